// Fused bf16 forward scan: one thread-block cluster per head, every stage of a
// frame in one kernel, nothing but the inputs and outputs crossing HBM.
//
// The scan runs in its affine form (gdn_internal.h):
//   S_t = g_t (S_{t-1} - M_t S_{t-1}) + b_t,
//   M_t = K~^T diag(beta) K~,  b_t = K~^T diag(beta) V_t,  O_t = Q_t S_t / sqrt(D).
// Value columns of the state evolve independently (column j of S_t depends only
// on column j of S_{t-1} and of b_t), so a head is split over NC = D/16 CTAs of
// one cluster, CTA r owning the 16 value columns J_r = [16r, 16r + 16).  Per
// frame t, CTA r:
//   gram    : [M_t[:, J_r] | b_t[:, J_r]] = K^T diag(beta) [K[:, J_r] | V[:, J_r]]
//             on tcgen05 (A = K tile, MN-major; B = beta-scaled columns, with
//             beta V split into bf16 hi + lo so b_t keeps ~16 significant bits);
//             fp32 accumulators in TMEM.
//   exchange: M_t's column block J_r (bf16) is written into this CTA's M image
//             and bulk-copied into the M image of every other CTA of the cluster
//             (distributed shared memory), so every CTA holds all of M_t.
//   scan    : P = M_t S_{t-1}[:, J_r] (tcgen05, the state as bf16 hi + lo), then
//             S_t[:, J_r] = g_t (S_{t-1} - P) + b_t in fp32 registers.
//   readout : O_t[:, J_r] = Q_t S_t[:, J_r] / sqrt(D) per 128-token tile (tcgen05),
//             stored as bf16 straight from registers.
// K and Q tiles are needed by every CTA of the cluster: each tile is fetched
// once from global memory and multicast into all of them (the CTA of rank
// tile % NC issues it); the cluster's CTAs also prefetch upcoming frames into
// L2, each its 1/NC share.  V[:, J_r] is loaded by CTA r alone.
//
// Roles (448 threads): warps 0-3 scan (thread i = state row i), warps 4-7
// read-out epilogue (thread = token of a tile), warps 8-11 beta scaling, warp 12
// TMA producer, warp 13 MMA issuer.  Every wait is bounded (2 s) and reports
// GDN_ERR_TIMEOUT through the status word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gdn_internal.h"
#include "ptx.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int kKTok = 64;                     // tokens per gram tile
constexpr int kQTok = 128;                    // tokens per read-out tile (MMA M)
constexpr int kKAtom = kKTok * 128;           // one 64-column atom of a K tile (8 KB)
constexpr int kQAtom = kQTok * 128;           // one 64-column atom of a Q tile (16 KB)
constexpr int kVcOff = 2 * kKAtom;            // V[:, J_r] tile: 64 rows x 2W bytes
constexpr int kQStage = 2 * kQAtom;           // 32 KB
constexpr int kQStages = 2;
constexpr uint32_t kTmemCols = 512;

// Shape of the kernel for W value columns per CTA (16 or 32).
template <int W>
struct Cfg {
  static constexpr int kScanWarps = W / 4;             // 16 state columns per scan thread
  static constexpr int kOutWarp0 = kScanWarps;         // 4 read-out epilogue warps
  static constexpr int kConvWarp0 = kScanWarps + 4;    // 4 beta-scaling warps
  static constexpr int kTmaWarp = kScanWarps + 8;
  static constexpr int kMmaWarp = kScanWarps + 9;
  static constexpr int kThreads = 32 * (kScanWarps + 10);
  static constexpr int kBgOff = kVcOff + kKTok * 2 * W;          // gram B operand (3W columns, 64-column atoms)
  static constexpr int kBgAtoms = (3 * W + 63) / 64;
  static constexpr int kKStage = kBgOff + kBgAtoms * kKAtom;     // 26 KB (W = 16) or 36 KB (W = 32)
  static constexpr int kKStages = 3;
  static constexpr int kMBufs = W == 16 ? 2 : 1;                 // M images in flight
  static constexpr int kSAtom = W * 128;                         // state image atom: W rows x 128 B
  static constexpr int kSImg = 2 * kSAtom;
  static constexpr uint32_t kAccG = 0;                           // gram accumulators at b * 128 (3W columns)
  static constexpr uint32_t kAccP = 256 - W;                     // scan accumulator (W columns)
  static constexpr uint32_t kAccO = 256;                         // read-out accumulators (W columns each)
  static constexpr int kOutSlots = 256 / W;
};

struct FusedArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* beta;
  const float* g;
  const float* state_in;
  __nv_bfloat16* out;
  float* state_out;
  int T, S, D, NC, NA;
  int gate_logits;
  float m_scale, b_scale, o_scale;
  unsigned int* status;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Bounded wait that also gives up when another role of this CTA has aborted; a
// timeout is recorded in the status word and raises the CTA's abort flag.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              unsigned int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kWaitTimeoutNs) {
        report_device_error(status, kTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// A bounded wait used only while tearing down.
__device__ __forceinline__ void wait_bounded(uint32_t bar, uint32_t parity, uint64_t ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > ns) return;
}

// Ring position plus, per slot, the parity of its last fill (for the teardown
// drain of the slots' release barriers).
struct Ring {
  int n, stage = 0;
  uint32_t phase = 0, used = 0, last = 0;
  __device__ explicit Ring(int n_) : n(n_) {}
  __device__ void fill() {
    used |= 1u << stage;
    last = (last & ~(1u << stage)) | (phase << stage);
  }
  __device__ void advance() {
    if (++stage == n) {
      stage = 0;
      phase ^= 1;
    }
  }
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// x -> bf16 hi + lo with hi = rne(x), lo = rne(x - hi), two values at a time.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}

__device__ __forceinline__ void unpack8(const uint4& w, float (&x)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[e]));
    x[2 * e] = f.x;
    x[2 * e + 1] = f.y;
  }
}

// Prefetches CTA `r`'s 1/NC share of a contiguous frame-head tile into L2.
__device__ __forceinline__ void prefetch_share(const __nv_bfloat16* base, long long f, int S, int D, int r, int NC) {
  const size_t tile = (size_t)S * D * 2;
  const size_t part = (((tile + NC - 1) / NC) + 15) & ~size_t(15);
  const size_t off = (size_t)r * part;
  if (off >= tile) return;
  const size_t len = tile - off < part ? tile - off : part;
  const uint8_t* p = reinterpret_cast<const uint8_t*>(base) + (size_t)f * tile + off;
  for (size_t o = 0; o < len; o += 65536) prefetch_l2(p + o, (uint32_t)(len - o < 65536 ? len - o : 65536));
}

template <int W>
__global__ void __launch_bounds__(Cfg<W>::kThreads, 1)
    tc_fused_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                    const __grid_constant__ CUtensorMap mapQ, FusedArgs a) {
  using C = Cfg<W>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int T = a.T, S = a.S, D = a.D, NC = a.NC, NA = a.NA;
  const int KS = D / 16;        // MMA K-steps over the head dim
  const int RM = NC * W;        // rows of an M image atom (key dims 16r.. of every CTA; >= D)
  const int mb = 2 * RM * 128;  // one M image: 2 atoms (m = key dim i, 64 each) x RM rows x 128 B
  uint8_t* kring = smem;
  uint8_t* qring = kring + C::kKStages * C::kKStage;
  uint8_t* mimg = qring + kQStages * kQStage;
  uint8_t* simg = mimg + ((C::kMBufs * mb + 1023) & ~1023);
  uint8_t* simg_lo = simg + C::kSImg;
  uint64_t* bars = reinterpret_cast<uint64_t*>(simg + 2 * C::kSImg);
  uint64_t* kfull = bars;
  uint64_t* kconv = kfull + C::kKStages;
  uint64_t* kempty = kconv + C::kKStages;
  uint64_t* qfull = kempty + C::kKStages;
  uint64_t* qempty = qfull + kQStages;
  uint64_t* gfull = qempty + kQStages;
  uint64_t* gempty = gfull + 2;
  uint64_t* mfull = gempty + 2;
  uint64_t* mempty = mfull + C::kMBufs;
  uint64_t* ofull = mempty + C::kMBufs;
  uint64_t* oempty = ofull + C::kOutSlots;
  uint64_t* pfull = oempty + C::kOutSlots;
  uint64_t* sready = pfull + 1;
  uint64_t* mma_done = sready + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const uint32_t r = cluster_rank();
  const long long bh = blockIdx.x / NC;
  const uint16_t all = (uint16_t)((1u << NC) - 1u);
  const int c0 = W * (int)r;  // first value column of this CTA

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(smem_u32(&kfull[s]), 1);
      mbar_init(smem_u32(&kconv[s]), 4);
      mbar_init(smem_u32(&kempty[s]), NC);
    }
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(smem_u32(&qfull[s]), 1);
      mbar_init(smem_u32(&qempty[s]), NC);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&gfull[b]), 1);
      mbar_init(smem_u32(&gempty[b]), C::kScanWarps);
    }
    for (int b = 0; b < C::kMBufs; ++b) {
      mbar_init(smem_u32(&mfull[b]), 1);
      mbar_init(smem_u32(&mempty[b]), NC);
    }
    for (int s = 0; s < C::kOutSlots; ++s) {
      mbar_init(smem_u32(&ofull[s]), 1);
      mbar_init(smem_u32(&oempty[s]), 4);
    }
    mbar_init(smem_u32(pfull), 1);
    mbar_init(smem_u32(sready), 1);
    mbar_init(smem_u32(mma_done), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Rows 64..127 of the gram A operand are key dims >= 64: zero when D <= 64
  // (TMA never writes that atom then).
  if (NA == 1)
    for (int s = 0; s < C::kKStages; ++s)
      for (int idx = threadIdx.x; idx < kKAtom / 16; idx += blockDim.x)
        reinterpret_cast<uint4*>(kring + s * C::kKStage + kKAtom)[idx] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == C::kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // barriers of every CTA initialised before any remote arrive or copy
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nkc = (S + kKTok - 1) / kKTok;
  const int nqc = (S + kQTok - 1) / kQTok;

  if (warp == C::kTmaWarp) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&mapK);
      prefetch_tmap(&mapV);
      prefetch_tmap(&mapQ);
      for (int u = 0; u < 2 && u < T; ++u) {
        prefetch_share(a.k, bh * T + u, S, D, r, NC);
        prefetch_share(a.v, bh * T + u, S, D, r, NC);
      }
      prefetch_share(a.q, bh * T, S, D, r, NC);
      Ring kr(C::kKStages), qr(kQStages);
      bool ok = true;
      auto load_k = [&](int u) {
        const long long f = bh * T + u;
        if (u + 2 < T) {
          prefetch_share(a.k, f + 2, S, D, r, NC);
          prefetch_share(a.v, f + 2, S, D, r, NC);
        }
        if (u + 1 < T) prefetch_share(a.q, f + 1, S, D, r, NC);
        for (int ch = 0; ok && ch < nkc; ++ch) {
          if (!wait_or_abort(smem_u32(&kempty[kr.stage]), kr.phase ^ 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          uint8_t* st = kring + kr.stage * C::kKStage;
          const uint32_t fb = smem_u32(&kfull[kr.stage]);
          mbar_arrive_expect_tx(fb, NA * kKAtom + kKTok * 2 * W);
          if (ch % NC == (int)r)
            for (int at = 0; at < NA; ++at)
              tma_load_3d_mc(smem_u32(st + at * kKAtom), &mapK, fb, 64 * at, ch * kKTok, (int)f, all);
          tma_load_3d(smem_u32(st + kVcOff), &mapV, fb, c0, ch * kKTok, (int)f);
          kr.fill();
          kr.advance();
        }
      };
      auto load_q = [&](int u) {
        const long long f = bh * T + u;
        for (int ch = 0; ok && ch < nqc; ++ch) {
          if (!wait_or_abort(smem_u32(&qempty[qr.stage]), qr.phase ^ 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          uint8_t* st = qring + qr.stage * kQStage;
          const uint32_t fb = smem_u32(&qfull[qr.stage]);
          mbar_arrive_expect_tx(fb, NA * kQAtom);
          if (ch % NC == (int)r)
            for (int at = 0; at < NA; ++at)
              tma_load_3d_mc(smem_u32(st + at * kQAtom), &mapQ, fb, 64 * at, ch * kQTok, (int)f, all);
          qr.fill();
          qr.advance();
        }
      };
      load_k(0);
      for (int t = 0; ok && t < T; ++t) {
        if (t + 1 < T) load_k(t + 1);
        if (t >= 1) load_q(t - 1);
      }
      if (ok) load_q(T - 1);
      // Every CTA's release of every slot has landed here: no remote arrive remains.
      for (int s = 0; s < C::kKStages; ++s)
        if (kr.used & (1u << s)) wait_bounded(smem_u32(&kempty[s]), (kr.last >> s) & 1u, 500000000ull);
      for (int s = 0; s < kQStages; ++s)
        if (qr.used & (1u << s)) wait_bounded(smem_u32(&qempty[s]), (qr.last >> s) & 1u, 500000000ull);
      // ...and every fill issued into this CTA has landed.
      for (int s = 0; s < C::kKStages; ++s)
        if (kr.used & (1u << s)) wait_bounded(smem_u32(&kfull[s]), (kr.last >> s) & 1u, 500000000ull);
      for (int s = 0; s < kQStages; ++s)
        if (qr.used & (1u << s)) wait_bounded(smem_u32(&qfull[s]), (qr.last >> s) & 1u, 500000000ull);
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_g = idesc_bf16(128, 3 * W, 1, 1);  // A K^T (MN-major), B beta-scaled (MN-major)
      const uint32_t id_s = idesc_bf16(128, W, 1, 0);      // A M_t (MN-major), B state (K-major)
      const uint32_t id_o = idesc_bf16(128, W, 0, 0);      // A Q (K-major), B state (K-major)
      int ks = 0, qs = 0, os = 0;
      uint32_t kph = 0, qph = 0, oph = 0;
      bool ok = true;
      auto gram = [&](int u) {
        const int b = u & 1;
        if (!wait_or_abort(smem_u32(&gempty[b]), ((u >> 1) & 1) ^ 1, abort_flag, a.status)) {
          ok = false;
          return;
        }
        tc_fence_after();
        const uint32_t acc = tmem + C::kAccG + b * 128;
        for (int ch = 0; ch < nkc; ++ch) {
          if (!wait_or_abort(smem_u32(&kconv[ks]), kph, abort_flag, a.status)) {
            ok = false;
            return;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(kring + ks * C::kKStage);
#pragma unroll
          for (int kk = 0; kk < kKTok / 16; ++kk)
            mma_bf16(acc, smem_desc(st + kk * 2048, kKAtom, 1024),
                     smem_desc(st + C::kBgOff + kk * 2048, kKAtom, 1024), id_g, (ch > 0 || kk > 0) ? 1u : 0u);
          mma_commit_mc(smem_u32(&kempty[ks]), all);
          if (++ks == C::kKStages) { ks = 0; kph ^= 1; }
        }
        mma_commit(smem_u32(&gfull[b]));
      };
      auto readout = [&](int u) {
        // S_u is state image completion u + 1.
        if (!wait_or_abort(smem_u32(sready), (u + 1) & 1, abort_flag, a.status)) {
          ok = false;
          return;
        }
        for (int ch = 0; ch < nqc; ++ch) {
          if (!wait_or_abort(smem_u32(&qfull[qs]), qph, abort_flag, a.status) ||
              !wait_or_abort(smem_u32(&oempty[os]), oph ^ 1, abort_flag, a.status)) {
            ok = false;
            return;
          }
          tc_fence_after();
          const uint32_t qb = smem_u32(qring + qs * kQStage);
          const uint32_t acc = tmem + C::kAccO + os * W;
          for (int kk = 0; kk < KS; ++kk) {
            const uint32_t ko = (kk >> 2) * kQAtom + (kk & 3) * 32;
            const uint32_t so = (kk >> 2) * C::kSAtom + (kk & 3) * 32;
            const uint64_t ad = smem_desc(qb + ko, 16, 1024);
            mma_bf16(acc, ad, smem_desc(smem_u32(simg) + so, 16, 1024), id_o, kk > 0 ? 1u : 0u);
            mma_bf16(acc, ad, smem_desc(smem_u32(simg_lo) + so, 16, 1024), id_o, 1u);
          }
          mma_commit_mc(smem_u32(&qempty[qs]), all);
          mma_commit(smem_u32(&ofull[os]));
          if (++qs == kQStages) { qs = 0; qph ^= 1; }
          if (++os == C::kOutSlots) { os = 0; oph ^= 1; }
        }
      };
      auto scan = [&](int t) {
        const int b = t % C::kMBufs;
        if (!wait_or_abort(smem_u32(&mfull[b]), (t / C::kMBufs) & 1, abort_flag, a.status) ||
            !wait_or_abort(smem_u32(sready), t & 1, abort_flag, a.status)) {
          ok = false;
          return;
        }
        tc_fence_after();
        const uint32_t mbase = smem_u32(mimg + b * mb);
        for (int kk = 0; kk < KS; ++kk) {
          const uint64_t ad = smem_desc(mbase + kk * 2048, RM * 128, 1024);
          const uint32_t so = (kk >> 2) * C::kSAtom + (kk & 3) * 32;
          mma_bf16(tmem + C::kAccP, ad, smem_desc(smem_u32(simg) + so, 16, 1024), id_s, kk > 0 ? 1u : 0u);
          mma_bf16(tmem + C::kAccP, ad, smem_desc(smem_u32(simg_lo) + so, 16, 1024), id_s, 1u);
        }
        mma_commit(smem_u32(pfull));
        mma_commit_mc(smem_u32(&mempty[b]), all);
      };
      gram(0);
      for (int t = 0; ok && t < T; ++t) {
        if (t + 1 < T) gram(t + 1);
        if (ok && t >= 1) readout(t - 1);
        if (ok) scan(t);
      }
      if (ok) readout(T - 1);
    }
  } else if (warp >= C::kConvWarp0) {
    // ------------------------------------------------------------------ beta scaling
    // thread = (token, part): part 0 scales K[:, J_r], part 1 splits beta V[:, J_r].
    const int ct = threadIdx.x - 32 * C::kConvWarp0;
    const int tok = ct & (kKTok - 1), part = ct >> 6;
    const int kat = c0 >> 6, kcol = c0 & 63;  // K columns J_r inside the tile
    int ks = 0;
    uint32_t kph = 0;
    for (int u = 0; u < T; ++u) {
      const long long f = bh * T + u;
      const float* bf = a.beta + f * S;
      for (int ch = 0; ch < nkc; ++ch) {
        const int s = ch * kKTok + tok;
        const float bs = s < S ? beta_of(__ldg(bf + s), a.gate_logits) : 0.f;
        if (!__all_sync(0xffffffffu, wait_or_abort(smem_u32(&kfull[ks]), kph, abort_flag, a.status))) goto done;
        uint8_t* st = kring + ks * C::kKStage;
        uint8_t* bg = st + C::kBgOff;
#pragma unroll
        for (int c = 0; c < W; c += 8) {
          float x[8];
          if (part == 0) {
            unpack8(*reinterpret_cast<const uint4*>(st + kat * kKAtom + sw128_off(tok, kcol + c)), x);
            uint4 o;
            o.x = pack_bf16(bs * x[0], bs * x[1]);
            o.y = pack_bf16(bs * x[2], bs * x[3]);
            o.z = pack_bf16(bs * x[4], bs * x[5]);
            o.w = pack_bf16(bs * x[6], bs * x[7]);
            *reinterpret_cast<uint4*>(bg + sw128_off(tok, c)) = o;
          } else {
            unpack8(*reinterpret_cast<const uint4*>(st + kVcOff + tok * 2 * W + 2 * c), x);
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) split2(bs * x[2 * e], bs * x[2 * e + 1], hi[e], lo[e]);
            const int nh = W + c, nl = 2 * W + c;  // Bg columns of the hi and lo parts
            *reinterpret_cast<uint4*>(bg + (nh >> 6) * kKAtom + sw128_off(tok, nh & 63)) =
                make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(bg + (nl >> 6) * kKAtom + sw128_off(tok, nl & 63)) =
                make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&kconv[ks]));
        if (++ks == C::kKStages) { ks = 0; kph ^= 1; }
      }
    }
  } else if (warp >= C::kOutWarp0) {
    // ------------------------------------------------------------------ read-out epilogue
    const int q4 = warp & 3;
    const int tok = q4 * 32 + lane;
    int os = 0;
    uint32_t oph = 0;
    for (int u = 0; u < T; ++u) {
      const long long f = bh * T + u;
      for (int ch = 0; ch < nqc; ++ch) {
        if (!__all_sync(0xffffffffu, wait_or_abort(smem_u32(&ofull[os]), oph, abort_flag, a.status))) goto done;
        tc_fence_after();
        float v[W];
#pragma unroll
        for (int c = 0; c < W; c += 16)
          tmem_ld16(tmem + ((uint32_t)(q4 * 32) << 16) + C::kAccO + os * W + c, *reinterpret_cast<float(*)[16]>(&v[c]));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&oempty[os]));
        const int s = ch * kQTok + tok;
        if (s < S) {
          __nv_bfloat16* dst = a.out + ((size_t)f * S + s) * D + c0;
#pragma unroll
          for (int c = 0; c < W; c += 16) {
            if (c0 + c < D) {
              uint4 o0, o1;
              o0.x = pack_bf16(v[c + 0] * a.o_scale, v[c + 1] * a.o_scale);
              o0.y = pack_bf16(v[c + 2] * a.o_scale, v[c + 3] * a.o_scale);
              o0.z = pack_bf16(v[c + 4] * a.o_scale, v[c + 5] * a.o_scale);
              o0.w = pack_bf16(v[c + 6] * a.o_scale, v[c + 7] * a.o_scale);
              o1.x = pack_bf16(v[c + 8] * a.o_scale, v[c + 9] * a.o_scale);
              o1.y = pack_bf16(v[c + 10] * a.o_scale, v[c + 11] * a.o_scale);
              o1.z = pack_bf16(v[c + 12] * a.o_scale, v[c + 13] * a.o_scale);
              o1.w = pack_bf16(v[c + 14] * a.o_scale, v[c + 15] * a.o_scale);
              reinterpret_cast<uint4*>(dst + c)[0] = o0;
              reinterpret_cast<uint4*>(dst + c)[1] = o1;
            }
          }
        }
        if (++os == C::kOutSlots) { os = 0; oph ^= 1; }
      }
    }
  } else {
    // ------------------------------------------------------------------ scan
    // thread (i, h) owns row i of 16 state columns: S[i][c0 + 16h .. c0 + 16h + 16).
    const int i = threadIdx.x & 127;
    const int h = warp >> 2;
    const int cj = c0 + 16 * h;  // first state column of this thread
    const bool row = i < D;
    const bool cols = cj < D;
    const int nscan = 32 * C::kScanWarps;
    float x[16], bcur[16], bnext[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      x[j] = 0.f;
      bcur[j] = 0.f;
      bnext[j] = 0.f;
    }
    if (row && cols && a.state_in) {
      const float4* si = reinterpret_cast<const float4*>(a.state_in + ((size_t)bh * D + i) * D + cj);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 w = si[q];
        x[4 * q] = w.x;
        x[4 * q + 1] = w.y;
        x[4 * q + 2] = w.z;
        x[4 * q + 3] = w.w;
      }
    }
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    // State image (B operand, K-major: row n = value column, k = i): element i of
    // rows 16h .. 16h + 15.
    auto write_state = [&]() {
      if (!row) return;
      uint8_t* hi = simg + (i >> 6) * C::kSAtom;
      uint8_t* lo = simg_lo + (i >> 6) * C::kSAtom;
#pragma unroll
      for (int n = 0; n < 16; n += 2) {
        uint32_t hv, lv;
        split2(x[n], x[n + 1], hv, lv);
        const uint32_t o0 = sw128_off(16 * h + n, i & 63), o1 = sw128_off(16 * h + n + 1, i & 63);
        *reinterpret_cast<uint16_t*>(hi + o0) = (uint16_t)(hv & 0xFFFF);
        *reinterpret_cast<uint16_t*>(hi + o1) = (uint16_t)(hv >> 16);
        *reinterpret_cast<uint16_t*>(lo + o0) = (uint16_t)(lv & 0xFFFF);
        *reinterpret_cast<uint16_t*>(lo + o1) = (uint16_t)(lv >> 16);
      }
    };
    // Gram epilogue of frame u: M_u[:, J_r] into every CTA's M image, b_u -> bdst.
    auto gram_epi = [&](int u, float (&bdst)[16]) -> bool {
      const int b = u & 1, mbuf = u % C::kMBufs;
      bool ok = __all_sync(0xffffffffu, wait_or_abort(smem_u32(&gfull[b]), (u >> 1) & 1, abort_flag, a.status));
      float m[16];
      if (ok) {
        tc_fence_after();
        float hv[16], lv[16];
        const uint32_t acc = tmem + lane_base + C::kAccG + b * 128 + 16 * h;
        tmem_ld16(acc, m);
        tmem_ld16(acc + W, hv);
        tmem_ld16(acc + 2 * W, lv);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) bdst[j] = a.b_scale * (hv[j] + lv[j]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&gempty[b]));
        // every CTA has finished the scan MMA that last read this M buffer
        ok = __all_sync(0xffffffffu, wait_or_abort(smem_u32(&mempty[mbuf]), ((u / C::kMBufs) & 1) ^ 1, abort_flag,
                                                   a.status));
      }
      if (ok) {
        // M image (A operand, MN-major): row k = c0 + 16h + j holds M[0..127][k];
        // thread i writes element i of each of its 16 rows.
        uint8_t* mi = mimg + mbuf * mb + (i >> 6) * (RM * 128);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          *reinterpret_cast<__nv_bfloat16*>(mi + sw128_off(cj + j, i & 63)) = __float2bfloat16_rn(a.m_scale * m[j]);
        fence_proxy_async_smem();
      }
      if (barrier_any(1, nscan, !ok || *abort_flag)) return false;
      if (threadIdx.x == 0) {
        const uint32_t fb = smem_u32(&mfull[mbuf]);
        mbar_arrive_expect_tx(fb, (uint32_t)(NC - 1) * 2 * (W * 128));
        const uint32_t src = smem_u32(mimg + mbuf * mb) + c0 * 128;
        for (int p = 0; p < NC; ++p) {
          if (p == (int)r) continue;
          const uint32_t dst = map_to_rank(src, p);
          const uint32_t rb = map_to_rank(fb, p);
          bulk_s2dsmem(dst, src, W * 128, rb);
          bulk_s2dsmem(dst + RM * 128, src + RM * 128, W * 128, rb);
        }
      }
      return true;
    };
    write_state();
    fence_proxy_async_smem();
    if (barrier_any(1, nscan, *abort_flag)) goto done;
    if (threadIdx.x == 0) mbar_arrive(smem_u32(sready));
    if (T > 0 && !gram_epi(0, bcur)) goto done;
    for (int t = 0; t < T; ++t) {
      if (t + 1 < T && !gram_epi(t + 1, bnext)) goto done;
      const long long f = bh * T + t;
      const float gt = decay_of(__ldg(a.g + f), a.gate_logits);
      const bool ok = __all_sync(0xffffffffu, wait_or_abort(smem_u32(pfull), t & 1, abort_flag, a.status));
      if (ok) {
        tc_fence_after();
        float p[16];
        tmem_ld16(tmem + lane_base + C::kAccP + 16 * h, p);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = fmaf(gt, x[j] - p[j], bcur[j]);
        tc_fence_before();
        write_state();
        fence_proxy_async_smem();
      }
      if (barrier_any(1, nscan, !ok || *abort_flag)) goto done;
      if (threadIdx.x == 0) mbar_arrive(smem_u32(sready));
#pragma unroll
      for (int j = 0; j < 16; ++j) bcur[j] = bnext[j];
    }
    if (row && cols && a.state_out) {
      float4* so = reinterpret_cast<float4*>(a.state_out + ((size_t)bh * D + i) * D + cj);
#pragma unroll
      for (int q = 0; q < 4; ++q) so[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    }
    // Every CTA's release of the last M images has landed here.
    if (threadIdx.x == 0)
      for (int u = T - C::kMBufs; u < T; ++u)
        if (u >= 0) wait_bounded(smem_u32(&mempty[u % C::kMBufs]), (u / C::kMBufs) & 1, 500000000ull);
  }
done:
  if (warp == C::kMmaWarp && lane == 0) {  // every MMA this CTA issued has completed
    mma_commit(smem_u32(mma_done));
    wait_bounded(smem_u32(mma_done), 0, 500000000ull);
  }
  tc_fence_before();
  cluster_sync();  // no CTA leaves while a peer may still write into it
  if (warp == C::kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 3D view [frames][S][D] of a bf16 [B,H,T,S,D] tensor with a cols x rows x 1 box.
bool make_map(CUtensorMap* m, const void* base, int D, int S, long long F, int cols, int rows,
              CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)F};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)S * D * 2};
  cuuint32_t box[3] = {(cuuint32_t)cols, (cuuint32_t)rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int W>
int fused_smem(int D) {
  using C = Cfg<W>;
  const int NC = (D + W - 1) / W;
  const int mb = 2 * NC * W * 128;
  return C::kKStages * C::kKStage + kQStages * kQStage + ((C::kMBufs * mb + 1023) & ~1023) + 2 * C::kSImg + 512 +
         1024;
}

template <int W>
int launch_fused(const Problem& p, const CUtensorMap& mapK, const CUtensorMap& mapQ, cudaStream_t st) {
  const long long F = p.BHT();
  CUtensorMap mapV;
  if (!make_map(&mapV, p.v, p.D, p.S, F, W, kKTok, CU_TENSOR_MAP_SWIZZLE_NONE)) return kCuda;
  const int NC = (p.D + W - 1) / W;
  const int smem = fused_smem<W>(p.D);
  if (cudaFuncSetAttribute(tc_fused_kernel<W>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return kCuda;
  FusedArgs fa{static_cast<const __nv_bfloat16*>(p.q),
               static_cast<const __nv_bfloat16*>(p.k),
               static_cast<const __nv_bfloat16*>(p.v),
               p.beta,
               p.g,
               p.state_in,
               static_cast<__nv_bfloat16*>(p.out),
               p.state_out,
               p.T,
               p.S,
               p.D,
               NC,
               (p.D + 63) / 64,
               p.gate_logits,
               p.key_scale * p.key_scale,
               p.key_scale,
               p.out_scale,
               p.status};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.BH() * NC));
  cfg.blockDim = dim3(Cfg<W>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = NC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  {
    ProfScope ps(st, W == 16 ? "tc_fused16" : "tc_fused32");
    e = cudaLaunchKernelEx(&cfg, tc_fused_kernel<W>, mapK, mapV, mapQ, fa);
  }
  return e == cudaSuccess ? kOk : kCuda;
}

// Value columns per CTA.  16 gives each CTA the least tensor work per frame but
// needs clusters of D/16 CTAs, of which fewer fit on the GPU at once (15 of 7 on
// a B300); 32 halves the cluster size.  GDN_FUSED_COLS=16|32 overrides.
int fused_cols(const Problem& p) {
  static int forced = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    const char* e = getenv("GDN_FUSED_COLS");
    forced = e ? atoi(e) : 0;
  });
  if (forced == 16 || forced == 32) return forced;
  if (p.D <= 16) return 16;
  int dev = 0, n16 = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 32;
  cudaLaunchConfig_t cfg = {};
  const int NC = p.D / 16;
  cfg.gridDim = dim3((unsigned)NC);
  cfg.blockDim = dim3(Cfg<16>::kThreads);
  cfg.dynamicSmemBytes = fused_smem<16>(p.D);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = NC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaFuncSetAttribute(tc_fused_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, cfg.dynamicSmemBytes) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n16, tc_fused_kernel<16>, &cfg) != cudaSuccess)
    return 32;
  return p.BH() <= n16 ? 16 : 32;
}

}  // namespace

bool fused_supported(const Problem& p) {
  return p.dtype == 1 && p.D % 16 == 0 && p.D >= 16 && p.D <= 128 && fused_smem<16>(p.D) <= 227 * 1024 &&
         fused_smem<32>(p.D) <= 227 * 1024;
}

int fused_forward(const Problem& p, cudaStream_t st) {
  const long long F = p.BHT();
  CUtensorMap mapK, mapQ;
  if (!make_map(&mapK, p.k, p.D, p.S, F, 64, kKTok, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&mapQ, p.q, p.D, p.S, F, 64, kQTok, CU_TENSOR_MAP_SWIZZLE_128B))
    return kCuda;
  return fused_cols(p) == 16 ? launch_fused<16>(p, mapK, mapQ, st) : launch_fused<32>(p, mapK, mapQ, st);
}

}  // namespace gdn
