// bf16 tensor-core path of the frame-wise GDN forward scan (sm_103a: tcgen05
// MMAs with TMEM accumulators, operands staged by TMA / bulk copies).
//
// The scan runs in its transition form (gdn_internal.h):
//   gram    : [M_t | b_t] = (diag(beta) K)^T [K | V], every frame-head in
//             parallel.  diag(beta)K is split into bf16 hi + lo parts (the lo
//             part only feeds b_t, whose precision sets the state's);
//             M_t -> bf16 image (the scan's B operand), b_t -> fp32.
//   scan    : per head, frame by frame: P^T = S^T M_t on the tensor core with S
//             split into bf16 hi + lo (A operand), then S <- g (S - P) + b_t in
//             fp32 registers.  Writes S_t as a bf16 hi/lo image for the read-out.
//   readout : O_t^T = S_t^T Q_t^T (A = S image, B = Q tile, N = 128 tokens),
//             epilogue x 1/sqrt(D) -> bf16 -> TMA store.
//
// Shared-memory tiles use 128-byte rows with the 128-byte swizzle.  A 16-bit
// matrix with more than 64 columns is kept as "atoms" of 64 columns each, one
// region per atom.  Descriptor conventions (canonical tcgen05 layouts):
//   K-major operand (K contiguous): SBO = 1024 (8 rows x 128 B); one MMA K-step of
//     16 elements advances the start address 32 bytes inside an atom.
//   MN-major operand (M/N contiguous): LBO = byte stride between 64-wide MN atoms,
//     SBO = 1024 (8 K-rows x 128 B); one K-step of 16 rows advances 2048 bytes.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <utility>

#include "../../include/gdn.h"
#include "gdn_internal.h"
#include "ptx.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int kGramTok = 64;                   // tokens per gram stage
constexpr int kGramRegion = kGramTok * 128;    // one 64-column atom of a stage
constexpr int kGramThreads = 448;              // 4 epilogue, 8 convert, 1 TMA, 1 MMA warps
constexpr int kOutTok = 128;                   // tokens per read-out tile (MMA M)
constexpr int kOutQStages = 2;
constexpr int kOutAcc = 4;                     // TMEM accumulators in flight
constexpr int kOutThreads = 320;               // 4 epilogue, 1 TMA, 1 MMA, 4 query-prep warps

__host__ __device__ inline int num_atoms(int D) { return (D + 63) / 64; }

// ---------------------------------------------------------------- workspace layout
struct TcLayout {
  size_t m_off, b_off, s_off, total;
  size_t m_bytes, b_bytes, s_bytes;  // per frame-head
  size_t maps_off, starts_off;       // prefix form: chunk maps [A|b] and chunk starts
};

constexpr int kTcChunkFrames = 16;  // frames per chunk of the prefix form

TcLayout tc_layout(const Problem& p, int mode = GDN_MODE_SPLIT) {
  TcLayout L{};
  const int NA = num_atoms(p.D);
  L.m_bytes = (size_t)NA * p.D * 128;      // M_t image: NA regions of D rows x 128 B
  L.b_bytes = (size_t)p.D * p.D * 4;       // b_t: fp32 column blocks [D/16][i][16]
  L.s_bytes = (size_t)2 * NA * p.D * 128;  // S_t image: hi/lo x NA regions of D rows
  const size_t F = (size_t)p.BHT();
  L.m_off = 0;
  L.b_off = align_up(L.m_off + F * L.m_bytes, 1024);
  L.s_off = align_up(L.b_off + F * L.b_bytes, 1024);
  L.total = align_up(L.s_off + F * L.s_bytes, 1024);
  if (mode == GDN_MODE_PREFIX) {
    const size_t nch = (size_t)((p.T + kTcChunkFrames - 1) / kTcChunkFrames);
    const size_t mat = (size_t)p.D * p.D * 4;
    L.maps_off = L.total;
    L.starts_off = align_up(L.maps_off + (size_t)p.BH() * nch * 2 * mat, 1024);
    L.total = align_up(L.starts_off + (size_t)p.BH() * nch * mat, 1024);
  }
  return L;
}

// ---------------------------------------------------------------- tensor maps
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

// 3D view [frames][S][D] of a bf16 [B,H,T,S,D] tensor; box = 64 columns x rows x 1 frame.
bool make_map(CUtensorMap* m, const void* base, int D, int S, long long F, int rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)F};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)S * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Bounded wait that also gives up when another role has aborted; a timeout is
// recorded in the status word and raises the CTA's abort flag.  After a first
// check the thread waits suspended (try_wait with a suspend-time hint: the
// hardware wakes it when the phase completes, or after the hint), so a waiting
// warp does not take issue slots from the warps sharing its sub-partition.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              unsigned int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (mbar_try_wait_suspend(bar, parity, kWaitSuspendNs)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kWaitTimeoutNs) {
      report_device_error(status, kTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

// A bounded wait used only while tearing down after an abort.
__device__ __forceinline__ void wait_bounded(uint32_t bar, uint32_t parity, uint64_t ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > ns) return;
}

// Pipeline ring position plus, per slot, the parity of the last fill issued into
// it, so that an aborting producer can wait for its own copies still in flight.
template <int N>
struct Ring {
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued_mask = 0;
  uint32_t last_phase_mask = 0;
  __device__ void mark_issued() {
    issued_mask |= 1u << stage;
    last_phase_mask = (last_phase_mask & ~(1u << stage)) | (phase << stage);
  }
  __device__ void advance() {
    if (++stage == N) {
      stage = 0;
      phase ^= 1;
    }
  }
  // Waits (bounded) for the last fill of every slot to land on its `full` barrier.
  __device__ void drain(const uint64_t* full) const {
    for (int s = 0; s < N; ++s)
      if (issued_mask & (1u << s)) wait_bounded(smem_u32(&full[s]), (last_phase_mask >> s) & 1u, 500000000ull);
  }
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Splits x into bf16 hi + lo with hi = rne(x), lo = rne(x - hi).
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}

// =============================================================================
// gram: [M_t | b_t] = (diag(beta) K)^T [K | V] per frame-head.
//
// Persistent CTAs stream K and V tiles of 64 tokens through a 4-deep ring (TMA);
// eight warps scale each tile by beta and split it into bf16 hi + lo parts in a
// 2-deep ring of their own; one thread issues the MMAs; four warps drain the
// fp32 accumulators (double-buffered in TMEM) into
//   the M_t image: bf16, the scan's A operand (K-major, 128-byte swizzle, NA
//     atoms of D rows x 128 B), staged in shared memory and bulk-stored;
//   b_t: fp32 in column blocks of 16 ([D/16][D rows][16]), so each block the
//     scan's column-split CTAs read is contiguous.
// =============================================================================
constexpr int kGramRaw = 4;
constexpr int kGramConv = 2;
constexpr int kRawStage = 4 * kGramRegion;   // K atoms (NA) then V atoms (NA): 32 KB
constexpr int kConvStage = 4 * kGramRegion;  // AH atoms (2) then AL atoms (2): 32 KB

struct GramArgs {
  const float* beta;
  int gate_logits;
  int variant;
  uint8_t* m_img;  // F x NA x D rows x 128 B
  float* b_blk;    // F x (D/16) x D x 16
  long long nitems;
  int S, D, NA;
  float m_scale, b_scale;
  unsigned int* status;
  // 1: only the b part, with beta = 1 (the backward's Q^T dO: K holds Q, V holds
  // dO); no M image.  The A operand is then the Q tile itself, exact in bf16: the
  // MMA reads it straight from the TMA ring and the beta-scaling warps sit out.
  int b_only;
  size_t m_span, b_span;  // extents (bytes) of the M image and b block regions (debug checks)
};

constexpr int kGramTmaWarp = 12, kGramMmaWarp = 13;  // warps 0-3 epilogue, 4-11 converters

__global__ void __launch_bounds__(kGramThreads, 1)
    tc_gram_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV, GramArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int NA = a.NA, D = a.D, S = a.S;
  uint8_t* raw = smem;
  uint8_t* conv = raw + kGramRaw * kRawStage;
  uint8_t* mstage = conv + kGramConv * kConvStage;  // NA x D rows x 128 B
  uint64_t* bars = reinterpret_cast<uint64_t*>(mstage + NA * D * 128);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + kGramRaw;
  uint64_t* conv_full = raw_empty + kGramRaw;
  uint64_t* conv_empty = conv_full + kGramConv;
  uint64_t* accfull = conv_empty + kGramConv;
  uint64_t* accempty = accfull + 2;
  uint64_t* mma_done = accempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGramRaw; ++s) {
      mbar_init(smem_u32(&raw_full[s]), 1);
      mbar_init(smem_u32(&raw_empty[s]), 1);
    }
    for (int s = 0; s < kGramConv; ++s) {
      mbar_init(smem_u32(&conv_full[s]), 8);
      mbar_init(smem_u32(&conv_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&accfull[b]), 1);
      mbar_init(smem_u32(&accempty[b]), 4);
    }
    mbar_init(smem_u32(mma_done), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // The A operands span 128 rows of M (key dims); with one atom (D <= 64) the
  // second atom's rows are never converted: zero them once, so those accumulator
  // rows, which nothing reads, stay finite.
  if (NA == 1)
    for (int s = 0; s < kGramConv; ++s)
      for (int idx = threadIdx.x; idx < kGramRegion / 16; idx += blockDim.x) {
        reinterpret_cast<uint4*>(conv + s * kConvStage + kGramRegion)[idx] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4*>(conv + s * kConvStage + 3 * kGramRegion)[idx] = make_uint4(0, 0, 0, 0);
      }
  fence_proxy_async_smem();
  if (warp == kGramMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nchunks = (S + kGramTok - 1) / kGramTok;
  // (launched with programmatic stream serialization: everything above overlaps
  // the preceding kernel; no global memory is touched before this wait)
  griddep_wait();
  griddep_launch_dependents();

  if (warp == kGramTmaWarp) {
    // ---------------- TMA producer
    if (lane == 0) {
      prefetch_tmap(&mapK);
      prefetch_tmap(&mapV);
      Ring<kGramRaw> r;
      bool ok = true;
      for (long long f = blockIdx.x; ok && f < a.nitems; f += gridDim.x) {
        for (int c = 0; c < nchunks; ++c) {
          if (!wait_or_abort(smem_u32(&raw_empty[r.stage]), r.phase ^ 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          uint8_t* st = raw + r.stage * kRawStage;
          const uint32_t fb = smem_u32(&raw_full[r.stage]);
          mbar_arrive_expect_tx(fb, 2 * NA * kGramRegion);
          for (int at = 0; at < NA; ++at) {
            tma_load_3d(smem_u32(st + at * kGramRegion), &mapK, fb, 64 * at, c * kGramTok, (int)f);
            tma_load_3d(smem_u32(st + (NA + at) * kGramRegion), &mapV, fb, 64 * at, c * kGramTok, (int)f);
          }
          r.mark_issued();
          r.advance();
        }
      }
      r.drain(raw_full);  // every issued load has landed before the CTA may exit
    }
  } else if (warp == kGramMmaWarp) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t id1 = idesc_bf16(128, NA * 64 + D, 1, 1);
      const uint32_t id2 = idesc_bf16(128, D, 1, 1);
      // Descriptors of ring stage 0 and K-step 0; a stage or K-step only moves the
      // start address (the low 14-bit field, in 16-byte units; every address here
      // stays below 2^18, so the sum never carries into the next field).  Building
      // each descriptor afresh per MMA cost the issuing warp ~100 cycles an MMA.
      const uint64_t dK0 = smem_desc(smem_u32(raw), kGramRegion, 1024);
      const uint64_t dV0 = smem_desc(smem_u32(raw + NA * kGramRegion), kGramRegion, 1024);
      const uint64_t dH0 = smem_desc(smem_u32(conv), kGramRegion, 1024);
      const uint64_t dL0 = smem_desc(smem_u32(conv + 2 * kGramRegion), kGramRegion, 1024);
      const uint32_t accb = NA * 64;
      int rs = 0, cs = 0, ab = 0;
      uint32_t rph = 0, cph = 0, aph = 0;
      for (long long f = blockIdx.x; f < a.nitems; f += gridDim.x) {
        if (!wait_or_abort(smem_u32(&accempty[ab]), aph ^ 1, abort_flag, a.status)) goto done;
        tc_fence_after();
        const uint32_t acc = tmem + ab * 256;
        for (int c = 0; c < nchunks; ++c) {
          if (!wait_or_abort(a.b_only ? smem_u32(&raw_full[rs]) : smem_u32(&conv_full[cs]), a.b_only ? rph : cph,
                             abort_flag, a.status))
            goto done;
          tc_fence_after();
          const uint64_t ro = (uint64_t)((rs * kRawStage) >> 4), co = (uint64_t)((cs * kConvStage) >> 4);
#pragma unroll
          for (int kk = 0; kk < kGramTok / 16; ++kk) {
            const uint64_t ko = (uint64_t)((kk * 2048) >> 4);
            const uint32_t accum = (c > 0 || kk > 0) ? 1u : 0u;
            if (a.b_only) {
              mma_bf16(acc + accb, dK0 + ro + ko, dV0 + ro + ko, id2, accum);
              continue;
            }
            mma_bf16(acc, dH0 + co + ko, dK0 + ro + ko, id1, accum);
            mma_bf16(acc + accb, dL0 + co + ko, dV0 + ro + ko, id2, 1u);
          }
          mma_commit(smem_u32(&raw_empty[rs]));
          if (++rs == kGramRaw) { rs = 0; rph ^= 1; }
          if (!a.b_only) {
            mma_commit(smem_u32(&conv_empty[cs]));
            if (++cs == kGramConv) { cs = 0; cph ^= 1; }
          }
        }
        mma_commit(smem_u32(&accfull[ab]));
        if (++ab == 2) { ab = 0; aph ^= 1; }
      }
    }
  } else if (warp >= 4) {
    // ---------------- beta scaling: A = diag(beta) K, split into bf16 hi + lo.
    // Elementwise, so each 16-byte chunk is transformed where it lies in the
    // swizzled tile (the hi / lo tiles share the K tile's layout).
    if (a.b_only) goto done;  // the MMA reads the raw tiles
    const int ct = threadIdx.x - 128;
    int rs = 0, cs = 0;
    uint32_t rph = 0, cph = 0;
    const int units = NA * kGramTok * 8;  // 16-byte chunks of K per tile (at most 4 per thread)
    const bool relu_k = a.variant == kReluLinear;
    // This thread's chunks lie in tile rows r0 and r0 + 32; their beta values are
    // loaded one tile ahead so the load latency stays off the critical path.
    const int r0 = ct >> 3;
    auto beta_at = [&](long long f, int c, int rw) {
      const int s = c * kGramTok + rw;
      // raw value, mapped when used: mapping here would wait for the load
      if (!(f < a.nitems && s < S)) return -INFINITY;
      return (a.variant == kReluLinear || a.b_only) ? 1.f : __ldg(a.beta + f * S + s);
    };
    long long fn = blockIdx.x;
    int cn = 0;
    // beta of token rows r0 and r0 + 32: raw values loaded one tile ahead, mapped
    // (rows past S, loaded as -inf, give 0) after the current tile is converted.
    auto mapped = [&](float x) {
      return x == -INFINITY ? 0.f : ((a.variant == kReluLinear || a.b_only) ? x : beta_of(x, a.gate_logits));
    };
    float bn0 = beta_at(fn, 0, r0), bn1 = beta_at(fn, 0, r0 + 32);
    float b0 = mapped(bn0), b1 = mapped(bn1);
    for (long long f = blockIdx.x; f < a.nitems; f += gridDim.x) {
      for (int c = 0; c < nchunks; ++c) {
        if (++cn == nchunks) { cn = 0; fn += gridDim.x; }
        bn0 = beta_at(fn, cn, r0);
        bn1 = beta_at(fn, cn, r0 + 32);
        const bool ok = wait_or_abort(smem_u32(&raw_full[rs]), rph, abort_flag, a.status) &&
                        wait_or_abort(smem_u32(&conv_empty[cs]), cph ^ 1, abort_flag, a.status);
        if (!__all_sync(0xffffffffu, ok)) goto done;
        const uint8_t* kt = raw + rs * kRawStage;
        uint8_t* ah = conv + cs * kConvStage;
        // This thread's (at most four) 16-byte chunks: every load issued before any
        // arithmetic, so the shared-memory latencies overlap.  (Chunks of key
        // columns past D hold the tile's zero fill and convert to zeros.)
        uint4 kv[4];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
          if (ct + 256 * rr < units) kv[rr] = *reinterpret_cast<const uint4*>(kt + (ct + 256 * rr) * 16);
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          if (ct + 256 * rr >= units) break;
          const float bs = (rr & 1) ? b1 : b0;
          const uint32_t w[4] = {kv[rr].x, kv[rr].y, kv[rr].z, kv[rr].w};
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
            if (relu_k)
              split2(bs * fmaxf(x.x, 0.f), bs * fmaxf(x.y, 0.f), hi[e], lo[e]);
            else
              split2(bs * x.x, bs * x.y, hi[e], lo[e]);
          }
          const int u = ct + 256 * rr;
          *reinterpret_cast<uint4*>(ah + u * 16) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(ah + 2 * kGramRegion + u * 16) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&conv_full[cs]));
        if (++rs == kGramRaw) { rs = 0; rph ^= 1; }
        if (++cs == kGramConv) { cs = 0; cph ^= 1; }
        b0 = mapped(bn0);
        b1 = mapped(bn1);
      }
    }
  } else if (warp < 4) {
    // ---------------- epilogue: TMEM -> M image (bf16, staged) and b (fp32 column blocks)
    const int i = warp * 32 + lane;  // accumulator row = key index
    const int ncb = D / 16;
    int ab = 0;
    uint32_t aph = 0;
    for (long long f = blockIdx.x; f < a.nitems; f += gridDim.x) {
      if (threadIdx.x == 0) bulk_wait_read0();  // the previous M image store has read the stage
      const bool ok = __all_sync(0xffffffffu, wait_or_abort(smem_u32(&accfull[ab]), aph, abort_flag, a.status));
      if (barrier_any(1, 128, !ok || *abort_flag)) goto done;
      tc_fence_after();
      const uint32_t acc = tmem + ((uint32_t)(warp * 32) << 16) + ab * 256;
      for (int c0 = 0; c0 < (a.b_only ? 0 : D); c0 += 16) {
        float v[16];
        tmem_ld16(acc + c0, v);
        tmem_ld_wait();
        if (i < D) {
          uint8_t* reg = mstage + (c0 >> 6) * D * 128;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint4 o;
            o.x = pack_bf16(v[8 * h + 0] * a.m_scale, v[8 * h + 1] * a.m_scale);
            o.y = pack_bf16(v[8 * h + 2] * a.m_scale, v[8 * h + 3] * a.m_scale);
            o.z = pack_bf16(v[8 * h + 4] * a.m_scale, v[8 * h + 5] * a.m_scale);
            o.w = pack_bf16(v[8 * h + 6] * a.m_scale, v[8 * h + 7] * a.m_scale);
            *reinterpret_cast<uint4*>(reg + sw128_off(i, (c0 & 63) + 8 * h)) = o;
          }
        }
      }
      for (int cb = 0; cb < ncb; ++cb) {
        float v[16];
        tmem_ld16(acc + NA * 64 + 16 * cb, v);
        tmem_ld_wait();
        if (i < D && in_region(((((size_t)f * ncb + cb) * D + i) * 16 + 16) * 4, a.b_span, a.status)) {
          // row i of the block: 64 contiguous bytes (the workspace is 256-byte aligned)
          float* dst = a.b_blk + (((size_t)f * ncb + cb) * D + i) * 16;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(v[8 * q + e] * a.b_scale);
            st_global_v8(dst + 8 * q, w);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&accempty[ab]));
      if (++ab == 2) { ab = 0; aph ^= 1; }
      fence_proxy_async_smem();
      named_barrier(1, 128);
      if (threadIdx.x == 0 && !a.b_only) {
        if (in_region(((size_t)f + 1) * NA * D * 128, a.m_span, a.status))
          bulk_s2g(a.m_img + (size_t)f * NA * D * 128, smem_u32(mstage), NA * D * 128);
        bulk_commit();
      }
    }
  }
done:
  if (threadIdx.x == 0) bulk_wait0();  // M image stores complete
  if (warp == kGramMmaWarp && lane == 0) {  // every MMA this CTA issued has completed
    mma_commit(smem_u32(mma_done));
    wait_bounded(smem_u32(mma_done), 0, 500000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kGramMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// =============================================================================
// scan: S_t[:, J] = g_t (S_{t-1}[:, J] - M_t S_{t-1}[:, J]) + b_t[:, J], frame by frame.
//
// Columns of the state evolve independently, so each head is split over D/16
// CTAs, CTA c owning the value columns J = [16c, 16c + 16): no communication.
// Per frame: P = M_t S_{t-1}[:, J] on the tensor core (A = the M_t image, B =
// the state block as bf16 hi and lo side by side, N = 32, the two halves summed
// in the epilogue), then the update in fp32 registers (thread i = state row i).
// M_t and the b_t block stream in through a ring of bulk copies; the new state
// block goes back to the read-out's S_t image with bulk stores (hi / lo, NA
// atoms, rows 16c .. 16c + 15 of each).
//
// Chunked forms (the prefix composition of the affine maps; zhichai.net SANA-WM
// summary, training pipeline Stage 3): the frames of a head are cut into chunks
// of `chunk` frames, one CTA per (head, chunk, column block), all in parallel.
//   summary : each chunk's composed map [A_c | b_c] (S_end = A_c S_start + b_c):
//             the A columns start as the identity's columns and take no b_t
//             term, the b columns start at zero; written to `maps`.
//   replay  : each chunk from its true initial state (`starts`), writing the
//             S_t images as the single pass does.
// =============================================================================
// Warps 0-7 epilogue (two per TMEM lane quadrant, 8 of the block's 16 columns
// each), warp 8 copies, warp 9 issues the MMAs.
constexpr int kScanEpiWarps = 8, kScanCopyWarp = 8, kScanMmaWarp = 9;
constexpr int kScanThreads = 320;
constexpr int kScanMStage = 2 * 128 * 128;  // M image: 2 atoms x 128 rows x 128 B
constexpr int kScanBStage = 128 * 64;       // b block: up to 128 rows x 16 floats
constexpr int kScanImg = 2 * 32 * 128;      // state block image: 2 atoms x 32 rows (hi 0-15, lo 16-31) x 128 B
constexpr int kScanImgBufs = 3;             // image buffers: MMA input, epilogue output, store in flight

struct ScanArgs {
  const uint8_t* m_img;
  const float* b_blk;
  const float* g;
  int gate_logits;
  int variant;
  const float* state_in;
  uint8_t* s_img;
  float* state_out;
  int T, D, NA;
  unsigned int* status;
  // 1: the backward pass's state-gradient scan, U_{t-1} = g_t (U_t - M_t U_t) + E_{t-1}
  // over t = T-1 .. 0.  b_blk holds E; state_in is dS_T and the scan starts from
  // U_{T-1} = dS_T + E_{T-1}; image slot t receives U_t (t = T-1 .. 0); state_out
  // receives dS_0 = g_0 (U_0 - M_0 U_0).  Not chunked.
  int reverse;
  // Chunking: frames per chunk and the number of chunks (T and 1 for one pass).
  int chunk, nchunks;
  // replay: the initial state of every chunk, [BH][nchunks][D][D] float32
  // (null: state_in, for one pass).  state_out is written by the last chunk.
  const float* starts;
  // summary: [BH][nchunks][D][2D] float32, row i = [A_c row i | b_c row i]; the
  // grid then has 2 D/16 column blocks per chunk (A's, then b's) and no image or
  // state_out is written.
  float* maps;
  // extents (bytes) of the M image, b block, state image, maps and starts regions
  // (debug checks)
  size_t m_span, b_span, s_span, maps_span, starts_span;
};

template <int STAGES>
__global__ void __launch_bounds__(kScanThreads, (STAGES <= 2 ? 2 : 1)) tc_scan_kernel(ScanArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int NA = a.NA, D = a.D, T = a.T;
  const int ncb = D / 16, KS = D / 16;
  uint8_t* mring = smem;
  uint8_t* bring = mring + STAGES * kScanMStage;
  uint8_t* img = bring + STAGES * kScanBStage;  // kScanImgBufs buffers
  uint64_t* bars = reinterpret_cast<uint64_t*>(img + kScanImgBufs * kScanImg);
  uint64_t* full = bars;
  uint64_t* empty = full + STAGES;
  uint64_t* pfull = empty + STAGES;
  uint64_t* sready = pfull + 1;
  uint64_t* mma_done = sready + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  // block -> (head, chunk, column block); in summary form column blocks 0 .. ncb-1
  // are A's (identity start, no b term), ncb .. 2 ncb - 1 are b's
  const int ncbx = a.maps ? 2 * ncb : ncb;
  const int cbx = (int)(blockIdx.x % ncbx);
  const long long hc = blockIdx.x / ncbx;
  const int chunk_id = (int)(hc % a.nchunks);
  const long long bh = hc / a.nchunks;
  const bool ident = a.maps != nullptr && cbx < ncb;
  const int cb = cbx < ncb ? cbx : cbx - ncb;
  const int t0 = chunk_id * a.chunk;
  const int nsteps = min(T, t0 + a.chunk) - t0;
  const bool use_b = !ident;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1 + kScanEpiWarps);  // the MMA's commit + each epilogue warp (b read)
    }
    mbar_init(smem_u32(pfull), 1);
    mbar_init(smem_u32(sready), kScanEpiWarps);  // each epilogue warp, once its part of the state image is written
    mbar_init(smem_u32(mma_done), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // M image rows D..127 of each atom (never copied in) must be finite: zero them once.
  {
    const int tail = (128 - D) * 8;  // 16-byte chunks per atom
    for (int idx = threadIdx.x; idx < STAGES * 2 * tail; idx += blockDim.x) {
      const int region = idx / tail, c = idx % tail;  // region = stage * 2 + atom
      reinterpret_cast<uint4*>(mring + region * (128 * 128) + D * 128)[c] = make_uint4(0, 0, 0, 0);
    }
  }
  fence_proxy_async_smem();
  if (warp == kScanMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 32);  // P_hi (columns 0-15) and P_lo (16-31)
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();  // no global memory is touched before the preceding kernel completes
  griddep_launch_dependents();

  if (warp == kScanCopyWarp) {
    // ---------------- copies in: M_t image (NA atoms of D rows) and the b_t block
    if (lane == 0) {
      Ring<STAGES> r;
      for (int j = 0; j < nsteps; ++j) {
        if (!wait_or_abort(smem_u32(&empty[r.stage]), r.phase ^ 1, abort_flag, a.status)) break;
        const int t = a.reverse ? T - 1 - j : t0 + j;
        const long long f = bh * T + t;
        // the b term of step j: b_t forward, E_{t-1} in reverse (frame 0's block,
        // unused, stands in for E_{-1})
        const long long fbk = a.reverse ? bh * T + (t > 0 ? t - 1 : 0) : f;
        const uint32_t fb = smem_u32(&full[r.stage]);
        mbar_arrive_expect_tx(fb, NA * D * 128 + (use_b ? D * 64 : 0));
        const uint8_t* src = a.m_img + (size_t)f * NA * D * 128;
        if (in_region(((size_t)f + 1) * NA * D * 128, a.m_span, a.status))
          for (int at = 0; at < NA; ++at)
            bulk_g2s(smem_u32(mring + r.stage * kScanMStage + at * 128 * 128), src + at * D * 128, D * 128, fb);
        if (use_b && in_region(((size_t)fbk * ncb + cb + 1) * D * 64, a.b_span, a.status))
          bulk_g2s(smem_u32(bring + r.stage * kScanBStage), a.b_blk + ((size_t)fbk * ncb + cb) * D * 16, D * 64, fb);
        r.mark_issued();
        r.advance();
      }
      r.drain(full);
    }
  } else if (warp == kScanMmaWarp) {
    // ---------------- MMA: P = M_t S_{t-1}[:, J]
    if (lane == 0) {
      const uint32_t id = idesc_bf16(128, 32, 0, 0);
      const bool store = a.s_img != nullptr;
      // the state block after step u (image buffer (u + 1) % 3; u = -1 is the
      // initial state) to global memory, laid out as in shared memory: the slot
      // of frame t0 + u, or in reverse slot T - 2 - u (the frame index of the
      // gradient U it holds)
      auto store_block = [&](int u) {
        const long long f = bh * T + (a.reverse ? T - 2 - u : t0 + u);
        if (in_region(((size_t)f * ncb + cb + 1) * NA * (32 * 128), a.s_span, a.status))
          bulk_s2g(a.s_img + ((size_t)f * ncb + cb) * NA * (32 * 128),
                   smem_u32(img + ((u + 1) % kScanImgBufs) * kScanImg), NA * 32 * 128);
        bulk_commit();
      };
      // Descriptors of stage 0 / buffer 0; the other stages and buffers only move
      // the start address (a 16-byte-unit field, well inside its 14 bits here).
      uint64_t ad0[8], bd0[8];
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        ad0[kk] = smem_desc(smem_u32(mring) + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024);
        bd0[kk] = smem_desc(smem_u32(img) + (kk >> 2) * (32 * 128) + (kk & 3) * 32, 16, 1024);
      }
      int stage = 0, buf = 0;  // buf = j % 3: the image buffer S_{j-1} is in
      uint32_t phase = 0;
      for (int j = 0; j < nsteps; ++j) {
        if (!wait_or_abort(smem_u32(&full[stage]), phase, abort_flag, a.status)) goto done;
        if (!wait_or_abort(smem_u32(sready), j & 1, abort_flag, a.status)) goto done;
        tc_fence_after();
        // The store of S_{j-3} (issued two steps ago) has read its buffer, which S_j
        // may overwrite once pfull(j) fires; the store of S_{j-2} may still be
        // reading.  Waiting here, before the MMAs, keeps the store issue below off
        // the frame's critical path.
        asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        const uint64_t ao = (uint64_t)((stage * kScanMStage) >> 4);
        const uint64_t bo = (uint64_t)((buf * kScanImg) >> 4);
        if (++buf == kScanImgBufs) buf = 0;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          if (kk < KS) mma_bf16(tmem, ad0[kk] + ao, bd0[kk] + bo, id, kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(pfull));
        mma_commit(smem_u32(&empty[stage]));
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
        if (store && (j >= 1 || a.reverse)) store_block(j - 1);
      }
      if (store && nsteps > 0 && !a.reverse) {  // the reverse scan's last result is dS_0 (state_out only)
        if (!wait_or_abort(smem_u32(sready), nsteps & 1, abort_flag, a.status)) goto done;
        store_block(nsteps - 1);
      }
    }
  } else {
    // ---------------- epilogue (8 warps): thread (i, h) owns row i of the column
    // block, columns 8h .. 8h + 7 (i = 32 (warp % 4) + lane, h = warp / 4; a warp
    // reads TMEM lanes 32 (warp % 4) ..)
    const int i = (warp & 3) * 32 + lane, h8 = 8 * (warp >> 2);
    const bool row = i < D;
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = (ident && i == 16 * cb + h8 + j) ? 1.f : 0.f;
    const float* s_init = a.starts ? a.starts + (size_t)(bh * a.nchunks + chunk_id) * D * D
                                   : (a.maps ? nullptr : (a.state_in ? a.state_in + (size_t)bh * D * D : nullptr));
    // (rows past D read nothing, so they check nothing)
    const bool init_ok = !a.starts || !row ||
                         in_region(((size_t)(bh * a.nchunks + chunk_id) * D * D + (size_t)i * D + 16 * cb + h8 + 8) * 4,
                                   a.starts_span, a.status);
    if (row && s_init && init_ok) {
      const float4* si = reinterpret_cast<const float4*>(s_init + (size_t)i * D + 16 * cb + h8);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float4 w = si[q];
        x[4 * q] = w.x;
        x[4 * q + 1] = w.y;
        x[4 * q + 2] = w.z;
        x[4 * q + 3] = w.w;
      }
    }
    if (row && a.reverse && T > 0) {  // U_{T-1} = dS_T + E_{T-1}
      const float4* e =
          reinterpret_cast<const float4*>(a.b_blk + (((size_t)(bh * T + T - 1) * ncb + cb) * D + i) * 16 + h8);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float4 w = e[q];
        x[4 * q] += w.x;
        x[4 * q + 1] += w.y;
        x[4 * q + 2] += w.z;
        x[4 * q + 3] += w.w;
      }
    }
    // state block image (B operand, K-major: row n = value column 16cb + n for the
    // hi part, row 16 + n for the lo part; k = i)
    auto write_img = [&](uint8_t* im) {
      if (!row) return;
      uint8_t* at = im + (i >> 6) * (32 * 128);
#pragma unroll
      for (int n = 0; n < 8; n += 2) {
        uint32_t hv, lv;
        split2(x[n], x[n + 1], hv, lv);
        *reinterpret_cast<uint16_t*>(at + sw128_off(h8 + n, i & 63)) = (uint16_t)(hv & 0xFFFF);
        *reinterpret_cast<uint16_t*>(at + sw128_off(h8 + n + 1, i & 63)) = (uint16_t)(hv >> 16);
        *reinterpret_cast<uint16_t*>(at + sw128_off(16 + h8 + n, i & 63)) = (uint16_t)(lv & 0xFFFF);
        *reinterpret_cast<uint16_t*>(at + sw128_off(17 + h8 + n, i & 63)) = (uint16_t)(lv >> 16);
      }
    };
    write_img(img);  // the initial state into buffer 0
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(sready));
    int stage = 0;
    uint32_t phase = 0;
    const bool relu_lin = a.variant == kReluLinear;  // g = 1, no delta-rule term
    // raw decay of the next step's frame; mapped when used
    float gnext = (nsteps > 0 && !relu_lin) ? __ldg(a.g + bh * T + (a.reverse ? T - 1 : t0)) : 0.f;
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16) + h8;
    for (int j = 0; j < nsteps; ++j) {  // j counts steps; the step's frame is fr
      const int fr = a.reverse ? T - 1 - j : t0 + j;
      const long long f = bh * T + fr;
      const float gt = relu_lin ? 1.f : decay_of(gnext, a.gate_logits);
      if (j + 1 < nsteps && !relu_lin) gnext = __ldg(a.g + (a.reverse ? f - 1 : f + 1));
      const bool add_b = use_b && !(a.reverse && fr == 0);  // E_{-1} = 0
      const bool ok = wait_or_abort(smem_u32(pfull), j & 1, abort_flag, a.status) &&
                      wait_or_abort(smem_u32(&full[stage]), phase, abort_flag, a.status);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        float p[8], pl[8];
        tmem_ld8(tl, p);
        tmem_ld8(tl + 16, pl);
        float bv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) bv[q] = 0.f;
        if (row && use_b) {
          const float4* bp = reinterpret_cast<const float4*>(bring + stage * kScanBStage + i * 64 + h8 * 4);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const float4 w = bp[q];
            bv[4 * q] = w.x;
            bv[4 * q + 1] = w.y;
            bv[4 * q + 2] = w.z;
            bv[4 * q + 3] = w.w;
          }
        }
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[stage]));
        if (row) {
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            x[jj] = relu_lin ? x[jj] + bv[jj] : fmaf(gt, x[jj] - (p[jj] + pl[jj]), add_b ? bv[jj] : 0.f);
        }
        // S_j goes into the buffer of S_{j-3}, whose store has read it (the MMA
        // thread waited for that before issuing step j's MMAs).
        write_img(img + ((j + 1) % kScanImgBufs) * kScanImg);
        fence_proxy_async_smem();
      }
      if (++stage == STAGES) { stage = 0; phase ^= 1; }
      if (!__all_sync(0xffffffffu, ok)) goto done;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(sready));
    }
    if (row && a.maps) {
      const size_t mo_end =
          ((size_t)(bh * a.nchunks + chunk_id) * D + i) * 2 * D + (ident ? 0 : D) + 16 * cb + h8 + 8;
      float4* mo = reinterpret_cast<float4*>(a.maps + mo_end - 8);
      if (in_region(mo_end * 4, a.maps_span, a.status)) {
#pragma unroll
        for (int q = 0; q < 2; ++q) mo[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
      }
    } else if (row && a.state_out && chunk_id == a.nchunks - 1) {
      float4* so = reinterpret_cast<float4*>(a.state_out + ((size_t)bh * D + i) * D + 16 * cb + h8);
#pragma unroll
      for (int q = 0; q < 2; ++q) so[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    }
  }
done:
  if (warp == kScanMmaWarp && lane == 0) {
    bulk_wait0();  // state block stores complete
    mma_commit(smem_u32(mma_done));
    wait_bounded(smem_u32(mma_done), 0, 500000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kScanMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 32);
  }
}

// =============================================================================
// readout: O_t = Q_t S_t / sqrt(D) per frame-head and 128-token tile.
//
// Persistent CTAs.  Whole frame-heads are dealt round-robin while every CTA gets
// one; the tiles of the frame-heads left over are then split into contiguous
// ranges as equal as whole tiles allow, one per CTA (so a call of few
// frame-heads still fills every SM).  Per frame-head of its work a CTA gathers
// the S_t image (bf16 hi + lo, the B operand: K-major, row n = value column, D
// rows) from the scan's column blocks (2 KB bulk copies) into one of two
// buffers; Q tiles of 128 tokens stream through a 2-deep TMA ring; per tile
// two MMA chains (hi, lo) accumulate O_tile (128 tokens x D) in one of four
// TMEM accumulators.  Each epilogue warp owns 32 token rows: it scales and
// rounds them to bf16 into its own slice of a staging tile and TMA-stores the
// slice, waiting only for its own previous store.
// =============================================================================
// A read-out CTA's work: units u = f * ntiles + tile, the k-th of count.
struct TileSched {
  long long per1;   // units in the round-robin phase (whole frame-heads)
  long long base;   // first unit of this CTA's tail range
  long long count;  // units in all
  int ntiles;
  __device__ TileSched(long long F, int nt) : ntiles(nt) {
    const long long G = gridDim.x, rounds = F / G, tail = (F - rounds * G) * nt;
    const long long r0 = tail * blockIdx.x / G, r1 = tail * (blockIdx.x + 1) / G;
    per1 = rounds * nt;
    base = rounds * G * nt + r0;
    count = per1 + (r1 - r0);
  }
  // frame-head and tile of unit 0
  __device__ void start(long long& f, int& tile) const {
    f = per1 > 0 ? (long long)blockIdx.x : base / ntiles;
    tile = per1 > 0 ? 0 : (int)(base % ntiles);
  }
  // from unit k to unit k + 1 (no division but at the phase change)
  __device__ void advance(long long k, long long& f, int& tile) const {
    if (k + 1 == per1) {
      f = base / ntiles;
      tile = (int)(base % ntiles);
    } else if (++tile == ntiles) {
      tile = 0;
      f += k < per1 ? (long long)gridDim.x : 1;
    }
  }
  // unit k starts / ends this CTA's share of its frame-head
  __device__ bool first(long long k, int tile) const { return k == 0 || k == per1 || tile == 0; }
  __device__ bool last(long long k, int tile) const { return k + 1 == count || tile == ntiles - 1; }
};

struct OutArgs {
  const uint8_t* s_img;
  int variant;  // kReluLinear: relu(Q) is applied to each Q tile in shared memory
  __nv_bfloat16* out;
  long long nitems;
  int S, D, NA;
  float scale;
  unsigned int* status;
  // 1: multiply by S_t^T instead (the backward's dQ = dO S_t^T / sqrt(D)): the
  // same image read as an MN-major B operand.
  int transpose_s;
  size_t s_span;  // extent (bytes) of the state image region (debug checks)
};

__global__ void __launch_bounds__(kOutThreads, 1)
    tc_readout_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapO, OutArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int NA = a.NA, D = a.D, S = a.S;
  const int img_bytes = 2 * NA * D * 128;                 // one S image (hi, lo)
  const int img_stride = (img_bytes + 1023) & ~1023;
  const int q_bytes = NA * kOutTok * 128;                 // one Q tile
  uint8_t* imgs = smem;
  uint8_t* qst = imgs + 2 * img_stride;
  uint8_t* stg = qst + kOutQStages * q_bytes;  // output staging: NA atoms of 128 rows x 128 B
  uint64_t* bars = reinterpret_cast<uint64_t*>(stg + NA * kOutTok * 128);
  uint64_t* afull = bars;
  uint64_t* aempty = bars + 2;
  uint64_t* qfull = bars + 4;
  uint64_t* qempty = qfull + kOutQStages;
  uint64_t* accfull = qempty + kOutQStages;
  uint64_t* accempty = accfull + kOutAcc;
  uint64_t* mma_done = accempty + kOutAcc;
  uint64_t* qready = mma_done + 1;  // kReluLinear: the tile's relu(Q) is in place
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(qready + kOutQStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const bool relu_q = a.variant == kReluLinear;

  const int warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&afull[b]), 1);
      mbar_init(smem_u32(&aempty[b]), 1);
    }
    for (int s = 0; s < kOutQStages; ++s) {
      mbar_init(smem_u32(&qfull[s]), 1);
      mbar_init(smem_u32(&qempty[s]), 1);
      mbar_init(smem_u32(&qready[s]), 4);
    }
    for (int b = 0; b < kOutAcc; ++b) {
      mbar_init(smem_u32(&accfull[b]), 1);
      mbar_init(smem_u32(&accempty[b]), 4);
    }
    mbar_init(smem_u32(mma_done), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ntiles = (S + kOutTok - 1) / kOutTok;
  const TileSched sc(a.nitems, ntiles);
  griddep_wait();  // no global memory is touched before the preceding kernel completes
  griddep_launch_dependents();

  if (warp == 4) {
    // ---------------- producer: S image per frame-head, Q tiles per tile
    if (lane == 0) {
      prefetch_tmap(&mapQ);
      Ring<2> ra;
      Ring<kOutQStages> rq;
      long long f;
      int tile;
      sc.start(f, tile);
      for (long long k = 0; k < sc.count; sc.advance(k++, f, tile)) {
        if (sc.first(k, tile)) {
          if (!wait_or_abort(smem_u32(&aempty[ra.stage]), ra.phase ^ 1, abort_flag, a.status)) break;
          const uint32_t afb = smem_u32(&afull[ra.stage]);
          mbar_arrive_expect_tx(afb, img_bytes);
          // block cb of the scan = [atom][hi 16 rows | lo 16 rows][128 B]
          const uint8_t* src = a.s_img + (size_t)f * img_bytes;
          if (in_region(((size_t)f + 1) * img_bytes, a.s_span, a.status))
            for (int cb = 0; cb < D / 16; ++cb)
              for (int at = 0; at < NA; ++at)
                for (int hl = 0; hl < 2; ++hl)
                  bulk_g2s(smem_u32(imgs + ra.stage * img_stride + (hl * NA + at) * D * 128 + cb * 16 * 128),
                           src + ((size_t)cb * NA + at) * (32 * 128) + hl * 16 * 128, 16 * 128, afb);
          ra.mark_issued();
          ra.advance();
        }
        if (!wait_or_abort(smem_u32(&qempty[rq.stage]), rq.phase ^ 1, abort_flag, a.status)) break;
        const uint32_t qfb = smem_u32(&qfull[rq.stage]);
        mbar_arrive_expect_tx(qfb, q_bytes);
        for (int at = 0; at < NA; ++at)
          tma_load_3d(smem_u32(qst + rq.stage * q_bytes + at * kOutTok * 128), &mapQ, qfb, 64 * at, tile * kOutTok,
                      (int)f);
        rq.mark_issued();
        rq.advance();
      }
      ra.drain(afull);
      rq.drain(qfull);
    }
  } else if (warp == 5) {
    // ---------------- MMA: O_tile (128 tokens x D) = Q_tile S_hi + Q_tile S_lo
    if (lane == 0) {
      const uint32_t id = idesc_bf16(128, D, 0, a.transpose_s ? 1 : 0);
      // Descriptors of buffer 0 / stage 0 / K-step 0; the rest only move the start
      // address (the low 14-bit field in 16-byte units; no carry below 2^18).
      // K-major image: rows = value columns, K-steps of 16 key dims inside an atom;
      // MN-major (transposed): K-steps of 16 rows (value columns), LBO = atom stride.
      const uint64_t dQ0 = smem_desc(smem_u32(qst), 16, 1024);
      const uint64_t dI0 = smem_desc(smem_u32(imgs), a.transpose_s ? D * 128 : 16, 1024);
      const uint64_t lo_off = (uint64_t)((NA * D * 128) >> 4);
      int ab = 0, qs = 0, cb = 0;
      uint32_t aph = 0, qph = 0, cph = 0;
      long long f;
      int tile;
      sc.start(f, tile);
      for (long long k = 0; k < sc.count; sc.advance(k++, f, tile)) {
        if (sc.first(k, tile))
          if (!wait_or_abort(smem_u32(&afull[ab]), aph, abort_flag, a.status)) goto done;
        const uint64_t io = (uint64_t)((ab * img_stride) >> 4);
        {
          if (!wait_or_abort(smem_u32(&accempty[cb]), cph ^ 1, abort_flag, a.status)) goto done;
          if (!wait_or_abort(smem_u32(relu_q ? &qready[qs] : &qfull[qs]), qph, abort_flag, a.status)) goto done;
          tc_fence_after();
          const uint64_t qo = (uint64_t)((qs * q_bytes) >> 4);
          const uint32_t acc = tmem + cb * 128;
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t ad = dQ0 + qo + (uint64_t)(((kk >> 2) * (kOutTok * 128) + (kk & 3) * 32) >> 4);
            const uint32_t so = a.transpose_s ? kk * 2048 : (kk >> 2) * (D * 128) + (kk & 3) * 32;
            const uint64_t bd = dI0 + io + (uint64_t)(so >> 4);
            mma_bf16(acc, ad, bd, id, kk > 0 ? 1u : 0u);
            mma_bf16(acc, ad, bd + lo_off, id, 1u);
          }
          mma_commit(smem_u32(&qempty[qs]));
          mma_commit(smem_u32(&accfull[cb]));
          if (++qs == kOutQStages) { qs = 0; qph ^= 1; }
          if (++cb == kOutAcc) { cb = 0; cph ^= 1; }
        }
        if (sc.last(k, tile)) {  // the frame-head's last tile in this CTA's work
          mma_commit(smem_u32(&aempty[ab]));
          if (++ab == 2) { ab = 0; aph ^= 1; }
        }
      }
    }
  } else if (warp >= 6) {
    // ---------------- query prep (kReluLinear only): relu(Q) in place, tile by tile
    if (relu_q) {
      const int pt = threadIdx.x - 192;  // 0 .. 127
      int qs = 0;
      uint32_t qph = 0;
      const __nv_bfloat162 zero = __floats2bfloat162_rn(0.f, 0.f);
      for (long long k = 0; k < sc.count; ++k) {
        {
          if (!__all_sync(0xffffffffu, wait_or_abort(smem_u32(&qfull[qs]), qph, abort_flag, a.status))) goto done;
          uint4* qt = reinterpret_cast<uint4*>(qst + qs * q_bytes);
          for (int idx = pt; idx < q_bytes / 16; idx += 128) {
            uint4 w = qt[idx];
            __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
            for (int e = 0; e < 4; ++e) h[e] = __hmax2(h[e], zero);
            qt[idx] = w;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&qready[qs]));
          if (++qs == kOutQStages) { qs = 0; qph ^= 1; }
        }
      }
    }
  } else {
    // ---------------- epilogue: warp w owns token rows 32w .. 32w + 31 of each tile
    const int row = warp * 32 + lane;
    int cb = 0;
    uint32_t cph = 0;
    long long f;
    int tile;
    sc.start(f, tile);
    for (long long k = 0; k < sc.count; sc.advance(k++, f, tile)) {
      {
        if (!__all_sync(0xffffffffu, wait_or_abort(smem_u32(&accfull[cb]), cph, abort_flag, a.status))) goto done;
        tc_fence_after();
        if (lane == 0) bulk_wait_read0();  // this warp's previous store has read its slice
        __syncwarp();
        const uint32_t acc = tmem + ((uint32_t)(warp * 32) << 16) + cb * 128;
        for (int c0 = 0; c0 < D; c0 += 32) {
          float v[32];
          tmem_ld16(acc + c0, *reinterpret_cast<float(*)[16]>(&v[0]));
          if (c0 + 16 < D) tmem_ld16(acc + c0 + 16, *reinterpret_cast<float(*)[16]>(&v[16]));
          tmem_ld_wait();
          uint8_t* reg = stg + (c0 >> 6) * (kOutTok * 128);
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            if (c0 + 8 * h < D) {
              uint4 o;
              o.x = pack_bf16(v[8 * h + 0] * a.scale, v[8 * h + 1] * a.scale);
              o.y = pack_bf16(v[8 * h + 2] * a.scale, v[8 * h + 3] * a.scale);
              o.z = pack_bf16(v[8 * h + 4] * a.scale, v[8 * h + 5] * a.scale);
              o.w = pack_bf16(v[8 * h + 6] * a.scale, v[8 * h + 7] * a.scale);
              *reinterpret_cast<uint4*>(reg + sw128_off(row, (c0 & 63) + 8 * h)) = o;
            }
          }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&accempty[cb]));
          for (int at = 0; at < NA; ++at)
            tma_store_3d(&mapO, smem_u32(stg + at * (kOutTok * 128) + warp * 32 * 128), 64 * at,
                         tile * kOutTok + warp * 32, (int)f);
          bulk_commit();
        }
        if (++cb == kOutAcc) { cb = 0; cph ^= 1; }
      }
    }
  }
done:
  if (warp < 4 && lane == 0) bulk_wait0();  // this warp's output stores are complete
  if (warp == 5 && lane == 0) {
    mma_commit(smem_u32(mma_done));
    wait_bounded(smem_u32(mma_done), 0, 500000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// =============================================================================
// Backward pass (gdn_frame_bwd, bf16 I/O).  The forward kernels above supply
// most of it: the gram (M_t, b_t) and scan (every S_t image) recompute the
// states; the gram's b-only form gives E_t = Q_t^T dO_t / sqrt(D); the scan's
// reverse form runs the state gradient U back through the adjoint map; the
// read-out's transposed form gives dQ = dO S_t^T / sqrt(D).  The kernel below
// does the rest.  With K~ = K / sqrt(D*S), P = K~ S_{t-1} and dR = K~ U_t, the
// gradients of a frame are
//   dV = diag(beta) dR,
//   dK~ = diag(beta) ((V - g P) U_t^T - g dR S_{t-1}^T),
//   dbeta_s = <dR_s, V_s - g P_s>,  dg = <U_t, S_{t-1}> - sum_s beta_s <dR_s, P_s>.
// With the symmetric D x D matrix W_t = S_{t-1} U_t^T + U_t S_{t-1}^T, formed once
// per frame-head,  P U_t^T + dR S_{t-1}^T = K~ W_t,  <dR_s, P_s> = k~_s W_t k~_s^T / 2
// and <U_t, S_{t-1}> = tr(W_t) / 2, so
//   dK~ = diag(beta) (V U_t^T - g K~ W_t),
//   dbeta_s = <k~_s, (V U_t^T)_s> - (g / 2) <k~_s, (K~ W_t)_s>,
//   dg = tr(W_t) / 2 - (1 / 2) sum_s beta_s <k~_s, (K~ W_t)_s>:
// three products per token tile, K U_t, V U_t^T and K W_t, whose A operands are
// the bf16 inputs themselves (exact) and whose B operands are bf16 hi + lo images,
// then element-wise work in fp32 registers.
// =============================================================================

// The initial state of every head as a scan block image (bf16 hi + lo), the
// backward's S_{-1}; zeros when `state` is null.  grid = (heads, D/16); thread =
// key dim (all 64 * NA positions written, those past D as zeros).
__global__ void __launch_bounds__(128) tc_state_image_kernel(const float* __restrict__ state,
                                                             uint8_t* __restrict__ img, int D, int NA) {
  const long long bh = blockIdx.x;
  const int cb = blockIdx.y, ncb = gridDim.y, i = threadIdx.x;
  if (i >= NA * 64) return;
  float x[16];
#pragma unroll
  for (int n = 0; n < 16; ++n) x[n] = (state && i < D) ? state[((size_t)bh * D + i) * D + 16 * cb + n] : 0.f;
  uint8_t* at = img + ((size_t)bh * ncb + cb) * NA * (32 * 128) + (i >> 6) * (32 * 128);
#pragma unroll
  for (int n = 0; n < 16; n += 2) {
    uint32_t hv, lv;
    split2(x[n], x[n + 1], hv, lv);
    *reinterpret_cast<uint16_t*>(at + sw128_off(n, i & 63)) = (uint16_t)(hv & 0xFFFF);
    *reinterpret_cast<uint16_t*>(at + sw128_off(n + 1, i & 63)) = (uint16_t)(hv >> 16);
    *reinterpret_cast<uint16_t*>(at + sw128_off(16 + n, i & 63)) = (uint16_t)(lv & 0xFFFF);
    *reinterpret_cast<uint16_t*>(at + sw128_off(17 + n, i & 63)) = (uint16_t)(lv >> 16);
  }
}

constexpr int kKvTok = 128;      // tokens per tile (MMA M)
constexpr int kKvThreads = 320;  // 8 element-wise warps, 1 MMA warp, 1 copy warp
// TMEM columns: X1 = K U_t, X2 = V U_t^T, X3 = K W_t (one tile each), W_t
constexpr uint32_t kTX1 = 0, kTX2 = 128, kTX3 = 256, kTW = 384;

struct KvArgs {
  const uint8_t* s_img;   // S_t images (F slots, the scan's block layout)
  const uint8_t* s0_img;  // S_{-1} images (one slot per head)
  const uint8_t* u_img;   // U_t images (F slots)
  const float* g;
  const float* beta;
  const __nv_bfloat16* k;  // K and V themselves (L2 prefetches of coming tiles)
  const __nv_bfloat16* v;
  int gate_logits;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* dbeta;
  float* dg_part;  // [F][ntiles]
  long long nitems;
  int T, S, D, NA;
  float ck;  // 1/sqrt(D*S)
  unsigned int* status;
  size_t s_span, s0_span, u_span;  // extents (bytes) of the image regions (debug checks)
  // dk and dv are 32-byte aligned: each thread writes its 16 columns of a row in
  // one 32-byte store (a row is 2 D bytes, a multiple of 32)
  int wide_stores;
};

// Persistent CTAs over frame-heads.  Per frame-head: the S_{t-1} and U_t images
// (bf16 hi + lo) are gathered; the MMA warp forms W_t in TMEM (six products per
// K-step: S_hi U_hi, S_hi U_lo, S_lo U_hi and the same with S and U swapped); the
// element-wise warps turn it into a bf16 hi + lo image in place of S_{t-1}'s
// (row i of W is row i of its K-major image, W being symmetric) and sum its
// trace.  Then per 128-token tile (K in a 2-deep ring, V single):
//   warp 8 (MMA)    : X1 = K U_t, then X3 = K W_t (K-major images) and
//                     X2 = V U_t^T (U_t read MN-major), into TMEM as two groups
//                     with their own full / empty barriers;
//   warps 0-7       : two per TMEM lane quadrant, alternate 16-column chunks:
//                     dV from X1 (the X2 / X3 products run meanwhile), then dK~
//                     from X2 and X3 (the next tile's X1 runs meanwhile), both
//                     straight from registers to global memory, and the partial
//                     dots of dbeta and dg (halves combined in shared memory,
//                     fixed order);
//   warp 9 (copies) : K and V tiles by TMA, the images by bulk copies.
__global__ void __launch_bounds__(kKvThreads, 1)
    tc_kv_grad_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV, KvArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int NA = a.NA, D = a.D, S = a.S, T = a.T, KS = D / 16;
  const int img_bytes = 2 * NA * D * 128;  // one image: hi, then lo (a multiple of 1024)
  const int lo = NA * D * 128;             // offset of the lo part
  const int tile_bytes = NA * kKvTok * 128;
  uint8_t* imgU = smem;
  uint8_t* imgW = imgU + img_bytes;  // S_{t-1}, then W_t
  uint8_t* tK = imgW + img_bytes;    // 2 slots
  uint8_t* tV = tK + 2 * tile_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(tV + tile_bytes);
  uint64_t* ifull = bars;        // images landed
  uint64_t* iempty = bars + 1;   // images free (the frame-head's last MMAs done)
  uint64_t* wacc = bars + 2;     // W_t in TMEM
  uint64_t* wimg = bars + 3;     // W_t image written (8 warps)
  uint64_t* kfull = bars + 4;    // [2]
  uint64_t* kempty = bars + 6;   // [2] (8 warps: K rows read after the tile's MMAs)
  uint64_t* vfull = bars + 8;
  uint64_t* vempty = bars + 9;   // the tile's MMAs done
  uint64_t* x1full = bars + 10;   // X1 in TMEM
  uint64_t* x1empty = bars + 11;  // X1 read (8 warps)
  uint64_t* mma_done = bars + 12;
  uint64_t* x23full = bars + 13;   // X2, X3 in TMEM (and every MMA of the tile done)
  uint64_t* x23empty = bars + 14;  // X2, X3 read (8 warps)
  float* red = reinterpret_cast<float*>(bars + 16);  // [2][8] per-warp dg partial sums, by tile parity
  float* dbh = red + 2 * 8;                          // [2][128] dbeta halves of warps 4-7, by tile parity
  float* trw = dbh + 2 * kKvTok;                     // [2][8] trace partials of W, by frame-head parity
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(trw + 2 * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  constexpr int wmma = 8, wcopy = 9;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(ifull), 1);
    mbar_init(smem_u32(iempty), 1);
    mbar_init(smem_u32(wacc), 1);
    mbar_init(smem_u32(wimg), 8);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&kfull[b]), 1);
      mbar_init(smem_u32(&kempty[b]), 8);
    }
    mbar_init(smem_u32(vfull), 1);
    mbar_init(smem_u32(vempty), 1);
    mbar_init(smem_u32(x1full), 1);
    mbar_init(smem_u32(x1empty), 8);
    mbar_init(smem_u32(x23full), 1);
    mbar_init(smem_u32(x23empty), 8);
    mbar_init(smem_u32(mma_done), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == wmma) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ntiles = (S + kKvTok - 1) / kKvTok;

  if (warp == wcopy) {
    // ---------------- copies in
    if (lane == 0) {
      prefetch_tmap(&mapK);
      prefetch_tmap(&mapV);
      Ring<1> ri, rv;
      Ring<2> rk;
      bool ok = true;
      for (long long f = blockIdx.x; ok && f < a.nitems; f += gridDim.x) {
        for (int tile = 0; ok && tile < ntiles; ++tile) {
          if (!wait_or_abort(smem_u32(&kempty[rk.stage]), rk.phase ^ 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          const uint32_t kb = smem_u32(&kfull[rk.stage]);
          mbar_arrive_expect_tx(kb, tile_bytes);
          for (int at = 0; at < NA; ++at)
            tma_load_3d(smem_u32(tK + rk.stage * tile_bytes + at * kKvTok * 128), &mapK, kb, 64 * at,
                        tile * kKvTok, (int)f);
          rk.mark_issued();
          rk.advance();
          {  // into L2: this tile's V rows and the next tile's K rows (contiguous in memory)
            const int rows = min(kKvTok, S - tile * kKvTok);
            prefetch_l2(a.v + ((size_t)f * S + (size_t)tile * kKvTok) * D, (uint32_t)rows * D * 2);
            const bool last = tile + 1 == ntiles;
            const long long fn = last ? f + gridDim.x : f;
            const int tn = last ? 0 : tile + 1;
            if (fn < a.nitems)
              prefetch_l2(a.k + ((size_t)fn * S + (size_t)tn * kKvTok) * D,
                          (uint32_t)min(kKvTok, S - tn * kKvTok) * D * 2);
          }
          if (tile == 0) {  // the frame-head's images, once the previous one's last MMAs are done
            if (!wait_or_abort(smem_u32(iempty), ri.phase ^ 1, abort_flag, a.status)) {
              ok = false;
              break;
            }
            const int t = (int)(f % T);
            const uint8_t* srcS =
                t > 0 ? a.s_img + (size_t)(f - 1) * img_bytes : a.s0_img + (size_t)(f / T) * img_bytes;
            const uint8_t* srcU = a.u_img + (size_t)f * img_bytes;
            const uint32_t ib = smem_u32(ifull);
            mbar_arrive_expect_tx(ib, 2 * img_bytes);
            const bool s_ok = t > 0 ? in_region((size_t)f * img_bytes, a.s_span, a.status)
                                    : in_region((size_t)(f / T + 1) * img_bytes, a.s0_span, a.status);
            const bool u_ok = in_region(((size_t)f + 1) * img_bytes, a.u_span, a.status);
            // block cb of the scan = [atom][hi 16 rows | lo 16 rows][128 B]
            for (int cb = 0; cb < D / 16; ++cb)
              for (int at = 0; at < NA; ++at)
                for (int hl = 0; hl < 2; ++hl) {
                  const size_t so = ((size_t)cb * NA + at) * (32 * 128) + hl * 16 * 128;
                  const uint32_t dof = hl * lo + at * D * 128 + cb * 16 * 128;
                  if (s_ok) bulk_g2s(smem_u32(imgW + dof), srcS + so, 16 * 128, ib);
                  if (u_ok) bulk_g2s(smem_u32(imgU + dof), srcU + so, 16 * 128, ib);
                }
            ri.mark_issued();
            ri.advance();
            const long long fn = f + gridDim.x;  // the next frame-head's images, into L2
            if (fn < a.nitems) {
              const int tn = (int)(fn % T);
              prefetch_l2(tn > 0 ? a.s_img + (size_t)(fn - 1) * img_bytes : a.s0_img + (size_t)(fn / T) * img_bytes,
                          (uint32_t)img_bytes);
              prefetch_l2(a.u_img + (size_t)fn * img_bytes, (uint32_t)img_bytes);
            }
          }
          if (!wait_or_abort(smem_u32(vempty), rv.phase ^ 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          const uint32_t vb = smem_u32(vfull);
          mbar_arrive_expect_tx(vb, tile_bytes);
          for (int at = 0; at < NA; ++at)
            tma_load_3d(smem_u32(tV + at * kKvTok * 128), &mapV, vb, 64 * at, tile * kKvTok, (int)f);
          rv.mark_issued();
          rv.advance();
        }
      }
      ri.drain(ifull);
      rk.drain(kfull);
      rv.drain(vfull);
    }
  } else if (warp == wmma) {
    // ---------------- MMAs
    if (lane == 0) {
      const uint32_t idK = idesc_bf16(128, D, 0, 0);  // A K-major (tile), B K-major (image, K = key dim)
      const uint32_t idT = idesc_bf16(128, D, 0, 1);  // A K-major (V tile), B MN-major (U image, K = value dim)
      const uint32_t idW = idesc_bf16(128, D, 1, 1);  // A and B MN-major (images, K = value dim)
      // Descriptors at offset 0 of each region; offsets only move the start address
      // (the low 14-bit field in 16-byte units; no carry below 2^18).
      const uint64_t uK = smem_desc(smem_u32(imgU), 16, 1024), wK = smem_desc(smem_u32(imgW), 16, 1024);
      const uint64_t uM = smem_desc(smem_u32(imgU), D * 128, 1024), wM = smem_desc(smem_u32(imgW), D * 128, 1024);
      const uint64_t tK0 = smem_desc(smem_u32(tK), 16, 1024), tV0 = smem_desc(smem_u32(tV), 16, 1024);
      const uint64_t lo16 = (uint64_t)(lo >> 4);
      int ks = 0;
      uint32_t kph = 0, vph = 0, x1ph = 0, x23ph = 0, iph = 0, wph = 0;
      for (long long f = blockIdx.x; f < a.nitems; f += gridDim.x) {
        if (!wait_or_abort(smem_u32(ifull), iph, abort_flag, a.status)) goto done;
        iph ^= 1;
        tc_fence_after();
        // W_t = S U^T + U S^T (K = value dim j; the images are [j][i], so both
        // operands are MN-major); the lo x lo terms are below fp32 rounding
        for (int kk = 0; kk < KS; ++kk) {
          const uint64_t mo = (uint64_t)((kk * 2048) >> 4);
          const uint64_t sh = wM + mo, sl = wM + lo16 + mo;
          const uint64_t uh = uM + mo, ul = uM + lo16 + mo;
          mma_bf16(tmem + kTW, sh, uh, idW, kk > 0 ? 1u : 0u);
          mma_bf16(tmem + kTW, sh, ul, idW, 1u);
          mma_bf16(tmem + kTW, sl, uh, idW, 1u);
          mma_bf16(tmem + kTW, uh, sh, idW, 1u);
          mma_bf16(tmem + kTW, uh, sl, idW, 1u);
          mma_bf16(tmem + kTW, ul, sh, idW, 1u);
        }
        mma_commit(smem_u32(wacc));
        // the W image replaces S_{t-1}'s
        if (!wait_or_abort(smem_u32(wimg), wph, abort_flag, a.status)) goto done;
        wph ^= 1;
        // Two accumulator groups per tile, so the element-wise warps' dV pass (X1)
        // runs beside the X2 / X3 products and the next tile's X1 beside their
        // dK pass (X2, X3).
        for (int tile = 0; tile < ntiles; ++tile) {
          if (!wait_or_abort(smem_u32(&kfull[ks]), kph, abort_flag, a.status)) goto done;
          if (!wait_or_abort(smem_u32(x1empty), x1ph ^ 1, abort_flag, a.status)) goto done;
          tc_fence_after();
          const uint64_t kso = (uint64_t)((ks * tile_bytes) >> 4);
          for (int kk = 0; kk < KS; ++kk) {  // K-dim = key dim i
            const uint64_t ko = (uint64_t)((((kk >> 2) * (kKvTok * 128) + (kk & 3) * 32)) >> 4);
            const uint64_t so = (uint64_t)((((kk >> 2) * (D * 128) + (kk & 3) * 32)) >> 4);
            const uint64_t ad = tK0 + kso + ko;
            mma_bf16(tmem + kTX1, ad, uK + so, idK, kk > 0 ? 1u : 0u);
            mma_bf16(tmem + kTX1, ad, uK + lo16 + so, idK, 1u);
          }
          mma_commit(smem_u32(x1full));
          x1ph ^= 1;
          if (!wait_or_abort(smem_u32(vfull), vph, abort_flag, a.status)) goto done;
          if (!wait_or_abort(smem_u32(x23empty), x23ph ^ 1, abort_flag, a.status)) goto done;
          tc_fence_after();
          for (int kk = 0; kk < KS; ++kk) {  // K-dim = key dim i
            const uint64_t ko = (uint64_t)((((kk >> 2) * (kKvTok * 128) + (kk & 3) * 32)) >> 4);
            const uint64_t so = (uint64_t)((((kk >> 2) * (D * 128) + (kk & 3) * 32)) >> 4);
            const uint64_t ad = tK0 + kso + ko;
            mma_bf16(tmem + kTX3, ad, wK + so, idK, kk > 0 ? 1u : 0u);
            mma_bf16(tmem + kTX3, ad, wK + lo16 + so, idK, 1u);
          }
          for (int kk = 0; kk < KS; ++kk) {  // K-dim = value dim j
            const uint64_t ko = (uint64_t)((((kk >> 2) * (kKvTok * 128) + (kk & 3) * 32)) >> 4);
            const uint64_t mo = (uint64_t)((kk * 2048) >> 4);
            const uint64_t ad = tV0 + ko;
            mma_bf16(tmem + kTX2, ad, uM + mo, idT, kk > 0 ? 1u : 0u);
            mma_bf16(tmem + kTX2, ad, uM + lo16 + mo, idT, 1u);
          }
          mma_commit(smem_u32(x23full));
          mma_commit(smem_u32(vempty));
          if (tile == ntiles - 1) mma_commit(smem_u32(iempty));
          x23ph ^= 1;
          vph ^= 1;
          if (++ks == 2) { ks = 0; kph ^= 1; }
        }
      }
    }
  } else if (warp < 8) {
    // ---------------- element-wise: warp w owns TMEM lane quadrant w % 4 (token rows
    // 32 (w % 4) .. + 31, or key rows of W) and the 16-column chunks c with c % 2 == w / 4
    const int quad = warp & 3, half = warp >> 2;
    const int row = quad * 32 + lane;
    const int et = threadIdx.x;  // 0 .. 255
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const float ck = a.ck;
    long long n = 0;  // tiles of this CTA so far
    int ks = 0;
    uint32_t kph = 0, x1ph = 0, x23ph = 0, wph = 0;
    int fpar = 0;  // frame-head parity (trace buffers)
    for (long long f = blockIdx.x; f < a.nitems; f += gridDim.x, fpar ^= 1) {
      const float gt = decay_of(__ldg(a.g + f), a.gate_logits);
      // ---- W_t out of TMEM into its hi + lo image (row i of W = image row i)
      if (!__all_sync(0xffffffffu, wait_or_abort(smem_u32(wacc), wph, abort_flag, a.status))) goto done;
      wph ^= 1;
      tc_fence_after();
      float tr = 0.f;
      for (int c0 = 16 * half; c0 < D; c0 += 32) {
        float w[16];
        tmem_ld16(tmem + lane_base + kTW + c0, w);
        tmem_ld_wait();
        if (row < D) {
          uint8_t* at = imgW + (c0 >> 6) * (D * 128);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t hv[4], lv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) split2(w[8 * h + 2 * e], w[8 * h + 2 * e + 1], hv[e], lv[e]);
            const uint32_t off = sw128_off(row, (c0 & 63) + 8 * h);
            *reinterpret_cast<uint4*>(at + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            *reinterpret_cast<uint4*>(at + lo + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
          }
          if (row >= c0 && row < c0 + 16) {
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (row == c0 + e) tr += w[e];
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tr += __shfl_xor_sync(0xffffffffu, tr, o);
      if (lane == 0) trw[8 * fpar + warp] = tr;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(wimg));
      // ---- the frame-head's tiles
      for (int tile = 0; tile < ntiles; ++tile, ++n) {
        const int par = (int)(n & 1);
        const int s = tile * kKvTok + row;
        const bool valid = s < S;
        const float bt = valid ? beta_of(__ldg(a.beta + f * S + s), a.gate_logits) : 0.f;
        const float btck = bt * ck, gck = gt * ck;
        __nv_bfloat16* dvrow = a.dv + (f * S + s) * D;
        __nv_bfloat16* dkrow = a.dk + (f * S + s) * D;
        // dV = beta ck X1 (the X1 group)
        if (!__all_sync(0xffffffffu, wait_or_abort(smem_u32(x1full), x1ph, abort_flag, a.status))) goto done;
        x1ph ^= 1;
        tc_fence_after();
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int c0 = 16 * half + 32 * m;
          if (c0 >= D) break;
          float x1b[16];
          tmem_ld16(tmem + lane_base + kTX1 + c0, x1b);
          tmem_ld_wait();
          uint32_t ov[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) ov[e] = pack_bf16(btck * x1b[2 * e], btck * x1b[2 * e + 1]);
          if (valid && a.wide_stores) {
            st_global_v8(dvrow + c0, ov);
          } else if (valid) {
            reinterpret_cast<uint4*>(dvrow + c0)[0] = make_uint4(ov[0], ov[1], ov[2], ov[3]);
            reinterpret_cast<uint4*>(dvrow + c0)[1] = make_uint4(ov[4], ov[5], ov[6], ov[7]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(x1empty));
        }
        // dK~, the dbeta and dg dots (the X2, X3 group)
        if (!__all_sync(0xffffffffu, wait_or_abort(smem_u32(x23full), x23ph, abort_flag, a.status))) goto done;
        x23ph ^= 1;
        tc_fence_after();
        const uint8_t* kt = tK + ks * (NA * kKvTok * 128);
        float dot2 = 0.f, dot3 = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int c0 = 16 * half + 32 * m;
          if (c0 >= D) break;
          float x2[16], x3[16];
          tmem_ld16(tmem + lane_base + kTX2 + c0, x2);
          tmem_ld16(tmem + lane_base + kTX3 + c0, x3);
          tmem_ld_wait();
          uint32_t ok[8];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 kv = *reinterpret_cast<const uint4*>(kt + (c0 >> 6) * (kKvTok * 128) +
                                                             sw128_off(row, (c0 & 63) + 8 * h));
            const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 k2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kw[e]));
              const int j = 8 * h + 2 * e;
              dot2 = fmaf(k2.x, x2[j], fmaf(k2.y, x2[j + 1], dot2));
              dot3 = fmaf(k2.x, x3[j], fmaf(k2.y, x3[j + 1], dot3));
              ok[4 * h + e] = pack_bf16(btck * fmaf(-gck, x3[j], x2[j]), btck * fmaf(-gck, x3[j + 1], x2[j + 1]));
            }
          }
          if (valid && a.wide_stores) {
            st_global_v8(dkrow + c0, ok);
          } else if (valid) {
            reinterpret_cast<uint4*>(dkrow + c0)[0] = make_uint4(ok[0], ok[1], ok[2], ok[3]);
            reinterpret_cast<uint4*>(dkrow + c0)[1] = make_uint4(ok[4], ok[5], ok[6], ok[7]);
          }
        }
        // this tile's X2, X3 and K rows are read
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(x23empty));
          mbar_arrive(smem_u32(&kempty[ks]));
        }
        if (++ks == 2) { ks = 0; kph ^= 1; }
        // dbeta_s = ck <k_s, X2_s> - (g / 2) ck^2 <k_s, X3_s>, this half's columns
        const float db = ck * dot2 - 0.5f * gt * ck * ck * dot3;
        // dg partial: -(1/2) ck^2 sum_s beta_s <k_s, X3_s> (rows past S have beta 0)
        float part = -0.5f * ck * ck * bt * dot3;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) red[8 * par + warp] = part;
        if (half == 1) dbh[kKvTok * par + row] = db;
        named_barrier(1, 256);  // partial sums and dbeta halves in place
        if (half == 0 && valid) {
          const float dbt = db + dbh[kKvTok * par + row];
          a.dbeta[f * S + s] = a.gate_logits ? dbt * bt * (1.f - bt) : dbt;
        }
        if (et == 0) {
          float tot = 0.f;
          for (int w8 = 0; w8 < 8; ++w8) tot += red[8 * par + w8];
          if (tile == 0) {  // <U_t, S_{t-1}> = tr(W_t) / 2
            float t2 = 0.f;
            for (int w8 = 0; w8 < 8; ++w8) t2 += trw[8 * fpar + w8];
            tot += 0.5f * t2;
          }
          a.dg_part[f * ntiles + tile] = tot;
        }
      }
    }
  }
done:
  if (warp == wmma && lane == 0) {
    mma_commit(smem_u32(mma_done));
    wait_bounded(smem_u32(mma_done), 0, 500000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == wmma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Launches `kernel` with programmatic stream serialization: it may begin (its
// prologue: barriers, TMEM, descriptors) while the preceding kernel in the stream
// finishes; each such kernel waits (griddep_wait) before its first global access.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, int smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

constexpr int kBarBytes = 256;
constexpr int kKvBarBytes = 1792;  // barriers, partial sums, dbeta halves and trace partials of tc_kv_grad_kernel

// Every kernel here asks for more than half of the SM's shared memory, so two of
// them never share an SM (the gram and read-out kernels allocate all of TMEM).
int gram_smem(int NA, int D) {
  return kGramRaw * kRawStage + kGramConv * kConvStage + NA * D * 128 + kBarBytes + 1024;
}
int kv_smem(int NA, int D) { return 4 * NA * D * 128 + 3 * NA * kKvTok * 128 + kKvBarBytes + 1024; }
static_assert(4 * 2 * 128 * 128 + 3 * 2 * kKvTok * 128 + 1792 + 1024 <= 232448, "kv_grad shared memory at D = 128");
template <int STAGES>
int scan_smem() { return STAGES * (kScanMStage + kScanBStage) + kScanImgBufs * kScanImg + kBarBytes + 1024; }

constexpr int kTcChunk = kTcChunkFrames;

// A one-pass scan's arguments (not chunked).
ScanArgs one_pass(const uint8_t* m_img, const float* b_blk, const float* g, int gate_logits, int variant,
                  const float* state_in, uint8_t* s_img, float* state_out, int T, int D, unsigned int* status,
                  int reverse) {
  ScanArgs sa{m_img, b_blk, g, gate_logits, variant, state_in, s_img, state_out, T, D, num_atoms(D), status, reverse};
  sa.chunk = T;
  sa.nchunks = 1;
  sa.starts = nullptr;
  sa.maps = nullptr;
  sa.m_span = sa.b_span = sa.s_span = sa.maps_span = sa.starts_span = 0;
  return sa;
}

template <int STAGES>
int launch_scan(const ScanArgs& sa, long long ctas, cudaStream_t st, const char* name) {
  const int smem = scan_smem<STAGES>();
  if (cudaFuncSetAttribute(tc_scan_kernel<STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return kCuda;
  ProfScope ps(st, name);
  return launch_pdl(tc_scan_kernel<STAGES>, (unsigned)ctas, kScanThreads, smem, st, sa) == cudaSuccess ? kOk : kCuda;
}
int out_smem(int NA, int D) {
  return 2 * ((2 * NA * D * 128 + 1023) & ~1023) + (kOutQStages + 1) * NA * kOutTok * 128 + kBarBytes + 1024;
}

}  // namespace

// Sequential and split forms: the gram, the one-pass scan and the read-out,
// through a workspace.  Prefix form: the gram, the chunked scan's summaries, the
// fold over chunk boundaries, the chunked replay and the read-out; its workspace
// is the split form's plus the chunk maps and starts.
size_t tc_workspace_bytes(const Problem& p, int mode) { return tc_layout(p, mode).total; }

namespace {

// The gram over every frame-head of the call on persistent CTAs: the M_t images
// and b_t blocks (regions of m_span and b_span bytes).
int launch_gram(const Problem& p, uint8_t* m_img, float* b_mat, size_t m_span, size_t b_span, cudaStream_t st) {
  const int NA = num_atoms(p.D);
  const long long F = p.BHT();
  CUtensorMap mapK, mapV;
  if (!make_map(&mapK, p.k, p.D, p.S, F, kGramTok) || !make_map(&mapV, p.v, p.D, p.S, F, kGramTok)) return kCuda;
  const int smem = gram_smem(NA, p.D);
  if (cudaFuncSetAttribute(tc_gram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return kCuda;
  GramArgs ga{p.beta, p.gate_logits, p.variant, m_img, b_mat, F, p.S, p.D, NA, p.key_scale * p.key_scale,
              p.key_scale, p.status, 0, m_span, b_span};
  const int nsm = num_sms();
  const unsigned grid = (unsigned)(F < nsm ? F : nsm);
  ProfScope ps(st, "tc_gram");
  return launch_pdl(tc_gram_kernel, grid, kGramThreads, smem, st, mapK, mapV, ga) == cudaSuccess ? kOk : kCuda;
}

// The read-out over every frame-head of the call on persistent CTAs.
int launch_readout(const Problem& p, const CUtensorMap& mapQ, const CUtensorMap& mapO, const uint8_t* s_img,
                   size_t s_span, cudaStream_t st) {
  const long long F = p.BHT();
  const int nsm = num_sms();
  const int NA = num_atoms(p.D);
  const int smem = out_smem(NA, p.D);
  if (cudaFuncSetAttribute(tc_readout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return kCuda;
  const size_t shrink = debug_shrink();
  OutArgs oa{s_img, p.variant, static_cast<__nv_bfloat16*>(p.out), F, p.S, p.D, NA, p.out_scale, p.status, 0,
             s_span > shrink ? s_span - shrink : 1};
  const long long units = F * ((p.S + kOutTok - 1) / kOutTok);  // (frame-head, tile) pairs
  const unsigned grid = (unsigned)(units < nsm ? units : nsm);
  ProfScope ps(st, "tc_readout");
  return launch_pdl(tc_readout_kernel, grid, kOutThreads, smem, st, mapQ, mapO, oa) == cudaSuccess ? kOk : kCuda;
}

// The chunked scan's summary form: [A_c | b_c] of every (head, chunk) into `maps`.
int launch_chunk_summaries(const Problem& p, const TcLayout& L, const uint8_t* m_img, const float* b_mat,
                           float* maps, int nch, cudaStream_t st) {
  ScanArgs sa = one_pass(m_img, b_mat, p.g, p.gate_logits, p.variant, nullptr, nullptr, nullptr, p.T, p.D,
                         p.status, 0);
  sa.chunk = kTcChunk;
  sa.nchunks = nch;
  sa.maps = maps;
  sa.m_span = L.b_off - L.m_off;
  sa.b_span = L.s_off - L.b_off;
  sa.maps_span = L.starts_off - L.maps_off;
  return launch_scan<2>(sa, p.BH() * nch * 2 * (p.D / 16), st, "tc_chunk_summary");
}

}  // namespace

int tc_chunk_maps(const Problem& p, void* ws, float** maps, int* nchunks, cudaStream_t st) {
  const TcLayout L = tc_layout(p, GDN_MODE_PREFIX);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const int nch = (p.T + kTcChunk - 1) / kTcChunk;
  float* mp = reinterpret_cast<float*>(w + L.maps_off);
  int rc = launch_gram(p, w + L.m_off, reinterpret_cast<float*>(w + L.b_off), L.b_off - L.m_off, L.s_off - L.b_off,
                       st);
  if (rc != kOk) return rc;
  rc = launch_chunk_summaries(p, L, w + L.m_off, reinterpret_cast<float*>(w + L.b_off), mp, nch, st);
  if (rc != kOk) return rc;
  *maps = mp;
  *nchunks = nch;
  return kOk;
}

int tc_forward(const Problem& p, void* ws, cudaStream_t st) {
  const TcLayout L = tc_layout(p, p.mode);
  const int NA = num_atoms(p.D);
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint8_t* m_img = w + L.m_off;
  float* b_mat = reinterpret_cast<float*>(w + L.b_off);
  uint8_t* s_img = w + L.s_off;
  const long long F = p.BHT();

  CUtensorMap mapQ, mapO;
  if (!make_map(&mapQ, p.q, p.D, p.S, F, kOutTok) || !make_map(&mapO, p.out, p.D, p.S, F, 32)) return kCuda;

  const size_t m_span = L.b_off - L.m_off, b_span = L.s_off - L.b_off;
  const size_t s_span = (p.mode == GDN_MODE_PREFIX ? L.maps_off : L.total) - L.s_off;
  int rc = launch_gram(p, m_img, b_mat, m_span, b_span, st);
  if (rc != kOk) return rc;
  if (p.mode == GDN_MODE_PREFIX) {
    // chunk summaries [A_c | b_c] -> the fold over chunk boundaries (float32) ->
    // every chunk replayed from its true initial state
    const int nch = (p.T + kTcChunk - 1) / kTcChunk;
    float* maps = reinterpret_cast<float*>(w + L.maps_off);
    float* starts = reinterpret_cast<float*>(w + L.starts_off);
    rc = launch_chunk_summaries(p, L, m_img, b_mat, maps, nch, st);
    if (rc != kOk) return rc;
    const size_t maps_span = L.starts_off - L.maps_off, starts_span = L.total - L.starts_off;
    rc = launch_chunk_fold(maps, maps + p.D, 2LL * p.D * p.D, 2 * p.D, nch, p.state_in, starts, nullptr, nullptr,
                           nullptr, p.BH(), p.D, st, maps_span, maps_span - p.D * 4, starts_span);
    if (rc != kOk) return rc;
    ScanArgs sa = one_pass(m_img, b_mat, p.g, p.gate_logits, p.variant, nullptr, s_img, p.state_out, p.T, p.D,
                           p.status, 0);
    sa.chunk = kTcChunk;
    sa.nchunks = nch;
    sa.starts = starts;
    sa.m_span = m_span;
    sa.b_span = b_span;
    sa.s_span = s_span;
    sa.starts_span = starts_span;
    rc = launch_scan<2>(sa, p.BH() * nch * (p.D / 16), st, "tc_chunk_replay");
    if (rc != kOk) return rc;
  } else {
    ScanArgs sa = one_pass(m_img, b_mat, p.g, p.gate_logits, p.variant, p.state_in, s_img, p.state_out, p.T, p.D,
                           p.status, 0);
    sa.m_span = m_span;
    sa.b_span = b_span;
    sa.s_span = s_span;
    rc = launch_scan<4>(sa, p.BH() * (p.D / 16), st, "tc_scan");
    if (rc != kOk) return rc;
  }
  return launch_readout(p, mapQ, mapO, s_img, s_span, st);
}


// ---------------------------------------------------------------- backward pass
namespace {

struct TcBwdLayout {
  size_t m_off, e_off, s_off, u_off, s0_off, dg_off, total;
  size_t img_bytes;  // one S / U image slot
  int ntiles;
};

TcBwdLayout tc_bwd_layout(const Problem& p) {
  TcBwdLayout L{};
  const int NA = num_atoms(p.D);
  const size_t F = (size_t)p.BHT();
  L.img_bytes = (size_t)2 * NA * p.D * 128;
  L.ntiles = (p.S + kKvTok - 1) / kKvTok;
  L.m_off = 0;
  L.e_off = align_up(L.m_off + F * NA * p.D * 128, 1024);
  L.s_off = align_up(L.e_off + F * p.D * p.D * 4, 1024);
  L.u_off = align_up(L.s_off + F * L.img_bytes, 1024);
  L.s0_off = align_up(L.u_off + F * L.img_bytes, 1024);
  L.dg_off = align_up(L.s0_off + (size_t)p.BH() * L.img_bytes, 1024);
  L.total = align_up(L.dg_off + F * L.ntiles * 4, 1024);
  return L;
}

}  // namespace

size_t tc_bwd_workspace_bytes(const Problem& p) { return tc_bwd_layout(p).total; }

// The forward split form's scratch (tc_layout) is the backward layout's first
// three regions, so a forward call's states can be reused in place.
bool tc_bwd_layout_extends_forward(const Problem& p) {
  const TcLayout f = tc_layout(p);
  const TcBwdLayout b = tc_bwd_layout(p);
  return f.m_off == b.m_off && f.b_off == b.e_off && f.s_off == b.s_off && f.total <= b.total;
}

int tc_backward(const Problem& p, const BwdGrads& gr, void* ws, cudaStream_t st, bool states_ready) {
  const TcBwdLayout L = tc_bwd_layout(p);
  if (states_ready && !tc_bwd_layout_extends_forward(p)) return kInvalidArg;
  const int NA = num_atoms(p.D), D = p.D;
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint8_t* m_img = w + L.m_off;
  float* e_blk = reinterpret_cast<float*>(w + L.e_off);
  uint8_t* s_img = w + L.s_off;
  uint8_t* u_img = w + L.u_off;
  uint8_t* s0_img = w + L.s0_off;
  float* dg_part = reinterpret_cast<float*>(w + L.dg_off);
  const long long F = p.BHT();
  const int nsm = num_sms();
  const unsigned pgrid = (unsigned)(F < nsm ? F : nsm);

  CUtensorMap mapK, mapV, mapQ, mapDO, mapDO128, mapDQ;
  if (!make_map(&mapK, p.k, D, p.S, F, kGramTok) || !make_map(&mapV, p.v, D, p.S, F, kGramTok) ||
      !make_map(&mapQ, p.q, D, p.S, F, kGramTok) || !make_map(&mapDO, gr.dout, D, p.S, F, kGramTok) ||
      !make_map(&mapDO128, gr.dout, D, p.S, F, kOutTok) || !make_map(&mapDQ, gr.dq, D, p.S, F, 32))
    return kCuda;
  CUtensorMap mapK128, mapV128;
  if (!make_map(&mapK128, p.k, D, p.S, F, kKvTok) || !make_map(&mapV128, p.v, D, p.S, F, kKvTok)) return kCuda;

  const int gsmem = gram_smem(NA, D);
  if (cudaFuncSetAttribute(tc_gram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, gsmem) != cudaSuccess)
    return kCuda;
  const long long sgrid = p.BH() * (D / 16);

  // forward states: M_t (image), b_t (into the E blocks), S_t (images), unless a
  // forward call left them in the workspace (tc_layout's regions are this layout's first three)
  if (!states_ready) {
    {
      GramArgs ga{p.beta, p.gate_logits, kGdn, m_img, e_blk, F, p.S, D, NA, p.key_scale * p.key_scale, p.key_scale,
                  p.status, 0, L.e_off - L.m_off, L.s_off - L.e_off};
      ProfScope ps(st, "tc_gram");
      tc_gram_kernel<<<pgrid, kGramThreads, gsmem, st>>>(mapK, mapV, ga);
    }
    if (cudaGetLastError() != cudaSuccess) return kCuda;
    ScanArgs sa = one_pass(m_img, e_blk, p.g, p.gate_logits, kGdn, p.state_in, s_img, nullptr, p.T, D, p.status, 0);
    sa.m_span = L.e_off - L.m_off;
    sa.b_span = L.s_off - L.e_off;
    sa.s_span = L.u_off - L.s_off;
    const int rc = launch_scan<4>(sa, sgrid, st, "tc_scan");
    if (rc != kOk) return rc;
  }
  // E_t = Q_t^T dO_t / sqrt(D) (overwrites b_t, which the scan has consumed)
  {
    GramArgs ga{nullptr, 0, kGdn, nullptr, e_blk, F, p.S, D, NA, 0.f, p.out_scale, p.status, 1, 0, L.s_off - L.e_off};
    ProfScope ps(st, "tc_bwd_qdo");
    tc_gram_kernel<<<pgrid, kGramThreads, gsmem, st>>>(mapQ, mapDO, ga);
  }
  if (cudaGetLastError() != cudaSuccess) return kCuda;
  // U_t for every frame and dS_0, by the reverse scan
  {
    ScanArgs sa = one_pass(m_img, e_blk, p.g, p.gate_logits, kGdn, gr.dstate_out, u_img, gr.dstate_in, p.T, D,
                           p.status, 1);
    sa.m_span = L.e_off - L.m_off;
    sa.b_span = L.s_off - L.e_off;
    sa.s_span = L.s0_off - L.u_off;
    const int rc = launch_scan<4>(sa, sgrid, st, "tc_bwd_rscan");
    if (rc != kOk) return rc;
  }
  {
    ProfScope ps(st, "tc_bwd_s0_image");
    tc_state_image_kernel<<<dim3((unsigned)p.BH(), D / 16), 128, 0, st>>>(p.state_in, s0_img, D, NA);
  }
  if (cudaGetLastError() != cudaSuccess) return kCuda;
  {
    const int smem = kv_smem(NA, D);
    if (cudaFuncSetAttribute(tc_kv_grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return kCuda;
    KvArgs ka{s_img, s0_img, u_img, p.g, p.beta, static_cast<const __nv_bfloat16*>(p.k),
              static_cast<const __nv_bfloat16*>(p.v), p.gate_logits,
              static_cast<__nv_bfloat16*>(gr.dk),
              static_cast<__nv_bfloat16*>(gr.dv), gr.dbeta, dg_part, F, p.T, p.S, D, NA, p.key_scale, p.status,
              L.u_off - L.s_off, L.dg_off - L.s0_off, L.s0_off - L.u_off,
              ((reinterpret_cast<uintptr_t>(gr.dk) | reinterpret_cast<uintptr_t>(gr.dv)) & 31) == 0 ? 1 : 0};
    ProfScope ps(st, "tc_bwd_kv_grad");
    tc_kv_grad_kernel<<<pgrid, kKvThreads, smem, st>>>(mapK128, mapV128, ka);
  }
  if (cudaGetLastError() != cudaSuccess) return kCuda;
  // dQ = dO S_t^T / sqrt(D)
  {
    const int smem = out_smem(NA, D);
    if (cudaFuncSetAttribute(tc_readout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return kCuda;
    OutArgs oa{s_img, kGdn, static_cast<__nv_bfloat16*>(gr.dq), F, p.S, D, NA, p.out_scale, p.status, 1,
               L.u_off - L.s_off};
    ProfScope ps(st, "tc_bwd_q_grad");
    tc_readout_kernel<<<pgrid, kOutThreads, smem, st>>>(mapDO128, mapDQ, oa);
  }
  if (cudaGetLastError() != cudaSuccess) return kCuda;
  return launch_dg_sum(dg_part, p.g, gr.dg, F, L.ntiles, p.gate_logits, st);
}

}  // namespace gdn
