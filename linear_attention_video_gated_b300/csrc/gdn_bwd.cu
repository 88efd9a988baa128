// Backward pass of the frame-wise GDN scan (gdn_frame_bwd): the gradients of
// every input of the forward scan.  This file holds the C ABI, the float32 I/O
// path (CUDA cores, float32 arithmetic) and the dg reduction both paths share;
// bf16 I/O runs on the tensor cores (tc_backward in gdn_tc.cu).
//
// The pages train the model with this layer but give no backward pass; it is
// the forward definition differentiated.  With U_t the gradient with respect to
// the state after frame t, E_t = Q_t^T dO_t / sqrt(D) the read-out's share and
// M_t = K~^T diag(beta) K~ (the forward's transition term):
//
//   U_{T-1} = dS_T + E_{T-1},   U_{t-1} = E_{t-1} + g_t (U_t - M_t^T U_t),
//   dS_0 = g_0 (U_0 - M_0^T U_0)
//
// -- the adjoint of the forward's affine map S_t = g_t (S_{t-1} - M_t S_{t-1}) + b_t,
// run from the last frame to the first.  Columns of U evolve independently, as
// the state's do in the forward.  Per frame, with P = K~ S_{t-1} and dR = K~ U_t:
//
//   dV = diag(beta) dR,   dbeta_s = <dR_s, V_s - g P_s>,   dP = -g diag(beta) dR,
//   dK = (R U_t^T + dP S_{t-1}^T) / sqrt(D*S),   R = diag(beta)(V - g P),
//   dQ = dO S_t^T / sqrt(D),   dg = <U_t, S_{t-1}> - sum_s beta_s <dR_s, P_s>.
//
// Kernels, in launch order:
//   forward states : M_t, b_t and every S_t (the float32 forward's gram + scan);
//   qdo            : E_t for every frame-head in parallel (overwrites b_t);
//   rscan          : the reverse scan of U, one CTA per (head, 16 state columns);
//   kv_grad        : dK, dV, dbeta and the partial dg sums, per (frame-head,
//                    32-token tile), every frame in parallel;
//   q_grad         : dQ, per (frame-head, 64-token tile);
//   dg_sum         : dg per frame-head from the partial sums.
#include <cmath>
#include <cstdint>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kTok = 32;        // tokens staged per iteration of the Q^T dO product
constexpr int kRows = 32;       // tokens per kv_grad CTA
constexpr int kQRows = 64;      // tokens per q_grad CTA
constexpr int kColBlock = 16;   // columns of U per rscan CTA
constexpr int kScanThreads = 128;  // rscan: one 4 x 4 tile of U per thread (D/4 x 4 tiles)

// E_t = co Q_t^T dO_t.  One CTA per frame-head; each thread owns up to four
// 4 x 4 tiles of the D x D result.
template <typename TIn>
__global__ void __launch_bounds__(kThreads) qdo_kernel(const TIn* __restrict__ q, const TIn* __restrict__ dout,
                                                       float* __restrict__ Ews, int S, int D, float co) {
  extern __shared__ float smem[];
  float* sQ = smem;             // [kTok][D]
  float* sO = smem + kTok * D;  // [kTok][D]
  const long long f = blockIdx.x;
  const TIn* qf = q + f * S * D;
  const TIn* of = dout + f * S * D;
  const int nt4 = D / 4;
  const int ntiles = nt4 * nt4;
  float acc[4][16];
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[u][e] = 0.f;
  for (int s0 = 0; s0 < S; s0 += kTok) {
    const int n = min(kTok, S - s0);
    for (int idx = threadIdx.x; idx < kTok * D; idx += blockDim.x) {
      const int s = idx / D;
      const long long o = (long long)(s0 + s) * D + (idx % D);
      sQ[idx] = s < n ? to_f32(qf[o]) : 0.f;
      sO[idx] = s < n ? to_f32(of[o]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int tile = threadIdx.x + u * kThreads;
      if (tile < ntiles) {
        const int i0 = (tile / nt4) * 4, j0 = (tile % nt4) * 4;
        for (int s = 0; s < n; ++s) {
          const float4 a = *reinterpret_cast<const float4*>(sQ + s * D + i0);
          const float4 x = *reinterpret_cast<const float4*>(sO + s * D + j0);
          const float av[4] = {a.x, a.y, a.z, a.w};
          const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[u][r * 4 + c] = fmaf(av[r], xv[c], acc[u][r * 4 + c]);
        }
      }
    }
    __syncthreads();
  }
  float* C = Ews + f * D * D;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int tile = threadIdx.x + u * kThreads;
    if (tile < ntiles) {
      const int i0 = (tile / nt4) * 4, j0 = (tile % nt4) * 4;
#pragma unroll
      for (int r = 0; r < 4; ++r)
        *reinterpret_cast<float4*>(C + (i0 + r) * D + j0) =
            make_float4(acc[u][r * 4 + 0] * co, acc[u][r * 4 + 1] * co, acc[u][r * 4 + 2] * co,
                        acc[u][r * 4 + 3] * co);
    }
  }
}

// Reverse scan of the state gradient over kColBlock columns of one head:
// U_{T-1} = dS_T + E_{T-1}; U_{t-1} = E_{t-1} + g_t (U_t - M_t^T U_t); writes every
// U_t and dS_0 = g_0 (U_0 - M_0^T U_0).  grid = (heads, D / kColBlock).
__global__ void __launch_bounds__(kScanThreads) rscan_kernel(const float* __restrict__ Mws,
                                                             const float* __restrict__ Ews,
                                                             const float* __restrict__ g,
                                                             const float* __restrict__ dstate_out,
                                                             float* __restrict__ Uws, float* __restrict__ dstate_in,
                                                             int T, int D, int logits) {
  extern __shared__ float smem[];
  float* sM = smem;          // [D][D]
  float* sU = smem + D * D;  // [D][kColBlock]
  constexpr int W = kColBlock;
  const long long bh = blockIdx.x;
  const int j0 = blockIdx.y * W;
  const size_t DD = (size_t)D * D;
  {
    const float* E = Ews + (bh * T + T - 1) * DD;
    for (int idx = threadIdx.x; idx < D * W; idx += blockDim.x) {
      const int i = idx / W, c = idx % W;
      float u = E[i * D + j0 + c];
      if (dstate_out) u += dstate_out[bh * DD + i * D + j0 + c];
      sU[idx] = u;
    }
  }
  const bool active = (int)threadIdx.x < D;  // D/4 row tiles x 4 column tiles
  const int i0 = (threadIdx.x / 4) * 4, c0 = (threadIdx.x % 4) * 4;
  for (int t = T - 1; t >= 0; --t) {
    const long long f = bh * T + t;
    __syncthreads();  // sU complete; sM free
    for (int idx = threadIdx.x; idx < D * W; idx += blockDim.x) {
      const int i = idx / W, c = idx % W;
      Uws[f * DD + i * D + j0 + c] = sU[idx];
    }
    const float4* Mg = reinterpret_cast<const float4*>(Mws + f * DD);
    for (int idx = threadIdx.x; idx < D * D / 4; idx += blockDim.x) reinterpret_cast<float4*>(sM)[idx] = Mg[idx];
    __syncthreads();
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    if (active) {
      // (M^T U)[i][c] = sum_k M[k][i] U[k][c]: both operands read along rows.
      for (int kk = 0; kk < D; ++kk) {
        const float4 m = *reinterpret_cast<const float4*>(sM + kk * D + i0);
        const float4 x = *reinterpret_cast<const float4*>(sU + kk * W + c0);
        const float mv[4] = {m.x, m.y, m.z, m.w};
        const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[r * 4 + c] = fmaf(mv[r], xv[c], acc[r * 4 + c]);
      }
    }
    __syncthreads();  // every product read the old U
    if (active) {
      const float gt = decay_of(g[f], logits);
      const float* E = t > 0 ? Ews + (f - 1) * DD : nullptr;
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int i = i0 + r, cc = c0 + c;
          float u = gt * (sU[i * W + cc] - acc[r * 4 + c]);
          if (E) u += E[i * D + j0 + cc];
          sU[i * W + cc] = u;
        }
    }
  }
  __syncthreads();
  if (dstate_in)
    for (int idx = threadIdx.x; idx < D * W; idx += blockDim.x) {
      const int i = idx / W, c = idx % W;
      dstate_in[bh * DD + i * D + j0 + c] = sU[idx];
    }
}

// Rows x D product C = A B for A [kRows][D] and B [D][D] in shared memory, every
// thread computing 4 x 4 tiles `task`, `task + kThreads`, ... of C.
__device__ __forceinline__ void rows_times_matrix_tile(const float* A, const float* Bm, int D, int tile,
                                                       float acc[16]) {
  const int ntj = D / 4;
  const int r0 = (tile / ntj) * 4, j0 = (tile % ntj) * 4;
  for (int kk = 0; kk < D; ++kk) {
    const float4 x = *reinterpret_cast<const float4*>(Bm + kk * D + j0);
    const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float a = A[(r0 + r) * D + kk];
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r * 4 + c] = fmaf(a, xv[c], acc[r * 4 + c]);
    }
  }
}

// dK, dV, dbeta and the partial dg sums of kRows tokens of one frame-head.
// grid = (frame-heads, token tiles).  dg_part[f * ntiles + tile] receives
// -sum_s beta_s <dR_s, P_s> over the tile's tokens, plus <U_t, S_{t-1}> in tile 0.
template <typename TIn>
__global__ void __launch_bounds__(kThreads) kv_grad_kernel(
    const TIn* __restrict__ k, const TIn* __restrict__ v, const float* __restrict__ g,
    const float* __restrict__ beta, const float* __restrict__ state_in, const float* __restrict__ Sws,
    const float* __restrict__ Uws, TIn* __restrict__ dk, TIn* __restrict__ dv, float* __restrict__ dbeta,
    float* __restrict__ dg_part, int T, int S, int D, float ck, int logits) {
  extern __shared__ float smem[];
  float* sSp = smem;              // [D][D]  S_{t-1}; transposed before phase 2
  float* sU = sSp + D * D;        // [D][D]  U_t;     transposed before phase 2
  float* sK = sU + D * D;         // [kRows][D]  K~
  float* sV = sK + kRows * D;     // [kRows][D]  V
  float* sA = sV + kRows * D;     // [kRows][D]  P, then R
  float* sB = sA + kRows * D;     // [kRows][D]  dR, then dP
  __shared__ float sBeta[kRows];
  __shared__ float sRed[kThreads / 32];
  const long long f = blockIdx.x;
  const long long bh = f / T;
  const int t = (int)(f % T);
  const int s0 = blockIdx.y * kRows;
  const int n = min(kRows, S - s0);
  const size_t DD = (size_t)D * D;
  const float* Sp = t > 0 ? Sws + (f - 1) * DD : (state_in ? state_in + bh * DD : nullptr);
  for (int idx = threadIdx.x; idx < D * D / 4; idx += blockDim.x) {
    reinterpret_cast<float4*>(sSp)[idx] = Sp ? reinterpret_cast<const float4*>(Sp)[idx] : make_float4(0, 0, 0, 0);
    reinterpret_cast<float4*>(sU)[idx] = reinterpret_cast<const float4*>(Uws + f * DD)[idx];
  }
  for (int idx = threadIdx.x; idx < kRows * D; idx += blockDim.x) {
    const int s = idx / D;
    const long long o = (f * S + s0 + s) * D + idx % D;
    sK[idx] = s < n ? ck * to_f32(k[o]) : 0.f;
    sV[idx] = s < n ? to_f32(v[o]) : 0.f;
  }
  if (threadIdx.x < kRows)
    sBeta[threadIdx.x] = (int)threadIdx.x < n ? beta_of(beta[f * S + s0 + threadIdx.x], logits) : 0.f;
  const float gt = decay_of(g[f], logits);
  __syncthreads();

  // phase 1: P = K~ S_{t-1} -> sA, dR = K~ U_t -> sB
  const int ntile = (kRows / 4) * (D / 4);
  for (int task = threadIdx.x; task < 2 * ntile; task += kThreads) {
    const int which = task / ntile, tile = task % ntile;
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    rows_times_matrix_tile(sK, which ? sU : sSp, D, tile, acc);
    float* C = which ? sB : sA;
    const int r0 = (tile / (D / 4)) * 4, j0 = (tile % (D / 4)) * 4;
#pragma unroll
    for (int r = 0; r < 4; ++r)
      *reinterpret_cast<float4*>(C + (r0 + r) * D + j0) =
          make_float4(acc[r * 4 + 0], acc[r * 4 + 1], acc[r * 4 + 2], acc[r * 4 + 3]);
  }
  // <U_t, S_{t-1}> (tile 0 of each frame-head only); independent of phase 1.
  float dg_mat = 0.f;
  if (blockIdx.y == 0)
    for (int idx = threadIdx.x; idx < D * D; idx += blockDim.x) dg_mat = fmaf(sU[idx], sSp[idx], dg_mat);
  __syncthreads();

  // element-wise: R, dP into sA, sB; dV and dbeta out; row sums by warp shuffles
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  float dg_tok = 0.f;
  for (int s = warp; s < kRows; s += kThreads / 32) {
    const float b = sBeta[s];
    float db = 0.f, dp = 0.f;
    for (int j = lane; j < D; j += 32) {
      const float p = sA[s * D + j], dr = sB[s * D + j];
      const float res = sV[s * D + j] - gt * p;
      db = fmaf(dr, res, db);
      dp = fmaf(dr, p, dp);
      sA[s * D + j] = b * res;
      sB[s * D + j] = -gt * b * dr;
      if (s < n) from_f32(dv[(f * S + s0 + s) * D + j], b * dr);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      db += __shfl_xor_sync(0xffffffffu, db, o);
      dp += __shfl_xor_sync(0xffffffffu, dp, o);
    }
    if (lane == 0 && s < n) dbeta[f * S + s0 + s] = logits ? db * b * (1.f - b) : db;
    dg_tok -= b * dp;
  }
  // block sum of dg_mat (every lane) and dg_tok (lane 0 of each warp)
  float part = dg_mat + (lane == 0 ? dg_tok : 0.f);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if (lane == 0) sRed[warp] = part;
  // transpose S_{t-1} and U_t in place for phase 2 (each pair i < j swapped by one thread)
  for (int idx = threadIdx.x; idx < D * D; idx += blockDim.x) {
    const int i = idx / D, j = idx % D;
    if (i < j) {
      float a = sSp[i * D + j];
      sSp[i * D + j] = sSp[j * D + i];
      sSp[j * D + i] = a;
      a = sU[i * D + j];
      sU[i * D + j] = sU[j * D + i];
      sU[j * D + i] = a;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) tot += sRed[w];
    dg_part[f * gridDim.y + blockIdx.y] = tot;
  }

  // phase 2: dK~ = R U_t^T + dP S_{t-1}^T  (sU, sSp now hold the transposes)
  for (int tile = threadIdx.x; tile < ntile; tile += kThreads) {
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    rows_times_matrix_tile(sA, sU, D, tile, acc);
    rows_times_matrix_tile(sB, sSp, D, tile, acc);
    const int r0 = (tile / (D / 4)) * 4, i0 = (tile % (D / 4)) * 4;
#pragma unroll
    for (int r = 0; r < 4; ++r)
      if (r0 + r < n) {
        TIn* o = dk + (f * S + s0 + r0 + r) * D + i0;
#pragma unroll
        for (int c = 0; c < 4; ++c) from_f32(o[c], ck * acc[r * 4 + c]);
      }
  }
}

// dQ = co dO S_t^T for kQRows tokens of one frame-head.  grid = (frame-heads, token tiles).
template <typename TIn>
__global__ void __launch_bounds__(kThreads) q_grad_kernel(const TIn* __restrict__ dout, const float* __restrict__ Sws,
                                                          TIn* __restrict__ dq, int S, int D, float co) {
  extern __shared__ float smem[];
  float* sT = smem;          // [D][D]  S_t transposed
  float* sO = smem + D * D;  // [kQRows][D]
  const long long f = blockIdx.x;
  const int s0 = blockIdx.y * kQRows;
  const int n = min(kQRows, S - s0);
  const float* St = Sws + f * (size_t)D * D;
  for (int idx = threadIdx.x; idx < D * D; idx += blockDim.x) sT[(idx % D) * D + idx / D] = St[idx];
  for (int idx = threadIdx.x; idx < kQRows * D; idx += blockDim.x) {
    const int s = idx / D;
    sO[idx] = s < n ? to_f32(dout[(f * S + s0 + s) * D + idx % D]) : 0.f;
  }
  __syncthreads();
  const int ntile = (kQRows / 4) * (D / 4);
  for (int tile = threadIdx.x; tile < ntile; tile += kThreads) {
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    rows_times_matrix_tile(sO, sT, D, tile, acc);
    const int r0 = (tile / (D / 4)) * 4, i0 = (tile % (D / 4)) * 4;
#pragma unroll
    for (int r = 0; r < 4; ++r)
      if (r0 + r < n) {
        TIn* o = dq + (f * S + s0 + r0 + r) * D + i0;
#pragma unroll
        for (int c = 0; c < 4; ++c) from_f32(o[c], co * acc[r * 4 + c]);
      }
  }
}

// dg[f] = sum of the frame-head's partial sums (times dg/dlogit for logits).
__global__ void dg_sum_kernel(const float* __restrict__ dg_part, const float* __restrict__ g, float* __restrict__ dg,
                              long long nframes, int ntiles, int logits) {
  const long long f = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (f >= nframes) return;
  float s = 0.f;
  for (int i = 0; i < ntiles; ++i) s += dg_part[f * ntiles + i];
  if (logits) {
    const float gt = decay_of(g[f], 1);
    s *= -gt * (1.f - gt);
  }
  dg[f] = s;
}

struct BwdLayout {
  size_t m_off, e_off, s_off, u_off, dg_off, total;
  int ntiles;
};

BwdLayout bwd_layout(const Problem& p) {
  BwdLayout L{};
  const size_t per = align_up((size_t)p.BHT() * p.D * p.D * sizeof(float), 256);
  L.ntiles = (p.S + kRows - 1) / kRows;
  L.m_off = 0;
  L.e_off = L.m_off + per;
  L.s_off = L.e_off + per;
  L.u_off = L.s_off + per;
  L.dg_off = L.u_off + per;
  L.total = L.dg_off + align_up((size_t)p.BHT() * L.ntiles * sizeof(float), 256);
  return L;
}

using Grads = BwdGrads;

template <typename TIn>
int run_bwd(const Problem& p, const Grads& gr, void* ws, cudaStream_t st, bool states_ready) {
  const BwdLayout L = bwd_layout(p);
  char* w = static_cast<char*>(ws);
  float* Mws = reinterpret_cast<float*>(w + L.m_off);
  float* Ews = reinterpret_cast<float*>(w + L.e_off);
  float* Sws = reinterpret_cast<float*>(w + L.s_off);
  float* Uws = reinterpret_cast<float*>(w + L.u_off);
  float* dg_part = reinterpret_cast<float*>(w + L.dg_off);
  const int D = p.D;
  const size_t mat = (size_t)D * D * sizeof(float);

  // forward states (b_t lands in the E buffer and is overwritten below), unless a
  // forward call left them in the workspace: the float32 forward's scratch (M_t,
  // b_t, S_t, each BHT x D x D, 256-byte aligned) is this layout's first three regions
  if (!states_ready) {
    Problem pf = p;
    pf.out = nullptr;
    pf.state_out = nullptr;
    const int rc = simt_states(pf, Mws, Ews, Sws, st);
    if (rc != kOk) return rc;
  }

  {
    ProfScope ps(st, "bwd_qdo");
    qdo_kernel<TIn><<<(unsigned)p.BHT(), kThreads, 2 * kTok * D * sizeof(float), st>>>(
        static_cast<const TIn*>(p.q), static_cast<const TIn*>(gr.dout), Ews, p.S, D, p.out_scale);
  }
  if (cudaGetLastError() != cudaSuccess) return kCuda;

  const size_t rsmem = mat + (size_t)D * kColBlock * sizeof(float);
  if (cudaFuncSetAttribute(rscan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rsmem) != cudaSuccess)
    return kCuda;
  {
    ProfScope ps(st, "bwd_rscan");
    rscan_kernel<<<dim3((unsigned)p.BH(), D / kColBlock), kScanThreads, rsmem, st>>>(
        Mws, Ews, p.g, gr.dstate_out, Uws, gr.dstate_in, p.T, D, p.gate_logits);
  }
  if (cudaGetLastError() != cudaSuccess) return kCuda;

  const size_t ksmem = 2 * mat + 4 * (size_t)kRows * D * sizeof(float);
  if (cudaFuncSetAttribute(kv_grad_kernel<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ksmem) !=
      cudaSuccess)
    return kCuda;
  {
    ProfScope ps(st, "bwd_kv_grad");
    kv_grad_kernel<TIn><<<dim3((unsigned)p.BHT(), L.ntiles), kThreads, ksmem, st>>>(
        static_cast<const TIn*>(p.k), static_cast<const TIn*>(p.v), p.g, p.beta, p.state_in, Sws, Uws,
        static_cast<TIn*>(gr.dk), static_cast<TIn*>(gr.dv), gr.dbeta, dg_part, p.T, p.S, D, p.key_scale,
        p.gate_logits);
  }
  if (cudaGetLastError() != cudaSuccess) return kCuda;

  const size_t qsmem = mat + (size_t)kQRows * D * sizeof(float);
  if (cudaFuncSetAttribute(q_grad_kernel<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)qsmem) !=
      cudaSuccess)
    return kCuda;
  {
    ProfScope ps(st, "bwd_q_grad");
    q_grad_kernel<TIn><<<dim3((unsigned)p.BHT(), (p.S + kQRows - 1) / kQRows), kThreads, qsmem, st>>>(
        static_cast<const TIn*>(gr.dout), Sws, static_cast<TIn*>(gr.dq), p.S, D, p.out_scale);
  }
  if (cudaGetLastError() != cudaSuccess) return kCuda;

  return launch_dg_sum(dg_part, p.g, gr.dg, p.BHT(), L.ntiles, p.gate_logits, st);
}

// The backward's own layout, and never less than any forward form needs for the
// shape, so one workspace serves a forward call and the backward that reuses its
// states.
size_t workspace_of(const Problem& p) {
  const size_t own = p.dtype == GDN_BF16 ? tc_bwd_workspace_bytes(p) : bwd_layout(p).total;
  Problem pf = p;
  pf.mode = GDN_MODE_PREFIX;  // the largest forward form
  const size_t fwd = scratch_bytes(pf);
  return own > fwd ? own : fwd;
}


// Validation shared by gdn_frame_bwd and gdn_bwd_workspace_bytes; fills p and gr.
int check_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta, const float* state_in,
              const void* dout, const float* dstate_out, void* dq, void* dk, void* dv, float* dg, float* dbeta,
              float* dstate_in, int B, int H, int T, int S, int D, int dtype, Problem* p, Grads* gr) {
  // the forward's checks (dout stands in for `out`: same dtype, shape and alignment)
  int rc = check_args(q, k, v, g, beta, state_in, const_cast<void*>(dout), nullptr, B, H, T, S, D, dtype,
                      GDN_MODE_SEQUENTIAL, p);
  if (rc != kOk) return rc;
  // token tiles are the second grid dimension (at most 65535)
  if ((S + kRows - 1) / kRows > 65535) return kUnsupported;
  if (T > 0) {
    if (!dq || !dk || !dv || !dg || !dbeta) return kInvalidArg;
    if (!aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16)) return kMisaligned;
    if (!aligned(dg, 4) || !aligned(dbeta, 4)) return kMisaligned;
  }
  if (dstate_out && !aligned(dstate_out, 16)) return kMisaligned;
  if (dstate_in && !aligned(dstate_in, 16)) return kMisaligned;
  p->out = nullptr;
  gr->dout = dout;
  gr->dstate_out = dstate_out;
  gr->dq = dq;
  gr->dk = dk;
  gr->dv = dv;
  gr->dg = dg;
  gr->dbeta = dbeta;
  gr->dstate_in = dstate_in;
  return kOk;
}

int frame_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta, const float* state_in,
              const void* dout, const float* dstate_out, void* dq, void* dk, void* dv, float* dg, float* dbeta,
              float* dstate_in, int B, int H, int T, int S, int D, int dtype, void* workspace,
              size_t workspace_bytes, void* stream, int flags) {
  if (flags & ~(GDN_BWD_STATES_IN_WORKSPACE | GDN_BWD_GATE_LOGITS)) return kInvalidArg;
  Problem p{};
  Grads gr{};
  int rc = check_bwd(q, k, v, g, beta, state_in, dout, dstate_out, dq, dk, dv, dg, dbeta, dstate_in, B, H, T, S, D,
                     dtype, &p, &gr);
  if (rc != kOk) return rc;
  p.gate_logits = (flags & GDN_BWD_GATE_LOGITS) ? 1 : 0;
  const bool states_ready = (flags & GDN_BWD_STATES_IN_WORKSPACE) != 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0) {  // the initial state's gradient is the final state's
    if (!dstate_in) return kOk;
    const size_t bytes = (size_t)p.BH() * D * D * sizeof(float);
    const cudaError_t e = dstate_out ? cudaMemcpyAsync(dstate_in, dstate_out, bytes, cudaMemcpyDeviceToDevice, st)
                                     : cudaMemsetAsync(dstate_in, 0, bytes, st);
    return e == cudaSuccess ? kOk : kCuda;
  }
  if (!workspace || workspace_bytes < workspace_of(p)) return kWorkspace;
  if (!aligned(workspace, 256)) return kMisaligned;
  p.status = device_status_word();
  if (!p.status) return kCuda;
  return dtype == GDN_F32 ? run_bwd<float>(p, gr, workspace, st, states_ready)
                          : tc_backward(p, gr, workspace, st, states_ready);
}

}  // namespace

int launch_dg_sum(const float* dg_part, const float* g, float* dg, long long nframes, int ntiles, int logits,
                  cudaStream_t st) {
  {
    ProfScope ps(st, "bwd_dg_sum");
    dg_sum_kernel<<<(unsigned)((nframes + 255) / 256), 256, 0, st>>>(dg_part, g, dg, nframes, ntiles, logits);
  }
  return cudaGetLastError() == cudaSuccess ? kOk : kCuda;
}

}  // namespace gdn

using namespace gdn;

extern "C" size_t gdn_bwd_workspace_bytes(int B, int H, int T, int S, int D, int dtype) {
  static const char dummy[16] __attribute__((aligned(16))) = {0};
  const void* d = dummy;
  float* fd = const_cast<float*>(reinterpret_cast<const float*>(dummy));
  Problem p{};
  Grads gr{};
  if (check_bwd(d, d, d, fd, fd, nullptr, d, nullptr, const_cast<void*>(d), const_cast<void*>(d),
                const_cast<void*>(d), fd, fd, nullptr, B, H, T, S, D, dtype, &p, &gr) != kOk)
    return 0;
  return T == 0 ? 0 : workspace_of(p);
}

extern "C" int gdn_frame_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                             const float* state_in, const void* dout, const float* dstate_out, void* dq, void* dk,
                             void* dv, float* dg, float* dbeta, float* dstate_in, int B, int H, int T, int S, int D,
                             int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  return frame_bwd(q, k, v, g, beta, state_in, dout, dstate_out, dq, dk, dv, dg, dbeta, dstate_in, B, H, T, S, D,
                   dtype, workspace, workspace_bytes, stream, 0);
}

extern "C" int gdn_frame_bwd_ex(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                const float* state_in, const void* dout, const float* dstate_out, void* dq, void* dk,
                                void* dv, float* dg, float* dbeta, float* dstate_in, int B, int H, int T, int S,
                                int D, int dtype, int flags, void* workspace, size_t workspace_bytes, void* stream) {
  return frame_bwd(q, k, v, g, beta, state_in, dout, dstate_out, dq, dk, dv, dg, dbeta, dstate_in, B, H, T, S, D,
                   dtype, workspace, workspace_bytes, stream, flags);
}

extern "C" int gdn_frame_bwd_from_logits(const void* q, const void* k, const void* v, const float* g_logit,
                                         const float* beta_logit, const float* state_in, const void* dout,
                                         const float* dstate_out, void* dq, void* dk, void* dv, float* dg_logit,
                                         float* dbeta_logit, float* dstate_in, int B, int H, int T, int S, int D,
                                         int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  return frame_bwd(q, k, v, g_logit, beta_logit, state_in, dout, dstate_out, dq, dk, dv, dg_logit, dbeta_logit,
                   dstate_in, B, H, T, S, D, dtype, workspace, workspace_bytes, stream, GDN_BWD_GATE_LOGITS);
}
