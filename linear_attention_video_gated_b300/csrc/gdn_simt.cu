// SIMT (CUDA-core, float32 FMA) implementation of the frame-wise GDN forward
// scan in its transition form (see gdn_internal.h).  It serves float32 I/O,
// where the result must match the fp64 definition to ~1e-6 relative, which
// bf16 tensor-core operands cannot give.  Three kernels per call:
//
//   gram    : M_t = K~^T diag(beta) K~ and b_t = K~^T diag(beta) V_t, every frame
//             in parallel (one CTA per frame-head and output matrix);
//   scan    : S_t = g_t (S_{t-1} - M_t S_{t-1}) + b_t, one CTA per head, frame by
//             frame, the state resident in shared memory;
//   readout : O_t = Q_t S_t / sqrt(D), every frame and token tile in parallel.
//
// Workspace per frame-head: M_t, b_t and S_t, each D x D float32.
//
// Prefix mode (GDN_MODE_PREFIX) composes the maps chunk by chunk instead of
// frame by frame: compose (per head and chunk, parallel) -> boundary scan (per
// head, over chunks) -> replay (per head and chunk, parallel) -> readout.
#include <cuda_bf16.h>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kTok = 32;       // tokens staged per gram iteration
constexpr int kOutRows = 64;   // tokens per readout CTA
constexpr int kChunk = 16;     // frames per chunk in prefix mode

// C[i][j] = scale * sum_s (beta_s A[s][i]) X[s][j]; which = 0 -> X = K (gives M),
// which = 1 -> X = V (gives b).  One CTA per (frame-head, which).
template <typename TIn>
__global__ void __launch_bounds__(kThreads) gram_kernel(const TIn* __restrict__ k, const TIn* __restrict__ v,
                                                        const float* __restrict__ beta, float* __restrict__ Mws,
                                                        float* __restrict__ bws, int S, int D, float ck, int logits,
                                                        int variant) {
  extern __shared__ float smem[];
  float* sA = smem;             // [kTok][D]  beta * k
  float* sX = smem + kTok * D;  // [kTok][D]  k or v
  const long long f = blockIdx.x;
  const int which = blockIdx.y;
  const TIn* kf = k + f * S * D;
  const TIn* xf = (which == 0 ? k : v) + f * S * D;
  const float* bf = beta + f * S;
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
      float a = 0.f, x = 0.f;
      if (s < n) {
        const long long o = (long long)(s0 + s) * D + (idx % D);
        const float bt = variant == kReluLinear ? 1.f : beta_of(bf[s0 + s], logits);
        a = bt * relu_if(to_f32(kf[o]), variant);
        x = to_f32(xf[o]);
      }
      sA[idx] = a;
      sX[idx] = x;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int tile = threadIdx.x + u * kThreads;
      if (tile < ntiles) {
        const int i0 = (tile / nt4) * 4, j0 = (tile % nt4) * 4;
        for (int s = 0; s < n; ++s) {
          const float4 a = *reinterpret_cast<const float4*>(sA + s * D + i0);
          const float4 x = *reinterpret_cast<const float4*>(sX + s * D + j0);
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
  float* C = (which == 0 ? Mws : bws) + f * D * D;
  const float sc = which == 0 ? ck * ck : ck;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int tile = threadIdx.x + u * kThreads;
    if (tile < ntiles) {
      const int i0 = (tile / nt4) * 4, j0 = (tile % nt4) * 4;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        float4 o = make_float4(acc[u][r * 4 + 0] * sc, acc[u][r * 4 + 1] * sc, acc[u][r * 4 + 2] * sc,
                               acc[u][r * 4 + 3] * sc);
        *reinterpret_cast<float4*>(C + (i0 + r) * D + j0) = o;
      }
    }
  }
}

// X <- A-map applied: X_new = g (X - M X) + c * b, for a D x W state X held in
// shared memory (W = D for a state, 2D for a composed map [A | b]).
// Each thread owns up to 8 4x4 output tiles.
__device__ void affine_step(float* sX, const float* sM, const float* __restrict__ bglob, float g, int D, int W,
                            int b_col0, float* __restrict__ out_glob) {
  const int nti = D / 4, ntj = W / 4;
  const int ntiles = nti * ntj;
  float acc[8][16];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int tile = threadIdx.x + u * kThreads;
    if (tile < ntiles) {
      const int i0 = (tile / ntj) * 4, j0 = (tile % ntj) * 4;
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[u][e] = 0.f;
      for (int kk = 0; kk < D; ++kk) {
        const float m[4] = {sM[(i0 + 0) * D + kk], sM[(i0 + 1) * D + kk], sM[(i0 + 2) * D + kk],
                            sM[(i0 + 3) * D + kk]};
        const float4 x = *reinterpret_cast<const float4*>(sX + kk * W + j0);
        const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[u][r * 4 + c] = fmaf(m[r], xv[c], acc[u][r * 4 + c]);
      }
    }
  }
  __syncthreads();  // every product read the old X
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int tile = threadIdx.x + u * kThreads;
    if (tile < ntiles) {
      const int i0 = (tile / ntj) * 4, j0 = (tile % ntj) * 4;
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int i = i0 + r, j = j0 + c;
          float x = g * (sX[i * W + j] - acc[u][r * 4 + c]);
          if (bglob != nullptr && j >= b_col0) x += bglob[i * D + (j - b_col0)];
          sX[i * W + j] = x;
          if (out_glob != nullptr) out_glob[i * W + j] = x;
        }
    }
  }
  __syncthreads();
}

// Sequential scan: one CTA per head.
__global__ void __launch_bounds__(kThreads) scan_kernel(const float* __restrict__ Mws, const float* __restrict__ bws,
                                                        const float* __restrict__ g, const float* state_in,
                                                        float* __restrict__ Sws, float* state_out, int T, int D,
                                                        int logits, int variant) {
  extern __shared__ float smem[];
  float* sS = smem;          // [D][D]
  float* sM = smem + D * D;  // [D][D]
  const long long bh = blockIdx.x;
  for (int idx = threadIdx.x; idx < D * D; idx += blockDim.x)
    sS[idx] = state_in ? state_in[bh * D * D + idx] : 0.f;
  __syncthreads();
  for (int t = 0; t < T; ++t) {
    const long long f = bh * T + t;
    for (int idx = threadIdx.x; idx < D * D; idx += blockDim.x)
      sM[idx] = variant == kReluLinear ? 0.f : Mws[f * D * D + idx];
    __syncthreads();
    affine_step(sS, sM, bws + f * D * D, (variant == kReluLinear ? 1.f : decay_of(g[f], logits)), D, D, 0, Sws + f * D * D);
  }
  if (state_out)
    for (int idx = threadIdx.x; idx < D * D; idx += blockDim.x) state_out[bh * D * D + idx] = sS[idx];
}

// Prefix mode, pass 1: composed map of each chunk of frames, [A_c | b_c] (D x 2D),
// starting from [I | 0].  One CTA per (head, chunk).
__global__ void __launch_bounds__(kThreads) compose_kernel(const float* __restrict__ Mws, const float* __restrict__ bws,
                                                           const float* __restrict__ g, float* __restrict__ maps,
                                                           int T, int D, int nchunks, int logits, int variant) {
  extern __shared__ float smem[];
  float* sX = smem;              // [D][2D]
  float* sM = smem + 2 * D * D;  // [D][D]
  const long long bh = blockIdx.x / nchunks;
  const int c = blockIdx.x % nchunks;
  const int t0 = c * kChunk, t1 = min(T, t0 + kChunk);
  for (int idx = threadIdx.x; idx < 2 * D * D; idx += blockDim.x) {
    const int i = idx / (2 * D), j = idx % (2 * D);
    sX[idx] = (j == i) ? 1.f : 0.f;
  }
  __syncthreads();
  for (int t = t0; t < t1; ++t) {
    const long long f = bh * T + t;
    for (int idx = threadIdx.x; idx < D * D; idx += blockDim.x)
      sM[idx] = variant == kReluLinear ? 0.f : Mws[f * D * D + idx];
    __syncthreads();
    affine_step(sX, sM, bws + f * D * D, (variant == kReluLinear ? 1.f : decay_of(g[f], logits)), D, 2 * D, D, nullptr);
  }
  float* dst = maps + (bh * nchunks + c) * 2 * D * D;
  for (int idx = threadIdx.x; idx < 2 * D * D; idx += blockDim.x) dst[idx] = sX[idx];
}

// Prefix mode, pass 2: exclusive scan over chunk boundaries, S_c = A_c S_{c-1} + b_c,
// one CTA per head.  Writes the initial state of every chunk; and the final state.
__global__ void __launch_bounds__(kThreads) boundary_kernel(const float* __restrict__ maps, const float* state_in,
                                                            float* __restrict__ starts, float* state_out, int D,
                                                            int nchunks) {
  extern __shared__ float smem[];
  float* sS = smem;          // [D][D]
  float* sA = smem + D * D;  // [D][2D]
  const long long bh = blockIdx.x;
  for (int idx = threadIdx.x; idx < D * D; idx += blockDim.x)
    sS[idx] = state_in ? state_in[bh * D * D + idx] : 0.f;
  __syncthreads();
  const int nti = D / 4;
  const int ntiles = nti * nti;
  for (int c = 0; c < nchunks; ++c) {
    for (int idx = threadIdx.x; idx < D * D; idx += blockDim.x) starts[(bh * nchunks + c) * D * D + idx] = sS[idx];
    const float* mp = maps + (bh * nchunks + c) * 2 * D * D;
    for (int idx = threadIdx.x; idx < 2 * D * D; idx += blockDim.x) sA[idx] = mp[idx];
    __syncthreads();
    float acc[4][16];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int tile = threadIdx.x + u * kThreads;
      if (tile < ntiles) {
        const int i0 = (tile / nti) * 4, j0 = (tile % nti) * 4;
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[u][r * 4 + q] = sA[(i0 + r) * 2 * D + D + j0 + q];  // b_c
        for (int kk = 0; kk < D; ++kk) {
          const float4 x = *reinterpret_cast<const float4*>(sS + kk * D + j0);
          const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const float a = sA[(i0 + r) * 2 * D + kk];
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[u][r * 4 + q] = fmaf(a, xv[q], acc[u][r * 4 + q]);
          }
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int tile = threadIdx.x + u * kThreads;
      if (tile < ntiles) {
        const int i0 = (tile / nti) * 4, j0 = (tile % nti) * 4;
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int q = 0; q < 4; ++q) sS[(i0 + r) * D + j0 + q] = acc[u][r * 4 + q];
      }
    }
    __syncthreads();
  }
  if (state_out)
    for (int idx = threadIdx.x; idx < D * D; idx += blockDim.x) state_out[bh * D * D + idx] = sS[idx];
}

// Prefix mode, pass 3: replay each chunk from its true initial state, writing S_t.
__global__ void __launch_bounds__(kThreads) replay_kernel(const float* __restrict__ Mws, const float* __restrict__ bws,
                                                          const float* __restrict__ g, const float* __restrict__ starts,
                                                          float* __restrict__ Sws, int T, int D, int nchunks,
                                                          int logits, int variant) {
  extern __shared__ float smem[];
  float* sS = smem;
  float* sM = smem + D * D;
  const long long bh = blockIdx.x / nchunks;
  const int c = blockIdx.x % nchunks;
  const int t0 = c * kChunk, t1 = min(T, t0 + kChunk);
  const float* st = starts + (bh * nchunks + c) * D * D;
  for (int idx = threadIdx.x; idx < D * D; idx += blockDim.x) sS[idx] = st[idx];
  __syncthreads();
  for (int t = t0; t < t1; ++t) {
    const long long f = bh * T + t;
    for (int idx = threadIdx.x; idx < D * D; idx += blockDim.x)
      sM[idx] = variant == kReluLinear ? 0.f : Mws[f * D * D + idx];
    __syncthreads();
    affine_step(sS, sM, bws + f * D * D, (variant == kReluLinear ? 1.f : decay_of(g[f], logits)), D, D, 0, Sws + f * D * D);
  }
}

// O_t = Q_t S_t * co for a tile of kOutRows tokens.  grid = (frame-heads, token tiles).
template <typename TIn>
__global__ void __launch_bounds__(kThreads) readout_kernel(const TIn* __restrict__ q, const float* __restrict__ Sws,
                                                           TIn* __restrict__ out, int S, int D, float co, int variant) {
  extern __shared__ float smem[];
  float* sS = smem;          // [D][D]
  float* sQ = smem + D * D;  // [kOutRows][D]
  const long long f = blockIdx.x;
  const int s0 = blockIdx.y * kOutRows;
  const int n = min(kOutRows, S - s0);
  for (int idx = threadIdx.x; idx < D * D; idx += blockDim.x) sS[idx] = Sws[f * D * D + idx];
  for (int idx = threadIdx.x; idx < kOutRows * D; idx += blockDim.x) {
    const int s = idx / D;
    sQ[idx] = s < n ? relu_if(to_f32(q[(f * S + s0 + s) * D + idx % D]), variant) : 0.f;
  }
  __syncthreads();
  const int ntj = D / 4;
  const int ntiles = (kOutRows / 4) * ntj;
  for (int tile = threadIdx.x; tile < ntiles; tile += blockDim.x) {
    const int r0 = (tile / ntj) * 4, j0 = (tile % ntj) * 4;
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    for (int kk = 0; kk < D; ++kk) {
      const float4 x = *reinterpret_cast<const float4*>(sS + kk * D + j0);
      const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float a = sQ[(r0 + r) * D + kk];
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r * 4 + c] = fmaf(a, xv[c], acc[r * 4 + c]);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if (r0 + r < n) {
        TIn* o = out + (f * S + s0 + r0 + r) * D + j0;
#pragma unroll
        for (int c = 0; c < 4; ++c) from_f32(o[c], acc[r * 4 + c] * co);
      }
    }
  }
}

// Fold of affine maps over chunks, float32 (used by both I/O dtypes): per head,
// x_{c+1} = A_c x_c + b_c for c = 0 .. nchunks - 1.  One CTA per (head, 16-column
// block of x): columns of x evolve independently, so a CTA holds its D x 16 block
// in registers (thread i = row i) and stages each A_c in shared memory.
//   boundary form (A_out null): x_0 = state_in (or zeros); writes x_c into
//     `starts` (the initial state of every chunk) and the last x into `x_out`.
//   summary form (A_out set): the composed map of all chunks, [A | b]: 2 D/16
//     column blocks per head, the first D columns starting as the identity and
//     taking no b term (A = A_{n-1} ... A_0), the last D starting at zero (b).
struct FoldArgs {
  const float* A;
  const float* b;
  long long chunk_stride;  // floats between consecutive chunk maps (and heads: nchunks of them)
  int ld;                  // floats between rows of A_c and of b_c
  int nchunks, D;
  const float* state_in;
  float* starts;
  float* x_out;
  float* A_out;
  float* b_out;
  unsigned int* status;
  size_t a_span, b_span, starts_span;  // extents (bytes) from A, b and starts (debug checks)
};

constexpr int kFoldThreads = 128;

__global__ void __launch_bounds__(kFoldThreads) chunk_fold_kernel(FoldArgs a) {
  extern __shared__ float fsm[];
  const int D = a.D, ncb = D / 16;
  float* sA = fsm;                // [D][D + 1]: the padding keeps row reads conflict-free
  float* sx = sA + D * (D + 1);   // [D][16]
  const bool summary = a.A_out != nullptr;
  const int ncbx = summary ? 2 * ncb : ncb;
  const long long bh = blockIdx.x / ncbx;
  const int cbx = (int)(blockIdx.x % ncbx);
  const bool ident = summary && cbx < ncb;
  const int cb = cbx < ncb ? cbx : cbx - ncb;
  const int i = threadIdx.x;
  const bool row = i < D;
  float x[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) x[j] = (ident && i == 16 * cb + j) ? 1.f : 0.f;
  if (!summary && a.state_in && row) {
#pragma unroll
    for (int j = 0; j < 16; ++j) x[j] = a.state_in[((size_t)bh * D + i) * D + 16 * cb + j];
  }
  for (int c = 0; c < a.nchunks; ++c) {
    const size_t mo = (size_t)(bh * a.nchunks + c) * a.chunk_stride;
    if (row) {
      if (a.starts && in_region((((size_t)(bh * a.nchunks + c) * D + i) * D + 16 * cb + 16) * 4, a.starts_span,
                                a.status)) {
        float* dst = a.starts + ((size_t)(bh * a.nchunks + c) * D + i) * D + 16 * cb;
#pragma unroll
        for (int j = 0; j < 16; ++j) dst[j] = x[j];
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) sx[i * 16 + j] = x[j];
      const float4* ar = reinterpret_cast<const float4*>(a.A + mo + (size_t)i * a.ld);
      const bool a_ok = in_region((mo + (size_t)i * a.ld + D) * 4, a.a_span, a.status);
      for (int k4 = 0; a_ok && k4 < D / 4; ++k4) {
        const float4 w = ar[k4];
        sA[i * (D + 1) + 4 * k4] = w.x;
        sA[i * (D + 1) + 4 * k4 + 1] = w.y;
        sA[i * (D + 1) + 4 * k4 + 2] = w.z;
        sA[i * (D + 1) + 4 * k4 + 3] = w.w;
      }
    }
    __syncthreads();
    if (row) {
      float y[16];
      const float* br = a.b + mo + (size_t)i * a.ld + 16 * cb;
      const bool b_ok = !ident && in_region((mo + (size_t)i * a.ld + 16 * cb + 16) * 4, a.b_span, a.status);
#pragma unroll
      for (int j = 0; j < 16; ++j) y[j] = b_ok ? br[j] : 0.f;
      for (int k = 0; k < D; ++k) {
        const float aik = sA[i * (D + 1) + k];
        const float4* xr = reinterpret_cast<const float4*>(sx + k * 16);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 w = xr[q];
          y[4 * q] = fmaf(aik, w.x, y[4 * q]);
          y[4 * q + 1] = fmaf(aik, w.y, y[4 * q + 1]);
          y[4 * q + 2] = fmaf(aik, w.z, y[4 * q + 2]);
          y[4 * q + 3] = fmaf(aik, w.w, y[4 * q + 3]);
        }
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) x[j] = y[j];
    }
    __syncthreads();
  }
  float* dst = summary ? (ident ? a.A_out : a.b_out) : a.x_out;
  if (row && dst) {
#pragma unroll
    for (int j = 0; j < 16; ++j) dst[((size_t)bh * D + i) * D + 16 * cb + j] = x[j];
  }
}

struct SimtLayout {
  size_t m_off, b_off, s_off, maps_off, starts_off, total;
  int nchunks;
};

SimtLayout simt_layout(const Problem& p, int mode) {
  SimtLayout L{};
  const size_t mat = (size_t)p.D * p.D * sizeof(float);
  const size_t per = (size_t)p.BHT() * mat;
  L.m_off = 0;
  L.b_off = align_up(L.m_off + per, 256);
  L.s_off = align_up(L.b_off + per, 256);
  L.total = align_up(L.s_off + per, 256);
  L.nchunks = (p.T + kChunk - 1) / kChunk;
  if (mode == 1) {
    L.maps_off = L.total;
    L.starts_off = align_up(L.maps_off + (size_t)p.BH() * L.nchunks * 2 * mat, 256);
    L.total = align_up(L.starts_off + (size_t)p.BH() * L.nchunks * mat, 256);
  }
  return L;
}

// The transition terms M_t, b_t of every frame, then the state S_t after every
// frame (sequential scan, or the prefix form's compose / boundary / replay when
// `prefix`).  Writes p.state_out when it is not null.
template <typename TIn>
int states(const Problem& p, float* Mws, float* bws, float* Sws, char* w, const SimtLayout& L, bool prefix,
           cudaStream_t st) {
  const int D = p.D;
  const size_t mat = (size_t)D * D * sizeof(float);

  const size_t gram_smem = 2 * kTok * D * sizeof(float);
  {
    ProfScope pg(st, "simt_gram");
    gram_kernel<TIn><<<dim3((unsigned)p.BHT(), 2), kThreads, gram_smem, st>>>(
        static_cast<const TIn*>(p.k), static_cast<const TIn*>(p.v), p.beta, Mws, bws, p.S, D, p.key_scale,
        p.gate_logits, p.variant);
  }
  if (cudaGetLastError() != cudaSuccess) return kCuda;

  if (!prefix) {
    const size_t smem = 2 * mat;
    if (cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return kCuda;
    {
      ProfScope ps(st, "simt_scan");
      scan_kernel<<<(unsigned)p.BH(), kThreads, smem, st>>>(Mws, bws, p.g, p.state_in, Sws, p.state_out, p.T, D,
                                                             p.gate_logits, p.variant);
    }
    if (cudaGetLastError() != cudaSuccess) return kCuda;
  } else {
    float* maps = reinterpret_cast<float*>(w + L.maps_off);
    float* starts = reinterpret_cast<float*>(w + L.starts_off);
    const size_t csmem = 3 * mat;
    if (cudaFuncSetAttribute(compose_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csmem) != cudaSuccess)
      return kCuda;
    {
      ProfScope pc(st, "simt_compose");
      compose_kernel<<<(unsigned)(p.BH() * L.nchunks), kThreads, csmem, st>>>(Mws, bws, p.g, maps, p.T, D, L.nchunks,
                                                                               p.gate_logits, p.variant);
    }
    if (cudaGetLastError() != cudaSuccess) return kCuda;
    if (cudaFuncSetAttribute(boundary_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csmem) !=
        cudaSuccess)
      return kCuda;
    {
      ProfScope pb(st, "simt_boundary");
      boundary_kernel<<<(unsigned)p.BH(), kThreads, csmem, st>>>(maps, p.state_in, starts, p.state_out, D, L.nchunks);
    }
    if (cudaGetLastError() != cudaSuccess) return kCuda;
    const size_t rsmem = 2 * mat;
    if (cudaFuncSetAttribute(replay_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rsmem) != cudaSuccess)
      return kCuda;
    {
      ProfScope pr(st, "simt_replay");
      replay_kernel<<<(unsigned)(p.BH() * L.nchunks), kThreads, rsmem, st>>>(Mws, bws, p.g, starts, Sws, p.T, D,
                                                                            L.nchunks, p.gate_logits, p.variant);
    }
    if (cudaGetLastError() != cudaSuccess) return kCuda;
  }
  return kOk;
}

template <typename TIn>
int run(const Problem& p, void* ws, cudaStream_t st) {
  const SimtLayout L = simt_layout(p, p.mode);
  char* w = static_cast<char*>(ws);
  float* Mws = reinterpret_cast<float*>(w + L.m_off);
  float* bws = reinterpret_cast<float*>(w + L.b_off);
  float* Sws = reinterpret_cast<float*>(w + L.s_off);
  const int D = p.D;
  const size_t mat = (size_t)D * D * sizeof(float);
  // sequential and split forms are the same three stages here
  const int rc = states<TIn>(p, Mws, bws, Sws, w, L, p.mode == 1, st);
  if (rc != kOk) return rc;

  const size_t osmem = mat + kOutRows * D * sizeof(float);
  if (cudaFuncSetAttribute(readout_kernel<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)osmem) !=
      cudaSuccess)
    return kCuda;
  {
    ProfScope po(st, "simt_readout");
    readout_kernel<TIn><<<dim3((unsigned)p.BHT(), (p.S + kOutRows - 1) / kOutRows), kThreads, osmem, st>>>(
        static_cast<const TIn*>(p.q), Sws, static_cast<TIn*>(p.out), p.S, D, p.out_scale, p.variant);
  }
  if (cudaGetLastError() != cudaSuccess) return kCuda;
  return kOk;
}

}  // namespace

int launch_chunk_fold(const float* A, const float* b, long long chunk_stride, int ld, int nchunks,
                      const float* state_in, float* starts, float* x_out, float* A_out, float* b_out, long long BH,
                      int D, cudaStream_t st, size_t a_span, size_t b_span, size_t starts_span) {
  const int smem = (D * (D + 1) + D * 16) * (int)sizeof(float);
  if (cudaFuncSetAttribute(chunk_fold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return kCuda;
  FoldArgs fa{A, b, chunk_stride, ld, nchunks, D, state_in, starts, x_out, A_out, b_out, device_status_word(),
              a_span, b_span, starts_span};
  const long long ctas = BH * (D / 16) * (A_out ? 2 : 1);
  ProfScope ps(st, A_out ? "chunk_fold_summary" : "chunk_fold");
  chunk_fold_kernel<<<(unsigned)ctas, kFoldThreads, smem, st>>>(fa);
  return cudaGetLastError() == cudaSuccess ? kOk : kCuda;
}

size_t simt_workspace_bytes(const Problem& p, int mode) { return simt_layout(p, mode).total; }

int simt_chunk_maps(const Problem& p, void* ws, float** maps, int* nchunks, cudaStream_t st) {
  const SimtLayout L = simt_layout(p, GDN_MODE_PREFIX);
  char* w = static_cast<char*>(ws);
  float* Mws = reinterpret_cast<float*>(w + L.m_off);
  float* bws = reinterpret_cast<float*>(w + L.b_off);
  const int D = p.D;
  const size_t mat = (size_t)D * D * sizeof(float);
  {
    ProfScope pg(st, "simt_gram");
    if (p.dtype == GDN_F32)
      gram_kernel<float><<<dim3((unsigned)p.BHT(), 2), kThreads, 2 * kTok * D * sizeof(float), st>>>(
          static_cast<const float*>(p.k), static_cast<const float*>(p.v), p.beta, Mws, bws, p.S, D, p.key_scale,
          p.gate_logits, p.variant);
    else
      gram_kernel<__nv_bfloat16><<<dim3((unsigned)p.BHT(), 2), kThreads, 2 * kTok * D * sizeof(float), st>>>(
          static_cast<const __nv_bfloat16*>(p.k), static_cast<const __nv_bfloat16*>(p.v), p.beta, Mws, bws, p.S, D,
          p.key_scale, p.gate_logits, p.variant);
  }
  if (cudaGetLastError() != cudaSuccess) return kCuda;
  float* mp = reinterpret_cast<float*>(w + L.maps_off);
  const size_t csmem = 3 * mat;
  if (cudaFuncSetAttribute(compose_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csmem) != cudaSuccess)
    return kCuda;
  {
    ProfScope pc(st, "simt_compose");
    compose_kernel<<<(unsigned)(p.BH() * L.nchunks), kThreads, csmem, st>>>(Mws, bws, p.g, mp, p.T, D, L.nchunks,
                                                                             p.gate_logits, p.variant);
  }
  if (cudaGetLastError() != cudaSuccess) return kCuda;
  *maps = mp;
  *nchunks = L.nchunks;
  return kOk;
}

int simt_forward(const Problem& p, void* ws, cudaStream_t st) {
  if (p.dtype == 0) return run<float>(p, ws, st);
  return run<__nv_bfloat16>(p, ws, st);
}

int simt_states(const Problem& p, float* Mws, float* bws, float* Sws, cudaStream_t st) {
  const SimtLayout L{};  // the sequential scan uses no chunk buffers
  if (p.dtype == 0) return states<float>(p, Mws, bws, Sws, nullptr, L, false, st);
  return states<__nv_bfloat16>(p, Mws, bws, Sws, nullptr, L, false, st);
}

}  // namespace gdn
