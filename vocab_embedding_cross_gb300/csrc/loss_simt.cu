// fp32 cross-entropy path (SIMT FMA, fp32 exp/log).
//
// Used when the problem is stored in fp32: tensor-core tf32 would not keep the
// fp32 results within 1e-5 of the exact values, so this path keeps every
// product and sum in fp32 FMA. Same method as the bf16 path ("Vocabulary
// shards: look up locally and normalize globally", paragraphs 3-4): per work
// unit (a column range inside one shard) a running maximum and sum of exp, the
// target logit from its owning unit, and for the backward
// G = (p - onehot) * g / N_valid over column chunks followed by two GEMMs.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"

namespace vce {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;

// z tile [64 tokens x 64 columns] = h[m0.., :] . W[v0.., :]^T into acc; rows
// >= T and columns >= vlim read as zero.
__device__ __forceinline__ void z_tile(const float* __restrict__ h, const float* __restrict__ W, int T, int H,
                                       int m0, int64_t vt0, int64_t vlim, float (&acc)[4][4],
                                       float (*hs)[TM + 4], float (*ws)[TN + 4]) {
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  for (int k0 = 0; k0 < H; k0 += TK) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int idx = tid + 256 * q, r = idx >> 4, kk = idx & 15;
      const int gr = m0 + r, gk = k0 + kk;
      hs[kk][r] = (gr < T && gk < H) ? h[static_cast<int64_t>(gr) * H + gk] : 0.0f;
      const int64_t v = vt0 + r;
      ws[kk][r] = (v < vlim && gk < H) ? W[v * H + gk] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = hs[kk][4 * ty + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = ws[kk][4 * tx + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
}

__device__ __forceinline__ float hmax16(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float hsum16(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// grid (ceil(T/64), n_units): running max / sum of exp of one unit for 64 tokens.
__global__ void __launch_bounds__(256) simt_fwd_kernel(ProbDev pd, UnitGrid ug, const float* __restrict__ h,
                                                       const float* __restrict__ W,
                                                       const int64_t* __restrict__ targets, float2* __restrict__ part,
                                                       float* __restrict__ ztgt, int32_t* merge_ctr) {
  __shared__ float hs[TK][TM + 4];
  if (merge_ctr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *merge_ctr = 0;   // for the merge after it
  __shared__ float ws[TK][TN + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.x * TM;
  const int u = blockIdx.y;
  const int k_sh = u / ug.ups, j_u = u - k_sh * ug.ups;
  const int64_t lo = shard_lo(k_sh, pd.Vp, pd.S), hi = shard_lo(k_sh + 1, pd.Vp, pd.S);
  const int64_t vb = lo + static_cast<int64_t>(j_u) * ug.uw;
  const int64_t ve = vb + ug.uw < hi ? vb + ug.uw : hi;
  const int64_t vlim = ve < pd.V_real ? ve : pd.V_real;
  float m_run[4], s_run[4];
  int64_t y[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m_run[i] = -INFINITY;
    s_run[i] = 0.0f;
    const int r = m0 + 4 * ty + i;
    y[i] = r < pd.T ? targets[r] : -1;
  }
  for (int64_t vt0 = vb; vt0 < vlim; vt0 += TN) {
    float acc[4][4];
    z_tile(h, W, pd.T, pd.H, m0, vt0, vlim, acc, hs, ws);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float lm = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (vt0 + 4 * tx + j < vlim) lm = fmaxf(lm, acc[i][j]);
      const float tmax = hmax16(lm);
      const float mn = fmaxf(m_run[i], tmax);
      if (mn != -INFINITY) {
        float ls = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (vt0 + 4 * tx + j < vlim) ls += expf(acc[i][j] - mn);
        ls = hsum16(ls);
        s_run[i] = s_run[i] * expf(m_run[i] - mn) + ls;
        m_run[i] = mn;
      }
      const int r = m0 + 4 * ty + i;
      const int64_t c0 = vt0 + 4 * tx;
      if (r < pd.T && y[i] >= c0 && y[i] < c0 + 4 && y[i] < vlim) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (c0 + j == y[i]) ztgt[r] = acc[i][j];
      }
    }
  }
  if (tx == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = m0 + 4 * ty + i;
      if (r < pd.T) part[static_cast<int64_t>(r) * ug.n_units + u] = make_float2(m_run[i], s_run[i]);
    }
  }
}

// (max, argmax) pair reduction over the 16 lanes holding one row: larger
// value first, lower column on a tie (columns < 0 mean "none").
__device__ __forceinline__ void hargmax16(float& v, int32_t& c) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int32_t c2 = __shfl_xor_sync(0xffffffffu, c, o);
    if (c2 >= 0 && (c < 0 || v2 > v || (v2 == v && c2 < c))) {
      v = v2;
      c = c2;
    }
  }
}

// grid (ceil(T/64), n_units): largest real logit of one unit and its lowest
// column, for 64 tokens (greedy decoding over the sharded head).
__global__ void __launch_bounds__(256) simt_argmax_kernel(ProbDev pd, UnitGrid ug, const float* __restrict__ h,
                                                          const float* __restrict__ W, float2* __restrict__ part) {
  __shared__ float hs[TK][TM + 4];
  __shared__ float ws[TK][TN + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.x * TM;
  const int u = blockIdx.y;
  const int k_sh = u / ug.ups, j_u = u - k_sh * ug.ups;
  const int64_t lo = shard_lo(k_sh, pd.Vp, pd.S), hi = shard_lo(k_sh + 1, pd.Vp, pd.S);
  const int64_t vb = lo + static_cast<int64_t>(j_u) * ug.uw;
  const int64_t ve = vb + ug.uw < hi ? vb + ug.uw : hi;
  const int64_t vlim = ve < pd.V_real ? ve : pd.V_real;
  float m_run[4];
  int32_t c_run[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m_run[i] = -INFINITY;
    c_run[i] = -1;
  }
  for (int64_t vt0 = vb; vt0 < vlim; vt0 += TN) {
    float acc[4][4];
    z_tile(h, W, pd.T, pd.H, m0, vt0, vlim, acc, hs, ws);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float bv = -INFINITY;
      int32_t bc = -1;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t v = vt0 + 4 * tx + j;
        if (v < vlim && (bc < 0 || acc[i][j] > bv)) {
          bv = acc[i][j];
          bc = static_cast<int32_t>(v);
        }
      }
      hargmax16(bv, bc);
      if (bc >= 0 && (c_run[i] < 0 || bv > m_run[i])) {   // later tiles hold higher columns
        m_run[i] = bv;
        c_run[i] = bc;
      }
    }
  }
  if (tx == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = m0 + 4 * ty + i;
      if (r < pd.T) part[static_cast<int64_t>(r) * ug.n_units + u] = make_float2(m_run[i], __int_as_float(c_run[i]));
    }
  }
}

// grid (ceil(T/64), ceil(vc/64)): G[t, v - v0] = (exp(z - lse) - [v == y]) * g / N_valid.
__global__ void __launch_bounds__(256) simt_grad_kernel(ProbDev pd, const float* __restrict__ h,
                                                        const float* __restrict__ W,
                                                        const int64_t* __restrict__ targets,
                                                        const float* __restrict__ lse,
                                                        const int32_t* __restrict__ n_valid, float g, int v0, int vc,
                                                        float* __restrict__ G) {
  __shared__ float hs[TK][TM + 4];
  __shared__ float ws[TK][TN + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.x * TM;
  const int64_t vt0 = v0 + static_cast<int64_t>(blockIdx.y) * TN;
  const int64_t vend = static_cast<int64_t>(v0) + vc;
  const int64_t vlim = vend < pd.V_real ? vend : pd.V_real;
  float acc[4][4];
  z_tile(h, W, pd.T, pd.H, m0, vt0, vlim, acc, hs, ws);
  const int nv = n_valid[0];
  const float scale = nv > 0 ? g / static_cast<float>(nv) : 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = m0 + 4 * ty + i;
    if (r >= pd.T) continue;
    const int64_t y = targets[r];
    const bool row_ok = (y >= 0) && (y < pd.V_real);
    const float l = lse[r];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t v = vt0 + 4 * tx + j;
      if (v >= vend) continue;
      float gv = 0.0f;
      if (row_ok && v < pd.V_real) {
        const float p = expf(acc[i][j] - l);
        gv = (p - (v == y ? 1.0f : 0.0f)) * scale;
      }
      G[static_cast<int64_t>(r) * vc + (v - v0)] = gv;
    }
  }
}

__global__ void __launch_bounds__(256) sgemm_kernel(int M, int N, int K, const float* __restrict__ A, int64_t sam,
                                                    int64_t sak, const float* __restrict__ B, int64_t sbk,
                                                    int64_t sbn, float* __restrict__ C, int64_t ldc, int beta) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  for (int k0 = 0; k0 < K; k0 += TK) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int idx = tid + 256 * q;
      {
        const int r = idx >> 4, kk = idx & 15;
        const int gm = m0 + r, gk = k0 + kk;
        As[kk][r] = (gm < M && gk < K) ? A[gm * sam + gk * sak] : 0.0f;
      }
      {
        const int kk = idx >> 6, c = idx & 63;
        const int gk = k0 + kk, gn = n0 + c;
        Bs[kk][c] = (gk < K && gn < N) ? B[gk * sbk + gn * sbn] : 0.0f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][4 * ty + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][4 * tx + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + 4 * ty + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + 4 * tx + j;
      if (gn >= N) continue;
      float* c = C + gm * ldc + gn;
      *c = beta ? (*c + acc[i][j]) : acc[i][j];
    }
  }
}

}  // namespace

cudaError_t launch_simt_fwd(const ProbDev& pd, const UnitGrid& ug, const float* h, const float* W,
                            const int64_t* targets, float2* part, float* ztgt, int32_t* merge_ctr, cudaStream_t st) {
  dim3 grid(static_cast<unsigned>(ceil_div(pd.T, TM)), static_cast<unsigned>(ug.n_units));
  simt_fwd_kernel<<<grid, 256, 0, st>>>(pd, ug, h, W, targets, part, ztgt, merge_ctr);
  note_launch(VCE_K_SIMT_FWD, st);
  return cudaGetLastError();
}

cudaError_t launch_simt_argmax(const ProbDev& pd, const UnitGrid& ug, const float* h, const float* W, float2* part,
                               cudaStream_t st) {
  dim3 grid(static_cast<unsigned>(ceil_div(pd.T, TM)), static_cast<unsigned>(ug.n_units));
  simt_argmax_kernel<<<grid, 256, 0, st>>>(pd, ug, h, W, part);
  note_launch(VCE_K_SIMT_ARGMAX, st);
  return cudaGetLastError();
}

cudaError_t launch_simt_grad(const ProbDev& pd, const float* h, const float* W, const int64_t* targets,
                             const float* lse, const int32_t* n_valid, float g, int v0, int vc, float* G,
                             cudaStream_t st) {
  dim3 grid(static_cast<unsigned>(ceil_div(pd.T, TM)), static_cast<unsigned>(ceil_div(vc, TN)));
  simt_grad_kernel<<<grid, 256, 0, st>>>(pd, h, W, targets, lse, n_valid, g, v0, vc, G);
  note_launch(VCE_K_SIMT_GRAD, st);
  return cudaGetLastError();
}

cudaError_t launch_sgemm(int M, int N, int K, const float* A, int64_t sam, int64_t sak, const float* B,
                         int64_t sbk, int64_t sbn, float* C, int64_t ldc, int beta, cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(ceil_div(N, TN)), static_cast<unsigned>(ceil_div(M, TM)));
  sgemm_kernel<<<grid, 256, 0, st>>>(M, N, K, A, sam, sak, B, sbk, sbn, C, ldc, beta);
  note_launch(VCE_K_SGEMM, st);
  return cudaGetLastError();
}

}  // namespace vce
