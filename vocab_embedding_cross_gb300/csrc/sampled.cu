// Candidate list of the sampled softmax ("Sampled Softmax with Over-Tokenized
// Transformer", Setup: the loss scores the batch's targets plus random
// negatives, P tokens in all, and takes the cross-entropy at each target's
// position in that list).
//
// One CTA: mark the valid targets in a dense byte map over the vocabulary,
// scan the map to list the distinct targets in ascending order (and each
// target's rank), then take negatives in draw order from the caller's distinct
// uniform draws, skipping targets, until P entries. The loss itself then runs
// on the existing kernels: gather W[cand] (embedding lookup), cross-entropy
// over the P gathered rows, and the candidate rows of dW scattered back with
// the embedding backward.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace vce {
namespace {

constexpr int kThreads = 1024;

__device__ __forceinline__ int cta_excl_scan(int v, int* sh_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int w = sh_warp[lane];
    int s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    sh_warp[lane] = s - w;
    if (lane == 31) sh_warp[32] = s;
  }
  __syncthreads();
  const int res = sh_warp[warp] + x - v;
  *total = sh_warp[32];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(kThreads, 1)
    sampled_cand_kernel(const int64_t* __restrict__ targets, int64_t T, int64_t V_real, int64_t ignore_index,
                        const int64_t* __restrict__ draws, int64_t n_draws, int64_t P, uint8_t* mark, int32_t* rank,
                        int64_t* cand, int64_t* pos, int32_t* n_unique, int32_t* status) {
  __shared__ int sh_warp[33];
  const int tid = threadIdx.x;
  for (int64_t v = tid; v < V_real; v += kThreads) mark[v] = 0;
  __syncthreads();
  bool bad = false;
  for (int64_t t = tid; t < T; t += kThreads) {
    const int64_t y = targets[t];
    if (y >= 0 && y < V_real)
      mark[y] = 1;
    else if (y != ignore_index)
      bad = true;
  }
  if (bad && status) atomicCAS(status, 0, static_cast<int>(VCE_ERR_BAD_INDEX));
  __syncthreads();

  // Distinct targets in ascending order: scan of the map (contiguous ranges
  // of the vocabulary per thread).
  const int64_t per = (V_real + kThreads - 1) / kThreads;
  const int64_t v0 = tid * per, v1 = v0 + per < V_real ? v0 + per : V_real;
  int cnt = 0;
  for (int64_t v = v0; v < v1; ++v) cnt += mark[v];
  int nu;
  int r = cta_excl_scan(cnt, sh_warp, &nu);
  for (int64_t v = v0; v < v1; ++v) {
    if (mark[v]) {
      rank[v] = r;
      if (r < P) cand[r] = v;
      ++r;
    }
  }
  if (tid == 0) n_unique[0] = nu;
  __syncthreads();
  if (nu > P) {   // more distinct targets than candidates: a data error
    if (tid == 0 && status) atomicCAS(status, 0, static_cast<int>(VCE_ERR_ARG));
    // Defined outputs: an empty list (id -1 gathers a zero row and is skipped
    // by the embedding backward) and every target ignored.
    for (int64_t i = tid; i < P; i += kThreads) cand[i] = -1;
    for (int64_t t = tid; t < T; t += kThreads) pos[t] = ignore_index;
    return;
  }

  // Negatives: the draws that are not targets, in draw order, until P.
  const int64_t per2 = (n_draws + kThreads - 1) / kThreads;
  const int64_t i0 = tid * per2, i1 = i0 + per2 < n_draws ? i0 + per2 : n_draws;
  int c2 = 0;
  for (int64_t i = i0; i < i1; ++i) {
    const int64_t d = draws[i];
    c2 += (d >= 0 && d < V_real && !mark[d]) ? 1 : 0;
  }
  int avail;
  int q = cta_excl_scan(c2, sh_warp, &avail);
  for (int64_t i = i0; i < i1; ++i) {
    const int64_t d = draws[i];
    if (d >= 0 && d < V_real && !mark[d]) {
      if (nu + q < P) cand[nu + q] = d;
      ++q;
    }
  }
  if (nu + avail < P) {   // too few usable draws: the tail of the list stays empty (-1)
    if (tid == 0 && status) atomicCAS(status, 0, static_cast<int>(VCE_ERR_ARG));
    for (int64_t i = nu + avail + tid; i < P; i += kThreads) cand[i] = -1;
  }
  __syncthreads();

  // Position of each target in the list (ignore_index where not a valid target).
  for (int64_t t = tid; t < T; t += kThreads) {
    const int64_t y = targets[t];
    pos[t] = (y >= 0 && y < V_real) ? static_cast<int64_t>(rank[y]) : ignore_index;
  }
}

}  // namespace

size_t sampled_ws_bytes(const vce_problem& p) {
  return align_up(static_cast<size_t>(p.V_real), kWsAlign) + align_up(sizeof(int32_t) * p.V_real, kWsAlign);
}

cudaError_t launch_sampled_candidates(const vce_problem& p, const int64_t* targets, const int64_t* draws,
                                      int64_t n_draws, int64_t P, int64_t* cand, int64_t* pos, int32_t* n_unique,
                                      void* ws, int32_t* status, cudaStream_t st) {
  uint8_t* mark = static_cast<uint8_t*>(ws);
  int32_t* rank = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + align_up(static_cast<size_t>(p.V_real), kWsAlign));
  sampled_cand_kernel<<<1, kThreads, 0, st>>>(targets, p.T, p.V_real, p.ignore_index, draws, n_draws, P, mark, rank,
                                              cand, pos, n_unique, status);
  note_launch(VCE_K_SAMPLED_CAND, st);
  return cudaGetLastError();
}

}  // namespace vce
