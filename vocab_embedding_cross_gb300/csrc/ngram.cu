// Hashed n-gram input embeddings ("Sampled Softmax with Over-Tokenized
// Transformer", Setup and its loss listing: the input embedding of every token
// gains the hashed 2-gram and 3-gram embeddings that end at it).
//
// Hash: the n-gram (x[t-n+1], ..., x[t]) of the input ids x, read as a number
// in base V (x[t] the lowest digit), reduced mod the table's row count M:
//     idx_n(t) = (sum_j x[t-j] * V^j) mod M,   j = 0 .. n-1,
// evaluated by Horner's rule with a reduction after every step, so every
// intermediate stays below 2^62 (M, V < 2^31). Positions with fewer than n-1
// earlier tokens in their sequence (sequences of seq_len tokens) and n-grams
// holding an invalid id (outside [0, V)) have no n-gram: index -1, zero row,
// no gradient.
//
// Forward: E[t] = ((W[x_t] + T2[idx_2(t)]) + T3[idx_3(t)]) in fp32, a missing
// term read as +0, rounded once to the storage type (round to nearest even).
// Backward: each table receives the deterministic embedding backward of dE
// with its own index list (sorted (index, t), runs of 32, fp32, one rounding).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace vce {
namespace {

__device__ __forceinline__ int64_t ngram_index(const int64_t* __restrict__ ids, int64_t t, int n, int64_t V,
                                               int64_t M, int64_t seq_len) {
  if (M <= 0) return -1;
  const int64_t pos = seq_len > 0 ? t % seq_len : t;
  if (pos < n - 1) return -1;
  const uint64_t vm = static_cast<uint64_t>(V % M);
  uint64_t hsh = 0;
  for (int j = n - 1; j >= 0; --j) {   // oldest token first: Horner in base V
    const int64_t x = ids[t - j];
    if (x < 0 || x >= V) return -1;
    hsh = (hsh * vm + static_cast<uint64_t>(x % M)) % static_cast<uint64_t>(M);
  }
  return static_cast<int64_t>(hsh);
}

__global__ void __launch_bounds__(256) ngram_hash_kernel(const int64_t* __restrict__ ids, int64_t T, int n,
                                                         int64_t V, int64_t M, int64_t seq_len,
                                                         int64_t* __restrict__ out) {
  for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < T;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[t] = ngram_index(ids, t, n, V, M, seq_len);
}

// Both tables' row indices in one launch (the backward's plan needs both).
__global__ void __launch_bounds__(256) ngram_hash_pair_kernel(const int64_t* __restrict__ ids, int64_t T, int64_t V,
                                                              int64_t M2, int64_t M3, int64_t seq_len,
                                                              int64_t* __restrict__ out2, int64_t* __restrict__ out3) {
  for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < T;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    out2[t] = ngram_index(ids, t, 2, V, M2, seq_len);
    out3[t] = ngram_index(ids, t, 3, V, M3, seq_len);
  }
}

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = acc[2 * i] + __uint_as_float(w[i] << 16);
    acc[2 * i + 1] = acc[2 * i + 1] + __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t bf16_rne_pair(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// One warp per token: 16-byte lanes over the row, three gathered rows summed
// in fp32 and stored once.
template <bool BF16>
__global__ void __launch_bounds__(256)
    ngram_embed_fwd_kernel(const int64_t* __restrict__ ids, const uint4* __restrict__ W,
                           const uint4* __restrict__ T2, const uint4* __restrict__ T3, uint4* __restrict__ E,
                           int64_t T, int64_t V, int64_t M2, int64_t M3, int64_t seq_len, int row_vecs) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (t >= T) return;
  const int64_t x = ids[t];
  const int64_t i1 = (x >= 0 && x < V) ? x : -1;
  const int64_t i2 = ngram_index(ids, t, 2, V, M2, seq_len);
  const int64_t i3 = ngram_index(ids, t, 3, V, M3, seq_len);
  const uint4* r1 = i1 >= 0 ? W + i1 * row_vecs : nullptr;
  const uint4* r2 = i2 >= 0 ? T2 + i2 * row_vecs : nullptr;
  const uint4* r3 = i3 >= 0 ? T3 + i3 * row_vecs : nullptr;
  uint4* dst = E + t * row_vecs;
  for (int i = lane; i < row_vecs; i += 32) {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    const uint4 a = r1 ? __ldg(r1 + i) : z;
    const uint4 b = r2 ? __ldg(r2 + i) : z;
    const uint4 c = r3 ? __ldg(r3 + i) : z;
    if constexpr (BF16) {
      float acc[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
      // (0 + w) is w exactly, except -0 + 0 = +0: the same rule as a missing term.
      add_bf16x8(acc, a);
      add_bf16x8(acc, b);
      add_bf16x8(acc, c);
      dst[i] = make_uint4(bf16_rne_pair(acc[0], acc[1]), bf16_rne_pair(acc[2], acc[3]),
                          bf16_rne_pair(acc[4], acc[5]), bf16_rne_pair(acc[6], acc[7]));
    } else {
      float4 o;
      o.x = ((0.0f + __uint_as_float(a.x)) + __uint_as_float(b.x)) + __uint_as_float(c.x);
      o.y = ((0.0f + __uint_as_float(a.y)) + __uint_as_float(b.y)) + __uint_as_float(c.y);
      o.z = ((0.0f + __uint_as_float(a.z)) + __uint_as_float(b.z)) + __uint_as_float(c.z);
      o.w = ((0.0f + __uint_as_float(a.w)) + __uint_as_float(b.w)) + __uint_as_float(c.w);
      dst[i] = *reinterpret_cast<const uint4*>(&o);
    }
  }
}

}  // namespace

cudaError_t launch_ngram_hash(const int64_t* ids, int64_t T, int n, int64_t V, int64_t M, int64_t seq_len,
                              int64_t* out, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const DevInfo di = current_device_info();
  int64_t blocks = ceil_div(T, 256);
  if (blocks > di.num_sms * 8) blocks = di.num_sms * 8;
  ngram_hash_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(ids, T, n, V, M, seq_len, out);
  note_launch(VCE_K_NGRAM_HASH, st);
  return cudaGetLastError();
}

cudaError_t launch_ngram_hash_pair(const int64_t* ids, int64_t T, int64_t V, int64_t M2, int64_t M3, int64_t seq_len,
                                   int64_t* out2, int64_t* out3, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const DevInfo di = current_device_info();
  int64_t blocks = ceil_div(T, 256);
  if (blocks > di.num_sms * 8) blocks = di.num_sms * 8;
  ngram_hash_pair_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(ids, T, V, M2, M3, seq_len, out2, out3);
  note_launch(VCE_K_NGRAM_HASH, st);
  return cudaGetLastError();
}

cudaError_t launch_ngram_embed_fwd(const vce_problem& p, const int64_t* ids, const void* W, const void* T2,
                                   int64_t M2, const void* T3, int64_t M3, int64_t seq_len, void* E,
                                   cudaStream_t st) {
  if (p.T == 0) return cudaSuccess;
  const int esize = p.dtype == VCE_BF16 ? 2 : 4;
  const int row_vecs = static_cast<int>(p.H * esize / 16);
  const unsigned blocks = static_cast<unsigned>(ceil_div(p.T, 8));
  if (p.dtype == VCE_BF16)
    ngram_embed_fwd_kernel<true><<<blocks, 256, 0, st>>>(
        ids, static_cast<const uint4*>(W), static_cast<const uint4*>(T2), static_cast<const uint4*>(T3),
        static_cast<uint4*>(E), p.T, p.V_real, M2, M3, seq_len, row_vecs);
  else
    ngram_embed_fwd_kernel<false><<<blocks, 256, 0, st>>>(
        ids, static_cast<const uint4*>(W), static_cast<const uint4*>(T2), static_cast<const uint4*>(T3),
        static_cast<uint4*>(E), p.T, p.V_real, M2, M3, seq_len, row_vecs);
  note_launch(VCE_K_NGRAM_FWD, st);
  return cudaGetLastError();
}

}  // namespace vce
