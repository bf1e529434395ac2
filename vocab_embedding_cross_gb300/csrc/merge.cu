// Merge of the forward partials into one maximum and one denominator per token.
//
// "Vocabulary shards: look up locally and normalize globally", paragraphs 3-4:
// the loss needs the global maximum over the valid classes of every shard and
// one global denominator; the target logit comes from its unique owner. The
// forward kernels leave, for every (token, work unit) with a unit lying inside
// one shard, the unit's maximum m_u and its sum s_u = sum exp(z - m_u). Here
// they are combined with the rescaling rule
//     (m, s) + (m', s') = (M, s*exp(m - M) + s'*exp(m' - M)),  M = max(m, m'),
// which equals the page's "subtract the global maximum, sum, combine" schedule
// (paragraph 4: fused implementations may use other reduction schedules).
// The loss is then averaged once over the valid tokens ("Sequence-parallel
// normalization", paragraph 3) with a fixed-order, deterministic reduction,
// by the last merge block to finish.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"

namespace vce {
namespace {

constexpr int kMergeWarps = 8;

__device__ __forceinline__ void combine(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  if (m2 > m) {
    s = s * expf(m - m2) + s2;
    m = m2;
  } else {
    s = s + s2 * expf(m2 - m);
  }
}

// The last block to finish (an atomic counter, zeroed by the forward kernel
// before this one) also takes the mean: the block partials are added in block
// order, each thread a contiguous range in double, then a fixed tree, so the
// result does not depend on which block comes last.
__global__ void __launch_bounds__(kMergeWarps * 32)
    merge_kernel(ProbDev pd, UnitGrid ug, const int64_t* __restrict__ targets, const float2* __restrict__ part,
                 const float* __restrict__ ztgt, float* __restrict__ lse, float* __restrict__ token_loss,
                 int32_t* __restrict__ target_owner, int32_t* __restrict__ max_owner, float* block_sums,
                 int32_t* counter, float* __restrict__ loss, int32_t* status) {
  __shared__ float sh_loss[kMergeWarps];
  __shared__ int sh_cnt[kMergeWarps];
  __shared__ double sh_a[kMergeWarps * 32];
  __shared__ long long sh_c[kMergeWarps * 32];
  __shared__ int s_last;
  grid_dep_launch();   // launched as a dependent launch: wait for the kernel before
  grid_dep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kMergeWarps + warp;
  float my_loss = 0.0f;
  int my_cnt = 0;
  if (t < pd.T) {
    float m = -INFINITY, s = 0.0f, bm = -INFINITY;
    int bu = 0x7FFFFFFF;
    const float2* row = part + t * ug.n_units;
    for (int u = lane; u < ug.n_units; u += 32) {
      const float2 ms = row[u];
      combine(m, s, ms.x, ms.y);
      if (ms.x > bm) {          // units ascend with the lane, so the first maximum wins
        bm = ms.x;
        bu = u;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      const float bm2 = __shfl_xor_sync(0xffffffffu, bm, o);
      const int bu2 = __shfl_xor_sync(0xffffffffu, bu, o);
      // combine in lane order so every lane ends with the same bits
      if ((lane & o) == 0) {
        combine(m, s, m2, s2);
      } else {
        float mm = m2, ss = s2;
        combine(mm, ss, m, s);
        m = mm;
        s = ss;
      }
      if (bm2 > bm || (bm2 == bm && bu2 < bu)) {
        bm = bm2;
        bu = bu2;
      }
    }
    if (lane == 0) {
      const float l = m + logf(s);
      lse[t] = l;
      const int64_t y = targets[t];
      const bool valid = (y >= 0) && (y < pd.V_real);
      if (!valid && y != pd.ignore_index && status) atomicCAS(status, 0, static_cast<int>(VCE_ERR_BAD_INDEX));
      const float tl = valid ? (l - ztgt[t]) : 0.0f;
      if (token_loss) token_loss[t] = tl;
      if (target_owner) target_owner[t] = valid ? shard_of(y, pd.Vp, pd.S) : -1;
      if (max_owner) max_owner[t] = (bu < ug.n_units) ? bu / ug.ups : -1;
      my_loss = tl;
      my_cnt = valid ? 1 : 0;
    }
  }
  if (lane == 0) {
    sh_loss[warp] = my_loss;
    sh_cnt[warp] = my_cnt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.0f;
    int c = 0;
    for (int w = 0; w < kMergeWarps; ++w) {
      a += sh_loss[w];
      c += sh_cnt[w];
    }
    block_sums[2 * blockIdx.x] = a;
    block_sums[2 * blockIdx.x + 1] = __int_as_float(c);
    __threadfence();
    s_last = atomicAdd(counter, 1) == static_cast<int>(gridDim.x) - 1 ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  constexpr int kT = kMergeWarps * 32;
  const int nblocks = static_cast<int>(gridDim.x);
  const int per = (nblocks + kT - 1) / kT;
  const int b0 = static_cast<int>(threadIdx.x) * per;
  double a = 0.0;
  long long c = 0;
  for (int b = b0; b < min(nblocks, b0 + per); ++b) {
    a += static_cast<double>(__ldcg(block_sums + 2 * b));
    c += __float_as_int(__ldcg(block_sums + 2 * b + 1));
  }
  sh_a[threadIdx.x] = a;
  sh_c[threadIdx.x] = c;
  __syncthreads();
  for (int o = kT / 2; o > 0; o >>= 1) {
    if (static_cast<int>(threadIdx.x) < o) {
      sh_a[threadIdx.x] += sh_a[threadIdx.x + o];
      sh_c[threadIdx.x] += sh_c[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) loss[0] = sh_c[0] > 0 ? static_cast<float>(sh_a[0] / static_cast<double>(sh_c[0])) : 0.0f;
}

__global__ void __launch_bounds__(1024) count_valid_kernel(ProbDev pd, const int64_t* __restrict__ targets,
                                                           int32_t* n_valid, int32_t* status) {
  grid_dep_launch();   // launched as a dependent launch: wait for the kernel before
  grid_dep_wait();
  __shared__ int sh[32];
  int c = 0;
  bool bad = false;
  for (int64_t t = threadIdx.x; t < pd.T; t += blockDim.x) {
    const int64_t y = targets[t];
    const bool v = (y >= 0) && (y < pd.V_real);
    c += v ? 1 : 0;
    bad |= (!v && y != pd.ignore_index);
  }
  if (bad && status) atomicCAS(status, 0, static_cast<int>(VCE_ERR_BAD_INDEX));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int s = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) s += sh[w];
    n_valid[0] = s;
  }
}

// Greedy decoding: the units' (max, column) pairs of one token are merged to
// the global maximum and its lowest column; the owner is the shard of that
// column ("Tensor Parallelism (TP)", on-device sampling: the argmax is found
// across the sharded logits without gathering them).
__global__ void __launch_bounds__(kMergeWarps * 32)
    argmax_merge_kernel(ProbDev pd, UnitGrid ug, const float2* __restrict__ part, int64_t* __restrict__ argmax,
                        float* __restrict__ max_logit, int32_t* __restrict__ owner) {
  grid_dep_launch();   // launched as a dependent launch: wait for the kernel before
  grid_dep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kMergeWarps + warp;
  if (t >= pd.T) return;
  float m = -INFINITY;
  int32_t c = -1;
  const float2* row = part + t * ug.n_units;
  for (int u = lane; u < ug.n_units; u += 32) {
    const float2 mc = row[u];
    const int32_t c2 = __float_as_int(mc.y);
    if (c2 >= 0 && (c < 0 || mc.x > m || (mc.x == m && c2 < c))) {
      m = mc.x;
      c = c2;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const int32_t c2 = __shfl_xor_sync(0xffffffffu, c, o);
    if (c2 >= 0 && (c < 0 || m2 > m || (m2 == m && c2 < c))) {
      m = m2;
      c = c2;
    }
  }
  if (lane == 0) {
    argmax[t] = c;
    if (max_logit) max_logit[t] = m;
    if (owner) owner[t] = c >= 0 ? shard_of(c, pd.Vp, pd.S) : -1;
  }
}

// dH in bf16: out[i] = bf16(acc[i]) or, accumulating, bf16(float(out[i]) + acc[i]),
// rounded to nearest even once. Four elements per step (8-byte stores).
__global__ void __launch_bounds__(256) dh_to_bf16_kernel(const float4* __restrict__ acc, uint2* __restrict__ out,
                                                         int64_t n4, int accumulate) {
  grid_dep_launch();   // launched as a dependent launch: wait for the kernel before
  grid_dep_wait();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 a = __ldcs(acc + i);
    if (accumulate) {
      const uint2 o = out[i];
      a.x = a.x + __uint_as_float(o.x << 16);
      a.y = a.y + __uint_as_float(o.x & 0xFFFF0000u);
      a.z = a.z + __uint_as_float(o.y << 16);
      a.w = a.w + __uint_as_float(o.y & 0xFFFF0000u);
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y), hi = __floats2bfloat162_rn(a.z, a.w);
    out[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
  }
}

}  // namespace

int merge_blocks(int64_t T) { return static_cast<int>(ceil_div(T, kMergeWarps)); }

cudaError_t launch_dh_to_bf16(const float* acc, void* out, int64_t n, bool accumulate, cudaStream_t st) {
  const int64_t n4 = n / 4;
  if (n4 == 0) return cudaSuccess;
  const DevInfo di = current_device_info();
  int64_t blocks = ceil_div(n4, 256 * 4);
  const int64_t cap = static_cast<int64_t>(di.num_sms) * 8;
  if (blocks > cap) blocks = cap;
  const cudaError_t e = launch_dependent(dh_to_bf16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st,
                                         reinterpret_cast<const float4*>(acc), static_cast<uint2*>(out), n4,
                                         accumulate ? 1 : 0);
  note_launch(VCE_K_DH_BF16, st);
  return e;
}

cudaError_t launch_argmax_merge(const ProbDev& pd, const UnitGrid& ug, const float2* part, int64_t* argmax,
                                float* max_logit, int32_t* owner, cudaStream_t st) {
  const cudaError_t e = launch_dependent(argmax_merge_kernel, dim3(merge_blocks(pd.T)), dim3(kMergeWarps * 32), 0, st,
                                         pd, ug, part, argmax, max_logit, owner);
  note_launch(VCE_K_ARGMAX_MERGE, st);
  return e;
}

cudaError_t launch_merge(const ProbDev& pd, const UnitGrid& ug, const int64_t* targets, const float2* part,
                         const float* ztgt, float* lse, float* token_loss, int32_t* target_owner,
                         int32_t* max_owner, float* block_sums, int32_t* counter, float* loss, int32_t* status,
                         cudaStream_t st) {
  const int nb = merge_blocks(pd.T);
  const cudaError_t e = launch_dependent(merge_kernel, dim3(nb), dim3(kMergeWarps * 32), 0, st, pd, ug, targets, part,
                                         ztgt, lse, token_loss, target_owner, max_owner, block_sums, counter, loss,
                                         status);
  note_launch(VCE_K_MERGE, st);
  return e;
}

cudaError_t launch_count_valid(const ProbDev& pd, const int64_t* targets, int32_t* n_valid, int32_t* status,
                               cudaStream_t st) {
  const cudaError_t e = launch_dependent(count_valid_kernel, dim3(1), dim3(1024), 0, st, pd, targets, n_valid, status);
  note_launch(VCE_K_COUNT_VALID, st);
  return e;
}

}  // namespace vce
