// Sampled softmax ("Sampled Softmax with Over-Tokenized Transformer", Setup:
// the loss scores the batch's targets plus random negatives, P tokens in all,
// and takes the cross-entropy at each target's position in that list).
//
// Candidate list: one CTA keeps a bitmap of the vocabulary and the prefix
// count of every 32-bit word in shared memory (V_real/4 bytes; in the
// workspace when that exceeds the shared-memory budget).
//   1. set the bit of every valid target;
//   2. scan the words' popcounts: the distinct targets in ascending order and
//      the rank of each (its word's prefix plus the bits below it);
//   3. pos[t] = rank of targets[t];
//   4. negatives in draw order, 4096 draws per round (four consecutive draws
//      per thread): a draw is kept when it is in [0, V_real), its bit is clear
//      (not a target, not an earlier negative) and no earlier draw of the same
//      round has the same value (a shared-memory hash table keeps the smallest
//      index per value); the kept draws are ranked by a block scan and their
//      bits set before the next round. Rounds stop once the list holds P
//      entries. The kept draws are the first occurrences of their values, so
//      the list does not depend on the round size.
// Every step is a fixed function of the inputs, so the list is deterministic.
//
// dW scatter: candidates are distinct by construction, so each candidate row
// of dW receives exactly one addition of its gradient row (one fp32 rounding).
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "internal.h"

namespace vce {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kDrawsPerThread = 4;
constexpr int kRoundDraws = kThreads * kDrawsPerThread;
constexpr int kHashSlots = 2 * kRoundDraws;
constexpr size_t kHashBytes = 2 * sizeof(int32_t) * kHashSlots;   // keys and smallest indices, dynamic shared memory
constexpr size_t kCandSmemBudget = 200 * 1024;   // hash table + bitmap + word prefixes held in shared memory up to this

// Exclusive block scan of one int per thread; *total gets the sum.
__device__ __forceinline__ int block_excl_scan(int v, int* sh_warp, int* total) {
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
    const int w = lane < kWarps ? sh_warp[lane] : 0;
    int s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kWarps) sh_warp[lane] = s - w;
    if (lane == 31) sh_warp[32] = s;
  }
  __syncthreads();
  const int res = sh_warp[warp] + x - v;
  *total = sh_warp[32];
  __syncthreads();
  return res;
}

__device__ __forceinline__ uint32_t hash_slot(int32_t d) {
  return (static_cast<uint32_t>(d) * 2654435761u) >> (32 - 13);   // 13 bits: kHashSlots = 8192
}
static_assert(kHashSlots == 8192, "hash_slot takes 13 bits");

__global__ void __launch_bounds__(kThreads, 1)
    sampled_cand_kernel(const int64_t* __restrict__ targets, int32_t T, int32_t V_real, int64_t ignore_index,
                        const int64_t* __restrict__ draws, int64_t n_draws, int32_t P, uint32_t* g_bits,
                        int32_t* g_wpre, bool use_smem, int64_t* __restrict__ cand, int64_t* __restrict__ pos,
                        int32_t* __restrict__ n_unique, int32_t* status) {
  extern __shared__ __align__(16) uint32_t dsm[];
  __shared__ int sh_warp[33];
  int32_t* hkey = reinterpret_cast<int32_t*>(dsm);
  int32_t* hidx = hkey + kHashSlots;
  const int tid = threadIdx.x;
  const int NW = (V_real + 31) >> 5;
  uint32_t* bits = use_smem ? dsm + 2 * kHashSlots : g_bits;
  int32_t* wpre = use_smem ? reinterpret_cast<int32_t*>(dsm + 2 * kHashSlots + NW) : g_wpre;

  for (int w = tid; w < NW; w += kThreads) bits[w] = 0u;
  __syncthreads();
  bool bad = false;
  // Targets kBatch per thread at a time, every load issued before the first
  // use, so a thread waits for one round trip per batch, not per target.
  constexpr int kBatch = 8;
  for (int t0 = 0; t0 < T; t0 += kThreads * kBatch) {
    int64_t yv[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int t = t0 + j * kThreads + tid;
      yv[j] = t < T ? targets[t] : ignore_index;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int64_t y = yv[j];
      if (y >= 0 && y < V_real) {
        // a hot target's bit is set once; later copies find it set and skip
        // the atomic, which would queue behind the others on one word
        const uint32_t m = 1u << (y & 31);
        if (!(bits[y >> 5] & m)) atomicOr(&bits[y >> 5], m);
      } else if (y != ignore_index) {
        bad = true;
      }
    }
  }
  if (bad && status) atomicCAS(status, 0, static_cast<int>(VCE_ERR_BAD_INDEX));
  __syncthreads();

  // Word prefixes: contiguous words per thread, block scan of their popcounts.
  const int per = (NW + kThreads - 1) / kThreads;
  const int w0 = tid * per, w1 = min(w0 + per, NW);
  int cnt = 0;
  for (int w = w0; w < w1; ++w) cnt += __popc(bits[w]);
  int nu;
  int r = block_excl_scan(cnt, sh_warp, &nu);
  for (int w = w0; w < w1; ++w) {
    wpre[w] = r;
    r += __popc(bits[w]);
  }
  if (tid == 0) n_unique[0] = nu;
  __syncthreads();

  if (nu > P) {   // more distinct targets than candidates: a data error
    if (tid == 0 && status) atomicCAS(status, 0, static_cast<int>(VCE_ERR_ARG));
    // Defined outputs: an empty list (id -1 gathers a zero row and is skipped
    // by the scatter) and every target ignored.
    for (int i = tid; i < P; i += kThreads) cand[i] = -1;
    for (int t = tid; t < T; t += kThreads) pos[t] = ignore_index;
    return;
  }
  // The distinct targets, ascending.
  for (int w = w0; w < w1; ++w) {
    uint32_t b = bits[w];
    int k = wpre[w];
    while (b) {
      const int bit = __ffs(b) - 1;
      b &= b - 1;
      cand[k++] = static_cast<int64_t>(w) * 32 + bit;
    }
  }
  // Each target's position, the targets loaded in batches as above.
  for (int t0 = 0; t0 < T; t0 += kThreads * kBatch) {
    int64_t yv[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int t = t0 + j * kThreads + tid;
      yv[j] = t < T ? targets[t] : ignore_index;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int t = t0 + j * kThreads + tid;
      const int64_t y = yv[j];
      int64_t q = ignore_index;
      if (y >= 0 && y < V_real) {
        const int w = static_cast<int>(y >> 5);
        q = wpre[w] + __popc(bits[w] & ((1u << (y & 31)) - 1u));
      }
      if (t < T) pos[t] = q;
    }
  }

  // Negatives in draw order, a round of kRoundDraws draws at a time; thread
  // tid takes the round's draws [tid * R, tid * R + R), so the block scan of
  // the threads' kept counts ranks the kept draws in draw order.
  constexpr int R = kDrawsPerThread;
  int have = nu;
  for (int64_t r0 = 0; r0 < n_draws && have < P; r0 += kRoundDraws) {
    for (int s = tid; s < kHashSlots; s += kThreads) {
      hkey[s] = -1;
      hidx[s] = INT_MAX;
    }
    __syncthreads();
    int32_t d[R];
    bool ok[R];
    uint32_t slot[R];
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int64_t i = r0 + static_cast<int64_t>(tid) * R + j;
      const int64_t d64 = i < n_draws ? draws[i] : -1;
      d[j] = static_cast<int32_t>(d64);
      ok[j] = d64 >= 0 && d64 < V_real;
    }
#pragma unroll
    for (int j = 0; j < R; ++j) {
      ok[j] = ok[j] && !((bits[d[j] >> 5] >> (d[j] & 31)) & 1u);
      slot[j] = 0;
      if (ok[j]) {
        uint32_t sl = hash_slot(d[j]);
        for (int probe = 0; probe < kHashSlots; ++probe) {   // at most kRoundDraws keys in 2*kRoundDraws slots
          const int32_t k = atomicCAS(&hkey[sl], -1, d[j]);
          if (k == -1 || k == d[j]) break;
          sl = (sl + 1) & (kHashSlots - 1);
        }
        slot[j] = sl;
        atomicMin(&hidx[sl], tid * R + j);
      }
    }
    __syncthreads();
    int mine = 0;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      ok[j] = ok[j] && hidx[slot[j]] == tid * R + j;   // the first draw of this value in the round
      mine += ok[j] ? 1 : 0;
    }
    int kept;
    int q = block_excl_scan(mine, sh_warp, &kept);
#pragma unroll
    for (int j = 0; j < R; ++j) {
      if (ok[j]) {
        if (have + q < P) cand[have + q] = d[j];
        atomicOr(&bits[d[j] >> 5], 1u << (d[j] & 31));
        ++q;
      }
    }
    have += kept;
    __syncthreads();
  }
  if (have < P) {   // too few usable draws: the tail of the list stays empty (-1)
    if (tid == 0 && status) atomicCAS(status, 0, static_cast<int>(VCE_ERR_ARG));
    for (int i = have + tid; i < P; i += kThreads) cand[i] = -1;
  }
}

// dW[cand[i], :] += dWc[i, :] for candidate rows in [0, V_real); float4 lanes.
__global__ void __launch_bounds__(256)
    sampled_scatter_kernel(const int64_t* __restrict__ cand, int32_t P, int32_t V_real, int32_t H,
                           const float4* __restrict__ dWc, float4* __restrict__ dW) {
  constexpr int U = 4;
  const int hq = H >> 2;
  const int64_t n = static_cast<int64_t>(P) * hq;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < n; base += stride * U) {
    float4 g[U], w[U];
    int64_t dst[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t e = base + u * stride;
      dst[u] = -1;
      if (e < n) {
        const int64_t row = e / hq;
        const int64_t c = cand[row];
        if (c >= 0 && c < V_real) {
          dst[u] = c * hq + (e - row * hq);
          g[u] = dWc[e];
          w[u] = dW[dst[u]];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (dst[u] >= 0) {
        w[u].x += g[u].x;
        w[u].y += g[u].y;
        w[u].z += g[u].z;
        w[u].w += g[u].w;
        dW[dst[u]] = w[u];
      }
    }
  }
}

size_t cand_table_bytes(int64_t V_real) { return 2 * sizeof(uint32_t) * static_cast<size_t>((V_real + 31) / 32); }

}  // namespace

size_t sampled_ws_bytes(const vce_problem& p) { return align_up(cand_table_bytes(p.V_real), kWsAlign); }

cudaError_t launch_sampled_candidates(const vce_problem& p, const int64_t* targets, const int64_t* draws,
                                      int64_t n_draws, int64_t P, int64_t* cand, int64_t* pos, int32_t* n_unique,
                                      void* ws, int32_t* status, cudaStream_t st) {
  const size_t table = cand_table_bytes(p.V_real);
  const bool use_smem = kHashBytes + table <= kCandSmemBudget;
  const size_t smem = kHashBytes + (use_smem ? table : 0);
  static std::atomic<uint64_t> configured{0};
  if (device_pending(configured)) {
    cudaError_t e = cudaFuncSetAttribute(sampled_cand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kCandSmemBudget));
    if (e != cudaSuccess) return e;
    mark_device_done(configured);
  }
  uint32_t* g_bits = static_cast<uint32_t*>(ws);
  int32_t* g_wpre = reinterpret_cast<int32_t*>(g_bits + (p.V_real + 31) / 32);
  sampled_cand_kernel<<<1, kThreads, smem, st>>>(targets, static_cast<int32_t>(p.T), static_cast<int32_t>(p.V_real),
                                                 p.ignore_index, draws, n_draws, static_cast<int32_t>(P), g_bits,
                                                 g_wpre, use_smem, cand, pos, n_unique, status);
  note_launch(VCE_K_SAMPLED_CAND, st);
  return cudaGetLastError();
}

cudaError_t launch_sampled_scatter(const int64_t* cand, int64_t P, const vce_problem& p, const float* dWc, float* dW,
                                   cudaStream_t st) {
  const int64_t n = P * (p.H / 4);
  if (n == 0) return cudaSuccess;
  const DevInfo di = current_device_info();
  int64_t blocks = ceil_div(n, 256 * 4);
  const int64_t cap = static_cast<int64_t>(di.num_sms) * 8;
  if (blocks > cap) blocks = cap;
  sampled_scatter_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
      cand, static_cast<int32_t>(P), static_cast<int32_t>(p.V_real), static_cast<int32_t>(p.H),
      reinterpret_cast<const float4*>(dWc), reinterpret_cast<float4*>(dW));
  note_launch(VCE_K_SAMPLED_SCATTER, st);
  return cudaGetLastError();
}

}  // namespace vce
