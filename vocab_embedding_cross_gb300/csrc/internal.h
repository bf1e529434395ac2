// Internal declarations shared by the translation units of libvocabce.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/vce.h"

namespace vce {

constexpr int kEmbedBwdChunk = 32;      // run length of the embedding backward's order
constexpr int kTcUnitWidth = 2048;      // widest forward work unit (tensor cores), in vocab columns
constexpr int kSimtUnitWidth = 256;     // vocab columns per forward work unit (fp32 SIMT)
constexpr size_t kWsAlign = 256;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Programmatic dependent launch (sm_90 and later). A kernel launched with the
// programmatic-serialisation attribute may start once every CTA of the
// previous kernel in the stream has called grid_dep_launch() or exited;
// grid_dep_wait() then blocks until that kernel has completed and its writes
// are visible. Both are no-ops in a kernel launched the ordinary way.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launches `kern` with programmatic stream serialisation: it may start while
// the previous kernel in the stream is still running, and must call
// grid_dep_wait() before it touches anything that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Shard owning a row id in [0, Vp): the largest k with floor(k*Vp/S) <= id,
// i.e. ceil((id+1)*S/Vp) - 1.
__host__ __device__ inline int32_t shard_of(int64_t id, int64_t Vp, int32_t S) {
  return static_cast<int32_t>(((id + 1) * static_cast<int64_t>(S) + Vp - 1) / Vp - 1);
}
__host__ __device__ inline int64_t shard_lo(int64_t k, int64_t Vp, int32_t S) { return (k * Vp) / S; }

// Forward work units: each shard is cut into `ups` units of `uw` columns
// (the last one of a shard may be shorter or empty).
struct UnitGrid {
  int32_t uw, ups, n_units;
};
inline UnitGrid unit_grid(const vce_problem& p, int uw) {
  int64_t max_rows = ceil_div(p.Vp, p.S);
  int32_t ups = static_cast<int32_t>(ceil_div(max_rows, uw));
  if (ups < 1) ups = 1;
  return UnitGrid{uw, ups, static_cast<int32_t>(ups * static_cast<int64_t>(p.S))};
}

// Device-side view of a problem (plain values, passed by value to kernels).
struct ProbDev {
  int32_t T, H, Vp, V_real, S;
  int64_t ignore_index;
};
inline ProbDev prob_dev(const vce_problem& p) {
  return ProbDev{static_cast<int32_t>(p.T), static_cast<int32_t>(p.H), static_cast<int32_t>(p.Vp),
                 static_cast<int32_t>(p.V_real), p.S, p.ignore_index};
}

// Host-side argument rules shared by every entry point that takes a problem
// (shapes, flags, dtype, the ignore value, 32-bit work-item numbering).
vce_status check_problem(const vce_problem* p);
// VCE_OK, or VCE_ERR_CUDA with the error's name and text kept for
// vce_last_error (the sticky error is cleared).
vce_status cuda_status(cudaError_t e);
// Returns `s` and keeps `why` as the calling thread's vce_last_error text.
vce_status refuse(vce_status s, const char* why);

// Workspace of the loss forward: status word (and, 4 bytes on, the merge's
// last-block counter), per-(token, unit) partials, target logits and the
// mean's block sums, each 256-byte aligned.
struct FwdLayout {
  size_t status, part, ztgt, block_sums, total;
  UnitGrid ug;
};
FwdLayout fwd_layout(const vce_problem& p);

struct DevInfo {
  int device = -1;
  int num_sms = 0;
};
DevInfo current_device_info();

// Per-device one-time setup (a kernel's shared-memory limit is a property of
// the device): true until mark_device_done has run for the current device.
// Two threads may both see "not done" and both do the (idempotent) setup.
inline bool device_pending(const std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev < 0 || dev >= 64 || (done.load(std::memory_order_acquire) & (uint64_t(1) << dev)) == 0;
}
inline void mark_device_done(std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64) done.fetch_or(uint64_t(1) << dev, std::memory_order_release);
}
uint64_t wait_limit_ns();
// Called after every kernel launch: counts it and, when a table is installed,
// records the next timing event on `st` (see vce_set_launch_events).
void note_launch(int kind, cudaStream_t st);

// Encodes a row-major 2-D tensor map (driver entry point fetched at run time).
// rows x cols elements of `esize` bytes, row stride `ld` elements.
bool make_tmap_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t cols,
                  uint64_t rows, uint64_t ld, uint32_t box_cols, uint32_t box_rows, bool swizzle128);

// ---------------------------------------------------------------------------
// Launchers. Each returns cudaSuccess or the launch error.
// ---------------------------------------------------------------------------
cudaError_t launch_embed_fwd(const vce_problem& p, const int64_t* ids, const void* W, void* E, int32_t* owner,
                             int32_t* local, cudaStream_t st);
// The lookup and the embedding backward's plan in one sequence: the plan's
// launches first, then the lookup as their dependent, running beside the sort.
cudaError_t launch_embed_fwd_plan(const vce_problem& p, const int64_t* ids, const void* W, void* E, int32_t* owner,
                                  int32_t* local, void* ws, cudaStream_t st);

size_t embed_bwd_ws_bytes(const vce_problem& p);
// False when the embedding backward's work items would not fit in 32 bits.
bool embed_bwd_supported(const vce_problem& p);
// The backward is a plan (the sort of the ids into runs, kept in the
// workspace) followed by its application to dE. launch_embed_bwd does both;
// the apply leaves the plan unchanged, so it can be applied again.
cudaError_t launch_embed_bwd(const vce_problem& p, const int64_t* ids, const void* dE, float* dW, void* ws,
                             int32_t* status, cudaStream_t st);
cudaError_t launch_embed_bwd_plan(const vce_problem& p, const int64_t* ids, void* ws, cudaStream_t st);
cudaError_t launch_embed_bwd_apply(const vce_problem& p, const void* dE, float* dW, void* ws, int32_t* status,
                                   cudaStream_t st);
// n (1 to 3) backward problems with the same T, H and dtype and the same dE,
// each with its own ids, dW and workspace (embed_bwd_ws_bytes of it): one
// header-zeroing launch, one sort per problem, one reduce over all of them.
cudaError_t launch_embed_bwd_multi(const vce_problem* ps, const int64_t* const* ids, float* const* dW,
                                   void* const* ws, int n, const void* dE, int32_t* status, cudaStream_t st);
// The same in its two parts: the plans of the n problems (one zeroing launch,
// one sort each), and one reduce that applies them all to dE.
cudaError_t launch_embed_bwd_plan_multi(const vce_problem* ps, const int64_t* const* ids, void* const* ws, int n,
                                        cudaStream_t st);
cudaError_t launch_embed_bwd_apply_multi(const vce_problem* ps, float* const* dW, void* const* ws, int n,
                                         const void* dE, int32_t* status, cudaStream_t st);

// Merge of the forward partials into lse, per-token loss and the mean. The
// forward kernel before it zeroes `counter` (the merge's last-block counter).
cudaError_t launch_merge(const ProbDev& pd, const UnitGrid& ug, const int64_t* targets, const float2* part,
                         const float* ztgt, float* lse, float* token_loss, int32_t* target_owner,
                         int32_t* max_owner, float* block_sums, int32_t* counter, float* loss, int32_t* status,
                         cudaStream_t st);
int merge_blocks(int64_t T);
cudaError_t launch_count_valid(const ProbDev& pd, const int64_t* targets, int32_t* n_valid, int32_t* status,
                               cudaStream_t st);
// dH[T,H] in bf16 from its fp32 sum (n = T*H, a multiple of 4): rounded once,
// after adding the bf16 values already there when accumulating.
cudaError_t launch_dh_to_bf16(const float* acc, void* out, int64_t n, bool accumulate, cudaStream_t st);
// Greedy argmax: merge of the units' (max, column) partials (column stored as the float's bits).
cudaError_t launch_argmax_merge(const ProbDev& pd, const UnitGrid& ug, const float2* part, int64_t* argmax,
                                float* max_logit, int32_t* owner, cudaStream_t st);

// fp32 SIMT path.
cudaError_t launch_simt_fwd(const ProbDev& pd, const UnitGrid& ug, const float* h, const float* W,
                            const int64_t* targets, float2* part, float* ztgt, int32_t* merge_ctr, cudaStream_t st);
cudaError_t launch_simt_argmax(const ProbDev& pd, const UnitGrid& ug, const float* h, const float* W, float2* part,
                               cudaStream_t st);
cudaError_t launch_simt_grad(const ProbDev& pd, const float* h, const float* W, const int64_t* targets,
                             const float* lse, const int32_t* n_valid, float g, int v0, int vc, float* G,
                             cudaStream_t st);
// C[M,N] = beta*C + sum_k A(m,k) B(k,n), A(m,k) = A[m*sam + k*sak], B(k,n) = B[k*sbk + n*sbn],
// C row-major with leading dimension ldc. beta is 0 or 1.
cudaError_t launch_sgemm(int M, int N, int K, const float* A, int64_t sam, int64_t sak, const float* B,
                         int64_t sbk, int64_t sbn, float* C, int64_t ldc, int beta, cudaStream_t st);

// bf16 tensor-core path.
cudaError_t launch_tc_fwd(const vce_problem& p, const UnitGrid& ug, const void* h, const void* W,
                          const int64_t* targets, float2* part, float* ztgt, int32_t* merge_ctr, int32_t* status,
                          cudaStream_t st);
cudaError_t launch_tc_argmax(const vce_problem& p, const UnitGrid& ug, const void* h, const void* W, float2* part,
                             int32_t* status, cudaStream_t st);
cudaError_t launch_tc_bwd_chunk(const vce_problem& p, const void* h, const void* W, const int64_t* targets,
                                const float* lse, float g, int v0, int vc_act,
                                void* G, int g_ld, float* dH, bool dH_accumulate, float* dW, bool dW_accumulate,
                                int32_t* dh_flags, int dh_parts, int32_t* status, cudaStream_t st);
// Number of K parts for the dH GEMM of one column chunk (fills the waves of
// the persistent grid); at most kMaxDhParts.
constexpr int kMaxDhParts = 8;
int tc_dh_parts(const vce_problem& p, int vc_act);
// Forward unit width (a multiple of 256, at most kTcUnitWidth) that balances
// the persistent grid's waves for this problem on the current device.
int tc_unit_width(const vce_problem& p);

cudaError_t launch_wait_selftest(uint64_t limit_ns, int32_t* status, cudaStream_t st);

// Hashed n-gram embeddings.
cudaError_t launch_ngram_hash(const int64_t* ids, int64_t T, int n, int64_t V, int64_t M, int64_t seq_len,
                              int64_t* out, cudaStream_t st);
// The 2-gram and 3-gram row indices (M2, M3 > 0) in one launch.
cudaError_t launch_ngram_hash_pair(const int64_t* ids, int64_t T, int64_t V, int64_t M2, int64_t M3, int64_t seq_len,
                                   int64_t* out2, int64_t* out3, cudaStream_t st);
cudaError_t launch_ngram_embed_fwd(const vce_problem& p, const int64_t* ids, const void* W, const void* T2,
                                   int64_t M2, const void* T3, int64_t M3, int64_t seq_len, void* E,
                                   cudaStream_t st);

// Sampled-softmax candidate list.
size_t sampled_ws_bytes(const vce_problem& p);
cudaError_t launch_sampled_candidates(const vce_problem& p, const int64_t* targets, const int64_t* draws,
                                      int64_t n_draws, int64_t P, int64_t* cand, int64_t* pos, int32_t* n_unique,
                                      void* ws, int32_t* status, cudaStream_t st);
// dW[cand[i], :] += dWc[i, :] for the distinct candidates (rows with cand < 0 skipped).
cudaError_t launch_sampled_scatter(const int64_t* cand, int64_t P, const vce_problem& p, const float* dWc, float* dW,
                                   cudaStream_t st);

}  // namespace vce
