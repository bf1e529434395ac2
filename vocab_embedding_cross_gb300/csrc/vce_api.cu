// The C ABI of libvocabce: argument checks, workspace layout, tensor-map
// encoding and the launch sequence of each call. No device memory is
// allocated here; every buffer comes from the caller.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace vce {

namespace {
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
DevInfo g_dev[64];
std::mutex g_dev_mu;
}  // namespace

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

namespace {
std::atomic<uint64_t> g_launches{0};
std::mutex g_prof_mu;
bool g_prof_on = false;
cudaEvent_t g_prof_start = nullptr;
cudaEvent_t* g_prof_ev = nullptr;
int32_t* g_prof_kind = nullptr;
int32_t g_prof_cap = 0;
int32_t g_prof_n = 0;

void prof_release() {
  for (int i = 0; i < g_prof_cap; ++i)
    if (g_prof_ev[i]) cudaEventDestroy(g_prof_ev[i]);
  if (g_prof_start) cudaEventDestroy(g_prof_start);
  delete[] g_prof_ev;
  delete[] g_prof_kind;
  g_prof_ev = nullptr;
  g_prof_kind = nullptr;
  g_prof_start = nullptr;
  g_prof_cap = g_prof_n = 0;
  g_prof_on = false;
}
}  // namespace

void note_launch(int kind, cudaStream_t st) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (g_prof_on && g_prof_n < g_prof_cap) {
    g_prof_kind[g_prof_n] = kind;
    cudaEventRecord(g_prof_ev[g_prof_n], st);
    ++g_prof_n;
  }
}

DevInfo current_device_info() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return DevInfo{dev, 148};
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_dev[dev].device != dev) {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    g_dev[dev] = DevInfo{dev, sms > 0 ? sms : 148};
  }
  return g_dev[dev];
}

bool make_tmap_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t cols,
                  uint64_t rows, uint64_t ld, uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode || cols == 0 || rows == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * static_cast<uint64_t>(esize)};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {
int esize_of(const vce_problem& p) { return p.dtype == VCE_BF16 ? 2 : 4; }
bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }
thread_local char g_last_err[256] = "";
}  // namespace

vce_status check_problem(const vce_problem* p) {
  if (!p) return VCE_ERR_ARG;
  if ((p->flags & ~(VCE_FLAG_ACCUMULATE_DH | VCE_FLAG_DH_BF16)) != 0) return VCE_ERR_ARG;
  if (p->dtype != VCE_F32 && p->dtype != VCE_BF16) return VCE_ERR_UNSUPPORTED;
  if (p->T < 0 || p->H < 1 || p->V_real < 1 || p->S < 1) return VCE_ERR_ARG;
  if (p->Vp < 64 || p->Vp % 64 != 0) return VCE_ERR_ARG;   // the padded vocabulary must be 64-aligned
  if (p->V_real > p->Vp || p->S > p->Vp) return VCE_ERR_ARG;
  if (p->tied_weights != 0 && p->tied_weights != 1) return VCE_ERR_ARG;
  // The ignore value must not name a real class: a target equal to it could
  // then not be told from a target of that class.
  if (p->ignore_index >= 0 && p->ignore_index < p->V_real) return VCE_ERR_ARG;
  if (p->T >= (int64_t(1) << 31) || p->Vp >= (int64_t(1) << 31) || p->H > 65536) return VCE_ERR_UNSUPPORTED;
  if ((p->H * esize_of(*p)) % 16 != 0) return VCE_ERR_UNSUPPORTED;
  // Work items of the tensor-core kernels ((token block, unit or column block)
  // pairs) are numbered in 32 bits.
  if ((p->T / 256 + 1) * (p->Vp / 256 + p->S) >= (int64_t(1) << 31)) return VCE_ERR_UNSUPPORTED;
  return VCE_OK;
}

vce_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return VCE_OK;
  snprintf(g_last_err, sizeof(g_last_err), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  cudaGetLastError();
  return VCE_ERR_CUDA;
}

vce_status refuse(vce_status s, const char* why) {
  snprintf(g_last_err, sizeof(g_last_err), "%s", why);
  return s;
}

FwdLayout fwd_layout(const vce_problem& p) {
  FwdLayout L{};
  L.ug = unit_grid(p, p.dtype == VCE_BF16 ? tc_unit_width(p) : kSimtUnitWidth);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, kWsAlign);
    return o;
  };
  L.status = take(16);
  L.part = take(sizeof(float2) * static_cast<size_t>(p.T) * L.ug.n_units);
  L.ztgt = take(sizeof(float) * static_cast<size_t>(p.T));
  L.block_sums = take(sizeof(float) * 2 * static_cast<size_t>(merge_blocks(p.T)));
  L.total = off;
  return L;
}

namespace {

// Greedy argmax: one (max, column) pair per (token, unit).
size_t argmax_ws_bytes(const vce_problem& p) {
  const UnitGrid ug = unit_grid(p, p.dtype == VCE_BF16 ? tc_unit_width(p) : kSimtUnitWidth);
  return align_up(sizeof(float2) * static_cast<size_t>(p.T) * ug.n_units, kWsAlign) + kWsAlign;
}

constexpr size_t kBwdHeader = 256;   // status word, N_valid
size_t g_esize(const vce_problem& p) { return p.dtype == VCE_BF16 ? 2 : 4; }
int64_t vocab_cols_cap(const vce_problem& p) { return ceil_div(p.V_real, 256) * 256; }
size_t bwd_bytes_for(const vce_problem& p, int64_t vc) {
  return kBwdHeader + align_up(static_cast<size_t>(p.T) * static_cast<size_t>(vc) * g_esize(p), kWsAlign);
}
// Column chunk that fits the given workspace (multiple of 256), 0 if none.
int64_t bwd_chunk_cols(const vce_problem& p, size_t ws_bytes) {
  if (p.T == 0) return vocab_cols_cap(p);
  if (ws_bytes < kBwdHeader) return 0;
  int64_t vc = static_cast<int64_t>((ws_bytes - kBwdHeader) / (static_cast<size_t>(p.T) * g_esize(p)));
  vc = vc / 256 * 256;
  const int64_t cap = vocab_cols_cap(p);
  return vc > cap ? cap : vc;
}
int64_t bwd_recommended_cols(const vce_problem& p) {
  if (p.T == 0) return 256;
  // Fewest passes with at most 1.5 GiB of G per pass, the columns split evenly
  // between the passes (each pass costs three launches and a pipeline fill).
  const size_t per_col = static_cast<size_t>(p.T) * g_esize(p);
  const size_t cap_bytes = size_t(3) << 29;
  const int64_t cols = vocab_cols_cap(p);
  int64_t max_cols = static_cast<int64_t>(cap_bytes / per_col) / 256 * 256;
  if (max_cols < 256) max_cols = 256;
  const int64_t passes = ceil_div(cols, max_cols);
  int64_t vc = ceil_div(ceil_div(cols, passes), 256) * 256;
  return vc > cols ? cols : vc;
}
// Counters of the dH GEMM's K parts (bf16 path): one per (256 x 256 tile of
// dH, CTA of the pair, epilogue warp).
size_t dh_flag_bytes(const vce_problem& p) {
  if (p.dtype != VCE_BF16 || p.T == 0) return 0;
  return align_up(static_cast<size_t>(ceil_div(p.T, 256)) * static_cast<size_t>(ceil_div(p.H, 256)) * 16 *
                      sizeof(int32_t),
                  kWsAlign);
}

// fp32 sum of dH when dH itself is bf16 (VCE_FLAG_DH_BF16), at the front of
// the backward's workspace.
size_t dh_acc_bytes(const vce_problem& p) {
  if ((p.flags & VCE_FLAG_DH_BF16) == 0 || p.T == 0) return 0;
  return align_up(static_cast<size_t>(p.T) * static_cast<size_t>(p.H) * sizeof(float), kWsAlign);
}

// ----- sampled softmax: the sub-problems and the workspace layout -----
// Candidate table: P rows, padded to a multiple of 64 for the loss kernels.
int64_t cand_rows(int64_t P) { return ceil_div(P, 64) * 64; }
// Gather W[cand] (and scatter into dW): T = P ids into the full table.
vce_problem sampled_table_problem(const vce_problem& p, int64_t P, int32_t dtype) {
  vce_problem q = p;
  q.T = P;
  q.dtype = dtype;
  q.tied_weights = 0;
  return q;
}
// Cross-entropy over the candidate columns: one dense table, no vocabulary shards.
vce_problem sampled_loss_problem(const vce_problem& p, int64_t P) {
  vce_problem q = p;
  q.Vp = cand_rows(P);
  q.V_real = P;
  q.S = 1;
  q.tied_weights = 0;
  return q;
}
struct SampledLayout {
  size_t Wc, dWc, lse, loss, scratch, scratch_min, total, total_min;
};
// Wc[Pc,H] | dWc[Pc,H] fp32 | lse[T] | loss | scratch shared by the steps,
// which run one after the other on the caller's stream.
SampledLayout sampled_layout(const vce_problem& p, int64_t P) {
  SampledLayout L{};
  const vce_problem pl = sampled_loss_problem(p, P);
  const size_t rows = static_cast<size_t>(cand_rows(P)), H = static_cast<size_t>(p.H);
  L.Wc = 0;
  L.dWc = align_up(rows * H * esize_of(p), kWsAlign);
  L.lse = L.dWc + align_up(rows * H * sizeof(float), kWsAlign);
  L.loss = L.lse + align_up(sizeof(float) * static_cast<size_t>(p.T), kWsAlign);
  L.scratch = L.loss + kWsAlign;
  size_t common = sampled_ws_bytes(p);
  common = common > fwd_layout(pl).total ? common : fwd_layout(pl).total;
  const size_t bwd_min = dh_acc_bytes(pl) + bwd_bytes_for(pl, pl.T == 0 ? 0 : 256);
  const size_t bwd_rec = dh_acc_bytes(pl) + bwd_bytes_for(pl, bwd_recommended_cols(pl)) + dh_flag_bytes(pl);
  L.scratch_min = common > bwd_min ? common : bwd_min;
  const size_t rec = common > bwd_rec ? common : bwd_rec;
  L.total = L.scratch + rec;
  L.total_min = L.scratch + L.scratch_min;
  return L;
}

}  // namespace
}  // namespace vce

using namespace vce;

extern "C" {

const char* vce_status_str(vce_status s) {
  switch (s) {
    case VCE_OK: return "VCE_OK";
    case VCE_ERR_ARG: return "VCE_ERR_ARG: invalid argument or shape";
    case VCE_ERR_UNSUPPORTED: return "VCE_ERR_UNSUPPORTED: unsupported dtype, alignment or size";
    case VCE_ERR_CUDA: return "VCE_ERR_CUDA: CUDA call or launch failed";
    case VCE_ERR_BAD_INDEX: return "VCE_ERR_BAD_INDEX: target outside [0, V_real) and not ignore_index";
    case VCE_ERR_TIMEOUT: return "VCE_ERR_TIMEOUT: a bounded wait inside a kernel ran out";
    case VCE_ERR_WORKSPACE: return "VCE_ERR_WORKSPACE: workspace missing, too small or misaligned";
  }
  return "unknown vce_status";
}

int32_t vce_embed_bwd_chunk(void) { return kEmbedBwdChunk; }
const char* vce_last_error(void) { return g_last_err; }
uint64_t vce_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }
vce_status vce_profile_begin(int32_t capacity, void* stream) {
  if (capacity < 1 || capacity > (1 << 20)) return VCE_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (g_prof_on) prof_release();
  g_prof_ev = new cudaEvent_t[capacity]();
  g_prof_kind = new int32_t[capacity]();
  g_prof_cap = capacity;
  g_prof_n = 0;
  cudaError_t e = cudaEventCreate(&g_prof_start);
  for (int i = 0; e == cudaSuccess && i < capacity; ++i) e = cudaEventCreate(&g_prof_ev[i]);
  if (e == cudaSuccess) e = cudaEventRecord(g_prof_start, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    prof_release();
    return cuda_status(e);
  }
  g_prof_on = true;
  return VCE_OK;
}

int32_t vce_profile_end(float* ms, int32_t* kinds, int32_t capacity) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on) return -1;
  const int n = g_prof_n;
  int32_t out = n < capacity ? n : capacity;
  if (n > 0 && cudaEventSynchronize(g_prof_ev[n - 1]) != cudaSuccess) out = -1;
  for (int i = 0; out >= 0 && i < out; ++i) {
    float t = 0.0f;
    if (cudaEventElapsedTime(&t, i == 0 ? g_prof_start : g_prof_ev[i - 1], g_prof_ev[i]) != cudaSuccess) {
      out = -1;
      break;
    }
    if (ms) ms[i] = t;
    if (kinds) kinds[i] = g_prof_kind[i];
  }
  prof_release();
  cudaGetLastError();
  return out;
}
int32_t vce_version(void) { return 100; }
void vce_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns ? ns : 1, std::memory_order_relaxed); }

size_t vce_workspace_size(const vce_problem* p, int32_t op) {
  if (check_problem(p) != VCE_OK) return SIZE_MAX;
  switch (op) {
    case VCE_OP_EMBED_FWD: return 0;
    case VCE_OP_EMBED_BWD: return embed_bwd_ws_bytes(*p);
    case VCE_OP_LOSS_FWD: return fwd_layout(*p).total;
    case VCE_OP_LOSS_BWD:
      return dh_acc_bytes(*p) + bwd_bytes_for(*p, bwd_recommended_cols(*p)) + dh_flag_bytes(*p);
    case VCE_OP_SAMPLED_CANDIDATES: return sampled_ws_bytes(*p);
    case VCE_OP_GREEDY_ARGMAX: return argmax_ws_bytes(*p);
  }
  return SIZE_MAX;
}

size_t vce_workspace_size_min(const vce_problem* p, int32_t op) {
  if (check_problem(p) != VCE_OK) return SIZE_MAX;
  if (op == VCE_OP_LOSS_BWD) return dh_acc_bytes(*p) + bwd_bytes_for(*p, p->T == 0 ? 0 : 256);
  return vce_workspace_size(p, op);
}

vce_status vce_embed_fwd(const vce_problem* p, const int64_t* ids, const void* W, void* E, int32_t* owner,
                         int32_t* local, int32_t* dev_status, void* stream) {
  (void)dev_status;
  vce_status s = check_problem(p);
  if (s != VCE_OK) return s;
  if (p->T == 0) return VCE_OK;
  if (!ids || !W || !E) return VCE_ERR_ARG;
  if (!aligned(ids, 8) || !aligned(W, 16) || !aligned(E, 16) || !aligned(owner, 4) || !aligned(local, 4))
    return VCE_ERR_UNSUPPORTED;
  return cuda_status(launch_embed_fwd(*p, ids, W, E, owner, local, static_cast<cudaStream_t>(stream)));
}

vce_status vce_embed_fwd_plan(const vce_problem* p, const int64_t* ids, const void* W, void* E, int32_t* owner,
                              int32_t* local, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  (void)dev_status;
  vce_status s = check_problem(p);
  if (s != VCE_OK) return s;
  if (p->T == 0) return VCE_OK;
  if (!ids || !W || !E) return VCE_ERR_ARG;
  if (!aligned(ids, 8) || !aligned(W, 16) || !aligned(E, 16) || !aligned(owner, 4) || !aligned(local, 4))
    return VCE_ERR_UNSUPPORTED;
  if (!embed_bwd_supported(*p)) return VCE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, kWsAlign) || ws_bytes < embed_bwd_ws_bytes(*p)) return VCE_ERR_WORKSPACE;
  return cuda_status(launch_embed_fwd_plan(*p, ids, W, E, owner, local, ws, static_cast<cudaStream_t>(stream)));
}

vce_status vce_embed_bwd(const vce_problem* p, const int64_t* ids, const void* dE, float* dW, void* ws,
                         size_t ws_bytes, int32_t* dev_status, void* stream) {
  vce_status s = check_problem(p);
  if (s != VCE_OK) return s;
  if (p->T == 0) return VCE_OK;
  if (!ids || !dE || !dW) return VCE_ERR_ARG;
  if (!aligned(ids, 8) || !aligned(dE, 16) || !aligned(dW, 16)) return VCE_ERR_UNSUPPORTED;
  if (!embed_bwd_supported(*p)) return VCE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, kWsAlign) || ws_bytes < embed_bwd_ws_bytes(*p)) return VCE_ERR_WORKSPACE;
  return cuda_status(launch_embed_bwd(*p, ids, dE, dW, ws, dev_status, static_cast<cudaStream_t>(stream)));
}

vce_status vce_embed_bwd_plan(const vce_problem* p, const int64_t* ids, void* ws, size_t ws_bytes,
                              int32_t* dev_status, void* stream) {
  (void)dev_status;
  vce_status s = check_problem(p);
  if (s != VCE_OK) return s;
  if (p->T == 0) return VCE_OK;
  if (!ids) return VCE_ERR_ARG;
  if (!aligned(ids, 8)) return VCE_ERR_UNSUPPORTED;
  if (!embed_bwd_supported(*p)) return VCE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, kWsAlign) || ws_bytes < embed_bwd_ws_bytes(*p)) return VCE_ERR_WORKSPACE;
  return cuda_status(launch_embed_bwd_plan(*p, ids, ws, static_cast<cudaStream_t>(stream)));
}

vce_status vce_embed_bwd_apply(const vce_problem* p, const void* dE, float* dW, void* ws, size_t ws_bytes,
                               int32_t* dev_status, void* stream) {
  vce_status s = check_problem(p);
  if (s != VCE_OK) return s;
  if (p->T == 0) return VCE_OK;
  if (!dE || !dW) return VCE_ERR_ARG;
  if (!aligned(dE, 16) || !aligned(dW, 16)) return VCE_ERR_UNSUPPORTED;
  if (!embed_bwd_supported(*p)) return VCE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, kWsAlign) || ws_bytes < embed_bwd_ws_bytes(*p)) return VCE_ERR_WORKSPACE;
  return cuda_status(launch_embed_bwd_apply(*p, dE, dW, ws, dev_status, static_cast<cudaStream_t>(stream)));
}

vce_status vce_loss_fwd(const vce_problem* p, const void* h, const void* W, const int64_t* targets, float* loss,
                        float* lse, float* token_loss, int32_t* target_owner, int32_t* max_owner, void* ws,
                        size_t ws_bytes, int32_t* dev_status, void* stream) {
  vce_status s = check_problem(p);
  if (s != VCE_OK) return s;
  if (!loss) return VCE_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p->T == 0) return cuda_status(cudaMemsetAsync(loss, 0, sizeof(float), st));
  if (!h || !W || !targets || !lse) return VCE_ERR_ARG;
  if (!aligned(h, 16) || !aligned(W, 16) || !aligned(targets, 8) || !aligned(loss, 4) || !aligned(lse, 4) ||
      !aligned(token_loss, 4) || !aligned(target_owner, 4) || !aligned(max_owner, 4))
    return VCE_ERR_UNSUPPORTED;
  const FwdLayout L = fwd_layout(*p);
  if (!ws || !aligned(ws, kWsAlign) || ws_bytes < L.total) return VCE_ERR_WORKSPACE;
  char* b = static_cast<char*>(ws);
  int32_t* status = dev_status;
  if (!status) {
    status = reinterpret_cast<int32_t*>(b + L.status);
    if (cudaError_t me = cudaMemsetAsync(status, 0, sizeof(int32_t), st)) return cuda_status(me);
  }
  float2* part = reinterpret_cast<float2*>(b + L.part);
  float* ztgt = reinterpret_cast<float*>(b + L.ztgt);
  float* bsum = reinterpret_cast<float*>(b + L.block_sums);
  int32_t* merge_ctr = reinterpret_cast<int32_t*>(b + L.status + 4);
  const ProbDev pd = prob_dev(*p);
  cudaError_t e;
  if (p->dtype == VCE_BF16)
    e = launch_tc_fwd(*p, L.ug, h, W, targets, part, ztgt, merge_ctr, status, st);
  else
    e = launch_simt_fwd(pd, L.ug, static_cast<const float*>(h), static_cast<const float*>(W), targets, part, ztgt,
                        merge_ctr, st);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_merge(pd, L.ug, targets, part, ztgt, lse, token_loss, target_owner, max_owner, bsum,
                                  merge_ctr, loss, status, st));
}

vce_status vce_loss_bwd(const vce_problem* p, const void* h, const void* W, const int64_t* targets,
                        const float* lse, float g, void* dH_out, float* dW, void* ws, size_t ws_bytes,
                        int32_t* dev_status, void* stream) {
  vce_status s = check_problem(p);
  if (s != VCE_OK) return s;
  if (!dW) return VCE_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t row_bytes = static_cast<size_t>(p->H) * sizeof(float);
  if (p->T == 0) {
    if (!p->tied_weights) return cuda_status(cudaMemsetAsync(dW, 0, row_bytes * p->Vp, st));
    return VCE_OK;
  }
  if (!h || !W || !targets || !lse || !dH_out) return VCE_ERR_ARG;
  if (!aligned(h, 16) || !aligned(W, 16) || !aligned(targets, 8) || !aligned(lse, 4) || !aligned(dH_out, 16) ||
      !aligned(dW, 16))
    return VCE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, kWsAlign)) return VCE_ERR_WORKSPACE;
  // A bf16 dH is summed in fp32 at the front of the workspace and rounded once
  // at the end; the rest of the layout follows it.
  const size_t acc_bytes = dh_acc_bytes(*p);
  if (ws_bytes < acc_bytes) return VCE_ERR_WORKSPACE;
  float* dH = acc_bytes ? static_cast<float*>(ws) : static_cast<float*>(dH_out);
  ws = static_cast<char*>(ws) + acc_bytes;
  ws_bytes -= acc_bytes;
  // Layout: header | dH K-part counters (when the workspace has room) | G chunk.
  const size_t part_bytes = dh_flag_bytes(*p);
  const bool use_parts = part_bytes > 0 && ws_bytes >= bwd_bytes_for(*p, 256) + part_bytes;
  const int64_t vc = bwd_chunk_cols(*p, use_parts ? ws_bytes - part_bytes : ws_bytes);
  if (vc < 256) return VCE_ERR_WORKSPACE;
  char* b = static_cast<char*>(ws);
  int32_t* status = dev_status;
  int32_t* n_valid = reinterpret_cast<int32_t*>(b + 16);
  if (!status) {
    status = reinterpret_cast<int32_t*>(b);
    if (cudaError_t me = cudaMemsetAsync(status, 0, sizeof(int32_t), st)) return cuda_status(me);
  }
  int32_t* dh_flags = use_parts ? reinterpret_cast<int32_t*>(b + kBwdHeader) : nullptr;
  void* G = b + kBwdHeader + (use_parts ? part_bytes : 0);
  const ProbDev pd = prob_dev(*p);
  // The fp32 path counts the valid targets first; the tensor-core GRAD kernel
  // counts them itself.
  if (p->dtype != VCE_BF16)
    if (cudaError_t ce = launch_count_valid(pd, targets, n_valid, status, st)) return cuda_status(ce);
  if (!p->tied_weights && p->Vp > p->V_real) {
    if (cudaMemsetAsync(dW + static_cast<size_t>(p->V_real) * p->H, 0, row_bytes * (p->Vp - p->V_real), st) !=
        cudaSuccess)
      return VCE_ERR_CUDA;
  }
  const bool acc_out = (p->flags & VCE_FLAG_ACCUMULATE_DH) != 0;
  const bool acc_dh = acc_out && acc_bytes == 0;   // a bf16 dH is added in the rounding step
  for (int64_t c0 = 0; c0 < p->V_real; c0 += vc) {
    const int vc_act = static_cast<int>((p->V_real - c0) < vc ? (p->V_real - c0) : vc);
    cudaError_t e;
    if (p->dtype == VCE_BF16) {
      const int parts = dh_flags ? tc_dh_parts(*p, vc_act) : 1;
      e = launch_tc_bwd_chunk(*p, h, W, targets, lse, g, static_cast<int>(c0), vc_act, G,
                              static_cast<int>(vc), dH, c0 > 0 || acc_dh, dW, p->tied_weights != 0, dh_flags, parts,
                              status, st);
    } else {
      float* Gf = static_cast<float*>(G);
      const float* hf = static_cast<const float*>(h);
      const float* Wf = static_cast<const float*>(W);
      e = launch_simt_grad(pd, hf, Wf, targets, lse, n_valid, g, static_cast<int>(c0), vc_act, Gf, st);
      if (e == cudaSuccess)   // dH (+)= G W[c0:c0+vc_act]
        e = launch_sgemm(pd.T, pd.H, vc_act, Gf, vc_act, 1, Wf + c0 * p->H, p->H, 1, dH, p->H,
                         (c0 > 0 || acc_dh) ? 1 : 0, st);
      if (e == cudaSuccess)   // dW[c0:c0+vc_act] (+)= G^T h
        e = launch_sgemm(vc_act, pd.H, pd.T, Gf, 1, vc_act, hf, p->H, 1, dW + c0 * p->H, p->H,
                         p->tied_weights ? 1 : 0, st);
    }
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (acc_bytes)
    return cuda_status(launch_dh_to_bf16(dH, dH_out, p->T * p->H, acc_out, st));
  return VCE_OK;
}

vce_status vce_sampled_candidates(const vce_problem* p, const int64_t* targets, const int64_t* draws,
                                  int64_t n_draws, int64_t P, int64_t* cand, int64_t* pos, int32_t* n_unique,
                                  void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  vce_status s = check_problem(p);
  if (s != VCE_OK) return s;
  if (P < 1 || P > p->V_real || n_draws < 0) return VCE_ERR_ARG;
  if (!cand || !n_unique || (p->T > 0 && (!targets || !pos)) || (n_draws > 0 && !draws)) return VCE_ERR_ARG;
  if (!aligned(targets, 8) || !aligned(draws, 8) || !aligned(cand, 8) || !aligned(pos, 8) || !aligned(n_unique, 4))
    return VCE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, kWsAlign) || ws_bytes < sampled_ws_bytes(*p)) return VCE_ERR_WORKSPACE;
  return cuda_status(launch_sampled_candidates(*p, targets, draws, n_draws, P, cand, pos, n_unique, ws, dev_status,
                                               static_cast<cudaStream_t>(stream)));
}

size_t vce_sampled_workspace_size(const vce_problem* p, int64_t P) {
  if (check_problem(p) != VCE_OK || P < 1 || P > p->V_real) return SIZE_MAX;
  return sampled_layout(*p, P).total;
}

vce_status vce_sampled_loss(const vce_problem* p, const void* h, const void* W, const int64_t* targets,
                            const int64_t* draws, int64_t n_draws, int64_t P, float g, float* loss, float* lse,
                            void* dH, float* dW, int64_t* cand, int64_t* pos, int32_t* n_unique, void* ws,
                            size_t ws_bytes, int32_t* dev_status, void* stream) {
  vce_status s = check_problem(p);
  if (s != VCE_OK) return s;
  if (P < 1 || P > p->V_real || n_draws < 0) return VCE_ERR_ARG;
  if (!W || !dW || !cand || !n_unique || !loss || (n_draws > 0 && !draws)) return VCE_ERR_ARG;
  if (p->T > 0 && (!h || !targets || !dH || !pos)) return VCE_ERR_ARG;
  if (!aligned(dW, 16) || !aligned(loss, 4) || !aligned(lse, 4)) return VCE_ERR_UNSUPPORTED;
  const SampledLayout L = sampled_layout(*p, P);
  if (!ws || !aligned(ws, kWsAlign) || ws_bytes < L.total_min) return VCE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* b = static_cast<char*>(ws);
  void* Wc = b + L.Wc;
  float* dWc = reinterpret_cast<float*>(b + L.dWc);
  float* lse_c = lse ? lse : reinterpret_cast<float*>(b + L.lse);
  void* scratch = b + L.scratch;
  const size_t scratch_bytes = ws_bytes - L.scratch;
  const vce_problem pg = sampled_table_problem(*p, P, p->dtype);
  const vce_problem pl = sampled_loss_problem(*p, P);
  // 1. candidate list and each target's position in it
  s = vce_sampled_candidates(p, targets, draws, n_draws, P, cand, pos, n_unique, scratch, scratch_bytes, dev_status,
                             stream);
  if (s != VCE_OK) return s;
  // 2. Wc = W[cand]; the padding rows of the table are zero
  const size_t row_bytes = static_cast<size_t>(p->H) * esize_of(*p);
  if (pl.Vp > P) {
    if (cudaError_t me = cudaMemsetAsync(static_cast<char*>(Wc) + P * row_bytes, 0, (pl.Vp - P) * row_bytes, st))
      return cuda_status(me);
  }
  s = vce_embed_fwd(&pg, cand, W, Wc, nullptr, nullptr, dev_status, stream);
  if (s != VCE_OK) return s;
  // 3. cross-entropy over the candidate columns, targets remapped to positions
  s = vce_loss_fwd(&pl, h, Wc, pos, loss, lse_c, nullptr, nullptr, nullptr, scratch, scratch_bytes, dev_status,
                   stream);
  if (s != VCE_OK) return s;
  // 4. dH and the candidate rows' gradient dWc (overwritten)
  s = vce_loss_bwd(&pl, h, Wc, pos, lse_c, g, dH, dWc, scratch, scratch_bytes, dev_status, stream);
  if (s != VCE_OK) return s;
  // 5. dW[cand[i]] += dWc[i]: the candidates are distinct, one addition per element
  return cuda_status(launch_sampled_scatter(cand, P, *p, dWc, dW, st));
}

vce_status vce_greedy_argmax(const vce_problem* p, const void* h, const void* W, int64_t* argmax,
                             float* max_logit, int32_t* owner, void* ws, size_t ws_bytes, int32_t* dev_status,
                             void* stream) {
  vce_status s = check_problem(p);
  if (s != VCE_OK) return s;
  if (p->T == 0) return VCE_OK;
  if (!h || !W || !argmax) return VCE_ERR_ARG;
  if (!aligned(h, 16) || !aligned(W, 16) || !aligned(argmax, 8) || !aligned(max_logit, 4) || !aligned(owner, 4))
    return VCE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, kWsAlign) || ws_bytes < argmax_ws_bytes(*p)) return VCE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const UnitGrid ug = unit_grid(*p, p->dtype == VCE_BF16 ? tc_unit_width(*p) : kSimtUnitWidth);
  const ProbDev pd = prob_dev(*p);
  char* b = static_cast<char*>(ws);
  int32_t* status = dev_status;
  if (!status) {
    status = reinterpret_cast<int32_t*>(b);
    if (cudaError_t me = cudaMemsetAsync(status, 0, sizeof(int32_t), st)) return cuda_status(me);
  }
  float2* part = reinterpret_cast<float2*>(b + kWsAlign);
  cudaError_t e = p->dtype == VCE_BF16
                      ? launch_tc_argmax(*p, ug, h, W, part, status, st)
                      : launch_simt_argmax(pd, ug, static_cast<const float*>(h), static_cast<const float*>(W), part,
                                           st);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_argmax_merge(pd, ug, part, argmax, max_logit, owner, st));
}

vce_status vce_ngram_hash(const int64_t* ids, int64_t T, int32_t n, int64_t V, int64_t M, int64_t seq_len,
                          int64_t* out, void* stream) {
  if (T < 0 || T >= (int64_t(1) << 31) || n < 1 || V < 1 || V >= (int64_t(1) << 31) || M < 1 ||
      M >= (int64_t(1) << 31) || seq_len < 0)
    return VCE_ERR_ARG;
  if (T == 0) return VCE_OK;
  if (!ids || !out) return VCE_ERR_ARG;
  if (!aligned(ids, 8) || !aligned(out, 8)) return VCE_ERR_UNSUPPORTED;
  return cuda_status(launch_ngram_hash(ids, T, n, V, M, seq_len, out, static_cast<cudaStream_t>(stream)));
}

namespace {
bool ngram_tables_ok(int64_t M2, const void* T2, int64_t M3, const void* T3) {
  const int64_t lim = int64_t(1) << 31;
  return M2 >= 0 && M2 < lim && M3 >= 0 && M3 < lim && (M2 == 0 || T2) && (M3 == 0 || T3);
}
// The embedding backward of one n-gram table: a problem whose "vocabulary" is the table's rows.
vce_problem ngram_table_problem(const vce_problem& p, int64_t M) {
  vce_problem q = p;
  q.Vp = M;
  q.V_real = M;
  q.S = 1;
  q.tied_weights = 0;
  return q;
}
}  // namespace

vce_status vce_ngram_embed_fwd(const vce_problem* p, const int64_t* ids, const void* W, const void* T2,
                               int64_t M2, const void* T3, int64_t M3, int64_t seq_len, void* E,
                               int32_t* dev_status, void* stream) {
  (void)dev_status;
  vce_status s = check_problem(p);
  if (s != VCE_OK) return s;
  if (!ngram_tables_ok(M2, T2, M3, T3) || seq_len < 0) return VCE_ERR_ARG;
  if (p->T == 0) return VCE_OK;
  if (!ids || !W || !E) return VCE_ERR_ARG;
  if (!aligned(ids, 8) || !aligned(W, 16) || !aligned(T2, 16) || !aligned(T3, 16) || !aligned(E, 16))
    return VCE_ERR_UNSUPPORTED;
  return cuda_status(launch_ngram_embed_fwd(*p, ids, W, M2 ? T2 : nullptr, M2, M3 ? T3 : nullptr, M3, seq_len, E,
                                            static_cast<cudaStream_t>(stream)));
}

size_t vce_ngram_workspace_size(const vce_problem* p) {
  if (check_problem(p) != VCE_OK) return SIZE_MAX;
  // the two n-gram row-index arrays, then one embedding-backward workspace per table
  return 2 * align_up(sizeof(int64_t) * static_cast<size_t>(p->T), kWsAlign) + 3 * embed_bwd_ws_bytes(*p);
}

namespace {
// The n-gram backward's problems: the token table, then the 2-gram and 3-gram
// tables that are present, each with its row indices and its part of the
// workspace (the two row-index arrays, then one embedding-backward workspace
// per table).
struct NgramBwd {
  vce_problem ps[3];
  const int64_t* pid[3];
  float* pdw[3];
  void* pws[3];
  int n;
  int64_t* idx2;
  int64_t* idx3;
};
NgramBwd ngram_bwd(const vce_problem& p, const int64_t* ids, float* dW, float* dT2, int64_t M2, float* dT3,
                   int64_t M3, void* ws) {
  NgramBwd g{};
  char* b = static_cast<char*>(ws);
  const size_t ids_bytes = align_up(sizeof(int64_t) * static_cast<size_t>(p.T), kWsAlign);
  const size_t ews_bytes = embed_bwd_ws_bytes(p);
  g.idx2 = reinterpret_cast<int64_t*>(b);
  g.idx3 = reinterpret_cast<int64_t*>(b + ids_bytes);
  g.ps[0] = p;
  g.pid[0] = ids;
  g.pdw[0] = dW;
  g.pws[0] = b + 2 * ids_bytes;
  g.n = 1;
  if (M2 > 0) {
    g.ps[g.n] = ngram_table_problem(p, M2);
    g.pid[g.n] = g.idx2;
    g.pdw[g.n] = dT2;
    g.pws[g.n] = b + 2 * ids_bytes + ews_bytes;
    ++g.n;
  }
  if (M3 > 0) {
    g.ps[g.n] = ngram_table_problem(p, M3);
    g.pid[g.n] = g.idx3;
    g.pdw[g.n] = dT3;
    g.pws[g.n] = b + 2 * ids_bytes + 2 * ews_bytes;
    ++g.n;
  }
  return g;
}

// Row indices of the present tables, then their plans.
cudaError_t ngram_plan(const vce_problem& p, const int64_t* ids, int64_t M2, int64_t M3, int64_t seq_len,
                       const NgramBwd& g, cudaStream_t st) {
  if (M2 > 0 && M3 > 0) {
    if (cudaError_t e = launch_ngram_hash_pair(ids, p.T, p.V_real, M2, M3, seq_len, g.idx2, g.idx3, st)) return e;
  } else if (M2 > 0) {
    if (cudaError_t e = launch_ngram_hash(ids, p.T, 2, p.V_real, M2, seq_len, g.idx2, st)) return e;
  } else if (M3 > 0) {
    if (cudaError_t e = launch_ngram_hash(ids, p.T, 3, p.V_real, M3, seq_len, g.idx3, st)) return e;
  }
  return launch_embed_bwd_plan_multi(g.ps, g.pid, g.pws, g.n, st);
}

// The backward's size and workspace rules (after check_problem, for T > 0).
vce_status ngram_bwd_check(const vce_problem* p, const void* ws, size_t ws_bytes) {
  if (!embed_bwd_supported(*p)) return VCE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, kWsAlign) || ws_bytes < vce_ngram_workspace_size(p)) return VCE_ERR_WORKSPACE;
  return VCE_OK;
}
}  // namespace

vce_status vce_ngram_embed_bwd(const vce_problem* p, const int64_t* ids, const void* dE, float* dW, float* dT2,
                               int64_t M2, float* dT3, int64_t M3, int64_t seq_len, void* ws, size_t ws_bytes,
                               int32_t* dev_status, void* stream) {
  vce_status s = check_problem(p);
  if (s != VCE_OK) return s;
  if (!ngram_tables_ok(M2, dT2, M3, dT3) || seq_len < 0) return VCE_ERR_ARG;
  if (p->T == 0) return VCE_OK;
  if (!ids || !dE || !dW) return VCE_ERR_ARG;
  if (!aligned(ids, 8) || !aligned(dE, 16) || !aligned(dW, 16) || !aligned(dT2, 16) || !aligned(dT3, 16))
    return VCE_ERR_UNSUPPORTED;
  if ((s = ngram_bwd_check(p, ws, ws_bytes)) != VCE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The row indices first; then the tables' backward problems are sorted one
  // after the other and reduced in one launch.
  const NgramBwd g = ngram_bwd(*p, ids, dW, dT2, M2, dT3, M3, ws);
  if (cudaError_t e = ngram_plan(*p, ids, M2, M3, seq_len, g, st)) return cuda_status(e);
  return cuda_status(launch_embed_bwd_apply_multi(g.ps, g.pdw, g.pws, g.n, dE, dev_status, st));
}

vce_status vce_ngram_embed_bwd_plan(const vce_problem* p, const int64_t* ids, int64_t M2, int64_t M3,
                                    int64_t seq_len, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  (void)dev_status;
  vce_status s = check_problem(p);
  if (s != VCE_OK) return s;
  const int64_t lim = int64_t(1) << 31;
  if (M2 < 0 || M2 >= lim || M3 < 0 || M3 >= lim || seq_len < 0) return VCE_ERR_ARG;
  if (p->T == 0) return VCE_OK;
  if (!ids) return VCE_ERR_ARG;
  if (!aligned(ids, 8)) return VCE_ERR_UNSUPPORTED;
  if ((s = ngram_bwd_check(p, ws, ws_bytes)) != VCE_OK) return s;
  const NgramBwd g = ngram_bwd(*p, ids, nullptr, nullptr, M2, nullptr, M3, ws);
  return cuda_status(ngram_plan(*p, ids, M2, M3, seq_len, g, static_cast<cudaStream_t>(stream)));
}

vce_status vce_ngram_embed_bwd_apply(const vce_problem* p, const void* dE, float* dW, float* dT2, int64_t M2,
                                     float* dT3, int64_t M3, void* ws, size_t ws_bytes, int32_t* dev_status,
                                     void* stream) {
  vce_status s = check_problem(p);
  if (s != VCE_OK) return s;
  if (!ngram_tables_ok(M2, dT2, M3, dT3)) return VCE_ERR_ARG;
  if (p->T == 0) return VCE_OK;
  if (!dE || !dW) return VCE_ERR_ARG;
  if (!aligned(dE, 16) || !aligned(dW, 16) || !aligned(dT2, 16) || !aligned(dT3, 16)) return VCE_ERR_UNSUPPORTED;
  if ((s = ngram_bwd_check(p, ws, ws_bytes)) != VCE_OK) return s;
  const NgramBwd g = ngram_bwd(*p, nullptr, dW, dT2, M2, dT3, M3, ws);
  return cuda_status(
      launch_embed_bwd_apply_multi(g.ps, g.pdw, g.pws, g.n, dE, dev_status, static_cast<cudaStream_t>(stream)));
}

vce_status vce_wait_selftest(uint64_t limit_ns, int32_t* dev_status, void* stream) {
  if (!dev_status) return VCE_ERR_ARG;
  return cuda_status(launch_wait_selftest(limit_ns, dev_status, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
