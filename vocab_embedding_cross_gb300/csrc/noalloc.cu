// Loss forward for callers that cannot allocate device memory.
//
// vce_loss_fwd needs a caller-provided workspace for its per-tile partial
// results. Some callers cannot provide one: code that runs inside a host
// framework which owns every byte of device memory and only hands a plugin its
// inputs and outputs, or a hot path that must never call cudaMalloc (which can
// synchronise the device, fragment a pooled allocator, or fail under memory
// pressure in the middle of a step). vce_loss_fwd_noalloc runs the same
// kernels as vce_loss_fwd with its scratch in a fixed array that lives in the
// library's own device memory for as long as the library is loaded.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "internal.h"

namespace vce {
namespace {

// 16 MiB of scratch, reserved on every GPU that loads the library until the
// process exits. Enough for the forward of T = 8192 tokens over a 151936-entry
// vocabulary in 8 shards (about 5.3 MB) or T = 16384 over 201088 at H = 2048 (about 13.7 MB).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[64] = {};

// Device address of the scratch array for the current device. In host code the
// array's name only stands for the symbol; its device address is asked for
// once per device, with that device current, and kept. A device reset after
// that first call would leave the kept address stale; that is not supported.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool aligned_to(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

}  // namespace
}  // namespace vce

using namespace vce;

extern "C" {

size_t vce_loss_fwd_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

vce_status vce_loss_fwd_noalloc(const vce_problem* p, const void* h, const void* W, const int64_t* targets,
                                float* loss, float* lse, float* token_loss, int32_t* target_owner,
                                int32_t* max_owner, int32_t* dev_status, void* stream) {
  // The argument rules and the scratch layout are vce_loss_fwd's own.
  vce_status s = check_problem(p);
  if (s != VCE_OK) return s;
  if (!loss) return VCE_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p->T == 0) return cuda_status(cudaMemsetAsync(loss, 0, sizeof(float), st));
  if (!h || !W || !targets || !lse) return VCE_ERR_ARG;
  if (!aligned_to(h, 16) || !aligned_to(W, 16) || !aligned_to(targets, 8) || !aligned_to(loss, 4) ||
      !aligned_to(lse, 4) || !aligned_to(token_loss, 4) || !aligned_to(target_owner, 4) ||
      !aligned_to(max_owner, 4))
    return VCE_ERR_UNSUPPORTED;
  const FwdLayout L = fwd_layout(*p);
  if (L.total > kNoAllocScratchBytes) {   // problem too large for the fixed scratch: nothing is enqueued
    char why[160];
    snprintf(why, sizeof(why),
             "vce_loss_fwd_noalloc: the forward needs %zu bytes of scratch, more than the fixed %zu-byte array",
             L.total, kNoAllocScratchBytes);
    return refuse(VCE_ERR_WORKSPACE, why);
  }
  void* base = nullptr;
  if (cudaError_t e = scratch_address(&base)) return cuda_status(e);
  char* b = static_cast<char*>(base);
  int32_t* status = dev_status;
  if (!status) {   // the shared status word must start at zero on every call
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

}  // extern "C"
