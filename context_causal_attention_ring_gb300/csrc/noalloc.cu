// Forward entry point that allocates nothing.
//
// Some callers cannot call cudaMalloc: a plugin running inside a host
// program that owns the whole device-memory pool and hands its plugins no
// allocator, or a serving path that must never enter the allocator (no
// allocation latency, no out-of-memory failure in the middle of a request).
// They still own their inputs and outputs, but cannot provide the forward's
// fp32 workspace. This entry point takes that workspace from a fixed array in
// the library's own device image instead.
#include <cstring>
#include <string>

#include "kernels.h"

namespace {

// Fixed scratch for the forward workspace (the fp32 running output, or the
// Pass-Q partial slots). A device holds these bytes from the moment the
// library's device image is loaded on it (its first kernel launch or symbol
// lookup, under CUDA's lazy module loading) until the process exits.
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the current context. In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with the device current. The lookup runs on every call and allocates
// nothing: an address kept from an earlier call could belong to a context
// that has since been destroyed (cudaDeviceReset, or a host program that
// makes its own context current on the same device).
cp_attn_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return cpa::fail(CP_ATTN_ERR_CUDA, "forward_noalloc: no current CUDA device");
  }
  void* ptr = nullptr;
  const cudaError_t err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (err != cudaSuccess || ptr == nullptr) {
    cudaGetLastError();
    // the library's device image (and with it the array) is loaded on the
    // first call on each device; that load can run out of device memory
    const cp_attn_status st =
        err == cudaErrorMemoryAllocation ? CP_ATTN_ERR_OOM : CP_ATTN_ERR_CUDA;
    return cpa::fail(st, std::string("forward_noalloc: cudaGetSymbolAddress failed on device ") +
                             std::to_string(dev) + ": " + cudaGetErrorString(err));
  }
  *out = ptr;
  return CP_ATTN_OK;
}

}  // namespace

extern "C" {

size_t cp_attn_forward_noalloc_capacity(void) { return kNoAllocScratchBytes; }

cp_attn_status cp_attn_forward_noalloc(cp_attn_plan_t plan, const void* q, const void* k,
                                       const void* v, void* o, float* lse, void* stream) {
  cpa::clear_error();
  if (!plan) return cpa::fail(CP_ATTN_ERR_INVALID_ARG, "forward_noalloc: null plan");
  size_t need = 0;
  cp_attn_status st = cp_attn_workspace_size(plan, CP_ATTN_OP_FORWARD, &need);
  if (st != CP_ATTN_OK) return st;
  if (need > kNoAllocScratchBytes)
    return cpa::fail(CP_ATTN_ERR_SHAPE,
                     "forward_noalloc: the plan needs " + std::to_string(need) +
                         " bytes of forward workspace, more than the fixed " +
                         std::to_string(kNoAllocScratchBytes) +
                         " bytes; use cp_attn_forward with a caller-provided workspace");
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != CP_ATTN_OK) return st;
  // Nothing in the scratch needs clearing: step 0 (Pass KV) overwrites every
  // accumulator row and every Pass-Q step writes every row of its slot
  // before anything reads them.
  return cp_attn_forward(plan, q, k, v, o, lse, scratch, need, stream);
}

}  // extern "C"
