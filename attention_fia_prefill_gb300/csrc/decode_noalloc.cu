// fia_decode_no_alloc: incremental attention for callers that cannot allocate
// device memory.
//
// fia_decode needs a caller-provided workspace (the device status word, the
// split plan and the per-split partial results).  Some callers only ever hold
// the input and output buffers they were handed -- plugin hosts and inference
// servers that own the device memory budget, code that runs where a device
// allocation is forbidden or would break a fixed memory pool -- and cannot call
// cudaMalloc (or an allocating framework routine) to create one.  This entry
// point gives them fia_decode with the workspace taken from a fixed array that
// lives in the library itself.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes; every
// GPU that loads this library holds it until the process exits.  Nothing here
// calls cudaMalloc, cudaFree or any allocating routine.
#include "../../include/fia.h"

#include <cuda_runtime.h>

#include <cstdio>

#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the calling thread's current
// context.  In host code `g_decode_scratch` names a host-side stand-in, not
// device memory, so the address must come from cudaGetSymbolAddress with the
// target device current.  The address belongs to a CUDA context, not to a
// device index: a host that makes another context current (driver API) or
// resets the device gets a different one.  The lookup is therefore repeated
// on every call (it allocates nothing); the first call in a context also loads
// the library's kernels into it.
fia_status scratch_for_current_context(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    fia::set_last_error(FIA_ERR_CUDA, cudaGetErrorString(e));
    return FIA_ERR_CUDA;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_decode_scratch);
  if (e != cudaSuccess || p == nullptr) {
    fia::set_last_error(FIA_ERR_CUDA, e != cudaSuccess ? cudaGetErrorString(e) : "null scratch address");
    return FIA_ERR_CUDA;
  }
  *out = p;
  return FIA_OK;
}

}  // namespace

extern "C" fia_status fia_decode_no_alloc(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                                          const fia_tensor* query_rope, const fia_tensor* key_rope,
                                          const fia_tensor* block_table, const fia_tensor* atten_mask,
                                          const fia_params* params, const fia_tensor* attention_out,
                                          const fia_tensor* softmax_lse, void* stream) {
  size_t need = 0;
  fia_status st = fia_decode_get_workspace_size(query, key, value, query_rope, key_rope, block_table, atten_mask,
                                                params, attention_out, softmax_lse, &need);
  if (st != FIA_OK) return st;
  if (need > kNoAllocScratchBytes) {
    char msg[160];
    snprintf(msg, sizeof(msg), "fia_decode_no_alloc: this call needs %zu bytes of scratch, the built-in maximum is %zu",
             need, kNoAllocScratchBytes);
    fia::set_last_error(FIA_ERR_WORKSPACE, msg);
    return FIA_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  st = scratch_for_current_context(&ws);
  if (st != FIA_OK) return st;
  return fia_decode(query, key, value, query_rope, key_rope, block_table, atten_mask, params, attention_out,
                    softmax_lse, ws, kNoAllocScratchBytes, stream);
}
