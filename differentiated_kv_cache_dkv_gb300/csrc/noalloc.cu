// noalloc.cu -- dkv_compact_noalloc: the compaction call for callers that
// cannot allocate device memory themselves.
//
// dkv_compact needs a scratch workspace from its caller.  Some callers have
// no way to provide one: an engine whose device memory is entirely reserved
// up front by its own pool allocator, or a caller (a plugin, a different
// language runtime) that has no device allocator at all.  This entry point
// takes its scratch from a file-scope __device__ array of fixed size instead,
// so the caller passes only its inputs and outputs.  The array lives in every
// GPU that loads the library until the process exits.
//
// This convenience has no counterpart in the DiffKV paper.
#include <cuda_runtime.h>


#include "dkv_internal.cuh"

namespace {

constexpr size_t kScratchBytes = DKV_NOALLOC_SCRATCH_BYTES;

// Shared by every call on a device; contents are scratch (dkv_compact resets
// all it relies on at the start of each call).
__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch in the current context (host code cannot use
// the symbol's own address: it names a host-side stand-in).  Resolved on every
// call: after cudaDeviceReset, or in another context on the same device, the
// module is loaded again and the address can change; the lookup is cheap next
// to the launches it precedes.
cudaError_t scratch_address(void **out) {
  void *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" {

int32_t dkv_compact_noalloc(const dkv_batch *b, const dkv_params *p, const dkv_pool *pool, const dkv_tables *t,
                            void *stream) {
  size_t need = 0;
  if (dkv_workspace_size(b, &need) != DKV_OK) return DKV_E_INVAL;
  if (need > kScratchBytes) return DKV_E_INVAL;  // batch too large for the built-in scratch
  void *ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return DKV_E_CUDA;
  return dkv_compact(b, p, pool, t, ws, kScratchBytes, stream);
}

}  // extern "C"
