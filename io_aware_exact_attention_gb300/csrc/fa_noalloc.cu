// fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.
//
// fa_bwd needs a workspace (the per-row D values and the float32 dQ accumulator)
// that the caller allocates.  Some callers cannot: a plugin loaded into a host
// application that owns every device allocation and hands the plugin no allocator,
// or a latency-critical path where cudaMalloc (which may synchronise the device)
// is not allowed.  For them this entry point uses a scratch array that lives in
// the library itself: a file-scope __device__ array of FA_BWD_NOALLOC_MAX_BYTES,
// which every GPU that loads the library keeps until the process exits.
//
// The array's name in host code is only a host-side handle, not a device address.
// Every call looks the device address up with cudaGetSymbolAddress on the current
// device (a host-side query, no allocation) and passes it to the existing backward
// kernels like any caller-owned workspace.  Looking it up on every call rather than
// caching it keeps the address right after a device reset reloads the module.
// Nothing here calls cudaMalloc, cudaFree or any allocating library routine.
#include <cuda_runtime.h>

#include "../../include/fa_gb300.h"
#include "fa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[FA_BWD_NOALLOC_MAX_BYTES];

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                    const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                    float scale, int causal, const uint8_t* block_mask, const int32_t* kv_len,
                                    int dtype, void* stream) {
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || N == 0) {
    // nothing to compute; fa_bwd applies its own argument checks and launches nothing
    return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, nullptr, 0, B, H, N, d, scale, causal, block_mask, kv_len,
                  dtype, stream);
  }
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  if (need == 0 || need > static_cast<size_t>(FA_BWD_NOALLOC_MAX_BYTES)) return FA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&scratch, g_bwd_scratch);
  if (e != cudaSuccess) return static_cast<fa_status>(fa::cuda_status(e));
  if (scratch == nullptr) return static_cast<fa_status>(fa::cuda_status(cudaErrorInvalidSymbol));
  // fa_bwd's first stage writes D and zeroes the dQ accumulator in the scratch, so
  // whatever an earlier call left there is overwritten before it is read.
  return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, scratch, static_cast<size_t>(FA_BWD_NOALLOC_MAX_BYTES), B, H, N,
                d, scale, causal, block_mask, kv_len, dtype, stream);
}
