// Internal interface between the host entry points (fa_api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

constexpr int kTile = 128;  // query and key tile edge (rows)

// Arguments common to the attention kernels (forward and backward).
struct AttnArgs {
  int B, H, N, d;
  int n_tiles;                // ceil(N / 128)
  float scale;                // softmax scale
  float scale_log2;           // scale * log2(e): scores go straight to the exp2 domain
                              // (FP8 forward: times the scales of Q and K)
  float o_scale;              // factor on O / l (FP8 forward: the scale of V; otherwise 1)
  int causal;
  const uint8_t* block_mask;  // [n_tiles, n_tiles] or null
  const int32_t* kv_len;      // [B] or null
  unsigned int* status;       // device status word
  // Split-KV forward only (otherwise nk = N, nk_tiles = n_tiles, n_chunks = 0): N and
  // n_tiles count query rows and tiles, nk and nk_tiles key rows and tiles.  Each CTA
  // takes key tiles [c * chunk_tiles, (c + 1) * chunk_tiles) of one query tile and writes
  // two partial results (its even and its odd key tiles) for the combine kernel.
  int nk, nk_tiles;
  int n_chunks, chunk_tiles;
  float* part_o;              // [2 * n_chunks, B*H, N, d] float32, O of each partial (normalised)
  float* part_lse;            // [2 * n_chunks, B*H, N] float32, LSE of each partial (-inf: no key)
};

// Tensor maps for [B*H, N, d] bf16 tensors, boxes of 64 x 128 with 128-byte swizzle
// (FP8 forward: q, k E4M3 [B*H, N, 128] in 128 x 128 boxes, v the E4M3 V^T
// [B*H, 128, ldv] in 128-key x 128-row boxes, o bf16 as above).
struct FwdMaps {
  CUtensorMap q, k, v, o;
  void* o_ptr;  // O itself, for rows written with plain stores
};

struct BwdMaps {
  CUtensorMap q, k, v, dout, dk, dv;
  CUtensorMap dq_acc;  // float32 [B*H, N, d], 32 x 32 boxes, 128-byte swizzle (reduce-add target)
  CUtensorMap dk32, dv32;  // dK, dV again with 32 x 32 boxes and 64-byte swizzle (one warp's block)
};

// Launches `kernel` on `stream` with programmatic stream serialization, so that its CTAs
// may be scheduled while the previous kernel of the stream finishes (each kernel calls
// griddep_wait before touching global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Records `e` as this host thread's last CUDA error (read by fa_last_cuda_error) and
// returns the public status for it: FA_OK for cudaSuccess, FA_ERR_CUDA otherwise.
int cuda_status(cudaError_t e);

// Streaming multiprocessors of the current device (cached after the first call).
int sm_count();

// Raises a kernel's dynamic shared memory limit to `bytes` once per (kernel, device), so
// that repeated launches (and launches under stream capture) make no attribute call.
cudaError_t ensure_smem_limit(const void* kernel, int bytes);

cudaError_t launch_fwd_bf16(const FwdMaps& maps, float* lse, const AttnArgs& a, cudaStream_t stream);

cudaError_t launch_fwd_fp8(const FwdMaps& maps, float* lse, const AttnArgs& a, cudaStream_t stream);

// Split-KV forward (d = 128, bf16): the partial pass then the combine kernel.
cudaError_t launch_fwd_splitkv(const FwdMaps& maps, void* o, float* lse, const AttnArgs& a, cudaStream_t stream);

cudaError_t launch_fwd_fp32(const float* q, const float* k, const float* v, float* o, float* lse,
                            const AttnArgs& a, cudaStream_t stream);

cudaError_t launch_bwd_preprocess(const void* o, const void* dout, float* dsum, float* dq_acc,
                                  const AttnArgs& a, cudaStream_t stream);

cudaError_t launch_bwd_main_bf16(const BwdMaps& maps, const float* lse, const float* dsum, const AttnArgs& a,
                                 cudaStream_t stream);

cudaError_t launch_wait_timeout_selftest(unsigned int* status, cudaStream_t stream);

cudaError_t launch_bwd_postprocess(const float* dq_acc, void* dq, const AttnArgs& a, cudaStream_t stream);

}  // namespace fa
