/*
 * fa_gb300.h -- C ABI of the exact tiled attention library for one NVIDIA GB300
 * (sm_103a).
 *
 * The library computes exact scaled-dot-product attention with online softmax:
 *
 *   S = scale * Q K^T,   P = softmax(S) row by row,   O = P V
 *
 * as defined in "FlashAttention: how a memory trick unlocked today's giant AI
 * models" (khetwal.com), section "The Quadratic Memory Bottleneck" (the three
 * steps, with the scale written into the score step) and section "The Trick:
 * Online Softmax" (the softmax formula and the running max / running sum that
 * let it be computed one key tile at a time).  Following section "Tiling" and
 * the "FlashAttention (Conceptual)" listing, query tiles of 128 rows stream key
 * and value tiles of 128 rows through on-chip memory; the N x N matrices S and P
 * are never written to device memory, so memory use is linear in N.  The
 * backward pass keeps only the per-row softmax statistic (the log-sum-exp) and
 * recomputes P from it ("How FlashAttention Eliminates Transformer Memory
 * Bottlenecks", galileo blog, Innovation #3).  Tiles that a causal or block mask
 * zeroes out are skipped (same blog, Innovation #5).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors Q, K, V, O, dO, dQ, dK, dV are contiguous [B, H, N, d], d fastest,
 *    in device memory owned by the caller.  LSE is contiguous [B, H, N] float32.
 *  - dtype FA_BF16: those tensors hold bfloat16; arithmetic is bf16 x bf16 with
 *    float32 accumulation, softmax in float32.  dtype FA_FP32 (forward only):
 *    float32 tensors, float32 arithmetic on CUDA cores.
 *  - d must be 64 or 128; B, H, N >= 0 (a call with B, H or N equal to 0 does
 *    nothing and returns FA_OK).  scale must be finite and > 0.
 *  - LSE[b,h,i] = max_j S_ij + ln(sum_j exp(S_ij - max_j S_ij)) over the keys row
 *    i sees (natural log, scale included).  A row that sees no key gets O = 0,
 *    LSE = -inf and dQ = 0.
 *  - causal != 0: query i sees key j only if j <= i.
 *  - kv_len (device, int32 [B], may be NULL): keys j >= kv_len[b] are masked for
 *    every query of sequence b (key padding).  Values are clamped to [0, N].
 *  - block_mask (device, uint8 [T, T] row-major with T = ceil(N / 128), may be
 *    NULL): query tile i sees key tile j only if block_mask[i*T + j] != 0.  One
 *    mask is shared by all B*H heads; masked tiles are skipped, kept tiles are
 *    computed in full.  The three masks combine by AND.
 *  - Pointers to the [B,H,N,d] tensors and to workspaces must be 16-byte aligned
 *    (the kernels move tiles with TMA); lse must be 4-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  All calls are
 *    asynchronous with respect to the host; they enqueue kernels on `stream` and
 *    return.  The library allocates no device memory.
 *
 * Errors: argument checks run on the host before anything is enqueued; a failed
 * check returns FA_ERR_INVALID_ARG or FA_ERR_UNSUPPORTED and launches nothing.
 * A CUDA error while encoding descriptors or launching returns FA_ERR_CUDA.
 * Every device-side wait is bounded; a wait that gives up records FA_ERR_TIMEOUT
 * in a device status word that fa_get_device_status() reads.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, negative size, bad scale, small workspace */
  FA_ERR_UNSUPPORTED = 2,  /* d not in {64,128}, unknown dtype, fp32 backward */
  FA_ERR_CUDA = 3,         /* CUDA runtime/driver error on the host side */
  FA_ERR_TIMEOUT = 4       /* a device-side wait gave up (reported by fa_get_device_status) */
} fa_status;

typedef enum { FA_BF16 = 0, FA_FP32 = 1 } fa_dtype;

/* Forward pass: O = softmax(scale * Q K^T) V and LSE, as defined above.
 * q, k, v: inputs [B,H,N,d]; o: output [B,H,N,d]; lse: output [B,H,N] float32.
 * One kernel launch.  The tiles of S live only in tensor memory and registers. */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, float scale, int causal,
                 const uint8_t* block_mask, const int32_t* kv_len, int dtype, void* stream);

/* Forward pass with 8-bit inputs (OCP FP8 E4M3: 1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits, largest finite value 448) and one scale per tensor.  The pages
 * quote an 8-bit forward only as a throughput figure ("How FlashAttention Bypasses
 * the GPU Memory Bottleneck to Enable Long-Context AI", factlen.com, the paragraphs
 * on FlashAttention-3 for Hopper: 8-bit floating point on H100); the arithmetic
 * below is this library's reading.
 * The attention inputs are Q = descale_q * q, K = descale_k * k, V = descale_v * v
 * where q, k, v are the E4M3 codes; the result is the forward of fa_fwd on those
 * values: O = softmax(scale * Q K^T) V (bf16) and LSE (float32), with the masks,
 * empty-row rule and LSE definition given above.
 *  - q, k: E4M3 [B, H, N, d], d fastest.
 *  - vt: E4M3 V transposed, [B, H, d, ldv]: vt[b,h,c,j] = v[b,h,j,c]; ldv (row stride
 *    in elements = bytes) must be >= N and a multiple of 16; columns j >= N are not
 *    read.
 *  - o: bf16 [B, H, N, d]; lse: float32 [B, H, N].
 *  - d must be 128 (anything else returns FA_ERR_UNSUPPORTED).  scale and the three
 *    descale factors must be finite and > 0.
 * Arithmetic: S = Q K^T and P V are 8-bit tensor-core products accumulated in float
 * registers of the tensor memory; the softmax is float32.  P (values in (0, 256],
 * relative to a row max that trails the true one by at most 8 log2 units) is rounded
 * to E4M3 for the P V product, which moves each probability by at most 2^-4 of
 * itself (2^-10 absolute below 2^-6); the row sum and LSE use the unrounded values.
 * O is therefore accurate to a few percent relative (not to bf16 precision); LSE is
 * as accurate as the score products.
 * One kernel launch; pointers 16-byte aligned (lse 4-byte); errors as for fa_fwd. */
fa_status fa_fwd_fp8(const void* q, const void* k, const void* vt, int ldv, void* o, float* lse,
                     int B, int H, int N, int d, float scale, float descale_q, float descale_k, float descale_v,
                     int causal, const uint8_t* block_mask, const int32_t* kv_len, void* stream);

/* Split-KV forward for short query blocks against long keys (decode and chunked
 * prefill).  Not on the pages: their kernels split work over query tiles, which
 * leaves most SMs idle when B*H*ceil(Nq/128) is small; this entry point also splits
 * the keys of each query tile into n_splits chunks processed in parallel and merges
 * the partial results by their log-sum-exp, which gives the same softmax over all keys
 * (the online-softmax rescaling of "The Trick: Online Softmax" applied across chunks
 * instead of across tiles).
 *  - q: bf16 [B, H, Nq, d]; k, v: bf16 [B, H, Nk, d] (Nq and Nk independent, either
 *    may exceed the other); o: bf16 [B, H, Nq, d]; lse: float32 [B, H, Nq].
 *  - No causal or block mask: every query row sees keys j < kv_len[b] (all Nk keys if
 *    kv_len is NULL; lengths clamped to [0, Nk]).  Rows that see no key get O = 0,
 *    LSE = -inf; so does every row when Nk = 0 (k and v may then be NULL).
 *  - d must be 128 (anything else returns FA_ERR_UNSUPPORTED).
 *  - n_splits: key chunks per 128-row query tile, 1..1024; each chunk of
 *    ceil(ceil(Nk/128) / n_splits) key tiles yields two partial results (its even and
 *    odd key tiles, processed side by side by one CTA).  fa_fwd_splitkv_pick_splits
 *    suggests a value for the current device.
 *  - workspace: caller-owned device memory of at least
 *    fa_fwd_splitkv_workspace_size(B, H, Nq, d, n_splits) bytes, 16-byte aligned:
 *    float32 partial O [2*n_splits, B*H, Nq, d] and partial LSE [2*n_splits, B*H, Nq].
 * Two kernel launches (partials, then the combine).  Errors as for fa_fwd. */
fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int Nq, int Nk, int d, float scale, const int32_t* kv_len,
                         int n_splits, void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes fa_fwd_splitkv needs (0 for an empty problem or n_splits < 1). */
size_t fa_fwd_splitkv_workspace_size(int B, int H, int Nq, int d, int n_splits);

/* A key-chunk count for fa_fwd_splitkv on the current device: about six CTAs per SM
 * for query blocks of at most 16 rows (decode), about half a CTA per SM otherwise; at
 * least two key tiles per chunk, at most 1024; 1 for empty shapes. */
int fa_fwd_splitkv_pick_splits(int B, int H, int Nq, int Nk);

/* Bytes of device workspace fa_bwd needs: D = rowsum(dO * O) (float32 [B,H,N])
 * and the float32 dQ accumulator [B,H,N,d], each 256-byte aligned.  Linear in N. */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/* Backward pass (bf16 only): given the forward's inputs, its outputs O and LSE and
 * the output gradient dO, writes dQ, dK, dV [B,H,N,d] for L = sum(O * dO):
 *   dP = dO V^T,  D_i = sum_c dO_ic O_ic,  dS = P * (dP - D),
 *   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO,
 * with P recomputed from Q, K and LSE.  The pages give no backward formulas; these
 * are the chain rule applied to the forward definition.  Keys that no query sees
 * get dK = dV = 0.  workspace: caller-owned device memory of at least
 * fa_bwd_workspace_size() bytes (contents on entry are ignored).
 * Equivalent to fa_bwd_preprocess + fa_bwd_main + fa_bwd_postprocess. */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                 int B, int H, int N, int d, float scale, int causal,
                 const uint8_t* block_mask, const int32_t* kv_len, int dtype, void* stream);

/* Backward stage 1: D = rowsum(dO * O) into the workspace and zero the float32 dQ
 * accumulator.  Memory-bound.  o, dout: bf16 [B,H,N,d]. */
fa_status fa_bwd_preprocess(const void* o, const void* dout, void* workspace, size_t workspace_bytes,
                            int B, int H, int N, int d, void* stream);

/* Backward stage 2: one CTA per 128-key tile recomputes P for every query tile that
 * sees it and accumulates dK, dV (written as bf16) and dQ (added into the workspace's
 * float32 accumulator by TMA reduce-add, cp.reduce.async.bulk.tensor .add, one 32x32
 * block at a time).  Needs stage 1 to have run on the same workspace. */
fa_status fa_bwd_main(const void* q, const void* k, const void* v, const float* lse, const void* dout,
                      void* dk, void* dv, void* workspace, size_t workspace_bytes,
                      int B, int H, int N, int d, float scale, int causal,
                      const uint8_t* block_mask, const int32_t* kv_len, void* stream);

/* Backward stage 3: dQ (bf16) = the float32 accumulator in the workspace. */
fa_status fa_bwd_postprocess(void* dq, const void* workspace, size_t workspace_bytes,
                             int B, int H, int N, int d, void* stream);

/* Size of the scratch array fa_bwd_noalloc uses: 64 MiB, held by every GPU that
 * loads this library until the process exits. */
#define FA_BWD_NOALLOC_MAX_BYTES (64u * 1024u * 1024u)

/* Backward pass for callers that cannot allocate device memory.  The pages have
 * no counterpart to this entry point: it is a deployment convenience.
 * Some callers are not allowed to allocate -- for example a plugin whose host
 * application owns all device memory and gives it no allocator, or a
 * latency-critical path where cudaMalloc's possible device synchronisation is
 * unacceptable.  This call takes the same arguments as fa_bwd minus the
 * workspace: its scratch (D and the float32 dQ accumulator) is a 64 MiB array
 * inside the library, so it calls no cudaMalloc, cudaFree or allocating routine.
 * Limits and behaviour:
 *  - returns FA_ERR_INVALID_ARG, launching nothing, when the problem needs more
 *    scratch than FA_BWD_NOALLOC_MAX_BYTES (that is, when
 *    fa_bwd_workspace_size(B,H,N,d) > FA_BWD_NOALLOC_MAX_BYTES; for d = 64 about
 *    258k query rows B*H*N, for d = 128 about 130k);
 *  - every call looks up the array's device address on the current device with
 *    cudaGetSymbolAddress (a host-side query that allocates nothing); the first
 *    call on a device may also load the library's module there, so make that
 *    first call before any stream capture;
 *  - every call on a device shares the one array and leaves its contents behind;
 *    the call clears what must start at zero itself, but calls whose work
 *    overlaps on the GPU (different streams, no ordering) race on the array and
 *    give wrong gradients -- order them on one stream or with events.
 * Other arguments, layouts and errors are those of fa_bwd. */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dout, void* dq, void* dk, void* dv,
                         int B, int H, int N, int d, float scale, int causal,
                         const uint8_t* block_mask, const int32_t* kv_len, int dtype, void* stream);

/* Synchronises `stream`, then returns and clears the device status word:
 * FA_OK, FA_ERR_TIMEOUT, or FA_ERR_CUDA if the synchronisation itself failed. */
fa_status fa_get_device_status(void* stream);

/* Failure-path self-test (no counterpart in the pages): enqueues one small
 * kernel whose bounded wait on a barrier that nothing arrives on gives up after
 * about one second and records FA_ERR_TIMEOUT in the device status word, exactly
 * as a stalled attention kernel would.  Nothing faults or hangs; a following
 * fa_get_device_status(stream) returns FA_ERR_TIMEOUT and clears the word. */
fa_status fa_selftest_wait_timeout(void* stream);

/* Static, human-readable name of a status code. */
const char* fa_status_string(int status);

/* Name of the last CUDA runtime error that made a call on this host thread return
 * FA_ERR_CUDA ("no error" if none).  Diagnostic only. */
const char* fa_last_cuda_error(void);

/* Library ABI version (major * 100 + minor). */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
