// Host side of the C ABI declared in include/fa_gb300.h: argument checks, TMA
// descriptor encoding, workspace carving and kernel launches on the caller's
// stream.  No device memory is allocated here; the only device state is one
// status word per device (a __device__ variable) that bounded waits write to.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/fa_gb300.h"
#include "fa_internal.h"

namespace {

__device__ unsigned int g_fa_status = 0u;

constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 1024;  // split-KV: key chunks per query tile
constexpr float kLog2e = 1.44269504088896340736f;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0u; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0u; }

size_t round256(size_t x) { return (x + 255u) & ~size_t(255u); }

// Checks shared by every entry point.  `empty` is set when there is nothing to do.
fa_status check_shape(int B, int H, int N, int d, bool* empty) {
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  *empty = (B == 0 || H == 0 || N == 0);
  if (*empty) return FA_OK;
  const long long bh = static_cast<long long>(B) * H;
  const long long tiles = (static_cast<long long>(N) + fa::kTile - 1) / fa::kTile;
  if (bh > INT_MAX || tiles * bh > INT_MAX) return FA_ERR_INVALID_ARG;  // one CTA per (tile, head)
  if (bh * N > (1LL << 40)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

fa_status check_scale(float scale) {
  if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

// Address of this device's status word (looked up once per device).
unsigned int* status_word() {
  static unsigned int* addr[kMaxDevices] = {};
  static std::mutex mu;
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_status) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned int*>(p);
  }
  return addr[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [B*H, N, d] bf16 tensor, boxes of 64 columns x 128 rows, 128-byte swizzle.
// Rows past N read as zero and are not written.
bool encode_bf16(CUtensorMap* map, const void* base, int BH, int N, int d) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(fa::kTile), 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [B*H, N, d] bf16 tensor, boxes of 32 columns x 32 rows with 64-byte swizzle (the
// block one warp of the d = 64 backward writes of dK or dV).
bool encode_bf16_block32(CUtensorMap* map, const void* base, int BH, int N, int d) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 8-bit [B*H, rows, cols] tensor with row stride ld >= cols bytes, boxes of 128 x 128
// with 128-byte swizzle.  Columns past `cols` and rows past `rows` read as zero.
bool encode_u8(CUtensorMap* map, const void* base, int BH, int rows, int cols, int ld) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld), static_cast<cuuint64_t>(rows) * ld};
  const cuuint32_t box[3] = {128, 128, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// float32 [B*H, N, d] tensor (the dQ accumulator), boxes of 32 x 32 with 128-byte
// swizzle; the backward kernel reduce-adds 32x32 blocks into it.
bool encode_f32_acc(CUtensorMap* map, const void* base, int BH, int N, int d) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(N) * d * 4};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

fa::AttnArgs make_args(int B, int H, int N, int d, float scale, int causal, const uint8_t* block_mask,
                       const int32_t* kv_len) {
  fa::AttnArgs a;
  a.B = B;
  a.H = H;
  a.N = N;
  a.d = d;
  a.n_tiles = (N + fa::kTile - 1) / fa::kTile;
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.o_scale = 1.f;
  a.nk = N;
  a.nk_tiles = a.n_tiles;
  a.n_chunks = 0;
  a.chunk_tiles = 0;
  a.part_o = nullptr;
  a.part_lse = nullptr;
  a.causal = causal ? 1 : 0;
  a.block_mask = block_mask;
  a.kv_len = kv_len;
  a.status = status_word();
  return a;
}

struct Workspace {
  float* dsum;
  float* dq_acc;
};

size_t workspace_bytes_for(int B, int H, int N, int d) {
  const size_t rows = static_cast<size_t>(B) * H * N;
  return round256(rows * sizeof(float)) + round256(rows * d * sizeof(float));
}

Workspace carve(void* ws, int B, int H, int N) {
  const size_t rows = static_cast<size_t>(B) * H * N;
  char* p = static_cast<char*>(ws);
  return Workspace{reinterpret_cast<float*>(p), reinterpret_cast<float*>(p + round256(rows * sizeof(float)))};
}

thread_local cudaError_t t_last_cuda_error = cudaSuccess;

fa_status launch_status(cudaError_t e) {
  if (e == cudaSuccess) return FA_OK;
  t_last_cuda_error = e;
  return FA_ERR_CUDA;
}

}  // namespace

namespace fa {
int cuda_status(cudaError_t e) { return launch_status(e); }

cudaError_t ensure_smem_limit(const void* kernel, int bytes) {
  struct Entry {
    const void* kernel;
    int device, bytes;
  };
  static std::vector<Entry> done;
  static std::mutex mu;
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : done)
    if (e.kernel == kernel && e.device == dev && e.bytes >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.push_back({kernel, dev, bytes});
  return e;
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n = 152;
  }
  return n;
}
}  // namespace fa

extern "C" {

int fa_version(void) { return 100; }

const char* fa_last_cuda_error(void) { return cudaGetErrorString(t_last_cuda_error); }

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    default: return "FA_ERR_UNKNOWN";
  }
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, const uint8_t* block_mask, const int32_t* kv_len, int dtype, void* stream) {
  bool empty = false;
  fa_status st = check_shape(B, H, N, d, &empty);
  if (st != FA_OK) return st;
  if (dtype != FA_BF16 && dtype != FA_FP32) return FA_ERR_UNSUPPORTED;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (empty) return FA_OK;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse)) return FA_ERR_INVALID_ARG;
  const fa::AttnArgs a = make_args(B, H, N, d, scale, causal, block_mask, kv_len);
  if (a.status == nullptr) return FA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == FA_FP32)
    return launch_status(fa::launch_fwd_fp32(static_cast<const float*>(q), static_cast<const float*>(k),
                                             static_cast<const float*>(v), static_cast<float*>(o), lse, a, s));
  fa::FwdMaps maps;
  const int BH = B * H;
  if (!encode_bf16(&maps.q, q, BH, N, d) || !encode_bf16(&maps.k, k, BH, N, d) || !encode_bf16(&maps.v, v, BH, N, d) ||
      !encode_bf16(&maps.o, o, BH, N, d))
    return FA_ERR_CUDA;
  maps.o_ptr = o;
  return launch_status(fa::launch_fwd_bf16(maps, lse, a, s));
}

fa_status fa_fwd_fp8(const void* q, const void* k, const void* vt, int ldv, void* o, float* lse, int B, int H, int N,
                     int d, float scale, float descale_q, float descale_k, float descale_v, int causal,
                     const uint8_t* block_mask, const int32_t* kv_len, void* stream) {
  bool empty = false;
  fa_status st = check_shape(B, H, N, d, &empty);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if ((st = check_scale(scale)) != FA_OK || (st = check_scale(descale_q)) != FA_OK ||
      (st = check_scale(descale_k)) != FA_OK || (st = check_scale(descale_v)) != FA_OK)
    return st;
  const float sl2 = scale * descale_q * descale_k * kLog2e;
  if (!(sl2 > 0.f) || !std::isfinite(sl2)) return FA_ERR_INVALID_ARG;
  if (empty) return FA_OK;
  if (ldv < N || ldv % 16 != 0) return FA_ERR_INVALID_ARG;
  if (!q || !k || !vt || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o) || !aligned4(lse)) return FA_ERR_INVALID_ARG;
  fa::AttnArgs a = make_args(B, H, N, d, scale, causal, block_mask, kv_len);
  if (a.status == nullptr) return FA_ERR_CUDA;
  a.scale_log2 = sl2;
  a.o_scale = descale_v;
  fa::FwdMaps maps;
  const int BH = B * H;
  if (!encode_u8(&maps.q, q, BH, N, d, d) || !encode_u8(&maps.k, k, BH, N, d, d) ||
      !encode_u8(&maps.v, vt, BH, d, N, ldv) || !encode_bf16(&maps.o, o, BH, N, d))
    return FA_ERR_CUDA;
  maps.o_ptr = o;
  return launch_status(fa::launch_fwd_fp8(maps, lse, a, static_cast<cudaStream_t>(stream)));
}

size_t fa_fwd_splitkv_workspace_size(int B, int H, int Nq, int d, int n_splits) {
  if (B <= 0 || H <= 0 || Nq <= 0 || d <= 0 || n_splits <= 0) return 0;
  const size_t rows = static_cast<size_t>(B) * H * Nq * 2 * static_cast<size_t>(n_splits);
  return round256(rows * d * sizeof(float)) + round256(rows * sizeof(float));
}

int fa_fwd_splitkv_pick_splits(int B, int H, int Nq, int Nk) {
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0) return 1;
  const long long ctas_per_split = static_cast<long long>(B) * H * ((Nq + fa::kTile - 1) / fa::kTile);
  const long long key_tiles = (Nk + fa::kTile - 1) / fa::kTile;
  // The pass streams K and V from HBM.  With a few query rows the partial results are a
  // few hundred bytes, and six CTAs per SM keep more loads in flight (measured on the
  // 1-row, 32k-key decode shape: 1.05x over one CTA per SM).  A full 128-row block's
  // partials (2 x 64 KB per CTA) cost more than they hide, so half an SM's worth of
  // CTAs per split is enough there (128 rows x 32k keys: one split was fastest).
  const long long sms = fa::sm_count();
  const long long want = Nq <= 16 ? 6 * sms : sms / 2;
  long long n = (want + ctas_per_split - 1) / ctas_per_split;
  const long long most = (key_tiles + 1) / 2;  // two key tiles per CTA at least
  if (n > most) n = most;
  if (n > kMaxSplits) n = kMaxSplits;
  return static_cast<int>(n < 1 ? 1 : n);
}

fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                         int d, float scale, const int32_t* kv_len, int n_splits, void* workspace,
                         size_t workspace_bytes, void* stream) {
  bool empty = false;
  fa_status st = check_shape(B, H, Nq, d, &empty);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (Nk < 0 || n_splits < 1 || n_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (empty) return FA_OK;
  bool empty_k = false;
  if (Nk > 0 && (st = check_shape(B, H, Nk, d, &empty_k)) != FA_OK) return st;
  const long long grid = static_cast<long long>(B) * H * ((Nq + fa::kTile - 1) / fa::kTile) * n_splits;
  if (grid > INT_MAX) return FA_ERR_INVALID_ARG;
  if (!q || !o || !lse || !workspace || (Nk > 0 && (!k || !v))) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o) || !aligned4(lse) || !aligned16(workspace) ||
      (Nk > 0 && (!aligned16(k) || !aligned16(v))))
    return FA_ERR_INVALID_ARG;
  if (workspace_bytes < fa_fwd_splitkv_workspace_size(B, H, Nq, d, n_splits)) return FA_ERR_INVALID_ARG;
  fa::AttnArgs a = make_args(B, H, Nq, d, scale, 0, nullptr, kv_len);
  if (a.status == nullptr) return FA_ERR_CUDA;
  a.nk = Nk;
  a.nk_tiles = (Nk + fa::kTile - 1) / fa::kTile;
  a.n_chunks = n_splits;
  a.chunk_tiles = a.nk_tiles > 0 ? (a.nk_tiles + n_splits - 1) / n_splits : 0;
  const size_t parts_rows = static_cast<size_t>(B) * H * Nq * 2 * static_cast<size_t>(n_splits);
  a.part_o = static_cast<float*>(workspace);
  a.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + round256(parts_rows * d * sizeof(float)));
  fa::FwdMaps maps;
  const int BH = B * H;
  if (!encode_bf16(&maps.q, q, BH, Nq, d)) return FA_ERR_CUDA;
  if (Nk > 0 && (!encode_bf16(&maps.k, k, BH, Nk, d) || !encode_bf16(&maps.v, v, BH, Nk, d))) return FA_ERR_CUDA;
  maps.o = maps.q;  // not used by the partial pass
  maps.o_ptr = o;
  return launch_status(fa::launch_fwd_splitkv(maps, o, lse, a, static_cast<cudaStream_t>(stream)));
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0 || d <= 0) return 0;
  return workspace_bytes_for(B, H, N, d);
}

fa_status fa_bwd_preprocess(const void* o, const void* dout, void* workspace, size_t workspace_bytes, int B, int H,
                            int N, int d, void* stream) {
  bool empty = false;
  fa_status st = check_shape(B, H, N, d, &empty);
  if (st != FA_OK || empty) return st;
  if (!o || !dout || !workspace) return FA_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(dout) || !aligned16(workspace)) return FA_ERR_INVALID_ARG;
  if (workspace_bytes < workspace_bytes_for(B, H, N, d)) return FA_ERR_INVALID_ARG;
  const fa::AttnArgs a = make_args(B, H, N, d, 1.f, 0, nullptr, nullptr);
  const Workspace w = carve(workspace, B, H, N);
  return launch_status(fa::launch_bwd_preprocess(o, dout, w.dsum, w.dq_acc, a, static_cast<cudaStream_t>(stream)));
}

fa_status fa_bwd_main(const void* q, const void* k, const void* v, const float* lse, const void* dout, void* dk,
                      void* dv, void* workspace, size_t workspace_bytes, int B, int H, int N, int d, float scale,
                      int causal, const uint8_t* block_mask, const int32_t* kv_len, void* stream) {
  bool empty = false;
  fa_status st = check_shape(B, H, N, d, &empty);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (empty) return FA_OK;
  if (!q || !k || !v || !lse || !dout || !dk || !dv || !workspace) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned4(lse) || !aligned16(dout) || !aligned16(dk) ||
      !aligned16(dv) || !aligned16(workspace))
    return FA_ERR_INVALID_ARG;
  if (workspace_bytes < workspace_bytes_for(B, H, N, d)) return FA_ERR_INVALID_ARG;
  const fa::AttnArgs a = make_args(B, H, N, d, scale, causal, block_mask, kv_len);
  if (a.status == nullptr) return FA_ERR_CUDA;
  fa::BwdMaps maps;
  const int BH = B * H;
  if (!encode_bf16(&maps.q, q, BH, N, d) || !encode_bf16(&maps.k, k, BH, N, d) || !encode_bf16(&maps.v, v, BH, N, d) ||
      !encode_bf16(&maps.dout, dout, BH, N, d) || !encode_bf16(&maps.dk, dk, BH, N, d) ||
      !encode_bf16(&maps.dv, dv, BH, N, d))
    return FA_ERR_CUDA;
  const Workspace w = carve(workspace, B, H, N);
  if (!encode_f32_acc(&maps.dq_acc, w.dq_acc, BH, N, d)) return FA_ERR_CUDA;
  if (d == 64 && (!encode_bf16_block32(&maps.dk32, dk, BH, N, d) || !encode_bf16_block32(&maps.dv32, dv, BH, N, d)))
    return FA_ERR_CUDA;
  return launch_status(fa::launch_bwd_main_bf16(maps, lse, w.dsum, a, static_cast<cudaStream_t>(stream)));
}

fa_status fa_bwd_postprocess(void* dq, const void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                             void* stream) {
  bool empty = false;
  fa_status st = check_shape(B, H, N, d, &empty);
  if (st != FA_OK || empty) return st;
  if (!dq || !workspace || !aligned16(dq) || !aligned16(workspace)) return FA_ERR_INVALID_ARG;
  if (workspace_bytes < workspace_bytes_for(B, H, N, d)) return FA_ERR_INVALID_ARG;
  const fa::AttnArgs a = make_args(B, H, N, d, 1.f, 0, nullptr, nullptr);
  const Workspace w = carve(const_cast<void*>(workspace), B, H, N);
  return launch_status(fa::launch_bwd_postprocess(w.dq_acc, dq, a, static_cast<cudaStream_t>(stream)));
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                 float scale, int causal, const uint8_t* block_mask, const int32_t* kv_len, int dtype, void* stream) {
  bool empty = false;
  fa_status st = check_shape(B, H, N, d, &empty);
  if (st != FA_OK) return st;
  if (dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (empty) return FA_OK;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace))
    return FA_ERR_INVALID_ARG;
  if (workspace_bytes < workspace_bytes_for(B, H, N, d)) return FA_ERR_INVALID_ARG;
  if ((st = fa_bwd_preprocess(o, dout, workspace, workspace_bytes, B, H, N, d, stream)) != FA_OK) return st;
  if ((st = fa_bwd_main(q, k, v, lse, dout, dk, dv, workspace, workspace_bytes, B, H, N, d, scale, causal, block_mask,
                        kv_len, stream)) != FA_OK)
    return st;
  return fa_bwd_postprocess(dq, workspace, workspace_bytes, B, H, N, d, stream);
}

fa_status fa_selftest_wait_timeout(void* stream) {
  unsigned int* word = status_word();
  if (word == nullptr) return FA_ERR_CUDA;
  return launch_status(fa::launch_wait_timeout_selftest(word, static_cast<cudaStream_t>(stream)));
}

fa_status fa_get_device_status(void* stream) {
  unsigned int* word = status_word();
  if (word == nullptr) return FA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int value = 0;
  if (cudaMemcpyAsync(&value, word, sizeof(value), cudaMemcpyDeviceToHost, s) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaMemsetAsync(word, 0, sizeof(value), s) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
  return value == 0u ? FA_OK : static_cast<fa_status>(value);
}

}  // extern "C"
