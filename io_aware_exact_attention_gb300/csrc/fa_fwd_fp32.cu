// Forward pass for float32 inputs, on CUDA cores in float32 arithmetic.
//
// Same tiled online-softmax schedule as the bf16 kernel ("FlashAttention
// (Conceptual)" listing, khetwal.com), sized for true fp32 accuracy: tensor-core
// tf32 would round Q and K to 10 mantissa bits.  A CTA of 128 threads owns 32
// query rows; four adjacent lanes share a row, each holding a quarter of its q
// and output columns (interleaved in float4 groups so shared-memory reads are
// conflict-free).  Keys and values stream through shared memory in chunks of 32;
// per chunk the row max is updated once, the accumulator rescaled once, and the
// chunk's exp-weighted values added.
#include <math.h>

#include "fa_internal.h"
#include "fa_tiles.cuh"

namespace fa {
namespace {

constexpr int kRows = 32;    // query rows per CTA
constexpr int kChunk = 32;   // keys per shared-memory chunk
constexpr int kThreads = 128;

template <int D>
__global__ void __launch_bounds__(kThreads)
    fwd_fp32_kernel(const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
                    float* __restrict__ o, float* __restrict__ lse_out, const AttnArgs a) {
  constexpr int G = D / 16;  // float4 groups per thread
  __shared__ __align__(16) float ks[kChunk][D];
  __shared__ __align__(16) float vs[kChunk][D];

  const int head = blockIdx.y;
  const int b = head / a.H;
  const int N = a.N;
  const int row0 = blockIdx.x * kRows;
  const int lane = threadIdx.x & 31;
  const int r = (threadIdx.x >> 2);  // row within the CTA (0..31)
  const int g = threadIdx.x & 3;     // quarter of the columns
  const int i = row0 + r;
  const bool row_ok = i < N;
  const int kv_len = clamp_kv_len(a.kv_len, b, N);
  const size_t base = static_cast<size_t>(head) * N * D;
  const int qtile = row0 / kTile;  // the 32 rows lie in one 128-row tile

  float4 qv[G], acc[G];
#pragma unroll
  for (int t = 0; t < G; ++t) {
    const int c = 4 * (g + 4 * t);
    qv[t] = row_ok ? *reinterpret_cast<const float4*>(q + base + static_cast<size_t>(i) * D + c)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    acc[t] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float m_run = -INFINITY, l_run = 0.f;
  const int last_row = min(row0 + kRows, N) - 1;
  int key_end = kv_len;
  if (a.causal) key_end = min(key_end, last_row + 1);

  for (int j0 = 0; j0 < key_end; j0 += kChunk) {
    if (a.block_mask != nullptr && a.block_mask[qtile * a.n_tiles + j0 / kTile] == 0) continue;
    __syncthreads();
    for (int e = threadIdx.x; e < kChunk * D / 4; e += kThreads) {
      const int jj = e / (D / 4), c = 4 * (e % (D / 4));
      const int j = j0 + jj;
      float4 kx = make_float4(0.f, 0.f, 0.f, 0.f), vx = kx;
      if (j < N) {
        kx = *reinterpret_cast<const float4*>(k + base + static_cast<size_t>(j) * D + c);
        vx = *reinterpret_cast<const float4*>(v + base + static_cast<size_t>(j) * D + c);
      }
      *reinterpret_cast<float4*>(&ks[jj][c]) = kx;
      *reinterpret_cast<float4*>(&vs[jj][c]) = vx;
    }
    __syncthreads();
    float s[kChunk];
    float mx = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < kChunk; ++jj) {
      float part = 0.f;
#pragma unroll
      for (int t = 0; t < G; ++t) {
        const float4 kx = *reinterpret_cast<const float4*>(&ks[jj][4 * (g + 4 * t)]);
        part = fmaf(qv[t].x, kx.x, part);
        part = fmaf(qv[t].y, kx.y, part);
        part = fmaf(qv[t].z, kx.z, part);
        part = fmaf(qv[t].w, kx.w, part);
      }
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      const int j = j0 + jj;
      const bool vis = j < kv_len && (!a.causal || j <= i);
      s[jj] = vis ? part * a.scale : -INFINITY;
      mx = fmaxf(mx, s[jj]);
    }
    const float m_new = fmaxf(m_run, mx);
    if (m_new == -INFINITY) continue;  // nothing visible for this row yet
    const float alpha = expf(m_run - m_new);
    l_run *= alpha;
#pragma unroll
    for (int t = 0; t < G; ++t) {
      acc[t].x *= alpha; acc[t].y *= alpha; acc[t].z *= alpha; acc[t].w *= alpha;
    }
#pragma unroll
    for (int jj = 0; jj < kChunk; ++jj) {
      const float p = expf(s[jj] - m_new);
      l_run += p;
#pragma unroll
      for (int t = 0; t < G; ++t) {
        const float4 vx = *reinterpret_cast<const float4*>(&vs[jj][4 * (g + 4 * t)]);
        acc[t].x = fmaf(p, vx.x, acc[t].x);
        acc[t].y = fmaf(p, vx.y, acc[t].y);
        acc[t].z = fmaf(p, vx.z, acc[t].z);
        acc[t].w = fmaf(p, vx.w, acc[t].w);
      }
    }
    m_run = m_new;
  }
  (void)lane;
  if (!row_ok) return;
  const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
  for (int t = 0; t < G; ++t) {
    const float4 y = make_float4(acc[t].x * inv_l, acc[t].y * inv_l, acc[t].z * inv_l, acc[t].w * inv_l);
    *reinterpret_cast<float4*>(o + base + static_cast<size_t>(i) * D + 4 * (g + 4 * t)) = y;
  }
  if (g == 0) lse_out[static_cast<size_t>(head) * N + i] = l_run > 0.f ? m_run + logf(l_run) : -INFINITY;
}

}  // namespace

cudaError_t launch_fwd_fp32(const float* q, const float* k, const float* v, float* o, float* lse,
                            const AttnArgs& a, cudaStream_t stream) {
  dim3 grid((a.N + kRows - 1) / kRows, a.B * a.H);
  if (a.d == 64)
    fwd_fp32_kernel<64><<<grid, kThreads, 0, stream>>>(q, k, v, o, lse, a);
  else
    fwd_fp32_kernel<128><<<grid, kThreads, 0, stream>>>(q, k, v, o, lse, a);
  return cudaGetLastError();
}

}  // namespace fa
