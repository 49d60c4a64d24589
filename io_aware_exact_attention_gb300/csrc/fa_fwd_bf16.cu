// Forward pass, bf16 in / fp32 accumulate, on the fifth-generation tensor cores.
//
// One CTA owns one 128-row query tile Q_i of one (batch, head) and streams the
// key/value tiles K_j, V_j it may see, as in the "FlashAttention (Conceptual)"
// listing of "FlashAttention: how a memory trick unlocked..." (khetwal.com): per
// key tile it forms the score block, updates the running row max and row sum,
// rescales the output accumulator and adds P V ("The Trick: Online Softmax").
// The GB300 mapping:
//   warp 0       TMA producer: Q_i once, then K_j/V_j into a ring of shared-memory
//                stages (128-byte swizzle), skipping tiles the masks zero out;
//   warp 1       allocates tensor memory and issues tcgen05.mma:
//                  S_j = Q_i K_j^T into one of two TMEM score buffers, then
//                  O  += P_j V_j into the TMEM output accumulator;
//   warps 2..5   softmax: each thread owns one query row (one TMEM lane), reads its
//                score row, masks, takes the max, exponentiates with exp2 (log2(e)
//                folded into the scale), writes P (bf16) to shared memory, rescales
//                O in TMEM when the row max grew, and finally writes O / l (bf16,
//                by TMA) and LSE = m + ln l (fp32).
// The score MMA of tile j+1 is issued before P_j V_j, so the exponentials of one
// tile overlap the tensor-core work of its neighbour.  S and P never reach HBM.
#include "fa_internal.h"
#include "fa_tiles.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kFwdThreads = 192;
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct FwdLayout {
  static constexpr int kStages = D == 64 ? 3 : 2;
  static constexpr int kTileBytes = kTile * D * 2;  // one 128-row tile of Q, K or V (bf16)
  static constexpr int kSubBytes = kTile * 64 * 2;  // one 64-column swizzle sub-tile
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kP = kV + kStages * kTileBytes;
  static constexpr int kEnd = kP + kTile * kTile * 2;
  static constexpr int kSmemBytes = kEnd + 1024;  // slack for aligning the base to 1024
  static constexpr uint32_t kColS = 0;            // two score buffers: columns [0,128), [128,256)
  static constexpr uint32_t kColO = 256;          // output accumulator: columns [256, 256 + D)
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

template <int D>
struct FwdBarriers {
  uint64_t q_full;
  uint64_t kv_full[FwdLayout<D>::kStages];
  uint64_t kv_empty[FwdLayout<D>::kStages];
  uint64_t s_full[2];
  uint64_t s_empty[2];
  uint64_t p_full;
  uint64_t o_done;
  uint64_t drain;
};

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    float* __restrict__ lse_out, const AttnArgs a) {
  using L = FwdLayout<D>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) FwdBarriers<D> bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = a.n_tiles;
  const int head = blockIdx.x / T;  // b * H + h
  const int qt = a.causal ? (T - 1 - static_cast<int>(blockIdx.x % T)) : static_cast<int>(blockIdx.x % T);
  const int b = head / a.H;
  const int kv_len = clamp_kv_len(a.kv_len, b, a.N);
  const WaitCtx wc{&abort_flag, a.status};

  uint8_t* smQ = smem + L::kQ;
  uint8_t* smK = smem + L::kK;
  uint8_t* smV = smem + L::kV;
  uint8_t* smP = smem + L::kP;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar.q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&bar.kv_full[s], 1);
      mbar_init(&bar.kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar.s_full[s], 1);
      mbar_init(&bar.s_empty[s], 128);
    }
    mbar_init(&bar.p_full, 128);
    mbar_init(&bar.o_done, 1);
    mbar_init(&bar.drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&bar.q_full, L::kTileBytes);
      for (int h = 0; h < D / 64; ++h)
        tma_load_3d(smQ + h * L::kSubBytes, &tm_q, &bar.q_full, h * 64, qt * kTile, head);
      int it = 0;
      bool ok = true;
      for (int kt = next_key_tile(qt, 0, kv_len, a.causal, a.block_mask, T); kt < T;
           kt = next_key_tile(qt, kt + 1, kv_len, a.causal, a.block_mask, T), ++it) {
        const int s = it % S;
        if (it >= S && !(ok = mbar_wait(&bar.kv_empty[s], ((it / S) - 1) & 1, wc))) break;
        mbar_arrive_expect_tx(&bar.kv_full[s], 2 * L::kTileBytes);
        for (int h = 0; h < D / 64; ++h) {
          tma_load_3d(smK + s * L::kTileBytes + h * L::kSubBytes, &tm_k, &bar.kv_full[s], h * 64, kt * kTile, head);
          tma_load_3d(smV + s * L::kTileBytes + h * L::kSubBytes, &tm_v, &bar.kv_full[s], h * 64, kt * kTile, head);
        }
      }
      if (!ok) {
        // let the loads already issued land before the CTA can exit
        mbar_drain(&bar.q_full, 0, 100000000ull);
        for (int j = (it > S ? it - S : 0); j < it; ++j) mbar_drain(&bar.kv_full[j % S], (j / S) & 1, 100000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, false, true);
      const uint32_t q0 = smem_u32(smQ), k0 = smem_u32(smK), v0 = smem_u32(smV), p0 = smem_u32(smP);
      bool ok = mbar_wait(&bar.q_full, 0, wc);
      int it = 0;
      auto issue_pv = [&](int t) -> bool {
        if (!mbar_wait(&bar.p_full, t & 1, wc)) return false;
        tc_fence_after();
        const uint32_t vs = v0 + (t % S) * L::kTileBytes;
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k) {
          const uint64_t ad = sdesc_sw128(p0 + (k / 4) * L::kSubBytes + (k % 4) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(vs + k * 2048, L::kSubBytes, 1024);
          mma_bf16_ss(tmem + L::kColO, ad, bd, idesc_o, (t > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(&bar.o_done);
        mma_commit(&bar.kv_empty[t % S]);
        return true;
      };
      if (ok) {
        for (int kt = next_key_tile(qt, 0, kv_len, a.causal, a.block_mask, T); kt < T;
             kt = next_key_tile(qt, kt + 1, kv_len, a.causal, a.block_mask, T), ++it) {
          const int s = it % S;
          const int buf = it & 1;
          if (!(ok = mbar_wait(&bar.kv_full[s], (it / S) & 1, wc))) break;
          if (it >= 2 && !(ok = mbar_wait(&bar.s_empty[buf], ((it >> 1) - 1) & 1, wc))) break;
          tc_fence_after();
          const uint32_t ks = k0 + s * L::kTileBytes;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint64_t ad = sdesc_sw128(q0 + (k / 4) * L::kSubBytes + (k % 4) * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(ks + (k / 4) * L::kSubBytes + (k % 4) * 32, 16, 1024);
            mma_bf16_ss(tmem + L::kColS + buf * 128, ad, bd, idesc_s, k > 0 ? 1u : 0u);
          }
          mma_commit(&bar.s_full[buf]);
          if (it >= 1 && !(ok = issue_pv(it - 1))) break;
        }
        if (ok && it >= 1) ok = issue_pv(it - 1);
      }
      if (!ok) {
        mma_commit(&bar.drain);
        mbar_drain(&bar.drain, 0, 100000000ull);
      }
    }
  } else {
    // --------------------------------------------------- softmax + epilogue
    const int wq = warp & 3;  // TMEM lane quarter this warp may access
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const int q_row = qt * kTile + r;
    const float sl2 = a.scale_log2;
    float m_run = neg_inf();  // running max, log2 domain (already multiplied by scale*log2 e)
    float l_run = 0.f;        // running sum of exp2(s - m_run)
    bool ok = true;
    int it = 0;
    for (int kt = next_key_tile(qt, 0, kv_len, a.causal, a.block_mask, T); kt < T;
         kt = next_key_tile(qt, kt + 1, kv_len, a.causal, a.block_mask, T), ++it) {
      const int buf = it & 1;
      ok = mbar_wait(&bar.s_full[buf], (it >> 1) & 1, wc);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      float s[kTile];
#pragma unroll
      for (int c0 = 0; c0 < kTile; c0 += 32) {
        uint32_t t[32];
        tmem_ld32(tmem + lane_off + L::kColS + buf * 128 + c0, t);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c0 + i] = __uint_as_float(t[i]);
      }
      tc_fence_before();
      mbar_arrive(&bar.s_empty[buf]);

      // element mask: key padding tail, causal diagonal (N tail is covered by kv_len <= N)
      const int key0 = kt * kTile;
      if (key0 + kTile > kv_len || (a.causal && kt == qt)) {
        const int lim = a.causal ? min(kv_len, q_row + 1) : kv_len;  // keys [key0, lim) visible
#pragma unroll
        for (int c = 0; c < kTile; ++c)
          if (key0 + c >= lim) s[c] = neg_inf();
      }
      float mx = neg_inf();
#pragma unroll
      for (int c = 0; c < kTile; ++c) mx = fmaxf(mx, s[c]);
      const float m_new = fmaxf(m_run, mx * sl2);
      const float m_use = (m_new == neg_inf()) ? 0.f : m_new;
      const float alpha = ex2(m_run - m_use);
      uint32_t pk[kTile / 2];
      float rowsum = 0.f;
#pragma unroll
      for (int c = 0; c < kTile; c += 2) {
        const float p0 = ex2(fmaf(s[c], sl2, -m_use));
        const float p1 = ex2(fmaf(s[c + 1], sl2, -m_use));
        rowsum += p0 + p1;
        pk[c / 2] = pack_bf16x2(p0, p1);
      }
      l_run = l_run * alpha + rowsum;
      m_run = m_new;

      if (it >= 1) {
        // P_{j-1} V_{j-1} must have finished before O is rescaled and P is overwritten
        ok = mbar_wait(&bar.o_done, (it - 1) & 1, wc);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha < 1.f)) {
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t t[32];
            tmem_ld32(tmem + lane_off + L::kColO + c0, t);
#pragma unroll
            for (int i = 0; i < 32; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
            tmem_st32(tmem + lane_off + L::kColO + c0, t);
          }
        }
      }
      const uint32_t prow = smem_u32(smP);
#pragma unroll
      for (int g = 0; g < kTile / 8; ++g)
        st_shared_v4(prow + (g / 8) * L::kSubBytes + sw128_offset(r, g % 8), pk[4 * g], pk[4 * g + 1],
                     pk[4 * g + 2], pk[4 * g + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar.p_full);
    }

    // epilogue: O = O_acc / l (bf16, staged in the Q buffer, stored by TMA); LSE = m + ln l
    const int n_vis = it;
    bool have_o = ok && n_vis > 0;
    if (have_o) {
      ok = mbar_wait(&bar.o_done, (n_vis - 1) & 1, wc);
      have_o = __all_sync(0xffffffffu, ok);
      tc_fence_after();
    }
    const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
    const uint32_t orow = smem_u32(smQ);
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t t[32];
      if (have_o) {
        tmem_ld32(tmem + lane_off + L::kColO + c0, t);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) t[i] = 0u;
      }
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        w[i] = pack_bf16x2(__uint_as_float(t[2 * i]) * inv_l, __uint_as_float(t[2 * i + 1]) * inv_l);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st_shared_v4(orow + (c0 / 64) * L::kSubBytes + sw128_offset(r, ((c0 % 64) / 8) + q), w[4 * q],
                     w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
    fence_proxy_async_smem();
    named_barrier(1, 128);
    if (warp == 2 && lane == 0) {
      for (int h = 0; h < D / 64; ++h) tma_store_3d(&tm_o, smQ + h * L::kSubBytes, h * 64, qt * kTile, head);
      tma_store_commit();
      tma_store_wait_all();
    }
    if (q_row < a.N) {
      const float lse = (n_vis > 0 && l_run > 0.f) ? (m_run + log2f(l_run)) * kLn2 : neg_inf();
      lse_out[static_cast<size_t>(head) * a.N + q_row] = lse;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int D>
cudaError_t launch_fwd_d(const FwdMaps& maps, float* lse, const AttnArgs& a, cudaStream_t stream) {
  using L = FwdLayout<D>;
  static bool configured = false;  // attribute set once per process (host-side, idempotent)
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fwd_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const long long grid = static_cast<long long>(a.n_tiles) * a.B * a.H;
  fwd_bf16_kernel<D><<<static_cast<unsigned>(grid), kFwdThreads, L::kSmemBytes, stream>>>(maps.q, maps.k, maps.v,
                                                                                         maps.o, lse, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdMaps& maps, float* lse, const AttnArgs& a, cudaStream_t stream) {
  return a.d == 64 ? launch_fwd_d<64>(maps, lse, a, stream) : launch_fwd_d<128>(maps, lse, a, stream);
}

}  // namespace fa
