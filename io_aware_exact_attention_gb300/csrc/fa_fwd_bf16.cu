// Forward pass, bf16 in / fp32 accumulate, on the fifth-generation tensor cores.
//
// One CTA owns two adjacent 128-row query tiles Q_a, Q_b of one (batch, head) and
// streams the key/value tiles K_j, V_j either may see, as in the "FlashAttention
// (Conceptual)" listing of "FlashAttention: how a memory trick unlocked..."
// (khetwal.com): per key tile it forms the score block, updates the running row
// max and row sum, rescales the output accumulator and adds P V ("The Trick:
// Online Softmax").  The GB300 mapping:
//   warp 0       TMA producer: both query tiles once, then K_j and V_j into a ring
//                of shared-memory stages (128-byte swizzle), skipping masked tiles;
//   warp 1       allocates tensor memory and issues tcgen05.mma:
//                  S_a = Q_a K_j^T, S_b = Q_b K_j^T into two TMEM score buffers,
//                  O_a += P_a V_j, O_b += P_b V_j with P read from TMEM (the score
//                  buffer it replaced) and V N-major straight from its TMA tile;
//   warps 2..5   softmax of tile a, warps 6..9 softmax of tile b: one thread per
//                query row (one TMEM lane) loads its score row, masks, takes the
//                max, exponentiates with exp2 (log2 e folded into the scale),
//                writes P as bf16 pairs back into TMEM, rescales O in TMEM when
//                needed, and at the end writes O / l (bf16, by TMA) and
//                LSE = m + ln l (fp32).
// While one softmax warpgroup exponentiates its tile, the tensor cores work on the
// other tile, so exp and MMA overlap.  The row max used for the exponentials is
// raised only when a tile's max exceeds it by more than kRescaleSlack (in log2
// units); the result is still exact because O and l always use the same max, and
// most tiles then skip the O rescale.  S and P never reach HBM.
#include "fa_internal.h"
#include "fa_tiles.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleSlack = 8.0f;  // P values stay below 2^8 before a rescale is forced

// NQ query tiles per CTA.  NQ = 2 (d = 128): one CTA per SM, the two tiles'
// softmax phases overlap each other's MMAs.  NQ = 1 (d = 64): a lighter CTA with
// 256 TMEM columns and ~81 KB of shared memory, so two CTAs share an SM and one
// CTA's set-up, loads and epilogue overlap the other's main loop.
template <int D, int NQ>
struct FwdLayout {
  static constexpr int kThreads = 64 + 128 * NQ;  // producer warp, MMA warp, one softmax warpgroup per tile
  static constexpr int kCtasPerSm = NQ == 1 ? 2 : 1;
  static constexpr int kStages = NQ == 1 ? 2 : (D == 64 ? 4 : 2);
  static constexpr int kTileBytes = kTile * D * 2;  // one 128-row tile of Q, K or V (bf16)
  static constexpr int kSubBytes = kTile * 64 * 2;  // one 64-column swizzle sub-tile
  static constexpr int kQ = 0;                      // NQ query tiles
  static constexpr int kK = kQ + NQ * kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kEnd = kV + kStages * kTileBytes;
  static constexpr int kSmemBytes = kEnd + 1024;  // slack for aligning the base to 1024
  static constexpr uint32_t kTmemCols = NQ == 1 ? 256 : 512;
  // TMEM columns: score/P buffer of tile i at 128*i, output accumulator of tile i after all score buffers
  __device__ static constexpr uint32_t col_s(int i) { return 128u * static_cast<uint32_t>(i); }
  __device__ static constexpr uint32_t col_o(int i) { return 128u * NQ + static_cast<uint32_t>(D * i); }
  static_assert(128 * NQ + D * NQ <= static_cast<int>(kTmemCols), "TMEM budget");
  static_assert(kSmemBytes <= (NQ == 1 ? 112 * 1024 : 227 * 1024), "shared memory budget");
};

template <int D, int NQ>
struct FwdBarriers {
  uint64_t q_full;
  uint64_t k_full[FwdLayout<D, NQ>::kStages];
  uint64_t v_full[FwdLayout<D, NQ>::kStages];
  uint64_t kv_empty[FwdLayout<D, NQ>::kStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t drain;
};

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// Key tile kt is loaded when either query tile of the CTA sees it.
__device__ __forceinline__ bool pair_sees(const int (&qt)[2], int kt, int kv_len, const AttnArgs& a) {
  if (tile_pair_visible(qt[0], kt, kv_len, a.causal, a.block_mask, a.n_tiles)) return true;
  return qt[1] < a.n_tiles && tile_pair_visible(qt[1], kt, kv_len, a.causal, a.block_mask, a.n_tiles);
}

__device__ __forceinline__ int next_union_tile(const int (&qt)[2], int kt, int kv_len, const AttnArgs& a) {
  while (kt < a.n_tiles && !pair_sees(qt, kt, kv_len, a)) ++kt;
  return kt;
}

template <int D, int NQ>
__global__ void __launch_bounds__(FwdLayout<D, NQ>::kThreads, FwdLayout<D, NQ>::kCtasPerSm)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    float* __restrict__ lse_out, const AttnArgs a) {
  using L = FwdLayout<D, NQ>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) FwdBarriers<D, NQ> bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = a.n_tiles;
  const int n_groups = (T + NQ - 1) / NQ;
  const int head = blockIdx.x / n_groups;  // b * H + h
  const int gr = static_cast<int>(blockIdx.x % n_groups);
  const int group = a.causal ? (n_groups - 1 - gr) : gr;  // causal: heaviest groups first
  const int qt[2] = {NQ * group, NQ == 2 ? 2 * group + 1 : T};  // qt[1] >= T: no second tile
  const bool has_b = qt[1] < T;
  const int b = head / a.H;
  const int kv_len = clamp_kv_len(a.kv_len, b, a.N);
  const WaitCtx wc{&abort_flag, a.status};

  uint8_t* smQ = smem + L::kQ;
  uint8_t* smK = smem + L::kK;
  uint8_t* smV = smem + L::kV;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar.q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&bar.k_full[s], 1);
      mbar_init(&bar.v_full[s], 1);
      mbar_init(&bar.kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.s_full[i], 1);
      mbar_init(&bar.p_full[i], 128);
      mbar_init(&bar.o_done[i], 1);
    }
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
      mbar_arrive_expect_tx(&bar.q_full, (has_b ? 2 : 1) * L::kTileBytes);
      for (int i = 0; i < (has_b ? 2 : 1); ++i)
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(smQ + i * L::kTileBytes + h * L::kSubBytes, &tm_q, &bar.q_full, h * 64, qt[i] * kTile, head);
      int u = 0;
      bool ok = true;
      for (int kt = next_union_tile(qt, 0, kv_len, a); kt < T; kt = next_union_tile(qt, kt + 1, kv_len, a), ++u) {
        const int s = u % S;
        if (u >= S && !(ok = mbar_wait(&bar.kv_empty[s], ((u / S) - 1) & 1, wc))) break;
        mbar_arrive_expect_tx(&bar.k_full[s], L::kTileBytes);
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(smK + s * L::kTileBytes + h * L::kSubBytes, &tm_k, &bar.k_full[s], h * 64, kt * kTile, head);
        mbar_arrive_expect_tx(&bar.v_full[s], L::kTileBytes);
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(smV + s * L::kTileBytes + h * L::kSubBytes, &tm_v, &bar.v_full[s], h * 64, kt * kTile, head);
      }
      if (!ok) {
        // let the loads already issued land before the CTA can exit
        mbar_drain(&bar.q_full, 0, 100000000ull);
        for (int j = (u > S ? u - S : 0); j < u; ++j) {
          mbar_drain(&bar.k_full[j % S], (j / S) & 1, 100000000ull);
          mbar_drain(&bar.v_full[j % S], (j / S) & 1, 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, false, true);
      const uint32_t q0 = smem_u32(smQ), k0 = smem_u32(smK), v0 = smem_u32(smV);
      bool ok = mbar_wait(&bar.q_full, 0, wc);
      int n[2] = {0, 0};  // P V products issued per query tile
      int u = 0;          // position in the union list of key tiles
      // S_i for key tile kt into tile i's TMEM buffer.  That buffer still holds P_i of the
      // last P V, which this thread issued earlier: MMAs from one thread execute in issue
      // order, so the new scores overwrite P only after that P V has read it.
      auto issue_scores = [&](int i, int kt_s, int stage) -> bool {
        tc_fence_after();
        const uint32_t qs = q0 + i * L::kTileBytes, ks = k0 + stage * L::kTileBytes;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k / 4) * L::kSubBytes + (k % 4) * 32;
          mma_bf16_ss(tmem + L::col_s(i), sdesc_sw128(qs + off, 16, 1024), sdesc_sw128(ks + off, 16, 1024), idesc_s,
                      k > 0 ? 1u : 0u);
        }
        mma_commit(&bar.s_full[i]);
        (void)kt_s;
        return true;
      };
      int kt = next_union_tile(qt, 0, kv_len, a);
      if (ok && kt < T) {
        ok = mbar_wait(&bar.k_full[0], 0, wc);
        for (int i = 0; ok && i < 2; ++i)
          if (i == 0 || has_b)
            if (tile_pair_visible(qt[i], kt, kv_len, a.causal, a.block_mask, T)) ok = issue_scores(i, kt, 0);
      }
      // Per key tile: P_i V for each tile i, and right after it tile i's scores for the
      // next key tile, so each softmax warpgroup gets its next scores without waiting
      // for the other tile.
      while (ok && kt < T) {
        const int s = u % S;
        const int kt_next = next_union_tile(qt, kt + 1, kv_len, a);
        bool f[2], fn[2];
        f[0] = tile_pair_visible(qt[0], kt, kv_len, a.causal, a.block_mask, T);
        f[1] = has_b && tile_pair_visible(qt[1], kt, kv_len, a.causal, a.block_mask, T);
        fn[0] = kt_next < T && tile_pair_visible(qt[0], kt_next, kv_len, a.causal, a.block_mask, T);
        fn[1] = kt_next < T && has_b && tile_pair_visible(qt[1], kt_next, kv_len, a.causal, a.block_mask, T);
        if (!(ok = mbar_wait(&bar.v_full[s], (u / S) & 1, wc))) break;
        const uint32_t vs = v0 + s * L::kTileBytes;
        bool next_k_ready = false;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (f[i]) {
            if (!(ok = mbar_wait(&bar.p_full[i], n[i] & 1, wc))) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < kTile / 16; ++k)
              mma_bf16_ts(tmem + L::col_o(i), tmem + L::col_s(i) + k * 8,
                          sdesc_sw128(vs + k * 2048, L::kSubBytes, 1024), idesc_o, (n[i] > 0 || k > 0) ? 1u : 0u);
            mma_commit(&bar.o_done[i]);
            ++n[i];
          }
          if (fn[i]) {
            if (!next_k_ready) {
              if (!(ok = mbar_wait(&bar.k_full[(u + 1) % S], ((u + 1) / S) & 1, wc))) break;
              next_k_ready = true;
            }
            if (!(ok = issue_scores(i, kt_next, (u + 1) % S))) break;
          }
        }
        if (!ok) break;
        mma_commit(&bar.kv_empty[s]);
        kt = kt_next;
        ++u;
      }
      if (!ok) {
        mma_commit(&bar.drain);
        mbar_drain(&bar.drain, 0, 100000000ull);
      }
    }
  } else {
    // --------------------------------------------------- softmax + epilogue
    const int wg = (warp - 2) >> 2;  // which query tile of the pair
    const int my_qt = qt[wg];
    const int wq = warp & 3;  // TMEM lane quarter this warp may access
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off + L::col_s(wg);
    const uint32_t t_o = tmem + lane_off + L::col_o(wg);
    const int q_row = my_qt * kTile + r;
    const float sl2 = a.scale_log2;
    if (my_qt < T) {
      float m_run = neg_inf();  // max used for the exponentials, log2 domain (scale * log2 e applied)
      float l_run = 0.f;        // running sum of exp2(s - m_run)
      bool ok = true;
      int n = 0;
      for (int kt = next_key_tile(my_qt, 0, kv_len, a.causal, a.block_mask, T); kt < T;
           kt = next_key_tile(my_qt, kt + 1, kv_len, a.causal, a.block_mask, T), ++n) {
        ok = mbar_wait(&bar.s_full[wg], n & 1, wc);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        float s[kTile];
#pragma unroll
        for (int c0 = 0; c0 < kTile; c0 += 64) {
          uint32_t t[64];
          tmem_ld64(t_s + c0, t);
#pragma unroll
          for (int i = 0; i < 64; ++i) s[c0 + i] = __uint_as_float(t[i]);
        }
        // element mask: key padding tail, causal diagonal (the N tail is covered by kv_len <= N)
        const int key0 = kt * kTile;
        if (key0 + kTile > kv_len || (a.causal && kt == my_qt)) {
          const int lim = a.causal ? min(kv_len, q_row + 1) : kv_len;  // keys [key0, lim) visible
#pragma unroll
          for (int c = 0; c < kTile; ++c)
            if (key0 + c >= lim) s[c] = neg_inf();
        }
        float mx0 = neg_inf(), mx1 = neg_inf();
#pragma unroll
        for (int c = 0; c < kTile; c += 4) {
          mx0 = fmax3(mx0, s[c], s[c + 1]);
          mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
        }
        const float mx = fmaxf(mx0, mx1) * sl2;
        const float m_new = (mx > m_run + kRescaleSlack) ? mx : m_run;
        const float m_use = (m_new == neg_inf()) ? 0.f : m_new;
        const float alpha = ex2(m_run - m_use);
        // all exponentials first (independent, so they overlap), then sums and packing;
        // scale-and-subtract and the sums run two lanes per instruction
#pragma unroll
        for (int c = 0; c < kTile; c += 2) {
          ffma2(s[c], s[c + 1], s[c], s[c + 1], sl2, -m_use);
          s[c] = ex2(s[c]);
          s[c + 1] = ex2(s[c + 1]);
        }
        float sum0 = 0.f, sum1 = 0.f, sum2 = 0.f, sum3 = 0.f;
#pragma unroll
        for (int c = 0; c < kTile; c += 4) {
          fadd2(sum0, sum1, s[c], s[c + 1]);
          fadd2(sum2, sum3, s[c + 2], s[c + 3]);
        }
        uint32_t pk[kTile / 2];
#pragma unroll
        for (int c = 0; c < kTile; c += 2) pk[c / 2] = pack_bf16x2(s[c], s[c + 1]);
        l_run = l_run * alpha + ((sum0 + sum1) + (sum2 + sum3));
        m_run = m_new;
        // P replaces S in the tile's TMEM buffer (bf16 pairs, columns [0, 64))
        tmem_st32(t_s, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
        tmem_st32(t_s + 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
        if (n > 0 && __any_sync(0xffffffffu, alpha < 1.f)) {
          // the previous P V must be done before O is rescaled
          ok = mbar_wait(&bar.o_done[wg], (n - 1) & 1, wc);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t t[32];
            tmem_ld32(t_o + c0, t);
#pragma unroll
            for (int i = 0; i < 32; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
            tmem_st32(t_o + c0, t);
          }
        }
        tc_fence_before();
        mbar_arrive(&bar.p_full[wg]);
      }

      // epilogue: O = O_acc / l (bf16, staged in this tile's Q buffer, stored by TMA); LSE = m + ln l
      bool have_o = ok && n > 0;
      if (have_o) {
        ok = mbar_wait(&bar.o_done[wg], (n - 1) & 1, wc);
        have_o = __all_sync(0xffffffffu, ok);
        tc_fence_after();
      }
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      uint8_t* stage = smQ + wg * L::kTileBytes;
      const uint32_t orow = smem_u32(stage);
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t t[32];
        if (have_o) {
          tmem_ld32(t_o + c0, t);
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
      named_barrier(1 + wg, 128);
      if (wq == 2 && lane == 0) {
        for (int h = 0; h < D / 64; ++h)
          tma_store_3d(&tm_o, stage + h * L::kSubBytes, h * 64, my_qt * kTile, head);
        tma_store_commit();
        tma_store_wait_all();
      }
      if (q_row < a.N) {
        const float lse = (n > 0 && l_run > 0.f) ? (m_run + log2f(l_run)) * kLn2 : neg_inf();
        lse_out[static_cast<size_t>(head) * a.N + q_row] = lse;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int D, int NQ>
cudaError_t launch_fwd_d(const FwdMaps& maps, float* lse, const AttnArgs& a, cudaStream_t stream) {
  using L = FwdLayout<D, NQ>;
  cudaError_t e = cudaFuncSetAttribute(fwd_bf16_kernel<D, NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       L::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>((a.n_tiles + NQ - 1) / NQ) * a.B * a.H;
  fwd_bf16_kernel<D, NQ><<<static_cast<unsigned>(grid), L::kThreads, L::kSmemBytes, stream>>>(maps.q, maps.k, maps.v,
                                                                                             maps.o, lse, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdMaps& maps, float* lse, const AttnArgs& a, cudaStream_t stream) {
  return a.d == 64 ? launch_fwd_d<64, 1>(maps, lse, a, stream) : launch_fwd_d<128, 2>(maps, lse, a, stream);
}

}  // namespace fa
