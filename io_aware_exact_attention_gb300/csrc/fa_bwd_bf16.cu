// Backward pass, bf16 in / fp32 accumulate.
//
// The pages keep only the per-row softmax statistics after the forward pass and
// recompute what back-propagation needs ("How FlashAttention Eliminates
// Transformer Memory Bottlenecks", galileo blog, Innovation #3).  They give no
// formulas; these kernels apply the chain rule to S = scale Q K^T, P = softmax(S),
// O = P V with L = sum(O * dO):
//   P  = exp(S - LSE)            (recomputed, one exp per score)
//   dV = P^T dO,   dP = dO V^T,  D = rowsum(dO * O),  dS = P * (dP - D)
//   dK = scale dS^T Q,           dQ = scale dS K
// Three launches:
//   1. preprocess: D per query row, and the float32 dQ accumulator set to zero;
//   2. main: one CTA per 128-row key tile K_j, V_j (kept in shared memory) loops
//      over the query tiles Q_i that see it.  Five tcgen05 MMAs per tile pair:
//        S = Q_i K_j^T and dP = dO_i V_j^T (TMEM, lanes = query rows),
//        dV += P^T dO_i and dK += dS^T Q_i (TMEM accumulators, lanes = key rows),
//        dQ_i = dS K_j (TMEM), scaled and added into the float32 accumulator by
//        TMA reduce-add from shared memory, 32x32 blocks at a time.
//      P and then dS occupy one shared buffer as bf16 in a 128-byte-swizzled
//      [query][key] layout; the same bytes serve as a K-major operand (dQ) and,
//      read M-major, as the transposed operand (dV, dK).  Q is double-buffered so
//      the next tile's scores can start as soon as this tile's dK, dQ are issued.
//      Roles: warp 0 TMA producer, warp 1 MMA issuer, warps 2..5 P and dS,
//      warps 6..9 dQ drain and the dK, dV epilogue.
//      At d = 64 the main step is a persistent kernel instead: one CTA per SM walks
//      key tiles with two K/V buffers, and both compute warpgroups share P, dS and
//      the dQ drain by key halves (bwd_persistent_kernel).
//   3. postprocess: dQ (bf16) from the float32 accumulator.
#include "fa_internal.h"
#include "fa_tiles.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kBwdThreads = 320;
constexpr float kLog2e = 1.44269504088896340736f;

// d = 128, one CTA per key tile.  TMEM: S and dP take turns in one 128-column region
// (S is read out before dP is written, dP before the next S), which leaves dV, dK and
// dQ 128 columns each, so the dQ drain (warps 6..9) only has to finish before the next
// dQ and never holds up the next dP.  Warps 2..5 compute P and dS.
template <int D>
struct BwdLayout {
  static_assert(D == 128, "the one-CTA-per-key-tile backward is the d = 128 kernel");
  static constexpr int kQStages = 2;
  static constexpr int kDoStages = 1;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kSubBytes = kTile * 64 * 2;
  static constexpr int kStageBytes = 32 * 32 * 4;  // one 32x32 fp32 dQ block
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;
  static constexpr int kDO = kQ + kQStages * kTileBytes;
  static constexpr int kPS = kDO + kDoStages * kTileBytes;   // P, then dS, of the current tile pair
  static constexpr int kDQ = kPS + kTile * kTile * 2;        // 4 drain warps x 2 buffers of 32x32 fp32
  static constexpr int kEnd = kDQ + 4 * 2 * kStageBytes;
  static constexpr int kSmemBytes = kEnd + 1024;
  static constexpr uint32_t kColSP = 0;  // S, then dP, of the current tile pair
  static constexpr uint32_t kColDV = 128;
  static constexpr uint32_t kColDK = 128 + D;
  static constexpr uint32_t kColDQ = 128 + 2 * D;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kComputeArrivals = 128u;  // one warpgroup per role
  static_assert(kColDQ + D <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// The eight K = 16 steps of a 128-deep product over 128-byte-swizzled bf16 tiles, in
// descriptor units (16 bytes): a K-major operand moves 32 bytes inside a 64-element
// sub-tile, then to the next sub-tile (kSubBytes on); an M- or N-major operand moves 16
// rows of 128 bytes (2048 bytes).  kk: both K-major (S, dP); mn: both M/N-major (dV,
// dK); kn: A K-major, B N-major (dQ).
static_assert(BwdLayout<128>::kSubBytes == 1024 * 16, "K-major step offsets below");
__device__ __forceinline__ void mma_steps_kk(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  mma8_bf16_ss<0, 2, 4, 6, 1024, 1026, 1028, 1030, 0, 2, 4, 6, 1024, 1026, 1028, 1030>(d, a, b, idesc, acc);
}
__device__ __forceinline__ void mma_steps_mn(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  mma8_bf16_ss<0, 128, 256, 384, 512, 640, 768, 896, 0, 128, 256, 384, 512, 640, 768, 896>(d, a, b, idesc, acc);
}
__device__ __forceinline__ void mma_steps_kn(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  mma8_bf16_ss<0, 2, 4, 6, 1024, 1026, 1028, 1030, 0, 128, 256, 384, 512, 640, 768, 896>(d, a, b, idesc, acc);
}

template <int D>
struct BwdBarriers {
  uint64_t kv_full;
  uint64_t q_full[BwdLayout<D>::kQStages];
  uint64_t q_empty[BwdLayout<D>::kQStages];
  uint64_t do_full[BwdLayout<D>::kDoStages];
  uint64_t do_empty[BwdLayout<D>::kDoStages];
  uint64_t s_full, s_free, dp_full, dp_free, p_full, dv_done, ds_full, dq_free, dkdq_done, drain;
};

__device__ __forceinline__ float pos_inf() { return __int_as_float(0x7f800000); }

// 3-D tiled reduce-add of one box from shared memory into global memory (bulk group).
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, const void* smem_src, int c0, int c1,
                                                  int c2) {
  asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::
                   "l"(reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(smem_src))
               : "memory");
}

__device__ __forceinline__ void bulk_wait_read_le1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                    const __grid_constant__ CUtensorMap tm_dq, const float* __restrict__ lse,
                    const float* __restrict__ dsum, const AttnArgs a) {
  using L = BwdLayout<D>;
  griddep_launch_dependents();
  griddep_wait();  // every global access of this kernel comes after the previous kernel of the stream
  constexpr int QS = L::kQStages;
  constexpr int DS = L::kDoStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) BwdBarriers<D> bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = a.n_tiles;
  const int head = blockIdx.x / T;
  const int kt = blockIdx.x % T;  // key tile owned by this CTA
  const int b = head / a.H;
  const int kv_len = clamp_kv_len(a.kv_len, b, a.N);
  const int qt_first = a.causal ? kt : 0;
  const WaitCtx wc{&abort_flag, a.status};

  uint8_t* smK = smem + L::kK;
  uint8_t* smV = smem + L::kV;
  uint8_t* smQ = smem + L::kQ;
  uint8_t* smDO = smem + L::kDO;
  uint8_t* smPS = smem + L::kPS;
  uint8_t* smDQ = smem + L::kDQ;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar.kv_full, 1);
    for (int s = 0; s < QS; ++s) {
      mbar_init(&bar.q_full[s], 1);
      mbar_init(&bar.q_empty[s], 1);
    }
    for (int s = 0; s < DS; ++s) {
      mbar_init(&bar.do_full[s], 1);
      mbar_init(&bar.do_empty[s], 1);
    }
    mbar_init(&bar.s_full, 1);
    mbar_init(&bar.s_free, L::kComputeArrivals);
    mbar_init(&bar.dp_full, 1);
    mbar_init(&bar.dp_free, L::kComputeArrivals);
    mbar_init(&bar.p_full, L::kComputeArrivals);
    mbar_init(&bar.dv_done, 1);
    mbar_init(&bar.ds_full, L::kComputeArrivals);
    mbar_init(&bar.dq_free, L::kComputeArrivals);
    mbar_init(&bar.dkdq_done, 1);
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
  const int first = next_query_tile(qt_first, kt, kv_len, a.causal, a.block_mask, T);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      if (first < T) {
        mbar_arrive_expect_tx(&bar.kv_full, 2 * L::kTileBytes);
        for (int h = 0; h < D / 64; ++h) {
          tma_load_3d(smK + h * L::kSubBytes, &tm_k, &bar.kv_full, h * 64, kt * kTile, head);
          tma_load_3d(smV + h * L::kSubBytes, &tm_v, &bar.kv_full, h * 64, kt * kTile, head);
        }
      }
      for (int qt = first; qt < T; qt = next_query_tile(qt + 1, kt, kv_len, a.causal, a.block_mask, T), ++it) {
        const int sq = it % QS, sd = it % DS;
        if (it >= QS && !(ok = mbar_wait(&bar.q_empty[sq], ((it / QS) - 1) & 1, wc))) break;
        mbar_arrive_expect_tx(&bar.q_full[sq], L::kTileBytes);
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(smQ + sq * L::kTileBytes + h * L::kSubBytes, &tm_q, &bar.q_full[sq], h * 64, qt * kTile, head);
        if (it >= DS && !(ok = mbar_wait(&bar.do_empty[sd], ((it / DS) - 1) & 1, wc))) break;
#ifdef FA_TEST_SKIP_LOAD
        // failure-path test build only: CTA 0 never loads its second dO tile, so the MMA
        // issuer's bounded wait on it gives up and the CTA takes its abort path
        if (it == 1 && blockIdx.x == 0) continue;
#endif
        mbar_arrive_expect_tx(&bar.do_full[sd], L::kTileBytes);
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(smDO + sd * L::kTileBytes + h * L::kSubBytes, &tm_do, &bar.do_full[sd], h * 64, qt * kTile,
                      head);
      }
      if (!ok) {
        // let the loads already issued land before the CTA can exit
        if (first < T) mbar_drain(&bar.kv_full, 0, 100000000ull);
        for (int j = (it > QS ? it - QS : 0); j <= it; ++j) mbar_drain(&bar.q_full[j % QS], (j / QS) & 1, 100000000ull);
        for (int j = (it > DS ? it - DS : 0); j < it; ++j) mbar_drain(&bar.do_full[j % DS], (j / DS) & 1, 100000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, 128, false, false);   // S, dP
      constexpr uint32_t id_t = idesc_bf16_f32(128, D, true, true);       // dV, dK (transposed A)
      constexpr uint32_t id_q = idesc_bf16_f32(128, D, false, true);      // dQ
      const uint64_t kd = sdesc_sw128(smem_u32(smK), 16, 1024);          // K, K-major (S)
      const uint64_t kn = sdesc_sw128(smem_u32(smK), L::kSubBytes, 1024);  // K, N-major (dQ)
      const uint64_t vd = sdesc_sw128(smem_u32(smV), 16, 1024);          // V, K-major (dP)
      const uint64_t pt = sdesc_sw128(smem_u32(smPS), L::kSubBytes, 1024);  // P, dS read M-major (dV, dK)
      const uint64_t pk = sdesc_sw128(smem_u32(smPS), 16, 1024);           // dS read K-major (dQ)
      bool ok = true;
      int it = 0;
      // S = Q_i K_j^T into the S/dP columns
      auto issue_scores = [&](int stage) {
        const uint64_t qd = sdesc_sw128(smem_u32(smQ + stage * L::kTileBytes), 16, 1024);
        tc_fence_after();
        mma_steps_kk(tmem + L::kColSP, qd, kd, id_s, 0u);
        mma_commit(&bar.s_full);
      };
      if (first < T) {
        ok = mbar_wait(&bar.kv_full, 0, wc) && mbar_wait(&bar.q_full[0], 0, wc);
        if (ok) issue_scores(0);
      }
      if (ok) {
        // Per query tile: dP (once S is read out), dV, the next S (once dP is read
        // out), dK, then dQ (once the previous dQ is drained).
        for (int qt = first; qt < T; ++it) {
          const int qt_next = next_query_tile(qt + 1, kt, kv_len, a.causal, a.block_mask, T);
          const int sq = it % QS, sd = it % DS;
          const uint64_t qn = sdesc_sw128(smem_u32(smQ + sq * L::kTileBytes), L::kSubBytes, 1024);
          const uint64_t dod = sdesc_sw128(smem_u32(smDO + sd * L::kTileBytes), 16, 1024);
          const uint64_t don = sdesc_sw128(smem_u32(smDO + sd * L::kTileBytes), L::kSubBytes, 1024);
          // dP = dO_i V_j^T
          if (!(ok = mbar_wait(&bar.do_full[sd], (it / DS) & 1, wc))) break;
          if (!(ok = mbar_wait(&bar.s_free, it & 1, wc))) break;
          tc_fence_after();
          mma_steps_kk(tmem + L::kColSP, dod, vd, id_s, 0u);
          mma_commit(&bar.dp_full);
          // dV += P^T dO_i
          if (!(ok = mbar_wait(&bar.p_full, it & 1, wc))) break;
          tc_fence_after();
          mma_steps_mn(tmem + L::kColDV, pt, don, id_t, it > 0 ? 1u : 0u);
          mma_commit(&bar.dv_done);
          mma_commit(&bar.do_empty[sd]);
          // the next scores
          if (qt_next < T) {
            if (!(ok = mbar_wait(&bar.q_full[(it + 1) % QS], ((it + 1) / QS) & 1, wc))) break;
            if (!(ok = mbar_wait(&bar.dp_free, it & 1, wc))) break;
            issue_scores((it + 1) % QS);
          }
          // dK += dS^T Q_i (the last reader of Q_i)
          if (!(ok = mbar_wait(&bar.ds_full, it & 1, wc))) break;
          tc_fence_after();
          mma_steps_mn(tmem + L::kColDK, pt, qn, id_t, it > 0 ? 1u : 0u);
          mma_commit(&bar.q_empty[sq]);
          // dQ_i = dS K_j
          if (it >= 1 && !(ok = mbar_wait(&bar.dq_free, (it - 1) & 1, wc))) break;
          tc_fence_after();
          mma_steps_kn(tmem + L::kColDQ, pk, kn, id_q, 0u);
          mma_commit(&bar.dkdq_done);  // dS is no longer read, dQ_i is complete
          qt = qt_next;
        }
      }
      if (!ok) {
        mma_commit(&bar.drain);
        mbar_drain(&bar.drain, 0, 100000000ull);
      }
    }
  } else if (warp < 6) {
    // ------------------------------------------------- P and dS (warps 2..5)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // query row inside the tile
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = a.scale_log2;
    const int key0 = kt * kTile;
    const uint32_t psrow = smem_u32(smPS);
    bool ok = true;
    int it = 0;
    int qt = first;
    // per-row statistics of the current query tile, loaded one tile ahead
    auto load_stats = [&](int t, float& lse_v, float& d_v) {
      const int row = t * kTile + r;
      if (t < T && row < a.N) {
        const size_t idx = static_cast<size_t>(head) * a.N + row;
        lse_v = ld_global_pinned(lse + idx);
        d_v = ld_global_pinned(dsum + idx);
      } else {
        lse_v = pos_inf();
        d_v = 0.f;
      }
    };
    float lse_r, d_r;
    load_stats(qt, lse_r, d_r);
    for (; qt < T; ++it) {
      const int qt_next = next_query_tile(qt + 1, kt, kv_len, a.causal, a.block_mask, T);
      float lse_n, d_n;
      load_stats(qt_next, lse_n, d_n);
      const int q_row = qt * kTile + r;
      if (lse_r == -pos_inf()) lse_r = pos_inf();  // a row that sees no key contributes nothing
      const float lse2 = lse_r * kLog2e;
      const bool need_mask = (key0 + kTile > kv_len) || (a.causal && kt == qt);
      const int lim = a.causal ? min(kv_len, q_row + 1) : kv_len;  // keys [key0, lim) visible

      // P = exp2(S scale log2e - LSE log2e), one 64-column half at a time through one loop
      // body (see the dS loop below); the MMA warp may write dP over S once both halves are
      // in registers.  The first half's bf16 pairs are held while the second is formed,
      // then both are stored once the previous dS is no longer read.
      ok = mbar_wait(&bar.s_full, it & 1, wc);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t pk0[32];
#pragma unroll 1
      for (int c0 = 0; c0 < kTile; c0 += 64) {
        uint32_t t[64];
        tmem_ld64(tmem + lane_off + L::kColSP + c0, t);
        if (c0 == 64) {
          tc_fence_before();
          mbar_arrive(&bar.s_free);
        }
        float f[64];
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          ffma2(f[i], f[i + 1], __uint_as_float(t[i]), __uint_as_float(t[i + 1]), sl2, -lse2);
          f[i] = ex2(f[i]);
          f[i + 1] = ex2(f[i + 1]);
        }
        if (need_mask) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (key0 + c0 + i >= lim) f[i] = 0.f;
        }
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 64; i += 2) pk[i / 2] = pack_bf16x2(f[i], f[i + 1]);
        if (c0 == 0) {
#pragma unroll
          for (int j = 0; j < 32; ++j) pk0[j] = pk[j];
        } else {
          if (it >= 1) {
            ok = mbar_wait(&bar.dkdq_done, (it - 1) & 1, wc);  // dS_{i-1} no longer read by the dK, dQ MMAs
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          }
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            st_shared_v4(psrow + sw128_offset(r, g), pk0[4 * g], pk0[4 * g + 1], pk0[4 * g + 2], pk0[4 * g + 3]);
            st_shared_v4(psrow + L::kSubBytes + sw128_offset(r, g), pk[4 * g], pk[4 * g + 1], pk[4 * g + 2],
                         pk[4 * g + 3]);
          }
        }
      }
      if (!ok) break;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar.p_full);

      // dS = P * (dP - D), one 64-column half at a time, P read back from the rows of the
      // shared buffer this thread wrote.  dS replaces P there once the dV MMA has read P
      // (waited before the first half is written); the MMA warp may write the next S over
      // dP once the second half is loaded (the pipe is still busy with dV until about
      // then).  The halves run through one loop body: with P in registers both halves
      // were separate code, and this kernel's roles together outgrew the instruction
      // cache (64% hits); one body, and one for the dQ drain below, took 9% off its time.
      ok = mbar_wait(&bar.dp_full, it & 1, wc);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int c0 = 0; c0 < kTile; c0 += 64) {
        uint32_t t[64];
        tmem_ld64(tmem + lane_off + L::kColSP + c0, t);
        if (c0 == 64) {
          tc_fence_before();
          mbar_arrive(&bar.dp_free);
        }
        uint32_t pp[32];
#pragma unroll
        for (int g = 0; g < 8; ++g)
          ld_shared_v4(psrow + (c0 / 64) * L::kSubBytes + sw128_offset(r, g), pp[4 * g], pp[4 * g + 1], pp[4 * g + 2],
                       pp[4 * g + 3]);
        float f[64];
#pragma unroll
        for (int i = 0; i < 64; i += 2)
          fsubmul2(f[i], f[i + 1], __uint_as_float(t[i]), __uint_as_float(t[i + 1]), d_r, bf16lo(pp[i / 2]),
                   bf16hi(pp[i / 2]));
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 64; i += 2) w[i / 2] = pack_bf16x2(f[i], f[i + 1]);
        if (c0 == 0) {
          ok = mbar_wait(&bar.dv_done, it & 1, wc);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        }
#pragma unroll
        for (int g = 0; g < 8; ++g)
          st_shared_v4(psrow + (c0 / 64) * L::kSubBytes + sw128_offset(r, g), w[4 * g], w[4 * g + 1], w[4 * g + 2],
                       w[4 * g + 3]);
      }
      if (!ok) break;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar.ds_full);
      qt = qt_next;
      lse_r = lse_n;
      d_r = d_n;
    }
  } else {
    // ------------------------------- dQ drain and the dK, dV epilogue (warps 6..9)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // query row (dQ) or key row (dK, dV) inside the tile
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    uint8_t* stage_dq = smDQ + wq * 2 * L::kStageBytes;  // this warp's two 32x32 fp32 staging blocks
    bool ok = true;
    int it = 0;
    int nblk = 0;
    for (int qt = first; qt < T; qt = next_query_tile(qt + 1, kt, kv_len, a.causal, a.block_mask, T), ++it) {
      // dQ_i = dS K_j in its own TMEM columns: scale it and add it into the float32
      // accumulator; it only has to be drained before dQ_{i+1} is formed
      ok = mbar_wait(&bar.dkdq_done, it & 1, wc);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int c64 = 0; c64 < D; c64 += 64) {
        uint32_t t[64];
        tmem_ld64(tmem + lane_off + L::kColDQ + c64, t);
#pragma unroll
        for (int h = 0; h < 2; ++h, ++nblk) {
          uint8_t* blk = stage_dq + (nblk & 1) * L::kStageBytes;
          if (lane == 0) bulk_wait_read_le1();  // the block written two steps ago has been read
          __syncwarp();
          const uint32_t row = smem_u32(blk);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            st_shared_v4(row + sw128_offset(lane, q), __float_as_uint(__uint_as_float(t[32 * h + 4 * q]) * a.scale),
                         __float_as_uint(__uint_as_float(t[32 * h + 4 * q + 1]) * a.scale),
                         __float_as_uint(__uint_as_float(t[32 * h + 4 * q + 2]) * a.scale),
                         __float_as_uint(__uint_as_float(t[32 * h + 4 * q + 3]) * a.scale));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_3d(&tm_dq, blk, c64 + 32 * h, qt * kTile + wq * 32, head);
            tma_store_commit();
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bar.dq_free);
    }
    if (lane == 0) tma_store_wait_all();

    // epilogue: dV_j and scale * dK_j as bf16 through shared memory (the two Q
    // stages: the last dK, which the final dkdq_done follows, was their last reader)
    // and TMA
    const bool have = ok && it > 0;
    tc_fence_after();
    uint8_t* stv = smQ;
    uint8_t* stk = smQ + L::kTileBytes;
    const uint32_t stage_v = smem_u32(stv), stage_k = smem_u32(stk);
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t tv[32], tk[32];
      if (have) {
        tmem_ld32(tmem + lane_off + L::kColDV + c0, tv);
        tmem_ld32(tmem + lane_off + L::kColDK + c0, tk);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) tv[i] = tk[i] = 0u;
      }
      uint32_t wv[16], wk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        wv[i] = pack_bf16x2(__uint_as_float(tv[2 * i]), __uint_as_float(tv[2 * i + 1]));
        wk[i] = pack_bf16x2(__uint_as_float(tk[2 * i]) * a.scale, __uint_as_float(tk[2 * i + 1]) * a.scale);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t off = (c0 / 64) * L::kSubBytes + sw128_offset(r, ((c0 % 64) / 8) + q);
        st_shared_v4(stage_v + off, wv[4 * q], wv[4 * q + 1], wv[4 * q + 2], wv[4 * q + 3]);
        st_shared_v4(stage_k + off, wk[4 * q], wk[4 * q + 1], wk[4 * q + 2], wk[4 * q + 3]);
      }
    }
    fence_proxy_async_smem();
    named_barrier(1, 128);
    if (warp == 6 && lane == 0) {
      for (int h = 0; h < D / 64; ++h) {
        tma_store_3d(&tm_dv, stv + h * L::kSubBytes, h * 64, kt * kTile, head);
        tma_store_3d(&tm_dk, stk + h * L::kSubBytes, h * 64, kt * kTile, head);
      }
      tma_store_commit();
      tma_store_wait_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// Persistent backward for d = 64: one CTA per SM walks key tiles c, c + G, c + 2G, ...
// (G = grid size), with two K/V buffers so the next key tile loads while this one is
// processed, and two P/dS buffers so the next P is written while dK, dQ still read
// this dS.  The P/dS work (a full 128-key row per thread regardless of d) is split by
// key halves over both compute warpgroups; each warp drains its 32 x 32 block of dQ
// and writes its 32 x 32 blocks of dV, dK through one private staging block.  Across
// items the work overlaps: the next item's first scores go out after this item's last
// dV, and this item's last dQ drain and its dV, dK epilogue run in the next item's
// first tile pair, after that P is stored (BERT-sized items of <= 4 tiles: -10%).
template <int D>
struct PBwdLayout {
  static_assert(D == 64, "the persistent backward is the d = 64 kernel");
  static constexpr int kQStages = 2;
  static constexpr int kDoStages = 2;
  static constexpr int kKvBuffers = 2;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kSubBytes = kTile * 64 * 2;
  static constexpr int kStageBytes = 32 * 32 * 4;  // one 32x32 fp32 dQ block
  static constexpr int kKV = 0;                                   // [K, V] per buffer
  static constexpr int kQ = kKV + kKvBuffers * 2 * kTileBytes;
  static constexpr int kDO = kQ + kQStages * kTileBytes;
  static constexpr int kPSBytes = kTile * kTile * 2;
  static constexpr int kPS = kDO + kDoStages * kTileBytes;   // 2 buffers: P, then dS, of tile pair i in buffer i % 2
  static constexpr int kDQ = kPS + 2 * kPSBytes;             // 8 staging blocks (one per compute warp)
  static constexpr int kEnd = kDQ + 8 * kStageBytes;
  static constexpr int kSmemBytes = kEnd + 1024;
  // TMEM columns: S, dP, dV, dK, dQ side by side (128 + 128 + 3 * 64 <= 512).
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColDP = 128;
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + D;
  static constexpr uint32_t kColDQ = 256 + 2 * D;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kComputeArrivals = 256u;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

template <int D>
struct PBwdBarriers {
  uint64_t kv_full[PBwdLayout<D>::kKvBuffers];
  uint64_t kv_empty[PBwdLayout<D>::kKvBuffers];
  uint64_t q_full[PBwdLayout<D>::kQStages];
  uint64_t q_empty[PBwdLayout<D>::kQStages];
  uint64_t do_full[PBwdLayout<D>::kDoStages];
  uint64_t do_empty[PBwdLayout<D>::kDoStages];
  uint64_t dkdq_done[2];  // tile pair i completes dkdq_done[i % 2]
  uint64_t s_full, dp_full, p_full, dv_done, ds_full, dq_free, acc_free, drain;
};


// One unit of persistent backward work: a 128-row key tile of one (batch, head).
struct BwdItem {
  int head, kt, kv_len, first;  // first query tile that sees the key tile (T if none)
};

// Items are taken key-tile-major, so every CTA gets an even mix of causal work
// (early key tiles have the most query tiles).  `kv_len_raw` is the item's entry of
// the key-padding lengths (item_kv_len), loaded ahead so no role waits on it.
__device__ __forceinline__ BwdItem bwd_item(int item, int kv_len_raw, const AttnArgs& a) {
  BwdItem w;
  const int BH = a.B * a.H;
  w.head = item % BH;
  w.kt = item / BH;
  w.kv_len = kv_len_raw < 0 ? 0 : (kv_len_raw > a.N ? a.N : kv_len_raw);
  w.first = next_query_tile(a.causal ? w.kt : 0, w.kt, w.kv_len, a.causal, a.block_mask, a.n_tiles);
  return w;
}

// Key-padding length of item `item`'s batch (N without padding or past the last item).
__device__ __forceinline__ int item_kv_len(int item, int n_items, const AttnArgs& a) {
  if (a.kv_len == nullptr || item >= n_items) return a.N;
  return ld_global_pinned(a.kv_len + (item % (a.B * a.H)) / a.H);
}

// kv_len of a CTA's items two items ahead: next() returns the current item's value and
// issues the load for the item two steps on, which has a whole item to arrive.
struct KvLenAhead {
  int n0, n1, step, n_items;
  __device__ __forceinline__ KvLenAhead(int first, int g, int n, const AttnArgs& a)
      : n0(item_kv_len(first, n, a)), n1(item_kv_len(first + g, n, a)), step(g), n_items(n) {}
  __device__ __forceinline__ int next(int item, const AttnArgs& a) {
    const int cur = n0;
    n0 = n1;
    n1 = item_kv_len(item + 2 * step, n_items, a);
    return cur;
  }
  __device__ __forceinline__ int peek() const { return n0; }  // the next item's, after next()
};

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_persistent_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                    const __grid_constant__ CUtensorMap tm_dq, const float* __restrict__ lse,
                    const float* __restrict__ dsum, const AttnArgs a) {
  using L = PBwdLayout<D>;
  griddep_launch_dependents();
  griddep_wait();  // every global access of this kernel comes after the previous kernel of the stream
  constexpr int QS = L::kQStages;
  constexpr int DS = L::kDoStages;
  constexpr int KB = L::kKvBuffers;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) PBwdBarriers<D> bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = a.n_tiles;
  const int n_items = T * a.B * a.H;
  const WaitCtx wc{&abort_flag, a.status};

  uint8_t* smKV = smem + L::kKV;
  uint8_t* smQ = smem + L::kQ;
  uint8_t* smDO = smem + L::kDO;
  uint8_t* smPS = smem + L::kPS;
  uint8_t* smDQ = smem + L::kDQ;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < KB; ++s) {
      mbar_init(&bar.kv_full[s], 1);
      mbar_init(&bar.kv_empty[s], 1);
    }
    for (int s = 0; s < QS; ++s) {
      mbar_init(&bar.q_full[s], 1);
      mbar_init(&bar.q_empty[s], 1);
    }
    for (int s = 0; s < DS; ++s) {
      mbar_init(&bar.do_full[s], 1);
      mbar_init(&bar.do_empty[s], 1);
    }
    mbar_init(&bar.s_full, 1);
    mbar_init(&bar.dp_full, 1);
    mbar_init(&bar.p_full, L::kComputeArrivals);
    mbar_init(&bar.dv_done, 1);
    mbar_init(&bar.ds_full, L::kComputeArrivals);
    mbar_init(&bar.dkdq_done[0], 1);
    mbar_init(&bar.dkdq_done[1], 1);
    mbar_init(&bar.dq_free, L::kComputeArrivals);
    mbar_init(&bar.acc_free, L::kComputeArrivals);
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
      int git = 0;  // query-tile iterations over all items of this CTA
      int kvu = 0;  // items with work (K/V buffer uses)
      bool ok = true;
      KvLenAhead kvl(blockIdx.x, gridDim.x, n_items, a);
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const BwdItem w = bwd_item(item, kvl.next(item, a), a);
        if (w.first >= T) continue;  // no query sees this key tile: nothing to load
        const int kb = kvu % KB;
        if (kvu >= KB && !(ok = mbar_wait(&bar.kv_empty[kb], ((kvu / KB) - 1) & 1, wc))) break;
        uint8_t* kvs = smKV + kb * 2 * L::kTileBytes;
        mbar_arrive_expect_tx(&bar.kv_full[kb], 2 * L::kTileBytes);
        for (int h = 0; h < D / 64; ++h) {
          tma_load_3d(kvs + h * L::kSubBytes, &tm_k, &bar.kv_full[kb], h * 64, w.kt * kTile, w.head);
          tma_load_3d(kvs + L::kTileBytes + h * L::kSubBytes, &tm_v, &bar.kv_full[kb], h * 64, w.kt * kTile, w.head);
        }
        ++kvu;
        for (int qt = w.first; qt < T; qt = next_query_tile(qt + 1, w.kt, w.kv_len, a.causal, a.block_mask, T), ++git) {
          const int sq = git % QS, sd = git % DS;
          if (git >= QS && !(ok = mbar_wait(&bar.q_empty[sq], ((git / QS) - 1) & 1, wc))) break;
          mbar_arrive_expect_tx(&bar.q_full[sq], L::kTileBytes);
          for (int h = 0; h < D / 64; ++h)
            tma_load_3d(smQ + sq * L::kTileBytes + h * L::kSubBytes, &tm_q, &bar.q_full[sq], h * 64, qt * kTile,
                        w.head);
          if (git >= DS && !(ok = mbar_wait(&bar.do_empty[sd], ((git / DS) - 1) & 1, wc))) break;
          mbar_arrive_expect_tx(&bar.do_full[sd], L::kTileBytes);
          for (int h = 0; h < D / 64; ++h)
            tma_load_3d(smDO + sd * L::kTileBytes + h * L::kSubBytes, &tm_do, &bar.do_full[sd], h * 64, qt * kTile,
                        w.head);
        }
      }
      if (!ok) {
        // let the loads already issued land before the CTA can exit
        for (int j = (kvu > KB ? kvu - KB : 0); j < kvu; ++j)
          mbar_drain(&bar.kv_full[j % KB], (j / KB) & 1, 100000000ull);
        for (int j = (git > QS ? git - QS : 0); j <= git; ++j)
          mbar_drain(&bar.q_full[j % QS], (j / QS) & 1, 100000000ull);
        for (int j = (git > DS ? git - DS : 0); j < git; ++j)
          mbar_drain(&bar.do_full[j % DS], (j / DS) & 1, 100000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, 128, false, false);   // S, dP
      constexpr uint32_t id_t = idesc_bf16_f32(128, D, true, true);       // dV, dK (transposed A)
      constexpr uint32_t id_q = idesc_bf16_f32(128, D, false, true);      // dQ
      const uint32_t ps0 = smem_u32(smPS);
      // P, dS: read M-major (the transposed A of dV, dK) and K-major (the A of dQ)
      const uint64_t pt_desc = sdesc_sw128(ps0, L::kSubBytes, 1024);
      const uint64_t pk_desc = sdesc_sw128(ps0, 16, 1024);
      bool ok = true;
      int git = 0, kvu = 0;
      int accu = 0;  // items whose dK, dV accumulators were used
      // S = Q K_j^T into the S columns (free once the previous P has been read out)
      auto issue_scores = [&](int stage, uint32_t k0) {
        const uint64_t qa = sdesc_sw128(smem_u32(smQ + stage * L::kTileBytes), 16, 1024);
        const uint64_t kb = sdesc_sw128(k0, 16, 1024);
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k / 4) * L::kSubBytes + (k % 4) * 32;
          mma_bf16_ss(tmem + L::kColS, sdesc_adv(qa, off), sdesc_adv(kb, off), id_s, k > 0 ? 1u : 0u);
        }
        mma_commit(&bar.s_full);
      };
      KvLenAhead kvl(blockIdx.x, gridDim.x, n_items, a);
      bool s_ahead = false;  // this item's first scores went out during the previous item
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const BwdItem w = bwd_item(item, kvl.next(item, a), a);
        if (w.first >= T) continue;
        const int kb = kvu % KB;
        const uint32_t k0 = smem_u32(smKV + kb * 2 * L::kTileBytes), v0 = k0 + L::kTileBytes;
        if (!s_ahead) {
          if (!(ok = mbar_wait(&bar.kv_full[kb], (kvu / KB) & 1, wc))) break;
          if (!(ok = mbar_wait(&bar.q_full[git % QS], (git / QS) & 1, wc))) break;
          issue_scores(git % QS, k0);
        }
        s_ahead = false;
        // Per query tile: dP, dV, then the next tile's scores (so the P/dS warps can
        // move straight on; after an item's last dV, the next item's first scores, its
        // K, V being in the other buffer), then dK and dQ.
        int itl = 0;
        for (int qt = w.first; qt < T; ++itl, ++git) {
          const int qt_next = next_query_tile(qt + 1, w.kt, w.kv_len, a.causal, a.block_mask, T);
          const int sq = git % QS, sd = git % DS;
          const uint32_t q0 = smem_u32(smQ + sq * L::kTileBytes), do0 = smem_u32(smDO + sd * L::kTileBytes);
          const uint32_t psb = static_cast<uint32_t>(git & 1) * L::kPSBytes;
          // dP = dO_i V_j^T (when dQ shares dP's columns, the previous dQ must have been drained)
          if (!(ok = mbar_wait(&bar.do_full[sd], (git / DS) & 1, wc))) break;
          tc_fence_after();
          {
            const uint64_t da = sdesc_sw128(do0, 16, 1024), vb = sdesc_sw128(v0, 16, 1024);
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
              const uint32_t off = (k / 4) * L::kSubBytes + (k % 4) * 32;
              mma_bf16_ss(tmem + L::kColDP, sdesc_adv(da, off), sdesc_adv(vb, off), id_s, k > 0 ? 1u : 0u);
            }
          }
          mma_commit(&bar.dp_full);
          // dV += P^T dO_i; the first of an item overwrites the accumulators, which the
          // previous item's epilogue must have read out
          if (!(ok = mbar_wait(&bar.p_full, git & 1, wc))) break;
          if (itl == 0 && accu > 0 && !(ok = mbar_wait(&bar.acc_free, (accu - 1) & 1, wc))) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k)
            mma_bf16_ss(tmem + L::kColDV, sdesc_adv(pt_desc, psb + k * 2048), sdesc_adv(sdesc_sw128(do0, L::kSubBytes, 1024), k * 2048),
                        id_t, (itl > 0 || k > 0) ? 1u : 0u);
          mma_commit(&bar.dv_done);
          mma_commit(&bar.do_empty[sd]);
          // next tile's scores: the S columns were read out before p_full
          if (qt_next < T) {
            if (!(ok = mbar_wait(&bar.q_full[(git + 1) % QS], ((git + 1) / QS) & 1, wc))) break;
            issue_scores((git + 1) % QS, k0);
          } else if (item + static_cast<int>(gridDim.x) < n_items) {
            // the next item's first scores (its K, V are in the other buffer)
            const BwdItem wn = bwd_item(item + gridDim.x, kvl.peek(), a);
            if (wn.first < T) {
              const int kbn = (kvu + 1) % KB;
              if (!(ok = mbar_wait(&bar.kv_full[kbn], ((kvu + 1) / KB) & 1, wc))) break;
              if (!(ok = mbar_wait(&bar.q_full[(git + 1) % QS], ((git + 1) / QS) & 1, wc))) break;
              issue_scores((git + 1) % QS, smem_u32(smKV + kbn * 2 * L::kTileBytes));
              s_ahead = true;
            }
          }
          // dK += dS^T Q_i ; dQ_i = dS K_j
          if (!(ok = mbar_wait(&bar.ds_full, git & 1, wc))) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k)
            mma_bf16_ss(tmem + L::kColDK, sdesc_adv(pt_desc, psb + k * 2048), sdesc_adv(sdesc_sw128(q0, L::kSubBytes, 1024), k * 2048),
                        id_t, (itl > 0 || k > 0) ? 1u : 0u);
          if (git >= 1 && !(ok = mbar_wait(&bar.dq_free, (git - 1) & 1, wc))) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k)
            mma_bf16_ss(tmem + L::kColDQ, sdesc_adv(pk_desc, psb + (k / 4) * L::kSubBytes + (k % 4) * 32),
                        sdesc_adv(sdesc_sw128(k0, L::kSubBytes, 1024), k * 2048), id_q, k > 0 ? 1u : 0u);
          mma_commit(&bar.dkdq_done[git & 1]);
          mma_commit(&bar.q_empty[sq]);
          qt = qt_next;
        }
        if (!ok) break;
        mma_commit(&bar.kv_empty[kb]);  // K_j, V_j are free once this item's MMAs finish
        ++kvu;
        ++accu;
      }
      if (!ok) {
        mma_commit(&bar.drain);
        mbar_drain(&bar.drain, 0, 100000000ull);
      }
    }
  } else {
    // ------- d = 64: P, dS, the dQ drain and the dK, dV epilogue, split by halves (warps 2..9)
    const int hc = (warp - 2) >> 2;  // keys [64 hc, 64 hc + 64) of P and dS; dQ, dK, dV columns [32 hc, 32 hc + 32)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // query row (P, dS, dQ) or key row (dK, dV) inside the tile
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = a.scale_log2;
    const uint32_t ps_half = smem_u32(smPS) + hc * L::kSubBytes;
    uint8_t* blk = smDQ + (hc * 4 + wq) * L::kStageBytes;  // this warp's staging block (dQ, then dV | dK)
    bool ok = true;
    int git = 0;
    bool pending = false;  // dQ of iteration git-1 not yet drained
    int pend_qt = 0, pend_head = 0;
    // LSE and D of query row `row` of head `head` (+inf and 0 past the last tile)
    auto load_stats = [&](int head, int t, float& lse_v, float& d_v) {
      const int row = t * kTile + r;
      if (t < T && row < a.N) {
        const size_t idx = static_cast<size_t>(head) * a.N + row;
        lse_v = ld_global_pinned(lse + idx);
        d_v = ld_global_pinned(dsum + idx);
      } else {
        lse_v = pos_inf();
        d_v = 0.f;
      }
    };
    // dQ of query tile qt_d of head h_d (this warp's 32 rows x 32 columns): TMEM ->
    // swizzled shared block -> TMA reduce-add into the float32 accumulator
    auto drain_dq = [&](int qt_d, int h_d) {
      uint32_t t[32];
      tmem_ld32(tmem + lane_off + L::kColDQ + 32 * hc, t);
      if (lane == 0) bulk_wait_read_all();  // the block's last bulk copy has read it
      __syncwarp();
      const uint32_t row = smem_u32(blk);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st_shared_v4(row + sw128_offset(lane, q), __float_as_uint(__uint_as_float(t[4 * q]) * a.scale),
                     __float_as_uint(__uint_as_float(t[4 * q + 1]) * a.scale),
                     __float_as_uint(__uint_as_float(t[4 * q + 2]) * a.scale),
                     __float_as_uint(__uint_as_float(t[4 * q + 3]) * a.scale));
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_reduce_add_3d(&tm_dq, blk, 32 * hc, qt_d * kTile + wq * 32, h_d);
        tma_store_commit();
      }
    };
    // wait for the dK, dQ MMAs of iteration j (tile pair j completes dkdq_done[j % 2])
    auto wait_dkdq = [&](int j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bar.dkdq_done[j & 1], (j >> 1) & 1, wc));
      return ok;
    };
    // The statistics of an item's first query tile are loaded one item ahead.
    KvLenAhead kvl(blockIdx.x, gridDim.x, n_items, a);
    float lse_c = pos_inf(), d_c = 0.f;
    if (static_cast<int>(blockIdx.x) < n_items) {
      const BwdItem w0 = bwd_item(blockIdx.x, kvl.peek(), a);
      load_stats(w0.head, w0.first, lse_c, d_c);
    }
    // The epilogue of an item: this warp's 32 key rows x 32 columns of dV_j and scale * dK_j
    // as bf16, staged in its own block (64-byte rows, 64-byte swizzle) and stored by TMA;
    // key tiles no query sees get zeros.  `have`: the item's MMAs are all done and its
    // accumulators hold dV_j, dK_j.
    auto epilogue = [&](bool have, int kt_e, int head_e) {
      uint32_t wv[16], wk[16];
      {
        uint32_t tv[32], tk[32];
        if (have) {
          tc_fence_after();
          tmem_ld32(tmem + lane_off + L::kColDV + 32 * hc, tv);
          tmem_ld32(tmem + lane_off + L::kColDK + 32 * hc, tk);
          tc_fence_before();
          mbar_arrive(&bar.acc_free);  // the accumulators may now be overwritten by the next item
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) tv[i] = tk[i] = 0u;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          wv[i] = pack_bf16x2(__uint_as_float(tv[2 * i]), __uint_as_float(tv[2 * i + 1]));
          wk[i] = pack_bf16x2(__uint_as_float(tk[2 * i]) * a.scale, __uint_as_float(tk[2 * i + 1]) * a.scale);
        }
      }
      if (lane == 0) bulk_wait_read_all();  // the block's last bulk copy (a dQ reduce) has read it
      __syncwarp();
      const uint32_t sv = smem_u32(blk), sk = sv + 2048;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        st_shared_v4(sv + sw64_offset(lane, q), wv[4 * q], wv[4 * q + 1], wv[4 * q + 2], wv[4 * q + 3]);
        st_shared_v4(sk + sw64_offset(lane, q), wk[4 * q], wk[4 * q + 1], wk[4 * q + 2], wk[4 * q + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&tm_dv, blk, 32 * hc, kt_e * kTile + wq * 32, head_e);
        tma_store_3d(&tm_dk, blk + 2048, 32 * hc, kt_e * kTile + wq * 32, head_e);
        tma_store_commit();
      }
    };
    // An item's last dQ drain and its epilogue are deferred into the next item's first
    // tile pair, after its P is stored: the next P then overlaps the item's last dK, dQ.
    bool epi_pending = false, epi_have = false;
    int epi_kt = 0, epi_head = 0;
    auto flush_item = [&]() {
      if (pending) {
        if (ok && wait_dkdq(git - 1)) {
          tc_fence_after();
          drain_dq(pend_qt, pend_head);
          tc_fence_before();
          mbar_arrive(&bar.dq_free);
        }
        pending = false;
      }
      if (epi_pending) {
        epilogue(epi_have && ok, epi_kt, epi_head);
        epi_pending = false;
      }
    };
    // Every warp walks every item; an aborted CTA (ok == false) only skips the work.
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const BwdItem w = bwd_item(item, kvl.next(item, a), a);
      const bool work = w.first < T;
      float lse_x = pos_inf(), d_x = 0.f;  // the next item's first tile, in flight during this item
      if (item + static_cast<int>(gridDim.x) < n_items) {
        const BwdItem wn = bwd_item(item + gridDim.x, kvl.peek(), a);
        load_stats(wn.head, wn.first, lse_x, d_x);
      }
      const int key0 = w.kt * kTile + 64 * hc;
      float lse_r = lse_c, d_r = d_c;
      for (int qt = w.first; ok && qt < T; ++git) {
        const int qt_next = next_query_tile(qt + 1, w.kt, w.kv_len, a.causal, a.block_mask, T);
        float lse_n, d_n;
        load_stats(w.head, qt_next, lse_n, d_n);
        const int q_row = qt * kTile + r;
        if (lse_r == -pos_inf()) lse_r = pos_inf();  // a row that sees no key contributes nothing
        const float lse2 = lse_r * kLog2e;
        const bool need_mask = (w.kt * kTile + kTile > w.kv_len) || (a.causal && w.kt == qt);
        const int lim = a.causal ? min(w.kv_len, q_row + 1) : w.kv_len;  // keys [kt*128, lim) visible
        const uint32_t psrow = ps_half + static_cast<uint32_t>(git & 1) * L::kPSBytes;

        ok = mbar_wait(&bar.s_full, git & 1, wc);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        uint32_t pk[32];
        {
          uint32_t t[64];
          tmem_ld64(tmem + lane_off + L::kColS + 64 * hc, t);
          float f[64];
#pragma unroll
          for (int i = 0; i < 64; i += 2) {
            ffma2(f[i], f[i + 1], __uint_as_float(t[i]), __uint_as_float(t[i + 1]), sl2, -lse2);
            f[i] = ex2(f[i]);
            f[i + 1] = ex2(f[i + 1]);
          }
          if (need_mask) {
#pragma unroll
            for (int i = 0; i < 64; ++i)
              if (key0 + i >= lim) f[i] = 0.f;
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
        }
        // this buffer last held dS of iteration git-2: its dK, dQ MMAs must be done
        if (git >= 2 && !wait_dkdq(git - 2)) break;
#pragma unroll
        for (int g = 0; g < 8; ++g)
          st_shared_v4(psrow + sw128_offset(r, g), pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bar.p_full);
        // the previous dQ drains while the MMA warp runs dV and the next scores
        if (pending) {
          if (!wait_dkdq(git - 1)) break;
          tc_fence_after();
          drain_dq(pend_qt, pend_head);
          tc_fence_before();
          mbar_arrive(&bar.dq_free);
          pending = false;
        }
        if (epi_pending) {
          epilogue(epi_have, epi_kt, epi_head);
          epi_pending = false;
        }

        ok = mbar_wait(&bar.dp_full, git & 1, wc);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        uint32_t wds[32];
        {
          uint32_t t[64];
          tmem_ld64(tmem + lane_off + L::kColDP + 64 * hc, t);
          float f[64];
#pragma unroll
          for (int i = 0; i < 64; i += 2)
            fsubmul2(f[i], f[i + 1], __uint_as_float(t[i]), __uint_as_float(t[i + 1]), d_r, bf16lo(pk[i / 2]),
                     bf16hi(pk[i / 2]));
#pragma unroll
          for (int i = 0; i < 32; ++i) wds[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
        }
        // dS replaces P in the shared buffer once the dV MMA has read P
        ok = mbar_wait(&bar.dv_done, git & 1, wc);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
#pragma unroll
        for (int g = 0; g < 8; ++g)
          st_shared_v4(psrow + sw128_offset(r, g), wds[4 * g], wds[4 * g + 1], wds[4 * g + 2], wds[4 * g + 3]);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bar.ds_full);
        pending = true;
        pend_qt = qt;
        pend_head = w.head;
        qt = qt_next;
        lse_r = lse_n;
        d_r = d_n;
      }
      lse_c = lse_x;
      d_c = d_x;
      if (work) {
        // this item's first tile pair ran the previous item's epilogue; one still pending
        // here means that pair gave up (ok == false), and it only writes zeros
        if (epi_pending) flush_item();
        epi_pending = true;
        epi_have = ok;
        epi_kt = w.kt;
        epi_head = w.head;
      } else {
        flush_item();
        epilogue(false, w.kt, w.head);
      }
    }
    flush_item();
    if (lane == 0) tma_store_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// D_i = sum_c dO_ic O_ic (float32) for every row, and dq_acc = 0.
// Eight bf16 per lane; D / 8 lanes share a row.
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout,
                                                             float* __restrict__ dsum, float4* __restrict__ dq_acc,
                                                             long long rows) {
  griddep_launch_dependents();
  griddep_wait();
  constexpr int kLanesPerRow = D / 8;
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
  // rows handled in groups so every lane of a warp stays active for the shuffles
  const long long row_slots = (rows * kLanesPerRow + 31) / 32 * 32;
  for (long long e = tid; e < row_slots; e += nthreads) {
    const long long row = e / kLanesPerRow;
    const int part = static_cast<int>(e % kLanesPerRow);
    float acc = 0.f;
    if (row < rows) {
      const uint4 x = o[row * kLanesPerRow + part];
      const uint4 y = dout[row * kLanesPerRow + part];
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc = fmaf(bf16lo(xs[i]), bf16lo(ys[i]), acc);
        acc = fmaf(bf16hi(xs[i]), bf16hi(ys[i]), acc);
      }
    }
#pragma unroll
    for (int off = kLanesPerRow / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && part == 0) dsum[row] = acc;
  }
  const long long n4 = rows * D / 4;
  for (long long e = tid; e < n4; e += nthreads) dq_acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// dq (bf16) = dq_acc (float32), eight elements per thread.
__global__ void __launch_bounds__(256) bwd_postprocess_kernel(const float4* __restrict__ dq_acc,
                                                              uint4* __restrict__ dq, long long n8) {
  griddep_launch_dependents();
  griddep_wait();
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long e = tid; e < n8; e += nthreads) {
    const float4 x = dq_acc[2 * e], y = dq_acc[2 * e + 1];
    dq[e] = make_uint4(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w), pack_bf16x2(y.x, y.y), pack_bf16x2(y.z, y.w));
  }
}

unsigned grid_for(long long work, int per_block) {
  long long blocks = (work + per_block - 1) / per_block;
  const long long cap = static_cast<long long>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  return static_cast<unsigned>(blocks < 1 ? 1 : blocks);
}

template <int D>
cudaError_t launch_bwd_main_d(const BwdMaps& m, const float* lse, const float* dsum, const AttnArgs& a,
                              cudaStream_t stream) {
  const long long n_items = static_cast<long long>(a.n_tiles) * a.B * a.H;
  if constexpr (D == 64) {
    // persistent: one CTA per SM walks the key tiles
    using L = PBwdLayout<D>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(bwd_persistent_kernel<D>), L::kSmemBytes);
    if (e != cudaSuccess) return e;
    const long long grid = n_items < sm_count() ? n_items : sm_count();
    return launch_pdl(bwd_persistent_kernel<D>, static_cast<unsigned>(grid), kBwdThreads, L::kSmemBytes, stream, m.q,
                      m.k, m.v, m.dout, m.dk32, m.dv32, m.dq_acc, lse, dsum, a);
  } else {
    // one CTA per key tile
    using L = BwdLayout<D>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(bwd_main_kernel<D>), L::kSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(bwd_main_kernel<D>, static_cast<unsigned>(n_items), kBwdThreads, L::kSmemBytes, stream, m.q, m.k,
                      m.v, m.dout, m.dk, m.dv, m.dq_acc, lse, dsum, a);
  }
}

}  // namespace

cudaError_t launch_bwd_preprocess(const void* o, const void* dout, float* dsum, float* dq_acc, const AttnArgs& a,
                                  cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.B) * a.H * a.N;
  const unsigned grid = grid_for(rows * (a.d / 8), 256);
  const uint4* o4 = static_cast<const uint4*>(o);
  const uint4* do4 = static_cast<const uint4*>(dout);
  float4* acc = reinterpret_cast<float4*>(dq_acc);
  if (a.d == 64) return launch_pdl(bwd_preprocess_kernel<64>, grid, 256, 0, stream, o4, do4, dsum, acc, rows);
  return launch_pdl(bwd_preprocess_kernel<128>, grid, 256, 0, stream, o4, do4, dsum, acc, rows);
}

cudaError_t launch_bwd_main_bf16(const BwdMaps& maps, const float* lse, const float* dsum, const AttnArgs& a,
                                 cudaStream_t stream) {
  return a.d == 64 ? launch_bwd_main_d<64>(maps, lse, dsum, a, stream) : launch_bwd_main_d<128>(maps, lse, dsum, a, stream);
}

cudaError_t launch_bwd_postprocess(const float* dq_acc, void* dq, const AttnArgs& a, cudaStream_t stream) {
  const long long n8 = static_cast<long long>(a.B) * a.H * a.N * a.d / 8;
  return launch_pdl(bwd_postprocess_kernel, grid_for(n8, 256), 256, 0, stream, reinterpret_cast<const float4*>(dq_acc),
                    static_cast<uint4*>(dq), n8);
}

}  // namespace fa
