// Forward pass on the fifth-generation tensor cores: bf16 inputs (d = 64 or 128) or
// FP8 E4M3 inputs (d = 128), fp32 accumulation, bf16 O and fp32 LSE.
//
// One CTA owns two adjacent 128-row query tiles Q_a, Q_b of one (batch, head) and
// streams the key/value tiles K_j, V_j either may see, as in the "FlashAttention
// (Conceptual)" listing of "FlashAttention: how a memory trick unlocked..."
// (khetwal.com): per key tile it forms the score block, updates the running row
// max and row sum, rescales the output accumulator and adds P V ("The Trick:
// Online Softmax").  The GB300 mapping:
//   warp 0       TMA producer: lane 0 both query tiles once, then K_j, lane 1 V_j,
//                each into a ring of shared-memory stages (128-byte swizzle) with
//                its own release barrier, skipping masked tiles;
//   warps 1, 10  MMA issuers, one per query tile (warp 1 also allocates tensor
//                memory), taking turns: tile i's O_i += P_i V_j with P read from
//                TMEM (the score buffer it replaced) and V N-major straight from
//                its TMA tile, then S_i = Q_i K_{j+1}^T into that score buffer;
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
//
// The FP8 variant runs the same kernel with 8-bit tiles.  Q and K arrive as E4M3
// [B*H, N, 128] (one 128-byte swizzle row per token); V arrives transposed, E4M3
// [B*H, 128, ldv], so that the P V product reads it K-major (keys contiguous) like
// the score product reads K.  Both products are kind::f8f6f4 MMAs of K = 32.  The
// per-tensor scales of Q and K are folded into the score scale and that of V into
// 1/l.  P is rounded to E4M3 (its values lie in (0, 2^8], see kRescaleSlack) and
// packed four to a TMEM column; the row sum l is taken over the unrounded values.
// O (bf16) is staged in a region of its own, the 8-bit Q tiles being half its size.
#include "fa_internal.h"
#include "fa_tiles.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleSlack = 8.0f;  // P values stay below 2^8 before a rescale is forced
// bf16: a key tile whose exponentials against the running max sum to at most 2^8 keeps it
constexpr float kFastSumLimit = 256.0f;  // = 2^kRescaleSlack

// NQ query tiles per CTA.  NQ = 2 (d = 128): one CTA per SM, the two tiles'
// softmax phases overlap each other's MMAs.  NQ = 1 (d = 64): a lighter CTA with
// 256 TMEM columns and ~81 KB of shared memory, so two CTAs share an SM and one
// CTA's set-up, loads and epilogue overlap the other's main loop.
// F8: E4M3 tiles (d = 128, two query tiles).
template <int D, int NQ, bool F8>
struct FwdLayout {
  static_assert(!F8 || (D == 128 && NQ == 2), "the FP8 forward runs d = 128 with two query tiles per CTA");
  static constexpr int kElem = F8 ? 1 : 2;        // bytes per Q, K or V element
  // warp 0 producer, warp 1 MMA issuer of tile a, warps 2.. one softmax warpgroup per
  // tile, then (NQ = 2) the MMA issuer of tile b
  static constexpr int kIssuerB = NQ == 2 ? 2 + 4 * NQ : -1;
  static constexpr int kThreads = 64 + 128 * NQ + (NQ == 2 ? 32 : 0);
  static constexpr int kCtasPerSm = NQ == 1 ? 2 : 1;
  static constexpr int kStages = F8 ? 4 : (NQ == 1 ? 2 : (D == 64 ? 4 : 2));
  static constexpr int kTileBytes = kTile * D * kElem;  // one tile of Q, K or V (F8: V^T, d rows x 128 keys)
  static constexpr int kSubBytes = kTile * 128;         // one swizzle sub-tile: 128 rows of 128 bytes
  static constexpr int kSubElems = 128 / kElem;         // elements in one sub-tile row
  static constexpr int kOTileBytes = kTile * D * 2;     // one bf16 O tile
  static constexpr int kQ = 0;                          // NQ query tiles
  static constexpr int kK = kQ + NQ * kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kOStage = kV + kStages * kTileBytes;  // F8: O staging; bf16 stages O in the Q tiles
  static constexpr int kEnd = F8 ? kOStage + NQ * kOTileBytes : kOStage;
  static constexpr int kSmemBytes = kEnd + 1024;  // slack for aligning the base to 1024
  static constexpr uint32_t kTmemCols = NQ == 1 ? 256 : 512;
  // TMEM columns: score/P buffer of tile i at 128*i, output accumulator of tile i after all score buffers
  __device__ static constexpr uint32_t col_s(int i) { return 128u * static_cast<uint32_t>(i); }
  __device__ static constexpr uint32_t col_o(int i) { return 128u * NQ + static_cast<uint32_t>(D * i); }
  static_assert(128 * NQ + D * NQ <= static_cast<int>(kTmemCols), "TMEM budget");
  static_assert(kSmemBytes <= (NQ == 1 ? 112 * 1024 : 227 * 1024), "shared memory budget");
};

template <int S>
struct FwdBarriers {
  uint64_t q_full;
  uint64_t k_full[S];
  uint64_t v_full[S];
  uint64_t k_empty[S];  // both score products have read the K tile of the stage
  uint64_t v_empty[S];  // both P V products have read the V tile of the stage
  uint64_t s_full[2];
  uint64_t p_full[2];  // P of the tile is in TMEM and O rescaled if it had to be (FP8: keys [0, 64) of P)
  uint64_t p_hi[2];    // FP8 only: P of keys [64, 128) is in TMEM
  uint64_t o_done[2];
  uint64_t drain[2];  // one per MMA issuer
  uint64_t tok[2];    // tok[i]: issuer i has issued its batch (the other issuer's turn)
};

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// Waits of the MMA issuers, which have nothing else to do meanwhile: try_wait with a
// suspend-time hint, so the thread sleeps until the phase completes (or the hint runs
// out) instead of re-issuing the test, leaving the issue slots of its sub-partition
// to the softmax warps that share it.  Bounded like mbar_wait.  (In the backward
// kernels the same change made the issuers react later and cost ~3%, so they poll.)
constexpr uint32_t kIssuerSleepNs = 2000;

__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kIssuerSleepNs)
      : "memory");
  return ok != 0u;
}

__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long start = globaltimer();
  uint32_t tries = 0;
  while (true) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if ((++tries & 7u) == 0u) {
      if (*w.abort_flag) return false;
      if (globaltimer() - start > kWaitLimitNs) {
        *w.abort_flag = 1;
        if (w.status) atomicCAS(w.status, 0u, kErrTimeout);
        return false;
      }
    }
  }
}

// Maximum of a 128-value row: eight independent 3-input max chains of eight steps,
// then a three-level tree (a two-chain loop is a 32-step latency chain).
__device__ __forceinline__ float row_max128(const float (&v)[kTile]) {
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = fmaxf(v[2 * k], v[2 * k + 1]);
#pragma unroll
  for (int c = 16; c < kTile; c += 16)
#pragma unroll
    for (int k = 0; k < 8; ++k) m[k] = fmax3(m[k], v[c + 2 * k], v[c + 2 * k + 1]);
  return fmaxf(fmax3(m[0], m[1], m[2]), fmax3(m[3], m[4], fmax3(m[5], m[6], m[7])));
}

// Sum of a 128-value row: eight independent accumulators (four paired adds per step).
__device__ __forceinline__ float row_sum128(const float (&v)[kTile]) {
  float a[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) a[k] = v[k];
#pragma unroll
  for (int c = 8; c < kTile; c += 8)
#pragma unroll
    for (int k = 0; k < 8; k += 2) fadd2(a[k], a[k + 1], v[c + k], v[c + k + 1]);
  return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
}

// Registers -> TMEM, 32 lanes x 16 columns in one store and one wait.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Sum of 64 values v[c0 .. c0+63]: eight independent accumulators (paired adds).
__device__ __forceinline__ float half_sum64(const float (&v)[kTile], int c0) {
  float a[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) a[k] = v[c0 + k];
#pragma unroll
  for (int c = 8; c < 64; c += 8)
#pragma unroll
    for (int k = 0; k < 8; k += 2) fadd2(a[k], a[k + 1], v[c0 + c + k], v[c0 + c + k + 1]);
  return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
}

// Key tile kt is loaded when either query tile of the CTA sees it.
__device__ __forceinline__ bool pair_sees(const int (&qt)[2], int kt, int kv_len, const AttnArgs& a) {
  if (tile_pair_visible(qt[0], kt, kv_len, a.causal, a.block_mask, a.n_tiles)) return true;
  return qt[1] < a.n_tiles && tile_pair_visible(qt[1], kt, kv_len, a.causal, a.block_mask, a.n_tiles);
}

__device__ __forceinline__ int next_union_tile(const int (&qt)[2], int kt, int kv_len, const AttnArgs& a) {
  while (kt < a.n_tiles && !pair_sees(qt, kt, kv_len, a)) ++kt;
  return kt;
}

// SPLIT: split-KV partial pass (bf16, d = 128): the CTA's two query-tile slots hold the
// same query tile and see the even / odd key tiles of one key chunk; each slot writes a
// normalised float32 O and its LSE as one partial result instead of O.
template <int D, int NQ, bool F8, bool SPLIT = false>
__device__ __forceinline__ void fwd_body(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                         const CUtensorMap& tm_o, float* __restrict__ lse_out, const AttnArgs& a) {
  using L = FwdLayout<D, NQ, F8>;
  griddep_launch_dependents();
  griddep_wait();  // every global access of this kernel comes after the previous kernel of the stream
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) FwdBarriers<S> bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = a.n_tiles;                  // query tiles
  const int TK = SPLIT ? a.nk_tiles : T;    // key tiles
  int head, qt[2], chunk = 0;
  if constexpr (SPLIT) {
    const int per_head = T * a.n_chunks;
    head = blockIdx.x / per_head;
    const int rem = static_cast<int>(blockIdx.x % per_head);
    qt[0] = qt[1] = rem / a.n_chunks;
    chunk = rem % a.n_chunks;
  } else {
    const int n_groups = (T + NQ - 1) / NQ;
    head = blockIdx.x / n_groups;  // b * H + h
    const int gr = static_cast<int>(blockIdx.x % n_groups);
    const int group = a.causal ? (n_groups - 1 - gr) : gr;  // causal: heaviest groups first
    qt[0] = NQ * group;
    qt[1] = NQ == 2 ? 2 * group + 1 : T;  // qt[1] >= T: no second tile
  }
  const bool has_b = qt[1] < T;
  const int b = head / a.H;
  const int kv_len = clamp_kv_len(a.kv_len, b, SPLIT ? a.nk : a.N);
  const int kvt = (kv_len + kTile - 1) / kTile;
  // SPLIT: key tiles [k_lo, k_hi) of this CTA; slot i sees those at even (i = 0) or odd
  // (i = 1) positions from k_lo.
  const int k_lo = SPLIT ? chunk * a.chunk_tiles : 0;
  const int k_hi = SPLIT ? min(k_lo + a.chunk_tiles, kvt) : TK;
  // does slot i see key tile kt; first key tile >= kt that slot i sees / either slot sees
  auto pair_vis = [&](int i, int kt) -> bool {
    if constexpr (SPLIT) return kt >= k_lo && kt < k_hi && ((kt - k_lo) & 1) == i;
    else return tile_pair_visible(qt[i], kt, kv_len, a.causal, a.block_mask, T);
  };
  auto next_vis = [&](int i, int kt) -> int {
    if constexpr (SPLIT) {
      kt = max(kt, k_lo);
      kt += ((kt - k_lo) & 1) != i;
      return kt < k_hi ? kt : TK;
    } else {
      return next_key_tile(qt[i], kt, kv_len, a.causal, a.block_mask, T);
    }
  };
  auto next_union = [&](int kt) -> int {
    if constexpr (SPLIT) {
      kt = max(kt, k_lo);
      return kt < k_hi ? kt : TK;
    } else {
      return next_union_tile(qt, kt, kv_len, a);
    }
  };
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
      mbar_init(&bar.k_empty[s], has_b ? 2 : 1);  // one commit per MMA issuer
      mbar_init(&bar.v_empty[s], has_b ? 2 : 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.s_full[i], 1);
      mbar_init(&bar.p_full[i], 128);
      mbar_init(&bar.p_hi[i], 128);
      mbar_init(&bar.o_done[i], 1);
      mbar_init(&bar.drain[i], 1);
      mbar_init(&bar.tok[i], 1);
    }
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
    // lane 0: both query tiles, then the K tiles; lane 1: the V tiles.  K and V stages
    // are released separately (a K tile is done once both score products have read
    // it, a V tile once both P V products have).  The two lanes run one loop, so their
    // loads go out in step; starting the K lane's loop one key tile further ahead
    // measured no faster (and slower for FP8).
    if (lane < 2) {
      const bool is_k = lane == 0;
      if (is_k) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        mbar_arrive_expect_tx(&bar.q_full, (has_b ? 2 : 1) * L::kTileBytes);
        for (int i = 0; i < (has_b ? 2 : 1); ++i)
          for (int h = 0; h < L::kTileBytes / L::kSubBytes; ++h)
            tma_load_3d(smQ + i * L::kTileBytes + h * L::kSubBytes, &tm_q, &bar.q_full, h * L::kSubElems,
                        qt[i] * kTile, head);
      } else {
        tma_prefetch_desc(&tm_v);
      }
      uint64_t* full = is_k ? bar.k_full : bar.v_full;
      uint64_t* empty = is_k ? bar.k_empty : bar.v_empty;
      int u = 0;
      bool ok = true;
      for (int kt = next_union(0); kt < TK; kt = next_union(kt + 1), ++u) {
        const int s = u % S;
        if (u >= S && !(ok = mbar_wait(&empty[s], ((u / S) - 1) & 1, wc))) break;
#ifdef FA_TEST_SKIP_LOAD
        // failure-path test build only: CTA 0 never loads its second K tile, so the
        // MMA issuer's bounded wait on it gives up and the CTA takes its abort path
        if (is_k && u == 1 && blockIdx.x == 0 && !SPLIT) continue;
#endif
        mbar_arrive_expect_tx(&full[s], L::kTileBytes);
        if (is_k) {
          for (int h = 0; h < L::kTileBytes / L::kSubBytes; ++h)
            tma_load_3d(smK + s * L::kTileBytes + h * L::kSubBytes, &tm_k, &full[s], h * L::kSubElems, kt * kTile,
                        head);
        } else if constexpr (F8) {
          // V^T tile: d rows of 128 keys
          tma_load_3d(smV + s * L::kTileBytes, &tm_v, &full[s], kt * kTile, 0, head);
        } else {
          for (int h = 0; h < D / 64; ++h)
            tma_load_3d(smV + s * L::kTileBytes + h * L::kSubBytes, &tm_v, &full[s], h * 64, kt * kTile, head);
        }
      }
      if (!ok) {
        // let the loads already issued land before the CTA can exit
        if (is_k) mbar_drain(&bar.q_full, 0, 100000000ull);
        for (int j = (u > S ? u - S : 0); j < u; ++j) mbar_drain(&full[j % S], (j / S) & 1, 100000000ull);
      }
    }
  } else if (warp == 1 || warp == L::kIssuerB) {
    // ------------------------------------------------------------ MMA issuers
    // One issuing thread per query tile: warp 1 for tile a, warp kIssuerB for tile b.
    // An MMA holds its issuing thread about as long as the tensor pipe takes to run it,
    // so with a single issuer its waits and bookkeeping leave the pipe idle.  Here the
    // two issuers take turns: a batch (tile i's P V, then its next scores) is issued only
    // after the other tile's batch, signalled through tok[] as soon as its last MMA is
    // issued; each thread's waits and commits then overlap the other's MMAs, and the
    // alternation keeps one softmax running while the other tile's products execute.
    // The two tiles' accumulators and score buffers are disjoint; a K or V stage is
    // released once both issuers have committed it (k_empty and v_empty count one
    // arrival per issuer, one commit per key tile of the union list whether the tile
    // used it or not).  Each issuer runs one batch per key tile of the union list plus
    // the first scores, used or empty, so the token phases of the two threads stay in
    // step.
    const int i = warp == 1 ? 0 : 1;
    if (lane == 0 && (i == 0 || has_b)) {
      constexpr uint32_t idesc_s = F8 ? idesc_e4m3_f32(128, 128) : idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_o = F8 ? idesc_e4m3_f32(128, D) : idesc_bf16_f32(128, D, false, true);
      const uint32_t qs = smem_u32(smQ) + i * L::kTileBytes, k0 = smem_u32(smK), v0 = smem_u32(smV);
      // Without a block mask the key tiles are [0, end_union) and tile i sees [0, end_i),
      // which spares the issuer the per-tile visibility tests.
      const bool dense = !SPLIT && a.block_mask == nullptr;
      const int end_i = min(kvt, a.causal ? qt[i] + 1 : T);
      const int end_union = has_b ? min(kvt, a.causal ? qt[1] + 1 : T) : min(kvt, a.causal ? qt[0] + 1 : T);
      auto union_from = [&](int kt) { return dense ? (kt < end_union ? kt : TK) : next_union(kt); };
      auto sees = [&](int kt) { return dense ? kt < end_i : pair_vis(i, kt); };
      bool ok = mbar_wait(&bar.q_full, 0, wc);
      int n = 0;  // P V products issued for this tile
      int u = 0;  // position in the union list of key tiles
      // batch j of tile a follows batch j-1 of tile b; batch j of tile b follows batch j of a
      auto take_turn = [&](int j) -> bool {
        if (!has_b) return true;
        if (i == 0) return j == 0 || mbar_wait_sleep(&bar.tok[1], (j - 1) & 1, wc);
        return mbar_wait_sleep(&bar.tok[0], j & 1, wc);
      };
      auto pass_turn = [&]() {
        if (has_b) mbar_arrive(&bar.tok[i]);
      };
      // S_i for the key tile in `stage` into tile i's TMEM buffer.  That buffer still holds
      // P_i of the last P V, which this thread issued earlier: MMAs from one thread execute
      // in issue order, so the new scores overwrite P only after that P V has read it.
      auto issue_scores = [&](int stage) {
        tc_fence_after();
        const uint32_t ks = k0 + stage * L::kTileBytes;
        if constexpr (F8) {
          // four K = 32 steps, 32 bytes each inside the 128-byte rows
          mma4_f8_ss<0, 2, 4, 6, 0, 2, 4, 6>(tmem + L::col_s(i), sdesc_sw128(qs, 16, 1024), sdesc_sw128(ks, 16, 1024),
                                              idesc_s, 0u);
        } else if constexpr (D == 128) {
          // eight K = 16 steps: 32 bytes inside a 64-element sub-tile, then the next sub-tile
          static_assert(L::kSubBytes == 1024 * 16, "step offsets in 16-byte units");
          mma8_bf16_ss<0, 2, 4, 6, 1024, 1026, 1028, 1030, 0, 2, 4, 6, 1024, 1026, 1028, 1030>(
              tmem + L::col_s(i), sdesc_sw128(qs, 16, 1024), sdesc_sw128(ks, 16, 1024), idesc_s, 0u);
        } else {
#pragma unroll
          for (int k = 0; k < D * L::kElem / 32; ++k) {  // 32 bytes of each row per MMA
            const uint32_t off = (k / 4) * L::kSubBytes + (k % 4) * 32;
            mma_bf16_ss(tmem + L::col_s(i), sdesc_sw128(qs + off, 16, 1024), sdesc_sw128(ks + off, 16, 1024), idesc_s,
                        k > 0 ? 1u : 0u);
          }
        }
      };
      int kt = union_from(0);
      if (ok && kt < TK) {
        const bool f0 = sees(kt);
        if (f0) ok = mbar_wait(&bar.k_full[0], 0, wc);
        if (ok) ok = take_turn(0);
        if (ok) {
          if (f0) {
            issue_scores(0);
            mma_commit(&bar.s_full[i]);
          }
          pass_turn();
          mma_commit(&bar.k_empty[0]);
        }
      }
      // Per key tile of the union list: P_i V, then S_i for the next key tile, so the
      // softmax warpgroup gets its next scores as early as possible.  Every V stage is
      // waited for and every stage committed, used or not: the V wait keeps this thread
      // from committing a stage ahead of the other issuer's use of its previous contents.
      while (ok && kt < TK) {
        const int s = u % S;
        const int kt_next = union_from(kt + 1);
        const bool f = sees(kt), fn = kt_next < TK && sees(kt_next);
        // all waits before the turn: inside it only MMAs and the score commit are issued
        if (!(ok = mbar_wait_sleep(&bar.v_full[s], (u / S) & 1, wc))) break;
        if (f && !(ok = mbar_wait_sleep(&bar.p_full[i], n & 1, wc))) break;
        if (fn && !(ok = mbar_wait_sleep(&bar.k_full[(u + 1) % S], ((u + 1) / S) & 1, wc))) break;
        if (!(ok = take_turn(u + 1))) break;
        if (f) {
          tc_fence_after();
          const uint32_t vs = v0 + s * L::kTileBytes;
          if constexpr (F8) {
            // V^T K-major: 32 keys = 32 bytes per step; P: four keys per TMEM column.  P V on
            // keys [0, 64) while the softmax warps finish keys [64, 128), then the rest.
            const uint64_t vdesc = sdesc_sw128(vs, 16, 1024);
            mma2_f8_ts<0, 2>(tmem + L::col_o(i), tmem + L::col_s(i), vdesc, idesc_o, n > 0 ? 1u : 0u);
            if (!(ok = mbar_wait(&bar.p_hi[i], n & 1, wc))) break;
            tc_fence_after();
            mma2_f8_ts<4, 6>(tmem + L::col_o(i), tmem + L::col_s(i) + 16, vdesc, idesc_o, 1u);
          } else {
            // V N-major: 16 keys = 2048 bytes per step; P: two keys (eight per K step) per TMEM column
            mma8_bf16_ts<0, 128, 256, 384, 512, 640, 768, 896>(tmem + L::col_o(i), tmem + L::col_s(i),
                                                                sdesc_sw128(vs, L::kSubBytes, 1024), idesc_o,
                                                                n > 0 ? 1u : 0u);
          }
        }
        if (fn) {
          issue_scores((u + 1) % S);
          mma_commit(&bar.s_full[i]);
        }
        pass_turn();
        // The P V completion (o_done) is signalled after the next scores: the softmax waits
        // for it only after it has waited for those scores, which complete no earlier.
        if (f) {
          mma_commit(&bar.o_done[i]);
          ++n;
        }
        mma_commit(&bar.v_empty[s]);
        if (kt_next < TK) mma_commit(&bar.k_empty[(u + 1) % S]);
        kt = kt_next;
        ++u;
      }
      if (!ok) {
        mma_commit(&bar.drain[i]);
        mbar_drain(&bar.drain[i], 0, 100000000ull);
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
      for (int kt = next_vis(wg, 0); kt < TK; kt = next_vis(wg, kt + 1), ++n) {
        ok = mbar_wait(&bar.s_full[wg], n & 1, wc);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        // S of this key tile into registers, masked: key padding tail, causal diagonal
        // (the N tail is covered by kv_len <= N)
        float s[kTile];
        const int key0 = kt * kTile;
        const bool edge = key0 + kTile > kv_len || (a.causal && kt == my_qt);
        auto load_scores = [&]() {
#pragma unroll
          for (int c0 = 0; c0 < kTile; c0 += 64) {
            uint32_t t[64];
            tmem_ld64(t_s + c0, t);
#pragma unroll
            for (int i = 0; i < 64; ++i) s[c0 + i] = __uint_as_float(t[i]);
          }
          if (edge) {
            const int lim = a.causal ? min(kv_len, q_row + 1) : kv_len;  // keys [key0, lim) visible
#pragma unroll
            for (int c = 0; c < kTile; ++c)
              if (key0 + c >= lim) s[c] = neg_inf();
          }
        };
        load_scores();
        // The stabiliser m_use of the exponentials.  bf16, after the first key tile: the
        // exponentials are formed against the running max first, and kept when they sum to
        // at most 2^8.  P >= 0, so then every term is at most 2^8: the tile's max lies
        // within kRescaleSlack of the running max, where the max rule below keeps the
        // running max too, and the values are exactly the ones that rule would form.  A
        // larger (or NaN or infinite) sum falls back to the rule, with S reloaded from TMEM.
        // This skips the row max, a sixth of the softmax's instructions, whenever the max
        // does not move.  The first tile and FP8 (P formed in halves) always take the rule.
        //
        // P replaces S in the tile's TMEM buffer.  All exponentials of a batch first
        // (independent, so they overlap), then sums and packing; scale-and-subtract and
        // the sums run two lanes per instruction.  bf16: one batch of 128 keys, P as bf16
        // pairs in columns [0, 64).  FP8: two batches of 64 keys, P as E4M3 quads in
        // columns [0, 16) then [16, 32), so that the MMA warp starts P V on keys [0, 64)
        // while the exponentials and the (costlier) E4M3 packing of [64, 128) run.
        constexpr int kFirst = F8 ? kTile / 2 : kTile;
        float m_new = m_run, m_use = m_run, alpha = 1.f, tile_sum = 0.f;
        bool with_max = F8 || n == 0;
#pragma unroll 1
        for (int pass = 0;; ++pass) {
          if (with_max) {
            if (pass > 0) load_scores();
            const float mx = row_max128(s) * sl2;
            m_new = (mx > m_run + kRescaleSlack) ? mx : m_run;
            m_use = (m_new == neg_inf()) ? 0.f : m_new;
            alpha = ex2(m_run - m_use);
          }
#pragma unroll
          for (int c = 0; c < kFirst; c += 2) {
            ffma2(s[c], s[c + 1], s[c], s[c + 1], sl2, -m_use);
            s[c] = ex2(s[c]);
            s[c + 1] = ex2(s[c + 1]);
          }
          if constexpr (F8) break;
          tile_sum = row_sum128(s);
          if (with_max || !__any_sync(0xffffffffu, !(tile_sum <= kFastSumLimit))) break;
          with_max = true;
        }
        if constexpr (F8) {
          tile_sum = half_sum64(s, 0);
          uint32_t pk[kTile / 8];
#pragma unroll
          for (int c = 0; c < kTile / 2; c += 4) pk[c / 4] = pack_e4m3x4(s[c], s[c + 1], s[c + 2], s[c + 3]);
          tmem_st16(t_s, pk);
        } else {
          uint32_t pk[kTile / 2];
#pragma unroll
          for (int c = 0; c < kTile; c += 2) pk[c / 2] = pack_bf16x2(s[c], s[c + 1]);
          tmem_st32(t_s, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
          tmem_st32(t_s + 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
        }
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
        if constexpr (F8) {
#pragma unroll
          for (int c = kTile / 2; c < kTile; c += 2) {
            ffma2(s[c], s[c + 1], s[c], s[c + 1], sl2, -m_use);
            s[c] = ex2(s[c]);
            s[c + 1] = ex2(s[c + 1]);
          }
          uint32_t pk[kTile / 8];
#pragma unroll
          for (int c = kTile / 2; c < kTile; c += 4)
            pk[(c - kTile / 2) / 4] = pack_e4m3x4(s[c], s[c + 1], s[c + 2], s[c + 3]);
          tmem_st16(t_s + kTile / 8, pk);
          tc_fence_before();
          mbar_arrive(&bar.p_hi[wg]);
          tile_sum += half_sum64(s, kTile / 2);
        }
        l_run = l_run * alpha + tile_sum;
        m_run = m_new;
      }

      // epilogue: O = O_acc / l (bf16, staged in this tile's Q buffer, stored by TMA); LSE = m + ln l
      bool have_o = ok && n > 0;
      if (have_o) {
        ok = mbar_wait(&bar.o_done[wg], (n - 1) & 1, wc);
        have_o = __all_sync(0xffffffffu, ok);
        tc_fence_after();
      }
      const float inv_l = l_run > 0.f ? a.o_scale / l_run : 0.f;
      if constexpr (SPLIT) {
        // partial result (slot wg of key chunk `chunk`): normalised O in float32 and LSE,
        // written straight from registers, 512 bytes per row; the TMEM loads are
        // warp-wide, only the stores are limited to rows below N
        const bool row_ok = q_row < a.N;
        const size_t part = static_cast<size_t>(2 * chunk + wg) * (static_cast<size_t>(a.B) * a.H) + head;
        float4* dst = reinterpret_cast<float4*>(a.part_o + (part * a.N + (row_ok ? q_row : 0)) * D);
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t t[32];
          if (have_o) {
            tmem_ld32(t_o + c0, t);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) t[i] = 0u;
          }
          if (row_ok) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[c0 / 4 + q] = make_float4(__uint_as_float(t[4 * q]) * inv_l, __uint_as_float(t[4 * q + 1]) * inv_l,
                                            __uint_as_float(t[4 * q + 2]) * inv_l, __uint_as_float(t[4 * q + 3]) * inv_l);
          }
        }
        if (row_ok)
          a.part_lse[part * a.N + q_row] = (n > 0 && l_run > 0.f) ? (m_run + log2f(l_run)) * kLn2 : neg_inf();
      } else {
      if (!F8 && n == 0) {
        // no score MMA has read this Q tile, so its TMA load may still be landing in
        // the buffer the zero O is about to be staged in
        ok = mbar_wait(&bar.q_full, 0, wc);
        __syncwarp();
      }
      uint8_t* stage = F8 ? smem + L::kOStage + wg * L::kOTileBytes : smQ + wg * L::kTileBytes;
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
      }  // !SPLIT
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
__global__ void __launch_bounds__(FwdLayout<D, NQ, false>::kThreads, FwdLayout<D, NQ, false>::kCtasPerSm)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    float* __restrict__ lse_out, const AttnArgs a) {
  fwd_body<D, NQ, false>(tm_q, tm_k, tm_v, tm_o, lse_out, a);
}

// Split-KV partial pass: tm_q maps Q ([B*H, N, 128]), tm_k and tm_v K and V
// ([B*H, nk, 128]); tm_o and lse_out are not used.
__global__ void __launch_bounds__(FwdLayout<128, 2, false>::kThreads, FwdLayout<128, 2, false>::kCtasPerSm)
    fwd_splitkv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                       float* __restrict__ lse_out, const AttnArgs a) {
  fwd_body<128, 2, false, true>(tm_q, tm_k, tm_v, tm_o, lse_out, a);
}

// Combine of the split-KV partials, one warp per query row (d = 128, four columns per
// lane): LSE = M + ln sum_p exp(LSE_p - M) with M = max_p LSE_p, and
// O = sum_p exp(LSE_p - LSE) O_p, which is the softmax over all keys because each O_p is
// normalised by its own sum exp(LSE_p).  A row without keys (every LSE_p = -inf, or no
// partials) gets O = 0 and LSE = -inf.
__global__ void __launch_bounds__(256) splitkv_combine_kernel(const float* __restrict__ part_o,
                                                              const float* __restrict__ part_lse,
                                                              uint16_t* __restrict__ o, float* __restrict__ lse,
                                                              long long rows, int parts) {
  griddep_launch_dependents();
  griddep_wait();
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float m = neg_inf();
  for (int p = lane; p < parts; p += 32) m = fmaxf(m, part_lse[p * rows + row]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float total = neg_inf();
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (m != neg_inf()) {
    float sum = 0.f;
    for (int p = lane; p < parts; p += 32) sum += expf(part_lse[p * rows + row] - m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    total = m + logf(sum);
    for (int p = 0; p < parts; ++p) {
      const float w = expf(part_lse[p * rows + row] - total);
      if (w == 0.f) continue;  // the same for every lane of the warp
      const float4 x = reinterpret_cast<const float4*>(part_o + (p * rows + row) * 128)[lane];
      acc.x += w * x.x;
      acc.y += w * x.y;
      acc.z += w * x.z;
      acc.w += w * x.w;
    }
  }
  reinterpret_cast<uint2*>(o + row * 128)[lane] = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
  if (lane == 0) lse[row] = total;
}

// tm_v maps V^T (E4M3 [B*H, 128, ldv]).
__global__ void __launch_bounds__(FwdLayout<128, 2, true>::kThreads, FwdLayout<128, 2, true>::kCtasPerSm)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   float* __restrict__ lse_out, const AttnArgs a) {
  fwd_body<128, 2, true>(tm_q, tm_k, tm_v, tm_o, lse_out, a);
}

// Persistent forward for d = 64: two CTAs per SM, each walking (query tile, head) items
// so that TMEM is allocated once per CTA and the next item's loads and first score MMA
// overlap this item's epilogue.  P has TMEM columns of its own (S 128, P 64, O 64), so
// the scores of the next key tile are computed while the softmax of this one runs: the
// MMA warp issues S_{u+1} as soon as the softmax warps have read S_u out of TMEM.
// K and V have rings of their own (a K stage is free once its score MMA is done, a V
// stage once its P V is), filled by two producer lanes that run the same loop, and a
// third lane loads Q.  The two lanes stay converged, so the load of K for pair u + 1
// goes out together with V for pair u.  That pacing measured fastest: 4-5% ahead of one
// lane streaming K two pairs ahead of V, and ahead of K and V loads issued each as soon
// as its stage is free (separate code paths per lane, or one thread polling all rings).
// Q is double-buffered by item; an item's Q buffer is the staging tile of its O.
//
// The per-item barriers (q_full, q_empty, o_free) count only items with at least one
// visible key tile, in every role: with items skipped by one role but counted by
// another, a parity wait could see a phase two completions away.  An item without a
// visible key writes its zero rows of O with plain stores and touches no barrier.
template <int D>
struct PFwdLayout {
  static_assert(D == 64, "the persistent forward is the d = 64 kernel");
  static constexpr int kThreads = 192;  // producer warp, MMA warp, one softmax warpgroup
  static constexpr int kStages = 2;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kSubBytes = kTile * 64 * 2;
  static constexpr int kQ = 0;  // 2 Q buffers (item j in buffer j % 2)
  static constexpr int kK = kQ + 2 * kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kEnd = kV + kStages * kTileBytes;
  static constexpr int kSmemBytes = kEnd + 1024;
  static constexpr uint32_t kTmemCols = 256;
  static constexpr uint32_t kColS = 0;    // scores, float32, 128 columns
  static constexpr uint32_t kColP = 128;  // P as bf16 pairs, 64 columns
  static constexpr uint32_t kColO = 192;  // output accumulator, 64 columns
  static_assert(kSmemBytes <= 113 * 1024, "two CTAs per SM");
};

struct PFwdBarriers {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full, s_free, p_full, o_done, o_free;
  uint64_t drain;
};

// Item j of CTA c (rounds in snake order so that, with the heaviest items first,
// every CTA gets a similar total); -1 once the CTA has no more items.
__device__ __forceinline__ int pfwd_item(int j, int c, int G, int n_items) {
  const int idx = j * G + ((j & 1) ? (G - 1 - c) : c);
  return idx < n_items ? idx : -1;
}

struct FwdItem {
  int qt, head, kv_len;
};

__device__ __forceinline__ FwdItem pfwd_decode(int idx, const AttnArgs& a) {
  FwdItem w;
  const int BH = a.B * a.H;
  const int qi = idx / BH;
  w.head = idx % BH;
  w.qt = a.causal ? (a.n_tiles - 1 - qi) : qi;  // causal: longest rows first
  w.kv_len = clamp_kv_len(a.kv_len, w.head / a.H, a.N);
  return w;
}

// Position in a CTA's sequence of (item, visible key tile) pairs; j < 0 past the end.
struct FwdCursor {
  int j, kt;
  int k;       // index of the item among the CTA's items with a visible key tile
  bool first;  // the item's first key tile
  FwdItem w;
};

// First pair at or after item j, whose item is the k-th with a visible key tile
// (items without one are skipped).
__device__ __forceinline__ FwdCursor pfwd_cursor_from(int j, int k, int c, int G, int n_items, const AttnArgs& a) {
  FwdCursor cur;
  cur.first = true;
  cur.k = k;
  for (;; ++j) {
    const int idx = pfwd_item(j, c, G, n_items);
    if (idx < 0) {
      cur.j = -1;
      cur.kt = a.n_tiles;
      return cur;
    }
    cur.w = pfwd_decode(idx, a);
    cur.kt = next_key_tile(cur.w.qt, 0, cur.w.kv_len, a.causal, a.block_mask, a.n_tiles);
    if (cur.kt < a.n_tiles) {
      cur.j = j;
      return cur;
    }
  }
}

__device__ __forceinline__ FwdCursor pfwd_cursor_next(const FwdCursor& cur, int c, int G, int n_items,
                                                      const AttnArgs& a) {
  FwdCursor nxt = cur;
  nxt.kt = next_key_tile(cur.w.qt, cur.kt + 1, cur.w.kv_len, a.causal, a.block_mask, a.n_tiles);
  nxt.first = false;
  if (nxt.kt < a.n_tiles) return nxt;
  return pfwd_cursor_from(cur.j + 1, cur.k + 1, c, G, n_items, a);
}

template <int D>
__global__ void __launch_bounds__(PFwdLayout<D>::kThreads, 2)
    fwd_persistent_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                          uint16_t* __restrict__ o_out, float* __restrict__ lse_out, const AttnArgs a) {
  using L = PFwdLayout<D>;
  griddep_launch_dependents();
  griddep_wait();  // every global access of this kernel comes after the previous kernel of the stream
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) PFwdBarriers bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = a.n_tiles;
  const int n_items = T * a.B * a.H;
  const int G = gridDim.x, c = blockIdx.x;
  const WaitCtx wc{&abort_flag, a.status};
  uint8_t* smQ = smem + L::kQ;
  uint8_t* smK = smem + L::kK;
  uint8_t* smV = smem + L::kV;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.q_full[i], 1);
      mbar_init(&bar.q_empty[i], 1);
      mbar_init(&bar.k_full[i], 1);
      mbar_init(&bar.k_empty[i], 1);
      mbar_init(&bar.v_full[i], 1);
      mbar_init(&bar.v_empty[i], 1);
    }
    mbar_init(&bar.s_full, 1);
    mbar_init(&bar.s_free, 128);
    mbar_init(&bar.p_full, 128);
    mbar_init(&bar.o_done, 1);
    mbar_init(&bar.o_free, 128);
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
    if (lane == 0 || lane == 2) {
      // lane 0: K, lane 2: V of every (item, key tile) pair, each through its own ring;
      // one loop for both lanes, which keeps them in step (see above)
      const bool is_k = lane == 0;
      tma_prefetch_desc(is_k ? &tm_k : &tm_v);
      uint64_t* full = is_k ? bar.k_full : bar.v_full;
      uint64_t* empty = is_k ? bar.k_empty : bar.v_empty;
      uint8_t* ring = is_k ? smK : smV;
      const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
      int u = 0;
      bool ok = true;
      for (FwdCursor cu = pfwd_cursor_from(0, 0, c, G, n_items, a); cu.j >= 0;
           cu = pfwd_cursor_next(cu, c, G, n_items, a)) {
        const int s = u % S;
        if (u >= S && !(ok = mbar_wait(&empty[s], ((u / S) - 1) & 1, wc))) break;
        mbar_arrive_expect_tx(&full[s], L::kTileBytes);
        tma_load_3d(ring + s * L::kTileBytes, tm, &full[s], 0, cu.kt * kTile, cu.w.head);
        ++u;
      }
      if (!ok) {
        // let the loads already issued land before the CTA can exit
        for (int i = (u > S ? u - S : 0); i < u; ++i) mbar_drain(&full[i % S], (i / S) & 1, 100000000ull);
      }
    } else if (lane == 1) {
      // Q of every item with a visible key tile; the k-th goes to buffer k % 2, which
      // the epilogue of the (k-2)-th frees
      tma_prefetch_desc(&tm_q);
      int k = 0;
      bool ok = true;
      for (int j = 0, idx; ok && (idx = pfwd_item(j, c, G, n_items)) >= 0; ++j) {
        const FwdItem w = pfwd_decode(idx, a);
        if (next_key_tile(w.qt, 0, w.kv_len, a.causal, a.block_mask, T) >= T) continue;
        const int qb = k & 1;
        if (k >= 2 && !(ok = mbar_wait(&bar.q_empty[qb], ((k >> 1) - 1) & 1, wc))) break;
        mbar_arrive_expect_tx(&bar.q_full[qb], L::kTileBytes);
        tma_load_3d(smQ + qb * L::kTileBytes, &tm_q, &bar.q_full[qb], 0, w.qt * kTile, w.head);
        ++k;
      }
      if (!ok)
        for (int i = (k > 2 ? k - 2 : 0); i < k; ++i) mbar_drain(&bar.q_full[i & 1], (i >> 1) & 1, 100000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, false, true);
      const uint64_t kdesc = sdesc_sw128(smem_u32(smK), 16, 1024);
      const uint64_t vdesc = sdesc_sw128(smem_u32(smV), L::kSubBytes, 1024);
      bool ok = true;
      // S = Q K^T of pair `cur` from K/V stage `stage` into the S columns
      auto issue_scores = [&](const FwdCursor& cur, int stage) {
        const uint64_t qdesc = sdesc_sw128(smem_u32(smQ + (cur.k & 1) * L::kTileBytes), 16, 1024);
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_bf16_ss(tmem + L::kColS, sdesc_adv(qdesc, k * 32), sdesc_adv(kdesc, stage * L::kTileBytes + k * 32),
                      idesc_s, k > 0 ? 1u : 0u);
        mma_commit(&bar.s_full);
        mma_commit(&bar.k_empty[stage]);
      };
      int u = 0;  // pairs so far (= S and P V products, = K/V ring uses)
      FwdCursor cur = pfwd_cursor_from(0, 0, c, G, n_items, a);
      if (cur.j >= 0) {
        ok = mbar_wait_sleep(&bar.q_full[0], 0, wc) && mbar_wait_sleep(&bar.k_full[0], 0, wc);
        if (ok) issue_scores(cur, 0);
      }
      // The next scores go out as soon as the softmax warps have read these out of TMEM,
      // before this pair's P V, also when they are the next item's first: that item's Q
      // buffer is freed by the epilogue two items back, which waits for no later P V.
      // (Issuing them after the item's last P V instead left each item boundary ~5000
      // clk longer than a pair: 5% of the GPT-2-shaped forward.)
      auto next_scores = [&](const FwdCursor& cur, const FwdCursor& nxt) -> bool {
        if (nxt.j != cur.j && !mbar_wait_sleep(&bar.q_full[nxt.k & 1], (nxt.k >> 1) & 1, wc)) return false;
        if (!mbar_wait_sleep(&bar.k_full[(u + 1) % S], ((u + 1) / S) & 1, wc)) return false;
        if (!mbar_wait_sleep(&bar.s_free, u & 1, wc)) return false;
        issue_scores(nxt, (u + 1) % S);
        return true;
      };
      while (ok && cur.j >= 0) {
        const FwdCursor nxt = pfwd_cursor_next(cur, c, G, n_items, a);
        const int s = u % S;
        if (nxt.j >= 0 && !(ok = next_scores(cur, nxt))) break;
        // O (+)= P V; the first product of an item overwrites the accumulator, which the
        // epilogue of the CTA's previous item with a visible key tile must have read out
        if (!(ok = mbar_wait_sleep(&bar.v_full[s], (u / S) & 1, wc))) break;
        if (!(ok = mbar_wait_sleep(&bar.p_full, u & 1, wc))) break;
        if (cur.first && cur.k >= 1 && !(ok = mbar_wait_sleep(&bar.o_free, (cur.k - 1) & 1, wc))) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k)
          mma_bf16_ts(tmem + L::kColO, tmem + L::kColP + k * 8, sdesc_adv(vdesc, s * L::kTileBytes + k * 2048),
                      idesc_o, (!cur.first || k > 0) ? 1u : 0u);
        mma_commit(&bar.o_done);
        mma_commit(&bar.v_empty[s]);
        cur = nxt;
        ++u;
      }
      if (!ok) {
        mma_commit(&bar.drain);
        mbar_drain(&bar.drain, 0, 100000000ull);
      }
    }
  } else {
    // --------------------------------------------------- softmax + epilogue (warps 2..5)
    const int wq = warp & 3;  // TMEM lane quarter this warp may access
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off + L::kColS;
    const uint32_t t_p = tmem + lane_off + L::kColP;
    const uint32_t t_o = tmem + lane_off + L::kColO;
    const float sl2 = a.scale_log2;
    bool ok = true;
    int u = 0;  // pairs so far, over all items
    int k = 0;  // items with a visible key tile so far
    // Every warp walks every item; an item with a visible key tile reaches the epilogue
    // barrier once, also after a wait has given up (ok == false), so the named barrier
    // stays matched.
    for (int j = 0, idx; (idx = pfwd_item(j, c, G, n_items)) >= 0; ++j) {
      const FwdItem w = pfwd_decode(idx, a);
      const int q_row = w.qt * kTile + r;
      if (next_key_tile(w.qt, 0, w.kv_len, a.causal, a.block_mask, T) >= T) {
        // no key visible: O = 0 and LSE = -inf, by plain stores; no barrier involved
        if (q_row < a.N) {
          uint4* orow = reinterpret_cast<uint4*>(o_out + (static_cast<size_t>(w.head) * a.N + q_row) * D);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) orow[i] = make_uint4(0u, 0u, 0u, 0u);
          lse_out[static_cast<size_t>(w.head) * a.N + q_row] = neg_inf();
        }
        continue;
      }
      const int qb = k & 1;
      float m_run = neg_inf();  // max used for the exponentials, log2 domain (scale * log2 e applied)
      float l_run = 0.f;        // running sum of exp2(s - m_run)
      int n = 0;                // key tiles of this item
      for (int kt = next_key_tile(w.qt, 0, w.kv_len, a.causal, a.block_mask, T); ok && kt < T;
           kt = next_key_tile(w.qt, kt + 1, w.kv_len, a.causal, a.block_mask, T), ++n, ++u) {
        ok = mbar_wait(&bar.s_full, u & 1, wc);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        float sv[kTile];
        {
          uint32_t t[kTile];
          tmem_ld128(t_s, t);
#pragma unroll
          for (int i = 0; i < kTile; ++i) sv[i] = __uint_as_float(t[i]);
        }
        tc_fence_before();
        mbar_arrive(&bar.s_free);  // the MMA warp may overwrite S with the next scores
        // element mask: key padding tail, causal diagonal (the N tail is covered by kv_len <= N)
        const int key0 = kt * kTile;
        if (key0 + kTile > w.kv_len || (a.causal && kt == w.qt)) {
          const int lim = a.causal ? min(w.kv_len, q_row + 1) : w.kv_len;  // keys [key0, lim) visible
#pragma unroll
          for (int cc = 0; cc < kTile; ++cc)
            if (key0 + cc >= lim) sv[cc] = neg_inf();
        }
        const float mx = row_max128(sv) * sl2;
        const float m_new = (mx > m_run + kRescaleSlack) ? mx : m_run;
        const float m_use = (m_new == neg_inf()) ? 0.f : m_new;
        const float alpha = ex2(m_run - m_use);
#pragma unroll
        for (int cc = 0; cc < kTile; cc += 2) {
          ffma2(sv[cc], sv[cc + 1], sv[cc], sv[cc + 1], sl2, -m_use);
          sv[cc] = ex2(sv[cc]);
          sv[cc + 1] = ex2(sv[cc + 1]);
        }
        const float tile_sum = row_sum128(sv);
        uint32_t pk[kTile / 2];
#pragma unroll
        for (int cc = 0; cc < kTile; cc += 2) pk[cc / 2] = pack_bf16x2(sv[cc], sv[cc + 1]);
        l_run = l_run * alpha + tile_sum;
        m_run = m_new;
        // the previous P V has read P and updated O
        if (u > 0) {
          ok = mbar_wait(&bar.o_done, (u - 1) & 1, wc);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
        }
        tmem_st64(t_p, pk);
        if (n > 0 && __any_sync(0xffffffffu, alpha < 1.f)) {
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
        mbar_arrive(&bar.p_full);
      }

      // epilogue: O = O_acc / l (bf16) staged in this item's Q buffer and stored by TMA; LSE = m + ln l
      bool have_o = ok && n > 0;
      if (have_o) {
        ok = mbar_wait(&bar.o_done, (u - 1) & 1, wc);  // this item's last P V
        have_o = __all_sync(0xffffffffu, ok);
        ok = have_o;
        tc_fence_after();
      }
      uint32_t wo[D / 2];
      {
        const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
        uint32_t t[D];
        if (have_o) {
          tmem_ld64(t_o, t);
        } else {
#pragma unroll
          for (int i = 0; i < D; ++i) t[i] = 0u;
        }
#pragma unroll
        for (int i = 0; i < D / 2; ++i)
          wo[i] = pack_bf16x2(__uint_as_float(t[2 * i]) * inv_l, __uint_as_float(t[2 * i + 1]) * inv_l);
      }
      tc_fence_before();
      mbar_arrive(&bar.o_free);  // the accumulator may be overwritten by the next item with a visible key
      // the Q tile has landed and no MMA reads it any more
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar.q_full[qb], (k >> 1) & 1, wc));
      const uint32_t orow = smem_u32(smQ + qb * L::kTileBytes);
#pragma unroll
      for (int q = 0; q < D / 8; ++q)
        st_shared_v4(orow + sw128_offset(r, q), wo[4 * q], wo[4 * q + 1], wo[4 * q + 2], wo[4 * q + 3]);
      fence_proxy_async_smem();
      named_barrier(1, 128);
      if (wq == 2 && lane == 0) {
        tma_store_3d(&tm_o, smQ + qb * L::kTileBytes, 0, w.qt * kTile, w.head);
        tma_store_commit();
        bulk_wait_read_all();
        mbar_arrive(&bar.q_empty[qb]);  // the staging tile has been read: the producer may load the Q two items on
      }
      if (q_row < a.N) {
        const float lse = (n > 0 && l_run > 0.f) ? (m_run + log2f(l_run)) * kLn2 : neg_inf();
        lse_out[static_cast<size_t>(w.head) * a.N + q_row] = lse;
      }
      ++k;
    }
    if (wq == 2 && lane == 0) tma_store_wait_all();
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
  using L = FwdLayout<D, NQ, false>;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(fwd_bf16_kernel<D, NQ>), L::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>((a.n_tiles + NQ - 1) / NQ) * a.B * a.H;
  return launch_pdl(fwd_bf16_kernel<D, NQ>, static_cast<unsigned>(grid), L::kThreads, L::kSmemBytes, stream, maps.q,
                    maps.k, maps.v, maps.o, lse, a);
}

}  // namespace

cudaError_t launch_fwd_splitkv(const FwdMaps& maps, void* o, float* lse, const AttnArgs& a, cudaStream_t stream) {
  using L = FwdLayout<128, 2, false>;
  const long long rows = static_cast<long long>(a.B) * a.H * a.N;
  if (a.n_chunks > 0 && a.nk > 0) {
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(fwd_splitkv_kernel), L::kSmemBytes);
    if (e != cudaSuccess) return e;
    const long long grid = static_cast<long long>(a.n_tiles) * a.n_chunks * a.B * a.H;
    e = launch_pdl(fwd_splitkv_kernel, static_cast<unsigned>(grid), L::kThreads, L::kSmemBytes, stream, maps.q, maps.k,
                   maps.v, maps.o, lse, a);
    if (e != cudaSuccess) return e;
  }
  const int parts = (a.n_chunks > 0 && a.nk > 0) ? 2 * a.n_chunks : 0;
  const long long blocks = (rows * 32 + 255) / 256;
  return launch_pdl(splitkv_combine_kernel, static_cast<unsigned>(blocks), 256, 0, stream,
                    static_cast<const float*>(a.part_o), static_cast<const float*>(a.part_lse),
                    static_cast<uint16_t*>(o), lse, rows, parts);
}

cudaError_t launch_fwd_fp8(const FwdMaps& maps, float* lse, const AttnArgs& a, cudaStream_t stream) {
  using L = FwdLayout<128, 2, true>;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(fwd_fp8_kernel), L::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>((a.n_tiles + 1) / 2) * a.B * a.H;
  return launch_pdl(fwd_fp8_kernel, static_cast<unsigned>(grid), L::kThreads, L::kSmemBytes, stream, maps.q, maps.k,
                    maps.v, maps.o, lse, a);
}

cudaError_t launch_fwd_bf16(const FwdMaps& maps, float* lse, const AttnArgs& a, cudaStream_t stream) {
  if (a.d == 128) return launch_fwd_d<128, 2>(maps, lse, a, stream);
  // d = 64: persistent, two CTAs per SM
  using L = PFwdLayout<64>;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(fwd_persistent_kernel<64>), L::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long n_items = static_cast<long long>(a.n_tiles) * a.B * a.H;
  const long long slots = 2LL * sm_count();
  const long long grid = n_items < slots ? n_items : slots;
  return launch_pdl(fwd_persistent_kernel<64>, static_cast<unsigned>(grid), L::kThreads, L::kSmemBytes, stream, maps.q,
                    maps.k, maps.v, maps.o, static_cast<uint16_t*>(maps.o_ptr), lse, a);
}

}  // namespace fa
