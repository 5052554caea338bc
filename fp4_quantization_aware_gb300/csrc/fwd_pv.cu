// Attn-QAT forward, pass 2 at D = 128 (sm_103a): P, P^, O' and O from the LSE.
//
// "Attn-QAT: 4-Bit Attention With Quantization-Aware Training" (Method, Fix 1)
// and "NVFP4 Attention QAT Backward" (cuDNN frontend docs, Overview):
//   P   = exp(scale * Q^ K^T - LSE)     (the normalised probabilities, FP32)
//   O'  = P V^                          (auxiliary high-precision output, BF16)
//   O   = fake_nvfp4(P) V^              (groups of 16 keys of the normalised P)
// The LSE comes from pass 1 (fwd_lse.cu), so every key tile's P is final when
// it is formed and O', O accumulate in TMEM with no rescaling.
//
// One CTA per 128-row query tile, key tiles of 64. S of a key tile is ready
// for the softmax warps once its S MMA has run, and its buffer can take the
// S of a later tile only once the O' and O MMAs that read P and P^ from it
// have completed. With three S buffers the S MMA runs up to three tiles ahead
// of those MMAs, so the softmax warps always find a computed S and the tensor
// core always finds P of an earlier tile to multiply: neither waits for the
// other's latest step (with two buffers of 128 keys, S(t + 2) queued behind
// the O', O MMAs of tile t + 1 and each side idled while the other worked).
//
// TMEM columns: S buffer b (key tile t, b = t % 3) at 64 b; scale factors of
// the block-scaled S MMA at 192 + 4 ks (Q) and 200 + 8 (t % 4) + 4 ks (K of
// key tile t), 4 columns per K = 64 step, 4-column aligned; O' at 256, O at
// 384. A tile's 64 keys are split into kParts parts of kPartKeys keys, one
// softmax warp per part and lane quarter; the warp of part p writes P (BF16
// pairs) over the first half of the S columns it read, [kPartKeys p,
// + kPartKeys / 2), and P^ over the second half, and the O' and O MMAs take
// their A operand from TMEM there, 16 keys per MMA.
//
// Warps: 4 kParts softmax (warp w: lane quarter w % 4, key part w / 4; the
// last part of each half of the parts also writes the K scale factors of K
// step (its half), three tiles ahead), then the TMA producer and the MMA
// issuers of O', O and S, on SM sub-partitions 0-3 (an issuing thread slows
// the softmax warps of its own sub-partition, so the issue work is spread
// out).
// Shared memory: V^ x6 (16 KiB a tile), NVFP4 Q 8 KiB, NVFP4 K x6 (4 KiB).
#include "attn_common.cuh"
#include "fp4_mma.cuh"
#include "checked.cuh"

namespace attnqat {
namespace {

constexpr int kParts = 4;                    // key parts of a tile (softmax warps per lane quarter)
constexpr int kPartKeys = 64 / kParts;       // keys of a tile per softmax warp
constexpr int kGroups = kPartKeys / 16;      // NVFP4 groups of P per softmax warp and tile
constexpr int kSoftWarpsV = 4 * kParts;
constexpr int kThreadsV = (kSoftWarpsV + 4) * 32;
constexpr int kWarpTmaV = kSoftWarpsV;       // sub-partition 0
constexpr int kWarpMmaOP = kSoftWarpsV + 1;  // O' += P V^ (and TMEM allocation)
constexpr int kWarpMmaOV = kSoftWarpsV + 2;  // O += P^ V^
constexpr int kWarpMmaSV = kSoftWarpsV + 3;  // S
constexpr int kKeysV = 64;                   // keys per tile
constexpr int kRing = 3;                     // S buffers
constexpr int kSfSlots = 4;                  // K scale-factor slots

struct PvLayout {
  static constexpr int kStages = 6;                       // K and V tiles in flight
  static constexpr uint32_t kVBlock = kKeysV * 128;       // 64 keys x 64 values of D (128 bytes a row)
  static constexpr uint32_t kVTile = 2 * kVBlock;         // both 64-wide halves of D
  static constexpr uint32_t kFp4Row = 64;                 // 128 E2M1 values
  static constexpr uint32_t kQ4Tile = 128 * kFp4Row;
  static constexpr uint32_t kK4Tile = kKeysV * kFp4Row;
  static constexpr uint32_t kV0 = 0;                      // stage s at kV0 + s * kVTile
  static constexpr uint32_t kQ4 = kV0 + kStages * kVTile;
  static constexpr uint32_t kK40 = kQ4 + kQ4Tile;         // stage s at kK40 + s * kK4Tile
  static constexpr uint32_t kBar = kK40 + kStages * kK4Tile;
  static constexpr uint32_t kBytes = kBar + 512;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static constexpr uint32_t kColSFQ = kRing * kKeysV;     // 192 (+ 4 ks)
  static constexpr uint32_t kColSFK = kColSFQ + 8;        // 200 (+ 8 slot + 4 ks)
  static constexpr uint32_t kColOP = 256;
  static constexpr uint32_t kColO = 384;
  // epilogue: O' then O as BF16, each two blocks of 128 rows x 64 columns, over the V^ stages
  static constexpr uint32_t kOutBlock = 128 * 128;
  static_assert(4 * kOutBlock <= kStages * kVTile, "output staging fits the V^ stages");
  // split tiles: FP32 O' then O, each four blocks of 128 rows x 32 columns,
  // over the V^, Q and K stages (free once every MMA is done)
  static constexpr uint32_t kSplitBlock = 128 * 32 * 4;
  static_assert(8 * kSplitBlock <= kBar && kV0 == 0, "split staging fits below the barriers");
  static_assert(kVBlock % 1024 == 0 && kQ4 % 1024 == 0 && kK40 % 1024 == 0 && kK4Tile % 512 == 0,
                "swizzled tiles need 1024-byte (128-byte swizzle) or 512-byte (64-byte swizzle) alignment");
  static_assert(kColSFQ % 4 == 0 && kColSFK % 4 == 0 && kColSFK + 8 * kSfSlots <= kColOP,
                "scale factors: 4-column aligned, between the S ring and O'");
  static_assert(kAlloc <= 227 * 1024, "shared memory");
};

struct PvBars {
  uint64_t q_full;
  uint64_t k_full[PvLayout::kStages], k_empty[PvLayout::kStages];
  uint64_t v_full[PvLayout::kStages], v_empty[PvLayout::kStages];
  uint64_t s_full[kRing];    // S of the buffer's tile complete
  uint64_t p_ready[kRing];   // P and P^ of the buffer's tile in place (and later K scales written)
  uint64_t pv_read[kRing];   // the O' and O MMAs of the buffer's tile complete
  uint64_t o_done;           // one phase: every O' and O MMA has completed
  uint64_t sf_init;          // Q scales and the first three tiles' K scales in TMEM
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
  uint32_t split_order;      // split tiles: this CTA's place in the slot's count (0 or 1)
  uint64_t split_in;         // split tiles, second CTA: the other CTA's partial rows loaded
};
static_assert(sizeof(PvBars) <= 512, "barrier block");

struct PvArgs {
  const uint8_t* q_sf;   // NVFP4 scales of Q, K ((B*H, S, 8) E4M3)
  const uint8_t* k_sf;
  const float* lse;      // natural-log LSE of every query row (pass 1)
  bf16* o;
  bf16* o_hp;
  int Sq, Sk;
  int n_qtiles, n_ktiles;   // 128-row query tiles, 64-key tiles
  int n_full;               // CTAs 0 .. n_full - 1 own whole query tiles; then two CTAs per split tile
  float* split_acc;         // split tiles: FP32 [slot][rank][O', O][128][128] (also as tm_slot)
  uint32_t* split_cnt;      // ... and zeroed counters
  int causal;
  float c2;                 // scale * log2(e)
  uint32_t* err;
  uint64_t timeout_ns;
  ATTNQAT_CHECKED_ONLY(int64_t rows_q; int64_t rows_k; int64_t n_split;)   // debug build: B*H*Sq, B*H*Sk, split tiles
};

// 16 TMEM columns of this warp's 32 lanes, without waiting: tmem_wait_ld16
// waits for the load, and the registers pass through its asm block, so no use
// of them moves above the wait.
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_st4_nowait(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}

__global__ void __launch_bounds__(kThreadsV, 1)
    fwd_pv_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q4,
                  const __grid_constant__ CUtensorMap tm_k4, const __grid_constant__ CUtensorMap tm_ohp,
                  const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_slot,
                  const PvArgs a) {
  using L = PvLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  PvBars& B = *reinterpret_cast<PvBars*>(smem + L::kBar);

  const int warp = warp_id();
  const int lane = lane_id();
  // 1-D grid, query tiles fastest within a head (causal: the longest first).
  // CTA n_full + 2 u + rank works on split tile n_full + u: rank 0 takes the
  // first half of its key tiles (rounded up), rank 1 the rest.
  const int lin = static_cast<int>(blockIdx.x);
  const bool split_cta = lin >= a.n_full;
  const int sidx = split_cta ? (lin - a.n_full) >> 1 : 0;
  const int rank = split_cta ? ((lin - a.n_full) & 1) : 0;
  const int tile = split_cta ? a.n_full + sidx : lin;
  const int bh = tile / a.n_qtiles;
  const int i = a.causal ? (a.n_qtiles - 1 - tile % a.n_qtiles) : tile % a.n_qtiles;
  const int n_total = a.causal ? min(a.n_ktiles, 2 * i + 2) : a.n_ktiles;
  const int n_half0 = split_cta ? (n_total + 1) / 2 : n_total;
  // this CTA's key tiles: kt0 + t for t < nt (t indexes buffers, stages and phases)
  const int kt0 = rank == 0 ? 0 : n_half0;
  const int nt = rank == 0 ? n_half0 : n_total - n_half0;

  if (threadIdx.x == 0) {
    B.abort_flag = 0;
    mbar_init(&B.q_full, 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&B.k_full[s], 1), mbar_init(&B.k_empty[s], 1);
      mbar_init(&B.v_full[s], 1), mbar_init(&B.v_empty[s], 2);   // read by the O' and the O MMAs
    }
    for (int b = 0; b < kRing; ++b) {
      mbar_init(&B.s_full[b], 1);
      mbar_init(&B.p_ready[b], kSoftWarpsV * 32);
      mbar_init(&B.pv_read[b], 2);   // one commit each from the O' and O issuers
    }
    mbar_init(&B.o_done, 2);
    mbar_init(&B.split_in, 1);
    mbar_init(&B.sf_init, 2 * 128);   // key parts 1 and 3
    mbar_init(&B.drain, 3);           // one commit per MMA-issuing thread
    fence_mbar_init();
  }
  if (warp == kWarpMmaOP) {
    tmem_alloc(&B.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B.tmem_base;
  const WaitCtl ctl{&B.abort_flag, a.err, a.timeout_ns};
  // Launched as a programmatic dependent of the LSE pass, which let this one
  // start only after the quantize step had completed: its NVFP4 Q, K, scales
  // and V^ are readable now, the LSE only after grid_dep_wait (softmax warps).

  if (warp == kWarpTmaV) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_v), tma_prefetch_desc(&tm_q4), tma_prefetch_desc(&tm_k4);
      tma_prefetch_desc(&tm_ohp), tma_prefetch_desc(&tm_o);
      mbar_arrive_expect_tx(&B.q_full, L::kQ4Tile);
      tma_load_3d(smem + L::kQ4, &tm_q4, &B.q_full, 0, i * 128, bh);
      int k_uses[L::kStages] = {}, v_uses[L::kStages] = {};
      for (int t = 0; t < nt; ++t) {
        const int s = t % L::kStages, use = t / L::kStages;
        if (use >= 1 && !mbar_wait(&B.k_empty[s], (use - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(&B.k_full[s], L::kK4Tile);
        tma_load_3d(smem + L::kK40 + s * L::kK4Tile, &tm_k4, &B.k_full[s], 0, (kt0 + t) * kKeysV, bh);
        ++k_uses[s];
        if (use >= 1 && !mbar_wait(&B.v_empty[s], (use - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(&B.v_full[s], L::kVTile);
        for (int h = 0; h < 2; ++h)
          tma_load_3d(smem + L::kV0 + s * L::kVTile + h * L::kVBlock, &tm_v, &B.v_full[s], h * 64, (kt0 + t) * kKeysV,
                      bh);
        ++v_uses[s];
      }
      // every copy issued above lands before shared memory is released
      mbar_wait_drain(&B.q_full, 0, ctl);
      for (int s = 0; s < L::kStages; ++s) {
        if (k_uses[s]) mbar_wait_drain(&B.k_full[s], (k_uses[s] - 1) & 1, ctl);
        if (v_uses[s]) mbar_wait_drain(&B.v_full[s], (v_uses[s] - 1) & 1, ctl);
      }
    }
  } else if (warp == kWarpMmaSV) {
    // ------------------------------------------------------------ S issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_nvfp4(128, kKeysV);
      const uint64_t dq = sdesc_sw64(sbase + L::kQ4);
      const uint64_t dk0 = sdesc_sw64(sbase + L::kK40);
      bool ok = mbar_wait(&B.q_full, 0, ctl) && mbar_wait(&B.sf_init, 0, ctl);
      for (int t = 0; ok && t < nt; ++t) {
        const int b = t % kRing, s = t % L::kStages;
        const bool kf = mbar_try_wait(&B.k_full[s], (t / L::kStages) & 1);
        // S(t) goes where S(t - 3) was, once the O' and O MMAs reading P(t - 3)
        // and P^(t - 3) from there have completed. The softmax warps wrote key
        // tile t's K scales before their p_ready arrival for tile t - 3, whose
        // phase (complete by then) is also waited for here, so that the writes
        // are ordered before this thread's MMA directly.
        if ((t >= kRing && !mbar_wait_both(&B.p_ready[b], ((t / kRing) - 1) & 1, &B.pv_read[b],
                                           ((t / kRing) - 1) & 1, ctl)) ||
            (!kf && !mbar_wait(&B.k_full[s], (t / L::kStages) & 1, ctl))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dk = sdesc_advance(dk0, s * L::kK4Tile);
        const uint32_t sfk = L::kColSFK + 8 * (t % kSfSlots);
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          umma_nvfp4(tmem + b * kKeysV, sdesc_advance(dq, ks * 32), sdesc_advance(dk, ks * 32), kIdS,
                     tmem + L::kColSFQ + 4 * ks, tmem + sfk + 4 * ks, ks > 0);
        umma_commit(&B.s_full[b]);
        umma_commit(&B.k_empty[s]);
      }
      umma_commit(&B.drain);
      mbar_wait_drain(&B.drain, 0, ctl);
    }
  } else if (warp == kWarpMmaOP || warp == kWarpMmaOV) {
    // ------------------------------------------------------------ O', O issuers
    // O' += P V^ (A at 64 b + 16 kk), O += P^ V^ (A at 64 b + 16 kk + 8): one
    // MMA per 16 keys, V^ MN-major in shared memory (16 rows of 128 bytes per
    // K = 16 step, the two halves of D kVBlock apart).
    if (lane == 0) {
      const bool is_op = warp == kWarpMmaOP;
      constexpr uint32_t kIdO = idesc_bf16(128, 128, false, true);
      const uint64_t dv0 = sdesc_sw128(sbase + L::kV0, L::kVBlock, 1024);
      const uint32_t dcol = is_op ? L::kColOP : L::kColO;
      const uint32_t acol = is_op ? 0u : 8u * kGroups;   // P, then P^, in each part's columns
      bool ok = true;
      for (int t = 0; ok && t < nt; ++t) {
        const int b = t % kRing, s = t % L::kStages;
        if (!mbar_wait_both(&B.v_full[s], (t / L::kStages) & 1, &B.p_ready[b], (t / kRing) & 1, ctl)) break;
        tc_fence_after();
        const uint64_t dv = sdesc_advance(dv0, s * L::kVTile);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_tmem_a(tmem + dcol, tmem + b * kKeysV + (kk / kGroups) * kPartKeys + 8 * (kk % kGroups) + acol,
                           sdesc_advance(dv, kk * 2048), kIdO,
                           (t > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&B.v_empty[s]);
        umma_commit(&B.pv_read[b]);
        if (t == nt - 1) umma_commit(&B.o_done);
      }
      umma_commit(&B.drain);
      mbar_wait_drain(&B.drain, 0, ctl);
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 0-15)
    const uint32_t quarter = warp & 3, part = warp >> 2;
    // the last part of each half of the tile's parts writes the K scales of
    // K step (its half)
    constexpr uint32_t kHalf = kParts / 2;
    const bool sf_writer = part % kHalf == kHalf - 1;
    const int ks = static_cast<int>(part / kHalf);
    const uint32_t r = quarter * 32 + lane;
    const uint32_t lane_off = (quarter * 32u) << 16;
    const int qrow = i * 128 + static_cast<int>(r);
    const int kend = a.causal ? min(a.Sk, qrow + 1) : a.Sk;
    const int64_t kbase = static_cast<int64_t>(bh) * a.Sk;
    auto k_scales = [&](int t, uint32_t (&w)[4]) {   // this CTA's tile t; rows past the tile's 64 stay 0
      const int kt = kt0 + t;
      const int rows = min(kKeysV, a.Sk - kt * kKeysV);
      load_scales(a.k_sf, kbase + static_cast<int64_t>(kt) * kKeysV,
                  ATTNQAT_IN_BOUNDS(kbase + static_cast<int64_t>(kt) * kKeysV + rows <= a.rows_k) ? rows : 0, ks, w);
    };
    // K scales written at tile t (those of tile t + 3), loaded one tile ahead.
    // The prologue issues all of its scale loads before the first TMEM store.
    uint32_t sfw[4] = {0u, 0u, 0u, 0u};
    if (sf_writer) {
      uint32_t w[1 + kRing][4];
      load_scales(a.q_sf, static_cast<int64_t>(bh) * a.Sq + i * 128,
                  ATTNQAT_IN_BOUNDS(static_cast<int64_t>(bh) * a.Sq + i * 128 + min(128, a.Sq - i * 128) <= a.rows_q)
                      ? min(128, a.Sq - i * 128) : 0,
                  ks, w[0]);
#pragma unroll
      for (int kt = 0; kt < kRing; ++kt)
        if (kt < nt) k_scales(kt, w[1 + kt]);
      if (kRing < nt) k_scales(kRing, sfw);
      tmem_st4_nowait(tmem + lane_off + L::kColSFQ + 4 * ks, w[0]);
#pragma unroll
      for (int kt = 0; kt < kRing; ++kt)
        if (kt < nt) tmem_st4_nowait(tmem + lane_off + L::kColSFK + 8 * (kt % kSfSlots) + 4 * ks, w[1 + kt]);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&B.sf_init);
    }
    grid_dep_wait();
    const float lse2 = qrow < a.Sq && ATTNQAT_IN_BOUNDS(static_cast<int64_t>(bh) * a.Sq + qrow < a.rows_q)
                           ? __ldg(a.lse + static_cast<size_t>(bh) * a.Sq + qrow) * kLog2e : 0.0f;
    const float2 c22 = make_float2(a.c2, a.c2), nl = make_float2(-lse2, -lse2);
    // One tile: P = exp2(S c2 - lse2), P^ = fake_nvfp4(P) over this warp's S
    // columns, key tile t + 3's K scales from `sf_now` into their slot, key
    // tile t + 4's scales loaded into `sf_next` (written a tile later; the
    // loop below alternates the two arrays, so no copy waits for the load).
    auto tile = [&](int t, const uint32_t (&sf_now)[4], uint32_t (&sf_next)[4]) -> bool {
      const int b = t % kRing;
      const int valid = kend - ((kt0 + t) * kKeysV + static_cast<int>(part) * kPartKeys);
      if (sf_writer && t + kRing + 1 < nt) k_scales(t + kRing + 1, sf_next);
      if (!warp_wait(&B.s_full[b], (t / kRing) & 1, ctl)) return false;
      tc_fence_after();
      // this warp's S columns; P of group g over columns 8 g, P^ over 8 kGroups + 8 g
      const uint32_t pcol = tmem + lane_off + b * kKeysV + part * kPartKeys;
      uint32_t v[kGroups][16];
#pragma unroll
      for (int g = 0; g < kGroups; ++g) tmem_ld16_nowait(pcol + 16 * g, v[g]);
#pragma unroll
      for (int g = 0; g < kGroups; ++g) tmem_wait_ld16(v[g]);
#pragma unroll
      for (int g = 0; g < kGroups; ++g) {
        float P[16];
#pragma unroll
        for (int k = 0; k < 16; k += 2) {
          const float2 e = ffma2(make_float2(__uint_as_float(v[g][k]), __uint_as_float(v[g][k + 1])), c22, nl);
          P[k] = ex2(e.x), P[k + 1] = ex2(e.y);
        }
        if (valid < 16 * (g + 1)) {   // masked keys: P = 0
#pragma unroll
          for (int k = 0; k < 16; ++k)
            if (16 * g + k >= valid) P[k] = 0.0f;
        }
        // P in words 0-7, P^ in words 8-15: with one group per warp their
        // columns (8 g and 8 kGroups + 8 g) are adjacent, one 16-column store
        uint32_t pw[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) pw[k] = pack_bf16x2(P[2 * k], P[2 * k + 1]);
        fake_nvfp4_16_pack_nonneg<false>(P, 1.0f, pw + 8);
        if constexpr (kGroups == 1) {
          tmem_st16_nowait(pcol, pw);
        } else {
          tmem_st8_nowait(pcol + 8 * g, pw);
          tmem_st8_nowait(pcol + 8 * kGroups + 8 * g, pw + 8);
        }
      }
      // key tile t + 3's K scales into slot (t + 3) % 4, last read by S(t - 1),
      // which is complete since S(t) is; S(t + 3) is issued only after the
      // O' and O MMAs that wait for this tile's p_ready
      if (sf_writer && t + kRing < nt)
        tmem_st4_nowait(tmem + lane_off + L::kColSFK + 8 * ((t + kRing) % kSfSlots) + 4 * ks, sf_now);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&B.p_ready[b]);
      return true;
    };
    uint32_t sfo[4] = {0u, 0u, 0u, 0u};
    bool ok = true;
    for (int t = 0; ok && t < nt; t += 2) {
      ok = tile(t, sfw, sfo);
      if (ok && t + 1 < nt) ok = tile(t + 1, sfo, sfw);
    }
    // epilogue: part p stores columns [128 / kParts p, + 128 / kParts) of O'
    // and O (a one-shot barrier committed after the last O' and O MMAs). The
    // two CTAs of a split tile store their FP32 rows in the tile's slot; the
    // one that counts second adds the other's and stores the BF16 sums.
    const bool have = ok && nt > 0 && warp_wait(&B.o_done, 0, ctl);
    if (have) tc_fence_after();
    constexpr int kCols = 128 / kParts;
    if (!split_cta) {
      // O' and O as BF16 in the free V^ area (all O', O MMAs are done), two
      // 64-column 128-byte-swizzled blocks each, then four TMA stores, so the
      // rows go out coalesced (rows past Sq are clipped by the tensor maps)
      if (have) {
#pragma unroll
        for (int o = 0; o < 2; ++o) {
#pragma unroll
          for (int c = 0; c < kCols; c += 32) {
            const uint32_t col = part * kCols + c;
            uint32_t v[32], w[16];
            tmem_ld32(tmem + lane_off + (o == 0 ? L::kColOP : L::kColO) + col, v);
#pragma unroll
            for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]));
            const uint32_t blk = sbase + L::kV0 + o * 2 * L::kOutBlock + (col / 64) * L::kOutBlock;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              st_shared_v4(sw128_chunk(blk, r, (col % 64) / 8 + j), w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
          }
        }
        fence_proxy_async_smem();
      }
      named_bar_sync(1, kSoftWarpsV * 32);
      if (have && warp == 0 && lane == 0) {
#pragma unroll
        for (int o = 0; o < 2; ++o)
#pragma unroll
          for (int h = 0; h < 2; ++h)
            tma_store_3d(o == 0 ? &tm_ohp : &tm_o, smem + L::kV0 + (2 * o + h) * L::kOutBlock, 64 * h, i * 128, bh);
        bulk_commit_group();
        bulk_wait_group_read<0>();   // shared memory read: the CTA may exit
      }
    } else {
      // The two CTAs of a split tile: each stages its FP32 partial O' and O
      // rows in shared memory (the free V^, Q, K stages: eight 128-row x
      // 32-column blocks, 128-byte swizzled) and stores them to its slot with
      // TMA; the one that counts second loads the other's slot back with TMA,
      // adds its own partial and stores the BF16 sums as the whole tiles do.
      uint32_t v[2][32];
#pragma unroll
      for (int o = 0; o < 2; ++o) {
        if (have) {
          tmem_ld32(tmem + lane_off + (o == 0 ? L::kColOP : L::kColO) + part * 32, v[o]);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) v[o][k] = 0u;   // no key tiles: adds nothing
        }
        const uint32_t blk = sbase + (o * 4 + part) * L::kSplitBlock;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          st_shared_v4(sw128_chunk(blk, r, j), v[o][4 * j], v[o][4 * j + 1], v[o][4 * j + 2], v[o][4 * j + 3]);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, kSoftWarpsV * 32);
      const int row0 = (sidx * 2 + rank) * 2 * 128, orow0 = (sidx * 2 + (rank ^ 1)) * 2 * 128;
      if (warp == 0 && lane == 0) {
#pragma unroll
        for (int o = 0; o < 2; ++o)
#pragma unroll
          for (int pp = 0; pp < 4; ++pp)
            tma_store_3d(&tm_slot, smem + (o * 4 + pp) * L::kSplitBlock, 32 * pp, row0 + o * 128, 0);
        bulk_commit_group();
        bulk_wait_group<0>();        // this CTA's rows are written (and its staging read)
        fence_proxy_async_all();
        __threadfence();
        B.split_order = ATTNQAT_IN_BOUNDS(sidx < a.n_split) ? atomicAdd(a.split_cnt + sidx, 1u) : 0u;
        if (B.split_order == 1u) {   // the other CTA's rows are written too
          __threadfence();
          fence_proxy_async_all();
          mbar_arrive_expect_tx(&B.split_in, 8 * L::kSplitBlock);
#pragma unroll
          for (int o = 0; o < 2; ++o)
#pragma unroll
            for (int pp = 0; pp < 4; ++pp)
              tma_load_3d(smem + (o * 4 + pp) * L::kSplitBlock, &tm_slot, &B.split_in, 32 * pp, orow0 + o * 128, 0);
        }
      }
      named_bar_sync(1, kSoftWarpsV * 32);
      if (*reinterpret_cast<volatile uint32_t*>(&B.split_order) == 1u) {
        const bool in = warp_wait(&B.split_in, 0, ctl);
#pragma unroll
        for (int o = 0; o < 2; ++o) {
          const uint32_t blk = (o * 4 + part) * L::kSplitBlock;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 x = *reinterpret_cast<const float4*>(smem + (sw128_chunk(sbase + blk, r, j) - sbase));
            v[o][4 * j] = __float_as_uint(__uint_as_float(v[o][4 * j]) + x.x);
            v[o][4 * j + 1] = __float_as_uint(__uint_as_float(v[o][4 * j + 1]) + x.y);
            v[o][4 * j + 2] = __float_as_uint(__uint_as_float(v[o][4 * j + 2]) + x.z);
            v[o][4 * j + 3] = __float_as_uint(__uint_as_float(v[o][4 * j + 3]) + x.w);
          }
        }
        named_bar_sync(1, kSoftWarpsV * 32);   // every thread has read the FP32 blocks
#pragma unroll
        for (int o = 0; o < 2; ++o) {
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(__uint_as_float(v[o][2 * k]), __uint_as_float(v[o][2 * k + 1]));
          const uint32_t col = part * 32;
          const uint32_t blk = sbase + L::kV0 + o * 2 * L::kOutBlock + (col / 64) * L::kOutBlock;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            st_shared_v4(sw128_chunk(blk, r, (col % 64) / 8 + j), w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, kSoftWarpsV * 32);
        if (in && warp == 0 && lane == 0) {
#pragma unroll
          for (int o = 0; o < 2; ++o)
#pragma unroll
            for (int h = 0; h < 2; ++h)
              tma_store_3d(o == 0 ? &tm_ohp : &tm_o, smem + L::kV0 + (2 * o + h) * L::kOutBlock, 64 * h, i * 128, bh);
          bulk_commit_group();
          bulk_wait_group_read<0>();
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaOP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_fwd_pv(const Problem& p, const bf16* vh, const uint8_t* q4, const uint8_t* qsf,
                          const uint8_t* k4, const uint8_t* ksf, const float* lse, bf16* o, bf16* o_hp,
                          float* split_acc, uint32_t* split_cnt, uint32_t* err, cudaStream_t st) {
  if (p.D != 128 || vh == nullptr || q4 == nullptr || qsf == nullptr || k4 == nullptr || ksf == nullptr ||
      lse == nullptr)
    return cudaErrorInvalidValue;
  CUtensorMap tv, tq4, tk4;
  const uint64_t bh = p.bh();
  CUtensorMap tohp, to;
  if (!make_tile_map(&tv, vh, false, 128, p.Sk, bh, 64, kKeysV) || !make_fp4_map(&tq4, q4, p.Sq, bh, 128) ||
      !make_fp4_map(&tk4, k4, p.Sk, bh, kKeysV) || !make_tile_map(&tohp, o_hp, false, 128, p.Sq, bh, 64, 128) ||
      !make_tile_map(&to, o, false, 128, p.Sq, bh, 64, 128))
    return cudaErrorInvalidValue;
  PvArgs a;
  a.q_sf = qsf, a.k_sf = ksf, a.lse = lse;
  a.o = o, a.o_hp = o_hp;
  a.Sq = static_cast<int>(p.Sq), a.Sk = static_cast<int>(p.Sk);
  a.n_qtiles = static_cast<int>((p.Sq + 127) / 128);
  a.n_ktiles = static_cast<int>((p.Sk + kKeysV - 1) / kKeysV);
  a.causal = p.causal ? 1 : 0;
  a.c2 = p.scale * kLog2e;
  a.err = err, a.timeout_ns = wait_timeout_ns();
  const SplitPlan plan = fwd_pv_split_plan(p, device_sm_count());
  a.n_full = static_cast<int>(plan.n_full);
  a.split_acc = split_acc, a.split_cnt = split_cnt;
  ATTNQAT_CHECKED_ONLY(a.rows_q = static_cast<int64_t>(p.bh()) * p.Sq; a.rows_k = static_cast<int64_t>(p.bh()) * p.Sk;
                       a.n_split = plan.n_split;)
  const int64_t blocks = plan.n_full + 2 * plan.n_split;
  if (blocks > 0x7fffffff || (plan.n_split > 0 && (split_acc == nullptr || split_cnt == nullptr)))
    return cudaErrorInvalidValue;
  // the split slots as one FP32 matrix of [slot][rank][O', O] 128-row blocks,
  // 128 columns, read and written in 32-column boxes
  CUtensorMap tslot = tv;   // not read without split tiles
  if (plan.n_split > 0 && !make_tile_map(&tslot, split_acc, true, 128, static_cast<uint64_t>(plan.n_split) * 4 * 128, 1,
                                         32, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem(reinterpret_cast<const void*>(&fwd_pv_kernel), PvLayout::kAlloc);
  if (e != cudaSuccess) return e;
  return launch_dependent(fwd_pv_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kThreadsV), PvLayout::kAlloc, st,
                          tv, tq4, tk4, tohp, to, tslot, a);
}

// The query tiles of a partial last wave (or, when every tile's two halves fit
// one wave, all of them) get two CTAs each, as in the backward: the key loop
// of a non-causal tile splits evenly, and two halves of a tile take about 0.6
// of a whole tile's time.
SplitPlan fwd_pv_split_plan(const Problem& p, int sms) {
  const int64_t nk = (p.Sk + kKeysV - 1) / kKeysV;
  const int64_t tiles = ((p.Sq + 127) / 128) * p.bh();
  int64_t s = 0;
  if (nk >= 2 && sms > 0) {
    if (2 * tiles <= sms) {
      s = tiles;
    } else if (!p.causal) {
      const int64_t r = tiles % sms;
      s = 2 * r <= sms ? r : 0;
    }
  }
  if (s > kMaxSplitTiles) s = 0;
  return SplitPlan{tiles - s, s};
}

// the debug build's count of skipped accesses in this file's kernels
ATTNQAT_OOB_READER(oob_read_fwd_pv)

}  // namespace attnqat
