// Attn-QAT forward main kernel (sm_103a): O, O' and LSE.
//
// "Attn-QAT: 4-Bit Attention With Quantization-Aware Training" (Method, Fix 1)
// and "NVFP4 Attention QAT Backward" (cuDNN frontend docs, Overview):
//   P   = softmax(scale * Q^ K^T)  (FP32)
//   O'  = P V^                     (auxiliary high-precision output, BF16)
//   O   = fake_nvfp4(P) V^         (groups of 16 keys of the normalised P)
//   LSE = natural-log log-sum-exp of the scaled logits (FP32)
//
// fake_nvfp4 is applied to the normalised probabilities, and fake(c x) differs
// from c fake(x) unless c is a power of two, so P^ needs the final LSE. The
// kernel therefore makes two passes over the key tiles of its 128-row query
// tile: pass 1 computes S and the row max/sum (LSE); pass 2 recomputes S,
// forms the final P and P^, and accumulates O' and O in TMEM with no
// rescaling.
//
// TMEM columns: S double-buffered [0,128) and [128,256); O' [256,256+D);
// O [256+D,256+2D). In pass 2 the softmax warps write P and P^ (BF16 pairs)
// back over the S tile they read: the warps of key part p (keys 32p..32p+31)
// put P in columns 32p + [0,16) and P^ in 32p + [16,32) of that S buffer,
// columns only they read, and the O' and O MMAs take their A operand from
// TMEM there. The next S goes into a buffer once the O' and O MMAs reading
// its P and P^ have completed (their commits). Warp roles (20 warps): 0-15
// softmax (warp w: lanes 32*(w%4).., key columns [32*(w/4), +32)); 16 TMA
// producer; 17, 18, 19 MMA issuers of O', O and S, one per SM sub-partition
// 1-3 (an issuing thread slows the softmax warps of its own sub-partition).
// K^ and V^ tiles are triple-buffered in shared memory.
//
// D = 128: both passes compute S on the block-scaled NVFP4 tensor-core MMA
// (2 MMAs of K = 64 per tile instead of 8 BF16 ones) from the NVFP4 encoding
// of Q and K, whose values are exactly Q^ and K^. The MMA's scale factors sit
// in TMEM. For pass 1 and the first two pass-2 tiles they are in the O'
// columns, which hold no accumulator yet: Q at O' + [0,8), K of tile t at
// O' + 16 + 16 (t % 2) + [0,8). For a later pass-2 tile t + 1 they are in
// columns 64h + [56,64) of S(t)'s buffer (K step h), written by the softmax
// warps of key part 2h + 1 as soon as they have read S(t). The P^ of each key
// half's last 16 keys, whose columns those are, goes through shared memory
// instead.
// Shared memory: V^ x3 96K, NVFP4 Q 8K, NVFP4 K x3 24K, last-16-key P^ x2.
// D = 64: S on BF16 MMAs from Q^, K^ in both passes. Shared memory: V^ x3,
// Q^, K^ x3.
#include "attn_common.cuh"
#include "fp4_mma.cuh"

namespace attnqat {
namespace {

constexpr int kSoftWarpsF = 16;                 // 4 per lane quarter, 32 keys of a tile each
constexpr int kThreadsFwd = (kSoftWarpsF + 4) * 32;
constexpr int kWarpTmaF = kSoftWarpsF;       // SM sub-partition 0
// The MMAs are issued from three warps on sub-partitions 1, 2 and 3: a thread
// issuing tcgen05.mma slows the softmax warps that share its sub-partition,
// so the issue work is spread out.
constexpr int kWarpMmaF = kSoftWarpsF + 1;   // O' += P V^ (and TMEM allocation)
constexpr int kWarpMmaO = kSoftWarpsF + 2;   // O += P^ V^
constexpr int kWarpMmaS = kSoftWarpsF + 3;   // S

template <int D>
struct FwdLayout {
  static constexpr bool kFp4 = D == 128;                 // S on the block-scaled NVFP4 MMA
  static constexpr uint32_t kTile = 128 * D * 2;
  static constexpr uint32_t kFp4Tile = 128 * 64;         // 128 rows x 64 bytes of E2M1 pairs
  static constexpr int kStages = 3;                     // K and V tiles in flight
  static constexpr uint32_t kV0 = 0;                     // V^ stage s at kV0 + s * kTile
  // D = 64: BF16 Q^, K^ (stage s at kK0 + s * kTile)
  static constexpr uint32_t kQ = kV0 + kStages * kTile;
  static constexpr uint32_t kK0 = kQ + kTile;
  // D = 128: NVFP4 Q, K (stage s at kK40 + s * kFp4Tile)
  static constexpr uint32_t kQ4 = kV0 + kStages * kTile;
  static constexpr uint32_t kK40 = kQ4 + kFp4Tile;
  // D = 128: P^ of each key half's last 16 keys, per pass-2 tile parity: two
  // 64-key K-major blocks (128-byte swizzle) of which only bytes 96..127 of
  // each row are written and read
  static constexpr uint32_t kPL0 = kK40 + kStages * kFp4Tile;
  // 128 rows x (m, l) of key parts 1..3, then 128 lse2
  static constexpr uint32_t kML = kFp4 ? kPL0 + 2 * 2 * kBlockBytes : kK0 + kStages * kTile;
  static constexpr uint32_t kBar = kML + 3 * 128 * 8 + 128 * 4;
  static constexpr uint32_t kBytes = kBar + 256;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static constexpr uint32_t kColS0 = 0;
  static constexpr uint32_t kColOP = 256;
  static constexpr uint32_t kColO = 256 + D;
  static constexpr uint32_t kColSFQ = kColOP;            // pass 1 and pass-2 tiles 0, 1
  static constexpr uint32_t kColSFK0 = kColOP + 16;
  static constexpr uint32_t kColSFK1 = kColOP + 32;
  // later pass-2 tiles: + 128 * buffer + 64 * ks, over the P^ columns of the
  // key half's last 16 keys (read by the last O MMA of that half)
  static constexpr uint32_t kColSFQ2 = 56;
  static constexpr uint32_t kColSFK2 = 60;
  static_assert(!kFp4 || kPL0 % 1024 == 0, "P^ blocks need 1024-byte alignment for the 128-byte swizzle");
  static_assert(kColSFQ2 % 4 == 0 && kColSFK2 == kColSFQ2 + 4 && kColSFK2 + 4 == 64,
                "pass-2 scale factors: 4-column aligned, over the last 8 P^ columns of a key half");
};

struct FwdBars {
  uint64_t q_full;
  uint64_t k_full[3];    // per K / V stage
  uint64_t k_empty[3];
  uint64_t v_full[3];
  uint64_t v_empty[3];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_ready[2];   // per S buffer: P and P^ of a pass-2 tile are in place
  uint64_t pv_read[2];   // per S buffer: the O' and O MMAs of a pass-2 tile are done with it
  uint64_t o_done;       // one phase: every O' and O MMA has completed
  uint64_t ml_ready;
  uint64_t lse_ready;
  uint64_t drain;
  uint64_t sf_init;      // pass 1: Q scales and tile 0 and 1 K scales are in TMEM
  uint32_t tmem_base;
  uint32_t abort_flag;
};

struct FwdArgs {
  const uint8_t* q_sf;   // NVFP4 scales of Q, K ((B*H, S, D/16) E4M3), D = 128
  const uint8_t* k_sf;
  bf16* o;
  bf16* o_hp;
  float* lse;
  const float* lse_in;   // not null: pass 1 is skipped, this is the LSE (natural log)
  int Sq, Sk;
  int n_qtiles, n_ktiles;
  int causal;
  float c2;   // scale * log2(e)
  uint32_t* err;
  uint64_t timeout_ns;
};

template <int D>
__global__ void __launch_bounds__(kThreadsFwd, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q4,
               const __grid_constant__ CUtensorMap tm_k4, const FwdArgs a) {
  using L = FwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  FwdBars& B = *reinterpret_cast<FwdBars*>(smem + L::kBar);
  float* ml = reinterpret_cast<float*>(smem + L::kML);

  const int warp = warp_id();
  const int lane = lane_id();
  // Causal tiles have i + 1 key tiles: launch the longest first.
  const int i = a.causal ? (a.n_qtiles - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
  const int bh = blockIdx.y;
  const int nk = a.causal ? i + 1 : a.n_ktiles;
  // Tiles t of the sequence: pass 1 (t < P1, key tile t), then pass 2 (key
  // tile t - P1). With lse_in given (D = 128: the paired LSE kernel has
  // computed the LSE), only pass 2 runs.
  const int P1 = a.lse_in != nullptr ? 0 : nk;
  const int nt = P1 + nk;

  if (threadIdx.x == 0) {
    B.abort_flag = 0;
    mbar_init(&B.q_full, 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&B.k_full[s], 1), mbar_init(&B.k_empty[s], 1);
      mbar_init(&B.v_full[s], 1), mbar_init(&B.v_empty[s], 2);   // read by the O' and the O MMAs
    }
    for (int s = 0; s < 2; ++s) mbar_init(&B.s_full[s], 1), mbar_init(&B.s_free[s], kSoftWarpsF * 32);
    mbar_init(&B.p_ready[0], kSoftWarpsF * 32);
    mbar_init(&B.p_ready[1], kSoftWarpsF * 32);
    mbar_init(&B.pv_read[0], 2), mbar_init(&B.pv_read[1], 2);   // one commit each from the O' and O issuers
    mbar_init(&B.o_done, 2);
    mbar_init(&B.ml_ready, 3 * 128);   // key parts 1..3
    mbar_init(&B.lse_ready, 128);      // key part 0
    mbar_init(&B.drain, 3);            // one commit per MMA-issuing thread
    mbar_init(&B.sf_init, 2 * 128);    // key parts 1 and 3
    fence_mbar_init();
  }
  if (warp == kWarpMmaF) {
    tmem_alloc(&B.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B.tmem_base;
  const WaitCtl ctl{&B.abort_flag, a.err, a.timeout_ns};

  if (warp == kWarpTmaF) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q), tma_prefetch_desc(&tm_k), tma_prefetch_desc(&tm_v);
      if (L::kFp4) tma_prefetch_desc(&tm_q4), tma_prefetch_desc(&tm_k4);
      int k_uses[L::kStages] = {}, v_uses[L::kStages] = {};
      if constexpr (L::kFp4) {                          // NVFP4 Q only
        mbar_arrive_expect_tx(&B.q_full, L::kFp4Tile);
        tma_load_3d(smem + L::kQ4, &tm_q4, &B.q_full, 0, i * 128, bh);
      } else {
        mbar_arrive_expect_tx(&B.q_full, L::kTile);
        for (int b = 0; b < D / 64; ++b)
          tma_load_3d(smem + L::kQ + b * kBlockBytes, &tm_q, &B.q_full, b * 64, i * 128, bh);
      }
      for (int t = 0; t < nt; ++t) {
        const int jt = t < P1 ? t : t - P1;
        const int s = t % L::kStages, use = t / L::kStages;
        if (use >= 1 && !mbar_wait(&B.k_empty[s], (use - 1) & 1, ctl)) break;
        if constexpr (L::kFp4) {                           // NVFP4 K in both passes
          mbar_arrive_expect_tx(&B.k_full[s], L::kFp4Tile);
          tma_load_3d(smem + L::kK40 + s * L::kFp4Tile, &tm_k4, &B.k_full[s], 0, jt * 128, bh);
        } else {
          mbar_arrive_expect_tx(&B.k_full[s], L::kTile);
          for (int b = 0; b < D / 64; ++b)
            tma_load_3d(smem + L::kK0 + s * L::kTile + b * kBlockBytes, &tm_k, &B.k_full[s], b * 64, jt * 128, bh);
        }
        ++k_uses[s];
        if (t >= P1) {
          const int tv = t - P1, sv = tv % L::kStages, vuse = tv / L::kStages;
          if (vuse >= 1 && !mbar_wait(&B.v_empty[sv], (vuse - 1) & 1, ctl)) break;
          mbar_arrive_expect_tx(&B.v_full[sv], L::kTile);
          for (int b = 0; b < D / 64; ++b)
            tma_load_3d(smem + L::kV0 + sv * L::kTile + b * kBlockBytes, &tm_v, &B.v_full[sv], b * 64, jt * 128, bh);
          ++v_uses[sv];
        }
      }
      mbar_wait_drain(&B.q_full, 0, ctl);
      for (int s = 0; s < L::kStages; ++s) {
        if (k_uses[s]) mbar_wait_drain(&B.k_full[s], (k_uses[s] - 1) & 1, ctl);
        if (v_uses[s]) mbar_wait_drain(&B.v_full[s], (v_uses[s] - 1) & 1, ctl);
      }
    }
  } else if (warp == kWarpMmaF || warp == kWarpMmaO || warp == kWarpMmaS) {
    // ------------------------------------------------------------ MMA issuers
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdO = idesc_bf16(128, D, false, true);
      // Descriptors built once, advanced by constants per k-step (few issue
      // instructions per MMA for a thread that shares its sub-partition).
      const uint64_t kmaj = sdesc_sw128(sbase, 16, 1024);
      const uint64_t mnmaj = sdesc_sw128(sbase, kBlockBytes, 1024);
      // use index of pass-2 tile t's S buffer among pass-2 tiles (one barrier
      // per buffer, so the softmax warps running ahead cannot alias phases)
      auto pr_use = [&](int t) { return (t >> 1) - ((P1 + 1 - (t & 1)) >> 1); };
      bool ok = true;
      if (warp == kWarpMmaS) {
        auto issue_s = [&](int t) -> bool {
          const int s = t & 1, ks_ = t % L::kStages;
          // The buffer's previous tile u = t - 2 must be done with: a pass-1 S
          // once the softmax warps have read it, a pass-2 buffer (P(u), P^(u))
          // once the O' and O MMAs of tile u have completed.
          const int u = t - 2;
          // D = 128, pass-2 tiles from the third on: the scale factors are in the
          // previous tile's S buffer, written there once the softmax warps have
          // read that S (they arrive on its s_free in both passes).
          const bool sf_in_s = L::kFp4 && t >= P1 + 2;
          const bool prev_s = u >= 0 && u < P1;   // exclusive with sf_in_s
          uint64_t* sbar = prev_s ? &B.s_free[s] : (sf_in_s ? &B.s_free[(t - 1) & 1] : nullptr);
          const uint32_t spar = prev_s ? ((u >> 1) & 1) : (((t - 1) >> 1) & 1);
          const bool pv_wait = u >= P1;
          const bool kf = mbar_try_wait(&B.k_full[ks_], (t / L::kStages) & 1);
          if (!mbar_wait_both(sbar, spar, pv_wait ? &B.pv_read[s] : nullptr, pv_wait ? (pr_use(u) & 1) : 0u, ctl))
            return false;
          if (!kf && !mbar_wait(&B.k_full[ks_], (t / L::kStages) & 1, ctl)) return false;
          tc_fence_after();
          if constexpr (L::kFp4) {
            const uint64_t d4q = sdesc_sw64(sbase + L::kQ4), d4k = sdesc_sw64(sbase + L::kK40 + ks_ * L::kFp4Tile);
            const uint32_t sfq = sf_in_s ? L::kColS0 + ((t - 1) & 1) * 128 + L::kColSFQ2 : L::kColSFQ;
            const uint32_t sfk = sf_in_s ? L::kColS0 + ((t - 1) & 1) * 128 + L::kColSFK2 : (s ? L::kColSFK1 : L::kColSFK0);
            const uint32_t step = sf_in_s ? 64u : 4u;      // column distance between the K = 64 steps' factors
#pragma unroll
            for (int ks = 0; ks < 2; ++ks)
              umma_nvfp4(tmem + L::kColS0 + s * 128, sdesc_advance(d4q, ks * 32), sdesc_advance(d4k, ks * 32),
                         idesc_nvfp4(128, 128), tmem + sfq + ks * step, tmem + sfk + ks * step, ks > 0);
          } else {
            const uint64_t dq = sdesc_advance(kmaj, L::kQ);
            const uint64_t db = sdesc_advance(kmaj, L::kK0 + ks_ * L::kTile);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t o = (kk >> 2) * kBlockBytes + (kk & 3) * 32;
              umma_bf16(tmem + L::kColS0 + s * 128, sdesc_advance(dq, o), sdesc_advance(db, o), kIdS, kk > 0);
            }
          }
          umma_commit(&B.s_full[s]);
          umma_commit(&B.k_empty[ks_]);
          return true;
        };
        ok = mbar_wait(&B.q_full, 0, ctl) && (!L::kFp4 || mbar_wait(&B.sf_init, 0, ctl));
        for (int t = 0; ok && t < nt; ++t) ok = issue_s(t);
      } else {
        // O' += P V^ (warp kWarpMmaF) or O += P^ V^ (warp kWarpMmaO) for every
        // pass-2 tile, A from TMEM at the tile's S buffer (keys 32p .. 32p + 31
        // in columns 32p + [0,16) for P and 32p + [16,32) for P^), V^ MN-major
        // in shared memory. D = 128: the P^ of each key half's last 16 keys
        // comes from shared memory (its TMEM columns hold the next S's scale
        // factors).
        const bool is_op = warp == kWarpMmaF;
        // The scale factors of pass 1 and of pass-2 tiles 0, 1 sit in the O'
        // columns: the first O' MMA waits until S of those tiles has completed.
        if (is_op && L::kFp4 && P1 < nt) {
          const int t0 = P1, t1 = P1 + 1;
          ok = mbar_wait_both(&B.s_full[t0 & 1], (t0 >> 1) & 1, t1 < nt ? &B.s_full[t1 & 1] : nullptr,
                              (t1 >> 1) & 1, ctl);
        }
        for (int t = P1; ok && t < nt; ++t) {
          const int tv = t - P1, sv = tv % L::kStages;
          if (!mbar_wait_both(&B.v_full[sv], (tv / L::kStages) & 1, &B.p_ready[t & 1], pr_use(t) & 1, ctl)) break;
          tc_fence_after();
          const uint64_t dv = sdesc_advance(mnmaj, L::kV0 + sv * L::kTile);
          const uint32_t sc = L::kColS0 + (t & 1) * 128;
          if (is_op) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t ac = sc + (kk >> 1) * 32 + (kk & 1) * 8;
              umma_bf16_tmem_a(tmem + L::kColOP, tmem + ac, sdesc_advance(dv, kk * 2048), kIdO,
                               (tv > 0 || kk > 0) ? 1u : 0u);
            }
          } else {
            const uint64_t dl = sdesc_advance(kmaj, L::kPL0 + (tv & 1) * 2 * kBlockBytes);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t acc = (tv > 0 || kk > 0) ? 1u : 0u;
              if (L::kFp4 && (kk & 3) == 3) {
                umma_bf16(tmem + L::kColO, sdesc_advance(dl, (kk >> 2) * kBlockBytes + 3 * 32),
                          sdesc_advance(dv, kk * 2048), kIdO, acc);
              } else {
                const uint32_t ac = sc + 16 + (kk >> 1) * 32 + (kk & 1) * 8;
                umma_bf16_tmem_a(tmem + L::kColO, tmem + ac, sdesc_advance(dv, kk * 2048), kIdO, acc);
              }
            }
          }
          umma_commit(&B.v_empty[sv]);
          umma_commit(&B.pv_read[t & 1]);
          if (tv == nk - 1) umma_commit(&B.o_done);
        }
      }
      umma_commit(&B.drain);
      mbar_wait_drain(&B.drain, 0, ctl);
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 0-15)
    // Warp w owns lane quarter w % 4 (32 query rows) and key part w / 4 (keys
    // 32 p .. 32 p + 31 of every tile, S columns [32 p, 32 p + 32)). In pass 2
    // it writes P over columns 32 p + [0,16) and P^ over 32 p + [16,32). Parts
    // 1 and 3 also write the scale factors (K step p / 2); in pass 2 those go
    // over their P^ columns 32 p + [24,32), whose P^ goes to shared memory.
    const uint32_t quarter = warp & 3, part = warp >> 2;
    const bool sf_writer = (part & 1u) != 0;
    const int ks = static_cast<int>(part >> 1);
    const uint32_t r = quarter * 32 + lane;
    const uint32_t lane_off = (quarter * 32u) << 16;
    const int qrow = i * 128 + r;
    const int kend = a.causal ? min(a.Sk, qrow + 1) : a.Sk;
    const int64_t kbase = static_cast<int64_t>(bh) * a.Sk;
    bool ok = true;
    if (L::kFp4 && sf_writer) {   // pass-1 scale factors of K step ks
      uint32_t w[4];
      load_scales(a.q_sf, static_cast<int64_t>(bh) * a.Sq + i * 128, min(128, a.Sq - i * 128), ks, w);
      tmem_st4(tmem + lane_off + L::kColSFQ + 4 * ks, w);
      load_scales(a.k_sf, kbase, min(128, a.Sk), ks, w);
      tmem_st4(tmem + lane_off + L::kColSFK0 + 4 * ks, w);
      const int kt1 = nk > 1 ? 1 : 0;   // tile 1 is pass 2's first when nk = 1
      load_scales(a.k_sf, kbase + kt1 * 128, min(128, a.Sk - kt1 * 128), ks, w);
      tmem_st4(tmem + lane_off + L::kColSFK1 + 4 * ks, w);
      tc_fence_before();
      mbar_arrive(&B.sf_init);
    }

    // pass 1: running max and sum of exp2(S * c2) over this thread's 32 key columns
    const float2 c22 = make_float2(a.c2, a.c2);
    float m = -INFINITY, l = 0.0f;
    // K scales written at tile t (those of tile t + 2, up to pass 2's second
    // tile) are loaded one tile ahead, so their latency is off the hand-off
    auto kt_of = [&](int u) { return u < P1 ? u : u - P1; };
    uint32_t sfw[4] = {0u, 0u, 0u, 0u}, sfw_next[4] = {0u, 0u, 0u, 0u};
    if (L::kFp4 && sf_writer && 2 < nt)
      load_scales(a.k_sf, kbase + kt_of(2) * 128, min(128, a.Sk - kt_of(2) * 128), ks, sfw);
    for (int t = 0; t < P1; ++t) {
      const int s = t & 1;
      const int valid = kend - (t * 128 + static_cast<int>(part) * 32);
      // K scales of tile t + 2 (up to pass 2's second tile, key tile 1)
      const bool more = L::kFp4 && sf_writer && t + 2 < nt;
      if (L::kFp4 && sf_writer && t + 3 < nt && t + 1 < P1)
        load_scales(a.k_sf, kbase + kt_of(t + 3) * 128, min(128, a.Sk - kt_of(t + 3) * 128), ks, sfw_next);
      if (!warp_wait(&B.s_full[s], (t >> 1) & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32(tmem + lane_off + L::kColS0 + s * 128 + part * 32, v);
      // tile t + 2's K scales into the slot S(t) used (S(t) is complete);
      // releasing S(t) below also certifies them to the S issuer
      if (more) tmem_st4(tmem + lane_off + (s ? L::kColSFK1 : L::kColSFK0) + 4 * ks, sfw);
      tc_fence_before();
      mbar_arrive(&B.s_free[s]);
#pragma unroll
      for (int q = 0; q < 4; ++q) sfw[q] = sfw_next[q];
      if (valid < 32) {   // masked keys: -inf
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (k >= valid) v[k] = 0xFF800000u;
      }
      // Row max of the raw S (two chains of 3-input max); c2 > 0 and rounding
      // is monotonic, so max(S) * c2 is the max of the scaled logits.
      float mq[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        float acc = fmaxf(__uint_as_float(v[16 * u]), __uint_as_float(v[16 * u + 1]));
#pragma unroll
        for (int k = 2; k < 16; k += 2) acc = fmax3(acc, __uint_as_float(v[16 * u + k]), __uint_as_float(v[16 * u + k + 1]));
        mq[u] = acc;
      }
      const float mx = fmaxf(m, fmaxf(mq[0], mq[1]) * a.c2);
      if (mx == -INFINITY) continue;
      // sum of exp2(S * c2 - mx), arguments and partial sums as packed pairs
      const float2 nm = make_float2(-mx, -mx);
      float2 sc[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                      make_float2(0.0f, 0.0f)};
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float2 e = ffma2(make_float2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1])), c22, nm);
        sc[k & 3] = fadd2(sc[k & 3], make_float2(ex2(e.x), ex2(e.y)));
      }
      const float2 st = fadd2(fadd2(sc[0], sc[1]), fadd2(sc[2], sc[3]));
      l = l * ex2(m - mx) + (st.x + st.y);
      m = mx;
    }
    // Combine the four key parts of each row: parts 1..3 hand (m, l) to part
    // 0, which forms lse2 = log2 sum 2^(S*c2), stores LSE and hands lse2 back.
    float lse2 = 0.0f;
    float* lse_s = ml + 3 * 256;
    if (P1 == 0) {   // pass 2 only: the LSE of this row from lse_in
      if (qrow < a.Sq) lse2 = __ldg(a.lse_in + (size_t)bh * a.Sq + qrow) * kLog2e;
    } else if (ok && part != 0) {
      ml[(part - 1) * 256 + r * 2] = m;
      ml[(part - 1) * 256 + r * 2 + 1] = l;
      mbar_arrive(&B.ml_ready);
      if (warp_wait(&B.lse_ready, 0, ctl))
        lse2 = lse_s[r];
      else
        ok = false;
    } else if (ok) {
      if (warp_wait(&B.ml_ready, 0, ctl)) {
        float mp[4] = {m, ml[r * 2], ml[256 + r * 2], ml[512 + r * 2]};
        float lp[4] = {l, ml[r * 2 + 1], ml[256 + r * 2 + 1], ml[512 + r * 2 + 1]};
        const float M = fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3]));
        float Lsum = 0.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) Lsum += mp[q] == -INFINITY ? 0.0f : lp[q] * ex2(mp[q] - M);
        lse2 = M + lg2(Lsum);
        lse_s[r] = lse2;
        mbar_arrive(&B.lse_ready);
        if (qrow < a.Sq) a.lse[(size_t)bh * a.Sq + qrow] = lse2 * kLn2;
      } else {
        ok = false;
      }
    }

    // pass 2: P = exp2(S * c2 - lse2), P^ = fake_nvfp4(P); hand both to the MMA warps
    uint32_t sfq[4] = {0u, 0u, 0u, 0u};   // D = 128: K step ks of the Q scale factors (parts 1, 3)
    if (L::kFp4 && sf_writer)
      load_scales(a.q_sf, static_cast<int64_t>(bh) * a.Sq + i * 128, min(128, a.Sq - i * 128), ks, sfq);
    uint32_t sfk[4] = {0u, 0u, 0u, 0u};
    for (int t = P1; ok && t < nt; ++t) {
      const int s = t & 1, tv = t - P1;
      const int valid = kend - (tv * 128 + static_cast<int>(part) * 32);
      // D = 128: parts 1 and 3 put the scale factors of S(t + 1) (pass-2
      // tiles from the third on; K step ks) into S(t)'s buffer, over the P^
      // columns of the key half's last 16 keys
      const bool wsf = L::kFp4 && sf_writer && tv >= 1 && t + 1 < nt;
      // sfk holds key tile tv + 1's scales (loaded one tile ahead); fetch tv + 2's
      uint32_t sfk_next[4] = {0u, 0u, 0u, 0u};
      if (L::kFp4 && sf_writer && tv + 2 < nk)
        load_scales(a.k_sf, kbase + (tv + 2) * 128, min(128, a.Sk - (tv + 2) * 128), ks, sfk_next);
      if (!warp_wait(&B.s_full[s], (t >> 1) & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      const uint32_t pcol = tmem + lane_off + L::kColS0 + s * 128 + part * 32;   // this warp's S columns
      float P[32];
      {
        uint32_t v[32];
        tmem_ld32(pcol, v);
        if constexpr (L::kFp4) {   // S(t) is read: scale factors of S(t + 1), then release it
          if (wsf) {
            tmem_st4(pcol + 24, sfq);
            tmem_st4(pcol + 28, sfk);
          }
          tc_fence_before();
          mbar_arrive(&B.s_free[s]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) sfk[q] = sfk_next[q];
        const float2 nl = make_float2(-lse2, -lse2);
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          const float2 e = ffma2(make_float2(__uint_as_float(v[k]), __uint_as_float(v[k + 1])), c22, nl);
          P[k] = ex2(e.x), P[k + 1] = ex2(e.y);
        }
      }
      if (valid < 32) {   // masked keys: P = 0
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (k >= valid) P[k] = 0.0f;
      }
      uint32_t pw[16], phw[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) pw[k] = pack_bf16x2(P[2 * k], P[2 * k + 1]);
#pragma unroll
      for (int g = 0; g < 2; ++g) fake_nvfp4_16_pack_nonneg<false>(P + 16 * g, 1.0f, phw + 8 * g);
      // P over columns [0,16) of this warp's S columns, P^ over [16,32). D = 128:
      // parts 1 and 3 send the P^ of the key half's last 16 keys to shared
      // memory instead (bytes 96..127 of the row of the half's 64-key block),
      // as its columns may hold the scale factors of S(t + 1); the buffer's
      // previous tile, t - 2, is complete since S(t) is.
      tmem_st16_nowait(pcol, pw);
      if (L::kFp4 && sf_writer) {
        tmem_st8_nowait(pcol + 16, phw);
        const uint32_t blk = sbase + L::kPL0 + (tv & 1) * 2 * kBlockBytes + ks * kBlockBytes;
        st_shared_v4(sw128_chunk(blk, r, 6), phw[8], phw[9], phw[10], phw[11]);
        st_shared_v4(sw128_chunk(blk, r, 7), phw[12], phw[13], phw[14], phw[15]);
        fence_proxy_async_smem();
      } else {
        tmem_st16_nowait(pcol + 16, phw);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&B.p_ready[s]);
    }
    // epilogue: O' and O rows (a one-shot barrier committed after the last O'
    // and O MMAs). D = 128: part p stores columns [32 p, 32 p + 32) of both;
    // D = 64: parts 0, 1 store O' columns [32 (p % 2), +32), parts 2, 3 O's.
    if (ok && warp_wait(&B.o_done, 0, ctl)) {
      tc_fence_after();
      const size_t row = (size_t)bh * a.Sq + qrow;
      uint32_t v[32];
      if constexpr (D == 128) {
        const uint32_t col = part * 32;
        tmem_ld32(tmem + lane_off + L::kColOP + col, v);
        if (qrow < a.Sq) store_row32_bf16(a.o_hp + row * D + col, v, 1.0f);
        tmem_ld32(tmem + lane_off + L::kColO + col, v);
        if (qrow < a.Sq) store_row32_bf16(a.o + row * D + col, v, 1.0f);
      } else {
        const uint32_t col = (part & 1) * 32;
        tmem_ld32(tmem + lane_off + (part < 2 ? L::kColOP : L::kColO) + col, v);
        if (qrow < a.Sq) store_row32_bf16((part < 2 ? a.o_hp : a.o) + row * D + col, v, 1.0f);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaF) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_fwd(const Problem& p, const bf16* qh, const bf16* kh, const bf16* vh, const uint8_t* q4,
                       const uint8_t* qsf, const uint8_t* k4, const uint8_t* ksf, bf16* o, bf16* o_hp, float* lse,
                       uint32_t* err, cudaStream_t st) {
  CUtensorMap tq, tk, tv, tq4, tk4;
  const uint64_t bh = p.bh();
  if (!make_tile_map(&tq, qh, false, p.D, p.Sq, bh, 64, 128) || !make_tile_map(&tk, kh, false, p.D, p.Sk, bh, 64, 128) ||
      !make_tile_map(&tv, vh, false, p.D, p.Sk, bh, 64, 128))
    return cudaErrorInvalidValue;
  const bool fp4 = p.D == 128;
  if (fp4 && (q4 == nullptr || qsf == nullptr || k4 == nullptr || ksf == nullptr)) return cudaErrorInvalidValue;
  if (fp4) {
    if (!make_fp4_map(&tq4, q4, p.Sq, bh, 128) || !make_fp4_map(&tk4, k4, p.Sk, bh, 128)) return cudaErrorInvalidValue;
  } else {
    tq4 = tq, tk4 = tk;   // not read at D = 64
  }
  FwdArgs a;
  a.q_sf = qsf, a.k_sf = ksf;
  a.o = o, a.o_hp = o_hp, a.lse = lse;
  a.Sq = static_cast<int>(p.Sq), a.Sk = static_cast<int>(p.Sk);
  a.n_qtiles = static_cast<int>((p.Sq + kBlockM - 1) / kBlockM);
  a.n_ktiles = static_cast<int>((p.Sk + kBlockN - 1) / kBlockN);
  a.causal = p.causal ? 1 : 0;
  a.c2 = p.scale * kLog2e;
  a.err = err, a.timeout_ns = wait_timeout_ns();
  a.lse_in = nullptr;
  const dim3 grid(static_cast<unsigned>(a.n_qtiles), static_cast<unsigned>(bh));
  if (fp4) {
    // D = 128: pass 1 (the LSE) in the paired kernel of fwd_lse.cu, then pass
    // 2 here reading it
    cudaError_t e = launch_fwd_lse(p, q4, qsf, k4, ksf, lse, err, st);
    if (e != cudaSuccess) return e;
    a.lse_in = lse;
    e = set_smem(reinterpret_cast<const void*>(&fwd_kernel<128>), FwdLayout<128>::kAlloc);
    if (e != cudaSuccess) return e;
    fwd_kernel<128><<<grid, kThreadsFwd, FwdLayout<128>::kAlloc, st>>>(tq, tk, tv, tq4, tk4, a);
  } else {
    cudaError_t e = set_smem(reinterpret_cast<const void*>(&fwd_kernel<64>), FwdLayout<64>::kAlloc);
    if (e != cudaSuccess) return e;
    fwd_kernel<64><<<grid, kThreadsFwd, FwdLayout<64>::kAlloc, st>>>(tq, tk, tv, tq4, tk4, a);
  }
  return cudaGetLastError();
}

}  // namespace attnqat
