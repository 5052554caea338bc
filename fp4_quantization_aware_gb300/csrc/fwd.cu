// Attn-QAT forward at D = 64 (sm_103a): O, O' and LSE in one kernel.
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
// rescaling. (At D = 128 the two passes are separate kernels, fwd_lse.cu and
// fwd_pv.cu, with S on the block-scaled NVFP4 MMA.)
//
// S = Q^ K^T on BF16 MMAs from the quantize step's Q^, K^. TMEM columns: S
// double-buffered [0,128) and [128,256); O' [256,320); O [320,384). In pass 2
// the softmax warps write P and P^ (BF16 pairs) back over the S tile they
// read: the warps of key part p (keys 32p..32p+31) put P in columns
// 32p + [0,16) and P^ in 32p + [16,32) of that S buffer, columns only they
// read, and the O' and O MMAs take their A operand from TMEM there. The next S
// goes into a buffer once the O' and O MMAs reading its P and P^ have
// completed (their commits). Warp roles (20 warps): 0-15 softmax (warp w:
// lanes 32*(w%4).., key columns [32*(w/4), +32)); 16 TMA producer; 17, 18, 19
// MMA issuers of O', O and S, one per SM sub-partition 1-3 (an issuing thread
// slows the softmax warps of its own sub-partition).
// Shared memory: V^ x3, Q^, K^ x3.
#include "attn_common.cuh"
#include "checked.cuh"

namespace attnqat {
namespace {

constexpr int kD = 64;
constexpr int kSoftWarpsF = 16;                 // 4 per lane quarter, 32 keys of a tile each
constexpr int kThreadsFwd = (kSoftWarpsF + 4) * 32;
constexpr int kWarpTmaF = kSoftWarpsF;       // SM sub-partition 0
constexpr int kWarpMmaF = kSoftWarpsF + 1;   // O' += P V^ (and TMEM allocation)
constexpr int kWarpMmaO = kSoftWarpsF + 2;   // O += P^ V^
constexpr int kWarpMmaS = kSoftWarpsF + 3;   // S

struct FwdLayout {
  static constexpr uint32_t kTile = 128 * kD * 2;      // one 64-column (128-byte) block of 128 rows
  static constexpr int kStages = 3;                     // K and V tiles in flight
  static constexpr uint32_t kV0 = 0;                     // V^ stage s at kV0 + s * kTile
  static constexpr uint32_t kQ = kV0 + kStages * kTile;
  static constexpr uint32_t kK0 = kQ + kTile;            // K^ stage s at kK0 + s * kTile
  static constexpr uint32_t kML = kK0 + kStages * kTile;   // 128 rows x (m, l) of key parts 1..3, then 128 lse2
  static constexpr uint32_t kBar = kML + 3 * 128 * 8 + 128 * 4;
  static constexpr uint32_t kBytes = kBar + 256;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static constexpr uint32_t kColS0 = 0;
  static constexpr uint32_t kColOP = 256;
  static constexpr uint32_t kColO = 256 + kD;
  static_assert(kTile == kBlockBytes, "D = 64: one 128-byte-swizzled block per tile");
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
  uint32_t tmem_base;
  uint32_t abort_flag;
};

struct FwdArgs {
  bf16* o;
  bf16* o_hp;
  float* lse;
  int Sq, Sk;
  int n_qtiles, n_ktiles;
  int causal;
  float c2;   // scale * log2(e)
  uint32_t* err;
  uint64_t timeout_ns;
  ATTNQAT_CHECKED_ONLY(int64_t rows_q; int64_t rows_k;)   // debug build: B*H*Sq, B*H*Sk
};

__global__ void __launch_bounds__(kThreadsFwd, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  using L = FwdLayout;
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
  // Tiles t of the sequence: pass 1 (t < nk, key tile t), then pass 2 (key
  // tile t - nk).
  const int nt = 2 * nk;

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
      int k_uses[L::kStages] = {}, v_uses[L::kStages] = {};
      mbar_arrive_expect_tx(&B.q_full, L::kTile);
      tma_load_3d(smem + L::kQ, &tm_q, &B.q_full, 0, i * 128, bh);
      for (int t = 0; t < nt; ++t) {
        const int jt = t < nk ? t : t - nk;
        const int s = t % L::kStages, use = t / L::kStages;
        if (use >= 1 && !mbar_wait(&B.k_empty[s], (use - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(&B.k_full[s], L::kTile);
        tma_load_3d(smem + L::kK0 + s * L::kTile, &tm_k, &B.k_full[s], 0, jt * 128, bh);
        ++k_uses[s];
        if (t >= nk) {
          const int tv = t - nk, sv = tv % L::kStages, vuse = tv / L::kStages;
          if (vuse >= 1 && !mbar_wait(&B.v_empty[sv], (vuse - 1) & 1, ctl)) break;
          mbar_arrive_expect_tx(&B.v_full[sv], L::kTile);
          tma_load_3d(smem + L::kV0 + sv * L::kTile, &tm_v, &B.v_full[sv], 0, jt * 128, bh);
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
      constexpr uint32_t kIdO = idesc_bf16(128, kD, false, true);
      // Descriptors built once, advanced by constants per k-step (few issue
      // instructions per MMA for a thread that shares its sub-partition).
      const uint64_t kmaj = sdesc_sw128(sbase, 16, 1024);
      const uint64_t mnmaj = sdesc_sw128(sbase, kBlockBytes, 1024);
      // use index of pass-2 tile t's S buffer among pass-2 tiles (one barrier
      // per buffer, so the softmax warps running ahead cannot alias phases)
      auto pr_use = [&](int t) { return (t >> 1) - ((nk + 1 - (t & 1)) >> 1); };
      bool ok = true;
      if (warp == kWarpMmaS) {
        auto issue_s = [&](int t) -> bool {
          const int s = t & 1, ks_ = t % L::kStages;
          // The buffer's previous tile u = t - 2 must be done with: a pass-1 S
          // once the softmax warps have read it, a pass-2 buffer (P(u), P^(u))
          // once the O' and O MMAs of tile u have completed.
          const int u = t - 2;
          const bool prev_s = u >= 0 && u < nk;
          const bool pv_wait = u >= nk;
          const bool kf = mbar_try_wait(&B.k_full[ks_], (t / L::kStages) & 1);
          if (!mbar_wait_both(prev_s ? &B.s_free[s] : nullptr, (u >> 1) & 1, pv_wait ? &B.pv_read[s] : nullptr,
                              pv_wait ? (pr_use(u) & 1) : 0u, ctl))
            return false;
          if (!kf && !mbar_wait(&B.k_full[ks_], (t / L::kStages) & 1, ctl)) return false;
          tc_fence_after();
          const uint64_t dq = sdesc_advance(kmaj, L::kQ);
          const uint64_t db = sdesc_advance(kmaj, L::kK0 + ks_ * L::kTile);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            umma_bf16(tmem + L::kColS0 + s * 128, sdesc_advance(dq, kk * 32), sdesc_advance(db, kk * 32), kIdS, kk > 0);
          umma_commit(&B.s_full[s]);
          umma_commit(&B.k_empty[ks_]);
          return true;
        };
        ok = mbar_wait(&B.q_full, 0, ctl);
        for (int t = 0; ok && t < nt; ++t) ok = issue_s(t);
      } else {
        // O' += P V^ (warp kWarpMmaF) or O += P^ V^ (warp kWarpMmaO) for every
        // pass-2 tile, A from TMEM at the tile's S buffer (keys 32p .. 32p + 31
        // in columns 32p + [0,16) for P and 32p + [16,32) for P^), V^ MN-major
        // in shared memory.
        const bool is_op = warp == kWarpMmaF;
        const uint32_t acc_col = is_op ? L::kColOP : L::kColO;
        const uint32_t a_off = is_op ? 0u : 16u;
        for (int t = nk; ok && t < nt; ++t) {
          const int tv = t - nk, sv = tv % L::kStages;
          if (!mbar_wait_both(&B.v_full[sv], (tv / L::kStages) & 1, &B.p_ready[t & 1], pr_use(t) & 1, ctl)) break;
          tc_fence_after();
          const uint64_t dv = sdesc_advance(mnmaj, L::kV0 + sv * L::kTile);
          const uint32_t sc = L::kColS0 + (t & 1) * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ac = sc + a_off + (kk >> 1) * 32 + (kk & 1) * 8;
            umma_bf16_tmem_a(tmem + acc_col, tmem + ac, sdesc_advance(dv, kk * 2048), kIdO,
                             (tv > 0 || kk > 0) ? 1u : 0u);
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
    // it writes P over columns 32 p + [0,16) and P^ over 32 p + [16,32).
    const uint32_t quarter = warp & 3, part = warp >> 2;
    const uint32_t r = quarter * 32 + lane;
    const uint32_t lane_off = (quarter * 32u) << 16;
    const int qrow = i * 128 + r;
    const int kend = a.causal ? min(a.Sk, qrow + 1) : a.Sk;
    bool ok = true;

    // pass 1: running max and sum of exp2(S * c2) over this thread's 32 key columns
    const float2 c22 = make_float2(a.c2, a.c2);
    float m = -INFINITY, l = 0.0f;
    for (int t = 0; t < nk; ++t) {
      const int s = t & 1;
      const int valid = kend - (t * 128 + static_cast<int>(part) * 32);
      if (!warp_wait(&B.s_full[s], (t >> 1) & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32(tmem + lane_off + L::kColS0 + s * 128 + part * 32, v);
      tc_fence_before();
      mbar_arrive(&B.s_free[s]);
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
    if (ok && part != 0) {
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
        if (qrow < a.Sq && ATTNQAT_IN_BOUNDS(static_cast<int64_t>(bh) * a.Sq + qrow < a.rows_q))
          a.lse[(size_t)bh * a.Sq + qrow] = lse2 * kLn2;
      } else {
        ok = false;
      }
    }

    // pass 2: P = exp2(S * c2 - lse2), P^ = fake_nvfp4(P); hand both to the MMA warps
    for (int t = nk; ok && t < nt; ++t) {
      const int s = t & 1, tv = t - nk;
      const int valid = kend - (tv * 128 + static_cast<int>(part) * 32);
      if (!warp_wait(&B.s_full[s], (t >> 1) & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      const uint32_t pcol = tmem + lane_off + L::kColS0 + s * 128 + part * 32;   // this warp's S columns
      float P[32];
      {
        uint32_t v[32];
        tmem_ld32(pcol, v);
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
      // P over columns [0,16) of this warp's S columns, P^ over [16,32)
      tmem_st16_nowait(pcol, pw);
      tmem_st16_nowait(pcol + 16, phw);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&B.p_ready[s]);
    }
    // epilogue: O' and O rows (a one-shot barrier committed after the last O'
    // and O MMAs); parts 0, 1 store O' columns [32 (p % 2), +32), parts 2, 3 O's.
    if (ok && warp_wait(&B.o_done, 0, ctl)) {
      tc_fence_after();
      const size_t row = (size_t)bh * a.Sq + qrow;
      uint32_t v[32];
      const uint32_t col = (part & 1) * 32;
      tmem_ld32(tmem + lane_off + (part < 2 ? L::kColOP : L::kColO) + col, v);
      if (qrow < a.Sq && ATTNQAT_IN_BOUNDS(static_cast<int64_t>(row) < a.rows_q))
        store_row32_bf16((part < 2 ? a.o_hp : a.o) + row * kD + col, v, 1.0f);
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
                       float* split_acc, uint32_t* split_cnt, uint32_t* err, cudaStream_t st) {
  if (p.D == 128) {
    // pass 1 (the LSE) in the paired kernel of fwd_lse.cu, then pass 2
    // (fwd_pv.cu) reading it; S on the block-scaled NVFP4 MMA in both
    if (vh == nullptr || q4 == nullptr || qsf == nullptr || k4 == nullptr || ksf == nullptr)
      return cudaErrorInvalidValue;
    cudaError_t e = launch_fwd_lse(p, q4, qsf, k4, ksf, lse, err, st);
    if (e != cudaSuccess) return e;
    return launch_fwd_pv(p, vh, q4, qsf, k4, ksf, lse, o, o_hp, split_acc, split_cnt, err, st);
  }
  if (p.D != kD) return cudaErrorInvalidValue;
  CUtensorMap tq, tk, tv;
  const uint64_t bh = p.bh();
  if (!make_tile_map(&tq, qh, false, kD, p.Sq, bh, 64, 128) || !make_tile_map(&tk, kh, false, kD, p.Sk, bh, 64, 128) ||
      !make_tile_map(&tv, vh, false, kD, p.Sk, bh, 64, 128))
    return cudaErrorInvalidValue;
  FwdArgs a;
  a.o = o, a.o_hp = o_hp, a.lse = lse;
  a.Sq = static_cast<int>(p.Sq), a.Sk = static_cast<int>(p.Sk);
  a.n_qtiles = static_cast<int>((p.Sq + kBlockM - 1) / kBlockM);
  a.n_ktiles = static_cast<int>((p.Sk + kBlockN - 1) / kBlockN);
  a.causal = p.causal ? 1 : 0;
  a.c2 = p.scale * kLog2e;
  a.err = err, a.timeout_ns = wait_timeout_ns();
  ATTNQAT_CHECKED_ONLY(a.rows_q = static_cast<int64_t>(p.bh()) * p.Sq; a.rows_k = static_cast<int64_t>(p.bh()) * p.Sk;)
  cudaError_t e = set_smem(reinterpret_cast<const void*>(&fwd_kernel), FwdLayout::kAlloc);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(a.n_qtiles), static_cast<unsigned>(bh));
  fwd_kernel<<<grid, kThreadsFwd, FwdLayout::kAlloc, st>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

// the debug build's count of skipped accesses in this file's kernels
ATTNQAT_OOB_READER(oob_read_fwd)

}  // namespace attnqat
