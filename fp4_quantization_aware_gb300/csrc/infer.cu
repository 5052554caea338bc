// Attn-QAT inference forward (sm_103a): O = softmax(scale * Q K^T) V with Q and
// K in NVFP4 (E2M1 values, one E4M3 scale per 16) on the block-scaled FP4
// tensor-core MMA and V in BF16.
//
// "Attn-QAT: 4-Bit Attention With Quantization-Aware Training" (Key claims,
// Results; TMEM overlap schedule): block-scaled NVFP4 on the QK MMA, BF16 on
// PV ("FP4 only where it's free"); FastVideo attn_qat_infer page: NVFP4 per-16
// E4M3 scale factors for Q and K, fa4_pv_mode "bf16". The NVFP4 values of Q and
// K are exactly fake_nvfp4(Q), fake_nvfp4(K), so O equals the training
// forward's O' with an unquantized V.
//
// One CTA per 128-row query tile of one (b, h), one pass over the key tiles
// with an online softmax:
//   S(j) = Q K(j)^T            2 FP4 MMAs (K = 64 each) into TMEM buffer j % 2
//   m    = running row max; O and l are rescaled only when the tile's max
//          exceeds the reference by more than kRescaleLog2 (P <= 2^8 otherwise)
//   P(j) = exp2(S * c2 - m) in BF16, written back over S(j) in TMEM
//   O   += P(j) V(j)           8 BF16 MMAs with A read from TMEM
// O = O / l at the end; LSE = (m + log2 l) * ln 2.
//
// The softmax work is split over 8 warps: warp w owns lane quarter w % 4 (32
// query rows) and key half w / 4 (64 of the tile's 128 keys). The two warps of
// a quarter exchange their half-row maxima through shared memory once per
// tile (a 64-thread named barrier), so both take the same rescaling decision.
// S and PV are issued by two threads (on different SM sub-partitions, as an
// issuing thread slows the softmax warps of its own): S(j+2) overwrites buffer
// j % 2 once PV(j), which read P(j) from it, has completed (its commit).
//
// The block-scaled MMA's operand and scale-factor layouts are in fp4_mma.cuh.
//
// TMEM columns: S0 [0,128), S1 [128,256), O [256,384), Q scales [384,392),
// K scales x2 [400,408) and [416,424). Warps: 0-7 softmax, 8 TMA producer,
// 9 PV issuer, 10 S issuer.
#include "attn_common.cuh"
#include "checked.cuh"
#include "fp4_mma.cuh"

namespace attnqat {
namespace {

constexpr int kWarpTmaI = 8;    // SM sub-partition 0
// A thread issuing tcgen05.mma slows the softmax warps of its sub-partition:
// PV and S come from warps on two different ones.
constexpr int kWarpMmaI = 9;    // PV (and TMEM allocation), sub-partition 1
constexpr int kWarpMmaS = 10;   // S, sub-partition 2
constexpr int kThreadsInf = 11 * 32;
constexpr int kD = 128;
constexpr int kStagesK = 3;
constexpr int kStagesV = 3;
constexpr float kRescaleLog2 = 8.0f;

struct InfLayout {
  static constexpr uint32_t kFp4Tile = 128 * 64;          // 128 rows x 64 bytes
  static constexpr uint32_t kVTile = 128 * kD * 2;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + kFp4Tile;
  static constexpr uint32_t kV = kK + kStagesK * kFp4Tile;   // 1024-aligned
  static constexpr uint32_t kBar = kV + kStagesV * kVTile;
  static constexpr uint32_t kXchg = kBar + 512;               // maxima, flags [2][2][128], sums [2][128]
  static constexpr uint32_t kBytes = kXchg + 10 * 128 * 4;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static constexpr uint32_t kColS0 = 0;
  static constexpr uint32_t kColO = 256;
  static constexpr uint32_t kColSFQ = 384;
  static constexpr uint32_t kColSFK0 = 400;
  static constexpr uint32_t kColSFK1 = 416;
};
static_assert(InfLayout::kV % 1024 == 0, "V stages need 1024-byte alignment");
static_assert(InfLayout::kAlloc <= 227 * 1024, "shared memory");

struct InfBars {
  uint64_t q_full;
  uint64_t sf_init;       // Q scales and the K scales of tiles 0 and 1 are in TMEM
  uint64_t k_full[kStagesK];
  uint64_t k_empty[kStagesK];
  uint64_t v_full[kStagesV];
  uint64_t v_empty[kStagesV];
  uint64_t s_full[2];
  uint64_t p_ready[2];    // P(j) is in TMEM over S(j), and the K scales of tile j + 2
  uint64_t pv_done;       // one phase per PV(j) (waited only before rescaling O)
  uint64_t pv_read[2];    // per S buffer: PV(j) is done with P(j)
  uint64_t o_done;
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
};
static_assert(sizeof(InfBars) <= 512, "barrier area");

struct InfArgs {
  const uint8_t* q_sf;    // (B*H, Sq, 8) E4M3
  const uint8_t* k_sf;    // (B*H, Sk, 8)
  bf16* o;
  float* lse;             // may be null
  int Sq, Sk;
  int n_qtiles, n_ktiles;
  int causal;
  float c2;               // scale * log2(e)
  uint32_t* err;
  uint64_t timeout_ns;
  ATTNQAT_CHECKED_ONLY(int64_t rows_q; int64_t rows_k;)   // debug build: B*H*Sq, B*H*Sk
};

// Three warps share SM sub-partitions 0-2: at most 168 registers a thread.
__global__ void __maxnreg__(168)
    infer_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const InfArgs a) {
  using L = InfLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  InfBars& B = *reinterpret_cast<InfBars*>(smem + L::kBar);
  float* xmax = reinterpret_cast<float*>(smem + L::kXchg);        // [slot 2][half 2][row 128]
  uint32_t* xok = reinterpret_cast<uint32_t*>(xmax + 4 * 128);    // [slot 2][half 2][row 128]
  float* xsum = xmax + 8 * 128;                                   // [half 2][row 128]

  const int warp = warp_id();
  const int lane = lane_id();
  const int i = a.causal ? (a.n_qtiles - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
  const int bh = blockIdx.y;
  const int nk = a.causal ? i + 1 : a.n_ktiles;

  if (threadIdx.x == 0) {
    B.abort_flag = 0;
    mbar_init(&B.q_full, 1);
    mbar_init(&B.sf_init, 256);
    for (int s = 0; s < kStagesK; ++s) mbar_init(&B.k_full[s], 1), mbar_init(&B.k_empty[s], 1);
    for (int s = 0; s < kStagesV; ++s) mbar_init(&B.v_full[s], 1), mbar_init(&B.v_empty[s], 1);
    for (int s = 0; s < 2; ++s) mbar_init(&B.s_full[s], 1), mbar_init(&B.p_ready[s], 256);
    mbar_init(&B.pv_done, 1);
    mbar_init(&B.pv_read[0], 1), mbar_init(&B.pv_read[1], 1);
    mbar_init(&B.o_done, 1);
    mbar_init(&B.drain, 2);   // one commit per MMA-issuing thread
    fence_mbar_init();
  }
  if (warp == kWarpMmaI) {
    tmem_alloc(&B.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B.tmem_base;
  const WaitCtl ctl{&B.abort_flag, a.err, a.timeout_ns};

  if (warp == kWarpTmaI) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q), tma_prefetch_desc(&tm_k), tma_prefetch_desc(&tm_v);
      int k_uses[kStagesK] = {}, v_uses[kStagesV] = {};
      auto load_k = [&](int j) -> bool {
        const int s = j % kStagesK;
        if (j >= kStagesK && !mbar_wait(&B.k_empty[s], ((j / kStagesK) - 1) & 1, ctl)) return false;
        mbar_arrive_expect_tx(&B.k_full[s], L::kFp4Tile);
        tma_load_3d(smem + L::kK + s * L::kFp4Tile, &tm_k, &B.k_full[s], 0, j * 128, bh);
        ++k_uses[s];
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int s = j % kStagesV;
        if (j >= kStagesV && !mbar_wait(&B.v_empty[s], ((j / kStagesV) - 1) & 1, ctl)) return false;
        mbar_arrive_expect_tx(&B.v_full[s], L::kVTile);
        for (int b = 0; b < kD / 64; ++b)
          tma_load_3d(smem + L::kV + s * L::kVTile + b * kBlockBytes, &tm_v, &B.v_full[s], b * 64, j * 128, bh);
        ++v_uses[s];
        return true;
      };
      mbar_arrive_expect_tx(&B.q_full, L::kFp4Tile);
      tma_load_3d(smem + L::kQ, &tm_q, &B.q_full, 0, i * 128, bh);
      bool ok = load_k(0);
      for (int j = 0; ok && j < nk; ++j) {
        if (j + 1 < nk) ok = load_k(j + 1);
        if (ok) ok = load_v(j);
      }
      mbar_wait_drain(&B.q_full, 0, ctl);
      for (int s = 0; s < kStagesK; ++s)
        if (k_uses[s]) mbar_wait_drain(&B.k_full[s], (k_uses[s] - 1) & 1, ctl);
      for (int s = 0; s < kStagesV; ++s)
        if (v_uses[s]) mbar_wait_drain(&B.v_full[s], (v_uses[s] - 1) & 1, ctl);
    }
  } else if (warp == kWarpMmaS) {
    // ------------------------------------------------------------ S issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_nvfp4(128, 128);
      const uint64_t dq = sdesc_sw64(sbase + L::kQ);
      bool ok = mbar_wait(&B.q_full, 0, ctl) && mbar_wait(&B.sf_init, 0, ctl);
      for (int j = 0; ok && j < nk; ++j) {
        const int s = j % kStagesK, b = j & 1;
        // S(j) goes over P(j-2): once PV(j-2) is done with it. The K scales of
        // tile j were written with P(j-2) (p_ready). The polls overlap.
        const bool kf = mbar_try_wait(&B.k_full[s], (j / kStagesK) & 1);
        if (j >= 2 && !mbar_wait_both(&B.pv_read[b], ((j - 2) >> 1) & 1, &B.p_ready[b], ((j - 2) >> 1) & 1, ctl)) break;
        if (!kf && !mbar_wait(&B.k_full[s], (j / kStagesK) & 1, ctl)) break;
        tc_fence_after();
        const uint64_t dk = sdesc_sw64(sbase + L::kK + s * L::kFp4Tile);
        const uint32_t sfk = b ? L::kColSFK1 : L::kColSFK0;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          umma_nvfp4(tmem + L::kColS0 + b * 128, sdesc_advance(dq, ks * 32), sdesc_advance(dk, ks * 32), kIdS,
                     tmem + L::kColSFQ + ks * 4, tmem + sfk + ks * 4, ks > 0);
        umma_commit(&B.s_full[b]);
        umma_commit(&B.k_empty[s]);
      }
      umma_commit(&B.drain);
      mbar_wait_drain(&B.drain, 0, ctl);
    }
  } else if (warp == kWarpMmaI) {
    // ------------------------------------------------------------ PV issuer
    if (lane == 0) {
      constexpr uint32_t kIdO = idesc_bf16(128, kD, false, true);
      const uint64_t mnmaj = sdesc_sw128(sbase, kBlockBytes, 1024);
      bool ok = true;
      for (int j = 0; ok && j < nk; ++j) {
        const int sv = j % kStagesV, b = j & 1;
        if (!mbar_wait_both(&B.v_full[sv], (j / kStagesV) & 1, &B.p_ready[b], (j >> 1) & 1, ctl)) break;
        tc_fence_after();
        const uint64_t dv = sdesc_advance(mnmaj, L::kV + sv * L::kVTile);
        const uint32_t pc = L::kColS0 + b * 128;   // keys 64h + 2c, +1 of P in column pc + 64h + c
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16_tmem_a(tmem + L::kColO, tmem + pc + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_advance(dv, kk * 2048),
                           kIdO, (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&B.v_empty[sv]);
        umma_commit(&B.pv_done);
        umma_commit(&B.pv_read[b]);
        if (j == nk - 1) umma_commit(&B.o_done);
      }
      umma_commit(&B.drain);
      mbar_wait_drain(&B.drain, 0, ctl);
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 0-7)
    const uint32_t quarter = warp & 3, half = warp >> 2;
    const uint32_t r = quarter * 32 + lane;
    const uint32_t lane_off = (quarter * 32u) << 16;
    const uint32_t bar_id = 1 + quarter;                          // the quarter's two warps
    const int qrow = i * 128 + static_cast<int>(r);
    const int kend = a.causal ? min(a.Sk, qrow + 1) : a.Sk;
    const int64_t qbase = static_cast<int64_t>(bh) * a.Sq, kbase = static_cast<int64_t>(bh) * a.Sk;
    {
      uint32_t w[4];
      load_scales(a.q_sf, qbase + i * 128, ATTNQAT_IN_BOUNDS(qbase + i * 128 + min(128, a.Sq - i * 128) <= a.rows_q) ? min(128, a.Sq - i * 128) : 0, half, w);
      tmem_st4(tmem + lane_off + L::kColSFQ + 4 * half, w);
      load_scales(a.k_sf, kbase, ATTNQAT_IN_BOUNDS(kbase + min(128, a.Sk) <= a.rows_k) ? min(128, a.Sk) : 0, half, w);
      tmem_st4(tmem + lane_off + L::kColSFK0 + 4 * half, w);
      if (nk > 1) {
        load_scales(a.k_sf, kbase + 128, ATTNQAT_IN_BOUNDS(kbase + 128 + min(128, a.Sk - 128) <= a.rows_k) ? min(128, a.Sk - 128) : 0, half, w);
        tmem_st4(tmem + lane_off + L::kColSFK1 + 4 * half, w);
      }
      tc_fence_before();
      mbar_arrive(&B.sf_init);
    }

    float mref = -INFINITY;                    // reference max, in exp2 units
    float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
    bool ok = true, fail = false;
    for (int j = 0; j < nk; ++j) {
      const int b = j & 1;
      const bool more = j + 2 < nk;
      uint32_t sfw[4] = {0u, 0u, 0u, 0u};
      if (more)
        load_scales(a.k_sf, kbase + (j + 2) * 128,
                    ATTNQAT_IN_BOUNDS(kbase + (j + 2) * 128 + min(128, a.Sk - (j + 2) * 128) <= a.rows_k) ? min(128, a.Sk - (j + 2) * 128) : 0, half, sfw);
      const uint32_t scol = tmem + lane_off + L::kColS0 + b * 128 + 64 * half;
      uint32_t v[64];
      const bool got = !fail && warp_wait(&B.s_full[b], (j >> 1) & 1, ctl);
      if (got) {
        tc_fence_after();
        tmem_ld64(scol, v);
      } else {
#pragma unroll
        for (int k = 0; k < 64; ++k) v[k] = 0u;
      }
      const int valid = kend - j * 128 - 64 * static_cast<int>(half);
      if (valid < 64) {
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (k >= valid) v[k] = __float_as_uint(-INFINITY);
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int k = 0; k < 64; k += 8) {
        mx[0] = fmax3(mx[0], __uint_as_float(v[k]), __uint_as_float(v[k + 1]));
        mx[1] = fmax3(mx[1], __uint_as_float(v[k + 2]), __uint_as_float(v[k + 3]));
        mx[2] = fmax3(mx[2], __uint_as_float(v[k + 4]), __uint_as_float(v[k + 5]));
        mx[3] = fmax3(mx[3], __uint_as_float(v[k + 6]), __uint_as_float(v[k + 7]));
      }
      // half-row maxima and health flags through shared memory (both warps
      // of the quarter always reach this barrier the same number of times)
      const int slot = (j & 1) * 2;
      xmax[(slot + half) * 128 + r] = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3]));
      xok[(slot + half) * 128 + r] = got ? 1u : 0u;
      named_bar_sync(bar_id, 64);
      const float tmax = fmaxf(xmax[(slot + half) * 128 + r], xmax[(slot + (half ^ 1)) * 128 + r]);
      if (!got || xok[(slot + (half ^ 1)) * 128 + r] == 0u) {
        ok = false;
        break;
      }
      const float ms = tmax * a.c2;
      // The rescaling decision is per row, but the wait and the TMEM accesses
      // below are warp-collective: the whole warp enters when any of its rows
      // needs it (rows that do not use the factor 1). Both warps of a quarter
      // hold the same rows, so they take the same branch.
      const bool need = j > 0 && ms > mref + kRescaleLog2;
      if (j == 0) mref = ms;
      if (__any_sync(0xffffffffu, need)) {
        const float f = need ? ex2(mref - ms) : 1.0f;
        if (need) mref = ms;
        const float2 f2 = make_float2(f, f);
        acc0 = fmul2(acc0, f2), acc1 = fmul2(acc1, f2);
        // O holds PV(0..j-1): wait for PV(j-1), then rescale this half's columns
        if (warp_wait(&B.pv_done, (j - 1) & 1, ctl)) {
          tc_fence_after();
          uint32_t o[32];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint32_t oc = tmem + lane_off + L::kColO + 64 * half + 32 * c;
            tmem_ld32(oc, o);
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              const float2 t = fmul2(make_float2(__uint_as_float(o[k]), __uint_as_float(o[k + 1])), f2);
              o[k] = __float_as_uint(t.x), o[k + 1] = __float_as_uint(t.y);
            }
            tmem_st32(oc, o);
          }
        } else {
          fail = true;
        }
      }
      const float2 c2v = make_float2(a.c2, a.c2), nm = make_float2(-mref, -mref);
      uint32_t pw[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float2 x = ffma2(make_float2(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1])), c2v, nm);
        const float2 p = make_float2(ex2(x.x), ex2(x.y));
        if (c & 1) acc1 = fadd2(acc1, p);
        else acc0 = fadd2(acc0, p);
        pw[c] = pack_bf16x2(p.x, p.y);
      }
      tmem_st32(scol, pw);                                   // over this warp's own S columns
      if (more) tmem_st4(tmem + lane_off + (b ? L::kColSFK1 : L::kColSFK0) + 4 * half, sfw);
      tc_fence_before();
      mbar_arrive(&B.p_ready[b]);
    }
    const float2 lt = fadd2(acc0, acc1);
    const float l = lt.x + lt.y;
    xsum[half * 128 + r] = l;
    named_bar_sync(bar_id, 64);
    const float ltot = l + xsum[(half ^ 1) * 128 + r];

    // epilogue: this half's 64 columns of O / l; LSE
    if (ok && !fail && warp_wait(&B.o_done, 0, ctl)) {
      tc_fence_after();
      const float inv = ltot > 0.0f ? 1.0f / ltot : 0.0f;
      bf16* out = a.o + (qbase + qrow) * kD + 64 * half;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + L::kColO + 64 * half + 32 * c, o);
        if (qrow < a.Sq && ATTNQAT_IN_BOUNDS(qbase + qrow < a.rows_q)) store_row32_bf16(out + 32 * c, o, inv);
      }
      if (half == 0 && a.lse != nullptr && qrow < a.Sq && ATTNQAT_IN_BOUNDS(qbase + qrow < a.rows_q))
        a.lse[qbase + qrow] = (mref + lg2(ltot)) * kLn2;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaI) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_infer(const Problem& p, const uint8_t* q_fp4, const uint8_t* q_sf, const uint8_t* k_fp4,
                         const uint8_t* k_sf, const bf16* v, bf16* o, float* lse, uint32_t* err, cudaStream_t st) {
  if (p.D != kD) return cudaErrorInvalidValue;
  CUtensorMap tq, tk, tv;
  const uint64_t bh = p.bh();
  if (!make_fp4_map(&tq, q_fp4, p.Sq, bh, 128) || !make_fp4_map(&tk, k_fp4, p.Sk, bh, 128) ||
      !make_tile_map(&tv, v, false, p.D, p.Sk, bh, 64, 128))
    return cudaErrorInvalidValue;
  InfArgs a;
  a.q_sf = q_sf, a.k_sf = k_sf, a.o = o, a.lse = lse;
  a.Sq = static_cast<int>(p.Sq), a.Sk = static_cast<int>(p.Sk);
  a.n_qtiles = static_cast<int>((p.Sq + kBlockM - 1) / kBlockM);
  a.n_ktiles = static_cast<int>((p.Sk + kBlockN - 1) / kBlockN);
  a.causal = p.causal ? 1 : 0;
  a.c2 = p.scale * kLog2e;
  a.err = err, a.timeout_ns = wait_timeout_ns();
  ATTNQAT_CHECKED_ONLY(a.rows_q = static_cast<int64_t>(p.bh()) * p.Sq; a.rows_k = static_cast<int64_t>(p.bh()) * p.Sk;)
  cudaError_t e = set_smem(reinterpret_cast<const void*>(&infer_kernel), InfLayout::kAlloc);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(a.n_qtiles), static_cast<unsigned>(bh));
  infer_kernel<<<grid, kThreadsInf, InfLayout::kAlloc, st>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

// the debug build's count of skipped accesses in this file's kernels
ATTNQAT_OOB_READER(oob_read_infer)

}  // namespace attnqat
