// Attn-QAT forward, recipe R2 (sm_103a): one pass over the key tiles with an
// online softmax that fake-quantizes each tile's unnormalised probabilities.
//
// The review of the FastVideo pull request "Add Attn-QAT training Triton
// kernels" shows a one-pass forward whose row statistic is summed from the
// unquantized probabilities while P itself is quantized per tile. Per query
// row and key tile j (128 keys):
//   m_j  = max(m_{j-1}, max S_j)                     exact running max
//   P^_j = fake_nvfp4(exp(S_j - m_j))                groups of 16 keys
//   l    = rowsum of exp(S - m), O' = P V^ / l, LSE  as in the standard forward
//   O    = sum_j exp(m_j - m) P^_j V^_j / l
// (O' and LSE equal the standard recipe's, so the backward is unchanged.)
// The FP8-P variant (the branch that review is about) replaces fake_nvfp4 by
// an FP8 cast of each element of P_j, round to nearest even: E5M2 (Triton's
// tl.float8e5, which the review names) or E4M3. The kernel is a template on
// this P format (kPNvfp4, kPE5M2, kPE4M3).
//
// The accumulators use a reference max m_ref that moves only when the running
// max exceeds it by more than kRescaleLog2 (then O', O and l are rescaled), so
// that O' and O are rarely read back from TMEM. Each tile's quantization grid
// still follows the exact running max: P_q = exp2(S c2 - m_j) is
// fake-quantized and its P^ is scaled by 2^(m_j - m_ref) into the reference
// of the accumulators; P = P_q 2^(m_j - m_ref) feeds O' and l.
//
// One CTA per 128-row query tile of one (b, h). TMEM columns: S double-
// buffered [0,128) and [128,256), O' [256,256+D), O [256+D,256+2D); the
// softmax warps write P and P^ (BF16 pairs) back over the S tile they read
// (key half h: P in 64h + [0,32), P^ in 64h + [32,64)), and the O' and O MMAs
// take their A operand there. Warps: 0-7 softmax (warp w: lane quarter w % 4,
// key half w / 4; the two warps of a quarter exchange their half-row maxima
// once per tile), 8 TMA producer, 9 MMA issuer. Tensor-pipe order: S(0) S(1)
// PV(0) S(2) PV(1) ...; MMAs from one thread execute in issue order, so S(j+2)
// overwrites buffer j % 2 only after PV(j) has read P(j) and P^(j) from it.
#include "attn_common.cuh"
#include "checked.cuh"
#include "fp4_mma.cuh"

namespace attnqat {
namespace {

constexpr int kThreadsR2 = 10 * 32;
constexpr int kWarpTmaR2 = 8;
constexpr int kWarpMmaR2 = 9;
constexpr float kRescaleLog2R2 = 8.0f;

// P^ of one tile for the P formats: 16 unnormalised probabilities (>= 0,
// <= 1) of one thread, times g (the scale into the accumulators' reference),
// as 8 BF16 pairs. NVFP4: fake_nvfp4 of the group. FP8: the hardware
// conversion cvt.rn.satfinite.{e5m2x2,e4m3x2}.f32 (round to nearest even)
// and back to FP16, which holds both formats exactly.
template <int PF>
__device__ __forceinline__ void p_hat_16(const float* x, float g, uint32_t* out8) {
  if constexpr (PF == kPNvfp4) {
    fake_nvfp4_16_pack_nonneg<true>(x, g, out8);
  } else {
    const float2 g2 = make_float2(g, g);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint32_t h2;
      if constexpr (PF == kPE5M2) {
        asm("{\n\t.reg .b16 t;\n\t"
            "cvt.rn.satfinite.e5m2x2.f32 t, %1, %2;\n\t"
            "cvt.rn.f16x2.e5m2x2 %0, t;\n\t}"
            : "=r"(h2)
            : "f"(x[2 * k + 1]), "f"(x[2 * k]));
      } else {
        asm("{\n\t.reg .b16 t;\n\t"
            "cvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\t"
            "cvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
            : "=r"(h2)
            : "f"(x[2 * k + 1]), "f"(x[2 * k]));
      }
      const float2 y = fmul2(make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu))),
                                         __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)))),
                             g2);
      out8[k] = pack_bf16x2(y.x, y.y);
    }
  }
}

template <int D>
struct R2Layout {
  static constexpr uint32_t kTile = 128 * D * 2;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK0 = kQ + kTile;
  static constexpr uint32_t kK1 = kK0 + kTile;
  static constexpr uint32_t kV0 = kK1 + kTile;
  static constexpr uint32_t kV1 = kV0 + kTile;
  static constexpr uint32_t kBar = kV1 + kTile;
  static constexpr uint32_t kXchg = kBar + 256;           // maxima, flags [2][2][128], sums [2][128]
  static constexpr uint32_t kBytes = kXchg + 10 * 128 * 4;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static constexpr uint32_t kColS0 = 0;
  static constexpr uint32_t kColOP = 256;
  static constexpr uint32_t kColO = 256 + D;
};

struct R2Bars {
  uint64_t q_full;
  uint64_t k_full[2];
  uint64_t k_empty[2];
  uint64_t v_full[2];
  uint64_t v_empty[2];
  uint64_t s_full[2];
  uint64_t p_ready[2];   // P and P^ of tile j are in TMEM over S(j)
  uint64_t pv_done;      // one phase per tile's O' and O MMAs (waited only before rescaling)
  uint64_t o_done;
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
};

struct R2Args {
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

template <int D, int PF>
__global__ void __launch_bounds__(kThreadsR2, 1)
    fwd_r2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const R2Args a) {
  using L = R2Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  R2Bars& B = *reinterpret_cast<R2Bars*>(smem + L::kBar);
  float* xmax = reinterpret_cast<float*>(smem + L::kXchg);        // [slot 2][half 2][row 128]
  uint32_t* xok = reinterpret_cast<uint32_t*>(xmax + 4 * 128);    // [slot 2][half 2][row 128]
  float* xsum = xmax + 8 * 128;                                   // [half 2][row 128]

  const int warp = warp_id();
  const int lane = lane_id();
  // Causal tiles have i + 1 key tiles: launch the longest first.
  const int i = a.causal ? (a.n_qtiles - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
  const int bh = blockIdx.y;
  const int nk = a.causal ? i + 1 : a.n_ktiles;

  if (threadIdx.x == 0) {
    B.abort_flag = 0;
    mbar_init(&B.q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&B.k_full[s], 1), mbar_init(&B.k_empty[s], 1);
      mbar_init(&B.v_full[s], 1), mbar_init(&B.v_empty[s], 1);
      mbar_init(&B.s_full[s], 1), mbar_init(&B.p_ready[s], 256);
    }
    mbar_init(&B.pv_done, 1);
    mbar_init(&B.o_done, 1);
    mbar_init(&B.drain, 1);
    fence_mbar_init();
  }
  if (warp == kWarpMmaR2) {
    tmem_alloc(&B.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B.tmem_base;
  const WaitCtl ctl{&B.abort_flag, a.err, a.timeout_ns};

  if (warp == kWarpTmaR2) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q), tma_prefetch_desc(&tm_k), tma_prefetch_desc(&tm_v);
      int k_uses[2] = {0, 0}, v_uses[2] = {0, 0};
      auto load_k = [&](int j) -> bool {
        const int s = j & 1;
        if (j >= 2 && !mbar_wait(&B.k_empty[s], ((j >> 1) - 1) & 1, ctl)) return false;
        mbar_arrive_expect_tx(&B.k_full[s], L::kTile);
        for (int b = 0; b < D / 64; ++b)
          tma_load_3d(smem + (s ? L::kK1 : L::kK0) + b * kBlockBytes, &tm_k, &B.k_full[s], b * 64, j * 128, bh);
        ++k_uses[s];
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int s = j & 1;
        if (j >= 2 && !mbar_wait(&B.v_empty[s], ((j >> 1) - 1) & 1, ctl)) return false;
        mbar_arrive_expect_tx(&B.v_full[s], L::kTile);
        for (int b = 0; b < D / 64; ++b)
          tma_load_3d(smem + (s ? L::kV1 : L::kV0) + b * kBlockBytes, &tm_v, &B.v_full[s], b * 64, j * 128, bh);
        ++v_uses[s];
        return true;
      };
      mbar_arrive_expect_tx(&B.q_full, L::kTile);
      for (int b = 0; b < D / 64; ++b)
        tma_load_3d(smem + L::kQ + b * kBlockBytes, &tm_q, &B.q_full, b * 64, i * 128, bh);
      bool ok = load_k(0);
      for (int j = 0; ok && j < nk; ++j) {
        if (j + 1 < nk) ok = load_k(j + 1);
        if (ok) ok = load_v(j);
      }
      mbar_wait_drain(&B.q_full, 0, ctl);
      for (int s = 0; s < 2; ++s) {
        if (k_uses[s]) mbar_wait_drain(&B.k_full[s], (k_uses[s] - 1) & 1, ctl);
        if (v_uses[s]) mbar_wait_drain(&B.v_full[s], (v_uses[s] - 1) & 1, ctl);
      }
    }
  } else if (warp == kWarpMmaR2) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdO = idesc_bf16(128, D, false, true);
      const uint64_t kmaj = sdesc_sw128(sbase, 16, 1024);
      const uint64_t mnmaj = sdesc_sw128(sbase, kBlockBytes, 1024);
      const uint64_t dq = sdesc_advance(kmaj, L::kQ);
      auto issue_s = [&](int j) -> bool {
        const int s = j & 1;
        if (!mbar_wait(&B.k_full[s], (j >> 1) & 1, ctl)) return false;
        tc_fence_after();
        const uint64_t db = sdesc_advance(kmaj, s ? L::kK1 : L::kK0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = (kk >> 2) * kBlockBytes + (kk & 3) * 32;
          umma_bf16(tmem + L::kColS0 + s * 128, sdesc_advance(dq, o), sdesc_advance(db, o), kIdS, kk > 0);
        }
        umma_commit(&B.s_full[s]);
        umma_commit(&B.k_empty[s]);
        return true;
      };
      // O (+)= A[128 q x 128 keys] V^[128 keys x D], A from TMEM at a_col
      // (keys 0..63 in columns a_col + [0,32), keys 64..127 in a_col + 64 + [0,32)).
      auto mma_pv = [&](uint32_t a_col, uint32_t v_off, uint32_t col, bool acc) {
        const uint64_t dv = sdesc_advance(mnmaj, v_off);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t ac = a_col + (kk >> 2) * 64 + (kk & 3) * 8;
          umma_bf16_tmem_a(tmem + col, tmem + ac, sdesc_advance(dv, kk * 2048), kIdO, (acc || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(&B.q_full, 0, ctl) && issue_s(0) && (nk < 2 || issue_s(1));
      for (int j = 0; ok && j < nk; ++j) {
        const int s = j & 1;
        if (!mbar_wait(&B.v_full[s], (j >> 1) & 1, ctl)) break;
        if (!mbar_wait(&B.p_ready[s], (j >> 1) & 1, ctl)) break;
        tc_fence_after();
        const uint32_t vb = s ? L::kV1 : L::kV0;
        const uint32_t sc = L::kColS0 + s * 128;
        mma_pv(sc, vb, L::kColOP, j > 0);        // O' += P V^
        mma_pv(sc + 32, vb, L::kColO, j > 0);    // O  += P^ V^
        umma_commit(&B.v_empty[s]);
        umma_commit(&B.pv_done);
        if (j == nk - 1) umma_commit(&B.o_done);
        if (j + 2 < nk && !issue_s(j + 2)) break;
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
    const int64_t qbase = static_cast<int64_t>(bh) * a.Sq;

    float mref = -INFINITY;                    // accumulators' reference max (exp2 units)
    float mrun = -INFINITY;                    // exact running max (exp2 units)
    float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
    bool ok = true, fail = false;
    for (int j = 0; j < nk; ++j) {
      const int b = j & 1;
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
      // every row has a live key in every tile it visits, so tmax is finite
      mrun = fmaxf(mrun, tmax * a.c2);
      // The reference moves per row, but the wait and the TMEM accesses below
      // are warp-collective: the whole warp enters when any of its rows needs
      // it (rows that do not use the factor 1). Both warps of a quarter hold
      // the same rows, so they take the same branch.
      const bool need = j > 0 && mrun > mref + kRescaleLog2R2;
      if (j == 0) mref = mrun;
      if (__any_sync(0xffffffffu, need)) {
        const float f = need ? ex2(mref - mrun) : 1.0f;
        if (need) mref = mrun;
        const float2 f2 = make_float2(f, f);
        acc0 = fmul2(acc0, f2), acc1 = fmul2(acc1, f2);
        // O' and O hold PV(0..j-1): wait for PV(j-1), then rescale this
        // warp's columns of both
        if (warp_wait(&B.pv_done, (j - 1) & 1, ctl)) {
          tc_fence_after();
          uint32_t o[32];
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const uint32_t oc = tmem + lane_off + (t ? L::kColO : L::kColOP) + half * (D / 2) + 32 * c;
              tmem_ld32(oc, o);
#pragma unroll
              for (int k = 0; k < 32; k += 2) {
                const float2 x = fmul2(make_float2(__uint_as_float(o[k]), __uint_as_float(o[k + 1])), f2);
                o[k] = __float_as_uint(x.x), o[k + 1] = __float_as_uint(x.y);
              }
              tmem_st32(oc, o);
            }
          }
        } else {
          fail = true;
        }
      }
      // P_q = exp2(S c2 - m_j) relative to the running max (the recipe's
      // quantization grid); P = P_q G with G = 2^(m_j - m_ref) for O' and l.
      const float G = ex2(mrun - mref);
      const float2 c2v = make_float2(a.c2, a.c2), nm = make_float2(-mrun, -mrun), g2 = make_float2(G, G);
      float pq[64];
      uint32_t pw[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float2 x = ffma2(make_float2(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1])), c2v, nm);
        pq[2 * c] = ex2(x.x), pq[2 * c + 1] = ex2(x.y);
        const float2 p = fmul2(make_float2(pq[2 * c], pq[2 * c + 1]), g2);
        if (c & 1) acc1 = fadd2(acc1, p);
        else acc0 = fadd2(acc0, p);
        pw[c] = pack_bf16x2(p.x, p.y);
      }
      uint32_t phw[32];
#pragma unroll
      for (int g = 0; g < 4; ++g) p_hat_16<PF>(pq + 16 * g, G, phw + 8 * g);
      tmem_st32(scol, pw);                                   // over this warp's own S columns
      tmem_st32(scol + 32, phw);
      tc_fence_before();
      mbar_arrive(&B.p_ready[b]);
    }
    const float2 lt = fadd2(acc0, acc1);
    const float l = lt.x + lt.y;
    xsum[half * 128 + r] = l;
    named_bar_sync(bar_id, 64);
    const float ltot = l + xsum[(half ^ 1) * 128 + r];

    // epilogue: this warp's columns of O' / l and O / l; LSE
    if (ok && !fail && warp_wait(&B.o_done, 0, ctl)) {
      tc_fence_after();
      const float inv = ltot > 0.0f ? 1.0f / ltot : 0.0f;
      const size_t row = (size_t)qbase + qrow;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const uint32_t col = half * (D / 2) + c * 32;
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + L::kColOP + col, o);
        if (qrow < a.Sq && ATTNQAT_IN_BOUNDS(static_cast<int64_t>(row) < a.rows_q))
          store_row32_bf16(a.o_hp + row * D + col, o, inv);
        tmem_ld32(tmem + lane_off + L::kColO + col, o);
        if (qrow < a.Sq && ATTNQAT_IN_BOUNDS(static_cast<int64_t>(row) < a.rows_q))
          store_row32_bf16(a.o + row * D + col, o, inv);
      }
      if (half == 0 && qrow < a.Sq && ATTNQAT_IN_BOUNDS(static_cast<int64_t>(row) < a.rows_q))
        a.lse[row] = (mref + lg2(ltot)) * kLn2;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaR2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int PF>
cudaError_t launch_r2(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const R2Args& a,
                      dim3 grid, cudaStream_t st) {
  cudaError_t e = set_smem(reinterpret_cast<const void*>(&fwd_r2_kernel<D, PF>), R2Layout<D>::kAlloc);
  if (e != cudaSuccess) return e;
  fwd_r2_kernel<D, PF><<<grid, kThreadsR2, R2Layout<D>::kAlloc, st>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_r2_fmt(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const R2Args& a,
                          dim3 grid, int p_format, cudaStream_t st) {
  switch (p_format) {
    case kPNvfp4: return launch_r2<D, kPNvfp4>(tq, tk, tv, a, grid, st);
    case kPE5M2: return launch_r2<D, kPE5M2>(tq, tk, tv, a, grid, st);
    case kPE4M3: return launch_r2<D, kPE4M3>(tq, tk, tv, a, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_fwd_r2(const Problem& p, const bf16* qh, const bf16* kh, const bf16* vh, bf16* o, bf16* o_hp,
                          float* lse, int p_format, uint32_t* err, cudaStream_t st) {
  CUtensorMap tq, tk, tv;
  const uint64_t bh = p.bh();
  if (!make_tile_map(&tq, qh, false, p.D, p.Sq, bh, 64, 128) || !make_tile_map(&tk, kh, false, p.D, p.Sk, bh, 64, 128) ||
      !make_tile_map(&tv, vh, false, p.D, p.Sk, bh, 64, 128))
    return cudaErrorInvalidValue;
  R2Args a;
  a.o = o, a.o_hp = o_hp, a.lse = lse;
  a.Sq = static_cast<int>(p.Sq), a.Sk = static_cast<int>(p.Sk);
  a.n_qtiles = static_cast<int>((p.Sq + kBlockM - 1) / kBlockM);
  a.n_ktiles = static_cast<int>((p.Sk + kBlockN - 1) / kBlockN);
  a.causal = p.causal ? 1 : 0;
  a.c2 = p.scale * kLog2e;
  a.err = err, a.timeout_ns = wait_timeout_ns();
  ATTNQAT_CHECKED_ONLY(a.rows_q = static_cast<int64_t>(p.bh()) * p.Sq; a.rows_k = static_cast<int64_t>(p.bh()) * p.Sk;)
  const dim3 grid(static_cast<unsigned>(a.n_qtiles), static_cast<unsigned>(bh));
  return p.D == 128 ? launch_r2_fmt<128>(tq, tk, tv, a, grid, p_format, st)
                    : launch_r2_fmt<64>(tq, tk, tv, a, grid, p_format, st);
}

// the debug build's count of skipped accesses in this file's kernels
ATTNQAT_OOB_READER(oob_read_fwd_r2)

}  // namespace attnqat
