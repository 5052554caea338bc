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
// One CTA per 128-row query tile of one (b, h). Two passes over the key tiles,
// so that no accumulator is ever rescaled:
//   pass 1: S = Q K^T (2 FP4 MMAs of K = 64 per tile), row max only;
//   pass 2: S again, P = exp2(S * c2 - m) in BF16 written back over S in TMEM,
//           O += P V (8 BF16 MMAs with A from TMEM), row sum l.
// O = O / l at the end; LSE = (m + log2 l) * ln 2.
//
// Block-scaled MMA operands (measured contract): A and B K-major with 64-byte
// rows (128 E2M1 values, even element in the low nibble) and the 64-byte
// swizzle, 32 bytes per K = 64 step; scale factors in TMEM, 4 columns per K = 64
// step, lane r (in every lane quarter) holding in column j the four E4M3 bytes
// of row r + 32 j; scale-factor column addresses are multiples of 4.
//
// TMEM columns: S0 [0,128), S1 [128,256), O [256,384), Q scales [384,392),
// K scales x2 [400,408) and [416,424). Warps: 0-3 softmax (thread = query row,
// all 128 keys of a tile), 4 TMA producer, 5 MMA issuer.
// Shared memory: Q 8K, K x2 16K, V x2 64K.
#include "attn_common.cuh"

namespace attnqat {
namespace {

constexpr int kThreadsInf = 6 * 32;
constexpr int kWarpTmaI = 4;
constexpr int kWarpMmaI = 5;
constexpr int kD = 128;

struct InfLayout {
  static constexpr uint32_t kFp4Tile = 128 * 64;          // 128 rows x 64 bytes
  static constexpr uint32_t kVTile = 128 * kD * 2;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK0 = kQ + kFp4Tile;
  static constexpr uint32_t kK1 = kK0 + kFp4Tile;
  static constexpr uint32_t kV0 = kK1 + kFp4Tile;          // 1024-aligned: 24 KiB
  static constexpr uint32_t kV1 = kV0 + kVTile;
  static constexpr uint32_t kBar = kV1 + kVTile;
  static constexpr uint32_t kBytes = kBar + 256;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static constexpr uint32_t kColS0 = 0;
  static constexpr uint32_t kColO = 256;
  static constexpr uint32_t kColSFQ = 384;
  static constexpr uint32_t kColSFK0 = 400;
  static constexpr uint32_t kColSFK1 = 416;
};

struct InfBars {
  uint64_t q_full;
  uint64_t sfq_ready;
  uint64_t k_full[2];
  uint64_t k_empty[2];
  uint64_t v_full[2];
  uint64_t v_empty[2];
  uint64_t s_full[2];
  uint64_t s_free[2];     // pass 1: the softmax warps have read S
  uint64_t sf_ready[2];   // the K scales of the next tile in this buffer are in TMEM
  uint64_t p_ready[2];    // pass 2: P (BF16) is in TMEM over S
  uint64_t o_done;
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
};

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
};

// Shared-memory descriptor of a K-major tile with 64-byte rows and the 64-byte
// swizzle (8-row atoms of 512 bytes).
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(512 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)4 << 61;                       // SWIZZLE_64B
  return d;
}

// Instruction descriptor of tcgen05.mma kind::mxf4nvf4 with E2M1 A and B,
// UE4M3 scales, FP32 D.
__host__ __device__ constexpr uint32_t idesc_nvfp4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_nvfp4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

// Scales of a 128-row tile (rows row0.., `rows` valid) into the 8 TMEM columns
// at `col` of this warp's lane quarter, in the replicated layout above. Every
// softmax warp writes the same values into its own quarter.
__device__ __forceinline__ void write_scales(uint32_t taddr_quarter, const uint8_t* sf, int64_t row0, int rows) {
  const int r = static_cast<int>(lane_id());
  uint32_t w[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int row = r + 32 * j;
    uint2 v = make_uint2(0u, 0u);
    if (row < rows) v = __ldg(reinterpret_cast<const uint2*>(sf + (row0 + row) * 8));
    w[j] = v.x;          // K step 0: groups 0..3
    w[4 + j] = v.y;      // K step 1: groups 4..7
  }
  tmem_st8(taddr_quarter, w);
}

__global__ void __launch_bounds__(kThreadsInf, 1)
    infer_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const InfArgs a) {
  using L = InfLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  InfBars& B = *reinterpret_cast<InfBars*>(smem + L::kBar);

  const int warp = warp_id();
  const int lane = lane_id();
  const int i = a.causal ? (a.n_qtiles - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
  const int bh = blockIdx.y;
  const int nk = a.causal ? i + 1 : a.n_ktiles;
  const int nt = 2 * nk;                     // pass 1: T < nk; pass 2: T >= nk

  if (threadIdx.x == 0) {
    B.abort_flag = 0;
    mbar_init(&B.q_full, 1);
    mbar_init(&B.sfq_ready, 128);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&B.k_full[s], 1), mbar_init(&B.k_empty[s], 1);
      mbar_init(&B.v_full[s], 1), mbar_init(&B.v_empty[s], 1);
      mbar_init(&B.s_full[s], 1), mbar_init(&B.s_free[s], 128);
      mbar_init(&B.sf_ready[s], 128), mbar_init(&B.p_ready[s], 128);
    }
    mbar_init(&B.o_done, 1);
    mbar_init(&B.drain, 1);
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
      int k_uses[2] = {0, 0}, v_uses[2] = {0, 0};
      mbar_arrive_expect_tx(&B.q_full, L::kFp4Tile);
      tma_load_3d(smem + L::kQ, &tm_q, &B.q_full, 0, i * 128, bh);
      for (int T = 0; T < nt; ++T) {
        const int jt = T < nk ? T : T - nk;
        const int s = T & 1;
        if (T >= 2 && !mbar_wait(&B.k_empty[s], ((T >> 1) - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(&B.k_full[s], L::kFp4Tile);
        tma_load_3d(smem + (s ? L::kK1 : L::kK0), &tm_k, &B.k_full[s], 0, jt * 128, bh);
        ++k_uses[s];
        if (T >= nk) {
          const int tv = T - nk, sv = tv & 1;
          if (tv >= 2 && !mbar_wait(&B.v_empty[sv], ((tv >> 1) - 1) & 1, ctl)) break;
          mbar_arrive_expect_tx(&B.v_full[sv], L::kVTile);
          for (int b = 0; b < kD / 64; ++b)
            tma_load_3d(smem + (sv ? L::kV1 : L::kV0) + b * kBlockBytes, &tm_v, &B.v_full[sv], b * 64, jt * 128, bh);
          ++v_uses[sv];
        }
      }
      mbar_wait_drain(&B.q_full, 0, ctl);
      for (int s = 0; s < 2; ++s) {
        if (k_uses[s]) mbar_wait_drain(&B.k_full[s], (k_uses[s] - 1) & 1, ctl);
        if (v_uses[s]) mbar_wait_drain(&B.v_full[s], (v_uses[s] - 1) & 1, ctl);
      }
    }
  } else if (warp == kWarpMmaI) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_nvfp4(128, 128);
      constexpr uint32_t kIdO = idesc_bf16(128, kD, false, true);
      const uint64_t dq = sdesc_sw64(sbase + L::kQ);
      const uint64_t mnmaj = sdesc_sw128(sbase, kBlockBytes, 1024);
      auto issue_s = [&](int T) -> bool {
        const int s = T & 1;
        if (!mbar_wait(&B.k_full[s], (T >> 1) & 1, ctl)) return false;
        // previous occupant of this S buffer: read by the softmax warps (pass 1),
        // or its P read by the PV MMA issued earlier by this thread (in order)
        const int u = T - 2;
        if (u >= 0 && u < nk && !mbar_wait(&B.s_free[s], (u >> 1) & 1, ctl)) return false;
        if (!mbar_wait(&B.sf_ready[s], (T >> 1) & 1, ctl)) return false;
        tc_fence_after();
        const uint64_t dk = sdesc_sw64(sbase + (s ? L::kK1 : L::kK0));
        const uint32_t sfk = s ? L::kColSFK1 : L::kColSFK0;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          umma_nvfp4(tmem + L::kColS0 + s * 128, sdesc_advance(dq, ks * 32), sdesc_advance(dk, ks * 32), kIdS,
                     tmem + L::kColSFQ + ks * 4, tmem + sfk + ks * 4, ks > 0);
        umma_commit(&B.s_full[s]);
        umma_commit(&B.k_empty[s]);
        return true;
      };
      bool ok = mbar_wait(&B.q_full, 0, ctl) && mbar_wait(&B.sfq_ready, 0, ctl) && issue_s(0);
      for (int T = 0; ok && T < nt; ++T) {
        if (T + 1 < nt && !issue_s(T + 1)) break;
        if (T >= nk) {
          const int tv = T - nk, sv = tv & 1;
          if (!mbar_wait(&B.v_full[sv], (tv >> 1) & 1, ctl)) break;
          const int pr_use = (T >> 1) - ((nk + 1 - (T & 1)) >> 1);
          if (!mbar_wait(&B.p_ready[T & 1], pr_use & 1, ctl)) break;
          tc_fence_after();
          const uint64_t dv = sdesc_advance(mnmaj, sv ? L::kV1 : L::kV0);
          const uint32_t pc = L::kColS0 + (T & 1) * 128;    // P: keys 2c, 2c+1 in column pc + c
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_bf16_tmem_a(tmem + L::kColO, tmem + pc + kk * 8, sdesc_advance(dv, kk * 2048), kIdO,
                             (tv > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&B.v_empty[sv]);
          if (tv == nk - 1) umma_commit(&B.o_done);
        }
      }
      umma_commit(&B.drain);
      mbar_wait_drain(&B.drain, 0, ctl);
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 0-3)
    const uint32_t quarter = warp;
    const uint32_t r = quarter * 32 + lane;
    const uint32_t lane_off = (quarter * 32u) << 16;
    const int qrow = i * 128 + static_cast<int>(r);
    const int kend = a.causal ? min(a.Sk, qrow + 1) : a.Sk;
    const int64_t qbase = static_cast<int64_t>(bh) * a.Sq, kbase = static_cast<int64_t>(bh) * a.Sk;
    bool ok = true;
    auto k_scales = [&](int T) {   // K scales of global tile T into its buffer
      const int jt = T < nk ? T : T - nk;
      write_scales(tmem + lane_off + ((T & 1) ? L::kColSFK1 : L::kColSFK0), a.k_sf, kbase + jt * 128,
                   min(128, a.Sk - jt * 128));
      tc_fence_before();
      mbar_arrive(&B.sf_ready[T & 1]);
    };
    write_scales(tmem + lane_off + L::kColSFQ, a.q_sf, qbase + i * 128, min(128, a.Sq - i * 128));
    tc_fence_before();
    mbar_arrive(&B.sfq_ready);
    k_scales(0);
    if (nt > 1) k_scales(1);

    // pass 1: row max of S * c2
    float m = -INFINITY;
    for (int T = 0; T < nk; ++T) {
      const int s = T & 1;
      const int valid = kend - T * 128;
      if (!warp_wait(&B.s_full[s], (T >> 1) & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      float mc[4] = {m, m, m, m};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v[64];
        tmem_ld64(tmem + lane_off + L::kColS0 + s * 128 + h * 64, v);
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (h * 64 + k < valid) mc[k & 3] = fmaxf(mc[k & 3], __uint_as_float(v[k]) * a.c2);
      }
      tc_fence_before();
      mbar_arrive(&B.s_free[s]);
      m = fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3]));
      if (T + 2 < nt) k_scales(T + 2);
    }
    if (m == -INFINITY) m = 0.0f;   // a row with no live key (not reached for rows < Sq)

    // pass 2: P = exp2(S * c2 - m) as BF16 over S; row sum
    float lc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int T = nk; ok && T < nt; ++T) {
      const int s = T & 1, tv = T - nk;
      const int valid = kend - tv * 128;
      if (!warp_wait(&B.s_full[s], (T >> 1) & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      const uint32_t scol = tmem + lane_off + L::kColS0 + s * 128;
      uint32_t pw[64];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v[64];
        tmem_ld64(scol + h * 64, v);
#pragma unroll
        for (int k = 0; k < 64; k += 2) {
          const float p0 = (h * 64 + k < valid) ? ex2(fmaf(__uint_as_float(v[k]), a.c2, -m)) : 0.0f;
          const float p1 = (h * 64 + k + 1 < valid) ? ex2(fmaf(__uint_as_float(v[k + 1]), a.c2, -m)) : 0.0f;
          lc[k & 3] += p0;
          lc[(k + 1) & 3] += p1;
          pw[h * 32 + k / 2] = pack_bf16x2(p0, p1);
        }
      }
      uint32_t half0[32], half1[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) half0[k] = pw[k], half1[k] = pw[32 + k];
      tmem_st32(scol, half0);          // keys 0..63 in columns 0..31
      tmem_st32(scol + 32, half1);     // keys 64..127 in columns 32..63
      tc_fence_before();
      mbar_arrive(&B.p_ready[s]);
      if (T + 2 < nt) k_scales(T + 2);
    }
    const float l = (lc[0] + lc[1]) + (lc[2] + lc[3]);

    // epilogue: O / l, LSE
    if (ok && warp_wait(&B.o_done, 0, ctl)) {
      tc_fence_after();
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      bf16* out = a.o + (qbase + qrow) * kD;
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + L::kColO + c * 32, v);
        if (qrow < a.Sq) store_row32_bf16(out + c * 32, v, inv);
      }
      if (a.lse != nullptr && qrow < a.Sq) a.lse[qbase + qrow] = (m + lg2(l)) * kLn2;
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
  a.err = err, a.timeout_ns = kWaitTimeoutNs;
  cudaError_t e = set_smem(reinterpret_cast<const void*>(&infer_kernel), InfLayout::kAlloc);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(a.n_qtiles), static_cast<unsigned>(bh));
  infer_kernel<<<grid, kThreadsInf, InfLayout::kAlloc, st>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace attnqat
