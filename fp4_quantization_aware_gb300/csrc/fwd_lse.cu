// Attn-QAT forward, pass 1 at D = 128 (sm_103a): the natural-log LSE of two
// query tiles of one head per CTA.
//
// "Attn-QAT: 4-Bit Attention With Quantization-Aware Training" (Method, Fix 1)
// and "NVFP4 Attention QAT Backward" (cuDNN frontend docs, Overview, High-level
// wrapper): P^ = fake_nvfp4(P) is taken of the normalised probabilities, so the
// forward first needs LSE = ln sum_j exp(scale * Q^ K^T)_j of every query row;
// the second pass (fwd_pv.cu, reading this kernel's LSE) forms P, P^, O' and O.
//
// This pass issues one small MMA per key tile (S on the block-scaled NVFP4
// MMA) and is bound by the exp2 work of the softmax warps. A CTA takes two
// query tiles A, B of one head, which share each K tile (loaded once).
//
// Each softmax thread owns one query row of one tile: it loads the row's 128
// S values of a key tile from TMEM, releases the S buffer (so the next S MMA
// of its tile can run while it computes), and keeps the row's running max and
// sum of exp2(S * scale * log2 e) by itself. The per-tile costs of a hand-off
// (barrier poll, TMEM load, release) are paid once per 128 keys of a row, and
// the row's LSE needs no combining across threads. The warps of tile A and of
// tile B share each SM sub-partition, so one tile's waits overlap the other's
// arithmetic.
//
// TMEM: S_A [0,128), S_B [128,256) (one buffer each: S_X(j+1) is issued once
// the softmax warps of tile X have loaded S_X(j)); scale factors of the MMAs in
// columns of their own: Q of tile X at 256 + 8 X + 4 ks, K of key tile j at
// 272 + 8 (j % 2) + 4 ks (4 columns per K = 64 step; lane r holds in column c
// the four scale bytes of row r + 32 c). Key tile j + 2's K scales go into
// slot j % 2 once the last S of step j (which read it) is complete; they are
// written by the warps of tile B (of tile A when the CTA has no tile B), which
// see every step.
//
// Warps (10): 0-7 softmax (warp w: tile w / 4, lane quarter w % 4); 8 TMA
// producer; 9 MMA issuer (and TMEM allocation).
#include "attn_common.cuh"
#include "fp4_mma.cuh"
#include "checked.cuh"

namespace attnqat {
namespace {

constexpr int kSoftWarpsL = 8;
constexpr int kWarpTmaL = 8;
constexpr int kWarpMmaL = 9;
constexpr int kThreadsL = 10 * 32;

struct LseLayout {
  static constexpr int kStages = 4;                      // NVFP4 K tiles in flight
  static constexpr uint32_t kFp4Tile = 128 * 64;         // 128 rows x 64 bytes of E2M1 pairs
  static constexpr uint32_t kQ4 = 0;                     // tile X at kQ4 + X * kFp4Tile
  static constexpr uint32_t kK0 = 2 * kFp4Tile;          // stage s at kK0 + s * kFp4Tile
  static constexpr uint32_t kBar = kK0 + kStages * kFp4Tile;
  static constexpr uint32_t kBytes = kBar + 256;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static constexpr uint32_t kColSFQ = 256;               // + 8 X + 4 ks
  static constexpr uint32_t kColSFK = 272;               // + 8 slot + 4 ks
  static_assert(kK0 % 1024 == 0, "swizzled tiles need 1024-byte alignment");
};

struct LseBars {
  uint64_t q_full;
  uint64_t k_full[4], k_empty[4];
  uint64_t s_full[2];   // per tile: S_X(j) complete
  uint64_t s_free[2];   // per tile: S_X(j) loaded (and, for the scale writers, key tile j + 2's K scales written)
  uint64_t sf_init;     // Q scales of both tiles, K scales of key tiles 0 and 1 written
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
};

struct LseArgs {
  const uint8_t* q_sf;   // NVFP4 scales of Q, K ((B*H, S, 8) E4M3)
  const uint8_t* k_sf;
  float* lse;
  int Sq, Sk;
  int n_qtiles, n_ktiles, n_pairs;
  int causal;
  float c2;              // scale * log2(e)
  uint32_t* err;
  uint64_t timeout_ns;
  ATTNQAT_CHECKED_ONLY(int64_t rows_q; int64_t rows_k;)   // debug build: B*H*Sq, B*H*Sk
};

// 32 TMEM columns of this warp's 32 lanes, without waiting.
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// 128 TMEM columns of this warp's 32 lanes in one load, without waiting.
__device__ __forceinline__ void tmem_ld128_nowait(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
}

// Ties 32 registers to a point in the instruction stream: with `wait` set the
// asm block also waits for this thread's TMEM loads, so no use of the
// registers can move above the wait.
template <bool kWait>
__device__ __forceinline__ void tmem_tie32(uint32_t* r) {
  if constexpr (kWait) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
  } else {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
  }
}

__device__ __forceinline__ void tmem_st4_nowait(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}

__global__ void __launch_bounds__(kThreadsL, 1)
    fwd_lse_kernel(const __grid_constant__ CUtensorMap tm_q4, const __grid_constant__ CUtensorMap tm_k4,
                   const LseArgs a) {
  using L = LseLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  LseBars& B = *reinterpret_cast<LseBars*>(smem + L::kBar);

  const int warp = warp_id();
  const int lane = lane_id();
  // Causal pairs have 2p + 1 and 2p + 2 key tiles: launch the longest first.
  const int pr = a.causal ? (a.n_pairs - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
  const int bh = blockIdx.y;
  const int i0 = 2 * pr, i1 = 2 * pr + 1;            // query tiles A, B
  const bool hasB = i1 < a.n_qtiles;
  const int nA = a.causal ? i0 + 1 : a.n_ktiles;
  const int nB = hasB ? (a.causal ? i1 + 1 : a.n_ktiles) : 0;
  const int n_steps = max(nA, nB);                    // nA <= nB whenever B exists

  if (threadIdx.x == 0) {
    B.abort_flag = 0;
    mbar_init(&B.q_full, 1);
    for (int s = 0; s < L::kStages; ++s) mbar_init(&B.k_full[s], 1), mbar_init(&B.k_empty[s], 1);
    for (int x = 0; x < 2; ++x) mbar_init(&B.s_full[x], 1), mbar_init(&B.s_free[x], 4 * 32);   // the tile's warps
    mbar_init(&B.sf_init, kSoftWarpsL * 32);
    mbar_init(&B.drain, 1);
    fence_mbar_init();
  }
  if (warp == kWarpMmaL) {
    tmem_alloc(&B.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B.tmem_base;
  const WaitCtl ctl{&B.abort_flag, a.err, a.timeout_ns};
  // launched as a programmatic dependent of the quantize step: its NVFP4 Q,
  // K and scales are read after grid_dep_wait; pass 2 may then start
  grid_dep_wait();
  grid_dep_launch();

  if (warp == kWarpTmaL) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q4), tma_prefetch_desc(&tm_k4);
      mbar_arrive_expect_tx(&B.q_full, (hasB ? 2 : 1) * L::kFp4Tile);
      tma_load_3d(smem + L::kQ4, &tm_q4, &B.q_full, 0, i0 * 128, bh);
      if (hasB) tma_load_3d(smem + L::kQ4 + L::kFp4Tile, &tm_q4, &B.q_full, 0, i1 * 128, bh);
      int uses[L::kStages] = {};
      for (int j = 0; j < n_steps; ++j) {
        const int s = j % L::kStages, use = j / L::kStages;
        if (use >= 1 && !mbar_wait(&B.k_empty[s], (use - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(&B.k_full[s], L::kFp4Tile);
        tma_load_3d(smem + L::kK0 + s * L::kFp4Tile, &tm_k4, &B.k_full[s], 0, j * 128, bh);
        ++uses[s];
      }
      // every copy issued above lands before shared memory is released
      mbar_wait_drain(&B.q_full, 0, ctl);
      for (int s = 0; s < L::kStages; ++s)
        if (uses[s]) mbar_wait_drain(&B.k_full[s], (uses[s] - 1) & 1, ctl);
    }
  } else if (warp == kWarpMmaL) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kId = idesc_nvfp4(128, 128);
      const uint64_t dk0 = sdesc_sw64(sbase + L::kK0);
      bool ok = mbar_wait(&B.q_full, 0, ctl) && mbar_wait(&B.sf_init, 0, ctl);
      auto issue = [&](int x, int j) {
        const uint64_t dq = sdesc_sw64(sbase + L::kQ4 + x * L::kFp4Tile);
        const uint64_t dk = sdesc_advance(dk0, (j % L::kStages) * L::kFp4Tile);
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          umma_nvfp4(tmem + x * 128u, sdesc_advance(dq, ks * 32), sdesc_advance(dk, ks * 32), kId,
                     tmem + L::kColSFQ + 8 * x + 4 * ks, tmem + L::kColSFK + 8 * (j & 1) + 4 * ks, ks > 0);
        umma_commit(&B.s_full[x]);
      };
      // Key tile j's K scales were written at step j - 2 before the scale
      // writers released their tile's S; this thread waited for that release
      // before issuing an S of step j - 1, so the writes precede these MMAs.
      for (int j = 0; ok && j < n_steps; ++j) {
        const int s = j % L::kStages;
        const bool kf = mbar_try_wait(&B.k_full[s], (j / L::kStages) & 1);
        const bool doA = j < nA, doB = hasB && j < nB;
        // S_X(j) goes where S_X(j - 1) was, once the softmax warps have loaded it
        if (doA) {
          if ((j >= 1 && !mbar_wait(&B.s_free[0], (j - 1) & 1, ctl)) ||
              (!kf && !mbar_wait(&B.k_full[s], (j / L::kStages) & 1, ctl))) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue(0, j);
        }
        if (doB) {
          if ((j >= 1 && !mbar_wait(&B.s_free[1], (j - 1) & 1, ctl)) ||
              (!doA && !kf && !mbar_wait(&B.k_full[s], (j / L::kStages) & 1, ctl))) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue(1, j);
        }
        umma_commit(&B.k_empty[s]);
      }
      umma_commit(&B.drain);
      mbar_wait_drain(&B.drain, 0, ctl);
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 0-7)
    const int x = warp >> 2;                       // tile A or B
    const uint32_t quarter = warp & 3;
    const uint32_t r = quarter * 32 + lane;
    const uint32_t lane_off = (quarter * 32u) << 16;
    const bool active = x == 0 || hasB;
    const bool sf_writer = x == (hasB ? 1 : 0);   // writes the K scales (both K steps)
    const int nX = x == 0 ? nA : nB;
    const int qi = x == 0 ? i0 : i1;
    const int qrow = qi * 128 + static_cast<int>(r);
    const int kend = a.causal ? min(a.Sk, qrow + 1) : a.Sk;
    const int64_t kbase = static_cast<int64_t>(bh) * a.Sk;
    auto k_scales = [&](int kt, uint32_t (&w)[2][4]) {
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)
        load_scales(a.k_sf, kbase + kt * 128,
                    ATTNQAT_IN_BOUNDS(kbase + kt * 128 + min(128, a.Sk - kt * 128) <= a.rows_k) ? min(128, a.Sk - kt * 128) : 0,
                    ks, w[ks]);
    };
    // Q scales of this warp's tile; K scales of key tiles 0, 1 (slots 0, 1)
    // from the scale writers. Every softmax thread arrives on sf_init.
    uint32_t sfw[2][4] = {}, sfo[2][4] = {};   // K scales written at step j (key tile j + 2's)
    if (active) {
      uint32_t wq[2][4], wk[2][2][4];
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)
        load_scales(a.q_sf, static_cast<int64_t>(bh) * a.Sq + qi * 128,
                    ATTNQAT_IN_BOUNDS(static_cast<int64_t>(bh) * a.Sq + qi * 128 + min(128, a.Sq - qi * 128) <= a.rows_q)
                        ? min(128, a.Sq - qi * 128) : 0,
                    ks, wq[ks]);
      if (sf_writer) {
#pragma unroll
        for (int kt = 0; kt < 2; ++kt)
          if (kt < n_steps) k_scales(kt, wk[kt]);
        if (2 < n_steps) k_scales(2, sfw);
      }
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) tmem_st4_nowait(tmem + lane_off + L::kColSFQ + 8 * x + 4 * ks, wq[ks]);
      if (sf_writer) {
#pragma unroll
        for (int kt = 0; kt < 2; ++kt)
          if (kt < n_steps) {
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) tmem_st4_nowait(tmem + lane_off + L::kColSFK + 8 * kt + 4 * ks, wk[kt][ks]);
          }
      }
      tmem_wait_st();
      tc_fence_before();
    }
    mbar_arrive(&B.sf_init);

    const float2 c22 = make_float2(a.c2, a.c2);
    float m = -INFINITY, l = 0.0f;
    // One key tile of this row: S (128 values) loaded and the buffer released,
    // then the running max and sum updated. `sf_now` holds key tile j + 2's
    // K scales (written here by the scale writers), `sf_next` receives key
    // tile j + 3's (the loop alternates the two, so no copy waits for a load).
    auto step = [&](int j, const uint32_t (&sf_now)[2][4], uint32_t (&sf_next)[2][4]) -> bool {
      if (sf_writer && j + 3 < n_steps) k_scales(j + 3, sf_next);
      if (!warp_wait(&B.s_full[x], j & 1, ctl)) return false;
      tc_fence_after();
      uint32_t v[128];
      tmem_ld128_nowait(tmem + lane_off + x * 128u, v);
      tmem_tie32<true>(v);
      tmem_tie32<false>(v + 32);
      tmem_tie32<false>(v + 64);
      tmem_tie32<false>(v + 96);
      // S_X(j) is loaded; for the scale writers every S of step j is complete
      // (S_A(j) was issued before S_B(j)), so key tile j + 2's K scales go
      // into slot j % 2, which those MMAs read
      if (sf_writer && j + 2 < n_steps) {
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) tmem_st4_nowait(tmem + lane_off + L::kColSFK + 8 * (j & 1) + 4 * ks, sf_now[ks]);
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(&B.s_free[x]);
      const int valid = kend - j * 128;
      if (valid < 128) {   // masked keys: -inf
#pragma unroll
        for (int k = 0; k < 128; ++k)
          if (k >= valid) v[k] = 0xFF800000u;
      }
      // row max of the raw S in four chains (c2 > 0: max(S) * c2 is the max
      // of the scaled logits)
      float mq[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float acc = fmaxf(__uint_as_float(v[32 * u]), __uint_as_float(v[32 * u + 1]));
#pragma unroll
        for (int k = 2; k < 32; k += 2)
          acc = fmax3(acc, __uint_as_float(v[32 * u + k]), __uint_as_float(v[32 * u + k + 1]));
        mq[u] = acc;
      }
      const float mx = fmaxf(m, fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * a.c2);
      if (mx == -INFINITY) return true;   // every key of the row so far masked
      // sum of exp2(S * c2 - mx), arguments and partial sums as packed pairs
      const float2 nm = make_float2(-mx, -mx);
      float2 sc[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) sc[k] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int k = 0; k < 64; ++k) {
        const float2 e = ffma2(make_float2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1])), c22, nm);
        sc[k & 7] = fadd2(sc[k & 7], make_float2(ex2(e.x), ex2(e.y)));
      }
      const float2 s4 = fadd2(fadd2(fadd2(sc[0], sc[1]), fadd2(sc[2], sc[3])), fadd2(fadd2(sc[4], sc[5]), fadd2(sc[6], sc[7])));
      l = l * ex2(m - mx) + (s4.x + s4.y);
      m = mx;
      return true;
    };
    bool ok = true;
    for (int j = 0; active && ok && j < nX; j += 2) {
      ok = step(j, sfw, sfo);
      if (ok && j + 1 < nX) ok = step(j + 1, sfo, sfw);
    }
    if (active && ok && qrow < a.Sq && ATTNQAT_IN_BOUNDS(static_cast<int64_t>(bh) * a.Sq + qrow < a.rows_q))
      a.lse[(size_t)bh * a.Sq + qrow] = (m + lg2(l)) * kLn2;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaL) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_fwd_lse(const Problem& p, const uint8_t* q4, const uint8_t* qsf, const uint8_t* k4,
                           const uint8_t* ksf, float* lse, uint32_t* err, cudaStream_t st) {
  if (p.D != 128 || q4 == nullptr || qsf == nullptr || k4 == nullptr || ksf == nullptr) return cudaErrorInvalidValue;
  CUtensorMap tq4, tk4;
  const uint64_t bh = p.bh();
  if (!make_fp4_map(&tq4, q4, p.Sq, bh, 128) || !make_fp4_map(&tk4, k4, p.Sk, bh, 128)) return cudaErrorInvalidValue;
  LseArgs a;
  a.q_sf = qsf, a.k_sf = ksf, a.lse = lse;
  a.Sq = static_cast<int>(p.Sq), a.Sk = static_cast<int>(p.Sk);
  a.n_qtiles = static_cast<int>((p.Sq + kBlockM - 1) / kBlockM);
  a.n_ktiles = static_cast<int>((p.Sk + kBlockN - 1) / kBlockN);
  a.n_pairs = (a.n_qtiles + 1) / 2;
  a.causal = p.causal ? 1 : 0;
  a.c2 = p.scale * kLog2e;
  a.err = err, a.timeout_ns = wait_timeout_ns();
  ATTNQAT_CHECKED_ONLY(a.rows_q = static_cast<int64_t>(p.bh()) * p.Sq; a.rows_k = static_cast<int64_t>(p.bh()) * p.Sk;)
  const dim3 grid(static_cast<unsigned>(a.n_pairs), static_cast<unsigned>(bh));
  cudaError_t e = set_smem(reinterpret_cast<const void*>(&fwd_lse_kernel), LseLayout::kAlloc);
  if (e != cudaSuccess) return e;
  return launch_dependent(fwd_lse_kernel, grid, dim3(kThreadsL), LseLayout::kAlloc, st, tq4, tk4, a);
}

// the debug build's count of skipped accesses in this file's kernels
ATTNQAT_OOB_READER(oob_read_fwd_lse)

}  // namespace attnqat
