// Attn-QAT forward, pass 1 at D = 128 (sm_103a): the natural-log LSE of two
// query tiles of one head per CTA.
//
// "Attn-QAT: 4-Bit Attention With Quantization-Aware Training" (Method, Fix 1)
// and "NVFP4 Attention QAT Backward" (cuDNN frontend docs, Overview, High-level
// wrapper): P^ = fake_nvfp4(P) is taken of the normalised probabilities, so the
// forward first needs LSE = ln sum_j exp(scale * Q^ K^T)_j of every query row;
// the second pass (fwd.cu, reading this kernel's LSE) forms P, P^, O' and O.
//
// This pass issues one small MMA per key tile (S on the block-scaled NVFP4
// MMA) and is bound by the softmax warps' exp2 work and their hand-offs. A CTA
// takes two query tiles A, B of one head and alternates between them: while
// the softmax warps reduce S_A(j), the tensor core computes S_B(j), and the
// other way round, so each MMA's latency hides behind the other tile's work.
// Both tiles read the same K tile j, loaded once.
//
// TMEM: S_A [0,128), S_B [128,256) (one buffer each: S_X(j+1) is issued once
// the softmax warps have read S_X(j)); scale factors of the MMAs in columns of
// their own: Q of tile X at 256 + 8 X + 4 ks, K of key tile j at 272 + 8 (j %
// 2) + 4 ks (4 columns per K = 64 step; lane r holds in column c the four
// scale bytes of row r + 32 c). Key tile j + 2's K scales go into slot j % 2
// once the last S of step j (which read it) is complete.
//
// Warps (18): 0-15 softmax (warp w: lane quarter w % 4, keys 32 (w / 4) .. +31
// of every tile; parts 1 and 3 write the K scale factors of K step part / 2);
// 16 TMA producer; 17 MMA issuer (and TMEM allocation).
#include "attn_common.cuh"
#include "fp4_mma.cuh"

namespace attnqat {
namespace {

constexpr int kSoftWarpsL = 16;
constexpr int kWarpTmaL = 16;
constexpr int kWarpMmaL = 17;
constexpr int kThreadsL = 18 * 32;

struct LseLayout {
  static constexpr int kStages = 4;                      // NVFP4 K tiles in flight
  static constexpr uint32_t kFp4Tile = 128 * 64;         // 128 rows x 64 bytes of E2M1 pairs
  static constexpr uint32_t kQ4 = 0;                     // tile X at kQ4 + X * kFp4Tile
  static constexpr uint32_t kK0 = 2 * kFp4Tile;          // stage s at kK0 + s * kFp4Tile
  static constexpr uint32_t kML = kK0 + kStages * kFp4Tile;   // [tile][part 1..3][row][m, l]
  static constexpr uint32_t kBar = kML + 2 * 3 * 128 * 8;
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
  uint64_t s_free[2];   // per tile: S_X(j) read (and, for a step's last S, key tile j + 2's K scales written)
  uint64_t sf_init;     // Q scales of both tiles, K scales of key tiles 0 and 1 written
  uint64_t ml_ready;
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
};

__global__ void __launch_bounds__(kThreadsL, 1)
    fwd_lse_kernel(const __grid_constant__ CUtensorMap tm_q4, const __grid_constant__ CUtensorMap tm_k4,
                   const LseArgs a) {
  using L = LseLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  LseBars& B = *reinterpret_cast<LseBars*>(smem + L::kBar);
  float* ml = reinterpret_cast<float*>(smem + L::kML);

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
    for (int x = 0; x < 2; ++x) mbar_init(&B.s_full[x], 1), mbar_init(&B.s_free[x], kSoftWarpsL * 32);
    mbar_init(&B.sf_init, 2 * 128);   // key parts 1 and 3
    mbar_init(&B.ml_ready, 3 * 128);  // key parts 1..3
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
      for (int j = 0; ok && j < n_steps; ++j) {
        const int s = j % L::kStages;
        const bool kf = mbar_try_wait(&B.k_full[s], (j / L::kStages) & 1);
        const bool doA = j < nA, doB = hasB && j < nB;
        // S_X(j) goes where S_X(j - 1) was, once the softmax warps have read it
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
    // ------------------------------------------------------------ softmax (warps 0-15)
    const uint32_t quarter = warp & 3, part = warp >> 2;
    const bool sf_writer = (part & 1u) != 0;
    const int ks = static_cast<int>(part >> 1);
    const uint32_t r = quarter * 32 + lane;
    const uint32_t lane_off = (quarter * 32u) << 16;
    const int64_t kbase = static_cast<int64_t>(bh) * a.Sk;
    const int qrow[2] = {i0 * 128 + static_cast<int>(r), i1 * 128 + static_cast<int>(r)};
    const int kend[2] = {a.causal ? min(a.Sk, qrow[0] + 1) : a.Sk, a.causal ? min(a.Sk, qrow[1] + 1) : a.Sk};
    bool ok = true;
    // K scales written at step j (key tile j + 2's), loaded one step ahead
    uint32_t sfw[4] = {0u, 0u, 0u, 0u};
    if (sf_writer) {
      uint32_t w[4];
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int qi = x == 0 ? i0 : i1;
        if (x == 0 || hasB) {
          load_scales(a.q_sf, static_cast<int64_t>(bh) * a.Sq + qi * 128, min(128, a.Sq - qi * 128), ks, w);
          tmem_st4(tmem + lane_off + L::kColSFQ + 8 * x + 4 * ks, w);
        }
      }
#pragma unroll
      for (int kt = 0; kt < 2; ++kt) {
        if (kt < n_steps) {
          load_scales(a.k_sf, kbase + kt * 128, min(128, a.Sk - kt * 128), ks, w);
          tmem_st4(tmem + lane_off + L::kColSFK + 8 * kt + 4 * ks, w);
        }
      }
      if (2 < n_steps) load_scales(a.k_sf, kbase + 2 * 128, min(128, a.Sk - 2 * 128), ks, sfw);
      tc_fence_before();
      mbar_arrive(&B.sf_init);
    }

    const float2 c22 = make_float2(a.c2, a.c2);
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};
    for (int j = 0; j < n_steps; ++j) {
      const bool doA = j < nA, doB = hasB && j < nB;
      // key tile j + 3's scales, for the write at step j + 1
      uint32_t sfw_next[4] = {0u, 0u, 0u, 0u};
      if (sf_writer && j + 3 < n_steps)
        load_scales(a.k_sf, kbase + (j + 3) * 128, min(128, a.Sk - (j + 3) * 128), ks, sfw_next);
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (x == 0 ? !doA : !doB) continue;
        if (!warp_wait(&B.s_full[x], j & 1, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + x * 128u + part * 32, v);
        // the step's last S is read: both S MMAs of key tile j are complete,
        // so key tile j + 2's K scales go into the slot they read
        const bool last = x == 1 || !doB;
        if (last && sf_writer && j + 2 < n_steps) tmem_st4(tmem + lane_off + L::kColSFK + 8 * (j & 1) + 4 * ks, sfw);
        tc_fence_before();
        mbar_arrive(&B.s_free[x]);
        const int valid = kend[x] - (j * 128 + static_cast<int>(part) * 32);
        if (valid < 32) {   // masked keys: -inf
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (k >= valid) v[k] = 0xFF800000u;
        }
        // row max of the raw S (c2 > 0: max(S) * c2 is the max of the scaled logits)
        float mq[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          float acc = fmaxf(__uint_as_float(v[16 * u]), __uint_as_float(v[16 * u + 1]));
#pragma unroll
          for (int k = 2; k < 16; k += 2)
            acc = fmax3(acc, __uint_as_float(v[16 * u + k]), __uint_as_float(v[16 * u + k + 1]));
          mq[u] = acc;
        }
        const float mx = fmaxf(m[x], fmaxf(mq[0], mq[1]) * a.c2);
        if (mx != -INFINITY) {
          const float2 nm = make_float2(-mx, -mx);
          float2 sc[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                          make_float2(0.0f, 0.0f)};
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 e = ffma2(make_float2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1])), c22, nm);
            sc[k & 3] = fadd2(sc[k & 3], make_float2(ex2(e.x), ex2(e.y)));
          }
          const float2 st = fadd2(fadd2(sc[0], sc[1]), fadd2(sc[2], sc[3]));
          l[x] = l[x] * ex2(m[x] - mx) + (st.x + st.y);
          m[x] = mx;
        }
      }
      if (!ok) break;
#pragma unroll
      for (int q = 0; q < 4; ++q) sfw[q] = sfw_next[q];
    }
    // The four key parts of each row: parts 1..3 hand (m, l) of both tiles to
    // part 0, which forms lse = ln sum exp(S * scale) and stores it.
    if (ok && part != 0) {
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        ml[((x * 3) + (part - 1)) * 256 + r * 2] = m[x];
        ml[((x * 3) + (part - 1)) * 256 + r * 2 + 1] = l[x];
      }
      mbar_arrive(&B.ml_ready);
    } else if (ok && warp_wait(&B.ml_ready, 0, ctl)) {
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (x == 1 && !hasB) break;
        const float* mlx = ml + x * 3 * 256;
        float mp[4] = {m[x], mlx[r * 2], mlx[256 + r * 2], mlx[512 + r * 2]};
        float lp[4] = {l[x], mlx[r * 2 + 1], mlx[256 + r * 2 + 1], mlx[512 + r * 2 + 1]};
        const float M = fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3]));
        float Lsum = 0.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) Lsum += mp[q] == -INFINITY ? 0.0f : lp[q] * ex2(mp[q] - M);
        if (qrow[x] < a.Sq) a.lse[(size_t)bh * a.Sq + qrow[x]] = (M + lg2(Lsum)) * kLn2;
      }
    }
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
  const dim3 grid(static_cast<unsigned>(a.n_pairs), static_cast<unsigned>(bh));
  cudaError_t e = set_smem(reinterpret_cast<const void*>(&fwd_lse_kernel), LseLayout::kAlloc);
  if (e != cudaSuccess) return e;
  fwd_lse_kernel<<<grid, kThreadsL, LseLayout::kAlloc, st>>>(tq4, tk4, a);
  return cudaGetLastError();
}

}  // namespace attnqat
