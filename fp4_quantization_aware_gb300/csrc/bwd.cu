// Attn-QAT backward main kernel (sm_103a): dK, dV and the dQ contributions.
//
// "NVFP4 Attention QAT Backward" (cuDNN frontend docs, Overview):
//   dS = P * (dO V^T - delta),  delta = rowsum(O' * dO)
//   dQ = scale * dS K^,  dK = scale * dS^T Q^,  dV = fake_nvfp4(P)^T dO
// with P recomputed from the forward's LSE ("Attn-QAT" paper summary, Fix 2)
// and fake-quantized in registers in groups of 16 keys before the P^T dO MMA.
// dQ and dK use the unquantized P (straight-through estimator).
//
// One CTA owns a 128-key tile of one (b, h) and walks the 128-row query tiles
// (causal: from the diagonal tile on, keeping the element mask on the
// diagonal; tiles past Sq/Sk are zero-filled by TMA and masked). The last
// n_split key tiles of the grid are each shared by two CTAs, one per half of
// the query tiles, so that a partial last wave of CTAs runs half as long
// (bwd_split_plan). Both add their FP32 partial dK, dV rows into a zeroed
// workspace slot; the one that counts second stores the BF16 sums.
//
// Two kernels share this structure. bwd_fp4_kernel (D = 128, described with
// its layout below) recomputes S on the block-scaled NVFP4 MMA and gives P^
// and dS a buffer each. bwd_kernel (D = 64) is the all-BF16 form:
//
// Per query tile i (all MMAs tcgen05 kind::f16, BF16 in, FP32 in TMEM):
//   S  = Q^_i K^T        (128 columns, lane = query row)
//   dP = dO_i V^T        (128 columns)
//   dV += P^T dO_i       (cols [256,256+D), lane = key)   A = P^ from smem (MN-major)
//   dQ_i = dS K^         (over dP_i once it is read)      A = dS (K-major)
//   dK += dS^T Q^_i      (cols [256+D,256+2D))            A = dS from smem (MN-major)
// S, dP and dQ share two 128-column TMEM regions R0 = [0,128), R1 = [128,256).
// Step `it` keeps dP and then dQ in R[(it+1)%2]; S of step it >= 1 is there
// too (read before dP is written), S of step 0 is in R0. So dP of a step waits
// only for the softmax warps to read that step's S, and S of the next step
// goes into the region whose dQ was drained one step earlier: the dQ drain is
// off the critical path.
// Warp roles (14 warps, both kernels):
//   0-7  softmax: P = exp2(S*c - lse2), P^ = fake_nvfp4(P) -> smem, scale*dS -> smem
//        (warp w reads TMEM lanes 32*(w%4).., columns [64*(w/4), +64) of a tile)
//   8-11 dQ drain: TMEM -> FP32 swizzled smem -> TMA reduce-add into
//        the workspace's FP32 dQ accumulator (one 32x32 box per warp and chunk)
//   12   TMA producer (lane 0)
//   13   MMA issuer (lane 0); the whole warp allocates and frees TMEM
// Shared memory (D = 64): K^ 16K, V^ 16K, Q^ x2 32K, dO 16K, P^/dS 32K,
// dQ staging 32K.
#include "attn_common.cuh"
#include "fp4_mma.cuh"
#include "checked.cuh"

namespace attnqat {
namespace {

constexpr int kThreadsBwd = 14 * 32;
constexpr int kWarpTma = 12;
constexpr int kWarpMma = 13;

template <int D>
struct BwdLayout {
  static constexpr uint32_t kTile = 128 * D * 2;
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kK + kTile;
  static constexpr uint32_t kQ0 = kV + kTile;
  static constexpr uint32_t kQ1 = kQ0 + kTile;
  static constexpr uint32_t kDO = kQ1 + kTile;
  static constexpr uint32_t kPS = kDO + kTile;          // 128 x 128 BF16
  static constexpr uint32_t kDQ = kPS + 2 * kBlockBytes; // 4 warps x 2 stages x 4 KiB
  static constexpr uint32_t kBar = kDQ + 32768;
  static constexpr uint32_t kBytes = kBar + 256;
  static constexpr uint32_t kAlloc = kBytes + 1024;      // room to align the base to 1024
  // TMEM columns
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + D;
};

// TMEM column of the region holding S of step `it`, and of dP / dQ of step `it`.
__device__ __forceinline__ uint32_t s_region(int it) { return it == 0 ? 0u : ((it + 1) & 1) * 128u; }
__device__ __forceinline__ uint32_t dp_region(int it) { return ((it + 1) & 1) * 128u; }

struct BwdBars {
  uint64_t kv_full;
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t do_full;
  uint64_t do_empty;
  uint64_t s_full;
  uint64_t s_free;
  uint64_t dp_full;
  uint64_t dq_free;
  uint64_t p_ready;
  uint64_t dv_done;
  uint64_t ds_ready;
  uint64_t buf_free;
  uint64_t dq_full;
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
  uint32_t split_order;  // split key tile: this CTA's position in the slot's count (0 or 1)
};

struct BwdArgs {
  const float* lse;
  const float* delta;
  bf16* dk;
  bf16* dv;
  int Sq, Sk;
  int n_qtiles, n_ktiles;
  int causal;
  int n_full;           // CTAs 0 .. n_full-1 own whole key tiles; then two CTAs per split tile
  float* split_acc;     // [split tile][dK, dV][128 rows][D] FP32, zeroed by the preprocess
  uint32_t* split_cnt;  // [split tile] CTAs done, zeroed by the preprocess
  float scale;
  float c2;   // scale * log2(e)
  const uint8_t* q_sf;  // NVFP4 E4M3 group scales of Q^ and K^ (B*H, S, 8): the D = 128 kernel
  const uint8_t* k_sf;
  uint32_t* err;
  uint64_t timeout_ns;
  ATTNQAT_CHECKED_ONLY(int64_t rows_q; int64_t rows_k; int64_t n_split;)   // debug build: B*H*Sq, B*H*Sk, split tiles
};

// Epilogue of the softmax warps (256 threads): warps 0-3 own dK rows, warps
// 4-7 dV rows, one key row per thread, read from the TMEM columns at `tcol`
// (this warp's lanes). A whole key tile stores BF16 rows. A split key tile
// adds its FP32 partial rows into the tile's workspace slot; after both CTAs
// have counted (device-scope fences around the count), the second one stores
// the BF16 sums. Neither waits for the other. The softmax scale of dK is
// already in dS.
template <int D>
__device__ __forceinline__ void store_dk_dv(const BwdArgs& a, uint32_t tcol, bool have, bool split_cta, int sidx,
                                            uint32_t half, int krow, int bh, uint32_t r, bool leader,
                                            uint32_t* split_order) {
  bf16* out = (half == 0 ? a.dk : a.dv) + ((size_t)bh * a.Sk + krow) * D;
  if (!split_cta) {
    if (have) {
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tcol + c * 32, v);
        if (krow < a.Sk && ATTNQAT_IN_BOUNDS(static_cast<int64_t>(bh) * a.Sk + krow < a.rows_k))
          store_row32_bf16(out + c * 32, v, 1.0f);
      }
    }
    return;
  }
  float* slot = a.split_acc + ((size_t)(sidx * 2 + half) * 128 + r) * D;
  if (have && ATTNQAT_IN_BOUNDS(sidx < a.n_split)) {
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(tcol + c * 32, v);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        red_add_v4(slot + c * 32 + 4 * q, __uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                   __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
    }
  }
  __threadfence();
  named_bar_sync(1, 256);                                  // all partial rows of this CTA are added
  if (leader) *split_order = ATTNQAT_IN_BOUNDS(sidx < a.n_split) ? atomicAdd(a.split_cnt + sidx, 1u) : 0u;
  named_bar_sync(1, 256);
  if (*reinterpret_cast<volatile uint32_t*>(split_order) == 1u) {   // the other CTA's rows are in too
    __threadfence();
    if (krow < a.Sk && ATTNQAT_IN_BOUNDS(static_cast<int64_t>(bh) * a.Sk + krow < a.rows_k)) {
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 t = __ldcg(reinterpret_cast<const float4*>(slot + c * 32 + 4 * q));
          v[4 * q] = __float_as_uint(t.x), v[4 * q + 1] = __float_as_uint(t.y);
          v[4 * q + 2] = __float_as_uint(t.z), v[4 * q + 3] = __float_as_uint(t.w);
        }
        store_row32_bf16(out + c * 32, v, 1.0f);
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreadsBwd, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dq, const BwdArgs a) {
  using L = BwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  BwdBars& B = *reinterpret_cast<BwdBars*>(smem + L::kBar);

  const int warp = warp_id();
  const int lane = lane_id();
  // 1-D grid, key tiles fastest within a head. CTA n_full + 2 t + rank works
  // on split key tile n_full + t: rank 0 takes the first half of its query
  // tiles (rounded up), rank 1 the rest.
  const int lin = static_cast<int>(blockIdx.x);
  const bool split_cta = lin >= a.n_full;
  const int sidx = split_cta ? (lin - a.n_full) >> 1 : 0;
  const int rank = split_cta ? ((lin - a.n_full) & 1) : 0;
  const int tile = split_cta ? a.n_full + sidx : lin;
  const int j = tile % a.n_ktiles;          // key tile
  const int bh = tile / a.n_ktiles;
  const int i_first = a.causal ? j : 0;     // BM == BN: the diagonal tile index equals j
  const int n_total = a.n_qtiles - i_first;
  const int n_half0 = split_cta ? (n_total + 1) / 2 : n_total;
  const int i_begin = rank == 0 ? i_first : i_first + n_half0;
  const int n_it = rank == 0 ? n_half0 : n_total - n_half0;

  if (threadIdx.x == 0) {
    B.abort_flag = 0;
    mbar_init(&B.kv_full, 1);
    for (int s = 0; s < 2; ++s) mbar_init(&B.q_full[s], 1), mbar_init(&B.q_empty[s], 1);
    mbar_init(&B.do_full, 1);
    mbar_init(&B.do_empty, 1);
    mbar_init(&B.s_full, 1);
    mbar_init(&B.s_free, 256);
    mbar_init(&B.dp_full, 1);
    mbar_init(&B.dq_free, 128);
    mbar_init(&B.p_ready, 256);
    mbar_init(&B.dv_done, 1);
    mbar_init(&B.ds_ready, 256);
    mbar_init(&B.buf_free, 1);
    mbar_init(&B.dq_full, 1);
    mbar_init(&B.drain, 1);
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&B.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B.tmem_base;
  const WaitCtl ctl{&B.abort_flag, a.err, a.timeout_ns};

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_it > 0) {
      tma_prefetch_desc(&tm_q), tma_prefetch_desc(&tm_k), tma_prefetch_desc(&tm_v), tma_prefetch_desc(&tm_do);
      int q_uses[2] = {0, 0}, do_uses = 0;
      mbar_arrive_expect_tx(&B.kv_full, 2 * L::kTile);
      for (int b = 0; b < D / 64; ++b) {
        tma_load_3d(smem + L::kK + b * kBlockBytes, &tm_k, &B.kv_full, b * 64, j * 128, bh);
        tma_load_3d(smem + L::kV + b * kBlockBytes, &tm_v, &B.kv_full, b * 64, j * 128, bh);
      }
      for (int it = 0; it < n_it; ++it) {
        const int i = i_begin + it, s = it & 1;
        if (it >= 2 && !mbar_wait(&B.q_empty[s], ((it >> 1) - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(&B.q_full[s], L::kTile);
        for (int b = 0; b < D / 64; ++b)
          tma_load_3d(smem + (s ? L::kQ1 : L::kQ0) + b * kBlockBytes, &tm_q, &B.q_full[s], b * 64, i * 128, bh);
        ++q_uses[s];
        if (it >= 1 && !mbar_wait(&B.do_empty, (it - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(&B.do_full, L::kTile);
        for (int b = 0; b < D / 64; ++b)
          tma_load_3d(smem + L::kDO + b * kBlockBytes, &tm_do, &B.do_full, b * 64, i * 128, bh);
        ++do_uses;
      }
      // Let every copy this CTA issued land before shared memory is released.
      mbar_wait_drain(&B.kv_full, 0, ctl);
      for (int s = 0; s < 2; ++s)
        if (q_uses[s]) mbar_wait_drain(&B.q_full[s], (q_uses[s] - 1) & 1, ctl);
      if (do_uses) mbar_wait_drain(&B.do_full, (do_uses - 1) & 1, ctl);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);   // S, dP
      constexpr uint32_t kIdT = idesc_bf16(128, D, true, true);       // dV, dK
      constexpr uint32_t kIdQ = idesc_bf16(128, D, false, true);      // dQ
      // Descriptors are built once and advanced by constants per k-step: the
      // issuing thread shares its SM sub-partition with two softmax warps, so
      // few instructions per MMA keep the tensor pipe fed.
      const uint64_t kmaj = sdesc_sw128(sbase, 16, 1024);             // K-major view at offset 0
      const uint64_t mnmaj = sdesc_sw128(sbase, kBlockBytes, 1024);   // MN-major view at offset 0
      // X[128 x 128] = A[128 x D] B[128 x D]^T, both K-major (K = D).
      auto mma_nt = [&](uint32_t a_off, uint32_t b_off, uint32_t col) {
        const uint64_t da = sdesc_advance(kmaj, a_off), db = sdesc_advance(kmaj, b_off);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = (kk >> 2) * kBlockBytes + (kk & 3) * 32;
          umma_bf16(tmem + col, sdesc_advance(da, o), sdesc_advance(db, o), kIdS, kk > 0);
        }
      };
      // X[128 keys x D] (+)= A^T B with A = [128 q x 128 keys] and B = [128 q x D],
      // both read MN-major (K = 128 query rows, 16 per step).
      auto mma_tn = [&](uint32_t a_off, uint32_t b_off, uint32_t col, bool acc) {
        const uint64_t da = sdesc_advance(mnmaj, a_off), db = sdesc_advance(mnmaj, b_off);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16(tmem + col, sdesc_advance(da, kk * 2048), sdesc_advance(db, kk * 2048), kIdT,
                    (acc || kk > 0) ? 1u : 0u);
      };
      // dQ[128 q x D] = dS[128 q x 128 keys] K^[128 keys x D]: A K-major, B MN-major.
      auto mma_dq = [&](uint32_t col) {
        const uint64_t da = sdesc_advance(kmaj, L::kPS), db = sdesc_advance(mnmaj, L::kK);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16(tmem + col, sdesc_advance(da, (kk >> 2) * kBlockBytes + (kk & 3) * 32),
                    sdesc_advance(db, kk * 2048), kIdQ, kk > 0);
      };

      bool ok = n_it > 0 && mbar_wait(&B.kv_full, 0, ctl) && mbar_wait(&B.q_full[0], 0, ctl);
      if (ok) {
        tc_fence_after();
        mma_nt(L::kQ0, L::kK, s_region(0));
        umma_commit(&B.s_full);
      }
      for (int it = 0; ok && it < n_it; ++it) {
        const int s = it & 1;
        if (!mbar_wait(&B.do_full, it & 1, ctl)) break;
        // dP_it goes where S_it is (it >= 1): wait until the softmax warps read S_it.
        if (it >= 1 && !mbar_wait(&B.s_free, it & 1, ctl)) break;
        tc_fence_after();
        mma_nt(L::kDO, L::kV, dp_region(it));
        umma_commit(&B.dp_full);

        if (!mbar_wait(&B.p_ready, it & 1, ctl)) break;
        tc_fence_after();
        mma_tn(L::kPS, L::kDO, L::kColDV, it > 0);
        umma_commit(&B.dv_done);
        umma_commit(&B.do_empty);

        if (it + 1 < n_it) {
          const int s1 = (it + 1) & 1;
          if (!mbar_wait(&B.q_full[s1], ((it + 1) >> 1) & 1, ctl)) break;
          // S_{it+1} goes to region it%2: after S_0 is read (it == 0), else after dQ_{it-1} is drained.
          if (it == 0 ? !mbar_wait(&B.s_free, 0, ctl) : !mbar_wait(&B.dq_free, (it - 1) & 1, ctl)) break;
          tc_fence_after();
          mma_nt(s1 ? L::kQ1 : L::kQ0, L::kK, s_region(it + 1));
          umma_commit(&B.s_full);
        }

        if (!mbar_wait(&B.ds_ready, it & 1, ctl)) break;
        tc_fence_after();
        // dQ first, so that its drain (which frees the region S of step
        // it + 2 goes to) starts one GEMM earlier
        mma_dq(dp_region(it));
        umma_commit(&B.dq_full);
        mma_tn(L::kPS, s ? L::kQ1 : L::kQ0, L::kColDK, it > 0);
        umma_commit(&B.q_empty[s]);
        umma_commit(&B.buf_free);
      }
      // Every MMA issued above completes before TMEM and smem are released.
      umma_commit(&B.drain);
      mbar_wait_drain(&B.drain, 0, ctl);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax / quant
    const uint32_t quarter = warp & 3, half = warp >> 2;
    const uint32_t r = quarter * 32 + lane;                  // row of the query tile
    const uint32_t lane_off = (quarter * 32u) << 16;
    const uint32_t ps_block = sbase + L::kPS + half * kBlockBytes;
    const int key0 = j * 128 + half * 64;                    // first key of my 64 columns
    bool ok = true;
    // LSE and delta of the row, loaded one step ahead (rows past Sq: P = 0).
    auto row_stats = [&](int it, float& lse_out, float& dlt_out) {
      const int row = (i_begin + it) * 128 + static_cast<int>(r);
      lse_out = INFINITY, dlt_out = 0.0f;
      if (it < n_it && row < a.Sq && ATTNQAT_IN_BOUNDS(static_cast<int64_t>(bh) * a.Sq + row < a.rows_q)) {
        lse_out = __ldg(a.lse + (size_t)bh * a.Sq + row);
        dlt_out = __ldg(a.delta + (size_t)bh * a.Sq + row);
      }
    };
    const float2 c22 = make_float2(a.c2, a.c2), sc2 = make_float2(a.scale, a.scale);
    float lse_next, dlt_next;
    row_stats(0, lse_next, dlt_next);
    for (int it = 0; it < n_it; ++it) {
      const int i = i_begin + it;
      const int qrow = i * 128 + r;
      const float lse2 = lse_next * kLog2e, dlt = dlt_next;
      row_stats(it + 1, lse_next, dlt_next);
      const int kend = a.causal ? min(a.Sk, qrow + 1) : a.Sk;
      const int valid = kend - key0;                         // columns [0, valid) are live keys

      if (!warp_wait(&B.s_full, it & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      float P[64];
      {
        uint32_t v[64];
        tmem_ld64(tmem + lane_off + s_region(it) + half * 64, v);
        const float2 nl = make_float2(-lse2, -lse2);
#pragma unroll
        for (int k = 0; k < 64; k += 2) {
          const float2 e = ffma2(make_float2(__uint_as_float(v[k]), __uint_as_float(v[k + 1])), c22, nl);
          P[k] = ex2(e.x), P[k + 1] = ex2(e.y);
        }
      }
      if (valid < 64) {   // masked keys: P = 0
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (k >= valid) P[k] = 0.0f;
      }
      tc_fence_before();
      mbar_arrive(&B.s_free);

      uint32_t ph[32];
#pragma unroll
      for (int g = 0; g < 4; ++g) fake_nvfp4_16_pack_nonneg<false>(P + 16 * g, 1.0f, ph + 8 * g);
      if (it > 0 && !warp_wait(&B.buf_free, (it - 1) & 1, ctl)) { ok = false; break; }
      store_row64(ps_block, r, ph);
      fence_proxy_async_smem();
      mbar_arrive(&B.p_ready);

      if (!warp_wait(&B.dp_full, it & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      uint32_t ds[32];
      {
        uint32_t v[64];
        tmem_ld64(tmem + lane_off + dp_region(it) + half * 64, v);
        // dS carries the softmax scale of dQ and dK: scale * P (dP - delta)
        // = P (scale dP - scale delta), one FMA and one multiply per pair
        const float2 nsd = make_float2(-dlt * a.scale, -dlt * a.scale);
#pragma unroll
        for (int k = 0; k < 64; k += 2) {
          const float2 d = fmul2(make_float2(P[k], P[k + 1]),
                                 ffma2(make_float2(__uint_as_float(v[k]), __uint_as_float(v[k + 1])), sc2, nsd));
          ds[k / 2] = pack_bf16x2(d.x, d.y);
        }
      }
      tc_fence_before();
      if (!warp_wait(&B.dv_done, it & 1, ctl)) { ok = false; break; }
      store_row64(ps_block, r, ds);
      fence_proxy_async_smem();
      mbar_arrive(&B.ds_ready);
    }
    const bool have = ok && n_it > 0 && warp_wait(&B.buf_free, (n_it - 1) & 1, ctl);
    if (have) tc_fence_after();
    store_dk_dv<D>(a, tmem + lane_off + (half == 0 ? L::kColDK : L::kColDV), have, split_cta, sidx, half,
                   j * 128 + static_cast<int>(r), bh, r, warp == 0 && lane == 0, &B.split_order);
  } else {
    // ------------------------------------------------------------ dQ drain (warps 8-11)
    const uint32_t quarter = warp & 3;
    const uint32_t lane_off = (quarter * 32u) << 16;
    const uint32_t stage0 = sbase + L::kDQ + quarter * 8192;   // two 4 KiB stages of 32 rows x 128 B
    uint8_t* stage0_ptr = smem + L::kDQ + quarter * 8192;
    int chunk = 0;
    for (int it = 0; it < n_it; ++it) {
      const int i = i_begin + it;
      if (!warp_wait(&B.dq_full, it & 1, ctl)) break;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c, ++chunk) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + dp_region(it) + c * 32, v);
        if (c == D / 32 - 1) {
          tc_fence_before();
          mbar_arrive(&B.dq_free);
        }
        const uint32_t b = chunk & 1;
        if (lane == 0) bulk_wait_group_read<1>();            // the reduce that last read stage b is done
        __syncwarp();
        const uint32_t st = stage0 + b * 4096;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          st_shared_v4(sw128_chunk(st, lane, k), v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(&tm_dq, stage0_ptr + b * 4096, c * 32, i * 128 + quarter * 32, bh);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}


// ---------------------------------------------------------------------------
// D = 128: S on the block-scaled NVFP4 MMA, separate P^ and dS buffers.
//
// S = Q^ K^T is recomputed from the NVFP4 encodings of Q^ and K^ (their values
// are exactly fake_nvfp4(Q), fake_nvfp4(K)) with tcgen05.mma kind::mxf4nvf4:
// 16 KiB of operands instead of 64, and a quarter of the BF16 MMA time. That
// frees one BF16 Q^ buffer (the FP4 tile feeds S, the BF16 tile only dK), so
// P^ and dS get a 32 KiB buffer each and the softmax warps no longer wait for
// the dK MMAs of the previous step before storing P^. MMA order per step:
//   [scale factors of S(it+1) written] S(it+1), [dS(it) stored] dQ(it), dK(it),
//   [S(it+1) read] dP(it+1), [P^(it+1) stored] dV(it+1)
// S(it+1) reads its scale factors from the region of dP(it): the softmax warps
// write them there once they have read dP(it), before computing dS(it), so
// S(it+1) runs while they do; dQ(it), issued after S(it+1), then overwrites
// that region (tcgen05 MMAs of one thread execute in issue order). Barrier
// polls take long while the tensor core streams operands from shared memory,
// so the waits whose phase is normally complete already (buffer releases,
// loaded tiles) are polled early and checked late, off the hand-off path.
// TMEM: R0 = [0,128), R1 = [128,256): S(t), dP(t), dQ(t) in R[t % 2]; the
// scale factors of S(t) in R[(t+1) % 2] (each 64-column half h: Q scales at
// column 56, K scales at 60, K step h); dV [256,384), dK [384,512).
// Shared memory: K^, V^, Q^, dO, P^, dS 32 KiB each, dQ staging 16 KiB,
// NVFP4 K^ and Q^ 8 KiB each = 224 KiB.
struct BwdFp4Layout {
  static constexpr uint32_t kTile = 128 * 128 * 2;
  static constexpr uint32_t kFp4Tile = 128 * 64;
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kK + kTile;
  static constexpr uint32_t kQ = kV + kTile;
  static constexpr uint32_t kDO = kQ + kTile;
  static constexpr uint32_t kP = kDO + kTile;
  static constexpr uint32_t kDS = kP + kTile;
  static constexpr uint32_t kDQ = kDS + kTile;           // 4 warps x 4 KiB
  static constexpr uint32_t kK4 = kDQ + 16384;
  static constexpr uint32_t kQ4 = kK4 + kFp4Tile;
  static constexpr uint32_t kBar = kQ4 + kFp4Tile;
  static constexpr uint32_t kBytes = kBar + 256;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 384;
  static constexpr uint32_t kColSFQ = 56;                // inside a 64-column half
  static constexpr uint32_t kColSFK = 60;
};
static_assert(BwdFp4Layout::kAlloc <= 232448, "shared memory of the D = 128 backward");

struct BwdFp4Bars {
  uint64_t kv_full, q_full, q_empty, q4_full, q4_empty, do_full, do_empty;
  uint64_t s_full, s_free, dp_full, p_ready, p_free, ds_ready, ds_free, dq_full, dq_free, sf_init, sf_ready, drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
  uint32_t split_order;
};
static_assert(sizeof(BwdFp4Bars) <= 256, "barrier block");

// Four warps share each SM sub-partition's 16K registers: at most 128 a thread.
__global__ void __maxnreg__(128)
    bwd_fp4_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_q4,
                   const __grid_constant__ CUtensorMap tm_k4, const BwdArgs a) {
  using L = BwdFp4Layout;
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  BwdFp4Bars& B = *reinterpret_cast<BwdFp4Bars*>(smem + L::kBar);

  const int warp = warp_id();
  const int lane = lane_id();
  const int lin = static_cast<int>(blockIdx.x);
  const bool split_cta = lin >= a.n_full;
  const int sidx = split_cta ? (lin - a.n_full) >> 1 : 0;
  const int rank = split_cta ? ((lin - a.n_full) & 1) : 0;
  const int tile = split_cta ? a.n_full + sidx : lin;
  const int j = tile % a.n_ktiles;
  const int bh = tile / a.n_ktiles;
  const int i_first = a.causal ? j : 0;
  const int n_total = a.n_qtiles - i_first;
  const int n_half0 = split_cta ? (n_total + 1) / 2 : n_total;
  const int i_begin = rank == 0 ? i_first : i_first + n_half0;
  const int n_it = rank == 0 ? n_half0 : n_total - n_half0;

  if (threadIdx.x == 0) {
    B.abort_flag = 0;
    mbar_init(&B.kv_full, 1), mbar_init(&B.q_full, 1), mbar_init(&B.q_empty, 1);
    mbar_init(&B.q4_full, 1), mbar_init(&B.q4_empty, 1), mbar_init(&B.do_full, 1), mbar_init(&B.do_empty, 1);
    mbar_init(&B.s_full, 1), mbar_init(&B.dp_full, 1), mbar_init(&B.p_free, 1), mbar_init(&B.ds_free, 1);
    mbar_init(&B.dq_full, 1), mbar_init(&B.drain, 1);
    mbar_init(&B.s_free, 256), mbar_init(&B.p_ready, 256), mbar_init(&B.ds_ready, 256), mbar_init(&B.sf_init, 256);
    mbar_init(&B.sf_ready, 256);
    mbar_init(&B.dq_free, 128);
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&B.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B.tmem_base;
  const WaitCtl ctl{&B.abort_flag, a.err, a.timeout_ns};

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_it > 0) {
      tma_prefetch_desc(&tm_q), tma_prefetch_desc(&tm_k), tma_prefetch_desc(&tm_v), tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_q4), tma_prefetch_desc(&tm_k4);
      mbar_arrive_expect_tx(&B.kv_full, 2 * L::kTile + L::kFp4Tile);
      for (int b = 0; b < 2; ++b) {
        tma_load_3d(smem + L::kK + b * kBlockBytes, &tm_k, &B.kv_full, b * 64, j * 128, bh);
        tma_load_3d(smem + L::kV + b * kBlockBytes, &tm_v, &B.kv_full, b * 64, j * 128, bh);
      }
      tma_load_3d(smem + L::kK4, &tm_k4, &B.kv_full, 0, j * 128, bh);
      auto load_q4 = [&](int t) {
        mbar_arrive_expect_tx(&B.q4_full, L::kFp4Tile);
        tma_load_3d(smem + L::kQ4, &tm_q4, &B.q4_full, 0, (i_begin + t) * 128, bh);
      };
      auto load_bf16 = [&](uint32_t dst, const CUtensorMap* m, uint64_t* bar, int t) {
        mbar_arrive_expect_tx(bar, L::kTile);
        for (int b = 0; b < 2; ++b) tma_load_3d(smem + dst + b * kBlockBytes, m, bar, b * 64, (i_begin + t) * 128, bh);
      };
      int n_q4 = 0, n_do = 0, n_q = 0;   // copies issued
      load_q4(0), ++n_q4;
      load_bf16(L::kDO, &tm_do, &B.do_full, 0), ++n_do;
      load_bf16(L::kQ, &tm_q, &B.q_full, 0), ++n_q;
      // In time order: S(t) done, dV(t) done, dK(t) done.
      for (int t = 0; t + 1 < n_it; ++t) {
        if (!mbar_wait(&B.q4_empty, t & 1, ctl)) break;
        load_q4(t + 1), ++n_q4;
        if (!mbar_wait(&B.do_empty, t & 1, ctl)) break;
        load_bf16(L::kDO, &tm_do, &B.do_full, t + 1), ++n_do;
        if (!mbar_wait(&B.q_empty, t & 1, ctl)) break;
        load_bf16(L::kQ, &tm_q, &B.q_full, t + 1), ++n_q;
      }
      // Let every copy this CTA issued land before shared memory is released
      // (copy u of a buffer completes phase u of its barrier).
      mbar_wait_drain(&B.kv_full, 0, ctl);
      mbar_wait_drain(&B.q4_full, (n_q4 - 1) & 1, ctl);
      mbar_wait_drain(&B.do_full, (n_do - 1) & 1, ctl);
      mbar_wait_drain(&B.q_full, (n_q - 1) & 1, ctl);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS4 = idesc_nvfp4(128, 128);                // S
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);    // dP
      constexpr uint32_t kIdT = idesc_bf16(128, D, true, true);        // dV, dK
      constexpr uint32_t kIdQ = idesc_bf16(128, D, false, true);       // dQ
      const uint64_t kmaj = sdesc_sw128(sbase, 16, 1024);
      const uint64_t mnmaj = sdesc_sw128(sbase, kBlockBytes, 1024);
      const uint64_t d4q = sdesc_sw64(sbase + L::kQ4), d4k = sdesc_sw64(sbase + L::kK4);
      // S(t) into R[t % 2] from the NVFP4 tiles, scale factors in R[(t + 1) % 2]
      auto issue_s = [&](int t) {
        const uint32_t sf = tmem + ((t + 1) & 1) * 128u;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          umma_nvfp4(tmem + (t & 1) * 128u, sdesc_advance(d4q, ks * 32), sdesc_advance(d4k, ks * 32), kIdS4,
                     sf + 64 * ks + L::kColSFQ, sf + 64 * ks + L::kColSFK, ks > 0 ? 1u : 0u);
        umma_commit(&B.s_full);
        umma_commit(&B.q4_empty);
      };
      // X[128 x 128] = A[128 x D] B[128 x D]^T, both K-major (K = D).
      auto mma_nt = [&](uint32_t a_off, uint32_t b_off, uint32_t col) {
        const uint64_t da = sdesc_advance(kmaj, a_off), db = sdesc_advance(kmaj, b_off);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = (kk >> 2) * kBlockBytes + (kk & 3) * 32;
          umma_bf16(tmem + col, sdesc_advance(da, o), sdesc_advance(db, o), kIdS, kk > 0);
        }
      };
      // X[128 keys x D] (+)= A^T B, A = [128 q x 128 keys], B = [128 q x D], both MN-major.
      auto mma_tn = [&](uint32_t a_off, uint32_t b_off, uint32_t col, bool acc) {
        const uint64_t da = sdesc_advance(mnmaj, a_off), db = sdesc_advance(mnmaj, b_off);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16(tmem + col, sdesc_advance(da, kk * 2048), sdesc_advance(db, kk * 2048), kIdT,
                    (acc || kk > 0) ? 1u : 0u);
      };
      // dQ[128 q x D] = dS[128 q x 128 keys] K^[128 keys x D]: A K-major, B MN-major.
      auto mma_dq = [&](uint32_t col) {
        const uint64_t da = sdesc_advance(kmaj, L::kDS), db = sdesc_advance(mnmaj, L::kK);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16(tmem + col, sdesc_advance(da, (kk >> 2) * kBlockBytes + (kk & 3) * 32),
                    sdesc_advance(db, kk * 2048), kIdQ, kk > 0);
      };
      // dP(t) over S(t) once it is read, then dV(t) once P^(t) is stored.
      auto issue_dp_dv = [&](int t, bool do_ready) -> bool {
        if (!mbar_wait_both(do_ready ? nullptr : &B.do_full, t & 1, &B.s_free, t & 1, ctl)) return false;
        tc_fence_after();
        mma_nt(L::kDO, L::kV, (t & 1) * 128u);
        umma_commit(&B.dp_full);
        if (!mbar_wait(&B.p_ready, t & 1, ctl)) return false;
        tc_fence_after();
        mma_tn(L::kP, L::kDO, L::kColDV, t > 0);
        umma_commit(&B.p_free);
        umma_commit(&B.do_empty);
        return true;
      };

      bool ok = n_it > 0 && mbar_wait(&B.kv_full, 0, ctl) && mbar_wait(&B.q4_full, 0, ctl) &&
                mbar_wait(&B.sf_init, 0, ctl);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        ok = issue_dp_dv(0, false);
      }
      for (int it = 0; ok && it < n_it; ++it) {
        // Inputs of S(it+1) that are ready long before its scale factors are
        // checked first (a poll takes long while the tensor core streams shared
        // memory). S(it+1) goes to the region dQ(it-1) used: after that is drained.
        // S(it+1) as soon as its scale factors are in place (the softmax warps
        // write them once they have read dP(it), before computing dS(it)).
        // The three polls are issued together, so their latencies overlap.
        if (it + 1 < n_it) {
          const bool q4r = mbar_try_wait(&B.q4_full, (it + 1) & 1);
          const bool dqr = it < 1 || mbar_try_wait(&B.dq_free, (it - 1) & 1);
          if (!mbar_wait(&B.sf_ready, it & 1, ctl)) break;
          if (!q4r && !mbar_wait(&B.q4_full, (it + 1) & 1, ctl)) break;
          if (!dqr && !mbar_wait(&B.dq_free, (it - 1) & 1, ctl)) break;
          tc_fence_after();
          issue_s(it + 1);
        }
        // the BF16 Q^ tile is needed by dK(it) only; its load follows dK(it-1)
        const bool q_ready = mbar_try_wait(&B.q_full, it & 1);
        if (!mbar_wait(&B.ds_ready, it & 1, ctl)) break;
        const bool do_ready = it + 1 < n_it && mbar_try_wait(&B.do_full, (it + 1) & 1);
        tc_fence_after();
        mma_dq((it & 1) * 128u);
        umma_commit(&B.dq_full);
        if (!q_ready && !mbar_wait(&B.q_full, it & 1, ctl)) break;
        tc_fence_after();
        mma_tn(L::kDS, L::kQ, L::kColDK, it > 0);
        umma_commit(&B.q_empty);
        umma_commit(&B.ds_free);
        if (it + 1 < n_it && !issue_dp_dv(it + 1, do_ready)) break;
      }
      // Every MMA issued above completes before TMEM and smem are released.
      umma_commit(&B.drain);
      mbar_wait_drain(&B.drain, 0, ctl);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax / quant
    const uint32_t quarter = warp & 3, half = warp >> 2;
    const uint32_t r = quarter * 32 + lane;
    const uint32_t lane_off = (quarter * 32u) << 16;
    const uint32_t p_block = sbase + L::kP + half * kBlockBytes;
    const uint32_t ds_block = sbase + L::kDS + half * kBlockBytes;
    const int key0 = j * 128 + half * 64;
    const int64_t qbase = static_cast<int64_t>(bh) * a.Sq, kbase = static_cast<int64_t>(bh) * a.Sk;
    bool ok = true;
    auto row_stats = [&](int it, float& lse_out, float& dlt_out) {
      const int row = (i_begin + it) * 128 + static_cast<int>(r);
      lse_out = INFINITY, dlt_out = 0.0f;
      if (it < n_it && row < a.Sq && ATTNQAT_IN_BOUNDS(static_cast<int64_t>(bh) * a.Sq + row < a.rows_q)) {
        lse_out = __ldg(a.lse + (size_t)bh * a.Sq + row);
        dlt_out = __ldg(a.delta + (size_t)bh * a.Sq + row);
      }
    };
    // scale factors of K step `half`: K's are fixed; Q's follow the query tile
    auto q_scales = [&](int it, uint32_t (&w)[4]) {
      const int qt = i_begin + it;
      if (it < n_it)
        load_scales(a.q_sf, qbase + qt * 128,
                    ATTNQAT_IN_BOUNDS(qbase + qt * 128 + min(128, a.Sq - qt * 128) <= a.rows_q) ? min(128, a.Sq - qt * 128) : 0,
                    static_cast<int>(half), w);
      else w[0] = w[1] = w[2] = w[3] = 0u;
    };
    uint32_t sfk[4], sfq[4];
    load_scales(a.k_sf, kbase + j * 128,
                ATTNQAT_IN_BOUNDS(kbase + j * 128 + min(128, a.Sk - j * 128) <= a.rows_k) ? min(128, a.Sk - j * 128) : 0,
                static_cast<int>(half), sfk);
    q_scales(0, sfq);
    tmem_st4(tmem + lane_off + 128 + 64 * half + L::kColSFQ, sfq);   // S(0)'s, in R1
    tmem_st4(tmem + lane_off + 128 + 64 * half + L::kColSFK, sfk);
    tc_fence_before();
    mbar_arrive(&B.sf_init);
    q_scales(1, sfq);

    const float2 c22 = make_float2(a.c2, a.c2), sc2 = make_float2(a.scale, a.scale);
    float lse_next, dlt_next;
    row_stats(0, lse_next, dlt_next);
    for (int it = 0; it < n_it; ++it) {
      const int i = i_begin + it;
      const int qrow = i * 128 + r;
      const uint32_t reg = (it & 1) * 128u + half * 64;   // this warp's columns of R[it % 2]
      const float lse2 = lse_next * kLog2e, dlt = dlt_next;
      row_stats(it + 1, lse_next, dlt_next);
      const int kend = a.causal ? min(a.Sk, qrow + 1) : a.Sk;
      const int valid = kend - key0;

      if (!warp_wait(&B.s_full, it & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      float P[64];
      uint32_t pf = 0u;   // P^ buffer free (dV(it-1) done): polled now, used before the P^ store
      {
        uint32_t v[64];
        tmem_ld64(tmem + lane_off + reg, v);
        if (it > 0) pf = warp_poll(&B.p_free, (it - 1) & 1);
        const float2 nl = make_float2(-lse2, -lse2);
#pragma unroll
        for (int k = 0; k < 64; k += 2) {
          const float2 e = ffma2(make_float2(__uint_as_float(v[k]), __uint_as_float(v[k + 1])), c22, nl);
          P[k] = ex2(e.x), P[k + 1] = ex2(e.y);
        }
      }
      if (valid < 64) {
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (k >= valid) P[k] = 0.0f;
      }
      tc_fence_before();
      mbar_arrive(&B.s_free);

      uint32_t ph[32];
#pragma unroll
      for (int g = 0; g < 4; ++g) fake_nvfp4_16_pack_nonneg<false>(P + 16 * g, 1.0f, ph + 8 * g);
      if (it > 0 && !warp_wait_polled(pf, &B.p_free, (it - 1) & 1, ctl)) { ok = false; break; }
      store_row64(p_block, r, ph);
      fence_proxy_async_smem();
      mbar_arrive(&B.p_ready);

      if (!warp_wait(&B.dp_full, it & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      uint32_t ds[32];
      uint32_t df = 0u;   // dS buffer free (dK(it-1) done): polled now, used before the dS store
      {
        // dP in two 32-column loads, so that fewer values are live at once
        const float2 nsd = make_float2(-dlt * a.scale, -dlt * a.scale);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + reg + 32 * h, v);
          if (h == 0 && it > 0) df = warp_poll(&B.ds_free, (it - 1) & 1);
          if (h == 1 && it + 1 < n_it) {
            // dP(it) is read: S(it+1)'s scale factors go over its last 8
            // columns of this half (Q's then K's, adjacent: one store, one
            // wait), and S(it+1) may start
            static_assert(L::kColSFK == L::kColSFQ + 4, "Q and K scale columns adjacent");
            const uint32_t sf8[8] = {sfq[0], sfq[1], sfq[2], sfq[3], sfk[0], sfk[1], sfk[2], sfk[3]};
            tmem_st8_nowait(tmem + lane_off + reg + L::kColSFQ, sf8);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&B.sf_ready);
            q_scales(it + 2, sfq);
          }
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const float2 d = fmul2(make_float2(P[32 * h + k], P[32 * h + k + 1]),
                                   ffma2(make_float2(__uint_as_float(v[k]), __uint_as_float(v[k + 1])), sc2, nsd));
            ds[16 * h + k / 2] = pack_bf16x2(d.x, d.y);
          }
        }
      }
      if (it > 0 && !warp_wait_polled(df, &B.ds_free, (it - 1) & 1, ctl)) { ok = false; break; }
      store_row64(ds_block, r, ds);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&B.ds_ready);
    }
    const bool have = ok && n_it > 0 && warp_wait(&B.ds_free, (n_it - 1) & 1, ctl);
    if (have) tc_fence_after();
    store_dk_dv<D>(a, tmem + lane_off + (half == 0 ? L::kColDK : L::kColDV), have, split_cta, sidx, half,
                   j * 128 + static_cast<int>(r), bh, r, warp == 0 && lane == 0, &B.split_order);
  } else {
    // ------------------------------------------------------------ dQ drain (warps 8-11)
    const uint32_t quarter = warp & 3;
    const uint32_t lane_off = (quarter * 32u) << 16;
    const uint32_t stage = sbase + L::kDQ + quarter * 4096;   // 32 rows x 128 B
    uint8_t* stage_ptr = smem + L::kDQ + quarter * 4096;
    for (int it = 0; it < n_it; ++it) {
      const int i = i_begin + it;
      if (!warp_wait(&B.dq_full, it & 1, ctl)) break;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + (it & 1) * 128u + c * 32, v);
        if (c == D / 32 - 1) {
          tc_fence_before();
          mbar_arrive(&B.dq_free);
        }
        if (lane == 0) bulk_wait_group_read<0>();            // the previous reduce has read the stage
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          st_shared_v4(sw128_chunk(stage, lane, k), v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(&tm_dq, stage_ptr, c * 32, i * 128 + quarter * 32, bh);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_bwd(const Problem& p, const bf16* qh, const bf16* kh, const bf16* vh, const bf16* dout,
                       const float* lse, const float* delta, float* dq_acc, bf16* dk, bf16* dv, float* split_acc,
                       uint32_t* split_cnt, const uint8_t* q4, const uint8_t* qsf, const uint8_t* k4,
                       const uint8_t* ksf, uint32_t* err, cudaStream_t st) {
  CUtensorMap tq, tk, tv, tdo, tdq;
  const uint64_t bh = p.bh();
  if (!make_tile_map(&tq, qh, false, p.D, p.Sq, bh, 64, 128) || !make_tile_map(&tk, kh, false, p.D, p.Sk, bh, 64, 128) ||
      !make_tile_map(&tv, vh, false, p.D, p.Sk, bh, 64, 128) || !make_tile_map(&tdo, dout, false, p.D, p.Sq, bh, 64, 128) ||
      !make_tile_map(&tdq, dq_acc, true, p.D, p.Sq, bh, 32, 32))
    return cudaErrorInvalidValue;
  BwdArgs a;
  a.lse = lse, a.delta = delta, a.dk = dk, a.dv = dv;
  a.Sq = static_cast<int>(p.Sq), a.Sk = static_cast<int>(p.Sk);
  a.n_qtiles = static_cast<int>((p.Sq + kBlockM - 1) / kBlockM);
  a.n_ktiles = static_cast<int>((p.Sk + kBlockN - 1) / kBlockN);
  a.causal = p.causal ? 1 : 0;
  a.scale = p.scale, a.c2 = p.scale * kLog2e;
  a.q_sf = qsf, a.k_sf = ksf;
  a.err = err, a.timeout_ns = wait_timeout_ns();
  const SplitPlan plan = bwd_split_plan(p, device_sm_count());
  a.n_full = static_cast<int>(plan.n_full);
  a.split_acc = split_acc, a.split_cnt = split_cnt;
  ATTNQAT_CHECKED_ONLY(a.rows_q = static_cast<int64_t>(p.bh()) * p.Sq; a.rows_k = static_cast<int64_t>(p.bh()) * p.Sk;
                       a.n_split = plan.n_split;)
  const int64_t blocks = plan.n_full + 2 * plan.n_split;
  if (blocks > 0x7fffffff || (plan.n_split > 0 && (split_acc == nullptr || split_cnt == nullptr)))
    return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(blocks));
  if (p.D == 128) {   // NVFP4 S: the packed Q^, K^ and their scales are required
    CUtensorMap tq4, tk4;
    if (q4 == nullptr || qsf == nullptr || k4 == nullptr || ksf == nullptr || !make_fp4_map(&tq4, q4, p.Sq, bh, 128) ||
        !make_fp4_map(&tk4, k4, p.Sk, bh, 128))
      return cudaErrorInvalidValue;
    cudaError_t e = set_smem(reinterpret_cast<const void*>(&bwd_fp4_kernel), BwdFp4Layout::kAlloc);
    if (e != cudaSuccess) return e;
    bwd_fp4_kernel<<<grid, kThreadsBwd, BwdFp4Layout::kAlloc, st>>>(tq, tk, tv, tdo, tdq, tq4, tk4, a);
  } else {
    cudaError_t e = set_smem(reinterpret_cast<const void*>(&bwd_kernel<64>), BwdLayout<64>::kAlloc);
    if (e != cudaSuccess) return e;
    bwd_kernel<64><<<grid, kThreadsBwd, BwdLayout<64>::kAlloc, st>>>(tq, tk, tv, tdo, tdq, a);
  }
  return cudaGetLastError();
}

int device_sm_count() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 148;
  if (dev >= 0 && dev < 64) cache[dev] = sms;
  return sms;
}

// Key tiles are uniform in a non-causal problem: with q full waves of
// CTAs and r tiles left over, splitting those r tiles in two lets the last
// wave run 2r half-length CTAs (when 2r <= SMs) instead of r full ones. A
// problem whose every tile split fits one wave is split throughout.
SplitPlan bwd_split_plan(const Problem& p, int sms) {
  const int64_t nq = (p.Sq + kBlockM - 1) / kBlockM;
  const int64_t tiles = ((p.Sk + kBlockN - 1) / kBlockN) * p.bh();
  int64_t s = 0;
  if (nq >= 2 && sms > 0) {
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
ATTNQAT_OOB_READER(oob_read_bwd)

}  // namespace attnqat
