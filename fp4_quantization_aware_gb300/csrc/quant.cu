// HBM-bound kernels of the Attn-QAT path:
//  - fake_nvfp4 of BF16 and FP32 matrices (groups of 16 along rows),
//  - the fused preprocess: Q^, K^, V^ along D ("NVFP4 Attention QAT Backward",
//    Overview: fused Q fake-quantization/delta preprocessing and K/V
//    fake-quantization), delta = rowsum(O' * dO), and zeroing of the FP32 dQ
//    accumulator that the backward kernel adds into,
//  - the dQ FP32 -> BF16 conversion,
//  - the bounded-wait self-test.
// One thread owns one 16-value group (32 bytes of BF16): a warp moves 1 KiB
// contiguous per access, and the D/16 threads of a row reduce delta with
// shuffles. (Two or four groups per thread with every load issued first was
// slower here: twice the registers halve the CTAs resident per SM.) The dQ
// conversion gives a thread four float4s a block apart, loaded first.
#include "kernels.h"
#include "nvfp4.cuh"
#include "checked.cuh"

namespace attnqat {
namespace {

constexpr int kThreads = 256;
constexpr int kConvU = 4;   // float4 per dQ-conversion thread

__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float* f) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

__device__ __forceinline__ void load16(const bf16* p, float (&f)[16]) {
  const uint4* v = reinterpret_cast<const uint4*>(p);
  unpack8(__ldg(v), f);
  unpack8(__ldg(v + 1), f + 8);
}

__device__ __forceinline__ void store16(bf16* p, const float (&f)[16]) {
  uint4* v = reinterpret_cast<uint4*>(p);
  v[0] = pack8(f);
  v[1] = pack8(f + 8);
}

// ------------------------------------------------------------ generic quantizers
__global__ void __launch_bounds__(kThreads) fake_bf16_kernel(const bf16* x, bf16* y,
                                                             int64_t rows, int64_t cols) {
  const int64_t gpr = (cols + 15) / 16;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (g >= rows * gpr) return;
  const int64_t r = g / gpr, c0 = (g % gpr) * 16;
  const int64_t base = r * cols + c0;
  float f[16];
  if ((cols & 15) == 0) {
    load16(x + base, f);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) f[i] = (c0 + i < cols) ? __bfloat162float(x[base + i]) : 0.0f;
  }
  fake_nvfp4_16(f);
  if ((cols & 15) == 0) {
    store16(y + base, f);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (c0 + i < cols) y[base + i] = __float2bfloat16_rn(f[i]);
  }
}

__global__ void __launch_bounds__(kThreads) fake_f32_kernel(const float* x, float* y,
                                                            int64_t rows, int64_t cols) {
  const int64_t gpr = (cols + 15) / 16;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (g >= rows * gpr) return;
  const int64_t r = g / gpr, c0 = (g % gpr) * 16;
  const int64_t base = r * cols + c0;
  float f[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) f[i] = (c0 + i < cols) ? x[base + i] : 0.0f;
  fake_nvfp4_16(f);
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if (c0 + i < cols) y[base + i] = f[i];
}

// ------------------------------------------------------------ NVFP4 packing
// One thread per 16-value group of a BF16 (rows, cols) matrix, cols % 16 == 0:
// 8 bytes of E2M1 pairs to `packed` (row-major, cols/2 bytes per row) and one
// E4M3 scale byte to `scales` (cols/16 per row).
__global__ void __launch_bounds__(kThreads) nvfp4_pack_kernel(const bf16* __restrict__ x, uint8_t* __restrict__ packed,
                                                              uint8_t* __restrict__ scales, int64_t groups) {
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (g >= groups) return;
  float f[16];
  load16(x + g * 16, f);
  uint8_t b[8];
  scales[g] = nvfp4_encode_16(f, b);
  uint2 w;
  w.x = b[0] | (uint32_t)b[1] << 8 | (uint32_t)b[2] << 16 | (uint32_t)b[3] << 24;
  w.y = b[4] | (uint32_t)b[5] << 8 | (uint32_t)b[6] << 16 | (uint32_t)b[7] << 24;
  reinterpret_cast<uint2*>(packed)[g] = w;
}

// ------------------------------------------------------------ fused preprocess
struct PrepArgs {
  const bf16* src[3];   // q, k, v
  bf16* dst[3];         // q^, k^, v^ (q^, k^ may be null when packed[] is set)
  int64_t groups[3];    // 16-groups per tensor
  const bf16* o_hp;     // null: forward (no delta, no dQ accumulator)
  const bf16* dout;
  float* delta;
  float* dq_acc;
  float* zero;          // blockIdx.y == 3: zero_n16 runs of 16 floats set to 0
  int64_t zero_n16;
  uint8_t* packed[2];   // Q, K as NVFP4 (E2M1 pairs), or null
  uint8_t* scales[2];   // their E4M3 group scales
};

// blockIdx.y selects the tensor (0: Q with delta, 1: K, 2: V) or (3) the
// range to zero.
template <int D>
__global__ void __launch_bounds__(kThreads) prep_kernel(PrepArgs a) {
  constexpr int kGroupsPerRow = D / 16;
  const int t = blockIdx.y;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (t == 3) {
    if (g < a.zero_n16) {
      float4* z = reinterpret_cast<float4*>(a.zero + g * 16);
      const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
      z[0] = zero, z[1] = zero, z[2] = zero, z[3] = zero;
    }
    return;
  }
  const bool live = g < a.groups[t];
  if (blockIdx.x * static_cast<int64_t>(kThreads) >= a.groups[t]) return;   // whole block out of range
  float f[16];
  if (live) {
    load16(a.src[t] + g * 16, f);
    if (t < 2 && a.packed[t] != nullptr) {   // the same values, NVFP4-encoded
      uint8_t b[8];
      a.scales[t][g] = nvfp4_encode_16(f, b);
      uint2 w;
      w.x = b[0] | (uint32_t)b[1] << 8 | (uint32_t)b[2] << 16 | (uint32_t)b[3] << 24;
      w.y = b[4] | (uint32_t)b[5] << 8 | (uint32_t)b[6] << 16 | (uint32_t)b[7] << 24;
      reinterpret_cast<uint2*>(a.packed[t])[g] = w;
    }
    if (a.dst[t] != nullptr) {   // null: only the NVFP4 encoding is wanted
      fake_nvfp4_16(f);
      store16(a.dst[t] + g * 16, f);
    }
  }
  if (t != 0 || a.o_hp == nullptr) return;
  // delta = rowsum(O' * dO); every lane of the warp takes part in the shuffles.
  float part = 0.0f;
  if (live) {
    float o[16], d[16];
    load16(a.o_hp + g * 16, o);
    load16(a.dout + g * 16, d);
#pragma unroll
    for (int i = 0; i < 16; ++i) part = fmaf(o[i], d[i], part);
    float4* z = reinterpret_cast<float4*>(a.dq_acc + g * 16);
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    z[0] = zero, z[1] = zero, z[2] = zero, z[3] = zero;
  }
#pragma unroll
  for (int off = 1; off < kGroupsPerRow; off <<= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
  if (live && (g % kGroupsPerRow) == 0) a.delta[g / kGroupsPerRow] = part;
}

// Thread x of block b converts float4s (b kConvU + u) kThreads + x.
__global__ void __launch_bounds__(kThreads) dq_convert_kernel(const float4* __restrict__ acc, uint2* __restrict__ dq,
                                                              int64_t n4) {
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * (kThreads * kConvU) + threadIdx.x;
  float4 v[kConvU];
#pragma unroll
  for (int u = 0; u < kConvU; ++u)
    if (i0 + u * kThreads < n4) v[u] = acc[i0 + u * kThreads];
#pragma unroll
  for (int u = 0; u < kConvU; ++u)
    if (i0 + u * kThreads < n4)
      dq[i0 + u * kThreads] = make_uint2(pack_bf16x2(v[u].x, v[u].y), pack_bf16x2(v[u].z, v[u].w));
}

// The debug build's self-test of its bounds checks: thread i of n + extra
// writes element i of an n-element buffer behind the same guard as the
// kernels' accesses, so the extra threads' writes are skipped and counted.
// Only the debug build has it.
#ifdef ATTNQAT_CHECKED
__global__ void __launch_bounds__(kThreads) bounds_selftest_kernel(float* buf, int64_t n, int64_t total) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (i < total && ATTNQAT_IN_BOUNDS(i < n)) buf[i] = static_cast<float>(i);
}
#endif

// One CTA waits on a barrier that nothing arrives at; the bounded wait gives
// up after timeout_ns, records the error and the kernel returns.
__global__ void wait_timeout_kernel(uint32_t* err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    WaitCtl c{&abort_flag, err, timeout_ns};
    (void)mbar_wait(&bar, 0, c);
  }
  __syncthreads();
}

// Every E4M3 scale s (126 positive values) times every FP32 a of either sign
// with |a| / s in [1/8, 16): div_by_scale against IEEE division, bit for bit.
// out[0] counts mismatches; out[1], out[2] keep the bits of one (a, s).
constexpr int64_t kQuotPerScale = int64_t(7) << 23;   // 7 binades of FP32
constexpr int64_t kQuotTotal = 126 * kQuotPerScale * 2;

__device__ __forceinline__ float e4m3_value(int code) {   // code 1..126
  const int e = code >> 3, m = code & 7;
  return e == 0 ? m * 0x1p-9f : ldexpf(1.0f + m / 8.0f, e - 7);
}

__global__ void __launch_bounds__(kThreads) quotient_selftest_kernel(unsigned long long* out) {
  unsigned long long bad = 0;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < kQuotTotal;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t j = i >> 1;
    const int code = 1 + static_cast<int>(j / kQuotPerScale);
    const float s = e4m3_value(code);
    const uint32_t lo = __float_as_uint(s * 0.125f);
    float a = __uint_as_float(lo + static_cast<uint32_t>(j % kQuotPerScale));
    if (i & 1) a = -a;
    const float r = rcp_scale(s);
    const float got = copysignf(div_by_scale(a, s, r), a);
    const float want = __fdiv_rn(a, s);
    if (__float_as_uint(got) != __float_as_uint(want)) {
      ++bad;
      if (atomicCAS(out + 1, 0ull, static_cast<unsigned long long>(__float_as_uint(a)) | 1ull << 32) == 0ull)
        out[2] = __float_as_uint(s);
    }
  }
  if (bad) atomicAdd(out, bad);
}

// The quantizer's scale arithmetic against IEEE arithmetic, and the packing
// variant for non-negative inputs against the generic quantizer:
//  out[0] (out[3]): FP32 amax in (kZeroScaleAmax, FLT_MAX] whose div6 differs
//                   from __fdiv_rn(amax, 6) (the bits of one);
//  out[1] (out[4]): positive E4M3 scales whose rcp_scale differs from __frcp_rn;
//  out[2] (out[5]): pseudo-random groups of 16 non-negative values (zeros,
//                   and magnitudes from 2^-23 to 2, so both paths run) whose
//                   packed BF16 results differ from fake_nvfp4_16's (the index).
constexpr int64_t kNonnegGroups = int64_t(1) << 24;

__device__ __forceinline__ uint32_t mix32(uint32_t h) {   // an integer hash (xorshift-multiply rounds)
  h ^= h >> 16, h *= 0x7feb352du;
  h ^= h >> 15, h *= 0x846ca68bu;
  return h ^ (h >> 16);
}

__global__ void __launch_bounds__(kThreads) scale_selftest_kernel(unsigned long long* out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  unsigned long long bad[3] = {0, 0, 0};
  const uint32_t lo = __float_as_uint(kZeroScaleAmax) + 1u, hi = 0x7F7FFFFFu;
  for (int64_t i = t0; i <= static_cast<int64_t>(hi - lo); i += stride) {
    const float a = __uint_as_float(lo + static_cast<uint32_t>(i));
    if (__float_as_uint(div6(a)) != __float_as_uint(__fdiv_rn(a, 6.0f))) {
      ++bad[0];
      atomicCAS(out + 3, 0ull, static_cast<unsigned long long>(__float_as_uint(a)) | 1ull << 32);
    }
  }
  if (t0 < 126) {
    const float sc = e4m3_value(1 + static_cast<int>(t0));
    if (__float_as_uint(rcp_scale(sc)) != __float_as_uint(__frcp_rn(sc))) {
      ++bad[1];
      atomicCAS(out + 4, 0ull, static_cast<unsigned long long>(__float_as_uint(sc)) | 1ull << 32);
    }
  }
  for (int64_t gi = t0; gi < kNonnegGroups; gi += stride) {
    float x[16], y[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint32_t h = mix32(static_cast<uint32_t>(gi) * 16u + static_cast<uint32_t>(k) + 0x9e3779b9u);
      const float v = ldexpf(1.0f + static_cast<float>(h & 0x7FFFFFu) * 0x1p-23f, -static_cast<int>((h >> 23) % 24u));
      x[k] = (h >> 28) == 0u ? 0.0f : v;
      y[k] = x[k];
    }
    fake_nvfp4_16(y);
    uint32_t w[8];
    fake_nvfp4_16_pack_nonneg<false>(x, 1.0f, w);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (w[k] != pack_bf16x2(y[2 * k], y[2 * k + 1])) {
        ++bad[2];
        atomicCAS(out + 5, 0ull, static_cast<unsigned long long>(gi) | 1ull << 40);
        break;
      }
    }
  }
  for (int k = 0; k < 3; ++k)
    if (bad[k]) atomicAdd(out + k, bad[k]);
}

inline unsigned blocks_for(int64_t n) { return static_cast<unsigned>((n + kThreads - 1) / kThreads); }

}  // namespace

cudaError_t launch_fake_bf16(const bf16* x, bf16* y, int64_t rows, int64_t cols, cudaStream_t st) {
  const int64_t n = rows * ((cols + 15) / 16);
  if (n == 0) return cudaSuccess;
  fake_bf16_kernel<<<blocks_for(n), kThreads, 0, st>>>(x, y, rows, cols);
  return cudaGetLastError();
}

cudaError_t launch_fake_f32(const float* x, float* y, int64_t rows, int64_t cols, cudaStream_t st) {
  const int64_t n = rows * ((cols + 15) / 16);
  if (n == 0) return cudaSuccess;
  fake_f32_kernel<<<blocks_for(n), kThreads, 0, st>>>(x, y, rows, cols);
  return cudaGetLastError();
}

cudaError_t launch_prep(const Problem& p, const bf16* q, const bf16* k, const bf16* v, const bf16* o_hp,
                        const bf16* dout, bf16* qh, bf16* kh, bf16* vh, float* delta, float* dq_acc,
                        float* zero, int64_t zero_n, uint8_t* q4, uint8_t* qsf, uint8_t* k4, uint8_t* ksf,
                        cudaStream_t st) {
  if (zero_n % 16 != 0) return cudaErrorInvalidValue;
  PrepArgs a;
  a.packed[0] = q4, a.scales[0] = qsf, a.packed[1] = k4, a.scales[1] = ksf;
  a.src[0] = q, a.src[1] = k, a.src[2] = v;
  a.dst[0] = qh, a.dst[1] = kh, a.dst[2] = vh;
  a.groups[0] = p.bh() * p.Sq * (p.D / 16);
  a.groups[1] = a.groups[2] = p.bh() * p.Sk * (p.D / 16);
  a.o_hp = o_hp, a.dout = dout, a.delta = delta, a.dq_acc = dq_acc;
  a.zero = zero, a.zero_n16 = zero == nullptr ? 0 : zero_n / 16;
  int64_t most = a.groups[0] > a.groups[1] ? a.groups[0] : a.groups[1];
  if (a.zero_n16 > most) most = a.zero_n16;
  dim3 grid(blocks_for(most), a.zero_n16 > 0 ? 4 : 3);
  if (p.D == 128)
    prep_kernel<128><<<grid, kThreads, 0, st>>>(a);
  else
    prep_kernel<64><<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_nvfp4_pack(const bf16* x, uint8_t* packed, uint8_t* scales, int64_t rows, int64_t cols,
                              cudaStream_t st) {
  const int64_t groups = rows * (cols / 16);
  if (groups == 0) return cudaSuccess;
  nvfp4_pack_kernel<<<blocks_for(groups), kThreads, 0, st>>>(x, packed, scales, groups);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const Problem& p, const float* dq_acc, bf16* dq, cudaStream_t st) {
  const int64_t n4 = p.bh() * p.Sq * p.D / 4;
  if (n4 == 0) return cudaSuccess;
  dq_convert_kernel<<<blocks_for((n4 + kConvU - 1) / kConvU), kThreads, 0, st>>>(
      reinterpret_cast<const float4*>(dq_acc), reinterpret_cast<uint2*>(dq), n4);
  return cudaGetLastError();
}

cudaError_t launch_scale_selftest(unsigned long long* out, cudaStream_t st) {
  scale_selftest_kernel<<<152 * 8, kThreads, 0, st>>>(out);
  return cudaGetLastError();
}

cudaError_t launch_quotient_selftest(unsigned long long* out, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(out, 0, 3 * sizeof(unsigned long long), st);
  if (e != cudaSuccess) return e;
  quotient_selftest_kernel<<<152 * 8, kThreads, 0, st>>>(out);
  return cudaGetLastError();
}

cudaError_t launch_bounds_selftest(float* buf, int64_t n, int64_t extra, cudaStream_t st) {
#ifdef ATTNQAT_CHECKED
  const int64_t total = n + extra;
  if (n < 0 || extra < 0 || total == 0) return cudaErrorInvalidValue;
  bounds_selftest_kernel<<<blocks_for(total), kThreads, 0, st>>>(buf, n, total);
  return cudaGetLastError();
#else
  (void)buf, (void)n, (void)extra, (void)st;
  return cudaErrorNotSupported;   // no guard in the product build: never launched
#endif
}

cudaError_t launch_wait_timeout(uint32_t* err, uint64_t timeout_ns, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(err, timeout_ns);
  return cudaGetLastError();
}

// the debug build's count of skipped accesses in this file's kernels
ATTNQAT_OOB_READER(oob_read_quant)

}  // namespace attnqat
