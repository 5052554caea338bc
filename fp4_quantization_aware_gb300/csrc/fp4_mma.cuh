// Block-scaled NVFP4 tensor-core MMA (tcgen05.mma kind::mxf4nvf4, scale_vec
// 4X: one E4M3 scale per 16 E2M1 values) for a 128 x N x 128 product from
// 128-row tiles of packed NVFP4 data. Shared by the inference forward and the
// QAT forward's first pass.
//
// Measured contract (a probe against a float64 product of decoded codes):
//  - A and B are K-major with 64-byte rows (128 E2M1 values, the even element
//    in the low nibble) and the 64-byte swizzle (16-byte chunk c of row r at
//    c ^ ((r >> 1) & 3), which is what a TMA load with CU_TENSOR_MAP_SWIZZLE_64B
//    writes); one instruction covers K = 64, the next starts 32 bytes on;
//  - scale factors sit in TMEM, 4 columns per K = 64 step: lane r (the same in
//    every lane quarter) holds in column c the four scale bytes (groups
//    4 ks .. 4 ks + 3) of row r + 32 c;
//  - scale-factor column addresses must be multiples of 4 (an unaligned one
//    faults).
#pragma once
#include "attn_common.cuh"

namespace attnqat {

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

__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
      : "memory");
}

// The scale bytes one thread writes for one K = 64 step (`ks`) of a 128-row
// tile: word c = the four E4M3 scales of groups 4 ks .. 4 ks + 3 of row
// lane + 32 c (0 past `rows`).
__device__ __forceinline__ void load_scales(const uint8_t* sf, int64_t row0, int rows, int ks, uint32_t (&w)[4]) {
  const int r = static_cast<int>(lane_id());
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int row = r + 32 * c;
    w[c] = row < rows ? __ldg(reinterpret_cast<const uint32_t*>(sf + (row0 + row) * 8 + ks * 4)) : 0u;
  }
}

}  // namespace attnqat
