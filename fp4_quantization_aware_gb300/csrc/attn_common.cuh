// Pieces shared by the forward and backward attention kernels.
#pragma once
#include "kernels.h"
#include "nvfp4.cuh"
#include "ptx.cuh"

namespace attnqat {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// A 128-row BF16 tile with 64-column (128-byte) blocks, 128-byte swizzled:
// row r of block b starts at b * 16 KiB + r * 128 and its 16-byte chunk c is
// stored at chunk position c ^ (r % 8). This is the layout TMA writes for a
// {64, 128} box with CU_TENSOR_MAP_SWIZZLE_128B and the layout the tcgen05
// descriptors read.
constexpr uint32_t kBlockBytes = 128 * 128;   // 128 rows x 128 bytes

__device__ __forceinline__ uint32_t sw128_chunk(uint32_t block_base, uint32_t row, uint32_t chunk) {
  return block_base + row * 128u + ((chunk ^ (row & 7u)) << 4);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Warp-uniform bounded wait. Every lane first polls the barrier word (one
// shared-memory access for the warp) and a vote decides, so a phase that is
// already complete costs no divergent branch or broadcast; otherwise lane 0
// waits, the verdict is broadcast, and the warp re-converges. Either way the
// warp-collective tcgen05 loads that follow are never reached by only part
// of a warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& c) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  uint32_t ok = 0;
  if (lane_id() == 0) ok = mbar_wait(bar, parity, c) ? 1u : 0u;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// Early, non-blocking poll of a barrier phase by lane 0 (1 if complete). Its
// verdict is consumed by warp_wait_polled later, so the poll's latency (long
// while the tensor core streams operands from shared memory) overlaps the
// work issued in between.
__device__ __forceinline__ uint32_t warp_poll(uint64_t* bar, uint32_t parity) {
  return lane_id() == 0 && mbar_try_wait(bar, parity) ? 1u : 0u;
}

// warp_wait that lane 0 skips when its earlier warp_poll saw the phase done.
__device__ __forceinline__ bool warp_wait_polled(uint32_t polled, uint64_t* bar, uint32_t parity,
                                                 const WaitCtl& c) {
  uint32_t ok = polled;
  if (lane_id() == 0 && ok == 0u) ok = mbar_wait(bar, parity, c) ? 1u : 0u;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}


// Store one thread's 64 packed BF16 values (32 words) as row `row` of the
// 64-column block at `block_base`.
__device__ __forceinline__ void store_row64(uint32_t block_base, uint32_t row, const uint32_t* w) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    st_shared_v4(sw128_chunk(block_base, row, c), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}

// Store 32 FP32 values (packed to BF16) of one row to global memory.
__device__ __forceinline__ void store_row32_bf16(bf16* dst, const uint32_t (&v)[32], float mul) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 u;
    u.x = pack_bf16x2(__uint_as_float(v[8 * c + 0]) * mul, __uint_as_float(v[8 * c + 1]) * mul);
    u.y = pack_bf16x2(__uint_as_float(v[8 * c + 2]) * mul, __uint_as_float(v[8 * c + 3]) * mul);
    u.z = pack_bf16x2(__uint_as_float(v[8 * c + 4]) * mul, __uint_as_float(v[8 * c + 5]) * mul);
    u.w = pack_bf16x2(__uint_as_float(v[8 * c + 6]) * mul, __uint_as_float(v[8 * c + 7]) * mul);
    d[c] = u;
  }
}

// ------------------------------------------------------------ host helpers
// 3-D tiled tensor map over a contiguous (outer, rows, inner) array with a
// {box_inner, box_rows, 1} box and 128-byte swizzle; rows past `rows` read as
// zero and are clipped on reduce.
bool make_tile_map(CUtensorMap* m, const void* base, bool fp32, uint64_t inner, uint64_t rows, uint64_t outer,
                   uint32_t box_inner, uint32_t box_rows);

// 3-D tiled tensor map over packed NVFP4 data, (outer, rows, 64 bytes) with
// two E2M1 values per byte (D = 128), a {64, box_rows, 1} box and the 64-byte
// swizzle; rows past `rows` read as zero.
bool make_fp4_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t outer, uint32_t box_rows);

// Opt the kernel into `bytes` of dynamic shared memory (once per kernel).
cudaError_t set_smem(const void* kernel, int bytes);

}  // namespace attnqat
