// Host-side launchers of the CUDA kernels (internal to libattnqat).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attnqat {

using bf16 = __nv_bfloat16;

// Launch `kernel` as a programmatic dependent of the previous kernel in the
// stream: its CTAs may start while that kernel finishes, and the kernel waits
// (grid_dep_wait) before it reads that kernel's results.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid, cfg.blockDim = block, cfg.dynamicSmemBytes = smem, cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr, cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

struct Problem {
  int64_t B, H, Sq, Sk, D;
  bool causal;
  float scale;
  int64_t bh() const { return B * H; }
};

// Kernel tile sizes: 128 query rows x 128 keys per step in both directions.
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;

// Default wait limit of the attention kernels' barrier waits.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;
// The limit the next launches use: kWaitTimeoutNs unless a test has set
// another through attnqat_selftest_set_wait_limit.
uint64_t wait_timeout_ns();

cudaError_t launch_fake_bf16(const bf16* x, bf16* y, int64_t rows, int64_t cols, cudaStream_t st);
cudaError_t launch_fake_f32(const float* x, float* y, int64_t rows, int64_t cols, cudaStream_t st);

// Q^, K^, V^ (and, when o_hp != nullptr, delta = rowsum(O' * dO) and a zeroed
// FP32 dQ accumulator); `zero_n` floats at `zero` are set to 0 as well (the
// backward's split-tile counters and slots). When q4 / k4 are not null, Q and
// K are also written NVFP4-encoded ((rows, D/2) bytes of E2M1 pairs and
// (rows, D/16) E4M3 scales): the forward's first pass reads them.
cudaError_t launch_prep(const Problem& p, const bf16* q, const bf16* k, const bf16* v, const bf16* o_hp,
                        const bf16* dout, bf16* qh, bf16* kh, bf16* vh, float* delta, float* dq_acc,
                        float* zero, int64_t zero_n, uint8_t* q4, uint8_t* qsf, uint8_t* k4, uint8_t* ksf,
                        cudaStream_t st);

cudaError_t launch_nvfp4_pack(const bf16* x, uint8_t* packed, uint8_t* scales, int64_t rows, int64_t cols,
                              cudaStream_t st);

cudaError_t launch_dq_convert(const Problem& p, const float* dq_acc, bf16* dq, cudaStream_t st);

// The debug build (ATTNQAT_CHECKED, checked.cuh): each file's count of the
// accesses its bounds checks skipped (added to *out; cleared when asked; the
// product build's readers add nothing), and the checks' self-test, which
// writes n + extra elements of an n-element buffer (product build:
// cudaErrorNotSupported, nothing launched).
cudaError_t oob_read_fwd_lse(unsigned long long* out, bool clear);
cudaError_t oob_read_fwd_pv(unsigned long long* out, bool clear);
cudaError_t oob_read_fwd(unsigned long long* out, bool clear);
cudaError_t oob_read_fwd_r2(unsigned long long* out, bool clear);
cudaError_t oob_read_bwd(unsigned long long* out, bool clear);
cudaError_t oob_read_infer(unsigned long long* out, bool clear);
cudaError_t oob_read_quant(unsigned long long* out, bool clear);
cudaError_t launch_bounds_selftest(float* buf, int64_t n, int64_t extra, cudaStream_t st);

// The forward; q4, qsf, k4, ksf: NVFP4 Q and K for the first pass's
// block-scaled S (D = 128; null for D = 64, which stays on BF16).
cudaError_t launch_fwd(const Problem& p, const bf16* qh, const bf16* kh, const bf16* vh, const uint8_t* q4,
                       const uint8_t* qsf, const uint8_t* k4, const uint8_t* ksf, bf16* o, bf16* o_hp, float* lse,
                       float* split_acc, uint32_t* split_cnt, uint32_t* err, cudaStream_t st);

// Pass 1 of the D = 128 forward: the natural-log LSE of every query row, two
// query tiles of a head per CTA (S on the block-scaled NVFP4 MMA).
cudaError_t launch_fwd_lse(const Problem& p, const uint8_t* q4, const uint8_t* qsf, const uint8_t* k4,
                           const uint8_t* ksf, float* lse, uint32_t* err, cudaStream_t st);

// Pass 2 of the D = 128 forward: O' = P V^ and O = fake_nvfp4(P) V^ from pass
// 1's LSE, one 128-row query tile per CTA over 64-key tiles (S on the
// block-scaled NVFP4 MMA).
// The query tiles of fwd_pv_split_plan's split share two CTAs each, which
// store their FP32 partial O', O rows in slots of split_acc (fwd_split_slot_floats
// each); the one that counts second (counters at split_cnt, zeroed) adds them.
cudaError_t launch_fwd_pv(const Problem& p, const bf16* vh, const uint8_t* q4, const uint8_t* qsf,
                          const uint8_t* k4, const uint8_t* ksf, const float* lse, bf16* o, bf16* o_hp,
                          float* split_acc, uint32_t* split_cnt, uint32_t* err, cudaStream_t st);

// How a kernel shares its work units between CTAs: the first n_full units
// (in grid order) get one CTA each, the last n_split two CTAs each (half the
// unit's loop apiece), whose FP32 partial results meet in a workspace slot.
// The backward's units are key tiles (its loop runs over query tiles), the
// forward pass 2's are query tiles (its loop runs over key tiles).
constexpr int64_t kMaxSplitTiles = 96;
struct SplitPlan {
  int64_t n_full, n_split;
};
SplitPlan bwd_split_plan(const Problem& p, int sms);
SplitPlan fwd_pv_split_plan(const Problem& p, int sms);
int device_sm_count();   // SMs of the current device (148 if it cannot be read)

// Split-tile workspace: kMaxSplitTiles counters (rounded to 64 words), then
// min(tiles, kMaxSplitTiles) slots of two FP32 [128][D] outputs ([dK, dV] in
// the backward, [O', O] in the forward).
inline int64_t split_cnt_words() { return 64 * ((kMaxSplitTiles + 63) / 64); }
inline int64_t split_slot_floats(const Problem& p) { return 2 * 128 * p.D; }
inline int64_t fwd_split_slot_floats(const Problem& p) { return 2 * 2 * 128 * p.D; }   // both ranks' [O', O]

// The forward in recipe R2 (one pass; P^ of each key tile quantized before
// normalisation) from the quantize step's Q^, K^, V^; same outputs as launch_fwd.
// Probability formats of recipe R2 (the values of attnqat_p_format).
constexpr int kPNvfp4 = 0;
constexpr int kPE5M2 = 1;
constexpr int kPE4M3 = 2;

cudaError_t launch_fwd_r2(const Problem& p, const bf16* qh, const bf16* kh, const bf16* vh, bf16* o, bf16* o_hp,
                          float* lse, int p_format, uint32_t* err, cudaStream_t st);

cudaError_t launch_bwd(const Problem& p, const bf16* qh, const bf16* kh, const bf16* vh, const bf16* dout,
                       const float* lse, const float* delta, float* dq_acc, bf16* dk, bf16* dv, float* split_acc,
                       uint32_t* split_cnt, const uint8_t* q4, const uint8_t* qsf, const uint8_t* k4,
                       const uint8_t* ksf, uint32_t* err, cudaStream_t st);

// Inference forward: O = softmax(scale * Q K^T) V with packed NVFP4 Q and K
// ((B*H, S, 64) bytes of E2M1 pairs, (B*H, S, 8) E4M3 scales) and BF16 V;
// lse may be null. D = 128 only.
cudaError_t launch_infer(const Problem& p, const uint8_t* q_fp4, const uint8_t* q_sf, const uint8_t* k_fp4,
                         const uint8_t* k_sf, const bf16* v, bf16* o, float* lse, uint32_t* err, cudaStream_t st);

cudaError_t launch_quotient_selftest(unsigned long long* out, cudaStream_t st);
cudaError_t launch_scale_selftest(unsigned long long* out, cudaStream_t st);

cudaError_t launch_wait_timeout(uint32_t* err, uint64_t timeout_ns, cudaStream_t st);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda). Returns nullptr if the driver does not provide it.
void* tensor_map_encoder();

}  // namespace attnqat
