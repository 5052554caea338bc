/*
 * attnqat: Attn-QAT (scaled dot-product attention trained with NVFP4 fake
 * quantization) for GB300 (sm_103a) behind a C ABI.
 *
 * The method ("NVFP4 Attention QAT Backward", cuDNN frontend docs, Overview;
 * "Attn-QAT: 4-Bit Attention With Quantization-Aware Training", Method):
 *
 *   Q^, K^, V^ = fake_nvfp4(Q), fake_nvfp4(K), fake_nvfp4(V)  (16-groups along D)
 *   P   = softmax(softmax_scale * Q^ K^T)                     (FP32)
 *   O   = fake_nvfp4(P) V^                                    (16-groups of keys)
 *   O'  = P V^                       (high-precision auxiliary output, "Fix 1")
 *   LSE = natural-log log-sum-exp of the scaled logits
 *   dS  = P * (dO V^T - rowsum(O' * dO))
 *   dQ  = softmax_scale * dS K^,  dK = softmax_scale * dS^T Q^
 *   dV  = fake_nvfp4(P)^T dO         (P recomputed from LSE, "Fix 2")
 *
 * fake_nvfp4 of a group of 16 values: s = RNE_E4M3(amax / 6) with IEEE
 * division (saturating to 448); y = RNE_E2M1(x / s) * s with IEEE division
 * (saturating to 6); y = +-0 when s == 0.
 *
 * Conventions shared by every entry point:
 *  - Tensors are device pointers to contiguous BHSD storage: Q, O, O', dO, dQ
 *    are (B, H, Sq, D); K, V, dK, dV are (B, H, Sk, D); LSE is (B, H, Sq).
 *    Activations are BF16 (passed as void*), LSE is FP32. Every pointer must
 *    be 16-byte aligned and all of them must live on the current device.
 *  - The caller owns every buffer. No entry point allocates device memory;
 *    scratch space comes from the caller's workspace.
 *  - `stream` is a cudaStream_t (NULL is the legacy default stream). All work
 *    is enqueued on it in order; nothing synchronizes the host.
 *  - Argument, shape, alignment and workspace checks run on the host before
 *    any launch and return an error without enqueuing anything.
 *  - Every wait inside a kernel is bounded. A wait that runs out of time makes
 *    the kernel return early and records ATTNQAT_ERR_TIMEOUT in a device
 *    error word, read by attnqat_device_status().
 */
#ifndef ATTNQAT_H_
#define ATTNQAT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum attnqat_status {
  ATTNQAT_OK = 0,
  ATTNQAT_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad scale */
  ATTNQAT_ERR_UNSUPPORTED = 2,   /* D not in {64, 128}; causal with Sq != Sk */
  ATTNQAT_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned */
  ATTNQAT_ERR_WORKSPACE = 4,     /* workspace null, misaligned or too small */
  ATTNQAT_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed */
  ATTNQAT_ERR_TIMEOUT = 6        /* a bounded device wait ran out of time */
} attnqat_status;

/* One attention problem. MHA only (equal query and key/value head counts,
 * cuDNN page "Current support and limitations"). is_causal drops keys j > i
 * and needs Sq == Sk; softmax_scale must be finite and > 0 (the pages'
 * default is 1/sqrt(128)) and must be the same in the forward and backward. */
typedef struct attnqat_problem {
  int64_t B, H, Sq, Sk, D;
  int32_t is_causal;
  float softmax_scale;
} attnqat_problem;

/* Library version (major * 10000 + minor * 100 + patch). */
int attnqat_version(void);

/* A static, human-readable name of a status code. */
const char* attnqat_status_string(int status);

/* Detail of the last error returned on the calling thread (empty if none). */
const char* attnqat_last_error_message(void);

/* Host-only check of a problem: ATTNQAT_OK if the kernels support it.
 * B, H >= 1; Sq, Sk >= 1 and below 2^31; D in {64, 128}; causal needs
 * Sq == Sk. Launches nothing and needs no GPU. */
attnqat_status attnqat_check_support(const attnqat_problem* p);

/* Workspace bytes for attnqat_fwd / attnqat_bwd (0 if the problem is not
 * supported). Forward: Q^, K^, V^ (BF16). Backward: Q^, K^, V^, delta (FP32,
 * B*H*Sq), an FP32 dQ accumulator (B*H*Sq*D), and FP32 partial-dK/dV slots
 * for up to 96 key tiles that the backward shares between two CTAs (the
 * preprocess step zeroes what a call uses). At D = 128 both add the NVFP4
 * encodings of Q^ and K^ (packed E2M1 pairs and E4M3 scales, 72 bytes per
 * row) that the S = Q^ K^T MMAs read. */
size_t attnqat_fwd_workspace_bytes(const attnqat_problem* p);
size_t attnqat_bwd_workspace_bytes(const attnqat_problem* p);

/* fake_nvfp4 of a row-major (rows, cols) BF16 matrix, groups of 16 along the
 * contiguous axis starting at column 0 (a ragged last group is padded with
 * zeros). x and y are device pointers (16-byte aligned) and may alias.
 * Source: cuDNN page, Overview (the Q/K/V quantizer). */
attnqat_status attnqat_fake_nvfp4(const void* x_bf16, void* y_bf16, int64_t rows, int64_t cols, void* stream);

/* The same quantizer on FP32 input and output: the exact device routine the
 * attention kernels apply to the probabilities P (groups of 16 keys). */
attnqat_status attnqat_fake_nvfp4_f32(const float* x, float* y, int64_t rows, int64_t cols, void* stream);

/* Forward. Inputs q, k, v (BF16). Outputs o = fake_nvfp4(P) V^, o_hp = P V^
 * (both BF16, shape of q) and lse (FP32, natural log). Needs a workspace of
 * attnqat_fwd_workspace_bytes(p) bytes, 256-byte aligned. Same outputs as
 * attnqat_quantize_qkv followed by attnqat_fwd_main; at D = 128 its quantize
 * step writes only what the forward kernel reads (the NVFP4 Q, K and the
 * BF16 V^), not the BF16 Q^, K^. */
attnqat_status attnqat_fwd(const attnqat_problem* p, const void* q, const void* k, const void* v, void* o,
                           void* o_hp, float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* Backward. Inputs dO, q, k, v, o_hp (the matching forward's O' = P V^, not
 * O; any other auxiliary gives wrong gradients) and lse (the matching
 * forward's FP32 natural-log LSE). Outputs dq, dk, dv (BF16). Needs a
 * workspace of attnqat_bwd_workspace_bytes(p) bytes, 256-byte aligned.
 * Equivalent to attnqat_bwd_preprocess, attnqat_bwd_main, attnqat_bwd_dq_convert. */
attnqat_status attnqat_bwd(const attnqat_problem* p, const void* dout, const void* q, const void* k,
                           const void* v, const void* o_hp, const float* lse, void* dq, void* dk, void* dv,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Backward with every input and output in host memory (page-locked, so that
 * the copies overlap the kernels): the backward of the cuDNN page (Overview),
 * computed by the same kernels as attnqat_bwd on groups of heads. The B*H
 * heads are split into contiguous groups of n = ceil(B*H / chunks) heads
 * (chunks clamped to 1..B*H), except the first and the last groups, which
 * hold about n / 2 (the transfers bound this call: a short first group
 * starts the kernels early, a short last group leaves less after the last
 * copy in). While group c runs on `stream`, group c + 1 is copied in and
 * group c - 1 out on two copy streams the library creates once per device.
 * Arguments as for
 * attnqat_bwd, with dout, q, k, v, o_hp, lse, dq, dk, dv host pointers in the
 * same BHSD layouts. The device workspace of
 * attnqat_bwd_host_workspace_bytes(p, chunks) bytes (256-byte aligned) holds
 * two groups' inputs, outputs and backward workspace. The call returns once
 * everything is enqueued; `stream` then waits for the last copy out, so
 * synchronizing it makes dq, dk, dv readable. The host buffers must stay
 * valid and unmodified until then. Results equal attnqat_bwd's up to the order
 * of the FP32 additions of dQ and of split key tiles' partial dK, dV. Errors
 * as attnqat_bwd; a failing CUDA call returns ATTNQAT_ERR_CUDA with part of
 * the work enqueued. */
size_t attnqat_bwd_host_workspace_bytes(const attnqat_problem* p, int chunks);
attnqat_status attnqat_bwd_host(const attnqat_problem* p, const void* dout, const void* q, const void* k,
                                const void* v, const void* o_hp, const float* lse, void* dq, void* dk, void* dv,
                                int chunks, void* workspace, size_t workspace_bytes, void* stream);

/* ---- the steps of attnqat_fwd / attnqat_bwd, for callers that time or
 * schedule them separately. Each takes the same workspace. ---- */

/* Forward step 1: Q^, K^, V^ into the workspace (HBM-bound). At D = 128 it
 * also clears the counters with which step 2 combines the partial outputs of
 * its split query tiles, so each attnqat_fwd_main needs an
 * attnqat_quantize_qkv on the same workspace before it. */
attnqat_status attnqat_quantize_qkv(const attnqat_problem* p, const void* q, const void* k, const void* v,
                                    void* workspace, size_t workspace_bytes, void* stream);

/* Forward step 2: the attention kernel on the workspace's Q^, K^, V^ (pass 1:
 * LSE; pass 2: P, fake_nvfp4(P), O' and O). At D = 128 it reads Q^ and K^ in
 * their NVFP4 encoding only. */
attnqat_status attnqat_fwd_main(const attnqat_problem* p, void* o, void* o_hp, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream);

/* ---- forward recipe R2 ---- */

/* The forward in recipe R2: one pass over the key tiles with an online
 * softmax that fake-quantizes each 128-key tile's unnormalised probabilities
 * (the FastVideo pull request "Add Attn-QAT training Triton kernels", review
 * of its FP8-P branch: the row statistic is summed from the unquantized P).
 * Per query row and key tile j: m_j = running max of the scaled logits,
 * P^_j = fake_nvfp4(exp(S_j - m_j)) in groups of 16 keys, and
 * O = sum_j exp(m_j - m) P^_j V^_j / l. O' = P V^ and the natural-log LSE are
 * the standard forward's (so attnqat_bwd applies unchanged); only O differs.
 * Same arguments, workspace and outputs as attnqat_fwd. */
attnqat_status attnqat_fwd_r2(const attnqat_problem* p, const void* q, const void* k, const void* v, void* o,
                              void* o_hp, float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* Step 2 of attnqat_fwd_r2, after attnqat_quantize_qkv. */
attnqat_status attnqat_fwd_main_r2(const attnqat_problem* p, void* o, void* o_hp, float* lse, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* Probability quantizers of recipe R2: NVFP4 (fake_nvfp4 in 16-key groups,
 * attnqat_fwd_r2), or the FP8-P variant of the same review ("when dtype is
 * tl.float8e5 (FP8) ..."): every element of a tile's unnormalised P cast to
 * FP8, round to nearest even, E5M2 (Triton's tl.float8e5, the type the review
 * names) or E4M3FN. */
typedef enum { ATTNQAT_P_NVFP4 = 0, ATTNQAT_P_FP8_E5M2 = 1, ATTNQAT_P_FP8_E4M3 = 2 } attnqat_p_format;

/* attnqat_fwd_r2 with the probability quantizer p_format (an
 * attnqat_p_format; any other value returns ATTNQAT_ERR_INVALID_ARG before
 * any launch). In the FP8 formats P^_j = fp8(exp(S_j - m_j)) element by
 * element; l still sums the unquantized P, and O', LSE are unchanged. Same
 * arguments, workspace and outputs as attnqat_fwd. */
attnqat_status attnqat_fwd_r2_p(const attnqat_problem* p, const void* q, const void* k, const void* v, void* o,
                                void* o_hp, float* lse, int p_format, void* workspace, size_t workspace_bytes,
                                void* stream);

/* Step 2 of attnqat_fwd_r2_p, after attnqat_quantize_qkv. */
attnqat_status attnqat_fwd_main_r2_p(const attnqat_problem* p, void* o, void* o_hp, float* lse, int p_format,
                                     void* workspace, size_t workspace_bytes, void* stream);

/* Backward step 1: Q^, K^, V^ (and at D = 128 their NVFP4 encodings),
 * delta = rowsum(O' * dO) into the workspace, the FP32 dQ accumulator and the
 * split-tile slots zeroed (one HBM-bound kernel). */
attnqat_status attnqat_bwd_preprocess(const attnqat_problem* p, const void* dout, const void* q, const void* k,
                                      const void* v, const void* o_hp, void* workspace, size_t workspace_bytes,
                                      void* stream);

/* Backward step 2: the dK/dV kernel (one CTA per 128-key tile; when the
 * tiles leave a partial last wave on the GPU, the last tiles get two CTAs
 * each, half the query tiles apiece), which also adds every tile's dQ
 * contribution into the workspace's FP32 accumulator. */
attnqat_status attnqat_bwd_main(const attnqat_problem* p, const void* dout, const float* lse, void* dk, void* dv,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Backward step 3: dQ (BF16) from the FP32 accumulator. */
attnqat_status attnqat_bwd_dq_convert(const attnqat_problem* p, void* dq, void* workspace, size_t workspace_bytes,
                                      void* stream);

/* The backward for callers that cannot allocate device memory (code running
 * where cudaMalloc is not allowed or not possible, or a fixed memory budget
 * with no allocator hook). The paper has no counterpart: it exists only so
 * that such callers need no workspace. It computes exactly what attnqat_bwd
 * computes, with the scratch space in a 32 MiB static device array that the
 * library declares; problems whose attnqat_bwd_workspace_bytes() exceed
 * 32 MiB return ATTNQAT_ERR_WORKSPACE. It calls no allocator. Every GPU that
 * loads the library's module holds the array until exit; all calls share it
 * and it keeps the last call's contents (each call's preprocess clears the
 * parts that must start at zero), so calls that overlap on the GPU race.
 * The first call on a device looks up the array's address. Under CUDA's lazy
 * module loading (the default) that lookup is also what loads the module and
 * reserves the 32 MiB on that device, so the first call can fail with
 * ATTNQAT_ERR_CUDA when the device is full: make it at start-up, before any
 * stream capture and before a memory budget applies. The address is cached
 * per device for the life of the CUDA context: do not reset the device
 * (cudaDeviceReset) between calls. */
attnqat_status attnqat_bwd_noalloc(const attnqat_problem* p, const void* dout, const void* q, const void* k,
                                   const void* v, const void* o_hp, const float* lse, void* dq, void* dk, void* dv,
                                   void* stream);

/* ---- NVFP4 inference forward ("Attn-QAT: 4-Bit Attention With
 * Quantization-Aware Training", Results: block-scaled NVFP4 on the QK MMA,
 * BF16 on PV; FastVideo attn_qat_infer page: Q and K packed to NVFP4 with
 * per-16 E4M3 scale factors, fa4_pv_mode "bf16"). ---- */

/* Real NVFP4 encoding of a row-major (rows, cols) BF16 matrix, groups of 16
 * along the contiguous axis; cols must be a multiple of 16. Writes `packed`
 * (rows * cols / 2 bytes: byte j of a row holds elements 2j (low nibble) and
 * 2j + 1 (high nibble) as E2M1 codes, sign in bit 3) and `scales` (rows *
 * cols / 16 E4M3FN bytes, one per group in order). The decoded values are
 * bit for bit those of attnqat_fake_nvfp4. A group whose scale rounds to 0
 * gets scale byte 0 and codes 0 or 8 (the element's sign). Device pointers,
 * 16-byte aligned; the caller owns them. */
attnqat_status attnqat_nvfp4_pack(const void* x_bf16, void* packed, void* scales, int64_t rows, int64_t cols,
                                  void* stream);

/* Workspace bytes of attnqat_infer_fwd (0 if the problem is not supported by
 * it): packed Q and K and their scale factors, each 256-byte aligned. */
size_t attnqat_infer_fwd_workspace_bytes(const attnqat_problem* p);

/* Inference forward on pre-packed Q and K: O = softmax(softmax_scale *
 * Q^ K^T) V with Q^, K^ the values q_fp4 / k_fp4 encode (attnqat_nvfp4_pack
 * layout over (B*H*S, 128): q_fp4 (B, H, Sq, 64) bytes, q_sf (B, H, Sq, 8);
 * k_fp4, k_sf likewise over Sk) and V BF16 (B, H, Sk, D) unquantized. Writes
 * o (BF16, (B, H, Sq, D)) and, when lse is not NULL, the natural-log LSE
 * (FP32, (B, H, Sq)). D must be 128 (ATTNQAT_ERR_UNSUPPORTED otherwise). No
 * probability quantization and no O': it serves inference only. */
attnqat_status attnqat_infer_fwd_packed(const attnqat_problem* p, const void* q_fp4, const void* q_sf,
                                        const void* k_fp4, const void* k_sf, const void* v, void* o, float* lse,
                                        void* stream);

/* Inference forward from BF16 q, k, v: packs Q and K into the workspace
 * (attnqat_nvfp4_pack) and runs attnqat_infer_fwd_packed. Needs
 * attnqat_infer_fwd_workspace_bytes(p) bytes of workspace. */
attnqat_status attnqat_infer_fwd(const attnqat_problem* p, const void* q, const void* k, const void* v, void* o,
                                 float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* ---- device status ---- */

/* Synchronizes the current device, then returns ATTNQAT_OK or the first
 * device-side error recorded since the last clear (ATTNQAT_ERR_TIMEOUT), or
 * ATTNQAT_ERR_CUDA if the synchronization failed. clear != 0 resets it. */
attnqat_status attnqat_device_status(int clear);

/* Checks the quantizer's division-free quotient against IEEE FP32 division,
 * bit for bit, for every positive E4M3 scale s and every FP32 a of either
 * sign with |a| / s in [1/8, 16) (about 7.4e9 pairs; below 1/8 the E2M1 code
 * is 0 and above 16 it saturates either way). `out` is a device pointer to 3
 * unsigned 64-bit words, written on `stream`: the mismatch count, then the
 * bits of one mismatching a (| 1 << 32) and s. Supports the "precise
 * division" requirement of the cuDNN page (Overview). */
attnqat_status attnqat_selftest_quotient(unsigned long long* out, void* stream);

/* Checks the quantizer's scale arithmetic and its packing variant for
 * non-negative inputs, bit for bit: (0) the FMA-corrected amax / 6 against IEEE
 * FP32 division for every FP32 amax above the zero-scale bound 6 * 2^-10;
 * (1) the refined reciprocal against IEEE reciprocal for all 126 positive
 * E4M3 scales; (2) the non-negative variant (the one the attention kernels
 * apply to P) against the generic quantizer on 2^24 pseudo-random groups. `out`
 * is a device pointer to 6 unsigned 64-bit words, written on `stream` and
 * expected zero-initialised: the three mismatch counts, then an example of
 * each (bits of amax, bits of the scale, group index; bit 32 or 40 set). */
attnqat_status attnqat_selftest_scale(unsigned long long* out, void* stream);

/* Launches one CTA that waits on a barrier that nothing arrives at, with a
 * limit of timeout_ns nanoseconds; it then records ATTNQAT_ERR_TIMEOUT in the
 * device error word and returns. Exercises the bounded-wait path without
 * faulting or hanging the GPU. */
attnqat_status attnqat_selftest_wait_timeout(uint64_t timeout_ns, void* stream);

/* The default limit, in nanoseconds, of the attention kernels' barrier waits. */
#define ATTNQAT_DEFAULT_WAIT_LIMIT_NS 2000000000ull

/* Test export: sets the limit, in nanoseconds, of the barrier waits of every
 * attention kernel launched afterwards by this process (above 10 s returns
 * ATTNQAT_ERR_INVALID_ARG; ATTNQAT_DEFAULT_WAIT_LIMIT_NS restores the
 * default). A limit of 0 makes every wait give up at the first poll that
 * finds its phase incomplete: the kernel's CTAs then record
 * ATTNQAT_ERR_TIMEOUT in the device error word (attnqat_device_status) and
 * return, which exercises the abort path of the real kernels. (A poll may
 * suspend until its phase completes, so a short nonzero limit does not
 * reliably make a wait run out.) The waits at a CTA's teardown, which let its
 * own copies and MMAs land before its shared memory and TMEM are released,
 * keep their 2 s limit. Outputs of an aborted call are undefined. Not for
 * use concurrently with other calls. */
attnqat_status attnqat_selftest_set_wait_limit(uint64_t timeout_ns);

/* ---- debug build (libattnqat_checked.so, compiled with ATTNQAT_CHECKED) ----
 * Every plain global load and store of the attention kernels (TMA copies are
 * clipped by their tensor maps) checks that its element index lies inside the
 * extent of the buffer it addresses; an access that would not is skipped and
 * counted in device counters, so a bad index shows up as a count, never as a
 * fault. No page defines these; they stand in for a memory checker. */

/* 1 in the debug build, 0 in the product build (libattnqat.so). */
int attnqat_checked_build(void);

/* The number of accesses the debug build's checks skipped since the last
 * clear (synchronizes the device; clear != 0 resets the counters). The product
 * build returns ATTNQAT_ERR_UNSUPPORTED. */
attnqat_status attnqat_debug_oob_count(unsigned long long* count, int clear);

/* Self-test of the checks: n + extra threads each write one element of the
 * n-element device buffer buf (float) behind the same guard, so the last
 * `extra` writes are skipped and counted (read with attnqat_debug_oob_count).
 * The product build returns ATTNQAT_ERR_UNSUPPORTED and launches nothing. */
attnqat_status attnqat_selftest_bounds(float* buf, int64_t n, int64_t extra, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTNQAT_H_ */
