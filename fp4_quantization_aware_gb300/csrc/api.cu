// C ABI of libattnqat: argument validation, workspace layout and launches.
// Every check runs on the host before anything is enqueued.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <initializer_list>

#include <atomic>
#include <mutex>

#include "../../include/attnqat.h"
#include "attn_common.cuh"

namespace attnqat {

// The device error word that bounded waits write on timeout.
__device__ uint32_t g_device_error;

namespace {

thread_local char g_msg[256] = "";

attnqat_status fail(attnqat_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
attnqat_status fail(attnqat_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}

attnqat_status cuda_fail(cudaError_t e, const char* where) {
  return fail(ATTNQAT_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t qh, kh, vh, delta, dq_acc, split, split_slots, q4, qsf, k4, ksf, total;
  bool packed;   // D = 128: NVFP4 Q^, K^ and their scales for the S MMAs
};

Problem to_problem(const attnqat_problem& p) {
  return Problem{p.B, p.H, p.Sq, p.Sk, p.D, p.is_causal != 0, p.softmax_scale};
}

WsLayout layout(const attnqat_problem& p, bool bwd) {
  const size_t bh = static_cast<size_t>(p.B) * p.H;
  WsLayout w{};
  size_t off = 0;
  w.qh = off, off += round256(bh * p.Sq * p.D * 2);
  w.kh = off, off += round256(bh * p.Sk * p.D * 2);
  w.vh = off, off += round256(bh * p.Sk * p.D * 2);
  if (bwd) {
    w.delta = off, off += round256(bh * p.Sq * 4);
    w.dq_acc = off, off += round256(bh * p.Sq * p.D * 4);
    // split key tiles of the backward: counters, then FP32 [dK, dV] slots
    const int64_t tiles = ((p.Sk + kBlockN - 1) / kBlockN) * static_cast<int64_t>(bh);
    w.split_slots = static_cast<size_t>(tiles < kMaxSplitTiles ? tiles : kMaxSplitTiles);
    w.split = off,
    off += round256((split_cnt_words() + w.split_slots * split_slot_floats(to_problem(p))) * 4);
  }
  if (!bwd && p.D == 128) {
    // split query tiles of the forward's pass 2: counters, then the two CTAs'
    // FP32 [O', O] slots
    const int64_t tiles = ((p.Sq + 127) / 128) * static_cast<int64_t>(bh);
    w.split_slots = static_cast<size_t>(tiles < kMaxSplitTiles ? tiles : kMaxSplitTiles);
    w.split = off,
    off += round256((split_cnt_words() + w.split_slots * fwd_split_slot_floats(to_problem(p))) * 4);
  }
  if (p.D == 128) {   // NVFP4 Q^, K^ for the S MMAs (forward passes, backward recompute)
    w.packed = true;
    w.q4 = off, off += round256(bh * p.Sq * 64);
    w.qsf = off, off += round256(bh * p.Sq * 8);
    w.k4 = off, off += round256(bh * p.Sk * 64);
    w.ksf = off, off += round256(bh * p.Sk * 8);
  }
  w.total = off;
  return w;
}

attnqat_status check_problem(const attnqat_problem* p) {
  if (p == nullptr) return fail(ATTNQAT_ERR_INVALID_ARG, "problem is null");
  if (p->B < 1 || p->H < 1 || p->Sq < 1 || p->Sk < 1 || p->D < 1)
    return fail(ATTNQAT_ERR_INVALID_ARG, "sizes must be >= 1 (B=%lld H=%lld Sq=%lld Sk=%lld D=%lld)",
                (long long)p->B, (long long)p->H, (long long)p->Sq, (long long)p->Sk, (long long)p->D);
  if (!(std::isfinite(p->softmax_scale) && p->softmax_scale > 0.0f))
    return fail(ATTNQAT_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
  if (p->D != 64 && p->D != 128) return fail(ATTNQAT_ERR_UNSUPPORTED, "head dimension %lld not in {64, 128}", (long long)p->D);
  if (p->is_causal && p->Sq != p->Sk) return fail(ATTNQAT_ERR_UNSUPPORTED, "causal attention needs Sq == Sk");
  if (p->Sq >= (int64_t(1) << 31) - 256 || p->Sk >= (int64_t(1) << 31) - 256)
    return fail(ATTNQAT_ERR_UNSUPPORTED, "sequence length beyond 2^31");
  // each factor first, so that the product cannot wrap
  if (p->B > 65535 || p->H > 65535 || p->B * p->H > 65535) return fail(ATTNQAT_ERR_UNSUPPORTED, "B*H above 65535");
  return ATTNQAT_OK;
}

attnqat_status check_ptrs(std::initializer_list<const void*> ptrs) {
  for (const void* q : ptrs) {
    if (q == nullptr) return fail(ATTNQAT_ERR_INVALID_ARG, "a tensor pointer is null");
    if (!aligned16(q)) return fail(ATTNQAT_ERR_MISALIGNED, "a tensor pointer is not 16-byte aligned");
  }
  return ATTNQAT_OK;
}

attnqat_status check_ws(const void* ws, size_t bytes, size_t need) {
  if (ws == nullptr) return fail(ATTNQAT_ERR_WORKSPACE, "workspace is null");
  if (!aligned16(ws)) return fail(ATTNQAT_ERR_WORKSPACE, "workspace is not 16-byte aligned");
  if (bytes < need) return fail(ATTNQAT_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", bytes, need);
  return ATTNQAT_OK;
}

// The device address of g_device_error, looked up once per device (under a
// lock: calls may come from several host threads) and cached for the life of
// the CUDA context.
uint32_t* device_error_word(attnqat_status* st) {
  static std::mutex lock;
  static uint32_t* cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *st = cuda_fail(e, "cudaGetDevice");
    return nullptr;
  }
  std::lock_guard<std::mutex> guard(lock);
  if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_device_error);
  if (e != cudaSuccess) {
    *st = cuda_fail(e, "cudaGetSymbolAddress");
    return nullptr;
  }
  if (dev >= 0 && dev < 64) cache[dev] = static_cast<uint32_t*>(p);
  return static_cast<uint32_t*>(p);
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

#define ATTNQAT_TRY(x)                      \
  do {                                      \
    attnqat_status s_ = (x);                \
    if (s_ != ATTNQAT_OK) return s_;        \
  } while (0)

#define ATTNQAT_CUDA(x, where)                   \
  do {                                           \
    cudaError_t e_ = (x);                        \
    if (e_ != cudaSuccess) return cuda_fail(e_, where); \
  } while (0)

}  // namespace

// ------------------------------------------------------------ shared host helpers
void set_error_message(const char* msg) { snprintf(g_msg, sizeof(g_msg), "%s", msg); }

void* tensor_map_encoder() {
  static void* fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return f;
  }();
  return fn;
}

bool make_tile_map(CUtensorMap* m, const void* base, bool fp32, uint64_t inner, uint64_t rows, uint64_t outer,
                   uint32_t box_inner, uint32_t box_rows) {
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  auto enc = reinterpret_cast<Encode>(tensor_map_encoder());
  if (enc == nullptr) return false;
  const uint64_t es = fp32 ? 4 : 2;
  const cuuint64_t dims[3] = {inner, rows, outer};
  const cuuint64_t strides[2] = {inner * es, inner * rows * es};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_fp4_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t outer, uint32_t box_rows) {
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  auto enc = reinterpret_cast<Encode>(tensor_map_encoder());
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {64, rows, outer};
  const cuuint64_t strides[2] = {64, 64 * rows};
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t set_smem(const void* kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

std::atomic<uint64_t> g_wait_limit_ns{kWaitTimeoutNs};
uint64_t wait_timeout_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

}  // namespace attnqat

using namespace attnqat;

extern "C" {

int attnqat_version(void) { return 100; }

const char* attnqat_status_string(int s) {
  switch (s) {
    case ATTNQAT_OK: return "ok";
    case ATTNQAT_ERR_INVALID_ARG: return "invalid argument";
    case ATTNQAT_ERR_UNSUPPORTED: return "unsupported problem";
    case ATTNQAT_ERR_MISALIGNED: return "misaligned pointer";
    case ATTNQAT_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTNQAT_ERR_CUDA: return "CUDA error";
    case ATTNQAT_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

const char* attnqat_last_error_message(void) { return g_msg; }

attnqat_status attnqat_check_support(const attnqat_problem* p) { return check_problem(p); }

size_t attnqat_fwd_workspace_bytes(const attnqat_problem* p) {
  return check_problem(p) == ATTNQAT_OK ? layout(*p, false).total : 0;
}

size_t attnqat_bwd_workspace_bytes(const attnqat_problem* p) {
  return check_problem(p) == ATTNQAT_OK ? layout(*p, true).total : 0;
}

attnqat_status attnqat_fake_nvfp4(const void* x, void* y, int64_t rows, int64_t cols, void* stream) {
  if (rows < 0 || cols < 0) return fail(ATTNQAT_ERR_INVALID_ARG, "negative size");
  if (rows == 0 || cols == 0) return ATTNQAT_OK;
  ATTNQAT_TRY(check_ptrs({x, y}));
  ATTNQAT_CUDA(launch_fake_bf16(static_cast<const bf16*>(x), static_cast<bf16*>(y), rows, cols,
                                static_cast<cudaStream_t>(stream)),
               "fake_nvfp4");
  return ATTNQAT_OK;
}

attnqat_status attnqat_fake_nvfp4_f32(const float* x, float* y, int64_t rows, int64_t cols, void* stream) {
  if (rows < 0 || cols < 0) return fail(ATTNQAT_ERR_INVALID_ARG, "negative size");
  if (rows == 0 || cols == 0) return ATTNQAT_OK;
  ATTNQAT_TRY(check_ptrs({x, y}));
  ATTNQAT_CUDA(launch_fake_f32(x, y, rows, cols, static_cast<cudaStream_t>(stream)), "fake_nvfp4_f32");
  return ATTNQAT_OK;
}

// The forward's split-tile counters (D = 128), which the quantize step clears.
int64_t fwd_split_zero_floats(const attnqat_problem& p, const WsLayout& w) {
  (void)p;
  return w.packed ? split_cnt_words() : 0;
}

attnqat_status attnqat_quantize_qkv(const attnqat_problem* p, const void* q, const void* k, const void* v,
                                    void* ws, size_t ws_bytes, void* stream) {
  ATTNQAT_TRY(check_problem(p));
  ATTNQAT_TRY(check_ptrs({q, k, v}));
  const WsLayout w = layout(*p, false);
  ATTNQAT_TRY(check_ws(ws, ws_bytes, w.total));
  ATTNQAT_CUDA(launch_prep(to_problem(*p), static_cast<const bf16*>(q), static_cast<const bf16*>(k),
                           static_cast<const bf16*>(v), nullptr, nullptr, at<bf16>(ws, w.qh), at<bf16>(ws, w.kh),
                           at<bf16>(ws, w.vh), nullptr, nullptr, w.packed ? at<float>(ws, w.split) : nullptr,
                           fwd_split_zero_floats(*p, w),
                           w.packed ? at<uint8_t>(ws, w.q4) : nullptr, w.packed ? at<uint8_t>(ws, w.qsf) : nullptr,
                           w.packed ? at<uint8_t>(ws, w.k4) : nullptr, w.packed ? at<uint8_t>(ws, w.ksf) : nullptr,
                           static_cast<cudaStream_t>(stream)),
               "quantize_qkv");
  return ATTNQAT_OK;
}

attnqat_status attnqat_fwd_main(const attnqat_problem* p, void* o, void* o_hp, float* lse, void* ws,
                                size_t ws_bytes, void* stream) {
  ATTNQAT_TRY(check_problem(p));
  ATTNQAT_TRY(check_ptrs({o, o_hp, lse}));
  const WsLayout w = layout(*p, false);
  ATTNQAT_TRY(check_ws(ws, ws_bytes, w.total));
  attnqat_status st = ATTNQAT_OK;
  uint32_t* err = device_error_word(&st);
  if (!err) return st;
  ATTNQAT_CUDA(launch_fwd(to_problem(*p), at<bf16>(ws, w.qh), at<bf16>(ws, w.kh), at<bf16>(ws, w.vh),
                          w.packed ? at<uint8_t>(ws, w.q4) : nullptr, w.packed ? at<uint8_t>(ws, w.qsf) : nullptr,
                          w.packed ? at<uint8_t>(ws, w.k4) : nullptr, w.packed ? at<uint8_t>(ws, w.ksf) : nullptr,
                          static_cast<bf16*>(o), static_cast<bf16*>(o_hp), lse,
                          w.packed ? at<float>(ws, w.split) + split_cnt_words() : nullptr,
                          w.packed ? at<uint32_t>(ws, w.split) : nullptr, err, static_cast<cudaStream_t>(stream)),
               "fwd_main");
  return ATTNQAT_OK;
}

attnqat_status attnqat_fwd(const attnqat_problem* p, const void* q, const void* k, const void* v, void* o,
                           void* o_hp, float* lse, void* ws, size_t ws_bytes, void* stream) {
  ATTNQAT_TRY(check_problem(p));
  ATTNQAT_TRY(check_ptrs({q, k, v, o, o_hp, lse}));
  ATTNQAT_TRY(check_ws(ws, ws_bytes, layout(*p, false).total));
  const WsLayout w = layout(*p, false);
  if (!w.packed) {
    ATTNQAT_TRY(attnqat_quantize_qkv(p, q, k, v, ws, ws_bytes, stream));
    return attnqat_fwd_main(p, o, o_hp, lse, ws, ws_bytes, stream);
  }
  // D = 128: the forward kernel reads Q and K only in their NVFP4 encoding,
  // so the BF16 Q^, K^ are not written (V^ is: the PV MMAs read it)
  ATTNQAT_CUDA(launch_prep(to_problem(*p), static_cast<const bf16*>(q), static_cast<const bf16*>(k),
                           static_cast<const bf16*>(v), nullptr, nullptr, nullptr, nullptr, at<bf16>(ws, w.vh),
                           nullptr, nullptr, at<float>(ws, w.split), fwd_split_zero_floats(*p, w),
                           at<uint8_t>(ws, w.q4), at<uint8_t>(ws, w.qsf),
                           at<uint8_t>(ws, w.k4), at<uint8_t>(ws, w.ksf), static_cast<cudaStream_t>(stream)),
               "fwd quantize");
  return attnqat_fwd_main(p, o, o_hp, lse, ws, ws_bytes, stream);
}

attnqat_status attnqat_fwd_main_r2_p(const attnqat_problem* p, void* o, void* o_hp, float* lse, int p_format,
                                     void* ws, size_t ws_bytes, void* stream) {
  ATTNQAT_TRY(check_problem(p));
  ATTNQAT_TRY(check_ptrs({o, o_hp, lse}));
  if (p_format != ATTNQAT_P_NVFP4 && p_format != ATTNQAT_P_FP8_E5M2 && p_format != ATTNQAT_P_FP8_E4M3)
    return fail(ATTNQAT_ERR_INVALID_ARG, "p_format must be ATTNQAT_P_NVFP4, ATTNQAT_P_FP8_E5M2 or ATTNQAT_P_FP8_E4M3");
  const WsLayout w = layout(*p, false);
  ATTNQAT_TRY(check_ws(ws, ws_bytes, w.total));
  attnqat_status st = ATTNQAT_OK;
  uint32_t* err = device_error_word(&st);
  if (!err) return st;
  ATTNQAT_CUDA(launch_fwd_r2(to_problem(*p), at<bf16>(ws, w.qh), at<bf16>(ws, w.kh), at<bf16>(ws, w.vh),
                             static_cast<bf16*>(o), static_cast<bf16*>(o_hp), lse, p_format, err,
                             static_cast<cudaStream_t>(stream)),
               "fwd_main_r2");
  return ATTNQAT_OK;
}

attnqat_status attnqat_fwd_main_r2(const attnqat_problem* p, void* o, void* o_hp, float* lse, void* ws,
                                   size_t ws_bytes, void* stream) {
  return attnqat_fwd_main_r2_p(p, o, o_hp, lse, ATTNQAT_P_NVFP4, ws, ws_bytes, stream);
}

attnqat_status attnqat_fwd_r2_p(const attnqat_problem* p, const void* q, const void* k, const void* v, void* o,
                                void* o_hp, float* lse, int p_format, void* ws, size_t ws_bytes, void* stream) {
  ATTNQAT_TRY(check_problem(p));
  ATTNQAT_TRY(check_ptrs({q, k, v, o, o_hp, lse}));
  if (p_format != ATTNQAT_P_NVFP4 && p_format != ATTNQAT_P_FP8_E5M2 && p_format != ATTNQAT_P_FP8_E4M3)
    return fail(ATTNQAT_ERR_INVALID_ARG, "p_format must be ATTNQAT_P_NVFP4, ATTNQAT_P_FP8_E5M2 or ATTNQAT_P_FP8_E4M3");
  ATTNQAT_TRY(check_ws(ws, ws_bytes, layout(*p, false).total));
  ATTNQAT_TRY(attnqat_quantize_qkv(p, q, k, v, ws, ws_bytes, stream));
  return attnqat_fwd_main_r2_p(p, o, o_hp, lse, p_format, ws, ws_bytes, stream);
}

attnqat_status attnqat_fwd_r2(const attnqat_problem* p, const void* q, const void* k, const void* v, void* o,
                              void* o_hp, float* lse, void* ws, size_t ws_bytes, void* stream) {
  return attnqat_fwd_r2_p(p, q, k, v, o, o_hp, lse, ATTNQAT_P_NVFP4, ws, ws_bytes, stream);
}

attnqat_status attnqat_bwd_preprocess(const attnqat_problem* p, const void* dout, const void* q, const void* k,
                                      const void* v, const void* o_hp, void* ws, size_t ws_bytes, void* stream) {
  ATTNQAT_TRY(check_problem(p));
  ATTNQAT_TRY(check_ptrs({dout, q, k, v, o_hp}));
  const WsLayout w = layout(*p, true);
  ATTNQAT_TRY(check_ws(ws, ws_bytes, w.total));
  ATTNQAT_CUDA(launch_prep(to_problem(*p), static_cast<const bf16*>(q), static_cast<const bf16*>(k),
                           static_cast<const bf16*>(v), static_cast<const bf16*>(o_hp),
                           static_cast<const bf16*>(dout), at<bf16>(ws, w.qh), at<bf16>(ws, w.kh),
                           at<bf16>(ws, w.vh), at<float>(ws, w.delta), at<float>(ws, w.dq_acc),
                           at<float>(ws, w.split),
                           split_cnt_words() + bwd_split_plan(to_problem(*p), device_sm_count()).n_split *
                                                   split_slot_floats(to_problem(*p)),
                           w.packed ? at<uint8_t>(ws, w.q4) : nullptr, w.packed ? at<uint8_t>(ws, w.qsf) : nullptr,
                           w.packed ? at<uint8_t>(ws, w.k4) : nullptr, w.packed ? at<uint8_t>(ws, w.ksf) : nullptr,
                           static_cast<cudaStream_t>(stream)),
               "bwd_preprocess");
  return ATTNQAT_OK;
}

attnqat_status attnqat_bwd_main(const attnqat_problem* p, const void* dout, const float* lse, void* dk, void* dv,
                                void* ws, size_t ws_bytes, void* stream) {
  ATTNQAT_TRY(check_problem(p));
  ATTNQAT_TRY(check_ptrs({dout, lse, dk, dv}));
  const WsLayout w = layout(*p, true);
  ATTNQAT_TRY(check_ws(ws, ws_bytes, w.total));
  attnqat_status st = ATTNQAT_OK;
  uint32_t* err = device_error_word(&st);
  if (!err) return st;
  ATTNQAT_CUDA(launch_bwd(to_problem(*p), at<bf16>(ws, w.qh), at<bf16>(ws, w.kh), at<bf16>(ws, w.vh),
                          static_cast<const bf16*>(dout), lse, at<float>(ws, w.delta), at<float>(ws, w.dq_acc),
                          static_cast<bf16*>(dk), static_cast<bf16*>(dv), at<float>(ws, w.split) + split_cnt_words(),
                          at<uint32_t>(ws, w.split), w.packed ? at<uint8_t>(ws, w.q4) : nullptr,
                          w.packed ? at<uint8_t>(ws, w.qsf) : nullptr, w.packed ? at<uint8_t>(ws, w.k4) : nullptr,
                          w.packed ? at<uint8_t>(ws, w.ksf) : nullptr, err, static_cast<cudaStream_t>(stream)),
               "bwd_main");
  return ATTNQAT_OK;
}

attnqat_status attnqat_bwd_dq_convert(const attnqat_problem* p, void* dq, void* ws, size_t ws_bytes, void* stream) {
  ATTNQAT_TRY(check_problem(p));
  ATTNQAT_TRY(check_ptrs({dq}));
  const WsLayout w = layout(*p, true);
  ATTNQAT_TRY(check_ws(ws, ws_bytes, w.total));
  ATTNQAT_CUDA(launch_dq_convert(to_problem(*p), at<float>(ws, w.dq_acc), static_cast<bf16*>(dq),
                                 static_cast<cudaStream_t>(stream)),
               "bwd_dq_convert");
  return ATTNQAT_OK;
}

attnqat_status attnqat_bwd(const attnqat_problem* p, const void* dout, const void* q, const void* k, const void* v,
                           const void* o_hp, const float* lse, void* dq, void* dk, void* dv, void* ws,
                           size_t ws_bytes, void* stream) {
  ATTNQAT_TRY(check_problem(p));
  ATTNQAT_TRY(check_ptrs({dout, q, k, v, o_hp, lse, dq, dk, dv}));
  ATTNQAT_TRY(check_ws(ws, ws_bytes, layout(*p, true).total));
  ATTNQAT_TRY(attnqat_bwd_preprocess(p, dout, q, k, v, o_hp, ws, ws_bytes, stream));
  ATTNQAT_TRY(attnqat_bwd_main(p, dout, lse, dk, dv, ws, ws_bytes, stream));
  return attnqat_bwd_dq_convert(p, dq, ws, ws_bytes, stream);
}

attnqat_status attnqat_nvfp4_pack(const void* x, void* packed, void* scales, int64_t rows, int64_t cols,
                                  void* stream) {
  if (rows < 0 || cols < 0) return fail(ATTNQAT_ERR_INVALID_ARG, "negative size");
  if (cols % 16 != 0) return fail(ATTNQAT_ERR_INVALID_ARG, "cols (%lld) is not a multiple of 16", (long long)cols);
  if (rows == 0 || cols == 0) return ATTNQAT_OK;
  ATTNQAT_TRY(check_ptrs({x, packed, scales}));
  ATTNQAT_CUDA(launch_nvfp4_pack(static_cast<const bf16*>(x), static_cast<uint8_t*>(packed),
                                 static_cast<uint8_t*>(scales), rows, cols, static_cast<cudaStream_t>(stream)),
               "nvfp4_pack");
  return ATTNQAT_OK;
}

namespace {

attnqat_status check_infer(const attnqat_problem* p) {
  ATTNQAT_TRY(check_problem(p));
  if (p->D != 128) return fail(ATTNQAT_ERR_UNSUPPORTED, "the inference forward needs D == 128 (got %lld)", (long long)p->D);
  return ATTNQAT_OK;
}

struct InferWs {
  size_t q_fp4, q_sf, k_fp4, k_sf, total;
};

InferWs infer_layout(const attnqat_problem& p) {
  const size_t bh = static_cast<size_t>(p.B) * p.H;
  InferWs w{};
  size_t off = 0;
  w.q_fp4 = off, off += round256(bh * p.Sq * 64);
  w.q_sf = off, off += round256(bh * p.Sq * 8);
  w.k_fp4 = off, off += round256(bh * p.Sk * 64);
  w.k_sf = off, off += round256(bh * p.Sk * 8);
  w.total = off;
  return w;
}

}  // namespace

size_t attnqat_infer_fwd_workspace_bytes(const attnqat_problem* p) {
  return check_infer(p) == ATTNQAT_OK ? infer_layout(*p).total : 0;
}

attnqat_status attnqat_infer_fwd_packed(const attnqat_problem* p, const void* q_fp4, const void* q_sf,
                                        const void* k_fp4, const void* k_sf, const void* v, void* o, float* lse,
                                        void* stream) {
  ATTNQAT_TRY(check_infer(p));
  ATTNQAT_TRY(check_ptrs({q_fp4, q_sf, k_fp4, k_sf, v, o}));
  if (lse != nullptr && !aligned16(lse)) return fail(ATTNQAT_ERR_MISALIGNED, "lse is not 16-byte aligned");
  attnqat_status st = ATTNQAT_OK;
  uint32_t* err = device_error_word(&st);
  if (!err) return st;
  ATTNQAT_CUDA(launch_infer(to_problem(*p), static_cast<const uint8_t*>(q_fp4), static_cast<const uint8_t*>(q_sf),
                            static_cast<const uint8_t*>(k_fp4), static_cast<const uint8_t*>(k_sf),
                            static_cast<const bf16*>(v), static_cast<bf16*>(o), lse, err,
                            static_cast<cudaStream_t>(stream)),
               "infer_fwd");
  return ATTNQAT_OK;
}

attnqat_status attnqat_infer_fwd(const attnqat_problem* p, const void* q, const void* k, const void* v, void* o,
                                 float* lse, void* ws, size_t ws_bytes, void* stream) {
  ATTNQAT_TRY(check_infer(p));
  ATTNQAT_TRY(check_ptrs({q, k, v, o}));
  const InferWs w = infer_layout(*p);
  ATTNQAT_TRY(check_ws(ws, ws_bytes, w.total));
  const int64_t bh = p->B * p->H;
  ATTNQAT_TRY(attnqat_nvfp4_pack(q, at<uint8_t>(ws, w.q_fp4), at<uint8_t>(ws, w.q_sf), bh * p->Sq, p->D, stream));
  ATTNQAT_TRY(attnqat_nvfp4_pack(k, at<uint8_t>(ws, w.k_fp4), at<uint8_t>(ws, w.k_sf), bh * p->Sk, p->D, stream));
  return attnqat_infer_fwd_packed(p, at<uint8_t>(ws, w.q_fp4), at<uint8_t>(ws, w.q_sf), at<uint8_t>(ws, w.k_fp4),
                                  at<uint8_t>(ws, w.k_sf), v, o, lse, stream);
}

attnqat_status attnqat_device_status(int clear) {
  attnqat_status st = ATTNQAT_OK;
  uint32_t* err = device_error_word(&st);
  if (!err) return st;
  ATTNQAT_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  uint32_t v = 0;
  ATTNQAT_CUDA(cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost), "read device error word");
  if (clear) ATTNQAT_CUDA(cudaMemset(err, 0, sizeof(uint32_t)), "clear device error word");
  if (clear) ATTNQAT_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  return v == kDevTimeout ? fail(ATTNQAT_ERR_TIMEOUT, "a device wait ran out of time") : ATTNQAT_OK;
}

int attnqat_checked_build(void) {
#ifdef ATTNQAT_CHECKED
  return 1;
#else
  return 0;
#endif
}

attnqat_status attnqat_debug_oob_count(unsigned long long* count, int clear) {
  ATTNQAT_TRY(check_ptrs({count}));
  if (!attnqat_checked_build()) return fail(ATTNQAT_ERR_UNSUPPORTED, "bounds checks are in the debug build only");
  ATTNQAT_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  unsigned long long n = 0;
  for (auto* rd : {oob_read_fwd_lse, oob_read_fwd_pv, oob_read_fwd, oob_read_fwd_r2, oob_read_bwd, oob_read_infer,
                   oob_read_quant})
    ATTNQAT_CUDA(rd(&n, clear != 0), "read bounds-check counters");
  *count = n;
  return ATTNQAT_OK;
}

attnqat_status attnqat_selftest_bounds(float* buf, int64_t n, int64_t extra, void* stream) {
  if (!attnqat_checked_build()) return fail(ATTNQAT_ERR_UNSUPPORTED, "bounds checks are in the debug build only");
  if (buf == nullptr || n < 1 || extra < 0) return fail(ATTNQAT_ERR_INVALID_ARG, "buf null, n < 1 or extra < 0");
  ATTNQAT_CUDA(launch_bounds_selftest(buf, n, extra, static_cast<cudaStream_t>(stream)), "selftest_bounds");
  return ATTNQAT_OK;
}

attnqat_status attnqat_selftest_quotient(unsigned long long* out, void* stream) {
  ATTNQAT_TRY(check_ptrs({out}));
  ATTNQAT_CUDA(launch_quotient_selftest(out, static_cast<cudaStream_t>(stream)), "selftest_quotient");
  return ATTNQAT_OK;
}

attnqat_status attnqat_selftest_scale(unsigned long long* out, void* stream) {
  ATTNQAT_TRY(check_ptrs({out}));
  ATTNQAT_CUDA(launch_scale_selftest(out, static_cast<cudaStream_t>(stream)), "selftest_scale");
  return ATTNQAT_OK;
}

attnqat_status attnqat_selftest_set_wait_limit(uint64_t timeout_ns) {
  if (timeout_ns > 10000000000ull) return fail(ATTNQAT_ERR_INVALID_ARG, "wait limit above 10 s");
  attnqat::g_wait_limit_ns.store(timeout_ns, std::memory_order_relaxed);
  return ATTNQAT_OK;
}

attnqat_status attnqat_selftest_wait_timeout(uint64_t timeout_ns, void* stream) {
  attnqat_status st = ATTNQAT_OK;
  uint32_t* err = device_error_word(&st);
  if (!err) return st;
  if (timeout_ns > 10000000000ull) return fail(ATTNQAT_ERR_INVALID_ARG, "timeout above 10 s");
  ATTNQAT_CUDA(launch_wait_timeout(err, timeout_ns, static_cast<cudaStream_t>(stream)), "selftest_wait_timeout");
  return ATTNQAT_OK;
}

}  // extern "C"
