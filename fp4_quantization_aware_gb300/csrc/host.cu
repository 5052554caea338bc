// attnqat_bwd_host: the backward with its inputs and outputs in host memory.
//
// The B*H heads are processed in contiguous groups. Group c's kernels run on
// the caller's stream (attnqat_bwd on a problem of the group's heads) while
// group c + 1 is copied in on one of the library's copy streams and group
// c - 1 is copied out on the other, so the host<->device transfers overlap
// the kernels. Two device slots, each holding one group's inputs, outputs and
// backward workspace, alternate between groups; events order each slot's
// reuse. The copy-in of group c + 2 waits only for group c's kernels (the
// last readers of the slot's inputs), so the inputs stream in back to back;
// group c + 2's kernels wait for the copy-out of group c (the slot's
// outputs) as well as for their own inputs.
//
// The groups hold ceil(B*H / chunks) heads each, except the first and the last
// ones, which hold half of that: the kernels start after a shorter first copy,
// and less work is left once the last inputs are in (the copies, not the
// kernels, bound this call).
//
// The copy streams and events are created once per device and shared by all
// calls, so calls on one device must not run concurrently from several host
// threads.
#include <mutex>

#include "../../include/attnqat.h"
#include "kernels.h"

namespace attnqat {
void set_error_message(const char* msg);
}

namespace {

constexpr int kMaxDevices = 64;

struct CopyStreams {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t in[2] = {}, done[2] = {}, out[2] = {};   // per slot: copied in, kernels done, copied out
};

std::mutex g_mutex;
CopyStreams g_streams[kMaxDevices];

size_t r256(size_t x) { return (x + 255) & ~size_t(255); }

// Byte offsets of one slot's buffers for a group of `hc` heads.
struct SlotLayout {
  size_t dout, q, o_hp, k, v, lse, dq, dk, dv, ws, ws_bytes, total;
};

attnqat_problem group_problem(const attnqat_problem& p, int64_t heads) {
  attnqat_problem g = p;
  g.B = 1, g.H = heads;
  return g;
}

SlotLayout slot_layout(const attnqat_problem& p, int64_t hc) {
  const size_t nq = static_cast<size_t>(hc) * p.Sq * p.D * 2, nk = static_cast<size_t>(hc) * p.Sk * p.D * 2;
  const attnqat_problem g = group_problem(p, hc);
  SlotLayout s{};
  size_t off = 0;
  s.dout = off, off += r256(nq);
  s.q = off, off += r256(nq);
  s.o_hp = off, off += r256(nq);
  s.k = off, off += r256(nk);
  s.v = off, off += r256(nk);
  s.lse = off, off += r256(static_cast<size_t>(hc) * p.Sq * 4);
  s.dq = off, off += r256(nq);
  s.dk = off, off += r256(nk);
  s.dv = off, off += r256(nk);
  s.ws = off;
  s.ws_bytes = attnqat_bwd_workspace_bytes(&g);
  off += r256(s.ws_bytes);
  s.total = off;
  return s;
}

// Heads per group: ceil(B*H / chunks), chunks clamped to 1..B*H.
int64_t group_heads(const attnqat_problem& p, int chunks) {
  const int64_t bh = p.B * p.H;
  const int64_t n = chunks < 1 ? 1 : (chunks > bh ? bh : chunks);
  return (bh + n - 1) / n;
}

// The first head and the head count of group g of the call's groups (see the
// file comment): sizes half, full, ..., full, then the remainder, of which a
// full-size last group is halved.
struct GroupPlan {
  int64_t bh, hc, first, n_mid, rest_a, rest_b;   // group sizes: first, n_mid x hc, rest_a, rest_b
  int64_t groups() const { return 1 + n_mid + (rest_a > 0) + (rest_b > 0); }
  void group(int64_t g, int64_t& h0, int64_t& nh) const {
    if (g == 0) { h0 = 0, nh = first; return; }
    if (g <= n_mid) { h0 = first + (g - 1) * hc, nh = hc; return; }
    h0 = first + n_mid * hc;
    if (g == n_mid + 1 && rest_a > 0) { nh = rest_a; return; }
    h0 += rest_a, nh = rest_b;
  }
};

GroupPlan plan_groups(int64_t bh, int64_t hc) {
  GroupPlan p{bh, hc, 0, 0, 0, 0};
  p.first = hc > 1 ? (hc + 1) / 2 : 1;
  if (p.first >= bh) {
    p.first = bh;
    return p;
  }
  int64_t rest = bh - p.first;
  p.n_mid = rest / hc;
  rest -= p.n_mid * hc;
  if (rest == 0 && p.n_mid > 0 && hc > 1) {   // the last full group becomes two halves
    --p.n_mid;
    rest = hc;
  }
  if (rest > (hc + 1) / 2 && hc > 1) {
    p.rest_a = rest - (hc + 1) / 2;
    p.rest_b = (hc + 1) / 2;
  } else {
    p.rest_a = rest;
  }
  return p;
}

attnqat_status streams_for(int dev, CopyStreams** out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  CopyStreams& s = g_streams[dev];
  if (s.h2d == nullptr) {
    CopyStreams c;
    bool ok = cudaStreamCreateWithFlags(&c.h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&c.start, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < 2; ++i)
      ok = cudaEventCreateWithFlags(&c.in[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&c.done[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&c.out[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      attnqat::set_error_message("attnqat_bwd_host: could not create the copy streams and events");
      return ATTNQAT_ERR_CUDA;
    }
    s = c;
  }
  *out = &s;
  return ATTNQAT_OK;
}

}  // namespace

extern "C" size_t attnqat_bwd_host_workspace_bytes(const attnqat_problem* p, int chunks) {
  if (attnqat_check_support(p) != ATTNQAT_OK) return 0;
  const SlotLayout s = slot_layout(*p, group_heads(*p, chunks));
  return s.ws_bytes == 0 ? 0 : 2 * s.total;
}

extern "C" attnqat_status attnqat_bwd_host(const attnqat_problem* p, const void* dout, const void* q,
                                           const void* k, const void* v, const void* o_hp, const float* lse,
                                           void* dq, void* dk, void* dv, int chunks, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  attnqat_status st = attnqat_check_support(p);
  if (st != ATTNQAT_OK) return st;
  for (const void* ptr : {dout, q, k, v, o_hp, static_cast<const void*>(lse), static_cast<const void*>(dq),
                          static_cast<const void*>(dk), static_cast<const void*>(dv)})
    if (ptr == nullptr) {
      attnqat::set_error_message("attnqat_bwd_host: a host tensor pointer is null");
      return ATTNQAT_ERR_INVALID_ARG;
    }
  const int64_t bh = p->B * p->H, hc = group_heads(*p, chunks);
  const GroupPlan plan = plan_groups(bh, hc);
  const int64_t groups = plan.groups();
  const SlotLayout L = slot_layout(*p, hc);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < 2 * L.total) {
    attnqat::set_error_message("attnqat_bwd_host: the device workspace is null, not 256-byte aligned, or "
                               "smaller than attnqat_bwd_host_workspace_bytes(p, chunks)");
    return ATTNQAT_ERR_WORKSPACE;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    attnqat::set_error_message("attnqat_bwd_host: no usable current device");
    return ATTNQAT_ERR_CUDA;
  }
  CopyStreams* S = nullptr;
  if ((st = streams_for(dev, &S)) != ATTNQAT_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  bool ok = true;
  auto cuda = [&](cudaError_t e) {
    if (e != cudaSuccess && ok) {
      attnqat::set_error_message(cudaGetErrorString(e));
      ok = false;
    }
    return ok;
  };
  // Copies start after the work already on the caller's stream (which may use
  // the workspace or write the inputs).
  cuda(cudaEventRecord(S->start, cs));
  cuda(cudaStreamWaitEvent(S->h2d, S->start, 0));
  cuda(cudaStreamWaitEvent(S->d2h, S->start, 0));
  const size_t qrow = static_cast<size_t>(p->Sq) * p->D * 2, krow = static_cast<size_t>(p->Sk) * p->D * 2;
  const size_t lrow = static_cast<size_t>(p->Sq) * 4;
  const uint8_t* hin[6] = {static_cast<const uint8_t*>(dout), static_cast<const uint8_t*>(q),
                           static_cast<const uint8_t*>(o_hp), static_cast<const uint8_t*>(k),
                           static_cast<const uint8_t*>(v), reinterpret_cast<const uint8_t*>(lse)};
  const size_t in_off[6] = {L.dout, L.q, L.o_hp, L.k, L.v, L.lse};
  const size_t in_row[6] = {qrow, qrow, qrow, krow, krow, lrow};
  uint8_t* hout[3] = {static_cast<uint8_t*>(dq), static_cast<uint8_t*>(dk), static_cast<uint8_t*>(dv)};
  const size_t out_off[3] = {L.dq, L.dk, L.dv};
  const size_t out_row[3] = {qrow, krow, krow};
  for (int64_t g = 0; ok && g < groups; ++g) {
    const int s = static_cast<int>(g & 1);
    int64_t h0 = 0, nh = 0;
    plan.group(g, h0, nh);
    uint8_t* base = static_cast<uint8_t*>(workspace) + s * L.total;
    if (g >= 2) cuda(cudaStreamWaitEvent(S->h2d, S->done[s], 0));   // slot s's inputs read (group g - 2)
    for (int i = 0; i < 6 && ok; ++i)
      cuda(cudaMemcpyAsync(base + in_off[i], hin[i] + h0 * in_row[i], nh * in_row[i], cudaMemcpyHostToDevice,
                           S->h2d));
    cuda(cudaEventRecord(S->in[s], S->h2d));
    cuda(cudaStreamWaitEvent(cs, S->in[s], 0));
    if (g >= 2) cuda(cudaStreamWaitEvent(cs, S->out[s], 0));         // slot s's outputs copied out (group g - 2)
    if (!ok) break;
    const attnqat_problem gp = group_problem(*p, nh);
    st = attnqat_bwd(&gp, base + L.dout, base + L.q, base + L.k, base + L.v, base + L.o_hp,
                     reinterpret_cast<const float*>(base + L.lse), base + L.dq, base + L.dk, base + L.dv,
                     base + L.ws, L.ws_bytes, stream);
    if (st != ATTNQAT_OK) return st;
    cuda(cudaEventRecord(S->done[s], cs));
    cuda(cudaStreamWaitEvent(S->d2h, S->done[s], 0));
    for (int i = 0; i < 3 && ok; ++i)
      cuda(cudaMemcpyAsync(hout[i] + h0 * out_row[i], base + out_off[i], nh * out_row[i], cudaMemcpyDeviceToHost,
                           S->d2h));
    cuda(cudaEventRecord(S->out[s], S->d2h));
  }
  // The caller's stream waits for the last copy out of both slots.
  for (int64_t g = groups - 2; ok && g < groups; ++g)
    if (g >= 0) cuda(cudaStreamWaitEvent(cs, S->out[g & 1], 0));
  return ok ? ATTNQAT_OK : ATTNQAT_ERR_CUDA;
}
