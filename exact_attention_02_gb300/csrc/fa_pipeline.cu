// fa_fwd_bwd_host: forward + backward of host-resident tensors, with the host<->device
// copies overlapped with the kernels.
//
// The heads are independent, so the call cuts the B*H heads into contiguous groups and runs
// each group through three stages on three internal streams:
//   copy-in  : Q, K, V, dO of the group, host -> device slot
//   compute  : fa_fwd, fa_bwd_preprocess, fa_bwd on the slot (the group as B = 1, H = heads)
//   copy-out : O, LSE, dQ, dK, dV of the group, device slot -> host
// Three device slots rotate, so group g's copy-in overlaps group g-1's kernels and the
// copy-outs of groups g-1 and g-2; with two slots, the copy-in of a group had to wait for
// the copy-out of the group two before it, which left the kernels idle between groups.
// Events order the stages at the granularity the kernels need: the forward starts once
// Q, K and V have landed (dO is still on its way), and O and LSE go back to the host while
// the backward runs; a slot is refilled only after its previous group's copy-out has
// read it. The call forks from the caller's stream (the internal
// streams wait on an event recorded there) and joins back into it (the caller's stream
// waits on the last copy-out), so it enqueues work and returns without synchronising.
//
// Only the first group's copy-in and the last group's copy-out overlap no kernel, so the
// default schedule makes those two groups half the size of the others (1:2:2:2:1).
#include <algorithm>
#include <mutex>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kMaxChunks = 16;
constexpr int kSlots = 3;
constexpr int kEventsPerChunk = 5;
constexpr int kRing = kMaxChunks * kEventsPerChunk + 1;  // + the fork event
constexpr int kJoinEvents = 3;                            // error join: one per internal stream

size_t round_up(size_t x) { return (x + 255) / 256 * 256; }

// Per-slot layout for `hc` heads.
struct SlotLayout {
  size_t q, k, v, dO, o, dq, dk, dv, lse, D, acc, bytes;
};

SlotLayout slot_layout(int64_t hc, int N, int d) {
  const size_t el = (size_t)hc * N * d * 2, rows = (size_t)hc * N * 4;
  SlotLayout s;
  size_t off = 0;
  auto take = [&](size_t n) {
    const size_t at = off;
    off += round_up(n);
    return at;
  };
  s.q = take(el);
  s.k = take(el);
  s.v = take(el);
  s.dO = take(el);
  s.o = take(el);
  s.dq = take(el);
  s.dk = take(el);
  s.dv = take(el);
  s.lse = take(rows);
  s.D = take(rows);
  s.acc = take((size_t)hc * N * d * 4);
  s.bytes = off;
  return s;
}

struct DeviceQueues {
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  cudaEvent_t ring[kRing] = {};
  cudaEvent_t join[kJoinEvents] = {};
  bool ok = false;
};

// Streams and events are created once per device and reused; a mutex serialises the
// enqueueing of concurrent calls (each event is waited on before it is recorded again,
// and a wait captures the event's state when it is enqueued).
std::mutex g_mu;
DeviceQueues g_queues[64];

DeviceQueues* queues_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  DeviceQueues& q = g_queues[dev];
  if (!q.ok) {
    bool ok = cudaStreamCreateWithFlags(&q.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&q.comp, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&q.out, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; ok && i < kRing; ++i) ok = cudaEventCreateWithFlags(&q.ring[i], cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < kJoinEvents; ++i)
      ok = cudaEventCreateWithFlags(&q.join[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) return nullptr;
    q.ok = true;
  }
  return &q;
}

// Group g holds heads start[g] .. start[g+1] - 1.
struct Groups {
  int n = 0;
  int64_t start[kMaxChunks + 1] = {};
  int64_t largest = 0;
};

// chunks > 0: that many equal groups (at most B*H and 16; the last may be smaller).
// chunks == 0: with at least 8 heads, five groups in the ratio 1:2:2:2:1; else up to 4
// equal groups.
Groups make_groups(int64_t heads, int chunks) {
  Groups g;
  if (chunks <= 0 && heads >= 8) {
    const int64_t q = heads / 8, rem = heads - 2 * q;
    const int64_t size[5] = {q, rem / 3 + (rem % 3 > 0), rem / 3 + (rem % 3 > 1), rem / 3, q};
    g.n = 5;
    for (int i = 0; i < 5; ++i) g.start[i + 1] = g.start[i] + size[i];
  } else {
    const int c = (int)std::max<int64_t>(1, std::min<int64_t>({(int64_t)(chunks <= 0 ? 4 : chunks), heads,
                                                               (int64_t)kMaxChunks}));
    const int64_t hc = (heads + c - 1) / c;
    g.n = (int)((heads + hc - 1) / hc);
    for (int i = 0; i < g.n; ++i) g.start[i + 1] = std::min<int64_t>(heads, g.start[i] + hc);
  }
  for (int i = 0; i < g.n; ++i) g.largest = std::max(g.largest, g.start[i + 1] - g.start[i]);
  return g;
}

}  // namespace
}  // namespace fa

extern "C" size_t fa_fwd_bwd_host_workspace_size(int B, int H, int N, int d, int dtype, int chunks) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128) || dtype != FA_DTYPE_BF16) return 0;
  const fa::Groups g = fa::make_groups((int64_t)B * H, chunks);
  return fa::kSlots * fa::slot_layout(g.largest, N, d).bytes;
}

namespace fa {
namespace {

// Enqueues every group's copy-in, kernels and copy-out on the internal streams (which have
// already forked from the caller's stream) and joins the caller's stream to the last
// copy-out. Returns at the first failure, with some work possibly enqueued.
fa_status_t enqueue_groups(const void* Q, const void* K, const void* V, const void* dO, void* O, float* LSE,
                           void* dQ, void* dK, void* dV, void* workspace, int N, int d, float scale, int causal,
                           int dtype, const Groups& G, const SlotLayout& L, DeviceQueues* qs, int& ev,
                           cudaStream_t caller) {
  auto next_event = [&]() { return qs->ring[ev++]; };
  const int ng = G.n;
  const size_t head_el = (size_t)N * d * 2, head_rows = (size_t)N * 4;
#define FA_TRY(x)                                   \
  do {                                              \
    const cudaError_t e_ = (x);                     \
    if (e_ != cudaSuccess) return FA_ERR_CUDA;      \
  } while (0)
  cudaEvent_t out_done[kMaxChunks] = {};
  for (int g = 0; g < ng; ++g) {
    const int64_t h0 = G.start[g], nh = G.start[g + 1] - h0;
    char* slot = static_cast<char*>(workspace) + (size_t)(g % kSlots) * L.bytes;
    const size_t el = (size_t)nh * head_el, rows = (size_t)nh * head_rows;
    const size_t off = (size_t)h0 * head_el, roff = (size_t)h0 * head_rows;
    // copy-in, once the slot's previous group has been copied out
    if (g >= kSlots) FA_TRY(cudaStreamWaitEvent(qs->in, out_done[g - kSlots], 0));
    FA_TRY(cudaMemcpyAsync(slot + L.q, static_cast<const char*>(Q) + off, el, cudaMemcpyHostToDevice, qs->in));
    FA_TRY(cudaMemcpyAsync(slot + L.k, static_cast<const char*>(K) + off, el, cudaMemcpyHostToDevice, qs->in));
    FA_TRY(cudaMemcpyAsync(slot + L.v, static_cast<const char*>(V) + off, el, cudaMemcpyHostToDevice, qs->in));
    cudaEvent_t qkv_in = next_event();
    FA_TRY(cudaEventRecord(qkv_in, qs->in));
    FA_TRY(cudaMemcpyAsync(slot + L.dO, static_cast<const char*>(dO) + off, el, cudaMemcpyHostToDevice, qs->in));
    cudaEvent_t do_in = next_event();
    FA_TRY(cudaEventRecord(do_in, qs->in));
    // compute (its outputs overwrite the slot's previous outputs, which copy-in already
    // waited for): the forward needs Q, K, V only
    cudaStream_t comp = qs->comp;
    FA_TRY(cudaStreamWaitEvent(comp, qkv_in, 0));
    const int nhi = (int)nh;
    fa_status_t r = fa_fwd(slot + L.q, slot + L.k, slot + L.v, slot + L.o, reinterpret_cast<float*>(slot + L.lse), 1,
                           nhi, N, d, scale, causal, dtype, comp);
    if (r != FA_OK) return r;
    cudaEvent_t fwd_done = next_event();
    FA_TRY(cudaEventRecord(fwd_done, comp));
    FA_TRY(cudaStreamWaitEvent(comp, do_in, 0));
    r = fa_bwd_preprocess(slot + L.o, slot + L.dO, reinterpret_cast<float*>(slot + L.D), 1, nhi, N, d, dtype, comp);
    if (r != FA_OK) return r;
    r = fa_bwd(slot + L.q, slot + L.k, slot + L.v, slot + L.o, slot + L.dO, reinterpret_cast<float*>(slot + L.lse),
               reinterpret_cast<float*>(slot + L.D), slot + L.dq, slot + L.dk, slot + L.dv, slot + L.acc,
               (size_t)nh * N * d * 4, 1, nhi, N, d, scale, causal, dtype, comp);
    if (r != FA_OK) return r;
    cudaEvent_t bwd_done = next_event();
    FA_TRY(cudaEventRecord(bwd_done, comp));
    // copy-out: O and LSE as soon as the forward is done, the gradients after the backward
    FA_TRY(cudaStreamWaitEvent(qs->out, fwd_done, 0));
    FA_TRY(cudaMemcpyAsync(static_cast<char*>(O) + off, slot + L.o, el, cudaMemcpyDeviceToHost, qs->out));
    FA_TRY(cudaMemcpyAsync(reinterpret_cast<char*>(LSE) + roff, slot + L.lse, rows, cudaMemcpyDeviceToHost, qs->out));
    FA_TRY(cudaStreamWaitEvent(qs->out, bwd_done, 0));
    FA_TRY(cudaMemcpyAsync(static_cast<char*>(dQ) + off, slot + L.dq, el, cudaMemcpyDeviceToHost, qs->out));
    FA_TRY(cudaMemcpyAsync(static_cast<char*>(dK) + off, slot + L.dk, el, cudaMemcpyDeviceToHost, qs->out));
    FA_TRY(cudaMemcpyAsync(static_cast<char*>(dV) + off, slot + L.dv, el, cudaMemcpyDeviceToHost, qs->out));
    out_done[g] = next_event();
    FA_TRY(cudaEventRecord(out_done[g], qs->out));
  }
  // join: the caller's stream continues after the last copy-out (which follows every
  // kernel and copy of the call)
  FA_TRY(cudaStreamWaitEvent(caller, out_done[ng - 1], 0));
#undef FA_TRY
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" fa_status_t fa_fwd_bwd_host(const void* Q, const void* K, const void* V, const void* dO, void* O,
                                       float* LSE, void* dQ, void* dK, void* dV, void* workspace,
                                       size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
                                       int dtype, int chunks, void* stream) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP32) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f && scale < INFINITY)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  for (const void* p : {Q, K, V, dO, (const void*)O, (const void*)LSE, (const void*)dQ, (const void*)dK,
                        (const void*)dV})
    if (!p) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 || (d != 64 && d != 128)) return FA_ERR_UNSUPPORTED;
  if ((int64_t)B * H * N > INT32_MAX) return FA_ERR_UNSUPPORTED;
  const size_t need = fa_fwd_bwd_host_workspace_size(B, H, N, d, dtype, chunks);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID_ARG;

  const fa::Groups G = fa::make_groups((int64_t)B * H, chunks);
  const fa::SlotLayout L = fa::slot_layout(G.largest, N, d);

  std::lock_guard<std::mutex> lock(fa::g_mu);
  fa::DeviceQueues* qs = fa::queues_for_current_device();
  if (!qs) return FA_ERR_CUDA;
  cudaStream_t caller = static_cast<cudaStream_t>(stream);
  int ev = 0;
  // fork: every internal stream starts after the work already queued on the caller's stream
  cudaEvent_t start = qs->ring[ev++];
  if (cudaEventRecord(start, caller) != cudaSuccess) return FA_ERR_CUDA;
  fa_status_t r = FA_OK;
  if (cudaStreamWaitEvent(qs->in, start, 0) != cudaSuccess || cudaStreamWaitEvent(qs->comp, start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(qs->out, start, 0) != cudaSuccess)
    r = FA_ERR_CUDA;
  if (r == FA_OK)
    r = fa::enqueue_groups(Q, K, V, dO, O, LSE, dQ, dK, dV, workspace, N, d, scale, causal, dtype, G, L, qs, ev,
                           caller);
  if (r != FA_OK) {
    // Work already enqueued on the internal streams keeps running after a failure: the
    // caller's stream waits for all of it, so that synchronising that stream before freeing
    // or reusing the buffers is safe even after an error.
    const cudaStream_t internal[fa::kJoinEvents] = {qs->in, qs->comp, qs->out};
    for (int i = 0; i < fa::kJoinEvents; ++i)
      if (cudaEventRecord(qs->join[i], internal[i]) == cudaSuccess) cudaStreamWaitEvent(caller, qs->join[i], 0);
  }
  return r;
}

