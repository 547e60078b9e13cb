// fa_backward_host: the backward pass for tensors that live in host memory.
//
// The B*H heads are independent (each head's dQ, dK, dV depend only on that
// head's Q, K, V, O, dO, L), so the batch is cut into groups of heads that
// stream through a caller-provided device workspace with three slots:
// while group c is computed on the caller's stream, group c+1 is copied in on
// one internal stream and group c-1 is copied out on another.  Host buffers
// should be page-locked, or the copies cannot overlap.

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kSlots = 3;
constexpr int kMaxDevices = 64;

struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t ev_in[kSlots] = {}, ev_comp[kSlots] = {}, ev_out[kSlots] = {};
  bool ready = false;
};
std::mutex g_mu;
HostPipe g_pipe[kMaxDevices];
// One call at a time per device: the streams and events above are shared, and
// a second host thread re-recording ev_comp[s] between another call's record
// and its wait would make that call copy out the wrong group's results.
std::mutex g_call_mu[kMaxDevices];

// Streams and events are created once per device and reused by every call.
HostPipe* pipe_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  HostPipe& hp = g_pipe[dev];
  if (hp.ready) return &hp;
  const unsigned f = cudaEventDisableTiming;
  bool ok = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&hp.start, f) == cudaSuccess && cudaEventCreateWithFlags(&hp.done, f) == cudaSuccess;
  for (int s = 0; ok && s < kSlots; ++s)
    ok = cudaEventCreateWithFlags(&hp.ev_in[s], f) == cudaSuccess &&
         cudaEventCreateWithFlags(&hp.ev_comp[s], f) == cudaSuccess &&
         cudaEventCreateWithFlags(&hp.ev_out[s], f) == cudaSuccess;
  if (!ok) {  // release whatever was created; the next call tries again
    for (cudaEvent_t* ev : {&hp.start, &hp.done})
      if (*ev) cudaEventDestroy(*ev);
    for (int s = 0; s < kSlots; ++s)
      for (cudaEvent_t ev : {hp.ev_in[s], hp.ev_comp[s], hp.ev_out[s]})
        if (ev) cudaEventDestroy(ev);
    if (hp.in) cudaStreamDestroy(hp.in);
    if (hp.out) cudaStreamDestroy(hp.out);
    hp = HostPipe();
    return nullptr;
  }
  hp.ready = true;
  return &hp;
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Byte offsets of one slot's buffers for a group of `g` heads.
struct SlotLayout {
  size_t q, k, v, o, dO, dq, dk, dv, L, D, acc, bytes;
};
// p is normalised (N_k set).
SlotLayout slot_layout(const fa_problem& p, int g) {
  const size_t es = p.dtype == FA_BF16 ? 2 : 4;
  const size_t qhead = (size_t)p.N * p.d * es, khead = (size_t)p.N_k * p.d * es;
  const size_t rows = (size_t)g * p.N * 4;
  const size_t acc = (size_t)g * ceil_div(p.N, kTileRows) * kTileRows * p.d * 4 * dq_slices(p);
  SlotLayout s;
  size_t off = 0;
  for (size_t* f : {&s.q, &s.k, &s.v, &s.o, &s.dO, &s.dq, &s.dk, &s.dv}) {
    *f = off;
    const bool kshaped = f == &s.k || f == &s.v || f == &s.dk || f == &s.dv;
    off += align256(g * (kshaped ? khead : qhead));
  }
  s.L = off;
  off += align256(rows);
  s.D = off;
  off += align256(rows);
  s.acc = off;
  off += align256(acc);
  s.bytes = off;
  return s;
}

int default_group(const fa_problem& p) {
  const int heads = p.B * p.H;
  // about eight groups: the copies in are the bound, and smaller groups
  // shorten the tail (the last group's compute and copy out) until the
  // per-group launches stop filling the GPU (measured on 1x32x8192x128:
  // 4 heads per group 2.36 ms, 8 heads 2.45 ms, 3 heads 2.44 ms)
  return heads <= 4 ? 1 : (heads + 7) / 8;
}

}  // namespace
}  // namespace fa

extern "C" {

size_t fa_backward_host_workspace_bytes(const fa_problem* p, int32_t heads_per_group) {
  fa_problem pn;
  if (!fa::normalize_problem(p, &pn)) return 0;
  const int g = heads_per_group > 0 ? heads_per_group : fa::default_group(pn);
  return fa::kSlots * fa::slot_layout(pn, g).bytes;
}

fa_status fa_backward_host(const fa_problem* p, const void* hQ, const void* hK, const void* hV, const void* hO,
                           const void* hdO, const float* hL, void* hdQ, void* hdK, void* hdV, void* workspace,
                           size_t workspace_bytes, int32_t heads_per_group, void* stream) {
  fa::NvtxRange range("fa_backward_host");
  fa_problem pn;
  if (!fa::normalize_problem(p, &pn)) return p ? FA_ERR_UNSUPPORTED : FA_ERR_INVALID_ARG;
  if (!hQ || !hK || !hV || !hO || !hdO || !hL || !hdQ || !hdK || !hdV || !workspace) return FA_ERR_INVALID_ARG;
  if (heads_per_group < 0) return FA_ERR_INVALID_ARG;
  // host tensors are dense [B, H, N, d] and [B, H, N_k, d]
  if (pn.stride_n != pn.d || pn.stride_h != (int64_t)pn.N * pn.d || pn.stride_b != (int64_t)pn.H * pn.N * pn.d ||
      pn.kstride_n != pn.d || pn.kstride_h != (int64_t)pn.N_k * pn.d ||
      pn.kstride_b != (int64_t)pn.H * pn.N_k * pn.d)
    return FA_ERR_INVALID_ARG;
  const int heads = pn.B * pn.H;
  const int g = heads_per_group > 0 ? (heads_per_group < heads ? heads_per_group : heads) : fa::default_group(pn);
  const fa::SlotLayout lay = fa::slot_layout(pn, g);
  if (workspace_bytes < fa::kSlots * lay.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return FA_ERR_INVALID_ARG;
  fa::HostPipe* hp = fa::pipe_for_current_device();
  if (!hp) return FA_ERR_CUDA;
  // held from the first record to the final join, so that concurrent calls on
  // one device enqueue one after the other
  std::lock_guard<std::mutex> call_lock(fa::g_call_mu[hp - fa::g_pipe]);
  cudaStream_t cs = (cudaStream_t)stream;
  const size_t es = pn.dtype == FA_BF16 ? 2 : 4;
  const size_t qhead_bytes = (size_t)pn.N * pn.d * es, khead_bytes = (size_t)pn.N_k * pn.d * es;
  const size_t row_bytes = (size_t)pn.N * 4;
  auto H2D = cudaMemcpyHostToDevice;
  auto D2H = cudaMemcpyDeviceToHost;

  cudaError_t e = cudaEventRecord(hp->start, cs);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->in, hp->start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->out, hp->start, 0);
  const int groups = (heads + g - 1) / g;
  fa_status st = FA_OK;
  for (int c = 0; c < groups && e == cudaSuccess; ++c) {
    const int s = c % fa::kSlots;
    const int h0 = c * g;
    const int gh = heads - h0 < g ? heads - h0 : g;
    uint8_t* base = static_cast<uint8_t*>(workspace) + s * lay.bytes;
    const size_t qoff = (size_t)h0 * qhead_bytes, qn = (size_t)gh * qhead_bytes;
    const size_t koff = (size_t)h0 * khead_bytes, kn = (size_t)gh * khead_bytes;
    // copy in (the slot's previous group must have been copied out)
    if (c >= fa::kSlots) e = cudaStreamWaitEvent(hp->in, hp->ev_out[s], 0);
    const void* srcs[5] = {hQ, hK, hV, hO, hdO};
    const size_t dsts[5] = {lay.q, lay.k, lay.v, lay.o, lay.dO};
    const bool ksh[5] = {false, true, true, false, false};
    for (int t = 0; t < 5 && e == cudaSuccess; ++t)
      e = cudaMemcpyAsync(base + dsts[t], static_cast<const uint8_t*>(srcs[t]) + (ksh[t] ? koff : qoff),
                          ksh[t] ? kn : qn, H2D, hp->in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(base + lay.L, reinterpret_cast<const uint8_t*>(hL) + (size_t)h0 * row_bytes,
                          (size_t)gh * row_bytes, H2D, hp->in);
    if (e == cudaSuccess) e = cudaEventRecord(hp->ev_in[s], hp->in);
    // compute on the caller's stream
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, hp->ev_in[s], 0);
    if (e != cudaSuccess) break;
    fa_problem pc = pn;  // the group: B = 1, H = gh, dense slots
    pc.B = 1;
    pc.H = gh;
    pc.stride_n = pn.d;
    pc.stride_h = (int64_t)pn.N * pn.d;
    pc.stride_b = (int64_t)gh * pn.N * pn.d;
    pc.kstride_n = pn.d;
    pc.kstride_h = (int64_t)pn.N_k * pn.d;
    pc.kstride_b = (int64_t)gh * pn.N_k * pn.d;
    st = fa_backward(&pc, base + lay.q, base + lay.k, base + lay.v, base + lay.o, base + lay.dO,
                     reinterpret_cast<const float*>(base + lay.L), reinterpret_cast<float*>(base + lay.D),
                     reinterpret_cast<float*>(base + lay.acc), base + lay.dq, base + lay.dk, base + lay.dv, cs);
    if (st != FA_OK) break;
    e = cudaEventRecord(hp->ev_comp[s], cs);
    // copy out
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->out, hp->ev_comp[s], 0);
    void* outs[3] = {hdQ, hdK, hdV};
    const size_t srcs_out[3] = {lay.dq, lay.dk, lay.dv};
    for (int t = 0; t < 3 && e == cudaSuccess; ++t)
      e = cudaMemcpyAsync(static_cast<uint8_t*>(outs[t]) + (t ? koff : qoff), base + srcs_out[t], t ? kn : qn, D2H,
                          hp->out);
    if (e == cudaSuccess) e = cudaEventRecord(hp->ev_out[s], hp->out);
  }
  // The caller's stream continues only after the last copy out, also when a
  // group failed, so that no copy of this call is still running when the
  // caller reuses or frees its buffers.
  cudaError_t j = cudaEventRecord(hp->done, hp->in);
  if (j == cudaSuccess) j = cudaStreamWaitEvent(cs, hp->done, 0);
  if (j == cudaSuccess) j = cudaEventRecord(hp->done, hp->out);
  if (j == cudaSuccess) j = cudaStreamWaitEvent(cs, hp->done, 0);
  if (st != FA_OK) return st;
  return e == cudaSuccess && j == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
