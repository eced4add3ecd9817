// Forward + backward between host buffers (flashmask_fwd_bwd_host): the
// classification, forward and backward of the C ABI run chunk by chunk over
// groups of heads, with the copies in and out of each chunk overlapped with the
// kernels of its neighbours on three streams. Nothing here allocates device
// memory: the three chunk slots are carved from the caller's workspace.
#include <cmath>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "flashmask.h"

namespace {

constexpr int kSlots = 3;        // chunk c uses slot c % 3: copy-in, kernels, copy-out in flight
constexpr int kMaxDevices = 256;

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Heads [h0, h0 + ch) of one batch entry read whole mask heads: either the chunk
// lies inside one group of H / Hm heads, or it covers whole groups.
bool chunk_ok(int H, int Hm, int ch) {
  if (ch <= 0 || H % ch != 0) return false;
  const int G = H / Hm;
  return (G % ch == 0) || (ch % G == 0);
}
int chunk_mask_heads(int H, int Hm, int ch) {
  const int G = H / Hm;
  return ch >= G ? ch / G : 1;
}

// Byte offsets inside one slot.
struct Slot {
  size_t q, k, v, dout, o, dq, dk, dv, lse, lts, lte, uts, ute, ws, ws_bytes, total;
};

Slot slot_layout(int ch, int Hmc, int N, int d) {
  Slot s;
  const size_t t = static_cast<size_t>(ch) * N * d * 2;  // one bf16 [ch, N, d] tensor
  const size_t m = static_cast<size_t>(Hmc) * N * 4;     // one int32 [Hmc, N] bound vector
  size_t off = 0;
  size_t* tens[8] = {&s.q, &s.k, &s.v, &s.dout, &s.o, &s.dq, &s.dk, &s.dv};
  for (size_t* p : tens) {
    *p = off;
    off += up256(t);
  }
  s.lse = off;
  off += up256(static_cast<size_t>(ch) * N * 4);
  size_t* bounds[4] = {&s.lts, &s.lte, &s.uts, &s.ute};
  for (size_t* p : bounds) {
    *p = off;
    off += up256(m);
  }
  s.ws = off;
  s.ws_bytes = flashmask_workspace_bytes(1, ch, Hmc, N, d, 1);
  off += up256(s.ws_bytes);
  s.total = off;
  return s;
}

// Streams and events of one device, made on first use and kept.
struct DeviceState {
  std::mutex lock;  // one pipelined call per device at a time
  bool ready = false;
  cudaStream_t in = nullptr, work = nullptr, out = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t copied_in[kSlots] = {}, computed[kSlots] = {}, copied_out[kSlots] = {};
};
DeviceState g_dev[kMaxDevices];
std::mutex g_init;

fm_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FM_ERR_UNSUPPORTED;
  DeviceState& st = g_dev[dev];
  std::lock_guard<std::mutex> g(g_init);
  if (!st.ready) {
    const unsigned ev = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&st.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&st.work, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&st.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&st.start, ev) == cudaSuccess;
    for (int s = 0; ok && s < kSlots; ++s)
      ok = cudaEventCreateWithFlags(&st.copied_in[s], ev) == cudaSuccess &&
           cudaEventCreateWithFlags(&st.computed[s], ev) == cudaSuccess &&
           cudaEventCreateWithFlags(&st.copied_out[s], ev) == cudaSuccess;
    if (!ok) return FM_ERR_CUDA;
    st.ready = true;
  }
  *out = &st;
  return FM_OK;
}

}  // namespace

extern "C" {

size_t flashmask_host_workspace_bytes(int B, int H, int Hm, int N, int d, int chunk_heads) {
  if (flashmask_workspace_bytes(B, H, Hm, N, d, 1) == 0) return 0;  // unsupported shape
  if (!chunk_ok(H, Hm, chunk_heads)) return 0;
  const Slot s = slot_layout(chunk_heads, chunk_mask_heads(H, Hm, chunk_heads), N, d);
  return kSlots * s.total;
}

fm_status flashmask_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dout,
                                 const fm_mask* mask, int B, int H, int N, int d, float scale,
                                 void* o, float* lse, void* dq, void* dk, void* dv, void* dev_ws,
                                 size_t ws_bytes, int chunk_heads, void* stream) {
  if (!q || !k || !v || !dout || !o || !lse || !dq || !dk || !dv || !mask) return FM_ERR_INVALID_ARG;
  if (!mask->lts || !mask->lte || ((mask->uts == nullptr) != (mask->ute == nullptr)))
    return FM_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FM_ERR_INVALID_ARG;
  const int Hm = mask->Hm;
  if (Hm <= 0 || flashmask_workspace_bytes(B, H, Hm, N, d, 1) == 0) return FM_ERR_UNSUPPORTED;
  if (!chunk_ok(H, Hm, chunk_heads)) return FM_ERR_UNSUPPORTED;
  const int ch = chunk_heads, G = H / Hm, Hmc = chunk_mask_heads(H, Hm, ch);
  const Slot L = slot_layout(ch, Hmc, N, d);
  if (!dev_ws || (reinterpret_cast<uintptr_t>(dev_ws) & 255u) != 0 || ws_bytes < kSlots * L.total)
    return FM_ERR_WORKSPACE;

  DeviceState* st = nullptr;
  fm_status rc = device_state(&st);
  if (rc != FM_OK) return rc;
  std::lock_guard<std::mutex> g(st->lock);

  // everything below runs after the work already queued on the caller's stream
  cudaStream_t caller = static_cast<cudaStream_t>(stream);
  if (cudaEventRecord(st->start, caller) != cudaSuccess) return FM_ERR_CUDA;
  for (cudaStream_t s : {st->in, st->work, st->out})
    if (cudaStreamWaitEvent(s, st->start, 0) != cudaSuccess) return FM_ERR_CUDA;

  // each slot's device status word (at the start of its workspace) starts at zero
  for (int s = 0; s < kSlots; ++s)
    if (cudaMemsetAsync(static_cast<char*>(dev_ws) + s * L.total + L.ws, 0, 16, st->work) !=
        cudaSuccess)
      return FM_ERR_CUDA;

  const size_t tb = static_cast<size_t>(ch) * N * d * 2;  // bytes of one chunk tensor
  const size_t lb = static_cast<size_t>(ch) * N * 4;      // bytes of one chunk's LSE
  const size_t mb = static_cast<size_t>(Hmc) * N * 4;     // bytes of one chunk bound vector
  const int per_b = H / ch, nchunks = B * per_b;
  long long held[kSlots][2];  // (batch, first mask head) whose mask slot s holds, or -1
  for (auto& h : held) h[0] = h[1] = -1;
  const cudaMemcpyKind H2D = cudaMemcpyHostToDevice, D2H = cudaMemcpyDeviceToHost;
  bool cuda_ok = true;

  for (int c = 0; c < nchunks && cuda_ok && rc == FM_OK; ++c) {
    const int s = c % kSlots, b = c / per_b, h0 = (c % per_b) * ch, hm0 = h0 / G;
    char* base = static_cast<char*>(dev_ws) + s * L.total;
    const size_t head0 = static_cast<size_t>(b) * H + h0;  // first [N, d] head of the chunk
    const size_t toff = head0 * N * d * 2, loff = head0 * N;
    const size_t moff = (static_cast<size_t>(b) * Hm + hm0) * N;
    const bool new_mask = held[s][0] != b || held[s][1] != hm0;

    // copy in (after the slot's previous chunk has been copied out)
    if (c >= kSlots) cuda_ok = cudaStreamWaitEvent(st->in, st->copied_out[s], 0) == cudaSuccess;
    const void* srcs[4] = {q, k, v, dout};
    const size_t dsts[4] = {L.q, L.k, L.v, L.dout};
    for (int i = 0; i < 4 && cuda_ok; ++i)
      cuda_ok = cudaMemcpyAsync(base + dsts[i], static_cast<const char*>(srcs[i]) + toff, tb, H2D,
                                st->in) == cudaSuccess;
    if (new_mask) {
      const int32_t* msrc[4] = {mask->lts, mask->lte, mask->uts, mask->ute};
      const size_t mdst[4] = {L.lts, L.lte, L.uts, L.ute};
      for (int i = 0; i < 4 && cuda_ok; ++i)
        if (msrc[i])
          cuda_ok = cudaMemcpyAsync(base + mdst[i], msrc[i] + moff, mb, H2D, st->in) == cudaSuccess;
    }
    if (cuda_ok) cuda_ok = cudaEventRecord(st->copied_in[s], st->in) == cudaSuccess;

    // kernels
    if (cuda_ok) cuda_ok = cudaStreamWaitEvent(st->work, st->copied_in[s], 0) == cudaSuccess;
    if (!cuda_ok) break;
    fm_mask dm;
    dm.lts = reinterpret_cast<const int32_t*>(base + L.lts);
    dm.lte = reinterpret_cast<const int32_t*>(base + L.lte);
    dm.uts = mask->uts ? reinterpret_cast<const int32_t*>(base + L.uts) : nullptr;
    dm.ute = mask->ute ? reinterpret_cast<const int32_t*>(base + L.ute) : nullptr;
    dm.Hm = Hmc;
    dm.causal = mask->causal;
    void* ws = base + L.ws;
    void* w = st->work;
    char* dq_d = base + L.dq;
    float* lse_d = reinterpret_cast<float*>(base + L.lse);
    if (new_mask) rc = flashmask_classify(&dm, 1, N, ws, L.ws_bytes, w);
    if (rc == FM_OK)
      rc = flashmask_fwd(base + L.q, base + L.k, base + L.v, &dm, 1, ch, N, d, scale, base + L.o,
                         lse_d, ws, L.ws_bytes, 1, w);
    if (rc == FM_OK)
      rc = flashmask_bwd_preprocess(base + L.o, lse_d, base + L.dout, 1, ch, Hmc, N, d, ws,
                                    L.ws_bytes, w);
    if (rc == FM_OK)
      rc = flashmask_bwd_main(base + L.q, base + L.k, base + L.v, base + L.dout, &dm, 1, ch, N, d,
                              scale, base + L.dk, base + L.dv, ws, L.ws_bytes, w);
    if (rc == FM_OK)
      rc = flashmask_bwd_finalize(1, ch, Hmc, N, d, scale, dq_d, ws, L.ws_bytes, w);
    if (rc != FM_OK) break;
    held[s][0] = b;
    held[s][1] = hm0;
    cuda_ok = cudaEventRecord(st->computed[s], st->work) == cudaSuccess;

    // copy out
    if (cuda_ok) cuda_ok = cudaStreamWaitEvent(st->out, st->computed[s], 0) == cudaSuccess;
    void* outs[4] = {o, dq, dk, dv};
    const size_t srco[4] = {L.o, L.dq, L.dk, L.dv};
    for (int i = 0; i < 4 && cuda_ok; ++i)
      cuda_ok = cudaMemcpyAsync(static_cast<char*>(outs[i]) + toff, base + srco[i], tb, D2H,
                                st->out) == cudaSuccess;
    if (cuda_ok)
      cuda_ok = cudaMemcpyAsync(lse + loff, base + L.lse, lb, D2H, st->out) == cudaSuccess;
    if (cuda_ok) cuda_ok = cudaEventRecord(st->copied_out[s], st->out) == cudaSuccess;
  }

  // wait for everything queued, then read (and clear) each used slot's status word
  const bool synced = cudaStreamSynchronize(st->in) == cudaSuccess &&
                      cudaStreamSynchronize(st->work) == cudaSuccess &&
                      cudaStreamSynchronize(st->out) == cudaSuccess;
  if (rc != FM_OK) return rc;
  if (!cuda_ok || !synced) return FM_ERR_CUDA;
  for (int s = 0; s < kSlots && s < nchunks; ++s) {
    const fm_status cs =
        flashmask_check_status(static_cast<char*>(dev_ws) + s * L.total + L.ws, st->work, nullptr);
    if (cs != FM_OK) return cs;
  }
  return FM_OK;
}

}  // extern "C"
