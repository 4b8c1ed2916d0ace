// ckda_host.cu -- the forward over host buffers.
//
// The token axis is cut into slices of a multiple of 64 tokens.  Slice s is
// copied in (one 2-D copy per input: B*H rows of the slice's tokens) on one
// stream while slice s-1 is computed on the caller's stream and slice s-2's
// o is copied out on a third, through two device buffers.  Every (sequence,
// head) carries its fp32 state from slice to slice in device memory (the
// forward's h0 -> hT, which may alias); slice boundaries fall on chunk
// boundaries, so the result is the same as one ckda_fwd over the whole
// sequence.
#include "ckda_internal.cuh"

#include <mutex>

namespace ckda {
namespace {

constexpr int kBufs = 2;
constexpr int kMaxDevices = 64;

struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, fin = nullptr;
  cudaEvent_t in_done[kBufs] = {}, comp_done[kBufs] = {}, out_done[kBufs] = {};
  bool ready = false;
};
std::mutex g_mu;
HostPipe g_pipe[kMaxDevices];

// The copy streams and events of the current device, created on first use.
ckda_status pipe_for_current_device(HostPipe** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CKDA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CKDA_ERR_UNSUPPORTED;
  HostPipe& p = g_pipe[dev];
  if (!p.ready) {
    bool ok = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.fin, cudaEventDisableTiming) == cudaSuccess;
    for (int b = 0; ok && b < kBufs; ++b)
      ok = cudaEventCreateWithFlags(&p.in_done[b], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&p.comp_done[b], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&p.out_done[b], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) return CKDA_ERR_CUDA;
    p.ready = true;
  }
  *out = &p;
  return CKDA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Byte offsets within the caller's scratch: the status word, the carried
// state, then kBufs slice buffers of q, k, alpha, v, beta and o.
struct Layout {
  size_t state;
  size_t q, k, a, v, b, o;  // within one slice buffer
  size_t buf0, buf_bytes, total;
};
Layout make_layout(int B, int H, int Ts, int dk, int dv, size_t es) {
  Layout L{};
  const size_t rows = (size_t)B * H * Ts;
  size_t off = kWsStatusBytes;
  L.state = off;
  off = align256(off + (size_t)B * H * dk * dv * sizeof(float));
  size_t in = 0;
  L.q = in; in = align256(in + rows * dk * es);
  L.k = in; in = align256(in + rows * dk * es);
  L.a = in; in = align256(in + rows * dk * es);
  L.v = in; in = align256(in + rows * dv * es);
  L.b = in; in = align256(in + rows * es);
  L.o = in; in = align256(in + rows * dv * es);
  L.buf0 = off;
  L.buf_bytes = in;
  L.total = off + kBufs * in;
  return L;
}

// Slice length: the caller's (a multiple of 64), else about a quarter of the
// sequence, at least 512 tokens (shorter slices make the 2-D copies, B*H rows
// each, too fine to run at full copy bandwidth).
int slice_length(int T, int slice_tokens) {
  if (slice_tokens > 0) return slice_tokens;
  int ts = ((T + 3) / 4 + 63) / 64 * 64;
  ts = ts < 512 ? 512 : ts;
  return T < ts ? ((T + 63) / 64) * 64 : ts;
}

}  // namespace
}  // namespace ckda

extern "C" size_t ckda_fwd_host_scratch_bytes(int B, int H, int T, int dk, int dv,
                                              ckda_dtype io_dtype, int slice_tokens) {
  using namespace ckda;
  if (B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1 || slice_tokens < 0 || (slice_tokens % 64) != 0)
    return 0;
  const size_t es = io_dtype == CKDA_BF16 ? 2 : 4;
  return make_layout(B, H, slice_length(T, slice_tokens), dk, dv, es).total;
}

extern "C" ckda_status ckda_fwd_host(const void* q, const void* k, const void* v,
                                     const void* alpha, const void* beta, const float* h0,
                                     void* o, float* hT, int B, int H, int T, int dk, int dv,
                                     ckda_dtype io_dtype, float scale, int slice_tokens,
                                     void* dev_scratch, size_t dev_scratch_bytes, void* stream) {
  using namespace ckda;
  if (io_dtype != CKDA_F32 && io_dtype != CKDA_BF16) return CKDA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1) return CKDA_ERR_INVALID_ARG;
  if (slice_tokens < 0 || (slice_tokens % 64) != 0) return CKDA_ERR_INVALID_ARG;
  if ((long long)B * H * T > 0x7fffffffLL) return CKDA_ERR_UNSUPPORTED;
  if (!(scale == scale)) return CKDA_ERR_INVALID_ARG;
  if (T > 0 && (!q || !k || !v || !alpha || !beta || !o)) return CKDA_ERR_INVALID_ARG;
  if (dk > 128 || dv > 128) return CKDA_ERR_UNSUPPORTED;
  const size_t es = io_dtype == CKDA_BF16 ? 2 : 4;
  const int Ts = slice_length(T, slice_tokens);
  const Layout L = make_layout(B, H, Ts, dk, dv, es);
  if (!dev_scratch || dev_scratch_bytes < L.total) return CKDA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(dev_scratch) & 255) != 0) return CKDA_ERR_WORKSPACE;

  std::lock_guard<std::mutex> lock(g_mu);  // the copy streams and events are shared
  HostPipe* P = nullptr;
  if (ckda_status st = pipe_for_current_device(&P); st != CKDA_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(dev_scratch);
  int* status = reinterpret_cast<int*>(base);
  float* state = reinterpret_cast<float*>(base + L.state);
  const bool tensor_path = fwd_tensor_path(io_dtype, dk, dv);
  const size_t units = (size_t)B * H;

#define CK(call)                                  \
  do {                                            \
    if ((call) != cudaSuccess) return CKDA_ERR_CUDA; \
  } while (0)
  CK(cudaMemsetAsync(status, 0, sizeof(int), cs));
  CK(cudaEventRecord(P->start, cs));
  CK(cudaStreamWaitEvent(P->in, P->start, 0));
  CK(cudaStreamWaitEvent(P->out, P->start, 0));
  if (h0)
    CK(cudaMemcpyAsync(state, h0, units * dk * dv * sizeof(float), cudaMemcpyHostToDevice, P->in));

  const int nslices = (T + Ts - 1) / Ts;
  for (int s = 0; s < nslices; ++s) {
    const int b = s % kBufs;
    const int t0 = s * Ts, len = T - t0 < Ts ? T - t0 : Ts;
    char* buf = base + L.buf0 + b * L.buf_bytes;
    // in: the buffer's previous slice must be computed before it is overwritten
    if (s >= kBufs) CK(cudaStreamWaitEvent(P->in, P->comp_done[b], 0));
    auto copy_in = [&](size_t dst_off, const void* src, int d) {
      const size_t row = (size_t)len * d * es;
      return cudaMemcpy2DAsync(buf + dst_off, row, static_cast<const char*>(src) + (size_t)t0 * d * es,
                               (size_t)T * d * es, row, units, cudaMemcpyHostToDevice, P->in);
    };
    CK(copy_in(L.q, q, dk));
    CK(copy_in(L.k, k, dk));
    CK(copy_in(L.a, alpha, dk));
    CK(copy_in(L.v, v, dv));
    CK(copy_in(L.b, beta, 1));
    CK(cudaEventRecord(P->in_done[b], P->in));
    // compute: on the caller's stream, once the slice is in and the buffer's
    // previous o has been copied out
    CK(cudaStreamWaitEvent(cs, P->in_done[b], 0));
    if (s >= kBufs) CK(cudaStreamWaitEvent(cs, P->out_done[b], 0));
    FwdArgs a{};
    a.q = buf + L.q; a.k = buf + L.k; a.alpha = buf + L.a; a.v = buf + L.v; a.beta = buf + L.b;
    a.o = buf + L.o;
    a.h0 = (s == 0 && !h0) ? nullptr : state;
    a.hT = state;
    a.cu_seqlens = nullptr;
    a.order = nullptr;
    a.status = status;
    a.num_units_seq = B;
    a.B = B; a.H = H; a.T = len; a.dk = dk; a.dv = dv;
    a.scale = scale; a.io = io_dtype;
    CK(tensor_path ? launch_fwd(a, cs) : launch_fwd_recurrent(a, cs));
    CK(cudaEventRecord(P->comp_done[b], cs));
    // out: o of this slice into its rows of the host o
    CK(cudaStreamWaitEvent(P->out, P->comp_done[b], 0));
    const size_t orow = (size_t)len * dv * es;
    CK(cudaMemcpy2DAsync(static_cast<char*>(o) + (size_t)t0 * dv * es, (size_t)T * dv * es,
                         buf + L.o, orow, orow, units, cudaMemcpyDeviceToHost, P->out));
    CK(cudaEventRecord(P->out_done[b], P->out));
  }
  if (hT) {
    if (nslices == 0) {  // no tokens: the final state is h0 (or zero)
      if (h0)
        CK(cudaMemcpyAsync(hT, h0, units * dk * dv * sizeof(float), cudaMemcpyHostToHost, P->out));
      else
        CK(cudaMemsetAsync(state, 0, units * dk * dv * sizeof(float), P->out));
    }
    if (nslices > 0 || !h0)
      CK(cudaMemcpyAsync(hT, state, units * dk * dv * sizeof(float), cudaMemcpyDeviceToHost, P->out));
  }
  CK(cudaEventRecord(P->fin, P->out));
  CK(cudaStreamWaitEvent(cs, P->fin, 0));
#undef CK
  return CKDA_OK;
}
