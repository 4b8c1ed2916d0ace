// ckda_api.cu -- the C ABI of libckda: argument validation, dispatch to the
// kernels, the workspace status word, the longest-first order of packed
// sequences and the bounded-wait self-test.
#include "ckda_internal.cuh"
#include "sm103.cuh"

namespace ckda {
namespace {

// Rank of each packed sequence by length, longest first (ties by index):
// order[rank] = sequence.  One block; O(n^2 / threads) work, used up to
// kMaxRankSeqs sequences; longer lists keep their natural order.
constexpr int kMaxRankSeqs = 16384;

__global__ void seq_order_kernel(const int32_t* cu, int n, int32_t* order) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int li = cu[i + 1] - cu[i];
    int rank = 0;
    for (int j = 0; j < n; ++j) {
      const int lj = cu[j + 1] - cu[j];
      rank += (lj > li) || (lj == li && j < i);
    }
    order[rank] = i;
  }
}

__global__ void seq_order_identity_kernel(int n, int32_t* order) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    order[i] = i;
}

// Waits on an mbarrier that no one will ever complete, with a bounded number
// of polls, then records CKDA_ERR_TIMEOUT.  Exercises the same bounded wait
// the tensor-core kernel uses, without hanging.
__global__ void selftest_timeout_kernel(int* status, unsigned spin_limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  bool ok = mbar_wait(&bar, 0, spin_limit, 1000u);
  if (!ok && threadIdx.x == 0) set_status(status, CKDA_ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_seq_order(const int32_t* cu, int n, int32_t* order, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (n <= kMaxRankSeqs)
    seq_order_kernel<<<1, 1024, 0, s>>>(cu, n, order);
  else
    seq_order_identity_kernel<<<(n + 255) / 256, 256, 0, s>>>(n, order);
  return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(int* status, unsigned spin_limit, cudaStream_t s) {
  selftest_timeout_kernel<<<1, 32, 0, s>>>(status, spin_limit);
  return cudaGetLastError();
}

}  // namespace ckda

using namespace ckda;

extern "C" {

int ckda_version(void) { return 10000; }

const char* ckda_status_string(ckda_status s) {
  switch (s) {
    case CKDA_OK: return "CKDA_OK";
    case CKDA_ERR_INVALID_ARG: return "CKDA_ERR_INVALID_ARG";
    case CKDA_ERR_UNSUPPORTED: return "CKDA_ERR_UNSUPPORTED";
    case CKDA_ERR_CUDA: return "CKDA_ERR_CUDA";
    case CKDA_ERR_TIMEOUT: return "CKDA_ERR_TIMEOUT";
    case CKDA_ERR_WORKSPACE: return "CKDA_ERR_WORKSPACE";
    case CKDA_ERR_RANGE: return "CKDA_ERR_RANGE";
  }
  return "CKDA_ERR_UNKNOWN";
}

size_t ckda_fwd_workspace_bytes(int num_seqs, int H) {
  (void)H;
  size_t n = num_seqs > 0 ? (size_t)num_seqs : 0;
  return kWsStatusBytes + ((n * sizeof(int32_t) + 255) / 256) * 256;
}

}  // extern "C"

namespace {

// ckda_fwd, and with raw = 1 ckda_fwd_raw (tensor-core shapes only).
ckda_status fwd_impl(const void* q, const void* k, const void* v, const void* alpha,
                     const void* beta, const float* h0, void* o, float* hT,
                     const int32_t* cu_seqlens, int num_seqs, int B, int H, int T, int dk,
                     int dv, ckda_dtype io_dtype, float scale, int chunk_size, void* workspace,
                     size_t workspace_bytes, void* stream, int raw, int normalize_q,
                     float norm_eps) {
  if (io_dtype != CKDA_F32 && io_dtype != CKDA_BF16) return CKDA_ERR_INVALID_ARG;
  if (raw && (!(norm_eps >= 0.f) || norm_eps > 3.0e38f)) return CKDA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1) return CKDA_ERR_INVALID_ARG;
  if ((long long)B * H * T > 0x7fffffffLL) return CKDA_ERR_UNSUPPORTED;
  if (!(scale == scale)) return CKDA_ERR_INVALID_ARG;
  if (cu_seqlens) {
    if (B != 1 || num_seqs < 1) return CKDA_ERR_INVALID_ARG;
  } else if (num_seqs != 0 && num_seqs != B) {
    return CKDA_ERR_INVALID_ARG;
  }
  if (T > 0 && (!q || !k || !v || !alpha || !beta || !o)) return CKDA_ERR_INVALID_ARG;
  if (dk > 128 || dv > 128) return CKDA_ERR_UNSUPPORTED;
  if (chunk_size != 0 && chunk_size != 16 && chunk_size != 32 && chunk_size != 64)
    return CKDA_ERR_UNSUPPORTED;
  const bool tensor_path = fwd_tensor_path(io_dtype, dk, dv);
  if (raw && !tensor_path) return CKDA_ERR_UNSUPPORTED;
  if (tensor_path && chunk_size != 0 && chunk_size != 64) return CKDA_ERR_UNSUPPORTED;
  const int nseq = cu_seqlens ? num_seqs : B;
  const size_t need = ckda_fwd_workspace_bytes(cu_seqlens ? num_seqs : 0, H);
  if (!workspace || workspace_bytes < need) return CKDA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return CKDA_ERR_WORKSPACE;
  if (tensor_path) {
    // TMA needs 16-byte aligned bases
    const void* ptrs[4] = {q, k, v, alpha};
    for (const void* p : ptrs)
      if (T > 0 && (reinterpret_cast<uintptr_t>(p) & 15) != 0) return CKDA_ERR_INVALID_ARG;
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(workspace);
  int32_t* order = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + kWsStatusBytes);

  FwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta;
  a.h0 = h0; a.o = o; a.hT = hT;
  a.cu_seqlens = cu_seqlens;
  a.order = nullptr;
  a.status = status;
  a.num_units_seq = nseq;
  a.B = B; a.H = H; a.T = T; a.dk = dk; a.dv = dv;
  a.scale = scale; a.io = io_dtype;
  a.raw = raw;
  a.normalize_q = normalize_q;
  a.norm_eps = norm_eps;

  cudaError_t err = cudaMemsetAsync(status, 0, sizeof(int), s);
  if (err != cudaSuccess) return CKDA_ERR_CUDA;
  if (tensor_path && cu_seqlens) {
    err = launch_seq_order(cu_seqlens, num_seqs, order, s);
    if (err != cudaSuccess) return CKDA_ERR_CUDA;
    a.order = order;
  }
  err = tensor_path ? launch_fwd(a, s) : launch_fwd_recurrent(a, s);
  return err == cudaSuccess ? CKDA_OK : CKDA_ERR_CUDA;
}

}  // namespace

extern "C" {

ckda_status ckda_fwd(const void* q, const void* k, const void* v, const void* alpha,
                     const void* beta, const float* h0, void* o, float* hT,
                     const int32_t* cu_seqlens, int num_seqs, int B, int H, int T, int dk,
                     int dv, ckda_dtype io_dtype, float scale, int chunk_size, void* workspace,
                     size_t workspace_bytes, void* stream) {
  return fwd_impl(q, k, v, alpha, beta, h0, o, hT, cu_seqlens, num_seqs, B, H, T, dk, dv,
                  io_dtype, scale, chunk_size, workspace, workspace_bytes, stream, 0, 0, 0.f);
}

ckda_status ckda_fwd_raw(const void* q_raw, const void* k_raw, const void* v, const void* a_raw,
                         const void* b_raw, const float* h0, void* o, float* hT,
                         const int32_t* cu_seqlens, int num_seqs, int B, int H, int T, int dk,
                         int dv, ckda_dtype io_dtype, float scale, int normalize_q,
                         float norm_eps, void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_impl(q_raw, k_raw, v, a_raw, b_raw, h0, o, hT, cu_seqlens, num_seqs, B, H, T, dk,
                  dv, io_dtype, scale, 0, workspace, workspace_bytes, stream, 1,
                  normalize_q ? 1 : 0, norm_eps);
}

ckda_status ckda_fwd_status(void* workspace, void* stream) {
  if (!workspace) return CKDA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int host = 0;
  if (cudaMemcpyAsync(&host, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return CKDA_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(int), s) != cudaSuccess) return CKDA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return CKDA_ERR_CUDA;
  return static_cast<ckda_status>(host);
}

ckda_status ckda_decode_step(const void* q, const void* k, const void* v, const void* alpha,
                             const void* beta, float* state, void* o, int B, int H, int dk,
                             int dv, ckda_dtype io_dtype, float scale, void* stream) {
  if (io_dtype != CKDA_F32 && io_dtype != CKDA_BF16) return CKDA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || dk < 1 || dv < 1) return CKDA_ERR_INVALID_ARG;
  if (!q || !k || !v || !alpha || !beta || !state || !o) return CKDA_ERR_INVALID_ARG;
  if (!(scale == scale)) return CKDA_ERR_INVALID_ARG;
  if (dk > 128 || dv > 128) return CKDA_ERR_UNSUPPORTED;
  if ((long long)B * H > 0x7fffffffLL) return CKDA_ERR_UNSUPPORTED;
  if (dk == 128 && dv == 128 && (reinterpret_cast<uintptr_t>(state) & 15) != 0)
    return CKDA_ERR_INVALID_ARG;
  DecodeArgs a{};
  a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta;
  a.state = state; a.o = o;
  a.B = B; a.H = H; a.dk = dk; a.dv = dv;
  a.scale = scale; a.io = io_dtype;
  return launch_decode(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? CKDA_OK
                                                                             : CKDA_ERR_CUDA;
}

ckda_status ckda_decode_step_raw(const void* q_raw, const void* k_raw, const void* v,
                                 const void* a_raw, const void* b_raw, float* state, void* o,
                                 int B, int H, int dk, int dv, ckda_dtype io_dtype, float scale,
                                 int normalize_q, float norm_eps, void* stream) {
  if (io_dtype != CKDA_F32 && io_dtype != CKDA_BF16) return CKDA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || dk < 1 || dv < 1) return CKDA_ERR_INVALID_ARG;
  if (!q_raw || !k_raw || !v || !a_raw || !b_raw || !state || !o) return CKDA_ERR_INVALID_ARG;
  if (!(scale == scale)) return CKDA_ERR_INVALID_ARG;
  if (!(norm_eps >= 0.f) || norm_eps > 3.0e38f) return CKDA_ERR_INVALID_ARG;
  if (dk != 128 || dv != 128) return CKDA_ERR_UNSUPPORTED;
  if ((long long)B * H > 0x7fffffffLL) return CKDA_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(state) & 15) != 0) return CKDA_ERR_INVALID_ARG;
  DecodeArgs a{};
  a.q = q_raw; a.k = k_raw; a.v = v; a.alpha = a_raw; a.beta = b_raw;
  a.state = state; a.o = o;
  a.B = B; a.H = H; a.dk = dk; a.dv = dv;
  a.scale = scale; a.io = io_dtype;
  return launch_decode_raw(a, normalize_q, norm_eps, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? CKDA_OK
             : CKDA_ERR_CUDA;
}

ckda_status ckda_selftest_timeout(void* workspace, size_t workspace_bytes, unsigned int spin_limit,
                                  void* stream) {
  if (!workspace || workspace_bytes < kWsStatusBytes) return CKDA_ERR_WORKSPACE;
  if (cudaMemsetAsync(workspace, 0, sizeof(int), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return CKDA_ERR_CUDA;
  return launch_selftest_timeout(static_cast<int*>(workspace), spin_limit,
                                 static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? CKDA_OK
             : CKDA_ERR_CUDA;
}

}  // extern "C"
