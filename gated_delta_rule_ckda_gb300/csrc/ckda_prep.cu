// ckda_prep.cu -- fused input preparation for the CKDA forward and decode:
// unit-norm keys (and, on request, queries) and the paper's gate
// parameterisation, in one pass over HBM.
//
// Per token ("Complex KDA" discussion slides, backup frame "practical gates
// differ from exact theoretical endpoints"; paper App. E-G.1; the paper's
// Sec. 6 "Implementation" fuses the gate's sign handling into the key
// normalisation in the same way):
//
//   r = tanh(a / 2),  s = +1 if r >= 0 else -1,  alpha = s [eps + (1 - eps)|r|],
//   eps = e^-5,       beta = 2 sigma(b),
//   k <- k / sqrt(sum_i k_i^2 + norm_eps)            (paper Sec. 2: ||k_t|| = 1)
//
// One warp per token row; arithmetic in fp32, one rounding to the I/O dtype.
// Bound: HBM (each byte read or written once).  ckda_prep_bwd, the backward
// of the same map, follows the same layout.
#include "ckda_internal.cuh"

namespace ckda {
namespace {


struct PrepArgs {
  const void* q_raw;
  const void* k_raw;
  const void* a_raw;
  const void* b_raw;
  void* q;
  void* k;
  void* alpha;
  void* beta;
  long long rows;
  int dk;
  int normalize_q;
  float norm_eps;
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t bf_pack(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// bf16, dk = 128: lane l owns channels 4l .. 4l + 3 (8-byte accesses); each
// warp takes kRows rows and issues all their loads before using any.
constexpr int kRows = 2;
__global__ void __launch_bounds__(256) prep128_bf16_kernel(const PrepArgs a) {
  const int lane = threadIdx.x & 31;
  const long long row_base = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * kRows;
  uint2 kw[kRows], aw[kRows], qw[kRows];
  float b[kRows];
#pragma unroll
  for (int e = 0; e < kRows; ++e) {
    const long long row = row_base + e;
    kw[e] = aw[e] = qw[e] = make_uint2(0u, 0u);
    b[e] = 0.f;
    if (row < a.rows) {
      const size_t off = (size_t)row * 32 + lane;  // in uint2 units
      kw[e] = static_cast<const uint2*>(a.k_raw)[off];
      aw[e] = static_cast<const uint2*>(a.a_raw)[off];
      if (a.q_raw) qw[e] = static_cast<const uint2*>(a.q_raw)[off];
      if (lane == 0) b[e] = __bfloat162float(static_cast<const __nv_bfloat16*>(a.b_raw)[row]);
    }
  }
#pragma unroll
  for (int e = 0; e < kRows; ++e) {
    const long long row = row_base + e;
    if (row >= a.rows) break;  // warp-uniform
    const size_t off = (size_t)row * 32 + lane;
    const float k0 = bf_lo(kw[e].x), k1 = bf_hi(kw[e].x), k2 = bf_lo(kw[e].y), k3 = bf_hi(kw[e].y);
    const float ik = rsqrtf(warp_sum(k0 * k0 + k1 * k1 + k2 * k2 + k3 * k3) + a.norm_eps);
    static_cast<uint2*>(a.k)[off] =
        make_uint2(bf_pack(k0 * ik, k1 * ik), bf_pack(k2 * ik, k3 * ik));
    if (a.q_raw) {
      const float q0 = bf_lo(qw[e].x), q1 = bf_hi(qw[e].x), q2 = bf_lo(qw[e].y), q3 = bf_hi(qw[e].y);
      float iq = 1.f;
      if (a.normalize_q) iq = rsqrtf(warp_sum(q0 * q0 + q1 * q1 + q2 * q2 + q3 * q3) + a.norm_eps);
      static_cast<uint2*>(a.q)[off] =
          make_uint2(bf_pack(q0 * iq, q1 * iq), bf_pack(q2 * iq, q3 * iq));
    }
    static_cast<uint2*>(a.alpha)[off] =
        make_uint2(bf_pack(gate_alpha(bf_lo(aw[e].x)), gate_alpha(bf_hi(aw[e].x))),
                   bf_pack(gate_alpha(bf_lo(aw[e].y)), gate_alpha(bf_hi(aw[e].y))));
    if (lane == 0)
      static_cast<__nv_bfloat16*>(a.beta)[row] = __float2bfloat16_rn(gate_beta(b[e]));
  }
}

// Any dk <= 128 and either I/O dtype: lane l owns channels l, l + 32, ...
template <typename T>
__global__ void __launch_bounds__(256) prep_kernel(const PrepArgs a) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= a.rows) return;
  const size_t base = (size_t)row * a.dk;
  const T* kr = static_cast<const T*>(a.k_raw) + base;
  const T* ar = static_cast<const T*>(a.a_raw) + base;
  float kv[4], qv[4], av[4];
  float sk = 0.f, sq = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = lane + 32 * j;
    kv[j] = qv[j] = av[j] = 0.f;
    if (c < a.dk) {
      kv[j] = ld_io<T>(kr + c);
      av[j] = ld_io<T>(ar + c);
      if (a.q_raw) qv[j] = ld_io<T>(static_cast<const T*>(a.q_raw) + base + c);
    }
    sk = fmaf(kv[j], kv[j], sk);
    sq = fmaf(qv[j], qv[j], sq);
  }
  const float ik = rsqrtf(warp_sum(sk) + a.norm_eps);
  float iq = 1.f;
  if (a.q_raw && a.normalize_q) iq = rsqrtf(warp_sum(sq) + a.norm_eps);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = lane + 32 * j;
    if (c < a.dk) {
      st_io<T>(static_cast<T*>(a.k) + base + c, kv[j] * ik);
      st_io<T>(static_cast<T*>(a.alpha) + base + c, gate_alpha(av[j]));
      if (a.q_raw) st_io<T>(static_cast<T*>(a.q) + base + c, qv[j] * iq);
    }
  }
  if (lane == 0)
    st_io<T>(static_cast<T*>(a.beta) + row, gate_beta(ld_io<T>(static_cast<const T*>(a.b_raw) + row)));
}

// ------------------------------------------------------------- backward
// Gradients with respect to the raw inputs from those with respect to the
// prepared ones, per token row:
//   k = x / n, n = sqrt(sum x^2 + norm_eps):  dx = (dk - k (k . dk)) / n
//   (q likewise when normalised, else dq passes through),
//   da = dalpha * gate_alpha_grad(a),  db = dbeta * gate_beta_grad(b).
// One HBM pass; fp32 arithmetic, one rounding to the I/O dtype.
struct PrepBwdArgs {
  const void* q_raw;
  const void* k_raw;
  const void* a_raw;
  const void* b_raw;
  const void* dq;
  const void* dk;
  const void* dalpha;
  const void* dbeta;
  void* dq_raw;
  void* dk_raw;
  void* da_raw;
  void* db_raw;
  long long rows;
  int dk_width;
  int normalize_q;
  float norm_eps;
};

// (x, g) -> (g - k (k . g)) / n for one row held as four channels per lane
// (any assignment of channels to lanes; unused channels are zero).
__device__ __forceinline__ void unit_norm_bwd4(float (&x)[4], const float (&g)[4], float eps) {
  const float in = rsqrtf(warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]) + eps);
  float kx[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) kx[i] = x[i] * in;
  const float dot = warp_sum(kx[0] * g[0] + kx[1] * g[1] + kx[2] * g[2] + kx[3] * g[3]);
#pragma unroll
  for (int i = 0; i < 4; ++i) x[i] = (g[i] - kx[i] * dot) * in;
}
__device__ __forceinline__ void unpack4(uint2 w, float (&f)[4]) {
  f[0] = bf_lo(w.x); f[1] = bf_hi(w.x); f[2] = bf_lo(w.y); f[3] = bf_hi(w.y);
}
__device__ __forceinline__ uint2 pack4(const float (&f)[4]) {
  return make_uint2(bf_pack(f[0], f[1]), bf_pack(f[2], f[3]));
}

// bf16, dk = 128: lane l owns channels 4l .. 4l + 3; kRows rows per warp,
// every load in flight before any use.
__global__ void __launch_bounds__(256) prep_bwd128_bf16_kernel(const PrepBwdArgs a) {
  const int lane = threadIdx.x & 31;
  const long long row_base = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * kRows;
  uint2 kw[kRows], aw[kRows], qw[kRows], gk[kRows], ga[kRows], gq[kRows];
  float b[kRows], gb[kRows];
#pragma unroll
  for (int e = 0; e < kRows; ++e) {
    const long long row = row_base + e;
    kw[e] = aw[e] = qw[e] = gk[e] = ga[e] = gq[e] = make_uint2(0u, 0u);
    b[e] = gb[e] = 0.f;
    if (row < a.rows) {
      const size_t off = (size_t)row * 32 + lane;  // in uint2 units
      kw[e] = static_cast<const uint2*>(a.k_raw)[off];
      aw[e] = static_cast<const uint2*>(a.a_raw)[off];
      gk[e] = static_cast<const uint2*>(a.dk)[off];
      ga[e] = static_cast<const uint2*>(a.dalpha)[off];
      if (a.q_raw) {
        qw[e] = static_cast<const uint2*>(a.q_raw)[off];
        gq[e] = static_cast<const uint2*>(a.dq)[off];
      }
      if (lane == 0) {
        b[e] = __bfloat162float(static_cast<const __nv_bfloat16*>(a.b_raw)[row]);
        gb[e] = __bfloat162float(static_cast<const __nv_bfloat16*>(a.dbeta)[row]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < kRows; ++e) {
    const long long row = row_base + e;
    if (row >= a.rows) break;  // warp-uniform
    const size_t off = (size_t)row * 32 + lane;
    float x[4], g[4];
    unpack4(kw[e], x);
    unpack4(gk[e], g);
    unit_norm_bwd4(x, g, a.norm_eps);
    static_cast<uint2*>(a.dk_raw)[off] = pack4(x);
    if (a.q_raw) {
      if (a.normalize_q) {
        unpack4(qw[e], x);
        unpack4(gq[e], g);
        unit_norm_bwd4(x, g, a.norm_eps);
        static_cast<uint2*>(a.dq_raw)[off] = pack4(x);
      } else {
        static_cast<uint2*>(a.dq_raw)[off] = gq[e];
      }
    }
    unpack4(aw[e], x);
    unpack4(ga[e], g);
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = g[i] * gate_alpha_grad(x[i]);
    static_cast<uint2*>(a.da_raw)[off] = pack4(x);
    if (lane == 0)
      static_cast<__nv_bfloat16*>(a.db_raw)[row] = __float2bfloat16_rn(gb[e] * gate_beta_grad(b[e]));
  }
}

// Any dk <= 128 and either I/O dtype: lane l owns channels l, l + 32, ...
template <typename T>
__global__ void __launch_bounds__(256) prep_bwd_kernel(const PrepBwdArgs a) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= a.rows) return;
  const size_t base = (size_t)row * a.dk_width;
  float kv[4], qv[4], av[4], gk[4], gq[4], ga[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = lane + 32 * j;
    kv[j] = qv[j] = av[j] = gk[j] = gq[j] = ga[j] = 0.f;
    if (c < a.dk_width) {
      kv[j] = ld_io<T>(static_cast<const T*>(a.k_raw) + base + c);
      av[j] = ld_io<T>(static_cast<const T*>(a.a_raw) + base + c);
      gk[j] = ld_io<T>(static_cast<const T*>(a.dk) + base + c);
      ga[j] = ld_io<T>(static_cast<const T*>(a.dalpha) + base + c);
      if (a.q_raw) {
        qv[j] = ld_io<T>(static_cast<const T*>(a.q_raw) + base + c);
        gq[j] = ld_io<T>(static_cast<const T*>(a.dq) + base + c);
      }
    }
  }
  float bb = 0.f, gb = 0.f;
  if (lane == 0) {
    bb = ld_io<T>(static_cast<const T*>(a.b_raw) + row);
    gb = ld_io<T>(static_cast<const T*>(a.dbeta) + row);
  }
  unit_norm_bwd4(kv, gk, a.norm_eps);
  const bool qn = a.q_raw && a.normalize_q;
  if (qn) unit_norm_bwd4(qv, gq, a.norm_eps);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = lane + 32 * j;
    if (c < a.dk_width) {
      st_io<T>(static_cast<T*>(a.dk_raw) + base + c, kv[j]);
      st_io<T>(static_cast<T*>(a.da_raw) + base + c, ga[j] * gate_alpha_grad(av[j]));
      if (a.q_raw) st_io<T>(static_cast<T*>(a.dq_raw) + base + c, qn ? qv[j] : gq[j]);
    }
  }
  if (lane == 0) st_io<T>(static_cast<T*>(a.db_raw) + row, gb * gate_beta_grad(bb));
}

}  // namespace
}  // namespace ckda

using namespace ckda;

extern "C" ckda_status ckda_prep_bwd(const void* q_raw, const void* k_raw, const void* a_raw,
                                     const void* b_raw, const void* d_q, const void* d_k,
                                     const void* d_alpha, const void* d_beta, void* d_q_raw,
                                     void* d_k_raw, void* d_a_raw, void* d_b_raw, long long rows,
                                     int dk, ckda_dtype io_dtype, int normalize_q,
                                     float norm_eps, void* stream) {
  if (io_dtype != CKDA_F32 && io_dtype != CKDA_BF16) return CKDA_ERR_INVALID_ARG;
  if (rows < 0 || dk < 1) return CKDA_ERR_INVALID_ARG;
  if (!(norm_eps >= 0.f) || norm_eps > 3.0e38f) return CKDA_ERR_INVALID_ARG;
  if ((q_raw == nullptr) != (d_q == nullptr) || (q_raw == nullptr) != (d_q_raw == nullptr))
    return CKDA_ERR_INVALID_ARG;
  if (rows > 0 && (!k_raw || !a_raw || !b_raw || !d_k || !d_alpha || !d_beta || !d_k_raw ||
                   !d_a_raw || !d_b_raw))
    return CKDA_ERR_INVALID_ARG;
  if (dk > 128) return CKDA_ERR_UNSUPPORTED;
  if (rows > (long long)0x7fffffff * 8) return CKDA_ERR_UNSUPPORTED;
  if (rows == 0) return CKDA_OK;
  PrepBwdArgs a{q_raw, k_raw, a_raw, b_raw, d_q, d_k, d_alpha, d_beta, d_q_raw, d_k_raw,
                d_a_raw, d_b_raw, rows, dk, normalize_q, norm_eps};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool vec = io_dtype == CKDA_BF16 && dk == 128;
  for (const void* p : {q_raw, k_raw, a_raw, d_q, d_k, d_alpha, static_cast<const void*>(d_q_raw),
                        static_cast<const void*>(d_k_raw), static_cast<const void*>(d_a_raw)})
    if (p && (reinterpret_cast<uintptr_t>(p) & 7) != 0) vec = false;
  if (vec)
    prep_bwd128_bf16_kernel<<<(unsigned)((rows + 8 * kRows - 1) / (8 * kRows)), 256, 0, s>>>(a);
  else if (io_dtype == CKDA_BF16)
    prep_bwd_kernel<__nv_bfloat16><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(a);
  else
    prep_bwd_kernel<float><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? CKDA_OK : CKDA_ERR_CUDA;
}

extern "C" ckda_status ckda_prep(const void* q_raw, const void* k_raw, const void* a_raw,
                                 const void* b_raw, void* q, void* k, void* alpha, void* beta,
                                 long long rows, int dk, ckda_dtype io_dtype, int normalize_q,
                                 float norm_eps, void* stream) {
  if (io_dtype != CKDA_F32 && io_dtype != CKDA_BF16) return CKDA_ERR_INVALID_ARG;
  if (rows < 0 || dk < 1) return CKDA_ERR_INVALID_ARG;
  if (!(norm_eps >= 0.f) || norm_eps > 3.0e38f) return CKDA_ERR_INVALID_ARG;
  if ((q_raw == nullptr) != (q == nullptr)) return CKDA_ERR_INVALID_ARG;
  if (rows > 0 && (!k_raw || !a_raw || !b_raw || !k || !alpha || !beta))
    return CKDA_ERR_INVALID_ARG;
  if (dk > 128) return CKDA_ERR_UNSUPPORTED;
  if (rows > (long long)0x7fffffff * 8) return CKDA_ERR_UNSUPPORTED;
  if (rows == 0) return CKDA_OK;
  PrepArgs a{q_raw, k_raw, a_raw, b_raw, q, k, alpha, beta, rows, dk, normalize_q, norm_eps};
  const unsigned blocks = (unsigned)((rows + 7) / 8);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool vec = io_dtype == CKDA_BF16 && dk == 128;
  for (const void* p : {q_raw, k_raw, a_raw, static_cast<const void*>(q), static_cast<const void*>(k),
                        static_cast<const void*>(alpha)})
    if (p && (reinterpret_cast<uintptr_t>(p) & 7) != 0) vec = false;
  if (vec)
    prep128_bf16_kernel<<<(unsigned)((rows + 8 * kRows - 1) / (8 * kRows)), 256, 0, s>>>(a);
  else if (io_dtype == CKDA_BF16)
    prep_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(a);
  else
    prep_kernel<float><<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? CKDA_OK : CKDA_ERR_CUDA;
}
