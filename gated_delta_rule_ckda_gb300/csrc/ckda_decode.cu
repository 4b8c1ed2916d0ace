// ckda_decode.cu -- one decode step on a resident fp32 state, in place.
//
// Per (batch, head), with the state H (dk x dv, rows = key channels) and one
// token (q, k, v, alpha, beta), the step is the bounded case study's
// read-compare-correct with per-channel decay ("Kimi Delta Attention: a
// bounded case study", worked case A/B), written per column j:
//     r_j  = sum_i H_ij alpha_i k_i          (read through the decayed state)
//     u_j  = beta (v_j - r_j)                (compare)
//     H'_ij = alpha_i H_ij + k_i u_j         (decay + correct)
//     o_j  = scale * sum_i H'_ij q_i         (readout of the updated state)
//
// The step moves the whole state once in and once out (128 KiB per head at
// dk = dv = 128) and does ~7 flop per state element, so it is bound by HBM
// bandwidth.  The 128 x 128 kernel below reads and writes the state with
// 16-byte vector accesses: a block of 256 threads owns one (batch, head);
// thread (g, c) holds rows 16g..16g+15 of columns 4c..4c+3 in registers, so a
// warp's access covers one whole 512-byte state row.  The two column sums
// (r and o) are reduced over the 8 row groups through shared memory.
#include "ckda_internal.cuh"

namespace ckda {
namespace {

// RAW: the token inputs are raw (q and k not normalised, a and b the gate
// logits), and the step first applies the input preparation of ckda_prep to
// them (unit-norm k, and q when normalize_q; alpha and beta from the logits).
// A separate instance, so that the plain step carries none of it.
template <typename IO, bool RAW>
__global__ void __launch_bounds__(256, 2) decode128_kernel(DecodeArgs a, int normalize_q,
                                                           float norm_eps) {
  __shared__ float s_ak[128], s_a[128], s_k[128], s_q[128], s_v[128];
  __shared__ float4 s_red[8][32];
  __shared__ float s_beta;
  const int p = blockIdx.x;  // (batch, head)
  const int tid = threadIdx.x, g = tid >> 5, c = tid & 31;
  float4* S = reinterpret_cast<float4*>(a.state + (size_t)p * 128 * 128);

  float4 h[16];
#pragma unroll
  for (int r = 0; r < 16; ++r) h[r] = __ldcs(S + (16 * g + r) * 32 + c);

  const IO* q = static_cast<const IO*>(a.q) + (size_t)p * 128;
  const IO* k = static_cast<const IO*>(a.k) + (size_t)p * 128;
  const IO* al = static_cast<const IO*>(a.alpha) + (size_t)p * 128;
  const IO* v = static_cast<const IO*>(a.v) + (size_t)p * 128;
  if (!RAW) {
    if (tid < 128) {
      float av = ld_io(al + tid), kv = ld_io(k + tid);
      s_a[tid] = av;
      s_k[tid] = kv;
      s_ak[tid] = av * kv;
      s_q[tid] = a.scale * ld_io(q + tid);
    } else {
      s_v[tid - 128] = ld_io(v + (tid - 128));
      if (tid == 128) s_beta = ld_io(static_cast<const IO*>(a.beta) + p);
    }
    __syncthreads();
  } else {
    // every warp reads all of k and q (four channels per lane) and reduces
    // the two norms itself, so that the step keeps a single block barrier
    float k4[4], q4[4], ss_k = 0.f, ss_q = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      k4[e] = ld_io(k + 4 * c + e);
      q4[e] = ld_io(q + 4 * c + e);
      ss_k = fmaf(k4[e], k4[e], ss_k);
      ss_q = fmaf(q4[e], q4[e], ss_q);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
      ss_k += __shfl_xor_sync(0xffffffffu, ss_k, m);
      ss_q += __shfl_xor_sync(0xffffffffu, ss_q, m);
    }
    const float ik = rsqrtf(ss_k + norm_eps);
    const float iq = normalize_q ? rsqrtf(ss_q + norm_eps) : 1.f;
    if (tid < 128) {  // warps 0-3 publish k, alpha, alpha k and scale q, one channel a lane
      const int i = tid;
      const float kv = ld_io(k + i) * ik, av = gate_alpha(ld_io(al + i));
      s_k[i] = kv;
      s_a[i] = av;
      s_ak[i] = av * kv;
      s_q[i] = a.scale * (ld_io(q + i) * iq);
    } else {
      s_v[tid - 128] = ld_io(v + (tid - 128));
      if (tid == 128) s_beta = gate_beta(ld_io(static_cast<const IO*>(a.beta) + p));
    }
    __syncthreads();
  }

  // r = H^T (alpha * k), partial over this thread's 16 rows
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const float w = s_ak[16 * g + r];
    acc.x = fmaf(h[r].x, w, acc.x);
    acc.y = fmaf(h[r].y, w, acc.y);
    acc.z = fmaf(h[r].z, w, acc.z);
    acc.w = fmaf(h[r].w, w, acc.w);
  }
  s_red[g][c] = acc;
  __syncthreads();
  float4 rr = s_red[0][c];
#pragma unroll
  for (int gg = 1; gg < 8; ++gg) {
    const float4 t = s_red[gg][c];
    rr.x += t.x; rr.y += t.y; rr.z += t.z; rr.w += t.w;
  }
  const float b = s_beta;
  const float4 vv = reinterpret_cast<const float4*>(s_v)[c];
  const float4 u = make_float4(b * (vv.x - rr.x), b * (vv.y - rr.y), b * (vv.z - rr.z),
                               b * (vv.w - rr.w));

  // H' = Diag(alpha) H + k u^T, and the partial readout o = H'^T q
  float4 oacc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const int i = 16 * g + r;
    const float ai = s_a[i], ki = s_k[i], qi = s_q[i];
    h[r].x = fmaf(ai, h[r].x, ki * u.x);
    h[r].y = fmaf(ai, h[r].y, ki * u.y);
    h[r].z = fmaf(ai, h[r].z, ki * u.z);
    h[r].w = fmaf(ai, h[r].w, ki * u.w);
    oacc.x = fmaf(h[r].x, qi, oacc.x);
    oacc.y = fmaf(h[r].y, qi, oacc.y);
    oacc.z = fmaf(h[r].z, qi, oacc.z);
    oacc.w = fmaf(h[r].w, qi, oacc.w);
  }
#pragma unroll
  for (int r = 0; r < 16; ++r) __stcs(S + (16 * g + r) * 32 + c, h[r]);
  __syncthreads();  // every thread has read s_red before it is reused
  s_red[g][c] = oacc;
  __syncthreads();
  if (g == 0) {
    float4 oo = s_red[0][c];
#pragma unroll
    for (int gg = 1; gg < 8; ++gg) {
      const float4 t = s_red[gg][c];
      oo.x += t.x; oo.y += t.y; oo.z += t.z; oo.w += t.w;
    }
    IO* o = static_cast<IO*>(a.o) + (size_t)p * 128 + 4 * c;
    st_io(o + 0, oo.x);
    st_io(o + 1, oo.y);
    st_io(o + 2, oo.z);
    st_io(o + 3, oo.w);
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  const int units = a.B * a.H;
  if (units == 0) return cudaSuccess;
  if (a.dk == 128 && a.dv == 128) {
    if (a.io == CKDA_F32)
      decode128_kernel<float, false><<<units, 256, 0, s>>>(a, 0, 0.f);
    else
      decode128_kernel<__nv_bfloat16, false><<<units, 256, 0, s>>>(a, 0, 0.f);
    return cudaGetLastError();
  }
  // Other shapes: the token-serial forward with T = 1 and the state as both
  // its initial and its final state (each thread reads its column first).
  FwdArgs f{};
  f.q = a.q; f.k = a.k; f.v = a.v; f.alpha = a.alpha; f.beta = a.beta;
  f.h0 = a.state; f.o = a.o; f.hT = a.state;
  f.cu_seqlens = nullptr; f.order = nullptr; f.status = nullptr;
  f.num_units_seq = a.B;
  f.B = a.B; f.H = a.H; f.T = 1; f.dk = a.dk; f.dv = a.dv;
  f.scale = a.scale; f.io = a.io;
  return launch_fwd_recurrent(f, s);
}

}  // namespace ckda

namespace ckda {

cudaError_t launch_decode_raw(const DecodeArgs& a, int normalize_q, float norm_eps,
                              cudaStream_t s) {
  const int units = a.B * a.H;
  if (units == 0) return cudaSuccess;
  if (a.io == CKDA_F32)
    decode128_kernel<float, true><<<units, 256, 0, s>>>(a, normalize_q, norm_eps);
  else
    decode128_kernel<__nv_bfloat16, true><<<units, 256, 0, s>>>(a, normalize_q, norm_eps);
  return cudaGetLastError();
}

}  // namespace ckda
