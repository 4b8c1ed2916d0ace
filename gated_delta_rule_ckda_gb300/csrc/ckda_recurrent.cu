// ckda_recurrent.cu -- token-serial CUDA-core forward for every shape the
// tensor-core kernel does not take (fp32 I/O, or dk/dv other than 128).
//
// The state columns evolve independently: the transition acts on the columns
// of H ("Complex KDA: Understanding and Enhancing the Expressivity of Kimi
// Delta Attention", Sec. 2, Eq. (1): "the transition applied to its
// columns").  So thread j of a block owns column j of one (sequence, head)
// state in registers and runs the bounded case study's three steps per token
// (decay row i by alpha_i, read v_hat_j = sum_i S_ij k_i, correct
// S_ij += beta k_i (v_j - v_hat_j)), then reads out o_j = sum_i S_ij q_i.
// No thread ever needs another thread's column; the block only shares the
// per-token vectors q, k, alpha, beta through shared memory.
#include "ckda_internal.cuh"

namespace ckda {
namespace {

constexpr int kTile = 16;  // tokens staged per shared-memory fill

template <typename IO, int DK>
__global__ void __launch_bounds__(128) fwd_recurrent_kernel(FwdArgs a) {
  __shared__ float sq[kTile][DK], sk[kTile][DK], sa[kTile][DK], sb[kTile];
  const IO* q = static_cast<const IO*>(a.q);
  const IO* k = static_cast<const IO*>(a.k);
  const IO* v = static_cast<const IO*>(a.v);
  const IO* al = static_cast<const IO*>(a.alpha);
  const IO* be = static_cast<const IO*>(a.beta);
  IO* o = static_cast<IO*>(a.o);

  const int unit = blockIdx.x;
  const int n = unit / a.H, h = unit % a.H;
  long row0;  // row of token 0 of this (sequence, head) in the [B*H*T] row space
  int len;
  if (a.cu_seqlens) {
    int t0 = a.cu_seqlens[n];
    len = a.cu_seqlens[n + 1] - t0;
    row0 = (long)h * a.T + t0;
  } else {
    len = a.T;
    row0 = ((long)n * a.H + h) * a.T;
  }
  const int j = threadIdx.x;
  const bool col = j < a.dv;
  const int dk = a.dk, dv = a.dv;
  const size_t sidx = ((size_t)n * a.H + h) * (size_t)dk * dv;

  float S[DK];
#pragma unroll
  for (int i = 0; i < DK; ++i) S[i] = 0.f;
  if (col && a.h0) {
#pragma unroll
    for (int i = 0; i < DK; ++i)
      if (i < dk) S[i] = a.h0[sidx + (size_t)i * dv + j];
  }

  for (int t0 = 0; t0 < len; t0 += kTile) {
    const int nt = min(kTile, len - t0);
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * DK; e += blockDim.x) {
      int tt = e / DK, i = e % DK;
      float qv = 0.f, kv = 0.f, av = 1.f;  // padded channels: no key, unit gate
      if (tt < nt && i < dk) {
        size_t off = (size_t)(row0 + t0 + tt) * dk + i;
        qv = ld_io(q + off);
        kv = ld_io(k + off);
        av = ld_io(al + off);
      }
      sq[tt][i] = qv;
      sk[tt][i] = kv;
      sa[tt][i] = av;
    }
    for (int tt = threadIdx.x; tt < kTile; tt += blockDim.x)
      sb[tt] = tt < nt ? ld_io(be + row0 + t0 + tt) : 0.f;
    __syncthreads();
    if (!col) continue;
    for (int tt = 0; tt < nt; ++tt) {
      const size_t r = (size_t)(row0 + t0 + tt);
      const float vj = ld_io(v + r * dv + j);
      float pred = 0.f;
#pragma unroll
      for (int i = 0; i < DK; ++i) {
        S[i] *= sa[tt][i];
        pred = fmaf(S[i], sk[tt][i], pred);
      }
      const float u = sb[tt] * (vj - pred);
      float oj = 0.f;
#pragma unroll
      for (int i = 0; i < DK; ++i) {
        S[i] = fmaf(sk[tt][i], u, S[i]);
        oj = fmaf(S[i], sq[tt][i], oj);
      }
      st_io(o + r * dv + j, a.scale * oj);
    }
  }
  if (col && a.hT) {
#pragma unroll
    for (int i = 0; i < DK; ++i)
      if (i < dk) a.hT[sidx + (size_t)i * dv + j] = S[i];
  }
}

template <typename IO>
cudaError_t launch_io(const FwdArgs& a, cudaStream_t s) {
  const int units = a.num_units_seq * a.H;
  if (units == 0) return cudaSuccess;
  dim3 grid(units), block(((a.dv + 31) / 32) * 32);
  if (a.dk <= 16)
    fwd_recurrent_kernel<IO, 16><<<grid, block, 0, s>>>(a);
  else if (a.dk <= 32)
    fwd_recurrent_kernel<IO, 32><<<grid, block, 0, s>>>(a);
  else if (a.dk <= 64)
    fwd_recurrent_kernel<IO, 64><<<grid, block, 0, s>>>(a);
  else
    fwd_recurrent_kernel<IO, 128><<<grid, block, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_recurrent(const FwdArgs& a, cudaStream_t s) {
  return a.io == CKDA_F32 ? launch_io<float>(a, s) : launch_io<__nv_bfloat16>(a, s);
}

}  // namespace ckda
