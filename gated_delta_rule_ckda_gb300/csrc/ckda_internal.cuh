// ckda_internal.cuh -- declarations shared by the translation units of libckda.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include "../../include/ckda.h"

namespace ckda {

// Workspace layout (bytes):
//   [0, 4)        device status word (int32, a ckda_status; 0 = OK)
//   [256, ...)    int32 order[num_seqs]: packed sequences, longest first
constexpr size_t kWsStatusBytes = 256;

// Records a device-side error; the first one wins.
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* alpha;
  const void* beta;
  const float* h0;
  void* o;
  float* hT;
  const int32_t* cu_seqlens;  // device, or nullptr
  const int32_t* order;       // device work order (packed), or nullptr
  int* status;                // device status word
  int num_units_seq;          // N (sequences) -- dense: B
  int B, H, T, dk, dv;
  float scale;
  ckda_dtype io;
  // Raw inputs (tensor-core path): q, k are unnormalised and alpha, beta
  // hold the gate logits a, b; the kernel applies ckda_prep's maps itself.
  int raw;
  int normalize_q;
  float norm_eps;
  // Sequence split (dense layout, tensor-core path): each sequence runs as
  // nseg segments of seg_len tokens (a multiple of 64; the last may be
  // shorter).  split_pass 1: segment 0 from h0 (its o, and its final state into
  // seg_state[1]) and, for segments 1..nseg-2, the final state from zero
  // (seg_F) and the transition (seg_P: the final state from [I | 0] with
  // v = 0).  split_pass 2: segments 1..nseg-1 from seg_state (o, and hT from
  // the last).  Buffers are [B * H][nseg][dk][128] fp32.  0 = no split.
  int split_pass;
  int nseg, seg_len;
  float* seg_state;
  float* seg_P;
  float* seg_F;
  // Packed split (cu_seqlens set): the plan in the workspace, int32
  // S[N] (segments of each sequence, >= 1), slot0[N + 1] (its first state
  // slot; slot x of head h is tile (slot0[i] + x) * H + h), off1[N + 1] and
  // off2[N + 1] (its first work item in pass 1 and 2), and the number of
  // work items per head this pass launches (an upper bound on off[N]).
  const int32_t* split_plan;
  int split_items;
};

// Shapes the chunkwise tensor-core kernel takes: bf16 I/O, dv = 128 and
// dk = 128, or dk = 64 (the reduced key dimension of a state-reduced head,
// "On State Reduction in Linear Attention"), which has an instance of its own.
inline bool fwd_tensor_path(ckda_dtype io, int dk, int dv) {
  return io == CKDA_BF16 && dv == 128 && (dk == 128 || dk == 64);
}
// The driver's cuTensorMapEncodeTiled, looked up once (null if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
// Chunkwise tcgen05 forward (fwd_tensor_path shapes, chunk 64), dense or
// packed, or one pass of the sequence split (a.split_pass != 0).
cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t s);
// Token-serial CUDA-core forward (any dk, dv <= 128).
cudaError_t launch_fwd_recurrent(const FwdArgs& a, cudaStream_t s);
// CTAs of one pass of the sequence split, per (sequence, head).
__host__ __device__ inline int split_ctas_per_unit(int pass, int nseg) {
  return pass == 1 ? (nseg >= 3 ? 2 * nseg - 3 : 1) : nseg - 1;
}
// The scan between the passes: seg_state[s + 1] = seg_P[s] seg_state[s] +
// seg_F[s] for s = 1..nseg-2, per (sequence, head); with a packed split's
// plan, per (sequence i, head) over its own S[i] segments.
cudaError_t launch_seg_scan(float* state, const float* P, const float* F, int units, int nseg,
                            int dk, cudaStream_t s, const int32_t* plan = nullptr, int N = 0,
                            int H = 0);
// The packed split's plan (see FwdArgs::split_plan) from cu_seqlens.
cudaError_t launch_split_plan(const int32_t* cu, const int32_t* order, int N, int seg_len,
                              int32_t* plan, cudaStream_t s);
// Longest-first order of packed sequences.
cudaError_t launch_seq_order(const int32_t* cu, int n, int32_t* order, cudaStream_t s);

struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* alpha;
  const void* beta;
  float* state;
  void* o;
  int B, H, dk, dv;
  float scale;
  ckda_dtype io;
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
// The decode step on raw inputs (q_raw, k_raw, gate logits a, b in the
// q, k, alpha, beta fields): dk = dv = 128 only.
cudaError_t launch_decode_raw(const DecodeArgs& a, int normalize_q, float norm_eps,
                              cudaStream_t s);

cudaError_t launch_selftest_timeout(int* status, unsigned spin_limit, cudaStream_t s);

// The paper's gate parameterisation ("Complex KDA" discussion slides, backup
// frame "practical gates differ from exact theoretical endpoints"), in fp32:
// alpha = s [e^-5 + (1 - e^-5) |tanh(a / 2)|] with s = +1 for tanh(a/2) >= 0,
// else -1; beta = 2 sigma(b), with the exponential of a non-positive argument
// on either side so that large |b| neither overflows nor loses the tail.
constexpr float kGateEps = 0.006737947f;  // e^-5
__device__ __forceinline__ float gate_alpha(float a) {
  const float r = tanhf(0.5f * a);
  const float s = r >= 0.f ? 1.f : -1.f;
  return s * fmaf(1.f - kGateEps, fabsf(r), kGateEps);
}
__device__ __forceinline__ float gate_beta(float b) {
  if (b >= 0.f) return 2.f / (1.f + expf(-b));
  const float e = expf(b);
  return 2.f * e / (1.f + e);
}

// Their derivatives, for the backward of the input preparation.  The sign s
// is piecewise constant and carries no gradient, and |tanh(a/2)| takes the
// subgradient 0 at a = 0, so d alpha / d a = (1 - e^-5) (1 - r^2) / 2 for
// a != 0 and 0 at a = 0; 1 - r^2 = 4 e / (1 + e)^2 with e = exp(-|a|) keeps
// its relative accuracy for large |a|.  d beta / d b = 2 sigma(b)(1 - sigma(b))
// = 2 e / (1 + e)^2 with e = exp(-|b|).
__device__ __forceinline__ float gate_alpha_grad(float a) {
  if (a == 0.f) return 0.f;
  const float e = expf(-fabsf(a));
  const float d = 1.f + e;
  return 2.f * (1.f - kGateEps) * e / (d * d);
}
__device__ __forceinline__ float gate_beta_grad(float b) {
  const float e = expf(-fabsf(b));
  const float d = 1.f + e;
  return 2.f * e / (d * d);
}

// Element loads/stores in the I/O dtype.
template <typename T>
__device__ __forceinline__ float ld_io(const T* p);
template <>
__device__ __forceinline__ float ld_io<float>(const float* p) {
  return *p;
}
template <>
__device__ __forceinline__ float ld_io<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void st_io(T* p, float x);
template <>
__device__ __forceinline__ void st_io<float>(float* p, float x) {
  *p = x;
}
template <>
__device__ __forceinline__ void st_io<__nv_bfloat16>(__nv_bfloat16* p, float x) {
  *p = __float2bfloat16_rn(x);
}

}  // namespace ckda
