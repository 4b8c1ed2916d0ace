// ckda_split.cu -- the sequence-split forward: few long sequences spread over
// many SMs by a two-level scan over segment operators.
//
// The state after a segment is an affine function of the state before it
// ("Kimi Delta Attention: a bounded case study", "Chunkwise execution": the
// chunk operator is Diag(gamma_C) - (k*rho)^T W applied to the state plus the
// chunk's write, and a product of such operators is again one; the
// sequence-parallel scan over these operators is the one step beyond
// chunking that splits a single sequence):
//
//     H_out = P H_in + F,   P = prod of the segment's transitions (dk x dk),
//                           F = the segment's final state from H_in = 0.
//
// Pass 1 runs, in parallel, segment 0 from h0 (its outputs are final), and
// for every middle segment F (from zero) and P (the final state from
// [I | 0] with v = 0: both are the tensor-core forward with a different
// initial state and value input).  The scan below then gives the state
// entering every segment, and pass 2 runs segments 1..S-1 from those states.
// Results equal one pass over the whole sequence up to rounding.
#include "ckda_internal.cuh"

#include <algorithm>

namespace ckda {
namespace {

constexpr int kScanCols = 16;      // state columns per CTA
constexpr int kScanThreads = 256;  // 16 row groups x 16 columns

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}

// One (sequence, head) and 16 state columns per CTA.  Thread (g, j) owns rows
// g, g + 16, ... of column j, so that the two row groups of a warp read
// neighbouring rows of P (different banks) and the same H entries
// (broadcast).  P_s (rows padded by 4 floats) is double-buffered: P_{s+1} is
// copied in while step s computes.  The column block of H stays in shared
// memory between steps; each output is an fp32 dot product over m in order.
// Dense: unit ui has nseg segments at tiles ui * nseg + x.  Packed (plan
// set): unit ui = (sequence i, head h) has S[i] segments at tiles
// (slot0[i] + x) * H + h.
template <int DK>
__global__ void __launch_bounds__(kScanThreads) seg_scan_kernel(float* state, const float* P,
                                                                const float* F, int nseg,
                                                                const int32_t* plan, int N,
                                                                int H) {
  extern __shared__ float4 scan_smem[];
  constexpr int LDP = DK + 4;
  constexpr int R = DK / 16;
  constexpr size_t tile = (size_t)DK * 128;
  float* Ps = reinterpret_cast<float*>(scan_smem);   // [2][DK][LDP]
  float* Hs = Ps + 2 * DK * LDP;                     // [DK][16]
  const int ui = blockIdx.x, j0 = blockIdx.y * kScanCols;
  const int tid = threadIdx.x, g = tid >> 4, j = tid & 15;
  size_t t0 = (size_t)ui * nseg, tstride = 1;   // tile of slot x: t0 + x * tstride
  if (plan) {
    const int i = ui / H, h = ui % H;
    nseg = plan[i];
    t0 = (size_t)plan[N + i] * H + h;
    tstride = H;
  }
  if (nseg < 3) return;
  auto at = [&](int x) { return (t0 + (size_t)x * tstride) * tile; };
  auto fetch_p = [&](int s) {
    const float* Pg = P + at(s);
    float* dst = Ps + (s & 1) * DK * LDP;
    for (int e = tid; e < DK * DK / 4; e += kScanThreads) {
      const int i = e / (DK / 4), m4 = e % (DK / 4);
      cp_async16(dst + i * LDP + 4 * m4, Pg + (size_t)i * 128 + 4 * m4);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  fetch_p(1);
  // H_1 (written by pass 1)
  for (int e = tid; e < DK * kScanCols; e += kScanThreads) {
    const int m = e / kScanCols, c = e % kScanCols;
    Hs[e] = state[at(1) + (size_t)m * 128 + j0 + c];
  }
  for (int s = 1; s + 1 < nseg; ++s) {
    if (s + 2 < nseg) {
      fetch_p(s + 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();   // P_s and H_s in place
    const float* Pb = Ps + (s & 1) * DK * LDP;
    const float* Fg = F + at(s);
    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = Fg[(size_t)(16 * r + g) * 128 + j0 + j];
#pragma unroll 4
    for (int m = 0; m < DK; m += 4) {
      const float h0 = Hs[(m + 0) * kScanCols + j], h1 = Hs[(m + 1) * kScanCols + j];
      const float h2 = Hs[(m + 2) * kScanCols + j], h3 = Hs[(m + 3) * kScanCols + j];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float4 p = *reinterpret_cast<const float4*>(Pb + (16 * r + g) * LDP + m);
        acc[r] = fmaf(p.w, h3, fmaf(p.z, h2, fmaf(p.y, h1, fmaf(p.x, h0, acc[r]))));
      }
    }
    __syncthreads();   // every read of H_s and of this P buffer is done
    float* Hg = state + at(s + 1);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      Hs[(16 * r + g) * kScanCols + j] = acc[r];
      Hg[(size_t)(16 * r + g) * 128 + j0 + j] = acc[r];
    }
  }
}


// The packed split's plan (one block): per sequence i (the i-th in `order`,
// longest first) of length L_i,
// S[i] = max(1, ceil(L_i / seg_len)) segments, and exclusive prefix sums of
// S (slot0), of the pass-1 work items (1 for S <= 2, else 2 S - 3: segment 0,
// S - 2 zero-start finals, S - 2 transitions) and of the pass-2 items (S - 1).
// Layout: S[N], slot0[N + 1], off1[N + 1], off2[N + 1].
__global__ void __launch_bounds__(1024) split_plan_kernel(const int32_t* cu, const int32_t* order,
                                                          int N, int seg_len, int32_t* plan) {
  __shared__ int carry[3];
  __shared__ int part[3][32];
  int32_t* Sn = plan;
  int32_t* slot0 = plan + N;
  int32_t* off1 = slot0 + N + 1;
  int32_t* off2 = off1 + N + 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < 3) carry[tid] = 0;
  __syncthreads();
  for (int base = 0; base < N; base += 1024) {
    const int i = base + tid;
    int v[3] = {0, 0, 0};
    if (i < N) {
      const int n = order ? order[i] : i;
      const int L = cu[n + 1] - cu[n];
      const int S = max(1, (L + seg_len - 1) / seg_len);
      Sn[i] = S;
      v[0] = S;
      v[1] = S >= 3 ? 2 * S - 3 : 1;
      v[2] = S - 1;
    }
    int incl[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      int x = v[k];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
      }
      incl[k] = x;
      if (lane == 31) part[k][warp] = x;
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        int x = part[k][lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, d);
          if (lane >= d) x += y;
        }
        part[k][lane] = x;   // inclusive over warps
      }
    }
    __syncthreads();
    if (i < N) {
      int32_t* outs[3] = {slot0, off1, off2};
#pragma unroll
      for (int k = 0; k < 3; ++k)
        outs[k][i] = carry[k] + (warp ? part[k][warp - 1] : 0) + incl[k] - v[k];
    }
    __syncthreads();
    if (tid < 3) carry[tid] += part[tid][31];
    __syncthreads();
  }
  if (tid == 0) {
    slot0[N] = carry[0];
    off1[N] = carry[1];
    off2[N] = carry[2];
  }
}

}  // namespace

cudaError_t launch_seg_scan(float* state, const float* P, const float* F, int units, int nseg,
                            int dk, cudaStream_t s, const int32_t* plan, int N, int H) {
  if (units == 0 || (!plan && nseg < 3)) return cudaSuccess;
  const dim3 grid(units, 128 / kScanCols);
  const size_t smem = (2 * (size_t)dk * (dk + 4) + (size_t)dk * kScanCols) * sizeof(float);
  auto kern = dk == 64 ? seg_scan_kernel<64> : seg_scan_kernel<128>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  kern<<<grid, kScanThreads, smem, s>>>(state, P, F, nseg, plan, N, H);
  return cudaGetLastError();
}

cudaError_t launch_split_plan(const int32_t* cu, const int32_t* order, int N, int seg_len,
                              int32_t* plan, cudaStream_t s) {
  split_plan_kernel<<<1, 1024, 0, s>>>(cu, order, N, seg_len, plan);
  return cudaGetLastError();
}

}  // namespace ckda

using namespace ckda;

namespace {

size_t split_state_tile_bytes(int dk) { return (size_t)dk * 128 * sizeof(float); }

// Segments and tokens per segment for a requested count: segments hold
// ceil(chunks / S) chunks each, so the count actually used may be lower.
void split_shape(int T, int segments, int* nseg, int* seg_len) {
  const int nch = (T + 63) / 64;
  const int sc = std::max(1, (nch + segments - 1) / segments);
  *seg_len = sc * 64;
  *nseg = std::max(1, (nch + sc - 1) / sc);
}

int device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace

extern "C" {

int ckda_fwd_split_segments(int B, int H, int T, int dk, int dv, ckda_dtype io_dtype,
                            int num_sms) {
  if (B < 1 || H < 1 || T < 1 || num_sms < 0) return 1;
  if (!fwd_tensor_path(io_dtype, dk, dv)) return 1;
  if (num_sms == 0) num_sms = device_sms();
  if (num_sms < 1) return 1;
  const long long units = (long long)B * H;
  const int nch = (T + 63) / 64;
  auto waves = [&](long long ctas) { return (ctas + num_sms - 1) / num_sms; };
  // time in chunk steps: both passes (each in whole waves of CTAs), one step
  // of state I/O per pass, and about half a step per scan step
  double best = (double)waves(units) * nch;
  int best_s = 1;
  for (int S = 2; S <= 16 && S <= nch; ++S) {
    int ns = 0, sl = 0;
    split_shape(T, S, &ns, &sl);
    if (ns != S) continue;
    const double t = (double)(waves(units * split_ctas_per_unit(1, S)) +
                              waves(units * split_ctas_per_unit(2, S))) * (sl / 64) +
                     2.0 + 0.5 * (S - 2);
    if (t < 0.9 * best) {
      best = t;
      best_s = S;
    }
  }
  return best_s;
}

size_t ckda_fwd_split_workspace_bytes(int B, int H, int T, int dk, int dv, ckda_dtype io_dtype,
                                      int segments) {
  if (B < 1 || H < 1 || T < 0 || dk < 1 || segments < 0) return 0;
  if (segments == 0) segments = ckda_fwd_split_segments(B, H, T, dk, dv, io_dtype, 0);
  size_t bytes = ckda_fwd_workspace_bytes(0, H);
  if (segments < 2 || T == 0) return bytes;
  int nseg = 0, seg_len = 0;
  split_shape(T, segments, &nseg, &seg_len);
  if (nseg < 2) return bytes;
  const size_t per = (size_t)B * H * nseg * split_state_tile_bytes(dk);
  return bytes + per * (nseg >= 3 ? 3 : 1);
}

ckda_status ckda_fwd_split(const void* q, const void* k, const void* v, const void* alpha,
                           const void* beta, const float* h0, void* o, float* hT, int B, int H,
                           int T, int dk, int dv, ckda_dtype io_dtype, float scale, int segments,
                           void* workspace, size_t workspace_bytes, void* stream) {
  if (segments < 0) return CKDA_ERR_INVALID_ARG;
  if (segments == 0) {
    if (io_dtype != CKDA_F32 && io_dtype != CKDA_BF16) return CKDA_ERR_INVALID_ARG;
    segments = ckda_fwd_split_segments(B, H, T, dk, dv, io_dtype, 0);
  }
  int nseg = 1, seg_len = 0;
  if (segments >= 2 && T > 0) split_shape(T, segments, &nseg, &seg_len);
  if (nseg < 2)
    return ckda_fwd(q, k, v, alpha, beta, h0, o, hT, nullptr, 0, B, H, T, dk, dv, io_dtype, scale,
                    0, workspace, workspace_bytes, stream);

  // the checks of ckda_fwd, for the shapes the split takes
  if (io_dtype != CKDA_F32 && io_dtype != CKDA_BF16) return CKDA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || dk < 1 || dv < 1) return CKDA_ERR_INVALID_ARG;
  if ((long long)B * H * T > 0x7fffffffLL) return CKDA_ERR_UNSUPPORTED;
  if (!(scale == scale)) return CKDA_ERR_INVALID_ARG;
  if (!q || !k || !v || !alpha || !beta || !o) return CKDA_ERR_INVALID_ARG;
  if (!fwd_tensor_path(io_dtype, dk, dv)) return CKDA_ERR_UNSUPPORTED;
  for (const void* p : {q, k, v, alpha})
    if ((reinterpret_cast<uintptr_t>(p) & 15) != 0) return CKDA_ERR_INVALID_ARG;
  const size_t need = ckda_fwd_split_workspace_bytes(B, H, T, dk, dv, io_dtype, segments);
  if (!workspace || workspace_bytes < need) return CKDA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return CKDA_ERR_WORKSPACE;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const size_t per = (size_t)B * H * nseg * split_state_tile_bytes(dk);
  float* seg_state = reinterpret_cast<float*>(ws + kWsStatusBytes);
  float* seg_P = nseg >= 3 ? reinterpret_cast<float*>(ws + kWsStatusBytes + per) : nullptr;
  float* seg_F = nseg >= 3 ? reinterpret_cast<float*>(ws + kWsStatusBytes + 2 * per) : nullptr;

  FwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta;
  a.h0 = h0; a.o = o; a.hT = hT;
  a.status = static_cast<int*>(workspace);
  a.num_units_seq = B;
  a.B = B; a.H = H; a.T = T; a.dk = dk; a.dv = dv;
  a.scale = scale; a.io = io_dtype;
  a.nseg = nseg; a.seg_len = seg_len;
  a.seg_state = seg_state; a.seg_P = seg_P; a.seg_F = seg_F;

  if (cudaMemsetAsync(a.status, 0, sizeof(int), s) != cudaSuccess) return CKDA_ERR_CUDA;
  a.split_pass = 1;
  if (launch_fwd(a, s) != cudaSuccess) return CKDA_ERR_CUDA;
  if (launch_seg_scan(seg_state, seg_P, seg_F, B * H, nseg, dk, s) != cudaSuccess)
    return CKDA_ERR_CUDA;
  a.split_pass = 2;
  if (launch_fwd(a, s) != cudaSuccess) return CKDA_ERR_CUDA;
  return CKDA_OK;
}

}  // extern "C"

namespace {

// Packed split sizes: state slots (an upper bound on the sum over sequences of
// max(1, ceil(L / seg_len))) and work items per head in each pass.
long long varlen_slots(int N, int T, int seg_len) { return (long long)T / seg_len + 1 + N; }
long long varlen_items(int pass, int N, int T, int seg_len) {
  return pass == 1 ? 2 * varlen_slots(N, T, seg_len) : (long long)T / seg_len + 1;
}
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
size_t varlen_plan_offset(int N) { return align256(kWsStatusBytes + 4 * (size_t)N); }
size_t varlen_state_offset(int N) {
  return varlen_plan_offset(N) + align256(4 * (size_t)(4 * N + 3));
}

}  // namespace

extern "C" {

int ckda_fwd_split_varlen_seg_len(int num_seqs, int H, int T, int dk, int dv,
                                  ckda_dtype io_dtype, int num_sms) {
  if (num_seqs < 1 || H < 1 || T < 1 || num_sms < 0) return 0;
  if (!fwd_tensor_path(io_dtype, dk, dv)) return 0;
  if (num_sms == 0) num_sms = device_sms();
  if (num_sms < 1) return 0;
  // a sequence longer than the average work per SM (in chunk steps) is cut
  // into segments of about that length; shorter ones run whole
  const long long work = (long long)((T + 63) / 64 + num_seqs) * H;
  const long long per_sm = std::max<long long>(16, (work + num_sms - 1) / num_sms);
  return (int)std::min<long long>(per_sm * 64, 1LL << 24);
}

size_t ckda_fwd_split_varlen_workspace_bytes(int num_seqs, int H, int T, int dk, int seg_len) {
  if (num_seqs < 1 || H < 1 || T < 0 || dk < 1 || seg_len < 64 || seg_len % 64) return 0;
  const size_t tile = (size_t)dk * 128 * sizeof(float);
  return varlen_state_offset(num_seqs) +
         3 * (size_t)varlen_slots(num_seqs, T, seg_len) * H * tile;
}

ckda_status ckda_fwd_split_varlen(const void* q, const void* k, const void* v, const void* alpha,
                                  const void* beta, const float* h0, void* o, float* hT,
                                  const int32_t* cu_seqlens, int num_seqs, int H, int T, int dk,
                                  int dv, ckda_dtype io_dtype, float scale, int seg_len,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  if (io_dtype != CKDA_F32 && io_dtype != CKDA_BF16) return CKDA_ERR_INVALID_ARG;
  if (num_seqs < 1 || H < 1 || T < 0 || dk < 1 || dv < 1 || !cu_seqlens)
    return CKDA_ERR_INVALID_ARG;
  if (seg_len < 0 || seg_len % 64) return CKDA_ERR_INVALID_ARG;
  if ((long long)H * T > 0x7fffffffLL) return CKDA_ERR_UNSUPPORTED;
  if (!(scale == scale)) return CKDA_ERR_INVALID_ARG;
  if (!q || !k || !v || !alpha || !beta || !o) return CKDA_ERR_INVALID_ARG;
  if (!fwd_tensor_path(io_dtype, dk, dv)) return CKDA_ERR_UNSUPPORTED;
  for (const void* p : {q, k, v, alpha})
    if ((reinterpret_cast<uintptr_t>(p) & 15) != 0) return CKDA_ERR_INVALID_ARG;
  if (seg_len == 0) seg_len = ckda_fwd_split_varlen_seg_len(num_seqs, H, T, dk, dv, io_dtype, 0);
  if (seg_len < 64) return CKDA_ERR_CUDA;
  const size_t need = ckda_fwd_split_varlen_workspace_bytes(num_seqs, H, T, dk, seg_len);
  if (!workspace || workspace_bytes < need) return CKDA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return CKDA_ERR_WORKSPACE;
  const long long items1 = varlen_items(1, num_seqs, T, seg_len);
  if (items1 * H > 0x7fffffffLL) return CKDA_ERR_UNSUPPORTED;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const size_t per = (size_t)varlen_slots(num_seqs, T, seg_len) * H * dk * 128 * sizeof(float);
  int32_t* order = reinterpret_cast<int32_t*>(ws + kWsStatusBytes);
  int32_t* plan = reinterpret_cast<int32_t*>(ws + varlen_plan_offset(num_seqs));
  char* st = ws + varlen_state_offset(num_seqs);

  FwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta;
  a.h0 = h0; a.o = o; a.hT = hT;
  a.cu_seqlens = cu_seqlens;
  a.order = order;
  a.status = static_cast<int*>(workspace);
  a.num_units_seq = num_seqs;
  a.B = 1; a.H = H; a.T = T; a.dk = dk; a.dv = dv;
  a.scale = scale; a.io = io_dtype;
  a.seg_len = seg_len;
  a.seg_state = reinterpret_cast<float*>(st);
  a.seg_P = reinterpret_cast<float*>(st + per);
  a.seg_F = reinterpret_cast<float*>(st + 2 * per);
  a.split_plan = plan;

  if (cudaMemsetAsync(a.status, 0, sizeof(int), s) != cudaSuccess) return CKDA_ERR_CUDA;
  if (launch_seq_order(cu_seqlens, num_seqs, order, s) != cudaSuccess) return CKDA_ERR_CUDA;
  if (launch_split_plan(cu_seqlens, order, num_seqs, seg_len, plan, s) != cudaSuccess)
    return CKDA_ERR_CUDA;
  a.split_pass = 1;
  a.split_items = (int)items1;
  if (launch_fwd(a, s) != cudaSuccess) return CKDA_ERR_CUDA;
  if (launch_seg_scan(a.seg_state, a.seg_P, a.seg_F, num_seqs * H, 0, dk, s, plan, num_seqs, H) !=
      cudaSuccess)
    return CKDA_ERR_CUDA;
  a.split_pass = 2;
  a.split_items = (int)varlen_items(2, num_seqs, T, seg_len);
  if (launch_fwd(a, s) != cudaSuccess) return CKDA_ERR_CUDA;
  return CKDA_OK;
}

}  // extern "C"
