// ckda_bwd.cu -- backward of the CKDA recurrence on CUDA cores, token by token.
//
// Gradients of L = sum_t <o_t, do_t> + <H_T, dH_T> with respect to q, k, v,
// alpha, beta and h0, by reverse-mode differentiation of the recurrence of
// "Complex KDA: Understanding and Enhancing the Expressivity of Kimi Delta
// Attention" (Sec. 2, Eq. (1); App. B.2, Eq. (9)), taken in the bounded case
// study's step order.  Forward step t, state S (dk x dv, rows = key channels):
//
//   G = Diag(alpha) S,   p = G^T k,   u = beta (v - p),   S' = G + k u^T,
//   o = S'^T (scale q).
//
// Reverse step t, with D = dL/dS' (starting from dH_T):
//
//   D += (scale q) do^T,   du = D^T k,   dv = beta du,   dp = -beta du,
//   dbeta = <du, v - p>,   dk = D u + Diag(alpha) S dp,
//   dG = D + k dp^T,       dalpha_i = sum_j dG_ij S_ij,   D <- Diag(alpha) dG;
//
// dq = scale S' do comes from the forward pass, and dh0 is the final D.
//
// One block of 512 threads owns one (sequence, head).  S and D live in
// shared memory as 128 x 129 fp32 tiles (the padding makes both a column walk
// and a row walk conflict-free), so that each step alternates a column phase
// (lane j = state column: p, u, du, dv, D += q do^T) and a row phase (lane i
// = key channel: dk, dalpha, the update of D, and dq).  Each lane is four
// threads, each walking a quarter of the other index; the quarters' partial
// sums meet in shared memory.  Pass 1 runs the forward and stores the state
// before every 64th token (a checkpoint).  Pass 2 takes the chunks of 64
// tokens in reverse: it recomputes the chunk from its checkpoint, storing the
// state before each token in the unit's chunk buffer and writing dq, then
// walks the chunk backward, reading the next state back with cp.async into a
// second tile while the current one is in use and fetching the next token's
// vectors into registers.  Arithmetic is fp32.
#include "ckda_internal.cuh"

namespace ckda {
namespace {

constexpr int NB = 512;   // threads per block: 128 lanes x 4 parts
constexpr int NL = 128;   // lanes: state columns (column phases) or key channels (row phases)
constexpr int LD = 129;   // padded row stride of the shared tiles

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* alpha;
  const void* beta;
  const void* dout;
  const float* h0;
  const float* dhT;
  void* gq;                 // gradients, in the I/O dtype
  void* gk;
  void* gv;
  void* galpha;
  void* gbeta;
  float* gh0;               // fp32
  float* states;            // workspace: checkpoints, then one chunk buffer per unit
  const int32_t* cu_seqlens;
  int N;                    // sequences (packed) or B (dense)
  int B, H, T, dk, dv;
  float scale;
};

constexpr int CK = 64;    // tokens per checkpoint interval (and per recomputed chunk)

// Workspace, in dk x dv fp32 tiles: the checkpoints (the state before every
// CK-th token of each unit), then CK tiles per unit for the states of the
// chunk being walked.  Dense units own ceil(T / CK) checkpoint slots each;
// packed sequences share their head's ceil(T / CK) + N slots (sequence n
// starting at token t0 takes slots floor(t0 / CK) + n onward, which never
// overlap the next sequence's).
__host__ __device__ inline size_t bwd_ck_slots(bool packed, int N, int H, int T) {
  const size_t per = ((size_t)T + CK - 1) / CK;
  return packed ? (size_t)H * (per + (size_t)N) : (size_t)N * H * per;
}

// two state tiles (pass 2 double-buffers them), the gradient tile D, seven
// per-token vectors and five [4][128] tables of per-part partial sums
constexpr size_t kSmemFloats = (size_t)3 * NL * LD + 7 * NL + 5 * 4 * NL + 32;
constexpr size_t kSmemBytes = kSmemFloats * sizeof(float);

__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <typename IO>
__global__ void __launch_bounds__(NB, 1) bwd_kernel(const BwdArgs a) {
  extern __shared__ float smf[];
  float* Sb[2] = {smf, smf + NL * LD};   // [128][LD] each
  float* D = smf + 2 * NL * LD;          // [128][LD]
  float* kv = D + NL * LD;               // k_t
  float* av = kv + NL;                   // alpha_t
  float* qv = av + NL;                   // scale * q_t
  float* dov = qv + NL;                  // do_t
  float* vv = dov + NL;                  // v_t
  float* uv = vv + NL;                   // u_t
  float* dpv = uv + NL;                  // dp_t
  float* P0 = dpv + NL;                  // [4][128] per-part partial sums
  float* P1 = P0 + 4 * NL;
  float* P2 = P1 + 4 * NL;
  float* P3 = P2 + 4 * NL;
  float* P4 = P3 + 4 * NL;
  float* red = P4 + 4 * NL;              // [0..3] dbeta per warp of part 0, [8] beta_t

  const IO* q = static_cast<const IO*>(a.q);
  const IO* k = static_cast<const IO*>(a.k);
  const IO* v = static_cast<const IO*>(a.v);
  const IO* al = static_cast<const IO*>(a.alpha);
  const IO* be = static_cast<const IO*>(a.beta);
  const IO* dout = static_cast<const IO*>(a.dout);

  const int unit = blockIdx.x;
  const int n = unit / a.H, h = unit % a.H;
  long row0;
  int len;
  if (a.cu_seqlens) {
    const int t0 = a.cu_seqlens[n];
    len = a.cu_seqlens[n + 1] - t0;
    row0 = (long)h * a.T + t0;
  } else {
    len = a.T;
    row0 = ((long)n * a.H + h) * a.T;
  }
  const int tid = threadIdx.x;
  const int x = tid & (NL - 1);          // lane: column j or channel i
  const int part = tid >> 7;             // which quarter of the other index
  const int dk = a.dk, dv = a.dv;
  const int lo = 32 * part;              // this part's range of the other index
  const int hi_k = min(lo + 32, dk), hi_v = min(lo + 32, dv);
  const bool colx = x < dv, rowx = x < dk;
  const size_t sidx = ((size_t)n * a.H + h) * (size_t)dk * dv;
  const size_t tile = (size_t)dk * dv;

  // token vectors, fetched one token ahead into registers by part 0
  float rk = 0.f, ra = 1.f, rq = 0.f, rv = 0.f, rdo = 0.f, rb = 0.f;
  auto fetch = [&](int t) {
    if (part != 0 || t < 0 || t >= len) return;
    const long r = row0 + t;
    if (rowx) {
      rk = ld_io(k + (size_t)r * dk + x);
      ra = ld_io(al + (size_t)r * dk + x);
      rq = a.scale * ld_io(q + (size_t)r * dk + x);
    }
    if (colx) {
      rv = ld_io(v + (size_t)r * dv + x);
      rdo = ld_io(dout + (size_t)r * dv + x);
    }
    if (x == 0) rb = ld_io(be + r);
  };
  auto publish_vectors = [&]() {
    if (part != 0) return;
    if (rowx) { kv[x] = rk; av[x] = ra; qv[x] = rq; }
    if (colx) { vv[x] = rv; dov[x] = rdo; }
    if (x == 0) red[8] = rb;
  };

  // checkpoint slots and this unit's chunk buffer (in tiles)
  const size_t per_unit_ck = ((size_t)a.T + CK - 1) / CK;
  const size_t ck0 = a.cu_seqlens
                         ? (size_t)h * (per_unit_ck + a.N) + (size_t)(a.cu_seqlens[n] / CK) + n
                         : (size_t)unit * per_unit_ck;
  float* chunkbuf = a.states + (bwd_ck_slots(a.cu_seqlens != nullptr, a.N, a.H, a.T) +
                                (size_t)unit * CK) * tile;
  auto ck_tile = [&](int m) { return a.states + (ck0 + m) * tile; };

  // one forward step on the tile S (token t's vectors published and visible):
  // S <- Diag(alpha) S + k u^T with u = beta (v - (Diag(alpha) S)^T k)
  auto forward_step = [&](float* S) {
    if (colx) {
      float p = 0.f;
#pragma unroll 4
      for (int i = lo; i < hi_k; ++i) p = fmaf(kv[i] * av[i], S[i * LD + x], p);
      P0[part * NL + x] = p;
    }
    __syncthreads();
    if (colx) {
      const float p = P0[x] + P0[NL + x] + P0[2 * NL + x] + P0[3 * NL + x];
      const float u = red[8] * (vv[x] - p);
#pragma unroll 4
      for (int i = lo; i < hi_k; ++i) S[i * LD + x] = fmaf(av[i], S[i * LD + x], kv[i] * u);
    }
    __syncthreads();
  };
  auto store_tile = [&](const float* S, float* dst) {  // this thread's rows of column x
    if (colx)
      for (int i = lo; i < hi_k; ++i) dst[(size_t)i * dv + x] = S[i * LD + x];
  };

  // ------------------------------------------------ pass 1: checkpoints
  float* S = Sb[0];
  if (colx)
    for (int i = lo; i < hi_k; ++i) S[i * LD + x] = a.h0 ? a.h0[sidx + (size_t)i * dv + x] : 0.f;
  fetch(0);
  for (int t = 0; t < len; ++t) {
    publish_vectors();
    if (t % CK == 0) store_tile(S, ck_tile(t / CK));
    __syncthreads();
    fetch(t + 1);
    forward_step(S);
  }

  // ------------------------------------------------ pass 2: reverse, by chunk
  if (colx)
    for (int i = lo; i < hi_k; ++i) D[i * LD + x] = a.dhT ? a.dhT[sidx + (size_t)i * dv + x] : 0.f;
  // the state before token t (of the chunk starting at t0) goes to tile t mod 2
  auto fetch_state = [&](int t, int t0) {
    if (t < t0 || !colx) return;
    const float* st = chunkbuf + (size_t)(t - t0) * tile + x;
    float* dst = Sb[t & 1];
    for (int i = lo; i < hi_k; ++i) cp_async4(dst + i * LD + x, st + (size_t)i * dv);
  };
  const int nck = (len + CK - 1) / CK;
  for (int m = nck - 1; m >= 0; --m) {
    const int t0 = m * CK, t1 = min(len, t0 + CK);
    // (a) recompute the chunk from its checkpoint, storing the state before
    // each token and writing dq = scale S' do
    __syncthreads();  // the previous walk's last reads of the tiles are done
    if (colx) {
      const float* src = ck_tile(m);
      for (int i = lo; i < hi_k; ++i) S[i * LD + x] = src[(size_t)i * dv + x];
    }
    fetch(t0);
    for (int t = t0; t < t1; ++t) {
      const long r = row0 + t;
      publish_vectors();
      store_tile(S, chunkbuf + (size_t)(t - t0) * tile);
      __syncthreads();
      if (t + 1 < t1) fetch(t + 1);
      forward_step(S);
      if (rowx) {  // dq_i = scale * sum_j S'_ij do_j (scale is applied below)
        float acc = 0.f;
#pragma unroll 4
        for (int j = lo; j < hi_v; ++j) acc = fmaf(S[x * LD + j], dov[j], acc);
        P1[part * NL + x] = acc;
      }
      __syncthreads();
      if (part == 0 && rowx)
        st_io(static_cast<IO*>(a.gq) + (size_t)r * dk + x,
              a.scale * (P1[x] + P1[NL + x] + P1[2 * NL + x] + P1[3 * NL + x]));
    }
    __syncthreads();  // the recompute's reads of S and its global stores are done
    // (b) walk the chunk backward
    fetch_state(t1 - 1, t0);
    cp_async_commit();
    fetch(t1 - 1);
    for (int t = t1 - 1; t >= t0; --t) {
      const long r = row0 + t;
      float* St = Sb[t & 1];
      cp_async_wait_all();
      publish_vectors();
      __syncthreads();  // S_t, the vectors, and the previous step's D are visible
      fetch_state(t - 1, t0);
      cp_async_commit();
      if (t - 1 >= t0) fetch(t - 1);
      if (colx) {
        const float doj = dov[x];
        float p = 0.f, du = 0.f;
#pragma unroll 4
        for (int i = lo; i < hi_k; ++i) {
          const float d = fmaf(qv[i], doj, D[i * LD + x]);
          D[i * LD + x] = d;
          p = fmaf(kv[i] * av[i], St[i * LD + x], p);
          du = fmaf(kv[i], d, du);
        }
        P0[part * NL + x] = p;
        P1[part * NL + x] = du;
      }
      __syncthreads();
      if (part == 0) {
        const float bt = red[8];
        float dbp = 0.f;
        if (colx) {
          const float p = P0[x] + P0[NL + x] + P0[2 * NL + x] + P0[3 * NL + x];
          const float du = P1[x] + P1[NL + x] + P1[2 * NL + x] + P1[3 * NL + x];
          const float vj = vv[x];
          uv[x] = bt * (vj - p);
          dpv[x] = -bt * du;
          st_io(static_cast<IO*>(a.gv) + (size_t)r * dv + x, bt * du);
          dbp = du * (vj - p);
        }
#pragma unroll
        for (int mm = 16; mm >= 1; mm >>= 1) dbp += __shfl_xor_sync(0xffffffffu, dbp, mm);
        if ((x & 31) == 0) red[x >> 5] = dbp;
      }
      __syncthreads();
      if (rowx) {
        const float ki = kv[x], ai = av[x];
        float gk = 0.f, gs = 0.f, ga = 0.f;
#pragma unroll 4
        for (int j = lo; j < hi_v; ++j) {
          const float d = D[x * LD + j], s = St[x * LD + j], dpj = dpv[j];
          gk = fmaf(d, uv[j], gk);
          gs = fmaf(s, dpj, gs);
          const float dG = fmaf(ki, dpj, d);
          ga = fmaf(dG, s, ga);
          D[x * LD + j] = ai * dG;
        }
        P2[part * NL + x] = fmaf(ai, gs, gk);
        P3[part * NL + x] = ga;
      }
      __syncthreads();
      if (part == 0 && rowx) {
        st_io(static_cast<IO*>(a.gk) + (size_t)r * dk + x,
              P2[x] + P2[NL + x] + P2[2 * NL + x] + P2[3 * NL + x]);
        st_io(static_cast<IO*>(a.galpha) + (size_t)r * dk + x,
              P3[x] + P3[NL + x] + P3[2 * NL + x] + P3[3 * NL + x]);
      }
      if (tid == 0) st_io(static_cast<IO*>(a.gbeta) + r, red[0] + red[1] + red[2] + red[3]);
    }
    cp_async_wait_all();
  }
  __syncthreads();
  if (a.gh0 && colx)
    for (int i = lo; i < hi_k; ++i) a.gh0[sidx + (size_t)i * dv + x] = D[i * LD + x];
}

template <typename IO>
cudaError_t launch_io(const BwdArgs& a, int units, cudaStream_t s) {
  cudaError_t err = cudaFuncSetAttribute(bwd_kernel<IO>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  bwd_kernel<IO><<<units, NB, kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace
}  // namespace ckda

using namespace ckda;

extern "C" size_t ckda_bwd_workspace_bytes(int num_seqs, int B, int H, int T, int dk, int dv) {
  if (B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1 || num_seqs < 0) return 0;
  const bool packed = num_seqs > 0;
  const int N = packed ? num_seqs : B;
  const size_t tiles = bwd_ck_slots(packed, N, H, T) + (size_t)N * H * CK;
  return tiles * (size_t)dk * dv * sizeof(float);
}

extern "C" ckda_status ckda_bwd(const void* q, const void* k, const void* v, const void* alpha,
                                const void* beta, const float* h0, const void* d_o,
                                const float* d_hT, void* d_q, void* d_k, void* d_v,
                                void* d_alpha, void* d_beta, float* d_h0,
                                const int32_t* cu_seqlens, int num_seqs, int B, int H, int T,
                                int dk, int dv, ckda_dtype io_dtype, float scale, void* workspace,
                                size_t workspace_bytes, void* stream) {
  if (io_dtype != CKDA_F32 && io_dtype != CKDA_BF16) return CKDA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1) return CKDA_ERR_INVALID_ARG;
  if (!(scale == scale)) return CKDA_ERR_INVALID_ARG;
  if (cu_seqlens) {
    if (B != 1 || num_seqs < 1) return CKDA_ERR_INVALID_ARG;
  } else if (num_seqs != 0 && num_seqs != B) {
    return CKDA_ERR_INVALID_ARG;
  }
  if (T > 0 && (!q || !k || !v || !alpha || !beta || !d_o || !d_q || !d_k || !d_v ||
                !d_alpha || !d_beta))
    return CKDA_ERR_INVALID_ARG;
  if (dk > NL || dv > NL) return CKDA_ERR_UNSUPPORTED;
  if ((long long)B * H * T > 0x7fffffffLL) return CKDA_ERR_UNSUPPORTED;
  const size_t need = ckda_bwd_workspace_bytes(cu_seqlens ? num_seqs : 0, B, H, T, dk, dv);
  if (need > 0 && (!workspace || workspace_bytes < need)) return CKDA_ERR_WORKSPACE;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 15) != 0) return CKDA_ERR_WORKSPACE;
  const int units = (cu_seqlens ? num_seqs : B) * H;
  BwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.dout = d_o;
  a.h0 = h0; a.dhT = d_hT;
  a.gq = d_q; a.gk = d_k; a.gv = d_v; a.galpha = d_alpha; a.gbeta = d_beta; a.gh0 = d_h0;
  a.states = static_cast<float*>(workspace);
  a.cu_seqlens = cu_seqlens;
  a.N = cu_seqlens ? num_seqs : B;
  a.B = B; a.H = H; a.T = T; a.dk = dk; a.dv = dv;
  a.scale = scale;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t err = io_dtype == CKDA_F32 ? launch_io<float>(a, units, s)
                                               : launch_io<__nv_bfloat16>(a, units, s);
  return err == cudaSuccess ? CKDA_OK : CKDA_ERR_CUDA;
}
