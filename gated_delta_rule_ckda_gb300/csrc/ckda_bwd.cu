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
//   dbeta = <du, v - p>,   dk = D u + G dp,
//   dG = D + k dp^T,       dalpha_i = sum_j dG_ij S_ij,   D <- Diag(alpha) dG;
//
// dq = scale S' do comes from a forward pass, and dh0 is the final D.
//
// Every column j of S evolves on its own; only p and du sum over the rows of
// a column, while dq, dk, dalpha and dbeta sum over the columns.  So the
// state is split by columns: a cluster of ceil(dv / 32) CTAs owns one
// (sequence, head), each CTA 32 columns, and each of its 256 threads 16 rows
// (16g .. 16g + 15) of one column of S and of D, in registers.  A column's
// sums are 3-step shuffles among its 8 row groups (lanes of one warp).  The
// sums over columns are reduced over the 4 columns of a warp by halving
// exchanges, over the 8 warps in shared memory, and over the cluster's CTAs
// through distributed shared memory, once per 8 tokens, in a fixed order.
//
// Recomputation: pass 1 runs the forward and keeps the state slice before
// every 64th token (a checkpoint).  Pass 2 takes the 64-token chunks in
// reverse: (a) it reruns the chunk from its checkpoint, keeping the state
// before every 2nd token (a sub-checkpoint) and forming dq; (b) it takes the
// chunk's 2-token groups in reverse, reruns each from its sub-checkpoint with
// both states kept in registers, and walks them backward.  Two tokens per
// group keep a thread at 128 registers, so that 2 CTAs share an SM (16 warps)
// and 76 clusters of 4 run at once on 152 SMs.  Arithmetic is fp32.
#include "ckda_internal.cuh"

namespace ckda {
namespace {

constexpr int CW = 32;           // state columns per CTA
constexpr int NTH = 8 * CW;      // threads per CTA: warps of 4 columns x 8 row groups
constexpr int NW = NTH / 32;     // warps per CTA
constexpr int MIN_CTAS = 512 / NTH;  // CTAs per SM at 128 registers a thread
constexpr int RPT = 16;          // rows per thread
constexpr int CK = 64;           // tokens per checkpoint interval
constexpr int SG = 2;            // tokens per group (sub-checkpoint interval)
constexpr int NSG = CK / SG;     // groups per chunk
constexpr int VP = 20;           // padded stride of a row group in a channel vector
constexpr int VEC = 8 * VP;      // one padded channel vector (128 channels)
constexpr int SLOT = NTH * RPT;  // floats of one CTA's state slice
constexpr int PART = 2 * 128 + 4;  // per token: dk (128), dalpha (128), dbeta
constexpr int RT = 8;            // tokens per reduction over the cluster
static_assert(NTH >= 128, "one thread per key channel publishes the token vectors");
static_assert(SG * CW + SG <= NTH, "threads that load v, do and beta");
static_assert(CK % SG == 0 && RT % SG == 0, "groups tile chunks and reduction rounds");

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
  float* states;            // workspace: checkpoints, then each CTA's sub-checkpoints
  const int32_t* cu_seqlens;
  int N;                    // sequences (packed) or B (dense)
  int B, H, T, dk, dv;
  int ncb;                  // CTAs (column blocks) per (sequence, head)
  float scale;
};

// Checkpoint slots per workspace: dense units own ceil(T / CK) each; packed
// sequences share their head's ceil(T / CK) + N (sequence n starting at token
// t0 takes slots floor(t0 / CK) + n onward, which never overlap the next
// sequence's).  A slot holds ncb state slices.
__host__ __device__ inline size_t bwd_ck_slots(bool packed, int N, int H, int T) {
  const size_t per = ((size_t)T + CK - 1) / CK;
  return packed ? (size_t)H * (per + (size_t)N) : (size_t)N * H * per;
}

// Shared memory, in floats.
constexpr int SM_VEC = 0;                        // [2][SG][3][VEC]: k, alpha, scale q
constexpr int SM_CV = SM_VEC + 2 * SG * 3 * VEC;  // [2][SG][2][CW]: v, do of this CTA's columns
constexpr int SM_BV = SM_CV + 2 * SG * 2 * CW;   // [2][SG]: beta
constexpr int SM_RED = SM_BV + 2 * SG;           // [2][SG][NW][2][VEC]: per-warp sums over columns
constexpr int SM_REDB = SM_RED + 2 * SG * NW * 2 * VEC;  // [2][SG][NW]: per-warp dbeta
constexpr int SM_PART = SM_REDB + 2 * SG * NW;   // [2][RT][PART]: the CTA's sums, per token
constexpr int SM_TOK = SM_PART + 2 * RT * PART;  // [2][RT] int: the token of each PART row
constexpr int SM_FLOATS = SM_TOK + 2 * RT;
constexpr size_t kSmemBytes = (size_t)SM_FLOATS * sizeof(float);

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// every thread of every CTA of the cluster; orders the shared-memory writes
// before it with the distributed reads after it
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// a float of CTA `rank`'s shared memory, at the offset of p in this CTA's
__device__ __forceinline__ float ld_cluster(const float* p, uint32_t rank) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}
// the sum over the cluster's ncb CTAs of the float at p, in rank order: every
// remote load is issued before the first add waits
__device__ __forceinline__ float sum_cluster(const float* p, int ncb) {
  float x[8];
#pragma unroll
  for (int rr = 0; rr < 8; ++rr) x[rr] = rr < ncb ? ld_cluster(p, (uint32_t)rr) : 0.f;
  float acc = x[0];
#pragma unroll
  for (int rr = 1; rr < 8; ++rr) acc += x[rr];
  return acc;
}

// Sums x over the 4 columns of a warp (lanes l, l ^ 8, l ^ 16, l ^ 24 share a
// row group).  N = 16: afterwards lane (cw, g) holds rows 16g + 4cw + e,
// e < 4.  N = 32 (two quantities of 16 rows): quantity cw >> 1, rows
// 16g + 8 (cw & 1) + e, e < 8.
template <int N>
__device__ __forceinline__ void sum_columns(float (&x)[N], float (&z)[N / 4], int lane) {
  constexpr int H1 = N / 2, H2 = N / 4;
  float y[H1];
  const bool hi = (lane & 16) != 0, hi2 = (lane & 8) != 0;
#pragma unroll
  for (int e = 0; e < H1; ++e) {
    const float send = hi ? x[e] : x[e + H1];
    const float keep = hi ? x[e + H1] : x[e];
    y[e] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int e = 0; e < H2; ++e) {
    const float send = hi2 ? y[e] : y[e + H2];
    const float keep = hi2 ? y[e + H2] : y[e];
    z[e] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}
__device__ __forceinline__ float sum_rows(float x) {   // over the 8 row groups of a column
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x + __shfl_xor_sync(0xffffffffu, x, 4);
}

template <typename IO>
__global__ void __launch_bounds__(NTH, MIN_CTAS) bwd_kernel(const BwdArgs a) {
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  const IO* q = static_cast<const IO*>(a.q);
  const IO* k = static_cast<const IO*>(a.k);
  const IO* v = static_cast<const IO*>(a.v);
  const IO* al = static_cast<const IO*>(a.alpha);
  const IO* be = static_cast<const IO*>(a.beta);
  const IO* dout = static_cast<const IO*>(a.dout);

  const uint32_t rank = cluster_rank();        // column block
  const int unit = blockIdx.x / a.ncb;
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
  const int dk = a.dk, dv = a.dv;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int g = lane & 7, cw = lane >> 3;
  const int c = 4 * w + cw;                    // column within the block
  const int j = (int)rank * CW + c;            // state column
  const bool colok = j < dv;
  const size_t sidx = ((size_t)n * a.H + h) * (size_t)dk * dv;

  // ---- per-token vectors, a group of SG tokens at a time, double-buffered
  float rk[SG], ra[SG], rq[SG], rv = 0.f, rdo = 0.f, rb = 0.f;
  auto fetch = [&](int t0) {   // tokens t0 .. t0 + SG - 1 into registers
#pragma unroll
    for (int s = 0; s < SG; ++s) {
      const int t = t0 + s;
      rk[s] = 0.f; ra[s] = 1.f; rq[s] = 0.f;   // channels past dk, tokens past len: identity
      if (t >= 0 && t < len && tid < dk) {
        const size_t o = (size_t)(row0 + t) * dk + tid;
        rk[s] = ld_io(k + o);
        ra[s] = ld_io(al + o);
        rq[s] = a.scale * ld_io(q + o);
      }
    }
    rv = 0.f; rdo = 0.f; rb = 0.f;
    if (tid < SG * CW) {
      const int t = t0 + tid / CW, jj = (int)rank * CW + tid % CW;
      if (t >= 0 && t < len && jj < dv) {
        const size_t o = (size_t)(row0 + t) * dv + jj;
        rv = ld_io(v + o);
        rdo = ld_io(dout + o);
      }
    } else if (tid >= SG * CW && tid < SG * CW + SG) {
      const int t = t0 + tid - SG * CW;
      if (t >= 0 && t < len) rb = ld_io(be + (row0 + t));
    }
  };
  auto publish = [&](int vb) {
    float* V = sm + SM_VEC + vb * SG * 3 * VEC;
    const int pi = VP * (tid >> 4) + (tid & 15);
    if (tid < 128) {
#pragma unroll
      for (int s = 0; s < SG; ++s) {
        V[(s * 3 + 0) * VEC + pi] = rk[s];
        V[(s * 3 + 1) * VEC + pi] = ra[s];
        V[(s * 3 + 2) * VEC + pi] = rq[s];
      }
    }
    if (tid < SG * CW) {
      float* C = sm + SM_CV + vb * SG * 2 * CW;
      C[(tid / CW) * 2 * CW + tid % CW] = rv;
      C[(tid / CW) * 2 * CW + CW + tid % CW] = rdo;
    } else if (tid >= SG * CW && tid < SG * CW + SG) {
      sm[SM_BV + vb * SG + tid - SG * CW] = rb;
    }
  };
  // L2 prefetch of the group starting at t0 (one ahead of the register fetch)
  auto prefetch_group = [&](int t0) {
#pragma unroll
    for (int s = 0; s < SG; ++s) {
      const int t = t0 + s;
      if (t >= 0 && t < len && tid < dk) {
        const size_t o = (size_t)(row0 + t) * dk + tid;
        prefetch_l2(k + o);
        prefetch_l2(al + o);
        prefetch_l2(q + o);
      }
    }
    if (tid < SG * CW) {
      const int t = t0 + tid / CW, jj = (int)rank * CW + tid % CW;
      if (t >= 0 && t < len && jj < dv) {
        prefetch_l2(v + (size_t)(row0 + t) * dv + jj);
        prefetch_l2(dout + (size_t)(row0 + t) * dv + jj);
      }
    }
  };
  int vg = 0;   // running count of vector groups (buffer = parity)
  // loads the group fetched last, fetches the one starting at next0 into
  // registers and prefetches the one after it (at next0 + step) into L2
  auto next_group = [&](int next0, int step) -> int {
    const int vb = vg & 1;
    ++vg;
    publish(vb);
    __syncthreads();
    fetch(next0);
    prefetch_group(next0 + step);
    return vb;
  };
  auto K_of = [&](int vb, int s) { return sm + SM_VEC + (vb * SG + s) * 3 * VEC + VP * g; };
  auto v_of = [&](int vb, int s) { return sm[SM_CV + (vb * SG + s) * 2 * CW + c]; };
  auto do_of = [&](int vb, int s) { return sm[SM_CV + (vb * SG + s) * 2 * CW + CW + c]; };
  auto beta_of = [&](int vb, int s) { return sm[SM_BV + vb * SG + s]; };

  // one forward step of this thread's rows of column j: Sn = alpha S + k u
  auto forward = [&](const float (&S)[RPT], float (&Sn)[RPT], int vb, int s) {
    const float* K = K_of(vb, s);
    float gq[RPT];
    float p = 0.f;
#pragma unroll
    for (int m = 0; m < RPT / 4; ++m) {
      const float4 k4 = *reinterpret_cast<const float4*>(K + 4 * m);
      const float4 a4 = *reinterpret_cast<const float4*>(K + VEC + 4 * m);
      gq[4 * m + 0] = a4.x * S[4 * m + 0];
      gq[4 * m + 1] = a4.y * S[4 * m + 1];
      gq[4 * m + 2] = a4.z * S[4 * m + 2];
      gq[4 * m + 3] = a4.w * S[4 * m + 3];
      p = fmaf(k4.x, gq[4 * m + 0], p);
      p = fmaf(k4.y, gq[4 * m + 1], p);
      p = fmaf(k4.z, gq[4 * m + 2], p);
      p = fmaf(k4.w, gq[4 * m + 3], p);
    }
    p = sum_rows(p);
    const float u = beta_of(vb, s) * (v_of(vb, s) - p);
#pragma unroll
    for (int m = 0; m < RPT / 4; ++m) {
      const float4 k4 = *reinterpret_cast<const float4*>(K + 4 * m);
      Sn[4 * m + 0] = fmaf(k4.x, u, gq[4 * m + 0]);
      Sn[4 * m + 1] = fmaf(k4.y, u, gq[4 * m + 1]);
      Sn[4 * m + 2] = fmaf(k4.z, u, gq[4 * m + 2]);
      Sn[4 * m + 3] = fmaf(k4.w, u, gq[4 * m + 3]);
    }
  };

  int rg = 0;   // running count of cluster reduction rounds (partial buffer = parity)
  int gcount = 0;   // running count of reduced groups (per-warp sum buffer = parity)
  float* red = sm + SM_RED;
  float* part = sm + SM_PART;
  int* tok = reinterpret_cast<int*>(sm + SM_TOK);
  // the CTA's sum over its NW warps of the per-warp sums of token s of group
  // buffer gb (after a barrier), into row `slot` of partial buffer pb
  auto cta_sum = [&](int gb, int s, int pb, int slot, int nq) {
    const float* R = red + (gb * SG + s) * NW * 2 * VEC;
    for (int e = tid; e < nq * 128; e += NTH) {
      const int qq = e >> 7, i = e & 127;
      const int off = qq * VEC + VP * (i >> 4) + (i & 15);
      float x = 0.f;
#pragma unroll
      for (int ww = 0; ww < NW; ++ww) x += R[ww * 2 * VEC + off];
      part[(pb * RT + slot) * PART + e] = x;
    }
  };
  // the cluster's sums of the cnt tokens in partial buffer pb: each CTA
  // takes every ncb-th item; dq (nq = 1) or dk, dalpha and dbeta (nq = 2)
  auto cluster_reduce = [&](int pb, int cnt, int nq) {
    cluster_sync();
    const int per = nq * dk;
    const int items = cnt * per + (nq == 2 ? cnt : 0);
    for (int it = (int)rank + a.ncb * tid; it < items; it += a.ncb * NTH) {
      int slot, e;
      if (it < cnt * per) {
        slot = it / per;
        const int rem = it % per;
        e = (rem / dk) * 128 + rem % dk;
      } else {
        slot = it - cnt * per;
        e = 256;
      }
      const int t = tok[pb * RT + slot];
      const float x = sum_cluster(part + (pb * RT + slot) * PART + e, a.ncb);
      if (t < len) {
        const size_t row = (size_t)(row0 + t);
        if (nq == 1) st_io(static_cast<IO*>(a.gq) + row * dk + e, a.scale * x);
        else if (e == 256) st_io(static_cast<IO*>(a.gbeta) + row, x);
        else if (e < 128) st_io(static_cast<IO*>(a.gk) + row * dk + e, x);
        else st_io(static_cast<IO*>(a.galpha) + row * dk + (e - 128), x);
      }
    }
  };

  float S[RPT], D[RPT];
  const int i0 = 16 * g;
  // ------------------------------------------------ pass 1: checkpoints
#pragma unroll
  for (int r = 0; r < RPT; ++r)
    S[r] = (a.h0 && colok && i0 + r < dk) ? a.h0[sidx + (size_t)(i0 + r) * dv + j] : 0.f;
  const size_t per_unit_ck = ((size_t)a.T + CK - 1) / CK;
  const size_t ck0 = a.cu_seqlens
                         ? (size_t)h * (per_unit_ck + a.N) + (size_t)(a.cu_seqlens[n] / CK) + n
                         : (size_t)unit * per_unit_ck;
  auto ck_slot = [&](int m) { return a.states + ((ck0 + m) * a.ncb + rank) * SLOT; };
  float* subck = a.states + (bwd_ck_slots(a.cu_seqlens != nullptr, a.N, a.H, a.T) * a.ncb +
                             ((size_t)unit * a.ncb + rank) * NSG) * SLOT;
  auto store_slice = [&](const float (&X)[RPT], float* dst) {
#pragma unroll
    for (int r = 0; r < RPT; ++r) dst[r * NTH + tid] = X[r];
  };
  auto load_slice = [&](float (&X)[RPT], const float* src) {
#pragma unroll
    for (int r = 0; r < RPT; ++r) X[r] = src[r * NTH + tid];
  };

  const int ngr = (len + SG - 1) / SG;
  fetch(0);
  prefetch_group(SG);
  for (int gi = 0; gi < ngr; ++gi) {
    if (gi % NSG == 0) store_slice(S, ck_slot(gi / NSG));
    const int vb = next_group((gi + 1) * SG, SG);
#pragma unroll
    for (int s = 0; s < SG; ++s) {
      float Sn[RPT];
      forward(S, Sn, vb, s);
#pragma unroll
      for (int r = 0; r < RPT; ++r) S[r] = Sn[r];
    }
  }

  // ------------------------------------------------ pass 2: reverse, by chunk
#pragma unroll
  for (int r = 0; r < RPT; ++r)
    D[r] = (a.dhT && colok && i0 + r < dk) ? a.dhT[sidx + (size_t)(i0 + r) * dv + j] : 0.f;
  IO* gv_o = static_cast<IO*>(a.gv);
  const int nck = (len + CK - 1) / CK;
  for (int m = nck - 1; m >= 0; --m) {
    const int g0 = m * NSG, g1 = min(ngr, g0 + NSG);
    // (a) rerun the chunk, keeping sub-checkpoints, and form dq
    load_slice(S, ck_slot(m));
    __syncthreads();   // the previous walk's reads of the vector buffers are done
    fetch(g0 * SG);
    prefetch_group((g0 + 1) * SG);
    int pend = 0;   // tokens in the current partial buffer
    for (int gi = g0; gi < g1; ++gi) {
      store_slice(S, subck + (size_t)(gi - g0) * SLOT);
      const int vb = next_group((gi + 1) * SG, SG);
      const int gb = gcount & 1;
      ++gcount;
#pragma unroll
      for (int s = 0; s < SG; ++s) {
        float Sn[RPT];
        forward(S, Sn, vb, s);
        const float dov = do_of(vb, s);
        float x[RPT], z[RPT / 4];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
          S[r] = Sn[r];
          x[r] = Sn[r] * dov;
        }
        sum_columns<RPT>(x, z, lane);
        *reinterpret_cast<float4*>(red + ((gb * SG + s) * NW + w) * 2 * VEC + VP * g + 4 * cw) =
            make_float4(z[0], z[1], z[2], z[3]);
      }
      __syncthreads();
      const int pb = rg & 1;
#pragma unroll
      for (int s = 0; s < SG; ++s) {
        cta_sum(gb, s, pb, pend + s, 1);
        if (tid == 0) tok[pb * RT + pend + s] = gi * SG + s;
      }
      pend += SG;
      if (pend == RT || gi == g1 - 1) {   // dq of these tokens
        cluster_reduce(pb, pend, 1);
        ++rg;
        pend = 0;
      }
    }
    // (b) walk the chunk's groups backward
    __syncthreads();   // (a)'s reads of the vector buffers are done
    fetch((g1 - 1) * SG);
    prefetch_group((g1 - 2) * SG);
    // the first group's vectors; each later group's are published at the
    // end of the group before it, under that group's barrier
    int vb = next_group((g1 - 2) * SG, -SG);
    pend = 0;
    for (int gi = g1 - 1; gi >= g0; --gi) {
      float st[SG][RPT];
      load_slice(st[0], subck + (size_t)(gi - g0) * SLOT);
      if (gi > g0) {   // the next group's sub-checkpoint into L1
#pragma unroll
        for (int r = 0; r < RPT; ++r) prefetch_l1(subck + (size_t)(gi - 1 - g0) * SLOT + r * NTH + tid);
      }
      const int gb = gcount & 1;
      ++gcount;
#pragma unroll
      for (int s = 0; s + 1 < SG; ++s) forward(st[s], st[s + 1], vb, s);
#pragma unroll
      for (int s = SG - 1; s >= 0; --s) {
        const int t = gi * SG + s;
        const float* K = K_of(vb, s);
        const float dov = do_of(vb, s), vj = v_of(vb, s), bt = beta_of(vb, s);
        float p = 0.f, du = 0.f;
#pragma unroll
        for (int mm = 0; mm < RPT / 4; ++mm) {
          const float4 k4 = *reinterpret_cast<const float4*>(K + 4 * mm);
          const float4 a4 = *reinterpret_cast<const float4*>(K + VEC + 4 * mm);
          const float4 q4 = *reinterpret_cast<const float4*>(K + 2 * VEC + 4 * mm);
          const float kk[4] = {k4.x, k4.y, k4.z, k4.w}, aa[4] = {a4.x, a4.y, a4.z, a4.w};
          const float qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = 4 * mm + e;
            D[r] = fmaf(qq[e], dov, D[r]);
            p = fmaf(kk[e] * aa[e], st[s][r], p);
            du = fmaf(kk[e], D[r], du);
          }
        }
        p = sum_rows(p);
        du = sum_rows(du);
        const float u = bt * (vj - p), dp = -bt * du;
        if (g == 0 && colok && t < len) st_io(gv_o + (size_t)(row0 + t) * dv + j, bt * du);
        float x[2 * RPT];
#pragma unroll
        for (int mm = 0; mm < RPT / 4; ++mm) {
          const float4 k4 = *reinterpret_cast<const float4*>(K + 4 * mm);
          const float4 a4 = *reinterpret_cast<const float4*>(K + VEC + 4 * mm);
          const float kk[4] = {k4.x, k4.y, k4.z, k4.w}, aa[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = 4 * mm + e;
            const float sp = st[s][r];
            x[r] = fmaf(D[r], u, aa[e] * sp * dp);        // dk
            const float dG = fmaf(kk[e], dp, D[r]);
            x[RPT + r] = dG * sp;                         // dalpha
            D[r] = aa[e] * dG;
          }
        }
        float z[2 * RPT / 4];
        sum_columns<2 * RPT>(x, z, lane);
        float* R = red + ((gb * SG + s) * NW + w) * 2 * VEC + (cw >> 1) * VEC + VP * g +
                   8 * (cw & 1);
        *reinterpret_cast<float4*>(R) = make_float4(z[0], z[1], z[2], z[3]);
        *reinterpret_cast<float4*>(R + 4) = make_float4(z[4], z[5], z[6], z[7]);
        // dbeta over this warp's 4 columns
        float db = (g == 0) ? du * (vj - p) : 0.f;
        db += __shfl_xor_sync(0xffffffffu, db, 8);
        db += __shfl_xor_sync(0xffffffffu, db, 16);
        if (lane == 0) sm[SM_REDB + (gb * SG + s) * NW + w] = db;
      }
      // the next group's vectors (fetched during this one) into the other
      // buffer, whose last reader was the group before this one
      const int vb_next = vg & 1;
      if (gi > g0) {
        ++vg;
        publish(vb_next);
      }
      __syncthreads();   // this group's per-warp sums and the next group's vectors
      if (gi > g0) {
        fetch((gi - 2) * SG);
        prefetch_group((gi - 3) * SG);
      }
      const int pb = rg & 1;
#pragma unroll
      for (int s = 0; s < SG; ++s) {
        cta_sum(gb, s, pb, pend + s, 2);
        if (tid == 0) {
          const float* RB = sm + SM_REDB + (gb * SG + s) * NW;
          float x = 0.f;
          for (int ww = 0; ww < NW; ++ww) x += RB[ww];
          part[(pb * RT + pend + s) * PART + 256] = x;
          tok[pb * RT + pend + s] = gi * SG + s;
        }
      }
      pend += SG;
      if (pend == RT || gi == g0) {   // dk, dalpha, dbeta of these tokens
        cluster_reduce(pb, pend, 2);
        ++rg;
        pend = 0;
      }
      vb = vb_next;
    }
  }
  if (a.gh0 && colok) {
#pragma unroll
    for (int r = 0; r < RPT; ++r)
      if (i0 + r < dk) a.gh0[sidx + (size_t)(i0 + r) * dv + j] = D[r];
  }
  cluster_sync();   // no CTA leaves while another may still read its shared memory
}

template <typename IO>
cudaError_t launch_io(const BwdArgs& a, int units, cudaStream_t s) {
  const cudaError_t err = cudaFuncSetAttribute(
      bwd_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(units * a.ncb));
  cfg.blockDim = dim3(NTH);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)a.ncb;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bwd_kernel<IO>, a);
}

}  // namespace
}  // namespace ckda

using namespace ckda;

extern "C" size_t ckda_bwd_workspace_bytes(int num_seqs, int B, int H, int T, int dk, int dv) {
  if (B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1 || num_seqs < 0) return 0;
  const bool packed = num_seqs > 0;
  const int N = packed ? num_seqs : B;
  const size_t ncb = (size_t)(dv + CW - 1) / CW;
  const size_t slices = bwd_ck_slots(packed, N, H, T) * ncb + (size_t)N * H * ncb * NSG;
  return slices * SLOT * sizeof(float);
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
  if (dk > 128 || dv > 128) return CKDA_ERR_UNSUPPORTED;
  if ((long long)B * H * T > 0x7fffffffLL) return CKDA_ERR_UNSUPPORTED;
  const int units = (cu_seqlens ? num_seqs : B) * H;
  const int ncb = (dv + CW - 1) / CW;
  if ((long long)units * ncb > 0x7fffffffLL) return CKDA_ERR_UNSUPPORTED;
  const size_t need = ckda_bwd_workspace_bytes(cu_seqlens ? num_seqs : 0, B, H, T, dk, dv);
  if (need > 0 && (!workspace || workspace_bytes < need)) return CKDA_ERR_WORKSPACE;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 15) != 0) return CKDA_ERR_WORKSPACE;
  BwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.dout = d_o;
  a.h0 = h0; a.dhT = d_hT;
  a.gq = d_q; a.gk = d_k; a.gv = d_v; a.galpha = d_alpha; a.gbeta = d_beta; a.gh0 = d_h0;
  a.states = static_cast<float*>(workspace);
  a.cu_seqlens = cu_seqlens;
  a.N = cu_seqlens ? num_seqs : B;
  a.B = B; a.H = H; a.T = T; a.dk = dk; a.dv = dv;
  a.ncb = ncb;
  a.scale = scale;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t err = io_dtype == CKDA_F32 ? launch_io<float>(a, units, s)
                                               : launch_io<__nv_bfloat16>(a, units, s);
  return err == cudaSuccess ? CKDA_OK : CKDA_ERR_CUDA;
}
