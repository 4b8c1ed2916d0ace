// ckda_chunk.cu -- chunkwise CKDA forward on tcgen05 tensor cores (sm_103a).
//
// One CTA owns one (sequence, head) and walks its tokens in chunks of C = 64
// with the fp32 state H^T (dv x dk = 128 x 128) resident in tensor memory.
// The chunk algebra is the WY/UT form of a product of diagonal-plus-rank-one
// transitions ("Complex KDA: Understanding and Enhancing the Expressivity of
// Kimi Delta Attention", Sec. 2: KDA keeps "efficient WY-based chunk-wise
// implementations"; "Kimi Delta Attention: a bounded case study",
// "Chunkwise execution": carrying the state block to block changes cost,
// never the numbers).  For a chunk with initial state H (per channel i,
// Gamma(t<-s) = prod_{s<r<=t} alpha_r, gamma_t = Gamma(t<-0),
// rho_s = Gamma(C<-s)):
//
//   M[t,s] = beta_t sum_i k_ti k_si Gamma(t<-s)_i      (s < t)
//   A[t,s] = sum_i q_ti k_si Gamma(t<-s)_i             (s <= t)
//   T  = (I + M)^-1,   TB = T Diag(beta)
//   W  = TB (k * gamma),           U~ = TB V
//   U  = U~ - W H
//   O  = (q * gamma) H + A U                            -> o (scaled)
//   H' = Diag(gamma_C) H + (k * rho)^T U
//
// Gate products are formed by multiplication only -- never as a ratio of
// prefix products and never in log space -- because alpha may be negative or
// exactly zero (paper Sec. 6 "Implementation": the KDA kernels keep gate
// magnitudes in log space, which signed gates break).  The strictly-lower
// pairs of M and A are split by a binary tree over the chunk: a pair (t, s)
// first separated at tree level L lies in one aligned segment of 2L tokens
// with s in the lower and t in the upper half, and with m the last position
// of the lower half Gamma(t<-s) = [prod_{m<r<=t} alpha_r][prod_{s<r<=m}
// alpha_r]; every level is then one dense contraction of gated operands on
// the tensor cores.  Two levels share one 128 x 64 MMA tile (3 rounds).
//
// Precision: operands of every contraction that touches the state, the
// Grams and A are fp16 (11-bit significand); T Diag(beta), k * gamma and the
// raw bf16 inputs are bf16; all accumulation is fp32 in TMEM, T is fp32.
//
// This version runs the phases of a chunk one after another with all 256
// threads cooperating between barriers; one thread issues every MMA.
#include "ckda_internal.cuh"
#include "sm103.cuh"

#include <cudaTypedefs.h>
#include <mutex>

namespace ckda {
namespace {

constexpr int C = 64;
constexpr int NT = 256;

// ---- shared memory map (bytes from a 1024-aligned base) ----
constexpr uint32_t S_TQ = 0;        // bf16 q tile     [64 t][128 i]  (TMA)
constexpr uint32_t S_TK = 16384;    // bf16 k tile
constexpr uint32_t S_TA = 32768;    // bf16 alpha tile
constexpr uint32_t S_TV = 49152;    // bf16 v tile     [64 s][128 j]  (MN-major A of U~)
constexpr uint32_t S_KH = 65536;    // fp16 K^ = (k*rho)^T  [128 i][64 s]  B of H-MMA
constexpr uint32_t S_WM = 81920;    // fp16 -W          [64 t][128 i]  B of U-MMA
constexpr uint32_t S_AQ = 98304;    // fp16 A           [64 t][64 s]   B of O-MMA
constexpr uint32_t S_TB = 106496;   // bf16 T Diag(beta)[64 t][64 s]   B of W/U~
constexpr uint32_t S_GB = 114688;   // 48 KiB scratch, reused within a chunk:
constexpr uint32_t S_GX = S_GB;            //   Gram X  fp16 [128 rows][128 i]
constexpr uint32_t S_GY = S_GB + 32768;    //   Gram Y  fp16 [64 rows][128 i]
constexpr uint32_t S_TF = S_GB;            //   T       fp32 [64][64]
constexpr uint32_t S_KGT = S_GB + 16384;   //   (k*gamma)^T bf16 [128 i][64 s]  A of W-MMA
constexpr uint32_t S_QG = S_GB + 32768;    //   q*gamma fp16 [64 t][128 i]  B of O-MMA
constexpr uint32_t S_RT = S_GB + 32768;    //   T-inverse temporaries (before q*gamma)
constexpr uint32_t S_HT = 163840;   // fp16 H^T         [128 j][128 i]  A of U/O
constexpr uint32_t S_UT = 196608;   // fp16 U^T         [128 j][64 s]   A of O/H
constexpr uint32_t S_MF = S_UT;     //   M fp32 [64][64] while the Grams are assembled
constexpr uint32_t S_SMALL = 212992;
constexpr uint32_t S_BETA = S_SMALL;          // fp32 [64]
constexpr uint32_t S_GC = S_SMALL + 256;      // fp32 [128] gamma_C
constexpr uint32_t S_BAR = S_SMALL + 768;     // mbarriers
constexpr uint32_t S_MISC = S_SMALL + 832;    // tmem base, abort flag
constexpr uint32_t SMEM_USED = S_SMALL + 1024;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;  // + alignment slack

// ---- tensor memory columns ----
constexpr uint32_t T_H = 0;     // H^T fp32 [128 j][128 i]
constexpr uint32_t T_U = 128;   // U^T fp32 [128 j][64 t]
constexpr uint32_t T_O = 192;   // O^T fp32 [128 j][64 t]
constexpr uint32_t T_G = 256;   // 3 Gram tiles [128 x][64 y]
constexpr uint32_t T_W = 448;   // W^T fp32 [128 i][64 t]
constexpr uint32_t TMEM_COLS = 512;

constexpr uint32_t TILE_BYTES = 16384;

__device__ __forceinline__ float bf16_at(const uint8_t* tile, int r, int c) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + sw128_off(64, r, c)));
}
__device__ __forceinline__ float2 bf16x2_at(const uint8_t* tile, int r, int c) {
  __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(tile + sw128_off(64, r, c));
  return __bfloat1622float2(v);
}
__device__ __forceinline__ bool fp16_ok(float x) { return fabsf(x) <= 65504.f; }

// Builds the Gram operands of one round: levels La (X rows 0..63, Y rows
// 0..31) and La/2 (X rows 64..127, Y rows 32..63).  X rows per level: 32
// k-rows then 32 q-rows of the upper-half tokens; Y rows: the lower-half tokens.
__device__ void build_gram_operands(uint8_t* sm, int La, int lenc) {
  const int tid = threadIdx.x, cp = tid & 63, grp = tid >> 6;
  const int c0 = 2 * cp;
  const uint8_t* tq = sm + S_TQ;
  const uint8_t* tk = sm + S_TK;
  const uint8_t* ta = sm + S_TA;
  const int L = (grp & 1) ? La / 2 : La;
  if (grp < 2) {
    uint8_t* X = sm + S_GX;
    const int xbase = (grp & 1) ? 64 : 0;
    for (int sg = 0; sg < 32 / L; ++sg) {
      float f0 = 1.f, f1 = 1.f;
      for (int w = 0; w < L; ++w) {
        const int t = sg * 2 * L + L + w;
        float2 a = t < lenc ? bf16x2_at(ta, t, c0) : make_float2(1.f, 1.f);
        f0 *= a.x;
        f1 *= a.y;
        const float2 kk = bf16x2_at(tk, t, c0);
        const float2 qq = bf16x2_at(tq, t, c0);
        const int rk = xbase + sg * L + w;
        *reinterpret_cast<uint32_t*>(X + sw128_off(128, rk, c0)) = pack_half2(kk.x * f0, kk.y * f1);
        *reinterpret_cast<uint32_t*>(X + sw128_off(128, rk + 32, c0)) =
            pack_half2(qq.x * f0, qq.y * f1);
      }
    }
  } else {
    uint8_t* Y = sm + S_GY;
    const int ybase = (grp & 1) ? 32 : 0;
    for (int sg = 0; sg < 32 / L; ++sg) {
      float b0 = 1.f, b1 = 1.f;
      for (int w = L - 1; w >= 0; --w) {
        const int s = sg * 2 * L + w;
        const float2 kk = bf16x2_at(tk, s, c0);
        *reinterpret_cast<uint32_t*>(Y + sw128_off(64, ybase + sg * L + w, c0)) =
            pack_half2(kk.x * b0, kk.y * b1);
        float2 a = s < lenc ? bf16x2_at(ta, s, c0) : make_float2(1.f, 1.f);
        b0 *= a.x;
        b1 *= a.y;
      }
    }
  }
}

// Reads Gram round r out of TMEM into M (fp32, scaled by beta_t) and A (fp16).
__device__ void extract_gram(uint8_t* sm, uint32_t tmem, int r) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int x = 32 * (warp & 3) + lane;  // X row = TMEM lane
  const int half = warp >> 2;
  const int La = 32 >> (2 * r);
  const bool lvb = x >= 64;
  const int L = lvb ? La / 2 : La;
  const int xr = x & 63;
  const bool qrow = xr >= 32;
  const int jx = xr & 31;
  const int t = (jx / L) * 2 * L + L + (jx % L);
  const uint32_t col0 = T_G + 64 * r + (lvb ? 32 : 0) + 16 * half;
  uint32_t v[16];
  tmem_ld32<16>(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + col0, v);
  tmem_ld_wait();
  const float* beta = reinterpret_cast<const float*>(sm + S_BETA);
  float* Mf = reinterpret_cast<float*>(sm + S_MF);
  uint8_t* AQ = sm + S_AQ;
#pragma unroll
  for (int cc = 0; cc < 16; ++cc) {
    const int jy = 16 * half + cc;
    if (jy / L != jx / L) continue;
    const int s = (jy / L) * 2 * L + (jy % L);
    const float g = __uint_as_float(v[cc]);
    if (qrow)
      *reinterpret_cast<__half*>(AQ + sw128_off(64, t, s)) = __float2half_rn(g);
    else
      Mf[t * 64 + s] = beta[t] * g;
  }
}

// T = (I + M)^-1 for the strictly lower M (fp32), by 16 x 16 blocks:
// diagonal blocks by forward substitution, then block rows by distance.
__device__ void invert_unit_lower(uint8_t* sm) {
  const int tid = threadIdx.x;
  const float* Mf = reinterpret_cast<const float*>(sm + S_MF);
  float* Tf = reinterpret_cast<float*>(sm + S_TF);
  float* R = reinterpret_cast<float*>(sm + S_RT);
  if (tid < 64) {
    const int blk = tid >> 4, c = tid & 15, o = 16 * blk;
    float x[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      float acc = (t == c) ? 1.f : 0.f;
#pragma unroll
      for (int s = 0; s < t; ++s) acc = fmaf(-Mf[(o + t) * 64 + o + s], x[s], acc);
      x[t] = acc;
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) Tf[(o + t) * 64 + o + c] = x[t];
  }
  __syncthreads();
  for (int d = 1; d < 4; ++d) {
    const int nb = 4 - d;
    for (int e = tid; e < nb * 256; e += NT) {
      const int J = e >> 8, I = J + d, a = (e >> 4) & 15, b = e & 15;
      float acc = 0.f;
      for (int K = J; K < I; ++K)
#pragma unroll
        for (int m = 0; m < 16; ++m)
          acc = fmaf(Mf[(16 * I + a) * 64 + 16 * K + m], Tf[(16 * K + m) * 64 + 16 * J + b], acc);
      R[e] = acc;
    }
    __syncthreads();
    for (int e = tid; e < nb * 256; e += NT) {
      const int J = e >> 8, I = J + d, a = (e >> 4) & 15, b = e & 15;
      float acc = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m)
        acc = fmaf(Tf[(16 * I + a) * 64 + 16 * I + m], R[(J << 8) + (m << 4) + b], acc);
      Tf[(16 * I + a) * 64 + 16 * J + b] = -acc;
    }
    __syncthreads();
  }
}

struct Unit {
  long row0;
  int len;
  size_t sidx;  // offset of this unit's state in h0/hT (elements)
};

__device__ __forceinline__ Unit unit_of(const FwdArgs& a) {
  Unit u;
  const int b = blockIdx.x;
  const int h = b % a.H;
  int n = b / a.H;
  if (a.cu_seqlens) {
    if (a.order) n = a.order[n];
    const int t0 = a.cu_seqlens[n];
    u.len = a.cu_seqlens[n + 1] - t0;
    u.row0 = (long)h * a.T + t0;
  } else {
    u.len = a.T;
    u.row0 = ((long)n * a.H + h) * a.T;
  }
  u.sidx = ((size_t)n * a.H + h) * 128 * 128;
  return u;
}

__global__ void __launch_bounds__(NT, 1)
    fwd_chunk_kernel(const __grid_constant__ FwdArgs a, const __grid_constant__ CUtensorMap mq,
                     const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap ma,
                     const __grid_constant__ CUtensorMap mv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wq = warp & 3, half = warp >> 2;
  const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
  uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + S_BAR);
  uint64_t* bar_mma = bar_tma + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S_MISC);
  float* beta_s = reinterpret_cast<float*>(sm + S_BETA);
  float* gC = reinterpret_cast<float*>(sm + S_GC);

  const Unit u = unit_of(a);
  const int nchunks = (u.len + C - 1) / C;

  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
    tma_prefetch_desc(&mq);
    tma_prefetch_desc(&mk);
    tma_prefetch_desc(&ma);
    tma_prefetch_desc(&mv);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto issue_tiles = [&](int c, bool qka, bool v) {
    const int y = (int)(u.row0 + (long)c * C);
    if (qka) {
      mbar_arrive_expect_tx(bar_tma, 4 * TILE_BYTES);
      tma_load_2d(sm + S_TQ, &mq, bar_tma, 0, y);
      tma_load_2d(sm + S_TQ + 8192, &mq, bar_tma, 64, y);
      tma_load_2d(sm + S_TK, &mk, bar_tma, 0, y);
      tma_load_2d(sm + S_TK + 8192, &mk, bar_tma, 64, y);
      tma_load_2d(sm + S_TA, &ma, bar_tma, 0, y);
      tma_load_2d(sm + S_TA + 8192, &ma, bar_tma, 64, y);
    }
    if (v) {
      tma_load_2d(sm + S_TV, &mv, bar_tma, 0, y);
      tma_load_2d(sm + S_TV + 8192, &mv, bar_tma, 64, y);
    }
  };
  if (tid == 0 && nchunks > 0) issue_tiles(0, true, true);

  // Initial state: H^T[j][i] = h0[i][j] (or 0) into TMEM and as fp16 into smem.
  {
    const int j = 32 * wq + lane;
    uint8_t* HT = sm + S_HT;
    for (int c16 = 0; c16 < 4; ++c16) {
      const int i0 = 64 * half + 16 * c16;
      uint32_t r[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        r[e] = __float_as_uint(a.h0 ? a.h0[u.sidx + (size_t)(i0 + e) * 128 + j] : 0.f);
      tmem_st32<16>(tmem + lane_base + T_H + i0, r);
#pragma unroll
      for (int e = 0; e < 16; e += 8) {
        uint4 pk;
        pk.x = pack_half2(__uint_as_float(r[e]), __uint_as_float(r[e + 1]));
        pk.y = pack_half2(__uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
        pk.z = pack_half2(__uint_as_float(r[e + 4]), __uint_as_float(r[e + 5]));
        pk.w = pack_half2(__uint_as_float(r[e + 6]), __uint_as_float(r[e + 7]));
        *reinterpret_cast<uint4*>(HT + sw128_chunk(128, j, (i0 + e) >> 3)) = pk;
      }
    }
    tmem_st_wait();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  uint32_t mma_phase = 0;
  bool ovf = false;
  bool tma_pending = nchunks > 0;
  int tma_next = 0;  // chunk whose tiles were issued last
  bool aborted = false;  // uniform across the block: decided by __syncthreads_or
  auto wait_mma = [&]() -> bool {
    const bool ok = mbar_wait(bar_mma, mma_phase);
    mma_phase ^= 1;
    if (!ok) set_status(a.status, CKDA_ERR_TIMEOUT);
    tc_fence_after();
    aborted = __syncthreads_or(ok ? 0 : 1) != 0;
    return !aborted;
  };
  auto sync_for_mma = [&]() {
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };

  const uint32_t sb = smem_u32(sm);
  const uint32_t idx_f16_n64 = idesc_f16(128, 64, 0, 0, 0);
  const uint32_t idx_f16_n128 = idesc_f16(128, 128, 0, 0, 0);
  const uint32_t idx_bf16_n64 = idesc_f16(128, 64, 1, 0, 0);
  const uint32_t idx_bf16_mn_n64 = idesc_f16(128, 64, 1, 1, 0);

  for (int c = 0; c < nchunks; ++c) {
    const int lenc = min(C, u.len - c * C);
    // ---------------------------------------------------------- tiles of c
    {
      const bool ok = mbar_wait(bar_tma, (uint32_t)(c & 1));
      if (!ok) set_status(a.status, CKDA_ERR_TIMEOUT);
      aborted = __syncthreads_or(ok ? 0 : 1) != 0;
      if (aborted) break;
      tma_pending = false;
    }
    if (tid < C) {
      const long r = u.row0 + (long)c * C + tid;
      beta_s[tid] = tid < lenc ? ld_io(static_cast<const __nv_bfloat16*>(a.beta) + r) : 0.f;
    }
    {  // zero M (fp32) and A (fp16) for this chunk
      float4* mz = reinterpret_cast<float4*>(sm + S_MF);
      for (int e = tid; e < 64 * 64 / 4; e += NT) mz[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      uint4* az = reinterpret_cast<uint4*>(sm + S_AQ);
      for (int e = tid; e < 8192 / 16; e += NT) az[e] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    // ------------------------------------------------- gated Grams (3 rounds)
    bool alive = true;
    for (int r = 0; r < 3 && alive; ++r) {
      build_gram_operands(sm, 32 >> (2 * r), lenc);
      sync_for_mma();
      if (tid == 0) {
        for (int k = 0; k < 8; ++k)
          umma_ss(tmem + T_G + 64 * r, kmajor_desc(sb + S_GX, 128, k),
                  kmajor_desc(sb + S_GY, 64, k), idx_f16_n64, k > 0);
        umma_commit(bar_mma);
      }
      alive = wait_mma();
    }
    if (!alive) break;
    for (int r = 0; r < 3; ++r) extract_gram(sm, tmem, r);
    {  // diagonal of A: q_t . k_t
      const int t = tid >> 2, part = tid & 3;
      float acc = 0.f;
      for (int i = 32 * part; i < 32 * part + 32; i += 2) {
        const float2 qq = bf16x2_at(sm + S_TQ, t, i), kk = bf16x2_at(sm + S_TK, t, i);
        acc = fmaf(qq.x, kk.x, fmaf(qq.y, kk.y, acc));
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      if (part == 0) *reinterpret_cast<__half*>(sm + S_AQ + sw128_off(64, t, t)) = __float2half_rn(acc);
    }
    __syncthreads();
    // ------------------------------------------------------- T and T Diag(beta)
    invert_unit_lower(sm);
    {
      const float* Tf = reinterpret_cast<const float*>(sm + S_TF);
      for (int e = tid; e < 64 * 32; e += NT) {
        const int t = e >> 5, s = 2 * (e & 31);
        const float v0 = s <= t ? Tf[t * 64 + s] * beta_s[s] : 0.f;
        const float v1 = s + 1 <= t ? Tf[t * 64 + s + 1] * beta_s[s + 1] : 0.f;
        *reinterpret_cast<uint32_t*>(sm + S_TB + sw128_off(64, t, s)) = pack_bf162(v0, v1);
      }
    }
    __syncthreads();
    // --------------------------- (k*gamma)^T, q*gamma, (k*rho)^T and gamma_C
    if (tid < 128) {
      const int i = tid;
      float g = 1.f;
      uint32_t pk[4];
      for (int s = 0; s < C; ++s) {
        const float al = s < lenc ? bf16_at(sm + S_TA, s, i) : 1.f;
        g *= al;
        const float kg = bf16_at(sm + S_TK, s, i) * g;
        const float qg = bf16_at(sm + S_TQ, s, i) * g;
        if (s < lenc) ovf |= !fp16_ok(qg);
        *reinterpret_cast<__half*>(sm + S_QG + sw128_off(64, s, i)) = __float2half_rn(qg);
        const int e = s & 7;
        if (e & 1) {
          const float prev = __uint_as_float(pk[e >> 1]);
          pk[e >> 1] = pack_bf162(prev, kg);
        } else {
          pk[e >> 1] = __float_as_uint(kg);
        }
        if (e == 7)
          *reinterpret_cast<uint4*>(sm + S_KGT + sw128_chunk(128, i, s >> 3)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      gC[i] = g;
    } else {
      const int i = tid - 128;
      float rho = 1.f;
      float vals[8];
      for (int s = C - 1; s >= 0; --s) {
        vals[s & 7] = bf16_at(sm + S_TK, s, i) * rho;
        const float al = s < lenc ? bf16_at(sm + S_TA, s, i) : 1.f;
        rho *= al;
        if ((s & 7) == 0) {
          uint4 pk;
          pk.x = pack_half2(vals[0], vals[1]);
          pk.y = pack_half2(vals[2], vals[3]);
          pk.z = pack_half2(vals[4], vals[5]);
          pk.w = pack_half2(vals[6], vals[7]);
          *reinterpret_cast<uint4*>(sm + S_KH + sw128_chunk(128, i, s >> 3)) = pk;
        }
      }
    }
    sync_for_mma();
    // ------------------------------------------------------------ W = TB (k*gamma)
    if (tid == 0) {
      for (int k = 0; k < 4; ++k)
        umma_ss(tmem + T_W, kmajor_desc(sb + S_KGT, 128, k), kmajor_desc(sb + S_TB, 64, k),
                idx_bf16_n64, k > 0);
      umma_commit(bar_mma);
      // q, k, alpha of this chunk are no longer read: prefetch the next chunk's
      if (c + 1 < nchunks) issue_tiles(c + 1, true, false);
    }
    if (!wait_mma()) break;
    {  // -W as fp16 [t][i]: lane = i, columns = t
      const int i = 32 * wq + lane;
      uint32_t v[32];
      tmem_ld32<32>(tmem + lane_base + T_W + 32 * half, v);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e)
        *reinterpret_cast<__half*>(sm + S_WM + sw128_off(64, 32 * half + e, i)) =
            __float2half_rn(-__uint_as_float(v[e]));
    }
    {  // H^T <- H^T Diag(gamma_C) in TMEM (column i scaled by gamma_C[i])
      for (int c16 = 0; c16 < 4; ++c16) {
        const int i0 = 64 * half + 16 * c16;
        uint32_t v[16];
        tmem_ld32<16>(tmem + lane_base + T_H + i0, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * gC[i0 + e]);
        tmem_st32<16>(tmem + lane_base + T_H + i0, v);
      }
      tmem_st_wait();
    }
    sync_for_mma();
    // ------------------------------- U = TB V - W H ;  O = (q*gamma) H
    if (tid == 0) {
      for (int k = 0; k < 4; ++k)
        umma_ss(tmem + T_U, mnmajor_desc(sb + S_TV, 64, k), kmajor_desc(sb + S_TB, 64, k),
                idx_bf16_mn_n64, k > 0);
      for (int k = 0; k < 8; ++k)
        umma_ss(tmem + T_U, kmajor_desc(sb + S_HT, 128, k), kmajor_desc(sb + S_WM, 64, k),
                idx_f16_n64, 1);
      for (int k = 0; k < 8; ++k)
        umma_ss(tmem + T_O, kmajor_desc(sb + S_HT, 128, k), kmajor_desc(sb + S_QG, 64, k),
                idx_f16_n64, k > 0);
      umma_commit(bar_mma);
    }
    if (!wait_mma()) break;
    if (c + 1 < nchunks) {
      if (tid == 0) issue_tiles(c + 1, false, true);
      tma_pending = true;
      tma_next = c + 1;
    }
    {  // U^T -> fp16 [j][s]
      const int j = 32 * wq + lane;
      uint32_t v[32];
      tmem_ld32<32>(tmem + lane_base + T_U + 32 * half, v);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        uint4 pk;
        float f[8];
#pragma unroll
        for (int z = 0; z < 8; ++z) {
          f[z] = __uint_as_float(v[e + z]);
          ovf |= !fp16_ok(f[z]);
        }
        pk.x = pack_half2(f[0], f[1]);
        pk.y = pack_half2(f[2], f[3]);
        pk.z = pack_half2(f[4], f[5]);
        pk.w = pack_half2(f[6], f[7]);
        *reinterpret_cast<uint4*>(sm + S_UT + sw128_chunk(128, j, (32 * half + e) >> 3)) = pk;
      }
    }
    sync_for_mma();
    // ------------------------------ O += A U ;  H^T += U^T (k*rho)
    if (tid == 0) {
      for (int k = 0; k < 4; ++k)
        umma_ss(tmem + T_O, kmajor_desc(sb + S_UT, 128, k), kmajor_desc(sb + S_AQ, 64, k),
                idx_f16_n64, 1);
      for (int k = 0; k < 4; ++k)
        umma_ss(tmem + T_H, kmajor_desc(sb + S_UT, 128, k), kmajor_desc(sb + S_KH, 128, k),
                idx_f16_n128, 1);
      umma_commit(bar_mma);
    }
    if (!wait_mma()) break;
    {  // outputs of this chunk: o[t][j] for t < lenc
      const int j = 32 * wq + lane;
      uint32_t v[32];
      tmem_ld32<32>(tmem + lane_base + T_O + 32 * half, v);
      tmem_ld_wait();
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.o);
      const long rbase = u.row0 + (long)c * C;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int t = 32 * half + e;
        if (t < lenc) o[(size_t)(rbase + t) * 128 + j] = __float2bfloat16_rn(a.scale * __uint_as_float(v[e]));
      }
    }
    if (c + 1 < nchunks) {  // H^T -> fp16 [j][i] for the next chunk
      const int j = 32 * wq + lane;
      for (int c32 = 0; c32 < 2; ++c32) {
        const int i0 = 64 * half + 32 * c32;
        uint32_t v[32];
        tmem_ld32<32>(tmem + lane_base + T_H + i0, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          float f[8];
#pragma unroll
          for (int z = 0; z < 8; ++z) {
            f[z] = __uint_as_float(v[e + z]);
            ovf |= !fp16_ok(f[z]);
          }
          uint4 pk;
          pk.x = pack_half2(f[0], f[1]);
          pk.y = pack_half2(f[2], f[3]);
          pk.z = pack_half2(f[4], f[5]);
          pk.w = pack_half2(f[6], f[7]);
          *reinterpret_cast<uint4*>(sm + S_HT + sw128_chunk(128, j, (i0 + e) >> 3)) = pk;
        }
      }
    }
    sync_for_mma();
  }

  // ------------------------------------------------------------ final state
  if (!aborted && a.hT) {
    const int j = 32 * wq + lane;
    for (int c32 = 0; c32 < 2; ++c32) {
      const int i0 = 64 * half + 32 * c32;
      uint32_t v[32];
      tmem_ld32<32>(tmem + lane_base + T_H + i0, v);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) a.hT[u.sidx + (size_t)(i0 + e) * 128 + j] = __uint_as_float(v[e]);
    }
  }
  if (__syncthreads_or(ovf ? 1 : 0) && tid == 0) set_status(a.status, CKDA_ERR_RANGE);
  if (tid == 0 && tma_pending && aborted) {
    // a load of the next chunk may still be landing in shared memory
    mbar_wait(bar_tma, (uint32_t)(tma_next & 1));
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, uint64_t rows) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t gdim[2] = {128, rows};
  cuuint64_t gstride[1] = {128 * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_fwd_chunk(const FwdArgs& a, cudaStream_t s) {
  const int units = a.num_units_seq * a.H;
  if (units == 0) return cudaSuccess;
  const uint64_t rows = (uint64_t)a.B * a.H * a.T;
  CUtensorMap mq, mk, ma, mv;
  if (rows == 0) {
    // every sequence is empty: the kernel only copies h0 to hT, no tile is loaded
    mq = mk = ma = mv = CUtensorMap{};
  } else if (!make_map(&mq, a.q, rows) || !make_map(&mk, a.k, rows) ||
             !make_map(&ma, a.alpha, rows) || !make_map(&mv, a.v, rows)) {
    return cudaErrorInvalidValue;
  }
  // per device and cheap: set on every launch
  cudaError_t attr_err = cudaFuncSetAttribute(
      fwd_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
  if (attr_err != cudaSuccess) return attr_err;
  fwd_chunk_kernel<<<units, NT, SMEM_ALLOC, s>>>(a, mq, mk, ma, mv);
  return cudaGetLastError();
}

}  // namespace ckda
