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
// alpha_r]: a prefix product within an aligned block of L tokens times an
// exclusive suffix product within one.  Every level is one dense contraction
// of gated operands on the tensor cores; two levels share a 128 x 64 MMA tile.
//
// Precision: operands of every contraction that touches the state, the
// Grams and A are fp16 (11-bit significand); T Diag(beta), k * gamma and the
// raw bf16 inputs are bf16; all accumulation is fp32 in TMEM, gate products
// and T are fp32.  An fp16 overflow is reported as CKDA_ERR_RANGE.
//
// Warp roles (384 threads):
//   warps 0-7  PREP: per chunk, gate products, gated Grams, T, W and the
//              operands of the state step; thread (j, tq) owns channels
//              8j..8j+7 of tokens 4tq..4tq+3.  Prep of chunk c+1 runs while
//              the state warps step chunk c.
//   warps 8-11 STATE: the serial state step on TMEM (thread = TMEM lane = j).
// Handoffs use release/acquire counters in shared memory; MMA and TMA
// completion use mbarriers.  Every wait is bounded.
#include "ckda_internal.cuh"
#include "sm103.cuh"

#include <cudaTypedefs.h>
#include <mutex>

namespace ckda {
namespace {

constexpr int C = 64;
constexpr int NPREP = 256;
constexpr int NSTATE = 128;
constexpr int NT = NPREP + NSTATE;
constexpr int BAR_PREP = 1;   // named barrier ids
constexpr int BAR_STATE = 2;

// ---- shared memory map (bytes from a 1024-aligned base) ----
// q, k, alpha tiles; once read they hold the second Gram operand buffer
// (X over q and k, Y over alpha) until the last Gram MMA, then the next
// chunk's tiles are fetched into them
constexpr uint32_t S_TQ = 0;         // bf16 q tile   [64 t][128 i]  (TMA)
constexpr uint32_t S_TK = 16384;     // bf16 k tile
constexpr uint32_t S_TA = 32768;     // bf16 alpha tile
constexpr uint32_t S_V = 49152;      // bf16 v tile   [64 s][128 j]  MN-major A of U~   (TMA)
constexpr uint32_t S_TB = 65536;     // bf16 T Diag(beta) [64 t][64 s] K-major B of U~, W
constexpr uint32_t S_W = 73728;      // fp16 -W^T     [128 i][64 t]  MN-major B of U
constexpr uint32_t S_QG = 90112;     // fp16 q*gamma  [64 t][128 i]  K-major B of O
constexpr uint32_t S_KH = 106496;    // fp16 k*rho    [64 s][128 i]  MN-major B of H
constexpr uint32_t S_KGT = 122880;   // bf16 k*gamma  [64 s][128 i]  MN-major A of W
constexpr uint32_t S_AQ = 139264;    // fp16 A        [64 t][64 s]   K-major B of O
constexpr uint32_t S_GX = 147456;    // fp16 Gram X   [128 rows][128 i] K-major A
constexpr uint32_t S_GY = 180224;    // fp16 Gram Y   [64 rows][128 i]  K-major B
constexpr uint32_t S_GX2 = S_TQ;     // second Gram buffer (the tile region)
constexpr uint32_t S_GY2 = S_TA;
// after the Gram MMAs the 48 KiB of X and Y hold the inverse's 64 x 64 tiles
// (fp16, one 64-column panel each).  A tile read as a 128-row A operand also
// reads the 8 KiB after it; those rows only feed TMEM lanes that are ignored.
constexpr uint32_t S_TD = S_GX + 8192;       // D: inverses of the 16 x 16 diagonal blocks
constexpr uint32_t S_TE = S_GX + 16384;      // E = D N
constexpr uint32_t S_TG = S_GX + 24576;      // G = I + E^2
constexpr uint32_t S_TFm = S_GY;             // F = (I - E) G
// written by the Gram read-out while later Gram MMAs still read X and Y:
constexpr uint32_t S_TN = 196608;            // fp16 N: block-strictly-lower part of M
constexpr uint32_t S_MD = 204800;            // fp32 diagonal 16 x 16 blocks of M [4][16][20]
constexpr int kMdRow = 20, kMdBlk = 16 * kMdRow;  // padded rows spread the banks
constexpr uint32_t S_SMALL = 209920;
constexpr uint32_t S_BETA = S_SMALL;         // fp32 [2][64]
constexpr uint32_t S_GC = S_SMALL + 512;     // fp32 [2][128] gamma_C
constexpr uint32_t S_DIAG = S_SMALL + 1536;  // fp32 [16][64] partial q.k
constexpr uint32_t S_TOT = S_SMALL + 5632;   // fp32 [2][16][8] half-chunk gate totals
constexpr uint32_t S_BAR = S_SMALL + 6656;   // mbarriers
constexpr uint32_t SMEM_USED = S_SMALL + 6912;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
static_assert(SMEM_ALLOC <= 232448, "shared memory budget");

// ---- tensor memory columns ----
constexpr uint32_t T_H = 0;     // H^T fp32 [128 j][128 i]     state accumulator
constexpr uint32_t T_HA = 128;  // H^T fp16 [128 j][128 i]     A operand (2 per column)
constexpr uint32_t T_U = 192;   // U^T fp32 [128 j][64 t]
constexpr uint32_t T_UA = 256;  // U^T fp16 [128 j][64 t]      A operand
constexpr uint32_t T_O = 288;   // O^T fp32 [128 j][64 t]
constexpr uint32_t T_G0 = 352;  // Gram rounds use G0, G1, G0; the inverse chain uses
constexpr uint32_t T_G1 = 416;  //   E:G1, E^2:G0, EG:G1, T:G0; then W^T:G1 (read by the state)
constexpr uint32_t TMEM_COLS = 512;

constexpr uint32_t TILE_BYTES = 16384;

struct Unit {
  long row0;
  int len;
  size_t sidx;
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

__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ uint4 pack_half8(const float (&f)[8]) {
  return make_uint4(pack_half2(f[0], f[1]), pack_half2(f[2], f[3]), pack_half2(f[4], f[5]),
                    pack_half2(f[6], f[7]));
}
__device__ __forceinline__ uint4 pack_bf8(const float (&f)[8]) {
  return make_uint4(pack_bf162(f[0], f[1]), pack_bf162(f[2], f[3]), pack_bf162(f[4], f[5]),
                    pack_bf162(f[6], f[7]));
}
// bf16 x 8 -> fp16 x 8 (through fp32; exact in the fp16 normal range)
__device__ __forceinline__ uint4 bf16x8_to_half8(const uint4& v) {
  float f[8];
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
  return make_uint4(pack_half2(f[0], f[1]), pack_half2(f[2], f[3]), pack_half2(f[4], f[5]),
                    pack_half2(f[6], f[7]));
}
// x (fp16 x 8) times the gate factors f (fp32 x 8, rounded to fp16) -> fp16 x 8
__device__ __forceinline__ uint4 hmul8(const uint4& x, const float (&f)[8]) {
  const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
  uint32_t r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 a = *reinterpret_cast<const __half2*>(&xs[i]);
    const __half2 b = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
    const __half2 p = __hmul2(a, b);
    r[i] = *reinterpret_cast<const uint32_t*>(&p);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}
// elementwise product of two fp16 x 8 vectors
__device__ __forceinline__ uint4 hmul8h(const uint4& x, const uint4& y) {
  uint4 r;
  const __half2 p0 = __hmul2(*reinterpret_cast<const __half2*>(&x.x), *reinterpret_cast<const __half2*>(&y.x));
  const __half2 p1 = __hmul2(*reinterpret_cast<const __half2*>(&x.y), *reinterpret_cast<const __half2*>(&y.y));
  const __half2 p2 = __hmul2(*reinterpret_cast<const __half2*>(&x.z), *reinterpret_cast<const __half2*>(&y.z));
  const __half2 p3 = __hmul2(*reinterpret_cast<const __half2*>(&x.w), *reinterpret_cast<const __half2*>(&y.w));
  r.x = *reinterpret_cast<const uint32_t*>(&p0);
  r.y = *reinterpret_cast<const uint32_t*>(&p1);
  r.z = *reinterpret_cast<const uint32_t*>(&p2);
  r.w = *reinterpret_cast<const uint32_t*>(&p3);
  return r;
}
__device__ __forceinline__ uint4 to_half8(const float (&f)[8]) {
  return make_uint4(pack_half2(f[0], f[1]), pack_half2(f[2], f[3]), pack_half2(f[4], f[5]),
                    pack_half2(f[6], f[7]));
}
// fp16 x 8 -> bf16 x 8
__device__ __forceinline__ uint4 half8_to_bf8(const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    r[i] = pack_bf162(t.x, t.y);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}
__device__ __forceinline__ float absmax8(const float (&f)[8]) {
  float m = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(f[e]));
  return m;
}
__device__ __forceinline__ void unpack_half8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
// true iff no lane of an fp16 x 8 vector is inf or NaN
__device__ __forceinline__ bool half8_finite(const uint4& v) {
  const uint32_t m = 0x7c007c00u;
  return ((v.x & m) != m) && ((v.y & m) != m) && ((v.z & m) != m) && ((v.w & m) != m) &&
         (((v.x >> 10) & 0x1f) != 0x1f) && (((v.x >> 26) & 0x1f) != 0x1f) &&
         (((v.y >> 10) & 0x1f) != 0x1f) && (((v.y >> 26) & 0x1f) != 0x1f) &&
         (((v.z >> 10) & 0x1f) != 0x1f) && (((v.z >> 26) & 0x1f) != 0x1f) &&
         (((v.w >> 10) & 0x1f) != 0x1f) && (((v.w >> 26) & 0x1f) != 0x1f);
}
__device__ __forceinline__ bool fp16_ok8(const float (&f)[8]) {
  float m = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(f[e]));
  return m <= 65504.f;  // false for NaN too
}

// Per-thread state of one prep chunk: tokens t = 4 tq + u, channels 8 j + e.
// Gate factors are kept as packed fp16 pairs (4 words = 8 channels): they
// only ever multiply fp16 operands.  gamma_C, which scales the fp32 state,
// is formed in fp32 separately.
struct Prep {
  uint4 k[4], q[4];      // k, q rows as fp16 (8 channels; exact for |x| >= 2^-14)
  uint4 lp[4], ls[4];    // in-quad inclusive prefix / exclusive suffix products
  uint4 a1, a2, a3;      // alpha of quad tokens 1, 2, 3 (levels 1 and 2)
  uint4 F8, F16, F32;    // per level: in-group prefix (upper) or suffix (lower)
  uint4 E16, X16;        // whole-chunk exclusive prefix / suffix of quad totals
  int tq;

  // Gate factor of token u of this quad at tree level L: the product of
  // alpha over (m, t] for an upper-half token, over (s, m] for a lower one.
  template <int L>
  __device__ __forceinline__ uint4 factor(int u) const {
    const int t = 4 * tq + u;
    const bool upper = (t % (2 * L)) >= L;
    const uint4 one = make_uint4(0x3c003c00u, 0x3c003c00u, 0x3c003c00u, 0x3c003c00u);
    if (L == 1) return upper ? (u == 1 ? a1 : a3) : one;
    if (L == 2) {
      if (upper) return u == 2 ? a2 : ls[1];  // a2, a2 a3
      return u == 0 ? a1 : one;
    }
    if (L == 4) return upper ? lp[u] : ls[u];
    const uint4& F = L == 8 ? F8 : (L == 16 ? F16 : F32);
    return hmul8h(F, upper ? lp[u] : ls[u]);
  }
  __device__ __forceinline__ uint4 gamma(int u) const { return hmul8h(E16, lp[u]); }
  __device__ __forceinline__ uint4 rho(int u) const { return hmul8h(ls[u], X16); }
};

// Segmented exclusive prefix / suffix products of quad totals within aligned
// groups of 2, 4, 8, 16 quads, over the 16 quads of a chunk (lanes tq of a
// 16-wide shuffle segment).  Level L = 8, 16, 32 needs the prefix if this
// quad is in the upper half of its 2L segment and the suffix otherwise.
// Quads tq_lo = 0..7 of one half of the chunk sit on the 8 lanes of a
// shuffle segment; the two halves are in different warps and meet through
// shared memory (`tot`, after a barrier of the prep role).
__device__ __forceinline__ void quad_scans(Prep& P, const float (&Bq)[8], float (&E16f)[8],
                                           float* tot, int j) {
  const int tq = P.tq, tq_lo = tq & 7, tq_hi = tq >> 3;
  float I[8], J[8], E[8], X[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    I[e] = Bq[e];
    J[e] = Bq[e];
    E[e] = 1.f;
    X[e] = 1.f;
  }
#pragma unroll
  for (int lg = 0; lg < 3; ++lg) {
    const int g = 1 << lg;
    const int base = tq_lo & ~(2 * g - 1);
    const int srcE = base + g - 1;  // last quad of the first half
    const int srcX = base + g;      // first quad of the second half
    const bool second = (tq_lo & g) != 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float vi = __shfl_sync(0xffffffffu, I[e], srcE, 8);
      const float vj = __shfl_sync(0xffffffffu, J[e], srcX, 8);
      if (second) E[e] *= vi; else X[e] *= vj;
      I[e] = E[e] * Bq[e];
      J[e] = X[e] * Bq[e];
    }
    // groups of 2g quads = blocks of 8g tokens serve tree level L = 8g
    const bool upper = (tq & (2 * g)) != 0;
    float sel[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) sel[e] = upper ? E[e] : X[e];
    if (lg == 0) P.F8 = to_half8(sel);
    if (lg == 1) P.F16 = to_half8(sel);
    if (lg == 2) P.F32 = to_half8(sel);
  }
  // whole chunk: the other half's total comes from the other warp
  if (tq_lo == 7) {
#pragma unroll
    for (int e = 0; e < 8; ++e) tot[(tq_hi * 16 + j) * 8 + e] = I[e];
  }
  named_sync(1, 256);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    if (tq_hi) E[e] *= tot[j * 8 + e];           // first half's total
    else X[e] *= tot[(16 + j) * 8 + e];          // second half's total
  }
  P.E16 = to_half8(E);
  P.X16 = to_half8(X);
#pragma unroll
  for (int e = 0; e < 8; ++e) E16f[e] = E[e];
}

// Row of token t in level L's operands: upper tokens -> X rank, lower -> Y rank.
__device__ __forceinline__ int level_rank(int t, int L) {
  const int seg = t / (2 * L), w = t % (2 * L);
  return seg * L + (w >= L ? w - L : w);
}

__device__ __forceinline__ void store16(uint8_t* p, const uint4& v) {
  *reinterpret_cast<uint4*>(p) = v;
}

// Builds the Gram operands of one round: levels La (X rows 0..63, Y rows
// 0..31) and La/2 (X rows 64..127, Y rows 32..63).  X rows of a level are
// 32 k-rows then 32 q-rows of its upper-half tokens; Y rows its lower-half
// tokens, each gated by the token's factor at that level.
template <int L>
__device__ __forceinline__ void write_level(uint8_t* X, uint8_t* Y, const Prep& P, int j,
                                            int xbase, int ybase) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int t = 4 * P.tq + u;
    const bool upper = (t % (2 * L)) >= L;
    const int rank = level_rank(t, L);
    const uint4 f = P.factor<L>(u);
    // |factor| <= 1, so the products stay within the range of k and q
    if (upper) {
      store16(X + sw128_chunk(128, xbase + rank, j), hmul8h(P.k[u], f));
      store16(X + sw128_chunk(128, xbase + 32 + rank, j), hmul8h(P.q[u], f));
    } else {
      store16(Y + sw128_chunk(64, ybase + rank, j), hmul8h(P.k[u], f));
    }
  }
}

// Reads one tree level out of TMEM (lanes = its X rows) into M (fp32,
// beta_t scaled) and A (fp16).  Lane x of a level: rows 0..31 are k-rows,
// 32..63 q-rows of upper rank x & 31; its valid columns are the L sources of
// its own segment, columns [sg*L, sg*L + L) of the level's 32.
template <int L>
__device__ __forceinline__ void extract_level(uint8_t* sm, uint32_t taddr, int xr,
                                              const float* beta, uint8_t* AQ) {
  const bool qrow = xr >= 32;
  const int jr = xr & 31;
  const int sg = jr / L;
  const int t = sg * 2 * L + L + (jr % L);
  const int s0 = sg * 2 * L;  // first source of the segment
  uint32_t v[32];
  tmem_ld32<32>(taddr, v);
  tmem_ld_wait();
  float g[L];
#pragma unroll
  for (int c = 0; c < L; ++c) g[c] = 0.f;
#pragma unroll
  for (int sgc = 0; sgc < 32 / L; ++sgc) {
    if (sgc == sg) {
#pragma unroll
      for (int c = 0; c < L; ++c) g[c] = __uint_as_float(v[sgc * L + c]);
    }
  }
  if (qrow) {
    if (L == 1) {
      *reinterpret_cast<__half*>(AQ + sw128_off(64, t, s0)) = __float2half_rn(g[0]);
    } else if (L < 8) {
#pragma unroll
      for (int c = 0; c < L; c += 2)
        *reinterpret_cast<uint32_t*>(AQ + sw128_off(64, t, s0 + c)) = pack_half2(g[c], g[c + 1]);
    } else {
#pragma unroll
      for (int c = 0; c < L; c += 8) {
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = g[c + e];
        store16(AQ + sw128_off(64, t, s0 + c), pack_half8(f));
      }
    }
  } else {
    const float bt = beta[t];
    if (L >= 16) {
      // pairs in different 16-token blocks: fp16 tile N[t][s]
#pragma unroll
      for (int c = 0; c < L; c += 8) {
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = bt * g[c + e];
        store16(sm + S_TN + sw128_off(64, t, s0 + c), pack_half8(f));
      }
    } else {
      // pairs inside one 16-token block: fp32 [block][t mod 16][s mod 16]
      float* Md = reinterpret_cast<float*>(sm + S_MD) + (t >> 4) * kMdBlk + (t & 15) * kMdRow;
      const int sl = s0 & 15;
      if (L >= 4) {
#pragma unroll
        for (int c = 0; c < L; c += 4)
          *reinterpret_cast<float4*>(Md + sl + c) =
              make_float4(bt * g[c], bt * g[c + 1], bt * g[c + 2], bt * g[c + 3]);
      } else {
#pragma unroll
        for (int c = 0; c < L; ++c) Md[sl + c] = bt * g[c];
      }
    }
  }
}

template <int La>
__device__ __forceinline__ void extract_round(uint8_t* sm, uint32_t tmem, uint32_t col, int wq,
                                              int lane, const float* beta, uint8_t* AQ) {
  const int x = 32 * wq + lane;  // warp-uniform level: lanes 0..63 level La, 64..127 La/2
  const uint32_t base = tmem + ((uint32_t)(32 * wq) << 16) + col;
  if (x < 64)
    extract_level<La>(sm, base, x & 63, beta, AQ);
  else
    extract_level<La / 2>(sm, base + 32, x & 63, beta, AQ);
}

// D (tmem) (+)= A (tmem) x B (smem), issued by a single thread.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Inverses of the four unit-lower 16 x 16 diagonal blocks of I + M, by
// right-looking substitution (one column per thread), written as fp16 into
// the diagonal blocks of D.  Threads 0..63.
__device__ __forceinline__ void invert_diag_blocks(uint8_t* sm, int p) {
  const int blk = p >> 4, c = p & 15, o = 16 * blk;
  const float* Md = reinterpret_cast<const float*>(sm + S_MD) + blk * kMdBlk;
  float x[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) x[t] = (t == c) ? 1.f : 0.f;
#pragma unroll
  for (int s = 0; s < 15; ++s) {
#pragma unroll
    for (int t = s + 1; t < 16; ++t) x[t] = fmaf(-Md[t * kMdRow + s], x[s], x[t]);
  }
#pragma unroll
  for (int t = 0; t < 16; ++t)
    *reinterpret_cast<__half*>(sm + S_TD + sw128_off(64, o + t, o + c)) = __float2half_rn(x[t]);
}

__global__ void __launch_bounds__(NT, 1)
    fwd_chunk_kernel(const __grid_constant__ FwdArgs a, const __grid_constant__ CUtensorMap mq,
                     const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap ma,
                     const __grid_constant__ CUtensorMap mv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* bar_v = reinterpret_cast<uint64_t*>(sm + S_BAR);
  uint64_t* bar_w = bar_v + 2;
  uint64_t* bar_s1 = bar_v + 3;
  uint64_t* bar_s3 = bar_v + 4;
  uint64_t* bar_t = bar_v + 5;
  uint64_t* bar_qka = bar_v + 6;
  // prep -> state handoffs, one barrier per chunk parity so that a waiter can
  // never fall a whole phase behind: operands of chunk c complete, gamma_C
  // of chunk c published.  The state -> prep direction uses bar_s1 (TB, W
  // free) and bar_s3 (q*gamma, k*rho, A free) directly.
  uint64_t* bar_ready = bar_v + 7;   // [2]
  uint64_t* bar_gc = bar_v + 9;      // [2]
  // one barrier per Gram round: rounds 1 and 2 are both in flight before
  // round 1 is waited for, so a shared barrier could run two phases ahead
  uint64_t* bar_r = bar_v + 11;      // [3]
  int* s_abort = reinterpret_cast<int*>(sm + S_BAR + 128);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S_BAR + 136);

  const Unit u = unit_of(a);
  const int nchunks = (u.len + C - 1) / C;

  if (tid == 0) {
    mbar_init(bar_v, 1);
    mbar_init(bar_w, 1);
    mbar_init(bar_s1, 1);
    mbar_init(bar_s3, 1);
    mbar_init(bar_t, 1);
    mbar_init(bar_qka, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_ready + i, 1);
      mbar_init(bar_gc + i, 1);
    }
    for (int i = 0; i < 3; ++i) mbar_init(bar_r + i, 1);
    *s_abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&mq);
    tma_prefetch_desc(&mk);
    tma_prefetch_desc(&ma);
    tma_prefetch_desc(&mv);
  }
  // A's upper triangle and N's blocks on and above the 16-block diagonal are
  // never written again, so zero both tiles once
  for (int e = tid; e < 8192 / 16; e += NT) {
    reinterpret_cast<uint4*>(sm + S_AQ)[e] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(sm + S_TN)[e] = make_uint4(0, 0, 0, 0);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sb = smem_u32(sm);
  bool ovf = false;

  if (tid < NPREP) {
    // =================================================================== PREP
    const int p = tid;
    const int w = p >> 5;
    // a warp holds 8 quads (32 tokens) x 4 channel chunks: its 16-byte tile
    // accesses then fall on 8 distinct swizzle positions (conflict-free)
    const int j = 4 * (w >> 1) + (lane >> 3);  // channel chunk
    const int tq = 8 * (w & 1) + (lane & 7);   // token quad
    const int wq = w & 3, half = w >> 2;
    const __nv_bfloat16* gb = static_cast<const __nv_bfloat16*>(a.beta);
    uint32_t t_phase = 0;
    bool alive = true;
    float beta_next[4] = {0.f, 0.f, 0.f, 0.f};
    if (j == 0 && nchunks > 0) {
      const int len0 = min(C, u.len);
#pragma unroll
      for (int uu = 0; uu < 4; ++uu) {
        const int t = 4 * tq + uu;
        beta_next[uu] = t < len0 ? __bfloat162float(gb[u.row0 + t]) : 0.f;
      }
    }
    // q, k, alpha tiles of chunk cc (issued by one thread)
    auto issue_qka = [&](int cc) {
      const int y = (int)(u.row0 + (long)cc * C);
      mbar_arrive_expect_tx(bar_qka, 3 * TILE_BYTES);
      tma_load_2d(sm + S_TQ, &mq, bar_qka, 0, y);
      tma_load_2d(sm + S_TQ + 8192, &mq, bar_qka, 64, y);
      tma_load_2d(sm + S_TK, &mk, bar_qka, 0, y);
      tma_load_2d(sm + S_TK + 8192, &mk, bar_qka, 64, y);
      tma_load_2d(sm + S_TA, &ma, bar_qka, 0, y);
      tma_load_2d(sm + S_TA + 8192, &ma, bar_qka, 64, y);
    };
    if (p == 0 && nchunks > 0) issue_qka(0);
    // waits on an mbarrier fed by this role's MMAs or copies; the AND over
    // the role decides, uniformly, whether to go on
    auto prep_wait = [&](uint64_t* bar, uint32_t& phase) -> bool {
      const bool ok = mbar_wait(bar, phase & 1);
      ++phase;
      const bool all = named_and(BAR_PREP, NPREP, ok);
      tc_fence_after();
      return all;
    };
    // waits for the state role's MMA of chunk cc (bar_s1 or bar_s3); nothing
    // to wait for before the first chunk
    auto prep_state = [&](uint64_t* bar, int cc) -> bool {
      const bool ok = cc < 0 ? true : mbar_wait(bar, (uint32_t)(cc & 1));
      return named_and(BAR_PREP, NPREP, ok);
    };
    // the MMA of the inverse chain: D[lanes 0..63] = A (rows 0..63 used) x B
    auto t_mma = [&](uint32_t d_col, uint32_t a_tile, uint32_t b_tile) {
      const uint64_t da = kmajor_desc(sb + a_tile, 128, 0), db = mnmajor_desc(sb + b_tile, 64, 0);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        umma_ss(tmem + d_col, da + (uint64_t)(2 * k), db + (uint64_t)(128 * k),
                idesc_f16(128, 64, 0, 0, 1), k > 0);
      umma_commit(bar_t);
    };
    auto gram_mma = [&](uint32_t d_col, uint32_t xbuf, uint32_t ybuf, uint64_t* bar) {
      const uint64_t d_gx = kmajor_desc(sb + xbuf, 128, 0), d_gy = kmajor_desc(sb + ybuf, 64, 0);
#pragma unroll
      for (int k = 0; k < 8; ++k)  // K steps: 32 bytes in a panel, panels R*128 apart
        umma_ss(tmem + d_col, d_gx + (uint64_t)((k >> 2) * 1024 + (k & 3) * 2),
                d_gy + (uint64_t)((k >> 2) * 512 + (k & 3) * 2), idesc_f16(128, 64, 0, 0, 0),
                k > 0);
      umma_commit(bar);
    };
    const bool tconv = wq < 2;  // warps 0,1,4,5 reach TMEM lanes 0..63
    const int trow = 32 * wq + lane;
    const uint32_t tl = (uint32_t)(32 * (wq & 1)) << 16;
    const uint32_t tlw = (uint32_t)(32 * wq) << 16;
    uint8_t* AQ = sm + S_AQ;

    uint8_t* X1 = sm + S_GX;   // Gram operand buffers: the dedicated one and the tile region
    uint8_t* Y1 = sm + S_GY;
    uint8_t* X2 = sm + S_GX2;
    uint8_t* Y2 = sm + S_GY2;
    float* dg = reinterpret_cast<float*>(sm + S_DIAG);
    for (int c = 0; c < nchunks && alive; ++c) {
      const int lenc = min(C, u.len - c * C);
      const int buf = c & 1;
      const long rbase = u.row0 + (long)c * C;
      // ---- this chunk's q, k, alpha tiles
      {
        uint32_t ph = (uint32_t)c;
        if (!prep_wait(bar_qka, ph)) { alive = false; break; }
      }
      Prep P;
      P.tq = tq;
      float Bq[8];
      {
        float al[4][8];
        uint32_t inf_or_nan = 0;
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
          const int t = 4 * tq + uu;
          const uint32_t off = sw128_chunk(64, t, j);
          float kk[8], qq[8];
          unpack_bf16x8(*reinterpret_cast<const uint4*>(sm + S_TK + off), kk);
          unpack_bf16x8(*reinterpret_cast<const uint4*>(sm + S_TQ + off), qq);
          unpack_bf16x8(*reinterpret_cast<const uint4*>(sm + S_TA + off), al[uu]);
          float sacc = 0.f;  // partial q.k over this thread's 8 channels
#pragma unroll
          for (int e = 0; e < 8; ++e) sacc = fmaf(qq[e], kk[e], sacc);
          P.k[uu] = to_half8(kk);
          P.q[uu] = to_half8(qq);
          if (lenc < C && t >= lenc) {  // past the end of the sequence: identity transition
            P.k[uu] = make_uint4(0, 0, 0, 0);
            P.q[uu] = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int e = 0; e < 8; ++e) al[uu][e] = 1.f;
            sacc = 0.f;
          }
          dg[j * 64 + t] = sacc;
          // an input outside the fp16 range turns into inf here
          const uint32_t w4[4] = {P.q[uu].x | P.k[uu].x, P.q[uu].y | P.k[uu].y,
                                  P.q[uu].z | P.k[uu].z, P.q[uu].w | P.k[uu].w};
#pragma unroll
          for (int z = 0; z < 4; ++z) inf_or_nan |= __vcmpeq2(w4[z] & 0x7c007c00u, 0x7c007c00u);
        }
        ovf |= inf_or_nan != 0;
        // in-quad prefix / suffix products (fp32, then packed halves)
        float lp[8], ls[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) { lp[e] = al[0][e]; ls[e] = 1.f; }
        P.lp[0] = to_half8(lp);
#pragma unroll
        for (int uu = 1; uu < 4; ++uu) {
#pragma unroll
          for (int e = 0; e < 8; ++e) lp[e] *= al[uu][e];
          P.lp[uu] = to_half8(lp);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) Bq[e] = lp[e];
        P.ls[3] = to_half8(ls);
#pragma unroll
        for (int uu = 2; uu >= 0; --uu) {
#pragma unroll
          for (int e = 0; e < 8; ++e) ls[e] *= al[uu + 1][e];
          P.ls[uu] = to_half8(ls);
        }
        P.a1 = to_half8(al[1]);
        P.a2 = to_half8(al[2]);
        P.a3 = to_half8(al[3]);
      }
      // beta: this chunk's values were loaded one chunk ahead
      float* beta_s = reinterpret_cast<float*>(sm + S_BETA) + 64 * buf;
      if (j == 0) {
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) beta_s[4 * tq + uu] = beta_next[uu];
        if (c + 1 < nchunks) {
          const int lenn = min(C, u.len - (c + 1) * C);
#pragma unroll
          for (int uu = 0; uu < 4; ++uu) {
            const int t = 4 * tq + uu;
            beta_next[uu] = t < lenn ? __bfloat162float(gb[rbase + C + t]) : 0.f;
          }
        }
      }
      // ---- gate products across quads (the scan's barrier also ends the
      // reads of the tile region, which now becomes Gram buffer 2)
      float E16f[8];
      quad_scans(P, Bq, E16f, reinterpret_cast<float*>(sm + S_TOT), j);
      // gamma_C (fp32: it scales the fp32 state): the last quad publishes it
      float* gC = reinterpret_cast<float*>(sm + S_GC) + 128 * buf;
      if (tq == 15) {
#pragma unroll
        for (int e = 0; e < 8; ++e) gC[8 * j + e] = E16f[e] * Bq[e];
      }
      // ---- Gram round 1: levels 8 and 4 (pairs inside 16-token blocks)
      write_level<8>(X2, Y2, P, j, 0, 0);
      write_level<4>(X2, Y2, P, j, 64, 32);
      fence_proxy_async_smem();
      named_sync(BAR_PREP, NPREP);
      if (p == 0) {
        mbar_arrive(bar_gc + (c & 1));
        tc_fence_after();
        gram_mma(T_G0, S_GX2, S_GY2, bar_r + 0);
      }
      // ---- round 2: levels 2 and 1.  Its TMEM tile G1 last held W of the
      // previous chunk, which the state warps convert before their U-MMA.
      write_level<2>(X1, Y1, P, j, 0, 0);
      write_level<1>(X1, Y1, P, j, 64, 32);
      fence_proxy_async_smem();
      if (!prep_state(bar_s1, c - 1)) { alive = false; break; }
      if (p == 0) { tc_fence_after(); gram_mma(T_G1, S_GX, S_GY, bar_r + 1); }
      // ---- k*gamma (bf16, A of the W-MMA; the previous W-MMA is done with it)
      {
        const bool ok = c == 0 ? true : mbar_wait(bar_w, (uint32_t)((c - 1) & 1));
        if (!named_and(BAR_PREP, NPREP, ok)) { alive = false; break; }
      }
#pragma unroll
      for (int uu = 0; uu < 4; ++uu) {
        const int t = 4 * tq + uu;
        store16(sm + S_KGT + sw128_chunk(64, t, j), half8_to_bf8(hmul8h(P.k[uu], P.gamma(uu))));
      }
      // ---- q*gamma, k*rho: the previous chunk's last MMA must have read them
      // (and A, which the Gram read-out below overwrites)
      if (!prep_state(bar_s3, c - 1)) { alive = false; break; }
#pragma unroll
      for (int uu = 0; uu < 4; ++uu) {
        const int t = 4 * tq + uu;
        store16(sm + S_QG + sw128_chunk(64, t, j), hmul8h(P.q[uu], P.gamma(uu)));
        store16(sm + S_KH + sw128_chunk(64, t, j), hmul8h(P.k[uu], P.rho(uu)));
      }
      // ---- round 3 (levels 32 and 16) goes into buffer 2 once round 1 is done
      uint32_t rph = (uint32_t)c;
      if (!prep_wait(bar_r + 0, rph)) { alive = false; break; }
      if (half == 0) extract_round<8>(sm, tmem, T_G0, wq, lane, beta_s, AQ);
      write_level<32>(X2, Y2, P, j, 0, 0);
      write_level<16>(X2, Y2, P, j, 64, 32);
      fence_proxy_async_smem();
      tc_fence_before();
      named_sync(BAR_PREP, NPREP);
      if (p == 0) { tc_fence_after(); gram_mma(T_G0, S_GX2, S_GY2, bar_r + 2); }
      rph = (uint32_t)c;
      if (!prep_wait(bar_r + 1, rph)) { alive = false; break; }  // round 2
      if (half == 1) extract_round<2>(sm, tmem, T_G1, wq, lane, beta_s, AQ);
      // D lives where Gram X was: zero it (its diagonal blocks come next)
      for (int e = p; e < 8192 / 16; e += NPREP) store16(sm + S_TD + 16 * e, make_uint4(0, 0, 0, 0));
      tc_fence_before();
      named_sync(BAR_PREP, NPREP);
      // ---- T = (I + M)^-1 = (I - E)(I + E^2) D with D the inverse of the
      // block diagonal of I + M and E = D N (E^4 = 0: N is strictly lower by
      // 16-blocks); D is formed while round 3 runs, the products on tensor cores
      if (p < 64) invert_diag_blocks(sm, p);
      rph = (uint32_t)c;
      if (!prep_wait(bar_r + 2, rph)) { alive = false; break; }  // round 3
      // the tile region is free: fetch the next chunk's q, k, alpha
      if (p == 0 && c + 1 < nchunks) issue_qka(c + 1);
      if (half == 0) extract_round<32>(sm, tmem, T_G0, wq, lane, beta_s, AQ);
      else if (p >= 128 && p < 192) {
        const int t = p - 128;
        float sacc = 0.f;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) sacc += dg[jj * 64 + t];
        *reinterpret_cast<__half*>(AQ + sw128_off(64, t, t)) = __float2half_rn(sacc);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_sync(BAR_PREP, NPREP);
      if (p == 0) { tc_fence_after(); t_mma(T_G1, S_TD, S_TN); }       // E = D N
      if (!prep_wait(bar_t, t_phase)) { alive = false; break; }
      if (tconv) {
        uint32_t v[32];
        tmem_ld32<32>(tmem + tl + T_G1 + 32 * half, v);
        tmem_ld_wait();
#pragma unroll
        for (int z = 0; z < 32; z += 8) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(v[z + e]);
          store16(sm + S_TE + sw128_chunk(64, trow, (32 * half + z) >> 3), pack_half8(f));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_sync(BAR_PREP, NPREP);
      if (p == 0) { tc_fence_after(); t_mma(T_G0, S_TE, S_TE); }       // E^2
      if (!prep_wait(bar_t, t_phase)) { alive = false; break; }
      float gv[32];  // G = I + E^2, kept for F
      if (tconv) {
        uint32_t v[32];
        tmem_ld32<32>(tmem + tl + T_G0 + 32 * half, v);
        tmem_ld_wait();
#pragma unroll
        for (int z = 0; z < 32; ++z)
          gv[z] = __uint_as_float(v[z]) + ((32 * half + z) == trow ? 1.f : 0.f);
#pragma unroll
        for (int z = 0; z < 32; z += 8) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = gv[z + e];
          store16(sm + S_TG + sw128_chunk(64, trow, (32 * half + z) >> 3), pack_half8(f));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_sync(BAR_PREP, NPREP);
      if (p == 0) { tc_fence_after(); t_mma(T_G1, S_TE, S_TG); }       // E G
      if (!prep_wait(bar_t, t_phase)) { alive = false; break; }
      if (tconv) {
        uint32_t v[32];
        tmem_ld32<32>(tmem + tl + T_G1 + 32 * half, v);
        tmem_ld_wait();
#pragma unroll
        for (int z = 0; z < 32; z += 8) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = gv[z + e] - __uint_as_float(v[z + e]);  // F = G - E G
          store16(sm + S_TFm + sw128_chunk(64, trow, (32 * half + z) >> 3), pack_half8(f));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_sync(BAR_PREP, NPREP);
      if (p == 0) { tc_fence_after(); t_mma(T_G0, S_TFm, S_TD); }      // T = F D
      if (!prep_wait(bar_t, t_phase)) { alive = false; break; }
      // ---- T Diag(beta) as bf16 (TB is single-buffered: the previous
      // chunk's U-MMA read it before this chunk's round 2 was issued)
      if (tconv) {
        uint32_t v[32];
        tmem_ld32<32>(tmem + tl + T_G0 + 32 * half, v);
        tmem_ld_wait();
#pragma unroll
        for (int z = 0; z < 32; z += 8) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int s = 32 * half + z + e;
            f[e] = s <= trow ? __uint_as_float(v[z + e]) * beta_s[s] : 0.f;
          }
          store16(sm + S_TB + sw128_chunk(64, trow, (32 * half + z) >> 3), pack_bf8(f));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_sync(BAR_PREP, NPREP);
      if (p == 0) {
        tc_fence_after();
        // W^T[i][t] = sum_s (k*gamma)[s][i] TB[t][s], into G1; the state warps
        // read it out
        const uint64_t da = mnmajor_desc(sb + S_KGT, 64, 0), db = kmajor_desc(sb + S_TB, 64, 0);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_ss(tmem + T_G1, da + (uint64_t)(128 * k), db + (uint64_t)(2 * k),
                  idesc_f16(128, 64, 1, 1, 0), k > 0);
        umma_commit(bar_w);
        mbar_arrive(bar_ready + (c & 1));
      }
    }
    if (!alive) *reinterpret_cast<volatile int*>(s_abort) = 1;
  } else {
    // ================================================================== STATE
    const int s = tid - NPREP;   // 0..127 = TMEM lane = value column j
    const int wq = s >> 5;       // warps 8..11 -> lane groups 0..3
    const uint32_t lb = (uint32_t)(32 * wq) << 16;
    const bool lead = s == 0;
    float* hT = a.hT;
    bool alive = true;
    if (lead && nchunks > 0) {
      mbar_arrive_expect_tx(bar_v, TILE_BYTES);
      tma_load_2d(sm + S_V, &mv, bar_v, 0, (int)u.row0);
      tma_load_2d(sm + S_V + 8192, &mv, bar_v, 64, (int)u.row0);
    }
    const float* gc_all = reinterpret_cast<const float*>(sm + S_GC);
    // H^T as the fp16 A operand (TMEM) and, in TMEM, H^T Diag(gamma_C) of
    // the chunk about to start (column i times gC[i])
    auto convert_and_scale = [&](int c_next, bool from_h0) {
      const float* gC = gc_all + 128 * (c_next & 1);
#pragma unroll 1
      for (int i0 = 0; i0 < 128; i0 += 32) {
        float f[32];
        if (from_h0) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            f[e] = a.h0 ? a.h0[u.sidx + (size_t)(i0 + e) * 128 + s] : 0.f;
        } else {
          uint32_t v[32];
          tmem_ld32<32>(tmem + lb + T_H + i0, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v[e]);
        }
        uint32_t h[16];
        float mx = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          h[e] = pack_half2(f[2 * e], f[2 * e + 1]);
          mx = fmaxf(mx, fmaxf(fabsf(f[2 * e]), fabsf(f[2 * e + 1])));
        }
        ovf |= !(mx <= 65504.f);
        tmem_st32<16>(tmem + lb + T_HA + (i0 >> 1), h);
        uint32_t o[16];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
          for (int e = 0; e < 16; e += 4) {
            const float4 g4 = *reinterpret_cast<const float4*>(gC + i0 + 16 * hh + e);
            o[e] = __float_as_uint(f[16 * hh + e] * g4.x);
            o[e + 1] = __float_as_uint(f[16 * hh + e + 1] * g4.y);
            o[e + 2] = __float_as_uint(f[16 * hh + e + 2] * g4.z);
            o[e + 3] = __float_as_uint(f[16 * hh + e + 3] * g4.w);
          }
          tmem_st32<16>(tmem + lb + T_H + i0 + 16 * hh, o);
        }
      }
      tmem_st_wait();
    };
    if (nchunks > 0) {
      const bool ok = mbar_wait(bar_gc, 0);
      alive = named_and(BAR_STATE, NSTATE, ok);
      if (alive) convert_and_scale(0, true);
    } else if (hT) {
      for (int i = 0; i < 128; ++i)
        hT[u.sidx + (size_t)i * 128 + s] = a.h0 ? a.h0[u.sidx + (size_t)i * 128 + s] : 0.f;
    }
    tc_fence_before();
    named_sync(BAR_STATE, NSTATE);

    const uint64_t d_v = mnmajor_desc(sb + S_V, 64, 0), d_tb = kmajor_desc(sb + S_TB, 64, 0);
    const uint64_t d_w = mnmajor_desc(sb + S_W, 128, 0), d_qg = kmajor_desc(sb + S_QG, 64, 0);
    const uint64_t d_kh = mnmajor_desc(sb + S_KH, 64, 0), d_aq = kmajor_desc(sb + S_AQ, 64, 0);
    __nv_bfloat16* go = static_cast<__nv_bfloat16*>(a.o);
    for (int c = 0; c < nchunks && alive; ++c) {
      const int lenc = min(C, u.len - c * C);
      {  // prep operands of chunk c, its W^T in TMEM, and its v tile
        bool ok = mbar_wait(bar_ready + (c & 1), (uint32_t)((c >> 1) & 1));
        if (ok) ok = mbar_wait(bar_w, c & 1);
        if (ok) ok = mbar_wait(bar_v, c & 1);
        if (!named_and(BAR_STATE, NSTATE, ok)) { alive = false; break; }
        tc_fence_after();
      }
      {  // -W^T as fp16 [i][t] (MN-major B of the U-MMA): lane = i
        float mx = 0.f;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t v[32];
          tmem_ld32<32>(tmem + lb + T_G1 + 32 * h2, v);
          tmem_ld_wait();
#pragma unroll
          for (int z = 0; z < 32; z += 8) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              f[e] = -__uint_as_float(v[z + e]);
              mx = fmaxf(mx, fabsf(f[e]));
            }
            store16(sm + S_W + sw128_chunk(128, s, (32 * h2 + z) >> 3), pack_half8(f));
          }
        }
        ovf |= !(mx <= 65504.f);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_sync(BAR_STATE, NSTATE);
      if (lead) {
        tc_fence_after();
        // U^T = V^T TB^T - H^T W^T
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_ss(tmem + T_U, d_v + (uint64_t)(128 * k), d_tb + (uint64_t)(2 * k),
                  idesc_f16(128, 64, 1, 1, 0), k > 0);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          umma_ts(tmem + T_U, tmem + T_HA + 8 * k, d_w + (uint64_t)(128 * k),
                  idesc_f16(128, 64, 0, 0, 1), 1);
        umma_commit(bar_s1);
        // O^T = H^T (q*gamma)^T
#pragma unroll
        for (int k = 0; k < 8; ++k)
          umma_ts(tmem + T_O, tmem + T_HA + 8 * k,
                  d_qg + (uint64_t)((k >> 2) * 512 + (k & 3) * 2), idesc_f16(128, 64, 0, 0, 0),
                  k > 0);
      }
      {
        const bool ok = mbar_wait(bar_s1, c & 1);
        if (!named_and(BAR_STATE, NSTATE, ok)) { alive = false; break; }
        tc_fence_after();
      }
      if (lead) {
        if (c + 1 < nchunks) {  // the v tile is free: fetch the next one
          mbar_arrive_expect_tx(bar_v, TILE_BYTES);
          tma_load_2d(sm + S_V, &mv, bar_v, 0, (int)(u.row0 + (long)(c + 1) * C));
          tma_load_2d(sm + S_V + 8192, &mv, bar_v, 64, (int)(u.row0 + (long)(c + 1) * C));
        }
      }
      // U^T -> fp16 A operand in TMEM
      {
        uint32_t v[32];
        float mx = 0.f;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          tmem_ld32<32>(tmem + lb + T_U + 32 * h2, v);
          tmem_ld_wait();
          uint32_t hh[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float x0 = __uint_as_float(v[2 * e]), x1 = __uint_as_float(v[2 * e + 1]);
            hh[e] = pack_half2(x0, x1);
            mx = fmaxf(mx, fmaxf(fabsf(x0), fabsf(x1)));
          }
          tmem_st32<16>(tmem + lb + T_UA + 16 * h2, hh);
        }
        ovf |= !(mx <= 65504.f);
        tmem_st_wait();
      }
      tc_fence_before();
      named_sync(BAR_STATE, NSTATE);
      if (lead) {
        tc_fence_after();
        // H^T += U^T (k*rho);  O^T += U^T A^T
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_ts(tmem + T_H, tmem + T_UA + 8 * k, d_kh + (uint64_t)(128 * k),
                  idesc_f16(128, 128, 0, 0, 1), 1);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_ts(tmem + T_O, tmem + T_UA + 8 * k, d_aq + (uint64_t)(2 * k),
                  idesc_f16(128, 64, 0, 0, 0), 1);
        umma_commit(bar_s3);
      }
      {
        const bool ok = mbar_wait(bar_s3, c & 1);
        if (!named_and(BAR_STATE, NSTATE, ok)) { alive = false; break; }
        tc_fence_after();
      }
      // outputs o[t][j] = scale * O^T[j][t]
      {
        const long rbase = u.row0 + (long)c * C;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t v[32];
          tmem_ld32<32>(tmem + lb + T_O + 32 * h2, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int t = 32 * h2 + e;
            if (t < lenc)
              go[(size_t)(rbase + t) * 128 + s] = __float2bfloat16_rn(a.scale * __uint_as_float(v[e]));
          }
        }
      }
      if (c + 1 < nchunks) {
        const bool ok = mbar_wait(bar_gc + ((c + 1) & 1), (uint32_t)(((c + 1) >> 1) & 1));
        if (!named_and(BAR_STATE, NSTATE, ok)) { alive = false; break; }
        convert_and_scale(c + 1, false);
        tc_fence_before();
        named_sync(BAR_STATE, NSTATE);
      }
    }
    if (alive && nchunks > 0 && hT) {
      for (int i0 = 0; i0 < 128; i0 += 32) {
        uint32_t v[32];
        tmem_ld32<32>(tmem + lb + T_H + i0, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) hT[u.sidx + (size_t)(i0 + e) * 128 + s] = __uint_as_float(v[e]);
      }
    }
    if (!alive) *reinterpret_cast<volatile int*>(s_abort) = 1;
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  const int any_ovf = __syncthreads_or(ovf ? 1 : 0);
  if (tid == 0) {
    if (any_ovf) set_status(a.status, CKDA_ERR_RANGE);
    if (*reinterpret_cast<volatile int*>(s_abort)) {
      set_status(a.status, CKDA_ERR_TIMEOUT);
      // let any MMA or copy still in flight land before the memory is released
      for (int i = 0; i < 3; ++i) mbar_wait(bar_r + i, 0, 1u << 16);
      mbar_wait(bar_t, 0, 1u << 16);
      mbar_wait(bar_w, 0, 1u << 16);
      mbar_wait(bar_s1, 0, 1u << 16);
      mbar_wait(bar_s3, 0, 1u << 16);
      mbar_wait(bar_v, 0, 1u << 16);
      mbar_wait(bar_qka, 0, 1u << 16);
    }
    (void)s_abort;
  }
  __syncthreads();
  tc_fence_after();
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
    mq = mk = ma = mv = CUtensorMap{};  // every sequence is empty: no tile is ever loaded
  } else if (!make_map(&mq, a.q, rows) || !make_map(&mk, a.k, rows) ||
             !make_map(&ma, a.alpha, rows) || !make_map(&mv, a.v, rows)) {
    return cudaErrorInvalidValue;
  }
  cudaError_t err = cudaFuncSetAttribute(
      fwd_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
  if (err != cudaSuccess) return err;
  fwd_chunk_kernel<<<units, NT, SMEM_ALLOC, s>>>(a, mq, mk, ma, mv);
  return cudaGetLastError();
}

}  // namespace ckda
