// ckda_chunk.cu -- chunkwise CKDA forward on tcgen05 tensor cores (sm_103a).
//
// One CTA owns one (sequence, head) and walks its tokens in chunks of C = 64
// with the fp32 state H^T (dv x dk = 128 x 128) resident in tensor memory.
// A 64-wide key (dk = 64) runs as 128 channels whose last 64 have zero keys
// and queries and unit gates: their state rows stay zero and add nothing.
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
//   O  = (q * gamma) H + A U                            -> o
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
// T is formed from D, the inverses of the 16 x 16 diagonal blocks of I + M
// (CUDA cores, fp32), and E = D N with N the rest of M: E is strictly lower
// by blocks, so E^4 = 0 and T = (I + E^2)(I - E) D.  One tensor-core step
// gives E^2 and F = (I - E) D together (operands [E ; I - E] x [E | D]), the
// next T = F + E^2 F with F kept in fp32 in tensor memory.
//
// Precision: operands of every contraction that touches the state, the
// Grams and A are fp16 (11-bit significand); T Diag(beta), k * gamma and the
// raw bf16 inputs are bf16; all accumulation is fp32 in TMEM.  Gate factors
// inside a 16-token block are fp16 product chains; block totals, gamma_C and
// T are fp32.  An fp16 operand that overflows turns into inf and reaches o
// (or the final state); a non-finite o or final state is reported as
// CKDA_ERR_RANGE.
//
// Warp roles (512 threads):
//   warps 0-7   PREP: per chunk, gate products, the gated Grams and their
//               read-outs, D and the operands of the state step.  For the
//               elementwise work thread (blk, panel, lane) owns channels
//               64 panel + 2 lane, +1 of the 16 tokens 16 blk .. 16 blk + 15,
//               so every gate product inside a block is a register chain and
//               every shared-memory access is a conflict-free 4-byte access at
//               a compile-time swizzle.
//   warps 8-11  STATE: the serial state step on TMEM (thread = TMEM lane = j);
//               thread 0 issues its MMAs.
//   warps 12-15 INVERSE CHAIN: once the prep role has handed chunk c's E = D N
//               over, they finish T and W^T (thread = TMEM lane) while the
//               prep role starts chunk c+1.  Lane 0 of warp 12 issues every
//               tensor-core step outside the state role and every copy into
//               shared memory, so that no prep warp stalls on an issue.
// Handoffs are mbarriers (MMA and TMA completion, operand hand-over) and
// named barriers within a role.  Every wait is bounded.
#include "ckda_internal.cuh"
#include "sm103.cuh"

#include <cudaTypedefs.h>
#include <mutex>

namespace ckda {
namespace {

constexpr int C = 64;
constexpr int NPREP = 256;
constexpr int NSTATE = 128;
// A fourth warpgroup finishes each chunk's inverse chain and issues the
// prep role's tensor-core steps and copies.
constexpr int NT = NPREP + NSTATE + 128;
constexpr int MMA_WARP = (NPREP + NSTATE) / 32;
// Registers per thread: 128 at launch (65536 / 512); the prep warpgroups
// raise theirs to 144 and the fourth warpgroup lowers its to 96, which adds up
// to the launch's 512 x 128 exactly (the state warpgroup keeps 128).
constexpr int kRegsLaunch = 128, kRegsPrep = 144, kRegsAux = 96;
static_assert(NPREP * (kRegsPrep - kRegsLaunch) <= 128 * (kRegsLaunch - kRegsAux),
              "register split exceeds what the fourth warpgroup gives up");
constexpr int NTAIL = 128;    // the fourth warpgroup
constexpr int BAR_PREP = 1;   // named barrier ids
constexpr int BAR_STATE = 2;
constexpr int BAR_TAIL = 3;

// ---- shared memory map (bytes from a 1024-aligned base) ----
// q, k, alpha tiles; once read they hold the second Gram operand buffer
// (X over q and k, Y over alpha) until round 3 is done, then the next
// chunk's tiles are fetched into them
constexpr uint32_t S_TQ = 0;         // bf16 q tile   [64 t][128 i]  (TMA)
constexpr uint32_t S_TK = 16384;     // bf16 k tile
constexpr uint32_t S_TA = 32768;     // bf16 alpha tile
constexpr uint32_t S_V = 49152;      // bf16 v tile   [64 s][128 j]  MN-major A of U~   (TMA)
constexpr uint32_t S_GX2 = S_TQ;     // second Gram buffer (the tile region)
constexpr uint32_t S_GY2 = S_TA;
constexpr uint32_t S_GX = 65536;     // fp16 Gram X   [128 rows][128 i] K-major A
constexpr uint32_t S_GY = 98304;     // fp16 Gram Y   [64 rows][128 i]  K-major B
// once round 3 is done, the inverse's 64 x 64 fp16 tiles E and I - E live
// in Gram X:
constexpr uint32_t S_TE = S_GX;            // E, then F = (I - E) D
constexpr uint32_t S_TIE = S_GX + 8192;    // I - E, then E^2
constexpr uint32_t S_TB = 114688;    // bf16 T Diag(beta) [64 t][64 s]
constexpr uint32_t S_TD = S_TB + 8192;     // fp16 D: inverses of the 16 x 16 diagonal blocks
constexpr uint32_t S_WQ = 131072;    // fp16 [-W^T | (q*gamma)^T] [128 i][64 t] x 2 panels, MN-major B of [U|O]
constexpr uint32_t S_AK = 163840;    // fp16 [A ; (k*rho)^T] [64 t + 128 i][64 s]  K-major B of O, H
constexpr uint32_t S_KG = 188416;    // bf16 k*gamma  [64 s][128 i]  MN-major A of W^T
constexpr uint32_t S_TN = 204800;    // fp16 N: block-strictly-lower part of M [64 t][64 s]
constexpr uint32_t S_MD = 212992;    // fp32 diagonal 16 x 16 blocks of M [4][16][20]
constexpr int kMdRow = 20, kMdBlk = 16 * kMdRow;  // padded rows spread the banks
constexpr uint32_t S_SMALL = 218112;
constexpr uint32_t S_BETA = S_SMALL;         // fp32 [2][64]
constexpr uint32_t S_GC = S_SMALL + 512;     // fp32 [2][128] gamma_C
constexpr uint32_t S_DIAG = S_SMALL + 1536;  // fp32 [2 panels][64] partial q.k
constexpr uint32_t S_TOT = S_SMALL + 2048;   // fp32 [4 blocks][128] block totals of alpha
constexpr uint32_t S_BAR = S_SMALL + 4096;   // mbarriers
constexpr uint32_t S_A2 = 223232;    // fp16 A of odd chunks [64 t][64 s] (even chunks' is S_AK's top)
constexpr uint32_t SMEM_USED = S_A2 + 8192;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
static_assert(S_A2 >= S_SMALL + 4352 && S_A2 % 1024 == 0, "second A tile");

// ---- tensor memory columns ----
// [U | O] is the accumulator of the first state MMA and [O | H] of the second
constexpr uint32_t T_U = 0;     // U^T fp32 [128 j][64 t]
constexpr uint32_t T_O = 64;    // O^T fp32 [128 j][64 t]
constexpr uint32_t T_H = 128;   // H^T fp32 [128 j][128 i]     state accumulator
constexpr uint32_t T_HA = 256;  // H^T fp16 [128 j][128 i]     A operand (2 per column)
constexpr uint32_t T_UA = 320;  // U^T fp16 [128 j][64 t]      A operand
constexpr uint32_t T_G0 = 352;  // prep: Gram rounds G0, G1, G0; then E in G1,
constexpr uint32_t T_G1 = 416;  //   [E^2 | F] in G0..G1, T in G1, W^T in G1
constexpr uint32_t TMEM_COLS = 512;

// ---- mbarriers ----
// prep -> issuer "operands ready" (Gram rounds and E) and MMA -> waiters
// "step done", one pair per tensor-core step outside the state role
enum Step : int { ST_R1 = 0, ST_R2, ST_R3, ST_E, ST_X, ST_T, ST_W, ST_COUNT };
enum Bar : int {
  B_QKA = 0,                   // q, k, alpha tiles (TMA)
  B_V,                         // v tile (TMA)
  B_OPS,                       // [ST_COUNT]
  B_DONE = B_OPS + ST_COUNT,   // [ST_COUNT]
  B_S1 = B_DONE + ST_COUNT,    // state: [U | O] MMA done
  B_S3,                        // state: [O | H] MMA done
  B_READY,                     // [2] prep and warp 12 -> state: chunk operands in place
  B_GC = B_READY + 2,          // [2] prep -> state: gamma_C published
  B_BETA = B_GC + 2,           // warp 12 -> prep: a chunk's beta is in shared memory (32 arrivals)
  B_COUNT
};
static_assert(B_COUNT * 8 <= 192, "mbarrier area");

constexpr uint32_t TILE_BYTES = 16384;

// What one CTA runs: its rows, its initial and final state, and (in the
// sequence split) whether its initial state is [I | 0], its v is zero and its
// o is stored.
struct Unit {
  long row0;
  int len;
  size_t sidx;       // plain kernel: offset of the (sequence, head) in h0 and hT
  const float* h0;   // split: [DK][128] initial state, or null: zero (or [I | 0] if ident)
  float* hT;         // split: [DK][128] final state, or null: not stored
  bool ident, zero_v, write_o;
};

template <int DK, bool SPLIT>
__device__ __forceinline__ Unit unit_of(const FwdArgs& a) {
  Unit u;
  constexpr size_t tile = (size_t)DK * 128;
  u.ident = false;
  u.zero_v = false;
  u.write_o = true;
  if constexpr (SPLIT) {
    // dense layout; CTA b is (sequence, head) ui, role r of its pass
    const int S = a.nseg;
    const int per = split_ctas_per_unit(a.split_pass, S);
    const int ui = (int)blockIdx.x / per, r = (int)blockIdx.x % per;
    const size_t slot0 = (size_t)ui * S;
    int seg;
    u.h0 = nullptr;
    u.hT = nullptr;
    if (a.split_pass == 1) {
      u.write_o = r == 0;
      if (r == 0) {          // segment 0 from h0; its final state enters segment 1
        seg = 0;
        u.h0 = a.h0 ? a.h0 + (size_t)ui * tile : nullptr;
        u.hT = a.seg_state + (slot0 + 1) * tile;
      } else if (r <= S - 2) {  // final state of segment r from zero
        seg = r;
        u.hT = a.seg_F + (slot0 + seg) * tile;
      } else {               // transition of segment r - (S - 2): from [I | 0], v = 0
        seg = r - (S - 2);
        u.ident = true;
        u.zero_v = true;
        u.hT = a.seg_P + (slot0 + seg) * tile;
      }
    } else {
      seg = 1 + r;
      u.h0 = a.seg_state + (slot0 + seg) * tile;
      u.hT = (seg == S - 1 && a.hT) ? a.hT + (size_t)ui * tile : nullptr;
    }
    u.row0 = (long)ui * a.T + (long)seg * a.seg_len;
    u.len = min(a.seg_len, a.T - seg * a.seg_len);
  } else {
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
    u.sidx = ((size_t)n * a.H + h) * tile;
  }
  return u;
}

__device__ __forceinline__ uint4 pack_half8(const float (&f)[8]) {
  return make_uint4(pack_half2(f[0], f[1]), pack_half2(f[2], f[3]), pack_half2(f[4], f[5]),
                    pack_half2(f[6], f[7]));
}
__device__ __forceinline__ uint4 pack_bf8(const float (&f)[8]) {
  return make_uint4(pack_bf162(f[0], f[1]), pack_bf162(f[2], f[3]), pack_bf162(f[4], f[5]),
                    pack_bf162(f[6], f[7]));
}
__device__ __forceinline__ void store16(uint8_t* p, const uint4& v) {
  *reinterpret_cast<uint4*>(p) = v;
}
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// ------------------------------------------------ prep elementwise mapping
// Thread part of the byte offset of the channel pair (64 panel + 2 lane, +1)
// in a 128B-swizzled tile of R rows with 64-column panels: the panel, the
// 16-byte chunk (lane >> 2, bits 4..6) and the word in it.
template <uint32_t R>
__device__ __forceinline__ uint32_t pair_tb(int panel, int lane) {
  return (uint32_t)panel * R * 128u + (((uint32_t)lane >> 2) << 4) + (((uint32_t)lane & 3u) << 2);
}
// Offset of that pair in row rowbase + rc (rowbase a multiple of 8, rc a
// compile-time constant): the row's swizzle is an XOR of bits 4..6.
__device__ __forceinline__ uint32_t pair_at(uint32_t tb, uint32_t rowbase, uint32_t rc) {
  return (tb ^ ((rc & 7u) << 4)) + (rowbase + rc) * 128u;
}
__device__ __forceinline__ void st_pair(uint8_t* p, __half2 v) {
  *reinterpret_cast<uint32_t*>(p) = h2u(v);
}

// One 16-token block of one channel pair: k, scale * q and alpha as fp16
// pairs, the fp32 partial q.k of each token and the fp32 block total of alpha.
struct Blk {
  __half2 a[16], k[16], q[16];
  float dqk[16];
  float2 tot;
};
// Loads the block from the q, k, alpha tiles.  Tokens at or past `live` (the
// end of the sequence, relative to the block) become identity transitions.
// With pad set (channels past a 64-wide key) nothing is read: k = q = 0 and
// alpha = 1, so that the state's rows for them stay zero and add nothing.
template <bool kMask>
__device__ __forceinline__ void load_block(Blk& B, const uint8_t* sm, int blk, int panel, int lane,
                                           float scale, int live, bool pad = false) {
  B.tot = make_float2(1.f, 1.f);
  const uint32_t tb = pair_tb<64>(panel, lane);
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const uint32_t off = pair_at(tb, 16 * blk, r);
    uint32_t kw = 0u, qw = 0u, aw = 0x3F803F80u;  // bf16 pairs (0, 0) and (1, 1)
    if (!pad) {
      kw = *reinterpret_cast<const uint32_t*>(sm + S_TK + off);
      qw = *reinterpret_cast<const uint32_t*>(sm + S_TQ + off);
      aw = *reinterpret_cast<const uint32_t*>(sm + S_TA + off);
    }
    float2 kf = make_float2(__uint_as_float(kw << 16), __uint_as_float(kw & 0xffff0000u));
    float2 qf = make_float2(__uint_as_float(qw << 16) * scale,
                            __uint_as_float(qw & 0xffff0000u) * scale);
    float2 af = make_float2(__uint_as_float(aw << 16), __uint_as_float(aw & 0xffff0000u));
    if (kMask && r >= live) {
      kf = make_float2(0.f, 0.f);
      qf = make_float2(0.f, 0.f);
      af = make_float2(1.f, 1.f);
    }
    B.dqk[r] = fmaf(qf.x, kf.x, qf.y * kf.y);
    B.k[r] = __float22half2_rn(kf);
    B.q[r] = __float22half2_rn(qf);
    B.a[r] = __float22half2_rn(af);
    B.tot.x *= af.x;
    B.tot.y *= af.y;
  }
}
// Sums v[r] over the 32 lanes of a warp by halving exchanges; afterwards lanes
// 2m and 2m+1 both hold the sum for r = m.
__device__ __forceinline__ float warp_sum16(float (&v)[16], int lane) {
#pragma unroll
  for (int w = 16, n = 8; w >= 2; w >>= 1, n >>= 1) {
    const bool hi = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float send = hi ? v[i] : v[i + n];
      const float keep = hi ? v[i + n] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// Gram operands of one tree level L <= 8 (pairs inside a 16-token block):
// X rows xrow.. (k rows) and xrow+32.. (q rows) of its upper tokens, Y rows
// yrow.. of its lower tokens, each gated by the token's factor: the product
// of alpha from the start of its upper half to t, or over (s, end of its
// lower half].  A block holds 8 upper and 8 lower ranks of every such level.
template <int L, uint32_t XT, uint32_t YT, int XROW, int YROW>
__device__ __forceinline__ void write_level_in(uint8_t* sm, const Blk& B, int blk, int panel,
                                               int lane) {
  const uint32_t tx = pair_tb<128>(panel, lane), ty = pair_tb<64>(panel, lane);
  uint8_t* X = sm + XT + 8 * blk * 128;
  uint8_t* Y = sm + YT + 8 * blk * 128;
#pragma unroll
  for (int seg = 0; seg < 16; seg += 2 * L) {
    const int rk0 = (seg / (2 * L)) * L;
    __half2 f = B.a[seg + L];
#pragma unroll
    for (int uu = 0; uu < L; ++uu) {
      const int r = seg + L + uu;
      if (uu > 0) f = __hmul2(f, B.a[r]);
      st_pair(X + pair_at(tx, XROW, rk0 + uu), __hmul2(B.k[r], f));
      st_pair(X + pair_at(tx, XROW + 32, rk0 + uu), __hmul2(B.q[r], f));
    }
    __half2 b = B.a[seg + L - 1];
#pragma unroll
    for (int uu = L - 1; uu >= 0; --uu) {
      const int r = seg + uu;
      if (uu < L - 2) b = __hmul2(b, B.a[r + 1]);
      st_pair(Y + pair_at(ty, YROW, rk0 + uu), uu == L - 1 ? B.k[r] : __hmul2(B.k[r], b));
    }
  }
}
// Cross-block levels 32 and 16 of block BLK: level 32 into X rows x32 (k),
// x32 + 32 (q) or Y rows y32, level 16 into x16 / y16.  Block b is upper at
// level 16 if b is odd and at level 32 if b >= 2.  Upper factors are the
// running in-block prefix product of alpha (times block 2's total in block 3
// at level 32); lower factors the running in-block exclusive suffix product
// (times block 1's total in block 0 at level 32).  Ranks: 16 (b >> 1) + r at
// level 16, 16 (b mod 2) + r at level 32.
template <int BLK, uint32_t XT, uint32_t YT>
__device__ __forceinline__ void write_cross(uint8_t* sm, const Blk& B, __half2 t1, __half2 t2,
                                            int panel, int lane) {
  constexpr bool up16 = (BLK & 1) != 0, up32 = BLK >= 2;
  constexpr int rb16 = 16 * (BLK >> 1), rb32 = 16 * (BLK & 1);
  constexpr int x32 = 0, x16 = 64, y32 = 0, y16 = 32;
  const uint32_t tx = pair_tb<128>(panel, lane), ty = pair_tb<64>(panel, lane);
  uint8_t* X = sm + XT;
  uint8_t* Y = sm + YT;
  if (up16 || up32) {
    __half2 pr = B.a[0];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      if (r > 0) pr = __hmul2(pr, B.a[r]);
      if (up16) {
        st_pair(X + pair_at(tx, x16 + rb16, r), __hmul2(B.k[r], pr));
        st_pair(X + pair_at(tx, x16 + 32 + rb16, r), __hmul2(B.q[r], pr));
      }
      if (up32) {
        const __half2 f = BLK == 3 ? __hmul2(t2, pr) : pr;
        st_pair(X + pair_at(tx, x32 + rb32, r), __hmul2(B.k[r], f));
        st_pair(X + pair_at(tx, x32 + 32 + rb32, r), __hmul2(B.q[r], f));
      }
    }
  }
  if (!up16 || !up32) {
    __half2 sr = B.a[15];
#pragma unroll
    for (int r = 15; r >= 0; --r) {
      if (r < 14) sr = __hmul2(sr, B.a[r + 1]);
      if (!up16) st_pair(Y + pair_at(ty, y16 + rb16, r), r == 15 ? B.k[r] : __hmul2(B.k[r], sr));
      if (!up32) {
        const __half2 g = BLK == 0 ? (r == 15 ? t1 : __hmul2(sr, t1)) : sr;
        st_pair(Y + pair_at(ty, y32 + rb32, r),
                (BLK == 1 && r == 15) ? B.k[r] : __hmul2(B.k[r], g));
      }
    }
  }
}
// Rows i0 = 64 panel + 2 lane and i0 + 1 of a transposed [i][t] tile (one
// 64-column panel, rows of 128 bytes): the 16 tokens of block blk are two
// 16-byte chunks per row, assembled from the per-token channel pairs.  Lanes
// 4..7 mod 8 write their second chunk first: the rows of one store then fall
// in 4 swizzle phases x 2 chunks, 8 distinct bank groups.
__device__ __forceinline__ void store_transposed(uint8_t* tile, const __half2 (&v)[16], int blk,
                                                 int panel, int lane) {
  const uint32_t flip = ((uint32_t)lane >> 2) & 1u;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const uint32_t i = (uint32_t)(64 * panel + 2 * lane + e);
    const uint32_t sel = e ? 0x7632u : 0x5410u;
    uint32_t w[2][4];
#pragma unroll
    for (int hc = 0; hc < 2; ++hc)
#pragma unroll
      for (int m = 0; m < 4; ++m)
        w[hc][m] = __byte_perm(h2u(v[8 * hc + 2 * m]), h2u(v[8 * hc + 2 * m + 1]), sel);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint32_t hc = (uint32_t)k ^ flip;
      const uint4 x = hc ? make_uint4(w[1][0], w[1][1], w[1][2], w[1][3])
                         : make_uint4(w[0][0], w[0][1], w[0][2], w[0][3]);
      const uint32_t ch = (uint32_t)(2 * blk) + hc;
      store16(tile + i * 128u + ((ch ^ (i & 7u)) << 4), x);
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

// Inverses of the four unit-lower 16 x 16 diagonal blocks of I + M, one
// column per thread by left-looking substitution: x_c = 1 and, for t > c,
// x_t = -sum_{s<t} M[t][s] x_s (x_s = 0 for s < c), each row of the block
// read once as float4s; written as fp16 into the diagonal blocks of D.
// Threads 0..63.
__device__ __forceinline__ float f4c(const float4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}
// Rows are taken four at a time: the four dot products with the earlier
// rows' x are independent, then a 4 x 4 triangular step finishes the block.
__device__ __forceinline__ void invert_diag_blocks(uint8_t* sm, int p) {
  const int blk = p >> 4, c = p & 15, o = 16 * blk;
  const float* Md = reinterpret_cast<const float*>(sm + S_MD) + blk * kMdBlk;
  float x[16];
#pragma unroll
  for (int ib = 0; ib < 4; ++ib) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q4 = 0; q4 < ib; ++q4) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float4 m = *reinterpret_cast<const float4*>(Md + (4 * ib + r) * kMdRow + 4 * q4);
        acc[r] = fmaf(m.w, x[4 * q4 + 3],
                      fmaf(m.z, x[4 * q4 + 2], fmaf(m.y, x[4 * q4 + 1], fmaf(m.x, x[4 * q4], acc[r]))));
      }
    }
    float4 mr[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) mr[r] = *reinterpret_cast<const float4*>(Md + (4 * ib + r) * kMdRow + 4 * ib);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int t = 4 * ib + r;
      float a = acc[r];
#pragma unroll
      for (int r2 = 0; r2 < r; ++r2) a = fmaf(f4c(mr[r], r2), x[4 * ib + r2], a);
      x[t] = t < c ? 0.f : (t == c ? 1.f : -a);
    }
  }
#pragma unroll
  for (int t = 0; t < 16; ++t)
    *reinterpret_cast<__half*>(sm + S_TD + sw128_off(64, o + t, o + c)) = __float2half_rn(x[t]);
}

// DK: the caller's key width, 128 or 64 (a compile-time constant, so that
// the 128-wide kernel carries nothing for the narrower one).  SPLIT: one pass
// of the sequence split (per-CTA roles from unit_of); the plain kernel
// carries none of it.
template <int DK, bool SPLIT>
__global__ void __launch_bounds__(NT, 1)
    fwd_chunk_kernel(const __grid_constant__ FwdArgs a, const __grid_constant__ CUtensorMap mq,
                     const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap ma,
                     const __grid_constant__ CUtensorMap mv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S_BAR);
  uint64_t* bar_qka = bars + B_QKA;
  uint64_t* bar_v = bars + B_V;
  uint64_t* bar_ops = bars + B_OPS;
  uint64_t* bar_done = bars + B_DONE;
  uint64_t* bar_s1 = bars + B_S1;
  uint64_t* bar_s3 = bars + B_S3;
  uint64_t* bar_ready = bars + B_READY;
  uint64_t* bar_gc = bars + B_GC;
  uint64_t* bar_beta = bars + B_BETA;
  int* s_abort = reinterpret_cast<int*>(sm + S_BAR + 192);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S_BAR + 200);

  static_assert(DK == 128 || DK == 64, "key width");
  const Unit u = unit_of<DK, SPLIT>(a);
  const bool zero_v = SPLIT && u.zero_v;    // no v tile is read; U~ = 0
  const int nchunks = (u.len + C - 1) / C;

  if (tid == 0) {
    for (int i = 0; i < B_COUNT; ++i)
      mbar_init(bars + i, i == B_BETA ? 32 : (i == B_READY || i == B_READY + 1) ? 2 : 1);
    *s_abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&mq);
    tma_prefetch_desc(&mk);
    tma_prefetch_desc(&ma);
    tma_prefetch_desc(&mv);
  }
  // A's upper triangle and N's blocks on and above the 16-block diagonal are
  // never written: clear them once
  for (int e = tid; e < 8192 / 16; e += NT) {
    reinterpret_cast<uint4*>(sm + S_AK)[e] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(sm + S_A2)[e] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(sm + S_TN)[e] = make_uint4(0, 0, 0, 0);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sb = smem_u32(sm);
  bool ovf = false;
  if (warp < NPREP / 32) setmaxnreg_inc<kRegsPrep>();
  else if (warp >= MMA_WARP) setmaxnreg_dec<kRegsAux>();

  // q, k, alpha tiles of chunk cc (one thread)
  // (with dk = 64 only the first 64-channel panel of each tile is loaded;
  // the prep role treats channels 64..127 as padding)
  constexpr bool dk64 = DK == 64;
  auto issue_qka = [&](int cc) {
    const int y = (int)(u.row0 + (long)cc * C);
    mbar_arrive_expect_tx(bar_qka, dk64 ? 3 * TILE_BYTES / 2 : 3 * TILE_BYTES);
    tma_load_2d(sm + S_TQ, &mq, bar_qka, 0, y);
    tma_load_2d(sm + S_TK, &mk, bar_qka, 0, y);
    tma_load_2d(sm + S_TA, &ma, bar_qka, 0, y);
    if (!dk64) {
      tma_load_2d(sm + S_TQ + 8192, &mq, bar_qka, 64, y);
      tma_load_2d(sm + S_TK + 8192, &mk, bar_qka, 64, y);
      tma_load_2d(sm + S_TA + 8192, &ma, bar_qka, 64, y);
    }
  };

  if (tid < NPREP) {
    // =================================================================== PREP
    // Chunk cn: loads, gate products, the Gram rounds and their read-outs and
    // D; E = D N is handed to the fourth warpgroup, which finishes the chunk
    // (T, W) while this role stores the chunk's operands of the state step
    // (once the state has released their tiles) and starts the next chunk.
    const int p = tid;
    const int w = p >> 5;
    const int blk = w >> 1, panel = w & 1;     // elementwise mapping
    const int wq = w & 3, half = w >> 2;       // TMEM lane quarter, column half
    bool alive = true;
    // waits for a completion of chunk cc on `bar` (one phase per chunk); the
    // AND over the role decides, uniformly, whether to go on
    auto prep_wait = [&](uint64_t* bar, int cc) -> bool {
      const bool ok = cc < 0 ? true : mbar_wait(bar, (uint32_t)(cc & 1));
      const bool all = named_and(BAR_PREP, NPREP, ok);
      tc_fence_after();
      return all;
    };
    // makes every operand written so far visible to the tensor cores
    auto publish = [&]() {
      fence_proxy_async_smem();
      tc_fence_before();
      named_sync(BAR_PREP, NPREP);
    };
    float* dg = reinterpret_cast<float*>(sm + S_DIAG);
    float2* totv = reinterpret_cast<float2*>(sm + S_TOT);
    Blk B;
    for (int cn = 0; cn < nchunks && alive; ++cn) {
      const int c = cn - 1;                    // the chunk the fourth warpgroup finishes meanwhile
      const int lenn = min(C, u.len - cn * C);
      // A alternates between two tiles by chunk parity, so that its entries
      // are written as they are read out (the state's step two chunks back
      // was the last reader of this one)
      uint8_t* AQ = sm + ((cn & 1) ? S_A2 : S_AK);
      float* beta_n = reinterpret_cast<float*>(sm + S_BETA) + 64 * (cn & 1);
      // ---- q, k, alpha
      if (!prep_wait(bar_qka, cn)) { alive = false; break; }
      const bool pad = dk64 && panel == 1;
      if (lenn == C) load_block<false>(B, sm, blk, panel, lane, a.scale, C, pad);
      else load_block<true>(B, sm, blk, panel, lane, a.scale, lenn - 16 * blk, pad);
      {
        const float sq = warp_sum16(B.dqk, lane);   // q.k over this panel's 64 channels
        if ((lane & 1) == 0) dg[64 * panel + 16 * blk + (lane >> 1)] = sq;
      }
      totv[64 * blk + 32 * panel + lane] = B.tot;
      // (block totals visible; the tile reads are done, so the tile region
      // becomes Gram buffer 2)
      named_sync(BAR_PREP, NPREP);
      __half2 Gb, Ga, t1, t2;
      {
        float2 T4[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) T4[b] = totv[64 * b + 32 * panel + lane];
        float2 gbf = make_float2(1.f, 1.f), gaf = make_float2(1.f, 1.f);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          if (b < blk) { gbf.x *= T4[b].x; gbf.y *= T4[b].y; }
          if (b > blk) { gaf.x *= T4[b].x; gaf.y *= T4[b].y; }
        }
        Gb = __float22half2_rn(gbf);
        Ga = __float22half2_rn(gaf);
        t1 = __float22half2_rn(T4[1]);
        t2 = __float22half2_rn(T4[2]);
        // gamma_C (fp32: it scales the fp32 state)
        float* gC = reinterpret_cast<float*>(sm + S_GC) + 128 * (cn & 1);
        if (blk == 0)
          reinterpret_cast<float2*>(gC)[32 * panel + lane] = make_float2(
              T4[0].x * T4[1].x * T4[2].x * T4[3].x, T4[0].y * T4[1].y * T4[2].y * T4[3].y);
      }
      // Gram round 1: levels 8 and 4 (pairs inside 16-token blocks), buffer 2
      write_level_in<8, S_GX2, S_GY2, 0, 0>(sm, B, blk, panel, lane);
      write_level_in<4, S_GX2, S_GY2, 64, 32>(sm, B, blk, panel, lane);
      publish();
      if (p == 0) {
        mbar_arrive(bar_ops + ST_R1);
        mbar_arrive(bar_gc + (cn & 1));
      }
      // Gram round 3 (levels 32 and 16) into buffer 1, once the previous
      // chunk's T step has read its E and I - E tiles there
      if (!prep_wait(bar_done + ST_T, c)) { alive = false; break; }
      switch (blk) {
        case 0: write_cross<0, S_GX, S_GY>(sm, B, t1, t2, panel, lane); break;
        case 1: write_cross<1, S_GX, S_GY>(sm, B, t1, t2, panel, lane); break;
        case 2: write_cross<2, S_GX, S_GY>(sm, B, t1, t2, panel, lane); break;
        default: write_cross<3, S_GX, S_GY>(sm, B, t1, t2, panel, lane); break;
      }
      publish();
      if (p == 0) mbar_arrive(bar_ops + ST_R3);
      // round 1 done (and the chunk's beta, first used by the read-out, in
      // place): warps 0-3 read it out while the rest start round 2 (levels 2
      // and 1) in buffer 2
      {
        bool ok = mbar_wait(bar_done + ST_R1, (uint32_t)(cn & 1));
        if (ok) ok = mbar_wait(bar_beta, (uint32_t)(cn & 1));
        if (!named_and(BAR_PREP, NPREP, ok)) { alive = false; break; }
        tc_fence_after();
      }
      if (half == 0) extract_round<8>(sm, tmem, T_G0, wq, lane, beta_n, AQ);
      write_level_in<2, S_GX2, S_GY2, 0, 0>(sm, B, blk, panel, lane);
      write_level_in<1, S_GX2, S_GY2, 64, 32>(sm, B, blk, panel, lane);
      publish();
      if (p == 0) mbar_arrive(bar_ops + ST_R2);                  // (G0 has been read out)
      // gamma_t = (earlier blocks' totals) x prefix_t, a running product;
      // k*gamma (bf16, A of the W^T step: the previous chunk's has read it);
      // (q*gamma) and (k*rho), rho_s = exclusive suffix x later blocks'
      // totals, stay in registers until the state releases their tiles
      if (!prep_wait(bar_done + ST_W, c)) { alive = false; break; }
      __half2 gq[16], kr[16];
      {
        __half2 g = Gb;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          g = __hmul2(g, B.a[r]);
          const float2 kg = __half22float2(__hmul2(B.k[r], g));
          *reinterpret_cast<uint32_t*>(sm + S_KG + pair_at(pair_tb<64>(panel, lane), 16 * blk, r)) =
              pack_bf162(kg.x, kg.y);
          gq[r] = __hmul2(B.q[r], g);
        }
        __half2 rr = Ga;
#pragma unroll
        for (int r = 15; r >= 0; --r) {
          if (r < 15) rr = __hmul2(rr, B.a[r + 1]);
          kr[r] = __hmul2(B.k[r], rr);
        }
      }
      // round 2 done: warps 4-7 read it out; the tile region is free, so
      // chunk cn+1's q, k, alpha are fetched now; D (in its own tile) is
      // cleared for its diagonal blocks
      if (!prep_wait(bar_done + ST_R2, cn)) { alive = false; break; }
      if (p == 0 && cn + 1 < nchunks) issue_qka(cn + 1);
      if (half == 1) extract_round<2>(sm, tmem, T_G0, wq, lane, beta_n, AQ);
      for (int e = p; e < 8192 / 16; e += NPREP) store16(sm + S_TD + 16 * e, make_uint4(0, 0, 0, 0));
      tc_fence_before();
      named_sync(BAR_PREP, NPREP);
      // T = (I + M)^-1: warps 0-1 invert D's diagonal blocks while warps 2-5
      // (one per TMEM lane quarter) read round 3 out and warps 6-7 add up A's
      // diagonal
      bool ok = true;
      if (w < 2) {
        invert_diag_blocks(sm, p);
      } else if (w < 6) {
        ok = mbar_wait(bar_done + ST_R3, (uint32_t)(cn & 1));
        tc_fence_after();
        if (ok) extract_round<32>(sm, tmem, T_G1, wq, lane, beta_n, AQ);
      } else {
        const int t = p - 192;
        *reinterpret_cast<__half*>(AQ + sw128_off(64, t, t)) = __float2half_rn(dg[t] + dg[64 + t]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      if (!named_and(BAR_PREP, NPREP, ok)) { alive = false; break; }
      if (p == 0) mbar_arrive(bar_ops + ST_E);                   // E = D N
      // the state step's operands: (q*gamma)^T next to -W^T and (k*rho)^T,
      // once the previous chunk's [O | H] MMAs (issued after its [U | O] MMA
      // had completed) have read them
      if (!prep_wait(bar_s3, c)) { alive = false; break; }
      store_transposed(sm + S_WQ + 16384, gq, blk, panel, lane);
      store_transposed(sm + S_AK + 8192, kr, blk, panel, lane);
      fence_proxy_async_smem();
      named_sync(BAR_PREP, NPREP);
      if (p == 0) mbar_arrive(bar_ready + (cn & 1));             // (with warp 12's)
    }
    if (!alive) *reinterpret_cast<volatile int*>(s_abort) = 1;
  } else if (tid < NPREP + NSTATE) {
    // ================================================================== STATE
    const int s = tid - NPREP;   // 0..127 = TMEM lane = value column j
    const int wq = s >> 5;       // warps 8..11 -> lane groups 0..3
    const uint32_t lb = (uint32_t)(32 * wq) << 16;
    const bool lead = s == 0;
    // the final state of this CTA's (sequence, head) is hT + hoff, or none
    float* hT = SPLIT ? u.hT : a.hT;
    const size_t hoff = SPLIT ? 0 : u.sidx;
    bool alive = true;
    const float* gc_all = reinterpret_cast<const float*>(sm + S_GC);
    // H^T as the fp16 A operand (TMEM) and, in TMEM, H^T Diag(gamma_C) of
    // the chunk about to start (column i times gC[i])
    auto convert_and_scale = [&](int c_next, bool from_h0) {
      const float* gC = gc_all + 128 * (c_next & 1);
#pragma unroll 1
      for (int i0 = 0; i0 < 128; i0 += 16) {
        float f[16];
        if (from_h0) {
          if constexpr (SPLIT) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              f[e] = 0.f;
              if (i0 + e < DK) {
                if (u.h0) f[e] = u.h0[(size_t)(i0 + e) * 128 + s];
                else if (u.ident && i0 + e == s) f[e] = 1.f;
              }
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e)
              f[e] = (a.h0 && i0 + e < DK) ? a.h0[u.sidx + (size_t)(i0 + e) * 128 + s] : 0.f;
          }
        } else {
          uint32_t v[16];
          tmem_ld32<16>(tmem + lb + T_H + i0, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) f[e] = __uint_as_float(v[e]);
        }
        uint32_t h[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = pack_half2(f[2 * e], f[2 * e + 1]);
        tmem_st32<8>(tmem + lb + T_HA + (i0 >> 1), h);
        uint32_t o[16];
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          const float4 g4 = *reinterpret_cast<const float4*>(gC + i0 + e);
          o[e] = __float_as_uint(f[e] * g4.x);
          o[e + 1] = __float_as_uint(f[e + 1] * g4.y);
          o[e + 2] = __float_as_uint(f[e + 2] * g4.z);
          o[e + 3] = __float_as_uint(f[e + 3] * g4.w);
        }
        tmem_st32<16>(tmem + lb + T_H + i0, o);
      }
      tmem_st_wait();
    };
    if (nchunks > 0) {
      const bool ok = mbar_wait(bar_gc, 0);
      alive = named_and(BAR_STATE, NSTATE, ok);
      if (alive) convert_and_scale(0, true);
    } else if (hT) {
      const float* h0 = SPLIT ? u.h0 : a.h0;
      for (int i = 0; i < DK; ++i)
        hT[hoff + (size_t)i * 128 + s] =
            h0 ? h0[hoff + (size_t)i * 128 + s] : ((SPLIT && u.ident && i == s) ? 1.f : 0.f);
    }
    tc_fence_before();
    named_sync(BAR_STATE, NSTATE);

    __nv_bfloat16* go = static_cast<__nv_bfloat16*>(a.o);
    float fin = 0.f;  // becomes NaN once any output is inf or NaN
    for (int c = 0; c < nchunks && alive; ++c) {
      const int lenc = min(C, u.len - c * C);
      {  // O starts from zero (the previous chunk's has been read out), and
         // so does U when v is zero (no U~ step)
        const uint32_t z[16] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
        for (int i0 = 0; i0 < 64; i0 += 16) tmem_st32<16>(tmem + lb + T_O + i0, z);
        if (zero_v) {
#pragma unroll
          for (int i0 = 0; i0 < 64; i0 += 16) tmem_st32<16>(tmem + lb + T_U + i0, z);
        }
        tmem_st_wait();
        tc_fence_before();
      }
      {  // prep operands of chunk c in shared memory, and its v tile
        bool ok = mbar_wait(bar_ready + (c & 1), (uint32_t)((c >> 1) & 1));
        if (ok && !zero_v) ok = mbar_wait(bar_v, (uint32_t)(c & 1));
        if (!named_and(BAR_STATE, NSTATE, ok)) { alive = false; break; }
        tc_fence_after();
      }
      if (lead) {
        // U~^T = V^T TB^T, then [U^T | O^T] += H^T [-W^T | (q*gamma)^T]
        if (!zero_v) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_ss(tmem + T_U, mnmajor_desc(sb + S_V, 64, k), kmajor_desc(sb + S_TB, 64, k),
                    idesc_f16(128, 64, 1, 1, 0), k > 0);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
          umma_ts(tmem + T_U, tmem + T_HA + 8 * k, mnmajor_desc(sb + S_WQ, 128, k),
                  idesc_f16(128, 128, 0, 0, 1), 1);
        umma_commit(bar_s1);
      }
      {
        const bool ok = mbar_wait(bar_s1, c & 1);
        if (!named_and(BAR_STATE, NSTATE, ok)) { alive = false; break; }
        tc_fence_after();
      }
      if (lead && c + 1 < nchunks && !zero_v) {  // the v tile is free: fetch the next one
        const int y = (int)(u.row0 + (long)(c + 1) * C);
        mbar_arrive_expect_tx(bar_v, TILE_BYTES);
        tma_load_2d(sm + S_V, &mv, bar_v, 0, y);
        tma_load_2d(sm + S_V + 8192, &mv, bar_v, 64, y);
      }
      // U^T -> fp16 A operand in TMEM
      {
        uint32_t v[32];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          tmem_ld32<32>(tmem + lb + T_U + 32 * h2, v);
          tmem_ld_wait();
          uint32_t hh[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            hh[e] = pack_half2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
          tmem_st32<16>(tmem + lb + T_UA + 16 * h2, hh);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      named_sync(BAR_STATE, NSTATE);
      if (lead) {
        tc_fence_after();
        // O^T += U^T A^T (A of this chunk's parity), H^T += U^T (k*rho)
        const uint32_t sa = (c & 1) ? S_A2 : S_AK;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_ts(tmem + T_O, tmem + T_UA + 8 * k, kmajor_desc(sb + sa, 64, k),
                  idesc_f16(128, 64, 0, 0, 0), 1);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_ts(tmem + T_H, tmem + T_UA + 8 * k, kmajor_desc(sb + S_AK + 8192, 128, k),
                  idesc_f16(128, 128, 0, 0, 0), 1);
        umma_commit(bar_s3);
      }
      {
        const bool ok = mbar_wait(bar_s3, c & 1);
        if (!named_and(BAR_STATE, NSTATE, ok)) { alive = false; break; }
        tc_fence_after();
      }
      // outputs o[t][j] = O^T[j][t]
      if (!SPLIT || u.write_o) {
        const long rbase = u.row0 + (long)c * C;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t v[32];
          tmem_ld32<32>(tmem + lb + T_O + 32 * h2, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int t = 32 * h2 + e;
            const float x = __uint_as_float(v[e]);
            if (t < lenc) {
              go[(size_t)(rbase + t) * 128 + s] = __float2bfloat16_rn(x);
              fin = fmaf(x, 0.f, fin);
            }
          }
        }
      }
      tc_fence_before();
      named_sync(BAR_STATE, NSTATE);
      if (c + 1 < nchunks) {
        const bool ok = mbar_wait(bar_gc + ((c + 1) & 1), (uint32_t)(((c + 1) >> 1) & 1));
        if (!named_and(BAR_STATE, NSTATE, ok)) { alive = false; break; }
        convert_and_scale(c + 1, false);
        tc_fence_before();
        named_sync(BAR_STATE, NSTATE);
      }
    }
    if (alive && nchunks > 0 && hT) {
      for (int i0 = 0; i0 < DK; i0 += 32) {
        uint32_t v[32];
        tmem_ld32<32>(tmem + lb + T_H + i0, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float x = __uint_as_float(v[e]);
          hT[hoff + (size_t)(i0 + e) * 128 + s] = x;
          fin = fmaf(x, 0.f, fin);
        }
      }
    }
    ovf = !(fin == 0.f);
    if (!alive) *reinterpret_cast<volatile int*>(s_abort) = 1;
  } else {
    // ======================================================= INVERSE CHAIN
    // Warps 12-15 (one per TMEM lane quarter) finish chunk c after the prep
    // role has handed over E = D N: [E ; I - E] and its product with [E | D],
    // T = F + E^2 F, T Diag(beta) and W^T, each a tensor-core step issued by
    // lane 0 of warp 12 as soon as the warpgroup has written its operands.
    // Between those steps the same thread issues chunk c+1's Gram rounds and
    // E step as the prep role hands their operands over, and L2 prefetches;
    // warp 12 loads beta.
    const int tq = warp - MMA_WARP;            // TMEM lane quarter (= warp % 4)
    const int row = 32 * tq + lane;            // this thread's TMEM lane
    const uint32_t tl = (uint32_t)(32 * tq) << 16;
    const bool issuer = warp == MMA_WARP && lane == 0;
    bool alive = true;
    auto tail_wait = [&](uint64_t* bar, int cc, bool ok) -> bool {
      if (ok && cc >= 0) ok = mbar_wait(bar, (uint32_t)(cc & 1));
      const bool all = named_and(BAR_TAIL, NTAIL, ok);
      tc_fence_after();
      return all;
    };
    auto tail_publish = [&]() {
      fence_proxy_async_smem();
      tc_fence_before();
      named_sync(BAR_TAIL, NTAIL);
    };
    const uint32_t id64 = idesc_f16(128, 64, 0, 0, 0);
    auto prefetch_l2 = [&](int cc) {
      const int y = (int)(u.row0 + (long)cc * C);
#pragma unroll
      for (int x0 = 0; x0 < 128; x0 += 64) {
        if (x0 < DK) {
          tma_prefetch_2d_l2(&mq, x0, y);
          tma_prefetch_2d_l2(&mk, x0, y);
          tma_prefetch_2d_l2(&ma, x0, y);
        }
        if (!zero_v) tma_prefetch_2d_l2(&mv, x0, y);
      }
    };
    // beta of chunk cc, two tokens per lane of warp 12: fetched a chunk ahead
    // into registers (as raw bf16, so that nothing waits on the load before
    // the store), stored into its parity buffer once that is free; every
    // lane arrives (the barrier counts 32)
    const unsigned short* gbeta = static_cast<const unsigned short*>(a.beta);
    uint32_t braw0 = 0, braw1 = 0;
    auto fetch_beta = [&](int cc) {
      const int len = min(C, u.len - cc * C);
      const unsigned short* src = gbeta + u.row0 + (long)cc * C;
      braw0 = lane < len ? (uint32_t)src[lane] : 0u;
      braw1 = lane + 32 < len ? (uint32_t)src[lane + 32] : 0u;
    };
    auto store_beta = [&](int cc) {
      float* dst = reinterpret_cast<float*>(sm + S_BETA) + 64 * (cc & 1);
      uint32_t b0 = braw0, b1 = braw1;
      asm volatile("" : "+r"(b0), "+r"(b1));  // the first use is here, not earlier
      dst[lane] = __uint_as_float(b0 << 16);
      dst[lane + 32] = __uint_as_float(b1 << 16);
      mbar_arrive(bar_beta);
    };
    // Gram round: D (128 x 64) = X (128 rows) Y^T (64 rows), K = 128
    auto gram = [&](uint32_t d_col, uint32_t xbuf, uint32_t ybuf) {
      const uint64_t d_gx = kmajor_desc(sb + xbuf, 128, 0), d_gy = kmajor_desc(sb + ybuf, 64, 0);
#pragma unroll
      for (int k = 0; k < 8; ++k)  // K steps: 32 bytes in a panel, panels R*128 apart
        umma_ss(tmem + d_col, d_gx + (uint64_t)((k >> 2) * 1024 + (k & 3) * 2),
                d_gy + (uint64_t)((k >> 2) * 512 + (k & 3) * 2), id64, k > 0);
    };
    // issuer only: waits for the prep role's operands of step st of chunk cc
    auto wait_ops = [&](int st, int cc) -> bool {
      if (!mbar_wait(bar_ops + st, (uint32_t)(cc & 1))) return false;
      tc_fence_after();
      return true;
    };
    // issuer only: round 1 of chunk cc (buffer 2 -> G0)
    auto issue_r1 = [&](int cc) -> bool {
      if (!wait_ops(ST_R1, cc)) return false;
      gram(T_G0, S_GX2, S_GY2);
      umma_commit(bar_done + ST_R1);
      return true;
    };
    // issuer only: rounds 2 (buffer 2 -> G0, once round 1 has been read out;
    // D waits for it) and 3 (buffer 1 -> G1) of chunk cc, then its E step
    auto issue_rest = [&](int cc) -> bool {
      if (!wait_ops(ST_R2, cc)) return false;
      gram(T_G0, S_GX2, S_GY2);
      umma_commit(bar_done + ST_R2);
      if (!wait_ops(ST_R3, cc)) return false;
      gram(T_G1, S_GX, S_GY);
      umma_commit(bar_done + ST_R3);
      if (cc + 2 < nchunks) prefetch_l2(cc + 2);
      // E = D N (rows 0..63 of G1)
      if (!wait_ops(ST_E, cc)) return false;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        umma_ss(tmem + T_G1, kmajor_desc(sb + S_TD, 128, k), mnmajor_desc(sb + S_TN, 64, k),
                idesc_f16(128, 64, 0, 0, 1), k > 0);
      umma_commit(bar_done + ST_E);
      return true;
    };
    bool ok = true;                            // the issuer's waits so far
    if (nchunks > 0 && warp == MMA_WARP) {
      if (lane == 0) {
        issue_qka(0);
        if (!zero_v) {
          mbar_arrive_expect_tx(bar_v, TILE_BYTES);
          tma_load_2d(sm + S_V, &mv, bar_v, 0, (int)u.row0);
          tma_load_2d(sm + S_V + 8192, &mv, bar_v, 64, (int)u.row0);
        }
        if (nchunks > 1) prefetch_l2(1);
      }
      fetch_beta(0);
      store_beta(0);
      if (nchunks > 1) fetch_beta(1);
      if (lane == 0) {
        ok = issue_r1(0);
        if (ok) ok = issue_rest(0);
      }
      __syncwarp();
      // only once chunk 0's prep has passed its wait for beta: a second
      // completion before that would alias the phase it waits for
      if (nchunks > 1) store_beta(1);
    }
    for (int c = 0; c < nchunks && alive; ++c) {
      const int cn = c + 1;
      const bool nx = cn < nchunks;
      const float* beta_c = reinterpret_cast<const float*>(sm + S_BETA) + 64 * (c & 1);
      // chunk c+2's beta, stored once chunk c+1's prep has passed its wait
      if (warp == MMA_WARP && c + 2 < nchunks) fetch_beta(c + 2);
      // ---- E -> [E ; I - E] (rows t of two tiles): lanes 0..63
      if (!tail_wait(bar_done + ST_E, c, ok)) { alive = false; break; }
      if (tq < 2) {
        uint32_t v[64];
        tmem_ld32<32>(tmem + tl + T_G1, *reinterpret_cast<uint32_t(*)[32]>(v));
        tmem_ld32<32>(tmem + tl + T_G1 + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
        tmem_ld_wait();
#pragma unroll
        for (int z = 0; z < 64; z += 8) {
          float f[8], g[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            f[e] = __uint_as_float(v[z + e]);
            g[e] = ((z + e) == row ? 1.f : 0.f) - f[e];
          }
          store16(sm + S_TE + sw128_chunk(64, row, (uint32_t)z >> 3), pack_half8(f));
          store16(sm + S_TIE + sw128_chunk(64, row, (uint32_t)z >> 3), pack_half8(g));
        }
      }
      tail_publish();
      if (issuer) {
        // [E ; I - E] x [E | D]: E^2 in G0 rows 0..63, F = (I - E) D in G1
        // rows 64..127 (D is the second 64-wide panel of B)
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_ss(tmem + T_G0, kmajor_desc(sb + S_TE, 128, k),
                  sw128_desc(sb + S_TE + (uint32_t)k * 2048u, S_TD - S_TE, 1024u),
                  idesc_f16(128, 128, 0, 0, 1), k > 0);
        umma_commit(bar_done + ST_X);
      }
      // ---- E^2 (G0, lanes 0..63) and F (G1, lanes 64..127) as fp16
      if (!tail_wait(bar_done + ST_X, c, true)) { alive = false; break; }
      {
        const bool e2 = tq < 2;
        const int r = e2 ? row : row - 64;
        uint8_t* dst = sm + (e2 ? S_TIE : S_TE);
        uint32_t v[64];
        tmem_ld32<32>(tmem + tl + (e2 ? T_G0 : T_G1), *reinterpret_cast<uint32_t(*)[32]>(v));
        tmem_ld32<32>(tmem + tl + (e2 ? T_G0 : T_G1) + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
        tmem_ld_wait();
#pragma unroll
        for (int z = 0; z < 64; z += 8) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(v[z + e]);
          store16(dst + sw128_chunk(64, r, (uint32_t)z >> 3), pack_half8(f));
        }
      }
      tail_publish();
      if (issuer) {
        // T = F + E^2 F in G1 rows 64..127 (A rows 64..127 = E^2, B = F)
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_ss(tmem + T_G1, kmajor_desc(sb + S_TE, 128, k), mnmajor_desc(sb + S_TE, 64, k),
                  idesc_f16(128, 64, 0, 0, 1), 1);
        umma_commit(bar_done + ST_T);
        // round 1 of chunk cn (G0 is free: E^2 has been read)
        if (nx) ok = issue_r1(cn);
      }
      // ---- T Diag(beta) as bf16 (T is in G1, lanes 64..127; its upper
      // triangle is exactly zero), once the previous chunk's U~ step has read
      // the last one
      if (!tail_wait(bar_done + ST_T, c, ok)) { alive = false; break; }
      if (!tail_wait(bar_s1, c - 1, true)) { alive = false; break; }
      if (tq >= 2) {
        const int r = row - 64;
        uint32_t v[64];
        tmem_ld32<32>(tmem + tl + T_G1, *reinterpret_cast<uint32_t(*)[32]>(v));
        tmem_ld32<32>(tmem + tl + T_G1 + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
        tmem_ld_wait();
#pragma unroll
        for (int z = 0; z < 64; z += 8) {
          const float4 b0 = *reinterpret_cast<const float4*>(beta_c + z);
          const float4 b1 = *reinterpret_cast<const float4*>(beta_c + z + 4);
          const float f[8] = {__uint_as_float(v[z]) * b0.x, __uint_as_float(v[z + 1]) * b0.y,
                              __uint_as_float(v[z + 2]) * b0.z, __uint_as_float(v[z + 3]) * b0.w,
                              __uint_as_float(v[z + 4]) * b1.x, __uint_as_float(v[z + 5]) * b1.y,
                              __uint_as_float(v[z + 6]) * b1.z, __uint_as_float(v[z + 7]) * b1.w};
          store16(sm + S_TB + sw128_chunk(64, r, (uint32_t)z >> 3), pack_bf8(f));
        }
      }
      tail_publish();
      if (issuer) {
        // W^T = (k*gamma)^T TB^T in G1 (lane = i)
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_ss(tmem + T_G1, mnmajor_desc(sb + S_KG, 64, k), kmajor_desc(sb + S_TB, 64, k),
                  idesc_f16(128, 64, 1, 1, 0), k > 0);
        umma_commit(bar_done + ST_W);
      }
      // ---- -W^T (fp16, panel 0 of [-W^T | (q*gamma)^T]; W^T is in G1,
      // lane = i); then chunk c is ready for the state step (with the prep
      // role's part)
      if (!tail_wait(bar_done + ST_W, c, true)) { alive = false; break; }
      {
        uint32_t v[64];
        tmem_ld32<32>(tmem + tl + T_G1, *reinterpret_cast<uint32_t(*)[32]>(v));
        tmem_ld32<32>(tmem + tl + T_G1 + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
        tmem_ld_wait();
#pragma unroll
        for (int z = 0; z < 64; z += 8) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = -__uint_as_float(v[z + e]);
          store16(sm + S_WQ + sw128_chunk(64, row, (uint32_t)z >> 3), pack_half8(f));
        }
      }
      tail_publish();
      if (warp == MMA_WARP) {
        if (lane == 0) {
          mbar_arrive(bar_ready + (c & 1));
          if (nx) ok = issue_rest(cn);     // G1 is free: W^T has been read
        }
        __syncwarp();
        // chunk c+2's beta buffer was last read by this chunk's T Diag(beta),
        // and chunk c+1's prep has passed its wait for its own (a later
        // completion of the barrier would alias that phase)
        if (c + 2 < nchunks) store_beta(c + 2);
      }
    }
    if (!alive || !ok) *reinterpret_cast<volatile int*>(s_abort) = 1;
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  const int any_ovf = __syncthreads_or(ovf ? 1 : 0);
  if (tid == 0) {
    if (any_ovf) set_status(a.status, CKDA_ERR_RANGE);
    if (*reinterpret_cast<volatile int*>(s_abort)) {
      set_status(a.status, CKDA_ERR_TIMEOUT);
      // let any MMA or copy still in flight land before the memory is released
      for (int i = 0; i < ST_COUNT; ++i) mbar_wait(bar_done + i, 0, 1u << 12, 1000u);
      mbar_wait(bar_s1, 0, 1u << 12, 1000u);
      mbar_wait(bar_s3, 0, 1u << 12, 1000u);
      if (!zero_v) mbar_wait(bar_v, 0, 1u << 12, 1000u);
      mbar_wait(bar_qka, 0, 1u << 12, 1000u);
    }
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------ host side
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t width) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t gdim[2] = {width, rows};
  cuuint64_t gstride[1] = {width * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

cudaError_t launch_fwd_chunk(const FwdArgs& a, cudaStream_t s) {
  const int units = a.num_units_seq * a.H;
  if (units == 0) return cudaSuccess;
  const uint64_t rows = (uint64_t)a.B * a.H * a.T;
  CUtensorMap mq, mk, ma, mv;
  if (rows == 0) {
    mq = mk = ma = mv = CUtensorMap{};  // every sequence is empty: no tile is ever loaded
  } else if (!make_map(&mq, a.q, rows, a.dk) || !make_map(&mk, a.k, rows, a.dk) ||
             !make_map(&ma, a.alpha, rows, a.dk) || !make_map(&mv, a.v, rows, 128)) {
    return cudaErrorInvalidValue;
  }
  auto kern = a.split_pass ? (a.dk == 64 ? fwd_chunk_kernel<64, true> : fwd_chunk_kernel<128, true>)
                           : (a.dk == 64 ? fwd_chunk_kernel<64, false> : fwd_chunk_kernel<128, false>);
  const long long grid =
      a.split_pass ? (long long)a.B * a.H * split_ctas_per_unit(a.split_pass, a.nseg) : units;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
  if (err != cudaSuccess) return err;
  kern<<<(unsigned)grid, NT, SMEM_ALLOC, s>>>(a, mq, mk, ma, mv);
  return cudaGetLastError();
}

}  // namespace ckda
