// chunk_tc.cu -- fused chunked forward of delta-rule attention on the 5th-
// generation tensor cores (tcgen05 + TMEM + TMA), bf16 I/O, dk = dv = 128,
// chunk C = 64, any n_h (Gated DeltaProduct), gated or not.
//
// The algorithm is the chunkwise form of "08 · linear 路线（三）：delta rule 与
// DPLR 统一框架" -- the UT transform of §2.2, the state passing of §2.3 and
// the gated variant of §3 -- run on the extended sequence of "DeltaProduct：
// 通过 Householder 乘积增强线性 RNN 的状态追踪" §4.1.  Per chunk of 64 rows:
//
//   gc   = inclusive cumsum of the log gate (log g_t at each token's first
//          sub-step, 0 elsewhere; clamped at -80 so g = 0 stays finite)
//   A    = strictLower(diag(beta) (Gam * K K^T)),  Gam_ij = exp(gc_i - gc_j)
//   T    = (I + A)^{-1} diag(beta)
//   W    = T (K * exp(gc)),  U = T V
//   O    = (Q * exp(gc)) S + P (U - W S),   P = Q K^T * Gam * M (M incl. diag)
//   S   <- exp(gc_C) S + Kd^T (U - W S),    Kd = K * exp(gc_C - gc)
//
// Everything that does not involve the state is folded into two per-chunk
// matrices, so that the sequential state chain is ONE tensor-core product:
//
//   M - I = (exp(gc_C) - 1) I - Kd^T W          (dk x dk)
//   Q'    = Q * exp(gc) - P W                    (readout rows x dk)
//   S    <- S + (M - I) S + Kd^T U               (the chain)
//   O     = Q' S + P U
//
// This is an exact rewrite of the same chunk step (the state enters both
// products once, as in U - W S).  All products are computed TRANSPOSED, so
// that every tensor-core product has M = 128 (a d axis) and the state S^T
// lives in TMEM as an fp32 accumulator [dv lanes x dk columns]:
//
//   G     = [K; Q] K^T                  SS  N=64  K=128  (-> A, P)
//   W^T   = K^T (T diag exp gc)^T       SS  N=64  K=64
//   U^T   = V^T T^T                     SS  N=64  K=64
//   (M-I)^T = -W^T Kd                   TS  N=128 K=64   (A = W^T bf16 in TMEM)
//   Q'^T  = -W^T P^T (+ exp(gc) Q^T)    TS  N=64  K=64
//   O^T   = U^T P^T + S^T Q'^T          TS  N=64  K=64 + K=128
//   S^T  += S^T (M-I)^T + U^T Kd        TS  N=128 K=128 + K=64   (chain)
//
// W, U, T, M, Q' and P never leave the SM.  HBM traffic is q, k, v, beta, g
// in and out, h0/hT once per head.
//
// Warp roles (448 threads ungated, 480 gated; one CTA per (b, h) head):
//   warp 0       TMA producer: K/Q/V tiles (128-byte swizzle, 3 stages, the
//                chunk after them prefetched into L2) + beta / log-gate rows
//   warp 1       TMEM owner and MMA issuer (gated: the state-recurrence
//                products; warp 14 issues the look-ahead W, U, G products)
//   warps 2-5    prep (chunk n+2): G -> A, P -> UT solve -> T tiles
//   warps 6-9    feed-forward (chunk n+1): W^T, U^T -> bf16 TMEM operands,
//                Kd, (M-I)^T -> smem operand
//   warps 10-13  chain (chunk n): S^T -> bf16 operand, the outputs (staged
//                through the V slot by transposing 8x8 stores), hT; then Q'
//                of chunk n+1 -> smem operand, in the same fragment layout
// Every mbarrier wait is bounded; a timeout sets a device error word and the
// kernel winds down instead of hanging.
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm100.cuh"
#include "tma_host.h"

namespace delta {

// Set by the tensor-core kernel when a bounded wait gives up (1 + role id).
__device__ unsigned int g_tc_error = 0;

namespace {
using namespace sm100;

constexpr int C = 64;
constexpr int D = 128;
constexpr int NS = 3;  // TMA stages
// Gated, a second MMA-issuing warp (14) takes the look-ahead products; the
// ungated step keeps one issuer and its priority order (measured faster)
__host__ __device__ constexpr bool dual_issue(bool gated) { return gated; }
__host__ __device__ constexpr bool look_wu(bool gated) { return true; }  // W, U on warp 14
__host__ __device__ constexpr bool look_g(bool gated) { return true; }   // G on warp 14
__host__ __device__ constexpr int threads_for(bool gated) { return dual_issue(gated) ? 480 : 448; }
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLogGateFloor = -80.0f;
// Down to this cumulative log2 gate within a chunk the decay factors are
// formed as 2^gc_i * 2^-gc_j (no overflow); below it, exactly per entry.
constexpr float kRatioFloor = -100.0f;

// ---- shared memory layout (offsets from a 1024-byte aligned base) ----
constexpr uint32_t STAGE_BYTES = 49152;
constexpr uint32_t ST_K0 = 0, ST_Q0 = 8192, ST_K1 = 16384, ST_Q1 = 24576;
constexpr uint32_t ST_V0 = 32768;  // V (64 x 128), later Kd, same layout
constexpr uint32_t OFF_MS = NS * STAGE_BYTES;  // (M-I)^T bf16 [128 j][128 i], MN-major B
constexpr uint32_t OFF_TU = OFF_MS + 32768;    // T bf16 [64][64], K-major
constexpr uint32_t OFF_TW = OFF_TU + 8192;     // T diag(exp gc)
constexpr uint32_t OFF_P = OFF_TW + 8192;      // 2 x P bf16 [64][64], K-major
constexpr uint32_t OFF_AX = OFF_P + 16384;     // A (upper, transposed) / X (lower) fp32 [64][64]
constexpr uint32_t OFF_SM = OFF_AX + 16384;    // small arrays and barriers
constexpr uint32_t SM_BETA = 0;                // [NS][64]
constexpr uint32_t SM_LAM = SM_BETA + NS * 256;  // [NS][64] log2 gate
constexpr uint32_t SM_EG = SM_LAM + NS * 256;    // prep: 2^gc
constexpr uint32_t SM_IEG = SM_EG + 256;         // prep: 2^-gc
constexpr uint32_t SM_BGC = SM_IEG + 256;        // prep: beta 2^gc
constexpr uint32_t SM_DEC = SM_BGC + 256;        // feed-forward: 2^(gc_C - gc)
constexpr uint32_t SM_GQ = SM_DEC + 256;         // feed-forward: 2^gc at readout rows
constexpr uint32_t SM_BAR = SM_GQ + 256;

// ---- barrier indices ----
enum {
  B_FULL = 0,        // [NS] producer -> all: K, Q tiles, beta, log gate loaded (count 2 + tx)
  B_EMPTY = NS,      // [NS] MMA -> producer: K, Q tiles of the stage consumed
  B_GFULL = 2 * NS,  // MMA -> prep: G in TMEM
  B_GFREE,           // prep -> MMA: G read (one arrival per warp)
  B_TFULL,           // prep -> MMA: T tiles and P written (per warp)
  B_WFULL,           // MMA -> ff, prep: W^T, U^T in TMEM (T tiles consumed)
  B_CWD,             // ff -> MMA: W^T, U^T bf16 in TMEM, Kd in smem (per warp)
  B_MFULL,           // MMA -> ff: (M-I)^T in TMEM
  B_MRDY,            // ff -> MMA: (M-I)^T in smem, TMEM free (per warp)
  B_QFULL,           // MMA -> ff: -W^T P^T in TMEM
  B_QRDY,            // ff -> MMA: Q' in smem, TMEM free (per warp)
  B_SRDY,            // chain -> MMA: S^T bf16 in TMEM (per warp)
  B_SFULL,           // MMA -> chain, ff: state step done
  B_OFULL,           // MMA -> chain: O^T in TMEM
  B_OFREE,           // chain -> MMA: O^T read (per warp)
  B_PFREE0,          // MMA -> prep: P buffer 0 consumed
  B_PFREE1,          //                        1
  B_DRAIN,           // MMA: everything issued has completed
  B_VFULL,           // [NS] producer -> MMA: the V tile of a stage loaded (count 1 + tx)
  B_VEMPTY = B_VFULL + NS,  // [NS] chain -> producer: V slot free (per warp; it stages the outputs)
  NBARS = B_VEMPTY + NS
};
constexpr uint32_t SM_MISC = SM_BAR + NBARS * 8;  // tmem slot, abort flag, gate of the chunk
constexpr uint32_t SMEM_TOTAL = OFF_SM + SM_MISC + 16;
constexpr uint32_t SMEM_ALLOC = 232448;
static_assert(SMEM_TOTAL <= SMEM_ALLOC, "shared memory budget");

// ---- TMEM columns ----
constexpr uint32_t TM_S = 0;      // S^T fp32 [dv][dk]                128
constexpr uint32_t TM_SBF = 128;  // S^T bf16 (packed)                 64
constexpr uint32_t TM_O = 192;    // -W^T P^T, then O^T fp32           64
constexpr uint32_t TM_X1 = 256;   // W^T | U^T fp32, then (M-I)^T     128
constexpr uint32_t TM_G = 384;    // G fp32                            64
constexpr uint32_t TM_WB = 448;   // W^T bf16 (packed)                 32
constexpr uint32_t TM_UB = 480;   // U^T bf16 (packed)                 32
constexpr uint32_t TM_COLS = 512;

struct TcParams {
  const float *beta, *g, *h0;
  __nv_bfloat16 *out;
  float *hT;
  int H, T, L, n_h, nchunks;
};

struct Smem {
  uint8_t *base;
  __device__ uint8_t *stage(int s) const { return base + s * STAGE_BYTES; }
  __device__ float *arr(uint32_t off) const { return reinterpret_cast<float *>(base + OFF_SM + off); }
  __device__ float *beta(int s) const { return arr(SM_BETA + s * 256); }
  __device__ float *lam(int s) const { return arr(SM_LAM + s * 256); }
  __device__ uint64_t *bar(int i) const {
    return reinterpret_cast<uint64_t *>(base + OFF_SM + SM_BAR) + i;
  }
  __device__ uint32_t *tmem_slot() const { return reinterpret_cast<uint32_t *>(base + OFF_SM + SM_MISC); }
  __device__ volatile int *abort_flag() const {
    return reinterpret_cast<volatile int *>(base + OFF_SM + SM_MISC + 4);
  }
  __device__ float *gate_c() const { return reinterpret_cast<float *>(base + OFF_SM + SM_MISC + 8); }
  // set when a drain wait ran out: TMEM is then not freed at exit
  __device__ volatile int *keep_tmem() const {
    return reinterpret_cast<volatile int *>(base + OFF_SM + SM_MISC + 12);
  }
  __device__ float *AX() const { return reinterpret_cast<float *>(base + OFF_AX); }
};

// Bounded wait that also gives up at once when another role has aborted.
// The first poll is inline; the loop stays out of line (it is called from
// many places) and takes only scalars, so nothing goes through local memory.
__device__ __noinline__ bool wait_bar_slow(uint8_t *base, int idx, uint32_t parity, int role) {
  Smem sm;
  sm.base = base;
  uint64_t *b = sm.bar(idx);
  for (uint32_t i = 0; i < (1u << 22); ++i) {
    if (mbar_try_wait(b, parity)) return true;
    if ((i & 63) == 63 && *sm.abort_flag()) return false;
  }
  *sm.abort_flag() = 1;
  atomicCAS(&g_tc_error, 0u, (unsigned)(1 + role) | ((unsigned)idx << 8));
  return false;
}
__device__ __forceinline__ bool wait_bar(const Smem &sm, int idx, uint32_t parity, int role) {
  if (mbar_try_wait(sm.bar(idx), parity)) return true;
  return wait_bar_slow(sm.base, idx, parity, role);
}

// Wait for the completion of TMA copies or tensor-core products that were
// already issued.  They complete on their own, so this wait does NOT give up
// when another role has aborted (shared memory and TMEM must not be released
// under them); it is still bounded.  If it runs out, the error word records
// it and the CTA keeps its TMEM columns at exit instead of freeing them
// under work that may still be writing them.
__device__ __noinline__ bool wait_bar_drain(uint8_t *base, int idx, uint32_t parity, int role) {
  Smem sm;
  sm.base = base;
  uint64_t *b = sm.bar(idx);
  for (uint32_t i = 0; i < (1u << 24); ++i)
    if (mbar_try_wait(b, parity)) return true;
  *sm.abort_flag() = 1;
  *sm.keep_tmem() = 1;
  atomicCAS(&g_tc_error, 0u, (unsigned)(1 + role) | ((unsigned)idx << 8));
  return false;
}

// fp32 64x64 matrices in shared memory are stored row-major with the column
// XOR-swizzled by the row (bits 2..4), which keeps float4 runs along a row
// contiguous and makes the tf32 MMA fragment loads below conflict-free.
__device__ __forceinline__ int swz(int r, int c) { return r * 64 + (c ^ ((r & 7) << 2)); }

// The solve's 64x64 array holds A_ij (i > j) at (j, i) -- the upper triangle --
// and X_ij = ((I + A)^{-1})_ij (i > j) at (i, j) -- the lower triangle.  The
// diagonal holds the chunk's cumulative log gate (X_ii = 1 is implicit).
__device__ __forceinline__ float ldA(const float *AX, int i, int j) { return AX[swz(j, i)]; }
// X_rc of a block that touches the diagonal: 1 on it, 0 above it.
__device__ __forceinline__ float ldXm(const float *M, int r, int c) {
  const float v = M[swz(r, c)];
  return r > c ? v : (r == c ? 1.f : 0.f);
}

// D(16x8) += A(16x8) B(8x8) on the warp-level tensor-core path, tf32 inputs
// (fp32 bit patterns; the MMA ignores the low mantissa bits).
// Fragments: a = {A[g][t], A[g+8][t], A[g][t+4], A[g+8][t+4]},
// b = {B[t][g], B[t+4][g]}, d = {D[g][2t], D[g][2t+1], D[g+8][2t], D[g+8][2t+1]}
// with g = lane / 4, t = lane % 4.
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Operand fragments of the tf32 MMA read from the solve array.  KIND 0: a
// block of A (stored transposed in the upper triangle); KIND 1: a block of X
// that may touch the diagonal (1 on it, 0 above it).
template <int KIND>
__device__ __forceinline__ uint32_t lsol(const float *AX, int r, int c) {
  return __float_as_uint(KIND == 0 ? ldA(AX, r, c) : ldXm(AX, r, c));
}
template <int KIND>
__device__ __forceinline__ void frag_a(uint32_t (&a)[4], const float *AX, int r0, int k0, int lane) {
  const int g = lane >> 2, t = lane & 3;
  a[0] = lsol<KIND>(AX, r0 + g, k0 + t);
  a[1] = lsol<KIND>(AX, r0 + g + 8, k0 + t);
  a[2] = lsol<KIND>(AX, r0 + g, k0 + t + 4);
  a[3] = lsol<KIND>(AX, r0 + g + 8, k0 + t + 4);
}
template <int KIND>
__device__ __forceinline__ void frag_b(uint32_t (&b)[2], const float *AX, int k0, int n0, int lane) {
  const int g = lane >> 2, t = lane & 3;
  b[0] = lsol<KIND>(AX, k0 + t, n0 + g);
  b[1] = lsol<KIND>(AX, k0 + t + 4, n0 + g);
}
// B fragment for k-step ks (rows 8 ks .. 8 ks + 7) of a matrix Y held as MMA
// results: y[h] is the 16x8 accumulator of rows 16 h .. 16 h + 15.  Row r,
// column c of a 16x8 accumulator lives in lane (r % 8) * 4 + c / 2, element
// (r / 8) * 2 + c % 2: two candidates are shuffled in and one is kept.
template <int NH>
__device__ __forceinline__ void frag_b_acc(uint32_t (&b)[2], const float (&y)[NH][4], int ks,
                                           int lane) {
  const int g = lane >> 2, t = lane & 3, h = ks >> 1, e = (ks & 1) * 2;
  const int s0 = t * 4 + (g >> 1), s1 = (t + 4) * 4 + (g >> 1);
  const float a0 = __shfl_sync(0xffffffffu, y[h][e], s0);
  const float a1 = __shfl_sync(0xffffffffu, y[h][e + 1], s0);
  const float c0 = __shfl_sync(0xffffffffu, y[h][e], s1);
  const float c1 = __shfl_sync(0xffffffffu, y[h][e + 1], s1);
  b[0] = __float_as_uint((g & 1) ? a1 : a0);
  b[1] = __float_as_uint((g & 1) ? c1 : c0);
}

// T_U[r][c] = x beta_c and T_W[r][c] = x beta_c exp(gc_c) (bf16 tiles).
__device__ __forceinline__ void put_t(uint8_t *tu, uint8_t *tw, int r, int c, float x, float bc,
                                      float wc) {
  const uint32_t off = sw128_offset(r, c, 64);
  *reinterpret_cast<__nv_bfloat16 *>(tu + off) = __float2bfloat16_rn(x * bc);
  *reinterpret_cast<__nv_bfloat16 *>(tw + off) = __float2bfloat16_rn(x * wc);
}

// T tiles from a 16x8 fragment of (scale * D) at rows r0.., columns n0...
__device__ __forceinline__ void frag_to_t(uint8_t *tu, uint8_t *tw, int r0, int n0,
                                          const float (&d)[4], float scale, const float *beta,
                                          const float *bgc, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const int c = n0 + 2 * t;
  const float b0 = beta[c], b1 = beta[c + 1], w0 = bgc[c], w1 = bgc[c + 1];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const float x0 = d[2 * hh] * scale, x1 = d[2 * hh + 1] * scale;
    const int r = r0 + g + 8 * hh;
    *reinterpret_cast<uint32_t *>(tu + sw128_offset(r, c, 64)) = pack_bf16(x0 * b0, x1 * b1);
    *reinterpret_cast<uint32_t *>(tw + sw128_offset(r, c, 64)) = pack_bf16(x0 * w0, x1 * w1);
  }
}

// Store a 16x8 fragment (scaled) into swizzled fp32 smem at (r0, n0).
__device__ __forceinline__ void warp_store_16x8(float *M, int r0, int n0, const float (&d)[4],
                                                float scale, int lane) {
  const int g = lane >> 2, t = lane & 3;
  M[swz(r0 + g, n0 + 2 * t)] = d[0] * scale;
  M[swz(r0 + g, n0 + 2 * t + 1)] = d[1] * scale;
  M[swz(r0 + g + 8, n0 + 2 * t)] = d[2] * scale;
  M[swz(r0 + g + 8, n0 + 2 * t + 1)] = d[3] * scale;
}

// One warp inverts the unit lower-triangular 16x16 diagonal block at offset
// o of (I + A): closed-form 4x4 leaves, then the merges 4 -> 8 -> 16, each
// X21 = -X22 (A21 X11).  Every entry of A the warp needs is loaded at once;
// the partial inverses move between lanes by shuffles, not through shared
// memory.  X goes to the lower triangle of the solve array and, scaled, to
// the T tiles.
__device__ __forceinline__ void invert_diag16(float *AX, uint8_t *tu, uint8_t *tw,
                                              const float *beta, const float *bgc, int o,
                                              int lane) {
  const unsigned full = 0xffffffffu;
  // leaf lanes (0..11): leaf a, column cc;  merge-1 lanes: (hh, r4, c4);
  // merge-2 lanes: (r8, c0 and c0 + 4)
  const int a = lane < 12 ? lane / 3 : 0, cc = lane < 12 ? lane - 3 * (lane / 3) : 0;
  const int b0 = o + 4 * a;
  const int hh = lane >> 4, r4 = (lane >> 2) & 3, c4 = lane & 3, o8 = o + 8 * hh;
  const int r8 = lane >> 2, c0 = lane & 3;
  const float a10 = ldA(AX, b0 + 1, b0), a20 = ldA(AX, b0 + 2, b0), a21 = ldA(AX, b0 + 2, b0 + 1);
  const float a30 = ldA(AX, b0 + 3, b0), a31 = ldA(AX, b0 + 3, b0 + 1), a32 = ldA(AX, b0 + 3, b0 + 2);
  float am1[4], am2[8];
#pragma unroll
  for (int m = 0; m < 4; ++m) am1[m] = ldA(AX, o8 + 4 + r4, o8 + m);
#pragma unroll
  for (int m = 0; m < 8; ++m) am2[m] = ldA(AX, o + 8 + r8, o + m);

  // ---- leaves: column cc of leaf a by forward substitution ----
  const float x0 = cc == 0 ? 1.f : 0.f;
  const float x1 = cc == 1 ? 1.f : (cc < 1 ? -(a10 * x0) : 0.f);
  const float x2 = cc == 2 ? 1.f : (cc < 2 ? -fmaf(a21, x1, a20 * x0) : 0.f);
  const float x3 = -fmaf(a32, x2, fmaf(a31, x1, a30 * x0));
  if (lane < 12) {
    const int col = b0 + cc;
    const float bc = beta[col], wc = bgc[col];
    if (cc < 1) {
      AX[swz(b0 + 1, col)] = x1;
      put_t(tu, tw, b0 + 1, col, x1, bc, wc);
    }
    if (cc < 2) {
      AX[swz(b0 + 2, col)] = x2;
      put_t(tu, tw, b0 + 2, col, x2, bc, wc);
    }
    AX[swz(b0 + 3, col)] = x3;
    put_t(tu, tw, b0 + 3, col, x3, bc, wc);
  }
  if (lane < 16) put_t(tu, tw, o + lane, o + lane, 1.f, beta[o + lane], bgc[o + lane]);

  // ---- 4 -> 8: X[o8+4+r4][o8+c4] ----
  float xm1;
  {
    // X11 = leaf 2 hh, column c4 (lane 6 hh + c4); X11[m][c4] for m > c4
    const int s11 = 6 * hh + c4;
    const float u1 = __shfl_sync(full, x1, s11), u2 = __shfl_sync(full, x2, s11),
                u3 = __shfl_sync(full, x3, s11);
    const float xc[4] = {c4 == 0 ? 1.f : 0.f, c4 == 1 ? 1.f : (c4 < 1 ? u1 : 0.f),
                         c4 == 2 ? 1.f : (c4 < 2 ? u2 : 0.f), c4 == 3 ? 1.f : u3};
    float y = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) y = fmaf(am1[m], xc[m], y);
    // Y[m][c4] from lane (hh, m, c4); X22[r4][m] = leaf 2 hh + 1, column m, row r4
    float z = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float ym = __shfl_sync(full, y, (lane & 16) | (m << 2) | c4);
      float xr = 1.f;
      if (m < 3) {
        const int s22 = 6 * hh + 3 + m;
        const float w1 = __shfl_sync(full, x1, s22), w2 = __shfl_sync(full, x2, s22),
                    w3 = __shfl_sync(full, x3, s22);
        xr = r4 == 1 ? w1 : (r4 == 2 ? w2 : w3);
      }
      if (m < r4) z = fmaf(xr, ym, z);
      if (m == r4) z += ym;
    }
    xm1 = -z;
    AX[swz(o8 + 4 + r4, o8 + c4)] = xm1;
    put_t(tu, tw, o8 + 4 + r4, o8 + c4, xm1, beta[o8 + c4], bgc[o8 + c4]);
  }

  // ---- 8 -> 16: X[o+8+r8][o+c0] and X[o+8+r8][o+c0+4] ----
  {
    // column c0 of X11 = X[o..o+8][o..o+8]: rows < 4 from leaf 0 (lane c0),
    // rows >= 4 from the 4 -> 8 merge (lane (0, m-4, c0))
    const float u1 = __shfl_sync(full, x1, c0), u2 = __shfl_sync(full, x2, c0),
                u3 = __shfl_sync(full, x3, c0);
    // column c0 + 4: rows >= 4 from leaf 1 (lane 3 + c0)
    const float v1 = __shfl_sync(full, x1, 3 + c0), v2 = __shfl_sync(full, x2, 3 + c0),
                v3 = __shfl_sync(full, x3, 3 + c0);
    float y0 = 0.f, y1 = 0.f;
    const float lo[4] = {c0 == 0 ? 1.f : 0.f, c0 == 1 ? 1.f : (c0 < 1 ? u1 : 0.f),
                         c0 == 2 ? 1.f : (c0 < 2 ? u2 : 0.f), c0 == 3 ? 1.f : u3};
    const float hi[4] = {c0 == 0 ? 1.f : 0.f, c0 == 1 ? 1.f : (c0 < 1 ? v1 : 0.f),
                         c0 == 2 ? 1.f : (c0 < 2 ? v2 : 0.f), c0 == 3 ? 1.f : v3};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      y0 = fmaf(am2[m], lo[m], y0);
      const float wm = __shfl_sync(full, xm1, (m << 2) | c0);
      y0 = fmaf(am2[m + 4], wm, y0);
      y1 = fmaf(am2[m + 4], hi[m], y1);
    }
    // X22 = X[o+8..o+16][o+8..o+16]: rows < 4 from leaf 2, rows >= 4 from
    // leaf 3 (same columns) or, for columns < 4, from the 4 -> 8 merge (hh 1)
    float z0 = 0.f, z1 = 0.f;
    const int rr = r8 & 3;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float ya = __shfl_sync(full, y0, (m << 2) | c0);
      const float yb = __shfl_sync(full, y1, (m << 2) | c0);
      float xr;
      if ((m & 3) < 3) {
        // leaf 2 (r8 < 4) or leaf 3 (r8 >= 4), column m & 3, row r8 & 3
        const int sl = (r8 < 4 ? 6 : 9) + (m & 3);
        const float w1 = __shfl_sync(full, x1, sl), w2 = __shfl_sync(full, x2, sl),
                    w3 = __shfl_sync(full, x3, sl);
        xr = rr == 1 ? w1 : (rr == 2 ? w2 : w3);
      } else {
        xr = 0.f;
      }
      if (m < 4) {
        const float xq = __shfl_sync(full, xm1, 16 | ((r8 & 3) << 2) | m);
        if (r8 >= 4) xr = xq;
      }
      if (m < r8) {
        z0 = fmaf(xr, ya, z0);
        z1 = fmaf(xr, yb, z1);
      }
      if (m == r8) {
        z0 += ya;
        z1 += yb;
      }
    }
    AX[swz(o + 8 + r8, o + c0)] = -z0;
    AX[swz(o + 8 + r8, o + c0 + 4)] = -z1;
    put_t(tu, tw, o + 8 + r8, o + c0, -z0, beta[o + c0], bgc[o + c0]);
    put_t(tu, tw, o + 8 + r8, o + c0 + 4, -z1, beta[o + c0 + 4], bgc[o + c0 + 4]);
  }
}

// 2^x on the MUFU unit (relative error ~2^-22; flushes to 0 far below 1)
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_sync(int id) {
  asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}

// Named barrier over 128 threads that also ORs `cond` across them, so that
// every participant takes the same decision (used to leave a loop together
// once any role has aborted).
__device__ __forceinline__ bool named_sync_or(int id, bool cond) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %2, 0;\n\t"
      "bar.red.or.pred q, %1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(id), "r"((uint32_t)cond)
      : "memory");
  return r != 0;
}

// One arrival per warp once every lane's prior work (fenced by the caller) is
// done: the warp converges, then lane 0 arrives.
__device__ __forceinline__ void arrive_warp(uint64_t *bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// Inclusive prefix sum over the 64 log-gate entries of a chunk, per warp:
// lane holds entries lane and lane + 32.
__device__ __forceinline__ void warp_scan64(const float *lam, int lane, float &lo, float &hi) {
  lo = lam[lane];
  hi = lam[lane + 32];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float a = __shfl_up_sync(0xffffffffu, lo, o);
    const float c = __shfl_up_sync(0xffffffffu, hi, o);
    if (lane >= o) {
      lo += a;
      hi += c;
    }
  }
  hi += __shfl_sync(0xffffffffu, lo, 31);
}

// 16-byte shared-memory load at a 32-bit shared address
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void st_chunk(uint8_t *p, const uint32_t (&v)[4]) {
  *reinterpret_cast<uint4 *>(p) = make_uint4(v[0], v[1], v[2], v[3]);
}

// readout rows of chunk n: tokens t_lo .. t_lo + Cp - 1 (their last sub-step
// falls in the chunk); row r reads out after extended step pos(r)
struct Rows {
  int e0, t_lo, Cp;
  __device__ Rows(int n, int n_h, int T) {
    e0 = n * C;
    t_lo = e0 / n_h;
    int t_hi = (e0 + C - n_h) / n_h;
    if (t_hi > T - 1) t_hi = T - 1;
    Cp = t_hi - t_lo + 1;
  }
  __device__ int pos(int r, int n_h) const { return (t_lo + r) * n_h + (n_h - 1) - e0; }
};

// 14 warps: at most 4 per SM sub-partition, so 128 registers per thread
template <bool GATED>
__global__ void __launch_bounds__(threads_for(GATED), 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem sm;
  // pointer arithmetic on the shared array (not integer casts) keeps every
  // access below in the shared state space
  sm.base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __builtin_assume(__isShared(sm.base));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the layout needs SMEM_TOTAL bytes after the 1024-byte alignment
  if ((uint32_t)(sm.base - smem_raw) + SMEM_TOTAL > SMEM_ALLOC) {
    if (tid == 0) atomicCAS(&g_tc_error, 0u, 0xFFu);
    return;
  }
  const int bh = blockIdx.x;
  const int b = bh / p.H, h = bh % p.H;
  const int n_h = p.n_h, NT = p.nchunks;
  const int QR = n_h == 1 ? 64 : 32;  // query rows loaded per chunk

  // ---- set-up: zero shared memory, init barriers, allocate TMEM ----
  {
    uint4 *z = reinterpret_cast<uint4 *>(sm.base);
    for (uint32_t i = tid; i < SMEM_TOTAL / 16; i += threads_for(GATED)) z[i] = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(sm.bar(B_FULL + s), 2);
      mbar_init(sm.bar(B_EMPTY + s), 1);
      mbar_init(sm.bar(B_VEMPTY + s), 4);
    }
    const int cnt[B_VFULL - 2 * NS] = {1, 4, 4, 1, 4, 1, 4, 1, 4, 4, 1, 1, 4, 1, 1, dual_issue(GATED) ? 2 : 1};
    for (int i = 2 * NS; i < B_VFULL; ++i) mbar_init(sm.bar(i), cnt[i - 2 * NS]);
    for (int s = 0; s < NS; ++s) mbar_init(sm.bar(B_VFULL + s), 1);
    *sm.abort_flag() = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sm.tmem_slot(), TM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_q);
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot();

  if (warp == 0) {
    // ===================================================== TMA producer
    // beta and the log gate of a chunk are read from global memory one chunk
    // ahead (registers), so that a stage is complete as soon as its tiles land
    float nb[2], nl[2];
    auto fetch = [&](int n) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int e = n * C + lane + 32 * k;
        float bt = 0.f, lg = 0.f;
        if (n < NT && e < p.L) {
          bt = p.beta[((size_t)b * p.L + e) * p.H + h];
          if (GATED && (e % n_h) == 0)
            lg = fmaxf(logf(p.g[((size_t)b * p.T + e / n_h) * p.H + h]), kLogGateFloor) * kLog2e;
        }
        nb[k] = bt;
        nl[k] = lg;
      }
    };
    fetch(0);
    int issued = 0, issued_v = 0;
    for (int n = 0; n < NT; ++n) {
      const int s = n % NS;
      int ok = 1;
      if (n >= NS && lane == 0) ok = wait_bar(sm, B_EMPTY + s, ((n / NS) - 1) & 1, 0);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      const int e0 = n * C;
      const int t_lo = e0 / n_h;
      uint8_t *st = sm.stage(s);
      if (lane == 0) {
        // keep the chunk after the ones in the ring warm in L2
        for (int pf = (n == 0 ? NS : n + NS); pf <= n + NS && pf < NT; ++pf) {
          const int pe = pf * C, pt = pe / n_h;
          tma_prefetch_4d(&map_k, 0, h, pe, b);
          tma_prefetch_4d(&map_k, 64, h, pe, b);
          tma_prefetch_4d(&map_v, 0, h, pe, b);
          tma_prefetch_4d(&map_v, 64, h, pe, b);
          tma_prefetch_4d(&map_q, 0, h, pt, b);
          tma_prefetch_4d(&map_q, 64, h, pt, b);
        }
        // K and Q first, on their own barrier (the G product waits for them
        // only); V, needed later, on a second one
        mbar_arrive_expect_tx(sm.bar(B_FULL + s), 2u * (8192u + (uint32_t)QR * 128u));
        uint64_t *fb = sm.bar(B_FULL + s);
        tma_load_4d(st + ST_K0, &map_k, fb, 0, h, e0, b);
        tma_load_4d(st + ST_K1, &map_k, fb, 64, h, e0, b);
        tma_load_4d(st + ST_Q0, &map_q, fb, 0, h, t_lo, b);
        tma_load_4d(st + ST_Q1, &map_q, fb, 64, h, t_lo, b);
      }
      issued = n + 1;
      float *sb = sm.beta(s), *sl = sm.lam(s);
      sb[lane] = nb[0];
      sb[lane + 32] = nb[1];
      sl[lane] = nl[0];
      sl[lane + 32] = nl[1];
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(B_FULL + s));
      // V on its own barrier: its slot stages the outputs of the chunk NS
      // back, until the chain warps have written them out
      if (n >= NS && lane == 0) ok = wait_bar(sm, B_VEMPTY + s, ((n / NS) - 1) & 1, 0);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (lane == 0) {
        uint64_t *vb = sm.bar(B_VFULL + s);
        mbar_arrive_expect_tx(vb, 2u * 8192u);
        tma_load_4d(st + ST_V0, &map_v, vb, 0, h, e0, b);
        tma_load_4d(st + ST_V0 + 8192, &map_v, vb, 64, h, e0, b);
      }
      issued_v = n + 1;
      fetch(n + 1);
    }
    // copies still in flight must land before the CTA's shared memory goes
    if (lane == 0) {
      for (int n = (issued > NS ? issued - NS : 0); n < issued; ++n)
        wait_bar_drain(sm.base, B_FULL + n % NS, (n / NS) & 1, 0);
      for (int n = (issued_v > NS ? issued_v - NS : 0); n < issued_v; ++n)
        wait_bar_drain(sm.base, B_VFULL + n % NS, (n / NS) & 1, 0);
    }
    __syncwarp();
  } else if (warp == 1 || (dual_issue(GATED) && warp == 14)) {
    // ===================================================== MMA issuers
    // Gated: warp 1 issues the products on the state recurrence (op, the
    // state step with the rest of the output, M, the Q' helper) and warp 14
    // the look-ahead products for later chunks (W, U, G).  Each commits the
    // barriers of its own products; the hand-offs between the two kinds are
    // barriers already.  Ungated: warp 1 issues everything.
    constexpr bool kDual = dual_issue(GATED);
    const bool crit = warp == 1;
    // which thread issues the look-ahead kinds
    const bool do_wu = !kDual || (look_wu(GATED) ? warp == 14 : crit);
    const bool do_g = !kDual || (look_g(GATED) ? warp == 14 : crit);
    if (lane == 0) {
      constexpr uint32_t id_uw = idesc_bf16(128, 64, true, false);
      constexpr uint32_t id_m = idesc_bf16(128, 128, false, true, true);  // B = Kd, MN-major, negated
      constexpr uint32_t id_q = idesc_bf16(128, 64, false, false, true);  // B = P, negated
      constexpr uint32_t id_op = idesc_bf16(128, 64, false, false);       // B = P
      constexpr uint32_t id_s = idesc_bf16(128, 128, false, true);        // B = (M-I)^T or Kd, MN-major
      constexpr uint32_t id_o = idesc_bf16(128, 64, false, false);        // B = Q' (K-major)
      const uint32_t a_tu = smem_u32(sm.base + OFF_TU), a_tw = smem_u32(sm.base + OFF_TW);
      const uint32_t a_ms = smem_u32(sm.base + OFF_MS), a_p = smem_u32(sm.base + OFF_P);
      auto rdy = [&](int idx, int k) -> bool { return mbar_test_wait(sm.bar(idx), k & 1); };
      auto kd_desc = [&](int m, int k) -> uint64_t {  // B = Kd (gated: V slot) or K
        const uint32_t kq = smem_u32(sm.stage(m % NS));
        return GATED ? sdesc_sw128(kq + ST_V0 + k * 2048, 8192, 1024)
                     : sdesc_sw128(kq + ST_K0 + k * 2048, 16384, 1024);
      };
      // Every product of chunk k is issued as soon as its inputs are ready,
      // each kind in chunk order; the barriers are the whole dependency graph
      // (each phase is waited for once, in order).  The tensor pipe runs in
      // order and a thread's issue blocks while it is busy, so the products
      // on the state recurrence (chain -> outputs -> Q' -> op -> chain) go
      // first and the look-ahead work for later chunks after them, in 4-MMA
      // pieces.  In priority order:
      //   op(k): QRDY(k)   chain(n): op(n) issued, SRDY(n), MRDY(n)
      //   m(k): CWD(k)     q(k): M(k) issued, OFREE(k-1)
      //   W(k): TFULL(k), MRDY(k-1)   U(k): after W(k), VFULL(k)   (they release the T tiles)
      //   G(k) halves: FULL(k), GFREE(k-1)
      constexpr uint32_t id_g = idesc_bf16(128, 64, false, false);
      int c_ch = 0, c_op = 0, c_q = 0, c_m = 0, c_w = 0, c_u = 0, c_g2 = 0;
      uint32_t idle = 0, nap = 16;
      while (crit ? c_ch < NT : ((do_wu && c_u < NT) || (do_g && c_g2 < 2 * NT))) {
        if (crit && c_op < c_q && rdy(B_QRDY, c_op)) {
          // ---- O^T = U^T P^T (first part of the output) ----
          const int m = c_op++;
          tc_fence_after();
          const uint32_t pb = a_p + (m & 1) * 8192;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ts(tmem + TM_O, tmem + TM_UB + k * 8, sdesc_sw128(pb + k * 32, 0, 1024), id_op, k > 0);
          mma_commit(sm.bar(B_PFREE0 + (m & 1)));
        } else if (crit && c_ch < c_op && rdy(B_SRDY, c_ch) && rdy(B_MRDY, c_ch)) {
          // ---- the state step and the rest of O(n) ----
          const int n = c_ch++;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ts(tmem + TM_S, tmem + TM_SBF + k * 8, sdesc_sw128(a_ms + k * 2048, 16384, 1024), id_s, true);
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_ts(tmem + TM_S, tmem + TM_UB + k * 8, kd_desc(n, k), id_s, true);
          mma_commit(sm.bar(B_SFULL));
          const uint32_t st = smem_u32(sm.stage(n % NS));
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t qa = st + (k < 4 ? ST_Q0 : ST_Q1) + (k & 3) * 32;
            mma_ts(tmem + TM_O, tmem + TM_SBF + k * 8, sdesc_sw128(qa, 0, 1024), id_o, true);
          }
          mma_commit(sm.bar(B_OFULL));
          mma_commit(sm.bar(B_EMPTY + n % NS));
        } else if (crit && (do_wu ? c_m < c_u : c_m < NT) && rdy(B_CWD, c_m)) {  // CWD(m): U(m) done, converted
          // ---- (M-I)^T = -W^T Kd ----
          const int m = c_m++;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_ts(tmem + TM_X1, tmem + TM_WB + k * 8, kd_desc(m, k), id_m, k > 0);
          mma_commit(sm.bar(B_MFULL));
        } else if (crit && c_q < c_m && (c_q == 0 || rdy(B_OFREE, c_q - 1))) {
          // ---- -W^T P^T (the rest of Q' is added on the CUDA cores) ----
          const int m = c_q++;
          tc_fence_after();
          const uint32_t pb = a_p + (m & 1) * 8192;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ts(tmem + TM_O, tmem + TM_WB + k * 8, sdesc_sw128(pb + k * 32, 0, 1024), id_q, k > 0);
          mma_commit(sm.bar(B_QFULL));
        } else if (do_wu && c_w < NT && c_w == c_u && rdy(B_TFULL, c_w) && (c_w == 0 || rdy(B_MRDY, c_w - 1))) {
          // ---- W^T = K^T (T diag exp gc)^T ----
          const int m = c_w++;
          tc_fence_after();
          const uint32_t kq = smem_u32(sm.stage(m % NS));
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + TM_X1, sdesc_sw128(kq + ST_K0 + k * 2048, 16384, 1024),
                   sdesc_sw128(a_tw + k * 32, 0, 1024), id_uw, k > 0);
        } else if (do_wu && c_u < c_w && rdy(B_VFULL + c_u % NS, c_u / NS)) {
          // ---- U^T = V^T T^T ----
          const int m = c_u++;
          tc_fence_after();
          const uint32_t kq = smem_u32(sm.stage(m % NS));
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + TM_X1 + 64, sdesc_sw128(kq + ST_V0 + k * 2048, 8192, 1024),
                   sdesc_sw128(a_tu + k * 32, 0, 1024), id_uw, k > 0);
          mma_commit(sm.bar(B_WFULL));
        } else if (do_g && c_g2 < 2 * NT && ((c_g2 & 1) ||
                                     (rdy(B_FULL + (c_g2 >> 1) % NS, (c_g2 >> 1) / NS) &&
                                      (c_g2 == 0 || rdy(B_GFREE, (c_g2 >> 1) - 1))))) {
          // ---- G = [K;Q] K^T, one 64-column half of the K dimension ----
          const int m = c_g2 >> 1, hf = c_g2 & 1;
          ++c_g2;
          tc_fence_after();
          const uint32_t kq = smem_u32(sm.stage(m % NS)) + hf * 16384;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + TM_G, sdesc_sw128(kq + k * 32, 0, 1024), sdesc_sw128(kq + k * 32, 0, 1024), id_g,
                   hf > 0 || k > 0);
          if (hf) mma_commit(sm.bar(B_GFULL));
        } else {
          // nothing ready: back off (exponentially, so that the polling
          // leaves the issue slots of this SM sub-partition to the solve),
          // give up after ~1 s
          if (++idle > (1u << 22) || ((idle & 63) == 0 && *sm.abort_flag())) {
            *sm.abort_flag() = 1;
            atomicCAS(&g_tc_error, 0u, 2u | (0xEEu << 8));
            break;
          }
          __nanosleep(nap);
          if (nap < 256) nap <<= 1;
          continue;
        }
        idle = 0;
        nap = 16;
      }
      mma_commit(sm.bar(B_DRAIN));  // every issuer arrives
      wait_bar_drain(sm.base, B_DRAIN, 0, 1);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ===================================================== prep warps
    const int q4 = warp & 3;              // TMEM lane quarter
    const int L = q4 * 32 + lane;         // TMEM lane of this thread
    const int pw = warp - 2;              // 0..3
    const int pt = tid - 64;              // 0..127 within the group
    float *AX = sm.AX();
    float *eg = sm.arr(SM_EG), *ieg = sm.arr(SM_IEG), *bgc = sm.arr(SM_BGC);
    uint8_t *tu = sm.base + OFF_TU;
    uint8_t *tw = sm.base + OFF_TW;
    for (int m = 0; m < NT; ++m) {
      const int s = m % NS;
      // every warp of the group is done with the previous chunk (its gate
      // factors and beta exp(gc) are rewritten below)
      if (named_sync_or(1, *sm.abort_flag() != 0)) break;
      // a failed wait sets the abort flag; every thread still reaches the
      // next named barrier and all of them leave together after it
      wait_bar(sm, B_FULL + s, (m / NS) & 1, 2);
      const float *sb = sm.beta(s);
      if (GATED && warp == 2) {
        float lo, hi;
        warp_scan64(sm.lam(s), lane, lo, hi);
        AX[swz(lane, lane)] = lo;
        AX[swz(lane + 32, lane + 32)] = hi;
        const float e0 = fast_exp2(lo), e1 = fast_exp2(hi);
        eg[lane] = e0;
        eg[lane + 32] = e1;
        ieg[lane] = fast_exp2(-lo);
        ieg[lane + 32] = fast_exp2(-hi);
        bgc[lane] = sb[lane] * e0;
        bgc[lane + 32] = sb[lane + 32] * e1;
      }
      if (!GATED && pt < 64) bgc[pt] = sb[pt];
      if (named_sync_or(1, *sm.abort_flag() != 0)) break;
      const Rows rw(m, n_h, p.T);
      // exact per-entry decay only when the chunk's gate product leaves the
      // range of the ratio form
      const bool ratio = !GATED || AX[swz(63, 63)] >= kRatioFloor;

      // the P buffer is rewritten from here on
      if (m >= 2) wait_bar(sm, B_PFREE0 + (m & 1), ((m >> 1) - 1) & 1, 2);
      // ---- one row of G = [K;Q] K^T per thread (TMEM lane L), 16 columns at a time:
      //      rows 0..63 give A (upper triangle of the solve array, transposed),
      //      rows 64..127 give P ----
      wait_bar(sm, B_GFULL, m & 1, 2);
      tc_fence_after();
      {
        const int i = L, r = L - 64;
        const bool arow = L < 64;
        const float bi = arow ? sb[i] : 0.f;
        const float gi = (GATED && arow) ? AX[swz(i, i)] : 0.f;
        const float bie = (GATED && arow) ? bi * eg[i] : bi;
        const int pos = (!arow && r < rw.Cp) ? rw.pos(r, n_h) : -1;
        const float gp = (GATED && pos >= 0) ? AX[swz(pos, pos)] : 0.f;
        const float ep = (GATED && pos >= 0) ? eg[pos] : 1.f;
        // entry (row, j) = G(row, j) * f_j: f_j = bx (ungated); rf 2^-gc_j
        // (the ratio form, while the chunk's gate product stays in range);
        // else bx 2^(gr - gc_j) exactly.  The branch is uniform per chunk.
        const float bx = arow ? bi : 1.f, rf = arow ? bie : ep, gr = arow ? gi : gp;
        uint8_t *prow = sm.base + OFF_P + (m & 1) * 8192;
#pragma unroll 1
        for (int jb = 0; jb < 64; jb += 16) {
          uint32_t g[16];
          tmem_ld16(tmem_addr(tmem + TM_G, q4 * 32, jb), g);
          float cf[16];
          if (!GATED) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) cf[jj] = bx;
          } else if (ratio) {
#pragma unroll
            for (int jj = 0; jj < 16; jj += 4) {
              const float4 e4 = *reinterpret_cast<const float4 *>(ieg + jb + jj);
              cf[jj] = rf * e4.x;
              cf[jj + 1] = rf * e4.y;
              cf[jj + 2] = rf * e4.z;
              cf[jj + 3] = rf * e4.w;
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) cf[jj] = bx * fast_exp2(gr - AX[swz(jb + jj, jb + jj)]);
          }
          tmem_wait_ld_regs(g);
          if (arow) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int j = jb + jj;
              if (j < i) AX[swz(j, i)] = cf[jj] * __uint_as_float(g[jj]);
            }
          } else {
            uint32_t pk[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int j = jb + 2 * u;
              const float v0 = j <= pos ? __uint_as_float(g[2 * u]) * cf[2 * u] : 0.f;
              const float v1 = j + 1 <= pos ? __uint_as_float(g[2 * u + 1]) * cf[2 * u + 1] : 0.f;
              pk[u] = pack_bf16(v0, v1);
            }
            st_chunk(prow + sw128_offset(r, jb, 64), {pk[0], pk[1], pk[2], pk[3]});
            st_chunk(prow + sw128_offset(r, jb + 8, 64), {pk[4], pk[5], pk[6], pk[7]});
          }
        }
        tc_fence_before();
        arrive_warp(sm.bar(B_GFREE), lane);
      }
      if (named_sync_or(1, *sm.abort_flag() != 0)) break;  // A complete

      // ---- X = (I + A)^{-1}: 16x16 diagonal blocks, one per warp; the T
      //      tiles are rewritten from here on ----
      if (m >= 1) wait_bar(sm, B_WFULL, (m - 1) & 1, 2);
      invert_diag16(AX, tu, tw, sb, bgc, 16 * pw, lane);
      named_sync(1);
      {
        // ---- merge 16 -> 32: X21 = -X22 (A21 X11) in each 32-row half;
        //      warp = (half, 8-column slab), the product A21 X11 stays in registers ----
        const int o = 32 * (pw >> 1), n0 = o + 8 * (pw & 1);
        uint32_t fa[2][4], fx[2][2], fz[2][4];
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          frag_a<0>(fa[ks], AX, o + 16, o + 8 * ks, lane);
          frag_b<1>(fx[ks], AX, o + 8 * ks, n0, lane);
          frag_a<1>(fz[ks], AX, o + 16, o + 16 + 8 * ks, lane);
        }
        float y[1][4] = {{0.f, 0.f, 0.f, 0.f}}, z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) mma_tf32(y[0], fa[ks], fx[ks]);
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          uint32_t bb[2];
          frag_b_acc<1>(bb, y, ks, lane);
          mma_tf32(z, fz[ks], bb);
        }
        warp_store_16x8(AX, o + 16, n0, z, -1.f, lane);
        frag_to_t(tu, tw, o + 16, n0, z, -1.f, sb, bgc, lane);
      }
      named_sync(1);
      {
        // ---- merge 32 -> 64: rows 32..63, columns 8 pw .. 8 pw + 7 of X,
        //      straight into the T tiles ----
        const int n0 = 8 * pw;
        float y[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          uint32_t fa[2][4][4], fx[4][2];
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            frag_b<1>(fx[ks], AX, 8 * ks, n0, lane);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) frag_a<0>(fa[mt][ks], AX, 32 + 16 * mt, 8 * ks, lane);
          }
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) mma_tf32(y[mt], fa[mt][ks], fx[ks]);
        }
        float z[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          uint32_t fz[2][4][4];
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) frag_a<1>(fz[mt][ks], AX, 32 + 16 * mt, 32 + 8 * ks, lane);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            uint32_t bb[2];
            frag_b_acc<2>(bb, y, ks, lane);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) mma_tf32(z[mt], fz[mt][ks], bb);
          }
        }
        frag_to_t(tu, tw, 32, n0, z[0], -1.f, sb, bgc, lane);
        frag_to_t(tu, tw, 48, n0, z[1], -1.f, sb, bgc, lane);
      }
      fence_proxy_async_smem();
      arrive_warp(sm.bar(B_TFULL), lane);
    }
  } else if (warp < 10) {
    // ===================================================== feed-forward warps
    const int q4 = warp & 3;
    const int L = q4 * 32 + lane;  // TMEM lane: a d index
    const int ft = tid - 192;      // 0..127 within the group
    float *dec = sm.arr(SM_DEC);
    for (int c = 0; c < NT; ++c) {
      const int s = c % NS;
      // every warp of the group is done with the previous chunk's gate
      // factors before they are rewritten
      if (named_sync_or(2, *sm.abort_flag() != 0)) break;
      if (GATED) {
        wait_bar(sm, B_FULL + s, (c / NS) & 1, 3);
        if (warp == 6) {
          float lo, hi;
          warp_scan64(sm.lam(s), lane, lo, hi);
          const float tot = __shfl_sync(0xffffffffu, hi, 31);
          dec[lane] = fast_exp2(tot - lo);
          dec[lane + 32] = fast_exp2(tot - hi);
          if (lane == 0) *sm.gate_c() = fast_exp2(tot);
        }
        named_sync(2);
      }

      // ---- W^T, U^T -> bf16 operands; Kd ----
      wait_bar(sm, B_WFULL, c & 1, 3);
      tc_fence_after();
      {
        uint32_t r[64], pw_[32];
        tmem_ld32(tmem_addr(tmem + TM_X1, q4 * 32, 0), *reinterpret_cast<uint32_t (*)[32]>(&r[0]));
        tmem_ld32(tmem_addr(tmem + TM_X1, q4 * 32, 32), *reinterpret_cast<uint32_t (*)[32]>(&r[32]));
        tmem_wait_ld_regs(r);
#pragma unroll
        for (int u = 0; u < 32; ++u)
          pw_[u] = pack_bf16(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
        // W^T bf16 of the previous chunk is read by its -W^T P^T product
        // (after its M product, whose completion was waited for already)
        if (c >= 1) {
          wait_bar(sm, B_QFULL, (c - 1) & 1, 3);
          tc_fence_after();
        }
        tmem_st32(tmem_addr(tmem + TM_WB, q4 * 32, 0), pw_);
      }
      if (GATED) {
        // Kd = diag(exp(gc_C - gc)) K into the V slot (V was consumed by U)
        const uint8_t *kt = sm.stage(s);
        uint8_t *kd = sm.stage(s) + ST_V0;
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int qi = ft + 128 * it;  // 16-byte chunk: 512 per 64-column half
          const int half = qi >> 9, rem = qi & 511, row = rem >> 3;
          const uint4 v = *reinterpret_cast<const uint4 *>(kt + half * 16384 + rem * 16);
          const float dr = dec[row];
          const uint32_t in[4] = {v.x, v.y, v.z, v.w};
          uint32_t o4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            o4[u] = pack_bf16(__uint_as_float(in[u] << 16) * dr, __uint_as_float(in[u] & 0xFFFF0000u) * dr);
          st_chunk(kd + half * 8192 + rem * 16, o4);
        }
        fence_proxy_async_smem();
      }
      uint32_t pu[32];
      {
        uint32_t r[64];
        tmem_ld32(tmem_addr(tmem + TM_X1, q4 * 32, 64), *reinterpret_cast<uint32_t (*)[32]>(&r[0]));
        tmem_ld32(tmem_addr(tmem + TM_X1, q4 * 32, 96), *reinterpret_cast<uint32_t (*)[32]>(&r[32]));
        tmem_wait_ld_regs(r);
#pragma unroll
        for (int u = 0; u < 32; ++u)
          pu[u] = pack_bf16(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
      }
      // U^T bf16 is read by the state step of the previous chunk until it ends
      if (c >= 1) wait_bar(sm, B_SFULL, (c - 1) & 1, 3);
      tmem_st32(tmem_addr(tmem + TM_UB, q4 * 32, 0), pu);
      tmem_wait_st();
      tc_fence_before();
      arrive_warp(sm.bar(B_CWD), lane);

      // ---- (M-I)^T -> bf16 smem operand (row L = j, columns i) ----
      wait_bar(sm, B_MFULL, c & 1, 3);
      tc_fence_after();
      const float gm1 = GATED ? *sm.gate_c() - 1.f : 0.f;
#pragma unroll 1
      for (int cb = 0; cb < 128; cb += 32) {
        uint32_t r[32];
        tmem_ld32(tmem_addr(tmem + TM_X1, q4 * 32, cb), r);
        tmem_wait_ld_regs(r);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t o4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            o4[u] = pack_bf16(__uint_as_float(r[q * 8 + 2 * u]), __uint_as_float(r[q * 8 + 2 * u + 1]));
          st_chunk(sm.base + OFF_MS + sw128_offset(L, cb + q * 8, 128), o4);
        }
      }
      if (GATED) {
        // the (exp(gc_C) - 1) I term, on this thread's own diagonal entry
        __nv_bfloat16 *dg = reinterpret_cast<__nv_bfloat16 *>(sm.base + OFF_MS + sw128_offset(L, L, 128));
        *dg = __float2bfloat16_rn(__bfloat162float(*dg) + gm1);
      }
      tc_fence_before();
      fence_proxy_async_smem();
      arrive_warp(sm.bar(B_MRDY), lane);

    }
  } else {
    // ===================================================== chain warps
    const int q4 = warp & 3;
    const int L = q4 * 32 + lane;  // TMEM lane = value column dv
    float *gq = sm.arr(SM_GQ);
    // Q'(c) = exp(gc) Q - P W, in place over the Q tile of chunk c (same
    // K-major layout: the output product reads it as its B operand); the
    // scan for exp(gc) at the readout rows first
    auto qprime = [&](int c) {
      const int s = c % NS;
      const Rows rw(c, n_h, p.T);
      if (GATED) wait_bar(sm, B_FULL + s, (c / NS) & 1, 4);  // the chunk's log-gate row
      if (GATED && warp == 10) {
        float lo, hi;
        warp_scan64(sm.lam(s), lane, lo, hi);
        const float elo = fast_exp2(lo), ehi = fast_exp2(hi);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int r = lane + 32 * hf;
          const int pos = rw.pos(r, n_h);
          const float a = __shfl_sync(0xffffffffu, elo, pos & 31);
          const float e = __shfl_sync(0xffffffffu, ehi, pos & 31);
          gq[r] = r < rw.Cp ? (pos < 32 ? a : e) : 0.f;
        }
      }
      if (GATED) named_sync(3);
      wait_bar(sm, B_QFULL, c & 1, 4);
      tc_fence_after();
      {
        // Warp-MMA fragments throughout: the tile of this warp (d = 32 q4 ..
        // 32 q4 + 31, all 64 rows) goes in 8x8 pieces; a thread holds the
        // pairs (d = t / 4 (+ 8), rows 8 g + 2 (t % 4), + 1) of TMEM, of Q
        // (transposing 8x8 loads) and of Q' (transposing 8x8 stores, to the
        // addresses the loads came from)
        const int tq = lane & 3;
        float2 gv[8];
#pragma unroll
        for (int g = 0; g < 8; ++g)
          gv[g] = GATED ? *reinterpret_cast<const float2 *>(gq + 8 * g + 2 * tq) : make_float2(1.f, 1.f);
        const int cp = rw.Cp;
        const uint32_t qh = smem_u32(sm.stage(s) + ((q4 >> 1) ? ST_Q1 : ST_Q0));
        const int mi = lane >> 3, mr = lane & 7;  // the 8x8 piece and row this lane addresses
#pragma unroll
        for (int b16 = 0; b16 < 32; b16 += 16) {
          uint32_t hreg[32];
          tmem_ld16x256b_x8(tmem_addr(tmem + TM_O, q4 * 32 + b16, 0), hreg);
          tmem_wait_ld_regs(hreg);
          const int ck = (32 * (q4 & 1) + b16) / 8 + (mi & 1);  // 16-byte piece of the row
          // all loads of this half first (the stores go to the same places)
          uint32_t addr[4], qd[4][4];
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const int row = 16 * cc + 8 * (mi >> 1) + mr;
            addr[cc] = qh + (row >> 3) * 1024 + (row & 7) * 128 + ((ck ^ (row & 7)) << 4);
            ldsm_x4_trans(addr[cc], qd[cc]);
          }
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t o4[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const int g = 2 * cc + (m >> 1), j = 4 * g + 2 * (m & 1);
              const int r0 = 8 * g + 2 * tq;
              const float v0 = fmaf(gv[g].x, __uint_as_float(qd[cc][m] << 16), __uint_as_float(hreg[j]));
              const float v1 = fmaf(gv[g].y, __uint_as_float(qd[cc][m] & 0xFFFF0000u), __uint_as_float(hreg[j + 1]));
              o4[m] = pack_bf16(r0 < cp ? v0 : 0.f, r0 + 1 < cp ? v1 : 0.f);
            }
            stsm_x4_trans(addr[cc], o4);
          }
        }
        tc_fence_before();
      }
      fence_proxy_async_smem();
      arrive_warp(sm.bar(B_QRDY), lane);
      if (GATED) named_sync(3);  // gq is rewritten for the next chunk
    };
    // ---- initial state S^T (lane = dv, column = dk) ----
    {
      const float *h0 = p.h0 ? p.h0 + (size_t)bh * D * D : nullptr;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t f[32], pk[16];
#pragma unroll
        for (int u = 0; u < 32; u += 2) {
          const float x0 = h0 ? h0[(size_t)(c0 + u) * D + L] : 0.f;
          const float x1 = h0 ? h0[(size_t)(c0 + u + 1) * D + L] : 0.f;
          f[u] = __float_as_uint(x0);
          f[u + 1] = __float_as_uint(x1);
          pk[u >> 1] = pack_bf16(x0, x1);
        }
        tmem_st32(tmem_addr(tmem + TM_S, q4 * 32, c0), f);
        tmem_st16(tmem_addr(tmem + TM_SBF, q4 * 32, c0 / 2), pk);
      }
      tmem_wait_st();
      tc_fence_before();
      arrive_warp(sm.bar(B_SRDY), lane);
    }
    if (!named_sync_or(3, *sm.abort_flag() != 0)) qprime(0);
    for (int n = 0; n < NT; ++n) {
      if (named_sync_or(3, *sm.abort_flag() != 0)) break;
      const Rows rw(n, n_h, p.T);
      // ---- state: S^T -> bf16 operand for the next chunk, or hT ----
      wait_bar(sm, B_SFULL, n & 1, 4);
      tc_fence_after();
      if (n + 1 < NT) {
        uint32_t pk[64];
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t r[32];
          tmem_ld32(tmem_addr(tmem + TM_S, q4 * 32, cb * 32), r);
          tmem_wait_ld_regs(r);
#pragma unroll
          for (int u = 0; u < 16; ++u)
            pk[cb * 16 + u] = pack_bf16(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
        }
        // the output products of chunk n read the bf16 copy until they end
        wait_bar(sm, B_OFULL, n & 1, 4);
        tc_fence_after();
        tmem_st32(tmem_addr(tmem + TM_SBF, q4 * 32, 0), *reinterpret_cast<uint32_t (*)[32]>(&pk[0]));
        tmem_st32(tmem_addr(tmem + TM_SBF, q4 * 32, 32), *reinterpret_cast<uint32_t (*)[32]>(&pk[32]));
        tmem_wait_st();
        tc_fence_before();
        arrive_warp(sm.bar(B_SRDY), lane);
      } else if (p.hT) {
        float *hT = p.hT + (size_t)bh * D * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tmem_addr(tmem + TM_S, q4 * 32, c0), r);
          tmem_wait_ld_regs(r);
#pragma unroll
          for (int u = 0; u < 32; ++u) hT[(size_t)(c0 + u) * D + L] = __uint_as_float(r[u]);
        }
      }
      // ---- outputs of this chunk: the accumulator is read at once (TMEM is
      //      released early), staged as bf16 rows in the V slot of this chunk
      //      (its last reader, the U product or, gated, the state step on Kd,
      //      has completed) by transposing 8x8 stores, then written out in
      //      16-byte pieces ----
      wait_bar(sm, B_OFULL, n & 1, 4);
      tc_fence_after();
      uint32_t o0[32], o1[32];
      tmem_ld16x256b_x8(tmem_addr(tmem + TM_O, q4 * 32, 0), o0);
      tmem_ld16x256b_x8(tmem_addr(tmem + TM_O, q4 * 32 + 16, 0), o1);
      tmem_wait_ld_regs(o0);
      tmem_wait_ld_regs(o1);
      tc_fence_before();
      arrive_warp(sm.bar(B_OFREE), lane);
      {
        // staging row r (a readout row): 256 bytes, the 16-byte piece k
        // (values 8 k .. 8 k + 7) at (k ^ (r % 8)) * 16
        const uint32_t sv = smem_u32(sm.stage(n % NS) + ST_V0);
        auto srow = [&](int r) -> uint32_t { return sv + r * 256; };
        const int mi = lane >> 3, mr = lane & 7;
#pragma unroll
        for (int b16 = 0; b16 < 32; b16 += 16) {
          const uint32_t(&ov)[32] = b16 ? o1 : o0;
          const int k = (32 * q4 + b16) / 8 + (mi & 1);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t o4[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const int j = 4 * (2 * cc + (m >> 1)) + 2 * (m & 1);
              o4[m] = pack_bf16(__uint_as_float(ov[j]), __uint_as_float(ov[j + 1]));
            }
            const int r = 16 * cc + 8 * (mi >> 1) + mr;
            stsm_x4_trans(srow(r) + ((k ^ (r & 7)) << 4), o4);
          }
        }
        named_sync(3);  // every value column of every row staged
        const int ct = tid - 320;  // 0..127 within the group
        const int k = ct & 15, cp = rw.Cp;
        __nv_bfloat16 *obase = p.out + (((size_t)b * p.T + rw.t_lo) * p.H + h) * D + 8 * k;
        const size_t rstride = (size_t)p.H * D;
        uint4 v[8];  // every load before the first store
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int r = 8 * it + (ct >> 4);
          v[it] = lds128(srow(r) + ((k ^ (r & 7)) << 4));
        }
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int r = 8 * it + (ct >> 4);
          if (r < cp) *reinterpret_cast<uint4 *>(obase + r * rstride) = v[it];
        }
        // the V slot is free once every warp has read its rows
        arrive_warp(sm.bar(B_VEMPTY + n % NS), lane);
      }
      if (n + 1 < NT) qprime(n + 1);
    }
  }

  // ---- teardown ----
  tc_fence_before();
  __syncthreads();
  if (warp == 1 && !*sm.keep_tmem()) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

}  // namespace

bool chunk_tc_supports(const FwdArgs &a) {
  return a.bf16 && a.dk == D && a.dv == D && a.chunk == C && a.T > 0 &&
         a.L < (int64_t(1) << 30) && a.B * a.H < (int64_t(1) << 31);
}

namespace {
// The bounded-wait path on its own: a barrier nobody arrives on.
__global__ void wait_selftest_kernel(unsigned int polls) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    sm100::mbar_init(&bar, 1);
    sm100::fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    bool done = false;
    for (unsigned int i = 0; i < polls && !done; ++i) done = sm100::mbar_try_wait(&bar, 0);
    if (!done) atomicCAS(&g_tc_error, 0u, (1u + 7u) | (253u << 8));
  }
}
}  // namespace

cudaError_t launch_wait_selftest(unsigned int polls, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(polls);
  return cudaGetLastError();
}

cudaError_t read_and_clear_tc_error(unsigned int *word) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(word, g_tc_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(unsigned int));
}

cudaError_t launch_chunk_tc(const FwdArgs &a, cudaStream_t s) {
  if (!chunk_tc_supports(a)) return cudaErrorNotSupported;
  CUtensorMap mq, mk, mv;
  const uint32_t qr = a.n_h == 1 ? 64 : 32;
  cudaError_t e;
  if ((e = make_map_4d_bf16(&mq, a.q, D, a.H, a.T, a.B, 64, 1, qr, 1, true)) != cudaSuccess) return e;
  if ((e = make_map_4d_bf16(&mk, a.k, D, a.H, a.L, a.B, 64, 1, 64, 1, true)) != cudaSuccess) return e;
  if ((e = make_map_4d_bf16(&mv, a.v, D, a.H, a.L, a.B, 64, 1, 64, 1, true)) != cudaSuccess) return e;
  TcParams p;
  p.beta = a.beta;
  p.g = a.g;
  p.h0 = a.h0;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.hT = a.hT;
  p.H = (int)a.H;
  p.T = (int)a.T;
  p.L = (int)a.L;
  p.n_h = a.n_h;
  p.nchunks = (int)((a.L + C - 1) / C);
  auto kern = a.g ? chunk_tc_kernel<true> : chunk_tc_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)(a.B * a.H), threads_for(a.g != nullptr), SMEM_ALLOC, s>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace delta
