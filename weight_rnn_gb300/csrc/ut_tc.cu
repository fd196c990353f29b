// ut_tc.cu -- the intra-chunk pass of the chunked forward on the 5th-
// generation tensor cores: for every chunk of 64 steps of every (b, h) head,
// in parallel over all chunks of all heads,
//
//   gc = inclusive cumsum of the log gate (log g_t at each token's first
//        sub-step, 0 elsewhere; clamped at -80 so g = 0 stays finite)
//   A  = strictLower(diag(beta) (Gam * K K^T)),   Gam_ij = exp(gc_i - gc_j)
//   T  = (I + A)^{-1} diag(beta)                   (the UT transform)
//
// as in "08 · linear 路线（三）：delta rule 与 DPLR 统一框架" §2.2 (the UT
// transform: A from the keys and beta, T by forward substitution, in SRAM)
// and §3 (the gated chunk form: the decay ratios inside A), on the extended
// sequence of "DeltaProduct：通过 Householder 乘积增强线性 RNN 的状态追踪" §4.1
// (n_h sub-steps per token; the gate at each token's first one).  T is
// written as bf16, row-major [chunks][64][64] (chunk = (b * H + h) * NT + n);
// the state pass reads it back.  Rows past the end of the sequence are
// identity steps (k = 0, beta = 0, log g = 0), so T is 0 there except for
// the unit diagonal times beta = 0.
//
// A CTA takes two chunks at a time (a "pair", consecutive in the global
// chunk order).  Their keys are stacked into one 128-row operand and one
// tcgen05 product G = [K_a; K_b] [K_a; K_b]^T (M = N = 128, K = 128) gives
// both Gram matrices on its diagonal blocks.  The solve is blocked: the four
// 16x16 diagonal blocks of I + A are inverted one per warp, then two block
// merges X21 = -X22 (A21 X11) run on warp-level tf32 MMAs.
//
// Warp roles (320 threads, two CTAs per SM, persistent over pairs):
//   warps 0, 1, 4, 5   chunk a of the pair: A formation, solve, T store
//   warps 2, 3, 6, 7   chunk b
//   warp 8             TMA producer: the pair's key tiles, beta, log gate
//   warp 9             TMEM owner and MMA issuer
// The key tiles of a pair occupy one of two 32 KB slots; once the Gram
// product has read them, the slot holds the two solve arrays.  Every
// mbarrier wait is bounded; a timeout sets a device error word and the
// kernel winds down instead of hanging.
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm100.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace delta {

// Set by the UT kernel when a bounded wait gives up (1 + role id, barrier << 8).
__device__ unsigned int g_ut_error = 0;

namespace {
using namespace sm100;
using namespace tc;

constexpr int C = 64;
constexpr int D = 128;
constexpr int UT_THREADS = 320;
constexpr int UT_CTAS_PER_SM = 2;

// ---- shared memory layout (offsets from a 1024-byte aligned base) ----
constexpr uint32_t SLOT_BYTES = 32768;  // [K_a lo | K_b lo | K_a hi | K_b hi], later AX_a | AX_b
constexpr uint32_t OFF_T = 2 * SLOT_BYTES;  // two bf16 T tiles (chunk a, chunk b), 8 KB each
constexpr uint32_t OFF_SM = OFF_T + 2 * 8192;
constexpr uint32_t SM_BETA = 0;                   // [slot][chunk][64]
constexpr uint32_t SM_LAM = SM_BETA + 4 * 256;    // [slot][chunk][64] log2 gate
constexpr uint32_t SM_GC = SM_LAM + 4 * 256;      // [chunk][64] cumulative log2 gate
constexpr uint32_t SM_IEG = SM_GC + 2 * 256;      // [chunk][64] 2^-gc
constexpr uint32_t SM_BEG = SM_IEG + 2 * 256;     // [chunk][64] beta 2^gc
constexpr uint32_t SM_BAR = SM_BEG + 2 * 256;
enum {
  B_FULL = 0,   // [2] producer -> all: the slot's key tiles, beta, log gate (count 1 + tx)
  B_FREE = 2,   // [2] solve groups -> producer: the slot's solve arrays released (count 2)
  B_GFULL = 4,  // MMA -> solve: G in TMEM
  B_GFREE,      // solve -> MMA: G read (one arrival per solve warp, 8)
  B_DRAIN,      // MMA: every product issued has completed
  NBARS
};
constexpr uint32_t SM_MISC = SM_BAR + NBARS * 8;  // tmem slot, abort flag, keep-TMEM flag
constexpr uint32_t SMEM_TOTAL = OFF_SM + ((SM_MISC + 16 + 15) & ~15u);
constexpr uint32_t UT_SMEM_ALLOC = SMEM_TOTAL + 1024;  // + worst-case alignment
static_assert(UT_CTAS_PER_SM * (UT_SMEM_ALLOC + 1024) <= 233472, "two CTAs per SM");
constexpr uint32_t TM_COLS = 128;

struct UtParams {
  const float *beta, *g;
  int H, T, L, n_h, nchunks;  // chunks per head
  long long total;            // chunks over all heads
  long long pairs;
};

struct Smem {
  uint8_t *base;
  __device__ uint8_t *slot(int s) const { return base + s * SLOT_BYTES; }
  __device__ float *arr(uint32_t off) const { return reinterpret_cast<float *>(base + OFF_SM + off); }
  __device__ uint64_t *bar(int i) const {
    return reinterpret_cast<uint64_t *>(base + OFF_SM + SM_BAR) + i;
  }
  __device__ uint32_t *tmem_slot() const { return reinterpret_cast<uint32_t *>(base + OFF_SM + SM_MISC); }
  __device__ volatile int *abort_flag() const {
    return reinterpret_cast<volatile int *>(base + OFF_SM + SM_MISC + 4);
  }
  __device__ volatile int *keep_tmem() const {
    return reinterpret_cast<volatile int *>(base + OFF_SM + SM_MISC + 8);
  }
};

__device__ __noinline__ bool wait_bar_slow(uint8_t *base, int idx, uint32_t parity, int role) {
  Smem sm;
  sm.base = base;
  uint64_t *b = sm.bar(idx);
  for (uint32_t i = 0; i < (1u << 22); ++i) {
    if (mbar_try_wait(b, parity)) return true;
    if ((i & 63) == 63 && *sm.abort_flag()) return false;
  }
  *sm.abort_flag() = 1;
  atomicCAS(&g_ut_error, 0u, (unsigned)(1 + role) | ((unsigned)idx << 8));
  return false;
}
// Bounded wait that also gives up at once when another role has aborted.
__device__ __forceinline__ bool wait_bar(const Smem &sm, int idx, uint32_t parity, int role) {
  if (mbar_try_wait(sm.bar(idx), parity)) return true;
  return wait_bar_slow(sm.base, idx, parity, role);
}
// Wait for copies or products already issued: ignores the abort flag (they
// complete on their own), still bounded; if it runs out on the products
// (which write TMEM), TMEM is kept at exit.
__device__ __noinline__ bool wait_bar_drain(uint8_t *base, int idx, uint32_t parity, int role,
                                            bool tmem_writer) {
  Smem sm;
  sm.base = base;
  uint64_t *b = sm.bar(idx);
  for (uint32_t i = 0; i < (1u << 24); ++i)
    if (mbar_try_wait(b, parity)) return true;
  *sm.abort_flag() = 1;
  if (tmem_writer) *sm.keep_tmem() = 1;
  atomicCAS(&g_ut_error, 0u, (unsigned)(1 + role) | ((unsigned)idx << 8));
  return false;
}

// fp32 64x64 matrices in shared memory are stored row-major with the column
// XOR-swizzled by the row (bits 2..4), which keeps float4 runs along a row
// contiguous and makes the tf32 MMA fragment loads below conflict-free.
__device__ __forceinline__ int swz(int r, int c) { return r * 64 + (c ^ ((r & 7) << 2)); }

// The solve's 64x64 array holds A_ij (i > j) at (j, i) -- the upper triangle --
// and X_ij = ((I + A)^{-1})_ij (i > j) at (i, j) -- the lower triangle.  The
// diagonal is never read (X_ii = 1 is implicit).
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

// T[r][c] = x beta_c, into the bf16 T tile (128-byte swizzled rows).
__device__ __forceinline__ void put_t(uint8_t *tu, int r, int c, float x, float bc) {
  *reinterpret_cast<__nv_bfloat16 *>(tu + sw128_offset(r, c, 64)) = __float2bfloat16_rn(x * bc);
}

// The T tile from a 16x8 fragment of (scale * X) at rows r0.., columns n0...
__device__ __forceinline__ void frag_to_t(uint8_t *tu, int r0, int n0, const float (&d)[4],
                                          float scale, const float *beta, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const int c = n0 + 2 * t;
  const float b0 = beta[c], b1 = beta[c + 1];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const float x0 = d[2 * hh] * scale, x1 = d[2 * hh + 1] * scale;
    const int r = r0 + g + 8 * hh;
    *reinterpret_cast<uint32_t *>(tu + sw128_offset(r, c, 64)) = pack_bf16(x0 * b0, x1 * b1);
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
// o of (I + A) by column-oriented forward substitution: lane j (and lane
// j + 16, which repeats it) carries column j of X = (I + A_oo)^{-1} in
// registers, starting from e_j.  At step k its entry k is final; it is x_kj,
// and every row i > k takes -A_ik x_kj.  Column k of A sits in row o + k of
// the solve array's upper triangle (A_ik at (k, i)), read as float4 groups
// that every lane shares.  The dependent chain is one multiply-add per step.
// X goes to the lower triangle of the solve array and, scaled by beta of its
// column, to the T tile.
__device__ __forceinline__ void invert_diag16(float *AX, uint8_t *tu, const float *beta, int o,
                                              int lane) {
  const int j = lane & 15;
  float x[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = i == j ? 1.f : 0.f;
#pragma unroll
  for (int k = 0; k < 15; ++k) {
    // A_{o+i, o+k} for i = 0..15 from row o + k (the 128-bit groups keep
    // their 4 columns together under the row swizzle)
    const float *row = AX + (o + k) * 64;
    float a[16];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      if (4 * g + 3 <= k) continue;  // every column of the group is at or left of the diagonal
      const float4 v = *reinterpret_cast<const float4 *>(row + ((o + 4 * g) ^ (((o + k) & 7) << 2)));
      a[4 * g] = v.x;
      a[4 * g + 1] = v.y;
      a[4 * g + 2] = v.z;
      a[4 * g + 3] = v.w;
    }
    const float xk = x[k];
#pragma unroll
    for (int i = k + 1; i < 16; ++i) x[i] = fmaf(-a[i], xk, x[i]);
  }
  if (lane < 16) {
    const float bj = beta[o + j];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i > j) AX[swz(o + i, o + j)] = x[i];
      if (i >= j) put_t(tu, o + i, o + j, x[i], bj);
    }
  }
}

// Named barrier of solve group gi (ids 1 and 2, immediate operands, so that
// the kernel reserves only the barriers it uses).
__device__ __forceinline__ void group_sync(int gi) {
  if (gi == 0)
    named_sync(1);
  else
    named_sync(2);
}
__device__ __forceinline__ bool group_sync_or(int gi, bool cond) {
  return gi == 0 ? named_sync_or(1, cond) : named_sync_or(2, cond);
}

template <bool GATED>
__global__ void __launch_bounds__(UT_THREADS, UT_CTAS_PER_SM)
ut_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_t,
          UtParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem sm;
  sm.base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __builtin_assume(__isShared(sm.base));
  const int tid = threadIdx.x, lane = tid & 31;
  // the warp index through a shuffle from lane 0: the compiler then knows it
  // is the same in every lane, so that branches on a warp's role are not
  // divergent and need no reconvergence code around the warp-wide
  // instructions in them (a much smaller kernel)
  const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
  if ((uint32_t)(sm.base - smem_raw) + SMEM_TOTAL > UT_SMEM_ALLOC) {
    if (tid == 0) atomicCAS(&g_ut_error, 0u, 0xFFu);
    return;
  }
  // pairs of this CTA: blockIdx.x, blockIdx.x + gridDim.x, ...
  const long long npairs = p.pairs;
  const int mine = (int)((npairs - blockIdx.x + gridDim.x - 1) / gridDim.x);
  auto pair_of = [&](int i) -> long long { return (long long)blockIdx.x + (long long)i * gridDim.x; };

  // ---- set-up ----
  {
    // the two T tiles (the solve writes their lower triangle and diagonal
    // only, the same entries for every pair, so the strict upper triangle
    // stays zero from here on), the small arrays, the barriers and the flags
    uint4 *z = reinterpret_cast<uint4 *>(sm.base + OFF_T);
    for (uint32_t i = tid; i < (SMEM_TOTAL - OFF_T) / 16; i += UT_THREADS) z[i] = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  if (tid == 0) {
    *sm.abort_flag() = 0;
    *sm.keep_tmem() = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(sm.bar(B_FULL + s), 1);
      mbar_init(sm.bar(B_FREE + s), 2);
    }
    mbar_init(sm.bar(B_GFULL), 1);
    mbar_init(sm.bar(B_GFREE), 8);
    mbar_init(sm.bar(B_DRAIN), 1);
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(sm.tmem_slot(), TM_COLS);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_t);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot();

  if (warp == 8) {
    // ===================================================== TMA producer
    // beta and the linear gate of a pair's two chunks are read into registers
    // one pair ahead (lanes: steps lane and lane + 32 of each chunk), so that
    // the loads are in flight while the producer waits for a free slot
    float pb[4], pg[4];
    auto fetch = [&](int i) {
      const long long pr = pair_of(i);
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const long long c = 2 * pr + x;
        const bool live = i < mine && c < p.total;
        const int bh = live ? (int)(c / p.nchunks) : 0, n = live ? (int)(c % p.nchunks) : 0;
        const int b = bh / p.H, h = bh % p.H;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int e = n * C + lane + 32 * k;
          const bool in = live && e < p.L;
          pb[2 * x + k] = in ? __ldg(p.beta + ((size_t)b * p.L + e) * p.H + h) : 0.f;
          pg[2 * x + k] = (GATED && in && (e % p.n_h) == 0)
                              ? __ldg(p.g + ((size_t)b * p.T + e / p.n_h) * p.H + h)
                              : 1.f;
        }
      }
    };
    fetch(0);
    int issued = 0;
    for (int i = 0; i < mine; ++i) {
      const int s = i & 1;
      int ok = 1;
      if (i >= 2 && lane == 0) ok = wait_bar(sm, B_FREE + s, ((i >> 1) - 1) & 1, 0);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      const long long pr = pair_of(i);
      uint32_t bytes = 0;
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        float *sb = sm.arr(SM_BETA + (s * 2 + x) * 256), *sl = sm.arr(SM_LAM + (s * 2 + x) * 256);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          sb[lane + 32 * k] = pb[2 * x + k];
          // the log2 gate (log g at each token's first sub-step, clamped so
          // that g = 0 stays finite; 0 elsewhere and past the end)
          sl[lane + 32 * k] = GATED ? gate_log2(pg[2 * x + k]) : 0.f;
        }
        if (2 * pr + x < p.total) bytes += 16384u;
      }
      __syncwarp();
      if (lane == 0) {
        uint64_t *fb = sm.bar(B_FULL + s);
        mbar_arrive_expect_tx(fb, bytes);
        uint8_t *st = sm.slot(s);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const long long c = 2 * pr + x;
          if (c < p.total) {
            const int bh = (int)(c / p.nchunks), n = (int)(c % p.nchunks);
            const int b = bh / p.H, h = bh % p.H;
            tma_load_4d(st + x * 8192, &map_k, fb, 0, h, n * C, b);
            tma_load_4d(st + 16384 + x * 8192, &map_k, fb, 64, h, n * C, b);
          }
        }
      }
      issued = i + 1;
      fetch(i + 1);
    }
    // copies still in flight must land before the CTA's shared memory goes
    if (lane == 0)
      for (int i = (issued > 2 ? issued - 2 : 0); i < issued; ++i)
        wait_bar_drain(sm.base, B_FULL + (i & 1), (i >> 1) & 1, 0, false);
    __syncwarp();
  } else if (warp == 9) {
    // ===================================================== MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_g = idesc_bf16(128, 128, false, false);
      for (int i = 0; i < mine; ++i) {
        const int s = i & 1;
        if (!wait_bar(sm, B_FULL + s, (i >> 1) & 1, 1)) break;
        if (i >= 1 && !wait_bar(sm, B_GFREE, (i - 1) & 1, 1)) break;
        tc_fence_after();
        const uint32_t kq = smem_u32(sm.slot(s));
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t dsc = sdesc_sw128(kq + (k >> 2) * 16384 + (k & 3) * 32, 0, 1024);
          mma_ss(tmem, dsc, dsc, id_g, k > 0);
        }
        mma_commit(sm.bar(B_GFULL));
      }
      mma_commit(sm.bar(B_DRAIN));
      wait_bar_drain(sm.base, B_DRAIN, 0, 1, true);
    }
    __syncwarp();
  } else {
    // ===================================================== solve groups
    const int gi = (warp >> 1) & 1;                     // chunk of the pair
    const int pw = (warp & 1) | ((warp >> 2) << 1);     // warp within the group
    const int q = warp & 1, hf = warp >> 2;             // rows 32 q.., column half
    const int row = 32 * q + lane;                      // row of the chunk (TMEM lane 64 gi + row)
    float *gc = sm.arr(SM_GC + gi * 256), *ieg = sm.arr(SM_IEG + gi * 256),
          *beg = sm.arr(SM_BEG + gi * 256);
    uint8_t *tu = sm.base + OFF_T + gi * 8192;
    const bool issuer = pw == 0 && lane == 0;  // the group's T store
    for (int i = 0; i < mine; ++i) {
      const int s = i & 1;
      if (group_sync_or(gi, *sm.abort_flag() != 0)) break;
      wait_bar(sm, B_FULL + s, (i >> 1) & 1, 2);
      const float *sb = sm.arr(SM_BETA + (s * 2 + gi) * 256);
      if (pw == 0) {
        if (GATED) {
          float lo, hi;
          warp_scan64(sm.arr(SM_LAM + (s * 2 + gi) * 256), lane, lo, hi);
          gc[lane] = lo;
          gc[lane + 32] = hi;
          ieg[lane] = fast_exp2(-lo);
          ieg[lane + 32] = fast_exp2(-hi);
          beg[lane] = sb[lane] * fast_exp2(lo);
          beg[lane + 32] = sb[lane + 32] * fast_exp2(hi);
        } else {
          beg[lane] = sb[lane];
          beg[lane + 32] = sb[lane + 32];
        }
      }
      if (group_sync_or(gi, *sm.abort_flag() != 0)) break;
      // exact per-entry decay only when the chunk's gate product leaves the
      // range of the ratio form (uniform per chunk)
      const bool ratio = !GATED || gc[63] >= kRatioFloor;
      float *AX = reinterpret_cast<float *>(sm.slot(s) + gi * 16384);

      // ---- A = strictLower(diag(beta) (Gam * K K^T)) from the Gram block of
      //      this chunk (TMEM lanes 64 gi.., columns 64 gi..), into the upper
      //      triangle of the solve array: A_ir sits at (r, i) for i > r, and
      //      as K K^T is symmetric, row r of that triangle comes from TMEM row
      //      r of the Gram block, A_ir = beta_i 2^gc_i * 2^-gc_r * G_ri: each
      //      thread writes its own row in 16-byte pieces.  Rows 32..63 have no
      //      entry in columns 0..31, so that warp has nothing to do ----
      wait_bar(sm, B_GFULL, i & 1, 2);
      tc_fence_after();
      if (!(q == 1 && hf == 0)) {
        const int clo = 32 * hf;
        // ratio regime: row factor 2^-gc_r (column factors beta_i 2^gc_i in beg)
        const float rf = (GATED && ratio) ? ieg[row] : 1.f, gr = GATED ? gc[row] : 0.f;
        float *arow = AX + row * 64;
        const int sw = (row & 7) << 2;
#pragma unroll 1
        for (int jb = clo; jb < clo + 32; jb += 16) {
          uint32_t g[16];
          tmem_ld16(tmem_addr(tmem, 32 * (warp & 3), 64 * gi + jb), g);
          float cf[16];
          if (!GATED || ratio) {
#pragma unroll
            for (int jj = 0; jj < 16; jj += 4) {
              const float4 e4 = *reinterpret_cast<const float4 *>(beg + jb + jj);
              cf[jj] = rf * e4.x;
              cf[jj + 1] = rf * e4.y;
              cf[jj + 2] = rf * e4.z;
              cf[jj + 3] = rf * e4.w;
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) cf[jj] = sb[jb + jj] * fast_exp2(gc[jb + jj] - gr);
          }
          tmem_wait_ld_regs(g);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int c0 = jb + 4 * t;
            // a piece wholly at or below the diagonal holds no entry of A (the
            // lower triangle is written with X later and never read before)
            if (c0 + 3 > row)
              *reinterpret_cast<float4 *>(arow + (c0 ^ sw)) =
                  make_float4(cf[4 * t] * __uint_as_float(g[4 * t]),
                              cf[4 * t + 1] * __uint_as_float(g[4 * t + 1]),
                              cf[4 * t + 2] * __uint_as_float(g[4 * t + 2]),
                              cf[4 * t + 3] * __uint_as_float(g[4 * t + 3]));
          }
        }
      }
      {
        tc_fence_before();
        arrive_warp(sm.bar(B_GFREE), lane);
      }
      // the T tile is rewritten from here on: the previous store has read it
      if (issuer) bulk_wait_read0();
      if (group_sync_or(gi, *sm.abort_flag() != 0)) break;  // A complete

      // ---- X = (I + A)^{-1}: 16x16 diagonal blocks, one per warp ----
      invert_diag16(AX, tu, sb, 16 * pw, lane);
      group_sync(gi);
      {
        // ---- merge 16 -> 32: X21 = -X22 (A21 X11) in each 32-row half;
        //      warp = (half, 8-column slab), A21 X11 stays in registers ----
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
        frag_to_t(tu, o + 16, n0, z, -1.f, sb, lane);
      }
      group_sync(gi);
      {
        // ---- merge 32 -> 64: rows 32..63, columns 8 pw .. 8 pw + 7 of X,
        //      straight into the T tile ----
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
        frag_to_t(tu, 32, n0, z[0], -1.f, sb, lane);
        frag_to_t(tu, 48, n0, z[1], -1.f, sb, lane);
      }
      fence_proxy_async_smem();
      group_sync(gi);  // the T tile is complete; the solve array is no longer read
      if (issuer) {
        const long long c = 2 * pair_of(i) + gi;
        if (c < p.total) {
          tma_store_3d(&map_t, tu, 0, 0, (int)c);
          bulk_commit();
        }
        mbar_arrive(sm.bar(B_FREE + s));
      }
    }
    // every store has completed before the CTA ends
    if (issuer) bulk_wait0();
  }

  // ---- teardown ----
  tc_fence_before();
  __syncthreads();
  if (warp == 9 && !*sm.keep_tmem()) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

}  // namespace

bool ut_supports(const FwdArgs &a) {
  return a.bf16 && a.dk == D && a.chunk == C && a.T > 0 && a.L < (int64_t(1) << 30) &&
         a.B * a.H < (int64_t(1) << 31) && a.B * a.H * ((a.L + C - 1) / C) < (int64_t(1) << 31);
}

int64_t ut_workspace_bytes(const FwdArgs &a) {
  return a.B * a.H * ((a.L + C - 1) / C) * (int64_t)(C * C * 2);
}

cudaError_t make_t_map(CUtensorMap *map, const void *t_mat, int64_t total_chunks) {
  return make_map_3d_bf16_sw128(map, t_mat, C, C, (uint64_t)total_chunks, C, C, 1);
}

cudaError_t launch_ut(const FwdArgs &a, void *t_mat, cudaStream_t s) {
  if (!ut_supports(a)) return cudaErrorNotSupported;
  const int nt = (int)((a.L + C - 1) / C);
  const int64_t total = a.B * a.H * nt;
  CUtensorMap mk, mt;
  cudaError_t e;
  if ((e = make_map_4d_bf16(&mk, a.k, D, a.H, a.L, a.B, 64, 1, 64, 1, true)) != cudaSuccess) return e;
  if ((e = make_t_map(&mt, t_mat, total)) != cudaSuccess) return e;
  UtParams p;
  p.beta = a.beta;
  p.g = a.g;
  p.H = (int)a.H;
  p.T = (int)a.T;
  p.L = (int)a.L;
  p.n_h = a.n_h;
  p.nchunks = nt;
  p.total = total;
  p.pairs = (total + 1) / 2;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long grid = p.pairs < (long long)UT_CTAS_PER_SM * sms ? p.pairs : (long long)UT_CTAS_PER_SM * sms;
  auto kern = a.g ? ut_kernel<true> : ut_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)UT_SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)grid, UT_THREADS, UT_SMEM_ALLOC, s>>>(mk, mt, p);
  return cudaGetLastError();
}

cudaError_t read_and_clear_ut_error(unsigned int *word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, g_ut_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_ut_error, &zero, sizeof(unsigned int));
}

}  // namespace delta
