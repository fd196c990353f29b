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
//   Vt   = U - W S                               (pseudo-values)
//   O    = (Q * exp(gc)) S + (Q K^T * Gam * M) Vt   (token readout rows only)
//   S   <- exp(gc_C) S + (K * exp(gc_C - gc))^T Vt
//
// Design (one CTA per (b, h) head, the 128x128 state on chip for the whole
// sequence): everything is computed TRANSPOSED so that every tensor-core
// product has M = 128 (the dk or dv axis) and the state S^T lives in TMEM as
// an fp32 accumulator [dv lanes x dk columns]:
//
//   G     = [K; Q] K^T                 SS  M=128 N=64  K=128   (TMEM)
//   U^T   = V^T T^T                    SS  M=128 N=64  K=64    (TMEM, becomes Vt^T)
//   W^T   = K^T (T diag(exp gc))^T     SS  M=128 N=64  K=64    (TMEM -> smem bf16)
//   Vt^T += S^T (-W^T)                 TS  M=128 N=64  K=128   (A = S^T bf16 in TMEM)
//   S^T  += (Vt^T diag(exp(gc_C-gc))) K  TS M=128 N=128 K=64   (S^T pre-scaled by exp gc_C)
//   O1^T  = S^T Q^T                    TS  M=128 N=64  K=128
//   O2^T  = Vt^T P^T                   TS  M=128 N=64  K=64    (A = Vt^T bf16 in TMEM)
//   out   = exp(gc) * O1 + O2          (epilogue; O2 accumulates into O1 when ungated)
//
// W and U never leave the SM.  HBM traffic is q, k, v, beta, g in and out,
// h0/hT once per head.  The UT solve runs on the CUDA cores: 16x16 diagonal
// blocks by forward substitution in registers (rows exchanged with warp
// shuffles), then two block merges on the warp-level tensor cores (tf32).
//
// Warp roles (320 threads):
//   warp 0      TMA producer: K/Q/V tiles (128-byte swizzle, 3 stages, the
//               next chunk prefetched into L2) + beta/log-gate rows
//   warp 1      TMEM owner and the single MMA-issuing thread
//   warps 2-5   "prep": G -> A, P -> UT solve -> T tiles     (S-independent)
//   warps 6-9   "chain": Vt^T -> bf16 TMEM operands, S^T -> bf16 copy and
//               gate decay, W^T -> smem operand, output epilogue, final state
// The prep stage of chunk n+1 overlaps the state-dependent chain of chunk n.
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
constexpr int kThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLogGateFloor = -80.0f;

// ---- shared memory layout (offsets from a 1024-byte aligned base) ----
constexpr uint32_t STAGE_BYTES = 49152;  // [K0 | Q0 | K1 | Q1] 32 KB + [V0 | V1] 16 KB
constexpr uint32_t OFF_W = NS * STAGE_BYTES;     // W^T bf16 [128 d][64 c], MN-major
constexpr uint32_t OFF_TU = OFF_W + 16384;       // T    bf16 [64][64], K-major
constexpr uint32_t OFF_TW = OFF_TU + 8192;       // T diag(exp gc)
constexpr uint32_t OFF_P = OFF_TW + 8192;        // 2 x P bf16 [64][64]
constexpr uint32_t OFF_A = OFF_P + 16384;        // A^T fp32 [64][64] (entry (j, i) = A_ij)
constexpr uint32_t OFF_X = OFF_A + 16384;        // X = (I + A)^{-1} fp32 [64][64]
constexpr uint32_t SMEM_TOTAL = OFF_X + 16384;
// A^T rows 32..63 only ever hold entries of columns 32..63 (A_ij with
// i > j >= 32): the first 128 bytes of each of those rows are free and carry
// the small per-chunk arrays and the barriers, one 128-byte slice per row.
constexpr int SL_BETA = 0;    // [NS] arrays of 64 floats, 2 slices each
constexpr int SL_LAM = SL_BETA + 2 * NS;
constexpr int SL_GCP = SL_LAM + 2 * NS;
constexpr int SL_DEC = SL_GCP + 2;   // [2]
constexpr int SL_GAM = SL_DEC + 4;   // [2]
constexpr int SL_BGC = SL_GAM + 4;
constexpr int SL_BAR = SL_BGC + 2;   // 16 barriers per slice
constexpr int NBARS = 2 * NS + 14;
constexpr int SL_MISC = SL_BAR + (NBARS + 15) / 16;
static_assert(SL_MISC < 32, "small region must fit in the free slices of A^T");
constexpr uint32_t SMEM_ALLOC = SMEM_TOTAL + 1024;
static_assert(SMEM_ALLOC <= 232448, "shared memory budget");

// ---- TMEM columns ----
constexpr uint32_t TM_S = 0;        // S^T fp32            [dv][dk]   128 cols
constexpr uint32_t TM_SBF = 128;    // 2 x S^T bf16 (packed)         2x64 cols
constexpr uint32_t TM_GW = 256;     // G, then W^T fp32                64 cols
constexpr uint32_t TM_UV = 320;     // U^T -> Vt^T -> (gated) O2^T     64 cols
constexpr uint32_t TM_O = 384;      // O1^T fp32                       64 cols
constexpr uint32_t TM_VBF = 448;    // Vt^T bf16 (packed)              32 cols
constexpr uint32_t TM_VDEC = 480;   // Vt^T diag(exp(gc_C - gc)) bf16  32 cols
constexpr uint32_t TM_COLS = 512;

// ---- barrier indices ----
enum {
  B_FULL = 0,             // [NS] producer -> consumers (count 2 + tx)
  B_EMPTY = NS,           // [NS] MMA commit -> producer
  B_GFULL = 2 * NS,       // MMA -> prep: G ready in TMEM
  B_TFULL,                // prep -> MMA: T, P in smem (128)
  B_WFULL,                // MMA -> chain, prep: U, W^T ready (T tiles consumed)
  B_WREADY,               // chain -> MMA: W in smem, TMEM GW free (128)
  B_WFREE,                // MMA -> chain: W smem consumed
  B_SREADY,               // chain -> MMA: S^T bf16 ready, S^T decayed (128)
  B_VTFULL,               // MMA -> chain: Vt^T ready
  B_VTREADY,              // chain -> MMA: Vt^T bf16 operands ready (128)
  B_SFULL,                // MMA -> chain: S^T updated
  B_OFULL,                // MMA -> chain: O1 (and O2) complete
  B_OFREE,                // chain -> MMA: O1 / O2 read (128)
  B_PQFREE0,              // MMA -> prep: P buffer 0 free
  B_PQFREE1,              //                          1
  B_DRAIN,                // MMA: everything issued has completed
};

struct TcParams {
  const float *beta, *g, *h0;
  __nv_bfloat16 *out;
  float *hT;
  int H, T, L, n_h, nchunks;
};

// 64 floats split over two 128-byte slices.
struct Arr64 {
  uint8_t *p0, *p1;
  __device__ float &operator[](int e) const {
    return reinterpret_cast<float *>(e < 32 ? p0 : p1)[e & 31];
  }
};

struct Smem {
  uint8_t *base;
  __device__ uint8_t *stage(int s) const { return base + s * STAGE_BYTES; }
  __device__ uint8_t *slice(int k) const { return base + OFF_A + (32 + k) * 256; }
  __device__ Arr64 arr(int k) const { return Arr64{slice(k), slice(k + 1)}; }
  __device__ Arr64 beta(int s) const { return arr(SL_BETA + 2 * s); }
  __device__ Arr64 lam(int s) const { return arr(SL_LAM + 2 * s); }
  __device__ Arr64 gcp() const { return arr(SL_GCP); }
  __device__ Arr64 dec(int b) const { return arr(SL_DEC + 2 * b); }
  __device__ Arr64 gam(int b) const { return arr(SL_GAM + 2 * b); }
  __device__ Arr64 bgc() const { return arr(SL_BGC); }
  __device__ uint64_t *bar(int i) const {
    return reinterpret_cast<uint64_t *>(slice(SL_BAR + (i >> 4))) + (i & 15);
  }
  __device__ uint32_t *tmem_slot() const { return reinterpret_cast<uint32_t *>(slice(SL_MISC)); }
  __device__ volatile int *abort_flag() const { return reinterpret_cast<volatile int *>(slice(SL_MISC) + 4); }
  __device__ float *At() const { return reinterpret_cast<float *>(base + OFF_A); }
  __device__ float *X() const { return reinterpret_cast<float *>(base + OFF_X); }
};

// Bounded wait that also gives up at once when another role has aborted.
__device__ __forceinline__ bool wait_bar(const Smem &sm, int idx, uint32_t parity, int role) {
  uint64_t *b = sm.bar(idx);
  for (uint32_t i = 0; i < (1u << 22); ++i) {
    if (mbar_try_wait(b, parity)) return true;
    if ((i & 63) == 63 && *sm.abort_flag()) return false;
  }
  *sm.abort_flag() = 1;
  atomicCAS(&g_tc_error, 0u, (unsigned)(1 + role) | ((unsigned)idx << 8));
  return false;
}

// fp32 64x64 matrices in shared memory are stored row-major with the column
// XOR-swizzled by the row (bits 2..4), which keeps float4 runs along a row
// contiguous and makes the tf32 MMA fragment loads below conflict-free.
__device__ __forceinline__ int swz(int r, int c) { return r * 64 + (c ^ ((r & 7) << 2)); }


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

// One warp: D(16x8) (+)= M1[r0.., k0..k0+K) * M2[k2.., n0..n0+8) (and a second
// tile at n0 + 8 when TWO) with both operands read from swizzled fp32 smem;
// M1 is read through its transpose when `m1t` (A^T holds A).  The fp32 bits
// are fed to the tf32 MMA as they are (the low mantissa bits are ignored).
template <int K, bool TWO>
__device__ __forceinline__ void warp_gemm(float (&d0)[4], float (&d1)[4], const float *M1, bool m1t,
                                          int r0, int k0, const float *M2, int k2, int n0, int lane) {
  const int g = lane >> 2, t = lane & 3;
  uint32_t a[K / 8][4], b0[K / 8][2], b1[K / 8][2];
#pragma unroll
  for (int ks = 0; ks < K / 8; ++ks) {
    const int c = k0 + 8 * ks;
    if (m1t) {
      a[ks][0] = __float_as_uint(M1[swz(c + t, r0 + g)]);
      a[ks][1] = __float_as_uint(M1[swz(c + t, r0 + g + 8)]);
      a[ks][2] = __float_as_uint(M1[swz(c + t + 4, r0 + g)]);
      a[ks][3] = __float_as_uint(M1[swz(c + t + 4, r0 + g + 8)]);
    } else {
      a[ks][0] = __float_as_uint(M1[swz(r0 + g, c + t)]);
      a[ks][1] = __float_as_uint(M1[swz(r0 + g + 8, c + t)]);
      a[ks][2] = __float_as_uint(M1[swz(r0 + g, c + t + 4)]);
      a[ks][3] = __float_as_uint(M1[swz(r0 + g + 8, c + t + 4)]);
    }
    const int kr = k2 + 8 * ks;
    b0[ks][0] = __float_as_uint(M2[swz(kr + t, n0 + g)]);
    b0[ks][1] = __float_as_uint(M2[swz(kr + t + 4, n0 + g)]);
    if (TWO) {
      b1[ks][0] = __float_as_uint(M2[swz(kr + t, n0 + 8 + g)]);
      b1[ks][1] = __float_as_uint(M2[swz(kr + t + 4, n0 + 8 + g)]);
    }
  }
#pragma unroll
  for (int ks = 0; ks < K / 8; ++ks) {
    mma_tf32(d0, a[ks], b0[ks]);
    if (TWO) mma_tf32(d1, a[ks], b1[ks]);
  }
}

// T_U = x * beta_j and T_W = x * beta_j exp(gc_j) of a 16x8 fragment of
// (scale * D) at rows r0.., columns n0.. of the bf16 T tiles.
__device__ __forceinline__ void frag_to_t(uint8_t *tu, uint8_t *tw, int r0, int n0,
                                          const float (&d)[4], float scale, const Arr64 &bcol,
                                          const Arr64 &bgcol, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const int c = n0 + 2 * t;
  const float b0 = bcol[c], b1 = bcol[c + 1], w0 = bgcol[c], w1 = bgcol[c + 1];
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

// Inclusive prefix sum over the 64 log-gate entries of a chunk, per warp:
// lane holds entries lane and lane + 32.
__device__ __forceinline__ void warp_scan64(const Arr64 &lam, int lane, float &lo, float &hi) {
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

// 16-byte store of 8 packed bf16 values into a swizzled tile row.
__device__ __forceinline__ void st_chunk(uint8_t *tile, uint32_t off, const uint32_t (&p)[4]) {
  *reinterpret_cast<uint4 *>(tile + off) = make_uint4(p[0], p[1], p[2], p[3]);
}

template <bool GATED>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem sm;
  sm.base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                        ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x;
  const int b = bh / p.H, h = bh % p.H;
  const int n_h = p.n_h, NT = p.nchunks;
  const int QR = n_h == 1 ? 64 : 32;  // query rows loaded per chunk

  // ---- set-up: zero shared memory, init barriers, allocate TMEM ----
  {
    uint4 *z = reinterpret_cast<uint4 *>(sm.base);
    for (uint32_t i = tid; i < SMEM_TOTAL / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(sm.bar(B_FULL + s), 2);
      mbar_init(sm.bar(B_EMPTY + s), 1);
    }
    mbar_init(sm.bar(B_GFULL), 1);
    mbar_init(sm.bar(B_TFULL), 128);
    mbar_init(sm.bar(B_WFULL), 1);
    mbar_init(sm.bar(B_WREADY), 128);
    mbar_init(sm.bar(B_WFREE), 1);
    mbar_init(sm.bar(B_SREADY), 128);
    mbar_init(sm.bar(B_VTFULL), 1);
    mbar_init(sm.bar(B_VTREADY), 128);
    mbar_init(sm.bar(B_SFULL), 1);
    mbar_init(sm.bar(B_OFULL), 1);
    mbar_init(sm.bar(B_OFREE), 128);
    mbar_init(sm.bar(B_PQFREE0), 1);
    mbar_init(sm.bar(B_PQFREE1), 1);
    mbar_init(sm.bar(B_DRAIN), 1);
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
        mbar_arrive_expect_tx(sm.bar(B_FULL + s), 2u * (8192u + 8192u + (uint32_t)QR * 128u));
        uint64_t *fb = sm.bar(B_FULL + s);
        tma_load_4d(st + 0, &map_k, fb, 0, h, e0, b);
        tma_load_4d(st + 16384, &map_k, fb, 64, h, e0, b);
        tma_load_4d(st + 8192, &map_q, fb, 0, h, t_lo, b);
        tma_load_4d(st + 24576, &map_q, fb, 64, h, t_lo, b);
        tma_load_4d(st + 32768, &map_v, fb, 0, h, e0, b);
        tma_load_4d(st + 40960, &map_v, fb, 64, h, e0, b);
      }
      const Arr64 sb = sm.beta(s), sl = sm.lam(s);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int r = lane + 32 * k;
        const int e = e0 + r;
        float bt = 0.f, lg = 0.f;
        if (e < p.L) {
          bt = p.beta[((size_t)b * p.L + e) * p.H + h];
          if (GATED && (e % n_h) == 0)
            lg = fmaxf(logf(p.g[((size_t)b * p.T + e / n_h) * p.H + h]), kLogGateFloor) * kLog2e;
        }
        sb[r] = bt;
        sl[r] = lg;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(B_FULL + s));
    }
  } else if (warp == 1) {
    // ===================================================== MMA issuer
    if (lane == 0) {
      bool ok = true;
      const uint32_t id_g = idesc_bf16(128, 64, false, false);
      const uint32_t id_uw = idesc_bf16(128, 64, true, false);
      const uint32_t id_vt = idesc_bf16(128, 64, false, true, true);  // B = W^T MN-major, negated
      const uint32_t id_o = idesc_bf16(128, 64, false, false);
      const uint32_t id_s = idesc_bf16(128, 128, false, true);
      const uint32_t a_tu = smem_u32(sm.base + OFF_TU), a_tw = smem_u32(sm.base + OFF_TW);
      const uint32_t a_w = smem_u32(sm.base + OFF_W);

      auto issue_g = [&](int m) -> bool {  // G(m) = [K;Q] K^T
        const int s = m % NS;
        if (!wait_bar(sm, B_FULL + s, (m / NS) & 1, 1)) return false;
        tc_fence_after();
        const uint32_t kq = smem_u32(sm.stage(s));
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
          mma_ss(tmem + TM_GW, sdesc_sw128(kq + off, 0, 1024), sdesc_sw128(kq + off, 0, 1024),
                 id_g, k > 0);
        }
        mma_commit(sm.bar(B_GFULL));
        return true;
      };
      auto issue_w = [&](int m) {  // W(m)^T = K^T (T diag(exp gc))^T
        const uint32_t kq = smem_u32(sm.stage(m % NS));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tmem + TM_GW, sdesc_sw128(kq + k * 2048, 16384, 1024),
                 sdesc_sw128(a_tw + k * 32, 0, 1024), id_uw, k > 0);
      };
      auto issue_u = [&](int m) {  // U(m)^T = V^T T^T
        const uint32_t vv = smem_u32(sm.stage(m % NS)) + 32768;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tmem + TM_UV, sdesc_sw128(vv + k * 2048, 8192, 1024),
                 sdesc_sw128(a_tu + k * 32, 0, 1024), id_uw, k > 0);
      };

      ok = issue_g(0) && wait_bar(sm, B_TFULL, 0, 1);
      if (ok) {
        tc_fence_after();
        issue_w(0);
        issue_u(0);
        mma_commit(sm.bar(B_WFULL));
      }
      for (int n = 0; ok && n < NT; ++n) {
        const int s = n % NS;
        const uint32_t kq = smem_u32(sm.stage(s));
        const uint32_t sbf = tmem + TM_SBF + (n & 1) * 64;
        if (!wait_bar(sm, B_WREADY, n & 1, 1)) break;
        // G of the next chunk as soon as W^T(n) has left TMEM: its solve
        // overlaps this chunk's state-dependent chain
        if (n + 1 < NT && !issue_g(n + 1)) break;
        if (!wait_bar(sm, B_SREADY, n & 1, 1)) break;
        tc_fence_after();
        // Vt^T = U^T - S^T W^T                                (critical chain)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ts(tmem + TM_UV, sbf + k * 8, sdesc_sw128(a_w + k * 2048, 8192, 1024), id_vt, true);
        mma_commit(sm.bar(B_VTFULL));
        mma_commit(sm.bar(B_WFREE));
        if (!wait_bar(sm, B_VTREADY, n & 1, 1)) break;
        tc_fence_after();
        // S^T += Vt^T diag(dec) K                             (critical chain)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ts(tmem + TM_S, tmem + (GATED ? TM_VDEC : TM_VBF) + k * 8,
                 sdesc_sw128(kq + k * 2048, 16384, 1024), id_s, true);
        mma_commit(sm.bar(B_SFULL));
        // O1^T = S^T Q^T ; O2^T = Vt^T P^T (into the same accumulator when ungated)
        if (n >= 1 && !wait_bar(sm, B_OFREE, (n - 1) & 1, 1)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ts(tmem + TM_O, sbf + k * 8,
                 sdesc_sw128(kq + 8192 + (k >> 2) * 16384 + (k & 3) * 32, 0, 1024), id_o, k > 0);
        const uint32_t pb = smem_u32(sm.base + OFF_P) + (n & 1) * 8192;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ts(tmem + (GATED ? TM_UV : TM_O), tmem + TM_VBF + k * 8,
                 sdesc_sw128(pb + k * 32, 0, 1024), id_o, GATED ? (k > 0) : true);
        mma_commit(sm.bar(B_OFULL));
        mma_commit(sm.bar(B_EMPTY + s));
        mma_commit(sm.bar(B_PQFREE0 + (n & 1)));
        // W (and U) of the next chunk
        if (n + 1 < NT) {
          if (!wait_bar(sm, B_TFULL, (n + 1) & 1, 1)) break;
          tc_fence_after();
          issue_w(n + 1);
          if (GATED) {
            // U overwrites O2(n) in TMEM: wait until the epilogue has read it
            if (!wait_bar(sm, B_OFREE, n & 1, 1)) break;
            tc_fence_after();
          }
          issue_u(n + 1);
          mma_commit(sm.bar(B_WFULL));
        }
      }
      mma_commit(sm.bar(B_DRAIN));
      wait_bar(sm, B_DRAIN, 0, 1);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ===================================================== prep warps
    const int q4 = warp & 3;              // TMEM lane quarter
    const int L = q4 * 32 + lane;         // TMEM lane of this thread
    const int pw = warp - 2;              // 0..3
    const int pt = tid - 64;              // 0..127 within the group
    float *At = sm.At();                  // A^T: entry (j, i) holds A_ij
    float *X = sm.X();
    const Arr64 gcp = sm.gcp();
    const Arr64 bgc = sm.bgc();
    uint8_t *tu = sm.base + OFF_TU;
    uint8_t *tw = sm.base + OFF_TW;
    for (int m = 0; m < NT; ++m) {
      const int s = m % NS;
      // a failed wait sets the abort flag; every thread still reaches the
      // next named barrier and all of them leave together after it
      wait_bar(sm, B_FULL + s, (m / NS) & 1, 2);
      const Arr64 sb = sm.beta(s);
      if (GATED && warp == 2) {
        float lo, hi;
        warp_scan64(sm.lam(s), lane, lo, hi);
        gcp[lane] = lo;
        gcp[lane + 32] = hi;
      }
      if (named_sync_or(1, *sm.abort_flag() != 0)) break;
      if (pt < 64) bgc[pt] = GATED ? sb[pt] * fast_exp2(gcp[pt]) : sb[pt];
      const int e0 = m * C;
      const int t_lo = e0 / n_h;
      int t_hi = (e0 + C - n_h) / n_h;
      if (t_hi > p.T - 1) t_hi = p.T - 1;
      const int Cp = t_hi - t_lo + 1;  // readout rows of this chunk

      // ---- one row of G = [K;Q] K^T per thread (TMEM lane L) ----
      wait_bar(sm, B_GFULL, m & 1, 2);
      tc_fence_after();
      uint32_t g[64];
      tmem_ld32(tmem_addr(tmem + TM_GW, q4 * 32, 0), *reinterpret_cast<uint32_t (*)[32]>(&g[0]));
      tmem_ld32(tmem_addr(tmem + TM_GW, q4 * 32, 32), *reinterpret_cast<uint32_t (*)[32]>(&g[32]));
      tmem_wait_ld_regs(g);
      tc_fence_before();

      if (L < 64) {
        // ---- row i of A = beta_i Gam_ij (k_i . k_j), j < i, into A^T; blocks
        //      right of the diagonal block are never read and not stored ----
        const int i = L, blk = i >> 4;
        const float bi = sb[i];
        const float gi = GATED ? gcp[i] : 0.f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          if ((j >> 4) > blk) continue;
          const float v = bi * __uint_as_float(g[j]) * (GATED ? fast_exp2(gi - gcp[j]) : 1.f);
          At[swz(j, i)] = ((j >> 4) == blk && j >= i) ? 0.f : v;
        }
      } else {
        // ---- row r of P = (q_r . k_j) Gam, j <= pos(r) ----
        const int r = L - 64;
        const bool valid = r < Cp;
        const int pos = valid ? (t_lo + r) * n_h + (n_h - 1) - e0 : -1;
        const float gp = (GATED && valid) ? gcp[pos] : 0.f;
        if (m >= 2) wait_bar(sm, B_PQFREE0 + (m & 1), ((m >> 1) - 1) & 1, 2);
        uint8_t *ptile = sm.base + OFF_P + (m & 1) * 8192;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint32_t pk[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j0 = q * 8 + 2 * u;
            const float v0 =
                (j0 <= pos) ? __uint_as_float(g[j0]) * (GATED ? fast_exp2(gp - gcp[j0]) : 1.f) : 0.f;
            const float v1 = (j0 + 1 <= pos)
                                 ? __uint_as_float(g[j0 + 1]) * (GATED ? fast_exp2(gp - gcp[j0 + 1]) : 1.f)
                                 : 0.f;
            pk[u] = pack_bf16(v0, v1);
          }
          st_chunk(ptile, sw128_offset(r, q * 8, 64), pk);
        }
      }
      // the T tiles are rewritten from here on: U/W of the previous chunk
      // must have consumed them
      if (m >= 1) wait_bar(sm, B_WFULL, (m - 1) & 1, 2);
      if (named_sync_or(1, *sm.abort_flag() != 0)) break;  // A^T, P, bgc ready

      {
        // ---- 16x16 diagonal blocks of X = (I + A)^{-1}: column jj of block
        //      blk, rows split over a lane pair, right-looking forward
        //      substitution; X and the T tiles written as columns finish ----
        const int blk = pt >> 5, jj = (pt >> 1) & 15, half = pt & 1, o = 16 * blk;
        const int col = o + jj;
        const float bcol = sb[col], wcol = bgc[col];
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        float4 n0 = *reinterpret_cast<const float4 *>(At + swz(o, o + 8 * half));
        float4 n1 = *reinterpret_cast<const float4 *>(At + swz(o, o + 8 * half + 4));
#pragma unroll
        for (int mm = 0; mm < 16; ++mm) {
          const float cur[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
          if (mm + 1 < 16) {
            n0 = *reinterpret_cast<const float4 *>(At + swz(o + mm + 1, o + 8 * half));
            n1 = *reinterpret_cast<const float4 *>(At + swz(o + mm + 1, o + 8 * half + 4));
          }
          const int owner = mm >> 3;
          const float xo = (mm == jj) ? 1.f : ((mm > jj) ? -acc[mm & 7] : 0.f);
          const float x = __shfl_sync(0xffffffffu, xo, (lane & ~1) | owner);
          if (half == owner) {
            X[swz(o + mm, col)] = x;
            const uint32_t off = sw128_offset(o + mm, col, 64);
            *reinterpret_cast<__nv_bfloat16 *>(tu + off) = __float2bfloat16_rn(x * bcol);
            *reinterpret_cast<__nv_bfloat16 *>(tw + off) = __float2bfloat16_rn(x * wcol);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (8 * half + i > mm) acc[i] = fmaf(cur[i], x, acc[i]);
        }
      }
      named_sync(1);
      {
        // ---- merge 16 -> 32: X21' = -X22' (A21' X11') in each 32-row half ----
        const int o = (pw >> 1) * 32, nt = pw & 1;
        float y[4] = {0.f, 0.f, 0.f, 0.f}, unused[4];
        warp_gemm<16, false>(y, unused, At, true, o + 16, o, X, o, o + 8 * nt, lane);
        // scratch: the unused upper-right 32x32 block of X
        const int sr = (pw >> 1) * 16, scol = 32 + (pw >> 1) * 16 + 8 * nt;
        warp_store_16x8(X, sr, scol, y, 1.f, lane);
        __syncwarp();
        float z[4] = {0.f, 0.f, 0.f, 0.f};
        warp_gemm<16, false>(z, unused, X, false, o + 16, o + 16, X, sr, scol, lane);
        warp_store_16x8(X, o + 16, o + 8 * nt, z, -1.f, lane);
        frag_to_t(tu, tw, o + 16, o + 8 * nt, z, -1.f, sb, bgc, lane);
      }
      named_sync(1);
      {
        // ---- merge 32 -> 64: Y = A21 X11 into the upper-right block, then
        //      X21 = -X22 Y straight into the T tiles ----
        const int mr = (pw >> 1) * 16, nc = (pw & 1) * 16;
        float y0[4] = {0.f, 0.f, 0.f, 0.f}, y1[4] = {0.f, 0.f, 0.f, 0.f};
        warp_gemm<32, true>(y0, y1, At, true, 32 + mr, 0, X, 0, nc, lane);
        warp_store_16x8(X, mr, 32 + nc, y0, 1.f, lane);
        warp_store_16x8(X, mr, 32 + nc + 8, y1, 1.f, lane);
        named_sync(1);
        float z0[4] = {0.f, 0.f, 0.f, 0.f}, z1[4] = {0.f, 0.f, 0.f, 0.f};
        warp_gemm<32, true>(z0, z1, X, false, 32 + mr, 32, X, 0, 32 + nc, lane);
        frag_to_t(tu, tw, 32 + mr, nc, z0, -1.f, sb, bgc, lane);
        frag_to_t(tu, tw, 32 + mr, nc + 8, z1, -1.f, sb, bgc, lane);
      }
      fence_proxy_async_smem();
      mbar_arrive(sm.bar(B_TFULL));
    }
  } else {
    // ===================================================== chain warps
    const int q4 = warp & 3;
    const int L = q4 * 32 + lane;  // TMEM lane = value column dv
    // gate of a chunk: 2^(sum of its log2 gates)
    auto chunk_decay = [&](int n) -> float {
      if (!GATED) return 1.f;
      const Arr64 lam = sm.lam(n % NS);
      float t = lam[lane] + lam[lane + 32];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      return fast_exp2(t);
    };
    // W^T of chunk m (TMEM, lane = d) -> bf16 smem operand, row d
    auto convert_w = [&](int m) {
      wait_bar(sm, B_WFULL, m & 1, 3);
      if (m >= 1) wait_bar(sm, B_WFREE, (m - 1) & 1, 3);
      tc_fence_after();
      uint8_t *wt = sm.base + OFF_W;
      uint32_t r[64];
      tmem_ld32(tmem_addr(tmem + TM_GW, q4 * 32, 0), *reinterpret_cast<uint32_t (*)[32]>(&r[0]));
      tmem_ld32(tmem_addr(tmem + TM_GW, q4 * 32, 32), *reinterpret_cast<uint32_t (*)[32]>(&r[32]));
      tmem_wait_ld_regs(r);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint32_t pk[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          pk[u] = pack_bf16(__uint_as_float(r[q * 8 + 2 * u]), __uint_as_float(r[q * 8 + 2 * u + 1]));
        st_chunk(wt, sw128_offset(L, q * 8, 128), pk);
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(sm.bar(B_WREADY));
    };
    // the whole chain group proceeds only if every thread saw chunk 0 arrive
    const bool ok = !named_sync_or(2, !wait_bar(sm, B_FULL + 0, 0, 3));
    // ---- initial state S^T (lane = dv, column = dk) ----
    if (ok) {
      const float d0 = chunk_decay(0);
      const float *h0 = p.h0 ? p.h0 + (size_t)bh * D * D : nullptr;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t f[32], pk[16];
#pragma unroll
        for (int u = 0; u < 32; u += 2) {
          const float x0 = h0 ? h0[(size_t)(c0 + u) * D + L] : 0.f;
          const float x1 = h0 ? h0[(size_t)(c0 + u + 1) * D + L] : 0.f;
          f[u] = __float_as_uint(x0 * d0);
          f[u + 1] = __float_as_uint(x1 * d0);
          pk[u >> 1] = pack_bf16(x0, x1);
        }
        tmem_st32(tmem_addr(tmem + TM_S, q4 * 32, c0), f);
        tmem_st16(tmem_addr(tmem + TM_SBF, q4 * 32, c0 / 2), pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(sm.bar(B_SREADY));
      convert_w(0);
    }
    for (int n = 0; ok && n < NT; ++n) {
      const int s = n % NS;
      const int e0 = n * C;
      const int t_lo = e0 / n_h;
      int t_hi = (e0 + C - n_h) / n_h;
      if (t_hi > p.T - 1) t_hi = p.T - 1;
      const int Cp = t_hi - t_lo + 1;
      // ---- pseudo-values: Vt^T -> bf16 operands ----
      wait_bar(sm, B_VTFULL, n & 1, 3);
      tc_fence_after();
      const Arr64 dec = sm.dec(n & 1);
      const Arr64 gam = sm.gam(n & 1);
      if (GATED) {
        wait_bar(sm, B_FULL + s, (n / NS) & 1, 3);
        if (warp == 6) {
          float lo, hi;
          warp_scan64(sm.lam(s), lane, lo, hi);
          const float tot = __shfl_sync(0xffffffffu, hi, 31);
          dec[lane] = fast_exp2(tot - lo);
          dec[lane + 32] = fast_exp2(tot - hi);
          gam[lane] = fast_exp2(lo);
          gam[lane + 32] = fast_exp2(hi);
        }
        if (named_sync_or(2, *sm.abort_flag() != 0)) break;
      }
      {
        uint32_t r[64];
        tmem_ld32(tmem_addr(tmem + TM_UV, q4 * 32, 0), *reinterpret_cast<uint32_t (*)[32]>(&r[0]));
        tmem_ld32(tmem_addr(tmem + TM_UV, q4 * 32, 32), *reinterpret_cast<uint32_t (*)[32]>(&r[32]));
        tmem_wait_ld_regs(r);
        uint32_t pk[32];
#pragma unroll
        for (int u = 0; u < 32; ++u)
          pk[u] = pack_bf16(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
        tmem_st32(tmem_addr(tmem + TM_VBF, q4 * 32, 0), pk);
        if (GATED) {
#pragma unroll
          for (int u = 0; u < 32; ++u)
            pk[u] = pack_bf16(__uint_as_float(r[2 * u]) * dec[2 * u],
                              __uint_as_float(r[2 * u + 1]) * dec[2 * u + 1]);
          tmem_st32(tmem_addr(tmem + TM_VDEC, q4 * 32, 0), pk);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(sm.bar(B_VTREADY));

      // ---- state: S^T -> bf16 copy for the next chunk (+ its decay), or hT ----
      wait_bar(sm, B_SFULL, n & 1, 3);
      tc_fence_after();
      if (n + 1 < NT) {
        float dn = 1.f;
        if (GATED) {
          wait_bar(sm, B_FULL + (n + 1) % NS, ((n + 1) / NS) & 1, 3);
          dn = chunk_decay(n + 1);
        }
        const uint32_t sbf = tmem + TM_SBF + ((n + 1) & 1) * 64;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 64) {
          uint32_t r[64], pk[32];
          tmem_ld32(tmem_addr(tmem + TM_S, q4 * 32, c0), *reinterpret_cast<uint32_t (*)[32]>(&r[0]));
          tmem_ld32(tmem_addr(tmem + TM_S, q4 * 32, c0 + 32), *reinterpret_cast<uint32_t (*)[32]>(&r[32]));
          tmem_wait_ld_regs(r);
#pragma unroll
          for (int u = 0; u < 32; ++u)
            pk[u] = pack_bf16(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
          tmem_st32(tmem_addr(sbf, q4 * 32, c0 / 2), pk);
          if (GATED) {
#pragma unroll
            for (int u = 0; u < 64; ++u) r[u] = __float_as_uint(__uint_as_float(r[u]) * dn);
            tmem_st32(tmem_addr(tmem + TM_S, q4 * 32, c0), *reinterpret_cast<uint32_t (*)[32]>(&r[0]));
            tmem_st32(tmem_addr(tmem + TM_S, q4 * 32, c0 + 32), *reinterpret_cast<uint32_t (*)[32]>(&r[32]));
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(sm.bar(B_SREADY));
      } else if (p.hT) {
        float *hT = p.hT + (size_t)bh * D * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tmem_addr(tmem + TM_S, q4 * 32, c0), r);
          tmem_wait_ld_regs(r);
#pragma unroll
          for (int u = 0; u < 32; ++u) hT[(size_t)(c0 + u) * D + L] = __uint_as_float(r[u]);
        }
      }
      // ---- outputs of this chunk: o = exp(gc) O1 + O2 per readout row ----
      wait_bar(sm, B_OFULL, n & 1, 3);
      tc_fence_after();
      float o[64];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t r1[32];
        tmem_ld32(tmem_addr(tmem + TM_O, q4 * 32, hf * 32), r1);
        if (GATED) {
          uint32_t r2[32];
          tmem_ld32(tmem_addr(tmem + TM_UV, q4 * 32, hf * 32), r2);
          tmem_wait_ld_regs(r1);
          tmem_wait_ld_regs(r2);
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const int rr = hf * 32 + u;
            const int pos = (t_lo + rr) * n_h + (n_h - 1) - e0;
            const float gm = rr < Cp ? gam[pos] : 0.f;
            o[rr] = fmaf(gm, __uint_as_float(r1[u]), __uint_as_float(r2[u]));
          }
        } else {
          tmem_wait_ld_regs(r1);
#pragma unroll
          for (int u = 0; u < 32; ++u) o[hf * 32 + u] = __uint_as_float(r1[u]);
        }
      }
      tc_fence_before();
      mbar_arrive(sm.bar(B_OFREE));
      // W^T of the next chunk before the stores: it gates the next chain step
      if (n + 1 < NT) convert_w(n + 1);
      // 8x8 transposes within groups of 8 lanes: lane k of a group then holds
      // 8 consecutive value columns of row 8 rg + k -> one 16-byte store
      {
        const int k = lane & 7;
        const size_t col = (size_t)q4 * 32 + (lane >> 3) * 8;
#pragma unroll
        for (int rg = 0; rg < 8; ++rg) {
          float v[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = o[rg * 8 + j];
#pragma unroll
          for (int sh = 1; sh < 8; sh <<= 1) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (j & sh) continue;
              const float send = (k & sh) ? v[j] : v[j | sh];
              const float recv = __shfl_xor_sync(0xffffffffu, send, sh);
              if (k & sh)
                v[j] = recv;
              else
                v[j | sh] = recv;
            }
          }
          const int row = rg * 8 + k;
          if (row < Cp) {
            const uint4 pkt = make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]),
                                         pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
            *reinterpret_cast<uint4 *>(p.out + (((size_t)b * p.T + t_lo + row) * p.H + h) * D + col) = pkt;
          }
        }
      }
    }
  }

  // ---- teardown ----
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

}  // namespace

bool chunk_tc_supports(const FwdArgs &a) {
  return a.bf16 && a.dk == D && a.dv == D && a.chunk == C && a.T > 0 &&
         a.L < (int64_t(1) << 30) && a.B * a.H < (int64_t(1) << 31);
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
  kern<<<(unsigned)(a.B * a.H), kThreads, SMEM_ALLOC, s>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace delta
