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
//   O^T   = S^T (Q * exp gc)^T         TS  M=128 N=64  K=128
//   O^T  += Vt^T P^T                   TS  M=128 N=64  K=64    (A = Vt^T bf16 in TMEM)
//   S^T  += (Vt^T diag(exp(gc_C-gc))) K  TS M=128 N=128 K=64   (S^T pre-scaled by exp gc_C)
//
// W and U never leave the SM.  HBM traffic is q, k, v, beta, g in and out,
// h0/hT once per head.
//
// Warp roles (320 threads):
//   warp 0      TMA producer: K/Q/V tiles (128-byte swizzle) + beta/log-gate rows
//   warp 1      TMEM owner and the single MMA-issuing thread
//   warps 2-5   "prep": G -> UT solve -> T tiles, P = Q K^T * Gam, gated Q,
//               then W^T (TMEM) -> bf16 smem operand        (S-independent)
//   warps 6-9   "chain": Vt^T -> bf16 TMEM operands, S^T -> bf16 copy and
//               gate decay, output epilogue, final state     (S-dependent)
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
constexpr int NS = 2;  // TMA stages
constexpr int kThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLogGateFloor = -80.0f;

// ---- shared memory layout (offsets from a 1024-byte aligned base) ----
constexpr uint32_t STAGE_BYTES = 49152;  // [K0 | Q0 | K1 | Q1] 32 KB + [V0 | V1] 16 KB
constexpr uint32_t OFF_W = NS * STAGE_BYTES;     // W^T bf16 [128 d][64 c], MN-major
constexpr uint32_t OFF_TU = OFF_W + 16384;       // T    bf16 [64][64], K-major
constexpr uint32_t OFF_TW = OFF_TU + 8192;       // T diag(exp gc)
constexpr uint32_t OFF_P = OFF_TW + 8192;        // 2 x P bf16 [64][64]
constexpr uint32_t OFF_QG = OFF_P + 16384;       // 2 x gated Q, interleaved blocks
constexpr uint32_t OFF_AT = OFF_QG + 32768;      // A^T fp32 [64][64]
constexpr uint32_t OFF_X = OFF_AT + 16384;       // X = (I + A)^{-1} fp32 [64][64]
constexpr uint32_t OFF_STG = OFF_X + 16384;      // output staging bf16 [64][128]
constexpr uint32_t OFF_SMALL = OFF_STG + 16384;
// small region
constexpr uint32_t SM_BETA = 0;                  // float [NS][64]
constexpr uint32_t SM_LAM = SM_BETA + NS * 256;  // float [NS][64]  (log2 units)
constexpr uint32_t SM_GCP = SM_LAM + NS * 256;   // float [64] prep's cumsum (log2 units)
constexpr uint32_t SM_DEC = SM_GCP + 256;        // float [64] chain's exp2(gc_C - gc)
constexpr uint32_t SM_BAR = SM_DEC + 256;        // mbarriers
constexpr int NBARS = 2 * NS + 15;
constexpr uint32_t SM_TMEM = SM_BAR + NBARS * 8;
constexpr uint32_t SM_ABORT = SM_TMEM + 4;
constexpr uint32_t SMALL_BYTES = SM_ABORT + 12;
constexpr uint32_t SMEM_TOTAL = OFF_SMALL + SMALL_BYTES;
constexpr uint32_t SMEM_ALLOC = SMEM_TOTAL + 1024;
static_assert(SMEM_ALLOC <= 232448, "shared memory budget");

// ---- TMEM columns ----
constexpr uint32_t TM_S = 0;        // S^T fp32            [dv][dk]   128 cols
constexpr uint32_t TM_SBF = 128;    // 2 x S^T bf16 (packed)         2x64 cols
constexpr uint32_t TM_GW = 256;     // G, then W^T fp32                64 cols
constexpr uint32_t TM_UV = 320;     // U^T -> Vt^T fp32                64 cols
constexpr uint32_t TM_O = 384;      // O^T fp32                        64 cols
constexpr uint32_t TM_VBF = 448;    // Vt^T bf16 (packed)              32 cols
constexpr uint32_t TM_VDEC = 480;   // Vt^T diag(exp(gc_C - gc)) bf16  32 cols
constexpr uint32_t TM_COLS = 512;

// ---- barrier indices ----
enum {
  B_FULL = 0,             // [NS] producer -> consumers (count 2 + tx)
  B_EMPTY = NS,           // [NS] MMA commit -> producer
  B_GFULL = 2 * NS,       // MMA -> prep: G ready in TMEM
  B_TFULL,                // prep -> MMA: T, P, gated Q in smem (128)
  B_WFULL,                // MMA -> prep, chain: U, W^T ready (T tiles free)
  B_WREADY,               // chain -> MMA: W in smem, TMEM W free (128)
  B_WFREE,                // MMA -> chain: W smem consumed
  B_SREADY,               // chain -> MMA: S^T bf16 ready, S^T decayed (128)
  B_VTFULL,               // MMA -> chain: Vt^T ready
  B_VTREADY,              // chain -> MMA: Vt^T bf16 operands ready (128)
  B_SFULL,                // MMA -> chain: S^T updated
  B_OFULL,                // MMA -> chain: O^T complete
  B_OFREE,                // chain -> MMA: O^T read (128)
  B_PQFREE0,              // MMA -> prep: P / gated Q buffer 0 free
  B_PQFREE1,              //                                  1
  B_DRAIN,                // MMA: everything issued has completed
};

struct TcParams {
  const float *beta, *g, *h0;
  __nv_bfloat16 *out;
  float *hT;
  int H, T, L, n_h, nchunks;
};

struct Smem {
  uint8_t *base;
  __device__ uint8_t *stage(int s) const { return base + s * STAGE_BYTES; }
  __device__ float *beta(int s) const { return reinterpret_cast<float *>(base + OFF_SMALL + SM_BETA) + s * 64; }
  __device__ float *lam(int s) const { return reinterpret_cast<float *>(base + OFF_SMALL + SM_LAM) + s * 64; }
  __device__ float *gcp() const { return reinterpret_cast<float *>(base + OFF_SMALL + SM_GCP); }
  __device__ float *dec() const { return reinterpret_cast<float *>(base + OFF_SMALL + SM_DEC); }
  __device__ uint64_t *bar(int i) const { return reinterpret_cast<uint64_t *>(base + OFF_SMALL + SM_BAR) + i; }
  __device__ uint32_t *tmem_slot() const { return reinterpret_cast<uint32_t *>(base + OFF_SMALL + SM_TMEM); }
  __device__ volatile int *abort_flag() const { return reinterpret_cast<volatile int *>(base + OFF_SMALL + SM_ABORT); }
  __device__ float *At() const { return reinterpret_cast<float *>(base + OFF_AT); }
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

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// D(16x8) += A(16x8) B(8x8) on the warp-level tensor-core path, tf32 inputs.
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

// One warp: D(16x8) = M1[r0.., k0..k0+K) * M2[k0'.., n0..] with both operands
// read from swizzled fp32 smem.  M1 is read through its transpose when
// `m1_transposed` (At holds A^T).  K is a multiple of 8.
template <int K>
__device__ __forceinline__ void warp_gemm_16x8(float (&d)[4], const float *M1, bool m1_transposed,
                                               int r0, int k0, const float *M2, int k2, int n0,
                                               int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int ks = 0; ks < K / 8; ++ks) {
    const int c = k0 + 8 * ks;
    uint32_t a[4];
    if (m1_transposed) {
      a[0] = to_tf32(M1[swz(c + t, r0 + g)]);
      a[1] = to_tf32(M1[swz(c + t, r0 + g + 8)]);
      a[2] = to_tf32(M1[swz(c + t + 4, r0 + g)]);
      a[3] = to_tf32(M1[swz(c + t + 4, r0 + g + 8)]);
    } else {
      a[0] = to_tf32(M1[swz(r0 + g, c + t)]);
      a[1] = to_tf32(M1[swz(r0 + g + 8, c + t)]);
      a[2] = to_tf32(M1[swz(r0 + g, c + t + 4)]);
      a[3] = to_tf32(M1[swz(r0 + g + 8, c + t + 4)]);
    }
    const int kr = k2 + 8 * ks;
    const uint32_t b[2] = {to_tf32(M2[swz(kr + t, n0 + g)]), to_tf32(M2[swz(kr + t + 4, n0 + g)])};
    mma_tf32(d, a, b);
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

  // ---- set-up: zero the operand buffers, init barriers, allocate TMEM ----
  {
    uint4 *z = reinterpret_cast<uint4 *>(sm.base);
    for (uint32_t i = tid; i < OFF_SMALL / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
  }
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
        // keep the chunks after the ones in the ring warm in L2
        for (int pf = (n == 0 ? NS : n + NS); pf <= n + NS + 1 && pf < NT; ++pf) {
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
      float *sb = sm.beta(s), *sl = sm.lam(s);
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
      const uint32_t id_uw = idesc_bf16(128, 64, true, false);
      const uint32_t id_vt = idesc_bf16(128, 64, false, true, true);  // B = W^T MN-major, negated
      const uint32_t id_o = idesc_bf16(128, 64, false, false);
      const uint32_t id_s = idesc_bf16(128, 128, false, true);
      const uint32_t a_tu = smem_u32(sm.base + OFF_TU), a_tw = smem_u32(sm.base + OFF_TW);
      const uint32_t a_w = smem_u32(sm.base + OFF_W);

      const uint32_t id_g = idesc_bf16(128, 64, false, false);
      auto prep_g = [&](int m) -> bool {  // G(m) = [K;Q] K^T
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
      auto prep_uw = [&](int m) -> bool {  // U(m)^T, W(m)^T
        const int s = m % NS;
        if (!wait_bar(sm, B_TFULL, m & 1, 1)) return false;
        tc_fence_after();
        const uint32_t kq = smem_u32(sm.stage(s));
        const uint32_t vv = kq + 32768;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tmem + TM_UV, sdesc_sw128(vv + k * 2048, 8192, 1024),
                 sdesc_sw128(a_tu + k * 32, 0, 1024), id_uw, k > 0);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tmem + TM_GW, sdesc_sw128(kq + k * 2048, 16384, 1024),
                 sdesc_sw128(a_tw + k * 32, 0, 1024), id_uw, k > 0);
        mma_commit(sm.bar(B_WFULL));
        return true;
      };

      ok = prep_g(0) && prep_uw(0);
      for (int n = 0; ok && n < NT; ++n) {
        const int s = n % NS;
        const uint32_t kq = smem_u32(sm.stage(s));
        const uint32_t sbf = tmem + TM_SBF + (n & 1) * 64;
        if (!wait_bar(sm, B_WREADY, n & 1, 1)) break;
        // G of the next chunk as soon as W^T(n) has left TMEM: its solve
        // overlaps this chunk's state-dependent chain
        if (n + 1 < NT && !prep_g(n + 1)) break;
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
        // O^T = S^T (Q * exp gc)^T + Vt^T P^T; afterwards the stage is free
        if (n >= 1 && !wait_bar(sm, B_OFREE, (n - 1) & 1, 1)) break;
        tc_fence_after();
        const uint32_t qb = GATED ? smem_u32(sm.base + OFF_QG) + (n & 1) * 8192 : kq + 8192;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ts(tmem + TM_O, sbf + k * 8, sdesc_sw128(qb + (k >> 2) * 16384 + (k & 3) * 32, 0, 1024),
                 id_o, k > 0);
        const uint32_t pb = smem_u32(sm.base + OFF_P) + (n & 1) * 8192;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ts(tmem + TM_O, tmem + TM_VBF + k * 8, sdesc_sw128(pb + k * 32, 0, 1024), id_o, true);
        mma_commit(sm.bar(B_OFULL));
        mma_commit(sm.bar(B_EMPTY + s));
        mma_commit(sm.bar(B_PQFREE0 + (n & 1)));
        // U, W of the next chunk
        if (n + 1 < NT && !prep_uw(n + 1)) break;
      }
      mma_commit(sm.bar(B_DRAIN));
      wait_bar(sm, B_DRAIN, 0, 1);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ===================================================== prep warps
    const int q4 = warp & 3;              // TMEM lane quarter
    const int L = q4 * 32 + lane;         // TMEM lane of this thread
    float *At = sm.At();
    float *X = sm.X();
    float *gcp = sm.gcp();
    for (int m = 0; m < NT; ++m) {
      const int s = m % NS;
      // a failed wait sets the abort flag; every thread still reaches the
      // next named barrier and all of them leave together after it
      wait_bar(sm, B_FULL + s, (m / NS) & 1, 2);
      const float *sb = sm.beta(s);
      if (GATED && warp == 2) {
        float lo, hi;
        warp_scan64(sm.lam(s), lane, lo, hi);
        gcp[lane] = lo;
        gcp[lane + 32] = hi;
      }
      if (named_sync_or(1, *sm.abort_flag() != 0)) break;
      const int e0 = m * C;
      const int t_lo = e0 / n_h;
      int t_hi = (e0 + C - n_h) / n_h;
      if (t_hi > p.T - 1) t_hi = p.T - 1;
      const int Cp = t_hi - t_lo + 1;  // readout rows of this chunk

      // ---- one row of G = [K;Q] K^T per thread (TMEM lane L), 16 columns at a time ----
      const int pw = warp - 2;  // 0..3
      wait_bar(sm, B_GFULL, m & 1, 2);
      tc_fence_after();
      if (L < 64) {
        // row i of A = beta_i Gam_ij (k_i . k_j) for j < i, stored transposed
        const int i = L;
        const float bi = sb[i];
        const float gi = GATED ? gcp[i] : 0.f;
        uint32_t r[64];
        tmem_ld32(tmem_addr(tmem + TM_GW, q4 * 32, 0), *reinterpret_cast<uint32_t (*)[32]>(&r[0]));
        tmem_ld32(tmem_addr(tmem + TM_GW, q4 * 32, 32), *reinterpret_cast<uint32_t (*)[32]>(&r[32]));
        tmem_wait_ld_regs(r);
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          float a = 0.f;
          if (j < i) a = bi * __uint_as_float(r[j]) * (GATED ? fast_exp2(gi - gcp[j]) : 1.f);
          At[swz(j, i)] = a;
        }
      } else {
        // row r of P = (q_r . k_j) Gam, j <= pos(r)
        const int r = L - 64;
        const bool valid = r < Cp;
        const int pos = valid ? (t_lo + r) * n_h + (n_h - 1) - e0 : -1;
        const float gp = (GATED && valid) ? gcp[pos] : 0.f;
        if (m >= 2) wait_bar(sm, B_PQFREE0 + (m & 1), ((m >> 1) - 1) & 1, 2);
        uint8_t *ptile = sm.base + OFF_P + (m & 1) * 8192;
        uint32_t g64[64];
        tmem_ld32(tmem_addr(tmem + TM_GW, q4 * 32, 0), *reinterpret_cast<uint32_t (*)[32]>(&g64[0]));
        tmem_ld32(tmem_addr(tmem + TM_GW, q4 * 32, 32), *reinterpret_cast<uint32_t (*)[32]>(&g64[32]));
        tmem_wait_ld_regs(g64);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint32_t pk[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j0 = q * 8 + 2 * u;
            const float v0 =
                (j0 <= pos) ? __uint_as_float(g64[j0]) * (GATED ? fast_exp2(gp - gcp[j0]) : 1.f) : 0.f;
            const float v1 = (j0 + 1 <= pos)
                                 ? __uint_as_float(g64[j0 + 1]) * (GATED ? fast_exp2(gp - gcp[j0 + 1]) : 1.f)
                                 : 0.f;
            pk[u] = pack_bf16(v0, v1);
          }
          st_chunk(ptile, sw128_offset(r, q * 8, 64), pk);
        }
      }
      tc_fence_before();
      if (named_sync_or(1, *sm.abort_flag() != 0)) break;  // A^T complete

      if (L < 64) {
        // ---- diagonal 16x16 blocks of X = (I + A)^{-1}: column jj of block
        //      b, right-looking forward substitution, next column prefetched ----
        const int o = (L >> 4) * 16, jj = L & 15;
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
        float4 nx[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) nx[q] = *reinterpret_cast<const float4 *>(At + swz(o, o + 4 * q));
#pragma unroll
        for (int mm = 0; mm < 16; ++mm) {
          float cur[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            cur[4 * q] = nx[q].x; cur[4 * q + 1] = nx[q].y;
            cur[4 * q + 2] = nx[q].z; cur[4 * q + 3] = nx[q].w;
          }
          if (mm + 1 < 16) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              nx[q] = *reinterpret_cast<const float4 *>(At + swz(o + mm + 1, o + 4 * q));
          }
          const float x = (mm == jj) ? 1.f : ((mm > jj) ? -acc[mm] : 0.f);
          X[swz(o + mm, o + jj)] = x;
#pragma unroll
          for (int i = mm + 1; i < 16; ++i) acc[i] = fmaf(cur[i], x, acc[i]);
        }
      } else if (GATED) {
        // ---- gated query row r: q_r * exp(gc_pos), zero beyond the readout set ----
        const int r = L - 64;
        const bool valid = r < Cp;
        const int pos = valid ? (t_lo + r) * n_h + (n_h - 1) - e0 : 0;
        const float sc = valid ? fast_exp2(gcp[pos]) : 0.f;
        const uint8_t *qt = sm.stage(s) + 8192;
        uint8_t *qg = sm.base + OFF_QG + (m & 1) * 8192;
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t off = blk * 16384 + sw128_offset(r, q * 8, 64);
            const uint4 v = *reinterpret_cast<const uint4 *>(qt + off);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              __nv_bfloat162 b2;
              *reinterpret_cast<uint32_t *>(&b2) = w[u];
              const float2 f = __bfloat1622float2(b2);
              o4[u] = pack_bf16(f.x * sc, f.y * sc);
            }
            st_chunk(qg, off, o4);
          }
        }
      }
      named_sync(1);  // diagonal blocks of X done
      {
        // ---- merge 16 -> 32: X21' = -X22' (A21' X11') in each 32-row half ----
        const int o = (pw >> 1) * 32, nt = pw & 1;
        float y[4] = {0.f, 0.f, 0.f, 0.f};
        warp_gemm_16x8<16>(y, At, true, o + 16, o, X, o, o + 8 * nt, lane);
        // scratch: the unused upper-right 32x32 block of X
        const int sr = (pw >> 1) * 16, scol = 32 + (pw >> 1) * 16 + 8 * nt;
        warp_store_16x8(X, sr, scol, y, 1.f, lane);
        __syncwarp();
        float z[4] = {0.f, 0.f, 0.f, 0.f};
        warp_gemm_16x8<16>(z, X, false, o + 16, o + 16, X, sr, scol, lane);
        warp_store_16x8(X, o + 16, o + 8 * nt, z, -1.f, lane);
      }
      named_sync(1);
      {
        // ---- merge 32 -> 64: Y = A21 X11 into the upper-right block ----
        const int mr = (pw >> 1) * 16, nc = (pw & 1) * 16;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          float y[4] = {0.f, 0.f, 0.f, 0.f};
          warp_gemm_16x8<32>(y, At, true, 32 + mr, 0, X, 0, nc + 8 * nt, lane);
          warp_store_16x8(X, mr, 32 + nc + 8 * nt, y, 1.f, lane);
        }
        named_sync(1);
        // ---- X21 = -X22 Y ----
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          float z[4] = {0.f, 0.f, 0.f, 0.f};
          warp_gemm_16x8<32>(z, X, false, 32 + mr, 32, X, 0, 32 + nc + 8 * nt, lane);
          warp_store_16x8(X, 32 + mr, nc + 8 * nt, z, -1.f, lane);
        }
      }
      named_sync(1);
      if (m >= 1) wait_bar(sm, B_WFULL, (m - 1) & 1, 2);  // T tiles consumed by U/W(m-1)
      // ---- T = X diag(beta) and T diag(beta exp gc) as bf16 operand tiles
      //      (entries above the diagonal of X hold scratch: masked) ----
      {
        const int i = (tid & 127) >> 1, jh = (tid & 1) * 32;
        uint8_t *tu = sm.base + OFF_TU;
        uint8_t *tw = sm.base + OFF_TW;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t pu[4], pwv[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = jh + q * 8 + 2 * u;
            const float2 x2 = *reinterpret_cast<const float2 *>(X + swz(i, j));
            const float u0 = (j <= i) ? x2.x * sb[j] : 0.f;
            const float u1 = (j + 1 <= i) ? x2.y * sb[j + 1] : 0.f;
            pu[u] = pack_bf16(u0, u1);
            if (GATED)
              pwv[u] = pack_bf16(u0 * fast_exp2(gcp[j]), u1 * fast_exp2(gcp[j + 1]));
            else
              pwv[u] = pu[u];
          }
          st_chunk(tu, sw128_offset(i, jh + q * 8, 64), pu);
          st_chunk(tw, sw128_offset(i, jh + q * 8, 64), pwv);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(sm.bar(B_TFULL));

    }
  } else {
    // ===================================================== chain warps
    const int q4 = warp & 3;
    const int L = q4 * 32 + lane;  // TMEM lane = value column dv
    const int ct = tid - 192;      // 0..127 within the chain group
    float *dec = sm.dec();
    // gate of a chunk: 2^(sum of its log2 gates)
    auto chunk_decay = [&](int n) -> float {
      if (!GATED) return 1.f;
      const float *lam = sm.lam(n % NS);
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
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t r[32];
        tmem_ld32(tmem_addr(tmem + TM_GW, q4 * 32, half * 32), r);
        tmem_wait_ld_regs(r);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t pk[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            pk[u] = pack_bf16(__uint_as_float(r[q * 8 + 2 * u]), __uint_as_float(r[q * 8 + 2 * u + 1]));
          st_chunk(wt, sw128_offset(L, half * 32 + q * 8, 128), pk);
        }
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
      // ---- pseudo-values: Vt^T -> bf16 operands ----
      wait_bar(sm, B_VTFULL, n & 1, 3);
      tc_fence_after();
      if (GATED) {
        wait_bar(sm, B_FULL + s, (n / NS) & 1, 3);
        if (warp == 6) {
          float lo, hi;
          warp_scan64(sm.lam(s), lane, lo, hi);
          const float tot = __shfl_sync(0xffffffffu, hi, 31);
          dec[lane] = fast_exp2(tot - lo);
          dec[lane + 32] = fast_exp2(tot - hi);
        }
        if (named_sync_or(2, *sm.abort_flag() != 0)) break;
      }
      {
        uint32_t r[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          tmem_ld32(tmem_addr(tmem + TM_UV, q4 * 32, half * 32), r);
          tmem_wait_ld_regs(r);
          uint32_t pk[16], pd[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const float a = __uint_as_float(r[2 * u]), c = __uint_as_float(r[2 * u + 1]);
            pk[u] = pack_bf16(a, c);
            if (GATED) pd[u] = pack_bf16(a * dec[half * 32 + 2 * u], c * dec[half * 32 + 2 * u + 1]);
          }
          tmem_st16(tmem_addr(tmem + TM_VBF, q4 * 32, half * 16), pk);
          if (GATED) tmem_st16(tmem_addr(tmem + TM_VDEC, q4 * 32, half * 16), pd);
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
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t r[32], pk[16];
          tmem_ld32(tmem_addr(tmem + TM_S, q4 * 32, c0), r);
          tmem_wait_ld_regs(r);
#pragma unroll
          for (int u = 0; u < 16; ++u)
            pk[u] = pack_bf16(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
          tmem_st16(tmem_addr(sbf, q4 * 32, c0 / 2), pk);
          if (GATED) {
#pragma unroll
            for (int u = 0; u < 32; ++u) r[u] = __float_as_uint(__uint_as_float(r[u]) * dn);
            tmem_st32(tmem_addr(tmem + TM_S, q4 * 32, c0), r);
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
      // ---- epilogue: token outputs of this chunk, staged for 16-byte stores ----
      wait_bar(sm, B_OFULL, n & 1, 3);
      tc_fence_after();
      {
        const int e0 = n * C;
        const int t_lo = e0 / n_h;
        int t_hi = (e0 + C - n_h) / n_h;
        if (t_hi > p.T - 1) t_hi = p.T - 1;
        const int Cp = t_hi - t_lo + 1;
        __nv_bfloat16 *stg = reinterpret_cast<__nv_bfloat16 *>(sm.base + OFF_STG);
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tmem_addr(tmem + TM_O, q4 * 32, c0), r);
          tmem_wait_ld_regs(r);
#pragma unroll
          for (int u = 0; u < 32; ++u) stg[(c0 + u) * D + L] = __float2bfloat16_rn(__uint_as_float(r[u]));
        }
        tc_fence_before();
        mbar_arrive(sm.bar(B_OFREE));
        // W^T of the next chunk before the copy-out: it gates the next chain step
        if (n + 1 < NT) convert_w(n + 1);
        if (named_sync_or(2, *sm.abort_flag() != 0)) break;
        // rows of 256 bytes: 16 threads per row, 8 rows per pass
        const int chunk16 = ct & 15;
        uint4 *og = reinterpret_cast<uint4 *>(p.out);
        const uint4 *sg = reinterpret_cast<const uint4 *>(stg);
        for (int rr = ct >> 4; rr < Cp; rr += 8) {
          const size_t row = ((size_t)b * p.T + t_lo + rr) * p.H + h;
          og[row * (D / 8) + chunk16] = sg[rr * (D / 8) + chunk16];
        }
        named_sync(2);
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
