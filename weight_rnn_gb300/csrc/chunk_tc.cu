// chunk_tc.cu -- the state pass of the chunked forward of delta-rule
// attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), bf16
// I/O, dk = dv = 128, chunk C = 64, any n_h (Gated DeltaProduct), gated or
// not.  It takes the UT transform T = (I + A)^{-1} diag(beta) of every chunk
// from the intra-chunk pass (ut_tc.cu) and runs the state chain.
//
// The algorithm is the chunkwise form of "08 · linear 路线（三）：delta rule 与
// DPLR 统一框架" -- the WY vectors of §2.2, the state passing of §2.3 and the
// gated variant of §3 -- run on the extended sequence of "DeltaProduct：通过
// Householder 乘积增强线性 RNN 的状态追踪" §4.1.  Per chunk of 64 rows:
//
//   gc   = inclusive cumsum of the log gate (log g_t at each token's first
//          sub-step, 0 elsewhere; clamped at -80 so g = 0 stays finite)
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
//   G     = [K; Q] K^T                  SS  N=64  K=128  (rows 64.. -> P)
//   W^T   = K^T (T diag exp gc)^T       SS  N=64  K=64
//   U^T   = V^T T^T                     SS  N=64  K=64
//   (M-I)^T = -W^T Kd                   TS  N=128 K=64   (A = W^T bf16 in TMEM)
//   Q'^T  = -W^T P^T (+ exp(gc) Q^T)    TS  N=64  K=64
//   S^T  += S^T (M-I)^T + U^T Kd        TS  N=128 K=128 + K=64   (chain)
//   O^T   = U^T P^T + S^T Q'^T          TS  N=64  K=64 + K=128   (after the chain step)
//
// The state step does not wait for the outputs: the output group of chunk n
// is issued right behind its state step (it reads the same bf16 S^T), and
// Q' is prepared by other warps while the chain runs.  W, U, M, Q' and P never
// leave the SM.  HBM traffic is q, k, v, beta, g and T in, out, h0/hT once per
// head.
//
// Warp roles (512 threads; one CTA per (b, h) head):
//   warp 0       TMA producer: K/Q/V tiles (128-byte swizzle, 3 stages, the
//                chunk after them prefetched into L2), the T tile (2-slot
//                ring), beta / log-gate rows
//   warps 1, 14, 15  MMA issuers (one thread each): the recurrence (state
//                step, output group); M and the Q' helper; the look-ahead
//                G, W, U.  Warp 1 owns the TMEM allocation.
//   warps 2-5    prep: P from G (chunk n+2), T diag(exp gc) for W, and Q' of
//                the chunk in flight -> smem operand (warp-MMA fragments)
//   warps 6-9    feed-forward (chunk n+1): W^T, U^T -> bf16 TMEM operands,
//                Kd, (M-I)^T -> smem operand
//   warps 10-13  chain (chunk n): S^T -> bf16 operand, the outputs (staged
//                through the V slot by transposing 8x8 stores), hT
// Every mbarrier wait is bounded; a timeout sets a device error word and the
// kernel winds down instead of hanging.
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm100.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace delta {

// Set by the tensor-core kernel when a bounded wait gives up (1 + role id).
__device__ unsigned int g_tc_error = 0;

namespace {
using namespace sm100;
using namespace tc;

constexpr int C = 64;
constexpr int D = 128;
constexpr int NS = 3;  // TMA stages
// Three MMA-issuing threads (warps 1, 14, 15), each blocking on its own
// barriers in a fixed order; 16 warps = 512 threads, 128 registers each
constexpr int kThreads = 512;

// ---- shared memory layout (offsets from a 1024-byte aligned base) ----
constexpr uint32_t STAGE_BYTES = 49152;
constexpr uint32_t ST_K0 = 0, ST_Q0 = 8192, ST_K1 = 16384, ST_Q1 = 24576;
constexpr uint32_t ST_V0 = 32768;  // V (64 x 128), later Kd, same layout
constexpr uint32_t OFF_MS = NS * STAGE_BYTES;  // (M-I)^T bf16 [128 j][128 i], MN-major B
constexpr uint32_t OFF_TW = OFF_MS + 32768;    // T diag(exp gc) bf16 [64][64], K-major
constexpr uint32_t OFF_P = OFF_TW + 8192;      // 2 x P bf16 [64][64], K-major
constexpr uint32_t OFF_TR = OFF_P + 16384;     // 2 x T bf16 [64][64] (TMA ring), K-major
constexpr uint32_t OFF_SM = OFF_TR + 16384;    // small arrays and barriers
constexpr uint32_t SM_BETA = 0;                // [NS][64]
constexpr uint32_t SM_LAM = SM_BETA + NS * 256;  // [NS][64] log2 gate
constexpr uint32_t SM_EG = SM_LAM + NS * 256;    // prep: 2^gc
constexpr uint32_t SM_IEG = SM_EG + 256;         // prep: 2^-gc
constexpr uint32_t SM_GC = SM_IEG + 256;         // prep: gc (cumulative log2 gate)
constexpr uint32_t SM_DEC = SM_GC + 256;         // feed-forward: 2^(gc_C - gc)
constexpr uint32_t SM_GQ = SM_DEC + 256;         // feed-forward: 2^gc at readout rows
constexpr uint32_t SM_BAR = SM_GQ + 256;

// ---- barrier indices ----
enum {
  B_FULL = 0,        // [NS] producer -> all: K, Q tiles, beta, log gate loaded (count 2 + tx)
  B_EMPTY = NS,      // [NS] MMA -> producer: K, Q tiles of the stage consumed
  B_GFULL = 2 * NS,  // MMA -> prep: G in TMEM
  B_GFREE,           // prep -> MMA: G read (per P warp, 2)
  B_TFULL,           // prep -> MMA: T diag(exp gc) and P written (per warp)
  B_WFULL,           // MMA -> ff, prep: W^T, U^T in TMEM (T diag(exp gc) consumed)
  B_CWDW,            // ff -> MMA: W^T bf16 in TMEM, Kd in smem, TM_X1 read (per warp)
  B_MFULL,           // MMA -> ff: (M-I)^T in TMEM
  B_MRDY,            // ff -> MMA: (M-I)^T in smem, TMEM free (per warp)
  B_QFULL,           // MMA -> prep, ff: -W^T P^T in TMEM (W^T bf16 consumed)
  B_QRDY,            // prep -> MMA: Q' in smem, TMEM read (per warp)
  B_SRDY,            // chain -> MMA: S^T bf16 in TMEM (per warp)
  B_SFULL,           // MMA -> chain, ff: state step done
  B_OFULL,           // MMA -> chain, ff: the output group (U^T P^T + S^T Q'^T) done
  B_OFREE,           // chain -> MMA: O^T read (per warp)
  B_PFREE0,          // MMA -> prep: P buffer 0 consumed
  B_PFREE1,          //                        1
  B_DRAIN,           // MMA: everything issued has completed
  B_CWDU,            // ff -> MMA: U^T bf16 in TMEM (per warp)
  B_VFULL,           // [NS] producer -> MMA: the V tile of a stage loaded (count 1 + tx)
  B_VEMPTY = B_VFULL + NS,  // [NS] chain -> producer: V slot free (per warp; it stages the outputs)
  B_TRFULL = B_VEMPTY + NS,  // [2] producer -> prep: the chunk's T tile loaded (count 1 + tx)
  B_TREMPTY = B_TRFULL + 2,  // [2] MMA -> producer: the T tile consumed (by the U product)
  NBARS = B_TREMPTY + 2
};
constexpr uint32_t SM_MISC = SM_BAR + NBARS * 8;  // tmem slot, abort flag, gate of the chunk
constexpr uint32_t SMEM_TOTAL = OFF_SM + ((SM_MISC + 16 + 15) & ~15u);
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
// it; if the work waited for writes TMEM (the products), the CTA keeps its
// TMEM columns at exit instead of freeing them under products that may still
// be writing them.
__device__ __noinline__ bool wait_bar_drain(uint8_t *base, int idx, uint32_t parity, int role,
                                            bool tmem_writer) {
  Smem sm;
  sm.base = base;
  uint64_t *b = sm.bar(idx);
  for (uint32_t i = 0; i < (1u << 24); ++i)
    if (mbar_try_wait(b, parity)) return true;
  *sm.abort_flag() = 1;
  if (tmem_writer) *sm.keep_tmem() = 1;
  atomicCAS(&g_tc_error, 0u, (unsigned)(1 + role) | ((unsigned)idx << 8));
  return false;
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
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_t,
                TcParams p) {
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
    for (uint32_t i = tid; i < SMEM_TOTAL / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(sm.bar(B_FULL + s), 2);
      mbar_init(sm.bar(B_EMPTY + s), 1);
      mbar_init(sm.bar(B_VEMPTY + s), 4);
    }
    const int cnt[B_VFULL - 2 * NS] = {1, 2, 4, 1, 4, 1, 4, 1, 4, 4, 1, 1, 4, 1, 1, 3, 4};
    for (int i = 2 * NS; i < B_VFULL; ++i) mbar_init(sm.bar(i), cnt[i - 2 * NS]);
    for (int s = 0; s < NS; ++s) mbar_init(sm.bar(B_VFULL + s), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(sm.bar(B_TRFULL + s), 1);
      mbar_init(sm.bar(B_TREMPTY + s), 1);
    }
    *sm.abort_flag() = 0;
    *sm.keep_tmem() = 0;
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
    tma_prefetch_desc(&map_t);
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
    int issued = 0, issued_v = 0, issued_t = 0;
    const int tc0 = bh * NT;  // this head's first chunk in the T tensor
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
          tma_prefetch_3d(&map_t, 0, 0, tc0 + pf);
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
      // T of the chunk (written by the UT pass) into its 2-slot ring; the U
      // product of the chunk two back is its last reader
      if (n >= 2 && lane == 0) ok = wait_bar(sm, B_TREMPTY + (n & 1), ((n >> 1) - 1) & 1, 0);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (lane == 0) {
        uint64_t *tb = sm.bar(B_TRFULL + (n & 1));
        mbar_arrive_expect_tx(tb, 8192u);
        tma_load_3d(sm.base + OFF_TR + (n & 1) * 8192, &map_t, tb, 0, 0, tc0 + n);
      }
      issued_t = n + 1;
      fetch(n + 1);
    }
    // copies still in flight must land before the CTA's shared memory goes
    if (lane == 0) {
      for (int n = (issued > NS ? issued - NS : 0); n < issued; ++n)
        wait_bar_drain(sm.base, B_FULL + n % NS, (n / NS) & 1, 0, false);
      for (int n = (issued_v > NS ? issued_v - NS : 0); n < issued_v; ++n)
        wait_bar_drain(sm.base, B_VFULL + n % NS, (n / NS) & 1, 0, false);
      for (int n = (issued_t > 2 ? issued_t - 2 : 0); n < issued_t; ++n)
        wait_bar_drain(sm.base, B_TRFULL + (n & 1), (n >> 1) & 1, 0, false);
    }
    __syncwarp();
  } else if (warp == 1 || warp >= 14) {
    // ===================================================== MMA issuers
    // Three threads, each issuing one kind of work in a fixed order and
    // blocking on the barriers of its inputs (a blocked try_wait wakes within
    // ~100 cycles of the arrival; the tensor pipe interleaves their products
    // in issue order):
    //   warp 1   the recurrence: state step n (SRDY, MRDY, CWDU), then the
    //            output group of n (QRDY), which reads the same bf16 S^T
    //   warp 14  M(n) (CWDW), then the -W^T P^T helper of Q'(n) (OFREE(n-1))
    //   warp 15  the look-ahead: G(0); per chunk W(m) (TFULL, MRDY(m-1)),
    //            U(m) (VFULL), G(m+1) (FULL, GFREE(m))
    // Each commits the barriers of its own products; every hand-off between
    // kinds is a barrier.
    if (lane == 0) {
      constexpr uint32_t id_uw = idesc_bf16(128, 64, true, false);
      constexpr uint32_t id_m = idesc_bf16(128, 128, false, true, true);  // B = Kd, MN-major, negated
      constexpr uint32_t id_q = idesc_bf16(128, 64, false, false, true);  // B = P, negated
      constexpr uint32_t id_op = idesc_bf16(128, 64, false, false);       // B = P
      constexpr uint32_t id_s = idesc_bf16(128, 128, false, true);        // B = (M-I)^T or Kd, MN-major
      constexpr uint32_t id_o = idesc_bf16(128, 64, false, false);        // B = Q' (K-major)
      constexpr uint32_t id_g = idesc_bf16(128, 64, false, false);
      const uint32_t a_tr = smem_u32(sm.base + OFF_TR), a_tw = smem_u32(sm.base + OFF_TW);
      const uint32_t a_ms = smem_u32(sm.base + OFF_MS), a_p = smem_u32(sm.base + OFF_P);
      auto kd_desc = [&](int m, int k) -> uint64_t {  // B = Kd (gated: V slot) or K
        const uint32_t kq = smem_u32(sm.stage(m % NS));
        return GATED ? sdesc_sw128(kq + ST_V0 + k * 2048, 8192, 1024)
                     : sdesc_sw128(kq + ST_K0 + k * 2048, 16384, 1024);
      };
      if (warp == 1) {
        for (int n = 0; n < NT; ++n) {
          // ---- the state step ----
          if (!wait_bar(sm, B_SRDY, n & 1, 1) || !wait_bar(sm, B_MRDY, n & 1, 1) ||
              !wait_bar(sm, B_CWDU, n & 1, 1))
            break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ts(tmem + TM_S, tmem + TM_SBF + k * 8, sdesc_sw128(a_ms + k * 2048, 16384, 1024), id_s, true);
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_ts(tmem + TM_S, tmem + TM_UB + k * 8, kd_desc(n, k), id_s, true);
          mma_commit(sm.bar(B_SFULL));
          // ---- the output group: O^T = U^T P^T + S^T Q'^T ----
          if (!wait_bar(sm, B_QRDY, n & 1, 1)) break;
          tc_fence_after();
          const uint32_t pb = a_p + (n & 1) * 8192;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ts(tmem + TM_O, tmem + TM_UB + k * 8, sdesc_sw128(pb + k * 32, 0, 1024), id_op, k > 0);
          const uint32_t st = smem_u32(sm.stage(n % NS));
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t qa = st + (k < 4 ? ST_Q0 : ST_Q1) + (k & 3) * 32;
            mma_ts(tmem + TM_O, tmem + TM_SBF + k * 8, sdesc_sw128(qa, 0, 1024), id_o, true);
          }
          mma_commit(sm.bar(B_OFULL));
          mma_commit(sm.bar(B_PFREE0 + (n & 1)));
          mma_commit(sm.bar(B_EMPTY + n % NS));
        }
      } else if (warp == 14) {
        for (int m = 0; m < NT; ++m) {
          // ---- (M-I)^T = -W^T Kd ----
          if (!wait_bar(sm, B_CWDW, m & 1, 1)) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_ts(tmem + TM_X1, tmem + TM_WB + k * 8, kd_desc(m, k), id_m, k > 0);
          mma_commit(sm.bar(B_MFULL));
          // ---- -W^T P^T (the rest of Q' is added on the CUDA cores) ----
          if (m >= 1 && !wait_bar(sm, B_OFREE, (m - 1) & 1, 1)) break;
          tc_fence_after();
          const uint32_t pb = a_p + (m & 1) * 8192;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ts(tmem + TM_O, tmem + TM_WB + k * 8, sdesc_sw128(pb + k * 32, 0, 1024), id_q, k > 0);
          mma_commit(sm.bar(B_QFULL));
        }
      } else if (warp == 15) {
        // ---- G = [K;Q] K^T of chunk m ----
        auto issue_g = [&](int m) -> bool {
          if (!wait_bar(sm, B_FULL + m % NS, (m / NS) & 1, 1)) return false;
          if (m >= 1 && !wait_bar(sm, B_GFREE, (m - 1) & 1, 1)) return false;
          tc_fence_after();
          const uint32_t kq0 = smem_u32(sm.stage(m % NS));
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const uint32_t kq = kq0 + hf * 16384;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ss(tmem + TM_G, sdesc_sw128(kq + k * 32, 0, 1024), sdesc_sw128(kq + k * 32, 0, 1024),
                     id_g, hf > 0 || k > 0);
          }
          mma_commit(sm.bar(B_GFULL));
          return true;
        };
        bool ok = issue_g(0);
        for (int m = 0; ok && m < NT; ++m) {
          // ---- W^T = K^T (T diag exp gc)^T (ungated: T itself) ----
          if (!wait_bar(sm, B_TFULL, m & 1, 1)) break;
          if (m >= 1 && !wait_bar(sm, B_MRDY, (m - 1) & 1, 1)) break;
          tc_fence_after();
          const uint32_t kq = smem_u32(sm.stage(m % NS));
          const uint32_t wb = GATED ? a_tw : a_tr + (m & 1) * 8192;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + TM_X1, sdesc_sw128(kq + ST_K0 + k * 2048, 16384, 1024),
                   sdesc_sw128(wb + k * 32, 0, 1024), id_uw, k > 0);
          // ---- U^T = V^T T^T ----
          if (!wait_bar(sm, B_VFULL + m % NS, (m / NS) & 1, 1)) break;
          tc_fence_after();
          const uint32_t tb = a_tr + (m & 1) * 8192;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + TM_X1 + 64, sdesc_sw128(kq + ST_V0 + k * 2048, 8192, 1024),
                   sdesc_sw128(tb + k * 32, 0, 1024), id_uw, k > 0);
          mma_commit(sm.bar(B_WFULL));
          mma_commit(sm.bar(B_TREMPTY + (m & 1)));
          if (m + 1 < NT) ok = issue_g(m + 1);
        }
      }
      mma_commit(sm.bar(B_DRAIN));  // every issuer arrives
      wait_bar_drain(sm.base, B_DRAIN, 0, 1, true);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ===================================================== prep warps
    // warps 2, 3 (TMEM lanes 64..127): P from rows 64..127 of G;
    // warps 4, 5: the T tile of the UT pass, scaled to T diag(exp gc) for the
    // W product (gated; ungated the W product reads T itself)
    const int q4 = warp & 3;              // TMEM lane quarter
    const int L = q4 * 32 + lane;         // TMEM lane of this thread
    float *eg = sm.arr(SM_EG), *ieg = sm.arr(SM_IEG), *gcs = sm.arr(SM_GC);
    float *gq = sm.arr(SM_GQ);
    // Q'(c) = exp(gc) Q - P W, in place over the Q tile of chunk c (same
    // K-major layout: the output product reads it as its B operand); the
    // scan for exp(gc) at the readout rows first
    auto qprime = [&](int c) {
      const int s = c % NS;
      const Rows rw(c, n_h, p.T);
      if (GATED) wait_bar(sm, B_FULL + s, (c / NS) & 1, 2);  // the chunk's log-gate row
      if (GATED && warp == 2) {
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
      if (GATED) named_sync(1);
      wait_bar(sm, B_QFULL, c & 1, 2);
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
    };
    for (int m = 0; m < NT; ++m) {
      const int s = m % NS;
      // every warp of the group is done with the previous chunk's gate
      // factors (they are rewritten below)
      if (named_sync_or(1, *sm.abort_flag() != 0)) break;
      // a failed wait sets the abort flag; every thread still reaches the
      // next named barrier and all of them leave together after it
      wait_bar(sm, B_FULL + s, (m / NS) & 1, 2);
      if (GATED && warp == 2) {
        float lo, hi;
        warp_scan64(sm.lam(s), lane, lo, hi);
        gcs[lane] = lo;
        gcs[lane + 32] = hi;
        eg[lane] = fast_exp2(lo);
        eg[lane + 32] = fast_exp2(hi);
        ieg[lane] = fast_exp2(-lo);
        ieg[lane + 32] = fast_exp2(-hi);
      }
      if (named_sync_or(1, *sm.abort_flag() != 0)) break;
      if (warp < 4) {
        // ---- P = Q K^T * Gam * M: one readout row per thread, 16 columns
        //      at a time, into the P buffer of this chunk ----
        const Rows rw(m, n_h, p.T);
        // exact per-entry decay only when the chunk's gate product leaves
        // the range of the ratio form (uniform per chunk)
        const bool ratio = !GATED || gcs[63] >= kRatioFloor;
        if (m >= 2) wait_bar(sm, B_PFREE0 + (m & 1), ((m >> 1) - 1) & 1, 2);
        wait_bar(sm, B_GFULL, m & 1, 2);
        tc_fence_after();
        const int r = L - 64;
        const int pos = r < rw.Cp ? rw.pos(r, n_h) : -1;
        const float gp = (GATED && pos >= 0) ? gcs[pos] : 0.f;
        const float ep = (GATED && pos >= 0) ? eg[pos] : 1.f;
        uint8_t *prow = sm.base + OFF_P + (m & 1) * 8192;
#pragma unroll 1
        for (int jb = 0; jb < 64; jb += 16) {
          uint32_t g[16];
          tmem_ld16(tmem_addr(tmem + TM_G, q4 * 32, jb), g);
          float cf[16];
          if (!GATED) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) cf[jj] = 1.f;
          } else if (ratio) {
#pragma unroll
            for (int jj = 0; jj < 16; jj += 4) {
              const float4 e4 = *reinterpret_cast<const float4 *>(ieg + jb + jj);
              cf[jj] = ep * e4.x;
              cf[jj + 1] = ep * e4.y;
              cf[jj + 2] = ep * e4.z;
              cf[jj + 3] = ep * e4.w;
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) cf[jj] = fast_exp2(gp - gcs[jb + jj]);
          }
          tmem_wait_ld_regs(g);
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
        tc_fence_before();
        arrive_warp(sm.bar(B_GFREE), lane);
      } else {
        // ---- the T tile of this chunk (UT pass) has landed; gated, T diag(exp gc)
        //      into its own buffer, free once the previous chunk's W and U ended ----
        wait_bar(sm, B_TRFULL + (m & 1), (m >> 1) & 1, 2);
        if (GATED) {
          if (m >= 1) wait_bar(sm, B_WFULL, (m - 1) & 1, 2);
          const uint8_t *tt = sm.base + OFF_TR + (m & 1) * 8192;
          uint8_t *tw = sm.base + OFF_TW;
          const int ft = tid - 128;  // 0..63
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            // 16-byte piece qi of the swizzled tile: row qi / 8, columns
            // 8 ((qi % 8) ^ (row % 8)) .. + 7
            const int qi = ft + 64 * it, row = qi >> 3;
            const int c0 = 8 * ((qi & 7) ^ (row & 7));
            const uint4 v = *reinterpret_cast<const uint4 *>(tt + qi * 16);
            const float4 e0 = *reinterpret_cast<const float4 *>(eg + c0);
            const float4 e1 = *reinterpret_cast<const float4 *>(eg + c0 + 4);
            const float ev[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
            const uint32_t in[4] = {v.x, v.y, v.z, v.w};
            uint32_t o4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
              o4[u] = pack_bf16(__uint_as_float(in[u] << 16) * ev[2 * u],
                                __uint_as_float(in[u] & 0xFFFF0000u) * ev[2 * u + 1]);
            st_chunk(tw + qi * 16, o4);
          }
        }
      }
      fence_proxy_async_smem();
      arrive_warp(sm.bar(B_TFULL), lane);
      // Q' of the previous chunk, as soon as its -W^T P^T helper is in TMEM
      if (m >= 1) {
        if (named_sync_or(1, *sm.abort_flag() != 0)) break;
        qprime(m - 1);
      }
    }
    if (NT >= 1 && !named_sync_or(1, *sm.abort_flag() != 0)) qprime(NT - 1);
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

      // ---- W^T, U^T -> bf16 operands (both read out of TM_X1 first, so
      //      that the M product may overwrite it); Kd ----
      wait_bar(sm, B_WFULL, c & 1, 3);
      tc_fence_after();
      uint32_t pw_[32], pu[32];
      {
        uint32_t r[64];
        tmem_ld32(tmem_addr(tmem + TM_X1, q4 * 32, 0), *reinterpret_cast<uint32_t (*)[32]>(&r[0]));
        tmem_ld32(tmem_addr(tmem + TM_X1, q4 * 32, 32), *reinterpret_cast<uint32_t (*)[32]>(&r[32]));
        tmem_wait_ld_regs(r);
#pragma unroll
        for (int u = 0; u < 32; ++u)
          pw_[u] = pack_bf16(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
      }
      {
        uint32_t r[64];
        tmem_ld32(tmem_addr(tmem + TM_X1, q4 * 32, 64), *reinterpret_cast<uint32_t (*)[32]>(&r[0]));
        tmem_ld32(tmem_addr(tmem + TM_X1, q4 * 32, 96), *reinterpret_cast<uint32_t (*)[32]>(&r[32]));
        tmem_wait_ld_regs(r);
#pragma unroll
        for (int u = 0; u < 32; ++u)
          pu[u] = pack_bf16(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
      }
      // W^T bf16 of the previous chunk is read by its M and -W^T P^T products
      // (the -W^T P^T product is issued after M and commits QFULL)
      if (c >= 1) {
        wait_bar(sm, B_QFULL, (c - 1) & 1, 3);
        tc_fence_after();
      }
      tmem_st32(tmem_addr(tmem + TM_WB, q4 * 32, 0), pw_);
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
      tmem_wait_st();
      tc_fence_before();
      arrive_warp(sm.bar(B_CWDW), lane);
      // U^T bf16 of the previous chunk is read by its state step and its
      // output group (U^T P^T) until the output group ends
      if (c >= 1) {
        wait_bar(sm, B_OFULL, (c - 1) & 1, 3);
        tc_fence_after();
      }
      tmem_st32(tmem_addr(tmem + TM_UB, q4 * 32, 0), pu);
      tmem_wait_st();
      tc_fence_before();
      arrive_warp(sm.bar(B_CWDU), lane);

      // ---- (M-I)^T -> bf16 smem operand (row L = j, columns i); the state
      //      step of the previous chunk reads the old one until it ends ----
      wait_bar(sm, B_MFULL, c & 1, 3);
      if (c >= 1) wait_bar(sm, B_SFULL, (c - 1) & 1, 3);
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
  return a.bf16 && a.dk == D && a.dv == D && a.chunk == C && a.T > 0 && ut_supports(a);
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

cudaError_t launch_chunk_tc(const FwdArgs &a, const void *t_mat, cudaStream_t s) {
  if (!chunk_tc_supports(a)) return cudaErrorNotSupported;
  CUtensorMap mq, mk, mv, mt;
  const uint32_t qr = a.n_h == 1 ? 64 : 32;
  const int nt = (int)((a.L + C - 1) / C);
  cudaError_t e;
  if ((e = make_map_4d_bf16(&mq, a.q, D, a.H, a.T, a.B, 64, 1, qr, 1, true)) != cudaSuccess) return e;
  if ((e = make_map_4d_bf16(&mk, a.k, D, a.H, a.L, a.B, 64, 1, 64, 1, true)) != cudaSuccess) return e;
  if ((e = make_map_4d_bf16(&mv, a.v, D, a.H, a.L, a.B, 64, 1, 64, 1, true)) != cudaSuccess) return e;
  if ((e = make_map_3d_bf16_sw128(&mt, t_mat, C, C, (uint64_t)(a.B * a.H * nt), C, C, 1)) != cudaSuccess)
    return e;
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
  p.nchunks = nt;
  auto kern = a.g ? chunk_tc_kernel<true> : chunk_tc_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)(a.B * a.H), kThreads, SMEM_ALLOC, s>>>(mq, mk, mv, mt, p);
  return cudaGetLastError();
}

}  // namespace delta
