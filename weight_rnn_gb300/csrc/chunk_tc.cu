// chunk_tc.cu -- the state pass of the chunked forward of delta-rule
// attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), bf16
// I/O, dk = dv = 128, chunk C = 64, any n_h (Gated DeltaProduct), gated or
// not.  It takes the UT transform T = (I + A)^{-1} diag(beta) of every chunk
// from the intra-chunk pass (ut_tc.cu) and runs the state chain.
//
// The algorithm is the chunkwise form of "08 · linear 路线（三）：delta rule 与
// DPLR 统一框架" -- the WY vectors of §2.2, the state passing of §2.3 and the
// gated variant of §3 -- run on the extended sequence of "DeltaProduct：通过
// Householder 乘积增强线性 RNN 的状态追踪" §4.1.  Per chunk of 64 rows, with
// gc the inclusive cumsum of the log gate (log g_t at each token's first
// sub-step, 0 elsewhere; clamped at -80 so g = 0 stays finite):
//
//   W    = T (K * exp(gc)),  U = T V                      (the WY vectors)
//   V~   = U - W S                                        (pseudo-values)
//   O    = (Q * exp(gc)) S + P V~,   P = Q K^T * Gam * M  (M incl. diag)
//   S   <- exp(gc_C) S + Kd^T V~,    Kd = K * exp(gc_C - gc)
//
// All products are computed TRANSPOSED, so that every tensor-core product has
// M = 128 (a d axis) and the state S^T lives in TMEM as an fp32 accumulator
// [dv lanes x dk columns]:
//
//   G     = [K; Q] K^T                  SS  N=64  K=128  (rows 64.. -> P)
//   W^T   = K^T (T diag exp gc)^T       SS  N=64  K=64   -> bf16 smem operand
//   U^T   = V^T T^T                     SS  N=64  K=64   (into the V~ accumulator)
//   V~^T -= S^T W^T                     TS  N=64  K=128  (A = S^T bf16 in TMEM)
//   S^T  += (V~ diag dec)^T K           TS  N=128 K=64   (= V~^T Kd, dec = exp(gc_C - gc);
//                                                         S^T scaled by exp(gc_C) first)
//   O^T   = S^T (Q exp gc)^T + V~^T P^T TS  N=64  K=128 + K=64
//
// The recurrence is S^T -> bf16 -> V~ -> bf16 -> S^T: two products and two
// conversions per chunk.  Everything else (G, P, W, Q exp(gc), the
// outputs) is prepared or drained by other warps around it.  W, U, V~ and P
// never leave the SM.  HBM traffic is q, k, v, beta, g and T in, out, h0/hT
// once per head.
//
// Warp roles (512 threads; one CTA per (b, h) head):
//   warp 0       TMA producer: K/Q/V tiles (128-byte swizzle, 3 stages)
//                and the T tile (2-slot ring); beta is inside T, and the
//                prep warps read the gate
//   warps 1, 14, 15  MMA issuers (one thread each): the recurrence (U, V~,
//                the state update); the outputs; the look-ahead G, W.
//                Warp 1 owns the TMEM allocation.
//   warps 2-5    prep: P from G, T diag(exp gc)
//   warps 6-9    feed-forward: W^T -> bf16 smem operand and Q exp(gc) in
//                place (one chunk ahead),
//                the outputs (staged through the V slot by transposing 8x8
//                stores, then 16-byte global stores)
//   warps 10-13  chain: V~^T -> bf16 operands (plain, and scaled by dec for
//                the state update), S^T -> bf16 operand and the exp(gc_C)
//                scaling, hT
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
constexpr uint32_t ST_K0 = 0, ST_Q0 = 8192, ST_K1 = 16384, ST_Q1 = 24576;  // Q later Q*exp(gc)
constexpr uint32_t ST_V0 = 32768;  // V (64 x 128), later the staged output rows
constexpr uint32_t OFF_WS = NS * STAGE_BYTES;  // 2 x W^T bf16 [128 dk][64], MN-major B
constexpr uint32_t OFF_TW = OFF_WS + 32768;    // T diag(exp gc) bf16 [64][64], K-major
constexpr uint32_t OFF_P = OFF_TW + 8192;      // 2 x P bf16 [64][64], K-major
constexpr uint32_t OFF_TR = OFF_P + 16384;     // 2 x T bf16 [64][64] (TMA ring), K-major
constexpr uint32_t OFF_SM = OFF_TR + 16384;    // small arrays and barriers
constexpr uint32_t SM_LAM = 0;                 // prep: the chunk's log2 gate
constexpr uint32_t SM_EG = SM_LAM + 256;         // prep: 2^gc
constexpr uint32_t SM_GC = SM_EG + 256;          // prep: gc (cumulative log2 gate)
constexpr uint32_t SM_DEC = SM_GC + 256;         // [4][64] prep -> chain: 2^(gc_C - gc) / sigma'
constexpr uint32_t SM_QF = SM_DEC + 1024;        // [4][64] prep -> ff: 2^gc at each readout row's sub-step
constexpr uint32_t SM_PLAN = SM_QF + 1024;       // [4] ChunkPlan, prep -> chain, MMA, ff
constexpr uint32_t SM_BAR = SM_PLAN + 64;

// ---- barrier indices ----
enum {
  B_FULL = 0,        // [NS] producer -> all: K, Q tiles loaded (count 1 + tx)
  B_EMPTY = NS,      // [NS] MMA -> producer: the stage consumed (state and output issuers, 2)
  B_VFULL = 2 * NS,  // [NS] producer -> MMA: the V tile of a stage loaded (count 1 + tx)
  B_VEMPTY = 3 * NS, // [NS] ff -> producer: V slot free (per warp; it stages the outputs)
  B_TRFULL = 4 * NS, // [2] producer -> prep: the chunk's T tile loaded (count 1 + tx)
  B_TREMPTY = 4 * NS + 2,  // [2] MMA -> producer: the T tile consumed (U and W products, 2)
  B_WSFREE = 4 * NS + 4,   // [2] MMA -> ff: the W^T operand buffer consumed (by the S W product)
  B_PFREE = 4 * NS + 6,    // [2] MMA -> prep: P buffer consumed (by the V~ P product)
  B_WCVT = 4 * NS + 8,     // [2] ff -> MMA: W^T bf16 operand buffer filled (per warp)
  B_TFULL = 4 * NS + 10,   // [2] prep -> MMA: T (gated: T diag exp gc) of a chunk ready (warps 4, 5)
  B_PLAN = 4 * NS + 12,    // [4] prep -> chain, MMA, ff: the chunk's ChunkPlan, dec and readout factors (gated)
  B_PRDY = 4 * NS + 16,    // [2] prep -> MMA: P of a chunk in shared memory (warps 2, 3)
  B_GFULL = 4 * NS + 18,   // MMA -> prep: G in TMEM
  B_GFREE,           // prep -> MMA: G read (per P warp, 2)
  B_WFULL,           // MMA -> ff, prep: W^T in TMEM (T diag(exp gc) consumed)
  B_WREAD,           // ff -> MMA: W^T read out of TMEM (per warp)
  B_VDONE,           // MMA -> chain: V~^T = U^T - S^T W^T in TMEM
  B_VRDY,            // chain -> MMA: V~^T bf16 in TMEM, TM_V read (per warp)
  B_SFULL,           // MMA -> chain, ff: the state update done
  B_SRDY,            // chain -> MMA: S^T bf16 in TMEM, S^T scaled by exp(gc_C) (per warp)
  B_SQDONE,          // MMA -> chain: the S^T (Q exp gc)^T product done (S^T bf16 consumed)
  B_OFULL,           // MMA -> ff, chain: O^T in TMEM
  B_OFREE,           // ff -> MMA: O^T read (per warp)
  B_DRAIN,           // MMA: everything issued has completed (3 issuers)
  NBARS
};
constexpr uint32_t SM_MISC = SM_BAR + NBARS * 8;  // tmem slot, abort flag, spare, keep-TMEM flag
constexpr uint32_t SMEM_TOTAL = OFF_SM + ((SM_MISC + 16 + 15) & ~15u);
constexpr uint32_t SMEM_ALLOC = 232448;
static_assert(SMEM_TOTAL + 1023 <= SMEM_ALLOC, "shared memory budget");

// ---- TMEM columns ----
constexpr uint32_t TM_S = 0;      // S^T fp32 [dv][dk]                   128
constexpr uint32_t TM_SBF = 128;  // S^T bf16 (packed)                    64
constexpr uint32_t TM_O = 192;    // O^T fp32 [dv][readout rows]          64
constexpr uint32_t TM_G = 256;    // G fp32                               64
constexpr uint32_t TM_W = 320;    // W^T fp32 [dk][64]                    64
constexpr uint32_t TM_V = 384;    // U^T, then V~^T fp32 [dv][64]         64
constexpr uint32_t TM_VB = 448;   // V~^T bf16 (packed)                   32
constexpr uint32_t TM_VBD = 480;  // (V~ diag exp(gc_C - gc))^T bf16      32  (gated)
constexpr uint32_t TM_COLS = 512;

// Gated: TMEM holds S~ = S / sigma, sigma = 2^ls.  Each chunk's decay
// exp(gc_C) goes into sigma (sigma' = exp(gc_C) sigma) and the accumulator is
// only added to, until sigma would fall below 2^-kSigmaRange: then the state
// is rescaled in TMEM instead (sigma' = 1), so S~ stays within 2^64 |S|.
constexpr float kSigmaRange = 64.f;

// The per-chunk decisions of the gated state update, made by the prep warps
// (in chunk order, ahead of the chain) and read by the others.
struct ChunkPlan {
  float rs;   // TMEM factor before the chunk's update (1 unless rescaled)
  float sig;  // sigma of the state after the chunk's update
  int ratio;  // the chunk is in the ratio regime (decay product >= 2^-100)
  int pad;
};

struct TcParams {
  const float *beta, *g, *h0;
  __nv_bfloat16 *out;
  float *hT;
  int H, T, n_h, nchunks;
};

struct Smem {
  uint8_t *base;
  __device__ uint8_t *stage(int s) const { return base + s * STAGE_BYTES; }
  __device__ float *arr(uint32_t off) const { return reinterpret_cast<float *>(base + OFF_SM + off); }
  __device__ float *lam() const { return arr(SM_LAM); }
  __device__ volatile ChunkPlan *plan(int m) const {
    return reinterpret_cast<volatile ChunkPlan *>(base + OFF_SM + SM_PLAN) + (m & 3);
  }
  __device__ uint64_t *bar(int i) const {
    return reinterpret_cast<uint64_t *>(base + OFF_SM + SM_BAR) + i;
  }
  __device__ uint32_t *tmem_slot() const { return reinterpret_cast<uint32_t *>(base + OFF_SM + SM_MISC); }
  __device__ volatile int *abort_flag() const {
    return reinterpret_cast<volatile int *>(base + OFF_SM + SM_MISC + 4);
  }
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

// Exact regime of the gated path: the Q rows of a stage times their readout
// factor qf, in place (thread ft of the 128 takes the 16-byte pieces ft,
// ft + 128, ... of both 64-column halves).  Out of line: it runs only for the
// chunks whose decay leaves the range of the ratio form, and inline it would
// spread the hot code over more instruction cache lines.
__device__ __noinline__ void scale_q_rows(uint8_t *qt, const float *qf, int ft) {
#pragma unroll 2
  for (int it = 0; it < 8; ++it) {
    const int qi = ft + 128 * it;  // 16-byte piece: 512 per 64-column half
    uint8_t *pc = qt + ((qi >> 9) ? ST_Q1 : ST_Q0) + (qi & 511) * 16;
    const uint4 v = *reinterpret_cast<const uint4 *>(pc);
    const float f = qf[(qi & 511) >> 3];
    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
    uint32_t o4[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      o4[u] = pack_bf16(__uint_as_float(in[u] << 16) * f, __uint_as_float(in[u] & 0xFFFF0000u) * f);
    *reinterpret_cast<uint4 *>(pc) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
  }
}

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
  const int tid = threadIdx.x, lane = tid & 31;
  // the warp index through a shuffle from lane 0: the compiler then knows it
  // is the same in every lane, so that branches on a warp's role are not
  // divergent and need no reconvergence code around the warp-wide
  // instructions in them (a much smaller kernel)
  const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
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
      mbar_init(sm.bar(B_FULL + s), 1);
      mbar_init(sm.bar(B_EMPTY + s), 2);
      mbar_init(sm.bar(B_VFULL + s), 1);
      mbar_init(sm.bar(B_VEMPTY + s), 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(sm.bar(B_TRFULL + s), 1);
      mbar_init(sm.bar(B_TREMPTY + s), 2);
      mbar_init(sm.bar(B_WSFREE + s), 1);
      mbar_init(sm.bar(B_PFREE + s), 1);
      mbar_init(sm.bar(B_WCVT + s), 4);
      mbar_init(sm.bar(B_TFULL + s), 2);
      mbar_init(sm.bar(B_PRDY + s), 2);
    }
    for (int s = 0; s < 4; ++s) mbar_init(sm.bar(B_PLAN + s), 1);
    // count per barrier, from B_GFULL on
    const int cnt[NBARS - B_GFULL] = {1, 2, 1, 4, 1, 4, 1, 4, 1, 1, 4, 3};
    for (int i = B_GFULL; i < NBARS; ++i) mbar_init(sm.bar(i), cnt[i - B_GFULL]);
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
    // (tiles only: beta is inside T, and the prep warps read the gate)
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
    // blocking on the barriers of its inputs; the tensor pipe executes their
    // products in issue order.
    //   warp 1   the recurrence, per chunk n: U^T = V^T T^T into TM_V (the
    //            T slot loaded, V~ of n-1 read), V~^T -= S^T W^T (SRDY, the
    //            W^T slot filled), then S^T += (V~ diag dec)^T K (VRDY)
    // A thread waits for phase k of a barrier only where phase k+1 needs one
    // of that thread's own later products (else a slow thread could see two
    // completions as none): ring barriers carry the slot index.
    //   warp 14  the outputs of n: O^T = S^T (Q exp gc)^T behind the S W
    //            product (VDONE, OFREE(n-1)), O^T += V~^T P^T behind the
    //            state update (SFULL, PRDY(n))
    //   warp 15  the look-ahead: G(0); per chunk W(m) (TFULL, WREAD(m-1)),
    //            then G(m+1) (FULL, GFREE(m))
    // Each commits the barriers of its own products; every hand-off between
    // kinds is a barrier.  A descriptor's address field is the byte address
    // / 16 and every operand lies below 256 KiB, so a K step of an operand is
    // the descriptor plus its byte offset / 16.  Only the two products on the recurrence (S W and
    // the state update) are unrolled: the kernel's hot code has to fit the
    // SM's instruction cache, and with every SM of a GPC running this kernel
    // the refills of a miss are slow.
    if (lane == 0) {
      constexpr uint32_t id_uw = idesc_bf16(128, 64, true, false);        // A = K^T or V^T (MN-major), B = T
      constexpr uint32_t id_sw = idesc_bf16(128, 64, false, true, true);  // B = W^T (MN-major), negated
      constexpr uint32_t id_kd = idesc_bf16(128, 128, false, true);       // B = K (MN-major)
      constexpr uint32_t id_o = idesc_bf16(128, 64, false, false);        // B = Q exp(gc) or P (K-major)
      constexpr uint32_t id_g = idesc_bf16(128, 64, false, false);
      const uint32_t a_tr = smem_u32(sm.base + OFF_TR), a_tw = smem_u32(sm.base + OFF_TW);
      const uint32_t a_ws = smem_u32(sm.base + OFF_WS), a_p = smem_u32(sm.base + OFF_P);
      if (warp == 1) {
        for (int n = 0; n < NT; ++n) {
          const int s = n % NS;
          const uint32_t st = smem_u32(sm.stage(s));
          // ---- U^T = V^T T^T ----
          // (every wait here and below is on a barrier whose next phase
          // needs this thread's own later products, so no phase can be
          // skipped: the T ring slot is refilled only after this U product)
          if (!wait_bar(sm, B_TRFULL + (n & 1), (n >> 1) & 1, 1) ||
              !wait_bar(sm, B_VFULL + s, (n / NS) & 1, 1))
            break;
          if (n >= 1 && !wait_bar(sm, B_VRDY, (n - 1) & 1, 1)) break;
          tc_fence_after();
          const uint64_t du = sdesc_sw128(st + ST_V0, 8192, 1024);
          const uint64_t dt = sdesc_sw128(a_tr + (n & 1) * 8192, 0, 1024);
#pragma unroll 1
          for (int k = 0; k < 4; ++k) mma_ss(tmem + TM_V, du + k * 128, dt + k * 2, id_uw, k > 0);
          mma_commit(sm.bar(B_TREMPTY + (n & 1)));
          // ---- V~^T = U^T - S^T W^T ----
          if (!wait_bar(sm, B_WCVT + (n & 1), (n >> 1) & 1, 1) || !wait_bar(sm, B_SRDY, n & 1, 1)) break;
          tc_fence_after();
          const uint64_t dw = sdesc_sw128(a_ws + (n & 1) * 16384, 8192, 1024);
#pragma unroll
          for (int k = 0; k < 8; ++k) mma_ts(tmem + TM_V, tmem + TM_SBF + k * 8, dw + k * 128, id_sw, true);
          mma_commit(sm.bar(B_VDONE));
          mma_commit(sm.bar(B_WSFREE + (n & 1)));
          // ---- S^T += V~^T Kd = (V~ diag exp(gc_C - gc))^T K (S^T was scaled by
          //      exp(gc_C) by the chain warps) ----
          if (!wait_bar(sm, B_VRDY, n & 1, 1)) break;
          tc_fence_after();
          // (gated: S~ += ((V~ diag dec) / sigma')^T K, the decay carried by
          // the scale sigma of the accumulator)
          const uint32_t vb = GATED ? TM_VBD : TM_VB;
          const uint64_t dk = sdesc_sw128(st + ST_K0, 16384, 1024);
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_ts(tmem + TM_S, tmem + vb + k * 8, dk + k * 128, id_kd, true);
          mma_commit(sm.bar(B_SFULL));
          mma_commit(sm.bar(B_EMPTY + s));
        }
      } else if (warp == 14) {
        for (int n = 0; n < NT; ++n) {
          const int s = n % NS;
          const uint32_t st = smem_u32(sm.stage(s));
          // ---- O^T = S^T (Q exp gc)^T, behind the S W product (it reads the
          //      same bf16 S^T, which is rewritten once both ended) ----
          if (n >= 1 && !wait_bar(sm, B_OFREE, (n - 1) & 1, 1)) break;
          if (!wait_bar(sm, B_VDONE, n & 1, 1)) break;
          tc_fence_after();
          // (the two 64-column halves of Q are 16 KiB apart)
          const uint64_t dq = sdesc_sw128(st + ST_Q0, 0, 1024);
#pragma unroll 1
          for (int k = 0; k < 8; ++k)
            mma_ts(tmem + TM_O, tmem + TM_SBF + k * 8, dq + (k >> 2) * 1024 + (k & 3) * 2, id_o, k > 0);
          mma_commit(sm.bar(B_SQDONE));
          // ---- O^T += V~^T P^T, behind the state update (gated, ratio
          //      regime: the dec-scaled copy of V~, P carrying 1 / dec) ----
          if (!wait_bar(sm, B_PRDY + (n & 1), (n >> 1) & 1, 1)) break;
          if (GATED && !wait_bar(sm, B_PLAN + (n & 3), (n >> 2) & 1, 1)) break;
          if (!wait_bar(sm, B_SFULL, n & 1, 1)) break;
          tc_fence_after();
          const uint64_t dp = sdesc_sw128(a_p + (n & 1) * 8192, 0, 1024);
          const uint32_t vsrc = (GATED && sm.plan(n)->ratio) ? TM_VBD : TM_VB;
#pragma unroll 1
          for (int k = 0; k < 4; ++k) mma_ts(tmem + TM_O, tmem + vsrc + k * 8, dp + k * 2, id_o, true);
          mma_commit(sm.bar(B_OFULL));
          mma_commit(sm.bar(B_PFREE + (n & 1)));
          mma_commit(sm.bar(B_EMPTY + s));
        }
      } else if (warp == 15) {
        // ---- G = [K;Q] K^T of chunk m ----
        auto issue_g = [&](int m) -> bool {
          if (!wait_bar(sm, B_FULL + m % NS, (m / NS) & 1, 1)) return false;
          // TM_G is free once the P warps have read chunk m-1's G
          if (m >= 1 && !wait_bar(sm, B_GFREE, (m - 1) & 1, 1)) return false;
          tc_fence_after();
          // [K;Q] is 128 rows (K then Q, 64 rows = 8 KiB each) per 64-column
          // half, the halves 16 KiB apart
          const uint64_t dg = sdesc_sw128(smem_u32(sm.stage(m % NS)), 0, 1024);
#pragma unroll 1
          for (int k = 0; k < 8; ++k) {
            const uint64_t d = dg + (k >> 2) * 1024 + (k & 3) * 2;
            mma_ss(tmem + TM_G, d, d, id_g, k > 0);
          }
          mma_commit(sm.bar(B_GFULL));
          return true;
        };
        bool ok = issue_g(0);
        for (int m = 0; ok && m < NT; ++m) {
          // ---- W^T = K^T (T diag exp gc)^T (ungated: T itself) ----
          if (!wait_bar(sm, B_TFULL + (m & 1), (m >> 1) & 1, 1)) break;
          if (m >= 1 && !wait_bar(sm, B_WREAD, (m - 1) & 1, 1)) break;
          tc_fence_after();
          const uint64_t dk = sdesc_sw128(smem_u32(sm.stage(m % NS)) + ST_K0, 16384, 1024);
          const uint64_t dt = sdesc_sw128(GATED ? a_tw : a_tr + (m & 1) * 8192, 0, 1024);
#pragma unroll 1
          for (int k = 0; k < 4; ++k) mma_ss(tmem + TM_W, dk + k * 128, dt + k * 2, id_uw, k > 0);
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
    // per chunk m: P = Q K^T * Gam * M from rows 64..127 of G, then GFREE
    // and PRDY (warps 2, 3); T diag(exp gc) for the W product, then TFULL
    // (warps 4, 5; ungated: TFULL once the T tile has landed)
    const int q4 = warp & 3;              // TMEM lane quarter
    const int L = q4 * 32 + lane;         // TMEM lane of this thread
    float *eg = sm.arr(SM_EG), *gcs = sm.arr(SM_GC);
    float ls = 0.f;  // P warps, gated: log2 sigma of the state before chunk m's update
    // gated, warp 2: the linear gate of the tokens whose first sub-step lies
    // in a chunk, one token per lane (and lane + 32), and that sub-step's
    // place in the chunk (-1: no such token); read one chunk ahead so that
    // the loads are in flight while the chunk before is prepared
    float gnx[2] = {1.f, 1.f};
    int gpos[2] = {-1, -1};
    auto gate_fetch = [&](int m) {
      const int e0 = m * C;
      const int t0 = (e0 + n_h - 1) / n_h;  // the first token that starts in the chunk
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int t = t0 + lane + 32 * k, e = t * n_h - e0;
        const bool in = m < NT && e < C && t < p.T;
        gpos[k] = in ? e : -1;
        gnx[k] = in ? p.g[((size_t)b * p.T + t) * p.H + h] : 1.f;
      }
    };
    if (GATED && warp == 2) gate_fetch(0);
    for (int m = 0; m < NT; ++m) {
      // every warp of the group is done with the previous chunk's gate
      // factors (they are rewritten below)
      if (named_sync_or(1, *sm.abort_flag() != 0)) break;
      // a failed wait sets the abort flag; every thread still reaches the
      // next named barrier and all of them leave together after it
      if (GATED && warp == 2) {
        // log2 g at each token's first sub-step, 0 at the others
        float *lam = sm.lam();
        lam[lane] = 0.f;
        lam[lane + 32] = 0.f;
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 2; ++k)
          if (gpos[k] >= 0) lam[gpos[k]] = gate_log2(gnx[k]);
        __syncwarp();
        gate_fetch(m + 1);
        float lo, hi;
        warp_scan64(lam, lane, lo, hi);
        gcs[lane] = lo;
        gcs[lane + 32] = hi;
        eg[lane] = fast_exp2(lo);
        eg[lane + 32] = fast_exp2(hi);
      }
      if (named_sync_or(1, *sm.abort_flag() != 0)) break;
      const Rows rw(m, n_h, p.T);
      if (warp < 4) {
        // ---- P: one readout row per thread, 16 columns at a time ----
        // exact per-entry decay only when the chunk's gate product leaves
        // the range of the ratio form (uniform per chunk)
        const bool ratio = !GATED || gcs[63] >= kRatioFloor;
        if (m >= 2) wait_bar(sm, B_PFREE + (m & 1), ((m >> 1) - 1) & 1, 2);
        float cp = 1.f;  // ratio regime: the uniform factor of P
        if (GATED) {
          // ---- the plan of chunk m's state update.  Both P warps track sigma
          //      alike and take the same decisions; warp 2 publishes them with
          //      dec = exp(gc_C - gc) / sigma' (the chain's factor of V~) and
          //      the readout factor 2^gc of each readout row (0 past the last
          //      one).  Slot m % 4 was last read for chunk m - 4, whose readers
          //      all finished before the V~ P product of chunk m - 2 (waited for
          //      just above) was issued ----
          const float gl = gcs[63];
          const float e = -(gl + ls);
          float rs = 1.f;
          if (e < kSigmaRange) {
            ls = -e;
          } else {
            ls = 0.f;
            rs = fast_exp2(-e);
          }
          // the V~ P product reads V~ diag(dec): P = Q K^T * M * 2^(ls' - gc_C)
          // (the readout row's own 2^gc is applied to the output row)
          cp = fast_exp2(ls - gl);
          if (warp == 2) {
            float *dec = sm.arr(SM_DEC + (m & 3) * 256), *qf = sm.arr(SM_QF + (m & 3) * 256);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int j = lane + 32 * hf;
              dec[j] = fast_exp2(gl - gcs[j] - ls);
              qf[j] = j < rw.Cp ? eg[rw.pos(j, n_h)] : 0.f;
            }
            if (lane == 0) {
              volatile ChunkPlan *pl = sm.plan(m);
              pl->rs = rs;
              pl->sig = fast_exp2(ls);
              pl->ratio = ratio ? 1 : 0;
            }
            arrive_warp(sm.bar(B_PLAN + (m & 3)), lane);
          }
        }
        wait_bar(sm, B_GFULL, m & 1, 2);
        tc_fence_after();
        const int r = L - 64;
        const int pos = r < rw.Cp ? rw.pos(r, n_h) : -1;
        const float gp = (GATED && pos >= 0) ? gcs[pos] : 0.f;
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
            for (int jj = 0; jj < 16; ++jj) cf[jj] = cp;
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
        //      into its own buffer, free once the previous chunk's W product ended ----
        wait_bar(sm, B_TRFULL + (m & 1), (m >> 1) & 1, 2);
        if (GATED) {
          if (m >= 1) wait_bar(sm, B_WFULL, (m - 1) & 1, 2);
          const uint8_t *tt = sm.base + OFF_TR + (m & 1) * 8192;
          uint8_t *tw = sm.base + OFF_TW;
          const int ft = tid - 128;  // 0..63
#pragma unroll 2
          for (int it = 0; it < 8; ++it) {
            const uint4 v = *reinterpret_cast<const uint4 *>(tt + (ft + 64 * it) * 16);
            // 16-byte piece qi of the swizzled tile: row qi / 8, columns
            // 8 ((qi % 8) ^ (row % 8)) .. + 7
            const int qi = ft + 64 * it, row = qi >> 3;
            const int c0 = 8 * ((qi & 7) ^ (row & 7));
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
      // P goes to the V~ P product; T diag(exp gc) to the W product, which
      // thus does not wait for P
      fence_proxy_async_smem();
      arrive_warp(sm.bar((warp < 4 ? B_PRDY : B_TFULL) + (m & 1)), lane);
    }
  } else if (warp < 10) {
    // ===================================================== feed-forward warps
    // W^T(m) -> bf16 operand in shared memory and (gated) Q exp(gc) in place,
    // one chunk ahead; the outputs of chunk m -> global memory
    const int q4 = warp & 3;
    const int L = q4 * 32 + lane;  // TMEM lane: a d index
    const int ft = tid - 192;      // 0..127 within the group
    auto w_convert = [&](int m) {
      // ---- W^T (row L = a dk index, 64 columns) -> bf16 rows of the MN-major
      //      operand W^T [dk][64] ----
      wait_bar(sm, B_WFULL, m & 1, 3);
      tc_fence_after();
      uint32_t pw_[32];
      {
        uint32_t r[64];
        tmem_ld32(tmem_addr(tmem + TM_W, q4 * 32, 0), *reinterpret_cast<uint32_t (*)[32]>(&r[0]));
        tmem_ld32(tmem_addr(tmem + TM_W, q4 * 32, 32), *reinterpret_cast<uint32_t (*)[32]>(&r[32]));
        tmem_wait_ld_regs(r);
        tc_fence_before();
        arrive_warp(sm.bar(B_WREAD), lane);
#pragma unroll
        for (int u = 0; u < 32; ++u)
          pw_[u] = pack_bf16(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
      }
      // the S W product of the chunk two back reads this buffer until it ends
      if (m >= 2) wait_bar(sm, B_WSFREE + (m & 1), ((m >> 1) - 1) & 1, 3);
      uint8_t *ws = sm.base + OFF_WS + (m & 1) * 16384;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st_chunk(ws + sw128_offset(L, 8 * q, 128), {pw_[4 * q], pw_[4 * q + 1], pw_[4 * q + 2], pw_[4 * q + 3]});
      if (GATED) {
        // ---- the readout factor exp(gc) at each readout row's sub-step
        //      (published by prep warp 2 with the chunk's plan).  Ratio
        //      regime (the chunk's decay stays above 2^-100; P' = Q K^T *
        //      2^-gc_j): the output rows are scaled by it at write-out.
        //      Exact regime: Q exp(gc) in place (rows past the readouts
        //      zeroed) and no output scaling.  The G product (which read Q)
        //      completed before P and W; the output product that reads Q
        //      waits for the S W product, which waits for WCVT ----
        // (the plan of chunk m + 4 needs this thread's W^T of chunk m + 2)
        wait_bar(sm, B_PLAN + (m & 3), (m >> 2) & 1, 3);
        if (!sm.plan(m)->ratio) {
          wait_bar(sm, B_FULL + m % NS, (m / NS) & 1, 3);  // the Q tile landed
          scale_q_rows(sm.stage(m % NS), sm.arr(SM_QF + (m & 3) * 256), ft);
        }
      }
      fence_proxy_async_smem();
      arrive_warp(sm.bar(B_WCVT + (m & 1)), lane);
    };
    if (!named_sync_or(2, *sm.abort_flag() != 0)) w_convert(0);
    for (int n = 0; n < NT; ++n) {
      if (named_sync_or(2, *sm.abort_flag() != 0)) break;
      if (n + 1 < NT) w_convert(n + 1);
      const Rows rw(n, n_h, p.T);
      // ---- outputs of chunk n: the accumulator is read at once (TMEM is
      //      released early), staged as bf16 rows in the V slot of this chunk
      //      (its reader, the U product, has completed) by transposing 8x8
      //      stores, then written out in 16-byte pieces ----
      // read O^T only once the chain's TMEM work of this chunk (the S^T
      // conversion, SRDY phase n + 1) is done; the next SRDY phase needs
      // this chunk's OFREE (through the output product of the next chunk)
      wait_bar(sm, B_OFULL, n & 1, 3);
      if (n + 1 < NT) wait_bar(sm, B_SRDY, (n + 1) & 1, 3);
      tc_fence_after();
      uint32_t o0[32], o1[32];
      tmem_ld16x256b_x8(tmem_addr(tmem + TM_O, q4 * 32, 0), o0);
      tmem_ld16x256b_x8(tmem_addr(tmem + TM_O, q4 * 32 + 16, 0), o1);
      tmem_wait_ld_regs(o0);
      tmem_wait_ld_regs(o1);
      tc_fence_before();
      arrive_warp(sm.bar(B_OFREE), lane);
      {
        if (GATED && sm.plan(n)->ratio) {
          // ratio regime: every output row times its readout factor
          const int tq = lane & 3;
          const float *qf = sm.arr(SM_QF + (n & 3) * 256);
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            // register 4 g + j holds output row (column of O^T) 8 g + 2 tq + j % 2
            const float2 f = *reinterpret_cast<const float2 *>(qf + 8 * g + 2 * tq);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float fj = (j & 1) ? f.y : f.x;
              o0[4 * g + j] = __float_as_uint(__uint_as_float(o0[4 * g + j]) * fj);
              o1[4 * g + j] = __float_as_uint(__uint_as_float(o1[4 * g + j]) * fj);
            }
          }
        }
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
            for (int mm = 0; mm < 4; ++mm) {
              const int j = 4 * (2 * cc + (mm >> 1)) + 2 * (mm & 1);
              o4[mm] = pack_bf16(__uint_as_float(ov[j]), __uint_as_float(ov[j + 1]));
            }
            const int r = 16 * cc + 8 * (mi >> 1) + mr;
            stsm_x4_trans(srow(r) + ((k ^ (r & 7)) << 4), o4);
          }
        }
        named_sync(2);  // every value column of every row staged
        const int k = ft & 15, cp = rw.Cp;
        __nv_bfloat16 *obase = p.out + (((size_t)b * p.T + rw.t_lo) * p.H + h) * D + 8 * k;
        const size_t rstride = (size_t)p.H * D;
        uint4 v[8];  // every load before the first store
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int r = 8 * it + (ft >> 4);
          v[it] = lds128(srow(r) + ((k ^ (r & 7)) << 4));
        }
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int r = 8 * it + (ft >> 4);
          if (r < cp) *reinterpret_cast<uint4 *>(obase + r * rstride) = v[it];
        }
        // the V slot is free once every warp has read its rows
        arrive_warp(sm.bar(B_VEMPTY + n % NS), lane);
      }
    }
  } else {
    // ===================================================== chain warps
    // the recurrence: V~^T -> bf16 operand (gated: V~ diag dec); the updated
    // state S^T -> bf16 operand (gated: sigma S~^T, and the rare rescale of
    // TMEM the plan of the next chunk asks for); hT
    const int q4 = warp & 3;
    const int L = q4 * 32 + lane;  // TMEM lane = value column dv
    // ---- initial state: S^T bf16 = h0^T, S~^T fp32 = h0^T (sigma = 1) ----
    {
      const float *h0 = p.h0 ? p.h0 + (size_t)bh * D * D : nullptr;
      float r0 = 1.f;
      if (GATED) {
        wait_bar(sm, B_PLAN, 0, 4);
        r0 = sm.plan(0)->rs;
      }
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t f[32], pk[16];
#pragma unroll
        for (int u = 0; u < 32; u += 2) {
          const float x0 = h0 ? h0[(size_t)(c0 + u) * D + L] : 0.f;
          const float x1 = h0 ? h0[(size_t)(c0 + u + 1) * D + L] : 0.f;
          f[u] = __float_as_uint(x0 * r0);
          f[u + 1] = __float_as_uint(x1 * r0);
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
      // ---- V~^T -> bf16 operands: gated, (V~ diag dec / sigma')^T for the
      //      state update (and, in the ratio regime, for the V~ P product);
      //      V~^T itself for the V~ P product otherwise.  The products of the
      //      previous chunk read the old ones until the output group ended (it
      //      is issued after the state update) ----
      if (n >= 1) wait_bar(sm, B_OFULL, (n - 1) & 1, 4);
      wait_bar(sm, B_VDONE, n & 1, 4);
      tc_fence_after();
      // (the plan of chunk n was waited for at the previous chunk's end)
      const bool plain = !GATED || !sm.plan(n)->ratio;
      const float *dec = sm.arr(SM_DEC + (n & 3) * 256);
#pragma unroll 1
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t r[32], pv[16];
        tmem_ld32(tmem_addr(tmem + TM_V, q4 * 32, 32 * hf), r);
        tmem_wait_ld_regs(r);
        if (plain) {
#pragma unroll
          for (int u = 0; u < 16; ++u) pv[u] = pack_bf16(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
          tmem_st16(tmem_addr(tmem + TM_VB, q4 * 32, 16 * hf), pv);
        }
        if (GATED) {
#pragma unroll
          for (int u = 0; u < 16; u += 2) {
            const float4 d4 = *reinterpret_cast<const float4 *>(dec + 32 * hf + 2 * u);
            pv[u] = pack_bf16(__uint_as_float(r[2 * u]) * d4.x, __uint_as_float(r[2 * u + 1]) * d4.y);
            pv[u + 1] = pack_bf16(__uint_as_float(r[2 * u + 2]) * d4.z, __uint_as_float(r[2 * u + 3]) * d4.w);
          }
          tmem_st16(tmem_addr(tmem + TM_VBD, q4 * 32, 16 * hf), pv);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      arrive_warp(sm.bar(B_VRDY), lane);
      // ---- the updated state: S^T -> bf16 operand for the next chunk (gated:
      //      sigma S~^T, and the rescale of the next chunk's plan), or hT; the
      //      S W and S (Q) products of this chunk read the old bf16 copy ----
      // (the waits that usually completed earlier go first, so that the
      // state update's is the last one)
      float rs = 1.f;
      if (n + 1 < NT) {
        if (GATED) {
          wait_bar(sm, B_PLAN + ((n + 1) & 3), ((n + 1) >> 2) & 1, 4);
          rs = sm.plan(n + 1)->rs;
        }
        wait_bar(sm, B_SQDONE, n & 1, 4);
      }
      wait_bar(sm, B_SFULL, n & 1, 4);
      tc_fence_after();
      const float sig = GATED ? sm.plan(n)->sig : 1.f;  // sigma of S~ in TMEM now
      if (n + 1 < NT) {
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t r[64], pk[32];
          tmem_ld32(tmem_addr(tmem + TM_S, q4 * 32, 64 * hf), *reinterpret_cast<uint32_t (*)[32]>(&r[0]));
          tmem_ld32(tmem_addr(tmem + TM_S, q4 * 32, 64 * hf + 32), *reinterpret_cast<uint32_t (*)[32]>(&r[32]));
          tmem_wait_ld_regs(r);
#pragma unroll
          for (int u = 0; u < 32; ++u)
            pk[u] = pack_bf16(__uint_as_float(r[2 * u]) * sig, __uint_as_float(r[2 * u + 1]) * sig);
          tmem_st32(tmem_addr(tmem + TM_SBF, q4 * 32, 32 * hf), pk);
          if (GATED && rs != 1.f) {
            // the next chunk's sigma' would fall below 2^-64: TMEM <-
            // exp(gc_C) S, with sigma' = 1
#pragma unroll
            for (int u = 0; u < 64; ++u) r[u] = __float_as_uint(__uint_as_float(r[u]) * rs);
            tmem_st32(tmem_addr(tmem + TM_S, q4 * 32, 64 * hf), *reinterpret_cast<uint32_t (*)[32]>(&r[0]));
            tmem_st32(tmem_addr(tmem + TM_S, q4 * 32, 64 * hf + 32), *reinterpret_cast<uint32_t (*)[32]>(&r[32]));
          }
        }
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
          for (int u = 0; u < 32; ++u) hT[(size_t)(c0 + u) * D + L] = __uint_as_float(r[u]) * sig;
        }
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
  return a.bf16 && a.dk == D && a.dv == D && a.chunk == C && a.T > 0 && !a.alpha && ut_supports(a);
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
  p.n_h = a.n_h;
  p.nchunks = nt;
  auto kern = a.g ? chunk_tc_kernel<true> : chunk_tc_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)(a.B * a.H), kThreads, SMEM_ALLOC, s>>>(mq, mk, mv, mt, p);
  return cudaGetLastError();
}

}  // namespace delta
