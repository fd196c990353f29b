// backward.cu -- gradients of the forward of delta_fwd, float32 on CUDA
// cores.  The pages state no backward formulas; these follow from the
// recurrence of "DeltaProduct：通过 Householder 乘积增强线性 RNN 的状态追踪"
// §2.6 (gate once per token, then n_h delta sub-steps, readout after the
// last) by reverse-mode differentiation, one sub-step at a time.  With P the
// state a sub-step reads (after the token's gate) and r = v - P^T k:
//
//   S = (I - beta k k^T) P + beta k v^T,   o = S^T q at a readout
//   dS += q do^T (readout);  dq = S do
//   dv = beta dS^T k;  dbeta = k^T dS r;  dk = beta (dS r - P dS^T k)
//   dP = dS - beta k (k^T dS);  at a gate: dg = <dP, S_prev>, dS_prev = g dP
//
// One CTA per (b, h) keeps S and dS [dk][dv] in shared memory.  A first sweep
// runs the forward and stores the state at the start of every block of kBlk
// sub-steps in scratch; the backward sweep walks the blocks in reverse,
// recomputes the block's states from its start (stored per sub-step in
// scratch) and runs the reverse recurrence over them.  A correctness path:
// every step is a few dependent reductions over the state.
#include <cuda_bf16.h>

#include "kernels.h"

namespace delta {
namespace {

constexpr int kThreads = 256;
constexpr int kBlk = 64;  // sub-steps per recomputed block

__device__ __forceinline__ float ld(const void *p, int64_t i, bool bf16) {
  return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i])
              : static_cast<const float *>(p)[i];
}

// block-wide sum of one value per thread (red: kThreads / 32 floats)
__device__ __forceinline__ float block_sum(float x, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = x;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < kThreads / 32; ++w) t += red[w];
  return t;
}

__global__ void __launch_bounds__(kThreads) bwd_kernel(BwdArgs a) {
  extern __shared__ float sm[];
  const int dk = a.dk, dv = a.dv, n_h = a.n_h, tid = threadIdx.x;
  const int64_t T = a.T, H = a.H, L = a.T * a.n_h;
  const int64_t bh = blockIdx.x, b = bh / H, h = bh % H;
  const int64_t DD = (int64_t)dk * dv;
  float *S = sm;             // [dk][dv]
  float *dS = S + DD;        // [dk][dv]
  float *kk = dS + DD;       // [dk]
  float *qq = kk + dk;       // [dk]
  float *vec = qq + dk;      // [dv]: v, then r
  float *u = vec + dv;       // [dv]: P^T k, dS^T k, ...
  float *w = u + dv;         // [dk]: dS r, P dS^T k, ...
  float *red = w + dk;       // [kThreads / 32]
  const int64_t nblk = (L + kBlk - 1) / kBlk;
  float *ckpt = a.scratch + bh * (nblk + 1) * DD;       // block starts (+ final)
  float *steps = a.scratch2 + bh * (int64_t)kBlk * DD;  // the states inside one block

  auto load_k = [&](int64_t e) {
    for (int d = tid; d < dk; d += kThreads) kk[d] = ld(a.k, ((b * L + e) * H + h) * dk + d, a.bf16);
  };
  // one sub-step e on the state in S: gate (at a token's first sub-step),
  // then S += beta k (v - S^T k)^T.  `before` (optional) gets the state the
  // update read (after the gate).
  auto fwd_step = [&](int64_t e, float *before) {
    const int64_t t = e / n_h;
    if (a.g && (e % n_h) == 0) {
      const float gt = a.g[(b * T + t) * H + h];
      for (int64_t i = tid; i < DD; i += kThreads) S[i] *= gt;
    }
    load_k(e);
    for (int c = tid; c < dv; c += kThreads) vec[c] = ld(a.v, ((b * L + e) * H + h) * dv + c, a.bf16);
    __syncthreads();
    if (before)
      for (int64_t i = tid; i < DD; i += kThreads) before[i] = S[i];
    for (int c = tid; c < dv; c += kThreads) {
      float acc = 0.f;
      for (int d = 0; d < dk; ++d) acc = fmaf(S[d * dv + c], kk[d], acc);
      u[c] = vec[c] - acc;  // r
    }
    __syncthreads();
    const float bt = a.beta[(b * L + e) * H + h];
    for (int64_t i = tid; i < DD; i += kThreads) S[i] = fmaf(bt * kk[i / dv], u[i % dv], S[i]);
    __syncthreads();
  };

  // ---- forward sweep: block starts into ckpt ----
  for (int64_t i = tid; i < DD; i += kThreads) S[i] = a.h0 ? a.h0[bh * DD + i] : 0.f;
  __syncthreads();
  for (int64_t blk = 0; blk < nblk; ++blk) {
    for (int64_t i = tid; i < DD; i += kThreads) ckpt[blk * DD + i] = S[i];
    for (int64_t e = blk * kBlk; e < L && e < (blk + 1) * kBlk; ++e) fwd_step(e, nullptr);
  }
  // ---- backward sweep ----
  for (int64_t i = tid; i < DD; i += kThreads) dS[i] = a.dhT ? a.dhT[bh * DD + i] : 0.f;
  __syncthreads();
  for (int64_t blk = nblk - 1; blk >= 0; --blk) {
    const int64_t e_lo = blk * kBlk, e_hi = (e_lo + kBlk < L) ? e_lo + kBlk : L;
    // recompute: steps[j] = the state after the gate of sub-step e_lo + j
    // (what its update reads); S ends as the state after the block
    for (int64_t i = tid; i < DD; i += kThreads) S[i] = ckpt[blk * DD + i];
    __syncthreads();
    for (int64_t e = e_lo; e < e_hi; ++e) fwd_step(e, steps + (e - e_lo) * DD);
    for (int64_t e = e_hi - 1; e >= e_lo; --e) {
      const int64_t t = e / n_h;
      const float *P = steps + (e - e_lo) * DD;
      // S = the state after sub-step e: rebuilt from P (the next iteration
      // needs only P of e - 1, so S holds the state after e here)
      load_k(e);
      for (int c = tid; c < dv; c += kThreads) vec[c] = ld(a.v, ((b * L + e) * H + h) * dv + c, a.bf16);
      __syncthreads();
      const float bt = a.beta[(b * L + e) * H + h];
      for (int c = tid; c < dv; c += kThreads) {
        float acc = 0.f;
        for (int d = 0; d < dk; ++d) acc = fmaf(P[d * dv + c], kk[d], acc);
        vec[c] -= acc;  // r = v - P^T k
      }
      __syncthreads();
      for (int64_t i = tid; i < DD; i += kThreads) S[i] = fmaf(bt * kk[i / dv], vec[i % dv], P[i]);
      __syncthreads();
      // readout at the token's last sub-step: dS += q do^T, dq = S do
      if ((int)(e % n_h) == n_h - 1) {
        for (int d = tid; d < dk; d += kThreads) qq[d] = ld(a.q, ((b * T + t) * H + h) * dk + d, a.bf16);
        for (int c = tid; c < dv; c += kThreads) u[c] = ld(a.dout, ((b * T + t) * H + h) * dv + c, a.bf16);
        __syncthreads();
        for (int d = tid; d < dk; d += kThreads) {
          float acc = 0.f;
          for (int c = 0; c < dv; ++c) acc = fmaf(S[d * dv + c], u[c], acc);
          a.gq[((b * T + t) * H + h) * dk + d] = acc;
        }
        for (int64_t i = tid; i < DD; i += kThreads) dS[i] = fmaf(qq[i / dv], u[i % dv], dS[i]);
        __syncthreads();
      }
      // dv = beta dS^T k;  u = dS^T k
      for (int c = tid; c < dv; c += kThreads) {
        float acc = 0.f;
        for (int d = 0; d < dk; ++d) acc = fmaf(dS[d * dv + c], kk[d], acc);
        u[c] = acc;
        a.gv[((b * L + e) * H + h) * dv + c] = bt * acc;
      }
      // w = dS r (over the value index)
      for (int d = tid; d < dk; d += kThreads) {
        float acc = 0.f;
        for (int c = 0; c < dv; ++c) acc = fmaf(dS[d * dv + c], vec[c], acc);
        w[d] = acc;
      }
      __syncthreads();
      // dbeta = k^T dS r
      float part = 0.f;
      for (int d = tid; d < dk; d += kThreads) part = fmaf(kk[d], w[d], part);
      const float dbeta = block_sum(part, red);
      if (tid == 0) a.gbeta[(b * L + e) * H + h] = dbeta;
      // dk = beta (dS r - P dS^T k)
      for (int d = tid; d < dk; d += kThreads) {
        float acc = 0.f;
        for (int c = 0; c < dv; ++c) acc = fmaf(P[d * dv + c], u[c], acc);
        a.gk[((b * L + e) * H + h) * dk + d] = bt * (w[d] - acc);
      }
      __syncthreads();
      // dP = dS - beta k (k^T dS) = dS - beta k u^T
      for (int64_t i = tid; i < DD; i += kThreads) dS[i] = fmaf(-bt * kk[i / dv], u[i % dv], dS[i]);
      __syncthreads();
      // the gate before this sub-step: P = g S_prev
      if (a.g && (e % n_h) == 0) {
        const float gt = a.g[(b * T + t) * H + h];
        // dg = <dP, S_prev> with S_prev the state before the gate: the block
        // start for the block's first sub-step, else the previous sub-step's
        // result P_{e-1} + beta_{e-1} k_{e-1} r_{e-1}^T, rebuilt here (no
        // division by g, which may be 0)
        float pdot = 0.f;
        if (e == e_lo) {
          const float *Sprev = ckpt + blk * DD;
          for (int64_t i = tid; i < DD; i += kThreads) pdot = fmaf(dS[i], Sprev[i], pdot);
        } else {
          const float *Pp = steps + (e - 1 - e_lo) * DD;
          load_k(e - 1);
          for (int c = tid; c < dv; c += kThreads)
            vec[c] = ld(a.v, ((b * L + e - 1) * H + h) * dv + c, a.bf16);
          __syncthreads();
          for (int c = tid; c < dv; c += kThreads) {
            float acc = 0.f;
            for (int d = 0; d < dk; ++d) acc = fmaf(Pp[d * dv + c], kk[d], acc);
            u[c] = vec[c] - acc;
          }
          __syncthreads();
          const float bp = a.beta[(b * L + e - 1) * H + h];
          for (int64_t i = tid; i < DD; i += kThreads)
            pdot = fmaf(dS[i], fmaf(bp * kk[i / dv], u[i % dv], Pp[i]), pdot);
        }
        const float dg = block_sum(pdot, red);
        if (tid == 0) a.gg[(b * T + t) * H + h] = dg;
        for (int64_t i = tid; i < DD; i += kThreads) dS[i] *= gt;
        __syncthreads();
      }
    }
  }
  if (a.gh0)
    for (int64_t i = tid; i < DD; i += kThreads) a.gh0[bh * DD + i] = dS[i];
}

}  // namespace

int64_t bwd_scratch_floats(const BwdArgs &a, int64_t *second) {
  const int64_t DD = (int64_t)a.dk * a.dv, L = a.T * a.n_h;
  const int64_t nblk = (L + kBlk - 1) / kBlk;
  *second = a.B * a.H * (int64_t)kBlk * DD;
  return a.B * a.H * (nblk + 1) * DD;
}

cudaError_t launch_bwd(const BwdArgs &a, cudaStream_t s) {
  const size_t smem = (size_t)(2 * a.dk * a.dv + 3 * a.dk + 2 * a.dv + kThreads / 32) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  bwd_kernel<<<(unsigned)(a.B * a.H), kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace delta
