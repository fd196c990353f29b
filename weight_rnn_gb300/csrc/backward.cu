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
// One CTA per (b, h) keeps S, dS and the state a sub-step reads, P, [dk][dv]
// in shared memory.  A first sweep runs the forward and stores the state at
// the start of every block of kBlk sub-steps in scratch; the backward sweep
// walks the blocks in reverse, recomputes the block's states from its start
// (stored per sub-step in scratch) and runs the reverse recurrence over them.
// A correctness path: every step is a few dependent matrix-vector products
// over the state.  The dims are powers of two (16 ... 128), so every index
// below is a shift or a mask; each thread owns one column of the elementwise
// passes, and both kinds of matrix-vector product split their sum over
// kThreads / dim parts that meet in `part`.
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
  const int DD = dk * dv;
  const int lgv = __ffs(dv) - 1, lgk = __ffs(dk) - 1;
  float *S = sm;              // [dk][dv]
  float *dS = S + DD;         // [dk][dv]
  float *Ps = dS + DD;        // [dk][dv]: the state the current sub-step read
  float *kk = Ps + DD;        // [dk]
  float *qq = kk + dk;        // [dk]
  float *w = qq + dk;         // [dk]: dS r
  float *vec = w + dk;        // [dv]: v, then r
  float *u = vec + dv;        // [dv]: P^T k, dS^T k, do, ...
  float *red = u + dv;        // [kThreads / 32]
  float *part = red + kThreads / 32;  // [kThreads]
  const int64_t nblk = (L + kBlk - 1) / kBlk;
  float *ckpt = a.scratch + bh * (nblk + 1) * (int64_t)DD;  // block starts
  float *steps = a.scratch2 + bh * (int64_t)kBlk * DD;      // the states inside one block

  // elementwise passes: this thread's column ec, rows er0, er0 + estep, ...
  const int ec = tid & (dv - 1), er0 = tid >> lgv, estep = kThreads >> lgv;
  // y[c] = sum_d M[d][c] x[d]; `out(c, y)` runs on threads c < dv
  auto col_product = [&](const float *M, const float *x, auto out) {
    const int np = kThreads >> lgv, len = dk / np, d0 = (tid >> lgv) * len;
    float acc = 0.f;
    for (int d = d0; d < d0 + len; ++d) acc = fmaf(M[(d << lgv) + ec], x[d], acc);
    part[tid] = acc;
    __syncthreads();
    if (tid < dv) {
      float y = 0.f;
      for (int q = 0; q < np; ++q) y += part[(q << lgv) + tid];
      out(tid, y);
    }
    __syncthreads();
  };
  // y[r] = sum_c M[r][c] x[c]; each part walks its columns from a row-skewed
  // start, so the lanes of a warp (consecutive rows) hit distinct banks
  auto row_product = [&](const float *M, const float *x, auto out) {
    const int r = tid & (dk - 1), np = kThreads >> lgk, len = dv / np, c0 = (tid >> lgk) * len;
    float acc = 0.f;
    for (int j = 0; j < len; ++j) {
      const int c = c0 + ((j + r) & (len - 1));
      acc = fmaf(M[(r << lgv) + c], x[c], acc);
    }
    part[tid] = acc;
    __syncthreads();
    if (tid < dk) {
      float y = 0.f;
      for (int q = 0; q < np; ++q) y += part[(q << lgk) + tid];
      out(tid, y);
    }
    __syncthreads();
  };
  auto load_kv = [&](int64_t e) {
    for (int d = tid; d < dk; d += kThreads) kk[d] = ld(a.k, ((b * L + e) * H + h) * dk + d, a.bf16);
    for (int c = tid; c < dv; c += kThreads) vec[c] = ld(a.v, ((b * L + e) * H + h) * dv + c, a.bf16);
  };
  // r = v - M^T k into vec (vec holds v, kk holds k)
  auto residual = [&](const float *M) {
    col_product(M, kk, [&](int c, float y) { vec[c] -= y; });
  };
  // one sub-step e on the state in S: gate (at a token's first sub-step),
  // then S += beta k (v - S^T k)^T.  `before` (optional) gets the state the
  // update read (after the gate).
  auto fwd_step = [&](int64_t e, float *before) {
    const int64_t t = e / n_h;
    const float gt = (a.g && (e % n_h) == 0) ? a.g[(b * T + t) * H + h] : 1.f;
    const float bt = a.beta[(b * L + e) * H + h];
    load_kv(e);
    for (int r = er0; r < dk; r += estep) {
      const int i = (r << lgv) + ec;
      const float x = S[i] * gt;
      S[i] = x;
      if (before) before[i] = x;
    }
    __syncthreads();
    residual(S);
    const float ur = vec[ec];
    for (int r = er0; r < dk; r += estep) {
      const int i = (r << lgv) + ec;
      S[i] = fmaf(bt * kk[r], ur, S[i]);
    }
    __syncthreads();
  };

  // ---- forward sweep: block starts into ckpt ----
  for (int r = er0; r < dk; r += estep) {
    const int i = (r << lgv) + ec;
    S[i] = a.h0 ? a.h0[bh * DD + i] : 0.f;
  }
  __syncthreads();
  for (int64_t blk = 0; blk < nblk; ++blk) {
    float *dst = ckpt + blk * DD;
    for (int r = er0; r < dk; r += estep) dst[(r << lgv) + ec] = S[(r << lgv) + ec];
    for (int64_t e = blk * kBlk; e < L && e < (blk + 1) * kBlk; ++e) fwd_step(e, nullptr);
  }
  // ---- backward sweep ----
  for (int r = er0; r < dk; r += estep) {
    const int i = (r << lgv) + ec;
    dS[i] = a.dhT ? a.dhT[bh * DD + i] : 0.f;
  }
  __syncthreads();
  bool preloaded = false;  // Ps already holds the state the next sub-step read
  for (int64_t blk = nblk - 1; blk >= 0; --blk) {
    const int64_t e_lo = blk * kBlk, e_hi = (e_lo + kBlk < L) ? e_lo + kBlk : L;
    // recompute: steps[j] = the state after the gate of sub-step e_lo + j
    // (what its update reads)
    const float *src = ckpt + blk * DD;
    for (int r = er0; r < dk; r += estep) S[(r << lgv) + ec] = src[(r << lgv) + ec];
    __syncthreads();
    for (int64_t e = e_lo; e < e_hi; ++e) fwd_step(e, steps + (e - e_lo) * DD);
    preloaded = false;
    for (int64_t e = e_hi - 1; e >= e_lo; --e) {
      const int64_t t = e / n_h;
      const float bt = a.beta[(b * L + e) * H + h];
      if (!preloaded) {
        const float *P = steps + (e - e_lo) * DD;
        for (int r = er0; r < dk; r += estep) Ps[(r << lgv) + ec] = P[(r << lgv) + ec];
      }
      preloaded = false;
      load_kv(e);
      __syncthreads();
      residual(Ps);  // r = v - P^T k
      // S = the state after sub-step e, rebuilt from P
      {
        const float ur = vec[ec];
        for (int r = er0; r < dk; r += estep) {
          const int i = (r << lgv) + ec;
          S[i] = fmaf(bt * kk[r], ur, Ps[i]);
        }
      }
      __syncthreads();
      // readout at the token's last sub-step: dq = S do, dS += q do^T
      if ((int)(e % n_h) == n_h - 1) {
        for (int d = tid; d < dk; d += kThreads) qq[d] = ld(a.q, ((b * T + t) * H + h) * dk + d, a.bf16);
        for (int c = tid; c < dv; c += kThreads) u[c] = ld(a.dout, ((b * T + t) * H + h) * dv + c, a.bf16);
        __syncthreads();
        float *gq = a.gq + ((b * T + t) * H + h) * dk;
        row_product(S, u, [&](int d, float y) { gq[d] = y; });
        const float uo = u[ec];
        for (int r = er0; r < dk; r += estep) {
          const int i = (r << lgv) + ec;
          dS[i] = fmaf(qq[r], uo, dS[i]);
        }
        __syncthreads();
      }
      // u = dS^T k, dv = beta u
      float *gv = a.gv + ((b * L + e) * H + h) * dv;
      col_product(dS, kk, [&](int c, float y) {
        u[c] = y;
        gv[c] = bt * y;
      });
      // w = dS r
      row_product(dS, vec, [&](int d, float y) { w[d] = y; });
      // dbeta = k^T dS r
      float pk = 0.f;
      for (int d = tid; d < dk; d += kThreads) pk = fmaf(kk[d], w[d], pk);
      const float dbeta = block_sum(pk, red);
      if (tid == 0) a.gbeta[(b * L + e) * H + h] = dbeta;
      // dk = beta (dS r - P dS^T k)
      float *gk = a.gk + ((b * L + e) * H + h) * dk;
      row_product(Ps, u, [&](int d, float y) { gk[d] = bt * (w[d] - y); });
      // dP = dS - beta k (k^T dS) = dS - beta k u^T
      {
        const float uc = u[ec];
        for (int r = er0; r < dk; r += estep) {
          const int i = (r << lgv) + ec;
          dS[i] = fmaf(-bt * kk[r], uc, dS[i]);
        }
      }
      __syncthreads();
      // the gate before this sub-step: P = g S_prev
      if (a.g && (e % n_h) == 0) {
        const float gt = a.g[(b * T + t) * H + h];
        // dg = <dP, S_prev> with S_prev the state before the gate: the block
        // start for the block's first sub-step, else the previous sub-step's
        // result P_{e-1} + beta_{e-1} k_{e-1} r_{e-1}^T, rebuilt here (no
        // division by g, which may be 0); P_{e-1} stays in Ps for the next
        // iteration
        float pdot = 0.f;
        if (e == e_lo) {
          for (int r = er0; r < dk; r += estep) {
            const int i = (r << lgv) + ec;
            pdot = fmaf(dS[i], src[i], pdot);
          }
        } else {
          const float *Pp = steps + (e - 1 - e_lo) * DD;
          for (int r = er0; r < dk; r += estep) Ps[(r << lgv) + ec] = Pp[(r << lgv) + ec];
          preloaded = true;
          load_kv(e - 1);
          __syncthreads();
          residual(Ps);
          const float bp = a.beta[(b * L + e - 1) * H + h];
          const float ur = vec[ec];
          for (int r = er0; r < dk; r += estep) {
            const int i = (r << lgv) + ec;
            pdot = fmaf(dS[i], fmaf(bp * kk[r], ur, Ps[i]), pdot);
          }
        }
        const float dg = block_sum(pdot, red);
        if (tid == 0) a.gg[(b * T + t) * H + h] = dg;
        for (int r = er0; r < dk; r += estep) dS[(r << lgv) + ec] *= gt;
        __syncthreads();
      }
    }
  }
  if (a.gh0)
    for (int r = er0; r < dk; r += estep) {
      const int i = (r << lgv) + ec;
      a.gh0[bh * DD + i] = dS[i];
    }
}

}  // namespace

int64_t bwd_scratch_floats(const BwdArgs &a, int64_t *second) {
  const int64_t DD = (int64_t)a.dk * a.dv, L = a.T * a.n_h;
  const int64_t nblk = (L + kBlk - 1) / kBlk;
  *second = a.B * a.H * (int64_t)kBlk * DD;
  return a.B * a.H * (nblk + 1) * DD;
}

cudaError_t launch_bwd(const BwdArgs &a, cudaStream_t s) {
  const size_t smem =
      (size_t)(3 * a.dk * a.dv + 3 * a.dk + 2 * a.dv + kThreads / 32 + kThreads) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  bwd_kernel<<<(unsigned)(a.B * a.H), kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace delta
