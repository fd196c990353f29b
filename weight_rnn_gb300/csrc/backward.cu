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
// The delta update acts on every column of the state alone (S[:, c] depends
// only on k, beta and v_c), and so does its reverse: dS[:, c] needs nothing
// from the other columns.  So each (b, h) is split into groups of kCols
// value columns, one CTA per group, which keeps its columns of S, dS and of
// the state a sub-step reads, P, in shared memory.  The gradients that sum
// over the value columns (dq, dk, dbeta, dg) leave each CTA as partial sums,
// which a second kernel adds up in group order (deterministic); dv and dh0
// are per column.  A first sweep runs the forward and stores the state at
// the start of every block of kBlk sub-steps in scratch; the backward sweep
// walks the blocks in reverse, recomputes the block's states from its start
// (stored per sub-step in scratch) and runs the reverse recurrence over
// them.  A correctness path: every step is a few dependent matrix-vector
// products over the state.  The dims are powers of two (16 ... 128), so every
// index below is a shift or a mask; each thread owns one column of the
// elementwise passes, and both kinds of matrix-vector product split their
// sum over several parts that meet in `part`.
#include <cuda_bf16.h>

#include "kernels.h"

namespace delta {
namespace {

constexpr int kThreads = 256;
constexpr int kBlk = 64;   // sub-steps per recomputed block
constexpr int kCols = 32;  // value columns per CTA

__host__ __device__ inline int col_groups(int dv) { return dv > kCols ? dv / kCols : 1; }

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

// sizes of the four summed gradients, each rounded up to 4 floats so that
// every partial array starts 16-byte aligned
struct PartSizes {
  int64_t q, k, b, g;
  __host__ __device__ PartSizes(const BwdArgs &a) {
    const int64_t L = a.T * a.n_h;
    q = (a.B * a.T * a.H * a.dk + 3) & ~int64_t(3);
    k = (a.B * L * a.H * a.dk + 3) & ~int64_t(3);
    b = (a.B * L * a.H + 3) & ~int64_t(3);
    g = a.g ? (a.B * a.T * a.H + 3) & ~int64_t(3) : 0;
  }
  __host__ __device__ int64_t total() const { return q + k + b + g; }
};

__global__ void __launch_bounds__(kThreads, 4) bwd_kernel(BwdArgs a) {
  extern __shared__ float sm[];
  const int dk = a.dk, dv = a.dv, n_h = a.n_h, tid = threadIdx.x;
  const int ng = col_groups(dv), dvs = dv / ng;  // this CTA's columns: cb .. cb + dvs - 1
  const int64_t T = a.T, H = a.H, L = a.T * a.n_h;
  const int64_t cta = blockIdx.x, bh = cta / ng, b = bh / H, h = bh % H;
  const int grp = (int)(cta % ng), cb = grp * dvs;
  const int DD = dk * dvs;
  const int lgv = __ffs(dvs) - 1, lgk = __ffs(dk) - 1;
  float *S = sm;              // [dk][dvs]
  float *dS = S + DD;         // [dk][dvs]
  float *Ps = dS + DD;        // [dk][dvs]: the state the current sub-step read
  float *kk = Ps + DD;        // [dk]
  float *qq = kk + dk;        // [dk]
  float *w = qq + dk;         // [dk]: dS r
  float *vec = w + dk;        // [dvs]: v, then r
  float *u = vec + dvs;       // [dvs]: dS^T k, do, ...
  float *red = u + dvs;       // [kThreads / 32]
  float *part = red + kThreads / 32;  // [kThreads]
  const int64_t nblk = (L + kBlk - 1) / kBlk;
  float *ckpt = a.scratch + cta * (nblk + 1) * (int64_t)DD;  // block starts
  float *steps = a.scratch2 + cta * (int64_t)kBlk * DD;      // the states inside one block
  // the summed gradients: straight to the outputs with one group, else into
  // this group's partial arrays
  float *oq = a.gq, *ok = a.gk, *ob = a.gbeta, *og = a.gg;
  if (ng > 1) {
    const PartSizes ps(a);
    float *base = a.scratch3 + grp * ps.total();
    oq = base;
    ok = base + ps.q;
    ob = ok + ps.k;
    og = a.g ? ob + ps.b : nullptr;
  }

  // elementwise passes: this thread's column ec, rows er0, er0 + estep, ...
  const int ec = tid & (dvs - 1), er0 = tid >> lgv, estep = kThreads >> lgv;
  // state element (r, c) of this group in a [dk][dv] float32 array
  auto gidx = [&](int r, int c) { return (int64_t)r * dv + cb + c; };
  // y[c] = sum_d M[d][c] x[d]; `out(c, y)` runs on threads c < dvs
  auto col_product = [&](const float *M, const float *x, auto out) {
    const int np = kThreads >> lgv, len = dk / np, d0 = (tid >> lgv) * len;
    float acc = 0.f;
    for (int d = d0; d < d0 + len; ++d) acc = fmaf(M[(d << lgv) + ec], x[d], acc);
    part[tid] = acc;
    __syncthreads();
    if (tid < dvs) {
      float y = 0.f;
      for (int q = 0; q < np; ++q) y += part[(q << lgv) + tid];
      out(tid, y);
    }
    __syncthreads();
  };
  // y[r] = sum_c M[r][c] x[c] over this group's columns; each part walks its
  // columns from a row-skewed start, so that the lanes of a warp
  // (consecutive rows) hit distinct banks
  auto row_product = [&](const float *M, const float *x, auto out) {
    const int r = tid & (dk - 1), np = kThreads >> lgk, len = dvs / np, c0 = (tid >> lgk) * len;
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
    for (int c = tid; c < dvs; c += kThreads)
      vec[c] = ld(a.v, ((b * L + e) * H + h) * dv + cb + c, a.bf16);
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
  for (int r = er0; r < dk; r += estep)
    S[(r << lgv) + ec] = a.h0 ? a.h0[bh * dk * dv + gidx(r, ec)] : 0.f;
  __syncthreads();
  for (int64_t blk = 0; blk < nblk; ++blk) {
    float *dst = ckpt + blk * DD;
    for (int r = er0; r < dk; r += estep) dst[(r << lgv) + ec] = S[(r << lgv) + ec];
    for (int64_t e = blk * kBlk; e < L && e < (blk + 1) * kBlk; ++e) fwd_step(e, nullptr);
  }
  // ---- backward sweep ----
  for (int r = er0; r < dk; r += estep)
    dS[(r << lgv) + ec] = a.dhT ? a.dhT[bh * dk * dv + gidx(r, ec)] : 0.f;
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
        for (int c = tid; c < dvs; c += kThreads)
          u[c] = ld(a.dout, ((b * T + t) * H + h) * dv + cb + c, a.bf16);
        __syncthreads();
        float *gq = oq + ((b * T + t) * H + h) * dk;
        row_product(S, u, [&](int d, float y) { gq[d] = y; });
        const float uo = u[ec];
        for (int r = er0; r < dk; r += estep) {
          const int i = (r << lgv) + ec;
          dS[i] = fmaf(qq[r], uo, dS[i]);
        }
        __syncthreads();
      }
      // u = dS^T k, dv = beta u
      float *gv = a.gv + ((b * L + e) * H + h) * dv + cb;
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
      if (tid == 0) ob[(b * L + e) * H + h] = dbeta;
      // dk = beta (dS r - P dS^T k)
      float *gk = ok + ((b * L + e) * H + h) * dk;
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
        if (tid == 0) og[(b * T + t) * H + h] = dg;
        for (int r = er0; r < dk; r += estep) dS[(r << lgv) + ec] *= gt;
        __syncthreads();
      }
    }
  }
  if (a.gh0)
    for (int r = er0; r < dk; r += estep) a.gh0[bh * dk * dv + gidx(r, ec)] = dS[(r << lgv) + ec];
}

// out[i] = sum over the groups g = 0, 1, ... of part[g * stride + i], in
// group order; n floats (16-byte aligned arrays, float4 where n allows)
__global__ void __launch_bounds__(256, 4) bwd_sum_kernel(const float *__restrict__ part, int64_t stride,
                                                      int ng, float *__restrict__ out, int64_t n) {
  const int64_t n4 = n >> 2;
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += step) {
    float4 acc = reinterpret_cast<const float4 *>(part)[i];
    for (int g = 1; g < ng; ++g) {
      const float4 x = reinterpret_cast<const float4 *>(part + g * stride)[i];
      acc.x += x.x;
      acc.y += x.y;
      acc.z += x.z;
      acc.w += x.w;
    }
    reinterpret_cast<float4 *>(out)[i] = acc;
  }
  for (int64_t i = 4 * n4 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += step) {
    float acc = part[i];
    for (int g = 1; g < ng; ++g) acc += part[g * stride + i];
    out[i] = acc;
  }
}

}  // namespace

int64_t bwd_ctas(const BwdArgs &a) { return a.B * a.H * col_groups(a.dv); }

int64_t bwd_scratch_floats(const BwdArgs &a, int64_t *second, int64_t *third) {
  const int64_t DD = (int64_t)a.dk * a.dv, L = a.T * a.n_h;
  const int64_t nblk = (L + kBlk - 1) / kBlk;
  const int ng = col_groups(a.dv);
  *second = a.B * a.H * (int64_t)kBlk * DD;
  *third = ng > 1 ? ng * PartSizes(a).total() : 0;
  return a.B * a.H * (nblk + 1) * DD;
}

cudaError_t launch_bwd(const BwdArgs &a, cudaStream_t s) {
  const int ng = col_groups(a.dv), dvs = a.dv / ng;
  const size_t smem =
      (size_t)(3 * a.dk * dvs + 3 * a.dk + 2 * dvs + kThreads / 32 + kThreads) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  bwd_kernel<<<(unsigned)(a.B * a.H * ng), kThreads, smem, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess || ng == 1) return e;
  // add up the groups' partial sums of the gradients that sum over columns
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const PartSizes ps(a);
  const int64_t L = a.T * a.n_h;
  struct {
    int64_t off, n;
    float *out;
  } parts[4] = {{0, a.B * a.T * a.H * a.dk, a.gq},
                {ps.q, a.B * L * a.H * a.dk, a.gk},
                {ps.q + ps.k, a.B * L * a.H, a.gbeta},
                {ps.q + ps.k + ps.b, a.g ? a.B * a.T * a.H : 0, a.gg}};
  for (const auto &p : parts) {
    if (p.n == 0) continue;
    int64_t blocks = (p.n / 4 + 255) / 256;
    if (blocks > 8LL * sms) blocks = 8LL * sms;
    if (blocks < 1) blocks = 1;
    bwd_sum_kernel<<<(unsigned)blocks, 256, 0, s>>>(a.scratch3 + p.off, ps.total(), ng, p.out, p.n);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace delta
