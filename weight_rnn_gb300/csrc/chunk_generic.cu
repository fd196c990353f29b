// chunk_generic.cu -- chunked delta-rule forward on CUDA cores, float32.
//
// The chunkwise algorithm of "08 · linear 路线（三）：delta rule 与 DPLR 统一框架":
// the UT transform of §2.2, the state passing of §2.3 and the gated form of §3
// (cumulative log decay gc within a chunk, Gam_ij = exp(gc_i - gc_j)), run on
// the extended sequence of "DeltaProduct" §4.1 (n_h sub-steps per token, the
// log gate of token t at its first sub-step and 0 elsewhere, readout at each
// token's last sub-step).  Per chunk of C rows of the extended sequence:
//
//   A   = strictLower(diag(beta) (Gam * K K^T))
//   T   = (I + A)^{-1} diag(beta)                 forward substitution
//   W   = T (K * exp(gc)),  U = T V
//   Vt  = U - W S                                 pseudo-values
//   O   = (Q * exp(gc)) S + (Q K^T * Gam) Vt      readout rows only
//   S  <- exp(gc_C) S + (K * exp(gc_C - gc))^T Vt
//
// With a channel-wise gate (the KDA row of the family table in §1.4: S_t =
// (I - beta k k^T) Diag(alpha_t) S_{t-1} + beta k v^T), gc is a vector per row
// (the cumulative log alpha of each key channel) and every Gam factor above
// becomes the per-channel ratio inside the key dimension's sum:
//
//   A_rj = beta_r sum_d k_rd k_jd exp(gc_rd - gc_jd),  P_rj likewise with q_r
//   W    = T (K * exp(gc)),  O = (Q * exp(gc)) S + P Vt
//   S   <- Diag(exp(gc_C)) S + (K * exp(gc_C - gc))^T Vt
//
// A ragged tail is padded with identity steps (k = v = 0, beta = 0, log g = 0).
// log g is clamped at -80 so that g = 0 (a reset) stays finite: exp(-80) is
// far below float32 resolution relative to the state.
//
// This kernel serves every supported shape and both I/O dtypes; it is the
// float32 path (accurate to ~1e-6) and the fallback for shapes the
// tensor-core kernel does not take.  One CTA handles one (b, h) head and a
// slab of BV value columns; every array lives in shared memory.  The rows of
// K (and of the channel-wise cumulative gate) are padded to dk + 1 floats:
// forming A and P, the lanes of a warp read one key channel of 32 different
// rows, which an unpadded stride of dk floats would put in one bank.
#include <cuda_bf16.h>

#include "kernels.h"

namespace delta {
namespace {

constexpr int kThreads = 256;
constexpr float kLogGateFloor = -80.0f;

__device__ __forceinline__ float load_io(const void *p, int64_t i, bool bf16) {
  return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i])
              : static_cast<const float *>(p)[i];
}

__device__ __forceinline__ void store_io(void *p, int64_t i, float x, bool bf16) {
  if (bf16)
    static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
  else
    static_cast<float *>(p)[i] = x;
}

struct Smem {
  float *S, *K, *Q, *V, *A, *X, *P, *W, *U, *beta, *gc, *eg, *ed, *gcd;
  static __host__ __device__ size_t floats(int C, int dk, int BV, bool kda) {
    return (size_t)dk * BV + (size_t)C * (dk + 1) + 2 * (size_t)C * dk + 2 * (size_t)C * BV +
           3 * (size_t)C * C + 4 * (size_t)C + (kda ? (size_t)C * (dk + 1) : 0);
  }
  __device__ Smem(float *base, int C, int dk, int BV) {
    S = base;
    K = S + dk * BV;        // [C][dk + 1]
    Q = K + C * (dk + 1);
    W = Q + C * dk;
    V = W + C * dk;
    U = V + C * BV;
    A = U + C * BV;
    X = A + C * C;
    P = X + C * C;
    beta = P + C * C;
    gc = beta + C;
    eg = gc + C;   // exp(gc_j), scalar gate
    ed = eg + C;   // exp(gc_C - gc_j), scalar gate
    gcd = ed + C;  // [C][dk + 1], channel-wise gate only
  }
};

template <bool KDA>
__global__ void __launch_bounds__(kThreads)
chunk_generic_kernel(FwdArgs a, int BV) {
  extern __shared__ float smem_raw[];
  const int C = a.chunk, dk = a.dk, n_h = a.n_h;
  Smem sm(smem_raw, C, dk, BV);
  const int tid = threadIdx.x;
  const int64_t bh = blockIdx.x;
  const int64_t b = bh / a.H, h = bh % a.H;
  const int v0 = blockIdx.y * BV;
  const int ks = dk + 1;  // row stride of K and gcd
  const int64_t L = a.L, T = a.T, H = a.H;
  constexpr bool kda = KDA;  // channel-wise gate a.alpha (else the scalar a.g)

  // initial state slab
  for (int i = tid; i < dk * BV; i += kThreads) {
    const int d = i / BV, c = i % BV;
    sm.S[i] = a.h0 ? a.h0[((b * H + h) * dk + d) * a.dv + v0 + c] : 0.0f;
  }

  const int64_t nchunks = (L + C - 1) / C;
  for (int64_t n = 0; n < nchunks; ++n) {
    __syncthreads();  // previous chunk fully consumed
    const int64_t e0 = n * C;
    // ---- load the chunk (extended rows e = t * n_h + j) ----
    for (int i = tid; i < C * dk; i += kThreads) {
      const int r = i / dk, d = i % dk;
      const int64_t e = e0 + r;
      float kv = 0.0f, qv = 0.0f;
      if (e < L) {
        kv = load_io(a.k, ((b * L + e) * H + h) * dk + d, a.bf16);
        if ((int)(e % n_h) == n_h - 1)
          qv = load_io(a.q, ((b * T + e / n_h) * H + h) * dk + d, a.bf16);
      }
      sm.K[r * ks + d] = kv;
      sm.Q[i] = qv;
    }
    for (int i = tid; i < C * BV; i += kThreads) {
      const int r = i / BV, c = i % BV;
      const int64_t e = e0 + r;
      sm.V[i] = e < L ? load_io(a.v, ((b * L + e) * H + h) * a.dv + v0 + c, a.bf16) : 0.0f;
    }
    for (int r = tid; r < C; r += kThreads) {
      const int64_t e = e0 + r;
      float bt = 0.0f, lg = 0.0f;
      if (e < L) {
        bt = a.beta[(b * L + e) * H + h];
        if (a.g && (e % n_h) == 0)
          lg = fmaxf(logf(a.g[(b * T + e / n_h) * H + h]), kLogGateFloor);
      }
      sm.beta[r] = bt;
      sm.gc[r] = lg;
    }
    __syncthreads();
    // inclusive cumulative log gate (C <= 64: one thread; channel-wise: one
    // thread per key channel)
    if (!kda) {
      if (tid == 0) {
        float acc = 0.0f;
        for (int r = 0; r < C; ++r) {
          acc += sm.gc[r];
          sm.gc[r] = acc;
        }
      }
      __syncthreads();
      for (int j = tid; j < C; j += kThreads) {
        sm.eg[j] = expf(sm.gc[j]);
        sm.ed[j] = expf(sm.gc[C - 1] - sm.gc[j]);
      }
    } else {
      for (int d = tid; d < dk; d += kThreads) {
        float acc = 0.0f;
        for (int r = 0; r < C; ++r) {
          const int64_t e = e0 + r;
          if (e < L && (e % n_h) == 0)
            acc += fmaxf(logf(a.alpha[((b * T + e / n_h) * H + h) * dk + d]), kLogGateFloor);
          sm.gcd[r * ks + d] = acc;
        }
      }
    }
    __syncthreads();
    // ---- A (strictly lower, gated) and P (lower incl. diagonal) ----
    for (int i = tid; i < C * C; i += kThreads) {
      const int r = i / C, j = i % C;
      float av = 0.0f, pv = 0.0f, xv = (r == j) ? 1.0f : 0.0f;
      if (j <= r && !kda) {
        const float gam = expf(sm.gc[r] - sm.gc[j]);
        float kk = 0.0f, qk = 0.0f;
        for (int d = 0; d < dk; ++d) {
          const float kj = sm.K[j * ks + d];
          kk = fmaf(sm.K[r * ks + d], kj, kk);
          qk = fmaf(sm.Q[r * dk + d], kj, qk);
        }
        pv = qk * gam;
        if (j < r) av = sm.beta[r] * kk * gam;
      } else if (j <= r) {
        // the ratio of each channel's decay inside the sum (exponent <= 0)
        float kk = 0.0f, qk = 0.0f;
        for (int d = 0; d < dk; ++d) {
          const float kj = sm.K[j * ks + d] * expf(sm.gcd[r * ks + d] - sm.gcd[j * ks + d]);
          kk = fmaf(sm.K[r * ks + d], kj, kk);
          qk = fmaf(sm.Q[r * dk + d], kj, qk);
        }
        pv = qk;
        if (j < r) av = sm.beta[r] * kk;
      }
      sm.A[i] = av;
      sm.P[i] = pv;
      sm.X[i] = xv;
    }
    __syncthreads();
    // ---- X = (I + A)^{-1} by forward substitution, row by row ----
    for (int r = 1; r < C; ++r) {
      for (int j = tid; j < r; j += kThreads) {
        float acc = 0.0f;
        for (int m = j; m < r; ++m) acc = fmaf(sm.A[r * C + m], sm.X[m * C + j], acc);
        sm.X[r * C + j] = -acc;
      }
      __syncthreads();
    }
    // T = X diag(beta), in place in A (A is no longer needed)
    for (int i = tid; i < C * C; i += kThreads) sm.A[i] = sm.X[i] * sm.beta[i % C];
    __syncthreads();
    // ---- W = T (K * exp(gc)), U = T V ----
    for (int i = tid; i < C * dk; i += kThreads) {
      const int r = i / dk, d = i % dk;
      float acc = 0.0f;
      for (int j = 0; j <= r; ++j)
        acc = fmaf(sm.A[r * C + j], sm.K[j * ks + d] * (kda ? expf(sm.gcd[j * ks + d]) : sm.eg[j]), acc);
      sm.W[i] = acc;
    }
    for (int i = tid; i < C * BV; i += kThreads) {
      const int r = i / BV, c = i % BV;
      float acc = 0.0f;
      for (int j = 0; j <= r; ++j) acc = fmaf(sm.A[r * C + j], sm.V[j * BV + c], acc);
      sm.U[i] = acc;
    }
    __syncthreads();
    // ---- Vt = U - W S (in place in U) ----
    for (int i = tid; i < C * BV; i += kThreads) {
      const int r = i / BV, c = i % BV;
      float acc = sm.U[i];
      for (int d = 0; d < dk; ++d) acc = fmaf(-sm.W[r * dk + d], sm.S[d * BV + c], acc);
      sm.U[i] = acc;
    }
    __syncthreads();
    // ---- readout rows: O = (Q * exp(gc)) S + (Q K^T * Gam) Vt ----
    for (int i = tid; i < C * BV; i += kThreads) {
      const int r = i / BV, c = i % BV;
      const int64_t e = e0 + r;
      if (e >= L || (int)(e % n_h) != n_h - 1) continue;
      float qs = 0.0f;
      if (kda) {
        for (int d = 0; d < dk; ++d)
          qs = fmaf(sm.Q[r * dk + d] * expf(sm.gcd[r * ks + d]), sm.S[d * BV + c], qs);
      } else {
        for (int d = 0; d < dk; ++d) qs = fmaf(sm.Q[r * dk + d], sm.S[d * BV + c], qs);
        qs *= sm.eg[r];
      }
      float acc = qs;
      for (int j = 0; j <= r; ++j) acc = fmaf(sm.P[r * C + j], sm.U[j * BV + c], acc);
      store_io(a.out, ((b * T + e / n_h) * H + h) * a.dv + v0 + c, acc, a.bf16);
    }
    __syncthreads();
    // ---- S <- exp(gc_C) S + (K * exp(gc_C - gc))^T Vt ----
    for (int i = tid; i < dk * BV; i += kThreads) {
      const int d = i / BV, c = i % BV;
      float acc;
      if (kda) {
        const float *g = sm.gcd + d;  // this row's cumulative log gate
        const float gl = g[(C - 1) * ks];
        acc = sm.S[i] * expf(gl);
        for (int j = 0; j < C; ++j)
          acc = fmaf(sm.K[j * ks + d] * expf(gl - g[j * ks]), sm.U[j * BV + c], acc);
      } else {
        acc = sm.S[i] * sm.eg[C - 1];
        for (int j = 0; j < C; ++j) acc = fmaf(sm.K[j * ks + d] * sm.ed[j], sm.U[j * BV + c], acc);
      }
      sm.S[i] = acc;
    }
  }
  __syncthreads();
  if (a.hT) {
    for (int i = tid; i < dk * BV; i += kThreads) {
      const int d = i / BV, c = i % BV;
      a.hT[((b * H + h) * dk + d) * a.dv + v0 + c] = sm.S[i];
    }
  }
}

__global__ void state_passthrough_kernel(const float *h0, float *hT, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    hT[i] = h0 ? h0[i] : 0.0f;
}

}  // namespace

cudaError_t launch_chunk_generic(const FwdArgs &a, cudaStream_t s) {
  const int BV = a.dv < 32 ? a.dv : 32;
  const bool kda = a.alpha != nullptr;
  const size_t bytes = Smem::floats(a.chunk, a.dk, BV, kda) * sizeof(float);
  auto kern = kda ? chunk_generic_kernel<true> : chunk_generic_kernel<false>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (err != cudaSuccess) return err;
  dim3 grid((unsigned)(a.B * a.H), (unsigned)(a.dv / BV));
  kern<<<grid, kThreads, bytes, s>>>(a, BV);
  return cudaGetLastError();
}

cudaError_t launch_state_passthrough(const FwdArgs &a, cudaStream_t s) {
  if (!a.hT || a.hT == a.h0) return cudaSuccess;
  const int64_t n = a.B * a.H * a.dk * a.dv;
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  state_passthrough_kernel<<<(unsigned)blocks, 256, 0, s>>>(a.h0, a.hT, n);
  return cudaGetLastError();
}

}  // namespace delta
