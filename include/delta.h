/*
 * delta.h -- C ABI of libdelta: the forward pass of delta-rule linear
 * attention (DeltaNet, Gated DeltaNet, Gated DeltaProduct) and its
 * single-token decode step, for one NVIDIA GB300 (sm_103a); around them the
 * input prologue (delta_prologue and the *_prologue calls), the channel-wise
 * gate (delta_fwd_kda, delta_step_kda), the gradients (delta_bwd) and two
 * diagnostics on the outputs (delta_state_erank, delta_attention_map).
 *
 * The operation.  For every batch row b and head h, independently, a state
 * S in R^{dk x dv} runs through the recurrence
 *
 *     S <- g_t * S                                    (once per token)
 *     for j = 0 .. n_h-1:                             (n_h sub-steps)
 *         S <- (I - beta_tj k_tj k_tj^T) S + beta_tj k_tj v_tj^T
 *     o_t = S^T q_t                                   (after the update)
 *
 * as defined in "08 · linear 路线（三）：delta rule 与 DPLR 统一框架"
 * (llm-infra-atlas), §1.2 (the simplified Householder form) and §3 (Gated
 * DeltaNet, scalar gate), and in "DeltaProduct：通过 Householder 乘积增强线性
 * RNN 的状态追踪" (reading notes), §2.2 (n_h Householder sub-steps per token)
 * and §2.6 (the gate applied once, before the sub-steps).  delta_fwd computes
 * it chunkwise through the WY representation and the UT transform
 * (§2.1-§2.3 and §3 "chunkwise 形式" of the first page), treating DeltaProduct
 * as DeltaNet on the extended sequence of length n_h*T (§4.1 of the second).
 *
 * Conventions common to both calls
 *   - There is no query scale: callers pre-scale q.
 *   - Inputs are used as given: keys are not normalised and beta is not
 *     clamped (||k|| = 1 and beta in [0, 2] keep the recurrence stable).
 *   - g is the LINEAR gate in [0, 1]; g = 0 resets the state.  NULL means 1.
 *   - Every pointer is device memory owned by the caller, contiguous in the
 *     layout given, and 16-byte aligned.  The library keeps no state between
 *     calls and is thread-safe.  The one device allocation it makes is the
 *     scratch of delta_fwd's tensor-core path (below).
 *   - The calls only enqueue work on `stream` and return; they never
 *     synchronise.  Argument errors are returned before anything is enqueued.
 *     A failed launch returns DELTA_ERR_CUDA.  NaN/Inf inputs propagate and
 *     are not detected.
 *   - `out` must not overlap any input.  `hT`/`state` may be updated in place
 *     (hT == h0 is allowed) but must not partially overlap anything else.
 *
 * Supported set: dk, dv in {16, 32, 64, 128}; chunk in {16, 32, 64};
 * 1 <= n_h <= 4; B, H, T >= 0 with B*H < 2^31.  Anything else returns
 * DELTA_ERR_UNSUPPORTED.  Empty problems (B*H*T == 0) are valid.
 *
 * Fast path.  Only DELTA_BF16 with dk = dv = 128 and chunk = 64 (any n_h,
 * gated or not, any T with n_h*T < 2^30 and B*H*ceil(n_h*T/64) < 2^31) runs
 * on the tensor cores (tcgen05, TMEM, TMA), in two kernels: the UT pass
 * (delta_ut_transform) over every chunk at once, then the state pass
 * (delta_fwd_with_ut), one CTA per (b, h).  Every other shape in the
 * supported set -- all DELTA_F32 I/O, head dims below 128, chunk 16 or 32 --
 * runs a float32 CUDA-core kernel meant for correctness checks, about two
 * hundred times slower (39.5 ms against 0.18 ms at B8 H16 T4096, d = 128).
 * delta_step has one kernel for every supported shape (HBM-bound at
 * dk = dv = 128).
 */
#ifndef DELTA_H_
#define DELTA_H_

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* == cudaStream_t; NULL is the legacy default stream */

typedef enum {
    DELTA_OK = 0,
    DELTA_ERR_INVALID = -1,     /* NULL pointer, negative size, bad dtype, overlap */
    DELTA_ERR_UNSUPPORTED = -2, /* outside the supported set above */
    DELTA_ERR_ALIGN = -3,       /* a pointer is not 16-byte aligned */
    DELTA_ERR_CUDA = -4         /* a CUDA call failed; see delta_last_error() */
} delta_status;

typedef enum {
    DELTA_F32 = 0,  /* q, k, v, out are float32 */
    DELTA_BF16 = 1  /* q, k, v, out are bfloat16 (outputs rounded to nearest even) */
} delta_dtype;

/* phi of "DeltaProduct" §2.2, the map from a raw projection to beta */
typedef enum {
    DELTA_BETA_SIGMOID = 0,  /* beta = sigmoid(x), in (0, 1) */
    DELTA_BETA_2SIGMOID = 1  /* beta = 2 sigmoid(x), in (0, 2): reflections allowed */
} delta_beta_map;

/*
 * delta_fwd -- chunked forward over a whole sequence.
 *
 *   q    [B, T, H, dk]        dtype   queries, one per token
 *   k    [B, T, n_h, H, dk]   dtype   keys, one per sub-step
 *   v    [B, T, n_h, H, dv]   dtype   values, one per sub-step
 *   beta [B, T, n_h, H]       float32 write strengths
 *   g    [B, T, H]            float32 linear gate per token, or NULL (=> 1)
 *   h0   [B, H, dk, dv]       float32 initial state (row = key index), or NULL (=> 0)
 *   out  [B, T, H, dv]        dtype   o_t after token t's last sub-step
 *   hT   [B, H, dk, dv]       float32 state after the last token, or NULL (=> not written)
 *   chunk                      rows of the extended sequence per chunk
 *
 * For n_h == 1 the sub-step axis has extent 1, i.e. k is [B, T, H, dk].
 *
 * Scratch.  On the tensor-core path the call takes B*H*ceil(n_h*T/64) * 8 KiB
 * of device memory (the T tiles of every chunk, see delta_ut_transform) as a
 * stream-ordered allocation from a memory pool the library creates once per
 * device, on the current device, and releases it, stream-ordered, before
 * returning; the pool keeps the memory for the next call until the process
 * exits.  Concurrent calls on different streams each get their own block.
 * Callers that manage this memory themselves call delta_ut_transform and
 * delta_fwd_with_ut instead.  An allocation failure returns DELTA_ERR_CUDA
 * with nothing enqueued.
 */
int delta_fwd(const void *q, const void *k, const void *v, const float *beta,
              const float *g, const float *h0, void *out, float *hT,
              int B, int H, int T, int dk, int dv, int n_h, int chunk,
              delta_dtype dtype, struct CUstream_st *stream);

/*
 * delta_fwd_kda -- delta_fwd with a channel-wise gate instead of the scalar
 * one: the KDA row of the family table in "08 · linear 路线（三）" §1.4,
 *
 *   S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *   o_t = S_t^T q_t,
 *
 * the decay of each key row of the state first, then the delta update on the
 * decayed state (§5 of the same page gives it as the DPLR form with w =
 * alpha_t, a = -beta k, b = alpha_t * k).  With n_h > 1 the gate acts once per
 * token, before its sub-steps, as g does in delta_fwd.
 *
 *   alpha [B, T, H, dk]  float32  per-channel linear gate in [0, 1]
 *                                 (log alpha is clamped at -80 inside)
 *   everything else      as in delta_fwd (without g)
 *
 * Runs the float32 CUDA-core chunk kernel for every shape (the tensor-core
 * path takes the scalar gate only): a correctness path, several hundred times
 * slower than delta_fwd's fast path.  Errors as in delta_fwd; alpha must be
 * 16-byte aligned and must not overlap out or hT.
 */
int delta_fwd_kda(const void *q, const void *k, const void *v, const float *beta,
                  const float *alpha, const float *h0, void *out, float *hT,
                  int B, int H, int T, int dk, int dv, int n_h, int chunk,
                  delta_dtype dtype, struct CUstream_st *stream);

/*
 * delta_bwd -- gradients of delta_fwd's outputs and final state with
 * respect to every input, for training.  The pages state no backward
 * formulas: these are the reverse-mode derivatives of the recurrence of
 * "DeltaProduct" §2.6 (gate once per token, then the n_h delta sub-steps,
 * readout after the last), taken one sub-step at a time in float32.
 *
 *   q, k, v, beta, g, h0   as in delta_fwd (g and h0 may be NULL)
 *   dout  [B, T, H, dv]    dtype    gradient of the loss w.r.t. out
 *   dhT   [B, H, dk, dv]   float32  gradient w.r.t. hT, or NULL (=> 0)
 *   grad_q    [B, T, H, dk]       float32  out
 *   grad_k    [B, T, n_h, H, dk]  float32  out
 *   grad_v    [B, T, n_h, H, dv]  float32  out
 *   grad_beta [B, T, n_h, H]      float32  out
 *   grad_g    [B, T, H]           float32  out, required when g is given (else unused)
 *   grad_h0   [B, H, dk, dv]      float32  out, or NULL (=> not written)
 *
 * The update and its reverse act on each value column of the state alone,
 * so every (b, h) is split into groups of 32 value columns (one group when
 * dv <= 32), one CTA per group on the CUDA cores, holding its columns of the
 * state and of its gradient in shared memory.  A CTA runs the forward once
 * storing the state every 64 sub-steps, then walks the sequence backwards,
 * recomputing 64 states at a time.  grad_q, grad_k, grad_beta and grad_g sum
 * over the columns: with several groups each CTA writes partial sums, which a
 * second kernel adds in group order, so results are deterministic.  Scratch:
 * B*H*(ceil(n_h*T/64) + 1 + 64)*dk*dv*4 bytes, plus, when dv > 32, dv/32
 * times the sizes of grad_q, grad_k, grad_beta and grad_g (each rounded up to
 * 16 bytes); stream-ordered from the pool delta_fwd uses, released before
 * returning.  A correctness path (float32 throughout; no tensor cores).  dk, dv in {16, 32, 64, 128},
 * n_h in [1, 4], any dtype; the grad_ outputs must overlap no input and no other
 * output (DELTA_ERR_INVALID); every pointer 16-byte aligned.
 */
int delta_bwd(const void *q, const void *k, const void *v, const float *beta,
              const float *g, const float *h0, const void *dout, const float *dhT,
              float *grad_q, float *grad_k, float *grad_v, float *grad_beta,
              float *grad_g, float *grad_h0, int B, int H, int T, int dk, int dv, int n_h,
              delta_dtype dtype, struct CUstream_st *stream);

/*
 * delta_prologue -- the input prologue on its own: the keys of "DeltaProduct"
 * §2.2, k = psi(x) / ||psi(x)||_2 over the key dimension with psi = SiLU,
 * the queries likewise (the query path of the layer design in "08 · linear
 * 路线（三）" §3: SiLU, then L2 norm), and beta = phi(x), phi = sigmoid or
 * 2 sigmoid.  A vector whose SiLU is all zero becomes the zero vector.
 *
 *   q_raw    [B, T, H, dk]       dtype   in    q_out    same shape, dtype   out
 *   k_raw    [B, T, n_h, H, dk]  dtype   in    k_out    same shape, dtype   out
 *   beta_raw [B, T, n_h, H]      float32 in    beta_out same shape, float32 out
 *
 * One kernel, one read of each input and one write of each output, float32
 * arithmetic (outputs rounded to dtype, nearest even).  All buffers are
 * caller-owned device memory, 16-byte aligned; no output may overlap an input
 * or another output (DELTA_ERR_INVALID).  dk must be in {16, 32, 64, 128}.
 */
int delta_prologue(const void *q_raw, const void *k_raw, const float *beta_raw,
                   void *q_out, void *k_out, float *beta_out, int B, int H, int T, int dk,
                   int n_h, delta_dtype dtype, delta_beta_map beta_map,
                   struct CUstream_st *stream);

/*
 * delta_fwd_prologue -- delta_fwd on raw projections: first the input
 * prologue of "DeltaProduct" §2.2 (each key k = psi(x) / ||psi(x)||_2 over
 * the key dimension with psi = SiLU, beta = phi(x) with phi = sigmoid or
 * 2 sigmoid) with the query path of the layer design in "08 · linear 路线
 * （三）" §3 (SiLU, then the same L2 norm), then delta_fwd on the results.
 *
 *   q_raw    [B, T, H, dk]       dtype   raw query projections
 *   k_raw    [B, T, n_h, H, dk]  dtype   raw key projections
 *   beta_raw [B, T, n_h, H]      float32 raw beta projections
 *   beta_map                      DELTA_BETA_SIGMOID or DELTA_BETA_2SIGMOID
 *   everything else               as in delta_fwd
 *
 * A key or query whose SiLU is all zero is used as the zero vector.  The
 * prologue is delta_prologue's kernel: a single read of q_raw, k_raw and
 * beta_raw and a single write of the normalised q and k (in dtype) and of
 * beta (float32) into stream-ordered scratch from the pool delta_fwd uses (B*H*(T + n_h*T)
 * *dk*sizeof(dtype) + B*H*n_h*T*4 bytes, 256-byte rounded per part),
 * released before the call returns.  Errors as in delta_fwd, plus
 * DELTA_ERR_INVALID for an unknown beta_map.
 */
int delta_fwd_prologue(const void *q_raw, const void *k_raw, const void *v,
                       const float *beta_raw, const float *g, const float *h0, void *out,
                       float *hT, int B, int H, int T, int dk, int dv, int n_h, int chunk,
                       delta_dtype dtype, delta_beta_map beta_map,
                       struct CUstream_st *stream);

/*
 * delta_fwd_static_scratch -- delta_fwd for callers that cannot allocate
 * device memory.  The pages have no counterpart: it is delta_fwd's
 * tensor-core path with its scratch (the T tiles handed from the UT pass to
 * the state pass) in a static device array of the library instead of the
 * memory pool.  Arguments, layouts and results as in delta_fwd.
 *
 *   - Allocates nothing.  The array holds 32 MiB: the T tiles of at most
 *     4096 chunks, i.e. B*H*ceil(n_h*T/64) <= 4096 (e.g. B=1, H=32,
 *     T=8192).  Larger problems return DELTA_ERR_UNSUPPORTED, with the
 *     sizes in delta_last_error(), before anything is enqueued.
 *   - Only DELTA_BF16 with dk = dv = 128 and chunk = 64 (DELTA_ERR_UNSUPPORTED
 *     otherwise); T = 0 copies h0 to hT as delta_fwd does.
 *   - The first call on each device looks up the array's device address
 *     (with that device current) and keeps it; make that first call before
 *     any stream capture.
 *   - Nothing in the array needs clearing: each call writes every tile it
 *     reads.
 *   - There is one array per device: calls that overlap in time on the same
 *     device (on any streams, from any threads) race on it and give wrong
 *     results.  Callers serialise them, e.g. on one stream.
 */
int delta_fwd_static_scratch(const void *q, const void *k, const void *v, const float *beta,
                             const float *g, const float *h0, void *out, float *hT,
                             int B, int H, int T, int dk, int dv, int n_h, int chunk,
                             delta_dtype dtype, struct CUstream_st *stream);

/*
 * delta_ut_transform -- the intra-chunk pass of delta_fwd on its own: the UT
 * transform of "08 · linear 路线（三）" §2.2 with the gated decay of §3, for
 * every chunk n of 64 steps of the extended sequence (length L = n_h*T,
 * "DeltaProduct" §4.1) of every (b, h):
 *
 *   gc_r   = sum_{e <= r} log g_e      (within the chunk; log g_e = log g_t at
 *                                       each token's first sub-step, else 0)
 *   A      = strictLower(diag(beta) (Gam * K K^T)),  Gam_ij = exp(gc_i - gc_j)
 *   T      = (I + A)^{-1} diag(beta)
 *
 *   k, beta, g     as in delta_fwd (bf16 keys, dk = 128)
 *   t_mat [B, H, NT, 64, 64]  bfloat16, row-major, NT = ceil(L / 64); T of
 *                              chunk n; rows past L are identity steps
 *                              (k = 0, beta = 0), i.e. zero rows and columns
 *
 * Only bf16 with dk = 128 and chunk = 64 is supported (DELTA_ERR_UNSUPPORTED
 * otherwise).  t_mat is caller-owned device memory of B*H*NT*8192 bytes,
 * 16-byte aligned, overlapping no input.  The entries are rounded to bf16
 * (nearest even) from a float32 / tf32 solve.
 */
int delta_ut_transform(const void *k, const float *beta, const float *g, void *t_mat,
                       int B, int H, int T, int dk, int n_h, int chunk,
                       delta_dtype dtype, struct CUstream_st *stream);

/*
 * delta_fwd_with_ut -- the state pass of delta_fwd on its own, given the
 * t_mat that delta_ut_transform wrote for the same k, beta and g: W = T (K *
 * exp(gc)), U = T V, the outputs and the state update of "08 · linear 路线
 * （三）" §2.3 and §3, chunk after chunk.  Arguments as in delta_fwd plus
 * t_mat (read only; it must overlap no other argument).  Only bf16 with
 * dk = dv = 128 and chunk = 64 is supported.  Allocates nothing.
 */
int delta_fwd_with_ut(const void *q, const void *k, const void *v, const float *beta,
                      const float *g, const float *h0, const void *t_mat, void *out,
                      float *hT, int B, int H, int T, int dk, int dv, int n_h, int chunk,
                      delta_dtype dtype, struct CUstream_st *stream);

/*
 * delta_step -- one decode token for every (b, h): the recurrent form of
 * "08 · linear 路线（三）" §2.3 (the decode path) with the sub-steps and gate of
 * "DeltaProduct" §2.6.  The float32 state is read once and written once, in
 * place.
 *
 *   q     [B, H, dk]          dtype
 *   k     [B, n_h, H, dk]     dtype
 *   v     [B, n_h, H, dv]     dtype
 *   beta  [B, n_h, H]         float32
 *   g     [B, H]              float32 linear gate, or NULL (=> 1)
 *   state [B, H, dk, dv]      float32, in/out
 *   out   [B, H, dv]          dtype
 *
 * The kernel runs one block per (b, h) and 32-column slab of the state, so
 * B*H*max(1, dv/32) must stay below 2^31; larger sizes return
 * DELTA_ERR_UNSUPPORTED.
 */
int delta_step(const void *q, const void *k, const void *v, const float *beta,
               const float *g, float *state, void *out,
               int B, int H, int dk, int dv, int n_h,
               delta_dtype dtype, struct CUstream_st *stream);

/*
 * delta_step_kda -- delta_step with the channel-wise gate of delta_fwd_kda:
 * alpha [B, H, dk] float32 in place of g.  The decayed state Diag(alpha) S
 * is formed in the same single read of the state; HBM-bound like delta_step.
 * Errors as in delta_step; alpha must be 16-byte aligned and overlap neither
 * state nor out.
 */
int delta_step_kda(const void *q, const void *k, const void *v, const float *beta,
                   const float *alpha, float *state, void *out,
                   int B, int H, int dk, int dv, int n_h,
                   delta_dtype dtype, struct CUstream_st *stream);

/*
 * delta_step_prologue -- delta_step on raw projections, with the input
 * prologue of delta_fwd_prologue ("DeltaProduct" §2.2; "08 · linear 路线
 * （三）" §3) applied inside the decode kernel: q_raw, k_raw and beta_raw
 * take the places of q, k and beta (same shapes and types), beta_map picks
 * phi.  No extra pass over memory and no scratch.  Errors as in delta_step,
 * plus DELTA_ERR_INVALID for an unknown beta_map.
 */
int delta_step_prologue(const void *q_raw, const void *k_raw, const void *v,
                        const float *beta_raw, const float *g, float *state, void *out,
                        int B, int H, int dk, int dv, int n_h, delta_dtype dtype,
                        delta_beta_map beta_map, struct CUstream_st *stream);

/*
 * delta_state_erank -- the effective rank of each state matrix, the spectral
 * diagnostic of "DeltaProduct" §4.6:
 *
 *   erank(S) = exp(-sum_k p_k log p_k),  p_k = sigma_k / sum_j sigma_j
 *
 * over the singular values sigma_k of S (1 <= erank <= rank(S) for S != 0).
 *
 *   state [B, H, dk, dv]  float32 (e.g. hT of delta_fwd, or delta_step's state)
 *   erank [B, H]          float32, written
 *
 * The singular values come from a one-sided Jacobi SVD of each matrix in
 * float32 (columns rotated until every pair is orthogonal to 1e-5 of their
 * norms, at most 40 sweeps).  A zero matrix, where the definition does not
 * apply, gives 0.  dk, dv in {16, 32, 64, 128}; pointers 16-byte aligned,
 * erank not overlapping state.
 */
int delta_state_erank(const float *state, float *erank, int B, int H, int dk, int dv,
                      struct CUstream_st *stream);

/*
 * delta_attention_map -- the fully parallel form of "08 · linear 路线（三）"
 * §2.4 with the gated decay of §3: for a block of N <= 64 steps per (b, h)
 * (n_h = 1, zero initial state), the N x N matrix with o_i = sum_j A_ij v_j,
 *
 *   A = (Q K^T * Gam * M) T,   T = (I + strictLower(diag(beta) (Gam * K K^T)))^{-1} diag(beta)
 *
 * with Gam_ij = exp(gc_i - gc_j), gc the inclusive cumulative log gate, and M
 * the causal mask including the diagonal.
 *
 *   q, k  [B, N, H, dk]   dtype
 *   beta  [B, N, H]       float32
 *   g     [B, N, H]       float32 linear gate, or NULL (=> 1)
 *   attn  [B, H, N, N]    float32, written (row i = readout step i; 0 above the diagonal)
 *
 * float32 arithmetic throughout; log g is clamped at -80 as in delta_fwd.
 * N > 64 returns DELTA_ERR_UNSUPPORTED; dk in {16, 32, 64, 128}.
 */
int delta_attention_map(const void *q, const void *k, const float *beta, const float *g,
                        float *attn, int B, int H, int N, int dk, delta_dtype dtype,
                        struct CUstream_st *stream);

/*
 * delta_fwd_kernel_count -- how many kernels one delta_fwd call with these
 * sizes enqueues (0 for an empty batch), or -1 if delta_fwd would reject
 * them.  Pure host function; nothing is enqueued.
 */
int delta_fwd_kernel_count(int B, int H, int T, int dk, int dv, int n_h, int chunk,
                           delta_dtype dtype);

/* Static English text for a delta_status value. */
const char *delta_status_string(int status);

/*
 * Detail of the last non-OK status returned on the calling thread (for
 * DELTA_ERR_CUDA the CUDA error name and the call that failed).  The pointer
 * stays valid until the next call on the same thread.
 */
const char *delta_last_error(void);

/*
 * delta_check_device -- diagnostic, SYNCHRONOUS: waits for all work on the
 * current device, then reports whether a library kernel gave up on one of its
 * bounded internal waits since the last check (DELTA_ERR_CUDA with the detail
 * in delta_last_error()) and clears that record.  A kernel that gives up ends
 * early instead of hanging; the outputs of that call are then invalid.
 * Also returns DELTA_ERR_CUDA for any pending CUDA error on the device.
 */
int delta_check_device(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int delta_version(void);

/*
 * delta_inject_failure -- test hook: the next `count` calls of delta_fwd,
 * delta_bwd, delta_fwd_kda, delta_step_kda, delta_prologue,
 * delta_fwd_prologue, delta_ut_transform, delta_fwd_with_ut, delta_step,
 * delta_step_prologue, delta_state_erank and delta_attention_map (together)
 * return DELTA_ERR_CUDA, with "injected failure" in delta_last_error(),
 * right after their arguments pass validation and before
 * anything is enqueued.  count = 0 clears a pending injection; count < 0 is
 * DELTA_ERR_INVALID.  The counter is process-wide.
 */
int delta_inject_failure(int count);

/*
 * delta_selftest_wait -- diagnostic: enqueues one warp on `stream` that
 * waits, giving up after `polls` (1 .. 2^24) tries, on a shared-memory
 * barrier that nothing completes -- the bounded-wait path every library
 * kernel takes when a hand-off never arrives.  It gives up and records role
 * 7, barrier 253 in the device error word; the next delta_check_device()
 * returns DELTA_ERR_CUDA and clears it.  Nothing faults, and the context stays
 * usable.  Returns DELTA_ERR_INVALID for polls out of range, DELTA_ERR_CUDA
 * if the launch fails.
 */
int delta_selftest_wait(int polls, struct CUstream_st *stream);

#ifdef __cplusplus
}
#endif

#endif /* DELTA_H_ */
