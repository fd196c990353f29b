// kernels.h -- internal launch interface between the C-ABI layer (api.cu)
// and the CUDA kernels.  Not installed; callers use include/delta.h.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

namespace delta {

// Arguments of one forward call after validation.  Sizes are widened to
// 64 bits; `L` is the extended sequence length n_h * T.
struct FwdArgs {
  const void *q, *k, *v;
  const float *beta, *g, *h0;
  void *out;
  float *hT;
  int64_t B, H, T, L;
  int dk, dv, n_h, chunk;
  bool bf16;
  // channel-wise gate [B, T, H, dk] (KDA), instead of g; nullptr: none
  const float *alpha = nullptr;
};

struct StepArgs {
  const void *q, *k, *v;
  const float *beta, *g;
  float *state;
  void *out;
  int64_t B, H;
  int dk, dv, n_h;
  bool bf16;
  // channel-wise gate [B, H, dk] (KDA), instead of g; nullptr: none
  const float *alpha = nullptr;
  // input prologue applied in the kernel: -1 none (q, k, beta as given);
  // 0: q, k -> SiLU -> L2 norm, beta -> sigmoid; 1: the same, beta -> 2 sigmoid
  int beta_map = -1;
};

// The input prologue as one pass over raw inputs: rows of dk elements
// (rows_q query rows, then rows_k key rows) -> SiLU -> L2 norm, written to
// q_out / k_out in the input dtype; n_beta betas -> sigmoid (beta_map 0) or
// 2 sigmoid (beta_map 1), float32.
struct PrologueArgs {
  const void *q, *k;
  const float *beta;
  void *q_out, *k_out;
  float *beta_out;
  int64_t rows_q, rows_k, n_beta;
  int dk, beta_map;
  bool bf16;
};
cudaError_t launch_prologue(const PrologueArgs &a, cudaStream_t s);

// Gradients of the forward (float32, CUDA cores): inputs as FwdArgs plus the
// loss gradients dout (dtype) and dhT (float32, or nullptr); outputs, all
// float32: gq [B,T,H,dk], gk [B,L,H,dk], gv [B,L,H,dv], gbeta [B,L,H], gg
// [B,T,H] (when g is set) and gh0 [B,H,dk,dv] (or nullptr).  scratch holds
// bwd_scratch_floats() floats (block-start states), scratch2 `second` floats
// (the states inside one block), scratch3 `third` floats (the per-column-group
// partial sums of gq, gk, gbeta and gg; none when one group covers dv).
struct BwdArgs {
  const void *q, *k, *v, *dout;
  const float *beta, *g, *h0, *dhT;
  float *gq, *gk, *gv, *gbeta, *gg, *gh0;
  float *scratch, *scratch2, *scratch3;
  int64_t B, H, T;
  int dk, dv, n_h;
  bool bf16;
};
int64_t bwd_scratch_floats(const BwdArgs &a, int64_t *second, int64_t *third);
int64_t bwd_ctas(const BwdArgs &a);  // the grid of the backward kernel
cudaError_t launch_bwd(const BwdArgs &a, cudaStream_t s);

// Generic chunked forward on CUDA cores, float32 arithmetic, any supported
// shape.  Returns the launch error (cudaSuccess if enqueued).
cudaError_t launch_chunk_generic(const FwdArgs &a, cudaStream_t s);

// Tensor-core chunked forward (tcgen05 + TMEM + TMA) for bf16 I/O with
// dk = dv = 128 and chunk = 64: the state pass, given the T tiles the UT pass
// (launch_ut) wrote to t_mat.  Returns cudaErrorNotSupported when the shape
// is outside that set.
cudaError_t launch_chunk_tc(const FwdArgs &a, const void *t_mat, cudaStream_t s);
bool chunk_tc_supports(const FwdArgs &a);
// kernels one tensor-core forward launches (UT pass + state pass)
constexpr int kChunkTcKernels = 2;

// The intra-chunk UT transform T = (I + A)^{-1} diag(beta) of every chunk,
// bf16 [B*H*NT][64][64] row-major (tensor cores; bf16 keys, dk = 128,
// chunk = 64).  t_mat must hold ut_workspace_bytes(a) bytes, 16-byte aligned.
bool ut_supports(const FwdArgs &a);
int64_t ut_workspace_bytes(const FwdArgs &a);
cudaError_t launch_ut(const FwdArgs &a, void *t_mat, cudaStream_t s);

// Read and clear the word the tensor-core kernels set when one of their
// bounded waits gives up (0 = no error).  Synchronises the device.
cudaError_t read_and_clear_tc_error(unsigned int *word);
cudaError_t read_and_clear_ut_error(unsigned int *word);

// One warp waits, at most `polls` tries, on a barrier that nothing completes,
// then records its giving up in the same device error word.
cudaError_t launch_wait_selftest(unsigned int polls, cudaStream_t s);

// hT <- h0 (or 0) for an empty sequence (T == 0).
cudaError_t launch_state_passthrough(const FwdArgs &a, cudaStream_t s);

// One decode step, state updated in place.
cudaError_t launch_step(const StepArgs &a, cudaStream_t s);

// Effective rank of each of the BH state matrices [dk][dv] (float32) into
// erank[BH]; one block per matrix with erank_smem_bytes of shared memory.
int64_t erank_smem_bytes(int dk, int dv);
cudaError_t launch_erank(const float *state, float *erank, int64_t BH, int dk, int dv,
                         cudaStream_t s);

// The attention map of the fully parallel form for N <= 64 steps (n_h = 1):
// q, k [B][N][H][dk] (bf16 or float32), beta, g [B][N][H], attn [B][H][N][N].
cudaError_t launch_attention_map(const void *q, const void *k, const float *beta, const float *g,
                                 float *attn, int64_t B, int64_t H, int N, int dk, bool bf16,
                                 cudaStream_t s);

}  // namespace delta
