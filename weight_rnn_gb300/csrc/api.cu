// api.cu -- the C ABI declared in include/delta.h: argument validation,
// kernel selection, scratch memory for the tensor-core forward and error
// reporting.  Nothing is synchronised: each call enqueues work on the
// caller's stream and returns.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdarg>
#include <cstring>
#include <mutex>

#include "../../include/delta.h"
#include "kernels.h"

// Scratch of delta_fwd_static_scratch: the T tiles of at most 4096 chunks
// (8 KiB each), in a file-scope device array, so that the call allocates
// nothing.  Every tile the state pass reads is written by the same call's UT
// pass first, so nothing in it has to start at zero.
constexpr int64_t kStaticScratchBytes = int64_t(32) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {

thread_local char g_last_error[256] = "no error";
// calls still to fail on purpose (delta_inject_failure)
std::atomic<int> g_inject{0};

// true (and one injection used up) when this call is to fail on purpose
bool take_injection() {
  int n = g_inject.load();
  while (n > 0)
    if (g_inject.compare_exchange_weak(n, n - 1)) return true;
  return false;
}

int fail(int status, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int status, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t err, const char *what) {
  return fail(DELTA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(err),
              cudaGetErrorString(err));
}

bool supported_dim(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool supported_chunk(int c) { return c == 16 || c == 32 || c == 64; }
bool aligned16(const void *p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
};
Range range(const void *p, int64_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return Range{lo, lo + (uintptr_t)bytes};
}
bool overlap(Range a, Range b) {
  return a.lo != 0 && b.lo != 0 && a.hi > a.lo && b.hi > b.lo && a.lo < b.hi && b.lo < a.hi;
}

// Scratch for the T tiles handed from the UT pass to the state pass: stream-
// ordered allocations from one memory pool per device, owned by the library,
// that keeps freed memory for reuse (release threshold: unlimited), so calls
// after the first reuse it without reaching the driver.
constexpr int kMaxDevices = 64;
std::mutex g_pool_mu;
cudaMemPool_t g_pool[kMaxDevices] = {};

cudaError_t scratch_pool(cudaMemPool_t *out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_pool_mu);
  if (!g_pool[dev]) {
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool;
    if ((e = cudaMemPoolCreate(&pool, &props)) != cudaSuccess) return e;
    uint64_t keep = UINT64_MAX;
    if ((e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
      cudaMemPoolDestroy(pool);
      return e;
    }
    g_pool[dev] = pool;
  }
  *out = g_pool[dev];
  return cudaSuccess;
}

// Device address of g_static_scratch on the current device, looked up (with
// that device current) the first time each device asks.
std::mutex g_static_mu;
void *g_static_addr[kMaxDevices] = {};

cudaError_t static_scratch(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[dev]) {
    void *p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_static_scratch)) != cudaSuccess) return e;
    g_static_addr[dev] = p;
  }
  *out = g_static_addr[dev];
  return cudaSuccess;
}

// Checks shared by the forward entry points; fills `a` on success.
int validate_fwd(const void *q, const void *k, const void *v, const float *beta,
                 const float *g, const float *h0, void *out, float *hT, int B, int H,
                 int T, int dk, int dv, int n_h, int chunk, delta_dtype dtype,
                 delta::FwdArgs &a) {
  if (B < 0 || H < 0 || T < 0)
    return fail(DELTA_ERR_INVALID, "negative size B=%d H=%d T=%d", B, H, T);
  if (dtype != DELTA_F32 && dtype != DELTA_BF16)
    return fail(DELTA_ERR_INVALID, "unknown dtype %d", (int)dtype);
  if (!supported_dim(dk) || !supported_dim(dv))
    return fail(DELTA_ERR_UNSUPPORTED, "dk=%d dv=%d not in {16,32,64,128}", dk, dv);
  if (!supported_chunk(chunk))
    return fail(DELTA_ERR_UNSUPPORTED, "chunk=%d not in {16,32,64}", chunk);
  if (n_h < 1 || n_h > 4) return fail(DELTA_ERR_UNSUPPORTED, "n_h=%d not in [1,4]", n_h);
  if ((int64_t)B * H >= (int64_t(1) << 31))
    return fail(DELTA_ERR_UNSUPPORTED, "B*H=%lld too large", (long long)B * H);

  const int64_t esz = dtype == DELTA_BF16 ? 2 : 4;
  const int64_t BH = (int64_t)B * H;
  const int64_t L = (int64_t)T * n_h;
  const int64_t state_bytes = BH * dk * dv * 4;
  a = delta::FwdArgs{};
  a.q = q; a.k = k; a.v = v; a.beta = beta; a.g = g; a.h0 = h0;
  a.out = out; a.hT = hT;
  a.B = B; a.H = H; a.T = T; a.L = L;
  a.dk = dk; a.dv = dv; a.n_h = n_h; a.chunk = chunk;
  a.bf16 = dtype == DELTA_BF16;
  if (BH == 0) return DELTA_OK;
  if (T > 0 && (!q || !k || !v || !beta || !out))
    return fail(DELTA_ERR_INVALID, "q, k, v, beta and out must be non-NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(beta) ||
      !aligned16(g) || !aligned16(h0) || !aligned16(out) || !aligned16(hT))
    return fail(DELTA_ERR_ALIGN, "every pointer must be 16-byte aligned");

  const Range r_out = range(out, BH * T * dv * esz);
  const Range r_hT = range(hT, state_bytes);
  const Range inputs[] = {range(q, BH * T * dk * esz), range(k, BH * L * dk * esz),
                          range(v, BH * L * dv * esz),  range(beta, BH * L * 4),
                          range(g, g ? BH * T * 4 : 0), range(h0, h0 ? state_bytes : 0)};
  for (const Range &r : inputs)
    if (overlap(r_out, r)) return fail(DELTA_ERR_INVALID, "out overlaps an input");
  for (int i = 0; i < 5; ++i)
    if (overlap(r_hT, inputs[i])) return fail(DELTA_ERR_INVALID, "hT overlaps an input");
  if (overlap(r_hT, r_out)) return fail(DELTA_ERR_INVALID, "hT overlaps out");
  if (hT && h0 && (const void *)hT != (const void *)h0 && overlap(r_hT, inputs[5]))
    return fail(DELTA_ERR_INVALID, "hT partially overlaps h0");
  return DELTA_OK;
}

// t_mat of the tensor-core shape: present, aligned and clear of the rest.
int validate_t_mat(const delta::FwdArgs &a, const void *t_mat, bool with_outputs) {
  if (!t_mat) return fail(DELTA_ERR_INVALID, "t_mat must be non-NULL");
  if (!aligned16(t_mat)) return fail(DELTA_ERR_ALIGN, "t_mat must be 16-byte aligned");
  const int64_t BH = a.B * a.H;
  const Range r_t = range(t_mat, delta::ut_workspace_bytes(a));
  const Range others[] = {range(a.k, BH * a.L * a.dk * 2), range(a.beta, BH * a.L * 4),
                          range(a.g, a.g ? BH * a.T * 4 : 0),
                          range(with_outputs ? a.q : nullptr, BH * a.T * a.dk * 2),
                          range(with_outputs ? a.v : nullptr, BH * a.L * a.dv * 2),
                          range(with_outputs ? a.h0 : nullptr, a.h0 ? BH * a.dk * a.dv * 4 : 0),
                          range(with_outputs ? a.out : nullptr, BH * a.T * a.dv * 2),
                          range(with_outputs ? a.hT : nullptr, BH * a.dk * a.dv * 4)};
  for (const Range &r : others)
    if (overlap(r_t, r)) return fail(DELTA_ERR_INVALID, "t_mat overlaps another argument");
  return DELTA_OK;
}

// The forward of a validated call (B*H > 0): the tensor-core path with its
// T-tile scratch, the state pass-through for T = 0, or the generic kernel.
int run_fwd(const delta::FwdArgs &a, cudaStream_t s) {
  cudaError_t err;
  if (a.T == 0) {
    err = delta::launch_state_passthrough(a, s);
    return err == cudaSuccess ? DELTA_OK : cuda_fail(err, "state passthrough launch");
  }
  if (delta::chunk_tc_supports(a)) {
    // the T tiles of every chunk live in stream-ordered scratch between the
    // two passes and are released (stream-ordered) after the second
    cudaMemPool_t pool;
    if ((err = scratch_pool(&pool)) != cudaSuccess) return cuda_fail(err, "scratch pool");
    void *t_mat = nullptr;
    err = cudaMallocFromPoolAsync(&t_mat, (size_t)delta::ut_workspace_bytes(a), pool, s);
    if (err != cudaSuccess) return cuda_fail(err, "scratch allocation");
    err = delta::launch_ut(a, t_mat, s);
    const char *what = "UT-pass kernel launch";
    if (err == cudaSuccess) {
      err = delta::launch_chunk_tc(a, t_mat, s);
      what = "tensor-core chunk kernel launch";
    }
    const cudaError_t ef = cudaFreeAsync(t_mat, s);
    if (err != cudaSuccess) return cuda_fail(err, what);
    return ef == cudaSuccess ? DELTA_OK : cuda_fail(ef, "scratch release");
  }
  err = delta::launch_chunk_generic(a, s);
  return err == cudaSuccess ? DELTA_OK : cuda_fail(err, "generic chunk kernel launch");
}

// Checks of delta_prologue's arguments (rows of q and k, betas).
int validate_prologue(const void *q_raw, const void *k_raw, const float *beta_raw, void *q_out,
                      void *k_out, float *beta_out, int B, int H, int T, int dk, int n_h,
                      delta_dtype dtype, delta_beta_map beta_map) {
  if (beta_map != DELTA_BETA_SIGMOID && beta_map != DELTA_BETA_2SIGMOID)
    return fail(DELTA_ERR_INVALID, "unknown beta_map %d", (int)beta_map);
  if (B < 0 || H < 0 || T < 0)
    return fail(DELTA_ERR_INVALID, "negative size B=%d H=%d T=%d", B, H, T);
  if (dtype != DELTA_F32 && dtype != DELTA_BF16)
    return fail(DELTA_ERR_INVALID, "unknown dtype %d", (int)dtype);
  if (!supported_dim(dk)) return fail(DELTA_ERR_UNSUPPORTED, "dk=%d not in {16,32,64,128}", dk);
  if (n_h < 1 || n_h > 4) return fail(DELTA_ERR_UNSUPPORTED, "n_h=%d not in [1,4]", n_h);
  const int64_t BH = (int64_t)B * H, esz = dtype == DELTA_BF16 ? 2 : 4;
  if (BH * T == 0) return DELTA_OK;
  if (!q_raw || !k_raw || !beta_raw || !q_out || !k_out || !beta_out)
    return fail(DELTA_ERR_INVALID, "every pointer must be non-NULL");
  if (!aligned16(q_raw) || !aligned16(k_raw) || !aligned16(beta_raw) || !aligned16(q_out) ||
      !aligned16(k_out) || !aligned16(beta_out))
    return fail(DELTA_ERR_ALIGN, "every pointer must be 16-byte aligned");
  const int64_t L = (int64_t)T * n_h;
  const Range outs[] = {range(q_out, BH * T * dk * esz), range(k_out, BH * L * dk * esz),
                        range(beta_out, BH * L * 4)};
  const Range ins[] = {range(q_raw, BH * T * dk * esz), range(k_raw, BH * L * dk * esz),
                       range(beta_raw, BH * L * 4)};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 3; ++j)
      if (overlap(outs[i], ins[j])) return fail(DELTA_ERR_INVALID, "an output overlaps an input");
    for (int j = i + 1; j < 3; ++j)
      if (overlap(outs[i], outs[j])) return fail(DELTA_ERR_INVALID, "two outputs overlap");
  }
  return DELTA_OK;
}

delta::PrologueArgs prologue_args(const void *q_raw, const void *k_raw, const float *beta_raw,
                                  void *q_out, void *k_out, float *beta_out, int64_t BH, int64_t T,
                                  int dk, int n_h, bool bf16, delta_beta_map beta_map) {
  delta::PrologueArgs p;
  p.q = q_raw; p.k = k_raw; p.beta = beta_raw;
  p.q_out = q_out; p.k_out = k_out; p.beta_out = beta_out;
  p.rows_q = BH * T; p.rows_k = BH * T * n_h; p.n_beta = BH * T * n_h;
  p.dk = dk; p.beta_map = beta_map == DELTA_BETA_2SIGMOID ? 1 : 0; p.bf16 = bf16;
  return p;
}

// Checks of delta_step's arguments.
int validate_step(const void *q, const void *k, const void *v, const float *beta,
                  const float *g, float *state, void *out, int B, int H, int dk, int dv,
                  int n_h, delta_dtype dtype) {
  if (B < 0 || H < 0) return fail(DELTA_ERR_INVALID, "negative size B=%d H=%d", B, H);
  if (dtype != DELTA_F32 && dtype != DELTA_BF16)
    return fail(DELTA_ERR_INVALID, "unknown dtype %d", (int)dtype);
  if (!supported_dim(dk) || !supported_dim(dv))
    return fail(DELTA_ERR_UNSUPPORTED, "dk=%d dv=%d not in {16,32,64,128}", dk, dv);
  if (n_h < 1 || n_h > 4) return fail(DELTA_ERR_UNSUPPORTED, "n_h=%d not in [1,4]", n_h);
  if ((int64_t)B * H >= (int64_t(1) << 31))
    return fail(DELTA_ERR_UNSUPPORTED, "B*H=%lld too large", (long long)B * H);
  const int64_t BH = (int64_t)B * H;
  if (BH == 0) return DELTA_OK;
  // one CTA per (b, h) and 32-column slab of the state: the grid must fit
  // gridDim.x
  if (BH * (dv < 32 ? 1 : dv / 32) > INT32_MAX)
    return fail(DELTA_ERR_UNSUPPORTED, "B*H*(dv/32)=%lld blocks exceed 2^31-1",
                (long long)(BH * (dv < 32 ? 1 : dv / 32)));
  if (!q || !k || !v || !beta || !state || !out)
    return fail(DELTA_ERR_INVALID, "q, k, v, beta, state and out must be non-NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(beta) ||
      !aligned16(g) || !aligned16(state) || !aligned16(out))
    return fail(DELTA_ERR_ALIGN, "every pointer must be 16-byte aligned");
  const int64_t esz = dtype == DELTA_BF16 ? 2 : 4;
  const Range r_state = range(state, BH * dk * dv * 4);
  const Range r_out = range(out, BH * dv * esz);
  const Range inputs[] = {range(q, BH * dk * esz), range(k, BH * n_h * dk * esz),
                          range(v, BH * n_h * dv * esz), range(beta, BH * n_h * 4),
                          range(g, g ? BH * 4 : 0)};
  for (const Range &r : inputs) {
    if (overlap(r_out, r)) return fail(DELTA_ERR_INVALID, "out overlaps an input");
    if (overlap(r_state, r)) return fail(DELTA_ERR_INVALID, "state overlaps an input");
  }
  if (overlap(r_state, r_out)) return fail(DELTA_ERR_INVALID, "state overlaps out");
  return DELTA_OK;
}

int run_step(const void *q, const void *k, const void *v, const float *beta, const float *g,
             float *state, void *out, int B, int H, int dk, int dv, int n_h, delta_dtype dtype,
             int beta_map, struct CUstream_st *stream, const float *alpha = nullptr,
             bool kda = false) {
  const int st = validate_step(q, k, v, beta, g, state, out, B, H, dk, dv, n_h, dtype);
  if (st != DELTA_OK || (int64_t)B * H == 0) return st;
  if (kda) {
    if (!alpha) return fail(DELTA_ERR_INVALID, "alpha must be non-NULL");
    if (!aligned16(alpha)) return fail(DELTA_ERR_ALIGN, "every pointer must be 16-byte aligned");
    const int64_t BH = (int64_t)B * H, esz = dtype == DELTA_BF16 ? 2 : 4;
    const Range r_a = range(alpha, BH * dk * 4);
    if (overlap(r_a, range(state, BH * dk * dv * 4)))
      return fail(DELTA_ERR_INVALID, "state overlaps alpha");
    if (overlap(r_a, range(out, BH * dv * esz))) return fail(DELTA_ERR_INVALID, "out overlaps alpha");
  }
  if (take_injection()) return fail(DELTA_ERR_CUDA, "injected failure (delta_inject_failure)");
  delta::StepArgs a;
  a.q = q; a.k = k; a.v = v; a.beta = beta; a.g = g; a.state = state; a.out = out;
  a.B = B; a.H = H; a.dk = dk; a.dv = dv; a.n_h = n_h;
  a.bf16 = dtype == DELTA_BF16;
  a.beta_map = beta_map;
  a.alpha = alpha;
  const cudaError_t err = delta::launch_step(a, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? DELTA_OK : cuda_fail(err, "decode step launch");
}

}  // namespace

extern "C" {

const char *delta_status_string(int status) {
  switch (status) {
    case DELTA_OK: return "success";
    case DELTA_ERR_INVALID: return "invalid argument";
    case DELTA_ERR_UNSUPPORTED: return "unsupported shape or option";
    case DELTA_ERR_ALIGN: return "pointer not 16-byte aligned";
    case DELTA_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

const char *delta_last_error(void) { return g_last_error; }

int delta_version(void) { return 100; }

int delta_inject_failure(int count) {
  if (count < 0) return fail(DELTA_ERR_INVALID, "count=%d is negative", count);
  g_inject.store(count);
  return DELTA_OK;
}

int delta_selftest_wait(int polls, struct CUstream_st *stream) {
  if (polls < 1 || polls > (1 << 24)) return fail(DELTA_ERR_INVALID, "polls=%d not in [1, 2^24]", polls);
  const cudaError_t err = delta::launch_wait_selftest((unsigned)polls, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? DELTA_OK : cuda_fail(err, "wait self-test launch");
}

int delta_check_device(void) {
  unsigned int word = 0, ut_word = 0;
  cudaError_t err = delta::read_and_clear_tc_error(&word);
  if (err == cudaSuccess) err = delta::read_and_clear_ut_error(&ut_word);
  if (err != cudaSuccess) return cuda_fail(err, "device check");
  if (word != 0)
    return fail(DELTA_ERR_CUDA,
                "a kernel wait gave up (role %u, barrier %u): results of that call are invalid",
                (word & 0xffu) - 1, word >> 8);
  if (ut_word != 0)
    return fail(DELTA_ERR_CUDA,
                "a UT-pass wait gave up (role %u, barrier %u): results of that call are invalid",
                (ut_word & 0xffu) - 1, ut_word >> 8);
  return DELTA_OK;
}

int delta_fwd(const void *q, const void *k, const void *v, const float *beta,
              const float *g, const float *h0, void *out, float *hT, int B, int H,
              int T, int dk, int dv, int n_h, int chunk, delta_dtype dtype,
              struct CUstream_st *stream) {
  delta::FwdArgs a;
  const int st = validate_fwd(q, k, v, beta, g, h0, out, hT, B, H, T, dk, dv, n_h, chunk, dtype, a);
  if (st != DELTA_OK || a.B * a.H == 0) return st;
  if (take_injection()) return fail(DELTA_ERR_CUDA, "injected failure (delta_inject_failure)");
  return run_fwd(a, reinterpret_cast<cudaStream_t>(stream));
}

int delta_fwd_prologue(const void *q_raw, const void *k_raw, const void *v, const float *beta_raw,
                       const float *g, const float *h0, void *out, float *hT, int B, int H,
                       int T, int dk, int dv, int n_h, int chunk, delta_dtype dtype,
                       delta_beta_map beta_map, struct CUstream_st *stream) {
  if (beta_map != DELTA_BETA_SIGMOID && beta_map != DELTA_BETA_2SIGMOID)
    return fail(DELTA_ERR_INVALID, "unknown beta_map %d", (int)beta_map);
  delta::FwdArgs a;
  const int st = validate_fwd(q_raw, k_raw, v, beta_raw, g, h0, out, hT, B, H, T, dk, dv, n_h,
                              chunk, dtype, a);
  if (st != DELTA_OK || a.B * a.H == 0) return st;
  if (take_injection()) return fail(DELTA_ERR_CUDA, "injected failure (delta_inject_failure)");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) return run_fwd(a, s);
  // the normalised q and k and the mapped beta, in stream-ordered scratch
  // (one allocation, 256-byte aligned parts), released after the forward
  const int64_t BH = a.B * a.H, esz = a.bf16 ? 2 : 4;
  const auto up = [](int64_t n) { return (n + 255) & ~int64_t(255); };
  const int64_t bq = up(BH * a.T * dk * esz), bk = up(BH * a.L * dk * esz), bb = up(BH * a.L * 4);
  cudaMemPool_t pool;
  cudaError_t err = scratch_pool(&pool);
  if (err != cudaSuccess) return cuda_fail(err, "scratch pool");
  void *scratch = nullptr;
  err = cudaMallocFromPoolAsync(&scratch, (size_t)(bq + bk + bb), pool, s);
  if (err != cudaSuccess) return cuda_fail(err, "scratch allocation");
  uint8_t *base = static_cast<uint8_t *>(scratch);
  const delta::PrologueArgs p =
      prologue_args(q_raw, k_raw, beta_raw, base, base + bq,
                    reinterpret_cast<float *>(base + bq + bk), BH, a.T, dk, n_h, a.bf16, beta_map);
  err = delta::launch_prologue(p, s);
  int rc = DELTA_OK;
  if (err != cudaSuccess) {
    rc = cuda_fail(err, "prologue kernel launch");
  } else {
    a.q = p.q_out; a.k = p.k_out; a.beta = p.beta_out;
    rc = run_fwd(a, s);
  }
  const cudaError_t ef = cudaFreeAsync(scratch, s);
  if (rc != DELTA_OK) return rc;
  return ef == cudaSuccess ? DELTA_OK : cuda_fail(ef, "scratch release");
}

int delta_fwd_kda(const void *q, const void *k, const void *v, const float *beta,
                  const float *alpha, const float *h0, void *out, float *hT, int B, int H, int T,
                  int dk, int dv, int n_h, int chunk, delta_dtype dtype,
                  struct CUstream_st *stream) {
  delta::FwdArgs a;
  const int st = validate_fwd(q, k, v, beta, nullptr, h0, out, hT, B, H, T, dk, dv, n_h, chunk,
                              dtype, a);
  if (st != DELTA_OK || a.B * a.H == 0) return st;
  if (T > 0) {
    if (!alpha) return fail(DELTA_ERR_INVALID, "alpha must be non-NULL");
    if (!aligned16(alpha)) return fail(DELTA_ERR_ALIGN, "every pointer must be 16-byte aligned");
    const int64_t esz = a.bf16 ? 2 : 4, BH = a.B * a.H;
    const Range r_a = range(alpha, BH * a.T * dk * 4);
    if (overlap(r_a, range(out, BH * a.T * dv * esz)))
      return fail(DELTA_ERR_INVALID, "out overlaps alpha");
    if (overlap(r_a, range(hT, BH * dk * dv * 4)))
      return fail(DELTA_ERR_INVALID, "hT overlaps alpha");
  }
  if (take_injection()) return fail(DELTA_ERR_CUDA, "injected failure (delta_inject_failure)");
  a.alpha = alpha;
  return run_fwd(a, reinterpret_cast<cudaStream_t>(stream));
}

int delta_bwd(const void *q, const void *k, const void *v, const float *beta, const float *g,
              const float *h0, const void *dout, const float *dhT, float *dq, float *dk,
              float *dv, float *dbeta, float *dg, float *dh0, int B, int H, int T, int dk_,
              int dv_, int n_h, delta_dtype dtype, struct CUstream_st *stream) {
  if (B < 0 || H < 0 || T < 0)
    return fail(DELTA_ERR_INVALID, "negative size B=%d H=%d T=%d", B, H, T);
  if (dtype != DELTA_F32 && dtype != DELTA_BF16)
    return fail(DELTA_ERR_INVALID, "unknown dtype %d", (int)dtype);
  if (!supported_dim(dk_) || !supported_dim(dv_))
    return fail(DELTA_ERR_UNSUPPORTED, "dk=%d dv=%d not in {16,32,64,128}", dk_, dv_);
  if (n_h < 1 || n_h > 4) return fail(DELTA_ERR_UNSUPPORTED, "n_h=%d not in [1,4]", n_h);
  if ((int64_t)B * H >= (int64_t(1) << 31))
    return fail(DELTA_ERR_UNSUPPORTED, "B*H=%lld too large", (long long)B * H);
  const int64_t BH = (int64_t)B * H, L = (int64_t)T * n_h, esz = dtype == DELTA_BF16 ? 2 : 4;
  if (BH == 0) return DELTA_OK;
  if (T > 0 && (!q || !k || !v || !beta || !dout || !dq || !dk || !dv || !dbeta))
    return fail(DELTA_ERR_INVALID, "q, k, v, beta, dout, dq, dk, dv and dbeta must be non-NULL");
  if (T > 0 && g && !dg) return fail(DELTA_ERR_INVALID, "dg must be non-NULL when g is given");
  const void *ptrs[] = {q, k, v, beta, g, h0, dout, dhT, dq, dk, dv, dbeta, dg, dh0};
  for (const void *p : ptrs)
    if (!aligned16(p)) return fail(DELTA_ERR_ALIGN, "every pointer must be 16-byte aligned");
  const int64_t DD = (int64_t)dk_ * dv_;
  const Range ins[] = {range(q, BH * T * dk_ * esz), range(k, BH * L * dk_ * esz),
                       range(v, BH * L * dv_ * esz), range(beta, BH * L * 4),
                       range(g, g ? BH * T * 4 : 0), range(h0, h0 ? BH * DD * 4 : 0),
                       range(dout, BH * T * dv_ * esz), range(dhT, dhT ? BH * DD * 4 : 0)};
  const Range outs[] = {range(dq, BH * T * dk_ * 4), range(dk, BH * L * dk_ * 4),
                        range(dv, BH * L * dv_ * 4), range(dbeta, BH * L * 4),
                        range(g ? dg : nullptr, BH * T * 4), range(dh0, dh0 ? BH * DD * 4 : 0)};
  for (int i = 0; i < 6; ++i) {
    for (const Range &r : ins)
      if (overlap(outs[i], r)) return fail(DELTA_ERR_INVALID, "an output overlaps an input");
    for (int j = i + 1; j < 6; ++j)
      if (overlap(outs[i], outs[j])) return fail(DELTA_ERR_INVALID, "two outputs overlap");
  }
  if (take_injection()) return fail(DELTA_ERR_CUDA, "injected failure (delta_inject_failure)");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {
    // no step: dh0 = dhT
    if (!dh0) return DELTA_OK;
    const cudaError_t e = dhT ? cudaMemcpyAsync(dh0, dhT, (size_t)(BH * DD * 4), cudaMemcpyDeviceToDevice, s)
                              : cudaMemsetAsync(dh0, 0, (size_t)(BH * DD * 4), s);
    return e == cudaSuccess ? DELTA_OK : cuda_fail(e, "dh0 copy");
  }
  delta::BwdArgs a;
  a.q = q; a.k = k; a.v = v; a.dout = dout;
  a.beta = beta; a.g = g; a.h0 = h0; a.dhT = dhT;
  a.gq = dq; a.gk = dk; a.gv = dv; a.gbeta = dbeta; a.gg = g ? dg : nullptr; a.gh0 = dh0;
  a.B = B; a.H = H; a.T = T; a.dk = dk_; a.dv = dv_; a.n_h = n_h;
  a.bf16 = dtype == DELTA_BF16;
  if (delta::bwd_ctas(a) > INT32_MAX)
    return fail(DELTA_ERR_UNSUPPORTED, "B*H=%lld too large for the backward grid", (long long)BH);
  int64_t second = 0, third = 0;
  const int64_t first = delta::bwd_scratch_floats(a, &second, &third);
  cudaMemPool_t pool;
  cudaError_t err = scratch_pool(&pool);
  if (err != cudaSuccess) return cuda_fail(err, "scratch pool");
  void *scr = nullptr;
  err = cudaMallocFromPoolAsync(&scr, (size_t)((first + second + third) * 4), pool, s);
  if (err != cudaSuccess) return cuda_fail(err, "scratch allocation");
  a.scratch = static_cast<float *>(scr);
  a.scratch2 = a.scratch + first;
  a.scratch3 = a.scratch2 + second;
  err = delta::launch_bwd(a, s);
  const cudaError_t ef = cudaFreeAsync(scr, s);
  if (err != cudaSuccess) return cuda_fail(err, "backward kernel launch");
  return ef == cudaSuccess ? DELTA_OK : cuda_fail(ef, "scratch release");
}

int delta_prologue(const void *q_raw, const void *k_raw, const float *beta_raw, void *q_out,
                   void *k_out, float *beta_out, int B, int H, int T, int dk, int n_h,
                   delta_dtype dtype, delta_beta_map beta_map, struct CUstream_st *stream) {
  const int st = validate_prologue(q_raw, k_raw, beta_raw, q_out, k_out, beta_out, B, H, T, dk,
                                   n_h, dtype, beta_map);
  if (st != DELTA_OK || (int64_t)B * H * T == 0) return st;
  if (take_injection()) return fail(DELTA_ERR_CUDA, "injected failure (delta_inject_failure)");
  const delta::PrologueArgs p = prologue_args(q_raw, k_raw, beta_raw, q_out, k_out, beta_out,
                                              (int64_t)B * H, T, dk, n_h, dtype == DELTA_BF16,
                                              beta_map);
  const cudaError_t err = delta::launch_prologue(p, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? DELTA_OK : cuda_fail(err, "prologue kernel launch");
}

int delta_fwd_static_scratch(const void *q, const void *k, const void *v, const float *beta,
                             const float *g, const float *h0, void *out, float *hT, int B,
                             int H, int T, int dk, int dv, int n_h, int chunk,
                             delta_dtype dtype, struct CUstream_st *stream) {
  delta::FwdArgs a;
  const int st = validate_fwd(q, k, v, beta, g, h0, out, hT, B, H, T, dk, dv, n_h, chunk, dtype, a);
  if (st != DELTA_OK || a.B * a.H == 0) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (T == 0) {
    err = delta::launch_state_passthrough(a, s);
    return err == cudaSuccess ? DELTA_OK : cuda_fail(err, "state passthrough launch");
  }
  if (!delta::chunk_tc_supports(a))
    return fail(DELTA_ERR_UNSUPPORTED,
                "the static-scratch forward runs for bf16 with dk = dv = 128 and chunk = 64 only");
  const int64_t need = delta::ut_workspace_bytes(a);
  if (need > kStaticScratchBytes)
    return fail(DELTA_ERR_UNSUPPORTED,
                "the T tiles of B*H*ceil(n_h*T/64) = %lld chunks need %lld bytes; the static "
                "scratch holds %lld bytes (4096 chunks)",
                (long long)(need / 8192), (long long)need, (long long)kStaticScratchBytes);
  void *t_mat = nullptr;
  if ((err = static_scratch(&t_mat)) != cudaSuccess) return cuda_fail(err, "static scratch address");
  err = delta::launch_ut(a, t_mat, s);
  if (err != cudaSuccess) return cuda_fail(err, "UT-pass kernel launch");
  err = delta::launch_chunk_tc(a, t_mat, s);
  return err == cudaSuccess ? DELTA_OK : cuda_fail(err, "tensor-core chunk kernel launch");
}

int delta_ut_transform(const void *k, const float *beta, const float *g, void *t_mat, int B,
                       int H, int T, int dk, int n_h, int chunk, delta_dtype dtype,
                       struct CUstream_st *stream) {
  if (B < 0 || H < 0 || T < 0)
    return fail(DELTA_ERR_INVALID, "negative size B=%d H=%d T=%d", B, H, T);
  if (dtype != DELTA_F32 && dtype != DELTA_BF16)
    return fail(DELTA_ERR_INVALID, "unknown dtype %d", (int)dtype);
  if (n_h < 1 || n_h > 4) return fail(DELTA_ERR_UNSUPPORTED, "n_h=%d not in [1,4]", n_h);
  if ((int64_t)B * H >= (int64_t(1) << 31))
    return fail(DELTA_ERR_UNSUPPORTED, "B*H=%lld too large", (long long)B * H);
  delta::FwdArgs a{};
  a.k = k; a.beta = beta; a.g = g;
  a.B = B; a.H = H; a.T = T; a.L = (int64_t)T * n_h;
  a.dk = dk; a.dv = dk; a.n_h = n_h; a.chunk = chunk;
  a.bf16 = dtype == DELTA_BF16;
  if (a.B * a.H == 0 || T == 0) return DELTA_OK;
  if (!delta::ut_supports(a))
    return fail(DELTA_ERR_UNSUPPORTED,
                "the UT pass runs for bf16 keys with dk = 128 and chunk = 64 only");
  if (!k || !beta) return fail(DELTA_ERR_INVALID, "k and beta must be non-NULL");
  if (!aligned16(k) || !aligned16(beta) || !aligned16(g))
    return fail(DELTA_ERR_ALIGN, "every pointer must be 16-byte aligned");
  int st;
  if ((st = validate_t_mat(a, t_mat, false)) != DELTA_OK) return st;
  if (take_injection()) return fail(DELTA_ERR_CUDA, "injected failure (delta_inject_failure)");
  const cudaError_t err = delta::launch_ut(a, t_mat, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? DELTA_OK : cuda_fail(err, "UT-pass kernel launch");
}

int delta_fwd_with_ut(const void *q, const void *k, const void *v, const float *beta,
                      const float *g, const float *h0, const void *t_mat, void *out, float *hT,
                      int B, int H, int T, int dk, int dv, int n_h, int chunk, delta_dtype dtype,
                      struct CUstream_st *stream) {
  delta::FwdArgs a;
  int st = validate_fwd(q, k, v, beta, g, h0, out, hT, B, H, T, dk, dv, n_h, chunk, dtype, a);
  if (st != DELTA_OK || a.B * a.H == 0 || T == 0) return st;
  if (!delta::chunk_tc_supports(a))
    return fail(DELTA_ERR_UNSUPPORTED,
                "the state pass runs for bf16 with dk = dv = 128 and chunk = 64 only");
  if ((st = validate_t_mat(a, t_mat, true)) != DELTA_OK) return st;
  if (take_injection()) return fail(DELTA_ERR_CUDA, "injected failure (delta_inject_failure)");
  const cudaError_t err = delta::launch_chunk_tc(a, t_mat, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? DELTA_OK : cuda_fail(err, "tensor-core chunk kernel launch");
}

int delta_state_erank(const float *state, float *erank, int B, int H, int dk, int dv,
                      struct CUstream_st *stream) {
  if (B < 0 || H < 0) return fail(DELTA_ERR_INVALID, "negative size B=%d H=%d", B, H);
  if (!supported_dim(dk) || !supported_dim(dv))
    return fail(DELTA_ERR_UNSUPPORTED, "dk=%d dv=%d not in {16,32,64,128}", dk, dv);
  if ((int64_t)B * H >= (int64_t(1) << 31))
    return fail(DELTA_ERR_UNSUPPORTED, "B*H=%lld too large", (long long)B * H);
  const int64_t BH = (int64_t)B * H;
  if (BH == 0) return DELTA_OK;
  if (!state || !erank) return fail(DELTA_ERR_INVALID, "state and erank must be non-NULL");
  if (!aligned16(state) || !aligned16(erank))
    return fail(DELTA_ERR_ALIGN, "every pointer must be 16-byte aligned");
  if (overlap(range(state, BH * dk * dv * 4), range(erank, BH * 4)))
    return fail(DELTA_ERR_INVALID, "erank overlaps state");
  if (take_injection()) return fail(DELTA_ERR_CUDA, "injected failure (delta_inject_failure)");
  const cudaError_t err = delta::launch_erank(state, erank, BH, dk, dv, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? DELTA_OK : cuda_fail(err, "effective-rank kernel launch");
}

int delta_attention_map(const void *q, const void *k, const float *beta, const float *g,
                        float *attn, int B, int H, int N, int dk, delta_dtype dtype,
                        struct CUstream_st *stream) {
  if (B < 0 || H < 0 || N < 0) return fail(DELTA_ERR_INVALID, "negative size B=%d H=%d N=%d", B, H, N);
  if (dtype != DELTA_F32 && dtype != DELTA_BF16)
    return fail(DELTA_ERR_INVALID, "unknown dtype %d", (int)dtype);
  if (!supported_dim(dk)) return fail(DELTA_ERR_UNSUPPORTED, "dk=%d not in {16,32,64,128}", dk);
  if (N > 64) return fail(DELTA_ERR_UNSUPPORTED, "N=%d: the attention map is built for N <= 64", N);
  if ((int64_t)B * H >= (int64_t(1) << 31))
    return fail(DELTA_ERR_UNSUPPORTED, "B*H=%lld too large", (long long)B * H);
  const int64_t BH = (int64_t)B * H;
  if (BH == 0 || N == 0) return DELTA_OK;
  if (!q || !k || !beta || !attn) return fail(DELTA_ERR_INVALID, "q, k, beta and attn must be non-NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(beta) || !aligned16(g) || !aligned16(attn))
    return fail(DELTA_ERR_ALIGN, "every pointer must be 16-byte aligned");
  const int64_t esz = dtype == DELTA_BF16 ? 2 : 4;
  const Range r_a = range(attn, BH * N * N * 4);
  const Range inputs[] = {range(q, BH * N * dk * esz), range(k, BH * N * dk * esz),
                          range(beta, BH * N * 4), range(g, g ? BH * N * 4 : 0)};
  for (const Range &r : inputs)
    if (overlap(r_a, r)) return fail(DELTA_ERR_INVALID, "attn overlaps an input");
  if (take_injection()) return fail(DELTA_ERR_CUDA, "injected failure (delta_inject_failure)");
  const cudaError_t err = delta::launch_attention_map(q, k, beta, g, attn, B, H, N, dk,
                                                     dtype == DELTA_BF16,
                                                     reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? DELTA_OK : cuda_fail(err, "attention-map kernel launch");
}

int delta_fwd_kernel_count(int B, int H, int T, int dk, int dv, int n_h, int chunk,
                           delta_dtype dtype) {
  if (B < 0 || H < 0 || T < 0 || (dtype != DELTA_F32 && dtype != DELTA_BF16) ||
      !supported_dim(dk) || !supported_dim(dv) || !supported_chunk(chunk) || n_h < 1 ||
      n_h > 4 || (int64_t)B * H >= (int64_t(1) << 31))
    return -1;
  if ((int64_t)B * H == 0) return 0;
  delta::FwdArgs a{};
  a.B = B; a.H = H; a.T = T; a.L = (int64_t)T * n_h;
  a.dk = dk; a.dv = dv; a.n_h = n_h; a.chunk = chunk;
  a.bf16 = dtype == DELTA_BF16;
  if (T == 0) return 1;
  return delta::chunk_tc_supports(a) ? delta::kChunkTcKernels : 1;
}

int delta_step(const void *q, const void *k, const void *v, const float *beta,
               const float *g, float *state, void *out, int B, int H, int dk, int dv,
               int n_h, delta_dtype dtype, struct CUstream_st *stream) {
  return run_step(q, k, v, beta, g, state, out, B, H, dk, dv, n_h, dtype, -1, stream);
}

int delta_step_kda(const void *q, const void *k, const void *v, const float *beta,
                   const float *alpha, float *state, void *out, int B, int H, int dk, int dv,
                   int n_h, delta_dtype dtype, struct CUstream_st *stream) {
  return run_step(q, k, v, beta, nullptr, state, out, B, H, dk, dv, n_h, dtype, -1, stream, alpha,
                  true);
}

int delta_step_prologue(const void *q_raw, const void *k_raw, const void *v, const float *beta_raw,
                        const float *g, float *state, void *out, int B, int H, int dk, int dv,
                        int n_h, delta_dtype dtype, delta_beta_map beta_map,
                        struct CUstream_st *stream) {
  if (beta_map != DELTA_BETA_SIGMOID && beta_map != DELTA_BETA_2SIGMOID)
    return fail(DELTA_ERR_INVALID, "unknown beta_map %d", (int)beta_map);
  return run_step(q_raw, k_raw, v, beta_raw, g, state, out, B, H, dk, dv, n_h, dtype,
                  beta_map == DELTA_BETA_2SIGMOID ? 1 : 0, stream);
}

}  // extern "C"
