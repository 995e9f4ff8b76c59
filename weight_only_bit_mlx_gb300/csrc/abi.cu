// abi.cu - the extern "C" entry points of libqlinear.so: argument checks, launch
// geometry and the small auxiliary kernels (SwiGLU control, wait probe, status word).
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/qlinear.h"
#include "common.cuh"
#include "pgemm.cuh"
#include "qmv.cuh"
#include "sync.cuh"

namespace qlk {

// Device status word (one per device that loads the library).  Kernels receive its
// address as a parameter; qlinear_last_error() reads and clears it.
__device__ int g_status_word = 0;

static std::atomic<uint64_t> g_wait_budget_ns{2000000000ull};

uint64_t wait_budget_ns() { return g_wait_budget_ns.load(std::memory_order_relaxed); }

constexpr int kMaxDevices = 64;
static std::mutex g_dev_mu;
static int g_dev_state[kMaxDevices];     // 0 unknown, 1 ok, -1 wrong arch
static int *g_dev_status[kMaxDevices];   // device address of g_status_word

// Checks that the current device is sm_103 and returns the status-word address.
int device_setup(int **status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QL_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_dev_state[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return QL_ERR_CUDA;
    if (major != 10 || minor != 3) {
      g_dev_state[dev] = -1;
    } else {
      void *p = nullptr;
      if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return QL_ERR_CUDA;
      g_dev_status[dev] = static_cast<int *>(p);
      g_dev_state[dev] = 1;
    }
  }
  if (g_dev_state[dev] < 0) return QL_ERR_ARCH;
  if (status) *status = g_dev_status[dev];
  return QL_OK;
}

static bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_weight(const ql_weight *w) {
  if (w == nullptr || w->wq == nullptr || w->scales == nullptr || w->biases == nullptr) return QL_ERR_NULL;
  if (w->group != 64) return QL_ERR_GROUP;
  if (w->bits != 4 && w->bits != 6 && w->bits != 8) return QL_ERR_BITS;
  if (w->n <= 0 || w->k <= 0 || (w->k % 64) != 0 || w->k > 65536) return QL_ERR_SHAPE;
  if (!aligned(w->wq, 16) || !aligned(w->scales, 2) || !aligned(w->biases, 2)) return QL_ERR_ALIGN;
  return QL_OK;
}

static int check_x(const uint16_t *x, int32_t rows, int64_t ldx, int32_t k) {
  if (x == nullptr) return QL_ERR_NULL;
  if (rows < 1 || rows > 16) return QL_ERR_ROWS;
  if (!aligned(x, 16) || (ldx % 8) != 0 || (rows > 1 && ldx < k)) return QL_ERR_ALIGN;
  return QL_OK;
}

static int launch_status(cudaError_t e) {
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return QL_ERR_LAUNCH;
  }
  return QL_OK;
}

static MvMat make_mat(const ql_weight *w, void *out, int64_t ldo) {
  MvMat m;
  m.wq = w->wq;
  m.s = w->scales;
  m.b = w->biases;
  m.out = out;
  m.ldo = ldo;
  m.n = w->n;
  return m;
}

// ---------------------------------------------------------------------------------
// SwiGLU on its own (the "fusion off" control of the fused FFN step)
// ---------------------------------------------------------------------------------
__global__ void swiglu_kernel(const float *a, const float *c, int rows, int n, int64_t lda, uint16_t *h,
                              int64_t ldh) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // as in swiglu_vec4_kernel
  const int64_t total = (int64_t)rows * n;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / n, j = i % n;
    h[r * ldh + j] = swiglu_bf16(a[r * lda + j], c[r * lda + j]);
  }
}

// Contiguous rows and 16-byte aligned data: four elements per thread step.
__global__ void swiglu_vec4_kernel(const float4 *a, const float4 *c, int64_t n4, uint2 *h) {
  // a kernel launched after this one with programmatic dependent launch (the next prompt
  // GEMM call's code conversion, which reads only its weights) may start now; every
  // library kernel waits for this one before it reads what this one writes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
    const float4 av = a[i], cv = c[i];
    const uint32_t h0 = swiglu_bf16(av.x, cv.x), h1 = swiglu_bf16(av.y, cv.y);
    const uint32_t h2 = swiglu_bf16(av.z, cv.z), h3 = swiglu_bf16(av.w, cv.w);
    h[i] = make_uint2(h0 | (h1 << 16), h2 | (h3 << 16));
  }
}

// One thread waits on a barrier nothing will ever complete; the bounded wait gives
// up after budget_ns and records QL_ERR_TIMEOUT.
__global__ void wait_probe_kernel(int *status, uint64_t budget_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait_bounded(&bar, 0u, budget_ns, nullptr)) record_status(status, kErrTimeout);
  }
}

}  // namespace qlk

using namespace qlk;

extern "C" {

int qlinear_mv_rows(const ql_weight *w, const uint16_t *x, int32_t rows, int64_t ldx, float *y, int64_t ldy,
                    void *stream) {
  int e = check_weight(w);
  if (e) return e;
  if ((e = check_x(x, rows, ldx, w->k))) return e;
  if (y == nullptr) return QL_ERR_NULL;
  if (rows > 1 && ldy < w->n) return QL_ERR_ALIGN;
  int *status = nullptr;
  if ((e = device_setup(&status))) return e;
  MvParams p;
  std::memset(&p, 0, sizeof(p));
  (void)status;  // the decode kernels have no device-side waits to report
  p.m[0] = make_mat(w, y, ldy);
  p.x = x;
  p.ldx = ldx;
  p.rows = rows;
  p.k = w->k;
  const int tiles = (w->n + 15) / 16;
  return launch_status(launch_mv(p, kMvPlain, w->bits, tiles, static_cast<cudaStream_t>(stream)));
}

int qlinear_mv_resid_norm(const ql_weight *w, const uint16_t *x, int32_t rows, int64_t ldx, uint16_t *resid,
                          int64_t ldr, const uint16_t *gamma, float eps, uint16_t *out, int64_t ldo, void *stream) {
  int e = check_weight(w);
  if (e) return e;
  if ((e = check_x(x, rows, ldx, w->k))) return e;
  if (resid == nullptr || gamma == nullptr || out == nullptr) return QL_ERR_NULL;
  if (!(eps >= 0.0f)) return QL_ERR_SHAPE;
  if ((w->n + 15) / 16 > kMvResidMaxTiles) return QL_ERR_SHAPE;
  if ((rows > 1 && (ldr < w->n || ldo < w->n)) || !aligned(resid, 2) || !aligned(out, 2) || !aligned(gamma, 2))
    return QL_ERR_ALIGN;
  int *status = nullptr;
  if ((e = device_setup(&status))) return e;
  MvParams p;
  std::memset(&p, 0, sizeof(p));
  if (mv_resid_scratch(&p.part, &p.counter)) return QL_ERR_CUDA;
  (void)status;  // the decode kernels have no device-side waits to report
  p.m[0] = make_mat(w, nullptr, 0);
  p.x = x;
  p.ldx = ldx;
  p.rows = rows;
  p.k = w->k;
  p.resid = resid;
  p.ldr = ldr;
  p.gamma = gamma;
  p.eps = eps;
  p.nout = out;
  p.ldn = ldo;
  const int tiles = (w->n + 15) / 16;
  p.ntiles = tiles;
  return launch_status(launch_mv(p, kMvResid, w->bits, tiles, static_cast<cudaStream_t>(stream)));
}

int qlinear_mv(const ql_weight *w, const uint16_t *x, float *y, void *stream) {
  return qlinear_mv_rows(w, x, 1, w ? w->k : 0, y, w ? w->n : 0, stream);
}

int qffn_swiglu_mv(const ql_weight *w1, const ql_weight *w3, const uint16_t *x, int32_t rows, int64_t ldx,
                   uint16_t *h, int64_t ldh, void *stream) {
  int e = check_weight(w1);
  if (e) return e;
  if ((e = check_weight(w3))) return e;
  if (w1->bits != w3->bits) return QL_ERR_BITS;
  if (w1->n != w3->n || w1->k != w3->k) return QL_ERR_SHAPE;
  if ((e = check_x(x, rows, ldx, w1->k))) return e;
  if (h == nullptr) return QL_ERR_NULL;
  if (rows > 1 && ldh < w1->n) return QL_ERR_ALIGN;
  int *status = nullptr;
  if ((e = device_setup(&status))) return e;
  MvParams p;
  std::memset(&p, 0, sizeof(p));
  (void)status;  // the decode kernels have no device-side waits to report
  p.m[0] = make_mat(w1, h, ldh);
  p.m[1] = make_mat(w3, h, ldh);
  p.x = x;
  p.ldx = ldx;
  p.rows = rows;
  p.k = w1->k;
  const int tiles = (w1->n + 15) / 16;
  return launch_status(launch_mv(p, kMvFfn, w1->bits, tiles, static_cast<cudaStream_t>(stream)));
}

int qattn_proj_mv(const ql_weight *wq, const ql_weight *wk, const ql_weight *wv, const ql_weight *wg,
                  const uint16_t *x, int32_t rows, int64_t ldx, float *q, float *k, float *v, float *g,
                  void *stream) {
  const ql_weight *ws[4] = {wq, wk, wv, wg};
  float *outs[4] = {q, k, v, g};
  int e;
  for (int i = 0; i < 4; ++i) {
    if ((e = check_weight(ws[i]))) return e;
    if (outs[i] == nullptr) return QL_ERR_NULL;
    if (ws[i]->bits != wq->bits) return QL_ERR_BITS;
    if (ws[i]->k != wq->k) return QL_ERR_SHAPE;
  }
  if ((e = check_x(x, rows, ldx, wq->k))) return e;
  int *status = nullptr;
  if ((e = device_setup(&status))) return e;
  MvParams p;
  std::memset(&p, 0, sizeof(p));
  (void)status;  // the decode kernels have no device-side waits to report
  int tiles = 0;
  for (int i = 0; i < 4; ++i) {
    p.m[i] = make_mat(ws[i], outs[i], ws[i]->n);
    tiles += (ws[i]->n + 15) / 16;
    p.tile_end[i] = tiles;
  }
  p.x = x;
  p.ldx = ldx;
  p.rows = rows;
  p.k = wq->k;
  return launch_status(launch_mv(p, kMvAttn, wq->bits, tiles, static_cast<cudaStream_t>(stream)));
}

int qlinear_pgemm(const ql_weight *w, const uint16_t *X, int32_t m, int64_t ldx, float *Y, int64_t ldy,
                  void *stream) {
  int e = check_weight(w);
  if (e) return e;
  if (m < 0) return QL_ERR_SHAPE;
  if (m == 0) return QL_OK;  // an empty window: nothing to read or write (pointers may be NULL)
  if (X == nullptr || Y == nullptr) return QL_ERR_NULL;
  if (!aligned(X, 16) || (ldx % 8) != 0 || ldx < w->k || ldy < w->n || !aligned(Y, 4)) return QL_ERR_ALIGN;
  int *status = nullptr;
  if ((e = device_setup(&status))) return e;
  return pgemm_run(w, X, m, ldx, Y, ldy, static_cast<cudaStream_t>(stream), status);
}

constexpr int kPgemmMultiMax = 16;  // weights of one qlinear_pgemm_multi call

// Each weight checked as qlinear_pgemm checks it, every k equal; then one row-sum
// pre-pass and the weights' GEMMs in turn.
int qlinear_pgemm_multi(const ql_weight *const *w, int32_t nw, const uint16_t *X, int32_t m, int64_t ldx,
                        float *const *Y, const int64_t *ldy, void *stream) {
  if (w == nullptr || Y == nullptr || ldy == nullptr) return QL_ERR_NULL;
  if (nw < 1 || nw > kPgemmMultiMax) return QL_ERR_SHAPE;
  int e = QL_OK;
  for (int i = 0; i < nw; ++i) {
    if ((e = check_weight(w[i]))) return e;
    if (w[i]->k != w[0]->k) return QL_ERR_SHAPE;
  }
  if (m < 0) return QL_ERR_SHAPE;
  if (m == 0) return QL_OK;  // an empty window: nothing to read or write
  if (X == nullptr) return QL_ERR_NULL;
  if (!aligned(X, 16) || (ldx % 8) != 0 || ldx < w[0]->k) return QL_ERR_ALIGN;
  for (int i = 0; i < nw; ++i) {
    if (Y[i] == nullptr) return QL_ERR_NULL;
    if (ldy[i] < w[i]->n || !aligned(Y[i], 4)) return QL_ERR_ALIGN;
  }
  int *status = nullptr;
  if ((e = device_setup(&status))) return e;
  return pgemm_run_multi(w, nw, X, m, ldx, Y, ldy, static_cast<cudaStream_t>(stream), status);
}

// Same checks as qlinear_pgemm, then the fixed-scratch variant (allocates nothing).
int qlinear_pgemm_noalloc(const ql_weight *w, const uint16_t *X, int32_t m, int64_t ldx, float *Y, int64_t ldy,
                          void *stream) {
  int e = check_weight(w);
  if (e) return e;
  if (m < 0) return QL_ERR_SHAPE;
  if (m == 0) return QL_OK;
  if (X == nullptr || Y == nullptr) return QL_ERR_NULL;
  if (!aligned(X, 16) || (ldx % 8) != 0 || ldx < w->k || ldy < w->n || !aligned(Y, 4)) return QL_ERR_ALIGN;
  const int64_t lds = ((3 * (int64_t)(w->k / 64) + 63) / 64) * 64;
  if ((int64_t)m * lds > pgemm_noalloc_max_elems()) return QL_ERR_TOO_LARGE;
  int *status = nullptr;
  if ((e = device_setup(&status))) return e;
  return pgemm_run_noalloc(w, X, m, ldx, Y, ldy, static_cast<cudaStream_t>(stream), status);
}

// The prompt GEMM of the FFN's up projection with the SwiGLU as its epilogue.
int qlinear_pgemm_swiglu(const ql_weight *w3, const uint16_t *X, int32_t m, int64_t ldx, const float *A, int64_t lda,
                         uint16_t *H, int64_t ldh, void *stream) {
  int e = check_weight(w3);
  if (e) return e;
  if (m < 0) return QL_ERR_SHAPE;
  if (m == 0) return QL_OK;
  if (X == nullptr || A == nullptr || H == nullptr) return QL_ERR_NULL;
  if (!aligned(X, 16) || (ldx % 8) != 0 || ldx < w3->k || lda < w3->n || ldh < w3->n || !aligned(A, 4) ||
      !aligned(H, 2))
    return QL_ERR_ALIGN;
  int *status = nullptr;
  if ((e = device_setup(&status))) return e;
  PgEpilogue epi = {kPgSwiglu, A, lda, H, ldh};
  return pgemm_run(w3, X, m, ldx, nullptr, 0, static_cast<cudaStream_t>(stream), status, &epi);
}

// The prompt GEMM of w2 / o with the post-add as its epilogue, then the next-norm.
int qlinear_pgemm_resid_norm(const ql_weight *w, const uint16_t *X, int32_t m, int64_t ldx, uint16_t *resid,
                             int64_t ldr, const uint16_t *gamma, float eps, uint16_t *out, int64_t ldo, void *stream) {
  int e = check_weight(w);
  if (e) return e;
  if (m < 0) return QL_ERR_SHAPE;
  if (m == 0) return QL_OK;
  if (X == nullptr || resid == nullptr || gamma == nullptr || out == nullptr) return QL_ERR_NULL;
  if (!(eps >= 0.0f)) return QL_ERR_SHAPE;
  if (!aligned(X, 16) || (ldx % 8) != 0 || ldx < w->k || ldr < w->n || ldo < w->n || !aligned(resid, 2) ||
      !aligned(out, 2) || !aligned(gamma, 2))
    return QL_ERR_ALIGN;
  int *status = nullptr;
  if ((e = device_setup(&status))) return e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PgEpilogue epi = {kPgResid, nullptr, 0, resid, ldr};
  if ((e = pgemm_run(w, X, m, ldx, nullptr, 0, st, status, &epi))) return e;
  return launch_status(launch_resid_rmsnorm(nullptr, 0, resid, ldr, m, w->n, gamma, eps, out, ldo, st));
}

int qswiglu(const float *a, const float *c, int32_t rows, int32_t n, int64_t lda, uint16_t *h, int64_t ldh,
            void *stream) {
  if (a == nullptr || c == nullptr || h == nullptr) return QL_ERR_NULL;
  if (rows < 1 || n < 1) return QL_ERR_SHAPE;
  if (lda < n || ldh < n) return QL_ERR_ALIGN;
  int e;
  if ((e = device_setup(nullptr))) return e;
  const int64_t total = (int64_t)rows * n;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((rows == 1 || (lda == n && ldh == n)) && total % 4 == 0 && aligned(a, 16) && aligned(c, 16) &&
      aligned(h, 8)) {
    const int64_t n4 = total / 4;
    int blocks = (int)((n4 + 255) / 256);
    if (blocks > 152 * 16) blocks = 152 * 16;
    swiglu_vec4_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4 *>(a), reinterpret_cast<const float4 *>(c),
                                               n4, reinterpret_cast<uint2 *>(h));
  } else {
    int blocks = (int)((total + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    swiglu_kernel<<<blocks, 256, 0, st>>>(a, c, rows, n, lda, h, ldh);
  }
  return launch_status(cudaGetLastError());
}

int qlinear_last_error(void *stream) {
  int *status = nullptr;
  int e = device_setup(&status);
  if (e) return e;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return QL_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return QL_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return QL_ERR_CUDA;
  // a post-add / next-norm launch that gave up may have left its tile counter part-way
  if (v != QL_OK && mv_resid_counter_reset() != 0) return QL_ERR_CUDA;
  return v;
}

uint64_t qlinear_set_wait_budget_ns(uint64_t ns) { return g_wait_budget_ns.exchange(ns); }

int qlinear_wait_probe(uint64_t budget_ns, void *stream) {
  int *status = nullptr;
  int e = device_setup(&status);
  if (e) return e;
  wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, budget_ns);
  return launch_status(cudaGetLastError());
}

const char *qlinear_strerror(int code) {
  switch (code) {
    case QL_OK: return "ok";
    case QL_ERR_NULL: return "a required pointer is NULL";
    case QL_ERR_SHAPE: return "invalid or mismatched shape (n, k, m)";
    case QL_ERR_BITS: return "bits must be 4, 6 or 8 (and equal across fused weights)";
    case QL_ERR_GROUP: return "group must be 64";
    case QL_ERR_ROWS: return "rows must be in 1..16";
    case QL_ERR_ALIGN: return "misaligned pointer or leading dimension";
    case QL_ERR_ARCH: return "the current device is not sm_103 (GB300)";
    case QL_ERR_LAUNCH: return "kernel launch failed";
    case QL_ERR_TIMEOUT: return "a bounded device-side wait gave up";
    case QL_ERR_CUDA: return "CUDA runtime error";
    case QL_ERR_NOMEM: return "could not allocate scratch memory";
    case QL_ERR_TOO_LARGE: return "m * round_up(3*k/64, 64) exceeds the 1,048,576-value fixed scratch";
    default: return "unknown qlinear status";
  }
}

int qlinear_version(void) { return (0 << 16) | 1; }

}  // extern "C"
