// qpost.cu - the decoder steps that follow the quantized projections (sm_103a):
// QK norm with partial RoPE and the KV store, and the post-add / next-norm step.
//
// TensorFold PR #1696 (later revision), "What it adds": kernels for "QK norm with
// partial RoPE", decode "fuses ... RoPE with the KV store", per-stream "KV rings";
// PR #1514 "What changes": "post-add/next-norm fusion" keeping the retained rounding
// boundaries.  The pages print no formula; the definitions used (every constant an
// argument) are:
//   QK norm:   xhat_j = x_j / sqrt(mean(x^2) + eps) * w_j, per head (q and k weights)
//   RoPE:      rotate-half on the first rot_dim dimensions of a head,
//              theta_i = pos * base^(-2i/rot_dim), i < rot_dim/2:
//              (a, b) = (x_i, x_{i+rot/2}) -> (a cos - b sin, a sin + b cos)
//   KV store:  k (normed, rotated) and v of stream r to slot pos[r] mod ring_len of
//              that stream's ring, bf16; q (normed, rotated) to q_out, bf16
//   post-add:  r' = bf16(r + y) (the stored residual), out = bf16(r' * rstd * gamma)
// One warp per head (QK norm): the sum of squares is a fixed xor-butterfly, so every
// head's result depends on that head's data only.  The angles are formed and turned
// reduced modulo 2*pi in double precision, then turned into (cos, sin) in fp32;
// everything else is fp32, rounded to bf16 once.
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/qlinear.h"
#include "common.cuh"

namespace qlk {

constexpr int kHeadWarps = 4;          // heads per CTA
constexpr int kMaxHeadDim = 256;
constexpr int kNormThreads = 256;      // post-add / next-norm: one CTA per row

__device__ __forceinline__ float warp_sum_xor(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

struct QkParams {
  const float *q, *k, *v;
  int64_t ldq, ldk, ldv;
  int rows, nq, nkv, hd, rot;
  double base;
  float eps;
  const uint16_t *qw, *kw;
  const int32_t *pos;
  uint16_t *q_out;
  int64_t ldqo;
  uint16_t *k_ring, *v_ring;
  int ring_len;
};

// The rotation angles of one position: theta_i = pos * base^(-2i/rot) formed in
// float64 (positions up to 2^31 keep ~1e-7 rad absolute accuracy), reduced to
// [-pi, pi] in float64 (2*pi as a two-part constant), then cos / sin of the remainder
// in fp32.
__device__ __forceinline__ float2 rope_cos_sin(double pos, int i, int rot, double base) {
  const double theta = pos * pow(base, -2.0 * (double)i / (double)rot);
  const double kTwoPiHi = 6.283185307179586;       // 2*pi rounded to double
  const double kTwoPiLo = 2.4492935982947064e-16;  // 2*pi - kTwoPiHi
  const double n = rint(theta * 0.15915494309189535);  // theta / (2*pi)
  const double r = fma(-n, kTwoPiLo, fma(-n, kTwoPiHi, theta));
  float sn, cs;
  sincosf((float)r, &sn, &cs);
  return make_float2(cs, sn);
}

// grid: (ceil((nq + nkv) / kHeadWarps), rows); warp = one head of q (head < nq) or k
// (head >= nq, which also stores that kv head's v).  The CTA's angle table (one row,
// one position) is built first, once per CTA.
__global__ void __launch_bounds__(kHeadWarps * 32) qk_norm_rope_kv_kernel(const __grid_constant__ QkParams p) {
  __shared__ float hbuf[kHeadWarps][kMaxHeadDim];
  __shared__ float2 cs_tab[kMaxHeadDim / 2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.x * kHeadWarps + warp;
  const int r = blockIdx.y;
  const int half = p.rot >> 1;
  // positions and norm weights are not written by a preceding kernel
  const double pos = (double)p.pos[r];
  for (int i = threadIdx.x; i < half; i += kHeadWarps * 32) cs_tab[i] = rope_cos_sin(pos, i, p.rot, p.base);
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __syncthreads();
  if (head >= p.nq + p.nkv) return;
  const bool is_q = head < p.nq;
  const int kvh = head - p.nq;
  const float *src = is_q ? p.q + (size_t)r * p.ldq + (size_t)head * p.hd : p.k + (size_t)r * p.ldk + (size_t)kvh * p.hd;
  const uint16_t *w = is_q ? p.qw : p.kw;
  const int per = p.hd >> 5;  // values per lane (head_dim % 32 == 0)
  float x[kMaxHeadDim / 32];
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxHeadDim / 32; ++i) {
    if (i < per) {
      x[i] = src[lane + 32 * i];
      ss = __fmaf_rn(x[i], x[i], ss);
    }
  }
  ss = warp_sum_xor(ss);
  const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)p.hd), p.eps)));
#pragma unroll
  for (int i = 0; i < kMaxHeadDim / 32; ++i)
    if (i < per) hbuf[warp][lane + 32 * i] = __fmul_rn(__fmul_rn(x[i], rstd), bf16_to_f32(ldg_u16(w + lane + 32 * i)));
  __syncwarp();
  uint16_t *dst;
  if (is_q) {
    dst = p.q_out + (size_t)r * p.ldqo + (size_t)head * p.hd;
  } else {
    int slot = p.pos[r] % p.ring_len;
    if (slot < 0) slot += p.ring_len;
    const size_t off = ((size_t)r * p.ring_len + slot) * ((size_t)p.nkv * p.hd) + (size_t)kvh * p.hd;
    dst = p.k_ring + off;
    // v of this kv head, rounded to bf16, into the same slot
    const float *vs = p.v + (size_t)r * p.ldv + (size_t)kvh * p.hd;
    for (int j = lane; j < p.hd; j += 32) p.v_ring[off + j] = f32_to_bf16_rn(vs[j]);
  }
  for (int j = lane; j < p.hd; j += 32) {
    float out;
    if (j < p.rot) {
      const int i = j < half ? j : j - half;
      const float c = cs_tab[i].x, s = cs_tab[i].y;
      const float a = hbuf[warp][i], b = hbuf[warp][i + half];
      out = j < half ? __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, s)) : __fadd_rn(__fmul_rn(a, s), __fmul_rn(b, c));
    } else {
      out = hbuf[warp][j];
    }
    dst[j] = f32_to_bf16_rn(out);
  }
}

// post-add / next-norm: one CTA per row; the sum of squares is reduced in a fixed order
// (per-thread sums over its elements in order, then a tree over the warps'
// xor-butterfly results in warp order).  Vector form (16-byte rows and n % 8 == 0):
// each thread owns chunks of 8 consecutive elements, c = tid + 256 k; the first
// kVecKeep chunks of the stored residual stay in registers for the second pass.
constexpr int kVecKeep = 4;

__device__ __forceinline__ float block_sum_fixed(float ss, float *wsum) {
  ss = warp_sum_xor(ss);
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = wsum[0];
  for (int i = 1; i < kNormThreads / 32; ++i) tot = __fadd_rn(tot, wsum[i]);
  return tot;
}

// kAdd: r' = bf16(r + y) is stored first; otherwise r' is the stored residual as it is
// (the post-add already done by the producing GEMM's epilogue) and y is not read.
template <bool kAdd>
__global__ void __launch_bounds__(kNormThreads) resid_rmsnorm_vec_kernel(const float *y, int64_t ldy, uint16_t *resid,
                                                                       int64_t ldr, int n, const uint16_t *gamma,
                                                                       float eps, uint16_t *out, int64_t ldo) {
  __shared__ float wsum[kNormThreads / 32];
  const int r = blockIdx.x;
  const int nch = n >> 3;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float *yr = y + (size_t)r * ldy;
  uint16_t *rr = resid + (size_t)r * ldr;
  // chunk c of this row: r' = bf16(r + y), stored; returns the packed r' and adds its
  // squares to ss in element order
  auto add_chunk = [&](int c, float &ss) -> uint4 {
    const uint4 rv = *reinterpret_cast<const uint4 *>(rr + 8 * c);
    const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
    float yv[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    if constexpr (kAdd) {
      const float4 y0 = *reinterpret_cast<const float4 *>(yr + 8 * c);
      const float4 y1 = *reinterpret_cast<const float4 *>(yr + 8 * c + 4);
      yv[0] = y0.x; yv[1] = y0.y; yv[2] = y0.z; yv[3] = y0.w;
      yv[4] = y1.x; yv[5] = y1.y; yv[6] = y1.z; yv[7] = y1.w;
    }
    uint32_t nw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint16_t lo = (uint16_t)(rw[e] & 0xFFFFu), hi = (uint16_t)(rw[e] >> 16);
      if constexpr (kAdd) {
        lo = f32_to_bf16_rn(__fadd_rn(bf16_to_f32(lo), yv[2 * e]));
        hi = f32_to_bf16_rn(__fadd_rn(bf16_to_f32(hi), yv[2 * e + 1]));
      }
      const float vl = bf16_to_f32(lo), vh = bf16_to_f32(hi);
      ss = __fmaf_rn(vl, vl, ss);
      ss = __fmaf_rn(vh, vh, ss);
      nw[e] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    const uint4 nv = make_uint4(nw[0], nw[1], nw[2], nw[3]);
    if constexpr (kAdd) *reinterpret_cast<uint4 *>(rr + 8 * c) = nv;
    return nv;
  };
  uint4 keep[kVecKeep];
  float ss = 0.0f;
#pragma unroll
  for (int k = 0; k < kVecKeep; ++k) {
    const int c = threadIdx.x + k * kNormThreads;
    if (c < nch) keep[k] = add_chunk(c, ss);
  }
  for (int c = threadIdx.x + kVecKeep * kNormThreads; c < nch; c += kNormThreads) (void)add_chunk(c, ss);
  const float tot = block_sum_fixed(ss, wsum);
  const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)n), eps)));
  uint16_t *orow = out + (size_t)r * ldo;
  auto norm_chunk = [&](int c, const uint4 &nv) {
    const uint4 gv = *reinterpret_cast<const uint4 *>(gamma + 8 * c);
    const uint32_t nw[4] = {nv.x, nv.y, nv.z, nv.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t ow[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint16_t lo = f32_to_bf16_rn(__fmul_rn(__fmul_rn(bf16_to_f32(nw[e] & 0xFFFFu), rstd),
                                                   bf16_to_f32(gw[e] & 0xFFFFu)));
      const uint16_t hi = f32_to_bf16_rn(__fmul_rn(__fmul_rn(bf16_to_f32(nw[e] >> 16), rstd), bf16_to_f32(gw[e] >> 16)));
      ow[e] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    *reinterpret_cast<uint4 *>(orow + 8 * c) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
  };
#pragma unroll
  for (int k = 0; k < kVecKeep; ++k) {
    const int c = threadIdx.x + k * kNormThreads;
    if (c < nch) norm_chunk(c, keep[k]);
  }
  for (int c = threadIdx.x + kVecKeep * kNormThreads; c < nch; c += kNormThreads)
    norm_chunk(c, *reinterpret_cast<const uint4 *>(rr + 8 * c));
}

// Scalar form (any n, strides and alignment): the same arithmetic one element at a time.
template <bool kAdd>
__global__ void __launch_bounds__(kNormThreads) resid_rmsnorm_kernel(const float *y, int64_t ldy, uint16_t *resid,
                                                                   int64_t ldr, int n, const uint16_t *gamma, float eps,
                                                                   uint16_t *out, int64_t ldo) {
  __shared__ float wsum[kNormThreads / 32];
  const int r = blockIdx.x;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float *yr = y + (size_t)r * ldy;
  uint16_t *rr = resid + (size_t)r * ldr;
  float ss = 0.0f;
  for (int j = threadIdx.x; j < n; j += kNormThreads) {
    uint16_t nb = rr[j];
    if constexpr (kAdd) {
      nb = f32_to_bf16_rn(__fadd_rn(bf16_to_f32(nb), yr[j]));
      rr[j] = nb;
    }
    const float v = bf16_to_f32(nb);
    ss = __fmaf_rn(v, v, ss);
  }
  const float tot = block_sum_fixed(ss, wsum);
  const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)n), eps)));
  uint16_t *orow = out + (size_t)r * ldo;
  for (int j = threadIdx.x; j < n; j += kNormThreads)
    orow[j] = f32_to_bf16_rn(__fmul_rn(__fmul_rn(bf16_to_f32(rr[j]), rstd), bf16_to_f32(gamma[j])));
}

static cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, void **args, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_qk_norm_rope_kv(const QkParams &p, cudaStream_t st) {
  QkParams pp = p;
  void *args[] = {&pp};
  const dim3 grid((unsigned)((p.nq + p.nkv + kHeadWarps - 1) / kHeadWarps), (unsigned)p.rows);
  return launch_pdl(reinterpret_cast<const void *>(&qk_norm_rope_kv_kernel), grid, dim3(kHeadWarps * 32), args, st);
}

cudaError_t launch_resid_rmsnorm(const float *y, int64_t ldy, uint16_t *resid, int64_t ldr, int rows, int n,
                                 const uint16_t *gamma, float eps, uint16_t *out, int64_t ldo, cudaStream_t st) {
  void *args[] = {&y, &ldy, &resid, &ldr, &n, &gamma, &eps, &out, &ldo};
  auto a16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) % 16) == 0; };
  // y == nullptr: the residual already holds r' (added by the GEMM's epilogue); normalise only
  const bool add = y != nullptr;
  const bool vec = (n % 8) == 0 && (!add || ((ldy % 4) == 0 && a16(y))) && (ldr % 8) == 0 && (ldo % 8) == 0 &&
                   a16(resid) && a16(out) && a16(gamma);
  const void *fn = add ? (vec ? reinterpret_cast<const void *>(&resid_rmsnorm_vec_kernel<true>)
                              : reinterpret_cast<const void *>(&resid_rmsnorm_kernel<true>))
                       : (vec ? reinterpret_cast<const void *>(&resid_rmsnorm_vec_kernel<false>)
                              : reinterpret_cast<const void *>(&resid_rmsnorm_kernel<false>));
  return launch_pdl(fn, dim3((unsigned)rows), dim3(kNormThreads), args, st);
}

}  // namespace qlk

using namespace qlk;

namespace qlk {
int device_setup(int **status);
}

static bool al(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

extern "C" {

int qattn_qknorm_rope_kv(const float *q, int64_t ldq, const float *k, int64_t ldk, const float *v, int64_t ldv,
                         int32_t rows, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t rot_dim,
                         float rope_base, float eps, const uint16_t *q_norm_w, const uint16_t *k_norm_w,
                         const int32_t *pos, uint16_t *q_out, int64_t ldqo, uint16_t *k_ring, uint16_t *v_ring,
                         int32_t ring_len, void *stream) {
  if (!q || !k || !v || !q_norm_w || !k_norm_w || !pos || !q_out || !k_ring || !v_ring) return QL_ERR_NULL;
  if (rows < 1 || rows > 16) return QL_ERR_ROWS;
  if (n_q_heads < 1 || n_kv_heads < 1 || head_dim < 32 || head_dim > kMaxHeadDim || (head_dim % 32) != 0 ||
      rot_dim < 0 || rot_dim > head_dim || (rot_dim % 2) != 0 || ring_len < 1 || !(rope_base > 0.0f) || !(eps >= 0.0f))
    return QL_ERR_SHAPE;
  if (ldq < (int64_t)n_q_heads * head_dim || ldk < (int64_t)n_kv_heads * head_dim ||
      ldv < (int64_t)n_kv_heads * head_dim || ldqo < (int64_t)n_q_heads * head_dim || !al(q, 4) || !al(k, 4) ||
      !al(v, 4) || !al(q_out, 2) || !al(k_ring, 2) || !al(v_ring, 2) || !al(pos, 4))
    return QL_ERR_ALIGN;
  int e = device_setup(nullptr);
  if (e) return e;
  QkParams p;
  p.q = q; p.k = k; p.v = v;
  p.ldq = ldq; p.ldk = ldk; p.ldv = ldv;
  p.rows = rows; p.nq = n_q_heads; p.nkv = n_kv_heads; p.hd = head_dim; p.rot = rot_dim;
  p.base = (double)rope_base;
  p.eps = eps;
  p.qw = q_norm_w; p.kw = k_norm_w;
  p.pos = pos;
  p.q_out = q_out; p.ldqo = ldqo;
  p.k_ring = k_ring; p.v_ring = v_ring; p.ring_len = ring_len;
  if (launch_qk_norm_rope_kv(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    (void)cudaGetLastError();
    return QL_ERR_LAUNCH;
  }
  return QL_OK;
}

int qresid_rmsnorm(const float *y, int64_t ldy, uint16_t *resid, int64_t ldr, int32_t rows, int32_t n,
                   const uint16_t *gamma, float eps, uint16_t *out, int64_t ldo, void *stream) {
  if (!y || !resid || !gamma || !out) return QL_ERR_NULL;
  if (rows < 1) return QL_ERR_ROWS;
  if (n < 1 || !(eps >= 0.0f)) return QL_ERR_SHAPE;
  if (ldy < n || ldr < n || ldo < n || !al(y, 4) || !al(resid, 2) || !al(out, 2) || !al(gamma, 2)) return QL_ERR_ALIGN;
  int e = device_setup(nullptr);
  if (e) return e;
  if (launch_resid_rmsnorm(y, ldy, resid, ldr, rows, n, gamma, eps, out, ldo, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return QL_ERR_LAUNCH;
  }
  return QL_OK;
}

}  // extern "C"
