// qmv_core.cuh - the arithmetic of the decode kernels (sm_103a): code extraction,
// activation fragments, scale/bias pairs and the per-group tensor-core step
// mv_group(), kept apart from the kernel's data movement so that any kernel splitting
// the same work the same way computes bit-identical results.
#pragma once

#include <cstdint>

#include "common.cuh"
#include "qmv.cuh"
#include "sync.cuh"

namespace qlk {

template <int BITS> struct Geo;
// chunks per span (2, computing the first half while the second lands, measured slower
// on the decode pass)
constexpr int kNch = 1;
// spans of 32 groups (4-bit) or 16 groups (6/8-bit), split over the compute warps and chunks
template <> struct Geo<4> {
  static constexpr int kLw = 2;                          // words per lane per row per group
  static constexpr int kGpw = 32 / (kMvWarps * kNch);    // groups per compute warp per chunk
};
template <> struct Geo<6> { static constexpr int kLw = 3; static constexpr int kGpw = 16 / (kMvWarps * kNch); };
template <> struct Geo<8> { static constexpr int kLw = 4; static constexpr int kGpw = 16 / (kMvWarps * kNch); };
static_assert(Geo<6>::kGpw >= 1, "every compute warp owns at least one group per chunk");
template <int BITS> __host__ __device__ constexpr int gbytes() { return 8 * BITS; }                  // bytes per row per group
template <int BITS> __host__ __device__ constexpr int gpc() { return kMvWarps * Geo<BITS>::kGpw; }  // groups per chunk
template <int BITS> __host__ __device__ constexpr int span_g() { return kNch * gpc<BITS>(); }        // groups per span
template <int BITS> __host__ __device__ constexpr int wpitch() { return span_g<BITS>() * gbytes<BITS>() + 32; }  // padded row pitch

// Lane (g4, c) of a warp holds, for each of its two rows (g4, g4 + 8), the 16 codes
// j = 64*g + 16*c + i (i = 0..15) of group g.  MMA j (0..3) of the group takes k
// slots {2c, 2c+1} <- i = {2j, 2j+1} and {2c+8, 2c+9} <- i = {8+2j, 9+2j}; the B
// fragments use the same mapping, so they are plain 16-byte reads of x.
template <int BITS>
__device__ __forceinline__ void lds_lane_words(const uint8_t *p, uint32_t (&w)[Geo<BITS>::kLw]) {
  if constexpr (BITS == 4) {
    const uint2 v = *reinterpret_cast<const uint2 *>(p);
    w[0] = v.x; w[1] = v.y;
  } else if constexpr (BITS == 8) {
    const uint4 v = *reinterpret_cast<const uint4 *>(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else {
    const uint32_t *q = reinterpret_cast<const uint32_t *>(p);
    w[0] = q[0]; w[1] = q[1]; w[2] = q[2];
  }
}

// bf16 pairs of centred codes q - z for MMA j: lo = codes (j, j+4) / (2j, 2j+1),
// hi = codes (8+j, 12+j) / (8+2j, 9+2j) for 4 / 6 and 8 bits; zc is the row's offset
// constant (group_factors)
template <int BITS>
__device__ __forceinline__ void lane_pairs(const uint32_t (&w)[Geo<BITS>::kLw], int j, uint32_t zc, uint32_t &lo,
                                           uint32_t &hi) {
  if constexpr (BITS == 4) {
    lo = q4_split_pair(w[0], j, zc);
    hi = q4_split_pair(w[1], j, zc);
  } else if constexpr (BITS == 8) {
    lo = q8_pair(w[j >> 1], j & 1, __uint_as_float(zc));
    hi = q8_pair(w[2 + (j >> 1)], j & 1, __uint_as_float(zc));
  } else {
    lo = q6_pair(bits96_at(w[0], w[1], w[2], 12 * j), zc);
    hi = q6_pair(bits96_at(w[0], w[1], w[2], 48 + 12 * j), zc);
  }
}

// The factors of one (row, group): (scale s, centred bias b + s*z, offset constant, 0)
// with the group's zero point z = round(-b / s) clamped to the code range.  The group
// contributes s * sum (q - z) x + (b + s*z) * S, the same linear map as s*P + b*S, but
// now |w_j| >= |b + s*z| and s*|q_j - z| <= 2|w_j| for every j of the group (the zero
// point is the code nearest to where w changes sign, or an end of the range if w has
// one sign), so no term of the factored sum exceeds twice sum |w x| and the fp32
// rounding of every step is relative to |w x|.  Where the dequantized weights vanish
// (q = c, b = -s*c) z = c and both terms are exactly zero.  The offset constant is
// -(128 + z) as a bf16 pair (4 and 6 bits, exact for z <= 63) or 2^23 + z as fp32
// (8 bits); a zero scale gives z = 0.
template <int BITS>
__device__ __forceinline__ float4 group_factors(float s, float b) {
  constexpr float kMaxQ = (float)((1 << BITS) - 1);
  const float z = fminf(fmaxf(rintf(__fdiv_rn(-b, s)), 0.0f), kMaxQ);  // a NaN quotient becomes 0
  uint32_t zc;
  if constexpr (BITS == 8) {
    zc = __float_as_uint(__fadd_rn(8388608.0f, z));
  } else {
    const uint32_t h = f32_to_bf16_rn(-(128.0f + z));
    zc = h | (h << 16);
  }
  return make_float4(s, __fmaf_rn(s, z, b), __uint_as_float(zc), 0.0f);
}

__device__ __forceinline__ uint32_t u4get(const uint4 &v, int j) {
  return j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
}

// 16 bytes global -> shared, asynchronously (bypassing L1); completion per thread by
// cp_async_wait_all
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

constexpr int kMvThreads = kMvWarps * 32;  // compute warps (each also copies its weight bytes)
constexpr int kMvComputeThreads = kMvWarps * 32;
constexpr int kBarCompute = 1;                   // named barrier of the compute warps

// activation fragment of lane (g4, c) for one group: x[row][64g + 16c .. +16) as two
// 16-byte pieces; 4-bit takes each 8-value block in the order x0 x4 x1 x5 x2 x6 x3 x7,
// the order in which q4_split_pair pairs the codes of a word
template <bool kPair4>
__device__ __forceinline__ void load_x_frag(const uint16_t *px, uint4 &a, uint4 &b) {
  a = ldg_v4(px);
  b = ldg_v4(px + 8);
  if constexpr (kPair4) {
    a = make_uint4(__byte_perm(a.x, a.z, 0x5410), __byte_perm(a.x, a.z, 0x7632), __byte_perm(a.y, a.w, 0x5410),
                   __byte_perm(a.y, a.w, 0x7632));
    b = make_uint4(__byte_perm(b.x, b.z, 0x5410), __byte_perm(b.x, b.z, 0x7632), __byte_perm(b.y, b.w, 0x5410),
                   __byte_perm(b.y, b.w, 0x7632));
  }
}

// One group of one warp: S of the group for this lane's output columns (MMA with
// A = 1), then for each of the NMAT matrices the exact centred codes q - z of rows g4 and g4 + 8
// (wrow: the lane's bytes of row 0 of matrix 0 of the group; rows WP bytes apart,
// matrices 16 rows apart) on the tensor cores with a fresh accumulator, and the
// group's affine step y = fma(s, P', y); y = fma(b', S, y) with the factors of rows g4
// and g4 + 8 (group_factors; fg: matrix 0's factors of the group, 16 rows; matrices
// fstride apart).
template <int BITS, int NB, int NMAT>
__device__ __forceinline__ void mv_group(const uint8_t *wrow, int WP, const float4 *fg, int fstride,
                                         const uint4 (&X0)[NB], const uint4 (&X1)[NB], int g4,
                                         float (&y)[NMAT * NB * 4]) {
  constexpr int LW = Geo<BITS>::kLw;
  const uint32_t ones[4] = {kBf16One2, kBf16One2, kBf16One2, kBf16One2};
  float S[NB][4];
#pragma unroll
  for (int h = 0; h < NB; ++h) {
    S[h][0] = S[h][1] = S[h][2] = S[h][3] = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) mma_bf16_16816(S[h], ones, u4get(X0[h], j), u4get(X1[h], j), S[h]);
  }
#pragma unroll
  for (int t = 0; t < NMAT; ++t) {
    uint32_t W0[LW], W1[LW];
    lds_lane_words<BITS>(wrow + (t * 16 + g4) * WP, W0);
    lds_lane_words<BITS>(wrow + (t * 16 + g4 + 8) * WP, W1);
    // offset constants of rows g4 and g4 + 8 now, their (scale, centred bias) after the MMAs
    const uint32_t zc0 = __float_as_uint(fg[t * fstride + g4].z);
    const uint32_t zc1 = __float_as_uint(fg[t * fstride + g4 + 8].z);
    float P[NB][4];
#pragma unroll
    for (int h = 0; h < NB; ++h) P[h][0] = P[h][1] = P[h][2] = P[h][3] = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t a[4];
      lane_pairs<BITS>(W0, j, zc0, a[0], a[2]);
      lane_pairs<BITS>(W1, j, zc1, a[1], a[3]);
#pragma unroll
      for (int h = 0; h < NB; ++h) mma_bf16_16816(P[h], a, u4get(X0[h], j), u4get(X1[h], j), P[h]);
    }
    const float2 f0 = *reinterpret_cast<const float2 *>(&fg[t * fstride + g4]);
    const float2 f1 = *reinterpret_cast<const float2 *>(&fg[t * fstride + g4 + 8]);
#pragma unroll
    for (int h = 0; h < NB; ++h) {
      float *yy = &y[(t * NB + h) * 4];
      yy[0] = __fmaf_rn(f0.x, P[h][0], yy[0]); yy[0] = __fmaf_rn(f0.y, S[h][0], yy[0]);
      yy[1] = __fmaf_rn(f0.x, P[h][1], yy[1]); yy[1] = __fmaf_rn(f0.y, S[h][1], yy[1]);
      yy[2] = __fmaf_rn(f1.x, P[h][2], yy[2]); yy[2] = __fmaf_rn(f1.y, S[h][0], yy[2]);
      yy[3] = __fmaf_rn(f1.x, P[h][3], yy[3]); yy[3] = __fmaf_rn(f1.y, S[h][1], yy[3]);
    }
  }
}

}  // namespace qlk
