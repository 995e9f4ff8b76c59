// common.cuh - small device helpers shared by the qlinear kernels (sm_103a only).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ != 1030)
#error "qlinear kernels are written for sm_103a only"
#endif

namespace qlk {

constexpr int kGroup = 64;
constexpr int kErrTimeout = -9;

// activations: keep them in L1, they are re-read by every CTA on the SM
__device__ __forceinline__ uint4 ldg_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_u16(const uint16_t *p) {
  unsigned short v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// round-to-nearest-even float -> bf16 bits (finite inputs; NaN stays NaN)
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  uint16_t h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
  return h;
}

// bf16x2 a*b + c, round to nearest
__device__ __forceinline__ uint32_t fma_bf16x2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// pack two floats into bf16x2 (lo in bits 0..15), round to nearest (exact for the
// small integers it is used on)
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// ---------------------------------------------------------------------------------
// Exact conversion of unsigned codes to bf16 pairs.  A bf16 with biased exponent
// 134 (0x4300 = 128.0) has a unit in the last place of exactly 1 over [128, 256),
// so OR-ing a code q < 128 into its mantissa gives 128 + q exactly; one bf16x2 fma
// (x * 1 - 128) then yields q exactly.  Pairs are (lower-k value, higher-k value).
// ---------------------------------------------------------------------------------
constexpr uint32_t kBf16Magic2 = 0x43004300u;  // (128.0, 128.0)
constexpr uint32_t kBf16One2 = 0x3F803F80u;    // (1.0, 1.0)
constexpr uint32_t kBf16Neg128x2 = 0xC300C300u;  // (-128.0, -128.0)

// 4-bit: natural pair t (nibbles 2t and 2t+1) of word w; w4 = w >> 4
__device__ __forceinline__ uint32_t q4_pair(uint32_t w, uint32_t w4, int t) {
  // byte 0 <- w.byte[t] (low nibble = nibble 2t), byte 2 <- w4.byte[t] (low nibble = 2t+1)
  const uint32_t sel = (uint32_t)t | ((uint32_t)t << 4) | ((uint32_t)(4 + t) << 8) | ((uint32_t)(4 + t) << 12);
  uint32_t v = __byte_perm(w, w4, sel);
  v = (v & 0x000F000Fu) | kBf16Magic2;
  return fma_bf16x2(v, kBf16One2, kBf16Neg128x2);
}

// 4-bit: codes t and t+4 of word w (t = 0..3) as the exact bf16 pair
// (q_t - z, q_{t+4} - z).  Nibble t sits at bits 4t..4t+3 and nibble t+4 at bits
// 16+4t..16+4t+3, so one shift puts both at the bottom of their 16-bit halves; the
// mask-or places them in the mantissas of (128, 128) and one bf16x2 fma adds
// zc = -(128 + z) in both halves (z = 0: the codes themselves).  Pairing t with t+4
// (instead of 2t with 2t+1) saves the byte permute; the activations are loaded in the
// same order.
__device__ __forceinline__ uint32_t q4_split_pair(uint32_t w, int t, uint32_t zc = kBf16Neg128x2) {
  const uint32_t v = ((t == 0 ? w : (w >> (4 * t))) & 0x000F000Fu) | kBf16Magic2;
  return fma_bf16x2(v, kBf16One2, zc);
}

// 6-bit: a 12-bit field f (two 6-bit codes, lower code in bits 0..5) as the exact bf16
// pair (q0 - z, q1 - z), zc = -(128 + z) in both halves
__device__ __forceinline__ uint32_t q6_pair(uint32_t f, uint32_t zc = kBf16Neg128x2) {
  uint32_t v = (f & 0x3Fu) | ((f << 10) & 0x003F0000u) | kBf16Magic2;
  return fma_bf16x2(v, kBf16One2, zc);
}

// 8-bit: natural pair t (bytes 2t and 2t+1) of word w as the exact bf16 pair
// (q0 - z, q1 - z), through float32 2^23 + q; zf = 2^23 + z
__device__ __forceinline__ uint32_t q8_pair(uint32_t w, int t, float zf = 8388608.0f) {
  const uint32_t m = 0x4B000000u;  // bytes (0, 0, 0, 0x4B)
  const uint32_t s0 = (uint32_t)(2 * t) | (4u << 4) | (4u << 8) | (7u << 12);
  const uint32_t s1 = (uint32_t)(2 * t + 1) | (4u << 4) | (4u << 8) | (7u << 12);
  float lo = __fsub_rn(__uint_as_float(__byte_perm(w, m, s0)), zf);
  float hi = __fsub_rn(__uint_as_float(__byte_perm(w, m, s1)), zf);
  return pack_bf16x2(lo, hi);
}

// 12-bit window starting at bit `off` (0 <= off <= 84) of a 96-bit little-endian
// value held in three words
__device__ __forceinline__ uint32_t bits96_at(uint32_t w0, uint32_t w1, uint32_t w2, int off) {
  if (off < 32) return __funnelshift_r(w0, w1, off);
  if (off < 64) return __funnelshift_r(w1, w2, off - 32);
  return w2 >> (off - 64);
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + C, fp32 accumulate.  A pure function
// of its registers (not volatile), so the compiler may interleave independent MMAs
// with the loads and conversions of other groups.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1, const float (&c)[4]) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

// SwiGLU element: bf16(silu(a) * c), silu(t) = t / (1 + exp(-t)) in float32.
__device__ __forceinline__ uint16_t swiglu_bf16(float a, float c) {
  float sa = __fdiv_rn(a, __fadd_rn(1.0f, expf(-a)));
  return f32_to_bf16_rn(__fmul_rn(sa, c));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

}  // namespace qlk
