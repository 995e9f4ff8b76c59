// qmv.cu - decode matvecs over MLX affine 4/6/8-bit group-64 weights (sm_103a).
//
// One kernel template serves qlinear_mv / qlinear_mv_rows (one weight), the fused
// w1 + w3 + SwiGLU step (two weights, bf16 output) and the fused q/k/v/gate step
// (four weights, one launch).  TensorFold PR #1696 (later revision), "What it adds":
// N-row matvecs summing each row as the one-row kernels do; decode fuses w1 + w3 +
// SwiGLU and the four attention matvecs.
//
// Work decomposition (a function of k and bits only, never of the number of rows R,
// of n or of the fused/unfused choice):
//   * a CTA owns a 16-row tile of W (both w1 and w3 in the fused FFN) and a k-span;
//     CTAs of a cluster split k into spans, a span is processed in chunks of
//     span_g<BITS>() groups (2048 k for 4-bit, 1024 k for 6/8-bit);
//   * each of the 4 warps owns Geo::kGpw consecutive groups of the chunk.  Its lanes
//     start one bulk copy (cp.async.bulk) per weight row of the slice - contiguous
//     runs of 192-256 bytes straight from HBM into shared memory, so the weight
//     stream leaves the SM as few large requests, all issued at kernel start;
//   * scales and biases are staged in shared memory as fp32; activations (the only
//     input a preceding kernel may write) are bulk-copied in after
//     griddepcontrol.wait, so with programmatic dependent launch the weight stream of
//     this kernel overlaps the tail of the previous one;
//   * per group the codes are converted exactly to bf16 and multiplied on the tensor
//     cores with mma.sync m16n8k16 (rows of W as A, activation rows as B):
//       P_g = sum_{j in g} q_j x_j      (fresh fp32 accumulator per group)
//       S_g = sum_{j in g} x_j          (same MMA with A = 1)
//       y   = fma(scale_g, P_g, y);  y = fma(bias_g, S_g, y)   (groups in order)
//   * warp partials are added in warp order through shared memory, CTA partials in
//     rank order through distributed shared memory.  No atomics, no scratch memory.
// The tensor core computes every output column (activation row) from that column's
// data alone, so a row's result does not depend on how many rows share the call.
#include <cooperative_groups.h>

#include "common.cuh"
#include "qmv.cuh"
#include "sync.cuh"

namespace cg = cooperative_groups;

namespace qlk {

template <int BITS> struct Geo;
template <> struct Geo<4> {
  static constexpr int kLw = 2;     // words per lane per row per group
  static constexpr int kGpw = 8;    // groups per warp slice
};
template <> struct Geo<6> { static constexpr int kLw = 3; static constexpr int kGpw = 4; };
template <> struct Geo<8> { static constexpr int kLw = 4; static constexpr int kGpw = 4; };
template <int BITS> __host__ __device__ constexpr int gbytes() { return 8 * BITS; }                           // bytes per row per group
template <int BITS> __host__ __device__ constexpr int span_g() { return kMvWarps * Geo<BITS>::kGpw; }          // groups per chunk
template <int BITS> __host__ __device__ constexpr int wpitch() { return span_g<BITS>() * gbytes<BITS>() + 32; }  // padded row pitch
__host__ __device__ constexpr int xpitch(int sg) { return sg * 64 + 8; }                                       // bf16 elements

int mv_span_g(int bits) { return bits == 4 ? span_g<4>() : (bits == 6 ? span_g<6>() : span_g<8>()); }

// Lane (g4, c) of a warp holds, for each of its two rows (g4, g4 + 8), the 16 codes
// j = 64*g + 16*c + i (i = 0..15) of group g.  MMA j (0..3) of the group takes k
// slots {2c, 2c+1} <- i = {2j, 2j+1} and {2c+8, 2c+9} <- i = {8+2j, 9+2j}; the B
// fragments use the same mapping, so they are plain 16-byte reads of x.
template <int BITS>
__device__ __forceinline__ void lds_lane_words(const uint8_t *p, uint32_t (&w)[Geo<BITS>::kLw]) {
  const uint32_t a = smem_addr(p);
  if constexpr (BITS == 4) {
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "r"(a));
  } else if constexpr (BITS == 8) {
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(a));
  } else {
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[0]) : "r"(a));
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[1]) : "r"(a + 4));
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[2]) : "r"(a + 8));
  }
}

// bf16 pairs for MMA j: lo = codes (2j, 2j+1), hi = codes (8+2j, 9+2j)
template <int BITS>
__device__ __forceinline__ void lane_pairs(const uint32_t (&w)[Geo<BITS>::kLw], int j, uint32_t &lo, uint32_t &hi) {
  if constexpr (BITS == 4) {
    lo = q4_pair(w[0], w[0] >> 4, j);
    hi = q4_pair(w[1], w[1] >> 4, j);
  } else if constexpr (BITS == 8) {
    lo = q8_pair(w[j >> 1], j & 1);
    hi = q8_pair(w[2 + (j >> 1)], j & 1);
  } else {
    lo = q6_pair(bits96_at(w[0], w[1], w[2], 12 * j));
    hi = q6_pair(bits96_at(w[0], w[1], w[2], 48 + 12 * j));
  }
}

__device__ __forceinline__ uint32_t u4get(const uint4 &v, int j) {
  return j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
}

__device__ __forceinline__ uint4 lds_v4(const void *p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// Shared-memory layout of one CTA (dynamic, 128-byte aligned):
//   wsm [NMAT][16][wpitch]                   weight rows of the chunk (one bulk copy per row)
//   sbs [NMAT][2][16][span] bf16             scales, biases of the chunk
//   red [kMvWarps][NV][32] fp32              warp partials
//   csum[NV][32] fp32                        CTA partial (read by cluster rank 0)
//   bars[2]                                  weights+scales barrier, activation barrier
//   xs  [rows][xpitch] bf16                  activations of the chunk
template <int BITS, int NB, int MODE> struct MvLayout {
  static constexpr int NMAT = (MODE == kMvFfn) ? 2 : 1;
  static constexpr int NV = NMAT * NB * 4;
  static constexpr int kW = 0;
  static constexpr int kSb = kW + NMAT * 16 * wpitch<BITS>();
  static constexpr int kRed = kSb + NMAT * 2 * 16 * span_g<BITS>() * 2;
  static constexpr int kCsum = kRed + kMvWarps * NV * 32 * 4;
  static constexpr int kBar = kCsum + NV * 32 * 4;
  static constexpr int kX = ((kBar + 2 * 8) + 127) / 128 * 128;
  static int bytes(int rows) { return kX + rows * xpitch(span_g<BITS>()) * 2; }
};

template <int BITS, int NB, int MODE>
__global__ void __launch_bounds__(kMvWarps * 32) qmv_kernel(const __grid_constant__ MvParams p) {
  using Lay = MvLayout<BITS, NB, MODE>;
  constexpr int NMAT = Lay::NMAT;
  constexpr int NV = Lay::NV;
  constexpr int LW = Geo<BITS>::kLw;
  constexpr int GPW = Geo<BITS>::kGpw;
  constexpr int SPAN = span_g<BITS>();
  constexpr int GB = gbytes<BITS>();
  constexpr int WP = wpitch<BITS>();
  constexpr int XP = xpitch(SPAN);
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t *sbs = reinterpret_cast<uint16_t *>(smem + Lay::kSb);
  float *red = reinterpret_cast<float *>(smem + Lay::kRed);
  float *csum = reinterpret_cast<float *>(smem + Lay::kCsum);
  uint64_t *wbar = reinterpret_cast<uint64_t *>(smem + Lay::kBar);
  uint64_t *xbar = wbar + 1;
  uint16_t *xs = reinterpret_cast<uint16_t *>(smem + Lay::kX);

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = p.cs > 1 ? (int)cluster.block_rank() : 0;
  const int tile_g = blockIdx.x / p.cs;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int g4 = lane >> 2, c = lane & 3;
  uint8_t *wsm = smem + Lay::kW;

  int mi = 0, tile = tile_g;
  if constexpr (MODE == kMvAttn) {
    while (mi < 3 && tile_g >= p.tile_end[mi]) ++mi;
    tile = tile_g - (mi ? p.tile_end[mi - 1] : 0);
  }
  const int n = p.m[mi].n;
  const size_t row_bytes = (size_t)p.groups * GB;

  // this CTA's k-span: groups [gs0, gs1), in chunks of SPAN groups
  const int gs0 = rank * p.span_g, gs1 = min(p.groups, gs0 + p.span_g);

  if (threadIdx.x == 0) {
    mbar_init(wbar, 1);
    mbar_init(xbar, 1);
    fence_mbar_init();
  }
  __syncwarp();

  float y[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) y[i] = 0.0f;
  const uint32_t ones[4] = {kBf16One2, kBf16One2, kBf16One2, kBf16One2};
  uint32_t phase = 0;

  for (int ch0 = gs0; ch0 < gs1; ch0 += SPAN) {
    const int ch1 = min(gs1, ch0 + SPAN);
    const int gw0 = ch0 + warp * GPW;  // this warp's slice
    const int gcnt = max(0, min(GPW, ch1 - gw0));
    // ---- 1. weights (and, with 16-byte aligned rows, scales and biases) of the
    //         chunk: warp 0 starts one bulk copy per row, HBM -> smem, at once
    const int cg_n = ch1 - ch0;
    if (warp == 0) {
      const int t = lane >> 4, r = lane & 15;
      const int row = tile * 16 + r;
      const bool mine = lane < NMAT * 16 && row < n;
      const uint32_t wb = (uint32_t)(cg_n * GB), sbb = (uint32_t)(cg_n * 2);
      uint32_t bytes = mine ? wb + (p.sb_bulk ? 2u * sbb : 0u) : 0u;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
      if (lane == 0) {
        if (ch0 != gs0) fence_proxy_async_smem();
        mbar_arrive_expect_tx(wbar, bytes);
      }
      __syncwarp();
      if (mine) {
        const uint8_t *src = reinterpret_cast<const uint8_t *>(p.m[mi + t].wq) + (size_t)row * row_bytes +
                             (size_t)ch0 * GB;
        bulk_g2s(wsm + (t * 16 + r) * WP, src, wb, wbar);
        if (p.sb_bulk) {
          const size_t off = (size_t)row * p.groups + ch0;
          bulk_g2s(sbs + ((t * 2 + 0) * 16 + r) * SPAN, p.m[mi + t].s + off, sbb, wbar);
          bulk_g2s(sbs + ((t * 2 + 1) * 16 + r) * SPAN, p.m[mi + t].b + off, sbb, wbar);
        }
      }
    }
    if (ch0 != gs0) __syncthreads();  // the previous chunk's activations are fully read
    // ---- 2. scales and biases the slow way (rows not 16-byte aligned)
    if (!p.sb_bulk) {
      if (ch0 != gs0) __syncthreads();
      for (int e = threadIdx.x; e < NMAT * 16 * cg_n; e += blockDim.x) {
        const int t = e / (16 * cg_n), rr = (e / cg_n) % 16, gg = e % cg_n;
        const int row = tile * 16 + rr;
        uint16_t sv = 0, bv = 0;
        if (row < n) {
          const size_t off = (size_t)row * p.groups + ch0 + gg;
          sv = (uint16_t)ldg_u16(p.m[mi + t].s + off);
          bv = (uint16_t)ldg_u16(p.m[mi + t].b + off);
        }
        sbs[((t * 2 + 0) * 16 + rr) * SPAN + gg] = sv;
        sbs[((t * 2 + 1) * 16 + rr) * SPAN + gg] = bv;
      }
    }
    // ---- 3. activations: a preceding kernel may write them, so they are read only
    //         after the programmatic-dependency wait; one bulk copy per row
    if (ch0 == gs0) {
      asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
      asm volatile("griddepcontrol.wait;" ::: "memory");
    }
    __syncthreads();  // scales/biases visible; barriers initialised
    if (threadIdx.x == 0) {
      fence_proxy_async_smem();
      const uint32_t xb = (uint32_t)(ch1 - ch0) * 128u;
      mbar_arrive_expect_tx(xbar, xb * (uint32_t)p.rows);
      for (int r = 0; r < p.rows; ++r)
        bulk_g2s(xs + r * XP, p.x + (size_t)r * p.ldx + (size_t)ch0 * 64, xb, xbar);
    }
    bool ok = mbar_wait_bounded(xbar, phase, p.budget_ns, nullptr) &&
              mbar_wait_bounded(wbar, phase, p.budget_ns, nullptr);
    phase ^= 1u;
    ok = __syncthreads_and(ok) != 0;
    if (!ok) {
      if (threadIdx.x == 0) record_status(p.status, kErrTimeout);
      break;
    }
    // ---- 4. per group: exact-code MMAs, then the affine step in group order
    bool xv[NB];
#pragma unroll
    for (int h = 0; h < NB; ++h) xv[h] = (8 * h + g4) < p.rows;
#pragma unroll
    for (int gi = 0; gi < GPW; ++gi) {
      if (gi < gcnt) {
        const int gl = gw0 + gi - ch0;  // group index within the chunk
        uint4 X0[NB], X1[NB];
#pragma unroll
        for (int h = 0; h < NB; ++h) {
          if (xv[h]) {
            const uint16_t *px = xs + (8 * h + g4) * XP + gl * 64 + 16 * c;
            X0[h] = lds_v4(px);
            X1[h] = lds_v4(px + 8);
          } else {
            X0[h] = make_uint4(0, 0, 0, 0);
            X1[h] = make_uint4(0, 0, 0, 0);
          }
        }
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
          lds_lane_words<BITS>(wsm + (t * 16 + g4) * WP + gl * GB + c * 4 * LW, W0);
          lds_lane_words<BITS>(wsm + (t * 16 + g4 + 8) * WP + gl * GB + c * 4 * LW, W1);
          float P[NB][4];
#pragma unroll
          for (int h = 0; h < NB; ++h) P[h][0] = P[h][1] = P[h][2] = P[h][3] = 0.0f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t a[4];
            lane_pairs<BITS>(W0, j, a[0], a[2]);
            lane_pairs<BITS>(W1, j, a[1], a[3]);
#pragma unroll
            for (int h = 0; h < NB; ++h) mma_bf16_16816(P[h], a, u4get(X0[h], j), u4get(X1[h], j), P[h]);
          }
          const float2 sb0 = make_float2(bf16_to_f32(sbs[((t * 2 + 0) * 16 + g4) * SPAN + gl]),
                                         bf16_to_f32(sbs[((t * 2 + 1) * 16 + g4) * SPAN + gl]));
          const float2 sb1 = make_float2(bf16_to_f32(sbs[((t * 2 + 0) * 16 + g4 + 8) * SPAN + gl]),
                                         bf16_to_f32(sbs[((t * 2 + 1) * 16 + g4 + 8) * SPAN + gl]));
#pragma unroll
          for (int h = 0; h < NB; ++h) {
            float *yy = &y[(t * NB + h) * 4];
            yy[0] = __fmaf_rn(sb0.x, P[h][0], yy[0]); yy[0] = __fmaf_rn(sb0.y, S[h][0], yy[0]);
            yy[1] = __fmaf_rn(sb0.x, P[h][1], yy[1]); yy[1] = __fmaf_rn(sb0.y, S[h][1], yy[1]);
            yy[2] = __fmaf_rn(sb1.x, P[h][2], yy[2]); yy[2] = __fmaf_rn(sb1.y, S[h][0], yy[2]);
            yy[3] = __fmaf_rn(sb1.x, P[h][3], yy[3]); yy[3] = __fmaf_rn(sb1.y, S[h][1], yy[3]);
          }
        }
      }
    }
    __syncthreads();  // every warp is done with the chunk before it is refilled
  }

  // ---- partials: warps in order, then cluster ranks in order
#pragma unroll
  for (int i = 0; i < NV; ++i) red[(warp * NV + i) * 32 + lane] = y[i];
  __syncthreads();
  for (int v = threadIdx.x; v < NV * 32; v += blockDim.x) {
    const int i = v >> 5, ln = v & 31;
    float acc = red[i * 32 + ln];
    for (int w = 1; w < nwarps; ++w) acc = __fadd_rn(acc, red[(w * NV + i) * 32 + ln]);
    csum[i * 32 + ln] = acc;
  }
  if (p.cs > 1) cluster.sync();
  else __syncthreads();
  if (rank == 0) {
    constexpr int NO = NB * 4;  // outputs per lane per matrix
    for (int v = threadIdx.x; v < NO * 32; v += blockDim.x) {
      const int i = v >> 5, ln = v & 31;
      float acc[NMAT];
#pragma unroll
      for (int t = 0; t < NMAT; ++t) acc[t] = csum[(t * NO + i) * 32 + ln];
      for (int r = 1; r < p.cs; ++r) {
        const float *rs = cluster.map_shared_rank(csum, r);
#pragma unroll
        for (int t = 0; t < NMAT; ++t) acc[t] = __fadd_rn(acc[t], rs[(t * NO + i) * 32 + ln]);
      }
      // value i of lane ln: half h = i / 4, element e = i % 4
      const int h = i >> 2, e = i & 3;
      const int row = tile * 16 + (ln >> 2) + ((e & 2) ? 8 : 0);
      const int xr = 8 * h + 2 * (ln & 3) + (e & 1);
      if (row < n && xr < p.rows) {
        const MvMat &M = p.m[mi];
        if constexpr (MODE == kMvFfn) {
          static_cast<uint16_t *>(M.out)[(size_t)xr * M.ldo + row] = swiglu_bf16(acc[0], acc[1]);
        } else {
          static_cast<float *>(M.out)[(size_t)xr * M.ldo + row] = acc[0];
        }
      }
    }
  }
  if (p.cs > 1) cluster.sync();
}

template <int BITS, int NB, int MODE>
static cudaError_t launch_t(const MvParams &p, int nwarps, int tiles, cudaStream_t st) {
  using Lay = MvLayout<BITS, NB, MODE>;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(qmv_kernel<BITS, NB, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay::bytes(16));
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * p.cs));
  cfg.blockDim = dim3((unsigned)(nwarps * 32));
  cfg.dynamicSmemBytes = (size_t)Lay::bytes(p.rows);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, qmv_kernel<BITS, NB, MODE>, p);
}

template <int MODE>
static cudaError_t launch_mode(const MvParams &p, int bits, int nwarps, int tiles, cudaStream_t st) {
  const bool two = p.rows > 8;
  switch (bits) {
    case 4: return two ? launch_t<4, 2, MODE>(p, nwarps, tiles, st) : launch_t<4, 1, MODE>(p, nwarps, tiles, st);
    case 6: return two ? launch_t<6, 2, MODE>(p, nwarps, tiles, st) : launch_t<6, 1, MODE>(p, nwarps, tiles, st);
    default: return two ? launch_t<8, 2, MODE>(p, nwarps, tiles, st) : launch_t<8, 1, MODE>(p, nwarps, tiles, st);
  }
}

// k-decomposition used by every decode launch (a function of k and bits only):
// CTAs per cluster cs = min(8, ceil(groups / span)), each CTA takes ceil(groups / cs)
// groups in chunks of the span; warps = ceil(min(groups, span) / gpw) <= kMvWarps.
void mv_geometry(int k, int bits, int &groups, int &span_g_out, int &nwarps, int &cs) {
  groups = k / kGroup;
  const int span = mv_span_g(bits);
  const int gpw = span / kMvWarps;
  const int need = (groups + span - 1) / span;
  cs = need < kMvMaxCluster ? need : kMvMaxCluster;
  span_g_out = (groups + cs - 1) / cs;
  const int chunk = span_g_out < span ? span_g_out : span;
  nwarps = (chunk + gpw - 1) / gpw;
}

cudaError_t launch_mv(MvParams &p, int mode, int bits, int tiles, cudaStream_t st) {
  int nwarps;
  mv_geometry(p.k, bits, p.groups, p.span_g, nwarps, p.cs);
  p.wpr = p.k * bits / 32;
  // scale/bias rows of a chunk can be bulk-copied when every copy starts and ends on
  // a 16-byte boundary: groups and the per-CTA span multiples of 8, pointers aligned
  const int nm = mode == kMvAttn ? 4 : (mode == kMvFfn ? 2 : 1);
  bool sb = (p.groups % 8) == 0 && (p.span_g % 8) == 0;
  for (int i = 0; i < nm; ++i)
    sb = sb && (reinterpret_cast<uintptr_t>(p.m[i].s) % 16) == 0 && (reinterpret_cast<uintptr_t>(p.m[i].b) % 16) == 0;
  p.sb_bulk = sb ? 1 : 0;
  switch (mode) {
    case kMvFfn: return launch_mode<kMvFfn>(p, bits, nwarps, tiles, st);
    case kMvAttn: return launch_mode<kMvAttn>(p, bits, nwarps, tiles, st);
    default: return launch_mode<kMvPlain>(p, bits, nwarps, tiles, st);
  }
}

}  // namespace qlk
