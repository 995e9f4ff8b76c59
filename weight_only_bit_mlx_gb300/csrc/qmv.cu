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
//   * a warp owns a 16-row tile of W and a k-slice of kGpw consecutive 64-wide groups;
//   * per group the packed codes are loaded straight from HBM into registers with
//     vector loads, converted exactly to bf16, and multiplied on the tensor cores with
//     mma.sync m16n8k16 (rows of W as A, up to 8 activation rows per B half):
//       P_g = sum_{j in g} q_j x_j      (fresh fp32 accumulator per group)
//       S_g = sum_{j in g} x_j          (same MMA with A = 1)
//       y   = fma(scale_g, P_g, y);  y = fma(bias_g, S_g, y)   (groups in order)
//   * warps of a CTA take consecutive slices; CTAs of a cluster split k further;
//     partials are added in (CTA rank, warp) order through shared and distributed
//     shared memory.  No atomics, no scratch memory.
// The tensor core computes every output column (activation row) from that column's
// data alone, so a row's result does not depend on how many rows share the call.
#include <cooperative_groups.h>

#include "common.cuh"
#include "qmv.cuh"

namespace cg = cooperative_groups;

namespace qlk {

template <int BITS> struct Geo;
template <> struct Geo<4> { static constexpr int kWpg = 8;  static constexpr int kLw = 2; };
template <> struct Geo<6> { static constexpr int kWpg = 12; static constexpr int kLw = 3; };
template <> struct Geo<8> { static constexpr int kWpg = 16; static constexpr int kLw = 4; };

// Lane (g4, c) of a warp holds, for each of its two rows (g4, g4 + 8), the 16 codes
// j = 64*g + 16*c + i (i = 0..15) of group g.  MMA j (0..3) of the group takes k
// slots {2c, 2c+1} <- i = {2j, 2j+1} and {2c+8, 2c+9} <- i = {8+2j, 9+2j}; the B
// fragments use the same mapping, so they are plain 16-byte loads of x.
template <int BITS>
__device__ __forceinline__ void load_lane_words(const uint32_t *row, int g, int c, uint32_t (&w)[Geo<BITS>::kLw]) {
  const uint32_t *p = row + g * Geo<BITS>::kWpg + c * Geo<BITS>::kLw;
  if constexpr (BITS == 4) {
    uint2 v = ldg_nc_v2(p);
    w[0] = v.x; w[1] = v.y;
  } else if constexpr (BITS == 8) {
    uint4 v = ldg_nc_v4(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else {
    w[0] = ldg_nc_u32(p); w[1] = ldg_nc_u32(p + 1); w[2] = ldg_nc_u32(p + 2);
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

template <int BITS, int NB, int MODE>
__global__ void __launch_bounds__(kMvMaxWarps * 32) qmv_kernel(const __grid_constant__ MvParams p) {
  constexpr int NMAT = (MODE == kMvFfn) ? 2 : 1;
  constexpr int LW = Geo<BITS>::kLw;
  constexpr int NV = NMAT * NB * 4;  // partial values per lane
  __shared__ float red[kMvMaxWarps][NV][32];
  __shared__ float csum[NV][32];

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int tile_g = blockIdx.x / p.cs;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int g4 = lane >> 2, c = lane & 3;

  int mi = 0, tile = tile_g;
  if constexpr (MODE == kMvAttn) {
    while (mi < 3 && tile_g >= p.tile_end[mi]) ++mi;
    tile = tile_g - (mi ? p.tile_end[mi - 1] : 0);
  }
  const int n = p.m[mi].n;
  const int row0 = tile * 16 + g4, row1 = row0 + 8;
  const bool v0 = row0 < n, v1 = row1 < n;

  const uint32_t *wrow[NMAT][2];
  const uint16_t *srow[NMAT][2], *brow[NMAT][2];
#pragma unroll
  for (int t = 0; t < NMAT; ++t) {
    const MvMat &M = p.m[mi + t];
    wrow[t][0] = M.wq + (size_t)(v0 ? row0 : 0) * p.wpr;
    wrow[t][1] = M.wq + (size_t)(v1 ? row1 : 0) * p.wpr;
    srow[t][0] = M.s + (size_t)(v0 ? row0 : 0) * p.groups;
    srow[t][1] = M.s + (size_t)(v1 ? row1 : 0) * p.groups;
    brow[t][0] = M.b + (size_t)(v0 ? row0 : 0) * p.groups;
    brow[t][1] = M.b + (size_t)(v1 ? row1 : 0) * p.groups;
  }
  const uint16_t *xrow[NB];
  bool xv[NB];
#pragma unroll
  for (int h = 0; h < NB; ++h) {
    const int r = 8 * h + g4;
    xv[h] = r < p.rows;
    xrow[h] = p.x + (size_t)(xv[h] ? r : 0) * p.ldx + 16 * c;
  }

  float y[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) y[i] = 0.0f;

  const uint32_t ones[4] = {kBf16One2, kBf16One2, kBf16One2, kBf16One2};

  const int slice_stride = nwarps * p.cs;
  for (int sl = rank * nwarps + warp; sl < p.slices; sl += slice_stride) {
    const int gbeg = sl * kMvGpw;
    const int gcnt = min(kMvGpw, p.groups - gbeg);
    // ---- all HBM loads of the slice first: packed codes, scales, biases
    uint32_t W[NMAT][kMvGpw][2][LW];
    uint32_t SB[NMAT][kMvGpw][4];
#pragma unroll
    for (int gi = 0; gi < kMvGpw; ++gi) {
#pragma unroll
      for (int t = 0; t < NMAT; ++t) {
        if (gi < gcnt) {
          const int g = gbeg + gi;
          if (v0) load_lane_words<BITS>(wrow[t][0], g, c, W[t][gi][0]);
          else for (int q = 0; q < LW; ++q) W[t][gi][0][q] = 0u;
          if (v1) load_lane_words<BITS>(wrow[t][1], g, c, W[t][gi][1]);
          else for (int q = 0; q < LW; ++q) W[t][gi][1][q] = 0u;
          SB[t][gi][0] = v0 ? ldg_u16(srow[t][0] + g) : 0u;
          SB[t][gi][1] = v1 ? ldg_u16(srow[t][1] + g) : 0u;
          SB[t][gi][2] = v0 ? ldg_u16(brow[t][0] + g) : 0u;
          SB[t][gi][3] = v1 ? ldg_u16(brow[t][1] + g) : 0u;
        }
      }
    }
    // ---- activations (L1/L2 resident) for the slice
    uint4 X0[kMvGpw][NB], X1[kMvGpw][NB];
#pragma unroll
    for (int gi = 0; gi < kMvGpw; ++gi) {
#pragma unroll
      for (int h = 0; h < NB; ++h) {
        if (gi < gcnt && xv[h]) {
          const uint16_t *px = xrow[h] + (size_t)(gbeg + gi) * kGroup;
          X0[gi][h] = ldg_v4(px);
          X1[gi][h] = ldg_v4(px + 8);
        } else {
          X0[gi][h] = make_uint4(0, 0, 0, 0);
          X1[gi][h] = make_uint4(0, 0, 0, 0);
        }
      }
    }
    // ---- per group: exact-code MMAs, then the affine step in group order
#pragma unroll
    for (int gi = 0; gi < kMvGpw; ++gi) {
      if (gi < gcnt) {
        float S[NB][4];
#pragma unroll
        for (int h = 0; h < NB; ++h) {
          S[h][0] = S[h][1] = S[h][2] = S[h][3] = 0.0f;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            mma_bf16_16816(S[h], ones, u4get(X0[gi][h], j), u4get(X1[gi][h], j), S[h]);
        }
#pragma unroll
        for (int t = 0; t < NMAT; ++t) {
          float P[NB][4];
#pragma unroll
          for (int h = 0; h < NB; ++h) P[h][0] = P[h][1] = P[h][2] = P[h][3] = 0.0f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t a[4];
            lane_pairs<BITS>(W[t][gi][0], j, a[0], a[2]);
            lane_pairs<BITS>(W[t][gi][1], j, a[1], a[3]);
#pragma unroll
            for (int h = 0; h < NB; ++h)
              mma_bf16_16816(P[h], a, u4get(X0[gi][h], j), u4get(X1[gi][h], j), P[h]);
          }
          const float s0 = bf16_to_f32(SB[t][gi][0]), s1 = bf16_to_f32(SB[t][gi][1]);
          const float b0 = bf16_to_f32(SB[t][gi][2]), b1 = bf16_to_f32(SB[t][gi][3]);
#pragma unroll
          for (int h = 0; h < NB; ++h) {
            float *yy = &y[(t * NB + h) * 4];
            yy[0] = __fmaf_rn(s0, P[h][0], yy[0]); yy[0] = __fmaf_rn(b0, S[h][0], yy[0]);
            yy[1] = __fmaf_rn(s0, P[h][1], yy[1]); yy[1] = __fmaf_rn(b0, S[h][1], yy[1]);
            yy[2] = __fmaf_rn(s1, P[h][2], yy[2]); yy[2] = __fmaf_rn(b1, S[h][0], yy[2]);
            yy[3] = __fmaf_rn(s1, P[h][3], yy[3]); yy[3] = __fmaf_rn(b1, S[h][1], yy[3]);
          }
        }
      }
    }
  }

  // ---- partials: warps in order, then cluster ranks in order
#pragma unroll
  for (int i = 0; i < NV; ++i) red[warp][i][lane] = y[i];
  __syncthreads();
  for (int v = threadIdx.x; v < NV * 32; v += blockDim.x) {
    const int i = v >> 5, ln = v & 31;
    float acc = red[0][i][ln];
    for (int w = 1; w < nwarps; ++w) acc = __fadd_rn(acc, red[w][i][ln]);
    csum[i][ln] = acc;
  }
  cluster.sync();
  if (rank == 0) {
    constexpr int NO = NB * 4;  // outputs per lane per matrix
    for (int v = threadIdx.x; v < NO * 32; v += blockDim.x) {
      const int i = v >> 5, ln = v & 31;
      float acc[NMAT];
#pragma unroll
      for (int t = 0; t < NMAT; ++t) acc[t] = csum[t * NO + i][ln];
      for (int r = 1; r < p.cs; ++r) {
        const float *rs = cluster.map_shared_rank(&csum[0][0], r);
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
  cluster.sync();
}

template <int BITS, int NB, int MODE>
static cudaError_t launch_t(const MvParams &p, int nwarps, int tiles, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * p.cs));
  cfg.blockDim = dim3((unsigned)(nwarps * 32));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
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

void mv_geometry(int k, int &groups, int &slices, int &nwarps, int &cs) {
  groups = k / kGroup;
  slices = (groups + kMvGpw - 1) / kMvGpw;
  nwarps = slices < kMvMaxWarps ? slices : kMvMaxWarps;
  int need = (slices + nwarps - 1) / nwarps;
  cs = need < kMvMaxCluster ? need : kMvMaxCluster;
}

cudaError_t launch_mv(MvParams &p, int mode, int bits, int tiles, cudaStream_t st) {
  int nwarps;
  mv_geometry(p.k, p.groups, p.slices, nwarps, p.cs);
  p.wpr = p.k * bits / 32;
  switch (mode) {
    case kMvFfn: return launch_mode<kMvFfn>(p, bits, nwarps, tiles, st);
    case kMvAttn: return launch_mode<kMvAttn>(p, bits, nwarps, tiles, st);
    default: return launch_mode<kMvPlain>(p, bits, nwarps, tiles, st);
  }
}

}  // namespace qlk
