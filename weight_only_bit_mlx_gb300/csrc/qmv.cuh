// qmv.cuh - launch interface of the decode matvec kernels (host side).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace qlk {

constexpr int kMvGpw = 2;         // 64-wide groups per warp slice
constexpr int kMvMaxWarps = 8;    // warps (k-slices) per CTA
constexpr int kMvMaxCluster = 8;  // CTAs per cluster along k

enum { kMvPlain = 0, kMvFfn = 1, kMvAttn = 2 };

struct MvMat {
  const uint32_t *wq;
  const uint16_t *s;
  const uint16_t *b;
  void *out;     // float [rows, ldo] (plain, attn) or bf16 bits [rows, ldo] (ffn, in m[0])
  int64_t ldo;
  int n;
};

struct MvParams {
  MvMat m[4];        // plain: m[0]; ffn: m[0] = w1, m[1] = w3; attn: q, k, v, gate
  int tile_end[4];   // attn: cumulative 16-row tile counts of m[0..3]
  const uint16_t *x;
  int64_t ldx;
  int rows;
  int k;
  // filled by launch_mv from k and bits
  int groups;
  int wpr;
  int slices;
  int cs;
};

// k-decomposition used by every decode launch (function of k only)
void mv_geometry(int k, int &groups, int &slices, int &nwarps, int &cs);

// Enqueue one decode launch over `tiles` 16-row tiles.
cudaError_t launch_mv(MvParams &p, int mode, int bits, int tiles, cudaStream_t st);

}  // namespace qlk
