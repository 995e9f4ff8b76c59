// qmv.cuh - launch interface of the decode matvec kernels (host side).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace qlk {

// warps per CTA, each owning a slice of the CTA's k-span (4 measured slower on the decode pass)
constexpr int kMvWarps = 8;
constexpr int kMvMaxCluster = 8;  // CTAs per cluster along k

enum { kMvPlain = 0, kMvFfn = 1, kMvAttn = 2, kMvResid = 3 };

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
  int sb_bulk;           // scales/biases rows are 16-byte aligned: read as 16-byte vectors
  // kMvResid: the post-add / next-norm epilogue (one weight, like kMvPlain)
  uint16_t *resid;       // bf16 [rows, ldr], read and overwritten with bf16(resid + y)
  int64_t ldr;
  const uint16_t *gamma; // bf16 [n]
  float eps;
  uint16_t *nout;        // bf16 [rows, ldn]: the normalised stored residual times gamma
  int64_t ldn;
  float *part;           // [tiles][16] per-tile sums of squares (library scratch)
  unsigned *counter;     // tiles finished (library scratch, zero between calls)
  int ntiles;            // 16-row tiles of the launch
  // filled by launch_mv from k and bits
  int groups;
  int wpr;
  int span_g;            // groups per CTA (processed in chunks of the per-bits span)
  int cs;                // CTAs per cluster along k
};

// groups per k-span of one CTA for the given code width
int mv_span_g(int bits);

// k-decomposition used by every decode launch (a function of k and bits only)
void mv_geometry(int k, int bits, int &groups, int &span_g, int &nwarps, int &cs);

// Maximum 16-row tiles of a kMvResid launch (n <= 65536) and the device addresses of its
// per-tile partial sums and finished-tile counter (current device); reset the counter.
constexpr int kMvResidMaxTiles = 4096;
int mv_resid_scratch(float **part, unsigned **counter);
int mv_resid_counter_reset();

// Enqueue one decode launch over `tiles` 16-row tiles.
cudaError_t launch_mv(MvParams &p, int mode, int bits, int tiles, cudaStream_t st);

}  // namespace qlk
