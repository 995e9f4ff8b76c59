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
//     CTAs of a cluster split k into spans;
//   * compute warp w owns kGpw consecutive groups of the span; at kernel start it copies
//     exactly those bytes of every row of the tile from HBM into shared memory with
//     16-byte cp.async pieces (a warp instruction reads four whole 128-byte lines), and
//     waits only for its own copies.  Measured against one bulk copy (cp.async.bulk)
//     per row, all issued by warp 0 (32 per CTA in the fused FFN): 0.269 against
//     0.283-0.287 ms per 4-bit R = 1 decode pass;
//   * scales and biases are read by the compute threads (16-byte vectors of 8 groups
//     when the rows allow it) before the dependency wait; activations (the only input
//     a preceding kernel may write) are loaded after griddepcontrol.wait, so with
//     programmatic dependent launch the weight stream of this kernel overlaps the
//     tail of the previous one;
//   * compute warp w owns kGpw consecutive groups of every chunk.  Per group the
//     codes are converted exactly to bf16 and multiplied on the tensor cores with
//     mma.sync m16n8k16 (rows of W as A, activation rows as B), a fresh fp32
//     accumulator per group, and the affine step follows in group order:
//       P'_g = sum_{j in g} (q_j - z) x_j;   y = fma(s, P'_g, y); y = fma(b + s*z, S_g, y)
//     with the group's zero point z = round(-b/s) in the code range (the codes are
//     centred as they are converted, at no extra instruction; see group_factors)
//     and S_g = sum_{j in g} x_j from the same tensor-core path (A = 1), once per
//     activation row and group;
//   * warp partials are added in warp order through shared memory, CTA partials in
//     rank order through distributed shared memory.  No atomics, no scratch memory.
// The tensor core computes every output column (activation row) from that column's
// data alone, so a row's result does not depend on how many rows share the call.
#include <cooperative_groups.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "qmv.cuh"
#include "qmv_core.cuh"
#include "sync.cuh"

namespace cg = cooperative_groups;

namespace qlk {

// per-tile sums of squares and the finished-tile counter of kMvResid launches (one per
// device that loads the library; the counter is back at zero after every launch)
__device__ float g_resid_part[kMvResidMaxTiles * 16];
__device__ unsigned g_resid_counter = 0;

// Device addresses of the two arrays, looked up once per device (with that device
// current) and cached: in host code the arrays' names are only host-side stand-ins.
// The first post-add / next-norm call on a device does the lookup, so it should come
// before any stream capture.
static std::mutex g_resid_mu;
static float *g_resid_part_addr[64];
static unsigned *g_resid_counter_addr[64];

int mv_resid_scratch(float **part, unsigned **counter) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::lock_guard<std::mutex> lk(g_resid_mu);
  if (g_resid_part_addr[dev] == nullptr) {
    void *a = nullptr, *b = nullptr;
    if (cudaGetSymbolAddress(&a, g_resid_part) != cudaSuccess ||
        cudaGetSymbolAddress(&b, g_resid_counter) != cudaSuccess) {
      (void)cudaGetLastError();
      return -1;
    }
    g_resid_counter_addr[dev] = static_cast<unsigned *>(b);
    g_resid_part_addr[dev] = static_cast<float *>(a);
  }
  *part = g_resid_part_addr[dev];
  *counter = g_resid_counter_addr[dev];
  return 0;
}

int mv_resid_counter_reset() {
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_resid_counter, &zero, sizeof(zero)) == cudaSuccess ? 0 : -1;
}

int mv_span_g(int bits) { return bits == 4 ? span_g<4>() : (bits == 6 ? span_g<6>() : span_g<8>()); }

// Shared-memory layout of one CTA (dynamic, 128-byte aligned):
//   wsm [NMAT][16][wpitch]             weight rows of the span (each warp copies its groups);
//                                      after the last group it holds the warp partials
//                                      red[kMvWarps][NV][32] (without a cluster they are
//                                      added in warp order where the outputs are stored)
//   sbf [NMAT][span][16] float4        per (group, row): group_factors (scale, centred
//                                      bias, offset constant)
//   cpart[cs][NV][32] fp32             with a cluster of cs > 1 CTAs: every rank's CTA
//                                      partial (only rank 0's copy is read); a region of
//                                      its own, since other ranks write it while this
//                                      CTA may still be reading its weights
// Activations never pass through shared memory: each lane loads the 16-byte pieces
// its MMA fragments take straight from global memory (L1/L2).
template <int BITS, int NB, int MODE> struct MvLayout {
  static constexpr int NMAT = (MODE == kMvFfn) ? 2 : 1;
  static constexpr int NV = NMAT * NB * 4;
  static constexpr int kW = 0;
  static constexpr int kRed = 0;                                // aliases wsm
  static constexpr int kCsum = kRed + kMvWarps * NV * 32 * 4;   // aliases wsm
  static constexpr int kPartBytes = kCsum + NV * 32 * 4;
  static constexpr int kWBytes = NMAT * 16 * wpitch<BITS>() > kPartBytes ? NMAT * 16 * wpitch<BITS>() : kPartBytes;
  static constexpr int kSbf = kWBytes;
  static constexpr int kCpart = (kSbf + NMAT * span_g<BITS>() * 16 * 16 + 15) / 16 * 16;
  static constexpr int kBytes = kCpart;  // without a cluster
  static int bytes(int cs) { return cs > 1 ? kCpart + cs * NV * 32 * 4 : kBytes; }
  static int max_bytes() { return bytes(kMvMaxCluster); }
};

// Four CTAs of 256 threads per SM: 64 registers a thread, and every variant (one or
// two row blocks) equally resident.  Measured on the decode pass: 3 per SM (80
// registers) and 5 per SM (48 registers, spills) are both slower.
constexpr int kMvCtasPerSm = 4;

// The post-add / next-norm epilogue after the tile's residual rows are stored
// (TensorFold PR #1514, "What changes": post-add/next-norm fusion): the tile's sum of
// squares per activation row (its 16 channels in order) goes to its slot; the CTA that
// finishes last (a device counter) adds the slots in tile order, and normalises every
// channel of every row from the stored residual: out = bf16(r' / sqrt(mean r'^2 + eps)
// * gamma).  No CTA waits for another; every order is fixed, so the result is
// deterministic and each activation row's depends on that row alone.
template <int NB>
__device__ __forceinline__ void resid_norm_tail(const MvParams &p, int tile, float (*s_sq)[17]) {
  __shared__ float s_wsum[kMvWarps][8 * NB];
  __shared__ float s_rstd[8 * NB];
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = p.m[0].n;
  __syncthreads();  // s_sq complete
  if (tid < p.rows) {
    float sacc = 0.0f;
#pragma unroll
    for (int c = 0; c < 16; ++c) sacc = __fadd_rn(sacc, s_sq[tid][c]);
    p.part[(size_t)tile * 16 + tid] = sacc;
  }
  __threadfence();  // this tile's residual rows and slot are visible device-wide
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(p.counter, 1u) == (unsigned)(p.ntiles - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // sums of squares per activation row: tiles strided over the threads, then each
  // warp's butterfly, then the warps in order
  float a[8 * NB];
#pragma unroll
  for (int r = 0; r < 8 * NB; ++r) a[r] = 0.0f;
  for (int tl = tid; tl < p.ntiles; tl += kMvThreads) {
#pragma unroll
    for (int r = 0; r < 8 * NB; ++r)
      if (r < p.rows) a[r] = __fadd_rn(a[r], __ldcg(p.part + (size_t)tl * 16 + r));
  }
#pragma unroll
  for (int r = 0; r < 8 * NB; ++r) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a[r] = __fadd_rn(a[r], __shfl_xor_sync(0xffffffffu, a[r], o));
    if (lane == 0) s_wsum[warp][r] = a[r];
  }
  __syncthreads();
  if (tid < p.rows) {
    float tot = s_wsum[0][tid];
    for (int w = 1; w < kMvWarps; ++w) tot = __fadd_rn(tot, s_wsum[w][tid]);
    s_rstd[tid] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)n), p.eps)));
  }
  __syncthreads();
  const bool vec = (n % 8) == 0 && (p.ldr % 8) == 0 && (p.ldn % 8) == 0 &&
                   ((reinterpret_cast<uintptr_t>(p.resid) | reinterpret_cast<uintptr_t>(p.nout) |
                     reinterpret_cast<uintptr_t>(p.gamma)) & 15) == 0;
  if (vec) {
    // 8 channels per 16-byte access, several accesses of each thread in flight
    const int nch = n >> 3, total = p.rows * nch;
#pragma unroll 4
    for (int c = tid; c < total; c += kMvThreads) {
      const int xr = c / nch, i = (c - xr * nch) * 8;
      const uint4 rv = __ldcg(reinterpret_cast<const uint4 *>(p.resid + (size_t)xr * p.ldr + i));
      const uint4 gv = __ldg(reinterpret_cast<const uint4 *>(p.gamma + i));
      const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
      const float rs = s_rstd[xr];
      uint32_t ow[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint16_t lo = f32_to_bf16_rn(__fmul_rn(__fmul_rn(bf16_to_f32(rw[q] & 0xFFFFu), rs), bf16_to_f32(gw[q] & 0xFFFFu)));
        const uint16_t hi = f32_to_bf16_rn(__fmul_rn(__fmul_rn(bf16_to_f32(rw[q] >> 16), rs), bf16_to_f32(gw[q] >> 16)));
        ow[q] = (uint32_t)lo | ((uint32_t)hi << 16);
      }
      *reinterpret_cast<uint4 *>(p.nout + (size_t)xr * p.ldn + i) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    }
  } else {
#pragma unroll 4
    for (int e = tid; e < p.rows * n; e += kMvThreads) {
      const int xr = e / n, i = e - xr * n;
      const float v = bf16_to_f32(__ldcg(p.resid + (size_t)xr * p.ldr + i));
      p.nout[(size_t)xr * p.ldn + i] = f32_to_bf16_rn(__fmul_rn(__fmul_rn(v, s_rstd[xr]), bf16_to_f32(p.gamma[i])));
    }
  }
  if (tid == 0) atomicExch(p.counter, 0u);  // ready for the next launch (stream order)
}

template <int BITS, int NB, int MODE>
__global__ void __launch_bounds__(kMvThreads, kMvCtasPerSm) qmv_kernel(const __grid_constant__ MvParams p) {
  using Lay = MvLayout<BITS, NB, MODE>;
  constexpr int NMAT = Lay::NMAT;
  constexpr int NV = Lay::NV;
  constexpr int LW = Geo<BITS>::kLw;
  constexpr int GPW = Geo<BITS>::kGpw;
  constexpr int GPC = gpc<BITS>();
  constexpr int SPAN = span_g<BITS>();
  constexpr int GB = gbytes<BITS>();
  constexpr int WP = wpitch<BITS>();
  constexpr bool kPair4 = BITS == 4;  // 4-bit codes paired (t, t+4): activations in that order
  extern __shared__ __align__(128) uint8_t smem[];
  float4 *sbf = reinterpret_cast<float4 *>(smem + Lay::kSbf);
  float *red = reinterpret_cast<float *>(smem + Lay::kRed);
  float *csum = reinterpret_cast<float *>(smem + (p.cs > 1 ? Lay::kCpart : Lay::kCsum));
  uint8_t *wsm = smem + Lay::kW;

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = p.cs > 1 ? (int)cluster.block_rank() : 0;
  const int tile_g = blockIdx.x / p.cs;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g4 = lane >> 2, c = lane & 3;

  int mi = 0, tile = tile_g;
  if constexpr (MODE == kMvAttn) {
    while (mi < 3 && tile_g >= p.tile_end[mi]) ++mi;
    tile = tile_g - (mi ? p.tile_end[mi - 1] : 0);
  }
  const int n = p.m[mi].n;
  const size_t row_bytes = (size_t)p.groups * GB;

  // this CTA's k-span: groups [gs0, gs1), in spans of SPAN groups
  const int gs0 = rank * p.span_g, gs1 = min(p.groups, gs0 + p.span_g);

  float y[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) y[i] = 0.0f;

  for (int ch0 = gs0; ch0 < gs1; ch0 += SPAN) {
    const int ch1 = min(gs1, ch0 + SPAN);
    const int ng = ch1 - ch0;
    {
      // ---- every warp starts the copies of the weight bytes it will read: its groups of
      //      the span, every row of the tile, as 16-byte pieces (consecutive lanes on
      //      consecutive pieces of a row, so a warp instruction reads whole 128-byte
      //      lines); no other warp reads them, so the warp waits only for its own
      static_assert(kNch == 1, "one chunk per span");
      const int gw0 = ch0 + warp * GPW;
      const int gcnt = max(0, min(GPW, ch1 - gw0));
      auto piece = [&](int rr, int pc) {
        const int row = tile * 16 + (rr & 15);
        if (row < n)
          cp_async16(wsm + rr * WP + (gw0 - ch0) * GB + pc * 16,
                     reinterpret_cast<const uint8_t *>(p.m[mi + (rr >> 4)].wq) + (size_t)row * row_bytes +
                         (size_t)gw0 * GB + pc * 16);
      };
      constexpr int PC = GPW * GB / 16;  // pieces per row with all of the warp's groups
      if (gcnt == GPW && (PC & (PC - 1)) == 0) {
        // (4 and 8 bits) a power-of-two count per row: unrolled, no division (6 bits keeps
        // the loop below: unrolled, its FFN variant spills and the pass measured slower)
        static_assert((NMAT * 16 * PC) % 32 == 0, "whole warp instructions");
#pragma unroll
        for (int i = 0; i < NMAT * 16 * PC / 32; ++i) {
          const int e = lane + 32 * i;
          piece(e / PC, e % PC);
        }
      } else {
        const int pieces = gcnt * (GB / 16);  // per row
        for (int e = lane; e < NMAT * 16 * pieces; e += 32) {
          const int rr = e / pieces;
          piece(rr, e - rr * pieces);
        }
      }
      cp_async_commit();
    }
    {
      // ---- every warp computes
      const int tid = threadIdx.x;  // 0 .. kMvComputeThreads-1
      // Scales and biases of the span (not written by a preceding kernel, so read
      // before the dependency wait) -> per-group factors (group_factors).  16-byte vectors of 8
      // groups when the rows allow it, else one value at a time.
      if (p.sb_bulk) {
        const int v8 = ng >> 3;  // vectors per row
        for (int e = tid; e < NMAT * 16 * v8; e += kMvComputeThreads) {
          const int t = e / (16 * v8), rr = (e / v8) % 16, v = e % v8;
          const int row = tile * 16 + rr;
          uint4 sv = make_uint4(0, 0, 0, 0), bv = make_uint4(0, 0, 0, 0);
          if (row < n) {
            const size_t off = (size_t)row * p.groups + ch0 + 8 * v;
            sv = ldg_v4(p.m[mi + t].s + off);
            bv = ldg_v4(p.m[mi + t].b + off);
          }
          const uint32_t ss[4] = {sv.x, sv.y, sv.z, sv.w}, bb[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
          for (int q2 = 0; q2 < 8; ++q2) {
            const float s1 = bf16_to_f32((ss[q2 >> 1] >> (16 * (q2 & 1))) & 0xFFFFu);
            const float b1 = bf16_to_f32((bb[q2 >> 1] >> (16 * (q2 & 1))) & 0xFFFFu);
            sbf[(t * SPAN + 8 * v + q2) * 16 + rr] = group_factors<BITS>(s1, b1);
          }
        }
      } else {
        for (int e = tid; e < NMAT * 16 * ng; e += kMvComputeThreads) {
          const int t = e / (16 * ng), rr = (e / ng) % 16, gg = e % ng;
          const int row = tile * 16 + rr;
          float s1 = 0.0f, b1 = 0.0f;
          if (row < n) {
            const size_t off = (size_t)row * p.groups + ch0 + gg;
            s1 = bf16_to_f32(ldg_u16(p.m[mi + t].s + off));
            b1 = bf16_to_f32(ldg_u16(p.m[mi + t].b + off));
          }
          sbf[(t * SPAN + gg) * 16 + rr] = group_factors<BITS>(s1, b1);
        }
      }
      // Activations: a preceding kernel may write them, so they are read only after
      // the programmatic-dependency wait.
      if (ch0 == gs0) {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        asm volatile("griddepcontrol.wait;" ::: "memory");
      }
      named_bar_sync(kBarCompute, kMvComputeThreads);  // group factors visible
      bool xv[NB];
#pragma unroll
      for (int h = 0; h < NB; ++h) xv[h] = (8 * h + g4) < p.rows;
      for (int cc = 0; cc < kNch; ++cc) {
        const int ga = ch0 + cc * GPC;
        if (ga >= ch1) break;
        const int gw0 = ga + warp * GPW;  // this warp's groups of the chunk
        const int gcnt = max(0, min(GPW, ch1 - gw0));
        // the first group's activations are in flight while the chunk's weights land
        uint4 Xa[NB], Xb[NB];
#pragma unroll
        for (int h = 0; h < NB; ++h) {
          Xa[h] = make_uint4(0, 0, 0, 0);
          Xb[h] = make_uint4(0, 0, 0, 0);
          if (xv[h] && gcnt > 0)
            load_x_frag<kPair4>(p.x + (size_t)(8 * h + g4) * p.ldx + (size_t)gw0 * 64 + 16 * c, Xa[h], Xb[h]);
        }
        cp_async_wait_all();  // this warp's weight bytes have landed
        __syncwarp();
#pragma unroll
        for (int gi = 0; gi < GPW; ++gi) {
          if (gi < gcnt) {
            const int gl = gw0 + gi - ch0;  // group index within the span
            uint4 X0[NB], X1[NB];
#pragma unroll
            for (int h = 0; h < NB; ++h) {
              if (NB == 1 || gi == 0) {
                // one activation row block: the next group's fragments are loaded a
                // group ahead; with two blocks they are loaded when used (registers)
                X0[h] = Xa[h];
                X1[h] = Xb[h];
                if (NB == 1 && xv[h] && gi + 1 < gcnt)
                  load_x_frag<kPair4>(p.x + (size_t)(8 * h + g4) * p.ldx + (size_t)(gw0 + gi + 1) * 64 + 16 * c, Xa[h],
                                    Xb[h]);
              } else if (xv[h]) {
                load_x_frag<kPair4>(p.x + (size_t)(8 * h + g4) * p.ldx + (size_t)(gw0 + gi) * 64 + 16 * c, X0[h], X1[h]);
              } else {
                X0[h] = make_uint4(0, 0, 0, 0);
                X1[h] = make_uint4(0, 0, 0, 0);
              }
            }
            mv_group<BITS, NB, NMAT>(wsm + gl * GB + c * 4 * LW, WP, sbf + gl * 16, SPAN * 16, X0, X1, g4, y);
          }
        }
      }
    }
    if (ch1 < gs1) __syncthreads();  // the span's buffers are fully read before the next span refills them
  }
  cp_async_wait_all();  // (a warp with no groups started no copies)

  // ---- partials: warps in order, then cluster ranks in order.  The partials reuse
  //      the weight area, so every compute warp is past its last group first.  In a
  //      cluster each rank writes its CTA partial into slot `rank` of rank 0's cpart
  //      (distributed shared memory); after one cluster barrier rank 0 adds the slots
  //      in rank order and the other ranks may exit (nobody reads their shared memory).
  {
    named_bar_sync(kBarCompute, kMvComputeThreads);
#pragma unroll
    for (int i = 0; i < NV; ++i) red[(warp * NV + i) * 32 + lane] = y[i];
    named_bar_sync(kBarCompute, kMvComputeThreads);
    if (p.cs > 1) {
      float *dst = cluster.map_shared_rank(csum, 0) + rank * NV * 32;
      for (int v = threadIdx.x; v < NV * 32; v += kMvComputeThreads) {
        const int i = v >> 5, ln = v & 31;
        float acc = red[i * 32 + ln];
#pragma unroll
        for (int w = 1; w < kMvWarps; ++w) acc = __fadd_rn(acc, red[(w * NV + i) * 32 + ln]);
        dst[i * 32 + ln] = acc;
      }
    }
  }
  // without a cluster the warp partials are added in warp order right below, where
  // they are stored (the same order; the barrier above made them visible)
  if (p.cs > 1) cluster.sync();
  if (rank == 0) {
    constexpr int NO = NB * 4;  // outputs per lane per matrix
    __shared__ float s_sq[MODE == kMvResid ? 8 * NB : 1][17];  // [activation row][channel of the tile]
    for (int v = threadIdx.x; v < NO * 32; v += kMvThreads) {
      const int i = v >> 5, ln = v & 31;
      float acc[NMAT];
      if (p.cs > 1) {
#pragma unroll
        for (int t = 0; t < NMAT; ++t) acc[t] = csum[(t * NO + i) * 32 + ln];
        for (int r = 1; r < p.cs; ++r) {
#pragma unroll
          for (int t = 0; t < NMAT; ++t) acc[t] = __fadd_rn(acc[t], csum[r * NV * 32 + (t * NO + i) * 32 + ln]);
        }
      } else {
#pragma unroll
        for (int t = 0; t < NMAT; ++t) {
          acc[t] = red[(t * NO + i) * 32 + ln];
#pragma unroll
          for (int w = 1; w < kMvWarps; ++w) acc[t] = __fadd_rn(acc[t], red[(w * NV + t * NO + i) * 32 + ln]);
        }
      }
      // value i of lane ln: half h = i / 4, element e = i % 4
      const int h = i >> 2, e = i & 3;
      const int row = tile * 16 + (ln >> 2) + ((e & 2) ? 8 : 0);
      const int xr = 8 * h + 2 * (ln & 3) + (e & 1);
      if constexpr (MODE == kMvResid) {
        // post-add: the stored residual r' = bf16(r + y) and its square
        float sq = 0.0f;
        if (row < n && xr < p.rows) {
          uint16_t *rp = p.resid + (size_t)xr * p.ldr + row;
          const uint16_t nb = f32_to_bf16_rn(__fadd_rn(bf16_to_f32(*rp), acc[0]));
          *rp = nb;
          const float v = bf16_to_f32(nb);
          sq = __fmul_rn(v, v);
        }
        s_sq[xr][(ln >> 2) + ((e & 2) ? 8 : 0)] = sq;
      } else if (row < n && xr < p.rows) {
        const MvMat &M = p.m[mi];
        if constexpr (MODE == kMvFfn) {
          static_cast<uint16_t *>(M.out)[(size_t)xr * M.ldo + row] = swiglu_bf16(acc[0], acc[1]);
        } else {
          static_cast<float *>(M.out)[(size_t)xr * M.ldo + row] = acc[0];
        }
      }
    }
    if constexpr (MODE == kMvResid) resid_norm_tail<NB>(p, tile, s_sq);
  }
}

template <int BITS, int NB, int MODE>
static cudaError_t launch_t(const MvParams &p, int tiles, cudaStream_t st) {
  using Lay = MvLayout<BITS, NB, MODE>;
  static std::atomic<bool> attr_done[64];  // per device; setting the attributes twice is harmless
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev].load(std::memory_order_relaxed)) {
    cudaError_t e = cudaFuncSetAttribute(qmv_kernel<BITS, NB, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay::max_bytes());
    if (e != cudaSuccess) return e;
    // every decode kernel asks for the largest shared-memory carveout, so CTAs of
    // consecutive launches (programmatic dependent launch) can share an SM
    e = cudaFuncSetAttribute(qmv_kernel<BITS, NB, MODE>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_done[dev].store(true, std::memory_order_relaxed);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * p.cs));
  cfg.blockDim = dim3((unsigned)kMvThreads);
  cfg.dynamicSmemBytes = (size_t)Lay::bytes(p.cs);
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
static cudaError_t launch_mode(const MvParams &p, int bits, int tiles, cudaStream_t st) {
  const bool two = p.rows > 8;
  switch (bits) {
    case 4: return two ? launch_t<4, 2, MODE>(p, tiles, st) : launch_t<4, 1, MODE>(p, tiles, st);
    case 6: return two ? launch_t<6, 2, MODE>(p, tiles, st) : launch_t<6, 1, MODE>(p, tiles, st);
    default: return two ? launch_t<8, 2, MODE>(p, tiles, st) : launch_t<8, 1, MODE>(p, tiles, st);
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
  // scale/bias rows of a span can be read as 16-byte vectors when every vector starts on
  // a 16-byte boundary: groups and the per-CTA span multiples of 8, pointers aligned
  const int nm = mode == kMvAttn ? 4 : (mode == kMvFfn ? 2 : 1);
  bool sb = (p.groups % 8) == 0 && (p.span_g % 8) == 0;
  for (int i = 0; i < nm; ++i)
    sb = sb && (reinterpret_cast<uintptr_t>(p.m[i].s) % 16) == 0 && (reinterpret_cast<uintptr_t>(p.m[i].b) % 16) == 0;
  p.sb_bulk = sb ? 1 : 0;
  switch (mode) {
    case kMvFfn: return launch_mode<kMvFfn>(p, bits, tiles, st);
    case kMvAttn: return launch_mode<kMvAttn>(p, bits, tiles, st);
    case kMvResid: return launch_mode<kMvResid>(p, bits, tiles, st);
    default: return launch_mode<kMvPlain>(p, bits, tiles, st);
  }
}

}  // namespace qlk
