// qmv.cu - decode matvecs over MLX affine 4/6/8-bit group-64 weights (sm_103a).
//
// One kernel template serves qlinear_mv / qlinear_mv_rows (one weight), the fused
// w1 + w3 + SwiGLU step (two weights, bf16 output), the fused q/k/v/gate step (four
// weights, one launch) and the matvec with the post-add / next-norm epilogue.
// TensorFold PR #1696 (later revision), "What it adds": N-row matvecs summing each
// row as the one-row kernels do; decode fuses w1 + w3 + SwiGLU and the four attention
// matvecs.  PR #1514, "What changes": post-add/next-norm fusion.
//
// Data movement: one CTA per SM.  CTA c owns a contiguous range of 16-row tiles (both
// w1 and w3 rows of a tile in the fused FFN); a tile's k-range is cut into spans of 32
// groups (4-bit) or 16 groups (6/8-bit), and every (tile, span) is one slot of a ring
// in shared memory: the weight rows, and with them the span's scales and biases, each
// arrive by one bulk copy (cp.async.bulk) per row straight from HBM.  Warp 0 fills the
// whole ring at kernel start, before the programmatic-dependency wait, and refills a
// slot as soon as every warp is done with it, so the weight stream of a launch runs
// while the previous launch still computes.  The CTA is small enough (at most 140 KB
// of shared memory for two weights, 80 KB for one; 256 threads) that the next launch's
// CTA fits beside it on the same SM and starts streaming its own weights in turn.
// Activations - the only input a preceding kernel writes - are read after
// griddepcontrol.wait, straight into the registers of the MMA fragments.
//
// Arithmetic (qmv_core.cuh): warp w owns groups w*gpw .. w*gpw + gpw - 1 of every span
// (gpw = 4 for 4-bit, 2 otherwise).  Per group the codes are converted exactly to bf16,
// centred on the group's zero point z, and multiplied on the tensor cores with
// mma.sync m16n8k16 (rows of W as A, activation rows as B), a fresh fp32 accumulator
// per group; the affine step follows in group order:
//   P'_g = sum_{j in g} (q_j - z) x_j;   y = fma(s, P'_g, y); y = fma(b + s*z, S_g, y)
// with S_g = sum_{j in g} x_j from the same tensor-core path (A = 1).  A warp's partial
// runs over its groups of every span of the tile in k order; the warps' partials are
// then added in warp order.  This order is a function of k and bits only - never of
// the number of activation rows, of n, of the tile-to-CTA assignment or of fused vs
// unfused - and the tensor core computes every output column (activation row) from
// that column's data alone, so a row's result does not depend on how many rows share
// the call.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "qmv.cuh"
#include "qmv_core.cuh"
#include "sync.cuh"

namespace qlk {

// per-tile sums of squares and the finished-CTA counter of kMvResid launches (one per
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

// Shared-memory layout of one CTA (dynamic):
//   ring[NS] slots, each: weights [NMAT][16 rows][wpitch] (one bulk copy per row),
//            scales [NMAT][16][span] bf16, biases [NMAT][16][span] bf16
//   red[2][kMvWarps][NV][32] fp32     warp partials of a tile (two tiles in flight)
//   fac[kMvWarps][gpw][NMAT][16] float4  each warp's group factors of the current slot
//   full[NS]                          mbarrier per ring slot (bulk-copy bytes)
template <int BITS, int NB, int MODE> struct MvLayout {
  static constexpr int NMAT = (MODE == kMvFfn) ? 2 : 1;
  static constexpr int NV = NMAT * NB * 4;  // accumulators per lane
  static constexpr int SPAN = span_g<BITS>();
  static constexpr int kWBytes = NMAT * 16 * wpitch<BITS>();
  static constexpr int kSBRow = SPAN * 2;   // bytes of one row's scales (or biases) in a slot
  static constexpr int kSlot = kWBytes + 2 * NMAT * 16 * kSBRow;
  static constexpr int kRed = kMvWarps * NV * 32 * 4;
  static constexpr int kFac = kMvWarps * Geo<BITS>::kGpw * NMAT * 16 * 16;
  // two weights (the fused FFN) may take 148 KB, one weight 76 KB: any two consecutive
  // launches of a decode layer fit one SM together
  static constexpr int kBudget = (NMAT == 2 ? 148 : 76) * 1024;
  static constexpr int NS = (kBudget - 2 * kRed - kFac - 256) / kSlot;
  static constexpr int kOffRed = NS * kSlot;
  static constexpr int kOffFac = kOffRed + 2 * kRed;
  static constexpr int kOffBar = kOffFac + kFac;
  static constexpr int kBytes = kOffBar + NS * 8;
  static_assert(NS >= 2, "at least two ring slots");
  static_assert(kBytes <= kBudget, "shared-memory budget");
};

// The post-add / next-norm epilogue after the last CTA has stored its tiles' residual
// rows and their sums of squares (TensorFold PR #1514, "What changes": post-add/next-
// norm fusion): the CTA that finishes last (a device counter) adds the per-tile slots in
// tile order and normalises every channel of every row from the stored residual:
// out = bf16(r' / sqrt(mean r'^2 + eps) * gamma).  No CTA waits for another; every order
// is fixed, so the result is deterministic and each activation row's depends on that
// row alone.
template <int NB>
__device__ __forceinline__ void resid_norm_tail(const MvParams &p) {
  __shared__ float s_wsum[kMvWarps][8 * NB];
  __shared__ float s_rstd[8 * NB];
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = p.m[0].n;
  __threadfence();  // this CTA's residual rows and slots are visible device-wide
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(p.counter, 1u) == gridDim.x - 1;
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
__global__ void __launch_bounds__(kMvThreads, 2) qmv_kernel(const __grid_constant__ MvParams p) {
  using Lay = MvLayout<BITS, NB, MODE>;
  constexpr int NMAT = Lay::NMAT;
  constexpr int NV = Lay::NV;
  constexpr int NO = NB * 4;  // outputs per lane per matrix
  constexpr int NS = Lay::NS;
  constexpr int SPAN = Lay::SPAN;
  constexpr int LW = Geo<BITS>::kLw;
  constexpr int GPW = Geo<BITS>::kGpw;
  constexpr int GB = gbytes<BITS>();
  constexpr int WP = wpitch<BITS>();
  constexpr bool kPair4 = BITS == 4;  // 4-bit codes paired (t, t+4): activations in that order
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lay::kOffBar);
  float *red = reinterpret_cast<float *>(smem + Lay::kOffRed);
  float4 *fac = reinterpret_cast<float4 *>(smem + Lay::kOffFac);
  __shared__ int s_abort;
  __shared__ float s_sq[MODE == kMvResid ? 8 * NB : 1][17];  // [activation row][channel of the tile]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g4 = lane >> 2, c = lane & 3;
  const int G = p.groups, nspan = p.nspan;
  const int t0 = (int)(((long long)blockIdx.x * p.ntiles) / gridDim.x);
  const int t1 = (int)(((long long)(blockIdx.x + 1) * p.ntiles) / gridDim.x);
  const int J = (t1 - t0) * nspan;  // ring slots this CTA consumes
  const size_t row_bytes = (size_t)G * GB;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();

  // matrix and 16-row tile within it of a tile index of the launch
  auto tile_mat = [&](int t, int &mi, int &lt) {
    mi = 0;
    if constexpr (MODE == kMvAttn) {
      while (mi < 3 && t >= p.tile_end[mi]) ++mi;
    }
    lt = t - (mi ? p.tile_end[mi - 1] : 0);
  };

  // warp 0: one bulk copy per weight row of slot j (lane l: matrix l / 16, row l % 16),
  // and of its scale and bias rows, into ring buffer j % NS
  int issued = 0;  // slots issued so far (warp 0)
  auto issue = [&](int j) {
    const int t = t0 + j / nspan, sp = j - (j / nspan) * nspan;
    int mi, lt;
    tile_mat(t, mi, lt);
    const int g0 = sp * SPAN, ng = min(SPAN, G - g0);
    const int mt = lane >> 4, r = lane & 15;
    const int row = lt * 16 + r;
    const bool mine = mt < NMAT && row < p.m[mi + (mt < NMAT ? mt : 0)].n;
    uint32_t bytes = mine ? (uint32_t)(ng * GB + (p.sb_bulk ? 4 * ng : 0)) : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
    uint64_t *bar = &full[j % NS];
    uint8_t *slot = smem + (j % NS) * Lay::kSlot;
    if (lane == 0) mbar_arrive_expect_tx(bar, bytes);
    __syncwarp();
    if (mine) {
      const MvMat &M = p.m[mi + mt];
      bulk_g2s(slot + (mt * 16 + r) * WP, reinterpret_cast<const uint8_t *>(M.wq) + (size_t)row * row_bytes +
                                              (size_t)g0 * GB,
               (uint32_t)(ng * GB), bar);
      if (p.sb_bulk) {
        uint8_t *sb = slot + Lay::kWBytes + (mt * 16 + r) * Lay::kSBRow;
        bulk_g2s(sb, M.s + (size_t)row * G + g0, (uint32_t)(2 * ng), bar);
        bulk_g2s(sb + NMAT * 16 * Lay::kSBRow, M.b + (size_t)row * G + g0, (uint32_t)(2 * ng), bar);
      }
    }
  };

  // ---- the weight stream starts before the dependency wait: it reads nothing a
  //      preceding kernel writes
  if (warp == 0) {
    const int first = J < NS ? J : NS;
    for (int j = 0; j < first; ++j) issue(j);
    issued = first;
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  bool xv[NB];
#pragma unroll
  for (int h = 0; h < NB; ++h) xv[h] = (8 * h + g4) < p.rows;
  float y[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) y[i] = 0.0f;
  bool ok = true;

  // With one span per tile (k <= 2048 at 4 bits, k <= 1024 otherwise) every slot of the
  // CTA covers the same groups: the activation fragments and sums of the warp's groups
  // are loaded and formed once, at the first slot, and kept in registers.
  const bool hoist = NB == 1 && nspan == 1;  // (two row blocks: kept per group, registers)
  uint4 Xh0[GPW][NB], Xh1[GPW][NB];
  float Sh[GPW][NB][4];
  constexpr int NQ = GPW * NMAT * 16;  // group factors per warp per slot
  float4 *fw = fac + warp * NQ;
  for (int j = 0; j < J; ++j) {
    const int ti = j / nspan, sp = j - ti * nspan, buf = j % NS;
    int mi, lt;
    tile_mat(t0 + ti, mi, lt);
    const int g0 = sp * SPAN, ng = min(SPAN, G - g0);
    const uint8_t *slot = smem + buf * Lay::kSlot;
    if (sp == 0) {
#pragma unroll
      for (int i = 0; i < NV; ++i) y[i] = 0.0f;
    }
    if (ok && !mbar_wait_bounded(&full[buf], (uint32_t)(j / NS) & 1u, p.budget_ns, &s_abort)) {
      ok = false;
      s_abort = 1;
    }
    const int gw0 = warp * GPW;  // this warp's first group of the span
    if (ok && gw0 < ng) {
      const int gcnt = min(GPW, ng - gw0);
      // the factors of the warp's groups of this slot (lane q: group q / (16 NMAT),
      // matrix (q / 16) % NMAT, row q % 16)
      for (int q = lane; q < NQ; q += 32) {
        const int gi = q / (NMAT * 16), mt = (q >> 4) % NMAT, r = q & 15;
        const int gl = gw0 + gi, row = lt * 16 + r;
        float s1 = 0.0f, b1 = 0.0f;
        if (gi < gcnt && row < p.m[mi + mt].n) {
          if (p.sb_bulk) {
            const uint16_t *sb = reinterpret_cast<const uint16_t *>(slot + Lay::kWBytes) + (mt * 16 + r) * SPAN + gl;
            s1 = bf16_to_f32(sb[0]);
            b1 = bf16_to_f32(sb[NMAT * 16 * SPAN]);
          } else {
            const size_t off = (size_t)row * G + g0 + gl;
            s1 = bf16_to_f32(ldg_u16(p.m[mi + mt].s + off));
            b1 = bf16_to_f32(ldg_u16(p.m[mi + mt].b + off));
          }
        }
        fw[q] = group_factors<BITS>(s1, b1);
      }
      __syncwarp();
      if (hoist) {
        if (j == 0) {
#pragma unroll
          for (int gi = 0; gi < GPW; ++gi) {
#pragma unroll
            for (int h = 0; h < NB; ++h) {
              Xh0[gi][h] = make_uint4(0, 0, 0, 0);
              Xh1[gi][h] = make_uint4(0, 0, 0, 0);
              if (xv[h] && gi < gcnt)
                load_x_frag<kPair4>(p.x + (size_t)(8 * h + g4) * p.ldx + (size_t)(g0 + gw0 + gi) * 64 + 16 * c,
                                    Xh0[gi][h], Xh1[gi][h]);
            }
          }
#pragma unroll
          for (int gi = 0; gi < GPW; ++gi)
            if (gi < gcnt) mv_sums<NB>(Xh0[gi], Xh1[gi], Sh[gi]);
        }
#pragma unroll
        for (int gi = 0; gi < GPW; ++gi) {
          if (gi < gcnt)
            mv_group_s<BITS, NB, NMAT>(slot + (gw0 + gi) * GB + c * 4 * LW, WP, fw + gi * NMAT * 16, 16, Xh0[gi],
                                       Xh1[gi], Sh[gi], g4, y);
        }
      } else {
#pragma unroll
        for (int gi = 0; gi < GPW; ++gi) {
          if (gi < gcnt) {
            uint4 X0[NB], X1[NB];
            float S[NB][4];
#pragma unroll
            for (int h = 0; h < NB; ++h) {
              X0[h] = make_uint4(0, 0, 0, 0);
              X1[h] = make_uint4(0, 0, 0, 0);
              if (xv[h])
                load_x_frag<kPair4>(p.x + (size_t)(8 * h + g4) * p.ldx + (size_t)(g0 + gw0 + gi) * 64 + 16 * c,
                                    X0[h], X1[h]);
            }
            mv_sums<NB>(X0, X1, S);
            mv_group_s<BITS, NB, NMAT>(slot + (gw0 + gi) * GB + c * 4 * LW, WP, fw + gi * NMAT * 16, 16, X0, X1, S,
                                       g4, y);
          }
        }
      }
    }
    const bool last = sp == nspan - 1;
    float *rb = red + (ti & 1) * (kMvWarps * NV * 32);
    if (last) {
#pragma unroll
      for (int i = 0; i < NV; ++i) rb[(warp * NV + i) * 32 + lane] = y[i];
    }
    // every warp is done with slot j (it may be refilled) and the tile's partials are visible
    named_bar_sync(kBarSlot, kMvThreads);
    if (s_abort) ok = false;
    if (warp == 0 && ok && issued < J) {
      if (lane == 0) fence_proxy_async_smem();
      __syncwarp();
      issue(issued);
      ++issued;
    }
    if (last) {
      // the tile's outputs: the warps' partials added in warp order
      for (int v = tid; v < NO * 32; v += kMvThreads) {
        const int i = v >> 5, ln = v & 31;
        float acc[NMAT];
#pragma unroll
        for (int t = 0; t < NMAT; ++t) {
          acc[t] = rb[(t * NO + i) * 32 + ln];
#pragma unroll
          for (int w = 1; w < kMvWarps; ++w) acc[t] = __fadd_rn(acc[t], rb[(w * NV + t * NO + i) * 32 + ln]);
        }
        // value i of lane ln: half h = i / 4, element e = i % 4
        const int h = i >> 2, e = i & 3;
        const int ch = (ln >> 2) + ((e & 2) ? 8 : 0);
        const int row = lt * 16 + ch;
        const int xr = 8 * h + 2 * (ln & 3) + (e & 1);
        const MvMat &M = p.m[mi];
        if constexpr (MODE == kMvResid) {
          // post-add: the stored residual r' = bf16(r + y) and its square
          float sq = 0.0f;
          if (ok && row < M.n && xr < p.rows) {
            uint16_t *rp = p.resid + (size_t)xr * p.ldr + row;
            const uint16_t nb = f32_to_bf16_rn(__fadd_rn(bf16_to_f32(*rp), acc[0]));
            *rp = nb;
            const float vv = bf16_to_f32(nb);
            sq = __fmul_rn(vv, vv);
          }
          s_sq[xr][ch] = sq;
        } else if (ok && row < M.n && xr < p.rows) {
          if constexpr (MODE == kMvFfn) {
            static_cast<uint16_t *>(M.out)[(size_t)xr * M.ldo + row] = swiglu_bf16(acc[0], acc[1]);
          } else {
            static_cast<float *>(M.out)[(size_t)xr * M.ldo + row] = acc[0];
          }
        }
      }
      if constexpr (MODE == kMvResid) {
        // the tile's sum of squares per activation row, its 16 channels in order
        __syncthreads();
        if (tid < p.rows) {
          float sacc = 0.0f;
#pragma unroll
          for (int ch = 0; ch < 16; ++ch) sacc = __fadd_rn(sacc, s_sq[tid][ch]);
          p.part[(size_t)(t0 + ti) * 16 + tid] = sacc;
        }
        __syncthreads();
      }
    }
  }
  if (!ok && lane == 0) record_status(p.status, kErrTimeout);
  if (warp == 0 && lane == 0) {
    // copies issued but not consumed (only after a wait gave up) land before the CTA exits
    for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
      (void)mbar_wait_bounded(&full[j % NS], (uint32_t)(j / NS) & 1u, kMvDrainNs, nullptr);
  }
  if constexpr (MODE == kMvResid) resid_norm_tail<NB>(p);
}

// SMs of the current device (cached per device)
static int mv_sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int c = cached[dev].load(std::memory_order_relaxed);
  if (c == 0) {
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0) c = 1;
    cached[dev].store(c, std::memory_order_relaxed);
  }
  return c;
}

template <int BITS, int NB, int MODE>
static cudaError_t launch_t(const MvParams &p, int tiles, cudaStream_t st) {
  using Lay = MvLayout<BITS, NB, MODE>;
  static std::atomic<bool> attr_done[64];  // per device; setting the attributes twice is harmless
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev].load(std::memory_order_relaxed)) {
    cudaError_t e = cudaFuncSetAttribute(qmv_kernel<BITS, NB, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay::kBytes);
    if (e != cudaSuccess) return e;
    // the largest shared-memory carveout, so CTAs of consecutive launches (programmatic
    // dependent launch) share an SM
    e = cudaFuncSetAttribute(qmv_kernel<BITS, NB, MODE>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_done[dev].store(true, std::memory_order_relaxed);
  }
  const int sms = mv_sm_count();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles < sms ? tiles : sms));
  cfg.blockDim = dim3((unsigned)kMvThreads);
  cfg.dynamicSmemBytes = (size_t)Lay::kBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
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

cudaError_t launch_mv(MvParams &p, int mode, int bits, int tiles, cudaStream_t st) {
  p.groups = p.k / kGroup;
  const int span = bits == 4 ? span_g<4>() : (bits == 6 ? span_g<6>() : span_g<8>());
  p.nspan = (p.groups + span - 1) / span;
  p.ntiles = tiles;
  if (mode != kMvAttn) p.tile_end[0] = tiles;
  // scale/bias rows of a span can be bulk-copied when every copy starts and ends on a
  // 16-byte boundary: groups a multiple of 8 (spans are), pointers 16-byte aligned
  const int nm = mode == kMvAttn ? 4 : (mode == kMvFfn ? 2 : 1);
  bool sb = (p.groups % 8) == 0;
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
