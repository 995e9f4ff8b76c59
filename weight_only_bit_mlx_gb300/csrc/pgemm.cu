// pgemm.cu - prompt-window GEMM over MLX affine 4/6/8-bit group-64 weights on the
// sm_103a tensor cores (TMA -> exact dequant into shared memory -> tcgen05.mma).
//
// TensorFold PR #1696 (later revision), "What it adds" > "Prompt GEMM": prompt
// windows take a GEMM that dequantizes the 4-bit weights as it loads each weight
// tile; every output sums an fma chain per 64-wide k block and adds the blocks in
// order, so a row's sum does not depend on how the prompt is cut.
//
// For output Y[m][n] with 64-wide blocks b = 0..G-1:
//   P_b[n][m] = sum_{j in b} q[n][j] * X[m][j]      tcgen05.mma, bf16 x bf16 -> fp32
//               A = codes of the weight rows converted exactly to bf16 and written
//                   into shared memory in the UMMA 128-byte-swizzle K-major layout;
//               B = the X tile (256 rows), staged by TMA in shared memory; fresh
//               accumulator per block, double-buffered in tensor memory
//   y = fma(scale[n][b], P_b, y)  for b = 0..G-1 in order      (epilogue registers)
//   Y = (y + B_0) + B_1,  B_0 + B_1 = sum_b bias[n][b] * S_b[m]   (added last)
// with S_b[m] = sum_{j in b} X[m][j] computed by a pre-pass in fp32 and split
// exactly into three bf16 parts, so the bias term is one more small tcgen05
// contraction (k' = 3G) instead of a second fma per element and block; its k blocks
// alternate between the two accumulators like all others, giving two partial sums
// B_0 (the part holding the first bias block) and B_1.
//
// CTA pairs: a cluster of two CTAs computes a 256-channel x 256-row tile with
// tcgen05.mma.cta_group::2 at M = 256, N = 256, K = 16, issued by the first CTA.
// Each CTA stages its own 128 channels of W (A's half) and its own 128 rows of X (B's
// half) at the same shared-memory offsets, and its tensor memory receives its 128
// channels x all 256 rows; so each SM stages and reads half the X tile that a single
// CTA would.  The accumulator holds output channels in tensor-memory lanes, so an
// epilogue thread owns one channel: one scale per block, and the 32 lanes of a warp
// store 32 consecutive channels of a row (coalesced).
// Every quantity of row m depends only on X[m][:] and W: the tensor core computes
// each output from its own row and column, tiles out of range are zero-filled by
// TMA, and nothing (split-K, tile shape, order) depends on m or on the window.
//
// Warp roles (each CTA of the pair, 512 threads = four warpgroups):
//   warpgroup 0 (warps 0-3, 56 registers)
//     warp 0    TMA producer (this CTA's half of the X tile, or of the S-part tile,
//               and its packed W tile, per k block; scale and bias boxes)
//     warps 1-2 first CTA: MMA issuers (one thread each), warp 1 the even k blocks of
//               the pair's running block count and accumulator 0, warp 2 the odd ones
//               and accumulator 1; second CTA: warp 1 relays "my halves of block g are
//               staged" to the first CTA's pair_full barriers.  Warp 1 of both CTAs
//               allocates the pair's tensor memory (two accumulators of 256 columns).
//     warp 3    idle
//   warpgroup 1 (warps 4-7, 88 registers): converters, one channel row per thread,
//               packed codes -> bf16 A tile in shared memory, scales -> fp32
//   warpgroups 2-3 (warps 8-15, 184 registers): epilogue, tensor memory -> registers,
//               scale chain, bias add, and the store of the output (or the SwiGLU /
//               post-add epilogue, template EPI); two warps per lane quarter, 128 rows
//               of X each, held in registers across the k loop
// The launch gives every thread 128 registers; setmaxnreg moves them from the first two
// warpgroups to the epilogue, whose running sums (128 fp32 per thread) need them.
//
// Windows of 2048 rows and more: the codes are converted once per call into a bf16
// buffer (wconv_kernel, the same values the converters write), and the GEMM (BITS = 0)
// TMA-loads ready A tiles; its converters only stage the scales.  A call enqueues the
// conversion (for those windows), the row-sum pre-pass and the GEMM, each with
// programmatic dependent launch.  The GEMM triggers its dependents once each CTA has
// started its last tile, so the next call's conversion (into the other of two
// alternating buffers) runs on the SMs the last round leaves idle; the row sums and the
// GEMM wait for the kernel before them before they touch X, the sums or the outputs.
// Several weights on one X (pgemm_run_multi): one row-sum pre-pass, then each weight's
// conversion and GEMM in turn.
// Every wait is a bounded mbarrier wait (sync.cuh); a wait that gives up records
// QL_ERR_TIMEOUT, the CTA drains its own copies and MMAs, and both CTAs pass a final
// cluster barrier (neither leaves while the other may still touch its shared memory)
// before the pair's tensor memory is freed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "pgemm.cuh"
#include "sync.cuh"

namespace qlk {

namespace pg {

constexpr int BM = 256;   // rows of X per tile (MMA N)
constexpr int BMH = 128;  // rows of X staged by each CTA of the pair (its half of the MMA's N)
constexpr int BN = 128;   // output channels of each CTA (its half of the MMA's M = 256; tensor-memory lanes)
constexpr int BK = 64;
constexpr int kPairRing = 4;  // barriers on which the second CTA reports its staged halves
constexpr int kScStages = 8;  // fp32 scale rows (deep enough to need no release barrier, see converters)
constexpr int kConvWarps = 4;   // one channel row per thread
constexpr int kEpiWarps = 8;    // two per tensor-memory lane quarter, 128 rows of X each
constexpr int kRoleWarps = 4;   // producer, two MMA issuers (second CTA: the relay), one idle - warp 1 allocates tensor memory
constexpr int kThreads = (kRoleWarps + kConvWarps + kEpiWarps) * 32;
// registers per thread: at launch, and per warpgroup after setmaxnreg (multiples of 8)
constexpr int kRegsLaunch = 65536 / kThreads;
constexpr int kRegsRole = 56;
constexpr int kRegsConv = 88;
constexpr int kRegsEpi = 184;
static_assert(kThreads == 512 && kRoleWarps == 4 && kConvWarps == 4 && kEpiWarps == 8, "warpgroup layout");
static_assert(128 * (kRegsRole + kRegsConv) + 256 * kRegsEpi <= kThreads * kRegsLaunch,
              "the register split must fit in the registers the block is launched with");
constexpr int kEpiWarp0 = kRoleWarps + kConvWarps;
constexpr int kConvThreads = kConvWarps * 32;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kEpiRows = BM / (kEpiWarps / 4);  // rows of X per epilogue thread
constexpr int kXBytes = BMH * BK * 2;           // this CTA's half of the X tile: 128 rows x 64 bf16, 128-byte swizzle
constexpr int kABytes = BN * BK * 2;            // converted W tile: 128 rows x 64 bf16, 128-byte swizzle
constexpr int kABufs = 4;  // converted weight blocks the converters may run ahead of the MMA
constexpr int kTmemCols = 512;  // two accumulators of BM fp32 columns
static_assert(2 * BM <= kTmemCols, "tensor memory budget");
constexpr uint64_t kDrainBudgetNs = 2000000000ull;
constexpr int kBiasG = 128;  // groups of bias staged in shared memory (k <= 8192); larger k reads global
constexpr int kPf = 2;       // k blocks of scale/bias prefetch (no-TMA path)
constexpr int kLdCols = 16;   // accumulator columns per epilogue tensor-memory load (two in flight)
static_assert(kEpiRows % kLdCols == 0, "epilogue loads cover the thread's rows");
constexpr int kEpiBatch = 8;  // rows of the fused epilogues' global loads in flight together
constexpr int kEpiPrefetchLead = 8;  // k blocks before a tile's end at which its epilogue inputs are prefetched
static_assert(kScStages >= kABufs + 2 + 1, "scale ring must outlast the converter/epilogue lag");

// BITS = 4, 6, 8: packed W tiles, converted in the kernel.  BITS = 0 (kPre): the A
// operand arrives ready as bf16 (codes converted once per call by wconv_kernel, bias
// blocks appended), loaded by TMA with the 128-byte swizzle straight into the stage.
template <int BITS> struct Cfg {
  static constexpr bool kPre = BITS == 0;
  static constexpr int kRowBytes = kPre ? BK * 2 : BK * BITS / 8;  // bytes of one row per k block
  static constexpr int kWBytes = BN * kRowBytes;         // packed W tile (kPre: the bf16 A tile)
  static constexpr int kStages = 4;                      // TMA stages in flight (X/S half tile + W tile)
  static constexpr int kOffX = 0;
  static constexpr int kOffW = kOffX + kStages * kXBytes;
  static constexpr int kOffA = (kOffW + kStages * kWBytes + 1023) / 1024 * 1024;
  static constexpr int kOffSc = kOffA + (kPre ? 0 : kABufs * kABytes);
  // biases of the tile's rows, bf16, boxes of 8 groups: [kBiasG / 8][BN][8]
  static constexpr int kOffBias = kOffSc + kScStages * BN * 4;
  // scale boxes streamed by TMA, bf16 [2][BN][8]
  static constexpr int kOffScBox = kOffBias + (kPre ? 0 : BN * kBiasG * 2);
  static constexpr int kOffBar = kOffScBox + 2 * BN * 8 * 2;
  // barriers: tma_full, tma_empty, a_full[kABufs], a_empty[kABufs], acc_full[2], acc_empty[2],
  //           sc_full, scb_full[2], scb_empty[2], bias_full, bias_empty, mma_done[2], pair_full[kPairRing]
  static constexpr int kNumBars = 2 * kStages + 2 * kABufs + 4 + kScStages + 4 + 2 + 2 + kPairRing;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;  // tmem address, abort flag
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

struct Params {
  const uint8_t *wq;     // packed codes, rows of w_row_bytes (for the L2 prefetch of a tile's rows)
  int64_t w_row_bytes;
  const uint16_t *scales;
  const uint16_t *biases;
  int sc_tma;  // scales arrive as TMA boxes of 8 groups (k % 512 == 0, 16-byte aligned)
  int bi_tma;  // biases arrive as TMA boxes too (additionally k <= 64 * kBiasG)
  float *Y;
  int64_t ldy;
  const float *A;  // kPgSwiglu: the gate projection's output
  int64_t lda;
  uint16_t *H;     // kPgSwiglu: output; kPgResid: the residual, read and overwritten
  int64_t ldh;
  int epi_pf;      // the rows the fused epilogue reads may be prefetched in 16-byte pieces
  int M, N, G, NBB;
  int tiles_n, tiles;  // 256-channel tiles per 256-row band; tiles in all
  int *status;
  uint64_t budget_ns;
  // A GEMM of a multi-weight call after the first (windows below the pre-conversion
  // size): it reads only X and the row sums, complete before the GEMM before it could
  // release this one, and writes its own output, so it skips the dependency wait at the
  // start and runs beside that GEMM; one thread waits for it before the CTA exits, so
  // that the last GEMM of the call still ends after every other.
  int follow;
};

// ---- PTX wrappers --------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_addr(dst)),
      "l"(map), "r"(smem_addr(bar)), "r"(x), "r"(y)
      : "memory");
}

// a hint: bring `bytes` (a multiple of 16) at the 16-byte aligned global `p` into L2
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// programmatic dependent launch: wait until the preceding kernels of the stream are
// complete and their writes visible (a no-op when launched without the attribute)
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16u >> 4) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// instruction descriptor: kind::f16, A = B = bf16, D = f32, both K-major, M x N
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T on the CTA pair: issued by the first CTA; A's 256
// rows are the two CTAs' 128-row halves and B's N columns their two halves, both at the
// same shared-memory offsets in either CTA; each CTA's tensor memory receives its rows
__device__ __forceinline__ void mma_bf16_ss2(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void sts128(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// one arrival, once this thread's earlier MMAs are complete, on the barrier at `bar`'s
// offset in each CTA of the pair named by `mask` (bit r: CTA rank r)
__device__ __forceinline__ void mma_commit2(uint64_t *bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"(mask)
      : "memory");
}

// the shared::cluster address of the same variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_rank(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}

// arrive on a barrier of another CTA of the cluster, with the default semantics
// (release at CTA scope): what the arrival publishes is tensor-memory reads ordered by
// tcgen05.fence, or shared-memory tiles whose completion this thread observed; a
// cluster-scope release would also wait for the thread's outstanding global stores
// (the epilogue's output rows)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive columns of this warp's 32 lanes: r[j] = column taddr + j of this thread's lane
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// per-warpgroup register budget (all four warps of the warpgroup execute it)
template <int N> __device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N> __device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ uint4 lds128(const void *p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

// bits [off, off + 32) of a little-endian array of 32-bit words (off is a constant
// after unrolling; the word after the last is never needed for the fields used)
template <int NW>
__device__ __forceinline__ uint32_t window32(const uint32_t (&w)[NW], int off) {
  const int i = off >> 5, s = off & 31;
  if (s == 0) return w[i];
  const uint32_t hi = (i + 1 < NW) ? w[i + 1] : 0u;
  return __funnelshift_r(w[i], hi, s);
}

// Chunk c (8 codes, k = 8c .. 8c+7 of the held words) -> four bf16 pairs in k order.
template <int BITS, int NW>
__device__ __forceinline__ void convert_chunk(const uint32_t (&w)[NW], int c, uint32_t *o) {
  if constexpr (BITS == 4) {
    const uint32_t x = w[c], x4 = x >> 4;
    o[0] = q4_pair(x, x4, 0); o[1] = q4_pair(x, x4, 1); o[2] = q4_pair(x, x4, 2); o[3] = q4_pair(x, x4, 3);
  } else if constexpr (BITS == 8) {
    o[0] = q8_pair(w[2 * c], 0); o[1] = q8_pair(w[2 * c], 1);
    o[2] = q8_pair(w[2 * c + 1], 0); o[3] = q8_pair(w[2 * c + 1], 1);
  } else {
    o[0] = q6_pair(window32(w, 48 * c));
    o[1] = q6_pair(window32(w, 48 * c + 12));
    o[2] = q6_pair(window32(w, 48 * c + 24));
    o[3] = q6_pair(window32(w, 48 * c + 36));
  }
}

// ---- the GEMM kernel -------------------------------------------------------------
// Persistent: one CTA per SM walks the tiles t = blockIdx.x, blockIdx.x + gridDim.x, ...
// (128-channel tiles fastest, so CTAs working at the same time share 256-row bands of
// X in L2).  Every role keeps running counters across tiles (k blocks g, main blocks
// h, scale boxes, accumulator uses), so the next tile's copies, conversions and MMAs
// overlap this tile's epilogue.
template <int BITS, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    pgemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                 const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmSc,
                 const __grid_constant__ CUtensorMap tmBi, const __grid_constant__ Params p) {
  using C = Cfg<BITS>;
  constexpr bool kPre = C::kPre;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sX = smem + C::kOffX;
  uint8_t *sW = smem + C::kOffW;
  uint8_t *sA = smem + C::kOffA;
  float *sSc = reinterpret_cast<float *>(smem + C::kOffSc);
  uint16_t *sbias = reinterpret_cast<uint16_t *>(smem + C::kOffBias);
  uint16_t *scbox = reinterpret_cast<uint16_t *>(smem + C::kOffScBox);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint64_t *tma_full = bars;
  uint64_t *tma_empty = tma_full + C::kStages;
  uint64_t *a_full = tma_empty + C::kStages;
  uint64_t *a_empty = a_full + kABufs;
  uint64_t *acc_full = a_empty + kABufs;
  uint64_t *acc_empty = acc_full + 2;
  uint64_t *sc_full = acc_empty + 2;
  uint64_t *scb_full = sc_full + kScStages;
  uint64_t *scb_empty = scb_full + 2;
  uint64_t *bias_full = scb_empty + 2;
  uint64_t *bias_empty = bias_full + 1;
  uint64_t *mma_done = bias_empty + 1;
  uint64_t *pair_full = mma_done + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G, KB = p.G + p.NBB;
  const uint64_t budget = p.budget_ns;
  // the CTA pair: rank 0 issues the MMAs for both; each CTA stages its own 128 channels
  // of W and its own 128 rows of X and receives its 128 channels of the accumulator
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) { mbar_init(&tma_full[i], 1); mbar_init(&tma_empty[i], 1 + kConvThreads); }
    for (int i = 0; i < kABufs; ++i) {
      mbar_init(&a_full[i], kConvThreads);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      // the first CTA's epilogue threads, and one arrival per epilogue warp of the second
      mbar_init(&acc_empty[i], kEpiThreads + kEpiWarps);
      mbar_init(&scb_full[i], 1);
      mbar_init(&scb_empty[i], kConvThreads);
    }
    for (int i = 0; i < kPairRing; ++i) mbar_init(&pair_full[i], 1);
    for (int i = 0; i < kScStages; ++i) mbar_init(&sc_full[i], kConvThreads);
    mbar_init(bias_full, 1);
    mbar_init(bias_empty, kConvThreads);
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmS);
    if (p.sc_tma) prefetch_tmap(&tmSc);
    if (p.bi_tma) prefetch_tmap(&tmBi);
  }
  // both CTAs are running and their barriers initialised before either allocates tensor
  // memory for the pair or arrives on the other's barriers
  cluster_sync_all();
  if (warp == 1) {
    // one warp of each CTA of the pair allocates, collectively
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto give_up = [&]() {
    *abort_flag = 1;
    record_status(p.status, kErrTimeout);
  };
  // the wait for the kernels before this one (none at the start for a follower)
  auto dep_wait = [&]() {
    if (!p.follow) griddep_wait();
  };

  // Each role first sets its warpgroup's register budget (the warpgroups that give
  // registers up do so before the epilogue's increase can be granted).
  if (warp < kRoleWarps) {
    regs_dec<kRegsRole>();
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        int g = 0, box = 0, tj = 0, bias_sets = 0;
        bool alive = true;
        bool dep_done = false;  // griddep_wait() passed: X and the row sums may be read
        bool released = false;  // the kernels launched after this one may start
        for (int t = pair; t < p.tiles && alive; t += npairs, ++tj) {
          const bool last_tile = t + npairs >= p.tiles;
          // this CTA's channels and rows of X of tile t
          const int n0 = (t % p.tiles_n) * (2 * BN) + (int)rank * BN, m0 = (t / p.tiles_n) * BM + (int)rank * BMH;
          if constexpr (!kPre) {
            // the tile's packed rows (contiguous) into L2 ahead of their TMA loads: a
            // prompt window reads each weight tile once, straight from HBM
            const int rows = min(BN, p.N - n0);
            if (rows > 0) prefetch_l2_bulk(p.wq + (size_t)n0 * p.w_row_bytes, (uint32_t)(rows * p.w_row_bytes));
          }
          if (p.bi_tma) {
            // every bias of the tile's channels, once per tile (read only by its bias
            // blocks), after the previous tile's bias blocks are converted
            if (tj > 0 && !mbar_wait_bounded(bias_empty, (uint32_t)((tj - 1) & 1), budget, abort_flag)) {
              give_up();
              break;
            }
            const int nbox = (G + 7) / 8;
            mbar_arrive_expect_tx(bias_full, (uint32_t)(nbox * BN * 16));
            for (int i = 0; i < nbox; ++i) tma_load_2d(sbias + i * BN * 8, &tmBi, bias_full, 8 * i, n0);
            ++bias_sets;
          }
          for (int kb = 0; kb < KB; ++kb) {
            if (EPI != kPgStore && p.epi_pf && kb == (G > kEpiPrefetchLead ? G - kEpiPrefetchLead : 0)) {
              // the tile's rows of the fused epilogue's input (the gate output, or the
              // residual), this CTA's channels, into L2 ahead of the tile's end
              const int mt = (t / p.tiles_n) * BM;
              const int nch = min(BN, p.N - n0);
              const uint32_t esz = EPI == kPgSwiglu ? 4u : 2u;
              const uint32_t bytes = ((uint32_t)nch * esz) & ~15u;
              if (nch > 0 && bytes > 0) {
                for (int r = 0; r < BM && mt + r < p.M; ++r) {
                  const void *src = EPI == kPgSwiglu
                                        ? static_cast<const void *>(p.A + (size_t)(mt + r) * p.lda + n0)
                                        : static_cast<const void *>(p.H + (size_t)(mt + r) * p.ldh + n0);
                  prefetch_l2_bulk(src, bytes);
                }
              }
            }
            if (p.sc_tma && kb < G && (kb & 7) == 0) {
              // scales of blocks kb .. kb+7 for the tile's channels, two boxes in flight
              const int slot = box & 1;
              if (!mbar_wait_bounded(&scb_empty[slot], ((uint32_t)(box >> 1) & 1u) ^ 1u, budget, abort_flag)) {
                give_up();
                alive = false;
                break;
              }
              mbar_arrive_expect_tx(&scb_full[slot], (uint32_t)(BN * 16));
              tma_load_2d(scbox + slot * BN * 8, &tmSc, &scb_full[slot], kb, n0);
              ++box;
            }
            const int s = g % C::kStages;
            const uint32_t ph = (uint32_t)(g / C::kStages) & 1u;
            if (!mbar_wait_bounded(&tma_empty[s], ph ^ 1u, budget, abort_flag)) {
              give_up();
              alive = false;
              break;
            }
            if constexpr (kPre) {
              // the bf16 A tile (main or bias block) and X or the row-sum parts; A is
              // written by the conversion pre-pass, so both wait for the earlier kernels
              if (!dep_done) {
                dep_wait();
                dep_done = true;
              }
              mbar_arrive_expect_tx(&tma_full[s], (uint32_t)(kXBytes + C::kWBytes));
              tma_load_2d(sW + s * C::kWBytes, &tmW, &tma_full[s], kb * BK, n0);
              if (kb < G)
                tma_load_2d(sX + s * kXBytes, &tmX, &tma_full[s], kb * BK, m0);
              else
                tma_load_2d(sX + s * kXBytes, &tmS, &tma_full[s], (kb - G) * BK, m0);
            } else if (kb < G) {
              mbar_arrive_expect_tx(&tma_full[s], (uint32_t)(kXBytes + C::kWBytes));
              tma_load_2d(sW + s * C::kWBytes, &tmW, &tma_full[s], kb * (BK * BITS / 32), n0);
              if (!dep_done) {  // the weights are constant; X is written by earlier kernels
                dep_wait();
                dep_done = true;
              }
              tma_load_2d(sX + s * kXBytes, &tmX, &tma_full[s], kb * BK, m0);
            } else {
              mbar_arrive_expect_tx(&tma_full[s], (uint32_t)kXBytes);
              if (!dep_done) {
                dep_wait();
                dep_done = true;
              }
              tma_load_2d(sX + s * kXBytes, &tmS, &tma_full[s], (kb - G) * BK, m0);
            }
            ++g;
            if (last_tile && dep_done && !released) {
              // This CTA has started its last tile: a kernel launched after this one
              // with programmatic dependent launch (the next call's code conversion)
              // may take the SMs that the pairs without a tile left leave idle.  Only
              // after the dependency wait, so that every kernel before this one has ended
              // (a follower's predecessor released it only after its own wait).
              asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
              released = true;
            }
          }
        }
        // drain: every copy this CTA started must land before its shared memory goes away
        for (int j = (box > 2 ? box - 2 : 0); j < box; ++j)
          (void)mbar_wait_bounded(&scb_full[j & 1], (uint32_t)(j >> 1) & 1u, kDrainBudgetNs, nullptr);
        if (bias_sets > 0) (void)mbar_wait_bounded(bias_full, (uint32_t)((bias_sets - 1) & 1), kDrainBudgetNs, nullptr);
        for (int s = 0; s < C::kStages && s < g; ++s) {
          const int uses = (g - 1 - s) / C::kStages + 1;
          (void)mbar_wait_bounded(&tma_full[s], (uint32_t)(uses - 1) & 1u, kDrainBudgetNs, nullptr);
        }
      }
    } else if (warp == 1 || warp == 2) {
      // ------------------------------------------------------------ MMA issuers (first CTA)
      // The k blocks of the pair (all tiles, main and bias blocks) alternate between the
      // two issuers and the two accumulators by their running index g: issuer par takes
      // g % 2 == par into accumulator par.  A main block is one use of the accumulator;
      // the bias blocks of a tile that fall to one issuer chain into one use (so each
      // accumulator holds half of the bias contraction).  Strict alternation keeps each
      // issuer at most one block ahead of the other, so no wait is ever more than one
      // phase ahead of a barrier's last completion.  A block is issued once both CTAs
      // have staged their halves: this CTA's own barriers, and pair_full, on which the
      // second CTA's relay reports its halves.  Each commit arrives on the barrier at the
      // same offset in both CTAs (mask 0b11).
      // ------------------------------------------------------------ relay (second CTA)
      // Warp 1 waits, block by block, for this CTA's X (or S) half and converted W tile
      // and reports them on the first CTA's pair_full.
      const int par = warp - 1;
      if (lane == 0 && leader) {
        constexpr uint32_t idesc = idesc_bf16(2 * BN, BM);
        bool any = false, alive = true;
        int g = 0, uses = 0;  // k blocks of the pair so far; uses of accumulator par so far
        for (int t = pair; t < p.tiles && alive; t += npairs) {
          const int g0 = g;
          // this issuer's first and last bias block of the tile
          const int kb_first = G + ((g0 + G) % 2 == par ? 0 : 1);
          const int kb_last = (g0 + KB - 1) % 2 == par ? KB - 1 : KB - 2;
          for (int kb = 0; kb < KB; ++kb, ++g) {
            if ((g & 1) != par) continue;
            const int s = g % C::kStages, ab = g % kABufs;
            if (!mbar_wait_bounded(&tma_full[s], (uint32_t)(g / C::kStages) & 1u, budget, abort_flag) ||
                !mbar_wait_bounded(&a_full[ab], (uint32_t)(g / kABufs) & 1u, budget, abort_flag) ||
                !mbar_wait_bounded(&pair_full[g % kPairRing], (uint32_t)(g / kPairRing) & 1u, budget, abort_flag)) {
              give_up();
              alive = false;
              break;
            }
            const bool opens = kb < G || kb == kb_first;   // a new use of the accumulator
            const bool closes = kb < G || kb == kb_last;
            if (opens) {  // both CTAs' epilogues have read the accumulator's last use
              if (!mbar_wait_bounded(&acc_empty[par], ((uint32_t)uses & 1u) ^ 1u, budget, abort_flag)) {
                give_up();
                alive = false;
                break;
              }
            }
            tc_fence_after();
            const uint32_t d = tmem_base + (uint32_t)(par * BM);
            const uint64_t ad = sw128_desc(smem_addr(kPre ? sW + s * C::kWBytes : sA + ab * kABytes));
            const uint64_t bd = sw128_desc(smem_addr(sX + s * kXBytes));
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint32_t acc = (kk > 0 || !opens) ? 1u : 0u;
              mma_bf16_ss2(d, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc, acc);
            }
            any = true;
            mma_commit2(&tma_empty[s], 3);
            mma_commit2(&a_empty[ab], 3);
            if (closes) {
              mma_commit2(&acc_full[par], 3);
              ++uses;
            }
          }
        }
        if (any) {
          mma_commit2(&mma_done[par], 1);
          (void)mbar_wait_bounded(&mma_done[par], 0u, kDrainBudgetNs, nullptr);
        }
      } else if (lane == 0 && par == 0) {
        const uint32_t pf0 = mapa_rank(pair_full, 0);
        bool alive = true;
        int g = 0;
        for (int t = pair; t < p.tiles && alive; t += npairs) {
          for (int kb = 0; kb < KB; ++kb, ++g) {
            const int s = g % C::kStages, ab = g % kABufs;
            if (!mbar_wait_bounded(&tma_full[s], (uint32_t)(g / C::kStages) & 1u, budget, abort_flag) ||
                !mbar_wait_bounded(&a_full[ab], (uint32_t)(g / kABufs) & 1u, budget, abort_flag)) {
              give_up();
              alive = false;
              break;
            }
            mbar_arrive_cluster(pf0 + (uint32_t)((g % kPairRing) * 8));
          }
        }
      }
    }     // warp 3: idle
  } else if (warp < kEpiWarp0) {
    regs_dec<kRegsConv>();
    // ------------------------------------------------------------ converters
    // Thread = one channel row of the tile.  Its 64 codes of the block become 32 exact
    // bf16 pairs, written as eight 16-byte chunks of the row of the A tile in the
    // UMMA 128-byte-swizzle K-major layout: 8-row groups 1024 bytes apart, rows 128
    // bytes apart, chunk c of row r at position c ^ (r % 8).
    const int ct = 32 * (warp & 3) + lane;  // channel (row of the W tile)
    // (kPre: the A tiles arrive ready by TMA; the converters only stage the scales)
    const bool bias_smem = !kPre && G <= kBiasG;
    const uint32_t a_row = smem_addr(sA) + (uint32_t)((ct >> 3) * 1024 + (ct & 7) * 128);
    const uint32_t sw = (uint32_t)(ct & 7);
    bool alive = true;
    int g = 0, h = 0, box = 0, tj = 0;  // k blocks, main blocks, scale boxes, tiles
    for (int t = pair; t < p.tiles && alive; t += npairs, ++tj) {
      const int n = (t % p.tiles_n) * (2 * BN) + (int)rank * BN + ct;
      const bool nvalid = n < p.N;
      const uint16_t *srow = p.scales + (size_t)(nvalid ? n : 0) * G;
      const uint16_t *brow = p.biases + (size_t)(nvalid ? n : 0) * G;
      // Without TMA boxes (k % 512 != 0), the thread loads its channel's scale and bias
      // itself, kPf blocks ahead; the loop is unrolled by kPf so that each ring slot
      // stays in place while its load is in flight.
      uint32_t sr[kPf], br[kPf];
#pragma unroll
      for (int i = 0; i < kPf; ++i) {
        sr[i] = (!p.sc_tma && nvalid && i < G) ? ldg_u16(srow + i) : 0u;
        br[i] = (!p.bi_tma && bias_smem && nvalid && i < G) ? ldg_u16(brow + i) : 0u;
      }
      for (int kb0 = 0; kb0 < KB && alive; kb0 += kPf) {
#pragma unroll
        for (int u = 0; u < kPf; ++u) {
          const int kb = kb0 + u;
          if (kb >= KB || !alive) break;
          const int s = g % C::kStages, ab = g % kABufs;
          uint32_t s_cur = 0u, b_cur = 0u;
          if (kb < G) {
            if (p.sc_tma) {
              const int slot = box & 1;
              if ((kb & 7) == 0 &&
                  !mbar_wait_bounded(&scb_full[slot], (uint32_t)(box >> 1) & 1u, budget, abort_flag)) {
                give_up();
                alive = false;
                break;
              }
              s_cur = scbox[(slot * BN + ct) * 8 + (kb & 7)];
              if ((kb & 7) == 7 || kb == G - 1) {
                mbar_arrive(&scb_empty[slot]);
                ++box;
              }
            } else {
              s_cur = sr[u];
              sr[u] = (nvalid && kb + kPf < G) ? ldg_u16(srow + kb + kPf) : 0u;
            }
            if (!p.bi_tma && bias_smem) {
              b_cur = br[u];
              br[u] = (nvalid && kb + kPf < G) ? ldg_u16(brow + kb + kPf) : 0u;
            }
          }
          if (!mbar_wait_bounded(&tma_full[s], (uint32_t)(g / C::kStages) & 1u, budget, abort_flag) ||
              !mbar_wait_bounded(&a_empty[ab], ((uint32_t)(g / kABufs) & 1u) ^ 1u, budget, abort_flag)) {
            give_up();
            alive = false;
            break;
          }
          const uint32_t dst = a_row + (uint32_t)(ab * kABytes);
          if (kb < G) {
            if constexpr (!kPre) {
              constexpr int NW = BK * BITS / 32;  // words of the row
              uint32_t w[NW];
              const uint8_t *wp = sW + s * C::kWBytes + ct * C::kRowBytes;
#pragma unroll
              for (int i = 0; i < NW / 4; ++i) {
                uint4 v = lds128(wp + 16 * i);
                w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
              }
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                uint32_t o[4];
                convert_chunk<BITS, NW>(w, c, o);
                sts128(dst + ((((uint32_t)c) ^ sw) << 4), o[0], o[1], o[2], o[3]);
              }
              if (!p.bi_tma && bias_smem) sbias[((kb >> 3) * BN + ct) * 8 + (kb & 7)] = (uint16_t)b_cur;
            }
            // Scale slot h % kScStages was last read by the epilogue for main block
            // h - kScStages.  Passing a_empty for this block means the MMA of the block
            // kABufs earlier finished, which waited for the epilogue to release the
            // accumulator use two main blocks before that; kScStages >= kABufs + 3 keeps
            // the slot free.
            sSc[(h % kScStages) * BN + ct] = bf16_to_f32(s_cur);
          } else if constexpr (!kPre) {
            // bias block: column t of block jb is k' = 64*jb + t of the [part][group]
            // layout; its A value is bias[n][k' mod G] (zero past 3G)
            if (kb == G && p.bi_tma && !mbar_wait_bounded(bias_full, (uint32_t)(tj & 1), budget, abort_flag)) {
              give_up();
              alive = false;
              break;
            }
            const int base = (kb - G) * BK;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              uint32_t o[4] = {0u, 0u, 0u, 0u};
              int j = base + 8 * c;
              if (bias_smem && (G % 8) == 0) {
                // a run of 8 columns never crosses a multiple of G: one 16-byte row of a
                // staged bias box
                if (nvalid && j < 3 * G) {
                  if (j >= G) j -= G;
                  if (j >= G) j -= G;
                  const uint4 v = lds128(sbias + ((j >> 3) * BN + ct) * 8);
                  o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
                }
              } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  int jj = j + e;
                  uint32_t v = 0u;
                  if (nvalid && jj < 3 * G) {
                    if (jj >= G) jj -= G;
                    if (jj >= G) jj -= G;
                    v = bias_smem ? (uint32_t)sbias[((jj >> 3) * BN + ct) * 8 + (jj & 7)] : ldg_u16(brow + jj);
                  }
                  o[e >> 1] |= v << (16 * (e & 1));
                }
              }
              sts128(dst + ((((uint32_t)c) ^ sw) << 4), o[0], o[1], o[2], o[3]);
            }
          }
          if constexpr (!kPre) fence_proxy_async_smem();  // the A tile is read by the tensor core (async proxy)
          mbar_arrive(&a_full[ab]);
          if (kb < G) {
            mbar_arrive(&sc_full[h % kScStages]);
            ++h;
          }
          mbar_arrive(&tma_empty[s]);
          if (kb == KB - 1) mbar_arrive(bias_empty);  // the tile's bias boxes are read
          ++g;
        }
      }
    }
  } else {
    regs_inc<kRegsEpi>();
    // ------------------------------------------------------------ epilogue
    dep_wait();  // the outputs (and the fused epilogues' inputs) belong to earlier kernels until then
    constexpr int CW = kEpiRows;  // rows of X owned by one thread
    const int q = warp & 3;       // tensor-memory lane quarter this warp may access
    const int slice = (warp - kEpiWarp0) >> 2;
    const int ch_row = 32 * q + lane;  // output channel of this thread within the tile
    const uint32_t lane_base = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(slice * CW);
    uint32_t phase = 0u;   // bit b: parity of the completed uses of accumulator b
    int h = 0;             // main blocks so far
    int g0 = 0;            // running index of the tile's first k block (as the issuers count)
    bool ok = true;
    // an accumulator use is read: every thread of the first CTA arrives on its
    // acc_empty, the second CTA's warps once each (after all their lanes' loads)
    const uint32_t acc_empty0 = mapa_rank(acc_empty, 0);
    auto release = [&](int buf) {
      tc_fence_before();
      if (leader) {
        mbar_arrive(&acc_empty[buf]);
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty0 + (uint32_t)(buf * 8));
      }
    };
    for (int t = pair; t < p.tiles && ok; t += npairs, g0 += KB) {
      // this CTA's 128 channels; the accumulator holds all 256 rows of the tile
      const int n0 = (t % p.tiles_n) * (2 * BN) + (int)rank * BN, m0 = (t / p.tiles_n) * BM;
      // the running sums of the thread's CW rows, as pairs (rows 2j, 2j + 1) so that each
      // step is one packed fp32 fma per pair (round to nearest in each lane)
      float2 y[CW / 2];
#pragma unroll
      for (int i = 0; i < CW / 2; ++i) y[i] = make_float2(0.0f, 0.0f);
      for (int kb = 0; kb < G; ++kb, ++h) {
        const int buf = (g0 + kb) & 1, sc = h % kScStages;
        bool w_ok = mbar_wait_bounded(&acc_full[buf], (phase >> buf) & 1u, budget, abort_flag) &&
                    mbar_wait_bounded(&sc_full[sc], (uint32_t)(h / kScStages) & 1u, budget, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) {
          give_up();
          ok = false;
          break;
        }
        tc_fence_after();
        const float s1 = sSc[sc * BN + ch_row];
        const float2 sv = make_float2(s1, s1);
        // software-pipelined: the load of chunk c + 1 is in flight while chunk c is
        // accumulated (tcgen05.wait::ld then waits only for that one load)
        const uint32_t ta = lane_base + (uint32_t)(buf * BM);
        uint32_t r[2][kLdCols];
        tmem_ld16_nowait(ta, r[0]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < CW / kLdCols; ++c) {
          if (c + 1 < CW / kLdCols) tmem_ld16_nowait(ta + (uint32_t)((c + 1) * kLdCols), r[(c + 1) & 1]);
#pragma unroll
          for (int i = 0; i < kLdCols / 2; ++i)
            y[c * (kLdCols / 2) + i] = __ffma2_rn(
                sv, make_float2(__uint_as_float(r[c & 1][2 * i]), __uint_as_float(r[c & 1][2 * i + 1])),
                y[c * (kLdCols / 2) + i]);
          if (c + 1 < CW / kLdCols) tmem_wait_ld();
        }
        release(buf);
        phase ^= 1u << buf;
      }
      if (!ok) break;
      // the bias contraction of the tile: its blocks alternate between the two
      // accumulators; the part of the tile's first bias block is added first.  Each
      // accumulator is released before the stores, so the next tile's MMAs can start
      // while this tile is written out.
      const int nparts = p.NBB >= 2 ? 2 : 1;
      for (int part = 0; part < nparts && ok; ++part) {
        const int buf = (g0 + G + part) & 1;
        bool w_ok = mbar_wait_bounded(&acc_full[buf], (phase >> buf) & 1u, budget, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) {
          give_up();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ta = lane_base + (uint32_t)(buf * BM);
        uint32_t r[2][kLdCols];
        tmem_ld16_nowait(ta, r[0]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < CW / kLdCols; ++c) {
          if (c + 1 < CW / kLdCols) tmem_ld16_nowait(ta + (uint32_t)((c + 1) * kLdCols), r[(c + 1) & 1]);
#pragma unroll
          for (int i = 0; i < kLdCols / 2; ++i)
            y[c * (kLdCols / 2) + i] = __fadd2_rn(
                y[c * (kLdCols / 2) + i], make_float2(__uint_as_float(r[c & 1][2 * i]), __uint_as_float(r[c & 1][2 * i + 1])));
          if (c + 1 < CW / kLdCols) tmem_wait_ld();
        }
        release(buf);
        phase ^= 1u << buf;
      }
      if (!ok) break;
      // one channel per thread: lanes of a warp write 32 consecutive channels of a row
      const int n = n0 + ch_row;
      if (n < p.N) {
        const int mb = m0 + slice * CW;
        if constexpr (EPI == kPgStore) {
          float *yp = p.Y + (size_t)mb * p.ldy + n;
          if (mb + CW <= p.M) {
            // the whole slice is in range: one store per row, the pointer stepped by the pitch
#pragma unroll
            for (int i = 0; i < CW / 2; ++i) {
              yp[0] = y[i].x;
              yp[p.ldy] = y[i].y;
              yp += 2 * p.ldy;
            }
          } else {
#pragma unroll
            for (int i = 0; i < CW; ++i)
              if (mb + i < p.M) yp[(size_t)i * p.ldy] = (i & 1) ? y[i >> 1].y : y[i >> 1].x;
          }
        } else if constexpr (EPI == kPgSwiglu) {
          // the SwiGLU of the FFN: h = bf16(silu(a) * c), c = this output.  The gate
          // values are loaded kEpiBatch at a time before any store, so the loads are in
          // flight together (a store to h could otherwise alias the next load of a).
          const float *acol = p.A + (size_t)mb * p.lda + n;
          uint16_t *hcol = p.H + (size_t)mb * p.ldh + n;
#pragma unroll
          for (int i0 = 0; i0 < CW; i0 += kEpiBatch) {
            float av[kEpiBatch];
#pragma unroll
            for (int i = 0; i < kEpiBatch; ++i)
              av[i] = (mb + i0 + i < p.M) ? __ldg(acol + (size_t)(i0 + i) * p.lda) : 0.0f;
#pragma unroll
            for (int i = 0; i < kEpiBatch; ++i)
              if (mb + i0 + i < p.M)
                hcol[(size_t)(i0 + i) * p.ldh] = swiglu_bf16(av[i], ((i0 + i) & 1) ? y[(i0 + i) >> 1].y : y[(i0 + i) >> 1].x);
          }
        } else {
          // the post-add of the residual stream: r' = bf16(r + y), stored in place, the
          // residual read kEpiBatch rows at a time before the stores
          uint16_t *rcol = p.H + (size_t)mb * p.ldh + n;
#pragma unroll
          for (int i0 = 0; i0 < CW; i0 += kEpiBatch) {
            uint16_t rv[kEpiBatch];
#pragma unroll
            for (int i = 0; i < kEpiBatch; ++i) rv[i] = (mb + i0 + i < p.M) ? rcol[(size_t)(i0 + i) * p.ldh] : 0;
#pragma unroll
            for (int i = 0; i < kEpiBatch; ++i)
              if (mb + i0 + i < p.M)
                rcol[(size_t)(i0 + i) * p.ldh] = f32_to_bf16_rn(
                    __fadd_rn(bf16_to_f32(rv[i]), ((i0 + i) & 1) ? y[(i0 + i) >> 1].y : y[(i0 + i) >> 1].x));
            }
        }
      }
    }
  }

  if (p.follow && threadIdx.x == 0) griddep_wait();  // a follower ends after the GEMM before it
  // neither CTA leaves (or frees the pair's tensor memory) while the other may still
  // read its shared memory, write its barriers or run MMAs into its tensor memory
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                 : "memory");
  }
}

// ---- row sums, split exactly into three bf16 parts ------------------------------
// S[m][b] = sum_{j in b} X[m][j] (fp32, j in increasing order); written as
// out[m][p*G + b] = part p (p = 0: nearest bf16 of S, 1: of the remainder, 2: rest).
// A tile is kXsumPairs consecutive (m, b) pairs.  A CTA stages a tile's 128-byte blocks
// of X in shared memory with coalesced 16-byte loads (16-byte chunk c of pair q at
// position c ^ (q % 8), so neither the stores nor the reads below collide on a bank),
// then each thread sums its own block in order.  The grid is at most one wave: a CTA
// walks tiles gridDim.x apart and loads its next tile into registers while it sums the
// current one.
constexpr int kXsumPairs = 256;
__global__ void __launch_bounds__(kXsumPairs) xsum_split_kernel(const uint16_t *X, int M, int G, int64_t ldx,
                                                                uint16_t *out, int64_t ldo) {
  // the GEMM that follows may start its set-up now (it reads these sums only after
  // this kernel completes)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Launched with programmatic dependent launch, this kernel may start while the kernel
  // before it still runs (the code conversion, or the previous call's GEMM in its last
  // tiles); it waits for that kernel, and so for every kernel before it, to end before it
  // reads X (which a fused epilogue of the previous GEMM may have written) or writes the
  // sums (which the previous GEMM reads).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ __align__(16) uint4 stage[kXsumPairs * 8];
  const int total = M * G;  // the host keeps this below 2^31
  const int tiles = (total + kXsumPairs - 1) / kXsumPairs;
  uint4 v[8];
  auto load = [&](int t) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int qi = threadIdx.x + kXsumPairs * i;  // chunk qi % 8 of pair qi / 8
      const int pr = t * kXsumPairs + (qi >> 3);
      if (pr < total) {
        const int m = pr / G, b = pr - m * G;
        v[i] = ldg_v4(X + (int64_t)m * ldx + (int64_t)b * 64 + 8 * (qi & 7));
      }
    }
  };
  if ((int)blockIdx.x < tiles) load(blockIdx.x);
  for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int qi = threadIdx.x + kXsumPairs * i;
      const int q = qi >> 3, c = qi & 7;
      if (t * kXsumPairs + q < total) stage[q * 8 + (c ^ (q & 7))] = v[i];
    }
    __syncthreads();
    if (t + (int)gridDim.x < tiles) load(t + gridDim.x);
    const int q = threadIdx.x, pr = t * kXsumPairs + q;
    if (pr < total) {
      float s = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 u = stage[q * 8 + (i ^ (q & 7))];
        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          s = __fadd_rn(s, bf16_to_f32(wv[e] & 0xFFFFu));
          s = __fadd_rn(s, bf16_to_f32(wv[e] >> 16));
        }
      }
      const uint16_t h0 = f32_to_bf16_rn(s);
      const float r1 = __fsub_rn(s, bf16_to_f32(h0));
      const uint16_t h1 = f32_to_bf16_rn(r1);
      const float r2 = __fsub_rn(r1, bf16_to_f32(h1));
      const uint16_t h2 = f32_to_bf16_rn(r2);
      const int m = pr / G, b = pr - m * G;
      uint16_t *o = out + (int64_t)m * ldo + b;
      o[0] = h0;
      o[G] = h1;
      o[2 * G] = h2;
    }
    __syncthreads();  // the stage is refilled next
  }
}


// ---- the codes as exact bf16, once per call (large prompt windows) ------------------
// A[r][j], rows kp = k + lds apart: for j < k the code q[r][j] as an exact bf16; for
// k <= j < kp column j - k of the bias blocks, bias[r][(j - k) mod G] while j - k < 3G and
// 0 after.  These are the values the converters write into the A tiles, so the GEMM
// computes the same bits from either.
// A thread writes kWconvChunks 8-value chunks, kWconvThreads chunks apart (so each load and store
// instruction of a warp covers consecutive words and chunks); all code words are loaded
// before the first chunk is converted, so one launch of a single wave keeps the whole of
// W in flight instead of one word per thread.
constexpr int kWconvThreads = 256;
constexpr int kWconvChunks = 4;
template <int BITS>
__global__ void __launch_bounds__(kWconvThreads) wconv_kernel(const uint32_t *wq, const uint16_t *biases, int n,
                                                             int k, int64_t kp, uint16_t *A) {
  // It is launched with programmatic dependent launch: it may run while the GEMM before
  // it (which triggers on its last tiles) still works, on the SMs that GEMM leaves
  // idle.  It reads only W and writes only its own A buffer, which the GEMM before it
  // does not read (calls alternate between two buffers).  The row-sum pass that
  // follows may be launched at once; it waits for this kernel to end.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int G = k / 64;
  const int per_row = (int)(kp / 8);  // 8-value chunks per row
  const int total = n * per_row;      // the host keeps this below 2^31
  const int64_t wpr = (int64_t)k * BITS / 32;
  const int i0 = blockIdx.x * (kWconvThreads * kWconvChunks) + threadIdx.x;
  uint32_t raw[kWconvChunks][2];
#pragma unroll
  for (int u = 0; u < kWconvChunks; ++u) {
    const int i = i0 + u * kWconvThreads;
    raw[u][0] = raw[u][1] = 0u;
    if (i >= total) continue;
    const int r = i / per_row;
    const int j0 = (i - r * per_row) * 8;
    if (j0 >= k) continue;
    const uint32_t *row = wq + (int64_t)r * wpr;
    if constexpr (BITS == 4) {
      raw[u][0] = __ldg(row + j0 / 8);
    } else if constexpr (BITS == 8) {
      raw[u][0] = __ldg(row + j0 / 4);
      raw[u][1] = __ldg(row + j0 / 4 + 1);
    } else {
      // bits 6 j0 .. 6 j0 + 47 lie in words wi, wi + 1 (the shift below is 0 or 16)
      const int64_t wi = ((int64_t)6 * j0) >> 5;
      raw[u][0] = __ldg(row + wi);
      raw[u][1] = __ldg(row + wi + 1);
    }
  }
#pragma unroll
  for (int u = 0; u < kWconvChunks; ++u) {
    const int i = i0 + u * kWconvThreads;
    if (i >= total) continue;
    const int r = i / per_row;
    const int j0 = (i - r * per_row) * 8;
    uint32_t q[8];
    if (j0 < k) {
      if constexpr (BITS == 4) {
#pragma unroll
        for (int e = 0; e < 8; ++e) q[e] = (raw[u][0] >> (4 * e)) & 15u;
      } else if constexpr (BITS == 8) {
#pragma unroll
        for (int e = 0; e < 8; ++e) q[e] = (raw[u][e >> 2] >> (8 * (e & 3))) & 255u;
      } else {
        const int sh = (6 * j0) & 31;
        const uint64_t v = (uint64_t)raw[u][0] | ((uint64_t)raw[u][1] << 32);
#pragma unroll
        for (int e = 0; e < 8; ++e) q[e] = (uint32_t)(v >> (sh + 6 * e)) & 63u;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) q[e] = f32_to_bf16_rn((float)q[e]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int jj = j0 - k + e;
        q[e] = jj < 3 * G ? (uint32_t)biases[(int64_t)r * G + jj % G] : 0u;
      }
    }
    *reinterpret_cast<uint4 *>(A + (int64_t)r * kp + j0) =
        make_uint4(q[0] | (q[1] << 16), q[2] | (q[3] << 16), q[4] | (q[5] << 16), q[6] | (q[7] << 16));
  }
  // The grid ends only after the kernel before it has: one CTA waits for it, the
  // others leave their SMs as soon as their chunks are written.
  if (blockIdx.x == gridDim.x - 1) asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace pg

// ---- host side -----------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

static bool make_map(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t d0, uint64_t d1,
                     uint64_t stride_bytes, uint32_t b0, uint32_t b1, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {d0, d1};
  cuuint64_t strides[1] = {stride_bytes};
  cuuint32_t box[2] = {b0, b1};
  cuuint32_t es[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Library-owned scratch: one growable buffer per device and use (slot 0: the split row
// sums; slot 1: the codes converted once per call for large windows).
constexpr int kMaxDev = 64;
constexpr int kScratchSlots = 3;  // 0: split row sums; 1, 2: converted codes (alternating)
static std::mutex g_scratch_mu;
static void *g_scratch[kScratchSlots][kMaxDev];
static size_t g_scratch_bytes[kScratchSlots][kMaxDev];

static void *scratch_get(int slot, size_t bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_bytes[slot][dev] < bytes) {
    if (g_scratch[slot][dev] != nullptr) {
      // earlier launches may still read the old buffer
      if (cudaDeviceSynchronize() != cudaSuccess) return nullptr;
      cudaFree(g_scratch[slot][dev]);
      g_scratch[slot][dev] = nullptr;
      g_scratch_bytes[slot][dev] = 0;
    }
    size_t cap = bytes < (size_t(1) << 20) ? (size_t(1) << 20) : bytes;
    void *p = nullptr;
    if (cudaMalloc(&p, cap) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    g_scratch[slot][dev] = p;
    g_scratch_bytes[slot][dev] = cap;
  }
  return g_scratch[slot][dev];
}

// SMs of the current device (cached per device)
static int sm_count() {
  static std::atomic<int> cached[kMaxDev];  // per device, 0 until first queried
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 1;
  int c = cached[dev].load(std::memory_order_relaxed);
  if (c == 0) {
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0) c = 1;
    cached[dev].store(c, std::memory_order_relaxed);
  }
  return c;
}

template <int BITS, int EPI>
static int launch_pgemm(const ql_weight *w, const uint16_t *X, int m, int64_t ldx, float *Y, int64_t ldy,
                        const uint16_t *S, int64_t lds, cudaStream_t st, int *status, const PgEpilogue *epi,
                        const uint16_t *apre = nullptr, bool follow = false) {
  using C = pg::Cfg<BITS>;
  const int G = w->k / 64;
  CUtensorMap tmX, tmW, tmS, tmSc, tmBi;
  if (!make_map(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, (uint64_t)w->k, (uint64_t)m, (uint64_t)ldx * 2, pg::BK,
                pg::BMH, CU_TENSOR_MAP_SWIZZLE_128B))
    return QL_ERR_CUDA;
  if constexpr (C::kPre) {
    // the converted codes and bias blocks, bf16 [n][k + lds], boxes of 64 x 128 rows in
    // the 128-byte swizzle the tensor core reads
    const uint64_t kp = (uint64_t)w->k + (uint64_t)lds;
    if (!make_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, apre, kp, (uint64_t)w->n, kp * 2, pg::BK, pg::BN,
                  CU_TENSOR_MAP_SWIZZLE_128B))
      return QL_ERR_CUDA;
  } else {
    if (!make_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, w->wq, (uint64_t)w->k * BITS / 32, (uint64_t)w->n,
                  (uint64_t)w->k * BITS / 8, pg::BK * BITS / 32, pg::BN, CU_TENSOR_MAP_SWIZZLE_NONE))
      return QL_ERR_CUDA;
  }
  if (!make_map(&tmS, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, S, (uint64_t)(3 * G), (uint64_t)m, (uint64_t)lds * 2,
                pg::BK, pg::BMH, CU_TENSOR_MAP_SWIZZLE_128B))
    return QL_ERR_CUDA;
  // scales/biases as TMA boxes of 8 groups when their rows are 16-byte aligned
  const bool sb_ok = (G % 8) == 0 && (reinterpret_cast<uintptr_t>(w->scales) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(w->biases) & 15) == 0;
  const bool sc_tma = sb_ok && make_map(&tmSc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w->scales, (uint64_t)G,
                                        (uint64_t)w->n, (uint64_t)G * 2, 8, pg::BN, CU_TENSOR_MAP_SWIZZLE_NONE);
  const bool bi_tma = !C::kPre && sc_tma && G <= pg::kBiasG &&
                      make_map(&tmBi, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w->biases, (uint64_t)G, (uint64_t)w->n,
                               (uint64_t)G * 2, 8, pg::BN, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!sc_tma) tmSc = tmX;  // never read
  if (!bi_tma) tmBi = tmX;  // never read
  static std::atomic<bool> attr_set[kMaxDev];  // per device; setting the attribute twice is harmless
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < kMaxDev && !attr_set[dev].load(std::memory_order_relaxed)) {
    if (cudaFuncSetAttribute(pg::pgemm_kernel<BITS, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kAlloc) !=
        cudaSuccess)
      return QL_ERR_LAUNCH;
    // The warpgroups' setmaxnreg split assumes that the block is launched with exactly
    // kRegsLaunch registers per thread: with fewer, the epilogue's increase could never
    // be granted.  Refuse to launch a build that differs.
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, pg::pgemm_kernel<BITS, EPI>) != cudaSuccess || fa.numRegs != pg::kRegsLaunch) {
      (void)cudaGetLastError();
      return QL_ERR_LAUNCH;
    }
    attr_set[dev].store(true, std::memory_order_relaxed);
  }
  pg::Params p;
  p.wq = reinterpret_cast<const uint8_t *>(w->wq);
  p.w_row_bytes = C::kPre ? 0 : (int64_t)w->k * BITS / 8;
  p.scales = w->scales;
  p.biases = w->biases;
  p.sc_tma = sc_tma ? 1 : 0;
  p.bi_tma = bi_tma ? 1 : 0;
  p.Y = Y;
  p.ldy = ldy;
  p.A = epi ? epi->a : nullptr;
  p.lda = epi ? epi->lda : 0;
  p.H = epi ? epi->h : nullptr;
  p.ldh = epi ? epi->ldh : 0;
  // the epilogue's input rows start on 16-byte boundaries (every tile's first channel is a
  // multiple of 128): they can be prefetched
  p.epi_pf = 0;
  if (EPI == kPgSwiglu)
    p.epi_pf = (reinterpret_cast<uintptr_t>(p.A) % 16) == 0 && (p.lda % 4) == 0;
  else if (EPI == kPgResid)
    p.epi_pf = (reinterpret_cast<uintptr_t>(p.H) % 16) == 0 && (p.ldh % 8) == 0;
  p.M = m;
  p.N = w->n;
  p.G = G;
  p.NBB = (int)(lds / pg::BK);
  p.status = status;
  p.budget_ns = wait_budget_ns();
  p.follow = follow ? 1 : 0;
  p.tiles_n = (w->n + 2 * pg::BN - 1) / (2 * pg::BN);
  p.tiles = p.tiles_n * ((m + pg::BM - 1) / pg::BM);
  // persistent: one CTA pair per two SMs, as a cluster of two
  const int pairs_max = sm_count() / 2 > 0 ? sm_count() / 2 : 1;
  const int pairs = p.tiles < pairs_max ? p.tiles : pairs_max;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * pairs));
  cfg.blockDim = dim3((unsigned)pg::kThreads);
  cfg.dynamicSmemBytes = (size_t)C::kAlloc;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the CTAs start (barriers, tensor memory, tensor maps,
  // the first weight tiles) while the row-sum pre-pass still runs; X, the row sums and
  // the outputs are touched only after griddepcontrol.wait
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, pg::pgemm_kernel<BITS, EPI>, tmX, tmW, tmS, tmSc, tmBi, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return QL_ERR_LAUNCH;
  }
  return QL_OK;
}

// ---- the same GEMM with a fixed, statically allocated scratch ---------------------
// For callers that must not allocate device memory at call time: code whose device
// memory is owned by another allocator or held to a fixed budget, and code that must
// not stall on the device-wide synchronization that growing (freeing and
// reallocating) a scratch buffer costs.  The split row sums then live in this
// file-scope array instead of the library's growable buffer.  Every GPU that loads
// the library holds the array until the process exits.
constexpr int64_t kNoAllocScratchElems = int64_t(1) << 20;  // 1,048,576 bf16 values = 2 MiB
static __device__ __align__(256) uint16_t g_noalloc_scratch[kNoAllocScratchElems];

static std::mutex g_noalloc_mu;
static uint16_t *g_noalloc_addr[kMaxDev];

// Device address of the static array for the current device.  The name of a
// __device__ array in host code is only a host-side stand-in, so the address is
// looked up once per device, with that device current, and cached.
static int noalloc_scratch_addr(uint16_t **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return QL_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      (void)cudaGetLastError();
      return QL_ERR_CUDA;
    }
    g_noalloc_addr[dev] = static_cast<uint16_t *>(p);
  }
  *out = g_noalloc_addr[dev];
  return QL_OK;
}

int64_t pgemm_noalloc_max_elems() { return kNoAllocScratchElems; }

// The row-sum pre-pass over m rows, launched with programmatic dependent launch (the
// kernel waits for the kernel before it before it touches X or the sums).
static int launch_xsum(const uint16_t *X, int m, int G, int64_t ldx, uint16_t *S, int64_t lds, cudaStream_t st) {
  const int64_t total = (int64_t)m * G;
  if (total >= (int64_t(1) << 31)) return QL_ERR_TOO_LARGE;
  // at most one wave of CTAs (resident CTAs per SM, by the kernel's shared memory)
  static std::atomic<int> per_sm{0};
  int occ = per_sm.load(std::memory_order_relaxed);
  if (occ == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, pg::xsum_split_kernel, pg::kXsumPairs, 0) !=
            cudaSuccess ||
        occ <= 0) {
      (void)cudaGetLastError();
      occ = 1;
    }
    per_sm.store(occ, std::memory_order_relaxed);
  }
  const int64_t tiles = (total + pg::kXsumPairs - 1) / pg::kXsumPairs;
  const int64_t wave = (int64_t)occ * sm_count();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles < wave ? tiles : wave));
  cfg.blockDim = dim3((unsigned)pg::kXsumPairs);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, pg::xsum_split_kernel, X, m, G, ldx, S, lds) != cudaSuccess) {
    (void)cudaGetLastError();
    return QL_ERR_LAUNCH;
  }
  return QL_OK;
}

int pgemm_run_noalloc(const ql_weight *w, const uint16_t *X, int m, int64_t ldx, float *Y, int64_t ldy,
                      cudaStream_t st, int *status) {
  const int G = w->k / 64;
  const int64_t lds = ((3 * (int64_t)G + 63) / 64) * 64;
  if ((int64_t)m * lds > kNoAllocScratchElems) return QL_ERR_TOO_LARGE;
  uint16_t *S = nullptr;
  int e = noalloc_scratch_addr(&S);
  if (e) return e;
  // every scratch value the GEMM reads is written by this pre-pass first, so nothing
  // left by an earlier call needs clearing
  if (int e2 = launch_xsum(X, m, G, ldx, S, lds, st)) return e2;
  switch (w->bits) {
    case 4: return launch_pgemm<4, kPgStore>(w, X, m, ldx, Y, ldy, S, lds, st, status, nullptr);
    case 6: return launch_pgemm<6, kPgStore>(w, X, m, ldx, Y, ldy, S, lds, st, status, nullptr);
    default: return launch_pgemm<8, kPgStore>(w, X, m, ldx, Y, ldy, S, lds, st, status, nullptr);
  }
}

template <int BITS>
static int launch_epi(const ql_weight *w, const uint16_t *X, int m, int64_t ldx, float *Y, int64_t ldy,
                      const uint16_t *S, int64_t lds, cudaStream_t st, int *status, const PgEpilogue *epi,
                      const uint16_t *apre = nullptr, bool follow = false) {
  switch (epi ? epi->mode : kPgStore) {
    case kPgSwiglu: return launch_pgemm<BITS, kPgSwiglu>(w, X, m, ldx, Y, ldy, S, lds, st, status, epi, apre, follow);
    case kPgResid: return launch_pgemm<BITS, kPgResid>(w, X, m, ldx, Y, ldy, S, lds, st, status, epi, apre, follow);
    default: return launch_pgemm<BITS, kPgStore>(w, X, m, ldx, Y, ldy, S, lds, st, status, epi, apre, follow);
  }
}

// From this many rows on, the codes are converted once per call (wconv_kernel) and the
// GEMM loads them ready (Cfg<0>): the conversion then costs one pass over W instead of
// one per 256-row band.  Smaller windows convert inside the GEMM.  Both give the same bits.
constexpr int kPreRows = 2048;

// Per device, how many calls have converted their codes (the parity picks the buffer).
static unsigned apre_flip(int dev) {
  static std::atomic<unsigned> calls[kMaxDev];
  return calls[dev].fetch_add(1u, std::memory_order_relaxed);
}

// From kPreRows rows on (and while the converted codes stay below 2^31 chunks), the call
// converts its codes once into one of two alternating buffers (wconv_kernel, launched
// with programmatic dependent launch so that it may run in the previous GEMM's last
// tiles) and sets *apre; otherwise *apre stays null and the GEMM converts in the kernel.
static int pgemm_convert(const ql_weight *w, int m, int64_t lds, cudaStream_t st, uint16_t **apre) {
  *apre = nullptr;
  if (m < kPreRows || (int64_t)w->n * (((int64_t)w->k + lds) / 8) >= (int64_t(1) << 31)) return QL_OK;
  const int64_t kp = (int64_t)w->k + lds;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return QL_ERR_LAUNCH;
  // Consecutive calls write alternate buffers: this call's conversion may run while
  // the previous call's GEMM (reading the other buffer) finishes.
  const int slot = 1 + (int)(apre_flip(dev) & 1u);
  uint16_t *a = static_cast<uint16_t *>(scratch_get(slot, (size_t)w->n * (size_t)kp * 2));
  if (a == nullptr) return QL_ERR_NOMEM;
  const int64_t chunks = (int64_t)w->n * (kp / 8);
  constexpr int per_block = pg::kWconvThreads * pg::kWconvChunks;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((chunks + per_block - 1) / per_block));
  cfg.blockDim = dim3((unsigned)pg::kWconvThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t ce;
  switch (w->bits) {
    case 4: ce = cudaLaunchKernelEx(&cfg, pg::wconv_kernel<4>, w->wq, w->biases, w->n, w->k, kp, a); break;
    case 6: ce = cudaLaunchKernelEx(&cfg, pg::wconv_kernel<6>, w->wq, w->biases, w->n, w->k, kp, a); break;
    default: ce = cudaLaunchKernelEx(&cfg, pg::wconv_kernel<8>, w->wq, w->biases, w->n, w->k, kp, a); break;
  }
  if (ce != cudaSuccess) {
    (void)cudaGetLastError();
    return QL_ERR_LAUNCH;
  }
  *apre = a;
  return QL_OK;
}

// The GEMM of one weight on split row sums S already enqueued (pre-converted codes if
// apre is set).
static int pgemm_launch(const ql_weight *w, const uint16_t *X, int m, int64_t ldx, float *Y, int64_t ldy,
                        const uint16_t *S, int64_t lds, cudaStream_t st, int *status, const PgEpilogue *epi,
                        const uint16_t *apre, bool follow) {
  if (apre != nullptr) return launch_epi<0>(w, X, m, ldx, Y, ldy, S, lds, st, status, epi, apre);
  switch (w->bits) {
    case 4: return launch_epi<4>(w, X, m, ldx, Y, ldy, S, lds, st, status, epi, nullptr, follow);
    case 6: return launch_epi<6>(w, X, m, ldx, Y, ldy, S, lds, st, status, epi, nullptr, follow);
    default: return launch_epi<8>(w, X, m, ldx, Y, ldy, S, lds, st, status, epi, nullptr, follow);
  }
}

int pgemm_run(const ql_weight *w, const uint16_t *X, int m, int64_t ldx, float *Y, int64_t ldy, cudaStream_t st,
              int *status, const PgEpilogue *epi) {
  return pgemm_run_multi(&w, 1, X, m, ldx, &Y, &ldy, st, status, epi);
}

int pgemm_run_multi(const ql_weight *const *w, int nw, const uint16_t *X, int m, int64_t ldx, float *const *Y,
                    const int64_t *ldy, cudaStream_t st, int *status, const PgEpilogue *epi) {
  const int G = w[0]->k / 64;
  const int64_t lds = ((3 * (int64_t)G + 63) / 64) * 64;  // row pitch of the split sums (elements)
  if ((int64_t)m * G >= (int64_t(1) << 31)) return QL_ERR_TOO_LARGE;
  uint16_t *S = static_cast<uint16_t *>(scratch_get(0, (size_t)m * lds * 2));
  if (S == nullptr) return QL_ERR_NOMEM;
  // The first weight's conversion goes before the row sums, so that it can start in the
  // previous call's last tiles (the row sums must wait for the kernel before them).
  uint16_t *apre = nullptr;
  if (int e = pgemm_convert(w[0], m, lds, st, &apre)) return e;
  if (int e = launch_xsum(X, m, G, ldx, S, lds, st)) return e;
  for (int i = 0; i < nw; ++i) {
    if (i > 0)
      if (int e = pgemm_convert(w[i], m, lds, st, &apre)) return e;
    // below the pre-conversion size the later GEMMs run beside the ones before them
    const bool follow = i > 0 && m < kPreRows;
    if (int e = pgemm_launch(w[i], X, m, ldx, Y[i], ldy[i], S, lds, st, status, epi, apre, follow)) return e;
  }
  return QL_OK;
}

}  // namespace qlk
