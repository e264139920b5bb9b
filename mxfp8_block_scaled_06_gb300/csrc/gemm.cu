// gemm.cu - low-batch MXFP8 block-scaled GEMM on tcgen05 (sm_103a).
//
// out[M, N] = dequant(A[M, K]) x dequant(W[N, K])^T, bf16 out, fp32 accumulate.
//
// Swap-AB: the 128 weight rows of a tile are the MMA's M (the only M the
// block-scaled tcgen05.mma takes with one CTA) and the activation rows,
// padded to a multiple of 16, are the MMA's N, so 1..256 rows cost one MMA
// shape. The kernel is bound by the weight stream from HBM and by fixed
// latencies; everything below is arranged around those:
//  * grid = (N/128 weight tiles) x (K splits); the splits of one tile form a
//    thread-block cluster and reduce their partial sums through distributed
//    shared memory (no global workspace, no second kernel); the split count and
//    ring depth come from plan_gemm (a measured table for the decode shapes);
//  * copies issued by one thread are serviced one after another, so each ring
//    stage has its own issuing lane: warp 0 streams the 128x128-byte weight
//    boxes (SWIZZLE_128B), the first ring-full before the programmatic
//    grid-dependency wait; warp 3 the activation boxes after it (they are the
//    previous kernel's output); warp 2 the scale tiles of the whole K-range,
//    one bulk copy per operand; refills come from warp-uniform loops whose
//    issuing lane rotates;
//  * the MMA warp walks the chunks warp-uniformly and an elected lane issues
//    tcgen05.cp (scales -> TMEM) and four tcgen05.mma.kind::mxf8f6f4.block_scale
//    (K = 32 each) per chunk, with the smem descriptors advanced by 32-bit adds
//    (that one thread's instruction latency bounds the loop), then frees the
//    stage with tcgen05.commit;
//  * the four warps read the fp32 accumulator from TMEM (warp w owns lanes
//    32w..32w+31 = weight rows) and the split-K partials are summed over the
//    cluster in rank order: up to 16 rows every CTA pushes the partials of the
//    outputs another rank owns into that rank's shared memory (st.async,
//    counted on the owner's mbarrier; no cluster barrier after the MMAs), above
//    they are staged in shared memory and, after a cluster barrier, read by the
//    owning warp from every peer; each (row, 32-column block) is summed by one
//    warp, and the optional fused requantization (the chain's next MXFP8
//    activation) takes its 32 values as one block; a relaxed cluster barrier
//    keeps every CTA alive until its peers are done with its shared memory.
// Variants: bf16 activations quantized in the prologue into resident operand
// tiles (kFusedA), and grouped activations (weight tile t contracts the K-slice
// of its group of a wider activation).
// Every mbarrier wait is bounded; on expiry the kernel records MX_ERR_TIMEOUT,
// skips the remaining work, drains its outstanding copies and frees TMEM.
#include <cuda_bf16.h>

#include <algorithm>
#include <type_traits>

#include <cstdio>

#include "kernels.h"
#include "ptx.cuh"
#include "push.cuh"

namespace mx {
namespace {

constexpr int kThreads = 128;

// Timeline build (-DMX_TIMELINE): %globaltimer stamps of one CTA's phases,
// written to p.tl[cta * kTimelineSlots + slot]: 0 entry, 1 set-up done, 2 first
// weight box issued, 3 weight scale tiles landed, 4 grid-dependency wait
// returned, 5 first chunk landed, 6 accumulator complete, 7 reduction barrier
// passed, 8 reduction done, 9 exit, 10 SM id, 11 chunks in the K-range,
// 12 bf16 activations quantized, 13 RMS of the rows done, 14 first row batch
// landed (12-14: in-kernel quantization only), 15 last chunk landed, 16 every
// MMA issued, 17 ring stages already landed when the wait returned (a count),
// 18 second chunk landed.
#ifdef MX_TIMELINE
#define MX_TL(slot, v)                                                             \
  do {                                                                             \
    if (p.tl != nullptr)                                                           \
      p.tl[(blockIdx.y * gridDim.x + blockIdx.x) * kTimelineSlots + (slot)] = (v); \
  } while (0)
__device__ __forceinline__ unsigned long long tl_smid() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}
#else
#define MX_TL(slot, v) \
  do {                 \
  } while (0)
#endif
constexpr uint32_t kWTileBytes = 128 * 128;  // one weight box: 128 rows x 128 K-bytes
constexpr uint32_t kSfTileBytes = 512;       // one 128x4 scale tile

// Shared-memory carve-up of one CTA: a ring of `stages` (weight box, activation
// box) pairs, then the weight and activation scale tiles of the CTA's whole
// K-range (loaded once), then the mbarriers. With bf16 activations quantized in
// the kernel (`fused`), the ring holds weight boxes only and the activation
// tiles of the whole K-range are resident, after the scale tiles, followed by a
// staging area for up to kRowBatch bf16 rows of the K-range. With the RMS norm
// (norm_blocks = K/32) follow the norm weight's K-range, the staged rows'
// per-block sums of squares and the rows' reciprocal RMS (a float per tile row).
// Then the mbarriers, and with the push reduction the area where the peers'
// partials arrive (apart from the ring: a slower peer's MMAs may still be
// reading its ring when this CTA's partials reach it).
constexpr int kRowBatch = 32;
constexpr int kRedRows = 4;  // rows a warp reduces at once in the several-rows epilogue
struct Layout {
  uint32_t a_bytes, stage_bytes, ring_bytes, sfa_bytes, sfb_bytes, act, xraw, gam, ssq, inv, bars;
  uint32_t red_bar, red, red_bytes;
  int stages, nsfb, nmax;
  __host__ __device__ Layout(int mtile, int stages_, int nmax_, bool fused = false, int xrows = 0,
                             int norm_blocks = 0, uint32_t red_bytes_ = 0) {
    stages = stages_;
    nmax = nmax_;
    nsfb = (mtile + 127) / 128;
    a_bytes = static_cast<uint32_t>(mtile) * 128u;
    stage_bytes = fused ? kWTileBytes : (kWTileBytes + a_bytes + 1023u) & ~1023u;
    ring_bytes = static_cast<uint32_t>(stages) * stage_bytes;
    sfa_bytes = static_cast<uint32_t>(nmax) * kSfTileBytes;
    sfb_bytes = static_cast<uint32_t>(nmax * nsfb) * kSfTileBytes;
    act = (ring_bytes + sfa_bytes + sfb_bytes + 1023u) & ~1023u;
    xraw = act + (fused ? static_cast<uint32_t>(nmax) * a_bytes : 0u);
    gam = xraw + (fused ? static_cast<uint32_t>(xrows * nmax) * 256u : 0u);
    const bool norm = fused && norm_blocks > 0;
    ssq = gam + (norm ? static_cast<uint32_t>(nmax) * 256u : 0u);
    inv = ssq + (norm ? static_cast<uint32_t>(xrows * norm_blocks) * 4u : 0u);
    bars = inv + (norm ? static_cast<uint32_t>(mtile) * 4u : 0u);
    red_bar = bars + 8u * (2 * stages + 4) + 8u;
    red = (bars + bar_bytes() + 127u) & ~127u;
    red_bytes = red_bytes_;
  }
  __host__ __device__ uint32_t w_off(int s) const { return s * stage_bytes; }
  __host__ __device__ uint32_t a_off(int s) const { return s * stage_bytes + kWTileBytes; }
  __host__ __device__ uint32_t sfa_off(int i) const { return ring_bytes + i * kSfTileBytes; }
  __host__ __device__ uint32_t sfb_off(int rt, int i) const {
    return ring_bytes + sfa_bytes + (rt * nmax + i) * kSfTileBytes;
  }
  // full[stages], empty[stages], sfa, sfb, accum, x; then TMEM slot and abort
  // flag; then the push reduction's receive barrier
  __host__ __device__ uint32_t bar_bytes() const { return 8u * (2 * stages + 4) + 16u; }
  __host__ __device__ size_t total() const { return 1024 + (red_bytes ? red + red_bytes : bars + bar_bytes()); }
};

__host__ __device__ inline int tmem_sfa_col(int mtile) { return (mtile + 15) & ~15; }

// Whether the epilogue reduces whole rows per warp (16-byte peer loads) rather
// than 32-column items: measured on GB300, 3-4x faster with two or three K-splits
// once a warp has two or more rows (N = 8192, K = 5120, M = 128: 9.5 -> 3.0 us),
// no faster with six (N = 5120, K = 8192, M = 192: 6.5 -> 6.4 us); the peer loads
// of up to four ranks are issued together.
inline bool row_reduction(int M, int splits) { return splits <= 4 && M >= 8 * splits; }

// The 64 bytes at src (shared memory) into w[0..15] in order, read as four
// 16-byte loads that start at granule rot (0..3): threads that differ in rot
// hit different banks. The rotation is undone with selects, so every register
// index is a compile-time constant.
__device__ __forceinline__ void load_block64(const uint8_t* src, int rot, uint32_t (&w)[16]) {
  uint4 r[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) r[j] = *reinterpret_cast<const uint4*>(src + ((j + rot) & 3) * 16);
  // r[j] holds granule (j + rot) & 3: granule q is r[(q - rot) & 3]
  if (rot & 1) {
    const uint4 t = r[3];
    r[3] = r[2];
    r[2] = r[1];
    r[1] = r[0];
    r[0] = t;
  }
  if (rot & 2) {
    uint4 t = r[0];
    r[0] = r[2];
    r[2] = t;
    t = r[1];
    r[1] = r[3];
    r[3] = t;
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    w[4 * q] = r[q].x;
    w[4 * q + 1] = r[q].y;
    w[4 * q + 2] = r[q].z;
    w[4 * q + 3] = r[q].w;
  }
}

// kRed: how the K-splits' partials are summed (Reduction).
template <bool kRequant, bool kFusedA, int kRed>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_a,
                const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw_addr);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tile = blockIdx.x;
  const int S = gridDim.y;
  const int split = blockIdx.y;
  const int c_begin = split * p.nchunks / S;
  const int n = (split + 1) * p.nchunks / S - c_begin;
  const int stages = p.stages;
  // grouped activations: this tile's group reads its own K-slice of A
  const int a_k0 = p.group_tiles > 0 ? (tile / p.group_tiles) * p.K : 0;
  const bool norm = kFusedA && p.norm.gamma != nullptr;
  constexpr bool kPush = kRed == kReducePush || kRed == kReducePushCompact;
  constexpr bool compact = kRed == kReducePushCompact;
  const PushGeometry pgeo(p.M, kPush ? S : 1, kPush ? split : 0);
  const uint32_t slot = pgeo.slot;
  const Layout L(p.mtile, stages, (p.nchunks + S - 1) / S, kFusedA, min(p.M, kRowBatch),
                 norm ? p.K / 32 : 0, kPush ? push_area_bytes(p.M, S, compact) : 0u);
  const int nsfb = L.nsfb;
  // Whether anything consumes the output columns of the tile's 32-column block
  // q: a block nobody consumes (no bf16 output, outside the requantized and the
  // summed-square columns) is not reduced.
  auto want_q = [&](int q) {
    return p.out != nullptr || (kRequant && tile * 128 + q * 32 < p.q_cols) ||
           (p.ssq_out != nullptr && tile * 128 + q * 32 < p.ssq_cols);
  };
  if (threadIdx.x == 0) MX_TL(0, globaltimer());

  const uint32_t bars = base + L.bars;
  // full(s): weight box and activation box of stage s landed (two arrivals);
  // empty(s): the MMAs reading stage s completed
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (stages + s); };
  const uint32_t sfa_bar = bars + 16u * stages;
  const uint32_t sfb_bar = sfa_bar + 8u;
  const uint32_t accum_bar = sfa_bar + 16u;
  const uint32_t x_bar = sfa_bar + 24u;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + L.bars + 8 * (2 * stages + 4));
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full(s), kFusedA ? 1 : 2);
      mbar_init(empty(s), 1);
    }
    mbar_init(sfa_bar, 1);
    mbar_init(sfb_bar, 1);
    mbar_init(accum_bar, 1);
    mbar_init(x_bar, 1);
    mbar_init(base + L.red_bar, 1);
    if constexpr (kPush) {
      // armed now with the bytes the S - 1 peers will store for this rank's
      // wanted units (the peers start storing after the cluster barrier below)
      mbar_expect_tx(base + L.red_bar, push_expect_bytes(pgeo, want_q));
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_w);
    if (!kFusedA) prefetch_tmap(&tm_a);
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // push reduction: the receive barriers of the whole cluster are initialised
  // and armed before any peer stores to them (the wait is in the epilogue)
  if constexpr (kPush) cluster_arrive_release();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sfa_col = tmem_sfa_col(p.mtile);
  const uint32_t sfb_col = sfa_col + 4 * stages;
  if (threadIdx.x == 0) MX_TL(1, globaltimer());

  auto fail = [&]() {
    atomicOr(p.status, kStatusTimeout);
    *abort_flag = 1;
  };

  // Copies issued by one thread are serviced one after another, so each ring
  // stage has its own issuing lane: lane s of warp 0 streams the weight boxes of
  // stage s, lane s of warp 3 the activation boxes, and warp 2 loads the scale
  // tiles of the whole K-range with one bulk copy per operand.
  const uint64_t pol_w = policy_evict_first();
  const uint64_t pol_a = policy_evict_last();
  const bool w_lane = warp == 0 && lane < stages;
  const bool a_lane = !kFusedA && warp == 3 && lane < stages;
  int last = -1;      // last chunk this lane loaded (weight or activation warps)
  int issued_n = 0;   // chunks its warp has loaded so far (warp-uniform)
  auto issue_w = [&](int i, int s) {
    mbar_expect_tx(full(s), kWTileBytes);
    tma_load_2d(base + L.w_off(s), &tm_w, full(s), (c_begin + i) * 128, tile * 128, pol_w);
    last = i;
  };
  auto issue_a = [&](int i, int s) {
    mbar_expect_tx(full(s), L.a_bytes);
    tma_load_2d(base + L.a_off(s), &tm_a, full(s), a_k0 + (c_begin + i) * 128, 0, pol_a);
    last = i;
  };

  // ---------------- before the grid-dependency wait: weights only
  if (w_lane && lane < n) issue_w(lane, lane);
  if (warp == 0) issued_n = min(n, stages);
  if (warp == 0 && lane == 0) MX_TL(2, globaltimer());
  if (warp == 2 && lane == 0) {
    mbar_expect_tx(sfa_bar, static_cast<uint32_t>(n) * kSfTileBytes);
    bulk_load(base + L.sfa_off(0),
              p.w_scales + (static_cast<size_t>(tile) * p.nchunks + c_begin) * kSfTileBytes,
              static_cast<uint32_t>(n) * kSfTileBytes, sfa_bar, pol_w);
  }
  pdl_launch_dependents();
#ifdef MX_TIMELINE
  // the MMA warp, which has nothing to do before the grid-dependency wait,
  // watches the weight scale tiles land (a non-consuming wait); a lane of a warp
  // whose other lanes sit in griddepcontrol.wait could not record before it returns
  if (warp == 1 && mbar_wait(sfa_bar, 0) && lane == 0) MX_TL(3, globaltimer());
  if (threadIdx.x == 0) MX_TL(10, tl_smid());
  if (threadIdx.x == 0) MX_TL(11, static_cast<unsigned long long>(n));
#endif
  // In-kernel quantization: each 32-block of a row batch is split over tpb
  // threads (a power of two up to 8, as many as the CTA's threads allow for the
  // first batch, so a few rows still spread over the CTA); a thread's first
  // (row, block) of a batch and its stride, worked out here, before the wait,
  // where the divisions cost nothing (the empty asm keeps them here).
  int q_tpb = 1, q_row0 = 0, q_blk0 = 0, q_drow = 0, q_dblk = 0;
  if constexpr (kFusedA) {
    const int bpr = n * 4;
    const int total0 = min(p.M, kRowBatch) * bpr;
    q_tpb = total0 * 8 <= kThreads ? 8 : total0 * 4 <= kThreads ? 4 : total0 * 2 <= kThreads ? 2 : 1;
    const int w = static_cast<int>(threadIdx.x) / q_tpb, dw = kThreads / q_tpb;
    q_row0 = w / bpr;
    q_blk0 = w - q_row0 * bpr;
    q_drow = dw / bpr;
    q_dblk = dw - q_drow * bpr;
    asm volatile("" : "+r"(q_tpb), "+r"(q_row0), "+r"(q_blk0), "+r"(q_drow), "+r"(q_dblk));
  }
  if constexpr (kFusedA) {
    // shared memory only, so before the wait: zero rows [M, mtile) of every
    // activation chunk tile, and the activation scale tiles
    for (int idx = threadIdx.x; idx < n * (p.mtile - p.M) * 8; idx += kThreads) {
      const int i = idx / ((p.mtile - p.M) * 8), rem = idx % ((p.mtile - p.M) * 8);
      const int m = p.M + rem / 8;
      *reinterpret_cast<uint4*>(base_ptr + L.act + i * L.a_bytes + m * 128 + (rem % 8) * 16) =
          make_uint4(0, 0, 0, 0);
    }
    for (int idx = threadIdx.x; idx < n * nsfb * 32; idx += kThreads)
      *reinterpret_cast<uint4*>(base_ptr + L.sfb_off(idx / (n * 32), 0) + (idx % (n * 32)) * 16) =
          make_uint4(0, 0, 0, 0);
    // every zero is stored before any thread writes the quantized activation
    // (after the wait) over the same bytes
    __syncthreads();
  }
  pdl_wait();
  if (threadIdx.x == 0) MX_TL(4, globaltimer());
#ifdef MX_TIMELINE
  // ring stages whose copies had all landed when the wait returned
  if (warp == 1 && lane == 0) {
    unsigned long long landed = 0;
    for (int s = 0; s < min(n, stages); ++s) landed += mbar_test_wait(full(s), 0) ? 1 : 0;
    MX_TL(17, landed);
  }
#endif

  // ---------------- activations (written by the previous kernel on the stream)
  int x_batches = 0;  // bf16 row batches requested (fused), warp 3
  if constexpr (!kFusedA) {
    if (a_lane && lane < n) issue_a(lane, lane);
    if (warp == 3) issued_n = min(n, stages);
    if (warp == 2 && lane == 1) {
      mbar_expect_tx(sfb_bar, static_cast<uint32_t>(n * nsfb) * kSfTileBytes);
      for (int rt = 0; rt < nsfb; ++rt)
        bulk_load(base + L.sfb_off(rt, 0),
                  p.a_scales + (static_cast<size_t>(rt) * p.a_sf_chunks + a_k0 / 128 + c_begin) *
                                   kSfTileBytes,
                  static_cast<uint32_t>(n) * kSfTileBytes, sfb_bar, pol_a);
    }
  } else {
    // bf16 rows of the CTA's K-range -> MXFP8 codes in the 128-byte-swizzled
    // K-major operand layout and the 128x4 scale tiles, in shared memory (rows
    // [M, mtile) and the scale tiles were zeroed before the wait)
    const uint32_t at = L.a_bytes;
    float* const row_inv = reinterpret_cast<float*>(base_ptr + L.inv);
    const bool norm_out = norm && tile == 0;  // tile 0 writes y and the activation
    const int nblk = p.K >> 5;                // 32-blocks of a whole row (the norm's sum)
    const int blocks_per_row = n * 4;         // 32-blocks in the K-range
    for (int r0 = 0, batch = 0; r0 < p.M; r0 += kRowBatch, ++batch) {
      // every thread reads the flag after the previous batch's barrier: once a
      // wait has expired no further row batch is requested
      if (*abort_flag != 0) break;
      const int rb = min(kRowBatch, p.M - r0);
      const bool gam = norm && batch == 0;  // the norm weight's K-range comes with batch 0
      if (warp == 3) {
        // one lane per row: each row's K-range is contiguous; with the norm, lane
        // 31 also copies the batch's block sums of squares (contiguous rows), and
        // lane 30 the norm weight's K-range with the first batch
        const uint32_t ssq_bytes = static_cast<uint32_t>(rb * nblk) * 4u;
        if (lane == 0)
          mbar_expect_tx(x_bar, static_cast<uint32_t>(rb * n) * 256u + (norm ? ssq_bytes : 0u) +
                                    (gam ? static_cast<uint32_t>(n) * 256u : 0u));
        __syncwarp();
        if (lane < rb)
          bulk_load(base + L.xraw + lane * L.nmax * 256,
                    p.x + static_cast<size_t>(r0 + lane) * p.ldx + static_cast<size_t>(c_begin) * 128,
                    static_cast<uint32_t>(n) * 256u, x_bar, pol_a);
        if (norm && lane == 31)
          bulk_load(base + L.ssq, p.norm.ssq + static_cast<size_t>(r0) * nblk, ssq_bytes, x_bar, pol_a);
        if (gam && lane == 30)
          bulk_load(base + L.gam, p.norm.gamma + static_cast<size_t>(c_begin) * 128,
                    static_cast<uint32_t>(n) * 256u, x_bar, pol_a);
        x_batches = batch + 1;
      }
      if (gam && norm_out && p.norm.a_q_scales != nullptr) {
        // padding rows [M, ceil128(M)) of the K-range's scale columns
        const int mpad = (p.M + 127) & ~127;
        for (int idx = threadIdx.x; idx < (mpad - p.M) * n * 4; idx += kThreads)
          p.norm.a_q_scales[swz_offset(p.M + idx / (n * 4), c_begin * 4 + idx % (n * 4), nblk)] = 0;
      }
      if (!mbar_wait(x_bar, batch & 1)) fail();
      if (batch == 0 && threadIdx.x == 0) MX_TL(14, globaltimer());
      if (norm) {
        // reciprocal RMS of the batch's rows, one thread per row: the blocks'
        // sums of squares added in block order, as the stand-alone norm kernel does
        if (threadIdx.x < rb) {
          const float* const sq = reinterpret_cast<const float*>(base_ptr + L.ssq) + threadIdx.x * nblk;
          float ss = 0.f;
#pragma unroll 8
          for (int b = 0; b < nblk; ++b) ss = __fadd_rn(ss, sq[b]);
          row_inv[r0 + threadIdx.x] =
              __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(p.K)), p.norm.eps)));
        }
        __syncthreads();
        if (batch == 0 && threadIdx.x == 0) MX_TL(13, globaltimer());
      }
      // tpb threads per 32-block, vpt = 32 / tpb consecutive values each: the
      // block's amax by an xor-shuffle over its aligned group of tpb lanes (a
      // maximum, so the same bits for any split), then each thread's codes
      const int total = rb * blocks_per_row;
      const bool go = *abort_flag == 0;
      auto blocks = [&](auto tpb_c) {
        constexpr int TPB = decltype(tpb_c)::value;
        constexpr int VPT = 32 / TPB;  // values per thread
        constexpr int WPT = VPT / 2;   // 32-bit words (bf16 pairs) per thread
        const int sub = static_cast<int>(threadIdx.x) & (TPB - 1);
        int row = q_row0, blk = q_blk0;
        for (int b0 = 0; go && b0 < total; b0 += kThreads / TPB) {
          const bool act = b0 + static_cast<int>(threadIdx.x) / TPB < total;  // uniform over the group
          const int m = r0 + row;
          const int kg = c_begin * 128 + blk * 32 + sub * VPT;  // the thread's first column of K
          uint32_t xw[WPT];
          if (act) {
            const uint4* const src =
                reinterpret_cast<const uint4*>(base_ptr + L.xraw + row * L.nmax * 256 + blk * 64 + sub * VPT * 2);
            if constexpr (WPT == 16) {
              // a whole block per thread: its four 16-byte loads start at a
              // rotated one (pairs of threads), so a warp's loads spread over all banks
              load_block64(reinterpret_cast<const uint8_t*>(src), (threadIdx.x >> 1) & 3, xw);
            } else if constexpr (WPT >= 4) {
#pragma unroll
              for (int q = 0; q < WPT / 4; ++q) {
                const uint4 t = src[q];
                xw[4 * q] = t.x;
                xw[4 * q + 1] = t.y;
                xw[4 * q + 2] = t.z;
                xw[4 * q + 3] = t.w;
              }
            } else {
              const uint2 t = *reinterpret_cast<const uint2*>(src);
              xw[0] = t.x;
              xw[1] = t.y;
            }
          } else {
#pragma unroll
            for (int e = 0; e < WPT; ++e) xw[e] = 0;
          }
          float v[VPT];
#pragma unroll
          for (int e = 0; e < WPT; ++e) {
            v[2 * e] = __uint_as_float(xw[e] << 16);
            v[2 * e + 1] = __uint_as_float(xw[e] & 0xFFFF0000u);
          }
          if (norm && act) {
            // y = bf16((x * inv_rms) * gamma), as the stand-alone norm kernel
            const float inv = row_inv[m];
            uint32_t gw[WPT];
            const uint8_t* const gsrc = base_ptr + L.gam + blk * 64 + sub * VPT * 2;
            if constexpr (WPT == 16) {
              load_block64(gsrc, (threadIdx.x >> 1) & 3, gw);
            } else if constexpr (WPT >= 4) {
#pragma unroll
              for (int q = 0; q < WPT / 4; ++q) {
                const uint4 t = reinterpret_cast<const uint4*>(gsrc)[q];
                gw[4 * q] = t.x;
                gw[4 * q + 1] = t.y;
                gw[4 * q + 2] = t.z;
                gw[4 * q + 3] = t.w;
              }
            } else {
              const uint2 t = *reinterpret_cast<const uint2*>(gsrc);
              gw[0] = t.x;
              gw[1] = t.y;
            }
#pragma unroll
            for (int e = 0; e < WPT; ++e) {
              const float a = __fmul_rn(__fmul_rn(v[2 * e], inv), __uint_as_float(gw[e] << 16));
              const float b = __fmul_rn(__fmul_rn(v[2 * e + 1], inv), __uint_as_float(gw[e] & 0xFFFF0000u));
              const uint32_t ha = __bfloat16_as_ushort(__float2bfloat16_rn(a));
              const uint32_t hb = __bfloat16_as_ushort(__float2bfloat16_rn(b));
              xw[e] = ha | (hb << 16);
              v[2 * e] = __uint_as_float(ha << 16);
              v[2 * e + 1] = __uint_as_float(hb << 16);
            }
            if (norm_out && p.norm.y != nullptr) {
              uint32_t* const dst = reinterpret_cast<uint32_t*>(p.norm.y + static_cast<size_t>(m) * p.K + kg);
              if constexpr (WPT >= 4) {
#pragma unroll
                for (int q = 0; q < WPT / 4; ++q)
                  reinterpret_cast<uint4*>(dst)[q] =
                      make_uint4(xw[4 * q], xw[4 * q + 1], xw[4 * q + 2], xw[4 * q + 3]);
              } else {
                *reinterpret_cast<uint2*>(dst) = make_uint2(xw[0], xw[1]);
              }
            }
          }
          // max |v| as bits: at or above Inf's bits when any value is Inf or NaN
          uint32_t amax_bits = 0;
#pragma unroll
          for (int e = 0; e < VPT; ++e) amax_bits = max(amax_bits, __float_as_uint(v[e]) & 0x7FFFFFFFu);
#pragma unroll
          for (int o = 1; o < TPB; o <<= 1) amax_bits = max(amax_bits, __shfl_xor_sync(0xFFFFFFFFu, amax_bits, o));
          uint32_t sbyte;
          uint32_t cw[VPT / 4];
          if (amax_bits >= 0x7F800000u) {
            sbyte = 0xFFu;
#pragma unroll
            for (int c = 0; c < VPT / 4; ++c) cw[c] = 0x7F7F7F7Fu;
          } else {
            sbyte = mx_scale_byte(__uint_as_float(amax_bits));
            const float f = mx_inv_scale(sbyte);
#pragma unroll
            for (int c = 0; c < VPT / 4; ++c)
              cw[c] = cvt_e4m3x2(v[4 * c] * f, v[4 * c + 1] * f) |
                      (cvt_e4m3x2(v[4 * c + 2] * f, v[4 * c + 3] * f) << 16);
          }
          if (act) {
            // the thread's VPT codes in the chunk tile's 128-byte row m, whose
            // 16-byte granules are swizzled by m % 8: bytes [c, c + VPT) of the
            // row, c = 32 (blk % 4) + sub VPT
            const int ci = blk >> 2;
            const int c = (blk & 3) * 32 + sub * VPT;
            const uint32_t rowoff = ci * at + (m >> 3) * 1024 + (m & 7) * 128;
            if constexpr (VPT >= 16) {
#pragma unroll
              for (int hh = 0; hh < VPT / 16; ++hh)
                *reinterpret_cast<uint4*>(base_ptr + L.act + rowoff + ((((c >> 4) + hh) ^ (m & 7)) << 4)) =
                    make_uint4(cw[4 * hh], cw[4 * hh + 1], cw[4 * hh + 2], cw[4 * hh + 3]);
            } else if constexpr (VPT == 8) {
              *reinterpret_cast<uint2*>(base_ptr + L.act + rowoff + (((c >> 4) ^ (m & 7)) << 4) + (c & 15)) =
                  make_uint2(cw[0], cw[1]);
            } else {
              *reinterpret_cast<uint32_t*>(base_ptr + L.act + rowoff + (((c >> 4) ^ (m & 7)) << 4) + (c & 15)) =
                  cw[0];
            }
            if (sub == 0)
              base_ptr[L.sfb_off(m >> 7, ci) + (m & 31) * 16 + ((m & 127) >> 5) * 4 + (blk & 3)] =
                  static_cast<uint8_t>(sbyte);
            if (norm_out && p.norm.a_q != nullptr) {
              uint8_t* const dst = p.norm.a_q + static_cast<size_t>(m) * p.K + kg;
              if constexpr (VPT >= 16) {
#pragma unroll
                for (int hh = 0; hh < VPT / 16; ++hh)
                  reinterpret_cast<uint4*>(dst)[hh] =
                      make_uint4(cw[4 * hh], cw[4 * hh + 1], cw[4 * hh + 2], cw[4 * hh + 3]);
              } else if constexpr (VPT == 8) {
                *reinterpret_cast<uint2*>(dst) = make_uint2(cw[0], cw[1]);
              } else {
                *reinterpret_cast<uint32_t*>(dst) = cw[0];
              }
              if (sub == 0)
                p.norm.a_q_scales[swz_offset(m, (kg - sub * VPT) >> 5, p.K >> 5)] = static_cast<uint8_t>(sbyte);
            }
          }
          row += q_drow;
          blk += q_dblk;
          if (blk >= blocks_per_row) {
            blk -= blocks_per_row;
            ++row;
          }
        }
      };
      switch (q_tpb) {
        case 8: blocks(std::integral_constant<int, 8>{}); break;
        case 4: blocks(std::integral_constant<int, 4>{}); break;
        case 2: blocks(std::integral_constant<int, 2>{}); break;
        default: blocks(std::integral_constant<int, 1>{}); break;
      }
      __syncthreads();  // the next batch reuses the staging rows
    }
    fence_proxy_async_smem();  // written by the threads, read by the tensor cores
    __syncthreads();
    if (threadIdx.x == 0) MX_TL(12, globaltimer());
  }

  if (warp == 0 || warp == 3) {
    // ---------------- ring refills (warp-uniform): chunk i re-uses stage
    // i % stages once the MMAs of chunk i - stages have completed; the issuing
    // lane rotates, so consecutive copies come from different threads
    const bool weights = warp == 0;
    int s = 0, issuer = stages & 31;
    uint32_t ph = 0, empty_s = empty(0);
    for (int i = stages; i < (kFusedA && !weights ? 0 : n); ++i) {
      bool freed = mbar_try_wait(empty_s, ph);
      if (!__all_sync(0xFFFFFFFFu, freed)) freed = *abort_flag == 0 && mbar_wait(empty_s, ph);
      if (!__all_sync(0xFFFFFFFFu, freed)) {
        if (lane == 0) fail();
        break;
      }
      if (lane == issuer) {
        if (weights) issue_w(i, s);
        else issue_a(i, s);
      }
      issued_n = i + 1;
      __syncwarp();
      if (++issuer == 32) issuer = 0;
      if (++s == stages) {
        s = 0;
        ph ^= 1u;
        empty_s = empty(0);
      } else {
        empty_s += 8;
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA warp. The whole warp walks the ring (waits, counters,
    // descriptors: warp-uniform values) and one elected lane issues the tcgen05
    // ops. The issue latency of that one instruction stream bounds the loop, so
    // the smem descriptors advance by 32-bit adds on their low halves (address
    // field in 16-byte units) and stage, phase, barrier and TMEM addresses are
    // running values rather than divisions and products.
    const uint64_t wd = sdesc_k_sw128(base + L.w_off(0));
    const uint64_t ad = sdesc_k_sw128(base + (kFusedA ? L.act : L.a_off(0)));
    const uint64_t fd = sdesc_sf(base + L.sfa_off(0));
    const uint64_t gd = sdesc_sf(base + L.sfb_off(0, 0));
    const uint32_t op_hi = static_cast<uint32_t>(wd >> 32), sf_hi = static_cast<uint32_t>(fd >> 32);
    const uint32_t stage_units = L.stage_bytes >> 4;
    const uint32_t rt_units = (static_cast<uint32_t>(L.nmax) * kSfTileBytes) >> 4;
    const uint32_t id0 = idesc_mxf8(p.mtile, 0), id1 = idesc_mxf8(p.mtile, 1);
    const uint32_t id2 = idesc_mxf8(p.mtile, 2), id3 = idesc_mxf8(p.mtile, 3);
    // every wait below is taken by all lanes and decided by a warp vote, so the
    // warp stays converged for elect.sync and leaves the loop together
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(sfa_bar, 0) && (kFusedA || mbar_wait(sfb_bar, 0)))) {
      if (lane == 0) fail();
    } else {
      uint32_t w_lo = static_cast<uint32_t>(wd), a_lo = static_cast<uint32_t>(ad);
      uint32_t f_lo = static_cast<uint32_t>(fd), g_lo = static_cast<uint32_t>(gd);
      uint32_t ta = tmem + sfa_col, tb = tmem + sfb_col;
      uint32_t full_s = full(0), empty_s = empty(0);
      uint32_t ph = 0;
      int s = 0;
      for (int i = 0; i < n; ++i) {
        bool landed = mbar_try_wait(full_s, ph);
        if (!__all_sync(0xFFFFFFFFu, landed)) landed = *abort_flag == 0 && mbar_wait(full_s, ph);
        if (!__all_sync(0xFFFFFFFFu, landed)) {
          if (lane == 0) fail();
          break;
        }
        if (i == 0 && lane == 0) MX_TL(5, globaltimer());
        if (i == 1 && lane == 0) MX_TL(18, globaltimer());
        if (i == n - 1 && lane == 0) MX_TL(15, globaltimer());
        tc_fence_after();
        if (elect_one()) {
          tmem_cp_32x128b_x4_lh(ta, f_lo, sf_hi);
          tmem_cp_32x128b_x4_lh(tb, g_lo, sf_hi);
          if (nsfb > 1) tmem_cp_32x128b_x4_lh(tb + 4, g_lo + rt_units, sf_hi);
          mma_mxf8_lh(tmem, w_lo, op_hi, a_lo, op_hi, id0, ta, tb, i != 0);
          mma_mxf8_lh(tmem, w_lo + 2, op_hi, a_lo + 2, op_hi, id1, ta, tb, 1);
          mma_mxf8_lh(tmem, w_lo + 4, op_hi, a_lo + 4, op_hi, id2, ta, tb, 1);
          mma_mxf8_lh(tmem, w_lo + 6, op_hi, a_lo + 6, op_hi, id3, ta, tb, 1);
          if (i + stages < n) tc_commit(empty_s);  // only stages that will be refilled
        }
        __syncwarp();
        f_lo += kSfTileBytes >> 4;
        g_lo += kSfTileBytes >> 4;
        if (kFusedA) a_lo += L.a_bytes >> 4;  // resident tiles: one per chunk
        if (++s == stages) {
          s = 0;
          ph ^= 1u;
          w_lo = static_cast<uint32_t>(wd);
          if (!kFusedA) a_lo = static_cast<uint32_t>(ad);
          ta = tmem + sfa_col;
          tb = tmem + sfb_col;
          full_s = full(0);
          empty_s = empty(0);
        } else {
          w_lo += stage_units;
          if (!kFusedA) a_lo += stage_units;
          ta += 4;
          tb += 4 * nsfb;
          full_s += 8;
          empty_s += 8;
        }
      }
    }
    if (elect_one()) tc_commit(accum_bar);
    __syncwarp();
    if (lane == 0) MX_TL(16, globaltimer());
  }
  __syncwarp();

  // ---------------- epilogue: TMEM -> shared partials
  if (!mbar_wait(accum_bar, 0)) fail();
  if (threadIdx.x == 0) MX_TL(6, globaltimer());
  tc_fence_after();
  __syncwarp();
  float* const red = reinterpret_cast<float*>(base_ptr);
  // push: the slots of the ranks (of the peers when compact: ranks below this
  // one, then above it); this rank's own values
  float* const push = reinterpret_cast<float*>(base_ptr + L.red);
  float* const own = compact ? red : push + static_cast<uint32_t>(split) * (slot / 4);
  const bool ok = (*abort_flag == 0);
  if constexpr (kPush) {
    // warp q sends column block q of every row (push.cuh); this rank's own
    // units are stored locally (own slot, or over the ring when compact)
    cluster_wait_acquire();  // every peer's receive barrier is initialised and armed
    if (want_q(warp))
      push_send<compact>(pgeo, tmem + (static_cast<uint32_t>(warp * 32) << 16), warp, lane, base + L.red,
                         base + L.red_bar, own, ok);
    tc_fence_before();
    if (!mbar_wait(base + L.red_bar, 0)) fail();
    __syncthreads();  // this rank's own values, stored by every warp, are read by any warp
    if (threadIdx.x == 0) MX_TL(7, globaltimer());
    // every store into this CTA has landed: its part of the exit barrier (an
    // arrival waits for the thread's own stores to peers, by now delivered)
    cluster_arrive_relaxed();
  } else {
    if (ok) {
      for (int c0 = 0; c0 < p.mtile; c0 += 16) {
        float v[16];
        tmem_ld_32x32b_x16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) red[(c0 + j) * 128 + warp * 32 + lane] = v[j];
      }
    }
    tc_fence_before();
    cluster_sync();
    if (threadIdx.x == 0) MX_TL(7, globaltimer());
  }

  // ---------------- cluster reduction + bf16 (+ MXFP8) store
  if (ok) {
    const uint32_t red_addr = smem_u32(red);
    __nv_bfloat16* const out = static_cast<__nv_bfloat16*>(p.out);
    // Item = 32 columns of one row. An item nobody consumes is not reduced: a
    // peer's shared memory is read only for a value that is then used, so no
    // read is in flight when the peers exit.
    auto wanted = [&](int item) { return item < p.M * 4 && want_q(item & 3); };
    auto item_addr = [&](int item) {
      return red_addr + static_cast<uint32_t>((item >> 2) * 128 + (item & 3) * 32 + lane) * 4u;
    };
    // bf16 store and MX requantization of one reduced item (warp-uniform call)
    auto emit = [&](int item, float acc) {
      const int m = item >> 2;
      const int col = tile * 128 + (item & 3) * 32 + lane;
      const __nv_bfloat16 hb = __float2bfloat16_rn(acc);
      if (out != nullptr) out[static_cast<size_t>(m) * p.N + col] = hb;
      if (p.ssq_out != nullptr && tile * 128 + (item & 3) * 32 < p.ssq_cols) {
        // the block's sum of squares: the xor-shuffle tree over its 32 values
        const float v = __bfloat162float(hb);
        float sq = __fmul_rn(v, v);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq = __fadd_rn(sq, __shfl_xor_sync(0xFFFFFFFFu, sq, o));
        if (lane == 0) p.ssq_out[static_cast<size_t>(m) * (p.ssq_cols >> 5) + (col >> 5)] = sq;
      }
      if (kRequant && tile * 128 + (item & 3) * 32 < p.q_cols) {
        const float v = __bfloat162float(hb);
        // block amax in one reduction: non-negative floats order as their
        // bits, and an Inf or NaN puts the maximum at or above Inf's bits
        const uint32_t amax_bits = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(v)));
        uint32_t sbyte, code;
        if (amax_bits >= 0x7F800000u) {
          sbyte = 0xFFu;
          code = 0x7Fu;
        } else {
          sbyte = mx_scale_byte(__uint_as_float(amax_bits));
          code = cvt_e4m3x2(v * mx_inv_scale(sbyte), 0.f) & 0xFFu;
        }
        p.q[static_cast<size_t>(m) * p.q_cols + col] = static_cast<uint8_t>(code);
        if (lane == 0) p.q_scales[swz_offset(m, col >> 5, p.q_cols >> 5)] = static_cast<uint8_t>(sbyte);
      }
    };
    if constexpr (kPush) {
      push_sum<compact>(pgeo, warp, kThreads / 32, lane, push, own, want_q, emit);
    } else if (p.M <= S) {
      // at most one item per warp
      for (int item = split + S * warp; item < p.M * 4; item += 4 * S)
        if (wanted(item)) emit(item, cluster_sum(item_addr(item), S));
    } else if (kRed == kReduceItems) {
      // several items per warp: four items' peer loads in flight at once (the
      // warp is alone on its scheduler, so one item at a time would be
      // latency-bound), each still summed in rank order
      for (int i0 = split + S * warp; i0 < p.M * 4; i0 += 4 * S * kSumBatch) {
        uint32_t offs[kSumBatch];
        bool use[kSumBatch];
        float sums[kSumBatch];
#pragma unroll
        for (int b = 0; b < kSumBatch; ++b) {
          use[b] = wanted(i0 + b * 4 * S);
          offs[b] = item_addr(i0 + b * 4 * S);
        }
        cluster_sum_batch(offs, use, S, sums);
#pragma unroll
        for (int b = 0; b < kSumBatch; ++b)
          if (use[b]) emit(i0 + b * 4 * S, sums[b]);  // use[] is warp-uniform
      }
    } else {
      // Several rows per warp and at most four K-splits (row_reduction): a
      // warp reduces whole rows of the tile, lane l owning columns 4l .. 4l + 3,
      // with 16-byte peer loads; the loads of kRedRows rows x 4 ranks are in
      // flight at once, each column still summed in rank order. Row m goes to
      // CTA m % S, warp (m / S) % 4.
      const bool row_wanted = out != nullptr || (kRequant && tile * 128 < p.q_cols) ||
                              (p.ssq_out != nullptr && tile * 128 < p.ssq_cols);
      uint32_t rank_base[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) rank_base[r] = r < S ? map_shared_rank(red_addr, r) : 0u;
      const int col0 = tile * 128 + lane * 4;  // the lane's first output column
      for (int m0 = split + S * warp; row_wanted && m0 < p.M; m0 += 4 * S * kRedRows) {
        float4 acc[kRedRows];
#pragma unroll
        for (int b = 0; b < kRedRows; ++b) acc[b] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r0 = 0; r0 < 8; r0 += 4) {  // S <= 8: a cluster holds at most 8 CTAs
          if (r0 >= S) break;
          float4 v[kRedRows][4];
#pragma unroll
          for (int b = 0; b < kRedRows; ++b)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int m = m0 + b * 4 * S;
              v[b][r] = m < p.M && r0 + r < S
                            ? ld_shared_cluster_v4(rank_base[r0 + r] + static_cast<uint32_t>(m * 512 + lane * 16))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
          for (int b = 0; b < kRedRows; ++b)
#pragma unroll
            for (int r = 0; r < 4; ++r)
              if (r0 + r < S) {
                acc[b].x += v[b][r].x;
                acc[b].y += v[b][r].y;
                acc[b].z += v[b][r].z;
                acc[b].w += v[b][r].w;
              }
        }
#pragma unroll
        for (int b = 0; b < kRedRows; ++b) {
          const int m = m0 + b * 4 * S;
          if (m >= p.M) break;  // warp-uniform
          const float a4[4] = {acc[b].x, acc[b].y, acc[b].z, acc[b].w};
          uint32_t hb[4];
          float v4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            hb[e] = __bfloat16_as_ushort(__float2bfloat16_rn(a4[e]));
            v4[e] = __uint_as_float(hb[e] << 16);
          }
          if (out != nullptr)
            *reinterpret_cast<uint2*>(out + static_cast<size_t>(m) * p.N + col0) =
                make_uint2(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16));
          if (kRequant && tile * 128 < p.q_cols) {
            // 32-column block = 8 lanes: its amax over their 4 values each
            uint32_t amax_bits = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) amax_bits = max(amax_bits, __float_as_uint(v4[e]) & 0x7FFFFFFFu);
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) amax_bits = max(amax_bits, __shfl_xor_sync(0xFFFFFFFFu, amax_bits, o));
            uint32_t sbyte, codes;
            if (amax_bits >= 0x7F800000u) {
              sbyte = 0xFFu;
              codes = 0x7F7F7F7Fu;
            } else {
              sbyte = mx_scale_byte(__uint_as_float(amax_bits));
              const float f = mx_inv_scale(sbyte);
              codes = cvt_e4m3x2(v4[0] * f, v4[1] * f) | (cvt_e4m3x2(v4[2] * f, v4[3] * f) << 16);
            }
            *reinterpret_cast<uint32_t*>(p.q + static_cast<size_t>(m) * p.q_cols + col0) = codes;
            if ((lane & 7) == 0) p.q_scales[swz_offset(m, col0 >> 5, p.q_cols >> 5)] = static_cast<uint8_t>(sbyte);
          }
          if (p.ssq_out != nullptr && tile * 128 < p.ssq_cols) {
            // the block's sum of squares in the tree order of the one-item path:
            // element j = 4 (lane % 8) + e pairs with j ^ 16, j ^ 8, j ^ 4 (lanes
            // l ^ 4, l ^ 2, l ^ 1), then j ^ 2 and j ^ 1 (inside the lane)
            float s[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) s[e] = __fmul_rn(v4[e], v4[e]);
#pragma unroll
            for (int o = 4; o > 0; o >>= 1)
#pragma unroll
              for (int e = 0; e < 4; ++e) s[e] = __fadd_rn(s[e], __shfl_xor_sync(0xFFFFFFFFu, s[e], o));
            s[0] = __fadd_rn(s[0], s[2]);
            s[1] = __fadd_rn(s[1], s[3]);
            s[0] = __fadd_rn(s[0], s[1]);
            if ((lane & 7) == 0) p.ssq_out[static_cast<size_t>(m) * (p.ssq_cols >> 5) + (col0 >> 5)] = s[0];
          }
        }
      }
    }
    if (kRequant && split == 0 && tile * 128 < p.q_cols) {
      // padding rows of this tile's four scale columns
      const int mpad = (p.M + 127) & ~127;
      for (int idx = threadIdx.x; idx < (mpad - p.M) * 4; idx += kThreads) {
        const int m = p.M + (idx >> 2);
        p.q_scales[swz_offset(m, tile * 4 + (idx & 3), p.q_cols >> 5)] = 0;
      }
    }
  }
  if (threadIdx.x == 0) MX_TL(8, globaltimer());
  // the peers' reads of this CTA's partials have completed (their values were
  // consumed), so ordering the exits needs no memory release; with the push
  // reduction every CTA has arrived once all stores into it landed
  if constexpr (kPush)
    cluster_wait();
  else
    cluster_sync_relaxed();

  // ---------------- teardown
  if (*abort_flag != 0) {
    // wait (bounded) for the copies still in flight, so none lands after exit:
    // per stage, the last chunk loaded into it (an earlier one in the same stage
    // had landed before the stage was refilled)
    if (last >= 0 && last + stages >= issued_n) mbar_wait(full(last % stages), (last / stages) & 1);
    if (warp == 2 && lane == 0) mbar_wait(sfa_bar, 0);
    if (warp == 2 && lane == 1 && !kFusedA) mbar_wait(sfb_bar, 0);
    if (warp == 3 && lane == 0 && x_batches > 0) mbar_wait(x_bar, (x_batches - 1) & 1);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
  if (threadIdx.x == 0) MX_TL(9, globaltimer());
}

int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

}  // namespace

// K-splits (and, where it helps, the ring depth) of the decode step's projection
// shapes on a GB300 (152 SMs), chosen inside the graph-replayed chain of the
// three projections (bench.py --tune-chain: mx_gemm_chain, weights streamed from
// HBM), as the mxfp8 page picks its fixed tactics per row range in the chain
// rather than as isolated launches. Chain us, the table timed as back-to-back
// launches -> this one: 1 row 19.5 -> 18.5, 4 rows 20.3 -> 18.5, 16 rows
// 20.9 -> 20.6, 32 rows 23.9 -> 22.7, 64 rows 29.6 -> 26.8, 128 rows 50.8 ->
// 34.0, 192 rows 77.4 -> 42.6, 256 rows 55.5 -> 49.3 (from 32 rows four or
// fewer splits win once their partials are reduced as whole rows). G1's shape
// is also the stand-alone GEMM of the benchmark step: in the chain 4 splits with
// the whole K-range resident save 0.5 us at one to four rows but cost 0.3 us per
// stand-alone launch (4.58 -> 4.87 us at M = 1), and one table serves both, so
// that mx_gemm and the chain's G1 stay the same kernel (the chain equals the
// composition of its entry points bit for bit); G1 keeps 8 splits up to 16
// rows. Re-tuned with the push reduction (1 / 4 / 8 / 16 rows): only G2 at one
// or two rows moved, from 2 to 4 splits (chain at one row 17.6 -> 17.3 us); G1
// at 8 splits remains the fastest stand-alone (3.89 us at one row, against
// 4.23 with 6 and 4.51 with 5). G3 takes a ring of 4 stages from 5 to 12 rows:
// its CTAs then fit beside G2's with the push reduction's receive areas
// (chain at 8 rows 19.3 -> 18.4 us, at 12 rows 20.0 -> 19.5 us; at 1, 4 and 16
// rows 0.2-0.4 us slower, so there it keeps 5). After the fused-norm G2 the
// shallower ring is slower (chain-norm at 8 rows 20.9 -> 22.0 us): that chain
// asks for the planned depth. wo_b keeps the counts timed as back-to-back
// launches. stages = 0: the ring depth plan_gemm derives. Shapes not listed use
// the SM-count rule.
struct SplitEntry {
  int n, k, max_m, splits, stages;
};
constexpr SplitEntry kSplitTable[] = {
    {2048, 5120, 16, 8, 0},   {2048, 5120, 256, 4, 0},                            // G1
    {8192, 1536, 128, 4, 0},  {8192, 1536, 256, 2, 0},                            // G2
    {5120, 8192, 4, 6, 0},    {5120, 8192, 12, 6, 4},   {5120, 8192, 64, 6, 0},   // G3
    {5120, 8192, 256, 3, 0},
    {5120, 4096, 32, 8, 0},   {5120, 4096, 256, 6, 0},                            // wo_b
};

static const SplitEntry* table_entry(int M, int N, int K) {
  for (const SplitEntry& e : kSplitTable)
    if (e.n == N && e.k == K && M <= e.max_m) return &e;
  return nullptr;
}

// Tuning override for one weight shape, from MX_PLAN_AT ("NxK:splits[:stages],...",
// e.g. "8192x1536:4:3"; splits 1..8, stages 1..12); 0 where the shape is not listed.
static void plan_override(const char* e, int N, int K, int* splits, int* stages) {
  *splits = *stages = 0;
  while (*e != '\0') {
    int n = 0, k = 0, s = 0, st = 0, used = 0;
    const int got = sscanf(e, "%dx%d:%d%n:%d%n", &n, &k, &s, &used, &st, &used);
    if (got < 3) return;
    if (n == N && k == K) {
      if (s >= 1 && s <= 8) *splits = s;
      if (got >= 4 && st >= 1 && st <= 12) *stages = st;
      return;
    }
    e += used;
    if (*e == ',') ++e;
  }
}

PlanEnv read_plan_env() {
  PlanEnv env{};
  auto num = [](const char* name, int lo, int hi) {
    const char* e = getenv(name);
    const int v = e != nullptr ? atoi(e) : 0;
    return v >= lo && v <= hi ? v : 0;
  };
  env.splits = num("MX_SPLITS", 1, 8);  // a K-split cluster holds at most 8 CTAs
  env.stages = num("MX_STAGES", 1, 12);
  env.woa_splits = num("MX_WOA_SPLITS", 1, 8);
  // MX_PUSH_ROWS: the push reduction up to this many rows (0: never)
  const char* pr = getenv("MX_PUSH_ROWS");
  env.push_rows = pr != nullptr ? std::max(0, std::min(atoi(pr), 256)) : -1;
  if (const char* e = getenv("MX_PLAN_AT")) snprintf(env.plan_at, sizeof(env.plan_at), "%s", e);
  return env;
}

GemmPlan plan_gemm(int M, int N, int K, int sm_count, const PlanEnv& env, bool fused_a, bool norm,
                   int push_mode, bool table_depth) {
  int force_splits, force_stages;
  plan_override(env.plan_at, N, K, &force_splits, &force_stages);
  const int mtile = (M + 15) & ~15;
  const int tiles = N / 128;
  const int nchunks = K / 128;
  const int nsfb = (mtile + 127) / 128;
  const int xrows = std::min(M, kRowBatch);
  const int push_rows = env.push_rows >= 0 ? env.push_rows : kPushMaxRows;
  // the scale tiles of a CTA's K-range stay resident: at most 48 KB of them
  auto scale_bytes = [&](int sp) {
    return static_cast<size_t>((nchunks + sp - 1) / sp) * kSfTileBytes * (1 + nsfb);
  };
  // the plan for a given number of K splits
  auto plan_for = [&](int splits) {
    GemmPlan pl{};
    pl.mtile = mtile;
    while (splits < std::min(8, nchunks) && scale_bytes(splits) > 48 * 1024) ++splits;
    pl.splits = splits;
    const int per_cta = (nchunks + splits - 1) / splits;
    const Layout L1(mtile, 1, per_cta, fused_a, xrows, norm ? K / 32 : 0);
    // resident per CTA besides the ring: scale tiles (and, fused, the activation
    // tiles and the bf16 staging rows)
    const size_t scales = L1.bars - L1.ring_bytes;
    // Short K-ranges (all chunks in flight at once): about 100 KB per CTA, so
    // the next kernel's CTAs fit beside this one. Long ones: as deep a ring as
    // lets the whole grid be resident in one wave (CTAs per SM x shared memory).
    const int per_sm = (tiles * splits + sm_count - 1) / std::max(sm_count, 1);
    const size_t wave = per_sm <= 1 ? 180 * 1024 : 227 * 1024 / static_cast<size_t>(per_sm) - 4 * 1024;
    const size_t budget = per_cta <= 8 ? std::min<size_t>(100 * 1024, wave) : wave;
    int stages = budget > scales ? static_cast<int>((budget - scales) / L1.stage_bytes) : 0;
    stages = std::max(2, std::min(stages, 10));
    if (env.stages > 0) stages = env.stages;
    if (force_stages > 0) stages = force_stages;
    stages = std::min(stages, per_cta);
    // the epilogue stages the fp32 partials [mtile][128] over the ring and what follows it
    while (static_cast<size_t>(stages) * L1.stage_bytes + scales < static_cast<size_t>(mtile) * 512)
      ++stages;
    pl.stages = stages;
    pl.tmem_cols = pow2_at_least(tmem_sfa_col(mtile) + 4 * stages * (1 + nsfb));
    // the push reduction (where asked for and its receive area fits)
    const uint32_t area = push_area_bytes(M, splits, push_mode == kPushCompact);
    const bool push = push_mode != kPushNone && M <= push_rows &&
                      Layout(mtile, stages, per_cta, fused_a, xrows, norm ? K / 32 : 0, area).total() <=
                          kMaxDynamicSmem;
    pl.reduction = !push                         ? (row_reduction(M, splits) ? kReduceRows : kReduceItems)
                   : push_mode == kPushCompact ? kReducePushCompact
                                               : kReducePush;
    const Layout L(mtile, stages, per_cta, fused_a, xrows, norm ? K / 32 : 0, push ? area : 0u);
    // CTAs that can share an SM must fit their TMEM together: ask for enough
    // shared memory that at most 512 / tmem_cols of them are resident.
    const int max_res = 512 / pl.tmem_cols;
    const size_t min_smem = 233472 / static_cast<size_t>(max_res + 1) + 1;
    pl.smem = std::max(L.total(), min_smem);
    return pl;
  };
  int splits = std::max(1, sm_count / std::max(tiles, 1));
  // the table was measured with 152 SMs; other parts keep the SM-count rule
  const SplitEntry* te = sm_count == 152 ? table_entry(M, N, K) : nullptr;
  if (te != nullptr) splits = te->splits;
  if (te != nullptr && force_stages == 0 && table_depth) force_stages = te->stages;
  splits = std::min(splits, std::min(8, nchunks));
  bool forced = false;
  if (env.splits > 0) {
    splits = std::min(env.splits, nchunks);
    forced = true;
  }
  if (force_splits > 0) {
    splits = std::min(force_splits, nchunks);
    forced = true;
  }
  GemmPlan pl = plan_for(splits);
  // An accumulator of more than half the TMEM (mtile above ~230 rows) leaves
  // room for one CTA per SM: a grid beyond one CTA per SM would run in two
  // waves (M = 256, N = 5120, K = 8192: 240 CTAs, 36 us against 19 us at 192
  // rows), so such plans take at most one CTA per SM.
  if (!forced && pl.tmem_cols > 256 && tiles * pl.splits > sm_count)
    pl = plan_for(std::max(1, std::min(pl.splits, sm_count / std::max(tiles, 1))));
  return pl;
}

cudaError_t set_gemm_attributes() {
  const void* ks[16] = {
      reinterpret_cast<const void*>(&gemm_kernel<false, false, kReduceItems>),
      reinterpret_cast<const void*>(&gemm_kernel<true, false, kReduceItems>),
      reinterpret_cast<const void*>(&gemm_kernel<false, true, kReduceItems>),
      reinterpret_cast<const void*>(&gemm_kernel<true, true, kReduceItems>),
      reinterpret_cast<const void*>(&gemm_kernel<false, false, kReduceRows>),
      reinterpret_cast<const void*>(&gemm_kernel<true, false, kReduceRows>),
      reinterpret_cast<const void*>(&gemm_kernel<false, true, kReduceRows>),
      reinterpret_cast<const void*>(&gemm_kernel<true, true, kReduceRows>),
      reinterpret_cast<const void*>(&gemm_kernel<false, false, kReducePush>),
      reinterpret_cast<const void*>(&gemm_kernel<true, false, kReducePush>),
      reinterpret_cast<const void*>(&gemm_kernel<false, true, kReducePush>),
      reinterpret_cast<const void*>(&gemm_kernel<true, true, kReducePush>),
      reinterpret_cast<const void*>(&gemm_kernel<false, false, kReducePushCompact>),
      reinterpret_cast<const void*>(&gemm_kernel<true, false, kReducePushCompact>),
      reinterpret_cast<const void*>(&gemm_kernel<false, true, kReducePushCompact>),
      reinterpret_cast<const void*>(&gemm_kernel<true, true, kReducePushCompact>)};
  for (const void* k : ks) {
    // clusters of up to 16 K-splits (beyond the portable 8)
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    // the whole unified L1/shared array as shared memory, so that every plan's
    // CTAs-per-SM fit from the first launch on
    e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kMaxDynamicSmem));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_gemm(const CUtensorMap& tm_w, const CUtensorMap& tm_a, const GemmArgs& args,
                        const GemmPlan& plan, bool pdl, cudaStream_t stream) {
  if (plan.smem > kMaxDynamicSmem) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(args.N / 128, plan.splits, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  attrs[na].id = cudaLaunchAttributeClusterDimension;
  attrs[na].val.clusterDim.x = 1;
  attrs[na].val.clusterDim.y = plan.splits;
  attrs[na].val.clusterDim.z = 1;
  ++na;
  if (pdl) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  const bool rq = args.q != nullptr, fx = args.x != nullptr;
  auto go = [&](auto kernel) { return cudaLaunchKernelEx(&cfg, kernel, tm_w, tm_a, args); };
  auto pick = [&](auto red) {
    constexpr int R = decltype(red)::value;
    if (fx) return rq ? go(gemm_kernel<true, true, R>) : go(gemm_kernel<false, true, R>);
    return rq ? go(gemm_kernel<true, false, R>) : go(gemm_kernel<false, false, R>);
  };
  if (plan.reduction == kReducePush) return pick(std::integral_constant<int, kReducePush>{});
  if (plan.reduction == kReducePushCompact) return pick(std::integral_constant<int, kReducePushCompact>{});
  if (plan.reduction == kReduceRows) return pick(std::integral_constant<int, kReduceRows>{});
  return pick(std::integral_constant<int, kReduceItems>{});
}

}  // namespace mx
