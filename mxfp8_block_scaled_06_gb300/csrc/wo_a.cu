// wo_a.cu - grouped WO-A output projection with inverse RoPE, writing MXFP8.
//
// z[t, g R + r] = sum_k dX_g[t, k] dW_g[r, k],  X_g = the H heads of group g,
// each head = 448 "nope" dims followed by 64 "rope" dims rotated by -pos f_i;
// q, q_scales = MXFP8(bf16(z)) for the following wo_b GEMM.
//
// Grid = (G * R/128 weight tiles) x (K splits); the splits of a tile form a
// thread-block cluster. Per CTA:
//  1. weight boxes (TMA, 128 rows x 128 K-bytes, SWIZZLE_128B) are issued for
//     the whole ring, one lane per box, and the scale tiles of the CTA's K-range
//     with one bulk copy, before the programmatic grid-dependency wait (with
//     early_trigger, dependents may launch right after the TMEM allocation);
//  2. after the wait, one lane per token bulk-copies the token's contiguous
//     K-slice of x (bf16) into shared memory while the others stage the tokens'
//     cos/sin rows; the 8 warps then rotate the rope pairs in float32 (no
//     FMA), take each 32-block's amax with two xor-shuffles over the 4 lanes
//     holding it, and write E4M3 codes straight into the 128-byte-swizzled
//     K-major operand layout plus 128x4 scale tiles - the activation never
//     goes to global memory (unless the debug outputs are requested);
//  3. the MMA warp walks the chunks warp-uniformly and an elected lane issues
//     tcgen05.cp + tcgen05.mma.kind::mxf8f6f4.block_scale; weight refills come
//     from a warp-uniform loop whose issuing lane rotates (copies issued by one
//     thread are serviced one after another); 4. the cluster reduces the fp32
//     partials over distributed shared memory (up to 16 tokens by the push
//     exchange of push.cuh, above by peer loads after a cluster barrier),
//     rounds to bf16 and requantizes each 32-column block.
#include <cuda_bf16.h>

#include <algorithm>

#include "kernels.h"
#include "ptx.cuh"
#include "push.cuh"

namespace mx {
namespace {

constexpr int kThreads = 256;
constexpr uint32_t kWTileBytes = 128 * 128;
constexpr uint32_t kSfTileBytes = 512;
constexpr uint32_t kStageBytes = 16384;  // one weight box
constexpr int kTokenBatch = 32;          // tokens whose raw x slices are staged at once

// Timeline build (-DMX_TIMELINE): %globaltimer stamps of one CTA's phases in
// p.tl, in the GEMM's slot numbering: 0 entry, 4 grid-dependency wait returned,
// 5 first chunk landed, 6 accumulator complete, 7 partials exchanged (push:
// received; else the cluster barrier), 8 reduction done, 9 exit, 10 SM id,
// 12 activation quantized, 13 the first batch's barrier passed, 14 first token
// batch of x landed, 15 last chunk landed, 16 every MMA issued, 17 thread 0's
// units of the first batch quantized.
#ifdef MX_TIMELINE
#define MX_TL(slot, v)                                                             \
  do {                                                                             \
    if (p.tl != nullptr)                                                           \
      p.tl[(blockIdx.y * gridDim.x + blockIdx.x) * kTimelineSlots + (slot)] = (v); \
  } while (0)
#else
#define MX_TL(slot, v) \
  do {                 \
  } while (0)
#endif

struct WoaLayout {
  uint32_t ring, act, sfb, sfa, xraw, cs, misc, red_bar, red, total;
  // tbmax = tokens staged per batch (min(T, kTokenBatch)), nmax = chunks per CTA,
  // red_bytes = the push exchange's receive area (0: none)
  __host__ __device__ WoaLayout(int mtile, int stages, int nmax, int tbmax, uint32_t red_bytes = 0) {
    ring = 0;
    act = ring + stages * kStageBytes;                              // nmax x [mtile x 128] swizzled
    sfb = act + static_cast<uint32_t>(nmax) * mtile * 128;          // nmax x 512
    sfa = sfb + static_cast<uint32_t>(nmax) * kSfTileBytes;         // nmax x 512 (weight scales)
    xraw = sfa + static_cast<uint32_t>(nmax) * kSfTileBytes;        // tbmax x nmax x 256
    cs = xraw + static_cast<uint32_t>(tbmax) * nmax * 256;          // tbmax x 64 floats
    misc = cs + static_cast<uint32_t>(tbmax) * 64 * 4;
    // barriers: wfull[stages], empty[stages], accum, x, sfa; TMEM slot, abort
    // flag; the receive barrier
    red_bar = misc + 8 * (2 * stages + 3) + 8;
    total = misc + 8 * (2 * stages + 3) + 16;
    red = (total + 127u) & ~127u;
    if (red_bytes != 0) total = red + red_bytes;
  }
};

// kPush: the push split-K exchange (up to 16 tokens) instead of peer loads.
template <bool kPush>
__global__ void __launch_bounds__(kThreads, 1)
    wo_a_kernel(const __grid_constant__ CUtensorMap tm_w, const WoaArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* const bp = smem_raw + (base - raw_addr);
  if (threadIdx.x == 0) MX_TL(0, globaltimer());

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_per_group = p.R / 128;
  const int tile = blockIdx.x;
  const int g = tile / tiles_per_group;
  const int rt = tile % tiles_per_group;
  const int S = gridDim.y;
  const int split = blockIdx.y;
  const int kg = p.H * p.D;      // K of one group
  const int nchunks = kg / 128;
  const int c_begin = split * nchunks / S;
  const int n = (split + 1) * nchunks / S - c_begin;
  const int nmax = (nchunks + S - 1) / S;
  const int stages = p.stages;
  const PushGeometry pgeo(p.T, kPush ? S : 1, kPush ? split : 0);
  const uint32_t slot = pgeo.slot;
  const WoaLayout L(p.mtile, stages, nmax, min(p.T, kTokenBatch), kPush ? push_area_bytes(p.T, S, false) : 0u);
  auto want_all = [](int) { return true; };  // every column is requantized

  const uint32_t bars = base + L.misc;
  auto wfull = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (stages + s); };
  const uint32_t accum_bar = bars + 16u * stages;
  const uint32_t x_bar = accum_bar + 8u;
  const uint32_t sfa_bar = accum_bar + 16u;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(bp + L.misc + 8 * (2 * stages + 3));
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(wfull(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(accum_bar, 1);
    mbar_init(x_bar, 1);
    mbar_init(sfa_bar, 1);
    mbar_init(base + L.red_bar, 1);
    // armed now with the bytes the peers will store (after the cluster barrier below)
    if constexpr (kPush) mbar_expect_tx(base + L.red_bar, push_expect_bytes(pgeo, want_all));
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_w);
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // push: the receive barriers of the whole cluster are initialised and armed
  // before any peer stores to them (the wait is in the epilogue)
  if constexpr (kPush) cluster_arrive_release();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sfa_col = (p.mtile + 15) & ~15;
  const uint32_t sfb_col = sfa_col + 4 * stages;
  if (p.early_trigger) pdl_launch_dependents();

  auto fail = [&]() {
    atomicOr(p.status, kStatusTimeout);
    *abort_flag = 1;
  };

  const uint64_t pol_w = policy_evict_first();
  int last = -1;      // last chunk whose weight box this lane loaded (warp 0)
  int issued_n = 0;   // weight boxes warp 0 has loaded so far (warp-uniform)
  auto issue_w = [&](int i, int s) {
    mbar_expect_tx(wfull(s), kWTileBytes);
    tma_load_2d(base + L.ring + s * kStageBytes, &tm_w, wfull(s), (c_begin + i) * 128, tile * 128,
                pol_w);
    last = i;
  };
  if (warp == 0) {
    if (lane < min(n, stages)) issue_w(lane, lane);
    issued_n = min(n, stages);
  }
  if (warp == 2 && lane == 0) {
    mbar_expect_tx(sfa_bar, static_cast<uint32_t>(n) * kSfTileBytes);
    bulk_load(base + L.sfa, p.w_scales + (static_cast<size_t>(tile) * nchunks + c_begin) * kSfTileBytes,
              static_cast<uint32_t>(n) * kSfTileBytes, sfa_bar, pol_w);
  }
  int x_batches = 0;
  // shared memory only, so before the wait: zero the padding rows [T, mtile) of
  // every chunk tile and all scale tiles (the quantized rows are written over
  // them after the first batch's barrier below)
  const uint32_t act_tile_bytes = static_cast<uint32_t>(p.mtile) * 128u;
  {
    const int pad_rows = p.mtile - p.T;
    for (int idx = threadIdx.x; idx < n * pad_rows * 8; idx += kThreads) {
      const int i = idx / (pad_rows * 8);
      const int rem = idx % (pad_rows * 8);
      const int m = p.T + rem / 8;
      *reinterpret_cast<uint4*>(bp + L.act + i * act_tile_bytes + m * 128 + (rem % 8) * 16) =
          make_uint4(0, 0, 0, 0);
    }
    for (int idx = threadIdx.x; idx < n * 32; idx += kThreads)
      *reinterpret_cast<uint4*>(bp + L.sfb + idx * 16) = make_uint4(0, 0, 0, 0);
  }
  if (!p.early_trigger) pdl_launch_dependents();
  pdl_wait();
  if (threadIdx.x == 0) MX_TL(4, globaltimer());
#ifdef MX_TIMELINE
  if (threadIdx.x == 0) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    MX_TL(10, static_cast<unsigned long long>(smid));
  }
#endif

  // ---------------- prologue: RoPE + MX quantize into the swizzled operand
  const size_t xq_stride = static_cast<size_t>(p.G) * kg;
  const int units_per_token = n * 16;  // 8-element units in the CTA's K-slice
  const float inv_units = 1.f / static_cast<float>(units_per_token);
  for (int t0 = 0, batch = 0; t0 < p.T; t0 += kTokenBatch, ++batch) {
    const int tb = min(kTokenBatch, p.T - t0);
    if (warp == 0) {
      // one lane per token (tb <= 32)
      if (lane == 0) mbar_expect_tx(x_bar, static_cast<uint32_t>(tb) * n * 256u);
      __syncwarp();
      if (lane < tb) {
        const uint16_t* src = p.x + static_cast<size_t>(t0 + lane) * p.ldx +
                              static_cast<size_t>(g) * kg + static_cast<size_t>(c_begin) * 128;
        bulk_load(base + L.xraw + lane * nmax * 256, src, n * 256u, x_bar, pol_w);
      }
      x_batches = batch + 1;
    }
    // cos/sin rows of the batch's tokens
    float* const cs = reinterpret_cast<float*>(bp + L.cs);
    for (int idx = threadIdx.x; idx < tb * 64; idx += kThreads) {
      const int m = idx >> 6;
      long long pos = p.positions[t0 + m];
      if (pos < 0 || pos >= p.max_pos) {
        atomicOr(p.status, kStatusBadInput);  // position outside the cache: read row 0
        pos = 0;
      }
      cs[idx] = p.cos_sin[static_cast<size_t>(pos) * 64 + (idx & 63)];
    }
    if (!mbar_wait(x_bar, batch & 1)) fail();
    if (batch == 0 && threadIdx.x == 0) MX_TL(14, globaltimer());
    __syncthreads();
    if (batch == 0 && threadIdx.x == 0) MX_TL(13, globaltimer());
    const int total = tb * units_per_token;
    for (int b0 = 0; b0 < total; b0 += kThreads) {
      const int u = b0 + threadIdx.x;
      const bool valid = u < total && *abort_flag == 0;
      // token within the batch and 8-element unit within the slice: u split by
      // units_per_token through a float reciprocal, corrected to the exact
      // integer quotient (u < 32 tokens x 512 units: the estimate is off by at
      // most one)
      int ml = __float2int_rz(__int2float_rn(u) * inv_units);
      if ((ml + 1) * units_per_token <= u) ++ml;
      if (ml * units_per_token > u) --ml;
      const int ul = u - ml * units_per_token;
      const int blk = ul >> 2;                  // 32-block within the slice
      const int sub = ul & 3;
      const int kin = c_begin * 128 + ul * 8;   // K index within the group
      const int d = kin & (p.D - 1);            // D = 512 (448 + 64), a power of two
      float v[8];
      float amax = 0.f;
      uint32_t nonfinite = 0;
      if (valid) {
        const uint4 raw = *reinterpret_cast<const uint4*>(bp + L.xraw + ml * nmax * 256 + ul * 16);
        const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[2 * i] = __uint_as_float(w4[i] << 16);
          v[2 * i + 1] = __uint_as_float(w4[i] & 0xFFFF0000u);
        }
        if (d >= 448) {
          const float* row = cs + ml * 64;
          const int p0 = (d - 448) >> 1;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float c = row[p0 + i], s = row[32 + p0 + i];
            const float a = v[2 * i], b = v[2 * i + 1];
            v[2 * i] = __fadd_rn(__fmul_rn(a, c), __fmul_rn(b, s));
            v[2 * i + 1] = __fsub_rn(__fmul_rn(b, c), __fmul_rn(a, s));
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          amax = fmaxf(amax, fabsf(v[i]));
          nonfinite |= !isfinite(v[i]);
        }
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
      nonfinite |= __shfl_xor_sync(0xFFFFFFFFu, nonfinite, 1);
      nonfinite |= __shfl_xor_sync(0xFFFFFFFFu, nonfinite, 2);
      if (valid) {
        uint32_t sbyte, lo, hi;
        if (nonfinite) {
          sbyte = 0xFFu;
          lo = hi = 0x7F7F7F7Fu;
        } else {
          sbyte = mx_scale_byte(amax);
          const float f = mx_inv_scale(sbyte);
          lo = cvt_e4m3x2(v[0] * f, v[1] * f) | (cvt_e4m3x2(v[2] * f, v[3] * f) << 16);
          hi = cvt_e4m3x2(v[4] * f, v[5] * f) | (cvt_e4m3x2(v[6] * f, v[7] * f) << 16);
        }
        const int m = t0 + ml;
        const int ci = blk >> 2;                 // chunk within the slice
        const int kb = (blk & 3) * 32 + sub * 8;  // byte within the 128-byte row
        const uint32_t off = ci * act_tile_bytes + (m >> 3) * 1024 + (m & 7) * 128 +
                             (((kb >> 4) ^ (m & 7)) << 4) + (kb & 15);
        *reinterpret_cast<uint2*>(bp + L.act + off) = make_uint2(lo, hi);
        if (sub == 0)
          bp[L.sfb + ci * kSfTileBytes + (m & 31) * 16 + (m >> 5) * 4 + (blk & 3)] =
              static_cast<uint8_t>(sbyte);
        if (rt == 0) {
          const size_t kglob = static_cast<size_t>(g) * kg + kin;
          if (p.debug_xq)
            *reinterpret_cast<uint2*>(p.debug_xq + m * xq_stride + kglob) = make_uint2(lo, hi);
          if (p.debug_xs && sub == 0)
            p.debug_xs[m * (xq_stride / 32) + kglob / 32] = static_cast<uint8_t>(sbyte);
        }
      }
    }
    if (batch == 0 && threadIdx.x == 0) MX_TL(17, globaltimer());
    fence_proxy_async_smem();
    __syncthreads();  // the next batch reuses the raw slices
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (threadIdx.x == 0) MX_TL(12, globaltimer());

  if (warp == 0) {
    // ---------------- weight ring refills (warp-uniform, rotating issuing lane):
    // chunk i re-uses stage i % stages once the MMAs of chunk i - stages completed
    int s = 0, issuer = stages & 31;
    uint32_t ph = 0, empty_s = empty(0);
    for (int i = stages; i < n; ++i) {
      bool freed = mbar_try_wait(empty_s, ph);
      if (!__all_sync(0xFFFFFFFFu, freed)) freed = *abort_flag == 0 && mbar_wait(empty_s, ph);
      if (!__all_sync(0xFFFFFFFFu, freed)) {
        if (lane == 0) fail();
        break;
      }
      if (lane == issuer) issue_w(i, s);
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
    // ---------------- MMA warp: warp-uniform walk, one elected lane issues; the
    // smem descriptors advance by 32-bit adds on their low halves
    const uint64_t wd = sdesc_k_sw128(base + L.ring);
    const uint64_t ad = sdesc_k_sw128(base + L.act);
    const uint64_t fd = sdesc_sf(base + L.sfa);
    const uint64_t gd = sdesc_sf(base + L.sfb);
    const uint32_t op_hi = static_cast<uint32_t>(wd >> 32), sf_hi = static_cast<uint32_t>(fd >> 32);
    const uint32_t id0 = idesc_mxf8(p.mtile, 0), id1 = idesc_mxf8(p.mtile, 1);
    const uint32_t id2 = idesc_mxf8(p.mtile, 2), id3 = idesc_mxf8(p.mtile, 3);
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(sfa_bar, 0))) {
      if (lane == 0) fail();
    } else {
      uint32_t w_lo = static_cast<uint32_t>(wd), a_lo = static_cast<uint32_t>(ad);
      uint32_t f_lo = static_cast<uint32_t>(fd), g_lo = static_cast<uint32_t>(gd);
      uint32_t ta = tmem + sfa_col, tb = tmem + sfb_col;
      uint32_t full_s = wfull(0), empty_s = empty(0);
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
        if (i == n - 1 && lane == 0) MX_TL(15, globaltimer());
        tc_fence_after();
        if (elect_one()) {
          tmem_cp_32x128b_x4_lh(ta, f_lo, sf_hi);
          tmem_cp_32x128b_x4_lh(tb, g_lo, sf_hi);
          mma_mxf8_lh(tmem, w_lo, op_hi, a_lo, op_hi, id0, ta, tb, i != 0);
          mma_mxf8_lh(tmem, w_lo + 2, op_hi, a_lo + 2, op_hi, id1, ta, tb, 1);
          mma_mxf8_lh(tmem, w_lo + 4, op_hi, a_lo + 4, op_hi, id2, ta, tb, 1);
          mma_mxf8_lh(tmem, w_lo + 6, op_hi, a_lo + 6, op_hi, id3, ta, tb, 1);
          if (i + stages < n) tc_commit(empty_s);  // only stages that will be refilled
        }
        __syncwarp();
        f_lo += kSfTileBytes >> 4;
        g_lo += kSfTileBytes >> 4;
        a_lo += act_tile_bytes >> 4;
        if (++s == stages) {
          s = 0;
          ph ^= 1u;
          w_lo = static_cast<uint32_t>(wd);
          ta = tmem + sfa_col;
          tb = tmem + sfb_col;
          full_s = wfull(0);
          empty_s = empty(0);
        } else {
          w_lo += kStageBytes >> 4;
          ta += 4;
          tb += 4;
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

  // ---------------- epilogue
  if (!mbar_wait(accum_bar, 0)) fail();
  if (threadIdx.x == 0) MX_TL(6, globaltimer());
  tc_fence_after();
  __syncwarp();
  float* const red = reinterpret_cast<float*>(bp + L.ring);
  float* const push = reinterpret_cast<float*>(bp + L.red);
  const bool ok = (*abort_flag == 0);
  if constexpr (kPush) {
    // warps 0-3 (the accumulator's TMEM lanes) send their column blocks
    cluster_wait_acquire();  // every peer's receive barrier is initialised and armed
    if (warp < 4)
      push_send<false>(pgeo, tmem + (static_cast<uint32_t>(warp * 32) << 16), warp, lane, base + L.red,
                       base + L.red_bar, push + static_cast<uint32_t>(split) * (slot / 4), ok);
    tc_fence_before();
    if (!mbar_wait(base + L.red_bar, 0)) fail();
    __syncthreads();  // this rank's own values, stored by warps 0-3, are read by any warp
    if (threadIdx.x == 0) MX_TL(7, globaltimer());
    // every store into this CTA has landed: its part of the exit barrier
    cluster_arrive_relaxed();
  } else {
    if (ok && warp < 4) {
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
  if (ok) {
    const uint32_t red_addr = smem_u32(red);
    const int qcols = p.G * p.R;
    const int nwarps = kThreads / 32;
    // bf16 and MXFP8 of one reduced item (32 columns of token m; warp-uniform call)
    auto emit = [&](int item, float acc) {
      const int m = item >> 2;
      const int col = g * p.R + rt * 128 + (item & 3) * 32 + lane;
      const __nv_bfloat16 hb = __float2bfloat16_rn(acc);
      if (p.debug_z) p.debug_z[static_cast<size_t>(m) * qcols + col] = __bfloat16_as_ushort(hb);
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
      p.q[static_cast<size_t>(m) * qcols + col] = static_cast<uint8_t>(code);
      if (lane == 0) p.q_scales[swz_offset(m, col >> 5, qcols >> 5)] = static_cast<uint8_t>(sbyte);
    };
    if constexpr (kPush) {
      push_sum<false>(pgeo, warp, nwarps, lane, push, push + static_cast<uint32_t>(split) * (slot / 4), want_all,
                      emit);
    } else {
      // four items' peer loads in flight at once, each summed in rank order
      for (int i0 = split + S * warp; i0 < p.T * 4; i0 += nwarps * S * kSumBatch) {
        uint32_t offs[kSumBatch];
        bool use[kSumBatch];
        float sums[kSumBatch];
#pragma unroll
        for (int b = 0; b < kSumBatch; ++b) {
          const int item = i0 + b * nwarps * S;
          use[b] = item < p.T * 4;
          offs[b] = red_addr + static_cast<uint32_t>((item >> 2) * 128 + (item & 3) * 32 + lane) * 4u;
        }
        cluster_sum_batch(offs, use, S, sums);
#pragma unroll
        for (int b = 0; b < kSumBatch; ++b)
          if (use[b]) emit(i0 + b * nwarps * S, sums[b]);  // use[] is warp-uniform
      }
    }
    if (split == 0) {
      const int mpad = (p.T + 127) & ~127;
      for (int idx = threadIdx.x; idx < (mpad - p.T) * 4; idx += kThreads) {
        const int m = p.T + (idx >> 2);
        p.q_scales[swz_offset(m, (g * p.R + rt * 128) / 32 + (idx & 3), qcols >> 5)] = 0;
      }
    }
  }
  if (threadIdx.x == 0) MX_TL(8, globaltimer());
  // the peers' reads of this CTA's partials have completed (their values were
  // consumed), so ordering the exits needs no memory release; with the push
  // exchange every CTA has arrived once all stores into it landed
  if constexpr (kPush)
    cluster_wait();
  else
    cluster_sync_relaxed();

  if (*abort_flag != 0) {
    // wait (bounded) for the copies still in flight, so none lands after exit
    if (last >= 0 && last + stages >= issued_n) mbar_wait(wfull(last % stages), (last / stages) & 1);
    if (warp == 0 && lane == 0 && x_batches > 0) mbar_wait(x_bar, (x_batches - 1) & 1);
    if (warp == 2 && lane == 0) mbar_wait(sfa_bar, 0);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
  if (threadIdx.x == 0) MX_TL(9, globaltimer());
}

int pow2_at_least(int v) {
  int r = 32;
  while (r < v) r <<= 1;
  return r;
}

}  // namespace

WoaPlan plan_wo_a(int T, int G, int H, int R, int sm_count, const PlanEnv& env) {
  WoaPlan pl{};
  pl.mtile = (T + 15) & ~15;
  const int tiles = G * (R / 128);
  const int nchunks = H * 512 / 128;
  // Measured on a GB300 (4 groups x 1024 rows, 8 heads): up to 16 tokens the
  // fastest plan fills two co-resident CTAs per SM (T = 1: 6.5 us with 8 splits
  // vs 7.1 with 4); at 32 tokens the larger activation tiles favour one per SM.
  const int per_sm = T <= 16 ? 2 : 1;
  int splits = std::max(1, per_sm * sm_count / std::max(tiles, 1));
  splits = std::min(splits, std::min(8, nchunks));
  if (env.woa_splits > 0) splits = std::min(env.woa_splits, nchunks);
  const int tbmax = std::min(T, kTokenBatch);
  // more K-splits (fewer resident activation chunks) and a shallower weight
  // ring until the CTA fits in shared memory
  for (; splits <= std::min(8, nchunks); ++splits) {
    const int nmax = (nchunks + splits - 1) / splits;
    for (int stages = std::min(nmax, 4); stages >= 1; --stages) {
      // the fp32 partials [mtile][128] are staged in the weight ring
      if (static_cast<size_t>(stages) * kStageBytes < static_cast<size_t>(pl.mtile) * 512) break;
      pl.push = T <= kPushMaxRows;
      const WoaLayout L(pl.mtile, stages, nmax, tbmax, pl.push ? push_area_bytes(T, splits, false) : 0u);
      if (static_cast<size_t>(L.total) + 1024 > 232448) continue;
      pl.splits = splits;
      pl.stages = stages;
      pl.tmem_cols = pow2_at_least(((pl.mtile + 15) & ~15) + 8 * stages);
      const int max_res = 512 / pl.tmem_cols;
      const size_t min_smem = 233472 / static_cast<size_t>(max_res + 1) + 1;
      pl.smem = std::max(static_cast<size_t>(L.total) + 1024, min_smem);
      return pl;
    }
  }
  pl.smem = 0;  // no plan fits: rejected by launch_wo_a
  return pl;
}

cudaError_t set_wo_a_attributes() {
  for (const void* k : {reinterpret_cast<const void*>(&wo_a_kernel<false>),
                        reinterpret_cast<const void*>(&wo_a_kernel<true>)}) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_wo_a(const CUtensorMap& tm_w, const WoaArgs& args, const WoaPlan& plan,
                        cudaStream_t stream) {
  if (plan.smem == 0 || plan.smem > 232448) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(args.G * (args.R / 128), plan.splits, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 1;
  attrs[0].val.clusterDim.y = plan.splits;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  return plan.push ? cudaLaunchKernelEx(&cfg, wo_a_kernel<true>, tm_w, args)
                   : cudaLaunchKernelEx(&cfg, wo_a_kernel<false>, tm_w, args);
}

}  // namespace mx
