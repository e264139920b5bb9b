// quantize.cu - bf16 rows -> MXFP8 (E4M3 + one UE8M0 scale per 32 along K).
//
// One warp owns 8 consecutive 32-blocks (256 elements, 512 input bytes) of one
// row; each lane loads 16 bytes (8 bf16), four lanes form a block and combine
// their partial amax with two xor-shuffles. Loads are 512-byte coalesced per
// warp, stores 256 bytes. Padding of the swizzled scale buffer (rows up to a
// multiple of 128, block columns up to a multiple of 4) is written as zero by
// the same grid so the whole buffer is defined.
//
// Optionally (rope != null) the rows are attention heads of `head_dim` whose
// last dims from `d_nope` on are rotated first, the inverse RoPE of the WO-A
// projection: adjacent pairs (a, b) at rope dim 2i become (a c + b s, b c - a s)
// with c, s = the float32 cos/sin of the row's position (cache row [32 cos |
// 32 sin]), each product and sum rounded to float32 (no fused multiply-add).
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace mx {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kPadRows = 8;  // swizzled-scale padding rows zeroed by one warp

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    quantize_rows_kernel(const uint16_t* __restrict__ x, long ldx, int M, int K,
                         uint8_t* __restrict__ q, uint8_t* __restrict__ scales, int swizzled,
                         int rows_total, int groups_per_row, RopeArgs rope) {
  // Programmatic dependent launch: let the next kernel (typically a GEMM that
  // streams its weights first) start now; wait for the previous kernel before
  // touching memory it may produce or read.
  pdl_launch_dependents();
  // The warp's row and 32-block (or padding rows) touch no memory, so they are
  // worked out before the wait: its divisions stay off the path from the
  // previous kernel's end to the first load.
  const long gw = static_cast<long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int nblk = K >> 5;
  const int cpad4 = (nblk + 3) & ~3;
  const long real_warps = static_cast<long>(M) * groups_per_row;
  const bool pad = gw >= real_warps;
  long wq = (pad ? gw - real_warps : gw) / groups_per_row;
  int wgrp = static_cast<int>((pad ? gw - real_warps : gw) - wq * groups_per_row);
  asm volatile("" : "+l"(wq), "+r"(wgrp));  // computed before the wait, not sunk below it
  pdl_wait();
  if (pad) {
    // padding rows [M, rows_total) of the swizzled scales: zero, kPadRows rows per warp
    const int r0 = M + static_cast<int>(wq) * kPadRows;
    const int blk = wgrp * 8 + (lane >> 2);
    if (r0 >= rows_total || (lane & 3) != 0 || blk >= cpad4) return;
    for (int r = r0; r < min(r0 + kPadRows, rows_total); ++r) scales[swz_offset(r, blk, cpad4)] = 0;
    return;
  }
  const int row = static_cast<int>(wq);
  const int grp = wgrp;
  const int blk = grp * 8 + (lane >> 2);
  const int sub = lane & 3;
  const bool valid = row < M && blk < nblk;

  float v[8];
  float amax = 0.f;
  uint32_t nonfinite = 0;
  if (valid) {
    const uint4 raw =
        *reinterpret_cast<const uint4*>(x + static_cast<size_t>(row) * ldx + blk * 32 + sub * 8);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    const int d = (blk * 32 + sub * 8) % (rope.cos_sin != nullptr ? rope.head_dim : 1);
    if (rope.cos_sin != nullptr && d >= rope.d_nope) {
      long long pos = rope.positions[row];
      if (pos < 0 || pos >= rope.max_pos) {
        atomicOr(rope.status, kStatusBadInput);  // position outside the cache: row 0
        pos = 0;
      }
      const float* cs = rope.cos_sin + static_cast<size_t>(pos) * 64;
      const int p0 = (d - rope.d_nope) >> 1;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float c = cs[p0 + i], sn = cs[32 + p0 + i];
        const float a = v[2 * i], b = v[2 * i + 1];
        v[2 * i] = __fadd_rn(__fmul_rn(a, c), __fmul_rn(b, sn));
        v[2 * i + 1] = __fsub_rn(__fmul_rn(b, c), __fmul_rn(a, sn));
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

  uint32_t sbyte = 0;
  if (valid) {
    uint32_t lo, hi;
    if (nonfinite) {
      sbyte = 0xFFu;
      lo = hi = 0x7F7F7F7Fu;
    } else {
      sbyte = mx_scale_byte(amax);
      const float f = mx_inv_scale(sbyte);
      lo = cvt_e4m3x2(v[0] * f, v[1] * f) | (cvt_e4m3x2(v[2] * f, v[3] * f) << 16);
      hi = cvt_e4m3x2(v[4] * f, v[5] * f) | (cvt_e4m3x2(v[6] * f, v[7] * f) << 16);
    }
    *reinterpret_cast<uint2*>(q + static_cast<size_t>(row) * K + blk * 32 + sub * 8) =
        make_uint2(lo, hi);
  }
  if (sub == 0) {
    if (swizzled) {
      if (blk < cpad4) scales[swz_offset(row, blk, cpad4)] = static_cast<uint8_t>(sbyte);
    } else if (valid) {
      scales[static_cast<size_t>(row) * nblk + blk] = static_cast<uint8_t>(sbyte);
    }
  }
}

// RMS normalization + MX quantization of rows (the split between the first two
// decode projections): one warp per row; pass 1 sums the squares of the row in
// float32 in a fixed order (per 32-block a tree, then the blocks in order),
// pass 2 scales each element by 1/sqrt(mean + eps) (correctly rounded sqrt and
// division) and the row's weight, rounds to bf16 (optionally stored) and
// quantizes per 32-block as quantize_rows_kernel does.
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    rmsnorm_quantize_rows_kernel(const uint16_t* __restrict__ x, long ldx, int M, int K,
                                 const uint16_t* __restrict__ gamma, float eps,
                                 uint16_t* __restrict__ y, uint8_t* __restrict__ q,
                                 uint8_t* __restrict__ scales, int swizzled, int rows_total) {
  pdl_launch_dependents();
  pdl_wait();
  const int row = static_cast<int>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows_total) return;  // warp-uniform
  const int nblk = K >> 5;
  const int cpad4 = (nblk + 3) & ~3;
  const int groups = (cpad4 + 7) / 8;  // 8 blocks (256 elements) per pass of the warp
  const bool real = row < M;
  const uint16_t* const xr = x + static_cast<size_t>(row) * ldx;
  // Sum of squares: each 32-block's squares are added in the xor-shuffle tree
  // over the block's 32 elements (element j pairs with j ^ 16, then j ^ 8, ...:
  // the order the GEMM epilogue uses when it writes a row's block sums), and the
  // block sums in block order. Lane l holds elements 8 (l & 3) .. 8 (l & 3) + 7 of
  // block l / 4: the tree's first two levels pair lanes (l ^ 2, l ^ 1), the last
  // three pair elements within the lane.
  float ss = 0.f;
  for (int g = 0; g < groups; ++g) {
    const int blk = g * 8 + (lane >> 2);
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (real && blk < nblk) raw = *reinterpret_cast<const uint4*>(xr + blk * 32 + (lane & 3) * 8);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    float s[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = __uint_as_float(w[i] << 16), b = __uint_as_float(w[i] & 0xFFFF0000u);
      s[2 * i] = __fmul_rn(a, a);
      s[2 * i + 1] = __fmul_rn(b, b);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) s[e] = __fadd_rn(s[e], __shfl_xor_sync(0xFFFFFFFFu, s[e], 2));
#pragma unroll
    for (int e = 0; e < 8; ++e) s[e] = __fadd_rn(s[e], __shfl_xor_sync(0xFFFFFFFFu, s[e], 1));
#pragma unroll
    for (int e = 0; e < 4; ++e) s[e] = __fadd_rn(s[e], s[e + 4]);
    s[0] = __fadd_rn(s[0], s[2]);
    s[1] = __fadd_rn(s[1], s[3]);
    s[0] = __fadd_rn(s[0], s[1]);
    // block g * 8 + b sits in lanes 4b .. 4b + 3; every lane adds the same sequence
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const float blk_sum = __shfl_sync(0xFFFFFFFFu, s[0], 4 * b);
      if (g * 8 + b < nblk) ss = __fadd_rn(ss, blk_sum);
    }
  }
  const float inv = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(K)), eps)));
  for (int g = 0; g < groups; ++g) {
    const int blk = g * 8 + (lane >> 2);
    const int sub = lane & 3;
    const bool valid = real && blk < nblk;
    float v[8];
    float amax = 0.f;
    uint32_t nonfinite = 0;
    if (valid) {
      const int k0 = blk * 32 + sub * 8;
      const uint4 raw = *reinterpret_cast<const uint4*>(xr + k0);
      const uint4 graw = *reinterpret_cast<const uint4*>(gamma + k0);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
      const uint32_t gw[4] = {graw.x, graw.y, graw.z, graw.w};
      uint32_t packed[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = __fmul_rn(__fmul_rn(__uint_as_float(w[i] << 16), inv), __uint_as_float(gw[i] << 16));
        const float b = __fmul_rn(__fmul_rn(__uint_as_float(w[i] & 0xFFFF0000u), inv),
                                  __uint_as_float(gw[i] & 0xFFFF0000u));
        const uint32_t ha = __bfloat16_as_ushort(__float2bfloat16_rn(a));
        const uint32_t hb = __bfloat16_as_ushort(__float2bfloat16_rn(b));
        packed[i] = ha | (hb << 16);
        v[2 * i] = __uint_as_float(ha << 16);
        v[2 * i + 1] = __uint_as_float(hb << 16);
      }
      if (y != nullptr)
        *reinterpret_cast<uint4*>(y + static_cast<size_t>(row) * K + k0) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
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
    uint32_t sbyte = 0;
    if (valid) {
      uint32_t lo, hi;
      if (nonfinite) {
        sbyte = 0xFFu;
        lo = hi = 0x7F7F7F7Fu;
      } else {
        sbyte = mx_scale_byte(amax);
        const float f = mx_inv_scale(sbyte);
        lo = cvt_e4m3x2(v[0] * f, v[1] * f) | (cvt_e4m3x2(v[2] * f, v[3] * f) << 16);
        hi = cvt_e4m3x2(v[4] * f, v[5] * f) | (cvt_e4m3x2(v[6] * f, v[7] * f) << 16);
      }
      *reinterpret_cast<uint2*>(q + static_cast<size_t>(row) * K + blk * 32 + sub * 8) =
          make_uint2(lo, hi);
    }
    if (sub == 0) {
      if (swizzled) {
        if (blk < cpad4) scales[swz_offset(row, blk, cpad4)] = static_cast<uint8_t>(sbyte);
      } else if (valid) {
        scales[static_cast<size_t>(row) * nblk + blk] = static_cast<uint8_t>(sbyte);
      }
    }
  }
}

}  // namespace

cudaError_t launch_rmsnorm_quantize_rows(const void* x, long ldx, int M, int K, const void* gamma,
                                         float eps, void* y, void* q, void* scales, int swizzled,
                                         cudaStream_t stream) {
  const int rows_total = swizzled ? ((M + 127) / 128) * 128 : M;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows_total + kWarpsPerBlock - 1) / kWarpsPerBlock), 1, 1);
  cfg.blockDim = dim3(kWarpsPerBlock * 32, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, rmsnorm_quantize_rows_kernel, static_cast<const uint16_t*>(x), ldx,
                            M, K, static_cast<const uint16_t*>(gamma), eps, static_cast<uint16_t*>(y),
                            static_cast<uint8_t*>(q), static_cast<uint8_t*>(scales), swizzled,
                            rows_total);
}

cudaError_t launch_quantize_rows(const void* x, long ldx, int M, int K, void* q, void* scales,
                                 int swizzled, cudaStream_t stream, const RopeArgs& rope) {
  const int nblk = K / 32;
  const int cols = swizzled ? ((nblk + 3) & ~3) : nblk;
  const int groups_per_row = (cols + 7) / 8;
  const int rows_total = swizzled ? ((M + 127) / 128) * 128 : M;
  const long pad_warps = static_cast<long>((rows_total - M + kPadRows - 1) / kPadRows) * groups_per_row;
  const long warps = static_cast<long>(M) * groups_per_row + pad_warps;
  const long blocks = (warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kWarpsPerBlock * 32, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quantize_rows_kernel, static_cast<const uint16_t*>(x), ldx, M, K,
                            static_cast<uint8_t*>(q), static_cast<uint8_t*>(scales), swizzled,
                            rows_total, groups_per_row, rope);
}

// ------------------------------------------------------------ wait self-test
// One thread waits, through the same bounded mbar_wait the kernels use, on an
// mbarrier that nothing ever arrives on. The wait gives up after kWaitLimitNs,
// the thread records kStatusTimeout and the kernel returns: the failure path of
// every pipeline wait, taken on purpose and without a fault. Nothing is in
// flight on the barrier, so it is simply abandoned at exit.
__global__ void wait_selftest_kernel(int* status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  if (!mbar_wait(b, 0)) atomicOr(status, kStatusTimeout);
}

cudaError_t launch_wait_selftest(int* status, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 1, 0, stream>>>(status);
  return cudaGetLastError();
}

}  // namespace mx
