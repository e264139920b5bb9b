// gemm.cu - low-batch MXFP8 block-scaled GEMM on tcgen05 (sm_103a).
//
// out[M, N] = dequant(A[M, K]) x dequant(W[N, K])^T, bf16 out, fp32 accumulate.
//
// Swap-AB: the 128 weight rows of a tile are the MMA's M (the only M the
// block-scaled tcgen05.mma takes with one CTA) and the activation rows,
// padded to a multiple of 16, are the MMA's N, so 1..256 rows cost one MMA
// shape. The kernel is bound by the weight stream from HBM; everything below
// is arranged around keeping that stream saturated:
//  * grid = (N/128 weight tiles) x (K splits); the splits of one tile form a
//    thread-block cluster and reduce their partial sums through distributed
//    shared memory (no global workspace, no second kernel);
//  * one thread issues TMA loads of 128x128-byte weight boxes (SWIZZLE_128B)
//    and 512-byte scale tiles for the whole pipeline depth BEFORE the
//    programmatic-dependent-launch wait, so under PDL the weight read overlaps
//    the previous kernel on the stream; activations (produced by that kernel)
//    are loaded only after the wait;
//  * one thread issues tcgen05.cp (scales -> TMEM) and four
//    tcgen05.mma.kind::mxf8f6f4.block_scale (K = 32 each) per 128-wide chunk,
//    and frees the stage with tcgen05.commit;
//  * the four warps read the fp32 accumulator from TMEM (warp w owns lanes
//    32w..32w+31 = weight rows), stage it in shared memory, and after a cluster
//    barrier each (row, 32-column block) of the output is summed over the
//    cluster's partials by one warp; the optional fused requantization (the
//    chain's next MXFP8 activation) takes the warp's 32 values as one block.
// Every mbarrier wait is bounded; on expiry the kernel records MX_ERR_TIMEOUT,
// skips the remaining work, drains its outstanding copies and frees TMEM.
#include <cuda_bf16.h>

#include <algorithm>

#include "kernels.h"
#include "ptx.cuh"

namespace mx {
namespace {

constexpr int kThreads = 128;
constexpr uint32_t kWTileBytes = 128 * 128;  // one weight box: 128 rows x 128 K-bytes
constexpr uint32_t kSfTileBytes = 512;       // one 128x4 scale tile

struct Layout {
  uint32_t a_bytes, sfb_bytes, stage_bytes;
  __host__ __device__ Layout(int mtile) {
    a_bytes = static_cast<uint32_t>(mtile) * 128u;
    sfb_bytes = kSfTileBytes * static_cast<uint32_t>((mtile + 127) / 128);
    stage_bytes = (kWTileBytes + a_bytes + kSfTileBytes + sfb_bytes + 1023u) & ~1023u;
  }
  __host__ __device__ uint32_t w_off(int s) const { return s * stage_bytes; }
  __host__ __device__ uint32_t a_off(int s) const { return s * stage_bytes + kWTileBytes; }
  __host__ __device__ uint32_t sfa_off(int s) const { return a_off(s) + a_bytes; }
  __host__ __device__ uint32_t sfb_off(int s) const { return sfa_off(s) + kSfTileBytes; }
};

__host__ __device__ inline int tmem_sfa_col(int mtile) { return (mtile + 15) & ~15; }

template <bool kRequant>
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
  const int nsfb = (p.mtile + 127) / 128;
  const Layout L(p.mtile);

  const uint32_t bars = base + stages * L.stage_bytes;
  auto wfull = [&](int s) { return bars + 8u * s; };
  auto afull = [&](int s) { return bars + 8u * (stages + s); };
  auto empty = [&](int s) { return bars + 8u * (2 * stages + s); };
  const uint32_t accum_bar = bars + 24u * stages;
  uint32_t* const tmem_slot =
      reinterpret_cast<uint32_t*>(base_ptr + stages * L.stage_bytes + 8 * (3 * stages + 1));
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(wfull(s), 1);
      mbar_init(afull(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(accum_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_a);
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sfa_col = tmem_sfa_col(p.mtile);
  const uint32_t sfb_col = sfa_col + 4 * stages;

  auto fail = [&]() {
    atomicOr(p.status, kStatusTimeout);
    *abort_flag = 1;
  };

  // ---------------- weights first: they do not depend on the previous kernel
  const uint64_t pol_w = policy_evict_first();
  const uint64_t pol_a = policy_evict_last();
  auto issue_w = [&](int i) {
    const int s = i % stages;
    const int c = c_begin + i;
    mbar_expect_tx(wfull(s), kWTileBytes + kSfTileBytes);
    tma_load_2d(base + L.w_off(s), &tm_w, wfull(s), c * 128, tile * 128, pol_w);
    bulk_load(base + L.sfa_off(s),
              p.w_scales + (static_cast<size_t>(tile) * p.nchunks + c) * kSfTileBytes,
              kSfTileBytes, wfull(s), pol_w);
  };
  auto issue_a = [&](int i) {
    const int s = i % stages;
    const int c = c_begin + i;
    mbar_expect_tx(afull(s), L.a_bytes + L.sfb_bytes);
    tma_load_2d(base + L.a_off(s), &tm_a, afull(s), c * 128, 0, pol_a);
    for (int rt = 0; rt < nsfb; ++rt)
      bulk_load(base + L.sfb_off(s) + rt * kSfTileBytes,
                p.a_scales + (static_cast<size_t>(rt) * p.nchunks + c) * kSfTileBytes,
                kSfTileBytes, afull(s), pol_a);
  };
  const int npre = min(n, stages);
  int w_issued = 0, a_issued = 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < npre; ++i) issue_w(i);
    w_issued = npre;
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();

  if (threadIdx.x == 0) {
    // ---------------- producer
    for (int i = 0; i < npre; ++i) issue_a(i);
    a_issued = npre;
    for (int i = npre; i < n; ++i) {
      const int s = i % stages;
      if (*abort_flag || !mbar_wait(empty(s), ((i / stages) - 1) & 1)) {
        fail();
        break;
      }
      issue_w(i);
      ++w_issued;
      issue_a(i);
      ++a_issued;
    }
  } else if (threadIdx.x == 32) {
    // ---------------- MMA issuer
    for (int i = 0; i < n; ++i) {
      const int s = i % stages;
      const uint32_t ph = (i / stages) & 1;
      if (*abort_flag || !mbar_wait(wfull(s), ph) || !mbar_wait(afull(s), ph)) {
        fail();
        break;
      }
      tc_fence_after();
      const uint32_t ta = tmem + sfa_col + 4 * s;
      const uint32_t tb = tmem + sfb_col + 4 * nsfb * s;
      tmem_cp_32x128b_x4(ta, sdesc_sf(base + L.sfa_off(s)));
      for (int rt = 0; rt < nsfb; ++rt)
        tmem_cp_32x128b_x4(tb + 4 * rt, sdesc_sf(base + L.sfb_off(s) + rt * kSfTileBytes));
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_mxf8(tmem, sdesc_k_sw128(base + L.w_off(s) + 32 * kk),
                 sdesc_k_sw128(base + L.a_off(s) + 32 * kk), idesc_mxf8(p.mtile, kk), ta, tb,
                 (i | kk) != 0);
      }
      tc_commit(empty(s));
    }
    tc_commit(accum_bar);
  }

  // ---------------- epilogue: TMEM -> shared partials
  if (!mbar_wait(accum_bar, 0)) fail();
  tc_fence_after();
  __syncwarp();
  float* const red = reinterpret_cast<float*>(base_ptr);
  const bool ok = (*abort_flag == 0);
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

  // ---------------- cluster reduction + bf16 (+ MXFP8) store
  if (ok) {
    const uint32_t red_addr = smem_u32(red);
    __nv_bfloat16* const out = static_cast<__nv_bfloat16*>(p.out);
    for (int item = split + S * warp; item < p.M * 4; item += 4 * S) {
      const int m = item >> 2;
      const int nl = (item & 3) * 32 + lane;
      const uint32_t off = red_addr + static_cast<uint32_t>(m * 128 + nl) * 4u;
      const float acc = cluster_sum(off, S);
      const __nv_bfloat16 hb = __float2bfloat16_rn(acc);
      const int col = tile * 128 + nl;
      if (out != nullptr) out[static_cast<size_t>(m) * p.N + col] = hb;
      if (kRequant && tile * 128 + (item & 3) * 32 < p.q_cols) {
        const float v = __bfloat162float(hb);
        float amax = fabsf(v);
        uint32_t nonfinite = !isfinite(v);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
          nonfinite |= __shfl_xor_sync(0xFFFFFFFFu, nonfinite, o);
        }
        uint32_t sbyte, code;
        if (nonfinite) {
          sbyte = 0xFFu;
          code = 0x7Fu;
        } else {
          sbyte = mx_scale_byte(amax);
          code = cvt_e4m3x2(v * mx_inv_scale(sbyte), 0.f) & 0xFFu;
        }
        p.q[static_cast<size_t>(m) * p.q_cols + col] = static_cast<uint8_t>(code);
        if (lane == 0) p.q_scales[swz_offset(m, col >> 5, p.q_cols >> 5)] = static_cast<uint8_t>(sbyte);
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
  cluster_sync();

  // ---------------- teardown
  if (!ok && threadIdx.x == 0) {
    // wait (bounded) for every copy this CTA issued, so none lands after exit
    for (int i = 0; i < w_issued; ++i) mbar_wait(wfull(i % stages), (i / stages) & 1);
    for (int i = 0; i < a_issued; ++i) mbar_wait(afull(i % stages), (i / stages) & 1);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

}  // namespace

GemmPlan plan_gemm(int M, int N, int K, int sm_count) {
  GemmPlan pl{};
  pl.mtile = (M + 15) & ~15;
  const int tiles = N / 128;
  const int nchunks = K / 128;
  int splits = std::max(1, sm_count / std::max(tiles, 1));
  splits = std::min(splits, std::min(8, nchunks));
  if (const char* e = getenv("MX_SPLITS")) {
    const int v = atoi(e);
    if (v >= 1 && v <= 8) splits = std::min(v, nchunks);
  }
  pl.splits = splits;
  const int per_cta = (nchunks + splits - 1) / splits;
  const Layout L(pl.mtile);
  const size_t budget = 96 * 1024;
  int stages = static_cast<int>(budget / L.stage_bytes);
  stages = std::max(2, std::min(stages, 8));
  if (const char* e = getenv("MX_STAGES")) {
    const int v = atoi(e);
    if (v >= 1 && v <= 12) stages = v;
  }
  stages = std::min(stages, per_cta);
  // the epilogue stages the fp32 partials [mtile][128] in the pipeline buffers
  while (static_cast<size_t>(stages) * L.stage_bytes < static_cast<size_t>(pl.mtile) * 512) ++stages;
  pl.stages = stages;
  const int nsfb = (pl.mtile + 127) / 128;
  pl.tmem_cols = pow2_at_least(tmem_sfa_col(pl.mtile) + 4 * stages + 4 * nsfb * stages);
  size_t smem = 1024 + static_cast<size_t>(stages) * L.stage_bytes + 8 * (3 * stages + 1) + 16;
  // CTAs that can share an SM must fit their TMEM together: ask for enough
  // shared memory that at most 512 / tmem_cols of them are resident.
  const int max_res = 512 / pl.tmem_cols;
  const size_t min_smem = 233472 / static_cast<size_t>(max_res + 1) + 1;
  pl.smem = std::max(smem, min_smem);
  return pl;
}

cudaError_t set_gemm_attributes() {
  const void* ks[2] = {reinterpret_cast<const void*>(&gemm_kernel<false>),
                       reinterpret_cast<const void*>(&gemm_kernel<true>)};
  for (const void* k : ks) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_gemm(const CUtensorMap& tm_w, const CUtensorMap& tm_a, const GemmArgs& args,
                        const GemmPlan& plan, bool pdl, cudaStream_t stream) {
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
  if (args.q != nullptr) return cudaLaunchKernelEx(&cfg, gemm_kernel<true>, tm_w, tm_a, args);
  return cudaLaunchKernelEx(&cfg, gemm_kernel<false>, tm_w, tm_a, args);
}

}  // namespace mx
