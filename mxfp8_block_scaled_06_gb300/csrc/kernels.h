// kernels.h - host-side launchers of the CUDA kernels (internal to libmx).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mx {

// Largest dynamic shared memory one CTA may ask for on sm_103a.
constexpr size_t kMaxDynamicSmem = 232448;

// ------------------------------------------------------------ quantizer
// Inverse RoPE applied before quantizing (WO-A activation): rows are tokens of
// heads of head_dim, dims from d_nope on rotated by -pos * f; cos_sin null = none.
struct RopeArgs {
  const int64_t* positions;
  const float* cos_sin;  // [max_pos, 64]: 32 cos | 32 sin
  int max_pos, head_dim, d_nope;
  int* status;
};
cudaError_t launch_quantize_rows(const void* x, long ldx, int M, int K, void* q, void* scales,
                                 int swizzled, cudaStream_t stream,
                                 const RopeArgs& rope = RopeArgs{nullptr, nullptr, 0, 0, 0, nullptr});

// y = bf16(x / sqrt(mean(x^2) + eps) * gamma) per row (float32 arithmetic), then
// MX-quantized into q / scales; y may be null.
cudaError_t launch_rmsnorm_quantize_rows(const void* x, long ldx, int M, int K, const void* gamma,
                                         float eps, void* y, void* q, void* scales, int swizzled,
                                         cudaStream_t stream);

// One thread waits on an mbarrier nothing completes; after the bounded wait's
// limit it sets the timeout bit of *status and returns.
cudaError_t launch_wait_selftest(int* status, cudaStream_t stream);

// ------------------------------------------------------------ block-scaled GEMM
// Plan of one GEMM launch: activation tile (MMA N), K-splits per weight tile
// (a thread-block cluster along K), pipeline depth, TMEM columns, shared bytes.
struct GemmPlan {
  int mtile;
  int splits;
  int stages;
  int tmem_cols;
  size_t smem;
};

struct GemmArgs {
  int M, N, K;
  int mtile, stages, nchunks, tmem_cols;
  const uint8_t* a_scales;  // MXFP8 activations' swizzled scales (unused when x is set)
  const uint8_t* w_scales;
  // bf16 activations [M, K] (row stride ldx elements) quantized inside the
  // kernel instead of MXFP8 activations through tm_a / a_scales; null = MXFP8 in
  const uint16_t* x;
  long ldx;
  // Grouped activations (0 = not grouped): weight tile t belongs to group
  // g = t / group_tiles and contracts the group's K-slice [g K, (g + 1) K) of
  // a wider MXFP8 activation whose scale layout has a_sf_chunks 128-wide
  // column blocks per row tile (= K / 128 when not grouped).
  int group_tiles;
  int a_sf_chunks;
  void* out;          // bf16 [M, N] or null
  uint8_t* q;         // fused requantization of columns [0, q_cols): E4M3 [M, q_cols]
  uint8_t* q_scales;  // swizzled scales of q
  int q_cols;
  int* status;
#ifdef MX_TIMELINE
  unsigned long long* tl;  // kTimelineSlots %globaltimer stamps per CTA, or null
#endif
};

#ifdef MX_TIMELINE
// Timeline build only: stamps per CTA of one GEMM launch (see gemm.cu).
constexpr int kTimelineSlots = 12;
constexpr int kTimelineCtas = 512;
#endif

GemmPlan plan_gemm(int M, int N, int K, int sm_count, bool fused_a = false);
cudaError_t set_gemm_attributes();
cudaError_t launch_gemm(const CUtensorMap& tm_w, const CUtensorMap& tm_a, const GemmArgs& args,
                        const GemmPlan& plan, bool pdl, cudaStream_t stream);

// ------------------------------------------------------------ grouped WO-A
struct WoaPlan {
  int mtile;
  int splits;
  int stages;
  int tmem_cols;
  size_t smem;
};

struct WoaArgs {
  int T, G, H, R, D;  // tokens, groups, heads per group, o_lora_rank, head dim (512)
  int mtile, stages, tmem_cols;
  const uint16_t* x;  // bf16 bits
  long ldx;
  const int64_t* positions;
  const float* cos_sin;
  int max_pos;
  const uint8_t* w_scales;
  uint8_t* q;
  uint8_t* q_scales;
  uint16_t* debug_z;
  uint8_t* debug_xq;
  uint8_t* debug_xs;
  int early_trigger;
  int* status;
};

WoaPlan plan_wo_a(int T, int G, int H, int R, int sm_count);
cudaError_t set_wo_a_attributes();
cudaError_t launch_wo_a(const CUtensorMap& tm_w, const WoaArgs& args, const WoaPlan& plan,
                        cudaStream_t stream);

}  // namespace mx
