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
// Plan overrides for tuning, read from the environment once per handle (at
// mx_create): MX_SPLITS (K-splits of every GEMM, 1..8), MX_STAGES (ring depth),
// MX_PLAN_AT ("NxK:splits[:stages],..." for listed weight shapes),
// MX_WOA_SPLITS (fused WO-A K-splits). Zero / empty = none.
struct PlanEnv {
  int splits;
  int stages;
  int woa_splits;
  int push_rows;  // the push reduction up to this many rows (0: the default)
  char plan_at[256];
};
PlanEnv read_plan_env();

// How the K-splits' fp32 partials are summed (every form in rank order):
// items = a warp sums 32-column items from the peers' shared memory; rows = a
// warp sums whole rows with 16-byte peer loads; push = every CTA stores the
// partials of the units another rank owns straight into that rank's shared
// memory (st.async, counted on its mbarrier) and sums its own units locally,
// with a receive slot per rank, or (compact) per peer.
enum Reduction : int { kReduceItems = 0, kReduceRows = 1, kReducePush = 2, kReducePushCompact = 3 };
// Whether a plan may take the push reduction, and with which receive area.
enum PushMode : int { kPushNone = 0, kPushCompact = 1, kPushFull = 2 };

struct GemmPlan {
  int mtile;
  int splits;
  int stages;
  int tmem_cols;
  int reduction;  // Reduction
  size_t smem;
};

// RMS norm of the bf16 activation rows before their quantization (in-kernel
// quantization only; gamma null = none): y = bf16(x * 1/sqrt(mean(x^2) + eps) *
// gamma), the mean over the row's K values. The sum of squares is read, not
// computed: ssq [M, K/32] holds each 32-block's sum of its squares (written by
// the previous GEMM's epilogue, ssq_out), added here in block order. Tile 0's
// CTAs also write, over their K-range, the normalized rows to y [M, K] and the
// MXFP8 activation to a_q [M, K] and its swizzled scales a_q_scales (each null =
// not written).
struct GemmNorm {
  const uint16_t* gamma;
  float eps;
  const float* ssq;
  uint16_t* y;
  uint8_t* a_q;
  uint8_t* a_q_scales;
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
  GemmNorm norm;
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
  // per-32-block sums of squares of the bf16 output, columns [0, ssq_cols):
  // ssq_out[m * ssq_cols / 32 + c / 32], each the xor-shuffle tree over the
  // block's 32 values (null = not written)
  float* ssq_out;
  int ssq_cols;
  int* status;
#ifdef MX_TIMELINE
  unsigned long long* tl;  // kTimelineSlots %globaltimer stamps per CTA, or null
#endif
};

#ifdef MX_TIMELINE
// Timeline build only: stamps per CTA of one GEMM launch (see gemm.cu).
constexpr int kTimelineSlots = 20;
constexpr int kTimelineCtas = 512;
#endif

// fused_a: bf16 activations quantized in the kernel; norm: with the RMS norm;
// push_mode: whether the push reduction may be chosen, and its receive area;
// table_depth: the ring depth of the split table's row (false: as planned).
GemmPlan plan_gemm(int M, int N, int K, int sm_count, const PlanEnv& env, bool fused_a = false,
                   bool norm = false, int push_mode = kPushFull, bool table_depth = true);
cudaError_t set_gemm_attributes();
cudaError_t launch_gemm(const CUtensorMap& tm_w, const CUtensorMap& tm_a, const GemmArgs& args,
                        const GemmPlan& plan, bool pdl, cudaStream_t stream);

// ------------------------------------------------------------ persistent chain
// The three projections of mx_gemm_chain in one persistent kernel (chain.cu):
// clusters of kChainCluster CTAs, one CTA per SM, every CTA resident at once.
constexpr int kChainCluster = 8;
constexpr int kChainMaxUnits = 8;      // (tile, K split) work units per CTA, all projections
constexpr int kChainCounters = 16384;  // 32-bit words of the handle's chain workspace

// One projection as the chain kernel sees it.
struct ChainProj {
  const uint8_t* w_scales;  // swizzled [n, k/32]
  const uint8_t* a_scales;  // swizzled scales of the activation [M, k]
  int n, k;
  int splits;               // CTAs (ranks of one cluster) sharing a weight tile's K-range
  void* out;                // bf16 [M, n], or null
  uint8_t* q;               // MX requantization of columns [0, q_cols): the next activation
  uint8_t* q_scales;
  int q_cols;
};

// Shared-memory and TMEM plan of the chain kernel (offsets from the CTA's
// 1024-aligned base); ok == false: the three-launch path serves the call.
struct ChainPlan {
  bool ok;
  int clusters, ring, tmem_cols;
  int act_chunks[3], max_units[3];
  uint32_t off_act[3], off_asf[3], off_staged, off_recv[3], recv_unit_bytes[3], off_bars;
  size_t smem;
};

struct ChainArgs {
  int M, mtile, nsfb;
  ChainProj proj[3];
  ChainPlan plan;
  // workspace: [0] calls completed, [1] CTAs finished in this call, [2] abort,
  // then one counter per weight tile of the first two projections (from
  // cnt_off), zero at the start of every call
  unsigned* counters;
  int cnt_off[2];
  int* status;
#ifdef MX_TIMELINE
  unsigned long long* tl;  // kTimelineSlots %globaltimer stamps per CTA, or null
#endif
};

ChainPlan plan_chain(int M, const ChainProj (&proj)[3], int clusters);
// Clusters of kChainCluster CTAs of the chain kernel that can be resident at once.
int chain_max_clusters();
cudaError_t set_chain_attributes();
cudaError_t launch_chain(const CUtensorMap (&maps)[6], const ChainArgs& args, cudaStream_t stream);

// ------------------------------------------------------------ grouped WO-A
struct WoaPlan {
  int mtile;
  int splits;
  int stages;
  int tmem_cols;
  bool push;  // the push split-K reduction (full receive area)
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
#ifdef MX_TIMELINE
  unsigned long long* tl;  // kTimelineSlots %globaltimer stamps per CTA, or null
#endif
};

WoaPlan plan_wo_a(int T, int G, int H, int R, int sm_count, const PlanEnv& env);
cudaError_t set_wo_a_attributes();
cudaError_t launch_wo_a(const CUtensorMap& tm_w, const WoaArgs& args, const WoaPlan& plan,
                        cudaStream_t stream);

}  // namespace mx
