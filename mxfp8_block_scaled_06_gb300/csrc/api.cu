// api.cu - the C ABI of libmx (declared in include/mx.h): argument
// validation (always before any launch), launch plans, TMA tensor maps.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/mx.h"
#include "kernels.h"

// Tensor maps already encoded by this handle, by (address, rows, k, box rows):
// an eager caller reuses the same weight and activation buffers call after call,
// and encoding a map is host work on every launch otherwise. A map holds no
// device state, so a reused address with the same geometry gets the same map.
struct TmapEntry {
  const void* ptr;
  int rows;
  long k;
  int box_rows;
  CUtensorMap map;
};
constexpr int kTmapCache = 32;

// GEMM plans the handle has computed, by problem.
struct PlanEntry {
  int M, N, K;
  bool fused, norm;
  int push_mode;
  bool table_depth;
  mx::GemmPlan plan;
};
constexpr int kPlanCache = 64;

struct mx_handle {
  int device;
  int sm_count;
  size_t smem_per_sm;    // shared memory of an SM, and the reserve of each resident block
  size_t smem_reserved;
  mx::PlanEnv env;        // plan overrides, read once at mx_create
  bool chain_persistent;  // MX_CHAIN_PERSISTENT=1 at mx_create
  PlanEntry plans[kPlanCache];
  int plan_count;
  int plan_next;  // round-robin replacement
  int* d_status;
  unsigned* d_chain;   // persistent chain kernel's counters (kChainCounters words)
  int chain_clusters;  // clusters of 8 CTAs it may use (0: the three-launch path only)
  uint8_t* d_woa;      // wo_a_grouped's two-launch activation (kWoaScratchBytes)
  float* d_ssq;        // mx_gemm_chain_norm's block sums of squares (kSsqBytes)
  PFN_cuTensorMapEncodeTiled_v12000 encode;
  TmapEntry tmaps[kTmapCache];
  int tmap_count;
  int tmap_next;  // round-robin replacement
#ifdef MX_TIMELINE
  unsigned long long* d_tl;  // kTimelineLaunches x kTimelineCtas x kTimelineSlots stamps
  int tl_next;               // GEMM launches recorded since the last reset
#endif
};
// wo_a_grouped above kWoaFusedMaxTokens tokens runs the two-launch form and
// keeps its quantized activation in the handle: codes [T, G*H*D], then the
// swizzled scales at the next 256-byte boundary. Room for T = 128 tokens of
// G*H*D = 65536 (8 MiB of codes, 256 KiB of scales).
constexpr size_t kWoaScratchBytes = (size_t{8} << 20) + (size_t{256} << 10) + 256;
// Measured on GB300 (4 groups x 1024 rows, 8 heads of 512): the fused kernel
// is faster up to 8 tokens (7.5 against 8.1 us), the two launches from 12 on
// (8.3 against 8.4 us; 19 against 75 us at 128 tokens). Re-measured with both
// paths on the push split-K exchange: the two launches are faster from 10
// tokens on (7.85 / 7.85 / 8.12 us against 8.04 / 8.19 / 8.96 us at 10 / 12 /
// 16 tokens).
constexpr int kWoaFusedMaxTokens = 8;
// mx_gemm_chain_norm applies the RMS norm in G2's prologue up to this many rows
// (measured on GB300 with N1 = 2048, qr 1536, N2 = 8192, N3 = 5120; beyond, G2's
// CTAs each quantizing their K-range of every row cost more than a launch).
// Re-measured with the push split-K exchange: from 9 to 16 rows the fused form
// is still the faster (21.9 / 22.8 / 23.7 us against 25.4 / 25.0 / 25.6 us at
// 10 / 12 / 16 rows).
constexpr int kNormFusedMaxRows = 16;
// the block sums of squares G1 hands to G2 there: [M, g1_cols / 32] floats
constexpr size_t kSsqBytes = size_t{64} << 10;
#ifdef MX_TIMELINE
constexpr int kTimelineLaunches = 256;
constexpr size_t kTimelineBytes =
    sizeof(unsigned long long) * kTimelineLaunches * mx::kTimelineCtas * mx::kTimelineSlots;
#endif

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

int check_device(const mx_handle* h) {
  if (h == nullptr) return MX_ERR_INVALID_ARG;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return MX_ERR_CUDA;
  return cur == h->device ? MX_OK : MX_ERR_DEVICE;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MX_OK : MX_ERR_CUDA; }

// The GEMM plan of a problem, computed once per handle (mx_warmup computes those
// of the registered shapes ahead of the first call).
mx::GemmPlan get_plan(mx_handle* h, int M, int N, int K, bool fused = false, bool norm = false,
                      int push_mode = mx::kPushFull, bool table_depth = true) {
  for (int i = 0; i < h->plan_count; ++i) {
    const PlanEntry& e = h->plans[i];
    if (e.M == M && e.N == N && e.K == K && e.fused == fused && e.norm == norm && e.push_mode == push_mode &&
        e.table_depth == table_depth)
      return e.plan;
  }
  const mx::GemmPlan plan = mx::plan_gemm(M, N, K, h->sm_count, h->env, fused, norm, push_mode, table_depth);
  const int slot = h->plan_count < kPlanCache ? h->plan_count++ : h->plan_next;
  if (h->plan_count == kPlanCache) h->plan_next = (slot + 1) % kPlanCache;
  h->plans[slot] = PlanEntry{M, N, K, fused, norm, push_mode, table_depth, plan};
  return plan;
}

// A chain projection's plan, for the co-residency check below.
struct ChainShape {
  int N, K;
  bool fused, norm, table_depth;
};

// The push reduction of each projection of a three-launch chain (PushMode).
// Under PDL the next grid's CTAs start while the previous grid's still run, on
// the same SMs when both fit (shared memory, with the per-block reserve, and
// TMEM). For every pair of neighbours (G3 of the previous step before G1) that
// fits without the push reduction's receive areas, the chosen forms must fit
// too: where they do not, the later projection steps down first (full receive
// area, then the compact one, then none). plan(i, mode) is projection i's plan.
template <typename PlanFn>
void chain_push_modes(const ChainShape (&c)[3], int sm_count, size_t smem_per_sm, size_t smem_reserved,
                      PlanFn plan, int (&mode)[3]) {
  auto fits = [&](int pi, int pm, int i, int im) {
    const mx::GemmPlan prev = plan(pi, pm), next = plan(i, im);
    const int grid = c[pi].N / 128 * prev.splits;
    const size_t k = static_cast<size_t>((grid + sm_count - 1) / sm_count);
    return k * (prev.smem + smem_reserved) + next.smem + smem_reserved <= smem_per_sm &&
           k * prev.tmem_cols + next.tmem_cols <= 512;
  };
  auto mode_of = [](const mx::GemmPlan& pl) {
    return pl.reduction == mx::kReducePush          ? mx::kPushFull
           : pl.reduction == mx::kReducePushCompact ? mx::kPushCompact
                                                    : mx::kPushNone;
  };
  for (int i = 0; i < 3; ++i) mode[i] = mode_of(plan(i, mx::kPushFull));
  for (bool changed = true; changed;) {  // each pass steps one down, or ends
    changed = false;
    for (int i = 0; i < 3 && !changed; ++i) {
      const int pi = (i + 2) % 3;
      if (fits(pi, mx::kPushNone, i, mx::kPushNone) && !fits(pi, mode[pi], i, mode[i])) {
        const int j = mode[i] != mx::kPushNone ? i : pi;  // the later projection first
        mode[j] = mode[j] == mx::kPushFull && mode_of(plan(j, mx::kPushCompact)) == mx::kPushCompact
                      ? mx::kPushCompact
                      : mx::kPushNone;
        changed = true;
      }
    }
  }
}

void chain_push(mx_handle* h, int M, const ChainShape (&c)[3], int (&mode)[3]) {
  chain_push_modes(
      c, h->sm_count, h->smem_per_sm, h->smem_reserved,
      [&](int i, int m) { return get_plan(h, M, c[i].N, c[i].K, c[i].fused, c[i].norm, m, c[i].table_depth); },
      mode);
}

// mx_gemm_chain_norm applies the norm in G2's prologue (three launches) when
// the rows' block sums of squares fit the handle's buffer and the fused plan fits
// shared memory; otherwise the norm kernel runs between G1 and G2.
bool chain_norm_fused(int M, int g1_cols, size_t fused_g2_smem) {
  return M <= kNormFusedMaxRows && static_cast<size_t>(M) * (g1_cols / 32) * sizeof(float) <= kSsqBytes &&
         fused_g2_smem <= mx::kMaxDynamicSmem;
}

// 2-D uint8 tensor map over a row-major [rows, k] matrix, box {128 bytes, box_rows}
// with the 128-byte swizzle; out-of-range rows of a box read as zero.
int make_tmap(mx_handle* h, CUtensorMap* tm, const void* ptr, int rows, long k, int box_rows) {
  for (int i = 0; i < h->tmap_count; ++i) {
    const TmapEntry& e = h->tmaps[i];
    if (e.ptr == ptr && e.rows == rows && e.k == k && e.box_rows == box_rows) {
      *tm = e.map;
      return MX_OK;
    }
  }
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(k)};
  cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = h->encode(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return MX_ERR_CUDA;
  const int slot = h->tmap_count < kTmapCache ? h->tmap_count++ : h->tmap_next;
  if (h->tmap_count == kTmapCache) h->tmap_next = (slot + 1) % kTmapCache;
  h->tmaps[slot] = TmapEntry{ptr, rows, k, box_rows, *tm};
  return MX_OK;
}

int validate_gemm(mx_handle* h, int M, int N, int K, const void* a, const void* a_scales,
                  const void* w, const void* w_scales) {
  if (M < 1 || N < 1 || K < 1) return MX_ERR_INVALID_ARG;
  if (a == nullptr || a_scales == nullptr || w == nullptr || w_scales == nullptr)
    return MX_ERR_INVALID_ARG;
  if (!aligned(a, 16) || !aligned(a_scales, 16) || !aligned(w, 16) || !aligned(w_scales, 32))
    return MX_ERR_INVALID_ARG;
  if (K % 32 != 0) return MX_ERR_INVALID_ARG;
  if (M > 256 || N % 128 != 0 || K % 128 != 0) return MX_ERR_UNSUPPORTED;
  if (get_plan(h, M, N, K).smem > mx::kMaxDynamicSmem) return MX_ERR_UNSUPPORTED;
  return MX_OK;
}

// One GEMM launch, prepared (plan, tensor maps, arguments) before anything is
// enqueued, so that a call of several launches can fail before its first.
struct GemmLaunch {
  mx::GemmPlan plan;
  CUtensorMap tm_w, tm_a;
  mx::GemmArgs args;
};

// a = MXFP8 activations (+ a_scales), or x = bf16 activations with row stride
// ldx (quantized inside the kernel); exactly one of the two is non-null.
// groups > 1: a is [M, groups * K] and the weight tiles of group g (N / groups
// rows each) contract its K-slice g.
int gemm_prepare(mx_handle* h, GemmLaunch* L, int M, int N, int K, const void* a,
                 const void* a_scales, const void* w, const void* w_scales, void* out, uint8_t* q,
                 uint8_t* q_scales, int q_cols, const void* x = nullptr, long ldx = 0,
                 int groups = 1, const mx::GemmNorm* norm = nullptr, int push_mode = mx::kPushFull,
                 bool table_depth = true) {
  L->plan = get_plan(h, M, N, K, x != nullptr, norm != nullptr, push_mode, table_depth);
  int rc = make_tmap(h, &L->tm_w, w, N, K, 128);
  if (rc != MX_OK) return rc;
  if (x != nullptr) {
    L->tm_a = L->tm_w;  // not read by the fused kernel
  } else {
    rc = make_tmap(h, &L->tm_a, a, M, static_cast<long>(K) * groups, L->plan.mtile);
    if (rc != MX_OK) return rc;
  }
  mx::GemmArgs& args = L->args;
  args = mx::GemmArgs{};
  args.M = M;
  args.N = N;
  args.K = K;
  args.mtile = L->plan.mtile;
  args.stages = L->plan.stages;
  args.nchunks = K / 128;
  args.tmem_cols = L->plan.tmem_cols;
  args.a_scales = static_cast<const uint8_t*>(a_scales);
  args.w_scales = static_cast<const uint8_t*>(w_scales);
  args.x = static_cast<const uint16_t*>(x);
  args.ldx = ldx;
  args.group_tiles = groups > 1 ? N / groups / 128 : 0;
  args.a_sf_chunks = K / 128 * groups;
  args.out = out;
  args.q = q;
  args.q_scales = q_scales;
  args.q_cols = q_cols;
  if (norm != nullptr) args.norm = *norm;
  args.status = h->d_status;
  return MX_OK;
}

int gemm_run(mx_handle* h, GemmLaunch* L, bool pdl, cudaStream_t stream) {
#ifdef MX_TIMELINE
  L->args.tl = nullptr;
  if (h->d_tl != nullptr && (L->args.N / 128) * L->plan.splits <= mx::kTimelineCtas &&
      h->tl_next < kTimelineLaunches)
    L->args.tl = h->d_tl + static_cast<size_t>(h->tl_next++) * mx::kTimelineCtas * mx::kTimelineSlots;
#else
  (void)h;
#endif
  return cuda_status(mx::launch_gemm(L->tm_w, L->tm_a, L->args, L->plan, pdl, stream));
}

int gemm_launch(mx_handle* h, int M, int N, int K, const void* a, const void* a_scales,
                const void* w, const void* w_scales, void* out, uint8_t* q, uint8_t* q_scales,
                int q_cols, bool pdl, cudaStream_t stream, const void* x = nullptr, long ldx = 0,
                int groups = 1) {
  GemmLaunch L;
  const int rc = gemm_prepare(h, &L, M, N, K, a, a_scales, w, w_scales, out, q, q_scales, q_cols, x,
                              ldx, groups);
  return rc != MX_OK ? rc : gemm_run(h, &L, pdl, stream);
}

// The chain in one persistent kernel (chain.cu), when MX_CHAIN_PERSISTENT=1 and
// its plan exists (up to 16 rows, K splits of each projection's GEMM plan at
// most 8, enough resident clusters). Measured on GB300 it is slower than the
// three launches (39.6 vs 17.1 us at one row: its weight ring fills during each
// projection's dependency wait and every hand-off is a chain of ~0.5 us
// latencies), so the three launches are the default.
// Returns MX_OK after launching, MX_ERR_UNSUPPORTED when the three-launch path
// must serve the call, or an error before any launch.
int chain_persistent(mx_handle* h, int M, const void* a1, const void* a1_scales, const mx_weight w[3],
                     int g1_cols, void* a2, void* a2_scales, void* a3, void* a3_scales, void* out,
                     void* out1, void* out2, cudaStream_t stream) {
  if (!h->chain_persistent) return MX_ERR_UNSUPPORTED;
  if (h->chain_clusters < 1) return MX_ERR_UNSUPPORTED;
  mx::ChainArgs args = {};
  const void* acts[3] = {a1, a2, a3};
  const void* act_scales[3] = {a1_scales, a2_scales, a3_scales};
  void* outs[3] = {out1, out2, out};
  uint8_t* qs[3] = {static_cast<uint8_t*>(a2), static_cast<uint8_t*>(a3), nullptr};
  uint8_t* qscales[3] = {static_cast<uint8_t*>(a2_scales), static_cast<uint8_t*>(a3_scales), nullptr};
  const int qcols[3] = {g1_cols, w[1].n, 0};
  for (int p = 0; p < 3; ++p) {
    mx::ChainProj& P = args.proj[p];
    P.w_scales = static_cast<const uint8_t*>(w[p].w_scales);
    P.a_scales = static_cast<const uint8_t*>(act_scales[p]);
    P.n = w[p].n;
    P.k = w[p].k;
    P.splits = get_plan(h, M, w[p].n, w[p].k).splits;
    P.out = outs[p];
    P.q = qs[p];
    P.q_scales = qscales[p];
    P.q_cols = qcols[p];
  }
  args.plan = mx::plan_chain(M, args.proj, h->chain_clusters);
  if (!args.plan.ok) return MX_ERR_UNSUPPORTED;
  args.cnt_off[0] = 4;
  args.cnt_off[1] = 4 + w[0].n / 128;
  if (args.cnt_off[1] + w[1].n / 128 > mx::kChainCounters) return MX_ERR_UNSUPPORTED;
  args.M = M;
  args.mtile = (M + 15) & ~15;
  args.nsfb = 1;
  args.counters = h->d_chain;
  args.status = h->d_status;
  CUtensorMap maps[6];
  const int act_k[3] = {w[0].k, g1_cols, w[1].n};
  for (int p = 0; p < 3; ++p) {
    int rc = make_tmap(h, &maps[p], w[p].w, w[p].n, w[p].k, 128);
    if (rc != MX_OK) return rc;
    rc = make_tmap(h, &maps[3 + p], acts[p], M, act_k[p], args.mtile);
    if (rc != MX_OK) return rc;
  }
#ifdef MX_TIMELINE
  args.tl = nullptr;
  if (h->d_tl != nullptr && mx::kChainCluster * args.plan.clusters <= mx::kTimelineCtas &&
      h->tl_next < kTimelineLaunches)
    args.tl = h->d_tl + static_cast<size_t>(h->tl_next++) * mx::kTimelineCtas * mx::kTimelineSlots;
#endif
  return cuda_status(mx::launch_chain(maps, args, stream));
}

}  // namespace

extern "C" {

int mx_create(mx_handle** out, int device) {
  if (out == nullptr) return MX_ERR_INVALID_ARG;
  *out = nullptr;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return MX_ERR_CUDA;
  int major = 0, minor = 0, sms = 0, smem_sm = 0, smem_rsv = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, device) != cudaSuccess)
    return MX_ERR_CUDA;
  if (major != 10 || minor != 3) return MX_ERR_DEVICE;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return MX_ERR_CUDA;
  if (cudaSetDevice(device) != cudaSuccess) return MX_ERR_CUDA;
  mx_handle* h = new (std::nothrow) mx_handle();
  int rc = MX_OK;
  if (h == nullptr) {
    rc = MX_ERR_CUDA;
  } else {
    h->device = device;
    h->sm_count = sms;
    h->smem_per_sm = static_cast<size_t>(smem_sm);
    h->smem_reserved = static_cast<size_t>(smem_rsv);
    h->env = mx::read_plan_env();
    const char* pe = getenv("MX_CHAIN_PERSISTENT");
    h->chain_persistent = pe != nullptr && atoi(pe) == 1;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
      rc = MX_ERR_CUDA;
    } else {
      h->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      if (mx::set_gemm_attributes() != cudaSuccess || mx::set_wo_a_attributes() != cudaSuccess ||
          mx::set_chain_attributes() != cudaSuccess ||
          cudaMalloc(&h->d_status, 16) != cudaSuccess ||
          cudaMemset(h->d_status, 0, 16) != cudaSuccess ||
          cudaMalloc(&h->d_chain, mx::kChainCounters * sizeof(unsigned)) != cudaSuccess ||
          cudaMemset(h->d_chain, 0, mx::kChainCounters * sizeof(unsigned)) != cudaSuccess ||
          cudaMalloc(&h->d_woa, kWoaScratchBytes) != cudaSuccess ||
          cudaMalloc(&h->d_ssq, kSsqBytes) != cudaSuccess ||
#ifdef MX_TIMELINE
          cudaMalloc(&h->d_tl, kTimelineBytes) != cudaSuccess ||
          cudaMemset(h->d_tl, 0, kTimelineBytes) != cudaSuccess ||
#endif
          cudaDeviceSynchronize() != cudaSuccess)
        rc = MX_ERR_CUDA;
      // every CTA of the chain kernel must be resident at once: the largest
      // number of its clusters that fit (16 at most are used)
      if (rc == MX_OK) h->chain_clusters = std::min(16, mx::chain_max_clusters());
    }
  }
  if (rc != MX_OK && h != nullptr) {
    if (h->d_status) cudaFree(h->d_status);
    if (h->d_chain) cudaFree(h->d_chain);
    if (h->d_woa) cudaFree(h->d_woa);
    if (h->d_ssq) cudaFree(h->d_ssq);
    delete h;
    h = nullptr;
  }
  cudaSetDevice(prev);
  *out = h;
  return rc;
}

int mx_destroy(mx_handle* h) {
  if (h == nullptr) return MX_ERR_INVALID_ARG;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(h->device);
  cudaFree(h->d_status);
  cudaFree(h->d_chain);
  cudaFree(h->d_woa);
  cudaFree(h->d_ssq);
#ifdef MX_TIMELINE
  cudaFree(h->d_tl);
#endif
  cudaSetDevice(prev);
  delete h;
  return MX_OK;
}

size_t mx_scale_bytes(int rows, int k) {
  if (rows < 0 || k < 0 || k % 32 != 0) return 0;
  const size_t r = (static_cast<size_t>(rows) + 127) / 128 * 128;
  const size_t c = (static_cast<size_t>(k / 32) + 3) / 4 * 4;
  return r * c;
}

int mx_quantize_rows(mx_handle* h, int M, int K, const void* x, long ldx, void* q, void* scales,
                     int swizzled, void* stream) {
  int rc = check_device(h);
  if (rc != MX_OK) return rc;
  if (M < 1 || M > 65536 || K < 32 || K % 32 != 0 || ldx < K || ldx % 8 != 0)
    return MX_ERR_INVALID_ARG;
  if (x == nullptr || q == nullptr || scales == nullptr) return MX_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(q, 16)) return MX_ERR_INVALID_ARG;
  return cuda_status(mx::launch_quantize_rows(x, ldx, M, K, q, scales, swizzled,
                                              static_cast<cudaStream_t>(stream)));
}

int mx_rmsnorm_quantize_rows(mx_handle* h, int M, int K, const void* x, long ldx,
                             const void* norm_weight, float eps, void* y, void* q, void* scales,
                             int swizzled, void* stream) {
  int rc = check_device(h);
  if (rc != MX_OK) return rc;
  if (M < 1 || M > 65536 || K < 32 || K % 32 != 0 || ldx < K || ldx % 8 != 0)
    return MX_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || x == nullptr || norm_weight == nullptr || q == nullptr || scales == nullptr)
    return MX_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(norm_weight, 16) || !aligned(q, 16) || (y && !aligned(y, 16)))
    return MX_ERR_INVALID_ARG;
  return cuda_status(mx::launch_rmsnorm_quantize_rows(x, ldx, M, K, norm_weight, eps, y, q, scales,
                                                      swizzled, static_cast<cudaStream_t>(stream)));
}

int mx_gemm(mx_handle* h, int M, int N, int K, const void* a, const void* a_scales, const void* w,
            const void* w_scales, void* out, unsigned flags, void* stream) {
  int rc = check_device(h);
  if (rc != MX_OK) return rc;
  rc = validate_gemm(h, M, N, K, a, a_scales, w, w_scales);
  if (rc != MX_OK) return rc;
  if (out == nullptr || !aligned(out, 16)) return MX_ERR_INVALID_ARG;
  if (flags & ~MX_FLAG_PDL) return MX_ERR_INVALID_ARG;
  return gemm_launch(h, M, N, K, a, a_scales, w, w_scales, out, nullptr, nullptr, 0,
                     (flags & MX_FLAG_PDL) != 0, static_cast<cudaStream_t>(stream));
}

int mx_gemm_bf16(mx_handle* h, int M, int N, int K, const void* x, long ldx, const void* w,
                 const void* w_scales, void* out, unsigned flags, void* stream) {
  int rc = check_device(h);
  if (rc != MX_OK) return rc;
  if (M < 1 || N < 1 || K < 1 || x == nullptr || w == nullptr || w_scales == nullptr)
    return MX_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(w_scales, 32)) return MX_ERR_INVALID_ARG;
  if (K % 32 != 0 || ldx < K || ldx % 8 != 0) return MX_ERR_INVALID_ARG;
  if (out == nullptr || !aligned(out, 16)) return MX_ERR_INVALID_ARG;
  if (flags & ~MX_FLAG_PDL) return MX_ERR_INVALID_ARG;
  if (M > 256 || N % 128 != 0 || K % 128 != 0) return MX_ERR_UNSUPPORTED;
  if (get_plan(h, M, N, K, true).smem > mx::kMaxDynamicSmem) return MX_ERR_UNSUPPORTED;
  return gemm_launch(h, M, N, K, nullptr, nullptr, w, w_scales, out, nullptr, nullptr, 0,
                     (flags & MX_FLAG_PDL) != 0, static_cast<cudaStream_t>(stream), x, ldx);
}

// ------------------------------------------------------------------ warm-up
namespace {

// One weight per distinct (n, k), in increasing (n, k) order: indices into w.
std::vector<int> shape_representatives(const mx_weight* w, int nw) {
  std::vector<int> reps;
  for (int i = 0; i < nw; ++i) {
    bool seen = false;
    for (int j : reps) seen = seen || (w[j].n == w[i].n && w[j].k == w[i].k);
    if (!seen) reps.push_back(i);
  }
  std::sort(reps.begin(), reps.end(), [&](int a, int b) {
    return w[a].n != w[b].n ? w[a].n < w[b].n : w[a].k < w[b].k;
  });
  return reps;
}

// The zero activation's codes region, its scales region, and the outputs, in bytes.
bool warmup_layout(const mx_weight* w, int nw, const int* rows, int nrows, size_t* codes,
                   size_t* scales, size_t* outs) {
  if (w == nullptr || rows == nullptr || nw < 1 || nrows < 1) return false;
  *codes = *scales = *outs = 0;
  for (int i : shape_representatives(w, nw)) {
    if (w[i].n < 1 || w[i].k < 32 || w[i].k % 32 != 0) return false;
    for (int j = 0; j < nrows; ++j) {
      if (rows[j] < 1) return false;
      *codes = std::max(*codes, static_cast<size_t>(rows[j]) * w[i].k);
      *scales = std::max(*scales, mx_scale_bytes(rows[j], w[i].k));
      *outs += round256(static_cast<size_t>(rows[j]) * w[i].n * 2);
    }
  }
  *codes = round256(*codes);
  *scales = round256(*scales);
  return true;
}

}  // namespace

size_t mx_warmup_bytes(const mx_weight* w, int nw, const int* rows, int nrows) {
  size_t codes, scales, outs;
  return warmup_layout(w, nw, rows, nrows, &codes, &scales, &outs) ? codes + scales + outs : 0;
}

int mx_warmup(mx_handle* h, const mx_weight* w, int nw, const int* rows, int nrows, void* scratch,
              size_t scratch_bytes, void* stream) {
  int rc = check_device(h);
  if (rc != MX_OK) return rc;
  size_t codes, scales, outs;
  if (!warmup_layout(w, nw, rows, nrows, &codes, &scales, &outs)) return MX_ERR_INVALID_ARG;
  if (scratch == nullptr || !aligned(scratch, 256) || scratch_bytes < codes + scales + outs)
    return MX_ERR_INVALID_ARG;
  uint8_t* const base = static_cast<uint8_t*>(scratch);
  const std::vector<int> reps = shape_representatives(w, nw);
  // every launch is validated and prepared (plan, tensor maps) before the first
  std::vector<GemmLaunch> launches(reps.size() * static_cast<size_t>(nrows));
  size_t off = codes + scales;
  for (size_t r = 0; r < reps.size(); ++r) {
    const mx_weight& wr = w[reps[r]];
    for (int j = 0; j < nrows; ++j) {
      rc = validate_gemm(h, rows[j], wr.n, wr.k, base, base + codes, wr.w, wr.w_scales);
      if (rc == MX_OK)
        rc = gemm_prepare(h, &launches[r * nrows + j], rows[j], wr.n, wr.k, base, base + codes, wr.w,
                          wr.w_scales, base + off, nullptr, nullptr, 0);
      if (rc != MX_OK) return rc;
      off += round256(static_cast<size_t>(rows[j]) * wr.n * 2);
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the zero MXFP8 activation: zero codes, zero scale bytes (as the mxfp8 page's `_zeros`)
  rc = cuda_status(cudaMemsetAsync(base, 0, codes + scales, s));
  for (size_t i = 0; i < launches.size() && rc == MX_OK; ++i) rc = gemm_run(h, &launches[i], true, s);
  return rc;
}

int mx_gemm_chain(mx_handle* h, int M, const void* a1, const void* a1_scales, const mx_weight w[3],
                  int g1_cols, void* a2, void* a2_scales, void* a3, void* a3_scales, void* out,
                  void* debug_out1, void* debug_out2, void* stream) {
  int rc = check_device(h);
  if (rc != MX_OK) return rc;
  if (w == nullptr) return MX_ERR_INVALID_ARG;
  rc = validate_gemm(h, M, w[0].n, w[0].k, a1, a1_scales, w[0].w, w[0].w_scales);
  if (rc != MX_OK) return rc;
  rc = validate_gemm(h, M, w[1].n, w[1].k, a2, a2_scales, w[1].w, w[1].w_scales);
  if (rc != MX_OK) return rc;
  rc = validate_gemm(h, M, w[2].n, w[2].k, a3, a3_scales, w[2].w, w[2].w_scales);
  if (rc != MX_OK) return rc;
  if (g1_cols < 128 || g1_cols % 128 != 0 || g1_cols > w[0].n || w[1].k != g1_cols ||
      w[2].k != w[1].n)
    return MX_ERR_INVALID_ARG;
  if (out == nullptr || !aligned(out, 16)) return MX_ERR_INVALID_ARG;
  if ((debug_out1 && !aligned(debug_out1, 16)) || (debug_out2 && !aligned(debug_out2, 16)))
    return MX_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = chain_persistent(h, M, a1, a1_scales, w, g1_cols, a2, a2_scales, a3, a3_scales, out,
                        debug_out1, debug_out2, s);
  if (rc != MX_ERR_UNSUPPORTED) return rc;
  // three launches, every tensor map encoded before the first
  int push[3];
  chain_push(h, M,
             {{w[0].n, w[0].k, false, false, true}, {w[1].n, w[1].k, false, false, true},
              {w[2].n, w[2].k, false, false, true}},
             push);
  GemmLaunch L[3];
  rc = gemm_prepare(h, &L[0], M, w[0].n, w[0].k, a1, a1_scales, w[0].w, w[0].w_scales, debug_out1,
                    static_cast<uint8_t*>(a2), static_cast<uint8_t*>(a2_scales), g1_cols, nullptr, 0, 1,
                    nullptr, push[0]);
  if (rc == MX_OK)
    rc = gemm_prepare(h, &L[1], M, w[1].n, w[1].k, a2, a2_scales, w[1].w, w[1].w_scales, debug_out2,
                      static_cast<uint8_t*>(a3), static_cast<uint8_t*>(a3_scales), w[1].n, nullptr, 0, 1,
                      nullptr, push[1]);
  if (rc == MX_OK)
    rc = gemm_prepare(h, &L[2], M, w[2].n, w[2].k, a3, a3_scales, w[2].w, w[2].w_scales, out, nullptr,
                      nullptr, 0, nullptr, 0, 1, nullptr, push[2]);
  for (int i = 0; i < 3 && rc == MX_OK; ++i) rc = gemm_run(h, &L[i], true, s);
  return rc;
}

int mx_gemm_chain_norm(mx_handle* h, int M, const void* a1, const void* a1_scales,
                       const mx_weight w[3], int g1_cols, const void* norm_weight, float eps,
                       void* out1, void* a2, void* a2_scales, void* a3, void* a3_scales, void* out,
                       void* debug_y, void* debug_out2, void* stream) {
  int rc = check_device(h);
  if (rc != MX_OK) return rc;
  if (w == nullptr || norm_weight == nullptr || out1 == nullptr || !(eps >= 0.f))
    return MX_ERR_INVALID_ARG;
  rc = validate_gemm(h, M, w[0].n, w[0].k, a1, a1_scales, w[0].w, w[0].w_scales);
  if (rc != MX_OK) return rc;
  rc = validate_gemm(h, M, w[1].n, w[1].k, a2, a2_scales, w[1].w, w[1].w_scales);
  if (rc != MX_OK) return rc;
  rc = validate_gemm(h, M, w[2].n, w[2].k, a3, a3_scales, w[2].w, w[2].w_scales);
  if (rc != MX_OK) return rc;
  if (g1_cols < 128 || g1_cols % 128 != 0 || g1_cols > w[0].n || w[1].k != g1_cols ||
      w[2].k != w[1].n)
    return MX_ERR_INVALID_ARG;
  if (out == nullptr || !aligned(out, 16) || !aligned(out1, 16) || !aligned(norm_weight, 16) ||
      (debug_y && !aligned(debug_y, 16)) || (debug_out2 && !aligned(debug_out2, 16)))
    return MX_ERR_INVALID_ARG;
  // Up to kNormFusedMaxRows rows G2 applies the norm in its prologue (three
  // launches); beyond, every one of G2's CTAs would repeat the RMS pass over all
  // rows, and the stand-alone norm kernel between G1 and G2 is faster.
  const bool fused = chain_norm_fused(M, g1_cols, get_plan(h, M, w[1].n, w[1].k, true, true).smem);
  const mx::GemmNorm norm{static_cast<const uint16_t*>(norm_weight), eps, h->d_ssq,
                          static_cast<uint16_t*>(debug_y), static_cast<uint8_t*>(a2),
                          static_cast<uint8_t*>(a2_scales)};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // G1 -> bf16 out1 (qr | kv) and, fused, qr's block sums of squares; G2 reads
  // qr in bf16, normalizes and quantizes it in its prologue (writing a2 on the
  // way) or reads a2 written by the norm kernel, and requantizes into a3; G3.
  // Every tensor map is encoded before the first launch.
  // (four launches: the norm kernel sits between G1 and G2, so G1 and G2
  // are not neighbours; the check then takes G2 after G1 all the same). G3
  // keeps its planned ring depth here: the split table's shallower ring for G3
  // is measured after the plain G2 and is slower after the fused-norm one.
  int push[3];
  chain_push(h, M,
             {{w[0].n, w[0].k, false, false, true}, {w[1].n, w[1].k, fused, fused, true},
              {w[2].n, w[2].k, false, false, false}},
             push);
  GemmLaunch L[3];
  rc = gemm_prepare(h, &L[0], M, w[0].n, w[0].k, a1, a1_scales, w[0].w, w[0].w_scales, out1, nullptr,
                    nullptr, 0, nullptr, 0, 1, nullptr, push[0]);
  if (fused) {
    L[0].args.ssq_out = h->d_ssq;
    L[0].args.ssq_cols = g1_cols;
  }
  if (rc == MX_OK && fused)
    rc = gemm_prepare(h, &L[1], M, w[1].n, w[1].k, nullptr, nullptr, w[1].w, w[1].w_scales,
                      debug_out2, static_cast<uint8_t*>(a3), static_cast<uint8_t*>(a3_scales), w[1].n,
                      out1, w[0].n, 1, &norm, push[1]);
  else if (rc == MX_OK)
    rc = gemm_prepare(h, &L[1], M, w[1].n, w[1].k, a2, a2_scales, w[1].w, w[1].w_scales, debug_out2,
                      static_cast<uint8_t*>(a3), static_cast<uint8_t*>(a3_scales), w[1].n, nullptr, 0, 1,
                      nullptr, push[1]);
  if (rc == MX_OK)
    rc = gemm_prepare(h, &L[2], M, w[2].n, w[2].k, a3, a3_scales, w[2].w, w[2].w_scales, out, nullptr,
                      nullptr, 0, nullptr, 0, 1, nullptr, push[2], false);
  if (rc != MX_OK) return rc;
  rc = gemm_run(h, &L[0], true, s);
  if (rc != MX_OK) return rc;
  if (!fused) {
    rc = cuda_status(mx::launch_rmsnorm_quantize_rows(out1, w[0].n, M, g1_cols, norm_weight, eps,
                                                      debug_y, a2, a2_scales, 1, s));
    if (rc != MX_OK) return rc;
  }
  rc = gemm_run(h, &L[1], true, s);
  if (rc != MX_OK) return rc;
  return gemm_run(h, &L[2], true, s);
}

namespace {

// WO-A as two launches (inverse RoPE + MX quantization into xq, then one grouped
// GEMM with the requantization in its epilogue). The arguments are validated by
// the caller; returns MX_ERR_UNSUPPORTED before any launch when the GEMM has no
// plan for the shape.
int woa_two_launch(mx_handle* h, int T, const void* x, long ldx, const int64_t* positions,
                   const float* cos_sin, int max_pos, const void* w, const void* w_scales, int G,
                   int H, int d_nope, int d_rope, int R, void* xq, void* xq_scales, void* z,
                   void* q, void* q_scales, cudaStream_t s) {
  const int D = d_nope + d_rope;
  const long kx = static_cast<long>(G) * H * D;  // the activation's K (all groups)
  if (kx > (1L << 30) || get_plan(h, T, G * R, H * D).smem > mx::kMaxDynamicSmem)
    return MX_ERR_UNSUPPORTED;
  // 1. inverse RoPE + MX quantize of all heads -> xq (swizzled scales over G*H*D)
  const mx::RopeArgs rope{positions, cos_sin, max_pos, D, d_nope, h->d_status};
  int rc = cuda_status(mx::launch_quantize_rows(x, ldx, T, static_cast<int>(kx), xq, xq_scales, 1, s, rope));
  if (rc != MX_OK) return rc;
  // 2. one grouped GEMM: tile rows of group g contract xq's K-slice g; z rounded
  //    to bf16 and requantized in the epilogue
  return gemm_launch(h, T, G * R, H * D, xq, xq_scales, w, w_scales, z, static_cast<uint8_t*>(q),
                     static_cast<uint8_t*>(q_scales), G * R, true, s, nullptr, 0, G);
}

}  // namespace

int wo_a_grouped(mx_handle* h, int T, const void* x, long ldx, const int64_t* positions,
                 const float* cos_sin, int max_pos, const void* w, const void* w_scales, int G,
                 int H, int d_nope, int d_rope, int R, void* q, void* q_scales, void* debug_z,
                 void* debug_xq, void* debug_xs, int early_trigger, void* stream) {
  int rc = check_device(h);
  if (rc != MX_OK) return rc;
  if (x == nullptr || positions == nullptr || cos_sin == nullptr || w == nullptr ||
      w_scales == nullptr || q == nullptr || q_scales == nullptr)
    return MX_ERR_INVALID_ARG;
  if (T < 1 || G < 1 || H < 1 || R < 1 || max_pos < 1) return MX_ERR_INVALID_ARG;
  if (d_nope != 448 || d_rope != 64 || H > 8 || R % 128 != 0 || T > 128) return MX_ERR_UNSUPPORTED;
  const int D = d_nope + d_rope;
  if (ldx < static_cast<long>(G) * H * D || ldx % 8 != 0) return MX_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(w_scales, 32) || !aligned(q, 16) ||
      !aligned(q_scales, 16) || !aligned(cos_sin, 16) || !aligned(positions, 8))
    return MX_ERR_INVALID_ARG;
  if ((debug_z && !aligned(debug_z, 16)) || (debug_xq && !aligned(debug_xq, 16)))
    return MX_ERR_INVALID_ARG;
  // Above kWoaFusedMaxTokens the two launches are faster: every CTA of the fused
  // kernel quantizes its group's whole activation slice, which then outweighs
  // the weight stream. They need the handle's scratch for the activation, so
  // the fused kernel serves calls that ask for its debug copy of it.
  const long kx = static_cast<long>(G) * H * D;
  const size_t codes = (static_cast<size_t>(T) * kx + 255) & ~size_t{255};
  if (T > kWoaFusedMaxTokens && debug_xq == nullptr && debug_xs == nullptr && kx <= (1L << 24) &&
      codes + mx_scale_bytes(T, static_cast<int>(kx)) <= kWoaScratchBytes) {
    rc = woa_two_launch(h, T, x, ldx, positions, cos_sin, max_pos, w, w_scales, G, H, d_nope, d_rope,
                        R, h->d_woa, h->d_woa + codes, debug_z, q, q_scales,
                        static_cast<cudaStream_t>(stream));
    if (rc != MX_ERR_UNSUPPORTED) return rc;
  }
  const mx::WoaPlan plan = mx::plan_wo_a(T, G, H, R, h->sm_count, h->env);
  CUtensorMap tm_w;
  rc = make_tmap(h, &tm_w, w, G * R, H * D, 128);
  if (rc != MX_OK) return rc;
  mx::WoaArgs args = {};
  args.T = T;
  args.G = G;
  args.H = H;
  args.R = R;
  args.D = D;
  args.mtile = plan.mtile;
  args.stages = plan.stages;
  args.tmem_cols = plan.tmem_cols;
  args.x = static_cast<const uint16_t*>(x);
  args.ldx = ldx;
  args.positions = positions;
  args.cos_sin = cos_sin;
  args.max_pos = max_pos;
  args.w_scales = static_cast<const uint8_t*>(w_scales);
  args.q = static_cast<uint8_t*>(q);
  args.q_scales = static_cast<uint8_t*>(q_scales);
  args.debug_z = static_cast<uint16_t*>(debug_z);
  args.debug_xq = static_cast<uint8_t*>(debug_xq);
  args.debug_xs = static_cast<uint8_t*>(debug_xs);
  args.early_trigger = early_trigger;
  args.status = h->d_status;
#ifdef MX_TIMELINE
  args.tl = nullptr;
  if (h->d_tl != nullptr && G * (R / 128) * plan.splits <= mx::kTimelineCtas && h->tl_next < kTimelineLaunches)
    args.tl = h->d_tl + static_cast<size_t>(h->tl_next++) * mx::kTimelineCtas * mx::kTimelineSlots;
#endif
  return cuda_status(mx::launch_wo_a(tm_w, args, plan, static_cast<cudaStream_t>(stream)));
}

int wo_a_grouped_unfused(mx_handle* h, int T, const void* x, long ldx, const int64_t* positions,
                         const float* cos_sin, int max_pos, const void* w, const void* w_scales,
                         int G, int H, int d_nope, int d_rope, int R, void* xq, void* xq_scales,
                         void* z, void* q, void* q_scales, void* stream) {
  int rc = check_device(h);
  if (rc != MX_OK) return rc;
  if (x == nullptr || positions == nullptr || cos_sin == nullptr || w == nullptr ||
      w_scales == nullptr || xq == nullptr || xq_scales == nullptr || q == nullptr ||
      q_scales == nullptr)
    return MX_ERR_INVALID_ARG;
  if (T < 1 || G < 1 || H < 1 || R < 1 || max_pos < 1) return MX_ERR_INVALID_ARG;
  if (d_nope != 448 || d_rope != 64 || R % 128 != 0 || T > 256) return MX_ERR_UNSUPPORTED;
  const int D = d_nope + d_rope;
  const long kx = static_cast<long>(G) * H * D;  // the activation's K (all groups)
  if (ldx < kx || ldx % 8 != 0) return MX_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(w_scales, 32) || !aligned(xq, 16) ||
      !aligned(xq_scales, 16) || !aligned(q, 16) || !aligned(q_scales, 16) ||
      !aligned(cos_sin, 16) || !aligned(positions, 8) || (z && !aligned(z, 16)))
    return MX_ERR_INVALID_ARG;
  return woa_two_launch(h, T, x, ldx, positions, cos_sin, max_pos, w, w_scales, G, H, d_nope, d_rope,
                        R, xq, xq_scales, z, q, q_scales, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------ chain without allocation
// mx_gemm_chain_noalloc keeps the chain's two MXFP8 intermediates (codes and
// swizzled scales of the second and third projections' inputs) in this fixed
// device array instead of caller buffers. Every GPU that loads the library
// holds it until the process exits. Host code may not use the array's name as
// a device address (on the host it names a stand-in): the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
constexpr size_t kChainScratchBytes = size_t{1} << 20;
static __device__ __align__(256) uint8_t g_chain_scratch[kChainScratchBytes];

namespace {

constexpr int kScratchDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_address[kScratchDevices] = {};

// Device address of g_chain_scratch on `device` (the current device), looked up
// on the first call for that device.
int chain_scratch(int device, uint8_t** out) {
  if (device < 0 || device >= kScratchDevices) return MX_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_address[device] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_chain_scratch) != cudaSuccess || p == nullptr) return MX_ERR_CUDA;
    g_scratch_address[device] = p;
  }
  *out = static_cast<uint8_t*>(g_scratch_address[device]);
  return MX_OK;
}

}  // namespace

int mx_gemm_chain_noalloc(mx_handle* h, int M, const void* a1, const void* a1_scales,
                          const mx_weight w[3], int g1_cols, void* out, void* stream) {
  int rc = check_device(h);
  if (rc != MX_OK) return rc;
  if (w == nullptr || M < 1 || g1_cols < 1 || w[1].n < 1) return MX_ERR_INVALID_ARG;
  // a2 [M, g1_cols] + its scales, a3 [M, w[1].n] + its scales, each 256-byte aligned
  const size_t a2 = round256(static_cast<size_t>(M) * static_cast<size_t>(g1_cols));
  const size_t s2 = round256(mx_scale_bytes(M, g1_cols));
  const size_t a3 = round256(static_cast<size_t>(M) * static_cast<size_t>(w[1].n));
  const size_t s3 = round256(mx_scale_bytes(M, w[1].n));
  if (a2 + s2 + a3 + s3 > kChainScratchBytes) return MX_ERR_UNSUPPORTED;
  uint8_t* p = nullptr;
  rc = chain_scratch(h->device, &p);
  if (rc != MX_OK) return rc;
  return mx_gemm_chain(h, M, a1, a1_scales, w, g1_cols, p, p + a2, p + a2 + s2, p + a2 + s2 + a3,
                       out, nullptr, nullptr, stream);
}

static_assert(MX_REDUCE_ITEMS == mx::kReduceItems && MX_REDUCE_ROWS == mx::kReduceRows &&
                  MX_REDUCE_PUSH == mx::kReducePush && MX_REDUCE_PUSH_COMPACT == mx::kReducePushCompact,
              "mx.h reduction codes");
static_assert(MX_PUSH_NONE == mx::kPushNone && MX_PUSH_COMPACT == mx::kPushCompact && MX_PUSH_FULL == mx::kPushFull,
              "mx.h push codes");

int mx_plan_gemm(int M, int N, int K, int sm_count, int fused, int norm, int push, mx_plan_info* out) {
  if (out == nullptr || M < 1 || M > 256 || N < 128 || N % 128 != 0 || K < 128 || K % 128 != 0 ||
      sm_count < 1 || push < MX_PUSH_NONE || push > MX_PUSH_FULL || (norm && !fused))
    return MX_ERR_INVALID_ARG;
  const mx::GemmPlan pl = mx::plan_gemm(M, N, K, sm_count, mx::read_plan_env(), fused != 0, norm != 0, push);
  *out = mx_plan_info{pl.splits, pl.stages, pl.mtile, pl.tmem_cols, pl.reduction, pl.smem};
  return MX_OK;
}

int mx_plan_chain_push(int M, const mx_weight w[3], int norm, int sm_count, size_t smem_per_sm,
                       size_t smem_reserved, int modes[3]) {
  if (w == nullptr || modes == nullptr || M < 1 || M > 256 || sm_count < 1) return MX_ERR_INVALID_ARG;
  for (int i = 0; i < 3; ++i)
    if (w[i].n < 128 || w[i].n % 128 != 0 || w[i].k < 128 || w[i].k % 128 != 0) return MX_ERR_INVALID_ARG;
  if (w[1].k > w[0].n || w[2].k != w[1].n) return MX_ERR_INVALID_ARG;
  const mx::PlanEnv env = mx::read_plan_env();
  const bool fused =
      norm != 0 && chain_norm_fused(M, w[1].k, mx::plan_gemm(M, w[1].n, w[1].k, sm_count, env, true, true).smem);
  const ChainShape c[3] = {{w[0].n, w[0].k, false, false, true},
                           {w[1].n, w[1].k, fused, fused, true},
                           {w[2].n, w[2].k, false, false, norm == 0}};
  int m[3];
  chain_push_modes(
      c, sm_count, smem_per_sm, smem_reserved,
      [&](int i, int pm) {
        return mx::plan_gemm(M, c[i].N, c[i].K, sm_count, env, c[i].fused, c[i].norm, pm, c[i].table_depth);
      },
      m);
  for (int i = 0; i < 3; ++i) modes[i] = m[i];
  return MX_OK;
}

int mx_device_status(mx_handle* h, int* status) {
  int rc = check_device(h);
  if (rc != MX_OK) return rc;
  if (status == nullptr) return MX_ERR_INVALID_ARG;
  int v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return MX_ERR_CUDA;
  if (cudaMemcpy(&v, h->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MX_ERR_CUDA;
  if (cudaMemset(h->d_status, 0, sizeof(int)) != cudaSuccess) return MX_ERR_CUDA;
  // a failed chain call leaves its counters inconsistent: start them afresh
  if (v != 0 && cudaMemset(h->d_chain, 0, mx::kChainCounters * sizeof(unsigned)) != cudaSuccess)
    return MX_ERR_CUDA;
  *status = (v & 1) ? MX_ERR_TIMEOUT : (v & 2) ? MX_ERR_INVALID_ARG : MX_OK;
  return MX_OK;
}

int mx_wait_selftest(mx_handle* h, void* stream) {
  int rc = check_device(h);
  if (rc != MX_OK) return rc;
  return cuda_status(mx::launch_wait_selftest(h->d_status, static_cast<cudaStream_t>(stream)));
}

#ifdef MX_TIMELINE
// Timeline build only (not declared in mx.h): the stamps of the GEMM launches
// made since the last reset, launch after launch, kTimelineCtas x
// kTimelineSlots each. Copies min(bytes, recorded) to host memory and returns
// the number of launches recorded; reset clears the record.
int mx_timeline_read(mx_handle* h, void* host, size_t bytes, int* launches) {
  if (h == nullptr || host == nullptr || launches == nullptr) return MX_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MX_ERR_CUDA;
  const size_t per = sizeof(unsigned long long) * mx::kTimelineCtas * mx::kTimelineSlots;
  const size_t n = std::min(bytes, per * static_cast<size_t>(h->tl_next));
  if (cudaMemcpy(host, h->d_tl, n, cudaMemcpyDeviceToHost) != cudaSuccess) return MX_ERR_CUDA;
  *launches = h->tl_next;
  return MX_OK;
}
int mx_timeline_reset(mx_handle* h) {
  if (h == nullptr) return MX_ERR_INVALID_ARG;
  h->tl_next = 0;
  return cudaMemset(h->d_tl, 0, kTimelineBytes) == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}
#endif

const char* mx_status_string(int s) {
  switch (s) {
    case MX_OK: return "MX_OK";
    case MX_ERR_INVALID_ARG: return "MX_ERR_INVALID_ARG";
    case MX_ERR_UNSUPPORTED: return "MX_ERR_UNSUPPORTED";
    case MX_ERR_DEVICE: return "MX_ERR_DEVICE";
    case MX_ERR_CUDA: return "MX_ERR_CUDA";
    case MX_ERR_TIMEOUT: return "MX_ERR_TIMEOUT";
    default: return "MX_ERR_UNKNOWN";
  }
}

}  // extern "C"
