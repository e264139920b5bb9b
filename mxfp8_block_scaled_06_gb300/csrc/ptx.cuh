// ptx.cuh - thin inline-PTX wrappers for sm_103a: mbarrier, TMA (tensor and
// bulk), griddepcontrol, tcgen05 (alloc, mma block-scaled, cp, ld, commit),
// cluster shared memory. Every wait here is bounded (see mbar_wait).
#pragma once
#include <cstdint>
#include <cuda.h>

namespace mx {

// Bits of the device status word (mx_device_status maps them to MX_ERR_*).
constexpr int kStatusTimeout = 1;   // a bounded wait expired
constexpr int kStatusBadInput = 2;  // device-side data out of range (e.g. a position)
// Upper bound of any single wait on an mbarrier, in nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
// Bound of a wait for data a peer CTA sends at the end of its own pipeline: a
// peer reaches its send even after its own bounded waits expired (a few of
// them at most), so this bound outlasts any peer's way there.
constexpr uint64_t kPeerWaitLimitNs = 8 * kWaitLimitNs;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// Non-blocking: whether the phase with this parity has completed.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase of the given parity to complete; false after limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && globaltimer() - t0 > limit_ns) return false;
  }
}

// ----------------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
// 2-D tiled load of box {x.., y..} at element coordinates (x, y) into smem.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int x, int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
// Untiled bulk copy global -> shared; bytes % 16 == 0, both addresses 16-byte aligned.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------- programmatic dependent launch
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// -------------------------------------------------------------- async proxy
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Orders this thread's earlier generic-proxy accesses of global memory (e.g. an
// acquire of data another CTA wrote) before its later async-proxy ones (TMA).
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ------------------------------------------------------ global synchronization
__device__ __forceinline__ uint32_t ld_acquire_gpu(const unsigned* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Barrier among `threads` threads (whole warps) of the CTA on hardware barrier `id`.
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ------------------------------------------------------------------ cluster
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// Cluster barrier without memory ordering: for ordering execution only (e.g.
// no CTA exits before its peers have finished reading its shared memory). A
// release barrier would also wait for this thread's global stores to complete.
__device__ __forceinline__ void cluster_sync_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}
// The two halves of a cluster barrier, for a phase whose arrival and wait are
// far apart (arrive at set-up, wait just before the first access to a peer).
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Bulk copy from this CTA's shared memory into a peer's (dst and the peer's
// mbarrier from mapa), counted on that barrier (complete_tx); 16-byte aligned,
// bytes % 16 == 0. Committed to this thread's bulk async-group.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst, uint32_t src, uint32_t bytes,
                                                  uint32_t remote_bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "r"(src), "r"(bytes), "r"(remote_bar)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the source reads of this thread's committed bulk copies are done.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// 4-byte store into a peer CTA's shared memory (address from mapa), counted on
// the peer's mbarrier (its address from mapa) as 4 bytes of complete_tx: the
// peer sees the value once it observes that barrier's phase complete.
__device__ __forceinline__ void st_async_b32(uint32_t addr, uint32_t v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr),
               "r"(v), "r"(remote_bar)
               : "memory");
}
__device__ __forceinline__ void st_async_v2(uint32_t addr, float a, float b, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(
                   addr),
               "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(remote_bar)
               : "memory");
}
// 16 bytes (addr 16-byte aligned), as st_async_b32
__device__ __forceinline__ void st_async_v4(uint32_t addr, float a, float b, float c, float d,
                                            uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(__float_as_uint(c)),
               "r"(__float_as_uint(d)), "r"(remote_bar)
               : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Load from a peer CTA's shared memory. Volatile keeps it after the cluster
// barrier (volatile asm is never reordered against other volatile asm); no
// memory clobber, so consecutive loads are issued back to back.
__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
// 16 bytes from a peer CTA's shared memory (16-byte aligned), as above.
__device__ __forceinline__ float4 ld_shared_cluster_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}
// Sum of the float at shared offset `addr` over cluster ranks 0..S-1 (S <= 16),
// in rank order; the loads of each group of 8 ranks are issued before their adds.
__device__ __forceinline__ float cluster_sum(uint32_t addr, int S) {
  float acc = 0.f;
  for (int r0 = 0; r0 < S; r0 += 8) {
    float v[8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
      v[r] = r0 + r < S ? ld_shared_cluster_f32(map_shared_rank(addr, r0 + r)) : 0.f;
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r0 + r < S) acc += v[r];
  }
  return acc;
}

// cluster_sum for kSumBatch addresses at once: every (address, rank) load of a
// group of 8 ranks is issued before any add, so the items' latencies overlap;
// each sum is still taken in rank order (the same result as cluster_sum).
// Addresses with use[b] == false are not read and sum to 0.
constexpr int kSumBatch = 4;
__device__ __forceinline__ void cluster_sum_batch(const uint32_t (&addr)[kSumBatch],
                                                  const bool (&use)[kSumBatch], int S,
                                                  float (&sum)[kSumBatch]) {
#pragma unroll
  for (int b = 0; b < kSumBatch; ++b) sum[b] = 0.f;
  for (int r0 = 0; r0 < S; r0 += 8) {
    float v[kSumBatch][8];
#pragma unroll
    for (int b = 0; b < kSumBatch; ++b)
#pragma unroll
      for (int r = 0; r < 8; ++r)
        v[b][r] = use[b] && r0 + r < S ? ld_shared_cluster_f32(map_shared_rank(addr[b], r0 + r)) : 0.f;
#pragma unroll
    for (int b = 0; b < kSumBatch; ++b)
#pragma unroll
      for (int r = 0; r < 8; ++r)
        if (r0 + r < S) sum[b] += v[b][r];
  }
}

// ------------------------------------------------------------------ warp
// True in exactly one active lane of a converged warp (elect.sync); code around
// it stays warp-uniform, so its values can live in uniform registers.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b32 r;\n\t"
      "elect.sync r|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// ------------------------------------------------------------------ tcgen05
// Warp-wide: allocate ncols (power of two >= 32) TMEM columns, address -> smem.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive on an mbarrier once every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle
// layout written by a SWIZZLE_128B TMA box of 128-byte rows: 8-row atoms of
// 1024 bytes (stride-dimension offset 1024), leading offset unused.
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;            // leading byte offset (unused) = 16 B
  d |= static_cast<uint64_t>(1024 >> 4) << 32;    // stride byte offset = 1024 B
  d |= static_cast<uint64_t>(1) << 46;            // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;            // 128-byte swizzle
  return d;
}
// Descriptor of a 32-row x 16-byte scale-factor tile (512 contiguous bytes,
// rows 16 bytes apart) for tcgen05.cp .32x128b: no swizzle, 8-row core
// matrices 128 bytes apart, one 16-byte column.
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}
// Instruction descriptor of tcgen05.mma .kind::mxf8f6f4 .block_scale: E4M3 x
// E4M3, both K-major, UE8M0 scales, M = 128, N = n, scale byte `sf_id` of the
// 32-bit scale word for both operands, dense K = 32.
__device__ __forceinline__ uint32_t idesc_mxf8(uint32_t n, uint32_t sf_id) {
  return (sf_id << 4) | (0u << 7) | (0u << 10) | ((n >> 3) << 17) | (1u << 23) |
         ((128u >> 4) << 24) | (sf_id << 29);
}
// D[tmem] (+)= A[smem] x B[smem]^T with per-32 scales from TMEM.
// Each shared-memory descriptor is passed as its two 32-bit halves: a loop that
// walks a ring only changes the low half (the address field), so it advances
// descriptors with 32-bit adds and keeps the high halves in registers.
__device__ __forceinline__ void mma_mxf8_lh(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi,
                                            uint32_t b_lo, uint32_t b_hi, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "mov.b64 da, {%1, %2};\n\tmov.b64 db, {%3, %4};\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], da, db, %6, [%7], "
      "[%8], p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(accumulate), "r"(idesc), "r"(sfa_tmem),
      "r"(sfb_tmem)
      : "memory");
}
// Copy a 32x128-bit smem tile into TMEM lanes 0-31, replicated into all four
// 32-lane quarters (4 columns); the descriptor as its two 32-bit halves.
__device__ __forceinline__ void tmem_cp_32x128b_x4_lh(uint32_t taddr, uint32_t lo, uint32_t hi) {
  asm volatile("{\n\t.reg .b64 d;\n\tmov.b64 d, {%1, %2};\n\t"
               "tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], d;\n\t}" ::"r"(taddr),
               "r"(lo), "r"(hi)
               : "memory");
}
// Each thread of the warp reads 16 consecutive 32-bit columns of its TMEM lane,
// without waiting (tmem_ld_wait makes the registers valid).
__device__ __forceinline__ void tmem_ld_32x32b_x16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Each thread of the warp reads 16 consecutive 32-bit columns of its TMEM lane.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- MX rules
// Scale byte of a 32-block from its float amax: e = floor(log2 amax) - 8
// clamped below at -127, stored as e + 127; amax's exponent field gives
// floor(log2) exactly (every subnormal amax clamps).
__device__ __forceinline__ uint32_t mx_scale_byte(float amax) {
  const int ebits = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
  return static_cast<uint32_t>(max(ebits - 8, 0));
}
// 2^-e as a float for scale byte s (< 255): biased exponent 254 - s.
__device__ __forceinline__ float mx_inv_scale(uint32_t s) {
  return __uint_as_float((254u - s) << 23);
}
// Two floats -> two E4M3 bytes (lo in bits 0-7), nearest-even, saturating.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}
// Byte offset of scale (r, c) in the 128x4 swizzled layout with cpad4 = ceil4(K/32).
__device__ __forceinline__ uint32_t swz_offset(uint32_t r, uint32_t c, uint32_t cpad4) {
  return ((r >> 7) * (cpad4 >> 2) + (c >> 2)) * 512u + (r & 31u) * 16u + ((r & 127u) >> 5) * 4u +
         (c & 3u);
}

}  // namespace mx
