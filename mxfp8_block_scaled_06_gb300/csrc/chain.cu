// chain.cu - the three projections of a decode step's attention in one
// persistent kernel (sm_103a): fused_wqa_wkv (G1) -> wq_b (G2) -> wo_b (G3),
// each product rounded to bf16 and requantized to MXFP8 for the next, exactly
// as mx_gemm_chain defines them.
//
// Why one kernel: as three launches, every projection pays in series the
// programmatic-launch release after the previous grid has exited, the
// activation fetch, its split-K reduction and its exit, and the weight stream
// pauses between projections. Here every CTA streams its weights for all
// three projections through one ring without pause; only the MMAs wait for
// their activation, and then only for the 128-column tiles of the previous
// projection they read, not for the whole projection.
//
// Grid: Q clusters of 8 CTAs, one per SM, all resident at once (Q comes from
// the occupancy query, so every cross-cluster wait can be met). Projection p
// splits each weight tile's K-range over S_p ranks - the split mx_gemm's plan
// uses for that shape, with the same per-CTA chunk order and the same
// rank-order sum, so the results equal the composed entry points bit for bit.
// A cluster holds 8 / S_p tiles at a time and takes the batches c, c + Q, ...
// Warps:
//  0    weight producer: TMA boxes (128 rows x 128 K-bytes) and their scale
//       tiles for every unit of the CTA, in order, into a ring of slots; it
//       never waits for the previous kernel or for an activation;
//  1    activation loader and MMA issuer: per projection it waits until the
//       producing tiles' counters show this call's S_{p-1} publications
//       (acquire), TMA-loads the activation chunks of its K-range, copies the
//       scales to TMEM and issues tcgen05.mma per chunk into one of two
//       accumulators (alternating per unit, so the epilogue of one unit
//       overlaps the MMAs of the next);
//  2-5  epilogue (TMEM lane quarters): the split-K reduction - row m of a tile
//       is owned by group rank m % S; each warp stages its 32-column block of
//       every row by owner and sends each peer its rows with one bulk copy,
//       counted on that peer's barrier - then bf16, stores, the MX
//       requantization, and a release increment of the tile's counter.
// Every wait is bounded (a wait for a peer CTA or another cluster longer than
// any peer's own bounded path); a failure sets the status word and a
// workspace abort flag that the other CTAs' polls see, every CTA still sends
// what its peers wait for, drains its copies and frees TMEM.
#include <cuda_bf16.h>

#include <algorithm>

#include "kernels.h"
#include "ptx.cuh"

namespace mx {
namespace {

constexpr int kThreads = 192;

// Timeline build (-DMX_TIMELINE): %globaltimer stamps per CTA in a.tl[cta *
// kTimelineSlots + slot]: 0 entry, 1 second projection's MMAs issued, 2 last
// weight chunk issued, 3 grid-dependency wait returned, 4 first activation
// landed, 5 first projection's MMAs issued, 6 first unit's accumulator read,
// 7 first projection published, 8 second projection's tiles ready, 9 its
// activation landed, 10 second projection published, 11 third projection's
// tiles ready, 12 its activation landed, 13 second unit's accumulator read,
// 14 last unit stored, 15 exit.
#ifdef MX_TIMELINE
#define CH_TL(slot)                                                                   \
  do {                                                                                \
    if (a.tl != nullptr) a.tl[blockIdx.x * kTimelineSlots + (slot)] = globaltimer(); \
  } while (0)
#else
#define CH_TL(slot) \
  do {              \
  } while (0)
#endif
constexpr uint32_t kWBox = 128 * 128;    // one weight box
constexpr uint32_t kSfTile = 512;        // one 128x4 scale tile
constexpr uint32_t kSlot = kWBox + 1024; // weight box + its scale tile; slots 1024-aligned
constexpr int kMaxRows = 16;             // rows of the persistent path (one 16-column MMA N)

struct ChainMaps {
  CUtensorMap w[3];  // weights [n, k]
  CUtensorMap a[3];  // activations [M, k]: a1, then the requantized G1 and G2 outputs
};

// One work unit: weight tile `tile` of projection p, chunks [k0, k0 + nk) of its
// K-range, split index s of S; idx = its position among the CTA's units of p.
struct Unit {
  int p, tile, k0, nk, s, S, idx;
};

__device__ int build_units(const ChainArgs& a, int cluster, int rank, Unit* u) {
  int nu = 0;
  for (int p = 0; p < 3; ++p) {
    const ChainProj& P = a.proj[p];
    const int S = P.splits, g = kChainCluster / S;
    const int tiles = P.n / 128, chunks = P.k / 128;
    const int s = rank % S, tib = rank / S;
    if (tib >= g) continue;  // this rank has no place in a tile group of p
    const int k0 = s * chunks / S, k1 = (s + 1) * chunks / S;
    int idx = 0;
    for (int b = cluster; b * g < tiles; b += a.plan.clusters) {
      const int t = b * g + tib;
      if (t < tiles && nu < kChainMaxUnits) u[nu++] = Unit{p, t, k0, k1 - k0, s, S, idx++};
    }
  }
  return nu;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    chain_kernel(const __grid_constant__ ChainMaps maps, const __grid_constant__ ChainArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* const bp = smem_raw + (base - raw_addr);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cluster = blockIdx.x / kChainCluster;
  const int rank = blockIdx.x % kChainCluster;
  const ChainPlan& pl = a.plan;
  const int R = pl.ring;
  const int M = a.M;
  const int mtile = a.mtile;
  const int nsfb = a.nsfb;
  const uint32_t a_bytes = static_cast<uint32_t>(mtile) * 128u;

  Unit units[kChainMaxUnits];
  const int nu = build_units(a, cluster, rank, units);
  // receive barrier of unit (p, idx): red_first[p] + idx
  const int red_first[3] = {0, pl.max_units[0], pl.max_units[0] + pl.max_units[1]};

  const uint32_t bars = base + pl.off_bars;
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (R + s); };
  auto act_bar = [&](int p) { return bars + 8u * (2 * R + p); };
  auto acc_full = [&](int b) { return bars + 8u * (2 * R + 3 + b); };
  auto acc_empty = [&](int b) { return bars + 8u * (2 * R + 5 + b); };
  auto red_bar = [&](int i) { return bars + 8u * (2 * R + 7 + i); };
  uint32_t* const words = reinterpret_cast<uint32_t*>(bp + pl.off_bars + 8 * (2 * R + 7 + kChainMaxUnits));
  // words: [0] TMEM address, [1] abort, [2] chunks issued, [3] chunks consumed,
  // [4] activation loads open, [5] this CTA ends the call
  uint32_t* const tmem_slot = words;                        // TMEM base address
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(words + 1);
  volatile int* const issued_w = reinterpret_cast<volatile int*>(words + 2);    // warp 0's chunks issued
  volatile int* const consumed_w = reinterpret_cast<volatile int*>(words + 3);  // warp 1's chunks waited
  volatile int* const act_open = reinterpret_cast<volatile int*>(words + 4);    // act loads issued, not landed

  if (threadIdx.x == 0) CH_TL(0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < R; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int p = 0; p < 3; ++p) mbar_init(act_bar(p), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), 4);
    }
    for (int i = 0; i < kChainMaxUnits; ++i) mbar_init(red_bar(i), 1);
    // the peers' partials of each unit's owned rows may land any time from now on
    for (int u = 0; u < nu; ++u) {
      const Unit& U = units[u];
      const int own = U.S > 1 && U.s < M ? (M - U.s + U.S - 1) / U.S : 0;
      if (own > 0) mbar_expect_tx(red_bar(red_first[U.p] + U.idx), static_cast<uint32_t>(own * (U.S - 1)) * 512u);
    }
    *abort_flag = 0;
    *issued_w = 0;
    *consumed_w = 0;
    *act_open = 0;
    fence_mbar_init();
    for (int p = 0; p < 3; ++p) {
      prefetch_tmap(&maps.w[p]);
      prefetch_tmap(&maps.a[p]);
    }
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), pl.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Once this phase completes every CTA of the cluster has initialized its
  // barriers; each warp waits for it before its first access to a peer (or
  // before it would block anyway).
  cluster_arrive_release();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: two accumulators [0, 2 mtile), four weight-scale columns per
  // ring slot, 4 nsfb activation-scale columns per activation chunk
  const uint32_t sfa_col = 2u * mtile;
  const uint32_t sfb_col0 = sfa_col + 4u * R;
  pdl_launch_dependents();

  auto fail = [&]() {
    atomicOr(a.status, kStatusTimeout);
    *abort_flag = 1;
    atomicExch(a.counters + 2, 1u);
  };
  auto aborted = [&]() { return *abort_flag != 0; };

  if (warp == 0) {
    // ---------------- weight producer: every chunk of every unit, in order
    const uint64_t pol_w = policy_evict_first();
    int g = 0;
    bool paired = false, stop = false;
    for (int u = 0; u < nu && !stop; ++u) {
      const Unit& U = units[u];
      const ChainProj& P = a.proj[U.p];
      const int chunks = P.k / 128;
      for (int k = 0; k < U.nk; ++k, ++g) {
        const int slot = g % R;
        if (g >= R) {
          if (!paired) {
            cluster_wait_acquire();
            paired = true;
          }
          // the slot's previous chunk (g - R) has been consumed by the MMAs
          const uint32_t ph = static_cast<uint32_t>(((g / R) - 1) & 1);
          bool freed = mbar_try_wait(empty(slot), ph);
          if (!__all_sync(0xFFFFFFFFu, freed)) freed = !aborted() && mbar_wait(empty(slot), ph);
          if (!__all_sync(0xFFFFFFFFu, freed)) {
            if (lane == 0 && !aborted()) fail();
            stop = true;
            break;
          }
        }
        if (lane == (g & 31)) {
          mbar_expect_tx(full(slot), kWBox + kSfTile);
          tma_load_2d(base + slot * kSlot, &maps.w[U.p], full(slot), (U.k0 + k) * 128, U.tile * 128,
                      pol_w);
          bulk_load(base + slot * kSlot + kWBox,
                    P.w_scales + (static_cast<size_t>(U.tile) * chunks + U.k0 + k) * kSfTile, kSfTile,
                    full(slot), pol_w);
        }
        __syncwarp();
        if (lane == 0) *issued_w = g + 1;
      }
    }
    if (lane == 0) CH_TL(2);
    if (!paired) cluster_wait_acquire();
  } else if (warp == 1) {
    // ---------------- activation loader and MMA issuer
    pdl_wait();  // the first activation is the previous kernel's output
    if (lane == 0) CH_TL(3);
    cluster_wait_acquire();
    const uint64_t pol_a = policy_evict_last();
    const uint32_t id0 = idesc_mxf8(mtile, 0), id1 = idesc_mxf8(mtile, 1);
    const uint32_t id2 = idesc_mxf8(mtile, 2), id3 = idesc_mxf8(mtile, 3);
    const uint64_t sd = sdesc_sf(base);  // high half shared by every scale-tile descriptor
    const uint32_t sf_hi = static_cast<uint32_t>(sd >> 32);
    int g = 0, ub = 0, chunk_base = 0;
    for (int p = 0; p < 3; ++p) {
      int u0 = 0;
      while (u0 < nu && units[u0].p != p) ++u0;
      int u1 = u0;
      while (u1 < nu && units[u1].p == p) ++u1;
      if (u0 == u1) {
        chunk_base += pl.act_chunks[p];
        continue;
      }
      const ChainProj& P = a.proj[p];
      const int k0 = units[u0].k0, nk = units[u0].nk;
      bool ok = !aborted();
      if (p > 0 && ok) {
        // activation chunk j is tile k0 + j of the previous projection: ready once
        // its S_{p-1} ranks have published (the counters start every call at 0)
        const unsigned target = static_cast<unsigned>(a.proj[p - 1].splits);
        bool ready = true;
        if (lane < nk) {
          const unsigned* c = a.counters + a.cnt_off[p - 1] + k0 + lane;
          const uint64_t t0 = globaltimer();
          for (uint32_t i = 0;; ++i) {
            if (ld_acquire_gpu(c) >= target) break;
            if ((i & 31u) == 31u &&
                (ld_acquire_gpu(a.counters + 2) != 0 || globaltimer() - t0 > kPeerWaitLimitNs)) {
              ready = false;
              break;
            }
          }
        }
        ok = __all_sync(0xFFFFFFFFu, ready);
        if (lane == 0) CH_TL(p == 1 ? 8 : 11);
        if (!ok && lane == 0 && !aborted()) fail();
        // the tiles were written through the generic proxy; the TMA reads them
        // through the async proxy
        fence_proxy_async_global();
      }
      if (ok) {
        if (lane == 0) {
          mbar_expect_tx(act_bar(p), static_cast<uint32_t>(nk) * (a_bytes + nsfb * kSfTile));
          *act_open = *act_open | (1 << p);
        }
        __syncwarp();
        if (lane < nk)
          tma_load_2d(base + pl.off_act[p] + lane * a_bytes, &maps.a[p], act_bar(p), (k0 + lane) * 128, 0,
                      pol_a);
        if (lane == 31)
          for (int rt = 0; rt < nsfb; ++rt)
            bulk_load(base + pl.off_asf[p] + static_cast<uint32_t>(rt * pl.act_chunks[p]) * kSfTile,
                      P.a_scales + (static_cast<size_t>(rt) * (P.k / 128) + k0) * kSfTile,
                      static_cast<uint32_t>(nk) * kSfTile, act_bar(p), pol_a);
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(act_bar(p), 0));
        if (lane == 0) CH_TL(p == 0 ? 4 : p == 1 ? 9 : 12);
        if (!ok && lane == 0) fail();
        if (ok && lane == 0) *act_open = *act_open & ~(1 << p);
      }
      if (ok) {
        tc_fence_after();
        if (elect_one())
          for (int j = 0; j < nk; ++j)
            for (int rt = 0; rt < nsfb; ++rt)
              tmem_cp_32x128b_x4_lh(
                  tmem + sfb_col0 + 4u * nsfb * (chunk_base + j) + 4u * rt,
                  static_cast<uint32_t>(sdesc_sf(base + pl.off_asf[p] +
                                                 static_cast<uint32_t>(rt * pl.act_chunks[p] + j) * kSfTile)),
                  sf_hi);
        __syncwarp();
      }
      const uint64_t ad = sdesc_k_sw128(base + pl.off_act[p]);
      for (int u = u0; u < u1; ++u, ++ub) {
        const Unit& U = units[u];
        const int b = ub & 1;
        if (ub >= 2 && ok) {
          // the epilogue has read this accumulator's previous unit
          const bool freed = __all_sync(0xFFFFFFFFu, mbar_wait(acc_empty(b), static_cast<uint32_t>(((ub >> 1) - 1) & 1)));
          if (!freed) {
            if (lane == 0) fail();
            ok = false;
          }
        }
        tc_fence_after();
        for (int k = 0; k < U.nk; ++k, ++g) {
          const int slot = g % R;
          if (ok) {
            const uint32_t ph = static_cast<uint32_t>((g / R) & 1);
            bool landed = mbar_try_wait(full(slot), ph);
            if (!__all_sync(0xFFFFFFFFu, landed)) landed = !aborted() && mbar_wait(full(slot), ph);
            if (!__all_sync(0xFFFFFFFFu, landed)) {
              if (lane == 0 && !aborted()) fail();
              ok = false;
            } else if (lane == 0) {
              *consumed_w = g + 1;
            }
          }
          if (ok) {
            tc_fence_after();
            if (elect_one()) {
              const uint64_t wd = sdesc_k_sw128(base + slot * kSlot);
              const uint32_t w_lo = static_cast<uint32_t>(wd), op_hi = static_cast<uint32_t>(wd >> 32);
              const uint32_t a_lo = static_cast<uint32_t>(ad) + static_cast<uint32_t>(k) * (a_bytes >> 4);
              const uint32_t ta = tmem + sfa_col + 4u * slot;
              const uint32_t tb = tmem + sfb_col0 + 4u * nsfb * (chunk_base + k);
              const uint32_t acc = tmem + static_cast<uint32_t>(b * mtile);
              tmem_cp_32x128b_x4_lh(ta, static_cast<uint32_t>(sdesc_sf(base + slot * kSlot + kWBox)), sf_hi);
              mma_mxf8_lh(acc, w_lo, op_hi, a_lo, op_hi, id0, ta, tb, k != 0);
              mma_mxf8_lh(acc, w_lo + 2, op_hi, a_lo + 2, op_hi, id1, ta, tb, 1);
              mma_mxf8_lh(acc, w_lo + 4, op_hi, a_lo + 4, op_hi, id2, ta, tb, 1);
              mma_mxf8_lh(acc, w_lo + 6, op_hi, a_lo + 6, op_hi, id3, ta, tb, 1);
              tc_commit(empty(slot));  // the slot may be refilled once these complete
            }
            __syncwarp();
          }
        }
        // always signalled (no MMAs after a failure): the epilogue never waits in vain
        if (elect_one()) tc_commit(acc_full(b));
        __syncwarp();
      }
      if (p == 0 && lane == 0) CH_TL(5);
      if (p == 1 && lane == 0) CH_TL(1);
      chunk_base += pl.act_chunks[p];
    }
  } else {
    // ---------------- epilogue: warps 2..5 own TMEM lanes 32 q .. 32 q + 31
    const int q = warp & 3;
    cluster_wait_acquire();  // the peers' barriers are initialized before the first push
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    float* const staged = reinterpret_cast<float*>(bp + pl.off_staged);
    for (int u = 0; u < nu; ++u) {
      const Unit& U = units[u];
      const ChainProj& P = a.proj[U.p];
      const int b = u & 1;
      bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(acc_full(b), static_cast<uint32_t>((u >> 1) & 1)));
      if (!ok && lane == 0) fail();
      ok = ok && !aborted();
      tc_fence_after();
      float v[16];
      if (ok) tmem_ld_32x32b_x16(lane_base + static_cast<uint32_t>(b * mtile), v);
      if (warp == 2 && lane == 0 && u == 0) CH_TL(6);
      if (warp == 2 && lane == 0 && u == 1) CH_TL(13);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(b));
      const int S = U.S, s = U.s;
      const int col = U.tile * 128 + q * 32 + lane;
      __nv_bfloat16* const out = static_cast<__nv_bfloat16*>(P.out);
      const bool requant = P.q != nullptr && U.tile * 128 + q * 32 < P.q_cols;
      // one output block (row m, this warp's 32 columns): bf16 and its MX block
      auto store = [&](int m, float acc) {
        const __nv_bfloat16 hb = __float2bfloat16_rn(acc);
        if (out != nullptr) out[static_cast<size_t>(m) * P.n + col] = hb;
        if (requant) {
          const float x = __bfloat162float(hb);
          const uint32_t amax_bits = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(x)));
          uint32_t sbyte, code;
          if (amax_bits >= 0x7F800000u) {  // Inf or NaN in the block
            sbyte = 0xFFu;
            code = 0x7Fu;
          } else {
            sbyte = mx_scale_byte(__uint_as_float(amax_bits));
            code = cvt_e4m3x2(x * mx_inv_scale(sbyte), 0.f) & 0xFFu;
          }
          P.q[static_cast<size_t>(m) * P.q_cols + col] = static_cast<uint8_t>(code);
          if (lane == 0) P.q_scales[swz_offset(m, col >> 5, P.q_cols >> 5)] = static_cast<uint8_t>(sbyte);
        }
      };
      if (S == 1) {
        if (ok)
          for (int m = 0; m < M; ++m) store(m, v[m]);
      } else {
        // stage by owner: staged[o][q][j] = partial of row j S + o (o = m % S)
        const int rc = (M + S - 1) / S;
        int o = 0, jr = 0;
#pragma unroll
        for (int j = 0; j < kMaxRows; ++j) {
          if (ok && j < M) staged[((o * 4 + q) * rc + jr) * 32 + lane] = v[j];
          if (++o == S) {
            o = 0;
            ++jr;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        const uint32_t recv =
            base + pl.off_recv[U.p] + static_cast<uint32_t>(U.idx) * pl.recv_unit_bytes[U.p];
        const uint32_t rbar = red_bar(red_first[U.p] + U.idx);
        const int first = rank - s;  // cluster rank of the group's split 0
        // sent even after a failure (meaningless values then): an owner counts on
        // every byte arriving
        if (lane < S && lane != s) {
          const int cnt = lane < M ? (M - lane + S - 1) / S : 0;
          if (cnt > 0) {
            const int src = s < lane ? s : s - 1;
            bulk_copy_to_peer(map_shared_rank(recv + static_cast<uint32_t>((src * 4 + q) * rc) * 128u, first + lane),
                              base + pl.off_staged + static_cast<uint32_t>((lane * 4 + q) * rc) * 128u,
                              static_cast<uint32_t>(cnt) * 128u, map_shared_rank(rbar, first + lane));
            bulk_commit();
          }
        }
        if (lane < S) bulk_wait_read();
        __syncwarp();
        const int own = s < M ? (M - s + S - 1) / S : 0;
        if (own > 0) {
          const bool got = __all_sync(0xFFFFFFFFu, mbar_wait(rbar, 0, kPeerWaitLimitNs));
          if (!got && lane == 0) fail();
          ok = ok && got && !aborted();
          if (ok) {
            const float* const mine = staged + ((s * 4 + q) * rc) * 32 + lane;
            const float* const theirs = reinterpret_cast<const float*>(bp + (recv - base)) + q * rc * 32 + lane;
            for (int j = 0; j < own; ++j) {
              float w[8];
#pragma unroll
              for (int r = 0; r < 8; ++r)
                w[r] = r >= S ? 0.f : r == s ? mine[j * 32] : theirs[((r < s ? r : r - 1) * 4 * rc + j) * 32];
              float acc = 0.f;
#pragma unroll
              for (int r = 0; r < 8; ++r)
                if (r < S) acc += w[r];
              store(j * S + s, acc);
            }
          }
        }
      }
      if (ok && s == 0 && P.q != nullptr && U.tile * 128 < P.q_cols) {
        // the tile's four scale columns in the padding rows [M, ceil128(M))
        const int mpad = (M + 127) & ~127;
        for (int i = threadIdx.x - 64; i < (mpad - M) * 4; i += 128)
          P.q_scales[swz_offset(M + (i >> 2), U.tile * 4 + (i & 3), P.q_cols >> 5)] = 0;
      }
      if (U.p < 2 && P.q != nullptr && U.tile * 128 < P.q_cols) {
        // publish: every block of this rank's rows of the tile is stored
        named_barrier_sync(1, 128);
        if (warp == 2 && lane == 0 && !aborted()) {
          __threadfence();
          atomicAdd(a.counters + a.cnt_off[U.p] + U.tile, 1u);
          CH_TL(U.p == 0 ? 7 : 10);
        }
      }
      if (warp == 2 && lane == 0 && u == nu - 1) CH_TL(14);
    }
  }

  // ---------------- end of the call: the last CTA to get here (every tile has
  // been published and every poll has ended) clears the counters for the next
  // call, which touches them only after its grid-dependency wait on this one
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    words[5] = atomicAdd(a.counters + 1, 1u) == gridDim.x - 1 ? 1u : 0u;
  }
  __syncthreads();
  if (words[5] != 0) {
    const int n = a.cnt_off[1] + a.proj[1].n / 128;
    for (int i = a.cnt_off[0] + threadIdx.x; i < n; i += kThreads) a.counters[i] = 0u;
    if (threadIdx.x == 0) {
      a.counters[1] = 0u;  // CTAs finished
      a.counters[2] = 0u;  // abort (the status word keeps the failure)
      atomicAdd(a.counters, 1u);  // calls completed (diagnostic)
    }
  }
  if (aborted()) {
    // copies still in flight land before exit: the ring's issued, unconsumed
    // chunks (distinct slots) and activation loads that never completed
    if (warp == 0)
      for (int g = *consumed_w; g < *issued_w; ++g) mbar_wait(full(g % R), static_cast<uint32_t>((g / R) & 1));
    if (warp == 1 && lane < 3 && (*act_open & (1 << lane))) mbar_wait(act_bar(lane), 0);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, pl.tmem_cols);
  }
  if (threadIdx.x == 0) CH_TL(15);
}

int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

}  // namespace

ChainPlan plan_chain(int M, const ChainProj (&proj)[3], int clusters) {
  ChainPlan pl{};
  pl.ok = false;
  if (M < 1 || M > kMaxRows || clusters < 1) return pl;
  const int mtile = (M + 15) & ~15;
  const int nsfb = 1;
  const uint32_t a_bytes = static_cast<uint32_t>(mtile) * 128u;
  pl.clusters = clusters;
  int units = 0, chunks_total = 0;
  uint32_t staged = 0;
  for (int p = 0; p < 3; ++p) {
    const int S = proj[p].splits;
    if (S < 1 || S > kChainCluster) return pl;
    const int g = kChainCluster / S;
    const int tiles = proj[p].n / 128, chunks = proj[p].k / 128;
    if (tiles < 1 || chunks < S) return pl;
    pl.act_chunks[p] = (chunks + S - 1) / S;
    const int batches = (tiles + g - 1) / g;
    pl.max_units[p] = (batches + clusters - 1) / clusters;
    units += pl.max_units[p];
    chunks_total += pl.act_chunks[p];
    const int rc = (M + S - 1) / S;
    staged = std::max(staged, static_cast<uint32_t>(S * rc) * 512u);
    pl.recv_unit_bytes[p] = static_cast<uint32_t>((S - 1) * rc) * 512u;
  }
  if (units > kChainMaxUnits) return pl;
  // fixed part after the ring: activations, their scale tiles, staging, receive
  // areas, barriers
  uint32_t off = 0;
  uint32_t act[3], asf[3], rcv[3];
  for (int p = 0; p < 3; ++p) {
    act[p] = off;
    off += static_cast<uint32_t>(pl.act_chunks[p]) * a_bytes;  // multiples of 2 KB
  }
  for (int p = 0; p < 3; ++p) {
    asf[p] = off;
    off += static_cast<uint32_t>(nsfb * pl.act_chunks[p]) * kSfTile;
  }
  const uint32_t stg = off;
  off += staged;
  for (int p = 0; p < 3; ++p) {
    rcv[p] = off;
    off += static_cast<uint32_t>(pl.max_units[p]) * pl.recv_unit_bytes[p];
  }
  const uint32_t fixed = off;
  // ring slots in what remains of the largest allocation
  int ring = 16;
  auto total = [&](int r) {
    const uint32_t bar_bytes = 8u * (2 * r + 7 + kChainMaxUnits) + 32u;
    return static_cast<size_t>(1024 + r * kSlot + fixed) + ((bar_bytes + 7) & ~7u);
  };
  while (ring > 4 && total(ring) > kMaxDynamicSmem) --ring;
  if (total(ring) > kMaxDynamicSmem) return pl;
  pl.ring = ring;
  const uint32_t ring_bytes = static_cast<uint32_t>(ring) * kSlot;
  for (int p = 0; p < 3; ++p) {
    pl.off_act[p] = ring_bytes + act[p];
    pl.off_asf[p] = ring_bytes + asf[p];
    pl.off_recv[p] = ring_bytes + rcv[p];
  }
  pl.off_staged = ring_bytes + stg;
  pl.off_bars = (ring_bytes + fixed + 7u) & ~7u;
  pl.tmem_cols = pow2_at_least(2 * mtile + 4 * ring + 4 * nsfb * chunks_total);
  if (pl.tmem_cols > 512) return pl;
  pl.smem = total(ring);
  pl.ok = true;
  return pl;
}

int chain_max_clusters() {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = kChainCluster;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.gridDim = dim3(kChainCluster * 16, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kMaxDynamicSmem;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, chain_kernel, &cfg) != cudaSuccess) return 0;
  return n;
}

cudaError_t set_chain_attributes() {
  const void* k = reinterpret_cast<const void*>(&chain_kernel);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kMaxDynamicSmem));
}

cudaError_t launch_chain(const CUtensorMap (&maps)[6], const ChainArgs& args, cudaStream_t stream) {
  if (!args.plan.ok || args.plan.smem > kMaxDynamicSmem) return cudaErrorInvalidValue;
  ChainMaps m;
  for (int p = 0; p < 3; ++p) {
    m.w[p] = maps[p];
    m.a[p] = maps[3 + p];
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kChainCluster * args.plan.clusters, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = args.plan.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = kChainCluster;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, chain_kernel, m, args);
}

}  // namespace mx
