// push.cuh - the push split-K reduction of a K-split cluster (GEMM and WO-A).
//
// The S CTAs of a cluster hold fp32 partials of the same [M, 128] output tile
// in TMEM (lane 32 q + l = column 32 q + l, TMEM column m = row m). The outputs
// are cut into units of g rows (g = 4, or M when M < 3) by one 32-column block:
// unit u = 4 group + block, U = 4 ceil(M / g) units, and rank j owns the units
// [j U / S, (j + 1) U / S). Every CTA stores its values of a unit straight into
// the owner's receive area with one st.async of g floats, counted as bytes on
// the owner's receive barrier; the owner armed that barrier at set-up with the
// bytes it expects, so no cluster barrier is needed between the MMAs and the
// sums (only the one at set-up that makes the armed barriers visible). The
// owner then sums each of its values over the ranks in rank order, 0 first, as
// every reduction of these kernels does, so the results are the same bits.
//
// Receive area: a slot per rank of ceil(U / S) units x 32 lanes x g floats,
// the CTA's own values in its own slot; compact: a slot per peer (ranks below
// this one, then above it), the own values elsewhere (over the CTA's ring),
// 1/S less shared memory, ~0.1 us slower to sum on GB300.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace mx {

// The push reduction up to this many rows. Measured on GB300 (N = 2048, K = 5120,
// graph-replayed with PDL): 3.83-4.03 us against 4.51-4.68 us from one to eight
// rows, 4.51 against 5.11 at 16; from 32 rows on slower (6.5 against 5.8 us at
// 32), the owners' incoming 16-byte stores queueing.
constexpr int kPushMaxRows = 16;

__host__ __device__ inline int push_rows_per_unit(int M) { return M < 3 ? M : 4; }
__host__ __device__ inline int push_units(int M) {
  const int g = push_rows_per_unit(M);
  return 4 * ((M + g - 1) / g);
}
__host__ __device__ inline uint32_t push_slot_bytes(int M, int S) {
  return static_cast<uint32_t>((push_units(M) + S - 1) / S) * 128u * static_cast<uint32_t>(push_rows_per_unit(M));
}
__host__ __device__ inline uint32_t push_area_bytes(int M, int S, bool compact) {
  return static_cast<uint32_t>(compact ? S - 1 : S) * push_slot_bytes(M, S);
}

// The exchange's geometry for rank `split` of S, computed once at kernel start
// (its divisions stay off the path from the accumulator to the output).
struct PushGeometry {
  int M, S, split;
  int pg, units;         // rows per unit, units
  int own_lo, own_hi;    // this rank's units
  int lg;                // log2 of pg
  uint32_t slot;         // bytes of one slot
  __device__ __forceinline__ PushGeometry(int M_, int S_, int split_)
      : M(M_), S(S_), split(split_), pg(push_rows_per_unit(M_)), units(push_units(M_)),
        own_lo(split_ * units / S_), own_hi((split_ + 1) * units / S_), lg(pg == 4 ? 2 : pg - 1),
        slot(push_slot_bytes(M_, S_)) {}
};

// The bytes this rank's receive barrier expects: the S - 1 peers' values of
// its units whose column block q is wanted (want_q(q)).
template <typename WantQ>
__device__ __forceinline__ uint32_t push_expect_bytes(const PushGeometry& pg_, WantQ want_q) {
  uint32_t expect = 0;
  for (int u = pg_.own_lo; u < pg_.own_hi; ++u)
    if (want_q(u & 3)) expect += 128u * static_cast<uint32_t>(pg_.pg * (pg_.S - 1));
  return expect;
}

// Warp q's part of the exchange: its lanes' values of rows [0, M) (TMEM lanes
// 32 q .. 32 q + 31 from tmem_q, columns 0 .. M - 1) go unit by unit to their
// owners; `recv` and `recv_bar` are this CTA's receive area and barrier (the
// peers' by mapa), `own` where this rank keeps its own units. With ok false
// (a failed accumulator wait) zeros are sent, so that no owner waits for
// bytes that never come.
template <bool kCompact>
__device__ __forceinline__ void push_send(const PushGeometry& G, uint32_t tmem_q, int q, int lane, uint32_t recv,
                                          uint32_t recv_bar, float* own, bool ok) {
  const int M = G.M, S = G.S, split = G.split, pg = G.pg, units = G.units;
  const uint32_t slot = G.slot;
  int j = -1, lo = 0, hi = 0;  // the current owner and its units [lo, hi)
  uint32_t peer = 0, peer_bar = 0;
  auto send = [&](int u, float x0, float x1, float x2, float x3) {
    while (u >= hi) {
      ++j;
      lo = hi;
      hi = (j + 1) * units / S;
      peer = map_shared_rank(recv, j);
      peer_bar = map_shared_rank(recv_bar, j);
    }
    // at the owner: this rank's slot
    const uint32_t at = static_cast<uint32_t>((u - lo) * 32 + lane) * 4u * static_cast<uint32_t>(pg);
    const uint32_t off = static_cast<uint32_t>(kCompact && split > j ? split - 1 : split) * slot + at;
    if (j == split) {
      float* const d = own + at / 4;
      d[0] = x0;
      if (pg > 1) d[1] = x1;
      if (pg > 2) {
        d[2] = x2;
        d[3] = x3;
      }
    } else if (pg == 4) {
      st_async_v4(peer + off, x0, x1, x2, x3, peer_bar);
    } else if (pg == 2) {
      st_async_v2(peer + off, x0, x1, peer_bar);
    } else {
      st_async_b32(peer + off, __float_as_uint(x0), peer_bar);
    }
  };
  for (int c0 = 0; c0 < M; c0 += 16) {
    float v[16];
    if (ok) {
      tmem_ld_32x32b_x16(tmem_q + c0, v);
    } else {
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) v[jj] = 0.f;
    }
    // unit of rows [c0 + e0, c0 + e0 + g): one unit per 4 rows, or the only
    // unit when M < 3
#pragma unroll
    for (int e0 = 0; e0 < 16; e0 += 4) {
      if (c0 + e0 >= M) break;  // warp-uniform
      send(4 * ((c0 + e0) / 4) + q, v[e0], v[e0 + 1], v[e0 + 2], v[e0 + 3]);
    }
  }
}

// This rank's sums, once its receive barrier has completed and its own values
// are visible to every warp: the (unit, row) pairs of its wanted units are
// dealt over `nwarps` warps; each value's S <= 8 loads are issued together and
// added in rank order, then emit(item = 4 m + block, sum) (warp-uniform call).
template <bool kCompact, typename WantQ, typename Emit>
__device__ __forceinline__ void push_sum(const PushGeometry& G, int warp, int nwarps, int lane, const float* recv,
                                         const float* own, WantQ want_q, Emit emit) {
  const int M = G.M, S = G.S, split = G.split, pg = G.pg, own_lo = G.own_lo, own_hi = G.own_hi, lg = G.lg;
  const uint32_t slot = G.slot;
  for (int t = warp; t < ((own_hi - own_lo) << lg); t += nwarps) {
    const int u = own_lo + (t >> lg), e = t & (pg - 1), m = (u >> 2) * pg + e;
    if (m >= M || !want_q(u & 3)) continue;  // warp-uniform
    const uint32_t at = ((static_cast<uint32_t>(u - own_lo) * 32u + lane) << lg) + e;
    float v[8];
    if constexpr (kCompact) {
#pragma unroll
      for (int r = 0; r < 8; ++r)
        v[r] = r >= S ? 0.f : r == split ? own[at] : recv[static_cast<uint32_t>(r < split ? r : r - 1) * (slot / 4) + at];
    } else {
#pragma unroll
      for (int r = 0; r < 8; ++r) v[r] = r < S ? recv[static_cast<uint32_t>(r) * (slot / 4) + at] : 0.f;
    }
    float acc = 0.f;
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r < S) acc += v[r];
    emit(4 * m + (u & 3), acc);
  }
}

}  // namespace mx
