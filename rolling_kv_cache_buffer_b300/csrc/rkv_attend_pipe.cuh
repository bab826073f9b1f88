// rkv_attend_pipe.cuh -- the streaming side shared by the tensor-core
// attention kernels: stage geometry, the producer warp and the fine R(d) table.
//
// One persistent CTA per SM.  Lane 0 of warp 0 walks the CTA's share of the
// block list (rkv_attend_common.cuh) and, per block of TK slots, fills one
// shared-memory stage: the K and V tiles as one 4-D TMA box each (128-byte
// swizzle) and one or two (cos, sin) rows of the RoPE table.  Stages form a
// ring with a full barrier (copies landed) and an empty barrier (consumers done)
// each.  Between unit segments the producer waits for the consumers' merge,
// which reuses the stage memory.
#pragma once

#include "rkv_attend_common.cuh"

namespace rkv {

constexpr int SMEM_LIMIT = 227 * 1024;   // opt-in shared memory per CTA

template <int D, bool ROTK>
struct PipeCfg {
  static constexpr int HALF = D / 2;
  static constexpr int TILE = TK * D * 2;                 // bf16 K (or V) block tile
  static constexpr int TROW = ROTK ? HALF * 8 : 0;        // one (cos, sin) row
  static constexpr int STAGE = ((2 * TILE + 2 * TROW + 1023) / 1024) * 1024;
  static constexpr int FINE = ROTK ? TK * HALF * 8 : 0;   // R(d) table, d < TK
};

// Which table rows a block's stage carries (r0 = re-based position of the
// block's first slot):
//   KEY_BASES: row r0 and, when the block holds the ring's end, row
//     |r0 - W_ring| (the consumer flips its sine when r0 < W_ring, to get
//     R(r0 - W_ring));
//   NO_ROWS: none (the consumers derive the rows themselves).
enum TableRows { KEY_BASES = 1, NO_ROWS = 2 };

// 16-byte chunk `grp` of key row `row` (0..TK-1) of a block tile: the tile is
// D/64 boxes of TK rows x 128 bytes, 128-byte swizzled.
__device__ __forceinline__ uint32_t tile_swz(int row, int grp) {
  const int box = grp >> 3, cq = grp & 7;
  return static_cast<uint32_t>(box * (TK * 128) + row * 128 + ((cq ^ (row & 7)) << 4));
}

// Fine table: row d (0..TK-1) holds the rotation R(d) for every pair; 16-byte
// chunk k holds pairs 2k and 2k+1.  The chunk sits at position
// k ^ ((d mod NCH/4) * 4) of its row (NCH = D/4 chunks per row), so the two
// keys that one 8-lane phase of a 128-bit load reads (rows d, d+1, same k)
// fall into different halves of the 128-byte bank window.  Split-half chunks
// are (cos_2k, cos_2k+1, sin_2k, sin_2k+1), interleaved ones
// (cos_2k, sin_2k, cos_2k+1, sin_2k+1).
template <int D>
__device__ __forceinline__ uint32_t fine_chunk(int d, int k) {
  constexpr int NCH = D / 4;
  return static_cast<uint32_t>((k ^ ((d & (NCH / 4 - 1)) << 2)) << 4);
}

// The chunk kernel's layout of the same table: chunk k of row d at position
// k ^ (d mod 8), so that eight keys d..d+7 reading the same chunk k (one phase
// of a 128-bit load) hit eight different 16-byte bank groups.
template <int D>
__device__ __forceinline__ uint32_t fine_chunk_keys(int d, int k) {
  return static_cast<uint32_t>((k ^ (d & 7)) << 4);
}

// The rotation warps of the tcgen05 chunk kernel read the same table with
// eight lanes on eight consecutive keys d and one chunk j of pairs (2j, 2j+1)
// as (cos, cos, sin, sin) (the grouped table): chunk j of row d sits at
// position j ^ (d mod 8) of its row, so those eight reads hit eight different
// 16-byte bank groups.
__device__ __forceinline__ uint32_t fine_chunk_rot(int d, int j) {
  return static_cast<uint32_t>((j ^ (d & 7)) << 4);
}
// Threads t0, t0+nt, ... fill that table from rows 0..TK-1 of the grouped one.
template <int D>
__device__ __forceinline__ void load_fine_rot(const AttendParams& p, uint8_t* fine, int t0,
                                              int nt) {
  constexpr int HALF = D / 2;
  for (int idx = t0; idx < TK * HALF / 2; idx += nt) {
    const int d = idx / (HALF / 2), j = idx % (HALF / 2);
    const float4 v = __ldg(p.table_g + (size_t)d * (HALF / 2) + j);
    *reinterpret_cast<float4*>(fine + d * HALF * 8 + fine_chunk_rot(d, j)) = v;
  }
}

// Threads t0, t0+nt, ... fill the fine table from rows 0..TK-1 of the global
// (cos, sin) table (KEYS: in the chunk kernel's layout).
template <int D, int STYLE, bool KEYS = false>
__device__ __forceinline__ void load_fine(const AttendParams& p, uint8_t* fine, int t0, int nt) {
  constexpr int HALF = D / 2;
  for (int idx = t0; idx < TK * HALF / 2; idx += nt) {
    const int d = idx / (HALF / 2), k = idx % (HALF / 2);
    const float2 a = __ldg(p.table + (size_t)d * HALF + 2 * k);
    const float2 c = __ldg(p.table + (size_t)d * HALF + 2 * k + 1);
    const float4 v = STYLE == 0 ? make_float4(a.x, c.x, a.y, c.y)
                                : make_float4(a.x, a.y, c.x, c.y);
    *reinterpret_cast<float4*>(fine + d * HALF * 8 +
                               (KEYS ? fine_chunk_keys<D>(d, k) : fine_chunk<D>(d, k))) = v;
  }
}

// Threads t0, t0 + nt, ... of the CTA (all of them by default) bring its share
// of the queries into L2 (the queries are not written by the append kernel
// that may still be running).
__device__ __forceinline__ void prefetch_queries(const AttendParams& p, int D, int t0 = -1,
                                                 int nt = 0) {
  if (t0 < 0) { t0 = threadIdx.x; nt = blockDim.x; }
  const size_t qbytes = (size_t)p.L_att * p.sh.S * p.c * p.sh.Hq * D * (p.sh.q_bf16 ? 2 : 4);
  const size_t lines = (qbytes + 127) / 128;
  const size_t l0 = lines * blockIdx.x / gridDim.x, l1 = lines * (blockIdx.x + 1) / gridDim.x;
  for (size_t l = l0 + t0; l < l1; l += nt)
    prefetch_l2(static_cast<const uint8_t*>(p.q) + l * 128);
}

// Threads of the CTA bring the stream states into L2.  A prefetch reads
// nothing into the SM, so it may run before the previous kernel that writes
// the states has finished.
__device__ __forceinline__ void prefetch_states(const AttendParams& p) {
  const int lines = (p.sh.S * (int)sizeof(StreamState) + 127) / 128;
  for (int i = threadIdx.x; i < lines; i += blockDim.x)
    prefetch_l2(reinterpret_cast<const uint8_t*>(p.st) + (size_t)i * 128);
}

// The producer loop, run by lane 0 of warp 0 over blocks [rb, re).  Returns
// the number of stages it filled.  Stops early (status set, *abort raised) if
// a wait runs out.  The (cos, sin) rows come from `rows` (rows of D/2 float2
// of the global table, or of its grouped copy), p.table when null.
template <int D, bool ROTK, int ROWS>
__device__ __forceinline__ int produce(const AttendParams& p, const CUtensorMap* tmK,
                                       const CUtensorMap* tmV, uint8_t* stages, uint64_t* full,
                                       uint64_t* empty, uint64_t* mdone, const int* pre,
                                       const int* sa, const int* sfill, int rb, int re,
                                       volatile int* abort_flag, const float2* rows = nullptr) {
  using C = PipeCfg<D, ROTK>;
  const int NS = p.ns;
  const float2* rtab = rows ? rows : p.table;
  int stage = 0, round = 0, issued = 0, seg = 0;
  bool stop = false;
  const uint64_t pol = l2_evict_first_policy();   // every K/V row is read once
  for (int x = rb; x < re && !stop; ++seg) {
    // Per unit segment: the unit, then the block geometry advanced per block.
    const UnitRef u = unit_of_cached(x, p, pre, sa, sfill);
    // The merge of the previous segment uses the stage memory: wait for it.
    if (seg > 0 && !mbar_wait_or_abort(smem_u32(mdone), (seg - 1) & 1, abort_flag)) {
      *abort_flag = 1;
      p.st[u.s].status = STATUS_DEVICE_STATE;
      break;
    }
    const int x1 = min(u.uend, re);
    const int ug = static_cast<int>(unit_index(p, u));
    // Block geometry stepped in scalars (the producer is one thread that must
    // keep the ring full): j = block within the unit, the pinned prefix's npb
    // blocks first (slot block j, positions from 0), then the ring blocks
    // (slot block NP + br, first slot at position npin + r0r).
    const int Wg = p.sh.Wring, NBr = p.sh.NBr;
    const int npb = (u.npin + TK - 1) / TK;
    int j = x - u.ustart;
    int br = u.a / TK, r0r = 0;
    if (j >= npb) br = touched_block(u.a, j - npb, NBr);
    r0r = br * TK - u.a;
    if (r0r < 0) r0r += Wg;
    for (; x < x1; ++x, ++j) {
      const bool ring = j >= npb;
      const int blk = ring ? p.sh.NP + br : j;
      const int r0 = ring ? u.npin + r0r : j * TK;
      const int wrap_at = ring ? Wg - r0r : TK;
      if (*abort_flag) { stop = true; break; }
      if (round > 0 &&
          !mbar_wait_or_abort(smem_u32(empty + stage), (round - 1) & 1, abort_flag)) {
        *abort_flag = 1;
        p.st[u.s].status = STATUS_DEVICE_STATE;
        stop = true;
        break;
      }
      const uint32_t bar = smem_u32(full + stage);
      const uint32_t dst = smem_u32(stages + (size_t)stage * C::STAGE);
      const bool wraps = wrap_at < TK;
      uint32_t bytes = 2 * C::TILE;
      if constexpr (ROTK && ROWS != NO_ROWS) bytes += wraps ? 2 * C::TROW : C::TROW;
      mbar_arrive_expect_tx(bar, bytes);
      // One box per tile: {64 elements, TK rows, the D/64 row halves, one unit}.
      tma_load_4d_hint(dst, tmK, 0, blk * TK, 0, ug, bar, pol);
      tma_load_4d_hint(dst + C::TILE, tmV, 0, blk * TK, 0, ug, bar, pol);
      if constexpr (ROTK && ROWS != NO_ROWS) {
        const int rowA = r0, rowB = r0 >= Wg ? r0 - Wg : Wg - r0;
        bulk_load(dst + 2 * C::TILE, rtab + (size_t)rowA * C::HALF, C::TROW, bar);
        if (wraps)
          bulk_load(dst + 2 * C::TILE + C::TROW, rtab + (size_t)rowB * C::HALF, C::TROW, bar);
      }
      ++issued;
      if (++stage == NS) { stage = 0; ++round; }
      if (ring) {
        if (++br == NBr) br = 0;
        r0r += TK;
        if (r0r >= Wg) r0r -= Wg;
      }
    }
  }
  return issued;
}

}  // namespace rkv
