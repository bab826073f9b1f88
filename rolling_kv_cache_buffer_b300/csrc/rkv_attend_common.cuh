// rkv_attend_common.cuh -- pieces shared by the attention kernels: the block
// list of a call, the per-warp block sequence, and the log-sum-exp merge of
// the partial results of one (stream, layer, KV head) unit.
//
// Work layout.  A unit's window is cut into aligned slot blocks of TK slots;
// the units of all streams (stream-major, then layer, then KV head) are laid
// end to end and each persistent CTA takes one contiguous, equal share of the
// blocks.  Inside a CTA every unit segment is split into NWARP contiguous
// chunks, one per warp; each warp streams its chunk through its own ring of
// TMA stages and keeps an online-softmax state.  At the end of a segment the
// warps merge through shared memory; a unit split across CTAs is finished by
// the CTA that arrives last on the unit's ticket (no CTA waits on another).
#pragma once

#include "rkv_internal.h"

namespace rkv {

struct UnitRef {
  int s, l, g;          // stream, layer (within the call), KV head
  int nb;               // blocks per unit of this stream (pinned prefix, then ring)
  int ustart, uend;     // [ustart, uend): this unit's blocks in the call's list
  int a;                // origin mod W_ring (ring slot of the oldest retained pair)
  int fill;             // retained pairs
  int npin;             // pinned prefix pairs
};

__device__ __forceinline__ int stream_blocks(const AttendParams& p, int s) {
  const StreamState st = p.st[s];
  if (!state_ok(st, p.sh)) return 0;
  return unit_blocks(st.ring, st.fill, st.npin, p.sh.NBr);
}

// pre[s] = first block of stream s in the call's list, pre[S] = total.  One
// warp computes it (lane = its lane index); the caller synchronises the CTA
// afterwards.
__device__ __forceinline__ void build_prefix_warp(const AttendParams& p, int* pre, int lane) {
  const int per_unit = p.L_att * p.sh.Hkv;
  int carry = 0;
  if (lane == 0) pre[0] = 0;
  for (int base = 0; base < p.sh.S; base += 32) {
    const int s = base + lane;
    int v = (s < p.sh.S) ? stream_blocks(p, s) * per_unit : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += t;
    }
    if (s < p.sh.S) pre[s + 1] = carry + v;
    carry += __shfl_sync(0xffffffffu, v, 31);
  }
}
// Warp 0 of the CTA builds the prefix.
__device__ __forceinline__ void build_prefix(const AttendParams& p, int* pre) {
  if (threadIdx.x < 32) build_prefix_warp(p, pre, threadIdx.x);
}

// As build_prefix_warp, and also caches every stream's ring start a = origin
// mod W_ring with its pinned prefix pairs (pack_an; -1 for a stream whose
// state is not valid) and fill in shared memory, so later unit lookups need no
// global load; with `slag`, also the lag of stored-rotated keys that follow a
// re-basing epoch (0 otherwise).
__device__ __forceinline__ void build_prefix_cached(const AttendParams& p, int* pre, int* sa,
                                                    int* sfill, int lane, int* slag = nullptr) {
  const int per_unit = p.L_att * p.sh.Hkv;
  int carry = 0;
  if (lane == 0) pre[0] = 0;
  for (int base = 0; base < p.sh.S; base += 32) {
    const int s = base + lane;
    int v = 0;
    if (s < p.sh.S) {
      const StreamState st = p.st[s];
      const bool ok = state_ok(st, p.sh);
      sa[s] = ok ? pack_an(st.ring, st.npin) : -1;
      sfill[s] = ok ? st.fill : 0;
      if (slag) slag[s] = (ok && p.sh.epoch) ? st.pending : 0;
      v = ok ? unit_blocks(st.ring, st.fill, st.npin, p.sh.NBr) * per_unit : 0;
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += t;
    }
    if (s < p.sh.S) pre[s + 1] = carry + v;
    carry += __shfl_sync(0xffffffffu, v, 31);
  }
}

// The unit holding block x of the call's list, from the cached stream data.
__device__ __forceinline__ UnitRef unit_of_cached(int x, const AttendParams& p, const int* pre,
                                                  const int* sa, const int* sfill) {
  int lo = 0, hi = p.sh.S;  // pre[lo] <= x < pre[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid] <= x) lo = mid; else hi = mid;
  }
  UnitRef u;
  u.s = lo;
  u.a = sa[lo] & 0xffff;
  u.npin = sa[lo] >> 16;
  u.fill = sfill[lo];
  u.nb = unit_blocks(u.a, u.fill, u.npin, p.sh.NBr);
  const int xs = x - pre[lo];
  const int ul = xs / u.nb;
  u.l = ul / p.sh.Hkv;
  u.g = ul - u.l * p.sh.Hkv;
  u.ustart = pre[lo] + ul * u.nb;
  u.uend = u.ustart + u.nb;
  return u;
}

__device__ __forceinline__ UnitRef unit_of(int x, const AttendParams& p, const int* pre) {
  int lo = 0, hi = p.sh.S;  // pre[lo] <= x < pre[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid] <= x) lo = mid; else hi = mid;
  }
  UnitRef u;
  u.s = lo;
  const StreamState st = p.st[lo];
  u.a = st.ring;
  u.fill = st.fill;
  u.npin = st.npin;
  u.nb = unit_blocks(u.a, u.fill, u.npin, p.sh.NBr);
  const int xs = x - pre[lo];
  const int ul = xs / u.nb;
  u.l = ul / p.sh.Hkv;
  u.g = ul % p.sh.Hkv;
  u.ustart = pre[lo] + ul * u.nb;
  u.uend = u.ustart + u.nb;
  return u;
}

// Block y of unit u.  Its slots blk*TK .. blk*TK+TK-1 hold, for slot d of the
// block, re-based position r0 + d, or r0 + d - W_ring for d >= wrap_at (the
// ring's end falls inside the block); the slots at positions below lim are
// in the window.  Pinned prefix blocks (slots 0.., positions 0..npin-1) come
// first; a ring block's slot P + x holds retained pair (x - a) mod W_ring, at
// position npin + that.  Without pinned slots: blk = ring block, r0 =
// (blk*TK - a) mod W, wrap_at = W - r0, lim = fill.
struct BlockGeo {
  int blk;       // slot block
  int r0;        // re-based position of the block's first slot
  int wrap_at;   // slots d >= wrap_at sit at r0 + d - W_ring (>= TK: none do)
  int lim;       // slots at positions < lim are in the window
  int ring;      // 1 for a ring block, 0 for a pinned prefix block
};
__device__ __forceinline__ BlockGeo block_geo(int y, const UnitRef& u, const Shape& sh) {
  BlockGeo b;
  const int j = y - u.ustart;
  const int npb = (u.npin + TK - 1) / TK;
  if (j < npb) {
    b.blk = j;
    b.r0 = j * TK;
    b.wrap_at = TK;
    b.lim = u.npin;
    b.ring = 0;
    return b;
  }
  const int br = touched_block(u.a, j - npb, sh.NBr);
  int r0 = br * TK - u.a;
  if (r0 < 0) r0 += sh.Wring;
  b.blk = sh.NP + br;
  b.r0 = u.npin + r0;
  b.wrap_at = sh.Wring - r0;
  b.lim = u.npin + u.fill;
  b.ring = 1;
  return b;
}
// Position of slot d of block b.
__device__ __forceinline__ int slot_pos(const BlockGeo& b, int d, int Wring) {
  return b.r0 + d - (d >= b.wrap_at ? Wring : 0);
}

// Walks the blocks of one unit: the geometry of the current block, advanced
// by k blocks with additions and compares only (block_geo, with its
// remainder, runs once per segment and once where the walk leaves the pinned
// prefix for the ring).
struct BlockWalk {
  BlockGeo g;
  int j;     // block index within the unit
  int npb;   // pinned prefix blocks of the unit
  __device__ __forceinline__ void init(int y, const UnitRef& u, const Shape& sh) {
    j = y - u.ustart;
    npb = (u.npin + TK - 1) / TK;
    g = block_geo(y, u, sh);
  }
  // Returns the number of times the walk passed the ring's end (-1 when it
  // jumped from the pinned prefix to the ring).
  __device__ __forceinline__ int advance(int k, const UnitRef& u, const Shape& sh) {
    const int j2 = j + k;
    int wraps = 0;
    if (j >= npb) {
      int br = g.blk - sh.NP + k;
      while (br >= sh.NBr) br -= sh.NBr;
      int r0 = g.r0 - u.npin + k * TK;
      while (r0 >= sh.Wring) { r0 -= sh.Wring; ++wraps; }
      g.blk = sh.NP + br;
      g.r0 = u.npin + r0;
      g.wrap_at = sh.Wring - r0;
    } else if (j2 < npb) {
      g.blk = j2;
      g.r0 = j2 * TK;
    } else {
      g = block_geo(u.ustart + j2, u, sh);
      wraps = -1;
    }
    j = j2;
    return wraps;
  }
};

// The blocks one warp handles, in order: for each unit segment of the CTA's
// range, the warp's contiguous chunk of it.
struct WarpSeq {
  int x, re, w, y, ce;
  UnitRef u;
  __device__ __forceinline__ void init(int rb, int re_, int w_) {
    x = rb; re = re_; w = w_; y = 0; ce = 0;
  }
  __device__ __forceinline__ bool next(const AttendParams& p, const int* pre, int& by,
                                       UnitRef& ur) {
    while (y >= ce) {
      if (x >= re) return false;
      u = unit_of(x, p, pre);
      const int x1 = min(u.uend, re), n = x1 - x;
      y = x + (w * n) / NWARP;
      ce = x + ((w + 1) * n) / NWARP;
      x = x1;
    }
    by = y++;
    ur = u;
    return true;
  }
};

__device__ __forceinline__ size_t unit_index(const AttendParams& p, const UnitRef& u) {
  return ((size_t)u.s * p.sh.L + p.layer_begin + u.l) * p.sh.Hkv + u.g;
}
// out / q offset of (unit u, query row `row` = j*G + hh).
__device__ __forceinline__ size_t row_offset(const AttendParams& p, const UnitRef& u, int row) {
  const int j = row / p.sh.G, hh = row % p.sh.G;
  const int h = u.g * p.sh.G + hh;
  return ((((size_t)u.l * p.sh.S + u.s) * p.c + j) * p.sh.Hq + h) * p.sh.D;
}

// Zero the outputs of units whose stream has an empty window (nothing to
// attend to).  CTAs stride over the units; threads t0 .. t0+nt-1 of the CTA
// share a unit's rows.
__device__ __forceinline__ void zero_empty_units(const AttendParams& p, int t, int nt) {
  const int per_stream = p.L_att * p.sh.Hkv;
  const int units = p.sh.S * per_stream;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int s = u / per_stream;
    const StreamState st = p.st[s];
    if (!(state_ok(st, p.sh) && st.fill == 0 && st.npin == 0)) continue;
    UnitRef ur;
    ur.s = s;
    ur.l = (u % per_stream) / p.sh.Hkv;
    ur.g = u % p.sh.Hkv;
    for (int row = 0; row < p.R; ++row) {
      float* o = p.out + row_offset(p, ur, row);
      for (int d = t; d < p.sh.D; d += nt) o[d] = 0.f;
    }
  }
}
__device__ __forceinline__ void zero_empty_units(const AttendParams& p) {
  zero_empty_units(p, threadIdx.x, blockDim.x);
}
// As zero_empty_units, from the cached stream data.
__device__ __forceinline__ void zero_empty_units_cached(const AttendParams& p, const int* sa,
                                                        const int* sfill, int t, int nt) {
  const int per_stream = p.L_att * p.sh.Hkv;
  const int units = p.sh.S * per_stream;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int s = u / per_stream;
    // A valid state, no pinned prefix, no retained pair.
    if (!(sa[s] >= 0 && (sa[s] >> 16) == 0 && sfill[s] == 0)) continue;
    UnitRef ur;
    ur.s = s;
    ur.l = (u % per_stream) / p.sh.Hkv;
    ur.g = u % p.sh.Hkv;
    for (int row = 0; row < p.R; ++row) {
      float* o = p.out + row_offset(p, ur, row);
      for (int d = t; d < p.sh.D; d += nt) o[d] = 0.f;
    }
  }
}

// The last CTA of a split unit combines the unit's np partials (m, l and the
// unnormalised O of each row, one slot per CTA segment) into its output:
//   out = sum_k w_k O_k,  w_k = 2^(m_k - M) / sum_j 2^(m_j - M) l_j,  M = max_k m_k.
// The np x R weights go to shared scratch `scr` first (one load of every m and
// l, all in flight together); then thread t of nt sums Q output elements at a
// time, eight partials per pass, so that 8 Q loads are in flight.  Every thread
// of the nt calls it; `sync` synchronises them.  Scratch of 2 np R + 2 R
// floats; with less, the weights are recomputed per element instead.  With
// `store` false nothing but the scratch is written (a dry run that brings the
// code into the instruction caches).
template <int Q, typename Sync>
__device__ __forceinline__ void merge_unit_partials(const AttendParams& p, const UnitRef& u,
                                                    int T, int P, int t, int nt, float* scr,
                                                    int scr_floats, Sync sync,
                                                    bool store = true) {
  const int R = p.R, D = p.sh.D, RD = R * D;
  const int b0 = cta_of(u.ustart, T, P), b1 = cta_of(u.uend - 1, T, P), np = b1 - b0 + 1;
  const int rs0 = range_start(b0, T, P);
  // CTA b0 holds the unit in its second slot when its range starts before it.
  const float* first =
      p.partials + (size_t)(2 * b0 + (rs0 < u.ustart ? 1 : 0)) * p.slot_floats;
  auto part = [&](int k) {
    return k == 0 ? first : p.partials + (size_t)(2 * (b0 + k)) * p.slot_floats;
  };
  if (2 * np * R + 2 * R <= scr_floats) {
    float* wm = scr;                 // [np][R]: m, then the weight
    float* wl = scr + np * R;        // [np][R]: l
    float* rowM = wl + np * R;       // [R]: M
    float* rowI = rowM + R;          // [R]: 1 / sum_j 2^(m_j - M) l_j
    for (int i = t; i < np * R; i += nt) {
      const int k = i / R, h = i - k * R;
      wm[i] = __ldcg(part(k) + h);
      wl[i] = __ldcg(part(k) + R + h);
    }
    sync();
    for (int h = t; h < R; h += nt) {
      float M = NEG_BIG;
      for (int k = 0; k < np; ++k) M = fmaxf(M, wm[k * R + h]);
      float den = 0.f;
      for (int k = 0; k < np; ++k) den += exp2f(wm[k * R + h] - M) * wl[k * R + h];
      rowM[h] = M;
      rowI[h] = den > 0.f ? 1.f / den : 0.f;
    }
    sync();
    for (int i = t; i < np * R; i += nt) {
      const int h = i % R;
      wm[i] = exp2f(wm[i] - rowM[h]) * rowI[h];
    }
    sync();
    for (int i0 = t; i0 < RD; i0 += Q * nt) {
      float acc[Q];
      int h[Q], e[Q];
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        e[q] = min(i0 + q * nt, RD - 1);
        h[q] = e[q] / D;
        acc[q] = 0.f;
      }
      for (int k0 = 0; k0 < np; k0 += 8) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int k = k0 + kk < np ? k0 + kk : np - 1;
          const float on = k0 + kk < np ? 1.f : 0.f;
          const float* pp = part(k) + 2 * R;
#pragma unroll
          for (int q = 0; q < Q; ++q) acc[q] += on * wm[k * R + h[q]] * __ldcg(pp + e[q]);
        }
      }
#pragma unroll
      for (int q = 0; q < Q; ++q)
        if (store && i0 + q * nt < RD)
          p.out[row_offset(p, u, h[q]) + (e[q] - h[q] * D)] = acc[q];
    }
    return;
  }
  for (int i0 = t; i0 < RD; i0 += Q * nt) {
    float M[Q], num[Q], den[Q];
    int h[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      h[q] = min(i0 + q * nt, RD - 1) / D;
      M[q] = NEG_BIG;
      num[q] = 0.f;
      den[q] = 0.f;
    }
#pragma unroll 4
    for (int k = 0; k < np; ++k) {
      const float* pp = part(k);
#pragma unroll
      for (int q = 0; q < Q; ++q) M[q] = fmaxf(M[q], __ldcg(pp + h[q]));
    }
#pragma unroll 2
    for (int k = 0; k < np; ++k) {
      const float* pp = part(k);
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        const int e = min(i0 + q * nt, RD - 1);
        const float w = exp2f(__ldcg(pp + h[q]) - M[q]);
        den[q] += w * __ldcg(pp + R + h[q]);
        num[q] += w * __ldcg(pp + 2 * R + e);
      }
    }
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const int e = i0 + q * nt;
      if (store && e < RD)
        p.out[row_offset(p, u, h[q]) + (e - h[q] * D)] = den[q] > 0.f ? num[q] / den[q] : 0.f;
    }
  }
}

// Segment end.  `mrg` holds NWARP warp partials of `wstride` floats, each
// [m(R) | l(R) | o(R*D)] with m in log2 units.  All CTA threads call this
// right after a __syncthreads.  Writes the unit's output when the segment is
// the whole unit; otherwise stores the CTA partial (slot 0 for the CTA's first
// segment, slot 1 for its last), takes the unit's ticket and, if it is the
// last CTA of the unit to arrive, merges every CTA partial of the unit.
// T = blocks in the call's list, P = CTAs sharing them (every CTA below P has
// at least one block); `flag` is one int of shared scratch.  The caller
// synchronises the CTA before reusing `mrg` or `flag`.
__device__ __forceinline__ void finish_segment(const AttendParams& p, const UnitRef& u, int x0,
                                               int x1, int rb, int T, int P, const float* mrg,
                                               int wstride, int* flag) {
  const int R = p.R, D = p.sh.D;
  const int nthr = blockDim.x;
  const bool whole = (x0 == u.ustart) && (x1 == u.uend);
  float* part = nullptr;
  if (!whole) {
    const int kslot = (x0 == rb) ? 0 : 1;
    part = p.partials + (size_t)(2 * blockIdx.x + kslot) * p.slot_floats;
  }
  for (int idx = threadIdx.x; idx < R * D; idx += nthr) {
    const int row = idx / D, d = idx % D;
    float M = NEG_BIG;
#pragma unroll
    for (int w = 0; w < NWARP; ++w) M = fmaxf(M, mrg[w * wstride + row]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < NWARP; ++w) {
      const float sc = exp2f(mrg[w * wstride + row] - M);
      den += sc * mrg[w * wstride + R + row];
      num += sc * mrg[w * wstride + 2 * R + row * D + d];
    }
    if (whole) {
      p.out[row_offset(p, u, row) + d] = den > 0.f ? num / den : 0.f;
    } else {
      if (d == 0) { part[row] = M; part[R + row] = den; }
      part[2 * R + row * D + d] = num;
    }
  }
  if (whole) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    *flag = atomicAdd(&p.unit_tickets[unit_index(p, u)], 1);
  }
  __syncthreads();
  const int b0 = cta_of(u.ustart, T, P), b1 = cta_of(u.uend - 1, T, P);
  if (*flag != b1 - b0) return;  // another CTA finishes this unit
  __threadfence();
  merge_unit_partials<16>(p, u, T, P, threadIdx.x, nthr, const_cast<float*>(mrg),
                          NWARP * wstride, [] { __syncthreads(); });
  if (threadIdx.x == 0) p.unit_tickets[unit_index(p, u)] = 0;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace rkv
