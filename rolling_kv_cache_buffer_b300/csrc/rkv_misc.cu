// rkv_misc.cu -- bookkeeping + append (K0/K1), stored-rotated re-rotation (K4)
// and the stream-state setter.
//
// Bookkeeping follows the flowchart of "Audio8 ASR Infinite: What It Actually
// Takes to Listen Forever": a pair that does not fit makes the cache evict the
// oldest pair and shift the sliding origin forward.
#include <type_traits>

#include "rkv_internal.h"
#include "rkv_rows.cuh"

namespace rkv {

namespace {

constexpr int APPEND_THREADS = 512;
constexpr int APPEND_BATCH = 8;   // 16-byte chunks a thread has in flight

}  // namespace

// ----------------------------------------------------------------------------
// K0 + K1: bookkeeping and scatter of the new rows.  grid = (parts, S): every
// thread reads the old state and derives the same new state from it, the
// parts of a stream scatter its rows, and the new state is published once the
// stream's rows are written: by the CTA itself when a stream has one part,
// else by the part that arrives last on the stream's ticket (no CTA waits on
// another).
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(APPEND_THREADS) append_kernel(const AppendParams p) {
  pdl_trigger();   // the attention launched next may start its prologue now
  const Shape& sh = p.sh;
  const int s = blockIdx.y;
  const int part = blockIdx.x, parts = gridDim.x;
  const StreamState st = p.st[s];
  const int c = p.c, W = sh.W, D = sh.D, Hkv = sh.Hkv;
  // Stored-rotated: re-based before this append (every eviction), or, with an
  // epoch E, lagging by fewer than E evictions.
  const bool rebased = !sh.stored_rotated || (sh.epoch ? st.pending < sh.epoch : st.pending == 0);
  // Evict just enough of the oldest pairs that at most Wr (the retained
  // window, <= the W slots) stay.
  const bool ok = state_ok(st, sh) && c >= 1 && c <= sh.Wr && rebased;
  const int e = max(0, st.fill + c - sh.Wr);
  // Keys are stored rotated to p - o_ref: o_ref = o2 (every eviction) or
  // o2 - lag2 (epoch), lag2 = the evictions since the last re-rotation.
  const int lag2 = sh.epoch ? st.pending + e : 0;
  const long long o2 = st.origin + e;
  const int n2 = st.fill + c - e;
  const long long first = st.origin + st.fill;
  const int rows = sh.L * c * Hkv;                    // rows (l, j, g)
  const bool bf = sh.bf16 != 0;
  // Row -> (l, j, g) with row = (l * c + j) * Hkv + g.
  auto split_row = [&](int row, int& l, int& j, int& g) {
    const int lj = static_cast<int>(p.div_hkv.div(row));
    g = row - lj * Hkv;
    l = static_cast<int>(p.div_c.div(lj));
    j = lj - l * c;
  };
  // New pair j goes to ring slot first_ring + j (mod W_ring), i.e. slot P +
  // that (P pinned slots in front of the ring); the state keeps origin mod
  // W_ring.
  const int Wg = sh.Wring;
  const int first_ring = st.ring + st.fill < Wg ? st.ring + st.fill : st.ring + st.fill - Wg;
  const int first_slot = sh.P + first_ring;
  // Stored-rotated keys: a pinned prefix of npin pairs sits at positions
  // 0..npin-1 in front of the retained ones.
  const int npin = st.npin;

  if (!sh.stored_rotated) {
    // Pre-RoPE: a plain copy of each row in 16-byte chunks.  Each thread loads
    // up to APPEND_BATCH chunks before storing any, so the loads of a pass
    // overlap instead of paying one memory round trip each.  The loads do not
    // depend on the state and go out while it is still on its way; only the
    // stores wait for it (and are skipped for a bad state).
    const int esz = bf ? 2 : 4;
    const int lch = __ffs(D * esz / 16) - 1;          // log2(16-byte chunks per row)
    const int all = (2 * rows) << lch;                // K rows, then V rows
    const int lo = static_cast<int>((long long)all * part / parts);
    const int total = static_cast<int>((long long)all * (part + 1) / parts);
    for (int base = lo; base < total; base += APPEND_BATCH * blockDim.x) {
      uint4 v[APPEND_BATCH];
      int rr[APPEND_BATCH];
#pragma unroll
      for (int t = 0; t < APPEND_BATCH; ++t) {
        const int idx = base + t * blockDim.x + threadIdx.x;
        rr[t] = -1;
        if (idx >= total) continue;
        rr[t] = idx;
        const int kvrow = idx >> lch, q = idx & ((1 << lch) - 1);
        const int kv = kvrow >= rows;
        int l, j, g;
        split_row(kvrow - kv * rows, l, j, g);
        const size_t src = ((((size_t)l * sh.S + s) * c + j) * Hkv + g) * D;
        const uint8_t* from = static_cast<const uint8_t*>(kv ? p.v_new : p.k_new) + src * esz;
        v[t] = __ldg(reinterpret_cast<const uint4*>(from) + q);
      }
#pragma unroll
      for (int t = 0; t < APPEND_BATCH; ++t) {
        if (!ok || rr[t] < 0) continue;
        const int kvrow = rr[t] >> lch, q = rr[t] & ((1 << lch) - 1);
        const int kv = kvrow >= rows;
        int l, j, g;
        split_row(kvrow - kv * rows, l, j, g);
        const int slot = sh.P + (first_ring + j < Wg ? first_ring + j : first_ring + j - Wg);
        const size_t dst = ((((size_t)s * sh.L + l) * Hkv + g) * W + slot) * D;
        uint8_t* to = static_cast<uint8_t*>(kv ? p.v_pool : p.k_pool) + dst * esz;
        reinterpret_cast<uint4*>(to)[q] = v[t];
      }
    }
  } else if (ok) {
    // Stored-rotated: keys are stored as R(p - o_ref) k, four pairs per step.
    const int quads = D / 8;
    const int lo = static_cast<int>((long long)rows * quads * part / parts);
    const int hi = static_cast<int>((long long)rows * quads * (part + 1) / parts);
    for (int idx = lo + threadIdx.x; idx < hi; idx += blockDim.x) {
      const int row = idx / quads;
      const int i = (idx % quads) * 4;
      int l, j, g;
      split_row(row, l, j, g);
      const long long pos = first + j;
      const int slot = sh.P + (first_ring + j < Wg ? first_ring + j : first_ring + j - Wg);
      const size_t src = ((((size_t)l * sh.S + s) * c + j) * Hkv + g) * D;
      const size_t dst = ((((size_t)s * sh.L + l) * Hkv + g) * W + slot) * D;
      float ka[4], kb[4], va[4], vb[4];
      load_pairs(p.k_new, src, i, D, sh.style, bf, ka, kb);
      load_pairs(p.v_new, src, i, D, sh.style, bf, va, vb);
      float2 cs[4];
      load_cs4(p.table, (size_t)(npin + pos - o2 + lag2) * (D / 2), i, cs);
      rotate4(ka, kb, cs, 1.f);
      store_pairs(p.k_pool, dst, i, D, sh.style, bf, ka, kb);
      store_pairs(p.v_pool, dst, i, D, sh.style, bf, va, vb);
    }
  }
  __syncthreads();
  bool publish = threadIdx.x == 0;
  if (publish && parts > 1) {
    __threadfence();
    publish = atomicAdd(&p.tickets[s], 1) == parts - 1;
    if (publish) {
      __threadfence();
      p.tickets[s] = 0;
    }
  }
  if (publish) {
    StreamState ns = st;
    if (ok) {
      ns.origin = o2;
      ns.fill = n2;
      ns.ring = st.ring + e < Wg ? st.ring + e : st.ring + e - Wg;
      ns.pending = sh.stored_rotated ? (sh.epoch ? lag2 : e) : 0;
      ns.last_new = c;
    } else if (ns.status == 0) {
      ns.status = STATUS_DEVICE_STATE;
    }
    p.st[s] = ns;
    if (p.log) {
      long long* lg = p.log + 4 * (size_t)s;
      lg[0] = ok ? o2 : st.origin;
      lg[1] = ok ? n2 : st.fill;
      lg[2] = ok ? e : -1;
      lg[3] = ok ? first_slot : -1;
    }
  }
}

// ----------------------------------------------------------------------------
// K4: stored-rotated re-base.  Every retained key older than the last append is
// turned by R(-e), e = pairs that append evicted, in f32 and rounded back to
// the storage type.  With an epoch E, a stream is re-based only once its lag
// (evictions since the last re-rotation) reaches E, and then every retained
// key, new ones included, turns by R(-lag).  grid = (CTAs per stream, S), at
// most one resident wave (3 CTAs per SM).  Work item = eight rotary pairs of
// one key (two 16-byte loads of bf16); the CTAs stride over the stream's
// items.  The stride is a multiple of a key's D/16 items, so a thread always
// turns the same eight pairs and loads their (cos, sin) once.  A stream with
// nothing due costs one state read per CTA.
// ----------------------------------------------------------------------------
// Eight consecutive pool elements as f32, from / to their raw 16-byte words
// (one for bf16, two for f32).
template <bool BF>
__device__ __forceinline__ void widen8(const uint4* w, float (&x)[8]) {
  if constexpr (BF) {
    x[0] = bf_lo(w[0].x); x[1] = bf_hi(w[0].x); x[2] = bf_lo(w[0].y); x[3] = bf_hi(w[0].y);
    x[4] = bf_lo(w[0].z); x[5] = bf_hi(w[0].z); x[6] = bf_lo(w[0].w); x[7] = bf_hi(w[0].w);
  } else {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      x[4 * k] = __uint_as_float(w[k].x); x[4 * k + 1] = __uint_as_float(w[k].y);
      x[4 * k + 2] = __uint_as_float(w[k].z); x[4 * k + 3] = __uint_as_float(w[k].w);
    }
  }
}
template <bool BF>
__device__ __forceinline__ void narrow8(const float (&x)[8], uint4* w) {
  if constexpr (BF) {
    w[0] = make_uint4(pack_bf2(x[0], x[1]), pack_bf2(x[2], x[3]), pack_bf2(x[4], x[5]),
                      pack_bf2(x[6], x[7]));
  } else {
#pragma unroll
    for (int k = 0; k < 2; ++k)
      w[k] = make_uint4(__float_as_uint(x[4 * k]), __float_as_uint(x[4 * k + 1]),
                        __float_as_uint(x[4 * k + 2]), __float_as_uint(x[4 * k + 3]));
  }
}
// (x, y) -> (x cos + y sin, y cos - x sin): the rotation by minus the angle.
__device__ __forceinline__ void unrotate(float& x, float& y, float2 cs) {
  const float c = cs.x, s = -cs.y;
  const float x0 = x, y0 = y;
  x = x0 * c - y0 * s;
  y = y0 * c + x0 * s;
}

template <bool BF>
__global__ void __launch_bounds__(256, 3) rerotate_kernel(const RerotParams p) {
  pdl_wait();      // the state and the pool come from the kernel launched before
  pdl_trigger();   // the attention launched next may start its prologue now
  const Shape& sh = p.sh;
  const int s = blockIdx.y;
  const StreamState st = p.st[s];
  const int W = sh.W, D = sh.D;
  const bool work = sh.stored_rotated && state_ok(st, sh) &&
                    (sh.epoch ? st.pending >= sh.epoch : st.pending > 0);
  // Every CTA of the stream reads the same state (it changes only after the
  // last CTA's ticket below), so either all take a ticket or none does.
  if (!work) return;
  // Keys that predate the append (every eviction), or all of them (epoch).
  const int nr = max(sh.epoch ? st.fill : st.fill - st.last_new, 0);
  const int cshift = D == 128 ? 3 : 2;             // log2 of D / 16 items per key
  const int per_lg = nr << cshift;                 // items per (layer, KV head)
  const int LH = sh.L * sh.Hkv;
  const int stride = gridDim.x * blockDim.x;       // a multiple of D / 16
  const int t0 = blockIdx.x * blockDim.x + threadIdx.x;
  const int i = (t0 & ((1 << cshift) - 1)) * 8;    // the thread's first pair
  float2 cs[8];
  {
    const float4* t = reinterpret_cast<const float4*>(p.table + (size_t)st.pending * (D / 2) + i);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 v = __ldg(t + k);
      cs[2 * k] = make_float2(v.x, v.y);
      cs[2 * k + 1] = make_float2(v.z, v.w);
    }
  }
  // Element offsets (within a key) of the item's two groups of eight: the
  // pairs' first and second halves (split-half) or 16 consecutive elements.
  const int e0 = sh.style == 0 ? i : 2 * i, e1 = sh.style == 0 ? D / 2 + i : 2 * i + 8;
  constexpr int NW = BF ? 1 : 2;                   // 16-byte words per group
  using Elem = typename std::conditional<BF, uint16_t, float>::type;
  Elem* pool = static_cast<Elem*>(p.k_pool);
  // (layer * H_kv + head, item within it) of the thread's next item, advanced
  // by the stride without a division per item.
  int lg = per_lg ? t0 / per_lg : LH, rem = per_lg ? t0 - lg * per_lg : 0;
  const int dq = per_lg ? stride / per_lg : 0, dr = per_lg ? stride - dq * per_lg : 0;
  const size_t sbase = (size_t)s * LH * W;
  constexpr int NB = BF ? 4 : 2;   // items per thread in flight: all loads, then all stores
  while (lg < LH) {
    uint4 w[NB][2][NW];
    Elem* row[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      row[j] = nullptr;
      if (lg < LH) {
        // Retained pair r (oldest first) of the ring behind the P pinned
        // slots; a pinned prefix keeps its positions and is never turned.
        const int r = rem >> cshift;
        const int slot = sh.P + (st.ring + r < sh.Wring ? st.ring + r : st.ring + r - sh.Wring);
        row[j] = pool + (sbase + (size_t)lg * W + slot) * D;
#pragma unroll
        for (int k = 0; k < NW; ++k) {
          w[j][0][k] = reinterpret_cast<const uint4*>(row[j] + e0)[k];
          w[j][1][k] = reinterpret_cast<const uint4*>(row[j] + e1)[k];
        }
      }
      lg += dq;
      rem += dr;
      if (rem >= per_lg) { rem -= per_lg; ++lg; }
    }
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      if (!row[j]) continue;
      float u[8], v[8];
      widen8<BF>(w[j][0], u);
      widen8<BF>(w[j][1], v);
      if (sh.style == 0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) unrotate(u[k], v[k], cs[k]);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          unrotate(u[2 * k], u[2 * k + 1], cs[k]);
          unrotate(v[2 * k], v[2 * k + 1], cs[4 + k]);
        }
      }
      narrow8<BF>(u, w[j][0]);
      narrow8<BF>(v, w[j][1]);
#pragma unroll
      for (int k = 0; k < NW; ++k) {
        reinterpret_cast<uint4*>(row[j] + e0)[k] = w[j][0][k];
        reinterpret_cast<uint4*>(row[j] + e1)[k] = w[j][1][k];
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int old = atomicAdd(&p.tickets[s], 1);
    if (old == static_cast<int>(gridDim.x) - 1) {
      p.st[s].pending = 0;
      p.tickets[s] = 0;
    }
  }
}

__global__ void set_state_kernel(StreamState* st, int s, long long origin, int fill, int ring) {
  StreamState ns{};
  ns.origin = origin;
  ns.fill = fill;
  ns.ring = ring;
  st[s] = ns;
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t s) {
  // One CTA per stream unless a stream's rows need several batched passes.
  const int esz = p.sh.bf16 ? 2 : 4;
  const long long items = 2LL * p.sh.L * p.c * p.sh.Hkv * (p.sh.D * esz / 16);
  long long parts = (items + APPEND_THREADS * APPEND_BATCH - 1) / (APPEND_THREADS * APPEND_BATCH);
  parts = parts < 1 ? 1 : (parts > 64 ? 64 : parts);
  append_kernel<<<dim3((unsigned)parts, p.sh.S), APPEND_THREADS, 0, s>>>(p);
  return cudaGetLastError();
}
cudaError_t launch_rerotate(const RerotParams& p, int blocks_per_stream, cudaStream_t s) {
  // Programmatic dependent launch: the launch overlaps the previous kernel's
  // tail; the kernel waits for it before reading anything.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks_per_stream, p.sh.S);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return p.sh.bf16 ? cudaLaunchKernelEx(&cfg, rerotate_kernel<true>, p)
                   : cudaLaunchKernelEx(&cfg, rerotate_kernel<false>, p);
}
cudaError_t launch_set_state(StreamState* st, int s_idx, long long origin, int fill, int ring,
                             cudaStream_t s) {
  set_state_kernel<<<1, 1, 0, s>>>(st, s_idx, origin, fill, ring);
  return cudaGetLastError();
}

}  // namespace rkv
