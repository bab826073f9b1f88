// rkv_attend_mma.cu -- tensor-core decode attention over the rolling window
// (bf16 caches, one query token per stream, G = H_q/H_kv <= 8, D 64 or 128).
//
// What it computes is the attention over the window with exact re-basing of
// "Audio8 ASR Infinite: What It Actually Takes to Listen Forever" ("Inside the
// Rolling KV Cache and Exact RoPE Re-Basing"): for the query at r_q = fill - 1
// and every retained key at r = (slot - origin) mod W,
//   out = sum_r softmax(<R(r_q) q, R(r) k_r> * scale) v_r.
//
// Arithmetic.  The G query heads that share a KV head make S = Q K^T a dense
// contraction with M = G rows, and O^T = V^T P^T one with N = G columns, so
// both run on mma.sync m16n8k16 (bf16 operands, f32 accumulation):
//  * a block of TK = 32 slots starts at slot blk*TK, whose first slot sits at
//    re-based position r0; slot d of the block is at r0 + d, or r0 + d - W
//    past the ring's end;
//  * keys are rotated in f32 by R(d) only (d < 32, a shared-memory table) and
//    rounded to bf16; the block offset goes into the query instead:
//    rows 0..7 of the A operand hold R(r_q - r0) q and, in the one block of a
//    unit that holds the ring's end, rows 8..15 hold R(r_q - r0 + W) q, so
//    each key picks the row of its own base (<R(a) q, R(b) k> depends only on
//    b - a);
//  * the S accumulator fragment is exactly the B fragment P^T of the second
//    product, so probabilities never leave registers.
// Stored-rotated keys skip the key rotation and use R(r_q + lag) q alone (lag
// = 0 unless the keys follow a re-basing epoch).
//
// Pipeline (one persistent CTA per SM).  Warp 0 is the producer: one lane
// walks the CTA's share of the block list and streams every block's K and V
// tiles (one 4-D TMA box per tile, 128-byte swizzle) plus the (cos, sin) rows
// of the block's query rotations into a ring of NS shared-memory stages
// (full/empty mbarriers).  Warps 1..NCW are consumers in NCW/2 pairs: block j
// of the CTA's share goes to pair j mod (NCW/2), each warp of the pair takes
// 16 of the block's 32 keys and keeps an online-softmax state per unit
// segment.  At the end of a segment every warp writes its state to a slot
// that aliases the stage memory and the consumers combine the slots; the
// producer waits for that merge before it reuses the stages.  A unit split
// across CTAs is finished either by the CTA that arrives last on the unit's
// ticket (global partials), or, when the grid is exactly two CTAs per unit,
// by rank 0 of a 2-CTA cluster, into whose shared memory the warps of rank 1
// write their slots.  No CTA ever waits on a CTA that may not be resident.
//
// Fused step (FUSED): the same kernel also appends one pair per stream -- the
// geometry after the append comes from the old state, a prepass writes the
// new rows, the CTA that finishes a unit adds the new pair from the inputs,
// and the step's last launch publishes the new states.
#include <climits>
#include <type_traits>

#include "rkv_attend_pipe.cuh"
#include "rkv_rows.cuh"

#ifndef RKV_MMA_NCW
#define RKV_MMA_NCW 10
#endif

namespace rkv {

namespace {

constexpr int NCW = RKV_MMA_NCW;              // consumer warps
constexpr int CONS_THREADS = NCW * 32;
// Threads of a CTA: the producer warp, the consumer warps and, in a fused
// step, one side warp that writes the step's new pairs and publishes the new
// stream states (off the consumers' path to their first block).
template <bool FUSED>
constexpr int mma_threads() { return (1 + NCW + (FUSED ? 1 : 0)) * 32; }
constexpr int MMA_MAX_STAGES = 16;
constexpr int BAR_CONS = 1;                   // named barrier of the consumer warps
constexpr int BAR_PREFIX = 2;                 // the producer warp's block prefix is ready
constexpr int BAR_SIDE = 3;                   // the side warp's own barrier in its dry pass

constexpr int TKH = TK / 2;     // keys of a block each warp of a pair takes
constexpr int NPAIR = NCW / 2;  // consumer warp pairs
// Fewest blocks in a CTA's share for the dry run of the merge to pay off.
constexpr int DRY_MIN_BLOCKS = 32;
static_assert(NCW % 2 == 0, "consumer warps come in pairs");

template <int D, bool ROTK>
struct MmaCfg : PipeCfg<D, ROTK> {
  using PipeCfg<D, ROTK>::FINE;
  static constexpr int NGRP = D / 8;                      // 8-dim groups
  static constexpr int NKB = D / 16;                      // k-blocks of the QK product
  static constexpr int HG = NGRP / 2;
  static constexpr int QSTR = D + 8;                      // padded query row (floats)
  static constexpr int FR = 4 * NKB;                      // O^T fragment floats per lane
  // Warp partial: m[8], l[8], then the O^T fragment element-major: element i
  // of lane t at 16 + 32 i + t (every access pattern below is conflict-free).
  static constexpr int SLOT = 16 + 32 * FR;
  // Bytes after the stages (the warp slots of a segment merge alias the
  // stages), without the per-stream prefix: R(d) table, query rows, flags and
  // the merge-done barrier.
  // Query-base rows (cos, sin) of every consumer warp's current block and of
  // its wrap base, and the two constant steps R(-NPAIR*TK) and R(W).
  static constexpr int QROWS = ROTK ? (2 * NCW + 2) * (D / 2) * 8 : 0;
  static constexpr int FIXED =
      FINE + QROWS + 8 * QSTR * 4 + 10 * D * 4 + 16 + 16 + 32 + 2 * D * 4;
};

// `rx`: bytes of the cluster receive area (0 without cluster merge).
__host__ __device__ constexpr size_t mma_smem_bytes(int stage, int fixed, int ns, int S,
                                                    int rx = 0) {
  return 1024 + (size_t)ns * stage + (size_t)fixed + (size_t)ns * 16 + (size_t)(4 * S + 1) * 4 +
         (rx ? 16 + 16 + (size_t)rx : 0);
}
// Cluster merge: rank 0 receives rank 1's partial, already combined over its
// warps: per consumer thread, m and l of its head and its 4 (D/16) / NCW
// output elements (see the segment end), stored element-major.
template <int D>
constexpr int rx_per_thread() { return 2 + (4 * (D / 16) + NCW - 1) / NCW; }
template <int D>
constexpr int rx_floats() { return rx_per_thread<D>() * CONS_THREADS; }

__device__ __forceinline__ void rot(float& x, float& y, float c, float s) {
  const float a = x * c - y * s;
  y = y * c + x * s;
  x = a;
}

// Packed f32 pairs (the sm_100+ f32x2 pipe).
typedef unsigned long long f2;
__device__ __forceinline__ f2 f2_make(float a, float b) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_split(f2 v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
  f2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// Two split-half pairs held as bf16x2 words: x = dims (i, i+1), y = their
// partners (i+D/2, i+D/2+1).  Rotated in f32 by (cos, sin) = (c, s) per pair:
// x' = x c - y s, y' = y c + x s, then rounded to nearest even.
__device__ __forceinline__ void rot_pair2(uint32_t& x, uint32_t& y, float4 cs) {
  const f2 X = f2_make(bf_lo(x), bf_hi(x));
  const f2 Y = f2_make(bf_lo(y), bf_hi(y));
  const f2 C = f2_make(cs.x, cs.y), S = f2_make(cs.z, cs.w), NS = f2_make(-cs.z, -cs.w);
  const f2 Xr = f2_fma(Y, NS, f2_mul(X, C));
  const f2 Yr = f2_fma(X, S, f2_mul(Y, C));
  float a, b, c, d;
  f2_split(Xr, a, b);
  f2_split(Yr, c, d);
  x = pack_bf2(a, b);
  y = pack_bf2(c, d);
}

}  // namespace

// Fused decode step: what rkv_append of one pair would leave in a stream's
// state, from the state the step starts from (the bookkeeping of the append
// kernel: e = max(0, n + 1 - Wr), o' = o + e, n' = n + 1 - e; stored-rotated
// keys with a re-basing epoch E also carry their lag, which must be below E
// before the append and grows by e).
struct StepState {
  bool ok;
  int e, n2, ring2;   // evictions, fill and origin mod W_ring after the append
  int new_slot;       // slot of the new pair (behind the P pinned slots)
  int lag2;           // lag after the append (epoch), else 0
};
__device__ __forceinline__ StepState step_state(const StreamState& st, const Shape& sh) {
  const int Wg = sh.Wring;
  StepState r;
  r.ok = state_ok(st, sh) && (!sh.stored_rotated || (sh.epoch && st.pending < sh.epoch));
  r.e = max(0, st.fill + 1 - sh.Wr);
  r.n2 = st.fill + 1 - r.e;
  r.ring2 = st.ring + r.e < Wg ? st.ring + r.e : st.ring + r.e - Wg;
  r.new_slot = sh.P + (st.ring + st.fill < Wg ? st.ring + st.fill : st.ring + st.fill - Wg);
  r.lag2 = sh.epoch ? st.pending + r.e : 0;
  return r;
}

// Block prefix of a fused step: every stream's window after the append minus
// its new pair (the kernels read the new pair from the step's inputs, not from
// the pool), i.e. ring start ring', n' - 1 pairs; the query sits at n' - 1.
__device__ __forceinline__ void build_prefix_step(const AttendParams& p, int* pre, int* sa,
                                                  int* sfill, int* slag, int lane) {
  const int per_unit = p.L_att * p.sh.Hkv;
  int carry = 0;
  if (lane == 0) pre[0] = 0;
  for (int base = 0; base < p.sh.S; base += 32) {
    const int s = base + lane;
    int v = 0;
    if (s < p.sh.S) {
      const StreamState st = p.st[s];
      const StepState ss = step_state(st, p.sh);
      sa[s] = ss.ok ? pack_an(ss.ring2, st.npin) : -1;
      sfill[s] = ss.ok ? ss.n2 - 1 : 0;
      slag[s] = ss.ok ? ss.lag2 : 0;
      v = ss.ok ? unit_blocks(ss.ring2, ss.n2 - 1, st.npin, p.sh.NBr) * per_unit : 0;
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

// Fused step, every unit once (CTAs stride over the units, one warp per
// unit): the new pair goes into its slot in the pools (this step's attention
// takes it from the inputs and never reads that slot), and a unit whose window
// holds only the new pair gets v_new as its output.  Reads the post-append
// geometry from the CTA's cache (sa = ring start after the append with the
// pinned prefix pairs, or -1 for a bad state; sfill = fill after the append
// minus the new pair), so the new pair's slot is P + (a + sfill) mod W_ring.
// STORED: stored-rotated keys (with a re-basing epoch), whose new key goes in
// rotated.
template <int D, bool STORED>
__device__ __forceinline__ void step_prepass(const AttendParams& p, const int* sa,
                                             const int* sfill, const int* slag, int w, int nw,
                                             int lane) {
  const int per_stream = p.L_att * p.sh.Hkv;
  const int units = p.sh.S * per_stream;
  const int esz = p.sh.bf16 ? 2 : 4;
  const int t = lane, nt = 32;   // one warp per unit
  for (int u = blockIdx.x + gridDim.x * w; u < units; u += gridDim.x * nw) {
    const int s = u / per_stream;
    if (sa[s] < 0) continue;
    const int a = sa[s] & 0xffff, npin = sa[s] >> 16;
    int new_slot = a + sfill[s];
    if (new_slot >= p.sh.Wring) new_slot -= p.sh.Wring;
    new_slot += p.sh.P;
    const int l = (u % per_stream) / p.sh.Hkv, g = u % p.sh.Hkv;
    const size_t src = (((size_t)l * p.sh.S + s) * p.sh.Hkv + g) * D;
    const size_t dst =
        ((((size_t)s * p.sh.L + p.layer_begin + l) * p.sh.Hkv + g) * p.sh.W + new_slot) * D;
    const int chunks = D * esz / 16;
    if constexpr (STORED) {
      // Stored-rotated keys (with an epoch): the new key goes in rotated to
      // its position from o_ref, n' - 1 + lag', four pairs per lane.
      const size_t trow = (size_t)(npin + sfill[s] + slag[s]) * (D / 2);
      for (int i = t; i < D / 8; i += nt) {
        float ka[4], kb[4];
        float2 cs[4];
        load_pairs(p.k_new, src, 4 * i, D, p.sh.style, p.sh.bf16 != 0, ka, kb);
        load_cs4(p.table, trow, 4 * i, cs);
        rotate4(ka, kb, cs, 1.f);
        store_pairs(p.k_pool, dst, 4 * i, D, p.sh.style, p.sh.bf16 != 0, ka, kb);
      }
    }
    for (int i = t; i < 2 * chunks; i += nt) {
      const int kv = i >= chunks, q = i - kv * chunks;
      if (STORED && !kv) continue;   // rotated above
      const uint4* from = reinterpret_cast<const uint4*>(
          static_cast<const uint8_t*>(kv ? p.v_new : p.k_new) + src * esz) + q;
      uint4* to = reinterpret_cast<uint4*>(
          static_cast<uint8_t*>(kv ? p.v_pool : p.k_pool) + dst * esz) + q;
      *to = *from;
    }
    if (sfill[s] == 0 && npin == 0) {   // only the new pair: softmax over one key gives v_new
      UnitRef ur;
      ur.s = s; ur.l = l; ur.g = g;
      for (int i = t; i < p.sh.G * D; i += nt) {
        const int h = i / D, d = i % D;
        p.out[row_offset(p, ur, h) + d] = load_elem(p.v_new, src + d, p.sh.bf16);
      }
    }
  }
}

// The fused step's publish: every CTA reads the old states in its prologue and
// keeps what it needs in shared memory; once all have, the last CTA past this
// point writes the new ones (the append's bookkeeping), one stream per lane of
// the calling warp, on the step's last launch only.
__device__ __forceinline__ void step_publish(const AttendParams& p, int lane) {
  int last = 0;
  if (lane == 0) {
    __threadfence();
    last = atomicAdd(p.step_ticket, 1) == static_cast<int>(gridDim.x) - 1;
    if (last) __threadfence();
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  for (int s2 = lane; s2 < p.sh.S; s2 += 32) {
    const StreamState st = p.st[s2];
    const StepState ss = step_state(st, p.sh);
    StreamState ns = st;
    if (ss.ok) {
      ns.origin = st.origin + ss.e;
      ns.fill = ss.n2;
      ns.ring = ss.ring2;
      ns.pending = ss.lag2;
      ns.last_new = 1;
    } else if (ns.status == 0) {
      ns.status = STATUS_DEVICE_STATE;
    }
    p.st[s2] = ns;
    if (p.log) {
      long long* lg = p.log + 4 * (size_t)s2;
      lg[0] = ss.ok ? ns.origin : st.origin;
      lg[1] = ss.ok ? ns.fill : st.fill;
      lg[2] = ss.ok ? ss.e : -1;
      lg[3] = ss.ok ? ss.new_slot : -1;
    }
  }
  if (lane == 0) *p.step_ticket = 0;
}

template <int D, bool ROTK, int STYLE, bool FUSED, bool CL>
__global__ void __launch_bounds__(mma_threads<FUSED>(), 1)
    attend_mma_decode(const __grid_constant__ AttendParams p,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV) {
  using C = MmaCfg<D, ROTK>;
  constexpr int TILE = C::TILE, NGRP = C::NGRP, NKB = C::NKB, HALF = C::HALF, HG = C::HG;
  constexpr int QSTR = C::QSTR;
  const int G = p.sh.G, NS = p.ns;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  uint8_t* stages = smem;                                          // [NS][STAGE]
  float* slots = reinterpret_cast<float*>(smem);                   // [NCW][SLOT], between segments
  uint8_t* fine = stages + (size_t)NS * C::STAGE;                  // [TK][D/2] (cos, sin)
  float2* qrow = reinterpret_cast<float2*>(fine + C::FINE);        // [NCW][D/2] R(r_q - r0)
  float2* wrow = qrow + NCW * (D / 2);                             // [NCW][D/2] R(r_q - r0 + W)
  float2* srow = wrow + NCW * (D / 2);                             // [D/2] R(-NPAIR*TK)
  float2* Wrow = srow + D / 2;                                     // [D/2] R(W)
  float* qs = reinterpret_cast<float*>(fine + C::FINE + C::QROWS);  // [8][QSTR] raw query
  uint8_t* qraw = reinterpret_cast<uint8_t*>(qs + 8 * QSTR);       // [8][D] query, as stored
  uint8_t* nraw = qraw + 8 * D * 4;                                // [2][D] new pair, as stored
  int* flag = reinterpret_cast<int*>(nraw + 2 * D * 4);            // ticket, abort, issued
  uint64_t* mdone = reinterpret_cast<uint64_t*>(flag + 4);         // segment merged
  float* mx = reinterpret_cast<float*>(mdone + 2);                 // [8] new-key scores
  float* kvn = mx + 8;                                             // [2][D] new pair (fused)
  uint64_t* full = reinterpret_cast<uint64_t*>(kvn + 2 * D);       // [NS]
  uint64_t* empty = full + NS;                                     // [NS]
  int* pre = reinterpret_cast<int*>(empty + NS);                   // [S+1] block prefix
  int* sa = pre + p.sh.S + 1;                                      // [S] origin mod W
  int* sfill = sa + p.sh.S;                                        // [S] fill
  int* slag = sfill + p.sh.S;                                      // [S] lag (epoch)
  // Cluster merge (CL): the pair of CTAs that shares a unit meets here.
  uint64_t* rx_bar = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(slag + p.sh.S) + 15) & ~uintptr_t(15));
  float* rslots = reinterpret_cast<float*>(rx_bar + 2);            // rank 1's partial
  volatile int* abort_flag = flag + 1;

  constexpr int NTHR = mma_threads<FUSED>();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // The producer's first read after the dependency wait is the stream state:
  // bring it into L2 before anything else.
  prefetch_states(p);
  // Prologue that reads nothing the previous kernel of the stream writes: the
  // barriers and the R(d) table (written once when the handle was created).
  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(full + i), 1);
      mbar_init(smem_u32(empty + i), 2);   // both warps of the pair that takes the block
    }
    mbar_init(smem_u32(mdone), 1);
    if constexpr (CL) {
      // Completes once rank 1's partials (rx_floats() floats) have landed.
      mbar_init(smem_u32(rx_bar), 1);
      mbar_arrive_expect_tx(smem_u32(rx_bar), rx_floats<D>() * 4);
    }
    fence_mbar_init();
    flag[1] = 0;
    flag[2] = 0;
  }
  if constexpr (ROTK) {
    if (warp > 0 && warp <= NCW) {
      load_fine<D, STYLE>(p, fine, tid - 32, CONS_THREADS);
      // The constant steps of the query bases: R(-NPAIR*TK), the NPAIR-th
      // power of table row TK with its sine negated (rows stop below 2W, and
      // TK < 2W always), and R(W_ring) (row W_ring).
      for (int i = tid - 32; i < 2 * HALF; i += CONS_THREADS) {
        const int k = i % HALF;
        if (i < HALF) {
          const float2 c = __ldg(p.table + (size_t)TK * HALF + k);
          float2 a = c;
          for (int r = 1; r < NPAIR; ++r)
            a = make_float2(a.x * c.x - a.y * c.y, a.x * c.y + a.y * c.x);
          srow[k] = make_float2(a.x, -a.y);
        } else {
          Wrow[k] = __ldg(p.table + (size_t)p.sh.Wring * HALF + k);
        }
      }
    }
  }
  // The other warps bring this CTA's share of the queries (and of the step's
  // new pairs, which no earlier kernel of the step writes) into L2; warp 0
  // goes on to the stream state and its first copies.
  if (warp > 0) {
    prefetch_queries(p, D, tid - 32, NTHR - 32);
    if constexpr (FUSED) {
      const size_t nbytes = (size_t)p.L_att * p.sh.S * p.sh.Hkv * D * (p.sh.bf16 ? 2 : 4);
      const size_t lines = (nbytes + 127) / 128;
      const size_t l0 = lines * blockIdx.x / gridDim.x;
      const size_t l1 = lines * (blockIdx.x + 1) / gridDim.x;
      for (size_t l = l0 + tid - 32; l < l1; l += NTHR - 32) {
        prefetch_l2(static_cast<const uint8_t*>(p.k_new) + l * 128);
        prefetch_l2(static_cast<const uint8_t*>(p.v_new) + l * 128);
      }
    }
  }
  // Cluster merge: the partner's barrier must exist before this CTA touches
  // it; every thread arrives here and waits once it has work under way.
  if constexpr (CL) cluster_arrive_relaxed();
  pdl_wait();   // from here on: stream state, pools, queries, outputs
  pdl_trigger();   // a kernel launched next may start its own prologue
  // Warp 0 builds the block prefix and starts streaming at once; the
  // consumers pick the prefix up from the named barrier.
  if (warp == 0) {
    if constexpr (FUSED)
      build_prefix_step(p, pre, sa, sfill, slag, lane);
    else
      build_prefix_cached(p, pre, sa, sfill, lane, slag);
    __syncwarp();
    named_bar_arrive(BAR_PREFIX, NTHR);
  } else {
    named_bar_sync(BAR_PREFIX, NTHR);
  }
  const int T = pre[p.sh.S];
  const int P = min(static_cast<int>(gridDim.x), T);
  const int b = static_cast<int>(blockIdx.x);
  const int rb = b < P ? range_start(b, T, P) : 0, re = b < P ? range_start(b + 1, T, P) : 0;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0)
      flag[2] = produce<D, ROTK, NO_ROWS>(p, &tmK, &tmV, stages, full, empty, mdone, pre, sa,
                                          sfill, rb, re, abort_flag);
    __syncwarp();
    if constexpr (CL) cluster_wait();
  } else {
    // ------------------------------------------------------------------ consumers
    // In a fused step the side warp (warp NCW + 1) runs this code too, as a
    // dry pass only: one block body and the segment end, with nothing written
    // but its own scratch and its own barrier instead of the consumers' --
    // so that the consumers find that code in the instruction caches and need
    // no dry pass of their own -- and then does its own work (below).
    const bool side = FUSED && warp == NCW + 1;
    const int cw = warp - 1, ct = tid - 32;
    auto cbar = [&]() {
      named_bar_sync(side ? BAR_SIDE : BAR_CONS, side ? 32 : CONS_THREADS);
    };
    const int g = lane >> 2, cq = lane & 3;   // mma fragment coordinates
    // A unit's query rows (and, in a fused step, its new pair) reach shared
    // memory in two steps: `stage_unit` issues 16-byte asynchronous copies of the
    // rows as stored, `unstage_*` converts the chunks this thread copied to
    // f32 (`qs` rows >= G stay zero; `kvn` = [k_new | v_new]).
    const int qesz = p.sh.q_bf16 ? 2 : 4, kesz = p.sh.bf16 ? 2 : 4;
    const int qcpr = D * qesz / 16, kcpr = D * kesz / 16;   // 16-byte chunks per row
    auto stage_unit = [&](const UnitRef& un) {
      for (int i = ct; i < G * qcpr; i += CONS_THREADS) {
        const int h = i / qcpr, c = i - h * qcpr;
        cp_async16(smem_u32(qraw + (size_t)i * 16),
                   static_cast<const uint8_t*>(p.q) + row_offset(p, un, h) * qesz + c * 16);
      }
      if constexpr (FUSED) {
        const size_t r = (((size_t)un.l * p.sh.S + un.s) * p.sh.Hkv + un.g) * D;
        for (int i = ct; i < 2 * kcpr; i += CONS_THREADS) {
          const int kv = i >= kcpr, c = i - kv * kcpr;
          cp_async16(smem_u32(nraw + (size_t)i * 16),
                     static_cast<const uint8_t*>(kv ? p.v_new : p.k_new) + r * kesz + c * 16);
        }
      }
      cp_async_commit();
    };
    auto widen = [](const uint8_t* src, float* dst, bool bf) {
      const uint4 v = *reinterpret_cast<const uint4*>(src);
      if (bf) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          dst[2 * k] = bf_lo(w[k]);
          dst[2 * k + 1] = bf_hi(w[k]);
        }
      } else {
        dst[0] = __uint_as_float(v.x);
        dst[1] = __uint_as_float(v.y);
        dst[2] = __uint_as_float(v.z);
        dst[3] = __uint_as_float(v.w);
      }
    };
    auto unstage_q = [&]() {   // waits for this thread's copies
      cp_async_wait_all();
      for (int i = ct; i < G * qcpr; i += CONS_THREADS) {
        const int h = i / qcpr, c = i - h * qcpr;
        widen(qraw + (size_t)i * 16, qs + h * QSTR + c * (16 / qesz), p.sh.q_bf16);
      }
    };
    auto unstage_new = [&]() {   // after unstage_q
      for (int i = ct; i < 2 * kcpr; i += CONS_THREADS) {
        const int kv = i >= kcpr, c = i - kv * kcpr;
        widen(nraw + (size_t)i * 16, kvn + kv * D + c * (16 / kesz), p.sh.bf16);
      }
    };
    if (!side) {
      for (int i = ct; i < (8 - G) * D; i += CONS_THREADS)
        qs[(G + i / D) * QSTR + i % D] = 0.f;
      if (rb < re) stage_unit(unit_of_cached(rb, p, pre, sa, sfill));
      if constexpr (!FUSED) zero_empty_units_cached(p, sa, sfill, ct, CONS_THREADS);
      if (rb < re) {
        unstage_q();
        if constexpr (FUSED) unstage_new();
      }
    }
    cbar();
    if constexpr (CL) cluster_wait();   // long after both CTAs arrived
    // Dims of the thread's A-fragment elements: k-block kb, j in {0,1,2,3}:
    //   dim 16kb + (j>>1)*8 + 2cq + (j&1)
    auto qdim = [&](int kb, int j) { return 16 * kb + (j >> 1) * 8 + 2 * cq + (j & 1); };

    // Warp pair pi takes blocks pi, pi + NPAIR, ...; warp hh of the pair takes
    // keys 16*hh .. 16*hh+15 of each.
    const int pi = cw >> 1, hh = cw & 1;
    int jb = pi, stage = side ? 0 : pi, round = 0;   // the pair's next block and its stage (NS >= NPAIR)
    bool dead = false;
    // The first pass through the loop is a dry run of the segment end: no
    // block, nothing written (neither the slots, which alias the stages the
    // producer is filling, nor outputs, partials, tickets, the partner CTA or
    // the merge-done barrier), while the first tiles are still on their way.
    // It brings the merge's code into the instruction caches, so that the
    // real merge at the end of the stream does not fetch it from memory.  A
    // short share (a launch over one layer) has no time to hide it: there the
    // merge code is fetched when it runs.  In a fused step the side warp
    // makes this pass instead of the consumers.
    bool dry = FUSED ? side && rb < re : re - rb >= DRY_MIN_BLOCKS;
#pragma unroll 1
    for (int x = rb; x < re;) {
      const UnitRef u = unit_of_cached(x, p, pre, sa, sfill);
      const int x1 = min(u.uend, re);
      // The query's re-based position, behind the pinned prefix's npin pairs.
      const int rq = u.npin + u.fill - 1 + (FUSED ? 1 : 0);
      // The next segment's query (and new pair): copied now, converted once
      // this segment is done with `qs` (and `kvn`).
      const bool has_next = x1 < re;
      if (has_next && !dry) stage_unit(unit_of_cached(x1, p, pre, sa, sfill));
      // The CTA that finishes the unit adds the fused step's new pair.  It sits
      // at the query's own position, so its score is <q, k_new> (the rotations
      // cancel); warp h scores head h -- for the CTA's first segment here,
      // while the first tiles are on their way (q and k_new are in shared
      // memory since the barrier above), for a later one at its end.
      const bool add_new = FUSED && (CL ? x == u.ustart : x1 == u.uend);
      auto score_new = [&]() {
        if (add_new && cw < G) {
          float dot = 0.f;
          for (int d = lane; d < D; d += 32) dot += qs[cw * QSTR + d] * kvn[d];
          dot = warp_sum(dot);
          if (lane == 0) mx[cw] = dot * p.scale_log2;
        }
      };
      if (FUSED && !side && x == rb) score_new();

      // The raw query of head g (dims of the thread's A fragments), from `qs`.
      auto load_qf = [&](float (&qr)[NKB][4]) {
#pragma unroll
        for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
          for (int j = 0; j < 4; j += 2) {
            const float2 v = *reinterpret_cast<const float2*>(qs + g * QSTR + qdim(kb, j));
            qr[kb][j] = v.x;
            qr[kb][j + 1] = v.y;
          }
      };
      uint32_t qa[NKB][4];             // A fragments of the QK product
      float o[NKB][4];                 // O^T accumulators: m-tile = 16 dims
      float m_run = NEG_BIG, l_run = 0.f;
#pragma unroll
      for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          o[kb][j] = 0.f;
          qa[kb][j] = 0u;
        }
      if (!ROTK && !dry) {
        // Stored-rotated keys sit at r (+ the stream's lag, with a re-basing
        // epoch) already: one base, R(r_q + lag) q.
        const int lag = slag[u.s];
        const float2* t = p.table + (size_t)(rq + lag) * HALF;
        float qr[NKB][4];
        load_qf(qr);
        if constexpr (STYLE == 0) {
#pragma unroll
          for (int kb = 0; kb < NKB / 2; ++kb)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 cs = __ldg(t + qdim(kb, j));
              rot(qr[kb][j], qr[kb + NKB / 2][j], cs.x, cs.y);
            }
        } else {
#pragma unroll
          for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
            for (int j = 0; j < 4; j += 2) {
              const float2 cs = __ldg(t + qdim(kb, j) / 2);
              rot(qr[kb][j], qr[kb][j + 1], cs.x, cs.y);
            }
        }
#pragma unroll
        for (int kb = 0; kb < NKB; ++kb) {
          qa[kb][0] = pack_bf2(qr[kb][0], qr[kb][1]);
          qa[kb][2] = pack_bf2(qr[kb][2], qr[kb][3]);
        }
      }

      int r0 = -1;                     // re-based position of the block's first slot
      // The warp's query base R(r_q - r0) as a row of (cos, sin) per pair
      // (lane t holds pairs 2t and 2t+1 of `qrow`): seeded from the table for
      // the warp's first block of the segment, then stepped from block to
      // block by R(-NPAIR*TK), and by R(W_ring) where the ring wraps; seeded
      // again from the table where the blocks jump (pinned prefix to ring).
      float4 seed = make_float4(0.f, 0.f, 0.f, 0.f);
      bool seeded = true;
      float2* my_row = qrow + cw * HALF;
      auto table_row = [&](int r) {    // R(r_q - r) for this lane's two pairs
        const int m0 = rq - r;
        const int am = m0 < 0 ? -m0 : m0;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (2 * lane < HALF) {
          v = __ldg(reinterpret_cast<const float4*>(p.table + (size_t)am * HALF) + lane);
          if (m0 < 0) { v.y = -v.y; v.w = -v.w; }
        }
        return v;
      };
      if constexpr (ROTK) {
        if (rb + jb < x1 && !dry) {
          seed = table_row(block_geo(rb + jb, u, p.sh).r0);
          seeded = false;
        }
      }
      auto cmul_row = [&](float2* row, const float2* f) {   // row *= f, per pair
        if (2 * lane < HALF) {
          const float4 a = reinterpret_cast<const float4*>(row)[lane];
          const float4 b = reinterpret_cast<const float4*>(f)[lane];
          reinterpret_cast<float4*>(row)[lane] =
              make_float4(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x,
                          a.z * b.z - a.w * b.w, a.z * b.w + a.w * b.z);
        }
      };
      const int Wg = p.sh.Wring;
      BlockWalk wk{};
      if (rb + jb < x1 && !dry) wk.init(rb + jb, u, p.sh);
      // The side warp's dry pass also runs the block body once, on whatever
      // stage 0 holds: no wait, no release, no wrap (whose row it would write).
      bool dry_blk = side && dry;
      for (; dry_blk || (!dry && rb + jb < x1); jb += NPAIR) {
        if (r0 >= 0 && !dry_blk) {
          // NPAIR blocks further on: the query base turns by R(-NPAIR*TK), and
          // by R(W_ring) each time the ring's end is passed; where the blocks
          // jump (pinned prefix to ring) it is seeded from the table again.
          const int wraps = wk.advance(NPAIR, u, p.sh);
          if constexpr (ROTK) {
            if (wraps >= 0) {
              __syncwarp();
              cmul_row(my_row, srow);
              for (int i = 0; i < wraps; ++i) {
                __syncwarp();
                cmul_row(my_row, Wrow);
              }
            } else {
              const float4 v = table_row(wk.g.r0);
              __syncwarp();
              if (2 * lane < HALF) reinterpret_cast<float4*>(my_row)[lane] = v;
            }
          }
        }
        const BlockGeo& bg = wk.g;
        r0 = bg.r0;
        const int wrap_at = bg.wrap_at;  // keys d >= wrap_at sit at r0 + d - W_ring
        const bool wraps = wrap_at < TK && !dry_blk;
        const bool allvalid = wraps ? (u.fill == Wg) : (r0 + TK <= bg.lim);
        const bool plain = allvalid && !wraps;   // every key visible, one base
        {
          const int st_i = stage, st_r = round;
          // A pair only waits on every NPAIR-th stage, so it may reach one
          // before the stage's previous block has even landed.  Waiting first
          // for that block's release makes the full barrier's parity unambiguous.
          if (!dead && !dry_blk && st_r > 0 &&
              !mbar_wait_or_abort(smem_u32(empty + st_i), (st_r - 1) & 1, abort_flag))
            dead = true;
          if (!dead && !dry_blk &&
              !mbar_wait_or_abort(smem_u32(full + st_i), st_r & 1, abort_flag))
            dead = true;
          dead = __any_sync(0xffffffffu, dead);   // the warp stays converged
          if (dead && lane == 0 && !*abort_flag) {
            *abort_flag = 1;
            p.st[u.s].status = STATUS_DEVICE_STATE;
          }
          if (!dead) {
          const uint8_t* kt = stages + (size_t)st_i * C::STAGE;
          const uint8_t* vt = kt + TILE;
          const uint32_t kt_s = smem_u32(kt), vt_s = smem_u32(vt);
          // ---- query fragments for this block's base(s) ----
          if constexpr (ROTK) {
            {
              if (!seeded) {
                if (2 * lane < HALF) reinterpret_cast<float4*>(my_row)[lane] = seed;
                seeded = true;
              }
              __syncwarp();
              const float2* ta = my_row;
              const float sa = 1.f;
              // Rows 0..7 (hi = 0) or 8..15 (hi = 1) of the A operand.
              auto rotate_q = [&](const float2* tr, float sg, auto hi_c) {
                constexpr int hi = decltype(hi_c)::value;
                float qr[NKB][4];
                load_qf(qr);
                if constexpr (STYLE == 0) {
#pragma unroll
                  for (int kb = 0; kb < NKB / 2; ++kb)
#pragma unroll
                    for (int j = 0; j < 4; j += 2) {
                      const float4 a = *reinterpret_cast<const float4*>(tr + qdim(kb, j));
                      rot(qr[kb][j], qr[kb + NKB / 2][j], a.x, sg * a.y);
                      rot(qr[kb][j + 1], qr[kb + NKB / 2][j + 1], a.z, sg * a.w);
                    }
                } else {
#pragma unroll
                  for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
                    for (int j = 0; j < 4; j += 2) {
                      const float2 a = tr[qdim(kb, j) >> 1];
                      rot(qr[kb][j], qr[kb][j + 1], a.x, sg * a.y);
                    }
                }
#pragma unroll
                for (int kb = 0; kb < NKB; ++kb) {
                  qa[kb][hi] = pack_bf2(qr[kb][0], qr[kb][1]);
                  qa[kb][hi + 2] = pack_bf2(qr[kb][2], qr[kb][3]);
                }
              };
              rotate_q(ta, sa, std::integral_constant<int, 0>{});
              if (wraps) {
                // The keys past the ring's end take R(r_q - r0 + W).
                float2* wr = wrow + cw * HALF;
                if (2 * lane < HALF) reinterpret_cast<float4*>(wr)[lane] =
                    reinterpret_cast<const float4*>(my_row)[lane];
                cmul_row(wr, Wrow);
                __syncwarp();
                rotate_q(wr, 1.f, std::integral_constant<int, 1>{});
              }
            }
          }
          // ---- S = Q K^T per 8-key group; select each key's base ----
          float s[2][2];
#pragma unroll
          for (int nb = 0; nb < 2; ++nb) {
            uint32_t kf[NGRP];
            const int krow = hh * TKH + nb * 8 + (lane & 7);
#pragma unroll
            for (int g4 = 0; g4 < NGRP; g4 += 4)
              ldsm_x4(kt_s + tile_swz(krow, g4 + (lane >> 3)), kf[g4], kf[g4 + 1], kf[g4 + 2],
                      kf[g4 + 3]);
            if constexpr (ROTK) {
              const int dk = hh * TKH + nb * 8 + g;   // this thread's key within the block
              const uint8_t* frow = fine + dk * HALF * 8;
              if constexpr (STYLE == 0) {
#pragma unroll
                for (int gr = 0; gr < HG; ++gr) {
                  const int k = 4 * gr + cq;      // pairs 8gr + 2cq and 8gr + 2cq + 1
                  const float4 cs =
                      *reinterpret_cast<const float4*>(frow + fine_chunk<D>(dk, k));
                  rot_pair2(kf[gr], kf[gr + HG], cs);
                }
              } else {
#pragma unroll
                for (int gr = 0; gr < NGRP; ++gr) {
                  const int i = 4 * gr + cq;      // the pair in word gr
                  const float2 cs = *reinterpret_cast<const float2*>(
                      frow + fine_chunk<D>(dk, i >> 1) + ((i & 1) << 3));
                  float x0 = bf_lo(kf[gr]), x1 = bf_hi(kf[gr]);
                  rot(x0, x1, cs.x, cs.y);
                  kf[gr] = pack_bf2(x0, x1);
                }
              }
            }
            // Two interleaved accumulation chains (even and odd k-blocks).
            float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kb = 0; kb < NKB; kb += 2) {
              mma_bf16(acc0, qa[kb][0], qa[kb][1], qa[kb][2], qa[kb][3], kf[2 * kb],
                       kf[2 * kb + 1]);
              mma_bf16(acc1, qa[kb + 1][0], qa[kb + 1][1], qa[kb + 1][2], qa[kb + 1][3],
                       kf[2 * kb + 2], kf[2 * kb + 3]);
            }
            float accs[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) accs[i] = acc0[i] + acc1[i];
            if (plain) {
              s[nb][0] = accs[0] * p.scale_log2;
              s[nb][1] = accs[1] * p.scale_log2;
            } else {
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int d = hh * TKH + nb * 8 + 2 * cq + e;
                const bool wr = ROTK && d >= wrap_at;
                const int r = r0 + d - (d >= wrap_at ? Wg : 0);
                const bool vis = allvalid || r < bg.lim;
                s[nb][e] = vis ? (wr ? accs[2 + e] : accs[e]) * p.scale_log2 : NEG_BIG;
              }
            }
          }
          // ---- online softmax for head g (the 4 lanes of quad g) ----
          float tmax = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
          tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
          tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
          const float mnew = fmaxf(m_run, tmax);
          const float alpha = exp2f(m_run - mnew);
          float pr[2][2];
          float psum = 0.f;
#pragma unroll
          for (int nb = 0; nb < 2; ++nb)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              pr[nb][e] = s[nb][e] > 0.5f * NEG_BIG ? exp2f(s[nb][e] - mnew) : 0.f;
              psum += pr[nb][e];
            }
          l_run = l_run * alpha + psum;
          m_run = mnew;
          // Most blocks raise no running maximum once it settles: then every
          // alpha is 1 and the rescale is skipped.
          if (!__all_sync(0xffffffffu, alpha == 1.f)) {
            const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * cq);      // head 2cq
            const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * cq + 4);  // head 2cq+1
#pragma unroll
            for (int mt = 0; mt < NKB; ++mt) {
              o[mt][0] *= a0; o[mt][1] *= a1; o[mt][2] *= a0; o[mt][3] *= a1;
            }
          }
          // ---- O^T += V^T P^T over the 16 keys of this half ----
          {
            const uint32_t b0 = pack_bf2(pr[0][0], pr[0][1]);
            const uint32_t b1 = pack_bf2(pr[1][0], pr[1][1]);
            // V rows of keys outside the window are zeroed (they may hold anything).
            uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
            if (!allvalid) {
              auto ok = [&](int d) { return r0 + d - (d >= wrap_at ? Wg : 0) < bg.lim; };
              const int d0 = hh * TKH + 2 * cq;
              mlo = (ok(d0) ? 0x0000ffffu : 0u) | (ok(d0 + 1) ? 0xffff0000u : 0u);
              mhi = (ok(d0 + 8) ? 0x0000ffffu : 0u) | (ok(d0 + 9) ? 0xffff0000u : 0u);
            }
            const int vrow = hh * TKH + ((lane >> 4) << 3) + (lane & 7);
            if (allvalid) {
#pragma unroll
              for (int mt = 0; mt < NKB; ++mt) {
                uint32_t v0, v1, v2, v3;
                ldsm_x4_t(vt_s + tile_swz(vrow, 2 * mt + ((lane >> 3) & 1)), v0, v1, v2, v3);
                mma_bf16(o[mt], v0, v1, v2, v3, b0, b1);
              }
            } else {
#pragma unroll
              for (int mt = 0; mt < NKB; ++mt) {
                uint32_t v0, v1, v2, v3;
                ldsm_x4_t(vt_s + tile_swz(vrow, 2 * mt + ((lane >> 3) & 1)), v0, v1, v2, v3);
                mma_bf16(o[mt], v0 & mlo, v1 & mlo, v2 & mhi, v3 & mhi, b0, b1);
              }
            }
          }
          __syncwarp();
          if (lane == 0 && !dry_blk) mbar_arrive(smem_u32(empty + st_i));   // this warp's half is done
          }
        }
        if (dry_blk) {
          dry_blk = false;
          jb -= NPAIR;
          r0 = -1;
          continue;
        }
        stage += NPAIR;
        if (stage >= NS) { stage -= NS; ++round; }
      }

      // ---- segment end: merge the consumer warps ----
      // Once every consumer is done with the stages (the producer issues
      // nothing more until the merge is over), each warp leaves (m, l, O^T)
      // of its blocks in its slot, in the stage memory; after one more barrier
      // every thread combines the NCW slots for its output elements into this
      // CTA's partial.  In a 2-CTA cluster that splits the unit, rank 1 sends
      // its partial (per thread: m, l and its few elements) straight into rank
      // 0's receive area (asynchronous stores that complete bytes on rank 0's
      // barrier) and is done; rank 0 folds it into its own and writes the
      // output.  Otherwise the partial is the output (whole unit) or goes to
      // the unit's ticket merge in global memory.
      cbar();
      const bool whole = (x == u.ustart) && (x1 == u.uend);
      const bool ship = CL && !whole && x != u.ustart;      // rank 1: partial goes to rank 0
      const bool receive = CL && !whole && x == u.ustart;   // rank 0: waits for it
      {
        float lsum = l_run;
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
        if constexpr (FUSED) {
          if (x != rb) score_new();
        }
        if (!dry) {
          float* my = slots + cw * C::SLOT;
          if (cq == 0) { my[g] = m_run; my[8 + g] = lsum; }
#pragma unroll
          for (int i = 0; i < C::FR; ++i) my[16 + 32 * i + lane] = o[i >> 2][i & 3];
        }
      }
      cbar();
      if (has_next && !dry) unstage_q();
      const int R = p.R;   // == G for decode
      {
        // Thread ct takes fragment elements i = ct/32, ct/32 + NCW, ... of lane
        // lf: head h = 2(lf & 3) + (i & 1) is the same for all of them.
        constexpr int NE = (C::FR + NCW - 1) / NCW;   // output elements per thread (at most)
        const int lf = ct & 31, i0 = ct >> 5;
        const int h = 2 * (lf & 3) + (i0 & 1);
        float M = NEG_BIG;
#pragma unroll
        for (int w = 0; w < NCW; ++w) M = fmaxf(M, slots[w * C::SLOT + h]);
        float sc[NCW], L = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
          sc[w] = exp2f(slots[w * C::SLOT + h] - M);
          L += sc[w] * slots[w * C::SLOT + 8 + h];
        }
        float v[NE];
        int dd[NE];
        bool ok[NE];   // element i0 + k NCW exists (NCW need not divide FR)
#pragma unroll
        for (int k = 0; k < NE; ++k) {
          const int i = i0 + k * NCW;
          ok[k] = i < C::FR;
          dd[k] = ok[k] ? 16 * (i >> 2) + (lf >> 2) + (((i >> 1) & 1) << 3) : 0;
          float a = 0.f;
          if (ok[k]) {
#pragma unroll
            for (int w = 0; w < NCW; ++w) a += sc[w] * slots[w * C::SLOT + 16 + 32 * i + lf];
          }
          v[k] = a;
        }
        if (ship && !dry) {
          const uint32_t peer = cluster_rank() ^ 1u;
          const uint32_t dst = map_to_rank(smem_u32(rslots + ct), peer);
          const uint32_t bar = map_to_rank(smem_u32(rx_bar), peer);
          st_async_f32(dst, M, bar);
          st_async_f32(dst + 4u * CONS_THREADS, L, bar);
#pragma unroll
          for (int k = 0; k < NE; ++k) st_async_f32(dst + 4u * (2 + k) * CONS_THREADS, v[k], bar);
        } else {
          bool got = true;
          if (receive && !dry) {
            got = false;
            for (uint32_t i = 0; i < WAIT_LIMIT && !got; ++i)
              got = mbar_try_wait_cluster(smem_u32(rx_bar), 0);
            if (!got && ct == 0) {
              *abort_flag = 1;
              p.st[u.s].status = STATUS_DEVICE_STATE;
            }
            if (got) {
              // Rank 1's partial of the same elements.
              const float M1 = rslots[ct], L1 = rslots[CONS_THREADS + ct];
              const float Mx = fmaxf(M, M1);
              const float s0 = exp2f(M - Mx), s1 = exp2f(M1 - Mx);
              L = s0 * L + s1 * L1;
#pragma unroll
              for (int k = 0; k < NE; ++k) v[k] = s0 * v[k] + s1 * rslots[(2 + k) * CONS_THREADS + ct];
              M = Mx;
            }
          }
          if (add_new) {
            // The new pair: score mx[h], value v_new.
            const float Mx = fmaxf(M, mx[h]);
            const float s0 = exp2f(M - Mx), sn = exp2f(mx[h] - Mx);
            L = s0 * L + sn;
#pragma unroll
            for (int k = 0; k < NE; ++k) v[k] = s0 * v[k] + sn * kvn[D + dd[k]];
            M = Mx;
          }
          if (got && h < R && !dry) {
            if (whole || receive) {
              const float inv = L > 0.f ? 1.f / L : 0.f;
              float* out = p.out + row_offset(p, u, h);
#pragma unroll
              for (int k = 0; k < NE; ++k)
                if (ok[k]) out[dd[k]] = v[k] * inv;
            } else {
              float* part = p.partials + (size_t)(2 * b + (x == rb ? 0 : 1)) * p.slot_floats;
              if (lf < 4 && i0 < 2) { part[h] = M; part[R + h] = L; }
#pragma unroll
              for (int k = 0; k < NE; ++k)
                if (ok[k]) part[2 * R + h * D + dd[k]] = v[k];
            }
          }
        }
      }
      if (!whole && !CL) {
        // Publish this CTA's partial (one release by one thread after the
        // barrier); the last CTA of the unit to arrive merges them all, with
        // the raw-query area (free by now) as scratch.
        if (!dry) {
          named_bar_sync(BAR_CONS, CONS_THREADS);
          if (ct == 0) {
            __threadfence();
            flag[0] = atomicAdd(&p.unit_tickets[unit_index(p, u)], 1);
            __threadfence();
          }
          named_bar_sync(BAR_CONS, CONS_THREADS);
          const int b0 = cta_of(u.ustart, T, P), b1 = cta_of(u.uend - 1, T, P);
          if (flag[0] == b1 - b0) {
            merge_unit_partials<4>(p, u, T, P, ct, CONS_THREADS, reinterpret_cast<float*>(qraw),
                                   8 * D, [] { named_bar_sync(BAR_CONS, CONS_THREADS); });
            if (ct == 0) p.unit_tickets[unit_index(p, u)] = 0;
          }
        }
      }
      // The slots' generic-proxy accesses come before the producer's next
      // asynchronous copies into the same memory.
      fence_proxy_async();
      cbar();
      if (dry) {   // the real pass over the same segment
        if (side) break;
        dry = false;
        continue;
      }
      if (ct == 0) mbar_arrive(smem_u32(mdone));
      if constexpr (FUSED) {
        if (has_next) unstage_new();
      }
      x = x1;
    }
    if (side) {
      // The step's new pairs into their slots (every unit once over the grid),
      // then, on the step's last launch, the new stream states.
      step_prepass<D, !ROTK>(p, sa, sfill, slag, 0, 1, lane);
      if (p.publish) step_publish(p, lane);
    }
  }
  __syncthreads();
  if constexpr (CL) cluster_sync_all();   // neither CTA leaves while the other may reach it
  if (tid == 0 && *abort_flag) {
    // Normally every issued stage was waited on by its consumers.  After an
    // abort, no CTA exits with a copy still in flight into its shared memory:
    // wait (bounded) for the last NS stages this CTA issued.
    const int issued = flag[2];
    for (int j = max(0, issued - NS); j < issued; ++j)
      mbar_wait(smem_u32(full + (j % NS)), (j / NS) & 1);
  }
}

template <int D, bool ROTK>
static int mma_stages(int S) {
  using C = MmaCfg<D, ROTK>;
  int ns = MMA_MAX_STAGES;
  while (ns > NPAIR && mma_smem_bytes(C::STAGE, C::FIXED, ns, S) > (size_t)SMEM_LIMIT) --ns;
  return ns;
}

size_t attend_mma_smem(const Shape& sh, int c) {
  (void)c;
  const bool rotk = !sh.stored_rotated;
  if (sh.D == 128) {
    if (rotk) return mma_smem_bytes(MmaCfg<128, true>::STAGE, MmaCfg<128, true>::FIXED,
                                    mma_stages<128, true>(sh.S), sh.S);
    return mma_smem_bytes(MmaCfg<128, false>::STAGE, MmaCfg<128, false>::FIXED,
                          mma_stages<128, false>(sh.S), sh.S);
  }
  if (rotk) return mma_smem_bytes(MmaCfg<64, true>::STAGE, MmaCfg<64, true>::FIXED,
                                  mma_stages<64, true>(sh.S), sh.S);
  return mma_smem_bytes(MmaCfg<64, false>::STAGE, MmaCfg<64, false>::FIXED,
                        mma_stages<64, false>(sh.S), sh.S);
}

bool attend_mma_supported(const Shape& sh, int c) {
  return sh.bf16 && (sh.D == 64 || sh.D == 128) && sh.G <= 8 && c == 1 &&
         attend_mma_smem(sh, c) <= (size_t)SMEM_LIMIT;
}

// The pair of CTAs that shares a unit merges through distributed shared
// memory when every unit is cut into exactly two CTAs (one stream, grid = 2U).
inline bool use_cluster_merge(const AttendParams& p, int grid) {
  return p.sh.S == 1 && grid == 2 * p.L_att * p.sh.Hkv;
}

template <int D, bool ROTK, int STYLE, bool FUSED, bool CL>
static cudaError_t launch_mma_k(const AttendParams& p0, const CUtensorMap& tk,
                                const CUtensorMap& tv, int grid, cudaStream_t s) {
  using C = MmaCfg<D, ROTK>;
  AttendParams p = p0;
  const int rx = CL ? rx_floats<D>() * 4 : 0;
  int ns = MMA_MAX_STAGES;
  while (ns > NPAIR && mma_smem_bytes(C::STAGE, C::FIXED, ns, p.sh.S, rx) > (size_t)SMEM_LIMIT)
    --ns;
  p.ns = ns;
  const size_t smem = mma_smem_bytes(C::STAGE, C::FIXED, p.ns, p.sh.S, rx);
  if (smem > (size_t)SMEM_LIMIT) return cudaErrorNotSupported;
  auto kern = attend_mma_decode<D, ROTK, STYLE, FUSED, CL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // Programmatic dependent launch: the prologue overlaps the previous kernel.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(mma_threads<FUSED>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CL ? 2 : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CL ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, p, tk, tv);
}

template <int D, bool ROTK, int STYLE, bool FUSED = false>
static cudaError_t launch_mma_t(const AttendParams& p, const CUtensorMap& tk,
                                const CUtensorMap& tv, int grid, cudaStream_t s) {
  if (use_cluster_merge(p, grid)) return launch_mma_k<D, ROTK, STYLE, FUSED, true>(p, tk, tv, grid, s);
  return launch_mma_k<D, ROTK, STYLE, FUSED, false>(p, tk, tv, grid, s);
}

template <int D>
static cudaError_t launch_mma_d(const AttendParams& p, const CUtensorMap& tk,
                                const CUtensorMap& tv, int grid, cudaStream_t s) {
  const bool rotk = !p.sh.stored_rotated;
  if (p.sh.style == 0)
    return rotk ? launch_mma_t<D, true, 0>(p, tk, tv, grid, s)
                : launch_mma_t<D, false, 0>(p, tk, tv, grid, s);
  return rotk ? launch_mma_t<D, true, 1>(p, tk, tv, grid, s)
              : launch_mma_t<D, false, 1>(p, tk, tv, grid, s);
}

cudaError_t launch_attend_mma(const AttendParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              int grid, cudaStream_t s) {
  if (!attend_mma_supported(p.sh, p.c)) return cudaErrorNotSupported;
  if (p.sh.D == 128) return launch_mma_d<128>(p, tk, tv, grid, s);
  return launch_mma_d<64>(p, tk, tv, grid, s);
}

cudaError_t launch_step_mma(const AttendParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                            int grid, cudaStream_t s) {
  // Pre-RoPE keys, or stored-rotated keys that follow a re-basing epoch.
  if (!attend_mma_supported(p.sh, 1) || (p.sh.stored_rotated && !p.sh.epoch) || p.c != 1)
    return cudaErrorNotSupported;
  if (p.sh.stored_rotated) {
    if (p.sh.D == 128)
      return p.sh.style == 0 ? launch_mma_t<128, false, 0, true>(p, tk, tv, grid, s)
                             : launch_mma_t<128, false, 1, true>(p, tk, tv, grid, s);
    return p.sh.style == 0 ? launch_mma_t<64, false, 0, true>(p, tk, tv, grid, s)
                           : launch_mma_t<64, false, 1, true>(p, tk, tv, grid, s);
  }
  if (p.sh.D == 128)
    return p.sh.style == 0 ? launch_mma_t<128, true, 0, true>(p, tk, tv, grid, s)
                           : launch_mma_t<128, true, 1, true>(p, tk, tv, grid, s);
  return p.sh.style == 0 ? launch_mma_t<64, true, 0, true>(p, tk, tv, grid, s)
                         : launch_mma_t<64, true, 1, true>(p, tk, tv, grid, s);
}

}  // namespace rkv
