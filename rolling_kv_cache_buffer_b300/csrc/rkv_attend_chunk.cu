// rkv_attend_chunk.cu -- tensor-core attention for steps that insert a chunk of
// c > 1 tokens per stream (bf16 caches, R = c*G <= 96 query rows per
// (stream, layer, KV head), D 64 or 128).
//
// What it computes is the attention over the window with exact re-basing of
// "Audio8 ASR Infinite: What It Actually Takes to Listen Forever" ("Inside the
// Rolling KV Cache and Exact RoPE Re-Basing"), causal among the chunk: query j
// of the step sits at r_j = fill - c + j and sees the retained keys at
// r = (slot - origin) mod W with r <= r_j:
//   out_j = sum_{r <= r_j} softmax(<R(r_j) q_j, R(r) k_r> * scale) v_r.
//
// Arithmetic.  The rows (query j, head) that share a KV head make S = Q K^T and
// O^T = V^T P^T dense contractions, run on mma.sync m16n8k16 (bf16 operands,
// f32 accumulation).  Unlike the single-query kernel, every row has its own
// position, so the rotation goes to the keys in full: the key in slot d of a
// block whose first slot sits at r0 is turned by R(r0 + d) = R(r0) R(d) (or
// R(r0 - W) R(d) past the ring's end), composed in f32 from the block's table
// row and a shared-memory R(d) table, then rounded to bf16.  The queries are
// rotated once per unit, R(r_j) q_j.  Stored-rotated keys are used as stored.
//
// Work split: the R rows are cut into groups of 16; a team of ceil(R/16)
// consumer warps takes a block: the team first turns the block's keys in
// place in shared memory (each key once), then each warp takes one row group
// over all 32 keys of the block.  The producer, the stage ring and the merges are those of the
// single-query kernel (rkv_attend_pipe.cuh).
#include "rkv_attend_pipe.cuh"

namespace rkv {

namespace {

constexpr int CCW = 6;                        // consumer warps
constexpr int CH_THREADS = (CCW + 1) * 32;    // + the producer warp
constexpr int CCONS = CCW * 32;
constexpr int CH_MAX_STAGES = 16;
constexpr int CBAR_CONS = 1;                  // named barrier of the consumer warps
constexpr int CBAR_PREFIX = 2;                // the producer warp's block prefix is ready
constexpr int CBAR_TEAM0 = 3;                 // + team: the team's keys are rotated
constexpr int CH_MAX_ROWS = CCW * 16;

template <int D, bool ROTK>
struct ChunkCfg : PipeCfg<D, ROTK> {
  static constexpr int NGRP = D / 8;          // 8-dim groups
  static constexpr int NKB = D / 16;          // k-blocks of the QK product
  static constexpr int HG = NGRP / 2;
  static constexpr int QSTR = D + 8;          // padded query row (floats)
  static constexpr int OSTR = D + 4;          // padded output row (floats)
  static constexpr int SLOT = 32 + 16 * OSTR; // warp partial: m[16] l[16] o[16][OSTR]
};

// `slots`: bytes of merge slots of their own (0: they alias the stages).
__host__ __device__ constexpr size_t chunk_smem_bytes(int stage, int fine, int qstr, int rows16,
                                                      int ns, int S, int slots = 0) {
  return 1024 + (size_t)ns * stage + (size_t)fine + (size_t)rows16 * qstr * 4 + (size_t)slots +
         16 + 16 + (size_t)ns * 16 + (size_t)(3 * S + 1) * 4;
}
// Stages a launch must keep for the merge slots to get memory of their own.
constexpr int CH_OWN_SLOTS_MIN_STAGES = 10;

__device__ __forceinline__ void rotc(float& x, float& y, float c, float s) {
  const float a = x * c - y * s;
  y = y * c + x * s;
  x = a;
}

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
__device__ __forceinline__ f2 f2_sub(f2 a, f2 b) {
  f2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// Two split-half key pairs (bf16x2 words x = dims (i, i+1), y = their partners
// (i+D/2, i+D/2+1)) turned by R(base + d): `bs` = (cos_i, cos_i+1, sin_i,
// sin_i+1) of the base (a chunk of the grouped table; the sines times sg),
// `ds` the same of d.  Angles add: c = cb cd - sb sd, s = sb cd + cb sd; then
// x' = x c - y s, y' = y c + x s, rounded to nearest even: ten packed f32x2
// operations, the cosines and sines of both pairs each in one register pair.
__device__ __forceinline__ void rot_pair2_composed(uint32_t& x, uint32_t& y, float4 bs, float sg,
                                                   float4 ds) {
  const f2 CB = f2_make(bs.x, bs.y);
  f2 SB = f2_make(bs.z, bs.w);
  if (sg < 0.f) SB = f2_mul(SB, f2_make(-1.f, -1.f));
  const f2 CD = f2_make(ds.x, ds.y), SD = f2_make(ds.z, ds.w);
  const f2 C = f2_sub(f2_mul(CB, CD), f2_mul(SB, SD));
  const f2 S = f2_fma(SB, CD, f2_mul(CB, SD));
  const f2 X = f2_make(bf_lo(x), bf_hi(x));
  const f2 Y = f2_make(bf_lo(y), bf_hi(y));
  const f2 Xr = f2_sub(f2_mul(X, C), f2_mul(Y, S));
  const f2 Yr = f2_fma(X, S, f2_mul(Y, C));
  float a, b, e, f;
  f2_split(Xr, a, b);
  f2_split(Yr, e, f);
  x = pack_bf2(a, b);
  y = pack_bf2(e, f);
}

// Turns key slot d of a block tile in place by R(base + d): the 16-byte chunk
// m of its first half (dims 8m..8m+7) with its partners (dims D/2+8m..), i.e.
// split-half pairs 8m..8m+7; or, interleaved, the 4 pairs of chunk m.  `tb` is
// the base's row (sine times sg): of the grouped table for split-half pairs,
// (cos, sin) per pair for interleaved ones; `frow` the R(d) row of the fine
// table.
template <int D, int STYLE>
__device__ __forceinline__ void rotate_unit(uint8_t* kt, int d, int m, const float2* tb, float sg,
                                            const uint8_t* frow) {
  if constexpr (STYLE == 0) {
    uint4* px = reinterpret_cast<uint4*>(kt + tile_swz(d, m));
    uint4* py = reinterpret_cast<uint4*>(kt + tile_swz(d, m + D / 16));
    uint4 x = *px, y = *py;
    uint32_t* xw = reinterpret_cast<uint32_t*>(&x);
    uint32_t* yw = reinterpret_cast<uint32_t*>(&y);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int i = 8 * m + 2 * t;          // pairs i, i+1
      const float4 ds = *reinterpret_cast<const float4*>(frow + fine_chunk_keys<D>(d, i >> 1));
      const float4 bs = *reinterpret_cast<const float4*>(tb + i);
      rot_pair2_composed(xw[t], yw[t], bs, sg, ds);
    }
    *px = x;
    *py = y;
  } else {
    uint4* pz = reinterpret_cast<uint4*>(kt + tile_swz(d, m));
    uint4 z = *pz;
    uint32_t* zw = reinterpret_cast<uint32_t*>(&z);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int i = 4 * m + t;              // the pair in word t
      const float2 cd = *reinterpret_cast<const float2*>(frow + fine_chunk_keys<D>(d, i >> 1) +
                                                        ((i & 1) << 3));
      const float2 cb = tb[i];
      const float cbs = sg * cb.y;
      const float cc = cb.x * cd.x - cbs * cd.y;
      const float ss = cbs * cd.x + cb.x * cd.y;
      float x0 = bf_lo(zw[t]), x1 = bf_hi(zw[t]);
      rotc(x0, x1, cc, ss);
      zw[t] = pack_bf2(x0, x1);
    }
    *pz = z;
  }
}

}  // namespace

// OWN: the merge slots have shared memory of their own, so the producer goes
// on into the next unit segment as soon as the consumers are done with the
// stages (otherwise the slots alias the stages and the producer waits for
// the merge; the ring then drains at every segment boundary).
template <int D, bool ROTK, int STYLE, bool OWN>
__global__ void __launch_bounds__(CH_THREADS, 1)
    attend_mma_chunk(const __grid_constant__ AttendParams p,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV) {
  using C = ChunkCfg<D, ROTK>;
  constexpr int TILE = C::TILE, NGRP = C::NGRP, NKB = C::NKB, HALF = C::HALF;
  constexpr int QSTR = C::QSTR, OSTR = C::OSTR, SLOT = C::SLOT;
  const int G = p.sh.G, NS = p.ns, R = p.R, c = p.c;
  const int RG = (R + 15) >> 4;   // row groups = warps per team
  const int NTEAM = CCW / RG;     // teams (the launcher keeps RG <= CCW)
  const int R16 = RG * 16;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  uint8_t* stages = smem;                                          // [NS][STAGE]
  uint8_t* fine = stages + (size_t)NS * C::STAGE;                  // [TK][D/2] (cos, sin)
  float* qs = reinterpret_cast<float*>(fine + C::FINE);            // [R16][QSTR] raw queries
  // [CCW][SLOT] merge slots, used between segments: after the raw queries
  // (OWN) or over the stages.
  float* slots = OWN ? qs + R16 * QSTR : reinterpret_cast<float*>(smem);
  int* flag = reinterpret_cast<int*>(qs + R16 * QSTR + (OWN ? CCW * SLOT : 0));   // ticket, abort, issued
  uint64_t* mdone = reinterpret_cast<uint64_t*>(flag + 4);         // segment merged
  uint64_t* full = mdone + 2;                                      // [NS]
  uint64_t* empty = full + NS;                                     // [NS]
  int* pre = reinterpret_cast<int*>(empty + NS);                   // [S+1] block prefix
  int* sa = pre + p.sh.S + 1;                                      // [S] origin mod W
  int* sfill = sa + p.sh.S;                                        // [S] fill
  volatile int* abort_flag = flag + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // The producer's first read after the dependency wait is the stream state:
  // bring it into L2 before anything else.
  prefetch_states(p);
  // Prologue: nothing here reads what the previous kernel of the stream writes.
  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(full + i), 1);
      mbar_init(smem_u32(empty + i), RG);   // every warp of the team that takes the block
    }
    mbar_init(smem_u32(mdone), 1);
    fence_mbar_init();
    flag[1] = 0;
    flag[2] = 0;
  }
  if constexpr (ROTK) {
    if (warp > 0) load_fine<D, STYLE, true>(p, fine, tid - 32, CCONS);
  }
  if (warp > 0) prefetch_queries(p, D, tid - 32, CH_THREADS - 32);
  pdl_wait();   // from here on: stream state, pools, queries, outputs
  pdl_trigger();   // a kernel launched next may start its own prologue
  if (warp == 0) {
    build_prefix_cached(p, pre, sa, sfill, lane);
    __syncwarp();
    named_bar_arrive(CBAR_PREFIX, CH_THREADS);
  } else {
    named_bar_sync(CBAR_PREFIX, CH_THREADS);
  }
  const int T = pre[p.sh.S];
  const int P = min(static_cast<int>(gridDim.x), T);
  const int b = static_cast<int>(blockIdx.x);
  const int rb = b < P ? range_start(b, T, P) : 0, re = b < P ? range_start(b + 1, T, P) : 0;

  if (warp == 0) {
    if (lane == 0)
      flag[2] = produce<D, ROTK, KEY_BASES>(
          p, &tmK, &tmV, stages, full, empty, mdone, pre, sa, sfill, rb, re, abort_flag,
          STYLE == 0 ? reinterpret_cast<const float2*>(p.table_g) : nullptr);
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ consumers
    const int cw = warp - 1, ct = tid - 32;
    const int g = lane >> 2, cq = lane & 3;   // mma fragment coordinates
    const int team = cw / RG, rg = cw % RG;
    const bool active = team < NTEAM;
    // Raw queries of a unit into `qs` (rows >= R are zero).
    auto load_query = [&](const UnitRef& u) {
      for (int idx = ct; idx < R16 * D; idx += CCONS) {
        const int row = idx / D, d = idx % D;
        qs[row * QSTR + d] =
            row < R ? load_elem(p.q, row_offset(p, u, row) + d, p.sh.q_bf16) : 0.f;
      }
    };
    if (rb < re) load_query(unit_of_cached(rb, p, pre, sa, sfill));
    zero_empty_units_cached(p, sa, sfill, ct, CCONS);
    named_bar_sync(CBAR_CONS, CCONS);

    // Dims of the thread's A-fragment elements: k-block kb, j in {0,1,2,3}:
    //   dim 16kb + (j>>1)*8 + 2cq + (j&1)
    auto qdim = [&](int kb, int j) { return 16 * kb + (j >> 1) * 8 + 2 * cq + (j & 1); };

    // This warp's rows: rr[0] = 16rg + g and rr[1] = 16rg + g + 8.
    const int rr0 = 16 * rg + g, rr1 = rr0 + 8;
    int jb = team, stage = active ? team : 0, round = 0;   // the team's next block
    bool dead = false;
    for (int x = rb; x < re;) {
      const UnitRef u = unit_of_cached(x, p, pre, sa, sfill);
      const int x1 = min(u.uend, re);
      const bool has_next = x1 < re;
      // Positions of the two rows (query j = row / G at npin + fill - c + j,
      // behind the pinned prefix's npin pairs); rows past R see nothing.
      const int qbase = u.npin + u.fill - c;  // position of the chunk's first query
      const int rq0 = rr0 < R ? qbase + rr0 / G : -1;
      const int rq1 = rr1 < R ? qbase + rr1 / G : -1;
      const int rq_min = qbase;

      // ---- A fragments for the unit: rows rotated once, R(r_j) q ----
      uint32_t qa[NKB][4];
      {
        float q0[NKB][4], q1[NKB][4];
#pragma unroll
        for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
          for (int j = 0; j < 4; j += 2) {
            const float2 v0 = *reinterpret_cast<const float2*>(qs + rr0 * QSTR + qdim(kb, j));
            const float2 v1 = *reinterpret_cast<const float2*>(qs + rr1 * QSTR + qdim(kb, j));
            q0[kb][j] = v0.x; q0[kb][j + 1] = v0.y;
            q1[kb][j] = v1.x; q1[kb][j + 1] = v1.y;
          }
        {
          // Stored-rotated keys with a re-basing epoch sit at r + lag.
          const int lag = p.sh.epoch ? p.st[u.s].pending : 0;
          const float2* t0 = p.table + (size_t)(max(rq0, 0) + lag) * HALF;
          const float2* t1 = p.table + (size_t)(max(rq1, 0) + lag) * HALF;
          if constexpr (STYLE == 0) {
#pragma unroll
            for (int kb = 0; kb < NKB / 2; ++kb)
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float2 a = __ldg(t0 + qdim(kb, j));
                const float2 bq = __ldg(t1 + qdim(kb, j));
                rotc(q0[kb][j], q0[kb + NKB / 2][j], a.x, a.y);
                rotc(q1[kb][j], q1[kb + NKB / 2][j], bq.x, bq.y);
              }
          } else {
#pragma unroll
            for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
              for (int j = 0; j < 4; j += 2) {
                const float2 a = __ldg(t0 + qdim(kb, j) / 2);
                const float2 bq = __ldg(t1 + qdim(kb, j) / 2);
                rotc(q0[kb][j], q0[kb][j + 1], a.x, a.y);
                rotc(q1[kb][j], q1[kb][j + 1], bq.x, bq.y);
              }
          }
        }
#pragma unroll
        for (int kb = 0; kb < NKB; ++kb) {
          qa[kb][0] = pack_bf2(q0[kb][0], q0[kb][1]);
          qa[kb][1] = pack_bf2(q1[kb][0], q1[kb][1]);
          qa[kb][2] = pack_bf2(q0[kb][2], q0[kb][3]);
          qa[kb][3] = pack_bf2(q1[kb][2], q1[kb][3]);
        }
      }
      float o[NKB][2][4];              // O^T accumulators: m-tile = 16 dims, n-tile = 8 rows
      float m_run[2] = {NEG_BIG, NEG_BIG}, l_run[2] = {0.f, 0.f};
#pragma unroll
      for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 4; ++j) o[kb][nt][j] = 0.f;

      const int Wg = p.sh.Wring;
      BlockWalk wk;
      if (active && rb + jb < x1) wk.init(rb + jb, u, p.sh);
      for (bool first = true; active && rb + jb < x1; jb += NTEAM, first = false) {
        if (!first) wk.advance(NTEAM, u, p.sh);   // NTEAM blocks further on
        const BlockGeo& bg = wk.g;
        const int r0 = bg.r0;            // re-based position of the block's first slot
        const int wrap_at = bg.wrap_at;  // keys d >= wrap_at sit at r0 + d - W_ring
        const bool wraps = wrap_at < TK;
        const bool allvalid = wraps ? (u.fill == Wg) : (r0 + TK <= bg.lim);
        const int maxpos = wraps ? u.npin + Wg - 1 : r0 + TK - 1;
        const bool plain = allvalid && maxpos <= rq_min;   // every key seen by every row
        // A team only waits on every NTEAM-th stage, so it may reach one before
        // the stage's previous block has landed: wait for that block's release
        // first, so that the full barrier's parity is unambiguous.
        if (!dead && round > 0 &&
            !mbar_wait_or_abort(smem_u32(empty + stage), (round - 1) & 1, abort_flag))
          dead = true;
        if (!dead && !mbar_wait_or_abort(smem_u32(full + stage), round & 1, abort_flag))
          dead = true;
        dead = __any_sync(0xffffffffu, dead);   // the warp stays converged
        if (dead && lane == 0 && !*abort_flag) {
          *abort_flag = 1;
          p.st[u.s].status = STATUS_DEVICE_STATE;
        }
        if constexpr (ROTK) {
          // The team turns the block's keys in place, each warp a share of
          // the (key, chunk) units, then meets at the team barrier.
          if (!dead) {
            uint8_t* ktw = stages + (size_t)stage * C::STAGE;
            const float2* trA = reinterpret_cast<const float2*>(ktw + 2 * TILE);
            constexpr int UPK = STYLE == 0 ? D / 16 : D / 8;   // units per key
            for (int un = rg * 32 + lane; un < TK * UPK; un += RG * 32) {
              // Keys fastest: eight lanes take keys d..d+7 of the same chunk m,
              // which the tile swizzle and the table layout spread over all banks.
              const int d = un % TK, m = un / TK;
              // Past the ring's end: base R(r0 - W_ring), the stage's second
              // row |r0 - W_ring| with its sine negated when r0 < W_ring.
              const bool useB = d >= wrap_at;
              rotate_unit<D, STYLE>(ktw, d, m, useB ? trA + HALF : trA,
                                    useB && r0 < Wg ? -1.f : 1.f, fine + d * HALF * 8);
            }
            // These generic writes come before the next asynchronous copy into
            // the stage.
            fence_proxy_async();
          }
          if (RG > 1)
            named_bar_sync(CBAR_TEAM0 + team, RG * 32);
          else
            __syncwarp();
        }
        if (!dead) {
          const uint8_t* kt = stages + (size_t)stage * C::STAGE;
          const uint8_t* vt = kt + TILE;
          const uint32_t kt_s = smem_u32(kt), vt_s = smem_u32(vt);
          // ---- S = Q K^T per 8-key group ----
          float s[4][2][2];   // [key group][row 0/1][key pair element]
#pragma unroll
          for (int nb = 0; nb < 4; ++nb) {
            uint32_t kf[NGRP];
            const int krow = nb * 8 + (lane & 7);
#pragma unroll
            for (int g4 = 0; g4 < NGRP; g4 += 4)
              ldsm_x4(kt_s + tile_swz(krow, g4 + (lane >> 3)), kf[g4], kf[g4 + 1], kf[g4 + 2],
                      kf[g4 + 3]);
            float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kb = 0; kb < NKB; kb += 2) {
              mma_bf16(acc0, qa[kb][0], qa[kb][1], qa[kb][2], qa[kb][3], kf[2 * kb],
                       kf[2 * kb + 1]);
              mma_bf16(acc1, qa[kb + 1][0], qa[kb + 1][1], qa[kb + 1][2], qa[kb + 1][3],
                       kf[2 * kb + 2], kf[2 * kb + 3]);
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float a0 = (acc0[e] + acc1[e]) * p.scale_log2;       // row rr0
              const float a1 = (acc0[2 + e] + acc1[2 + e]) * p.scale_log2;  // row rr1
              if (plain) {
                s[nb][0][e] = a0;
                s[nb][1][e] = a1;
              } else {
                const int d = nb * 8 + 2 * cq + e;
                const int r = r0 + d - (d >= wrap_at ? Wg : 0);
                const bool in = r < bg.lim;
                s[nb][0][e] = (in && r <= rq0) ? a0 : NEG_BIG;
                s[nb][1][e] = (in && r <= rq1) ? a1 : NEG_BIG;
              }
            }
          }
          // ---- online softmax per row (rows g and g+8: the 4 lanes of quad g) ----
          float pr[4][2][2];
          float alpha[2];
#pragma unroll
          for (int rw = 0; rw < 2; ++rw) {
            float tmax = NEG_BIG;
#pragma unroll
            for (int nb = 0; nb < 4; ++nb) tmax = fmaxf(tmax, fmaxf(s[nb][rw][0], s[nb][rw][1]));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
            const float mnew = fmaxf(m_run[rw], tmax);
            alpha[rw] = exp2f(m_run[rw] - mnew);
            float psum = 0.f;
#pragma unroll
            for (int nb = 0; nb < 4; ++nb)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                pr[nb][rw][e] = s[nb][rw][e] > 0.5f * NEG_BIG ? exp2f(s[nb][rw][e] - mnew) : 0.f;
                psum += pr[nb][rw][e];
              }
            l_run[rw] = l_run[rw] * alpha[rw] + psum;
            m_run[rw] = mnew;
          }
          // o columns of this thread: rows nt*8 + 2cq (+1); their alphas sit in
          // quads 2cq and 2cq+1.  Once the running maxima settle, most blocks
          // raise none of them: every alpha is 1 and the rescale is skipped.
          if (!__all_sync(0xffffffffu, alpha[0] == 1.f && alpha[1] == 1.f)) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              const float ae = __shfl_sync(0xffffffffu, alpha[nt], 8 * cq);
              const float ao = __shfl_sync(0xffffffffu, alpha[nt], 8 * cq + 4);
#pragma unroll
              for (int mt = 0; mt < NKB; ++mt) {
                o[mt][nt][0] *= ae; o[mt][nt][1] *= ao; o[mt][nt][2] *= ae; o[mt][nt][3] *= ao;
              }
            }
          }
          // ---- O^T += V^T P^T ----
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            uint32_t bb[2][2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              bb[nt][0] = pack_bf2(pr[2 * kk][nt][0], pr[2 * kk][nt][1]);
              bb[nt][1] = pack_bf2(pr[2 * kk + 1][nt][0], pr[2 * kk + 1][nt][1]);
            }
            // V rows of keys outside the window are zeroed (they may hold anything).
            uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
            if (!allvalid) {
              auto ok = [&](int d) { return r0 + d - (d >= wrap_at ? Wg : 0) < bg.lim; };
              const int d0 = 16 * kk + 2 * cq;
              mlo = (ok(d0) ? 0x0000ffffu : 0u) | (ok(d0 + 1) ? 0xffff0000u : 0u);
              mhi = (ok(d0 + 8) ? 0x0000ffffu : 0u) | (ok(d0 + 9) ? 0xffff0000u : 0u);
            }
            const int vrow = 16 * kk + ((lane >> 4) << 3) + (lane & 7);
            if (allvalid) {
#pragma unroll
              for (int mt = 0; mt < NKB; ++mt) {
                uint32_t v0, v1, v2, v3;
                ldsm_x4_t(vt_s + tile_swz(vrow, 2 * mt + ((lane >> 3) & 1)), v0, v1, v2, v3);
                mma_bf16(o[mt][0], v0, v1, v2, v3, bb[0][0], bb[0][1]);
                mma_bf16(o[mt][1], v0, v1, v2, v3, bb[1][0], bb[1][1]);
              }
            } else {
#pragma unroll
              for (int mt = 0; mt < NKB; ++mt) {
                uint32_t v0, v1, v2, v3;
                ldsm_x4_t(vt_s + tile_swz(vrow, 2 * mt + ((lane >> 3) & 1)), v0, v1, v2, v3);
                v0 &= mlo; v1 &= mlo; v2 &= mhi; v3 &= mhi;
                mma_bf16(o[mt][0], v0, v1, v2, v3, bb[0][0], bb[0][1]);
                mma_bf16(o[mt][1], v0, v1, v2, v3, bb[1][0], bb[1][1]);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(empty + stage));   // this warp is done
        }
        stage += NTEAM;
        while (stage >= NS) { stage -= NS; ++round; }
      }

      // ---- segment end: merge the teams (rows of each row group) ----
      named_bar_sync(CBAR_CONS, CCONS);      // nobody reads the stages any more
      // With slots of their own the producer may fill the stages again now.
      if (OWN && ct == 0) mbar_arrive(smem_u32(mdone));
      {
        float lsum[2];
#pragma unroll
        for (int rw = 0; rw < 2; ++rw) {
          lsum[rw] = l_run[rw];
          lsum[rw] += __shfl_xor_sync(0xffffffffu, lsum[rw], 1);
          lsum[rw] += __shfl_xor_sync(0xffffffffu, lsum[rw], 2);
        }
        float* my = slots + cw * SLOT;
        if (cq == 0) {
          my[g] = m_run[0];
          my[8 + g] = m_run[1];
          my[16 + g] = lsum[0];
          my[24 + g] = lsum[1];
        }
#pragma unroll
        for (int mt = 0; mt < NKB; ++mt)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int row = nt * 8 + 2 * cq + (j & 1);
              const int d = 16 * mt + g + ((j >> 1) << 3);
              my[32 + row * OSTR + d] = o[mt][nt][j];
            }
      }
      named_bar_sync(CBAR_CONS, CCONS);
      const bool whole = (x == u.ustart) && (x1 == u.uend);
      float* part = nullptr;
      if (!whole) part = p.partials + (size_t)(2 * b + (x == rb ? 0 : 1)) * p.slot_floats;
      for (int idx = ct; idx < R * D; idx += CCONS) {
        const int row = idx / D, d = idx % D;
        const int grp = row >> 4, rl = row & 15;
        float M = NEG_BIG;
        for (int t = 0; t < NTEAM; ++t) M = fmaxf(M, slots[(t * RG + grp) * SLOT + rl]);
        float L = 0.f, v = 0.f;
        for (int t = 0; t < NTEAM; ++t) {
          const float* sw = slots + (t * RG + grp) * SLOT;
          const float sc = exp2f(sw[rl] - M);
          L += sc * sw[16 + rl];
          v += sc * sw[32 + rl * OSTR + d];
        }
        if (whole) {
          p.out[row_offset(p, u, row) + d] = L > 0.f ? v / L : 0.f;
        } else {
          if (d == 0) { part[row] = M; part[R + row] = L; }
          part[2 * R + row * D + d] = v;
        }
      }
      if (!whole) {
        // Publish this CTA's partial (one release by one thread after the
        // barrier); the last CTA of the unit to arrive merges them all.
        named_bar_sync(CBAR_CONS, CCONS);
        if (ct == 0) {
          __threadfence();
          flag[0] = atomicAdd(&p.unit_tickets[unit_index(p, u)], 1);
          __threadfence();
        }
        named_bar_sync(CBAR_CONS, CCONS);
        const int b0 = cta_of(u.ustart, T, P), b1 = cta_of(u.uend - 1, T, P);
        if (flag[0] == b1 - b0) {
          merge_unit_partials<16>(p, u, T, P, ct, CCONS, slots, CCW * SLOT,
                                  [] { named_bar_sync(CBAR_CONS, CCONS); });
          if (ct == 0) p.unit_tickets[unit_index(p, u)] = 0;
        }
      }
      if (has_next) load_query(unit_of_cached(x1, p, pre, sa, sfill));
      if constexpr (!OWN) {
        // The slots' generic-proxy accesses come before the producer's next
        // asynchronous copies into the same memory.
        fence_proxy_async();
      }
      named_bar_sync(CBAR_CONS, CCONS);
      if (!OWN && ct == 0) mbar_arrive(smem_u32(mdone));
      x = x1;
    }
  }
  __syncthreads();
  if (tid == 0 && *abort_flag) {
    // After an abort, no CTA exits with a copy still in flight into its shared
    // memory: wait (bounded) for the last NS stages this CTA issued.
    const int issued = flag[2];
    for (int j = max(0, issued - NS); j < issued; ++j)
      mbar_wait(smem_u32(full + (j % NS)), (j / NS) & 1);
  }
}

template <int D, bool ROTK>
static int chunk_stages(const Shape& sh, int R) {
  using C = ChunkCfg<D, ROTK>;
  const int rows16 = ((R + 15) / 16) * 16;
  const int nteam = CCW / ((R + 15) / 16);
  int ns = CH_MAX_STAGES;
  while (ns > nteam &&
         chunk_smem_bytes(C::STAGE, C::FINE, C::QSTR, rows16, ns, sh.S) > (size_t)SMEM_LIMIT)
    --ns;
  // The merge slots live in the stage memory.
  if ((size_t)ns * C::STAGE < (size_t)CCW * C::SLOT * 4) return 0;
  return ns;
}

// Stages with merge slots of their own, or 0 when fewer than
// CH_OWN_SLOTS_MIN_STAGES fit.
template <int D, bool ROTK>
static int chunk_stages_own(const Shape& sh, int R) {
  using C = ChunkCfg<D, ROTK>;
  const int rows16 = ((R + 15) / 16) * 16;
  int ns = CH_MAX_STAGES;
  while (ns >= CH_OWN_SLOTS_MIN_STAGES &&
         chunk_smem_bytes(C::STAGE, C::FINE, C::QSTR, rows16, ns, sh.S, CCW * C::SLOT * 4) >
             (size_t)SMEM_LIMIT)
    --ns;
  return ns >= CH_OWN_SLOTS_MIN_STAGES ? ns : 0;
}

template <int D, bool ROTK>
static size_t chunk_smem(const Shape& sh, int R) {
  using C = ChunkCfg<D, ROTK>;
  const int ns = chunk_stages<D, ROTK>(sh, R);
  return chunk_smem_bytes(C::STAGE, C::FINE, C::QSTR, ((R + 15) / 16) * 16, ns, sh.S);
}

bool attend_chunk_supported(const Shape& sh, int c) {
  const int R = c * sh.G;
  if (!(sh.bf16 && (sh.D == 64 || sh.D == 128) && c >= 2 && R <= CH_MAX_ROWS)) return false;
  const bool rotk = !sh.stored_rotated;
  int ns;
  size_t smem;
  if (sh.D == 128) {
    ns = rotk ? chunk_stages<128, true>(sh, R) : chunk_stages<128, false>(sh, R);
    smem = rotk ? chunk_smem<128, true>(sh, R) : chunk_smem<128, false>(sh, R);
  } else {
    ns = rotk ? chunk_stages<64, true>(sh, R) : chunk_stages<64, false>(sh, R);
    smem = rotk ? chunk_smem<64, true>(sh, R) : chunk_smem<64, false>(sh, R);
  }
  return ns >= CCW / ((R + 15) / 16) && smem <= (size_t)SMEM_LIMIT;
}

template <int D, bool ROTK, int STYLE>
static cudaError_t launch_chunk_t(const AttendParams& p0, const CUtensorMap& tk,
                                  const CUtensorMap& tv, int grid, cudaStream_t s) {
  using C = ChunkCfg<D, ROTK>;
  AttendParams p = p0;
  const int own = chunk_stages_own<D, ROTK>(p.sh, p.R);
  p.ns = own ? own : chunk_stages<D, ROTK>(p.sh, p.R);
  const size_t smem = own ? chunk_smem_bytes(C::STAGE, C::FINE, C::QSTR, ((p.R + 15) / 16) * 16,
                                             own, p.sh.S, CCW * C::SLOT * 4)
                          : chunk_smem<D, ROTK>(p.sh, p.R);
  auto kern = own ? attend_mma_chunk<D, ROTK, STYLE, true> : attend_mma_chunk<D, ROTK, STYLE, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(CH_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, tk, tv);
}

template <int D>
static cudaError_t launch_chunk_d(const AttendParams& p, const CUtensorMap& tk,
                                  const CUtensorMap& tv, int grid, cudaStream_t s) {
  const bool rotk = !p.sh.stored_rotated;
  if (p.sh.style == 0)
    return rotk ? launch_chunk_t<D, true, 0>(p, tk, tv, grid, s)
                : launch_chunk_t<D, false, 0>(p, tk, tv, grid, s);
  return rotk ? launch_chunk_t<D, true, 1>(p, tk, tv, grid, s)
              : launch_chunk_t<D, false, 1>(p, tk, tv, grid, s);
}

cudaError_t launch_attend_chunk(const AttendParams& p, const CUtensorMap& tk,
                                const CUtensorMap& tv, int grid, cudaStream_t s) {
  if (!attend_chunk_supported(p.sh, p.c)) return cudaErrorNotSupported;
  if (p.sh.D == 128) return launch_chunk_d<128>(p, tk, tv, grid, s);
  return launch_chunk_d<64>(p, tk, tv, grid, s);
}

}  // namespace rkv
