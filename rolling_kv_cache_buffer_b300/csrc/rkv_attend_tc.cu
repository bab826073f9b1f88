// rkv_attend_tc.cu -- chunk attention on the fifth-generation tensor cores
// (tcgen05, accumulators in tensor memory) for steps that insert c >= 2 tokens
// per stream: bf16 caches, R = c*G <= 128 query rows per (stream, layer, KV
// head) unit, D 64 or 128.
//
// What it computes is the attention over the window with exact re-basing of
// "Audio8 ASR Infinite: What It Actually Takes to Listen Forever" ("Inside the
// Rolling KV Cache and Exact RoPE Re-Basing"), causal among the chunk: query j
// sits at r_j = npin + fill - c + j and sees the keys at positions r <= r_j,
//   out_j = sum_{r <= r_j} softmax(<R(r_j) q_j, R(r) k_r> * scale) v_r.
//
// Per unit the rows (query j, head) form one M = 128 tile (rows >= R are
// zero), so S = Q K^T and O = P V are dense contractions issued as tcgen05.mma
// (kind::f16, bf16 operands, f32 accumulation in tensor memory):
//  * Q: [128 rows x D] bf16 in shared memory, K-major, 128-byte swizzle,
//    rotated once per unit by R(r_j) (plus the lag of stored-rotated keys
//    that follow a re-basing epoch);
//  * a key block (TK = 32 slots, one TMA box per tile, 128-byte swizzle) is
//    the B operand of S = Q K^T as it lands (stored-rotated keys) or after
//    the staging warps have turned each key in place to its position, R(r0+d)
//    = R(r0) R(d) composed in f32 (pre-RoPE keys), rounded to bf16;
//  * S (128 lanes x 32 columns f32, two buffers) is read by the softmax warps,
//    one row per thread: causal and window masks, running maximum with a lazy
//    rescale (O and l are rescaled only when the maximum grows by more than
//    2^8, which keeps every exponent below 2^8 and every partial sum exact
//    to f32 rounding), P = 2^(s - m) rounded to bf16 and written back to
//    tensor memory (two bf16 per column);
//  * O += P V takes P from tensor memory and the V tile from shared memory as
//    an MN-major operand (dims contiguous per key).
// A unit cut across CTAs is finished from their partials (m, l, O rows):
// when every unit is cut into exactly two CTAs, launched as a 2-CTA cluster,
// through distributed shared memory (rank 0 reads rank 1's); otherwise
// through global memory, by the last CTA to take the unit's ticket.
//
// Roles (one persistent CTA per SM, 16 warps): warp 0 the TMA producer (the
// stage ring of rkv_attend_pipe.cuh), warps 1-8 the softmax warps in two
// groups (warp w owns tensor-memory lanes 32 (w mod 4) .. +31), warps 10, 11,
// 14 and 15 the staging warps (they zero the V rows of slots outside the
// window and, for pre-RoPE keys, rotate the K tile), three MMA issuers (one
// lane each): warp 9 the products O += P V (the warp allocates and frees the
// tensor memory), warps 12 and 13 the products S = Q K^T of the first and the
// second key block of every step.  The staging warps sit on sub-partitions 2
// and 3, away from the softmax warps that hold rows when a unit has at most
// 64 (lane quarters 0 and 1: sub-partitions 0 and 1).  A tcgen05.mma costs the thread that issues
// it about a hundred cycles whatever its N (measured on B300), so one thread
// could not keep up with the twenty products of a 64-key step.  Every wait is
// bounded and falls back to the stream's status word.
#include "rkv_attend_pipe.cuh"

namespace rkv {

namespace {

constexpr int TC_SMW = 4;                       // softmax warps of one group
constexpr int TC_SMG = 2;                       // softmax groups (one stream of steps each)
constexpr int TC_RW = 4;                        // staging (rotation) warps
constexpr int TC_RG = 2;                        // staging groups (they take alternate blocks)
constexpr int W_SM0 = 1;
constexpr int W_MMA = 1 + TC_SMG * TC_SMW;       // P V issuer, owner of the tensor memory
constexpr int W_QK0 = W_MMA + 3;                 // Q K^T issuers: warps W_QK0, W_QK0 + 1
constexpr int TC_SMT = TC_SMG * TC_SMW * 32;    // softmax threads
// The staging warps: 10, 11, 14, 15.
__device__ __forceinline__ bool staging_warp(int w) { return (w & 2) && w > W_MMA; }
// Staging thread index (0 .. 127) of a thread of a staging warp: warps 10, 11
// form group 0, warps 14, 15 group 1.
__device__ __forceinline__ int staging_index(int tid) {
  const int w = tid >> 5;
  return ((w & 1) | (w >= W_QK0 + 2 ? 2 : 0)) * 32 + (tid & 31);
}
constexpr int TC_MAX_STAGES = 12;
constexpr int TC_ROWS = 128;                    // M of every product
constexpr int TBAR_PREFIX = 2;                  // named barrier: block prefix ready
constexpr int TBAR_SM = 3;                      // named barrier of the softmax warps
constexpr float TC_TAU = 8.f;                   // lazy rescale threshold (log2 units)
// A step of the softmax and of the products covers up to TC_KB key blocks
// (64 keys): S = Q K^T of the step's blocks lands side by side in one S
// buffer, the softmax reads it in two passes (maximum, then P), and O += P V
// takes the step's blocks one after the other.  Steps alternate between two
// streams, each with its own S, P and O in tensor memory and its own group
// of softmax warps (its own running maximum and sum), so that one group's
// softmax overlaps the other's; the two are combined row by row at the end
// of a segment.
constexpr int TC_KB = 2;
constexpr int TC_THREADS = 16 * 32;
static_assert(TC_KB == 2 && W_MMA == 9 && W_QK0 == 12, "warp roles");
// Tensor memory columns: S[2] (f32, TC_KB * TK each), P[2] (bf16 pairs,
// TC_KB * TK / 2 each), O[2] (f32, D columns each), one of each per stream.
constexpr int TM_SW = TC_KB * TK, TM_PW = TC_KB * TK / 2;
constexpr int TM_S = 0, TM_P = 2 * TM_SW, TM_O = TM_P + 2 * TM_PW, TM_COLS = 512;
static_assert(TM_O + 2 * 128 <= TM_COLS, "tensor memory columns");

template <int D, bool ROTK>
struct TcCfg : PipeCfg<D, ROTK> {
  static constexpr int QT = TC_ROWS * D * 2;    // Q tile bytes (D/64 boxes of 16 KB)
};

__host__ __device__ constexpr size_t tc_smem_bytes(int stage, int fine, int qt, int ns, int S) {
  // stages, Q tile, R(d) table, 3 barriers per stage, 13 more barriers, the
  // tensor memory address (16 B), flags (16 B), the per-stream cache.
  return 1024 + (size_t)ns * stage + (size_t)qt + (size_t)fine + (size_t)ns * 24 + 13 * 8 + 16 +
         16 + (size_t)(4 * S + 1) * 4;
}

// ---- tcgen05 wrappers ------------------------------------------------------
// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets, the sm_100 descriptor version (bit 46) and 128-byte swizzling.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// Instruction descriptor of kind::f16: f32 accumulator, bf16 A and B, A
// K-major, B K-major (tb = 0) or MN-major (tb = 1), M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int tb) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)tb << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void tc_mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                          int acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
               ::"r"(d), "l"(a), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void tc_mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id,
                                          int acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
               ::"r"(d), "r"(a), "l"(b), "r"(id), "r"(acc));
}
// The mbarrier completes once every tcgen05 operation this thread issued
// before it has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 columns of this warp's 32 lanes: thread t gets lane (base + t).
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// 2^x on the special-function unit (relative error about 2^-22; -inf gives 0):
// the softmax weights are rounded to bf16 right after.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Byte offset of element (row, col) of a K-major, 128-byte-swizzled tile of
// `rows` x 64 bf16 per box (col < 64 within the box).
__device__ __forceinline__ uint32_t swz128(int row, int col) {
  return static_cast<uint32_t>(row * 128 + ((((col * 2) >> 4) ^ (row & 7)) << 4) +
                               ((col * 2) & 15));
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
// Two rotary pairs (x0, y0), (x1, y1) -- X = (x0, x1), Y = (y0, y1) -- turned
// by the angle b + f: the cosines Bc and sines Bs of the base b of both pairs
// composed with those of f (angle addition), then x' = x c - y s,
// y' = y c + x s; ten packed f32x2 operations.
__device__ __forceinline__ void rot2_composed(f2& X, f2& Y, f2 Bc, f2 Bs, f2 Fc, f2 Fs) {
  const f2 Cc = f2_sub(f2_mul(Bc, Fc), f2_mul(Bs, Fs));
  const f2 Ss = f2_fma(Bc, Fs, f2_mul(Bs, Fc));
  const f2 Xr = f2_sub(f2_mul(X, Cc), f2_mul(Y, Ss));
  const f2 Yr = f2_fma(X, Ss, f2_mul(Y, Cc));
  X = Xr;
  Y = Yr;
}

// Staging warps, in TC_RG groups that take alternate blocks of the CTA's
// share (so that the load -> turn -> store chains of two blocks overlap): for
// every block of its group, in order, wait for its tiles, zero the V rows of slots outside the window (they may hold anything,
// and 0 * NaN would reach the output through P V), turn each key of the K
// tile in place to its position (pre-RoPE keys) -- slot d of the block at
// r0 + d, or r0 + d - W_ring past the ring's end -- and hand the stage on.  R(r0 + d) is the block's base row
// R(r0) (or R(r0 - W_ring): the stage's second row |r0 - W_ring|, its sine
// negated when r0 < W_ring) composed with R(d) from the resident table, both
// in the grouped layout (cosines of two pairs, then their sines).  Item
// `it` of a block is key d = it mod TK and group g = it / TK of eight rotary
// pairs: eight consecutive lanes take eight keys of one group, so their
// 16-byte reads of the swizzled tile and of the table fall in eight
// different bank groups and the base row is a broadcast.
template <int D, int STYLE, bool ROTK>
__device__ __forceinline__ void stage_tiles(const AttendParams& p, uint8_t* stages,
                                             const uint8_t* fine, uint64_t* full, uint64_t* rotd,
                                             const int* pre, const int* sa, const int* sfill,
                                             int rb, int re, volatile int* abort_flag, int rt) {
  using C = PipeCfg<D, ROTK>;
  constexpr int HALF = D / 2, NG = D / 16, ITEMS = TK * NG;
  constexpr int RT = TC_RW * 32 / TC_RG;   // threads of a group
  constexpr int VCH = D / 8;   // 16-byte chunks of a V row
  const int NS = p.ns, Wg = p.sh.Wring;
  const int lane = rt & 31, rg = rt / RT;
  rt -= rg * RT;
  int stage = 0, round = 0, jx = 0;
  for (int x = rb; x < re;) {
    const UnitRef u = unit_of_cached(x, p, pre, sa, sfill);
    const int x1 = min(u.uend, re);
    BlockWalk wk;
    wk.init(x, u, p.sh);
    for (bool first = true; x < x1; ++x, ++jx, first = false) {
      if (!first) wk.advance(1, u, p.sh);
      if (jx % TC_RG != rg) {   // the other group's block
        if (++stage == NS) { stage = 0; ++round; }
        continue;
      }
      // Every block passes through here in order, so the full barrier of a
      // stage is never more than one phase ahead of this wait.
      const bool bad = !mbar_wait_or_abort(smem_u32(full + stage), round & 1, abort_flag);
      if (__any_sync(0xffffffffu, bad)) {
        if (lane == 0 && !*abort_flag) {
          *abort_flag = 1;
          p.st[u.s].status = STATUS_DEVICE_STATE;
        }
        return;
      }
      uint8_t* kt = stages + (size_t)stage * C::STAGE;
      const int wrap_at = wk.g.wrap_at;
      // Slots outside the window may hold anything (NaN included): their V
      // rows are zeroed, since the product P V would turn 0 * NaN into NaN.
      // (Their K rows only reach masked scores.)
      const bool allvalid = wrap_at < TK ? (u.fill == Wg) : (wk.g.r0 + TK <= wk.g.lim);
      if (!allvalid) {
        for (int it = rt; it < TK * VCH; it += RT) {
          const int d = it % TK, ch = it / TK;
          if (slot_pos(wk.g, d, Wg) >= wk.g.lim)
            *reinterpret_cast<uint4*>(kt + C::TILE + tile_swz(d, ch)) = make_uint4(0, 0, 0, 0);
        }
      }
      if constexpr (ROTK) {
      const float4* base = reinterpret_cast<const float4*>(kt + 2 * C::TILE);   // R(r0)
      const float4* basew = base + HALF / 2;                                  // |r0 - W_ring|
      const bool neg = wk.g.r0 < Wg;
      static_assert(ITEMS % RT == 0, "every thread of a group takes the same number of items");
#pragma unroll
      for (int k0 = 0; k0 < ITEMS / RT; ++k0) {
        const int it = rt + k0 * RT;
        const int d = it & (TK - 1), g = it / TK;
        const bool wr = d >= wrap_at;
        const float4* bp = (wr ? basew : base) + 4 * g;
        const uint8_t* frow = fine + d * HALF * 8;
        const uint32_t offA = STYLE == 0 ? tile_swz(d, g) : tile_swz(d, 2 * g);
        const uint32_t offB = STYLE == 0 ? tile_swz(d, HALF / 8 + g) : tile_swz(d, 2 * g + 1);
        const uint4 A = *reinterpret_cast<const uint4*>(kt + offA);
        const uint4 B = *reinterpret_cast<const uint4*>(kt + offB);
        uint32_t w[8] = {A.x, A.y, A.z, A.w, B.x, B.y, B.z, B.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {   // pairs 8g + 2k and 8g + 2k + 1
          const float4 bb = bp[k];
          const float4 ff =
              *reinterpret_cast<const float4*>(frow + fine_chunk_rot(d, 4 * g + k));
          f2 Bs = f2_make(bb.z, bb.w);
          if (wr && neg) Bs = f2_mul(Bs, f2_make(-1.f, -1.f));
          // Split-half: x of the two pairs in word k of A, y in word k of B.
          // Interleaved: pair 8g + 2k + e is word 2k + e of A|B as (x, y).
          uint32_t& u0 = STYLE == 0 ? w[k] : w[2 * k];
          uint32_t& u1 = STYLE == 0 ? w[4 + k] : w[2 * k + 1];
          f2 X = STYLE == 0 ? f2_make(bf_lo(u0), bf_hi(u0)) : f2_make(bf_lo(u0), bf_lo(u1));
          f2 Y = STYLE == 0 ? f2_make(bf_lo(u1), bf_hi(u1)) : f2_make(bf_hi(u0), bf_hi(u1));
          rot2_composed(X, Y, f2_make(bb.x, bb.y), Bs, f2_make(ff.x, ff.y), f2_make(ff.z, ff.w));
          float x0, x1v, y0, y1;
          f2_split(X, x0, x1v);
          f2_split(Y, y0, y1);
          if (STYLE == 0) {
            u0 = pack_bf2(x0, x1v);
            u1 = pack_bf2(y0, y1);
          } else {
            u0 = pack_bf2(x0, y0);
            u1 = pack_bf2(x1v, y1);
          }
        }
        *reinterpret_cast<uint4*>(kt + offA) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(kt + offB) = make_uint4(w[4], w[5], w[6], w[7]);
      }
      }
      // The tensor cores read the tile through the async proxy.
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(rotd + stage));
      if (++stage == NS) { stage = 0; ++round; }
    }
  }
}

}  // namespace

// CL: the grid is one 2-CTA cluster per unit (every unit cut into exactly
// two CTAs).  Rank 1 leaves its partial (m, l and the unnormalised O rows) in
// its own stage memory, free once its one segment's products are done, and
// arrives on an mbarrier of rank 0; rank 0 reads it through distributed
// shared memory, folds it into its own rows and writes the output.
template <int D, bool ROTK, int STYLE, bool CL>
__global__ void __launch_bounds__(TC_THREADS, 1)
    attend_tc_chunk(const __grid_constant__ AttendParams p,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV) {
  using C = TcCfg<D, ROTK>;
  constexpr int HALF = D / 2, NKS = D / 16;   // k-steps of the QK product
  const int G = p.sh.G, NS = p.ns, R = p.R, c = p.c;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  uint8_t* stages = smem;                                        // [NS][STAGE]
  uint8_t* qt = stages + (size_t)NS * C::STAGE;                  // Q tile, 1024-aligned
  uint8_t* fine = qt + C::QT;                                    // R(d) table (pre-RoPE)
  uint64_t* full = reinterpret_cast<uint64_t*>(fine + C::FINE);  // [NS]
  uint64_t* empty = full + NS;                                   // [NS] stage consumed
  uint64_t* rotd = empty + NS;                                   // [NS] keys rotated
  uint64_t* sfull = rotd + NS;                                   // [2] S buffer written
  uint64_t* sfree = sfull + 2;                                   // [2] S buffer read
  uint64_t* pready = sfree + 2;                                  // [2] P buffer written
  uint64_t* qready = pready + 2;                                 // Q tile of the segment
  uint64_t* ofin = qready + 1;                                   // every product of a segment
  uint64_t* mdone = ofin + 1;                                    // a segment's products issued
  uint64_t* rxbar = mdone + 1;                                   // the peer's partial (CL)
  uint64_t* drain = rxbar + 1;                                   // [1 + TC_KB] issuers done
  uint32_t* tm_base = reinterpret_cast<uint32_t*>(drain + 1 + TC_KB);   // tensor memory address
  int* flag = reinterpret_cast<int*>(tm_base + 4);               // ticket, abort, issued
  int* pre = flag + 4;                                           // [S+1] block prefix
  int* sa = pre + p.sh.S + 1;                                    // [S] ring start | npin
  int* sfill = sa + p.sh.S;                                      // [S] fill
  int* slag = sfill + p.sh.S;                                    // [S] lag (epoch)
  volatile int* abort_flag = flag + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // The producer's first read after the dependency wait is the stream state:
  // bring it into L2 before anything else.
  prefetch_states(p);
  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(full + i), 1);
      mbar_init(smem_u32(empty + i), 1);      // the P V issuer's commit
      mbar_init(smem_u32(rotd + i), TC_RW / TC_RG);   // every warp of the block's group
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(sfull + i), TC_KB);   // every Q K^T issuer's commit
      mbar_init(smem_u32(sfree + i), TC_SMW);
      mbar_init(smem_u32(pready + i), TC_SMW);
    }
    mbar_init(smem_u32(qready), TC_SMG * TC_SMW);   // every softmax warp
    mbar_init(smem_u32(ofin), 1);
    mbar_init(smem_u32(mdone), 1);
    mbar_init(smem_u32(rxbar), TC_SMT);   // every softmax thread of rank 1
    for (int i = 0; i <= TC_KB; ++i) mbar_init(smem_u32(drain + i), 1);
    fence_mbar_init();
    flag[1] = 0;
    flag[2] = 0;
  }
  // Cluster barrier, phase 0: both CTAs have initialised their barriers once
  // it completes (waited on below, before any access to the peer).
  if constexpr (CL) cluster_arrive_relaxed();
  if (warp == W_MMA) {
    // The MMA warp owns the tensor memory: TM_COLS columns for the CTA.
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(tm_base)), "r"(TM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if constexpr (ROTK) {
    if (staging_warp(warp)) load_fine_rot<D>(p, fine, staging_index(tid), TC_RW * 32);
  }
  if (warp > 0) prefetch_queries(p, D, tid - 32, TC_THREADS - 32);
  pdl_wait();      // from here on: stream state, pools, queries, outputs
  pdl_trigger();   // a kernel launched next may start its own prologue
  tc_fence_before();
  if (warp == 0) {
    build_prefix_cached(p, pre, sa, sfill, lane, slag);
    __syncwarp();
    named_bar_arrive(TBAR_PREFIX, TC_THREADS);
  } else {
    named_bar_sync(TBAR_PREFIX, TC_THREADS);
  }
  tc_fence_after();
  if constexpr (CL) cluster_wait();
  const uint32_t tmem = *tm_base;
  const int T = pre[p.sh.S];
  const int P = min(static_cast<int>(gridDim.x), T);
  const int b = static_cast<int>(blockIdx.x);
  const int rb = b < P ? range_start(b, T, P) : 0, re = b < P ? range_start(b + 1, T, P) : 0;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0)
      flag[2] = produce<D, ROTK, ROTK ? KEY_BASES : NO_ROWS>(
          p, &tmK, &tmV, stages, full, empty, mdone, pre, sa, sfill, rb, re, abort_flag,
          reinterpret_cast<const float2*>(p.table_g));
    __syncwarp();
  } else if (staging_warp(warp)) {
    // ------------------------------------------------------------- staging warps
    stage_tiles<D, STYLE, ROTK>(p, stages, fine, full, rotd, pre, sa, sfill, rb, re, abort_flag,
                                staging_index(tid));
  } else if (warp == W_MMA || warp == W_QK0 || warp == W_QK0 + 1) {
    // -------------------------------------------------------------- MMA issuers
    // role -1: O += P V of every step (P from the step's P buffer, V from the
    // stages), each block's stage released by the commit after its products;
    // role i: S = Q K^T of block i of every step, over D in k-steps of 16 (32
    // bytes of a 128-byte row), into the block's 32 columns of the step's S
    // buffer.  Both Q K^T issuers commit to the S buffer's barrier (one with
    // nothing to issue commits all the same).
    if (lane == 0) {
      const int role = warp == W_MMA ? -1 : warp - W_QK0;
      const uint32_t id_qk = idesc_bf16(TC_ROWS, TK, 0);
      const uint32_t id_pv = idesc_bf16(TC_ROWS, D, 1);
      const uint32_t q_s = smem_u32(qt);
      uint64_t* ready = rotd;   // tiles staged (keys rotated, outside V rows zeroed)
      int jj = 0, t = 0, seg = 0;   // blocks and steps over the CTA, segments
      bool dead = false;
      auto wait = [&](uint64_t* bar, int parity) {
        if (!dead && !mbar_wait_or_abort(smem_u32(bar), parity, abort_flag)) dead = true;
        return !dead;
      };
      for (int x = rb; x < re && !dead; ++seg) {
        const UnitRef u = unit_of_cached(x, p, pre, sa, sfill);
        const int x1 = min(u.uend, re);
        if (role >= 0) {
          if (!wait(qready, seg & 1)) break;
          tc_fence_after();
        }
        bool first[2] = {true, true};   // each stream's first product into its O
        while (x < x1 && !dead) {
          const int nb = min(TC_KB, x1 - x), bs = t & 1;
          if (role >= 0) {
            // The S buffer was read by the softmax of step t - 2.
            if (t >= 2 && !wait(sfree + bs, ((t >> 1) - 1) & 1)) break;
            if (role < nb) {
              const int sb = (jj + role) % NS;
              if (!wait(ready + sb, ((jj + role) / NS) & 1)) break;
              tc_fence_after();
              const uint32_t k_s = smem_u32(stages + (size_t)sb * C::STAGE);
#pragma unroll
              for (int ks = 0; ks < NKS; ++ks) {
                const uint64_t a = sdesc(q_s + (ks >> 2) * (TC_ROWS * 128) + (ks & 3) * 32, 16, 1024);
                const uint64_t bd = sdesc(k_s + (ks >> 2) * (TK * 128) + (ks & 3) * 32, 16, 1024);
                tc_mma_ss(tmem + TM_S + bs * TM_SW + role * TK, a, bd, id_qk, ks > 0);
              }
            }
            tc_commit(smem_u32(sfull + bs));
          } else {
            if (!wait(pready + bs, (t >> 1) & 1)) break;
            tc_fence_after();
            for (int i = 0; i < nb; ++i) {
              const int sp = (jj + i) % NS;
              const uint32_t v_s = smem_u32(stages + (size_t)sp * C::STAGE + C::TILE);
#pragma unroll
              for (int ks = 0; ks < TK / 16; ++ks) {
                const uint64_t bd = sdesc(v_s + ks * 16 * 128, TK * 128, 1024);
                tc_mma_ts(tmem + TM_O + bs * D, tmem + TM_P + bs * TM_PW + i * (TK / 2) + ks * 8,
                          bd, id_pv, (first[bs] && i == 0 && ks == 0) ? 0 : 1);
              }
              tc_commit(smem_u32(empty + sp));
            }
            first[bs] = false;
          }
          jj += nb;
          x += nb;
          ++t;
        }
        if (dead) break;
        if (role < 0) {
          tc_commit(smem_u32(ofin));
          // The producer may go on with the next segment (its epilogue leaves
          // the stages alone).
          mbar_arrive(smem_u32(mdone));
        }
      }
      if (dead && !*abort_flag) {
        *abort_flag = 1;
        if (rb < re) p.st[unit_of_cached(rb, p, pre, sa, sfill).s].status = STATUS_DEVICE_STATE;
      }
      // Nothing leaves while this thread's products are in flight (after an
      // abort too): one last commit, waited on.
      tc_commit(smem_u32(drain + role + 1));
      mbar_wait(smem_u32(drain + role + 1), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps
    // Control flow is the same in all four warps (every decision below is
    // warp-uniform and the segment structure is shared), so the named
    // barriers of a split unit's merge are always reached by all of them,
    // also after a wait ran out (then the work is skipped, the barriers not).
    const int q4 = warp & 3;                  // tensor-memory lane quarter
    const int row = 32 * q4 + lane;           // this thread's row of every tile
    const uint32_t lane_addr = (uint32_t)(32 * q4) << 16;
    const int st = tid - 32 * W_SM0;          // 0 .. TC_SMT - 1
    const int grp = st / (TC_SMW * 32);       // the stream of steps this warp takes
    const bool warp_rows = 32 * q4 < R;       // the warp holds real rows
    zero_empty_units_cached(p, sa, sfill, st, TC_SMT);
    int jj = 0, t = 0, seg = 0;   // blocks and steps over the CTA, segments
    int jl1 = -1, jl2 = -1;       // the last blocks of the two previous steps
    bool dead = false;
    auto waited = [&](uint64_t* bar, int parity) {   // false (and dead) if it ran out
      if (dead) return false;
      if (__any_sync(0xffffffffu, !mbar_wait_or_abort(smem_u32(bar), parity, abort_flag))) {
        dead = true;
        if (lane == 0) *abort_flag = 1;   // the other roles stop waiting
      }
      return !dead;
    };
    for (int x = rb; x < re; ++seg) {
      const UnitRef u = unit_of_cached(x, p, pre, sa, sfill);
      const int x1 = min(u.uend, re);
      const bool whole = (x == u.ustart) && (x1 == u.uend);
      // A split unit's partial goes to slot 0 (the CTA's first segment) or 1;
      // in a cluster, rank 1 (the unit's second half) ships it to rank 0.
      const int kslot = x == rb ? 0 : 1;
      const bool ship = CL && !whole && x != u.ustart;
      const bool receive = CL && !whole && x == u.ustart;
      const int qbase = u.npin + u.fill - c;  // position of the chunk's first query
      const int rq = row < R ? qbase + row / G : -1;
      // ---- this segment's Q tile: row = (query j, head), rotated to r_j ----
      // (plus the lag of stored-rotated keys that follow a re-basing epoch);
      // rows >= R are zero.  The work is cut into chunks of eight rotary
      // pairs of one row (split-half pairs (i, i + D/2) from two 16-byte runs
      // of q, interleaved ones from one) dealt round-robin to every softmax
      // thread; each thread issues all the loads of a batch of its chunks
      // before it uses the first, so the tile costs one or two memory round
      // trips (the memory system is loaded by the stream, and dependent loads
      // would hold the segment's first product back by microseconds).
      {
        constexpr int NCK = STYLE == 0 ? HALF / 8 : D / 8;   // chunks per row
        constexpr int IB = STYLE == 0 ? 2 : 4;              // chunks per thread and batch
        auto qtile = [&](int r, int d0) {
          return reinterpret_cast<uint4*>(qt + (d0 >> 6) * (TC_ROWS * 128) + swz128(r, d0 & 63));
        };
        for (int i = st; i < (TC_ROWS - R) * (D / 8); i += TC_SMT)
          *qtile(R + i / (D / 8), 8 * (i % (D / 8))) = make_uint4(0, 0, 0, 0);
        auto load8 = [&](size_t off, float (&v)[8]) {
          if (p.sh.q_bf16) {
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(
                static_cast<const uint16_t*>(p.q) + off));
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) { v[2 * i] = bf_lo(ww[i]); v[2 * i + 1] = bf_hi(ww[i]); }
          } else {
            const float4* f = reinterpret_cast<const float4*>(static_cast<const float*>(p.q) + off);
            const float4 x0 = __ldg(f), x1v = __ldg(f + 1);
            v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
            v[4] = x1v.x; v[5] = x1v.y; v[6] = x1v.z; v[7] = x1v.w;
          }
        };
        auto store8 = [&](int r, int d0, const float (&v)[8]) {
          *qtile(r, d0) = make_uint4(pack_bf2(v[0], v[1]), pack_bf2(v[2], v[3]),
                                     pack_bf2(v[4], v[5]), pack_bf2(v[6], v[7]));
        };
        const int items = R * NCK;
#pragma unroll 1
        for (int i0 = st; i0 < items; i0 += IB * TC_SMT) {
          float xa[IB][8], xb[IB][8];
          float4 cs[IB][4];   // (cos, sin) of pairs 2k and 2k+1 = float4 k of a table row
#pragma unroll
          for (int k = 0; k < IB; ++k) {
            const int it = min(i0 + k * TC_SMT, items - 1);
            const int r = it / NCK, d0 = 8 * (it % NCK);
            const size_t qo = row_offset(p, u, r);
            const float4* tb = reinterpret_cast<const float4*>(
                p.table + (size_t)(qbase + r / G + slag[u.s]) * HALF);
            load8(qo + d0, xa[k]);
            if constexpr (STYLE == 0) {
              load8(qo + d0 + HALF, xb[k]);
#pragma unroll
              for (int e = 0; e < 4; ++e) cs[k][e] = __ldg(tb + d0 / 2 + e);
            } else {
              cs[k][0] = __ldg(tb + d0 / 4);
              cs[k][1] = __ldg(tb + d0 / 4 + 1);
            }
          }
#pragma unroll
          for (int k = 0; k < IB; ++k) {
            const int it = i0 + k * TC_SMT;
            if (it >= items) break;
            const int r = it / NCK, d0 = 8 * (it % NCK);
            if constexpr (STYLE == 0) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {   // pair d0 + i: (x, y) = (q[d0 + i], q[d0 + i + D/2])
                const float4 c4 = cs[k][i >> 1];
                const float cv = (i & 1) ? c4.z : c4.x, sv = (i & 1) ? c4.w : c4.y;
                const float x = xa[k][i], y = xb[k][i];
                xa[k][i] = x * cv - y * sv;
                xb[k][i] = y * cv + x * sv;
              }
              store8(r, d0, xa[k]);
              store8(r, d0 + HALF, xb[k]);
            } else {
#pragma unroll
              for (int i = 0; i < 4; ++i) {   // pair d0/2 + i: (x, y) = (q[d0 + 2i], q[d0 + 2i + 1])
                const float4 c4 = cs[k][i >> 1];
                const float cv = (i & 1) ? c4.z : c4.x, sv = (i & 1) ? c4.w : c4.y;
                const float x = xa[k][2 * i], y = xa[k][2 * i + 1];
                xa[k][2 * i] = x * cv - y * sv;
                xa[k][2 * i + 1] = y * cv + x * sv;
              }
              store8(r, d0, xa[k]);
            }
          }
        }
        // The tensor cores read the Q tile through the async proxy.
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(qready));
      }

      float m = NEG_BIG, l = 0.f;
      const int t0 = t;
      int nmine = 0;   // this group's steps in the segment
      BlockWalk wk;
      wk.init(x, u, p.sh);
      const int Wg = p.sh.Wring;
      // Scores of one block in log2 units; masked (-inf): outside the window
      // or after the row.  A block that holds no ring end, lies inside the
      // window and ends at or before the chunk's first query needs no mask.
      auto scores = [&](const BlockGeo& g, const uint32_t (&sr)[32], float (&sv)[32]) {
        if (g.wrap_at >= TK && g.r0 + TK <= g.lim && g.r0 + TK - 1 <= qbase) {
#pragma unroll
          for (int d = 0; d < 32; ++d) sv[d] = __uint_as_float(sr[d]) * p.scale_log2;
        } else {
#pragma unroll
          for (int d = 0; d < 32; ++d) {
            const int r = slot_pos(g, d, Wg);
            const bool vis = row < R && r < g.lim && r <= rq;
            sv[d] = vis ? __uint_as_float(sr[d]) * p.scale_log2 : -INFINITY;
          }
        }
      };
      auto load_s = [&](int col, uint32_t (&sr)[32]) {
        if (warp_rows) {
          tc_ld32(tmem + lane_addr + col, sr);
        } else {
#pragma unroll
          for (int d = 0; d < 32; ++d) sr[d] = 0u;
        }
      };
      for (bool first = true; x < x1; first = false) {
        const int nb = min(TC_KB, x1 - x), bs = t & 1;
        if (!first) wk.advance(TC_KB, u, p.sh);
        const int jl = jj + nb - 1;   // the step's last block
        auto next = [&]() {
          x += nb;
          jj += nb;
          ++t;
          jl2 = jl1;
          jl1 = jl;
        };
        if (bs != grp) { next(); continue; }   // the other stream's step
        ++nmine;
        if (!waited(sfull + bs, (t >> 1) & 1)) { next(); continue; }
        tc_fence_after();
        // A warp without real rows only keeps step with its group (its
        // arrivals below); its lanes of S, P and O are never used.
        if (warp_rows) {
        // One pass per block while no score exceeds the running maximum by
        // more than TC_TAU (the common case once a stream has had a step):
        // P = 2^(s - m) straight from the scores just read.  A block that
        // would move the maximum sends the whole step down the two-pass path
        // (maximum first, then P, which overwrites what was stored).
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
        bool quiet = t < 2;   // the P buffer and O are free (step t - 2 done)
        bool slow = false;
        {
          BlockWalk w = wk;
#pragma unroll 1
          for (int i = 0; i < nb; ++i) {
            if (i) w.advance(1, u, p.sh);
            uint32_t sr[32];
            float sv[32];
            load_s(TM_S + bs * TM_SW + i * TK, sr);
            scores(w.g, sr, sv);
            float mx[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
            for (int d = 4; d < 32; ++d) mx[d & 3] = fmaxf(mx[d & 3], sv[d]);
            const float bmi = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            if (__any_sync(0xffffffffu, bmi > m + TC_TAU)) { slow = true; break; }
            if (!quiet) {
              if (!waited(empty + jl2 % NS, (jl2 / NS) & 1)) break;
              tc_fence_after();
              quiet = true;
            }
            uint32_t pw[16];
#pragma unroll
            for (int d = 0; d < 32; d += 2) {
              const float p0 = ex2(sv[d] - m);
              const float p1 = ex2(sv[d + 1] - m);
              ps[(d >> 1) & 3] += p0 + p1;
              pw[d >> 1] = pack_bf2(p0, p1);
            }
            tc_st16(tmem + lane_addr + TM_P + bs * TM_PW + i * (TK / 2), pw);
          }
        }
        if (dead) { next(); continue; }
        if (slow) {
        ps[0] = ps[1] = ps[2] = ps[3] = 0.f;
        // Pass 1: the step's maximum.
        float bm = -INFINITY;
        {
          BlockWalk w = wk;
#pragma unroll 1
          for (int i = 0; i < nb; ++i) {
            if (i) w.advance(1, u, p.sh);
            uint32_t sr[32];
            float sv[32];
            load_s(TM_S + bs * TM_SW + i * TK, sr);
            scores(w.g, sr, sv);
            float mx[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
            for (int d = 4; d < 32; ++d) mx[d & 3] = fmaxf(mx[d & 3], sv[d]);
            bm = fmaxf(bm, fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])));
          }
        }
        // This stream's previous step (t - 2): its products read the P buffer
        // and wrote O; both are quiet once the commit after its last block
        // has completed.
        if (!quiet) {
          if (!waited(empty + jl2 % NS, (jl2 / NS) & 1)) { next(); continue; }
          tc_fence_after();
        }
        // Lazy rescale: the running maximum moves only when a score exceeds
        // it by more than TC_TAU; O and l are then rescaled (O holds products
        // of this segment once the stream had a step in it before).
        const bool grow = bm > m + TC_TAU;
        const float mnew = grow ? bm : m;
        if (__any_sync(0xffffffffu, grow && t >= t0 + 2)) {
          const float sc = ex2(m - mnew);
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 16) {
            uint32_t ov[16];
            tc_ld16(tmem + lane_addr + TM_O + bs * D + c0, ov);
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * sc);
            tc_st16(tmem + lane_addr + TM_O + bs * D + c0, ov);
          }
        }
        if (grow) l *= ex2(m - mnew);
        m = mnew;
        // Pass 2: P = 2^(s - m) (masked scores give 2^-inf = 0; m is always
        // finite), rounded to bf16, two per column of the P buffer.
        {
          BlockWalk w = wk;
#pragma unroll 1
          for (int i = 0; i < nb; ++i) {
            if (i) w.advance(1, u, p.sh);
            uint32_t sr[32];
            float sv[32];
            load_s(TM_S + bs * TM_SW + i * TK, sr);
            scores(w.g, sr, sv);
            uint32_t pw[16];
#pragma unroll
            for (int d = 0; d < 32; d += 2) {
              const float p0 = ex2(sv[d] - m);
              const float p1 = ex2(sv[d + 1] - m);
              ps[(d >> 1) & 3] += p0 + p1;
              pw[d >> 1] = pack_bf2(p0, p1);
            }
            tc_st16(tmem + lane_addr + TM_P + bs * TM_PW + i * (TK / 2), pw);
          }
        }
        }
        l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(sfree + bs));
          mbar_arrive(smem_u32(pready + bs));
        }
        next();
      }
      // ---- segment end: the two streams' rows combined, then the output ----
      // Each group publishes (m, l, steps) of its rows (in the Q tile, idle
      // until the next segment's), then group g writes columns
      // [g D/2, (g + 1) D/2) of every row:
      //   O = w_a O_a + w_b O_b,  l = w_a l_a + w_b l_b,  w = 2^(m - M),
      // M = max(m_a, m_b), a stream without steps in the segment left out.
      const bool fin = waited(ofin, seg & 1);
      tc_fence_after();
      float* xch = reinterpret_cast<float*>(qt);   // [2][3][128]
      xch[grp * 384 + row] = m;
      xch[grp * 384 + 128 + row] = l;
      xch[grp * 384 + 256 + row] = static_cast<float>(nmine);
      named_bar_sync(TBAR_SM, TC_SMT);
      // Rank 1's partial, in its stage memory: O rows first (16-byte chunk j
      // of row r at chunk j ^ (r mod 8), so that eight rows read at once hit
      // eight bank groups), then m, then l.
      auto rx_o = [&](int r, int col) {
        return static_cast<uint32_t>(4 * (r * D + ((((col >> 2) ^ (r & 7))) << 2)));
      };
      const uint32_t rx_m = static_cast<uint32_t>(4 * R * D), rx_l = rx_m + 4u * R;
      bool got = true;
      float M1 = NEG_BIG, L1 = 0.f;
      uint32_t peer = 0;
      if (receive) {
        got = false;
        for (uint32_t i = 0; i < WAIT_LIMIT && !got; ++i)
          got = mbar_try_wait_cluster(smem_u32(rxbar), 0);
        if (!got && st == 0) {
          *abort_flag = 1;
          p.st[u.s].status = STATUS_DEVICE_STATE;
        }
        peer = map_to_rank(smem_u32(stages), cluster_rank() ^ 1u);
        if (got && row < R) {
          M1 = ld_cluster_f32(peer + rx_m + 4u * row);
          L1 = ld_cluster_f32(peer + rx_l + 4u * row);
        }
      }
      if (fin && got) {
        const float ma = xch[row], la = xch[128 + row];
        const float mb = xch[384 + row], lb = xch[512 + row];
        const bool ha = xch[256 + row] > 0.f, hb = xch[640 + row] > 0.f;
        const float M = ha && hb ? fmaxf(ma, mb) : (ha ? ma : mb);
        const float wa = ha ? ex2(ma - M) : 0.f, wb = hb ? ex2(mb - M) : 0.f;
        float L = wa * la + wb * lb;
        // Rank 0: out = (s0 O + s1 O1) / (s0 L + s1 L1), s = 2^(m - max(M, M1)).
        float s0 = 1.f, s1 = 0.f;
        if (receive) {
          const float Mx = fmaxf(M, M1);
          s0 = ex2(M - Mx);
          s1 = ex2(M1 - Mx);
          L = s0 * L + s1 * L1;
        }
        constexpr int DH = D / 2;
#pragma unroll 1
        for (int c0 = grp * DH; c0 < (grp + 1) * DH; c0 += 16) {
          uint32_t oa[16], ob[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) oa[i] = ob[i] = 0u;
          if (warp_rows && ha) tc_ld16(tmem + lane_addr + TM_O + c0, oa);
          if (warp_rows && hb) tc_ld16(tmem + lane_addr + TM_O + D + c0, ob);
          float ov[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            ov[i] = (ha ? wa * __uint_as_float(oa[i]) : 0.f) +
                    (hb ? wb * __uint_as_float(ob[i]) : 0.f);
          if (row < R) {
            if (whole || receive) {
              const float inv = L > 0.f ? 1.f / L : 0.f;
              if (receive) {
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                  const float4 o1 = ld_cluster_f4(peer + rx_o(row, c0 + i));
                  ov[i] = s0 * ov[i] + s1 * o1.x;
                  ov[i + 1] = s0 * ov[i + 1] + s1 * o1.y;
                  ov[i + 2] = s0 * ov[i + 2] + s1 * o1.z;
                  ov[i + 3] = s0 * ov[i + 3] + s1 * o1.w;
                }
              }
              float* o = p.out + row_offset(p, u, row) + c0;
#pragma unroll
              for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4*>(o + i) =
                    make_float4(ov[i] * inv, ov[i + 1] * inv, ov[i + 2] * inv, ov[i + 3] * inv);
            } else if (ship) {
              uint8_t* rx = stages;
              if (c0 == 0) {
                *reinterpret_cast<float*>(rx + rx_m + 4 * row) = M;
                *reinterpret_cast<float*>(rx + rx_l + 4 * row) = L;
              }
#pragma unroll
              for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4*>(rx + rx_o(row, c0 + i)) =
                    make_float4(ov[i], ov[i + 1], ov[i + 2], ov[i + 3]);
            } else {
              // Split unit: this CTA's partial (m, l, unnormalised O) of the row.
              float* pp = p.partials + (size_t)(2 * b + kslot) * p.slot_floats;
              if (c0 == 0) { pp[row] = M; pp[R + row] = L; }
#pragma unroll
              for (int i = 0; i < 16; ++i) pp[2 * R + row * D + c0 + i] = ov[i];
            }
          }
        }
        tc_fence_before();
      }
      // Rank 1: every softmax thread releases its part of the partial.
      if (ship) mbar_arrive_remote(map_to_rank(smem_u32(rxbar), cluster_rank() ^ 1u));
      // The exchange area is the next segment's Q tile.
      named_bar_sync(TBAR_SM, TC_SMT);
      if (!whole && !CL) {
        // The last CTA of the unit to take its ticket merges the partials.
        named_bar_sync(TBAR_SM, TC_SMT);
        if (st == 0) {
          __threadfence();
          flag[0] = atomicAdd(&p.unit_tickets[unit_index(p, u)], 1);
          __threadfence();
        }
        named_bar_sync(TBAR_SM, TC_SMT);
        const int b0 = cta_of(u.ustart, T, P), b1 = cta_of(u.uend - 1, T, P);
        if (flag[0] == b1 - b0) {
          merge_unit_partials<8>(p, u, T, P, st, TC_SMT, reinterpret_cast<float*>(qt),
                                 C::QT / 4, [] { named_bar_sync(TBAR_SM, TC_SMT); });
          if (st == 0) p.unit_tickets[unit_index(p, u)] = 0;
        }
        named_bar_sync(TBAR_SM, TC_SMT);
      }
      x = x1;
    }
    if (dead && lane == 0 && !*abort_flag) {
      *abort_flag = 1;
      if (rb < re) p.st[unit_of_cached(rb, p, pre, sa, sfill).s].status = STATUS_DEVICE_STATE;
    }
  }
  tc_fence_before();
  // In a cluster neither CTA leaves while its peer may still read its memory.
  if constexpr (CL) cluster_sync_all(); else __syncthreads();
  tc_fence_after();
  if (warp == W_MMA) {
    // Every issuer drained its products before the barrier above.
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 ::"r"(tmem), "r"(TM_COLS));
  }
  if (tid == 0 && *abort_flag) {
    const int issued = flag[2];
    for (int j = max(0, issued - NS); j < issued; ++j)
      mbar_wait(smem_u32(full + (j % NS)), (j / NS) & 1);
  }
}

// ---------------------------------------------------------------------------
// Launch
// ---------------------------------------------------------------------------
template <int D, bool ROTK>
static int tc_stages(int S) {
  using C = TcCfg<D, ROTK>;
  int ns = TC_MAX_STAGES;
  while (ns > 2 && tc_smem_bytes(C::STAGE, C::FINE, C::QT, ns, S) > (size_t)SMEM_LIMIT) --ns;
  return ns;
}

bool attend_tc_supported(const Shape& sh, int c) {
  if (!(sh.bf16 && (sh.D == 64 || sh.D == 128) && c >= 2 && c * sh.G <= TC_ROWS)) return false;
  // A softmax group waits on the release of its previous step's last stage;
  // that stage must not be reused by the next three steps (the other
  // stream's step may complete meanwhile): at least 3 TC_KB + 1 stages.
  const bool rotk = !sh.stored_rotated;
  constexpr int need = 3 * TC_KB + 1;
  if (sh.D == 128)
    return rotk ? tc_stages<128, true>(sh.S) >= need : tc_stages<128, false>(sh.S) >= need;
  return rotk ? tc_stages<64, true>(sh.S) >= need : tc_stages<64, false>(sh.S) >= need;
}

template <int D, bool ROTK, int STYLE, bool CL>
static cudaError_t launch_tc_k(const AttendParams& p0, const CUtensorMap& tk,
                               const CUtensorMap& tv, int grid, cudaStream_t s) {
  using C = TcCfg<D, ROTK>;
  AttendParams p = p0;
  p.ns = tc_stages<D, ROTK>(p.sh.S);
  const size_t smem = tc_smem_bytes(C::STAGE, C::FINE, C::QT, p.ns, p.sh.S);
  if (smem > (size_t)SMEM_LIMIT) return cudaErrorNotSupported;
  auto kern = attend_tc_chunk<D, ROTK, STYLE, CL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(TC_THREADS);
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
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, p, tk, tv);
}

// The two CTAs that share a unit merge through distributed shared memory
// when every unit is cut into exactly two CTAs (one stream, grid = 2 units)
// and rank 1's partial (R rows of D floats, m and l) fits in its stages.
template <int D, bool ROTK>
static bool tc_cluster_merge(const AttendParams& p, int grid) {
  using C = TcCfg<D, ROTK>;
  return p.sh.S == 1 && grid == 2 * p.L_att * p.sh.Hkv &&
         (size_t)tc_stages<D, ROTK>(p.sh.S) * C::STAGE >= (size_t)(p.R * D + 2 * p.R) * 4;
}

template <int D, bool ROTK, int STYLE>
static cudaError_t launch_tc_s(const AttendParams& p, const CUtensorMap& tk,
                               const CUtensorMap& tv, int grid, cudaStream_t s) {
  return tc_cluster_merge<D, ROTK>(p, grid) ? launch_tc_k<D, ROTK, STYLE, true>(p, tk, tv, grid, s)
                                            : launch_tc_k<D, ROTK, STYLE, false>(p, tk, tv, grid, s);
}

template <int D>
static cudaError_t launch_tc_d(const AttendParams& p, const CUtensorMap& tk,
                               const CUtensorMap& tv, int grid, cudaStream_t s) {
  const bool rotk = !p.sh.stored_rotated;
  if (p.sh.style == 0)
    return rotk ? launch_tc_s<D, true, 0>(p, tk, tv, grid, s)
                : launch_tc_s<D, false, 0>(p, tk, tv, grid, s);
  return rotk ? launch_tc_s<D, true, 1>(p, tk, tv, grid, s)
              : launch_tc_s<D, false, 1>(p, tk, tv, grid, s);
}

cudaError_t launch_attend_tc(const AttendParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                             int grid, cudaStream_t s) {
  if (!attend_tc_supported(p.sh, p.c)) return cudaErrorNotSupported;
  if (p.sh.D == 128) return launch_tc_d<128>(p, tk, tv, grid, s);
  return launch_tc_d<64>(p, tk, tv, grid, s);
}

}  // namespace rkv
