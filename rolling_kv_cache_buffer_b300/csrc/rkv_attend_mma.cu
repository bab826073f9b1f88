// rkv_attend_mma.cu -- tensor-core decode attention over the rolling window
// (bf16 caches, one query token per stream, G = H_q/H_kv <= 8, D 64 or 128).
//
// What it computes is the attention over the window with exact re-basing of
// "Audio8 ASR Infinite: What It Actually Takes to Listen Forever" ("Inside the
// Rolling KV Cache and Exact RoPE Re-Basing"): for the query at r_q = fill - 1
// and every retained key at r = (slot - origin) mod W,
//   out = sum_r softmax(<R(r_q) q, R(r) k_r> * scale) v_r.
//
// The G query heads that share a KV head make S = Q K^T a dense contraction
// with M = G rows, and O^T = V^T P^T one with N = G columns, so both run on
// mma.sync m16n8k16 (bf16 operands, f32 accumulation):
//  * block of TK = 32 slots starting at slot blk*TK, whose first slot sits at
//    re-based position r0; slot d of the block is at r0 + d, or r0 + d - W
//    past the ring's end;
//  * keys are rotated in f32 by R(d) only (d < 32, a shared-memory table) and
//    rounded to bf16; the block offset goes into the query instead:
//    rows 0..7 of the A operand hold R(r_q - r0) q and rows 8..15 hold
//    R(r_q - r0 + W) q, so each key picks the row of its own base
//    (<R(a) q, R(b) k> depends only on b - a);
//  * the S accumulator fragment is exactly the B fragment P^T of the second
//    product, so probabilities never leave registers.
// Stored-rotated keys skip the key rotation and use R(r_q) q alone.
// K/V tiles come by 3-D TMA (128-byte swizzle) into a private 2-stage ring per
// warp, with the two (cos, sin) rows of the block's query rotations.
#include "rkv_attend_common.cuh"

namespace rkv {

namespace {

constexpr int MMA_NSW = 2;

template <int D, bool ROTK>
struct MmaCfg {
  static constexpr int TILE = TK * D * 2;                 // bf16 K (or V) tile
  static constexpr int NBOX = D / 64;                     // 128-byte boxes per row
  static constexpr int TROW = ROTK ? 2 * D * 4 : 0;       // two float2[D/2] table rows
  static constexpr int STAGE = ((2 * TILE + TROW + 1023) / 1024) * 1024;
  static constexpr int NGRP = D / 8;                      // 8-dim groups
  static constexpr int NKB = D / 16;                      // k-blocks of the QK product
  static constexpr int FINE = ROTK ? TK * (D / 2) * 8 : 0;  // fine (cos, sin) table
};

__device__ __forceinline__ uint32_t swz(int row, int grp) {
  const int box = grp >> 3, cq = grp & 7;
  return static_cast<uint32_t>(box * (TK * 128) + row * 128 + ((cq ^ (row & 7)) << 4));
}
// Fine table: row d (0..TK-1) holds (cos, sin)(d * w_i) for i < D/2, 16-byte
// chunks XOR-swizzled by (d & 7) so that 8 rows read together hit all banks.
__device__ __forceinline__ uint32_t fine_off(int d, int i) {
  const int q = i >> 1;
  return static_cast<uint32_t>(((q ^ (d & 7)) << 4) + ((i & 1) << 3));
}

__device__ __forceinline__ void rot(float& x, float& y, float c, float s) {
  const float a = x * c - y * s;
  y = y * c + x * s;
  x = a;
}

}  // namespace

template <int D, bool ROTK, int STYLE>
__global__ void __launch_bounds__(NWARP * 32, 1)
    attend_mma_decode(const __grid_constant__ AttendParams p,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV) {
  using C = MmaCfg<D, ROTK>;
  constexpr int NSW = MMA_NSW, TILE = C::TILE, NGRP = C::NGRP, NKB = C::NKB;
  constexpr int HALF = D / 2, HG = NGRP / 2;
  const int W = p.sh.W, NB = p.sh.NB, G = p.sh.G;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  uint8_t* stages = smem;                                               // [NWARP][NSW][STAGE]
  uint8_t* fine = stages + NWARP * NSW * C::STAGE;                      // [TK][D/2] float2
  uint64_t* bars = reinterpret_cast<uint64_t*>(fine + C::FINE);         // [NWARP][NSW]
  const int wstride = 8 * (D + 2);
  float* mrg = reinterpret_cast<float*>(bars + NWARP * NSW);            // [NWARP][wstride]
  int* flag = reinterpret_cast<int*>(mrg + NWARP * wstride);
  int* pre = flag + 4;

  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, cq = lane & 3;   // mma fragment coordinates
  if (tid == 0) {
    for (int i = 0; i < NWARP * NSW; ++i) mbar_init(smem_u32(bars + i), 1);
    fence_mbar_init();
  }
  if constexpr (ROTK) {
    for (int idx = tid; idx < TK * HALF; idx += blockDim.x) {
      const int d = idx / HALF, i = idx % HALF;
      *reinterpret_cast<float2*>(fine + d * HALF * 8 + fine_off(d, i)) =
          __ldg(p.table + (size_t)d * HALF + i);
    }
  }
  build_prefix(p, pre);
  __syncthreads();
  zero_empty_units(p);
  const int T = pre[p.sh.S];
  const int P = min(static_cast<int>(gridDim.x), T);
  const int b = static_cast<int>(blockIdx.x);
  const int rb = b < P ? range_start(b, T, P) : 0, re = b < P ? range_start(b + 1, T, P) : 0;

  uint8_t* my_st = stages + w * NSW * C::STAGE;
  uint64_t* my_bars = bars + w * NSW;
  float* my_m = mrg + w * wstride;

  WarpSeq iss;
  iss.init(rb, re, w);
  auto issue = [&](int slot_k) {
    int by;
    UnitRef ur;
    if (!iss.next(p, pre, by, ur)) return;
    const BlockGeo bg = block_geo(by, ur, W, NB);
    const int ug = static_cast<int>(unit_index(p, ur));
    const uint32_t bar = smem_u32(my_bars + slot_k);
    const uint32_t dst = smem_u32(my_st + slot_k * C::STAGE);
    mbar_arrive_expect_tx(bar, 2 * TILE + C::TROW);
#pragma unroll
    for (int bx = 0; bx < C::NBOX; ++bx) {
      tma_load_3d(dst + bx * TK * 128, &tmK, bx * 64, bg.blk * TK, ug, bar);
      tma_load_3d(dst + TILE + bx * TK * 128, &tmV, bx * 64, bg.blk * TK, ug, bar);
    }
    if constexpr (ROTK) {
      const int rq = ur.fill - 1;
      const int mA = rq - bg.r0, mB = mA + W;
      const float2* ta = p.table + (size_t)(mA < 0 ? -mA : mA) * HALF;
      const float2* tb = p.table + (size_t)mB * HALF;
      bulk_load(dst + 2 * TILE, ta, HALF * 8, bar);
      bulk_load(dst + 2 * TILE + HALF * 8, tb, HALF * 8, bar);
    }
  };
  if (lane == 0)
    for (int k = 0; k < NSW; ++k) issue(k);

  // The thread's query elements: head g, dims of its A fragments.
  //   k-block kb, j in {0,1,2,3}: dim 16kb + (j>>1)*8 + 2cq + (j&1)
  auto qdim = [&](int kb, int j) { return 16 * kb + (j >> 1) * 8 + 2 * cq + (j & 1); };

  bool dead = false;
  int k = 0;
  for (int x = rb; x < re;) {
    const UnitRef u = unit_of(x, p, pre);
    const int x1 = min(u.uend, re), n = x1 - x;
    const int cb = x + (w * n) / NWARP, ce = x + ((w + 1) * n) / NWARP;
    const int rq = u.fill - 1;

    float qf[NKB][4];                // raw query (f32), head g
    uint32_t qa[NKB][4];             // A fragments of the QK product
    float o[NKB][4];                 // O^T accumulators: m-tile = 16 dims
    float m_run = NEG_BIG, l_run = 0.f;
#pragma unroll
    for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
      for (int j = 0; j < 4; ++j) { o[kb][j] = 0.f; qf[kb][j] = 0.f; qa[kb][j] = 0u; }
    if (cb < ce && g < G) {
      const size_t qo = row_offset(p, u, g);
#pragma unroll
      for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
        for (int j = 0; j < 4; ++j) qf[kb][j] = load_elem(p.q, qo + qdim(kb, j), p.sh.q_bf16);
    }
    if constexpr (!ROTK) {
      // Stored-rotated keys sit at r already: one base, R(r_q) q.
      if (cb < ce && g < G) {
        const float2* t = p.table + (size_t)rq * HALF;
        float qr[NKB][4];
#pragma unroll
        for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
          for (int j = 0; j < 4; ++j) qr[kb][j] = qf[kb][j];
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
          qa[kb][1] = 0u;
          qa[kb][3] = 0u;
        }
      }
    }

    for (int y = cb; y < ce; ++y, ++k) {
      const int st = k % NSW;
      if (!dead && !mbar_wait(smem_u32(my_bars + st), (k / NSW) & 1)) {
        dead = true;
        if (lane == 0) p.st[u.s].status = STATUS_DEVICE_STATE;
      }
      if (!dead) {
        const uint8_t* kt = my_st + st * C::STAGE;
        const uint8_t* vt = kt + TILE;
        const uint32_t kt_s = smem_u32(kt), vt_s = smem_u32(vt);
        const BlockGeo bg = block_geo(y, u, W, NB);
        const int r0 = bg.r0;
        const int wrap_at = W - r0;               // keys d >= wrap_at use base B
        // ---- query fragments for this block's two bases ----
        if constexpr (ROTK) {
          if (g < G) {
            const float2* ta = reinterpret_cast<const float2*>(kt + 2 * TILE);
            const float2* tb = ta + HALF;
            const float sa = (rq - r0) < 0 ? -1.f : 1.f;
            float qA[NKB][4], qB[NKB][4];
#pragma unroll
            for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
              for (int j = 0; j < 4; ++j) { qA[kb][j] = qf[kb][j]; qB[kb][j] = qf[kb][j]; }
            if constexpr (STYLE == 0) {
#pragma unroll
              for (int kb = 0; kb < NKB / 2; ++kb)
#pragma unroll
                for (int j = 0; j < 4; j += 2) {
                  const int i = qdim(kb, j);
                  const float4 a = *reinterpret_cast<const float4*>(ta + i);
                  const float4 bb = *reinterpret_cast<const float4*>(tb + i);
                  rot(qA[kb][j], qA[kb + NKB / 2][j], a.x, sa * a.y);
                  rot(qA[kb][j + 1], qA[kb + NKB / 2][j + 1], a.z, sa * a.w);
                  rot(qB[kb][j], qB[kb + NKB / 2][j], bb.x, bb.y);
                  rot(qB[kb][j + 1], qB[kb + NKB / 2][j + 1], bb.z, bb.w);
                }
            } else {
#pragma unroll
              for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
                for (int j = 0; j < 4; j += 2) {
                  const int i = qdim(kb, j) >> 1;
                  const float2 a = ta[i], bb = tb[i];
                  rot(qA[kb][j], qA[kb][j + 1], a.x, sa * a.y);
                  rot(qB[kb][j], qB[kb][j + 1], bb.x, bb.y);
                }
            }
#pragma unroll
            for (int kb = 0; kb < NKB; ++kb) {
              qa[kb][0] = pack_bf2(qA[kb][0], qA[kb][1]);
              qa[kb][2] = pack_bf2(qA[kb][2], qA[kb][3]);
              qa[kb][1] = pack_bf2(qB[kb][0], qB[kb][1]);
              qa[kb][3] = pack_bf2(qB[kb][2], qB[kb][3]);
            }
          }
        }
        // ---- S = Q K^T per 8-key group; select each key's base ----
        float s[4][2];
        int nvalid = 0;
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) {
          uint32_t kf[NGRP];
          const int krow = nb * 8 + (lane & 7);
#pragma unroll
          for (int g4 = 0; g4 < NGRP; g4 += 4)
            ldsm_x4(kt_s + swz(krow, g4 + (lane >> 3)), kf[g4], kf[g4 + 1], kf[g4 + 2],
                    kf[g4 + 3]);
          if constexpr (ROTK) {
            const int dk = nb * 8 + g;          // this thread's key within the block
            const uint8_t* frow = fine + dk * HALF * 8;
            if constexpr (STYLE == 0) {
#pragma unroll
              for (int gr = 0; gr < HG; ++gr) {
                const int i = 8 * gr + 2 * cq;
                const float4 cs = *reinterpret_cast<const float4*>(frow + fine_off(dk, i));
                float x0 = bf_lo(kf[gr]), x1 = bf_hi(kf[gr]);
                float y0 = bf_lo(kf[gr + HG]), y1 = bf_hi(kf[gr + HG]);
                rot(x0, y0, cs.x, cs.y);
                rot(x1, y1, cs.z, cs.w);
                kf[gr] = pack_bf2(x0, x1);
                kf[gr + HG] = pack_bf2(y0, y1);
              }
            } else {
#pragma unroll
              for (int gr = 0; gr < NGRP; ++gr) {
                const int i = 4 * gr + cq;
                const float2 cs = *reinterpret_cast<const float2*>(frow + fine_off(dk, i));
                float x0 = bf_lo(kf[gr]), x1 = bf_hi(kf[gr]);
                rot(x0, x1, cs.x, cs.y);
                kf[gr] = pack_bf2(x0, x1);
              }
            }
          }
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kb = 0; kb < NKB; ++kb)
            mma_bf16(acc, qa[kb][0], qa[kb][1], qa[kb][2], qa[kb][3], kf[2 * kb], kf[2 * kb + 1]);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int d = nb * 8 + 2 * cq + e;
            const bool wr = ROTK && d >= wrap_at;
            int r = r0 + d;
            if (r >= W) r -= W;
            const bool vis = (r < u.fill) && (g < G);
            nvalid += (r < u.fill);
            s[nb][e] = vis ? (wr ? acc[2 + e] : acc[e]) * p.scale_log2 : NEG_BIG;
          }
        }
        // ---- online softmax for head g (the 4 lanes of quad g) ----
        float tmax = NEG_BIG;
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) tmax = fmaxf(tmax, fmaxf(s[nb][0], s[nb][1]));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
        const float mnew = fmaxf(m_run, tmax);
        const float alpha = exp2f(m_run - mnew);
        float pr[4][2];
        float psum = 0.f;
#pragma unroll
        for (int nb = 0; nb < 4; ++nb)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            pr[nb][e] = s[nb][e] > 0.5f * NEG_BIG ? exp2f(s[nb][e] - mnew) : 0.f;
            psum += pr[nb][e];
          }
        l_run = l_run * alpha + psum;
        m_run = mnew;
        const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * cq);      // head 2cq
        const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * cq + 4);  // head 2cq+1
#pragma unroll
        for (int mt = 0; mt < NKB; ++mt) {
          o[mt][0] *= a0; o[mt][1] *= a1; o[mt][2] *= a0; o[mt][3] *= a1;
        }
        // ---- O^T += V^T P^T ----
        const bool full = __all_sync(0xffffffffu, nvalid == 8);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const uint32_t b0 = pack_bf2(pr[2 * kk][0], pr[2 * kk][1]);
          const uint32_t b1 = pack_bf2(pr[2 * kk + 1][0], pr[2 * kk + 1][1]);
          // validity of the keys this thread's V^T elements belong to
          uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
          if (!full) {
            auto ok = [&](int d) {
              int r = r0 + d;
              if (r >= W) r -= W;
              return r < u.fill;
            };
            const int d0 = 16 * kk + 2 * cq;
            mlo = (ok(d0) ? 0x0000ffffu : 0u) | (ok(d0 + 1) ? 0xffff0000u : 0u);
            mhi = (ok(d0 + 8) ? 0x0000ffffu : 0u) | (ok(d0 + 9) ? 0xffff0000u : 0u);
          }
          const int vrow = 16 * kk + ((lane >> 4) << 3) + (lane & 7);
#pragma unroll
          for (int mt = 0; mt < NKB; ++mt) {
            uint32_t v0, v1, v2, v3;
            ldsm_x4_t(vt_s + swz(vrow, 2 * mt + ((lane >> 3) & 1)), v0, v1, v2, v3);
            mma_bf16(o[mt], v0 & mlo, v1 & mlo, v2 & mhi, v3 & mhi, b0, b1);
          }
        }
      }
      __syncwarp();
      if (lane == 0 && !dead) {
        fence_proxy_async();
        issue(st);
      }
    }

    // ---- segment end: warp partial -> shared (rows = heads), CTA merge ----
    float lsum = l_run;
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
    const int R = p.R;   // == G for decode
    if (cq == 0 && g < R) { my_m[g] = m_run; my_m[R + g] = lsum; }
#pragma unroll
    for (int mt = 0; mt < NKB; ++mt)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int h = 2 * cq + (j & 1);
        const int d = 16 * mt + g + ((j >> 1) << 3);
        if (h < R) my_m[2 * R + h * D + d] = o[mt][j];
      }
    __syncthreads();
    finish_segment(p, u, x, x1, rb, T, P, mrg, wstride, flag);
    __syncthreads();
    x = x1;
  }
  if (dead && lane == 0) {
    for (int i = 0; i < NSW; ++i) {
      const int kk = k + i;
      mbar_wait(smem_u32(my_bars + kk % NSW), (kk / NSW) & 1);
    }
  }
}

template <int D, bool ROTK>
static size_t mma_smem_t(int S) {
  using C = MmaCfg<D, ROTK>;
  size_t b = (size_t)NWARP * MMA_NSW * C::STAGE + C::FINE + NWARP * MMA_NSW * 8;
  b += (size_t)NWARP * 8 * (D + 2) * 4 + (4 + S + 1) * 4;
  return b + 1024;
}

size_t attend_mma_smem(const Shape& sh, int c) {
  (void)c;
  const bool rotk = !sh.stored_rotated;
  if (sh.D == 128) return rotk ? mma_smem_t<128, true>(sh.S) : mma_smem_t<128, false>(sh.S);
  return rotk ? mma_smem_t<64, true>(sh.S) : mma_smem_t<64, false>(sh.S);
}

bool attend_mma_supported(const Shape& sh, int c) {
  return sh.bf16 && sh.q_bf16 >= 0 && (sh.D == 64 || sh.D == 128) && sh.G <= 8 && c == 1;
}

template <int D, bool ROTK, int STYLE>
static cudaError_t launch_mma_t(const AttendParams& p, const CUtensorMap& tk,
                                const CUtensorMap& tv, int grid, cudaStream_t s) {
  const size_t smem = mma_smem_t<D, ROTK>(p.sh.S);
  auto kern = attend_mma_decode<D, ROTK, STYLE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, NWARP * 32, smem, s>>>(p, tk, tv);
  return cudaGetLastError();
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

}  // namespace rkv
