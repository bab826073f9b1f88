// rkv_attend_fma.cu -- CUDA-core attention over the rolling window (any query
// count c with c*G <= 16, bf16 or f32 storage, head_dim 64 or 128).
//
// Attention over the window with exact re-basing ("Audio8 ASR Infinite: What
// It Actually Takes to Listen Forever", "Inside the Rolling KV Cache and Exact
// RoPE Re-Basing"): key slot w holds position r = (w - origin) mod W, the
// query j of the step sits at r_j = fill - c + j, and
//   out = sum_{r <= r_j} softmax(<R(r_j) q, R(r) k_r> * scale) v_r.
// Pre-RoPE keys are rotated here in f32 with the (cos, sin) table row r;
// stored-rotated keys are used as stored.
//
// Mapping: one warp per block of TK = 32 slots; lane d owns key d for the dot
// products (the rotated queries are broadcast from shared memory) and owns
// D/32 output dims for P.V.  K/V tiles arrive by 3-D TMA (128-byte swizzle)
// into a private 2-stage ring per warp.
#include "rkv_attend_common.cuh"

namespace rkv {

namespace {

constexpr int FMA_NSW = 2;

template <int D, bool BF16>
struct FmaTile {
  static constexpr int ESZ = BF16 ? 2 : 4;
  static constexpr int E = 16 / ESZ;            // elements per 16-byte chunk
  static constexpr int NBOX = D * ESZ / 128;    // 128-byte boxes per row
  static constexpr int TILE = TK * D * ESZ;     // bytes of one K (or V) tile
  static constexpr int DPL = D / 32;            // output dims per lane
};

// Byte offset of 16-byte chunk q of row `row` in a 128B-swizzled tile.
__device__ __forceinline__ uint32_t swz(int row, int q) {
  const int box = q >> 3, cq = q & 7;
  return static_cast<uint32_t>(box * (TK * 128) + row * 128 + ((cq ^ (row & 7)) << 4));
}

template <bool BF16>
__device__ __forceinline__ void unpack_chunk(const uint8_t* p, float (&x)[BF16 ? 8 : 4]) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  if constexpr (BF16) {
    x[0] = bf_lo(v.x); x[1] = bf_hi(v.x); x[2] = bf_lo(v.y); x[3] = bf_hi(v.y);
    x[4] = bf_lo(v.z); x[5] = bf_hi(v.z); x[6] = bf_lo(v.w); x[7] = bf_hi(v.w);
  } else {
    x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
  }
}

}  // namespace

template <int D, bool BF16, int RMAX>
__global__ void __launch_bounds__(NWARP * 32, 1)
    attend_fma_kernel(const __grid_constant__ AttendParams p,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV) {
  using TT = FmaTile<D, BF16>;
  constexpr int E = TT::E, TILE = TT::TILE, DPL = TT::DPL, NSW = FMA_NSW;
  constexpr int HALF = D / 2;
  const int R = p.R, G = p.sh.G;
  const int style = p.sh.style;
  const bool rotk = !p.sh.stored_rotated;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  uint8_t* tiles = smem;                                             // [NWARP][NSW][K|V]
  uint64_t* bars = reinterpret_cast<uint64_t*>(tiles + NWARP * NSW * 2 * TILE);
  float* qs = reinterpret_cast<float*>(bars + NWARP * NSW);          // [NWARP][RMAX][D]
  float* pbuf = qs + NWARP * RMAX * D;                               // [NWARP][TK][RMAX]
  const int wstride = RMAX * (D + 2);
  float* mrg = pbuf + NWARP * TK * RMAX;                             // [NWARP][wstride]
  int* flag = reinterpret_cast<int*>(mrg + NWARP * wstride);         // [4]
  int* pre = flag + 4;                                               // [S+1]

  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < NWARP * NSW; ++i) mbar_init(smem_u32(bars + i), 1);
    fence_mbar_init();
  }
  build_prefix(p, pre);
  __syncthreads();
  zero_empty_units(p);
  const int T = pre[p.sh.S];
  // CTAs that share the blocks: at most one per block, so none has an empty range.
  const int P = min(static_cast<int>(gridDim.x), T);
  const int b = static_cast<int>(blockIdx.x);
  const int rb = b < P ? range_start(b, T, P) : 0, re = b < P ? range_start(b + 1, T, P) : 0;

  uint8_t* my_tiles = tiles + w * NSW * 2 * TILE;
  uint64_t* my_bars = bars + w * NSW;
  float* my_q = qs + w * RMAX * D;
  float* my_p = pbuf + w * TK * RMAX;
  float* my_m = mrg + w * wstride;

  // Issue side: lane 0 walks the warp's block sequence NSW blocks ahead.
  WarpSeq iss;
  iss.init(rb, re, w);
  auto issue = [&](int slot_k) {
    int by;
    UnitRef ur;
    if (!iss.next(p, pre, by, ur)) return;
    const BlockGeo bg = block_geo(by, ur, p.sh);
    const int ug = static_cast<int>(unit_index(p, ur));
    const uint32_t bar = smem_u32(my_bars + slot_k);
    const uint32_t kd = smem_u32(my_tiles + slot_k * 2 * TILE);
    mbar_arrive_expect_tx(bar, 2 * TILE);
#pragma unroll
    for (int bx = 0; bx < TT::NBOX; ++bx) {
      tma_load_3d(kd + bx * TK * 128, &tmK, bx * (128 / TT::ESZ), bg.blk * TK, ug, bar);
      tma_load_3d(kd + TILE + bx * TK * 128, &tmV, bx * (128 / TT::ESZ), bg.blk * TK, ug, bar);
    }
  };
  if (lane == 0)
    for (int k = 0; k < NSW; ++k) issue(k);

  bool dead = false;
  int k = 0;  // warp's block counter
  for (int x = rb; x < re;) {
    const UnitRef u = unit_of(x, p, pre);
    const int x1 = min(u.uend, re), n = x1 - x;
    const int cb = x + (w * n) / NWARP, ce = x + ((w + 1) * n) / NWARP;

    float m[RMAX], l[RMAX], o[RMAX][DPL];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      m[r] = NEG_BIG; l[r] = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[r][e] = 0.f;
    }
    if (cb < ce) {
      // Queries of this unit rotated to r_j = npin + fill - c + j (behind the
      // pinned prefix; + the stream's lag when stored-rotated keys follow a
      // re-basing epoch).
      const int lag = p.sh.epoch ? p.st[u.s].pending : 0;
      for (int idx = lane; idx < R * HALF; idx += 32) {
        const int row = idx / HALF, i = idx % HALF;
        const int rq = max(u.npin + u.fill - p.c + row / G, 0) + lag;
        const size_t qo = row_offset(p, u, row);
        const int d1 = pair_d1(i, D, style), d2 = pair_d2(i, D, style);
        const float a = load_elem(p.q, qo + d1, p.sh.q_bf16), b = load_elem(p.q, qo + d2, p.sh.q_bf16);
        const float2 cs = __ldg(p.table + (size_t)rq * HALF + i);
        my_q[row * D + d1] = a * cs.x - b * cs.y;
        my_q[row * D + d2] = b * cs.x + a * cs.y;
      }
      __syncwarp();
    }

    for (int y = cb; y < ce; ++y, ++k) {
      const int st = k % NSW;
      if (!dead && !mbar_wait(smem_u32(my_bars + st), (k / NSW) & 1)) {
        dead = true;
        if (lane == 0) p.st[u.s].status = STATUS_DEVICE_STATE;
      }
      if (!dead) {
        const uint8_t* kt = my_tiles + st * 2 * TILE;
        const uint8_t* vt = kt + TILE;
        const BlockGeo bg = block_geo(y, u, p.sh);
        const int r = slot_pos(bg, lane, p.sh.Wring);   // this lane's key position
        const bool valid = r < bg.lim;
        // ---- scores: lane = key ----
        float acc[RMAX];
#pragma unroll
        for (int rr = 0; rr < RMAX; ++rr) acc[rr] = 0.f;
        const float2* cs = p.table + (size_t)r * HALF;
        if (style == 0) {
#pragma unroll 2
          for (int q = 0; q < HALF / E; ++q) {
            float ka[E], kb[E];
            unpack_chunk<BF16>(kt + swz(lane, q), ka);
            unpack_chunk<BF16>(kt + swz(lane, q + HALF / E), kb);
            if (rotk) {
#pragma unroll
              for (int t = 0; t < E; ++t) {
                const float2 c = __ldg(cs + q * E + t);
                const float xa = ka[t], xb = kb[t];
                ka[t] = xa * c.x - xb * c.y;
                kb[t] = xb * c.x + xa * c.y;
              }
            }
#pragma unroll
            for (int rr = 0; rr < RMAX; ++rr) {
              if (rr < R) {
                const float* qa = my_q + rr * D + q * E;
                const float* qb = qa + HALF;
                float s = acc[rr];
#pragma unroll
                for (int t = 0; t < E; ++t) s = fmaf(qa[t], ka[t], fmaf(qb[t], kb[t], s));
                acc[rr] = s;
              }
            }
          }
        } else {
#pragma unroll 2
          for (int q = 0; q < D / E; ++q) {
            float kx[E];
            unpack_chunk<BF16>(kt + swz(lane, q), kx);
            if (rotk) {
#pragma unroll
              for (int t = 0; t < E / 2; ++t) {
                const float2 c = __ldg(cs + q * (E / 2) + t);
                const float xa = kx[2 * t], xb = kx[2 * t + 1];
                kx[2 * t] = xa * c.x - xb * c.y;
                kx[2 * t + 1] = xb * c.x + xa * c.y;
              }
            }
#pragma unroll
            for (int rr = 0; rr < RMAX; ++rr) {
              if (rr < R) {
                const float* qa = my_q + rr * D + q * E;
                float s = acc[rr];
#pragma unroll
                for (int t = 0; t < E; ++t) s = fmaf(qa[t], kx[t], s);
                acc[rr] = s;
              }
            }
          }
        }
        // ---- online softmax over the 32 keys (lanes) per row ----
        float alpha[RMAX];
#pragma unroll
        for (int rr = 0; rr < RMAX; ++rr) {
          if (rr < R) {
            const int rq = u.npin + u.fill - p.c + rr / G;
            const bool vis = valid && r <= rq;
            const float sc = vis ? acc[rr] * p.scale_log2 : NEG_BIG;
            const float mnew = fmaxf(m[rr], warp_max(sc));
            alpha[rr] = exp2f(m[rr] - mnew);
            const float pr = vis ? exp2f(sc - mnew) : 0.f;
            l[rr] = l[rr] * alpha[rr] + pr;
            m[rr] = mnew;
            my_p[lane * RMAX + rr] = pr;
          } else {
            alpha[rr] = 1.f;
          }
        }
        const unsigned vmask = __ballot_sync(0xffffffffu, valid);
        __syncwarp();
        // ---- P.V: lane owns dims lane*DPL .. +DPL ----
#pragma unroll
        for (int rr = 0; rr < RMAX; ++rr)
#pragma unroll
          for (int e = 0; e < DPL; ++e) o[rr][e] *= alpha[rr];
        const int d0 = lane * DPL;
        const int vq = d0 / E, voff = (d0 % E) * TT::ESZ;
        for (int key = 0; key < TK; ++key) {
          if (!((vmask >> key) & 1u)) continue;   // never touch slots outside the window
          float v[DPL];
          const uint8_t* vp = vt + swz(key, vq) + voff;
          if constexpr (BF16) {
            if constexpr (DPL == 4) {
              const uint2 wv = *reinterpret_cast<const uint2*>(vp);
              v[0] = bf_lo(wv.x); v[1] = bf_hi(wv.x); v[2] = bf_lo(wv.y); v[3] = bf_hi(wv.y);
            } else {
              const uint32_t wv = *reinterpret_cast<const uint32_t*>(vp);
              v[0] = bf_lo(wv); v[1] = bf_hi(wv);
            }
          } else {
#pragma unroll
            for (int e = 0; e < DPL; ++e) v[e] = reinterpret_cast<const float*>(vp)[e];
          }
          const float* pk = my_p + key * RMAX;
#pragma unroll
          for (int rr = 0; rr < RMAX; ++rr) {
            const float pr = pk[rr];
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[rr][e] = fmaf(pr, v[e], o[rr][e]);
          }
        }
      }
      __syncwarp();
      if (lane == 0 && !dead) {
        fence_proxy_async();
        issue(st);
      }
    }

    // ---- segment end: warp partial -> shared, CTA merge ----
#pragma unroll
    for (int rr = 0; rr < RMAX; ++rr) {
      const float lsum = warp_sum(l[rr]);
      if (rr < R) {
        if (lane == 0) { my_m[rr] = m[rr]; my_m[R + rr] = lsum; }
#pragma unroll
        for (int e = 0; e < DPL; ++e) my_m[2 * R + rr * D + lane * DPL + e] = o[rr][e];
      }
    }
    __syncthreads();
    finish_segment(p, u, x, x1, rb, T, P, mrg, wstride, flag);
    __syncthreads();
    x = x1;
  }
  // A warp that gave up on a wait lets its own copies in flight land first.
  if (dead && lane == 0) {
    for (int i = 0; i < NSW; ++i) {
      const int kk = k + i;
      mbar_wait(smem_u32(my_bars + kk % NSW), (kk / NSW) & 1);
    }
  }
}

template <int D, bool BF16, int RMAX>
static cudaError_t launch_fma_t(const AttendParams& p, const CUtensorMap& tk,
                                const CUtensorMap& tv, int grid, cudaStream_t s) {
  const size_t smem = attend_fma_smem(p.sh, RMAX);
  auto kern = attend_fma_kernel<D, BF16, RMAX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, NWARP * 32, smem, s>>>(p, tk, tv);
  return cudaGetLastError();
}

size_t attend_fma_smem(const Shape& sh, int rmax) {
  const int esz = sh.bf16 ? 2 : 4;
  const size_t tile = (size_t)TK * sh.D * esz;
  size_t b = NWARP * FMA_NSW * 2 * tile;
  b += NWARP * FMA_NSW * 8;
  b += (size_t)NWARP * rmax * sh.D * 4;
  b += (size_t)NWARP * TK * rmax * 4;
  b += (size_t)NWARP * rmax * (sh.D + 2) * 4;
  b += (4 + sh.S + 1) * 4;
  return b + 1024;  // alignment slack
}

template <int D, bool BF16>
static cudaError_t launch_fma_r(const AttendParams& p, const CUtensorMap& tk,
                                const CUtensorMap& tv, int grid, cudaStream_t s) {
  if (p.R <= 2) return launch_fma_t<D, BF16, 2>(p, tk, tv, grid, s);
  if (p.R <= 4) return launch_fma_t<D, BF16, 4>(p, tk, tv, grid, s);
  if (p.R <= 8) return launch_fma_t<D, BF16, 8>(p, tk, tv, grid, s);
  if (p.R <= 16) return launch_fma_t<D, BF16, 16>(p, tk, tv, grid, s);
  return cudaErrorNotSupported;
}

cudaError_t launch_attend_fma(const AttendParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              int grid, cudaStream_t s) {
  if (p.sh.D == 128 && p.sh.bf16) return launch_fma_r<128, true>(p, tk, tv, grid, s);
  if (p.sh.D == 64 && p.sh.bf16) return launch_fma_r<64, true>(p, tk, tv, grid, s);
  if (p.sh.D == 64 && !p.sh.bf16) return launch_fma_r<64, false>(p, tk, tv, grid, s);
  return cudaErrorNotSupported;
}

}  // namespace rkv
