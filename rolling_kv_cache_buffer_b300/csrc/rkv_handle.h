// rkv_handle.h -- definition of the opaque handle of include/rkv.h, shared by
// the host files of the library.  Not part of the public ABI.
#pragma once

#include <vector>

#include "rkv.h"
#include "rkv_internal.h"

struct rkv_handle {
  rkv_config cfg;
  rkv::Shape sh;
  rkv::WsLayout ws;
  void* k_pool;
  void* v_pool;
  rkv::StreamState* state;
  uint8_t* workspace;
  CUtensorMap tmK, tmV;     // 3-D views [units][W][D], boxes of 128 bytes x TK rows
  CUtensorMap tmK4, tmV4;   // bf16 pools: 4-D views, one box = a whole TK-row tile
  bool has_map4;
  int num_sms;
  int last_launches;
  float scale;
  std::vector<float2> host_table;  // kept alive until destroy
  std::vector<float4> host_table_g;
};

namespace rkv {
// Largest persistent grid of the attention kernels.
constexpr int kMaxCtas = 1024;
// Fewest blocks of a full window per CTA when a unit is split across CTAs.
constexpr int kMinBlocksPerCta = 8;

// Persistent grid of an attention call over n_layers layers.  The block list
// is cut into equal shares, CTA b taking [b*T/P, (b+1)*T/P).  With one stream
// every unit (layer, KV head) has the same number of blocks, so a grid of
// U*k CTAs (U units, k = #SMs / U) cuts each unit into exactly k equal parts:
// no CTA crosses a unit boundary and nothing is merged mid-stream.  With more
// units than SMs, a grid between 3/4 of the SMs and all of them that divides
// U gives every CTA whole units, again with nothing merged across CTAs (on
// B300 the encoder shape, 640 units of 24 blocks: 128 CTAs of 5 whole units
// take the step from 93.3 to 79.2 us against 148 CTAs that merge split
// units).  Several streams (fills unknown to the host) use one CTA per SM.
inline int attend_grid(const rkv_handle* h, int n_layers) {
  const int sms = h->num_sms < kMaxCtas ? h->num_sms : kMaxCtas;
  const int units = n_layers * h->sh.Hkv;
  if (h->sh.S == 1 && units <= sms) {
    // Every unit cut into the same number of CTAs, each with at least
    // kMinBlocksPerCta of a full window's blocks: a launch over few units (one
    // layer) streams its few MB from a few dozen SMs and merges few partials.
    int per = sms / units;
    const int cap = h->sh.NB / kMinBlocksPerCta;
    if (per > cap) per = cap > 1 ? cap : 1;
    return units * per;
  }
  if (h->sh.S == 1)
    for (int g = sms; g >= sms * 3 / 4; --g)
      if (units % g == 0) return g;
  return sms;
}

// Chunks of at least this many rows (c*G) run on tcgen05 under RKV_ATTEND_AUTO:
// below it most of the 128-row tile is padding and the mma.sync kernel wins
// (attention alone, measured on B300: 2 x 8 rows 59 us against 64 us, 3 x 8
// rows 61 against 86; 4 x 1 and 8 x 1 rows of the encoder shape 117 against
// 92-96 with split units, and the encoder's whole step 101 against 79 with
// whole units per CTA).
constexpr int kTcAutoMinRows = 16;

// Picks and launches the attention kernel for p.c queries per stream: the
// tensor-core kernels for bf16 caches (single query on mma.sync; a chunk on
// tcgen05 with RKV_ATTEND_TC, or with RKV_ATTEND_AUTO from kTcAutoMinRows
// rows, else on mma.sync for c*G <= 96 rows) unless the handle asks for the
// CUDA-core kernel, which serves f32 caches and c*G <= 16.
// RKV_ERR_UNSUPPORTED when no kernel takes the call.
inline rkv_status launch_attend_any(const rkv_handle* h, const AttendParams& p, int grid,
                                    cudaStream_t s) {
  const bool tc = h->cfg.attend_impl != RKV_ATTEND_FMA && h->has_map4;
  const bool want_tc = h->cfg.attend_impl == RKV_ATTEND_TC ||
                       (h->cfg.attend_impl == RKV_ATTEND_AUTO && p.R >= kTcAutoMinRows);
  cudaError_t e;
  if (tc && p.c == 1 && attend_mma_supported(h->sh, 1)) {
    e = launch_attend_mma(p, h->tmK4, h->tmV4, grid, s);
  } else if (want_tc && h->has_map4 && p.c > 1 && attend_tc_supported(h->sh, p.c)) {
    e = launch_attend_tc(p, h->tmK4, h->tmV4, grid, s);
  } else if (tc && p.c > 1 && attend_chunk_supported(h->sh, p.c)) {
    e = launch_attend_chunk(p, h->tmK4, h->tmV4, grid, s);
  } else {
    if (h->cfg.attend_impl == RKV_ATTEND_MMA || p.R > 16) return RKV_ERR_UNSUPPORTED;
    e = launch_attend_fma(p, h->tmK, h->tmV, grid, s);
  }
  if (e == cudaErrorNotSupported) return RKV_ERR_UNSUPPORTED;
  return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
}
}  // namespace rkv
