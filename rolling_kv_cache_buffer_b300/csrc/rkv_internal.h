// rkv_internal.h -- kernel parameter blocks and launchers shared by the host
// API (rkv_api.cu) and the kernel files.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "rkv_device.cuh"

namespace rkv {

// Division by a runtime constant d >= 1 for 0 <= x < 2^31, by multiply-high
// and shift (round-up reciprocal, the Granlund-Montgomery method).
struct FastDiv {
  uint32_t d, m, s;
  static FastDiv make(uint32_t d_) {
    FastDiv f;
    f.d = d_;
    f.s = 0;
    while ((1ull << f.s) < d_) ++f.s;
    f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << f.s) - d_)) / d_ + 1);
    return f;
  }
  __device__ __forceinline__ uint32_t div(uint32_t x) const {
    return static_cast<uint32_t>((static_cast<uint64_t>(__umulhi(x, m)) + x) >> s);
  }
};

// Geometry every kernel needs.
struct Shape {
  int S, L, Hq, Hkv, G, D, W, NB;  // W = slots per (stream, layer, KV head), NB = W / TK
  int P, NP;                       // pinned prefix slots 0..P-1, NP = P / TK blocks
  int Wring, NBr;                  // ring slots P..W-1: Wring = W - P, NBr = Wring / TK
  int Wr;                          // retained window (pairs kept), Wr <= Wring
  int bf16;                        // K/V pools hold bf16 (else f32)
  int q_bf16;                      // queries are bf16 (else f32)
  int style;                       // 0 split-half, 1 interleaved
  int stored_rotated;              // 1: keys kept rotated to (p - origin)
  int epoch;                       // stored-rotated lazy re-basing period E (0: every eviction)
};

__device__ __forceinline__ int state_ok(const StreamState& s, const Shape& sh) {
  return state_ok(s, sh.Wring, sh.Wr, sh.P);
}

// Workspace carve-up (byte offsets from the workspace base).
struct WsLayout {
  size_t table_off;        // float2 [2W][D/2]: (cos, sin)(m * w_i), m in [0, 2W)
  size_t table_g_off;      // float4 [2W][D/4]: the same, chunk j = (cos, cos, sin, sin) of
                           // pairs 2j and 2j+1 (the tcgen05 kernel's key rotation)
  size_t append_tk_off;    // int [S]  last-block tickets of the append kernel
  size_t rerot_tk_off;     // int [S]  last-block tickets of the re-rotation kernel
  size_t unit_tk_off;      // int [S*L*H_kv] tickets of split units (attention merge)
  size_t part_off;         // float [2 * max_ctas][slot_floats] split partials
  size_t total;
  int rmax;                // rows per unit a partial can hold (max_chunk * G)
  int slot_floats;         // rmax * (D + 2), rounded up to 4
  int max_ctas;
};

struct AppendParams {
  Shape sh;
  StreamState* st;
  const void* k_new;
  const void* v_new;
  void* k_pool;
  void* v_pool;
  long long* log;          // nullable, [S][4]
  int* tickets;            // [S] last-part tickets
  const float2* table;
  int c;                   // pairs appended this step
  FastDiv div_hkv, div_c;  // H_kv and c
};

struct RerotParams {
  Shape sh;
  StreamState* st;
  void* k_pool;
  int* tickets;
  const float2* table;
};

struct AttendParams {
  Shape sh;
  StreamState* st;
  const void* q;
  float* out;
  const float2* table;
  const float4* table_g;      // the table with each two pairs' cosines, then sines
  float* partials;
  int* unit_tickets;
  int layer_begin, L_att, c;  // layers of this call, queries per stream
  int R;                      // rows per unit = c * G
  int slot_floats;
  float scale_log2;           // softmax scale * log2(e)
  int ns;                     // pipeline stages (set by the launcher)
  // Fused decode step (rkv_step): the kernel also appends one pair per stream.
  int fused;                  // 0: attention only
  const void* k_new;          // [L][S][1][H_kv][D] of the cache type
  const void* v_new;
  void* k_pool;               // the pools (the fused step writes the new pair
  void* v_pool;               // into them; the attention reads them via TMA)
  long long* log;             // nullable, [S][4]
  int* step_ticket;           // one int: CTAs done with the step
  int publish;                // the step's last launch: publish the new states
};

cudaError_t launch_append(const AppendParams& p, cudaStream_t s);
cudaError_t launch_rerotate(const RerotParams& p, int blocks_per_stream, cudaStream_t s);
cudaError_t launch_set_state(StreamState* st, int s_idx, long long origin, int fill, int ring,
                             cudaStream_t s);

// Attention launchers; `grid` = persistent CTAs.  Return cudaErrorNotSupported
// when the shape has no instantiation.
cudaError_t launch_attend_fma(const AttendParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              int grid, cudaStream_t s);
cudaError_t launch_attend_mma(const AttendParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              int grid, cudaStream_t s);
// Fused decode step (append of one pair + pre-RoPE re-base + attention).
cudaError_t launch_step_mma(const AttendParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                            int grid, cudaStream_t s);
bool attend_mma_supported(const Shape& sh, int c);
// Tensor-core chunk attention (c >= 2 queries per stream, c*G <= 96 rows).
cudaError_t launch_attend_chunk(const AttendParams& p, const CUtensorMap& tk,
                                const CUtensorMap& tv, int grid, cudaStream_t s);
bool attend_chunk_supported(const Shape& sh, int c);
// Chunk attention on the tcgen05 tensor cores (c >= 2, c*G <= 128 rows).
cudaError_t launch_attend_tc(const AttendParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                             int grid, cudaStream_t s);
bool attend_tc_supported(const Shape& sh, int c);
size_t attend_fma_smem(const Shape& sh, int R);
size_t attend_mma_smem(const Shape& sh, int c);

}  // namespace rkv
