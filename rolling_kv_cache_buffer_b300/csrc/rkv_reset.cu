// rkv_reset.cu -- rkv_reset_stream: utterance reset of one stream, with an
// optional prefix (a constant prompt prepared once) at the start of its new
// window.
//
// "Audio8 ASR Infinite: What It Actually Takes to Listen Forever" resets the
// utterance state when the turn head predicts a completion (the flowchart of
// "Inside the Rolling KV Cache and Exact RoPE Re-Basing"), and the CPU runtime
// of "Reza2kn/Audio8-ASR-Infinite-Compressed" prepares an audio-independent
// prefix once and checks it again on every silence reset ("Linux CPU").
// Without pinned slots the prefix is the new window's first pairs, at
// re-based positions 0 .. n-1, and later appends evict it like any other pair.
// With P pinned slots it goes into slots 0 .. n-1, which no append touches,
// and the rolling window behind it starts empty.
#include <algorithm>

#include "rkv_handle.h"
#include "rkv_rows.cuh"

namespace rkv {
namespace {

struct ResetParams {
  Shape sh;
  StreamState* st;
  int s;               // the stream
  long long origin;    // its new origin
  int n;               // prefix pairs
  const void* k;       // [L][n][H_kv][D] of the cache type, keys before rotation
  const void* v;
  void* k_pool;
  void* v_pool;
  const float2* table;
};

// CTAs stride over the prefix's items.  Prefix pair j of row (l, j, g) goes to
// slot j (pinned) or P + ((origin + j) mod W_ring) = (origin + j) mod W (no
// pinned slots) of (s, l, g).  V rows and pre-RoPE keys are copied as raw
// 16-byte chunks; stored-rotated keys are rotated to their position j (in
// f32, rounded to the storage type, as the append kernel does), four pairs
// per item.  Thread 0 of CTA 0 writes the new state: nothing in this launch
// reads it, and the next kernel on the stream starts after this one has
// finished.
__global__ void __launch_bounds__(256) reset_stream_kernel(const ResetParams p) {
  const Shape& sh = p.sh;
  const int W = sh.W, D = sh.D, Hkv = sh.Hkv, Wg = sh.Wring;
  const int ring = static_cast<int>(p.origin % Wg);
  const bool bf = sh.bf16 != 0;
  const int esz = bf ? 2 : 4;
  const int chunks = D * esz / 16;                      // 16-byte chunks per row
  const int quads = D / 8;                              // rotation items per key
  const long long rows = (long long)sh.L * p.n * Hkv;
  // Items: the raw copies (V rows, and K rows unless they are rotated), then
  // the rotated keys.
  const long long raw = rows * chunks * (sh.stored_rotated ? 1 : 2);
  const long long items = raw + (sh.stored_rotated ? rows * quads : 0);
  auto slot_of = [&](int j) {
    if (sh.P) return j;
    return ring + j < Wg ? ring + j : ring + j - Wg;
  };
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < items;
       idx += (long long)gridDim.x * blockDim.x) {
    const bool rotk = idx >= raw;
    const long long it = rotk ? idx - raw : idx;
    const int per = rotk ? quads : chunks;
    const long long rowx = it / per;                   // (kv, row) for raw copies
    const int q = static_cast<int>(it % per);
    const bool is_v = !rotk && (sh.stored_rotated || rowx >= rows);
    const long long row = rotk ? rowx : (rowx >= rows ? rowx - rows : rowx);
    const int g = static_cast<int>(row % Hkv);
    const long long lj = row / Hkv;
    const int j = static_cast<int>(lj % p.n);
    const int l = static_cast<int>(lj / p.n);
    const size_t src = (size_t)row * D;
    const size_t dst = ((((size_t)p.s * sh.L + l) * Hkv + g) * W + slot_of(j)) * D;
    if (!rotk) {
      const uint4* from = reinterpret_cast<const uint4*>(
          static_cast<const uint8_t*>(is_v ? p.v : p.k) + src * esz) + q;
      uint4* to = reinterpret_cast<uint4*>(
          static_cast<uint8_t*>(is_v ? p.v_pool : p.k_pool) + dst * esz) + q;
      *to = __ldg(from);
    } else {
      const int i = q * 4;
      float ka[4], kb[4];
      load_pairs(p.k, src, i, D, sh.style, bf, ka, kb);
      float2 cs[4];
      load_cs4(p.table, (size_t)j * (D / 2), i, cs);
      rotate4(ka, kb, cs, 1.f);
      store_pairs(p.k_pool, dst, i, D, sh.style, bf, ka, kb);
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    StreamState ns{};   // status 0, lag 0
    ns.origin = p.origin;
    ns.fill = sh.P ? 0 : p.n;
    ns.ring = ring;
    ns.last_new = ns.fill;
    ns.npin = sh.P ? p.n : 0;
    p.st[p.s] = ns;
  }
}

bool aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

}  // namespace
}  // namespace rkv

rkv_status rkv_reset_stream(rkv_handle* h, int32_t s, int64_t origin, const void* k,
                            const void* v, int32_t n_prefix, void* stream) {
  if (!h || s < 0 || s >= h->sh.S || origin < 0 || n_prefix < 0 ||
      n_prefix > (h->sh.P ? h->sh.P : h->sh.Wr))
    return RKV_ERR_INVALID_ARG;
  if (n_prefix > 0 && (!k || !v || !rkv::aligned16(k) || !rkv::aligned16(v)))
    return RKV_ERR_INVALID_ARG;
  rkv::ResetParams p;
  p.sh = h->sh;
  p.st = h->state;
  p.s = s;
  p.origin = origin;
  p.n = n_prefix;
  p.k = k;
  p.v = v;
  p.k_pool = h->k_pool;
  p.v_pool = h->v_pool;
  p.table = reinterpret_cast<const float2*>(h->workspace + h->ws.table_off);
  const long long items = (long long)h->sh.L * n_prefix * h->sh.Hkv * (h->sh.D / 4);
  const long long grid = std::max(1LL, std::min((items + 255) / 256, 4LL * h->num_sms));
  rkv::reset_stream_kernel<<<(unsigned)grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
  h->last_launches = 1;
  return cudaGetLastError() == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
}
