// rkv_api.cu -- the C ABI declared in include/rkv.h: argument checks, the
// handle, workspace carve-up, TMA descriptors and kernel launches.  No call
// allocates device memory; only rkv_get_stream_state waits for the device.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "rkv_handle.h"

using rkv::Shape;
using rkv::WsLayout;

namespace {

using rkv::kMaxCtas;
constexpr int kMaxStreams = 1024;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

rkv_status check_config(const rkv_config* c) {
  if (!c) return RKV_ERR_INVALID_ARG;
  if (c->n_streams < 1 || c->n_layers < 1 || c->n_kv_heads < 1 || c->n_q_heads < 1 ||
      c->head_dim < 1 || c->capacity < 1 || c->max_chunk < 1 || c->rebase_epoch < 0 ||
      c->n_pinned < 0 || c->n_pinned >= c->capacity || c->n_pinned % rkv::TK ||
      c->window < 0 || c->window > c->capacity - c->n_pinned)
    return RKV_ERR_INVALID_ARG;
  if (c->n_q_heads % c->n_kv_heads) return RKV_ERR_INVALID_ARG;
  if (!(c->rope_theta > 1.0) || !std::isfinite(c->rope_theta)) return RKV_ERR_INVALID_ARG;
  if (c->softmax_scale < 0.f || !std::isfinite(c->softmax_scale)) return RKV_ERR_INVALID_ARG;
  if (c->kv_dtype != RKV_BF16 && c->kv_dtype != RKV_F32) return RKV_ERR_INVALID_ARG;
  if (c->q_dtype != RKV_BF16 && c->q_dtype != RKV_F32) return RKV_ERR_INVALID_ARG;
  if (c->layout != RKV_PRE_ROPE && c->layout != RKV_STORED_ROTATED) return RKV_ERR_INVALID_ARG;
  if (c->rope_style != RKV_ROPE_SPLIT_HALF && c->rope_style != RKV_ROPE_INTERLEAVED)
    return RKV_ERR_INVALID_ARG;
  if (c->attend_impl < RKV_ATTEND_AUTO || c->attend_impl > RKV_ATTEND_TC)
    return RKV_ERR_INVALID_ARG;
  // Retained window: by default every ring slot (those behind the pinned ones).
  const int wr = c->window ? c->window : c->capacity - c->n_pinned;
  if (c->max_chunk > wr) return RKV_ERR_CAPACITY;
  // Lazy re-basing: positions p - o_ref stay below 2W (the RoPE table's rows).
  if (c->rebase_epoch >= 2 &&
      (c->layout != RKV_STORED_ROTATED || c->rebase_epoch + c->max_chunk > wr + 1))
    return RKV_ERR_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return RKV_ERR_UNSUPPORTED;
  // A pinned key would need the lag in its own position too: not built.
  if (c->n_pinned && c->rebase_epoch >= 2) return RKV_ERR_UNSUPPORTED;
  if (c->capacity % rkv::TK || c->capacity > 65536) return RKV_ERR_UNSUPPORTED;
  if (c->n_streams > kMaxStreams) return RKV_ERR_UNSUPPORTED;
  if (c->kv_dtype == RKV_F32 && c->head_dim == 128) return RKV_ERR_UNSUPPORTED;
  const long long units = (long long)c->n_streams * c->n_layers * c->n_kv_heads;
  if (units * (c->capacity / rkv::TK) >= (1LL << 31)) return RKV_ERR_UNSUPPORTED;
  // The re-rotation kernel indexes a stream's work items in int32.
  if ((long long)c->n_layers * c->n_kv_heads * c->capacity * (c->head_dim / 8) >= (1LL << 31))
    return RKV_ERR_UNSUPPORTED;
  return RKV_OK;
}

Shape make_shape(const rkv_config* c) {
  Shape s;
  s.S = c->n_streams;
  s.L = c->n_layers;
  s.Hq = c->n_q_heads;
  s.Hkv = c->n_kv_heads;
  s.G = c->n_q_heads / c->n_kv_heads;
  s.D = c->head_dim;
  s.W = c->capacity;
  s.NB = c->capacity / rkv::TK;
  s.P = c->n_pinned;
  s.NP = c->n_pinned / rkv::TK;
  s.Wring = c->capacity - c->n_pinned;
  s.NBr = s.Wring / rkv::TK;
  s.Wr = c->window ? c->window : s.Wring;
  s.bf16 = c->kv_dtype == RKV_BF16;
  s.q_bf16 = c->q_dtype == RKV_BF16;
  s.style = c->rope_style;
  s.stored_rotated = c->layout == RKV_STORED_ROTATED;
  s.epoch = (s.stored_rotated && c->rebase_epoch >= 2) ? c->rebase_epoch : 0;
  return s;
}

WsLayout make_layout(const rkv_config* c) {
  WsLayout w;
  const Shape s = make_shape(c);
  size_t off = 0;
  w.table_off = off;
  off = align_up(off + (size_t)2 * s.W * (s.D / 2) * sizeof(float2), 256);
  w.table_g_off = off;
  off = align_up(off + (size_t)2 * s.W * (s.D / 2) * sizeof(float2), 256);
  w.append_tk_off = off;
  off = align_up(off + (size_t)s.S * 4, 256);
  w.rerot_tk_off = off;
  off = align_up(off + (size_t)s.S * 4, 256);
  w.unit_tk_off = off;
  off = align_up(off + (size_t)s.S * s.L * s.Hkv * 4, 256);
  w.rmax = c->max_chunk * s.G;
  w.slot_floats = static_cast<int>(align_up((size_t)w.rmax * (s.D + 2), 4));
  w.max_ctas = kMaxCtas;
  w.part_off = off;
  off = align_up(off + (size_t)2 * kMaxCtas * w.slot_floats * 4, 256);
  w.total = off;
  return w;
}

rkv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA; }

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 3-D view [units][W][D] of a pool; box = 128 bytes of one row x TK rows.
bool make_pool_map(CUtensorMap* tm, void* pool, const Shape& s) {
  auto enc = get_encode();
  if (!enc) return false;
  const int esz = s.bf16 ? 2 : 4;
  cuuint64_t dims[3] = {(cuuint64_t)s.D, (cuuint64_t)s.W, (cuuint64_t)s.S * s.L * s.Hkv};
  cuuint64_t strides[2] = {(cuuint64_t)s.D * esz, (cuuint64_t)s.W * s.D * esz};
  cuuint32_t box[3] = {(cuuint32_t)(128 / esz), (cuuint32_t)rkv::TK, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(tm, s.bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                   3, pool, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D view of a bf16 pool for whole-tile boxes: dims {64 elements, W rows,
// D/64 row halves, units} with strides {2D bytes, 128 bytes, 2WD bytes}; a box
// {64, TK, D/64, 1} (the keys of one block) lands in shared memory as D/64
// pieces of TK rows x 128 bytes one after the other.
bool make_pool_map4(CUtensorMap* tm, void* pool, const Shape& s) {
  auto enc = get_encode();
  if (!enc || !s.bf16) return false;
  const int nbox = s.D / 64;
  cuuint64_t dims[4] = {64, (cuuint64_t)s.W, (cuuint64_t)nbox, (cuuint64_t)s.S * s.L * s.Hkv};
  cuuint64_t strides[3] = {(cuuint64_t)s.D * 2, 128, (cuuint64_t)s.W * s.D * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)rkv::TK, (cuuint32_t)nbox, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, pool, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// (cos, sin)(m * w_i), w_i = theta^(-2i/D), for m in [0, 2W): computed in
// float64 and rounded to float32.
std::vector<float2> make_table(const Shape& s, double theta) {
  const int half = s.D / 2;
  std::vector<float2> t((size_t)2 * s.W * half);
  std::vector<double> w(half);
  for (int i = 0; i < half; ++i) w[i] = std::pow(theta, -2.0 * i / s.D);
  for (int m = 0; m < 2 * s.W; ++m)
    for (int i = 0; i < half; ++i) {
      const double a = (double)m * w[i];
      t[(size_t)m * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
    }
  return t;
}

// The same rows regrouped: chunk j of a row = (cos, cos, sin, sin) of pairs 2j
// and 2j+1, so that packed f32x2 arithmetic finds the two cosines (sines) of
// a chunk in one register pair.
std::vector<float4> group_table(const std::vector<float2>& t, const Shape& s) {
  const int half = s.D / 2;
  std::vector<float4> g(t.size() / 2);
  for (size_t m = 0; m < (size_t)2 * s.W; ++m)
    for (int j = 0; j < half / 2; ++j) {
      const float2 a = t[m * half + 2 * j], b = t[m * half + 2 * j + 1];
      g[m * (half / 2) + j] = make_float4(a.x, b.x, a.y, b.y);
    }
  return g;
}

}  // namespace

extern "C" {

int32_t rkv_abi_version(void) { return RKV_ABI_VERSION; }

const char* rkv_status_string(rkv_status s) {
  switch (s) {
    case RKV_OK: return "ok";
    case RKV_ERR_INVALID_ARG: return "invalid argument";
    case RKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case RKV_ERR_CAPACITY: return "more new tokens than the capacity";
    case RKV_ERR_CUDA: return "CUDA error";
    case RKV_ERR_DEVICE_STATE: return "device-side stream status set";
  }
  return "unknown status";
}

rkv_status rkv_required_bytes(const rkv_config* cfg, size_t* kv_pool_bytes_each,
                              size_t* state_bytes, size_t* workspace_bytes) {
  const rkv_status st = check_config(cfg);
  if (st != RKV_OK) return st;
  const Shape s = make_shape(cfg);
  if (kv_pool_bytes_each)
    *kv_pool_bytes_each = (size_t)s.S * s.L * s.Hkv * s.W * s.D * (s.bf16 ? 2 : 4);
  if (state_bytes) *state_bytes = align_up((size_t)s.S * sizeof(rkv::StreamState), 256);
  if (workspace_bytes) *workspace_bytes = make_layout(cfg).total;
  return RKV_OK;
}

rkv_status rkv_create(const rkv_config* cfg, const rkv_buffers* bufs, void* stream,
                      rkv_handle** out) {
  if (!out || !bufs) return RKV_ERR_INVALID_ARG;
  rkv_status st = check_config(cfg);
  if (st != RKV_OK) return st;
  // The tensor-core families take bf16 caches only.
  if ((cfg->attend_impl == RKV_ATTEND_MMA || cfg->attend_impl == RKV_ATTEND_TC) &&
      cfg->kv_dtype != RKV_BF16)
    return RKV_ERR_UNSUPPORTED;
  if (!bufs->k_pool || !bufs->v_pool || !bufs->state || !bufs->workspace)
    return RKV_ERR_INVALID_ARG;
  if (!aligned16(bufs->k_pool) || !aligned16(bufs->v_pool) || !aligned16(bufs->state) ||
      !aligned16(bufs->workspace))
    return RKV_ERR_INVALID_ARG;
  const WsLayout ws = make_layout(cfg);
  if (bufs->workspace_bytes < ws.total) return RKV_ERR_INVALID_ARG;

  rkv_handle* h = new (std::nothrow) rkv_handle();
  if (!h) return RKV_ERR_INVALID_ARG;
  h->cfg = *cfg;
  h->sh = make_shape(cfg);
  h->ws = ws;
  h->k_pool = bufs->k_pool;
  h->v_pool = bufs->v_pool;
  h->state = static_cast<rkv::StreamState*>(bufs->state);
  h->workspace = static_cast<uint8_t*>(bufs->workspace);
  h->scale = cfg->softmax_scale > 0.f ? cfg->softmax_scale : (float)(1.0 / std::sqrt((double)cfg->head_dim));
  h->last_launches = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    delete h;
    return RKV_ERR_CUDA;
  }
  if (!make_pool_map(&h->tmK, h->k_pool, h->sh) || !make_pool_map(&h->tmV, h->v_pool, h->sh)) {
    delete h;
    return RKV_ERR_CUDA;
  }
  h->has_map4 = h->sh.bf16 && make_pool_map4(&h->tmK4, h->k_pool, h->sh) &&
                make_pool_map4(&h->tmV4, h->v_pool, h->sh);
  if ((cfg->attend_impl == RKV_ATTEND_MMA || cfg->attend_impl == RKV_ATTEND_TC) && !h->has_map4) {
    delete h;
    return RKV_ERR_UNSUPPORTED;
  }
  h->host_table = make_table(h->sh, cfg->rope_theta);
  h->host_table_g = group_table(h->host_table, h->sh);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(h->state, 0, (size_t)h->sh.S * sizeof(rkv::StreamState), s);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(h->workspace + ws.append_tk_off, 0, ws.part_off - ws.append_tk_off, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(h->workspace + ws.table_off, h->host_table.data(),
                        h->host_table.size() * sizeof(float2), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(h->workspace + ws.table_g_off, h->host_table_g.data(),
                        h->host_table_g.size() * sizeof(float4), cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) {
    delete h;
    return RKV_ERR_CUDA;
  }
  *out = h;
  return RKV_OK;
}

rkv_status rkv_destroy(rkv_handle* h) {
  if (!h) return RKV_ERR_INVALID_ARG;
  delete h;
  return RKV_OK;
}

rkv_status rkv_append(rkv_handle* h, const void* k_new, const void* v_new, int32_t n_new,
                      int64_t* step_log, void* stream) {
  if (!h || !k_new || !v_new) return RKV_ERR_INVALID_ARG;
  if (n_new > h->sh.Wr) return RKV_ERR_CAPACITY;
  if (n_new < 1 || n_new > h->cfg.max_chunk) return RKV_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || (step_log && !aligned16(step_log)))
    return RKV_ERR_INVALID_ARG;
  rkv::AppendParams p;
  p.sh = h->sh;
  p.st = h->state;
  p.k_new = k_new;
  p.v_new = v_new;
  p.k_pool = h->k_pool;
  p.v_pool = h->v_pool;
  p.log = reinterpret_cast<long long*>(step_log);
  p.tickets = reinterpret_cast<int*>(h->workspace + h->ws.append_tk_off);
  p.table = reinterpret_cast<const float2*>(h->workspace + h->ws.table_off);
  p.c = n_new;
  p.div_hkv = rkv::FastDiv::make(static_cast<uint32_t>(h->sh.Hkv));
  p.div_c = rkv::FastDiv::make(static_cast<uint32_t>(n_new));
  h->last_launches = 1;
  return cuda_status(rkv::launch_append(p, static_cast<cudaStream_t>(stream)));
}

rkv_status rkv_attend(rkv_handle* h, const void* q, float* out, int32_t layer_begin,
                      int32_t n_layers, int32_t n_q, void* stream) {
  if (!h || !q || !out) return RKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out)) return RKV_ERR_INVALID_ARG;
  if (layer_begin < 0 || n_layers < 1 || layer_begin + n_layers > h->sh.L)
    return RKV_ERR_INVALID_ARG;
  if (n_q > h->sh.Wr) return RKV_ERR_CAPACITY;
  if (n_q < 1 || n_q > h->cfg.max_chunk) return RKV_ERR_INVALID_ARG;
  rkv::AttendParams p = {};
  p.sh = h->sh;
  p.st = h->state;
  p.q = q;
  p.out = out;
  p.k_pool = h->k_pool;   // read only through the tensor maps (and L2 prefetches)
  p.v_pool = h->v_pool;
  p.table = reinterpret_cast<const float2*>(h->workspace + h->ws.table_off);
  p.table_g = reinterpret_cast<const float4*>(h->workspace + h->ws.table_g_off);
  p.partials = reinterpret_cast<float*>(h->workspace + h->ws.part_off);
  p.unit_tickets = reinterpret_cast<int*>(h->workspace + h->ws.unit_tk_off);
  p.layer_begin = layer_begin;
  p.L_att = n_layers;
  p.c = n_q;
  p.R = n_q * h->sh.G;
  p.slot_floats = h->ws.slot_floats;
  p.scale_log2 = h->scale * 1.4426950408889634f;
  const int grid = rkv::attend_grid(h, n_layers);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const rkv_status st = rkv::launch_attend_any(h, p, grid, s);
  if (st == RKV_OK) h->last_launches = 1;
  return st;
}

rkv_status rkv_step_layers(rkv_handle* h, int32_t layer_begin, int32_t n_layers,
                           const void* k_new, const void* v_new, const void* q, float* out,
                           int64_t* step_log, int32_t last, void* stream) {
  if (!h || !k_new || !v_new || !q || !out) return RKV_ERR_INVALID_ARG;
  if (layer_begin < 0 || n_layers < 1 || layer_begin + n_layers > h->sh.L)
    return RKV_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(q) || !aligned16(out) ||
      (step_log && !aligned16(step_log)))
    return RKV_ERR_INVALID_ARG;
  if ((h->sh.stored_rotated && !h->sh.epoch) || !h->sh.bf16 || !h->has_map4 ||
      h->cfg.attend_impl == RKV_ATTEND_FMA || !rkv::attend_mma_supported(h->sh, 1))
    return RKV_ERR_UNSUPPORTED;
  rkv::AttendParams p = {};
  p.sh = h->sh;
  p.st = h->state;
  p.q = q;
  p.out = out;
  p.table = reinterpret_cast<const float2*>(h->workspace + h->ws.table_off);
  p.table_g = reinterpret_cast<const float4*>(h->workspace + h->ws.table_g_off);
  p.partials = reinterpret_cast<float*>(h->workspace + h->ws.part_off);
  p.unit_tickets = reinterpret_cast<int*>(h->workspace + h->ws.unit_tk_off);
  p.layer_begin = layer_begin;
  p.L_att = n_layers;
  p.c = 1;
  p.R = h->sh.G;
  p.slot_floats = h->ws.slot_floats;
  p.scale_log2 = h->scale * 1.4426950408889634f;
  p.fused = 1;
  p.k_new = k_new;
  p.v_new = v_new;
  p.k_pool = h->k_pool;
  p.v_pool = h->v_pool;
  p.log = last ? reinterpret_cast<long long*>(step_log) : nullptr;
  p.step_ticket = reinterpret_cast<int*>(h->workspace + h->ws.append_tk_off);
  p.publish = last ? 1 : 0;
  const int grid = rkv::attend_grid(h, n_layers);
  const cudaError_t e =
      rkv::launch_step_mma(p, h->tmK4, h->tmV4, grid, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return RKV_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return RKV_ERR_CUDA;
  h->last_launches = 1;
  return RKV_OK;
}

rkv_status rkv_step(rkv_handle* h, const void* k_new, const void* v_new, const void* q,
                    float* out, int64_t* step_log, void* stream) {
  if (!h) return RKV_ERR_INVALID_ARG;
  return rkv_step_layers(h, 0, h->sh.L, k_new, v_new, q, out, step_log, 1, stream);
}

rkv_status rkv_rebase(rkv_handle* h, void* stream) {
  if (!h) return RKV_ERR_INVALID_ARG;
  h->last_launches = 0;
  if (!h->sh.stored_rotated) return RKV_OK;  // re-basing is the origin update itself
  rkv::RerotParams p;
  p.sh = h->sh;
  p.st = h->state;
  p.k_pool = h->k_pool;
  p.tickets = reinterpret_cast<int*>(h->workspace + h->ws.rerot_tk_off);
  p.table = reinterpret_cast<const float2*>(h->workspace + h->ws.table_off);
  // One resident wave (3 CTAs of 256 threads per SM), split over the streams,
  // and no more CTAs than a stream's (key, eight-pair) items need.
  const long long items = (long long)h->sh.L * h->sh.Hkv * h->sh.W * (h->sh.D / 16);
  const long long need = (items + 255) / 256;
  const long long wave = std::max(1LL, (3LL * h->num_sms) / h->sh.S);
  const int bps = (int)std::max(1LL, std::min(need, wave));
  h->last_launches = 1;
  return cuda_status(rkv::launch_rerotate(p, bps, static_cast<cudaStream_t>(stream)));
}

rkv_status rkv_set_stream_state(rkv_handle* h, int32_t s, int64_t origin, int32_t fill,
                                void* stream) {
  if (!h || s < 0 || s >= h->sh.S || origin < 0 || fill < 0 || fill > h->sh.Wr)
    return RKV_ERR_INVALID_ARG;
  h->last_launches = 1;
  return cuda_status(
      rkv::launch_set_state(h->state, s, origin, fill, static_cast<int>(origin % h->sh.Wring),
                            static_cast<cudaStream_t>(stream)));
}

rkv_status rkv_get_stream_state(rkv_handle* h, int64_t* origins, int32_t* fills, int32_t* status,
                                void* stream) {
  if (!h) return RKV_ERR_INVALID_ARG;
  std::vector<rkv::StreamState> host(h->sh.S);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(host.data(), h->state, host.size() * sizeof(rkv::StreamState),
                                  cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return RKV_ERR_CUDA;
  for (int i = 0; i < h->sh.S; ++i) {
    if (origins) origins[i] = host[i].origin;
    if (fills) fills[i] = host[i].fill;
    if (status) status[i] = host[i].status;
  }
  return RKV_OK;
}

int32_t rkv_last_launch_count(const rkv_handle* h) { return h ? h->last_launches : 0; }

}  // extern "C"
