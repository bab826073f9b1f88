/*
 * rkv.h -- C ABI of the rolling KV cache with exact RoPE re-basing (B300, sm_103a).
 *
 * The operations follow "Audio8 ASR Infinite: What It Actually Takes to Listen
 * Forever" (its flowchart and the section "Inside the Rolling KV Cache and Exact
 * RoPE Re-Basing"): a fixed-capacity cache of key/value pairs per stream; when a
 * new pair does not fit, the oldest pair is evicted, the sliding origin moves
 * forward and every retained key and the query are placed at position
 * (p - origin), which preserves every query-key distance exactly.  The rotary
 * embedding uses theta = 1e6 ("Audio8-ASR-0.1B in audio.cpp", "Architecture")
 * and split-half pairing ("Audio8-ASR-Infinite-mlx", "Requires a patched
 * mlx-audio-swift"); the cache is stored in BF16
 * ("Reza2kn/Audio8-ASR-Infinite-Compressed", "Linux CPU").
 *
 * Conventions (all entry points):
 *  - Every buffer is caller-owned.  The library allocates no device memory;
 *    buffers must stay valid until rkv_destroy.  Device pointers must be
 *    16-byte aligned.
 *  - Work is enqueued on the caller's CUDA stream (passed as an opaque
 *    pointer, a cudaStream_t; NULL = legacy default stream).  Only
 *    rkv_get_stream_state waits for the device.
 *  - Argument errors are returned before anything is enqueued.  A failed
 *    launch returns RKV_ERR_CUDA.  Inconsistencies that only the device can
 *    see (a corrupt per-stream state, a query count larger than the window,
 *    a stored-rotated cache used without its re-base) set a sticky per-stream
 *    status word; kernels then skip that stream and rkv_get_stream_state
 *    reports it.
 *  - One handle is used from one CUDA stream at a time.  Calls on one handle
 *    that overlap on the GPU race.
 *
 * Notation: S streams, L layers, H_q query heads, H_kv KV heads (G = H_q/H_kv
 * query heads share one KV head: head h reads KV head floor(h/G)), D head_dim,
 * W capacity (slots per stream, layer and KV head), P pinned prefix slots
 * (rkv_config.n_pinned, usually 0) in front of a ring of W_ring = W - P slots,
 * W_r <= W_ring the retained window (pairs kept; W_r = W_ring unless
 * rkv_config.window says otherwise), c tokens per step.  Per stream the state
 * is (origin o, fill n <= W_r, npin pinned prefix pairs): retained absolute
 * positions are o .. o+n-1 and position p lives in slot P + (p mod W_ring);
 * prefix pair i lives in slot i.  Re-based positions: prefix pair i at i,
 * retained pair p at npin + (p - o) (npin = 0 without pinned slots).
 */
#ifndef RKV_H
#define RKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RKV_ABI_VERSION 2

typedef struct rkv_handle rkv_handle;  /* opaque, host memory owned by the library */

typedef enum {
  RKV_OK = 0,
  RKV_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or config field */
  RKV_ERR_UNSUPPORTED = 2,   /* valid but not built (e.g. head_dim 96)        */
  RKV_ERR_CAPACITY = 3,      /* more new tokens in one step than the capacity  */
  RKV_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed           */
  RKV_ERR_DEVICE_STATE = 5   /* a stream's device status word is set           */
} rkv_status;

typedef enum { RKV_BF16 = 0, RKV_F32 = 1 } rkv_dtype;

/* Key storage.  PRE_ROPE keeps keys unrotated and rotates them on the fly at
 * (p - origin) inside the attention kernels, so re-basing moves no data.
 * STORED_ROTATED keeps keys rotated at (p - origin) and re-rotates every
 * retained key by R(-e) after e evictions (rkv_rebase) -- the variant whose
 * repeated rounding "Audio8 ASR Infinite..." warns about in "Inside the
 * Rolling KV Cache and Exact RoPE Re-Basing" and "Failure Modes That Only
 * Appear on Day Three of a Session".  With rebase_epoch = E >= 2 the keys are
 * instead kept rotated at (p - o_ref), where o_ref = origin - lag trails the
 * origin by the evictions since the last re-rotation (lag < E + max_chunk);
 * the queries take the lag into their own rotation, and rkv_rebase turns all
 * retained keys by R(-lag) only once lag >= E: each key is rounded about
 * W / E + 1 times in its life instead of once per eviction, and the
 * re-rotation traffic drops by the factor E. */
typedef enum { RKV_PRE_ROPE = 0, RKV_STORED_ROTATED = 1 } rkv_layout;

/* Rotary pairing: split-half pairs element i with i + D/2 (rotate_half);
 * interleaved pairs 2i with 2i+1.  Pair i turns by angle r * theta^(-2i/D). */
typedef enum { RKV_ROPE_SPLIT_HALF = 0, RKV_ROPE_INTERLEAVED = 1 } rkv_rope_style;

/* Attention kernel family: AUTO picks the tensor-core kernels for bf16
 * caches -- single queries and chunks of fewer than 16 rows (c*G < 16) on
 * mma.sync, chunks of 16..128 rows on the fifth-generation tensor cores
 * (tcgen05, accumulators in tensor memory) -- and the CUDA-core kernel
 * otherwise; MMA keeps chunks on mma.sync (c*G <= 96); TC runs every chunk
 * with c*G <= 128 on tcgen05, single queries as AUTO. */
typedef enum {
  RKV_ATTEND_AUTO = 0, RKV_ATTEND_FMA = 1, RKV_ATTEND_MMA = 2, RKV_ATTEND_TC = 3
} rkv_attend_impl;

typedef struct {
  int32_t n_streams;     /* S, 1..1024                                    */
  int32_t n_layers;      /* L, >= 1; L * H_kv * W * D / 8 < 2^31          */
  int32_t n_q_heads;     /* H_q, multiple of n_kv_heads                   */
  int32_t n_kv_heads;    /* H_kv, >= 1                                    */
  int32_t head_dim;      /* D: 64 or 128                                  */
  int32_t capacity;      /* W: multiple of 32, 32..65536                  */
  int32_t max_chunk;     /* largest c passed to rkv_append / rkv_attend   */
  int32_t kv_dtype;      /* rkv_dtype of the K/V pools and new K/V rows    */
  int32_t q_dtype;       /* rkv_dtype of the queries                       */
  int32_t layout;        /* rkv_layout                                     */
  int32_t rope_style;    /* rkv_rope_style                                 */
  int32_t attend_impl;   /* rkv_attend_impl                                */
  double rope_theta;     /* > 1, e.g. 1e6                                  */
  float softmax_scale;   /* 0 => 1/sqrt(D)                                 */
  int32_t rebase_epoch;  /* STORED_ROTATED only: 0 re-rotates at every      */
                         /* eviction; E >= 2 re-rotates once every E        */
                         /* evictions (see rkv_rebase); E + max_chunk <= W_r+1 */
  int32_t window;        /* W_r, pairs retained per stream: 0 => W_ring,   */
                         /* else 1..W_ring.  A window that is not a multiple */
                         /* of 32 (the causal encoder's 750 frames,         */
                         /* "audio8-asr-infinite-p150", "At a glance") is   */
                         /* kept in a ring of W_ring >= W_r slots (768):    */
                         /* eviction follows W_r, slots follow W_ring;      */
                         /* max_chunk <= W_r                                */
  int32_t n_pinned;      /* P, pinned prefix slots: 0, or a multiple of 32  */
                         /* below W.  rkv_reset_stream then places its      */
                         /* prefix (<= P pairs) in slots 0.. that no append */
                         /* evicts; the window reads as "prefix, then the   */
                         /* retained pairs", numbered from 0 (a re-prefill: */
                         /* "audio8-asr-infinite-p150", "Limitations").    */
                         /* Not with rebase_epoch >= 2 (RKV_ERR_UNSUPPORTED) */
} rkv_config;

typedef struct {
  void* k_pool;           /* device, [S][L][H_kv][W][D] of kv_dtype           */
  void* v_pool;           /* device, same shape                               */
  void* state;            /* device, state_bytes (per-stream origin/fill/...) */
  void* workspace;        /* device, workspace_bytes (RoPE tables, partials)  */
  size_t workspace_bytes; /* size of workspace, >= rkv_required_bytes value   */
} rkv_buffers;

/* Sizes of the caller-owned buffers for cfg.  Host only; touches no GPU. */
rkv_status rkv_required_bytes(const rkv_config* cfg, size_t* kv_pool_bytes_each,
                              size_t* state_bytes, size_t* workspace_bytes);

/* Validates cfg and bufs, builds the handle and enqueues the initialisation
 * on `stream`: every stream's state becomes (origin 0, fill 0, status 0) and
 * the float32 sin/cos table (computed in float64 on the host) is uploaded into
 * the workspace.  Pool contents are not touched.  *out is set only on RKV_OK. */
rkv_status rkv_create(const rkv_config* cfg, const rkv_buffers* bufs, void* stream,
                      rkv_handle** out);

/* Appends n_new (1..max_chunk, <= W_r) pairs to every stream.
 * k_new, v_new: device, [L][S][n_new][H_kv][D] of kv_dtype.
 * Per stream (the flowchart of "Audio8 ASR Infinite...": "evict oldest pair",
 * "shift sliding origin forward"):
 *   e = max(0, n + n_new - W_r); o' = o + e; n' = n + n_new - e;
 *   new position o + n + j goes to slot (o + n + j) mod W in every layer and
 *   KV head.  STORED_ROTATED stores bf16/f32(R(p - o') k).
 * step_log: NULL or device int64 [S][4] receiving (o', n', e, first_slot).
 * One kernel launch.  In STORED_ROTATED, call rkv_rebase before the next
 * rkv_append or rkv_attend whenever this step evicted (the device flags a
 * missing re-base as RKV_ERR_DEVICE_STATE for that stream). */
rkv_status rkv_append(rkv_handle* h, const void* k_new, const void* v_new, int32_t n_new,
                      int64_t* step_log, void* stream);

/* Causal attention of the n_q newest tokens of every stream over its window,
 * for layers layer_begin .. layer_begin+n_layers-1.
 * q:   device, [n_layers][S][n_q][H_q][D] of q_dtype, before rotation.
 * out: device float32, same shape.
 * Query j sits at re-based position n' - n_q + j and sees keys r <= that
 * position; key r = p - o' is rotated to r (on the fly in PRE_ROPE).
 * out = sum_r softmax_r(<R(r_q) q, R(r) k_r> * scale) v_r, float32 math,
 * split across CTAs and merged by log-sum-exp.  An empty window gives 0.
 * n_q must not exceed the fill (device-checked). */
rkv_status rkv_attend(rkv_handle* h, const void* q, float* out, int32_t layer_begin,
                      int32_t n_layers, int32_t n_q, void* stream);

/* Re-base.  PRE_ROPE: nothing moves (the origin update of rkv_append is the
 * whole re-base) and nothing is launched.  STORED_ROTATED: one launch that
 * re-rotates every retained key older than the last append by R(-e), e = the
 * pairs that append evicted, in float32, rounded to nearest even.  With
 * rebase_epoch = E >= 2 the launch leaves a stream alone until its lag has
 * reached E and then turns all of its retained keys, the newest included, by
 * R(-lag) and sets the lag to 0; a stream with nothing due costs one state
 * read.  The launch is stream-ordered after the previous work on `stream`
 * (programmatic dependent launch lets it start its prologue early). */
rkv_status rkv_rebase(rkv_handle* h, void* stream);

/* One decode step in one kernel launch: rkv_append of one new pair per stream,
 * the (pre-RoPE, data-free) re-base and rkv_attend over every layer, fused.
 * k_new, v_new: device, [L][S][1][H_kv][D] of kv_dtype; q: device,
 * [L][S][1][H_q][D] of q_dtype; out: device float32, same shape as q;
 * step_log: NULL or device int64 [S][4] as for rkv_append.  Results, pool
 * contents and stream states equal those of rkv_append(k_new, v_new, 1),
 * rkv_rebase and rkv_attend(q, out, 0, L, 1) in sequence: the new pair is
 * written to its slot, and the attention takes it from k_new/v_new (its score
 * is <q, k_new>, the query and the key sharing a position) together with the
 * other retained pairs from the pools.  Served by the tensor-core kernel for
 * bf16 caches with PRE_ROPE keys, or STORED_ROTATED keys with a re-basing
 * epoch (rebase_epoch >= 2: the new key is stored rotated to its position
 * from o_ref and the lag grows by the evictions; call rkv_rebase after the
 * step as after rkv_append); anything else returns RKV_ERR_UNSUPPORTED before
 * touching the GPU (use the three calls instead).  The new states are
 * published by the last CTA of the launch to finish. */
rkv_status rkv_step(rkv_handle* h, const void* k_new, const void* v_new, const void* q,
                    float* out, int64_t* step_log, void* stream);

/* rkv_step for layers layer_begin .. layer_begin+n_layers-1 only, for a
 * decoder that runs its layers one after another (the new K/V and the query
 * of a layer exist only once the layer before it has run).  (The pages give
 * no interface; this is the per-layer form of the same step.)
 * k_new, v_new: [n_layers][S][1][H_kv][D]; q, out: [n_layers][S][1][H_q][D]
 * (the step's tensors from layer layer_begin on).  Every call derives the
 * step's geometry from the stream states as they were before the step, so the
 * calls of one step may come in any order and each layer range must be passed
 * exactly once; the call with last != 0 -- the step's final call, enqueued
 * after all the others -- publishes the new states and fills step_log (NULL
 * allowed).  Each call is one launch with no host synchronisation, so a
 * step's calls can be captured in a CUDA graph.  Same support as rkv_step;
 * a bad layer range returns RKV_ERR_INVALID_ARG. */
rkv_status rkv_step_layers(rkv_handle* h, int32_t layer_begin, int32_t n_layers,
                           const void* k_new, const void* v_new, const void* q, float* out,
                           int64_t* step_log, int32_t last, void* stream);

/* Size of the library-owned scratch array used by rkv_attend_static_scratch. */
#define RKV_STATIC_SCRATCH_BYTES (4u * 1024u * 1024u)

/* rkv_attend without caller-provided scratch.  (The pages have no counterpart:
 * this is a deployment convenience, not part of the method.)
 * Same arguments, layouts and result as rkv_attend, on the handle's pools,
 * state and RoPE table.  The scratch that rkv_attend keeps in the workspace --
 * split-softmax partials and merge tickets -- lives instead in one static
 * device array of RKV_STATIC_SCRATCH_BYTES that every GPU loading the library
 * holds until the process exits, so the call allocates nothing and writes
 * nothing to the workspace.  Meant for callers that cannot allocate device
 * memory where they attend (a host framework's fixed memory pool, a plugin
 * execute callback that forbids allocation, a real-time loop that must not
 * risk the device synchronisation of cudaMalloc).
 * Limits: S * L * H_kv <= 16384 and 2 * #SMs * max_chunk * G * (D + 2) * 4
 * bytes <= RKV_STATIC_SCRATCH_BYTES - 64 KiB; larger calls return
 * RKV_ERR_UNSUPPORTED before touching the GPU.
 * The first call on each device takes the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture.  Each call enqueues a clear of the tickets and one
 * kernel on `stream`.  All calls, from any handle, share the one array, which
 * keeps the last call's contents: calls that overlap on the GPU race. */
rkv_status rkv_attend_static_scratch(rkv_handle* h, const void* q, float* out,
                                     int32_t layer_begin, int32_t n_layers, int32_t n_q,
                                     void* stream);

/* Frees the handle (host memory only). */
rkv_status rkv_destroy(rkv_handle* h);

/* Utterance reset of stream s, with an optional prefix -- e.g. a constant
 * prompt prepared once: "Audio8 ASR Infinite..." resets the utterance state
 * when a turn completes, and "Reza2kn/Audio8-ASR-Infinite-Compressed" ("Linux
 * CPU") re-checks a prepared, audio-independent prefix on every silence
 * reset.  The stream's status is cleared; other streams are untouched.
 *  - Without pinned slots (n_pinned = 0): the stream restarts at `origin`
 *    holding the n_prefix pairs at positions origin .. origin + n_prefix - 1
 *    (re-based 0 .. n_prefix - 1) as the oldest pairs of its window; later
 *    appends evict them like any other pair.  0 <= n_prefix <= W_r.
 *  - With P = n_pinned > 0: the prefix goes into the pinned slots 0 ..
 *    n_prefix - 1 (re-based positions 0 .. n_prefix - 1), where no append
 *    evicts it; the rolling window restarts empty at `origin`, its pairs at
 *    re-based positions n_prefix + (p - o).  0 <= n_prefix <= P.
 * k, v: device, [L][n_prefix][H_kv][D] of kv_dtype, keys before rotation (the
 * call stores them rotated to 0 .. n_prefix - 1 for STORED_ROTATED), 16-byte
 * aligned; NULL allowed when n_prefix = 0 (an empty window, as
 * rkv_set_stream_state(s, origin, 0)).  0 <= s < S, origin >= 0, n_prefix in
 * range, else RKV_ERR_INVALID_ARG before touching the GPU.
 * One launch on `stream`, no host synchronisation. */
rkv_status rkv_reset_stream(rkv_handle* h, int32_t s, int64_t origin, const void* k,
                            const void* v, int32_t n_prefix, void* stream);

/* Sets stream s to (origin, fill) with no pinned prefix and clears its status,
 * enqueued on `stream`.  The caller must already hold that window's pairs in
 * slots P + ((origin+i) mod W_ring) (keys rotated to i for STORED_ROTATED).
 * Used to seed workloads and to jump the origin on an utterance reset.
 * origin >= 0, 0 <= fill <= W_r. */
rkv_status rkv_set_stream_state(rkv_handle* h, int32_t s, int64_t origin, int32_t fill,
                                void* stream);

/* Copies every stream's (origin, fill, status) to host arrays of length S
 * (any may be NULL) and waits for `stream`.  For tests and diagnostics. */
rkv_status rkv_get_stream_state(rkv_handle* h, int64_t* origins, int32_t* fills,
                                int32_t* status, void* stream);

/* Number of kernels the last enqueuing call on this handle launched: rkv_append,
 * rkv_attend, rkv_attend_static_scratch (its ticket clear is a memset, not a
 * kernel), rkv_rebase (0 for PRE_ROPE), rkv_step, rkv_step_layers,
 * rkv_reset_stream and rkv_set_stream_state. */
int32_t rkv_last_launch_count(const rkv_handle* h);

/* Static description of a status code. */
const char* rkv_status_string(rkv_status s);

/* RKV_ABI_VERSION of the loaded library. */
int32_t rkv_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* RKV_H */
