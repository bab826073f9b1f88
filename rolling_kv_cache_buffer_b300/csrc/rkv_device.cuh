// rkv_device.cuh -- device helpers shared by the rolling-KV kernels (sm_103a).
//
// Per-stream state, inline-PTX wrappers (mbarrier, TMA, ldmatrix, mma), bf16
// packing, and the work partition of the attention kernels: every stream's
// window is cut into aligned blocks of TK slots, all blocks of all (stream,
// layer, KV head) units are laid end to end, and each persistent CTA takes one
// contiguous, equal share of that list.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rkv {

// One stream's device state (32 bytes).  origin = absolute position of the
// oldest retained pair, fill = retained pairs; retained positions are
// origin .. origin+fill-1 and position p sits in slot P + (p mod W_ring) (P
// pinned slots in front of a ring of W_ring = W - P slots; P = 0 unless the
// handle pins a prefix).  npin pinned prefix pairs sit in slots 0..npin-1.
struct StreamState {
  long long origin;
  int fill;
  int status;     // 0, or an rkv_status code (sticky until rkv_set_stream_state)
  int pending;    // stored-rotated: evictions not yet re-based (the lag, with an epoch)
  int last_new;   // pairs inserted by the last append
  int ring;       // origin mod W_ring (ring slot of the oldest pair), kept by every writer
  int npin;       // pinned prefix pairs (0 without pinned slots)
};
static_assert(sizeof(StreamState) == 32, "state layout");

constexpr int TK = 32;            // slots per block (one warp's unit of work)
constexpr int NWARP = 4;          // consumer warps per attention CTA
constexpr float NEG_BIG = -1e30f; // "minus infinity" that keeps exp2 finite
constexpr uint32_t WAIT_LIMIT = 1u << 22;  // bounded mbarrier waits
constexpr int STATUS_DEVICE_STATE = 5;     // RKV_ERR_DEVICE_STATE

// ----------------------------------------------------------------------------
// Inline PTX
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity; gives up after WAIT_LIMIT tries.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < WAIT_LIMIT; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// Plain arrival (count 1) on an mbarrier.
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// As mbar_wait, but also gives up as soon as *abort becomes nonzero.
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity,
                                                   const volatile int* abort) {
  for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
  }
  return false;
}
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the previous kernel of the stream runs; it
// must call pdl_wait() before touching anything that kernel writes.  The
// previous kernel calls pdl_trigger() once its dependents may be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Named barrier `id` over `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Arrival on named barrier `id` without waiting (its writes become visible to
// the threads that complete the barrier with named_bar_sync).
__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Thread-block clusters: rank of this CTA, the shared::cluster address of a
// shared-memory word in CTA `rank`, asynchronous stores into a partner CTA's
// shared memory, a local wait that acquires at cluster scope, and the
// cluster-wide barrier.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
// Asynchronous 4-byte store into another CTA's shared memory that counts its
// bytes on that CTA's mbarrier (complete_tx).
__device__ __forceinline__ void st_async_f32(uint32_t cluster_addr, float v, uint32_t cluster_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
               ::"r"(cluster_addr), "r"(__float_as_uint(v)), "r"(cluster_bar)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Arrival on an mbarrier of another CTA of the cluster (a shared::cluster
// address from map_to_rank) that releases this thread's earlier writes at
// cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}
// Loads from another CTA's shared memory (shared::cluster addresses).
__device__ __forceinline__ float ld_cluster_f32(uint32_t cluster_addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t cluster_addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(cluster_addr)
               : "memory");
  return v;
}
// Split cluster barrier: arrive without ordering (after the barrier inits,
// whose fence already releases them to the cluster), wait later.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// 16-byte asynchronous global -> shared copy (both addresses 16-byte aligned),
// its group commit, and the wait for all of this thread's groups.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
// Hint: bring the 128-byte line holding p into L2.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 3-D tiled TMA load (global -> shared), completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
// Bring a tensor map (a kernel parameter) into the TMA unit's descriptor cache.
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}
// L2 policy for data read once: its lines are the first to go, so a stream of
// them does not push out what the kernel reads again (states, code, partials).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// 4-D tiled TMA load (global -> shared) under L2 cache policy `pol`,
// completion counted on `bar`.
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap* tm, int c0,
                                                 int c1, int c2, int c3, uint32_t bar,
                                                 uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar), "l"(pol)
      : "memory");
}
// 1-D bulk copy (global -> shared); both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D += A * B, m16n8k16, bf16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bf16 <-> f32.  A bf16 value is the upper 16 bits of the f32 with the same
// value, so widening is a shift; narrowing rounds to nearest even.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint16_t to_bf(float x) {
  return static_cast<uint16_t>(pack_bf2(x, 0.f) & 0xffffu);
}

// ----------------------------------------------------------------------------
// Element access for the two storage types
// ----------------------------------------------------------------------------
__device__ __forceinline__ float load_elem(const void* base, size_t i, bool bf16) {
  if (bf16) {
    uint16_t b = reinterpret_cast<const uint16_t*>(base)[i];
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  return reinterpret_cast<const float*>(base)[i];
}
__device__ __forceinline__ void store_elem(void* base, size_t i, float x, bool bf16) {
  if (bf16)
    reinterpret_cast<uint16_t*>(base)[i] = to_bf(x);
  else
    reinterpret_cast<float*>(base)[i] = x;
}

// Pair i of a head vector: split-half pairs (i, i + D/2), interleaved (2i, 2i+1).
__device__ __forceinline__ int pair_d1(int i, int D, int style) { return style ? 2 * i : i; }
__device__ __forceinline__ int pair_d2(int i, int D, int style) {
  return style ? 2 * i + 1 : i + D / 2;
}

// A usable stream state: no status set, 0 <= fill <= Wr (the retained window),
// 0 <= ring < Wring (the ring's slots) and 0 <= npin <= P (the pinned slots).
__device__ __forceinline__ int state_ok(const StreamState& s, int Wring, int Wr, int P) {
  return s.status == 0 && s.origin >= 0 && s.fill >= 0 && s.fill <= Wr && s.ring >= 0 &&
         s.ring < Wring && s.npin >= 0 && s.npin <= P;
}

// ----------------------------------------------------------------------------
// Work partition
// ----------------------------------------------------------------------------
// Blocks of TK slots touched by a window that starts at slot a (= origin mod W)
// and holds n pairs.  Blocks are aligned in slot space, so a block never
// crosses the end of the ring; a window that wraps touches blocks at the end
// and at the start.  W is a multiple of TK.
__host__ __device__ __forceinline__ int touched_blocks(int a, int n, int NB) {
  if (n <= 0) return 0;
  int first = a / TK;
  int last = (a + n - 1) / TK;  // may be >= NB when the window wraps
  int cnt = last - first + 1;
  return cnt > NB ? NB : cnt;
}
// Slot-block index of the j-th touched block.
__host__ __device__ __forceinline__ int touched_block(int a, int j, int NB) {
  return (a / TK + j) % NB;
}
// Blocks of one (stream, layer, KV head) unit: the ceil(npin / TK) blocks of
// the pinned prefix (slots 0..), then the ring blocks the window of n pairs
// starting at ring slot a touches.
__host__ __device__ __forceinline__ int unit_blocks(int a, int n, int npin, int NBr) {
  return (npin + TK - 1) / TK + touched_blocks(a, n, NBr);
}
// The cached per-stream word of the attention kernels: ring start a and pinned
// prefix pairs npin (both < 2^16), or -1 for a stream whose state is not usable.
__host__ __device__ __forceinline__ int pack_an(int a, int npin) { return a | (npin << 16); }
// First block index of CTA b when T blocks are shared by P CTAs.
__host__ __device__ __forceinline__ int range_start(int b, int T, int P) {
  return static_cast<int>((static_cast<long long>(b) * T) / P);
}
// The CTA whose range holds block x.
__host__ __device__ __forceinline__ int cta_of(int x, int T, int P) {
  return static_cast<int>(((static_cast<long long>(x) + 1) * P - 1) / T);
}

}  // namespace rkv
