// rkv_attend_static.cu -- rkv_attend_static_scratch: the attention call with its
// scratch in a library-owned device array, for callers that cannot allocate.
//
// rkv_attend keeps its scratch (the split-softmax partials of units shared by
// several CTAs and the per-unit merge tickets) in the caller's workspace.  Some
// callers cannot provide or grow device memory at the point where they attend:
// code running under a memory pool owned by a host framework or plugin API that
// forbids allocation inside its execute callback, and real-time loops where a
// cudaMalloc (which may synchronise the device) would stall the stream.  This
// entry point runs the same attention kernels with that scratch in a file-scope
// static __device__ array of RKV_STATIC_SCRATCH_BYTES instead.  It allocates
// nothing: no cudaMalloc, no cudaFree, no allocating library routine.
#include <mutex>

#include "rkv_handle.h"

namespace {

// Layout of the static scratch: merge tickets first, split partials after.
constexpr size_t kTicketBytes = 64 * 1024;                  // 16384 units
constexpr size_t kPartialBytes = RKV_STATIC_SCRATCH_BYTES - kTicketBytes;
static_assert(RKV_STATIC_SCRATCH_BYTES > kTicketBytes, "scratch layout");

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_rkv_scratch[RKV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_dev_ptr[kMaxDevices];   // device address of g_rkv_scratch, per device

// Device address of the scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, taken once per device with that device current.
rkv_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RKV_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_dev_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_rkv_scratch) != cudaSuccess || !p) return RKV_ERR_CUDA;
    g_dev_ptr[dev] = p;
  }
  *out = g_dev_ptr[dev];
  return RKV_OK;
}

}  // namespace

extern "C" rkv_status rkv_attend_static_scratch(rkv_handle* h, const void* q, float* out,
                                                int32_t layer_begin, int32_t n_layers,
                                                int32_t n_q, void* stream) {
  if (!h || !q || !out) return RKV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) & 15u) || (reinterpret_cast<uintptr_t>(out) & 15u))
    return RKV_ERR_INVALID_ARG;
  if (layer_begin < 0 || n_layers < 1 || layer_begin + n_layers > h->sh.L)
    return RKV_ERR_INVALID_ARG;
  if (n_q > h->sh.Wr) return RKV_ERR_CAPACITY;
  if (n_q < 1 || n_q > h->cfg.max_chunk) return RKV_ERR_INVALID_ARG;

  // Sizes first: a call that needs more scratch than the array holds is
  // rejected before anything touches the GPU.
  const int grid = rkv::attend_grid(h, n_layers);
  const size_t tickets = (size_t)h->sh.S * h->sh.L * h->sh.Hkv * sizeof(int);
  const size_t partials = (size_t)2 * grid * h->ws.slot_floats * sizeof(float);
  if (tickets > kTicketBytes || partials > kPartialBytes) return RKV_ERR_UNSUPPORTED;

  void* base = nullptr;
  rkv_status st = scratch_address(&base);
  if (st != RKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Every merge returns its unit's ticket to 0, so after a completed call the
  // tickets are already 0.  The clear guards against tickets left behind by a
  // call that aborted (a device-detected error stops a CTA before its merge)
  // or that used the array for another handle's shape.
  if (cudaMemsetAsync(base, 0, tickets, s) != cudaSuccess) return RKV_ERR_CUDA;

  rkv::AttendParams p = {};
  p.sh = h->sh;
  p.st = h->state;
  p.q = q;
  p.out = out;
  p.k_pool = h->k_pool;   // read only through the tensor maps (and L2 prefetches)
  p.v_pool = h->v_pool;
  p.table = reinterpret_cast<const float2*>(h->workspace + h->ws.table_off);
  p.table_g = reinterpret_cast<const float4*>(h->workspace + h->ws.table_g_off);
  p.partials = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kTicketBytes);
  p.unit_tickets = static_cast<int*>(base);
  p.layer_begin = layer_begin;
  p.L_att = n_layers;
  p.c = n_q;
  p.R = n_q * h->sh.G;
  p.slot_floats = h->ws.slot_floats;
  p.scale_log2 = h->scale * 1.4426950408889634f;
  const rkv_status ls = rkv::launch_attend_any(h, p, grid, s);
  if (ls == RKV_OK) h->last_launches = 1;   // the attention kernel (the clear is a memset)
  return ls;
}
