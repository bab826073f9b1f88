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
  CUtensorMap tmK, tmV;
  int num_sms;
  int last_launches;
  float scale;
  std::vector<float2> host_table;  // kept alive until destroy
};

namespace rkv {
// Largest persistent grid of the attention kernels.
constexpr int kMaxCtas = 1024;
}  // namespace rkv
