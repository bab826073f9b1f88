// rkv_rows.cuh -- f32 access to K/V rows and the rotation of their rotary
// pairs by (cos, sin) table entries, shared by the append kernel and the fused
// decode step.
#pragma once

#include "rkv_device.cuh"

namespace rkv {

// Four consecutive elements of a row, widened to f32.
__device__ __forceinline__ void load4(const void* base, size_t i, bool bf16, float (&x)[4]) {
  if (bf16) {
    uint2 w = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(base) + i);
    x[0] = bf_lo(w.x); x[1] = bf_hi(w.x); x[2] = bf_lo(w.y); x[3] = bf_hi(w.y);
  } else {
    float4 w = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + i);
    x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
  }
}
__device__ __forceinline__ void store4(void* base, size_t i, bool bf16, const float (&x)[4]) {
  if (bf16) {
    uint2 w = make_uint2(pack_bf2(x[0], x[1]), pack_bf2(x[2], x[3]));
    *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(base) + i) = w;
  } else {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + i) =
        make_float4(x[0], x[1], x[2], x[3]);
  }
}

// Rotates the 4 pairs held in (a, b) by the table entries cs[0..3]; `sgn` = +1
// rotates by +angle, -1 by -angle.  Pair (x, y) -> (x cos - y sin, y cos + x sin).
__device__ __forceinline__ void rotate4(float (&a)[4], float (&b)[4], const float2 (&cs)[4],
                                        float sgn) {
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    float c = cs[t].x, s = sgn * cs[t].y;
    float x = a[t], y = b[t];
    a[t] = x * c - y * s;
    b[t] = y * c + x * s;
  }
}

// Loads the two element groups of 4 pairs starting at pair i.  Split-half:
// a = dims i..i+3, b = dims i+D/2..i+D/2+3.  Interleaved: a = dims 2i,2i+2,..,
// b = dims 2i+1,2i+3,.. (8 consecutive elements).
__device__ __forceinline__ void load_pairs(const void* base, size_t row, int i, int D, int style,
                                           bool bf16, float (&a)[4], float (&b)[4]) {
  if (style == 0) {
    load4(base, row + i, bf16, a);
    load4(base, row + i + D / 2, bf16, b);
  } else {
    float x[4], y[4];
    load4(base, row + 2 * i, bf16, x);
    load4(base, row + 2 * i + 4, bf16, y);
    a[0] = x[0]; b[0] = x[1]; a[1] = x[2]; b[1] = x[3];
    a[2] = y[0]; b[2] = y[1]; a[3] = y[2]; b[3] = y[3];
  }
}
__device__ __forceinline__ void store_pairs(void* base, size_t row, int i, int D, int style,
                                            bool bf16, const float (&a)[4], const float (&b)[4]) {
  if (style == 0) {
    store4(base, row + i, bf16, a);
    store4(base, row + i + D / 2, bf16, b);
  } else {
    float x[4] = {a[0], b[0], a[1], b[1]};
    float y[4] = {a[2], b[2], a[3], b[3]};
    store4(base, row + 2 * i, bf16, x);
    store4(base, row + 2 * i + 4, bf16, y);
  }
}

__device__ __forceinline__ void load_cs4(const float2* table, size_t row_off, int i,
                                         float2 (&cs)[4]) {
  const float4* p = reinterpret_cast<const float4*>(table + row_off + i);
  float4 u = __ldg(p), v = __ldg(p + 1);
  cs[0] = make_float2(u.x, u.y); cs[1] = make_float2(u.z, u.w);
  cs[2] = make_float2(v.x, v.y); cs[3] = make_float2(v.z, v.w);
}


}  // namespace rkv
