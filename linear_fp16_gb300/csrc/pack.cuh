// Row repacking for operands TMA cannot read in place: x [R0, K] and W
// [R1, K] (2-byte aligned, any K) are copied into [R, Kp] buffers with
// Kp = K rounded up to 8 elements, so every row starts on a 16-byte
// boundary and the tcgen05 GEMM can load them with TMA.  The elements keep
// their bits (a pure copy: the contraction's arithmetic is untouched); the
// pad columns K .. Kp-1 are written as zeros (the tensor maps bound the
// inner dimension at K, so they are never read as operands anyway).
//
// Each thread moves one 16-byte chunk of a destination row (8 elements).
// The source chunk starts at row * K + 8c elements, so its alignment is the
// row start's: 16-, 8-, 4- or 2-byte loads as that alignment allows, all
// inside the row's own K elements; the row's last, partial chunk is read
// element by element.  Consecutive threads take consecutive chunks, so a
// warp reads and writes contiguous spans.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace poot {

struct PackArgs {
  const uint16_t* src[2];  // x, W (row pitch K elements)
  uint16_t* dst[2];        // packed copies (row pitch Kp elements, 16-byte aligned)
  long long rows[2];
  int K, Kp;
};

__device__ __forceinline__ uint4 pack_load8(const uint16_t* __restrict__ s) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(s);
  if ((a & 15u) == 0) return __ldg(reinterpret_cast<const uint4*>(s));
  if ((a & 7u) == 0) {
    const uint2 lo = __ldg(reinterpret_cast<const uint2*>(s));
    const uint2 hi = __ldg(reinterpret_cast<const uint2*>(s + 4));
    return make_uint4(lo.x, lo.y, hi.x, hi.y);
  }
  if ((a & 3u) == 0) {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(s);
    return make_uint4(__ldg(p), __ldg(p + 1), __ldg(p + 2), __ldg(p + 3));
  }
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) w[j] = (uint32_t)__ldg(s + 2 * j) | ((uint32_t)__ldg(s + 2 * j + 1) << 16);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void __launch_bounds__(256) pack_rows_kernel(const PackArgs a) {
  grid_dep_wait();  // x and W may come from the previous grid
  grid_dep_launch();
  const long long cpr = a.Kp / 8;  // 16-byte chunks per packed row
  const long long n0 = a.rows[0] * cpr;
  const long long total = n0 + a.rows[1] * cpr;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int t = i < n0 ? 0 : 1;
    const long long j = t ? i - n0 : i;
    const long long r = j / cpr;
    const int k0 = (int)(j - r * cpr) * 8;
    // (selects, not a.src[t]: a dynamic index would copy the arrays to local memory)
    const uint16_t* __restrict__ s = (t ? a.src[1] : a.src[0]) + r * a.K + k0;
    uint4 v;
    if (k0 + 8 <= a.K) {
      v = pack_load8(s);
    } else {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (k0 + e < a.K) w[e >> 1] |= (uint32_t)__ldg(s + e) << ((e & 1) * 16);
      v = make_uint4(w[0], w[1], w[2], w[3]);
    }
    *reinterpret_cast<uint4*>((t ? a.dst[1] : a.dst[0]) + r * a.Kp + k0) = v;
  }
}

}  // namespace poot
