// Second half of a split-K contraction: the S FP32 partial sums of each
// output element (workspace [S, M, N], written by the GEMM with K cut into
// S ranges) are added in split order (one legal FP32 summation order; the
// contract leaves the order free: "Tensor Programs, Part 1", section "One
// Program and One Numerical Contract", rule 1), then the epilogue of the
// contraction is applied exactly as the GEMM's own epilogue would:
// RN_h of the sum, RN_h(t + b[n]), the steps; or the FP32 sum (+ b).
#pragma once

#include "epilogue.cuh"
#include "ptx.cuh"

namespace poot {

struct SplitReduceArgs {
  const float* ws;  // [S, M, N] partial sums
  int S;
  int M, N;
  ElemEpilogue e;   // the contraction's epilogue, y row pitch N
};

// VEC = 4: four consecutive elements of one row per thread (N % 4 == 0, the
// workspace 16-byte aligned, y 8-byte / y32 16-byte aligned): one 16-byte
// load per split and one 8- or 16-byte store.  VEC = 1: one element.
template <int VEC>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const SplitReduceArgs a) {
  grid_dep_wait();  // the partial sums come from the previous grid
  grid_dep_launch();
  const long long MN = (long long)a.M * a.N;
  const long long units = MN / VEC;
  const int dt = a.e.dtype;
  for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < units;
       u += (long long)gridDim.x * blockDim.x) {
    const long long i = u * VEC;
    float s[VEC];
    if constexpr (VEC == 4) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(a.ws + i));
      s[0] = v.x; s[1] = v.y; s[2] = v.z; s[3] = v.w;
      for (int k = 1; k < a.S; ++k) {
        const float4 p = __ldg(reinterpret_cast<const float4*>(a.ws + (long long)k * MN + i));
        s[0] = __fadd_rn(s[0], p.x);
        s[1] = __fadd_rn(s[1], p.y);
        s[2] = __fadd_rn(s[2], p.z);
        s[3] = __fadd_rn(s[3], p.w);
      }
    } else {
      s[0] = __ldg(a.ws + i);
      for (int k = 1; k < a.S; ++k) s[0] = __fadd_rn(s[0], __ldg(a.ws + (long long)k * MN + i));
    }
    const int m = (int)(i / a.N), n0 = (int)(i - (long long)m * a.N);
    const ElemEpilogue& e = a.e;
    if (e.out_f32) {
#pragma unroll
      for (int j = 0; j < VEC; ++j)
        if (e.has_bias) s[j] = __fadd_rn(s[j], ep_widen(__ldg(e.b + n0 + j), dt));
      if constexpr (VEC == 4) {
        *reinterpret_cast<float4*>(e.y32 + i) = make_float4(s[0], s[1], s[2], s[3]);
      } else {
        e.y32[i] = s[0];
      }
      continue;
    }
    float t[VEC];
#pragma unroll
    for (int j = 0; j < VEC; ++j) t[j] = elem_head(e, s[j], m, n0 + j, n0 + j);
    if constexpr (VEC == 4) {
      *reinterpret_cast<uint2*>(e.y + i) = make_uint2(ep_pack(t[0], t[1], dt), ep_pack(t[2], t[3], dt));
    } else {
      e.y[i] = dt == kEpiBf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(t[0]))
                              : __half_as_ushort(__float2half_rn(t[0]));
    }
  }
}

}  // namespace poot
