// Device helpers of the widened contraction's epilogue ("ML compiler
// internals", section "The OpKind vocabulary": the ContractionEpilogue row —
// the head's result keeps its dtype and every step of the pointwise chain
// rounds through it — and section "SwiGLU and GeLU FFN": SiLU and GELU are
// compositions of the Neg, Exp, Add, Div, Mul and Erf primitives).
//
// Every primitive below is evaluated in FP32 and rounded to the head dtype
// (binary16 or bfloat16).  For +, *, / of two head-dtype values FP32 has at
// least 2p + 2 significand bits (p = 11 or 8), so FP32-then-round equals
// the correctly rounded head result (the double rounding is innocuous);
// the IEEE-rounded intrinsics (__fadd_rn, __fmul_rn, __fdiv_rn) keep the
// compiler from fusing two primitives into one rounding.  Exp and Erf use
// expf / erff and then round.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace poot {

enum EpiDtype : int { kEpiF16 = 0, kEpiBf16 = 1 };
enum EpiOp : int { kEpAdd = 1, kEpMul = 2, kEpSilu = 3, kEpGeluTanh = 4, kEpGeluErf = 5 };
constexpr int kEpiMaxSteps = 4;

// round one FP32 value to the head dtype and back (exact widening)
template <int DT>
__device__ __forceinline__ float ep_rh_t(float v) {
  if constexpr (DT == kEpiBf16) return __bfloat162float(__float2bfloat16_rn(v));
  else return __half2float(__float2half_rn(v));
}
__device__ __forceinline__ float ep_rh(float v, int dt) {
  return dt == kEpiBf16 ? __bfloat162float(__float2bfloat16_rn(v)) : __half2float(__float2half_rn(v));
}

// two FP32 values rounded to the head dtype, packed low = first
template <int DT>
__device__ __forceinline__ uint32_t ep_pack_t(float a, float b) {
  if constexpr (DT == kEpiBf16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
  } else {
    const __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
}
__device__ __forceinline__ uint32_t ep_pack(float a, float b, int dt) {
  if (dt == kEpiBf16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
  const __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// a packed pair of head-dtype values, widened exactly to FP32
template <int DT>
__device__ __forceinline__ float2 ep_unpack_t(uint32_t u) {
  if constexpr (DT == kEpiBf16) return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
  else return __half22float2(*reinterpret_cast<const __half2*>(&u));
}
__device__ __forceinline__ float2 ep_unpack(uint32_t u, int dt) {
  if (dt == kEpiBf16) return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
  return __half22float2(*reinterpret_cast<const __half2*>(&u));
}

__device__ __forceinline__ float ep_widen(uint16_t bits, int dt) {
  if (dt == kEpiBf16) return __uint_as_float((uint32_t)bits << 16);
  return __half2float(__ushort_as_half(bits));
}

// x / (1 + exp(-x)) over Neg, Exp, Add, Div
template <int DT>
__device__ __forceinline__ float ep_silu_t(float t) {
  const float e = ep_rh_t<DT>(expf(-t));  // -t is exact
  const float d = ep_rh_t<DT>(__fadd_rn(1.0f, e));
  return ep_rh_t<DT>(__fdiv_rn(t, d));
}

// the tanh approximation in its sigmoid form: x / (1 + exp(-c2 (x + c1 x^3)))
// c1 = RN(0.044715), c2 = RN(2 sqrt(2/pi)); the FP32 literals are within
// 2^-24 relative of the exact constants, far from a rounding boundary of
// either head dtype, so rounding them gives the same head values
template <int DT>
__device__ __forceinline__ float ep_gelu_tanh_t(float t) {
  const float c1 = ep_rh_t<DT>(0.044715f);
  const float c2 = ep_rh_t<DT>(1.5957691216057308f);
  const float s = ep_rh_t<DT>(__fmul_rn(t, t));
  const float c = ep_rh_t<DT>(__fmul_rn(s, t));
  const float u = ep_rh_t<DT>(__fmul_rn(c1, c));
  const float v = ep_rh_t<DT>(__fadd_rn(t, u));
  const float z = ep_rh_t<DT>(__fmul_rn(c2, v));
  const float e = ep_rh_t<DT>(expf(-z));
  const float d = ep_rh_t<DT>(__fadd_rn(1.0f, e));
  return ep_rh_t<DT>(__fdiv_rn(t, d));
}

// 0.5 x (1 + erf(x / sqrt 2)) over Mul, Erf, Add; c3 = RN(1/sqrt 2)
template <int DT>
__device__ __forceinline__ float ep_gelu_erf_t(float t) {
  const float c3 = ep_rh_t<DT>(0.70710678118654752f);
  const float s = ep_rh_t<DT>(__fmul_rn(c3, t));
  const float e = ep_rh_t<DT>(erff(s));
  const float d = ep_rh_t<DT>(__fadd_rn(1.0f, e));
  const float p = ep_rh_t<DT>(__fmul_rn(t, d));
  return ep_rh_t<DT>(__fmul_rn(0.5f, p));
}

template <int OP, int DT>
__device__ __forceinline__ float ep_activation_t(float t) {
  if constexpr (OP == kEpSilu) return ep_silu_t<DT>(t);
  else if constexpr (OP == kEpGeluTanh) return ep_gelu_tanh_t<DT>(t);
  else return ep_gelu_erf_t<DT>(t);
}

__device__ __forceinline__ float ep_activation(int op, float t, int dt) {
  const bool bf = dt == kEpiBf16;
  switch (op) {
    case kEpSilu: return bf ? ep_silu_t<kEpiBf16>(t) : ep_silu_t<kEpiF16>(t);
    case kEpGeluTanh: return bf ? ep_gelu_tanh_t<kEpiBf16>(t) : ep_gelu_tanh_t<kEpiF16>(t);
    case kEpGeluErf: return bf ? ep_gelu_erf_t<kEpiBf16>(t) : ep_gelu_erf_t<kEpiF16>(t);
    default: return t;
  }
}

// ---- packed pairs ------------------------------------------------------------
// Two head-dtype values in one 32-bit word (low = first).  Add and multiply
// of such pairs are the IEEE operations of the head dtype, rounded to
// nearest even (the correctly rounded result, the same value as the FP32
// operation followed by one rounding), two lanes of work per instruction;
// the _rn forms keep the compiler from contracting a multiply and an add
// into one fused (singly rounded) operation.  Division goes through the
// IEEE FP32 division and one rounding.
template <int DT>
__device__ __forceinline__ uint32_t ep_h2_add(uint32_t a, uint32_t b) {
  if constexpr (DT == kEpiBf16) {
    const __nv_bfloat162 r = __hadd2_rn(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                        *reinterpret_cast<const __nv_bfloat162*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
  } else {
    const __half2 r = __hadd2_rn(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
  }
}
template <int DT>
__device__ __forceinline__ uint32_t ep_h2_mul(uint32_t a, uint32_t b) {
  if constexpr (DT == kEpiBf16) {
    const __nv_bfloat162 r = __hmul2_rn(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                        *reinterpret_cast<const __nv_bfloat162*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
  } else {
    const __half2 r = __hmul2_rn(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
  }
}
template <int DT>
__device__ __forceinline__ uint32_t ep_h2_div(uint32_t a, uint32_t b) {
  const float2 fa = ep_unpack_t<DT>(a), fb = ep_unpack_t<DT>(b);
  return ep_pack_t<DT>(__fdiv_rn(fa.x, fb.x), __fdiv_rn(fa.y, fb.y));
}
// a constant in both halves, rounded to the head dtype
template <int DT>
__device__ __forceinline__ uint32_t ep_h2_const(float c) {
  return ep_pack_t<DT>(c, c);
}
// ADD / MUL step on a pair of head values and a pair of operand values
template <int DT>
__device__ __forceinline__ uint32_t ep_h2_binop(int op, uint32_t t, uint32_t r) {
  return op == kEpAdd ? ep_h2_add<DT>(t, r) : ep_h2_mul<DT>(t, r);
}
// exp of the negated pair: both evaluated in FP32 (expf), rounded
template <int DT>
__device__ __forceinline__ uint32_t ep_h2_exp_neg(uint32_t z) {
  const float2 f = ep_unpack_t<DT>(z);
  return ep_pack_t<DT>(expf(-f.x), expf(-f.y));  // -z is exact
}

// The activation OP over n packed pairs of head-dtype values, in place, with
// the same primitives and roundings as ep_activation_t, two lanes at a time;
// four pairs' chains in flight (inlined into the GEMM's rotated box loop,
// with 224 registers: GELU tanh 726 -> 704 us on 8192 x 14336 x 4096, the
// other forms within 2%, against two)
template <int OP, int DT, int N>
__device__ __forceinline__ void ep_activation_pairs(uint32_t* v) {
  const uint32_t one = ep_h2_const<DT>(1.0f);
#pragma unroll 4
  for (int i = 0; i < N; ++i) {
    const uint32_t t = v[i];
    if constexpr (OP == kEpSilu) {
      const uint32_t d = ep_h2_add<DT>(one, ep_h2_exp_neg<DT>(t));
      v[i] = ep_h2_div<DT>(t, d);
    } else if constexpr (OP == kEpGeluTanh) {
      // constants as in ep_gelu_tanh_t
      const uint32_t c1 = ep_h2_const<DT>(0.044715f), c2 = ep_h2_const<DT>(1.5957691216057308f);
      const uint32_t sq = ep_h2_mul<DT>(t, t);
      const uint32_t cu = ep_h2_mul<DT>(sq, t);
      const uint32_t u = ep_h2_mul<DT>(c1, cu);
      const uint32_t w = ep_h2_add<DT>(t, u);
      const uint32_t z = ep_h2_mul<DT>(c2, w);
      const uint32_t d = ep_h2_add<DT>(one, ep_h2_exp_neg<DT>(z));
      v[i] = ep_h2_div<DT>(t, d);
    } else {
      const uint32_t c3 = ep_h2_const<DT>(0.70710678118654752f), half = ep_h2_const<DT>(0.5f);
      const uint32_t sc = ep_h2_mul<DT>(c3, t);
      const float2 sf = ep_unpack_t<DT>(sc);
      const uint32_t e = ep_pack_t<DT>(erff(sf.x), erff(sf.y));
      const uint32_t d = ep_h2_add<DT>(one, e);
      v[i] = ep_h2_mul<DT>(half, ep_h2_mul<DT>(t, d));
    }
  }
}

// The widened contraction's epilogue for one output held as an FP32 sum by
// one lane (the GEMVs, the split-K reduce): y[m, n] (row pitch ldy) gets
// RN_h(s), then RN_h(t + b[n]), then the steps, every primitive rounded to
// the head dtype; or, with out_f32, the FP32 sum (+ b[n] in FP32).
struct ElemEpilogue {
  int dtype, out_f32, has_bias, num_steps;
  int op[kEpiMaxSteps];
  const uint16_t* ptr[kEpiMaxSteps];  // ADD / MUL operands [.., ld]
  long long ld[kEpiMaxSteps];
  const uint16_t* b;  // [N] head-dtype bits, or nullptr
  uint16_t* y;        // head-dtype bits (out_f32 == 0)
  float* y32;         // out_f32 == 1
  long long ldy;
};

// the head value after bias and steps (not yet stored); output row m and
// column n, bias element nb (n, or group * N + n for a grouped contraction)
__device__ __forceinline__ float elem_head(const ElemEpilogue& e, float s, int m, int n, int nb) {
  const int dt = e.dtype;
  float t = ep_rh(s, dt);
  if (e.has_bias) t = ep_rh(__fadd_rn(t, ep_widen(__ldg(e.b + nb), dt)), dt);
  for (int st = 0; st < e.num_steps; ++st) {
    const int op = e.op[st];
    if (op == kEpAdd || op == kEpMul) {
      const float r = ep_widen(__ldg(e.ptr[st] + (size_t)m * (size_t)e.ld[st] + n), dt);
      t = ep_rh(op == kEpAdd ? __fadd_rn(t, r) : __fmul_rn(t, r), dt);
    } else {
      t = ep_activation(op, t, dt);
    }
  }
  return t;
}

__device__ __forceinline__ void elem_store(const ElemEpilogue& e, float s, int m, int n, int nb) {
  const size_t i = (size_t)m * (size_t)e.ldy + n;
  if (e.out_f32) {
    e.y32[i] = e.has_bias ? __fadd_rn(s, ep_widen(__ldg(e.b + nb), e.dtype)) : s;
    return;
  }
  const float t = elem_head(e, s, m, n, nb);
  e.y[i] = e.dtype == kEpiBf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(t)) : __half_as_ushort(__float2half_rn(t));
}

// Eight consecutive elements (bits) of row `row`, columns c .. c+7, of an
// [M, ld] operand; zero outside [M) x [N).  `vec`: base 16-byte aligned and
// ld % 8 == 0 (c is a multiple of 8), so a full chunk is one 16-byte load.
__device__ __forceinline__ uint4 ep_load8(const uint16_t* __restrict__ base, long long ld, int row, int M, int c,
                                          int N, bool vec) {
  uint4 r = make_uint4(0u, 0u, 0u, 0u);
  if (row >= M) return r;
  const uint16_t* p = base + (size_t)row * (size_t)ld + c;
  if (vec && c + 8 <= N) return __ldg(reinterpret_cast<const uint4*>(p));
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t e = (c + j < N) ? (uint32_t)__ldg(p + j) : 0u;
    w[j >> 1] |= e << ((j & 1) * 16);
  }
  r.x = w[0]; r.y = w[1]; r.z = w[2]; r.w = w[3];
  return r;
}

// Row `lane` of a 32 x 32 box of an [M, ld] operand (columns c0 .. c0+31),
// copied by cp.async into a 32 x 64-byte shared-memory box with the 64-byte
// swizzle of the output staging boxes (16-byte chunk j of a row at position
// j ^ ((row >> 1) & 3), so that a warp's 16-byte accesses are free of bank
// conflicts); zero outside [M) x [N).  The operand must be 16-byte aligned
// with ld % 8 == 0 (c0 a multiple of 8).
__device__ __forceinline__ void ep_operand_box_async(uint32_t box, const uint16_t* __restrict__ base, long long ld,
                                                     int row, int M, int c0, int N, int lane) {
  const bool rok = row < M;
  const uint16_t* p = base + (size_t)(rok ? row : 0) * (size_t)ld + c0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = c0 + 8 * j;
    const int n = rok ? max(0, min(8, N - c)) : 0;  // elements of this chunk inside the operand
    cp_async_16(box + (uint32_t)(lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)), n > 0 ? (const void*)(p + 8 * j)
                                                                                       : (const void*)base,
                (uint32_t)(2 * n));
  }
}

}  // namespace poot
