// y = FP16(x . W^T) + b for M <= 16 rows: an HBM-bound stream of W.
//
// Each output feature n is one row of W ([N, K], read in place).  A block of
// eight warps stages x (all M rows, a chunk of K at a time) in shared memory
// and gives each W row to `wpr` warps (1, 2, 4 or 8; more warps per row when
// N is too small to fill the GPU).  Lanes stream W with 16-byte
// non-allocating loads, kGemvUnroll vectors in flight per lane, multiply by
// x in FP32 (each product of two binary16 numbers is exact) and accumulate
// in FP32.  Lane sums meet in a shuffle tree, the warps of one row in
// shared memory, in a fixed order.  Then proj = RN16(sum) and
// y = RN16(proj + b[n]) ("Tensor Programs, Part 1", section "One Program and
// One Numerical Contract", rules 1 and 2).
//
// The plan-time GEMV/GEMM split follows the MatMul entry of the poot "The
// Graph IR" page (one op; GEMV and GEMM specialised from static shapes).
#pragma once

#include "ptx.cuh"

namespace poot {

constexpr int kGemvWarps = 8;
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kGemvUnroll = 8;

struct GemvArgs {
  const __half* x;
  const __half* w;
  const __half* b;
  __half* y;
  int M, N, K;
  int wpr;  // warps per W row: 1, 2, 4 or 8
  int kc;   // K chunk staged in shared memory (multiple of 256)
};

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// MT: M rounded up to 1, 2, 4, 8 or 16.  VEC: 16-byte loads of x and W
// (K % 8 == 0 and both 16-byte aligned); otherwise 2-byte loads.
template <int MT, bool VEC>
__global__ void __launch_bounds__(kGemvThreads) gemv_f16_kernel(const GemvArgs a) {
  extern __shared__ uint4 gemv_smem[];
  __half* xs = reinterpret_cast<__half*>(gemv_smem);  // [MT][kc]
  __shared__ float red[kGemvWarps][MT];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wpr = a.wpr;
  const int row = blockIdx.x * (kGemvWarps / wpr) + warp / wpr;
  const int part = warp % wpr;
  const bool active = row < a.N;
  const int K = a.K, kc = a.kc;
  const __half* __restrict__ wrow = a.w + (size_t)(active ? row : 0) * K;

  float acc[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) acc[m] = 0.0f;

  for (int kc0 = 0; kc0 < K; kc0 += kc) {
    const int len = min(kc, K - kc0);
    __syncthreads();  // the previous chunk has been consumed
    if constexpr (VEC) {
      const int vpr = kc / 8;  // 16-byte vectors per staged row
      for (int i = threadIdx.x; i < MT * vpr; i += kGemvThreads) {
        const int m = i / vpr, v = i - m * vpr;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (m < a.M && v * 8 < len)
          val = *reinterpret_cast<const uint4*>(a.x + (size_t)m * K + kc0 + v * 8);
        reinterpret_cast<uint4*>(xs + (size_t)m * kc)[v] = val;
      }
    } else {
      for (int i = threadIdx.x; i < MT * kc; i += kGemvThreads) {
        const int m = i / kc, k = i - m * kc;
        xs[i] = (m < a.M && k < len) ? a.x[(size_t)m * K + kc0 + k] : __float2half_rn(0.0f);
      }
    }
    __syncthreads();
    if (!active) continue;

    if constexpr (VEC) {
      const int nvec = len / 8;
      const __half* wc = wrow + kc0;
      for (int v0 = part * 32; v0 < nvec; v0 += 32 * wpr * kGemvUnroll) {
        uint4 wv[kGemvUnroll];
#pragma unroll
        for (int u = 0; u < kGemvUnroll; ++u) {
          const int v = v0 + u * 32 * wpr + lane;
          wv[u] = (v < nvec) ? ldg_stream_16(wc + v * 8) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kGemvUnroll; ++u) {
          const int v = v0 + u * 32 * wpr + lane;
          if (v < nvec) {
            float wf[8];
            unpack8(wv[u], wf);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              float xf[8];
              unpack8(reinterpret_cast<const uint4*>(xs + (size_t)m * kc)[v], xf);
#pragma unroll
              for (int j = 0; j < 8; ++j) acc[m] = fmaf(wf[j], xf[j], acc[m]);
            }
          }
        }
      }
    } else {
      for (int k = part * 32 + lane; k < len; k += 32 * wpr) {
        const float wf = __half2float(wrow[kc0 + k]);
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = fmaf(wf, __half2float(xs[(size_t)m * kc + k]), acc[m]);
      }
    }
  }

  // lane sums -> warp sum (butterfly: every lane ends with the total)
#pragma unroll
  for (int m = 0; m < MT; ++m) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], off);
  }
  if (wpr > 1) {
    if (lane == 0) {
#pragma unroll
      for (int m = 0; m < MT; ++m) red[warp][m] = acc[m];
    }
    __syncthreads();
    if (part == 0) {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float s = red[warp][m];
        for (int j = 1; j < wpr; ++j) s += red[warp + j][m];
        acc[m] = s;
      }
    }
  }
  if (part == 0 && active) {
    const __half bn = a.b[row];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (lane == m && m < a.M) {
        const __half p = __float2half_rn(acc[m]);  // proj, rounded before the bias
        a.y[(size_t)m * a.N + row] = __hadd(p, bn);
      }
    }
  }
}

// K == 0: the sum is +0, so y[m, n] = RN16(+0 + b[n]) (a -0 bias gives +0).
__global__ void bias_only_kernel(const __half* __restrict__ b, __half* __restrict__ y, long long M,
                                 long long N) {
  const long long total = M * N;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    y[i] = __hadd(__float2half_rn(0.0f), b[i % N]);
  }
}

}  // namespace poot
