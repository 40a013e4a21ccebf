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

#include "epilogue.cuh"
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
  // the widened contraction (WIDE instantiations): x, W, b in the head
  // dtype, y by the per-element epilogue; `groups` independent contractions
  // (x [groups*M, K], W [groups*N, K], y and step operands [groups*M, ..],
  // b [groups*N]); 1 on the plain path
  ElemEpilogue e;
  int groups;
  int prefetch;  // tensor-core GEMV: bulk-prefetch each warp's W slice into L2 first
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

// eight binary16 (DT = kEpiF16) or bfloat16 values, widened exactly
template <int DT>
__device__ __forceinline__ void unpack8_t(const uint4 v, float (&f)[8]) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = ep_unpack_t<DT>(u[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// MT: M rounded up to 1, 2, 4, 8 or 16.  VEC: 16-byte loads of x and W
// (K % 8 == 0 and both 16-byte aligned); otherwise 2-byte loads.
template <int MT, bool VEC>
__global__ void __launch_bounds__(kGemvThreads) gemv_f16_kernel(const GemvArgs a) {
  grid_dep_wait();
  grid_dep_launch();
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

// M <= 2, 16-byte path: one warp per W row (or per K slice of a row when
// N is small), no shared-memory staging and no block barrier on the way.
// For each chunk of 32 * kGemvRowVpl vectors a lane issues all its W loads
// (16-byte vector v = chunk base + u * 32 + lane) before using any, then
// reads the matching x vectors through the read-only path (L2 once per SM,
// then L1) and accumulates in FP32.  On GB300 this streams W at about the
// rate of a plain read of the same bytes.
constexpr int kGemvRowWarps = 4;
constexpr int kGemvRowThreads = kGemvRowWarps * 32;
constexpr int kGemvRowVpl = 16;  // vectors per lane per chunk (16 * 32 * 8 = 4096 elements)

// DT: the operands' dtype; WIDE: the widened contraction's epilogue
// (a.e) instead of y = RN16(RN16(sum) + b).
template <int MT, int DT = kEpiF16, bool WIDE = false>
__global__ void __launch_bounds__(kGemvRowThreads, 8) gemv_f16_rows_kernel(const GemvArgs a) {
  __shared__ float red[kGemvRowWarps][MT];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wpr = a.wpr;
  const int row = blockIdx.x * (kGemvRowWarps / wpr) + warp / wpr;  // W row, over all groups
  const int part = warp % wpr;
  const bool active = row < a.N * a.groups;
  const int grp = WIDE ? row / a.N : 0;  // this row's group and column in it
  const int col = row - grp * a.N;
  const int nvec = a.K >> 3;
  // this warp's contiguous slice of the row, in whole chunks of 32 vectors
  const int segs = (nvec + 31) >> 5;
  const int seg_per_part = (segs + wpr - 1) / wpr;
  const int v_begin = min(nvec, part * seg_per_part * 32);
  const int v_end = min(nvec, (part + 1) * seg_per_part * 32);
  const uint4* __restrict__ wv = reinterpret_cast<const uint4*>(a.w + (size_t)(active ? row : 0) * a.K);
  const uint4* __restrict__ xv =
      reinterpret_cast<const uint4*>(a.x + (size_t)(active ? grp : 0) * (size_t)a.M * a.K);
  grid_dep_wait();

  // CH independent FMA chains per row (element j of a vector goes to chain
  // j % CH; the summation order is free): with one row the dependent chain,
  // not the loads, bounded the tail after the last W bytes arrive (GB300,
  // 1 x 4096 x 4096: 6.81 -> 6.69 us with four); two rows already have two
  // chains and more registers would cost occupancy
  constexpr int CH = MT == 1 ? 4 : 1;
  float acc[MT], part_acc[MT][CH];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int c = 0; c < CH; ++c) part_acc[m][c] = 0.0f;
  // b[row] is fetched now, beside the first W loads, not after the sum
  const __half bn = (!WIDE && active && part == 0) ? a.b[row] : __float2half_rn(0.0f);

  auto fma_vec = [&](const uint4 wvec, int v) {
    float wf[8];
    unpack8_t<DT>(wvec, wf);
#pragma unroll
    for (int m = 0; m < MT; ++m) {  // MT == M here (M <= 2)
      float xf[8];
      unpack8_t<DT>(__ldg(xv + (size_t)m * nvec + v), xf);
#pragma unroll
      for (int j = 0; j < 8; ++j) part_acc[m][j % CH] = fmaf(wf[j], xf[j], part_acc[m][j % CH]);
    }
  };
  if (active) {
    int c0 = v_begin;
    // whole chunks: no per-vector guards
    for (; c0 + 32 * kGemvRowVpl <= v_end; c0 += 32 * kGemvRowVpl) {
      uint4 wr[kGemvRowVpl];
#pragma unroll
      for (int u = 0; u < kGemvRowVpl; ++u) wr[u] = ldg_stream_16(wv + c0 + u * 32 + lane);
#pragma unroll
      for (int u = 0; u < kGemvRowVpl; ++u) fma_vec(wr[u], c0 + u * 32 + lane);
    }
    // tail: batches of four guarded vectors per lane
    for (; c0 < v_end; c0 += 32 * 4) {
      uint4 wr[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = c0 + u * 32 + lane;
        wr[u] = (v < v_end) ? ldg_stream_16(wv + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = c0 + u * 32 + lane;
        if (v < v_end) fma_vec(wr[u], v);
      }
    }
  }

#pragma unroll
  for (int m = 0; m < MT; ++m) {
    float t = part_acc[m][0];
#pragma unroll
    for (int c = 1; c < CH; ++c) t += part_acc[m][c];
    acc[m] = t;
  }
  // the W stream is done: let the next kernel in the stream start launching
  // (earlier, its blocks would compete with this grid's for SM slots)
  grid_dep_launch();
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
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (lane == m && m < a.M) {
        if constexpr (WIDE) {
          elem_store(a.e, acc[m], grp * a.M + m, col, row);
        } else {
          const __half p = __float2half_rn(acc[m]);  // proj, rounded before the bias
          a.y[(size_t)m * a.N + row] = __hadd(p, bn);
        }
      }
    }
  }
}

// 3 <= M <= 16, 16-byte path, on the tensor cores (mma.sync m16n8k16, FP16
// inputs, FP32 accumulators): on CUDA cores this range is bound by the
// FP32 FMAs, not by HBM.  A block owns a 16-row tile of W; its eight warps
// split K.  Per step of 32 along K, lane (g = lane / 4, t = lane % 4) loads
// the 16-byte vectors W[n0+g][k+8t .. +8), W[n0+g+8][k+8t .. +8) and
// x[g][k+8t .. +8) (and x[g+8][..] when M > 8).  The summation order is free
// (the contract's rule 1), so the K index inside a step is permuted: with
// that permutation these registers are exactly the A (W) and B (x^T)
// fragments of two m16n8k16 MMAs, and no shuffles are needed.  D[n][m]
// accumulates y^T; warps meet in shared memory in a fixed order.
// WARPS (8 or 16) split K: below two 16-row tiles per SM 16 warps keep
// twice the W bytes of a tile in flight; with more tiles 8 warps are better
// (GB300, M = 8, K = 4096, interleaved: N = 4096 7.15 us with 16 warps
// against 9.55 with 8; N = 6144 12.0 against 11.4; N = 8192 13.3 against
// 13.0; N = 14336 22.2 against 20.6).  The L2 bulk prefetch of each warp's
// slice pays only with few tiles (at most two for every three SMs), where
// it adds bytes in flight; with more it competes with the loads themselves
// (16 warps: N = 1024 4.9 us with the prefetch against 5.8 without; N =
// 4096 7.8 us without against 8.4 with).
constexpr int kGemvMmaWarpsFew = 16;
constexpr int kGemvMmaWarpsMany = 8;
// the 16-warp form for fewer than two 16-row tiles per SM
inline bool gemv_mma_few_tiles(long long tiles, int sm_count) { return tiles < 2LL * sm_count; }

__device__ __forceinline__ void mma_16816_f16_f32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                  uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// the same MMA on bfloat16 operands
__device__ __forceinline__ void mma_16816_bf16_f32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                   uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int DT>
__device__ __forceinline__ void mma_16816_f32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  if constexpr (DT == kEpiBf16) mma_16816_bf16_f32(d, a0, a1, a2, a3, b0, b1);
  else mma_16816_f16_f32(d, a0, a1, a2, a3, b0, b1);
}

// NT = number of 8-column blocks of m (1: M <= 8, 2: M <= 16); DT and WIDE
// as for gemv_f16_rows_kernel
template <int NT, int WARPS, int DT = kEpiF16, bool WIDE = false>
__global__ void __launch_bounds__(WARPS * 32) gemv_f16_mma_kernel(const GemvArgs a) {
  __shared__ float red[WARPS][32][4 * NT];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int K = a.K, N = a.N, M = a.M;
  // WIDE: 16-row tiles of W per group (a tile never spans two groups)
  int grp = 0, n0 = blockIdx.x * 16;
  if constexpr (WIDE) {
    const int tpg = (N + 15) / 16;
    grp = (int)blockIdx.x / tpg;
    n0 = ((int)blockIdx.x - grp * tpg) * 16;
  }
  const int nA = n0 + g, nB = n0 + g + 8;
  // this warp's K slice, a multiple of 32
  const int slice = ((K + WARPS * 32 - 1) / (WARPS * 32)) * 32;
  const int k_begin = min(K, warp * slice);
  const int k_end = min(K, k_begin + slice);
  const __half* __restrict__ wa = a.w + (size_t)(nA < N ? nA : 0) * K;
  const __half* __restrict__ wb = a.w + (size_t)(nB < N ? nB : 0) * K;
  const __half* __restrict__ x0 = a.x + (size_t)(g < M ? g : 0) * K;
  const __half* __restrict__ x1 = a.x + (size_t)(g + 8 < M ? g + 8 : 0) * K;
  if constexpr (WIDE) {
    // this group's W rows and x rows
    wa += (size_t)grp * N * K;
    wb += (size_t)grp * N * K;
    x0 += (size_t)grp * M * K;
    x1 += (size_t)grp * M * K;
  }
  const bool okA = nA < N, okB = nB < N, okx0 = g < M, okx1 = (NT > 1) && (g + 8 < M);
  // start this warp's K slice of its 16 W rows towards L2 while the
  // previous grid drains (lane 4g prefetches rows nA and nB)
  if (a.prefetch && t == 0 && k_end > k_begin) {
    if (okA) prefetch_l2_bulk(wa + k_begin, (uint32_t)(k_end - k_begin) * 2u);
    if (okB) prefetch_l2_bulk(wb + k_begin, (uint32_t)(k_end - k_begin) * 2u);
  }
  grid_dep_wait();
  grid_dep_launch();
  // bias of this lane's two output features, fetched early
  const float bA = (!WIDE && warp == 0 && okA) ? __half2float(a.b[nA]) : 0.0f;
  const float bB = (!WIDE && warp == 0 && okB) ? __half2float(a.b[nB]) : 0.0f;

  // two accumulator sets, even and odd steps along K, added at the end (the
  // summation order is free): halves the chain of dependent MMAs a warp
  // waits on once its loads have landed (GB300, 8 x 4096 x 4096: 7.68 ->
  // 7.11 us)
  float d[NT][4], d2[NT][4];
#pragma unroll
  for (int q = 0; q < NT; ++q) {
    d[q][0] = d[q][1] = d[q][2] = d[q][3] = 0.0f;
    d2[q][0] = d2[q][1] = d2[q][2] = d2[q][3] = 0.0f;
  }
  const uint4 zero = make_uint4(0, 0, 0, 0);

  constexpr int U = NT == 1 ? 8 : 4;  // steps of 32 along K per batch
  for (int k0 = k_begin; k0 < k_end; k0 += 32 * U) {
    uint4 va[U], vb[U], vx[U][NT];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int k = k0 + 32 * u + 8 * t;
      const bool in = k < k_end;  // K % 8 == 0: whole vector in or out
      va[u] = (in && okA) ? ldg_stream_16(wa + k) : zero;
      vb[u] = (in && okB) ? ldg_stream_16(wb + k) : zero;
      vx[u][0] = (in && okx0) ? __ldg(reinterpret_cast<const uint4*>(x0 + k)) : zero;
      if (NT > 1) vx[u][NT - 1] = (in && okx1) ? __ldg(reinterpret_cast<const uint4*>(x1 + k)) : zero;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int q = 0; q < NT; ++q) {
        float(&acc)[4] = (u & 1) ? d2[q] : d[q];
        mma_16816_f32<DT>(acc, va[u].x, vb[u].x, va[u].y, vb[u].y, vx[u][q].x, vx[u][q].y);
        mma_16816_f32<DT>(acc, va[u].z, vb[u].z, va[u].w, vb[u].w, vx[u][q].z, vx[u][q].w);
      }
    }
  }
#pragma unroll
  for (int q = 0; q < NT; ++q)
#pragma unroll
    for (int i = 0; i < 4; ++i) d[q][i] += d2[q][i];

#pragma unroll
  for (int q = 0; q < NT; ++q)
#pragma unroll
    for (int i = 0; i < 4; ++i) red[warp][lane][4 * q + i] = d[q][i];
  __syncthreads();
  if (warp != 0) return;
#pragma unroll
  for (int q = 0; q < NT; ++q) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float s = red[0][lane][4 * q + i];
      for (int wi = 1; wi < WARPS; ++wi) s += red[wi][lane][4 * q + i];
      // D[n][m]: i = 0, 1 -> (n = nA, m = 2t + i); i = 2, 3 -> (n = nB, m = 2t + i - 2)
      const int m = 8 * q + 2 * t + (i & 1);
      const int n = (i < 2) ? nA : nB;
      if (m < M && n < N) {
        if constexpr (WIDE) {
          elem_store(a.e, s, grp * M + m, n, grp * N + n);
        } else {
          const __half p = __float2half_rn(s);  // proj, rounded before the bias
          a.y[(size_t)m * N + n] = __hadd(p, __float2half_rn(i < 2 ? bA : bB));
        }
      }
    }
  }
}

// K == 0: the sum is +0, so y[m, n] = RN16(+0 + b[n]) (a -0 bias gives +0).
__global__ void bias_only_kernel(const __half* __restrict__ b, __half* __restrict__ y, long long M,
                                 long long N) {
  grid_dep_wait();
  grid_dep_launch();
  const long long total = M * N;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    y[i] = __hadd(__float2half_rn(0.0f), b[i % N]);
  }
}

}  // namespace poot
