// y = FP16(x . W^T) + b on the 5th-generation tensor cores (tcgen05).
//
// One persistent CTA per SM walks output tiles of 128 x BN in a grouped
// order (CTAs running together share rows of x and W in L2).  Warp roles:
//   warps 0-7  epilogue.  Warp w reads TMEM lanes 32*(w%4) .. +31 (tile
//              rows) and owns one half of the tile's columns.  After each K
//              chunk it moves the chunk's FP32 sums from TMEM into an FP32
//              register accumulator (tcgen05.ld + IEEE round-to-nearest
//              adds).  After the last chunk: proj = RN16(acc)
//              (cvt.rn.f16x2.f32), y = RN16(proj + b[n]) (HADD2), staged in
//              shared memory and written by TMA stores (plain stores when
//              y's pitch is not 16-byte aligned).  proj never reaches HBM.
//   warp 8     TMEM allocator and single-thread MMA issuer: per K block of 64,
//              four tcgen05.mma kind::f16 (M=128, N=BN, K=16) into one of two
//              TMEM chunk buffers; a chunk is chunk_kb K blocks.
//   warps 9+   producer: TMA tiles of x [128 x 64] and W [BN x 64], both
//              K-major with the 128-byte swizzle, into a ring of stages; or,
//              for row pitches TMA cannot address (K % 8 != 0 or unaligned
//              pointers), three warps that copy the same swizzled layout with
//              4-byte cp.async or 2-byte register copies.
// Tails in M, N and K: TMA zero-fills out-of-range reads (zeros add nothing
// to the sum) and clips stores; the copy producers zero-fill by predicate.
//
// Numerical contract ("Tensor Programs, Part 1", section "One Program and One
// Numerical Contract"): products enter an FP32 sum unrounded (the tensor
// core forms exact products of binary16 inputs), the FP32 result is rounded
// to FP16 before the bias is added, and y is FP16.  The chunked promotion
// keeps each tensor-core accumulation chain short: the tensor core aligns
// addends to the running sum with truncation, so a long chain against a
// large sum loses more than a round-to-nearest sum would; restarting every
// chunk and adding chunk sums in IEEE FP32 keeps the result within two FP16
// ulps of a sequential FP32 sum on cancelling sums as well.
#pragma once

#include "epilogue.cuh"
#include "ptx.cuh"

namespace poot {

enum LoadMode : int { kLoadTma = 0, kLoadCpAsync4 = 1, kLoadReg16 = 2 };

struct GemmArgs {
  const __half* x;
  const __half* w;
  const __half* b;
  __half* y;
  int M, N, K;
  int bn;        // output tile width: multiple of 32 in [64, 256] (the MMA's N)
  int stages;    // operand ring depth, 4 .. kGemmMaxStages
  int group_m;   // tile-order group height in M blocks
  int chunk_kb;  // K blocks accumulated in TMEM before promotion (>= 1)
  int num_m_blocks, num_n_blocks, num_k_blocks, num_tiles;
  int tma_store;  // 1: TMA store of y; 0: plain stores (any pitch/alignment)
  // 1: stages are filled, consumed and released in pairs, and a chunk's last
  // pair is released through the chunk-complete barrier (TMA producer, even
  // `stages`, every chunk an even number of at least `stages` K blocks);
  // 0: one stage at a time
  int paired;
  // The widened contraction (poot_contract).  general == 0: the plain
  // binary16 epilogue y = RN16(RN16(sum) + b).  general == 1: head dtype
  // `dtype`, optional bias, FP32 output or the epilogue steps.
  int general;
  int dtype;     // EpiDtype: x, W, b, step operands and y
  int out_f32;   // y32 = sum (+ b in FP32); no head rounding, no steps
  int has_bias;  // b is read (always 1 on the plain path)
  int y_vec;     // out_f32: 16-byte stores (y32 16-byte aligned, N % 4 == 0)
  int num_steps;
  int ep_op[kEpiMaxSteps];
  int ep_vec[kEpiMaxSteps];  // operand 16-byte aligned with ld % 8 == 0
  const uint16_t* ep_ptr[kEpiMaxSteps];
  long long ep_ld[kEpiMaxSteps];
  float* y32;
  // grouped contraction (GEN only): tile t belongs to group t / tiles_per_group;
  // x is [groups*M, K], W is [groups*N, K], y [groups, M, N], b [groups*N],
  // step operands [groups*M, ld]
  int groups;
  int tiles_per_group;
  // split K (GEN only, groups == split_k > 1): "group" g is split g of one
  // contraction, summing K blocks g*num_k_blocks .. (g+1)*num_k_blocks-1 of x
  // and W (no row offsets) into the FP32 partial tile y32 + g*M*N
  int split_k;
};

// Activation step over the 16 packed pairs of one 32-column box, the op and
// dtype dispatched once per box, so each loop body is straight-line code.
__device__ __forceinline__ void gemm_epi_activation16(uint32_t* v, int op, int dt) {
  if (dt == kEpiBf16) {
    switch (op) {
      case kEpSilu: ep_activation_pairs<kEpSilu, kEpiBf16, 16>(v); break;
      case kEpGeluTanh: ep_activation_pairs<kEpGeluTanh, kEpiBf16, 16>(v); break;
      case kEpGeluErf: ep_activation_pairs<kEpGeluErf, kEpiBf16, 16>(v); break;
      default: break;
    }
  } else {
    switch (op) {
      case kEpSilu: ep_activation_pairs<kEpSilu, kEpiF16, 16>(v); break;
      case kEpGeluTanh: ep_activation_pairs<kEpGeluTanh, kEpiF16, 16>(v); break;
      case kEpGeluErf: ep_activation_pairs<kEpGeluErf, kEpiF16, 16>(v); break;
      default: break;
    }
  }
}

// The same, out of line: the copy-producer kernels (168 registers, no
// register split) apply it box by box with the tile's sums live, and an
// inlined copy per box would cost them registers.
__device__ __noinline__ void gemm_epi_activation16_call(uint32_t* v, int op, int dt) {
  gemm_epi_activation16(v, op, dt);
}

enum GemmEpi : int { kEpiPlain = 0, kEpiHead = 1, kEpiFull = 2 };

constexpr int kGemmBM = 128;
constexpr int kGemmBK = 64;        // one 128-byte swizzle row of binary16
constexpr int kGemmMaxBN = 256;
constexpr int kGemmMaxStages = 8;
constexpr int kGemmEpiWarps = 8;
constexpr int kGemmMmaWarp = 8;
constexpr int kGemmProdWarp0 = 9;
constexpr int kGemmCopyThreads = 96;                 // copy producers: three warps
constexpr uint32_t kGemmTmemCols = 2 * kGemmMaxBN;  // two chunk buffers, 256 columns apart
constexpr int kGemmHalfCols = kGemmMaxBN / 2;        // columns per epilogue warp (max)

__host__ __device__ constexpr int gemm_prod_warps(int mode) { return mode == kLoadTma ? 1 : 3; }
// Register split of the TMA kernels.  A CTA of ten or twelve warps places
// three warps on some SM sub-partitions, whose 16K registers then cap every
// thread at 168: the epilogue warps, which hold a tile's FP32 sums, spilled
// there.  The TMA kernels therefore launch twelve warps (warps 10 and 11 do
// nothing) at 168 registers, and after the prologue the warpgroup of the
// MMA issuer and the producer gives registers back (setmaxnreg.dec to 56)
// while the two epilogue warpgroups take them (setmaxnreg.inc to 224):
// 256 * 224 + 128 * 56 = 384 * 168, so the increase never waits on
// registers that are not there (the host checks the launch count).
constexpr int kGemmLaunchRegs = 168;
constexpr int kGemmEpiRegs = 224;
constexpr int kGemmCtlRegs = 56;
static_assert(8 * 32 * kGemmEpiRegs + 4 * 32 * kGemmCtlRegs <= 12 * 32 * kGemmLaunchRegs,
              "the register split must fit the registers the CTA is launched with");
__host__ __device__ constexpr int gemm_threads(int mode) {
  return mode == kLoadTma ? 12 * 32 : (kGemmProdWarp0 + gemm_prod_warps(mode)) * 32;
}

// Shared-memory layout (offsets from a 1024-byte-aligned base).  The operand
// ring holds `stages` stages of A [128 x 64] followed by B [bn x 64]; every
// stage and both tiles start on 1024-byte boundaries (bn % 8 == 0).
struct GemmLayout {
  static constexpr int A_BYTES = kGemmBM * kGemmBK * 2;  // 16 KB
  static constexpr int RING_BYTES = 192 * 1024;
  static constexpr int STG_BYTES = 32 * 32 * 2;          // one 32 x 32 output box
  static constexpr int OFF_STG = RING_BYTES;
  static constexpr int OFF_BAR = OFF_STG + kGemmEpiWarps * 2 * STG_BYTES;
  static constexpr int NUM_BARS = 2 * kGemmMaxStages + 5;  // full, empty, cfull x2, cempty x2, drain
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
  static constexpr int BYTES = OFF_ABORT + 4;
  static constexpr int DYN_BYTES = BYTES + 1024;  // room to align the base
  static_assert(OFF_BAR % 8 == 0, "mbarriers are 8-byte objects");
  static_assert(DYN_BYTES <= 232448, "more shared memory than a CTA can have");
};

// W rows a CTA loads per stage: the whole tile width, or half of it when a
// CTA pair shares the W tile (2-SM MMA).
__host__ __device__ constexpr int gemm_b_rows(int bn, bool pair) { return pair ? bn / 2 : bn; }
__host__ __device__ constexpr int gemm_b_bytes(int bn, bool pair = false) { return gemm_b_rows(bn, pair) * kGemmBK * 2; }
__host__ __device__ constexpr int gemm_stage_bytes(int bn, bool pair = false) {
  return GemmLayout::A_BYTES + gemm_b_bytes(bn, pair);
}
__host__ __device__ constexpr int gemm_max_stages(int bn, bool pair = false) {
  return GemmLayout::RING_BYTES / gemm_stage_bytes(bn, pair) < kGemmMaxStages
             ? GemmLayout::RING_BYTES / gemm_stage_bytes(bn, pair) : kGemmMaxStages;
}
// Columns of the first epilogue half (a multiple of 32); the second half
// takes the rest.
__host__ __device__ constexpr int gemm_half0_cols(int bn) { return ((bn / 32 + 1) / 2) * 32; }

// Tile t -> (M block, N block): groups of group_m M blocks are walked column
// by column, so CTAs running at the same time share x rows and W rows in L2.
// Odd groups walk the columns from the far end: they start on the W rows
// the previous group read last, which L2 still holds (8192 x 14336 x 4096:
// DRAM reads 360 -> 350 MB).
__device__ __forceinline__ void gemm_tile_coords(int t, int num_m, int num_n, int group_m, int& mb,
                                                 int& nb) {
  const int span = group_m * num_n;
  const int g = t / span;
  const int first_m = g * group_m;
  const int gsize = min(num_m - first_m, group_m);
  const int local = t - g * span;
  mb = first_m + local % gsize;
  nb = local / gsize;
  if (g & 1) nb = num_n - 1 - nb;
}

// Register-copy producer (2-byte loads, any alignment): fills one operand
// tile (rows row0 .. row0+rows-1 of src, K block at k0) in the
// 128-byte-swizzled K-major layout, zero outside
// [nrows) x [K).  Row r, 16-byte chunk c lands at r*128 + ((c ^ (r & 7)) * 16).
// pt is the thread's index among the kGemmCopyThreads producer threads.
template <int MODE>
__device__ __forceinline__ void gemm_copy_tile(uint32_t dst_base, const __half* __restrict__ src,
                                               int rows, int row0, int nrows, int K, int k0, int pt) {
  constexpr int T = kGemmCopyThreads;
  static_assert(MODE == kLoadReg16, "the cp.async producers use gemm_copy_rows_cp");
  {
    // 16-byte chunks assembled from 2-byte loads: rows x 8 chunks, eight
    // chunks per thread in flight at a time.
    constexpr int PER = 8;
    const int chunks = rows * 8;
    for (int base = 0; base < chunks; base += T * PER) {
      uint32_t v[PER][4];
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int ch = base + pt + i * T;
        const int r = ch >> 3, c = ch & 7;
        const int grow = row0 + r, kb = k0 + c * 8;
        unsigned short e[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const bool ok = (ch < chunks) && (grow < nrows) && (kb + j < K);
          e[j] = ok ? __ldg(reinterpret_cast<const unsigned short*>(src) + (size_t)grow * K + kb + j)
                    : (unsigned short)0;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) v[i][j] = (uint32_t)e[2 * j] | ((uint32_t)e[2 * j + 1] << 16);
      }
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int ch = base + pt + i * T;
        if (ch < chunks) {
          const int r = ch >> 3, c = ch & 7;
          const uint32_t d = dst_base + r * 128 + ((c ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(d), "r"(v[i][0]), "r"(v[i][1]),
                       "r"(v[i][2]), "r"(v[i][3])
                       : "memory");
        }
      }
    }
  }
}

// cp.async producer: fills one operand tile with WB-byte words (4, or 8 when
// K % 4 == 0 and the operand is 8-byte aligned).  Copy warp cw of the three
// takes every third group of RPI rows; within a warp instruction lane l
// copies word l % LPR of row l / LPR, so one instruction moves 128 bytes of
// each of its rows.  Row r, byte b lands at r*128 + (((b >> 4) ^ (r & 7)) << 4)
// + (b & 15); words outside [nrows) x [K) are zero-filled.
template <int WB>
__device__ __forceinline__ void gemm_copy_rows_cp(uint32_t dst_base, const __half* __restrict__ src, int rows,
                                                  int row0, int nrows, int K, int k0, int cw, int lane) {
  constexpr int LPR = 128 / WB;  // lanes per row
  constexpr int RPI = 32 / LPR;  // rows per warp instruction
  constexpr int RSTEP = 3 * RPI;
  const int wl = lane % LPR;
  const int kk = k0 + wl * (WB / 2);
  const bool kok = kk < K;  // K is a multiple of WB / 2 elements: a word is all in or all out
  const uint32_t b = (uint32_t)(wl * WB);
  int r = cw * RPI + lane / LPR;
  const char* g = reinterpret_cast<const char*>(src) + ((size_t)(row0 + r) * K + kk) * 2;
  const size_t gstep = (size_t)RSTEP * K * 2;
  for (; r < rows; r += RSTEP, g += gstep) {
    const bool ok = kok && (row0 + r < nrows);
    const uint32_t d = dst_base + (uint32_t)r * 128u + ((((b >> 4) ^ (uint32_t)(r & 7))) << 4) + (b & 15u);
    if constexpr (WB == 8) cp_async_8(d, ok ? (const void*)g : (const void*)src, ok ? 8u : 0u);
    else cp_async_4(d, ok ? (const void*)g : (const void*)src, ok ? 4u : 0u);
  }
}

// CL = cluster size.  CL = 1: one CTA per 128 x BN tile.
// CL = 2: 2-SM MMA.  Two CTAs of a cluster (a pair: ranks 0 and 1) compute
// one 256 x BN output tile: each loads its 128 rows of x and BN/2 rows of W
// into its own shared memory, the even CTA issues tcgen05.mma.cta_group::2
// for both (each CTA's TMEM receives its 128 rows), and commits arrive in
// both CTAs.  The odd CTA's TMA loads complete on the even CTA's "full"
// barriers, and both CTAs' epilogue warps release chunk buffers on the even
// CTA's "cempty" barriers.  Per SM a stage holds 32 KB instead of 48 KB
// (BN = 256), so the ring is six stages deep, and W is read once per pair.
// EPI selects the epilogue compiled in: kEpiPlain, the plain binary16
// y = RN16(RN16(sum) + b) (the kernel ignores the fields that select the
// rest); kEpiHead, the widened contraction's head dtype and optional bias
// (groups included); kEpiFull, everything of the widened contraction (FP32
// output, epilogue steps, split-K partial sums).  The lighter forms keep
// fewer registers live in the epilogue.
template <int MODE, int CL, int EPI = kEpiPlain>
__global__ void __launch_bounds__(gemm_threads(MODE), 1)
    gemm_f16_tcgen05_kernel(const __grid_constant__ CUtensorMap tm_x,
                            const __grid_constant__ CUtensorMap tm_w,
                            const __grid_constant__ CUtensorMap tm_y, const GemmArgs args) {
  constexpr bool PAIR = CL >= 2;
  constexpr bool GEN = EPI != kEpiPlain;  // the widened contraction's fields are read
  constexpr bool FULL = EPI == kEpiFull;  // FP32 output, steps, split-K partial sums
  static_assert(CL == 1 || CL == 2, "one CTA or a CTA pair");
  static_assert(!PAIR || MODE == kLoadTma, "the CTA-pair kernel loads through TMA only");
  using L = GemmLayout;
  const int BN = args.bn;
  const int STAGES = args.stages;
  const int STAGE_BYTES = gemm_stage_bytes(BN, PAIR);
  // A and B both binary16, or both bfloat16 (bits 7-9 and 10-12: format 1)
  const uint32_t IDESC = idesc_f16_f32acc(PAIR ? 2 * kGemmBM : kGemmBM, (uint32_t)BN) |
                         ((GEN && args.dtype == kEpiBf16) ? ((1u << 7) | (1u << 10)) : 0u);
  const uint32_t crank = PAIR ? cluster_ctarank() : 0u;
  const uint32_t rank = crank & 1u;               // row half of the pair's tile
  const uint32_t lead_rank = crank & ~1u;         // even CTA of this pair
  const bool leader = (rank == 0);
  const int unit = (int)(blockIdx.x / CL);        // cluster (or CTA) index
  const int units = (int)(gridDim.x / CL);
  const int tile_rows = PAIR ? 2 * kGemmBM : kGemmBM;
  const int num_kb = args.num_k_blocks;
  const int chunk_kb = args.chunk_kb;
  const int num_chunks = (num_kb + chunk_kb - 1) / chunk_kb;

  // tile t -> (group, M block, N block)
  auto tile_decode = [&](int t, int& g, int& mb, int& nb) {
    int tl = t;
    g = 0;
    if constexpr (GEN) {
      g = t / args.tiles_per_group;
      tl = t - g * args.tiles_per_group;
    }
    gemm_tile_coords(tl, args.num_m_blocks, args.num_n_blocks, args.group_m, mb, nb);
  };

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + L::OFF_BAR;
  auto bar_full = [&](int s) { return bar0 + 8u * s; };
  auto bar_empty = [&](int s) { return bar0 + 8u * (kGemmMaxStages + s); };
  auto bar_cfull = [&](int a) { return bar0 + 8u * (2 * kGemmMaxStages + a); };
  auto bar_cempty = [&](int a) { return bar0 + 8u * (2 * kGemmMaxStages + 2 + a); };
  const uint32_t bar_drain = bar0 + 8u * (2 * kGemmMaxStages + 4);
  auto stage_a = [&](int s) { return sbase + (uint32_t)(s * STAGE_BYTES); };
  auto stage_b = [&](int s) { return sbase + (uint32_t)(s * STAGE_BYTES + L::A_BYTES); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEM_SLOT);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full(s), MODE == kLoadTma ? 1u : (uint32_t)kGemmCopyThreads);
      mbar_init(bar_empty(s), 1u);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_cfull(a), 1u);
      mbar_init(bar_cempty(a), (uint32_t)(PAIR ? 2 * kGemmEpiWarps : kGemmEpiWarps));
    }
    mbar_init(bar_drain, 1u);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kGemmMmaWarp) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_addr(tmem_slot), kGemmTmemCols);
      tmem_relinquish_alloc_permit_pair();
    } else {
      tmem_alloc(smem_addr(tmem_slot), kGemmTmemCols);
      tmem_relinquish_alloc_permit();
    }
  }
  if (MODE == kLoadTma && warp == kGemmProdWarp0 && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_w);
  }
  if (warp == 0 && lane == 0 && args.tma_store) tma_prefetch_desc(&tm_y);
  // the next kernel in the stream may start launching now: its CTAs can only
  // take SMs this grid leaves free, and it touches global memory only after
  // this grid has completed (its own grid_dep_wait)
  grid_dep_launch();
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // both CTAs' barriers exist before any remote signal
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // prologue done; global memory is touched only after the previous grid
  grid_dep_wait();

  if (warp >= kGemmMmaWarp) {
  // the MMA issuer's and the producers' warpgroup (setmaxnreg is executed by
  // every warp of a warpgroup together)
  if constexpr (MODE == kLoadTma) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kGemmCtlRegs) : "memory");
  if (MODE == kLoadTma && warp > kGemmProdWarp0) {
    // warps 10 and 11 of the TMA kernels: no role
  } else if (warp >= kGemmProdWarp0) {
    // ------------------------------------------------------------ producer
    if constexpr (MODE == kLoadTma) {
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        long long issued = 0;
        bool ok = true;
        // Paired stages (args.paired): stages 2p and 2p+1 are filled together
        // and released together through empty barrier p, and a chunk's last
        // pair is released by the chunk-complete barrier instead (every chunk
        // holds at least STAGES K blocks, so the fill at position STAGES - 2
        // of chunk ch reuses the pair of chunk ch - 1's end).  ck: position
        // in the chunk; ch: chunk count over this CTA's tiles (TMEM buffer and
        // barrier phase).
        const bool paired = args.paired != 0;
        const int step = paired ? 2 : 1;
        // x tiles are marked evict-last in L2: a group of M blocks is read
        // by every N block of its walk while W streams past it (8192 x
        // 14336 x 4096: DRAM reads 332 -> 327 MB; prefill 81.7 -> 81.0 us)
        const uint64_t xpol = l2_policy_evict_last();
        int ck = 0, ch = 0;
        for (int t = unit; t < args.num_tiles && ok; t += units) {
          int g, mb, nb;
          tile_decode(t, g, mb, nb);
          // rows of this group in the flattened x [groups*M, K] and W [groups*N, K]
          // (a tile that overhangs its group reads rows of the next one; they
          // only reach output rows or columns that are never stored)
          const bool ksplit = FULL && args.split_k > 1;
          const int xrow0 = ksplit ? 0 : g * args.M, wrow0 = ksplit ? 0 : g * args.N;
          const int kofs = ksplit ? g * num_kb * kGemmBK : 0;  // this split's first K element
          for (int kb = 0; kb < num_kb; kb += step) {
            const uint32_t eb = paired ? bar_empty(stage >> 1) : bar_empty(stage);
            if (paired && ck == STAGES - 2 && ch > 0) {
              const int pc = ch - 1;
              if (!mbar_wait(bar_cfull(pc & 1), (uint32_t)((pc >> 1) & 1), abort_flag)) { ok = false; break; }
              mbar_arrive(eb);  // in place of the MMA's commit
            }
            // the first pass over the ring and the first two chunk buffers
            // find them free: no wait (it would only add latency to the start)
            if (issued >= STAGES && !mbar_wait(eb, phase ^ 1u, abort_flag)) { ok = false; break; }
            if (paired && leader && ck == 0 && ch >= 2) {
              // the chunk's TMEM buffer must be drained before its first MMA;
              // that MMA waits on this stage's full barrier, so the producer
              // waits for the buffer before arming the barrier
              if (!mbar_wait(bar_cempty(ch & 1), (uint32_t)(((ch >> 1) & 1) ^ 1), abort_flag)) { ok = false; break; }
            }
            for (int h = 0; h < step; ++h) {
              const int st = stage + h, kc = kofs + (kb + h) * kGemmBK;
              const uint32_t fb = bar_full(st);
              if constexpr (PAIR) {
                // both CTAs' bytes complete on the even CTA's barrier
                const uint32_t fb0 = map_to_cta(fb, lead_rank);
                if (leader) mbar_arrive_expect_tx(fb, (uint32_t)(2 * STAGE_BYTES));
                const int arow = xrow0 + mb * tile_rows + (int)rank * kGemmBM;
                tma_load_2d_pair_hint(stage_a(st), &tm_x, fb0, kc, arow, xpol);
                tma_load_2d_pair(stage_b(st), &tm_w, fb0, kc, wrow0 + nb * BN + (int)rank * (BN / 2));
              } else {
                mbar_arrive_expect_tx(fb, (uint32_t)STAGE_BYTES);
                tma_load_2d_hint(stage_a(st), &tm_x, fb, kc, xrow0 + mb * kGemmBM, xpol);
                tma_load_2d(stage_b(st), &tm_w, fb, kc, wrow0 + nb * BN);
              }
            }
            if (ck + step >= chunk_kb || kb + step >= num_kb) { ck = 0; ++ch; } else { ck += step; }
            issued += step;
            stage += step;
            if (stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
        // Let the last loads land before the CTA can exit (their barrier
        // phases complete on their own; nothing else arrives there).  In a
        // pair the even CTA's barriers also count the odd CTA's bytes; the
        // odd CTA is held by the closing cluster barrier instead.
        if (leader) {
          int s = stage;
          uint32_t ph = phase;
          for (int i = 0; i < STAGES && i < issued; ++i) {
            if (s == 0) { s = STAGES - 1; ph ^= 1u; } else { --s; }
            mbar_wait(bar_full(s), ph, nullptr);
          }
        }
      }
    } else {
      const int pt = threadIdx.x - kGemmProdWarp0 * 32;  // 0 .. kGemmCopyThreads-1
      const int cw = pt >> 5;                             // copy warp 0 .. 2
      // cp.async: copies of a stage complete LAG fills after they are issued;
      // LAG < STAGES (STAGES >= 4) keeps the ring from deadlocking
      constexpr int LAG = (MODE == kLoadCpAsync4) ? 3 : 0;
      // 8-byte words when every row start and K slice is 8-byte aligned
      const bool w8 = (args.K % 4 == 0) && ((reinterpret_cast<uintptr_t>(args.x) | reinterpret_cast<uintptr_t>(args.w)) % 8 == 0);
      int stage = 0, done_stage = 0;  // ring slot to fill next; slot whose copies complete next
      uint32_t phase = 0;
      int filled = 0;                 // fills issued (saturates at LAG)
      bool ok = true;
      for (int t = unit; t < args.num_tiles && ok; t += units) {
        int g, mb, nb;
        tile_decode(t, g, mb, nb);
        const bool ksplit = FULL && args.split_k > 1;
        const __half* xg = ksplit ? args.x : args.x + (size_t)g * args.M * args.K;
        const __half* wg = ksplit ? args.w : args.w + (size_t)g * args.N * args.K;
        const int kofs = ksplit ? g * num_kb * kGemmBK : 0;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(bar_empty(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
          if constexpr (MODE == kLoadCpAsync4) {
            if (w8) {
              gemm_copy_rows_cp<8>(stage_a(stage), xg, kGemmBM, mb * kGemmBM, args.M, args.K, kofs + kb * kGemmBK, cw, lane);
              gemm_copy_rows_cp<8>(stage_b(stage), wg, BN, nb * BN, args.N, args.K, kofs + kb * kGemmBK, cw, lane);
            } else {
              gemm_copy_rows_cp<4>(stage_a(stage), xg, kGemmBM, mb * kGemmBM, args.M, args.K, kofs + kb * kGemmBK, cw, lane);
              gemm_copy_rows_cp<4>(stage_b(stage), wg, BN, nb * BN, args.N, args.K, kofs + kb * kGemmBK, cw, lane);
            }
            cp_async_commit();
            if (filled == LAG) {
              cp_async_wait_group<LAG>();
              fence_proxy_async_smem();
              mbar_arrive(bar_full(done_stage));
              if (++done_stage == STAGES) done_stage = 0;
            } else {
              ++filled;
            }
          } else {
            gemm_copy_tile<MODE>(stage_a(stage), xg, kGemmBM, mb * kGemmBM, args.M, args.K, kofs + kb * kGemmBK, pt);
            gemm_copy_tile<MODE>(stage_b(stage), wg, BN, nb * BN, args.N, args.K, kofs + kb * kGemmBK, pt);
            fence_proxy_async_smem();
            mbar_arrive(bar_full(stage));
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if constexpr (MODE == kLoadCpAsync4) {
        // the last `filled` fills (at most LAG) have not been signalled yet
        cp_async_wait_all();
        fence_proxy_async_smem();
        for (int j = 0; j < filled; ++j) {
          mbar_arrive(bar_full(done_stage));
          if (++done_stage == STAGES) done_stage = 0;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      const bool paired = MODE == kLoadTma && args.paired != 0;
      if (paired) {
        // Two K blocks (two stages, eight MMAs) per iteration over all of
        // this CTA's tiles, one commit each, every tcgen05 instruction
        // unconditional: measured on GB300, a commit under a branch (even one
        // never taken) or a wait and commit per four MMAs leaves gaps in the
        // tensor pipe, eight MMAs per wait and commit do not.  A chunk's
        // first MMA starts a fresh sum (accumulate off); its last pair
        // commits to the chunk-complete barrier, which also frees the pair
        // (the producers turn it into the pair's release), and the producer
        // has already waited for the chunk's TMEM buffer before arming it.
        const int my_tiles = unit < args.num_tiles ? (args.num_tiles - 1 - unit) / units + 1 : 0;
        const long long total = (long long)my_tiles * num_kb;
        int stage = 0;
        uint32_t phase = 0;
        int buf = 0;
        int ck = 0, kb = 0;  // K block within the chunk and within the tile
        for (long long g = 0; g < total; g += 2) {
          if (!mbar_wait(bar_full(stage), phase, abort_flag)) break;
          if (!mbar_wait(bar_full(stage + 1), phase, abort_flag)) break;
          tc_fence_after_sync();
          const bool last = (ck + 2 >= chunk_kb) || (kb + 2 >= num_kb);
          const uint32_t d_tmem = tmem_base + (uint32_t)(buf * kGemmMaxBN);
          const uint64_t a0 = sdesc_kmajor_sw128(stage_a(stage)), b0 = sdesc_kmajor_sw128(stage_b(stage));
          const uint64_t a1 = sdesc_kmajor_sw128(stage_a(stage + 1)), b1 = sdesc_kmajor_sw128(stage_b(stage + 1));
#pragma unroll
          for (int k = 0; k < kGemmBK / 16; ++k) {
            if constexpr (PAIR)
              umma_f16_pair(d_tmem, a0 + 2u * k, b0 + 2u * k, IDESC, (ck == 0 && k == 0) ? 0u : 1u);
            else
              umma_f16(d_tmem, a0 + 2u * k, b0 + 2u * k, IDESC, (ck == 0 && k == 0) ? 0u : 1u);
          }
#pragma unroll
          for (int k = 0; k < kGemmBK / 16; ++k) {
            if constexpr (PAIR)
              umma_f16_pair(d_tmem, a1 + 2u * k, b1 + 2u * k, IDESC, 1u);
            else
              umma_f16(d_tmem, a1 + 2u * k, b1 + 2u * k, IDESC, 1u);
          }
          const uint32_t cbar = last ? bar_cfull(buf) : bar_empty(stage >> 1);
          if constexpr (PAIR) umma_commit_pair(cbar, 3);
          else umma_commit(cbar);
          stage += 2;
          if (stage == STAGES) { stage = 0; phase ^= 1u; }
          buf ^= last ? 1 : 0;
          ck = last ? 0 : ck + 2;
          kb = (kb + 2 >= num_kb) ? 0 : kb + 2;
        }
      } else {
        int stage = 0;
        uint32_t phase = 0;
        int buf = 0;
        uint32_t buf_phase = 0;
        bool ok = true;
        for (int t = unit; t < args.num_tiles && ok; t += units) {
          for (int c = 0; c < num_chunks && ok; ++c) {
            if (!mbar_wait(bar_cempty(buf), buf_phase ^ 1u, abort_flag)) { ok = false; break; }
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem_base + (uint32_t)(buf * kGemmMaxBN);
            const int kb_end = min(num_kb, (c + 1) * chunk_kb);
            for (int kb = c * chunk_kb; kb < kb_end; ++kb) {
              if (!mbar_wait(bar_full(stage), phase, abort_flag)) { ok = false; break; }
              tc_fence_after_sync();
              const uint64_t adesc = sdesc_kmajor_sw128(stage_a(stage));
              const uint64_t bdesc = sdesc_kmajor_sw128(stage_b(stage));
              const bool first = (kb == c * chunk_kb);
#pragma unroll
              for (int k = 0; k < kGemmBK / 16; ++k) {
                // advance 16 elements = 32 bytes along K inside the swizzle row
                if constexpr (PAIR)
                  umma_f16_pair(d_tmem, adesc + 2u * k, bdesc + 2u * k, IDESC, (first && k == 0) ? 0u : 1u);
                else
                  umma_f16(d_tmem, adesc + 2u * k, bdesc + 2u * k, IDESC, (first && k == 0) ? 0u : 1u);
              }
              // frees the stage (in both CTAs of a pair) when these MMAs finish
              if constexpr (PAIR) umma_commit_pair(bar_empty(stage), 3);
              else umma_commit(bar_empty(stage));
              if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            // chunk sums ready for the epilogue(s)
            if constexpr (PAIR) umma_commit_pair(bar_cfull(buf), (uint16_t)(3u << lead_rank));
            else umma_commit(bar_cfull(buf));
            if (++buf == 2) { buf = 0; buf_phase ^= 1u; }
          }
        }
      }
      // every MMA this thread issued has finished before TMEM is released
      if constexpr (PAIR) umma_commit_pair(bar_drain, (uint16_t)(1u << lead_rank));
      else umma_commit(bar_drain);
      mbar_wait(bar_drain, 0u, nullptr);
    }
    __syncwarp();
  }
  } else {
    if constexpr (MODE == kLoadTma) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kGemmEpiRegs) : "memory");
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;   // TMEM lane quadrant: tile rows 32q .. 32q+31
    const int h = warp >> 2;  // column half
    const int half0 = gemm_half0_cols(BN);
    const int col0 = h == 0 ? 0 : half0;
    const int ngroups = (h == 0 ? half0 : BN - half0) / 32;  // 32-column groups, 1..4
    uint8_t* stg = smem + L::OFF_STG + warp * 2 * L::STG_BYTES;
    const uint32_t stg_addr = sbase + L::OFF_STG + warp * 2 * L::STG_BYTES;
    int sbuf = 0;
    int buf = 0;
    uint32_t buf_phase = 0;
    const int M = args.M, N = args.N;
    bool ok = true;
    // The first ADD / MUL step (num_steps if none).  With a 16-byte aligned
    // operand its boxes are staged by cp.async: the warp's second staging
    // buffer holds the operand box next in line (the first box of a tile is
    // requested when the tile starts, each next one as soon as the previous
    // one has been read), its first buffer the output boxes.
    int s_first = 0;
    if constexpr (FULL) {
      while (s_first < args.num_steps && args.ep_op[s_first] != kEpAdd && args.ep_op[s_first] != kEpMul) ++s_first;
    }
    const bool op_stage = FULL && s_first < args.num_steps && args.ep_vec[s_first] != 0;
    bool has_act = false;  // an activation among the steps
    if constexpr (FULL) {
      for (int s = 0; s < args.num_steps; ++s) has_act |= args.ep_op[s] != kEpAdd && args.ep_op[s] != kEpMul;
    }
    for (int t = unit; t < args.num_tiles && ok; t += units) {
      int grp, mb, nb;
      tile_decode(t, grp, mb, nb);
      const int m0 = mb * tile_rows + (int)rank * kGemmBM, n0 = nb * BN;
      // this warp's bias values, loaded now and used after the accumulators
      // are ready, so that their memory latency hides behind the main loop:
      // lane l holds b[n0 + col0 + 32g + l] for each 32-column box g
      // (measured: loaded after the last chunk, or prefetched into L1, the
      // first box waited about 0.4 us on them)
      const __half* bg = args.b + (size_t)grp * N;
      unsigned short bias16[kGemmHalfCols / 32];
#pragma unroll
      for (int g = 0; g < kGemmHalfCols / 32; ++g) {
        const int col = n0 + col0 + g * 32 + lane;
        bias16[g] = ((!GEN || args.has_bias) && g < ngroups && col < N) ? __half_as_ushort(__ldg(bg + col))
                                                                        : (unsigned short)0;
      }
      if (op_stage) {
        ep_operand_box_async(stg_addr + L::STG_BYTES, args.ep_ptr[s_first] + (size_t)grp * M * args.ep_ld[s_first],
                             args.ep_ld[s_first], m0 + q * 32 + lane, M, n0 + col0, N, lane);
        cp_async_commit();
      }
      float acc[kGemmHalfCols];
#pragma unroll
      for (int i = 0; i < kGemmHalfCols; ++i) acc[i] = 0.0f;
      for (int c = 0; c < num_chunks; ++c) {
        // warp-uniform decision: the TMEM loads below are warp-collective
        const bool got = mbar_wait(bar_cfull(buf), buf_phase, abort_flag);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kGemmMaxBN + col0);
#pragma unroll
        for (int g = 0; g < kGemmHalfCols / 32; ++g) {
          if (g < ngroups) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + (uint32_t)(g * 32), r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; j += 2)  // IEEE FP32 adds, round to nearest
              add_f32x2(acc[g * 32 + j], acc[g * 32 + j + 1], __uint_as_float(r[j]), __uint_as_float(r[j + 1]));
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR) mbar_arrive_cluster(map_to_cta(bar_cempty(buf), lead_rank));
          else mbar_arrive(bar_cempty(buf));
        }
        if (++buf == 2) { buf = 0; buf_phase ^= 1u; }
      }
      if (!ok) break;
      // final epilogue of this tile from registers; this tile's group: its
      // output (step operands below)
      __half* yg = args.y + (size_t)grp * M * N;
      if constexpr (FULL && MODE == kLoadTma) {
        if (has_act) {
          // Epilogue steps with an activation, one box at a time in a loop
          // that is not unrolled: the box in work is always acc[0..31] (the
          // sums rotate by one box per iteration, register moves), so each
          // activation is inlined once, and no call keeps the tile's sums
          // live across it (interleaved on 8192 x 14336 x 4096: SwiGLU
          // 786 -> 758 us, GELU tanh 780 -> 742; with K = 64, where the
          // epilogue alone sets the time, SiLU 377 -> 359, SwiGLU 476 ->
          // 439).  Steps without an activation keep the unrolled loop
          // below, whose boxes overlap better (residual: 593 against 638).
          const int dt = args.dtype;
          const int row = m0 + q * 32 + lane;
#pragma unroll 1
          for (int g = 0; g < kGemmHalfCols / 32; ++g) {
            if (g < ngroups) {
              const int nc = n0 + col0 + g * 32;
              const unsigned short blu = bias16[0];
              uint32_t packed[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                uint32_t t = ep_pack(acc[2 * i], acc[2 * i + 1], dt);
                const float b0 = ep_widen(__shfl_sync(0xffffffffu, blu, 2 * i), dt);
                const float b1 = ep_widen(__shfl_sync(0xffffffffu, blu, 2 * i + 1), dt);
                if (args.has_bias) {
                  const float2 tv = ep_unpack(t, dt);
                  t = ep_pack(__fadd_rn(tv.x, b0), __fadd_rn(tv.y, b1), dt);
                }
                packed[i] = t;
              }
              uint4 opv[4];
              if (op_stage) {
                cp_async_wait_all();
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                  opv[ch] = *reinterpret_cast<const uint4*>(stg + L::STG_BYTES + lane * 64 + ((ch ^ ((lane >> 1) & 3)) << 4));
                if (g + 1 < ngroups) {
                  ep_operand_box_async(stg_addr + L::STG_BYTES, args.ep_ptr[s_first] + (size_t)grp * M * args.ep_ld[s_first],
                                       args.ep_ld[s_first], row, M, nc + 32, N, lane);
                  cp_async_commit();
                }
              }
              for (int s = 0; s < args.num_steps; ++s) {
                const int op = args.ep_op[s];
                if (op == kEpAdd || op == kEpMul) {
                  const bool staged = op_stage && s == s_first;
#pragma unroll
                  for (int ch = 0; ch < 4; ++ch) {
                    const uint4 rv = staged ? opv[ch]
                                            : ep_load8(args.ep_ptr[s] + (size_t)grp * M * args.ep_ld[s], args.ep_ld[s],
                                                       row, M, nc + 8 * ch, N, args.ep_vec[s] != 0);
                    const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                    for (int p2 = 0; p2 < 4; ++p2)
                      packed[4 * ch + p2] = dt == kEpiBf16 ? ep_h2_binop<kEpiBf16>(op, packed[4 * ch + p2], rw[p2])
                                                           : ep_h2_binop<kEpiF16>(op, packed[4 * ch + p2], rw[p2]);
                  }
                } else {
                  gemm_epi_activation16(packed, op, dt);
                }
              }
              if (args.tma_store) {
                if (lane == 0) {
                  if (op_stage) bulk_wait_group_read<0>();
                  else bulk_wait_group_read<1>();
                }
                __syncwarp();
              }
              uint8_t* rowp = stg + sbuf * L::STG_BYTES + lane * 64;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int pos = j ^ ((lane >> 1) & 3);
                *reinterpret_cast<uint4*>(rowp + pos * 16) =
                    make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
              }
              if (args.tma_store) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                  tma_store_3d(&tm_y, stg_addr + sbuf * L::STG_BYTES, nc, m0 + q * 32, grp);
                  bulk_commit_group();
                }
              } else {
                __syncwarp();
                const uint8_t* box = stg + sbuf * L::STG_BYTES;
                const int col = nc + lane;
#pragma unroll 4
                for (int rr = 0; rr < 32; ++rr) {
                  const int r = m0 + q * 32 + rr;
                  if (r < M && col < N) {
                    const int pos = (lane >> 3) ^ ((rr >> 1) & 3);
                    yg[(size_t)r * N + col] =
                        *reinterpret_cast<const __half*>(box + rr * 64 + pos * 16 + (lane & 7) * 2);
                  }
                }
                __syncwarp();
              }
              if (!op_stage) sbuf ^= 1;
            }
#pragma unroll
            for (int i = 0; i < kGemmHalfCols - 32; ++i) acc[i] = acc[i + 32];
#pragma unroll
            for (int j = 0; j < kGemmHalfCols / 32 - 1; ++j) bias16[j] = bias16[j + 1];
          }
          continue;  // next tile
        }
      }
#pragma unroll
      for (int g = 0; g < kGemmHalfCols / 32; ++g) {
        if (g < ngroups) {
          const int nc = n0 + col0 + g * 32;  // first column of this 32-column box
          // bias of the box: lane l holds b[nc + l]; broadcast by shuffles
          const unsigned short blu = bias16[g];
          const int dt = GEN ? args.dtype : (int)kEpiF16;
          if (FULL && args.out_f32 && args.tma_store) {
            // FP32 output (the sum, + b rounded once in FP32) through the
            // staging boxes: the 32-column box as two 32 x 16 FP32 boxes
            // (64 bytes a row, the same 64-byte swizzle as the 16-bit box),
            // each stored by TMA through an FP32 map that clips at M and N
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t packed[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float bj = ep_widen(__shfl_sync(0xffffffffu, blu, 16 * h + j), dt);
                const float sj = acc[g * 32 + 16 * h + j];
                packed[j] = __float_as_uint(args.has_bias ? __fadd_rn(sj, bj) : sj);
              }
              if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous store has read it
              __syncwarp();
              uint8_t* rowp = stg + sbuf * L::STG_BYTES + lane * 64;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int pos = j ^ ((lane >> 1) & 3);
                *reinterpret_cast<uint4*>(rowp + pos * 16) =
                    make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(&tm_y, stg_addr + sbuf * L::STG_BYTES, nc + 16 * h, m0 + q * 32, grp);
                bulk_commit_group();
              }
              sbuf ^= 1;
            }
            continue;
          }
          if (FULL && args.out_f32) {
            // FP32 output without TMA (y32 not 16-byte aligned or N % 4 != 0):
            // lane = row, its 32 consecutive columns stored directly
            const int row = m0 + q * 32 + lane;
            float* yr = args.y32 + ((size_t)grp * M + (row < M ? row : 0)) * N + nc;
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
              float v[4];
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                const int j = 4 * i4 + jj;
                const float bj = ep_widen(__shfl_sync(0xffffffffu, blu, j), dt);
                v[jj] = args.has_bias ? __fadd_rn(acc[g * 32 + j], bj) : acc[g * 32 + j];
              }
              if (row < M) {
                if (args.y_vec && nc + 4 * i4 + 4 <= N) {
                  *reinterpret_cast<float4*>(yr + 4 * i4) = make_float4(v[0], v[1], v[2], v[3]);
                } else {
#pragma unroll
                  for (int jj = 0; jj < 4; ++jj)
                    if (nc + 4 * i4 + jj < N) yr[4 * i4 + jj] = v[jj];
                }
              }
            }
            continue;
          }
          uint32_t packed[16];
          if constexpr (!GEN) {
            // b[nc .. nc+31] as 16 column pairs, gathered from the lanes:
            // lane 2i + 1 sends its value up 16 bits to lane 2i first, so
            // each pair needs one broadcast shuffle
            const uint32_t up = (uint32_t)__shfl_down_sync(0xffffffffu, blu, 1);
            const uint32_t pairw = (uint32_t)blu | (up << 16);
            uint32_t bw[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) bw[i] = (uint32_t)__shfl_sync(0xffffffffu, pairw, 2 * i);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              // proj = RN16(acc) for two columns, then y = RN16(proj + b)
              const __half2 p = __floats2half2_rn(acc[g * 32 + 2 * i], acc[g * 32 + 2 * i + 1]);
              const __half2 yv = __hadd2(p, *reinterpret_cast<const __half2*>(&bw[i]));
              packed[i] = *reinterpret_cast<const uint32_t*>(&yv);
            }
          } else {
            // head value t = RN_h(sum), then RN_h(t + b), then the steps
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              uint32_t t = ep_pack(acc[g * 32 + 2 * i], acc[g * 32 + 2 * i + 1], dt);
              const float b0 = ep_widen(__shfl_sync(0xffffffffu, blu, 2 * i), dt);
              const float b1 = ep_widen(__shfl_sync(0xffffffffu, blu, 2 * i + 1), dt);
              if (args.has_bias) {
                const float2 tv = ep_unpack(t, dt);
                t = ep_pack(__fadd_rn(tv.x, b0), __fadd_rn(tv.y, b1), dt);
              }
              packed[i] = t;
            }
            const int row = m0 + q * 32 + lane;
            // the staged operand of this box into registers, then the next
            // box's request: it has this whole box's steps to land
            uint4 opv[4];
            if (op_stage) {
              cp_async_wait_all();  // this lane's row of the box has landed
#pragma unroll
              for (int ch = 0; ch < 4; ++ch)
                opv[ch] = *reinterpret_cast<const uint4*>(stg + L::STG_BYTES + lane * 64 + ((ch ^ ((lane >> 1) & 3)) << 4));
              if (g + 1 < ngroups) {
                ep_operand_box_async(stg_addr + L::STG_BYTES, args.ep_ptr[s_first] + (size_t)grp * M * args.ep_ld[s_first],
                                     args.ep_ld[s_first], row, M, nc + 32, N, lane);
                cp_async_commit();
              }
            }
            for (int s = 0; s < (FULL ? args.num_steps : 0); ++s) {
              const int op = args.ep_op[s];
              if (op == kEpAdd || op == kEpMul) {
                const bool staged = op_stage && s == s_first;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                  const uint4 rv =
                      staged ? opv[ch]
                             : ep_load8(args.ep_ptr[s] + (size_t)grp * M * args.ep_ld[s], args.ep_ld[s], row, M,
                                        nc + 8 * ch, N, args.ep_vec[s] != 0);
                  const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
                  // head-dtype pair arithmetic: the correctly rounded sum
                  // or product of two head values
#pragma unroll
                  for (int p2 = 0; p2 < 4; ++p2)
                    packed[4 * ch + p2] = dt == kEpiBf16 ? ep_h2_binop<kEpiBf16>(op, packed[4 * ch + p2], rw[p2])
                                                         : ep_h2_binop<kEpiF16>(op, packed[4 * ch + p2], rw[p2]);
                }
              } else {
                // the copy-producer kernels only (the TMA kernels run
                // activations in the rotated loop above)
                uint32_t tmp[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) tmp[i] = packed[i];
                gemm_epi_activation16_call(tmp, op, dt);
#pragma unroll
                for (int i = 0; i < 16; ++i) packed[i] = tmp[i];
              }
            }
          }
          if (args.tma_store) {
            // this buffer's previous store has read it (one output buffer
            // when the other stages the operand)
            if (lane == 0) {
              if (op_stage) bulk_wait_group_read<0>();
              else bulk_wait_group_read<1>();
            }
            __syncwarp();
          }
          // row `lane` of the 32 x 32 box, 64-byte swizzle: chunk j at j ^ ((row >> 1) & 3)
          uint8_t* rowp = stg + sbuf * L::STG_BYTES + lane * 64;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int pos = j ^ ((lane >> 1) & 3);
            *reinterpret_cast<uint4*>(rowp + pos * 16) =
                make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
          }
          if (args.tma_store) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              // the widened kernels store through a 3-D map [groups][M][N]
              if constexpr (GEN) tma_store_3d(&tm_y, stg_addr + sbuf * L::STG_BYTES, nc, m0 + q * 32, grp);
              else tma_store_2d_evict_first(&tm_y, stg_addr + sbuf * L::STG_BYTES, nc, m0 + q * 32);
              bulk_commit_group();
            }
          } else {
            __syncwarp();
            const uint8_t* box = stg + sbuf * L::STG_BYTES;
            const int col = nc + lane;
#pragma unroll 4
            for (int rr = 0; rr < 32; ++rr) {
              const int row = m0 + q * 32 + rr;
              if (row < M && col < N) {
                const int pos = (lane >> 3) ^ ((rr >> 1) & 3);
                yg[(size_t)row * N + col] =
                    *reinterpret_cast<const __half*>(box + rr * 64 + pos * 16 + (lane & 7) * 2);
              }
            }
            __syncwarp();
          }
          if (!op_stage) sbuf ^= 1;
        }
      }
    }
    // the staging buffers must have been read before the CTA exits; the
    // stores' writes complete with the grid (a dependent kernel's
    // grid_dep_wait sees them).  An operand box requested at a tile's start
    // is still in flight when a wait gave up (the abort path).
    if constexpr (FULL) cp_async_wait_all();
    if (args.tma_store && lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  // a pair's CTAs stay until the even CTA's MMAs (reading both CTAs' shared
  // memory and writing both TMEMs) and every remote arrive are done
  if constexpr (PAIR) cluster_sync();
  if (warp == kGemmMmaWarp) {
    tc_fence_after_sync();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, kGemmTmemCols);
    else tmem_dealloc(tmem_base, kGemmTmemCols);
  }
}

}  // namespace poot
