// C ABI of the GB300 FP16 linear library: argument checks, the plan-time
// choice between the GEMV and GEMM kernels, TMA descriptor encoding and the
// launches.  Declared in include/poot_linear.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <map>
#include <type_traits>
#include <functional>
#include <mutex>
#include <thread>
#include <utility>
#include <vector>

#include "poot_linear.h"
#include "gemm_tcgen05.cuh"
#include "gemv.cuh"
#include "pack.cuh"
#include "shards.cuh"
#include "splitk.cuh"

namespace {

using namespace poot;

constexpr int kVersion = 100;  // 0.1.0
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;
constexpr int kMaxDevices = 64;

using Layout = GemmLayout;
// K elements per TMEM accumulation chain before the FP32 register promotion.
// Measured on GB300 (8192x14336x4096, 1.38 M sampled outputs): chunks of
// 1024 leave 4 outputs beyond 2 FP16 ulps of a sequential FP32 sum (IEEE
// reorderings leave 2, one chain over all of K leaves 28) for about 1-2%
// of run time; 512 costs 2-3% more for no further gain.
constexpr int kDefaultChunkK = 1024;
// With epilogue steps the tile's final epilogue (an activation or an operand
// per element) outlasts the two chunks of the next tile that the TMEM double
// buffer lets it overlap; 2048-element chunks give it twice the window
// (GB300: SiLU on mlp_up 818 -> 692 us, SwiGLU 1086 -> 892 us, prefill SiLU
// 145 -> 120 us).  The longer tensor-core chains stay within the FP32
// accumulation bound that the contraction's tolerance checks.
constexpr int kStepsChunkK = 2048;

constexpr int kGemvSmemBudget = 64 * 1024;  // bytes of x staged per GEMV block

thread_local cudaError_t t_last_cuda_error = cudaSuccess;

struct DeviceState {
  bool ready = false;
  int status = POOT_OK;  // POOT_OK or POOT_ERR_UNSUPPORTED_DEVICE / CUDA
  int dev = 0;
  int sm_count = 0;
};

std::mutex g_mu;
DeviceState g_devices[kMaxDevices];
using EncodeTiledFn = decltype(&cuTensorMapEncodeTiled);
EncodeTiledFn g_encode_tiled = nullptr;

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = e;
  return POOT_ERR_CUDA;
}

template <int MODE, int CL, int EPI = kEpiPlain>
cudaError_t set_gemm_attrs() {
  if (MODE == kLoadTma) {
    // the TMA kernels rebalance registers between warpgroups (setmaxnreg):
    // the increase would wait forever unless the CTA is launched with the
    // registers the split adds up to
    cudaFuncAttributes fa;
    const cudaError_t e = cudaFuncGetAttributes(&fa, gemm_f16_tcgen05_kernel<MODE, CL, EPI>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kGemmLaunchRegs) return cudaErrorInvalidKernelImage;
  }
  return cudaFuncSetAttribute(gemm_f16_tcgen05_kernel<MODE, CL, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Layout::DYN_BYTES);
}

template <int MT, bool VEC>
cudaError_t set_gemv_attrs() {
  return cudaFuncSetAttribute(gemv_f16_kernel<MT, VEC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kGemvSmemBudget);
}

// One-time, per-device set-up: architecture check, SM count, kernel
// attributes, the driver's tensor-map encoder.
int device_state(int* dev_out, DeviceState** st_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return POOT_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_devices[dev];
  if (!st.ready) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e);
    if (major != 10 || minor != 3) {
      st.ready = true;
      st.status = POOT_ERR_UNSUPPORTED_DEVICE;
    } else {
      if (g_encode_tiled == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return cuda_fail(e);
        if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cuda_fail(cudaErrorNotSupported);
        g_encode_tiled = reinterpret_cast<EncodeTiledFn>(fn);
      }
      if ((e = set_gemm_attrs<kLoadTma, 1>()) != cudaSuccess || (e = set_gemm_attrs<kLoadTma, 2>()) != cudaSuccess ||
          (e = set_gemm_attrs<kLoadCpAsync4, 1>()) != cudaSuccess ||
          (e = set_gemm_attrs<kLoadReg16, 1>()) != cudaSuccess ||
          (e = set_gemm_attrs<kLoadTma, 1, kEpiHead>()) != cudaSuccess ||
          (e = set_gemm_attrs<kLoadTma, 2, kEpiHead>()) != cudaSuccess ||
          (e = set_gemm_attrs<kLoadCpAsync4, 1, kEpiHead>()) != cudaSuccess ||
          (e = set_gemm_attrs<kLoadReg16, 1, kEpiHead>()) != cudaSuccess ||
          (e = set_gemm_attrs<kLoadTma, 1, kEpiFull>()) != cudaSuccess ||
          (e = set_gemm_attrs<kLoadTma, 2, kEpiFull>()) != cudaSuccess ||
          (e = set_gemm_attrs<kLoadCpAsync4, 1, kEpiFull>()) != cudaSuccess ||
          (e = set_gemm_attrs<kLoadReg16, 1, kEpiFull>()) != cudaSuccess ||
          (e = set_gemv_attrs<1, true>()) != cudaSuccess || (e = set_gemv_attrs<2, true>()) != cudaSuccess ||
          (e = set_gemv_attrs<4, true>()) != cudaSuccess || (e = set_gemv_attrs<8, true>()) != cudaSuccess ||
          (e = set_gemv_attrs<16, true>()) != cudaSuccess ||
          (e = set_gemv_attrs<1, false>()) != cudaSuccess ||
          (e = set_gemv_attrs<2, false>()) != cudaSuccess ||
          (e = set_gemv_attrs<4, false>()) != cudaSuccess ||
          (e = set_gemv_attrs<8, false>()) != cudaSuccess ||
          (e = set_gemv_attrs<16, false>()) != cudaSuccess)
        return cuda_fail(e);
      st.dev = dev;
      st.sm_count = sms;
      st.status = POOT_OK;
      st.ready = true;
    }
  }
  *dev_out = dev;
  *st_out = &st;
  return st.status;
}

// Launch with programmatic stream serialisation (see grid_dep_wait in
// ptx.cuh): the kernel may be scheduled while the previous kernel in the
// stream drains; it waits for that kernel before touching global memory.
// cluster_x > 1 launches clusters of that many CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_clustered(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  std::memset(attr, 0, sizeof(attr));
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 1;
  if (cluster_x > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  cfg.attrs = attr;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                   Args&&... args) {
  return launch_clustered(kernel, grid, block, smem, stream, 1u, std::forward<Args>(args)...);
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline bool overlaps(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
  if (a == nullptr || b == nullptr || abytes <= 0 || bbytes <= 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(bbytes) && b0 < a0 + static_cast<uintptr_t>(abytes);
}

// Argument checks shared by every entry point (no CUDA calls).
int validate(const void* x, const void* w, const void* b, const void* y, int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return POOT_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return POOT_OK;
  if (y == nullptr || b == nullptr) return POOT_ERR_INVALID_ARG;
  if (K > 0 && (x == nullptr || w == nullptr)) return POOT_ERR_INVALID_ARG;
  if (!aligned(y, 2) || !aligned(b, 2)) return POOT_ERR_MISALIGNED;
  if (K > 0 && (!aligned(x, 2) || !aligned(w, 2))) return POOT_ERR_MISALIGNED;
  const int64_t ybytes = M * N * 2;
  if (overlaps(y, ybytes, b, N * 2)) return POOT_ERR_INVALID_ARG;
  if (K > 0 && (overlaps(y, ybytes, x, M * K * 2) || overlaps(y, ybytes, w, N * K * 2)))
    return POOT_ERR_INVALID_ARG;
  return POOT_OK;
}

bool xw_tma_ok(const void* x, const void* w, int64_t K) {
  return K % 8 == 0 && aligned(x, 16) && aligned(w, 16);
}

int choose_variant(const void* x, const void* w, int64_t M, int64_t N, int64_t K) {
  if (M == 0 || N == 0) return POOT_VARIANT_NONE;
  if (K == 0) return POOT_VARIANT_BIAS_ONLY;
  const bool tma = xw_tma_ok(x, w, K);
  if (M <= POOT_GEMV_MAX_M) return tma ? POOT_VARIANT_GEMV : POOT_VARIANT_GEMV_SCALAR;
  if (tma) return POOT_VARIANT_GEMM_TMA;
  return POOT_VARIANT_GEMM_PACKED;
}

// Whether a forced variant's preconditions hold.
bool variant_applicable(int v, const void* x, const void* w, int64_t M, int64_t N, int64_t K) {
  const bool empty = (M == 0 || N == 0);
  switch (v) {
    case POOT_VARIANT_NONE: return empty;
    case POOT_VARIANT_BIAS_ONLY: return !empty && K == 0;
    case POOT_VARIANT_GEMV: return !empty && K > 0 && M <= POOT_GEMV_MAX_M && xw_tma_ok(x, w, K);
    case POOT_VARIANT_GEMV_SCALAR: return !empty && K > 0 && M <= POOT_GEMV_MAX_M;
    case POOT_VARIANT_GEMM_TMA: return !empty && K > 0 && xw_tma_ok(x, w, K);
    case POOT_VARIANT_GEMM_CPASYNC: return !empty && K > 0 && K % 2 == 0 && aligned(x, 4) && aligned(w, 4);
    case POOT_VARIANT_GEMM_REG: return !empty && K > 0;
    case POOT_VARIANT_GEMM_PACKED: return !empty && K > 0;
    default: return false;
  }
}

// [slabs][outer][inner] tensor of FP32, box [1][box_outer][box_inner].
bool encode_3d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t slabs,
                   uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  const cuuint64_t dims[3] = {inner, outer, slabs};
  const cuuint64_t strides[2] = {inner * 4, inner * outer * 4};
  const cuuint32_t box[3] = {box_inner, box_outer, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Row-major [outer, inner] tensor of 2-byte elements (binary16, or bfloat16
// when bf16), rows `pitch` elements apart (default inner), box [box_outer,
// box_inner].
bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
               uint32_t box_outer, CUtensorMapSwizzle swizzle, bool bf16 = false, uint64_t pitch = 0) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {(pitch != 0 ? pitch : inner) * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode_tiled(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                                    2, const_cast<void*>(base), dims,
                                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [slabs][outer][inner] tensor of 2-byte elements, box [1][box_outer][box_inner]
// (each box stays inside one slab: stores clip at `outer` per slab).
bool encode_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t slabs,
               uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle, bool bf16) {
  const cuuint64_t dims[3] = {inner, outer, slabs};
  const cuuint64_t strides[2] = {inner * 2, inner * outer * 2};
  const cuuint32_t box[3] = {box_inner, box_outer, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode_tiled(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                                    3, const_cast<void*>(base), dims, strides, box, estr,
                                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct GemmPlan {
  int bn, stages, group_m, chunk_kb;
  int cluster;  // 1: single CTAs; 2: CTA pairs (2-SM MMA)
  bool pair;    // cluster == 2 (256-row tiles)
  int split;    // K ranges (split-K); 1 = none
};

// Tile plan from a cost model: each CTA runs ceil(tiles / SMs) tiles; a
// tile costs num_kb K blocks of max(MMA cycles, shared-memory operand
// cycles) / efficiency plus a fixed pipeline fill / drain.  MMA 128 x bn x 64
// takes 2 * bn cycles; its operands (16 KB + 128 * bn bytes) stream at about
// 128 B/cycle.  The efficiencies of narrower tiles (more x re-reads, more
// epilogue work per FLOP) were measured on GB300 for 224 (0.90 - 0.97) and
// extrapolated below it.  Ties go to the wider tile.
GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int sms, int bn_req, int group_req,
                   int chunk_req, int cluster_req, int split_req, bool allow_split, bool tma) {
  // CTA pairs (2-SM MMA) from M = 256 (one full pair tile); single CTAs
  // when M is smaller, for short K in one wave, or when the operands need
  // copies.
  int cluster = 1;
  bool short_k_wave = false;
  if (tma) {
    // short K in one wave of 128 x 64 single-CTA tiles: the pair's two
    // cluster barriers (about 0.5 us each) outweigh its gain (1024 x 1024 x
    // 768 on GB300: 6.5 us single, 8.0 us in pairs)
    const int64_t single64 = ((M + kGemmBM - 1) / kGemmBM) * ((N + 63) / 64);
    short_k_wave = (K + kGemmBK - 1) / kGemmBK <= 16 && single64 <= sms;
    // below 512 rows, 256-row pair tiles only where they pad M no more than
    // 128-row tiles do (384 x 4096 x 4096: 19.9 us single, 20.9 us in
    // pairs; 640 x 4096 x 4096: 29.0 us single, 24.2 us in pairs)
    const bool pair_rows = (M + 255) / 256 * 2 == (M + 127) / 128 || M >= 512;
    if (cluster_req != 0) cluster = cluster_req;
    else if (M >= 256 && N >= 256 && pair_rows && !short_k_wave) cluster = 2;
  }
  const bool pair = cluster >= 2;
  const int64_t bm = pair ? 2 * kGemmBM : kGemmBM;
  const int64_t slots = pair ? sms / 2 : sms;
  const int64_t num_m = (M + bm - 1) / bm;
  const int64_t num_kb = (K + kGemmBK - 1) / kGemmBK;
  int best_bn = 256;
  int64_t best = INT64_MAX;
  static const int cands[] = {256, 224, 192, 160, 128, 96, 64};
  static const int eff_pct[] = {100, 93, 88, 83, 78, 70, 60};
  for (int i = 0; i < 7; ++i) {
    const int bn = cands[i];
    if (bn_req != 0 && bn != bn_req) continue;
    const int64_t tiles = num_m * ((N + bn - 1) / bn);
    const int64_t waves = (tiles + slots - 1) / slots;
    const int64_t per_kb = (2 * bn > 128 + bn) ? 2 * bn : 128 + bn;
    const int64_t cost = waves * (num_kb * per_kb * 100 / eff_pct[i] + 2000);
    if (cost < best) { best = cost; best_bn = bn; }
  }
  if (bn_req != 0) best_bn = bn_req;
  else if (cluster == 1 && short_k_wave) best_bn = 64;  // most CTAs loading at once
  // Split-K, planned jointly with the tile width, when one wave of tiles
  // leaves more than a quarter of the CTA slots idle and K is long (or when
  // a split is requested without a tile width).  Here a tile's cost is
  // fitted to interleaved GB300 timings of every (width, split) filling at
  // most one wave on M = 64 .. 256, N x K = 1024 x 16384 .. 14336 x 4096 (the
  // chosen plan within 4% of the best measured on each): narrow tiles lose
  // less than above (their many CTAs stream W in parallel), and a split
  // costs about 4 us (the second kernel, the workspace's write and read)
  // plus its bytes.
  int split = split_req > 1 ? split_req : 1;
  {
    const int64_t tiles1 = num_m * ((N + best_bn - 1) / best_bn);
    const bool underfilled = tiles1 <= slots && tiles1 * 4 < slots * 3;
    const bool plan_joint = allow_split && cluster <= 2 &&
                            ((split_req == 0 && num_kb >= 16 && underfilled) || (split_req > 1 && bn_req == 0));
    if (plan_joint) {
      static const int eff_split[] = {100, 93, 88, 83, 86, 78, 70};
      static const int splits[] = {1, 2, 4, 8, 16};
      int64_t best_cost = INT64_MAX;
      int jbn = best_bn, jsplit = split;
      for (int i = 0; i < 7; ++i) {
        const int bn = cands[i];
        if (bn_req != 0 && bn != bn_req) continue;
        const int64_t tiles = num_m * ((N + bn - 1) / bn);
        for (int j = 0; j < 5; ++j) {
          const int S = splits[j];
          if (split_req > 1 && S != split_req) continue;
          if (split_req == 0 && S > 1 && (num_kb % S != 0 || num_kb / S < 8 || tiles * S > slots)) continue;
          const int64_t waves = (tiles * S + slots - 1) / slots;
          const int64_t per_kb = (2 * bn > 128 + bn) ? 2 * bn : 128 + bn;
          int64_t cost = waves * ((num_kb / S) * per_kb * 100 / eff_split[i] + 1000);
          if (S > 1) cost += 8000 + int64_t(S) * M * N * 4 / 1024;
          if (cost < best_cost) { best_cost = cost; jbn = bn; jsplit = S; }
        }
      }
      best_bn = jbn;
      split = jsplit;
    }
  }
  GemmPlan p;
  p.split = split;
  p.cluster = cluster;
  p.pair = pair;
  p.bn = best_bn;
  p.stages = gemm_max_stages(best_bn, pair);
  // Tiles are walked in groups of M blocks whose x rows (group x K x 2
  // bytes) stay within 32 MB of L2 while W streams past them: W is then
  // read from HBM once per group instead of once per 1024 rows.  Under the
  // power cap the saved HBM traffic buys SM clock: on 8192x14336x4096 with
  // CTA pairs, groups of 4096 rows ran 5% faster than 1024 rows (1365 vs
  // 1310 MHz) and 8192 rows 2% slower.
  int group_def = 1;
  {
    const int64_t rows_budget = (int64_t(32) << 20) / (2 * (K > 0 ? K : 1));
    while (int64_t(group_def) * 2 * bm <= rows_budget && group_def < 64) group_def *= 2;
  }
  p.group_m = group_req > 0 ? group_req : group_def;
  // K elements summed in TMEM before the FP32 register promotion
  const int chunk_k = chunk_req > 0 ? chunk_req : kDefaultChunkK;
  p.chunk_kb = chunk_k / kGemmBK;
  return p;
}

// ---- split-K workspace ------------------------------------------------------
struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::mutex g_ws_mu;
// key: (device, stream, thread): the thread is part of the key only for
// cudaStreamPerThread, one handle that names a different stream in each thread
struct WorkspaceKey {
  int dev;
  cudaStream_t stream;
  std::thread::id thread;
  bool operator<(const WorkspaceKey& o) const {
    if (dev != o.dev) return dev < o.dev;
    if (stream != o.stream) return std::less<cudaStream_t>()(stream, o.stream);
    return thread < o.thread;
  }
};
std::map<WorkspaceKey, Workspace> g_ws;
std::vector<void*> g_ws_retired;

struct WorkspaceRelease {
  ~WorkspaceRelease() {
    for (auto& kv : g_ws)
      if (kv.second.ptr != nullptr) cudaFree(kv.second.ptr);
    for (void* p : g_ws_retired) cudaFree(p);
  }
} g_ws_release;

// Workspace of a call (split-K partial sums, packed operands).  Outside
// stream capture: one buffer per (device, stream; thread for
// cudaStreamPerThread), grown by doubling and kept for the life of the process
// (calls on one stream are ordered, so they can share it; a buffer outgrown
// is kept too, as work queued earlier may still read it).  Under capture:
// a graph-owned allocation (cudaMallocAsync / cudaFreeAsync on the capturing
// stream become memory nodes of the graph), so that a graph never shares a
// buffer with calls made outside it.  nullptr: no workspace, no split.
struct WorkspaceLease {
  void* ptr = nullptr;
  bool graph_owned = false;
  cudaStream_t stream = nullptr;
  // a graph-owned workspace is freed on its stream after the last kernel
  // that reads it (or on any early return before those launches)
  cudaError_t release() {
    cudaError_t e = cudaSuccess;
    if (graph_owned) e = cudaFreeAsync(ptr, stream);
    graph_owned = false;
    return e;
  }
  WorkspaceLease() = default;
  WorkspaceLease(const WorkspaceLease&) = delete;
  WorkspaceLease& operator=(const WorkspaceLease&) = delete;
  WorkspaceLease(WorkspaceLease&& o) noexcept : ptr(o.ptr), graph_owned(o.graph_owned), stream(o.stream) {
    o.graph_owned = false;
  }
  WorkspaceLease& operator=(WorkspaceLease&& o) noexcept {
    if (this != &o) {
      (void)release();
      ptr = o.ptr;
      graph_owned = o.graph_owned;
      stream = o.stream;
      o.graph_owned = false;
    }
    return *this;
  }
  ~WorkspaceLease() { (void)release(); }
};

WorkspaceLease stream_workspace(int dev, cudaStream_t stream, size_t bytes) {
  WorkspaceLease lease;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    (void)cudaGetLastError();
    return lease;
  }
  if (cs != cudaStreamCaptureStatusNone) {
    if (cs != cudaStreamCaptureStatusActive || cudaMallocAsync(&lease.ptr, bytes, stream) != cudaSuccess) {
      (void)cudaGetLastError();
      lease.ptr = nullptr;
      return lease;
    }
    lease.graph_owned = true;
    lease.stream = stream;
    return lease;
  }
  std::lock_guard<std::mutex> lock(g_ws_mu);
  const std::thread::id tid = stream == cudaStreamPerThread ? std::this_thread::get_id() : std::thread::id();
  Workspace& ws = g_ws[WorkspaceKey{dev, stream, tid}];
  if (ws.bytes >= bytes) {
    lease.ptr = ws.ptr;
    return lease;
  }
  size_t want = bytes > 2 * ws.bytes ? bytes : 2 * ws.bytes;
  want = (want + (size_t(1) << 20) - 1) & ~((size_t(1) << 20) - 1);
  void* p = nullptr;
  if (cudaMalloc(&p, want) != cudaSuccess) {
    (void)cudaGetLastError();  // no split-K then; not an error of the call
    return lease;
  }
  if (ws.ptr != nullptr) g_ws_retired.push_back(ws.ptr);
  ws.ptr = p;
  ws.bytes = want;
  lease.ptr = p;
  return lease;
}

constexpr int kMaxSplitK = 16;

// The widened contraction's epilogue, as checked by poot_contract.
struct EpiConfig {
  int dtype, out_f32, num_steps;
  int op[kEpiMaxSteps];
  const void* ptr[kEpiMaxSteps];
  int64_t ld[kEpiMaxSteps];
};

int launch_gemm(int variant, const DeviceState& st, const void* x, const void* w, const void* b, void* y,
                int64_t M, int64_t N, int64_t K, int bn_req, int group_req, int chunk_req, int cluster_req,
                int split_req, cudaStream_t stream, const EpiConfig* epi = nullptr, int64_t G = 1,
                float* fixed_ws = nullptr, size_t fixed_ws_bytes = 0) {
  // GEMM_PACKED: x and W are first copied into 16-byte-pitched rows in the
  // workspace, then the TMA kernels run on the copies
  const bool packed = variant == POOT_VARIANT_GEMM_PACKED;
  if (packed && fixed_ws != nullptr) return POOT_ERR_INVALID_ARG;
  if (packed) variant = POOT_VARIANT_GEMM_TMA;
  const GemmPlan plan = plan_gemm(M, N, K, st.sm_count, bn_req, group_req, chunk_req,
                                  cluster_req, split_req, G == 1, variant == POOT_VARIANT_GEMM_TMA);
  const int bm = plan.pair ? 2 * kGemmBM : kGemmBM;
  GemmArgs a;
  a.x = static_cast<const __half*>(x);
  a.w = static_cast<const __half*>(w);
  a.b = static_cast<const __half*>(b);
  a.y = static_cast<__half*>(y);
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.bn = plan.bn;
  a.stages = plan.stages;
  a.group_m = plan.group_m;
  a.chunk_kb = plan.chunk_kb;
  a.num_m_blocks = static_cast<int>((M + bm - 1) / bm);
  // a group never spans more than all M blocks (keeps group_m * num_n_blocks
  // within the tile count, hence within int)
  if (a.group_m > a.num_m_blocks) a.group_m = a.num_m_blocks;
  a.num_n_blocks = static_cast<int>((N + plan.bn - 1) / plan.bn);
  const int64_t num_kb_all = (K + kGemmBK - 1) / kGemmBK;
  const int64_t tiles_per_group = int64_t(a.num_m_blocks) * a.num_n_blocks;
  // a requested split must divide the K blocks (and is not for groups); the
  // partial sums need a workspace
  if (split_req > 1 && (G != 1 || num_kb_all % split_req != 0)) return POOT_ERR_INVALID_ARG;
  int S = plan.split;
  WorkspaceLease lease;
  // workspace: [packed x | packed W | split-K partial sums], 256-byte aligned parts
  const int64_t Kp = (K + 7) / 8 * 8;
  auto round256 = [](size_t v) { return (v + 255) & ~size_t(255); };
  const size_t pack_x = packed ? round256(size_t(G) * M * Kp * 2) : 0;
  const size_t pack_w = packed ? round256(size_t(G) * N * Kp * 2) : 0;
  if (S > 1 && fixed_ws != nullptr) {
    // a caller-provided workspace (the no-allocation entry point)
    if (size_t(S) * M * N * sizeof(float) > fixed_ws_bytes) return POOT_ERR_INVALID_ARG;
  } else if (S > 1 || packed) {
    const size_t split_bytes = S > 1 ? size_t(S) * M * N * sizeof(float) : 0;
    lease = stream_workspace(st.dev, stream, pack_x + pack_w + split_bytes);
    if (lease.ptr == nullptr && packed) {
      // no room for the copies: the copy producers read x and W in place
      // (they cannot feed CTA pairs)
      if (cluster_req >= 2) return cuda_fail(cudaErrorMemoryAllocation);
      const int fallback = (K % 2 == 0 && aligned(x, 4) && aligned(w, 4)) ? POOT_VARIANT_GEMM_CPASYNC
                                                                          : POOT_VARIANT_GEMM_REG;
      return launch_gemm(fallback, st, x, w, b, y, M, N, K, bn_req, group_req, chunk_req, cluster_req, split_req,
                         stream, epi, G);
    }
    if (lease.ptr == nullptr) {
      if (split_req > 1) return cuda_fail(cudaErrorMemoryAllocation);
      S = 1;
    }
  }
  char* const ws_base = static_cast<char*>(lease.ptr);
  uint16_t* const xp = packed ? reinterpret_cast<uint16_t*>(ws_base) : nullptr;
  uint16_t* const wp = packed ? reinterpret_cast<uint16_t*>(ws_base + pack_x) : nullptr;
  float* const ws = fixed_ws != nullptr ? fixed_ws
                    : (S > 1 ? reinterpret_cast<float*>(ws_base + pack_x + pack_w) : nullptr);
  if (packed) {
    a.x = reinterpret_cast<const __half*>(xp);
    a.w = reinterpret_cast<const __half*>(wp);
  }
  a.num_k_blocks = static_cast<int>(num_kb_all / S);
  const int64_t tiles = tiles_per_group * (S > 1 ? S : G);
  if (tiles > INT32_MAX) return POOT_ERR_INVALID_ARG;
  a.num_tiles = static_cast<int>(tiles);
  a.groups = static_cast<int>(S > 1 ? S : G);
  a.tiles_per_group = static_cast<int>(tiles_per_group);
  a.split_k = S;
  a.tma_store = (N % 8 == 0 && aligned(y, 16)) ? 1 : 0;
  a.general = epi != nullptr ? 1 : 0;
  a.dtype = epi != nullptr ? epi->dtype : POOT_DTYPE_F16;
  a.out_f32 = (epi != nullptr && epi->out_f32) ? 1 : 0;
  a.has_bias = (epi == nullptr || b != nullptr) ? 1 : 0;
  a.y_vec = (N % 4 == 0 && aligned(y, 16)) ? 1 : 0;
  a.y32 = a.out_f32 ? static_cast<float*>(y) : nullptr;
  // FP32 output: TMA stores of 32 x 16 boxes need 16-byte rows
  if (a.out_f32) a.tma_store = (N % 4 == 0 && aligned(y, 16)) ? 1 : 0;
  a.num_steps = epi != nullptr ? epi->num_steps : 0;
  for (int s = 0; s < kEpiMaxSteps; ++s) {
    const bool used = s < a.num_steps;
    a.ep_op[s] = used ? epi->op[s] : 0;
    a.ep_ptr[s] = used ? static_cast<const uint16_t*>(epi->ptr[s]) : nullptr;
    a.ep_ld[s] = used ? epi->ld[s] : 0;
    a.ep_vec[s] = (used && a.ep_ptr[s] != nullptr && aligned(a.ep_ptr[s], 16) && a.ep_ld[s] % 8 == 0) ? 1 : 0;
  }
  // the reduce kernel applies the real epilogue after a split-K GEMM
  SplitReduceArgs ra;
  std::memset(&ra, 0, sizeof(ra));
  if (S > 1) {
    ra.ws = ws;
    ra.S = S;
    ra.M = a.M;
    ra.N = a.N;
    ra.e.dtype = a.dtype;
    ra.e.out_f32 = a.out_f32;
    ra.e.has_bias = a.has_bias;
    ra.e.num_steps = a.num_steps;
    for (int s = 0; s < kEpiMaxSteps; ++s) {
      ra.e.op[s] = a.ep_op[s];
      ra.e.ptr[s] = a.ep_ptr[s];
      ra.e.ld[s] = a.ep_ld[s];
    }
    ra.e.b = reinterpret_cast<const uint16_t*>(b);
    ra.e.y = a.out_f32 ? nullptr : static_cast<uint16_t*>(y);
    ra.e.y32 = a.out_f32 ? static_cast<float*>(y) : nullptr;
    ra.e.ldy = N;
    // the GEMM writes the unrounded partial sums of each split
    a.general = 1;
    a.out_f32 = 1;
    a.has_bias = 0;
    a.num_steps = 0;
    a.y32 = ws;
    a.y_vec = (N % 4 == 0) ? 1 : 0;
    a.tma_store = (N % 4 == 0) ? 1 : 0;  // the workspace is 256-byte aligned
  }
  const bool bf16 = a.dtype == POOT_DTYPE_BF16;
  // Paired stages (see GemmArgs::paired) need an even ring and every chunk
  // (the tile's last one included) an even number of at least `stages` K
  // blocks: the fill that reuses a chunk's last pair then lies in the next
  // chunk, and no chunk-complete barrier is two phases ahead of the producer.
  {
    const int nkb = a.num_k_blocks, ckb = plan.chunk_kb, tail = nkb % ckb;
    const int shortest = nkb <= ckb ? nkb : (tail == 0 ? ckb : tail);
    const int even_stages = plan.stages & ~1;
    a.paired = (variant == POOT_VARIANT_GEMM_TMA && ckb % 2 == 0 && nkb % 2 == 0 &&
                even_stages >= 4 && shortest >= even_stages)
                   ? 1
                   : 0;
    if (a.paired) a.stages = even_stages;
  }

  CUtensorMap tx, tw, ty;
  std::memset(&tx, 0, sizeof(tx));
  std::memset(&tw, 0, sizeof(tw));
  std::memset(&ty, 0, sizeof(ty));
  if (variant == POOT_VARIANT_GEMM_TMA) {
    // x and W of all groups as one flattened [G*M, K] and [G*N, K] tensor
    // (the packed copies: rows Kp elements apart, inner extent still K)
    const void* xs = packed ? static_cast<const void*>(xp) : x;
    const void* wsrc = packed ? static_cast<const void*>(wp) : w;
    const uint64_t pitch = packed ? static_cast<uint64_t>(Kp) : 0;
    if (!encode_2d(&tx, xs, K, G * M, kGemmBK, kGemmBM, CU_TENSOR_MAP_SWIZZLE_128B, bf16, pitch) ||
        !encode_2d(&tw, wsrc, K, G * N, kGemmBK, static_cast<uint32_t>(gemm_b_rows(plan.bn, plan.pair)),
                   CU_TENSOR_MAP_SWIZZLE_128B, bf16, pitch))
      return cuda_fail(cudaErrorInvalidValue);
  }
  if (a.tma_store) {
    // the widened kernels store through [G][M][N] so that boxes clip at each
    // group's M (FP32 output, split-K partial sums included: [groups][M][N]
    // FP32 with 32 x 16 boxes); the plain kernels through [M][N]
    bool ok;
    if (a.out_f32)
      ok = encode_3d_f32(&ty, a.y32, N, M, a.groups, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    else if (epi != nullptr)
      ok = encode_3d(&ty, y, N, M, G, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B, bf16);
    else
      ok = encode_2d(&ty, y, N, M, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B, bf16);
    if (!ok) return cuda_fail(cudaErrorInvalidValue);
  }

  cudaError_t e;
  if (packed) {
    PackArgs pa;
    pa.src[0] = static_cast<const uint16_t*>(x);
    pa.src[1] = static_cast<const uint16_t*>(w);
    pa.dst[0] = xp;
    pa.dst[1] = wp;
    pa.rows[0] = G * M;
    pa.rows[1] = G * N;
    pa.K = static_cast<int>(K);
    pa.Kp = static_cast<int>(Kp);
    const int64_t chunks = (G * M + G * N) * (Kp / 8);
    int64_t blocks = (chunks + 255) / 256;
    const int64_t cap = int64_t(st.sm_count) * 8;
    if (blocks > cap) blocks = cap;
    e = launch(pack_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, pa);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (epi != nullptr || S > 1) {
    // the widened epilogue (and the split-K partial sums) are compiled into
    // their own instantiations (CTA pairs or single CTAs)
    // head dtype and bias only: the lighter instantiation; FP32 output,
    // steps or split-K partial sums: the full one
    const bool full = S > 1 || a.out_f32 || a.num_steps > 0;
    auto launch_widened = [&](auto epi_tag) -> cudaError_t {
      constexpr int E = decltype(epi_tag)::value;
      if (plan.cluster == 2) {
        const int64_t pairs = st.sm_count / 2;
        const int grid = 2 * static_cast<int>(tiles < pairs ? tiles : pairs);
        return launch_clustered(gemm_f16_tcgen05_kernel<kLoadTma, 2, E>, dim3(grid), dim3(gemm_threads(kLoadTma)),
                                Layout::DYN_BYTES, stream, 2u, tx, tw, ty, a);
      }
      const int grid = static_cast<int>(tiles < st.sm_count ? tiles : st.sm_count);
      switch (variant) {
        case POOT_VARIANT_GEMM_TMA:
          return launch(gemm_f16_tcgen05_kernel<kLoadTma, 1, E>, dim3(grid), dim3(gemm_threads(kLoadTma)),
                        Layout::DYN_BYTES, stream, tx, tw, ty, a);
        case POOT_VARIANT_GEMM_CPASYNC:
          return launch(gemm_f16_tcgen05_kernel<kLoadCpAsync4, 1, E>, dim3(grid), dim3(gemm_threads(kLoadCpAsync4)),
                        Layout::DYN_BYTES, stream, tx, tw, ty, a);
        default:
          return launch(gemm_f16_tcgen05_kernel<kLoadReg16, 1, E>, dim3(grid), dim3(gemm_threads(kLoadReg16)),
                        Layout::DYN_BYTES, stream, tx, tw, ty, a);
      }
    };
    e = full ? launch_widened(std::integral_constant<int, kEpiFull>{})
             : launch_widened(std::integral_constant<int, kEpiHead>{});
    if (e == cudaSuccess && S > 1) {
      const bool vec = N % 4 == 0 && (ra.e.out_f32 ? aligned(y, 16) : aligned(y, 8));
      const int64_t units = vec ? M * N / 4 : M * N;
      int64_t blocks = (units + 255) / 256;
      const int64_t cap = int64_t(st.sm_count) * 8;
      if (blocks > cap) blocks = cap;
      e = vec ? launch(splitk_reduce_kernel<4>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, ra)
              : launch(splitk_reduce_kernel<1>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, ra);
    }
    const cudaError_t f = lease.release();
    if (e == cudaSuccess) e = f;
    return e == cudaSuccess ? POOT_OK : cuda_fail(e);
  }
  if (plan.cluster == 2) {
    const int64_t pairs = st.sm_count / 2;
    const int grid = 2 * static_cast<int>(tiles < pairs ? tiles : pairs);
    e = launch_clustered(gemm_f16_tcgen05_kernel<kLoadTma, 2>, dim3(grid), dim3(gemm_threads(kLoadTma)),
                         Layout::DYN_BYTES, stream, 2u, tx, tw, ty, a);
    return e == cudaSuccess ? POOT_OK : cuda_fail(e);
  }
  const int grid = static_cast<int>(tiles < st.sm_count ? tiles : st.sm_count);
  switch (variant) {
    case POOT_VARIANT_GEMM_TMA:
      e = launch(gemm_f16_tcgen05_kernel<kLoadTma, 1>, dim3(grid), dim3(gemm_threads(kLoadTma)),
                 Layout::DYN_BYTES, stream, tx, tw, ty, a);
      break;
    case POOT_VARIANT_GEMM_CPASYNC:
      e = launch(gemm_f16_tcgen05_kernel<kLoadCpAsync4, 1>, dim3(grid), dim3(gemm_threads(kLoadCpAsync4)),
                 Layout::DYN_BYTES, stream, tx, tw, ty, a);
      break;
    default:
      e = launch(gemm_f16_tcgen05_kernel<kLoadReg16, 1>, dim3(grid), dim3(gemm_threads(kLoadReg16)),
                 Layout::DYN_BYTES, stream, tx, tw, ty, a);
      break;
  }
  return e == cudaSuccess ? POOT_OK : cuda_fail(e);
}

template <bool VEC>
cudaError_t launch_gemv_mt(int mt, dim3 grid, size_t smem, cudaStream_t stream, const GemvArgs& a) {
  const dim3 block(kGemvThreads);
  switch (mt) {
    case 1: return launch(gemv_f16_kernel<1, VEC>, grid, block, smem, stream, a);
    case 2: return launch(gemv_f16_kernel<2, VEC>, grid, block, smem, stream, a);
    case 4: return launch(gemv_f16_kernel<4, VEC>, grid, block, smem, stream, a);
    case 8: return launch(gemv_f16_kernel<8, VEC>, grid, block, smem, stream, a);
    default: return launch(gemv_f16_kernel<16, VEC>, grid, block, smem, stream, a);
  }
}

int launch_gemv(int variant, const DeviceState& st, const void* x, const void* w, const void* b, void* y,
                int64_t M, int64_t N, int64_t K, int wpr_req, cudaStream_t stream) {
  int mt = 1;
  while (mt < M) mt *= 2;
  int wpr = wpr_req;
  if (wpr == 0) {
    // enough warps in flight to cover HBM latency: about 16 per SM
    const int64_t target = int64_t(st.sm_count) * 16;
    wpr = 1;
    while (wpr < kGemvWarps && N * wpr < target) wpr *= 2;
  }
  // K chunk staged in shared memory: a multiple of 256 elements
  int64_t kc = (kGemvSmemBudget / (2 * mt)) / 256 * 256;
  const int64_t kround = (K + 255) / 256 * 256;
  if (kc > kround) kc = kround;
  GemvArgs a;
  std::memset(&a, 0, sizeof(a));
  a.x = static_cast<const __half*>(x);
  a.w = static_cast<const __half*>(w);
  a.b = static_cast<const __half*>(b);
  a.y = static_cast<__half*>(y);
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.wpr = wpr;
  a.kc = static_cast<int>(kc);
  a.groups = 1;
  a.prefetch = 0;
  const int rows_per_block = kGemvWarps / wpr;
  const int64_t blocks = (N + rows_per_block - 1) / rows_per_block;
  if (blocks > INT32_MAX) return POOT_ERR_INVALID_ARG;
  const size_t smem = static_cast<size_t>(mt) * static_cast<size_t>(kc) * 2;
  cudaError_t e;
  if (variant == POOT_VARIANT_GEMV && mt <= 2 && wpr <= kGemvRowWarps) {
    const int rpb = kGemvRowWarps / wpr;
    const dim3 rgrid(static_cast<unsigned>((N + rpb - 1) / rpb));
    if (mt == 1)
      e = launch(gemv_f16_rows_kernel<1>, rgrid, dim3(kGemvRowThreads), 0, stream, a);
    else
      e = launch(gemv_f16_rows_kernel<2>, rgrid, dim3(kGemvRowThreads), 0, stream, a);
  } else if (variant == POOT_VARIANT_GEMV && wpr_req == 0) {
    // 3 <= M <= 16 on the tensor cores, 16 rows of W per block; 16 warps
    // along K below two such blocks per SM, the L2 prefetch up to two
    // blocks for every three SMs
    const int64_t tiles = (N + 15) / 16;
    const dim3 mgrid(static_cast<unsigned>(tiles));
    const bool few = gemv_mma_few_tiles(tiles, st.sm_count);
    a.prefetch = 3 * tiles <= 2 * int64_t(st.sm_count) ? 1 : 0;
    constexpr int WF = kGemvMmaWarpsFew, WM = kGemvMmaWarpsMany;
    // 9 <= M <= 16 always on eight warps: sixteen warps of the two-column-
    // block kernel need about 80 registers each, one block per SM, so 256
    // tiles took two waves (16 x 4096 x 4096 on GB300: 14.6 us against 9.2)
    if (M <= 8)
      e = few ? launch(gemv_f16_mma_kernel<1, WF>, mgrid, dim3(WF * 32), 0, stream, a)
              : launch(gemv_f16_mma_kernel<1, WM>, mgrid, dim3(WM * 32), 0, stream, a);
    else
      e = launch(gemv_f16_mma_kernel<2, WM>, mgrid, dim3(WM * 32), 0, stream, a);
  } else if (variant == POOT_VARIANT_GEMV) {
    e = launch_gemv_mt<true>(mt, dim3(static_cast<unsigned>(blocks)), smem, stream, a);
  } else {
    e = launch_gemv_mt<false>(mt, dim3(static_cast<unsigned>(blocks)), smem, stream, a);
  }
  return e == cudaSuccess ? POOT_OK : cuda_fail(e);
}

// The widened contraction for 1 <= M <= 16 (x and W 16-byte aligned,
// K % 8 == 0; G groups) on the GEMV kernels: the same W stream, the
// operands in the head dtype, each output through the per-element epilogue.
int launch_gemv_wide(const DeviceState& st, const void* x, const void* w, const void* b, void* y, int64_t M,
                     int64_t N, int64_t K, int64_t G, const EpiConfig& epi, cudaStream_t stream) {
  GemvArgs a;
  std::memset(&a, 0, sizeof(a));
  a.groups = static_cast<int>(G);
  a.x = static_cast<const __half*>(x);
  a.w = static_cast<const __half*>(w);
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.e.dtype = epi.dtype;
  a.e.out_f32 = epi.out_f32;
  a.e.has_bias = b != nullptr ? 1 : 0;
  a.e.num_steps = epi.num_steps;
  for (int s = 0; s < kEpiMaxSteps; ++s) {
    const bool used = s < epi.num_steps;
    a.e.op[s] = used ? epi.op[s] : 0;
    a.e.ptr[s] = used ? static_cast<const uint16_t*>(epi.ptr[s]) : nullptr;
    a.e.ld[s] = used ? epi.ld[s] : 0;
  }
  a.e.b = static_cast<const uint16_t*>(b);
  a.e.y = epi.out_f32 ? nullptr : static_cast<uint16_t*>(y);
  a.e.y32 = epi.out_f32 ? static_cast<float*>(y) : nullptr;
  a.e.ldy = N;
  const bool bf = epi.dtype == POOT_DTYPE_BF16;
  cudaError_t e;
  if (M <= 2) {
    // one warp per W row (or per K slice): about 16 warps per SM
    const int64_t target = int64_t(st.sm_count) * 16;
    int wpr = 1;
    while (wpr < kGemvRowWarps && G * N * wpr < target) wpr *= 2;
    a.wpr = wpr;
    const int rpb = kGemvRowWarps / wpr;
    const dim3 grid(static_cast<unsigned>((G * N + rpb - 1) / rpb)), block(kGemvRowThreads);
    if (M == 1)
      e = bf ? launch(gemv_f16_rows_kernel<1, kEpiBf16, true>, grid, block, 0, stream, a)
             : launch(gemv_f16_rows_kernel<1, kEpiF16, true>, grid, block, 0, stream, a);
    else
      e = bf ? launch(gemv_f16_rows_kernel<2, kEpiBf16, true>, grid, block, 0, stream, a)
             : launch(gemv_f16_rows_kernel<2, kEpiF16, true>, grid, block, 0, stream, a);
  } else {
    // the tensor-core GEMV, with the plain call's warp and prefetch rules
    // (16-row tiles per group)
    const int64_t tiles = G * ((N + 15) / 16);
    const dim3 grid(static_cast<unsigned>(tiles));
    const bool few = gemv_mma_few_tiles(tiles, st.sm_count);
    a.prefetch = 3 * tiles <= 2 * int64_t(st.sm_count) ? 1 : 0;
    constexpr int WF = kGemvMmaWarpsFew, WM = kGemvMmaWarpsMany;
    const dim3 block((few ? WF : WM) * 32);
    if (M <= 8) {
      if (bf)
        e = few ? launch(gemv_f16_mma_kernel<1, WF, kEpiBf16, true>, grid, block, 0, stream, a)
                : launch(gemv_f16_mma_kernel<1, WM, kEpiBf16, true>, grid, block, 0, stream, a);
      else
        e = few ? launch(gemv_f16_mma_kernel<1, WF, kEpiF16, true>, grid, block, 0, stream, a)
                : launch(gemv_f16_mma_kernel<1, WM, kEpiF16, true>, grid, block, 0, stream, a);
    } else {
      // eight warps for 9 <= M <= 16 (see launch_gemv)
      const dim3 block8(WM * 32);
      if (bf)
        e = launch(gemv_f16_mma_kernel<2, WM, kEpiBf16, true>, grid, block8, 0, stream, a);
      else
        e = launch(gemv_f16_mma_kernel<2, WM, kEpiF16, true>, grid, block8, 0, stream, a);
    }
  }
  return e == cudaSuccess ? POOT_OK : cuda_fail(e);
}

// GEMM options shared by run() and contract().
bool gemm_options_ok(const poot_linear_options& o) {
  if (o.gemm_tile_n != 0 && (o.gemm_tile_n < 64 || o.gemm_tile_n > kGemmMaxBN || o.gemm_tile_n % 32 != 0))
    return false;
  if (o.gemm_group_m < 0) return false;
  if (o.gemm_k_chunk < 0 || o.gemm_k_chunk % kGemmBK != 0) return false;
  if (o.gemm_split_k < 0 || o.gemm_split_k > kMaxSplitK) return false;
  return o.gemm_cluster == 0 || o.gemm_cluster == 1 || o.gemm_cluster == 2;
}

int run(const void* x, const void* w, const void* b, void* y, int64_t M, int64_t N, int64_t K,
        const poot_linear_options& o, cudaStream_t stream) {
  int rc = validate(x, w, b, y, M, N, K);
  if (rc != POOT_OK) return rc;
  int variant = o.variant;
  const int gemv_wpr = o.gemv_warps_per_row;
  if (variant < POOT_VARIANT_AUTO || variant > POOT_VARIANT_GEMM_PACKED) return POOT_ERR_INVALID_ARG;
  if (gemv_wpr != 0 && gemv_wpr != 1 && gemv_wpr != 2 && gemv_wpr != 4 && gemv_wpr != 8)
    return POOT_ERR_INVALID_ARG;
  if (!gemm_options_ok(o)) return POOT_ERR_INVALID_ARG;
  if (o.gemm_cluster > 1 && variant != POOT_VARIANT_AUTO && variant != POOT_VARIANT_GEMM_TMA &&
      variant != POOT_VARIANT_GEMM_PACKED)
    return POOT_ERR_INVALID_ARG;
  if (variant == POOT_VARIANT_AUTO) {
    variant = choose_variant(x, w, M, N, K);
  } else if (!variant_applicable(variant, x, w, M, N, K)) {
    return POOT_ERR_INVALID_ARG;
  }
  if (variant == POOT_VARIANT_NONE) return POOT_OK;

  int dev = 0;
  DeviceState* st = nullptr;
  rc = device_state(&dev, &st);
  if (rc != POOT_OK) return rc;

  switch (variant) {
    case POOT_VARIANT_BIAS_ONLY: {
      const int64_t total = M * N;
      int64_t blocks = (total + 255) / 256;
      const int64_t cap = int64_t(st->sm_count) * 8;
      if (blocks > cap) blocks = cap;
      const cudaError_t e = launch(bias_only_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                                   static_cast<const __half*>(b), static_cast<__half*>(y), (long long)M,
                                   (long long)N);
      return e == cudaSuccess ? POOT_OK : cuda_fail(e);
    }
    case POOT_VARIANT_GEMV:
    case POOT_VARIANT_GEMV_SCALAR:
      return launch_gemv(variant, *st, x, w, b, y, M, N, K, gemv_wpr, stream);
    default:
      return launch_gemm(variant, *st, x, w, b, y, M, N, K, o.gemm_tile_n, o.gemm_group_m, o.gemm_k_chunk,
                         o.gemm_cluster, o.gemm_split_k, stream);
  }
}

// The widened contraction (G groups; G = 1 for poot_contract): argument
// checks, GEMM variant, launch.
int contract(const void* x, const void* w, const void* b, void* y, int64_t G, int64_t M, int64_t N, int64_t K,
             const poot_contraction_spec* spec, const poot_linear_options* opts, cudaStream_t stream) {
  if (spec == nullptr) return POOT_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return POOT_ERR_INVALID_ARG;
  if (G < 1 || G > kMaxDim || G * M > kMaxDim || G * N > kMaxDim) return POOT_ERR_INVALID_ARG;
  if (spec->dtype != POOT_DTYPE_F16 && spec->dtype != POOT_DTYPE_BF16) return POOT_ERR_INVALID_ARG;
  if (spec->num_steps < 0 || spec->num_steps > POOT_EPILOGUE_MAX_STEPS) return POOT_ERR_INVALID_ARG;
  if (spec->out_f32 != 0 && spec->out_f32 != 1) return POOT_ERR_INVALID_ARG;
  if (spec->out_f32 && spec->num_steps != 0) return POOT_ERR_INVALID_ARG;
  EpiConfig epi;
  std::memset(&epi, 0, sizeof(epi));
  epi.dtype = spec->dtype;
  epi.out_f32 = spec->out_f32;
  epi.num_steps = spec->num_steps;
  for (int s = 0; s < spec->num_steps; ++s) {
    const poot_epilogue_step& st = spec->steps[s];
    if (st.op < POOT_EP_ADD || st.op > POOT_EP_GELU_ERF) return POOT_ERR_INVALID_ARG;
    epi.op[s] = st.op;
    if (st.op == POOT_EP_ADD || st.op == POOT_EP_MUL) {
      const int64_t ld = st.ld == 0 ? N : st.ld;
      if (st.operand == nullptr || ld < N || ld > kMaxDim) return POOT_ERR_INVALID_ARG;
      epi.ptr[s] = st.operand;
      epi.ld[s] = ld;
    }
  }
  poot_linear_options o;
  std::memset(&o, 0, sizeof(o));
  o.variant = POOT_VARIANT_AUTO;
  if (opts != nullptr) o = *opts;
  if (!gemm_options_ok(o)) return POOT_ERR_INVALID_ARG;
  if (o.variant != POOT_VARIANT_AUTO && o.variant != POOT_VARIANT_GEMV && o.variant != POOT_VARIANT_GEMM_TMA &&
      o.variant != POOT_VARIANT_GEMM_CPASYNC && o.variant != POOT_VARIANT_GEMM_REG &&
      o.variant != POOT_VARIANT_GEMM_PACKED)
    return POOT_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return POOT_OK;
  if (K == 0 || x == nullptr || w == nullptr || y == nullptr) return POOT_ERR_INVALID_ARG;
  if (!aligned(x, 2) || !aligned(w, 2) || (b != nullptr && !aligned(b, 2)) || !aligned(y, spec->out_f32 ? 4 : 2))
    return POOT_ERR_MISALIGNED;
  const int64_t ybytes = G * M * N * (spec->out_f32 ? 4 : 2);
  if (overlaps(y, ybytes, x, G * M * K * 2) || overlaps(y, ybytes, w, G * N * K * 2) ||
      (b != nullptr && overlaps(y, ybytes, b, G * N * 2)))
    return POOT_ERR_INVALID_ARG;
  for (int s = 0; s < epi.num_steps; ++s) {
    if (epi.ptr[s] == nullptr) continue;
    if (!aligned(epi.ptr[s], 2)) return POOT_ERR_MISALIGNED;
    if (overlaps(y, ybytes, epi.ptr[s], ((G * M - 1) * epi.ld[s] + N) * 2)) return POOT_ERR_INVALID_ARG;
  }
  // M <= 16 (operands readable by 16-byte loads, no GEMM split asked for):
  // the GEMV kernels with the per-element epilogue, any number of groups
  const bool gemv_ok = M <= POOT_GEMV_MAX_M && xw_tma_ok(x, w, K);
  if (o.variant == POOT_VARIANT_GEMV && !gemv_ok) return POOT_ERR_INVALID_ARG;
  if (o.variant == POOT_VARIANT_GEMV || (o.variant == POOT_VARIANT_AUTO && gemv_ok && o.gemm_split_k <= 1)) {
    int dev = 0;
    DeviceState* st = nullptr;
    const int rc = device_state(&dev, &st);
    if (rc != POOT_OK) return rc;
    return launch_gemv_wide(*st, x, w, b, y, M, N, K, G, epi, stream);
  }
  int variant = o.variant;
  if (variant == POOT_VARIANT_AUTO) {
    variant = xw_tma_ok(x, w, K) ? POOT_VARIANT_GEMM_TMA : POOT_VARIANT_GEMM_PACKED;
  } else if (!variant_applicable(variant, x, w, M, N, K)) {
    return POOT_ERR_INVALID_ARG;
  }
  if (o.gemm_cluster == 2 && variant != POOT_VARIANT_GEMM_TMA && variant != POOT_VARIANT_GEMM_PACKED)
    return POOT_ERR_INVALID_ARG;
  if (o.gemm_split_k > 1 && G > 1) return POOT_ERR_INVALID_ARG;
  int dev = 0;
  DeviceState* st = nullptr;
  const int rc = device_state(&dev, &st);
  if (rc != POOT_OK) return rc;
  const int chunk = (o.gemm_k_chunk == 0 && epi.num_steps > 0) ? kStepsChunkK : o.gemm_k_chunk;
  return launch_gemm(variant, *st, x, w, b, y, M, N, K, o.gemm_tile_n, o.gemm_group_m, chunk,
                     o.gemm_cluster, o.gemm_split_k, stream, &epi, G);
}

// ---- split-K without allocation -----------------------------------------------
// The partial sums of poot_linear_f16_splitk_noalloc live in this array,
// compiled into the library (one per device, in the module's global memory),
// so that callers that must not allocate — under a caching allocator that
// holds the device's memory budget, or in a serving loop that cannot take an
// allocation's implicit synchronisation — still get split-K.  Every element
// a call reads is written earlier in the same call, so it is never cleared.
// Calls that overlap in time race on it (one array per device).
static_assert(POOT_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size");
static __device__ __align__(256) float g_noalloc_scratch[POOT_NOALLOC_SCRATCH_BYTES / sizeof(float)];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Address of the array on device `dev` (the current device), looked up once.
int noalloc_scratch(int dev, float** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    g_noalloc_addr[dev] = p;
  }
  *out = static_cast<float*>(g_noalloc_addr[dev]);
  return POOT_OK;
}

int run_splitk_noalloc(const void* x, const void* w, const void* b, void* y, int64_t M, int64_t N, int64_t K,
                       int split_k, cudaStream_t stream) {
  int rc = validate(x, w, b, y, M, N, K);
  if (rc != POOT_OK) return rc;
  if (split_k < 2 || split_k > kMaxSplitK) return POOT_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return POOT_OK;
  const int64_t num_kb = (K + kGemmBK - 1) / kGemmBK;
  if (K == 0 || num_kb % split_k != 0) return POOT_ERR_INVALID_ARG;
  // split_k * M * N * 4 <= the array, without overflow (M, N < 2^31)
  if (M * N > int64_t(POOT_NOALLOC_SCRATCH_BYTES / sizeof(float)) / split_k) return POOT_ERR_INVALID_ARG;
  int variant = POOT_VARIANT_GEMM_REG;
  if (xw_tma_ok(x, w, K)) variant = POOT_VARIANT_GEMM_TMA;
  else if (K % 2 == 0 && aligned(x, 4) && aligned(w, 4)) variant = POOT_VARIANT_GEMM_CPASYNC;
  int dev = 0;
  DeviceState* st = nullptr;
  rc = device_state(&dev, &st);
  if (rc != POOT_OK) return rc;
  float* scratch = nullptr;
  rc = noalloc_scratch(dev, &scratch);
  if (rc != POOT_OK) return rc;
  return launch_gemm(variant, *st, x, w, b, y, M, N, K, 0, 0, 0, 0, split_k, stream, nullptr, 1, scratch,
                     POOT_NOALLOC_SCRATCH_BYTES);
}

// ---- tensor-parallel helpers -------------------------------------------------
// Shard plan of a tensor-parallel linear over `world` ranks: contiguous ranges
// of `extent` (N for a column split, K for a row split), every range but the
// last `width` elements wide, width a multiple of 8 so that every shard of a
// 16-byte-aligned operand stays 16-byte aligned (its TMA path applies).
int64_t tp_width(int64_t extent, int world) {
  int64_t w = (extent + world - 1) / world;
  w = (w + 7) / 8 * 8;
  return w < 8 ? 8 : w;
}

void tp_shard(int64_t extent, int world, int rank, int64_t* begin, int64_t* end) {
  const int64_t w = tp_width(extent, world);
  const int64_t b = int64_t(rank) * w, e = b + w;
  *begin = b < extent ? b : extent;
  *end = e < extent ? e : extent;
}

int gather_columns(const void* slots, void* y, int64_t M, int64_t N, int world, int64_t slot_elems,
                   cudaStream_t stream) {
  if (M < 0 || N < 0 || M > kMaxDim || N > kMaxDim || world < 1 || world > 65536 || slot_elems < 0)
    return POOT_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return POOT_OK;
  if (slots == nullptr || y == nullptr) return POOT_ERR_INVALID_ARG;
  if (!aligned(slots, 2) || !aligned(y, 2)) return POOT_ERR_MISALIGNED;
  const int64_t width = tp_width(N, world);
  // the first shard is the widest; every slot must hold it, and the shards
  // must cover N
  const int64_t w0 = width < N ? width : N;
  if (slot_elems < M * w0 || width * int64_t(world) < N) return POOT_ERR_INVALID_ARG;
  if (overlaps(y, M * N * 2, slots, int64_t(world) * slot_elems * 2)) return POOT_ERR_INVALID_ARG;
  int dev = 0;
  DeviceState* st = nullptr;
  const int rc = device_state(&dev, &st);
  if (rc != POOT_OK) return rc;
  GatherColumnsArgs a;
  a.slots = static_cast<const uint16_t*>(slots);
  a.y = static_cast<uint16_t*>(y);
  a.M = M;
  a.N = N;
  a.slot_elems = slot_elems;
  a.width = width;
  a.world = world;
  const int64_t chunks = M * ((N + 7) / 8);
  int64_t blocks = (chunks + 255) / 256;
  const int64_t cap = int64_t(st->sm_count) * 8;
  if (blocks > cap) blocks = cap;
  const cudaError_t e = launch(gather_columns_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, a);
  return e == cudaSuccess ? POOT_OK : cuda_fail(e);
}

int finish_f16(const float* S, const void* b, void* y, int64_t M, int64_t N, cudaStream_t stream) {
  if (M < 0 || N < 0 || M > kMaxDim || N > kMaxDim) return POOT_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return POOT_OK;
  if (S == nullptr || b == nullptr || y == nullptr) return POOT_ERR_INVALID_ARG;
  if (!aligned(S, 4) || !aligned(b, 2) || !aligned(y, 2)) return POOT_ERR_MISALIGNED;
  if (overlaps(y, M * N * 2, S, M * N * 4) || overlaps(y, M * N * 2, b, N * 2)) return POOT_ERR_INVALID_ARG;
  int dev = 0;
  DeviceState* st = nullptr;
  const int rc = device_state(&dev, &st);
  if (rc != POOT_OK) return rc;
  // the split-K reduce with one partial: y = RN16(RN16(S) + b)
  SplitReduceArgs ra;
  std::memset(&ra, 0, sizeof(ra));
  ra.ws = S;
  ra.S = 1;
  ra.M = static_cast<int>(M);
  ra.N = static_cast<int>(N);
  ra.e.dtype = POOT_DTYPE_F16;
  ra.e.has_bias = 1;
  ra.e.b = static_cast<const uint16_t*>(b);
  ra.e.y = static_cast<uint16_t*>(y);
  ra.e.ldy = N;
  const bool vec = N % 4 == 0 && aligned(S, 16) && aligned(y, 8);
  const int64_t units = vec ? M * N / 4 : M * N;
  int64_t blocks = (units + 255) / 256;
  const int64_t cap = int64_t(st->sm_count) * 8;
  if (blocks > cap) blocks = cap;
  const cudaError_t e = vec ? launch(splitk_reduce_kernel<4>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                                     stream, ra)
                            : launch(splitk_reduce_kernel<1>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                                     stream, ra);
  return e == cudaSuccess ? POOT_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

int poot_contract(const void* x, const void* w, const void* b, void* y, int64_t M, int64_t N, int64_t K,
                  const poot_contraction_spec* spec, const poot_linear_options* opts, poot_stream_t stream) {
  return contract(x, w, b, y, 1, M, N, K, spec, opts, reinterpret_cast<cudaStream_t>(stream));
}

int poot_contract_grouped(const void* x, const void* w, const void* b, void* y, int64_t G, int64_t M, int64_t N,
                          int64_t K, const poot_contraction_spec* spec, const poot_linear_options* opts,
                          poot_stream_t stream) {
  return contract(x, w, b, y, G, M, N, K, spec, opts, reinterpret_cast<cudaStream_t>(stream));
}

int poot_linear_f16_splitk_noalloc(const void* x, const void* w, const void* b, void* y, int64_t M, int64_t N,
                                   int64_t K, int split_k, poot_stream_t stream) {
  return run_splitk_noalloc(x, w, b, y, M, N, K, split_k, reinterpret_cast<cudaStream_t>(stream));
}

int poot_linear_gemm_plan(int64_t M, int64_t N, int64_t K, int sm_count, poot_gemm_plan* out) {
  if (M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxDim || sm_count < 2 || out == nullptr)
    return POOT_ERR_INVALID_ARG;
  const GemmPlan p = plan_gemm(M, N, K, sm_count, 0, 0, 0, 0, 0, true, true);
  const int64_t bm = p.pair ? 2 * kGemmBM : kGemmBM;
  std::memset(out, 0, sizeof(*out));
  out->tile_n = p.bn;
  out->cluster = p.cluster;
  out->split_k = p.split;
  out->k_chunk = p.chunk_kb * kGemmBK;
  out->tiles = static_cast<int>(((M + bm - 1) / bm) * ((N + p.bn - 1) / p.bn) * p.split);
  out->ctas = p.pair ? 2 * (sm_count / 2) : sm_count;
  return POOT_OK;
}

int poot_linear_tp_shard(int64_t extent, int world, int rank, int64_t* begin, int64_t* end) {
  if (extent < 0 || extent > kMaxDim || world < 1 || world > 65536 || rank < 0 || rank >= world ||
      begin == nullptr || end == nullptr)
    return POOT_ERR_INVALID_ARG;
  tp_shard(extent, world, rank, begin, end);
  return POOT_OK;
}

int poot_linear_gather_columns(const void* slots, void* y, int64_t M, int64_t N, int world, int64_t slot_elems,
                               poot_stream_t stream) {
  return gather_columns(slots, y, M, N, world, slot_elems, reinterpret_cast<cudaStream_t>(stream));
}

int poot_linear_f16_finish(const float* S, const void* b, void* y, int64_t M, int64_t N, poot_stream_t stream) {
  return finish_f16(S, b, y, M, N, reinterpret_cast<cudaStream_t>(stream));
}

int poot_linear_f16(const void* x, const void* w, const void* b, void* y, int64_t M, int64_t N, int64_t K,
                    poot_stream_t stream) {
  poot_linear_options o;
  std::memset(&o, 0, sizeof(o));
  o.variant = POOT_VARIANT_AUTO;
  return run(x, w, b, y, M, N, K, o, reinterpret_cast<cudaStream_t>(stream));
}

int poot_linear_f16_ex(const void* x, const void* w, const void* b, void* y, int64_t M, int64_t N, int64_t K,
                       const poot_linear_options* opts, poot_stream_t stream) {
  poot_linear_options o;
  std::memset(&o, 0, sizeof(o));
  o.variant = POOT_VARIANT_AUTO;
  if (opts != nullptr) o = *opts;
  return run(x, w, b, y, M, N, K, o, reinterpret_cast<cudaStream_t>(stream));
}

int poot_linear_f16_variant(const void* x, const void* w, const void* b, const void* y, int64_t M, int64_t N,
                            int64_t K) {
  const int rc = validate(x, w, b, y, M, N, K);
  if (rc != POOT_OK) return -rc;
  return choose_variant(x, w, M, N, K);
}

const char* poot_linear_status_string(int status) {
  switch (status) {
    case POOT_OK: return "ok";
    case POOT_ERR_INVALID_ARG: return "invalid argument";
    case POOT_ERR_MISALIGNED: return "pointer not 2-byte aligned";
    case POOT_ERR_UNSUPPORTED_DEVICE: return "unsupported device (sm_103 required)";
    case POOT_ERR_CUDA: return "CUDA error";
    case POOT_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

const char* poot_linear_last_cuda_error(void) { return cudaGetErrorName(t_last_cuda_error); }

int poot_linear_device_status(poot_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, poot::g_device_error, sizeof(word));
  if (e != cudaSuccess) return cuda_fail(e);
  if (word != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(poot::g_device_error, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e);
    return POOT_ERR_DEVICE_TIMEOUT;
  }
  return POOT_OK;
}

int poot_linear_version(void) { return kVersion; }

}  // extern "C"
