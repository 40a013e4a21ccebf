// The device steps of the tensor-parallel linear that are not the
// contraction itself: reassembling y from the column shards that an
// all-gather brought together, and the head epilogue of a K-split whose FP32
// partial sums an all-reduce has added ("The Graph IR", Primitive
// operations, the AllReduce / AllGather row; "Model and Distributed IR",
// section "Boundary between the layers": rank-local matmul tasks, a
// collective, and the reconstructed result).
//
// Shards are the contiguous ranges of the plan in poot_linear.cu
// (tp_shard): every shard but the last is `width` wide, so the shard of
// output column n is n / width.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace poot {

struct GatherColumnsArgs {
  const uint16_t* slots;  // [world][slot_elems]; slot r holds y_r [M, N_r] row-major
  uint16_t* y;            // [M, N] row-major
  long long M, N, slot_elems, width;
  int world;
};

// One thread per 8-element chunk of a y row.  A chunk inside one shard is
// copied with one 16-byte load and store when both addresses are 16-byte
// aligned; otherwise element by element (ragged shard edges, odd pitches).
__global__ void __launch_bounds__(256) gather_columns_kernel(const GatherColumnsArgs a) {
  grid_dep_wait();  // the gathered slots come from earlier work in the stream
  grid_dep_launch();
  const long long cpr = (a.N + 7) / 8;  // chunks per y row
  const long long total = a.M * cpr;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long m = i / cpr;
    const long long n0 = (i - m * cpr) * 8;
    const long long n1 = n0 + 8 < a.N ? n0 + 8 : a.N;
    const long long r0 = n0 / a.width, r1 = (n1 - 1) / a.width;
    uint16_t* dst = a.y + m * a.N + n0;
    if (r0 == r1 && n1 - n0 == 8) {
      const long long c0 = r0 * a.width;
      const long long nr = (c0 + a.width < a.N ? c0 + a.width : a.N) - c0;
      const uint16_t* src = a.slots + r0 * a.slot_elems + m * nr + (n0 - c0);
      if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u) == 0) {
        *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(src));
        continue;
      }
    }
    for (long long n = n0; n < n1; ++n) {
      const long long r = n / a.width;
      const long long c0 = r * a.width;
      const long long nr = (c0 + a.width < a.N ? c0 + a.width : a.N) - c0;
      dst[n - n0] = __ldg(a.slots + r * a.slot_elems + m * nr + (n - c0));
    }
  }
}

}  // namespace poot
