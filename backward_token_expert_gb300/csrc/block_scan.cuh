// Block-wide scan shared by the route-stats and selection kernels.
#pragma once

namespace lrm {

// Exclusive prefix sum of one int per thread over a 1024-thread block;
// *total receives the block sum.  Every thread of the block must call it.
__device__ __forceinline__ int block_exclusive_scan_1024(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int w = s_warp[lane];
    int z = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, z, o);
      if (lane >= o) z += y;
    }
    s_warp[lane] = z - w;
    if (lane == 31) *total = z;
  }
  __syncthreads();
  const int r = s_warp[warp] + x - v;
  __syncthreads();
  return r;
}

}  // namespace lrm
