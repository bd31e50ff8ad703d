// Second pass of the fused dbias: dbias[j] = sum over 128-row tiles t of ws[t][j].
//
// The quantize kernel leaves one fp32 partial column sum per 128-row tile in
// the workspace ws[row_tiles][N].  Here one CTA owns 32 columns; warp w sums
// tiles t = w, w + 8, w + 16, ... in fp64 (a coalesced 128-byte row per tile)
// and the eight warp sums are added in warp order, so the result does not
// depend on scheduling.  Like the quantize kernel it honours the device noop
// flag (the noop + reduce_dbias interaction raised in the review summary of
// "[Common] Experimental CuTeDSL MXFP8 backends in C++ via TVM-FFI").
#pragma once

#include <cstdint>

namespace mxfp8 {

constexpr int kReduceCols = 32;
constexpr int kReduceWarps = 8;

__global__ void __launch_bounds__(kReduceCols * kReduceWarps)
    dbias_reduce_kernel(const float *__restrict__ ws, int64_t row_tiles, int64_t N, float *__restrict__ dbias,
                        const float *noop)
{
    if (noop != nullptr && *noop == 1.0f)
        return;
    __shared__ double part[kReduceWarps][kReduceCols];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kReduceCols + lane;
    double acc = 0.0;
    if (j < N) {
#pragma unroll 4
        for (int64_t t = warp; t < row_tiles; t += kReduceWarps)
            acc += static_cast<double>(ws[t * N + j]);
    }
    part[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && j < N) {
        double s = part[0][lane];
#pragma unroll
        for (int w = 1; w < kReduceWarps; ++w)
            s += part[w][lane];
        dbias[j] = static_cast<float>(s);
    }
}

}  // namespace mxfp8
