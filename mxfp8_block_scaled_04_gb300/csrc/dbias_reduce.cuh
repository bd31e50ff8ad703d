// Second pass of the fused dbias: dbias[j] = sum over 128-row tiles t of ws[t][j].
//
// The quantize kernel leaves one fp32 partial column sum per 128-row tile in
// the workspace ws[row_tiles][N].  Here one CTA owns 32 columns; warp w sums
// tiles t = w, w + 16, w + 32, ... in fp32 (a coalesced 128-byte row per tile,
// all of a thread's loads in flight together) and the 16 warp sums are added
// in warp order, so the result does not
// depend on scheduling.  fp32 keeps the error of the whole dbias (tile sums
// included) below about 42 roundings of sum |x|, i.e. 2.5e-6 * sum |x|; GB300's
// fp64 rate is a small fraction of its fp32 rate.  Like the quantize kernel it
// honours the device noop flag (the noop + reduce_dbias interaction raised in the review summary of
// "[Common] Experimental CuTeDSL MXFP8 backends in C++ via TVM-FFI").
#pragma once

#include <cstdint>

namespace mxfp8 {

constexpr int kReduceCols = 32;
constexpr int kReduceWarps = 16;

__global__ void __launch_bounds__(kReduceCols * kReduceWarps)
    dbias_reduce_kernel(const float *__restrict__ ws, int64_t row_tiles, int64_t N, float *__restrict__ dbias,
                        const float *noop)
{
    if (noop != nullptr && *noop == 1.0f)
        return;
    __shared__ float part[kReduceWarps][kReduceCols];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kReduceCols + lane;
    float acc = 0.f;
    if (j < N) {
#pragma unroll 8
        for (int64_t t = warp; t < row_tiles; t += kReduceWarps)
            acc += ws[t * N + j];
    }
    part[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && j < N) {
        float s = part[0][lane];
#pragma unroll
        for (int w = 1; w < kReduceWarps; ++w)
            s += part[w][lane];
        dbias[j] = s;
    }
}

// Per-group dbias of the grouped call: dbias[g][j] = sum over the row tiles of
// group g of ws[t][j].  The grouped quantize kernel writes each group's first
// row tile into hdr[0..G] (hdr[G] = total), or hdr[0] = -1 when the offsets are
// invalid (then nothing is written here either).  CTA (column block, g) sums
// its group's tiles like the flat reduce: warp w takes tiles w, w+16, ... and
// the 16 warp sums are added in warp order.
__global__ void __launch_bounds__(kReduceCols * kReduceWarps)
    dbias_reduce_grouped_kernel(const float *__restrict__ ws, const int64_t *__restrict__ hdr, int64_t N,
                                float *__restrict__ dbias, const float *noop)
{
    if (noop != nullptr && *noop == 1.0f)
        return;
    if (hdr[0] < 0)
        return;
    __shared__ float part[kReduceWarps][kReduceCols];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = blockIdx.y;
    const int64_t start = hdr[g], nrt = hdr[g + 1] - hdr[g];
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kReduceCols + lane;
    float acc = 0.f;
    if (j < N) {
#pragma unroll 8
        for (int64_t t = warp; t < nrt; t += kReduceWarps)
            acc += ws[(start + t) * N + j];
    }
    part[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && j < N) {
        float s = part[0][lane];
#pragma unroll
        for (int w = 1; w < kReduceWarps; ++w)
            s += part[w][lane];
        dbias[static_cast<int64_t>(g) * N + j] = s;
    }
}

}  // namespace mxfp8
