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
// group g of ws[t][j].  The grouped quantize kernel numbers row tiles group by
// group (group g's tiles follow those of groups 0..g-1, ceil(rows/128) each),
// so CTA (column block, g) first finds its group's first row tile with a block
// sum over the offsets, re-checking them on the way (invalid offsets: write
// nothing, as the quantize kernel does), then sums like the flat reduce.
__global__ void __launch_bounds__(kReduceCols * kReduceWarps)
    dbias_reduce_grouped_kernel(const float *__restrict__ ws, const int64_t *__restrict__ offsets, int G,
                                int64_t total_rows, int64_t N, float *__restrict__ dbias, const float *noop)
{
    if (noop != nullptr && *noop == 1.0f)
        return;
    __shared__ long long s_start[kReduceWarps];
    __shared__ int s_bad[kReduceWarps];
    __shared__ float part[kReduceWarps][kReduceCols];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = blockIdx.y;
    long long start = 0;
    int bad = 0;
    for (int h = threadIdx.x; h < G; h += blockDim.x) {
        const int64_t a = offsets[h], b = offsets[h + 1];
        if (b < a || (b & 31))
            bad = 1;
        if (h < g)
            start += (b - a + 127) / 128;
    }
    if (threadIdx.x == 0 && (offsets[0] != 0 || offsets[G] != total_rows))
        bad = 1;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        start += __shfl_xor_sync(0xffffffffu, start, d);
        bad |= __shfl_xor_sync(0xffffffffu, bad, d);
    }
    if (lane == 0) {
        s_start[warp] = start;
        s_bad[warp] = bad;
    }
    __syncthreads();
    start = 0;
    bad = 0;
#pragma unroll
    for (int w = 0; w < kReduceWarps; ++w) {
        start += s_start[w];
        bad |= s_bad[w];
    }
    if (bad)
        return;
    const int64_t nrt = (offsets[g + 1] - offsets[g] + 127) / 128;
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
