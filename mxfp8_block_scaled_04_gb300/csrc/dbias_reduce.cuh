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

#include "ptx.cuh"
#include "quantize.cuh"  // kMaxGroups

namespace mxfp8 {

constexpr int kReduceCols = 32;
constexpr int kReduceWarps = 16;
#ifndef MXFP8_GREDUCE_WARPS
#define MXFP8_GREDUCE_WARPS 16
#endif
#ifndef MXFP8_GREDUCE_INFLIGHT
#define MXFP8_GREDUCE_INFLIGHT 16
#endif
constexpr int kGReduceWarps = MXFP8_GREDUCE_WARPS;        // grouped reduce: warps per 32-column CTA
constexpr int kGReduceInflight = MXFP8_GREDUCE_INFLIGHT;  // grouped reduce: tile loads in flight per warp

__global__ void __launch_bounds__(kReduceCols * kReduceWarps)
    dbias_reduce_kernel(const float *__restrict__ ws, int64_t row_tiles, int64_t N, float *__restrict__ dbias,
                        const float *noop)
{
    pdl_wait_and_release();
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
// row tile into hdr[0..G] (hdr[G] = T, the total), or hdr[0] = -1 when the
// offsets are invalid (then nothing is written here either).
//
// One CTA owns 32 columns of every group.  Its 16 warps split the T row tiles
// into contiguous ranges [T w / 16, T (w + 1) / 16); a warp sums the tiles of
// each group inside its range in tile order, with 16 tiles' loads in flight
// (8 measured 0.5% slower on the whole 64-expert call; 32 warps no better).  A group that lies wholly inside
// one range is written by that warp; the partial sums of a group that crosses
// ranges are left in shared memory, and the warp holding the group's last
// tile adds them in warp order.  The order of every sum depends only on T and
// hdr, so the result does not depend on scheduling.  Empty groups get zeros.
__global__ void __launch_bounds__(kReduceCols * kGReduceWarps)
    dbias_reduce_grouped_kernel(const float *__restrict__ ws, const int64_t *__restrict__ hdr, int num_groups,
                                int64_t N, float *__restrict__ dbias, const float *noop)
{
    pdl_wait_and_release();
    if (noop != nullptr && *noop == 1.0f)
        return;
    if (hdr[0] < 0)
        return;
    __shared__ int64_t first[kMaxGroups + 1];
    __shared__ float head[kGReduceWarps][kReduceCols];  // partial of a group that began in an earlier range
    __shared__ float tail[kGReduceWarps][kReduceCols];  // partial of a group that goes on into a later range
    const int G = num_groups;
    for (int i = threadIdx.x; i <= G; i += blockDim.x)
        first[i] = hdr[i];
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kReduceCols + lane;
    const int64_t T = first[G];
    const int64_t a = T * warp / kGReduceWarps, b = T * (warp + 1) / kGReduceWarps;

    for (int g = warp; g < G; g += kGReduceWarps)
        if (first[g] == first[g + 1] && j < N)
            dbias[static_cast<int64_t>(g) * N + j] = 0.f;

    int g0 = 0;  // the group of tile a: first[g0] <= a < first[g0 + 1]
    if (a < b) {
        int lo = 0, hi = G;  // first[lo] <= a < first[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (first[mid] <= a)
                lo = mid;
            else
                hi = mid;
        }
        g0 = lo;
        // a finished group's sum: written here, or left for the warp that completes it
        auto flush = [&](int g, float acc) {
            const bool before = first[g] < a, after = first[g + 1] > b;
            if (before)
                head[warp][lane] = acc;
            else if (after)
                tail[warp][lane] = acc;
            else if (j < N)
                dbias[static_cast<int64_t>(g) * N + j] = acc;
        };
        int g = g0;
        int64_t gend = first[g + 1];
        float acc = 0.f;
        // kGReduceInflight tiles' loads in flight at a time, whatever the group boundaries
        for (int64_t t0 = a; t0 < b; t0 += kGReduceInflight) {
            float v[kGReduceInflight];
#pragma unroll
            for (int k = 0; k < kGReduceInflight; ++k)
                v[k] = (t0 + k < b && j < N) ? ws[(t0 + k) * N + j] : 0.f;
#pragma unroll
            for (int k = 0; k < kGReduceInflight; ++k) {
                const int64_t t = t0 + k;
                if (t < b) {
                    if (t == gend) {  // warp-uniform: tile t starts the next non-empty group
                        flush(g, acc);
                        acc = 0.f;
                        do
                            ++g;
                        while (first[g + 1] <= t);
                        gend = first[g + 1];
                    }
                    acc += v[k];
                }
            }
        }
        flush(g, acc);
    }
    __syncthreads();
    // a group that began before this range and ends inside it: add the partials in warp order
    if (a < b && first[g0] < a && first[g0 + 1] <= b) {
        int w1 = warp - 1;  // the range holding the group's first tile
        while (w1 > 0 && T * w1 / kGReduceWarps > first[g0])
            --w1;
        float s = tail[w1][lane];
        for (int w = w1 + 1; w < warp; ++w)
            if (T * w / kGReduceWarps < T * (w + 1) / kGReduceWarps)
                s += head[w][lane];
        s += head[warp][lane];
        if (j < N)
            dbias[static_cast<int64_t>(g0) * N + j] = s;
    }
}

}  // namespace mxfp8
