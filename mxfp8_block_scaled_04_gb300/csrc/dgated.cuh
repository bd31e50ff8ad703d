// Backward of the gated activations: the MXFP8 cast of the gradient of
// x = [a | b] for y = act(a) * b (ReGLU, squared-ReLU GLU, GeGLU, SwiGLU,
// QGeGLU), given the gradient g of y:
//     da = g * b * act'(a),   db = g * act(a)      (fp32),
// da and db quantized as two [M, N] tensors laid side by side in [M, 2N]
// buffers (codes; scale_row [M, 2 ceil(N/32)], da's blocks first;
// scale_col [ceil(M/32), 2N]).
//
// Two kernels.  The first (squared-ReLU GLU, measured faster there): three
// BF16 inputs per element (g, a, b), so a stage holds three 128-row x
// 64-column boxes (48 KiB) and the kernel keeps two stages per CTA, two CTAs
// per SM (four tiles in flight per SM).  The phases follow the backward
// fusion's kernel:
//   - phase 1: warp w takes rows 32*(w>>1) + 16*(w&1) .. +15 of the tile, a
//     lane 4 columns x 8 rows; it forms da and db and their column maxima; the
//     two 16-row halves of a 32-row block meet in shared memory, where one
//     thread per (row block, column) forms both outputs' scales and column
//     multipliers;
//   - phase 2: warp w takes the 8-row groups 2w and 2w + 1; a lane 16
//     columns of one row: it forms da and db again (the same function of the
//     same inputs, so the same values), then both directions of both.
// act and act' come from the forward and derivative routines of the other
// kernels (one ex2 and one rcp shared between them).
#pragma once

#include <cstdint>
#include <cuda.h>

#include "dact.cuh"
#include "ptx.cuh"
#include "quantize.cuh"

namespace mxfp8 {

constexpr int kGStages = 2;
constexpr int kGStageBytes = 3 * kBoxBytes;                    // g, a, b boxes
constexpr int kGOffColMul = kGStages * kGStageBytes;           // float [2][4][64]
constexpr int kGOffPartF = kGOffColMul + 2 * 4 * kDBN * 4;     // float [2][2][4][64]
constexpr int kGOffBars = kGOffPartF + 2 * 2 * 4 * kDBN * 4;   // uint64 [kGStages]
constexpr int kGOffCoord = kGOffBars + 8 * kGStages;           // TileCoord [kGStages]
constexpr int kSmemDgated = kGOffCoord + 32 * kGStages + 1024;

// da = (g b) act'(a) and db = g act(a) for two elements (lanes of packed pairs); g b is
// a product of two BF16 values, exact in fp32.
template <int ACT>
__device__ __forceinline__ void dgate2(uint32_t gw, uint32_t aw, uint32_t bw, uint64_t &da, uint64_t &db)
{
    const uint64_t g = f2_pack(bf16_lo(gw), bf16_hi(gw));
    const uint64_t a = f2_pack(bf16_lo(aw), bf16_hi(aw));
    const uint64_t b = f2_pack(bf16_lo(bw), bf16_hi(bw));
    da = f2_mul(f2_mul(g, b), dactivation2<ACT>(a));
    db = f2_mul(g, activation2<ACT>(a));
}

template <int FMT, int ACT>
__global__ void __launch_bounds__(kThreads, 2)
    quantize_dgated_kernel(const __grid_constant__ CUtensorMap tmap_g, const __grid_constant__ CUtensorMap tmap_a,
                           const __grid_constant__ CUtensorMap tmap_b, const QuantParams p)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *colmul = reinterpret_cast<float *>(smem + kGOffColMul);  // [out][rb][64], rotated
    float *part_f = reinterpret_cast<float *>(smem + kGOffPartF);   // [out][half][rb][64]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kGOffBars);
    TileCoord *coords = reinterpret_cast<TileCoord *>(smem + kGOffCoord);

    pdl_wait_and_release();
    if (p.noop != nullptr && *p.noop == 1.0f)
        return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t N = p.N, N2 = 2 * p.N;
    const int64_t Cn = (N + 31) >> 5;  // scale columns of one half
    const int num_tiles = p.row_tiles * p.col_tiles;
    const int first = blockIdx.x, stride = gridDim.x;
    const int my_count = first < num_tiles ? (num_tiles - 1 - first) / stride + 1 : 0;
    if (my_count == 0)
        return;
    const bool do_row = p.out_row != nullptr, do_col = p.out_col != nullptr;
    const bool rows16 = (N & 15) == 0;  // both halves' FP8 rows 16-byte aligned (else 8-byte)

    if (tid == 0) {
        prefetch_tensormap(&tmap_g);
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
        for (int s = 0; s < kGStages; ++s)
            mbar_init(smem_u32(&bars[s]), 1);
        fence_mbar_init();
    }
    __syncthreads();

    auto issue = [&](int slot, int t) {
        const int rt = t / p.col_tiles, ct = t - rt * p.col_tiles;
        TileCoord c;
        c.row0 = static_cast<int64_t>(rt) * kBM;
        c.row_end = min(c.row0 + kBM, p.M);
        c.col0 = ct * kDBN;
        c.rt = rt;
        c.sb = rt * (kBM / 32);
        c.g = 0;
        coords[slot] = c;  // published to the consumers by the arrive below
        const uint32_t bar = smem_u32(&bars[slot]);
        const uint32_t dst = smem_u32(smem + slot * kGStageBytes);
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, kGStageBytes);
        tma_load_2d(dst, &tmap_g, bar, c.col0, static_cast<int32_t>(c.row0));
        tma_load_2d(dst + kBoxBytes, &tmap_a, bar, c.col0, static_cast<int32_t>(c.row0));
        tma_load_2d(dst + 2 * kBoxBytes, &tmap_b, bar, c.col0, static_cast<int32_t>(c.row0));
    };
    if (tid == 0)
        for (int s = 0; s < kGStages && s < my_count; ++s)
            issue(s, first + s * stride);

    for (int it = 0; it < my_count; ++it) {
        const int slot = it % kGStages;
        const uint32_t parity = static_cast<uint32_t>(it / kGStages) & 1u;
        const unsigned char *gbox = smem + slot * kGStageBytes;
        const unsigned char *abox = gbox + kBoxBytes;
        const unsigned char *bbox = gbox + 2 * kBoxBytes;
        const bool ok = mbar_wait_bounded(smem_u32(&bars[slot]), parity, kWaitLimitNs);
        const TileCoord tc = coords[slot];

        // ---- phase 1: both outputs' column maxima over 16-row halves ----
        if (ok) {
            const int rb = warp >> 1, hh = warp & 1;
            const int cq = lane & 15, q = lane >> 4;
            const int r0 = rb * 32 + hh * 16 + q * 8;  // r0 & 7 == 0
            float fa[4] = {0.f, 0.f, 0.f, 0.f}, fb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int off = (r0 + i) * 128 + (((cq >> 1) ^ i) << 4) + (cq & 1) * 8;
                const uint2 g = lds64(gbox + off), a = lds64(abox + off), b = lds64(bbox + off);
                uint64_t da01, db01, da23, db23;
                dgate2<ACT>(g.x, a.x, b.x, da01, db01);
                dgate2<ACT>(g.y, a.y, b.y, da23, db23);
                float v[4];
                f2_unpack(da01, v[0], v[1]);
                f2_unpack(da23, v[2], v[3]);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    fa[k] = fmaxf(fa[k], fabsf(v[k]));
                f2_unpack(db01, v[0], v[1]);
                f2_unpack(db23, v[2], v[3]);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    fb[k] = fmaxf(fb[k], fabsf(v[k]));
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                fa[k] = fmaxf(fa[k], __shfl_xor_sync(0xffffffffu, fa[k], 16));
                fb[k] = fmaxf(fb[k], __shfl_xor_sync(0xffffffffu, fb[k], 16));
            }
            if (q == 0) {
                const int o = (hh * 4 + rb) * kDBN + cq * 4;
                *reinterpret_cast<float4 *>(part_f + o) = make_float4(fa[0], fa[1], fa[2], fa[3]);
                *reinterpret_cast<float4 *>(part_f + 2 * 4 * kDBN + o) = make_float4(fb[0], fb[1], fb[2], fb[3]);
            }
        }
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicOr(&g_fault_word, 1u);
                for (int j = it; j < my_count && j < it + kGStages; ++j)
                    mbar_wait_bounded(smem_u32(&bars[j % kGStages]), static_cast<uint32_t>(j / kGStages) & 1u,
                                      kDrainLimitNs);
            }
            return;
        }
        // one thread per (32-row block, column): both outputs' scales and multipliers
        {
            const int rb = tid >> 6, c = tid & 63;
            const int64_t grow = tc.row0 + rb * 32, gcol = tc.col0 + c;
            const int sp = c >> 4, qq = (c >> 2) & 3;  // rotated layout, as in the main kernel
            const int rot = 4 * (4 * sp + ((qq + (sp >> 1)) & 3)) + (c & 3);
#pragma unroll
            for (int out = 0; out < 2; ++out) {
                const float *pf = part_f + out * 2 * 4 * kDBN;
                const float amax = fmaxf(pf[rb * kDBN + c], pf[(4 + rb) * kDBN + c]);
                const int e = block_exponent_f32<FMT>(__float_as_uint(amax));
                if (do_col && grow < tc.row_end && gcol < N)
                    p.scale_col[(grow >> 5) * N2 + out * N + gcol] = static_cast<uint8_t>(e);
                colmul[(out * 4 + rb) * kDBN + rot] = scale_multiplier(e);
            }
        }
        __syncthreads();

        // ---- phase 2: 16-column row segments of both outputs ----
        {
            const int rr = lane >> 2, sp = lane & 3;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int rg = 2 * warp + k;
                if (tc.row0 + rg * 8 >= tc.row_end)
                    continue;
                const int r = rg * 8 + rr;
                const int p0 = (2 * sp) ^ rr;
                const int o0 = r * 128 + p0 * 16, o1 = r * 128 + (p0 ^ 1) * 16;
                const uint4 GA = lds128(gbox + o0), GB = lds128(gbox + o1);
                const uint4 AA = lds128(abox + o0), AB = lds128(abox + o1);
                const uint4 BA = lds128(bbox + o0), BB = lds128(bbox + o1);
                const uint32_t gw[8] = {GA.x, GA.y, GA.z, GA.w, GB.x, GB.y, GB.z, GB.w};
                const uint32_t aw[8] = {AA.x, AA.y, AA.z, AA.w, AB.x, AB.y, AB.z, AB.w};
                const uint32_t bw[8] = {BA.x, BA.y, BA.z, BA.w, BB.x, BB.y, BB.z, BB.w};
                float ya[16], yb[16];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint64_t da, db;
                    dgate2<ACT>(gw[j], aw[j], bw[j], da, db);
                    f2_unpack(da, ya[2 * j], ya[2 * j + 1]);
                    f2_unpack(db, yb[2 * j], yb[2 * j + 1]);
                }
                const int64_t grow = tc.row0 + r, gcol = tc.col0 + sp * 16;
                const bool in = grow < tc.row_end && gcol < N;
                const bool half = gcol + 16 > N;
#pragma unroll
                for (int out = 0; out < 2; ++out) {
                    const float *y = out == 0 ? ya : yb;
                    if (do_row) {
                        float fm = 0.f;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            fm = fmaxf(fm, fabsf(y[i]));
                        fm = fmaxf(fm, __shfl_xor_sync(0xffffffffu, fm, 1));
                        const int er = block_exponent_f32<FMT>(__float_as_uint(fm));
                        const uint64_t rm = f2_splat(scale_multiplier(er));
                        uint32_t o[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            o[j] = cvt_fp8x2_scaled<FMT>(y[4 * j], y[4 * j + 1], rm) |
                                   (cvt_fp8x2_scaled<FMT>(y[4 * j + 2], y[4 * j + 3], rm) << 16);
                        if (in) {
                            store_codes(p.out_row + grow * N2 + out * N + gcol, o[0], o[1], o[2], o[3], rows16, half);
                            if ((sp & 1) == 0)
                                p.scale_row[grow * 2 * Cn + out * Cn + (gcol >> 5)] = static_cast<uint8_t>(er);
                        }
                    }
                    if (do_col) {
                        const float *cm = colmul + (out * 4 + (r >> 5)) * kDBN + sp * 16;
                        uint32_t o[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float4 c = lds128f(cm + 4 * ((j + (sp >> 1)) & 3));
                            o[j] = cvt_fp8x2_scaled<FMT>(y[4 * j], y[4 * j + 1], f2_pack(c.x, c.y)) |
                                   (cvt_fp8x2_scaled<FMT>(y[4 * j + 2], y[4 * j + 3], f2_pack(c.z, c.w)) << 16);
                        }
                        if (in)
                            store_codes(p.out_col + grow * N2 + out * N + gcol, o[0], o[1], o[2], o[3], rows16, half);
                    }
                }
            }
        }
        __syncthreads();  // stage and colmul are free again
        if (tid == 0 && it + kGStages < my_count)
            issue(slot, first + (it + kGStages) * stride);
    }
}

}  // namespace mxfp8

namespace mxfp8 {

// The gated backward with each product evaluated once (ReGLU, GeGLU, SwiGLU, QGeGLU).  For the
// transcendental activations their evaluation dominates the kernel above, which evaluates them in
// both phases because its 48 KiB stage cannot hold both fp32 products.  Here a tile is 64 rows x 64 columns
// (three 8 KiB boxes, three stages), and phase 1 writes da and db in fp32 to a 32 KiB keep area
// of the CTA; phase 2 reads them back, and the stage is refilled as soon as phase 1 is done.
//   - phase 1: warp w takes the 8 rows 32*(w>>2) + 8*(w&3) .. +7 of the tile, a lane 4 columns
//     x 4 rows; it forms da and db, keeps them, and their column maxima over its rows; the four
//     8-row parts of a 32-row block meet in shared memory, where one thread per (output, row
//     block, column) forms the scale and column multiplier;
//   - phase 2: warp w takes the 8-row group w; a lane 16 columns of one row, both outputs.
// Keep layout: output o, row r, 16-byte chunk c (four columns) at float offset
// ((o * 64 + r) * 16 + (c ^ ((c >> 3) << 1) ^ (r & 1))) * 4: the stores of phase 1 (a quarter
// warp: one row, chunks 0..7 or 8..15) and the loads of phase 2 (a quarter warp: two rows, chunks
// 4 sp + j) both meet eight distinct 16-byte bank groups.
constexpr int kKRows = 64;                                    // tile rows
constexpr int kKBoxBytes = kKRows * kDBN * 2;                 // 8 KiB
constexpr int kKStages = 3;
constexpr int kKStageBytes = 3 * kKBoxBytes;                  // g, a, b boxes
constexpr int kKOffKeep = kKStages * kKStageBytes;            // float [2][64][64]
constexpr int kKOffColMul = kKOffKeep + 2 * kKRows * kDBN * 4;  // float [2][2][64], rotated
constexpr int kKOffPart = kKOffColMul + 2 * 2 * kDBN * 4;     // float [2][4][2][64]
constexpr int kKOffBars = kKOffPart + 2 * 4 * 2 * kDBN * 4;   // uint64 [kKStages]
constexpr int kKOffCoord = kKOffBars + 8 * kKStages;          // TileCoord [kKStages]
constexpr int kSmemDgatedKeep = kKOffCoord + 32 * kKStages + 1024;

__device__ __forceinline__ int keep_chunk(int c, int r) { return c ^ ((c >> 3) << 1) ^ (r & 1); }

template <int FMT, int ACT>
__global__ void __launch_bounds__(kThreads, 2)
    quantize_dgated_keep_kernel(const __grid_constant__ CUtensorMap tmap_g, const __grid_constant__ CUtensorMap tmap_a,
                                const __grid_constant__ CUtensorMap tmap_b, const QuantParams p)
{
    static_assert(ACT != 2, "squared-ReLU GLU uses the 128-row kernel");
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *keep = reinterpret_cast<float *>(smem + kKOffKeep);
    float *colmul = reinterpret_cast<float *>(smem + kKOffColMul);  // [out][rb][64], rotated
    float *part = reinterpret_cast<float *>(smem + kKOffPart);      // [out][quarter][rb][64]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kKOffBars);
    TileCoord *coords = reinterpret_cast<TileCoord *>(smem + kKOffCoord);

    pdl_wait_and_release();
    if (p.noop != nullptr && *p.noop == 1.0f)
        return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t N = p.N, N2 = 2 * p.N;
    const int64_t Cn = (N + 31) >> 5;  // scale columns of one half
    const int num_tiles = p.row_tiles * p.col_tiles;
    const int first = blockIdx.x, stride = gridDim.x;
    const int my_count = first < num_tiles ? (num_tiles - 1 - first) / stride + 1 : 0;
    if (my_count == 0)
        return;
    const bool do_row = p.out_row != nullptr, do_col = p.out_col != nullptr;
    const bool rows16 = (N & 15) == 0;

    if (tid == 0) {
        prefetch_tensormap(&tmap_g);
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
        for (int s = 0; s < kKStages; ++s)
            mbar_init(smem_u32(&bars[s]), 1);
        fence_mbar_init();
    }
    __syncthreads();

    auto issue = [&](int slot, int t) {
        const int rt = t / p.col_tiles, ct = t - rt * p.col_tiles;
        TileCoord c;
        c.row0 = static_cast<int64_t>(rt) * kKRows;
        c.row_end = min(c.row0 + kKRows, p.M);
        c.col0 = ct * kDBN;
        c.rt = rt;
        c.sb = rt * (kKRows / 32);
        c.g = 0;
        coords[slot] = c;  // published to the consumers by the arrive below
        const uint32_t bar = smem_u32(&bars[slot]);
        const uint32_t dst = smem_u32(smem + slot * kKStageBytes);
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, kKStageBytes);
        tma_load_2d(dst, &tmap_g, bar, c.col0, static_cast<int32_t>(c.row0));
        tma_load_2d(dst + kKBoxBytes, &tmap_a, bar, c.col0, static_cast<int32_t>(c.row0));
        tma_load_2d(dst + 2 * kKBoxBytes, &tmap_b, bar, c.col0, static_cast<int32_t>(c.row0));
    };
    if (tid == 0)
        for (int s = 0; s < kKStages && s < my_count; ++s)
            issue(s, first + s * stride);

    for (int it = 0; it < my_count; ++it) {
        const int slot = it % kKStages;
        const uint32_t parity = static_cast<uint32_t>(it / kKStages) & 1u;
        const unsigned char *gbox = smem + slot * kKStageBytes;
        const unsigned char *abox = gbox + kKBoxBytes;
        const unsigned char *bbox = gbox + 2 * kKBoxBytes;
        const bool ok = mbar_wait_bounded(smem_u32(&bars[slot]), parity, kWaitLimitNs);
        const TileCoord tc = coords[slot];

        // ---- phase 1: da and db once, kept in fp32, and their column maxima over 4-row parts ----
        if (ok) {
            const int rb = warp >> 2, qt = warp & 3;
            const int cq = lane & 15, q = lane >> 4;
            const int r0 = rb * 32 + qt * 8 + q * 4;
            float fa[4] = {0.f, 0.f, 0.f, 0.f}, fb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = r0 + i;
                const int off = r * 128 + (((cq >> 1) ^ (r & 7)) << 4) + (cq & 1) * 8;
                const uint2 g = lds64(gbox + off), a = lds64(abox + off), b = lds64(bbox + off);
                uint64_t da01, db01, da23, db23;
                dgate2<ACT>(g.x, a.x, b.x, da01, db01);
                dgate2<ACT>(g.y, a.y, b.y, da23, db23);
                float va[4], vb[4];
                f2_unpack(da01, va[0], va[1]);
                f2_unpack(da23, va[2], va[3]);
                f2_unpack(db01, vb[0], vb[1]);
                f2_unpack(db23, vb[2], vb[3]);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    fa[k] = fmaxf(fa[k], fabsf(va[k]));
                    fb[k] = fmaxf(fb[k], fabsf(vb[k]));
                }
                const int kc = keep_chunk(cq, r) * 4;
                *reinterpret_cast<float4 *>(keep + r * kDBN + kc) = make_float4(va[0], va[1], va[2], va[3]);
                *reinterpret_cast<float4 *>(keep + (kKRows + r) * kDBN + kc) = make_float4(vb[0], vb[1], vb[2], vb[3]);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                fa[k] = fmaxf(fa[k], __shfl_xor_sync(0xffffffffu, fa[k], 16));
                fb[k] = fmaxf(fb[k], __shfl_xor_sync(0xffffffffu, fb[k], 16));
            }
            if (q == 0) {
                const int o = (qt * 2 + rb) * kDBN + cq * 4;
                *reinterpret_cast<float4 *>(part + o) = make_float4(fa[0], fa[1], fa[2], fa[3]);
                *reinterpret_cast<float4 *>(part + 4 * 2 * kDBN + o) = make_float4(fb[0], fb[1], fb[2], fb[3]);
            }
        }
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicOr(&g_fault_word, 1u);
                for (int j = it; j < my_count && j < it + kKStages; ++j)
                    mbar_wait_bounded(smem_u32(&bars[j % kKStages]), static_cast<uint32_t>(j / kKStages) & 1u,
                                      kDrainLimitNs);
            }
            return;
        }
        // the stage is read: phase 2 works from the keep area, so the next tile can land now
        if (tid == 0 && it + kKStages < my_count)
            issue(slot, first + (it + kKStages) * stride);

        // one thread per (output, 32-row block, column): the scale and the column multiplier
        {
            const int out = tid >> 7, rb = (tid >> 6) & 1, c = tid & 63;
            const float *pf = part + out * 4 * 2 * kDBN + rb * kDBN + c;
            const float amax = fmaxf(fmaxf(pf[0], pf[2 * kDBN]), fmaxf(pf[4 * kDBN], pf[6 * kDBN]));
            const int e = block_exponent_f32<FMT>(__float_as_uint(amax));
            const int64_t grow = tc.row0 + rb * 32, gcol = tc.col0 + c;
            if (do_col && grow < tc.row_end && gcol < N)
                p.scale_col[(grow >> 5) * N2 + out * N + gcol] = static_cast<uint8_t>(e);
            const int sp = c >> 4, qq = (c >> 2) & 3;  // rotated layout, as in the other kernels
            colmul[(out * 2 + rb) * kDBN + 4 * (4 * sp + ((qq + (sp >> 1)) & 3)) + (c & 3)] = scale_multiplier(e);
        }
        __syncthreads();

        // ---- phase 2: 16-column row segments of both outputs, from the keep area ----
        if (tc.row0 + warp * 8 < tc.row_end) {  // warp-uniform: the 8-row group exists
            const int rr = lane >> 2, sp = lane & 3;
            const int r = warp * 8 + rr;
            const int64_t grow = tc.row0 + r, gcol = tc.col0 + sp * 16;
            const bool in = grow < tc.row_end && gcol < N;
            const bool half = gcol + 16 > N;
#pragma unroll
            for (int out = 0; out < 2; ++out) {
                float y[16];
                const float *kr = keep + (out * kKRows + r) * kDBN;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 v = lds128f(kr + keep_chunk(4 * sp + j, r) * 4);
                    y[4 * j] = v.x;
                    y[4 * j + 1] = v.y;
                    y[4 * j + 2] = v.z;
                    y[4 * j + 3] = v.w;
                }
                if (do_row) {
                    float fm = 0.f;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        fm = fmaxf(fm, fabsf(y[i]));
                    fm = fmaxf(fm, __shfl_xor_sync(0xffffffffu, fm, 1));
                    const int er = block_exponent_f32<FMT>(__float_as_uint(fm));
                    const uint64_t rm = f2_splat(scale_multiplier(er));
                    uint32_t o[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        o[j] = cvt_fp8x2_scaled<FMT>(y[4 * j], y[4 * j + 1], rm) |
                               (cvt_fp8x2_scaled<FMT>(y[4 * j + 2], y[4 * j + 3], rm) << 16);
                    if (in) {
                        store_codes(p.out_row + grow * N2 + out * N + gcol, o[0], o[1], o[2], o[3], rows16, half);
                        if ((sp & 1) == 0)
                            p.scale_row[grow * 2 * Cn + out * Cn + (gcol >> 5)] = static_cast<uint8_t>(er);
                    }
                }
                if (do_col) {
                    const float *cm = colmul + (out * 2 + (r >> 5)) * kDBN + sp * 16;
                    uint32_t o[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 c = lds128f(cm + 4 * ((j + (sp >> 1)) & 3));
                        o[j] = cvt_fp8x2_scaled<FMT>(y[4 * j], y[4 * j + 1], f2_pack(c.x, c.y)) |
                               (cvt_fp8x2_scaled<FMT>(y[4 * j + 2], y[4 * j + 3], f2_pack(c.z, c.w)) << 16);
                    }
                    if (in)
                        store_codes(p.out_col + grow * N2 + out * N + gcol, o[0], o[1], o[2], o[3], rows16, half);
                }
            }
        }
        __syncthreads();  // the keep area and the multipliers are free for the next tile
    }
}

}  // namespace mxfp8
