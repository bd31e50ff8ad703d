// Backward fusion: the MXFP8 cast of dY * act'(X) (the `with_dact` field of
// the quantization config key on "[Common] Experimental CuTeDSL MXFP8
// backends in C++ via TVM-FFI", TransformerEngine PR #3137), with an optional
// fused dbias of the product.
//
// Two BF16 inputs per element, so a tile is 128 rows x 64 columns: each stage
// holds one 64-column TMA box of dY and one of X (16 KiB each, 128B swizzle),
// which keeps the 32 KiB stages and 2 CTAs per SM of the main kernel.
//   - phase 1: warp w takes rows 32*(w>>1) + 16*(w&1) .. +15 of the tile; a
//     lane takes 4 columns x 8 rows; the two 16-row halves of a 32-row block
//     meet in shared memory, where one thread per (row block, column) forms
//     the column's scale, multiplier and dbias partial.  Each fp32 product is
//     written back over its own two inputs (low half in the dY slot, high half
//     in the X slot: the same 4 bytes per element);
//   - phase 2: warp w takes the 8-row groups 2w and 2w + 1 (one 32-row block,
//     whose column multipliers it loads once per tile; dReLU: w and w + 8); a
//     lane takes 16 columns of one row, as in the main kernel, reading those
//     products back (one byte permute per element instead of a second
//     evaluation: measured faster for every activation, the ReLU family
//     included).
// The derivative is evaluated in fp32 with the same ex2 / rcp approximations
// as the forward activations; dReLU and dSReLU are exact.
//
// GATED: the same kernel casts a gated activation act(a) * b (ReGLU, squared-ReLU
// GLU, GeGLU, SwiGLU, QGeGLU) of an input x = [a | b], BF16 [M, 2N]: the dY slot
// holds the box of b (columns N.. of x), the X slot the box of a, and the forward
// activation takes the derivative's place.  No dbias.  GROUPED (gated only): the
// rows form groups, each quantized as its own flat problem, scheduled as in the
// grouped cast (no tile straddles two groups; a group's columnwise scale rows follow
// the previous group's); a partial last block leaves out the rows the tile loads
// past its group's end.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "ptx.cuh"
#include "quantize.cuh"

namespace mxfp8 {

constexpr int kDBN = 64;  // tile columns (one box per input)
constexpr int kDOffColMul = kStages * kStageBytes;         // float [4][64]
constexpr int kDOffDSum = kDOffColMul + 4 * kDBN * 4;      // float [4][64]
constexpr int kDOffPartF = kDOffDSum + 4 * kDBN * 4;       // float [2][4][64]
constexpr int kDOffPartD = kDOffPartF + 2 * 4 * kDBN * 4;  // float [2][4][64]
constexpr int kDOffBars = kDOffPartD + 2 * 4 * kDBN * 4;   // uint64 [kStages]
constexpr int kDOffCoord = kDOffBars + 8 * kStages;        // TileCoord [kStages]
constexpr int kSmemDact = kDOffCoord + 32 * kStages + 1024;
// grouped (gated cast only): the group schedule after the flat layout
constexpr int kDOffScan = kDOffCoord + 32 * kStages;                 // int64 [kThreads / 32]
constexpr int kDOffGOff = kDOffScan + 8 * (kThreads / 32);          // int64 [kMaxGroups + 1]
constexpr int kDOffGPre = kDOffGOff + 8 * (kMaxGroups + 1);         // int [kMaxGroups + 1]
constexpr int kDOffGSB = kDOffGPre + 4 * (kMaxGroups + 1);          // int [kMaxGroups + 1]
constexpr int kSmemDactGrouped = kDOffGSB + 4 * (kMaxGroups + 1) + 1024;

// Beyond |x| = 200 every derivative here is at its fp32 limit (1 for x > 0, -0 for
// x < 0).  The factors that overflow for huge |x| (x^2 in dGeLU's t', 1.702 x in
// dQGeLU) take x clamped there, or they would meet a zero factor (inf * 0 = NaN);
// dSiLU's x (1 - s) cannot overflow.
constexpr float kDactClamp = 200.f;

// dReLU and dSReLU in fp32 (exact).
template <int ACT>
__device__ __forceinline__ float dactivation(float x)
{
    static_assert(ACT == 1 || ACT == 2, "the transcendental derivatives are in dactivation2");
    if constexpr (ACT == 1)
        return x > 0.f ? 1.f : 0.f;
    else
        return x > 0.f ? 2.f * x : 0.f;
}

// act'(x) in fp32 for two values at once (lanes of a packed pair): 1 dReLU, 2 dSReLU
// (per lane, exact), 3 dGeLU (tanh form), 4 dSiLU, 5 dQGeLU (multiplies and adds as
// f32x2 operations, ex2 and rcp per lane).  sigmoid(t) = s and 1 - sigmoid(t) both come
// from h = 2^(-|t| log2(e) / 2), e = h h.  The derivative is s (1 + q) with
// q = x (1 - s) t', rather than s + x s (1 - s) t' (the sign of a tiny negative
// derivative survives), evaluated for t < 0 as (((1 + q) h) h) / (1 + e): multiplying
// 1 + q in before the second h keeps results that are fp32-subnormal where s alone would
// already have underflowed.
template <int ACT>
__device__ __forceinline__ uint64_t dactivation2(uint64_t x)
{
    float x0, x1;
    f2_unpack(x, x0, x1);
    if constexpr (ACT < 3) {
        return f2_pack(dactivation<ACT>(x0), dactivation<ACT>(x1));
    } else {
        const uint64_t one = f2_splat(1.f);
        float u0, u1, h0, h1;
        f2_unpack(half_log2e_arg2<ACT>(x), u0, u1);
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(h0) : "f"(-fabsf(u0)));
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(h1) : "f"(-fabsf(u1)));
        const float t0 = x0, t1 = x1;  // the sign tests only need sign(t) = sign(x)
        const uint64_t h = f2_pack(h0, h1);
        const uint64_t e = f2_mul(h, h);
        float o0, o1;
        f2_unpack(f2_add(e, one), o0, o1);
        const float i0 = rcp_1to2(o0), i1 = rcp_1to2(o1);
        float ei0, ei1;
        f2_unpack(f2_mul(e, f2_pack(i0, i1)), ei0, ei1);
        const uint64_t oms = f2_pack(t0 >= 0.f ? ei0 : i0, t1 >= 0.f ? ei1 : i1);
        uint64_t inner;
        if constexpr (ACT == 3) {
            const uint64_t xc = f2_pack(fminf(fmaxf(x0, -kDactClamp), kDactClamp),
                                        fminf(fmaxf(x1, -kDactClamp), kDactClamp));
            const uint64_t q = f2_mul(f2_splat(0.134145f), xc);
            const uint64_t tp = f2_mul(f2_splat(kGeluC0), f2_fma(q, xc, one));
            inner = f2_fma(f2_mul(xc, oms), tp, one);
        } else if constexpr (ACT == 4) {
            inner = f2_fma(x, oms, one);
        } else {
            const uint64_t xc = f2_pack(fminf(fmaxf(x0, -kDactClamp), kDactClamp),
                                        fminf(fmaxf(x1, -kDactClamp), kDactClamp));
            inner = f2_fma(f2_mul(f2_splat(1.702f), xc), oms, one);
        }
        const uint64_t a = f2_pack(t0 >= 0.f ? 1.f : h0, t1 >= 0.f ? 1.f : h1);
        return f2_mul(f2_mul(f2_mul(inner, a), a), f2_pack(i0, i1));
    }
}

template <int FMT, bool DBIAS, int ACT, bool GATED = false, bool GROUPED = false>
__global__ void __launch_bounds__(kThreads, 2)
    quantize_dact_kernel(const __grid_constant__ CUtensorMap tmap_g, const __grid_constant__ CUtensorMap tmap_x,
                         const QuantParams p)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *colmul = reinterpret_cast<float *>(smem + kDOffColMul);
    float *dsum = reinterpret_cast<float *>(smem + kDOffDSum);
    float *part_f = reinterpret_cast<float *>(smem + kDOffPartF);
    float *part_d = reinterpret_cast<float *>(smem + kDOffPartD);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kDOffBars);
    TileCoord *coords = reinterpret_cast<TileCoord *>(smem + kDOffCoord);

    static_assert(!(GATED && DBIAS), "the gated cast has no dbias");
    static_assert(!GROUPED || GATED, "the grouped two-input kernel is the gated cast");
    // act'(x) for the backward fusion, act(x) for the gated cast (two lanes)
    auto factor2 = [](uint64_t x) -> uint64_t {
        if constexpr (GATED)
            return activation2<ACT>(x);
        else
            return dactivation2<ACT>(x);
    };
    pdl_wait_and_release();
    if (p.noop != nullptr && *p.noop == 1.0f)
        return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t N = p.N;
    int64_t *goff = reinterpret_cast<int64_t *>(smem + kDOffGOff);
    int *gpre = reinterpret_cast<int *>(smem + kDOffGPre);
    int *gsb = reinterpret_cast<int *>(smem + kDOffGSB);
    int num_tiles;
    bool by_group = false;  // grouped schedule; with every offset a multiple of 32 the flat one
    if constexpr (GROUPED) {
        num_tiles = grouped_setup(p, goff, gpre, gsb, reinterpret_cast<int64_t *>(smem + kDOffScan));
        if (num_tiles < 0) {
            if (blockIdx.x == 0 && tid == 0 && p.err_flag != nullptr)
                atomicOr(p.err_flag, 1);
            return;
        }
        // With every group a whole number of 32-row blocks no block crosses a group and the
        // flat call on the concatenated rows writes the same bytes (scale_col row = row / 32):
        // flat 128-row tiles then skip the groups' partial last tiles.
        int unaligned = 0;
        for (int g = tid; g <= p.num_groups; g += kThreads)
            unaligned |= (goff[g] & 31) != 0;
        by_group = __syncthreads_or(unaligned) != 0;
        if (!by_group)
            num_tiles = p.row_tiles * p.col_tiles;
    } else {
        num_tiles = p.row_tiles * p.col_tiles;
    }
    const int first = blockIdx.x, stride = gridDim.x;
    const int my_count = first < num_tiles ? (num_tiles - 1 - first) / stride + 1 : 0;
    if (my_count == 0)
        return;
    const bool do_row = p.out_row != nullptr, do_col = p.out_col != nullptr;
    const bool rows16 = (N & 15) == 0;  // FP8 rows 16-byte aligned (else N % 16 == 8: 8-byte)

    if (tid == 0) {
        prefetch_tensormap(&tmap_g);
        prefetch_tensormap(&tmap_x);
        for (int s = 0; s < kStages; ++s)
            mbar_init(smem_u32(&bars[s]), 1);
        fence_mbar_init();
    }
    __syncthreads();

    auto issue = [&](int slot, int t) {
        TileCoord c;
        if (GROUPED && by_group) {
            c = tile_coord<true, kDBN>(t, p, goff, gpre, gsb);
        } else {
            const int rt = t / p.col_tiles, ct = t - rt * p.col_tiles;
            c.row0 = static_cast<int64_t>(rt) * kBM;
            c.row_end = min(c.row0 + kBM, p.M);
            c.col0 = ct * kDBN;
            c.rt = rt;
            c.sb = rt * (kBM / 32);
            c.g = 0;
        }
        coords[slot] = c;  // published to the consumers by the arrive below
        const uint32_t bar = smem_u32(&bars[slot]);
        const uint32_t dst = smem_u32(smem + slot * kStageBytes);
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, kStageBytes);
        tma_load_2d(dst, &tmap_g, bar, c.col0, static_cast<int32_t>(c.row0));
        tma_load_2d(dst + kBoxBytes, &tmap_x, bar, c.col0, static_cast<int32_t>(c.row0));
    };
    if (tid == 0)
        for (int s = 0; s < kStages && s < my_count; ++s)
            issue(s, first + s * stride);

    for (int it = 0; it < my_count; ++it) {
        const int slot = it % kStages;
        const uint32_t parity = static_cast<uint32_t>(it / kStages) & 1u;
        unsigned char *gbox = smem + slot * kStageBytes;
        unsigned char *xbox = gbox + kBoxBytes;
        const bool ok = mbar_wait_bounded(smem_u32(&bars[slot]), parity, kWaitLimitNs);
        const TileCoord tc = coords[slot];

        // ---- phase 1: column amax / sums over 16-row halves ----
        if (ok) {
            const int rb = warp >> 1, hh = warp & 1;
            const int cq = lane & 15, q = lane >> 4;
            const int r0 = rb * 32 + hh * 16 + q * 8;  // r0 & 7 == 0
            // rows of this lane's 8 that belong to the tile's group (grouped schedule)
            const int64_t left = tc.row_end - (tc.row0 + r0);
            const int live = left < 8 ? static_cast<int>(left) : 8;
            float f[4] = {0.f, 0.f, 0.f, 0.f}, d[4] = {0.f, 0.f, 0.f, 0.f};
            uint64_t d01 = 0, d23 = 0;  // packed column sums (+0.0 in both lanes)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int off = (r0 + i) * 128 + (((cq >> 1) ^ i) << 4) + (cq & 1) * 8;
                uint2 g = lds64(gbox + off);
                const uint2 xv = lds64(xbox + off);
                if (GROUPED && i >= live) {
                    g.x = 0u;  // a row after the group's end (the next group's): its products are +-0
                    g.y = 0u;
                }
                const uint64_t y01 = f2_mul(f2_pack(bf16_lo(g.x), bf16_hi(g.x)),
                                            factor2(f2_pack(bf16_lo(xv.x), bf16_hi(xv.x))));
                const uint64_t y23 = f2_mul(f2_pack(bf16_lo(g.y), bf16_hi(g.y)),
                                            factor2(f2_pack(bf16_lo(xv.y), bf16_hi(xv.y))));
                float y0, y1, y2, y3;
                f2_unpack(y01, y0, y1);
                f2_unpack(y23, y2, y3);
                f[0] = fmaxf(f[0], fabsf(y0));
                f[1] = fmaxf(f[1], fabsf(y1));
                f[2] = fmaxf(f[2], fabsf(y2));
                f[3] = fmaxf(f[3], fabsf(y3));
                if constexpr (DBIAS) {
                    d01 = f2_add(d01, y01);
                    d23 = f2_add(d23, y23);
                }
                {  // keep the products for phase 2 (see the top)
                    const uint32_t b0 = __float_as_uint(y0), b1 = __float_as_uint(y1);
                    const uint32_t b2 = __float_as_uint(y2), b3 = __float_as_uint(y3);
                    sts64(gbox + off, __byte_perm(b0, b1, 0x5410), __byte_perm(b2, b3, 0x5410));
                    sts64(xbox + off, __byte_perm(b0, b1, 0x7632), __byte_perm(b2, b3, 0x7632));
                }
            }
            fence_proxy_async_smem();  // these generic writes precede the stage's next TMA fill
            if constexpr (DBIAS) {
                f2_unpack(d01, d[0], d[1]);
                f2_unpack(d23, d[2], d[3]);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                f[k] = fmaxf(f[k], __shfl_xor_sync(0xffffffffu, f[k], 16));
                if constexpr (DBIAS)
                    d[k] += __shfl_xor_sync(0xffffffffu, d[k], 16);  // a + b == b + a
            }
            if (q == 0) {
                const int o = (hh * 4 + rb) * kDBN + cq * 4;
                *reinterpret_cast<float4 *>(part_f + o) = make_float4(f[0], f[1], f[2], f[3]);
                if constexpr (DBIAS)
                    *reinterpret_cast<float4 *>(part_d + o) = make_float4(d[0], d[1], d[2], d[3]);
            }
        }
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicOr(&g_fault_word, 1u);
                if (GROUPED && p.err_flag != nullptr)
                    atomicOr(p.err_flag, 2);
                for (int j = it; j < my_count && j < it + kStages; ++j)
                    mbar_wait_bounded(smem_u32(&bars[j % kStages]), static_cast<uint32_t>(j / kStages) & 1u,
                                      kDrainLimitNs);
            }
            return;
        }
        // one thread per (32-row block, column): scale, multiplier, dbias partial
        {
            const int rb = tid >> 6, c = tid & 63;
            const float amax = fmaxf(part_f[rb * kDBN + c], part_f[(4 + rb) * kDBN + c]);
            const int e = block_exponent_f32<FMT>(__float_as_uint(amax));
            const int64_t grow = tc.row0 + rb * 32, gcol = tc.col0 + c;
            if (do_col && grow < tc.row_end && gcol < N)
                p.scale_col[(GROUPED ? static_cast<int64_t>(tc.sb + rb) : grow >> 5) * N + gcol] =
                    static_cast<uint8_t>(e);
            const int sp = c >> 4, qq = (c >> 2) & 3;  // rotated layout, as in the main kernel
            colmul[rb * kDBN + 4 * (4 * sp + ((qq + (sp >> 1)) & 3)) + (c & 3)] = scale_multiplier(e);
            if constexpr (DBIAS)
                dsum[rb * kDBN + c] = grow < tc.row_end ? part_d[rb * kDBN + c] + part_d[(4 + rb) * kDBN + c] : 0.f;
        }
        __syncthreads();
        if constexpr (DBIAS) {
            if (tid < kDBN) {
                const int64_t gcol = tc.col0 + tid;
                if (gcol < N)
                    p.ws[static_cast<int64_t>(tc.rt) * N + gcol] =
                        ((dsum[tid] + dsum[kDBN + tid]) + dsum[2 * kDBN + tid]) + dsum[3 * kDBN + tid];
            }
        }

        // ---- phase 2: 16-column row segments ----
        {
            const int rr = lane >> 2, sp = lane & 3;
            // Except for dReLU (bound by memory: measured slower so), a warp's two tasks are
            // adjacent 8-row groups of one 32-row block, whose 16 column multipliers the lane
            // loads once per tile; dReLU's tasks step through the row blocks.
            constexpr bool kReuse = ACT >= 2;
            float4 cmv[4];
            if (kReuse && do_col) {
                const float *cm0 = colmul + (warp >> 1) * kDBN + sp * 16;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    cmv[j] = lds128f(cm0 + 4 * ((j + (sp >> 1)) & 3));
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int rg = kReuse ? 2 * warp + k : warp + 8 * k;
                if (tc.row0 + rg * 8 >= tc.row_end)
                    continue;
                const int r = rg * 8 + rr;
                const int p0 = (2 * sp) ^ rr;
                const uint4 GA = lds128(gbox + r * 128 + p0 * 16), GB = lds128(gbox + r * 128 + (p0 ^ 1) * 16);
                const uint4 XA = lds128(xbox + r * 128 + p0 * 16), XB = lds128(xbox + r * 128 + (p0 ^ 1) * 16);
                const uint32_t gw[8] = {GA.x, GA.y, GA.z, GA.w, GB.x, GB.y, GB.z, GB.w};
                const uint32_t xw[8] = {XA.x, XA.y, XA.z, XA.w, XB.x, XB.y, XB.z, XB.w};
                float y[16];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    // the products phase 1 left in the two slots
                    y[2 * j] = __uint_as_float(__byte_perm(gw[j], xw[j], 0x5410));
                    y[2 * j + 1] = __uint_as_float(__byte_perm(gw[j], xw[j], 0x7632));
                }
                const int64_t grow = tc.row0 + r, gcol = tc.col0 + sp * 16;
                const bool in = grow < tc.row_end && gcol < N;
                // two codes from two values and their multipliers (one f32x2 multiply)
                auto cvt_pair = [](float a, float b, float ma, float mb) -> uint32_t {
                    return cvt_fp8x2_scaled<FMT>(a, b, f2_pack(ma, mb));
                };
                if (do_row) {
                    float fm = 0.f;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        fm = fmaxf(fm, fabsf(y[i]));
                    fm = fmaxf(fm, __shfl_xor_sync(0xffffffffu, fm, 1));
                    const int er = block_exponent_f32<FMT>(__float_as_uint(fm));
                    const float rm = scale_multiplier(er);
                    uint32_t o[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        o[j] = cvt_pair(y[4 * j], y[4 * j + 1], rm, rm) |
                               (cvt_pair(y[4 * j + 2], y[4 * j + 3], rm, rm) << 16);
                    if (in) {
                        store_codes(p.out_row + grow * N + gcol, o[0], o[1], o[2], o[3], rows16, gcol + 16 > N);
                        if ((sp & 1) == 0)
                            p.scale_row[grow * ((N + 31) >> 5) + (gcol >> 5)] = static_cast<uint8_t>(er);
                    }
                }
                if (do_col) {
                    const float *cm = colmul + (r >> 5) * kDBN + sp * 16;
                    uint32_t o[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 c = kReuse ? cmv[j] : lds128f(cm + 4 * ((j + (sp >> 1)) & 3));
                        o[j] = cvt_pair(y[4 * j], y[4 * j + 1], c.x, c.y) |
                               (cvt_pair(y[4 * j + 2], y[4 * j + 3], c.z, c.w) << 16);
                    }
                    if (in)
                        store_codes(p.out_col + grow * N + gcol, o[0], o[1], o[2], o[3], rows16, gcol + 16 > N);
                }
            }
        }
        __syncthreads();  // stage, colmul and dsum are free again
        if (tid == 0 && it + kStages < my_count)
            issue(slot, first + (it + kStages) * stride);
    }
}

}  // namespace mxfp8
