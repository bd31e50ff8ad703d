// MXFP8 block-scaled quantize kernels for sm_103a (GB300).
//
// One pass over HBM: every BF16 element is read once (TMA, 128x128 tiles)
// and produces a rowwise FP8 byte (1x32 block along the row) and a
// columnwise FP8 byte (32x1 block down the column), plus the two E8M0 scale
// planes and, optionally, fp32 per-tile column partials for dbias.
//
// The operation is the MXFP8 cast of "[Common] Experimental CuTeDSL MXFP8
// backends in C++ via TVM-FFI" (TransformerEngine PR #3137): rowwise /
// colwise / with_dbias / with_noop config fields, 32-element blocks.
//
// Per block, amax is taken on the BF16 bit patterns (|x| ordering equals the
// integer ordering of bits & 0x7FFF for finite values) and the E8M0 exponent
//     e = clamp(ceil(log2(amax / Fmax)) + 127, 0, 254),  amax == 0 -> 127
// is computed exactly in integers: for a normal amax = (1 + m/128) 2^(E-127)
// with Fmax = 1.75 * 2^emax, ceil(log2(amax/Fmax)) = E - 127 - emax + [m > 96];
// a subnormal amax always clamps to e = 0.  Each element is then multiplied
// by 2^(127 - e) in fp32 (exact: BF16 has 8 significant bits, the factor is a
// power of two and subnormals are kept) and converted with
// cvt.rn.satfinite.{e4m3x2,e5m2x2}.f32.
//
// Tile pipeline (per CTA, persistent over a static round-robin tile list):
//   - thread 0 keeps STAGES tiles in flight: two 64-column TMA boxes per
//     128x128 tile, 128B-swizzled, completion on one mbarrier per stage;
//   - phase 1 (all 8 warps): column amax of the four 32-row blocks, read as
//     conflict-free 8-byte shared loads; writes scale_col and the fp32 column
//     multipliers (and dbias partial sums) to shared memory;
//   - phase 2 (all 8 warps): each thread takes 16 consecutive columns of one
//     row (two 16-byte shared loads), does the rowwise amax with one shuffle,
//     converts the 16 values twice (row multiplier, 16 column multipliers)
//     and writes two 16-byte global stores.
// Every wait on an mbarrier is bounded; on expiry the CTA records a fault,
// drains its own copies (again bounded) and returns.  The kernel is launched
// for programmatic dependent launch: it waits for the previous kernel on the
// stream to finish before its first global access and lets the next one start
// launching at once (pdl_wait_and_release).
#pragma once

#include <cstdint>
#include <cuda.h>

#include "ptx.cuh"

namespace mxfp8 {

constexpr int kBM = 128;                      // tile rows
constexpr int kBN = 128;                      // tile columns
constexpr int kBoxCols = 64;                  // TMA box width (128 bytes of BF16)
constexpr int kBoxBytes = kBM * kBoxCols * 2; // 16 KiB
constexpr int kStageBytes = 2 * kBoxBytes;    // 32 KiB
constexpr int kStages = 3;
constexpr int kThreads = 256;
constexpr int kMaxGroups = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr uint64_t kDrainLimitNs = 200000000ull;  // 0.2 s

// Shared-memory layout (bytes from a 1024-aligned base).
constexpr int kOffColMul = kStages * kStageBytes;      // float [4][128]
constexpr int kOffDSum = kOffColMul + 4 * kBN * 4;     // float [4][128]
constexpr int kOffBars = kOffDSum + 4 * kBN * 4;       // uint64 [kStages]
constexpr int kOffCoord = kOffBars + 8 * kStages;      // TileCoord [kStages]
constexpr int kOffScan = kOffCoord + 32 * kStages;     // int64 [kThreads / 32]
constexpr int kOffRowSc = kOffScan + 8 * (kThreads / 32);  // uint32 [kBM]: a tile's row scales
constexpr int kOffGOff = kOffRowSc + 4 * kBM;              // int64 [kMaxGroups + 1]
constexpr int kOffGPre = kOffGOff + 8 * (kMaxGroups + 1);  // int [kMaxGroups + 1]
constexpr int kOffGSB = kOffGPre + 4 * (kMaxGroups + 1);   // int [kMaxGroups + 1]
constexpr int kSmemFlat = kOffGOff + 1024;                 // + alignment slack
constexpr int kSmemGrouped = kOffGSB + 4 * (kMaxGroups + 1) + 1024;

struct QuantParams {
    uint8_t *out_row;
    uint8_t *scale_row;
    uint8_t *out_col;
    uint8_t *scale_col;
    float *ws;               // dbias partials [row_tiles][N], or nullptr
    const float *noop;       // device scalar or nullptr
    const int64_t *offsets;  // grouped: [num_groups + 1]
    int *err_flag;           // grouped: device flag or nullptr
    int64_t M;               // rows (total rows when grouped)
    int64_t N;
    int num_groups;
    int col_tiles;
    int row_tiles;           // flat only
    float *amax;             // per-tensor max |x| (device fp32, zeroed before the launch), AMAX variant
    int64_t *ws_hdr;         // grouped dbias: [num_groups + 1] first row tile of each group (-1: bad offsets)
};

// GEMM-ready layout: a scale matrix stored as 128-row x 4-column tiles of 512 bytes,
// row-tile major, entry (r, c) of a tile at 16 * (r % 32) + 4 * (r / 32) + c.  The
// byte of entry (r, c) within its tile (0 <= r < 128, 0 <= c < 4):
__device__ __forceinline__ int swizzled_in_tile(int r, int c)
{
    return ((r & 31) << 4) | (((r >> 5) & 3) << 2) | c;
}

// Library-wide device fault word (bit 0: a bounded wait expired).
__device__ unsigned int g_fault_word;

template <int FMT>
__device__ __forceinline__ int block_exponent(uint32_t amax_bits)
{
    constexpr int kEmax = FMT == 0 ? 8 : 15;
    int e = static_cast<int>(amax_bits >> 7) - kEmax + ((amax_bits & 0x7Fu) > 0x60u ? 1 : 0);
    e = e < 0 ? 0 : e;
    return amax_bits == 0 ? 127 : e;
}

// Same rule for an fp32 amax (the activated path): amax = (1 + m/2^23) 2^(E-127),
// ceil(log2(amax/Fmax)) = E - 127 - emax + [m > 0.75 * 2^23]; subnormal -> 0.
template <int FMT>
__device__ __forceinline__ int block_exponent_f32(uint32_t amax_bits)
{
    constexpr int kEmax = FMT == 0 ? 8 : 15;
    int e = static_cast<int>(amax_bits >> 23) - kEmax + ((amax_bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    e = e < 0 ? 0 : e;
    return amax_bits == 0 ? 127 : e;
}

// Activation applied to each input before the cast (fp32): 1 ReLU, 2 squared
// ReLU, 3 GeLU (tanh form, as x * sigmoid(2 sqrt(2/pi) (x + 0.044715 x^3))),
// 4 SiLU, 5 QGeLU (x * sigmoid(1.702 x)).  The sigmoid is 1 / (1 + e) or
// e / (1 + e) with e = 2^(-|t| log2 e): no overflow and no cancellation for
// large |t|.  It uses the hardware ex2 / rcp approximations in their
// flush-to-zero forms (a few ulps), which the parity tests allow for at decision
// boundaries.  e is formed as h h, h = 2^(z/2) from one bare ex2 (normal wherever
// e is within fp32's range); the reciprocal only ever sees 1 + e in [1, 2]; and
// for t < 0 the input is multiplied in between the two factors h, so that results
// in fp32's subnormal range come out as any fp32 product would give them.  (A
// guarded single ex2 -- 2^(z + 64) * 2^-64 for z < -64 -- costs six instructions
// instead of two; the activations measured 10-14% faster with the square, the
// derivatives 3-4%.)

// log2(e) / 2: the ex2 argument is z / 2 = -|t| log2(e) / 2.
constexpr float kHalfLog2e = 0.72134752044448170f;

// 1 / x for x in [1, 2].
__device__ __forceinline__ float rcp_1to2(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The sigmoid's argument t for GeLU (2 sqrt(2/pi) (x + 0.044715 x^3)), SiLU (x) and
// QGeLU (1.702 x), formed directly as u = t log2(e) / 2 with the constants folded in
// (GeLU: x (k c0 + k c1 x^2)).  t, and so u, has the sign of x for all three.
constexpr float kGeluC0 = 1.5957691216057308f;           // 2 sqrt(2/pi)
constexpr float kGeluC1 = 1.5957691216057308f * 0.044715f;
template <int ACT>
__device__ __forceinline__ uint64_t half_log2e_arg2(uint64_t x)
{
    if constexpr (ACT == 3)
        return f2_mul(x, f2_fma(f2_mul(x, x), f2_splat(kHalfLog2e * kGeluC1), f2_splat(kHalfLog2e * kGeluC0)));
    else if constexpr (ACT == 4)
        return f2_mul(f2_splat(kHalfLog2e), x);
    else
        return f2_mul(f2_splat(kHalfLog2e * 1.702f), x);
}

// ReLU and squared ReLU (exact in fp32).
template <int ACT>
__device__ __forceinline__ float relu_family(float x)
{
    if constexpr (ACT == 1)
        return x > 0.f ? x : 0.f;
    else
        return x > 0.f ? x * x : 0.f;
}

// The activations on two values at once (lanes lo and hi of a packed pair): the
// multiplies and adds run as f32x2 operations, ex2 and rcp per lane.  This is the
// only evaluation of the activations in the kernels (phase 1's column maxima and
// phase 2's elements both come from here), so every value a scale or a code is
// formed from is the same function of the BF16 input.
template <int ACT>
__device__ __forceinline__ uint64_t activation2(uint64_t x)
{
    float x0, x1;
    f2_unpack(x, x0, x1);
    if constexpr (ACT <= 2) {
        return f2_pack(relu_family<ACT>(x0), relu_family<ACT>(x1));
    } else {
        float u0, u1, h0, h1;
        f2_unpack(half_log2e_arg2<ACT>(x), u0, u1);
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(h0) : "f"(-fabsf(u0)));  // h = 2^(-|t| log2(e) / 2)
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(h1) : "f"(-fabsf(u1)));
        const uint64_t h = f2_pack(h0, h1);
        const uint64_t e = f2_mul(h, h);
        float o0, o1;
        f2_unpack(f2_add(e, f2_splat(1.f)), o0, o1);
        const float r0 = rcp_1to2(o0), r1 = rcp_1to2(o1);
        // x sigmoid(t) = x r for t >= 0 and ((x h) h) r for t < 0: multiplying x in
        // before the second h keeps results that are fp32-subnormal where e = h h
        // alone would already have underflowed (SiLU(-104) = -7e-44, for one)
        const uint64_t a = f2_pack(x0 >= 0.f ? 1.f : h0, x1 >= 0.f ? 1.f : h1);  // t >= 0 iff x >= 0
        return f2_mul(f2_mul(f2_mul(x, a), a), f2_pack(r0, r1));
    }
}

// Largest |act(x)| over x <= 0 (the activations above are monotone increasing for
// x > 0, and bounded in magnitude by this for x <= 0): SiLU's minimum is
// -0.2785 at x = -1.278; GeLU's and QGeLU's are smaller; ReLU's is 0.
template <int ACT>
__device__ __forceinline__ float negative_side_bound()
{
    return ACT <= 2 ? 0.f : 0.2785f * 1.01f;
}

// One step of a per-lane |x| maximum over BF16 bit pairs, and its final
// magnitudes.  XS: max.xorsign.abs.bf16x2, one instruction (measured faster in
// the grouped and dbias variants); else the integer form on bits & 0x7FFF
// (measured faster in the plain cast, notably on L2-resident inputs).
template <bool XS>
__device__ __forceinline__ uint32_t absmax_step(uint32_t m, uint32_t v)
{
    if constexpr (XS)
        return absmax_bf16x2(m, v);
    else
        return max_u16x2(m, v & 0x7FFF7FFFu);
}
template <bool XS>
__device__ __forceinline__ uint32_t absmax_done(uint32_t m)
{
    return XS ? m & 0x7FFF7FFFu : m;
}

// 2^(127 - e) as fp32, for 0 <= e <= 253.
__device__ __forceinline__ float scale_multiplier(int e)
{
    return __uint_as_float(static_cast<uint32_t>(254 - e) << 23);
}

struct TileCoord {
    int64_t row0;     // first row of the tile
    int64_t row_end;  // one past the last row that belongs to the tile
    int col0;
    int rt;           // flat row-tile index (dbias partial row)
    int sb;           // columnwise scale row of the tile's first 32-row block
    int g;            // the tile's group (0 for a flat call)
};
static_assert(sizeof(TileCoord) <= 32, "coordinate slot");

// Tile t's coordinates; BN is the tile's width in columns.
template <bool GROUPED, int BN = kBN>
__device__ __forceinline__ TileCoord tile_coord(int t, const QuantParams &p, const int64_t *goff,
                                                const int *gpre, const int *gsb)
{
    TileCoord c;
    if constexpr (GROUPED) {
        int lo = 0, hi = p.num_groups;  // gpre[lo] <= t < gpre[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (gpre[mid] <= t)
                lo = mid;
            else
                hi = mid;
        }
        const int local = t - gpre[lo];
        const int rtl = local / p.col_tiles;
        const int ct = local - rtl * p.col_tiles;
        c.row0 = goff[lo] + static_cast<int64_t>(rtl) * kBM;
        c.row_end = min(c.row0 + kBM, goff[lo + 1]);
        c.col0 = ct * BN;
        c.rt = gpre[lo] / p.col_tiles + rtl;  // global row-tile index (per-group dbias partial row)
        c.sb = gsb[lo] + rtl * (kBM / 32);     // the group's scale rows follow the groups before it
        c.g = lo;
    } else {
        const int rt = t / p.col_tiles;
        const int ct = t - rt * p.col_tiles;
        c.row0 = static_cast<int64_t>(rt) * kBM;
        c.row_end = min(c.row0 + kBM, p.M);
        c.col0 = ct * BN;
        c.rt = rt;
        c.sb = rt * (kBM / 32);
        c.g = 0;
    }
    return c;
}

// Grouped set-up: load and check the offsets, build the per-group prefixes of
// row tiles (gpre, in tiles of all column tiles) and of columnwise scale rows
// (gsb) in shared memory.  Returns the tile count, or -1 for bad offsets.
// Both prefixes come from one exclusive scan of a packed count (tiles in the
// high 32 bits, scale rows in the low: the low sum stays below 2^32, so it never
// carries); thread t counts groups 2t and 2t+1 (kMaxGroups == 2 * kThreads).
__device__ __forceinline__ int grouped_setup(const QuantParams &p, int64_t *goff, int *gpre, int *gsb,
                                             int64_t *scan)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = p.num_groups;
    for (int g = tid; g <= G; g += kThreads)
        goff[g] = p.offsets[g];
    __syncthreads();
    int bad = 0;
    for (int g = tid; g < G; g += kThreads)
        if (goff[g + 1] < goff[g])
            bad = 1;
    if (tid == 0 && (goff[0] != 0 || goff[G] != p.M))
        bad = 1;
    if (__syncthreads_or(bad))
        return -1;
    // a group of rows_g rows: ceil(rows_g / 128) row tiles (times the column tiles) and
    // ceil(rows_g / 32) columnwise scale rows
    int64_t c[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int g = 2 * tid + k;
        c[k] = 0;
        if (g < G) {
            const int64_t rows = goff[g + 1] - goff[g];
            c[k] = (((rows + kBM - 1) / kBM * p.col_tiles) << 32) + (rows + 31) / 32;
        }
    }
    int64_t incl = c[0] + c[1];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int64_t v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d)
            incl += v;
    }
    if (lane == 31)
        scan[warp] = incl;
    __syncthreads();
    int64_t base = 0, total = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
        base += w < warp ? scan[w] : 0;
        total += scan[w];
    }
    const int64_t e0 = base + incl - (c[0] + c[1]), e1 = e0 + c[0];
    if (2 * tid < G) {
        gpre[2 * tid] = static_cast<int>(e0 >> 32);
        gsb[2 * tid] = static_cast<int>(e0 & 0xFFFFFFFF);
    }
    if (2 * tid + 1 < G) {
        gpre[2 * tid + 1] = static_cast<int>(e1 >> 32);
        gsb[2 * tid + 1] = static_cast<int>(e1 & 0xFFFFFFFF);
    }
    if (tid == 0) {
        gpre[G] = static_cast<int>(total >> 32);
        gsb[G] = static_cast<int>(total & 0xFFFFFFFF);
    }
    __syncthreads();
    return static_cast<int>(total >> 32);
}

// SWZ: scale planes in the GEMM-ready layout; AMAX: also produce max |x|; ACT: an
// activation applied before the cast (0 = none).  All are template switches so the
// default variant carries no code for them.
template <int FMT, bool DBIAS, bool GROUPED, bool SWZ, bool AMAX, int ACT = 0>
__global__ void __launch_bounds__(kThreads, 2)
    quantize_kernel(const __grid_constant__ CUtensorMap tmap, const QuantParams p)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *colmul = reinterpret_cast<float *>(smem + kOffColMul);
    float *dsum = reinterpret_cast<float *>(smem + kOffDSum);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBars);
    TileCoord *coords = reinterpret_cast<TileCoord *>(smem + kOffCoord);
    int64_t *scan = reinterpret_cast<int64_t *>(smem + kOffScan);
    int64_t *goff = reinterpret_cast<int64_t *>(smem + kOffGOff);
    int *gpre = reinterpret_cast<int *>(smem + kOffGPre);
    int *gsb = reinterpret_cast<int *>(smem + kOffGSB);
    // warp-local: [kStages] warps done with a stage (in the scan's space, which the grouped
    // set-up has finished with before the counters are reset)
    unsigned *stage_done = reinterpret_cast<unsigned *>(smem + kOffScan);
    uint32_t *rowsc = reinterpret_cast<uint32_t *>(smem + kOffRowSc);

    constexpr bool kXS = GROUPED || DBIAS;  // form of the BF16 |x| maximum (absmax_step)
    // With a transcendental activation (bound on the SM side) a warp's phase-2 tasks are the
    // 8-row groups of the (32-row block, box) it handles in phase 1, so phase 2 reads only
    // shared data its own warp wrote: a warp barrier replaces the CTA barrier between the
    // phases, the lane's 16 column multipliers are loaded once per tile, and no CTA barrier
    // closes the tile either (the last warp done with a stage refills it): all measured
    // faster there.  Without one (bound by memory) the tasks step through the row blocks and
    // CTA barriers pace the tile: the order of the stores that measured fastest.
    constexpr bool kWarpLocal = ACT > 2;
    static_assert(!(kWarpLocal && DBIAS), "warp-local phases: casts without dbias");
    pdl_wait_and_release();
    if (p.noop != nullptr && *p.noop == 1.0f)
        return;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t N = p.N;

    int num_tiles;
    bool by_group = GROUPED;  // the grouped schedule (else the flat one)
    if constexpr (GROUPED) {
        num_tiles = grouped_setup(p, goff, gpre, gsb, scan);
        if (num_tiles < 0) {
            if (blockIdx.x == 0 && tid == 0) {
                if (p.err_flag != nullptr)
                    atomicOr(p.err_flag, 1);
                if (DBIAS)
                    p.ws_hdr[0] = -1;  // tells the dbias reduce to write nothing
            }
            return;
        }
        if (DBIAS && blockIdx.x == 0) {
            // each group's first row tile in the partials (and the total), for the dbias reduce
            for (int g = tid; g <= p.num_groups; g += kThreads)
                p.ws_hdr[g] = gpre[g] / p.col_tiles;
        }
        if constexpr (ACT != 0 && !SWZ) {
            // With every group a whole number of 32-row blocks the flat cast of the
            // concatenated rows writes the same bytes: flat tiles then skip the groups'
            // partial last tiles (measured faster for the activated casts only).
            int unaligned = 0;
            for (int g = tid; g <= p.num_groups; g += kThreads)
                unaligned |= (goff[g] & 31) != 0;
            if (!__syncthreads_or(unaligned)) {
                by_group = false;
                num_tiles = p.row_tiles * p.col_tiles;
            }
        }
    } else {
        num_tiles = p.row_tiles * p.col_tiles;
    }
    const int first = blockIdx.x, stride = gridDim.x;
    const int my_count = first < num_tiles ? (num_tiles - 1 - first) / stride + 1 : 0;
    if (my_count == 0)
        return;

    const bool do_row = p.out_row != nullptr;
    const bool do_col = p.out_col != nullptr;
    const bool rows16 = (N & 15) == 0;  // FP8 rows 16-byte aligned (else N % 16 == 8: 8-byte)

    if (tid == 0) {
        prefetch_tensormap(&tmap);
        for (int s = 0; s < kStages; ++s)
            mbar_init(smem_u32(&bars[s]), 1);
        fence_mbar_init();
        if constexpr (kWarpLocal)
            for (int s = 0; s < kStages; ++s)
                stage_done[s] = 0;
    }
    __syncthreads();

    auto issue = [&](int slot, int t) {
        const TileCoord c = by_group ? tile_coord<true>(t, p, goff, gpre, gsb) : tile_coord<false>(t, p, goff, gpre, gsb);
        coords[slot] = c;  // published to the consumers by the arrive below
        const uint32_t bar = smem_u32(&bars[slot]);
        const uint32_t dst = smem_u32(smem + slot * kStageBytes);
        const bool second = c.col0 + kBoxCols < N;  // skip a box that lies wholly past column N
        mbar_arrive_expect_tx(bar, second ? kStageBytes : kBoxBytes);
        tma_load_2d(dst, &tmap, bar, c.col0, static_cast<int32_t>(c.row0));
        if (second)
            tma_load_2d(dst + kBoxBytes, &tmap, bar, c.col0 + kBoxCols, static_cast<int32_t>(c.row0));
    };

    if (tid == 0) {
        for (int s = 0; s < kStages && s < my_count; ++s)
            issue(s, first + s * stride);
    }

    uint32_t amax_acc = 0;  // running max |value| as fp32 bits (amax output only)
    // GEMM-ready scale planes.  A flat call's planes are one swizzled matrix each; a grouped
    // call's are one per group, each swizzled on its own (padded to 128-row x 4-column tiles)
    // and laid out after the previous group's.  A 128 x 128 cast tile's scales fill exactly one
    // 512-byte tile of each plane: rowwise, its 128 rows x 4 row blocks; columnwise (the plane
    // of the transposed operand, N rows), its 128 columns x 4 column blocks.
    //  - rowwise plane tile (rt, ct), tiles of ceil(N/128) per tile row: index rt * col_tiles + ct.
    //    A grouped tile's rt counts the row tiles of the groups before it too (their planes come
    //    first), so the same index holds.
    //  - columnwise plane tile (ct, rt): flat, index ct * row_tiles + rt; grouped, group g's plane
    //    has N rows and ceil(rows_g/128) tile columns and starts after before * col_tiles tiles
    //    (before = the row tiles of the groups before g = rt - the tile's row tile in its group):
    //    index before * col_tiles + ct * ceil(rows_g/128) + (rt - before).
    static_assert(kBM == 128 && kBN == 128, "one plane tile per cast tile");
    const int64_t Cn = (N + 31) >> 5;  // scale columns of the plain rowwise plane
    auto swz_row_tile = [&](const TileCoord &tc) -> uint8_t * {
        return p.scale_row + (static_cast<int64_t>(tc.rt) * p.col_tiles + (tc.col0 >> 7)) * 512;
    };
    auto swz_col_tile = [&](const TileCoord &tc) -> uint8_t * {
        const int ct = tc.col0 >> 7;
        if constexpr (GROUPED) {
            const int64_t first = goff[tc.g];
            const int rtl = static_cast<int>((tc.row0 - first) >> 7);
            const int tiles_g = static_cast<int>((goff[tc.g + 1] - first + 127) >> 7);
            return p.scale_col + (static_cast<int64_t>(tc.rt - rtl) * p.col_tiles + static_cast<int64_t>(ct) * tiles_g +
                                  rtl) * 512;
        } else {
            return p.scale_col + (static_cast<int64_t>(ct) * p.row_tiles + tc.rt) * 512;
        }
    };
    // A row's four 32-column blocks of a tile have their scales in four contiguous bytes (plain:
    // scale columns col0/32 .. +3 of the row; GEMM-ready: the row's entries of its plane tile).
    // Outside the warp-local phases, phase 2 collects them in shared memory and the tile's end
    // stores each row's four with one store (one L2 request per row, not one per lane pair):
    // v holds block b in byte b.  Blocks at or past N are not stored (plain), or stored as the
    // plane's zero padding (GEMM-ready).  A 32-bit store where the destination allows it
    // (scale_row needs no alignment), bytes otherwise.
    const bool row_scales_aligned = (reinterpret_cast<uintptr_t>(p.scale_row) & 3) == 0 && (SWZ || (Cn & 3) == 0);
    auto store_row_scales = [&](const TileCoord &tc, int r, int64_t grow, uint32_t v) {
        const int64_t left = (N - tc.col0 + 31) >> 5;
        const int nb = left < 4 ? static_cast<int>(left) : 4;  // blocks of the row in this tile
        uint8_t *dst;
        if constexpr (SWZ) {
            dst = swz_row_tile(tc) + swizzled_in_tile(r, 0);
            if (nb < 4)
                v &= (1u << (8 * nb)) - 1u;
        } else {
            dst = p.scale_row + grow * Cn + (tc.col0 >> 5);
        }
        if (row_scales_aligned && (SWZ || nb == 4)) {
            *reinterpret_cast<uint32_t *>(dst) = v;
        } else {
            const int nw = SWZ ? 4 : nb;
            for (int b = 0; b < nw; ++b)
                dst[b] = static_cast<uint8_t>(v >> (8 * b));
        }
    };
    for (int it = 0; it < my_count; ++it) {
        const int slot = it % kStages;
        const uint32_t parity = static_cast<uint32_t>(it / kStages) & 1u;
        const unsigned char *stage = smem + slot * kStageBytes;

        bool ok = mbar_wait_bounded(smem_u32(&bars[slot]), parity, kWaitLimitNs);
        if constexpr (kWarpLocal)
            ok = __all_sync(0xffffffffu, ok);  // warp-uniform: phase 2 may skip on it, with shuffles inside
        const TileCoord tc = coords[slot];

        // ---- phase 1: column blocks (rb = 32-row block, box = 64-column half) ----
        const bool rb_live = tc.row0 + (warp >> 1) * 32 < tc.row_end;  // this warp's 32-row block exists
        if (ok && (do_col || DBIAS) && !rb_live) {
            if constexpr (DBIAS) {  // an absent row block adds nothing to the column sums
                const int rb = warp >> 1, box = warp & 1;
                if (lane < 16)
                    *reinterpret_cast<float4 *>(dsum + rb * kBN + box * kBoxCols + lane * 4) =
                        make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        if (ok && (do_col || DBIAS) && rb_live) {
            const int rb = warp >> 1, box = warp & 1;
            const int cq = lane & 15, half = lane >> 4;   // 4-column group, 16-row half
            const unsigned char *base = stage + box * kBoxBytes + (rb * 32 + half * 16) * 128 + (cq & 1) * 8;
            float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
            int e0, e1, e2, e3;
            uint32_t amax_bits;  // fp32 bits of the largest of the four column amaxes
            if constexpr (GROUPED) {
                // A group's last block may end inside this 32-row block: the rows after it
                // (the next group's, loaded with the tile) are zeroed in this warp's box, so
                // they add nothing to the block's amax or column sums (phase 2 does not store
                // them).  Flat tiles need this nowhere: rows past M are loaded as zeros.
                const int64_t left = tc.row_end - (tc.row0 + rb * 32);
                const int live = left < 32 ? static_cast<int>(left) : 32;
                if (live < 32) {
                    unsigned char *blk = const_cast<unsigned char *>(stage) + box * kBoxBytes + rb * 32 * 128;
                    for (int c = live * 8 + lane; c < 32 * 8; c += 32)
                        *reinterpret_cast<uint4 *>(blk + c * 16) = make_uint4(0u, 0u, 0u, 0u);
                    fence_proxy_async_smem();  // before the stage is refilled by TMA
                    __syncwarp();
                }
            }
            if constexpr (ACT == 0) {
                uint32_t mx0 = 0, mx1 = 0;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    // row r = rb*32 + half*16 + i has (r & 7) == (i & 7): 128B swizzle
                    const uint2 v = lds64(base + i * 128 + (((cq >> 1) ^ (i & 7)) << 4));
                    mx0 = absmax_step<kXS>(mx0, v.x);
                    mx1 = absmax_step<kXS>(mx1, v.y);
                    if constexpr (DBIAS) {
                        d0 = add_bf16_lo(d0, v.x);
                        d1 = add_bf16_hi(d1, v.x);
                        d2 = add_bf16_lo(d2, v.y);
                        d3 = add_bf16_hi(d3, v.y);
                    }
                }
                mx0 = absmax_done<kXS>(mx0);
                mx1 = absmax_done<kXS>(mx1);
                mx0 = max_u16x2(mx0, __shfl_xor_sync(0xffffffffu, mx0, 16));
                mx1 = max_u16x2(mx1, __shfl_xor_sync(0xffffffffu, mx1, 16));
                e0 = block_exponent<FMT>(mx0 & 0xFFFFu);
                e1 = block_exponent<FMT>(mx0 >> 16);
                e2 = block_exponent<FMT>(mx1 & 0xFFFFu);
                e3 = block_exponent<FMT>(mx1 >> 16);
                amax_bits = max(max(mx0 & 0xFFFFu, mx0 >> 16), max(mx1 & 0xFFFFu, mx1 >> 16)) << 16;
            } else {
                // On x > 0 every activation here is increasing, so a column's amax is
                // act(max x) whenever that exceeds anything x <= 0 can give; ReLU and
                // squared ReLU give 0 for x <= 0, so for them this is always exact.
                uint32_t m01 = 0xFF80FF80u, m23 = 0xFF80FF80u;  // BF16 pairs (-inf, -inf)
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint2 v = lds64(base + i * 128 + (((cq >> 1) ^ (i & 7)) << 4));
                    m01 = max_bf16x2(m01, v.x);
                    m23 = max_bf16x2(m23, v.y);
                }
                float xm[4] = {bf16_lo(m01), bf16_hi(m01), bf16_lo(m23), bf16_hi(m23)};
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    xm[k] = fmaxf(xm[k], __shfl_xor_sync(0xffffffffu, xm[k], 16));
                float f[4];
                f2_unpack(activation2<ACT>(f2_pack(xm[0], xm[1])), f[0], f[1]);
                f2_unpack(activation2<ACT>(f2_pack(xm[2], xm[3])), f[2], f[3]);
                bool slow = false;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    f[k] = xm[k] > 0.f ? f[k] : 0.f;
                    slow |= ACT > 2 && f[k] < negative_side_bound<ACT>();
                }
                if (__any_sync(0xffffffffu, slow)) {
                    // some column's amax may come from its negative entries: evaluate them all
                    float g[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint2 v = lds64(base + i * 128 + (((cq >> 1) ^ (i & 7)) << 4));
                        float a0, a1, a2, a3;
                        f2_unpack(activation2<ACT>(f2_pack(bf16_lo(v.x), bf16_hi(v.x))), a0, a1);
                        f2_unpack(activation2<ACT>(f2_pack(bf16_lo(v.y), bf16_hi(v.y))), a2, a3);
                        g[0] = fmaxf(g[0], fabsf(a0));
                        g[1] = fmaxf(g[1], fabsf(a1));
                        g[2] = fmaxf(g[2], fabsf(a2));
                        g[3] = fmaxf(g[3], fabsf(a3));
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        f[k] = fmaxf(g[k], __shfl_xor_sync(0xffffffffu, g[k], 16));
                }
                e0 = block_exponent_f32<FMT>(__float_as_uint(f[0]));
                e1 = block_exponent_f32<FMT>(__float_as_uint(f[1]));
                e2 = block_exponent_f32<FMT>(__float_as_uint(f[2]));
                e3 = block_exponent_f32<FMT>(__float_as_uint(f[3]));
                amax_bits = __float_as_uint(fmaxf(fmaxf(f[0], f[1]), fmaxf(f[2], f[3])));
            }
            if constexpr (DBIAS) {
                // 32-row column sums; a + b == b + a, so both halves agree bit for bit
                d0 += __shfl_xor_sync(0xffffffffu, d0, 16);
                d1 += __shfl_xor_sync(0xffffffffu, d1, 16);
                d2 += __shfl_xor_sync(0xffffffffu, d2, 16);
                d3 += __shfl_xor_sync(0xffffffffu, d3, 16);
            }
            const int64_t gcol = tc.col0 + box * kBoxCols + cq * 4;
            const int64_t grow = tc.row0 + rb * 32;
            if (AMAX && gcol < N)
                amax_acc = max(amax_acc, amax_bits);
            if (half == 0) {
                if (do_col && gcol < N && grow < tc.row_end) {
                    if constexpr (!SWZ) {
                        *reinterpret_cast<uint32_t *>(p.scale_col + static_cast<int64_t>(tc.sb + rb) * N + gcol) =
                            static_cast<uint32_t>(e0) | (static_cast<uint32_t>(e1) << 8) |
                            (static_cast<uint32_t>(e2) << 16) | (static_cast<uint32_t>(e3) << 24);
                    } else {
                        // the columnwise operand's scales: plane row = this column, plane column =
                        // the row block; the next three columns are the plane's next rows in the
                        // same 32-row group (box * 64 + cq * 4 is a multiple of 4): 16 bytes apart
                        uint8_t *sc = swz_col_tile(tc) + swizzled_in_tile(box * kBoxCols + cq * 4, rb);
                        sc[0] = static_cast<uint8_t>(e0);
                        sc[16] = static_cast<uint8_t>(e1);
                        sc[32] = static_cast<uint8_t>(e2);
                        sc[48] = static_cast<uint8_t>(e3);
                    }
                }
                if constexpr (DBIAS)
                    *reinterpret_cast<float4 *>(dsum + rb * kBN + box * kBoxCols + cq * 4) =
                        make_float4(d0, d1, d2, d3);
            } else {
                // column multipliers for phase 2: 4-column group q of segment sp is
                // stored at chunk 4*sp + ((q + (sp >> 1)) & 3) (bank-conflict free reads)
                const int sp = cq >> 2, q = cq & 3;
                const int chunk = 4 * sp + ((q + (sp >> 1)) & 3);
                *reinterpret_cast<float4 *>(colmul + rb * kBN + box * kBoxCols + chunk * 4) =
                    make_float4(scale_multiplier(e0), scale_multiplier(e1), scale_multiplier(e2),
                                scale_multiplier(e3));
            }
        }
        // GEMM-ready planes: the tile owns one 512-byte tile of each plane (the rowwise plane's
        // 128 rows x 4 scale columns, the columnwise plane's 128 rows (this tile's columns) x 4
        // scale columns (its 32-row blocks)).  The entries of those that hold no scale (rows past
        // the tile's end, columns past N) are zeroed here, so no separate padding pass is needed:
        // warp (rb, box) zeroes those of its 32 rows x 2 row blocks and of its 64 columns x 1
        // column block.  Every other entry is written by the phase that forms its scale.
        if constexpr (SWZ) {
            if (ok) {
                const int rb = warp >> 1, box = warp & 1;
                const int64_t grow = tc.row0 + rb * 32;
                if (do_row) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int64_t bc = tc.col0 + box * kBoxCols + j * 32;  // the block's first column
                        // (a live row's blocks past N are written with its other scales outside
                        // the warp-local phases)
                        if (grow + lane >= tc.row_end || (kWarpLocal && bc >= N))
                            swz_row_tile(tc)[swizzled_in_tile(rb * 32 + lane, box * 2 + j)] = 0;
                    }
                }
                if (do_col && lane < 16) {
                    const int64_t gcol = tc.col0 + box * kBoxCols + lane * 4;
                    if (grow >= tc.row_end || gcol >= N) {
                        uint8_t *sc = swz_col_tile(tc) + swizzled_in_tile(box * kBoxCols + lane * 4, rb);
                        sc[0] = 0;
                        sc[16] = 0;
                        sc[32] = 0;
                        sc[48] = 0;
                    }
                }
            }
        }
        // a bounded wait that expired: record it, drain this CTA's own copies, return
        auto give_up = [&]() {
            if (tid == 0) {
                atomicOr(&g_fault_word, 1u);
                if (GROUPED && p.err_flag != nullptr)
                    atomicOr(p.err_flag, 2);
                for (int j = it; j < my_count && j < it + kStages; ++j)
                    mbar_wait_bounded(smem_u32(&bars[j % kStages]), static_cast<uint32_t>(j / kStages) & 1u,
                                      kDrainLimitNs);
            }
        };
        if constexpr (kWarpLocal) {
            __syncwarp();  // phase 2 reads what this warp wrote in phase 1; the fault test is at the tile's end
        } else if (__syncthreads_or(!ok)) {
            give_up();
            return;
        }

        // dbias partial of this tile: the four 32-row block sums, in a fixed order
        if constexpr (DBIAS) {
            if (tid < kBN) {
                const int64_t gcol = tc.col0 + tid;
                if (gcol < N)
                    p.ws[static_cast<int64_t>(tc.rt) * N + gcol] =
                        ((dsum[tid] + dsum[kBN + tid]) + dsum[2 * kBN + tid]) + dsum[3 * kBN + tid];
            }
        }

        // ---- phase 2: row segments of 16 columns ----
        {
            const int rr = lane >> 2, sp = lane & 3;
            constexpr bool kReuse = kWarpLocal;
            float4 cmv[4];
            if (kReuse && do_col) {
                const float *cm0 = colmul + (warp >> 1) * kBN + (warp & 1) * kBoxCols + sp * 16;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    cmv[j] = lds128f(cm0 + 4 * ((j + (sp >> 1)) & 3));
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int task = warp + 8 * k;
                const int box = kReuse ? (warp & 1) : (task & 1);
                const int rg = kReuse ? (warp >> 1) * 4 + k : (task >> 1);
                if (tc.row0 + rg * 8 >= tc.row_end || (kWarpLocal && !ok))
                    continue;               // warp-uniform: the whole 8-row group is past the tile end
                const int r = rg * 8 + rr;  // (r & 7) == rr
                const unsigned char *rowp = stage + box * kBoxBytes + r * 128;
                const int p0 = (2 * sp) ^ rr;
                const uint4 A = lds128(rowp + p0 * 16);        // columns 16sp + 0..7
                const uint4 B = lds128(rowp + (p0 ^ 1) * 16);  // columns 16sp + 8..15
                const uint32_t w[8] = {A.x, A.y, A.z, A.w, B.x, B.y, B.z, B.w};
                const int64_t grow = tc.row0 + r;
                const int64_t gcol = tc.col0 + box * kBoxCols + sp * 16;
                const bool in = grow < tc.row_end && gcol < N;
                // the 16 values of the segment: the BF16 inputs, or their fp32 activations
                float y[16];
                if constexpr (ACT != 0) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        f2_unpack(activation2<ACT>(f2_pack(bf16_lo(w[j]), bf16_hi(w[j]))), y[2 * j], y[2 * j + 1]);
                }
                // two codes from two values and their multipliers (f32x2 multiplies pay
                // on the activation paths only: measured)
                auto cvt_pair = [](float a, float b, float ma, float mb) -> uint32_t {
                    if constexpr (ACT != 0)
                        return cvt_fp8x2_scaled<FMT>(a, b, f2_pack(ma, mb));
                    else
                        return cvt_fp8x2<FMT>(a * ma, b * mb);
                };
                auto val = [&](int i) -> float {
                    if constexpr (ACT == 0)
                        return (i & 1) ? bf16_hi(w[i >> 1]) : bf16_lo(w[i >> 1]);
                    else
                        return y[i];
                };
                if (do_row) {
                    int er;
                    uint32_t row_amax_bits;  // fp32 bits
                    if constexpr (ACT == 0) {
                        uint32_t m = 0;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            m = absmax_step<kXS>(m, w[j]);
                        m = absmax_done<kXS>(m);
                        uint32_t a = max(m & 0xFFFFu, m >> 16);
                        a = max(a, __shfl_xor_sync(0xffffffffu, a, 1));
                        er = block_exponent<FMT>(a);
                        row_amax_bits = a << 16;
                    } else {
                        float fm = 0.f;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            fm = fmaxf(fm, fabsf(y[i]));
                        fm = fmaxf(fm, __shfl_xor_sync(0xffffffffu, fm, 1));
                        er = block_exponent_f32<FMT>(__float_as_uint(fm));
                        row_amax_bits = __float_as_uint(fm);
                    }
                    const float rm = scale_multiplier(er);
                    uint32_t o[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t lo = cvt_pair(val(4 * j), val(4 * j + 1), rm, rm);
                        const uint32_t hi = cvt_pair(val(4 * j + 2), val(4 * j + 3), rm, rm);
                        o[j] = lo | (hi << 16);
                    }
                    if (in) {
                        store_codes(p.out_row + grow * N + gcol, o[0], o[1], o[2], o[3], rows16, gcol + 16 > N);
                        if ((sp & 1) == 0) {
                            if constexpr (!kWarpLocal)
                                reinterpret_cast<uint8_t *>(rowsc)[r * 4 + box * 2 + (sp >> 1)] = static_cast<uint8_t>(er);
                            else if constexpr (SWZ)
                                swz_row_tile(tc)[swizzled_in_tile(r, box * 2 + (sp >> 1))] = static_cast<uint8_t>(er);
                            else
                                p.scale_row[grow * Cn + (gcol >> 5)] = static_cast<uint8_t>(er);
                        }
                        if (AMAX && !do_col)
                            amax_acc = max(amax_acc, row_amax_bits);
                    }
                }
                if (do_col) {
                    const float *cm = colmul + (r >> 5) * kBN + box * kBoxCols + sp * 16;
                    uint32_t o[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 c = kReuse ? cmv[j] : lds128f(cm + 4 * ((j + (sp >> 1)) & 3));
                        const uint32_t lo = cvt_pair(val(4 * j), val(4 * j + 1), c.x, c.y);
                        const uint32_t hi = cvt_pair(val(4 * j + 2), val(4 * j + 3), c.z, c.w);
                        o[j] = lo | (hi << 16);
                    }
                    if (in)
                        store_codes(p.out_col + grow * N + gcol, o[0], o[1], o[2], o[3], rows16, gcol + 16 > N);
                }
            }
        }
        if constexpr (kWarpLocal) {
            // No CTA barrier: each warp counts itself done with the stage, and the eighth to
            // finish refills it.  A warp whose wait expired records the fault, drains the copies
            // that can still be in flight (tiles it .. it + kStages - 1: no later tile is issued
            // while this one is unfinished) and leaves; the stage it abandons is never refilled,
            // so the other warps' bounded waits expire in turn and they leave the same way.
            if (!ok) {
                if (lane == 0) {
                    atomicOr(&g_fault_word, 1u);
                    if (GROUPED && p.err_flag != nullptr)
                        atomicOr(p.err_flag, 2);
                    for (int j = it; j < my_count && j < it + kStages; ++j)
                        mbar_wait_bounded(smem_u32(&bars[j % kStages]), static_cast<uint32_t>(j / kStages) & 1u,
                                          kDrainLimitNs);
                }
                return;
            }
            __syncwarp();
            if (lane == 0) {
                unsigned before;
                asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                             : "=r"(before)
                             : "r"(smem_u32(&stage_done[slot]))
                             : "memory");
                if (before == kThreads / 32 - 1) {
                    stage_done[slot] = 0;  // no warp touches it again before the refill completes
                    if (it + kStages < my_count) {
                        fence_proxy_async_smem();
                        issue(slot, first + (it + kStages) * stride);
                    }
                }
            }
            continue;
        } else {
            __syncthreads();  // stage `slot` and colmul are free again; the tile's row scales are in rowsc
            if (do_row && tid < kBM && tc.row0 + tid < tc.row_end)
                store_row_scales(tc, tid, tc.row0 + tid, rowsc[tid]);
        }

        if (tid == 0 && it + kStages < my_count) {
            fence_proxy_async_smem();
            issue(slot, first + (it + kStages) * stride);
        }
    }
    if constexpr (AMAX) {
        // fp32 bits of a non-negative value order like the value itself
        const uint32_t m = __reduce_max_sync(0xffffffffu, amax_acc);
        if (lane == 0 && m != 0)
            atomicMax(reinterpret_cast<unsigned int *>(p.amax), m);
    }
}

}  // namespace mxfp8
