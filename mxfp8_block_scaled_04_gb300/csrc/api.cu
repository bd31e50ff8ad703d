// C ABI of the MXFP8 quantize library (declarations and contract in
// include/mxfp8.h).  Host-side validation, TMA descriptor encoding, kernel
// launches and the host-buffer pipeline; the device code is in quantize.cuh
// (the cast), dact.cuh (the backward fusion) and dbias_reduce.cuh.
#include <atomic>
#include <initializer_list>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <utility>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/mxfp8.h"
#include "dact.cuh"
#include "dbias_reduce.cuh"
#include "dgated.cuh"
#include "quantize.cuh"

namespace {

using namespace mxfp8;

constexpr int kMaxDevices = 64;

std::atomic<uint64_t> g_launches{0};

// Launch with programmatic stream serialisation: the kernel may begin while the
// previous kernel on the stream drains, and waits (griddepcontrol.wait) before
// its first global memory access, so stream order holds for every buffer.
// Only kernels that make that wait are launched this way.
template <typename... Params, typename... Args>
mxfp8_status_t launch_pdl(void (*kern)(Params...), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                          Args &&...args)
{
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
    const cudaError_t last = cudaGetLastError();
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return e == cudaSuccess && last == cudaSuccess ? MXFP8_OK : MXFP8_ERR_LAUNCH;
}

struct DeviceInfo {
    bool ready = false;
    int sm_count = 0;
    int ctas_per_sm[192] = {};  // indexed by kernel variant
    int dact_ctas_per_sm[48] = {};  // two-input kernels: FMT + 2 * DBIAS + 4 * ACT + 24 * GATED
    int dgated_ctas_per_sm[12] = {};  // gated backward: FMT + 2 * ACT
    int ggated_ctas_per_sm[12] = {};  // grouped gated cast: FMT + 2 * ACT
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Is p device (or managed) memory of `device`?  NULL passes.
bool on_device(const void *p, int device)
{
    if (p == nullptr)
        return true;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeManaged)
        return true;
    return a.type == cudaMemoryTypeDevice && a.device == device;
}

template <int FMT, bool DBIAS, bool GROUPED, bool SWZ, bool AMAX, int ACT>
int variant_index()
{
    return FMT + 2 * (DBIAS ? 1 : 0) + 4 * (GROUPED ? 1 : 0) + 8 * (SWZ ? 1 : 0) + 16 * (AMAX ? 1 : 0) + 32 * ACT;
}

// One-time per (device, variant) set-up: opt in to the large shared-memory
// carve-out and record how many CTAs fit per SM.
template <int FMT, bool DBIAS, bool GROUPED, bool SWZ, bool AMAX, int ACT>
mxfp8_status_t prepare(int device, int *grid_cap)
{
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (device < 0 || device >= kMaxDevices)
        return MXFP8_ERR_DEVICE;
    DeviceInfo &d = g_dev[device];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
            cudaGetLastError();  // leave no error behind for the caller
            return MXFP8_ERR_DEVICE;
        }
        d.ready = true;
    }
    const int v = variant_index<FMT, DBIAS, GROUPED, SWZ, AMAX, ACT>();
    if (d.ctas_per_sm[v] == 0) {
        const int smem = GROUPED ? kSmemGrouped : kSmemFlat;
        auto kern = quantize_kernel<FMT, DBIAS, GROUPED, SWZ, AMAX, ACT>;
        int n = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem) != cudaSuccess || n < 1) {
            cudaGetLastError();
            return MXFP8_ERR_LAUNCH;
        }
        d.ctas_per_sm[v] = n;
    }
    *grid_cap = d.ctas_per_sm[v] * d.sm_count;
    return MXFP8_OK;
}

// TMA map of a BF16 matrix [rows, N] whose rows are `pitch` elements apart (pitch >= N), in boxes
// of box_rows rows x 64 columns.
mxfp8_status_t make_tensor_map_pitch(CUtensorMap *map, const void *x, int64_t rows, int64_t N, int64_t pitch,
                                     int box_rows = kBM)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (enc == nullptr)
        return MXFP8_ERR_DEVICE;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch) * 2};
    cuuint32_t box[2] = {kBoxCols, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MXFP8_OK : MXFP8_ERR_LAUNCH;
}

mxfp8_status_t make_tensor_map(CUtensorMap *map, const void *x, int64_t rows, int64_t N)
{
    return make_tensor_map_pitch(map, x, rows, N, N);
}

// Shared host-side checks of the direction pointers.
mxfp8_status_t check_outputs(void *out_row, void *scale_row, void *out_col, void *scale_col)
{
    if ((out_row == nullptr) != (scale_row == nullptr) || (out_col == nullptr) != (scale_col == nullptr))
        return MXFP8_ERR_NULL;
    if (out_row == nullptr && out_col == nullptr)
        return MXFP8_ERR_NULL;
    if (!aligned(out_row, 16) || !aligned(out_col, 16) || !aligned(scale_col, 4))
        return MXFP8_ERR_ALIGN;
    return MXFP8_OK;
}

mxfp8_status_t current_device(int *device)
{
    if (cudaGetDevice(device) != cudaSuccess) {
        cudaGetLastError();
        return MXFP8_ERR_DEVICE;
    }
    return MXFP8_OK;
}

template <bool DBIAS, bool GROUPED, bool SWZ = false, bool AMAX = false, int ACT = 0>
mxfp8_status_t launch_quantize(int fmt, int device, const CUtensorMap &map, const QuantParams &p,
                               int64_t tile_bound, cudaStream_t stream)
{
    int cap = 0;
    mxfp8_status_t st = fmt == MXFP8_E4M3 ? prepare<0, DBIAS, GROUPED, SWZ, AMAX, ACT>(device, &cap)
                                          : prepare<1, DBIAS, GROUPED, SWZ, AMAX, ACT>(device, &cap);
    if (st != MXFP8_OK)
        return st;
    const int grid = static_cast<int>(tile_bound < cap ? tile_bound : cap);
    const int smem = GROUPED ? kSmemGrouped : kSmemFlat;
    if (fmt == MXFP8_E4M3)
        return launch_pdl(quantize_kernel<0, DBIAS, GROUPED, SWZ, AMAX, ACT>, grid, kThreads, smem, stream, map, p);
    return launch_pdl(quantize_kernel<1, DBIAS, GROUPED, SWZ, AMAX, ACT>, grid, kThreads, smem, stream, map, p);
}

// Per-tensor amax output: zero it before the quantize kernel (unless noop).
__global__ void amax_init_kernel(float *amax, const float *noop)
{
    if (noop != nullptr && *noop == 1.0f)
        return;
    *amax = 0.0f;
}

// Enqueue the flat quantize kernel (no validation: the caller has checked every
// argument).  ws != nullptr selects the dbias variant, which writes one fp32
// partial column sum per 128-row tile of this call to ws[tile][N].
// The backward-fusion kernel (dY * act'(X)): one-time set-up per (device, variant), then launch.
template <int FMT, bool DBIAS, int ACT, bool GATED = false, bool GROUPED = false>
mxfp8_status_t launch_dact_fmt(int device, const CUtensorMap &map_g, const CUtensorMap &map_x, const QuantParams &p,
                               int64_t tiles, cudaStream_t stream)
{
    constexpr int smem = GROUPED ? kSmemDactGrouped : kSmemDact;
    int cap = 0;
    {
        std::lock_guard<std::mutex> lock(g_dev_mu);
        if (device < 0 || device >= kMaxDevices)
            return MXFP8_ERR_DEVICE;
        DeviceInfo &d = g_dev[device];
        if (!d.ready) {
            if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
                cudaGetLastError();
                return MXFP8_ERR_DEVICE;
            }
            d.ready = true;
        }
        int &slot = GROUPED ? d.ggated_ctas_per_sm[FMT + 2 * ACT]
                            : d.dact_ctas_per_sm[FMT + 2 * (DBIAS ? 1 : 0) + 4 * ACT + (GATED ? 24 : 0)];
        if (slot == 0) {
            auto kern = quantize_dact_kernel<FMT, DBIAS, ACT, GATED, GROUPED>;
            int n = 0;
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem) != cudaSuccess || n < 1) {
                cudaGetLastError();
                return MXFP8_ERR_LAUNCH;
            }
            slot = n;
        }
        cap = slot * d.sm_count;
    }
    const int grid = static_cast<int>(tiles < cap ? tiles : cap);
    return launch_pdl(quantize_dact_kernel<FMT, DBIAS, ACT, GATED, GROUPED>, grid, kThreads, smem, stream, map_g,
                      map_x, p);
}

template <int ACT>
mxfp8_status_t launch_dact(int fmt, bool dbias, int device, const CUtensorMap &map_g, const CUtensorMap &map_x,
                           const QuantParams &p, int64_t tiles, cudaStream_t stream)
{
    if (fmt == MXFP8_E4M3)
        return dbias ? launch_dact_fmt<0, true, ACT>(device, map_g, map_x, p, tiles, stream)
                     : launch_dact_fmt<0, false, ACT>(device, map_g, map_x, p, tiles, stream);
    return dbias ? launch_dact_fmt<1, true, ACT>(device, map_g, map_x, p, tiles, stream)
                 : launch_dact_fmt<1, false, ACT>(device, map_g, map_x, p, tiles, stream);
}

template <int ACT, bool GROUPED = false>
mxfp8_status_t launch_gated(int fmt, int device, const CUtensorMap &map_b, const CUtensorMap &map_a,
                            const QuantParams &p, int64_t tiles, cudaStream_t stream)
{
    return fmt == MXFP8_E4M3 ? launch_dact_fmt<0, false, ACT, true, GROUPED>(device, map_b, map_a, p, tiles, stream)
                             : launch_dact_fmt<1, false, ACT, true, GROUPED>(device, map_b, map_a, p, tiles, stream);
}

// The gated backward kernel that evaluates each product once (64-row tiles): for ReGLU, GeGLU,
// SwiGLU and QGeGLU (measured 2-10% faster); squared-ReLU GLU runs 9% faster with the 128-row one.
template <int ACT>
constexpr bool kKeepDgated = ACT != MXFP8_ACT_SRELU;

// The gated backward kernel: one-time set-up per (device, variant), then launch.
template <int FMT, int ACT>
mxfp8_status_t launch_dgated_fmt(int device, const CUtensorMap &map_g, const CUtensorMap &map_a,
                                 const CUtensorMap &map_b, const QuantParams &p, int64_t tiles, cudaStream_t stream)
{
    int cap = 0;
    {
        std::lock_guard<std::mutex> lock(g_dev_mu);
        if (device < 0 || device >= kMaxDevices)
            return MXFP8_ERR_DEVICE;
        DeviceInfo &d = g_dev[device];
        if (!d.ready) {
            if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
                cudaGetLastError();
                return MXFP8_ERR_DEVICE;
            }
            d.ready = true;
        }
        const int v = FMT + 2 * ACT;
        if (d.dgated_ctas_per_sm[v] == 0) {
            auto kern = [] {
                if constexpr (kKeepDgated<ACT>)
                    return quantize_dgated_keep_kernel<FMT, ACT>;
                else
                    return quantize_dgated_kernel<FMT, ACT>;
            }();
            const int smem = kKeepDgated<ACT> ? kSmemDgatedKeep : kSmemDgated;
            int n = 0;
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem) != cudaSuccess || n < 1) {
                cudaGetLastError();
                return MXFP8_ERR_LAUNCH;
            }
            d.dgated_ctas_per_sm[v] = n;
        }
        cap = d.dgated_ctas_per_sm[v] * d.sm_count;
    }
    const int grid = static_cast<int>(tiles < cap ? tiles : cap);
    if constexpr (kKeepDgated<ACT>)
        return launch_pdl(quantize_dgated_keep_kernel<FMT, ACT>, grid, kThreads, kSmemDgatedKeep, stream, map_g, map_a,
                          map_b, p);
    else
        return launch_pdl(quantize_dgated_kernel<FMT, ACT>, grid, kThreads, kSmemDgated, stream, map_g, map_a, map_b,
                          p);
}

template <int ACT>
mxfp8_status_t launch_dgated(int fmt, int device, const CUtensorMap &map_g, const CUtensorMap &map_a,
                             const CUtensorMap &map_b, const QuantParams &p, int64_t tiles, cudaStream_t stream)
{
    return fmt == MXFP8_E4M3 ? launch_dgated_fmt<0, ACT>(device, map_g, map_a, map_b, p, tiles, stream)
                             : launch_dgated_fmt<1, ACT>(device, map_g, map_a, map_b, p, tiles, stream);
}

// Activated (ACT != 0) variants: flat, no dbias; swizzle and amax as template switches.
template <int ACT>
mxfp8_status_t launch_activated(int opts, int fmt, int device, const CUtensorMap &map, const QuantParams &p,
                                int64_t tiles, cudaStream_t stream)
{
    switch (opts) {
    case 0: return launch_quantize<false, false, false, false, ACT>(fmt, device, map, p, tiles, stream);
    case 1: return launch_quantize<false, false, true, false, ACT>(fmt, device, map, p, tiles, stream);
    case 2: return launch_quantize<false, false, false, true, ACT>(fmt, device, map, p, tiles, stream);
    default: return launch_quantize<false, false, true, true, ACT>(fmt, device, map, p, tiles, stream);
    }
}

mxfp8_status_t enqueue_flat(int device, int fmt, const void *x, int64_t M, int64_t N, void *out_row,
                            void *scale_row, void *out_col, void *scale_col, float *ws, const float *noop,
                            cudaStream_t stream, bool swizzled = false, float *amax = nullptr, int act = 0)
{
    CUtensorMap map;
    mxfp8_status_t st = make_tensor_map(&map, x, M, N);
    if (st != MXFP8_OK)
        return st;
    const int64_t row_tiles = (M + kBM - 1) / kBM, col_tiles = (N + kBN - 1) / kBN;
    QuantParams p{};
    p.out_row = static_cast<uint8_t *>(out_row);
    p.scale_row = static_cast<uint8_t *>(scale_row);
    p.out_col = static_cast<uint8_t *>(out_col);
    p.scale_col = static_cast<uint8_t *>(scale_col);
    p.ws = ws;
    p.noop = noop;
    p.M = M;
    p.N = N;
    p.row_tiles = static_cast<int>(row_tiles);
    p.col_tiles = static_cast<int>(col_tiles);
    p.amax = amax;
    const int64_t tiles = row_tiles * col_tiles;
    const int opts = (swizzled ? 1 : 0) + (amax != nullptr ? 2 : 0);
    if (act != MXFP8_ACT_NONE) {
        if (ws != nullptr)
            return MXFP8_ERR_FORMAT;
        switch (act) {
        case MXFP8_ACT_RELU: return launch_activated<1>(opts, fmt, device, map, p, tiles, stream);
        case MXFP8_ACT_SRELU: return launch_activated<2>(opts, fmt, device, map, p, tiles, stream);
        case MXFP8_ACT_GELU: return launch_activated<3>(opts, fmt, device, map, p, tiles, stream);
        case MXFP8_ACT_SILU: return launch_activated<4>(opts, fmt, device, map, p, tiles, stream);
        case MXFP8_ACT_QGELU: return launch_activated<5>(opts, fmt, device, map, p, tiles, stream);
        default: return MXFP8_ERR_FORMAT;
        }
    }
    if (ws != nullptr) {
        switch (opts) {
        case 0: return launch_quantize<true, false, false, false>(fmt, device, map, p, tiles, stream);
        case 1: return launch_quantize<true, false, true, false>(fmt, device, map, p, tiles, stream);
        case 2: return launch_quantize<true, false, false, true>(fmt, device, map, p, tiles, stream);
        default: return launch_quantize<true, false, true, true>(fmt, device, map, p, tiles, stream);
        }
    }
    switch (opts) {
    case 0: return launch_quantize<false, false, false, false>(fmt, device, map, p, tiles, stream);
    case 1: return launch_quantize<false, false, true, false>(fmt, device, map, p, tiles, stream);
    case 2: return launch_quantize<false, false, false, true>(fmt, device, map, p, tiles, stream);
    default: return launch_quantize<false, false, true, true>(fmt, device, map, p, tiles, stream);
    }
}

// Enqueue the dbias reduce over row_tiles partial rows of ws.
mxfp8_status_t enqueue_reduce(const float *ws, int64_t row_tiles, int64_t N, float *dbias, const float *noop,
                              cudaStream_t stream)
{
    const int64_t blocks = (N + kReduceCols - 1) / kReduceCols;
    return launch_pdl(dbias_reduce_kernel, static_cast<unsigned>(blocks), kReduceCols * kReduceWarps, 0, stream, ws,
                      row_tiles, N, dbias, noop);
}

// The grouped dbias workspace starts with an int64 header [num_groups + 1] (each
// group's first row tile), padded to 256 bytes; the fp32 partials follow.
int64_t grouped_header_floats(int num_groups)
{
    return ((static_cast<int64_t>(num_groups) + 1) * 8 + 255) / 256 * 256 / 4;
}

// The grouped call, with or without per-group dbias (ws and dbias both set).
mxfp8_status_t grouped_impl(const void *x, int64_t total_rows, int64_t N, int num_groups, const int64_t *offsets,
                            int fp8_fmt, void *out_row, void *scale_row, void *out_col, void *scale_col,
                            float *dbias, float *ws, const float *noop, int *err_flag, cudaStream_t stream,
                            int act = MXFP8_ACT_NONE, bool swizzled = false)
{
    if (fp8_fmt != MXFP8_E4M3 && fp8_fmt != MXFP8_E5M2)
        return MXFP8_ERR_FORMAT;
    if (act < MXFP8_ACT_NONE || act > MXFP8_ACT_QGELU || (act != MXFP8_ACT_NONE && dbias != nullptr) ||
        (swizzled && dbias != nullptr))
        return MXFP8_ERR_FORMAT;
    if (total_rows < 0 || N < 0 || N % 8 || total_rows >= (int64_t{1} << 31) || N >= (int64_t{1} << 31))
        return MXFP8_ERR_SHAPE;
    if (num_groups < 1 || num_groups > MXFP8_MAX_GROUPS || offsets == nullptr)
        return MXFP8_ERR_GROUPS;
    if (x == nullptr)
        return MXFP8_ERR_NULL;
    mxfp8_status_t st = check_outputs(out_row, scale_row, out_col, scale_col);
    if (st != MXFP8_OK)
        return st;
    if (!aligned(x, 16) || !aligned(offsets, 8) || !aligned(err_flag, 4) || !aligned(dbias, 4) || !aligned(ws, 16))
        return MXFP8_ERR_ALIGN;
    const int64_t col_tiles = (N + kBN - 1) / kBN;
    // Upper bound on the tile count: every non-empty group adds at most one partial row tile.
    const int64_t tile_bound = (total_rows / kBM + num_groups) * col_tiles;
    if (tile_bound >= (int64_t{1} << 31))
        return MXFP8_ERR_SHAPE;

    int device = 0;
    if ((st = current_device(&device)) != MXFP8_OK)
        return st;
    if (!on_device(x, device) || !on_device(offsets, device) || !on_device(out_row, device) ||
        !on_device(scale_row, device) || !on_device(out_col, device) || !on_device(scale_col, device) ||
        !on_device(noop, device) || !on_device(err_flag, device) || !on_device(dbias, device) ||
        !on_device(ws, device))
        return MXFP8_ERR_DEVICE;
    if (total_rows > 0 && N > 0) {
        CUtensorMap map;
        if ((st = make_tensor_map(&map, x, total_rows, N)) != MXFP8_OK)
            return st;
        QuantParams p{};
        p.out_row = static_cast<uint8_t *>(out_row);
        p.scale_row = static_cast<uint8_t *>(scale_row);
        p.out_col = static_cast<uint8_t *>(out_col);
        p.scale_col = static_cast<uint8_t *>(scale_col);
        p.ws = ws != nullptr ? ws + grouped_header_floats(num_groups) : nullptr;
        p.ws_hdr = reinterpret_cast<int64_t *>(ws);
        p.noop = noop;
        p.offsets = offsets;
        p.err_flag = err_flag;
        p.M = total_rows;
        p.N = N;
        p.num_groups = num_groups;
        p.col_tiles = static_cast<int>(col_tiles);
        p.row_tiles = static_cast<int>((total_rows + kBM - 1) / kBM);  // the flat schedule (aligned groups)
        auto launch_act = [&](auto swz_tag) -> mxfp8_status_t {
            constexpr bool S = decltype(swz_tag)::value;
            switch (act) {
            case MXFP8_ACT_RELU: return launch_quantize<false, true, S, false, 1>(fp8_fmt, device, map, p, tile_bound,
                                                                                 stream);
            case MXFP8_ACT_SRELU: return launch_quantize<false, true, S, false, 2>(fp8_fmt, device, map, p, tile_bound,
                                                                                  stream);
            case MXFP8_ACT_GELU: return launch_quantize<false, true, S, false, 3>(fp8_fmt, device, map, p, tile_bound,
                                                                                 stream);
            case MXFP8_ACT_SILU: return launch_quantize<false, true, S, false, 4>(fp8_fmt, device, map, p, tile_bound,
                                                                                 stream);
            case MXFP8_ACT_QGELU: return launch_quantize<false, true, S, false, 5>(fp8_fmt, device, map, p,
                                                                                  tile_bound, stream);
            default:
                if constexpr (S)
                    return launch_quantize<false, true, true, false>(fp8_fmt, device, map, p, tile_bound, stream);
                else
                    return dbias != nullptr
                               ? launch_quantize<true, true>(fp8_fmt, device, map, p, tile_bound, stream)
                               : launch_quantize<false, true>(fp8_fmt, device, map, p, tile_bound, stream);
            }
        };
        st = swizzled ? launch_act(std::true_type{}) : launch_act(std::false_type{});
        if (st != MXFP8_OK)
            return st;
    }
    if (dbias != nullptr && N > 0) {
        const unsigned blocks = static_cast<unsigned>((N + kReduceCols - 1) / kReduceCols);
        const float *partials = ws + grouped_header_floats(num_groups);
        const int64_t *hdr = reinterpret_cast<const int64_t *>(ws);
        st = launch_pdl(dbias_reduce_grouped_kernel, blocks, kReduceCols * kGReduceWarps, 0, stream, partials, hdr,
                        num_groups, N, dbias, noop);
        if (st != MXFP8_OK)
            return st;
    }
    return MXFP8_OK;
}

}  // namespace

extern "C" {

size_t mxfp8_quantize_workspace_bytes(int64_t M, int64_t N, int with_dbias)
{
    if (!with_dbias || M < 0 || N < 0 || N % 8)
        return 0;
    return static_cast<size_t>((M + kBM - 1) / kBM) * static_cast<size_t>(N) * sizeof(float);
}

size_t mxfp8_quantize_grouped_workspace_bytes(int64_t, int64_t, int) { return 0; }

mxfp8_status_t mxfp8_quantize(const void *x, int64_t M, int64_t N, int fp8_fmt, void *out_row, void *scale_row,
                              void *out_col, void *scale_col, float *dbias, void *workspace, const float *noop,
                              void *stream_)
{
    // ---- host-only checks, in a fixed order, before touching the device ----
    if (fp8_fmt != MXFP8_E4M3 && fp8_fmt != MXFP8_E5M2)
        return MXFP8_ERR_FORMAT;
    if (M < 0 || N < 0 || N % 8 || M >= (int64_t{1} << 31) || N >= (int64_t{1} << 31))
        return MXFP8_ERR_SHAPE;
    const bool empty = M == 0 || N == 0;  // nothing to read or write: data pointers may be NULL
    mxfp8_status_t st;
    if (!empty) {
        if (x == nullptr)
            return MXFP8_ERR_NULL;
        if ((st = check_outputs(out_row, scale_row, out_col, scale_col)) != MXFP8_OK)
            return st;
    }
    if (!aligned(x, 16) || !aligned(dbias, 4) || !aligned(workspace, 16))
        return MXFP8_ERR_ALIGN;
    const int64_t row_tiles = (M + kBM - 1) / kBM, col_tiles = (N + kBN - 1) / kBN;
    if (row_tiles * col_tiles >= (int64_t{1} << 31))
        return MXFP8_ERR_SHAPE;
    if (dbias != nullptr && workspace == nullptr && M > 0)
        return MXFP8_ERR_WORKSPACE;

    // ---- device checks ----
    int device = 0;
    if ((st = current_device(&device)) != MXFP8_OK)
        return st;
    if (!on_device(x, device) || !on_device(out_row, device) || !on_device(scale_row, device) ||
        !on_device(out_col, device) || !on_device(scale_col, device) || !on_device(dbias, device) ||
        !on_device(workspace, device) || !on_device(noop, device))
        return MXFP8_ERR_DEVICE;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);

    if (!empty) {
        st = enqueue_flat(device, fp8_fmt, x, M, N, out_row, scale_row, out_col, scale_col,
                          dbias != nullptr ? static_cast<float *>(workspace) : nullptr, noop, stream);
        if (st != MXFP8_OK)
            return st;
    }
    if (dbias != nullptr && N > 0) {
        st = enqueue_reduce(static_cast<const float *>(workspace), M > 0 ? row_tiles : 0, N, dbias, noop, stream);
        if (st != MXFP8_OK)
            return st;
    }
    return MXFP8_OK;
}

size_t mxfp8_scale_bytes(int64_t rows, int64_t scale_cols, int scale_layout)
{
    if (rows < 0 || scale_cols < 0)
        return 0;
    if (scale_layout == MXFP8_SCALES_PLAIN)
        return static_cast<size_t>(rows) * static_cast<size_t>(scale_cols);
    if (scale_layout == MXFP8_SCALES_SWIZZLED)
        return static_cast<size_t>((rows + 127) / 128 * 128) * static_cast<size_t>((scale_cols + 3) / 4 * 4);
    return 0;
}

mxfp8_status_t mxfp8_quantize_ex(const mxfp8_quantize_config_t *cfg, void *stream_)
{
    if (cfg == nullptr)
        return MXFP8_ERR_NULL;
    for (int r : cfg->reserved)
        if (r != 0)
            return MXFP8_ERR_FORMAT;
    if (cfg->scale_layout != MXFP8_SCALES_PLAIN && cfg->scale_layout != MXFP8_SCALES_SWIZZLED)
        return MXFP8_ERR_FORMAT;
    if (cfg->activation < MXFP8_ACT_NONE || cfg->activation > MXFP8_ACT_QGELU ||
        (cfg->activation != MXFP8_ACT_NONE && cfg->dbias != nullptr))
        return MXFP8_ERR_FORMAT;
    if (cfg->scale_layout == MXFP8_SCALES_PLAIN && cfg->amax == nullptr && cfg->activation == MXFP8_ACT_NONE)
        return mxfp8_quantize(cfg->x, cfg->M, cfg->N, cfg->fp8_fmt, cfg->out_row, cfg->scale_row, cfg->out_col,
                              cfg->scale_col, cfg->dbias, cfg->workspace, cfg->noop, stream_);

    const int64_t M = cfg->M, N = cfg->N;
    if (cfg->fp8_fmt != MXFP8_E4M3 && cfg->fp8_fmt != MXFP8_E5M2)
        return MXFP8_ERR_FORMAT;
    if (M < 0 || N < 0 || N % 8 || M >= (int64_t{1} << 31) || N >= (int64_t{1} << 31))
        return MXFP8_ERR_SHAPE;
    const bool swz = cfg->scale_layout == MXFP8_SCALES_SWIZZLED;
    const bool empty = M == 0 || N == 0;
    mxfp8_status_t st;
    if (!empty) {
        if (cfg->x == nullptr)
            return MXFP8_ERR_NULL;
        if ((cfg->out_row == nullptr) != (cfg->scale_row == nullptr) ||
            (cfg->out_col == nullptr) != (cfg->scale_col == nullptr) ||
            (cfg->out_row == nullptr && cfg->out_col == nullptr))
            return MXFP8_ERR_NULL;
    }
    if (!aligned(cfg->x, 16) || !aligned(cfg->out_row, 16) || !aligned(cfg->out_col, 16) ||
        (!swz && !aligned(cfg->scale_col, 4)) || !aligned(cfg->dbias, 4) || !aligned(cfg->workspace, 16) ||
        !aligned(cfg->amax, 4))
        return MXFP8_ERR_ALIGN;
    const int64_t row_tiles = (M + kBM - 1) / kBM, col_tiles = (N + kBN - 1) / kBN;
    if (row_tiles * col_tiles >= (int64_t{1} << 31))
        return MXFP8_ERR_SHAPE;
    if (cfg->dbias != nullptr && cfg->workspace == nullptr && M > 0)
        return MXFP8_ERR_WORKSPACE;
    int device = 0;
    if ((st = current_device(&device)) != MXFP8_OK)
        return st;
    if (!on_device(cfg->x, device) || !on_device(cfg->out_row, device) || !on_device(cfg->scale_row, device) ||
        !on_device(cfg->out_col, device) || !on_device(cfg->scale_col, device) || !on_device(cfg->dbias, device) ||
        !on_device(cfg->workspace, device) || !on_device(cfg->noop, device) || !on_device(cfg->amax, device))
        return MXFP8_ERR_DEVICE;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);

    if (cfg->amax != nullptr) {
        amax_init_kernel<<<1, 1, 0, stream>>>(cfg->amax, cfg->noop);
        g_launches.fetch_add(1, std::memory_order_relaxed);
    }
    if (cudaGetLastError() != cudaSuccess)
        return MXFP8_ERR_LAUNCH;
    if (!empty) {
        st = enqueue_flat(device, cfg->fp8_fmt, cfg->x, M, N, cfg->out_row, cfg->scale_row, cfg->out_col,
                          cfg->scale_col, cfg->dbias != nullptr ? static_cast<float *>(cfg->workspace) : nullptr,
                          cfg->noop, stream, swz, cfg->amax, cfg->activation);
        if (st != MXFP8_OK)
            return st;
    }
    if (cfg->dbias != nullptr && N > 0) {
        st = enqueue_reduce(static_cast<const float *>(cfg->workspace), M > 0 ? row_tiles : 0, N, cfg->dbias,
                            cfg->noop, stream);
        if (st != MXFP8_OK)
            return st;
    }
    return MXFP8_OK;
}

mxfp8_status_t mxfp8_quantize_grouped(const void *x, int64_t total_rows, int64_t N, int num_groups,
                                      const int64_t *offsets, int fp8_fmt, void *out_row, void *scale_row,
                                      void *out_col, void *scale_col, void *workspace, const float *noop,
                                      int *err_flag, void *stream_)
{
    (void)workspace;
    return grouped_impl(x, total_rows, N, num_groups, offsets, fp8_fmt, out_row, scale_row, out_col, scale_col,
                        nullptr, nullptr, noop, err_flag, static_cast<cudaStream_t>(stream_));
}

}  // extern "C"

namespace {

// The backward fusion's host checks and launches; with reduce false the dbias variant writes only
// its per-tile partial sums into workspace (the host pipeline reduces them once at its end).
mxfp8_status_t dact_impl(const void *grad, const void *act_input, int64_t M, int64_t N, int fp8_fmt, int activation,
                         void *out_row, void *scale_row, void *out_col, void *scale_col, float *dbias, void *workspace,
                         const float *noop, void *stream_, bool reduce)
{
    if (fp8_fmt != MXFP8_E4M3 && fp8_fmt != MXFP8_E5M2)
        return MXFP8_ERR_FORMAT;
    if (activation < MXFP8_ACT_RELU || activation > MXFP8_ACT_QGELU)
        return MXFP8_ERR_FORMAT;
    if (M < 0 || N < 0 || N % 8 || M >= (int64_t{1} << 31) || N >= (int64_t{1} << 31))
        return MXFP8_ERR_SHAPE;
    const bool empty = M == 0 || N == 0;
    mxfp8_status_t st;
    if (!empty) {
        if (grad == nullptr || act_input == nullptr)
            return MXFP8_ERR_NULL;
        if ((st = check_outputs(out_row, scale_row, out_col, scale_col)) != MXFP8_OK)
            return st;
    }
    if (!aligned(grad, 16) || !aligned(act_input, 16) || !aligned(dbias, 4) || !aligned(workspace, 16))
        return MXFP8_ERR_ALIGN;
    const int64_t row_tiles = (M + kBM - 1) / kBM, col_tiles = (N + kDBN - 1) / kDBN;
    if (row_tiles * col_tiles >= (int64_t{1} << 31))
        return MXFP8_ERR_SHAPE;
    if (dbias != nullptr && workspace == nullptr && M > 0)
        return MXFP8_ERR_WORKSPACE;
    int device = 0;
    if ((st = current_device(&device)) != MXFP8_OK)
        return st;
    if (!on_device(grad, device) || !on_device(act_input, device) || !on_device(out_row, device) ||
        !on_device(scale_row, device) || !on_device(out_col, device) || !on_device(scale_col, device) ||
        !on_device(dbias, device) || !on_device(workspace, device) || !on_device(noop, device))
        return MXFP8_ERR_DEVICE;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (!empty) {
        CUtensorMap map_g, map_x;
        if ((st = make_tensor_map(&map_g, grad, M, N)) != MXFP8_OK ||
            (st = make_tensor_map(&map_x, act_input, M, N)) != MXFP8_OK)
            return st;
        QuantParams p{};
        p.out_row = static_cast<uint8_t *>(out_row);
        p.scale_row = static_cast<uint8_t *>(scale_row);
        p.out_col = static_cast<uint8_t *>(out_col);
        p.scale_col = static_cast<uint8_t *>(scale_col);
        p.ws = dbias != nullptr ? static_cast<float *>(workspace) : nullptr;
        p.noop = noop;
        p.M = M;
        p.N = N;
        p.row_tiles = static_cast<int>(row_tiles);
        p.col_tiles = static_cast<int>(col_tiles);
        const bool db = dbias != nullptr;
        const int64_t tiles = row_tiles * col_tiles;
        switch (activation) {
        case MXFP8_ACT_RELU: st = launch_dact<1>(fp8_fmt, db, device, map_g, map_x, p, tiles, stream); break;
        case MXFP8_ACT_SRELU: st = launch_dact<2>(fp8_fmt, db, device, map_g, map_x, p, tiles, stream); break;
        case MXFP8_ACT_GELU: st = launch_dact<3>(fp8_fmt, db, device, map_g, map_x, p, tiles, stream); break;
        case MXFP8_ACT_SILU: st = launch_dact<4>(fp8_fmt, db, device, map_g, map_x, p, tiles, stream); break;
        default: st = launch_dact<5>(fp8_fmt, db, device, map_g, map_x, p, tiles, stream); break;
        }
        if (st != MXFP8_OK)
            return st;
    }
    if (reduce && dbias != nullptr && N > 0)
        return enqueue_reduce(static_cast<const float *>(workspace), M > 0 ? row_tiles : 0, N, dbias, noop, stream);
    return MXFP8_OK;
}

}  // namespace

extern "C" {

mxfp8_status_t mxfp8_quantize_dact(const void *grad, const void *act_input, int64_t M, int64_t N, int fp8_fmt,
                                   int activation, void *out_row, void *scale_row, void *out_col, void *scale_col,
                                   float *dbias, void *workspace, const float *noop, void *stream_)
{
    return dact_impl(grad, act_input, M, N, fp8_fmt, activation, out_row, scale_row, out_col, scale_col, dbias,
                     workspace, noop, stream_, true);
}

mxfp8_status_t mxfp8_quantize_gated(const void *x, int64_t M, int64_t N, int fp8_fmt, int activation, void *out_row,
                                    void *scale_row, void *out_col, void *scale_col, const float *noop,
                                    void *stream_)
{
    if (fp8_fmt != MXFP8_E4M3 && fp8_fmt != MXFP8_E5M2)
        return MXFP8_ERR_FORMAT;
    if (activation < MXFP8_ACT_RELU || activation > MXFP8_ACT_QGELU)
        return MXFP8_ERR_FORMAT;
    if (M < 0 || N < 0 || N % 8 || M >= (int64_t{1} << 31) || N >= (int64_t{1} << 30))
        return MXFP8_ERR_SHAPE;
    const bool empty = M == 0 || N == 0;
    mxfp8_status_t st;
    if (!empty) {
        if (x == nullptr)
            return MXFP8_ERR_NULL;
        if ((st = check_outputs(out_row, scale_row, out_col, scale_col)) != MXFP8_OK)
            return st;
    }
    if (!aligned(x, 16))
        return MXFP8_ERR_ALIGN;
    const int64_t row_tiles = (M + kBM - 1) / kBM, col_tiles = (N + kDBN - 1) / kDBN;
    if (row_tiles * col_tiles >= (int64_t{1} << 31))
        return MXFP8_ERR_SHAPE;
    int device = 0;
    if ((st = current_device(&device)) != MXFP8_OK)
        return st;
    if (!on_device(x, device) || !on_device(out_row, device) || !on_device(scale_row, device) ||
        !on_device(out_col, device) || !on_device(scale_col, device) || !on_device(noop, device))
        return MXFP8_ERR_DEVICE;
    if (empty)
        return MXFP8_OK;
    // a = columns 0 .. N-1 of x, b = columns N .. 2N-1 (16-byte aligned: N is a multiple of 8)
    CUtensorMap map_a, map_b;
    const void *b = static_cast<const uint16_t *>(x) + N;
    if ((st = make_tensor_map_pitch(&map_a, x, M, N, 2 * N)) != MXFP8_OK ||
        (st = make_tensor_map_pitch(&map_b, b, M, N, 2 * N)) != MXFP8_OK)
        return st;
    QuantParams p{};
    p.out_row = static_cast<uint8_t *>(out_row);
    p.scale_row = static_cast<uint8_t *>(scale_row);
    p.out_col = static_cast<uint8_t *>(out_col);
    p.scale_col = static_cast<uint8_t *>(scale_col);
    p.noop = noop;
    p.M = M;
    p.N = N;
    p.row_tiles = static_cast<int>(row_tiles);
    p.col_tiles = static_cast<int>(col_tiles);
    const int64_t tiles = row_tiles * col_tiles;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    switch (activation) {
    case MXFP8_ACT_RELU: return launch_gated<1>(fp8_fmt, device, map_b, map_a, p, tiles, stream);
    case MXFP8_ACT_SRELU: return launch_gated<2>(fp8_fmt, device, map_b, map_a, p, tiles, stream);
    case MXFP8_ACT_GELU: return launch_gated<3>(fp8_fmt, device, map_b, map_a, p, tiles, stream);
    case MXFP8_ACT_SILU: return launch_gated<4>(fp8_fmt, device, map_b, map_a, p, tiles, stream);
    default: return launch_gated<5>(fp8_fmt, device, map_b, map_a, p, tiles, stream);
    }
}

mxfp8_status_t mxfp8_quantize_grouped_swizzled(const void *x, int64_t total_rows, int64_t N, int num_groups,
                                               const int64_t *offsets, int fp8_fmt, int activation, void *out_row,
                                               void *scale_row, void *out_col, void *scale_col, const float *noop,
                                               int *err_flag, void *stream_)
{
    return grouped_impl(x, total_rows, N, num_groups, offsets, fp8_fmt, out_row, scale_row, out_col, scale_col,
                        nullptr, nullptr, noop, err_flag, static_cast<cudaStream_t>(stream_), activation, true);
}

size_t mxfp8_grouped_swizzled_scale_bytes(const int64_t *host_offsets, int num_groups, int64_t N, int colwise)
{
    if (host_offsets == nullptr || num_groups < 1 || num_groups > MXFP8_MAX_GROUPS || N < 0 || N % 8 ||
        host_offsets[0] != 0)
        return 0;
    int64_t tiles = 0;
    for (int g = 0; g < num_groups; ++g) {
        const int64_t rows = host_offsets[g + 1] - host_offsets[g];
        if (rows < 0)
            return 0;
        tiles += (rows + kBM - 1) / kBM;
    }
    const int64_t Cn = (N + 31) / 32;
    const int64_t per_tile = colwise ? 4 * ((N + 127) / 128 * 128) : 128 * ((Cn + 3) / 4 * 4);
    return static_cast<size_t>(tiles) * static_cast<size_t>(per_tile);
}

mxfp8_status_t mxfp8_quantize_grouped_activated(const void *x, int64_t total_rows, int64_t N, int num_groups,
                                                const int64_t *offsets, int fp8_fmt, int activation, void *out_row,
                                                void *scale_row, void *out_col, void *scale_col, const float *noop,
                                                int *err_flag, void *stream_)
{
    if (activation < MXFP8_ACT_RELU || activation > MXFP8_ACT_QGELU)
        return MXFP8_ERR_FORMAT;
    return grouped_impl(x, total_rows, N, num_groups, offsets, fp8_fmt, out_row, scale_row, out_col, scale_col,
                        nullptr, nullptr, noop, err_flag, static_cast<cudaStream_t>(stream_), activation);
}

mxfp8_status_t mxfp8_quantize_gated_grouped(const void *x, int64_t total_rows, int64_t N, int num_groups,
                                            const int64_t *offsets, int fp8_fmt, int activation, void *out_row,
                                            void *scale_row, void *out_col, void *scale_col, const float *noop,
                                            int *err_flag, void *stream_)
{
    if (fp8_fmt != MXFP8_E4M3 && fp8_fmt != MXFP8_E5M2)
        return MXFP8_ERR_FORMAT;
    if (activation < MXFP8_ACT_RELU || activation > MXFP8_ACT_QGELU)
        return MXFP8_ERR_FORMAT;
    if (total_rows < 0 || N < 0 || N % 8 || total_rows >= (int64_t{1} << 31) || N >= (int64_t{1} << 30))
        return MXFP8_ERR_SHAPE;
    if (num_groups < 1 || num_groups > MXFP8_MAX_GROUPS || offsets == nullptr)
        return MXFP8_ERR_GROUPS;
    if (x == nullptr)
        return MXFP8_ERR_NULL;
    mxfp8_status_t st = check_outputs(out_row, scale_row, out_col, scale_col);
    if (st != MXFP8_OK)
        return st;
    if (!aligned(x, 16) || !aligned(offsets, 8) || !aligned(err_flag, 4))
        return MXFP8_ERR_ALIGN;
    const int64_t col_tiles = (N + kDBN - 1) / kDBN;
    // every non-empty group adds at most one partial row tile
    const int64_t tile_bound = (total_rows / kBM + num_groups) * col_tiles;
    if (tile_bound >= (int64_t{1} << 31))
        return MXFP8_ERR_SHAPE;
    int device = 0;
    if ((st = current_device(&device)) != MXFP8_OK)
        return st;
    if (!on_device(x, device) || !on_device(offsets, device) || !on_device(out_row, device) ||
        !on_device(scale_row, device) || !on_device(out_col, device) || !on_device(scale_col, device) ||
        !on_device(noop, device) || !on_device(err_flag, device))
        return MXFP8_ERR_DEVICE;
    if (total_rows == 0 || N == 0)
        return MXFP8_OK;
    CUtensorMap map_a, map_b;
    const void *b = static_cast<const uint16_t *>(x) + N;  // 16-byte aligned: N is a multiple of 8
    if ((st = make_tensor_map_pitch(&map_a, x, total_rows, N, 2 * N)) != MXFP8_OK ||
        (st = make_tensor_map_pitch(&map_b, b, total_rows, N, 2 * N)) != MXFP8_OK)
        return st;
    QuantParams p{};
    p.out_row = static_cast<uint8_t *>(out_row);
    p.scale_row = static_cast<uint8_t *>(scale_row);
    p.out_col = static_cast<uint8_t *>(out_col);
    p.scale_col = static_cast<uint8_t *>(scale_col);
    p.noop = noop;
    p.offsets = offsets;
    p.err_flag = err_flag;
    p.M = total_rows;
    p.N = N;
    p.num_groups = num_groups;
    p.col_tiles = static_cast<int>(col_tiles);
    p.row_tiles = static_cast<int>((total_rows + kBM - 1) / kBM);  // the flat schedule (aligned groups)
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    switch (activation) {
    case MXFP8_ACT_RELU: return launch_gated<1, true>(fp8_fmt, device, map_b, map_a, p, tile_bound, stream);
    case MXFP8_ACT_SRELU: return launch_gated<2, true>(fp8_fmt, device, map_b, map_a, p, tile_bound, stream);
    case MXFP8_ACT_GELU: return launch_gated<3, true>(fp8_fmt, device, map_b, map_a, p, tile_bound, stream);
    case MXFP8_ACT_SILU: return launch_gated<4, true>(fp8_fmt, device, map_b, map_a, p, tile_bound, stream);
    default: return launch_gated<5, true>(fp8_fmt, device, map_b, map_a, p, tile_bound, stream);
    }
}

mxfp8_status_t mxfp8_quantize_dgated(const void *grad, const void *x, int64_t M, int64_t N, int fp8_fmt,
                                     int activation, void *out_row, void *scale_row, void *out_col,
                                     void *scale_col, const float *noop, void *stream_)
{
    if (fp8_fmt != MXFP8_E4M3 && fp8_fmt != MXFP8_E5M2)
        return MXFP8_ERR_FORMAT;
    if (activation < MXFP8_ACT_RELU || activation > MXFP8_ACT_QGELU)
        return MXFP8_ERR_FORMAT;
    if (M < 0 || N < 0 || N % 8 || M >= (int64_t{1} << 31) || N >= (int64_t{1} << 30))
        return MXFP8_ERR_SHAPE;
    const bool empty = M == 0 || N == 0;
    mxfp8_status_t st;
    if (!empty) {
        if (grad == nullptr || x == nullptr)
            return MXFP8_ERR_NULL;
        if ((st = check_outputs(out_row, scale_row, out_col, scale_col)) != MXFP8_OK)
            return st;
    }
    if (!aligned(grad, 16) || !aligned(x, 16))
        return MXFP8_ERR_ALIGN;
    const int tile_rows = activation != MXFP8_ACT_SRELU ? kKRows : kBM;  // see kKeepDgated
    const int64_t row_tiles = (M + tile_rows - 1) / tile_rows, col_tiles = (N + kDBN - 1) / kDBN;
    if (row_tiles * col_tiles >= (int64_t{1} << 31))
        return MXFP8_ERR_SHAPE;
    int device = 0;
    if ((st = current_device(&device)) != MXFP8_OK)
        return st;
    if (!on_device(grad, device) || !on_device(x, device) || !on_device(out_row, device) ||
        !on_device(scale_row, device) || !on_device(out_col, device) || !on_device(scale_col, device) ||
        !on_device(noop, device))
        return MXFP8_ERR_DEVICE;
    if (empty)
        return MXFP8_OK;
    CUtensorMap map_g, map_a, map_b;
    const void *b = static_cast<const uint16_t *>(x) + N;  // 16-byte aligned: N is a multiple of 8
    if ((st = make_tensor_map_pitch(&map_g, grad, M, N, N, tile_rows)) != MXFP8_OK ||
        (st = make_tensor_map_pitch(&map_a, x, M, N, 2 * N, tile_rows)) != MXFP8_OK ||
        (st = make_tensor_map_pitch(&map_b, b, M, N, 2 * N, tile_rows)) != MXFP8_OK)
        return st;
    QuantParams p{};
    p.out_row = static_cast<uint8_t *>(out_row);
    p.scale_row = static_cast<uint8_t *>(scale_row);
    p.out_col = static_cast<uint8_t *>(out_col);
    p.scale_col = static_cast<uint8_t *>(scale_col);
    p.noop = noop;
    p.M = M;
    p.N = N;
    p.row_tiles = static_cast<int>(row_tiles);
    p.col_tiles = static_cast<int>(col_tiles);
    const int64_t tiles = row_tiles * col_tiles;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    switch (activation) {
    case MXFP8_ACT_RELU: return launch_dgated<1>(fp8_fmt, device, map_g, map_a, map_b, p, tiles, stream);
    case MXFP8_ACT_SRELU: return launch_dgated<2>(fp8_fmt, device, map_g, map_a, map_b, p, tiles, stream);
    case MXFP8_ACT_GELU: return launch_dgated<3>(fp8_fmt, device, map_g, map_a, map_b, p, tiles, stream);
    case MXFP8_ACT_SILU: return launch_dgated<4>(fp8_fmt, device, map_g, map_a, map_b, p, tiles, stream);
    default: return launch_dgated<5>(fp8_fmt, device, map_g, map_a, map_b, p, tiles, stream);
    }
}

size_t mxfp8_quantize_grouped_dbias_workspace_bytes(int64_t total_rows, int64_t N, int num_groups)
{
    if (total_rows < 0 || N < 0 || num_groups < 1 || N % 8)
        return 0;
    return static_cast<size_t>(grouped_header_floats(num_groups)) * sizeof(float) +
           static_cast<size_t>((total_rows + kBM - 1) / kBM + num_groups) * static_cast<size_t>(N) * sizeof(float);
}

mxfp8_status_t mxfp8_quantize_grouped_dbias(const void *x, int64_t total_rows, int64_t N, int num_groups,
                                            const int64_t *offsets, int fp8_fmt, void *out_row, void *scale_row,
                                            void *out_col, void *scale_col, float *dbias, void *workspace,
                                            const float *noop, int *err_flag, void *stream_)
{
    if (dbias == nullptr)
        return MXFP8_ERR_NULL;
    if (workspace == nullptr && total_rows > 0)
        return MXFP8_ERR_WORKSPACE;
    return grouped_impl(x, total_rows, N, num_groups, offsets, fp8_fmt, out_row, scale_row, out_col, scale_col,
                        dbias, static_cast<float *>(workspace), noop, err_flag, static_cast<cudaStream_t>(stream_));
}

const char *mxfp8_status_string(int status)
{
    switch (status) {
    case MXFP8_OK: return "ok";
    case MXFP8_ERR_NULL: return "required pointer is NULL, a data/scale pair is half set, or no direction requested";
    case MXFP8_ERR_SHAPE: return "M must be >= 0, N a non-negative multiple of 8, both below 2^31";
    case MXFP8_ERR_ALIGN: return "x/out/workspace must be 16-byte aligned, scale_col/dbias 4-byte aligned";
    case MXFP8_ERR_FORMAT: return "fp8_fmt must be MXFP8_E4M3 (0) or MXFP8_E5M2 (1)";
    case MXFP8_ERR_WORKSPACE: return "dbias requested without a workspace";
    case MXFP8_ERR_DEVICE: return "no usable CUDA device, or a buffer is not on the current device";
    case MXFP8_ERR_LAUNCH: return "a CUDA call failed while preparing or launching a kernel";
    case MXFP8_ERR_GROUPS: return "num_groups out of range or offsets NULL";
    default: return "unknown status";
    }
}

uint64_t mxfp8_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"

namespace {

// Self-test of mbar_wait_bounded: the phase it waits for is never completed, so
// the wait expires and the expiry is recorded as a pipeline CTA records it.
__global__ void bounded_wait_selftest_kernel(uint64_t limit_ns, int *timed_out)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
        const bool ok = mbar_wait_bounded(smem_u32(&bar), 0, limit_ns);
        if (!ok)
            atomicOr(&g_fault_word, 1u);
        *timed_out = ok ? 0 : 1;
    }
}

// The fp32 value the cast kernels form from each BF16 input: act(x) through
// activation2 (the forward cast's only evaluation) or act'(x) through dactivation2
// (the backward fusion's), two inputs per thread as the kernels pair them.
template <int ACT, bool DERIV>
__global__ void activation_values_kernel(const uint16_t *__restrict__ x, int64_t n, float *__restrict__ out)
{
    const int64_t pairs = (n + 1) / 2;
    for (int64_t p = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; p < pairs;
         p += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t i = 2 * p;
        const bool two = i + 1 < n;
        const float a = __uint_as_float(static_cast<uint32_t>(x[i]) << 16);
        const float b = two ? __uint_as_float(static_cast<uint32_t>(x[i + 1]) << 16) : a;
        float ya, yb;
        if constexpr (DERIV)
            f2_unpack(dactivation2<ACT>(f2_pack(a, b)), ya, yb);
        else
            f2_unpack(activation2<ACT>(f2_pack(a, b)), ya, yb);
        out[i] = ya;
        if (two)
            out[i + 1] = yb;
    }
}

template <int ACT>
mxfp8_status_t launch_activation_values(const uint16_t *x, int64_t n, bool deriv, float *out, cudaStream_t stream)
{
    const int64_t pairs = (n + 1) / 2;
    const int64_t blocks64 = (pairs + 255) / 256;
    const unsigned blocks = static_cast<unsigned>(blocks64 < 4096 ? blocks64 : 4096);
    if (deriv)
        activation_values_kernel<ACT, true><<<blocks, 256, 0, stream>>>(x, n, out);
    else
        activation_values_kernel<ACT, false><<<blocks, 256, 0, stream>>>(x, n, out);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError() == cudaSuccess ? MXFP8_OK : MXFP8_ERR_LAUNCH;
}

}  // namespace

extern "C" {

mxfp8_status_t mxfp8_activation_values(const void *x, int64_t n, int activation, int derivative, float *out,
                                       void *stream)
{
    if (activation < MXFP8_ACT_RELU || activation > MXFP8_ACT_QGELU || (derivative != 0 && derivative != 1))
        return MXFP8_ERR_FORMAT;
    if (n < 0 || n >= (int64_t{1} << 40))
        return MXFP8_ERR_SHAPE;
    if (n == 0)
        return MXFP8_OK;
    if (x == nullptr || out == nullptr)
        return MXFP8_ERR_NULL;
    if (!aligned(x, 2) || !aligned(out, 4))
        return MXFP8_ERR_ALIGN;
    int device = 0;
    mxfp8_status_t st = current_device(&device);
    if (st != MXFP8_OK)
        return st;
    if (!on_device(x, device) || !on_device(out, device))
        return MXFP8_ERR_DEVICE;
    const uint16_t *xb = static_cast<const uint16_t *>(x);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool d = derivative != 0;
    switch (activation) {
    case MXFP8_ACT_RELU: return launch_activation_values<1>(xb, n, d, out, s);
    case MXFP8_ACT_SRELU: return launch_activation_values<2>(xb, n, d, out, s);
    case MXFP8_ACT_GELU: return launch_activation_values<3>(xb, n, d, out, s);
    case MXFP8_ACT_SILU: return launch_activation_values<4>(xb, n, d, out, s);
    default: return launch_activation_values<5>(xb, n, d, out, s);
    }
}

mxfp8_status_t mxfp8_selftest_bounded_wait(int64_t limit_ns, int *timed_out, void *stream)
{
    if (timed_out == nullptr)
        return MXFP8_ERR_NULL;
    if (limit_ns <= 0 || limit_ns > int64_t{10000000000})
        return MXFP8_ERR_SHAPE;
    int device = 0;
    mxfp8_status_t st = current_device(&device);
    if (st != MXFP8_OK)
        return st;
    if (!on_device(timed_out, device))
        return MXFP8_ERR_DEVICE;
    bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint64_t>(limit_ns),
                                                                                  timed_out);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError() == cudaSuccess ? MXFP8_OK : MXFP8_ERR_LAUNCH;
}

mxfp8_status_t mxfp8_device_fault_word(unsigned int *out, int clear)
{
    if (out == nullptr)
        return MXFP8_ERR_NULL;
    int device = 0;
    mxfp8_status_t st = current_device(&device);
    if (st != MXFP8_OK)
        return st;
    if (cudaMemcpyFromSymbol(out, g_fault_word, sizeof(unsigned int)) != cudaSuccess)
        return MXFP8_ERR_LAUNCH;
    if (clear) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(unsigned int)) != cudaSuccess)
            return MXFP8_ERR_LAUNCH;
    }
    return MXFP8_OK;
}

}  // extern "C"

// ---- dbias quantize without any allocation ------------------------------------
//
// For callers that cannot allocate device memory themselves: a plugin or callback
// that is handed only its input and output tensors and has no allocator or
// workspace to draw from, or code that must not allocate once it is running.
// The dbias workspace such a caller cannot provide lives in this file-scope device
// array instead: 8 MiB on each GPU where the library's device code is loaded (from
// the first use of its kernels, or of this call, on that device) until the process
// exits.

static __device__ __align__(256) unsigned char g_noalloc_scratch[MXFP8_NOALLOC_SCRATCH_BYTES];

namespace {
// Device address of g_noalloc_scratch per device (host code only holds a stand-in
// for the symbol, so the address is looked up once per device with it current).
void *g_noalloc_addr[kMaxDevices] = {};
std::mutex g_noalloc_mu;
}  // namespace

extern "C" {

mxfp8_status_t mxfp8_quantize_dbias_noalloc(const void *x, int64_t M, int64_t N, int fp8_fmt, void *out_row,
                                            void *scale_row, void *out_col, void *scale_col, float *dbias,
                                            const float *noop, void *stream)
{
    // the checks mxfp8_quantize makes first, in its order, then this call's own
    if (fp8_fmt != MXFP8_E4M3 && fp8_fmt != MXFP8_E5M2)
        return MXFP8_ERR_FORMAT;
    if (M < 0 || N < 0 || N % 8 || M >= (int64_t{1} << 31) || N >= (int64_t{1} << 31))
        return MXFP8_ERR_SHAPE;
    if (dbias == nullptr)
        return MXFP8_ERR_NULL;
    if (mxfp8_quantize_workspace_bytes(M, N, 1) > MXFP8_NOALLOC_SCRATCH_BYTES)
        return MXFP8_ERR_SHAPE;  // needs more than the static scratch array holds
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) {
        cudaGetLastError();
        return MXFP8_ERR_DEVICE;
    }
    if (device < 0 || device >= kMaxDevices)
        return MXFP8_ERR_DEVICE;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (g_noalloc_addr[device] == nullptr) {
            void *addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
                cudaGetLastError();
                return MXFP8_ERR_DEVICE;
            }
            g_noalloc_addr[device] = addr;
        }
        scratch = g_noalloc_addr[device];
    }
    // Every (row tile, column) entry of the workspace the call uses is written
    // before it is read, so nothing needs clearing between calls.
    return mxfp8_quantize(x, M, N, fp8_fmt, out_row, scale_row, out_col, scale_col, dbias, scratch, noop, stream);
}

}  // extern "C"

// ---- quantize from and to host memory, pipelined over row chunks ----------------
//
// Rows are cut into chunks of at most R rows (a multiple of 128, about 32 MiB of
// BF16); the first and last chunks ramp (R/8, R/4, R/2 ... R/2, R/4, R/8) so the
// copies that cannot overlap (the first upload, the last download) stay short.
// Chunk c goes through staging slot c % 3: host-to-device copy on an internal
// copy stream, the quantize kernel on the caller's stream, device-to-host copies
// of every requested output on a second internal copy stream.  Each arrow is an
// event wait, so the two copy directions and the kernels overlap.  With dbias,
// every chunk writes its 128-row tile partials into one workspace for the whole
// matrix and a single reduce runs after the last chunk, giving exactly the sums
// of the one-shot call.

namespace {

constexpr int64_t kHostChunkBytes = int64_t{32} << 20;  // BF16 bytes of x per full chunk (target)
constexpr int kHostSlots = 3;

size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

int64_t host_chunk_rows(int64_t M, int64_t N)
{
    int64_t r = (kHostChunkBytes / (2 * N)) / kBM * kBM;
    if (r < kBM)
        r = kBM;
    const int64_t m_up = (M + kBM - 1) / kBM * kBM;
    return r < m_up ? r : m_up;
}

// Chunk boundaries 0 = b[0] < b[1] < ... < b[k] = M; every b[i] < M is a multiple
// of 128 (so chunks start on dbias tiles) and no chunk exceeds R rows.
std::vector<int64_t> chunk_plan(int64_t M, int64_t R)
{
    std::vector<int64_t> ramp;
    for (int64_t d : {8, 4, 2}) {
        const int64_t r = R / d / kBM * kBM;
        if (r >= kBM)
            ramp.push_back(r);
    }
    int64_t ramp_rows = 0;
    for (int64_t r : ramp)
        ramp_rows += r;
    std::vector<int64_t> b{0};
    const int64_t M128 = M / kBM * kBM;  // the last chunk also takes the final M - M128 rows
    if (ramp.empty() || M128 <= 2 * ramp_rows + R) {  // no ramp (R < 256 rows) or too few rows for one
        for (int64_t r = R; r < M; r += R)
            b.push_back(r);
    } else {
        int64_t pos = 0;
        for (int64_t r : ramp)
            b.push_back(pos += r);
        const int64_t tail_start = M128 - ramp_rows;
        while (pos + R < tail_start)
            b.push_back(pos += R);
        if (pos < tail_start)
            b.push_back(pos = tail_start);
        for (auto it = ramp.rbegin(); it + 1 != ramp.rend(); ++it)
            b.push_back(pos += *it);
    }
    b.push_back(M);
    return b;
}

struct SlotLayout {
    size_t x, out_row, out_col, scale_row, scale_col, bytes;
};

// One chunk slot of R rows (a multiple of 128); with swz, the scale planes in the GEMM-ready
// layout (R rows x ceil(N/32) padded to 4 columns; ceil(N/128)*128 rows x R/32 columns).
SlotLayout slot_layout(int64_t R, int64_t N, bool swz = false)
{
    SlotLayout L;
    size_t o = 0;
    L.x = o;
    o += align256(static_cast<size_t>(R * N * 2));
    L.out_row = o;
    o += align256(static_cast<size_t>(R * N));
    L.out_col = o;
    o += align256(static_cast<size_t>(R * N));
    L.scale_row = o;
    const int64_t Cn = (N + 31) / 32;
    o += align256(static_cast<size_t>(swz ? R * ((Cn + 3) / 4 * 4) : R * Cn));
    L.scale_col = o;
    o += align256(static_cast<size_t>(swz ? (N + 127) / 128 * 128 * (R / 32) : R / 32 * N));
    L.bytes = o;
    return L;
}

struct HostPipe {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, end = nullptr, reduced = nullptr;
    cudaEvent_t h2d_done[kHostSlots] = {}, comp_done[kHostSlots] = {}, d2h_done[kHostSlots] = {};
};
HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mu;

// Streams and events of the host pipeline, created once per device (the device is current).
mxfp8_status_t host_pipe(int device, HostPipe **out)
{
    HostPipe &h = g_pipe[device];
    if (!h.ready) {
        const unsigned ef = cudaEventDisableTiming;
        bool ok = cudaStreamCreateWithFlags(&h.h2d, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&h.d2h, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&h.start, ef) == cudaSuccess &&
                  cudaEventCreateWithFlags(&h.end, ef) == cudaSuccess &&
                  cudaEventCreateWithFlags(&h.reduced, ef) == cudaSuccess;
        for (int k = 0; ok && k < kHostSlots; ++k)
            ok = cudaEventCreateWithFlags(&h.h2d_done[k], ef) == cudaSuccess &&
                 cudaEventCreateWithFlags(&h.comp_done[k], ef) == cudaSuccess &&
                 cudaEventCreateWithFlags(&h.d2h_done[k], ef) == cudaSuccess;
        if (!ok) {  // release whatever was created, so that a later call starts clean
            cudaGetLastError();
            for (cudaStream_t *s : {&h.h2d, &h.d2h})
                if (*s != nullptr) {
                    cudaStreamDestroy(*s);
                    *s = nullptr;
                }
            for (cudaEvent_t *e : {&h.start, &h.end, &h.reduced})
                if (*e != nullptr) {
                    cudaEventDestroy(*e);
                    *e = nullptr;
                }
            for (int k = 0; k < kHostSlots; ++k)
                for (cudaEvent_t *e : {&h.h2d_done[k], &h.comp_done[k], &h.d2h_done[k]})
                    if (*e != nullptr) {
                        cudaEventDestroy(*e);
                        *e = nullptr;
                    }
            cudaGetLastError();
            return MXFP8_ERR_LAUNCH;
        }
        h.ready = true;
    }
    *out = &h;
    return MXFP8_OK;
}

bool cuda_ok(cudaError_t e)
{
    if (e == cudaSuccess)
        return true;
    cudaGetLastError();
    return false;
}

// Device staging bytes of the flat host pipeline: three chunk slots, then (with dbias) the
// workspace of the whole matrix and an fp32 [N] vector, then (with amax) one fp32.
size_t host_staging_bytes(int64_t M, int64_t N, bool dbias, bool swz, bool amax)
{
    if (M <= 0 || N <= 0 || N % 8)
        return 0;
    size_t b = kHostSlots * slot_layout(host_chunk_rows(M, N), N, swz).bytes;
    if (dbias)
        b += align256(mxfp8_quantize_workspace_bytes(M, N, 1)) + align256(static_cast<size_t>(N) * 4);
    if (amax)
        b += 256;
    return b;
}

// The flat host pipeline (mxfp8_quantize_host, mxfp8_quantize_ex_host): x and the outputs in host
// memory, chunks of rows through three device slots.  act, swz and amax_host are the options of
// the config call; with swz the rowwise plane of a chunk is a contiguous run of whole tile rows of
// the matrix's plane, and the columnwise one a column band of it (one strided copy).
mxfp8_status_t host_pipeline(const void *x_host, int64_t M, int64_t N, int fp8_fmt, int act, bool swz,
                             void *out_row_host, void *scale_row_host, void *out_col_host, void *scale_col_host,
                             float *dbias_host, float *amax_host, void *staging, size_t staging_bytes,
                             void *stream_)
{
    if (fp8_fmt != MXFP8_E4M3 && fp8_fmt != MXFP8_E5M2)
        return MXFP8_ERR_FORMAT;
    if (M <= 0 || N <= 0 || N % 8 || M >= (int64_t{1} << 31) || N >= (int64_t{1} << 31))
        return MXFP8_ERR_SHAPE;
    if (x_host == nullptr || staging == nullptr)
        return MXFP8_ERR_NULL;
    mxfp8_status_t st = MXFP8_OK;
    if ((out_row_host == nullptr) != (scale_row_host == nullptr) ||
        (out_col_host == nullptr) != (scale_col_host == nullptr) ||
        (out_row_host == nullptr && out_col_host == nullptr))
        return MXFP8_ERR_NULL;
    if (!aligned(staging, 256))
        return MXFP8_ERR_ALIGN;
    if (staging_bytes < host_staging_bytes(M, N, dbias_host != nullptr, swz, amax_host != nullptr))
        return MXFP8_ERR_WORKSPACE;
    if ((M + kBM - 1) / kBM * ((N + kBN - 1) / kBN) >= (int64_t{1} << 31))
        return MXFP8_ERR_SHAPE;
    const int64_t row_tiles = (M + kBM - 1) / kBM;

    int device = 0;
    if ((st = current_device(&device)) != MXFP8_OK)
        return st;
    if (device < 0 || device >= kMaxDevices || !on_device(staging, device))
        return MXFP8_ERR_DEVICE;

    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe *hp = nullptr;
    if ((st = host_pipe(device, &hp)) != MXFP8_OK)
        return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const int64_t R = host_chunk_rows(M, N);
    const SlotLayout L = slot_layout(R, N, swz);
    unsigned char *base = static_cast<unsigned char *>(staging);
    float *ws = nullptr, *dbias_dev = nullptr;
    size_t tail = kHostSlots * L.bytes;  // after the slots: dbias workspace and vector, amax
    if (dbias_host != nullptr) {
        ws = reinterpret_cast<float *>(base + tail);
        tail += align256(mxfp8_quantize_workspace_bytes(M, N, 1));
        dbias_dev = reinterpret_cast<float *>(base + tail);
        tail += align256(static_cast<size_t>(N) * 4);
    }
    float *amax_dev = amax_host != nullptr ? reinterpret_cast<float *>(base + tail) : nullptr;
    const int64_t col_tiles = (N + kBN - 1) / kBN;  // GEMM-ready planes: tiles of 128 rows (or columns)
    const unsigned char *xh = static_cast<const unsigned char *>(x_host);

    if (!cuda_ok(cudaEventRecord(hp->start, stream)) || !cuda_ok(cudaStreamWaitEvent(hp->h2d, hp->start, 0)) ||
        !cuda_ok(cudaStreamWaitEvent(hp->d2h, hp->start, 0)))
        return MXFP8_ERR_LAUNCH;
    if (amax_dev != nullptr) {
        amax_init_kernel<<<1, 1, 0, stream>>>(amax_dev, nullptr);
        g_launches.fetch_add(1, std::memory_order_relaxed);
        if (cudaGetLastError() != cudaSuccess)
            return MXFP8_ERR_LAUNCH;
    }
    const std::vector<int64_t> plan = chunk_plan(M, R);
    const int64_t chunks = static_cast<int64_t>(plan.size()) - 1;
    for (int64_t c = 0; c < chunks; ++c) {
        const int k = static_cast<int>(c % kHostSlots);
        const int64_t row0 = plan[c], rows = plan[c + 1] - plan[c];
        unsigned char *slot = base + k * L.bytes;
        // host -> device, once the slot's previous outputs have left
        if (c >= kHostSlots && !cuda_ok(cudaStreamWaitEvent(hp->h2d, hp->d2h_done[k], 0)))
            return MXFP8_ERR_LAUNCH;
        if (!cuda_ok(cudaMemcpyAsync(slot + L.x, xh + row0 * N * 2, static_cast<size_t>(rows * N * 2),
                                     cudaMemcpyHostToDevice, hp->h2d)) ||
            !cuda_ok(cudaEventRecord(hp->h2d_done[k], hp->h2d)) ||
            !cuda_ok(cudaStreamWaitEvent(stream, hp->h2d_done[k], 0)))
            return MXFP8_ERR_LAUNCH;
        // quantize the chunk on the caller's stream
        const bool row = out_row_host != nullptr, col = out_col_host != nullptr;
        st = enqueue_flat(device, fp8_fmt, slot + L.x, rows, N, row ? slot + L.out_row : nullptr,
                          row ? slot + L.scale_row : nullptr, col ? slot + L.out_col : nullptr,
                          col ? slot + L.scale_col : nullptr, ws != nullptr ? ws + (row0 / kBM) * N : nullptr,
                          nullptr, stream, swz, amax_dev, act);
        if (st != MXFP8_OK)
            return st;
        if (!cuda_ok(cudaEventRecord(hp->comp_done[k], stream)) ||
            !cuda_ok(cudaStreamWaitEvent(hp->d2h, hp->comp_done[k], 0)))
            return MXFP8_ERR_LAUNCH;
        // device -> host of every requested output of the chunk
        bool ok = true;
        const int64_t rt0 = row0 / kBM, crt = (rows + kBM - 1) / kBM;  // the chunk's tile rows
        if (row) {
            ok = ok && cuda_ok(cudaMemcpyAsync(static_cast<unsigned char *>(out_row_host) + row0 * N, slot + L.out_row,
                                               static_cast<size_t>(rows * N), cudaMemcpyDeviceToHost, hp->d2h));
            const int64_t cr = (N + 31) / 32;
            if (swz)  // whole tile rows of the plane: col_tiles tiles of 512 bytes each
                ok = ok && cuda_ok(cudaMemcpyAsync(static_cast<unsigned char *>(scale_row_host) + rt0 * col_tiles * 512,
                                                   slot + L.scale_row, static_cast<size_t>(crt * col_tiles * 512),
                                                   cudaMemcpyDeviceToHost, hp->d2h));
            else
                ok = ok && cuda_ok(cudaMemcpyAsync(static_cast<unsigned char *>(scale_row_host) + row0 * cr,
                                                   slot + L.scale_row, static_cast<size_t>(rows * cr),
                                                   cudaMemcpyDeviceToHost, hp->d2h));
        }
        if (col) {
            ok = ok && cuda_ok(cudaMemcpyAsync(static_cast<unsigned char *>(out_col_host) + row0 * N, slot + L.out_col,
                                               static_cast<size_t>(rows * N), cudaMemcpyDeviceToHost, hp->d2h));
            if (swz)  // tile columns rt0 .. rt0 + crt of each of the plane's col_tiles tile rows
                ok = ok && cuda_ok(cudaMemcpy2DAsync(static_cast<unsigned char *>(scale_col_host) + rt0 * 512,
                                                     static_cast<size_t>(row_tiles * 512), slot + L.scale_col,
                                                     static_cast<size_t>(crt * 512), static_cast<size_t>(crt * 512),
                                                     static_cast<size_t>(col_tiles), cudaMemcpyDeviceToHost,
                                                     hp->d2h));
            else
                ok = ok && cuda_ok(cudaMemcpyAsync(static_cast<unsigned char *>(scale_col_host) + (row0 / 32) * N,
                                                   slot + L.scale_col, static_cast<size_t>(((rows + 31) / 32) * N),
                                                   cudaMemcpyDeviceToHost, hp->d2h));
        }
        if (!ok || !cuda_ok(cudaEventRecord(hp->d2h_done[k], hp->d2h)))
            return MXFP8_ERR_LAUNCH;
    }
    if (dbias_host != nullptr) {
        if ((st = enqueue_reduce(ws, row_tiles, N, dbias_dev, nullptr, stream)) != MXFP8_OK)
            return st;
        if (!cuda_ok(cudaEventRecord(hp->reduced, stream)) || !cuda_ok(cudaStreamWaitEvent(hp->d2h, hp->reduced, 0)) ||
            !cuda_ok(cudaMemcpyAsync(dbias_host, dbias_dev, static_cast<size_t>(N) * 4, cudaMemcpyDeviceToHost,
                                     hp->d2h)))
            return MXFP8_ERR_LAUNCH;
    }
    if (amax_dev != nullptr) {
        if (!cuda_ok(cudaEventRecord(hp->reduced, stream)) || !cuda_ok(cudaStreamWaitEvent(hp->d2h, hp->reduced, 0)) ||
            !cuda_ok(cudaMemcpyAsync(amax_host, amax_dev, 4, cudaMemcpyDeviceToHost, hp->d2h)))
            return MXFP8_ERR_LAUNCH;
    }
    // the caller's stream resumes once the last copy to the host is done
    if (!cuda_ok(cudaEventRecord(hp->end, hp->d2h)) || !cuda_ok(cudaStreamWaitEvent(stream, hp->end, 0)))
        return MXFP8_ERR_LAUNCH;
    return MXFP8_OK;
}

// The host pipeline of the two- and three-input calls (backward fusion, gated cast and its
// backward): up to two host inputs of b0 and b1 bytes per row, outputs of W bytes per row (the
// FP8 codes of each direction), SR bytes per row (row scales) and W bytes per 32 rows (column
// scales), all in the device calls' layouts.  Chunks of R rows (a multiple of 128) go through
// three slots as in the flat pipeline; enqueue(in0, in1, row0, rows, out_row, scale_row,
// out_col, scale_col) quantizes one chunk on the caller's stream.
struct RowsLayout {
    size_t in0, in1, out_row, out_col, scale_row, scale_col, bytes;
};

RowsLayout rows_layout(int64_t R, int64_t b0, int64_t b1, int64_t W, int64_t SR)
{
    RowsLayout L;
    size_t o = 0;
    L.in0 = o;
    o += align256(static_cast<size_t>(R * b0));
    L.in1 = o;
    o += align256(static_cast<size_t>(R * b1));
    L.out_row = o;
    o += align256(static_cast<size_t>(R * W));
    L.out_col = o;
    o += align256(static_cast<size_t>(R * W));
    L.scale_row = o;
    o += align256(static_cast<size_t>(R * SR));
    L.scale_col = o;
    o += align256(static_cast<size_t>(R / 32 * W));
    L.bytes = o;
    return L;
}

// Rows per chunk: about kHostChunkBytes of input, whole 128-row tiles.
int64_t rows_chunk(int64_t M, int64_t in_bytes_per_row)
{
    int64_t r = (kHostChunkBytes / in_bytes_per_row) / kBM * kBM;
    if (r < kBM)
        r = kBM;
    const int64_t m_up = (M + kBM - 1) / kBM * kBM;
    return r < m_up ? r : m_up;
}

template <class Enqueue>
mxfp8_status_t rows_pipeline(int device, cudaStream_t stream, const void *in0_host, int64_t b0, const void *in1_host,
                             int64_t b1, int64_t M, int64_t W, int64_t SR, void *out_row_host, void *scale_row_host,
                             void *out_col_host, void *scale_col_host, unsigned char *base, Enqueue &&enqueue)
{
    HostPipe *hp = nullptr;
    mxfp8_status_t st = host_pipe(device, &hp);
    if (st != MXFP8_OK)
        return st;
    const int64_t R = rows_chunk(M, b0 + b1);
    const RowsLayout L = rows_layout(R, b0, b1, W, SR);
    const unsigned char *h0 = static_cast<const unsigned char *>(in0_host);
    const unsigned char *h1 = static_cast<const unsigned char *>(in1_host);
    const bool row = out_row_host != nullptr, col = out_col_host != nullptr;
    if (!cuda_ok(cudaEventRecord(hp->start, stream)) || !cuda_ok(cudaStreamWaitEvent(hp->h2d, hp->start, 0)) ||
        !cuda_ok(cudaStreamWaitEvent(hp->d2h, hp->start, 0)))
        return MXFP8_ERR_LAUNCH;
    const std::vector<int64_t> plan = chunk_plan(M, R);
    const int64_t chunks = static_cast<int64_t>(plan.size()) - 1;
    for (int64_t c = 0; c < chunks; ++c) {
        const int k = static_cast<int>(c % kHostSlots);
        const int64_t row0 = plan[c], rows = plan[c + 1] - plan[c];
        unsigned char *slot = base + k * L.bytes;
        if (c >= kHostSlots && !cuda_ok(cudaStreamWaitEvent(hp->h2d, hp->d2h_done[k], 0)))
            return MXFP8_ERR_LAUNCH;
        if (!cuda_ok(cudaMemcpyAsync(slot + L.in0, h0 + row0 * b0, static_cast<size_t>(rows * b0),
                                     cudaMemcpyHostToDevice, hp->h2d)) ||
            (b1 > 0 && !cuda_ok(cudaMemcpyAsync(slot + L.in1, h1 + row0 * b1, static_cast<size_t>(rows * b1),
                                                cudaMemcpyHostToDevice, hp->h2d))) ||
            !cuda_ok(cudaEventRecord(hp->h2d_done[k], hp->h2d)) ||
            !cuda_ok(cudaStreamWaitEvent(stream, hp->h2d_done[k], 0)))
            return MXFP8_ERR_LAUNCH;
        st = enqueue(slot + L.in0, slot + L.in1, row0, rows, row ? slot + L.out_row : nullptr,
                     row ? slot + L.scale_row : nullptr, col ? slot + L.out_col : nullptr,
                     col ? slot + L.scale_col : nullptr);
        if (st != MXFP8_OK)
            return st;
        if (!cuda_ok(cudaEventRecord(hp->comp_done[k], stream)) ||
            !cuda_ok(cudaStreamWaitEvent(hp->d2h, hp->comp_done[k], 0)))
            return MXFP8_ERR_LAUNCH;
        bool ok = true;
        if (row) {
            ok = ok && cuda_ok(cudaMemcpyAsync(static_cast<unsigned char *>(out_row_host) + row0 * W, slot + L.out_row,
                                               static_cast<size_t>(rows * W), cudaMemcpyDeviceToHost, hp->d2h));
            ok = ok && cuda_ok(cudaMemcpyAsync(static_cast<unsigned char *>(scale_row_host) + row0 * SR,
                                               slot + L.scale_row, static_cast<size_t>(rows * SR),
                                               cudaMemcpyDeviceToHost, hp->d2h));
        }
        if (col) {
            ok = ok && cuda_ok(cudaMemcpyAsync(static_cast<unsigned char *>(out_col_host) + row0 * W, slot + L.out_col,
                                               static_cast<size_t>(rows * W), cudaMemcpyDeviceToHost, hp->d2h));
            ok = ok && cuda_ok(cudaMemcpyAsync(static_cast<unsigned char *>(scale_col_host) + (row0 / 32) * W,
                                               slot + L.scale_col, static_cast<size_t>(((rows + 31) / 32) * W),
                                               cudaMemcpyDeviceToHost, hp->d2h));
        }
        if (!ok || !cuda_ok(cudaEventRecord(hp->d2h_done[k], hp->d2h)))
            return MXFP8_ERR_LAUNCH;
    }
    return MXFP8_OK;
}

// The caller's stream resumes once the last copy to the host is done.
mxfp8_status_t rows_pipeline_end(int device, cudaStream_t stream)
{
    HostPipe *hp = nullptr;
    mxfp8_status_t st = host_pipe(device, &hp);
    if (st != MXFP8_OK)
        return st;
    if (!cuda_ok(cudaEventRecord(hp->end, hp->d2h)) || !cuda_ok(cudaStreamWaitEvent(stream, hp->end, 0)))
        return MXFP8_ERR_LAUNCH;
    return MXFP8_OK;
}

// Host checks shared by the three calls; `pointers` are the inputs, the staging buffer and the
// outputs as in the device calls.
mxfp8_status_t rows_host_checks(int fp8_fmt, int activation, int64_t M, int64_t N, int64_t n_limit, bool inputs_ok,
                                void *staging, void *out_row_host, void *scale_row_host, void *out_col_host,
                                void *scale_col_host, size_t staging_bytes, size_t need)
{
    if (fp8_fmt != MXFP8_E4M3 && fp8_fmt != MXFP8_E5M2)
        return MXFP8_ERR_FORMAT;
    if (activation < MXFP8_ACT_RELU || activation > MXFP8_ACT_QGELU)
        return MXFP8_ERR_FORMAT;
    if (M <= 0 || N <= 0 || N % 8 || M >= (int64_t{1} << 31) || N >= n_limit)
        return MXFP8_ERR_SHAPE;
    if (!inputs_ok || staging == nullptr)
        return MXFP8_ERR_NULL;
    if ((out_row_host == nullptr) != (scale_row_host == nullptr) ||
        (out_col_host == nullptr) != (scale_col_host == nullptr) ||
        (out_row_host == nullptr && out_col_host == nullptr))
        return MXFP8_ERR_NULL;
    if (!aligned(staging, 256))
        return MXFP8_ERR_ALIGN;
    if (staging_bytes < need)
        return MXFP8_ERR_WORKSPACE;
    return MXFP8_OK;
}

// Chunk boundaries of a grouped host call: the flat plan's, each interior one moved down to the
// nearest row a multiple of 32 rows after the start of the group that contains it.  A group cut
// by a boundary is then quantized as two pieces whose 32-row blocks are the group's own, so the
// chunks together give the one-shot call's bytes (each group is its own flat problem).  The flat
// plan's interior boundaries are at least 128 rows apart and move by less than 32, so they stay
// increasing, and a chunk holds at most R + 31 rows.  host_offsets are checked by the caller.
std::vector<int64_t> grouped_chunk_plan(const int64_t *off, int G, int64_t M, int64_t R)
{
    std::vector<int64_t> b = chunk_plan(M, R);
    int g = 0;
    for (size_t i = 1; i + 1 < b.size(); ++i) {
        while (g < G && off[g + 1] <= b[i])
            ++g;  // now off[g] <= b[i] < off[g + 1]
        b[i] = off[g] + (b[i] - off[g]) / 32 * 32;
    }
    return b;
}

// Device staging of one chunk of a grouped host call: up to Rcap rows of x and its outputs, the
// chunk's columnwise scale rows (at most Rcap/32 + G: each group piece rounds up once) and the
// chunk's group offsets.
struct GroupedSlotLayout {
    size_t x, out_row, out_col, scale_row, scale_col, off, bytes;
};

GroupedSlotLayout grouped_slot_layout(int64_t Rcap, int64_t N, int G)
{
    GroupedSlotLayout L;
    size_t o = 0;
    L.x = o;
    o += align256(static_cast<size_t>(Rcap * N * 2));
    L.out_row = o;
    o += align256(static_cast<size_t>(Rcap * N));
    L.out_col = o;
    o += align256(static_cast<size_t>(Rcap * N));
    L.scale_row = o;
    o += align256(static_cast<size_t>(Rcap * ((N + 31) / 32)));
    L.scale_col = o;
    o += align256(static_cast<size_t>((Rcap / 32 + G) * N));
    L.off = o;
    o += align256(static_cast<size_t>(G + 1) * 8);
    L.bytes = o;
    return L;
}

int64_t grouped_host_rcap(int64_t M, int64_t N) { return host_chunk_rows(M, N) + 32; }

// A chunk's group offsets, passed by value to a one-CTA kernel on the upload stream (so the
// upload needs no host staging buffer that must outlive the call).
constexpr int kOffsetPack = 257;
struct OffsetPack {
    int64_t v[kOffsetPack];
};

__global__ void fill_offsets_kernel(int64_t *dst, OffsetPack pack, int n)
{
    for (int i = threadIdx.x; i < n; i += blockDim.x)
        dst[i] = pack.v[i];
}

}  // namespace

extern "C" {

size_t mxfp8_quantize_host_staging_bytes(int64_t M, int64_t N, int with_dbias)
{
    return host_staging_bytes(M, N, with_dbias != 0, false, false);
}

mxfp8_status_t mxfp8_quantize_host(const void *x_host, int64_t M, int64_t N, int fp8_fmt, void *out_row_host,
                                   void *scale_row_host, void *out_col_host, void *scale_col_host,
                                   float *dbias_host, void *staging, size_t staging_bytes, void *stream_)
{
    return host_pipeline(x_host, M, N, fp8_fmt, MXFP8_ACT_NONE, false, out_row_host, scale_row_host, out_col_host,
                         scale_col_host, dbias_host, nullptr, staging, staging_bytes, stream_);
}

size_t mxfp8_quantize_ex_host_staging_bytes(const mxfp8_quantize_config_t *cfg)
{
    if (cfg == nullptr)
        return 0;
    return host_staging_bytes(cfg->M, cfg->N, cfg->dbias != nullptr, cfg->scale_layout == MXFP8_SCALES_SWIZZLED,
                              cfg->amax != nullptr);
}

mxfp8_status_t mxfp8_quantize_ex_host(const mxfp8_quantize_config_t *cfg, void *staging, size_t staging_bytes,
                                      void *stream_)
{
    if (cfg == nullptr)
        return MXFP8_ERR_NULL;
    for (int r : cfg->reserved)
        if (r != 0)
            return MXFP8_ERR_FORMAT;
    if (cfg->scale_layout != MXFP8_SCALES_PLAIN && cfg->scale_layout != MXFP8_SCALES_SWIZZLED)
        return MXFP8_ERR_FORMAT;
    if (cfg->activation < MXFP8_ACT_NONE || cfg->activation > MXFP8_ACT_QGELU ||
        (cfg->activation != MXFP8_ACT_NONE && cfg->dbias != nullptr))
        return MXFP8_ERR_FORMAT;
    // the workspace lives in the staging buffer; a skipped call would still copy stale bytes out
    if (cfg->workspace != nullptr || cfg->noop != nullptr)
        return MXFP8_ERR_FORMAT;
    return host_pipeline(cfg->x, cfg->M, cfg->N, cfg->fp8_fmt, cfg->activation,
                         cfg->scale_layout == MXFP8_SCALES_SWIZZLED, cfg->out_row, cfg->scale_row, cfg->out_col,
                         cfg->scale_col, cfg->dbias, cfg->amax, staging, staging_bytes, stream_);
}

size_t mxfp8_quantize_grouped_host_staging_bytes(int64_t total_rows, int64_t N, int num_groups)
{
    if (total_rows <= 0 || N <= 0 || N % 8 || num_groups < 1 || num_groups > MXFP8_MAX_GROUPS)
        return 0;
    return kHostSlots * grouped_slot_layout(grouped_host_rcap(total_rows, N), N, num_groups).bytes;
}

int64_t mxfp8_grouped_host_chunks(const int64_t *host_offsets, int num_groups, int64_t total_rows, int64_t N,
                                  int64_t *bounds, int64_t max_bounds)
{
    if (host_offsets == nullptr || num_groups < 1 || num_groups > MXFP8_MAX_GROUPS || total_rows <= 0 || N <= 0 ||
        N % 8 || host_offsets[0] != 0 || host_offsets[num_groups] != total_rows)
        return -1;
    for (int g = 0; g < num_groups; ++g)
        if (host_offsets[g + 1] < host_offsets[g])
            return -1;
    const std::vector<int64_t> b =
        grouped_chunk_plan(host_offsets, num_groups, total_rows, host_chunk_rows(total_rows, N));
    for (size_t i = 0; i < b.size() && static_cast<int64_t>(i) < max_bounds && bounds != nullptr; ++i)
        bounds[i] = b[i];
    return static_cast<int64_t>(b.size());
}

size_t mxfp8_quantize_dact_host_staging_bytes(int64_t M, int64_t N, int with_dbias)
{
    if (M <= 0 || N <= 0 || N % 8)
        return 0;
    const int64_t Cn = (N + 31) / 32;
    size_t b = kHostSlots * rows_layout(rows_chunk(M, 4 * N), 2 * N, 2 * N, N, Cn).bytes;
    if (with_dbias)
        b += align256(mxfp8_quantize_workspace_bytes(M, N, 1)) + align256(static_cast<size_t>(N) * 4);
    return b;
}

mxfp8_status_t mxfp8_quantize_dact_host(const void *grad_host, const void *act_input_host, int64_t M, int64_t N,
                                        int fp8_fmt, int activation, void *out_row_host, void *scale_row_host,
                                        void *out_col_host, void *scale_col_host, float *dbias_host, void *staging,
                                        size_t staging_bytes, void *stream_)
{
    mxfp8_status_t st = rows_host_checks(
        fp8_fmt, activation, M, N, int64_t{1} << 31, grad_host != nullptr && act_input_host != nullptr, staging,
        out_row_host, scale_row_host, out_col_host, scale_col_host, staging_bytes,
        mxfp8_quantize_dact_host_staging_bytes(M, N, dbias_host != nullptr));
    if (st != MXFP8_OK)
        return st;
    int device = 0;
    if ((st = current_device(&device)) != MXFP8_OK)
        return st;
    if (device < 0 || device >= kMaxDevices || !on_device(staging, device))
        return MXFP8_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const int64_t Cn = (N + 31) / 32;
    unsigned char *base = static_cast<unsigned char *>(staging);
    const size_t slots = kHostSlots * rows_layout(rows_chunk(M, 4 * N), 2 * N, 2 * N, N, Cn).bytes;
    float *ws = nullptr, *dbias_dev = nullptr;
    if (dbias_host != nullptr) {
        ws = reinterpret_cast<float *>(base + slots);
        dbias_dev = reinterpret_cast<float *>(base + slots + align256(mxfp8_quantize_workspace_bytes(M, N, 1)));
    }
    st = rows_pipeline(device, stream, grad_host, 2 * N, act_input_host, 2 * N, M, N, Cn, out_row_host,
                       scale_row_host, out_col_host, scale_col_host, base,
                       [&](unsigned char *g, unsigned char *x, int64_t row0, int64_t rows, void *orow, void *srow,
                           void *ocol, void *scol) {
                           // the dbias variant writes the chunk's tile partials; one reduce follows
                           return dact_impl(g, x, rows, N, fp8_fmt, activation, orow, srow, ocol, scol, dbias_dev,
                                            ws != nullptr ? ws + (row0 / kBM) * N : nullptr, nullptr, stream, false);
                       });
    if (st != MXFP8_OK)
        return st;
    if (dbias_host != nullptr) {
        HostPipe *hp = nullptr;
        if ((st = host_pipe(device, &hp)) != MXFP8_OK)
            return st;
        if ((st = enqueue_reduce(ws, (M + kBM - 1) / kBM, N, dbias_dev, nullptr, stream)) != MXFP8_OK)
            return st;
        if (!cuda_ok(cudaEventRecord(hp->reduced, stream)) || !cuda_ok(cudaStreamWaitEvent(hp->d2h, hp->reduced, 0)) ||
            !cuda_ok(cudaMemcpyAsync(dbias_host, dbias_dev, static_cast<size_t>(N) * 4, cudaMemcpyDeviceToHost,
                                     hp->d2h)))
            return MXFP8_ERR_LAUNCH;
    }
    return rows_pipeline_end(device, stream);
}

size_t mxfp8_quantize_gated_host_staging_bytes(int64_t M, int64_t N)
{
    if (M <= 0 || N <= 0 || N % 8)
        return 0;
    return kHostSlots * rows_layout(rows_chunk(M, 4 * N), 4 * N, 0, N, (N + 31) / 32).bytes;
}

mxfp8_status_t mxfp8_quantize_gated_host(const void *x_host, int64_t M, int64_t N, int fp8_fmt, int activation,
                                         void *out_row_host, void *scale_row_host, void *out_col_host,
                                         void *scale_col_host, void *staging, size_t staging_bytes, void *stream_)
{
    mxfp8_status_t st = rows_host_checks(fp8_fmt, activation, M, N, int64_t{1} << 30, x_host != nullptr, staging,
                                         out_row_host, scale_row_host, out_col_host, scale_col_host, staging_bytes,
                                         mxfp8_quantize_gated_host_staging_bytes(M, N));
    if (st != MXFP8_OK)
        return st;
    int device = 0;
    if ((st = current_device(&device)) != MXFP8_OK)
        return st;
    if (device < 0 || device >= kMaxDevices || !on_device(staging, device))
        return MXFP8_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    st = rows_pipeline(device, stream, x_host, 4 * N, nullptr, 0, M, N, (N + 31) / 32, out_row_host, scale_row_host,
                       out_col_host, scale_col_host, static_cast<unsigned char *>(staging),
                       [&](unsigned char *x, unsigned char *, int64_t, int64_t rows, void *orow, void *srow,
                           void *ocol, void *scol) {
                           return mxfp8_quantize_gated(x, rows, N, fp8_fmt, activation, orow, srow, ocol, scol,
                                                       nullptr, stream);
                       });
    return st != MXFP8_OK ? st : rows_pipeline_end(device, stream);
}

size_t mxfp8_quantize_dgated_host_staging_bytes(int64_t M, int64_t N)
{
    if (M <= 0 || N <= 0 || N % 8)
        return 0;
    return kHostSlots * rows_layout(rows_chunk(M, 6 * N), 2 * N, 4 * N, 2 * N, 2 * ((N + 31) / 32)).bytes;
}

mxfp8_status_t mxfp8_quantize_dgated_host(const void *grad_host, const void *x_host, int64_t M, int64_t N,
                                          int fp8_fmt, int activation, void *out_row_host, void *scale_row_host,
                                          void *out_col_host, void *scale_col_host, void *staging,
                                          size_t staging_bytes, void *stream_)
{
    mxfp8_status_t st = rows_host_checks(fp8_fmt, activation, M, N, int64_t{1} << 30,
                                         grad_host != nullptr && x_host != nullptr, staging, out_row_host,
                                         scale_row_host, out_col_host, scale_col_host, staging_bytes,
                                         mxfp8_quantize_dgated_host_staging_bytes(M, N));
    if (st != MXFP8_OK)
        return st;
    int device = 0;
    if ((st = current_device(&device)) != MXFP8_OK)
        return st;
    if (device < 0 || device >= kMaxDevices || !on_device(staging, device))
        return MXFP8_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    st = rows_pipeline(device, stream, grad_host, 2 * N, x_host, 4 * N, M, 2 * N, 2 * ((N + 31) / 32), out_row_host,
                       scale_row_host, out_col_host, scale_col_host, static_cast<unsigned char *>(staging),
                       [&](unsigned char *g, unsigned char *x, int64_t, int64_t rows, void *orow, void *srow,
                           void *ocol, void *scol) {
                           return mxfp8_quantize_dgated(g, x, rows, N, fp8_fmt, activation, orow, srow, ocol, scol,
                                                        nullptr, stream);
                       });
    return st != MXFP8_OK ? st : rows_pipeline_end(device, stream);
}

mxfp8_status_t mxfp8_quantize_grouped_host(const void *x_host, int64_t total_rows, int64_t N, int num_groups,
                                           const int64_t *host_offsets, int fp8_fmt, int activation,
                                           void *out_row_host, void *scale_row_host, void *out_col_host,
                                           void *scale_col_host, void *staging, size_t staging_bytes,
                                           void *stream_)
{
    if (fp8_fmt != MXFP8_E4M3 && fp8_fmt != MXFP8_E5M2)
        return MXFP8_ERR_FORMAT;
    if (activation < MXFP8_ACT_NONE || activation > MXFP8_ACT_QGELU)
        return MXFP8_ERR_FORMAT;
    if (total_rows <= 0 || N <= 0 || N % 8 || total_rows >= (int64_t{1} << 31) || N >= (int64_t{1} << 31))
        return MXFP8_ERR_SHAPE;
    if (num_groups < 1 || num_groups > MXFP8_MAX_GROUPS || host_offsets == nullptr)
        return MXFP8_ERR_GROUPS;
    // the offsets are on the host here, so a bad vector is rejected before any work
    if (host_offsets[0] != 0 || host_offsets[num_groups] != total_rows)
        return MXFP8_ERR_GROUPS;
    for (int g = 0; g < num_groups; ++g)
        if (host_offsets[g + 1] < host_offsets[g])
            return MXFP8_ERR_GROUPS;
    if (x_host == nullptr || staging == nullptr)
        return MXFP8_ERR_NULL;
    if ((out_row_host == nullptr) != (scale_row_host == nullptr) ||
        (out_col_host == nullptr) != (scale_col_host == nullptr) ||
        (out_row_host == nullptr && out_col_host == nullptr))
        return MXFP8_ERR_NULL;
    if (!aligned(staging, 256))
        return MXFP8_ERR_ALIGN;
    if (staging_bytes < mxfp8_quantize_grouped_host_staging_bytes(total_rows, N, num_groups))
        return MXFP8_ERR_WORKSPACE;

    int device = 0;
    mxfp8_status_t st = current_device(&device);
    if (st != MXFP8_OK)
        return st;
    if (device < 0 || device >= kMaxDevices || !on_device(staging, device))
        return MXFP8_ERR_DEVICE;

    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe *hp = nullptr;
    if ((st = host_pipe(device, &hp)) != MXFP8_OK)
        return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const GroupedSlotLayout L = grouped_slot_layout(grouped_host_rcap(total_rows, N), N, num_groups);
    unsigned char *base = static_cast<unsigned char *>(staging);
    const unsigned char *xh = static_cast<const unsigned char *>(x_host);
    const bool row = out_row_host != nullptr, col = out_col_host != nullptr;
    const int64_t Cn = (N + 31) / 32;

    if (!cuda_ok(cudaEventRecord(hp->start, stream)) || !cuda_ok(cudaStreamWaitEvent(hp->h2d, hp->start, 0)) ||
        !cuda_ok(cudaStreamWaitEvent(hp->d2h, hp->start, 0)))
        return MXFP8_ERR_LAUNCH;
    const std::vector<int64_t> plan =
        grouped_chunk_plan(host_offsets, num_groups, total_rows, host_chunk_rows(total_rows, N));
    const int64_t chunks = static_cast<int64_t>(plan.size()) - 1;
    int64_t s0 = 0;  // the chunk's first columnwise scale row
    OffsetPack pack;
    for (int64_t c = 0; c < chunks; ++c) {
        const int k = static_cast<int>(c % kHostSlots);
        const int64_t r0 = plan[c], r1 = plan[c + 1], rows = r1 - r0;
        unsigned char *slot = base + k * L.bytes;
        int64_t *off_dev = reinterpret_cast<int64_t *>(slot + L.off);
        // the slot is free once its previous outputs have left
        if (c >= kHostSlots && !cuda_ok(cudaStreamWaitEvent(hp->h2d, hp->d2h_done[k], 0)))
            return MXFP8_ERR_LAUNCH;
        // the chunk's offsets: every group's rows clipped to [r0, r1), relative to r0
        int64_t scale_rows = 0;
        for (int g0 = 0; g0 <= num_groups; g0 += kOffsetPack) {
            const int n = num_groups + 1 - g0 < kOffsetPack ? num_groups + 1 - g0 : kOffsetPack;
            for (int i = 0; i < n; ++i) {
                const int64_t o = host_offsets[g0 + i];
                pack.v[i] = (o < r0 ? r0 : o > r1 ? r1 : o) - r0;
            }
            fill_offsets_kernel<<<1, 256, 0, hp->h2d>>>(off_dev + g0, pack, n);
            g_launches.fetch_add(1, std::memory_order_relaxed);
        }
        for (int g = 0; g < num_groups; ++g) {
            const int64_t a = host_offsets[g] < r0 ? r0 : host_offsets[g] > r1 ? r1 : host_offsets[g];
            const int64_t e = host_offsets[g + 1] < r0 ? r0 : host_offsets[g + 1] > r1 ? r1 : host_offsets[g + 1];
            scale_rows += (e - a + 31) / 32;
        }
        if (!cuda_ok(cudaGetLastError()) ||
            !cuda_ok(cudaMemcpyAsync(slot + L.x, xh + r0 * N * 2, static_cast<size_t>(rows * N * 2),
                                     cudaMemcpyHostToDevice, hp->h2d)) ||
            !cuda_ok(cudaEventRecord(hp->h2d_done[k], hp->h2d)) ||
            !cuda_ok(cudaStreamWaitEvent(stream, hp->h2d_done[k], 0)))
            return MXFP8_ERR_LAUNCH;
        // the grouped cast of the chunk on the caller's stream
        st = grouped_impl(slot + L.x, rows, N, num_groups, off_dev, fp8_fmt, row ? slot + L.out_row : nullptr,
                          row ? slot + L.scale_row : nullptr, col ? slot + L.out_col : nullptr,
                          col ? slot + L.scale_col : nullptr, nullptr, nullptr, nullptr, nullptr, stream, activation);
        if (st != MXFP8_OK)
            return st;
        if (!cuda_ok(cudaEventRecord(hp->comp_done[k], stream)) ||
            !cuda_ok(cudaStreamWaitEvent(hp->d2h, hp->comp_done[k], 0)))
            return MXFP8_ERR_LAUNCH;
        bool ok = true;
        if (row) {
            ok = ok && cuda_ok(cudaMemcpyAsync(static_cast<unsigned char *>(out_row_host) + r0 * N, slot + L.out_row,
                                               static_cast<size_t>(rows * N), cudaMemcpyDeviceToHost, hp->d2h));
            ok = ok && cuda_ok(cudaMemcpyAsync(static_cast<unsigned char *>(scale_row_host) + r0 * Cn,
                                               slot + L.scale_row, static_cast<size_t>(rows * Cn),
                                               cudaMemcpyDeviceToHost, hp->d2h));
        }
        if (col) {
            ok = ok && cuda_ok(cudaMemcpyAsync(static_cast<unsigned char *>(out_col_host) + r0 * N, slot + L.out_col,
                                               static_cast<size_t>(rows * N), cudaMemcpyDeviceToHost, hp->d2h));
            ok = ok && cuda_ok(cudaMemcpyAsync(static_cast<unsigned char *>(scale_col_host) + s0 * N,
                                               slot + L.scale_col, static_cast<size_t>(scale_rows * N),
                                               cudaMemcpyDeviceToHost, hp->d2h));
        }
        if (!ok || !cuda_ok(cudaEventRecord(hp->d2h_done[k], hp->d2h)))
            return MXFP8_ERR_LAUNCH;
        s0 += scale_rows;
    }
    if (!cuda_ok(cudaEventRecord(hp->end, hp->d2h)) || !cuda_ok(cudaStreamWaitEvent(stream, hp->end, 0)))
        return MXFP8_ERR_LAUNCH;
    return MXFP8_OK;
}

}  // extern "C"
