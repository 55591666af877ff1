// api.cu -- the C ABI (include/sgemm.h): argument checks, the per-call plan,
// TMA tensor-map encoding, the device status word, and dispatch to the SIMT
// or tcgen05 launchers.  Nothing here allocates device memory.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/sgemm.h"
#include "common.cuh"
#include "internal.h"
#include "tune_table.h"

namespace sg {

// Device status word: set by kernels whose bounded waits run out.
__device__ unsigned int g_status_word;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    int num_sms = 0;
    int cc_major = 0, cc_minor = 0;
    unsigned int *status = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
std::atomic<int> g_default_mode{SGEMM_MODE_FP32};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Per-device facts, queried once with the device current.
const DeviceInfo *device_info(int *dev_out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    *dev_out = dev;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return nullptr;
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return nullptr;
        d.status = static_cast<unsigned int *>(addr);
        d.ready = true;
    }
    return &d;
}

struct SmemAttr {
    int dev;
    const void *kernel;
    int bytes;
};
std::mutex g_attr_mu;
std::vector<SmemAttr> g_attr;

bool get_encoder()
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode) return true;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return true;
}


// Scales C by beta (or zeroes it when beta == 0): the whole result when
// alpha == 0 or K == 0.  One thread per element, grid-stride.
__global__ void scale_c_kernel(float *C, int M, int N, long long ldc, long long sC, int Q,
                               float beta)
{
    const long long total = static_cast<long long>(Q) * M * N;
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long q = e / (static_cast<long long>(M) * N);
        const long long r = e - q * M * N;
        const long long i = r / N, j = r - i * N;
        float *c = C + q * sC + i * ldc + j;
        *c = (beta == 0.f) ? 0.f : beta * *c;
    }
}

// Split-K fix-up: for every split tile, sums its slices' partial tiles in
// slice order 0, 1, ..., splits-1 and writes C = alpha * sum + beta * C
// (C not read when beta == 0), masked at the M/N edges: the same result for
// the same inputs whatever order the slices ran in.  Block (x, y): split
// tile y, 256 consecutive float4 of it (one per thread).  It runs after the
// GEMM kernel on the same stream; when launched as a programmatic dependent
// it first waits for that kernel's completion and memory.
__global__ void __launch_bounds__(256) splitk_fixup_kernel(const GemmParams p, int bm, int bn)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int row_v4 = bn / 4;  // float4 per tile row
    const int tile_v4 = bm * row_v4;
    const int within = blockIdx.x * blockDim.x + threadIdx.x;
    if (within >= tile_v4) return;
    const long long sidx = blockIdx.y;
    const TileCoord tc = tile_coord(p.dp_tiles + sidx, p);
    const int r = within / row_v4, c = (within - r * row_v4) * 4;
    const int m = tc.tm * bm + r, n0 = tc.tn * bn + c;
    if (m >= p.M || n0 >= p.N) return;
    const float4 *slot = reinterpret_cast<const float4 *>(p.ws_part) +
                         sidx * p.splits * static_cast<long long>(tile_v4) + within;
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sl = 0; sl < p.splits; ++sl) {
        const float4 x = slot[static_cast<long long>(sl) * tile_v4];
        sum.x += x.x;
        sum.y += x.y;
        sum.z += x.z;
        sum.w += x.w;
    }
    const bool use_beta = p.beta != 0.f;
    float *crow = p.C + tc.q * p.sC + static_cast<long long>(m) * p.ldc;
    const float v[4] = {sum.x, sum.y, sum.z, sum.w};
    if (p.c_vec4 && n0 + 3 < p.N) {
        float4 o = make_float4(p.alpha * v[0], p.alpha * v[1], p.alpha * v[2], p.alpha * v[3]);
        float4 *dst = reinterpret_cast<float4 *>(crow + n0);
        if (use_beta) {
            const float4 old = *dst;
            o.x = fmaf(p.beta, old.x, o.x);
            o.y = fmaf(p.beta, old.y, o.y);
            o.z = fmaf(p.beta, old.z, o.z);
            o.w = fmaf(p.beta, old.w, o.w);
        }
        *dst = o;
    } else {
        for (int j = 0; j < 4 && n0 + j < p.N; ++j) {
            float o = p.alpha * v[j];
            if (use_beta) o = fmaf(p.beta, crow[n0 + j], o);
            crow[n0 + j] = o;
        }
    }
}

// Bounded-wait self test: one thread waits on an mbarrier that nobody arrives
// on, gives up after `limit` cycles, then completes the phase itself so the
// barrier is left in a clean state.
__global__ void wait_timeout_kernel(unsigned int *status, long long limit)
{
    __shared__ uint64_t bar;
    __shared__ int flag;
    mbar_init(&bar, 1);
    flag = 0;
    fence_mbar_init();
    const Abort ab{&flag, status, limit};
    mbar_wait(&bar, 0, ab, kStatusWaitTest);
    mbar_arrive(&bar);
}

}  // namespace

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(int M, int N, int K, float alpha, const void *A, int lda, const void *B, int ldb,
                const float *C, int ldc, int transA, int transB, long long sA, long long sB,
                long long sC, int Q)
{
    if (M < 0 || N < 0 || K < 0 || Q < 0) return SGEMM_ERR_INVALID_ARG;
    if (sA < 0 || sB < 0 || sC < 0) return SGEMM_ERR_INVALID_ARG;
    const long long a_row = transA ? M : K, b_row = transB ? K : N;
    if (lda < (a_row > 1 ? a_row : 1) || ldb < (b_row > 1 ? b_row : 1) || ldc < (N > 1 ? N : 1))
        return SGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0 || Q == 0) return SGEMM_OK;
    if (C == nullptr) return SGEMM_ERR_INVALID_ARG;
    if (Q > 1 && sC < static_cast<long long>(M - 1) * ldc + N) return SGEMM_ERR_INVALID_ARG;
    const bool reads_ab = (K > 0 && alpha != 0.f);
    if (reads_ab && (A == nullptr || B == nullptr)) return SGEMM_ERR_INVALID_ARG;
    return SGEMM_OK;
}

namespace {

int check_args(int mode, int M, int N, int K, float alpha, const float *A, int lda,
               const float *B, int ldb, float beta, float *C, int ldc, int transA, int transB,
               long long sA, long long sB, long long sC, int Q)
{
    (void)beta;
    if (mode != SGEMM_MODE_FP32 && mode != SGEMM_MODE_3XTF32 && mode != SGEMM_MODE_TF32)
        return SGEMM_ERR_INVALID_ARG;
    return check_shape(M, N, K, alpha, A, lda, B, ldb, C, ldc, transA, transB, sA, sB, sC, Q);
}

}  // namespace

namespace {
std::atomic<unsigned long long> g_launches{0};
}  // namespace

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

bool current_sm103(int *num_sms, unsigned int **status)
{
    int dev = 0;
    const DeviceInfo *di = device_info(&dev);
    if (di == nullptr || di->cc_major != 10 || di->cc_minor != 3) return false;
    *num_sms = di->num_sms;
    *status = di->status;
    return true;
}

namespace {

// Tensor maps already encoded, by their full description: a call that
// repeats pointers and shapes (the common case in a loop) takes the map from
// here instead of the driver (a map depends on nothing else, so an entry is
// never stale).  Direct-mapped, 128 entries.
struct MapKey {
    int dtype, swizzle, promo;
    const void *base;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
    bool operator==(const MapKey &o) const
    {
        return dtype == o.dtype && swizzle == o.swizzle && promo == o.promo && base == o.base &&
               std::memcmp(dims, o.dims, sizeof(dims)) == 0 &&
               std::memcmp(strides, o.strides, sizeof(strides)) == 0 &&
               std::memcmp(box, o.box, sizeof(box)) == 0;
    }
};
struct MapEntry {
    bool used = false;
    MapKey key;
    CUtensorMap map;
};
constexpr int kMapCache = 128;
std::mutex g_map_mu;
MapEntry g_maps[kMapCache];

size_t map_slot(const MapKey &k)
{
    uint64_t h = 1469598103934665603ull;
    auto mix = [&h](uint64_t v) { h = (h ^ v) * 1099511628211ull; };
    mix(static_cast<uint64_t>(k.dtype) | (static_cast<uint64_t>(k.swizzle) << 8) |
        (static_cast<uint64_t>(k.promo) << 16));
    mix(reinterpret_cast<uintptr_t>(k.base));
    for (int i = 0; i < 3; ++i) mix(k.dims[i] ^ (static_cast<uint64_t>(k.box[i]) << 40));
    for (int i = 0; i < 2; ++i) mix(k.strides[i]);
    return static_cast<size_t>(h % kMapCache);
}

// A rank-3 tiled map with unit element strides, no interleave and zero fill.
bool encode3(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
             const cuuint64_t (&dims)[3], const cuuint64_t (&strides)[2],
             const cuuint32_t (&box)[3], CUtensorMapSwizzle swizzle,
             CUtensorMapL2promotion promo)
{
    if (!get_encoder()) return false;
    MapKey k;
    std::memset(&k, 0, sizeof(k));
    k.dtype = static_cast<int>(dtype);
    k.swizzle = static_cast<int>(swizzle);
    k.promo = static_cast<int>(promo);
    k.base = base;
    std::memcpy(k.dims, dims, sizeof(k.dims));
    std::memcpy(k.strides, strides, sizeof(k.strides));
    std::memcpy(k.box, box, sizeof(k.box));
    const size_t slot = map_slot(k);
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        if (g_maps[slot].used && g_maps[slot].key == k) {
            *map = g_maps[slot].map;
            return true;
        }
    }
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(map, dtype, 3, const_cast<void *>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, promo,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    std::lock_guard<std::mutex> lk(g_map_mu);
    g_maps[slot].used = true;
    g_maps[slot].key = k;
    g_maps[slot].map = *map;
    return true;
}

}  // namespace

bool encode_operand(CUtensorMap *map, const float *base, bool kin, long long rows, long long K,
                    long long ld, int Q, long long stride, int box_rows, bool promote256)
{
    const bool batched = Q > 1 && stride != 0;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
    if (kin) {
        dims[0] = static_cast<cuuint64_t>(K);
        dims[1] = static_cast<cuuint64_t>(rows);
        box[0] = 32;
        box[1] = static_cast<cuuint32_t>(box_rows);
    } else {
        dims[0] = static_cast<cuuint64_t>(rows);
        dims[1] = static_cast<cuuint64_t>(K);
        box[0] = static_cast<cuuint32_t>(box_rows);
        box[1] = 32;
    }
    dims[2] = batched ? static_cast<cuuint64_t>(Q) : 1;
    box[2] = 1;
    strides[0] = static_cast<cuuint64_t>(ld) * 4;
    strides[1] = batched ? static_cast<cuuint64_t>(stride) * 4 : strides[0] * dims[1];
    return encode3(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, dims, strides, box,
                   kin ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   promote256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                              : CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
}

bool encode_operand_mn(CUtensorMap *map, const float *base, long long rows, long long K,
                       long long ld, int Q, long long stride, bool promote256)
{
    const bool batched = Q > 1 && stride != 0;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(K),
                          batched ? static_cast<cuuint64_t>(Q) : 1};
    cuuint64_t strides[2];
    strides[0] = static_cast<cuuint64_t>(ld) * 4;
    strides[1] = batched ? static_cast<cuuint64_t>(stride) * 4 : strides[0] * dims[1];
    cuuint32_t box[3] = {32, 32, 1};
    return encode3(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B,
                   promote256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                              : CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
}

bool encode_c_tiles(CUtensorMap *map, const float *C, long long M, long long N, long long ldc,
                    int Q, long long sC, int chunk_cols)
{
    const bool batched = Q > 1 && sC != 0;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M),
                          batched ? static_cast<cuuint64_t>(Q) : 1};
    cuuint64_t strides[2];
    strides[0] = static_cast<cuuint64_t>(ldc) * 4;
    strides[1] = batched ? static_cast<cuuint64_t>(sC) * 4 : strides[0] * dims[1];
    const bool wide = chunk_cols == 32;
    cuuint32_t box[3] = {wide ? 32u : 16u, 32, 1};
    return encode3(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, dims, strides, box,
                   wide ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
}

bool encode_operand16(CUtensorMap *map, const void *base, bool bf16, long long rows, long long K,
                      long long ld, int Q, long long stride, int box_rows)
{
    const bool batched = Q > 1 && stride != 0;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows),
                          batched ? static_cast<cuuint64_t>(Q) : 1};
    cuuint64_t strides[2];
    strides[0] = static_cast<cuuint64_t>(ld) * 2;
    strides[1] = batched ? static_cast<cuuint64_t>(stride) * 2 : strides[0] * dims[1];
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
    return encode3(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

bool smem_attr_once(const void *kernel, int bytes)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    for (const SmemAttr &a : g_attr)
        if (a.dev == dev && a.kernel == kernel && a.bytes >= bytes) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
        return false;
    g_attr.push_back(SmemAttr{dev, kernel, bytes});
    return true;
}

namespace {
std::atomic<int> g_force_route{kRouteAuto};
}  // namespace

int size_class(long long M, long long N, long long K, int Q)
{
    const double work = static_cast<double>(M) * N * K * (Q > 1 ? Q : 1);
    const int c = static_cast<int>(std::lround(std::log2(work > 1.0 ? work : 1.0) / 3.0));
    return c < kClassMin ? kClassMin : (c > kClassMax ? kClassMax : c);
}

namespace {
// A route the mode cannot take is the cost models' choice.
int applicable(int mode, int route)
{
    const bool fp32 = mode == SGEMM_MODE_FP32;
    if (route == kRouteSimtSmall) return fp32 ? route : kRouteAuto;
    if (route == kRouteTcPair || route == kRouteTcDirect || route == kRouteTcPlanes ||
        route == kRouteTcRaw || route == kRouteTcInline)
        return fp32 ? kRouteAuto : route;
    return kRouteAuto;
}
}  // namespace

int route_for(int mode, long long M, long long N, long long K, int Q)
{
    const int forced = g_force_route.load();
    if (forced == kRouteModels) return kRouteAuto;
    if (forced != kRouteAuto) return applicable(mode, forced);
    const int cls = size_class(M, N, K, Q);
    for (const TuneEntry &e : kTuneTable)
        if (e.mode == mode && e.size_class == cls && e.batched == (Q > 1 ? 1 : 0))
            return applicable(mode, e.route);
    return kRouteAuto;
}

int min_slice_k(int mode) { return mode == SGEMM_MODE_FP32 ? 64 : 256; }

// FLOP/s per multiprocessor each kernel sustains on GB300 (measured at
// 4092^3 with TMA-fed operands -- the FP32 kernel, the tensor-core pair
// kernel, the planes route's product alone -- and on the ragged
// 1000 x 1500 x 777 case, whose A TMA cannot describe: the FP32 kernel's
// cp.async fallback, the tensor-core direct kernel).
double path_rate_per_sm(int mode, int feed)
{
    if (mode == SGEMM_MODE_FP32) return feed == kFeedDirect ? 0.24e12 : 0.40e12;
    if (mode == SGEMM_MODE_3XTF32)
        return feed == kFeedDirect ? 0.47e12
               : feed == kFeedPlanes ? 2.45e12
               : feed == kFeedInline ? 2.35e12
                                     : 1.8e12;
    if (mode == kModeHalf) return 11.0e12;
    return feed == kFeedDirect ? 0.55e12 : feed == kFeedPlanes ? 6.4e12 : 3.6e12;
}

size_t splitk_workspace_bytes(long long split_tiles, int splits, int bm, int bn)
{
    if (splits <= 1 || split_tiles <= 0) return 0;
    return static_cast<size_t>(split_tiles) * splits * static_cast<size_t>(bm) * bn * sizeof(float);
}

namespace {
// The last plan's slice count (sgemm_last_split_count).
std::atomic<int> g_last_splits{1};
}  // namespace

SplitPlan choose_plan(long long num_tiles, int K, int slots, int mode, int bm, int bn, int feed,
                      size_t budget)
{
    SplitPlan best{1, num_tiles, 0, 0.0};
    if (num_tiles <= 0 || slots <= 0) return best;
    const int num_sms = slots;  // units running at once
    const long long full = num_tiles / num_sms, rem = num_tiles % num_sms;
    const double unit_rate =
        path_rate_per_sm(mode, feed) *
        ((feed == kFeedPair || feed == kFeedPlanes || feed == kFeedInline) ? 2 : 1);
    const double t_tile = 2.0 * bm * bn * static_cast<double>(K) / unit_rate;
    best.seconds = t_tile * static_cast<double>(full + (rem ? 1 : 0));
    if (rem == 0) return best;
    long long smax = K / min_slice_k(mode);
    if (smax > kMaxSplits) smax = kMaxSplits;
    const double t_whole = best.seconds;
    double best_t = t_whole;
    for (int s = 2; s <= smax; ++s) {
        const size_t ws = splitk_workspace_bytes(rem, s, bm, bn);
        if (ws > budget) continue;
        const long long waves = (rem * s + num_sms - 1) / num_sms;
        const double bw = ws <= (static_cast<size_t>(64) << 20) ? 8e12 : 3e12;
        const double t = t_tile * (static_cast<double>(full) + static_cast<double>(waves) / s) +
                         3e-6 + 2.0 * static_cast<double>(ws) / bw;
        if (t < best_t) {
            best_t = t;
            best = SplitPlan{s, full * num_sms, ws, t};
        }
    }
    if (best.splits > 1 && best_t > 0.99 * t_whole) best = SplitPlan{1, num_tiles, 0, t_whole};
    return best;
}

int plan_splits(Plan &plan, int bm, int bn, int feed, int slots)
{
    GemmParams &p = plan.p;
    p.splits = 1;
    p.dp_tiles = p.num_tiles;
    p.ws_part = nullptr;
    if (plan.ws != nullptr) {
        const SplitPlan sp =
            choose_plan(p.num_tiles, p.K, slots, plan.mode, bm, bn, feed, plan.ws_bytes);
        if (sp.splits > 1) {
            p.splits = sp.splits;
            p.dp_tiles = sp.dp_tiles;
            p.ws_part = static_cast<float *>(plan.ws);
        }
    }
    p.num_units = p.dp_tiles + (p.num_tiles - p.dp_tiles) * p.splits;
    g_last_splits.store(p.splits, std::memory_order_relaxed);
    return SGEMM_OK;
}

int launch_fixup(Plan &plan, int bm, int bn)
{
    const GemmParams &p = plan.p;
    const long long split_tiles = p.num_tiles - p.dp_tiles;
    if (split_tiles <= 0) return SGEMM_OK;
    if (split_tiles > 65535) return SGEMM_ERR_UNSUPPORTED;  // a split wave is < one per SM
    const int per_tile = (bm * bn / 4 + 255) / 256;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(per_tile), static_cast<unsigned>(split_tiles));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = plan.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, splitk_fixup_kernel, p, bm, bn) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    note_launch();
    return SGEMM_OK;
}

namespace {

// The plans of a call for every tile shape its mode may use (the FP32 path's
// depends on the operand layout, which the size queries do not take); the
// one needing the most workspace is reported, so that a workspace of that
// size serves the call whatever its layout.  one_wave: the allocation-free
// entry point's rule (see one_wave_plan).
SplitPlan plan_query(int mode, int M, int N, int K, int Q, bool one_wave)
{
    const SplitPlan none{1, 0, 0, 0.0};
    if (mode == SGEMM_MODE_DEFAULT) mode = g_default_mode.load();
    if (mode != SGEMM_MODE_FP32 && mode != SGEMM_MODE_3XTF32 && mode != SGEMM_MODE_TF32) return none;
    if (M <= 0 || N <= 0 || K <= 0 || Q <= 0) return none;
    int dev = 0;
    const DeviceInfo *di = device_info(&dev);
    if (di == nullptr) return none;
    const int sms = di->num_sms;
    SplitPlan out = none;
    // Whether the operands go through TMA depends on pointers and leading
    // dimensions the query does not take: plan for every kernel the mode
    // may run (FP32: the two tile shapes, each TMA-fed or not; tensor
    // cores: the direct kernel's 128 x 128 tiles, the pair kernel's 256 x 128).
    const bool small = mode == SGEMM_MODE_FP32 && route_for(mode, M, N, K, Q) == kRouteSimtSmall;
    for (int shape = 0; shape < (mode == SGEMM_MODE_FP32 ? (small ? 3 : 2) : 3); ++shape) {
        int bm = 0, bn = 0, slots = sms;
        int feeds[2] = {kFeedDirect, kFeedTma};
        if (mode == SGEMM_MODE_FP32) {
            if (shape == 2) simt_small_tile_dims(bm, bn);
            else simt_tile_dims(shape == 1, bm, bn);
        } else if (shape == 2) {  // the planes and raw routes' 256 x 256 pair tiles
            bm = bn = 256;
            slots = tc_pair_slots(sms);
            feeds[0] = kFeedPlanes;
            feeds[1] = mode == SGEMM_MODE_3XTF32 ? kFeedInline : kFeedPlanes;
        } else {
            tc_tile_dims(mode, K, shape == 1, bm, bn);
            if (shape == 1) {
                slots = tc_pair_slots(sms);
                feeds[0] = feeds[1] = kFeedPair;
            } else {
                feeds[1] = kFeedDirect;
            }
        }
        const long long tiles =
            static_cast<long long>(Q) * ((M + bm - 1) / bm) * ((N + bn - 1) / bn);
        SplitPlan sp{1, tiles, 0, 0.0};
        if (!one_wave) {
            for (int f = 0; f < 2; ++f) {
                const SplitPlan t =
                    choose_plan(tiles, K, slots, mode, bm, bn, feeds[f], ~static_cast<size_t>(0));
                if (t.ws_bytes > sp.ws_bytes) sp = t;
            }
        } else if (2 * tiles <= slots) {
            long long s = slots / tiles;
            const long long by_k = K / min_slice_k(mode);
            if (s > by_k) s = by_k;
            if (s > kMaxSplits) s = kMaxSplits;
            if (s >= 2)
                sp = SplitPlan{static_cast<int>(s), 0,
                               splitk_workspace_bytes(tiles, static_cast<int>(s), bm, bn), 0.0};
        }
        if (sp.ws_bytes > out.ws_bytes) out = sp;
    }
    return out;
}

}  // namespace

SplitPlan preferred_plan(int mode, int M, int N, int K, int Q)
{
    return plan_query(mode, M, N, K, Q, false);
}

SplitPlan one_wave_plan(int mode, int M, int N, int K, int Q)
{
    return plan_query(mode, M, N, K, Q, true);
}

}  // namespace sg

using namespace sg;

namespace {

// TMA can describe an operand when its base is 16-byte aligned and its row
// pitch and batch stride are multiples of 16 bytes.
bool tma_eligible(const float *p, long long ld, int Q, long long stride)
{
    if (!aligned16(p) || (ld % 4) != 0) return false;
    if (Q > 1 && stride != 0 && (stride % 4) != 0) return false;
    return true;
}

size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// Workspace a transposed copy of an operand takes: `outer` rows of
// round_up(inner, 4) floats per batch entry (one entry when broadcast).
size_t repack_bytes(long long inner, long long outer, int Q, bool broadcast)
{
    const long long ld = (inner + 3) / 4 * 4;
    return round256(static_cast<size_t>(broadcast ? 1 : Q) * static_cast<size_t>(outer) *
                    static_cast<size_t>(ld) * sizeof(float));
}

// FP32 path with a workspace: copies a K-inner A (when N >= kRepackMinN) and
// a K-inner B (when M >= kRepackMinM) into the front of the workspace,
// transposed, so that the product runs with A M-inner and B N-inner, the
// layout the FP32 kernel runs fastest (measured on GB300 at 4092^3: 69.2
// TFLOP/s against 64.2 with K-inner A, 55.9 with both K-inner).  The copy
// reads and writes the operand once; below the thresholds it costs more
// than it saves.  What remains of the workspace goes to the split plan.
int repack_for_simt(Plan &plan)
{
    GemmParams &p = plan.p;
    if (plan.ws == nullptr || plan.ws_bytes == 0) return SGEMM_OK;
    const bool want_a = !plan.transA && p.N >= kRepackMinN;
    const bool want_b = plan.transB && p.M >= kRepackMinM;
    const size_t a_bytes = want_a ? repack_bytes(p.M, p.K, p.Q, p.Q > 1 && p.sA == 0) : 0;
    const size_t b_bytes = want_b ? repack_bytes(p.N, p.K, p.Q, p.Q > 1 && p.sB == 0) : 0;
    bool do_a = want_a, do_b = want_b;
    if (a_bytes + b_bytes > plan.ws_bytes) {
        do_b = false;
        if (a_bytes > plan.ws_bytes) do_a = false;
    }
    if (!do_a && !do_b) return SGEMM_OK;
    char *w = static_cast<char *>(plan.ws);
    size_t used = 0;
    if (do_a) {
        // A (M x K, lda) -> A' stored K x M: op(A)[i][k] = A'[k * lda' + i]
        const long long ld = (p.M + 3) / 4 * 4;
        const int qa = (p.Q > 1 && p.sA == 0) ? 1 : p.Q;
        float *dst = reinterpret_cast<float *>(w + used);
        const int rc = launch_transpose(p.A, p.lda, p.sA, p.M, p.K, qa, dst, ld,
                                        static_cast<long long>(p.K) * ld, plan.num_sms, plan.stream);
        if (rc != SGEMM_OK) return rc;
        p.A = dst;
        p.lda = ld;
        p.sA = qa == 1 ? 0 : static_cast<long long>(p.K) * ld;
        p.a_vec4 = 1;
        plan.a_tma = true;
        plan.transA = true;
        used += a_bytes;
    }
    if (do_b) {
        // B stored N x K (ldb) -> B' stored K x N: op(B)[k][j] = B'[k * ldb' + j]
        const long long ld = (p.N + 3) / 4 * 4;
        const int qb = (p.Q > 1 && p.sB == 0) ? 1 : p.Q;
        float *dst = reinterpret_cast<float *>(w + used);
        const int rc = launch_transpose(p.B, p.ldb, p.sB, p.N, p.K, qb, dst, ld,
                                        static_cast<long long>(p.K) * ld, plan.num_sms, plan.stream);
        if (rc != SGEMM_OK) return rc;
        p.B = dst;
        p.ldb = ld;
        p.sB = qb == 1 ? 0 : static_cast<long long>(p.K) * ld;
        p.b_vec4 = 1;
        plan.b_tma = true;
        plan.transB = false;
        used += b_bytes;
    }
    plan.ws = used < plan.ws_bytes ? static_cast<void *>(w + used) : nullptr;
    plan.ws_bytes = used < plan.ws_bytes ? plan.ws_bytes - used : 0;
    return SGEMM_OK;
}

// Whether copying the operands TMA cannot describe pays for a call: the
// direct kernel's modelled time on the operands as they are, against the
// copies' (each operand read and written at HBM rate, ~4 us of launch and
// drain per copy) plus the pair kernel's.  Tiny problems keep the direct
// kernel: one launch instead of three.
bool repack_pays(const Plan &plan)
{
    const GemmParams &p = plan.p;
    const size_t any = ~static_cast<size_t>(0);
    int bm = 0, bn = 0;
    tc_tile_dims(plan.mode, p.K, false, bm, bn);
    long long tiles = static_cast<long long>(p.Q) * ((p.M + bm - 1) / bm) * ((p.N + bn - 1) / bn);
    const double t_direct =
        choose_plan(tiles, p.K, plan.num_sms, plan.mode, bm, bn, kFeedDirect, any).seconds;
    tc_tile_dims(plan.mode, p.K, true, bm, bn);
    tiles = static_cast<long long>(p.Q) * ((p.M + bm - 1) / bm) * ((p.N + bn - 1) / bn);
    double t = choose_plan(tiles, p.K, tc_pair_slots(plan.num_sms), plan.mode, bm, bn, kFeedPair,
                           any)
                   .seconds;
    if (!plan.a_tma) t += 4e-6 + 2.0 * 4.0 * p.Q * static_cast<double>(p.M) * p.K / 6.0e12;
    if (!plan.b_tma) t += 4e-6 + 2.0 * 4.0 * p.Q * static_cast<double>(p.N) * p.K / 6.0e12;
    return t < t_direct;
}

// Tensor-core paths with a workspace: an operand TMA cannot describe (row
// pitch or batch stride not a multiple of 16 bytes, unaligned base) is
// copied, in its own layout, into the workspace with rows padded to whole
// 128-byte lines, so that the product runs on the TMA-fed pair kernel
// instead of the direct-load one (measured on GB300, the ragged
// 1000 x 1500 x 777 case, lda = 777: 3xTF32 45.5 -> 74.3 TFLOP/s).  The
// cost models decide unless the caller forced the pair route (`force`).  What
// remains of the workspace goes to the split plan; without room for the
// copy the operand stays where it is and the direct kernel runs.
int repack_for_tc(Plan &plan, bool force)
{
    GemmParams &p = plan.p;
    if (plan.ws == nullptr || plan.ws_bytes == 0 || (plan.a_tma && plan.b_tma)) return SGEMM_OK;
    if (!force && !repack_pays(plan)) return SGEMM_OK;
    char *w = static_cast<char *>(plan.ws);
    size_t used = 0;
    for (int which = 0; which < 2; ++which) {
        const bool is_a = which == 0;
        if (is_a ? plan.a_tma : plan.b_tma) continue;
        // stored rows x row length of the operand as the caller holds it
        const bool trans = is_a ? plan.transA : plan.transB;
        const long long rows = is_a ? (trans ? p.K : p.M) : (trans ? p.N : p.K);
        const long long len = is_a ? (trans ? p.M : p.K) : (trans ? p.K : p.N);
        const long long ld = (len + 31) / 32 * 32;
        const long long stride = is_a ? p.sA : p.sB;
        const int q = (p.Q > 1 && stride == 0) ? 1 : p.Q;
        const size_t bytes = round256(static_cast<size_t>(q) * rows * ld * sizeof(float));
        if (used + bytes > plan.ws_bytes) continue;
        float *dst = reinterpret_cast<float *>(w + used);
        const float *src = is_a ? p.A : p.B;
        const long long lds = is_a ? p.lda : p.ldb;
        const int rc = launch_repack16(reinterpret_cast<const uint16_t *>(src), 2 * lds, 2 * stride,
                                       static_cast<int>(rows), static_cast<int>(2 * len), q, false,
                                       reinterpret_cast<uint16_t *>(dst), 2 * ld, 2 * rows * ld,
                                       plan.stream);
        if (rc != SGEMM_OK) return rc;
        if (is_a) {
            p.A = dst;
            p.lda = ld;
            p.sA = q == 1 ? 0 : rows * ld;
            p.a_q_step = q == 1 ? 0 : 1;
            p.a_vec4 = 1;
            plan.a_tma = true;
        } else {
            p.B = dst;
            p.ldb = ld;
            p.sB = q == 1 ? 0 : rows * ld;
            p.b_q_step = q == 1 ? 0 : 1;
            p.b_vec4 = 1;
            plan.b_tma = true;
        }
        used += bytes;
    }
    plan.ws = used < plan.ws_bytes ? static_cast<void *>(w + used) : nullptr;
    plan.ws_bytes = used < plan.ws_bytes ? plan.ws_bytes - used : 0;
    return SGEMM_OK;
}

int run(int mode, int M, int N, int K, float alpha, const float *A, int lda, const float *B,
        int ldb, float beta, float *C, int ldc, int transA, int transB, long long sA,
        long long sB, long long sC, int Q, void *stream, void *ws = nullptr,
        size_t ws_bytes = 0)
{
    if (mode == SGEMM_MODE_DEFAULT) mode = g_default_mode.load();
    int rc = check_args(mode, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, transA, transB, sA,
                        sB, sC, Q);
    if (rc != SGEMM_OK || M == 0 || N == 0 || Q == 0) return rc;

    int dev = 0;
    const DeviceInfo *di = device_info(&dev);
    if (di == nullptr) return SGEMM_ERR_UNSUPPORTED;
    if (di->cc_major != 10 || di->cc_minor != 3) return SGEMM_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    if (K == 0 || alpha == 0.f) {
        const long long total = static_cast<long long>(Q) * M * N;
        long long blocks = (total + 255) / 256;
        if (blocks > 8LL * di->num_sms) blocks = 8LL * di->num_sms;
        scale_c_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(C, M, N, ldc, sC, Q, beta);
        if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
        note_launch();
        return SGEMM_OK;
    }

    Plan plan{};
    GemmParams &p = plan.p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.Q = Q;
    p.alpha = alpha;
    p.beta = beta;
    p.A = A;
    p.B = B;
    p.C = C;
    p.lda = lda;
    p.ldb = ldb;
    p.ldc = ldc;
    p.sA = Q > 1 ? sA : 0;
    p.sB = Q > 1 ? sB : 0;
    p.sC = Q > 1 ? sC : 0;
    p.a_q_step = (Q > 1 && sA != 0) ? 1 : 0;
    p.b_q_step = (Q > 1 && sB != 0) ? 1 : 0;
    p.a_vec4 = aligned16(A) && lda % 4 == 0 && (p.sA % 4) == 0;
    p.b_vec4 = aligned16(B) && ldb % 4 == 0 && (p.sB % 4) == 0;
    p.c_vec4 = aligned16(C) && ldc % 4 == 0 && (p.sC % 4) == 0;
    p.status = di->status;
    p.wait_limit = kWaitLimitCycles;
    plan.transA = transA != 0;
    plan.transB = transB != 0;
    plan.mode = mode;
    plan.a_tma = tma_eligible(A, lda, Q, p.sA);
    plan.b_tma = tma_eligible(B, ldb, Q, p.sB);
    plan.num_sms = di->num_sms;
    plan.device = dev;
    plan.stream = st;
    plan.ws = ws;
    plan.ws_bytes = ws_bytes;

    const int route = route_for(mode, M, N, K, Q);
    if (mode == SGEMM_MODE_FP32) {
        if (route == kRouteSimtSmall) return launch_simt(plan, route);
        rc = repack_for_simt(plan);
        if (rc != SGEMM_OK) return rc;
        return launch_simt(plan, kRouteAuto);
    }
    bool taken = false;
    if (route == kRouteAuto || route == kRouteTcRaw || route == kRouteTcInline) {
        rc = run_raw(plan, taken, route != kRouteAuto, route);
        if (taken || rc != SGEMM_OK) return rc;
    }
    if (route == kRouteAuto || route == kRouteTcPlanes) {
        rc = run_planes(plan, taken, route == kRouteTcPlanes);
        if (taken || rc != SGEMM_OK) return rc;
    }
    if (route != kRouteTcDirect) {  // the direct kernel reads any layout as it is
        // the tuning table's pair route was measured on TMA-fed operands: only a
        // caller's explicit choice of it forces the copies
        rc = repack_for_tc(plan, g_force_route.load() == kRouteTcPair);
        if (rc != SGEMM_OK) return rc;
    }
    return launch_tc(plan, route);
}

}  // namespace

namespace sg {

size_t workspace_size_no_planes(int mode, int M, int N, int K, int Q)
{
    const size_t split = preferred_plan(mode, M, N, K, Q).ws_bytes;
    if (mode == SGEMM_MODE_DEFAULT) mode = g_default_mode.load();
    if (M <= 0 || N <= 0 || K <= 0 || Q <= 0) return split;
    if (mode == SGEMM_MODE_3XTF32 || mode == SGEMM_MODE_TF32) {
        // room for 128-byte-pitched copies of operands TMA cannot describe
        // (pointers, leading dimensions and layouts are not known here)
        auto copy = [Q, K](long long rows) {
            const long long r32k = rows * ((K + 31) / 32 * 32);
            const long long kr32 = static_cast<long long>(K) * ((rows + 31) / 32 * 32);
            return round256(static_cast<size_t>(Q) * (r32k > kr32 ? r32k : kr32) * 4);
        };
        return split + copy(M) + copy(N);
    }
    if (mode != SGEMM_MODE_FP32) return split;
    // room for the transposed operands the FP32 path may make (the layout
    // is not known here; a broadcast operand would need less)
    size_t repack = 0;
    if (N >= kRepackMinN) repack += repack_bytes(M, K, Q, false);
    if (M >= kRepackMinM) repack += repack_bytes(N, K, Q, false);
    return split + repack;
}

}  // namespace sg

extern "C" {

int sgemm(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb,
          float beta, float *C, int ldc, void *stream)
{
    return run(SGEMM_MODE_DEFAULT, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, 0, 0, 0, 0, 0,
               1, stream);
}

int sgemm_ex(int mode, int M, int N, int K, float alpha, const float *A, int lda, const float *B,
             int ldb, float beta, float *C, int ldc, void *stream)
{
    return run(mode, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, 0, 0, 0, 0, 0, 1, stream);
}

int sgemm_batched(int M, int N, int K, float alpha, const float *A, int lda, const float *B,
                  int ldb, float beta, float *C, int ldc, int transA, int transB,
                  long long strideA, long long strideB, long long strideC, int Q, void *stream)
{
    return run(SGEMM_MODE_DEFAULT, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, transA, transB,
               strideA, strideB, strideC, Q, stream);
}

int sgemm_batched_ex(int mode, int M, int N, int K, float alpha, const float *A, int lda,
                     const float *B, int ldb, float beta, float *C, int ldc, int transA,
                     int transB, long long strideA, long long strideB, long long strideC, int Q,
                     void *stream)
{
    return run(mode, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, transA, transB, strideA,
               strideB, strideC, Q, stream);
}

int sgemm_batched_ex_ws(int mode, int M, int N, int K, float alpha, const float *A, int lda,
                        const float *B, int ldb, float beta, float *C, int ldc, int transA,
                        int transB, long long strideA, long long strideB, long long strideC,
                        int Q, void *workspace, size_t workspace_bytes, void *stream)
{
    if (workspace_bytes > 0 &&
        (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return SGEMM_ERR_INVALID_ARG;
    return run(mode, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, transA, transB, strideA,
               strideB, strideC, Q, stream, workspace_bytes ? workspace : nullptr,
               workspace_bytes);
}

size_t sgemm_workspace_size(int mode, int M, int N, int K, int Q)
{
    const size_t base = workspace_size_no_planes(mode, M, N, K, Q);
    if (mode == SGEMM_MODE_DEFAULT) mode = g_default_mode.load();
    if (M <= 0 || N <= 0 || K <= 0 || Q <= 0) return base;
    if (mode != SGEMM_MODE_3XTF32 && mode != SGEMM_MODE_TF32) return base;
    // with route RAW (3xTF32: its lo planes) or where the planes route pays
    // for this shape (planes_pay; operands TMA cannot describe take it): the
    // planes (every batch entry stored) and the split plan of their tiles,
    // or the copies and plans of the other routes, whichever is larger
    const int route = route_for(mode, M, N, K, Q);
    if (route == kRouteTcPair || route == kRouteTcDirect || route == kRouteTcInline) return base;
    const int sms = num_sms_or_zero();
    size_t need = base;
    const size_t split = preferred_plan(mode, M, N, K, Q).ws_bytes;
    if (route == kRouteTcRaw) {  // 3xTF32: the lo pass's planes
        const size_t lo = raw_lo_bytes_max(mode, M, N, K, Q, Q) + split;
        if (lo > need) need = lo;
    }
    // operands TMA cannot describe take the planes route instead
    if (route == kRouteTcPlanes || (route != kRouteTcRaw && planes_pay(mode, M, N, K, Q, Q, Q, sms))) {
        const size_t planes = planes_bytes(mode, M, N, K, Q, Q) + split;
        if (planes > need) need = planes;
    }
    return need;
}

int sgemm_set_default_mode(int mode)
{
    if (mode != SGEMM_MODE_FP32 && mode != SGEMM_MODE_3XTF32 && mode != SGEMM_MODE_TF32)
        return SGEMM_ERR_INVALID_ARG;
    g_default_mode.store(mode);
    return SGEMM_OK;
}

int sgemm_get_default_mode(void) { return g_default_mode.load(); }

const char *sgemm_status_string(int status)
{
    switch (status) {
    case SGEMM_OK: return "success";
    case SGEMM_ERR_INVALID_ARG: return "invalid argument";
    case SGEMM_ERR_UNSUPPORTED: return "unsupported: needs a compute capability 10.3 GPU";
    case SGEMM_ERR_LAUNCH: return "CUDA launch or runtime error";
    case SGEMM_ERR_TIMEOUT: return "a kernel's bounded wait ran out (device status word)";
    case SGEMM_ERR_SCRATCH_LIMIT:
        return "the shape needs more split-K scratch than the built-in array holds";
    default: return "unknown status";
    }
}

int sgemm_poll_error(void *stream)
{
    int dev = 0;
    const DeviceInfo *di = device_info(&dev);
    if (di == nullptr) return SGEMM_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return SGEMM_ERR_LAUNCH;
    unsigned int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word)) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess)
            return SGEMM_ERR_LAUNCH;
        return SGEMM_ERR_TIMEOUT;
    }
    return SGEMM_OK;
}

int sgemm_selftest_wait_timeout(long long wait_cycles, void *stream)
{
    if (wait_cycles < 1 || wait_cycles > (1LL << 31)) return SGEMM_ERR_INVALID_ARG;
    int dev = 0;
    const DeviceInfo *di = device_info(&dev);
    if (di == nullptr) return SGEMM_ERR_UNSUPPORTED;
    wait_timeout_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(di->status,
                                                                          wait_cycles);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    note_launch();
    return SGEMM_OK;
}

int sgemm_peak_probe(int kind, long long iters, double *flops, void *stream)
{
    if (flops == nullptr || !sg::probe_args_ok(kind, iters)) return SGEMM_ERR_INVALID_ARG;
    int num_sms = 0;
    unsigned int *status = nullptr;
    if (!sg::current_sm103(&num_sms, &status)) return SGEMM_ERR_UNSUPPORTED;
    return sg::launch_peak_probe(kind, iters, num_sms, status, static_cast<cudaStream_t>(stream),
                                 flops);
}

unsigned long long sgemm_kernel_launches(void) { return sg::g_launches.load(); }

int sgemm_last_split_count(void) { return sg::g_last_splits.load(); }

int sgemm_tune_force(int route)
{
    if (route < 0 || route >= sg::kRouteCount) return SGEMM_ERR_INVALID_ARG;
    sg::g_force_route.store(route);
    return SGEMM_OK;
}

int sgemm_tune_route(int mode, int M, int N, int K, int Q)
{
    if (mode == SGEMM_MODE_DEFAULT) mode = g_default_mode.load();
    if (mode != SGEMM_MODE_FP32 && mode != SGEMM_MODE_3XTF32 && mode != SGEMM_MODE_TF32)
        return -1;
    if (M < 0 || N < 0 || K < 0 || Q < 0) return -1;
    return sg::route_for(mode, M, N, K, Q);
}

int sgemm_version(void) { return 100; }

}  // extern "C"
