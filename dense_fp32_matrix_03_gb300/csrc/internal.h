// internal.h -- host-side plan shared between the C-ABI layer (api.cu) and
// the kernel launchers.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "params.h"

namespace sg {

// Everything a launcher needs for one call, after validation.
struct Plan {
    GemmParams p;        // tile counts are filled in by the launcher
    int transA, transB;  // storage of A (K x M when set) and B (N x K when set)
    int mode;            // SGEMM_MODE_* (never DEFAULT here)
    bool a_tma, b_tma;   // operand can be described by a TMA tensor map
    bool even_k;         // K is a multiple of the K block
    int num_sms;         // multiprocessors of the current device
    int device;
    cudaStream_t stream;
    void *ws;            // caller's split-K workspace (may be null)
    size_t ws_bytes;
};

// A wait may spin for this many SM clock cycles (about a second at the
// GB300's clocks) before the kernel gives up and reports SGEMM_ERR_TIMEOUT.
constexpr long long kWaitLimitCycles = 1LL << 31;

// The planner's mode value for the 16-bit-input path (not a public mode).
constexpr int kModeHalf = 16;

bool aligned16(const void *p);
// Argument checks shared by every entry point (dimensions, leading
// dimensions, batch strides, pointers that will be read or written);
// returns SGEMM_OK or SGEMM_ERR_INVALID_ARG.
int check_shape(int M, int N, int K, float alpha, const void *A, int lda, const void *B, int ldb,
                const float *C, int ldc, int transA, int transB, long long sA, long long sB,
                long long sC, int Q);

// Split-K plan shared by the kernels (BM x BN output tiles, persistent: one
// CTA per multiprocessor, or one CTA pair per two for the tensor-core pair
// kernel).  With T tiles on G units at once (multiprocessors, or pairs) the
// grid runs floor(T/G) whole waves and a last wave of r = T mod G tiles that
// leaves the rest of the GPU idle.  The planner may cut the tiles of that last wave
// (all tiles when T < G) along K into `splits` slices, so that the slices
// spread over the whole GPU.  Each slice writes its partial tile, unscaled,
// to its own BM x BN fp32 slot of the workspace, and a fix-up kernel
// launched right after on the same stream sums every split tile's slots in
// slice order and applies alpha and beta.  Modelled time of s slices:
//     t_tile * (floor(T/G) + ceil(r * s / G) / s)
//       + (s > 1: 3 us + 2 * workspace bytes / (8 TB/s if they stay in L2,
//                                                 i.e. <= 64 MB, else 3 TB/s))
// with t_tile = 2 * BM * BN * K / (multiprocessors per unit x the kernel's
// per-multiprocessor rate, as measured on GB300: 0.40 TFLOP/s FP32, 1.8
// 3xTF32, 3.6 TF32 with TMA-fed operands; 0.24, 0.47, 0.55 for operands TMA
// cannot describe).  s runs over
// 1 .. min(16, K / min_slice_k(mode)); the best s is used only when it
// saves at least 1%.  Each slice is at least
// min_slice_k(mode) deep: 64 for the FP32 path, 256 for the tensor-core
// paths, whose per-unit pipeline start-up (copy, split, MMA, TMEM
// read-back) is longer (measured on GB300: shorter slices made 128^3..512^3
// slower).  The slices are whole k-blocks of the kernel that runs (each
// kernel's k-block is at most the minimum slice, so no slice is empty).  A
// plan whose workspace exceeds the caller's budget is not considered.
constexpr int kMaxSplits = 16;
// How a kernel is fed: operands loaded by the threads themselves (the FP32
// kernel's cp.async producer, the tensor-core direct kernel), by TMA on one
// CTA per unit, by TMA on a CTA pair per unit (two multiprocessors), or, on
// a CTA pair, as TF32 planes made by a pass before the product (planes.cu).
// kFeedInline: 3xTF32 on a CTA pair from the caller's matrices, the lo
// planes made in the kernel (raw.cu).
enum Feed { kFeedDirect = 0, kFeedTma = 1, kFeedPair = 2, kFeedPlanes = 3, kFeedInline = 4 };
struct SplitPlan {
    int splits;          // 1 = no split
    long long dp_tiles;  // tiles computed whole (they come first in unit order)
    size_t ws_bytes;     // workspace the plan needs
    double seconds;      // the model's time for the plan (0 when not modelled)
};
int min_slice_k(int mode);
// FLOP/s per multiprocessor of the kernel a mode and feed run (GB300).
double path_rate_per_sm(int mode, int feed);
size_t splitk_workspace_bytes(long long split_tiles, int splits, int bm, int bn);
// slots: units that run at once (multiprocessors, or CTA pairs for kFeedPair).
SplitPlan choose_plan(long long num_tiles, int K, int slots, int mode, int bm, int bn, int feed,
                      size_t budget);
// Fills p.splits / dp_tiles / num_units / ws_part for the launch (bm x bn
// tiles, operands through TMA or not) from the best plan that fits the
// caller's workspace.  Returns an sgemm status.
int plan_splits(Plan &plan, int bm, int bn, int feed, int slots);
// Output tile of each kernel (defined beside its launcher); the FP32 path's
// depends on whether both operands are K-inner.
void simt_tile_dims(bool both_k_inner, int &bm, int &bn);
// The FP32 path's tile on kRouteSimtSmall.
void simt_small_tile_dims(int &bm, int &bn);
// pair: the CTA-pair kernel's tile (the single-CTA kernels' otherwise).
void tc_tile_dims(int mode, int K, bool pair, int &bm, int &bn);
// CTA pairs of the pair kernel that fit on the device at once (cached).
int tc_pair_slots(int num_sms);
// Launches the CTA-pair tensor-core kernel (tile counts filled in by the
// caller) with the tensor maps of its A (128-row boxes) and B (64-row boxes).
int launch_tc_pair(Plan &plan, const CUtensorMap &tmA, const CUtensorMap &tmB, int slots);
// Enqueues the split-K fix-up for a launch whose plan split (bm x bn tiles).
int launch_fixup(Plan &plan, int bm, int bn);
// Workspace the TF32 planes of a 3xTF32 / TF32 call take (QA, QB: stored
// batch entries of A and B, 1 when broadcast).
size_t planes_bytes(int mode, long long M, long long N, long long K, int QA, int QB);
// The tensor-core paths' planes route (planes.cu): when the plan's workspace
// holds the planes, enqueues the pass over both operands and the product
// (taken = true) and returns its status; otherwise leaves the plan alone
// (taken = false).
// force: take the route whenever the planes fit (kRouteTcPlanes), without
// asking planes_pay.
int run_planes(Plan &plan, bool &taken, bool force = false);
// The tensor-core paths' raw route (raw.cu): both operands straight from
// the caller's matrices by TMA, K-major or M/N-major as stored; TF32 with no
// pass, 3xTF32 with a pass that writes the operands' lo planes into the
// workspace (the raw values are the hi planes).  Enqueues and sets taken
// when the operands allow it (and the workspace holds the lo planes) and
// either force is set or raw_pay says the route is expected to be fastest.
// With force, route is the one forced (kRouteTcRaw: 3xTF32 with a lo pass
// into the workspace; kRouteTcInline: 3xTF32 with the lo planes made in the
// kernel); without, the cost models' form (raw_choice).
int run_raw(Plan &plan, bool &taken, bool force = false, int route = 0);
// The form of the raw route the cost models pick for a call, if any:
// kRawNone, kRawPlain (TF32 on the raw operands) or kRawInline (3xTF32 with
// the lo planes made in the kernel) -- when its modelled time beats both the
// pair kernel's and the planes route's.  Each route's product takes the split
// planner's time for its tiles; the planes route adds its pass (12 bytes per
// operand value for 3xTF32, 8 for TF32, at 6.0 TB/s) and 7 us.  lines =
// false (some operand row off a 128-byte boundary) makes the raw product
// slower: 6% (3xTF32 inline) or 27% (TF32), as measured on GB300 at a
// 4092-float pitch against 4096.  (The raw route with a lo pass is taken
// only when forced: the inline form was faster on every shape measured.)
enum RawForm { kRawNone = 0, kRawPlain = 1, kRawInline = 2 };
int raw_choice(int mode, long long M, long long N, long long K, int QA, int QB, int Q,
               int num_sms, bool lines = true);
inline bool raw_pay(int mode, long long M, long long N, long long K, int QA, int QB, int Q,
                    int num_sms, bool lines = true)
{
    return raw_choice(mode, M, N, K, QA, QB, Q, num_sms, lines) != kRawNone;
}
// Workspace the raw route's lo planes take (3xTF32; 0 for TF32), for either
// layout of each operand (the larger of rows x round_up(K, 32) and
// K x round_up(rows, 32) values per stored entry).
size_t raw_lo_bytes_max(int mode, long long M, long long N, long long K, int QA, int QB);
// CTA pairs of the shared-memory-operand kernel that fit at once (cached).
int ss_slots(int num_sms);
// Whether the planes route is expected to beat the pair kernel for this
// shape (QA, QB: stored batch entries of A and B; num_sms 0: unknown, then
// false).  Each route's product takes the split planner's modelled time for
// its tiles (choose_plan: 256 x 256 pair tiles at the planes rate; the pair
// kernel's tiles at its rate), and the planes route adds its pass, which
// moves (QA * M + QB * N) * K * 4 * (1 + planes) bytes at 6.0 TB/s, and
// 7 us for its extra launch and the shorter grid's ramp (fitted on GB300,
// TFLOP/s pair / planes: 2048^3 3xTF32 213 / 208, TF32 393 / 376; 2560^3
// TF32 457 / 470; 4096 x 4096 x 1024 3xTF32 253 / 267; 2048 x 2048 x 8192
// 3xTF32 264 / 244).
bool planes_pay(int mode, long long M, long long N, long long K, int QA, int QB, int Q,
                int num_sms);
// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once: the attribute belongs to the function on each device and
// setting it is a driver call (about a microsecond), so the launchers ask
// here, which remembers (device, kernel) pairs already set.  False when the
// runtime refuses.
bool smem_attr_once(const void *kernel, int bytes);
// Multiprocessors of the current device, 0 when there is no usable one.
int num_sms_or_zero();
// sgemm_workspace_size without room for the planes (the host-buffer entry's
// per-panel calls would rewrite all of B once per panel).
size_t workspace_size_no_planes(int mode, int M, int N, int K, int Q);
// The plan sgemm_workspace_size reports for a call (no budget), or splits = 1.
SplitPlan preferred_plan(int mode, int M, int N, int K, int Q);
// The plan of the allocation-free entry point: a grid of at most half as many
// tiles as multiprocessors is cut into as many slices as keep every unit in
// one wave (at most 16, each at least min_slice_k deep); other grids run
// unsplit.  Its workspace is at most one partial tile per multiprocessor.
SplitPlan one_wave_plan(int mode, int M, int N, int K, int Q);

// Describes one operand for a TMA tensor map.
//  kin  : contiguous dimension is K (rows are `rows` long runs of K values)
//  rows : extent of the non-K dimension (M for A, N for B)
//  box_rows : tile extent along that dimension
// promote256: L2 fills of 256 bytes (else 128) -- measured on GB300, 256
// suits rows on 128-byte boundaries, 128 rows that are not (TF32 from a
// 4092-float pitch: 648 -> 725 TFLOP/s; a 4096-float pitch: equal).
// Returns false if the driver rejects the description (the caller then uses
// the cp.async producer).
bool encode_operand(CUtensorMap *map, const float *base, bool kin, long long rows, long long K,
                    long long ld, int Q, long long stride, int box_rows,
                    bool promote256 = true);

// Tensor map of an operand stored K x rows (rows-inner: A stored K x M, B
// stored K x N) for M/N-major staging: boxes of 32 rows-inner values by 32 k
// with the 128-byte swizzle of 32-byte atoms (dims rows, K, entries), the
// layout kind::tf32 reads M/N-major.
bool encode_operand_mn(CUtensorMap *map, const float *base, long long rows, long long K,
                       long long ld, int Q, long long stride, bool promote256 = true);

// Tensor map of C (Q entries sC apart when batched) in boxes of 32 rows by
// chunk_cols columns: 16 with the 64-byte swizzle, or 32 with the 128-byte
// one; the shared-memory-operand kernel's epilogue loads and stores C
// through it.  C must be 16-byte aligned with ldc and sC multiples of four
// values.
bool encode_c_tiles(CUtensorMap *map, const float *C, long long M, long long N, long long ldc,
                    int Q, long long sC, int chunk_cols);

// Tensor map of a K-inner 16-bit operand (bf16 or fp16): boxes of 64 k by
// box_rows rows with the 128-byte swizzle.
bool encode_operand16(CUtensorMap *map, const void *base, bool bf16, long long rows, long long K,
                      long long ld, int Q, long long stride, int box_rows);
// Copies Q matrices of 16-bit values into dst as rows x cols K-inner
// matrices (row pitch ldd, batch stride dstride): dst[r][c] = src[c][r] when
// trans (src stored cols x rows), else src[r][c] (src row pitch lds).
int launch_repack16(const uint16_t *src, long long lds, long long sstride, int rows, int cols,
                    int Q, bool trans, uint16_t *dst, long long ldd, long long dstride,
                    cudaStream_t stream);

// Transposes Q matrices of rows x cols (row pitch lds, batch stride sstride)
// into dst (row pitch ldd, batch stride dstride): dst[c][r] = src[r][c].
int launch_transpose(const float *src, long long lds, long long sstride, int rows, int cols, int Q,
                     float *dst, long long ldd, long long dstride, int num_sms, cudaStream_t stream);
// Smallest N (for A) and M (for B) at which the FP32 path transposes a
// K-inner operand into the workspace first (see repack_for_simt in api.cu).
constexpr int kRepackMinN = 1024, kRepackMinM = 1024;

// Multiprocessor count and device status word of the current device; false
// when it cannot be queried or is not a compute capability 10.3 GPU.
bool current_sm103(int *num_sms, unsigned int **status);
// Counts one kernel the library enqueued (reported by sgemm_kernel_launches).
void note_launch();

// A known probe kind with an iteration count inside its documented range.
bool probe_args_ok(int kind, long long iters);
// Enqueues one throughput probe (SGEMM_PROBE_*); *flops receives the
// operations it performs.  Returns an sgemm status.
int launch_peak_probe(int kind, long long iters, int num_sms, unsigned int *status,
                      cudaStream_t st, double *flops);

// Kernel families a call can run, the vocabulary of the tuning table
// (tune_table.h) and of sgemm_tune_force (include/sgemm.h):
//   kRouteAuto       the cost models (FP32: the tile for the layout; tensor
//                    cores: planes where planes_pay, else the pair kernel
//                    for TMA-describable operands, else the direct kernel);
//   kRouteSimtSmall  FP32 on 64 x 64 tiles (small grids);
//   kRouteTcPair     tensor cores on the CTA-pair kernel (never the planes);
//   kRouteTcDirect   tensor cores on the direct-load kernel (128 x 128);
//   kRouteTcPlanes   tensor cores on the planes route whenever the
//                    workspace holds the planes.
// A route the call's mode or operands cannot take falls back to kRouteAuto.
//   kRouteTcRaw      tensor cores on the caller's matrices as stored (raw.cu)
//                    whenever both operands are TMA-describable (and, for
//                    3xTF32, the workspace holds the lo planes).
//   kRouteTcInline   the raw route with 3xTF32's lo planes made inside the
//                    product kernel (TF32: the raw route).
//   kRouteModels     (forced only) the cost models' choice, the table
//                    ignored: the baseline the tuning sweep measures against.
enum Route { kRouteAuto = 0, kRouteSimtSmall = 1, kRouteTcPair = 2, kRouteTcDirect = 3,
             kRouteTcPlanes = 4, kRouteTcRaw = 5, kRouteTcInline = 6, kRouteModels = 7,
             kRouteCount = 8 };
// Size class of a call: round(log2(M * N * K * Q) / 3), clamped to
// [kClassMin, kClassMax] -- the log2 of the edge of a cube of the same work
// (4092^3: 12; the batched 32 x 1024 x 1024 x 512 workload: 11).
constexpr int kClassMin = 7, kClassMax = 13;
int size_class(long long M, long long N, long long K, int Q);
// The route of a call: the forced route (sgemm_tune_force) when one is set,
// else the tuning table's entry for (mode, size class, batched), else
// kRouteAuto.
int route_for(int mode, long long M, long long N, long long K, int Q);

int launch_simt(Plan &plan, int route);  // returns an sgemm status code
int launch_tc(Plan &plan, int route);    // tcgen05 paths (3xTF32 and TF32)

}  // namespace sg
