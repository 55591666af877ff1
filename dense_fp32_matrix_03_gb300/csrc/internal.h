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

// Split-K plan shared by both kernels (128 x 128 output tiles).  A grid with
// at most half as many tiles as multiprocessors is cut along K into `splits`
// slices, as many as keep all work units in one wave, each at least
// min_slice_k(mode) long: 64 for the FP32 path, 256 for the tensor-core
// paths, whose per-unit pipeline start-up (copy, split, MMA, TMEM read-back)
// is longer (measured on GB300: shorter slices made 128^3..512^3 slower).
// The slices are whole k-blocks of the kernel that runs (each kernel's
// k-block is at most the minimum slice, so no slice is empty).  The
// workspace holds one arrival counter per tile region and one fp32 partial
// tile per (tile, slice).
constexpr int kSplitTile = 128;            // output tile edge of both paths
constexpr int kSplitRegions = 8;           // counters per tile (>= warps writing a tile)
constexpr int kMaxSplits = 16;
int min_slice_k(int mode);
int choose_splits(long long num_tiles, int K, int num_sms, int mode);
size_t splitk_workspace_bytes(long long num_tiles, int splits);
// Fills p.splits / num_units / ws_* for the launch: splits if the plan's
// workspace is large enough (and clears its counters on the stream), else
// runs unsplit.  Returns an sgemm status.
int plan_splits(Plan &plan);

// Describes one operand for a TMA tensor map.
//  kin  : contiguous dimension is K (rows are `rows` long runs of K values)
//  rows : extent of the non-K dimension (M for A, N for B)
//  box_rows : tile extent along that dimension
// Returns false if the driver rejects the description (the caller then uses
// the cp.async producer).
bool encode_operand(CUtensorMap *map, const float *base, bool kin, long long rows, long long K,
                    long long ld, int Q, long long stride, int box_rows);

int launch_simt(Plan &plan);   // returns an sgemm status code
int launch_tc(Plan &plan);     // tcgen05 paths (3xTF32 and TF32)

}  // namespace sg
