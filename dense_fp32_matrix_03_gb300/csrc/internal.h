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
};

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
