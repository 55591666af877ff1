// params.h -- the launch parameters every SGEMM kernel receives, and the
// per-call plan the host builds.  Internal to the library (not part of the
// C ABI in include/sgemm.h).
#pragma once

#include <cstdint>

namespace sg {

// Device status word bits (read back by sgemm_poll_error()).
enum : unsigned int {
    kStatusWaitFull = 1u << 0,   // a consumer waited too long for a loaded stage
    kStatusWaitEmpty = 1u << 1,  // the producer waited too long for a free stage
    kStatusWaitMma = 1u << 2,    // a tensor-core completion never arrived
    kStatusWaitAcc = 1u << 3,    // the epilogue waited too long for an accumulator
    kStatusWaitTest = 1u << 4,   // the bounded-wait self test ran out (expected)
    kStatusWaitConv = 1u << 5,   // the MMA issuer waited too long for split operands
};

struct GemmParams {
    int M, N, K, Q;
    float alpha, beta;
    const float *A;
    const float *B;
    float *C;
    long long lda, ldb, ldc;
    long long sA, sB, sC;      // batch strides in elements (0 = broadcast)
    int tiles_m, tiles_n;      // output tiles per batch entry
    int k_blocks;              // ceil(K / BK)
    int group_m;               // rows of tiles per scheduler group
    long long num_tiles;       // Q * tiles_m * tiles_n
    int a_q_step, b_q_step;    // TMA batch coordinate multiplier (0 = broadcast)
    int a_vec4, b_vec4;        // fallback producer may copy 16 bytes at a time
    int c_vec4;                // epilogue may use 16-byte C accesses
    int c_tma;                 // the shared-memory-operand kernel's epilogue moves C by TMA
    unsigned int *status;      // device status word
    long long wait_limit;      // clock64 cycles a bounded wait may spin
    // split-K: tiles [0, dp_tiles) are whole work units (u = tile); every
    // later tile's k-blocks are cut into `splits` contiguous slices, unit
    // u = dp_tiles + (tile - dp_tiles) * splits + slice.  Each slice writes its
    // unscaled fp32 partial tile to its slot of ws_part; the fix-up kernel
    // then sums the slices, in slice order, and applies alpha and beta.
    // dp_tiles = 0 splits every tile (a grid smaller than the GPU); dp_tiles =
    // whole waves of tiles splits only the last, partial wave.
    int splits;                // 1 = no split
    long long dp_tiles;        // tiles computed whole (num_tiles when splits == 1)
    long long num_units;       // dp_tiles + (num_tiles - dp_tiles) * splits
    float *ws_part;            // one row-major BM x BN fp32 slot per split unit
};

}  // namespace sg
