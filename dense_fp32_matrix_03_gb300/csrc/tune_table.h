// tune_table.h -- kernel route per (mode, size class, batched) call, as
// measured by the sweep `python bench.py --tune` (which rewrites this file)
// on NVIDIA GB300, L2 flushed before every timed call, through the workspace entry.
// Size class and routes: internal.h (size_class, Route).  A (mode, class)
// without an entry takes the cost models' choice (kRouteAuto), which the
// sweep keeps unless another route is more than 2% faster; the
// shapes where it kept the cost models' choice:
//   3xtf32 128x128x128 (class 7): us models 13.2, pair 12.9, direct 15.6, planes 20.5, raw 18.7, inline 16.8
//   tf32 128x128x128 (class 7): us models 12.3, pair 12.3, direct 14.3, planes 17.7, raw 14.5
//   3xtf32 256x256x256 (class 8): us models 15.5, pair 15.2, direct 20.5, planes 23.4, raw 21.6, inline 20.5
//   tf32 256x256x256 (class 8): us models 13.3, pair 13.2, direct 18.4, planes 18.4, raw 16.4
//   3xtf32 512x512x512 (class 9): us models 18.4, pair 18.4, direct 22.5, planes 27.6, raw 25.7, inline 22.6
//   tf32 512x512x512 (class 9): us models 16.4, pair 16.4, direct 20.5, planes 21.7, raw 18.4
//   fp32 1024x1024x1024 (class 10): us models 55.3, small 73.7
//   tf32 1024x1024x1024 (class 10): us models 20.5, pair 20.8, direct 30.7, planes 27.6, raw 22.5
//   fp32 2048x2048x2048 (class 11): us models 309.2, small 469.0
//   3xtf32 2048x2048x2048 (class 11): us models 66.7, pair 82.0, direct 167.9, planes 84.0, raw 78.1, inline 67.2
//   tf32 2048x2048x2048 (class 11): us models 34.8, pair 43.0, direct 143.3, planes 46.1, raw 35.1
//   fp32 4092x4092x4092 (class 12): us models 1984.8, small 3663.9
//   3xtf32 4092x4092x4092 (class 12): us models 389.2, pair 487.6, direct 1142.9, planes 444.5, raw 443.4, inline 387.3
//   tf32 4092x4092x4092 (class 12): us models 194.7, pair 242.3, direct 1034.8, planes 203.9, raw 194.8
//   fp32 8192x8192x8192 (class 13): us models 15787.0, small 28818.4
//   3xtf32 8192x8192x8192 (class 13): us models 2889.7, pair 3726.3, direct 9046.0, planes 3077.1, raw 3146.8, inline 3093.5
//   fp32 1024x1024x512 Q=32 (class 11): us models 558.6, small 962.6
//   3xtf32 1024x1024x512 Q=32 (class 11): us models 110.6, pair 140.0, direct 335.6, planes 177.7, raw 164.4, inline 110.8
//   tf32 1024x1024x512 Q=32 (class 11): us models 65.5, pair 88.1, direct 270.6, planes 108.6, raw 65.6
#pragma once

namespace sg {

struct TuneEntry {
    int mode, size_class, batched, route;
};

// {mode (0 FP32, 1 3xTF32, 2 TF32), size class, batched, route}
constexpr TuneEntry kTuneTable[] = {
    {0, 7, 0, 1},  // fp32 128x128x128: small; us: models 22.5, small 10.3
    {0, 8, 0, 1},  // fp32 256x256x256: small; us: models 22.5, small 12.3
    {0, 9, 0, 1},  // fp32 512x512x512: small; us: models 22.8, small 18.8
    {1, 10, 0, 2},  // 3xtf32 1024x1024x1024: pair; us: models 26.7, pair 24.6, direct 32.8, planes 31.7, raw 29.7, inline 26.6
    {2, 13, 0, 5},  // tf32 8192x8192x8192: raw; us: models 1240.0, pair 1817.8, direct 7605.2, planes 1228.8, raw 1164.2
    {-1, 0, 0, 0},  // end of table
};

}  // namespace sg
