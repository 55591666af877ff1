// tune_table.h -- kernel route per (mode, size class, batched) call, as
// measured by the sweep `python bench.py --tune` (which rewrites this file)
// on NVIDIA GB300, L2 flushed before every timed call, through the workspace entry.
// Size class and routes: internal.h (size_class, Route).  A (mode, class)
// without an entry takes the cost models' choice (kRouteAuto), which the
// sweep keeps unless another route is more than 2% faster; the
// shapes where it kept the cost models' choice:
//   3xtf32 128x128x128 (class 7): us auto 12.3, pair 12.3, direct 14.4, planes 19.5
//   tf32 128x128x128 (class 7): us auto 12.3, pair 12.3, direct 14.4, planes 16.8
//   3xtf32 256x256x256 (class 8): us auto 14.5, pair 14.4, direct 19.9, planes 22.6
//   3xtf32 512x512x512 (class 9): us auto 18.4, pair 18.4, direct 22.5, planes 26.1
//   tf32 512x512x512 (class 9): us auto 16.4, pair 16.4, direct 20.5, planes 20.5
//   fp32 1024x1024x1024 (class 10): us auto 57.3, small 73.7
//   3xtf32 1024x1024x1024 (class 10): us auto 24.6, pair 24.6, direct 32.8, planes 31.8
//   tf32 1024x1024x1024 (class 10): us auto 20.5, pair 20.5, direct 30.7, planes 26.6
//   fp32 2048x2048x2048 (class 11): us auto 309.3, small 469.0
//   3xtf32 2048x2048x2048 (class 11): us auto 81.9, pair 82.0, direct 168.0, planes 82.0
//   tf32 2048x2048x2048 (class 11): us auto 43.0, pair 43.0, direct 142.3, planes 45.1
//   fp32 4092x4092x4092 (class 12): us auto 1985.8, small 3670.0
//   3xtf32 4092x4092x4092 (class 12): us auto 442.4, pair 488.2, direct 1147.4, planes 441.5
//   tf32 4092x4092x4092 (class 12): us auto 196.6, pair 241.6, direct 1035.3, planes 197.1
//   fp32 8192x8192x8192 (class 13): us auto 15813.6, small 28874.8
//   3xtf32 8192x8192x8192 (class 13): us auto 3076.1, pair 3720.2, direct 8913.9, planes 3074.0
//   tf32 8192x8192x8192 (class 13): us auto 1205.2, pair 1641.4, direct 7597.1, planes 1196.0
//   fp32 1024x1024x512 Q=32 (class 11): us auto 560.4, small 962.3
//   3xtf32 1024x1024x512 Q=32 (class 11): us auto 141.1, pair 140.1, direct 335.9, planes 178.4
//   tf32 1024x1024x512 Q=32 (class 11): us auto 87.8, pair 88.1, direct 270.6, planes 106.5
#pragma once

namespace sg {

struct TuneEntry {
    int mode, size_class, batched, route;
};

// {mode (0 FP32, 1 3xTF32, 2 TF32), size class, batched, route}
constexpr TuneEntry kTuneTable[] = {
    {0, 7, 0, 1},  // fp32 128x128x128: small; us: auto 21.5, small 10.3
    {0, 8, 0, 1},  // fp32 256x256x256: small; us: auto 22.5, small 12.3
    {2, 8, 0, 2},  // tf32 256x256x256: pair; us: auto 13.7, pair 12.8, direct 18.3, planes 18.4
    {0, 9, 0, 1},  // fp32 512x512x512: small; us: auto 22.5, small 18.5
    {-1, 0, 0, 0},  // end of table
};

}  // namespace sg
