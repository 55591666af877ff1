// tune_table.h -- kernel route per (mode, size class, batched) call, as
// measured by the sweep `python bench.py --tune` (which rewrites this file)
// on NVIDIA GB300, L2 flushed before every timed call, through the workspace entry.
// Size class and routes: internal.h (size_class, Route).  A (mode, class)
// without an entry takes the cost models' choice (kRouteAuto), which the
// sweep keeps unless another route is more than 2% faster; the
// shapes where it kept the cost models' choice:
//   tf32 128x128x128 (class 7): us models 12.5, pair 12.4, direct 14.3, planes 16.4, raw 14.3
//   3xtf32 256x256x256 (class 8): us models 15.4, pair 15.4, direct 20.5, planes 23.6, raw 22.5, inline 20.5
//   tf32 256x256x256 (class 8): us models 13.5, pair 13.3, direct 18.4, planes 19.5, raw 16.4
//   3xtf32 512x512x512 (class 9): us models 18.4, pair 18.4, direct 22.5, planes 27.6, raw 25.6, inline 22.5
//   tf32 512x512x512 (class 9): us models 16.4, pair 16.4, direct 20.5, planes 22.5, raw 18.6
//   fp32 1024x1024x1024 (class 10): us models 57.3, small 73.7
//   tf32 1024x1024x1024 (class 10): us models 20.8, pair 20.5, direct 30.7, planes 27.6, raw 22.5
//   fp32 2048x2048x2048 (class 11): us models 309.3, small 469.0
//   3xtf32 2048x2048x2048 (class 11): us models 67.8, pair 80.9, direct 167.9, planes 84.5, raw 78.8, inline 67.9
//   tf32 2048x2048x2048 (class 11): us models 34.8, pair 43.0, direct 142.6, planes 47.1, raw 35.1
//   fp32 4092x4092x4092 (class 12): us models 1985.0, small 3665.9
//   3xtf32 4092x4092x4092 (class 12): us models 409.6, pair 487.4, direct 1148.6, planes 443.6, raw 441.8, inline 407.6
//   tf32 4092x4092x4092 (class 12): us models 192.6, pair 242.2, direct 1037.3, planes 198.2, raw 192.5
//   fp32 8192x8192x8192 (class 13): us models 15787.0, small 28794.9
//   3xtf32 8192x8192x8192 (class 13): us models 2906.1, pair 3738.6, direct 8976.4, planes 3086.3, raw 3090.4, inline 3045.4
//   fp32 1024x1024x512 Q=32 (class 11): us models 560.0, small 959.7
//   3xtf32 1024x1024x512 Q=32 (class 11): us models 118.8, pair 139.3, direct 334.6, planes 178.7, raw 165.4, inline 119.3
//   tf32 1024x1024x512 Q=32 (class 11): us models 65.5, pair 86.5, direct 269.8, planes 112.6, raw 65.5
#pragma once

namespace sg {

struct TuneEntry {
    int mode, size_class, batched, route;
};

// {mode (0 FP32, 1 3xTF32, 2 TF32), size class, batched, route}
constexpr TuneEntry kTuneTable[] = {
    {0, 7, 0, 1},  // fp32 128x128x128: small; us: models 22.5, small 10.3
    {1, 7, 0, 2},  // 3xtf32 128x128x128: pair; us: models 13.0, pair 12.6, direct 15.1, planes 18.4, raw 17.4, inline 16.4
    {0, 8, 0, 1},  // fp32 256x256x256: small; us: models 22.5, small 12.6
    {0, 9, 0, 1},  // fp32 512x512x512: small; us: models 22.5, small 18.4
    {1, 10, 0, 2},  // 3xtf32 1024x1024x1024: pair; us: models 26.7, pair 24.6, direct 32.8, planes 32.6, raw 29.7, inline 27.4
    {2, 13, 0, 5},  // tf32 8192x8192x8192: raw; us: models 1254.4, pair 1821.0, direct 7535.6, planes 1208.3, raw 1179.6
    {-1, 0, 0, 0},  // end of table
};

}  // namespace sg
