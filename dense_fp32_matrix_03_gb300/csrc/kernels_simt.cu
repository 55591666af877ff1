// kernels_simt.cu -- instantiations and the host launcher of the FP32
// CUDA-core SGEMM kernel (simt_fp32.cuh).
#include <cstring>

#include "../../include/sgemm.h"
#include "internal.h"
#include "simt_fp32.cuh"

namespace sg {

namespace {

// Tile configurations of the FP32 path.  Where one operand's fragment comes
// in adjacent registers (every layout but A and B both K-inner), the FMAs are
// packed two per instruction, and a wide lane tile (8 x 16 outputs, 64 x 64
// per warp, 256 x 128 per CTA, two stages of 64 k) pays for the broadcast
// of the other operand over twice as many FMAs.  With both operands K-inner
// the FMAs stay scalar and the 8 x 8 lane tile (128 x 128 per CTA, three
// stages of 64 k) is faster.  Measured on GB300 at 4092^3 with the last wave
// split: nn 59.1 -> 63.6 TFLOP/s with the wide tile; nt 54.3 narrow, 51.6
// wide.  The wide tile reads A two k at a time (64-bit loads: fewer live
// fragment registers, 63.6 -> 64.0); the narrow one four at a time.
using SimtWide = SimtCfg<256, 128, 64, 64, 2, 2, 0, 2>;
using SimtNarrow = SimtCfg<128, 128, 64, 32, 3, 2, 1, 4>;
// Small grids (kRouteSimtSmall, chosen by the tuning table): 64 x 64 tiles,
// 32 x 32 per warp (4 x 8 outputs per lane), four warps, four stages of 32 k
// -- four times the tiles of the narrow tile, sixteen times those of the
// wide one, so that a 128^3 .. 512^3 product spreads over more
// multiprocessors before any split along K.
using SimtSmall = SimtCfg<64, 64, 32, 32, 4, 1, 1, 4>;
constexpr int kGroupM = 8;

template <class Cfg, bool A_KIN, bool B_KIN, bool USE_TMA, bool EVEN_K>
int launch_one(Plan &plan, const CUtensorMap &tmA, const CUtensorMap &tmB)
{
    auto kern = simt_sgemm_kernel<Cfg, A_KIN, B_KIN, USE_TMA, EVEN_K>;
    if (!smem_attr_once(reinterpret_cast<const void *>(kern), Cfg::SMEM_BYTES))
        return SGEMM_ERR_LAUNCH;
    long long grid = plan.p.num_units;
    if (grid > static_cast<long long>(plan.num_sms) * kMinBlocks)
        grid = static_cast<long long>(plan.num_sms) * kMinBlocks;
    kern<<<static_cast<unsigned>(grid), Cfg::THREADS, Cfg::SMEM_BYTES, plan.stream>>>(
        tmA, tmB, plan.p);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    note_launch();
    return plan.p.splits > 1 ? launch_fixup(plan, Cfg::BM, Cfg::BN) : SGEMM_OK;
}

// Plans and launches one layout with its tile configuration.
template <class Cfg, bool A_KIN, bool B_KIN>
int launch_cfg(Plan &plan)
{
    GemmParams &p = plan.p;
    p.tiles_m = (p.M + Cfg::BM - 1) / Cfg::BM;
    p.tiles_n = (p.N + Cfg::BN - 1) / Cfg::BN;
    p.k_blocks = (p.K + Cfg::BK - 1) / Cfg::BK;
    p.group_m = kGroupM;
    p.num_tiles = static_cast<long long>(p.Q) * p.tiles_m * p.tiles_n;
    plan.even_k = (p.K % Cfg::BK) == 0;

    alignas(64) CUtensorMap tmA;
    alignas(64) CUtensorMap tmB;
    std::memset(&tmA, 0, sizeof(tmA));
    std::memset(&tmB, 0, sizeof(tmB));
    bool use_tma = plan.a_tma && plan.b_tma;
    if (use_tma) {
        use_tma = encode_operand(&tmA, p.A, A_KIN, p.M, p.K, p.lda, p.Q, p.sA, Cfg::BM) &&
                  encode_operand(&tmB, p.B, B_KIN, p.N, p.K, p.ldb, p.Q, p.sB, Cfg::BN);
    }
    const int rc = plan_splits(plan, Cfg::BM, Cfg::BN, use_tma ? kFeedTma : kFeedDirect,
                               plan.num_sms);
    if (rc != SGEMM_OK) return rc;
    if (use_tma) return launch_one<Cfg, A_KIN, B_KIN, true, false>(plan, tmA, tmB);
    if (plan.even_k) return launch_one<Cfg, A_KIN, B_KIN, false, true>(plan, tmA, tmB);
    return launch_one<Cfg, A_KIN, B_KIN, false, false>(plan, tmA, tmB);
}

}  // namespace

void simt_small_tile_dims(int &bm, int &bn)
{
    bm = SimtSmall::BM;
    bn = SimtSmall::BN;
}

void simt_tile_dims(bool both_k_inner, int &bm, int &bn)
{
    bm = both_k_inner ? SimtNarrow::BM : SimtWide::BM;
    bn = both_k_inner ? SimtNarrow::BN : SimtWide::BN;
}

int launch_simt(Plan &plan, int route)
{
    static_assert(kMinBlocks == 1, "the split planner assumes one CTA per multiprocessor");
    const bool a_kin = !plan.transA, b_kin = plan.transB;
    if (route == kRouteSimtSmall) {
        if (a_kin && b_kin) return launch_cfg<SimtSmall, true, true>(plan);
        if (a_kin) return launch_cfg<SimtSmall, true, false>(plan);
        if (b_kin) return launch_cfg<SimtSmall, false, true>(plan);
        return launch_cfg<SimtSmall, false, false>(plan);
    }
    if (a_kin && b_kin) return launch_cfg<SimtNarrow, true, true>(plan);
    if (a_kin) return launch_cfg<SimtWide, true, false>(plan);
    if (b_kin) return launch_cfg<SimtWide, false, true>(plan);
    return launch_cfg<SimtWide, false, false>(plan);
}

}  // namespace sg
