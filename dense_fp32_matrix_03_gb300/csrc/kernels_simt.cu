// kernels_simt.cu -- instantiations and the host launcher of the FP32
// CUDA-core SGEMM kernel (simt_fp32.cuh).
#include <cstring>

#include "../../include/sgemm.h"
#include "internal.h"
#include "simt_fp32.cuh"

namespace sg {

namespace {

// Tile configuration of the FP32 path (overridable at build time for
// tuning sweeps): CTA tile BM x BN, warp tile WM x WN, pipeline stages of
// SUBS x 32 k.  Measured on GB300 at 4092^3 (nn): 4 stages of 32 k, 50.1
// TFLOP/s; 3 stages of 64 k, 52.8 (half the barrier round trips per FFMA).
#ifndef SG_SIMT_BM
#define SG_SIMT_BM 128
#define SG_SIMT_BN 128
#define SG_SIMT_WM 64
#define SG_SIMT_WN 32
#define SG_SIMT_STAGES 3
#endif
#ifndef SG_SIMT_SUBS
#define SG_SIMT_SUBS 2
#endif
using SimtMain = SimtCfg<SG_SIMT_BM, SG_SIMT_BN, SG_SIMT_WM, SG_SIMT_WN, SG_SIMT_STAGES, SG_SIMT_SUBS>;
constexpr int kGroupM = 8;

template <class Cfg, bool A_KIN, bool B_KIN, bool USE_TMA, bool EVEN_K>
int launch_one(Plan &plan, const CUtensorMap &tmA, const CUtensorMap &tmB)
{
    auto kern = simt_sgemm_kernel<Cfg, A_KIN, B_KIN, USE_TMA, EVEN_K>;
    // The attribute is per device; setting it on every call costs about a
    // microsecond and keeps the launcher free of per-device caches.
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::SMEM_BYTES) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    long long grid = plan.p.num_units;
    if (grid > static_cast<long long>(plan.num_sms) * kMinBlocks)
        grid = static_cast<long long>(plan.num_sms) * kMinBlocks;
    kern<<<static_cast<unsigned>(grid), Cfg::THREADS, Cfg::SMEM_BYTES, plan.stream>>>(
        tmA, tmB, plan.p);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    return plan.p.splits > 1 ? launch_fixup(plan, Cfg::BM, Cfg::BN) : SGEMM_OK;
}

template <class Cfg, bool USE_TMA, bool EVEN_K>
int dispatch_layout(Plan &plan, const CUtensorMap &tmA, const CUtensorMap &tmB)
{
    const bool a_kin = !plan.transA, b_kin = plan.transB;
    if (a_kin && !b_kin) return launch_one<Cfg, true, false, USE_TMA, EVEN_K>(plan, tmA, tmB);
    if (a_kin && b_kin) return launch_one<Cfg, true, true, USE_TMA, EVEN_K>(plan, tmA, tmB);
    if (!a_kin && !b_kin) return launch_one<Cfg, false, false, USE_TMA, EVEN_K>(plan, tmA, tmB);
    return launch_one<Cfg, false, true, USE_TMA, EVEN_K>(plan, tmA, tmB);
}

}  // namespace

int launch_simt(Plan &plan)
{
    using Cfg = SimtMain;
    GemmParams &p = plan.p;
    p.tiles_m = (p.M + Cfg::BM - 1) / Cfg::BM;
    p.tiles_n = (p.N + Cfg::BN - 1) / Cfg::BN;
    p.k_blocks = (p.K + Cfg::BK - 1) / Cfg::BK;
    p.group_m = kGroupM;
    p.num_tiles = static_cast<long long>(p.Q) * p.tiles_m * p.tiles_n;
    plan.even_k = (p.K % Cfg::BK) == 0;
    static_assert(Cfg::BM == kSplitTile && Cfg::BN == kSplitTile, "split-K workspace tile");
    static_assert(kMinBlocks == 1, "the split planner assumes one CTA per multiprocessor");
    const int rc = plan_splits(plan);
    if (rc != SGEMM_OK) return rc;

    alignas(64) CUtensorMap tmA;
    alignas(64) CUtensorMap tmB;
    std::memset(&tmA, 0, sizeof(tmA));
    std::memset(&tmB, 0, sizeof(tmB));
    bool use_tma = plan.a_tma && plan.b_tma;
    if (use_tma) {
        use_tma = encode_operand(&tmA, p.A, !plan.transA, p.M, p.K, p.lda, p.Q, p.sA, Cfg::BM) &&
                  encode_operand(&tmB, p.B, plan.transB, p.N, p.K, p.ldb, p.Q, p.sB, Cfg::BN);
    }
    if (use_tma) return dispatch_layout<Cfg, true, false>(plan, tmA, tmB);
    if (plan.even_k) return dispatch_layout<Cfg, false, true>(plan, tmA, tmB);
    return dispatch_layout<Cfg, false, false>(plan, tmA, tmB);
}

}  // namespace sg
