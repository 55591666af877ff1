// kernels_tc.cu -- host launcher of the tcgen05 tensor-core paths
// (tc_tf32.cuh): 3xTF32 (FP32 accuracy) and plain TF32.
#include <cstring>

#include "../../include/sgemm.h"
#include "internal.h"
#include "tc_tf32.cuh"

namespace sg {

namespace {

constexpr int kBN = 128;
constexpr int kGroupM = 8;

template <bool SPLIT3, bool A_KIN, bool B_KIN, bool USE_TMA>
int launch_one(Plan &plan, const CUtensorMap &tmA, const CUtensorMap &tmB)
{
    using C = tc::Cfg<kBN, SPLIT3, A_KIN, B_KIN, USE_TMA>;
    auto kern = tc::tc_sgemm_kernel<C>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    long long grid = plan.p.num_units;
    if (grid > plan.num_sms) grid = plan.num_sms;
    kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, plan.stream>>>(tmA, tmB,
                                                                                 plan.p);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    return plan.p.splits > 1 ? launch_fixup(plan, tc::BM, kBN) : SGEMM_OK;
}

template <bool SPLIT3, bool USE_TMA>
int dispatch_layout(Plan &plan, const CUtensorMap &tmA, const CUtensorMap &tmB)
{
    const bool a_kin = !plan.transA, b_kin = plan.transB;
    if (a_kin && !b_kin) return launch_one<SPLIT3, true, false, USE_TMA>(plan, tmA, tmB);
    if (a_kin && b_kin) return launch_one<SPLIT3, true, true, USE_TMA>(plan, tmA, tmB);
    if (!a_kin && !b_kin) return launch_one<SPLIT3, false, false, USE_TMA>(plan, tmA, tmB);
    return launch_one<SPLIT3, false, true, USE_TMA>(plan, tmA, tmB);
}

}  // namespace

void tc_tile_dims(int &bm, int &bn)
{
    bm = tc::BM;
    bn = kBN;
}

int launch_tc(Plan &plan)
{
    GemmParams &p = plan.p;
    p.tiles_m = (p.M + tc::BM - 1) / tc::BM;
    p.tiles_n = (p.N + kBN - 1) / kBN;
    p.k_blocks = (p.K + tc::BK - 1) / tc::BK;
    p.group_m = kGroupM;
    p.num_tiles = static_cast<long long>(p.Q) * p.tiles_m * p.tiles_n;
    plan.even_k = (p.K % tc::BK) == 0;

    alignas(64) CUtensorMap tmA;
    alignas(64) CUtensorMap tmB;
    std::memset(&tmA, 0, sizeof(tmA));
    std::memset(&tmB, 0, sizeof(tmB));
    bool use_tma = plan.a_tma && plan.b_tma;
    if (use_tma) {
        use_tma = encode_operand(&tmA, p.A, !plan.transA, p.M, p.K, p.lda, p.Q, p.sA, tc::BM) &&
                  encode_operand(&tmB, p.B, plan.transB, p.N, p.K, p.ldb, p.Q, p.sB, kBN);
    }
    const int rc = plan_splits(plan, tc::BM, kBN, use_tma);
    if (rc != SGEMM_OK) return rc;
    const bool split3 = plan.mode == SGEMM_MODE_3XTF32;
    if (split3) {
        return use_tma ? dispatch_layout<true, true>(plan, tmA, tmB)
                       : dispatch_layout<true, false>(plan, tmA, tmB);
    }
    return use_tma ? dispatch_layout<false, true>(plan, tmA, tmB)
                   : dispatch_layout<false, false>(plan, tmA, tmB);
}

}  // namespace sg
