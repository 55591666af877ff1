// kernels_tc.cu -- host launcher of the tcgen05 tensor-core paths: 3xTF32
// (FP32 accuracy) and plain TF32.  Operands TMA can describe run on the
// CTA-pair kernel (tc_pair.cuh, launched from kernels_tcp.cu): 256 x 128
// tiles, TMA-staged operands, each CTA of a pair converting half of B.
// Others (a row pitch or batch stride that is not a multiple of 16 bytes, an
// unaligned base) run on the direct kernel (tc_direct.cuh), whose converter
// warps load them from global memory themselves.  Measured on GB300: the
// direct kernel runs the ragged 1000 x 1500 x 777 case (lda = 777) at 43
// TFLOP/s where staging it with cp.async gave 19-25, but it is slower than
// TMA for aligned operands (114 TFLOP/s at 4092^3: its loads wait on L2
// latency that the TMA ring hides).
#include <cstring>

#include "../../include/sgemm.h"
#include "internal.h"
#include "tc_direct.cuh"
#include "tc_pair.cuh"

namespace sg {

namespace {

constexpr int kBN = 128;
constexpr int kGroupM = 8;

template <bool SPLIT3, bool A_KIN, bool B_KIN>
int launch_direct(Plan &plan)
{
    using C = tcd::Cfg<kBN, SPLIT3, A_KIN, B_KIN>;
    auto kern = tcd::tcd_sgemm_kernel<C>;
    if (!smem_attr_once(reinterpret_cast<const void *>(kern), C::SMEM_BYTES))
        return SGEMM_ERR_LAUNCH;
    long long grid = plan.p.num_units;
    if (grid > plan.num_sms) grid = plan.num_sms;
    kern<<<static_cast<unsigned>(grid), tcd::kThreads, C::SMEM_BYTES, plan.stream>>>(plan.p);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    note_launch();
    return plan.p.splits > 1 ? launch_fixup(plan, tc::BM, kBN) : SGEMM_OK;
}

template <bool SPLIT3>
int dispatch_direct(Plan &plan)
{
    const bool a_kin = !plan.transA, b_kin = plan.transB;
    if (a_kin && !b_kin) return launch_direct<SPLIT3, true, false>(plan);
    if (a_kin && b_kin) return launch_direct<SPLIT3, true, true>(plan);
    if (!a_kin && !b_kin) return launch_direct<SPLIT3, false, false>(plan);
    return launch_direct<SPLIT3, false, true>(plan);
}

}  // namespace

void tc_tile_dims(int mode, int K, bool pair, int &bm, int &bn)
{
    bm = pair ? tcp::PM : tc::BM;
    bn = pair ? tcp::pair_shape(tcp::pair_wide(mode == SGEMM_MODE_3XTF32, K)).bn : kBN;
}

int launch_tc(Plan &plan, int route)
{
    GemmParams &p = plan.p;
    p.k_blocks = (p.K + tc::BK - 1) / tc::BK;
    p.group_m = kGroupM;
    plan.even_k = (p.K % tc::BK) == 0;

    alignas(64) CUtensorMap tmA;
    alignas(64) CUtensorMap tmB;
    std::memset(&tmA, 0, sizeof(tmA));
    std::memset(&tmB, 0, sizeof(tmB));
    const tcp::PairShape sh =
        tcp::pair_shape(tcp::pair_wide(plan.mode == SGEMM_MODE_3XTF32, p.K));
    if (route != kRouteTcDirect && plan.a_tma && plan.b_tma &&
        encode_operand(&tmA, p.A, !plan.transA, p.M, p.K, p.lda, p.Q, p.sA, tcp::BM) &&
        encode_operand(&tmB, p.B, plan.transB, p.N, p.K, p.ldb, p.Q, p.sB, sh.hn)) {
        p.k_blocks = (p.K + sh.stage_k - 1) / sh.stage_k;  // the pair kernel's stages
        p.tiles_m = (p.M + tcp::PM - 1) / tcp::PM;
        p.tiles_n = (p.N + sh.bn - 1) / sh.bn;
        p.num_tiles = static_cast<long long>(p.Q) * p.tiles_m * p.tiles_n;
        const int slots = tc_pair_slots(plan.num_sms);
        const int rc = plan_splits(plan, tcp::PM, sh.bn, kFeedPair, slots);
        if (rc != SGEMM_OK) return rc;
        return launch_tc_pair(plan, tmA, tmB, slots);
    }
    p.tiles_m = (p.M + tc::BM - 1) / tc::BM;
    p.tiles_n = (p.N + kBN - 1) / kBN;
    p.num_tiles = static_cast<long long>(p.Q) * p.tiles_m * p.tiles_n;
    const int rc = plan_splits(plan, tc::BM, kBN, kFeedDirect, plan.num_sms);
    if (rc != SGEMM_OK) return rc;
    return plan.mode == SGEMM_MODE_3XTF32 ? dispatch_direct<true>(plan)
                                          : dispatch_direct<false>(plan);
}

}  // namespace sg
