// kernels_tcp.cu -- host launcher of the CTA-pair tcgen05 kernel
// (tc_pair.cuh): clusters of two CTAs, one pair per two multiprocessors,
// persistent over 256 x 128 tiles.
#include <atomic>

#include "../../include/sgemm.h"
#include "internal.h"
#include "tc_pair.cuh"

namespace sg {

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_slots[kMaxDevices];

template <bool SPLIT3, bool A_KIN, bool B_KIN, bool WIDE>
int launch_one(Plan &plan, const CUtensorMap &tmA, const CUtensorMap &tmB, int slots)
{
    using C = tcp::Cfg<SPLIT3, A_KIN, B_KIN, WIDE>;
    auto kern = tcp::tcp_sgemm_kernel<C>;
    if (!smem_attr_once(reinterpret_cast<const void *>(kern), C::SMEM_BYTES))
        return SGEMM_ERR_LAUNCH;
    long long pairs = plan.p.num_units;
    if (pairs > slots) pairs = slots;
    kern<<<static_cast<unsigned>(2 * pairs), tcp::kThreads, C::SMEM_BYTES, plan.stream>>>(
        tmA, tmB, plan.p);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    note_launch();
    return plan.p.splits > 1 ? launch_fixup(plan, tcp::PM, C::BN) : SGEMM_OK;
}

template <bool SPLIT3, bool WIDE>
int dispatch(Plan &plan, const CUtensorMap &tmA, const CUtensorMap &tmB, int slots)
{
    const bool a_kin = !plan.transA, b_kin = plan.transB;
    if (a_kin && !b_kin) return launch_one<SPLIT3, true, false, WIDE>(plan, tmA, tmB, slots);
    if (a_kin && b_kin) return launch_one<SPLIT3, true, true, WIDE>(plan, tmA, tmB, slots);
    if (!a_kin && !b_kin) return launch_one<SPLIT3, false, false, WIDE>(plan, tmA, tmB, slots);
    return launch_one<SPLIT3, false, true, WIDE>(plan, tmA, tmB, slots);
}

}  // namespace

// Pairs that can be resident at once: clusters of two need two free
// multiprocessors of one GPC, so this can be below num_sms / 2.  Asked of
// the runtime once per device (every configuration of the kernel has the
// same thread count and about the same shared memory: one CTA per SM).
int tc_pair_slots(int num_sms)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return num_sms / 2;
    const int cached = g_slots[dev].load();
    if (cached > 0) return cached;
    using C = tcp::Cfg<true, true, false>;
    auto kern = tcp::tcp_sgemm_kernel<C>;
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES) == cudaSuccess) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(2 * (num_sms / 2)));
        cfg.blockDim = dim3(tcp::kThreads);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();  // a refused query leaves no error behind
    if (n <= 0 || n > num_sms / 2) n = num_sms / 2;
    if (n < 1) n = 1;
    g_slots[dev].store(n);
    return n;
}

int launch_tc_pair(Plan &plan, const CUtensorMap &tmA, const CUtensorMap &tmB, int slots)
{
    if (plan.mode == SGEMM_MODE_3XTF32) return dispatch<true, false>(plan, tmA, tmB, slots);
    if (tcp::pair_wide(false, plan.p.K)) return dispatch<false, true>(plan, tmA, tmB, slots);
    return dispatch<false, false>(plan, tmA, tmB, slots);
}

}  // namespace sg
