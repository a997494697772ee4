// syncall_hard_kernels.cu -- the kernel table of the hard SYNCALL path with
// the cluster-barrier step: one syncall_kernel<HARD, workload, variant> per
// pair (a translation unit of its own, compiled in parallel with the others).
#include <array>
#include <utility>

#include "syncall_kernels.cuh"

namespace cns {
namespace {

template <int WL, int... Vs>
constexpr std::array<KernelFn, sizeof...(Vs)> hard_row(std::integer_sequence<int, Vs...>)
{
    return {{syncall_kernel<CNS_SYNCALL_HARD, WL, Vs, kHardStepClusterBarrier>...}};
}

template <int... WLs>
constexpr std::array<std::array<KernelFn, kBvCount>, sizeof...(WLs)> hard_table(std::integer_sequence<int, WLs...>)
{
    return {{hard_row<WLs>(std::make_integer_sequence<int, kBvCount>{})...}};
}

}  // namespace

KernelFn pick_hard_kernel(int wl, int variant)
{
    static constexpr auto t = hard_table(std::make_integer_sequence<int, CNS_WL_JACOBI + 1>{});
    return t[wl][variant];
}

}  // namespace cns
