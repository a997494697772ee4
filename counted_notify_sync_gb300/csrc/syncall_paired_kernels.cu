// syncall_paired_kernels.cu -- the kernel table of the hard SYNCALL path with
// the paired-mbarrier step (CNS_HARD_STEP_PAIRED_MBARRIER): one
// syncall_kernel<HARD, workload, variant, paired> per pair (a translation
// unit of its own, compiled in parallel with the others).
#include <array>
#include <utility>

#include "syncall_kernels.cuh"

namespace cns {
namespace {

template <int WL, int... Vs>
constexpr std::array<KernelFn, sizeof...(Vs)> paired_row(std::integer_sequence<int, Vs...>)
{
    return {{syncall_kernel<CNS_SYNCALL_HARD, WL, Vs, kHardStepPairedMbarrier>...}};
}

template <int... WLs>
constexpr std::array<std::array<KernelFn, kBvCount>, sizeof...(WLs)> paired_table(std::integer_sequence<int, WLs...>)
{
    return {{paired_row<WLs>(std::make_integer_sequence<int, kBvCount>{})...}};
}

}  // namespace

KernelFn pick_paired_kernel(int wl, int variant)
{
    static constexpr auto t = paired_table(std::make_integer_sequence<int, CNS_WL_JACOBI + 1>{});
    return t[wl][variant];
}

}  // namespace cns
