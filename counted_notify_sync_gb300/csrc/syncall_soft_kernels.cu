// syncall_soft_kernels.cu -- the kernel tables of the soft SYNCALL path: one
// syncall_kernel<SOFT, workload, variant> and one syncall_solo_kernel
// <workload, variant> per pair.  The hard path's tables live in translation
// units of their own, so that the builder compiles them in parallel.
#include <array>
#include <utility>

#include "syncall_kernels.cuh"

namespace cns {
namespace {

template <int WL, int... Vs>
constexpr std::array<KernelFn, sizeof...(Vs)> soft_row(std::integer_sequence<int, Vs...>)
{
    return {{syncall_kernel<CNS_SYNCALL_SOFT, WL, Vs>...}};
}

template <int... WLs>
constexpr std::array<std::array<KernelFn, kBvCount>, sizeof...(WLs)> soft_table(std::integer_sequence<int, WLs...>)
{
    return {{soft_row<WLs>(std::make_integer_sequence<int, kBvCount>{})...}};
}

template <int WL, int... Vs>
constexpr std::array<KernelFn, sizeof...(Vs)> solo_row(std::integer_sequence<int, Vs...>)
{
    return {{syncall_solo_kernel<WL, Vs>...}};
}

template <int... WLs>
constexpr std::array<std::array<KernelFn, kBvCount>, sizeof...(WLs)> solo_table(std::integer_sequence<int, WLs...>)
{
    return {{solo_row<WLs>(std::make_integer_sequence<int, kBvCount>{})...}};
}

}  // namespace

KernelFn pick_soft_kernel(int wl, int variant)
{
    static constexpr auto t = soft_table(std::make_integer_sequence<int, CNS_WL_JACOBI + 1>{});
    return t[wl][variant];
}

// Solo rounds exist for the empty workload and the rings (wl < CNS_WL_JACOBI).
KernelFn pick_solo_kernel(int wl, int variant)
{
    static constexpr auto t = solo_table(std::make_integer_sequence<int, CNS_WL_JACOBI>{});
    return t[wl][variant];
}

}  // namespace cns
