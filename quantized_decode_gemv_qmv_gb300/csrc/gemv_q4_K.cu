// GEMV instantiations for q4_K: streaming (units) kernel for every column count and
// mode, and the generic fallback.
#include "gemv_generic.cuh"
#include "gemv_units.cuh"
#include "kernels.h"

namespace qmv {

const void *gemv_stream_fn_q4_K(int mode, int nc)
{
    constexpr int F = FMT_Q4_K;
    if (mode == MODE_PLAIN) {
        switch (nc) {
        case 1: return reinterpret_cast<const void *>(&gemv_units_kernel<F, 1, MODE_PLAIN>);
        case 2: return reinterpret_cast<const void *>(&gemv_units_kernel<F, 2, MODE_PLAIN>);
        case 3: return reinterpret_cast<const void *>(&gemv_units_kernel<F, 3, MODE_PLAIN>);
        case 4: return reinterpret_cast<const void *>(&gemv_units_kernel<F, 4, MODE_PLAIN>);
        case 5: return reinterpret_cast<const void *>(&gemv_units_kernel<F, 5, MODE_PLAIN>);
        case 6: return reinterpret_cast<const void *>(&gemv_units_kernel<F, 6, MODE_PLAIN>);
        case 7: return reinterpret_cast<const void *>(&gemv_units_kernel<F, 7, MODE_PLAIN>);
        case 8: return reinterpret_cast<const void *>(&gemv_units_kernel<F, 8, MODE_PLAIN>);
        default: return nullptr;
        }
    }
#define QMV_MODE_CASES(MODE)                                                                     \
    switch (nc) {                                                                                \
    case 1: return reinterpret_cast<const void *>(&gemv_units_kernel<F, 1, MODE>);             \
    case 2: return reinterpret_cast<const void *>(&gemv_units_kernel<F, 2, MODE>);             \
    case 4: return reinterpret_cast<const void *>(&gemv_units_kernel<F, 4, MODE>);             \
    case 8: return reinterpret_cast<const void *>(&gemv_units_kernel<F, 8, MODE>);             \
    default: return nullptr;                                                                     \
    }
    if (mode == MODE_GATE) { QMV_MODE_CASES(MODE_GATE) }
    if (mode == MODE_MOE) { QMV_MODE_CASES(MODE_MOE) }
    if (mode == MODE_DEBUG) { QMV_MODE_CASES(MODE_DEBUG) }
#undef QMV_MODE_CASES
    return nullptr;
}

const void *gemv_generic_fn_q4_K(int mode)
{
    constexpr int F = FMT_Q4_K;
    switch (mode) {
    case MODE_PLAIN: return reinterpret_cast<const void *>(&gemv_generic_kernel<F, MODE_PLAIN>);
    case MODE_GATE: return reinterpret_cast<const void *>(&gemv_generic_kernel<F, MODE_GATE>);
    case MODE_MOE: return reinterpret_cast<const void *>(&gemv_generic_kernel<F, MODE_MOE>);
    case MODE_DEBUG: return reinterpret_cast<const void *>(&gemv_generic_kernel<F, MODE_DEBUG>);
    default: return nullptr;
    }
}

}  // namespace qmv
