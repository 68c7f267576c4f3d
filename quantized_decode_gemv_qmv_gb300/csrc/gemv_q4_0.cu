// GEMV instantiations for q4_0: the tile kernel for every column count and mode
// (gemv_tiles.cuh), and the generic fallback.
#include "gemv_generic.cuh"
#include "gemv_tiles.cuh"
#include "kernels.h"

namespace qmv {

const void *gemv_tiles_fn_q4_0(int mode, int nc, int rw) { return tiles_kernel_fn<FMT_Q4_0>(mode, nc, rw); }

const void *gemv_tiles_probe_fn_q4_0(int mode, int nc) { return tiles_probe_kernel_fn<FMT_Q4_0>(mode, nc); }

const void *gemv_tiles_yq_fn_q4_0(int mode, bool probe) { return tiles_yq_kernel_fn<FMT_Q4_0>(mode, probe); }

const void *gemv_generic_fn_q4_0(int mode)
{
    constexpr int F = FMT_Q4_0;
    switch (mode) {
    case MODE_PLAIN: return reinterpret_cast<const void *>(&gemv_generic_kernel<F, MODE_PLAIN>);
    case MODE_GATE: return reinterpret_cast<const void *>(&gemv_generic_kernel<F, MODE_GATE>);
    case MODE_MOE: return reinterpret_cast<const void *>(&gemv_generic_kernel<F, MODE_MOE>);
    case MODE_DEBUG: return reinterpret_cast<const void *>(&gemv_generic_kernel<F, MODE_DEBUG>);
    default: return nullptr;
    }
}

}  // namespace qmv
