// GEMV instantiations for q6_K: the tile kernel for every column count and mode
// (gemv_tiles.cuh), and the generic fallback.
#include "gemv_generic.cuh"
#include "gemv_tiles.cuh"
#include "kernels.h"

namespace qmv {

const void *gemv_tiles_fn_q6_K(int mode, int nc, int rw) { return tiles_kernel_fn<FMT_Q6_K>(mode, nc, rw); }

const void *gemv_tiles_probe_fn_q6_K(int mode, int nc) { return tiles_probe_kernel_fn<FMT_Q6_K>(mode, nc); }

const void *gemv_tiles_yq_fn_q6_K(int mode, bool probe) { return tiles_yq_kernel_fn<FMT_Q6_K>(mode, probe); }

const void *gemv_tiles_rowrun_fn_q6_K(int mode, int nc) { return tiles_rowrun_kernel_fn<FMT_Q6_K>(mode, nc); }

const void *gemv_generic_fn_q6_K(int mode)
{
    constexpr int F = FMT_Q6_K;
    switch (mode) {
    case MODE_PLAIN: return reinterpret_cast<const void *>(&gemv_generic_kernel<F, MODE_PLAIN>);
    case MODE_GATE: return reinterpret_cast<const void *>(&gemv_generic_kernel<F, MODE_GATE>);
    case MODE_MOE: return reinterpret_cast<const void *>(&gemv_generic_kernel<F, MODE_MOE>);
    case MODE_DEBUG: return reinterpret_cast<const void *>(&gemv_generic_kernel<F, MODE_DEBUG>);
    default: return nullptr;
    }
}

}  // namespace qmv
