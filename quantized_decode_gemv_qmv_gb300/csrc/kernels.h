// Host-side entry points of the kernel translation units (internal to libqmv).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace qmv {

struct GemvParams;

// q8_1 and weight quantizers (quantize.cu)
cudaError_t launch_quantize_q8_1(const float *x, int64_t K, int ncols, int64_t ldx, uint8_t *xq, cudaStream_t st,
                                 bool pdl);
cudaError_t launch_quantize_weights(int type, const float *w, int64_t M, int64_t K, int64_t ldw, uint8_t *W,
                                    int64_t row_bytes, cudaStream_t st);

// read-bandwidth probe (quantize.cu): every 16-byte piece of buf read once
cudaError_t launch_read_probe(const void *buf, int64_t bytes, unsigned int *sink, int num_sms, cudaStream_t st);

// Kernel function pointers of the GEMV instantiations (gemv_<type>.cu).
// Tile kernel: template columns nc_t (PLAIN: 1..8; other modes: 1, 2, 4, 8)
// and rows per tile rw.  Returns nullptr for a combination that is not
// instantiated.
const void *gemv_tiles_fn(int type, int mode, int nc_t, int rw);
const void *gemv_generic_fn(int type, int mode);

}  // namespace qmv
