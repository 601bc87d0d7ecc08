// dc_reduce_f16.cu -- fixed-order reduction kernels for f16 elements (the
// kernels themselves are in dc_reduce.cuh).
#include "dc_reduce.cuh"

DC_REDUCE_INSTANTIATE(kF16, f16)
