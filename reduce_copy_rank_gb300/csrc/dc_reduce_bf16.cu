// dc_reduce_bf16.cu -- fixed-order reduction kernels for bf16 elements (the
// kernels themselves are in dc_reduce.cuh).
#include "dc_reduce.cuh"

DC_REDUCE_INSTANTIATE(kBF16, bf16)
