// dc_reduce_f32.cu -- fixed-order reduction kernels for f32 elements (the
// kernels themselves are in dc_reduce.cuh).
#include "dc_reduce.cuh"

DC_REDUCE_INSTANTIATE(kF32, f32)
