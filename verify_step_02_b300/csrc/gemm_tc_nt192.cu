// Tensor-core skinny GEMM kernels for token tiles of 192 columns.
#include "gemm_tc.cuh"

SV_GEMM_TC_INSTANTIATE(192)

