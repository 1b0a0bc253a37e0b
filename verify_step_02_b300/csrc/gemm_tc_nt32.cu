// Tensor-core skinny GEMM kernels for token tiles of 32 columns.
#include "gemm_tc.cuh"

SV_GEMM_TC_INSTANTIATE(32)
SV_GEMM_TC_INSTANTIATE_SMALL(32)
