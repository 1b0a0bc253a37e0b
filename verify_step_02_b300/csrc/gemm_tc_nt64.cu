// Tensor-core skinny GEMM kernels for token tiles of 64 columns.
#include "gemm_tc.cuh"

SV_GEMM_TC_INSTANTIATE(64)
SV_GEMM_TC_INSTANTIATE_SMALL(64)
