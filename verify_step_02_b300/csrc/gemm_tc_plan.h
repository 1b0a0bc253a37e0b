// Shared-memory plan of the tensor-core skinny GEMM (gemm_tc.cuh): stage
// sizes, pipeline depth and K step per token tile width, as compile-time
// functions so that the host plan and the kernel instantiations agree.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include "internal.h"

namespace sv {
namespace tcg {

constexpr int kTcThreads = 384;     // warp 0 TMA, warp 1 MMA, warps 4-11 epilogue (two warpgroups)
constexpr int kTcThreadsW12 = 512;  // W12: warps 4-7 epilogue, warps 2, 3 and 8-15 rebuild weights
constexpr int kEpiThreads = 256;
constexpr int kYsLd = 33;                       // Ys row stride (floats)
constexpr int kABytes = kGemmBN * 128;          // weight tile of one 64-wide sub-tile: 128 rows x 64 bf16
constexpr int kSmemBudget = 225 * 1024;
constexpr int kW12Planes = 3 * 2 * 4096;        // one W12 unit: 3 planes x 2 row halves x 4 KB
constexpr int kW12Ring = 2;                     // rebuilt W12 weight tiles in flight
constexpr int kW12MaxNT = 64;                   // widest token tile of the W12 variant
constexpr int kClusterMaxNT = 64;               // widest token tile of the cluster split
constexpr int kClusterMaxSize = 8;              // CTAs per cluster (the portable maximum)

// One pipeline stage covers ks K-elements (ks / 64 swizzled sub-tiles of 64).
// bf16 weights: per sub-tile the weight tile, then the x tile(s). W12 weights
// (ks = 128): the three planes' 64 x 128 tiles of both row halves (24 KB),
// then the x tiles; the rebuilt bf16 weight tiles live in a separate ring.
constexpr int stage_bytes(int nt, bool pair, int ks, bool w12) {
  return w12 ? kW12Planes + (ks / 64) * nt * 128 * (pair ? 2 : 1) : (ks / 64) * (kABytes + nt * 128 * (pair ? 2 : 1));
}

// Token columns each rank of a cluster of cs CTAs reduces and finishes (a
// multiple of 4, so the slice reads are 16-byte vectors).
constexpr int cl_slice(int nt, int cs) { return ((nt + cs - 1) / cs + 3) / 4 * 4; }

// cs > 0: the cluster split, whose epilogue works on a slice of the tokens: its
// tile values Ys [128][slice + 1], its staged inputs Es [128][slice] and the
// slices every rank pushes to it, Rx [cs][128][slice], replace the stream-K
// Ys [128][33] and the launch's per-token data.
constexpr size_t tc_smem_bytes(int nt, bool pair, int ks, int stages, bool w12, int cs = 0) {
  return 1024 + static_cast<size_t>(stages) * stage_bytes(nt, pair, ks, w12) +
         (w12 ? static_cast<size_t>(kW12Ring) * (ks / 64) * kABytes : 0) +
         (cs > 0 ? sizeof(float) * kGemmBN * (cl_slice(nt, cs) * (cs + 2) + 1)
                 : sizeof(float) * kGemmBN * kYsLd + sizeof(TokData)) +
         sizeof(EpiSmem) + sizeof(uint64_t) * (2 * stages + 11) + 16;
}

constexpr int tc_stages_for(int nt, bool pair, int ks, bool w12, int cs = 0) {
  return (kSmemBudget - static_cast<int>(tc_smem_bytes(nt, pair, ks, 0, w12, cs) + 16 * sizeof(uint64_t))) /
                     stage_bytes(nt, pair, ks, w12) > 8
             ? 8
             : (kSmemBudget - static_cast<int>(tc_smem_bytes(nt, pair, ks, 0, w12, cs) + 16 * sizeof(uint64_t))) /
                   stage_bytes(nt, pair, ks, w12);
}

// K elements per pipeline stage for a token tile of nt columns: the widest of
// 256 / 128 / 64 that still leaves three stages (W12: always 128, its tile width).
constexpr int tc_ks_for(int nt, bool pair, bool w12) {
  return w12 ? 128
             : tc_stages_for(nt, pair, 256, false) >= 3 ? 256
             : tc_stages_for(nt, pair, 128, false) >= 3 ? 128
                                                        : 64;
}

// Launch of the kernel instantiation for token tile NT (gemm_tc_nt*.cu); CL:
// the cluster split (a.cl_size CTAs per cluster, a.cl_tiles tiles each).
template <int NT, bool PAIR, bool W12, bool CL>
cudaError_t gemm_tc_launch(const GemmArgs& a, const CUtensorMap& w, const CUtensorMap& x, cudaStream_t s);
// Clusters of cs CTAs of that instantiation (with `stages` pipeline stages) that fit on the device at once.
template <int NT, bool PAIR, bool W12, bool CL>
int gemm_tc_max_clusters(int cs, int stages);

}  // namespace tcg
}  // namespace sv
