// L2 prefetch of a later matrix product's weights (see L2Window).
//
// The step is a chain of weight-streaming products whose boundaries leave HBM
// idle: a kernel's tail (its last accumulators, the split reduction, the
// epilogue), the next kernel's start and its dependency wait. Every kernel
// requests part of the next product's weights into L2 as soon as its own
// loads are issued, so HBM keeps streaming through the boundary and the next
// kernel finds that part in L2.
#pragma once

#include "internal.h"
#include "tc_ptx.cuh"

namespace sv {
using tc::prefetch_l2_bulk;

// Run by one whole warp. cta / ncta: this kernel's CTA index and grid size.
__device__ __forceinline__ void l2_prefetch_window(const L2Window& pf, int cta, int ncta, int lane) {
  if (!pf.w || pf.count <= 0 || pf.grid_p <= 0) return;
  const char* w = static_cast<const char*>(pf.w);
  const int row_blocks = (pf.n_rows + 63) / 64;
  for (int tc = cta; tc < pf.grid_p; tc += ncta) {
    const long long u0 = tc * pf.U / pf.grid_p, u1 = (tc + 1) * pf.U / pf.grid_p;
    long long ua = u0 + pf.first;
    const long long ub = ua + pf.count < u1 ? ua + pf.count : u1;
    while (ua < ub) {
      const long long t = ua / pf.kb;
      const long long te = ub < (t + 1) * pf.kb ? ub : (t + 1) * pf.kb;
      const int kb0 = static_cast<int>(ua - t * pf.kb), kb1 = static_cast<int>(te - t * pf.kb);
      const int nt = static_cast<int>(t / pf.m_tiles);
      // the tile's two 64-row halves
      const int r0 = pf.pair == kPairSwiglu ? nt * (kGemmBN / 2) : nt * kGemmBN;
      const int r1 = pf.pair == kPairSwiglu ? pf.ffn + nt * (kGemmBN / 2) : r0 + kGemmBN / 2;
      if (pf.wdtype == SV_W12) {
        // plane p, half hh: tiles (row block, kb0 .. kb1 - 1) are contiguous
        if (lane < 6) {
          const int p = lane % 3, hh = lane / 3;
          const int rb = (hh ? r1 : r0) / 64;
          if (rb < row_blocks)
            prefetch_l2_bulk(w + p * pf.w12_plane + (static_cast<long long>(rb) * pf.w12_kt + kb0) * 4096,
                             static_cast<uint32_t>(kb1 - kb0) * 4096u);
        }
      } else {
        const int k_lo = kb0 * pf.ks, k_hi = kb1 * pf.ks < pf.K ? kb1 * pf.ks : pf.K;
        for (int i = lane; i < kGemmBN; i += 32) {
          const int r = i < kGemmBN / 2 ? r0 + i : r1 + i - kGemmBN / 2;
          if (r < pf.n_rows && k_hi > k_lo)
            prefetch_l2_bulk(w + (static_cast<long long>(r) * pf.K + k_lo) * 2, static_cast<uint32_t>(k_hi - k_lo) * 2u);
        }
      }
      ua = te;
    }
  }
}

}  // namespace sv
