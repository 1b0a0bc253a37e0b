// GEMM tile epilogues of the verify step, shared by the FMA and tcgen05 GEMMs.
//
// A finished tile holds, for kGemmBN weight rows and a run of tokens, the
// float32 sums y[m][n] = x[m] . W[n]. What happens next depends on the
// projection (DSpark summary, "Architecture": one target forward over the
// block; the decoder is the Llama-style pre-norm stack):
//   QKV   rotate q and k by RoPE at the row's absolute position (rotate-half
//         pairing i <-> i + hd/2, both halves of a head are in one tile),
//         write q for attention and k, v into the row's page slot;
//   O, down  add into the float32 residual stream;
//   gate|up  SiLU(gate) * up, both rows of a feature in one tile;
//   LM head  write logits and each token's (max, argmax) over the tile.
#pragma once

#include "device_util.cuh"
#include "internal.h"

namespace sv {

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// ys: tile values, element (t, c) at ys[t * ldys + c] for tile row t < kGemmBN and
// token c < mcount (global token m0 + c). nt: the weight tile index. The tile
// is shared by threads tid = 0 .. nthr-1 (nthr a multiple of 32).
__device__ __forceinline__ void epilogue_tile(const GemmArgs& a, int nt, const float* ys, int ldys, int m0,
                                              int mcount, int tid, int nthr) {
  const Epi& e = a.epi;
  constexpr int BN = kGemmBN;
  if (e.kind == kEpiStore || e.kind == kEpiResid) {
    for (int idx = tid; idx < BN * mcount; idx += nthr) {
      const int c = idx / BN, t = idx - c * BN;
      const int n = nt * BN + t;
      if (n >= a.n_rows) continue;
      const long long m = m0 + c;
      const float v = ys[t * ldys + c];
      if (e.kind == kEpiStore)
        e.y[m * e.ldy + n] = v;
      else
        e.h[m * e.ldh + n] += v;
    }
  } else if (e.kind == kEpiSwiglu) {
    constexpr int HB = BN / 2;
    for (int idx = tid; idx < HB * mcount; idx += nthr) {
      const int c = idx / HB, t = idx - c * HB;
      const int f = nt * HB + t;
      if (f >= e.ffn) continue;
      const float g = ys[t * ldys + c], u = ys[(t + HB) * ldys + c];
      store_x(e.act, e.act_plane, (long long)(m0 + c) * e.ffn + f, silu(g) * u, e.x_pair);
    }
  } else if (e.kind == kEpiQkv) {
    const int hd = e.head_dim, half = hd >> 1;
    const int nq = e.n_heads * hd;
    for (int idx = tid; idx < BN * mcount; idx += nthr) {
      const int c = idx / BN, t = idx - c * BN;
      const int n = nt * BN + t;
      if (n >= a.n_rows) continue;
      const int head = n / hd, i = n - head * hd;
      const int m = m0 + c;
      const int pos = e.row_pos[m];
      if (pos < 0) continue;  // flagged by the row preparation
      float v = ys[t * ldys + c];
      if (head < e.n_heads + e.n_kv_heads) {  // q or k: rotate
        const int ii = i < half ? i : i - half;
        const float2 cs = e.rope[(long long)pos * half + ii];
        if (i < half) {
          const float p = ys[(t + half) * ldys + c];
          v = v * cs.x - p * cs.y;
        } else {
          const float p = ys[(t - half) * ldys + c];
          v = v * cs.x + p * cs.y;
        }
      }
      if (n < nq) {
        e.q_out[(long long)m * nq + n] = v;
      } else {
        const bool is_k = head < e.n_heads + e.n_kv_heads;
        const int kvh = head - e.n_heads - (is_k ? 0 : e.n_kv_heads);
        const int r = e.row_req[m];
        const int pidx = pos / e.page_size;
        const int page = pidx < e.max_pages ? e.page_table[(long long)r * e.max_pages + pidx] : -1;
        if (page < 0 || page >= e.n_pages) {
          atomicOr(e.status, kStBadPage);
          continue;
        }
        const long long off = (((long long)page * e.n_kv_heads + kvh) * e.page_size + (pos - pidx * e.page_size)) *
                                  hd + i;
        store_act(is_k ? e.k_cache : e.v_cache, off, v, e.kv_bf16);
      }
    }
  } else if (e.kind == kEpiLogits) {
    if (e.logits) {
      for (int idx = tid; idx < BN * mcount; idx += nthr) {
        const int c = idx / BN, t = idx - c * BN;
        const int n = nt * BN + t;
        if (n < e.vocab) e.logits[(long long)(m0 + c) * e.vocab + n] = ys[t * ldys + c];
      }
    }
    const int lane = tid & 31, warp = tid >> 5, nw = nthr >> 5;
    for (int c = warp; c < mcount; c += nw) {
      float best = -INFINITY;
      int bi = 0x7fffffff;
      for (int t = lane; t < BN; t += 32) {
        const int n = nt * BN + t;
        if (n < e.vocab) argmax_merge(best, bi, ys[t * ldys + c], n);
      }
      warp_argmax(best, bi);
      if (lane == 0) e.argmax_part[(long long)(m0 + c) * a.n_tiles + nt] = make_float2(best, __int_as_float(bi));
    }
  }
}

// Split-K hand-off. Each split writes its partial tile; the last split to
// arrive (per-tile counter, no waiting) sums the partials in split order —
// a fixed order, so results do not depend on arrival order — resets the
// counter and returns true with the sum in ys.
__device__ __forceinline__ bool splitk_reduce(const GemmArgs& a, int tile_id, int split, const float* mine,
                                              float* ys, int ldys, int rows, int cols) {
  __shared__ unsigned s_last;
  const int tid = threadIdx.x, nthr = blockDim.x;
  float* base = a.partials + (long long)tile_id * a.k_splits * rows * cols;
  float* dst = base + (long long)split * rows * cols;
  for (int idx = tid; idx < rows * cols; idx += nthr) {
    const int t = idx / cols, c = idx - t * cols;
    __stcg(dst + idx, mine[t * ldys + c]);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.counters + tile_id, 1u) == (unsigned)(a.k_splits - 1);
  __syncthreads();
  if (!s_last) return false;
  __threadfence();
  for (int idx = tid; idx < rows * cols; idx += nthr) {
    float s = 0.f;
    for (int sp = 0; sp < a.k_splits; ++sp) s += __ldcg(base + (long long)sp * rows * cols + idx);
    const int t = idx / cols, c = idx - t * cols;
    ys[t * ldys + c] = s;
  }
  if (tid == 0) a.counters[tile_id] = 0u;
  __syncthreads();
  return true;
}

}  // namespace sv
