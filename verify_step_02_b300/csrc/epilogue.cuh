// GEMM tile epilogues of the verify step, shared by the FMA and tcgen05 GEMMs.
//
// A finished tile holds, for kGemmBN weight rows and a run of tokens, the
// float32 sums y[m][n] = x[m] . W[n]. What happens next depends on the
// projection (DSpark summary, "Architecture": one target forward over the
// block; the decoder is the Llama-style pre-norm stack):
//   QKV   rotate q and k by RoPE at the row's absolute position (rotate-half
//         pairing i <-> i + hd/2, both halves of a head are in one tile),
//         write q for attention and k, v into the row's page slot;
//   O, down  add into the float32 residual stream h, then write the next
//         projection's x tensor h * gain and the tile's sums of h^2 per token
//         (the statistics of the next RMSNorm);
//   gate|up  SiLU(gate) * up, both rows of a feature in one tile;
//   LM head  write logits and each token's (max, argmax) over the tile.
// RMSNorm is folded in: y = W (h * g / rms) = (W (h * g)) / rms, so the
// products consume x = h * g and their epilogues scale token m by
// 1 / rms_m = rsqrt(sum of the tiles' h^2 / d + eps), summed in tile order.
//
// Thread layout: thread tid owns tile row t = tid % kGemmBN and tokens
// tid / kGemmBN, + nthr / kGemmBN, ... (nthr a multiple of kGemmBN).
#pragma once

#include "device_util.cuh"
#include "internal.h"

namespace sv {

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// Per-token data of block row m: the RMSNorm scale 1 / rms (1 when the
// product's input is not a normed x), and for the QKV product the row's
// position and the page-pool row of its slot (kv head 0), or -1.
__device__ __forceinline__ void token_data(const Epi& e, int m, float& rs, int& pos, long long& kvo) {
  rs = 1.f;
  if (e.ss_in) {
    const float* p = e.ss_in + static_cast<long long>(m) * e.n_ss;
    float s = 0.f;
    for (int i0 = 0; i0 < e.n_ss; i0 += 8) {  // loads in flight together, sums in tile order
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = i0 + i < e.n_ss ? __ldcg(p + i0 + i) : 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) s += v[i];
    }
    rs = rsqrtf(s / static_cast<float>(e.d_model) + e.eps);
  }
  pos = -1;
  kvo = -1;
  if (e.kind == kEpiQkv) {
    pos = e.row_pos[m];
    if (pos >= 0) {
      const int r = e.row_req[m], pidx = pos / e.page_size;
      const int page = pidx < e.max_pages ? e.page_table[static_cast<long long>(r) * e.max_pages + pidx] : -1;
      if (page < 0 || page >= e.n_pages)
        atomicOr(e.status, kStBadPage);
      else
        kvo = static_cast<long long>(page) * e.n_kv_heads * e.page_size + (pos - pidx * e.page_size);
    }
  }
}

// Bring the global inputs the epilogue of tile nt will read (the residual h
// rows, the RoPE rows of the tokens' positions) into L1 ahead of time, so that
// a split tile's last arriver does not pay their latency after the reduction.
__device__ __forceinline__ void epilogue_prefetch(const GemmArgs& a, int nt, int m0, int mcount, int tid,
                                                  const TokData* td) {
  const Epi& e = a.epi;
  const int t = tid % kGemmBN, n = nt * kGemmBN + t;
  if (n >= a.n_rows) return;
  if (e.kind == kEpiResid) {
    if (e.next_gain)
      asm volatile("prefetch.global.L1 [%0];" ::"l"(static_cast<const char*>(e.next_gain) + (e.gain_bf16 ? 2 : 4) * n));
    for (int c = 0; c < mcount; ++c)
      asm volatile("prefetch.global.L1 [%0];" ::"l"(e.h + static_cast<long long>(m0 + c) * e.ldh + n));
  } else if (e.kind == kEpiQkv && td) {
    const int hd = e.head_dim, half = hd >> 1, head = n / hd, i = n - head * hd;
    if (head >= e.n_heads + e.n_kv_heads) return;  // v rows are not rotated
    const int ii = i < half ? i : i - half;
    for (int c = 0; c < mcount; ++c) {
      const int pos = td->pos[m0 + c];
      if (pos >= 0) asm volatile("prefetch.global.L1 [%0];" ::"l"(e.rope + static_cast<long long>(pos) * half + ii));
    }
  }
}

// ys: tile values, element (t, c) at ys[t * ldys + c] for tile row t < kGemmBN and
// token c < mcount <= 32 (global token m0 + c). nt: the weight tile index.
// td: the launch's per-token data, or nullptr (computed here, per tile).
// sync(): a barrier over the nthr threads that run the epilogue.
template <class Sync>
__device__ __forceinline__ void epilogue_tile(const GemmArgs& a, int nt, float* ys, int ldys, int m0, int mcount,
                                              int tid, int nthr, EpiSmem& sm, const TokData* td, Sync sync) {
  const Epi& e = a.epi;
  constexpr int BN = kGemmBN;
  const int t = tid % BN, cg = tid / BN, ng = nthr / BN;
  const int lane = tid & 31, rg = t >> 5;

  // ---- per-token data of the tile's tokens
  if (tid < mcount) {
    const int m = m0 + tid;
    if (td) {
      sm.rstd[tid] = td->rstd[m];
      sm.pos[tid] = td->pos[m];
      sm.kv[tid] = td->kv[m];
    } else {
      token_data(e, m, sm.rstd[tid], sm.pos[tid], sm.kv[tid]);
    }
  }
  sync();

  if (e.kind == kEpiStore) {
    const int n = nt * BN + t;
    if (n < a.n_rows)
      for (int c = cg; c < mcount; c += ng) e.y[static_cast<long long>(m0 + c) * e.ldy + n] = ys[t * ldys + c];
  } else if (e.kind == kEpiResid) {
    const int n = nt * BN + t;
    const bool valid = n < a.n_rows;
    const float g = (valid && e.next_gain) ? load_act(e.next_gain, n, e.gain_bf16) : 0.f;
    for (int c0 = cg; c0 < mcount; c0 += 16 * ng) {
      float hv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int c = c0 + i * ng;
        hv[i] = (valid && c < mcount) ? e.h[static_cast<long long>(m0 + c) * e.ldh + n] : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int c = c0 + i * ng;
        const bool live = valid && c < mcount;
        const float hn = live ? hv[i] + ys[t * ldys + c] : 0.f;
        if (live) {
          e.h[static_cast<long long>(m0 + c) * e.ldh + n] = hn;
          if (e.next_gain)
            store_x(e.x_out, e.x_out_plane, static_cast<long long>(m0 + c) * e.d_model + n, hn * g, e.x_pair);
        }
        if (c < mcount) ys[t * ldys + c] = hn * hn;  // this thread's own tile slot, already consumed
      }
    }
    if (e.ss_out) {
      // the tile's sum of h^2 per token: warp w sums tokens w, w + nthr/32, ..
      // over the 128 rows (rows lane + 32k, k in order, then a shuffle tree)
      sync();
      for (int c = tid >> 5; c < mcount; c += nthr >> 5) {
        float q = 0.f;
#pragma unroll
        for (int k = 0; k < BN / 32; ++k) q += ys[(lane + 32 * k) * ldys + c];
        q = warp_sum(q);
        if (lane == 0) e.ss_out[static_cast<long long>(m0 + c) * e.n_ss + nt] = q;
      }
    }
  } else if (e.kind == kEpiSwiglu) {
    constexpr int HB = BN / 2;
    const int f = nt * HB + t;
    if (t < HB && f < e.ffn) {
      for (int c = cg; c < mcount; c += ng) {
        const float rs = sm.rstd[c];
        const float gv = ys[t * ldys + c] * rs, uv = ys[(t + HB) * ldys + c] * rs;
        store_x(e.act, e.act_plane, static_cast<long long>(m0 + c) * e.ffn + f, silu(gv) * uv, e.x_pair);
      }
    }
  } else if (e.kind == kEpiQkv) {
    const int hd = e.head_dim, half = hd >> 1;
    const int nq = e.n_heads * hd;
    const int n = nt * BN + t;
    if (n < a.n_rows) {
      const int head = n / hd, i = n - head * hd;
      const bool rot = head < e.n_heads + e.n_kv_heads;  // q or k
      const int ii = i < half ? i : i - half;
      const int tp = i < half ? t + half : t - half;       // partner row of the rotation
      const float sgn = i < half ? -1.f : 1.f;
      const bool is_q = n < nq;
      const int kvh = is_q ? 0 : head - e.n_heads - (rot ? 0 : e.n_kv_heads);
      for (int c0 = cg; c0 < mcount; c0 += 16 * ng) {
        float2 cs[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int c = c0 + j * ng;
          const int pos = c < mcount ? sm.pos[c] : -1;
          cs[j] = (rot && pos >= 0) ? __ldg(e.rope + static_cast<long long>(pos) * half + ii) : make_float2(1.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int c = c0 + j * ng;
          if (c >= mcount) continue;
          const int pos = sm.pos[c];
          if (pos < 0) continue;  // flagged by the row preparation
          const float rs = sm.rstd[c];
          float v = ys[t * ldys + c] * rs;
          if (rot) v = v * cs[j].x + sgn * (ys[tp * ldys + c] * rs) * cs[j].y;
          const long long m = m0 + c;
          if (is_q) {
            if (e.q_pair)
              store_x(e.q_pair, e.q_plane, m * nq + n, v * e.q_scale, 1);
            else
              e.q_out[m * nq + n] = v;
          } else {
            const long long kvo = sm.kv[c];
            if (kvo < 0) continue;
            const long long off = (kvo + static_cast<long long>(kvh) * e.page_size) * hd + i;
            store_act(rot ? e.k_cache : e.v_cache, off, v, e.kv_bf16);
          }
        }
      }
    }
  } else if (e.kind == kEpiLogits) {
    const int n = nt * BN + t;
    const bool valid = n < e.vocab;
    for (int c = cg; c < mcount; c += ng) {
      const float v = valid ? ys[t * ldys + c] * sm.rstd[c] : -INFINITY;
      if (e.logits && valid) e.logits[static_cast<long long>(m0 + c) * e.vocab + n] = v;
      float best = v;
      int bi = valid ? n : 0x7fffffff;
      warp_argmax(best, bi);
      if (lane == 0) {
        sm.red[rg][c] = best;
        sm.redi[rg][c] = bi;
      }
    }
    sync();
    if (tid < mcount) {
      float best = sm.red[0][tid];
      int bi = sm.redi[0][tid];
      for (int g = 1; g < 4; ++g) argmax_merge(best, bi, sm.red[g][tid], sm.redi[g][tid]);
      e.argmax_part[static_cast<long long>(m0 + tid) * a.n_tiles + nt] = make_float2(best, __int_as_float(bi));
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
