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
      // the KV slot: the position, or for a token tree node C + its index
      const int slot = e.row_slot ? e.row_slot[m] : pos;
      const int r = e.row_req[m], pidx = slot / e.page_size;
      const int page = pidx < e.max_pages ? e.page_table[static_cast<long long>(r) * e.max_pages + pidx] : -1;
      if (pidx >= e.max_pages)
        atomicOr(e.status, kStNoPage);
      else if (page < 0 || page >= e.n_pages)
        atomicOr(e.status, kStBadPage);
      else
        kvo = static_cast<long long>(page) * e.n_kv_heads * e.page_size + (slot - pidx * e.page_size);
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

// Load the global inputs the epilogue of tile nt will read, for tokens
// m0 .. m0 + mcount - 1, into shared memory `es` (kGemmBN x mcount floats, in
// 32-token chunks of kGemmBN * 32): the residual rows h[m][n] (O and down
// products) at es[c * kGemmBN + t] and the tile rows' next-norm gains in
// sm.gain, or the RoPE (cos, sin) of each token's position (QKV product) as
// float2 at es[c * kGemmBN / 2 + ii], ii < head_dim/2.
// Run by nthr threads while the tile's weights stream, so the tile's epilogue
// needs no global loads. td: the launch's per-token data (positions), or
// nullptr when sm.pos already holds the positions of tokens m0 ...
__device__ __forceinline__ void stage_epilogue_inputs(const GemmArgs& a, int nt, int m0, int mcount, float* es,
                                                      EpiSmem& sm, const TokData* td, int tid, int nthr) {
  const Epi& e = a.epi;
  constexpr int U = 8;  // loads in flight per thread
  if (e.kind == kEpiResid) {
    for (int t = tid; t < kGemmBN; t += nthr) {
      const int n = nt * kGemmBN + t;
      sm.gain[t] = n < a.n_rows && e.next_gain ? load_act(e.next_gain, n, e.gain_bf16) : 0.f;
    }
    const int total = kGemmBN * mcount;
    for (int base = tid; base < total; base += U * nthr) {
      float v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int idx = base + u * nthr;
        const int c = idx / kGemmBN, t = idx - c * kGemmBN, n = nt * kGemmBN + t;
        v[u] = idx < total && n < a.n_rows ? e.h[static_cast<long long>(m0 + c) * e.ldh + n] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (base + u * nthr < total) es[base + u * nthr] = v[u];
    }
  } else if (e.kind == kEpiQkv) {
    const int half = e.head_dim >> 1;
    float2* es2 = reinterpret_cast<float2*>(es);
    const int total = (kGemmBN / 2) * mcount;
    for (int base = tid; base < total; base += U * nthr) {
      float2 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int idx = base + u * nthr;
        const int c = idx / (kGemmBN / 2), ii = idx - c * (kGemmBN / 2);
        const int pos = idx >= total ? -1 : td ? td->pos[m0 + c] : sm.pos[c];
        v[u] = pos >= 0 && ii < half ? __ldg(e.rope + static_cast<long long>(pos) * half + ii) : make_float2(1.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (base + u * nthr < total) es2[base + u * nthr] = v[u];
    }
  }
}

// Four float32 values as bf16 (round to nearest even), element 0 in the low half.
__device__ __forceinline__ uint2 bf16x4(float4 v) {
  return make_uint2(static_cast<uint32_t>(f32_to_bf16_bits(v.x)) | static_cast<uint32_t>(f32_to_bf16_bits(v.y)) << 16,
                    static_cast<uint32_t>(f32_to_bf16_bits(v.z)) | static_cast<uint32_t>(f32_to_bf16_bits(v.w)) << 16);
}

__device__ __forceinline__ float4 bf16x4_to_f32(uint2 b) {
  return make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xFFFF0000u), __uint_as_float(b.y << 16),
                     __uint_as_float(b.y & 0xFFFF0000u));
}

// Four consecutive x-tensor elements idx .. idx + 3 (idx and the plane offset
// multiples of 4): float32, or the hi/lo bf16 pair as one 8-byte store per plane.
__device__ __forceinline__ void store_x4(void* base, long long plane, long long idx, float4 v, int pair) {
  if (pair) {
    const uint2 hi = bf16x4(v);
    const float4 hf = bf16x4_to_f32(hi);
    const uint2 lo = bf16x4(make_float4(v.x - hf.x, v.y - hf.y, v.z - hf.z, v.w - hf.w));
    uint16_t* p = reinterpret_cast<uint16_t*>(base);
    *reinterpret_cast<uint2*>(p + idx) = hi;
    *reinterpret_cast<uint2*>(p + plane + idx) = lo;
  } else {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + idx) = v;
  }
}

// Four consecutive cache elements idx .. idx + 3 (idx a multiple of 4): bf16 or float32.
__device__ __forceinline__ void store_act4(void* base, long long idx, float4 v, int act_bf16) {
  if (act_bf16)
    *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(base) + idx) = bf16x4(v);
  else
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + idx) = v;
}

// The tile's epilogue. ys: tile values, element (t, c) at ys[t * ldys + c] for
// tile row t < kGemmBN and token c < mcount <= 32 (global token m0 + c); nt:
// the weight tile index; td: the launch's per-token data, or nullptr
// (computed here, per tile); sync(): a barrier over the nthr threads (a
// multiple of 32) that run it; es: this chunk's inputs staged by
// stage_epilogue_inputs (its 32-token chunk start), or nullptr to read them
// from global memory.
// Warp w takes tokens c = w, w + nthr / 32, ..; lane l takes tile rows
// 4l .. 4l + 3, so each warp writes a token's outputs with 8- or 16-byte
// stores and reduces over the tile's rows with a shuffle tree.
template <class Sync>
__device__ __forceinline__ void epilogue_tile(const GemmArgs& a, int nt, float* ys, int ldys, int m0, int mcount,
                                              int tid, int nthr, EpiSmem& sm, const TokData* td, Sync sync,
                                              const float* es = nullptr, bool tok_ready = false) {
  const Epi& e = a.epi;
  constexpr int BN = kGemmBN;
  const int lane = tid & 31, wid = tid >> 5, nw = nthr >> 5;
  const int t0 = lane * 4;                      // this lane's first tile row
  const int n0 = nt * BN + t0;                  // its first output row

  // ---- per-token data of the tile's tokens (already in sm when tok_ready)
  if (!tok_ready && tid < mcount) {
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
  auto tile4 = [&](int t, int c) {
    return make_float4(ys[t * ldys + c], ys[(t + 1) * ldys + c], ys[(t + 2) * ldys + c], ys[(t + 3) * ldys + c]);
  };

  if (e.kind == kEpiStore) {
    const bool vec = n0 + 3 < a.n_rows && (e.ldy & 3) == 0;
    for (int c = wid; c < mcount; c += nw) {
      const float4 v = tile4(t0, c);
      float* y = e.y + static_cast<long long>(m0 + c) * e.ldy + n0;
      if (vec) {
        *reinterpret_cast<float4*>(y) = v;
      } else {
        const float vv[4] = {v.x, v.y, v.z, v.w};
        for (int j = 0; j < 4; ++j)
          if (n0 + j < a.n_rows) y[j] = vv[j];
      }
    }
  } else if (e.kind == kEpiResid) {
    // h += value; x_out = h * next_gain; the tile's sum of h^2 per token
    const bool full = n0 + 3 < a.n_rows;
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f);
    if (e.next_gain) {
      if (es) {
        g = make_float4(sm.gain[t0], sm.gain[t0 + 1], sm.gain[t0 + 2], sm.gain[t0 + 3]);
      } else {
        float gg[4];
        for (int j = 0; j < 4; ++j) gg[j] = n0 + j < a.n_rows ? load_act(e.next_gain, n0 + j, e.gain_bf16) : 0.f;
        g = make_float4(gg[0], gg[1], gg[2], gg[3]);
      }
    }
    for (int c = wid; c < mcount; c += nw) {
      const long long m = m0 + c;
      float* hp = e.h + m * e.ldh + n0;
      float4 hv;
      if (es) {
        hv = *reinterpret_cast<const float4*>(es + c * BN + t0);
      } else if (full) {
        hv = *reinterpret_cast<const float4*>(hp);
      } else {
        float t4[4];
        for (int j = 0; j < 4; ++j) t4[j] = n0 + j < a.n_rows ? hp[j] : 0.f;
        hv = make_float4(t4[0], t4[1], t4[2], t4[3]);
      }
      const float4 v = tile4(t0, c);
      const float4 hn = make_float4(hv.x + v.x, hv.y + v.y, hv.z + v.z, hv.w + v.w);
      if (full) {
        *reinterpret_cast<float4*>(hp) = hn;
        if (e.next_gain)
          store_x4(e.x_out, e.x_out_plane, m * e.d_model + n0, make_float4(hn.x * g.x, hn.y * g.y, hn.z * g.z, hn.w * g.w),
                   e.x_pair);
      } else {
        const float hh[4] = {hn.x, hn.y, hn.z, hn.w}, gg[4] = {g.x, g.y, g.z, g.w};
        for (int j = 0; j < 4; ++j)
          if (n0 + j < a.n_rows) {
            hp[j] = hh[j];
            if (e.next_gain) store_x(e.x_out, e.x_out_plane, m * e.d_model + n0 + j, hh[j] * gg[j], e.x_pair);
          }
      }
      if (e.ss_out) {
        float q = 0.f;
        if (full) q = (hn.x * hn.x + hn.y * hn.y) + (hn.z * hn.z + hn.w * hn.w);
        else {
          const float hh[4] = {hn.x, hn.y, hn.z, hn.w};
          for (int j = 0; j < 4; ++j)
            if (n0 + j < a.n_rows) q += hh[j] * hh[j];
        }
        q = warp_sum(q);
        if (lane == 0) e.ss_out[m * e.n_ss + nt] = q;
      }
    }
  } else if (e.kind == kEpiSwiglu) {
    // tile rows t < BN/2 hold gate rows f0 + t, rows t >= BN/2 the up rows: lane l takes
    // features f0 + 2l and f0 + 2l + 1
    constexpr int HB = BN / 2;
    const int tf = 2 * lane, f = nt * HB + tf;
    if (f < e.ffn) {
      const bool two = f + 1 < e.ffn;
      for (int c = wid; c < mcount; c += nw) {
        const float rs = sm.rstd[c];
        const float g0 = ys[tf * ldys + c] * rs, g1 = ys[(tf + 1) * ldys + c] * rs;
        const float u0 = ys[(tf + HB) * ldys + c] * rs, u1 = ys[(tf + HB + 1) * ldys + c] * rs;
        const float o0 = silu(g0) * u0, o1 = silu(g1) * u1;
        const long long idx = static_cast<long long>(m0 + c) * e.ffn + f;
        if (two && e.x_pair && ((idx | e.act_plane) & 1) == 0) {
          const uint32_t hi = static_cast<uint32_t>(f32_to_bf16_bits(o0)) | static_cast<uint32_t>(f32_to_bf16_bits(o1)) << 16;
          const uint32_t lo = static_cast<uint32_t>(f32_to_bf16_bits(o0 - bf16_bits_to_f32(hi & 0xFFFFu))) |
                              static_cast<uint32_t>(f32_to_bf16_bits(o1 - bf16_bits_to_f32(hi >> 16))) << 16;
          uint16_t* p = reinterpret_cast<uint16_t*>(e.act);
          *reinterpret_cast<uint32_t*>(p + idx) = hi;
          *reinterpret_cast<uint32_t*>(p + e.act_plane + idx) = lo;
        } else {
          store_x(e.act, e.act_plane, idx, o0, e.x_pair);
          if (two) store_x(e.act, e.act_plane, idx + 1, o1, e.x_pair);
        }
      }
    }
  } else if (e.kind == kEpiQkv) {
    // the tile holds whole heads (head_dim 64 or 128): lane l's rows 4l .. 4l + 3 are
    // dims i .. i + 3 of one head; RoPE pairs them with dims i +- hd/2 (rows t0 +- hd/2)
    const int hd = e.head_dim, half = hd >> 1;
    const int nq = e.n_heads * hd;
    if (n0 < a.n_rows) {
      const int head = n0 / hd, i = n0 - head * hd;
      const bool rot = head < e.n_heads + e.n_kv_heads;  // q or k
      const int ii = i < half ? i : i - half;
      const int tp = i < half ? t0 + half : t0 - half;   // partner rows of the rotation
      const float sgn = i < half ? -1.f : 1.f;
      const bool is_q = n0 < nq;
      const int kvh = is_q ? 0 : head - e.n_heads - (rot ? 0 : e.n_kv_heads);
      for (int c = wid; c < mcount; c += nw) {
        const int pos = sm.pos[c];
        if (pos < 0) continue;  // flagged by the row preparation
        const float rs = sm.rstd[c];
        float4 v = tile4(t0, c);
        v = make_float4(v.x * rs, v.y * rs, v.z * rs, v.w * rs);
        if (rot) {
          float2 cs[4];
          if (es) {
            const float2* r2 = reinterpret_cast<const float2*>(es) + c * (BN / 2) + ii;
            for (int j = 0; j < 4; ++j) cs[j] = r2[j];
          } else {
            for (int j = 0; j < 4; ++j) cs[j] = __ldg(e.rope + static_cast<long long>(pos) * half + ii + j);
          }
          const float4 p = tile4(tp, c);
          v = make_float4(v.x * cs[0].x + sgn * (p.x * rs) * cs[0].y, v.y * cs[1].x + sgn * (p.y * rs) * cs[1].y,
                          v.z * cs[2].x + sgn * (p.z * rs) * cs[2].y, v.w * cs[3].x + sgn * (p.w * rs) * cs[3].y);
        }
        const long long m = m0 + c;
        if (is_q) {
          if (e.q_pair)
            store_x4(e.q_pair, e.q_plane, m * nq + n0,
                     make_float4(v.x * e.q_scale, v.y * e.q_scale, v.z * e.q_scale, v.w * e.q_scale), 1);
          else
            *reinterpret_cast<float4*>(e.q_out + m * nq + n0) = v;
        } else {
          const long long kvo = sm.kv[c];
          if (kvo < 0) continue;
          const long long off = (kvo + static_cast<long long>(kvh) * e.page_size) * hd + i;
          store_act4(rot ? e.k_cache : e.v_cache, off, v, e.kv_bf16);
        }
      }
    }
  } else if (e.kind == kEpiLogits) {
    // logits (when kept) and each token's (max, argmax) over the tile, lowest index on ties
    const bool vec = n0 + 3 < e.vocab && (e.vocab & 3) == 0;
    for (int c = wid; c < mcount; c += nw) {
      const float rs = sm.rstd[c];
      const float4 v4 = tile4(t0, c);
      const float vv[4] = {v4.x * rs, v4.y * rs, v4.z * rs, v4.w * rs};
      const long long m = m0 + c;
      if (e.logits) {
        float* lp = e.logits + m * e.vocab + n0;
        if (vec) {
          *reinterpret_cast<float4*>(lp) = make_float4(vv[0], vv[1], vv[2], vv[3]);
        } else {
          for (int j = 0; j < 4; ++j)
            if (n0 + j < e.vocab) lp[j] = vv[j];
        }
      }
      float best = -INFINITY;
      int bi = 0x7fffffff;
      for (int j = 0; j < 4; ++j)
        if (n0 + j < e.vocab) argmax_merge(best, bi, vv[j], n0 + j);
      warp_argmax(best, bi);
      if (lane == 0) e.argmax_part[m * a.n_tiles + nt] = make_float2(best, __int_as_float(bi));
    }
  }
}

}  // namespace sv
