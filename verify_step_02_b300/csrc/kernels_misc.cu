// Row preparation (embedding + the first RMSNorm statistics), acceptance +
// commit, RoPE table, W12 codec and Philox kernels of the verify step.
#include "device_util.cuh"
#include "internal.h"

namespace sv {
namespace {

constexpr int kNormThreads = 256;

// One CTA per block row: find the row's request and offset, gather the token's
// embedding into the residual stream h, and write the first projection's x
// tensor h * g (the first layer's attention-norm gain) with the row's sum of
// squares in ss[m][0] (the other tiles' slots zero): the QKV epilogue turns
// that into the RMSNorm scale.
//
// A token tree (p.parents): row j of request r is node j; its RoPE position
// is C + depth(j), its KV slot C + j, and row_anc[m] has bit i set for every
// node i on the path from the root to node j (the block keys it may see).
__global__ void __launch_bounds__(kNormThreads)
    prep_kernel(const PrepParams p, const int* tokens, const int* seq_len, int* row_req, int* row_pos, int* row_slot,
                unsigned long long* row_anc, int* req_row0_dev, const void* embed, const void* gain, float* h, void* u,
                long long u_plane, float* ss, int n_ss, int d, int vocab, int max_seq_len, int weights_bf16,
                int x_pair, unsigned* status) {
  __shared__ float red[32];
  pdl_wait();
  pdl_trigger();
  const int m = blockIdx.x;
  if (m == 0)
    for (int i = threadIdx.x; i <= p.B; i += blockDim.x) req_row0_dev[i] = p.req_row0[i];
  int lo = 0, hi = p.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.req_row0[mid] <= m) lo = mid; else hi = mid - 1;
  }
  const int r = lo, j = m - p.req_row0[r];
  int tok = tokens[(long long)r * p.gamma_stride + j];
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0) atomicOr(status, kStBadToken);
    tok = 0;
  }
  if (threadIdx.x == 0) {
    int depth = j;
    if (p.parents) {
      // walk to the root (parents strictly decrease: at most j steps); a bad
      // parent is flagged and the node treated as a chain row
      const int* par = p.parents + static_cast<long long>(r) * p.gamma_stride;
      unsigned long long anc = 1ull << j;
      depth = 0;
      for (int i = j; i > 0;) {
        const int q = par[i];
        if (q < 0 || q >= i) {
          atomicOr(status, kStBadTree);
          depth = j;
          anc = (2ull << j) - 1ull;
          break;
        }
        anc |= 1ull << q;
        i = q;
        ++depth;
      }
      row_anc[m] = anc;
    }
    // a row past the RoPE table / page budget gets position -1: the QKV
    // epilogue then writes nothing for it and the status word records it
    const int C = seq_len[r];
    int pos = C + depth, slot = C + j;  // (slot >= pos)
    if (C < 0 || slot >= max_seq_len) {
      atomicOr(status, kStBadPos);
      pos = slot = -1;
    }
    row_req[m] = r;
    row_pos[m] = pos;
    if (row_slot) row_slot[m] = slot;
  }
  float* hrow = h + (long long)m * d;
  float sq = 0.f;
  for (int k = threadIdx.x; k < d; k += blockDim.x) {
    const float x = load_act(embed, (long long)tok * d + k, weights_bf16);
    hrow[k] = x;
    sq = fmaf(x, x, sq);
    store_x(u, u_plane, (long long)m * d + k, x * load_act(gain, k, weights_bf16), x_pair);
  }
  const float tot = block_sum(sq, red);
  for (int i = threadIdx.x; i < n_ss; i += blockDim.x) ss[(long long)m * n_ss + i] = i == 0 ? tot : 0.f;
}

// ------------------------------------------------------------------ acceptance
constexpr int kAccThreads = 512;

struct SoftmaxRow {
  float mx;   // max of z / T
  float sum;  // sum of exp(z / T - mx)
};

__device__ SoftmaxRow softmax_stats(const float* z, int V, float invT, float* red) {
  float mx = -INFINITY;
  for (int v = threadIdx.x; v < V; v += blockDim.x) mx = fmaxf(mx, z[v] * invT);
  mx = block_max(mx, red);
  float s = 0.f;
  for (int v = threadIdx.x; v < V; v += blockDim.x) s += expf(z[v] * invT - mx);
  s = block_sum(s, red);
  return {mx, s};
}

// Inverse-CDF draw in token order over weights w(v) (v < V): the first v whose
// inclusive prefix sum exceeds u * total. Each thread owns a contiguous
// segment; segment sums are scanned across the block.
template <typename WFn>
__device__ int inverse_cdf_draw(WFn w, int V, float u, float* red, float* seg_pref, int* s_pick) {
  const int nt = blockDim.x, tid = threadIdx.x;
  const int seg = (V + nt - 1) / nt;
  const int v0 = min(V, tid * seg), v1 = min(V, v0 + seg);
  float mine = 0.f;
  for (int v = v0; v < v1; ++v) mine += w(v);
  seg_pref[tid] = mine;
  __syncthreads();
  if (tid == 0) {  // exclusive scan of the segment sums (nt <= 1024 values)
    float run = 0.f;
    for (int i = 0; i < nt; ++i) {
      const float t = seg_pref[i];
      seg_pref[i] = run;
      run += t;
    }
    red[0] = run;
    s_pick[0] = 0x7fffffff;
    s_pick[1] = -1;
  }
  __syncthreads();
  const float total = red[0];
  const float target = u * total;
  float run = seg_pref[tid];
  int last_pos = -1;
  for (int v = v0; v < v1; ++v) {
    const float wv = w(v);
    if (wv > 0.f) last_pos = v;
    run += wv;
    if (run > target) {
      atomicMin(s_pick, v);
      break;
    }
  }
  if (last_pos >= 0) atomicMax(s_pick + 1, last_pos);
  __syncthreads();
  const int pick = s_pick[0] != 0x7fffffff ? s_pick[0] : s_pick[1];
  __syncthreads();
  return pick < 0 ? 0 : pick;
}

__global__ void __launch_bounds__(kAccThreads) accept_kernel(const AcceptArgs a) {
  __shared__ float red[32];
  __shared__ float seg_pref[kAccThreads];
  __shared__ int s_pick[2];
  __shared__ int s_targ[kMaxGamma + 1];
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  pdl_trigger();
  const int row0 = a.req_row0[r], L = a.req_row0[r + 1] - row0 - 1;
  const int C = a.seq_len[r];
  const int* toks = a.tokens + (long long)r * a.gamma_stride;
  int k = 0, next = 0;
  if (a.temperature == 0.f) {
    // t_j = argmax over the LM head's per-tile partials, one warp per block row
    for (int j = warp; j <= L; j += blockDim.x >> 5) {
      const float2* part = a.argmax_part + (long long)(row0 + j) * a.n_tiles;
      float best = -INFINITY;
      int bi = 0x7fffffff;
      for (int t = lane; t < a.n_tiles; t += 32) {
        const float2 pv = part[t];
        argmax_merge(best, bi, pv.x, __float_as_int(pv.y));
      }
      warp_argmax(best, bi);
      if (lane == 0) s_targ[j] = bi;
    }
    __syncthreads();
    if (a.parents) {
      // token tree: node i is correct when its token is the target's greedy
      // token after its parent; the accepted path ends at the deepest node
      // whose every non-root ancestor and itself are correct (lowest index
      // among equally deep ones)
      if (tid == 0) {
        const int* par = a.parents + static_cast<long long>(r) * a.gamma_stride;
        unsigned long long okm = 1ull;  // bit i: node i accepted
        int depth[kMaxTreeNodes];
        depth[0] = 0;
        int end = 0;
        for (int i = 1; i <= L && i < kMaxTreeNodes; ++i) {
          const int q = par[i];
          const bool valid = q >= 0 && q < i;  // (a bad parent was flagged by the row preparation)
          depth[i] = valid ? depth[q] + 1 : 0;
          if (valid && ((okm >> q) & 1ull) && toks[i] == s_targ[q]) {
            okm |= 1ull << i;
            if (depth[i] > depth[end]) end = i;
          }
        }
        k = depth[end];
        next = s_targ[end];
        int* out = a.accepted_nodes + static_cast<long long>(r) * a.gamma_stride;
        for (int i = end, dd = k; dd >= 0; --dd) {
          out[dd] = i;
          i = dd > 0 ? par[i] : 0;
        }
      }
    } else {
      if (a.commit_all)
        k = L;  // prefill: the block is the prompt itself
      else
        while (k < L && toks[1 + k] == s_targ[k]) ++k;
      next = s_targ[k];
    }
  } else {
    const float invT = 1.0f / a.temperature;
    const long long req = a.request_ids ? a.request_ids[r] : r;
    bool rejected = false;
    for (int i = 1; i <= L; ++i) {
      const float* z = a.logits + (long long)(row0 + i - 1) * a.vocab;
      const SoftmaxRow st = softmax_stats(z, a.vocab, invT, red);
      int d = toks[i];
      if (d < 0 || d >= a.vocab) d = 0;
      const float* q = a.draft_probs + ((long long)r * a.max_gamma + (i - 1)) * a.vocab;
      const float pd = expf(z[d] * invT - st.mx) / st.sum;
      const float qd = q[d];
      const float u = philox_uniform(a.seed, req, (long long)C + i, 0u);
      if (u * qd < pd) {
        ++k;
        continue;
      }
      // residual max(0, p - q); if it is all zero, fall back to p
      const float invS = 1.0f / st.sum;
      float rs = 0.f;
      for (int v = tid; v < a.vocab; v += blockDim.x) rs += fmaxf(0.f, expf(z[v] * invT - st.mx) * invS - q[v]);
      rs = block_sum(rs, red);
      const float u2 = philox_uniform(a.seed, req, (long long)C + i, 1u);
      if (rs > 0.f) {
        next = inverse_cdf_draw([&](int v) { return fmaxf(0.f, expf(z[v] * invT - st.mx) * invS - q[v]); },
                                a.vocab, u2, red, seg_pref, s_pick);
      } else {
        next = inverse_cdf_draw([&](int v) { return expf(z[v] * invT - st.mx) * invS; }, a.vocab, u2, red,
                                seg_pref, s_pick);
      }
      rejected = true;
      break;
    }
    if (!rejected) {
      const float* z = a.logits + (long long)(row0 + L) * a.vocab;
      const SoftmaxRow st = softmax_stats(z, a.vocab, invT, red);
      const float invS = 1.0f / st.sum;
      const float u2 = philox_uniform(a.seed, req, (long long)C + L + 1, 1u);
      next = inverse_cdf_draw([&](int v) { return expf(z[v] * invT - st.mx) * invS; }, a.vocab, u2, red, seg_pref,
                              s_pick);
    }
  }
  if (tid == 0) {
    a.accepted_len[r] = k;
    a.next_token[r] = next;
    a.seq_len[r] = C + k + 1;  // commit the anchor and the accepted drafts
  }
}

// ------------------------------------------------------------------ tree commit
constexpr int kCompactThreads = 256;

// One CTA per (request, layer): for d = 1 .. k the accepted path's node p_d
// moves from slot C + p_d to slot C + d (p_d >= d, so in increasing d no
// source is overwritten before it is read: a slot C + e is written at step e
// and read, if at all, at the step d < e whose node is e). Each thread moves
// the same 16-byte pieces at every step, so its own program order keeps
// every read of a slot before the later write of it.
__global__ void __launch_bounds__(kCompactThreads) compact_kernel(const CompactArgs a) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, l = blockIdx.y;
  const int k = a.accepted_len[r];
  const int C = a.seq_len[r] - k - 1;
  if (k <= 0 || k >= kMaxTreeNodes || C < 0) return;
  const int* path = a.accepted_nodes + static_cast<long long>(r) * a.gamma_stride;
  const int* ptab = a.page_table + static_cast<long long>(r) * a.max_pages;
  const int pieces = a.row_bytes / 16;  // per kv head
  const int n = pieces * a.n_kv_heads;
  uint8_t* pools[2] = {static_cast<uint8_t*>(a.k[l]), static_cast<uint8_t*>(a.v[l])};
  // byte offset of (slot, kv head 0) in a pool, or -1 for a slot without a valid page
  auto slot_off = [&](int slot) -> long long {
    const int pidx = slot / a.page_size;
    const int page = pidx < a.max_pages ? ptab[pidx] : -1;
    if (page < 0 || page >= a.n_pages) return -1;
    return ((static_cast<long long>(page) * a.n_kv_heads) * a.page_size + (slot - pidx * a.page_size)) * a.row_bytes;
  };
  for (int dd = 1; dd <= k; ++dd) {
    const int node = path[dd];
    if (node == dd) continue;
    if (node < dd || node >= kMaxTreeNodes) return;
    const long long src = slot_off(C + node), dst = slot_off(C + dd);
    if (src < 0 || dst < 0) return;
    for (int i = threadIdx.x; i < 2 * n; i += kCompactThreads) {
      const int pool = i >= n, e = i - pool * n, h = e / pieces, piece = e - h * pieces;
      const long long ho = static_cast<long long>(h) * a.page_size * a.row_bytes + piece * 16;
      const uint4 v = *reinterpret_cast<const uint4*>(pools[pool] + src + ho);
      *reinterpret_cast<uint4*>(pools[pool] + dst + ho) = v;
    }
  }
}

// ------------------------------------------------------------------ RoPE table
__global__ void rope_table_kernel(float2* table, int max_seq_len, int half, int head_dim, double theta) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)max_seq_len * half) return;
  const int pos = static_cast<int>(idx / half), i = static_cast<int>(idx - (long long)pos * half);
  const double inv_freq = pow(theta, -2.0 * i / head_dim);
  double s, c;
  sincos(pos * inv_freq, &s, &c);
  table[idx] = make_float2(static_cast<float>(c), static_cast<float>(s));
}

// ------------------------------------------------------------------ W12
// stats[0]: min exponent over normal numbers, stats[1]: max exponent,
// stats[2]: elements that are not normal numbers. With base >= 0, stats[3]
// counts elements whose exponent exceeds base + 15.
__global__ void w12_scan_kernel(const uint16_t* b, long long n, int base, unsigned* stats) {
  unsigned emin = 255, emax = 0, bad = 0, wide = 0;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const unsigned e = (b[i] >> 7) & 0xFFu;
    if (e == 0 || e == 255) {
      ++bad;
    } else {
      emin = min(emin, e);
      emax = max(emax, e);
      if (base >= 0 && e > (unsigned)base + 15u) ++wide;
    }
  }
  for (int o = 16; o; o >>= 1) {
    emin = min(emin, __shfl_xor_sync(0xffffffffu, emin, o));
    emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, o));
    bad += __shfl_xor_sync(0xffffffffu, bad, o);
    wide += __shfl_xor_sync(0xffffffffu, wide, o);
  }
  if ((threadIdx.x & 31) == 0) {
    atomicMin(stats, emin);
    atomicMax(stats + 1, emax);
    atomicAdd(stats + 2, bad);
    atomicAdd(stats + 3, wide);
  }
}

__device__ __forceinline__ unsigned w12_code(uint16_t b, int base) {
  return (unsigned)(b >> 15) << 11 | (((b >> 7) & 0xFFu) - (unsigned)base) << 7 | (b & 0x7Fu);
}

// Element (within its group of 8) held by nibble slot s of a plane word: the
// even elements in slots 0-3, the odd ones in slots 4-7.
__device__ __forceinline__ int w12_slot_element(int s) { return s < 4 ? 2 * s : 2 * s - 7; }

// Planes are tiled: 64 rows x 128 elements per 4096-byte tile, tile (rt, kt)
// at byte (rt * kt_n + kt) * 4096, tile row r at r * 64 within it.
// One thread per plane byte b: tile b / 4096, tile row (b % 4096) / 64, group
// (b % 64) / 4, and nibble slots 2 (b % 4) and 2 (b % 4) + 1 of that group.
__global__ void w12_pack_kernel(const uint16_t* b, long long rows, long long cols, int kt_n, long long plane_bytes,
                                int base, uint8_t* planes) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= plane_bytes) return;
  const long long tile = idx >> 12;
  const int within = static_cast<int>(idx & 4095);
  const long long rt = tile / kt_n, kt = tile - rt * kt_n;
  const long long row = rt * 64 + (within >> 6);
  const int cb = within & 63;
  const long long g0 = kt * 128 + (cb >> 2) * 8;
  const int s0 = 2 * (cb & 3);
  const long long k0 = g0 + w12_slot_element(s0), k1 = g0 + w12_slot_element(s0 + 1);
  const unsigned c0 = row < rows && k0 < cols ? w12_code(b[row * cols + k0], base) : 0u;
  const unsigned c1 = row < rows && k1 < cols ? w12_code(b[row * cols + k1], base) : 0u;
#pragma unroll
  for (int p = 0; p < 3; ++p)
    planes[p * plane_bytes + idx] = static_cast<uint8_t>(((c0 >> (4 * p)) & 0xFu) | ((c1 >> (4 * p)) & 0xFu) << 4);
}

__global__ void w12_unpack_kernel(const uint8_t* planes, int base, long long rows, long long cols, int kt_n,
                                  long long plane_bytes, uint16_t* out) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * cols) return;
  const long long row = idx / cols, k = idx - row * cols;
  const int e = static_cast<int>(k & 7), slot = (e & 1) ? 4 + (e >> 1) : (e >> 1);
  const long long byte = (((row >> 6) * kt_n + (k >> 7)) << 12) + (row & 63) * 64 + ((k & 127) >> 3) * 4 + (slot >> 1);
  const int sh = (slot & 1) * 4;
  const unsigned c = ((planes[byte] >> sh) & 0xFu) | ((planes[plane_bytes + byte] >> sh) & 0xFu) << 4 |
                     ((planes[2 * plane_bytes + byte] >> sh) & 0xFu) << 8;
  out[idx] = static_cast<uint16_t>(((c & 0x7FFu) + ((unsigned)base << 7)) | ((c & 0x800u) << 4));
}

__global__ void philox_kernel(unsigned long long seed, long long req, long long pos0, int stream_id, int n,
                              float* out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = philox_uniform(seed, req, pos0 + i, static_cast<unsigned>(stream_id));
}

}  // namespace

cudaError_t launch_prep(const PrepParams& p, const int* tokens, const int* seq_len, int* row_req, int* row_pos,
                        int* row_slot, unsigned long long* row_anc, int* req_row0_dev, const void* embed,
                        const void* gain, float* h, void* u, long long u_plane, float* ss, int n_ss, int d, int vocab,
                        int max_seq_len, int weights_bf16, int x_pair, unsigned* status, cudaStream_t s) {
  return launch_k(prep_kernel, dim3(p.M), dim3(kNormThreads), 0, s, p.pdl != 0, p, tokens, seq_len, row_req, row_pos,
                  row_slot, row_anc, req_row0_dev, embed, gain, h, u, u_plane, ss, n_ss, d, vocab, max_seq_len,
                  weights_bf16, x_pair, status);
}

cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t s) {
  return launch_k(accept_kernel, dim3(a.B), dim3(kAccThreads), 0, s, a.pdl != 0, a);
}

cudaError_t launch_compact(const CompactArgs& a, cudaStream_t s) {
  return launch_k(compact_kernel, dim3(a.B, a.n), dim3(kCompactThreads), 0, s, a.pdl != 0, a);
}

cudaError_t launch_rope_table(float2* table, int max_seq_len, int head_dim, float theta, cudaStream_t s) {
  const int half = head_dim / 2;
  const long long n = (long long)max_seq_len * half;
  rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(table, max_seq_len, half, head_dim, (double)theta);
  return cudaGetLastError();
}

cudaError_t launch_w12_scan(const uint16_t* bf16, long long n, int base, unsigned* stats, cudaStream_t s) {
  long long blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  w12_scan_kernel<<<(unsigned)blocks, 256, 0, s>>>(bf16, n, base, stats);
  return cudaGetLastError();
}

cudaError_t launch_w12_pack(const uint16_t* bf16, long long rows, long long cols, int base, uint8_t* planes,
                            cudaStream_t s) {
  const int kt_n = static_cast<int>((cols + 127) / 128);
  const long long n = w12_plane_bytes(rows, cols);
  w12_pack_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(bf16, rows, cols, kt_n, n, base, planes);
  return cudaGetLastError();
}

cudaError_t launch_w12_unpack(const uint8_t* planes, int base, long long rows, long long cols, uint16_t* out,
                              cudaStream_t s) {
  const int kt_n = static_cast<int>((cols + 127) / 128);
  const long long n = rows * cols;
  w12_unpack_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(planes, base, rows, cols, kt_n,
                                                                 w12_plane_bytes(rows, cols), out);
  return cudaGetLastError();
}

cudaError_t launch_philox(unsigned long long seed, long long req, long long pos0, int stream_id, int n, float* out,
                          cudaStream_t s) {
  philox_kernel<<<(n + 255) / 256, 256, 0, s>>>(seed, req, pos0, stream_id, n, out);
  return cudaGetLastError();
}

}  // namespace sv
