// Block-causal paged-KV attention of the verify block.
//
// Request r's block rows j = 0 .. L_r sit at positions C_r + j; row j attends
// to the C_r cached positions and to block rows 0 .. j, whose K/V the QKV
// epilogue has just written into their page slots (DSpark summary,
// "Architecture"; AngelSpec, "Engineering": prefix-causal plus diagonal
// masking, partial softmaxes merged through their log-sum-exp). All query
// heads of one KV head (GQA group) and all block rows of the request share
// each K/V tile read from HBM.
//
// Work item = (request, kv head, chunk of keys). Each item keeps a running
// softmax (max m, sum l, unnormalized output O) over its keys, writes the
// partial, and the last item of a (request, kv head) to arrive merges the
// partials: out = sum_c O_c e^(m_c - M) / sum_c l_c e^(m_c - M), M = max_c m_c.
// No item waits on another.
#include "device_util.cuh"
#include "internal.h"

namespace sv {
namespace {

constexpr int KT = 32;  // keys per inner tile

template <typename KVT>
__device__ __forceinline__ float kv_load(const KVT* p, long long i) {
  if constexpr (sizeof(KVT) == 2)
    return bf16_bits_to_f32(p[i]);
  else
    return p[i];
}

template <typename KVT>
__global__ void __launch_bounds__(256) attn_fma_kernel(const AttnArgs a) {
  extern __shared__ __align__(16) float sm[];
  pdl_trigger();
  pdl_wait();
  const int hd = a.head_dim, nkv = a.n_kv_heads, group = a.n_heads / nkv;
  const int r = blockIdx.x / nkv, h = blockIdx.x - r * nkv, chunk = blockIdx.y;
  const int C = a.seq_len[r];
  const int row0 = a.req_row0[r], nrows = a.req_row0[r + 1] - row0;
  const int T = C + nrows;
  if (C < 0 || T > a.max_seq_len) {  // flagged by the row preparation; nothing is read or merged
    return;
  }
  const int kbeg = chunk * a.chunk;
  if (kbeg >= T) return;
  const int kend = min(T, kbeg + a.chunk);
  const int nchunks = (T + a.chunk - 1) / a.chunk;
  const int R = nrows * group;
  const int nq = a.n_heads * hd;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  float* Qs = sm;                         // [R][hd]
  float* Os = Qs + a.max_rows * hd;       // [R][hd]
  float* Ks = Os + a.max_rows * hd;       // [KT][hd + 1]
  float* Vs = Ks + KT * (hd + 1);         // [KT][hd]
  float* S = Vs + KT * hd;                // [R][KT]
  float* mrow = S + a.max_rows * KT;      // [R]
  float* lrow = mrow + a.max_rows;        // [R]
  float* crow = lrow + a.max_rows;        // [R]

  const float scale = rsqrtf(static_cast<float>(hd));
  for (int idx = tid; idx < R * hd; idx += blockDim.x) {
    const int rho = idx / hd, d = idx - rho * hd;
    const int j = rho / group, g = rho - j * group;
    Qs[idx] = a.q[(long long)(row0 + j) * nq + (h * group + g) * hd + d] * scale;
    Os[idx] = 0.f;
  }
  for (int rho = tid; rho < R; rho += blockDim.x) {
    mrow[rho] = -INFINITY;
    lrow[rho] = 0.f;
  }
  const KVT* kc = reinterpret_cast<const KVT*>(a.k_cache);
  const KVT* vc = reinterpret_cast<const KVT*>(a.v_cache);
  const int* ptab = a.page_table + (long long)r * a.max_pages;

  for (int kt0 = kbeg; kt0 < kend; kt0 += KT) {
    __syncthreads();
    for (int idx = tid; idx < KT * hd; idx += blockDim.x) {
      const int i = idx / hd, d = idx - i * hd;
      const int key = kt0 + i;
      float kv = 0.f, vv = 0.f;
      if (key < kend) {
        const int pidx = key / a.page_size;
        const int page = pidx < a.max_pages ? ptab[pidx] : -1;
        if (page >= 0 && page < a.n_pages) {
          const long long off = (((long long)page * nkv + h) * a.page_size + (key - pidx * a.page_size)) * hd + d;
          kv = kv_load(kc, off);
          vv = kv_load(vc, off);
        } else if (d == 0) {
          atomicOr(a.status, pidx >= a.max_pages ? kStNoPage : kStBadPage);
        }
      }
      Ks[i * (hd + 1) + d] = kv;
      Vs[i * hd + d] = vv;
    }
    __syncthreads();
    for (int idx = tid; idx < R * KT; idx += blockDim.x) {
      const int rho = idx / KT, i = idx - rho * KT;
      const int key = kt0 + i, j = rho / group;
      float s = -INFINITY;
      if (key < kend && key <= C + j) {
        const float* q = Qs + rho * hd;
        const float* k = Ks + i * (hd + 1);
        float acc = 0.f;
        for (int d = 0; d < hd; ++d) acc = fmaf(q[d], k[d], acc);
        s = acc;
      }
      S[idx] = s;
    }
    __syncthreads();
    for (int rho = warp; rho < R; rho += blockDim.x >> 5) {
      const float s = S[rho * KT + lane];
      const float mold = mrow[rho];
      const float mnew = fmaxf(mold, warp_max(s));
      const float p = s == -INFINITY ? 0.f : expf(s - mnew);
      const float corr = mold == -INFINITY ? 0.f : expf(mold - mnew);
      const float psum = warp_sum(p);
      S[rho * KT + lane] = p;
      if (lane == 0) {
        mrow[rho] = mnew;
        lrow[rho] = lrow[rho] * corr + psum;
        crow[rho] = corr;
      }
    }
    __syncthreads();
    for (int idx = tid; idx < R * hd; idx += blockDim.x) {
      const int rho = idx / hd, d = idx - rho * hd;
      const float* p = S + rho * KT;
      float o = Os[idx] * crow[rho];
#pragma unroll 8
      for (int i = 0; i < KT; ++i) o = fmaf(p[i], Vs[i * hd + d], o);
      Os[idx] = o;
    }
  }
  __syncthreads();

  // partial of this chunk: per row [m, l, O[hd]]
  const int item = blockIdx.x;  // (r, h)
  const int stride = hd + 2;
  float* part = a.partials + ((long long)item * a.max_chunks + chunk) * a.max_rows * stride;
  for (int idx = tid; idx < R * hd; idx += blockDim.x) {
    const int rho = idx / hd, d = idx - rho * hd;
    __stcg(part + rho * stride + 2 + d, Os[idx]);
  }
  for (int rho = tid; rho < R; rho += blockDim.x) {
    __stcg(part + rho * stride, mrow[rho]);
    __stcg(part + rho * stride + 1, lrow[rho]);
  }
  __threadfence();
  __syncthreads();
  __shared__ unsigned s_last;
  if (tid == 0) s_last = atomicAdd(a.counters + item, 1u) == (unsigned)(nchunks - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float* base = a.partials + (long long)item * a.max_chunks * a.max_rows * stride;
  const long long cstride = (long long)a.max_rows * stride;
  for (int rho = warp; rho < R; rho += blockDim.x >> 5) {
    float M = -INFINITY;
    for (int c = 0; c < nchunks; ++c) M = fmaxf(M, __ldcg(base + c * cstride + rho * stride));
    float L = 0.f;
    for (int c = 0; c < nchunks; ++c) {
      const float mc = __ldcg(base + c * cstride + rho * stride);
      if (mc != -INFINITY) L += __ldcg(base + c * cstride + rho * stride + 1) * expf(mc - M);
    }
    const int j = rho / group, g = rho - j * group;
    const long long orow = (long long)(row0 + j) * nq + (h * group + g) * hd;
    for (int d = lane; d < hd; d += 32) {
      float o = 0.f;
      for (int c = 0; c < nchunks; ++c) {
        const float mc = __ldcg(base + c * cstride + rho * stride);
        if (mc != -INFINITY) o += __ldcg(base + c * cstride + rho * stride + 2 + d) * expf(mc - M);
      }
      store_x(a.out, a.out_plane, orow + d, o / L, a.x_pair);
    }
  }
  if (tid == 0) a.counters[item] = 0u;
}

size_t attn_smem_bytes(const AttnArgs& a) {
  const int hd = a.head_dim;
  return sizeof(float) * ((size_t)2 * a.max_rows * hd + KT * (hd + 1) + KT * hd + (size_t)a.max_rows * KT +
                          3 * (size_t)a.max_rows);
}

}  // namespace

void plan_attention(AttnArgs& a, int max_batch, int max_seq_len, int max_gamma) {
  (void)max_batch;
  a.chunk = 256;
  a.max_seq_len = max_seq_len;
  a.max_chunks = (max_seq_len + a.chunk - 1) / a.chunk;
  a.max_rows = (max_gamma + 1) * (a.n_heads / a.n_kv_heads);
}

size_t attention_partial_floats(const AttnArgs& a, int max_batch) {
  return (size_t)max_batch * a.n_kv_heads * a.max_chunks * a.max_rows * (a.head_dim + 2);
}

cudaError_t launch_attention(const AttnArgs& a, int B, int kv_bf16, cudaStream_t s) {
  const size_t smem = attn_smem_bytes(a);
  const dim3 grid(B * a.n_kv_heads, a.max_chunks);
  if (kv_bf16) {
    cudaError_t e = cudaFuncSetAttribute(attn_fma_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    return launch_k(attn_fma_kernel<uint16_t>, grid, dim3(256), smem, s, a.pdl != 0, a);
  } else {
    cudaError_t e =
        cudaFuncSetAttribute(attn_fma_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_k(attn_fma_kernel<float>, grid, dim3(256), smem, s, a.pdl != 0, a);
  }
}

}  // namespace sv
