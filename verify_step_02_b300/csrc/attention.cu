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
// This CUDA-core kernel serves float32 models (bf16 caches run the tensor-core
// attention). Work item = (request, kv head, chunk of 256 keys). Each item
// keeps a running softmax (max m, sum l, unnormalized output O) over its keys
// in tiles of 32, writes the partial, and the last item of a (request, kv
// head) to arrive merges the partials:
// out = sum_c O_c e^(m_c - M) / sum_c l_c e^(m_c - M), M = max_c m_c.
// No item waits on another.
#include "device_util.cuh"
#include "internal.h"

namespace sv {
namespace {

constexpr int KT = 32;  // keys per inner tile

// 16-byte asynchronous copy global -> shared (completes with cp.async.wait_group).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// float32 KV: the chunk's page ids once, then K/V tiles of KT keys by 16-byte
// asynchronous copies into a double buffer (the next tile loads while this one
// is used), rows padded to hd + 4 floats so a warp's 16-byte reads of
// consecutive keys fall in distinct banks.
template <typename KVT>
__global__ void __launch_bounds__(256) attn_fma_kernel(const AttnArgs a) {
  static_assert(sizeof(KVT) == 4, "the CUDA-core attention reads float32 caches");
  extern __shared__ __align__(16) float sm[];
  // The lengths, row ranges, page table and the keys cached before this step
  // were written two or more kernels back (every kernel triggers its dependents
  // only after its own wait): they are read before the dependency wait; the
  // queries and the block's own keys after it.
  const int hd = a.head_dim, nkv = a.n_kv_heads, group = a.n_heads / nkv;
  const int r = blockIdx.x / nkv, h = blockIdx.x - r * nkv, chunk = blockIdx.y;
  const int C = a.seq_len[r];
  const int row0 = a.req_row0[r], nrows = a.req_row0[r + 1] - row0;
  const int T = C + nrows;
  if (C < 0 || T > a.max_seq_len) {  // flagged by the row preparation; nothing is read or merged
    pdl_wait();
    pdl_trigger();
    return;
  }
  const int kbeg = chunk * a.chunk;
  if (kbeg >= T) {
    pdl_wait();
    pdl_trigger();
    return;
  }
  const int kend = min(T, kbeg + a.chunk);
  const int nchunks = (T + a.chunk - 1) / a.chunk;
  const int R = nrows * group;
  const int nq = a.n_heads * hd;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int LD = hd + 4;  // padded K/V row (floats)

  float* Qs = sm;                          // [R][hd]
  float* Os = Qs + a.max_rows * hd;        // [R][hd]
  float* Kb = Os + a.max_rows * hd;        // [2][KT][LD]
  float* Vb = Kb + 2 * KT * LD;            // [2][KT][LD]
  float* S = Vb + 2 * KT * LD;             // [R][KT]
  float* mrow = S + a.max_rows * KT;       // [R]
  float* lrow = mrow + a.max_rows;         // [R]
  float* crow = lrow + a.max_rows;         // [R]
  int* pages = reinterpret_cast<int*>(crow + a.max_rows);  // [chunk / page_size]

  const int* ptab = a.page_table + (long long)r * a.max_pages;
  const int npg = (kend - kbeg + a.page_size - 1) / a.page_size;
  for (int i = tid; i < npg; i += blockDim.x) {
    const int pidx = kbeg / a.page_size + i;
    int page = pidx < a.max_pages ? ptab[pidx] : -1;
    if (page < 0 || page >= a.n_pages) {
      atomicOr(a.status, pidx >= a.max_pages ? kStNoPage : kStBadPage);
      page = -1;
    }
    pages[i] = page;
  }
  __syncthreads();
  const float* kc = reinterpret_cast<const float*>(a.k_cache);
  const float* vc = reinterpret_cast<const float*>(a.v_cache);
  const int q4 = hd / 4;  // 16-byte pieces per row
  // tile t of the chunk into buffer b: keys past the chunk or on a bad page are zeros
  auto load_tile = [&](int t, int b) {
    float* kb = Kb + b * KT * LD;
    float* vb = Vb + b * KT * LD;
    for (int idx = tid; idx < KT * q4; idx += blockDim.x) {
      const int i = idx / q4, d = (idx - i * q4) * 4;
      const int key = kbeg + t * KT + i;
      const int page = key < kend ? pages[(key - kbeg) / a.page_size] : -1;
      if (page >= 0) {
        const long long off = (((long long)page * nkv + h) * a.page_size + (key % a.page_size)) * hd + d;
        cp_async16(kb + i * LD + d, kc + off);
        cp_async16(vb + i * LD + d, vc + off);
      } else {
        *reinterpret_cast<float4*>(kb + i * LD + d) = make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(vb + i * LD + d) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    cp_async_commit();
  };
  // the first tile goes out before the wait when all its keys are cached context
  const bool early = kbeg + KT <= C;
  if (early) load_tile(0, 0);
  pdl_wait();
  pdl_trigger();
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
  __syncthreads();
  const int ntiles = (kend - kbeg + KT - 1) / KT;
  if (!early) load_tile(0, 0);
  for (int t = 0; t < ntiles; ++t) {
    const int b = t & 1;
    if (t + 1 < ntiles) {
      load_tile(t + 1, b ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const float* kb = Kb + b * KT * LD;
    const float* vb = Vb + b * KT * LD;
    const int kt0 = kbeg + t * KT;
    for (int idx = tid; idx < R * KT; idx += blockDim.x) {
      const int rho = idx / KT, i = idx - rho * KT;
      const int key = kt0 + i, j = rho / group;
      float sc = -INFINITY;
      // (a token tree row sees, of the block, only its ancestors and itself)
      if (key < kend && key <= C + j && pages[(key - kbeg) / a.page_size] >= 0 &&
          (!a.row_anc || key < C || ((a.row_anc[row0 + j] >> (key - C)) & 1ull))) {
        const float4* q = reinterpret_cast<const float4*>(Qs + rho * hd);
        const float4* k = reinterpret_cast<const float4*>(kb + i * LD);
        float acc = 0.f;
        for (int d = 0; d < q4; ++d) {
          const float4 qq = q[d], kk = k[d];
          acc = fmaf(qq.x, kk.x, acc);
          acc = fmaf(qq.y, kk.y, acc);
          acc = fmaf(qq.z, kk.z, acc);
          acc = fmaf(qq.w, kk.w, acc);
        }
        sc = acc;
      }
      S[idx] = sc;
    }
    __syncthreads();
    for (int rho = warp; rho < R; rho += blockDim.x >> 5) {
      const float sv = S[rho * KT + lane];
      const float mold = mrow[rho];
      const float mnew = fmaxf(mold, warp_max(sv));
      const float p = sv == -INFINITY ? 0.f : expf(sv - mnew);
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
    for (int idx = tid; idx < R * q4; idx += blockDim.x) {
      const int rho = idx / q4, d = (idx - rho * q4) * 4;
      const float* p = S + rho * KT;
      float4 o = *reinterpret_cast<const float4*>(Os + rho * hd + d);
      const float c = crow[rho];
      o = make_float4(o.x * c, o.y * c, o.z * c, o.w * c);
#pragma unroll 8
      for (int i = 0; i < KT; ++i) {
        const float pi = p[i];
        const float4 vv = *reinterpret_cast<const float4*>(vb + i * LD + d);
        o.x = fmaf(pi, vv.x, o.x);
        o.y = fmaf(pi, vv.y, o.y);
        o.z = fmaf(pi, vv.z, o.z);
        o.w = fmaf(pi, vv.w, o.w);
      }
      *reinterpret_cast<float4*>(Os + rho * hd + d) = o;
    }
    __syncthreads();  // the buffer is reloaded two tiles on
  }

  if (nchunks == 1) {
    // the only chunk: its running softmax is the row's, normalized here
    for (int idx = tid; idx < R * hd; idx += blockDim.x) {
      const int rho = idx / hd, d = idx - rho * hd;
      const int j = rho / group, g = rho - j * group;
      const float L = lrow[rho];
      store_x(a.out, a.out_plane, (long long)(row0 + j) * nq + (h * group + g) * hd + d, L > 0.f ? Os[idx] / L : 0.f,
              a.x_pair);
    }
    return;
  }
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
  return sizeof(float) * ((size_t)2 * a.max_rows * hd + 4 * KT * (hd + 4) + (size_t)a.max_rows * KT +
                          3 * (size_t)a.max_rows) +
         sizeof(int) * (a.chunk / a.page_size + 1);
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
  if (kv_bf16) {  // bf16 caches run the tensor-core attention
    return cudaErrorInvalidValue;
  } else {
    cudaError_t e =
        cudaFuncSetAttribute(attn_fma_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_k(attn_fma_kernel<float>, grid, dim3(256), smem, s, a.pdl != 0, a);
  }
}

}  // namespace sv
