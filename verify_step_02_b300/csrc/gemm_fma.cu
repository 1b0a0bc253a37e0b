// CUDA-core skinny GEMM: y[m][n] = x[m] . W[n] for float32, bf16 or W12 weights.
//
// This path serves float32 models (no TF32: float32 products keep the
// float32 model's accuracy) and bf16/W12 blocks too small for the tensor
// path. One CTA computes a 128-row x 32-token tile over one K range; the W
// tile is converted to float32 once into shared memory (W12 rebuilt from its
// three nibble planes to bf16 on the way, SpecPilot digest, "Reasons") and
// every thread then runs an 8 x 2 register-blocked FMA loop. Activations are
// read as float32 (a hi/lo pair is summed on load). K is split
// across CTAs (at most 8 splits) until the grid covers the GPU. The splits of
// a tile form one thread-block cluster: each rank sums a slice of the tile's
// rows over every split's partial (distributed shared memory, in split order,
// so results do not depend on timing) into rank 0, which runs the
// projection's epilogue.
#include "epilogue.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace sv {
namespace {

constexpr int BN = kGemmBN, BM = kFmaBM, KC = kFmaKC;
constexpr int WS_LD = BN + 4, XS_LD = BM + 4, YS_LD = BM + 1;

// W row of tile row t, or -1 when the tile row is past the matrix.
__device__ __forceinline__ int weight_row(const GemmArgs& a, int nt, int t) {
  if (a.pair == kPairSwiglu) {
    const int f = nt * (BN / 2) + (t & (BN / 2 - 1));
    if (f >= a.ffn) return -1;
    return t < BN / 2 ? f : a.ffn + f;
  }
  const int r = nt * BN + t;
  return r < a.n_rows ? r : -1;
}

// 16 consecutive weights of row `row` starting at k (k % 16 == 0), as float32.
template <int WT>
__device__ __forceinline__ void load_w16(const GemmArgs& a, int row, int k, float* v) {
  if (WT == SV_F32) {
    const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.w) + (long long)row * a.K + k);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 f = __ldg(p + j);
      v[4 * j] = f.x;
      v[4 * j + 1] = f.y;
      v[4 * j + 2] = f.z;
      v[4 * j + 3] = f.w;
    }
  } else if (WT == SV_BF16) {
    const uint4* p =
        reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.w) + (long long)row * a.K + k);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint4 u = __ldg(p + j);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[8 * j + 2 * q] = __uint_as_float(w[q] << 16);
        v[8 * j + 2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
      }
    }
  } else {  // W12: two 8-element groups of tile (row / 64, k / 128), tile row row % 64
    const uint8_t* base = reinterpret_cast<const uint8_t*>(a.w) +
                          ((((long long)(row >> 6) * a.w12_kt + (k >> 7)) << 12) + (row & 63) * 64 + ((k & 127) >> 1));
    const uint2 p0 = __ldg(reinterpret_cast<const uint2*>(base));
    const uint2 p1 = __ldg(reinterpret_cast<const uint2*>(base + a.w12_plane));
    const uint2 p2 = __ldg(reinterpret_cast<const uint2*>(base + 2 * a.w12_plane));
    // grouped W12: the row block's base, then the tile's escapes patched in
    const uint32_t ebase = static_cast<uint32_t>(a.w12_bases ? __ldg(a.w12_bases + (row >> 6)) : a.w12_base) << 7;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t b0 = h ? p0.y : p0.x, b1 = h ? p1.y : p1.x, b2 = h ? p2.y : p2.x;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int sh = 4 * ((e & 1) ? 4 + (e >> 1) : (e >> 1));  // nibble slot of element e
        const uint32_t c = ((b2 >> sh) & 0xFu) << 8 | ((b1 >> sh) & 0xFu) << 4 | ((b0 >> sh) & 0xFu);
        const uint32_t bits = ((c & 0x7FFu) + ebase) | ((c & 0x800u) << 4);
        v[8 * h + e] = __uint_as_float(bits << 16);
      }
    }
    if (a.w12_esc_off) {
      const long long tile = (long long)(row >> 6) * a.w12_kt + (k >> 7);
      const int o1 = __ldg(a.w12_esc_off + tile + 1), c0 = k & 127;
      for (int i = __ldg(a.w12_esc_off + tile); i < o1; ++i) {
        const uint32_t ent = __ldg(a.w12_esc + i);
        const int r = ent >> 23 & 63, c = (ent >> 16 & 127) - c0;
        if (r == (row & 63)) {
#pragma unroll
          for (int j = 0; j < 16; ++j)  // (a static index keeps v in registers)
            if (c == j) v[j] = __uint_as_float((ent & 0xFFFFu) << 16);
        }
      }
    }
  }
}

template <int WT, bool CL>
__global__ void __launch_bounds__(256) gemm_fma_kernel(const GemmArgs a) {
  __shared__ __align__(16) float Ws[KC][WS_LD];
  __shared__ __align__(16) float Xs[KC][XS_LD];
  __shared__ __align__(16) float Ys[BN * YS_LD];
  const int ks = blockIdx.x, nt = blockIdx.y, mt = blockIdx.z;
  const int tid = threadIdx.x;
  const int tr = (tid & 15) * 8, tc = (tid >> 4) * 2;
  const int m0 = mt * BM;
  const int kbeg = ks * a.k_chunk, kend = min(a.K, kbeg + a.k_chunk);
  float acc[8][2];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = 0.f;

  const int lrow = tid & (BN - 1), lkk = (tid >> 7) * 16;  // W loader: one row, 16 k
  const int wrow = weight_row(a, nt, lrow);
  const int xtok = tid >> 3, xkk = (tid & 7) * 4;          // X loader: one token, 4 k
  const int xm = m0 + xtok;
  // this thread's 16 weights of the K step at k0, one step ahead of the products
  float wv16[16];
  auto fetch_w = [&](int k0) {
    const int k = k0 + lkk;
    if (wrow >= 0 && k < kend) {
      load_w16<WT>(a, wrow, k, wv16);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) wv16[i] = 0.f;
    }
  };
  // the weights are never written by the step: the first step's are requested
  // before waiting for the kernels that produce x
  fetch_w(kbeg);
  pdl_wait();
  pdl_trigger();

  for (int k0 = kbeg; k0 < kend; k0 += KC) {
#pragma unroll
    for (int i = 0; i < 16; ++i) Ws[lkk + i][lrow] = wv16[i];
    {
      const int k = k0 + xkk;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float xv = 0.f;
        if (xm < a.M && k + i < kend) {
          xv = load_x(a.x, a.x_plane, (long long)xm * a.K + k + i, a.x_kind);
        }
        Xs[xkk + i][xtok] = xv;
      }
    }
    __syncthreads();
    if (k0 + KC < kend) fetch_w(k0 + KC);
#pragma unroll 4
    for (int k = 0; k < KC; ++k) {
      const float4 w0 = *reinterpret_cast<const float4*>(&Ws[k][tr]);
      const float4 w1 = *reinterpret_cast<const float4*>(&Ws[k][tr + 4]);
      const float2 x = *reinterpret_cast<const float2*>(&Xs[k][tc]);
      const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        acc[i][0] = fmaf(wv[i], x.x, acc[i][0]);
        acc[i][1] = fmaf(wv[i], x.y, acc[i][1]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    Ys[(tr + i) * YS_LD + tc] = acc[i][0];
    Ys[(tr + i) * YS_LD + tc + 1] = acc[i][1];
  }
  __syncthreads();
  const int mcount = min(BM, a.M - m0);
  if (CL) {
    // the tile's splits are one cluster, rank = split: rank r sums rows
    // [r rpr, (r + 1) rpr) of the live columns over every split, in split order
    const int cs = a.k_splits, rank = static_cast<int>(tc::cluster_ctarank());
    tc::cluster_sync();  // every split's partial is in its shared memory
    const int rpr = (BN + cs - 1) / cs, r0 = rank * rpr, r1 = min(BN, r0 + rpr);
    const int n = (r1 - r0) * mcount;
    const uint32_t ys0 = tc::smem_u32(Ys);
    for (int idx = tid; idx < n; idx += blockDim.x) {
      const int tt = idx / mcount, c = idx - tt * mcount;
      const uint32_t off = ys0 + 4u * static_cast<uint32_t>((r0 + tt) * YS_LD + c);
      float v[8];
#pragma unroll
      for (int p = 0; p < 8; ++p) v[p] = p < cs ? tc::ld_dsmem_f32(tc::mapa_shared(off, static_cast<uint32_t>(p))) : 0.f;
      float sum = 0.f;
#pragma unroll
      for (int p = 0; p < 8; ++p) sum += v[p];
      tc::st_dsmem_f32(tc::mapa_shared(off, 0u), sum);
    }
    tc::cluster_sync();  // rank 0 holds the sums; no rank leaves while its partial may be read
    if (rank != 0) return;
  }
  __shared__ EpiSmem esm;
  epilogue_tile(a, nt, Ys, YS_LD, m0, mcount, threadIdx.x, blockDim.x, esm, nullptr, [] { __syncthreads(); });
}

template <int WT>
cudaError_t launch_wt(const GemmArgs& a, dim3 grid, cudaStream_t s) {
  if (a.k_splits > 1) {
    if (a.cl_size != a.k_splits || a.cl_size > kFmaMaxCluster) return cudaErrorInvalidValue;
    return launch_k_cluster(gemm_fma_kernel<WT, true>, grid, dim3(256), 0, s, a.pdl != 0, a.cl_size, a);
  }
  return launch_k(gemm_fma_kernel<WT, false>, grid, dim3(256), 0, s, a.pdl != 0, a);
}

}  // namespace

void plan_gemm(GemmArgs& a, int M, int n_units, int K, int pair, int sm_count) {
  a.M = M;
  a.K = K;
  a.pair = pair;
  a.n_tiles = pair == kPairSwiglu ? (n_units + BN / 2 - 1) / (BN / 2) : (n_units + BN - 1) / BN;
  a.m_tiles = (M + BM - 1) / BM;
  const int base = a.n_tiles * a.m_tiles;
  const int target = 4 * sm_count;
  const int ksteps = (K + KC - 1) / KC;
  int splits = (target + base - 1) / base;
  if (splits > ksteps) splits = ksteps;
  if (splits > kFmaMaxCluster) splits = kFmaMaxCluster;
  if (splits < 1) splits = 1;
  const int steps_per = (ksteps + splits - 1) / splits;
  a.k_chunk = steps_per * KC;
  a.k_splits = (K + a.k_chunk - 1) / a.k_chunk;
  a.cl_size = a.k_splits > 1 ? a.k_splits : 0;
}

// (the splits meet in distributed shared memory: no partial tiles in global memory)
size_t gemm_partial_floats(const GemmArgs& a) {
  (void)a;
  return 0;
}

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s) {
  if (a.n_tiles > 65535 || a.m_tiles > 65535) return cudaErrorInvalidValue;  // grid y / z limits
  const dim3 grid(a.k_splits, a.n_tiles, a.m_tiles);  // a cluster spans one tile's splits (x)
  switch (a.wdtype) {
    case SV_F32: return launch_wt<SV_F32>(a, grid, s);
    case SV_BF16: return launch_wt<SV_BF16>(a, grid, s);
    case SV_W12: return launch_wt<SV_W12>(a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sv
