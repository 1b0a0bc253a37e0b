// Host side of the tensor-core skinny GEMM: tensor maps, the work plan and the
// dispatch to the kernel instantiation of the plan's token tile (the kernel
// itself is in gemm_tc.cuh, instantiated by gemm_tc_nt*.cu).
#include <cudaTypedefs.h>

#include <mutex>
#include <vector>

#include "gemm_tc_plan.h"
#include "internal.h"

namespace sv {
namespace {

using namespace tcg;

template <bool PAIR, bool CL>
cudaError_t launch_pair(const GemmArgs& a, const CUtensorMap& w, const CUtensorMap& x, cudaStream_t s) {
  if (a.wdtype == SV_W12 || CL) {
    const bool w12 = a.wdtype == SV_W12;
    switch (a.tc_nt) {
      case 32: return w12 ? gemm_tc_launch<32, PAIR, true, CL>(a, w, x, s) : gemm_tc_launch<32, PAIR, false, CL>(a, w, x, s);
      case 64: return w12 ? gemm_tc_launch<64, PAIR, true, CL>(a, w, x, s) : gemm_tc_launch<64, PAIR, false, CL>(a, w, x, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (a.tc_nt) {
    case 32: return gemm_tc_launch<32, PAIR, false, false>(a, w, x, s);
    case 64: return gemm_tc_launch<64, PAIR, false, false>(a, w, x, s);
    case 96: return gemm_tc_launch<96, PAIR, false, false>(a, w, x, s);
    case 128: return gemm_tc_launch<128, PAIR, false, false>(a, w, x, s);
    case 160: return gemm_tc_launch<160, PAIR, false, false>(a, w, x, s);
    case 192: return gemm_tc_launch<192, PAIR, false, false>(a, w, x, s);
    case 224: return gemm_tc_launch<224, PAIR, false, false>(a, w, x, s);
    case 256: return gemm_tc_launch<256, PAIR, false, false>(a, w, x, s);
    default: return cudaErrorInvalidValue;
  }
}

// Resident clusters of cs CTAs for the cluster-split instantiation of a plan,
// looked up once per (device, configuration).
int max_clusters(int nt, bool pair, bool w12, int cs, int stages) {
  struct Entry {
    int dev, nt, pair, w12, cs, stages, n;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : cache)
    if (e.dev == dev && e.nt == nt && e.pair == pair && e.w12 == w12 && e.cs == cs && e.stages == stages) return e.n;
  int n = 0;
#define SV_MC(NT, P, W) n = gemm_tc_max_clusters<NT, P, W, true>(cs, stages)
  if (nt == 32) {
    if (pair) { if (w12) SV_MC(32, true, true); else SV_MC(32, true, false); }
    else { if (w12) SV_MC(32, false, true); else SV_MC(32, false, false); }
  } else if (nt == 64) {
    if (pair) { if (w12) SV_MC(64, true, true); else SV_MC(64, true, false); }
    else { if (w12) SV_MC(64, false, true); else SV_MC(64, false, false); }
  }
#undef SV_MC
  cache.push_back({dev, nt, pair, w12, cs, stages, n});
  return n;
}

// ------------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

cudaError_t get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

cudaError_t encode_bf16_map(CUtensorMap* m, const void* p, long long rows, int K, int box_rows) {
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  if ((reinterpret_cast<uintptr_t>(p) & 15) || (K % 8) || rows < 1) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t tc_encode_weight_map(CUtensorMap* m, const void* w, long long rows, int K) {
  return encode_bf16_map(m, w, rows, K, kGemmBN / 2);
}

cudaError_t tc_encode_x_map(CUtensorMap* m, const void* x, long long rows, int K) {
  return encode_bf16_map(m, x, rows, K, 32);
}

cudaError_t tc_encode_kv_map(CUtensorMap* m, const void* pool, int n_pages, int n_kv, int head_dim) {
  return encode_bf16_map(m, pool, static_cast<long long>(n_pages) * n_kv * 16, head_dim, 16);
}

cudaError_t tc_encode_q_map(CUtensorMap* m, const void* q, int m_max, int n_heads, int head_dim, int group,
                            int rows) {
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  if ((reinterpret_cast<uintptr_t>(q) & 15) || (head_dim % 64) || group < 1 || group > 256 || rows < 1 ||
      rows > 256)
    return cudaErrorInvalidValue;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(n_heads),
                              static_cast<cuuint64_t>(2) * m_max};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                                 static_cast<cuuint64_t>(n_heads) * head_dim * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(rows)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

void plan_gemm_tc(GemmArgs& a, int M, int n_units, int K, int pair, int sm_count) {
  a.M = M;
  a.K = K;
  a.pair = pair;
  a.n_tiles = pair == kPairSwiglu ? (n_units + kGemmBN / 2 - 1) / (kGemmBN / 2) : (n_units + kGemmBN - 1) / kGemmBN;
  a.m_tiles = (M + 255) / 256;
  const int per = (M + a.m_tiles - 1) / a.m_tiles;
  a.tc_nt = (per + 31) / 32 * 32;
  const bool w12 = a.wdtype == SV_W12, pair2 = a.x_kind == kXPair;
  a.tc_ks = tc_ks_for(a.tc_nt, pair2, w12);
  a.kb = (K + a.tc_ks - 1) / a.tc_ks;
  const long long U = static_cast<long long>(a.n_tiles) * a.m_tiles * a.kb;
  a.grid_p = static_cast<int>(U < sm_count ? U : sm_count);
  a.tc_stages = w12 && a.tc_nt > kW12MaxNT ? 0 : tc_stages_for(a.tc_nt, pair2, a.tc_ks, w12);
  a.k_splits = 1;
  a.k_chunk = K;
  a.cl_size = 0;
  a.cl_tiles = 0;
  // Small token tiles: the cluster split, when some (CTAs per cluster 2 .. 8, one tile
  // per cluster) fits the device in one wave on at least 60% of the SMs with per-CTA
  // work within 1.5x of stream-K's: the fewest units per CTA wins, then the larger
  // cluster (a smaller slice per rank, so more pipeline stages). An SM streams about
  // 50 GB/s with this pipeline depth, so 96 CTAs still draw 4.7 TB/s, and the cluster's
  // hand-off through distributed shared memory ends about 5 us sooner than stream-K's
  // through global memory (8B-class q|k|v, 48 tiles: 96 CTAs in 16.8 us, stream-K
  // over 148 CTAs 19.7 us).
  if (a.tc_nt > kClusterMaxNT || a.m_tiles != 1 || a.tc_stages < 2) return;
  const long long ntt = static_cast<long long>(a.n_tiles) * a.m_tiles;
  const long long sk_work = (U + a.grid_p - 1) / a.grid_p;
  long long best_work = 0, best_ctas = 0;
  int best_cs = 0, best_tc = 0, best_st = 0;
  // power-of-two cluster sizes only: they tile the GPCs, so a whole wave of
  // clusters still fits while the previous kernel's CTAs leave their SMs
  for (int cs = 2; cs <= kClusterMaxSize && cs <= a.kb; cs *= 2) {
    const int st_cl = tc_stages_for(a.tc_nt, pair2, a.tc_ks, w12, cs);
    if (st_cl < 2) continue;
    int mc = -1;
    // one tile per cluster: with several, every tile's hand-off waits for the slowest
    // rank and the epilogue falls behind the MMAs (measured slower than stream-K)
    for (int tc = 1; tc <= 1; ++tc) {
      const long long ncl = (ntt + tc - 1) / tc;
      if (ncl * cs > sm_count || ncl * cs * 20 < 12LL * sm_count) continue;
      if (mc < 0) mc = max_clusters(a.tc_nt, pair2, w12, cs, st_cl);
      if (ncl > mc) continue;
      const long long work = static_cast<long long>(tc) * ((a.kb + cs - 1) / cs), ctas = ncl * cs;
      if (best_cs == 0 || work < best_work || (work == best_work && cs > best_cs)) {
        best_work = work;
        best_ctas = ctas;
        best_cs = cs;
        best_tc = tc;
        best_st = st_cl;
      }
    }
  }
  if (best_cs == 0 || best_work * 2 > sk_work * 3) return;
  a.cl_size = best_cs;
  a.cl_tiles = best_tc;
  a.grid_p = static_cast<int>(best_ctas);
  a.tc_stages = best_st;
}

size_t gemm_tc_partial_floats(const GemmArgs& a) {
  return static_cast<size_t>(a.grid_p) * 2 * kGemmBN * a.tc_nt;
}

// per tile: partials stored, then participants done (stream-K reduction)
size_t gemm_tc_counter_count(const GemmArgs& a) { return 2 * static_cast<size_t>(a.n_tiles) * a.m_tiles; }

bool gemm_tc_supported(int wdtype, int pair, int ffn) {
  // W12 row halves are whole 64-row plane tiles: gate|up needs ffn % 64 == 0
  return wdtype == SV_BF16 || (wdtype == SV_W12 && (pair != kPairSwiglu || ffn % 64 == 0));
}

cudaError_t launch_gemm_tc(const GemmArgs& a, const CUtensorMap& w, const CUtensorMap& x, cudaStream_t s) {
  if (!gemm_tc_supported(a.wdtype, a.pair, a.ffn) || a.tc_stages < 2) return cudaErrorInvalidValue;
  if (a.cl_size > 0)
    return a.x_kind == kXPair ? launch_pair<true, true>(a, w, x, s) : launch_pair<false, true>(a, w, x, s);
  return a.x_kind == kXPair ? launch_pair<true, false>(a, w, x, s) : launch_pair<false, false>(a, w, x, s);
}

}  // namespace sv
