// Weight-streaming skinny GEMM on the 5th-generation tensor cores (tcgen05).
//
// y[m][n] = x[m] . W[n] for bf16 weights W [rows][K] and bf16 activations, one
// plane or a hi/lo pair (x = hi + lo: both planes are multiplied into the same
// float32 accumulator). The verify block has M = sum(L_r + 1) rows, a few to a
// few hundred, so W is the big operand: it is the MMA's A operand (128 weight
// rows per tile, the MMA's M), and the block's tokens are its N (32 .. 256
// columns). Every weight byte is read from HBM exactly once per launch.
//
// Work split ("stream-K"): the launch has P <= #SM CTAs and U = tiles x K
// blocks of 64 units of work; CTA c takes units [c U / P, (c+1) U / P), so
// every SM streams the same number of weight bytes. A tile whose K range is
// shared by several CTAs is finished by the last of them to arrive, which sums
// the partial tiles in CTA order (a fixed order: results do not depend on
// timing) and runs the projection's epilogue. No CTA waits on another.
//
// Roles inside a CTA (256 threads):
//   warp 0     one thread issues TMA loads of the weight tile (two 64-row
//              boxes) and the x tile (32-row boxes per plane) into an S-stage
//              shared-memory ring;
//   warp 1     allocates the TMEM accumulators (two buffers of NT columns) and
//              one thread issues tcgen05.mma (M 128, N NT, K 16) per stage;
//   warps 4-7  read finished accumulators out of TMEM (warp w reads lanes
//              32 (w % 4) ..), and write partial tiles or run the epilogue.
// Every wait is bounded; a wait that runs out sets the status word's timeout
// bit and the whole CTA winds down (waits for its copies and MMAs in flight,
// frees TMEM, returns).
#include <cudaTypedefs.h>

#include <cstdlib>
#include <mutex>

#include "epilogue.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace sv {
namespace {

using namespace tc;

constexpr int kTcThreads = 384;  // warp 0 TMA, warp 1 MMA, warps 4-11 epilogue (two warpgroups)
constexpr int kEpiThreads = 256;
constexpr int kYsLd = 33;                       // Ys row stride (floats)
constexpr int kABytes = kGemmBN * 128;          // weight tile of one stage: 128 rows x 64 bf16
constexpr uint64_t kWaitNs = 2000000000ull;     // 2 s
constexpr uint64_t kDrainNs = 200000000ull;     // 0.2 s
constexpr int kSmemBudget = 225 * 1024;

// One pipeline stage covers ks K-elements (ks / 64 swizzled sub-tiles of 64).
__host__ __device__ constexpr int stage_bytes(int nt, bool pair, int ks) {
  return (ks / 64) * (kABytes + nt * 128 * (pair ? 2 : 1));
}

__host__ __device__ constexpr uint32_t tmem_cols(int nt) {
  return 2 * nt <= 32 ? 32u : 2 * nt <= 64 ? 64u : 2 * nt <= 128 ? 128u : 2 * nt <= 256 ? 256u : 512u;
}

// First CTA whose unit range contains unit x: the largest c with floor(c U / P) <= x.
__device__ __forceinline__ int cta_of_unit(long long x, long long U, int P) {
  return static_cast<int>(((x + 1) * P + U - 1) / U - 1);
}

template <int NT, bool PAIR, int KS>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmx,
                   const GemmArgs a) {
  constexpr int BX = NT * 128;              // bytes of one x plane per 64-wide sub-tile
  constexpr int SUB = kABytes + BX * (PAIR ? 2 : 1);  // one 64-wide sub-tile: weights, then x
  constexpr int NSUB = KS / 64;
  constexpr int STAGE = stage_bytes(NT, PAIR, KS);
  constexpr uint32_t TCOLS = tmem_cols(NT);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.tc_stages;
  float* Ys = reinterpret_cast<float*>(smem + static_cast<size_t>(S) * STAGE);
  EpiSmem* esm = reinterpret_cast<EpiSmem*>(Ys + kGemmBN * kYsLd);
  TokData* tok = reinterpret_cast<TokData*>(esm + 1);
  uint64_t* full = reinterpret_cast<uint64_t*>(tok + 1);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = a.grid_p, c = blockIdx.x;
  const long long U = static_cast<long long>(a.n_tiles) * a.m_tiles * a.kb;
  const long long u0 = c * U / P, u1 = (c + 1) * U / P;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(acc_full + i, 1);
      mbar_init(acc_empty + i, 128);  // the TMEM-reading warpgroup
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmw);
    prefetch_tmap(&tmx);
  }
  if (warp == 1) tmem_alloc(tmem_slot, TCOLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pw = policy_evict_first(), px = policy_evict_last();
      // weight boxes, all sub-tiles back to back: each row's KS elements are
      // requested together (contiguous bytes in HBM)
      auto load_w = [&](long long u, uint8_t* st, uint64_t* bar) {
        const long long t = u / a.kb;
        const int kb = static_cast<int>(u - t * a.kb);
        const int nt = static_cast<int>(t / a.m_tiles);
        const int r0 = a.pair == kPairSwiglu ? nt * (kGemmBN / 2) : nt * kGemmBN;
        const int r1 = a.pair == kPairSwiglu ? a.ffn + nt * (kGemmBN / 2) : r0 + kGemmBN / 2;
#pragma unroll
        for (int q = 0; q < NSUB; ++q) {
          tma_load_2d(st + q * SUB, &tmw, kb * KS + q * 64, r0, bar, pw);
          tma_load_2d(st + q * SUB + kABytes / 2, &tmw, kb * KS + q * 64, r1, bar, pw);
        }
      };
      auto load_x = [&](long long u, uint8_t* st, uint64_t* bar) {
        const long long t = u / a.kb;
        const int kb = static_cast<int>(u - t * a.kb);
        const int mt = static_cast<int>(t - (t / a.m_tiles) * a.m_tiles);
#pragma unroll
        for (int q = 0; q < NSUB; ++q) {
          uint8_t* sb = st + q * SUB + kABytes;
          const int k = kb * KS + q * 64;
#pragma unroll
          for (int j = 0; j < NT / 32; ++j) {
            tma_load_2d(sb + j * 4096, &tmx, k, mt * NT + j * 32, bar, px);
            if (PAIR) tma_load_2d(sb + BX + j * 4096, &tmx, k, a.x_lo_row + mt * NT + j * 32, bar, px);
          }
        }
      };
      // The weights of the first stages do not depend on earlier kernels:
      // request them before waiting for those kernels, then the activations.
      const long long npre = u1 - u0 < S ? u1 - u0 : S;
      for (long long i = 0; i < npre; ++i) {
        uint8_t* st = smem + static_cast<size_t>(i) * STAGE;
        mbar_arrive_expect_tx(full + i, STAGE);
        load_w(u0 + i, st, full + i);
      }
      pdl_wait();
      for (long long i = 0; i < npre; ++i) load_x(u0 + i, smem + static_cast<size_t>(i) * STAGE, full + i);
      int stage = static_cast<int>(npre % S);
      uint32_t phase = npre == S ? 1u : 0u;
      long long issued = npre;
      for (long long u = u0 + npre; u < u1; ++u) {
        if (!mbar_wait(empty + stage, phase ^ 1u, abort_flag, kWaitNs)) break;
        uint8_t* st = smem + static_cast<size_t>(stage) * STAGE;
        mbar_arrive_expect_tx(full + stage, STAGE);
        load_w(u, st, full + stage);
        load_x(u, st, full + stage);
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (*abort_flag) {
        // let the copies still in flight land before the CTA's shared memory goes away
        volatile int never = 0;
        const long long n = issued < S ? issued : S;
        for (long long i = 1; i <= n; ++i) {
          const long long q = issued - i;  // issue number
          mbar_wait(full + (q % S), static_cast<uint32_t>((q / S) & 1), &never, kDrainNs);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kGemmBN, NT);
      int stage = 0, seg = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (long long u = u0; u < u1 && ok;) {
        const long long t = u / a.kb;
        const long long uend = u1 < (t + 1) * a.kb ? u1 : (t + 1) * a.kb;
        const int b = seg & 1;
        if (!mbar_wait(acc_empty + b, ((seg >> 1) & 1) ^ 1u, abort_flag, kWaitNs)) break;
        tc_fence_after();
        const uint32_t d = tmem + b * NT;
        for (long long v = u; v < uend; ++v) {
          if (!mbar_wait(full + stage, phase, abort_flag, kWaitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + static_cast<size_t>(stage) * STAGE);
#pragma unroll
          for (int q = 0; q < NSUB; ++q) {
            const uint32_t sa = st + q * SUB, sb = sa + kABytes;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = smem_desc_sw128(sa + k * 32);
              mma_bf16(d, ad, smem_desc_sw128(sb + k * 32), idesc, (v > u || q > 0 || k > 0) ? 1u : 0u);
              if (PAIR) mma_bf16(d, ad, smem_desc_sw128(sb + BX + k * 32), idesc, 1u);
            }
          }
          mma_commit(empty + stage);  // frees the stage once these MMAs have read it
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(acc_full + b);
        ++seg;
        u = uend;
      }
      // every MMA issued above has completed once `drain` flips
      mma_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, &never, kDrainNs);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    // Warpgroup A (warps 4-7) reads the accumulators out of TMEM (warp w reads
    // lanes 32 (w % 4) ..) and writes partial tiles; both warpgroups share
    // the split reduction (16 columns each) and the tile epilogue.
    pdl_wait();  // reads what earlier kernels wrote (h, norm statistics, row maps)
    const int et2 = threadIdx.x - 128;          // 0 .. 255
    const bool grpA = et2 < 128;
    const int et = et2 & 127;                   // tile row
    // per-token data of the whole launch, while the weights stream in
    const TokData* td = a.M <= kTokMax ? tok : nullptr;
    if (td)
      for (int m = et2; m < a.M; m += kEpiThreads) token_data(a.epi, m, tok->rstd[m], tok->pos[m], tok->kv[m]);
    auto sync = [] { named_bar(1, kEpiThreads); };
    sync();
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int slot0_tile = static_cast<int>(u0 / a.kb);
    int seg = 0;
    for (long long u = u0; u < u1;) {
      const long long t = u / a.kb;
      const long long uend = u1 < (t + 1) * a.kb ? u1 : (t + 1) * a.kb;
      const int nt = static_cast<int>(t / a.m_tiles), mt = static_cast<int>(t - (long long)nt * a.m_tiles);
      const int b = seg & 1;
      // one thread waits and broadcasts, so all threads agree on the outcome
      if (et2 == 0) *s_flag = mbar_wait(acc_full + b, (seg >> 1) & 1, abort_flag, kWaitNs) ? 1 : 0;
      sync();
      const bool ok = *s_flag != 0;
      sync();
      if (!ok) break;
      tc_fence_after();
      const int cf = cta_of_unit(t * a.kb, U, P), cl = cta_of_unit((t + 1) * a.kb - 1, U, P);
      const bool alone = cf == cl;
      const int m_base = mt * NT;
      const int mtot = a.M - m_base < NT ? a.M - m_base : NT;
      const int slot = static_cast<int>(t) == slot0_tile ? 0 : 1;
      // partial tiles are column-major ([token][tile row]) so that a warp's
      // stores and the reducer's loads are 128-byte coalesced
      float* mine = a.partials + (static_cast<size_t>(c) * 2 + slot) * kGemmBN * NT + et;
      for (int ch = 0; ch * 32 < mtot; ++ch) {
        float v[32];
        if (grpA) tmem_ld32(tmem + lane_base + b * NT + ch * 32, v);
        if (alone) {
          if (grpA) {
#pragma unroll
            for (int i = 0; i < 32; ++i) Ys[et * kYsLd + i] = v[i];
          }
          sync();
          epilogue_tile(a, nt, Ys, kYsLd, m_base + ch * 32, mtot - ch * 32 < 32 ? mtot - ch * 32 : 32, et2,
                        kEpiThreads, *esm, td, sync);
          sync();
        } else if (grpA) {
#pragma unroll
          for (int i = 0; i < 32; ++i) __stcg(mine + (ch * 32 + i) * kGemmBN, v[i]);
        }
      }
      if (grpA) {
        tc_fence_before();
        mbar_arrive(acc_empty + b);
      }
      if (!alone) {
        epilogue_prefetch(a, nt, m_base, mtot < 32 ? mtot : 32, et, td);
        __threadfence();
        sync();
        if (et2 == 0) *s_flag = atomicAdd(a.counters + t, 1u) == static_cast<unsigned>(cl - cf) ? 1 : 0;
        sync();
        const bool last = *s_flag != 0;
        sync();
        if (last) {
          __threadfence();
          // the contributors' slots, in CTA order (a fixed summation order): a
          // tile is the first tile (slot 0) of every contributor after cf, and of
          // cf when cf's range starts at the tile's first unit
          const int ncon = cl - cf + 1;
          const int sl_first = static_cast<long long>(cf) * U / P == t * a.kb ? 0 : 1;
          const int col0 = grpA ? 0 : 16;  // each warpgroup sums 16 of the chunk's 32 columns
          for (int ch = 0; ch * 32 < mtot; ++ch) {
            float s[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) s[i] = 0.f;
#pragma unroll 2
            for (int j = 0; j < ncon; ++j) {
              const int cc = cf + j;
              const int sl = j == 0 ? sl_first : 0;
              const float* src = a.partials + (static_cast<size_t>(cc) * 2 + sl) * kGemmBN * NT + et;
              float v[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] = __ldcg(src + (ch * 32 + col0 + i) * kGemmBN);
#pragma unroll
              for (int i = 0; i < 16; ++i) s[i] += v[i];
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) Ys[et * kYsLd + col0 + i] = s[i];
            sync();
            epilogue_tile(a, nt, Ys, kYsLd, m_base + ch * 32, mtot - ch * 32 < 32 ? mtot - ch * 32 : 32, et2,
                          kEpiThreads, *esm, td, sync);
            sync();
          }
          if (et2 == 0) a.counters[t] = 0u;
        }
      }
      ++seg;
      u = uend;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TCOLS);
  }
  if (threadIdx.x == 0 && *abort_flag && a.epi.status) atomicOr(a.epi.status, kStTimeout);
}

size_t tc_smem_bytes(int nt, bool pair, int ks, int stages) {
  return 1024 + static_cast<size_t>(stages) * stage_bytes(nt, pair, ks) + sizeof(float) * kGemmBN * kYsLd +
         sizeof(EpiSmem) + sizeof(TokData) + sizeof(uint64_t) * (2 * stages + 5) + 16;
}

int tc_stages_for(int nt, bool pair, int ks) {
  const size_t fixed = tc_smem_bytes(nt, pair, ks, 0) + 16 * sizeof(uint64_t);
  int s = static_cast<int>((kSmemBudget - fixed) / stage_bytes(nt, pair, ks));
  if (s > 8) s = 8;
  return s;
}

// K elements per pipeline stage for a token tile of nt columns: the widest of
// 256 / 128 / 64 that still leaves three stages (two at the widest token tiles).
int tc_ks_for(int nt, bool pair) {
  if (const char* env = getenv("SV_GEMM_KS")) {
    const int v = atoi(env);
    if ((v == 64 || v == 128 || v == 256) && tc_stages_for(nt, pair, v) >= 2) return v;
  }
  for (int ks = 256; ks >= 64; ks /= 2)
    if (tc_stages_for(nt, pair, ks) >= 3) return ks;
  return 64;
}

template <int NT, bool PAIR, int KS>
cudaError_t launch_ks(const GemmArgs& a, const CUtensorMap& w, const CUtensorMap& x, cudaStream_t s) {
  const size_t smem = tc_smem_bytes(NT, PAIR, KS, a.tc_stages);
  static bool attr_set[64] = {};  // per device: allow the largest configuration this kernel may use
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<NT, PAIR, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBudget + 2048);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  return launch_k(gemm_tc_kernel<NT, PAIR, KS>, dim3(a.grid_p), dim3(kTcThreads), smem, s, a.pdl != 0, w, x, a);
}

template <int NT, bool PAIR>
cudaError_t launch_nt(const GemmArgs& a, const CUtensorMap& w, const CUtensorMap& x, cudaStream_t s) {
  switch (a.tc_ks) {
    case 64: return launch_ks<NT, PAIR, 64>(a, w, x, s);
    case 128: return launch_ks<NT, PAIR, 128>(a, w, x, s);
    case 256: return launch_ks<NT, PAIR, 256>(a, w, x, s);
    default: return cudaErrorInvalidValue;
  }
}

template <bool PAIR>
cudaError_t launch_pair(const GemmArgs& a, const CUtensorMap& w, const CUtensorMap& x, cudaStream_t s) {
  switch (a.tc_nt) {
    case 32: return launch_nt<32, PAIR>(a, w, x, s);
    case 64: return launch_nt<64, PAIR>(a, w, x, s);
    case 96: return launch_nt<96, PAIR>(a, w, x, s);
    case 128: return launch_nt<128, PAIR>(a, w, x, s);
    case 160: return launch_nt<160, PAIR>(a, w, x, s);
    case 192: return launch_nt<192, PAIR>(a, w, x, s);
    case 224: return launch_nt<224, PAIR>(a, w, x, s);
    case 256: return launch_nt<256, PAIR>(a, w, x, s);
    default: return cudaErrorInvalidValue;
  }
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
  a.tc_ks = tc_ks_for(a.tc_nt, a.x_kind == kXPair);
  a.kb = (K + a.tc_ks - 1) / a.tc_ks;
  const long long U = static_cast<long long>(a.n_tiles) * a.m_tiles * a.kb;
  a.grid_p = static_cast<int>(U < sm_count ? U : sm_count);
  a.tc_stages = tc_stages_for(a.tc_nt, a.x_kind == kXPair, a.tc_ks);
  a.k_splits = 1;
  a.k_chunk = K;
}

size_t gemm_tc_partial_floats(const GemmArgs& a) {
  return static_cast<size_t>(a.grid_p) * 2 * kGemmBN * a.tc_nt;
}

size_t gemm_tc_counter_count(const GemmArgs& a) { return static_cast<size_t>(a.n_tiles) * a.m_tiles; }

cudaError_t launch_gemm_tc(const GemmArgs& a, const CUtensorMap& w, const CUtensorMap& x, cudaStream_t s) {
  if (a.wdtype != SV_BF16 || a.tc_stages < 2) return cudaErrorInvalidValue;
  return a.x_kind == kXPair ? launch_pair<true>(a, w, x, s) : launch_pair<false>(a, w, x, s);
}

}  // namespace sv
