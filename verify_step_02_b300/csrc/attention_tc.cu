// Block-causal paged-KV attention of the verify block on the tcgen05 tensor
// cores, for bf16 KV caches.
//
// Request r's block rows j = 0 .. L_r sit at positions C_r + j; row j attends
// to the cached positions and to block rows 0 .. j (DSpark summary,
// "Architecture"; AngelSpec, "Engineering": prefix-causal plus diagonal
// masking, partial softmaxes merged through their log-sum-exp). All query
// heads of one KV head (the GQA group) and all block rows of the request are
// the MMA's 128 rows (rho = j * group + g), so every K/V byte is read once.
//
// One CTA = (request, kv head, 256-key chunk):
//   warp 4   TMA: the chunk's K and V pages (16 keys x 64 dims per box, two
//            boxes per page for hd 128) straight from the page pool;
//            and the Q tile: the QKV epilogue left q / sqrt(hd) as a hi/lo
//            bf16 pair (q = hi + lo to ~16 bits), which a 3D box (64 dims x
//            group heads x block rows) lands as rows rho = j * group + g;
//   warp 5   S = Q K^T (M 128, N 256, K hd; hi and lo into one accumulator);
//   warps 0-3 read their row of S from TMEM, mask it (key <= C_r + j), take
//            the chunk's max m and p = exp(s - m), sum l, and write P as a
//            hi/lo bf16 pair over the (now consumed) Q and K buffers;
//   warp 5   O = P V (M 128, N hd, K 256; V is the N-major operand);
//   warps 0-3 write the partial (m, l, O) of their row.
// A second kernel merges a row's chunk partials:
//   out = sum_c O_c e^(m_c - M) / sum_c l_c e^(m_c - M), M = max_c m_c,
// and writes the attention output as the next projection's x tensor.
#include <cudaTypedefs.h>

#include "device_util.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace sv {
namespace {

using namespace tc;

constexpr int kChunk = 256;
constexpr int kRowWarps = 16;                         // softmax warps: 4 lane groups x 4 column groups
constexpr int kRowThreads = kRowWarps * 32;
constexpr int kAttnThreads = kRowThreads + 64;        // + TMA warp + MMA warp
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 200000000ull;
constexpr uint32_t kTile = 16384;  // 128 rows x 128 bytes

// Shared-memory descriptor of an N-major (MN-major) bf16 operand in the
// 128-byte swizzled layout: 64 N-elements per 128-byte row, K rows 128 bytes
// apart, 8-row groups `sbo` bytes apart, 64-element N blocks `lbo` bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Two float32 values -> their bf16 pair (round to nearest even), low half first.
__device__ __forceinline__ uint32_t cvt_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 8 float32 values -> 16-byte hi chunk and lo chunk (x = hi + lo).
__device__ __forceinline__ void split8(const float* x, uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = cvt_bf16x2(x[2 * i], x[2 * i + 1]);
    l[i] = cvt_bf16x2(x[2 * i] - __uint_as_float(h[i] << 16), x[2 * i + 1] - __uint_as_float(h[i] & 0xFFFF0000u));
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Byte offset of 16-byte chunk `ch` (0..7) of row `row` in a 128-byte swizzled tile.
__device__ __forceinline__ uint32_t sw128(int row, int ch) {
  return static_cast<uint32_t>(row) * 128u + static_cast<uint32_t>((ch ^ (row & 7)) * 16);
}

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const AttnArgs a) {
  constexpr int NH = HD / 64;  // 64-dim halves of a head
  // shared memory: [P region 128 KB: Q (2 NH tiles), K (NH x 2 tiles)] [V: NH x 2 tiles] [barriers]
  constexpr uint32_t Q_OFF = 0, K_OFF = 2 * NH * kTile, V_OFF = 8 * kTile;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + V_OFF + NH * 2 * kTile);
  uint64_t* kv_full = bars;  // Q, K and V landed
  uint64_t* s_full = bars + 2;
  uint64_t* p_ready = bars + 3;
  uint64_t* o_full = bars + 4;
  uint64_t* drain = bars + 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 6);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_flag = abort_flag + 1;
  volatile uint32_t* valid_mask = reinterpret_cast<volatile uint32_t*>(abort_flag + 2);

  pdl_trigger();
  pdl_wait();
  const int nkv = a.n_kv_heads, group = a.n_heads / nkv;
  const int r = blockIdx.x / nkv, h = blockIdx.x - r * nkv, chunk = blockIdx.y;
  const int C = a.seq_len[r];
  const int row0 = a.req_row0[r], nrows = a.req_row0[r + 1] - row0;
  const int T = C + nrows;
  if (C < 0 || T > a.max_seq_len) return;  // flagged by the row preparation
  const int k0 = chunk * kChunk;
  if (k0 >= T) return;
  const int R = nrows * group;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;

  if (tid == 0) {
    mbar_init(kv_full, 1);
    mbar_init(s_full, 1);
    mbar_init(p_ready, kRowThreads);
    mbar_init(o_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kRowWarps + 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 256;

  if (warp == kRowWarps) {
    // ------------------------------------------------------------ TMA producer
    // lane p < 16 looks up page p of the chunk (all lookups in flight at once)
    const int key = k0 + 16 * lane;
    int page = -1;
    if (lane < 16 && key < T) {
      const int pidx = key >> 4;
      page = pidx < a.max_pages ? a.page_table[static_cast<long long>(r) * a.max_pages + pidx] : -1;
      if (page < 0 || page >= a.n_pages) {
        atomicOr(a.status, kStBadPage);
        page = -1;
      }
    }
    const uint32_t mask = __ballot_sync(0xffffffffu, page >= 0);
    if (lane == 0) {
      prefetch_tmap(&tmq);
      prefetch_tmap(&tmk);
      prefetch_tmap(&tmv);
      *valid_mask = mask;
      const uint32_t qbox = 128u * group * (a.max_rows / group);
      mbar_arrive_expect_tx(kv_full, static_cast<uint32_t>(__popc(mask)) * NH * 2 * 2048u + 2 * NH * qbox);
      const uint64_t polq = policy_evict_last();
#pragma unroll
      for (int pl = 0; pl < 2; ++pl)
#pragma unroll
        for (int hh = 0; hh < NH; ++hh)
          tma_load_3d(smem + Q_OFF + (pl * NH + hh) * kTile, &tmq, hh * 64, h * group, pl * a.q_lo_row + row0,
                      kv_full, polq);
    }
    __syncwarp();
    if (page >= 0) {  // the transaction count was raised above, before any of these copies
      const uint64_t pol = policy_evict_first();
      const int row = (page * nkv + h) * 16;
#pragma unroll
      for (int hh = 0; hh < NH; ++hh) {
        tma_load_2d(smem + K_OFF + hh * 2 * kTile + lane * 2048, &tmk, hh * 64, row, kv_full, pol);
        tma_load_2d(smem + V_OFF + hh * 2 * kTile + lane * 2048, &tmv, hh * 64, row, kv_full, pol);
      }
    }
    if (lane == 0) {
      volatile int never = 0;  // the copies land before the CTA can leave
      mbar_wait(kv_full, 0, &never, kWaitNs);
    }
    __syncwarp();
  } else if (warp == kRowWarps + 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(kv_full, 0, abort_flag, kWaitNs);
      if (ok) {
        tc_fence_after();
        const uint32_t q = smem_u32(smem + Q_OFF), k = smem_u32(smem + K_OFF);
        constexpr uint32_t idesc_s = idesc_bf16_f32(128, kChunk);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const int kh = ks >> 2;
          const uint32_t off = (ks & 3) * 32;
          const uint64_t b = smem_desc_sw128(k + kh * 2 * kTile + off);
          mma_bf16(tS, smem_desc_sw128(q + kh * kTile + off), b, idesc_s, ks > 0 ? 1u : 0u);
          mma_bf16(tS, smem_desc_sw128(q + (NH + kh) * kTile + off), b, idesc_s, 1u);
        }
        mma_commit(s_full);
        ok = mbar_wait(p_ready, 0, abort_flag, kWaitNs);
      }
      if (ok) {
        tc_fence_after();
        const uint32_t pb = smem_u32(smem), v = smem_u32(smem + V_OFF);
        constexpr uint32_t idesc_o = idesc_bf16_f32(128, HD) | (1u << 16);  // B (V) is N-major
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks) {
          const int kb = ks >> 2;
          const uint32_t off = (ks & 3) * 32;
          const uint64_t b = smem_desc_sw128_mn(v + ks * 2048, 2 * kTile, 1024);
          mma_bf16(tO, smem_desc_sw128(pb + kb * kTile + off), b, idesc_o, ks > 0 ? 1u : 0u);
          mma_bf16(tO, smem_desc_sw128(pb + (4 + kb) * kTile + off), b, idesc_o, 1u);
        }
        mma_commit(o_full);
      }
      mma_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, &never, kDrainNs);
    }
  } else {
    // ------------------------------------------------------------ rows: softmax, output
    // warp w reads TMEM lanes 32 (w % 4) .. (its rows) and columns of group
    // cg = w / 4: keys cg*64 .. cg*64+63 of S, dims cg*32 .. cg*32+31 of O
    const int lg = warp & 3, cg = warp >> 2;
    const int rho = lg * 32 + lane;
    const bool live = rho < R;
    const int j = live ? rho / group : 0;
    float* red = reinterpret_cast<float*>(bars + 8);  // [2][4][128]: partial max, partial sum
    auto sync = [] { named_bar(1, kRowThreads); };
    // (waiting on kv_full too makes the producer's page mask visible here)
    if (tid == 0)
      *s_flag = mbar_wait(kv_full, 0, abort_flag, kWaitNs) && mbar_wait(s_full, 0, abort_flag, kWaitNs) ? 1 : 0;
    sync();
    const bool ok = *s_flag != 0;
    sync();
    float m = -INFINITY, l = 0.f;
    if (ok) {
      tc_fence_after();
      const uint32_t lane_base = static_cast<uint32_t>(lg * 32) << 16;
      const uint32_t vmask = *valid_mask;
      const int lim = live ? C + j : -1;  // last key this row may see
      float v[64];
      tmem_ld32(tS + lane_base + cg * 64, v);
      tmem_ld32(tS + lane_base + cg * 64 + 32, v + 32);
      float mp = -INFINITY;
      if (k0 + cg * 64 + 63 <= C && ((vmask >> (cg * 4)) & 0xFu) == 0xFu) {
        // every key of this column group is cached context on loaded pages: no mask
#pragma unroll
        for (int i = 0; i < 64; ++i) mp = fmaxf(mp, v[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const int kk = cg * 64 + i;  // key within the chunk
          const bool vis = k0 + kk <= lim && ((vmask >> (kk >> 4)) & 1u);
          v[i] = vis ? v[i] : -INFINITY;
          mp = fmaxf(mp, v[i]);
        }
      }
      red[cg * 128 + rho] = mp;
      sync();
      m = fmaxf(fmaxf(red[rho], red[128 + rho]), fmaxf(red[256 + rho], red[384 + rho]));
      float lp = 0.f;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        v[i] = v[i] == -INFINITY ? 0.f : __expf(v[i] - m);
        lp += v[i];
      }
      red[512 + cg * 128 + rho] = lp;
      // keys cg*64 .. +63 are key block cg of P: 8 16-byte chunks per plane
#pragma unroll
      for (int c16 = 0; c16 < 8; ++c16) {
        uint4 hi, lo;
        split8(v + 8 * c16, hi, lo);
        *reinterpret_cast<uint4*>(smem + cg * kTile + sw128(rho, c16)) = hi;
        *reinterpret_cast<uint4*>(smem + (4 + cg) * kTile + sw128(rho, c16)) = lo;
      }
      // V rows of keys past the request's end or on unloaded pages hold stale
      // bytes (possibly not finite); zero them so P = 0 there contributes 0
      if (k0 + kChunk > T || vmask != 0xFFFFu)
      for (int idx = tid; idx < kChunk * NH * 8; idx += kRowThreads) {
        const int key_i = idx / (NH * 8), rem = idx - key_i * (NH * 8);
        const int hh = rem >> 3, c16 = rem & 7;
        if (k0 + key_i >= T || !((vmask >> (key_i >> 4)) & 1u))
          *reinterpret_cast<uint4*>(smem + V_OFF + hh * 2 * kTile + key_i * 128 + c16 * 16) = make_uint4(0, 0, 0, 0);
      }
    }
    tc_fence_before();
    fence_proxy_async_smem();
    mbar_arrive(p_ready);

    if (tid == 0) *s_flag = ok && mbar_wait(o_full, 0, abort_flag, kWaitNs) ? 1 : 0;
    sync();
    const bool ok2 = *s_flag != 0;
    if (ok2) {
      tc_fence_after();
      const uint32_t lane_base = static_cast<uint32_t>(lg * 32) << 16;
      const long long slot = (static_cast<long long>(blockIdx.x) * a.max_chunks + chunk) * a.max_rows + rho;
      if (cg < HD / 32) {  // O dims cg*32 .. +31 (hd 64: column groups 0 and 1)
        float4* po = reinterpret_cast<float4*>(a.partials + slot * HD + cg * 32);
        float o[32];
        tmem_ld32(tO + lane_base + cg * 32, o);
        if (live) {
#pragma unroll
          for (int i = 0; i < 8; ++i) __stcg(po + i, make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]));
        }
      }
      if (live && cg == 0) {
        l = red[512 + rho] + red[640 + rho] + red[768 + rho] + red[896 + rho];
        __stcg(reinterpret_cast<float2*>(a.partials + a.ml_offset) + slot, make_float2(m, l));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kRowWarps + 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (tid == 0 && *abort_flag) atomicOr(a.status, kStTimeout);
}

// One warp per (request, kv head, row): merge the row's chunk partials. Lanes
// read the chunks' (m, l) once, form the weights e^(m_c - M) in shared memory
// and the denominator; then each lane sums its hd / 32 output dims over the
// chunks.
template <int HD>
__global__ void __launch_bounds__(256) attn_merge_kernel(const AttnArgs a) {
  constexpr int D = HD / 32;
  extern __shared__ float s_w[];  // [8 warps][max_chunks]
  const int nkv = a.n_kv_heads, group = a.n_heads / nkv;
  const int item = blockIdx.x, r = item / nkv, h = item - r * nkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rho = blockIdx.y * 8 + warp;
  pdl_trigger();
  pdl_wait();
  const int C = a.seq_len[r];
  const int row0 = a.req_row0[r], nrows = a.req_row0[r + 1] - row0;
  const int T = C + nrows;
  if (C < 0 || T > a.max_seq_len || rho >= nrows * group) return;
  const int nchunks = (T + kChunk - 1) / kChunk;
  const long long slot0 = static_cast<long long>(item) * a.max_chunks * a.max_rows + rho;
  const float2* ml = reinterpret_cast<const float2*>(a.partials + a.ml_offset) + slot0;
  float* w = s_w + warp * a.max_chunks;
  float M = -INFINITY;
  for (int c = lane; c < nchunks; c += 32) {
    const float2 v = __ldcg(ml + static_cast<long long>(c) * a.max_rows);
    w[c] = v.x;
    M = fmaxf(M, v.x);
  }
  M = warp_max(M);
  float L = 0.f;
  for (int c = lane; c < nchunks; c += 32) {
    const float mc = w[c];
    const float wc = mc == -INFINITY ? 0.f : expf(mc - M);
    L += __ldcg(ml + static_cast<long long>(c) * a.max_rows).y * wc;
    w[c] = wc;
  }
  L = warp_sum(L);
  __syncwarp();
  float o[D];
#pragma unroll
  for (int i = 0; i < D; ++i) o[i] = 0.f;
  const float* po = a.partials + slot0 * HD + lane * D;
#pragma unroll 4
  for (int c = 0; c < nchunks; ++c) {
    const float wc = w[c];
    const float* p = po + static_cast<long long>(c) * a.max_rows * HD;
    if constexpr (D == 4) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(p));
      o[0] = fmaf(wc, v.x, o[0]);
      o[1] = fmaf(wc, v.y, o[1]);
      o[2] = fmaf(wc, v.z, o[2]);
      o[3] = fmaf(wc, v.w, o[3]);
    } else {
      const float2 v = __ldcg(reinterpret_cast<const float2*>(p));
      o[0] = fmaf(wc, v.x, o[0]);
      o[1] = fmaf(wc, v.y, o[1]);
    }
  }
  const int j = rho / group, g = rho - j * group;
  const long long orow = static_cast<long long>(row0 + j) * a.n_heads * HD + (h * group + g) * HD + lane * D;
  const float invL = 1.0f / L;
#pragma unroll
  for (int i = 0; i < D; ++i) store_x(a.out, a.out_plane, orow + i, o[i] * invL, a.x_pair);
}

size_t attn_tc_smem(int hd) {
  const int nh = hd / 64;
  return 1024 + 8 * kTile + static_cast<size_t>(nh) * 2 * kTile + 8 * 8 + sizeof(float) * 2 * 4 * 128;
}

template <int HD>
cudaError_t launch_hd(const AttnArgs& a, int B, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                      cudaStream_t s) {
  const size_t smem = attn_tc_smem(HD);
  static bool attr_set[64] = {};  // per device
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t e = cudaSuccess;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(attn_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_merge_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  e = launch_k(attn_tc_kernel<HD>, dim3(B * a.n_kv_heads, a.max_chunks), dim3(kAttnThreads), smem, s, a.pdl != 0, q,
               k, v, a);
  if (e != cudaSuccess) return e;
  const size_t msmem = sizeof(float) * 8 * a.max_chunks;
  return launch_k(attn_merge_kernel<HD>, dim3(B * a.n_kv_heads, (a.max_rows + 7) / 8), dim3(256), msmem, s,
                  a.pdl != 0, a);
}

}  // namespace

bool attention_tc_supported(int head_dim, int page_size, int max_rows, int max_seq_len) {
  const long long max_chunks = (static_cast<long long>(max_seq_len) + kChunk - 1) / kChunk;
  return (head_dim == 64 || head_dim == 128) && page_size == 16 && max_rows <= 128 &&
         max_chunks * 8 * sizeof(float) <= 200 * 1024;
}

cudaError_t launch_attention_tc(const AttnArgs& a, int B, const CUtensorMap& q, const CUtensorMap& k,
                                const CUtensorMap& v, cudaStream_t s) {
  if (a.chunk != kChunk || !attention_tc_supported(a.head_dim, a.page_size, a.max_rows, a.max_seq_len))
    return cudaErrorInvalidValue;
  return a.head_dim == 128 ? launch_hd<128>(a, B, q, k, v, s) : launch_hd<64>(a, B, q, k, v, s);
}

}  // namespace sv
