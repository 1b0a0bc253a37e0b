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
// The keys of one (request, kv head) are split over a thread-block cluster
// of CS CTAs (CS chosen by the host from the batch so the grid fills the
// SMs; each CTA's key range, a multiple of 64 keys, follows from the
// request's actual length on the device). Each CTA processes its range in
// sub-chunks of 64 keys through a three-stage K/V ring:
//   warp 16  TMA: the Q tile once (the QKV epilogue left q / sqrt(hd) as a
//            hi/lo bf16 pair, q = hi + lo to ~16 bits; a 3D box of 64 dims x
//            group heads x block rows lands it as rows rho = j * group + g),
//            the range's page-table entries (256 at a time), then each
//            sub-chunk's K and V pages (16 keys x 64 dims per box) straight
//            from the page pool into the free stage;
//   warp 17  S_j = Q K_j^T (M 128, N 64, K hd; hi and lo into one
//            accumulator; S buffer j mod 2 in TMEM) and O_b += P_j V_j
//            (b = j mod 2; V is the N-major operand), S_{j+1} issued before
//            O_b += P_j V_j;
//   warps 0-15, two sets of eight (set b takes the sub-chunks j = b mod 2, so
//            the two softmaxes overlap; two warps per row, 32 keys each): the
//            row's scores are masked (key <= C_r + j), the set keeps its running
//            maximum m_b and sum l_b, and writes P_j = exp(S_j - m_b) as a
//            hi/lo bf16 pair into the set's P buffer once O_b += P_{j-2}
//            V_{j-2} has completed. The maximum is raised only when a
//            sub-chunk exceeds it by more than 8 (then O_b and l_b are
//            rescaled by e^(m_old - m_new)); otherwise p <= e^8 and O_b, l_b
//            stay exact in float32 relative to the kept m_b.
// At the end each row merges its two sets' (m_b, l_b, O_b) through their
// log-sum-exp into the CTA's partial (m, l, O), kept in shared memory. After
// a cluster barrier, rank i merges rows i R / CS .. of all CS partials over
// distributed shared memory,
//   out = sum_c O_c e^(m_c - M) / sum_c l_c e^(m_c - M), M = max_c m_c,
// and writes the attention output as the next projection's x tensor.
#include <cudaTypedefs.h>

#include "device_util.cuh"
#include "epilogue.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace sv {
namespace {

using namespace tc;

constexpr int kSub = 64;                              // keys per sub-chunk
constexpr int kStages = 5;                            // K/V ring depth
constexpr int kPageBlock = 256;                       // page-table entries the producer holds at once
constexpr int kMaxCluster = 16;                       // CTAs per (request, kv head)
constexpr int kSetWarps = 8;                          // a softmax set: two warps per 32-lane TMEM group
constexpr int kSetThreads = kSetWarps * 32;
constexpr int kRowWarps = 2 * kSetWarps;              // two sets, for even and odd sub-chunks
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

// 2^x by the SFU's approximate base-2 exponential (2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset of 16-byte chunk `ch` (0..7) of row `row` in a 128-byte swizzled tile.
__device__ __forceinline__ uint32_t sw128(int row, int ch) {
  return static_cast<uint32_t>(row) * 128u + static_cast<uint32_t>((ch ^ (row & 7)) * 16);
}

// N consecutive TMEM columns of this thread's lane (N = 32, 16, 8).
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float* v) {
  if constexpr (N == 32) tmem_ld32(taddr, v);
  else if constexpr (N == 16) tmem_ld16(taddr, v);
  else tmem_ld8(taddr, v);
}
// N consecutive 32-bit TMEM columns of this thread's lane, issued without the
// completion wait (the registers are read at issue): tmem_wait_st() completes
// every earlier store of the thread, so several stores share one wait.
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t* v) {
  if constexpr (N == 16) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
  } else if constexpr (N == 8) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
  } else {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3])
                 : "memory");
  }
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

template <int HD, int QC>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const AttnArgs a) {
  constexpr int NH = HD / 64;                     // 64-dim halves of a head
  // QC copies of the tile's query rows fill the 128 MMA rows (QL lanes each);
  // copy c takes keys [c 64 / QC, (c + 1) 64 / QC) of every sub-chunk, so each
  // softmax warp (two per TMEM lane group and set) handles NKW keys per row
  constexpr int QL = 128 / QC;
  constexpr int NKW = 32 / QC;
  constexpr uint32_t QB = 2 * NH * kTile;         // Q: hi and lo planes, NH halves of 128 rows x 128 B
  constexpr uint32_t KT = kSub * 128;             // a half-head tile of one sub-chunk: 64 keys x 128 B
  constexpr uint32_t KVB = 2 * NH * KT;           // one stage: K (NH halves), then V (NH halves)
  constexpr uint32_t KV_OFF = QB;
  constexpr uint32_t PM_OFF = KV_OFF + kStages * KVB;  // partial row maxima, bf16 [set][hf][128]
  // once every MMA is done the K/V ring holds the CTA's partial (O, then (m, l)) and
  // the merge's scratch: the two sets' (m, l), then the cluster merge's weights
  // the partial's rows are HD + 4 floats apart: the lanes of a warp store consecutive
  // rows, which a stride of HD floats (a multiple of 128 bytes) would put in one bank
  constexpr int OLD = HD + 4;
  constexpr uint32_t XCH_OFF = KV_OFF + 128 * OLD * 4 + 128 * 8;
  constexpr uint32_t WTS_OFF = XCH_OFF + 4 * 128 * 8;
  constexpr uint32_t MLS_OFF = WTS_OFF + 128 * 16 * 4;
  constexpr uint32_t MLR_OFF = MLS_OFF + 128 * 16 * 8;  // the cluster's merged (m, l) of this rank's rows
  static_assert(MLR_OFF + 128 * 8 + 16 <= KV_OFF + kStages * KVB, "merge scratch must fit the K/V ring");
  constexpr uint32_t BAR_OFF = PM_OFF + 2 * 2 * 2 * 128 + 4 * 16;  // + the pair wait flags
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;                // [kStages]
  uint64_t* kv_empty = kv_full + kStages;      // [kStages]
  uint64_t* s_full = kv_empty + kStages;       // [2]: S buffer b holds S_j, j = b mod 2
  uint64_t* p_ready = s_full + 2;              // [2]: set b has read S_j and written P_j
  uint64_t* pv_done = p_ready + 2;             // [2]: O_b += P_j V_j complete
  uint64_t* o_full = pv_done + 2;
  uint64_t* drain = o_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile uint32_t* vmask_s = reinterpret_cast<volatile uint32_t*>(abort_flag + 1);  // [kStages]: pages loaded

  const int lin = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
  unsigned long long* const rec = a.trace ? a.trace + static_cast<size_t>(lin) * kTraceWords : nullptr;
  if (rec && threadIdx.x == 0) {
    rec[0] = (static_cast<unsigned long long>(kTrAttn) << 48) | (static_cast<unsigned long long>(sm_id()) << 32) |
             static_cast<unsigned>(lin);
    trace_mark(rec, 1);
  }
  // The lengths, row ranges and page table read here and the cached keys the
  // producer requests before its dependency wait were written two or more
  // kernels back (every kernel triggers its dependents only after its own
  // wait); the query tile and the block's own keys wait for the QKV product.
  const int nkv = a.n_kv_heads, group = a.n_heads / nkv;
  // blockIdx.x = (request, kv head, row tile): a row tile is a.q_rows block rows
  // (a.q_rows * group <= 128 MMA rows), so a long block spans several tiles
  const int rt = blockIdx.x % a.n_row_tiles, rh = blockIdx.x / a.n_row_tiles;
  const int r = rh / nkv, h = rh - r * nkv;
  const int CS = gridDim.y, rank = blockIdx.y;  // the cluster spans the grid's y dimension
  const int C = a.seq_len[r];
  const int row0 = a.req_row0[r], nrows = a.req_row0[r + 1] - row0;
  const int j0 = rt * a.q_rows;                                    // first block row of the tile
  const int ntok = nrows - j0 < a.q_rows ? nrows - j0 : a.q_rows;  // its block rows
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  // a request flagged by the row preparation, or a row tile past the block: every
  // CTA of the cluster leaves here
  if (C < 0 || C + nrows > a.max_seq_len || ntok <= 0) {
    if (tid == 0) trace_mark(rec, 6);
    return;
  }
  const int T = C + j0 + ntok;  // keys any row of the tile may see
  // this CTA's keys [k0, k0 + nkeys): the T keys in CS ranges of a multiple of 64
  // CC clusters per work item (grid z) split the keys further; their merged partials meet in
  // global memory, where the last of them to arrive for a row slice finishes it
  const int CC = gridDim.z, cc = blockIdx.z;
  const int NR = CS * CC, ri = cc * CS + rank;
  const int per = ((T + NR - 1) / NR + kSub - 1) / kSub * kSub;
  const int k0 = ri * per;
  const int nkeys = T - k0 < per ? T - k0 : per;  // <= 0: no keys (an empty partial)
  const int nsub = nkeys > 0 ? (nkeys + kSub - 1) / kSub : 0;
  const int R = ntok * group;
  // the CTA's partial (m, l, O) of each row, in the K/V ring once every MMA is done
  float* Os = reinterpret_cast<float*>(smem + KV_OFF);        // [128 rows][OLD]
  float2* ML = reinterpret_cast<float2*>(smem + KV_OFF + 128 * OLD * 4);  // [128 rows]

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int st = 0; st < kStages; ++st) {
      mbar_init(kv_full + st, 1);
      mbar_init(kv_empty + st, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full + b, 1);
      mbar_init(p_ready + b, kSetThreads);
      mbar_init(pv_done + b, 1);
    }
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
  // S buffers at columns 0 and 64; set b's O at 128 + b * HD; set b's P (hi, lo: 32
  // columns each, two bf16 keys per column) at 128 + 2 HD + 64 b
  const uint32_t tS = tmem, tO = tmem + 128, tP = tmem + 128 + 2 * HD;

  if (warp != kRowWarps) {
    pdl_wait();
    pdl_trigger();
    if (tid == 0) trace_mark(rec, 2);
  }
  if (nsub == 0) {
    // no keys in this CTA's range: an empty partial
    if (warp == kRowWarps) {
      pdl_wait();
      pdl_trigger();
    }
    for (int rho = tid; rho < 128; rho += kAttnThreads) ML[rho] = make_float2(-INFINITY, 0.f);
  } else if (warp == kRowWarps) {
    // ------------------------------------------------------------ TMA producer
    const int* ptab = a.page_table + static_cast<long long>(r) * a.max_pages;
    if (lane == 0) {
      prefetch_tmap(&tmq);
      prefetch_tmap(&tmk);
      prefetch_tmap(&tmv);
    }
    // the range's page ids, kPageBlock at a time with all lookups in flight:
    // page i of the block sits in lane i % 32, register i / 32; -1 for a bad entry
    const int npg = (nkeys + 15) >> 4;
    int pg[kPageBlock / 32];
    auto load_pages = [&](int blk) {
#pragma unroll
      for (int t = 0; t < kPageBlock / 32; ++t) {
        const int i = blk * kPageBlock + t * 32 + lane;
        int page = -1;
        if (i < npg) {
          const int pidx = (k0 >> 4) + i;
          page = pidx < a.max_pages ? ptab[pidx] : -1;
          if (page < 0 || page >= a.n_pages) {
            atomicOr(a.status, pidx >= a.max_pages ? kStNoPage : kStBadPage);
            page = -1;
          }
        }
        pg[t] = page;
      }
    };
    const uint64_t pol = policy_evict_first();
    int issued = 0;
    // sub-chunks whose keys all lie below C (cached before this step) go out
    // before the dependency wait, up to the ring's depth; the block's own keys
    // wait for the QKV product (the query tile is the MMA thread's to load)
    const int n_early = C - k0 >= kSub ? min(min(nsub, kStages), (C - k0) / kSub) : 0;
    auto dep_wait = [&]() {
      pdl_wait();
      pdl_trigger();
    };
    for (int j = 0; j < nsub; ++j) {
      const int st = j % kStages;
      const int pj = j * (kSub / 16);  // the sub-chunk's first page in the range
      if (j == n_early) dep_wait();
      if (pj % kPageBlock == 0) load_pages(pj / kPageBlock);
      int ok = 1;
      if (lane == 0 && j >= kStages) ok = mbar_wait(kv_empty + st, (j / kStages - 1) & 1, abort_flag, kWaitNs);
      // the first two sub-chunks go out alone: the rest wait until the first has
      // landed, so that it is not served behind every CTA's whole ring
      if (lane == 0 && j == 2) ok = mbar_wait(kv_full, 0, abort_flag, kWaitNs);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      // lane p < 4 takes page i = pj + p of the range, from lane i % 32,
      // register (i % kPageBlock) / 32 (the same register for the sub-chunk's four pages)
      const int pi = pj + (lane & 3);
      const int t_sel = (pj % kPageBlock) >> 5;
      int held = pg[0];
#pragma unroll
      for (int t = 1; t < kPageBlock / 32; ++t) held = t == t_sel ? pg[t] : held;
      int page = __shfl_sync(0xffffffffu, held, pi & 31);
      if (lane >= kSub / 16 || pi >= npg) page = -1;
      const uint32_t mask = __ballot_sync(0xffffffffu, page >= 0);
      uint8_t* buf = smem + KV_OFF + st * KVB;
      if (lane == 0) {
        vmask_s[st] = mask;
        mbar_arrive_expect_tx(kv_full + st, static_cast<uint32_t>(__popc(mask)) * NH * 2 * 2048u);
      }
      __syncwarp();
      if (page >= 0) {  // the transaction count was raised above, before any of these copies
        const int row = (page * nkv + h) * 16;
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
          tma_load_2d(buf + hh * KT + lane * 2048, &tmk, hh * 64, row, kv_full + st, pol);
          tma_load_2d(buf + (NH + hh) * KT + lane * 2048, &tmv, hh * 64, row, kv_full + st, pol);
        }
      }
      ++issued;
    }
    if (n_early == nsub) dep_wait();  // (every sub-chunk was early)
    if (lane == 0) {  // the copies land before the CTA can leave
      volatile int never = 0;
      for (int j = issued - kStages < 0 ? 0 : issued - kStages; j < issued; ++j)
        mbar_wait(kv_full + j % kStages, (j / kStages) & 1, &never, kWaitNs);
    }
    __syncwarp();
  } else if (warp == kRowWarps + 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kSub);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, HD) | (1u << 16);  // B (V) is N-major
      const uint32_t q = smem_u32(smem);
      {
        // the query tile (hi and lo planes), written by the QKV product (this warp has
        // waited for it above): QC copies of the tile's rows, at MMA rows 0, QL, ..
        const uint32_t qbox = 128u * group * a.q_rows;
        mbar_arrive_expect_tx(q_full, 2 * NH * qbox * QC);
        const uint64_t polq = policy_evict_last();
#pragma unroll
        for (int cp = 0; cp < QC; ++cp)
#pragma unroll
          for (int pl = 0; pl < 2; ++pl)
#pragma unroll
            for (int hh = 0; hh < NH; ++hh)
              tma_load_3d(smem + (pl * NH + hh) * kTile + cp * QL * 128, &tmq, hh * 64, h * group,
                          pl * a.q_lo_row + row0 + j0, q_full, polq);
      }
      bool ok = mbar_wait(q_full, 0, abort_flag, kWaitNs);
      auto issue_s = [&](int j) {
        const int b = j & 1;
        const uint32_t k = smem_u32(smem + KV_OFF + (j % kStages) * KVB);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const int kh = ks >> 2;
          const uint32_t off = (ks & 3) * 32;
          const uint64_t bd = smem_desc_sw128(k + kh * KT + off);
          mma_bf16(tS + b * kSub, smem_desc_sw128(q + kh * kTile + off), bd, idesc_s, ks > 0 ? 1u : 0u);
          mma_bf16(tS + b * kSub, smem_desc_sw128(q + (NH + kh) * kTile + off), bd, idesc_s, 1u);
        }
        mma_commit(s_full + b);
      };
      auto issue_pv = [&](int j) {
        const int st = j % kStages, b = j & 1;
        const uint32_t pt = tP + b * 64;  // P_j (hi, then lo) in TMEM: the MMA's A operand
        const uint32_t v = smem_u32(smem + KV_OFF + st * KVB + NH * KT);
        const uint32_t to = tO + b * HD;
#pragma unroll
        for (int ks = 0; ks < kSub / 16; ++ks) {
          const uint64_t bd = smem_desc_sw128_mn(v + ks * 2048, KT, 1024);
          mma_bf16_ts(to, pt + ks * 8, bd, idesc_o, (j >= 2 || ks > 0) ? 1u : 0u);
          mma_bf16_ts(to, pt + 32 + ks * 8, bd, idesc_o, 1u);
        }
        mma_commit(kv_empty + st);  // K_j / V_j no longer needed
        mma_commit(pv_done + b);    // P_j no longer needed, O_b complete through j
      };
      for (int j = 0; j < nsub && ok; ++j) {
        const int b = j & 1;
        ok = mbar_wait(kv_full + j % kStages, (j / kStages) & 1, abort_flag, kWaitNs);
        if (j == 0) trace_mark(rec, 3);
        if (j == nsub - 1) trace_mark(rec, 10);
        // S buffer b was last read by set b for sub-chunk j - 2
        if (ok && j >= 2) ok = mbar_wait(p_ready + b, ((j >> 1) - 1) & 1, abort_flag, kWaitNs);
        if (!ok) break;
        tc_fence_after();
        issue_s(j);
        if (j >= 1) {
          ok = mbar_wait(p_ready + ((j - 1) & 1), ((j - 1) >> 1) & 1, abort_flag, kWaitNs);
          if (!ok) break;
          if (j == 1) trace_mark(rec, 13);
          tc_fence_after();
          issue_pv(j - 1);
        }
      }
      if (ok) {
        const int j = nsub - 1;
        ok = mbar_wait(p_ready + (j & 1), (j >> 1) & 1, abort_flag, kWaitNs);
        if (ok) {
          trace_mark(rec, 11);
          tc_fence_after();
          issue_pv(j);
          mma_commit(o_full);
        }
      }
      trace_mark(rec, 4);
      mma_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, &never, kDrainNs);
      mbar_wait(q_full, 0, &never, kWaitNs);  // the query copy lands before the CTA can leave
    }
  } else {
    // ------------------------------------------------------------ rows: softmax, output
    // set = warp / 8 takes sub-chunks j = set (mod 2); warp w reads TMEM lanes
    // 32 (w % 4) ..; one thread per TMEM lane rho (copy cp, tile row `row`) and
    // key half hf = (w / 4) mod 2 of the copy's keys: NKW keys from kk0 of each
    // of the set's sub-chunks
    const int set = warp >> 3, lg = warp & 3, hf = (warp >> 2) & 1;
    const int rho = lg * 32 + lane;
    const int cp = rho / QL, row = rho - cp * QL;
    const int kk0 = cp * (64 / QC) + hf * NKW;
    const bool live = row < R;
    const int lim = live ? C + j0 + row / group : -1;  // last key this row may see
    // a token tree row sees, of the block keys, only its ancestors and itself (node < 64)
    const bool tree = a.row_anc != nullptr;
    const unsigned long long anc = tree && live ? a.row_anc[row0 + j0 + row / group] : 0ull;
    const uint32_t lane_base = static_cast<uint32_t>(lg * 32) << 16;
    const uint32_t to = tO + set * HD;
    const uint32_t tp = tP + set * 64 + lane_base;  // this row's P columns (set's hi at +0, lo at +32)
    // partial maxima of the two warps of a row, truncated to bf16 so both warps
    // take the same maximum: [set][hf][128]
    uint16_t* pmax = reinterpret_cast<uint16_t*>(smem + PM_OFF);
    volatile int* pok = reinterpret_cast<volatile int*>(smem + PM_OFF + 2 * 2 * 2 * 128);  // [set][hf][lg]
    const int pair_bar = 1 + set * 4 + lg;  // named barrier of the row's two warps
    float m = -INFINITY, l = 0.f;  // this set's running maximum; this warp's part of the sum
    bool ok = true;
    // a warp whose 32 rows are all padding only keeps the handshakes
    const bool idle = lg * 32 - (lg * 32 / QL) * QL >= R;
    if (QC > 1) {
      // a lane's P row holds only its copy's keys: the other columns stay zero
      float z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = 0.f;
      tmem_st32(tP + set * 64 + (static_cast<uint32_t>(lg * 32) << 16) + hf * 32, z);
    }
    constexpr float kLog2e = 1.4426950408889634f;
    for (int j = set; j < nsub; j += 2) {
      const int st = j % kStages;
      // (waiting on kv_full too makes the producer's page mask visible here)
      int okw = 1;
      if (lane == 0)
        okw = mbar_wait(kv_full + st, (j / kStages) & 1, abort_flag, kWaitNs) &&
              mbar_wait(s_full + set, (j >> 1) & 1, abort_flag, kWaitNs);
      __syncwarp();
      okw = __shfl_sync(0xffffffffu, okw, 0);
      if (j == 0 && warp == 0 && lane == 0) trace_mark(rec, 12);
      if (idle && !okw) {
        ok = false;
        break;
      }
      const uint32_t vmask = vmask_s[st];
      const int kb = k0 + j * kSub + kk0;  // first key of this warp's slice
      float v[NKW];
      float corr = 1.f;
      if (!idle) {
        // both warps of the row reach the pair barrier, and leave together if either failed
        if (lane == 0) pok[(set * 2 + hf) * 4 + lg] = okw;
        if (!okw) {
          named_bar(pair_bar, 64);
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_ld_cols<NKW>(tS + lane_base + set * kSub + kk0, v);
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        constexpr uint32_t pgm = NKW >= 16 ? (1u << (NKW / 16)) - 1u : 1u;  // the slice's pages
        if (kb + NKW - 1 <= C && ((vmask >> (kk0 >> 4)) & pgm) == pgm) {
          // every key is cached context on a loaded page: no mask
#pragma unroll
          for (int i = 0; i < NKW; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], v[i]);
        } else {
#pragma unroll
          for (int i = 0; i < NKW; ++i) {
            const bool vis = kb + i <= lim && ((vmask >> ((kk0 + i) >> 4)) & 1u) &&
                             (!tree || kb + i < C || ((anc >> (kb + i - C)) & 1ull));
            v[i] = vis ? v[i] : -INFINITY;
            mx4[i & 3] = fmaxf(mx4[i & 3], v[i]);
          }
        }
        const uint32_t own = __float_as_uint(fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]))) >> 16;
        pmax[(set * 2 + hf) * 128 + rho] = static_cast<uint16_t>(own);
        named_bar(pair_bar, 64);
        if (!pok[(set * 2 + (hf ^ 1)) * 4 + lg]) {
          ok = false;
          break;
        }
        const uint32_t other = pmax[(set * 2 + (hf ^ 1)) * 128 + rho];
        const float mx = fmaxf(__uint_as_float(own << 16), __uint_as_float(other << 16));
        // raise the kept maximum only when this sub-chunk exceeds it by more than 8
        const float m_new = (m == -INFINITY || mx > m + 8.f) ? mx : m;
        corr = (m == -INFINITY || m_new == m) ? 1.f : __expf(m - m_new);
        m = m_new;
        // p = 2^(s log2 e - m log2 e); masked keys (s = -inf) give 0
        const float ml2 = m == -INFINITY ? 0.f : m * kLog2e;
        float lp4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < NKW; ++i) {
          v[i] = ex2_approx(fmaf(v[i], kLog2e, -ml2));
          lp4[i & 3] += v[i];
        }
        l = l * corr + ((lp4[0] + lp4[1]) + (lp4[2] + lp4[3]));
      }
      if (j >= set + 2) {
        // O_set += P_{j-2} V_{j-2} has completed: P may be overwritten and O_set rescaled
        if (lane == 0) mbar_wait(pv_done + set, (((j - set) >> 1) - 1) & 1, abort_flag, kWaitNs);
        __syncwarp();
      }
      if (!idle) {
        // P_j row rho into TMEM: keys kk0 + 2 i and + 1 in column kk0 / 2 + i (hi, and lo 32 columns on)
        uint32_t ph[NKW / 2], pl[NKW / 2];
#pragma unroll
        for (int q = 0; q < NKW / 8; ++q) {
          uint4 hi, lo;
          split8(v + 8 * q, hi, lo);
          ph[4 * q] = hi.x, ph[4 * q + 1] = hi.y, ph[4 * q + 2] = hi.z, ph[4 * q + 3] = hi.w;
          pl[4 * q] = lo.x, pl[4 * q + 1] = lo.y, pl[4 * q + 2] = lo.z, pl[4 * q + 3] = lo.w;
        }
        tmem_st_cols<NKW / 2>(tp + kk0 / 2, ph);
        tmem_st_cols<NKW / 2>(tp + 32 + kk0 / 2, pl);
        tmem_wait_st();  // both halves in TMEM before the P-ready arrival below
      }
      if (j >= set + 2 && __any_sync(0xffffffffu, corr != 1.f)) {
        // this warp rescales O_set's dims hf * HD / 2 .. + HD / 2
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < HD / 64; ++c) {
          float o[32];
          const uint32_t ta = to + lane_base + hf * (HD / 2) + c * 32;
          tmem_ld32(ta, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= corr;
          tmem_st32(ta, o);
        }
      }
      // V rows of keys past the request's end or on unloaded pages hold stale
      // bytes (possibly not finite); zero them so P = 0 there contributes 0
      const int kb0 = k0 + j * kSub;
      if (kb0 + kSub > T || vmask != 0xFu) {
        uint8_t* vb = smem + KV_OFF + st * KVB + NH * KT;
        for (int idx = (warp & 7) * 32 + lane; idx < kSub * NH * 8; idx += kSetThreads) {
          const int key_i = idx / (NH * 8), rem = idx - key_i * (NH * 8);
          const int hh = rem >> 3, c16 = rem & 7;
          if (kb0 + key_i >= T || !((vmask >> (key_i >> 4)) & 1u))
            *reinterpret_cast<uint4*>(vb + hh * KT + key_i * 128 + c16 * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(p_ready + set);
    }

    // merge the two sets' (m, l, O) of each row into the CTA's partial, in shared memory
    int okw = 0;
    if (lane == 0) okw = ok && mbar_wait(o_full, 0, abort_flag, kWaitNs) ? 1 : 0;
    if (tid == 0) trace_mark(rec, 14);
    okw = __shfl_sync(0xffffffffu, okw, 0);
    float2* xch = reinterpret_cast<float2*>(smem + XCH_OFF);  // [set][hf][128]
    if (okw) xch[(set * 2 + hf) * 128 + rho] = make_float2(m, l);
    named_bar(9, kRowThreads);
    if (okw) {
      const float2 a0 = xch[rho], b0 = xch[128 + rho], a1 = xch[256 + rho], b1 = xch[384 + rho];
      const float m0 = a0.x, l0 = a0.y + b0.y, m1 = a1.x, l1 = a1.y + b1.y;
      const float M = fmaxf(m0, m1);
      const float w0 = m0 == -INFINITY ? 0.f : __expf(m0 - M);
      const float w1 = m1 == -INFINITY ? 0.f : __expf(m1 - M);
      const bool has1 = nsub > 1;  // set 1 accumulated at least one P V product
      tc_fence_after();
      // warp (set, hf) writes O dims (2 set + hf) HD / 4 .. + HD / 4 of the merged row
      const int qd = (set * 2 + hf) * (HD / 4);
#pragma unroll 1
      for (int c = 0; c < HD / 64; ++c) {
        const int col = qd + c * 16;
        float o0[16], o1[16];
        tmem_ld16(tO + lane_base + col, o0);
        if (has1) tmem_ld16(tO + HD + lane_base + col, o1);
        float4* po = reinterpret_cast<float4*>(Os + rho * OLD + col);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float x[4];
#pragma unroll
          for (int t = 0; t < 4; ++t)
            x[t] = (w0 != 0.f ? o0[4 * i + t] * w0 : 0.f) + (has1 && w1 != 0.f ? o1[4 * i + t] * w1 : 0.f);
          po[i] = make_float4(x[0], x[1], x[2], x[3]);
        }
      }
      if (set == 0 && hf == 0) ML[rho] = live ? make_float2(M, l0 * w0 + l1 * w1) : make_float2(-INFINITY, 0.f);
    } else if (set == 0 && hf == 0) {
      ML[rho] = make_float2(-INFINITY, 0.f);
    }
    if (tid == 0) trace_mark(rec, 15);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kRowWarps + 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (tid == 0) trace_mark(rec, 7);
  // every CTA of the cluster has its partial in shared memory
  if (CS > 1) cluster_sync();
  if (tid == 0) trace_mark(rec, 8);
  {
    // rank i merges rows [i rpr, (i + 1) rpr) of the NP = CS QC partials (rank k,
    // copy c: lane c QL + row of rank k) with the weights e^(m_p - M) / sum_p l_p
    // e^(m_p - M), 4 output dims per item: with at most 8 partials each item forms
    // its row's weights from loads issued with its O loads; with more, one thread
    // per row forms them first
    constexpr int NPMAX = kMaxCluster * QC;
    const int NP = CS * QC;
    const int rpr = (R + CS - 1) / CS;
    const int rr0 = rank * rpr, rr1 = rr0 + rpr < R ? rr0 + rpr : R;
    const uint32_t os_addr = smem_u32(Os), ml_addr = smem_u32(ML);
    const int nrr = rr1 - rr0;
    constexpr int D4 = HD / 4;
    constexpr int KB = 8;  // partials whose loads are in flight together
    static_assert(NPMAX % KB == 0, "partials in groups of KB");
    // the merged row: the output (one cluster), or with several clusters the row's
    // unnormalized partial and (M, L) for the last of them to arrive
    auto finish = [&](int rr, int d, float4 acc, float M, float L) {
      const int rho = rr0 + rr;
      if (CC > 1) {
        const size_t slot = static_cast<size_t>(blockIdx.x) * CC + cc;
        __stcg(reinterpret_cast<float4*>(a.xpart + (slot * 128 + rho) * HD + d), acc);
        if (d == 0) __stcg(a.xml + slot * 128 + rho, make_float2(M, L));
        return;
      }
      const int jrow = j0 + rho / group, g = rho % group;
      const long long orow = static_cast<long long>(row0 + jrow) * a.n_heads * HD + (h * group + g) * HD + d;
      store_x4(a.out, a.out_plane, orow, acc, a.x_pair);
    };
    if (NP <= KB) {
      // few partials: every item loads its row's (m, l) and O of each partial in one
      // round trip and forms the row's weights itself (the same arithmetic, in the
      // same order, as the two-phase merge below)
      if (tid == 0) trace_mark(rec, 9);
      for (int it = tid; it < nrr * D4; it += kAttnThreads) {
        const int rr = it / D4, rho = rr0 + rr, d = (it % D4) * 4;
        float2 ml[KB];
        float4 o[KB];
#pragma unroll
        for (int p = 0; p < KB; ++p)
          if (p < NP) {
            const uint32_t ln = static_cast<uint32_t>((p % QC) * QL + rho), rk = static_cast<uint32_t>(p / QC);
            ml[p] = ld_dsmem_f32x2(mapa_shared(ml_addr + 8u * ln, rk));
            o[p] = ld_dsmem_f32x4(mapa_shared(os_addr + 4u * (ln * OLD + d), rk));
          }
        float M = -INFINITY;
#pragma unroll
        for (int p = 0; p < KB; ++p)
          if (p < NP) M = fmaxf(M, ml[p].x);
        float w[KB];
        float L = 0.f;
#pragma unroll
        for (int p = 0; p < KB; ++p) {
          w[p] = p < NP && ml[p].x != -INFINITY ? __expf(ml[p].x - M) : 0.f;
          if (p < NP) L += ml[p].y * w[p];
        }
        // L = 0 only for rows whose keys were all on bad pages (flagged): output 0. With
        // several clusters the sum stays unnormalized until their partials meet.
        const float inv = CC > 1 ? 1.f : (L > 0.f ? 1.0f / L : 0.f);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int p = 0; p < KB; ++p) {
          const float wp = p < NP ? w[p] * inv : 0.f;
          if (wp != 0.f) {
            acc.x += o[p].x * wp;
            acc.y += o[p].y * wp;
            acc.z += o[p].z * wp;
            acc.w += o[p].w * wp;
          }
        }
        finish(rr, d, acc, M, L);
      }
    } else {
      float* wts = reinterpret_cast<float*>(smem + WTS_OFF);    // [rpr][NP]
      float2* mls = reinterpret_cast<float2*>(smem + MLS_OFF);  // [rpr][NP]
      // every partial's (m, l) of this rank's rows, all loads in flight
      for (int it = tid; it < nrr * NP; it += kAttnThreads) {
        const int rr = it / NP, p = it - rr * NP;
        const uint32_t ln = static_cast<uint32_t>((p % QC) * QL + rr0 + rr);
        mls[rr * NP + p] = ld_dsmem_f32x2(mapa_shared(ml_addr + 8u * ln, static_cast<uint32_t>(p / QC)));
      }
      __syncthreads();
      for (int rr = tid; rr < nrr; rr += kAttnThreads) {
        float M = -INFINITY;
        for (int p = 0; p < NP; ++p) M = fmaxf(M, mls[rr * NP + p].x);
        float L = 0.f;
        for (int p = 0; p < NP; ++p) {
          const float2 v = mls[rr * NP + p];
          const float w = v.x == -INFINITY ? 0.f : __expf(v.x - M);
          wts[rr * NP + p] = w;
          L += v.y * w;
        }
        // L = 0 only for rows whose keys were all on bad pages (flagged): output 0. With
        // several clusters the sum stays unnormalized until their partials meet.
        const float inv = CC > 1 ? 1.f : (L > 0.f ? 1.0f / L : 0.f);
        for (int p = 0; p < NP; ++p) wts[rr * NP + p] *= inv;
        if (CC > 1) reinterpret_cast<float2*>(smem + MLR_OFF)[rr] = make_float2(M, L);
      }
      __syncthreads();
      if (tid == 0) trace_mark(rec, 9);
      for (int it = tid; it < nrr * D4; it += kAttnThreads) {
        const int rr = it / D4, rho = rr0 + rr, d = (it % D4) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int p0 = 0; p0 < NP; p0 += KB) {
          float4 o[KB];
#pragma unroll
          for (int kk = 0; kk < KB; ++kk) {
            const int p = p0 + kk;
            if (p < NP && wts[rr * NP + p] != 0.f)
              o[kk] = ld_dsmem_f32x4(mapa_shared(os_addr + 4u * (((p % QC) * QL + rho) * OLD + d),
                                                 static_cast<uint32_t>(p / QC)));
          }
#pragma unroll
          for (int kk = 0; kk < KB; ++kk) {
            const float w = p0 + kk < NP ? wts[rr * NP + p0 + kk] : 0.f;
            if (w != 0.f) {
              acc.x += o[kk].x * w;
              acc.y += o[kk].y * w;
              acc.z += o[kk].z * w;
              acc.w += o[kk].w * w;
            }
          }
        }
        const float2 mlr = CC > 1 ? reinterpret_cast<const float2*>(smem + MLR_OFF)[rr] : make_float2(0.f, 0.f);
        finish(rr, d, acc, mlr.x, mlr.y);
      }
    }
    if (CC > 1) {
      // the last of the item's CC clusters to arrive for this rank's rows merges their partials
      volatile int* s_last = reinterpret_cast<volatile int*>(smem + MLR_OFF + 128 * 8);
      __threadfence();
      __syncthreads();
      unsigned* cnt = a.xcnt + static_cast<size_t>(blockIdx.x) * kMaxCluster + rank;
      if (tid == 0) *s_last = atomicAdd(cnt, 1u) == static_cast<unsigned>(CC - 1) ? 1 : 0;
      __syncthreads();
      if (*s_last) {
        __threadfence();
        for (int it = tid; it < nrr * D4; it += kAttnThreads) {
          const int rr = it / D4, rho = rr0 + rr, d = (it % D4) * 4;
          const size_t base = static_cast<size_t>(blockIdx.x) * CC;
          // every cluster's (m, l) and partial O of this row and 4 dims, all loads in flight
          float2 ml[kMaxCrossClusters];
          float4 o[kMaxCrossClusters];
#pragma unroll
          for (int c = 0; c < kMaxCrossClusters; ++c)
            if (c < CC) {
              ml[c] = __ldcg(a.xml + (base + c) * 128 + rho);
              o[c] = __ldcg(reinterpret_cast<const float4*>(a.xpart + ((base + c) * 128 + rho) * HD + d));
            }
          float M = -INFINITY;
#pragma unroll
          for (int c = 0; c < kMaxCrossClusters; ++c)
            if (c < CC) M = fmaxf(M, ml[c].x);
          float L = 0.f;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int c = 0; c < kMaxCrossClusters; ++c) {  // in cluster order: a fixed summation order
            const float w = c < CC && ml[c].x != -INFINITY ? __expf(ml[c].x - M) : 0.f;
            if (w == 0.f) continue;
            L += ml[c].y * w;
            acc.x += o[c].x * w;
            acc.y += o[c].y * w;
            acc.z += o[c].z * w;
            acc.w += o[c].w * w;
          }
          const float inv = L > 0.f ? 1.0f / L : 0.f;
          acc = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
          const int jrow = j0 + rho / group, g = rho % group;
          const long long orow = static_cast<long long>(row0 + jrow) * a.n_heads * HD + (h * group + g) * HD + d;
          store_x4(a.out, a.out_plane, orow, acc, a.x_pair);
        }
        if (tid == 0) *cnt = 0u;
      }
    }
  }
  if (tid == 0) trace_mark(rec, 5);
  // no CTA leaves while a rank of its cluster may still read its partial
  if (CS > 1) cluster_sync();
  if (tid == 0) {
    if (*abort_flag) atomicOr(a.status, kStTimeout);
    trace_mark(rec, 6);
  }
}

size_t attn_tc_smem(int hd) {
  const size_t nh = hd / 64, q = 2 * nh * kTile, kv = 2 * nh * kSub * 128;
  return 1024 + q + kStages * kv + 2 * 2 * 2 * 128 + 4 * 16 + (2 * kStages + 9) * 8 + 32;
}

template <int HD, int QC>
cudaError_t set_attrs() {
  static bool attr_set[64] = {};  // per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && attr_set[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<HD, QC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(attn_tc_smem(HD)));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_tc_kernel<HD, QC>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess && dev >= 0 && dev < 64) attr_set[dev] = true;
  return e;
}

template <int HD, int QC>
cudaError_t launch_hd(const AttnArgs& a, int B, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                      cudaStream_t s) {
  cudaError_t e = set_attrs<HD, QC>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B * a.n_kv_heads * a.n_row_tiles, a.cl_size, a.cl_count);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = attn_tc_smem(HD);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(a.cl_size);
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, attn_tc_kernel<HD, QC>, q, k, v, a);
}

template <int HD>
int max_clusters_hd(int cs) {
  if (set_attrs<HD, 1>() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, cs);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = attn_tc_smem(HD);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, attn_tc_kernel<HD, 1>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace

void attention_tc_split(long long items, int head_dim, int sm_count, int* cs_out, int* cc_out) {
  int cs = attention_tc_cluster(items, head_dim, sm_count), cc = 1;
  // few work items: several clusters per item (merged through global memory) so that
  // about every SM streams keys; cs * cc CTAs per item, all clusters co-resident
  if (items <= kCrossItems && items * cs * 2 <= sm_count) {
    int best = cs, bcs = cs, bcc = 1;
    for (int c = 2; c <= kMaxCrossClusters; c *= 2)
      for (int s = 2; s <= 8; s *= 2) {
        if (items * s * c > sm_count || s * c <= best) continue;
        const int mc = head_dim == 128 ? max_clusters_hd<128>(s) : max_clusters_hd<64>(s);
        if (mc < items * c) continue;  // every cluster of the launch resident at once
        best = s * c;
        bcs = s;
        bcc = c;
      }
    cs = bcs;
    cc = bcc;
  }
  *cs_out = cs;
  *cc_out = cc;
}

int attention_tc_cluster(long long items, int head_dim, int sm_count) {
  // CTAs per (request, kv head, row tile): about two waves of CTAs over the SMs,
  // at most kMaxCluster, halved while the device cannot hold the clusters one
  // wave needs
  long long want = (2LL * sm_count + items - 1) / items;
  int cs = 1;
  while (cs * 2 <= want && cs * 2 <= kMaxCluster) cs *= 2;
  for (; cs > 1; cs /= 2) {
    const int mc = head_dim == 128 ? max_clusters_hd<128>(cs) : max_clusters_hd<64>(cs);
    const long long need = items < sm_count / cs ? items : sm_count / cs;
    if (mc * 10LL >= need * 9) break;
  }
  return cs;
}

bool attention_tc_supported(int head_dim, int page_size, int max_rows, int max_seq_len) {
  (void)max_seq_len;
  (void)max_rows;  // any block length: rows beyond one MMA tile go to further row tiles
  return (head_dim == 64 || head_dim == 128) && page_size == 16;
}

cudaError_t launch_attention_tc(const AttnArgs& a, int B, const CUtensorMap& q, const CUtensorMap& k,
                                const CUtensorMap& v, cudaStream_t s) {
  const int qc = a.q_copies;
  if (a.cl_count < 1 || a.cl_count > kMaxCrossClusters ||
      (a.cl_count > 1 && (B * a.n_kv_heads * a.n_row_tiles > kCrossItems || !a.xpart || !a.xml || !a.xcnt)))
    return cudaErrorInvalidValue;
  if (a.cl_size < 1 || a.cl_size > kMaxCluster || a.q_rows < 1 || (qc != 1 && qc != 2 && qc != 4) ||
      a.q_rows * (a.n_heads / a.n_kv_heads) * qc > 128 || a.n_row_tiles < 1 ||
      !attention_tc_supported(a.head_dim, a.page_size, a.max_rows, a.max_seq_len))
    return cudaErrorInvalidValue;
  if (a.head_dim == 128)
    return qc == 4 ? launch_hd<128, 4>(a, B, q, k, v, s)
                   : qc == 2 ? launch_hd<128, 2>(a, B, q, k, v, s) : launch_hd<128, 1>(a, B, q, k, v, s);
  return qc == 4 ? launch_hd<64, 4>(a, B, q, k, v, s)
                 : qc == 2 ? launch_hd<64, 2>(a, B, q, k, v, s) : launch_hd<64, 1>(a, B, q, k, v, s);
}

}  // namespace sv
