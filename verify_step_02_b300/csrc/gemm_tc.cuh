// Weight-streaming skinny GEMM on the 5th-generation tensor cores (tcgen05).
//
// y[m][n] = x[m] . W[n] for bf16 weights W [rows][K] and bf16 activations, one
// plane or a hi/lo pair (x = hi + lo: both planes are multiplied into the same
// float32 accumulator). The verify block has M = sum(L_r + 1) rows, a few to a
// few hundred, so W is the big operand: it is the MMA's A operand (128 weight
// rows per tile, the MMA's M), and the block's tokens are its N (32 .. 256
// columns). Every weight byte is read from HBM exactly once per launch.
//
// Two ways to spread the K range of the tiles over the SMs:
//   stream-K   P <= #SM CTAs share U = tiles x K blocks units; CTA c takes
//              units [c U / P, (c+1) U / P), so every SM streams the same
//              bytes. With more tiles than CTAs, the first tiles - P tiles
//              are shared this way and then every CTA takes one whole tile
//              of its own, so that it ends on a local epilogue rather than
//              on a hand-off. A tile whose K range is shared by several CTAs
//              is finished by those of them whose shared ranges end inside
//              it: once every contributor's partial tile is in global memory,
//              each sums its own slice of the tile's tokens in CTA order and
//              runs the slice's epilogue, so no single SM reads the whole
//              tile's partials.
//   cluster    (token tiles of at most 64 columns, one weight tile per cluster:
//              the q|k|v, O and down projections) the CS CTAs of a cluster split the
//              tile's K blocks evenly. Each rank stores a 1/CS share of its
//              partial tile's tokens straight into the shared memory of the
//              rank that finishes those tokens (asynchronous stores counted on
//              that rank's mbarrier); rank r sums the CS shares in rank order
//              (a reduce-scatter) and runs their epilogue from inputs it
//              staged in shared memory while the weights streamed. The
//              hand-off at the end of the product then needs no round trip
//              through L2, which is what the end of a launch waits on.
// Both orders are fixed, so results do not depend on timing.
//
// Roles inside a CTA (384 threads; W12 weights: 512):
//   warp 0     one thread issues TMA loads of the weight tile (two 64-row
//              boxes) and the x tile (32-row boxes per plane) into an S-stage
//              shared-memory ring;
//   warp 1     allocates the TMEM accumulators (two buffers of NT columns) and
//              one thread issues tcgen05.mma (M 128, N NT, K 16) per stage;
//   warps 4-7  read finished accumulators out of TMEM (warp w reads lanes
//              32 (w % 4) ..), and hand off partial tiles or run the epilogue;
//              warps 8-11 share the reduction and the epilogue (bf16), or
//              with warps 2, 3 and 12-15 rebuild the W12 tiles.
// Every wait is bounded; a wait that runs out sets the status word's timeout
// bit and the whole CTA winds down (waits for its copies and MMAs in flight,
// frees TMEM, returns).
#pragma once

#include <cudaTypedefs.h>

#include "epilogue.cuh"
#include "gemm_tc_plan.h"
#include "internal.h"
#include "tc_ptx.cuh"

namespace sv {
namespace tcg {

using namespace tc;

constexpr uint64_t kWaitNs = 2000000000ull;     // 2 s
constexpr uint64_t kDrainNs = 200000000ull;     // 0.2 s

__host__ __device__ constexpr uint32_t tmem_cols(int nt) {
  return 2 * nt <= 32 ? 32u : 2 * nt <= 64 ? 64u : 2 * nt <= 128 ? 128u : 2 * nt <= 256 ? 256u : 512u;
}

// First CTA whose unit range contains unit x: the largest c with floor(c U / P) <= x.
__device__ __forceinline__ int cta_of_unit(long long x, long long U, int P) {
  return static_cast<int>(((x + 1) * P + U - 1) / U - 1);
}

// The units (tile, K block) of one CTA, in processing order: a contiguous
// range of the tile-major order of the stream-K tiles, then (with more tiles
// than CTAs) one whole tile of its own (stream-K), or every K block of the
// CTA's slice [k0, k1) of each tile in [t0, t1) (cluster split).
struct CtaUnits {
  long long u0, n;   // stream-K: first unit; both: units of this CTA
  long long nsk;     // stream-K: units of the shared range (then the whole tile tdp, if tdp >= 0)
  long long tdp;
  long long t0;      // cluster: first tile
  int k0, nk;        // cluster: first K block and K blocks per tile
  int kb;            // K blocks of a whole tile
  bool cl;
  __device__ __forceinline__ void at(long long i, long long& t, int& kbi) const {
    if (cl) {
      const long long q = i / nk;
      t = t0 + q;
      kbi = k0 + static_cast<int>(i - q * nk);
    } else if (i < nsk) {
      const long long u = u0 + i;
      t = u / kb;
      kbi = static_cast<int>(u - t * kb);
    } else {
      t = tdp;
      kbi = static_cast<int>(i - nsk);
    }
  }
  // one past the last unit of the tile that unit i belongs to
  __device__ __forceinline__ long long seg_end(long long i) const {
    if (cl) return (i / nk + 1) * nk;
    if (i >= nsk) return n;
    const long long t = (u0 + i) / kb;
    const long long e = (t + 1) * kb - u0;
    return e < nsk ? e : nsk;
  }
};

// Spin (bounded, like mbar_wait) until the counter at p reaches `target`; the
// load has acquire semantics at GPU scope.
__device__ __forceinline__ int wait_count(const unsigned* p, unsigned target, volatile int* abort, uint64_t limit_ns) {
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0;; ++i) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= target) return 1;
    if ((i & 15u) == 15u) {
      if (*abort) return 0;
      if (global_ns() - t0 > limit_ns) {
        *abort = 1;
        return 0;
      }
    }
    __nanosleep(32);
  }
}

template <int NT, bool PAIR, bool W12, bool CL>
__global__ void __launch_bounds__(W12 ? kTcThreadsW12 : kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmx,
                   const GemmArgs a) {
  constexpr int KS = tc_ks_for(NT, PAIR, W12);
  constexpr int BX = NT * 128;              // bytes of one x plane per 64-wide sub-tile
  constexpr int XQ = BX * (PAIR ? 2 : 1);   // x bytes per sub-tile
  constexpr int SUB = W12 ? XQ : kABytes + XQ;          // one 64-wide sub-tile: (weights,) then x
  constexpr int XOFF = W12 ? kW12Planes : kABytes;      // x of sub-tile q at q * SUB + XOFF
  constexpr int NSUB = KS / 64;
  constexpr int STAGE = stage_bytes(NT, PAIR, KS, W12);
  // hi/lo x planes: their tiles sit back to back in shared memory (rows 0 .. NT - 1,
  // then NT .. 2 NT - 1), so one MMA of N = 2 NT reads the weight tile once and
  // leaves W x_hi and W x_lo side by side in TMEM; the epilogue adds them
  constexpr bool FUSE = PAIR && 2 * NT <= 256;
  constexpr int ACC = FUSE ? 2 * NT : NT;               // accumulator columns per TMEM buffer
  constexpr uint32_t TCOLS = tmem_cols(ACC);
  constexpr int EPT = W12 ? 128 : kEpiThreads;          // epilogue threads (W12: warps 8-11 rebuild weights)
  constexpr int NCONV = kTcThreadsW12 / 32 - 6;         // W12 rebuild warps: 2, 3, 8 .. 15
  static_assert(!W12 || KS == 128, "W12 tiles are 128 elements wide");
  static_assert(!CL || NT <= kClusterMaxNT, "cluster split: token tiles of at most kClusterMaxNT columns");
  // (the cluster split takes 2 .. 8 CTAs per cluster, so a rank's slice is at most 32 tokens)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.tc_stages;
  uint8_t* aring = smem + static_cast<size_t>(S) * STAGE;  // W12: rebuilt bf16 weight tiles, 2 x NSUB x 16 KB
  // stream-K: Ys [128][33] and the launch's per-token data. Cluster split: the rank's
  // token slice of SL columns: Ys [128][SL + 1], staged epilogue inputs Es [128][SL],
  // and Rx [CS][128][SL], the slices of every rank's partial tile that the ranks
  // store into this CTA's shared memory
  const int SL = CL ? cl_slice(NT, a.cl_size) : 32;
  const int YLD = CL ? SL + 1 : kYsLd;
  float* Ys = reinterpret_cast<float*>(aring + (W12 ? kW12Ring * NSUB * kABytes : 0));
  EpiSmem* esm = reinterpret_cast<EpiSmem*>(Ys + kGemmBN * YLD);
  TokData* tok = reinterpret_cast<TokData*>(esm + 1);
  float* Rx = reinterpret_cast<float*>(esm + 1);
  float* Es = Rx + (CL ? a.cl_size : 0) * kGemmBN * SL;
  uint64_t* full = CL ? reinterpret_cast<uint64_t*>(Es + kGemmBN * SL) : reinterpret_cast<uint64_t*>(tok + 1);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* afull = drain + 1;     // W12 ring: rebuilt tile ready
  uint64_t* aempty = afull + 2;    // W12 ring: tile consumed by the MMAs
  uint64_t* rx_full = aempty + 2;  // cluster: every rank's slice for this CTA has landed (transaction bytes)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rx_full + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = a.grid_p, c = blockIdx.x;
  // stream-K: with more tiles than CTAs (and at least one unit per CTA left to share),
  // CTA c shares the first NTT - P tiles' units with the others, then takes tile
  // NTT - P + c whole, so that it ends on a tile of its own, not on a hand-off
  const long long NTT = static_cast<long long>(a.n_tiles) * a.m_tiles;
  const long long TSK = NTT > P && (NTT - P) * a.kb >= P ? NTT - P : NTT;  // tiles shared by stream-K
  const long long USK = TSK * a.kb;                                           // their units
  const int CS = CL ? a.cl_size : 1;
  const int rank = CL ? static_cast<int>(cluster_ctarank()) : 0;
  CtaUnits W;
  W.kb = a.kb;
  W.cl = CL;
  if (CL) {
    const long long ntt = static_cast<long long>(a.n_tiles) * a.m_tiles;
    W.t0 = static_cast<long long>(c / CS) * a.cl_tiles;
    const long long t1 = W.t0 + a.cl_tiles < ntt ? W.t0 + a.cl_tiles : ntt;
    W.k0 = rank * a.kb / CS;
    W.nk = (rank + 1) * a.kb / CS - W.k0;
    W.u0 = 0;
    W.n = (t1 > W.t0 ? t1 - W.t0 : 0) * W.nk;
    W.nsk = W.n;
    W.tdp = -1;
  } else {
    W.u0 = c * USK / P;
    W.nsk = (c + 1) * USK / P - W.u0;
    W.tdp = TSK < NTT ? TSK + c : -1;
    W.n = W.nsk + (W.tdp >= 0 ? a.kb : 0);
    W.t0 = 0;
    W.k0 = 0;
    W.nk = a.kb;
  }
  const long long NU = W.n;
  unsigned long long* const rec = a.trace ? a.trace + static_cast<size_t>(c) * kTraceWords : nullptr;
  if (rec && threadIdx.x == 0) {
    rec[0] = (static_cast<unsigned long long>(kTrGemm) << 48) | (static_cast<unsigned long long>(sm_id()) << 32) |
             static_cast<unsigned>(c);
    trace_mark(rec, 1);
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, W12 ? 1 + NCONV : 1);  // W12: the MMAs (x) and every rebuild warp (planes)
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(afull + i, NCONV);
      mbar_init(aempty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(acc_full + i, 1);
      mbar_init(acc_empty + i, 128);  // the TMEM-reading warpgroup
    }
    mbar_init(drain, 1);
    mbar_init(rx_full, 1);  // this CTA's own arrival (with the bytes it expects)
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    if (!W12) prefetch_tmap(&tmw);
    prefetch_tmap(&tmx);
  }
  if (warp == 1) tmem_alloc(tmem_slot, TCOLS);
  tc_fence_before();
  // cluster: every CTA's barriers exist before any rank arrives on them remotely
  if (CL)
    cluster_sync();
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pw = policy_evict_first(), px = policy_evict_last();
      const int w12_row_blocks = (a.n_rows + 63) / 64;
      // bytes one unit brings into its stage (W12: row halves past the matrix are not read)
      auto unit_bytes = [&](long long t) -> uint32_t {
        if (!W12) return STAGE;
        const int nt = static_cast<int>(t / a.m_tiles);
        const int r1 = a.pair == kPairSwiglu ? a.ffn + nt * (kGemmBN / 2) : nt * kGemmBN + kGemmBN / 2;
        return STAGE - (r1 / 64 < w12_row_blocks ? 0 : 3 * 4096);
      };
      // weight boxes, all sub-tiles back to back: each row's KS elements are
      // requested together (contiguous bytes in HBM)
      auto load_w = [&](long long t, int kb, uint8_t* st, uint64_t* bar) {
        const int nt = static_cast<int>(t / a.m_tiles);
        const int r0 = a.pair == kPairSwiglu ? nt * (kGemmBN / 2) : nt * kGemmBN;
        const int r1 = a.pair == kPairSwiglu ? a.ffn + nt * (kGemmBN / 2) : r0 + kGemmBN / 2;
        if constexpr (W12) {
          // the planes' 4096-byte tiles (row block, kb) of both row halves: contiguous reads
          const uint8_t* wb = static_cast<const uint8_t*>(a.w);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int rb = (hh ? r1 : r0) / 64;
            if (rb >= w12_row_blocks) continue;
            const long long off = (static_cast<long long>(rb) * a.w12_kt + kb) * 4096;
#pragma unroll
            for (int p = 0; p < 3; ++p)
              bulk_load(st + p * 8192 + hh * 4096, wb + p * a.w12_plane + off, 4096, bar, pw);
          }
        } else {
#pragma unroll
          for (int q = 0; q < NSUB; ++q) {
            tma_load_2d(st + q * SUB, &tmw, kb * KS + q * 64, r0, bar, pw);
            tma_load_2d(st + q * SUB + kABytes / 2, &tmw, kb * KS + q * 64, r1, bar, pw);
          }
        }
      };
      auto load_x = [&](long long t, int kb, uint8_t* st, uint64_t* bar) {
        const int mt = static_cast<int>(t - (t / a.m_tiles) * a.m_tiles);
#pragma unroll
        for (int q = 0; q < NSUB; ++q) {
          uint8_t* sb = st + q * SUB + XOFF;
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
      const long long npre = NU < S ? NU : S;
      for (long long i = 0; i < npre; ++i) {
        long long t;
        int kb;
        W.at(i, t, kb);
        uint8_t* st = smem + static_cast<size_t>(i) * STAGE;
        mbar_arrive_expect_tx(full + i, unit_bytes(t));
        load_w(t, kb, st, full + i);
      }
      pdl_wait();
      pdl_trigger();
      trace_mark(rec, 2);
      for (long long i = 0; i < npre; ++i) {
        long long t;
        int kb;
        W.at(i, t, kb);
        load_x(t, kb, smem + static_cast<size_t>(i) * STAGE, full + i);
      }
      int stage = static_cast<int>(npre % S);
      uint32_t phase = npre == S ? 1u : 0u;
      long long issued = npre;
      for (long long i = npre; i < NU; ++i) {
        if (!mbar_wait(empty + stage, phase ^ 1u, abort_flag, kWaitNs)) break;
        long long t;
        int kb;
        W.at(i, t, kb);
        uint8_t* st = smem + static_cast<size_t>(stage) * STAGE;
        mbar_arrive_expect_tx(full + stage, unit_bytes(t));
        load_w(t, kb, st, full + stage);
        load_x(t, kb, st, full + stage);
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
      constexpr uint32_t idesc = idesc_bf16_f32(kGemmBN, ACC);
      int stage = 0, seg = 0, ai = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (long long i = 0; i < NU && ok;) {
        const long long iend = W.seg_end(i);
        const int b = seg & 1;
        if (!mbar_wait(acc_empty + b, ((seg >> 1) & 1) ^ 1u, abort_flag, kWaitNs)) break;
        tc_fence_after();
        const uint32_t d = tmem + b * ACC;
        for (long long v = i; v < iend; ++v) {
          // W12: the rebuild warps saw this stage land before they filled the tile
          if (!mbar_wait(W12 ? afull + ai % kW12Ring : full + stage, W12 ? (ai / kW12Ring) & 1 : phase, abort_flag,
                         kWaitNs)) {
            ok = false;
            break;
          }
          if (ai == 0) trace_mark(rec, 3);
          tc_fence_after();
          const uint32_t st = smem_u32(smem + static_cast<size_t>(stage) * STAGE);
          const uint32_t at = smem_u32(aring + (ai % kW12Ring) * NSUB * kABytes);
#pragma unroll
          for (int q = 0; q < NSUB; ++q) {
            const uint32_t sa = W12 ? at + q * kABytes : st + q * SUB, sb = st + q * SUB + XOFF;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = smem_desc_sw128(sa + k * 32);
              mma_bf16(d, ad, smem_desc_sw128(sb + k * 32), idesc, (v > i || q > 0 || k > 0) ? 1u : 0u);
              if (PAIR && !FUSE) mma_bf16(d, ad, smem_desc_sw128(sb + BX + k * 32), idesc, 1u);
            }
          }
          mma_commit(empty + stage);  // frees the stage once these MMAs have read it
          if (W12) mma_commit(aempty + ai % kW12Ring);
          ++ai;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(acc_full + b);
        ++seg;
        i = iend;
      }
      trace_mark(rec, 4);
      // every MMA issued above has completed once `drain` flips
      mma_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, &never, kDrainNs);
    }
  } else if (W12 && (warp == 2 || warp == 3 || warp >= 8)) {
    // ------------------------------------------------------------ W12 rebuild
    // Each unit's three plane tiles become the bf16 weight tile, in the
    // 128-byte swizzled layout the MMA reads: per element, code
    // c = p0 | p1 << 4 | p2 << 8 and bf16 = ((c & 0x7FF) + (base << 7)) |
    // ((c & 0x800) << 4), two elements per 32-bit word (SpecPilot digest,
    // "Reasons": the planes are rebuilt to BF16 inside the GEMM). For a group
    // of 8 elements, X and Y hold p0 | p1 << 4 of the even and odd nibble
    // slots, Z0 and Z1 the p2 nibbles; one byte permute per output word puts
    // the two elements' codes into its 16-bit lanes.
    const int cw = warp < 4 ? warp - 2 : warp - 6;   // 0 .. NCONV - 1
    const int ct = cw * 32 + lane;
    // thread ct converts the 8-element groups g = ct mod 16 (a 4-byte word of
    // each plane, a 16-byte chunk of bf16) of rows r = ct / 16 + 2 NCONV k; a plane
    // tile row is 64 bytes at r * 64 (the two 64-row halves are 4096 bytes apart)
    const int g = ct & 15, r0 = ct >> 4;
    const int q = g >> 3, c16 = g & 7;
    // grouped W12: each 64-row half of the tile has its row block's base, and the
    // unit's escapes are written over the rebuilt elements by the thread that
    // rebuilt them (row r0 (mod 2 NCONV), group g), so no barrier is needed
    const bool grouped = a.w12_bases != nullptr;
    const int nrb = (a.n_rows + 63) / 64;
    // unit i's row-block bases and escape ranges, requested one unit ahead
    auto unit_meta = [&](long long i, uint32_t* b2h, int* eo, int* ee) {
      b2h[0] = b2h[1] = (static_cast<uint32_t>(a.w12_base) << 7) * 0x10001u;
      eo[0] = eo[1] = ee[0] = ee[1] = 0;
      if (!grouped || i >= NU) return;
      long long t;
      int kb;
      W.at(i, t, kb);
      const int nt = static_cast<int>(t / a.m_tiles);
      const int rh0 = a.pair == kPairSwiglu ? nt * (kGemmBN / 2) : nt * kGemmBN;
      const int rh1 = a.pair == kPairSwiglu ? a.ffn + nt * (kGemmBN / 2) : rh0 + kGemmBN / 2;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int rb = (hh ? rh1 : rh0) / 64;
        if (rb < nrb) {
          b2h[hh] = (static_cast<uint32_t>(__ldg(a.w12_bases + rb)) << 7) * 0x10001u;
          const long long tile = static_cast<long long>(rb) * a.w12_kt + kb;
          eo[hh] = __ldg(a.w12_esc_off + tile);
          ee[hh] = __ldg(a.w12_esc_off + tile + 1);
        }
      }
    };
    uint32_t nb2[2];
    int neo[2], nee[2];
    unit_meta(0, nb2, neo, nee);
    int stage = 0;
    uint32_t phase = 0;
    int ai = 0;
    for (long long i = 0; i < NU; ++i, ++ai) {
      const uint32_t b2h[2] = {nb2[0], nb2[1]};
      const int eo[2] = {neo[0], neo[1]}, ee[2] = {nee[0], nee[1]};
      unit_meta(i + 1, nb2, neo, nee);
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait(full + stage, phase, abort_flag, kWaitNs) &&
             mbar_wait(aempty + ai % kW12Ring, ((ai / kW12Ring) & 1) ^ 1u, abort_flag, kWaitNs);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      const uint8_t* pw = smem + static_cast<size_t>(stage) * STAGE + r0 * 64 + g * 4;
      uint8_t* aw = aring + (ai % kW12Ring) * NSUB * kABytes + q * kABytes;
#pragma unroll 2
      for (int r = r0; r < 128; r += NCONV * 2) {
        const int po = (r - r0) * 64;
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(pw + po);
        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(pw + 8192 + po);
        const uint32_t w2 = *reinterpret_cast<const uint32_t*>(pw + 16384 + po);
        // slots 0,2,4,6 hold elements 0,4,1,5; slots 1,3,5,7 hold 2,6,3,7
        const uint32_t X = (w0 & 0x0F0F0F0Fu) | ((w1 << 4) & 0xF0F0F0F0u);
        const uint32_t Y = ((w0 >> 4) & 0x0F0F0F0Fu) | (w1 & 0xF0F0F0F0u);
        // p2 nibbles with the sign moved from bit 3 to bit 7 of the byte: after the
        // byte permute a lane holds (c & 0x7FF) | (sign << 15)
        const uint32_t Z0 = (w2 & 0x07070707u) | ((w2 << 4) & 0x80808080u);
        const uint32_t Z1 = ((w2 >> 4) & 0x07070707u) | (w2 & 0x80808080u);
        const uint32_t cw4[4] = {__byte_perm(X, Z0, 0x6240), __byte_perm(Y, Z1, 0x6240), __byte_perm(X, Z0, 0x7351),
                                 __byte_perm(Y, Z1, 0x7351)};  // elements (0,1) (2,3) (4,5) (6,7)
        // ((c & 0x7FF) + (base << 7)) | (sign << 15) per 16-bit lane is one add: the
        // exponent sum base + e <= 254 (any code that packing accepted) stays below bit 15
        uint32_t o[4];
        const uint32_t b2 = r < 64 ? b2h[0] : b2h[1];
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = cw4[j] + b2;
        *reinterpret_cast<uint4*>(aw + r * 128 + ((c16 ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
        for (int e = eo[hh]; e < ee[hh]; ++e) {
          const uint32_t ent = __ldg(a.w12_esc + e);
          const int r = hh * 64 + static_cast<int>(ent >> 23 & 63u), col = static_cast<int>(ent >> 16 & 127u);
          if (r % (NCONV * 2) == r0 && (col >> 3) == g)
            *reinterpret_cast<uint16_t*>(aw + r * 128 + ((c16 ^ (r & 7)) << 4) + (col & 7) * 2) =
                static_cast<uint16_t>(ent & 0xFFFFu);
        }
      fence_proxy_async_smem();  // the MMAs read the tile through the async proxy
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(afull + ai % kW12Ring);
        mbar_arrive(empty + stage);  // planes consumed
      }
      if (++stage == S) {
        stage = 0;
        phase ^= 1u;
      }
    }
  } else if (warp >= 4 && warp < 4 + EPT / 32) {
    // ------------------------------------------------------------ epilogue
    // Warpgroup A (warps 4-7) reads the accumulators out of TMEM (warp w reads
    // lanes 32 (w % 4) ..); with two warpgroups both share the reduction (16
    // columns each) and the tile epilogue.
    pdl_wait();  // reads what earlier kernels wrote (h, norm statistics, row maps)
    pdl_trigger();
    const int et2 = threadIdx.x - 128;          // 0 .. EPT - 1
    const bool grpA = et2 < 128;
    const int et = et2 & 127;                   // tile row
    // per-token data of the whole launch, while the weights stream in
    const TokData* td = !CL && a.M <= kTokMax ? tok : nullptr;
    if (td)
      for (int m = et2; m < a.M; m += EPT) token_data(a.epi, m, tok->rstd[m], tok->pos[m], tok->kv[m]);
    if (CL) {
      // the cluster split has one token tile (M <= NT <= 64), so this rank's tokens are the
      // same for every tile: their per-token data once, into the epilogue's scratch
      const int mt0 = a.M < NT ? a.M : NT;
      const int sl = ((mt0 + CS - 1) / CS + 3) / 4 * 4;
      const int c0 = rank * sl, c1 = c0 + sl < mt0 ? c0 + sl : mt0;
      for (int c = et2; c < c1 - c0; c += EPT) token_data(a.epi, c0 + c, esm->rstd[c], esm->pos[c], esm->kv[c]);
    }
    auto sync = [] { named_bar(1, EPT); };
    sync();
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const long long slot0_tile = NU > 0 ? (W.u0 / a.kb) : 0;
    int seg = 0;
    for (long long i = 0; i < NU;) {
      const long long iend = W.seg_end(i);
      long long t;
      int kb_first;
      W.at(i, t, kb_first);
      const int nt = static_cast<int>(t / a.m_tiles), mt = static_cast<int>(t - (long long)nt * a.m_tiles);
      const int m_base = mt * NT;
      const int mtot = a.M - m_base < NT ? a.M - m_base : NT;
      const int b = seg & 1;
      // the hand-off of the CTA's last tile goes into the timeline
      unsigned long long* const trec = rec && iend == NU && et2 == 0 ? rec : nullptr;
      if (CL) {
        // the epilogue's global inputs of this rank's tokens, into shared memory while the tile accumulates
        const int sl = ((mtot + CS - 1) / CS + 3) / 4 * 4;
        const int c0 = rank * sl, c1 = c0 + sl < mtot ? c0 + sl : mtot;
        if (c0 < c1) stage_epilogue_inputs(a, nt, m_base + c0, c1 - c0, Es, *esm, nullptr, et2, EPT);
      }
      // one thread waits and broadcasts, so all threads agree on the outcome
      if (et2 == 0) *s_flag = mbar_wait(acc_full + b, (seg >> 1) & 1, abort_flag, kWaitNs) ? 1 : 0;
      sync();
      const bool ok = *s_flag != 0;
      sync();
      if (!ok) break;
      tc_fence_after();
      trace_mark(trec, 7);
      if constexpr (CL) {
        // ---- cluster split (one tile per cluster), reduce-scatter by pushes: every rank
        // stores the token slice [c0_r, c1_r) of its partial straight into rank r's shared
        // memory (st.async, counted on r's rx_full); rank r sums the CS slices in rank
        // order from its own shared memory and runs their epilogue
        const int sl = ((mtot + CS - 1) / CS + 3) / 4 * 4;
        const int c0 = rank * sl, c1 = c0 + sl < mtot ? c0 + sl : mtot;
        const int ncol4 = c1 > c0 ? (c1 - c0 + 3) / 4 * 4 : 0;  // columns this rank receives
        if (et2 == 0 && ncol4 > 0)
          mbar_arrive_expect_tx(rx_full, static_cast<uint32_t>(CS * kGemmBN * ncol4 * 4));
        if (grpA) {
          float v[2][32];
#pragma unroll
          for (int ch = 0; ch < NT / 32; ++ch)
            if (ch * 32 < mtot) {
              tmem_ld32(tmem + lane_base + b * ACC + ch * 32, v[ch]);
              if (FUSE) {  // the lo plane's products
                float w[32];
                tmem_ld32(tmem + lane_base + b * ACC + NT + ch * 32, w);
#pragma unroll
                for (int k = 0; k < 32; ++k) v[ch][k] += w[k];
              }
            }
          tc_fence_before();
          mbar_arrive(acc_empty + b);
          // token group c .. c + 3 (c a multiple of 4) goes to rank c / sl, slot (c % sl) / 4
          const uint32_t rx = smem_u32(Rx) + 4u * ((rank * kGemmBN + et) * SL), rxf = smem_u32(rx_full);
#pragma unroll
          for (int ch = 0; ch < NT / 32; ++ch)
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int c = ch * 32 + 4 * q;
              if (c < mtot) {
                const int r = c / sl;
                st_async_v4(mapa_shared(rx, static_cast<uint32_t>(r)) + 4u * (c - r * sl),
                            make_float4(v[ch][4 * q], v[ch][4 * q + 1], v[ch][4 * q + 2], v[ch][4 * q + 3]),
                            mapa_shared(rxf, static_cast<uint32_t>(r)));
              }
            }
        }
        trace_mark(trec, 8);
        if (ncol4 > 0) {
          if (et2 == 0) *s_flag = mbar_wait_cluster(rx_full, 0u, abort_flag, kWaitNs);
          sync();
          const bool okr = *s_flag != 0;
          sync();
          if (!okr) break;
          trace_mark(trec, 9);
          // thread (row et, sub) sums the 4-column groups sub, sub + NSUBT, .. in rank order
          constexpr int NSUBT = EPT / 128;
          const int sub = et2 >> 7;
          for (int g = sub; g * 4 < ncol4; g += NSUBT) {
            float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int r = 0; r < CS; ++r) {
              const float4 q = *reinterpret_cast<const float4*>(Rx + (r * kGemmBN + et) * SL + 4 * g);
              s4.x += q.x;
              s4.y += q.y;
              s4.z += q.z;
              s4.w += q.w;
            }
            Ys[et * YLD + 4 * g] = s4.x;
            Ys[et * YLD + 4 * g + 1] = s4.y;
            Ys[et * YLD + 4 * g + 2] = s4.z;
            Ys[et * YLD + 4 * g + 3] = s4.w;
          }
          trace_mark(trec, 13);
          sync();
          trace_mark(trec, 10);
          epilogue_tile(a, nt, Ys, YLD, m_base + c0, c1 - c0, et2, EPT, *esm, nullptr, sync, Es, true);
          sync();
          trace_mark(trec, 11);
        }
      } else {
        // ---- stream-K: partials through global memory, summed in token slices
        const bool own = t >= TSK;  // the CTA's own whole tile
        const int cf = own ? c : cta_of_unit(t * a.kb, USK, P), cl = own ? c : cta_of_unit((t + 1) * a.kb - 1, USK, P);
        const bool alone = cf == cl;
        const int slot = t == slot0_tile ? 0 : 1;
        // partial tiles are column-major ([token][tile row]) so that a warp's
        // stores and the reducer's loads are 128-byte coalesced
        float* mine = a.partials + (static_cast<size_t>(c) * 2 + slot) * kGemmBN * NT + et;
        for (int ch = 0; ch * 32 < mtot; ++ch) {
          float v[32];
          if (grpA) {
            tmem_ld32(tmem + lane_base + b * ACC + ch * 32, v);
            if (FUSE) {  // the lo plane's products
              float w[32];
              tmem_ld32(tmem + lane_base + b * ACC + NT + ch * 32, w);
#pragma unroll
              for (int k = 0; k < 32; ++k) v[k] += w[k];
            }
          }
          if (alone) {
            if (grpA) {
#pragma unroll
              for (int k = 0; k < 32; ++k) Ys[et * kYsLd + k] = v[k];
            }
            sync();
            epilogue_tile(a, nt, Ys, kYsLd, m_base + ch * 32, mtot - ch * 32 < 32 ? mtot - ch * 32 : 32, et2, EPT,
                          *esm, td, sync, nullptr);
            sync();
            trace_mark(trec, 11);
          } else if (grpA) {
#pragma unroll
            for (int k = 0; k < 32; ++k)  // (only the tile's tokens: the reducers read no others)
              if (ch * 32 + k < mtot) __stcg(mine + (ch * 32 + k) * kGemmBN, v[k]);
          }
        }
        if (grpA) {
          tc_fence_before();
          mbar_arrive(acc_empty + b);
        }
        if (!alone) {
          // Hand-off. A tile of one token chunk (at most 32 tokens) is summed by the
          // last contributor to arrive, so the others leave at once. A wider tile is
          // shared by its participants, the contributors whose ranges end inside it
          // (the tile is their last work): cf .. lp, where lp = cl unless cl's range
          // runs on past the tile. Once every partial is in, each sums its own token
          // slice, so no single SM reads the whole tile's partials.
          const bool share = mtot > 32;
          const int ncon = cl - cf + 1;
          const long long tend = (t + 1) * a.kb;
          const int lp = static_cast<long long>(cl + 1) * USK / P <= tend ? cl : cl - 1;
          const bool part = share && static_cast<long long>(c + 1) * USK / P <= tend;
          const int npart = share ? lp - cf + 1 : 1;
          const int ws = ((mtot + npart - 1) / npart + 3) / 4 * 4;
          const int s0 = share ? (c - cf) * ws : 0, s1 = share ? (s0 + ws < mtot ? s0 + ws : mtot) : mtot;
          if (!share || part) epilogue_prefetch(a, nt, m_base + s0, s1 - s0 < 32 ? s1 - s0 : 32, et, td);
          __threadfence();
          sync();
          trace_mark(trec, 8);
          if (share) {
            if (et2 == 0) {
              atomicAdd(a.counters + t, 1u);
              *s_flag = part ? wait_count(a.counters + t, static_cast<unsigned>(ncon), abort_flag, kWaitNs) : 0;
            }
          } else if (et2 == 0) {
            *s_flag = atomicAdd(a.counters + t, 1u) == static_cast<unsigned>(ncon - 1) ? 1 : 0;
          }
          sync();
          const bool reduce = *s_flag != 0;
          sync();
          trace_mark(trec, 9);
          if (reduce) {
            __threadfence();
            // the contributors' slots, in CTA order (a fixed summation order): a
            // tile is the first tile (slot 0) of every contributor after cf, and of
            // cf when cf's range starts at the tile's first unit
            const int sl_first = static_cast<long long>(cf) * USK / P == t * a.kb ? 0 : 1;
            constexpr int RW = 32 / (EPT / 128);  // columns of a chunk each warpgroup sums
            const int col0 = grpA ? 0 : RW;
            constexpr int NB = W12 ? 1 : 4;  // contributors whose loads are in flight together
            for (int cc = s0; cc < s1; cc += 32) {
              const int cn = s1 - cc < 32 ? s1 - cc : 32;
              // the next chunk's epilogue inputs into L1 while this chunk's partials load
              if (cc + 32 < s1) epilogue_prefetch(a, nt, m_base + cc + 32, s1 - cc - 32 < 32 ? s1 - cc - 32 : 32, et, td);
              float sm_[RW];
#pragma unroll
              for (int k = 0; k < RW; ++k) sm_[k] = 0.f;
              for (int j0 = 0; j0 < ncon; j0 += NB) {
                float v[NB][RW];
#pragma unroll
                for (int jj = 0; jj < NB; ++jj) {
                  const int j = j0 + jj;
                  if (j < ncon) {
                    const int sl = j == 0 ? sl_first : 0;
                    const float* src = a.partials + (static_cast<size_t>(cf + j) * 2 + sl) * kGemmBN * NT + et;
#pragma unroll
                    for (int k = 0; k < RW; ++k)
                      v[jj][k] = col0 + k < cn ? __ldcg(src + (cc + col0 + k) * kGemmBN) : 0.f;
                  }
                }
                // summed in CTA order, whatever the loads' completion order
#pragma unroll
                for (int jj = 0; jj < NB; ++jj)
                  if (j0 + jj < ncon) {
#pragma unroll
                    for (int k = 0; k < RW; ++k) sm_[k] += v[jj][k];
                  }
              }
#pragma unroll
              for (int k = 0; k < RW; ++k) Ys[et * kYsLd + col0 + k] = sm_[k];
              sync();
              trace_mark(trec, 10);
              epilogue_tile(a, nt, Ys, kYsLd, m_base + cc, cn, et2, EPT, *esm, td, sync, nullptr);
              sync();
              trace_mark(trec, 11);
            }
            if (!share) {
              if (et2 == 0) a.counters[t] = 0u;
            } else if (et2 == 0) {
              // the last participant to finish clears the tile's counters for the next launch
              __threadfence();
              unsigned* done = a.counters + static_cast<size_t>(a.n_tiles) * a.m_tiles;
              if (atomicAdd(done + t, 1u) == static_cast<unsigned>(npart - 1)) {
                a.counters[t] = 0u;
                done[t] = 0u;
              }
            }
          }
        }
      }
      ++seg;
      i = iend;
    }
    if (CL && NU > 0 && *abort_flag) {
      // after a timed-out wait: this CTA leaves only once the slices other ranks
      // store into it have landed (bounded); after a normal run they have
      const int mt0 = a.M < NT ? a.M : NT;
      const int sl = ((mt0 + CS - 1) / CS + 3) / 4 * 4;
      if (et2 == 0 && rank * sl < mt0) {
        volatile int never = 0;
        mbar_wait_cluster(rx_full, 0u, &never, kWaitNs);
      }
      sync();
    }
    if (et2 == 0) trace_mark(rec, 5);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TCOLS);
  }
  if (threadIdx.x == 0) {
    if (*abort_flag && a.epi.status) atomicOr(a.epi.status, kStTimeout);
    trace_mark(rec, 6);
  }
}

template <int NT, bool PAIR, bool W12, bool CL>
cudaError_t gemm_tc_launch(const GemmArgs& a, const CUtensorMap& w, const CUtensorMap& x, cudaStream_t s) {
  constexpr int KS = tc_ks_for(NT, PAIR, W12);
  const size_t smem = tc_smem_bytes(NT, PAIR, KS, a.tc_stages, W12, CL ? a.cl_size : 0);
  static bool attr_set[64] = {};  // per device: allow the largest configuration this kernel may use
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<NT, PAIR, W12, CL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget + 2048);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  if (CL) {
    if (a.cl_size < 1 || a.grid_p % a.cl_size) return cudaErrorInvalidValue;
    return launch_k_cluster(gemm_tc_kernel<NT, PAIR, W12, CL>, dim3(a.grid_p), dim3(W12 ? kTcThreadsW12 : kTcThreads),
                            smem, s, a.pdl != 0, a.cl_size, w, x, a);
  }
  return launch_k(gemm_tc_kernel<NT, PAIR, W12, CL>, dim3(a.grid_p), dim3(W12 ? kTcThreadsW12 : kTcThreads), smem, s,
                  a.pdl != 0, w, x, a);
}

// Clusters of `cs` CTAs of this instantiation that can be resident at once (0 on error).
template <int NT, bool PAIR, bool W12, bool CL>
int gemm_tc_max_clusters(int cs, int stages) {
  constexpr int KS = tc_ks_for(NT, PAIR, W12);
  const size_t smem = tc_smem_bytes(NT, PAIR, KS, stages, W12, CL ? cs : 0);
  if (cudaFuncSetAttribute(gemm_tc_kernel<NT, PAIR, W12, CL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBudget + 2048) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs);
  cfg.blockDim = dim3(W12 ? kTcThreadsW12 : kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<NT, PAIR, W12, CL>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace tcg
}  // namespace sv

// Explicit instantiations for token tile NT (one translation unit per NT, so
// the kernel variants compile in parallel). W12 and the cluster split stop at
// 64 columns.
#define SV_GEMM_TC_INSTANTIATE_ONE(NT, PAIR, W12, CL)                                                            \
  template cudaError_t sv::tcg::gemm_tc_launch<NT, PAIR, W12, CL>(const sv::GemmArgs&, const CUtensorMap&,       \
                                                                  const CUtensorMap&, cudaStream_t);             \
  template int sv::tcg::gemm_tc_max_clusters<NT, PAIR, W12, CL>(int, int);
#define SV_GEMM_TC_INSTANTIATE(NT)                \
  SV_GEMM_TC_INSTANTIATE_ONE(NT, true, false, false) \
  SV_GEMM_TC_INSTANTIATE_ONE(NT, false, false, false)
#define SV_GEMM_TC_INSTANTIATE_SMALL(NT)             \
  SV_GEMM_TC_INSTANTIATE_ONE(NT, true, true, false)  \
  SV_GEMM_TC_INSTANTIATE_ONE(NT, false, true, false) \
  SV_GEMM_TC_INSTANTIATE_ONE(NT, true, false, true)  \
  SV_GEMM_TC_INSTANTIATE_ONE(NT, false, false, true) \
  SV_GEMM_TC_INSTANTIATE_ONE(NT, true, true, true)   \
  SV_GEMM_TC_INSTANTIATE_ONE(NT, false, true, true)
