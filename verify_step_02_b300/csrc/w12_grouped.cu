// Grouped W12: the W12 planes (three 4-bit planes of 12-bit codes, rebuilt to
// bf16 inside the matrix kernels; SpecPilot digest, "Reasons") with one
// exponent base per 64-row block instead of one per tensor, plus a list of
// escapes for the elements the block's 16-binade window cannot hold (zeros,
// subnormals, inf/NaN, and exponents below the window). Real weights (e.g.
// N(0, sigma) with exact zeros) then round-trip bit-exactly.
//
//   base[rb] = max(1, (max E over the block's normal elements) - 15), or 1
//   escape  <=> the element is not a normal number, or E < base[rb]
//   code    = s << 11 | (E - base[rb]) << 7 | m, and 0 for an escape
//   escapes of plane tile (rb, kt) (64 rows x 128 columns, tiles in order
//   rb * KT + kt, row-major within a tile) are esc[off[i] .. off[i + 1]),
//   entry = row in block << 23 | column in tile << 16 | bf16 pattern.
#include "device_util.cuh"
#include "internal.h"

namespace sv {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ int bf16_exponent(uint16_t b) { return (b >> 7) & 0xFF; }
__device__ __forceinline__ bool w12g_escape(uint16_t b, int base) {
  const int e = bf16_exponent(b);
  return e < 1 || e > 254 || e < base;
}

// One CTA per 64-row block: its base.
__global__ void __launch_bounds__(kThreads) w12g_bases_kernel(const uint16_t* b, long long rows, long long cols,
                                                              uint8_t* bases) {
  __shared__ int red[kThreads / 32];
  const long long r0 = static_cast<long long>(blockIdx.x) * 64;
  const long long r1 = r0 + 64 < rows ? r0 + 64 : rows;
  int mx = 0;
  for (long long i = threadIdx.x; i < (r1 - r0) * cols; i += kThreads) {
    const int e = bf16_exponent(b[r0 * cols + i]);
    if (e >= 1 && e <= 254) mx = max(mx, e);
  }
  for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    int m = 0;
    for (int w = 0; w < kThreads / 32; ++w) m = max(m, red[w]);
    bases[blockIdx.x] = static_cast<uint8_t>(m == 0 ? 1 : max(1, m - 15));
  }
}

// Element (r, c) of plane tile `tile`, or false past the matrix.
__device__ __forceinline__ bool tile_element(int tile, int kt_n, int idx, long long rows, long long cols, long long& row,
                                             long long& col) {
  const int rb = tile / kt_n, kt = tile - rb * kt_n;
  row = static_cast<long long>(rb) * 64 + (idx >> 7);
  col = static_cast<long long>(kt) * 128 + (idx & 127);
  return row < rows && col < cols;
}

// One CTA per plane tile: its number of escapes.
__global__ void __launch_bounds__(kThreads) w12g_count_kernel(const uint16_t* b, long long rows, long long cols,
                                                              int kt_n, const uint8_t* bases, int* cnt) {
  __shared__ int red[kThreads / 32];
  const int tile = blockIdx.x, base = bases[tile / kt_n];
  int n = 0;
  for (int idx = threadIdx.x; idx < 64 * 128; idx += kThreads) {
    long long row, col;
    if (tile_element(tile, kt_n, idx, rows, cols, row, col) && w12g_escape(b[row * cols + col], base)) ++n;
  }
  for (int o = 16; o; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = n;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int w = 0; w < kThreads / 32; ++w) t += red[w];
    cnt[tile] = t;
  }
}

// One CTA per plane tile: its escapes in row-major order from esc[off[tile]].
__global__ void __launch_bounds__(kThreads) w12g_escape_kernel(const uint16_t* b, long long rows, long long cols,
                                                               int kt_n, const uint8_t* bases, const int* off,
                                                               uint32_t* esc) {
  __shared__ int warp_n[kThreads / 32];
  const int tile = blockIdx.x, base = bases[tile / kt_n];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int run = off[tile];
  for (int i0 = 0; i0 < 64 * 128; i0 += kThreads) {
    const int idx = i0 + threadIdx.x;
    long long row, col;
    uint16_t v = 0;
    bool f = false;
    if (tile_element(tile, kt_n, idx, rows, cols, row, col)) {
      v = b[row * cols + col];
      f = w12g_escape(v, base);
    }
    const uint32_t bal = __ballot_sync(0xffffffffu, f);
    if (lane == 0) warp_n[warp] = __popc(bal);
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      before += w < warp ? warp_n[w] : 0;
      total += warp_n[w];
    }
    if (f) {
      const int k = run + before + __popc(bal & ((1u << lane) - 1u));
      esc[k] = static_cast<uint32_t>((idx >> 7) << 23 | (idx & 127) << 16 | v);
    }
    run += total;
    __syncthreads();
  }
}

// Plane bytes as w12_pack_kernel writes them, with the row block's base and
// zero codes for escapes.
__device__ __forceinline__ unsigned w12g_code(uint16_t b, int base) {
  if (w12g_escape(b, base)) return 0u;
  return (unsigned)(b >> 15) << 11 | (unsigned)(bf16_exponent(b) - base) << 7 | (b & 0x7Fu);
}

__global__ void w12g_pack_kernel(const uint16_t* b, long long rows, long long cols, int kt_n, long long plane_bytes,
                                 const uint8_t* bases, uint8_t* planes) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= plane_bytes) return;
  const long long tile = idx >> 12;
  const int within = static_cast<int>(idx & 4095);
  const long long rt = tile / kt_n, kt = tile - rt * kt_n;
  const long long row = rt * 64 + (within >> 6);
  const int cb = within & 63;
  const long long g0 = kt * 128 + (cb >> 2) * 8;
  const int s0 = 2 * (cb & 3);
  // nibble slot s holds element 2s (s < 4) or 2(s - 4) + 1 of its group of 8
  const long long k0 = g0 + (s0 < 4 ? 2 * s0 : 2 * s0 - 7), k1 = g0 + (s0 + 1 < 4 ? 2 * s0 + 2 : 2 * s0 - 5);
  const int base = bases[rt];
  const unsigned c0 = row < rows && k0 < cols ? w12g_code(b[row * cols + k0], base) : 0u;
  const unsigned c1 = row < rows && k1 < cols ? w12g_code(b[row * cols + k1], base) : 0u;
#pragma unroll
  for (int p = 0; p < 3; ++p)
    planes[p * plane_bytes + idx] = static_cast<uint8_t>(((c0 >> (4 * p)) & 0xFu) | ((c1 >> (4 * p)) & 0xFu) << 4);
}

__global__ void w12g_unpack_kernel(const uint8_t* planes, const uint8_t* bases, long long rows, long long cols,
                                   int kt_n, long long plane_bytes, uint16_t* out) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= rows * cols) return;
  const long long row = idx / cols, k = idx - row * cols;
  const int e = static_cast<int>(k & 7), slot = (e & 1) ? 4 + (e >> 1) : (e >> 1);
  const long long byte = (((row >> 6) * kt_n + (k >> 7)) << 12) + (row & 63) * 64 + ((k & 127) >> 3) * 4 + (slot >> 1);
  const int sh = (slot & 1) * 4;
  const unsigned c = ((planes[byte] >> sh) & 0xFu) | ((planes[plane_bytes + byte] >> sh) & 0xFu) << 4 |
                     ((planes[2 * plane_bytes + byte] >> sh) & 0xFu) << 8;
  out[idx] = static_cast<uint16_t>(((c & 0x7FFu) + ((unsigned)bases[row >> 6] << 7)) | ((c & 0x800u) << 4));
}

// One CTA per plane tile: write its escapes' exact patterns.
__global__ void w12g_patch_kernel(const int* off, const uint32_t* esc, long long cols, int kt_n, uint16_t* out) {
  const int tile = blockIdx.x, rb = tile / kt_n, kt = tile - rb * kt_n;
  for (int i = off[tile] + threadIdx.x; i < off[tile + 1]; i += blockDim.x) {
    const uint32_t v = esc[i];
    const long long row = static_cast<long long>(rb) * 64 + (v >> 23 & 63), col = static_cast<long long>(kt) * 128 + (v >> 16 & 127);
    out[row * cols + col] = static_cast<uint16_t>(v & 0xFFFFu);
  }
}

}  // namespace

cudaError_t launch_w12g_bases(const uint16_t* bf16, long long rows, long long cols, uint8_t* bases, cudaStream_t s) {
  w12g_bases_kernel<<<(unsigned)((rows + 63) / 64), kThreads, 0, s>>>(bf16, rows, cols, bases);
  return cudaGetLastError();
}

cudaError_t launch_w12g_count(const uint16_t* bf16, long long rows, long long cols, const uint8_t* bases, int* cnt,
                              cudaStream_t s) {
  const int kt_n = static_cast<int>((cols + 127) / 128);
  w12g_count_kernel<<<(unsigned)(((rows + 63) / 64) * kt_n), kThreads, 0, s>>>(bf16, rows, cols, kt_n, bases, cnt);
  return cudaGetLastError();
}

cudaError_t launch_w12g_pack(const uint16_t* bf16, long long rows, long long cols, const uint8_t* bases,
                             const int* off, uint8_t* planes, uint32_t* esc, cudaStream_t s) {
  const int kt_n = static_cast<int>((cols + 127) / 128);
  const long long n = w12_plane_bytes(rows, cols);
  w12g_pack_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(bf16, rows, cols, kt_n, n, bases, planes);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess && esc) {
    w12g_escape_kernel<<<(unsigned)(((rows + 63) / 64) * kt_n), kThreads, 0, s>>>(bf16, rows, cols, kt_n, bases,
                                                                                    off, esc);
    e = cudaGetLastError();
  }
  return e;
}

cudaError_t launch_w12g_unpack(const uint8_t* planes, const uint8_t* bases, const int* off, const uint32_t* esc,
                               long long rows, long long cols, uint16_t* out, cudaStream_t s) {
  const int kt_n = static_cast<int>((cols + 127) / 128);
  const long long n = rows * cols;
  w12g_unpack_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(planes, bases, rows, cols, kt_n,
                                                                  w12_plane_bytes(rows, cols), out);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) {
    w12g_patch_kernel<<<(unsigned)(((rows + 63) / 64) * kt_n), 128, 0, s>>>(off, esc, cols, kt_n, out);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace sv
