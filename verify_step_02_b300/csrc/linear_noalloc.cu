// sv_linear_noalloc: the skinny weight-streaming product of sv_linear for
// callers that cannot allocate device memory. Its split-K scratch (partial
// tiles and tile counters) lives in one file-scope device array that every
// GPU loading this library holds until the process exits.
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB

// Device-side scratch. In host code this name is only a host stand-in for the
// symbol: kernels get the device address that cudaGetSymbolAddress returns.
static __device__ __align__(256) unsigned char g_linear_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_linear_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

sv_status reject(sv_status st, const char* msg) {
  sv::record_error(msg);
  return st;
}

}  // namespace

extern "C" sv_status sv_linear_noalloc(int32_t wdtype, const sv_matrix* w, int32_t N, int32_t K, const void* x,
                                       int32_t x_planes, int32_t M, float* y, void* stream) {
  using namespace sv;
  if (!w || !w->data || !x || !y) return reject(SV_ERR_INVALID_ARG, "NULL argument");
  if (wdtype < SV_F32 || wdtype > SV_W12) return reject(SV_ERR_INVALID_ARG, "bad wdtype");
  if (x_planes != 1 && !(x_planes == 2 && wdtype != SV_F32))
    return reject(SV_ERR_INVALID_ARG, "x_planes must be 1, or 2 for bf16/W12 weights");
  if (M < 1 || M > 4096 || N < 1 || K < 16 || K % 16) return reject(SV_ERR_INVALID_ARG, "need 1<=M<=4096, N>=1, K%16==0");
  if (wdtype == SV_W12 && !w->row_bases && (w->base < 1 || w->base > 254))
    return reject(SV_ERR_INVALID_ARG, "bad W12 base");
  if (wdtype == SV_W12 && w->row_bases && !w->esc_off) return reject(SV_ERR_INVALID_ARG, "grouped W12 without esc_off");
  int dev = 0, sm = 148;
  if (cudaGetDevice(&dev) != cudaSuccess) return reject(SV_ERR_CUDA, "cudaGetDevice failed");
  cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev);
  GemmArgs a;
  memset(&a, 0, sizeof a);
  a.wdtype = wdtype;
  a.w = w->data;
  a.w12_base = w->base;
  a.w12_bases = w->row_bases;
  a.w12_esc_off = w->esc_off;
  a.w12_esc = w->esc;
  a.w12_kt = (K + 127) / 128;
  a.w12_plane = w12_plane_bytes(N, K);
  a.n_rows = N;
  a.x = x;
  a.x_kind = wdtype == SV_F32 ? kXF32 : (x_planes == 2 ? kXPair : kXBf16);
  a.x_plane = (long long)M * K;
  plan_gemm(a, M, N, K, kPairNone, sm);
  const size_t cnt_bytes = ((size_t)a.n_tiles * a.m_tiles * sizeof(unsigned) + 255) & ~(size_t)255;
  const size_t need = cnt_bytes + gemm_partial_floats(a) * sizeof(float);
  if (need > kScratchBytes) {
    char buf[160];
    snprintf(buf, sizeof buf, "this shape needs %zu bytes of scratch, more than the %zu-byte static scratch", need,
             kScratchBytes);
    return reject(SV_ERR_INVALID_ARG, buf);
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return reject(SV_ERR_CUDA, cudaGetErrorString(e));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the tile counters must start at zero whatever an earlier call left behind
  e = cudaMemsetAsync(scratch, 0, cnt_bytes, s);
  if (e != cudaSuccess) return reject(SV_ERR_CUDA, cudaGetErrorString(e));
  a.counters = static_cast<unsigned*>(scratch);
  a.partials = reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) + cnt_bytes);
  a.epi.kind = kEpiStore;
  a.epi.y = y;
  a.epi.ldy = N;
  e = launch_gemm(a, s);
  if (e != cudaSuccess) return reject(SV_ERR_CUDA, cudaGetErrorString(e));
  return SV_OK;
}
