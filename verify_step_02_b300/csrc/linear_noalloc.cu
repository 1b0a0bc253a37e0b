// sv_linear_noalloc: the skinny weight-streaming product of sv_linear for
// callers that cannot allocate device memory. It runs the CUDA-core plan,
// whose K splits meet in distributed shared memory within thread-block
// clusters, so it needs no device scratch at all: no allocation, no shared
// state between calls.
#include <cstring>

#include "internal.h"

namespace {

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
  a.counters = nullptr;  // (the plan keeps its splits within one cluster: no counters, no partials)
  a.partials = nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  a.epi.kind = kEpiStore;
  a.epi.y = y;
  a.epi.ldy = N;
  const cudaError_t e = launch_gemm(a, s);
  if (e != cudaSuccess) return reject(SV_ERR_CUDA, cudaGetErrorString(e));
  return SV_OK;
}
