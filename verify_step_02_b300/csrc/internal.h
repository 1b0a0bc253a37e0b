// Internal declarations shared by the kernels and the host engine of libsv.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sv.h"

namespace sv {

constexpr int kMaxBatch = 1024;       // largest batch a verify may take
constexpr int kMaxGamma = 255;        // largest block beyond the anchor (drafts, or prefill rows)
constexpr int kGemmBN = 128;          // weight rows per GEMM tile (both GEMM paths)
constexpr int kFmaBM = 32;            // tokens per FMA GEMM tile
constexpr int kFmaKC = 32;            // K step of the FMA GEMM
constexpr int kFmaMaxCluster = 8;     // FMA GEMM: K splits reduced within one cluster (portable size)

// Device status word bits (sv_model_sync_status).
// kStBadPos and kStNoPage mean the block does not fit the request's KV capacity
// (a position reaches max_seq_len, or a page index is past the page table);
// the others are bad inputs or a timed-out wait.
enum : uint32_t {
  kStBadToken = 1u,
  kStBadPage = 2u,
  kStBadDraftProb = 4u,
  kStTimeout = 8u,
  kStBadPos = 16u,
  kStNoPage = 32u,
  kStBadTree = 64u,       // a token tree node whose parent does not precede it
};

// Token trees (sv_verify_tree): nodes per request, so that a node's ancestors
// fit one 64-bit mask.
constexpr int kMaxTreeNodes = 64;

enum EpiKind : int {
  kEpiStore = 0,   // y[m][n] = value                                  (sv_linear)
  kEpiQkv = 1,     // RoPE on q,k; q -> q_out; k,v -> paged cache      (QKV projection)
  kEpiResid = 2,   // h[m][n] += value                                 (O and down projections)
  kEpiSwiglu = 3,  // act[m][f] = SiLU(gate) * up                      (gate|up projection)
  kEpiLogits = 4,  // logits and per-tile (max, argmax)                (LM head)
};

// Row pairing of a GEMM tile. kPairNone: tile rows are W rows nt*BN + t.
// kPairSwiglu: tile rows t < BN/2 are gate rows f0 + t, rows t >= BN/2 the up
// rows ffn + f0 + t - BN/2, with f0 = nt * BN/2; the epilogue then sees the
// gate and up value of a feature in the same tile.
enum PairKind : int { kPairNone = 0, kPairSwiglu = 1 };

enum XKind : int { kXF32 = 0, kXBf16 = 1, kXPair = 2 };

// Activations that feed a matrix product ("x tensors": the normed residual,
// the attention output, the SwiGLU product) are float32 for float32 models.
// For bf16/W12 models they are a pair of bf16 planes, hi = bf16(x) and
// lo = bf16(x - hi), so that x = hi + lo to about 16 significant bits: the
// tensor-core product then runs on bf16 operands (hi and lo rows of one B
// tile) while keeping the activations near float32. A pair tensor stores hi
// at element i and lo at element plane + i.
struct Epi {
  int kind;
  int x_pair;              // x outputs (SwiGLU product) as hi/lo pairs (else float32)
  int kv_bf16;             // KV cache stored as bf16 (else float32)
  // kEpiStore
  float* y;
  int ldy;
  // kEpiQkv
  const int* row_req;      // [M] request of each row
  const int* row_pos;      // [M] absolute position of each row (RoPE)
  const int* row_slot;     // [M] KV slot of each row (token tree: C + node), or nullptr: the position
  const float2* rope;      // [max_seq_len][head_dim/2] (cos, sin)
  int n_heads, n_kv_heads, head_dim;
  float* q_out;            // [M][n_heads*head_dim], float32
  void* k_cache;           // layer's K pool [n_pages][n_kv][page_size][head_dim]
  void* v_cache;
  const int* page_table;
  int max_pages;
  int page_size;
  int n_pages;
  unsigned* status;
  // RMSNorm folded into the projections: the x tensors of the QKV, gate|up and
  // LM-head products hold h * gain (no 1/rms); their epilogues multiply each
  // token's results by rsqrt(sum_i ss_in[m][i] / d_model + eps), the sums of
  // squares that the producer of h left per 128-column tile.
  const float* ss_in;      // [M][n_ss] or nullptr (no scaling)
  int n_ss;                // ceil(d_model / 128)
  int d_model;
  float eps;
  // kEpiResid: h += value; then x_out = h * next_gain and ss_out[m][tile] = sum of h^2
  float* h;
  int ldh;
  const void* next_gain;   // [d_model], bf16 when gain_bf16 else float32; nullptr: no x_out
  int gain_bf16;
  void* x_out;             // x tensor [M][d_model] (float32 or hi/lo pair, x_pair)
  long long x_out_plane;
  float* ss_out;           // [M][n_ss]
  // kEpiQkv: q for the tensor-core attention as hi/lo bf16 planes, pre-scaled
  void* q_pair;            // [2][M][n_heads*head_dim] or nullptr (float32 q_out)
  long long q_plane;
  float q_scale;
  // kEpiSwiglu
  void* act;
  long long act_plane;     // element offset of the lo plane (x_pair)
  int ffn;
  // kEpiLogits
  float* logits;           // [M][vocab] or nullptr
  float2* argmax_part;     // [M][n_tiles]: (max value, index as float bits)
  int vocab;
};

// Per-token scratch of a GEMM tile epilogue (shared memory).
struct EpiSmem {
  float rstd[32];
  int pos[32];
  long long kv[32];        // page-pool row of the token's slot for kv head 0, or -1
  float red[4][32];
  int redi[4][32];
  float gain[kGemmBN];     // the tile rows' next-norm gain, when staged (stage_epilogue_inputs)
};

// Per-token epilogue data of a whole launch (block rows m < 256), computed once
// per CTA while the weights stream (tensor path).
constexpr int kTokMax = 256;
struct TokData {
  float rstd[kTokMax];
  int pos[kTokMax];
  long long kv[kTokMax];
};

// Per-CTA timeline (sv_model_set_trace): a traced launch writes one record of
// kTraceWords 64-bit words per CTA; word 0 = kind << 48 | smid << 32 | CTA,
// words 1-6 = %globaltimer (ns) at the kernel's milestones (0 = not reached):
// 1 start, 2 dependency wait returned, 3 first operands landed, 4 last MMA
// issued, 5 epilogue done, 6 exit. The projection kernels add the steps of
// their last tile's hand-off: 7 accumulator ready for the epilogue, 8 partial
// tile stored and signalled, 9 every contributor's partial in place (the
// stream-K participants; cluster split: the slice's owner), 10 the partials of
// the last token chunk summed, 11 tile epilogue done, 12 x tile landed, 13
// the cluster shares summed. The attention adds 7 partial (m, l, O) in shared
// memory, 8 the cluster's partials visible, 9 merge weights computed, 10 last
// K/V stage landed, 11 last softmax done, 12 first scores ready, 13 first
// softmax done, 14 every P·V product complete, 15 the two softmax sets merged.
constexpr int kTraceWords = 16;
enum TraceKind : int { kTrGemm = 1, kTrAttn = 2, kTrMerge = 3, kTrPrep = 4, kTrAccept = 5, kTrGemmFma = 6 };

struct GemmArgs {
  int wdtype;              // SV_F32, SV_BF16, SV_W12
  const void* w;           // weights (W12: planes back to back)
  int w12_base;
  int w12_kt;              // W12: 128-element tiles per row
  long long w12_plane;     // W12 bytes per plane
  const uint8_t* w12_bases;    // grouped W12: base per 64-row block (else nullptr: w12_base)
  const int* w12_esc_off;      // grouped W12: escapes of plane tile i at w12_esc[off[i] .. off[i + 1])
  const uint32_t* w12_esc;     //   (entry: row in block << 23 | column in tile << 16 | bf16 pattern)
  int n_rows;              // rows of W
  int K;
  const void* x;           // activations [M][K]
  int x_kind;              // kXF32, kXBf16 (one bf16 plane) or kXPair (hi/lo bf16 planes)
  long long x_plane;       // element offset of the lo plane (kXPair)
  int M;
  int pair;                // PairKind
  int ffn;                 // kPairSwiglu: gate rows [0, ffn), up rows [ffn, 2 ffn)
  int n_tiles;             // weight tiles
  int m_tiles;             // token tiles
  int k_splits;
  int k_chunk;             // K range of one split (multiple of the K step)
  float* partials;         // split-K partial tiles
  unsigned* counters;      // per tile arrivals (zero between launches)
  // tensor path (gemm_tc.cu)
  int tc_nt;               // token columns of one accumulator (multiple of 32, <= 256)
  int tc_ks;               // K elements per pipeline stage (64, 128 or 256)
  int kb;                  // K blocks of tc_ks per tile
  int grid_p;              // CTAs; CTA c owns units [c U / P, (c+1) U / P), U = n_tiles m_tiles kb
  int tc_stages;           // shared-memory pipeline depth
  int x_lo_row;            // row of the lo plane's first row in the x tensor map (kXPair)
  int pdl;                 // launched as a programmatic dependent of the previous kernel
  int cl_size;             // tensor path, cluster split: CTAs per cluster (0: stream-K)
  int cl_tiles;            // tensor path, cluster split: tiles per cluster
  unsigned long long* trace;  // this launch's per-CTA records, or nullptr
  Epi epi;
};

struct AttnArgs {
  const float* q;          // [M][n_heads*head_dim], float32
  void* out;               // [M][n_heads*head_dim], float32 or hi/lo pair
  long long out_plane;     // element offset of the lo plane (x_pair)
  const void* k_cache;
  const void* v_cache;
  const int* page_table;
  int max_pages;
  int page_size;
  int n_pages;
  const int* seq_len;      // [B] committed context C_r (before commit)
  const int* req_row0;     // [B+1] first block row of each request
  const unsigned long long* row_anc;  // [M] token tree: bit i set = the request's block row i is visible
                                      // (the row's ancestors and itself); nullptr: causal
  int n_heads, n_kv_heads, head_dim;
  int chunk;               // keys per work item
  int max_chunks;
  int max_rows;            // (max_gamma + 1) * group
  int max_seq_len;         // a request whose block ends past this is skipped (status kStBadPos)
  float* partials;         // CUDA-core kernel: chunk partials (max_batch*n_kv*max_chunks*max_rows*(head_dim+2) floats)
  int q_lo_row;            // tensor-core kernel: first token row of q's lo plane in the q tensor map
  unsigned* counters;      // [B*n_kv]
  unsigned* status;
  int x_pair;
  int kv_bf16;
  int pdl;                 // launched as a programmatic dependent of the previous kernel
  int cl_size;             // tensor-core kernel: CTAs per cluster (request, kv head, row tile)
  int cl_count;            // tensor-core kernel: clusters per (request, kv head, row tile), 1 .. kMaxCrossClusters
  float* xpart;            //   cl_count > 1: [item][cluster][128 rows][head_dim] unnormalized partial outputs
  float2* xml;             //   [item][cluster][128 rows] their (max, sum)
  unsigned* xcnt;          //   [item][16] arrivals per (item, rank), zero between launches
  int q_rows;              // tensor-core kernel: block rows per row tile (q_rows * group <= 128)
  int n_row_tiles;         // tensor-core kernel: row tiles per request (ceil((max_gamma + 1) / q_rows))
  int q_copies;            // tensor-core kernel: copies of a tile's query rows in the 128 MMA rows
                           // (1, 2 or 4; q_rows * group * q_copies <= 128), each taking 1/q_copies of the keys
  unsigned long long* trace;  // per-CTA records of the attention launch, or nullptr
};

struct AcceptArgs {
  int B;
  int vocab;
  int gamma_stride;        // 1 + max_gamma (tokens row stride)
  const int* tokens;       // [B][gamma_stride]
  const int* req_row0;     // [B+1]
  int* seq_len;            // [B] in/out
  const float* logits;     // [M][vocab] (sampled)
  const float2* argmax_part;  // [M][n_tiles] (greedy)
  int n_tiles;
  const float* draft_probs;   // [B][max_gamma][vocab]
  int max_gamma;
  float temperature;
  unsigned long long seed;
  const long long* request_ids;
  int* accepted_len;
  int* next_token;
  unsigned* status;
  int pdl;
  int commit_all;          // prefill: every row is committed and next_token = argmax of the last row
  const int* parents;      // token tree: [B][gamma_stride] parent of each node (greedy only), or nullptr
  int* accepted_nodes;     // token tree: [B][gamma_stride] out, the accepted path's nodes, root first
};

// Token tree commit: move the accepted path's keys and values from their
// nodes' slots C + node to C + depth (layers [l0, l0 + n) of one launch).
constexpr int kCompactLayers = 64;
struct CompactArgs {
  int B;
  int gamma_stride;
  const int* seq_len;         // [B] after the commit (C + accepted_len + 1)
  const int* accepted_len;    // [B]
  const int* accepted_nodes;  // [B][gamma_stride]
  const int* page_table;
  int max_pages;
  int page_size;
  int n_pages;
  int row_bytes;              // bytes of one position of one kv head (head_dim x element size)
  int n_kv_heads;
  int n;                      // layers in this launch
  void* k[kCompactLayers];
  void* v[kCompactLayers];
  int pdl;
};

struct PrepParams {
  int pdl;
  int B;
  int M;
  int gamma_stride;
  const int* parents;      // token tree: [B][gamma_stride] parent of each node, or nullptr (chain)
  int req_row0[kMaxBatch + 1];
};

// Set the message sv_last_error() returns on this thread.
void record_error(const char* msg);

// Launch `kern` on stream s; with pdl the launch may overlap the end of the
// previous kernel in the stream (the kernel calls pdl_wait before it reads
// what earlier kernels wrote).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// launch_k with thread-block clusters of `cluster` CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_k_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                             int cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// ---- launchers (defined in the .cu files) ----
cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s);
// Tensor path (tcgen05, gemm_tc.cu) for bf16 weights with bf16 or hi/lo-pair x.
// Weight maps: bf16 [rows][K], 64 x 64 boxes; x maps: bf16 [rows][K], 64 x 32
// boxes; both 128-byte swizzled, zero fill outside the tensor.
// bf16, or W12 whose gate|up row halves are whole plane tiles (ffn % 64 == 0);
// after plan_gemm_tc, tc_stages >= 2 says the token tile fits shared memory.
bool gemm_tc_supported(int wdtype, int pair, int ffn);
void plan_gemm_tc(GemmArgs& a, int M, int n_units, int K, int pair, int sm_count);
size_t gemm_tc_partial_floats(const GemmArgs& a);
size_t gemm_tc_counter_count(const GemmArgs& a);
cudaError_t tc_encode_weight_map(CUtensorMap* m, const void* w, long long rows, int K);
cudaError_t tc_encode_x_map(CUtensorMap* m, const void* x, long long rows, int K);
cudaError_t launch_gemm_tc(const GemmArgs& a, const CUtensorMap& w, const CUtensorMap& x, cudaStream_t s);
// Tensor-core attention (attention_tc.cu) for bf16 KV caches with 16-position
// pages and at most 128 query rows per (request, kv head); KV maps: a layer's
// pool as bf16 [n_pages * n_kv * 16][head_dim], 64 x 16 boxes.
bool attention_tc_supported(int head_dim, int page_size, int max_rows, int max_seq_len);
// CTAs per (request, kv head, row tile) for `items` of them (a power of two, 1 .. 16).
int attention_tc_cluster(long long items, int head_dim, int sm_count);
// Cluster size and clusters per item: several clusters per item only for few items (<= kCrossItems).
constexpr int kCrossItems = 64;
constexpr int kMaxCrossClusters = 4;
void attention_tc_split(long long items, int head_dim, int sm_count, int* cs, int* cc);
cudaError_t tc_encode_kv_map(CUtensorMap* m, const void* pool, int n_pages, int n_kv, int head_dim);
// q as hi/lo bf16 planes [2][m_max][n_heads][head_dim]; box (64 dims, group heads, rows tokens)
cudaError_t tc_encode_q_map(CUtensorMap* m, const void* q, int m_max, int n_heads, int head_dim, int group,
                            int rows);
cudaError_t launch_attention_tc(const AttnArgs& a, int B, const CUtensorMap& q, const CUtensorMap& k,
                                const CUtensorMap& v, cudaStream_t s);
void plan_gemm(GemmArgs& a, int M, int n_rows_or_pairs, int K, int pair, int sm_count);
size_t gemm_partial_floats(const GemmArgs& a);
cudaError_t launch_attention(const AttnArgs& a, int B, int kv_dtype_bf16, cudaStream_t s);
void plan_attention(AttnArgs& a, int max_batch, int max_seq_len, int max_gamma);
size_t attention_partial_floats(const AttnArgs& a, int max_batch);
// prep: weights_bf16 selects the embedding and gain type; x_pair the u output form.
// With p.parents (a token tree) it also writes each row's KV slot and ancestor mask.
cudaError_t launch_prep(const PrepParams& p, const int* tokens, const int* seq_len, int* row_req, int* row_pos,
                        int* row_slot, unsigned long long* row_anc, int* req_row0_dev, const void* embed,
                        const void* gain, float* h, void* u, long long u_plane, float* ss, int n_ss, int d, int vocab,
                        int max_seq_len, int weights_bf16, int x_pair, unsigned* status, cudaStream_t s);
cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t s);
cudaError_t launch_compact(const CompactArgs& a, cudaStream_t s);
cudaError_t launch_rope_table(float2* table, int max_seq_len, int head_dim, float theta, cudaStream_t s);
cudaError_t launch_w12_scan(const uint16_t* bf16, long long n, int base, unsigned* stats, cudaStream_t s);
// W12 planes: 64-row x 128-element tiles of 4096 bytes (see sv.h).
inline long long w12_plane_bytes(long long rows, long long cols) {
  return ((rows + 63) / 64) * ((cols + 127) / 128) * 4096;
}
cudaError_t launch_w12_pack(const uint16_t* bf16, long long rows, long long cols, int base, uint8_t* planes,
                            cudaStream_t s);
cudaError_t launch_w12_unpack(const uint8_t* planes, int base, long long rows, long long cols, uint16_t* out,
                              cudaStream_t s);
// grouped W12 (w12_grouped.cu)
cudaError_t launch_w12g_bases(const uint16_t* bf16, long long rows, long long cols, uint8_t* bases, cudaStream_t s);
cudaError_t launch_w12g_count(const uint16_t* bf16, long long rows, long long cols, const uint8_t* bases, int* cnt,
                              cudaStream_t s);
cudaError_t launch_w12g_pack(const uint16_t* bf16, long long rows, long long cols, const uint8_t* bases,
                             const int* off, uint8_t* planes, uint32_t* esc, cudaStream_t s);
cudaError_t launch_w12g_unpack(const uint8_t* planes, const uint8_t* bases, const int* off, const uint32_t* esc,
                               long long rows, long long cols, uint16_t* out, cudaStream_t s);
cudaError_t launch_philox(unsigned long long seed, long long req, long long pos0, int stream_id, int n, float* out,
                          cudaStream_t s);

}  // namespace sv
