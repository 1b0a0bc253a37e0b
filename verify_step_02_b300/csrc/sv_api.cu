// Host engine and C ABI of libsv: argument checks, workspace, and the
// launch sequence of one verify step (embedding, per layer QKV+RoPE+KV write,
// block-causal attention, O projection, MLP, then LM head and acceptance).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <utility>
#include <vector>

#include "internal.h"

using namespace sv;

namespace {

thread_local std::string g_err;

sv_status fail(sv_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

sv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(SV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define SV_CUDA(call, what)                         \
  do {                                              \
    cudaError_t e_ = (call);                        \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)


struct Timing {
  bool on = false;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pending[SV_KC_COUNT];
  std::vector<cudaEvent_t> spare;
  double ms[SV_KC_COUNT] = {};
  long long launches[SV_KC_COUNT] = {};
};

}  // namespace

void sv::record_error(const char* msg) { g_err = msg; }

struct sv_model {
  sv_config cfg;
  sv_weights w;
  std::vector<sv_layer_weights> layers;
  int wbf16 = 0;    // embedding, gains, KV cache in bf16 (else float32)
  int x_pair = 0;   // x tensors as hi/lo bf16 pairs (else float32)
  int sm_count = 148;
  int m_max = 0;
  int lm_tiles = 0;
  // workspace
  float* h = nullptr;
  float* ss = nullptr;   // [m_max][n_ss] per-tile sums of h^2 (RMSNorm statistics)
  int n_ss = 1;
  void* u = nullptr;
  void* q = nullptr;
  void* ao = nullptr;
  void* act = nullptr;
  long long u_plane = 0, ao_plane = 0, act_plane = 0;  // lo-plane offsets of the x tensors
  float* logits = nullptr;
  float2* argmax_part = nullptr;
  int* row_req = nullptr;
  int* row_pos = nullptr;
  int* row_slot = nullptr;             // token trees: KV slot of each row
  unsigned long long* row_anc = nullptr;  // token trees: visible block rows of each row
  int* req_row0 = nullptr;
  float2* rope = nullptr;
  float* gemm_part = nullptr;
  unsigned* gemm_cnt = nullptr;
  float* attn_part = nullptr;
  unsigned* attn_cnt = nullptr;
  float* attn_xpart = nullptr;     // tensor-core attention: partials of several clusters per item
  float2* attn_xml = nullptr;
  unsigned* attn_xcnt = nullptr;
  unsigned* status = nullptr;
  // staging for sv_verify_host
  int* d_tokens = nullptr;
  float* d_probs = nullptr;
  long long* d_reqids = nullptr;
  int* d_out = nullptr;  // accepted_len [max_batch], next_token [max_batch]
  std::vector<void*> allocs;
  // tensor path (bf16 weights): TMA maps of every weight matrix and of the x tensors
  bool use_tc = false;
  bool use_pdl = true;  // launch the step's kernels as programmatic dependents (overlapped prologues)
  std::vector<CUtensorMap> map_qkv, map_o, map_gu, map_d;
  CUtensorMap map_lm, map_u, map_ao, map_act;
  // tensor-core attention (bf16 KV): per-layer maps of the K and V page pools,
  // re-encoded when the caller passes other pools
  bool use_tc_attn = false;
  std::vector<CUtensorMap> map_k, map_v;
  std::vector<const void*> map_k_ptr, map_v_ptr;
  std::vector<int> map_kv_pages;
  // q maps for row tiles of q_rows[k] block rows, each tile's rows placed 1 << k
  // times into the 128 MMA rows (0: that layout does not fit)
  CUtensorMap map_q[3];
  int q_rows[3] = {0, 0, 0};
  bool last_logits = false;
  int last_m = 0;
  Timing timing;
  // per-CTA timeline (sv_model_set_trace)
  unsigned long long* trace = nullptr;
  long long trace_cap = 0, trace_used = 0;
  std::vector<long long> trace_launches;  // (first record, CTAs, kind) per traced launch
};

namespace {

template <typename T>
sv_status dalloc(sv_model* m, T** p, size_t bytes) {
  if (bytes == 0) bytes = 16;
  void* q = nullptr;
  const cudaError_t e = cudaMalloc(&q, bytes);
  if (e != cudaSuccess) return fail(SV_ERR_OUT_OF_MEMORY, "cudaMalloc(%zu): %s", bytes, cudaGetErrorString(e));
  m->allocs.push_back(q);
  *p = static_cast<T*>(q);
  return SV_OK;
}

void free_all(sv_model* m) {
  for (void* p : m->allocs) cudaFree(p);
  m->allocs.clear();
  for (auto& v : m->timing.pending)
    for (auto& pr : v) {
      cudaEventDestroy(pr.first);
      cudaEventDestroy(pr.second);
    }
  for (cudaEvent_t e : m->timing.spare) cudaEventDestroy(e);
}

int nqkv(const sv_config& c) { return (c.n_heads + 2 * c.n_kv_heads) * c.head_dim; }

sv_status check_config(const sv_config* c) {
  if (!c) return fail(SV_ERR_INVALID_ARG, "config is NULL");
  if (c->n_layers < 1 || c->d_model < 16 || c->n_heads < 1 || c->n_kv_heads < 1 || c->ffn < 16 || c->vocab < 2)
    return fail(SV_ERR_INVALID_ARG, "model sizes must be positive");
  if (c->n_heads % c->n_kv_heads) return fail(SV_ERR_INVALID_ARG, "n_heads must be a multiple of n_kv_heads");
  if (c->head_dim != 64 && c->head_dim != 128) return fail(SV_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (c->d_model % 16 || c->ffn % 16 || (c->n_heads * c->head_dim) % 16)
    return fail(SV_ERR_UNSUPPORTED, "d_model, ffn and n_heads*head_dim must be multiples of 16");
  if (c->weight_dtype < SV_F32 || c->weight_dtype > SV_W12) return fail(SV_ERR_INVALID_ARG, "bad weight_dtype");
  if (c->max_batch < 1 || c->max_batch > kMaxBatch) return fail(SV_ERR_INVALID_ARG, "max_batch must be 1..%d", kMaxBatch);
  if (c->max_gamma < 0 || c->max_gamma > kMaxGamma)
    return fail(SV_ERR_INVALID_ARG, "max_gamma must be 0..%d", kMaxGamma);
  if (c->page_size < 1 || c->page_size > 256) return fail(SV_ERR_INVALID_ARG, "page_size must be 1..256");
  if (c->weight_dtype != SV_F32 && c->page_size != 16)
    return fail(SV_ERR_UNSUPPORTED, "bf16/W12 models: page_size must be 16 (the tensor-core attention's page)");
  if (c->weight_dtype == SV_F32 && 256 % c->page_size)
    return fail(SV_ERR_UNSUPPORTED, "float32 models: page_size must divide 256 (the attention's key chunk)");
  if (c->max_seq_len < 1 || c->max_seq_len > (1 << 24)) return fail(SV_ERR_INVALID_ARG, "bad max_seq_len");
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return fail(SV_ERR_INVALID_ARG, "bad rms_eps or rope_theta");
  // float32 models run the CUDA-core attention, which holds a request's rows in shared memory
  if (c->weight_dtype == SV_F32 &&
      2LL * (c->n_heads / c->n_kv_heads) * (c->max_gamma + 1) * c->head_dim * 4 > 160 * 1024)
    return fail(SV_ERR_UNSUPPORTED,
                "float32 models: 2 * (n_heads / n_kv_heads) * (max_gamma + 1) * head_dim * 4 must be <= 160 KiB");
  return SV_OK;
}

// Sampled acceptance divides the logits by T in float32: below kMinTemperature
// z / T can overflow (and 1 / T does for T < ~3e-39), which would make every
// probability NaN, so such temperatures are refused (T = 0 is greedy).
constexpr float kMinTemperature = 1e-6f;

sv_status check_temperature(float T) {
  if (!(T >= 0.f) || std::isinf(T)) return fail(SV_ERR_INVALID_ARG, "temperature must be finite and >= 0");
  if (T > 0.f && T < kMinTemperature)
    return fail(SV_ERR_INVALID_ARG, "temperature %g is below the smallest sampled temperature %g (use 0 for greedy)",
                T, kMinTemperature);
  return SV_OK;
}

// ------------------------------------------------------------------ timing
void timed_begin(sv_model* m, int kc, cudaStream_t s, cudaEvent_t* ev) {
  *ev = nullptr;
  if (!m->timing.on) return;
  cudaEvent_t a, b;
  if (m->timing.spare.size() >= 2) {
    a = m->timing.spare.back();
    m->timing.spare.pop_back();
    b = m->timing.spare.back();
    m->timing.spare.pop_back();
  } else {
    cudaEventCreate(&a);
    cudaEventCreate(&b);
  }
  cudaEventRecord(a, s);
  m->timing.pending[kc].push_back({a, b});
  ev[0] = a;
}

void timed_end(sv_model* m, int kc, cudaStream_t s) {
  if (!m->timing.on) return;
  cudaEventRecord(m->timing.pending[kc].back().second, s);
  m->timing.launches[kc]++;
}

struct Timed {
  sv_model* m;
  int kc;
  cudaStream_t s;
  Timed(sv_model* m_, int kc_, cudaStream_t s_) : m(m_), kc(kc_), s(s_) {
    cudaEvent_t e;
    timed_begin(m, kc, s, &e);
  }
  ~Timed() { timed_end(m, kc, s); }
};

// Records for one traced launch of `ctas` CTAs, or nullptr (tracing off or full).
unsigned long long* trace_slot(sv_model* m, long long ctas, int kind) {
  if (!m->trace || m->trace_used + ctas > m->trace_cap) return nullptr;
  unsigned long long* p = m->trace + m->trace_used * kTraceWords;
  m->trace_launches.push_back(m->trace_used);
  m->trace_launches.push_back(ctas);
  m->trace_launches.push_back(kind);
  m->trace_used += ctas;
  return p;
}

// ------------------------------------------------------------------ GEMM helpers
GemmArgs gemm_base(sv_model* m, const sv_matrix& w, int n_rows, int K, const void* x, long long x_plane) {
  GemmArgs a;
  memset(&a, 0, sizeof a);
  a.wdtype = m->cfg.weight_dtype;
  a.w = w.data;
  a.w12_base = w.base;
  a.w12_kt = (K + 127) / 128;
  a.w12_plane = w12_plane_bytes(n_rows, K);
  a.w12_bases = w.row_bases;
  a.w12_esc_off = w.esc_off;
  a.w12_esc = w.esc;
  a.n_rows = n_rows;
  a.x = x;
  a.x_plane = x_plane;
  a.partials = m->gemm_part;
  a.counters = m->gemm_cnt;
  a.x_kind = m->x_pair ? kXPair : kXF32;
  a.epi.x_pair = m->x_pair;
  a.epi.kv_bf16 = m->wbf16;
  a.epi.status = m->status;
  a.epi.n_ss = m->n_ss;
  a.epi.d_model = m->cfg.d_model;
  a.epi.eps = m->cfg.rms_eps;
  a.epi.gain_bf16 = m->wbf16;
  a.pdl = m->use_pdl;
  return a;
}

// Largest split-K partial buffer and counter array any M in 1..m_max needs for a shape.
void gemm_ws_need(int sm, int m_max, int n_units, int K, int pair, size_t* part, size_t* cnt) {
  for (int M = 1; M <= m_max; ++M) {
    GemmArgs a;
    memset(&a, 0, sizeof a);
    plan_gemm(a, M, n_units, K, pair, sm);
    *part = std::max(*part, gemm_partial_floats(a));
    *cnt = std::max(*cnt, (size_t)a.n_tiles * a.m_tiles);
  }
}

// The tensor path where it applies and fits, else the FMA path: the larger need of both.
void gemm_tc_ws_need(int sm, int m_max, int n_units, int K, int pair, size_t* part, size_t* cnt, int wdtype) {
  gemm_ws_need(sm, m_max, n_units, K, pair, part, cnt);
  for (int M = 1; M <= m_max; ++M) {
    GemmArgs a;
    memset(&a, 0, sizeof a);
    a.x_kind = kXPair;
    a.wdtype = wdtype;
    plan_gemm_tc(a, M, n_units, K, pair, sm);
    *part = std::max(*part, gemm_tc_partial_floats(a));
    *cnt = std::max(*cnt, gemm_tc_counter_count(a));
  }
}

// wmap / xmap: the tensor maps of the weight and the x tensor (tensor path only).
sv_status run_gemm(sv_model* m, GemmArgs& a, int M, int n_units, int K, int pair, int kc, cudaStream_t s,
                   const char* what, const CUtensorMap* wmap = nullptr, const CUtensorMap* xmap = nullptr) {
  Timed t(m, kc, s);
  bool tc = m->use_tc && gemm_tc_supported(a.wdtype, pair, a.ffn);
  if (tc) {
    plan_gemm_tc(a, M, n_units, K, pair, m->sm_count);
    tc = a.tc_stages >= 2;
  }
  if (tc) {
    a.x_lo_row = m->m_max;
    a.trace = trace_slot(m, a.grid_p, kTrGemm);
    SV_CUDA(launch_gemm_tc(a, *wmap, *xmap, s), what);
  } else {
    plan_gemm(a, M, n_units, K, pair, m->sm_count);
    SV_CUDA(launch_gemm(a, s), what);
  }
  return SV_OK;
}

// Row-tile layout of the tensor-core attention for a call with block lengths
// lens[r] + 1: k = 0, 1, 2 places each tile's rows 1 << k times into the MMA
// rows, so that 1 << k TMEM lane groups share the softmax (each over 64 >> k
// keys of a sub-chunk); fewer rows per tile may mean more tiles, each reading
// the request's keys again. Cost per tile: K/V traffic (the larger part: a CTA's
// key stream is bound by the loads it can keep in flight) plus a softmax share.
int attention_layout(const sv_model* m, int B, const int* lens) {
  int best = 0;
  double best_cost = 0.0;
  for (int k = 0; k < 3; ++k) {
    if (m->q_rows[k] < 1) continue;
    long long tiles = 0;
    for (int r = 0; r < B; ++r) tiles += (lens[r] + m->q_rows[k]) / m->q_rows[k];
    const double cost = static_cast<double>(tiles) * (0.6 + 0.4 / (1 << k));
    if (k == 0 || cost < best_cost) {
      best = k;
      best_cost = cost;
    }
  }
  return best;
}

sv_status run_verify(sv_model* m, int B, const int* tokens, const int* lens, const sv_kv* kv, const float* probs,
                     float T, uint64_t seed, const long long* req_ids, int* acc_len, int* next_tok,
                     cudaStream_t s, bool commit_all = false, const int* parents = nullptr,
                     int* acc_nodes = nullptr) {
  const sv_config& c = m->cfg;
  if (B < 1 || B > c.max_batch) return fail(SV_ERR_INVALID_ARG, "batch %d outside 1..%d", B, c.max_batch);
  if (!tokens || !lens || !kv || !acc_len || !next_tok) return fail(SV_ERR_INVALID_ARG, "NULL argument");
  if (!kv->k || !kv->v || !kv->page_table || !kv->seq_len || kv->n_pages < 1 || kv->max_pages_per_seq < 1)
    return fail(SV_ERR_INVALID_ARG, "incomplete sv_kv");
  if (sv_status st = check_temperature(T)) return st;
  if (T > 0.f && !probs) return fail(SV_ERR_INVALID_ARG, "draft_probs required when temperature > 0");
  for (int l = 0; l < c.n_layers; ++l)
    if (!kv->k[l] || !kv->v[l]) return fail(SV_ERR_INVALID_ARG, "NULL KV pool for layer %d", l);
  static thread_local PrepParams p;
  int max_block = 1;  // the longest block (rows) of this call
  p.B = B;
  p.pdl = m->use_pdl;
  p.gamma_stride = c.max_gamma + 1;
  p.parents = parents;
  p.req_row0[0] = 0;
  for (int r = 0; r < B; ++r) {
    if (lens[r] < 0 || lens[r] > c.max_gamma)
      return fail(SV_ERR_INVALID_ARG, "verify_lens[%d] = %d outside 0..%d", r, lens[r], c.max_gamma);
    p.req_row0[r + 1] = p.req_row0[r] + lens[r] + 1;
    max_block = std::max(max_block, lens[r] + 1);
  }
  const int M = p.req_row0[B];
  p.M = M;
  const int d = c.d_model, hd = c.head_dim, nq = c.n_heads * hd, N3 = nqkv(c);
  const bool keep = T > 0.f || (c.flags & SV_FLAG_KEEP_LOGITS);
  {
    Timed t(m, SV_KC_NORM, s);
    SV_CUDA(launch_prep(p, tokens, kv->seq_len, m->row_req, m->row_pos, parents ? m->row_slot : nullptr,
                        m->row_anc, m->req_row0, m->w.embed,
                        m->layers[0].attn_norm, m->h, m->u, m->u_plane, m->ss, m->n_ss, d, c.vocab, c.max_seq_len,
                        m->wbf16, m->x_pair, m->status, s),
            "prep");
  }
  for (int l = 0; l < c.n_layers; ++l) {
    const sv_layer_weights& L = m->layers[l];
    {  // QKV projection, RoPE, q out, k/v into the page slots
      GemmArgs a = gemm_base(m, L.wqkv, N3, d, m->u, m->u_plane);
      a.epi.kind = kEpiQkv;
      a.epi.row_req = m->row_req;
      a.epi.row_pos = m->row_pos;
      a.epi.row_slot = parents ? m->row_slot : nullptr;
      a.epi.rope = m->rope;
      a.epi.n_heads = c.n_heads;
      a.epi.n_kv_heads = c.n_kv_heads;
      a.epi.head_dim = hd;
      a.epi.q_out = static_cast<float*>(m->q);
      if (m->use_tc_attn) {  // q as pre-scaled hi/lo bf16 planes for the tensor-core attention
        a.epi.q_pair = m->q;
        a.epi.q_plane = (long long)m->m_max * nq;
        a.epi.q_scale = 1.0f / std::sqrt(static_cast<float>(hd));
      }
      a.epi.ss_in = m->ss;
      a.epi.k_cache = kv->k[l];
      a.epi.v_cache = kv->v[l];
      a.epi.page_table = kv->page_table;
      a.epi.max_pages = kv->max_pages_per_seq;
      a.epi.page_size = c.page_size;
      a.epi.n_pages = kv->n_pages;
      sv_status st =
          run_gemm(m, a, M, N3, d, kPairNone, SV_KC_GEMM, s, "qkv gemm", &m->map_qkv[l], &m->map_u);
      if (st) return st;
    }
    {
      AttnArgs a;
      memset(&a, 0, sizeof a);
      a.q = static_cast<const float*>(m->q);
      a.out = m->ao;
      a.out_plane = m->ao_plane;
      a.k_cache = kv->k[l];
      a.v_cache = kv->v[l];
      a.page_table = kv->page_table;
      a.max_pages = kv->max_pages_per_seq;
      a.page_size = c.page_size;
      a.n_pages = kv->n_pages;
      a.seq_len = kv->seq_len;
      a.req_row0 = m->req_row0;
      a.row_anc = parents ? m->row_anc : nullptr;
      a.n_heads = c.n_heads;
      a.n_kv_heads = c.n_kv_heads;
      a.head_dim = hd;
      plan_attention(a, c.max_batch, c.max_seq_len, c.max_gamma);
      a.partials = m->attn_part;
      a.counters = m->attn_cnt;
      a.status = m->status;
      a.x_pair = m->x_pair;
      a.kv_bf16 = m->wbf16;
      a.pdl = m->use_pdl;
      if (m->use_tc_attn) {
        if (m->map_k_ptr[l] != kv->k[l] || m->map_v_ptr[l] != kv->v[l] || m->map_kv_pages[l] != kv->n_pages) {
          SV_CUDA(tc_encode_kv_map(&m->map_k[l], kv->k[l], kv->n_pages, c.n_kv_heads, hd), "K pool tensor map");
          SV_CUDA(tc_encode_kv_map(&m->map_v[l], kv->v[l], kv->n_pages, c.n_kv_heads, hd), "V pool tensor map");
          m->map_k_ptr[l] = kv->k[l];
          m->map_v_ptr[l] = kv->v[l];
          m->map_kv_pages[l] = kv->n_pages;
        }
        a.q_lo_row = m->m_max;
        const int ko = attention_layout(m, B, lens);
        a.q_rows = m->q_rows[ko];
        a.q_copies = 1 << ko;
        a.max_rows = a.q_rows * (c.n_heads / c.n_kv_heads);
        a.n_row_tiles = (max_block + a.q_rows - 1) / a.q_rows;
        const long long items = (long long)B * c.n_kv_heads * a.n_row_tiles;
        attention_tc_split(items, hd, m->sm_count, &a.cl_size, &a.cl_count);
        a.xpart = m->attn_xpart;
        a.xml = m->attn_xml;
        a.xcnt = m->attn_xcnt;
        a.trace = trace_slot(m, items * a.cl_size * a.cl_count, kTrAttn);
        Timed t(m, SV_KC_ATTENTION, s);
        SV_CUDA(launch_attention_tc(a, B, m->map_q[ko], m->map_k[l], m->map_v[l], s), "attention");
      } else {
        Timed t(m, SV_KC_ATTENTION, s);
        SV_CUDA(launch_attention(a, B, m->wbf16, s), "attention");
      }
    }
    {
      GemmArgs a = gemm_base(m, L.wo, d, nq, m->ao, m->ao_plane);
      a.epi.kind = kEpiResid;
      a.epi.h = m->h;
      a.epi.ldh = d;
      a.epi.next_gain = L.mlp_norm;
      a.epi.x_out = m->u;
      a.epi.x_out_plane = m->u_plane;
      a.epi.ss_out = m->ss;
      sv_status st = run_gemm(m, a, M, d, nq, kPairNone, SV_KC_GEMM, s, "o gemm", &m->map_o[l], &m->map_ao);
      if (st) return st;
    }
    {
      GemmArgs a = gemm_base(m, L.wgu, 2 * c.ffn, d, m->u, m->u_plane);
      a.ffn = c.ffn;
      a.epi.kind = kEpiSwiglu;
      a.epi.act = m->act;
      a.epi.act_plane = m->act_plane;
      a.epi.ffn = c.ffn;
      a.epi.ss_in = m->ss;
      sv_status st = run_gemm(m, a, M, c.ffn, d, kPairSwiglu, SV_KC_GEMM, s, "gate/up gemm", &m->map_gu[l],
                              &m->map_u);
      if (st) return st;
    }
    {
      GemmArgs a = gemm_base(m, L.wd, d, c.ffn, m->act, m->act_plane);
      a.epi.kind = kEpiResid;
      a.epi.h = m->h;
      a.epi.ldh = d;
      a.epi.next_gain = l + 1 < c.n_layers ? m->layers[l + 1].attn_norm : m->w.final_norm;
      a.epi.x_out = m->u;
      a.epi.x_out_plane = m->u_plane;
      a.epi.ss_out = m->ss;
      sv_status st =
          run_gemm(m, a, M, d, c.ffn, kPairNone, SV_KC_GEMM, s, "down gemm", &m->map_d[l], &m->map_act);
      if (st) return st;
    }
  }
  {
    GemmArgs a = gemm_base(m, m->w.lm_head, c.vocab, d, m->u, m->u_plane);
    a.epi.kind = kEpiLogits;
    a.epi.ss_in = m->ss;
    a.epi.logits = keep ? m->logits : nullptr;
    a.epi.argmax_part = m->argmax_part;
    a.epi.vocab = c.vocab;
    sv_status st = run_gemm(m, a, M, c.vocab, d, kPairNone, SV_KC_LM_HEAD, s, "lm head", &m->map_lm, &m->map_u);
    if (st) return st;
  }
  {
    AcceptArgs a;
    memset(&a, 0, sizeof a);
    a.B = B;
    a.vocab = c.vocab;
    a.gamma_stride = c.max_gamma + 1;
    a.tokens = tokens;
    a.req_row0 = m->req_row0;
    a.seq_len = kv->seq_len;
    a.logits = m->logits;
    a.argmax_part = m->argmax_part;
    a.n_tiles = m->lm_tiles;
    a.draft_probs = probs;
    a.max_gamma = c.max_gamma;
    a.temperature = T;
    a.seed = seed;
    a.request_ids = req_ids;
    a.accepted_len = acc_len;
    a.next_token = next_tok;
    a.status = m->status;
    a.pdl = m->use_pdl;
    a.commit_all = commit_all ? 1 : 0;
    a.parents = parents;
    a.accepted_nodes = acc_nodes;
    Timed t(m, SV_KC_ACCEPT, s);
    SV_CUDA(launch_accept(a, s), "accept");
  }
  if (parents) {
    // token tree: the accepted path's keys and values move to positions C .. C + k
    CompactArgs a;
    memset(&a, 0, sizeof a);
    a.B = B;
    a.gamma_stride = c.max_gamma + 1;
    a.seq_len = kv->seq_len;
    a.accepted_len = acc_len;
    a.accepted_nodes = acc_nodes;
    a.page_table = kv->page_table;
    a.max_pages = kv->max_pages_per_seq;
    a.page_size = c.page_size;
    a.n_pages = kv->n_pages;
    a.row_bytes = hd * (m->wbf16 ? 2 : 4);
    a.n_kv_heads = c.n_kv_heads;
    a.pdl = m->use_pdl;
    Timed t(m, SV_KC_ACCEPT, s);
    for (int l0 = 0; l0 < c.n_layers; l0 += kCompactLayers) {
      a.n = std::min(kCompactLayers, c.n_layers - l0);
      for (int i = 0; i < a.n; ++i) {
        a.k[i] = kv->k[l0 + i];
        a.v[i] = kv->v[l0 + i];
      }
      SV_CUDA(launch_compact(a, s), "tree commit");
    }
  }
  m->last_logits = keep;
  m->last_m = M;
  return SV_OK;
}

}  // namespace

extern "C" {

const char* sv_last_error(void) { return g_err.c_str(); }

int64_t sv_w12_plane_bytes(int64_t rows, int64_t cols) { return rows < 1 || cols < 1 ? 0 : w12_plane_bytes(rows, cols); }

sv_status sv_model_create(const sv_config* cfg, const sv_weights* weights, void* stream, sv_model** out) {
  if (!out) return fail(SV_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  sv_status st = check_config(cfg);
  if (st) return st;
  if (!weights || !weights->embed || !weights->final_norm || !weights->lm_head.data || !weights->layers)
    return fail(SV_ERR_INVALID_ARG, "incomplete sv_weights");
  // W12 matrices: a tensor-wide base in 1 .. 254, or grouped (row bases and escape offsets)
  auto bad_w12 = [&](const sv_matrix& w) {
    if (cfg->weight_dtype != SV_W12) return false;
    return w.row_bases ? !w.esc_off : (w.base < 1 || w.base > 254);
  };
  if (bad_w12(weights->lm_head)) return fail(SV_ERR_INVALID_ARG, "bad W12 lm_head (base or grouped arrays)");
  for (int l = 0; l < cfg->n_layers; ++l) {
    const sv_layer_weights& L = weights->layers[l];
    if (!L.attn_norm || !L.mlp_norm || !L.wqkv.data || !L.wo.data || !L.wgu.data || !L.wd.data)
      return fail(SV_ERR_INVALID_ARG, "incomplete weights for layer %d", l);
    if (bad_w12(L.wqkv) || bad_w12(L.wo) || bad_w12(L.wgu) || bad_w12(L.wd))
      return fail(SV_ERR_INVALID_ARG, "bad W12 matrix in layer %d (base or grouped arrays)", l);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  sv_model* m = new sv_model();
  m->cfg = *cfg;
  m->w = *weights;
  m->layers.assign(weights->layers, weights->layers + cfg->n_layers);
  m->w.layers = nullptr;
  m->wbf16 = cfg->weight_dtype == SV_F32 ? 0 : 1;
  m->use_pdl = (cfg->flags & SV_FLAG_NO_PDL) == 0;
  m->x_pair = m->wbf16;
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&m->sm_count, cudaDevAttrMultiProcessorCount, dev);
  const sv_config& c = *cfg;
  const int M = c.max_batch * (c.max_gamma + 1);
  m->m_max = M;
  m->lm_tiles = (c.vocab + kGemmBN - 1) / kGemmBN;
  const int d = c.d_model, nq = c.n_heads * c.head_dim;
  // x tensors: float32, or two bf16 planes of M rows each (the same bytes)
  const size_t ab = 4;
  m->u_plane = m->x_pair ? (long long)M * d : 0;
  m->ao_plane = m->x_pair ? (long long)M * nq : 0;
  m->act_plane = m->x_pair ? (long long)M * c.ffn : 0;
#define TRY(x)            \
  do {                    \
    st = (x);             \
    if (st) {             \
      free_all(m);        \
      delete m;           \
      return st;          \
    }                     \
  } while (0)
  TRY(dalloc(m, &m->h, sizeof(float) * M * d));
  m->n_ss = (d + kGemmBN - 1) / kGemmBN;
  TRY(dalloc(m, &m->ss, sizeof(float) * M * m->n_ss));
  TRY(dalloc(m, &m->u, ab * M * std::max(d, 16)));
  TRY(dalloc(m, &m->q, sizeof(float) * M * nq));
  TRY(dalloc(m, &m->ao, ab * M * nq));
  TRY(dalloc(m, &m->act, ab * M * c.ffn));
  TRY(dalloc(m, &m->logits, sizeof(float) * M * (size_t)c.vocab));
  TRY(dalloc(m, &m->argmax_part, sizeof(float2) * M * (size_t)m->lm_tiles));
  TRY(dalloc(m, &m->row_req, sizeof(int) * M));
  TRY(dalloc(m, &m->row_pos, sizeof(int) * M));
  TRY(dalloc(m, &m->row_slot, sizeof(int) * M));
  TRY(dalloc(m, &m->row_anc, sizeof(unsigned long long) * M));
  TRY(dalloc(m, &m->req_row0, sizeof(int) * (c.max_batch + 1)));
  TRY(dalloc(m, &m->rope, sizeof(float2) * (size_t)c.max_seq_len * (c.head_dim / 2)));
  size_t part = 0, cnt = 0;
  m->use_tc = (cfg->weight_dtype == SV_BF16 || cfg->weight_dtype == SV_W12) && !(cfg->flags & SV_FLAG_CUDA_CORE_GEMM);
  auto need = [&](int n_units, int K, int pair) {
    if (m->use_tc)
      gemm_tc_ws_need(m->sm_count, M, n_units, K, pair, &part, &cnt, cfg->weight_dtype);
    else
      gemm_ws_need(m->sm_count, M, n_units, K, pair, &part, &cnt);
  };
  need(nqkv(c), d, kPairNone);
  need(d, nq, kPairNone);
  need(c.ffn, d, kPairSwiglu);
  need(d, c.ffn, kPairNone);
  need(c.vocab, d, kPairNone);
  TRY(dalloc(m, &m->gemm_part, sizeof(float) * part));
  TRY(dalloc(m, &m->gemm_cnt, sizeof(unsigned) * cnt));
  AttnArgs aa;
  memset(&aa, 0, sizeof aa);
  aa.n_heads = c.n_heads;
  aa.n_kv_heads = c.n_kv_heads;
  aa.head_dim = c.head_dim;
  plan_attention(aa, c.max_batch, c.max_seq_len, c.max_gamma);
  TRY(dalloc(m, &m->attn_part, sizeof(float) * attention_partial_floats(aa, c.max_batch)));
  TRY(dalloc(m, &m->attn_cnt, sizeof(unsigned) * c.max_batch * c.n_kv_heads));
  if (m->wbf16) {  // the tensor-core attention's cross-cluster merge (few work items)
    const size_t slots = (size_t)kCrossItems * kMaxCrossClusters * 128;
    TRY(dalloc(m, &m->attn_xpart, sizeof(float) * slots * c.head_dim));
    TRY(dalloc(m, &m->attn_xml, sizeof(float2) * slots));
    TRY(dalloc(m, &m->attn_xcnt, sizeof(unsigned) * kCrossItems * 16));
  }
  TRY(dalloc(m, &m->status, sizeof(unsigned) * 4));
  TRY(dalloc(m, &m->d_tokens, sizeof(int) * c.max_batch * (c.max_gamma + 1)));
  TRY(dalloc(m, &m->d_probs, sizeof(float) * (size_t)c.max_batch * std::max(c.max_gamma, 1) * c.vocab));
  TRY(dalloc(m, &m->d_reqids, sizeof(long long) * c.max_batch));
  TRY(dalloc(m, &m->d_out, sizeof(int) * 2 * c.max_batch));
#undef TRY
  m->use_tc_attn = m->wbf16 && attention_tc_supported(c.head_dim, c.page_size, aa.max_rows, c.max_seq_len);
  if (m->use_tc_attn) {
    m->map_k.resize(c.n_layers);
    m->map_v.resize(c.n_layers);
    m->map_k_ptr.assign(c.n_layers, nullptr);
    m->map_v_ptr.assign(c.n_layers, nullptr);
    m->map_kv_pages.assign(c.n_layers, 0);
    // q of one attention row tile: q_rows block rows x the group's heads, times the
    // copies, <= 128 MMA rows
    const int group = c.n_heads / c.n_kv_heads;
    for (int k = 0; k < 3; ++k) {
      m->q_rows[k] = std::min(c.max_gamma + 1, (128 >> k) / group);
      if (m->q_rows[k] < 1) {
        m->q_rows[k] = 0;
        continue;
      }
      const cudaError_t qe = tc_encode_q_map(&m->map_q[k], m->q, M, c.n_heads, c.head_dim, group, m->q_rows[k]);
      if (qe != cudaSuccess) {
        free_all(m);
        delete m;
        return fail(SV_ERR_CUDA, "q tensor map: %s", cudaGetErrorString(qe));
      }
    }
  }
  if (m->use_tc) {
    cudaError_t me = cudaSuccess;
    auto enc_w = [&](CUtensorMap* mp, const sv_matrix& w, long long rows, int K) {
      // bf16 weights stream through tensor maps; W12 planes through contiguous tile copies
      if (me == cudaSuccess && cfg->weight_dtype == SV_BF16) me = tc_encode_weight_map(mp, w.data, rows, K);
    };
    const int L = c.n_layers;
    m->map_qkv.resize(L);
    m->map_o.resize(L);
    m->map_gu.resize(L);
    m->map_d.resize(L);
    for (int l = 0; l < L; ++l) {
      enc_w(&m->map_qkv[l], m->layers[l].wqkv, nqkv(c), d);
      enc_w(&m->map_o[l], m->layers[l].wo, d, nq);
      enc_w(&m->map_gu[l], m->layers[l].wgu, 2LL * c.ffn, d);
      enc_w(&m->map_d[l], m->layers[l].wd, d, c.ffn);
    }
    enc_w(&m->map_lm, m->w.lm_head, c.vocab, d);
    if (me == cudaSuccess) me = tc_encode_x_map(&m->map_u, m->u, 2LL * M, d);
    if (me == cudaSuccess) me = tc_encode_x_map(&m->map_ao, m->ao, 2LL * M, nq);
    if (me == cudaSuccess) me = tc_encode_x_map(&m->map_act, m->act, 2LL * M, c.ffn);
    if (me != cudaSuccess) {
      free_all(m);
      delete m;
      return fail(SV_ERR_INVALID_ARG, "tensor map encoding failed (weights must be 16-byte aligned): %s",
                  cudaGetErrorString(me));
    }
  }
  cudaError_t e = cudaMemsetAsync(m->gemm_cnt, 0, sizeof(unsigned) * cnt, s);
  if (e == cudaSuccess && m->attn_xcnt) e = cudaMemsetAsync(m->attn_xcnt, 0, sizeof(unsigned) * kCrossItems * 16, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(m->attn_cnt, 0, sizeof(unsigned) * c.max_batch * c.n_kv_heads, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(m->status, 0, sizeof(unsigned) * 4, s);
  if (e == cudaSuccess) e = launch_rope_table(m->rope, c.max_seq_len, c.head_dim, c.rope_theta, s);
  if (e != cudaSuccess) {
    free_all(m);
    delete m;
    return cuda_fail(e, "model init");
  }
  *out = m;
  return SV_OK;
}

void sv_model_destroy(sv_model* model) {
  if (!model) return;
  cudaDeviceSynchronize();
  free_all(model);
  delete model;
}

sv_status sv_verify(sv_model* model, int32_t batch, const int32_t* tokens, const int32_t* verify_lens,
                    const sv_kv* kv, const float* draft_probs, float temperature, uint64_t seed,
                    const int64_t* request_ids, int32_t* accepted_len, int32_t* next_token, void* stream) {
  if (sv_status st = check_temperature(temperature)) return st;
  if (!model) return fail(SV_ERR_INVALID_ARG, "model is NULL");
  return run_verify(model, batch, tokens, verify_lens, kv, draft_probs, temperature, seed,
                    reinterpret_cast<const long long*>(request_ids), accepted_len, next_token,
                    static_cast<cudaStream_t>(stream));
}

sv_status sv_verify_host(sv_model* model, int32_t batch, const int32_t* tokens, const int32_t* verify_lens,
                         const sv_kv* kv, const float* draft_probs, float temperature, uint64_t seed,
                         const int64_t* request_ids, int32_t* accepted_len, int32_t* next_token, void* stream) {
  if (sv_status st = check_temperature(temperature)) return st;
  if (!model) return fail(SV_ERR_INVALID_ARG, "model is NULL");
  const sv_config& c = model->cfg;
  if (batch < 1 || batch > c.max_batch) return fail(SV_ERR_INVALID_ARG, "batch %d outside 1..%d", batch, c.max_batch);
  if (!tokens || !accepted_len || !next_token) return fail(SV_ERR_INVALID_ARG, "NULL argument");
  if (temperature > 0.f && !draft_probs) return fail(SV_ERR_INVALID_ARG, "draft_probs required when temperature > 0");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t tok_bytes = sizeof(int) * batch * (c.max_gamma + 1);
  SV_CUDA(cudaMemcpyAsync(model->d_tokens, tokens, tok_bytes, cudaMemcpyHostToDevice, s), "copy tokens");
  const float* dp = nullptr;
  if (temperature > 0.f) {
    SV_CUDA(cudaMemcpyAsync(model->d_probs, draft_probs, sizeof(float) * batch * c.max_gamma * (size_t)c.vocab,
                            cudaMemcpyHostToDevice, s),
            "copy draft_probs");
    dp = model->d_probs;
  }
  const long long* rid = nullptr;
  if (request_ids) {
    SV_CUDA(cudaMemcpyAsync(model->d_reqids, request_ids, sizeof(long long) * batch, cudaMemcpyHostToDevice, s),
            "copy request_ids");
    rid = model->d_reqids;
  }
  sv_status st = run_verify(model, batch, model->d_tokens, verify_lens, kv, dp, temperature, seed, rid,
                            model->d_out, model->d_out + c.max_batch, s);
  if (st) return st;
  SV_CUDA(cudaMemcpyAsync(accepted_len, model->d_out, sizeof(int) * batch, cudaMemcpyDeviceToHost, s),
          "copy accepted_len");
  SV_CUDA(cudaMemcpyAsync(next_token, model->d_out + c.max_batch, sizeof(int) * batch, cudaMemcpyDeviceToHost, s),
          "copy next_token");
  SV_CUDA(cudaStreamSynchronize(s), "synchronize");
  return SV_OK;
}

sv_status sv_prefill(sv_model* model, int32_t batch, const int32_t* tokens, const int32_t* block_lens,
                     const sv_kv* kv, int32_t* next_token, void* stream) {
  if (!model) return fail(SV_ERR_INVALID_ARG, "model is NULL");
  if (!next_token) return fail(SV_ERR_INVALID_ARG, "NULL argument");
  return run_verify(model, batch, tokens, block_lens, kv, nullptr, 0.f, 0, nullptr, model->d_out, next_token,
                    static_cast<cudaStream_t>(stream), true);
}

sv_status sv_verify_tree(sv_model* model, int32_t batch, const int32_t* tokens, const int32_t* parents,
                         const int32_t* n_drafts, const sv_kv* kv, int32_t* accepted_len, int32_t* next_token,
                         int32_t* accepted_nodes, void* stream) {
  if (!model) return fail(SV_ERR_INVALID_ARG, "model is NULL");
  if (!parents || !n_drafts || !accepted_nodes) return fail(SV_ERR_INVALID_ARG, "NULL argument");
  const sv_config& c = model->cfg;
  if (batch < 1 || batch > c.max_batch) return fail(SV_ERR_INVALID_ARG, "batch %d outside 1..%d", batch, c.max_batch);
  const int lim = std::min(c.max_gamma, kMaxTreeNodes - 1);
  for (int r = 0; r < batch; ++r)
    if (n_drafts[r] < 0 || n_drafts[r] > lim)
      return fail(SV_ERR_INVALID_ARG, "n_drafts[%d] = %d outside 0..%d", r, n_drafts[r], lim);
  return run_verify(model, batch, tokens, n_drafts, kv, nullptr, 0.f, 0, nullptr, accepted_len, next_token,
                    static_cast<cudaStream_t>(stream), false, parents, accepted_nodes);
}

sv_status sv_model_logits(sv_model* model, float* dst, int32_t rows, void* stream) {
  if (!model || !dst) return fail(SV_ERR_INVALID_ARG, "NULL argument");
  if (!model->last_logits) return fail(SV_ERR_INVALID_ARG, "the last verify kept no logits");
  if (rows != model->last_m) return fail(SV_ERR_INVALID_ARG, "rows %d != last verify's M %d", rows, model->last_m);
  SV_CUDA(cudaMemcpyAsync(dst, model->logits, sizeof(float) * rows * (size_t)model->cfg.vocab,
                          cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream)),
          "copy logits");
  return SV_OK;
}

sv_status sv_model_sync_status(sv_model* model, void* stream) {
  if (!model) return fail(SV_ERR_INVALID_ARG, "model is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned word = 0;
  SV_CUDA(cudaMemcpyAsync(&word, model->status, sizeof word, cudaMemcpyDeviceToHost, s), "read status");
  SV_CUDA(cudaStreamSynchronize(s), "synchronize");
  SV_CUDA(cudaMemsetAsync(model->status, 0, sizeof(unsigned), s), "clear status");
  SV_CUDA(cudaStreamSynchronize(s), "synchronize");
  if (word) {
    // a block that only overran its KV capacity is SV_ERR_KV_CAPACITY; anything else a failed check
    const bool capacity_only = (word & ~(kStBadPos | kStNoPage)) == 0;
    return fail(capacity_only ? SV_ERR_KV_CAPACITY : SV_ERR_DEVICE_CHECK, "device check failed:%s%s%s%s%s%s%s",
                (word & kStBadToken) ? " token id out of range" : "", (word & kStBadPage) ? " page id out of range" : "",
                (word & kStTimeout) ? " wait timed out" : "",
                (word & kStBadPos) ? " a block position reaches max_seq_len" : "",
                (word & kStNoPage) ? " a block position is past the request's page table" : "",
                (word & kStBadDraftProb) ? " bad draft probability" : "",
                (word & kStBadTree) ? " a tree node's parent does not precede it" : "");
  }
  return SV_OK;
}

sv_status sv_model_set_timing(sv_model* model, int32_t enable) {
  if (!model) return fail(SV_ERR_INVALID_ARG, "model is NULL");
  Timing& t = model->timing;
  t.on = enable != 0;
  for (int k = 0; k < SV_KC_COUNT; ++k) {
    for (auto& pr : t.pending[k]) {
      t.spare.push_back(pr.first);
      t.spare.push_back(pr.second);
    }
    t.pending[k].clear();
    t.ms[k] = 0;
    t.launches[k] = 0;
  }
  return SV_OK;
}

sv_status sv_model_timing(sv_model* model, double* ms, int64_t* launches) {
  if (!model || !ms || !launches) return fail(SV_ERR_INVALID_ARG, "NULL argument");
  Timing& t = model->timing;
  for (int k = 0; k < SV_KC_COUNT; ++k) {
    for (auto& pr : t.pending[k]) {
      SV_CUDA(cudaEventSynchronize(pr.second), "event sync");
      float e = 0.f;
      SV_CUDA(cudaEventElapsedTime(&e, pr.first, pr.second), "event elapsed");
      t.ms[k] += e;
      t.spare.push_back(pr.first);
      t.spare.push_back(pr.second);
    }
    t.pending[k].clear();
    ms[k] = t.ms[k];
    launches[k] = t.launches[k];
  }
  return SV_OK;
}

sv_status sv_model_set_trace(sv_model* model, uint64_t* records, int64_t capacity) {
  if (!model) return fail(SV_ERR_INVALID_ARG, "model is NULL");
  if ((records == nullptr) != (capacity == 0) || capacity < 0)
    return fail(SV_ERR_INVALID_ARG, "records and capacity must both be set or both be 0");
  model->trace = reinterpret_cast<unsigned long long*>(records);
  model->trace_cap = capacity;
  model->trace_used = 0;
  model->trace_launches.clear();
  return SV_OK;
}

sv_status sv_model_trace_launches(sv_model* model, int64_t* launches, int64_t max_launches, int64_t* n_launches) {
  if (!model || !n_launches) return fail(SV_ERR_INVALID_ARG, "NULL argument");
  const int64_t n = static_cast<int64_t>(model->trace_launches.size() / 3);
  *n_launches = n;
  if (launches)
    for (int64_t i = 0; i < n && i < max_launches; ++i)
      for (int j = 0; j < 3; ++j) launches[3 * i + j] = model->trace_launches[3 * i + j];
  return SV_OK;
}

sv_status sv_pack_w12(const uint16_t* bf16, int64_t rows, int64_t cols, uint8_t* planes, int32_t* base_out,
                      int64_t* n_unrepresentable, void* stream) {
  if (!bf16 || !planes || !base_out || !n_unrepresentable) return fail(SV_ERR_INVALID_ARG, "NULL argument");
  if (rows < 1 || cols < 1) return fail(SV_ERR_INVALID_ARG, "rows and cols must be positive");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned* stats = nullptr;
  SV_CUDA(cudaMallocAsync(reinterpret_cast<void**>(&stats), 4 * sizeof(unsigned), s), "alloc stats");
  unsigned h[4] = {255u, 0u, 0u, 0u};
  sv_status st = SV_OK;
  cudaError_t e = cudaMemcpyAsync(stats, h, sizeof h, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = launch_w12_scan(bf16, rows * cols, -1, stats, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h, stats, sizeof h, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  long long bad = h[2];
  const int base = h[0] <= 254u ? static_cast<int>(h[0]) : 1;
  if (e == cudaSuccess && h[1] > h[0] + 15u && h[0] <= 254u) {
    unsigned z[4] = {255u, 0u, 0u, 0u};
    e = cudaMemcpyAsync(stats, z, sizeof z, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = launch_w12_scan(bf16, rows * cols, base, stats, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h, stats, sizeof h, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    bad += h[3];
  }
  if (e == cudaSuccess && bad == 0) e = launch_w12_pack(bf16, rows, cols, base, planes, s);
  cudaFreeAsync(stats, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "pack_w12");
  *n_unrepresentable = bad;
  *base_out = base;
  if (bad) st = fail(SV_ERR_NOT_REPRESENTABLE, "%lld elements are not representable in W12", bad);
  return st;
}

sv_status sv_unpack_w12(const uint8_t* planes, int32_t base, int64_t rows, int64_t cols, uint16_t* bf16_out,
                        void* stream) {
  if (!planes || !bf16_out) return fail(SV_ERR_INVALID_ARG, "NULL argument");
  if (rows < 1 || cols < 1 || base < 1 || base > 254) return fail(SV_ERR_INVALID_ARG, "bad sizes or base");
  SV_CUDA(launch_w12_unpack(planes, base, rows, cols, bf16_out, static_cast<cudaStream_t>(stream)),
          "unpack_w12");
  return SV_OK;
}

int64_t sv_w12_row_blocks(int64_t rows) { return rows < 1 ? 0 : (rows + 63) / 64; }
int64_t sv_w12_tiles(int64_t rows, int64_t cols) {
  return rows < 1 || cols < 1 ? 0 : ((rows + 63) / 64) * ((cols + 127) / 128);
}

sv_status sv_pack_w12_grouped(const uint16_t* bf16, int64_t rows, int64_t cols, uint8_t* planes, uint8_t* row_bases,
                              int32_t* esc_off, uint32_t* esc, int64_t esc_capacity, int64_t* n_escapes,
                              void* stream) {
  if (!bf16 || !planes || !row_bases || !esc_off || !n_escapes) return fail(SV_ERR_INVALID_ARG, "NULL argument");
  if (rows < 1 || cols < 1) return fail(SV_ERR_INVALID_ARG, "rows and cols must be positive");
  if (esc_capacity < 0 || (esc_capacity > 0 && !esc)) return fail(SV_ERR_INVALID_ARG, "bad escape buffer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t tiles = sv_w12_tiles(rows, cols);
  // per-tile escape counts into esc_off, their exclusive scan on the host, back to esc_off
  SV_CUDA(launch_w12g_bases(bf16, rows, cols, row_bases, s), "w12 grouped bases");
  SV_CUDA(launch_w12g_count(bf16, rows, cols, row_bases, esc_off, s), "w12 grouped count");
  std::vector<int32_t> off(static_cast<size_t>(tiles) + 1);
  SV_CUDA(cudaMemcpyAsync(off.data(), esc_off, sizeof(int32_t) * tiles, cudaMemcpyDeviceToHost, s), "read counts");
  SV_CUDA(cudaStreamSynchronize(s), "synchronize");
  long long total = 0;
  for (int64_t i = 0; i < tiles; ++i) {
    const long long c = off[i];
    off[i] = static_cast<int32_t>(total);
    total += c;
  }
  if (total > 0x7FFFFFFFll) return fail(SV_ERR_NOT_REPRESENTABLE, "too many escapes (%lld)", total);
  off[tiles] = static_cast<int32_t>(total);
  SV_CUDA(cudaMemcpyAsync(esc_off, off.data(), sizeof(int32_t) * (tiles + 1), cudaMemcpyHostToDevice, s),
          "write offsets");
  const bool fits = total <= esc_capacity;
  SV_CUDA(launch_w12g_pack(bf16, rows, cols, row_bases, esc_off, planes, fits && total > 0 ? esc : nullptr, s),
          "w12 grouped pack");
  SV_CUDA(cudaStreamSynchronize(s), "synchronize");
  *n_escapes = total;
  if (!fits && esc) return fail(SV_ERR_INVALID_ARG, "%lld escapes exceed the capacity %lld", total, (long long)esc_capacity);
  return SV_OK;
}

sv_status sv_unpack_w12_grouped(const uint8_t* planes, const uint8_t* row_bases, const int32_t* esc_off,
                                const uint32_t* esc, int64_t rows, int64_t cols, uint16_t* bf16_out, void* stream) {
  if (!planes || !row_bases || !esc_off || !bf16_out) return fail(SV_ERR_INVALID_ARG, "NULL argument");
  if (rows < 1 || cols < 1) return fail(SV_ERR_INVALID_ARG, "rows and cols must be positive");
  SV_CUDA(launch_w12g_unpack(planes, row_bases, esc_off, esc, rows, cols, bf16_out, static_cast<cudaStream_t>(stream)),
          "unpack_w12_grouped");
  return SV_OK;
}

size_t sv_linear_workspace_bytes(int32_t wdtype, int32_t M, int32_t N, int32_t K) {
  if (M < 1 || N < 1 || K < 1) return 0;
  int dev = 0, sm = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev);
  GemmArgs a;
  memset(&a, 0, sizeof a);
  size_t need = 0;
  if (wdtype == SV_BF16 || wdtype == SV_W12) {  // tensor path; the pair plan needs the most scratch
    a.x_kind = kXPair;
    a.wdtype = wdtype;
    plan_gemm_tc(a, M, N, K, kPairNone, sm);
    const size_t cnt = (gemm_tc_counter_count(a) * sizeof(unsigned) + 255) & ~(size_t)255;
    need = cnt + gemm_tc_partial_floats(a) * sizeof(float);
  }
  memset(&a, 0, sizeof a);  // the CUDA-core path (float32 weights, or a token tile too wide for the tensor path)
  plan_gemm(a, M, N, K, kPairNone, sm);
  const size_t cnt = ((size_t)a.n_tiles * a.m_tiles * sizeof(unsigned) + 255) & ~(size_t)255;
  return std::max(need, cnt + gemm_partial_floats(a) * sizeof(float));
}

sv_status sv_linear(int32_t wdtype, const sv_matrix* w, int32_t N, int32_t K, const void* x, int32_t x_planes,
                    int32_t M, float* y, void* workspace, size_t workspace_bytes, void* stream) {
  if (!w || !w->data || !x || !y || !workspace) return fail(SV_ERR_INVALID_ARG, "NULL argument");
  if (wdtype < SV_F32 || wdtype > SV_W12) return fail(SV_ERR_INVALID_ARG, "bad wdtype");
  if (x_planes != 1 && !(x_planes == 2 && wdtype != SV_F32))
    return fail(SV_ERR_INVALID_ARG, "x_planes must be 1, or 2 for bf16/W12 weights");
  if (M < 1 || M > 4096 || N < 1 || K < 16 || K % 16) return fail(SV_ERR_INVALID_ARG, "need 1<=M<=4096, N>=1, K%%16==0");
  if (wdtype == SV_W12 && !w->row_bases && (w->base < 1 || w->base > 254))
    return fail(SV_ERR_INVALID_ARG, "bad W12 base");
  if (wdtype == SV_W12 && w->row_bases && !w->esc_off) return fail(SV_ERR_INVALID_ARG, "grouped W12 without esc_off");
  const size_t need = sv_linear_workspace_bytes(wdtype, M, N, K);
  if (workspace_bytes < need) return fail(SV_ERR_INVALID_ARG, "workspace %zu < %zu bytes", workspace_bytes, need);
  int dev = 0, sm = 148;
  cudaGetDevice(&dev);
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
  a.epi.kind = kEpiStore;
  a.epi.y = y;
  a.epi.ldy = N;
  if (wdtype == SV_BF16 || wdtype == SV_W12) {
    plan_gemm_tc(a, M, N, K, kPairNone, sm);
    if (a.tc_stages >= 2) {
      const size_t cnt = (gemm_tc_counter_count(a) * sizeof(unsigned) + 255) & ~(size_t)255;
      a.counters = static_cast<unsigned*>(workspace);
      a.partials = reinterpret_cast<float*>(static_cast<char*>(workspace) + cnt);
      a.x_lo_row = M;
      CUtensorMap xm, wm;
      SV_CUDA(tc_encode_x_map(&xm, x, (long long)x_planes * M, K), "x tensor map");
      if (wdtype == SV_BF16)
        SV_CUDA(tc_encode_weight_map(&wm, w->data, N, K), "weight tensor map");
      else
        wm = xm;  // W12 planes are read by contiguous tile copies, not a tensor map
      SV_CUDA(launch_gemm_tc(a, wm, xm, static_cast<cudaStream_t>(stream)), "linear");
      return SV_OK;
    }
  }
  plan_gemm(a, M, N, K, kPairNone, sm);
  const size_t cnt = ((size_t)a.n_tiles * a.m_tiles * sizeof(unsigned) + 255) & ~(size_t)255;
  a.counters = static_cast<unsigned*>(workspace);
  a.partials = reinterpret_cast<float*>(static_cast<char*>(workspace) + cnt);
  SV_CUDA(launch_gemm(a, static_cast<cudaStream_t>(stream)), "linear");
  return SV_OK;
}

sv_status sv_philox_uniform(uint64_t seed, int64_t request_id, int64_t position0, int32_t stream_id, int32_t n,
                            float* out, void* stream) {
  if (!out || n < 0) return fail(SV_ERR_INVALID_ARG, "bad arguments");
  if (n == 0) return SV_OK;
  SV_CUDA(launch_philox(seed, request_id, position0, stream_id, n, out, static_cast<cudaStream_t>(stream)),
          "philox");
  return SV_OK;
}

}  // extern "C"
