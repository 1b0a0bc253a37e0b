/*
 * sv.h — C ABI of libsv, the target-model verify step of speculative decoding
 * on one B300 (sm_103a).
 *
 * What the step computes (DSpark summary, "Architecture": the decode round
 * with an anchor; LFM2.5-DSpark post, "How DSpark works": all drafted tokens
 * are verified in one forward pass of the target):
 *   B requests; request r has C_r committed positions in its paged KV cache,
 *   an anchor token a_r (the last emitted token, not yet cached) and L_r
 *   drafts d_{r,1..L_r}. The target decoder runs once over the M = sum(L_r+1)
 *   rows [a_r, d_{r,1}, .., d_{r,L_r}] at absolute positions C_r .. C_r+L_r,
 *   each row attending to the cached context and to the block rows before
 *   it. Acceptance then keeps the longest agreeing prefix of the drafts —
 *   greedy match at temperature 0 (LFM2.5-DSpark post, "Quality parity"),
 *   rejection sampling above it (DSpark summary, "Problem") — and emits one
 *   more token: the target's correction at the first rejection, or a bonus
 *   token when every draft is accepted. The KV rows of the anchor and the
 *   accepted drafts are committed: seq_len[r] += accepted_len[r] + 1.
 *
 * The target is a Llama-style pre-norm decoder (RMSNorm, GQA attention with
 * rotate-half RoPE, SwiGLU MLP, untied LM head). Its weights are float32,
 * bf16, or W12: bf16 stored losslessly as three 4-bit planes and rebuilt in
 * registers inside the matrix kernels (SpecPilot digest, "Reasons").
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" are CUDA device pointers on the current
 *     device; "host" pointers are ordinary host memory. The library never
 *     takes ownership of caller memory; the caller keeps it alive until the
 *     work queued on `stream` has finished.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). Calls queue work on it and return without waiting, except
 *     where a function says it synchronizes.
 *   - Every function returns an sv_status. Argument errors are detected on
 *     the host before anything is queued and leave no side effects.
 *     sv_last_error() gives a message for the last failure on this thread.
 *   - The library never aborts the process and never traps on the device.
 *     Device-side checks (token ids, page ids) record a status word that
 *     sv_model_sync_status() reads back; the offending rows are skipped.
 *   - Models and their tensor maps hold device addresses of the context they
 *     were made in. cudaDeviceReset ends that context: destroy every model
 *     before it.
 */
#ifndef SV_H
#define SV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1,       /* a size, pointer or option is out of range */
  SV_ERR_NOT_REPRESENTABLE = 2, /* W12: a value is not a normal number or the exponent window exceeds 16 binades */
  SV_ERR_KV_CAPACITY = 3,       /* a request's block did not fit its page table or max_seq_len (device-detected) */
  SV_ERR_OUT_OF_MEMORY = 4,     /* workspace allocation failed */
  SV_ERR_CUDA = 5,              /* a CUDA runtime/driver call failed; see sv_last_error() */
  SV_ERR_DEVICE_CHECK = 6,      /* a device-side check failed (bad token or page id) */
  SV_ERR_UNSUPPORTED = 7        /* a configuration this build does not implement */
} sv_status;

typedef enum {
  SV_F32 = 0,   /* float32 weights, float32 activations and KV cache */
  SV_BF16 = 1,  /* bf16 weights and KV cache; activations near float32 (hi/lo bf16 operand pairs) */
  SV_W12 = 2    /* W12 matrices (lossless bf16); otherwise as SV_BF16 */
} sv_dtype;

/* Model configuration. */
typedef struct {
  int32_t n_layers;
  int32_t d_model;
  int32_t n_heads;       /* query heads */
  int32_t n_kv_heads;    /* key/value heads; n_heads % n_kv_heads == 0 */
  int32_t head_dim;      /* 64 or 128 */
  int32_t ffn;           /* SwiGLU hidden size */
  int32_t vocab;
  float rope_theta;      /* RoPE base */
  float rms_eps;         /* RMSNorm epsilon */
  int32_t weight_dtype;  /* sv_dtype */
  int32_t max_batch;     /* largest B passed to sv_verify */
  int32_t max_gamma;     /* largest L_r (drafts per request, anchor excluded), 0 .. 255 */
  int32_t page_size;     /* KV positions per page: 16 */
  int32_t max_seq_len;   /* largest absolute position + 1 that any row may take */
  int32_t flags;         /* SV_FLAG_* */
} sv_config;

/* Also write the full float32 logits [M][vocab] of every verify into the
 * model's workspace (readable with sv_model_logits). Sampled verifies always
 * keep them. */
#define SV_FLAG_KEEP_LOGITS 1
/* Launch the step's kernels one after another, each starting when the one
 * before it has finished. By default every kernel is a programmatic dependent
 * of the previous one, so its prologue (barrier set-up, its first weight
 * loads) overlaps the end of that kernel. With this flag the step is slower,
 * but per-kernel event timing (sv_model_set_timing) adds up to the step. */
#define SV_FLAG_NO_PDL 2
/* Run every matrix product of the step on the CUDA cores (the warp-level FMA
 * kernel that float32 models use) instead of the tensor cores, for bf16/W12
 * models too. Same results within the bf16 tolerance; for measuring where
 * the tensor-core path starts to pay (small M). */
#define SV_FLAG_CUDA_CORE_GEMM 4

/* A weight matrix [rows][cols] (the output-major layout y = x W^T).
 * F32/BF16: `data` is a dense row-major device array of that type; the other
 *      fields are unused (0 / NULL).
 * W12: `data` holds plane 0, plane 1, plane 2 back to back, each
 *      sv_w12_plane_bytes(rows, cols) bytes (see sv_pack_w12), and `base` is
 *      the tensor's exponent base; row_bases, esc_off and esc are NULL.
 * Grouped W12 (sv_pack_w12_grouped): the same planes, `base` unused, and the
 *      device arrays row_bases [sv_w12_row_blocks(rows)], esc_off
 *      [sv_w12_tiles(rows, cols) + 1] and esc [esc_off[tiles]]. */
typedef struct {
  const void* data;
  int32_t base;
  const uint8_t* row_bases;
  const int32_t* esc_off;
  const uint32_t* esc;
} sv_matrix;

/* One decoder layer. Norm gains are float32 for SV_F32 models, bf16 otherwise. */
typedef struct {
  const void* attn_norm;  /* device [d_model] */
  sv_matrix wqkv;         /* [(n_heads + 2 n_kv_heads) head_dim][d_model]: q rows, then k rows, then v rows */
  sv_matrix wo;           /* [d_model][n_heads head_dim] */
  const void* mlp_norm;   /* device [d_model] */
  sv_matrix wgu;          /* [2 ffn][d_model]: gate rows, then up rows */
  sv_matrix wd;           /* [d_model][ffn] */
} sv_layer_weights;

typedef struct {
  const void* embed;               /* device [vocab][d_model]; float32 for SV_F32 models, bf16 otherwise */
  const void* final_norm;          /* device [d_model] */
  sv_matrix lm_head;               /* [vocab][d_model] */
  const sv_layer_weights* layers;  /* host array [n_layers]; copied by sv_model_create */
} sv_weights;

/* Paged KV cache. Pages of all requests come from one pool per layer.
 * K and V page pools of layer l: device [n_pages][n_kv_heads][page_size][head_dim],
 * float32 for SV_F32 models, bf16 otherwise. Position p of request r lives in
 * page page_table[r][p / page_size], slot p % page_size. */
typedef struct {
  void* const* k;              /* host array [n_layers] of device pointers */
  void* const* v;              /* host array [n_layers] of device pointers */
  int32_t n_pages;
  const int32_t* page_table;   /* device [batch][max_pages_per_seq] */
  int32_t max_pages_per_seq;
  int32_t* seq_len;            /* device [batch]: C_r in, C_r + accepted_len + 1 out */
} sv_kv;

typedef struct sv_model sv_model;

/* Create a model. The weight pointers are borrowed (not copied) and must
 * outlive the model; the layer array itself is copied. Allocates the
 * workspace for max_batch * (1 + max_gamma) rows and the RoPE table on the
 * current device, and queues their initialization on `stream`. */
sv_status sv_model_create(const sv_config* cfg, const sv_weights* weights, void* stream, sv_model** out);
void sv_model_destroy(sv_model* model);

/*
 * The verify step.
 *   batch        B, 1 <= B <= max_batch.
 *   tokens       device int32 [B][1 + max_gamma]: column 0 the anchor a_r,
 *                columns 1..L_r the drafts; other columns are ignored.
 *   verify_lens  HOST int32 [B]: L_r in 0..max_gamma. It is a host array
 *                because the launch shapes of every kernel depend on
 *                M = sum(L_r + 1), and the scheduler that chooses L_r runs on
 *                the host (DSpark summary, "Architecture", the prefix
 *                scheduler).
 *   kv           the paged cache; rows C_r..C_r+L_r must have pages.
 *   draft_probs  device float32 [B][max_gamma][vocab]: q_i, the distribution
 *                d_i was drawn from. Required when temperature > 0, ignored
 *                (may be NULL) when temperature == 0.
 *   temperature  0: greedy match; >= 1e-6: rejection sampling with target
 *                p = softmax(z / temperature): accept d_i iff
 *                u_i * q_i(d_i) < p_{i-1}(d_i); at the first rejection emit a
 *                draw from max(0, p_{i-1} - q_i) normalized, else a draw from
 *                p_{L_r}; draws by inverse CDF in token order.
 *   seed, request_ids (device int64 [B], or NULL for ids 0..B-1): Philox4x32-10
 *                key (seed) and counter (position, stream, request id) of the
 *                uniforms; position = absolute position of the emitted token,
 *                stream 0 = accept test, 1 = draw.
 *   accepted_len device int32 [B] out: k_r, the accepted drafts.
 *   next_token   device int32 [B] out: the correction or bonus token.
 * Writes the K/V of all M rows into their page slots, then commits
 * seq_len[r] += k_r + 1 (rows past the accepted prefix are left to be
 * overwritten). Asynchronous on `stream`.
 * CUDA graphs: every per-call choice is made on the host from B, verify_lens
 * and the model, and only kernels are launched, so after one call with the
 * same B, verify_lens, pointers, temperature and seed (all fixed in the graph),
 * a call made while `stream`
 * is being captured records the whole step (programmatic dependencies
 * included); replaying it recomputes with the current contents of the
 * captured buffers (tokens, seq_len, draft_probs, KV pools).
 * Errors: SV_ERR_INVALID_ARG (B, L_r, NULL pointers; a temperature that is
 *         negative, not finite, or positive but below 1e-6, where z / T
 *         could overflow in float32), SV_ERR_CUDA (launch failure).
 */
sv_status sv_verify(sv_model* model, int32_t batch, const int32_t* tokens, const int32_t* verify_lens,
                    const sv_kv* kv, const float* draft_probs, float temperature, uint64_t seed,
                    const int64_t* request_ids, int32_t* accepted_len, int32_t* next_token, void* stream);

/* sv_verify for callers whose per-step inputs and outputs live in host memory:
 * tokens [B][1 + max_gamma], draft_probs [B][max_gamma][vocab] (or NULL),
 * request_ids [B] (or NULL), accepted_len [B] and next_token [B] are HOST
 * pointers; the KV cache stays on the device. Copies the inputs into the
 * model's workspace, runs the step, copies the outputs back and synchronizes
 * `stream` before returning. */
sv_status sv_verify_host(sv_model* model, int32_t batch, const int32_t* tokens, const int32_t* verify_lens,
                         const sv_kv* kv, const float* draft_probs, float temperature, uint64_t seed,
                         const int64_t* request_ids, int32_t* accepted_len, int32_t* next_token, void* stream);

/*
 * Prefill (or autoregressive decode) through the verify step's kernels: the
 * target forward over the blocks [t_{r,0}, .., t_{r,L_r}] at positions
 * C_r .. C_r + L_r, committing every row: the KV of all rows is written and
 * seq_len[r] += L_r + 1. next_token[r] (device int32 out) is the greedy
 * token after the block (the argmax of row L_r's logits; lowest index on
 * ties). tokens and block_lens as in sv_verify (block_lens[r] = L_r = the
 * block's rows - 1, host, 0 .. max_gamma); a prompt longer than
 * max_gamma + 1 is fed as consecutive blocks. With L_r = 0 this is one step
 * of plain autoregressive greedy decoding (the baseline the speed-ups of
 * speculative decoding are quoted against). Asynchronous on `stream`; errors
 * as sv_verify.
 */
sv_status sv_prefill(sv_model* model, int32_t batch, const int32_t* tokens, const int32_t* block_lens,
                     const sv_kv* kv, int32_t* next_token, void* stream);

/*
 * Greedy verification of a token tree per request (SpecPilot digest,
 * "Reasons", names tree verification; this is the plain generalisation of
 * the block verify). Request r's tree has n_drafts[r] + 1 nodes: node 0 is
 * the anchor (the root), node i > 0 a draft whose parent is parents[r][i]
 * (0 <= parents[r][i] < i, so parents precede children). One target forward
 * runs over all nodes: node i sits at position C_r + depth(i) and attends to
 * the cached positions and to its own ancestors. With t_i the greedy token
 * after node i (argmax of its logits, lowest index on ties), node i is
 * correct when its token equals t_{parent(i)}; the accepted path ends at the
 * deepest node that is correct together with all its non-root ancestors (the
 * lowest index among equally deep ones). Outputs: accepted_len[r] = that
 * node's depth k, next_token[r] = t at its end, accepted_nodes[r][0..k] =
 * the path's nodes, root first. Commit: the path's keys and values are moved
 * to positions C_r .. C_r + k and seq_len[r] += k + 1.
 *
 * tokens [B][1 + max_gamma] and parents [B][1 + max_gamma]: device int32
 * (parents[r][0] is ignored); n_drafts: HOST int32 [B], 0 .. min(max_gamma,
 * 63) (at most 64 nodes per request); accepted_len, next_token [B] and
 * accepted_nodes [B][1 + max_gamma]: device int32 out. The tree's rows use
 * the KV slots C_r .. C_r + n_drafts[r] during the step, so the request must
 * have that capacity. Temperature 0 only. A parent that does not precede its
 * node is a device check (SV_ERR_DEVICE_CHECK on the next status read; the
 * node is then treated as a chain row). Asynchronous on `stream`; other
 * errors as sv_verify.
 */
sv_status sv_verify_tree(sv_model* model, int32_t batch, const int32_t* tokens, const int32_t* parents,
                         const int32_t* n_drafts, const sv_kv* kv, int32_t* accepted_len, int32_t* next_token,
                         int32_t* accepted_nodes, void* stream);

/* Copy the float32 logits [M][vocab] of the last verify (rows in request
 * order, anchor row first) to device `dst`. Valid after a sampled verify, or
 * after any verify when the model was created with SV_FLAG_KEEP_LOGITS;
 * otherwise SV_ERR_INVALID_ARG. `rows` must equal that verify's M. */
sv_status sv_model_logits(sv_model* model, float* dst, int32_t rows, void* stream);

/* Synchronize `stream`, read and clear the device status word. Since the last
 * call, if some request's block did not fit its KV capacity (a row position
 * reached max_seq_len, or its page index was past max_pages_per_seq) and
 * nothing else went wrong, returns SV_ERR_KV_CAPACITY; if a kernel saw a token
 * id outside [0, vocab), a page id outside [0, n_pages) or a wait that timed
 * out, returns SV_ERR_DEVICE_CHECK. sv_last_error() names every condition.
 * The offending rows were skipped: their KV was not written and their
 * attention ignored the missing pages; other requests are unaffected. */
sv_status sv_model_sync_status(sv_model* model, void* stream);

/* Kernel timing for measurement. When enabled, the library records CUDA
 * events around its launches on `stream` and accumulates per-kernel-class
 * device time; sv_model_timing synchronizes on the recorded events, adds
 * them up, and returns the totals (milliseconds) and launch counts of the
 * classes below since timing was last enabled. Recording events between
 * launches adds a little time to each step, so leave it off when timing
 * whole steps. */
enum { SV_KC_GEMM = 0, SV_KC_ATTENTION = 1, SV_KC_NORM = 2, SV_KC_LM_HEAD = 3, SV_KC_ACCEPT = 4, SV_KC_COUNT = 5 };
sv_status sv_model_set_timing(sv_model* model, int32_t enable);
sv_status sv_model_timing(sv_model* model, double* ms /* [SV_KC_COUNT] */, int64_t* launches /* [SV_KC_COUNT] */);

/* Per-CTA device timeline, for measurement. While records != NULL, each
 * traced kernel of a verify (the tensor-core projections, the tensor-core
 * attention and its merge) writes one record of 16 uint64 words per CTA into
 * `records` (device, capacity records, zero-filled by the caller): word 0 =
 * kind << 48 | SM id << 32 | CTA index (kinds: 1 projection, 2 attention,
 * 3 attention merge), words 1-6 = the %globaltimer value in ns when the CTA
 * started, returned from its dependency wait, had its first operands, issued
 * its last MMA, finished its epilogue, and exited (0 where a CTA has no such
 * step). Projections add, for the hand-off of the CTA's last tile: 7 the
 * accumulator ready for the epilogue, 8 its partial tile stored and fenced,
 * 9 its arrival counted, 10 the contributors' partials summed (last arriver
 * only), 11 the tile epilogue done. Launches that no longer fit are not
 * traced. Setting a new buffer (or
 * NULL, 0 to stop) restarts the count. sv_model_trace_launches writes
 * (first record, CTAs, kind) for each traced launch, in launch order, into
 * host int64 launches[3 * max_launches] and their number to *n_launches. */
sv_status sv_model_set_trace(sv_model* model, uint64_t* records, int64_t capacity);
sv_status sv_model_trace_launches(sv_model* model, int64_t* launches, int64_t max_launches, int64_t* n_launches);

/*
 * W12 codec (SpecPilot digest, "Reasons": BF16 split into three 4-bit
 * bit-planes and rebuilt bit-exactly in the GEMM's registers). The page
 * fixes no bit layout; this library's:
 *   bf16 b = s<<15 | E<<7 | m; base = min E over the tensor;
 *   code c = s<<11 | (E - base)<<7 | m (12 bits);
 *   plane p holds nibble p of c. A plane is tiled: the matrix is padded
 *   with zero codes to whole tiles of 64 rows x 128 columns; tile (rt, kt)
 *   (KT = ceil(cols/128) tiles per row block) is 4096 contiguous bytes at
 *   (rt*KT + kt)*4096, tile row r at r*64 within it. A tile row holds its
 *   128 elements in groups of 8, group q in the little-endian 32-bit word at
 *   bytes 4q..4q+3, whose nibble slot s (bits 4s..4s+3) holds element 8q+2s
 *   for s < 4 and 8q+2(s-4)+1 for s >= 4. Each tile is one contiguous read
 *   for the matrix kernels, and a shift and a mask put two elements into
 *   the two 16-bit lanes of a word.
 * A tensor is representable iff every element is a normal number (not
 * +-0, subnormal, inf or NaN) and max E - min E <= 15.
 */
int64_t sv_w12_plane_bytes(int64_t rows, int64_t cols);

/* Pack device bf16 [rows][cols] into device `planes` (3 *
 * sv_w12_plane_bytes(rows, cols) bytes, caller-allocated). Writes the base to
 * *base_out and the number of offending elements to *n_unrepresentable
 * (host). Synchronizes `stream`. Returns SV_ERR_NOT_REPRESENTABLE (planes
 * then undefined) when the tensor is not representable. */
sv_status sv_pack_w12(const uint16_t* bf16, int64_t rows, int64_t cols, uint8_t* planes, int32_t* base_out,
                      int64_t* n_unrepresentable, void* stream);

/* Rebuild device bf16 [rows][cols] from planes and base. Asynchronous. */
sv_status sv_unpack_w12(const uint8_t* planes, int32_t base, int64_t rows, int64_t cols, uint16_t* bf16_out,
                        void* stream);

/*
 * Grouped W12: any bf16 tensor, bit-exact. The planes keep the layout above;
 * each block of 64 rows (a plane tile's rows) has its own base, and the
 * elements its 16-binade window cannot hold are escapes, listed with their
 * exact pattern (and coded 0 in the planes):
 *   row_bases[rb] = max(1, (max E over the block's normal elements) - 15), or
 *     1 for a block without normal elements;
 *   an element escapes iff it is not a normal number or E < row_bases[rb];
 *   the escapes of plane tile (rb, kt) (tile i = rb * KT + kt, KT =
 *   ceil(cols / 128)) are esc[esc_off[i] .. esc_off[i + 1]), in row-major
 *   order, each entry = row in block << 23 | column in tile << 16 | pattern.
 * For N(0, 0.02) weights the escapes are the tail below 2^-16 of the block's
 * largest magnitude (about 1e-4 of the elements) and exact zeros.
 */
int64_t sv_w12_row_blocks(int64_t rows);            /* ceil(rows / 64) */
int64_t sv_w12_tiles(int64_t rows, int64_t cols);   /* row blocks x ceil(cols / 128) */

/* Pack device bf16 [rows][cols]: planes (3 * sv_w12_plane_bytes), row_bases,
 * esc_off as above (device, caller-allocated). The escapes go to `esc` (device,
 * esc_capacity entries) and their number to *n_escapes (host). With esc NULL
 * (capacity 0) only the count is computed; when the count exceeds the
 * capacity, SV_ERR_INVALID_ARG (planes, bases and offsets are still written).
 * Synchronizes `stream`. */
sv_status sv_pack_w12_grouped(const uint16_t* bf16, int64_t rows, int64_t cols, uint8_t* planes, uint8_t* row_bases,
                              int32_t* esc_off, uint32_t* esc, int64_t esc_capacity, int64_t* n_escapes,
                              void* stream);

/* Rebuild device bf16 [rows][cols] from grouped W12. Asynchronous. */
sv_status sv_unpack_w12_grouped(const uint8_t* planes, const uint8_t* row_bases, const int32_t* esc_off,
                                const uint32_t* esc, int64_t rows, int64_t cols, uint16_t* bf16_out, void* stream);

/*
 * Skinny weight-streaming matrix product y[M][N] = x[M][K] W^T with the
 * verify step's own kernels (the path every projection of the step takes):
 * W [N][K] of `wdtype` (F32, BF16 or W12 as in sv_matrix); y device float32
 * [M][N]; 1 <= M <= 4096, K a multiple of 16.
 * x (device): for F32 weights float32 [M][K] (x_planes = 1). For BF16/W12
 * weights bf16: x_planes = 1 gives one plane [M][K]; x_planes = 2 gives a hi
 * plane [M][K] followed by a lo plane [M][K] and the product uses hi + lo
 * (the verify step carries its activations this way, near float32 precision).
 * Uses `workspace` (device, at least sv_linear_workspace_bytes bytes,
 * caller-allocated, zero-filled before first use and left zeroed by every
 * call) for split-K partial sums and tile counters. Asynchronous.
 */
size_t sv_linear_workspace_bytes(int32_t wdtype, int32_t M, int32_t N, int32_t K);
sv_status sv_linear(int32_t wdtype, const sv_matrix* w, int32_t N, int32_t K, const void* x, int32_t x_planes,
                    int32_t M, float* y, void* workspace, size_t workspace_bytes, void* stream);

/*
 * sv_linear without any device allocation. The pages have no counterpart to
 * this entry point: it exists for callers that must not allocate device
 * memory while they run (cudaMalloc can synchronize the whole device and
 * stall other streams, and some hosts, such as inference servers with fixed
 * memory pools or plugins whose host owns every allocation, forbid it).
 * The same arguments as sv_linear, without the workspace. It always runs the
 * CUDA-core (FMA) plan of the product, whatever the weight type: its result
 * equals sv_linear's within rounding (not bit for bit, since sv_linear takes
 * the tensor-core path for bf16/W12 weights), and for large bf16/W12 shapes it
 * is much slower. That plan splits K over at most 8 CTAs of one thread-block
 * cluster, which add their partial tiles in distributed shared memory, so the
 * call needs no scratch: it allocates nothing, keeps no state between calls,
 * and calls on several streams or host threads may overlap. It launches one
 * kernel on `stream` and returns (asynchronous; capturable in a CUDA graph).
 * Errors: SV_ERR_INVALID_ARG as for sv_linear; SV_ERR_CUDA when the launch
 * fails (for example N beyond 65535 tiles of 128 rows).
 */
sv_status sv_linear_noalloc(int32_t wdtype, const sv_matrix* w, int32_t N, int32_t K, const void* x,
                            int32_t x_planes, int32_t M, float* y, void* stream);

/* Philox4x32-10 uniforms of the verify step: out[i] = u(seed, request_id,
 * position0 + i, stream_id) for i < n, device float32. Asynchronous. */
sv_status sv_philox_uniform(uint64_t seed, int64_t request_id, int64_t position0, int32_t stream_id, int32_t n,
                            float* out, void* stream);

/*
 * Hardware-aware prefix scheduler (DSpark summary, "Confidence-Scheduled
 * Verification"): choose every request's verify length from its draft
 * confidences and the measured step cost, to maximize the throughput
 * Theta = tau / T(M), tau = sum_r (1 + sum_{j <= L_r} a_{r,j}) the expected
 * tokens of the step, a_{r,j} = prod_{i <= j} c_{r,i} the survival
 * probability of draft j, M = sum_r (L_r + 1) the verified rows.
 *   conf        HOST float [batch][gamma]: c_{r,i} in [0, 1], the probability
 *               that draft i passes given drafts 1 .. i-1 did.
 *   step_us     HOST float [n_cost]: step_us[M - 1] = verify-step time for M
 *               rows (for example a bench sweep); n_cost >= batch. M past the
 *               table is never chosen.
 *   early_stop  nonzero: stop at the first admission that lowers Theta (the
 *               optimum when Theta is unimodal in M); zero: scan every M.
 *   verify_lens HOST int32 out [batch]: the chosen L_r.
 *   expected_tokens, throughput: HOST out (may be NULL): tau and Theta in
 *               tokens per second.
 * A global sort of the a_{r,j} admitted greedily visits the best choice of
 * drafts for every M (a_{r,j} never increases in j, so the M - B largest form
 * a prefix of each request's drafts). Host only; no GPU work.
 * Errors: SV_ERR_INVALID_ARG (sizes, NULL pointers, a confidence outside
 * [0, 1], a cost that is not finite and positive).
 */
sv_status sv_schedule_prefix(int32_t batch, int32_t gamma, const float* conf, const float* step_us, int32_t n_cost,
                             int32_t early_stop, int32_t* verify_lens, double* expected_tokens, double* throughput);

/* Message of the last failed call on this thread ("" if none). */
const char* sv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SV_H */
