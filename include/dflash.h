/*
 * dflash.h -- C ABI of a GB300 (sm_103a) library for one DFlash
 * speculative-decoding step: fuse -> inject -> draft -> verify -> accept ->
 * rollback.  Every stage runs as CUDA kernels of this library on the stream
 * the caller passes; the host only validates arguments and enqueues work.
 *
 * Sources (page titles as printed on the pages):
 *   [DD] "DFlash 深度解析：块扩散模型如何让 LLM 推理加速 6 倍——2026 投机解码完全指南"
 *        (chenxutan.com): §1.1 autoregressive decoding, §1.2 speculative
 *        decoding, §2.2 feature_fusion / kv_injection / draft_inference,
 *        §3.3 shared embedding and LM head, §5.1 one-forward block drafting,
 *        §8.2 linear verification.
 *   [LC] "从 ICML 论文到你的显卡：llama.cpp 吞下 DFlash，本地推理进入 2 倍速时代"
 *        (arex-research.com): KV injection into every drafter layer; keep the
 *        matching prefix, cut at the first error.
 *   [RD] "我在llama.cpp中测试了最新合并的DFlash在Qwen 3.6 27B本地AI上的表现"
 *        (bittide.aicompass.dev): greedy verification is lossless.
 *
 * Conventions
 *   - All pointers to tensors are DEVICE pointers owned by the caller unless
 *     stated otherwise; the library never frees them.  Row-major throughout.
 *   - Matrices are nn.Linear [out_features][in_features].
 *   - Element type of weights, KV caches, hidden states and captured states
 *     is the model's dtype (DFLASH_F32 or DFLASH_BF16); residual stream,
 *     logits and all reductions are float32.
 *   - Positions and lengths live on the device (per-sequence int32), so every
 *     call can be captured into a CUDA graph and replayed step after step.
 *   - Return values: DFLASH_OK (0) or a negative DFLASH_ERR_* code from the
 *     synchronous argument checks or from a failed CUDA launch.  Conditions
 *     detected inside kernels (capacity overflow, non-finite logits, a wait
 *     that ran out) set bits in the workspace's device status word, read with
 *     dflash_status(); kernels never trap.
 *   - Calls are asynchronous on `stream` and not thread-safe on one cache or
 *     workspace.
 */
#ifndef DFLASH_H_
#define DFLASH_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dflash_stream_t; /* = cudaStream_t */

enum {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = -1,
  DFLASH_ERR_UNSUPPORTED_SHAPE = -2,
  DFLASH_ERR_CUDA = -3,
  DFLASH_ERR_OOM = -4,
  DFLASH_ERR_TOO_LARGE = -5, /* a size above an entry point's fixed maximum */
};

/* device status bits (dflash_status) */
enum {
  DFLASH_STATUS_CAPACITY = 1,  /* a write beyond a cache's capacity was skipped */
  DFLASH_STATUS_NONFINITE = 2, /* a logit row held NaN/Inf */
  DFLASH_STATUS_TIMEOUT = 4,   /* a pipeline wait gave up (kernel returned early) */
  DFLASH_STATUS_BOUNDS = 8,    /* an index (token id, reference position) was out of range */
};

enum { DFLASH_F32 = 0, DFLASH_BF16 = 1 };

/* Dimensions of one decoder (target or drafter). head_dim: 64 or 128. */
typedef struct dflash_model_desc {
  int32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
  float rope_theta, rms_eps;
  int32_t dtype; /* DFLASH_F32 | DFLASH_BF16 */
} dflash_model_desc;

/* One pre-norm decoder layer.
 *   wqkv      [(nq + 2 nkv) * hd][H]  rows: q heads, then k heads, then v heads
 *   wo        [H][nq * hd]
 *   w_gate_up [2F][H]  row 2f is gate row f, row 2f+1 is up row f
 *   w_down    [H][F]
 *   attn_norm, ffn_norm [H] RMSNorm gains */
typedef struct dflash_layer_w {
  const void *attn_norm, *wqkv, *wo, *ffn_norm, *w_gate_up, *w_down;
} dflash_layer_w;

/* Target model.  capture[5]: 0-based layers whose output residual stream is
 * captured for feature fusion ([DD] §2.2: 5 layers from 2 to the
 * third-from-last, see dflash_capture_layers). */
typedef struct dflash_target {
  dflash_model_desc d;
  const void *embed;      /* [V][H] */
  const void *final_norm; /* [H] */
  const void *lm_head;    /* [V][H] */
  const dflash_layer_w *layers; /* HOST array of d.n_layers entries */
  int32_t capture[5];
} dflash_target;

/* Block-diffusion drafter.  It reuses the target's embedding and LM head
 * ([DD] §3.3).  w_kv_all packs, for every drafter layer l in order, that
 * layer's k rows then v rows of wqkv: [Ld * 2 * nkv * hd][H]; it holds the
 * same values as the layers' wqkv and lets one product project the fused
 * feature for all layers ([DD] §5.2 dflash_feature_injection).
 * cross_ctx: the drafter's cross-context window W ("如何使用 DFlash 试探式解码
 * 加速本地 LLM", §7, --spec-dflash-cross-ctx): W > 0 makes every drafter layer
 * attend only to the W most recent injected positions P-W..P-1 (all of them
 * when P <= W) plus the block's own rows; 0 attends to the whole context. */
typedef struct dflash_draft {
  dflash_model_desc d;
  const void *w_fc;       /* [H][5H] fusion Linear ([DD] §2.2 feature_fusion) */
  const void *fc_norm;    /* [H] fusion RMSNorm gain */
  const void *final_norm; /* [H] */
  const dflash_layer_w *layers; /* HOST array of d.n_layers entries */
  const void *w_kv_all;
  int32_t mask_id;
  int32_t cross_ctx;
} dflash_draft;

/* ------------------------------------------------------------------ caches
 * A KV cache holds, for `batch` sequences and `n_layers` layers, keys and
 * values [layer][seq][kv_head][capacity][head_dim] in the model dtype, a
 * device int32 length per sequence (starts at 0), and a float32 RoPE
 * cos/sin table for positions 0..capacity-1 (computed on the host in double
 * precision).  Library-owned device memory (cudaMalloc); free with
 * dflash_cache_free.  The target cache's length is the committed length P;
 * the drafter cache's length is the number of injected context rows.
 * Positions >= length are scratch: target_verify writes the block there and
 * dflash_draft_block writes its block's keys/values there. */
typedef struct dflash_cache dflash_cache;

int dflash_cache_alloc(const dflash_model_desc *d, int32_t n_layers, int32_t batch,
                       int32_t capacity, dflash_cache **out);

/* Storage of a cache's keys and values. */
enum { DFLASH_KV_MODEL = 0, DFLASH_KV_Q8 = 1 };
/* dflash_cache_alloc with a storage format.  DFLASH_KV_MODEL: the model dtype
 * (as dflash_cache_alloc).  DFLASH_KV_Q8 (bf16 models with head_dim 128; the
 * 8-bit K/V cache of DFlash 深度解析 §8.3 "显存优化" 方案3 and the
 * quantised cache types the datacamp tutorial runs, §5/§7, read as stated in
 * the oracle): each key or value row of 128 entries is kept as 8-bit codes
 * u = q + 128 (q in [-127, 127]) [layer][seq][kv_head][capacity][128] uint8
 * and one float32 scale s per row [layer][seq][kv_head][capacity]; the entry
 * is q * s, quantised from the float32 row x as s = max|x| / 127,
 * q = round-half-even(x / s) (a zero row keeps s = 0).  target_verify writes
 * its rows this way before attention reads them.  Attention computes in IEEE
 * half precision: the query is half, and each entry is read as the half
 * product of q and s rounded to half, half(q * half(s)).  Target caches only: the drafter's cache,
 * tree verification (target_verify_tree, dflash_accept_tree) and the fp32
 * configuration return DFLASH_ERR_UNSUPPORTED_SHAPE with a q8 cache.  A q8
 * cache's capacity is rounded up to a multiple of 8 positions. */
int dflash_cache_alloc_ex(const dflash_model_desc *d, int32_t n_layers, int32_t batch,
                          int32_t capacity, int32_t kv_format, dflash_cache **out);
/* The cache's storage format (DFLASH_KV_MODEL or DFLASH_KV_Q8), or -1. */
int32_t dflash_cache_kv_format(const dflash_cache *c);
int dflash_cache_free(dflash_cache *c);
/* A view of sequences [seq_begin, seq_begin + seq_count) sharing memory with
 * `c` (used to prefill a ragged batch one sequence at a time).  Free views
 * with dflash_cache_free before freeing their parent. */
int dflash_cache_view(dflash_cache *c, int32_t seq_begin, int32_t seq_count, dflash_cache **out);
/* Device pointer to the int32 lengths [batch] (for the caller to read). */
int32_t *dflash_cache_lengths(dflash_cache *c);
/* Synchronises `stream` and copies min(n, batch) lengths to host memory. */
int dflash_cache_get_lengths(dflash_cache *c, int32_t *host_out, int32_t n, dflash_stream_t stream);
/* Copy keys and values of positions [pos0, pos0 + n) of one layer and one
 * sequence from (write) or to (read) caller device buffers k, v laid out
 * [n_kv][n][head_dim] in the cache dtype.  Asynchronous device-to-device
 * copies; lengths are not changed.  Used to load a saved context. */
int dflash_cache_write(dflash_cache *c, int32_t layer, int32_t seq, int32_t pos0, int32_t n,
                       const void *k, const void *v, dflash_stream_t stream);
int dflash_cache_read(dflash_cache *c, int32_t layer, int32_t seq, int32_t pos0, int32_t n, void *k,
                      void *v, dflash_stream_t stream);
/* q8 caches: dflash_cache_write takes bf16 rows and quantises them on the
 * device (same rule as target_verify's writes); dflash_cache_read returns
 * DFLASH_ERR_INVALID_ARG, and dflash_cache_read_q8 copies the stored codes
 * u (uint8 [n_kv][n][128]) and scales (float32 [n_kv][n]) instead.  Either
 * output pair may be NULL. */
int dflash_cache_read_q8(dflash_cache *c, int32_t layer, int32_t seq, int32_t pos0, int32_t n,
                         void *k_codes, void *v_codes, float *k_scales, float *v_scales,
                         dflash_stream_t stream);
/* Copy every key, value (codes and scales for q8) and length of `src` into
 * `dst`, two caches (not views) of identical geometry and storage format
 * (asynchronous device-to-device copies). */
int dflash_cache_copy(dflash_cache *dst, const dflash_cache *src, dflash_stream_t stream);
/* Set the first n lengths from host memory (asynchronous). */
int dflash_cache_set_lengths(dflash_cache *c, const int32_t *host_len, int32_t n,
                             dflash_stream_t stream);
/* Set every length to 0 (asynchronous). */
int dflash_cache_reset(dflash_cache *c, dflash_stream_t stream);

/* --------------------------------------------------------------- workspace
 * Library-owned scratch for activations, split-K partial sums, attention
 * partials and the device status word.  Sized for both models, for up to
 * `max_rows` rows per call (batch x rows-per-sequence, <= 128) and contexts
 * up to `max_ctx` positions.  One workspace serves one stream at a time. */
typedef struct dflash_workspace dflash_workspace;

int dflash_workspace_alloc(const dflash_model_desc *target, const dflash_model_desc *draft,
                           int32_t max_rows, int32_t max_ctx, dflash_workspace **out);
int dflash_workspace_free(dflash_workspace *w);
/* Synchronises `stream`, returns the status bits in *status_out and clears them. */
int dflash_status(dflash_workspace *w, dflash_stream_t stream, int32_t *status_out);
/* Device pointer to one of the workspace's float32 logit buffers, row-major
 * [rows][vocab]: which = 0 the target's, written by target_verify (rows =
 * batch * n); which = 1 the drafter's, written by dflash_draft_block (rows =
 * batch * block).  Each holds the last RMSNorm'd residual times the LM head
 * ([DD] §1.1 next-token scores; §3.3 the drafter shares the head) until the
 * next such call on the workspace.  Owned by the workspace; NULL for a NULL
 * workspace or another `which`.  No synchronisation: read it on the stream. */
float *dflash_workspace_logits(dflash_workspace *w, int32_t which);
/* Failure-path testing: sets the limit, in nanoseconds, of the waits in the
 * main loop of the weight-product kernel (ring slots and accumulator) for
 * launches enqueued afterwards; a negative value restores the default of
 * 500 ms.  A limit of 0 expires at once, so the kernel gives up, sets
 * DFLASH_STATUS_TIMEOUT, still waits (with the default limit) for its copies
 * and products in flight, writes no result and returns.  Process-wide; not an
 * operation of the method. */
int dflash_debug_set_wait_limit(int64_t ns);
const char *dflash_strerror(int code);

/* Captured layers for a target of n_layers: 5 layers spread uniformly from
 * layer 2 to layer n_layers-3 ([DD] §2.2 feature_fusion), rounded half up. */
int dflash_capture_layers(int32_t n_layers, int32_t out[5]);

/* ------------------------------------------------------------------ stages
 * Sequence state shared by the stages (device int32 arrays, caller-owned):
 *   anchor[batch]  last emitted token; it sits at position P
 *   n_pend[batch]  captured rows not yet injected into the drafter cache;
 *                  they belong to positions P - n_pend .. P - 1
 * Invariant outside a stage: drafter length + n_pend == target length == P.
 * A step is: fuse + inject the pending rows, draft, verify, accept/rollback. */

/* Feature fusion ([DD] §2.2 feature_fusion): fused = RMSNorm(hcap · w_fcᵀ)
 * ⊙ fc_norm for `rows` rows.  hcap [rows][5H] holds the captured hidden
 * states of the 5 layers side by side (the concat); fused [rows][H]. */
int dflash_fuse_features(const dflash_draft *dr, const void *hcap, int32_t rows, void *fused,
                         dflash_workspace *ws, dflash_stream_t stream);

/* KV injection ([DD] §2.2 kv_injection, §5.2; [LC]): for every drafter layer
 * l, K = RoPE(fused · W_k,lᵀ) and V = fused · W_v,lᵀ are appended to layer
 * l's cache.  fused is [batch][rows_per_seq][H]; sequence b injects its first
 * n_pend[b] rows at positions len[b] .. len[b] + n_pend[b] - 1 of
 * draft_cache, then len[b] += n_pend[b] and n_pend[b] = 0 (the rows are
 * consumed). */
int dflash_inject_kv(const dflash_draft *dr, const void *fused, int32_t batch, int32_t rows_per_seq,
                     int32_t *n_pend, dflash_cache *draft_cache, dflash_workspace *ws,
                     dflash_stream_t stream);

/* Block drafting ([DD] §5.1, §2.2 draft_inference): one non-causal forward of
 * the block [anchor, MASK x (block-1)] at positions P .. P+block-1 (P = the
 * drafter cache length) through every drafter layer; each row attends to the
 * injected context 0..P-1 and to all block rows.  Tokens are embedded and
 * decoded with the target's embedding and LM head ([DD] §3.3).  Writes
 * draft_tokens[b][0] = anchor[b] and draft_tokens[b][j] = argmax of row j
 * (j >= 1).  block in [2, 16]. */
int dflash_draft_block(const dflash_draft *dr, const dflash_target *tg, const int32_t *anchor,
                       int32_t batch, int32_t block, dflash_cache *draft_cache,
                       int32_t *draft_tokens, dflash_workspace *ws, dflash_stream_t stream);

/* Target forward ([DD] §1.1, §1.2): tokens [batch][n] at positions
 * P .. P+n-1 (P = target cache length), causal, keys/values written into the
 * cache at those positions.  Outputs per row: argmax [batch][n] (lowest index
 * on ties), top2_gap [batch][n] (nullable; largest minus second-largest
 * logit) and hcap [batch][n][5H] (nullable), the residual stream after each
 * captured layer.  n in [1, 128], batch * n <= workspace max_rows.
 *   commit = 0  verification: lengths untouched (dflash_accept_rollback decides)
 *   commit = 1  prefill chunk: len += n, n_pend = n
 *   commit = 2  as 1, and the last row's greedy token becomes the anchor and
 *               is appended to the stream (last chunk of a prefill, or one
 *               autoregressive step) -- anchor/n_pend/stream may be NULL for
 *               commit = 0. */
int target_verify(const dflash_target *tg, const int32_t *tokens, int32_t batch, int32_t n,
                  int32_t commit, dflash_cache *target_cache, int32_t *argmax, float *top2_gap,
                  void *hcap, int32_t *anchor, int32_t *n_pend, int32_t *stream,
                  int32_t *stream_len, int32_t stream_cap, dflash_workspace *ws,
                  dflash_stream_t cuda_stream);

/* Acceptance and rollback ([DD] §1.2, §8.2; [LC]).  For each sequence b:
 *   a = the number of leading drafted tokens draft_tokens[b][i] (i >= 1) that
 *       equal the target's greedy choice argmax[b][i-1], stopping at the
 *       first mismatch (0 <= a <= block-1);
 *   emitted: argmax[b][0..a] (a drafted tokens + the target's own next token)
 *       are appended to stream[b][*] at stream_len[b] (capacity stream_cap);
 *   rollback: target len[b] = P + a + 1 (rows beyond are discarded in place,
 *       no data moves), anchor[b] = argmax[b][a], n_pend[b] = a + 1.
 * accept_len[batch] receives a (nullable). */
int dflash_accept_rollback(const int32_t *draft_tokens, const int32_t *argmax, int32_t batch,
                           int32_t block, dflash_cache *target_cache, int32_t *anchor,
                           int32_t *n_pend, int32_t *accept_len, int32_t *stream,
                           int32_t *stream_len, int32_t stream_cap, dflash_workspace *ws,
                           dflash_stream_t cuda_stream);

/* Teacher forcing (benchmark harness for random-init models, whose natural
 * acceptance is ~0).  For sequence b at step s = *step (device counter,
 * incremented by this call): k = k_draw[s][b], r = r_draw[s][b],
 * e = stream_len[b]; slots j = 1..min(k, block-1) take ref[b][e+j-1]; if
 * k+1 <= block-1, slot k+1 takes (ref[b][e+k] + 1 + r) mod vocab, which
 * differs from the reference; other slots keep the drafter's tokens.  With
 * ref the greedy stream, exactly min(k, block-1) drafts are then accepted. */
int dflash_teacher_force(int32_t *draft_tokens, int32_t batch, int32_t block, const int32_t *ref,
                         int32_t ref_stride, int32_t ref_len, const int32_t *stream_len,
                         const int32_t *k_draw, const int32_t *r_draw, int32_t max_steps,
                         int32_t *step, int32_t vocab, dflash_workspace *ws, dflash_stream_t stream);

/* ------------------------------------------------------ tree verification
 * "DFlash 深度解析" §8.2 (DDTree): one target forward explores several
 * branches of the drafter's guesses within a node budget instead of one
 * chain; the page prints no algorithm.  These calls take the following
 * reading (greedy):
 *   - candidates: per drafted slot j = 1..block-1, the drafter's top-K tokens
 *     by log-probability log q_j (softmax of the slot's logits; ties to the
 *     lower id);
 *   - the tree: the `budget` highest-scoring token prefixes, a prefix scoring
 *     the sum of its tokens' log q (best-first; every prefix's parent scores at
 *     least as high, so they form a tree rooted at the anchor); ties to the
 *     smaller depth, then the smaller rank, then the earlier parent;
 *   - verification: one target forward over the n = budget + 1 nodes (node 0
 *     the anchor), node i at position P + depth(i), attending to the context
 *     and to its own ancestors (itself included);
 *   - acceptance: from the root, move to the child whose token equals the
 *     target's greedy token after the current node while there is one; emit
 *     the path's tokens and the greedy token after its last node.
 * With K = 1 and budget = block - 1 the tree is the drafter's greedy chain and
 * the step equals linear verification.  Trees hold at most 64 nodes
 * (budget <= 63).  Per-sequence arrays are [batch][n], device memory owned by
 * the caller; tree_mask[b][i] has bit j set for every ancestor j of node i and
 * for i itself. */

/* After dflash_draft_block: build each sequence's tree from the drafter's
 * logits (workspace buffer 1).  topk in [1, 8]; budget in [1, 63] and at most
 * the number of prefixes the candidates allow, else DFLASH_ERR_INVALID_ARG. */
int dflash_draft_tree(const int32_t *anchor, int32_t batch, int32_t block, int32_t vocab, int32_t topk,
                      int32_t budget, int32_t *tree_tokens, int32_t *tree_parent, int32_t *tree_depth,
                      uint64_t *tree_mask, dflash_workspace *ws, dflash_stream_t stream);
/* Target forward of the trees (n = budget + 1 rows per sequence) at
 * positions P + depth, ancestor-masked; keys/values are written at the scratch
 * slots P .. P + n - 1 in node order; argmax [batch][n], top2_gap (nullable),
 * hcap [batch][n][5H] (nullable); lengths untouched. */
int target_verify_tree(const dflash_target *tg, const int32_t *tree_tokens, const int32_t *tree_depth,
                       const uint64_t *tree_mask, int32_t batch, int32_t n, dflash_cache *target_cache,
                       int32_t *argmax, float *top2_gap, void *hcap, dflash_workspace *ws,
                       dflash_stream_t cuda_stream);
/* The walk and the rollback: the accepted path's a drafted tokens and the
 * bonus are appended to stream; the path's keys/values (every target layer)
 * move from their node slots to positions P .. P + a and its captured rows
 * (hcap, nullable, [batch][n][5H]) to rows 0 .. a of the sequence's block;
 * len += a + 1, anchor = the bonus, n_pend = a + 1, accept_len = a
 * (nullable). */
int dflash_accept_tree(const dflash_target *tg, const int32_t *tree_tokens, const int32_t *tree_parent,
                       const int32_t *argmax, int32_t batch, int32_t n, dflash_cache *target_cache, void *hcap,
                       int32_t *anchor, int32_t *n_pend, int32_t *accept_len, int32_t *stream,
                       int32_t *stream_len, int32_t stream_cap, dflash_workspace *ws,
                       dflash_stream_t cuda_stream);

/* ------------------------------------------------------------ sampling mode
 * "DFlash 深度解析" §4.2: the speed-up holds at temperature 1 with the
 * output distribution unchanged; the page gives no rule.  These calls take
 * the standard speculative-sampling rule: with p_i = softmax(target logits of
 * row i / T) and q_j = softmax(drafter logits of slot j / T),
 *   - the drafter's slot j >= 1 is drawn from q_j;
 *   - drafted token d_i (i = 1..block-1) is accepted when u_i q_i(d_i) <
 *     p_{i-1}(d_i) (probability min(1, p/q)), stopping at the first rejection;
 *   - after a accepted drafts one more token is drawn: from the residual
 *     max(0, p_a - q_{a+1}) (renormalised; from p_a when it has no mass) when
 *     a < block-1, from p_{block-1} otherwise.
 * A draw from weights w with uniform v in [0, 1) is the smallest index whose
 * running sum exceeds v * sum(w); uniform numbers are caller-supplied device
 * float32 arrays.  Softmax statistics and running sums are float32 in a fixed
 * order.  temperature must be finite and > 0, else DFLASH_ERR_INVALID_ARG. */

/* After dflash_draft_block: draft_tokens[b][j] (j = 1..block-1) drawn from
 * the drafter's logits (workspace buffer 1) at temperature T with
 * w[b][j-1] ([batch][block-1]); slot 0 keeps the anchor. */
int dflash_draft_sample(int32_t batch, int32_t block, int32_t vocab, float temperature, const float *w,
                        int32_t *draft_tokens, dflash_workspace *ws, dflash_stream_t stream);
/* After target_verify of the drafted block (commit = 0): verification by the
 * rule above with u [batch][block-1] and v [batch], then the same rollback as
 * dflash_accept_rollback: emitted = d_1..d_a and the drawn token (a + 1
 * tokens) appended to stream; target len += a + 1; anchor = the drawn token;
 * n_pend = a + 1; accept_len[b] = a (nullable).  Reads both workspace logit
 * buffers; a drafted id outside [0, vocab) sets DFLASH_STATUS_BOUNDS and stops
 * that sequence's acceptance there. */
int dflash_accept_sample(const int32_t *draft_tokens, int32_t batch, int32_t block, int32_t vocab,
                         float temperature, const float *u, const float *v, dflash_cache *target_cache,
                         int32_t *anchor, int32_t *n_pend, int32_t *accept_len, int32_t *stream,
                         int32_t *stream_len, int32_t stream_cap, dflash_workspace *ws,
                         dflash_stream_t cuda_stream);
/* One draw per row of float32 logits [rows][vocab] at temperature T with
 * v[rows]: out[rows] (autoregressive sampling, the prefill's first token). */
int dflash_sample(const float *logits, int32_t rows, int32_t vocab, float temperature, const float *v,
                  int32_t *out, dflash_workspace *ws, dflash_stream_t stream);

/* -------------------------------------------------------- building blocks
 * The kernels behind the stages, exposed for unit parity tests. */

/* y[n][m] = sum_k x[n][k] w[m][k]; x [rows][K] (dtype), w [M][K] (dtype),
 * y [rows][M] float32.  rows <= 128. */
int dflash_linear(int32_t dtype, const void *x, const void *w, float *y, int32_t rows, int32_t M,
                  int32_t K, dflash_workspace *ws, dflash_stream_t stream);
/* y = x / sqrt(mean(x^2) + eps) * gain, x float32 [rows][H] -> y dtype. */
int dflash_rmsnorm(int32_t dtype, const float *x, const void *gain, void *y, int32_t rows,
                   int32_t H, float eps, dflash_stream_t stream);
/* Greedy token and top-2 gap of float32 logits [rows][V] ([DD] §1.1 greedy
 * choice; lowest index on ties). */
int dflash_argmax(const float *logits, int32_t rows, int32_t V, int32_t *argmax, float *gap,
                  dflash_workspace *ws, dflash_stream_t stream);
/* dflash_argmax without a workspace.  Not an operation of the method (the
 * pages have no counterpart): the same greedy token and top-2 gap of float32
 * logits [rows][V], for callers that cannot allocate device memory.  Such
 * callers hold no dflash_workspace, whose allocation needs both model
 * descriptors and reserves activation buffers sized for them, and cannot add
 * a cudaMalloc/cudaFree of their own: a sampler handed another engine's
 * logits in a serving loop whose memory is owned by a caching allocator, or
 * a loop where cudaFree's implicit device synchronisation would stall the
 * pipeline.
 *   Scratch: a fixed file-scope device array in the library (slice partials
 *   and per-row tickets, about 33 KiB per device) for at most
 *   DFLASH_ARGMAX_NOALLOC_MAX_ROWS rows; rows above it return
 *   DFLASH_ERR_TOO_LARGE before any CUDA call.  The library calls no
 *   allocator on this path.
 *   Set-up: the first call in each CUDA context (per device, with that device
 *   current) resolves the array's address (cudaGetSymbolAddress, return code
 *   checked; a failure returns DFLASH_ERR_CUDA and the next call retries).
 *   The library remembers the context's unique id and resolves again when it
 *   changes, e.g. after cudaDeviceReset.  Make the first call in a context
 *   before any stream capture begins.  Devices with an ordinal of 64 or more
 *   return DFLASH_ERR_INVALID_ARG.
 *   Each call clears the rows' tickets (an asynchronous memset on `stream`)
 *   and launches one kernel.  All calls on a device share the one array:
 *   calls that overlap in time (other streams, other host threads) race on
 *   it and must be serialised by the caller.
 *   argmax [rows] int32 and gap [rows] float32 (may be NULL) are device
 *   pointers; status (device int32, may be NULL) has DFLASH_STATUS_NONFINITE
 *   OR-ed in when a row holds NaN/Inf. */
#define DFLASH_ARGMAX_NOALLOC_MAX_ROWS 128
int dflash_argmax_noalloc(const float *logits, int32_t rows, int32_t V, int32_t *argmax,
                          float *gap, int32_t *status, dflash_stream_t stream);
/* Attention of q [batch][n][nq][hd] (dtype, RoPE applied) against layer
 * `layer` of `cache` (positions 0 .. len[b] + n - 1, the block's own keys
 * already written at len[b] ..), causal (row j sees 0..len+j) or not (every
 * row sees 0..len+n-1).  window > 0 drops the keys below len - window (the
 * drafter's cross-context window, see dflash_draft.cross_ctx); 0 keeps all.
 * out [batch][n][nq * hd] dtype.  q, out: device
 * pointers owned by the caller; q must be 16-byte aligned (the bf16 path
 * loads it by TMA), else DFLASH_ERR_INVALID_ARG before any CUDA call.  With
 * a DFLASH_KV_Q8 cache q is IEEE half precision (out stays bf16) and the
 * keys/values are the cache's codes times their row scales.
 * The scaled dot-product attention of "DFlash 深度解析" §2.2
 * draft_inference, evaluated per key group: the bf16 path splits the keys
 * into groups of a fixed number of 128-key tiles (a property of the cache),
 * keeps one running (max, sum, output) per row and group, and merges the
 * groups in order; the fp32 path does the same with 256-position chunks.
 * A row's result depends only on its own query and keys. */
int dflash_attention(const dflash_model_desc *d, const void *q, int32_t batch, int32_t n,
                     int32_t causal, int32_t window, dflash_cache *cache, int32_t layer, void *out,
                     dflash_workspace *ws, dflash_stream_t stream);

/* Kernel timing for measurement passes (not for graph capture): between
 * begin and end, the library brackets each weight-GEMM launch with a CUDA
 * event pair on the launching stream, up to max_records launches.  end
 * synchronises on the last event and returns per launch the elapsed
 * milliseconds and the tags (M, K, rows); *n_out = records returned. */
int dflash_profile_begin(int32_t max_records);
int dflash_profile_end(float *ms_out, int32_t *tags_out, int32_t max, int32_t *n_out);
/* Number of kernel launches this library has enqueued (or recorded into a
 * graph under capture) since it was loaded, counted on the host. */
long long dflash_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H_ */
