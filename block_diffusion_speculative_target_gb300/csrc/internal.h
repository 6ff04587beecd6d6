// Internal launcher interface between the C-ABI layer (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/dflash.h"

namespace dfl {

// fp32 GEMM epilogues: y[n][m] = sum_k x[n][k] w[m][k], then
enum EpiKind {
  EPI_F32 = 0,     // out f32 [n][ldo]            = y
  EPI_STORE = 1,   // out T   [n][ldo]            = T(y)
  EPI_RESID = 2,   // out f32 [n][ldo]           += y   (residual stream)
  EPI_SWIGLU = 3,  // out T   [n][ldo], col m/2   = T(silu(y[m]) * y[m+1]) for even m (gate/up interleaved)
};

struct Epi {
  int kind;
  void* out;
  int ldo;
};

// Maximum rows (tokens) one GEMM call handles.
constexpr int kMaxRows = 128;

// ------------------------------------------------------------------ bf16 GEMM
// Epilogues of the tensor-core weight product y[n][m] = sum_k x[n][k] w[m][k]:
enum GemmEpiKind {
  GE_F32 = 0,     // out f32 [rows][ldo] = y
  GE_RESID = 1,   // out f32 [rows][ldo] += y  (residual stream)
  GE_STORE = 2,   // out bf16 [rows][ldo] = y
  GE_SWIGLU = 3,  // out bf16 [rows][ldo], column m/2 = silu(y[m]) * y[m+1] (gate/up rows interleaved)
  GE_QKV = 4,     // 128-row tile t = head t of q|k|v: RoPE on q/k; q -> out [rows][nq][128], k/v -> cache
  GE_INJECT = 5,  // tile t = drafter layer t/(2 nkv), k or v head: RoPE on k; rows j < n_pend[b] -> cache
};

struct GemmEpi {
  int kind;
  void* out;
  int ldo;
  // GE_RESID: bf16 copies of the new residual into hcap [rows][5 cap_H], slots in cap_mask
  void* hcap;
  int cap_mask, cap_H;
  // GE_QKV / GE_INJECT: row n = b * rows_per_seq + j sits at position len[b] + j
  int nq, nkv, rows_per_seq, capacity;
  const int32_t* len;
  const float2* rope;      // [capacity][64] cos, sin
  const int32_t* n_pend;   // GE_INJECT
  const int32_t* rope_off; // GE_QKV, nullable: row n's RoPE position is len[b] + rope_off[n] (tree nodes)
  void* kc;
  void* vc;
  size_t layer_stride, seq_stride, head_stride;
  // GE_RESID, nullable: the next product's RMSNorm handed over -- the new
  // residual x also leaves as bf16(x * norm_gain) in norm_out [rows][ldo] (that
  // product's operand) and as sums of x^2 over each 32 consecutive columns in
  // norm_ssq [rows][ldo / 32]
  const void* norm_gain;
  void* norm_out;
  float* norm_ssq;
  // Any kind, nullable: this product's operand is such a bf16(x * gain); each
  // row's result is scaled by 1 / sqrt(sum(x^2) / in_cols + in_eps), the sum
  // taken over in_ssq [rows][in_cols / 32] in column order, before the epilogue
  const float* in_ssq;
  int in_cols;
  float in_eps;
  // GE_QKV with an 8-bit cache: keys/values leave as codes (kc/vc uint8) with
  // one scale per row in ks/vs (indexed like kc / 128), the query as fp16
  int kv_q8;
  float* ks;
  float* vs;
};

// bf16 weight product on tcgen05 with cluster split-K (M % 128 == 0, K % 64 == 0, rows <= 128).
cudaError_t gemm_bf16(const void* X, int ldx, int rows, const void* W, int M, int K, const GemmEpi& epi, int* status,
                      cudaStream_t s);
// Limit of the weight product's main-loop waits in nanoseconds (< 0: the
// default 500 ms); see dflash_debug_set_wait_limit.
void set_gemm_wait_ns(long long ns);
// K splits (cluster size) for an [M x K] weight: depends on M, K and the SM count only.
int gemm_splits(int M, int K);

// Fixed attention chunk length (positions); chunk boundaries sit at multiples of it.
constexpr int kAttnChunk = 256;

int num_sms();

// Launch with programmatic dependent launch allowed: the kernel may start
// while its predecessor finishes; every kernel of this library calls
// griddepcontrol.wait before touching data another kernel produces or reads.
#define DFL_RET(expr)                 \
  do {                                \
    cudaError_t e_ = (expr);          \
    if (e_ != cudaSuccess) return e_; \
  } while (0)

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
// Host-side count of kernel launches enqueued by the library (for measurement).
void count_launch(int n = 1);
long long launch_count();

// float32 weight product on the CUDA cores (fp32 configuration).
cudaError_t gemm_simt(const float* X, int ldx, int rows, const float* W, int M, int K, const Epi& epi,
                      cudaStream_t s);
// Shapes the bf16 tensor-core path accepts: M % 128 == 0, K % 64 == 0.
bool gemm_shape_ok(int dtype, int M, int K);

// Row-wise RMSNorm: y = T(x * 1/sqrt(mean(x^2)+eps) * g).
cudaError_t rmsnorm(int dtype, const float* x, const void* g, void* y, int rows, int H, float eps,
                    cudaStream_t s);
// Copy T(x) into column block `slot` of hcap [rows][5H].
cudaError_t capture(int dtype, const float* x, void* hcap, int rows, int H, int slot, cudaStream_t s);
// x[r] = float(E[token(r)]).  mode 0: token = tokens[r]; mode 1 (draft block):
// token = anchor[b] for slot 0 else mask_id, and draft_out[b][0] = anchor[b].
// With xg (bf16), also the first norm's hand-over: xg = bf16(x * norm_gain)
// and ssq [rows][H/32] (the sums of x^2 over each 32 consecutive columns).
cudaError_t embed(int dtype, const void* E, int V, int H, const int32_t* tokens, const int32_t* anchor,
                  int mask_id, int batch, int n, int mode, int32_t* draft_out, float* x, const void* norm_gain,
                  void* xg, float* ssq, int* status, cudaStream_t s);
// RoPE on the q and k parts of qkv (f32 [rows][(nq+2nkv)hd]); q -> qout (T), k/v -> cache at len[b]+j.
// rope_off (nullable): row r's RoPE position is len[b] + rope_off[r] instead of len[b] + j (tree nodes).
cudaError_t rope_qkv(int dtype, const float* qkv, int batch, int n, int nq, int nkv, int hd, void* qout,
                     void* kc, void* vc, size_t seq_stride, size_t head_stride, int capacity,
                     const int32_t* len, const float2* rope_tab, const int32_t* rope_off, int* status, cudaStream_t s);
// Inject: kv f32 [batch*rps][Ld][2][nkv][hd] -> drafter caches (layer stride given) at len[b]+j, j < n_pend[b].
cudaError_t inject_write(int dtype, const float* kv, int batch, int rps, int Ld, int nkv, int hd, void* kc,
                         void* vc, size_t layer_stride, size_t seq_stride, size_t head_stride, int capacity,
                         const int32_t* len, const int32_t* n_pend, const float2* rope_tab, int* status,
                         cudaStream_t s);
cudaError_t advance_len(int32_t* len, int32_t* n_pend, int batch, cudaStream_t s);

// Attention partials over fixed chunks + combine.
struct AttnScratch {
  float* o;    // [rows][nq][nchunk][hd]
  float* ml;   // [rows][nq][nchunk][2]
  int nchunk;  // chunk capacity per row
};
// TMA maps over a bf16 cache's keys/values viewed as [rows][128]; row0 is the
// row of (layer, first sequence of the view, head 0, position 0).
struct KvMaps {
  CUtensorMap k, v;
  long long row0;
  // 8-bit caches: the maps cover uint8 codes, and ks/vs are the float32 row
  // scales of the whole allocation, indexed by the same flattened row
  bool q8;
  const float* ks;
  const float* vs;
};
bool make_kv_maps(const void* k, const void* v, long long rows_total, CUtensorMap* mk, CUtensorMap* mv);
bool make_kv_maps_q8(const void* k, const void* v, long long rows_total, CUtensorMap* mk, CUtensorMap* mv);
// Quantise rows of bf16 keys/values [n_kv][n][128] into an 8-bit cache's codes
// (u = q + 128) and scales: k_dst/v_dst point at position pos0 of head 0
// (head stride `head_stride` codes), ks/vs at the matching scale (stride
// head_stride / 128).
cudaError_t kv_quant_write(const void* k, const void* v, int n_kv, int n, uint8_t* k_dst, uint8_t* v_dst, float* ks,
                           float* vs, size_t head_stride, cudaStream_t s);
// window > 0: keys below len[b] - window (a cross-context window) are not attended.
// gtiles: 128-key tiles per partial of the bf16 path (a property of the cache).
// tree_mask (nullable, non-causal calls with n <= 64): row b*n+j sees the
// context and block key len[b] + i only when bit i of tree_mask[b*n+j] is set.
cudaError_t attention(int dtype, const void* q, int batch, int n, int nq, int nkv, int hd, int causal, int window,
                      const void* kc, const void* vc, size_t seq_stride, size_t head_stride, int capacity, int gtiles,
                      const int32_t* len, const uint64_t* tree_mask, const KvMaps* maps, const AttnScratch& sc,
                      void* out, int* status, cudaStream_t s);
// The tiles per partial for a cache of `capacity` positions and nkv heads:
// about one unit per SM for one sequence at full capacity (a power of two in
// [2, 64], raised until those units fit in one wave); depends on nothing
// else, so results do not depend on the batch.
int attn_group_tiles(int capacity, int nkv);

// 3-D map over a bf16 query buffer [rows][nq][128]: boxes of 64 head-dim
// elements (128 B, swizzled) x G heads x min(16, rows) rows.  Encoded maps are cached by
// (pointer, rows, nq, G).
bool make_q_map(const void* q, int rows, int nq, int G, CUtensorMap* out);
// The bf16 attention kernel on tcgen05 (head_dim 128, G in {1, 2, 4, 5, 8}):
// one partial (max, sum, unnormalised output) per (row, head, tile group).
cudaError_t attention_fa(int G, const KvMaps& maps, const CUtensorMap& qmap, int batch, int n, int nq, int nkv,
                         int causal, int window, int capacity, int gtiles, const int32_t* len,
                         const uint64_t* tree_mask, const AttnScratch& sc, float scale_log2, int* status,
                         cudaStream_t s);

// Greedy token and top-2 gap per row.  If skip_first_of (>0), rows with
// (r % skip_first_of) == 0 are not written to argmax_out.
constexpr int kArgmaxSlices = 16;
struct ArgmaxScratch {
  float4* part;  // [max_rows][kArgmaxSlices] slice results
  int* tickets;  // [max_rows], zero between launches
  int max_rows;
};
cudaError_t argmax(const float* logits, int rows, int V, int32_t* argmax_out, float* gap, int skip_first_of,
                   const ArgmaxScratch& sc, int* status, cudaStream_t s);
// Stores e as the thread's last CUDA error (reported by dflash_strerror) and
// returns DFLASH_ERR_CUDA.
int record_cuda_error(cudaError_t e);

// Sampling mode: per-row (max, sum of 2^((z - max) log2e / T)); one inverse-CDF
// draw per row (rows r % skip_first_of == 0 skipped when skip_first_of > 0);
// speculative-sampling verification + rollback of one block per sequence.
cudaError_t softmax_stats(const float* logits, int rows, int V, float temperature, float2* stats, cudaStream_t s);
cudaError_t sample_rows(const float* logits, int rows, int V, float temperature, const float2* stats, const float* v,
                        int skip_first_of, int32_t* out, cudaStream_t s);
cudaError_t accept_sample(const int32_t* draft, const float* zt, const float* zd, const float2* tst, const float2* dst,
                          int batch, int block, int V, float temperature, const float* u, const float* v, int32_t* len,
                          int32_t* anchor, int32_t* n_pend, int32_t* accept_len, int32_t* stream, int32_t* stream_len,
                          int stream_cap, int* status, cudaStream_t s);

// Tree verification: the drafter's top-K per slot (rows r % block == 0 skipped),
// the best-first tree per sequence, the greedy walk + rollback (records the
// path, the old length and the accepted count), and the compaction of the
// path's keys/values (all layers) and captured rows.  Trees hold <= 64 nodes.
cudaError_t draft_topk(const float* logits, int batch, int block, int V, int K, const float2* stats, int32_t* tok,
                       float* lp, cudaStream_t s);
cudaError_t tree_build(const int32_t* cand_tok, const float* cand_lp, const int32_t* anchor, int batch, int D, int K,
                       int budget, int32_t* tokens, int32_t* parent, int32_t* depth, uint64_t* mask, cudaStream_t s);
cudaError_t accept_tree(const int32_t* tokens, const int32_t* parent, const int32_t* argmax, int batch, int n,
                        int32_t* len, int32_t* anchor, int32_t* n_pend, int32_t* accept_len, int32_t* stream,
                        int32_t* stream_len, int stream_cap, int32_t* path, int32_t* p0, int32_t* acc, int* status,
                        cudaStream_t s);
cudaError_t compact_kv(int dtype, void* kc, void* vc, int layers, int batch, int nkv, size_t layer_stride,
                       size_t seq_stride, size_t head_stride, int hd, int capacity, const int32_t* path,
                       const int32_t* p0, const int32_t* acc, cudaStream_t s);
cudaError_t compact_rows(int dtype, void* rows, size_t row_elems, int batch, int n, const int32_t* path,
                         const int32_t* acc, cudaStream_t s);

cudaError_t commit_rows(int32_t* len, int32_t* n_pend, int32_t* anchor, const int32_t* argmax, int batch, int n,
                        int emit, int32_t* stream, int32_t* stream_len, int stream_cap, int* status,
                        cudaStream_t s);
cudaError_t accept_rollback(const int32_t* draft, const int32_t* argmax, int batch, int block, int32_t* len,
                            int32_t* anchor, int32_t* n_pend, int32_t* accept_len, int32_t* stream,
                            int32_t* stream_len, int stream_cap, int* status, cudaStream_t s);
cudaError_t teacher_force(int32_t* draft, int batch, int block, const int32_t* ref, int ref_stride, int ref_len,
                          const int32_t* stream_len, const int32_t* k_draw, const int32_t* r_draw, int max_steps,
                          int32_t* step, int vocab, int* status, cudaStream_t s);

}  // namespace dfl
