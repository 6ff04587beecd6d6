// C ABI of the DFlash step library: caches, workspace, and the five stages
// (fuse, inject, draft, verify, accept/rollback) composed from the kernels.
// Host code validates arguments and enqueues kernels; it never synchronises
// except in dflash_status.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <vector>

#include "common.cuh"
#include "internal.h"

using namespace dfl;

struct dflash_cache {
  int32_t n_layers, batch, capacity, n_kv, head_dim, dtype;
  size_t elem;
  uint8_t* k;
  uint8_t* v;
  int32_t* len;
  float2* rope;
  size_t layer_stride, seq_stride, head_stride;  // elements
  bool owns;
  bool has_maps;          // bf16, head_dim 128: TMA maps over the whole allocation
  CUtensorMap tk, tv;
  int32_t total_batch;    // sequences of the allocation (views share it)
  int32_t seq_base;       // first sequence of this view
  int32_t attn_gtiles;    // 128-key tiles per attention partial (fixed for the cache's life)
  int32_t kv_format;      // DFLASH_KV_MODEL or DFLASH_KV_Q8
  float* ks;              // q8: row scales [layer][seq][kv_head][capacity] (null otherwise)
  float* vs;
};

static KvMaps kv_maps(const dflash_cache* c, int layer) {
  KvMaps m;
  m.k = c->tk;
  m.v = c->tv;
  m.row0 = ((long long)layer * c->total_batch + c->seq_base) * c->n_kv * c->capacity;
  m.q8 = c->kv_format == DFLASH_KV_Q8;
  // the scales of the whole allocation (row0 indexes them like the maps' rows)
  const size_t back = (size_t)c->seq_base * c->n_kv * c->capacity;
  m.ks = c->ks ? c->ks - back : nullptr;
  m.vs = c->vs ? c->vs - back : nullptr;
  return m;
}

struct dflash_workspace {
  int32_t max_rows, max_ctx;
  size_t x_elems, xn_elems, f32_elems, q_elems, act_elems, logit_elems;
  float* x;
  void* xn;
  float* ssq;  // [rows][H / 32] sums of squares of the residual's 32-column slices (fused RMSNorm)
  float* f32buf;
  void* q;
  void* attn;
  void* act;
  float* logits;   // the target's logits [rows][V] (target_verify)
  float* dlogits;  // the drafter's logits [rows][V] (dflash_draft_block)
  float2* tstats;  // sampling: per-row (max, sum) of the target's logits
  float2* dstats;  // sampling: the same for the drafter's logits
  int32_t* cand_tok;   // tree: drafter top-K tokens [rows][8]
  float* cand_lp;      // tree: their log-probabilities [rows][8]
  int32_t* tree_path;  // tree: accepted path per sequence [rows][64]
  int32_t* tree_p0;    // tree: length before the rollback [rows]
  int32_t* tree_a;     // tree: accepted count [rows]
  int32_t vocab;
  AttnScratch as;
  ArgmaxScratch am;
  int* status;
  std::vector<void*> allocs;
};

static thread_local cudaError_t g_last_cuda = cudaSuccess;

namespace dfl {
int record_cuda_error(cudaError_t e) {
  g_last_cuda = e;
  return DFLASH_ERR_CUDA;
}
}  // namespace dfl

#define CK(expr)                    \
  do {                              \
    cudaError_t e_ = (expr);        \
    if (e_ != cudaSuccess) {        \
      g_last_cuda = e_;             \
      return DFLASH_ERR_CUDA;       \
    }                               \
  } while (0)

#define REQ(cond)                          \
  do {                                     \
    if (!(cond)) return DFLASH_ERR_INVALID_ARG; \
  } while (0)

static size_t dtype_size(int dt) { return dt == DFLASH_BF16 ? 2 : 4; }

static bool desc_ok(const dflash_model_desc* d) {
  return d && d->n_layers > 0 && d->hidden > 0 && d->n_q_heads > 0 && d->n_kv_heads > 0 &&
         d->n_q_heads % d->n_kv_heads == 0 && (d->head_dim == 64 || d->head_dim == 128) && d->ffn > 0 &&
         d->vocab > 1 && (d->dtype == DFLASH_F32 || d->dtype == DFLASH_BF16) && d->hidden % 4 == 0;
}

static bool desc_shapes_ok(const dflash_model_desc* d) {
  if (d->dtype != DFLASH_BF16) return true;
  const int H = d->hidden, hd = d->head_dim;
  const int G = d->n_q_heads / d->n_kv_heads;
  return hd == 128 && (G == 1 || G == 2 || G == 4 || G == 5 || G == 8) &&
         gemm_shape_ok(DFLASH_BF16, (d->n_q_heads + 2 * d->n_kv_heads) * hd, H) &&
         gemm_shape_ok(DFLASH_BF16, H, d->n_q_heads * hd) && gemm_shape_ok(DFLASH_BF16, 2 * d->ffn, H) &&
         gemm_shape_ok(DFLASH_BF16, H, d->ffn) && gemm_shape_ok(DFLASH_BF16, d->vocab, H);
}

extern "C" {

const char* dflash_strerror(int code) {
  switch (code) {
    case DFLASH_OK: return "ok";
    case DFLASH_ERR_INVALID_ARG: return "invalid argument";
    case DFLASH_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case DFLASH_ERR_CUDA: return cudaGetErrorString(g_last_cuda);
    case DFLASH_ERR_OOM: return "out of device memory";
    case DFLASH_ERR_TOO_LARGE: return "size above the entry point's fixed maximum";
    default: return "unknown error";
  }
}

int dflash_capture_layers(int32_t n_layers, int32_t out[5]) {
  REQ(out && n_layers >= 6);
  const int lo = 2, hi = n_layers - 3;
  // lo + (hi - lo) * i / 4 rounded half up, in exact integer arithmetic
  for (int i = 0; i < 5; ++i) out[i] = lo + ((hi - lo) * i * 2 + 4) / 8;
  return DFLASH_OK;
}

// ------------------------------------------------------------------ caches
int dflash_cache_alloc(const dflash_model_desc* d, int32_t n_layers, int32_t batch, int32_t capacity,
                       dflash_cache** out) {
  return dflash_cache_alloc_ex(d, n_layers, batch, capacity, DFLASH_KV_MODEL, out);
}

int32_t dflash_cache_kv_format(const dflash_cache* c) { return c ? c->kv_format : -1; }

int dflash_cache_alloc_ex(const dflash_model_desc* d, int32_t n_layers, int32_t batch, int32_t capacity,
                          int32_t kv_format, dflash_cache** out) {
  REQ(out && desc_ok(d) && n_layers > 0 && batch > 0 && capacity > 0);
  REQ(kv_format == DFLASH_KV_MODEL || kv_format == DFLASH_KV_Q8);
  *out = nullptr;
  const bool q8 = kv_format == DFLASH_KV_Q8;
  if (q8 && (d->dtype != DFLASH_BF16 || d->head_dim != 128)) return DFLASH_ERR_UNSUPPORTED_SHAPE;
  // q8: rows of scales are fetched in 128-row copies that start 16-byte aligned
  if (q8) capacity = (capacity + 7) & ~7;
  dflash_cache* c = new dflash_cache();
  c->n_layers = n_layers;
  c->batch = batch;
  c->capacity = capacity;
  c->n_kv = d->n_kv_heads;
  c->head_dim = d->head_dim;
  c->dtype = d->dtype;
  c->kv_format = kv_format;
  c->elem = q8 ? 1 : dtype_size(d->dtype);
  c->head_stride = (size_t)capacity * d->head_dim;
  c->seq_stride = c->head_stride * d->n_kv_heads;
  c->layer_stride = c->seq_stride * batch;
  c->owns = true;
  const size_t bytes = c->layer_stride * n_layers * c->elem;
  const size_t sbytes = q8 ? c->layer_stride / d->head_dim * n_layers * sizeof(float) : 0;
  const int half = d->head_dim / 2;
  if (cudaMalloc(&c->k, bytes) != cudaSuccess || cudaMalloc(&c->v, bytes) != cudaSuccess ||
      cudaMalloc(&c->len, sizeof(int32_t) * batch) != cudaSuccess ||
      cudaMalloc(&c->rope, sizeof(float2) * (size_t)capacity * half) != cudaSuccess ||
      (q8 && (cudaMalloc(&c->ks, sbytes) != cudaSuccess || cudaMalloc(&c->vs, sbytes) != cudaSuccess))) {
    cudaGetLastError();
    cudaFree(c->k);
    cudaFree(c->v);
    cudaFree(c->len);
    cudaFree(c->rope);
    cudaFree(c->ks);
    cudaFree(c->vs);
    delete c;
    return DFLASH_ERR_OOM;
  }
  cudaMemset(c->len, 0, sizeof(int32_t) * batch);
  // every position holds a finite value from the start (q8: codes 128 with scale 0, i.e. zeros)
  cudaMemset(c->k, q8 ? 128 : 0, bytes);
  cudaMemset(c->v, q8 ? 128 : 0, bytes);
  if (q8) {
    cudaMemset(c->ks, 0, sbytes);
    cudaMemset(c->vs, 0, sbytes);
  }
  c->total_batch = batch;
  c->seq_base = 0;
  c->has_maps = false;
  c->attn_gtiles = attn_group_tiles(capacity, d->n_kv_heads);
  if (d->dtype == DFLASH_BF16 && d->head_dim == 128) {
    const long long rows = (long long)n_layers * batch * d->n_kv_heads * capacity;
    if (!(q8 ? make_kv_maps_q8(c->k, c->v, rows, &c->tk, &c->tv) : make_kv_maps(c->k, c->v, rows, &c->tk, &c->tv))) {
      dflash_cache_free(c);
      return DFLASH_ERR_CUDA;
    }
    c->has_maps = true;
  }
  // RoPE table in double precision: angle = pos * theta^(-2i/d)
  std::vector<float2> tab((size_t)capacity * half);
  for (int i = 0; i < half; ++i) {
    const double inv = pow((double)d->rope_theta, -2.0 * i / (double)d->head_dim);
    for (int p = 0; p < capacity; ++p) {
      const double a = (double)p * inv;
      tab[(size_t)p * half + i] = make_float2((float)cos(a), (float)sin(a));
    }
  }
  if (cudaMemcpy(c->rope, tab.data(), sizeof(float2) * tab.size(), cudaMemcpyHostToDevice) != cudaSuccess) {
    dflash_cache_free(c);
    return DFLASH_ERR_CUDA;
  }
  *out = c;
  return DFLASH_OK;
}

int dflash_cache_view(dflash_cache* c, int32_t seq_begin, int32_t seq_count, dflash_cache** out) {
  REQ(c && out && seq_begin >= 0 && seq_count > 0 && seq_begin + seq_count <= c->batch);
  dflash_cache* v = new dflash_cache(*c);
  v->k = c->k + (size_t)seq_begin * c->seq_stride * c->elem;
  v->v = c->v + (size_t)seq_begin * c->seq_stride * c->elem;
  v->len = c->len + seq_begin;
  if (c->ks) {
    v->ks = c->ks + (size_t)seq_begin * c->seq_stride / c->head_dim;
    v->vs = c->vs + (size_t)seq_begin * c->seq_stride / c->head_dim;
  }
  v->batch = seq_count;
  v->seq_base = c->seq_base + seq_begin;
  v->owns = false;
  *out = v;
  return DFLASH_OK;
}

int dflash_cache_free(dflash_cache* c) {
  if (!c) return DFLASH_OK;
  if (c->owns) {
    cudaFree(c->k);
    cudaFree(c->v);
    cudaFree(c->len);
    cudaFree(c->rope);
    cudaFree(c->ks);
    cudaFree(c->vs);
  }
  delete c;
  return DFLASH_OK;
}

int32_t* dflash_cache_lengths(dflash_cache* c) { return c ? c->len : nullptr; }

int dflash_cache_get_lengths(dflash_cache* c, int32_t* host_out, int32_t n, dflash_stream_t stream) {
  REQ(c && host_out && n > 0);
  CK(cudaStreamSynchronize((cudaStream_t)stream));
  CK(cudaMemcpy(host_out, c->len, sizeof(int32_t) * (n < c->batch ? n : c->batch), cudaMemcpyDeviceToHost));
  return DFLASH_OK;
}

static int cache_copy(dflash_cache* c, int32_t layer, int32_t seq, int32_t pos0, int32_t n, void* k, void* v,
                      bool to_cache, cudaStream_t s) {
  REQ(c && k && v && layer >= 0 && layer < c->n_layers && seq >= 0 && seq < c->batch && pos0 >= 0 && n > 0 &&
      pos0 + n <= c->capacity);
  const size_t es = c->elem;
  const size_t off = ((size_t)layer * c->layer_stride + (size_t)seq * c->seq_stride + (size_t)pos0 * c->head_dim) * es;
  if (c->kv_format == DFLASH_KV_Q8) {
    REQ(to_cache);  // the codes are read with dflash_cache_read_q8
    const size_t soff = off / c->head_dim;
    CK(kv_quant_write(k, v, c->n_kv, n, c->k + off, c->v + off, c->ks + soff, c->vs + soff, c->head_stride, s));
    return DFLASH_OK;
  }
  const size_t pitch_cache = c->head_stride * es, width = (size_t)n * c->head_dim * es;
  for (int t = 0; t < 2; ++t) {
    uint8_t* cbase = (t == 0 ? c->k : c->v) + off;
    void* ubuf = t == 0 ? k : v;
    if (to_cache)
      CK(cudaMemcpy2DAsync(cbase, pitch_cache, ubuf, width, width, c->n_kv, cudaMemcpyDeviceToDevice, s));
    else
      CK(cudaMemcpy2DAsync(ubuf, width, cbase, pitch_cache, width, c->n_kv, cudaMemcpyDeviceToDevice, s));
  }
  return DFLASH_OK;
}

int dflash_cache_write(dflash_cache* c, int32_t layer, int32_t seq, int32_t pos0, int32_t n, const void* k,
                       const void* v, dflash_stream_t stream) {
  return cache_copy(c, layer, seq, pos0, n, const_cast<void*>(k), const_cast<void*>(v), true, (cudaStream_t)stream);
}

int dflash_cache_read(dflash_cache* c, int32_t layer, int32_t seq, int32_t pos0, int32_t n, void* k, void* v,
                      dflash_stream_t stream) {
  return cache_copy(c, layer, seq, pos0, n, k, v, false, (cudaStream_t)stream);
}

int dflash_cache_read_q8(dflash_cache* c, int32_t layer, int32_t seq, int32_t pos0, int32_t n, void* k_codes,
                         void* v_codes, float* k_scales, float* v_scales, dflash_stream_t stream) {
  REQ(c && c->kv_format == DFLASH_KV_Q8 && layer >= 0 && layer < c->n_layers && seq >= 0 && seq < c->batch &&
      pos0 >= 0 && n > 0 && pos0 + n <= c->capacity);
  REQ((k_codes != nullptr) == (v_codes != nullptr) && (k_scales != nullptr) == (v_scales != nullptr));
  cudaStream_t s = (cudaStream_t)stream;
  const size_t row = (size_t)layer * c->layer_stride / c->head_dim + (size_t)seq * c->seq_stride / c->head_dim + pos0;
  const size_t rows_per_head = c->head_stride / c->head_dim;  // = capacity
  if (k_codes) {
    const size_t w = (size_t)n * c->head_dim;
    CK(cudaMemcpy2DAsync(k_codes, w, c->k + row * c->head_dim, c->head_stride, w, c->n_kv, cudaMemcpyDeviceToDevice, s));
    CK(cudaMemcpy2DAsync(v_codes, w, c->v + row * c->head_dim, c->head_stride, w, c->n_kv, cudaMemcpyDeviceToDevice, s));
  }
  if (k_scales) {
    const size_t w = (size_t)n * sizeof(float);
    CK(cudaMemcpy2DAsync(k_scales, w, c->ks + row, rows_per_head * sizeof(float), w, c->n_kv, cudaMemcpyDeviceToDevice,
                         s));
    CK(cudaMemcpy2DAsync(v_scales, w, c->vs + row, rows_per_head * sizeof(float), w, c->n_kv, cudaMemcpyDeviceToDevice,
                         s));
  }
  return DFLASH_OK;
}

int dflash_cache_copy(dflash_cache* dst, const dflash_cache* src, dflash_stream_t stream) {
  REQ(dst && src && dst != src && dst->owns && src->owns && dst->n_layers == src->n_layers &&
      dst->batch == src->batch && dst->capacity == src->capacity && dst->n_kv == src->n_kv &&
      dst->head_dim == src->head_dim && dst->dtype == src->dtype && dst->kv_format == src->kv_format);
  cudaStream_t s = (cudaStream_t)stream;
  const size_t bytes = dst->layer_stride * dst->n_layers * dst->elem;
  CK(cudaMemcpyAsync(dst->k, src->k, bytes, cudaMemcpyDeviceToDevice, s));
  CK(cudaMemcpyAsync(dst->v, src->v, bytes, cudaMemcpyDeviceToDevice, s));
  if (dst->ks) {
    const size_t sb = dst->layer_stride / dst->head_dim * dst->n_layers * sizeof(float);
    CK(cudaMemcpyAsync(dst->ks, src->ks, sb, cudaMemcpyDeviceToDevice, s));
    CK(cudaMemcpyAsync(dst->vs, src->vs, sb, cudaMemcpyDeviceToDevice, s));
  }
  CK(cudaMemcpyAsync(dst->len, src->len, sizeof(int32_t) * dst->batch, cudaMemcpyDeviceToDevice, s));
  return DFLASH_OK;
}

int dflash_cache_set_lengths(dflash_cache* c, const int32_t* host_len, int32_t n, dflash_stream_t stream) {
  REQ(c && host_len && n > 0 && n <= c->batch);
  for (int i = 0; i < n; ++i) REQ(host_len[i] >= 0 && host_len[i] <= c->capacity);
  CK(cudaMemcpyAsync(c->len, host_len, sizeof(int32_t) * n, cudaMemcpyHostToDevice, (cudaStream_t)stream));
  CK(cudaStreamSynchronize((cudaStream_t)stream));
  return DFLASH_OK;
}

int dflash_cache_reset(dflash_cache* c, dflash_stream_t stream) {
  REQ(c);
  CK(cudaMemsetAsync(c->len, 0, sizeof(int32_t) * c->batch, (cudaStream_t)stream));
  return DFLASH_OK;
}

// ------------------------------------------------------------------ workspace
int dflash_workspace_alloc(const dflash_model_desc* t, const dflash_model_desc* d, int32_t max_rows, int32_t max_ctx,
                           dflash_workspace** out) {
  REQ(out && desc_ok(t) && (!d || desc_ok(d)) && max_rows > 0 && max_rows <= kMaxRows && max_ctx > 0);
  if (d) REQ(d->dtype == t->dtype);
  *out = nullptr;
  dflash_workspace* w = new dflash_workspace();
  w->max_rows = max_rows;
  w->max_ctx = max_ctx;
  const size_t es = dtype_size(t->dtype);
  const dflash_model_desc* ds[2] = {t, d ? d : t};
  size_t H = 0, f32w = 0, qw = 0, F = 0, V = 0, nq = 0;
  for (const dflash_model_desc* m : ds) {
    const size_t hd = m->head_dim;
    H = std::max(H, (size_t)m->hidden);
    f32w = std::max(f32w, (size_t)(m->n_q_heads + 2 * m->n_kv_heads) * hd);
    f32w = std::max(f32w, (size_t)m->hidden);
    qw = std::max(qw, (size_t)m->n_q_heads * hd);
    F = std::max(F, (size_t)m->ffn);
    V = std::max(V, (size_t)m->vocab);
    nq = std::max(nq, (size_t)m->n_q_heads);
  }
  if (d) f32w = std::max(f32w, (size_t)d->n_layers * 2 * d->n_kv_heads * d->head_dim);
  const size_t R = max_rows;
  const int nchunk = (max_ctx + kAttnChunk - 1) / kAttnChunk;
  struct Req {
    void** p;
    size_t bytes;
  } reqs[] = {
      {(void**)&w->x, R * H * 4},
      {(void**)&w->xn, R * H * es},
      {(void**)&w->ssq, R * (H / 32 + 1) * 4},
      {(void**)&w->f32buf, R * f32w * 4},
      {(void**)&w->q, R * qw * es},
      {(void**)&w->attn, R * qw * es},
      {(void**)&w->act, R * F * es},
      {(void**)&w->logits, R * V * 4},
      {(void**)&w->dlogits, R * V * 4},
      {(void**)&w->tstats, R * 8},
      {(void**)&w->dstats, R * 8},
      {(void**)&w->cand_tok, R * 8 * 4},
      {(void**)&w->cand_lp, R * 8 * 4},
      {(void**)&w->tree_path, R * 64 * 4},
      {(void**)&w->tree_p0, R * 4},
      {(void**)&w->tree_a, R * 4},

      {(void**)&w->as.o, R * nq * nchunk * 128 * 4},
      {(void**)&w->as.ml, R * nq * nchunk * 2 * 4},
      {(void**)&w->status, 4},
      {(void**)&w->am.part, R * kArgmaxSlices * 16},
      {(void**)&w->am.tickets, R * 4},
  };
  for (auto& r : reqs) {
    void* p = nullptr;
    if (cudaMalloc(&p, r.bytes) != cudaSuccess) {
      cudaGetLastError();
      dflash_workspace_free(w);
      return DFLASH_ERR_OOM;
    }
    *r.p = p;
    w->allocs.push_back(p);
  }
  w->as.nchunk = nchunk;
  w->vocab = (int32_t)V;
  w->am.max_rows = (int)R;
  cudaMemset(w->am.tickets, 0, R * 4);

  cudaMemset(w->status, 0, 4);
  cudaMemset(w->x, 0, R * H * 4);
  if (cudaDeviceSynchronize() != cudaSuccess) {
    dflash_workspace_free(w);
    return DFLASH_ERR_CUDA;
  }
  *out = w;
  return DFLASH_OK;
}

int dflash_workspace_free(dflash_workspace* w) {
  if (!w) return DFLASH_OK;
  for (void* p : w->allocs) cudaFree(p);
  delete w;
  return DFLASH_OK;
}

float* dflash_workspace_logits(dflash_workspace* w, int32_t which) {
  if (!w || which < 0 || which > 1) return nullptr;
  return which == 0 ? w->logits : w->dlogits;
}

int dflash_debug_set_wait_limit(int64_t ns) {
  set_gemm_wait_ns((long long)ns);
  return DFLASH_OK;
}

int dflash_status(dflash_workspace* w, dflash_stream_t stream, int32_t* status_out) {
  REQ(w && status_out);
  int32_t v = 0;
  CK(cudaStreamSynchronize((cudaStream_t)stream));
  CK(cudaMemcpy(&v, w->status, 4, cudaMemcpyDeviceToHost));
  CK(cudaMemset(w->status, 0, 4));
  *status_out = v;
  return DFLASH_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ kernel timing
// While enabled (measurement passes only), every weight product is bracketed
// by a pair of CUDA events on its stream; tags record the kind (1: bf16
// tensor-core kernel, 0: fp32), the rows and the weight kilobytes.
namespace {
struct Profile {
  bool on = false;
  int max = 0, n = 0;
  std::vector<cudaEvent_t> ev;
  std::vector<int32_t> tags;  // kind, rows, weight KB per record
} g_prof;
}  // namespace

static cudaError_t prof_begin(cudaStream_t s) {
  if (g_prof.on && g_prof.n < g_prof.max) return cudaEventRecord(g_prof.ev[2 * g_prof.n], s);
  return cudaSuccess;
}
static cudaError_t prof_end(cudaStream_t s, int kind, int rows, double weight_bytes) {
  if (!(g_prof.on && g_prof.n < g_prof.max)) return cudaSuccess;
  cudaError_t e = cudaEventRecord(g_prof.ev[2 * g_prof.n + 1], s);
  if (e != cudaSuccess) return e;
  g_prof.tags[3 * g_prof.n] = kind;
  g_prof.tags[3 * g_prof.n + 1] = rows;
  g_prof.tags[3 * g_prof.n + 2] = (int32_t)(weight_bytes / 1024.0);
  ++g_prof.n;
  return cudaSuccess;
}

extern "C" long long dflash_launch_count(void) { return launch_count(); }

extern "C" int dflash_profile_begin(int32_t max_records) {
  REQ(max_records > 0 && max_records <= (1 << 20) && !g_prof.on);
  if ((int)g_prof.ev.size() < 2 * max_records) {
    const size_t old = g_prof.ev.size();
    g_prof.ev.resize(2 * max_records);
    for (size_t i = old; i < g_prof.ev.size(); ++i) CK(cudaEventCreate(&g_prof.ev[i]));
  }
  g_prof.tags.assign(3 * (size_t)max_records, 0);
  g_prof.max = max_records;
  g_prof.n = 0;
  g_prof.on = true;
  return DFLASH_OK;
}

extern "C" int dflash_profile_end(float* ms_out, int32_t* tags_out, int32_t max, int32_t* n_out) {
  REQ(g_prof.on && n_out);
  g_prof.on = false;
  const int n = g_prof.n < max ? g_prof.n : max;
  if (n > 0) CK(cudaEventSynchronize(g_prof.ev[2 * (n - 1) + 1]));
  for (int i = 0; i < n; ++i) {
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]));
    if (ms_out) ms_out[i] = ms;
    if (tags_out)
      for (int j = 0; j < 3; ++j) tags_out[3 * i + j] = g_prof.tags[3 * i + j];
  }
  *n_out = n;
  return DFLASH_OK;
}

// ------------------------------------------------------------------ weight products
static GemmEpi epi_of(int kind, void* out, int ldo) {
  GemmEpi e;
  memset(&e, 0, sizeof(e));
  e.kind = kind;
  e.out = out;
  e.ldo = ldo;
  return e;
}

static GemmEpi epi_cache(int kind, void* out, int ldo, dflash_cache* c, int layer, int nq, int rows_per_seq,
                         const int32_t* n_pend) {
  GemmEpi e = epi_of(kind, out, ldo);
  e.nq = nq;
  e.nkv = c->n_kv;
  e.rows_per_seq = rows_per_seq;
  e.capacity = c->capacity;
  e.len = c->len;
  e.rope = c->rope;
  e.n_pend = n_pend;
  e.kc = c->k + (size_t)layer * c->layer_stride * c->elem;
  e.vc = c->v + (size_t)layer * c->layer_stride * c->elem;
  e.layer_stride = c->layer_stride;
  e.seq_stride = c->seq_stride;
  e.head_stride = c->head_stride;
  if (c->kv_format == DFLASH_KV_Q8) {
    e.kv_q8 = 1;
    e.ks = c->ks + (size_t)layer * c->layer_stride / c->head_dim;
    e.vs = c->vs + (size_t)layer * c->layer_stride / c->head_dim;
  }
  return e;
}

static cudaError_t gemm_b16(const void* X, int ldx, int rows, const void* W, int M, int K, const GemmEpi& epi,
                            dflash_workspace* ws, cudaStream_t s) {
  DFL_RET(prof_begin(s));
  DFL_RET(gemm_bf16(X, ldx, rows, W, M, K, epi, ws->status, s));
  return prof_end(s, 1, rows, 2.0 * M * K);
}

static cudaError_t gemm_f32(const void* X, int ldx, int rows, const void* W, int M, int K, const Epi& epi,
                            cudaStream_t s) {
  DFL_RET(prof_begin(s));
  DFL_RET(gemm_simt((const float*)X, ldx, rows, (const float*)W, M, K, epi, s));
  return prof_end(s, 0, rows, 4.0 * M * K);
}

// ------------------------------------------------------------------ composed forward
static bool cache_matches(const dflash_cache* c, const dflash_model_desc& d, int n_layers) {
  return c && c->n_kv == d.n_kv_heads && c->head_dim == d.head_dim && c->dtype == d.dtype &&
         c->n_layers >= n_layers;
}

static int layer_forward_f32(const dflash_model_desc& d, const dflash_layer_w& w, dflash_cache* c, int layer,
                             int batch, int n, int causal, int window, const int32_t* rope_off,
                             const uint64_t* tree_mask, dflash_workspace* ws, cudaStream_t s) {
  const int rows = batch * n, H = d.hidden, hd = d.head_dim, nq = d.n_q_heads, nkv = d.n_kv_heads;
  const int qkvw = (nq + 2 * nkv) * hd, dt = d.dtype;
  uint8_t* kc = c->k + (size_t)layer * c->layer_stride * c->elem;
  uint8_t* vc = c->v + (size_t)layer * c->layer_stride * c->elem;
  CK(rmsnorm(dt, ws->x, w.attn_norm, ws->xn, rows, H, d.rms_eps, s));
  CK(gemm_f32(ws->xn, H, rows, w.wqkv, qkvw, H, Epi{EPI_F32, ws->f32buf, qkvw}, s));
  CK(rope_qkv(dt, ws->f32buf, batch, n, nq, nkv, hd, ws->q, kc, vc, c->seq_stride, c->head_stride, c->capacity,
              c->len, c->rope, rope_off, ws->status, s));
  CK(attention(dt, ws->q, batch, n, nq, nkv, hd, causal, window, kc, vc, c->seq_stride, c->head_stride, c->capacity,
               c->attn_gtiles, c->len, tree_mask, nullptr, ws->as, ws->attn, ws->status, s));
  CK(gemm_f32(ws->attn, nq * hd, rows, w.wo, H, nq * hd, Epi{EPI_RESID, ws->x, H}, s));
  CK(rmsnorm(dt, ws->x, w.ffn_norm, ws->xn, rows, H, d.rms_eps, s));
  CK(gemm_f32(ws->xn, H, rows, w.w_gate_up, 2 * d.ffn, H, Epi{EPI_SWIGLU, ws->act, d.ffn}, s));
  CK(gemm_f32(ws->act, d.ffn, rows, w.w_down, H, d.ffn, Epi{EPI_RESID, ws->x, H}, s));
  return DFLASH_OK;
}

// The decoder stack and LM head on x (already embedded).  Per layer: RMSNorm,
// QKV product (bf16: RoPE and the KV-cache write fused in its epilogue),
// attention, O product + residual, RMSNorm, gate/up product + SwiGLU, down
// product + residual.  Captured states (hcap != null) after the layers in
// capture[].  window > 0 limits attention to the last `window` cached
// positions (the drafter's cross-context window).  rope_off/tree_mask
// (nullable, tree verification): row n's RoPE position is len + rope_off[n]
// and it attends to the context and the block keys its mask selects.
// The gain of a stack's first RMSNorm: its first layer's attention norm (the final norm of an empty stack).
static const void* first_norm(const dflash_model_desc& d, const dflash_layer_w* layers, const void* final_norm) {
  return d.n_layers > 0 ? layers[0].attn_norm : final_norm;
}

// bf16: expects x and the first norm's hand-over (xn, ssq) already written, by the embedding.
static int decoder_stack(const dflash_model_desc& d, const dflash_layer_w* layers, dflash_cache* c, int batch, int n,
                         int causal, int window, const int32_t* rope_off, const uint64_t* tree_mask,
                         const int32_t* capture, void* hcap, const void* final_norm, const void* lm_head,
                         float* logits, dflash_workspace* ws, cudaStream_t s) {
  const int rows = batch * n, H = d.hidden, hd = d.head_dim, nq = d.n_q_heads, nkv = d.n_kv_heads, L = d.n_layers;
  for (int l = 0; l < L; ++l) {
    const dflash_layer_w& w = layers[l];
    REQ(w.attn_norm && w.wqkv && w.wo && w.ffn_norm && w.w_gate_up && w.w_down);
  }
  if (d.dtype != DFLASH_BF16) {
    for (int l = 0; l < L; ++l) {
      int rc = layer_forward_f32(d, layers[l], c, l, batch, n, causal, window, rope_off, tree_mask, ws, s);
      if (rc != DFLASH_OK) return rc;
      if (hcap)
        for (int si = 0; si < 5; ++si)
          if (capture[si] == l) CK(dfl::capture(d.dtype, ws->x, hcap, rows, H, si, s));
    }
    CK(rmsnorm(d.dtype, ws->x, final_norm, ws->xn, rows, H, d.rms_eps, s));
    CK(gemm_f32(ws->xn, H, rows, lm_head, d.vocab, H, Epi{EPI_F32, logits, d.vocab}, s));
    return DFLASH_OK;
  }
  // Every RMSNorm sits between a residual-add product and the next product:
  // the residual-add epilogue hands over bf16(x * gain) (the next operand, in
  // xn) with the rows' 32-column sums of squares (ssq), and the next product
  // scales its rows by 1 / rms.  Only the first norm runs on its own.
  const int qkvw = (nq + 2 * nkv) * hd;
  auto normed = [&](GemmEpi e) {
    e.in_ssq = ws->ssq;
    e.in_cols = H;
    e.in_eps = d.rms_eps;
    return e;
  };
  auto handover = [&](GemmEpi e, const void* gain) {
    e.norm_gain = gain;
    e.norm_out = ws->xn;
    e.norm_ssq = ws->ssq;
    return e;
  };
  // (the first norm's hand-over comes with the embedding rows)
  for (int l = 0; l < L; ++l) {
    const dflash_layer_w& w = layers[l];
    uint8_t* kc = c->k + (size_t)l * c->layer_stride * c->elem;
    uint8_t* vc = c->v + (size_t)l * c->layer_stride * c->elem;
    GemmEpi qkv = epi_cache(GE_QKV, ws->q, nq * hd, c, l, nq, n, nullptr);
    qkv.rope_off = rope_off;
    CK(gemm_b16(ws->xn, H, rows, w.wqkv, qkvw, H, normed(qkv), ws, s));
    const KvMaps maps = kv_maps(c, l);
    CK(attention(d.dtype, ws->q, batch, n, nq, nkv, hd, causal, window, kc, vc, c->seq_stride, c->head_stride, c->capacity,
                 c->attn_gtiles, c->len, tree_mask, &maps, ws->as, ws->attn, ws->status, s));
    CK(gemm_b16(ws->attn, nq * hd, rows, w.wo, H, nq * hd, handover(epi_of(GE_RESID, ws->x, H), w.ffn_norm), ws, s));
    CK(gemm_b16(ws->xn, H, rows, w.w_gate_up, 2 * d.ffn, H, normed(epi_of(GE_SWIGLU, ws->act, d.ffn)), ws, s));
    GemmEpi down = handover(epi_of(GE_RESID, ws->x, H), l + 1 < L ? layers[l + 1].attn_norm : final_norm);
    if (hcap) {
      for (int si = 0; si < 5; ++si)
        if (capture[si] == l) down.cap_mask |= 1 << si;
      down.hcap = hcap;
      down.cap_H = H;
    }
    CK(gemm_b16(ws->act, d.ffn, rows, w.w_down, H, d.ffn, down, ws, s));
  }
  CK(gemm_b16(ws->xn, H, rows, lm_head, d.vocab, H, normed(epi_of(GE_F32, logits, d.vocab)), ws, s));
  return DFLASH_OK;
}

extern "C" {

int target_verify(const dflash_target* tg, const int32_t* tokens, int32_t batch, int32_t n, int32_t commit,
                  dflash_cache* tc, int32_t* argmax_out, float* top2_gap, void* hcap, int32_t* anchor,
                  int32_t* n_pend, int32_t* stream, int32_t* stream_len, int32_t stream_cap, dflash_workspace* ws,
                  dflash_stream_t cuda_stream) {
  REQ(tg && tokens && argmax_out && ws && desc_ok(&tg->d) && tg->layers && tg->embed && tg->lm_head &&
      tg->final_norm);
  const dflash_model_desc& d = tg->d;
  if (!desc_shapes_ok(&d)) return DFLASH_ERR_UNSUPPORTED_SHAPE;
  REQ(batch > 0 && n > 0 && n <= kMaxRows && batch * n <= ws->max_rows && commit >= 0 && commit <= 2);
  REQ(cache_matches(tc, d, d.n_layers) && batch <= tc->batch && tc->capacity <= ws->max_ctx);
  if (commit == 2) REQ(anchor);
  for (int i = 0; i < 5; ++i) REQ(tg->capture[i] >= 0 && tg->capture[i] < d.n_layers);
  cudaStream_t s = (cudaStream_t)cuda_stream;
  const int rows = batch * n, H = d.hidden;
  const bool b16 = d.dtype == DFLASH_BF16;
  CK(embed(d.dtype, tg->embed, d.vocab, H, tokens, nullptr, 0, batch, n, 0, nullptr, ws->x,
           b16 ? first_norm(d, tg->layers, tg->final_norm) : nullptr, b16 ? ws->xn : nullptr, b16 ? ws->ssq : nullptr,
           ws->status, s));
  int rc = decoder_stack(d, tg->layers, tc, batch, n, 1, 0, nullptr, nullptr, tg->capture, hcap, tg->final_norm,
                         tg->lm_head, ws->logits, ws, s);
  if (rc != DFLASH_OK) return rc;
  CK(argmax(ws->logits, rows, d.vocab, argmax_out, top2_gap, 0, ws->am, ws->status, s));
  if (commit)
    CK(commit_rows(tc->len, n_pend, anchor, argmax_out, batch, n, commit == 2, stream, stream_len, stream_cap,
                   ws->status, s));
  return DFLASH_OK;
}

int dflash_fuse_features(const dflash_draft* dr, const void* hcap, int32_t rows, void* fused, dflash_workspace* ws,
                         dflash_stream_t stream) {
  REQ(dr && hcap && fused && ws && desc_ok(&dr->d) && dr->w_fc && dr->fc_norm);
  REQ(rows > 0 && rows <= ws->max_rows);
  const dflash_model_desc& d = dr->d;
  const int H = d.hidden;
  if (!gemm_shape_ok(d.dtype, H, 5 * H)) return DFLASH_ERR_UNSUPPORTED_SHAPE;
  cudaStream_t s = (cudaStream_t)stream;
  if (d.dtype != DFLASH_BF16) {
    CK(gemm_f32(hcap, 5 * H, rows, dr->w_fc, H, 5 * H, Epi{EPI_F32, ws->f32buf, H}, s));
    CK(rmsnorm(d.dtype, ws->f32buf, dr->fc_norm, fused, rows, H, d.rms_eps, s));
    return DFLASH_OK;
  }
  CK(gemm_b16(hcap, 5 * H, rows, dr->w_fc, H, 5 * H, epi_of(GE_F32, ws->f32buf, H), ws, s));
  CK(rmsnorm(d.dtype, ws->f32buf, dr->fc_norm, fused, rows, H, d.rms_eps, s));
  return DFLASH_OK;
}

int dflash_inject_kv(const dflash_draft* dr, const void* fused, int32_t batch, int32_t rows_per_seq,
                     int32_t* n_pend, dflash_cache* dc, dflash_workspace* ws, dflash_stream_t stream) {
  REQ(dr && fused && n_pend && ws && desc_ok(&dr->d) && dr->w_kv_all);
  if (dc && dc->kv_format != DFLASH_KV_MODEL) return DFLASH_ERR_UNSUPPORTED_SHAPE;  // the drafter's cache
  const dflash_model_desc& d = dr->d;
  REQ(cache_matches(dc, d, d.n_layers) && batch > 0 && batch <= dc->batch && rows_per_seq > 0 &&
      batch * rows_per_seq <= ws->max_rows);
  const int H = d.hidden, W = d.n_layers * 2 * d.n_kv_heads * d.head_dim;
  if (!gemm_shape_ok(d.dtype, W, H)) return DFLASH_ERR_UNSUPPORTED_SHAPE;
  cudaStream_t s = (cudaStream_t)stream;
  const int rows = batch * rows_per_seq;
  if (d.dtype != DFLASH_BF16) {
    CK(gemm_f32(fused, H, rows, dr->w_kv_all, W, H, Epi{EPI_F32, ws->f32buf, W}, s));
    CK(inject_write(d.dtype, ws->f32buf, batch, rows_per_seq, d.n_layers, d.n_kv_heads, d.head_dim, dc->k, dc->v,
                    dc->layer_stride, dc->seq_stride, dc->head_stride, dc->capacity, dc->len, n_pend, dc->rope,
                    ws->status, s));
  } else {
    REQ(d.head_dim == 128);
    CK(gemm_b16(fused, H, rows, dr->w_kv_all, W, H, epi_cache(GE_INJECT, nullptr, 0, dc, 0, 0, rows_per_seq, n_pend), ws,
                s));
  }
  CK(advance_len(dc->len, n_pend, batch, s));
  return DFLASH_OK;
}

int dflash_draft_block(const dflash_draft* dr, const dflash_target* tg, const int32_t* anchor, int32_t batch,
                       int32_t block, dflash_cache* dc, int32_t* draft_tokens, dflash_workspace* ws,
                       dflash_stream_t stream) {
  REQ(dr && tg && anchor && draft_tokens && ws && desc_ok(&dr->d) && dr->layers && dr->final_norm && tg->embed &&
      tg->lm_head);
  const dflash_model_desc& d = dr->d;
  if (!desc_shapes_ok(&d)) return DFLASH_ERR_UNSUPPORTED_SHAPE;
  REQ(d.hidden == tg->d.hidden && d.vocab == tg->d.vocab && d.dtype == tg->d.dtype);
  REQ(block >= 2 && block <= 16 && batch > 0 && batch * block <= ws->max_rows);
  REQ(cache_matches(dc, d, d.n_layers) && batch <= dc->batch && dc->capacity <= ws->max_ctx);
  if (dc->kv_format != DFLASH_KV_MODEL) return DFLASH_ERR_UNSUPPORTED_SHAPE;  // the drafter's cache
  REQ(dr->mask_id >= 0 && dr->mask_id < d.vocab && dr->cross_ctx >= 0);
  cudaStream_t s = (cudaStream_t)stream;
  const int rows = batch * block, H = d.hidden;
  const bool b16 = d.dtype == DFLASH_BF16;
  CK(embed(d.dtype, tg->embed, d.vocab, H, nullptr, anchor, dr->mask_id, batch, block, 1, draft_tokens, ws->x,
           b16 ? first_norm(d, dr->layers, dr->final_norm) : nullptr, b16 ? ws->xn : nullptr, b16 ? ws->ssq : nullptr,
           ws->status, s));
  int rc = decoder_stack(d, dr->layers, dc, batch, block, 0, dr->cross_ctx, nullptr, nullptr, nullptr, nullptr,
                         dr->final_norm, tg->lm_head, ws->dlogits, ws, s);
  if (rc != DFLASH_OK) return rc;
  CK(argmax(ws->dlogits, rows, d.vocab, draft_tokens, nullptr, block, ws->am, ws->status, s));
  return DFLASH_OK;
}

int dflash_accept_rollback(const int32_t* draft_tokens, const int32_t* argmax_in, int32_t batch, int32_t block,
                           dflash_cache* tc, int32_t* anchor, int32_t* n_pend, int32_t* accept_len, int32_t* stream,
                           int32_t* stream_len, int32_t stream_cap, dflash_workspace* ws, dflash_stream_t cuda_stream) {
  REQ(draft_tokens && argmax_in && tc && anchor && n_pend && ws);
  REQ(batch > 0 && batch <= tc->batch && block >= 2 && block <= 32);
  REQ(!stream || (stream_len && stream_cap > 0));
  CK(accept_rollback(draft_tokens, argmax_in, batch, block, tc->len, anchor, n_pend, accept_len, stream, stream_len,
                     stream_cap, ws->status, (cudaStream_t)cuda_stream));
  return DFLASH_OK;
}

int dflash_teacher_force(int32_t* draft_tokens, int32_t batch, int32_t block, const int32_t* ref, int32_t ref_stride,
                         int32_t ref_len, const int32_t* stream_len, const int32_t* k_draw, const int32_t* r_draw,
                         int32_t max_steps, int32_t* step, int32_t vocab, dflash_workspace* ws,
                         dflash_stream_t stream) {
  REQ(draft_tokens && ref && stream_len && k_draw && r_draw && step && ws);
  REQ(batch > 0 && batch <= 1024 && block >= 2 && ref_stride >= ref_len && ref_len > 0 && max_steps > 0 &&
      vocab > 1);
  CK(teacher_force(draft_tokens, batch, block, ref, ref_stride, ref_len, stream_len, k_draw, r_draw, max_steps, step,
                   vocab, ws->status, (cudaStream_t)stream));
  return DFLASH_OK;
}

// ------------------------------------------------------------------ sampling mode
int dflash_draft_sample(int32_t batch, int32_t block, int32_t vocab, float temperature, const float* w,
                        int32_t* draft_tokens, dflash_workspace* ws, dflash_stream_t stream) {
  REQ(ws && w && draft_tokens && batch > 0 && block >= 2 && batch * block <= ws->max_rows);
  REQ(vocab > 1 && vocab <= ws->vocab && temperature > 0.f && isfinite(temperature));
  cudaStream_t s = (cudaStream_t)stream;
  const int rows = batch * block;
  CK(softmax_stats(ws->dlogits, rows, vocab, temperature, ws->dstats, s));
  CK(sample_rows(ws->dlogits, rows, vocab, temperature, ws->dstats, w, block, draft_tokens, s));
  return DFLASH_OK;
}

int dflash_accept_sample(const int32_t* draft_tokens, int32_t batch, int32_t block, int32_t vocab, float temperature,
                         const float* u, const float* v, dflash_cache* tc, int32_t* anchor, int32_t* n_pend,
                         int32_t* accept_len, int32_t* stream, int32_t* stream_len, int32_t stream_cap,
                         dflash_workspace* ws, dflash_stream_t cuda_stream) {
  REQ(draft_tokens && u && v && tc && anchor && n_pend && ws);
  REQ(batch > 0 && batch <= tc->batch && block >= 2 && block <= 32 && batch * block <= ws->max_rows);
  REQ(vocab > 1 && vocab <= ws->vocab && temperature > 0.f && isfinite(temperature));
  REQ(!stream || (stream_len && stream_cap > 0));
  cudaStream_t s = (cudaStream_t)cuda_stream;
  CK(softmax_stats(ws->logits, batch * block, vocab, temperature, ws->tstats, s));
  CK(accept_sample(draft_tokens, ws->logits, ws->dlogits, ws->tstats, ws->dstats, batch, block, vocab, temperature, u,
                   v, tc->len, anchor, n_pend, accept_len, stream, stream_len, stream_cap, ws->status, s));
  return DFLASH_OK;
}

int dflash_sample(const float* logits, int32_t rows, int32_t vocab, float temperature, const float* v, int32_t* out,
                  dflash_workspace* ws, dflash_stream_t stream) {
  REQ(logits && v && out && ws && rows > 0 && rows <= ws->max_rows && vocab > 1);
  REQ(temperature > 0.f && isfinite(temperature));
  cudaStream_t s = (cudaStream_t)stream;
  CK(softmax_stats(logits, rows, vocab, temperature, ws->tstats, s));
  CK(sample_rows(logits, rows, vocab, temperature, ws->tstats, v, 0, out, s));
  return DFLASH_OK;
}

// ------------------------------------------------------------------ tree verification
static long long tree_capacity(int depth, int k, int limit) {  // number of prefixes, capped
  long long tot = 0, layer = 1;
  for (int d = 0; d < depth && tot < limit; ++d) {
    layer *= k;
    tot += layer;
    if (layer > limit) layer = limit;
  }
  return tot;
}

int dflash_draft_tree(const int32_t* anchor, int32_t batch, int32_t block, int32_t vocab, int32_t topk, int32_t budget,
                      int32_t* tree_tokens, int32_t* tree_parent, int32_t* tree_depth, uint64_t* tree_mask,
                      dflash_workspace* ws, dflash_stream_t stream) {
  REQ(anchor && tree_tokens && tree_parent && tree_depth && tree_mask && ws);
  REQ(batch > 0 && block >= 2 && batch * block <= ws->max_rows && vocab > 1 && vocab <= ws->vocab);
  REQ(topk >= 1 && topk <= 8 && budget >= 1 && budget <= 63 && tree_capacity(block - 1, topk, 64) >= budget);
  cudaStream_t s = (cudaStream_t)stream;
  CK(softmax_stats(ws->dlogits, batch * block, vocab, 1.0f, ws->dstats, s));
  CK(draft_topk(ws->dlogits, batch, block, vocab, topk, ws->dstats, ws->cand_tok, ws->cand_lp, s));
  CK(tree_build(ws->cand_tok, ws->cand_lp, anchor, batch, block - 1, topk, budget, tree_tokens, tree_parent,
                tree_depth, tree_mask, s));
  return DFLASH_OK;
}

int target_verify_tree(const dflash_target* tg, const int32_t* tree_tokens, const int32_t* tree_depth,
                       const uint64_t* tree_mask, int32_t batch, int32_t n, dflash_cache* tc, int32_t* argmax_out,
                       float* top2_gap, void* hcap, dflash_workspace* ws, dflash_stream_t cuda_stream) {
  REQ(tg && tree_tokens && tree_depth && tree_mask && argmax_out && ws && desc_ok(&tg->d) && tg->layers &&
      tg->embed && tg->lm_head && tg->final_norm);
  const dflash_model_desc& d = tg->d;
  if (!desc_shapes_ok(&d)) return DFLASH_ERR_UNSUPPORTED_SHAPE;
  REQ(batch > 0 && n >= 1 && n <= 64 && batch * n <= ws->max_rows);
  REQ(cache_matches(tc, d, d.n_layers) && batch <= tc->batch && tc->capacity <= ws->max_ctx);
  if (tc->kv_format != DFLASH_KV_MODEL) return DFLASH_ERR_UNSUPPORTED_SHAPE;
  for (int i = 0; i < 5; ++i) REQ(tg->capture[i] >= 0 && tg->capture[i] < d.n_layers);
  cudaStream_t s = (cudaStream_t)cuda_stream;
  const bool b16 = d.dtype == DFLASH_BF16;
  CK(embed(d.dtype, tg->embed, d.vocab, d.hidden, tree_tokens, nullptr, 0, batch, n, 0, nullptr, ws->x,
           b16 ? first_norm(d, tg->layers, tg->final_norm) : nullptr, b16 ? ws->xn : nullptr, b16 ? ws->ssq : nullptr,
           ws->status, s));
  int rc = decoder_stack(d, tg->layers, tc, batch, n, 0, 0, tree_depth, tree_mask, tg->capture, hcap, tg->final_norm,
                         tg->lm_head, ws->logits, ws, s);
  if (rc != DFLASH_OK) return rc;
  CK(argmax(ws->logits, batch * n, d.vocab, argmax_out, top2_gap, 0, ws->am, ws->status, s));
  return DFLASH_OK;
}

int dflash_accept_tree(const dflash_target* tg, const int32_t* tree_tokens, const int32_t* tree_parent,
                       const int32_t* argmax_in, int32_t batch, int32_t n, dflash_cache* tc, void* hcap,
                       int32_t* anchor, int32_t* n_pend, int32_t* accept_len, int32_t* stream, int32_t* stream_len,
                       int32_t stream_cap, dflash_workspace* ws, dflash_stream_t cuda_stream) {
  REQ(tg && tree_tokens && tree_parent && argmax_in && tc && anchor && n_pend && ws && desc_ok(&tg->d));
  REQ(batch > 0 && batch <= tc->batch && n >= 1 && n <= 64 && batch * n <= ws->max_rows);
  REQ(cache_matches(tc, tg->d, tg->d.n_layers));
  if (tc->kv_format != DFLASH_KV_MODEL) return DFLASH_ERR_UNSUPPORTED_SHAPE;
  REQ(!stream || (stream_len && stream_cap > 0));
  cudaStream_t s = (cudaStream_t)cuda_stream;
  CK(accept_tree(tree_tokens, tree_parent, argmax_in, batch, n, tc->len, anchor, n_pend, accept_len, stream,
                 stream_len, stream_cap, ws->tree_path, ws->tree_p0, ws->tree_a, ws->status, s));
  CK(compact_kv(tc->dtype, tc->k, tc->v, tc->n_layers, batch, tc->n_kv, tc->layer_stride, tc->seq_stride,
                tc->head_stride, tc->head_dim, tc->capacity, ws->tree_path, ws->tree_p0, ws->tree_a, s));
  if (hcap)
    CK(compact_rows(tg->d.dtype, hcap, (size_t)5 * tg->d.hidden, batch, n, ws->tree_path, ws->tree_a, s));
  return DFLASH_OK;
}

// ------------------------------------------------------------------ building blocks
int dflash_linear(int32_t dtype, const void* x, const void* w, float* y, int32_t rows, int32_t M, int32_t K,
                  dflash_workspace* ws, dflash_stream_t stream) {
  REQ(x && w && y && ws && rows > 0 && rows <= kMaxRows && rows <= ws->max_rows && M > 0 && K > 0);
  REQ(dtype == DFLASH_F32 || dtype == DFLASH_BF16);
  if (!gemm_shape_ok(dtype, M, K)) return DFLASH_ERR_UNSUPPORTED_SHAPE;
  cudaStream_t s = (cudaStream_t)stream;
  if (dtype != DFLASH_BF16) {
    CK(gemm_f32(x, K, rows, w, M, K, Epi{EPI_F32, y, M}, s));
    return DFLASH_OK;
  }
  CK(gemm_b16(x, K, rows, w, M, K, epi_of(GE_F32, y, M), ws, s));
  return DFLASH_OK;
}

int dflash_rmsnorm(int32_t dtype, const float* x, const void* gain, void* y, int32_t rows, int32_t H, float eps,
                   dflash_stream_t stream) {
  REQ(x && gain && y && rows > 0 && H > 0 && H % 4 == 0);
  REQ(dtype == DFLASH_F32 || dtype == DFLASH_BF16);
  CK(rmsnorm(dtype, x, gain, y, rows, H, eps, (cudaStream_t)stream));
  return DFLASH_OK;
}

int dflash_argmax(const float* logits, int32_t rows, int32_t V, int32_t* argmax_out, float* gap, dflash_workspace* ws,
                  dflash_stream_t stream) {
  REQ(logits && argmax_out && ws && rows > 0 && V > 0);
  REQ(rows <= ws->max_rows);
  CK(argmax(logits, rows, V, argmax_out, gap, 0, ws->am, ws->status, (cudaStream_t)stream));
  return DFLASH_OK;
}

int dflash_attention(const dflash_model_desc* d, const void* q, int32_t batch, int32_t n, int32_t causal,
                     int32_t window, dflash_cache* c, int32_t layer, void* out, dflash_workspace* ws,
                     dflash_stream_t stream) {
  REQ(desc_ok(d) && q && out && ws && batch > 0 && n > 0 && batch * n <= ws->max_rows && window >= 0);
  REQ(cache_matches(c, *d, layer + 1) && layer >= 0 && batch <= c->batch && c->capacity <= ws->max_ctx);
  REQ((reinterpret_cast<uintptr_t>(q) & 15) == 0);  // the bf16 path reads q by TMA
  if (!desc_shapes_ok(d)) return DFLASH_ERR_UNSUPPORTED_SHAPE;
  const uint8_t* kc = c->k + (size_t)layer * c->layer_stride * c->elem;
  const uint8_t* vc = c->v + (size_t)layer * c->layer_stride * c->elem;
  const KvMaps maps = kv_maps(c, layer);
  CK(attention(d->dtype, q, batch, n, d->n_q_heads, d->n_kv_heads, d->head_dim, causal ? 1 : 0, window, kc, vc,
               c->seq_stride, c->head_stride, c->capacity, c->attn_gtiles, c->len, nullptr, c->has_maps ? &maps : nullptr, ws->as, out,
               ws->status, (cudaStream_t)stream));
  return DFLASH_OK;
}

}  // extern "C"
