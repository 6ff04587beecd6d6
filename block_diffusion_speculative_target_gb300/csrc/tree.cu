// Tree verification kernels (DDTree): the drafter's top-K candidates per
// slot, the best-first tree of the highest-scoring token prefixes within a
// node budget, the greedy walk over the verified tree, and the compaction of
// the accepted path's keys/values and captured rows into consecutive
// positions.  Tree construction follows "DFlash 深度解析" §8.2 (several
// branches of the drafter's guesses verified in one target forward within a
// budget) in the reading the library's header states: a prefix's score is the
// sum of its tokens' log-probabilities under the drafter's per-slot
// distributions; ties go to the smaller depth, then the smaller rank, then the
// earlier parent.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace dfl {

namespace {
constexpr int kTopThreads = 1024;
constexpr int kMaxK = 8;
constexpr int kMaxNodes = 64;

struct Cand {
  float v;
  int i;
};
// a before b: larger value, then lower index
__device__ __forceinline__ bool cand_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}
}  // namespace

// Top-K (K <= 8) of each drafter slot row j >= 1 (rows r % block == 0 are the
// anchors' and skipped) with log-probabilities lp = (z - max) - ln(sum e^(z -
// max)) from the row's statistics; ties to the lower token id.  Output index
// b * (block - 1) + j - 1, K entries each, by rank.
__global__ void __launch_bounds__(kTopThreads) topk_kernel(const float* __restrict__ logits, int V, int block, int K,
                                                           const float2* __restrict__ stats, int32_t* __restrict__ tok,
                                                           float* __restrict__ lp) {
  __shared__ float sv[kTopThreads / 32];
  __shared__ int si[kTopThreads / 32], sw[kTopThreads / 32];
  __shared__ int winner;
  const int r = blockIdx.x;
  pdl_launch();
  pdl_wait();
  if (r % block == 0) return;  // uniform over the CTA
  const int out = (r / block) * (block - 1) + (r % block) - 1;
  const float* z = logits + (size_t)r * V;
  // per-thread sorted top-K over its strided elements (visited in index order)
  float v[kMaxK];
  int id[kMaxK];
#pragma unroll
  for (int k = 0; k < kMaxK; ++k) {
    v[k] = -INFINITY;
    id[k] = 0x7fffffff;
  }
  for (int t = threadIdx.x; t < V; t += blockDim.x) {
    const float x = z[t];
    if (!cand_before(x, t, v[K - 1], id[K - 1])) continue;
    // insert, keeping order (an equal value with a lower index stays ahead)
    int k = K - 1;
    while (k > 0 && cand_before(x, t, v[k - 1], id[k - 1])) {
      v[k] = v[k - 1];
      id[k] = id[k - 1];
      --k;
    }
    v[k] = x;
    id[k] = t;
  }
  // K rounds: the block's best head wins and its thread advances
  const float2 st = stats[r];
  const float lse = logf(st.y);
  int head = 0;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int k = 0; k < K; ++k) {
    float bv = head < K ? v[head] : -INFINITY;
    int bi = head < K ? id[head] : 0x7fffffff;
    int bw = threadIdx.x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const int ow = __shfl_xor_sync(0xffffffffu, bw, o);
      if (cand_before(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
        bw = ow;
      }
    }
    if (lane == 0) {
      sv[w] = bv;
      si[w] = bi;
      sw[w] = bw;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float gv = sv[0];
      int gi = si[0], gw = sw[0];
      for (int i = 1; i < (int)(blockDim.x >> 5); ++i)
        if (cand_before(sv[i], si[i], gv, gi)) {
          gv = sv[i];
          gi = si[i];
          gw = sw[i];
        }
      tok[(size_t)out * K + k] = gi == 0x7fffffff ? 0 : gi;
      lp[(size_t)out * K + k] = (gv - st.x) - lse;
      winner = gw;
    }
    __syncthreads();
    if (threadIdx.x == winner) ++head;
    __syncthreads();
  }
}

// The best-first tree of one sequence (one thread): see the file comment.
// Node 0 is the anchor; mask[i] has bit j set for every ancestor j of node i
// and for i itself.
__global__ void tree_build_kernel(const int32_t* __restrict__ cand_tok, const float* __restrict__ cand_lp,
                                  const int32_t* __restrict__ anchor, int D, int K, int budget,
                                  int32_t* __restrict__ tokens, int32_t* __restrict__ parent,
                                  int32_t* __restrict__ depth, uint64_t* __restrict__ mask) {
  __shared__ float f_sc[2 * kMaxNodes + 2];
  __shared__ int f_d[2 * kMaxNodes + 2], f_r[2 * kMaxNodes + 2], f_p[2 * kMaxNodes + 2];
  __shared__ float n_sc[kMaxNodes];
  __shared__ uint64_t n_mask[kMaxNodes];
  const int b = blockIdx.x;
  pdl_launch();
  pdl_wait();
  if (threadIdx.x != 0) return;
  const int32_t* ct = cand_tok + (size_t)b * D * K;
  const float* cl = cand_lp + (size_t)b * D * K;
  const int n = budget + 1;
  int32_t* tk = tokens + (size_t)b * n;
  int32_t* pa = parent + (size_t)b * n;
  int32_t* de = depth + (size_t)b * n;
  uint64_t* mk = mask + (size_t)b * n;
  tk[0] = anchor[b];
  pa[0] = -1;
  de[0] = 0;
  n_sc[0] = 0.f;
  n_mask[0] = 1ull;
  mk[0] = 1ull;
  int nf = 0, nodes = 1;
  if (D >= 1) {
    f_sc[0] = cl[0];
    f_d[0] = 1;
    f_r[0] = 0;
    f_p[0] = 0;
    nf = 1;
  }
  while (nf > 0 && nodes < n) {
    int best = 0;
    for (int e = 1; e < nf; ++e) {
      const bool better = f_sc[e] > f_sc[best] ||
                          (f_sc[e] == f_sc[best] &&
                           (f_d[e] < f_d[best] || (f_d[e] == f_d[best] && (f_r[e] < f_r[best] ||
                                                                          (f_r[e] == f_r[best] && f_p[e] < f_p[best])))));
      if (better) best = e;
    }
    const float sc = f_sc[best];
    const int d = f_d[best], r = f_r[best], par = f_p[best];
    f_sc[best] = f_sc[nf - 1];
    f_d[best] = f_d[nf - 1];
    f_r[best] = f_r[nf - 1];
    f_p[best] = f_p[nf - 1];
    --nf;
    const int node = nodes++;
    tk[node] = ct[(size_t)(d - 1) * K + r];
    pa[node] = par;
    de[node] = d;
    n_sc[node] = sc;
    n_mask[node] = n_mask[par] | (1ull << node);
    mk[node] = n_mask[node];
    if (r + 1 < K) {
      f_sc[nf] = n_sc[par] + cl[(size_t)(d - 1) * K + r + 1];
      f_d[nf] = d;
      f_r[nf] = r + 1;
      f_p[nf] = par;
      ++nf;
    }
    if (d + 1 <= D) {
      f_sc[nf] = sc + cl[(size_t)d * K];
      f_d[nf] = d + 1;
      f_r[nf] = 0;
      f_p[nf] = node;
      ++nf;
    }
  }
  for (int i = nodes; i < n; ++i) {  // unreachable under the host's budget check; kept well-formed
    tk[i] = tk[0];
    pa[i] = 0;
    de[i] = 1;
    mk[i] = 1ull | (1ull << i);
  }
}

// The greedy walk over one sequence's verified tree (one warp), the emitted
// stream and the rollback lengths; records the path for the compaction.
__global__ void accept_tree_kernel(const int32_t* __restrict__ tokens, const int32_t* __restrict__ parent,
                                   const int32_t* __restrict__ argmax, int n, int32_t* len, int32_t* anchor,
                                   int32_t* n_pend, int32_t* accept_len, int32_t* stream, int32_t* stream_len,
                                   int stream_cap, int32_t* path_out, int32_t* p0_out, int32_t* a_out, int* status) {
  __shared__ int path[kMaxNodes];
  __shared__ int na;
  const int b = blockIdx.x, lane = threadIdx.x;
  pdl_launch();
  pdl_wait();
  const int32_t* tk = tokens + (size_t)b * n;
  const int32_t* pa = parent + (size_t)b * n;
  const int32_t* g = argmax + (size_t)b * n;
  if (lane == 0) {
    int x = 0, a = 0;
    path[0] = 0;
    while (a + 1 < n) {
      const int want = g[x];
      int c = -1;
      for (int i = x + 1; i < n; ++i)
        if (pa[i] == x && tk[i] == want) {
          c = i;
          break;
        }
      if (c < 0) break;
      path[++a] = c;
      x = c;
    }
    na = a;
  }
  __syncwarp();
  const int a = na;
  const int e = stream_len ? stream_len[b] : 0;
  if (lane <= a && stream) {
    const int32_t t = lane < a ? tk[path[lane + 1]] : g[path[a]];
    if (e + lane < stream_cap)
      stream[(size_t)b * stream_cap + e + lane] = t;
    else
      set_status(status, DFLASH_STATUS_BOUNDS);
  }
  for (int i = lane; i < n; i += 32) path_out[(size_t)b * kMaxNodes + i] = i <= a ? path[i] : -1;
  __syncwarp();
  if (lane == 0) {
    p0_out[b] = len[b];
    a_out[b] = a;
    len[b] += a + 1;
    anchor[b] = g[path[a]];
    n_pend[b] = a + 1;
    if (accept_len) accept_len[b] = a;
    if (stream_len) stream_len[b] = min(e + a + 1, stream_cap);
  }
}

// Accepted path node i (slot p0 + path[i]) -> slot p0 + i, for every layer and
// KV head of one sequence; i ascending (path[i] >= i, so no source is
// overwritten before it is read).  One CTA per (head, sequence, layer).
template <typename T>
__global__ void compact_kv_kernel(T* kc, T* vc, size_t layer_stride, size_t seq_stride, size_t head_stride, int hd,
                                  int capacity, const int32_t* __restrict__ path, const int32_t* __restrict__ p0,
                                  const int32_t* __restrict__ acc) {
  const int h = blockIdx.x, b = blockIdx.y, l = blockIdx.z;
  pdl_launch();
  pdl_wait();
  const int P = p0[b], a = acc[b];
  const size_t base = (size_t)l * layer_stride + (size_t)b * seq_stride + (size_t)h * head_stride;
  for (int i = 1; i <= a; ++i) {
    const int src = path[(size_t)b * kMaxNodes + i];
    if (src != i && P + src < capacity) {
      for (int d = threadIdx.x; d < hd; d += blockDim.x) {
        const T k = kc[base + (size_t)(P + src) * hd + d];
        const T v = vc[base + (size_t)(P + src) * hd + d];
        kc[base + (size_t)(P + i) * hd + d] = k;
        vc[base + (size_t)(P + i) * hd + d] = v;
      }
    }
    __syncthreads();
  }
}

// Captured rows of the accepted path -> rows 0..a of the sequence's block
// (rows of `n` per sequence), i ascending.
template <typename T>
__global__ void compact_rows_kernel(T* rows, size_t row_elems, int n, const int32_t* __restrict__ path,
                                    const int32_t* __restrict__ acc) {
  const int b = blockIdx.x;
  pdl_launch();
  pdl_wait();
  const int a = acc[b];
  T* base = rows + (size_t)b * n * row_elems;
  for (int i = 1; i <= a; ++i) {
    const int src = path[(size_t)b * kMaxNodes + i];
    if (src != i)
      for (size_t e = threadIdx.x; e < row_elems; e += blockDim.x) base[(size_t)i * row_elems + e] = base[(size_t)src * row_elems + e];
    __syncthreads();
  }
}

cudaError_t draft_topk(const float* logits, int batch, int block, int V, int K, const float2* stats, int32_t* tok,
                       float* lp, cudaStream_t s) {
  if (K < 1 || K > kMaxK) return cudaErrorInvalidValue;
  DFL_RET(launch_pdl(topk_kernel, dim3(batch * block), dim3(kTopThreads), 0, s, logits, V, block, K, stats, tok, lp));
  count_launch();
  return cudaSuccess;
}

cudaError_t tree_build(const int32_t* cand_tok, const float* cand_lp, const int32_t* anchor, int batch, int D, int K,
                       int budget, int32_t* tokens, int32_t* parent, int32_t* depth, uint64_t* mask, cudaStream_t s) {
  if (budget < 1 || budget + 1 > kMaxNodes) return cudaErrorInvalidValue;
  DFL_RET(launch_pdl(tree_build_kernel, dim3(batch), dim3(32), 0, s, cand_tok, cand_lp, anchor, D, K, budget, tokens,
                     parent, depth, mask));
  count_launch();
  return cudaSuccess;
}

cudaError_t accept_tree(const int32_t* tokens, const int32_t* parent, const int32_t* argmax, int batch, int n,
                        int32_t* len, int32_t* anchor, int32_t* n_pend, int32_t* accept_len, int32_t* stream,
                        int32_t* stream_len, int stream_cap, int32_t* path, int32_t* p0, int32_t* acc, int* status,
                        cudaStream_t s) {
  if (n < 1 || n > kMaxNodes) return cudaErrorInvalidValue;
  DFL_RET(launch_pdl(accept_tree_kernel, dim3(batch), dim3(32), 0, s, tokens, parent, argmax, n, len, anchor, n_pend,
                     accept_len, stream, stream_len, stream_cap, path, p0, acc, status));
  count_launch();
  return cudaSuccess;
}

cudaError_t compact_kv(int dtype, void* kc, void* vc, int layers, int batch, int nkv, size_t layer_stride,
                       size_t seq_stride, size_t head_stride, int hd, int capacity, const int32_t* path,
                       const int32_t* p0, const int32_t* acc, cudaStream_t s) {
  const dim3 grid(nkv, batch, layers);
  if (dtype == DFLASH_BF16)
    DFL_RET(launch_pdl(compact_kv_kernel<bf16>, grid, dim3(64), 0, s, (bf16*)kc, (bf16*)vc, layer_stride, seq_stride,
                       head_stride, hd, capacity, path, p0, acc));
  else
    DFL_RET(launch_pdl(compact_kv_kernel<float>, grid, dim3(64), 0, s, (float*)kc, (float*)vc, layer_stride,
                       seq_stride, head_stride, hd, capacity, path, p0, acc));
  count_launch();
  return cudaSuccess;
}

cudaError_t compact_rows(int dtype, void* rows, size_t row_elems, int batch, int n, const int32_t* path,
                         const int32_t* acc, cudaStream_t s) {
  if (dtype == DFLASH_BF16)
    DFL_RET(launch_pdl(compact_rows_kernel<bf16>, dim3(batch), dim3(256), 0, s, (bf16*)rows, row_elems, n, path, acc));
  else
    DFL_RET(launch_pdl(compact_rows_kernel<float>, dim3(batch), dim3(256), 0, s, (float*)rows, row_elems, n, path,
                       acc));
  count_launch();
  return cudaSuccess;
}

}  // namespace dfl
