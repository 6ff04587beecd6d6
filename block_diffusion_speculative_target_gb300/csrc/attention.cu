// Block-vs-cache attention for the DFlash step.
//
// Keys are split into fixed 256-position chunks (boundaries at absolute
// multiples of 256); each CTA produces, per query row, the chunk's running
// max, softmax denominator and unnormalised output, and a combine kernel
// merges the chunks in chunk order.  A row's result therefore depends only on
// its own query and visible keys, not on how many rows share the launch.
//
// Visibility: causal (target verification and prefill) -- row j at position
// P+j sees keys 0..P+j; full (drafter block) -- every row sees 0..P+n-1 (the
// injected context plus the whole block).
//
// bf16 path (head_dim 128): the pipelined tcgen05 kernel (attention_fa.cu),
// one partial per group of `gtiles` 128-key tiles (a property of the cache).
// fp32 path: CUDA-core dot products, one CTA per (chunk, head, row).  This
// file also holds the chunk combine and the TMA maps over a cache.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dfl {

constexpr int kHD = 128;
// fp32: one CTA per (chunk, query head, row).
template <int NT>
__global__ void __launch_bounds__(NT)
    attn_f32_kernel(const float* __restrict__ q, int n, int nq, int nkv, int hd, int causal,
                    const float* __restrict__ kc, const float* __restrict__ vc, size_t seq_stride,
                    size_t head_stride, int capacity, int window, const int32_t* __restrict__ len,
                    const uint64_t* __restrict__ tree_mask, float* __restrict__ part_o, float* __restrict__ part_ml,
                    int nchunk, float scale_log2) {
  __shared__ float qs[kHD];
  __shared__ float sc[kAttnChunk];
  __shared__ float red[NT / 32];
  const int c = blockIdx.x, hq = blockIdx.y, r = blockIdx.z;
  const int b = r / n, j = r % n;
  const int hk = hq / (nq / nkv);
  pdl_launch();
  pdl_wait();
  const int P = len[b];
  const int lim = min(causal ? P + j + 1 : P + n, capacity);
  const int lo = window > 0 ? max(0, P - window) : 0;  // first key of a cross-context window
  const int kb = max(c * kAttnChunk, lo);
  if (kb >= lim || kb >= (c + 1) * kAttnChunk) return;
  const int ke = min((c + 1) * kAttnChunk, lim);
  const float* kbase = kc + (size_t)b * seq_stride + (size_t)hk * head_stride;
  const float* vbase = vc + (size_t)b * seq_stride + (size_t)hk * head_stride;
  for (int i = threadIdx.x; i < hd; i += NT) qs[i] = q[((size_t)r * nq + hq) * hd + i];
  __syncthreads();
  // tree verification: block key P + i is visible only when bit i is set (the node's ancestors)
  // (only then is n <= 64, so key - P < 64 keeps the shift defined)
  const uint64_t tm = tree_mask ? tree_mask[r] : 0ull;
  float mx = -INFINITY;
  for (int key = kb + threadIdx.x; key < ke; key += NT) {
    const float* kr = kbase + (size_t)key * hd;
    float acc = 0.f;
    for (int i = 0; i < hd; ++i) acc = fmaf(qs[i], kr[i], acc);
    acc *= scale_log2;
    if (tree_mask && key >= P && !((tm >> (key - P)) & 1ull)) acc = -INFINITY;
    sc[key - kb] = acc;
    mx = fmaxf(mx, acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  float m = red[0];
  for (int i = 1; i < NT / 32; ++i) m = fmaxf(m, red[i]);
  float ls = 0.f;
  for (int key = kb + threadIdx.x; key < ke; key += NT) {
    const float p = sc[key - kb] == -INFINITY ? 0.f : exp2f(sc[key - kb] - m);  // 0 for masked keys
    sc[key - kb] = p;
    ls += p;
  }
  const float l = block_sum<NT>(ls, red);  // contains __syncthreads: sc is complete afterwards
  const size_t row = ((size_t)r * nq + hq) * nchunk + c;
  for (int i = threadIdx.x; i < hd; i += NT) {
    float acc = 0.f;
    for (int key = kb; key < ke; ++key) acc = fmaf(sc[key - kb], vbase[(size_t)key * hd + i], acc);
    part_o[row * kHD + i] = acc;
  }
  if (threadIdx.x == 0) {
    part_ml[row * 2] = m;
    part_ml[row * 2 + 1] = l;
  }
}

// Merge of the key-group partials of one (row, head), two warps per pair
// (64 of the 128 columns each): with w_c = 2^(m_c - max m), out[d] =
// sum_c w_c o_c[d] / sum_c w_c l_c, the numerator summed over c in
// increasing order.  Lane l of half h owns columns 64 h + 2 l and + 1.  The
// row's length, the first 32 groups' maxima and sums and the
// first kCombineBatch groups' partial rows are all requested at once, before
// the row's group range is known (slots past it are read but never used), so
// a row with few groups needs one trip to memory.  The denominator's per-lane
// terms are added over a fixed butterfly.  The result depends only on the
// row's own groups.  The kernel holds no shared memory and at most 80
// registers a thread in 2-warp blocks (one (row, head) pair each), small
// enough to wait beside an attention CTA for it to finish.
constexpr int kCombineMaxChunks = 1024;
constexpr int kCombineWarps = 2;
constexpr int kCombineBatch = 16;  // partial rows in flight per lane

template <typename T>
__global__ void __launch_bounds__(kCombineWarps * 32, 12)
    attn_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml, int rows, int n, int nq,
                        int hd, int causal, int capacity, int window, int gk, const int32_t* __restrict__ len,
                        int nchunk, int swz_g, T* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int wi = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  const int item = wi >> 1, half = wi & 1;  // two warps per (row, head): 64 of the 128 dimensions each
  pdl_launch();
  pdl_wait();
  if (item >= rows * nq) return;  // warp-uniform
  const int r = item / nq, hq = item - r * nq;
  const int b = r / n, j = r - b * n;
  const size_t row0 = ((size_t)r * nq + hq) * nchunk;
  const float2* ml = reinterpret_cast<const float2*>(part_ml) + row0;
  // this lane's two columns 64 half + 2 lane: 16-byte chunk 16 half + lane / 2 of the row, which the
  // tcgen05 kernel leaves XOR-swizzled by (the row's index within its attention unit) & 7
  const int sw = swz_g > 0 ? (((j & 15) * swz_g + hq % swz_g) & 7) : 0;
  const float2* po = reinterpret_cast<const float2*>(part_o + row0 * kHD) +
                     ((((half * 16 + (lane >> 1)) ^ sw) << 1) | (lane & 1));  // group c: po[c * kHD / 2]
  const int P = len[b];
  const float2 ml0 = lane < nchunk ? ml[lane] : make_float2(-INFINITY, 0.f);  // group `lane`
  float2 v[kCombineBatch];
#pragma unroll
  for (int u = 0; u < kCombineBatch; ++u)
    if (u < nchunk) v[u] = po[(size_t)u * (kHD / 2)];
  const int lim = min(causal ? P + j + 1 : P + n, capacity);
  const int nch = min((lim + gk - 1) / gk, min(nchunk, kCombineMaxChunks));
  // groups below a cross-context window hold no partial
  const int clo = window > 0 ? min(max(0, P - window) / gk, nch) : 0;
  float m = (lane >= clo && lane < nch) ? ml0.x : -INFINITY;
  for (int c = 32 + lane; c < nch; c += 32)
    if (c >= clo) m = fmaxf(m, ml[c].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float M = m;
  float2 acc = make_float2(0.f, 0.f);
  float lsum = 0.f;
  for (int c0 = 0; c0 < nch; c0 += kCombineBatch) {
    if (c0 > 0) {
#pragma unroll
      for (int u = 0; u < kCombineBatch; ++u)
        if (c0 + u < nch) v[u] = po[(size_t)(c0 + u) * (kHD / 2)];
    }
    // lane u < kCombineBatch: group c0 + u's weight and its term of the denominator (groups below 32
    // come from the lane that loaded them)
    const int cu = c0 + lane;
    const float sx = __shfl_sync(0xffffffffu, ml0.x, cu & 31), sy = __shfl_sync(0xffffffffu, ml0.y, cu & 31);
    float2 mlu = make_float2(-INFINITY, 0.f);
    if (lane < kCombineBatch && cu >= clo && cu < nch) mlu = cu < 32 ? make_float2(sx, sy) : ml[cu];
    const float wu = mlu.x == -INFINITY ? 0.f : exp2f(mlu.x - M);
    lsum += wu * mlu.y;
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      const float w = __shfl_sync(0xffffffffu, wu, u);
      if (c0 + u >= clo && c0 + u < nch) {
        acc.x += w * v[u].x;
        acc.y += w * v[u].y;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
  const int d = half * 64 + 2 * lane;
  if (d < hd) {
    T* dst = out + ((size_t)r * nq + hq) * hd + d;
    dst[0] = from_f<T>(acc.x / lsum);
    dst[1] = from_f<T>(acc.y / lsum);
  }
}

typedef CUresult (*PFN_encodeTiled_t)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                      const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, fetched once (null if unavailable).
static PFN_encodeTiled_t encoder() {
  static const PFN_encodeTiled_t fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (PFN_encodeTiled_t) nullptr;
    return reinterpret_cast<PFN_encodeTiled_t>(p);
  }();
  return fn;
}

// 2-D maps over a whole bf16 cache viewed as [rows_total][128]: boxes of 64
// elements (128 B, swizzled) by 128 positions.
bool make_kv_maps(const void* k, const void* v, long long rows_total, CUtensorMap* mk, CUtensorMap* mv) {
  const PFN_encodeTiled_t fn = encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows_total};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t es[2] = {1, 1};
  for (int i = 0; i < 2; ++i)
    if (fn(i == 0 ? mk : mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(i == 0 ? k : v), dims, strides, box,
           es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  return true;
}

// 8-bit caches: codes [rows][128] uint8 in unswizzled 128-key boxes (the
// converter warps read them row by row).
bool make_kv_maps_q8(const void* k, const void* v, long long rows_total, CUtensorMap* mk, CUtensorMap* mv) {
  const PFN_encodeTiled_t fn = encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows_total};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t es[2] = {1, 1};
  for (int i = 0; i < 2; ++i)
    if (fn(i == 0 ? mk : mv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(i == 0 ? k : v), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  return true;
}

int attn_group_tiles(int capacity, int nkv) {
  // units of one sequence at full capacity ~ the SM count: tiles = cap/128 * nkv / SMs,
  // rounded to the nearest power of two, then raised until those units fit in one wave (one
  // CTA per SM): a second wave of a few units costs a whole unit's latency
  const int tiles = (capacity + 127) / 128, sms = num_sms();
  const double x = (double)tiles * nkv / (double)sms;
  int g = 2;
  while (g < 64 && (double)g * 1.41421356 < x) g *= 2;
  while (g < 64 && (long long)((tiles + g - 1) / g) * nkv > sms) ++g;
  return g;
}

bool make_q_map(const void* q, int rows, int nq, int G, CUtensorMap* out) {
  struct Entry {
    const void* q;
    int rows, nq, G;
    CUtensorMap map;
  };
  static Entry cache[16];
  static int used = 0, next = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].q == q && cache[i].rows == rows && cache[i].nq == nq && cache[i].G == G) {
      *out = cache[i].map;
      return true;
    }
  const PFN_encodeTiled_t fn = encoder();
  if (!fn || (reinterpret_cast<uintptr_t>(q) & 15) || rows <= 0) return false;
  CUtensorMap m;
  cuuint64_t dims[3] = {128, (cuuint64_t)nq, (cuuint64_t)rows};
  cuuint64_t strides[2] = {256, (cuuint64_t)nq * 256};
  cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)std::min(rows, 16)};
  cuuint32_t es[3] = {1, 1, 1};
  if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  Entry& e = cache[next];
  e = Entry{q, rows, nq, G, m};
  next = (next + 1) % 16;
  if (used < 16) ++used;
  *out = m;
  return true;
}

cudaError_t attention(int dtype, const void* q, int batch, int n, int nq, int nkv, int hd, int causal, int window,
                      const void* kc, const void* vc, size_t seq_stride, size_t head_stride, int capacity, int gtiles,
                      const int32_t* len, const uint64_t* tree_mask, const KvMaps* maps, const AttnScratch& sc,
                      void* out, int* status, cudaStream_t s) {
  if (batch * n <= 0) return cudaSuccess;
  if (tree_mask && (causal || n > 64)) return cudaErrorInvalidValue;  // tree rows: non-causal, at most 64 nodes
  const int nchunk_launch = (capacity + kAttnChunk - 1) / kAttnChunk;
  if (nchunk_launch > sc.nchunk || nchunk_launch > kCombineMaxChunks || hd > kHD) return cudaErrorInvalidValue;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)hd);
  const unsigned combine_blocks = (unsigned)((2 * batch * n * nq + kCombineWarps - 1) / kCombineWarps);
  if (dtype == DFLASH_BF16) {
    if (hd != kHD || !maps) return cudaErrorInvalidValue;
    const int G = nq / nkv;
    CUtensorMap qmap;
    if (!make_q_map(q, batch * n, nq, G, &qmap)) return cudaErrorInvalidValue;
    DFL_RET(attention_fa(G, *maps, qmap, batch, n, nq, nkv, causal, window, capacity, gtiles, len, tree_mask, sc,
                         scale_log2, status, s));
    DFL_RET(launch_pdl(attn_combine_kernel<bf16>, dim3(combine_blocks), dim3(kCombineWarps * 32), 0, s, sc.o, sc.ml,
                       batch * n, n, nq, hd, causal, capacity, window, gtiles * 128, len, sc.nchunk, G, (bf16*)out));
  } else {
    const dim3 grid(nchunk_launch, nq, batch * n);
    DFL_RET(launch_pdl(attn_f32_kernel<128>, grid, dim3(128), 0, s, (const float*)q, n, nq, nkv, hd, causal,
                       (const float*)kc, (const float*)vc, seq_stride, head_stride, capacity, window, len, tree_mask,
                       sc.o, sc.ml, sc.nchunk, scale_log2));
    DFL_RET(launch_pdl(attn_combine_kernel<float>, dim3(combine_blocks), dim3(kCombineWarps * 32), 0, s, sc.o, sc.ml,
                       batch * n, n, nq, hd, causal, capacity, window, kAttnChunk, len, sc.nchunk, 0, (float*)out));
  }
  count_launch(2);
  return cudaSuccess;
}

}  // namespace dfl
