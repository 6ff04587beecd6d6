// Bandwidth-bound and integer kernels of the DFlash step: embedding gather,
// RMSNorm, hidden-state capture, RoPE + KV-cache write, KV injection, greedy
// argmax with top-2 gap, acceptance/rollback and teacher forcing.
#include "common.cuh"
#include "internal.h"

#include <atomic>

namespace dfl {

static std::atomic<long long> g_launches{0};
void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
long long launch_count() { return g_launches.load(std::memory_order_relaxed); }

// ------------------------------------------------------------------ RMSNorm
// One CTA per row; fixed-order reduction, so a row's result does not depend
// on which other rows share the launch.
template <typename T, int NT>
__global__ void __launch_bounds__(NT) rmsnorm_kernel(const float* __restrict__ x, const T* __restrict__ g,
                                                     T* __restrict__ y, int H, float eps) {
  __shared__ float red[NT / 32];
  const float* xr = x + (size_t)blockIdx.x * H;
  T* yr = y + (size_t)blockIdx.x * H;
  pdl_launch();
  pdl_wait();
  float ss = 0.f;
  for (int i = threadIdx.x * 4; i < H; i += NT * 4) {
    float4 v = *reinterpret_cast<const float4*>(xr + i);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  const float tot = block_sum<NT>(ss, red);
  const float inv = 1.0f / sqrtf(tot / (float)H + eps);
  for (int i = threadIdx.x * 4; i < H; i += NT * 4) {
    float4 v = *reinterpret_cast<const float4*>(xr + i);
    yr[i + 0] = from_f<T>(v.x * inv * to_f<T>(g[i + 0]));
    yr[i + 1] = from_f<T>(v.y * inv * to_f<T>(g[i + 1]));
    yr[i + 2] = from_f<T>(v.z * inv * to_f<T>(g[i + 2]));
    yr[i + 3] = from_f<T>(v.w * inv * to_f<T>(g[i + 3]));
  }
}

cudaError_t rmsnorm(int dtype, const float* x, const void* g, void* y, int rows, int H, float eps,
                    cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (dtype == DFLASH_BF16)
    DFL_RET(launch_pdl(rmsnorm_kernel<bf16, 256>, dim3(rows), dim3(256), 0, s, x, (const bf16*)g, (bf16*)y, H, eps));
  else
    DFL_RET(launch_pdl(rmsnorm_kernel<float, 256>, dim3(rows), dim3(256), 0, s, x, (const float*)g, (float*)y, H, eps));
  count_launch();
  return cudaGetLastError();
}

// ------------------------------------------------------------------ 8-bit cache rows
// One warp per 128-entry row (lane l: entries 4 l .. 4 l + 3): s = max|x| /
// 127 and q = round-half-even(x / s) in float32 (IEEE division), stored as
// u = q + 128 with the scale.  Rows 0 .. n_kv * n - 1 are keys, the next as
// many values.
__global__ void __launch_bounds__(256) kv_quant_write_kernel(const bf16* __restrict__ k, const bf16* __restrict__ v,
                                                             int n_kv, int n, uint8_t* __restrict__ k_dst,
                                                             uint8_t* __restrict__ v_dst, float* __restrict__ ks,
                                                             float* __restrict__ vs, size_t head_stride) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  pdl_launch();
  pdl_wait();
  if (row >= 2 * n_kv * n) return;  // warp-uniform
  const int isv = row >= n_kv * n, r = isv ? row - n_kv * n : row;
  const int h = r / n, j = r - h * n;
  const bf16* src = (isv ? v : k) + (size_t)r * 128 + 4 * lane;
  float x[4], a = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[i] = __bfloat162float(src[i]);
    a = fmaxf(a, fabsf(x[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const float sc = __fdiv_rn(a, 127.0f);
  uchar4 u;
  uint8_t* ub = reinterpret_cast<uint8_t*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float q = sc > 0.f ? fminf(fmaxf(rintf(__fdiv_rn(x[i], sc)), -127.f), 127.f) : 0.f;
    ub[i] = (uint8_t)((int)q + 128);
  }
  const size_t crow = (size_t)h * head_stride + (size_t)j * 128;
  *reinterpret_cast<uchar4*>((isv ? v_dst : k_dst) + crow + 4 * lane) = u;
  if (lane == 0) (isv ? vs : ks)[crow / 128] = sc;
}

cudaError_t kv_quant_write(const void* k, const void* v, int n_kv, int n, uint8_t* k_dst, uint8_t* v_dst, float* ks,
                           float* vs, size_t head_stride, cudaStream_t s) {
  const int rows = 2 * n_kv * n;
  if (rows <= 0) return cudaSuccess;
  DFL_RET(launch_pdl(kv_quant_write_kernel, dim3((rows + 7) / 8), dim3(256), 0, s, (const bf16*)k, (const bf16*)v, n_kv,
                     n, k_dst, v_dst, ks, vs, head_stride));
  count_launch();
  return cudaGetLastError();
}

// ------------------------------------------------------------------ capture
template <typename T>
__global__ void capture_kernel(const float* __restrict__ x, T* __restrict__ hcap, int H, int slot) {
  const float* xr = x + (size_t)blockIdx.x * H;
  T* hr = hcap + (size_t)blockIdx.x * 5 * H + (size_t)slot * H;
  pdl_launch();
  pdl_wait();
  for (int i = threadIdx.x; i < H; i += blockDim.x) hr[i] = from_f<T>(xr[i]);
}

cudaError_t capture(int dtype, const float* x, void* hcap, int rows, int H, int slot, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (dtype == DFLASH_BF16)
    DFL_RET(launch_pdl(capture_kernel<bf16>, dim3(rows), dim3(256), 0, s, x, (bf16*)hcap, H, slot));
  else
    DFL_RET(launch_pdl(capture_kernel<float>, dim3(rows), dim3(256), 0, s, x, (float*)hcap, H, slot));
  count_launch();
  return cudaGetLastError();
}

// ------------------------------------------------------------------ embedding
// With `xg` given (bf16 only), the row also leaves as the first layer's
// norm operand, as a residual-add epilogue hands it over to the next
// product: bf16(x * g) and the sums of x^2 over each warp's 32-column slices
// (pass k, warp w: columns 256 k + 32 w .. + 31).
template <typename T>
__global__ void __launch_bounds__(256) embed_kernel(const T* __restrict__ E, int V, int H,
                                                    const int32_t* __restrict__ tokens,
                                                    const int32_t* __restrict__ anchor, int mask_id, int n, int mode,
                                                    int32_t* __restrict__ draft_out, float* __restrict__ x,
                                                    const bf16* __restrict__ g, bf16* __restrict__ xg,
                                                    float* __restrict__ ssq, int* status) {
  const int r = blockIdx.x, b = r / n, j = r % n;
  pdl_launch();
  pdl_wait();
  int tok;
  if (mode == 0) {
    tok = tokens[r];
  } else {
    tok = (j == 0) ? anchor[b] : mask_id;
    if (j == 0 && threadIdx.x == 0 && draft_out) draft_out[(size_t)b * n] = anchor[b];
  }
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) set_status(status, DFLASH_STATUS_BOUNDS);
    tok = 0;
  }
  const T* er = E + (size_t)tok * H;
  float* xr = x + (size_t)r * H;
  if constexpr (sizeof(T) == 2) {
    // eight entries per thread and pass: 16-byte loads of the row and the gains, 16-byte stores; the
    // sums of squares of each 32 columns over the four lanes that hold them
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    if (xg && (H & 255) == 0 && al16(er) && al16(xr) && al16(g) && al16(xg + (size_t)r * H)) {  // uniform
      for (int c = threadIdx.x; c < (H >> 3); c += blockDim.x) {
        const uint4 ew = reinterpret_cast<const uint4*>(er)[c];
        const uint4 gw = reinterpret_cast<const uint4*>(g)[c];
        const uint32_t e4[4] = {ew.x, ew.y, ew.z, ew.w}, g4[4] = {gw.x, gw.y, gw.z, gw.w};
        float v[8];
        uint32_t o4[4];
        float t = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 ev = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&e4[k]));
          const float2 gv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&g4[k]));
          v[2 * k] = ev.x;
          v[2 * k + 1] = ev.y;
          const __nv_bfloat162 pr = __floats2bfloat162_rn(ev.x * gv.x, ev.y * gv.y);
          o4[k] = *reinterpret_cast<const uint32_t*>(&pr);
          t += ev.x * ev.x;
          t += ev.y * ev.y;
        }
        reinterpret_cast<float4*>(xr)[2 * c] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4*>(xr)[2 * c + 1] = make_float4(v[4], v[5], v[6], v[7]);
        reinterpret_cast<uint4*>(xg + (size_t)r * H)[c] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
        t += __shfl_xor_sync(0xffffffffu, t, 1);
        t += __shfl_xor_sync(0xffffffffu, t, 2);
        if ((threadIdx.x & 3) == 0) ssq[(size_t)r * (H >> 5) + (c >> 2)] = t;
      }
      return;
    }
  }
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    const float v = to_f<T>(er[i]);
    xr[i] = v;
    if (xg) {  // uniform
      xg[(size_t)r * H + i] = __float2bfloat16_rn(v * __bfloat162float(g[i]));
      float t = v * v;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      if ((threadIdx.x & 31) == 0) ssq[(size_t)r * (H >> 5) + (i >> 5)] = t;
    }
  }
}

cudaError_t embed(int dtype, const void* E, int V, int H, const int32_t* tokens, const int32_t* anchor, int mask_id,
                  int batch, int n, int mode, int32_t* draft_out, float* x, const void* norm_gain, void* xg, float* ssq,
                  int* status, cudaStream_t s) {
  const int rows = batch * n;
  if (rows <= 0) return cudaSuccess;
  if (xg && (dtype != DFLASH_BF16 || H % 32 || !norm_gain || !ssq)) return cudaErrorInvalidValue;
  if (dtype == DFLASH_BF16)
    DFL_RET(launch_pdl(embed_kernel<bf16>, dim3(rows), dim3(256), 0, s, (const bf16*)E, V, H, tokens, anchor, mask_id,
                       n, mode, draft_out, x, (const bf16*)norm_gain, (bf16*)xg, ssq, status));
  else
    DFL_RET(launch_pdl(embed_kernel<float>, dim3(rows), dim3(256), 0, s, (const float*)E, V, H, tokens, anchor,
                       mask_id, n, mode, draft_out, x, (const bf16*)nullptr, (bf16*)nullptr, (float*)nullptr,
                       status));
  count_launch();
  return cudaGetLastError();
}

// ------------------------------------------------------------------ RoPE + KV write
// Rotate-half RoPE: pair (i, i + hd/2) rotated by pos * theta^(-2i/hd); the
// cos/sin table is per (position, i).
template <typename T>
__global__ void rope_qkv_kernel(const float* __restrict__ qkv, int n, int nq, int nkv, int hd, T* __restrict__ qout,
                                T* __restrict__ kc, T* __restrict__ vc, size_t seq_stride, size_t head_stride,
                                int capacity, const int32_t* __restrict__ len, const float2* __restrict__ tab,
                                const int32_t* __restrict__ rope_off, int* status) {
  const int r = blockIdx.x, b = r / n, j = r % n;
  const int half = hd / 2;
  const int width = (nq + 2 * nkv) * hd;
  pdl_launch();
  pdl_wait();
  const int pos = len[b] + j;
  const int rpos = rope_off ? len[b] + rope_off[r] : pos;  // RoPE position (a tree node's depth)
  const bool in_cap = pos < capacity && rpos >= 0 && rpos < capacity;
  if (!in_cap && threadIdx.x == 0) set_status(status, DFLASH_STATUS_CAPACITY);
  const float* src = qkv + (size_t)r * width;
  // q and k heads: nq + nkv heads x half pairs
  for (int t = threadIdx.x; t < (nq + nkv) * half; t += blockDim.x) {
    const int h = t / half, i = t % half;
    const float2 cs = in_cap ? tab[(size_t)rpos * half + i] : make_float2(1.f, 0.f);
    const float a = src[h * hd + i], c = src[h * hd + i + half];
    const float ra = a * cs.x - c * cs.y, rc = c * cs.x + a * cs.y;
    if (h < nq) {
      T* qo = qout + ((size_t)r * nq + h) * hd;
      qo[i] = from_f<T>(ra);
      qo[i + half] = from_f<T>(rc);
    } else if (in_cap) {
      T* ko = kc + (size_t)b * seq_stride + (size_t)(h - nq) * head_stride + (size_t)pos * hd;
      ko[i] = from_f<T>(ra);
      ko[i + half] = from_f<T>(rc);
    }
  }
  if (in_cap) {
    for (int t = threadIdx.x; t < nkv * hd; t += blockDim.x) {
      const int h = t / hd, i = t % hd;
      vc[(size_t)b * seq_stride + (size_t)h * head_stride + (size_t)pos * hd + i] =
          from_f<T>(src[(nq + nkv) * hd + t]);
    }
  }
}

cudaError_t rope_qkv(int dtype, const float* qkv, int batch, int n, int nq, int nkv, int hd, void* qout, void* kc,
                     void* vc, size_t seq_stride, size_t head_stride, int capacity, const int32_t* len,
                     const float2* tab, const int32_t* rope_off, int* status, cudaStream_t s) {
  const int rows = batch * n;
  if (rows <= 0) return cudaSuccess;
  if (dtype == DFLASH_BF16)
    DFL_RET(launch_pdl(rope_qkv_kernel<bf16>, dim3(rows), dim3(256), 0, s, qkv, n, nq, nkv, hd, (bf16*)qout, (bf16*)kc, (bf16*)vc, seq_stride,
                                               head_stride, capacity, len, tab, rope_off, status));
  else
    DFL_RET(launch_pdl(rope_qkv_kernel<float>, dim3(rows), dim3(256), 0, s, qkv, n, nq, nkv, hd, (float*)qout, (float*)kc, (float*)vc,
                                                seq_stride, head_stride, capacity, len, tab, rope_off, status));
  count_launch();
  return cudaGetLastError();
}

// ------------------------------------------------------------------ KV injection
template <typename T>
__global__ void inject_kernel(const float* __restrict__ kv, int rps, int Ld, int nkv, int hd, T* __restrict__ kc,
                              T* __restrict__ vc, size_t layer_stride, size_t seq_stride, size_t head_stride,
                              int capacity, const int32_t* __restrict__ len, const int32_t* __restrict__ n_pend,
                              const float2* __restrict__ tab, int* status) {
  const int r = blockIdx.x, b = r / rps, j = r % rps;
  pdl_launch();
  pdl_wait();
  if (j >= n_pend[b]) {
    return;
  }
  const int pos = len[b] + j;
  if (pos >= capacity) {
    if (threadIdx.x == 0) set_status(status, DFLASH_STATUS_CAPACITY);
    return;
  }
  const int half = hd / 2;
  const size_t width = (size_t)Ld * 2 * nkv * hd;
  const float* src = kv + (size_t)r * width;
  for (int t = threadIdx.x; t < Ld * nkv * half; t += blockDim.x) {
    const int l = t / (nkv * half), rem = t % (nkv * half), h = rem / half, i = rem % half;
    const float* ks = src + (size_t)l * 2 * nkv * hd + (size_t)h * hd;
    const float2 cs = tab[(size_t)pos * half + i];
    const float a = ks[i], c = ks[i + half];
    T* ko = kc + (size_t)l * layer_stride + (size_t)b * seq_stride + (size_t)h * head_stride + (size_t)pos * hd;
    ko[i] = from_f<T>(a * cs.x - c * cs.y);
    ko[i + half] = from_f<T>(c * cs.x + a * cs.y);
  }
  for (int t = threadIdx.x; t < Ld * nkv * hd; t += blockDim.x) {
    const int l = t / (nkv * hd), rem = t % (nkv * hd), h = rem / hd, i = rem % hd;
    const float* vs = src + (size_t)l * 2 * nkv * hd + (size_t)nkv * hd + (size_t)h * hd;
    vc[(size_t)l * layer_stride + (size_t)b * seq_stride + (size_t)h * head_stride + (size_t)pos * hd + i] =
        from_f<T>(vs[i]);
  }
}

cudaError_t inject_write(int dtype, const float* kv, int batch, int rps, int Ld, int nkv, int hd, void* kc, void* vc,
                         size_t layer_stride, size_t seq_stride, size_t head_stride, int capacity,
                         const int32_t* len, const int32_t* n_pend, const float2* tab, int* status,
                         cudaStream_t s) {
  const int rows = batch * rps;
  if (rows <= 0) return cudaSuccess;
  if (dtype == DFLASH_BF16)
    DFL_RET(launch_pdl(inject_kernel<bf16>, dim3(rows), dim3(256), 0, s, kv, rps, Ld, nkv, hd, (bf16*)kc, (bf16*)vc, layer_stride, seq_stride,
                                             head_stride, capacity, len, n_pend, tab, status));
  else
    DFL_RET(launch_pdl(inject_kernel<float>, dim3(rows), dim3(256), 0, s, kv, rps, Ld, nkv, hd, (float*)kc, (float*)vc, layer_stride,
                                              seq_stride, head_stride, capacity, len, n_pend, tab, status));
  count_launch();
  return cudaGetLastError();
}

// The injected rows are consumed: len += n_pend, n_pend = 0.
__global__ void advance_len_kernel(int32_t* len, int32_t* n_pend, int batch) {
  pdl_launch();
  pdl_wait();
  const int b = threadIdx.x;
  if (b < batch) {
    len[b] += n_pend[b];
    n_pend[b] = 0;
  }
}

cudaError_t advance_len(int32_t* len, int32_t* n_pend, int batch, cudaStream_t s) {
  DFL_RET(launch_pdl(advance_len_kernel, dim3(1), dim3(32 * ((batch + 31) / 32)), 0, s, len, n_pend, batch));
  count_launch();
  return cudaGetLastError();
}

// ------------------------------------------------------------------ argmax + top-2
struct Top2 {
  float v1, v2;
  int i1;
};

__device__ __forceinline__ Top2 top2_merge(Top2 a, Top2 b) {
  // winner: larger value, lower index on equal values
  const bool bw = (b.v1 > a.v1) || (b.v1 == a.v1 && b.i1 < a.i1);
  Top2 w = bw ? b : a, l = bw ? a : b;
  Top2 o;
  o.v1 = w.v1;
  o.i1 = w.i1;
  o.v2 = fmaxf(w.v2, l.v1);
  return o;
}

// Grid (rows, kArgmaxSlices): each CTA scans one contiguous slice of a row;
// the last CTA of the row (ticket) merges the slice results in slice order,
// so ties resolve to the lowest index and the result is deterministic.
template <int NT>
__global__ void __launch_bounds__(NT) argmax_kernel(const float* __restrict__ logits, int V, int32_t* __restrict__ out,
                                                    float* __restrict__ gap, int skip_first_of, float4* __restrict__ part,
                                                    int* __restrict__ tickets, int* status) {
  __shared__ Top2 sh[NT / 32];
  __shared__ int last;
  const int row_i = blockIdx.x, sl = blockIdx.y, ns = gridDim.y;
  const float* row = logits + (size_t)row_i * V;
  pdl_launch();
  pdl_wait();
  // 16-byte loads when the rows allow them (slices then start on multiples of 4 entries); each thread
  // takes its entries in increasing index order, so ties keep the lowest index
  const bool vec = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0;
  const int per = vec ? (((V + ns - 1) / ns + 3) & ~3) : (V + ns - 1) / ns;
  const int v0 = min(V, sl * per), v1 = min(V, v0 + per);
  Top2 t{-INFINITY, -INFINITY, 0x7fffffff};
  bool bad = false;
  auto take = [&](float v, int i) {
    bad |= !(fabsf(v) <= 3.0e38f);
    if (v > t.v1) {
      t.v2 = t.v1;
      t.v1 = v;
      t.i1 = i;
    } else if (v > t.v2) {
      t.v2 = v;
    }
  };
  if (vec) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const int q1 = v1 >> 2;
    int q = (v0 >> 2) + threadIdx.x;
    for (; q + 3 * NT < q1; q += 4 * NT) {  // four 16-byte loads in flight per thread
      float4 a[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) a[k] = r4[q + k * NT];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = 4 * (q + k * NT);
        take(a[k].x, i);
        take(a[k].y, i + 1);
        take(a[k].z, i + 2);
        take(a[k].w, i + 3);
      }
    }
    for (; q < q1; q += NT) {
      const float4 a = r4[q];
      take(a.x, 4 * q);
      take(a.y, 4 * q + 1);
      take(a.z, 4 * q + 2);
      take(a.w, 4 * q + 3);
    }
  } else {
    for (int i = v0 + threadIdx.x; i < v1; i += NT) take(row[i], i);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Top2 u;
    u.v1 = __shfl_xor_sync(0xffffffffu, t.v1, o);
    u.v2 = __shfl_xor_sync(0xffffffffu, t.v2, o);
    u.i1 = __shfl_xor_sync(0xffffffffu, t.i1, o);
    t = top2_merge(t, u);
  }
  bad = __any_sync(0xffffffffu, bad);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) sh[w] = t;
  if (bad && (threadIdx.x & 31) == 0) set_status(status, DFLASH_STATUS_NONFINITE);
  __syncthreads();
  if (threadIdx.x == 0) {
    Top2 r = sh[0];
    for (int i = 1; i < NT / 32; ++i) r = top2_merge(r, sh[i]);
    part[(size_t)row_i * ns + sl] = make_float4(r.v1, r.v2, __int_as_float(r.i1), 0.f);
    __threadfence();
    last = (atomicAdd(&tickets[row_i], 1) == ns - 1) ? 1 : 0;
  }
  __syncthreads();
  if (last && threadIdx.x == 0) {
    __threadfence();
    Top2 r{-INFINITY, -INFINITY, 0x7fffffff};
    for (int i = 0; i < ns; ++i) {
      const float4 p = __ldcg(&part[(size_t)row_i * ns + i]);
      r = top2_merge(r, Top2{p.x, p.y, __float_as_int(p.z)});
    }
    if (r.i1 == 0x7fffffff) r.i1 = 0;
    const bool skip = skip_first_of > 0 && (row_i % skip_first_of) == 0;
    if (!skip) out[row_i] = r.i1;
    if (gap) gap[row_i] = r.v1 - r.v2;
    tickets[row_i] = 0;
  }
}

cudaError_t argmax(const float* logits, int rows, int V, int32_t* out, float* gap, int skip_first_of,
                   const ArgmaxScratch& sc, int* status, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (rows > sc.max_rows) return cudaErrorInvalidValue;
  const int ns = V >= 16 * 1024 ? kArgmaxSlices : 1;
  DFL_RET(launch_pdl(argmax_kernel<256>, dim3(rows, ns), dim3(256), 0, s, logits, V, out, gap, skip_first_of, sc.part,
                     sc.tickets, status));
  count_launch();
  return cudaSuccess;
}

// ------------------------------------------------------------------ commit (prefill / AR)
__global__ void commit_kernel(int32_t* len, int32_t* n_pend, int32_t* anchor, const int32_t* argmax, int batch, int n,
                              int emit, int32_t* stream, int32_t* stream_len, int stream_cap, int* status) {
  pdl_launch();
  pdl_wait();
  const int b = threadIdx.x;
  if (b < batch) {
    len[b] += n;
    if (n_pend) n_pend[b] = n;
    if (emit) {
      const int32_t g = argmax[(size_t)b * n + (n - 1)];
      if (anchor) anchor[b] = g;
      if (stream && stream_len) {
        const int e = stream_len[b];
        if (e < stream_cap) {
          stream[(size_t)b * stream_cap + e] = g;
          stream_len[b] = e + 1;
        } else {
          set_status(status, DFLASH_STATUS_BOUNDS);
        }
      }
    }
  }
}

cudaError_t commit_rows(int32_t* len, int32_t* n_pend, int32_t* anchor, const int32_t* argmax, int batch, int n,
                        int emit, int32_t* stream, int32_t* stream_len, int stream_cap, int* status, cudaStream_t s) {
  DFL_RET(launch_pdl(commit_kernel, dim3(1), dim3(32 * ((batch + 31) / 32)), 0, s, len, n_pend, anchor, argmax, batch, n, emit, stream,
                                                       stream_len, stream_cap, status));
  count_launch();
  return cudaGetLastError();
}

// ------------------------------------------------------------------ accept + rollback
// One warp per sequence: lane i compares drafted slot i+1 with the target's
// greedy choice after slot i; the accepted count is the number of leading
// matches (first zero of the ballot).
__global__ void accept_kernel(const int32_t* __restrict__ draft, const int32_t* __restrict__ argmax, int batch,
                              int block, int32_t* len, int32_t* anchor, int32_t* n_pend, int32_t* accept_len,
                              int32_t* stream, int32_t* stream_len, int stream_cap, int* status) {
  pdl_launch();
  pdl_wait();
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= batch) {
    return;
  }
  const int32_t* d = draft + (size_t)b * block;
  const int32_t* g = argmax + (size_t)b * block;
  const bool match = (lane < block - 1) && (d[lane + 1] == g[lane]);
  const unsigned bal = __ballot_sync(0xffffffffu, match);
  const int a = __ffs(~bal) - 1;  // leading matches, <= block-1 since lanes >= block-1 vote 0
  const int e = stream_len ? stream_len[b] : 0;
  if (lane <= a && stream) {
    if (e + lane < stream_cap)
      stream[(size_t)b * stream_cap + e + lane] = g[lane];
    else
      set_status(status, DFLASH_STATUS_BOUNDS);
  }
  __syncwarp();
  if (lane == 0) {
    len[b] += a + 1;
    anchor[b] = g[a];
    n_pend[b] = a + 1;
    if (accept_len) accept_len[b] = a;
    if (stream_len) stream_len[b] = min(e + a + 1, stream_cap);
  }
}

cudaError_t accept_rollback(const int32_t* draft, const int32_t* argmax, int batch, int block, int32_t* len,
                            int32_t* anchor, int32_t* n_pend, int32_t* accept_len, int32_t* stream,
                            int32_t* stream_len, int stream_cap, int* status, cudaStream_t s) {
  const int warps = batch < 8 ? batch : 8;
  DFL_RET(launch_pdl(accept_kernel, dim3((batch + warps - 1) / warps), dim3(32 * warps), 0, s, draft, argmax, batch, block, len, anchor, n_pend,
                                                                   accept_len, stream, stream_len, stream_cap, status));
  count_launch();
  return cudaGetLastError();
}

// ------------------------------------------------------------------ teacher forcing
__global__ void teacher_force_kernel(int32_t* draft, int batch, int block, const int32_t* __restrict__ ref,
                                     int ref_stride, int ref_len, const int32_t* __restrict__ stream_len,
                                     const int32_t* __restrict__ k_draw, const int32_t* __restrict__ r_draw,
                                     int max_steps, int32_t* step, int vocab, int* status) {
  pdl_launch();
  pdl_wait();
  const int st = *step;
  const int b = threadIdx.x;
  if (b < batch) {
    if (st >= max_steps) {
      set_status(status, DFLASH_STATUS_BOUNDS);
    } else {
      const int k = k_draw[(size_t)st * batch + b];
      const int rr = r_draw[(size_t)st * batch + b];
      const int e = stream_len[b];
      const int kk = min(k, block - 1);
      int32_t* d = draft + (size_t)b * block;
      const int32_t* rf = ref + (size_t)b * ref_stride;
      if (e + kk >= ref_len || e < 1) {
        set_status(status, DFLASH_STATUS_BOUNDS);
      } else {
        for (int j = 1; j <= kk; ++j) d[j] = rf[e + j - 1];
        if (kk + 1 <= block - 1) d[kk + 1] = (int32_t)(((long long)rf[e + kk] + 1 + rr) % vocab);
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) *step = st + 1;
}

cudaError_t teacher_force(int32_t* draft, int batch, int block, const int32_t* ref, int ref_stride, int ref_len,
                          const int32_t* stream_len, const int32_t* k_draw, const int32_t* r_draw, int max_steps,
                          int32_t* step, int vocab, int* status, cudaStream_t s) {
  DFL_RET(launch_pdl(teacher_force_kernel, dim3(1), dim3(32 * ((batch + 31) / 32)), 0, s, draft, batch, block, ref, ref_stride, ref_len,
                                                              stream_len, k_draw, r_draw, max_steps, step, vocab,
                                                              status));
  count_launch();
  return cudaGetLastError();
}

}  // namespace dfl
