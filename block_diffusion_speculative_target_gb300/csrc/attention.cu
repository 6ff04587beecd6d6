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
// bf16 path (head_dim 128): one warp per query head of the GQA group, 16 block
// rows per warp, QK^T and PV on mma.sync m16n8k16 with fp32 accumulation;
// K/V sub-tiles of 64 keys double-buffered in shared memory (cp.async,
// XOR-swizzled 16-byte chunks so ldmatrix is conflict-free).
// fp32 path: CUDA-core dot products, one CTA per (chunk, head, row).
#include "common.cuh"
#include "internal.h"

namespace dfl {

constexpr int kHD = 128;
constexpr int kKT = 64;  // keys per shared-memory sub-tile
constexpr int kAttnSmem = 2 * 2 * kKT * kHD * 2;  // 2 buffers x (K + V) bf16

template <int G>
__global__ void __launch_bounds__(G * 32)
    attn_bf16_kernel(const bf16* __restrict__ q, int n, int nq, int causal, const bf16* __restrict__ kc,
                     const bf16* __restrict__ vc, size_t seq_stride, size_t head_stride, int capacity,
                     const int32_t* __restrict__ len, float* __restrict__ part_o, float* __restrict__ part_ml,
                     int nchunk, float scale_log2) {
  constexpr int NT = G * 32;
  extern __shared__ __align__(128) uint8_t smem[];
  const int c = blockIdx.x, hk = blockIdx.y;
  const int nrb = (n + 15) >> 4;
  const int b = blockIdx.z / nrb, rb = blockIdx.z % nrb;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq = hk * G + warp;
  const int g = lane >> 2, t = lane & 3;
  pdl_launch();
  pdl_wait();
  const int P = len[b];
  const int r_last = min(rb * 16 + 15, n - 1);
  const int kmax = min(causal ? P + r_last + 1 : P + n, capacity);
  const int k_begin = c * kAttnChunk;
  if (k_begin >= kmax) return;
  const int k_end = min(k_begin + kAttnChunk, kmax);
  const int i0 = rb * 16 + g, i1 = i0 + 8;
  const int lim0 = min(causal ? P + i0 + 1 : P + n, k_end);
  const int lim1 = min(causal ? P + i1 + 1 : P + n, k_end);

  const bf16* kbase = kc + (size_t)b * seq_stride + (size_t)hk * head_stride;
  const bf16* vbase = vc + (size_t)b * seq_stride + (size_t)hk * head_stride;

  uint32_t qa[8][4];
  {
    const bool v0 = i0 < n, v1 = i1 < n;
    const bf16* q0 = q + ((size_t)(b * n + (v0 ? i0 : 0)) * nq + hq) * kHD;
    const bf16* q1 = q + ((size_t)(b * n + (v1 ? i1 : 0)) * nq + hq) * kHD;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int col = kk * 16 + 2 * t;
      qa[kk][0] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + col) : 0u;
      qa[kk][1] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + col) : 0u;
      qa[kk][2] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + col + 8) : 0u;
      qa[kk][3] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + col + 8) : 0u;
    }
  }
  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float mr0 = -INFINITY, mr1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  const int nsub = (k_end - k_begin + kKT - 1) / kKT;
  const uint32_t sbase = smem_u32(smem);
  auto load = [&](int sub, int buf) {
    const int kb = k_begin + sub * kKT;
    const uint32_t ks = sbase + buf * (2 * kKT * kHD * 2);
    const uint32_t vs = ks + kKT * kHD * 2;
    for (int i = threadIdx.x; i < kKT * 16; i += NT) {
      const int key = i >> 4, ch = i & 15;
      const int gk = kb + key;
      const bool valid = gk < k_end;
      const size_t off = (size_t)(valid ? gk : k_begin) * kHD + ch * 8;
      const uint32_t dst = key * 256 + ((ch ^ (key & 7)) << 4);
      cp_async16_zfill(ks + dst, kbase + off, valid);
      cp_async16_zfill(vs + dst, vbase + off, valid);
    }
    cp_async_commit();
  };

  load(0, 0);
  for (int sub = 0; sub < nsub; ++sub) {
    if (sub + 1 < nsub) {
      load(sub + 1, (sub + 1) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t ks = sbase + (sub & 1) * (2 * kKT * kHD * 2);
    const uint32_t vs = ks + kKT * kHD * 2;
    const int kb = k_begin + sub * kKT;

    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
    const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int kp = 0; kp < 4; ++kp) {
        uint32_t r[4];
        const int key = j * 8 + rr;
        const int ch = kp * 4 + mi;
        ldmatrix_x4(r, ks + key * 256 + ((ch ^ (key & 7)) << 4));
        mma_bf16_16816(s[j], qa[2 * kp], r[0], r[1]);
        mma_bf16_16816(s[j], qa[2 * kp + 1], r[2], r[3]);
      }
    }
    // mask, running max
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = kb + j * 8 + 2 * t + e;
        s[j][e] = key < lim0 ? s[j][e] * scale_log2 : -INFINITY;
        s[j][2 + e] = key < lim1 ? s[j][2 + e] * scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, s[j][e]);
        mx1 = fmaxf(mx1, s[j][2 + e]);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(mr0, mx0), mn1 = fmaxf(mr1, mx1);
    const bool dead0 = (mn0 == -INFINITY), dead1 = (mn1 == -INFINITY);
    const float al0 = dead0 ? 1.f : exp2f(mr0 - mn0);
    const float al1 = dead1 ? 1.f : exp2f(mr1 - mn1);
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        s[j][e] = dead0 ? 0.f : exp2f(s[j][e] - mn0);
        s[j][2 + e] = dead1 ? 0.f : exp2f(s[j][2 + e] - mn1);
        ps0 += s[j][e];
        ps1 += s[j][2 + e];
      }
    }
    l0 = l0 * al0 + ps0;
    l1 = l1 * al1 + ps1;
    mr0 = mn0;
    mr1 = mn1;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      o[j][0] *= al0;
      o[j][1] *= al0;
      o[j][2] *= al1;
      o[j][3] *= al1;
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int jp = 0; jp < 8; ++jp) {
        uint32_t r[4];
        const int key = kk * 16 + (mi & 1) * 8 + rr;
        const int ch = 2 * jp + (mi >> 1);
        ldmatrix_x4_trans(r, vs + key * 256 + ((ch ^ (key & 7)) << 4));
        mma_bf16_16816(o[2 * jp], pa, r[0], r[1]);
        mma_bf16_16816(o[2 * jp + 1], pa, r[2], r[3]);
      }
    }
    __syncthreads();
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  if (i0 < n) {
    const size_t row = ((size_t)(b * n + i0) * nq + hq) * nchunk + c;
    float* po = part_o + row * kHD;
#pragma unroll
    for (int j = 0; j < 16; ++j) *reinterpret_cast<float2*>(po + j * 8 + 2 * t) = make_float2(o[j][0], o[j][1]);
    if (t == 0) *reinterpret_cast<float2*>(part_ml + row * 2) = make_float2(mr0, l0);
  }
  if (i1 < n) {
    const size_t row = ((size_t)(b * n + i1) * nq + hq) * nchunk + c;
    float* po = part_o + row * kHD;
#pragma unroll
    for (int j = 0; j < 16; ++j) *reinterpret_cast<float2*>(po + j * 8 + 2 * t) = make_float2(o[j][2], o[j][3]);
    if (t == 0) *reinterpret_cast<float2*>(part_ml + row * 2) = make_float2(mr1, l1);
  }
}

// fp32: one CTA per (chunk, query head, row).
template <int NT>
__global__ void __launch_bounds__(NT)
    attn_f32_kernel(const float* __restrict__ q, int n, int nq, int nkv, int hd, int causal,
                    const float* __restrict__ kc, const float* __restrict__ vc, size_t seq_stride,
                    size_t head_stride, int capacity, const int32_t* __restrict__ len, float* __restrict__ part_o,
                    float* __restrict__ part_ml, int nchunk, float scale_log2) {
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
  const int kb = c * kAttnChunk;
  if (kb >= lim) return;
  const int ke = min(kb + kAttnChunk, lim);
  const float* kbase = kc + (size_t)b * seq_stride + (size_t)hk * head_stride;
  const float* vbase = vc + (size_t)b * seq_stride + (size_t)hk * head_stride;
  for (int i = threadIdx.x; i < hd; i += NT) qs[i] = q[((size_t)r * nq + hq) * hd + i];
  __syncthreads();
  float mx = -INFINITY;
  for (int key = kb + threadIdx.x; key < ke; key += NT) {
    const float* kr = kbase + (size_t)key * hd;
    float acc = 0.f;
    for (int i = 0; i < hd; ++i) acc = fmaf(qs[i], kr[i], acc);
    acc *= scale_log2;
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
    const float p = exp2f(sc[key - kb] - m);
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

template <typename T>
__global__ void attn_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml, int n, int nq,
                                    int hd, int causal, int capacity, const int32_t* __restrict__ len, int nchunk,
                                    T* __restrict__ out) {
  const int r = blockIdx.x, hq = blockIdx.y;
  const int b = r / n, j = r % n;
  pdl_launch();
  pdl_wait();
  const int P = len[b];
  const int lim = min(causal ? P + j + 1 : P + n, capacity);
  const int nch = (lim + kAttnChunk - 1) / kAttnChunk;
  const size_t row0 = ((size_t)r * nq + hq) * nchunk;
  float M = -INFINITY;
  for (int c = 0; c < nch; ++c) M = fmaxf(M, part_ml[(row0 + c) * 2]);
  float L = 0.f;
  for (int c = 0; c < nch; ++c) {
    const float mc = part_ml[(row0 + c) * 2];
    if (mc != -INFINITY) L += part_ml[(row0 + c) * 2 + 1] * exp2f(mc - M);
  }
  const float invL = 1.0f / L;
  for (int i = threadIdx.x; i < hd; i += blockDim.x) {
    float acc = 0.f;
    for (int c = 0; c < nch; ++c) {
      const float mc = part_ml[(row0 + c) * 2];
      if (mc != -INFINITY) acc += part_o[(row0 + c) * kHD + i] * exp2f(mc - M);
    }
    out[((size_t)r * nq + hq) * hd + i] = from_f<T>(acc * invL);
  }
}

cudaError_t attention(int dtype, const void* q, int batch, int n, int nq, int nkv, int hd, int causal, const void* kc,
                      const void* vc, size_t seq_stride, size_t head_stride, int capacity, const int32_t* len,
                      const AttnScratch& sc, void* out, int* status, cudaStream_t s) {
  (void)status;
  if (batch * n <= 0) return cudaSuccess;
  const int nchunk_launch = (capacity + kAttnChunk - 1) / kAttnChunk;
  if (nchunk_launch > sc.nchunk || hd > kHD) return cudaErrorInvalidValue;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)hd);
  if (dtype == DFLASH_BF16) {
    if (hd != kHD) return cudaErrorInvalidValue;
    const int G = nq / nkv;
    const dim3 grid(nchunk_launch, nkv, batch * ((n + 15) / 16));
#define DFL_ATTN_CASE(GG)                                                                                     \
  case GG: {                                                                                                  \
    static bool set = false;                                                                                  \
    if (!set) {                                                                                               \
      DFL_RET(cudaFuncSetAttribute(attn_bf16_kernel<GG>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem)); \
      set = true;                                                                                             \
    }                                                                                                         \
    DFL_RET(launch_pdl(attn_bf16_kernel<GG>, grid, dim3(GG * 32), kAttnSmem, s, (const bf16*)q, n, nq, causal,  \
                       (const bf16*)kc, (const bf16*)vc, seq_stride, head_stride, capacity, len, sc.o, sc.ml,  \
                       sc.nchunk, scale_log2));                                                                \
    break;                                                                                                    \
  }
    switch (G) {
      DFL_ATTN_CASE(1)
      DFL_ATTN_CASE(2)
      DFL_ATTN_CASE(4)
      DFL_ATTN_CASE(5)
      DFL_ATTN_CASE(8)
      default:
        return cudaErrorInvalidValue;
    }
#undef DFL_ATTN_CASE
    DFL_RET(launch_pdl(attn_combine_kernel<bf16>, dim3(batch * n, nq), dim3(kHD), 0, s, sc.o, sc.ml, n, nq, hd,
                       causal, capacity, len, sc.nchunk, (bf16*)out));
  } else {
    const dim3 grid(nchunk_launch, nq, batch * n);
    DFL_RET(launch_pdl(attn_f32_kernel<128>, grid, dim3(128), 0, s, (const float*)q, n, nq, nkv, hd, causal,
                       (const float*)kc, (const float*)vc, seq_stride, head_stride, capacity, len, sc.o, sc.ml,
                       sc.nchunk, scale_log2));
    DFL_RET(launch_pdl(attn_combine_kernel<float>, dim3(batch * n, nq), dim3(hd), 0, s, sc.o, sc.ml, n, nq, hd,
                       causal, capacity, len, sc.nchunk, (float*)out));
  }
  count_launch(2);
  return cudaSuccess;
}

}  // namespace dfl
