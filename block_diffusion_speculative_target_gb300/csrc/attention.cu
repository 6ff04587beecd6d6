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
// rows per warp, QK^T and PV on mma.sync m16n8k16 with fp32 accumulation; the
// chunk's keys and values arrive by TMA in one go (see attn_tma_kernel).
// fp32 path: CUDA-core dot products, one CTA per (chunk, head, row).
#include "common.cuh"
#include "internal.h"

namespace dfl {

constexpr int kHD = 128;
constexpr int kKT = 64;  // keys per sub-tile of the online softmax

// bf16, whole 256-position chunk per CTA loaded by TMA (2-D maps over the
// cache, 128-byte swizzle): K and V of the chunk land in shared memory as
// [d-half][key][128 B] with the 16-byte chunk index XOR-ed by key % 8, so the
// ldmatrix reads below are conflict-free.  Two mbarriers split the chunk into
// keys 0..127 and 128..255.  KS warps serve each query head of the GQA group:
// warp (h, kh) handles key half kh, and the halves merge through shared
// memory in a fixed order.  kTmaWaitNs bounds every wait.
constexpr uint64_t kTmaWaitNs = 500000000ull;
// Warps per query head (key-half split) for group sizes up to 5 (build-time).
#ifndef DFL_ATTN_KS
#define DFL_ATTN_KS 2
#endif
constexpr int kKvBytes = 4 * 256 * 128;          // K/V x d-half x 256 keys x 128 B
constexpr int kMergeFloats = 32 * 68;            // per warp: 32 lanes x (64 o + m0 m1 l0 l1)

template <int G, int KS>
struct AttnCfg {
  static constexpr int THREADS = G * KS * 32;
  static constexpr int SMEM = kKvBytes + (KS > 1 ? G * kMergeFloats * 4 : 0) + 1024 + 64;
};

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <int G, int KS>
__global__ void __launch_bounds__(G * KS * 32)
    attn_tma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const bf16* __restrict__ q, int n, int nq, int causal, long long row0, int nkv, int capacity,
                    const int32_t* __restrict__ len, float* __restrict__ part_o, float* __restrict__ part_ml,
                    int nchunk, float scale_log2, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* merge = reinterpret_cast<float*>(smem + kKvBytes);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kKvBytes + (KS > 1 ? G * kMergeFloats * 4 : 0));
  const int c = blockIdx.x, hk = blockIdx.y;
  const int nrb = (n + 15) >> 4;
  const int b = blockIdx.z / nrb, rb = blockIdx.z % nrb;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hl = warp % G, kh = warp / G;  // head within the group, key half (KS == 2)
  const int hq = hk * G + hl;
  const int g = lane >> 2, t = lane & 3;
  pdl_launch();
  pdl_wait();
  const int P = len[b];
  const int r_last = min(rb * 16 + 15, n - 1);
  const int kmax = min(causal ? P + r_last + 1 : P + n, capacity);
  const int k_begin = c * kAttnChunk;
  if (k_begin >= kmax) return;
  const int k_end = min(k_begin + kAttnChunk, kmax);
  const int valid = k_end - k_begin;  // keys of this chunk inside the visible range
  const int nhalf = valid > 128 ? 2 : 1;
  const uint32_t sbase = smem_u32(smem);
  // regions: K d-half 0, K d-half 1, V d-half 0, V d-half 1; each [256 keys][128 B]
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_barrier_init();
    const int row = (int)(row0 + ((long long)b * nkv + hk) * capacity + k_begin);
    for (int h = 0; h < nhalf; ++h) {
      mbar_arrive_expect_tx(&bar[h], 4 * 128 * 128);
      for (int reg = 0; reg < 4; ++reg) {
        const CUtensorMap* map = reg < 2 ? &tmK : &tmV;
        tma_load_2d(smem + reg * 256 * 128 + h * 128 * 128, map, &bar[h], (reg & 1) * 64, row + h * 128);
      }
    }
  }
  const int i0 = rb * 16 + g, i1 = i0 + 8;
  const int lim0 = min(causal ? P + i0 + 1 : P + n, k_end);
  const int lim1 = min(causal ? P + i1 + 1 : P + n, k_end);

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
  __syncthreads();  // barriers initialised before anyone waits on them
  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float mr0 = -INFINITY, mr1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int nsub = (valid + kKT - 1) / kKT;
  const int mi = lane >> 3, rr = lane & 7;
  bool ok = true;
  // This warp's sub-tiles (64 keys each): KS == 1 all of them; KS == 2 the two of its key half.
  const int sub_lo = KS == 1 ? 0 : 2 * kh, sub_hi = KS == 1 ? nsub : min(nsub, 2 * kh + 2);
  for (int half = 0; half < 2; ++half) {
    if (KS == 2 && half != kh) continue;
    if (2 * half >= nsub) break;
    ok = mbar_wait(&bar[half], 0, kTmaWaitNs) && ok;
    // Rows past `valid` carry whatever the cache holds there; their weights
    // are zero, so clear their values (0 * NaN would poison the sum).
    const int z0 = valid > half * 128 ? valid : half * 128, z1 = (half + 1) * 128;
    if (z0 < z1) {
      const int nthr = KS == 2 ? G * 32 : G * KS * 32;
      const int tid = KS == 2 ? threadIdx.x - kh * G * 32 : threadIdx.x;
      named_sync(1 + half, nthr);
      for (int i = tid; i < (z1 - z0) * 16; i += nthr) {
        const int key = z0 + (i >> 4), part = i & 15;  // 16 x 16 B per key row over both d-halves
        uint4* dst = reinterpret_cast<uint4*>(smem + (2 + (part >> 3)) * 256 * 128 + key * 128 + (part & 7) * 16);
        *dst = make_uint4(0u, 0u, 0u, 0u);
      }
      named_sync(1 + half, nthr);
    }
    if (KS == 1 && half == 0 && nsub > 2) continue;  // single-warp-per-head: wait for both halves first
  }
  for (int sub = sub_lo; sub < sub_hi; ++sub) {
    const int kb = k_begin + sub * kKT;
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int kp = 0; kp < 4; ++kp) {
        uint32_t r[4];
        const int key = sub * kKT + j * 8 + rr;
        const int ch = kp * 4 + mi;  // 16-byte chunk of d (0..15)
        ldmatrix_x4(r, sbase + (ch >> 3) * 256 * 128 + key * 128 + (((ch & 7) ^ (key & 7)) << 4));
        mma_bf16_16816(s[j], qa[2 * kp], r[0], r[1]);
        mma_bf16_16816(s[j], qa[2 * kp + 1], r[2], r[3]);
      }
    }
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
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      // P enters the PV product as a bf16 hi/lo pair (p = hi + lo to ~2^-17
      // relative), so the probabilities are not rounded to bf16 on the way.
      uint32_t pa[4], pl[4];
      pack_bf16_hilo(s[2 * kk][0], s[2 * kk][1], pa[0], pl[0]);
      pack_bf16_hilo(s[2 * kk][2], s[2 * kk][3], pa[1], pl[1]);
      pack_bf16_hilo(s[2 * kk + 1][0], s[2 * kk + 1][1], pa[2], pl[2]);
      pack_bf16_hilo(s[2 * kk + 1][2], s[2 * kk + 1][3], pa[3], pl[3]);
#pragma unroll
      for (int jp = 0; jp < 8; ++jp) {
        uint32_t r[4];
        const int key = sub * kKT + kk * 16 + (mi & 1) * 8 + rr;
        const int ch = 2 * jp + (mi >> 1);
        ldmatrix_x4_trans(r, sbase + 2 * 256 * 128 + (ch >> 3) * 256 * 128 + key * 128 + (((ch & 7) ^ (key & 7)) << 4));
        mma_bf16_16816(o[2 * jp], pa, r[0], r[1]);
        mma_bf16_16816(o[2 * jp + 1], pa, r[2], r[3]);
        mma_bf16_16816(o[2 * jp], pl, r[0], r[1]);
        mma_bf16_16816(o[2 * jp + 1], pl, r[2], r[3]);
      }
    }
  }
  if (!ok) {
    if (lane == 0) set_status(status, DFLASH_STATUS_TIMEOUT);
    if (lane == 0)  // bounded drain of copies still in flight
      for (int h = 0; h < nhalf; ++h) mbar_wait(&bar[h], 0, kTmaWaitNs / 4);
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  if (KS == 2) {
    // key half 1 hands its state to key half 0 of the same head
    float* mb = merge + (size_t)(hl * 32 + lane) * 68;
    if (kh == 1) {
#pragma unroll
      for (int j = 0; j < 16; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) mb[j * 4 + e] = o[j][e];
      mb[64] = mr0;
      mb[65] = mr1;
      mb[66] = l0;
      mb[67] = l1;
    }
    __syncthreads();
    if (kh == 1) return;
    const float m0b = mb[64], m1b = mb[65], l0b = mb[66], l1b = mb[67];
    const float M0 = fmaxf(mr0, m0b), M1 = fmaxf(mr1, m1b);
    const float fa0 = M0 == -INFINITY ? 0.f : exp2f(mr0 - M0), fb0 = M0 == -INFINITY ? 0.f : exp2f(m0b - M0);
    const float fa1 = M1 == -INFINITY ? 0.f : exp2f(mr1 - M1), fb1 = M1 == -INFINITY ? 0.f : exp2f(m1b - M1);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      o[j][0] = o[j][0] * fa0 + mb[j * 4 + 0] * fb0;
      o[j][1] = o[j][1] * fa0 + mb[j * 4 + 1] * fb0;
      o[j][2] = o[j][2] * fa1 + mb[j * 4 + 2] * fb1;
      o[j][3] = o[j][3] * fa1 + mb[j * 4 + 3] * fb1;
    }
    l0 = l0 * fa0 + l0b * fb0;
    l1 = l1 * fa1 + l1b * fb1;
    mr0 = M0;
    mr1 = M1;
  }
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

// Merge the chunk partials of one (row, query head): weights w_c =
// 2^(m_c - max m) staged in shared memory, then out[d] = sum_c w_c o_c[d] /
// sum_c w_c l_c.  256 threads: thread (d, half) sums one half of the chunks
// (loads unrolled for memory-level parallelism); the halves are added in a
// fixed order, so the result does not depend on other rows.
constexpr int kCombineMaxChunks = 1024;

template <typename T>
__global__ void __launch_bounds__(256)
    attn_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml, int n, int nq, int hd,
                        int causal, int capacity, const int32_t* __restrict__ len, int nchunk, T* __restrict__ out) {
  __shared__ float w[kCombineMaxChunks];
  __shared__ float lsum[kCombineMaxChunks];
  __shared__ float half1[kHD];
  __shared__ float Msh, Lsh;
  const int r = blockIdx.x, hq = blockIdx.y;
  const int b = r / n, j = r % n;
  pdl_launch();
  pdl_wait();
  const int P = len[b];
  const int lim = min(causal ? P + j + 1 : P + n, capacity);
  const int nch = min((lim + kAttnChunk - 1) / kAttnChunk, kCombineMaxChunks);
  const size_t row0 = ((size_t)r * nq + hq) * nchunk;
  for (int c = threadIdx.x; c < nch; c += blockDim.x) {
    const float2 ml = *reinterpret_cast<const float2*>(part_ml + (row0 + c) * 2);
    w[c] = ml.x;
    lsum[c] = ml.y;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -INFINITY;
    for (int c = 0; c < nch; ++c) M = fmaxf(M, w[c]);
    Msh = M;
  }
  __syncthreads();
  const float M = Msh;
  for (int c = threadIdx.x; c < nch; c += blockDim.x) w[c] = (w[c] == -INFINITY) ? 0.f : exp2f(w[c] - M);
  __syncthreads();
  if (threadIdx.x == 0) {
    float L = 0.f;
    for (int c = 0; c < nch; ++c) L += w[c] * lsum[c];
    Lsh = L;
  }
  const int d = threadIdx.x & 127, h = threadIdx.x >> 7;
  const int cmid = nch / 2;
  const int c0 = h == 0 ? 0 : cmid, c1 = h == 0 ? cmid : nch;
  float acc = 0.f;
  if (d < hd) {
    const float* po = part_o + row0 * kHD + d;
    int c = c0;
    for (; c + 8 <= c1; c += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = po[(size_t)(c + u) * kHD];
#pragma unroll
      for (int u = 0; u < 8; ++u) acc += w[c + u] * v[u];
    }
    for (; c < c1; ++c) acc += w[c] * po[(size_t)c * kHD];
  }
  if (h == 1) half1[d] = acc;
  __syncthreads();
  if (h == 0 && d < hd) out[((size_t)r * nq + hq) * hd + d] = from_f<T>((acc + half1[d]) / Lsh);
}

typedef CUresult (*PFN_encodeTiled_t)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                      const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 2-D maps over a whole bf16 cache viewed as [rows_total][128]: boxes of 64
// elements (128 B, swizzled) by 128 positions.
bool make_kv_maps(const void* k, const void* v, long long rows_total, CUtensorMap* mk, CUtensorMap* mv) {
  static PFN_encodeTiled_t fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<PFN_encodeTiled_t>(p);
  }
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

cudaError_t attention(int dtype, const void* q, int batch, int n, int nq, int nkv, int hd, int causal, const void* kc,
                      const void* vc, size_t seq_stride, size_t head_stride, int capacity, const int32_t* len,
                      const KvMaps* maps, const AttnScratch& sc, void* out, int* status, cudaStream_t s) {
  if (batch * n <= 0) return cudaSuccess;
  const int nchunk_launch = (capacity + kAttnChunk - 1) / kAttnChunk;
  if (nchunk_launch > sc.nchunk || nchunk_launch > kCombineMaxChunks || hd > kHD) return cudaErrorInvalidValue;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)hd);
  if (dtype == DFLASH_BF16) {
    if (hd != kHD || !maps) return cudaErrorInvalidValue;
    const int G = nq / nkv;
    const dim3 grid(nchunk_launch, nkv, batch * ((n + 15) / 16));
#define DFL_ATTN_CASE(GG, KS)                                                                                 \
  case GG: {                                                                                                   \
    using AC = AttnCfg<GG, KS>;                                                                                \
    static bool set = false;                                                                                   \
    if (!set) {                                                                                                \
      DFL_RET(cudaFuncSetAttribute(attn_tma_kernel<GG, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize, AC::SMEM)); \
      set = true;                                                                                              \
    }                                                                                                          \
    DFL_RET(launch_pdl(attn_tma_kernel<GG, KS>, grid, dim3(AC::THREADS), AC::SMEM, s, maps->k, maps->v,         \
                       (const bf16*)q, n, nq, causal, maps->row0, nkv, capacity, len, sc.o, sc.ml, sc.nchunk,  \
                       scale_log2, status));                                                                   \
    break;                                                                                                     \
  }
    switch (G) {
      DFL_ATTN_CASE(1, DFL_ATTN_KS)
      DFL_ATTN_CASE(2, DFL_ATTN_KS)
      DFL_ATTN_CASE(4, DFL_ATTN_KS)
      DFL_ATTN_CASE(5, DFL_ATTN_KS)
      DFL_ATTN_CASE(8, 1)
      default:
        return cudaErrorInvalidValue;
    }
#undef DFL_ATTN_CASE
    DFL_RET(launch_pdl(attn_combine_kernel<bf16>, dim3(batch * n, nq), dim3(256), 0, s, sc.o, sc.ml, n, nq, hd,
                       causal, capacity, len, sc.nchunk, (bf16*)out));
  } else {
    const dim3 grid(nchunk_launch, nq, batch * n);
    DFL_RET(launch_pdl(attn_f32_kernel<128>, grid, dim3(128), 0, s, (const float*)q, n, nq, nkv, hd, causal,
                       (const float*)kc, (const float*)vc, seq_stride, head_stride, capacity, len, sc.o, sc.ml,
                       sc.nchunk, scale_log2));
    DFL_RET(launch_pdl(attn_combine_kernel<float>, dim3(batch * n, nq), dim3(256), 0, s, sc.o, sc.ml, n, nq, hd,
                       causal, capacity, len, sc.nchunk, (float*)out));
  }
  count_launch(2);
  return cudaSuccess;
}

}  // namespace dfl
