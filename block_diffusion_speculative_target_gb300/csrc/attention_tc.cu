// Block-vs-cache attention on the 5th-generation tensor cores (bf16, head_dim
// 128), one CTA per (256-position chunk, KV head, sequence, 16-row block).
//
// The G query heads that share the KV head are stacked into one M = 128 tile
// (row r = head (r / 16), block row (r % 16); rows past 16 G are zero), so
// one tcgen05.mma serves the whole GQA group:
//   1. TMA brings the chunk's keys (two 128-key halves) and values into
//      shared memory (128-byte swizzle); the threads stage the query tile.
//   2. S = Q K^T for each key half as soon as it lands, into TMEM (f32).
//   3. Exact softmax over the chunk: thread (warp w, lane l) owns row
//      32 (w % 4) + l and the 64-key quarter w / 4; the four quarters
//      exchange their row max and sum through shared memory in a fixed
//      order.  Masked keys (beyond the row's visible range or the chunk's
//      valid keys) get probability 0.
//   4. P enters the PV product as a bf16 hi/lo pair (p = hi + lo to about
//      2^-17 relative), written as K-major operands over the consumed key and
//      query tiles; O = P_hi V + P_lo V with V read as an MN-major operand.
//   5. O (TMEM) and the row's max/sum go out as the chunk's partial; the
//      combine kernel merges the chunks of a row in chunk order.
// A row's result depends only on its own query and keys: the chunk
// boundaries are absolute and every per-row computation is row-local.
#include "common.cuh"
#include "internal.h"

namespace dfl {

namespace {
constexpr int kTcThreads = 512;
constexpr uint32_t kRegK = 0;          // keys  [d-half][256 keys][128 B]; later P_hi [4 key-atoms][128 rows][128 B]
constexpr uint32_t kRegV = 65536;      // values [d-half][256 keys][128 B]
constexpr uint32_t kRegQ = 131072;     // query [d-half][128 rows][128 B]; later P_lo [4 key-atoms][128 rows][128 B] (64 KB)
constexpr uint32_t kStats = 196608;    // row max [4][128], row sum [4][128]
constexpr uint32_t kBars = kStats + 4096;
constexpr int kTcSmem = kBars + 64 + 1024;  // + barriers/slot/flag + alignment slack
constexpr uint32_t kTmemCols = 512;    // S: columns 0..255, O: 256..383
constexpr uint64_t kTcWaitNs = 500000000ull;

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2^x on the SFU (ex2.approx, flush-to-zero; exact 0 for -inf).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 32 lanes x 32 bits, 16 consecutive columns, without waiting for completion.
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// MN-major operand in 128-byte swizzled rows (the layout a TMA load of
// [key][64 x bf16] boxes writes): 8-row groups 1024 B apart (stride byte
// offset), 64-element column blocks `block_stride` bytes apart (leading byte
// offset).
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t addr, uint32_t block_stride) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)((block_stride >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
}  // namespace

template <int G>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const bf16* __restrict__ q, int n, int nq, int causal, long long row0, int nkv, int capacity,
                   const int32_t* __restrict__ len, float* __restrict__ part_o, float* __restrict__ part_ml,
                   int nchunk, float scale_log2, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* st_max = reinterpret_cast<float*>(sm + kStats);
  float* st_sum = st_max + 512;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kBars);  // K half 0, K half 1, V, S done, O done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 5);
  int* okf = reinterpret_cast<int*>(tslot + 1);
  const int c = blockIdx.x, hk = blockIdx.y;
  const int nrb = (n + 15) >> 4;
  const int b = blockIdx.z / nrb, rb = blockIdx.z % nrb;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_launch();
  pdl_wait();
  const int P = len[b];
  const int r_last = min(rb * 16 + 15, n - 1);
  const int kmax = min(causal ? P + r_last + 1 : P + n, capacity);
  const int k_begin = c * kAttnChunk;
  if (k_begin >= kmax) return;  // uniform over the CTA
  const int k_end = min(k_begin + kAttnChunk, kmax);
  const int valid = k_end - k_begin;
  const int nk = valid > 128 ? 2 : 1;

  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(&bar[i], 1);
    fence_barrier_init();
    *okf = 1;
    const int row = (int)(row0 + ((long long)b * nkv + hk) * capacity + k_begin);
    for (int h = 0; h < nk; ++h) {
      mbar_arrive_expect_tx(&bar[h], 2 * 128 * 128);
      for (int dh = 0; dh < 2; ++dh) tma_load_2d(sm + kRegK + dh * 32768 + h * 16384, &tmK, &bar[h], dh * 64, row + h * 128);
    }
    mbar_arrive_expect_tx(&bar[2], nk * 2 * 128 * 128);
    for (int h = 0; h < nk; ++h)
      for (int dh = 0; dh < 2; ++dh) tma_load_2d(sm + kRegV + dh * 32768 + h * 16384, &tmV, &bar[2], dh * 64, row + h * 128);
  }
  if (warp == 0) tmem_alloc(tslot, kTmemCols);
  {  // query tile: thread t stages a quarter (32 elements) of row t / 4 (zero rows past the group or the block)
    const int r = tid >> 2, part = tid & 3, dh = part >> 1;
    const int hl = r >> 4, qi = rb * 16 + (r & 15);
    const bool v = hl < G && qi < n;
    const bf16* src = q + ((size_t)(b * n + (v ? qi : 0)) * nq + hk * G + (v ? hl : 0)) * 128 + part * 32;
    uint8_t* dst = sm + kRegQ + dh * 16384 + r * 128;
    uint4 val[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) val[i] = v ? *reinterpret_cast<const uint4*>(src + i * 8) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int ch = (part & 1) * 4 + i;
      *reinterpret_cast<uint4*>(dst + ((ch ^ (r & 7)) << 4)) = val[i];
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tS = tmem, tO = tmem + 256;

  // ---- S = Q K^T per key half
  if (tid == 0) {
    const uint32_t idS = idesc_bf16_f32(128, 128);
    bool ok = true;
    for (int h = 0; h < nk && ok; ++h) {
      ok = mbar_wait(&bar[h], 0, kTcWaitNs);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int dh = kk >> 2;
        const uint64_t a = smem_desc_sw128(sm + kRegQ + dh * 16384) + (uint64_t)(((kk & 3) * 32) >> 4);
        const uint64_t bk = smem_desc_sw128(sm + kRegK + dh * 32768 + h * 16384) + (uint64_t)(((kk & 3) * 32) >> 4);
        tc_mma_f16(tS + h * 128, a, bk, idS, kk > 0 ? 1u : 0u);
      }
    }
    if (!ok) {
      *okf = 0;
      set_status(status, DFLASH_STATUS_TIMEOUT);
    }
    tc_commit(&bar[3]);
  }

  // ---- values: clear rows past the valid keys (their weight is 0, and 0 * NaN would poison the sum)
  bool okv = mbar_wait(&bar[2], 0, kTcWaitNs);
  if (okv && valid < nk * 128) {
    const int z0 = valid, z1 = nk * 128;
    for (int i = tid; i < (z1 - z0) * 16; i += kTcThreads) {
      const int key = z0 + (i >> 4), part = i & 15;
      *reinterpret_cast<uint4*>(sm + kRegV + (part >> 3) * 32768 + key * 128 + (part & 7) * 16) =
          make_uint4(0u, 0u, 0u, 0u);
    }
  }
  const bool oks = mbar_wait(&bar[3], 0, kTcWaitNs);
  tc_fence_after();
  if (!(okv && oks) && lane == 0) set_status(status, DFLASH_STATUS_TIMEOUT);

  // ---- softmax: row r, 64-key quarter cq
  const int q4 = warp & 3, cq = warp >> 2;
  const int r = q4 * 32 + lane;
  const int hl = r >> 4, qi = rb * 16 + (r & 15);
  const bool row_ok = hl < G && qi < n;
  // visible keys of this row in the chunk (0 for rows outside the group/block)
  const int lim = row_ok ? min(causal ? P + qi + 1 : P + n, k_end) - k_begin : 0;
  const int c0 = cq * 64;
  // warp-uniform: this quarter's scores exist and its rows are real (rows past 16 G are padding)
  const bool live = q4 * 32 < 16 * G;
  const bool have = live && c0 < nk * 128;
  float sv[64];
  float mx = -INFINITY;
  if (have) {
    uint32_t raw[4][16];
#pragma unroll
    for (int j = 0; j < 4; ++j) tmem_ld16_nowait(tS + ((uint32_t)(q4 * 32) << 16) + c0 + j * 16, raw[j]);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 16; ++e) sv[j * 16 + e] = __uint_as_float(raw[j][e]);
    if (lim >= c0 + 64) {
#pragma unroll
      for (int j = 0; j < 64; ++j) mx = fmaxf(mx, sv[j]);
    } else {
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        sv[j] = c0 + j < lim ? sv[j] : -INFINITY;
        mx = fmaxf(mx, sv[j]);
      }
    }
  }
  st_max[cq * 128 + r] = mx;
  __syncthreads();
  // chunk row max in log2 units (scale > 0, so max(s) * scale = max(s * scale))
  const float M = fmaxf(fmaxf(st_max[r], st_max[128 + r]), fmaxf(st_max[256 + r], st_max[384 + r])) * scale_log2;
  const float negM = M == -INFINITY ? 0.f : -M;
  float ls = 0.f;
  if (have) {
#pragma unroll
    for (int j8 = 0; j8 < 8; ++j8) {
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p0 = ex2(fmaf(sv[j8 * 8 + 2 * e], scale_log2, negM));
        const float p1 = ex2(fmaf(sv[j8 * 8 + 2 * e + 1], scale_log2, negM));
        ls += p0;
        ls += p1;
        pack_bf16_hilo(p0, p1, hi[e], lo[e]);
      }
      const uint32_t off = (uint32_t)cq * 16384 + r * 128 + ((j8 ^ (r & 7)) << 4);
      *reinterpret_cast<uint4*>(sm + kRegK + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(sm + kRegQ + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
  st_sum[cq * 128 + r] = ls;
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const float L = ((st_sum[r] + st_sum[128 + r]) + st_sum[256 + r]) + st_sum[384 + r];

  // ---- O = P_hi V + P_lo V
  if (tid == 0) {
    if (*okf && okv && oks) {
      const uint32_t idO = idesc_bf16_f32(128, 128) | (1u << 16);  // B (values) MN-major
      const int nks = (valid + 15) >> 4;
      for (int pass = 0; pass < 2; ++pass)
        for (int kk = 0; kk < nks; ++kk) {
          const uint64_t a = smem_desc_sw128(sm + (pass ? kRegQ : kRegK) + (kk >> 2) * 16384) +
                             (uint64_t)(((kk & 3) * 32) >> 4);
          const uint64_t bv = smem_desc_mn_sw128(smem_u32(sm + kRegV) + kk * 2048, 32768);
          tc_mma_f16(tO, a, bv, idO, (pass | kk) ? 1u : 0u);
        }
    }
    tc_commit(&bar[4]);
  }
  const bool oko = mbar_wait(&bar[4], 0, kTcWaitNs);
  tc_fence_after();
  const bool good = *okf && okv && oks && oko;
  if (!oko && lane == 0) set_status(status, DFLASH_STATUS_TIMEOUT);

  // ---- partial out: warp (q4, cq) writes columns 32 * cq .. +31 of its rows
  if (live) {
    uint32_t raw[2][16];
    tmem_ld16_nowait(tO + ((uint32_t)(q4 * 32) << 16) + cq * 32, raw[0]);
    tmem_ld16_nowait(tO + ((uint32_t)(q4 * 32) << 16) + cq * 32 + 16, raw[1]);
    tmem_ld_wait();
    if (row_ok && good) {
      const size_t prow = ((size_t)(b * n + qi) * nq + hk * G + hl) * nchunk + c;
      float4* po = reinterpret_cast<float4*>(part_o + prow * 128 + cq * 32);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        po[j] = make_float4(__uint_as_float(raw[j >> 2][(j & 3) * 4]), __uint_as_float(raw[j >> 2][(j & 3) * 4 + 1]),
                            __uint_as_float(raw[j >> 2][(j & 3) * 4 + 2]), __uint_as_float(raw[j >> 2][(j & 3) * 4 + 3]));
      if (cq == 0) *reinterpret_cast<float2*>(part_ml + prow * 2) = make_float2(M, L);
    }
  }
  if (!good && tid == 0) {  // bounded drain of copies that may still be in flight
    for (int h = 0; h < nk; ++h) mbar_wait(&bar[h], 0, kTcWaitNs / 4);
    mbar_wait(&bar[2], 0, kTcWaitNs / 4);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

cudaError_t attention_tc(int G, const KvMaps& maps, const bf16* q, int batch, int n, int nq, int nkv, int causal,
                         int capacity, const int32_t* len, const AttnScratch& sc, int nchunk_launch, float scale_log2,
                         int* status, cudaStream_t s) {
  const dim3 grid(nchunk_launch, nkv, batch * ((n + 15) / 16));
#define DFL_TC_CASE(GG)                                                                                       \
  case GG: {                                                                                                   \
    static bool set = false;                                                                                   \
    if (!set) {                                                                                                \
      DFL_RET(cudaFuncSetAttribute(attn_tc_kernel<GG>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem)); \
      set = true;                                                                                              \
    }                                                                                                          \
    DFL_RET(launch_pdl(attn_tc_kernel<GG>, grid, dim3(kTcThreads), kTcSmem, s, maps.k, maps.v, q, n, nq, causal, \
                       maps.row0, nkv, capacity, len, sc.o, sc.ml, sc.nchunk, scale_log2, status));            \
    return cudaSuccess;                                                                                        \
  }
  switch (G) {
    DFL_TC_CASE(1)
    DFL_TC_CASE(2)
    DFL_TC_CASE(4)
    DFL_TC_CASE(5)
    DFL_TC_CASE(8)
    default:
      return cudaErrorInvalidValue;
  }
#undef DFL_TC_CASE
}

}  // namespace dfl
