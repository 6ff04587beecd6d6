// Block-vs-cache attention on the 5th-generation tensor cores (bf16, head_dim
// 128).  A work item is one (256-position chunk, KV head, sequence, 16-row
// block); a persistent grid of at most one CTA per SM walks the items with the
// chunk index outermost, so every CTA gets an equal share of the context.
//
// The G query heads that share the KV head are stacked into one M = 128 tile
// (row r = block row (r / G), head (r % G); rows past 16 G are padding whose
// results are never read), so one tcgen05.mma serves the whole GQA group:
//   1. TMA brings the chunk's keys (two 128-key halves), its values and the
//      query tile (a [16 rows][G heads][64] box per head-dim half) into shared
//      memory, all with the 128-byte swizzle.
//   2. S = Q K^T for each key half as soon as it lands, into TMEM (f32).
//   3. Exact softmax over the chunk: thread (warp w, lane l) owns row
//      32 (w % 4) + l and keys [32 (w / 4), +32) of each 128-key half; the
//      four key groups exchange their row max and sum through shared memory
//      in a fixed order.  Masked keys (beyond the row's visible range or the
//      chunk's valid keys) get probability 0.
//   4. P enters the PV product as a bf16 hi/lo pair (p = hi + lo to about
//      2^-17 relative), written as K-major operands over the consumed key and
//      query tiles; O = P_hi V + P_lo V with V read as an MN-major operand.
//      The first half's product is issued as soon as its P is written and
//      runs while the second half is exponentiated.
//   5. O (TMEM) and the row's max/sum go out as the chunk's partial; the
//      combine kernel merges the chunks of a row in chunk order.
// As soon as an item's PV product has completed, its key, value and query
// tiles are dead: the next item's TMA loads are issued then, and land while
// this item's partial is written out.
// A row's result depends only on its own query and keys: the chunk
// boundaries are absolute and every per-row computation is row-local.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace dfl {

namespace {
constexpr int kTcThreads = 512;
constexpr int kIssuer = kTcThreads - 32;  // lane 0 of the last warp: PV products and later items' copies
constexpr uint32_t kRegK = 0;          // keys  [d-half][256 keys][128 B]; later P_hi [4 key-atoms][128 rows][128 B]
constexpr uint32_t kRegV = 65536;      // values [d-half][256 keys][128 B]
constexpr uint32_t kRegQ = 131072;     // query [d-half][128 rows][128 B]; later P_lo [4 key-atoms][128 rows][128 B] (64 KB)
constexpr uint32_t kStats = 196608;    // row max [4][128], row sum [4][128]
constexpr uint32_t kBars = kStats + 4096;
constexpr uint32_t kLens = kBars + 64;      // sequence lengths (batch <= 128)
constexpr uint32_t kNext = kLens + 512;     // the next item: index + TcItem fields
constexpr int kTcSmem = kNext + 32 + 1024;  // + alignment slack
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

// One work item: chunk c of KV head hk for 16-row block rb of sequence b.
struct TcItem {
  int c, hk, b, rb, P, k_begin, valid;
};

// Item t in chunk-major order; false when the chunk starts past the keys the
// block's rows can see (nothing to do).
__device__ __forceinline__ bool tc_item(int t, int nkv, int nrb, int batch, int n, int causal, int capacity,
                                        const int32_t* __restrict__ len, TcItem& it) {
  it.hk = t % nkv;
  int u = t / nkv;
  it.rb = u % nrb;
  u /= nrb;
  it.b = u % batch;
  it.c = u / batch;
  it.P = len[it.b];
  const int r_last = min(it.rb * 16 + 15, n - 1);
  const int kmax = min(causal ? it.P + r_last + 1 : it.P + n, capacity);
  it.k_begin = it.c * kAttnChunk;
  it.valid = min(kAttnChunk, kmax - it.k_begin);
  return it.valid > 0;
}

// First item at or after t (stride = grid size) that has work; nitems if none.
__device__ __forceinline__ int tc_next(int t, int nitems, int nkv, int nrb, int batch, int n, int causal,
                                       int capacity, const int32_t* __restrict__ len, TcItem& it) {
  for (; t < nitems; t += gridDim.x)
    if (tc_item(t, nkv, nrb, batch, n, causal, capacity, len, it)) break;
  return t;
}

template <int G>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmQ, int batch, int n, int nq, int causal, long long row0, int nkv,
                   int capacity, const int32_t* __restrict__ len, float* __restrict__ part_o,
                   float* __restrict__ part_ml, int nchunk, int nitems, float scale_log2, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* st_max = reinterpret_cast<float*>(sm + kStats);
  float* st_sum = st_max + 512;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kBars);  // K half 0, K half 1, V, S done, O done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 5);
  int* okf = reinterpret_cast<int*>(tslot + 1);
  int* pend = okf + 1;  // copies issued whose completion has not been seen yet
  int* len_s = reinterpret_cast<int*>(sm + kLens);
  int* next_s = reinterpret_cast<int*>(sm + kNext);
  const int nrb = (n + 15) >> 4;
  const int qbox = min(16, batch * n);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {  // the descriptors are kernel parameters: fetch them while the previous kernel drains
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  pdl_launch();
  pdl_wait();

  // Query, key and value tiles of an item: both 128-key halves always (a half
  // past the valid keys reads masked keys or the fill value), so each barrier
  // completes exactly once per item.  The query tile rides on the first key
  // half's barrier.  Query rows past the block (the next sequence's rows or
  // the fill value) are masked like the padding rows; so are rows at or past
  // the box height qbox = min(16, batch * n), which are past the block.
  auto issue_loads = [&](const TcItem& it) {
    const int row = (int)(row0 + ((long long)it.b * nkv + it.hk) * capacity + it.k_begin);
    mbar_arrive_expect_tx(&bar[0], 2 * 128 * 128 + 2 * 128 * G * qbox);
    for (int dh = 0; dh < 2; ++dh)
      tma_load_3d(sm + kRegQ + dh * 16384, &tmQ, &bar[0], dh * 64, it.hk * G, it.b * n + it.rb * 16);
    for (int h = 0; h < 2; ++h) {
      if (h) mbar_arrive_expect_tx(&bar[h], 2 * 128 * 128);
      for (int dh = 0; dh < 2; ++dh)
        tma_load_2d(sm + kRegK + dh * 32768 + h * 16384, &tmK, &bar[h], dh * 64, row + h * 128);
    }
    mbar_arrive_expect_tx(&bar[2], 2 * 2 * 128 * 128);
    for (int h = 0; h < 2; ++h)
      for (int dh = 0; dh < 2; ++dh)
        tma_load_2d(sm + kRegV + dh * 32768 + h * 16384, &tmV, &bar[2], dh * 64, row + h * 128);
  };
  TcItem cur;
  int t = tc_next(blockIdx.x, nitems, nkv, nrb, batch, n, causal, capacity, len, cur);
  if (t >= nitems) return;  // uniform over the CTA: no item with work
  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(&bar[i], 1);
    fence_barrier_init();
    *okf = 1;
    issue_loads(cur);
    *pend = 1;
  }
  if (warp == 0) tmem_alloc(tslot, kTmemCols);
  for (int i = tid; i < batch; i += kTcThreads) len_s[i] = len[i];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tS = tmem, tO = tmem + 256;

  // softmax roles: row r, 64-key quarter cq
  const int q4 = warp & 3, cq = warp >> 2;
  const int r = q4 * 32 + lane;
  const int ri = r / G, hl = r - ri * G;  // block row and head of tile row r
  // warp-uniform: this warp's rows are real (rows past 16 G are padding)
  const bool live = q4 * 32 < 16 * G;
  uint32_t ph = 0;
#pragma unroll 1
  while (t < nitems) {
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();  // the query tile is staged; the previous item's partial has been read out of TMEM
    tc_fence_after();
    if (!*okf) break;
    const int valid = cur.valid;
    if (tid == kIssuer) {  // decode the next item now, off the path from the PV product to its copies
      TcItem nx;
      next_s[0] = tc_next(t + gridDim.x, nitems, nkv, nrb, batch, n, causal, capacity, len_s, nx);
      next_s[1] = nx.c, next_s[2] = nx.hk, next_s[3] = nx.b, next_s[4] = nx.rb;
      next_s[5] = nx.P, next_s[6] = nx.k_begin, next_s[7] = nx.valid;
    }

    // ---- S = Q K^T per key half
    if (tid == 0) {
      const uint32_t idS = idesc_bf16_f32(128, 128);
      bool ok = true;
      for (int h = 0; h < 2 && ok; ++h) {
        ok = mbar_wait(&bar[h], ph, kTcWaitNs);
        if (!ok) break;
        tc_fence_after();
        if (h * 128 >= valid) continue;  // no valid key in this half
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int dh = kk >> 2;
          const uint64_t a = smem_desc_sw128(sm + kRegQ + dh * 16384) + (uint64_t)(((kk & 3) * 32) >> 4);
          const uint64_t bk =
              smem_desc_sw128(sm + kRegK + dh * 32768 + h * 16384) + (uint64_t)(((kk & 3) * 32) >> 4);
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
    const bool okv = mbar_wait(&bar[2], ph, kTcWaitNs);
    if (tid == 0 && okv && *okf) *pend = 0;  // thread 0 has seen all three copies land
    if (okv && valid < 256) {
      for (int i = tid; i < (256 - valid) * 16; i += kTcThreads) {
        const int key = valid + (i >> 4), part = i & 15;
        *reinterpret_cast<uint4*>(sm + kRegV + (part >> 3) * 32768 + key * 128 + (part & 7) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
    }
    const bool oks = mbar_wait(&bar[3], ph, kTcWaitNs);
    tc_fence_after();
    if (!(okv && oks) && lane == 0) {
      *okf = 0;
      set_status(status, DFLASH_STATUS_TIMEOUT);
    }

    // ---- softmax over the chunk, in two 128-key halves: thread (q4, cq) owns
    // row r and keys [32 cq, 32 cq + 32) of each half (sv[0..31], sv[32..63]).
    const int qi = cur.rb * 16 + ri;
    const bool row_ok = r < 16 * G && qi < n;
    // visible keys of this row in the chunk (0 for rows outside the group/block)
    const int lim = row_ok ? min(causal ? cur.P + qi + 1 : cur.P + n, cur.k_begin + valid) - cur.k_begin : 0;
    const int c0 = cq * 32;
    const bool have0 = live && c0 < valid, have1 = live && 128 + c0 < valid;
    float sv[64];
    float mx = -INFINITY;
    if (have0) {  // columns of a half with no valid key hold stale scores: all masked below
      const uint32_t lb = (uint32_t)(q4 * 32) << 16;
      uint32_t raw[4][16];
      tmem_ld16_nowait(tS + lb + c0, raw[0]);
      tmem_ld16_nowait(tS + lb + c0 + 16, raw[1]);
      tmem_ld16_nowait(tS + lb + 128 + c0, raw[2]);
      tmem_ld16_nowait(tS + lb + 128 + c0 + 16, raw[3]);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 16; ++e) sv[j * 16 + e] = __uint_as_float(raw[j][e]);
      if (lim >= 128 + c0 + 32) {
#pragma unroll
        for (int x = 0; x < 64; ++x) mx = fmaxf(mx, sv[x]);
      } else {
#pragma unroll
        for (int x = 0; x < 64; ++x) {
          const int key = (x < 32 ? 0 : 96) + c0 + x;
          sv[x] = key < lim ? sv[x] : -INFINITY;
          mx = fmaxf(mx, sv[x]);
        }
      }
    }
    st_max[cq * 128 + r] = mx;
    __syncthreads();
    // chunk row max in log2 units (scale > 0, so max(s) * scale = max(s * scale))
    const float M = fmaxf(fmaxf(st_max[r], st_max[128 + r]), fmaxf(st_max[256 + r], st_max[384 + r])) * scale_log2;
    const float negM = M == -INFINITY ? 0.f : -M;
    float ls = 0.f;
    // P of one half as bf16 hi/lo pairs: keys 128 hf + c0 + 8 j8 .. +7 sit in
    // 64-key atom 2 hf + (cq >> 1), 16-byte chunk 4 (cq & 1) + j8 of row r.
    auto write_p = [&](int hf) {
#pragma unroll
      for (int j8 = 0; j8 < 4; ++j8) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = ex2(fmaf(sv[hf * 32 + j8 * 8 + 2 * e], scale_log2, negM));
          const float p1 = ex2(fmaf(sv[hf * 32 + j8 * 8 + 2 * e + 1], scale_log2, negM));
          ls += p0;
          ls += p1;
          pack_bf16_hilo(p0, p1, hi[e], lo[e]);
        }
        const int ch = (cq & 1) * 4 + j8;
        const uint32_t off = (uint32_t)(2 * hf + (cq >> 1)) * 16384 + r * 128 + ((ch ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(sm + kRegK + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(sm + kRegQ + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    };
    // O += P_hi V + P_lo V over the 16-key steps [k0, k1) of the chunk
    const int nks = (valid + 15) >> 4;
    auto issue_pv = [&](int k0, int k1) {
      const uint32_t idO = idesc_bf16_f32(128, 128) | (1u << 16);  // B (values) MN-major
      for (int pass = 0; pass < 2; ++pass)
        for (int kk = k0; kk < k1; ++kk) {
          const uint64_t a = smem_desc_sw128(sm + (pass ? kRegQ : kRegK) + (kk >> 2) * 16384) +
                             (uint64_t)(((kk & 3) * 32) >> 4);
          const uint64_t bv = smem_desc_mn_sw128(smem_u32(sm + kRegV) + kk * 2048, 32768);
          tc_mma_f16(tO, a, bv, idO, (pass | kk) ? 1u : 0u);
        }
    };
    if (have0) write_p(0);
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();  // P of the first half is in place
    tc_fence_after();
    // issued from the last warp (padding rows whenever 16 G <= 96) so that no
    // row's second half waits for the issue; runs while the second half is exponentiated
    if (tid == kIssuer && *okf) issue_pv(0, min(nks, 8));
    if (have1) write_p(1);
    st_sum[cq * 128 + r] = ls;
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const float L = ((st_sum[r] + st_sum[128 + r]) + st_sum[256 + r]) + st_sum[384 + r];
    if (tid == kIssuer) {
      if (*okf && nks > 8) issue_pv(8, nks);
      tc_commit(&bar[4]);
    }
    const bool oko = mbar_wait(&bar[4], ph, kTcWaitNs);
    tc_fence_after();
    const bool good = *okf && okv && oks && oko;
    if (!oko && lane == 0) {
      *okf = 0;
      set_status(status, DFLASH_STATUS_TIMEOUT);
    }

    // ---- the tiles are dead: start the next item's loads.  The issuing lane
    // belongs to the last warp, which holds padding rows whenever 16 G <= 96, so
    // the copies go out while the other warps write the partial.
    if (tid == kIssuer && next_s[0] < nitems && good) {
      const TcItem nx{next_s[1], next_s[2], next_s[3], next_s[4], next_s[5], next_s[6], next_s[7]};
      issue_loads(nx);
      *pend = 1;
    }

    // ---- partial out, in two 64-column passes staged through shared memory so
    // that each row leaves as one contiguous 256-byte store: the staging area is
    // the second half of the P_lo region (dead once the PV product completed, and
    // outside the next item's copies), rows of 256 B with the 16-byte chunks
    // XOR-swizzled by (row & 7) so that eight lanes writing eight rows hit
    // distinct banks.
    uint8_t* stg = sm + kRegQ + 32768;
    const int rows_live = min(16 * G, 128);
    for (int pass = 0; pass < 2; ++pass) {
      if (live) {  // warp (q4, cq) moves columns 64 pass + 16 cq .. +15 of its rows
        uint32_t raw[16];
        tmem_ld16_nowait(tO + ((uint32_t)(q4 * 32) << 16) + pass * 64 + cq * 16, raw);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(stg + r * 256 + (((cq * 4 + c) ^ (r & 7)) << 4)) =
              make_uint4(raw[4 * c], raw[4 * c + 1], raw[4 * c + 2], raw[4 * c + 3]);
      }
      __syncthreads();
      if (good) {
        for (int idx = tid; idx < rows_live * 16; idx += kTcThreads) {
          const int rr = idx >> 4, ch = idx & 15;
          const int ir = rr / G, hr = rr - ir * G, qr = cur.rb * 16 + ir;
          if (qr < n) {
            const size_t prow = ((size_t)(cur.b * n + qr) * nq + cur.hk * G + hr) * nchunk + cur.c;
            *reinterpret_cast<uint4*>(part_o + prow * 128 + pass * 64 + ch * 4) =
                *reinterpret_cast<const uint4*>(stg + rr * 256 + ((ch ^ (rr & 7)) << 4));
          }
        }
      }
      if (pass == 0) __syncthreads();  // the staging area is rewritten by the second pass
    }
    if (live && row_ok && good && cq == 0) {
      const size_t prow = ((size_t)(cur.b * n + qi) * nq + cur.hk * G + hl) * nchunk + cur.c;
      *reinterpret_cast<float2*>(part_ml + prow * 2) = make_float2(M, L);
    }
    t = next_s[0];  // written before the syncs above
    cur = TcItem{next_s[1], next_s[2], next_s[3], next_s[4], next_s[5], next_s[6], next_s[7]};
    ph ^= 1;
  }
  __syncthreads();
  if (tid == 0 && *pend) {  // after a failure: bounded drain of copies that may still be in flight
    for (int h = 0; h < 3; ++h) mbar_wait(&bar[h], ph, kTcWaitNs / 4);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

cudaError_t attention_tc(int G, const KvMaps& maps, const CUtensorMap& qmap, int batch, int n, int nq, int nkv, int causal,
                         int capacity, const int32_t* len, const AttnScratch& sc, int nchunk_launch, float scale_log2,
                         int* status, cudaStream_t s) {
  const long long items = (long long)nchunk_launch * nkv * batch * ((n + 15) / 16);
  if (items <= 0) return cudaSuccess;
  if (items > INT32_MAX || batch > kMaxRows) return cudaErrorInvalidValue;
  const int nitems = (int)items;
  const dim3 grid((unsigned)std::min<long long>(items, num_sms()));
#define DFL_TC_CASE(GG)                                                                                       \
  case GG: {                                                                                                   \
    static bool set = false;                                                                                   \
    if (!set) {                                                                                                \
      DFL_RET(cudaFuncSetAttribute(attn_tc_kernel<GG>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem)); \
      set = true;                                                                                              \
    }                                                                                                          \
    DFL_RET(launch_pdl(attn_tc_kernel<GG>, grid, dim3(kTcThreads), kTcSmem, s, maps.k, maps.v, qmap, batch, n, nq, \
                       causal, maps.row0, nkv, capacity, len, sc.o, sc.ml, sc.nchunk, nitems, scale_log2,      \
                       status));                                                                               \
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
