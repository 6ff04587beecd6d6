// Block-vs-cache attention on the 5th-generation tensor cores (bf16, head_dim
// 128), warp-specialised and pipelined over 128-key tiles.
//
// Work unit (one CTA): KV head hk, 16-row block rb of sequence b, key group gi
// = `gtiles` consecutive 128-key tiles at absolute positions
// [gi * gtiles * 128, (gi + 1) * gtiles * 128).  The group size is a property
// of the cache (fixed when it is allocated), so the arithmetic below depends
// only on absolute positions: a row's result is the same whether it is
// computed alone or in a block, and in any batch.
//
// The G query heads that share the KV head are stacked into one M = 128 tile
// (row r = block row r / G, head r % G; rows past 16 G are padding), so one
// tcgen05.mma serves the whole GQA group.  Per tile t of the unit, per row:
//   S_t = Q K_t^T                         tensor cores, fp32 in TMEM (two buffers)
//   reference max M: set by the first tile with a visible key, raised to a
//     later tile's max only when that exceeds M by more than 8 (log2 units);
//     when it is raised, O and the row sum L are rescaled by 2^(M_old - M_new)
//   p = 2^(s - M) for visible keys (<= 2^8), else 0; L += sum of p
//   P_t = p as a bf16 hi/lo pair (p = hi + lo to about 2^-17 relative)
//         written over S_t in TMEM
//   O += P_hi V_t + P_lo V_t              tensor cores, A operand from TMEM,
//                                         O accumulated in TMEM over the unit
// and the unit writes one partial (M, L, O) per (row, head); the combine
// kernel merges the groups of a row in group order.  The decisions (when M
// moves) are row-local, so they too depend only on the row's keys.
//
// Roles (320 threads): warp 0 lane 0 streams Q and the K/V tiles through a
// TMA ring; warp 1 owns TMEM and its lane 0 issues the products (QK^T of tile
// t while P_{t-1} is being computed, PV of tile t-1 as soon as its P is in
// TMEM); warps 2..9 each own TMEM lane quarter (warp & 3) and one half of the
// key columns ((warp - 2) >> 2).  Each half writes P only over its own 64
// score columns; the two halves of a row exchange their maxima through
// shared memory on an mbarrier.  Every wait is bounded; a wait that gives up
// sets DFLASH_STATUS_TIMEOUT, the unit writes nothing, and the CTA drains its
// copies and products before releasing TMEM.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace dfl {

namespace {
constexpr int kFaThreads = 320;
constexpr uint32_t kTileBytes = 128 * 256;           // 128 keys x 128 dims bf16, two 64-dim halves
constexpr uint32_t kStageBytes = 2 * kTileBytes;     // keys then values
constexpr uint32_t kTmemCols = 512;                  // S0 S1 (P written over S) | O0 O1

// Shared-memory layout per GQA group size G: a 3-stage ring when the query
// tile (16 G rows) leaves room in its 128-row region for the two halves'
// row-maximum exchange [2 buffers][2 halves][128 rows] (G <= 5), else a
// 2-stage ring with the exchange after the query tile.
template <int G>
struct FaLayout {
  static constexpr int kStages = G <= 5 ? 3 : 2;
  static constexpr uint32_t kQ = kStages * kStageBytes;                     // query [d-half][128 rows][128 B]
  static constexpr uint32_t kXch = G <= 5 ? kQ + 16 * G * 128 : kQ + 32768; // exchange, 2 KB
  static constexpr uint32_t kBar = G <= 5 ? kQ + 32768 : kXch + 2048;       // barriers, TMEM slot, abort flag
  static constexpr int kSmem = kBar + 256 + 1024;                           // + alignment slack
  static_assert(G > 5 || 16 * G * 128 + 2048 <= 16384, "exchange must fit in the query tile's padding rows");
};

// 8-bit caches (G <= 5): a 3-stage ring of byte tiles as the TMA lands them
// (key codes, value codes, then their 128 key and 128 value scales), one
// half-precision key tile and one value tile built from them (the bf16
// ring's stage layout), the query tile, and in the query
// tile's padding rows the maxima exchange and the barriers.  Three byte
// stages keep more codes in flight against the DRAM latency than two byte
// and two half stages did.
template <int G>
struct FaLayoutQ8 {
  static constexpr int kU8Stages = 3;
  static constexpr uint32_t kU8Stage = 2 * 16384 + 2 * 512;
  static constexpr uint32_t kF = kU8Stages * kU8Stage;          // half keys, then half values
  static constexpr uint32_t kQ = kF + kStageBytes;
  static constexpr uint32_t kXch = kQ + 16 * G * 128;           // half 0 padding: exchange, 2 KB
  static constexpr uint32_t kBar = kQ + 16384 + 16 * G * 128;   // half 1 padding: barriers, TMEM slot, abort
  static constexpr int kSmem = kQ + 32768 + 1024;
  // (G > 5 leaves no padding rows: the launcher refuses 8-bit caches there)
  static_assert(G > 5 || 16 * G * 128 + 2048 <= 16384, "the exchange must fit in the padding rows");
  static_assert(kF % 1024 == 0 && kQ % 1024 == 0, "operand tiles are 1024-byte aligned");
  static_assert(kSmem <= 232448, "shared memory per block");
};
constexpr uint64_t kFaWaitNs = 500000000ull;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 32 lanes x 32 bits, 32 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem], kind::f16: A (M = 128 rows = TMEM lanes,
// K along the columns, two bf16 per 32-bit column) read from TMEM.
__device__ __forceinline__ void tc_mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// MN-major operand in 128-byte swizzled rows (a TMA load of [key][64 x bf16]
// boxes): 8-row groups 1024 B apart, 64-element column blocks `block_stride`
// bytes apart.
__device__ __forceinline__ uint64_t smem_desc_mn(uint32_t addr, uint32_t block_stride) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)((block_stride >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
}  // namespace

// Q8: the cache holds 8-bit codes u = q + 128 with a float32 scale per key or
// value row, and the products run in IEEE half precision.  The converter
// warps (those whose TMEM lane quarter holds only padding rows) turn each
// byte tile into half operands: a byte permute places u under the exponent
// of 1024 (the half 1024 + u, exact), a subtraction of 1152 leaves q, and a
// multiplication by the row's scale rounded to half gives the entry
// round(q * half(s)).  The keys of a tile are converted into the one half
// key tile as soon as the previous tile's Q K^T has read it (its S exists),
// its values into the one half value tile once the previous P V is done;
// each is released on its own barrier, so neither waits on the other, and
// the byte ring runs three tiles ahead.  The query arrives in half
// precision, P is a half hi/lo pair, and the softmax is the bf16 path's.
template <int G, bool Q8>
__global__ void __launch_bounds__(kFaThreads, 1)
    attn_fa_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmQ, int batch, int n, int nq, int nkv, int causal, int window,
                   long long row0, int capacity, int gtiles, int ngroups, const int32_t* __restrict__ len,
                   const uint64_t* __restrict__ tree_mask, const float* __restrict__ kscale,
                   const float* __restrict__ vscale, float* __restrict__ part_o, float* __restrict__ part_ml,
                   float scale_log2, int* status) {
  constexpr int kStages = Q8 ? 2 : FaLayout<G>::kStages;
  constexpr uint32_t kQ = Q8 ? FaLayoutQ8<G>::kQ : FaLayout<G>::kQ;
  constexpr uint32_t kXchOff = Q8 ? FaLayoutQ8<G>::kXch : FaLayout<G>::kXch;
  constexpr uint32_t kBarOff = Q8 ? FaLayoutQ8<G>::kBar : FaLayout<G>::kBar;
  // TMEM lane quarters holding real rows; in Q8 the warps of the others convert
  constexpr int kLiveQ = (16 * G + 31) / 32 < 4 ? (16 * G + 31) / 32 : 4;
  constexpr int kSoftWarps = Q8 ? 2 * kLiveQ : 8;  // warps that arrive on p_full / xch_full
  constexpr int kConvWarps = 8 - 2 * kLiveQ;
  static_assert(!Q8 || kConvWarps >= 2, "the 8-bit path needs padding quarters for its converter warps");
  // Q8: with only two converter warps (GQA 5) the softmax warps convert each tile's values, else the
  // converter warps convert keys and values
  constexpr bool kSoftV = Q8 && kConvWarps < 4;
  constexpr int kVConv = kSoftV ? kSoftWarps : kConvWarps;  // warps converting the values
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kBarOff);
  float* xch = reinterpret_cast<float*>(sm + kXchOff);  // [2][2][128] row maxima of each half
  uint64_t* kv_full = bar;        // [kStages] a tile's operands ready (bf16: landed; Q8: converted)
  uint64_t* kv_empty = bar + 3;   // [kStages] its products completed
  uint64_t* q_full = bar + 6;
  uint64_t* s_full = bar + 7;     // [2] S_t in TMEM
  uint64_t* p_full = bar + 9;     // [2] P_t in TMEM (one arrival per softmax warp)
  uint64_t* pv_done = bar + 11;   // [2] O += P_t V_t completed
  uint64_t* drain = bar + 13;     // every issued product completed
  uint64_t* xch_full = bar + 14;  // [2] both halves' maxima written (one arrival per softmax warp)
  // Q8: the byte ring's key half and value half land and are released separately
  constexpr int kU8S = FaLayoutQ8<G>::kU8Stages;  // byte stages (3)
  uint64_t* u8_full = bar + 16;   // Q8 [2][3] a tile's codes and scales landed ([kv * 3 + stage], kv 0: keys)
  uint64_t* u8_empty = bar + 22;  // Q8 [2][3] converted (one arrival per warp converting that kind)
  uint64_t* vf_full = bar + 28;   // Q8 the half value tile holds the next tile (kv_full[0]: the key tile)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + (Q8 ? 30 : 26));
  volatile int* abort_f = reinterpret_cast<volatile int*>(tslot + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Set-up that needs nothing from the previous kernel (barriers, TMEM, the
  // descriptors) runs before the wait on it.
  if (tid == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&kv_full[i], Q8 ? kConvWarps : 1);
      mbar_init(&kv_empty[i], 1);
    }
    if (Q8) {
      for (int i = 0; i < 2 * kU8S; ++i) {
        mbar_init(&u8_full[i], 1);
        mbar_init(&u8_empty[i], i < kU8S ? kConvWarps : kVConv);
      }
      mbar_init(vf_full, kVConv);
    }
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kSoftWarps);
      mbar_init(&pv_done[i], 1);
      mbar_init(&xch_full[i], kSoftWarps);
    }
    mbar_init(drain, 1);
    *abort_f = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  pdl_launch();

  // ---- the unit
  const int nrb = (n + 15) >> 4;
  int u = blockIdx.x;
  const int hk = u % nkv;
  u /= nkv;
  const int rb = u % nrb;
  u /= nrb;
  const int b = u % batch;
  const int gi = u / batch;
  const int r_last = min(rb * 16 + 15, n - 1);
  // the unit's key tiles [ta, ta + nt) when the sequence holds P positions before the block
  auto tile_range = [&](int P, int& ta_, int& nt_) {
    const int kmax = min(causal ? P + r_last + 1 : P + n, capacity);
    const int lo_ = window > 0 ? max(0, P - window) : 0;
    ta_ = max(gi * gtiles, lo_ >> 7);
    nt_ = min((gi + 1) * gtiles, (kmax + 127) >> 7) - ta_;
  };
  // Before the wait on the previous kernel (which may still be writing the block's rows of this cache),
  // the producer asks L2 for the unit's first ring stages of keys and values, so that their DRAM
  // latency overlaps the previous kernel's tail.  Every write lands in L2, so no copy requested here
  // is ever read stale; the length read here may be stale, which only misplaces the requests.
  if (warp == 0 && lane == 0) {
    int pta, pnt;
    tile_range(*reinterpret_cast<const volatile int32_t*>(len + b), pta, pnt);
    const long long rowp = row0 + ((long long)b * nkv + hk) * capacity;
    constexpr int kEarly = Q8 ? FaLayoutQ8<G>::kU8Stages : FaLayout<G>::kStages;
    for (int t = 0; t < min(pnt, kEarly); ++t) {
      const int key0 = (int)(rowp + (long long)(pta + t) * 128);
      if constexpr (Q8) {
        tma_prefetch_l2_2d(&tmK, 0, key0);
        tma_prefetch_l2_2d(&tmV, 0, key0);
        bulk_prefetch_l2(kscale + key0, 512);
        bulk_prefetch_l2(vscale + key0, 512);
      } else {
        for (int dh = 0; dh < 2; ++dh) {
          tma_prefetch_l2_2d(&tmK, dh * 64, key0);
          tma_prefetch_l2_2d(&tmV, dh * 64, key0);
        }
      }
    }
  }
  pdl_wait();
  const int P = len[b];
  const int lo = window > 0 ? max(0, P - window) : 0;
  int ta, nt;
  tile_range(P, ta, nt);
  if (nt <= 0) {  // uniform over the CTA: no key of this group is visible
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
    return;
  }
  const int q4w = warp & 3;
  const bool live = q4w * 32 < 16 * G;  // softmax warps: the quarter holds real rows
  const bool conv = Q8 && warp >= 2 && !live;

  // Q8: one byte-to-half conversion job -- kind kv (0 keys, 1 values) of tile t -- shared by `nparts`
  // warps, this one of rank `part`.  The converter warps convert the keys, and the values too unless
  // there are only two of them: then the softmax warps convert a tile's values right after writing
  // its P, while the next scores are computed.
  auto convert = [&](int kv, int t, int part, int nparts) -> bool {
    const int ct = part * 32 + lane, nct = nparts * 32;
    const int ch = ct & 7, row0 = ct >> 3, rstep = nct >> 3;
    // The 8 lanes of a quarter warp convert one row: lanes ch and ch + 4 fill the same swizzled chunk
    // positions of the two 64-entry halves, so the upper four store their second chunk first; each
    // store instruction then writes 8 distinct bank groups per quarter warp.
    const bool swap = ch >= 4;
    const int sw = row0 & 7, d0 = (((ch & 3) * 2) ^ sw) << 4, d1 = (((ch & 3) * 2 + 1) ^ sw) << 4;
    const int da = swap ? d1 : d0, db = swap ? d0 : d1;
    const __half2 off2 = __float2half2_rn(1152.f);
    const int s = t % kU8S;
    const uint8_t* src = sm + s * FaLayoutQ8<G>::kU8Stage;
    uint8_t* dst = sm + FaLayoutQ8<G>::kF;
    const float* scales = reinterpret_cast<const float*>(src + 32768);  // [128 keys | 128 values]
    // the half tile is free once the previous tile's product has read it: the keys once its S
    // exists, the values once its P V is done
    bool ok = mbar_wait(&u8_full[kv * kU8S + s], (uint32_t)(t / kU8S) & 1u, kFaWaitNs);
    if (ok && t >= 1)
      ok = kv == 0 ? mbar_wait(&s_full[(t - 1) & 1], (uint32_t)((t - 1) >> 1) & 1u, kFaWaitNs)
                   : mbar_wait(&pv_done[(t - 1) & 1], (uint32_t)((t - 1) >> 1) & 1u, kFaWaitNs);
    ok = __all_sync(0xffffffffu, ok);
    if (__any_sync(0xffffffffu, !ok || *abort_f)) {
      if (!ok) {
        *abort_f = 1;
        set_status(status, DFLASH_STATUS_TIMEOUT);
      }
      return false;
    }
    // this thread's 16-byte chunks: rows row0 + i * rstep, entries 16 ch .. + 15 (rstep is a multiple
    // of 8, so every row keeps the same swizzle phase)
    const uint8_t* sp = src + kv * 16384 + row0 * 128 + ch * 16;
    uint8_t* dp = dst + kv * kTileBytes + (ch >> 2) * 16384 + row0 * 128;
    const float* scp = scales + kv * 128 + row0;
#pragma unroll 4
    for (int row = row0; row < 128; row += rstep) {
      const uint4 w = *reinterpret_cast<const uint4*>(sp);
      const __half2 sc2 = __half2half2(__float2half_rn(*scp));
      // entries 0..7 of the chunk go to d0, 8..15 to d1; the first store takes the da half
      const uint32_t in[4] = {swap ? w.z : w.x, swap ? w.w : w.y, swap ? w.x : w.z, swap ? w.y : w.w};
      uint32_t o[8];
#pragma unroll
      for (int j2 = 0; j2 < 4; ++j2) {
        const uint32_t lo = __byte_perm(in[j2], 0x64646464u, 0x4140);  // halves 1024 + u of bytes 0, 1
        const uint32_t hi = __byte_perm(in[j2], 0x64646464u, 0x4342);  // bytes 2, 3
        const __half2 a = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&lo), off2), sc2);
        const __half2 b = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&hi), off2), sc2);
        o[2 * j2] = *reinterpret_cast<const uint32_t*>(&a);
        o[2 * j2 + 1] = *reinterpret_cast<const uint32_t*>(&b);
      }
      // half tile: 64-entry half ch >> 2, 16-byte chunks 2 (ch & 3) and + 1, 128-byte swizzle
      *reinterpret_cast<uint4*>(dp + da) = make_uint4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<uint4*>(dp + db) = make_uint4(o[4], o[5], o[6], o[7]);
      sp += rstep * 128;
      dp += rstep * 128;
      scp += rstep;
    }
    fence_proxy_async_smem();  // the tensor cores read the tiles through the async proxy
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(kv == 0 ? &kv_full[0] : vf_full);
      mbar_arrive(&u8_empty[kv * kU8S + s]);
    }
    return true;
  };

  int issued = 0;    // producer: tiles whose copies were issued (Q8: key halves)
  int issued_v = 0;  // Q8: value halves
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int qbox = min(16, batch * n);
      mbar_arrive_expect_tx(q_full, 2 * 128 * G * qbox);
      for (int dh = 0; dh < 2; ++dh)
        tma_load_3d(sm + kQ + dh * 16384, &tmQ, q_full, dh * 64, hk * G, b * n + rb * 16);
      const int rowb = (int)(row0 + ((long long)b * nkv + hk) * capacity);
      if constexpr (Q8) {
        // key halves and value halves in the converters' order: keys of tile t, then values of t - 1
        for (int t = 0; t <= nt && !*abort_f; ++t)
          for (int kv = 0; kv < 2; ++kv) {
            const int tt = t - kv;
            if (tt < 0 || tt >= nt) continue;
            const int s = tt % kU8S, bi = kv * kU8S + s;
            if (tt >= kU8S && !mbar_wait(&u8_empty[bi], (uint32_t)((tt / kU8S) - 1) & 1u, kFaWaitNs)) {
              *abort_f = 1;
              set_status(status, DFLASH_STATUS_TIMEOUT);
              break;
            }
            const int key0 = rowb + (ta + tt) * 128;
            uint8_t* st = sm + s * FaLayoutQ8<G>::kU8Stage;
            mbar_arrive_expect_tx(&u8_full[bi], 16384 + 512);
            tma_load_2d(st + kv * 16384, kv == 0 ? &tmK : &tmV, &u8_full[bi], 0, key0);
            bulk_load(st + 32768 + kv * 512, (kv == 0 ? kscale : vscale) + key0, 512, &u8_full[bi]);
            if (kv == 0)
              issued = tt + 1;
            else
              issued_v = tt + 1;
          }
      } else {
        for (int t = 0; t < nt; ++t) {
          const int s = t % kStages;
          if (t >= kStages && !mbar_wait(&kv_empty[s], (uint32_t)((t / kStages) - 1) & 1u, kFaWaitNs)) {
            *abort_f = 1;
            set_status(status, DFLASH_STATUS_TIMEOUT);
            break;
          }
          if (*abort_f) break;
          const int key0 = rowb + (ta + t) * 128;
          uint8_t* st = sm + s * kStageBytes;
          mbar_arrive_expect_tx(&kv_full[s], kStageBytes);
          for (int dh = 0; dh < 2; ++dh) tma_load_2d(st + dh * 16384, &tmK, &kv_full[s], dh * 64, key0);
          for (int dh = 0; dh < 2; ++dh) tma_load_2d(st + kTileBytes + dh * 16384, &tmV, &kv_full[s], dh * 64, key0);
          issued = t + 1;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ products
    if (lane == 0) {
      const uint32_t idS = Q8 ? idesc_f16_f32(128, 128) : idesc_bf16_f32(128, 128);
      const uint32_t idO = idS | (1u << 16);  // B (values) MN-major
      const uint32_t kOps = Q8 ? FaLayoutQ8<G>::kF : 0u;  // the operand ring (Q8: one key and one value tile)
      constexpr int kOpS = Q8 ? 1 : kStages;
      bool ok = mbar_wait(q_full, 0, kFaWaitNs);
      for (int t = 0; ok && t <= nt; ++t) {
        if (t < nt) {  // S_t = Q K_t^T into S[t & 1], once P_{t-2} (same buffer) has been consumed
          const int s = t % kOpS, sb = t & 1;
          ok = mbar_wait(&kv_full[s], (uint32_t)(t / kOpS) & 1u, kFaWaitNs);
          if (ok && t >= 2) ok = mbar_wait(&pv_done[sb], (uint32_t)((t - 2) >> 1) & 1u, kFaWaitNs);
          if (!ok || *abort_f) break;
          tc_fence_after();
          const uint8_t* kt = sm + kOps + s * kStageBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const int dh = kk >> 2;
            const uint64_t a = smem_desc_sw128(sm + kQ + dh * 16384) + (uint64_t)(((kk & 3) * 32) >> 4);
            const uint64_t bk = smem_desc_sw128(kt + dh * 16384) + (uint64_t)(((kk & 3) * 32) >> 4);
            tc_mma_f16(tmem + sb * 128, a, bk, idS, kk > 0 ? 1u : 0u);
          }
          tc_commit(&s_full[sb]);
        }
        if (t >= 1) {  // O += P_hi V + P_lo V for tile t-1 (P of key half j at columns 64 j: hi, then lo)
          const int w = t - 1, wb = w & 1, s = w % kOpS;
          ok = mbar_wait(&p_full[wb], (uint32_t)(w >> 1) & 1u, kFaWaitNs);
          if (Q8 && ok) ok = mbar_wait(vf_full, (uint32_t)w & 1u, kFaWaitNs);
          if (!ok || *abort_f) break;
          tc_fence_after();
          const uint32_t vt = smem_u32(sm + kOps + s * kStageBytes + kTileBytes);
#pragma unroll
          for (int pass = 0; pass < 2; ++pass)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              tc_mma_f16_tmem_a(tmem + 256, tmem + wb * 128 + (kk >> 2) * 64 + pass * 32 + (kk & 3) * 8,
                                smem_desc_mn(vt + kk * 2048, 16384), idO, (w | pass | kk) != 0 ? 1u : 0u);
          tc_commit(&pv_done[wb]);
          tc_commit(&kv_empty[s]);
        }
      }
      if (!ok) {
        *abort_f = 1;
        set_status(status, DFLASH_STATUS_TIMEOUT);
      }
      tc_commit(drain);  // arrives once every product issued above has completed
    }
    __syncwarp();
  } else if (conv) {
    // ------------------------------------------------------------ Q8: byte tiles -> fp16 operands
    if constexpr (Q8) {
      int cidx = 0;  // this warp's rank among the converter warps
      for (int w = 2; w < warp; ++w) cidx += (w & 3) * 32 >= 16 * G;
      // jobs in deadline order: keys of tile t (needed by its Q K^T) before the values of tile t-1
      // (needed only after tile t-1's softmax)
      for (int t = 0; t <= nt; ++t) {
        if (t < nt && !convert(0, t, cidx, kConvWarps)) break;
        if (!kSoftV && t >= 1 && !convert(1, t - 1, cidx, kConvWarps)) break;
      }

    }
  } else {
    // ------------------------------------------------------------ softmax
    const int q4 = q4w, h = (warp - 2) >> 2;
    int srank = warp - 2;  // this warp's rank among the softmax warps
    if (Q8)
      for (int w = 2; w < warp; ++w) srank -= (w & 3) * 32 >= 16 * G;
    const int r = q4 * 32 + lane;
    const int ri = r / G;
    const int qi = rb * 16 + ri;
    const bool row_ok = r < 16 * G && qi < n;
    const int lim = row_ok ? min(causal ? P + qi + 1 : P + n, capacity) : 0;  // visible keys [lo, lim)
    // tree verification: block key P + i is visible only when bit i is set (the node's ancestors)
    // (only then is n <= 64, so k - P < 64 keeps the shift defined)
    const bool tree = tree_mask != nullptr;
    const uint64_t tm = (tree && row_ok) ? tree_mask[(size_t)b * n + qi] : 0ull;
    const uint32_t lrow = (uint32_t)(q4 * 32) << 16;
    const uint32_t obase = tmem + lrow + 256 + h * 64;  // this half's 64 output columns
    float M = -INFINITY, Lh = 0.f;
    bool ok = true;
    for (int t = 0; ok && t < nt; ++t) {
      const int sb = t & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[sb], (uint32_t)(t >> 1) & 1u, kFaWaitNs));
      if (__any_sync(0xffffffffu, !ok || *abort_f)) break;  // warp-uniform
      tc_fence_after();
      const int k0 = (ta + t) * 128 + h * 64;                // this half's first key
      const uint32_t sbase = tmem + lrow + sb * 128 + h * 64;  // this half's 64 score columns
      uint32_t v[64];
      float lm = -INFINITY;
      // this row's visible keys of the half: [va, vb) (and, in tree mode, the ancestor bits)
      const int va = min(64, max(0, lo - k0)), vb = max(0, min(64, lim - k0));
      // warp-uniform fast path when every real row of the warp sees the whole half (padding rows -- past
      // 16 G or past the block -- are never read, so their values may be anything)
      const bool wfull = __all_sync(0xffffffffu, !row_ok || (!tree && va == 0 && vb == 64));
      // the visible entries as a bit mask (entry e: bit e & 31 of word e >> 5), so the masked loops
      // select instead of branching: keys [va, vb), and in tree mode the context or an ancestor
      uint32_t vw[2];
      if (!wfull) {
        auto range32 = [](int a, int b) -> uint32_t {  // bits [a, b) of a word, 0 <= a, b <= 32
          const uint32_t below_b = b >= 32 ? 0xffffffffu : ((1u << b) - 1u);
          const uint32_t below_a = a >= 32 ? 0xffffffffu : ((1u << a) - 1u);
          return a < b ? (below_b & ~below_a) : 0u;
        };
        vw[0] = range32(min(va, 32), min(vb, 32));
        vw[1] = range32(max(va - 32, 0), max(vb - 32, 0));
        if (tree) {  // entry e is key P + (d + e): context below d + e = 0, else bit d + e of the node's mask
          const int d = k0 - P;
          const uint64_t tv = d >= 64 ? 0ull : d >= 0 ? tm >> d : d > -64 ? (tm << -d) | ((1ull << -d) - 1ull) : ~0ull;
          vw[0] &= (uint32_t)tv;
          vw[1] &= (uint32_t)(tv >> 32);
        }
      }
      auto vis = [&](int e) { return ((vw[e >> 5] >> (e & 31)) & 1u) != 0u; };
      if (live) {  // this half's scores and their maximum over the visible keys
        tmem_ld32(sbase, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(sbase + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_ld_wait();
        if (wfull) {
#pragma unroll
          for (int e = 0; e < 64; ++e) lm = fmaxf(lm, __uint_as_float(v[e]));
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e) lm = fmaxf(lm, vis(e) ? __uint_as_float(v[e]) : -INFINITY);
        }
        xch[(sb * 2 + h) * 128 + r] = lm;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&xch_full[sb]);
      ok = __all_sync(0xffffffffu, mbar_wait(&xch_full[sb], (uint32_t)(t >> 1) & 1u, kFaWaitNs));
      if (__any_sync(0xffffffffu, !ok || *abort_f)) break;
      float Mn = M;
      bool resc = false;
      if (live) {
        const float mraw = fmaxf(lm, xch[(sb * 2 + (1 - h)) * 128 + r]);
        if (mraw != -INFINITY) {
          const float mt = mraw * scale_log2;  // scale > 0: max(s) * scale = max(s * scale)
          if (M == -INFINITY) {
            Mn = mt;
          } else if (mt > M + 8.f) {
            Mn = mt;
            resc = true;
          }
        }
        const float negm = Mn == -INFINITY ? 0.f : -Mn;
        const float sl = scale_log2;
        float lt = 0.f;
        uint32_t hi[32], lo_[32];
        // p of entries 2e, 2e+1 into the row sum and the P hi/lo pair (bf16, or half for Q8)
        auto emit = [&](int e, float p0, float p1) {
          lt += p0;
          lt += p1;
          if constexpr (Q8) {
            const __half2 hh = __floats2half2_rn(p0, p1);
            const float2 hf = __half22float2(hh);
            const __half2 ll = __floats2half2_rn(p0 - hf.x, p1 - hf.y);
            hi[e] = *reinterpret_cast<const uint32_t*>(&hh);
            lo_[e] = *reinterpret_cast<const uint32_t*>(&ll);
          } else {
            pack_bf16_hilo(p0, p1, hi[e], lo_[e]);
          }
        };
        // two separately unrolled loops: the common one has no per-entry test, so the
        // exponentials of different entries overlap freely
        if (wfull) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            emit(e, ex2f(fmaf(__uint_as_float(v[2 * e]), sl, negm)), ex2f(fmaf(__uint_as_float(v[2 * e + 1]), sl, negm)));
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e)  // a hidden entry: 2^-inf = +0
            emit(e, ex2f(vis(2 * e) ? fmaf(__uint_as_float(v[2 * e]), sl, negm) : -INFINITY),
                 ex2f(vis(2 * e + 1) ? fmaf(__uint_as_float(v[2 * e + 1]), sl, negm) : -INFINITY));
        }
        // every score of this half is in registers: P overwrites them (hi at +0..31, lo at +32..63)
        tmem_st16(sbase, *reinterpret_cast<const uint32_t(*)[16]>(&hi[0]));
        tmem_st16(sbase + 16, *reinterpret_cast<const uint32_t(*)[16]>(&hi[16]));
        tmem_st16(sbase + 32, *reinterpret_cast<const uint32_t(*)[16]>(&lo_[0]));
        tmem_st16(sbase + 48, *reinterpret_cast<const uint32_t(*)[16]>(&lo_[16]));
        const float f = resc ? ex2f(M - Mn) : 1.f;
        Lh = fmaf(Lh, f, lt);
        // a raised reference max rescales O once the products of the earlier tiles are done
        if (__any_sync(0xffffffffu, resc)) {
          ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[(t - 1) & 1], (uint32_t)((t - 1) >> 1) & 1u, kFaWaitNs));
          if (ok) {
            tc_fence_after();
            uint32_t o[64];
            tmem_ld32(obase, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
            tmem_ld32(obase + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 64; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_st16(obase + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(&o[c * 16]));
          }
        }
        tmem_st_wait();
        M = Mn;
      }
      if (__any_sync(0xffffffffu, !ok)) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sb]);
      if constexpr (kSoftV) {  // this tile's values, while the next tile's scores are computed
        if (!convert(1, t, srank, kSoftWarps)) {
          ok = false;
          break;
        }
      }
    }
    // the last product of the unit completes before O is read
    if (ok && !*abort_f)
      ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[(nt - 1) & 1], (uint32_t)((nt - 1) >> 1) & 1u, kFaWaitNs));
    if (!ok) {
      *abort_f = 1;
      set_status(status, DFLASH_STATUS_TIMEOUT);
    }
    // ---- the unit's partial, staged through the (dead) ring so that each
    // row leaves as one contiguous 512-byte store: row r at r * 512, its
    // 16-byte chunks XOR-swizzled by (r & 7).  Row sums of the two halves at
    // 64 KB, row maxima after them.  (Q8: every byte tile has been converted
    // once the last scores exist, so the 8-bit ring is dead here too.)
    float* stg = reinterpret_cast<float*>(sm);
    float* stg_l = stg + 128 * 128;
    float* stg_m = stg_l + 256;
    __syncthreads();
    const bool good = !*abort_f;
    if (good && live) {
      tc_fence_after();
      uint32_t o[64];
      tmem_ld32(obase, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
      tmem_ld32(obase + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int ch = h * 16 + c;
        *reinterpret_cast<uint4*>(stg + r * 128 + ((ch ^ (r & 7)) << 2)) =
            make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
      }
      stg_l[2 * r + h] = Lh;
      if (h == 0) stg_m[r] = M;
    }
    fence_proxy_async_smem();  // the staged rows leave through the bulk-copy engine
    __syncthreads();
    if (good) {
      const int rows_live = min(16 * G, 128);
      // lane l of this warp sends row srank + l kSoftWarps: its 512 bytes as they are staged (16-byte
      // chunks XOR-swizzled by the row's index in the unit, which the combine undoes) by one bulk copy,
      // its maximum and sum by a plain store
      const int rr = srank + lane * kSoftWarps;
      const int ir = rr / G, hr = rr - ir * G, qr = rb * 16 + ir;
      const bool mine = rr < rows_live && qr < n;
      if (mine) {
        const size_t prow = ((size_t)(b * n + qr) * nq + hk * G + hr) * ngroups + gi;
        bulk_store(part_o + prow * 128, stg + rr * 128, 512);
        bulk_store_commit();
        *reinterpret_cast<float2*>(part_ml + prow * 2) = make_float2(stg_m[rr], stg_l[2 * rr] + stg_l[2 * rr + 1]);
        bulk_store_wait();  // the copy has read the staged row and written it before the ring is released
      }
    }
  }
  if (warp < 2 || conv) {  // match the softmax warps' two block-wide barriers
    __syncthreads();
    __syncthreads();
  }
  // ---- teardown: copies and products still in flight complete before the
  // ring and TMEM are released
  if (warp == 0 && lane == 0 && *abort_f) {
    if (Q8) {  // the last byte tiles of each kind that were issued
      for (int kv = 0; kv < 2; ++kv) {
        const int last = kv == 0 ? issued : issued_v;
        for (int tt = last > kU8S ? last - kU8S : 0; tt < last; ++tt)
          mbar_wait(&u8_full[kv * kU8S + tt % kU8S], (uint32_t)(tt / kU8S) & 1u, kFaWaitNs / 4);
      }
    } else {
      const int first = issued > kStages ? issued - kStages : 0;
      for (int t = first; t < issued; ++t)
        mbar_wait(&kv_full[t % kStages], (uint32_t)(t / kStages) & 1u, kFaWaitNs / 4);
    }
  }
  if (warp == 1 && lane == 0) mbar_wait(drain, 0, kFaWaitNs / 4);
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

cudaError_t attention_fa(int G, const KvMaps& maps, const CUtensorMap& qmap, int batch, int n, int nq, int nkv,
                         int causal, int window, int capacity, int gtiles, const int32_t* len, const uint64_t* tree_mask,
                         const AttnScratch& sc, float scale_log2, int* status, cudaStream_t s) {
  if (gtiles < 2 || batch > kMaxRows) return cudaErrorInvalidValue;
  const int ngroups = (capacity + gtiles * 128 - 1) / (gtiles * 128);
  if (ngroups > sc.nchunk) return cudaErrorInvalidValue;  // partial slots per (row, head)
  const long long units = (long long)ngroups * nkv * batch * ((n + 15) / 16);
  if (units <= 0) return cudaSuccess;
  if (units > INT32_MAX) return cudaErrorInvalidValue;
  if (maps.q8 && (G > 5 || !maps.ks || !maps.vs)) return cudaErrorInvalidValue;
#define DFL_FA_CASE(GG, QQ, LY)                                                                                  \
  {                                                                                                              \
    static bool set = false;                                                                                     \
    if (!set) {                                                                                                  \
      DFL_RET(cudaFuncSetAttribute(attn_fa_kernel<GG, QQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,          \
                                   LY<GG>::kSmem));                                                              \
      set = true;                                                                                                \
    }                                                                                                            \
    DFL_RET(launch_pdl(attn_fa_kernel<GG, QQ>, dim3((unsigned)units), dim3(kFaThreads), LY<GG>::kSmem, s, maps.k, \
                       maps.v, qmap, batch, n, nq, nkv, causal, window, maps.row0, capacity, gtiles, sc.nchunk,   \
                       len, tree_mask, maps.ks, maps.vs, sc.o, sc.ml, scale_log2, status));                       \
    return cudaSuccess;                                                                                          \
  }
  if (maps.q8) {
    switch (G) {
      case 1: DFL_FA_CASE(1, true, FaLayoutQ8)
      case 2: DFL_FA_CASE(2, true, FaLayoutQ8)
      case 4: DFL_FA_CASE(4, true, FaLayoutQ8)
      case 5: DFL_FA_CASE(5, true, FaLayoutQ8)
      default: return cudaErrorInvalidValue;
    }
  }
  switch (G) {
    case 1: DFL_FA_CASE(1, false, FaLayout)
    case 2: DFL_FA_CASE(2, false, FaLayout)
    case 4: DFL_FA_CASE(4, false, FaLayout)
    case 5: DFL_FA_CASE(5, false, FaLayout)
    case 8: DFL_FA_CASE(8, false, FaLayout)
    default: return cudaErrorInvalidValue;
  }
#undef DFL_FA_CASE
}

}  // namespace dfl
