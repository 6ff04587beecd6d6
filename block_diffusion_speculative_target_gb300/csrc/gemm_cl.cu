// Weight-streaming GEMM on the tcgen05 tensor cores with cluster split-K.
//
//   y[n][m] = sum_k x[n][k] * w[m][k]        w: [M][K] bf16, x: [rows][K] bf16
//
// Swap-AB: a 128-row weight tile is the MMA's A operand, the 1..128 tokens
// the B operand (rows past `rows` are zero-filled by TMA), the fp32
// accumulator lives in TMEM.  Decode-sized products have few 128-row tiles,
// so K is split S ways (S depends only on M, K and the SM count) and the S
// CTAs that share a tile form one thread-block cluster.  Each CTA streams its
// K-slice of weights through a TMA ring with an evict-first L2 policy; at the
// end it parks its partial tile in its own shared memory (the drained ring),
// the cluster synchronises once, and CTA r reduces rows r, r+S, ... by reading
// the S partials over distributed shared memory in split order.  The result
// is deterministic and independent of the token count; no partial sum goes
// through global memory.
//
// Roles (128 threads): warp 0 lane 0 issues TMA (weights first: they do not
// depend on the previous kernel), warp 1 lane 0 issues MMAs, warp 2 owns TMEM,
// all four warps run the epilogue (warp w reads TMEM lanes 32w.., i.e. output
// features m0 + 32w + lane).
//
// Epilogues: f32 store, f32 residual add, bf16 store, SwiGLU on interleaved
// gate/up rows, and QKV / drafter-KV with rotate-half RoPE and the KV-cache
// write at each row's position.
//
// RMSNorm across a product boundary: a residual-add epilogue can hand the next
// product its operand bf16(x * gain) and each row's sums of x^2 over 32-column
// slices; that product's idle warps turn the slices into the row's
// 1 / rms during the main loop, and its epilogue scales the row's results by
// it.  No separate normalisation kernel runs between the two products.
#include <string.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dfl {

constexpr uint64_t kGemmWaitNs = 500000000ull;  // 500 ms per wait

// Limit of the main-loop waits (ring slots, accumulator); the drain after a
// time-out always waits the full kGemmWaitNs / 4 so that copies and products
// in flight complete before shared memory and TMEM are released.  Lowered only
// by dflash_debug_set_wait_limit (failure-path tests).
static std::atomic<unsigned long long> g_wait_ns{kGemmWaitNs};
void set_gemm_wait_ns(long long ns) { g_wait_ns.store(ns < 0 ? kGemmWaitNs : (unsigned long long)ns); }

template <int BN, int STAGES>
struct ClCfg {
  static constexpr int BM = 128, BK = 64;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = BN < 32 ? 32 : BN;
  static constexpr int RED_BYTES = BN * BM * 4;  // partial tile, aliases the ring
  static constexpr int RING = STAGES * STAGE_BYTES;
  static constexpr int TAIL = 256;   // barriers, TMEM slot, flags
  static constexpr int PRE = 2048;   // epilogue operands prefetched during the main loop
  static constexpr int RS = kMaxRows * 4;  // rows' 1 / rms of a fused RMSNorm
  static constexpr int SMEM = (RING > RED_BYTES ? RING : RED_BYTES) + 1024 + TAIL + PRE + RS;
  // a split CTA's summed rows (at most BN / 2 of them) in the dead ring past the partial tile
  static_assert(RED_BYTES + BN / 2 * BM * 4 <= RING, "the summed rows fit in the dead ring");
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The two halves of cluster_sync, for work that may run between them.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_dsmem(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// Sum of the SS split partials of one element (and of its RoPE partner) in
// split order, every load issued before the first add.
__device__ __forceinline__ float4 ld_dsmem4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Four consecutive columns of one row summed over the SS split partials in
// split order, every load issued before the first add (16-byte DSMEM loads:
// a remote request costs about the same whatever its width).
template <int SS>
__device__ __forceinline__ float4 sum_splits4(uint32_t red_local, uint32_t off) {
  float4 p[SS];
#pragma unroll
  for (int cc = 0; cc < SS; ++cc) p[cc] = ld_dsmem4(dsmem_addr(red_local, (uint32_t)cc) + off);
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int cc = 0; cc < SS; ++cc) {
    a.x += p[cc].x;
    a.y += p[cc].y;
    a.z += p[cc].z;
    a.w += p[cc].w;
  }
  return a;
}

// This CTA's rows n = r + j S of the split tile, warp w taking j = w, w + 4,
// ...: lane l sums columns 4l .. 4l + 3 of each over the SS partials (split
// order) and hands them to fn(j, n, sums).  The next row's loads are issued
// before fn runs on the current one, so a warp with several rows keeps one
// row's remote requests in flight behind its epilogue.
template <int SS, int BM, typename F>
__device__ __forceinline__ void split_rows4(uint32_t red_local, int r, int J, int warp, int lane, F&& fn) {
  float4 p[SS];
  auto issue = [&](int j) {
    const uint32_t off = (uint32_t)(((r + j * SS) * BM + lane * 4) * 4);
#pragma unroll
    for (int cc = 0; cc < SS; ++cc) p[cc] = ld_dsmem4(dsmem_addr(red_local, (uint32_t)cc) + off);
  };
  if (warp < J) issue(warp);
  for (int j = warp; j < J; j += 4) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int cc = 0; cc < SS; ++cc) {
      a.x += p[cc].x;
      a.y += p[cc].y;
      a.z += p[cc].z;
      a.w += p[cc].w;
    }
    if (j + 4 < J) issue(j + 4);
    fn(j, r + j * SS, a);
  }
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// The new residual x of output (n, m): stored, with its captured bf16 copies.
__device__ __forceinline__ void resid_store(const GemmEpi& e, int n, int m, float x) {
  reinterpret_cast<float*>(e.out)[(size_t)n * e.ldo + m] = x;
  if (e.cap_mask)
    for (int s = 0; s < 5; ++s)
      if (e.cap_mask & (1 << s))
        reinterpret_cast<bf16*>(e.hcap)[(size_t)n * 5 * e.cap_H + (size_t)s * e.cap_H + m] = __float2bfloat16_rn(x);
}

// The next product's RMSNorm handed over (GE_RESID with norm_out): bf16(x *
// gain) and the sum of x^2 over the warp's 32 consecutive columns.  Every lane
// of the warp calls it for the same row; `ok` is false after a time-out.
__device__ __forceinline__ void norm_handover(const GemmEpi& e, int n, int m, float x, bool ok, int lane) {
  if (ok)
    reinterpret_cast<bf16*>(e.norm_out)[(size_t)n * e.ldo + m] =
        __float2bfloat16_rn(x * __bfloat162float(reinterpret_cast<const bf16*>(e.norm_gain)[m]));
  float t = x * x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  if (ok && lane == 0) e.norm_ssq[(size_t)n * (e.ldo >> 5) + (m >> 5)] = t;
}

// RoPE / KV-cache epilogue of output (n, m) with the row's position and the
// cos/sin of this column's frequency at that position already at hand.
__device__ __forceinline__ void gemm_epi_rope(const GemmEpi& e, int n, int m, float v, float partner, int pos,
                                              float2 cs, int* status) {
  const int t = m >> 7, ml = m & 127;
  int kind, h, layer = 0;  // kind: 0 q, 1 k, 2 v
  if (e.kind == GE_QKV) {
    kind = t < e.nq ? 0 : (t < e.nq + e.nkv ? 1 : 2);
    h = kind == 0 ? t : (kind == 1 ? t - e.nq : t - e.nq - e.nkv);
  } else {
    layer = t / (2 * e.nkv);
    const int rem = t % (2 * e.nkv);
    kind = rem < e.nkv ? 1 : 2;
    h = rem % e.nkv;
  }
  const float r = kind == 2 ? v : (ml < 64 ? v * cs.x - partner * cs.y : v * cs.x + partner * cs.y);
  if (kind == 0) {
    reinterpret_cast<bf16*>(e.out)[((size_t)n * e.nq + h) * 128 + ml] = __float2bfloat16_rn(r);
    return;
  }
  if (pos >= e.capacity) {
    set_status(status, DFLASH_STATUS_CAPACITY);
    return;
  }
  const int b = n / e.rows_per_seq;
  bf16* dst = reinterpret_cast<bf16*>(kind == 1 ? e.kc : e.vc);
  dst[(size_t)layer * e.layer_stride + (size_t)b * e.seq_stride + (size_t)h * e.head_stride + (size_t)pos * 128 + ml] =
      __float2bfloat16_rn(r);
}

// GE_QKV into an 8-bit cache, output (n, m) with its RoPE partner and the
// row's position and cos/sin at hand: the query leaves as fp16; a key or
// value row -- the CTA's 128 columns are one head -- is quantised with
// s = max|x| / 127 over the CTA's 128 threads (two rounds of named barrier 1
// through `red`) and q = round-half-even(x / s), stored as q + 128 with s.
// Every thread of the CTA calls it for the same row (the kind is uniform over
// the CTA); `ok` is false after a time-out.
__device__ __forceinline__ void qkv_q8_out(const GemmEpi& e, int n, int m, float v, float partner, int pos,
                                           float2 cs, bool ok, float* red, int* status) {
  const int t = m >> 7, ml = m & 127;
  const int kind = t < e.nq ? 0 : (t < e.nq + e.nkv ? 1 : 2);  // 0 q, 1 k, 2 v
  const int h = kind == 0 ? t : (kind == 1 ? t - e.nq : t - e.nq - e.nkv);
  const float r = kind == 2 ? v : (ml < 64 ? v * cs.x - partner * cs.y : v * cs.x + partner * cs.y);
  if (kind == 0) {
    if (ok) reinterpret_cast<__half*>(e.out)[((size_t)n * e.nq + h) * 128 + ml] = __float2half_rn(r);
    return;
  }
  float a = fabsf(r);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  asm volatile("bar.sync 1, 128;" ::: "memory");
  const float amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  asm volatile("bar.sync 1, 128;" ::: "memory");  // `red` is rewritten for the next row
  const float sc = __fdiv_rn(amax, 127.0f);
  const float q = sc > 0.f ? fminf(fmaxf(rintf(__fdiv_rn(r, sc)), -127.f), 127.f) : 0.f;
  if (!ok || pos < 0) return;
  if (pos >= e.capacity) {
    set_status(status, DFLASH_STATUS_CAPACITY);
    return;
  }
  const int b = n / e.rows_per_seq;
  const size_t row = (size_t)b * (e.seq_stride >> 7) + (size_t)h * (e.head_stride >> 7) + (size_t)pos;
  reinterpret_cast<uint8_t*>(kind == 1 ? e.kc : e.vc)[row * 128 + ml] = (uint8_t)((int)q + 128);
  if (ml == 0) (kind == 1 ? e.ks : e.vs)[row] = sc;
}

// ---- the split path's epilogue, four columns per lane
// A warp applies the epilogue to one row of the tile: lane l holds columns
// m = m0 + 4l .. + 3 (the four sums it reduced), its RoPE partners (column
// ^ 64 within the head) sit in lane l ^ 16, and every store moves 4, 8 or 16
// bytes.  The arithmetic per element is the per-column epilogue's.

// Every pointer the epilogue touches is 16-byte aligned and every row stride a
// multiple of 4 elements: then the four-column stores stay aligned.
__device__ __forceinline__ bool epi_vec4_ok(const GemmEpi& e) {
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  bool ok = al(e.out) && (e.ldo & 3) == 0 && al(e.hcap) && (e.cap_H & 3) == 0 && al(e.norm_gain) && al(e.norm_out) &&
            al(e.rope) && al(e.kc) && al(e.vc);
  if (e.kind == GE_QKV || e.kind == GE_INJECT)
    ok = ok && (e.layer_stride & 3) == 0 && (e.seq_stride & 3) == 0 && (e.head_stride & 3) == 0;
  return ok;
}
__device__ __forceinline__ void st_bf16x4(void* p, float a, float b, float c, float d) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  *reinterpret_cast<uint2*>(p) = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}
__device__ __forceinline__ void st_halfx4(void* p, float a, float b, float c, float d) {
  const __half2 lo = __floats2half2_rn(a, b), hi = __floats2half2_rn(c, d);
  *reinterpret_cast<uint2*>(p) = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}

// Row n, columns m .. m + 3 with their values v (row scale applied).  j: the
// row's index among this CTA's rows; with `pf`, the residual's old values and
// the row's position and cos/sin were fetched during the main loop.  Every
// lane of the warp calls it for the same row; `ok` is false after a time-out.
__device__ __forceinline__ void gemm_epi4(const GemmEpi& e, int n, int m, float4 v, bool ok, int lane, bool pf, int j,
                                          const float* pre_x, const float2* pre_cs, const int* pre_pos, int* status) {
  const float vv[4] = {v.x, v.y, v.z, v.w};
  switch (e.kind) {
    case GE_F32:
      if (ok) *reinterpret_cast<float4*>(reinterpret_cast<float*>(e.out) + (size_t)n * e.ldo + m) = v;
      return;
    case GE_STORE:
      if (ok) st_bf16x4(reinterpret_cast<bf16*>(e.out) + (size_t)n * e.ldo + m, v.x, v.y, v.z, v.w);
      return;
    case GE_SWIGLU:
      if (ok) {
        const __nv_bfloat162 o = __floats2bfloat162_rn(silu_f(v.x) * v.y, silu_f(v.z) * v.w);
        *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<bf16*>(e.out) + (size_t)n * e.ldo + (m >> 1)) = o;
      }
      return;
    case GE_RESID: {
      float* xo = reinterpret_cast<float*>(e.out) + (size_t)n * e.ldo + m;
      float4 x;
      if (pf) {
        const float* px = pre_x + j * 128 + (m & 127);
        x = make_float4(px[0] + v.x, px[1] + v.y, px[2] + v.z, px[3] + v.w);
      } else {
        const float4 o = *reinterpret_cast<const float4*>(xo);
        x = make_float4(o.x + v.x, o.y + v.y, o.z + v.z, o.w + v.w);
      }
      if (ok) {
        *reinterpret_cast<float4*>(xo) = x;
        if (e.cap_mask)
          for (int s = 0; s < 5; ++s)
            if (e.cap_mask & (1 << s))
              st_bf16x4(reinterpret_cast<bf16*>(e.hcap) + (size_t)n * 5 * e.cap_H + (size_t)s * e.cap_H + m, x.x, x.y,
                        x.z, x.w);
      }
      if (e.norm_out) {  // the next product's operand bf16(x * g) and the sums of x^2 over 32 columns (8 lanes)
        const uint2 gw = *reinterpret_cast<const uint2*>(reinterpret_cast<const bf16*>(e.norm_gain) + m);
        const float2 g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw.x));
        const float2 g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw.y));
        if (ok)
          st_bf16x4(reinterpret_cast<bf16*>(e.norm_out) + (size_t)n * e.ldo + m, x.x * g01.x, x.y * g01.y,
                    x.z * g23.x, x.w * g23.y);
        float t = x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (ok && (lane & 7) == 0) e.norm_ssq[(size_t)n * (e.ldo >> 5) + (m >> 5)] = t;
      }
      return;
    }
    case GE_QKV:
    case GE_INJECT:
      break;
    default:
      return;
  }
  // GE_QKV / GE_INJECT: the head's 128 columns are this row's 32 lanes
  float pp[4];
  pp[0] = __shfl_xor_sync(0xffffffffu, v.x, 16);
  pp[1] = __shfl_xor_sync(0xffffffffu, v.y, 16);
  pp[2] = __shfl_xor_sync(0xffffffffu, v.z, 16);
  pp[3] = __shfl_xor_sync(0xffffffffu, v.w, 16);
  const int t = m >> 7, ml = m & 127;
  int kind, h, layer = 0;  // kind: 0 q, 1 k, 2 v
  if (e.kind == GE_QKV) {
    kind = t < e.nq ? 0 : (t < e.nq + e.nkv ? 1 : 2);
    h = kind == 0 ? t : (kind == 1 ? t - e.nq : t - e.nq - e.nkv);
  } else {
    layer = t / (2 * e.nkv);
    const int rem = t % (2 * e.nkv);
    kind = rem < e.nkv ? 1 : 2;
    h = rem % e.nkv;
  }
  const int b = n / e.rows_per_seq, jj = n % e.rows_per_seq;
  int pos;
  float2 cs[4];
  if (pf) {
    pos = pre_pos[j];
#pragma unroll
    for (int i = 0; i < 4; ++i) cs[i] = pre_cs[j * 64 + ((ml + i) & 63)];
  } else {
    const bool skip = e.kind == GE_INJECT && jj >= e.n_pend[b];
    pos = skip ? -1 : e.len[b] + jj;
    const int rpos = e.rope_off ? e.len[b] + e.rope_off[n] : e.len[b] + jj;  // RoPE position (a tree node's depth)
    if (rpos >= 0 && rpos < e.capacity) {
      const float4* c = reinterpret_cast<const float4*>(e.rope + (size_t)rpos * 64 + (ml & 63));
      const float4 c0 = c[0], c1 = c[1];
      cs[0] = make_float2(c0.x, c0.y);
      cs[1] = make_float2(c0.z, c0.w);
      cs[2] = make_float2(c1.x, c1.y);
      cs[3] = make_float2(c1.z, c1.w);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) cs[i] = make_float2(1.f, 0.f);
    }
  }
  float rr[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    rr[i] = kind == 2 ? vv[i] : (ml < 64 ? vv[i] * cs[i].x - pp[i] * cs[i].y : vv[i] * cs[i].x + pp[i] * cs[i].y);
  if (e.kv_q8) {  // GE_QKV into an 8-bit cache: s = max|x| / 127 over the row's 128 columns (this warp)
    if (kind == 0) {
      if (ok) st_halfx4(reinterpret_cast<__half*>(e.out) + ((size_t)n * e.nq + h) * 128 + ml, rr[0], rr[1], rr[2], rr[3]);
      return;
    }
    float a = fmaxf(fmaxf(fabsf(rr[0]), fabsf(rr[1])), fmaxf(fabsf(rr[2]), fabsf(rr[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const float sc = __fdiv_rn(a, 127.0f);
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float q = sc > 0.f ? fminf(fmaxf(rintf(__fdiv_rn(rr[i], sc)), -127.f), 127.f) : 0.f;
      word |= (uint32_t)((int)q + 128) << (8 * i);
    }
    if (!ok || pos < 0) return;
    if (pos >= e.capacity) {
      set_status(status, DFLASH_STATUS_CAPACITY);
      return;
    }
    const size_t row = (size_t)b * (e.seq_stride >> 7) + (size_t)h * (e.head_stride >> 7) + (size_t)pos;
    *reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(kind == 1 ? e.kc : e.vc) + row * 128 + ml) = word;
    if (ml == 0) (kind == 1 ? e.ks : e.vs)[row] = sc;
    return;
  }
  if (!ok || pos < 0) return;
  if (kind == 0) {
    st_bf16x4(reinterpret_cast<bf16*>(e.out) + ((size_t)n * e.nq + h) * 128 + ml, rr[0], rr[1], rr[2], rr[3]);
    return;
  }
  if (pos >= e.capacity) {
    set_status(status, DFLASH_STATUS_CAPACITY);
    return;
  }
  bf16* dst = reinterpret_cast<bf16*>(kind == 1 ? e.kc : e.vc);
  st_bf16x4(dst + (size_t)layer * e.layer_stride + (size_t)b * e.seq_stride + (size_t)h * e.head_stride + (size_t)pos * 128 +
                ml,
            rr[0], rr[1], rr[2], rr[3]);
}

// Final value y of output (n, m): apply the epilogue.  `partner` is y[n][m^1]
// (SwiGLU) or y[n][m^64] within the head (RoPE).
__device__ __forceinline__ void gemm_epi(const GemmEpi& e, int n, int m, float v, float partner, int* status) {
  switch (e.kind) {
    case GE_F32:
      reinterpret_cast<float*>(e.out)[(size_t)n * e.ldo + m] = v;
      break;
    case GE_RESID:
      resid_store(e, n, m, reinterpret_cast<const float*>(e.out)[(size_t)n * e.ldo + m] + v);
      break;
    case GE_STORE:
      reinterpret_cast<bf16*>(e.out)[(size_t)n * e.ldo + m] = __float2bfloat16_rn(v);
      break;
    case GE_SWIGLU:
      if ((m & 1) == 0)
        reinterpret_cast<bf16*>(e.out)[(size_t)n * e.ldo + (m >> 1)] = __float2bfloat16_rn(silu_f(v) * partner);
      break;
    case GE_QKV:
    case GE_INJECT: {
      const int t = m >> 7, ml = m & 127;
      int kind, h, layer = 0;  // kind: 0 q, 1 k, 2 v
      if (e.kind == GE_QKV) {
        kind = t < e.nq ? 0 : (t < e.nq + e.nkv ? 1 : 2);
        h = kind == 0 ? t : (kind == 1 ? t - e.nq : t - e.nq - e.nkv);
      } else {
        layer = t / (2 * e.nkv);
        const int rem = t % (2 * e.nkv);
        kind = rem < e.nkv ? 1 : 2;
        h = rem % e.nkv;
      }
      const int b = n / e.rows_per_seq, jj = n % e.rows_per_seq;
      if (e.kind == GE_INJECT && jj >= e.n_pend[b]) break;
      const int pos = e.len[b] + jj;
      const int rpos = e.rope_off ? e.len[b] + e.rope_off[n] : pos;  // RoPE position (a tree node's depth)
      float r = v;
      if (kind != 2) {
        const float2 cs = (rpos >= 0 && rpos < e.capacity) ? e.rope[(size_t)rpos * 64 + (ml & 63)] : make_float2(1.f, 0.f);
        r = ml < 64 ? v * cs.x - partner * cs.y : v * cs.x + partner * cs.y;
      }
      if (kind == 0) {
        reinterpret_cast<bf16*>(e.out)[((size_t)n * e.nq + h) * 128 + ml] = __float2bfloat16_rn(r);
        break;
      }
      if (pos >= e.capacity) {
        set_status(status, DFLASH_STATUS_CAPACITY);
        break;
      }
      bf16* dst = reinterpret_cast<bf16*>(kind == 1 ? e.kc : e.vc);
      dst[(size_t)layer * e.layer_stride + (size_t)b * e.seq_stride + (size_t)h * e.head_stride + (size_t)pos * 128 +
          ml] = __float2bfloat16_rn(r);
      break;
    }
  }
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(128)
    gemm_cl_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const GemmEpi epi,
                   const int rows, const int K, const int S, int* status, const uint64_t wait_ns) {
  using C = ClCfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * C::A_BYTES;
  float* red = reinterpret_cast<float*>(smem);  // [BN][128] partial tile after the main loop
  uint8_t* tail = smem + (C::RING > C::RED_BYTES ? C::RING : C::RED_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(tail);
  uint64_t* empty = full + STAGES;
  uint64_t* accb = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [0] abort
  // Prefetched epilogue operands of this CTA's rows (r, r + S, ...; at most
  // 4): old residual values [row][128], or RoPE cos/sin [row][64] and the
  // row's position (-1: row skipped).
  uint8_t* pre = tail + C::TAIL;
  float* pre_x = reinterpret_cast<float*>(pre);
  float2* pre_cs = reinterpret_cast<float2*>(pre);
  int* pre_pos = reinterpret_cast<int*>(tail + 192);  // [4], after the barriers and flags
  float* rsc = reinterpret_cast<float*>(tail + C::TAIL + C::PRE);  // [rows] 1 / rms of a fused RMSNorm
  float* red_q8 = reinterpret_cast<float*>(tail + 128);              // [4] row maxima of an 8-bit cache write

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = (int)cluster_rank();  // split index
  const int tile = blockIdx.y;
  const int KB = K / C::BK;
  const int kb0 = (int)((long long)r * KB / S), kb1 = (int)((long long)(r + 1) * KB / S);
  const int nkb = kb1 - kb0;
  const int m0 = tile * C::BM;
  const bool rope = epi.kind == GE_QKV || epi.kind == GE_INJECT;
  // prefetch the epilogue operands when this CTA owns at most 4 rows of a split tile
  const bool pf = S > 1 && (rows + S - 1) / S <= 4 && (epi.kind == GE_RESID || rope);

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(accb, 1);
    flags[0] = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch();

  int issued = 0;
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const int pre = nkb < STAGES ? nkb : STAGES;
      for (int i = 0; i < pre; ++i) {  // weights first: independent of the previous kernel
        mbar_arrive_expect_tx(&full[i], C::STAGE_BYTES);
        tma_load_2d_hint(sA + i * C::A_BYTES, &tmW, &full[i], (kb0 + i) * C::BK, m0, pol);
      }
      pdl_wait();
      for (int i = 0; i < pre; ++i) tma_load_2d(sB + i * C::B_BYTES, &tmX, &full[i], (kb0 + i) * C::BK, 0);
      issued = pre;
      for (int kb = pre; kb < nkb; ++kb) {
        const int s = kb % STAGES;
        if (!mbar_wait(&empty[s], (uint32_t)((kb / STAGES) - 1) & 1u, wait_ns) || flags[0]) {
          flags[0] = 1;
          set_status(status, DFLASH_STATUS_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
        tma_load_2d_hint(sA + s * C::A_BYTES, &tmW, &full[s], (kb0 + kb) * C::BK, m0, pol);
        tma_load_2d(sB + s * C::B_BYTES, &tmX, &full[s], (kb0 + kb) * C::BK, 0);
        issued = kb + 1;
      }
    }
    __syncwarp();
  } else if (warp >= 2) {
    // Idle during the main loop: fetch what the epilogue will need for this
    // CTA's rows, so no row waits on global memory there.
    const int gt = threadIdx.x - 64;
    if (pf || epi.in_ssq) pdl_wait();
    for (int j = 0; pf && j * S + r < rows; ++j) {
      const int n = r + j * S;
      if (epi.kind == GE_RESID) {
        const float2 v = *reinterpret_cast<const float2*>(reinterpret_cast<const float*>(epi.out) +
                                                          (size_t)n * epi.ldo + m0 + 2 * gt);
        pre_x[j * 128 + 2 * gt] = v.x;
        pre_x[j * 128 + 2 * gt + 1] = v.y;
      } else {  // GE_QKV / GE_INJECT
        const int b = n / epi.rows_per_seq, jj = n % epi.rows_per_seq;
        const bool skip = epi.kind == GE_INJECT && jj >= epi.n_pend[b];
        const int pos = epi.len[b] + jj;
        const int rpos = epi.rope_off ? epi.len[b] + epi.rope_off[n] : pos;
        if (gt == 0) pre_pos[j] = skip ? -1 : pos;
        pre_cs[j * 64 + gt] =
            (rpos >= 0 && rpos < epi.capacity) ? epi.rope[(size_t)rpos * 64 + gt] : make_float2(1.f, 0.f);
      }
    }
    if (epi.in_ssq) {
      // a fused RMSNorm: each of this CTA's rows' 1 / rms from its 32-column sums of squares, added in
      // column order per lane and then over a fixed butterfly (the same value in every CTA)
      const int nw = epi.in_cols >> 5;
      for (int n = r + (warp - 2) * S; n < rows; n += 2 * S) {
        const float* sp = epi.in_ssq + (size_t)n * nw;
        float t = 0.f;
#pragma unroll 4
        for (int c = lane; c < nw; c += 32) t += sp[c];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) rsc[n] = 1.0f / sqrtf(t / (float)epi.in_cols + epi.in_eps);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(C::BM, BN);
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % STAGES;
        if (!mbar_wait(&full[s], (uint32_t)(kb / STAGES) & 1u, wait_ns)) {
          flags[0] = 1;
          set_status(status, DFLASH_STATUS_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint64_t da = smem_desc_sw128(sA + s * C::A_BYTES);
        const uint64_t db = smem_desc_sw128(sB + s * C::B_BYTES);
#pragma unroll
        for (int k = 0; k < C::BK / 16; ++k) tc_mma_f16(tmem, da + 2 * k, db + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
        tc_commit(&empty[s]);
      }
      tc_commit(accb);
    }
    __syncwarp();
  }

  // ---------------------------------------------------------------- epilogue
  if (threadIdx.x == 0 && !mbar_wait(accb, 0, wait_ns)) {
    flags[0] = 1;
    set_status(status, DFLASH_STATUS_TIMEOUT);
  }
  __syncthreads();
  // Drain: after a time-out, wait (bounded) for the products and the loads
  // still in flight before the ring and TMEM are reused or released.
  if (flags[0] && warp == 0 && lane == 0) {
    mbar_wait(accb, 0, kGemmWaitNs / 4);
    const int first = issued > STAGES ? issued - STAGES : 0;
    for (int i = first; i < issued; ++i) mbar_wait(&full[i % STAGES], (uint32_t)(i / STAGES) & 1u, kGemmWaitNs / 4);
  }
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  const int ml = warp * 32 + lane;
  const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
  if (S == 1 && !rope) {
    // Unsplit tile: the accumulator is the result.  Read it straight from
    // TMEM, 16 rows at a time, and run the epilogue with the rows unrolled
    // (a residual's old values all in flight before the first add).  SwiGLU
    // and float outputs with 16-byte aligned rows leave through a staged slab.
    const bool slab = (epi.kind == GE_SWIGLU || epi.kind == GE_F32) &&
                      (reinterpret_cast<uintptr_t>(epi.out) & 15) == 0 && (epi.ldo & (epi.kind == GE_F32 ? 3 : 7)) == 0;
#pragma unroll 1
    for (int c = 0; c < BN / 16; ++c) {
      if (c * 16 >= rows) break;  // uniform
      float v[16];
      tmem_ld16(trow + c * 16, v);
      if (epi.in_ssq) {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] *= rsc[c * 16 + i];  // rows past `rows` are never stored
      }
      if (epi.kind == GE_RESID) {
        float* col = reinterpret_cast<float*>(epi.out) + m0 + ml;
        float old[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (c * 16 + i < rows) old[i] = col[(size_t)(c * 16 + i) * epi.ldo];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int n = c * 16 + i;
          if (n >= rows) break;  // uniform over the CTA
          const float x = old[i] + v[i];
          const bool ok = !flags[0];
          if (ok) resid_store(epi, n, m0 + ml, x);
          if (epi.norm_out) norm_handover(epi, n, m0 + ml, x, ok, lane);
        }
      } else if (slab) {
        // the 16-row slab staged in the dead ring, then stored in 16-byte row pieces (one store per
        // thread for SwiGLU's 16 x 64 bf16, four for 16 x 128 float)
        if (epi.kind == GE_SWIGLU) {
          bf16* st = reinterpret_cast<bf16*>(smem);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float partner = __shfl_xor_sync(0xffffffffu, v[i], 1);  // the up row of gate row ml
            if ((ml & 1) == 0) st[i * 64 + (ml >> 1)] = __float2bfloat16_rn(silu_f(v[i]) * partner);
          }
          __syncthreads();
          const int n = c * 16 + (ml >> 3);
          if (n < rows && !flags[0])
            *reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(epi.out) + (size_t)n * epi.ldo + (m0 >> 1) + (ml & 7) * 8) =
                reinterpret_cast<const uint4*>(smem)[ml];
        } else {  // GE_F32
          float* st = reinterpret_cast<float*>(smem);
#pragma unroll
          for (int i = 0; i < 16; ++i) st[i * 128 + ml] = v[i];
          __syncthreads();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int idx = k * 128 + ml, n = c * 16 + (idx >> 5);
            if (n < rows && !flags[0])
              *reinterpret_cast<float4*>(reinterpret_cast<float*>(epi.out) + (size_t)n * epi.ldo + m0 + (idx & 31) * 4) =
                  reinterpret_cast<const float4*>(smem)[idx];
          }
        }
        __syncthreads();  // the slab is rewritten for the next 16 rows
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int n = c * 16 + i;  // uniform over the CTA
          if (n < rows) {
            const float partner = __shfl_xor_sync(0xffffffffu, v[i], 1);
            if (!flags[0]) gemm_epi(epi, n, m0 + ml, v[i], partner, status);
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
      tc_fence_after();
      tmem_dealloc(tmem, C::TMEM_COLS);
    }
    return;
  }
  // park the partial tile: red[n][ml]
#pragma unroll 1
  for (int c = 0; c < BN / 16; ++c) {
    if (c * 16 >= rows) break;  // uniform
    float v[16];
    tmem_ld16(trow + c * 16, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) red[(c * 16 + i) * C::BM + ml] = flags[0] ? 0.f : v[i];
  }
  tc_fence_before();
  cluster_sync();  // every partial of the tile is in shared memory
  if (epi_vec4_ok(epi)) {
    // This CTA's rows n = r + j S, warp w taking rows j = w, w + 4, ...: each lane sums four columns
    // over the splits (split order) and applies the epilogue to them straight away.
    const uint32_t red_local = smem_u32(red);
    const int J = rows > r ? (rows - r + S - 1) / S : 0;
    const bool ok = !flags[0];
    auto row_epi = [&](int j, int n, float4 a) {
      if (epi.in_ssq) {
        const float sc = rsc[n];
        a = make_float4(a.x * sc, a.y * sc, a.z * sc, a.w * sc);
      }
      gemm_epi4(epi, n, m0 + lane * 4, a, ok, lane, pf, j, pre_x, pre_cs, pre_pos, status);
    };
    switch (S) {  // the split counts the policy produces
      case 2: split_rows4<2, C::BM>(red_local, r, J, warp, lane, row_epi); break;
      case 4: split_rows4<4, C::BM>(red_local, r, J, warp, lane, row_epi); break;
      case 8: split_rows4<8, C::BM>(red_local, r, J, warp, lane, row_epi); break;
      default:
        for (int j = warp; j < J; j += 4) {
          const int n = r + j * S;
          float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
          if (S == 1) {
            a = *reinterpret_cast<const float4*>(red + n * C::BM + lane * 4);
          } else {
            const uint32_t off = (uint32_t)((n * C::BM + lane * 4) * 4);
            for (int cc = 0; cc < S; ++cc) {
              const float4 p = ld_dsmem4(dsmem_addr(red_local, (uint32_t)cc) + off);
              a.x += p.x;
              a.y += p.y;
              a.z += p.z;
              a.w += p.w;
            }
          }
          row_epi(j, n, a);
        }
    }
    cluster_arrive();  // this CTA has read the other partials
  } else {
    // This CTA's rows n = r + j S summed over the splits: warp w takes rows j = w, w + 4, ..., each lane
    // four columns; the sums go to the dead ring past the partial tile.  (S = 1: the tile is the sum.)
    const float* sums = red;
    if (S > 1) {
      const uint32_t red_local = smem_u32(red);
      float* sbuf = reinterpret_cast<float*>(smem + C::RED_BYTES);  // [row j][128]
      const int J = rows > r ? (rows - r + S - 1) / S : 0;
      for (int j = warp; j < J; j += 4) {
        const uint32_t off = (uint32_t)(((r + j * S) * C::BM + lane * 4) * 4);
        float4 a;
        switch (S) {  // the split counts the policy produces
          case 2: a = sum_splits4<2>(red_local, off); break;
          case 4: a = sum_splits4<4>(red_local, off); break;
          case 8: a = sum_splits4<8>(red_local, off); break;
          default:
            a = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int cc = 0; cc < S; ++cc) {
              const float4 p = ld_dsmem4(dsmem_addr(red_local, (uint32_t)cc) + off);
              a.x += p.x;
              a.y += p.y;
              a.z += p.z;
              a.w += p.w;
            }
        }
        reinterpret_cast<float4*>(sbuf)[j * 32 + lane] = a;
      }
      __syncthreads();
      sums = sbuf;
    }
    // this CTA has read the other partials: its own may be released once every CTA has said so, which
    // the epilogue's stores overlap
    cluster_arrive();
    for (int n = r; n < rows; n += S) {
      const int j = (n - r) / S;
      float acc = sums[j * C::BM + ml], pacc = rope ? sums[j * C::BM + (ml ^ 64)] : 0.f;
      if (epi.in_ssq) {
        acc *= rsc[n];
        pacc *= rsc[n];
      }
      const bool ok = !flags[0];
      if (epi.kv_q8) {  // GE_QKV into an 8-bit cache
        int pos;
        float2 cs;
        if (pf) {
          const int j = (n - r) / S;
          pos = pre_pos[j];
          cs = pre_cs[j * 64 + (ml & 63)];
        } else {
          const int b = n / epi.rows_per_seq, jj = n % epi.rows_per_seq;
          pos = epi.len[b] + jj;
          const int rpos = epi.rope_off ? epi.len[b] + epi.rope_off[n] : pos;
          cs = (rpos >= 0 && rpos < epi.capacity) ? epi.rope[(size_t)rpos * 64 + (ml & 63)] : make_float2(1.f, 0.f);
        }
        qkv_q8_out(epi, n, m0 + ml, acc, pacc, pos, cs, ok, red_q8, status);
        continue;
      }
      if (pf) {  // operands already in shared memory
        const int j = (n - r) / S;
        if (epi.kind == GE_RESID) {
          const float x = pre_x[j * 128 + ml] + acc;
          if (ok) resid_store(epi, n, m0 + ml, x);
          if (epi.norm_out) norm_handover(epi, n, m0 + ml, x, ok, lane);
        } else if (ok && pre_pos[j] >= 0) {
          gemm_epi_rope(epi, n, m0 + ml, acc, pacc, pre_pos[j], pre_cs[j * 64 + (ml & 63)], status);
        }
        continue;
      }
      if (epi.kind == GE_RESID && epi.norm_out) {
        const float x = reinterpret_cast<const float*>(epi.out)[(size_t)n * epi.ldo + m0 + ml] + acc;
        if (ok) resid_store(epi, n, m0 + ml, x);
        norm_handover(epi, n, m0 + ml, x, ok, lane);
        continue;
      }
      const float partner = rope ? pacc : __shfl_xor_sync(0xffffffffu, acc, 1);
      if (ok) gemm_epi(epi, n, m0 + ml, acc, partner, status);
    }
  }
  cluster_wait();  // no CTA leaves while its partial may still be read
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*PFN_encodeTiled_t)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                      const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static PFN_encodeTiled_t encode_fn() {
  static PFN_encodeTiled_t fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled_t>(p);
  });
  return fn;
}

// 2-D bf16 map over a row-major [outer][inner] matrix with row stride `ld`
// elements, 128-byte swizzled boxes of box_inner x box_outer.
static bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                     uint32_t box_inner, uint32_t box_outer) {
  PFN_encodeTiled_t fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

bool gemm_shape_ok(int dtype, int M, int K) {
  if (dtype != DFLASH_BF16) return M > 0 && K > 0;
  return M > 0 && K > 0 && M % 128 == 0 && K % 64 == 0;
}

// Split count for an [M x K] weight: enough clusters to cover two CTAs per SM,
// at most 8 (portable cluster size), at least 4 k-blocks per CTA, rounded
// down to a power of two.
// Split policy (build-time): clusters of a power-of-two size, sized so the
// grid covers DFL_SPLIT_SLOTS CTAs per SM.  Power-of-two clusters pack the
// GPCs best on GB300 (measured: a 6-way QKV split ran 1.5x slower than 4-way).
#ifndef DFL_SPLIT_POW2
#define DFL_SPLIT_POW2 1
#endif
#ifndef DFL_SPLIT_SLOTS
#define DFL_SPLIT_SLOTS 2
#endif
#ifndef DFL_CL_STAGES_16
#define DFL_CL_STAGES_16 6
#endif
int gemm_splits(int M, int K) {
  const int tiles = M / 128, KB = K / 64;
  const int slots = DFL_SPLIT_SLOTS * num_sms();
  int s = tiles >= slots ? 1 : slots / tiles;
  if (s > 8) s = 8;
  if (s > KB / 4) s = KB / 4;
  if (DFL_SPLIT_POW2) {
    int p = 1;
    while (p * 2 <= s) p *= 2;
    s = p;
  }
  return s < 1 ? 1 : s;
}

template <int BN, int STAGES>
static cudaError_t launch_cl(const CUtensorMap& tw, const CUtensorMap& tx, const GemmEpi& epi, int rows, int M, int K,
                             int S, int* status, cudaStream_t s) {
  using C = ClCfg<BN, STAGES>;
  static bool set = false;
  if (!set) {
    DFL_RET(cudaFuncSetAttribute(gemm_cl_kernel<BN, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
    set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, M / 128, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = S;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  count_launch();
  return cudaLaunchKernelEx(&cfg, gemm_cl_kernel<BN, STAGES>, tw, tx, epi, rows, K, S, status,
                            (uint64_t)g_wait_ns.load(std::memory_order_relaxed));
}

cudaError_t gemm_bf16(const void* X, int ldx, int rows, const void* W, int M, int K, const GemmEpi& epi, int* status,
                      cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (rows > kMaxRows || !gemm_shape_ok(DFLASH_BF16, M, K)) return cudaErrorInvalidValue;
  if ((epi.kind == GE_QKV || epi.kind == GE_INJECT) && (!epi.len || !epi.rope || epi.rows_per_seq <= 0))
    return cudaErrorInvalidValue;
  const int S = gemm_splits(M, K);
  const int bn = rows <= 16 ? 16 : rows <= 32 ? 32 : rows <= 64 ? 64 : 128;
  CUtensorMap tw, tx;
  if (!make_map(&tw, W, (uint64_t)K, (uint64_t)M, (uint64_t)K, 64, 128)) return cudaErrorInvalidValue;
  if (!make_map(&tx, X, (uint64_t)K, (uint64_t)rows, (uint64_t)ldx, 64, (uint32_t)bn)) return cudaErrorInvalidValue;
  switch (bn) {
    case 16: return launch_cl<16, DFL_CL_STAGES_16>(tw, tx, epi, rows, M, K, S, status, s);
    case 32: return launch_cl<32, 5>(tw, tx, epi, rows, M, K, S, status, s);
    case 64: return launch_cl<64, 4>(tw, tx, epi, rows, M, K, S, status, s);
    default: return launch_cl<128, 3>(tw, tx, epi, rows, M, K, S, status, s);
  }
}

}  // namespace dfl
