// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA, for the dense products of the DFlash step at 1-128 tokens:
// fusion Linear, KV-injection projections, QKV / O / gate-up / down and the
// LM head.
//
//   y[n][m] = sum_k x[n][k] * w[m][k]        w: [M][K] bf16, x: [rows][K] bf16
//
// Swap-AB: a 128-row weight tile is the MMA's A operand, the tokens are the B
// operand (N = 16..128; rows past `rows` are zero-filled by TMA), the fp32
// accumulator lives in TMEM.  The weights dominate the bytes, so the kernel is
// persistent and balanced by bytes ("stream-K"): the (tile, 64-wide k-block)
// units of the whole product are cut into one contiguous range per CTA, one
// CTA per SM, and each CTA streams its range through a deep TMA ring with an
// evict-first L2 policy.  A tile whose k-range spans several CTAs is reduced
// by the last CTA to finish its part, summing the parts in k order, so the
// result is deterministic and independent of the token count (the cut depends
// only on M, K and the SM count).
//
// Roles (192 threads): warp 0 issues TMA, warp 1 owns TMEM and issues MMAs,
// warps 2-5 run the epilogue; epilogue warp w reads TMEM lanes
// 32*(w%4)..+31, i.e. output features m0 + 32*(w%4) + lane.  Two TMEM
// accumulators let the epilogue of one tile overlap the next tile's MMAs.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dfl {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Build-time shape of the persistent grid and of the TMA ring per token tile.
#ifndef DFL_GEMM_CTAS_PER_SM
#define DFL_GEMM_CTAS_PER_SM 2
#endif
#ifndef DFL_GEMM_STAGES_16
#define DFL_GEMM_STAGES_16 5
#endif
#ifndef DFL_GEMM_STAGES_32
#define DFL_GEMM_STAGES_32 5
#endif
#ifndef DFL_GEMM_STAGES_64
#define DFL_GEMM_STAGES_64 4
#endif
#ifndef DFL_GEMM_STAGES_128
#define DFL_GEMM_STAGES_128 3
#endif

template <int BN, int STAGES>
struct TcCfg {
  static constexpr int BM = 128, BK = 64;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int ACC_COLS = BN;                            // one accumulator
  static constexpr int TMEM_COLS = (2 * BN) < 32 ? 32 : 2 * BN;  // two accumulators
  static constexpr int THREADS = 192;
  static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + 512;
};

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Apply the epilogue to output (n, m).  `partner` is y[n][m ^ 1] (SwiGLU).
__device__ __forceinline__ void epi_apply(const Epi& e, int rows, int n, int m, float v, float partner) {
  if (n >= rows) return;
  switch (e.kind) {
    case EPI_F32:
      reinterpret_cast<float*>(e.out)[(size_t)n * e.ldo + m] = v;
      break;
    case EPI_STORE:
      reinterpret_cast<bf16*>(e.out)[(size_t)n * e.ldo + m] = __float2bfloat16_rn(v);
      break;
    case EPI_RESID:
      reinterpret_cast<float*>(e.out)[(size_t)n * e.ldo + m] += v;
      break;
    case EPI_SWIGLU:
      if ((m & 1) == 0)
        reinterpret_cast<bf16*>(e.out)[(size_t)n * e.ldo + (m >> 1)] = __float2bfloat16_rn(silu_f(v) * partner);
      break;
  }
}

__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// First unit of CTA c among G CTAs sharing U units.
__device__ __forceinline__ long long unit_begin(int c, long long U, int G) { return (long long)c * U / G; }
// CTA that processes unit u.
__device__ __forceinline__ int unit_owner(long long u, long long U, int G) {
  return (int)(((u + 1) * G - 1) / U);
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(192)
    gemm_sk_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const Epi epi,
                   const int rows, const int M, const int K, float* __restrict__ part, int* __restrict__ tickets,
                   int* status) {
  using C = TcCfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * C::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * C::B_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;  // [2]
  uint64_t* acc_empty = acc_full + 2;   // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [0] abort, [1] reducer flag

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int KB = K / C::BK;
  const long long U = (long long)(M / C::BM) * KB;
  const long long u0 = unit_begin(c, U, G), u1 = unit_begin(c + 1, U, G);
  const int nunits = (int)(u1 - u0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    flags[0] = 0;
    flags[1] = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch();  // dependents may be scheduled; they wait for this grid to complete

  int issued = 0;
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const int pre = nunits < STAGES ? nunits : STAGES;
      // Weights do not depend on the previous kernel: start streaming them first.
      for (int i = 0; i < pre; ++i) {
        const long long u = u0 + i;
        const int t = (int)(u / KB), kb = (int)(u % KB);
        mbar_arrive_expect_tx(&full[i], C::STAGE_BYTES);
        tma_load_2d_hint(sA + i * C::A_BYTES, &tmW, &full[i], kb * C::BK, t * C::BM, pol);
      }
      pdl_wait();
      for (int i = 0; i < pre; ++i) {
        const int kb = (int)((u0 + i) % KB);
        tma_load_2d(sB + i * C::B_BYTES, &tmX, &full[i], kb * C::BK, 0);
      }
      issued = pre;
      for (int i = pre; i < nunits; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait(&empty[s], (uint32_t)((i / STAGES) - 1) & 1u, kWaitLimitNs) || flags[0]) {
          flags[0] = 1;
          set_status(status, DFLASH_STATUS_TIMEOUT);
          break;
        }
        const long long u = u0 + i;
        const int t = (int)(u / KB), kb = (int)(u % KB);
        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
        tma_load_2d_hint(sA + s * C::A_BYTES, &tmW, &full[s], kb * C::BK, t * C::BM, pol);
        tma_load_2d(sB + s * C::B_BYTES, &tmX, &full[s], kb * C::BK, 0);
        issued = i + 1;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(C::BM, BN);
      int seg = 0;
      bool ok = true;
      for (int i = 0; i < nunits && ok; ++i) {
        const long long u = u0 + i;
        const int kb = (int)(u % KB);
        const bool first = (i == 0) || kb == 0;
        const bool last = (i + 1 == nunits) || kb == KB - 1;
        const int b = seg & 1;
        if (first && seg >= 2) {
          if (!mbar_wait(&acc_empty[b], (uint32_t)((seg >> 1) - 1) & 1u, kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        const int s = i % STAGES;
        if (!mbar_wait(&full[s], (uint32_t)(i / STAGES) & 1u, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t da = smem_desc_sw128(sA + s * C::A_BYTES);
        const uint64_t db = smem_desc_sw128(sB + s * C::B_BYTES);
        const uint32_t dt = tmem + (uint32_t)(b * C::ACC_COLS);
#pragma unroll
        for (int k = 0; k < C::BK / 16; ++k)  // 16 bf16 = 32 bytes per MMA step along K
          tc_mma_f16(dt, da + 2 * k, db + 2 * k, idesc, (!first || k > 0) ? 1u : 0u);
        tc_commit(&empty[s]);
        if (last) {
          tc_commit(&acc_full[b]);
          ++seg;
        }
      }
      if (!ok) {
        flags[0] = 1;
        set_status(status, DFLASH_STATUS_TIMEOUT);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter
    const int ml = q * 32 + lane;
    pdl_wait();
    int seg = 0;
    long long u = u0;
    while (u < u1) {
      const int t = (int)(u / KB);
      const int kb_begin = (int)(u - (long long)t * KB);
      const long long tile_end = (long long)(t + 1) * KB;
      const long long seg_end = u1 < tile_end ? u1 : tile_end;
      const bool whole = (kb_begin == 0) && (seg_end == tile_end);
      const int b = seg & 1;
      const int m = t * C::BM + ml;
      const bool got = mbar_wait(&acc_full[b], (uint32_t)(seg >> 1) & 1u, kWaitLimitNs);
      if (!got) {
        flags[0] = 1;
        if (lane == 0) set_status(status, DFLASH_STATUS_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * C::ACC_COLS);
      const int slot = (u0 >= (long long)t * KB) ? 0 : 1;
      float* mypart = part + ((size_t)(c * 2 + slot) * rows) * C::BM;
#pragma unroll 1
      for (int cc = 0; cc < BN / 16; ++cc) {
        if (cc * 16 >= rows) break;  // uniform
        float v[16];
        tmem_ld16(trow + cc * 16, v);
        if (whole) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float p = __shfl_xor_sync(0xffffffffu, v[i], 1);
            epi_apply(epi, rows, cc * 16 + i, m, v[i], p);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int n = cc * 16 + i;
            if (n < rows) mypart[(size_t)n * C::BM + ml] = v[i];
          }
        }
      }
      // release the accumulator to the MMA warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cnt1(&acc_empty[b]);
      if (!whole) {
        // hand in this part; the last CTA to do so reduces the tile in k order
        const int c_first = unit_owner((long long)t * KB, U, G);
        const int c_last = unit_owner(tile_end - 1, U, G);
        __threadfence();
        epi_bar_sync();
        if (warp == 2 && lane == 0) {
          const int prev = atomicAdd(&tickets[t], 1);
          flags[1] = (prev == c_last - c_first) ? 1 : 0;
        }
        epi_bar_sync();
        if (flags[1]) {
          __threadfence();
#pragma unroll 1
          for (int n0 = 0; n0 < rows; n0 += 8) {
            float acc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = 0.f;
            for (int cp = c_first; cp <= c_last; ++cp) {
              const int sl = (unit_begin(cp, U, G) >= (long long)t * KB) ? 0 : 1;
              const float* pp = part + ((size_t)(cp * 2 + sl) * rows) * C::BM + ml;
              float tv[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) tv[j] = (n0 + j < rows) ? __ldcg(pp + (size_t)(n0 + j) * C::BM) : 0.f;
#pragma unroll
              for (int j = 0; j < 8; ++j) acc[j] += tv[j];
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float p = __shfl_xor_sync(0xffffffffu, acc[j], 1);
              epi_apply(epi, rows, n0 + j, m, acc[j], p);
            }
          }
          if (warp == 2 && lane == 0) tickets[t] = 0;
        }
        epi_bar_sync();  // flags[1] is rewritten by the next partial tile
      }
      u = seg_end;
      ++seg;
    }
  }

  // Drain: after a time-out, wait (bounded) for loads still in flight before
  // the shared memory is released.
  __syncthreads();
  if (flags[0] && warp == 0 && lane == 0) {
    const int first = issued > STAGES ? issued - STAGES : 0;
    for (int i = first; i < issued; ++i) mbar_wait(&full[i % STAGES], (uint32_t)(i / STAGES) & 1u, kWaitLimitNs / 4);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
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

// CTAs of the stream-K cut for an [M x K] weight: one per SM, fewer only when
// the product has fewer units than SMs.  Depends on M, K and the GPU only.
int gemm_splits(int M, int K) {
  const long long U = (long long)(M / 128) * (K / 64);
  const int G = DFL_GEMM_CTAS_PER_SM * num_sms();
  return (int)(U < G ? U : G);
}

bool gemm_shape_ok(int dtype, int M, int K) {
  if (dtype != DFLASH_BF16) return M > 0 && K > 0;
  return M > 0 && K > 0 && M % 128 == 0 && K % 64 == 0;
}

template <int BN, int STAGES>
static cudaError_t launch_tc(const CUtensorMap& tw, const CUtensorMap& tx, const Epi& epi, int rows, int M, int K,
                             const GemmScratch& scr, int* status, cudaStream_t s) {
  using C = TcCfg<BN, STAGES>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_sk_kernel<BN, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(gemm_splits(M, K), 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launch();
  return cudaLaunchKernelEx(&cfg, gemm_sk_kernel<BN, STAGES>, tw, tx, epi, rows, M, K, scr.part, scr.tickets, status);
}

cudaError_t gemm_simt(const float* X, int ldx, int rows, const float* W, int M, int K, const Epi& epi, cudaStream_t s);

cudaError_t gemm(int dtype, const void* X, int ldx, int rows, const void* W, int M, int K, const Epi& epi,
                 const GemmScratch& scr, int* status, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (rows > kMaxRows) return cudaErrorInvalidValue;
  if (dtype != DFLASH_BF16) return gemm_simt((const float*)X, ldx, rows, (const float*)W, M, K, epi, s);
  if (!gemm_shape_ok(dtype, M, K)) return cudaErrorInvalidValue;
  const int G = gemm_splits(M, K);
  if ((size_t)G * 2 * rows * 128 > scr.part_elems || M / 128 > scr.n_tickets) return cudaErrorInvalidValue;
  const int bn = rows <= 16 ? 16 : rows <= 32 ? 32 : rows <= 64 ? 64 : 128;
  CUtensorMap tw, tx;
  if (!make_map(&tw, W, (uint64_t)K, (uint64_t)M, (uint64_t)K, 64, 128)) return cudaErrorInvalidValue;
  if (!make_map(&tx, X, (uint64_t)K, (uint64_t)rows, (uint64_t)ldx, 64, (uint32_t)bn)) return cudaErrorInvalidValue;
  switch (bn) {
    case 16: return launch_tc<16, DFL_GEMM_STAGES_16>(tw, tx, epi, rows, M, K, scr, status, s);
    case 32: return launch_tc<32, DFL_GEMM_STAGES_32>(tw, tx, epi, rows, M, K, scr, status, s);
    case 64: return launch_tc<64, DFL_GEMM_STAGES_64>(tw, tx, epi, rows, M, K, scr, status, s);
    default: return launch_tc<128, DFL_GEMM_STAGES_128>(tw, tx, epi, rows, M, K, scr, status, s);
  }
}

}  // namespace dfl
