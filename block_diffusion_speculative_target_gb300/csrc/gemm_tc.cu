// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA, for the dense products of the DFlash step at 1-128 tokens:
// fusion Linear, KV-injection projections, QKV / O / gate-up / down and the
// LM head.
//
//   y[n][m] = sum_k x[n][k] * w[m][k]        w: [M][K] bf16, x: [rows][K] bf16
//
// Swap-AB: the weight tile is the MMA's A operand (M = 128 output features),
// the tokens are the B operand (N = 16..128, rows past `rows` are zero-filled
// by TMA), the fp32 accumulator lives in TMEM.  Weights dominate the bytes, so
// each CTA streams one 128-row weight slab through a multi-stage TMA ring with
// an evict-first L2 policy.  Narrow outputs are split along K (the split count
// depends only on M, K and the SM count) and reduced in a fixed order by the
// last CTA of each tile, so results are deterministic and independent of the
// token count.
//
// Roles (128 threads): warp 0 lane 0 issues TMA, warp 1 lane 0 issues MMAs,
// warp 2 owns the TMEM allocation, and all four warps run the epilogue (warp w
// reads TMEM lanes 32w..32w+31 = output features m0+32w..).
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dfl {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

template <int BN, int STAGES>
struct TcCfg {
  static constexpr int BM = 128, BK = 64;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = BN < 32 ? 32 : BN;
  static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + 256;
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

template <int BN, int STAGES>
__global__ void __launch_bounds__(128, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const Epi epi,
                   const int rows, const int M, const int K, const int splits, float* __restrict__ part,
                   int* __restrict__ tickets, int* status) {
  using C = TcCfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * C::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * C::B_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* accb = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [0] abort, [1] last CTA of tile

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, split = blockIdx.y;
  const int KB = K / C::BK;
  const int kb0 = (int)((long long)split * KB / splits);
  const int kb1 = (int)((long long)(split + 1) * KB / splits);
  const int nkb = kb1 - kb0;
  const int m0 = tile * C::BM;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(accb, 1);
    flags[0] = 0;
    flags[1] = 0;
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

  int issued = 0;  // k-blocks whose loads were issued (producer only)
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const int pre = nkb < STAGES ? nkb : STAGES;
      // Weights do not depend on the previous kernel: start streaming them first.
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], C::STAGE_BYTES);
        tma_load_2d_hint(sA + i * C::A_BYTES, &tmW, &full[i], (kb0 + i) * C::BK, m0, pol);
      }
      pdl_wait();
      for (int i = 0; i < pre; ++i) tma_load_2d(sB + i * C::B_BYTES, &tmX, &full[i], (kb0 + i) * C::BK, 0);
      issued = pre;
      for (int kb = pre; kb < nkb; ++kb) {
        const int s = kb % STAGES;
        const uint32_t ph = (uint32_t)((kb / STAGES) - 1) & 1u;
        if (!mbar_wait(&empty[s], ph, kWaitLimitNs)) {
          flags[0] = 1;
          set_status(status, DFLASH_STATUS_TIMEOUT);
          break;
        }
        if (flags[0]) break;
        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
        tma_load_2d_hint(sA + s * C::A_BYTES, &tmW, &full[s], (kb0 + kb) * C::BK, m0, pol);
        tma_load_2d(sB + s * C::B_BYTES, &tmX, &full[s], (kb0 + kb) * C::BK, 0);
        issued = kb + 1;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(C::BM, BN);
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % STAGES;
        const uint32_t ph = (uint32_t)(kb / STAGES) & 1u;
        if (!mbar_wait(&full[s], ph, kWaitLimitNs)) {
          flags[0] = 1;
          set_status(status, DFLASH_STATUS_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint64_t da = smem_desc_sw128(sA + s * C::A_BYTES);
        const uint64_t db = smem_desc_sw128(sB + s * C::B_BYTES);
#pragma unroll
        for (int k = 0; k < C::BK / 16; ++k)  // 16 bf16 = 32 bytes per MMA step along K
          tc_mma_f16(tmem, da + 2 * k, db + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
        tc_commit(&empty[s]);
      }
      tc_commit(accb);
    }
    __syncwarp();
  }

  // ---------------------------------------------------------------- epilogue
  const bool acc_ok = mbar_wait(accb, 0, kWaitLimitNs);
  if (!acc_ok) {
    flags[0] = 1;
    if (lane == 0) set_status(status, DFLASH_STATUS_TIMEOUT);
  }
  tc_fence_after();
  pdl_wait();
  const int m = m0 + warp * 32 + lane;
  const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
  if (splits == 1) {
#pragma unroll 1
    for (int c = 0; c < BN / 16; ++c) {
      if (c * 16 >= rows) break;  // uniform across the CTA
      float v[16];
      tmem_ld16(trow + c * 16, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float p = __shfl_xor_sync(0xffffffffu, v[i], 1);
        epi_apply(epi, rows, c * 16 + i, m, v[i], p);
      }
    }
  } else {
#pragma unroll 1
    for (int c = 0; c < BN / 16; ++c) {
      if (c * 16 >= rows) break;
      float v[16];
      tmem_ld16(trow + c * 16, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int n = c * 16 + i;
        if (n < rows) part[((size_t)split * rows + n) * M + m] = v[i];
      }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const int t = atomicAdd(&tickets[tile], 1);
      flags[1] = (t == splits - 1) ? 1 : 0;
    }
    __syncthreads();
    if (flags[1]) {
      __threadfence();
#pragma unroll 1
      for (int n = 0; n < rows; ++n) {
        float acc = 0.f;
        for (int s = 0; s < splits; ++s) acc += __ldcg(&part[((size_t)s * rows + n) * M + m]);
        const float p = __shfl_xor_sync(0xffffffffu, acc, 1);
        epi_apply(epi, rows, n, m, acc, p);
      }
      if (threadIdx.x == 0) tickets[tile] = 0;
    }
  }
  pdl_launch();

  // Drain: after a time-out, wait (bounded) for loads still in flight before
  // the shared memory is released.
  if (flags[0] && warp == 0 && lane == 0) {
    const int first = issued > STAGES ? issued - STAGES : 0;
    for (int kb = first; kb < issued; ++kb)
      mbar_wait(&full[kb % STAGES], (uint32_t)(kb / STAGES) & 1u, kWaitLimitNs / 4);
  }
  tc_fence_before();
  __syncthreads();
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

int gemm_splits(int M, int K) {
  const int tiles = M / 128, KB = K / 64;
  const int slots = 2 * num_sms();  // two CTAs per SM
  int s = tiles >= slots ? 1 : slots / tiles;
  const int max_s = KB / 4 > 0 ? KB / 4 : 1;  // keep >= 4 k-blocks per CTA
  if (s > max_s) s = max_s;
  return s < 1 ? 1 : s;
}

bool gemm_shape_ok(int dtype, int M, int K) {
  if (dtype != DFLASH_BF16) return M > 0 && K > 0;
  return M > 0 && K > 0 && M % 128 == 0 && K % 64 == 0;
}

template <int BN, int STAGES>
static cudaError_t launch_tc(const CUtensorMap& tw, const CUtensorMap& tx, const Epi& epi, int rows, int M, int K,
                             int splits, const GemmScratch& scr, int* status, cudaStream_t s) {
  using C = TcCfg<BN, STAGES>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(M / 128, splits, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launch();
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, STAGES>, tw, tx, epi, rows, M, K, splits, scr.part,
                            scr.tickets, status);
}

cudaError_t gemm_simt(const float* X, int ldx, int rows, const float* W, int M, int K, const Epi& epi, cudaStream_t s);

cudaError_t gemm(int dtype, const void* X, int ldx, int rows, const void* W, int M, int K, const Epi& epi,
                 const GemmScratch& scr, int* status, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (rows > kMaxRows) return cudaErrorInvalidValue;
  if (dtype != DFLASH_BF16) return gemm_simt((const float*)X, ldx, rows, (const float*)W, M, K, epi, s);
  if (!gemm_shape_ok(dtype, M, K)) return cudaErrorInvalidValue;
  const int splits = gemm_splits(M, K);
  if (splits > 1) {
    if ((size_t)splits * rows * M > scr.part_elems || M / 128 > scr.n_tickets) return cudaErrorInvalidValue;
  }
  const int bn = rows <= 16 ? 16 : rows <= 32 ? 32 : rows <= 64 ? 64 : 128;
  CUtensorMap tw, tx;
  if (!make_map(&tw, W, (uint64_t)K, (uint64_t)M, (uint64_t)K, 64, 128)) return cudaErrorInvalidValue;
  if (!make_map(&tx, X, (uint64_t)K, (uint64_t)rows, (uint64_t)ldx, 64, (uint32_t)bn)) return cudaErrorInvalidValue;
  switch (bn) {
    case 16: return launch_tc<16, 6>(tw, tx, epi, rows, M, K, splits, scr, status, s);
    case 32: return launch_tc<32, 5>(tw, tx, epi, rows, M, K, splits, scr, status, s);
    case 64: return launch_tc<64, 4>(tw, tx, epi, rows, M, K, splits, scr, status, s);
    default: return launch_tc<128, 3>(tw, tx, epi, rows, M, K, splits, scr, status, s);
  }
}

}  // namespace dfl
