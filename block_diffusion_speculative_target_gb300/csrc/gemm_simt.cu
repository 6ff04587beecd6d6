// float32 GEMM on the CUDA cores for the fp32 configuration (tf32 tensor
// cores cannot hold a 1e-4 bound).  y[n][m] = sum_k x[n][k] w[m][k] with a
// fixed k order per output.  Each thread owns an (even, odd) pair of output
// features, so the gate/up SwiGLU epilogue stays inside one thread.
#include "common.cuh"
#include "internal.h"

namespace dfl {

constexpr int SB_M = 64, SB_N = 16, SB_K = 32;

__global__ void __launch_bounds__(256) gemm_f32_kernel(const float* __restrict__ X, int ldx, int rows,
                                                       const float* __restrict__ W, int M, int K, Epi epi) {
  __shared__ float Ws[SB_M][SB_K + 1];
  __shared__ float Xs[SB_N][SB_K + 1];
  const int m0 = blockIdx.x * SB_M, n0 = blockIdx.y * SB_N;
  const int tid = threadIdx.x;
  const int mp = tid & 31, nq = tid >> 5;  // m pair index, n pair index
  const int ml = 2 * mp, nl = 2 * nq;
  float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  pdl_launch();
  pdl_wait();
  for (int k0 = 0; k0 < K; k0 += SB_K) {
    for (int i = tid; i < SB_M * SB_K; i += 256) {
      const int r = i / SB_K, c = i % SB_K;
      const int gm = m0 + r, gk = k0 + c;
      Ws[r][c] = (gm < M && gk < K) ? W[(size_t)gm * K + gk] : 0.f;
    }
    for (int i = tid; i < SB_N * SB_K; i += 256) {
      const int r = i / SB_K, c = i % SB_K;
      const int gn = n0 + r, gk = k0 + c;
      Xs[r][c] = (gn < rows && gk < K) ? X[(size_t)gn * ldx + gk] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int c = 0; c < SB_K; ++c) {
      const float w0 = Ws[ml][c], w1 = Ws[ml + 1][c];
      const float x0 = Xs[nl][c], x1 = Xs[nl + 1][c];
      acc[0][0] = fmaf(x0, w0, acc[0][0]);
      acc[0][1] = fmaf(x0, w1, acc[0][1]);
      acc[1][0] = fmaf(x1, w0, acc[1][0]);
      acc[1][1] = fmaf(x1, w1, acc[1][1]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 2; ++a) {
    const int n = n0 + nl + a;
    if (n >= rows) continue;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int m = m0 + ml + b;
      if (m >= M) continue;
      const float v = acc[a][b];
      switch (epi.kind) {
        case EPI_F32:
        case EPI_STORE:
          reinterpret_cast<float*>(epi.out)[(size_t)n * epi.ldo + m] = v;
          break;
        case EPI_RESID:
          reinterpret_cast<float*>(epi.out)[(size_t)n * epi.ldo + m] += v;
          break;
        case EPI_SWIGLU:
          if (b == 0 && m + 1 < M) {
            const float g = v, u = acc[a][1];
            reinterpret_cast<float*>(epi.out)[(size_t)n * epi.ldo + (m >> 1)] = g / (1.0f + expf(-g)) * u;
          }
          break;
      }
    }
  }
}

cudaError_t gemm_simt(const float* X, int ldx, int rows, const float* W, int M, int K, const Epi& epi,
                      cudaStream_t s) {
  dim3 grid((M + SB_M - 1) / SB_M, (rows + SB_N - 1) / SB_N);
  DFL_RET(launch_pdl(gemm_f32_kernel, dim3(grid), dim3(256), 0, s, X, ldx, rows, W, M, K, epi));
  count_launch();
  return cudaGetLastError();
}

}  // namespace dfl
