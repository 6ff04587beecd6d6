// Sampling-mode kernels (temperature T > 0): softmax statistics of logit
// rows, inverse-CDF draws, and speculative-sampling verification with
// rollback.  Every reduction runs in a fixed order (per-thread contiguous
// slices of the row, then a fixed tree over the threads), so a draw depends
// only on the row's logits and the caller's uniform number.
//
// With c = log2(e) / T, a row's weights are e_t = 2^((z_t - max z) c) and its
// distribution is e_t / sum(e).  A draw with uniform v in [0, 1) is the
// smallest t whose running sum exceeds v * sum (the inverse CDF).
#include "common.cuh"
#include "internal.h"

namespace dfl {

namespace {
constexpr int kSampThreads = 1024;

__device__ __forceinline__ float ex2s(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Deterministic block-wide max and sum (fixed trees); every thread gets the result.
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = red[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) t = fmaxf(t, red[i]);
  return t;
}

// Inverse CDF over V weights given by wfn(t) >= 0, with the draw target
// v * total.  Thread i (of 1024) owns the contiguous slice [i * per,
// (i + 1) * per) and sums it in index order.  The slice sums are turned into
// boundaries ex_0 = 0 <= ex_1 <= ... <= ex_1024 = total by sequential adds
// (lane L of warp 0 runs over slices 32 L .. 32 L + 31, lane 0 then over the
// 32 lane sums); rounding is monotone, so the intervals [ex_i, ex_{i+1})
// tile [0, total) and exactly one slice holds the target.  Its thread walks
// the slice in order.  Returns the drawn index on every thread; sh_ex holds
// 1025 floats (sh_ex[1024] = total after the call), sh_out one int.
template <typename WF>
__device__ int block_inverse_cdf(int V, float v, WF wfn, float* sh_ex, int* sh_out) {
  const int tid = threadIdx.x;
  const int per = (V + kSampThreads - 1) / kSampThreads;
  const int t0 = min(V, tid * per), t1 = min(V, t0 + per);
  float own = 0.f;
  for (int t = t0; t < t1; ++t) own += wfn(t);
  __syncthreads();
  sh_ex[tid] = own;
  __syncthreads();
  if (tid < 32) {
    float run = 0.f;
    float part[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      part[k] = run;
      run += sh_ex[tid * 32 + k];
    }
    // lane prefixes over the 32 lane sums, in lane order
    float pre = 0.f, mine = 0.f;
    for (int l = 0; l < 32; ++l) {
      const float sl = __shfl_sync(0xffffffffu, run, l);
      if (l == tid) mine = pre;
      pre += sl;
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 32; ++k) sh_ex[tid * 32 + k] = mine + part[k];
    if (tid == 0) {
      sh_ex[kSampThreads] = pre;  // total
      *sh_out = -1;
    }
  }
  __syncthreads();
  const float total = sh_ex[kSampThreads];
  float target = v * total;
  if (total > 0.f && target >= total) target = __int_as_float(__float_as_int(total) - 1);  // v * total rounded up
  const float lo = sh_ex[tid], hi = sh_ex[tid + 1];
  if (lo <= target && target < hi) {
    int pick = -1, last = -1;
    float run = lo;
    for (int t = t0; t < t1; ++t) {
      const float w = wfn(t);
      if (w > 0.f) last = t;
      run += w;
      if (run > target) {
        pick = t;
        break;
      }
    }
    *sh_out = pick >= 0 ? pick : last;
  }
  __syncthreads();
  int r = *sh_out;
  if (r < 0) {  // no weight at all (total 0): index 0
    r = 0;
  }
  return r;
}
}  // namespace

// Per row: (max z, sum_t 2^((z_t - max) c)) of float32 logits [rows][V].
__global__ void __launch_bounds__(kSampThreads) softmax_stats_kernel(const float* __restrict__ logits, int V, float c,
                                                                     float2* __restrict__ stats) {
  __shared__ float red[kSampThreads / 32];
  const float* z = logits + (size_t)blockIdx.x * V;
  pdl_launch();
  pdl_wait();
  float m = -INFINITY;
  for (int t = threadIdx.x; t < V; t += blockDim.x) m = fmaxf(m, z[t]);
  m = block_max(m, red);
  float s = 0.f;
  for (int t = threadIdx.x; t < V; t += blockDim.x) s += ex2s((z[t] - m) * c);
  s = block_sum<kSampThreads>(s, red);
  if (threadIdx.x == 0) stats[blockIdx.x] = make_float2(m, s);
}

// One draw per row r from softmax(z_r / T) with uniform v[r] into out[r].
// When skip_first_of > 0, rows with r % skip_first_of == 0 are skipped and the
// draws are indexed by the remaining rows in order (the drafter's slots 1..B-1).
__global__ void __launch_bounds__(kSampThreads) sample_rows_kernel(const float* __restrict__ logits, int V, float c,
                                                                   const float2* __restrict__ stats,
                                                                   const float* __restrict__ v, int skip_first_of,
                                                                   int32_t* __restrict__ out) {
  __shared__ float sums[kSampThreads + 1];
  __shared__ int pick;
  const int r = blockIdx.x;
  pdl_launch();
  pdl_wait();
  int vi = r;
  if (skip_first_of > 0) {
    if (r % skip_first_of == 0) return;  // uniform over the CTA
    vi = (r / skip_first_of) * (skip_first_of - 1) + (r % skip_first_of) - 1;
  }
  const float* z = logits + (size_t)r * V;
  const float m = stats[r].x;
  const int t = block_inverse_cdf(V, v[vi], [&](int i) { return ex2s((z[i] - m) * c); }, sums, &pick);
  if (threadIdx.x == 0) out[r] = t;
}

// Speculative-sampling verification of one block per sequence (one CTA per
// sequence), then the rollback: see dflash_accept_sample.
__global__ void __launch_bounds__(kSampThreads)
    accept_sample_kernel(const int32_t* __restrict__ draft, const float* __restrict__ zt,
                         const float* __restrict__ zd, const float2* __restrict__ tst, const float2* __restrict__ dst,
                         int block, int V, float c, const float* __restrict__ u, const float* __restrict__ v,
                         int32_t* len, int32_t* anchor, int32_t* n_pend, int32_t* accept_len, int32_t* stream,
                         int32_t* stream_len, int stream_cap, int* status) {
  __shared__ float sums[kSampThreads + 1];
  __shared__ int pick, acc_s;
  const int b = blockIdx.x;
  pdl_launch();
  pdl_wait();
  const int32_t* d = draft + (size_t)b * block;
  const size_t row0 = (size_t)b * block;  // rows of this sequence in the logits buffers
  if (threadIdx.x == 0) {
    int a = 0;
    while (a < block - 1) {
      const int tok = d[a + 1];
      if (tok < 0 || tok >= V) {
        set_status(status, DFLASH_STATUS_BOUNDS);
        break;
      }
      const float2 sp = tst[row0 + a], sq = dst[row0 + a + 1];
      const float p = ex2s((zt[(row0 + a) * V + tok] - sp.x) * c) / sp.y;
      const float q = ex2s((zd[(row0 + a + 1) * V + tok] - sq.x) * c) / sq.y;
      if (!(u[(size_t)b * (block - 1) + a] * q < p)) break;
      ++a;
    }
    acc_s = a;
  }
  __syncthreads();
  const int a = acc_s;
  const float* p_row = zt + (row0 + a) * V;
  const float2 sp = tst[row0 + a];
  int t;
  if (a < block - 1) {  // residual max(0, p_a - q_{a+1})
    const float* q_row = zd + (row0 + a + 1) * V;
    const float2 sq = dst[row0 + a + 1];
    const float ip = 1.f / sp.y, iq = 1.f / sq.y;
    auto resid = [&](int i) {
      return fmaxf(ex2s((p_row[i] - sp.x) * c) * ip - ex2s((q_row[i] - sq.x) * c) * iq, 0.f);
    };
    t = block_inverse_cdf(V, v[b], resid, sums, &pick);
    if (!(sums[kSampThreads] > 0.f))  // no residual mass (p == q to rounding): sample the target
      t = block_inverse_cdf(V, v[b], [&](int i) { return ex2s((p_row[i] - sp.x) * c); }, sums, &pick);
  } else {  // bonus token from the last target row
    t = block_inverse_cdf(V, v[b], [&](int i) { return ex2s((p_row[i] - sp.x) * c); }, sums, &pick);
  }
  const int lane = threadIdx.x;
  if (lane <= a && stream) {
    const int e = stream_len[b];
    const int32_t tok = lane < a ? d[lane + 1] : t;
    if (e + lane < stream_cap)
      stream[(size_t)b * stream_cap + e + lane] = tok;
    else
      set_status(status, DFLASH_STATUS_BOUNDS);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    len[b] += a + 1;
    anchor[b] = t;
    n_pend[b] = a + 1;
    if (accept_len) accept_len[b] = a;
    if (stream_len) stream_len[b] = min(stream_len[b] + a + 1, stream_cap);
  }
}

cudaError_t softmax_stats(const float* logits, int rows, int V, float temperature, float2* stats, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const float c = 1.4426950408889634f / temperature;
  DFL_RET(launch_pdl(softmax_stats_kernel, dim3(rows), dim3(kSampThreads), 0, s, logits, V, c, stats));
  count_launch();
  return cudaSuccess;
}

cudaError_t sample_rows(const float* logits, int rows, int V, float temperature, const float2* stats, const float* v,
                        int skip_first_of, int32_t* out, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const float c = 1.4426950408889634f / temperature;
  DFL_RET(launch_pdl(sample_rows_kernel, dim3(rows), dim3(kSampThreads), 0, s, logits, V, c, stats, v, skip_first_of,
                     out));
  count_launch();
  return cudaSuccess;
}

cudaError_t accept_sample(const int32_t* draft, const float* zt, const float* zd, const float2* tst, const float2* dst,
                          int batch, int block, int V, float temperature, const float* u, const float* v, int32_t* len,
                          int32_t* anchor, int32_t* n_pend, int32_t* accept_len, int32_t* stream, int32_t* stream_len,
                          int stream_cap, int* status, cudaStream_t s) {
  const float c = 1.4426950408889634f / temperature;
  DFL_RET(launch_pdl(accept_sample_kernel, dim3(batch), dim3(kSampThreads), 0, s, draft, zt, zd, tst, dst, block, V, c,
                     u, v, len, anchor, n_pend, accept_len, stream, stream_len, stream_cap, status));
  count_launch();
  return cudaSuccess;
}

}  // namespace dfl
