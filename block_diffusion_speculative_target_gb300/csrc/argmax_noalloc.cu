// Greedy argmax + top-2 gap without a workspace: the same sliced vocabulary
// kernel as dflash_argmax, with its slice partials and per-row tickets held in
// a fixed file-scope device array instead of caller-allocated scratch.  The
// library calls no allocator on this path (no cudaMalloc/cudaFree, no
// allocating library routine).
#include "common.cuh"
#include "internal.h"

#include <atomic>
#include <mutex>

namespace {

constexpr int kMaxRows = DFLASH_ARGMAX_NOALLOC_MAX_ROWS;
constexpr int kMaxDevices = 64;

// Scratch of the sliced argmax for up to kMaxRows rows: 128 x 16 x 16 B of
// slice partials (32 KiB) and 128 tickets.  One copy per device (per context).
static __device__ __align__(256) float4 g_part[kMaxRows * dfl::kArgmaxSlices];
static __device__ __align__(256) int g_tickets[kMaxRows];

struct Slot {
  std::atomic<bool> ready{false};
  std::atomic<unsigned long long> ctx_id{0};  // unique id of the context the addresses belong to
  float4* part = nullptr;
  int* tickets = nullptr;
};
Slot g_slot[kMaxDevices];
std::mutex g_setup_mu;

typedef CUresult (*PFN_ctxGetCurrent_t)(CUcontext*);
typedef CUresult (*PFN_ctxGetId_t)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (0 when there is none or
// the driver cannot tell).  A device reset ends the context; the next one gets
// a new id, so addresses looked up in the old one are never reused.
unsigned long long current_ctx_id() {
  static PFN_ctxGetCurrent_t get_cur = nullptr;
  static PFN_ctxGetId_t get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PFN_ctxGetCurrent_t>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_ctxGetId_t>(p);
  });
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (!get_cur || !get_id || get_cur(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Resolves the device addresses of the scratch arrays in the current context
// of device `dev`: once per context (again after the context changes, e.g.
// after cudaDeviceReset); a failed lookup is not cached, so the next call
// retries.
cudaError_t scratch_of(int dev, dfl::ArgmaxScratch* out) {
  Slot& s = g_slot[dev];
  const unsigned long long id = current_ctx_id();
  if (!s.ready.load(std::memory_order_acquire) || id == 0 || s.ctx_id.load(std::memory_order_acquire) != id) {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!s.ready.load(std::memory_order_relaxed) || id == 0 || s.ctx_id.load(std::memory_order_relaxed) != id) {
      s.ready.store(false, std::memory_order_relaxed);
      void* p = nullptr;
      void* t = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&p, g_part);
      if (e != cudaSuccess) return e;
      e = cudaGetSymbolAddress(&t, g_tickets);
      if (e != cudaSuccess) return e;
      s.part = static_cast<float4*>(p);
      s.tickets = static_cast<int*>(t);
      s.ctx_id.store(id, std::memory_order_release);
      s.ready.store(true, std::memory_order_release);
    }
  }
  out->part = s.part;
  out->tickets = s.tickets;
  out->max_rows = kMaxRows;
  return cudaSuccess;
}

}  // namespace

extern "C" int dflash_argmax_noalloc(const float* logits, int32_t rows, int32_t V, int32_t* argmax, float* gap,
                                     int32_t* status, dflash_stream_t stream) {
  if (!logits || !argmax || rows <= 0 || V <= 0) return DFLASH_ERR_INVALID_ARG;
  if (rows > kMaxRows) return DFLASH_ERR_TOO_LARGE;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return dfl::record_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return DFLASH_ERR_INVALID_ARG;  // more devices than the table holds
  dfl::ArgmaxScratch sc;
  e = scratch_of(dev, &sc);
  if (e != cudaSuccess) return dfl::record_cuda_error(e);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // tickets count the finished slices of a row and must start at zero
  e = cudaMemsetAsync(sc.tickets, 0, sizeof(int) * (size_t)rows, s);
  if (e != cudaSuccess) return dfl::record_cuda_error(e);
  e = dfl::argmax(logits, rows, V, argmax, gap, 0, sc, reinterpret_cast<int*>(status), s);
  if (e != cudaSuccess) return dfl::record_cuda_error(e);
  return DFLASH_OK;
}
