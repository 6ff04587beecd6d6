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
  float4* part = nullptr;
  int* tickets = nullptr;
};
Slot g_slot[kMaxDevices];
std::mutex g_setup_mu;

// Resolves the device addresses of the scratch arrays on the current device,
// once per device; a failed lookup is not cached, so the next call retries.
cudaError_t scratch_of(int dev, dfl::ArgmaxScratch* out) {
  Slot& s = g_slot[dev];
  if (!s.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!s.ready.load(std::memory_order_relaxed)) {
      void* p = nullptr;
      void* t = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&p, g_part);
      if (e != cudaSuccess) return e;
      e = cudaGetSymbolAddress(&t, g_tickets);
      if (e != cudaSuccess) return e;
      s.part = static_cast<float4*>(p);
      s.tickets = static_cast<int*>(t);
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
  if (dev < 0 || dev >= kMaxDevices) return DFLASH_ERR_TOO_LARGE;
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
