// Device-driven miss staging.
//
// "Nanite for Experts" §5.4: expert tensors move as 256 KiB virtual tiles;
// persistent device page-table entries carry generations, so a slot whose
// tiles have not all landed is never read (§3.2 fail-closed). §3.4: the
// source is pinned host memory. "MawForge" §IV-C: a miss materialises the
// expert block into its slot.
//
// On GB300 the pinned store is reachable from the GPU over the coherent
// host link, so the copy is a kernel: after on-device admission wrote the
// fill list, a persistent grid walks the (fill, 32 KiB chunk) items; for
// each, a CTA issues all its 16-byte loads at once (eight per thread) and
// stores them; chunks never cross a matrix, and
// the 256 KiB tiles of each matrix remain the accounting unit. The CTA that
// lands a fill's last chunk publishes the slot's generation. No host round
// trip sits between routing and the FFN.
#include <algorithm>

#include "internal.h"
#include "pdl.cuh"

namespace moe {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 8;

// Streaming load of the store through its device alias (host memory).
__device__ __forceinline__ uint4 ld_host_stream(const uint4* p) { return __ldcs(p); }

// Persistent: CTA b copies work items b, b + gridDim.x, ... of the
// n_fills * chunks_per_expert items (item = fill * chunks_per_expert +
// chunk), so the launch does not depend on how many misses the step has.
__global__ void __launch_bounds__(kCopyThreads) stage_copy_kernel(StageArgs a) {
  pdl_wait();
  pdl_trigger();
  const int n = __ldcg(a.fills);
  const int cpe = a.chunks_per_expert;
  const int items = n * cpe;
  for (int w = blockIdx.x; w < items; w += gridDim.x) {
    const int f = w / cpe;
    const int e = __ldcg(a.fills + 1 + 2 * f);
    const int slot = __ldcg(a.fills + 2 + 2 * f);
    // chunk -> (matrix, offset); chunks never cross a matrix
    int j = w - f * cpe, m = 0;
    while (m < 2 && j >= a.chunks[m]) {
      j -= a.chunks[m];
      ++m;
    }
    const int64_t off = a.mat_off[m] + static_cast<int64_t>(j) * kStageChunkBytes;
    const int64_t len = min(kStageChunkBytes, a.mat_bytes[m] - static_cast<int64_t>(j) * kStageChunkBytes);
    const uint4* src = reinterpret_cast<const uint4*>(a.store + static_cast<int64_t>(e) * a.payload + off);
    uint4* dst = reinterpret_cast<uint4*>(a.pool + static_cast<int64_t>(slot) * a.slot_stride + off);
    const int nv = static_cast<int>(len / 16);
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int i = threadIdx.x + u * kCopyThreads;
      if (i < nv) v[u] = ld_host_stream(src + i);
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int i = threadIdx.x + u * kCopyThreads;
      if (i < nv) dst[i] = v[u];
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned prev = atomicAdd(a.done + f, 1u);
      if (prev + 1 == static_cast<unsigned>(cpe)) {
        // every chunk of this fill has landed: publish the slot's generation
        __threadfence();
        a.gen[slot] = __ldcg(a.sgen + slot);
        atomicAdd(reinterpret_cast<unsigned long long*>(a.stats + kStatTiles),
                  static_cast<unsigned long long>(a.tiles_per_expert));
        atomicAdd(reinterpret_cast<unsigned long long*>(a.stats + kStatBytes),
                  static_cast<unsigned long long>(a.payload));
      }
    }
  }
}

// One 4-byte load from every page of the bound store (the sum only keeps
// the loads alive): the device's first access to a page of host memory costs
// several times a later one, so binding takes that cost once, up front,
// instead of on a decode step's critical path.
__global__ void __launch_bounds__(256) touch_pages_kernel(const uint8_t* p, size_t n, size_t page, uint32_t* sink) {
  uint32_t acc = 0;
  const size_t step = static_cast<size_t>(gridDim.x) * blockDim.x * page;
  for (size_t i = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) * page; i < n; i += step)
    acc += __ldcv(reinterpret_cast<const uint32_t*>(p + i));
  if (acc == 0x9e3779b9u) *sink = acc;
}

// One 32-bit store, its value taken when the launch is enqueued (a copy
// from host memory would read the source only when it runs).
__global__ void set_word_kernel(uint32_t* dst, uint32_t v) { *dst = v; }

}  // namespace

cudaError_t launch_set_word(uint32_t* dst, uint32_t v, cudaStream_t st) {
  set_word_kernel<<<1, 1, 0, st>>>(dst, v);
  return cudaGetLastError();
}

cudaError_t launch_touch_pages(const uint8_t* dev_store, size_t bytes, int sms, uint32_t* sink, cudaStream_t st) {
  if (bytes < 4) return cudaSuccess;
  touch_pages_kernel<<<std::max(1, sms) * 8, 256, 0, st>>>(dev_store, bytes - 3, kTouchPage, sink);
  return cudaGetLastError();
}

cudaError_t launch_stage_copy(const StageArgs& a, cudaStream_t st) {
  if (a.max_fills <= 0) return cudaSuccess;
  static_assert(kStageChunkBytes == 16 * kCopyThreads * kCopyUnroll, "one chunk per CTA");
  const int grid = std::max(1, std::min(a.grid, a.chunks_per_expert * a.max_fills));
  const cudaError_t e = pdl_launch(stage_copy_kernel, dim3(grid), dim3(kCopyThreads), 0, st, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
