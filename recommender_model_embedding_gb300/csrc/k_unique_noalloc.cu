// Unique keys of one batch without any device allocation.
//
// Some callers cannot allocate device memory at the point where they need this: serving
// processes that pin their whole memory budget up front and forbid allocation on the
// request path, and plug-ins that are handed only their input and output buffers.  For them this entry point keeps its scratch -- an open-addressing hash
// set -- in a fixed-size array that is part of the library's device image, so a call
// touches only that array and the caller's buffers.
//
// The array holds kNoAllocSlots keys (8 bytes each) and their unique indices (4 bytes),
// 12 MiB in total, and every GPU that loads the library keeps it until the process exits.
// It is shared by all calls: each call first resets it, so two calls that overlap on the
// GPU (on different streams, or from different host threads) race and give wrong results.
#include <mutex>

#include "emb_internal.cuh"

namespace emb {
namespace {

constexpr int64_t kNoAllocMaxKeys = EMB_NOALLOC_MAX_KEYS;  // largest n accepted
constexpr uint32_t kNoAllocSlots = 1u << 20;               // >= 2 * kNoAllocMaxKeys
constexpr int kMaxDevices = 64;
static_assert(kNoAllocSlots >= 2 * kNoAllocMaxKeys, "set must stay at most half full");

struct NoAllocScratch {
  unsigned long long keys[kNoAllocSlots];  // all-ones = free
  uint32_t vals[kNoAllocSlots];            // unique index of each occupied slot
  uint32_t count;                          // unique keys so far
};

// File-scope scratch: in host code `g_noalloc` is only a handle, never a device address;
// the device address comes from cudaGetSymbolAddress (below).
static __device__ __align__(256) NoAllocScratch g_noalloc;

std::mutex g_mu;
NoAllocScratch* g_dev_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
cudaError_t scratch_address(NoAllocScratch** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_dev_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc);
    if (e != cudaSuccess) return e;
    g_dev_ptr[dev] = reinterpret_cast<NoAllocScratch*>(p);
  }
  *out = g_dev_ptr[dev];
  return cudaSuccess;
}

__global__ void k_na_clear(NoAllocScratch* sc) {
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < kNoAllocSlots;
       i += gridDim.x * blockDim.x)
    sc->keys[i] = ~0ull;
  if (blockIdx.x == 0 && threadIdx.x == 0) sc->count = 0;
}

// Insert every key; the lane whose CAS claims a slot numbers the key (one atomicAdd per
// block) and writes it to `uniq`.  `inverse` temporarily holds each key's slot (or -1).
__global__ void __launch_bounds__(256) k_na_insert(NoAllocScratch* sc, const int64_t* keys,
                                                   int64_t n, int64_t* uniq, int32_t* inverse) {
  __shared__ uint32_t warp_base[8];
  __shared__ uint32_t block_base;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x; i0 < n; i0 += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = i0 + threadIdx.x;
    bool won = false;
    int32_t slot = -1;
    int64_t key = -1;
    if (i < n) {
      key = keys[i];
      if (key >= 0) {
        uint32_t h = (uint32_t)mix64((uint64_t)key) & (kNoAllocSlots - 1);
        for (uint32_t probe = 0; probe < kNoAllocSlots; ++probe) {
          const unsigned long long k = reinterpret_cast<volatile unsigned long long*>(sc->keys)[h];
          if (k == (unsigned long long)key) {
            slot = (int32_t)h;
            break;
          }
          if (k == ~0ull) {
            const unsigned long long prev = atomicCAS(sc->keys + h, ~0ull, (unsigned long long)key);
            if (prev == ~0ull || prev == (unsigned long long)key) {
              won = prev == ~0ull;
              slot = (int32_t)h;
              break;
            }
          }
          h = (h + 1) & (kNoAllocSlots - 1);
        }
      }
      inverse[i] = slot;
    }
    const unsigned ball = __ballot_sync(0xFFFFFFFFu, won);
    if (lane == 0) warp_base[wid] = __popc(ball);
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t tot = 0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
        const uint32_t c = warp_base[w];
        warp_base[w] = tot;
        tot += c;
      }
      block_base = tot ? atomicAdd(&sc->count, tot) : 0u;
    }
    __syncthreads();
    if (won) {
      const uint32_t u = block_base + warp_base[wid] + __popc(ball & ((1u << lane) - 1u));
      sc->vals[slot] = u;
      uniq[u] = key;
    }
    __syncthreads();
  }
}

__global__ void k_na_finish(const NoAllocScratch* sc, int64_t n, int32_t* inverse,
                            int32_t* num_unique) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t slot = inverse[i];
    inverse[i] = slot >= 0 ? (int32_t)sc->vals[slot] : -1;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *num_unique = (int32_t)sc->count;
}

}  // namespace
}  // namespace emb

using namespace emb;

extern "C" emb_status emb_unique_keys_noalloc(const int64_t* d_keys, int64_t n, int64_t* d_unique,
                                              int32_t* d_inverse, int32_t* d_num_unique,
                                              void* stream) {
  if (n < 0 || n > kNoAllocMaxKeys || !d_num_unique) return EMB_EINVAL;
  if (n > 0 && (!d_keys || !d_unique || !d_inverse)) return EMB_EINVAL;
  NoAllocScratch* sc = nullptr;
  cudaError_t e = scratch_address(&sc);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return EMB_ECUDA;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  k_na_clear<<<256, 256, 0, s>>>(sc);
  if (n > 0) {
    const int grid = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
    k_na_insert<<<grid, 256, 0, s>>>(sc, d_keys, n, d_unique, d_inverse);
  }
  k_na_finish<<<n > 0 ? (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024) : 1, 256, 0, s>>>(
      sc, n, d_inverse, d_num_unique);
  e = cudaGetLastError();
  return e == cudaSuccess ? EMB_OK : EMB_ECUDA;
}
