// Gather + pool: pooled[b][t][:] = sum (or mean) of the rows looked up by bag b*T+t.
//
// Merlin Distributed Embeddings article, "Background", and HugeCTR interview, section 2:
// the lookup is bound by memory bandwidth, so the kernel is built around the row loads.
// A group of G lanes owns a bag; lane j of the group loads 16-byte chunks j, j+G, ... of
// each row (fp32: 4 elements per chunk, bf16: 8), so one row is a handful of fully
// coalesced 128-bit loads.  Eight rows are in flight per group: a multi-hot bag loads its
// row numbers eight at a time, one block ahead, and its rows back to back; with one ID per
// bag a group takes eight bags at once.  Accumulation is fp32 in lookup order; mean pooling
// divides the sum by the bag length L (rejected IDs count in L and add 0).
#include "emb_internal.cuh"

namespace emb {

constexpr int kMaxChunksPerLane = 4;  // D*esize <= 2 KB

constexpr int kPoolRows = 8;  // rows in flight per lane group

// 16 raw bytes of a row (chunk q), and their fp32 sum into acc (F4 float4s)
template <bool BF16>
__device__ __forceinline__ uint4 ld_chunk(const void* table, uint32_t row, int D, int q) {
  const int64_t base = (int64_t)row * D * (BF16 ? 2 : 4);
  return __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(table) + base) + q);
}
template <bool BF16>
__device__ __forceinline__ void add_chunk(uint4 raw, float4* acc) {
  if (BF16) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
    const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.z));
    const float2 d = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.w));
    acc[0] = f4_add(acc[0], make_float4(a.x, a.y, b.x, b.y));
    acc[1] = f4_add(acc[1], make_float4(c.x, c.y, d.x, d.y));
  } else {
    acc[0] = f4_add(acc[0], make_float4(__uint_as_float(raw.x), __uint_as_float(raw.y),
                                        __uint_as_float(raw.z), __uint_as_float(raw.w)));
  }
}

// CPL: 16-byte chunks of a row per lane (1 when a row has at most 32 chunks)
template <bool BF16, int CPL>
__global__ void __launch_bounds__(256) k_pool(Params p, int64_t nbags, int one_hot, int G,
                                              float* pooled) {
  constexpr int EPC = BF16 ? 8 : 4;       // elements per 16-byte chunk
  constexpr int F4 = EPC / 4;             // float4 accumulators per chunk
  constexpr int R = kPoolRows;
  const int D = p.D;
  const int chunks = D / EPC;
  const int lane = threadIdx.x & 31;
  const int sub = lane % G;               // lane within the group
  const int gpw = 32 / G;                 // groups per warp
  const int per = one_hot ? R : 1;        // bags per group per iteration
  const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  auto store = [&](int64_t bag, const float4* acc, float L) {
    float4* out = reinterpret_cast<float4*>(pooled + bag * D);
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
      const int q = sub + k * G;
      if (q >= chunks) continue;
#pragma unroll
      for (int f = 0; f < F4; ++f) {
        float4 v = acc[k * F4 + f];
        if (p.mean && L > 0.f) v = f4_div(v, L);
        out[q * F4 + f] = v;
      }
    }
  };
  for (int64_t b0 = gwarp * gpw * per; b0 < nbags; b0 += nwarps * gpw * per) {
    const int64_t g0 = b0 + (int64_t)(lane / G) * per;  // this group's first bag
    if (g0 >= nbags) continue;
    if (one_hot) {
      // R bags of one lookup each: row numbers, then the rows, then the outputs
      uint32_t r[R];
#pragma unroll
      for (int u = 0; u < R; ++u) r[u] = g0 + u < nbags ? p.row_of[g0 + u] : kNoRow;
      uint4 raw[R][CPL];
#pragma unroll
      for (int u = 0; u < R; ++u)
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
          const int q = sub + k * G;
          raw[u][k] = (r[u] != kNoRow && q < chunks) ? ld_chunk<BF16>(p.table, r[u], D, q)
                                                     : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
      for (int u = 0; u < R; ++u) {
        if (g0 + u >= nbags) break;
        float4 acc[CPL * F4];
#pragma unroll
        for (int e = 0; e < CPL * F4; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < CPL; ++k) add_chunk<BF16>(raw[u][k], acc + k * F4);
        store(g0 + u, acc, 1.f);
      }
      continue;
    }
    const int64_t bag = g0;
    int64_t beg = p.offs[bag], end = p.offs[bag + 1];
    if (beg < 0 || end < beg || end > p.nnz) end = beg = 0;  // flagged by the bag expansion
    float4 acc[CPL * F4];
#pragma unroll
    for (int e = 0; e < CPL * F4; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    uint32_t rn[R];  // row numbers of the next block
#pragma unroll
    for (int u = 0; u < R; ++u) rn[u] = beg + u < end ? p.row_of[beg + u] : kNoRow;
    for (int64_t i = beg; i < end; i += R) {
      uint32_t r[R];
#pragma unroll
      for (int u = 0; u < R; ++u) {
        r[u] = rn[u];
        rn[u] = i + R + u < end ? p.row_of[i + R + u] : kNoRow;
      }
      uint4 raw[R][CPL];
#pragma unroll
      for (int u = 0; u < R; ++u)
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
          const int q = sub + k * G;
          raw[u][k] = (r[u] != kNoRow && q < chunks) ? ld_chunk<BF16>(p.table, r[u], D, q)
                                                     : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
      for (int u = 0; u < R; ++u) {
        if (r[u] == kNoRow) continue;  // rejected ID or past the bag's end: adds nothing
#pragma unroll
        for (int k = 0; k < CPL; ++k) add_chunk<BF16>(raw[u][k], acc + k * F4);
      }
    }
    store(bag, acc, (float)(end - beg));
  }
}

cudaError_t launch_pool(Ctx* c, int64_t batch, float* pooled, cudaStream_t s) {
  const Params& p = c->p;
  const int64_t nbags = batch * p.T;
  const int chunks = p.D * (p.bf16 ? 2 : 4) / 16;
  int G = 1;
  while (G < chunks && G < 32) G <<= 1;
  const int one_hot = c->multi_hot ? 0 : 1;
  const int64_t groups = one_hot ? (nbags + kPoolRows - 1) / kPoolRows : nbags;
  const int64_t warps = (groups + (32 / G) - 1) / (32 / G);
  LaunchScope ls(c, K_POOL, s);
  const int grid = grid_for(c, warps * 32, 256, 8);
  const bool one = chunks <= 32;  // one chunk per lane
  if (p.bf16)
    one ? k_pool<true, 1><<<grid, 256, 0, s>>>(p, nbags, one_hot, G, pooled)
        : k_pool<true, kMaxChunksPerLane><<<grid, 256, 0, s>>>(p, nbags, one_hot, G, pooled);
  else
    one ? k_pool<false, 1><<<grid, 256, 0, s>>>(p, nbags, one_hot, G, pooled)
        : k_pool<false, kMaxChunksPerLane><<<grid, 256, 0, s>>>(p, nbags, one_hot, G, pooled);
  return cudaGetLastError();
}

}  // namespace emb
