// Gather + pool: pooled[b][t][:] = sum (or mean) of the rows looked up by bag b*T+t.
//
// Merlin Distributed Embeddings article, "Background", and HugeCTR interview, section 2:
// the lookup is bound by memory bandwidth, so the kernel is built around the row loads.
// A group of G lanes owns one bag; lane j of the group loads 16-byte chunks j, j+G, ... of
// each row (fp32: 4 elements per chunk, bf16: 8), so one row is a handful of fully
// coalesced 128-bit loads.  Row numbers of four lookups are fetched first and their rows
// loaded back to back, so several loads are in flight per lane.  Accumulation is fp32;
// mean pooling divides the sum by the bag length L (rejected IDs count in L and add 0).
#include "emb_internal.cuh"

namespace emb {

constexpr int kMaxChunksPerLane = 4;  // D*esize <= 2 KB

template <bool BF16>
__device__ __forceinline__ void accumulate_chunk(const void* table, uint32_t row, int D, int q,
                                                 float4* acc2) {
  if (BF16) {
    const __nv_bfloat16* r = reinterpret_cast<const __nv_bfloat16*>(table) + (int64_t)row * D;
    float4 lo, hi;
    ld_row8_bf16(r, q, lo, hi);
    acc2[0] = f4_add(acc2[0], lo);
    acc2[1] = f4_add(acc2[1], hi);
  } else {
    const float* r = reinterpret_cast<const float*>(table) + (int64_t)row * D;
    acc2[0] = f4_add(acc2[0], ld_row4_f32(r, q));
  }
}

template <bool BF16>
__global__ void __launch_bounds__(256) k_pool(Params p, int64_t nbags, int one_hot, int G,
                                              float* pooled) {
  constexpr int EPC = BF16 ? 8 : 4;       // elements per 16-byte chunk
  constexpr int F4 = EPC / 4;             // float4 accumulators per chunk
  const int D = p.D;
  const int chunks = D / EPC;
  const int lane = threadIdx.x & 31;
  const int sub = lane % G;               // lane within the group
  const int groups_per_warp = 32 / G;
  const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t b0 = gwarp * groups_per_warp; b0 < nbags; b0 += nwarps * groups_per_warp) {
    const int64_t bag = b0 + lane / G;
    if (bag >= nbags) continue;
    int64_t beg, end;
    if (one_hot) {
      beg = bag;
      end = bag + 1;
    } else {
      beg = p.offs[bag];
      end = p.offs[bag + 1];
      if (beg < 0 || end < beg || end > p.nnz) end = beg = 0;  // flagged by the bag expansion
    }
    float4 acc[kMaxChunksPerLane * F4];
#pragma unroll
    for (int k = 0; k < kMaxChunksPerLane * F4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    int64_t i = beg;
    for (; i + 4 <= end; i += 4) {
      uint32_t r[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) r[u] = p.row_of[i + u];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (r[u] == kNoRow) continue;
#pragma unroll
        for (int k = 0; k < kMaxChunksPerLane; ++k) {
          const int q = sub + k * G;
          if (q < chunks) accumulate_chunk<BF16>(p.table, r[u], D, q, acc + k * F4);
        }
      }
    }
    for (; i < end; ++i) {
      const uint32_t r = p.row_of[i];
      if (r == kNoRow) continue;
#pragma unroll
      for (int k = 0; k < kMaxChunksPerLane; ++k) {
        const int q = sub + k * G;
        if (q < chunks) accumulate_chunk<BF16>(p.table, r, D, q, acc + k * F4);
      }
    }
    const float L = (float)(end - beg);
    float4* out = reinterpret_cast<float4*>(pooled + bag * D);
#pragma unroll
    for (int k = 0; k < kMaxChunksPerLane; ++k) {
      const int q = sub + k * G;
      if (q >= chunks) continue;
#pragma unroll
      for (int f = 0; f < F4; ++f) {
        float4 v = acc[k * F4 + f];
        if (p.mean && L > 0.f) v = f4_div(v, L);
        out[q * F4 + f] = v;
      }
    }
  }
}

cudaError_t launch_pool(Ctx* c, int64_t batch, float* pooled, cudaStream_t s) {
  const Params& p = c->p;
  const int64_t nbags = batch * p.T;
  const int chunks = p.D * (p.bf16 ? 2 : 4) / 16;
  int G = 1;
  while (G < chunks && G < 32) G <<= 1;
  const int64_t warps = (nbags + (32 / G) - 1) / (32 / G);
  LaunchScope ls(c, K_POOL, s);
  const int grid = grid_for(c, warps * 32, 256, 8);
  if (p.bf16)
    k_pool<true><<<grid, 256, 0, s>>>(p, nbags, c->multi_hot ? 0 : 1, G, pooled);
  else
    k_pool<false><<<grid, 256, 0, s>>>(p, nbags, c->multi_hot ? 0 : 1, G, pooled);
  return cudaGetLastError();
}

}  // namespace emb
