// Backward: group the batch's lookups by unique row, reduce their gradients and apply
// sparse Adagrad to the touched rows only.
//
// Merlin Distributed Embeddings article, "synthetic model benchmark": the embeddings are
// trained with Adagrad; HugeCTR interview, section 3 (1): an efficient sparse optimiser
// implemented in a memory-saving way.  Update per touched row (per element):
//   acc += g*g;  w -= lr * g / (sqrt(acc) + eps)
// or row-wise (one accumulator per row):  acc += mean_j g_j^2;  w_j -= lr*g_j/(sqrt(acc)+eps).
// g is the sum of the gradients of all lookups of the row in the batch (times 1/L under
// mean pooling), so a row looked up k times takes one step, not k.
//
// Two gradient paths:
//  * from d_pooled (emb_backward_adagrad): counting sort of the lookups by unique row
//    (occurrence counts -> exclusive scan -> positions), then fixed chunks of kChunk
//    sorted positions per lane group.  A row whose lookups all fall inside one chunk is
//    reduced and updated by that group directly; a row cut by a chunk boundary (a hot row)
//    adds its partial sums into g[u] with vector reductions and is updated afterwards by
//    k_adagrad_from_g.  Every group does the same bounded amount of work however skewed
//    the ID distribution is.
//  * from the fused interaction backward, which has already added every row gradient into
//    g[u]: k_adagrad_from_g updates all U rows.
// k_adagrad_from_g also zeroes g[u] and frees the row's dedup-set slot, leaving both clean
// for the next batch.
#include "emb_internal.cuh"

namespace emb {

constexpr int kChunk = 32;  // sorted positions per lane group

// Lanes per row: a power of two such that each lane holds at most 4 chunks of 4 elements
// (D = 128 -> 8 lanes, 4 rows per warp).  Few lanes per row and several chunks per lane
// keep many independent row loads in flight per warp.
static int lanes_per_row(int D) {
  const int need = (D / 4 + 3) / 4;
  int G = 1;
  while (G < need && G < 32) G <<= 1;
  return G;
}

__device__ __forceinline__ float group_sum(float v, int G) {
  for (int o = G >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

template <bool BF16>
__device__ __forceinline__ float4 load_w4(const Params& p, uint32_t row, int kc) {
  const int64_t off = (int64_t)row * p.D + 4 * kc;
  if (BF16) {
    const uint2 raw = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(p.table) + off);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
  return *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.table) + off);
}

template <bool BF16>
__device__ __forceinline__ void store_w4(const Params& p, uint32_t row, int kc, float4 w) {
  const int64_t off = (int64_t)row * p.D + 4 * kc;
  if (BF16) {
    uint2 raw;
    *reinterpret_cast<__nv_bfloat162*>(&raw.x) = __floats2bfloat162_rn(w.x, w.y);
    *reinterpret_cast<__nv_bfloat162*>(&raw.y) = __floats2bfloat162_rn(w.z, w.w);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.table) + off) = raw;
  } else {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.table) + off) = w;
  }
}

__device__ __forceinline__ float adagrad_step(float w, float g, float denom, float lr) {
  return w - lr * g / denom;
}

// Adagrad on one row held by a group of G lanes; lane `sub` holds chunks sub, sub+G, ...
// in gk[] (up to 4 chunks).  Every load of the row (parameters and accumulators) is issued
// before any arithmetic, so one row costs one memory round trip.  All lanes of the warp
// must call this together (the row-wise variant reduces across the group).
template <bool BF16>
__device__ __forceinline__ void adagrad_row(const Params& p, uint32_t row, int sub, int G,
                                            const float4* gk, bool active) {
  const int KC = p.D / 4;
  float4 w[4], a[4];
  float ar = 0.f;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int kc = sub + m * G;
    if (active && kc < KC) {
      w[m] = load_w4<BF16>(p, row, kc);
      if (!p.rowwise) a[m] = reinterpret_cast<const float4*>(p.acc + (int64_t)row * p.D)[kc];
    }
  }
  if (p.rowwise) {
    if (active) ar = p.acc[row];
    float sq = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int kc = sub + m * G;
      if (active && kc < KC)
        sq += gk[m].x * gk[m].x + gk[m].y * gk[m].y + gk[m].z * gk[m].z + gk[m].w * gk[m].w;
    }
    sq = group_sum(sq, G);
    if (!active) return;
    ar += sq / (float)p.D;
    const float d = sqrtf(ar) + p.eps;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int kc = sub + m * G;
      if (kc >= KC) continue;
      const float4 g = gk[m];
      store_w4<BF16>(p, row, kc,
                     make_float4(adagrad_step(w[m].x, g.x, d, p.lr), adagrad_step(w[m].y, g.y, d, p.lr),
                                 adagrad_step(w[m].z, g.z, d, p.lr), adagrad_step(w[m].w, g.w, d, p.lr)));
    }
    if (sub == 0) p.acc[row] = ar;
    return;
  }
  if (!active) return;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int kc = sub + m * G;
    if (kc >= KC) continue;
    const float4 g = gk[m];
    float4 aa = a[m];
    aa.x += g.x * g.x;
    aa.y += g.y * g.y;
    aa.z += g.z * g.z;
    aa.w += g.w * g.w;
    reinterpret_cast<float4*>(p.acc + (int64_t)row * p.D)[kc] = aa;
    store_w4<BF16>(p, row, kc,
                   make_float4(adagrad_step(w[m].x, g.x, sqrtf(aa.x) + p.eps, p.lr),
                               adagrad_step(w[m].y, g.y, sqrtf(aa.y) + p.eps, p.lr),
                               adagrad_step(w[m].z, g.z, sqrtf(aa.z) + p.eps, p.lr),
                               adagrad_step(w[m].w, g.w, sqrtf(aa.w) + p.eps, p.lr)));
  }
}

// ------------------------------------------------------------------ counting sort

// unique index of each lookup and its rank among the lookups of that row
__global__ void k_inverse_count(Params p, int64_t nnz) {
  for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < nnz;
       q += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t sl = p.slot_of[q];
    uint32_t u = kNoRow;
    if (p.row_of[q] != kNoRow && sl != kEmpty32) {
      u = p.set_vals[sl];
      p.rank[q] = atomicAdd(p.cnt + u, 1u);
    }
    p.inv[q] = u;
  }
}

constexpr int kScanThreads = 256, kScanItems = 8, kScanTile = kScanThreads * kScanItems;

__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_tot,
                                                         uint32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t x = v;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[wid] = x;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t run = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
      const uint32_t t = warp_tot[w];
      warp_tot[w] = run;
      run += t;
    }
    *total = run;
  }
  __syncthreads();
  const uint32_t r = warp_tot[wid] + x - v;
  __syncthreads();
  return r;
}

// seg[i] = exclusive prefix of cnt within the tile; scan_tmp[tile] = tile total.
// Items i < U+1 take cnt[i] (cnt[U] is 0), so seg[U] ends up as the number of lookups.
__global__ void __launch_bounds__(kScanThreads) k_scan_local(Params p) {
  __shared__ uint32_t warp_tot[kScanThreads / 32];
  __shared__ uint32_t total;
  const int64_t n = (int64_t)p.counters[kU] + 1;
  const int64_t base = (int64_t)blockIdx.x * kScanTile + (int64_t)threadIdx.x * kScanItems;
  if ((int64_t)blockIdx.x * kScanTile >= n) {
    if (threadIdx.x == 0) p.scan_tmp[blockIdx.x] = 0;
    return;
  }
  uint32_t v[kScanItems];
  uint32_t sum = 0;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    v[k] = (base + k < n - 1) ? p.cnt[base + k] : 0u;
    sum += v[k];
  }
  uint32_t run = block_exclusive_scan(sum, warp_tot, &total);
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    if (base + k < n) p.seg[base + k] = run;
    run += v[k];
  }
  if (threadIdx.x == 0) p.scan_tmp[blockIdx.x] = total;
}

// exclusive scan of the tile totals, one block
__global__ void __launch_bounds__(1024) k_scan_blocks(Params p, int64_t ntiles) {
  __shared__ uint32_t warp_tot[32];
  __shared__ uint32_t total;
  const int64_t per = (ntiles + blockDim.x - 1) / blockDim.x;
  const int64_t b0 = (int64_t)threadIdx.x * per;
  uint32_t sum = 0;
  for (int64_t k = 0; k < per; ++k)
    if (b0 + k < ntiles) sum += p.scan_tmp[b0 + k];
  uint32_t run = block_exclusive_scan(sum, warp_tot, &total);
  for (int64_t k = 0; k < per; ++k) {
    if (b0 + k < ntiles) {
      const uint32_t t = p.scan_tmp[b0 + k];
      p.scan_tmp[b0 + k] = run;
      run += t;
    }
  }
}

__global__ void k_scan_add(Params p) {
  const int64_t n = (int64_t)p.counters[kU] + 1;
  const int64_t i = (int64_t)blockIdx.x * kScanTile + threadIdx.x;
  if ((int64_t)blockIdx.x * kScanTile >= n) return;
  const uint32_t add = p.scan_tmp[blockIdx.x];
  for (int64_t k = i; k < (int64_t)(blockIdx.x + 1) * kScanTile && k < n; k += blockDim.x)
    p.seg[k] += add;
}

__global__ void k_fill_perm(Params p, int64_t nnz) {
  for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < nnz;
       q += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t u = p.inv[q];
    if (u != kNoRow) p.perm[p.seg[u] + p.rank[q]] = (uint32_t)q;
  }
}

// ------------------------------------------------------------------ reduce + update

template <bool BF16>
__global__ void __launch_bounds__(256) k_segreduce_adagrad(Params p, const float* dpooled,
                                                           int one_hot, int G) {
  const int lane = threadIdx.x & 31;
  const int sub = lane % G;
  const int gpw = 32 / G;
  const int KC = p.D / 4;
  const uint32_t U = p.counters[kU];
  const int64_t NV = p.seg[U];
  const int64_t nchunks = (NV + kChunk - 1) / kChunk;
  const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t c0 = gwarp * gpw; c0 < nchunks; c0 += nwarps * gpw) {
    const int64_t c = c0 + lane / G;
    const bool live = c < nchunks;
    const int64_t p0 = live ? c * kChunk : 0;
    const int64_t p1 = live ? ((p0 + kChunk < NV) ? p0 + kChunk : NV) : 0;
    // every group walks kChunk steps so that the row-wise reduction stays warp-uniform
    float4 acc[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    int64_t run_start = p0;
    uint32_t cur = live && p0 < p1 ? p.inv[p.perm[p0]] : kNoRow;
    for (int step = 0; step <= kChunk; ++step) {
      const int64_t pos = p0 + step;
      const bool have = live && pos < p1;
      uint32_t q = 0, u = kNoRow;
      if (have) {
        q = p.perm[pos];
        u = p.inv[q];
      }
      // flush the run of `cur` when the row changes or the chunk ends
      const bool flush = live && cur != kNoRow && (!have || u != cur);
      const bool whole = flush && run_start == (int64_t)p.seg[cur] && pos == (int64_t)p.seg[cur + 1];
      // groups that finish a whole segment apply Adagrad (all lanes of the warp take part)
      const bool any_whole = __any_sync(0xFFFFFFFFu, whole);
      if (any_whole) adagrad_row<BF16>(p, whole ? p.uniq_row[cur] : 0u, sub, G, acc, whole);
      if (flush && !whole) {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int kc = sub + m * G;
          if (kc < KC) red_add_f4(p.g + (int64_t)cur * p.D + 4 * kc, acc[m]);
        }
      }
      if (flush) {
#pragma unroll
        for (int m = 0; m < 4; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        cur = u;
        run_start = pos;
      }
      if (have) {
        const uint32_t bag = one_hot ? q : p.bag_of[q];
        float scale = 1.f;
        if (p.mean && !one_hot) {
          const int32_t L = p.offs[bag + 1] - p.offs[bag];
          scale = 1.f / (float)L;
        }
        const float4* src = reinterpret_cast<const float4*>(dpooled + (int64_t)bag * p.D);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int kc = sub + m * G;
          if (kc < KC) {
            const float4 v = __ldg(src + kc);
            acc[m].x = fmaf(scale, v.x, acc[m].x);
            acc[m].y = fmaf(scale, v.y, acc[m].y);
            acc[m].z = fmaf(scale, v.z, acc[m].z);
            acc[m].w = fmaf(scale, v.w, acc[m].w);
          }
        }
        if (cur == kNoRow) {
          cur = u;
          run_start = pos;
        }
      }
    }
  }
}

// Update rows from g[u] (all rows, or only rows cut by a chunk boundary), zero g[u] and
// free the dedup-set slot of every unique row.
template <bool BF16>
__global__ void __launch_bounds__(256) k_adagrad_from_g(Params p, int split_only, int G) {
  const int lane = threadIdx.x & 31;
  const int sub = lane % G;
  const int gpw = 32 / G;
  const int KC = p.D / 4;
  const uint32_t U = p.counters[kU];
  const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t stride = nwarps * gpw;
  int64_t u = gwarp * gpw + lane / G;
  // Everything that decides an address or a predicate of the next iteration (its row, its
  // dedup-set slot, whether its segment was split) is loaded one iteration ahead: with
  // in-order issue, an instruction waiting on a fresh load would hold back the row loads
  // behind it for a whole memory round trip.
  uint32_t row = 0u, slot = 0u;
  bool split = true;
  if (u < U) {
    row = p.uniq_row[u];
    slot = p.uniq_slot[u];
    if (split_only) split = (p.seg[u] / kChunk) != ((p.seg[u + 1] - 1) / kChunk);
  }
  for (int64_t u0 = gwarp * gpw; u0 < U; u0 += stride, u += stride) {
    const bool live = u < U;
    const bool active = live && split;
    const uint32_t row_now = row, slot_now = slot;
    const int64_t un = u + stride;
    if (un < U) {
      row = p.uniq_row[un];
      slot = p.uniq_slot[un];
      if (split_only) split = (p.seg[un] / kChunk) != ((p.seg[un + 1] - 1) / kChunk);
    }
    float4 gk[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int kc = sub + m * G;
      gk[m] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (active && kc < KC) gk[m] = reinterpret_cast<const float4*>(p.g + u * p.D)[kc];
    }
    adagrad_row<BF16>(p, row_now, sub, G, gk, active);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int kc = sub + m * G;
      if (active && kc < KC)
        reinterpret_cast<float4*>(p.g + u * p.D)[kc] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (live && sub == 0) p.set_keys[slot_now] = kEmpty32;
  }
}

cudaError_t launch_backward_csr(Ctx* c, const float* dpooled, int64_t batch, int64_t nnz,
                                cudaStream_t s) {
  const Params& p = c->p;
  cudaError_t e = cudaMemsetAsync(p.cnt, 0, sizeof(uint32_t) * (size_t)(nnz + 1), s);
  if (e != cudaSuccess) return e;
  if (nnz > 0) {
    LaunchScope ls(c, K_INVERSE_COUNT, s);
    k_inverse_count<<<grid_for(c, nnz, 256), 256, 0, s>>>(p, nnz);
  }
  const int64_t ntiles = (nnz + 1 + kScanTile - 1) / kScanTile;
  {
    LaunchScope ls(c, K_SCAN_LOCAL, s);
    k_scan_local<<<(unsigned)ntiles, kScanThreads, 0, s>>>(p);
  }
  {
    LaunchScope ls(c, K_SCAN_BLOCKS, s);
    k_scan_blocks<<<1, 1024, 0, s>>>(p, ntiles);
  }
  {
    LaunchScope ls(c, K_SCAN_ADD, s);
    k_scan_add<<<(unsigned)ntiles, kScanThreads, 0, s>>>(p);
  }
  if (nnz > 0) {
    LaunchScope ls(c, K_FILL_PERM, s);
    k_fill_perm<<<grid_for(c, nnz, 256), 256, 0, s>>>(p, nnz);
  }
  const int G = lanes_per_row(p.D);
  if (nnz > 0) {
    const int64_t groups = (nnz + kChunk - 1) / kChunk;
    LaunchScope ls(c, K_SEGREDUCE_ADAGRAD, s);
    const int grid = grid_for(c, groups * G, 256, 8);
    if (p.bf16)
      k_segreduce_adagrad<true><<<grid, 256, 0, s>>>(p, dpooled, c->multi_hot ? 0 : 1, G);
    else
      k_segreduce_adagrad<false><<<grid, 256, 0, s>>>(p, dpooled, c->multi_hot ? 0 : 1, G);
  }
  {
    LaunchScope ls(c, K_ADAGRAD_FROM_G, s);
    const int grid = grid_for(c, (nnz > 0 ? nnz : 1) * G, 256, 8);
    if (p.bf16)
      k_adagrad_from_g<true><<<grid, 256, 0, s>>>(p, 1, G);
    else
      k_adagrad_from_g<false><<<grid, 256, 0, s>>>(p, 1, G);
  }
  return cudaGetLastError();
}

cudaError_t launch_adagrad_from_g(Ctx* c, int64_t max_unique, cudaStream_t s) {
  const Params& p = c->p;
  const int G = lanes_per_row(p.D);
  LaunchScope ls(c, K_ADAGRAD_FROM_G, s);
  const int grid = grid_for(c, (max_unique > 0 ? max_unique : 1) * G, 256, 8);
  if (p.bf16)
    k_adagrad_from_g<true><<<grid, 256, 0, s>>>(p, 0, G);
  else
    k_adagrad_from_g<false><<<grid, 256, 0, s>>>(p, 0, G);
  return cudaGetLastError();
}

}  // namespace emb
