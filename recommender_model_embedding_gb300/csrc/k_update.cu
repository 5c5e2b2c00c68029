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
//    (block-aggregated occurrence counts -> exclusive scan -> positions; the sorted order
//    keeps each lookup's unique index and bag), then fixed chunks of kChunk sorted
//    positions per lane group.  One-hot batches: a row whose lookups all fall inside one
//    chunk is reduced and updated by that group directly, its parameters prefetched when
//    its run starts; a row cut by a chunk boundary (a hot row) adds its partial sums into
//    g[u] with vector reductions and is updated afterwards by k_adagrad_from_g.  Multi-hot
//    batches: every run's sum goes into g[u] (stored when the row's lookups all fall in the
//    chunk, added otherwise) and k_adagrad_from_g updates all rows.  Every group does the
//    same bounded amount of work however skewed the ID distribution is.
//  * from the fused interaction backward, which has already added every row gradient into
//    g[u]: k_adagrad_from_g updates all U rows.
// k_adagrad_from_g also frees the row's dedup-set slot and, except after a multi-hot
// reduce, zeroes g[u], leaving both clean for the next batch.
#include "emb_internal.cuh"

namespace emb {

constexpr int kChunk = 32;  // sorted positions per lane group

// Lanes per row: a power of two such that each lane holds at most 4 chunks of 4 elements
// (D = 128 -> 8 lanes, 4 rows per warp).  Few lanes per row and several chunks per lane
// keep many independent row loads in flight per warp.
__host__ __device__ constexpr int lanes_per_row(int D) {
  int G = 1;
  while (G < (D / 4 + 3) / 4 && G < 32) G <<= 1;
  return G;
}

// Lanes per row of the segmented reduce: at most two 16-byte chunks per lane, so the
// gradient rows of kSegBlk positions and the row's parameters fit in registers together.
static int seg_lanes(int D) {
  const int need = (D / 4 + 1) / 2;
  int G = 1;
  while (G < need && G < 32) G <<= 1;
  return G;
}

// Tracked keys without admission holds: the work of k_admit for unique row u (its lookups
// added to the slot's count, saturating, and the step stamped), done by the kernel that
// visits u anyway in the fused step.
__device__ __forceinline__ void stamp_row(const Params& p, uint32_t u, uint32_t slot, uint32_t step) {
  const uint32_t c = p.cnt[u], f0 = (uint32_t)p.hstat[slot];
  const uint32_t f = f0 > 0xFFFFFFFFu - c ? 0xFFFFFFFFu : f0 + c;
  p.hstat[slot] = ((uint64_t)step << 32) | f;
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


// Adagrad on one row held by a group of G lanes; lane `sub` holds chunks sub, sub+G, ...
// (up to NCH chunks of 4 elements).  adagrad_load issues every load of the row (parameters
// and accumulators) so that the caller can overlap them with other work; adagrad_apply
// does the arithmetic and the stores.  All lanes of the warp must call adagrad_apply
// together (the row-wise variant reduces across the group).  With Adagrad Decay the load
// also fetches the period of the row's last update (lastp), and the apply discounts the
// accumulator by rate^(periods since then) before adding this step's squares.
// RW: 1 row-wise accumulators, 0 per element, -1 as the table is configured (p.rowwise);
// a kernel compiled for one kind keeps no registers for the other.
template <bool BF16, int NCH, bool DECAY, int RW = -1>
__device__ __forceinline__ void adagrad_load(const Params& p, uint32_t row, int sub, int G,
                                             bool active, float4 (&w)[NCH], float4 (&a)[NCH],
                                             float& ar, uint32_t& lastp) {
  const int KC = p.D / 4;
  if (DECAY && active) lastp = p.rperiod[row];
#pragma unroll
  for (int m = 0; m < NCH; ++m) {
    const int kc = sub + m * G;
    if (active && kc < KC) {
      w[m] = load_w4<BF16>(p, row, kc);
      if (!(RW < 0 ? p.rowwise : RW == 1))
        a[m] = reinterpret_cast<const float4*>(p.acc + (int64_t)row * p.D)[kc];
    }
  }
  if ((RW < 0 ? p.rowwise : RW == 1) && active) ar = p.acc[row];
}

template <bool BF16, int NCH, bool DECAY, int RW = -1>
__device__ __forceinline__ void adagrad_apply(const Params& p, uint32_t row, int sub, int G,
                                              const float4* gk, bool active,
                                              const float4 (&w)[NCH], const float4 (&a)[NCH],
                                              float ar, uint32_t lastp) {
  const int KC = p.D / 4;
  const float dec = DECAY ? acc_decay(lastp, p.period, p.decay_rate) : 1.f;
  if (DECAY && active && sub == 0) p.rperiod[row] = p.period;
  if (RW < 0 ? p.rowwise : RW == 1) {
    float sq = 0.f;
#pragma unroll
    for (int m = 0; m < NCH; ++m) {
      const int kc = sub + m * G;
      if (active && kc < KC)
        sq += gk[m].x * gk[m].x + gk[m].y * gk[m].y + gk[m].z * gk[m].z + gk[m].w * gk[m].w;
    }
    sq = group_sum(sq, G);
    if (!active) return;
    ar = DECAY ? ar * dec + sq / (float)p.D : ar + sq / (float)p.D;
    // one step size for the whole row, lr / (sqrt(acc) + eps) (IEEE square root and
    // division), then w_j - g_j * step: one rounding more than dividing each lr * g_j
    const float step = p.lr / (sqrtf(ar) + p.eps);
#pragma unroll
    for (int m = 0; m < NCH; ++m) {
      const int kc = sub + m * G;
      if (kc >= KC) continue;
      const float4 g = gk[m];
      store_w4<BF16>(p, row, kc,
                     make_float4(fmaf(-g.x, step, w[m].x), fmaf(-g.y, step, w[m].y),
                                 fmaf(-g.z, step, w[m].z), fmaf(-g.w, step, w[m].w)));
    }
    if (sub == 0) p.acc[row] = ar;
    return;
  }
  if (!active) return;
#pragma unroll
  for (int m = 0; m < NCH; ++m) {
    const int kc = sub + m * G;
    if (kc >= KC) continue;
    const float4 g = gk[m];
    float4 aa = DECAY ? f4_scale(a[m], dec) : a[m], ww = w[m];
    adagrad_elem(ww.x, aa.x, g.x, p.lr, p.eps);
    adagrad_elem(ww.y, aa.y, g.y, p.lr, p.eps);
    adagrad_elem(ww.z, aa.z, g.z, p.lr, p.eps);
    adagrad_elem(ww.w, aa.w, g.w, p.lr, p.eps);
    reinterpret_cast<float4*>(p.acc + (int64_t)row * p.D)[kc] = aa;
    store_w4<BF16>(p, row, kc, ww);
  }
}

// load and apply in one call (every load of the row issued before any arithmetic)
template <bool BF16, bool DECAY, int RW = -1>
__device__ __forceinline__ void adagrad_row(const Params& p, uint32_t row, int sub, int G,
                                            const float4* gk, bool active) {
  float4 w[4], a[4];
  float ar = 0.f;
  uint32_t lastp = 0;
  adagrad_load<BF16, 4, DECAY, RW>(p, row, sub, G, active, w, a, ar, lastp);
  adagrad_apply<BF16, 4, DECAY, RW>(p, row, sub, G, gk, active, w, a, ar, lastp);
}

// ------------------------------------------------------------------ counting sort

// Unique index of each lookup and its rank among the lookups of that row.  The counts are
// aggregated per block before they reach global memory: a block takes a tile of kAggTile
// lookups, counts each unique index of the tile in a shared-memory hash table (the count's
// old value is the lookup's rank inside the tile), then adds each index's tile count to its
// global count with one atomicAdd, whose old value is the tile's base.  A Zipf-hot row (the
// hottest key of the hashed workload takes ~9% of all lookups) then costs one global atomic
// per tile instead of one per warp, which serialised on its counter's L2 slice.
constexpr int kAggThreads = 512;
constexpr int kAggPer = 4;                          // lookups per thread per tile
constexpr int kAggTile = kAggThreads * kAggPer;     // 2048
constexpr int kAggSlots = 2 * kAggTile;             // shared hash table (at most half full)

// RANK = false (the fused steps, which need counts but no sorted order): no ranks; the unique
// index written per lookup is the inverse of k_inverse, with the once mark when mark_once,
// so the kernel replaces k_inverse there.  Either way block 0 copies U into the host-mapped
// mirror (h_unique, when given), which sizes the next batch's dedup set and its once-row
// choice.
template <bool RANK>
__global__ void __launch_bounds__(kAggThreads) k_inverse_count(Params p, int64_t nnz,
                                                               int mark_once, uint32_t* h_unique) {
  __shared__ uint32_t tkey[kAggSlots];  // unique index, kEmpty32 when free
  __shared__ uint32_t tval[kAggSlots];  // count of the tile, then the tile's global base
  if (h_unique && blockIdx.x == 0 && threadIdx.x == 0)
    *reinterpret_cast<volatile uint32_t*>(h_unique) = p.counters[kU];
  for (int64_t t0 = (int64_t)blockIdx.x * kAggTile; t0 < nnz; t0 += (int64_t)gridDim.x * kAggTile) {
    for (int e = threadIdx.x; e < kAggSlots; e += kAggThreads) {
      tkey[e] = kEmpty32;
      tval[e] = 0u;
    }
    __syncthreads();
    uint32_t u[kAggPer], ent[kAggPer], loc[kAggPer];
    uint32_t sl[kAggPer], rw[kAggPer];
#pragma unroll
    for (int j = 0; j < kAggPer; ++j) {
      const int64_t q = t0 + j * kAggThreads + threadIdx.x;
      sl[j] = q < nnz ? p.slot_of[q] : kEmpty32;
      rw[j] = q < nnz ? p.row_of[q] : kNoRow;
    }
#pragma unroll
    for (int j = 0; j < kAggPer; ++j)
      u[j] = (rw[j] != kNoRow && sl[j] != kEmpty32) ? p.set_vals[sl[j]] : kNoRow;
#pragma unroll
    for (int j = 0; j < kAggPer; ++j) {
      ent[j] = kEmpty32;
      loc[j] = 0u;
      if (u[j] == kNoRow) continue;
      uint32_t h = mix32(u[j]) & (kAggSlots - 1);
      for (int n = 0; n < kAggSlots; ++n) {  // at most half full: ends at a free or own slot
        const uint32_t k = atomicCAS(tkey + h, kEmpty32, u[j]);
        if (k == kEmpty32 || k == u[j]) break;
        h = (h + 1) & (kAggSlots - 1);
      }
      ent[j] = h;
      loc[j] = atomicAdd(tval + h, 1u);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kAggSlots; e += kAggThreads)
      if (tkey[e] != kEmpty32) tval[e] = atomicAdd(p.cnt + tkey[e], tval[e]);
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kAggPer; ++j) {
      const int64_t q = t0 + j * kAggThreads + threadIdx.x;
      if (q >= nnz) continue;
      uint32_t iv = u[j];
      if (RANK) {
        if (iv != kNoRow) p.rank[q] = tval[ent[j]] + loc[j];
      } else if (mark_once && iv != kNoRow && !(p.set_keys[sl[j]] & kSetMulti)) {
        p.uniq_once[iv] = 1;  // the only lookup of its row
        iv |= kInvOnce;
      }
      p.inv[q] = iv;
    }
    __syncthreads();  // the table is cleared for the next tile only after every read
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

// Lookups in unique-row order: position seg[u] + rank of each lookup gets its unique index
// and its bag (one 8-byte store at a scattered position).  zero_split (the summing reduce, which stores the sum of a row
// whose lookups fall in one chunk and adds partial sums of the others): the first lookup of
// a row whose positions cross a chunk boundary zeroes the row's g[u] for those additions.
__global__ void k_fill_perm(Params p, int64_t nnz, int one_hot, int zero_split) {
  for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < nnz;
       q += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t u = p.inv[q];
    if (u != kNoRow) {
      const uint32_t r = p.rank[q];
      const uint32_t pos = p.seg[u] + r;
      p.s_ub[pos] = make_uint2(u, one_hot ? (uint32_t)q : p.bag_of[q]);
      if (zero_split && r == 0 && pos / kChunk != (p.seg[u + 1] - 1) / kChunk) {
        float4* gu = reinterpret_cast<float4*>(p.g + (int64_t)u * p.D);
        for (int kc = 0; kc < p.D / 4; ++kc) gu[kc] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
}

// ------------------------------------------------------------------ reduce + update

constexpr int kSegBlk = 4;  // sorted positions whose gradient rows are loaded together

// One lane group per chunk of kChunk sorted positions.  A run (consecutive positions of one
// unique row) that starts inside the chunk prefetches the row's parameters at once; when
// the run ends inside the chunk (or the segment ends exactly at the chunk's end) the group
// applies Adagrad from registers; a run cut by a chunk boundary adds into g[u] instead.
template <bool BF16, bool DECAY, bool DIRECT>
__global__ void __launch_bounds__(256, DIRECT ? 2 : 4) k_segreduce_adagrad(Params p, const float* dpooled,
                                                           int one_hot, int G) {
  constexpr int NCH = 2;
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
    // (the direct form is one-hot only: the bag is the lookup, whose row is row_of[bag]; the
    // summing form needs no row)
    const uint2 first = live ? p.s_ub[p0] : make_uint2(kNoRow, 0u);
    uint32_t cur = first.x;
    uint32_t row = DIRECT && live ? p.row_of[first.y] : 0u;
    const bool cont_in = live && p0 > 0 && p.s_ub[p0 - 1].x == cur;
    const uint32_t u_last = live ? p.s_ub[p1 - 1].x : kNoRow;
    const bool cont_out = live && p1 < NV && p.s_ub[p1].x == u_last;
    // the current run may be its row's whole segment (DIRECT only: otherwise every run's
    // sum goes to g and the update kernel applies Adagrad to all rows; the compiler then
    // drops the parameter loads and updates below)
    bool whole = DIRECT && live && !cont_in;
    // (summing variant) the current run starts in this chunk: if it also ends here, its sum
    // is the row's whole gradient and is stored, not added
    bool starts_here = live && !cont_in;
    // hashed tables under admission: the row of a held key takes no update this step
    const bool hold_on = p.admit_min > 1;
    bool held = hold_on && live && p.uniq_hold[cur];
    float4 w[NCH], a[NCH];
    float ar = 0.f;
    uint32_t lp = 0;
    adagrad_load<BF16, NCH, DECAY>(p, row, sub, G, whole, w, a, ar, lp);
    float4 acc[NCH];
#pragma unroll
    for (int m = 0; m < NCH; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    // position data (unique index, row, bag) of the next block, loaded one block ahead
    uint32_t nu[kSegBlk], nr[kSegBlk], nbg[kSegBlk];
#pragma unroll
    for (int i = 0; i < kSegBlk; ++i) {
      const int64_t pos = p0 + i;
      const bool have = live && pos < p1;
      const uint2 e = have ? p.s_ub[pos] : make_uint2(kNoRow, 0u);
      nu[i] = e.x;
      nbg[i] = e.y;
      nr[i] = DIRECT && have ? p.row_of[e.y] : 0u;
    }
    for (int b0 = 0; b0 < kChunk; b0 += kSegBlk) {
      uint32_t uu[kSegBlk], rr[kSegBlk], bb[kSegBlk];
      float sc[kSegBlk];
      float4 v[kSegBlk][NCH];
#pragma unroll
      for (int i = 0; i < kSegBlk; ++i) {
        uu[i] = nu[i];
        rr[i] = nr[i];
        bb[i] = nbg[i];
        const int64_t pos = p0 + b0 + kSegBlk + i;
        const bool have = live && b0 + kSegBlk < kChunk && pos < p1;
        const uint2 e = have ? p.s_ub[pos] : make_uint2(kNoRow, 0u);
        nu[i] = e.x;
        nbg[i] = e.y;
        nr[i] = DIRECT && have ? p.row_of[e.y] : 0u;
      }
#pragma unroll
      for (int i = 0; i < kSegBlk; ++i) {
        const bool have = uu[i] != kNoRow;
        sc[i] = 1.f;
        if (p.mean && !one_hot && have) sc[i] = 1.f / (float)(p.offs[bb[i] + 1] - p.offs[bb[i]]);
        const float4* src = reinterpret_cast<const float4*>(dpooled + (int64_t)bb[i] * p.D);
#pragma unroll
        for (int m = 0; m < NCH; ++m) {
          const int kc = sub + m * G;
          v[i][m] = (have && kc < KC) ? __ldg(src + kc) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int i = 0; i < kSegBlk; ++i) {
        const bool have = uu[i] != kNoRow;
        const bool change = have && uu[i] != cur;
        const bool flush_whole = change && whole && !held;
        if (__any_sync(0xFFFFFFFFu, flush_whole))
          adagrad_apply<BF16, NCH, DECAY>(p, row, sub, G, acc, flush_whole, w, a, ar, lp);
        if (change) {
          if (!whole) {
#pragma unroll
            for (int m = 0; m < NCH; ++m) {
              const int kc = sub + m * G;
              float* dst = p.g + (int64_t)cur * p.D + 4 * kc;
              if (kc < KC) {
                if (!DIRECT && starts_here) *reinterpret_cast<float4*>(dst) = acc[m];
                else red_add_f4(dst, acc[m]);
              }
            }
          }
          starts_here = true;
#pragma unroll
          for (int m = 0; m < NCH; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
          cur = uu[i];
          row = rr[i];
          whole = DIRECT;
          held = hold_on && p.uniq_hold[cur];
          adagrad_load<BF16, NCH, DECAY>(p, row, sub, G, true, w, a, ar, lp);
        }
        if (have) {
#pragma unroll
          for (int m = 0; m < NCH; ++m) {
            acc[m].x = fmaf(sc[i], v[i][m].x, acc[m].x);
            acc[m].y = fmaf(sc[i], v[i][m].y, acc[m].y);
            acc[m].z = fmaf(sc[i], v[i][m].z, acc[m].z);
            acc[m].w = fmaf(sc[i], v[i][m].w, acc[m].w);
          }
        }
      }
    }
    // the chunk's last run (a held row that ends here is dropped; a cut run goes to g)
    const bool last_whole = live && whole && !cont_out;
    const bool fw = last_whole && !held;
    if (__any_sync(0xFFFFFFFFu, fw)) adagrad_apply<BF16, NCH, DECAY>(p, row, sub, G, acc, fw, w, a, ar, lp);
    if (live && !last_whole) {
      const bool store = !DIRECT && starts_here && !cont_out;
#pragma unroll
      for (int m = 0; m < NCH; ++m) {
        const int kc = sub + m * G;
        float* dst = p.g + (int64_t)cur * p.D + 4 * kc;
        if (kc < KC) {
          if (store) *reinterpret_cast<float4*>(dst) = acc[m];
          else red_add_f4(dst, acc[m]);
        }
      }
    }
  }
}

// Update rows from g[u] (all rows, or only rows whose segment of sorted positions crosses a
// multiple of `span`, the segmented reduce's chunk or tile), zero g[u] and free the
// dedup-set slot of every unique row.  With from_list, the rows are the counters[kMulti]
// entries (u, row, slot) that k_once_split listed in s_u, s_row and s_bag.  A key held by
// admission (hashed tables) has its g[u] cleared but its parameters left unchanged.
// STAMP (fused steps of tracked keys, no holds, not from_list): also stamps every row it
// visits (stamp_row).  keep_g (after the summing reduce, which stores or zeroes g[u] of every
// unique row itself): g[u] is read and left as it is.
template <bool BF16, bool DECAY, bool STAMP, int RW = -1>
__global__ void __launch_bounds__(256) k_adagrad_from_g(Params p, int split_only, int G,
                                                        int span, int from_list, uint32_t step,
                                                        int keep_g) {
  const int lane = threadIdx.x & 31;
  const int sub = lane % G;
  const int gpw = 32 / G;
  const int KC = p.D / 4;
  const uint32_t U = p.counters[from_list ? kMulti : kU];
  const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t stride = nwarps * gpw;
  int64_t i = gwarp * gpw + lane / G;
  // Everything that decides an address or a predicate of the next iteration (its unique
  // index, row, dedup-set slot, whether its segment was split) is loaded one iteration
  // ahead: with in-order issue, an instruction waiting on a fresh load would hold back the
  // row loads behind it for a whole memory round trip.
  uint32_t uq = 0u, row = 0u, slot = 0u;
  bool split = true, held = false;
  const bool hold_on = p.admit_min > 1;  // hashed tables under admission
  auto next = [&](int64_t ii) {
    if (from_list) {
      uq = p.s_u[ii];
      row = p.s_row[ii];
      slot = p.s_bag[ii];
    } else {
      uq = (uint32_t)ii;
      row = p.uniq_row[ii];
      slot = p.uniq_slot[ii];
      if (split_only) split = (p.seg[ii] / span) != ((p.seg[ii + 1] - 1) / span);
    }
    if (hold_on) held = p.uniq_hold[uq] != 0;
  };
  if (i < U) next(i);
  for (int64_t i0 = gwarp * gpw; i0 < U; i0 += stride, i += stride) {
    const bool live = i < U;
    const bool active = live && split;   // g[u] read and cleared
    const bool update = active && !held;  // parameters updated
    const uint32_t u = uq, row_now = row, slot_now = slot;
    const int64_t in = i + stride;
    if (in < U) next(in);
    float4 gk[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int kc = sub + m * G;
      gk[m] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (active && kc < KC) gk[m] = reinterpret_cast<const float4*>(p.g + (int64_t)u * p.D)[kc];
    }
    adagrad_row<BF16, DECAY, RW>(p, row_now, sub, G, gk, update);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int kc = sub + m * G;
      if (active && !keep_g && kc < KC)
        reinterpret_cast<float4*>(p.g + (int64_t)u * p.D)[kc] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (live && sub == 0) {
      p.set_keys[slot_now] = kEmpty32;
      if (STAMP) stamp_row(p, u, row_now, step);
    }
  }
}

// ------------------------------------------------------------------ staged update

// Every unique row u < U updated from g[u] (the all-rows form of k_adagrad_from_g, without
// Adagrad Decay, admission holds or stamps; D <= 128), with each tile of rows -- its
// gradient rows, parameter rows, accumulators, table rows and dedup-set slots -- copied
// into shared memory by cp.async kStages - 1 tiles ahead.
// The register form keeps one group of rows in flight per warp and waits for it; here the
// copies of later tiles stay in flight while a tile is computed, holding no registers.  A
// tile is one row per lane group: 256 / G rows.  Row strides are padded by 16 bytes per lane
// of a group (8 for bf16 parameters), so the two or four rows a quarter-warp reads start in
// different banks.  Used for row-wise tables (the multi-hot bf16 update: 0.359 -> 0.305 ms);
// on the fp32 per-element update of the Criteo shape it measured the same as the register
// form (0.193 against 0.192 ms), which stays there.  Three stages of about 31 KB (two CTAs
// per SM) measured best: four stages 0.321 ms, unpadded rows 0.309-0.315 ms.
constexpr int kStages = 3;

struct StagedLayout {
  int gs, ws, as;                  // padded row strides (bytes) of g, w, per-element acc
  int g, w, a, row, slot, bytes;   // offsets inside a stage, and its size
};

static inline StagedLayout staged_layout(int D, int G, bool bf16, bool rowwise) {
  StagedLayout L;
  const int R = 256 / G;
  L.gs = D * 4 + 16 * G;
  L.ws = bf16 ? D * 2 + 8 * G : D * 4 + 16 * G;
  L.as = D * 4 + 16 * G;
  L.g = 0;
  L.w = L.g + R * L.gs;
  L.a = L.w + R * L.ws;
  L.row = L.a + (rowwise ? (R * 4 + 15) / 16 * 16 : R * L.as);
  L.slot = L.row + R * 4;
  L.bytes = (L.slot + R * 4 + 15) / 16 * 16;
  return L;
}

__device__ __forceinline__ void cpa16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cpa4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// DT: the row length when known at compile time (64, the multi-hot shape: the copy loops'
// divisions become shifts; ncu showed the runtime-D copy issue-bound at 58% issue, and the
// multi-hot update went 0.292 -> 0.281 ms), else 0 (p.D).
template <bool BF16, int RW, int DT>
__global__ void __launch_bounds__(256) k_adagrad_staged(Params p, int Gr, int keep_g, StagedLayout L) {
  // bf16 parameters with per-element accumulators would need two chunk maps (8 and 4
  // elements per 16 bytes); that form is not built
  static_assert(!BF16 || RW == 1, "bf16 tables: row-wise accumulators only");
  extern __shared__ __align__(16) unsigned char sm[];
  constexpr int kMaxPer = 4;  // 16-byte chunks per thread and tile, each kind (D <= 128)
  const int tid = threadIdx.x, D = DT ? DT : p.D, KC = D / 4;
  const int G = DT ? lanes_per_row(DT) : Gr;
  const int R = 256 / G;
  const int wcpr = BF16 ? D / 8 : KC;  // 16-byte chunks of a parameter row
  const int row_bytes = BF16 ? D * 2 : D * 4;
  const uint32_t U = p.counters[kU];
  const int64_t ntiles = ((int64_t)U + R - 1) / R;
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(sm);
  auto tile_of = [&](int64_t k) { return (int64_t)blockIdx.x + k * (int64_t)gridDim.x; };
  // table rows of this thread's parameter (and per-element accumulator) chunks, and of its
  // row-wise accumulator, for the next tile to copy
  uint32_t rv[kMaxPer], rva = 0u;
  auto load_rows = [&](int64_t k) {
    const int64_t t = tile_of(k);
#pragma unroll
    for (int j = 0; j < kMaxPer; ++j) {
      const int c = tid + 256 * j;
      const int64_t u = t * R + c / wcpr;
      rv[j] = (t < ntiles && c < R * wcpr && u < U) ? p.uniq_row[u] : 0u;
    }
    if (RW == 1) {
      const int64_t u = t * R + tid;
      rva = (t < ntiles && tid < R && u < U) ? p.uniq_row[u] : 0u;
    }
  };
  auto issue = [&](int64_t k) {
    const int64_t t = tile_of(k);
    if (t < ntiles) {
      const int64_t u0 = t * R;
      const uint32_t st = sbase + (uint32_t)((k % kStages) * L.bytes);
      for (int c = tid; c < R * KC; c += 256) {  // gradient rows (consecutive u)
        const int r = c / KC, q = c % KC;
        if (u0 + r < U) cpa16(st + L.g + r * L.gs + q * 16, p.g + (u0 + r) * D + 4 * q);
      }
#pragma unroll
      for (int j = 0; j < kMaxPer; ++j) {  // parameter rows, per-element accumulator rows
        const int c = tid + 256 * j;
        if (c < R * wcpr) {
          const int r = c / wcpr, q = c % wcpr;
          if (u0 + r < U) {
            cpa16(st + L.w + r * L.ws + q * 16,
                  static_cast<const unsigned char*>(p.table) + (int64_t)rv[j] * row_bytes + 16 * q);
            if (RW != 1) cpa16(st + L.a + r * L.as + q * 16, p.acc + (int64_t)rv[j] * D + 4 * q);
          }
        }
      }
      if (RW == 1 && tid < R && u0 + tid < U) cpa4(st + L.a + tid * 4, p.acc + rva);
      for (int i = tid; i < 2 * R; i += 256) {  // table rows, dedup-set slots
        const int r = i < R ? i : i - R;
        if (u0 + r < U)
          cpa4(st + (i < R ? L.row : L.slot) + r * 4, (i < R ? p.uniq_row : p.uniq_slot) + u0 + r);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");  // empty past the last tile
  };

  load_rows(0);
  for (int k = 0; k < kStages - 1; ++k) {
    issue(k);
    load_rows(k + 1);
  }
  const int r = tid / G, sub = tid % G;
  for (int64_t k = 0; tile_of(k) < ntiles; ++k) {
    issue(k + kStages - 1);
    load_rows(k + kStages);
    asm volatile("cp.async.wait_group %0;" ::"n"(kStages - 1) : "memory");
    __syncthreads();
    const unsigned char* st = sm + (k % kStages) * L.bytes;
    const int64_t u = tile_of(k) * R + r;
    const bool active = u < U;
    float4 gk[4], w[4], a[4];
    float ar = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int kc = sub + m * G;
      gk[m] = w[m] = a[m] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (active && kc < KC) {
        gk[m] = *reinterpret_cast<const float4*>(st + L.g + r * L.gs + kc * 16);
        if (BF16) {
          const uint2 raw = *reinterpret_cast<const uint2*>(st + L.w + r * L.ws + kc * 8);
          const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
          const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
          w[m] = make_float4(lo.x, lo.y, hi.x, hi.y);
        } else {
          w[m] = *reinterpret_cast<const float4*>(st + L.w + r * L.ws + kc * 16);
        }
        if (RW != 1) a[m] = *reinterpret_cast<const float4*>(st + L.a + r * L.as + kc * 16);
      }
    }
    if (RW == 1 && active) ar = *reinterpret_cast<const float*>(st + L.a + r * 4);
    const uint32_t row = active ? *reinterpret_cast<const uint32_t*>(st + L.row + r * 4) : 0u;
    adagrad_apply<BF16, 4, false, RW>(p, row, sub, G, gk, active, w, a, ar, 0u);
    if (active) {
      if (sub == 0) p.set_keys[*reinterpret_cast<const uint32_t*>(st + L.slot + r * 4)] = kEmpty32;
      if (!keep_g) {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int kc = sub + m * G;
          if (kc < KC) reinterpret_cast<float4*>(p.g + u * D)[kc] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
    __syncthreads();
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// The staged update where it applies: row-wise accumulators, no decay or holds (and
// EMB_STAGED_UPDATE at context creation is not 0).
static bool staged_ok(const Ctx* c) {
  const Params& p = c->p;
  return c->staged_update && p.rowwise && !p.decay && p.admit_min <= 1 && p.D <= 128 &&
         p.D % (p.bf16 ? 8 : 4) == 0;
}

static cudaError_t launch_adagrad_staged(Ctx* c, int64_t max_unique, int keep_g, cudaStream_t s) {
  const Params& p = c->p;
  const int G = lanes_per_row(p.D);
  const StagedLayout L = staged_layout(p.D, G, p.bf16 != 0, p.rowwise != 0);
  const int smem = kStages * L.bytes;
  auto kern = p.D == 64 ? (p.bf16 ? k_adagrad_staged<true, 1, 64> : k_adagrad_staged<false, 1, 64>)
                        : (p.bf16 ? k_adagrad_staged<true, 1, 0> : k_adagrad_staged<false, 1, 0>);
  const int per_sm = std::max(1, resident_ctas(c, kern, 256, smem));
  const int64_t tiles = std::max<int64_t>(1, (max_unique + (256 / G) - 1) / (256 / G));
  const int grid = (int)std::min<int64_t>(tiles, (int64_t)per_sm * c->num_sms);
  LaunchScope ls(c, K_ADAGRAD_FROM_G, s);
  kern<<<grid, 256, smem, s>>>(p, G, keep_g, L);
  return cudaGetLastError();
}

// Steps that track once rows, before the update: free the dedup-set slot of every once row
// (the backward has updated it) and clear its mark; list every other unique row as
// (u, row, slot) in s_u, s_row, s_bag, counters[kMulti] entries (one atomicAdd per block).
// stamp: also does the work of k_admit for every unique row (tracked keys, no holds).
__global__ void __launch_bounds__(256) k_once_split(Params p, uint32_t step, int stamp) {
  __shared__ uint32_t warp_n[8];
  __shared__ uint32_t block_base;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const uint32_t U = p.counters[kU];
  for (int64_t u0 = (int64_t)blockIdx.x * blockDim.x; u0 < U; u0 += (int64_t)gridDim.x * blockDim.x) {
    const int64_t u = u0 + threadIdx.x;
    bool multi = false;
    uint32_t slot = 0u;
    if (u < U) {
      slot = p.uniq_slot[u];
      if (stamp) stamp_row(p, (uint32_t)u, p.uniq_row[u], step);
      if (p.uniq_once[u]) {
        p.set_keys[slot] = kEmpty32;
        p.uniq_once[u] = 0;
      } else {
        multi = true;
      }
    }
    const unsigned ball = __ballot_sync(0xFFFFFFFFu, multi);
    if (lane == 0) warp_n[wid] = __popc(ball);
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t tot = 0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
        const uint32_t cw = warp_n[w];
        warp_n[w] = tot;
        tot += cw;
      }
      block_base = tot ? atomicAdd(p.counters + kMulti, tot) : 0u;
    }
    __syncthreads();
    if (multi) {
      const uint32_t j = block_base + warp_n[wid] + __popc(ball & ((1u << lane) - 1u));
      p.s_u[j] = (uint32_t)u;
      p.s_row[j] = p.uniq_row[u];
      p.s_bag[j] = slot;
    }
    __syncthreads();
  }
}

// g[u] is zero between steps except after a multi-hot step (the summing reduce stores the
// rows' sums and the update leaves them): before a backward that adds into g, zero the rows
// such a step may have left.
cudaError_t clear_stale_g(Ctx* c, cudaStream_t s) {
  if (c->g_stale <= 0) return cudaSuccess;
  const cudaError_t e =
      cudaMemsetAsync(c->p.g, 0, sizeof(float) * (size_t)(c->g_stale * c->p.D), s);
  if (e == cudaSuccess) c->g_stale = 0;
  return e;
}

cudaError_t launch_backward_csr(Ctx* c, const float* dpooled, int64_t batch, int64_t nnz,
                                cudaStream_t s) {
  const Params& p = c->p;
  // One-hot batches apply Adagrad inside the segmented reduce to rows whose run ends in the
  // chunk (most runs are a few lookups long, and their parameters load while the run is
  // summed); multi-hot batches sum every run into g and update all rows in one streaming
  // pass, which keeps the parameter loads off the reduce's critical path (measured on the
  // multi-hot bf16 workload: reduce + update 1.39 -> 0.93 ms; on the hashed one-hot workload
  // the direct form is faster, 0.13 against 0.19 ms).  The summing form stores the sum of a
  // row whose lookups fall in one chunk and adds the partial sums of the others into g[u],
  // zeroed first by the sort; the update then leaves g[u] as it is.
  const int direct = c->multi_hot ? 0 : 1;
  cudaError_t e = direct ? clear_stale_g(c, s) : cudaSuccess;
  if (e == cudaSuccess) e = cudaMemsetAsync(p.cnt, 0, sizeof(uint32_t) * (size_t)(nnz + 1), s);
  if (e != cudaSuccess) return e;
  if (nnz > 0) {
    LaunchScope ls(c, K_INVERSE_COUNT, s);
    k_inverse_count<true>
        <<<grid_for(c, (nnz + kAggTile - 1) / kAggTile * kAggThreads, kAggThreads, 4),
           kAggThreads, 0, s>>>(p, nnz, 0, c->h_unique_dev);
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
  if (c->track) {  // counts, last step and admission holds of the step's keys
    cudaError_t e2 = launch_admit(c, s);
    if (e2 != cudaSuccess) return e2;
  }
  const int one_hot = c->multi_hot ? 0 : 1;
  if (nnz > 0) {
    LaunchScope ls(c, K_FILL_PERM, s);
    k_fill_perm<<<grid_for(c, nnz, 256), 256, 0, s>>>(p, nnz, one_hot, direct ? 0 : 1);
  }
  const int G = lanes_per_row(p.D);
  if (nnz > 0) {
    const int64_t chunks = (nnz + kChunk - 1) / kChunk;
    const int GS = seg_lanes(p.D);
    LaunchScope ls(c, K_SEGREDUCE_ADAGRAD, s);
    const int grid = grid_for(c, chunks * GS, 256, 8);
    auto kern = direct ? (p.bf16 ? (p.decay ? k_segreduce_adagrad<true, true, true>
                                            : k_segreduce_adagrad<true, false, true>)
                                 : (p.decay ? k_segreduce_adagrad<false, true, true>
                                            : k_segreduce_adagrad<false, false, true>))
                       : (p.bf16 ? (p.decay ? k_segreduce_adagrad<true, true, false>
                                            : k_segreduce_adagrad<true, false, false>)
                                 : (p.decay ? k_segreduce_adagrad<false, true, false>
                                            : k_segreduce_adagrad<false, false, false>));
    kern<<<grid, 256, 0, s>>>(p, dpooled, one_hot, GS);
  }
  if (!direct && staged_ok(c)) {
    e = launch_adagrad_staged(c, std::min<int64_t>(nnz, c->total_rows), 1, s);
    if (e != cudaSuccess) return e;
  } else {
    // direct: only rows cut by a chunk boundary are left to this kernel; otherwise all rows
    LaunchScope ls(c, K_ADAGRAD_FROM_G, s);
    const int grid = grid_for(c, (nnz > 0 ? nnz : 1) * G, 256, 8);
    const int split_only = direct, span = direct ? kChunk : 1;
    if (p.bf16)
      (p.decay ? k_adagrad_from_g<true, true, false>
               : (p.rowwise ? k_adagrad_from_g<true, false, false, 1> : k_adagrad_from_g<true, false, false>))
          <<<grid, 256, 0, s>>>(p, split_only, G, span, 0, c->step, direct ? 0 : 1);
    else
      (p.decay ? k_adagrad_from_g<false, true, false>
               : (p.rowwise ? k_adagrad_from_g<false, false, false, 1> : k_adagrad_from_g<false, false, false>))
          <<<grid, 256, 0, s>>>(p, split_only, G, span, 0, c->step, direct ? 0 : 1);
  }
  if (!direct) c->g_stale = std::max<int64_t>(c->g_stale, std::min<int64_t>(nnz, c->total_rows));
  return cudaGetLastError();
}

// Fused steps that track keys (hashed tables with admission or eviction, tiered tables): in
// the forward, one pass gives each lookup its unique index (as k_inverse) and each unique
// row its lookup count; the backward then only stamps counts and steps (launch_admit).
cudaError_t launch_inverse_counts(Ctx* c, int64_t nnz, cudaStream_t s) {
  const Params& p = c->p;
  cudaError_t e = cudaMemsetAsync(p.cnt, 0, sizeof(uint32_t) * (size_t)(nnz + 1), s);
  if (e != cudaSuccess || nnz <= 0) return e;
  LaunchScope ls(c, K_INVERSE_COUNT, s);
  k_inverse_count<false>
      <<<grid_for(c, (nnz + kAggTile - 1) / kAggTile * kAggThreads, kAggThreads, 4),
         kAggThreads, 0, s>>>(p, nnz, c->once_step ? 1 : 0, c->h_unique_dev);
  return cudaGetLastError();
}

// The same counts after a forward whose kernel recorded the unique indices itself.
cudaError_t launch_count_admit(Ctx* c, int64_t nnz, cudaStream_t s) {
  cudaError_t e = launch_inverse_counts(c, nnz, s);
  return e != cudaSuccess ? e : launch_admit(c, s);
}

cudaError_t launch_adagrad_from_g(Ctx* c, int64_t max_unique, cudaStream_t s, bool stamp) {
  const Params& p = c->p;
  const int G = lanes_per_row(p.D);
  const int from_list = c->once_step ? 1 : 0;
  if (from_list) {  // the split visits every unique row: it stamps them
    cudaError_t e = cudaMemsetAsync(p.counters + kMulti, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    LaunchScope ls(c, K_ONCE_SPLIT, s);
    k_once_split<<<grid_for(c, max_unique > 0 ? max_unique : 1, 256, 8), 256, 0, s>>>(
        p, c->step, stamp ? 1 : 0);
  }
  const bool st = stamp && !from_list;
  if (!from_list && !st && staged_ok(c)) return launch_adagrad_staged(c, max_unique, 0, s);
  LaunchScope ls(c, K_ADAGRAD_FROM_G, s);
  const int grid = grid_for(c, (max_unique > 0 ? max_unique : 1) * G, 256, 8);
  auto kern = p.bf16 ? (p.decay ? (st ? k_adagrad_from_g<true, true, true> : k_adagrad_from_g<true, true, false>)
                                : (st ? k_adagrad_from_g<true, false, true> : k_adagrad_from_g<true, false, false>))
                     : (p.decay ? (st ? k_adagrad_from_g<false, true, true> : k_adagrad_from_g<false, true, false>)
                                : (st ? k_adagrad_from_g<false, false, true> : k_adagrad_from_g<false, false, false>));
  kern<<<grid, 256, 0, s>>>(p, 0, G, 1, from_list, c->step, 0);
  return cudaGetLastError();
}

}  // namespace emb
