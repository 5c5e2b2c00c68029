// ID -> row mapping, the hashed table, the per-batch dedup set, table initialisation and
// the read-back kernels.
//
// HugeCTR interview (zhidx), section 2: IDs whose range is unknown in advance are first
// identified through a hash table before the embedding lookup; section 3 (1): the table
// lives on the GPU.  DeepRec announcement, "EmbeddingVariable": the table is lock-free and
// a new feature starts from the initializer value (generally 0).
//
// Hashed table: open addressing with linear probing over `capacity` slots of int64 keys
// (free slot = all-ones, evicted slot = all-ones but bit 0).  Insert is a single
// compare-and-swap on the key: the row values and accumulators of every slot are written at
// creation (w = hash_init, acc = init_acc) and again when its key is evicted, so a thread
// that loses or wins the CAS reads the same initial row and no value has to be published
// after the key.  Probing stops after kMaxProbe slots with EMB_FLAG_TABLE_FULL.
//
// Dedup set: a second open-addressing set of uint32 row numbers, sized to at least twice
// the largest batch of lookups so it never fills.  The lane whose CAS claims a slot owns
// that row: the block aggregates its winners and takes one atomicAdd on the unique
// counter, which numbers the unique rows 0..U-1 (in no fixed order).
#include <algorithm>

#include "emb_internal.cuh"

namespace emb {

// ------------------------------------------------------------------ initialisation

// SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): output number n of the stream `seed`.
__device__ __forceinline__ uint64_t splitmix_out(uint64_t seed, uint64_t n) {
  uint64_t z = seed + n * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Initial value of element `col` of row `id` of table `t`: counter ((t<<40)+id)*512+col,
// 24 top bits of the stream output as u in [0,1), v = lo + width*u with one rounding per
// float operation.
__device__ __forceinline__ float init_value(uint64_t seed, int t, int64_t id, int col, float lo,
                                            float width) {
  const uint64_t c = ((((uint64_t)t) << 40) + (uint64_t)id) * 512ull + (uint64_t)col;
  const uint64_t z = splitmix_out(seed, c + 1);
  const float u = __fmul_rn(__uint2float_rn((uint32_t)(z >> 40)), 1.0f / 16777216.0f);
  return __fadd_rn(lo, __fmul_rn(width, u));
}

template <bool BF16>
__global__ void k_init_table(void* table, int64_t row0, int64_t nrows, int D, int t,
                             uint64_t seed, float lo, float width) {
  const int64_t n = nrows * D;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t id = e / D;
    const int col = (int)(e - id * D);
    const float v = init_value(seed, t, id, col, lo, width);
    const int64_t off = row0 * D + e;
    if (BF16)
      reinterpret_cast<__nv_bfloat16*>(table)[off] = __float2bfloat16_rn(v);
    else
      reinterpret_cast<float*>(table)[off] = v;
  }
}

template <bool BF16>
__global__ void k_fill(void* dst, int64_t n, float v) {
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    if (BF16)
      reinterpret_cast<__nv_bfloat16*>(dst)[e] = __float2bfloat16_rn(v);
    else
      reinterpret_cast<float*>(dst)[e] = v;
  }
}

cudaError_t launch_init_table(Ctx* c, cudaStream_t s) {
  const Params& p = c->p;
  const float lo = c->cfg.init_lo;
  const float width = c->cfg.init_hi - c->cfg.init_lo;
  int64_t row0 = 0;
  for (int t = 0; t < p.T; ++t) {
    const int64_t nr = c->rows[t];
    if (nr > 0) {
      LaunchScope ls(c, K_INIT_TABLE, s);
      const int grid = grid_for(c, nr * p.D, 256, 16);
      if (p.bf16)
        k_init_table<true><<<grid, 256, 0, s>>>(p.table, row0, nr, p.D, t, c->cfg.seed, lo, width);
      else
        k_init_table<false><<<grid, 256, 0, s>>>(p.table, row0, nr, p.D, t, c->cfg.seed, lo, width);
    }
    row0 += nr;
  }
  const int64_t nacc = c->total_rows * (p.rowwise ? 1 : p.D);
  {
    LaunchScope ls(c, K_INIT_TABLE, s);
    k_fill<false><<<grid_for(c, nacc, 256, 16), 256, 0, s>>>(p.acc, nacc, p.init_acc);
  }
  return cudaGetLastError();
}

cudaError_t launch_init_hash(Ctx* c, cudaStream_t s) {
  const Params& p = c->p;
  cudaError_t e = cudaMemsetAsync(p.hkeys, 0xFF, sizeof(uint64_t) * (size_t)c->total_rows, s);
  if (e != cudaSuccess) return e;
  const int64_t nw = c->total_rows * p.D;
  const int64_t nacc = c->total_rows * (p.rowwise ? 1 : p.D);
  {
    LaunchScope ls(c, K_INIT_HASH, s);
    if (p.bf16)
      k_fill<true><<<grid_for(c, nw, 256, 16), 256, 0, s>>>(p.table, nw, c->cfg.hash_init);
    else
      k_fill<false><<<grid_for(c, nw, 256, 16), 256, 0, s>>>(p.table, nw, c->cfg.hash_init);
  }
  {
    LaunchScope ls(c, K_INIT_HASH, s);
    k_fill<false><<<grid_for(c, nacc, 256, 16), 256, 0, s>>>(p.acc, nacc, p.init_acc);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------ dedup set reset

// Free the set slots claimed by the last forward (slots of unique rows 0..U-1).
__global__ void k_reset_set(Params p, int64_t max_unique) {
  const uint32_t U = p.counters[kU];
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < U && u < max_unique;
       u += (int64_t)gridDim.x * blockDim.x)
  {
    p.set_keys[p.uniq_slot[u]] = kEmpty32;
    p.uniq_once[u] = 0;
  }
}

cudaError_t launch_reset_set(Ctx* c, cudaStream_t s) {
  LaunchScope ls(c, K_RESET_SET, s);
  k_reset_set<<<grid_for(c, c->max_lookups, 256), 256, 0, s>>>(c->p, c->max_lookups);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ map + dedup

// Bag of every lookup (multi-hot): eight lanes per bag, lane j storing entries j, j+8, ...
// of the bag's range, so each store instruction writes whole 32-byte segments (one thread
// per bag wrote 32 scattered words per instruction: 0.043 -> 0.017 ms on the multi-hot
// batch of 8.5M lookups).  A bag whose offsets are negative, decreasing or beyond nnz raises
// EMB_FLAG_BAD_OFFSETS and owns no lookup.
__global__ void k_expand_bags(Params p, const int32_t* offs, int64_t nbags, int64_t nnz) {
  const int sub = threadIdx.x & 7;
  const int64_t stride = ((int64_t)gridDim.x * blockDim.x) >> 3;
  for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 3; b < nbags; b += stride) {
    const int64_t beg = offs[b], end = offs[b + 1];
    if (beg < 0 || end < beg || end > nnz) {
      if (sub == 0) raise_flag(p.counters, EMB_FLAG_BAD_OFFSETS);
      continue;
    }
    for (int64_t i = beg + sub; i < end; i += 8) p.bag_of[i] = (uint32_t)b;
  }
}

// Find `key` in the hashed table or claim a slot for it, for every lane of a warp that has a
// key (`want`); all 32 lanes must call together.  Returns the slot or kNoRow
// (EMB_FLAG_TABLE_FULL) when the first kMaxProbe slots of its chain hold other keys.
//
// Linear probing: a probe passes live keys and tombstones (evicted slots) and ends at a free
// slot or after the whole probe range; an absent key then claims the first tombstone it
// passed, else that free slot, by CAS.  Inserts never run alongside an eviction, so slots
// only fill during a batch and no key can land before the first free slot a complete probe
// saw: when the CAS loses to another key, probing resumes right after the contested slot.
// Every lost CAS means one more slot of the probe range has been filled for good, so the
// probe ends after at most `limit` of them.
//
// Warp-cooperative: each lane first reads its key's home slot (one sector per key; at the
// load factors the workloads run at, most keys end there: found, or inserted into a free
// home slot).  Keys still unresolved -- a collision or a tombstone at home -- are then taken
// one at a time by the whole warp, which reads 32 consecutive slots per step (one coalesced
// 256-byte load), finds the first match, tombstone and free slot with ballots, and lets one
// lane do the CAS.
__device__ __forceinline__ uint32_t find_or_insert(const Params& p, uint64_t key, bool want,
                                                   bool& inserted, bool flag_full = true) {
  inserted = false;
  constexpr uint64_t kNone = ~0ull;
  const int lane = threadIdx.x & 31;
  const uint64_t limit = (p.hmask + 1 < (uint64_t)kMaxProbe) ? p.hmask + 1 : (uint64_t)kMaxProbe;
  volatile uint64_t* keys = reinterpret_cast<volatile uint64_t*>(p.hkeys);
  const uint64_t h0 = want ? (mix64(key) & p.hmask) : 0;
  uint32_t slot = kNoRow;
  bool open = false;  // unresolved after the home probe
  if (want) {
    const uint64_t k = keys[h0];
    if (k == key) {
      slot = (uint32_t)h0;
    } else if (k == kEmpty64) {
      const uint64_t prev = atomicCAS(reinterpret_cast<unsigned long long*>(p.hkeys + h0),
                                      (unsigned long long)kEmpty64, (unsigned long long)key);
      if (prev == kEmpty64) {
        slot = (uint32_t)h0;
        inserted = true;
      } else if (prev == key) {
        slot = (uint32_t)h0;
      } else {
        open = true;
      }
    } else {
      open = true;
    }
  }
  for (unsigned m = __ballot_sync(0xFFFFFFFFu, open); m; m &= m - 1) {
    const int leader = __ffs(m) - 1;
    const uint64_t kk = __shfl_sync(0xFFFFFFFFu, key, leader);
    const uint64_t hh = __shfl_sync(0xFFFFFFFFu, h0, leader);
    uint64_t i0 = 0;        // first probe position of the current window
    uint64_t tomb = kNone;  // first tombstone passed since the last resume
    uint32_t res = kNoRow;
    bool ins = false, done = false;
    for (uint64_t lost = 0; lost <= limit && !done;) {
      if (i0 >= limit) {  // the whole probe range holds other keys (or tombstones)
        if (tomb == kNone) break;
        uint64_t prev = 0;
        if (lane == 0)
          prev = atomicCAS(reinterpret_cast<unsigned long long*>(p.hkeys + ((hh + tomb) & p.hmask)),
                           (unsigned long long)kTomb64, (unsigned long long)kk);
        prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
        if (prev == kTomb64 || prev == kk) {
          res = (uint32_t)((hh + tomb) & p.hmask);
          ins = prev == kTomb64;
          done = true;
        } else {
          ++lost;
          i0 = tomb + 1;
          tomb = kNone;
        }
        continue;
      }
      const uint64_t i = i0 + (uint64_t)lane;
      const uint64_t k = i < limit ? keys[(hh + i) & p.hmask] : kk ^ 1u;  // past the range: no hit
      const unsigned emp = __ballot_sync(0xFFFFFFFFu, i < limit && k == kEmpty64);
      // only slots before the first free one belong to the chain
      const unsigned before = emp ? ((1u << (__ffs(emp) - 1)) - 1u) : 0xFFFFFFFFu;
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, i < limit && k == kk) & before;
      if (hit) {
        res = (uint32_t)((hh + i0 + (uint64_t)(__ffs(hit) - 1)) & p.hmask);
        done = true;
        break;
      }
      const unsigned tb = __ballot_sync(0xFFFFFFFFu, i < limit && k == kTomb64) & before;
      if (tomb == kNone && tb) tomb = i0 + (uint64_t)(__ffs(tb) - 1);
      if (!emp) {
        i0 += 32;
        continue;
      }
      // absent: claim the first tombstone passed, else the free slot
      const uint64_t j = tomb != kNone ? tomb : i0 + (uint64_t)(__ffs(emp) - 1);
      const uint64_t expect = tomb != kNone ? kTomb64 : kEmpty64;
      uint64_t prev = 0;
      if (lane == 0)
        prev = atomicCAS(reinterpret_cast<unsigned long long*>(p.hkeys + ((hh + j) & p.hmask)),
                         (unsigned long long)expect, (unsigned long long)kk);
      prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
      if (prev == expect || prev == kk) {
        res = (uint32_t)((hh + j) & p.hmask);
        ins = prev == expect;
        done = true;
      } else {
        ++lost;  // another key took the slot: resume right after it
        i0 = j + 1;
        tomb = kNone;
      }
    }
    if (lane == leader) {
      slot = res;
      inserted = ins;
      if (res == kNoRow && flag_full) raise_flag(p.counters, EMB_FLAG_TABLE_FULL);
    }
  }
  return slot;
}

constexpr int kSmallProbes = 64;  // probe window of the dedup set's small region

// Per lookup: row number (static: base[t] + id after a range check; hashed: the slot of
// the key, inserting it if new), then the row's slot in the dedup set.  Winners of a set
// slot get consecutive unique numbers, one atomicAdd per block.  With mark_multi (rows below
// 2^31 only), a lookup that finds its row already in the set sets kSetMulti in the slot's
// key: the key is in place before any lookup can find it, so the mark is never lost, and the
// probe compares keys with the mark masked off.
__global__ void __launch_bounds__(256) k_map_dedup(Params p, const int64_t* ids, int64_t nnz,
                                                   int one_hot, int mark_multi) {
  __shared__ uint32_t warp_base[8];
  __shared__ uint32_t block_base;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x; i0 < nnz;
       i0 += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = i0 + threadIdx.x;
    uint32_t row = kNoRow;
    bool fresh = false;  // tiered: this lookup brought its row into the cache
    uint64_t key = 0;    // hashed key, or global row of a tiered table, to find or insert
    bool want = false;
    if (i < nnz) {
      const uint32_t bag = one_hot ? (uint32_t)i : p.bag_of[i];
      if (bag != kNoRow) {
        const int64_t id = ids[i];
        if (!p.hashed) {
          const int t = (int)(bag % (uint32_t)p.T);
          const int64_t b0 = p.base[t], n = p.base[t + 1] - b0;
          if (id < 0 || id >= n) {
            raise_flag(p.counters, EMB_FLAG_ID_RANGE);
          } else if (!p.tiered) {
            row = (uint32_t)(b0 + id);
          } else {
            key = (uint64_t)(b0 + id);
            want = true;
          }
        } else {
          if (id < 0) {
            raise_flag(p.counters, EMB_FLAG_BAD_KEY);
          } else {
            key = (uint64_t)id;
            want = true;
          }
        }
      }
    }
    if (p.hashed || p.tiered) {  // the whole warp probes together
      const uint32_t r = find_or_insert(p, key, want, fresh);
      if (want) row = r;
    }
    if (i < nnz) p.row_of[i] = row;
    if (p.tiered) {  // list the cache slots to fill from the host tier (one atomicAdd per warp)
      const unsigned nb = __ballot_sync(0xFFFFFFFFu, fresh && row != kNoRow);
      if (nb) {
        const int leader = __ffs(nb) - 1;
        uint32_t base = 0;
        if (lane == leader) base = atomicAdd(p.counters + kFill, (uint32_t)__popc(nb));
        base = __shfl_sync(0xFFFFFFFFu, base, leader);
        if (fresh && row != kNoRow) p.fill_list[base + __popc(nb & ((1u << lane) - 1u))] = row;
      }
    }
    bool won = false;
    uint32_t sslot = kEmpty32, seen = 0u;
    if (row != kNoRow) {
      const uint32_t marked = mark_multi ? (row | kSetMulti) : row;
      // slot h holds the row, or takes it: the probe ends there
      auto visit = [&](uint32_t h) {
        const uint32_t k = reinterpret_cast<volatile uint32_t*>(p.set_keys)[h];
        if (k == row || k == marked) {
          sslot = h;
          seen = k;
          return true;
        }
        if (k == kEmpty32) {
          const uint32_t prev = atomicCAS(p.set_keys + h, kEmpty32, row);
          if (prev == kEmpty32) {
            won = true;
            sslot = h;
            return true;
          }
          if (prev == row || prev == marked) {
            sslot = h;
            seen = prev;
            return true;
          }
        }
        return false;
      };
      bool done = false;
      // the small region first (a window of kSmallProbes slots); slots only ever fill during
      // the pass, so every lookup of a row finds the same window full or stops in it at the
      // same row, and a row that finds the window full lives in the large region
      if (p.ssmall) {
        uint32_t h = mix32(row) & (p.ssmall - 1u);
        for (int n = 0; n < kSmallProbes && !done; ++n) {
          done = visit(h);
          h = (h + 1u) & (p.ssmall - 1u);
        }
      }
      if (!done) {
        uint32_t h = mix32(row ^ 0x9E3779B9u) & p.smask;
        for (uint32_t n = 0; n <= p.smask && !done; ++n) {
          done = visit(p.ssmall + h);
          h = (h + 1u) & p.smask;
        }
      }
    }
    if (i < nnz) p.slot_of[i] = sslot;
    // a second lookup of the row: mark the slot once (most repeats see the mark and skip)
    if (mark_multi && !won && sslot != kEmpty32 && !(seen & kSetMulti))
      atomicOr(p.set_keys + sslot, kSetMulti);
    const unsigned ball = __ballot_sync(0xFFFFFFFFu, won);
    if (lane == 0) warp_base[wid] = __popc(ball);
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t tot = 0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
        const uint32_t cw = warp_base[w];
        warp_base[w] = tot;
        tot += cw;
      }
      block_base = tot ? atomicAdd(p.counters + kU, tot) : 0u;
    }
    __syncthreads();
    if (won) {
      const uint32_t u = block_base + warp_base[wid] + __popc(ball & ((1u << lane) - 1u));
      p.set_vals[sslot] = u;
      p.uniq_row[u] = row;
      p.uniq_slot[u] = sslot;
    }
    __syncthreads();
  }
}

cudaError_t launch_map_dedup(Ctx* c, const int64_t* ids, const int32_t* offs, int64_t nnz,
                             int64_t batch, cudaStream_t s) {
  cudaError_t e;
  if (c->set_dirty) {  // slots of the previous batch (freed by index, whatever its set size)
    e = launch_reset_set(c, s);
    if (e != cudaSuccess) return e;
    c->set_dirty = false;
  }
  // The batch probes only the part of the dedup set it can fill at most half of (a power of
  // two >= 2 nnz): a multi-hot batch of 8.5M lookups uses 32M of the 128M slots allocated
  // for its largest possible size, so its probes touch fewer sectors and pages.  Every
  // kernel of the step sees the same mask.
  int64_t cap = 1024;
  while (cap < 2 * nnz && cap < c->set_cap) cap <<= 1;
  cap = std::min<int64_t>(cap, c->set_cap);
  // In front of it, where the allocation has room, a small region of at least four slots
  // per unique row of the previous batch (from the host mirror), which stays in L2: most
  // rows are found or placed there, and a row whose window there is full goes to the large
  // region, so the set never overflows whatever the batch.
  int64_t small = 0;
  const uint32_t u_prev = c->h_unique ? *reinterpret_cast<volatile const uint32_t*>(c->h_unique) : 0u;
  if (u_prev > 0) {
    small = 1024;
    while (small < 4 * (int64_t)u_prev) small <<= 1;
    if (small >= cap || small + cap > c->set_cap) small = 0;
  }
  c->p.ssmall = (uint32_t)small;
  c->p.smask = (uint32_t)(cap - 1);
  const Params& p = c->p;
  if (p.tiered && c->pf_pending) {  // rows prefetched for this batch are in before it looks
    e = cudaStreamWaitEvent(s, c->ev_prefetch, 0);
    if (e != cudaSuccess) return e;
    c->pf_pending = false;
  }
  e = cudaMemsetAsync(p.counters + kU, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess && p.tiered) e = cudaMemsetAsync(p.counters + kFill, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  const int64_t nbags = batch * p.T;
  if (offs) {
    e = cudaMemcpyAsync(p.offs, offs, sizeof(int32_t) * (size_t)(nbags + 1),
                        cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(p.bag_of, 0xFF, sizeof(uint32_t) * (size_t)nnz, s);
    if (e != cudaSuccess) return e;
    LaunchScope ls(c, K_EXPAND_BAGS, s);
    k_expand_bags<<<grid_for(c, nbags * 8, 256), 256, 0, s>>>(p, p.offs, nbags, nnz);
  }
  if (nnz > 0) {
    LaunchScope ls(c, K_MAP_DEDUP, s);
    k_map_dedup<<<grid_for(c, nnz, 256), 256, 0, s>>>(p, ids, nnz, offs ? 0 : 1,
                                                       c->once_step ? 1 : 0);
  }
  c->set_dirty = true;
  e = cudaGetLastError();
  if (e == cudaSuccess && p.tiered && nnz > 0) e = launch_tier_fill(c, nnz, s);
  // tiered: the cache holds this batch's rows from here on; a prefetch may start
  if (e == cudaSuccess && p.tiered) e = cudaEventRecord(c->ev_dedup, s);
  return e;
}

// Unique index of every lookup (after k_map_dedup has numbered the unique rows).
// (four lookups per thread, their loads issued together)  With mark_once, the only lookup
// of a row (its set key unmarked) carries kInvOnce and sets uniq_once[u] (zero otherwise;
// the update kernel or the set reset clears it again).  Block 0 also copies U into the
// host-mapped mirror.
__global__ void k_inverse(Params p, int64_t nnz, int mark_once, uint32_t* h_unique) {
  constexpr int kILP = 4;
  const int64_t span = (int64_t)blockDim.x * kILP;
  if (h_unique && blockIdx.x == 0 && threadIdx.x == 0)
    *reinterpret_cast<volatile uint32_t*>(h_unique) = p.counters[kU];
  for (int64_t q0 = (int64_t)blockIdx.x * span; q0 < nnz; q0 += (int64_t)gridDim.x * span) {
    uint32_t sl[kILP], rw[kILP];
#pragma unroll
    for (int j = 0; j < kILP; ++j) {
      const int64_t q = q0 + j * blockDim.x + threadIdx.x;
      sl[j] = q < nnz ? p.slot_of[q] : kEmpty32;
      rw[j] = q < nnz ? p.row_of[q] : kNoRow;
    }
#pragma unroll
    for (int j = 0; j < kILP; ++j) {
      const int64_t q = q0 + j * blockDim.x + threadIdx.x;
      if (q >= nnz) continue;
      uint32_t iv = kNoRow;
      if (rw[j] != kNoRow && sl[j] != kEmpty32) {
        iv = p.set_vals[sl[j]];
        if (mark_once && !(p.set_keys[sl[j]] & kSetMulti)) {
          p.uniq_once[iv] = 1;
          iv |= kInvOnce;
        }
      }
      p.inv[q] = iv;
    }
  }
}

cudaError_t launch_inverse(Ctx* c, int64_t nnz, cudaStream_t s) {
  if (nnz <= 0) return cudaSuccess;
  LaunchScope ls(c, K_INVERSE, s);
  k_inverse<<<grid_for(c, (nnz + 3) / 4, 256), 256, 0, s>>>(c->p, nnz, c->once_step ? 1 : 0,
                                                            c->h_unique_dev);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ read-back kernels

// Occurrence counts per unique row and the key of each unique row (hashed: the int64
// key of the slot; static: the global row).
__global__ void k_unique_count(Params p, int64_t nnz, uint32_t* counts, int64_t* keys) {
  const uint32_t U = p.counters[kU];
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nnz; i += stride) {
    const uint32_t sl = p.slot_of[i];
    if (p.row_of[i] != kNoRow && sl != kEmpty32) atomicAdd(counts + p.set_vals[sl], 1u);
  }
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < U; u += stride) {
    const uint32_t r = p.uniq_row[u];
    keys[u] = (p.hashed || p.tiered) ? (int64_t)p.hkeys[r] : (int64_t)r;
  }
}

// counts: zeroed [>= U] device buffer; keys: [>= U] device buffer
cudaError_t launch_unique_count(Ctx* c, int64_t nnz, uint32_t* counts, int64_t* keys,
                                cudaStream_t s) {
  LaunchScope ls(c, K_UNIQUE_COUNT, s);
  k_unique_count<<<grid_for(c, nnz > 0 ? nnz : 1, 256), 256, 0, s>>>(c->p, nnz, counts, keys);
  return cudaGetLastError();
}

__global__ void k_read_rows(Params p, const uint32_t* rows, int64_t n, float* w, float* acc) {
  const int AW = p.rowwise ? 1 : p.D;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n * p.D; e += stride) {
    const int64_t q = e / p.D;
    const int col = (int)(e - q * p.D);
    const uint32_t r = rows[q];
    float v = 0.0f;
    if (r != kNoRow) {
      const int64_t off = (int64_t)r * p.D + col;
      v = p.bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.table)[off])
                 : reinterpret_cast<const float*>(p.table)[off];
    }
    w[e] = v;
  }
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n * AW; e += stride) {
    const int64_t q = e / AW;
    const int col = (int)(e - q * AW);
    const uint32_t r = rows[q];
    acc[e] = (r != kNoRow) ? p.acc[(int64_t)r * AW + col] : 0.0f;
  }
}

cudaError_t launch_read_rows(Ctx* c, const uint32_t* rows, int64_t n, float* w, float* acc,
                             cudaStream_t s) {
  LaunchScope ls(c, K_READ_ROWS, s);
  k_read_rows<<<grid_for(c, n * c->p.D, 256), 256, 0, s>>>(c->p, rows, n, w, acc);
  return cudaGetLastError();
}

// Find-only probe of the hashed table.
__global__ void k_find_keys(Params p, const int64_t* keys, int64_t n, uint32_t* rows) {
  for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n;
       q += (int64_t)gridDim.x * blockDim.x) {
    const int64_t key = keys[q];
    uint32_t found = kNoRow;
    if (key >= 0) {
      uint64_t h = mix64((uint64_t)key) & p.hmask;
      const uint64_t limit = (p.hmask + 1 < (uint64_t)kMaxProbe) ? p.hmask + 1 : (uint64_t)kMaxProbe;
      for (uint64_t m = 0; m < limit; ++m) {
        const uint64_t k = p.hkeys[h];
        if (k == (uint64_t)key) {
          found = (uint32_t)h;
          break;
        }
        if (k == kEmpty64) break;
        h = (h + 1) & p.hmask;
      }
    }
    rows[q] = found;
  }
}

cudaError_t launch_find_keys(Ctx* c, const int64_t* keys, int64_t n, uint32_t* rows,
                             cudaStream_t s) {
  LaunchScope ls(c, K_READ_ROWS, s);
  k_find_keys<<<grid_for(c, n, 256), 256, 0, s>>>(c->p, keys, n, rows);
  return cudaGetLastError();
}

// Compact the slots of the hashed table that hold a key.
__global__ void k_export_hash(Params p, int64_t cap, int64_t* keys, uint32_t* rows,
                              uint32_t* count) {
  for (int64_t h = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; h <= (int64_t)p.hmask;
       h += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t k = p.hkeys[h];
    if (k != kEmpty64 && k != kTomb64) {
      const uint32_t idx = atomicAdd(count, 1u);
      if (idx < cap) {
        keys[idx] = (int64_t)k;
        rows[idx] = (uint32_t)h;
      }
    }
  }
}

cudaError_t launch_export_hash(Ctx* c, int64_t cap, int64_t* keys, uint32_t* rows, uint32_t* count,
                               cudaStream_t s) {
  LaunchScope ls(c, K_EXPORT_HASH, s);
  k_export_hash<<<grid_for(c, c->total_rows, 256), 256, 0, s>>>(c->p, cap, keys, rows,
                                                                count);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ admission / eviction
// DeepRec announcement, "EmbeddingVariable": feature admission and eviction strategies are
// named there, not defined.  Reading taken: a hashed key counts its lookups over all steps
// and its row takes a step's update only once the count (this step included) reaches the
// admission minimum; an eviction between steps removes keys idle for more than a number of
// steps or counted fewer than a minimum, and their slots start afresh.

// Per unique key of the step: add its lookups (cnt[u]) to the slot's count (saturating),
// stamp the step, and hold the update while the count is below the admission minimum.
__global__ void k_admit(Params p, uint32_t step) {
  const uint32_t U = p.counters[kU];
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < U;
       u += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t slot = p.uniq_row[u];
    const uint32_t c = p.cnt[u], f0 = (uint32_t)p.hstat[slot];
    const uint32_t f = f0 > 0xFFFFFFFFu - c ? 0xFFFFFFFFu : f0 + c;
    p.hstat[slot] = ((uint64_t)step << 32) | f;
    p.uniq_hold[u] = (p.admit_min > 1 && f < p.admit_min) ? 1 : 0;
  }
}

cudaError_t launch_admit(Ctx* c, cudaStream_t s) {
  LaunchScope ls(c, K_ADMIT, s);
  k_admit<<<grid_for(c, std::max<int64_t>(1, std::min<int64_t>(c->max_lookups, c->total_rows)),
                     256), 256, 0, s>>>(c->p, c->step);
  return cudaGetLastError();
}

// Between steps: a slot whose key is idle for more than max_idle steps (max_idle > 0) or
// counted fewer than min_count times becomes a tombstone; its row and accumulator return to
// their initial values and its counters to zero.  Each thread streams four consecutive
// slots per iteration (16-byte loads of keys and counters, all issued before any test);
// evictions are counted in counters[kEvicted] (one atomicAdd per warp).  Tiered tables
// write each evicted row back with the whole warp (one thread per row scattered its 16-byte
// stores over the host link).
template <bool BF16>
__device__ __forceinline__ void reset_slot(const Params& p, int64_t h, float hash_init) {
  const int AW = p.rowwise ? 1 : p.D;
  p.hkeys[h] = kTomb64;
  p.hstat[h] = 0;
  if (BF16) {
    __nv_bfloat16* w = reinterpret_cast<__nv_bfloat16*>(p.table) + h * p.D;
    const __nv_bfloat16 v = __float2bfloat16_rn(hash_init);
    for (int c = 0; c < p.D; ++c) w[c] = v;
  } else {
    float4* w = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.table) + h * p.D);
    for (int c = 0; c < p.D / 4; ++c) w[c] = make_float4(hash_init, hash_init, hash_init, hash_init);
  }
  float* a = p.acc + h * AW;
  for (int c = 0; c < AW; ++c) a[c] = p.init_acc;
}

// Tiered tables: copy the cached row of slot h (global row `key`) back to the host tier.
template <bool BF16>
__device__ __forceinline__ void write_back(const Params& p, int64_t h, uint64_t key) {
  const int AW = p.rowwise ? 1 : p.D;
  const int nw = p.D * (BF16 ? 2 : 4) / 16;  // 16-byte chunks of a stored row
  const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(p.table) + h * nw * 16);
  uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<char*>(p.htable) + (int64_t)key * nw * 16);
  for (int c = 0; c < nw; ++c) dst[c] = src[c];
  for (int c = 0; c < AW; ++c) p.hacc[(int64_t)key * AW + c] = p.acc[h * AW + c];
}

// The same, by the 32 lanes of a warp together: 16-byte chunks and accumulator words
// spread over the lanes, so each store to the host tier is one coalesced line.
template <bool BF16>
__device__ __forceinline__ void write_back_warp(const Params& p, int64_t h, uint64_t key,
                                                int lane) {
  const int AW = p.rowwise ? 1 : p.D;
  const int nw = p.D * (BF16 ? 2 : 4) / 16;
  const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(p.table) + h * nw * 16);
  uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<char*>(p.htable) + (int64_t)key * nw * 16);
  for (int c = lane; c < nw; c += 32) dst[c] = src[c];
  for (int c = lane; c < AW; c += 32) p.hacc[(int64_t)key * AW + c] = p.acc[h * AW + c];
}

// A hashed table's slot h back to the initial values, by the whole warp (coalesced stores;
// the key and statistics words are left to the caller).
template <bool BF16>
__device__ __forceinline__ void reset_row_warp(const Params& p, int64_t h, float hash_init,
                                               int lane) {
  const int AW = p.rowwise ? 1 : p.D;
  const int nw = p.D * (BF16 ? 2 : 4) / 16;  // 16-byte chunks of a stored row
  uint4 fill;
  if (BF16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(hash_init, hash_init);
    const uint32_t b = *reinterpret_cast<const uint32_t*>(&v);
    fill = make_uint4(b, b, b, b);
  } else {
    const uint32_t b = __float_as_uint(hash_init);
    fill = make_uint4(b, b, b, b);
  }
  uint4* w = reinterpret_cast<uint4*>(reinterpret_cast<char*>(p.table) + h * nw * 16);
  for (int c = lane; c < nw; c += 32) w[c] = fill;
  for (int c = lane; c < AW; c += 32) p.acc[h * AW + c] = p.init_acc;
}

// Evict the key of slot h: a tiered table writes the row back to the host tier (the next
// insert fills the slot from there); a hashed table resets it to the initial values.
template <bool BF16>
__device__ __forceinline__ void evict_slot(const Params& p, int64_t h, uint64_t key,
                                           float hash_init) {
  if (p.tiered) {
    write_back<BF16>(p, h, key);
    p.hkeys[h] = kTomb64;
    p.hstat[h] = 0;
  } else {
    reset_slot<BF16>(p, h, hash_init);
  }
}

__device__ __forceinline__ bool evictable(uint64_t k, uint64_t st, uint32_t step,
                                          uint32_t max_idle, uint32_t min_count, int exact_idle) {
  if (k == kEmpty64 || k == kTomb64) return false;
  // a prefetched row may carry the next step's number (counted as idle 0 until then)
  const int32_t d = (int32_t)(step - (uint32_t)(st >> 32));
  const bool idle = (exact_idle || max_idle > 0) && d > 0 && (uint32_t)d > max_idle;
  return idle || (uint32_t)st < min_count;
}

// thr_dev: the watermark variant -- evict keys idle for more than counters[kThresh] steps
// (any count), nothing when that word is all ones.
template <bool BF16>
__global__ void k_evict(Params p, uint32_t step, uint32_t max_idle, uint32_t min_count,
                        float hash_init, int thr_dev) {
  __shared__ uint32_t blk_n;  // evictions of the block, added to the counters once at the end
  const int lane = threadIdx.x & 31;
  if (thr_dev) {
    const uint32_t t = p.counters[kThresh];
    if (t == 0xFFFFFFFFu) return;
    min_count = 0;
    max_idle = t;  // idle > t (t = 0 allowed: keys not looked up in the current step)
  }
  if (threadIdx.x == 0) blk_n = 0;
  __syncthreads();
  const int64_t nslots = (int64_t)p.hmask + 1;
  const int64_t nquads = nslots / 4;  // capacities are powers of two: whole quads from 4 on
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t q0 = (int64_t)blockIdx.x * blockDim.x; q0 < nquads; q0 += stride) {
    const int64_t q = q0 + threadIdx.x;
    uint32_t n = 0;
    bool ev[4] = {false, false, false, false};
    uint64_t key[4] = {0, 0, 0, 0};
    if (q < nquads) {
      const ulonglong2* kp = reinterpret_cast<const ulonglong2*>(p.hkeys) + 2 * q;
      const ulonglong2* sp = reinterpret_cast<const ulonglong2*>(p.hstat) + 2 * q;
      const ulonglong2 k01 = kp[0], k23 = kp[1], s01 = sp[0], s23 = sp[1];
      const uint64_t k[4] = {k01.x, k01.y, k23.x, k23.y};
      const uint64_t st[4] = {s01.x, s01.y, s23.x, s23.y};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        ev[j] = evictable(k[j], st[j], step, max_idle, min_count, thr_dev);
        key[j] = k[j];
        n += ev[j] ? 1u : 0u;
      }
    }
    // the whole warp handles each evicted row in turn (coalesced 16-byte stores): tiered
    // tables copy it back to the host tier, hashed tables reset it (one thread per row
    // wrote 32 scattered words per store instruction)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      for (unsigned m = __ballot_sync(0xFFFFFFFFu, ev[j]); m; m &= m - 1) {
        const int src = __ffs(m) - 1;
        const int64_t h = 4 * __shfl_sync(0xFFFFFFFFu, q, src) + j;
        const uint64_t kh = __shfl_sync(0xFFFFFFFFu, key[j], src);
        if (p.tiered) write_back_warp<BF16>(p, h, kh, lane);
        else reset_row_warp<BF16>(p, h, hash_init, lane);
      }
      if (ev[j]) {
        p.hkeys[4 * q + j] = kTomb64;
        p.hstat[4 * q + j] = 0;
      }
    }
    n = __reduce_add_sync(0xFFFFFFFFu, n);
    if (lane == 0 && n) atomicAdd(&blk_n, n);
  }
  // one global atomic per block: one per warp and iteration serialised on the counter's L2
  // slice when many keys of a large table are evicted (64M slots: 0.51 -> 0.24 ms a call)
  __syncthreads();
  if (threadIdx.x == 0 && blk_n) {
    atomicAdd(p.counters + kEvicted, blk_n);
    if (p.tiered) atomicSub(p.counters + kOcc, blk_n);
  }
  // tables of fewer than four slots
  if (blockIdx.x == 0 && threadIdx.x < nslots - 4 * nquads) {
    const int64_t h = 4 * nquads + threadIdx.x;
    if (evictable(p.hkeys[h], p.hstat[h], step, max_idle, min_count, thr_dev)) {
      evict_slot<BF16>(p, h, p.hkeys[h], hash_init);
      atomicAdd(p.counters + kEvicted, 1u);
      if (p.tiered) atomicSub(p.counters + kOcc, 1u);
    }
  }
}

cudaError_t launch_evict(Ctx* c, uint32_t max_idle, uint32_t min_count, cudaStream_t s) {
  LaunchScope ls(c, K_EVICT, s);
  const int grid = grid_for(c, std::max<int64_t>(1, c->total_rows / 4), 256, 8);
  if (c->p.bf16)
    k_evict<true><<<grid, 256, 0, s>>>(c->p, c->step, max_idle, min_count, c->cfg.hash_init, 0);
  else
    k_evict<false><<<grid, 256, 0, s>>>(c->p, c->step, max_idle, min_count, c->cfg.hash_init, 0);
  return cudaGetLastError();
}

// Count and last step of the slots rows[q] (kNoRow: 0, 0).
__global__ void k_key_stats(Params p, const uint32_t* rows, int64_t n, uint32_t* freq,
                            uint32_t* last) {
  for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n;
       q += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t r = rows[q];
    const uint64_t st = r == kNoRow ? 0ull : p.hstat[r];
    freq[q] = (uint32_t)st;
    last[q] = (uint32_t)(st >> 32);
  }
}

cudaError_t launch_key_stats(Ctx* c, const uint32_t* rows, int64_t n, uint32_t* freq,
                             uint32_t* last, cudaStream_t s) {
  LaunchScope ls(c, K_READ_ROWS, s);
  k_key_stats<<<grid_for(c, n > 0 ? n : 1, 256), 256, 0, s>>>(c->p, rows, n, freq, last);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ tiered tables
// Tiered storage (a step beyond the pages' single tier; HugeCTR interview and Merlin article
// stress that embedding tables outgrow device memory): the static tables and their
// accumulators live in host memory that the GPU reads and writes directly (host-mapped,
// over NVLink-C2C on Grace systems); HBM holds a cache of `cache rows` rows indexed by the
// hashed-table machinery with the global row as key.  Dedup lists the cache slots a batch
// claims for rows it did not find; this kernel copies those rows in from the host tier
// before any kernel reads them, one warp per row (16-byte chunks).  Eviction writes rows
// back (k_evict), so the host tier plus the cache always hold the table's current values.
// cidx: the counter holding the list length (kFill for a step's own rows, kPfFill for a
// prefetch); stamp: the last step recorded for the rows brought in (0: counted later by the
// step's own bookkeeping).  Every row brought in adds one to the cache occupancy.
__global__ void __launch_bounds__(256) k_tier_fill(Params p, int cidx, uint32_t stamp) {
  const int lane = threadIdx.x & 31;
  const uint32_t n = p.counters[cidx];
  if (blockIdx.x == 0 && threadIdx.x == 0 && n) atomicAdd(p.counters + kOcc, n);
  const int AW = p.rowwise ? 1 : p.D;
  const int nw = p.D * (p.bf16 ? 2 : 4) / 16;
  const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t j = gwarp; j < n; j += nwarps) {
    const uint32_t slot = p.fill_list[j];
    const uint64_t key = p.hkeys[slot];
    const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(p.htable) + (int64_t)key * nw * 16);
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<char*>(p.table) + (int64_t)slot * nw * 16);
    for (int c = lane; c < nw; c += 32) dst[c] = src[c];
    for (int c = lane; c < AW; c += 32) p.acc[(int64_t)slot * AW + c] = p.hacc[(int64_t)key * AW + c];
    if (lane == 0) p.hstat[slot] = (uint64_t)stamp << 32;
  }
}

cudaError_t launch_tier_fill(Ctx* c, int64_t max_new, cudaStream_t s) {
  LaunchScope ls(c, K_TIER_FILL, s);
  k_tier_fill<<<grid_for(c, max_new * 32, 256), 256, 0, s>>>(c->p, kFill, 0u);
  return cudaGetLastError();
}

// Prefetch (tiered tables): find or insert the cache slot of every valid lookup of a batch
// (rows of a later step) and list the slots claimed, so that k_tier_fill brings those rows
// in ahead of that step's forward.  Nothing of the pending step is touched: its own rows
// were inserted and filled by its forward before the prefetch starts.  A full cache is not
// flagged here (the step's own forward retries and flags).  Rows found cached get their
// last step raised to `stamp`, rows brought in start with it.  One-hot: one lookup per thread;
// multi-hot: one bag per thread, the warp's lanes walking their bags in step.
__global__ void __launch_bounds__(256) k_prefetch(Params p, const int64_t* ids,
                                                  const int32_t* offs, int64_t nnz,
                                                  int64_t nbags, uint32_t stamp) {
  const int lane = threadIdx.x & 31;
  const int64_t n = offs ? nbags : nnz;
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x; i0 < n; i0 += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = i0 + threadIdx.x;
    int64_t beg = 0, end = 0;
    int t = 0;
    if (i < n) {
      if (offs) {
        beg = offs[i];
        end = offs[i + 1];
        if (beg < 0 || end < beg || end > nnz) end = beg;  // malformed: the forward flags it
        t = (int)(i % p.T);
      } else {
        beg = i;
        end = i + 1;
        t = (int)(i % p.T);
      }
    }
    const int64_t len = end - beg;
    const int64_t most = __reduce_max_sync(0xFFFFFFFFu, (unsigned)(len < 0 ? 0 : len));
    for (int64_t k = 0; k < most; ++k) {
      bool want = false;
      uint64_t key = 0;
      if (k < len) {
        const int64_t id = ids[beg + k];
        const int64_t b0 = p.base[t], rows = p.base[t + 1] - b0;
        if (id >= 0 && id < rows) {
          key = (uint64_t)(b0 + id);
          want = true;
        }
      }
      bool fresh = false;
      const uint32_t slot = find_or_insert(p, key, want, fresh, false);
      // a row already cached counts as used at `stamp` too, so that no eviction before its
      // step takes it out (the last-step half of its statistics word only; a Zipf-hot row
      // sees the raised stamp after its first lookups and skips the atomic)
      if (want && !fresh && slot != kNoRow &&
          (uint32_t)(reinterpret_cast<volatile uint64_t*>(p.hstat)[slot] >> 32) < stamp)
        atomicMax(reinterpret_cast<unsigned int*>(p.hstat + slot) + 1, stamp);
      const unsigned nb = __ballot_sync(0xFFFFFFFFu, want && fresh && slot != kNoRow);
      if (nb) {
        const int leader = __ffs(nb) - 1;
        uint32_t base = 0;
        if (lane == leader) base = atomicAdd(p.counters + kPfFill, (uint32_t)__popc(nb));
        base = __shfl_sync(0xFFFFFFFFu, base, leader);
        if (want && fresh && slot != kNoRow) p.fill_list[base + __popc(nb & ((1u << lane) - 1u))] = slot;
      }
    }
  }
}

cudaError_t launch_prefetch(Ctx* c, const int64_t* ids, const int32_t* offs, int64_t nnz,
                            int64_t batch, uint32_t stamp, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(c->p.counters + kPfFill, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess || nnz <= 0) return e;
  const int64_t nbags = batch * c->p.T;
  {
    LaunchScope ls(c, K_PREFETCH, s);
    k_prefetch<<<grid_for(c, offs ? nbags : nnz, 256), 256, 0, s>>>(c->p, ids, offs, nnz, nbags,
                                                                      stamp);
  }
  LaunchScope ls(c, K_TIER_FILL, s);
  k_tier_fill<<<grid_for(c, nnz * 32, 256), 256, 0, s>>>(c->p, kPfFill, stamp);
  return cudaGetLastError();
}

// Watermark check (tiered tables), after a backward step: when more than `high` cache slots
// are in use, count the occupied slots by idle steps (current step - last step, bins 0..62
// and 63 for 63 or more), then pick the smallest threshold t such that evicting every key
// idle for more than t brings the occupancy to `low` or below (t = 0: every key the current
// step did not look up); k_evict (threshold variant) then writes those rows back.  Below the
// watermark the threshold stays all ones and both kernels return at once.
constexpr int kIdleBins = 64;

// Watermark check, first pass: below the high mark every block leaves after one load (block
// 0 first sets "nothing to evict"); above it the blocks count the cached rows by idle steps
// (per-block shared-memory histograms added into tier_hist), and the last block to finish
// (a completion counter; no block waits for another) picks the smallest threshold t whose
// eviction -- every row idle for more than t steps -- brings the occupancy to `low` or
// below (t = 0 if nothing less does), then clears the histogram and the counter.
__global__ void __launch_bounds__(256) k_tier_hist(Params p, uint32_t step, uint32_t high,
                                                   uint32_t low) {
  __shared__ uint32_t h[kIdleBins];
  __shared__ uint32_t occ;
  __shared__ bool last;
  if (threadIdx.x == 0) occ = p.counters[kOcc];
  for (int b = threadIdx.x; b < kIdleBins; b += blockDim.x) h[b] = 0;
  __syncthreads();
  if (occ <= high) {  // the whole block leaves together
    if (blockIdx.x == 0 && threadIdx.x == 0) p.counters[kThresh] = 0xFFFFFFFFu;
    return;
  }
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i <= (int64_t)p.hmask;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t k = p.hkeys[i];
    if (k == kEmpty64 || k == kTomb64) continue;
    const int32_t d = (int32_t)(step - (uint32_t)(p.hstat[i] >> 32));
    const uint32_t idle = d > 0 ? (uint32_t)d : 0u;
    atomicAdd(h + (idle < kIdleBins - 1 ? idle : kIdleBins - 1), 1u);
  }
  __syncthreads();
  for (int b = threadIdx.x; b < kIdleBins; b += blockDim.x)
    if (h[b]) atomicAdd(p.tier_hist + b, h[b]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(p.counters + kTierDone, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last || threadIdx.x != 0) return;
  __threadfence();
  const uint32_t need = occ - low;
  uint32_t freed = 0, t = 0;  // evicting every key idle for more than 0 steps frees the most
  volatile const uint32_t* hist = p.tier_hist;
  for (int b = kIdleBins - 1; b >= 1; --b) {
    freed += hist[b];
    if (freed >= need) {
      t = (uint32_t)(b - 1);
      break;
    }
  }
  p.counters[kThresh] = t;
  for (int b = 0; b < kIdleBins; ++b) p.tier_hist[b] = 0;
  p.counters[kTierDone] = 0;
}

cudaError_t launch_tier_watermark(Ctx* c, uint32_t high, uint32_t low, cudaStream_t s) {
  // grids of a few blocks per SM (grid-stride loops): below the mark, which most steps are,
  // each launch costs little more than its dispatch
  {
    LaunchScope ls(c, K_TIER_WATERMARK, s);
    k_tier_hist<<<2 * c->num_sms, 256, 0, s>>>(c->p, c->step, high, low);
  }
  LaunchScope ls(c, K_EVICT, s);
  const int grid = std::min(4 * c->num_sms, grid_for(c, std::max<int64_t>(1, c->total_rows / 4), 256, 8));
  if (c->p.bf16)
    k_evict<true><<<grid, 256, 0, s>>>(c->p, c->step, 0, 0, c->cfg.hash_init, 1);
  else
    k_evict<false><<<grid, 256, 0, s>>>(c->p, c->step, 0, 0, c->cfg.hash_init, 1);
  return cudaGetLastError();
}

}  // namespace emb
