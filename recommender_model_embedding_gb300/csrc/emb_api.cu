// Host side of the C ABI declared in include/emb.h: configuration checks, device memory
// layout, call ordering and stream-ordered launches.
//
// Device memory held by a context (all allocated in emb_create, nothing allocated per
// call except the host-step staging buffers on first use and temporaries of the
// synchronous read-back calls):
//   table    [R][D] fp32|bf16   R = sum of rows (static) or capacity (hashed)
//   acc      [R][D] or [R] fp32
//   hkeys    [capacity] int64   (hashed; all-ones = free)
//   base     [T+1] int64        (static; first global row of each table)
//   dedup set keys/vals [S] u32, S = pow2 >= 2*max_lookups
//   per lookup: row_of, slot_of, bag_of, inv, rank, s_u, s_row, s_bag   [max_lookups] u32
//   per unique: uniq_row, uniq_slot [max_lookups], cnt, seg [max_lookups+1] u32,
//               uniq_once, uniq_hold [max_lookups] u8
//   hashed: hstat [capacity] u64 (lookup count | last step << 32 of each slot's key)
//   h_unique  one host-mapped pinned u32 (U of the last deduplicated batch)
//   g        [min(max_lookups, R)][D] fp32, zero between steps
//   offs     [max_batch*T+1] int32 copy of the last offsets
#include <sys/mman.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "emb_internal.cuh"
#include "interact_common.cuh"

namespace emb {

const char* const kKernelNames[K_NUM_KERNELS] = {
    "init_table",     "init_hash",      "reset_set",   "expand_bags",       "map_dedup",
    "pool",           "interact_fwd",   "interact_bwd", "fused_fwd",        "fused_bwd",
    "inverse_count",  "scan_local",     "scan_blocks", "scan_add",          "fill_perm",
    "segreduce_adagrad", "adagrad_from_g", "unique_count", "read_rows",     "export_hash",
    "inverse",        "once_split",     "admit",       "evict",             "tier_fill",
    "prefetch",       "tier_watermark"};

static cudaEvent_t take_event(Ctx* c) {
  if (!c->ev_pool.empty()) {
    cudaEvent_t e = c->ev_pool.back();
    c->ev_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

LaunchScope::LaunchScope(Ctx* c_, int kid_, cudaStream_t s_) : c(c_), kid(kid_), s(s_) {
  c->launches += 1;
  if (c->prof_on) {
    cudaEvent_t a = take_event(c);
    b = take_event(c);
    cudaEventRecord(a, s);
    c->recs.push_back(Ctx::Rec{kid, a, b});
  }
}

LaunchScope::~LaunchScope() {
  if (b) cudaEventRecord(b, s);
}

int grid_for(const Ctx* c, int64_t work_items, int threads, int blocks_per_sm) {
  int64_t blocks = (work_items + threads - 1) / threads;
  const int64_t cap = (int64_t)c->num_sms * blocks_per_sm;
  if (blocks > cap) blocks = cap;
  return (int)(blocks < 1 ? 1 : blocks);
}

static void free_all(Ctx* c) {
  for (void* p : c->allocs) cudaFree(p);
  c->allocs.clear();
  for (auto& r : c->recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  c->recs.clear();
  for (cudaEvent_t e : c->ev_pool) cudaEventDestroy(e);
  c->ev_pool.clear();
  for (cudaEvent_t* e : {&c->ev_inputs, &c->ev_dout, &c->ev_fwd, &c->ev_out, &c->ev_dedup,
                         &c->ev_prefetch}) {
    if (*e) cudaEventDestroy(*e);
    *e = nullptr;
  }
  for (auto& row : c->ev_chunk)
    for (cudaEvent_t& e : row) {
      if (e) cudaEventDestroy(e);
      e = nullptr;
    }
  for (cudaStream_t* q : {&c->st_h2d, &c->st_d2h}) {
    if (*q) cudaStreamDestroy(*q);
    *q = nullptr;
  }
  if (c->h_unique) cudaFreeHost(c->h_unique);
  c->h_unique = c->h_unique_dev = nullptr;
  void* hosts[2] = {c->host_table, c->host_acc};
  for (int i = 0; i < 2; ++i) {
    if (!hosts[i]) continue;
    if (c->host_map[i]) {
      cudaHostUnregister(hosts[i]);
      munmap(c->host_map[i], c->host_map_len[i]);
    } else {
      cudaFreeHost(hosts[i]);
    }
    c->host_map[i] = nullptr;
  }
  c->host_table = nullptr;
  c->host_acc = nullptr;
}

// Host-tier memory: anonymous memory on transparent huge pages (asked for with madvise,
// the start aligned to the huge-page size), pinned and mapped for the device.  The device
// reaches host memory through its own address translation, which covers a few GB: random
// 512-byte rows spread over 64 GB came at 9.8 GB/s from cudaHostAlloc memory and at 20.8
// GB/s from huge pages (209 GB/s within 8 GB, either way; GB300 with 64 KB base pages and
// 512 MB huge pages).  Falls back to cudaHostAlloc where the mapping or the registration
// is refused.  Returns the pointer the host uses; *map / *len describe the mapping (null
// for the fallback).
static void* host_tier_alloc(size_t bytes, void** map, size_t* len) {
  *map = nullptr;
  *len = 0;
  size_t huge = 2u << 20;
  if (FILE* f = std::fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
    unsigned long long v = 0;
    if (std::fscanf(f, "%llu", &v) == 1 && v >= 4096 && (v & (v - 1)) == 0) huge = (size_t)v;
    std::fclose(f);
  }
  const size_t total = bytes + huge;
  void* m = mmap(nullptr, total, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
  if (m != MAP_FAILED) {
    char* p = reinterpret_cast<char*>(((uintptr_t)m + huge - 1) & ~(uintptr_t)(huge - 1));
    madvise(p, bytes, MADV_HUGEPAGE);  // advisory: small pages where none is free
    if (cudaHostRegister(p, bytes, cudaHostRegisterMapped) == cudaSuccess) {
      *map = m;
      *len = total;
      return p;
    }
    cudaGetLastError();
    munmap(m, total);
  }
  void* h = nullptr;
  if (cudaHostAlloc(&h, bytes, cudaHostAllocMapped) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return h;
}

template <typename T>
static bool dalloc(Ctx* c, T** p, size_t count) {
  void* q = nullptr;
  if (count == 0) count = 1;
  if (cudaMalloc(&q, count * sizeof(T)) != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    return false;
  }
  c->allocs.push_back(q);
  *p = reinterpret_cast<T*>(q);
  return true;
}

static int64_t next_pow2(int64_t x) {
  int64_t p = 1;
  while (p < x) p <<= 1;
  return p;
}

static bool interaction_shape_ok(const Ctx* c) {
  return c->p.T + 1 <= kMaxF && c->p.D <= 128 && c->p.D % 4 == 0;
}

}  // namespace emb

using namespace emb;

struct emb_ctx : public Ctx {};

extern "C" {

const char* emb_status_str(emb_status s) {
  switch (s) {
    case EMB_OK: return "ok";
    case EMB_EINVAL: return "invalid argument";
    case EMB_ENOMEM: return "out of device memory";
    case EMB_ESTATE: return "call out of order";
    case EMB_ECUDA: return "CUDA error";
  }
  return "unknown status";
}

// cache_rows > 0: tiered static tables (host tier of all rows, HBM cache of cache_rows).
static emb_status create_impl(const emb_config* cfg, int64_t cache_rows, emb_ctx** out) {
  if (!cfg || !out) return EMB_EINVAL;
  *out = nullptr;
  const int T = cfg->num_tables, D = cfg->dim;
  if (T < 1 || T > 4096 || D < 1 || D > 512) return EMB_EINVAL;
  if (cfg->dtype != EMB_F32 && cfg->dtype != EMB_BF16) return EMB_EINVAL;
  const int esize = cfg->dtype == EMB_BF16 ? 2 : 4;
  if ((D * esize) % 16 != 0 || D % 4 != 0) return EMB_EINVAL;
  if (cfg->pooling != EMB_POOL_SUM && cfg->pooling != EMB_POOL_MEAN) return EMB_EINVAL;
  if (cfg->optimizer != EMB_ADAGRAD && cfg->optimizer != EMB_ADAGRAD_ROWWISE) return EMB_EINVAL;
  if (!(cfg->eps >= 0.0f) || !(cfg->lr == cfg->lr) || !(cfg->init_acc == cfg->init_acc))
    return EMB_EINVAL;
  if (cfg->max_batch < 1 || cfg->max_lookups < 1) return EMB_EINVAL;
  if (cfg->max_lookups >= (int64_t)1 << 31 || cfg->max_batch * T >= (int64_t)1 << 31)
    return EMB_EINVAL;
  int64_t total = 0;
  if (cfg->hashed) {
    const int64_t cap = cfg->capacity;
    if (cap < 2 || cap > ((int64_t)1 << 31) || (cap & (cap - 1)) != 0) return EMB_EINVAL;
    total = cap;
  } else {
    if (!cfg->rows || T >= (1 << 15)) return EMB_EINVAL;
    for (int t = 0; t < T; ++t) {
      if (cfg->rows[t] < 1 || cfg->rows[t] >= ((int64_t)1 << 40)) return EMB_EINVAL;
      total += cfg->rows[t];
      if (total >= (int64_t)0xFFFFFFFFll) return EMB_EINVAL;
    }
  }

  const bool tiered = cache_rows > 0;
  if (tiered && (cfg->hashed || cache_rows < 2 || cache_rows > ((int64_t)1 << 31) ||
                 (cache_rows & (cache_rows - 1)) != 0))
    return EMB_EINVAL;
  const int64_t host_rows = tiered ? total : 0;
  if (tiered) total = cache_rows;  // device arrays hold the cache

  emb_ctx* c = new (std::nothrow) emb_ctx();
  if (!c) return EMB_ENOMEM;
  c->cfg = *cfg;
  c->cfg.rows = nullptr;
  if (!cfg->hashed) c->rows.assign(cfg->rows, cfg->rows + T);
  c->total_rows = total;
  c->tiered = tiered;
  c->host_rows = host_rows;
  c->max_batch = cfg->max_batch;
  c->max_lookups = cfg->max_lookups;
  if (const char* impl = std::getenv("EMB_FUSED_FWD")) {
    if (std::strcmp(impl, "tc") == 0) c->fwd_impl = 1;
    else if (std::strcmp(impl, "simt") == 0) c->fwd_impl = 2;
  }
  if (const char* impl = std::getenv("EMB_FUSED_BWD")) {
    if (std::strcmp(impl, "tc") == 0) c->bwd_impl = 1;
    else if (std::strcmp(impl, "simt") == 0) c->bwd_impl = 2;
  }
  if (const char* od = std::getenv("EMB_ONCE_DIRECT")) {
    if (std::strcmp(od, "0") == 0) c->once_direct = 0;
    else if (std::strcmp(od, "1") == 0) c->once_direct = 1;
  }
  if (const char* nc = std::getenv("EMB_HOST_CHUNKS")) {
    const int n = std::atoi(nc);
    if (n >= 1 && n <= Ctx::kMaxChunks) c->host_chunks = n;
  }
  if (const char* su = std::getenv("EMB_STAGED_UPDATE")) c->staged_update = std::strcmp(su, "0") != 0;
  uint32_t first_wait_polls = (uint32_t)kWaitLimit;
  if (const char* wp = std::getenv("EMB_WAIT_POLLS")) {  // test knob: the give-up path
    const long n = std::atol(wp);
    if (n >= 0 && n < kWaitLimit) first_wait_polls = (uint32_t)n;
  }
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
    cudaGetLastError();
    delete c;
    return EMB_ECUDA;
  }
  Params& p = c->p;
  std::memset(&p, 0, sizeof(p));
  p.T = T;
  p.D = D;
  p.bf16 = cfg->dtype == EMB_BF16;
  p.mean = cfg->pooling == EMB_POOL_MEAN;
  p.rowwise = cfg->optimizer == EMB_ADAGRAD_ROWWISE;
  p.hashed = cfg->hashed ? 1 : 0;
  p.tiered = tiered ? 1 : 0;
  p.lr = cfg->lr;
  p.eps = cfg->eps;
  p.init_acc = cfg->init_acc;
  p.first_wait_polls = first_wait_polls;

  const int64_t L = cfg->max_lookups;
  const int64_t AW = p.rowwise ? 1 : D;
  c->set_cap = next_pow2(std::max<int64_t>(2 * L, 1024));
  const int64_t gmax = std::min<int64_t>(L, total);
  const int64_t ntiles = (L + 1 + 2047) / 2048 + 1;
  bool ok = true;
  void* table = nullptr;
  ok = ok && dalloc(c, reinterpret_cast<char**>(&table), (size_t)total * D * esize);
  p.table = table;
  ok = ok && dalloc(c, &p.acc, (size_t)(total * AW));
  if (p.hashed || tiered) {
    ok = ok && dalloc(c, &p.hkeys, (size_t)total) && dalloc(c, &p.hstat, (size_t)total);
    p.hmask = (uint64_t)total - 1;
  }
  if (!p.hashed) {
    int64_t* base = nullptr;
    ok = ok && dalloc(c, &base, (size_t)T + 1);
    p.base = base;
  }
  if (tiered) {  // host tier: every row and accumulator, in host-mapped pinned memory
    ok = ok && dalloc(c, &p.fill_list, (size_t)L);
    if (ok)
      c->host_table = host_tier_alloc((size_t)host_rows * D * esize, &c->host_map[0],
                                      &c->host_map_len[0]);
    if (ok)
      c->host_acc = static_cast<float*>(host_tier_alloc(sizeof(float) * (size_t)(host_rows * AW),
                                                        &c->host_map[1], &c->host_map_len[1]));
    void* dt = nullptr;
    void* da = nullptr;
    ok = ok && c->host_table && c->host_acc &&
         cudaHostGetDevicePointer(&dt, c->host_table, 0) == cudaSuccess &&
         cudaHostGetDevicePointer(&da, c->host_acc, 0) == cudaSuccess;
    cudaGetLastError();
    p.htable = dt;
    p.hacc = static_cast<float*>(da);
    c->track = true;  // eviction reads the per-key counts and last steps
    ok = ok && dalloc(c, &p.tier_hist, 64) &&
         cudaEventCreateWithFlags(&c->ev_dedup, cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&c->ev_prefetch, cudaEventDisableTiming) == cudaSuccess;
  }
  ok = ok && dalloc(c, &p.set_keys, (size_t)c->set_cap) && dalloc(c, &p.set_vals, (size_t)c->set_cap);
  p.smask = (uint32_t)(c->set_cap - 1);
  ok = ok && dalloc(c, &p.row_of, L) && dalloc(c, &p.slot_of, L) && dalloc(c, &p.bag_of, L) &&
       dalloc(c, &p.inv, L) && dalloc(c, &p.rank, L) && dalloc(c, &p.s_u, 3 * L) &&
       dalloc(c, &p.uniq_row, L) && dalloc(c, &p.uniq_slot, L) && dalloc(c, &p.uniq_once, L) &&
       dalloc(c, &p.uniq_hold, L) &&
       dalloc(c, &p.cnt, L + 1) &&
       dalloc(c, &p.seg, L + 1) && dalloc(c, &p.offs, (size_t)(cfg->max_batch * T + 1)) &&
       dalloc(c, &p.g, (size_t)(gmax * D)) && dalloc(c, &p.scan_tmp, (size_t)ntiles) &&
       dalloc(c, &p.counters, kNumCounters);
  if (ok) {  // one buffer: the once-row list's three arrays, or the sorted (u, bag) pairs
    p.s_row = p.s_u + L;
    p.s_bag = p.s_u + 2 * L;
    p.s_ub = reinterpret_cast<uint2*>(p.s_u);
  }
  float* zero_row = nullptr;
  ok = ok && dalloc(c, &zero_row, (size_t)D);
  p.zero_row = zero_row;
  if (ok) {
    void* h = nullptr;
    if (cudaHostAlloc(&h, sizeof(uint32_t), cudaHostAllocMapped) == cudaSuccess) {
      c->h_unique = static_cast<uint32_t*>(h);
      *c->h_unique = 0u;
      void* d = nullptr;
      if (cudaHostGetDevicePointer(&d, h, 0) == cudaSuccess)
        c->h_unique_dev = static_cast<uint32_t*>(d);
      else
        ok = false;
    } else {
      ok = false;
    }
    cudaGetLastError();
  }
  if (!ok) {
    free_all(c);
    delete c;
    return EMB_ENOMEM;
  }
  cudaStream_t s = 0;
  cudaError_t e = cudaMemsetAsync(p.counters, 0, sizeof(uint32_t) * kNumCounters, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(p.set_keys, 0xFF, sizeof(uint32_t) * c->set_cap, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(p.uniq_once, 0, (size_t)L, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(p.uniq_hold, 0, (size_t)L, s);
  if (e == cudaSuccess && (p.hashed || tiered))
    e = cudaMemsetAsync(p.hstat, 0, sizeof(uint64_t) * (size_t)total, s);
  if (e == cudaSuccess && tiered) e = cudaMemsetAsync(p.hkeys, 0xFF, sizeof(uint64_t) * (size_t)total, s);
  if (e == cudaSuccess && tiered) e = cudaMemsetAsync(p.tier_hist, 0, sizeof(uint32_t) * 64, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(p.g, 0, sizeof(float) * (size_t)(gmax * D), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(zero_row, 0, sizeof(float) * (size_t)D, s);
  if (e == cudaSuccess) {
    if (p.hashed) {
      e = launch_init_hash(c, s);
    } else {
      std::vector<int64_t> base(T + 1, 0);
      for (int t = 0; t < T; ++t) base[t + 1] = base[t] + c->rows[t];
      e = cudaMemcpy(const_cast<int64_t*>(p.base), base.data(), sizeof(int64_t) * (T + 1),
                     cudaMemcpyHostToDevice);
      if (e == cudaSuccess && !tiered) e = launch_init_table(c, s);
      if (e == cudaSuccess && tiered) {  // initial values written into the host tier
        void* tab = p.table;
        float* acc = p.acc;
        p.table = p.htable;
        p.acc = p.hacc;
        c->total_rows = host_rows;
        e = launch_init_table(c, s);
        p.table = tab;
        p.acc = acc;
        c->total_rows = total;
      }
    }
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaGetLastError();
    free_all(c);
    delete c;
    return EMB_ECUDA;
  }
  *out = c;
  return EMB_OK;
}

emb_status emb_create(const emb_config* cfg, emb_ctx** out) { return create_impl(cfg, 0, out); }

emb_status emb_create_tiered(const emb_config* cfg, int64_t cache_rows, emb_ctx** out) {
  if (!cfg || cache_rows < 1) return EMB_EINVAL;
  return create_impl(cfg, cache_rows, out);
}

void emb_destroy(emb_ctx* ctx) {
  if (!ctx) return;
  cudaDeviceSynchronize();
  free_all(ctx);
  delete ctx;
}

static emb_status check_launch(cudaError_t e) {
  if (e != cudaSuccess) {
    cudaGetLastError();
    return EMB_ECUDA;
  }
  return EMB_OK;
}

static emb_status check_lookup_args(const Ctx* c, const int64_t* ids, const int32_t* offs,
                                    int64_t nnz, int64_t batch) {
  if (batch < 0 || batch > c->max_batch || nnz < 0 || nnz > c->max_lookups) return EMB_EINVAL;
  if (nnz > 0 && !ids) return EMB_EINVAL;
  if (!offs && nnz != batch * c->p.T) return EMB_EINVAL;
  return EMB_OK;
}

// A backward step starts: number it (hashed tables stamp keys with the number) and set the
// Adagrad Decay period it belongs to.
static void begin_backward_step(Ctx* c) {
  c->step += 1;
  if (c->decay_steps) c->p.period = (c->step - 1 - c->decay_base) / c->decay_steps;
}

// Whether the step whose forward starts now tracks once rows (rows with a single lookup in
// the batch), which the tensor-core backward then updates itself.  Automatic choice: when
// the previous batch had at least kOnceFrac unique rows per lookup (read from the host
// mirror the inverse kernel writes; a value a step or two old only moves once rows between
// the two update paths, which compute the same values).  Measured on the Criteo shape
// (0.21 unique rows per lookup): step 0.666 ms with once rows against 0.738 without; with a
// quarter of its rows (0.17): 0.643 against 0.689 ms; on the uniform shape (0.97): 3.98
// against 6.9 ms.  The once path costs ~0.02 ms per step whatever the share.
constexpr double kOnceFrac = 0.1;
static bool decide_once_step(const Ctx* c) {
  if (!once_direct_ok(c) || c->once_direct == 0) return false;
  if (c->once_direct == 1) return true;
  if (c->last_nnz <= 0 || !c->h_unique) return false;
  const uint32_t u = *reinterpret_cast<volatile const uint32_t*>(c->h_unique);
  return (double)u >= kOnceFrac * (double)c->last_nnz;
}

emb_status emb_forward(emb_ctx* ctx, const int64_t* d_ids, const int32_t* d_offsets,
                       int64_t nnz, int64_t batch, float* d_pooled, void* stream) {
  if (!ctx) return EMB_EINVAL;
  emb_status st = check_lookup_args(ctx, d_ids, d_offsets, nnz, batch);
  if (st != EMB_OK) return st;
  if (batch > 0 && !d_pooled) return EMB_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  ctx->multi_hot = d_offsets != nullptr;
  ctx->p.nnz = nnz;
  ctx->once_step = false;
  cudaError_t e = launch_map_dedup(ctx, d_ids, d_offsets, nnz, batch, s);
  if (e == cudaSuccess && batch > 0) e = launch_pool(ctx, batch, d_pooled, s);
  ctx->last_batch = batch;
  ctx->last_nnz = nnz;
  ctx->fwd_kind = 1;
  return check_launch(e);
}

emb_status emb_interact(emb_ctx* ctx, const float* d_dense, const float* d_pooled,
                        int64_t batch, float* d_out, void* stream) {
  if (!ctx || batch < 0 || batch > ctx->max_batch || !interaction_shape_ok(ctx)) return EMB_EINVAL;
  if (batch == 0) return EMB_OK;
  if (!d_dense || !d_pooled || !d_out) return EMB_EINVAL;
  return check_launch(launch_interact_fwd(ctx, d_dense, d_pooled, batch, d_out,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

emb_status emb_interact_backward(emb_ctx* ctx, const float* d_dout, const float* d_dense,
                                 const float* d_pooled, int64_t batch, float* d_ddense,
                                 float* d_dpooled, void* stream) {
  if (!ctx || batch < 0 || batch > ctx->max_batch || !interaction_shape_ok(ctx)) return EMB_EINVAL;
  if (batch == 0) return EMB_OK;
  if (!d_dout || !d_dense || !d_pooled || !d_ddense || !d_dpooled) return EMB_EINVAL;
  return check_launch(launch_interact_bwd(ctx, d_dout, d_dense, d_pooled, batch, d_ddense,
                                          d_dpooled, reinterpret_cast<cudaStream_t>(stream)));
}

// Tiered contexts with a watermark: after each backward step, evict down to the low mark
// when the cache is fuller than the high mark (decided on the device; see
// launch_tier_watermark).  Waits for a pending prefetch first (no eviction alongside its
// inserts) and marks the cache as changed for the next prefetch.
static cudaError_t after_backward(Ctx* c, cudaStream_t s) {
  if (!c->tiered || c->wm_high == 0) return cudaSuccess;
  cudaError_t e = cudaSuccess;
  if (c->pf_pending) e = cudaStreamWaitEvent(s, c->ev_prefetch, 0);
  if (e == cudaSuccess) e = launch_tier_watermark(c, c->wm_high, c->wm_low, s);
  if (e == cudaSuccess) e = cudaEventRecord(c->ev_dedup, s);
  return e;
}

emb_status emb_backward_adagrad(emb_ctx* ctx, const float* d_dpooled, void* stream) {
  if (!ctx) return EMB_EINVAL;
  if (ctx->fwd_kind != 1) return EMB_ESTATE;
  if (ctx->last_batch > 0 && !d_dpooled) return EMB_EINVAL;
  begin_backward_step(ctx);
  cudaError_t e = launch_backward_csr(ctx, d_dpooled, ctx->last_batch, ctx->last_nnz,
                                      reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = after_backward(ctx, reinterpret_cast<cudaStream_t>(stream));
  ctx->fwd_kind = 0;
  ctx->set_dirty = false;
  return check_launch(e);
}

emb_status emb_forward_interact(emb_ctx* ctx, const int64_t* d_ids, const int32_t* d_offsets,
                                int64_t nnz, int64_t batch, const float* d_dense,
                                float* d_out, void* stream) {
  if (!ctx || !interaction_shape_ok(ctx)) return EMB_EINVAL;
  emb_status st = check_lookup_args(ctx, d_ids, d_offsets, nnz, batch);
  if (st != EMB_OK) return st;
  if (batch > 0 && (!d_dense || !d_out)) return EMB_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  ctx->multi_hot = d_offsets != nullptr;
  ctx->p.nnz = nnz;
  ctx->once_step = decide_once_step(ctx);
  cudaError_t e = launch_map_dedup(ctx, d_ids, d_offsets, nnz, batch, s);
  // tracked keys: the unique indices and the lookup counts the backward stamps, in one pass
  ctx->counted = ctx->track && !fused_fwd_records_inverse(ctx);
  if (e == cudaSuccess && !fused_fwd_records_inverse(ctx))
    e = ctx->counted ? launch_inverse_counts(ctx, nnz, s) : launch_inverse(ctx, nnz, s);
  if (e == cudaSuccess && batch > 0) e = launch_fused_fwd(ctx, d_dense, batch, d_out, s);
  ctx->last_batch = batch;
  ctx->last_nnz = nnz;
  ctx->fwd_kind = 2;
  return check_launch(e);
}

emb_status emb_backward_interact_adagrad(emb_ctx* ctx, const float* d_dout,
                                         const float* d_dense, float* d_ddense, void* stream) {
  if (!ctx) return EMB_EINVAL;
  if (ctx->fwd_kind != 2) return EMB_ESTATE;
  if (ctx->last_batch > 0 && (!d_dout || !d_dense || !d_ddense)) return EMB_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  begin_backward_step(ctx);
  if (ctx->last_batch > 0) {
    e = clear_stale_g(ctx, s);
    if (e == cudaSuccess) e = launch_fused_bwd(ctx, d_dout, d_dense, ctx->last_batch, d_ddense, s);
  }
  // counted keys without admission holds: the update kernels stamp them on the way
  const bool fold = ctx->track && ctx->counted && ctx->p.admit_min <= 1;
  if (e == cudaSuccess && ctx->track && !fold)
    e = ctx->counted ? launch_admit(ctx, s) : launch_count_admit(ctx, ctx->last_nnz, s);
  if (e == cudaSuccess)
    e = launch_adagrad_from_g(ctx, std::min<int64_t>(ctx->last_nnz, ctx->total_rows), s, fold);
  if (e == cudaSuccess) e = after_backward(ctx, s);
  ctx->fwd_kind = 0;
  ctx->set_dirty = false;
  return check_launch(e);
}

// Host-buffer step of the one-hot fp32 shapes, pipelined over sample chunks: the IDs go up
// first and are deduplicated for the whole batch; then chunk c's dense rows go up, its
// forward runs and its output comes down while the next chunk's rows go up; the same for
// dout, the backward and d_dense; the update runs once all gradients are summed.  Uploads
// use st_h2d, downloads st_d2h, kernels `s`; every side-stream copy waits for the event of
// what it needs, `s` waits for the uploads it consumes and, at the end, for the downloads.
// The per-chunk launches see the context's lookup arrays shifted to the chunk's first
// sample (the kernels index them by sample).
static emb_status step_host_chunked(Ctx* c, const int64_t* h_ids, int64_t nnz, int64_t batch,
                                    const float* h_dense, const float* h_dout, float* h_out,
                                    float* h_ddense, cudaStream_t s) {
  const int T = c->p.T, D = c->p.D, F = T + 1;
  const int64_t W = D + (int64_t)F * (F - 1) / 2;
  const int nc = (int)std::min<int64_t>(batch, c->host_chunks);
  const int64_t per = (batch + nc - 1) / nc;
  auto b0 = [&](int i) { return std::min<int64_t>(batch, per * i); };
  cudaEvent_t* ev_dense = c->ev_chunk[0];
  cudaEvent_t* ev_dout = c->ev_chunk[1];
  cudaEvent_t* ev_fwd = c->ev_chunk[2];
  cudaEvent_t* ev_bwd = c->ev_chunk[3];
  cudaError_t e = cudaEventRecord(c->ev_inputs, s);  // everything earlier on `s` is done
  if (e == cudaSuccess) e = cudaStreamWaitEvent(c->st_h2d, c->ev_inputs, 0);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(c->st_ids, h_ids, sizeof(int64_t) * (size_t)nnz, cudaMemcpyHostToDevice, s);
  for (int i = 0; i < nc && e == cudaSuccess; ++i) {
    const int64_t a = b0(i), n = b0(i + 1) - a;
    e = cudaMemcpyAsync(c->st_dense + a * D, h_dense + a * D, sizeof(float) * (size_t)(n * D),
                        cudaMemcpyHostToDevice, c->st_h2d);
    if (e == cudaSuccess) e = cudaEventRecord(ev_dense[i], c->st_h2d);
  }
  for (int i = 0; i < nc && e == cudaSuccess; ++i) {
    const int64_t a = b0(i), n = b0(i + 1) - a;
    e = cudaMemcpyAsync(c->st_dout + a * W, h_dout + a * W, sizeof(float) * (size_t)(n * W),
                        cudaMemcpyHostToDevice, c->st_h2d);
    if (e == cudaSuccess) e = cudaEventRecord(ev_dout[i], c->st_h2d);
  }
  c->multi_hot = false;
  c->p.nnz = nnz;
  c->once_step = decide_once_step(c);
  if (e == cudaSuccess) e = launch_map_dedup(c, c->st_ids, nullptr, nnz, batch, s);
  if (e == cudaSuccess) e = c->track ? launch_inverse_counts(c, nnz, s) : launch_inverse(c, nnz, s);
  const Params whole = c->p;
  auto shifted = [&](int64_t a) {
    c->p = whole;
    c->p.row_of += a * T;
    c->p.inv += a * T;
  };
  for (int i = 0; i < nc && e == cudaSuccess; ++i) {
    const int64_t a = b0(i), n = b0(i + 1) - a;
    e = cudaStreamWaitEvent(s, ev_dense[i], 0);
    shifted(a);
    if (e == cudaSuccess) e = launch_fused_fwd(c, c->st_dense + a * D, n, c->st_out + a * W, s);
    c->p = whole;
    if (e == cudaSuccess) e = cudaEventRecord(ev_fwd[i], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c->st_d2h, ev_fwd[i], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h_out + a * W, c->st_out + a * W, sizeof(float) * (size_t)(n * W),
                          cudaMemcpyDeviceToHost, c->st_d2h);
  }
  if (e == cudaSuccess) e = clear_stale_g(c, s);
  for (int i = 0; i < nc && e == cudaSuccess; ++i) {
    const int64_t a = b0(i), n = b0(i + 1) - a;
    e = cudaStreamWaitEvent(s, ev_dout[i], 0);
    shifted(a);
    if (e == cudaSuccess)
      e = launch_fused_bwd(c, c->st_dout + a * W, c->st_dense + a * D, n, c->st_ddense + a * D, s);
    c->p = whole;
    if (e == cudaSuccess) e = cudaEventRecord(ev_bwd[i], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c->st_d2h, ev_bwd[i], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h_ddense + a * D, c->st_ddense + a * D, sizeof(float) * (size_t)(n * D),
                          cudaMemcpyDeviceToHost, c->st_d2h);
  }
  begin_backward_step(c);
  const bool fold = c->track && c->p.admit_min <= 1;  // counted above; no holds to decide
  if (e == cudaSuccess && c->track && !fold) e = launch_admit(c, s);
  if (e == cudaSuccess)
    e = launch_adagrad_from_g(c, std::min<int64_t>(nnz, c->total_rows), s, fold);
  if (e == cudaSuccess) e = after_backward(c, s);
  // join both side streams into `s`, also on failure, so nothing outlives the call's order
  cudaEventRecord(c->ev_out, c->st_d2h);
  cudaStreamWaitEvent(s, c->ev_out, 0);
  cudaEventRecord(c->ev_dout, c->st_h2d);
  cudaStreamWaitEvent(s, c->ev_dout, 0);
  c->last_batch = batch;
  c->last_nnz = nnz;
  c->fwd_kind = 0;
  c->set_dirty = false;
  return check_launch(e);
}

emb_status emb_train_step_host(emb_ctx* ctx, const int64_t* h_ids, const int32_t* h_offsets,
                               int64_t nnz, int64_t batch, const float* h_dense,
                               const float* h_dout, float* h_out, float* h_ddense,
                               void* stream) {
  if (!ctx || !interaction_shape_ok(ctx)) return EMB_EINVAL;
  emb_status st = check_lookup_args(ctx, h_ids, h_offsets, nnz, batch);
  if (st != EMB_OK) return st;
  if (batch > 0 && (!h_dense || !h_dout || !h_out || !h_ddense)) return EMB_EINVAL;
  Ctx* c = ctx;
  const int T = c->p.T, D = c->p.D, F = T + 1;
  const int64_t W = D + (int64_t)F * (F - 1) / 2;
  if (!c->st_ids) {
    bool ok = dalloc(c, &c->st_ids, (size_t)c->max_lookups) &&
              dalloc(c, &c->st_offs, (size_t)(c->max_batch * T + 1)) &&
              dalloc(c, &c->st_dense, (size_t)(c->max_batch * D)) &&
              dalloc(c, &c->st_dout, (size_t)(c->max_batch * W)) &&
              dalloc(c, &c->st_out, (size_t)(c->max_batch * W)) &&
              dalloc(c, &c->st_ddense, (size_t)(c->max_batch * D));
    for (cudaStream_t* q : {&c->st_h2d, &c->st_d2h})
      ok = ok && cudaStreamCreateWithFlags(q, cudaStreamNonBlocking) == cudaSuccess;
    for (cudaEvent_t* ev : {&c->ev_inputs, &c->ev_dout, &c->ev_fwd, &c->ev_out})
      ok = ok && cudaEventCreateWithFlags(ev, cudaEventDisableTiming) == cudaSuccess;
    for (auto& row : c->ev_chunk)
      for (cudaEvent_t& ev : row)
        ok = ok && cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      c->st_ids = nullptr;
      return EMB_ENOMEM;
    }
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  c->multi_hot = h_offsets != nullptr;
  if (!h_offsets && batch > 0 && reg_supported(c) && use_tc_bwd(c))
    return step_host_chunked(c, h_ids, nnz, batch, h_dense, h_dout, h_out, h_ddense, s);
  // Three streams: `s` carries the inputs, the kernels and d_dense; st_h2d uploads dout
  // while the forward runs; st_d2h downloads out while the backward and update run.  Each
  // side stream starts behind the work already on `s` (so the staging buffers are free) and
  // `s` ends behind both, so synchronising `s` covers the whole step.
  cudaError_t e = cudaMemcpyAsync(c->st_ids, h_ids, sizeof(int64_t) * (size_t)nnz,
                                  cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && h_offsets)
    e = cudaMemcpyAsync(c->st_offs, h_offsets, sizeof(int32_t) * (size_t)(batch * T + 1),
                        cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(c->st_dense, h_dense, sizeof(float) * (size_t)(batch * D),
                        cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaEventRecord(c->ev_inputs, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(c->st_h2d, c->ev_inputs, 0);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(c->st_dout, h_dout, sizeof(float) * (size_t)(batch * W),
                        cudaMemcpyHostToDevice, c->st_h2d);
  if (e == cudaSuccess) e = cudaEventRecord(c->ev_dout, c->st_h2d);
  if (e != cudaSuccess) return check_launch(e);
  st = emb_forward_interact(ctx, c->st_ids, h_offsets ? c->st_offs : nullptr, nnz, batch,
                            c->st_dense, c->st_out, stream);
  if (st != EMB_OK) {
    cudaStreamWaitEvent(s, c->ev_dout, 0);
    return st;
  }
  e = cudaEventRecord(c->ev_fwd, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(c->st_d2h, c->ev_fwd, 0);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(h_out, c->st_out, sizeof(float) * (size_t)(batch * W),
                        cudaMemcpyDeviceToHost, c->st_d2h);
  if (e == cudaSuccess) e = cudaEventRecord(c->ev_out, c->st_d2h);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, c->ev_dout, 0);
  if (e != cudaSuccess) return check_launch(e);
  st = emb_backward_interact_adagrad(ctx, c->st_dout, c->st_dense, c->st_ddense, stream);
  if (st == EMB_OK) {
    e = cudaMemcpyAsync(h_ddense, c->st_ddense, sizeof(float) * (size_t)(batch * D),
                        cudaMemcpyDeviceToHost, s);
    st = check_launch(e);
  }
  cudaError_t j = cudaStreamWaitEvent(s, c->ev_out, 0);
  if (st == EMB_OK) st = check_launch(j);
  return st;
}

emb_status emb_get_status(emb_ctx* ctx, void* stream, uint32_t* flags) {
  if (!ctx || !flags) return EMB_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t f = 0;
  cudaError_t e = cudaMemcpyAsync(&f, ctx->p.counters + kFlags, sizeof(uint32_t),
                                  cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctx->p.counters + kFlags, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  *flags = f;
  return check_launch(e);
}

// temporary device buffer for the synchronous read-back calls
struct TmpBuf {
  void* p = nullptr;
  explicit TmpBuf(size_t bytes) {
    if (cudaMalloc(&p, bytes ? bytes : 1) != cudaSuccess) {
      cudaGetLastError();
      p = nullptr;
    }
  }
  ~TmpBuf() {
    if (p) cudaFree(p);
  }
};

// Tiered tables: a row cached in HBM is read there, any other from the host tier (host
// memory, read here directly after the device has finished).
static emb_status read_rows_tiered(Ctx* c, const std::vector<uint32_t>& grow, float* h_w,
                                   float* h_acc, int8_t* h_found) {
  const int64_t n = (int64_t)grow.size();
  const int D = c->p.D, AW = c->p.rowwise ? 1 : D;
  TmpBuf keys(sizeof(int64_t) * n), slots(sizeof(uint32_t) * n), w(sizeof(float) * n * D),
      acc(sizeof(float) * n * AW);
  if (!keys.p || !slots.p || !w.p || !acc.p) return EMB_ENOMEM;
  std::vector<int64_t> k(grow.begin(), grow.end());
  std::vector<uint32_t> hs(n);
  std::vector<float> hw((size_t)n * D), ha((size_t)n * AW);
  cudaError_t e = cudaMemcpy(keys.p, k.data(), sizeof(int64_t) * n, cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = launch_find_keys(c, reinterpret_cast<int64_t*>(keys.p), n,
                         reinterpret_cast<uint32_t*>(slots.p), 0);
  if (e == cudaSuccess)
    e = launch_read_rows(c, reinterpret_cast<uint32_t*>(slots.p), n, reinterpret_cast<float*>(w.p),
                         reinterpret_cast<float*>(acc.p), 0);
  if (e == cudaSuccess) e = cudaMemcpy(hs.data(), slots.p, sizeof(uint32_t) * n, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(hw.data(), w.p, sizeof(float) * n * D, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(ha.data(), acc.p, sizeof(float) * n * AW, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return check_launch(e);
  for (int64_t q = 0; q < n; ++q) {
    if (hs[q] == kNoRow) {  // not cached: the host tier holds the current values
      const int64_t r = grow[q];
      for (int j = 0; j < D; ++j) {
        if (c->p.bf16) {
          const uint16_t b = reinterpret_cast<const uint16_t*>(c->host_table)[r * D + j];
          uint32_t u = (uint32_t)b << 16;
          std::memcpy(&hw[q * D + j], &u, 4);
        } else {
          hw[q * D + j] = reinterpret_cast<const float*>(c->host_table)[r * D + j];
        }
      }
      for (int j = 0; j < AW; ++j) ha[q * AW + j] = c->host_acc[r * AW + j];
    }
    if (h_found) h_found[q] = 1;
  }
  if (h_w) std::memcpy(h_w, hw.data(), sizeof(float) * n * D);
  if (h_acc) std::memcpy(h_acc, ha.data(), sizeof(float) * n * AW);
  return EMB_OK;
}

emb_status emb_read_rows(emb_ctx* ctx, int32_t table, const int64_t* h_ids, int64_t n,
                         float* h_w, float* h_acc, int8_t* h_found) {
  if (!ctx || n < 0 || (n > 0 && !h_ids)) return EMB_EINVAL;
  if (n == 0) return EMB_OK;
  Ctx* c = ctx;
  const int AW = c->p.rowwise ? 1 : c->p.D;
  if (cudaDeviceSynchronize() != cudaSuccess) return check_launch(cudaErrorUnknown);
  TmpBuf rows(sizeof(uint32_t) * n), w(sizeof(float) * n * c->p.D), acc(sizeof(float) * n * AW);
  if (!rows.p || !w.p || !acc.p) return EMB_ENOMEM;
  std::vector<uint32_t> hrows(n);
  cudaError_t e = cudaSuccess;
  if (!c->p.hashed) {
    if (table < 0 || table >= c->p.T) return EMB_EINVAL;
    int64_t base = 0;
    for (int t = 0; t < table; ++t) base += c->rows[t];
    for (int64_t q = 0; q < n; ++q) {
      if (h_ids[q] < 0 || h_ids[q] >= c->rows[table]) return EMB_EINVAL;
      hrows[q] = (uint32_t)(base + h_ids[q]);
    }
    if (c->tiered) return read_rows_tiered(c, hrows, h_w, h_acc, h_found);
    e = cudaMemcpy(rows.p, hrows.data(), sizeof(uint32_t) * n, cudaMemcpyHostToDevice);
  } else {
    TmpBuf keys(sizeof(int64_t) * n);
    if (!keys.p) return EMB_ENOMEM;
    e = cudaMemcpy(keys.p, h_ids, sizeof(int64_t) * n, cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
      e = launch_find_keys(c, reinterpret_cast<int64_t*>(keys.p), n,
                           reinterpret_cast<uint32_t*>(rows.p), 0);
    if (e == cudaSuccess)
      e = cudaMemcpy(hrows.data(), rows.p, sizeof(uint32_t) * n, cudaMemcpyDeviceToHost);
  }
  if (e == cudaSuccess)
    e = launch_read_rows(c, reinterpret_cast<uint32_t*>(rows.p), n,
                         reinterpret_cast<float*>(w.p), reinterpret_cast<float*>(acc.p), 0);
  if (e == cudaSuccess && h_w)
    e = cudaMemcpy(h_w, w.p, sizeof(float) * n * c->p.D, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && h_acc)
    e = cudaMemcpy(h_acc, acc.p, sizeof(float) * n * AW, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && h_found)
    for (int64_t q = 0; q < n; ++q) h_found[q] = hrows[q] != kNoRow;
  return check_launch(e);
}

emb_status emb_set_adagrad_decay(emb_ctx* ctx, float rate, uint32_t period_steps) {
  if (!ctx) return EMB_EINVAL;
  if (period_steps > 0 && !(rate > 0.f && rate <= 1.f)) return EMB_EINVAL;
  if (ctx->fwd_kind != 0) return EMB_ESTATE;
  Params& p = ctx->p;
  if (period_steps > 0) {  // periods count from the next backward step; every row starts in 0
    if (!p.rperiod && !dalloc(ctx, &p.rperiod, (size_t)ctx->total_rows)) return EMB_ENOMEM;
    if (cudaMemset(p.rperiod, 0, sizeof(uint32_t) * (size_t)ctx->total_rows) != cudaSuccess)
      return check_launch(cudaErrorUnknown);
  }
  ctx->decay_steps = period_steps;
  ctx->decay_base = ctx->step;
  p.decay = period_steps > 0 ? 1 : 0;
  p.decay_rate = rate;
  p.period = 0;
  return EMB_OK;
}

emb_status emb_set_admission(emb_ctx* ctx, uint32_t min_count) {
  if (!ctx || !ctx->p.hashed) return EMB_EINVAL;
  if (ctx->fwd_kind != 0) return EMB_ESTATE;
  ctx->p.admit_min = min_count;
  ctx->track = true;
  return EMB_OK;
}

emb_status emb_evict(emb_ctx* ctx, uint32_t max_idle_steps, uint32_t min_count, void* stream,
                     int64_t* h_evicted) {
  if (!ctx || !(ctx->p.hashed || ctx->tiered)) return EMB_EINVAL;
  if (ctx->fwd_kind != 0 || !ctx->track) return EMB_ESTATE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (ctx->tiered && ctx->pf_pending) e = cudaStreamWaitEvent(s, ctx->ev_prefetch, 0);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctx->p.counters + kEvicted, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = launch_evict(ctx, max_idle_steps, min_count, s);
  if (e == cudaSuccess && ctx->tiered) e = cudaEventRecord(ctx->ev_dedup, s);  // cache changed
  if (e == cudaSuccess && h_evicted) {
    uint32_t n = 0;
    e = cudaMemcpyAsync(&n, ctx->p.counters + kEvicted, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    *h_evicted = n;
  }
  return check_launch(e);
}

emb_status emb_prefetch(emb_ctx* ctx, const int64_t* d_ids, const int32_t* d_offsets,
                        int64_t nnz, int64_t batch, void* stream) {
  if (!ctx || !ctx->tiered) return EMB_EINVAL;
  emb_status st = check_lookup_args(ctx, d_ids, d_offsets, nnz, batch);
  if (st != EMB_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // after the latest change of the cache (the pending forward's dedup and fill, or an
  // eviction); rows stamped with the step number their batch's backward will count them at
  // at the earliest, so a watermark check in between does not take them out again
  cudaError_t e = cudaStreamWaitEvent(s, ctx->ev_dedup, 0);
  if (e == cudaSuccess && ctx->pf_pending) e = cudaStreamWaitEvent(s, ctx->ev_prefetch, 0);
  const uint32_t stamp = ctx->step + (ctx->fwd_kind != 0 ? 1u : 0u);
  if (e == cudaSuccess) e = launch_prefetch(ctx, d_ids, d_offsets, nnz, batch, stamp, s);
  if (e == cudaSuccess) e = cudaEventRecord(ctx->ev_prefetch, s);
  if (e == cudaSuccess) ctx->pf_pending = true;
  return check_launch(e);
}

emb_status emb_set_tier_watermark(emb_ctx* ctx, int64_t high, int64_t low) {
  if (!ctx || !ctx->tiered) return EMB_EINVAL;
  if (high != 0 && (low < 0 || low >= high || high > ctx->total_rows)) return EMB_EINVAL;
  if (ctx->fwd_kind != 0) return EMB_ESTATE;
  ctx->wm_high = (uint32_t)high;
  ctx->wm_low = high ? (uint32_t)low : 0u;
  return EMB_OK;
}

emb_status emb_tier_occupancy(emb_ctx* ctx, int64_t* h_rows) {
  if (!ctx || !ctx->tiered || !h_rows) return EMB_EINVAL;
  uint32_t n = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess)
    e = cudaMemcpy(&n, ctx->p.counters + kOcc, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  *h_rows = n;
  return check_launch(e);
}

emb_status emb_read_key_stats(emb_ctx* ctx, const int64_t* h_keys, int64_t n, uint32_t* h_count,
                              uint32_t* h_last_step) {
  if (!ctx || !(ctx->p.hashed || ctx->tiered) || n < 0 || (n > 0 && !h_keys)) return EMB_EINVAL;
  if (n == 0) return EMB_OK;
  Ctx* c = ctx;
  if (cudaDeviceSynchronize() != cudaSuccess) return check_launch(cudaErrorUnknown);
  TmpBuf keys(sizeof(int64_t) * n), rows(sizeof(uint32_t) * n), cnt(sizeof(uint32_t) * n),
      last(sizeof(uint32_t) * n);
  if (!keys.p || !rows.p || !cnt.p || !last.p) return EMB_ENOMEM;
  cudaError_t e = cudaMemcpy(keys.p, h_keys, sizeof(int64_t) * n, cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = launch_find_keys(c, reinterpret_cast<int64_t*>(keys.p), n,
                         reinterpret_cast<uint32_t*>(rows.p), 0);
  if (e == cudaSuccess)
    e = launch_key_stats(c, reinterpret_cast<uint32_t*>(rows.p), n,
                         reinterpret_cast<uint32_t*>(cnt.p), reinterpret_cast<uint32_t*>(last.p), 0);
  if (e == cudaSuccess && h_count)
    e = cudaMemcpy(h_count, cnt.p, sizeof(uint32_t) * n, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && h_last_step)
    e = cudaMemcpy(h_last_step, last.p, sizeof(uint32_t) * n, cudaMemcpyDeviceToHost);
  return check_launch(e);
}

emb_status emb_read_unique(emb_ctx* ctx, int64_t* h_keys, int32_t* h_counts, int64_t cap,
                           int64_t* h_num_unique) {
  if (!ctx || !h_num_unique || cap < 0) return EMB_EINVAL;
  Ctx* c = ctx;
  if (c->last_nnz < 0) return EMB_ESTATE;
  if (cudaDeviceSynchronize() != cudaSuccess) return check_launch(cudaErrorUnknown);
  uint32_t U = 0;
  cudaError_t e = cudaMemcpy(&U, c->p.counters + kU, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return check_launch(e);
  *h_num_unique = U;
  TmpBuf counts(sizeof(uint32_t) * (U + 1)), keys(sizeof(int64_t) * (U + 1));
  if (!counts.p || !keys.p) return EMB_ENOMEM;
  e = cudaMemset(counts.p, 0, sizeof(uint32_t) * (U + 1));
  if (e == cudaSuccess)
    e = launch_unique_count(c, c->last_nnz, reinterpret_cast<uint32_t*>(counts.p),
                            reinterpret_cast<int64_t*>(keys.p), 0);
  const int64_t n = std::min<int64_t>(U, cap);
  if (e == cudaSuccess && h_keys && n > 0)
    e = cudaMemcpy(h_keys, keys.p, sizeof(int64_t) * n, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && h_counts && n > 0)
    e = cudaMemcpy(h_counts, counts.p, sizeof(int32_t) * n, cudaMemcpyDeviceToHost);
  return check_launch(e);
}

emb_status emb_export_hash(emb_ctx* ctx, int64_t* h_keys, float* h_w, float* h_acc,
                           int64_t cap, int64_t* h_count) {
  if (!ctx || !h_count || cap < 0) return EMB_EINVAL;
  Ctx* c = ctx;
  if (!c->p.hashed) return EMB_EINVAL;
  if (cudaDeviceSynchronize() != cudaSuccess) return check_launch(cudaErrorUnknown);
  TmpBuf cnt(sizeof(uint32_t));
  if (!cnt.p) return EMB_ENOMEM;
  cudaError_t e = cudaMemset(cnt.p, 0, sizeof(uint32_t));
  if (e == cudaSuccess)
    e = launch_export_hash(c, 0, nullptr, nullptr, reinterpret_cast<uint32_t*>(cnt.p), 0);
  uint32_t total = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&total, cnt.p, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return check_launch(e);
  *h_count = total;
  const int64_t n = std::min<int64_t>(total, cap);
  if (n == 0) return EMB_OK;
  const int AW = c->p.rowwise ? 1 : c->p.D;
  TmpBuf keys(sizeof(int64_t) * total), rows(sizeof(uint32_t) * total),
      w(sizeof(float) * n * c->p.D), acc(sizeof(float) * n * AW);
  if (!keys.p || !rows.p || !w.p || !acc.p) return EMB_ENOMEM;
  e = cudaMemset(cnt.p, 0, sizeof(uint32_t));
  if (e == cudaSuccess)
    e = launch_export_hash(c, total, reinterpret_cast<int64_t*>(keys.p),
                           reinterpret_cast<uint32_t*>(rows.p), reinterpret_cast<uint32_t*>(cnt.p), 0);
  if (e == cudaSuccess)
    e = launch_read_rows(c, reinterpret_cast<uint32_t*>(rows.p), n, reinterpret_cast<float*>(w.p),
                         reinterpret_cast<float*>(acc.p), 0);
  if (e == cudaSuccess && h_keys)
    e = cudaMemcpy(h_keys, keys.p, sizeof(int64_t) * n, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && h_w)
    e = cudaMemcpy(h_w, w.p, sizeof(float) * n * c->p.D, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && h_acc)
    e = cudaMemcpy(h_acc, acc.p, sizeof(float) * n * AW, cudaMemcpyDeviceToHost);
  return check_launch(e);
}

emb_status emb_profile(emb_ctx* ctx, int32_t enable) {
  if (!ctx) return EMB_EINVAL;
  ctx->prof_on = enable != 0;
  if (ctx->prof_on && ctx->ev_pool.size() < 4096) {
    while (ctx->ev_pool.size() < 4096) {
      cudaEvent_t e = nullptr;
      if (cudaEventCreate(&e) != cudaSuccess) return check_launch(cudaErrorUnknown);
      ctx->ev_pool.push_back(e);
    }
  }
  return EMB_OK;
}

static cudaError_t drain_records(Ctx* c) {
  cudaError_t err = cudaSuccess;
  for (auto& r : c->recs) {
    cudaError_t e = cudaEventSynchronize(r.b);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.a, r.b);
    if (e == cudaSuccess) {
      c->prof_ms[r.kid] += ms;
      c->prof_n[r.kid] += 1;
    } else {
      err = e;
      cudaGetLastError();
    }
    c->ev_pool.push_back(r.a);
    c->ev_pool.push_back(r.b);
  }
  c->recs.clear();
  return err;
}

emb_status emb_profile_read(emb_ctx* ctx, int32_t idx, const char** name, double* total_ms,
                            int64_t* launches) {
  if (!ctx || idx < 0 || idx >= K_NUM_KERNELS) return EMB_EINVAL;
  cudaError_t e = drain_records(ctx);
  if (name) *name = kKernelNames[idx];
  if (total_ms) *total_ms = ctx->prof_ms[idx];
  if (launches) *launches = ctx->prof_n[idx];
  return check_launch(e);
}

emb_status emb_profile_reset(emb_ctx* ctx) {
  if (!ctx) return EMB_EINVAL;
  cudaError_t e = drain_records(ctx);
  for (int k = 0; k < K_NUM_KERNELS; ++k) {
    ctx->prof_ms[k] = 0.0;
    ctx->prof_n[k] = 0;
  }
  return check_launch(e);
}

int64_t emb_launch_count(const emb_ctx* ctx) { return ctx ? ctx->launches : 0; }

emb_status emb_cross_forward(const float* d_x0, const float* d_xl, const float* d_w,
                             const float* d_b, int64_t B, int32_t K, float* d_out, void* stream) {
  if (B < 0 || K < 1 || K > EMB_CROSS_MAX_K) return EMB_EINVAL;
  if (B > 0 && (!d_x0 || !d_xl || !d_w || !d_b || !d_out)) return EMB_EINVAL;
  return check_launch(launch_cross_fwd(d_x0, d_xl, d_w, d_b, B, K, d_out,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

emb_status emb_cross_backward(const float* d_x0, const float* d_xl, const float* d_w,
                              const float* d_dout, int64_t B, int32_t K, float* d_dx0,
                              float* d_dxl, float* d_dw, float* d_db, void* stream) {
  if (B < 0 || K < 1 || K > EMB_CROSS_MAX_K || !d_dw || !d_db) return EMB_EINVAL;
  if (B > 0 && (!d_x0 || !d_xl || !d_w || !d_dout || !d_dx0 || !d_dxl)) return EMB_EINVAL;
  return check_launch(launch_cross_bwd(d_x0, d_xl, d_w, d_dout, B, K, d_dx0, d_dxl, d_dw, d_db,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

emb_status emb_quantize_rows(const float* d_x, int64_t n, int32_t d, int8_t* d_q,
                             float* d_scale, void* stream) {
  if (n < 0 || d < 1 || (n > 0 && (!d_x || !d_q || !d_scale))) return EMB_EINVAL;
  return check_launch(launch_quantize_rows(d_x, n, d, d_q, d_scale,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

emb_status emb_dequantize_rows(const int8_t* d_q, const float* d_scale, int64_t n, int32_t d,
                               float* d_x, void* stream) {
  if (n < 0 || d < 1 || (n > 0 && (!d_x || !d_q || !d_scale))) return EMB_EINVAL;
  return check_launch(launch_dequantize_rows(d_q, d_scale, n, d, d_x,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int32_t emb_step_tracks_once(const emb_ctx* ctx) {
  if (!ctx) return -1;
  return ctx->once_step ? 1 : 0;
}

}  // extern "C"
