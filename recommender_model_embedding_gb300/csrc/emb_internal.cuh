// Internal declarations shared by the translation units of libemb.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "emb.h"

namespace emb {

constexpr uint32_t kEmpty32 = 0xFFFFFFFFu;  // free slot of the dedup set
constexpr uint64_t kEmpty64 = ~0ull;        // free slot of the hashed table (key -1)
constexpr uint64_t kTomb64 = ~1ull;         // evicted slot (key -2): probes pass it, inserts reuse it
constexpr uint32_t kNoRow = 0xFFFFFFFFu;    // lookup that maps to no row (rejected ID)
// Rows looked up once ("once rows"), when a step tracks them (tables below 2^31 rows):
// bit 31 of a dedup-set key marks a row that a second lookup found; bit 31 of an inverse
// index marks the only lookup of a once row.  Unique indices stay below 2^31.
constexpr uint32_t kSetMulti = 0x80000000u;
constexpr uint32_t kInvOnce = 0x80000000u;
constexpr int kMaxF = 32;                   // interaction vectors per sample (T+1)
constexpr int kMaxProbe = 1 << 20;          // probe limit of the hashed table

// indices into the small device counter array
// kOcc: tiered cache slots in use; kPfFill: rows a prefetch brings in; kThresh: idle-time
// threshold the watermark check chose (all ones: nothing to evict); kTierDone: blocks of the
// watermark histogram pass that have finished (zero between checks)
enum Counter : int {
  kU = 0, kFlags = 1, kMulti = 2, kEvicted = 3, kFill = 4, kOcc = 5, kPfFill = 6, kThresh = 7,
  kTierDone = 8, kNumCounters = 9
};

// kernel ids for launch counting and optional event timing
enum KernelId : int {
  K_INIT_TABLE = 0,
  K_INIT_HASH,
  K_RESET_SET,
  K_EXPAND_BAGS,
  K_MAP_DEDUP,
  K_POOL,
  K_INTERACT_FWD,
  K_INTERACT_BWD,
  K_FUSED_FWD,
  K_FUSED_BWD,
  K_INVERSE_COUNT,
  K_SCAN_LOCAL,
  K_SCAN_BLOCKS,
  K_SCAN_ADD,
  K_FILL_PERM,
  K_SEGREDUCE_ADAGRAD,
  K_ADAGRAD_FROM_G,
  K_UNIQUE_COUNT,
  K_READ_ROWS,
  K_EXPORT_HASH,
  K_INVERSE,
  K_ONCE_SPLIT,
  K_ADMIT,
  K_EVICT,
  K_TIER_FILL,
  K_PREFETCH,
  K_TIER_WATERMARK,
  K_NUM_KERNELS
};
extern const char* const kKernelNames[K_NUM_KERNELS];

// Parameters every kernel family needs, passed by value.
struct Params {
  int T, D;
  int64_t nnz;           // lookups of the current batch (bound for offsets)
  int bf16, mean, rowwise, hashed;
  float lr, eps, init_acc;
  void* table;           // [rows][D] fp32 or bf16
  float* acc;            // [rows][D] or [rows]
  const int64_t* base;   // static: [T+1] first global row of each table
  int tiered;            // static tables in the host tier, cached in HBM (hkeys = global rows)
  void* htable;          // tiered: [host rows][D] parameters in host-mapped memory
  float* hacc;           // tiered: [host rows][D] or [host rows] accumulators, host-mapped
  uint32_t* fill_list;   // tiered: [L] cache slots claimed by the current batch
  uint64_t* hkeys;       // hashed: [capacity]; tiered: [cache rows], keys = global rows
  uint64_t hmask;        // capacity - 1
  uint64_t* hstat;       // hashed: [capacity] lookups counted over all steps (low 32 bits)
                         //   and the last step that counted the slot's key (high 32 bits)
  uint32_t admit_min;    // hashed: updates held until a key's count reaches this (0, 1: off)
  int decay;             // Adagrad Decay on: accumulators discounted per period of steps
  float decay_rate;      //   discount per period
  uint32_t period;       //   period of the current step
  uint32_t* rperiod;     //   [rows] period of each row's last update (allocated when on)
  uint32_t smask;        // dedup set: large region's capacity - 1
  uint32_t ssmall;       // dedup set: small region's capacity (slots [0, ssmall)), 0: none;
                         //   the large region follows it
  uint32_t* set_keys;    // [S] row of each occupied slot (| kSetMulti), kEmpty32 when free
  uint32_t* set_vals;    // [S] unique index of each occupied slot
  uint32_t* row_of;      // [L] row (static) or slot (hashed) of each lookup
  uint32_t* slot_of;     // [L] dedup-set slot of each lookup
  uint32_t* bag_of;      // [L] bag of each lookup (multi-hot)
  uint32_t* inv;         // [L] unique index of each lookup
  uint32_t* rank;        // [L] rank among the lookups of its unique row
  int32_t* offs;         // [B*T+1] device copy of the offsets (multi-hot)
  uint32_t* uniq_row;    // [L]
  uint32_t* uniq_slot;   // [L]
  uint8_t* uniq_once;    // [L] 1 when the unique row has one lookup (steps that track it);
                         //     0 between steps
  uint8_t* uniq_hold;    // [L] hashed: 1 when the unique key's update is held (admission)
  uint32_t* cnt;         // [L+1]
  uint32_t* seg;         // [L+1]
  // steps that track once rows: the list of the other unique rows (unique index, row,
  // dedup-set slot) that the update visits
  uint32_t* s_u;         // [L] listed unique index
  uint32_t* s_row;       // [L] table row (static) or slot (hashed), same order
  uint32_t* s_bag;       // [L] dedup-set slot, same order
  // unfused backward: lookups sorted by unique row, (unique index, bag) of each position
  // (one-hot: the bag is the lookup itself); the same memory as s_u and s_row (the two
  // uses belong to different backwards)
  uint2* s_ub;           // [L]
  float* g;              // [L][D] per-unique gradient rows, zero between steps
  const float* zero_row; // [D] zeros: bulk-copy source for a rejected lookup
  uint32_t* scan_tmp;    // block sums of the scan
  uint32_t* counters;    // kNumCounters
  uint32_t* tier_hist;   // tiered: [64] cache slots by idle steps (watermark check)
  uint32_t first_wait_polls;  // polls of the tensor-core backward's first bounded wait
                              // (normally the full limit; a test knob can lower it)
};

struct Ctx {
  emb_config cfg;
  Params p;
  int num_sms = 0;
  int device = 0;
  int64_t total_rows = 0;
  int64_t max_batch = 0, max_lookups = 0;
  int64_t set_cap = 0;
  std::vector<int64_t> rows;
  std::vector<void*> allocs;
  // state of the last forward
  int64_t last_batch = -1, last_nnz = -1;
  int fwd_kind = 0;  // 0: none pending, 1: emb_forward, 2: emb_forward_interact
  bool multi_hot = false;
  bool set_dirty = false;
  int fwd_impl = 0;  // fused interaction forward: 0 automatic, 1 tensor cores, 2 FMA pipes
  int bwd_impl = 0;  // fused interaction backward: 0 automatic, 1 tensor cores, 2 FMA pipes
  int host_chunks = 2;  // sample chunks of the pipelined host-buffer step
  bool staged_update = true;  // all-rows update through shared-memory staging where it applies
  uint32_t step = 0;    // backward steps run (hashed tables stamp keys with it)
  bool track = false;   // hashed: per-key counts and last steps kept (emb_set_admission)
  bool counted = false; // the pending fused forward also counted each unique row's lookups
  int64_t g_stale = 0;  // leading g rows a multi-hot step left non-zero (clear_stale_g)
  uint32_t decay_steps = 0;  // Adagrad Decay: backward steps per period (0: off)
  // tiered tables: rows of the host tier and its host-side addresses (total_rows = cache rows)
  bool tiered = false;
  int64_t host_rows = 0;
  void* host_table = nullptr;
  float* host_acc = nullptr;
  // the mappings behind them when they are huge-page host memory (else cudaHostAlloc'd)
  void* host_map[2] = {nullptr, nullptr};
  size_t host_map_len[2] = {0, 0};
  uint32_t decay_base = 0;   // backward steps run before Adagrad Decay was set
  // tiered tables: cache watermark (0, 0: off) and the prefetch's ordering events
  uint32_t wm_high = 0, wm_low = 0;
  cudaEvent_t ev_dedup = nullptr;     // recorded after each forward's dedup and cache fill
  cudaEvent_t ev_prefetch = nullptr;  // recorded at the end of each prefetch
  bool pf_pending = false;            // a prefetch the next forward or eviction must wait for
  // Once rows updated inside the tensor-core backward: -1 automatic, 0 never, 1 always
  int once_direct = -1;
  bool once_step = false;  // the pending step tracks once rows (decided at its forward)
  // U of the last deduplicated batch, in host-mapped pinned memory written by the inverse
  // kernel (host and device addresses of the same word)
  uint32_t* h_unique = nullptr;
  uint32_t* h_unique_dev = nullptr;
  // host-buffer step staging (allocated on first use)
  int64_t* st_ids = nullptr;
  int32_t* st_offs = nullptr;
  float *st_dense = nullptr, *st_dout = nullptr, *st_out = nullptr, *st_ddense = nullptr;
  // copy streams and events of the host-buffer step (created with the staging buffers)
  cudaStream_t st_h2d = nullptr, st_d2h = nullptr;
  cudaEvent_t ev_inputs = nullptr, ev_dout = nullptr, ev_fwd = nullptr, ev_out = nullptr;
  static constexpr int kMaxChunks = 8;  // pipeline chunks of the host-buffer step
  cudaEvent_t ev_chunk[4][kMaxChunks] = {};  // dense up, dout up, forward done, backward done
  // launch accounting / profiling
  int64_t launches = 0;
  bool prof_on = false;
  struct Rec {
    int kid;
    cudaEvent_t a, b;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> ev_pool;
  double prof_ms[K_NUM_KERNELS] = {};
  int64_t prof_n[K_NUM_KERNELS] = {};
};

// Launch bracket: counts the launch and, when profiling, records events around it.
struct LaunchScope {
  Ctx* c;
  int kid;
  cudaStream_t s;
  cudaEvent_t b = nullptr;
  LaunchScope(Ctx* c_, int kid_, cudaStream_t s_);
  ~LaunchScope();
};

int grid_for(const Ctx* c, int64_t work_items, int threads, int blocks_per_sm = 8);

// CTAs of `kern` that fit on one SM with `threads` threads and `smem` bytes of dynamic shared
// memory.  Registers: each of the SM's four scheduler partitions holds a quarter of the
// register file, allocated per warp in units of 256.  Shared memory: the whole per-SM
// amount (the driver sizes the carveout at launch; the runtime's occupancy query instead
// assumes the kernel's current carveout and can report fewer).  0 when a query fails.
template <typename K>
int resident_ctas(const Ctx* c, K kern, int threads, int smem) {
  cudaFuncAttributes fa{};
  int regs_sm = 0, smem_sm = 0, smem_rsv = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncGetAttributes(&fa, kern) != cudaSuccess ||
      cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, c->device) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const int warps = (threads + 31) / 32;
  const int regs_warp = ((fa.numRegs * 32 + 255) / 256) * 256;
  const int warps_sm = 4 * ((regs_sm / 4) / regs_warp);
  const int by_regs = warps_sm / warps;
  const int by_smem = smem_sm / (smem + (int)fa.sharedSizeBytes + smem_rsv);
  const int by_threads = 2048 / (warps * 32);
  int n = by_regs < by_smem ? by_regs : by_smem;
  return n < by_threads ? n : by_threads;
}

// ---- launchers (defined in the kernel translation units) ----
cudaError_t launch_init_table(Ctx* c, cudaStream_t s);
cudaError_t launch_init_hash(Ctx* c, cudaStream_t s);
cudaError_t launch_reset_set(Ctx* c, cudaStream_t s);
cudaError_t launch_map_dedup(Ctx* c, const int64_t* ids, const int32_t* offs, int64_t nnz,
                             int64_t batch, cudaStream_t s);
cudaError_t launch_pool(Ctx* c, int64_t batch, float* pooled, cudaStream_t s);
cudaError_t launch_interact_fwd(Ctx* c, const float* dense, const float* pooled, int64_t batch,
                                float* out, cudaStream_t s);
cudaError_t launch_interact_bwd(Ctx* c, const float* dout, const float* dense,
                                const float* pooled, int64_t batch, float* ddense,
                                float* dpooled, cudaStream_t s);
cudaError_t launch_fused_fwd(Ctx* c, const float* dense, int64_t batch, float* out,
                             cudaStream_t s);
cudaError_t launch_fused_bwd(Ctx* c, const float* dout, const float* dense, int64_t batch,
                             float* ddense, cudaStream_t s);
bool reg_supported(const Ctx* c);
// tensor-core forward (fp32 one-hot, D = 128, T+1 <= 32) and whether it is the one in use
bool tc_fwd_supported(const Ctx* c);
bool use_tc_fwd(const Ctx* c);
cudaError_t launch_fused_fwd_tc(Ctx* c, const float* dense, int64_t batch, float* out,
                                cudaStream_t s);
bool tc_supported(const Ctx* c);
bool fused_fwd_records_inverse(const Ctx* c);
bool use_tc_bwd(const Ctx* c);
// Whether the tensor-core backward can update once rows itself (per-element Adagrad only).
bool once_direct_ok(const Ctx* c);
cudaError_t launch_fused_bwd_tc(Ctx* c, const float* dout, const float* dense, int64_t batch,
                                float* ddense, cudaStream_t s);
cudaError_t launch_inverse(Ctx* c, int64_t nnz, cudaStream_t s);
cudaError_t launch_fused_fwd_reg(Ctx* c, const float* dense, int64_t batch, float* out,
                                 cudaStream_t s);
cudaError_t launch_fused_bwd_reg(Ctx* c, const float* dout, const float* dense, int64_t batch,
                                 float* ddense, cudaStream_t s);
cudaError_t launch_backward_csr(Ctx* c, const float* dpooled, int64_t batch, int64_t nnz,
                                cudaStream_t s);
// stamp: tracked keys without admission holds; the update (or, in a step with once rows, the
// split before it) also does k_admit's counting and stamping.
cudaError_t launch_adagrad_from_g(Ctx* c, int64_t max_unique, cudaStream_t s, bool stamp = false);
cudaError_t launch_unique_count(Ctx* c, int64_t nnz, uint32_t* counts, int64_t* keys,
                                cudaStream_t s);
cudaError_t launch_read_rows(Ctx* c, const uint32_t* rows, int64_t n, float* w, float* acc,
                             cudaStream_t s);
cudaError_t launch_find_keys(Ctx* c, const int64_t* keys, int64_t n, uint32_t* rows,
                             cudaStream_t s);
cudaError_t launch_export_hash(Ctx* c, int64_t cap, int64_t* keys, uint32_t* rows, uint32_t* count,
                               cudaStream_t s);
// hashed tables: per unique key of the step, count its lookups (p.cnt), stamp the step and
// set its admission hold
cudaError_t launch_admit(Ctx* c, cudaStream_t s);
cudaError_t launch_tier_fill(Ctx* c, int64_t max_new, cudaStream_t s);
// tiered: find or insert the rows of a (next) batch in the cache and copy the new ones in
// from the host tier, stamped with `stamp` as their last step
cudaError_t launch_prefetch(Ctx* c, const int64_t* ids, const int32_t* offs, int64_t nnz,
                            int64_t batch, uint32_t stamp, cudaStream_t s);
// tiered: when more than `high` cache slots are in use, evict the longest-idle rows down to
// at most `low` (threshold chosen on the device); otherwise nothing
cudaError_t launch_tier_watermark(Ctx* c, uint32_t high, uint32_t low, cudaStream_t s);
cudaError_t launch_count_admit(Ctx* c, int64_t nnz, cudaStream_t s);
cudaError_t clear_stale_g(Ctx* c, cudaStream_t s);
cudaError_t launch_inverse_counts(Ctx* c, int64_t nnz, cudaStream_t s);
cudaError_t launch_evict(Ctx* c, uint32_t max_idle, uint32_t min_count, cudaStream_t s);
// cross interaction (context-free)
cudaError_t launch_cross_fwd(const float* x0, const float* xl, const float* w, const float* b,
                             int64_t B, int K, float* out, cudaStream_t s);
cudaError_t launch_cross_bwd(const float* x0, const float* xl, const float* w, const float* dout,
                             int64_t B, int K, float* dx0, float* dxl, float* dw, float* db,
                             cudaStream_t s);
// int8 row codec (context-free)
cudaError_t launch_quantize_rows(const float* x, int64_t n, int d, int8_t* q, float* scale,
                                 cudaStream_t s);
cudaError_t launch_dequantize_rows(const int8_t* q, const float* scale, int64_t n, int d,
                                   float* x, cudaStream_t s);
cudaError_t launch_key_stats(Ctx* c, const uint32_t* rows, int64_t n, uint32_t* freq,
                             uint32_t* last, cudaStream_t s);

// ---- device helpers ----
#ifdef __CUDACC__

__device__ __forceinline__ void raise_flag(uint32_t* counters, uint32_t f) {
  atomicOr(counters + kFlags, f);
}

// Adagrad Decay: the accumulator discount of a row last updated in period `last`, now in
// period `now` (rate^(now - last); 1 within the same period).
__device__ __forceinline__ float acc_decay(uint32_t last, uint32_t now, float rate) {
  return now > last ? powf(rate, (float)(now - last)) : 1.f;
}

// Per-element Adagrad on one parameter w with accumulator a and gradient g: a += g*g, then
// w -= lr * g / (sqrt(a) + eps).  sqrt(a) is taken as a * rsqrt(a) and the quotient with
// the fast reciprocal (each within a few units in the last place, so the step carries a
// relative error below 1e-6); every kernel that updates rows per element uses this one
// sequence, so a row gets the same bits whichever kernel updates it.
__device__ __forceinline__ void adagrad_elem(float& w, float& a, float g, float lr, float eps) {
  a = __fmaf_rn(g, g, a);
  const float root = a > 0.f ? a * rsqrtf(a) : 0.f;
  w = w - __fdividef(lr * g, root + eps);
}

// murmur3 32-bit finaliser (Appleby), used to spread row numbers over the dedup set
__device__ __forceinline__ uint32_t mix32(uint32_t h) {
  h ^= h >> 16;
  h *= 0x85EBCA6Bu;
  h ^= h >> 13;
  h *= 0xC2B2AE35u;
  h ^= h >> 16;
  return h;
}

// murmur3 64-bit finaliser, used to spread keys over the hashed table
__device__ __forceinline__ uint64_t mix64(uint64_t k) {
  k ^= k >> 33;
  k *= 0xFF51AFD7ED558CCDull;
  k ^= k >> 33;
  k *= 0xC4CEB9FE1A85EC53ull;
  k ^= k >> 33;
  return k;
}

__device__ __forceinline__ float4 f4_add(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}
__device__ __forceinline__ float4 f4_scale(float4 a, float s) {
  return make_float4(a.x * s, a.y * s, a.z * s, a.w * s);
}
__device__ __forceinline__ float4 f4_div(float4 a, float s) {
  return make_float4(a.x / s, a.y / s, a.z / s, a.w / s);
}

// fp32 vector red (no return) into global memory; 16-byte aligned address
__device__ __forceinline__ void red_add_f4(float* addr, float4 v) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

// Load 16 bytes of a parameter row as fp32: chunk `q` of the row holds elements
// [4q, 4q+4) (fp32 table).  For bf16 tables a 16-byte load holds 8 elements; see
// load_row8_bf16.
__device__ __forceinline__ float4 ld_row4_f32(const float* row, int q) {
  return __ldg(reinterpret_cast<const float4*>(row) + q);
}

__device__ __forceinline__ void ld_row8_bf16(const __nv_bfloat16* row, int q, float4& lo,
                                             float4& hi) {
  uint4 raw = __ldg(reinterpret_cast<const uint4*>(row) + q);
  __nv_bfloat162 h0 = *reinterpret_cast<__nv_bfloat162*>(&raw.x);
  __nv_bfloat162 h1 = *reinterpret_cast<__nv_bfloat162*>(&raw.y);
  __nv_bfloat162 h2 = *reinterpret_cast<__nv_bfloat162*>(&raw.z);
  __nv_bfloat162 h3 = *reinterpret_cast<__nv_bfloat162*>(&raw.w);
  float2 a = __bfloat1622float2(h0), b = __bfloat1622float2(h1);
  float2 c = __bfloat1622float2(h2), d = __bfloat1622float2(h3);
  lo = make_float4(a.x, a.y, b.x, b.y);
  hi = make_float4(c.x, c.y, d.x, d.y);
}

#endif  // __CUDACC__

}  // namespace emb
