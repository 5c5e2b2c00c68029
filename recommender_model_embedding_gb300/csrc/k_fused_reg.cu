// Fused lookup + pooling + dot interaction (forward) and interaction backward + gradient
// scatter (backward) for fp32 one-hot tables with 26 features (F = 27 interaction vectors,
// D <= 128): the Criteo-shaped workload.
//
// OneEmbedding article, "operator optimisation" (FusedDotFeatureInteraction) and HugeCTR
// interview, section 3 (5) (pooling fused with its neighbour) name the fusion.
//
// Register-resident design: one warp per sample, lane l owns elements 4l..4l+3 of every
// vector, so a sample's X (27 x 128 fp32) lives in 27 float4 registers per lane and the
// arithmetic needs no shared-memory reads of X at all.  While a warp computes sample k from
// registers, the 27 rows of its next sample stream into the warp's own shared-memory slab
// with per-lane 16-byte cp.async copies; each lane copies and later reads only its own
// chunk of every row, so the slab needs no warp barrier, and every warp keeps one sample's
// 14 KB of random rows in flight.
//  - forward: each lane forms the 351 partial dot products over its 4 elements, 32 at a
//    time (the pair walk is unrolled at compile time, so every register index is fixed),
//    and a transpose through the warp's shared buffer leaves lane l with the sum of product
//    l of the chunk over all lanes, which it stores next to its neighbours'.
//  - backward: G is built in the warp's shared memory from the dout row (prefetched with
//    cp.async one sample ahead); dX rows 9g..9g+8 accumulate G[i][j] x_j with broadcast
//    coefficient loads; each row of a lookup goes to the per-unique-row gradient buffer with
//    one 512-byte vector reduction (red.global.add.v4.f32 per lane).
// Measured on GB300: 512-byte TMA bulk copies of scattered rows reached only ~1.5 TB/s of
// gathered data (few copies in flight per SM), and staging X in shared memory for a blocked
// FMA kernel made the shared-memory pipe and the staging latency the limit.
#include <utility>

#include "interact_common.cuh"

namespace emb {

constexpr int kRegF = 27;    // interaction vectors this kernel is built for (T = 26)
constexpr int kRegWarps = 2;  // warps per CTA
constexpr int kRegPairs = kRegF * (kRegF - 1) / 2;
constexpr int kRegDout = (128 + kRegPairs + 31) / 32;  // dout values per lane

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Copy this lane's chunk of sample s's rows into the slab: row 0 = dense, row t+1 = the row
// of feature t (r = that row, held by lane t; a rejected lookup copies the zero row).
__device__ __forceinline__ void stage_rows(const Params& p, float4* slab, int64_t s,
                                           const float* dense, uint32_t r, int lane) {
  const int T = kRegF - 1, D = p.D;
  const bool on = lane < (D >> 2);
  if (on) cp_async16(slab + lane, dense + s * D + 4 * lane);
#pragma unroll
  for (int t = 0; t < T; ++t) {
    const uint32_t rt = __shfl_sync(0xFFFFFFFFu, r, t);
    const float* src = rt != kNoRow ? reinterpret_cast<const float*>(p.table) + (int64_t)rt * D
                                    : p.zero_row;
    if (on) cp_async16(slab + (t + 1) * 32 + lane, src + 4 * lane);
  }
}

__device__ __forceinline__ void load_x(const float4* slab, float4 (&x)[kRegF], int lane, bool on) {
#pragma unroll
  for (int i = 0; i < kRegF; ++i) x[i] = on ? slab[i * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
}

// Packed two-lane fp32 arithmetic (one instruction for two independent fp32 operations).
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// a . b over four elements: (a.x b.x + a.z b.z) + (a.y b.y + a.w b.w) in two packed ops
__device__ __forceinline__ float dot4r(const float4& a, const float4& b) {
  uint64_t p, q;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(p) : "l"(pack2(a.x, a.y)), "l"(pack2(b.x, b.y)));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(pack2(a.z, a.w)), "l"(pack2(b.z, b.w)), "l"(p));
  float lo, hi;
  unpack2(q, lo, hi);
  return lo + hi;
}

constexpr int kChunkPairs = 32;  // partial products reduced together

// Sums over the warp of 32 values through a transpose in the warp's shared buffer:
// afterwards lane p returns the sum over all lanes of their value p.  Lane l writes its
// value p to row p, column l (each store of the warp fills one 128-byte row: no bank
// conflict); lane p reads row p back with eight 16-byte loads (rows 36 floats apart, so each
// quarter-warp's loads fall in distinct banks) and adds them pairwise with packed adds.
// Compared with a shuffle reduce-scatter this takes 56 instructions per 32 values instead of
// ~110 (the shuffles need two selects per value and stage).
constexpr int kRedStride = 36;  // floats per row of the transpose buffer

__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ float reduce_transpose32(const float (&v)[kChunkPairs], float* red,
                                                    int lane) {
#pragma unroll
  for (int q = 0; q < kChunkPairs; ++q) red[q * kRedStride + lane] = v[q];
  __syncwarp();
  const float4* row = reinterpret_cast<const float4*>(red + lane * kRedStride);
  uint64_t h[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 f = row[j];
    h[j] = add2(pack2(f.x, f.y), pack2(f.z, f.w));
  }
  __syncwarp();  // every lane has read its row before the buffer is written again
#pragma unroll
  for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) h[j] = add2(h[j], h[j + w]);
  float lo, hi;
  unpack2(h[0], lo, hi);
  return lo + hi;
}

// (a, b) of pair q in the order (1,0), (2,0), (2,1), (3,0), ...
constexpr int pair_a(int q) {
  int a = 1;
  while ((a + 1) * a / 2 <= q) ++a;
  return a;
}
constexpr int pair_b(int q) { return q - pair_a(q) * (pair_a(q) - 1) / 2; }

template <int Q>
struct PairIdx {
  static constexpr int a = Q < kRegPairs ? pair_a(Q) : 0;
  static constexpr int b = Q < kRegPairs ? pair_b(Q) : 0;
};

// Partial products of pairs Base..Base+31 (zero past the last pair), every register index
// fixed at compile time.
template <int Base, int... I>
__device__ __forceinline__ void chunk_products(const float4 (&x)[kRegF],
                                               float (&acc)[kChunkPairs],
                                               std::integer_sequence<int, I...>) {
  ((acc[I] = (Base + I < kRegPairs) ? dot4r(x[PairIdx<Base + I>::a], x[PairIdx<Base + I>::b])
                                    : 0.f),
   ...);
}

// Chunk C of the pair walk: 32 partial products, warp sum through the transpose buffer, one
// coalesced store; then chunk C+1.
template <int C>
__device__ __forceinline__ void pair_chunks(const float4 (&x)[kRegF], float (&acc)[kChunkPairs],
                                            float* red, float* prow, int lane) {
  constexpr int base = kChunkPairs * C;
  chunk_products<base>(x, acc, std::make_integer_sequence<int, kChunkPairs>{});
  const float r = reduce_transpose32(acc, red, lane);
  if (base + lane < kRegPairs) prow[base + lane] = r;
  if constexpr (base + kChunkPairs < kRegPairs) pair_chunks<C + 1>(x, acc, red, prow, lane);
}

// ---- forward ----

constexpr int kRegFwdWarpF4 = kRegF * 32 + 32 * kRedStride / 4;  // shared float4s per warp

// At most 168 registers (six CTAs' worth per SM): three warps fit in each scheduler
// partition's quarter of the register file instead of two.
__global__ void __launch_bounds__(kRegWarps * 32, 6) k_fused_fwd_reg(Params p, const float* dense,
                                                                  int64_t B, float* out) {
  extern __shared__ __align__(16) float4 smem_f4[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // per warp: the staging slab (27 rows x 32 lanes x 16 bytes), then the transpose buffer
  float4* slab = smem_f4 + warp * kRegFwdWarpF4;
  float* red = reinterpret_cast<float*>(slab + kRegF * 32);
  const int T = kRegF - 1, D = p.D;
  const bool on = lane < (D >> 2);
  const int64_t W = D + kRegPairs;
  const int64_t nw = (int64_t)gridDim.x * kRegWarps;
  int64_t s = (int64_t)blockIdx.x * kRegWarps + warp;
  uint32_t rnext = (s < B && lane < T) ? p.row_of[s * T + lane] : kNoRow;
  if (s < B) {
    stage_rows(p, slab, s, dense, rnext, lane);
    cp_async_commit();
  }
  rnext = (s + nw < B && lane < T) ? p.row_of[(s + nw) * T + lane] : kNoRow;
  for (; s < B; s += nw) {
    cp_async_wait_all();
    float4 x[kRegF];
    load_x(slab, x, lane, on);
    const int64_t sn = s + nw;
    if (sn < B) {
      stage_rows(p, slab, sn, dense, rnext, lane);
      cp_async_commit();
      rnext = (sn + nw < B && lane < T) ? p.row_of[(sn + nw) * T + lane] : kNoRow;
    }
    float* orow = out + s * W;
    if (on) {
      orow[4 * lane + 0] = x[0].x;
      orow[4 * lane + 1] = x[0].y;
      orow[4 * lane + 2] = x[0].z;
      orow[4 * lane + 3] = x[0].w;
    }
    float acc[kChunkPairs];
    pair_chunks<0>(x, acc, red, orow + D, lane);
  }
  cp_async_wait_all();
}

// ---- backward ----

// Shared memory per warp: slab [27][32] float4, G [27][48] floats (output rows 9g..9g+8 at
// columns 12g..12g+8 of contraction row j), dense-gradient passthrough [128], the next
// sample's dout row [15 * 32] (filled by cp.async), and per CTA the pair code of every
// dout position [15 * 32].
constexpr int kRegBwdWarpFloats = kRegF * 32 * 4 + kRegF * kGStride + 128 + kRegDout * 32;

__global__ void __launch_bounds__(kRegWarps * 32) k_fused_bwd_reg(Params p, const float* dout,
                                                                  const float* dense, int64_t B,
                                                                  float* ddense) {
  extern __shared__ __align__(16) float4 smem_f4[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* wbase = reinterpret_cast<float*>(smem_f4) + warp * kRegBwdWarpFloats;
  float4* slab = reinterpret_cast<float4*>(wbase);
  float* Gs = wbase + kRegF * 32 * 4;
  float* Ds = Gs + kRegF * kGStride;
  float* Db = Ds + 128;  // next sample's dout, element lane + 32m at Db[m * 32 + lane]
  int* code = reinterpret_cast<int*>(reinterpret_cast<float*>(smem_f4) +
                                     kRegWarps * kRegBwdWarpFloats);
  const int T = kRegF - 1, D = p.D;
  const int W = D + kRegPairs;
  const bool on = lane < (D >> 2);
  for (int e = lane; e < kRegF * kGStride; e += 32) Gs[e] = 0.f;  // diagonal/padding stay 0
  for (int e = threadIdx.x; e < kRegDout * 32; e += blockDim.x)
    code[e] = (e >= D && e < W) ? pair_code(e - D) : -1;
  __syncthreads();
  const int64_t nw = (int64_t)gridDim.x * kRegWarps;
  int64_t s = (int64_t)blockIdx.x * kRegWarps + warp;
  // dout row of sample ss into Db (each lane its own elements) and the unique index of the
  // lookup of feature `lane`
  auto stage_dout = [&](int64_t ss) {
    const float* drow = dout + ss * W;
#pragma unroll
    for (int m = 0; m < kRegDout; ++m) {
      const int e = lane + 32 * m;
      if (e < W) cp_async4(Db + m * 32 + lane, drow + e);
    }
  };
  uint32_t rnext = (s < B && lane < T) ? p.row_of[s * T + lane] : kNoRow;
  uint32_t inext = (s < B && lane < T) ? p.inv[s * T + lane] : kNoRow;
  if (s < B) {
    stage_rows(p, slab, s, dense, rnext, lane);
    stage_dout(s);
    cp_async_commit();
  }
  rnext = (s + nw < B && lane < T) ? p.row_of[(s + nw) * T + lane] : kNoRow;
  for (; s < B; s += nw) {
    cp_async_wait_all();
    float4 x[kRegF];
    load_x(slab, x, lane, on);
    float dcur[kRegDout];
#pragma unroll
    for (int m = 0; m < kRegDout; ++m) dcur[m] = Db[m * 32 + lane];
    const uint32_t icur = inext;
    const int64_t sn = s + nw;
    if (sn < B) {
      stage_rows(p, slab, sn, dense, rnext, lane);
      stage_dout(sn);
      cp_async_commit();
      rnext = (sn + nw < B && lane < T) ? p.row_of[(sn + nw) * T + lane] : kNoRow;
      inext = lane < T ? p.inv[sn * T + lane] : kNoRow;
    }
#pragma unroll
    for (int m = 0; m < kRegDout; ++m) {
      const int e = lane + 32 * m;
      if (e < D) {
        Ds[e] = dcur[m];
      } else if (e < W) {
        const int cd = code[m * 32 + lane];
        const int i = cd >> 8, j = cd & 255;
        Gs[j * kGStride + gcol(i)] = dcur[m];
        Gs[i * kGStride + gcol(j)] = dcur[m];
      }
    }
    __syncwarp();
#pragma unroll
    for (int g = 0; g < (kRegF + kRowsPerGroup - 1) / kRowsPerGroup; ++g) {
      float4 acc[kRowsPerGroup];
#pragma unroll
      for (int r = 0; r < kRowsPerGroup; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < kRegF; ++j) {
        const float* gr = Gs + j * kGStride + 12 * g;
        const float4 c0 = reinterpret_cast<const float4*>(gr)[0];
        const float4 c1 = reinterpret_cast<const float4*>(gr)[1];
        const float c8 = gr[8];
        const float cf[kRowsPerGroup] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w, c8};
#pragma unroll
        for (int r = 0; r < kRowsPerGroup; ++r) {
          acc[r].x = fmaf(cf[r], x[j].x, acc[r].x);
          acc[r].y = fmaf(cf[r], x[j].y, acc[r].y);
          acc[r].z = fmaf(cf[r], x[j].z, acc[r].z);
          acc[r].w = fmaf(cf[r], x[j].w, acc[r].w);
        }
      }
#pragma unroll
      for (int r = 0; r < kRowsPerGroup; ++r) {
        const int i = kRowsPerGroup * g + r;
        if (i >= kRegF) break;
        if (i == 0) {
          if (on)
            reinterpret_cast<float4*>(ddense + s * D)[lane] =
                f4_add(acc[0], reinterpret_cast<const float4*>(Ds)[lane]);
        } else {
          const uint32_t u = __shfl_sync(0xFFFFFFFFu, icur, i - 1);
          if (on && u != kNoRow) red_add_f4(p.g + (int64_t)u * D + 4 * lane, acc[r]);
        }
      }
    }
    __syncwarp();
  }
  cp_async_wait_all();
}

// ---- launchers ----

bool reg_supported(const Ctx* c) {
  return !c->p.bf16 && !c->multi_hot && c->p.T + 1 == kRegF && c->p.D <= 128;
}

template <typename K>
static int reg_grid(Ctx* c, K kern, int smem, int64_t B) {
  int per_sm = resident_ctas(c, kern, kRegWarps * 32, smem);
  if (per_sm < 1) per_sm = 1;
  int64_t grid = (int64_t)per_sm * c->num_sms;
  const int64_t need = (B + kRegWarps - 1) / kRegWarps;
  if (grid > need) grid = need;
  return (int)grid;
}

cudaError_t launch_fused_fwd_reg(Ctx* c, const float* dense, int64_t B, float* out,
                                 cudaStream_t s) {
  const int smem = kRegWarps * kRegFwdWarpF4 * 16;
  const int grid = reg_grid(c, k_fused_fwd_reg, smem, B);
  LaunchScope ls(c, K_FUSED_FWD, s);
  k_fused_fwd_reg<<<grid, kRegWarps * 32, smem, s>>>(c->p, dense, B, out);
  return cudaGetLastError();
}

cudaError_t launch_fused_bwd_reg(Ctx* c, const float* dout, const float* dense, int64_t B,
                                 float* ddense, cudaStream_t s) {
  const int smem = (kRegWarps * kRegBwdWarpFloats + kRegDout * 32) * 4;
  const int grid = reg_grid(c, k_fused_bwd_reg, smem, B);
  LaunchScope ls(c, K_FUSED_BWD, s);
  k_fused_bwd_reg<<<grid, kRegWarps * 32, smem, s>>>(c->p, dout, dense, B, ddense);
  return cudaGetLastError();
}

}  // namespace emb
