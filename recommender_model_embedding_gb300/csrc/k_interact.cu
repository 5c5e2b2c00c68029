// Pairwise dot feature interaction, forward and backward, standalone and fused with the
// row gather.
//
// OneEmbedding article, "operator optimisation": DLRM's feature interaction as one fused
// operator (FusedDotFeatureInteraction); "usability": interaction(dense_fields, embedding).
// HugeCTR interview, section 3 (5): pooling merged with its neighbouring operator so the
// pooled vectors never make a round trip through memory.
//
// Per sample b: X = [x_0 = dense_b; x_1..x_T = pooled_b,0..T-1]  (F = T+1 vectors of D).
//   forward : out_b = [dense_b || x_i . x_j for i = 1..F-1, j = 0..i-1]
//   backward: G_ij = G_ji = dout_b[D + pair(i,j)], G_ii = 0; dX = G X;
//             d_dense = dX_0 + dout_b[0:D]; d_pooled[t] = dX_{t+1}.
//
// Work split: one CTA per sample at a time, a few warps sharing the sample's X.  X sits in
// shared memory row-major as float4 chunks of 4 consecutive k: row i at slot(i) = i + i/4,
// row stride RS = (D/4)|1 chunks (odd).  With that layout the chunks one instruction
// touches fall in distinct bank groups for every access pattern used here: the forward
// reads x_{4I+r}[kc] for distinct I (slots 5I+r), the backward reads x_j[kc] with lane =
// kc, and staging writes row chunks with lane = chunk.
//  - forward: lane -> one 4x4 block (I >= J) of the lower triangle of X X^T; the warps of
//    the CTA split the k range and their partial blocks are summed through shared memory
//    (8 shared loads per 64 fp32 FMAs in the main loop);
//  - backward: warp g -> dX rows 9g..9g+8, lane -> chunk kc: dX[i][kc] += G[i][j] x_j[kc]
//    (4 shared loads per 36 FMAs); G is stored by contraction index j with the 9 rows of a
//    group in one aligned 12-float run, so a lane reads all 9 coefficients of row j at once.
//
// Fused fp32 one-hot path (the Criteo-shaped workload): each CTA keeps two X buffers and
// two mbarriers and runs a software pipeline over its samples -- while it computes sample
// k, the 27 rows of sample k+1 (dense vector + one table row per feature, 512 bytes each)
// are already on their way as TMA bulk copies (cp.async.bulk, completion counted in bytes
// on the buffer's mbarrier).  Every wait on an mbarrier is bounded; a wait that runs out
// raises EMB_FLAG_WAIT_LIMIT, waits (bounded) for the copies still in flight and leaves
// the kernel instead of hanging.  Other fused variants (multi-hot bags, bf16 storage)
// stage X with 16-byte register loads instead.  The fused backward adds each dX row
// (scaled by 1/L for mean pooling) into the per-unique-row gradient buffer with vector
// reductions.
#include <math.h>

#include "emb_internal.cuh"

namespace emb {

constexpr int kFwdWarps = 4;      // warps per CTA in the forward (split of the k range)
constexpr int kGStride = 48;      // floats per row of the backward coefficient table
constexpr int kRowsPerGroup = 9;  // dX rows per warp in the backward
constexpr int kMaxDoutPerLane = (128 + kMaxF * (kMaxF - 1) / 2 + 31) / 32;
constexpr int kMaxBlocks = 36;       // 4x4 blocks of the lower triangle for F <= 32
constexpr int kWaitLimit = 1 << 22;  // try_wait polls before a wait gives up

enum Src : int { SRC_POOLED = 0, SRC_GATHER = 1, SRC_TMA = 2 };

struct ILayout {
  int F, Fpad, KC, RS, nslots;
  int x_f4;       // float4 per X buffer
  int nbuf;       // X buffers per CTA
  int nblk;       // forward 4x4 blocks
  int nwarps;     // warps per CTA
  int p_f;        // floats of the forward partial sums
  int g_f;        // floats of the backward coefficient table
  int d_f;        // floats of the backward dense-gradient staging
  int cta_bytes;  // shared memory per CTA (16 bytes of mbarriers first)
};

static inline int host_slot(int i) { return i + (i >> 2); }
__device__ __forceinline__ int xslot(int i) { return i + (i >> 2); }
__device__ __forceinline__ int gcol(int i) { return 12 * (i / kRowsPerGroup) + i % kRowsPerGroup; }

static ILayout make_layout(int T, int D, bool bwd, bool tma) {
  ILayout L;
  L.F = T + 1;
  L.Fpad = (L.F + 3) & ~3;
  L.KC = D / 4;
  L.RS = L.KC | 1;
  L.nslots = host_slot(L.Fpad - 1) + 1;
  L.x_f4 = L.nslots * L.RS;
  L.nbuf = tma ? 2 : 1;
  const int R = L.Fpad / 4;
  L.nblk = R * (R + 1) / 2;
  L.nwarps = bwd ? (L.F + kRowsPerGroup - 1) / kRowsPerGroup : kFwdWarps;
  L.p_f = bwd ? 0 : L.nwarps * 16 * L.nblk + kMaxBlocks;  // + block coordinate table
  L.g_f = bwd ? L.F * kGStride : 0;
  L.d_f = bwd ? D : 0;
  const int bytes = 16 + L.nbuf * L.x_f4 * 16 + L.p_f * 4 + L.g_f * 4 + L.d_f * 4 + (bwd ? 4 * 32 : 0);
  L.cta_bytes = (bytes + 15) & ~15;
  return L;
}

// ---- mbarrier / bulk-copy primitives (PTX ISA: mbarrier, cp.async.bulk) ----

__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred P;\n mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n selp.u32 %0, "
      "1, 0, P;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; gives up after kWaitLimit polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  for (int n = 0; n < kWaitLimit; ++n)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Every thread of the CTA waits for buffer b of the two-buffer pipeline.  The CTA goes on
// only if every thread saw the phase complete; otherwise thread 0 flags the failure and
// gives the copies still in flight (this buffer's and, when issued, the other buffer's)
// one more bounded wait, and the whole CTA leaves the kernel together.
__device__ __forceinline__ bool cta_pipeline_wait(const Params& p, uint64_t* bar, int b,
                                                  uint32_t& phase0, uint32_t& phase1,
                                                  bool other_issued) {
  uint32_t& ph = b ? phase1 : phase0;
  const bool ok = mbar_wait_bounded(&bar[b], ph);
  if (__syncthreads_and(ok)) {
    ph ^= 1u;
    return true;
  }
  if (threadIdx.x == 0) {
    raise_flag(p.counters, EMB_FLAG_WAIT_LIMIT);
    mbar_wait_bounded(&bar[b], ph);
    if (other_issued) mbar_wait_bounded(&bar[b ^ 1], b ? phase0 : phase1);
  }
  __syncthreads();
  return false;
}

// ---- staging X of one sample ----

// Issue the bulk copies of sample s into buffer X (fp32 one-hot), one warp: lane t < T
// copies the row of feature t, lane T the dense vector; a rejected lookup gets a zero row
// instead.  With REC_INV (forward), lanes t < T also record the unique index of their
// lookup for the fused backward.
template <bool REC_INV>
__device__ __forceinline__ void tma_issue(const Params& p, const ILayout& L, float4* X,
                                          uint64_t* bar, int64_t s, const float* dense,
                                          int lane) {
  const int T = p.T, D = p.D;
  const uint32_t rb = (uint32_t)D * 4u;
  uint32_t r = kNoRow;
  if (lane < T) {
    const int64_t q = s * T + lane;
    r = p.row_of[q];
    if (REC_INV) {
      const uint32_t sl = p.slot_of[q];
      p.inv[q] = (r != kNoRow && sl != kEmpty32) ? p.set_vals[sl] : kNoRow;
    }
  }
  const bool copy = (lane == T) || (lane < T && r != kNoRow);
  const unsigned vm = __ballot_sync(0xFFFFFFFFu, copy);
  if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)__popc(vm) * rb);
  if (copy) {
    const float* src = (lane == T) ? dense + s * D
                                   : reinterpret_cast<const float*>(p.table) + (int64_t)r * D;
    fence_proxy_async();
    bulk_copy_g2s(X + xslot(lane == T ? 0 : lane + 1) * L.RS, src, rb, bar);
  } else if (lane < T) {
    float4* dst = X + xslot(lane + 1) * L.RS;
    for (int q = 0; q < L.KC; ++q) dst[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Synchronous staging (standalone interaction, multi-hot bags, bf16 storage): lane = chunk;
// warp w of NW stages the rows i with i % NW == w (row 0 = dense).
template <int SRC, bool BF16>
__device__ __forceinline__ void stage_x(const Params& p, const ILayout& L, float4* X, int64_t s,
                                        const float* dense, const float* pooled, int one_hot,
                                        int lane, int w, int NW) {
  const int D = p.D, T = p.T, KC = L.KC, RS = L.RS;
  if (w == 0)
    for (int kc = lane; kc < KC; kc += 32)
      X[xslot(0) * RS + kc] = __ldg(reinterpret_cast<const float4*>(dense + s * D) + kc);
  if (SRC == SRC_POOLED) {
    for (int t = (w + NW - 1) % NW; t < T; t += NW) {
      const float4* src = reinterpret_cast<const float4*>(pooled + (s * T + t) * D);
      for (int kc = lane; kc < KC; kc += 32) X[xslot(t + 1) * RS + kc] = __ldg(src + kc);
    }
    return;
  }
  constexpr int EPC = BF16 ? 8 : 4;  // elements per 16-byte load
  const int nchunk = D / EPC;
  for (int t = (w + NW - 1) % NW; t < T; t += NW) {
    const int64_t bag = s * T + t;
    int64_t beg = bag, end = bag + 1;
    if (!one_hot) {
      beg = p.offs[bag];
      end = p.offs[bag + 1];
      if (beg < 0 || end < beg || end > p.nnz) beg = end = 0;
    }
    const float Lb = (float)(end - beg);
    float4* dst = X + xslot(t + 1) * RS;
    for (int q = lane; q < nchunk; q += 32) {
      float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
      int64_t i = beg;
      for (; i + 2 <= end; i += 2) {  // two rows in flight per lane
        const uint32_t r0 = p.row_of[i], r1 = p.row_of[i + 1];
        if (BF16) {
          float4 l0, h0, l1, h1;
          l0 = h0 = l1 = h1 = make_float4(0.f, 0.f, 0.f, 0.f);
          if (r0 != kNoRow)
            ld_row8_bf16(reinterpret_cast<const __nv_bfloat16*>(p.table) + (int64_t)r0 * D, q, l0, h0);
          if (r1 != kNoRow)
            ld_row8_bf16(reinterpret_cast<const __nv_bfloat16*>(p.table) + (int64_t)r1 * D, q, l1, h1);
          a0 = f4_add(a0, f4_add(l0, l1));
          a1 = f4_add(a1, f4_add(h0, h1));
        } else {
          const float* tb = reinterpret_cast<const float*>(p.table);
          const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
          const float4 v0 = r0 != kNoRow ? ld_row4_f32(tb + (int64_t)r0 * D, q) : z;
          const float4 v1 = r1 != kNoRow ? ld_row4_f32(tb + (int64_t)r1 * D, q) : z;
          a0 = f4_add(a0, f4_add(v0, v1));
        }
      }
      for (; i < end; ++i) {
        const uint32_t r = p.row_of[i];
        if (r == kNoRow) continue;
        if (BF16) {
          float4 lo, hi;
          ld_row8_bf16(reinterpret_cast<const __nv_bfloat16*>(p.table) + (int64_t)r * D, q, lo, hi);
          a0 = f4_add(a0, lo);
          a1 = f4_add(a1, hi);
        } else {
          a0 = f4_add(a0, ld_row4_f32(reinterpret_cast<const float*>(p.table) + (int64_t)r * D, q));
        }
      }
      if (p.mean && Lb > 0.f) {
        a0 = f4_div(a0, Lb);
        a1 = f4_div(a1, Lb);
      }
      if (BF16) {
        dst[2 * q] = a0;
        dst[2 * q + 1] = a1;
      } else {
        dst[q] = a0;
      }
    }
  }
}

// Unique index of each lookup of sample s (fused forward, register staging), one warp.
__device__ __forceinline__ void record_inverse(const Params& p, int64_t s, int one_hot, int lane) {
  const int T = p.T;
  int64_t q0 = one_hot ? s * T : p.offs[s * T];
  int64_t q1 = one_hot ? (s + 1) * T : p.offs[(s + 1) * T];
  q0 = q0 < 0 ? 0 : q0;  // malformed offsets are flagged; stay inside [0, nnz)
  q1 = q1 > p.nnz ? p.nnz : q1;
  for (int64_t q = q0 + lane; q < q1; q += 32) {
    const uint32_t sl = p.slot_of[q];
    p.inv[q] = (p.row_of[q] != kNoRow && sl != kEmpty32) ? p.set_vals[sl] : kNoRow;
  }
}

// Zero the rows F..Fpad-1 of an X buffer (never written afterwards), whole CTA.
__device__ __forceinline__ void zero_pad_rows(const ILayout& L, float4* X) {
  const int n = (L.Fpad - L.F) * L.KC;
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int i = L.F + e / L.KC, kc = e % L.KC;
    X[xslot(i) * L.RS + kc] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// ---- forward compute ----

// Partial sums over kc in [kc0, kc1) of 4x4 block (I, J): acc[r*4+c] = x_{4I+r} . x_{4J+c}.
__device__ __forceinline__ void fwd_block(const ILayout& L, const float4* X, int I, int J, int kc0,
                                          int kc1, float* acc) {
  const int RS = L.RS;
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.f;
  const float4* ra = X + (5 * I) * RS;  // slot(4I + r) = 5I + r
  const float4* rb = X + (5 * J) * RS;
  for (int kc = kc0; kc < kc1; ++kc) {
    float4 a[4], b[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) a[r] = ra[r * RS + kc];
#pragma unroll
    for (int c = 0; c < 4; ++c) b[c] = rb[c * RS + kc];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r * 4 + c] = fmaf(a[r].x, b[c].x, acc[r * 4 + c]);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r * 4 + c] = fmaf(a[r].y, b[c].y, acc[r * 4 + c]);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r * 4 + c] = fmaf(a[r].z, b[c].z, acc[r * 4 + c]);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r * 4 + c] = fmaf(a[r].w, b[c].w, acc[r * 4 + c]);
  }
}

// ---- backward helpers ----

// This warp's share (m % NW == w) of the coefficient table of one sample:
// Gs[j*48 + gcol(i)] = G[i][j] and Ds[e] = dout[e] for e < D.  dv[m] = dout[lane + 32m];
// ptab[m] holds the (i, j) of pair lane + 32m - D.
__device__ __forceinline__ void build_g(float* Gs, float* Ds, const float* dv, const int* ptab,
                                        int D, int W, int lane, int w, int NW) {
#pragma unroll
  for (int m = 0; m < kMaxDoutPerLane; ++m) {
    if (m % NW != w) continue;
    const int e = lane + 32 * m;
    if (e < D) {
      Ds[e] = dv[m];
    } else if (e < W) {
      const int i = ptab[m] >> 8, j = ptab[m] & 255;
      Gs[j * kGStride + gcol(i)] = dv[m];
      Gs[i * kGStride + gcol(j)] = dv[m];
    }
  }
}

// dX rows 9g..9g+8 at chunk kc: acc[r] = sum_j G[9g+r][j] x_j[kc].
__device__ __forceinline__ void bwd_group(const ILayout& L, const float4* X, const float* Gs,
                                          int g, int kc, float4* acc) {
#pragma unroll
  for (int r = 0; r < kRowsPerGroup; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < L.F; ++j) {
    const float4 x = X[xslot(j) * L.RS + kc];
    const float* gr = Gs + j * kGStride + 12 * g;
    const float4 c0 = reinterpret_cast<const float4*>(gr)[0];
    const float4 c1 = reinterpret_cast<const float4*>(gr)[1];
    const float c8 = gr[8];
    const float cf[kRowsPerGroup] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w, c8};
#pragma unroll
    for (int r = 0; r < kRowsPerGroup; ++r) {
      acc[r].x = fmaf(cf[r], x.x, acc[r].x);
      acc[r].y = fmaf(cf[r], x.y, acc[r].y);
      acc[r].z = fmaf(cf[r], x.z, acc[r].z);
      acc[r].w = fmaf(cf[r], x.w, acc[r].w);
    }
  }
}

// This warp's share of the dout row of sample ss into registers (dv[m] = dout[ss][lane +
// 32m] for m % NW == w) and, for the fused one-hot path, the unique index of the lookup of
// feature `lane`.
__device__ __forceinline__ void load_dout(const Params& p, const float* dout, int64_t ss, int W,
                                          int T, bool fused_one_hot, int lane, int w, int NW,
                                          float* dv, uint32_t& iv) {
  const float* drow = dout + ss * W;
#pragma unroll
  for (int m = 0; m < kMaxDoutPerLane; ++m) {
    const int e = lane + 32 * m;
    dv[m] = (m % NW == w && e < W) ? __ldg(drow + e) : 0.f;
  }
  if (fused_one_hot && w == 0 && lane < T) iv = p.inv[ss * T + lane];
}

__device__ __forceinline__ int pair_code(int q) {
  int i = (int)((1.f + sqrtf(8.f * q + 1.f)) * 0.5f);
  while (i * (i - 1) / 2 > q) --i;
  while ((i + 1) * i / 2 <= q) ++i;
  const int j = q - i * (i - 1) / 2;
  return (i << 8) | j;
}

// ---- forward kernel ----

template <int SRC, bool BF16>
__global__ void __launch_bounds__(kFwdWarps * 32) k_interact_fwd(Params p, ILayout L,
                                                                 const float* dense,
                                                                 const float* pooled, int64_t B,
                                                                 float* out, int one_hot) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, NW = blockDim.x >> 5;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  float4* Xb = reinterpret_cast<float4*>(smem + 16);
  float* Ps = reinterpret_cast<float*>(Xb + L.nbuf * L.x_f4);   // [NW][16][nblk]
  int* Bij = reinterpret_cast<int*>(Ps + NW * 16 * L.nblk);      // (I << 8) | J per block
  const int D = p.D, F = L.F, nblk = L.nblk;
  const int64_t W = D + (int64_t)F * (F - 1) / 2;
  const int kc0 = (L.KC * w) / NW, kc1 = (L.KC * (w + 1)) / NW;
  const int64_t nw = gridDim.x;
  int64_t s = blockIdx.x;

  for (int b = 0; b < L.nbuf; ++b) zero_pad_rows(L, Xb + b * L.x_f4);
  if (threadIdx.x == 0) {
    int blk = 0;
    for (int I = 0; I < L.Fpad / 4; ++I)
      for (int J = 0; J <= I; ++J) Bij[blk++] = (I << 8) | J;
    if (SRC == SRC_TMA) {
      mbar_init(&bar[0], 1);
      mbar_init(&bar[1], 1);
      fence_mbar_init();
    }
  }
  __syncthreads();
  if (SRC == SRC_TMA && w == 0 && s < B) tma_issue<true>(p, L, Xb, &bar[0], s, dense, lane);
  uint32_t phase0 = 0, phase1 = 0;
  for (int k = 0; s < B; ++k, s += nw) {
    const int b = (SRC == SRC_TMA) ? (k & 1) : 0;
    const float4* X = Xb + b * L.x_f4;
    if (SRC == SRC_TMA) {
      const bool next = s + nw < B;
      if (w == 0 && next) tma_issue<true>(p, L, Xb + (b ^ 1) * L.x_f4, &bar[b ^ 1], s + nw, dense, lane);
      if (!cta_pipeline_wait(p, bar, b, phase0, phase1, next)) return;
    } else {
      stage_x<SRC, BF16>(p, L, Xb, s, dense, pooled, one_hot, lane, w, NW);
      if (SRC == SRC_GATHER && w == 0) record_inverse(p, s, one_hot, lane);
      __syncthreads();
    }
    for (int blk = lane; blk < nblk; blk += 32) {
      float acc[16];
      const int ij = Bij[blk];
      fwd_block(L, X, ij >> 8, ij & 255, kc0, kc1, acc);
#pragma unroll
      for (int e = 0; e < 16; ++e) Ps[(w * 16 + e) * nblk + blk] = acc[e];
    }
    __syncthreads();
    float* orow = out + s * W;
    const float* x0 = reinterpret_cast<const float*>(X);  // slot 0 = dense
    for (int e = threadIdx.x; e < D; e += blockDim.x) orow[e] = x0[e];
    for (int v = threadIdx.x; v < 16 * nblk; v += blockDim.x) {
      const int e = v / nblk, blk = v - e * nblk;
      const int ij = Bij[blk];
      const int i = 4 * (ij >> 8) + (e >> 2), j = 4 * (ij & 255) + (e & 3);
      if (i < F && j < i) {
        float sum = 0.f;
        for (int ww = 0; ww < NW; ++ww) sum += Ps[(ww * 16 + e) * nblk + blk];
        orow[D + i * (i - 1) / 2 + j] = sum;
      }
    }
    __syncthreads();
  }
}

// ---- backward kernel ----

template <int SRC, bool BF16>
__global__ void __launch_bounds__(128) k_interact_bwd(Params p, ILayout L, const float* dout,
                                                      const float* dense, const float* pooled,
                                                      int64_t B, float* ddense, float* dpooled,
                                                      int one_hot) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, NW = blockDim.x >> 5;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  float4* Xb = reinterpret_cast<float4*>(smem + 16);
  float* Gs = reinterpret_cast<float*>(Xb + L.nbuf * L.x_f4);
  float* Ds = Gs + L.g_f;
  uint32_t* Us = reinterpret_cast<uint32_t*>(Ds + L.d_f);  // unique index per feature
  const int D = p.D, T = p.T, F = L.F;
  const int W = D + F * (F - 1) / 2;
  const int g = w;  // dX rows 9g..9g+8
  const bool fused_one_hot = SRC != SRC_POOLED && one_hot;
  const int64_t nw = gridDim.x;
  int64_t s = blockIdx.x;

  for (int b = 0; b < L.nbuf; ++b) zero_pad_rows(L, Xb + b * L.x_f4);
  for (int e = threadIdx.x; e < L.g_f; e += blockDim.x) Gs[e] = 0.f;  // diagonal/padding stay 0
  int ptab[kMaxDoutPerLane];
#pragma unroll
  for (int m = 0; m < kMaxDoutPerLane; ++m) {
    const int e = lane + 32 * m;
    ptab[m] = (m % NW == w && e >= D && e < W) ? pair_code(e - D) : 0;
  }
  if (SRC == SRC_TMA && threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  float dcur[kMaxDoutPerLane], dnext[kMaxDoutPerLane];
  uint32_t icur = kNoRow, inext = kNoRow;
  if (s < B) {
    if (SRC == SRC_TMA && w == 0) tma_issue<false>(p, L, Xb, &bar[0], s, dense, lane);
    load_dout(p, dout, s, W, T, fused_one_hot, lane, w, NW, dcur, icur);
  }
  uint32_t phase0 = 0, phase1 = 0;
  for (int k = 0; s < B; ++k, s += nw) {
    const int b = (SRC == SRC_TMA) ? (k & 1) : 0;
    const float4* X = Xb + b * L.x_f4;
    const int64_t sn = s + nw;
    if (sn < B) {
      if (SRC == SRC_TMA && w == 0) tma_issue<false>(p, L, Xb + (b ^ 1) * L.x_f4, &bar[b ^ 1], sn, dense, lane);
      load_dout(p, dout, sn, W, T, fused_one_hot, lane, w, NW, dnext, inext);
    }
    if (SRC == SRC_TMA) {
      if (!cta_pipeline_wait(p, bar, b, phase0, phase1, sn < B)) return;
    } else {
      stage_x<SRC, BF16>(p, L, Xb, s, dense, pooled, one_hot, lane, w, NW);
    }
    build_g(Gs, Ds, dcur, ptab, D, W, lane, w, NW);
    if (fused_one_hot && w == 0 && lane < T) Us[lane] = icur;
    __syncthreads();
    for (int kc = lane; kc < L.KC; kc += 32) {
      float4 acc[kRowsPerGroup];
      bwd_group(L, X, Gs, g, kc, acc);
#pragma unroll
      for (int r = 0; r < kRowsPerGroup; ++r) {
        const int i = kRowsPerGroup * g + r;
        if (i >= F) break;
        float4 v = acc[r];
        if (i == 0) {
          v = f4_add(v, reinterpret_cast<const float4*>(Ds)[kc]);
          reinterpret_cast<float4*>(ddense + s * D)[kc] = v;
        } else if (SRC == SRC_POOLED) {
          reinterpret_cast<float4*>(dpooled + (s * T + (i - 1)) * D)[kc] = v;
        } else if (one_hot) {
          const uint32_t u = Us[i - 1];
          if (u != kNoRow) red_add_f4(p.g + (int64_t)u * D + 4 * kc, v);
        } else {
          const int64_t bag = s * T + (i - 1);
          int64_t q0 = p.offs[bag], q1 = p.offs[bag + 1];
          if (q0 < 0 || q1 < q0 || q1 > p.nnz) q0 = q1 = 0;
          if (p.mean && q1 > q0) v = f4_div(v, (float)(q1 - q0));
          for (int64_t q = q0; q < q1; ++q) {
            const uint32_t u = p.inv[q];
            if (u != kNoRow) red_add_f4(p.g + (int64_t)u * D + 4 * kc, v);
          }
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < kMaxDoutPerLane; ++m) dcur[m] = dnext[m];
    icur = inext;
  }
}

// ---- launchers ----

template <typename K>
static int persistent_grid(Ctx* c, K kern, int threads, size_t smem, int64_t B) {
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
  if (per_sm < 1) per_sm = 1;
  int64_t g = (int64_t)per_sm * c->num_sms;
  if (g > B) g = B;
  return (int)(g < 1 ? 1 : g);
}

static bool use_tma(const Ctx* c) { return !c->p.bf16 && !c->multi_hot; }

template <typename K>
static cudaError_t run_fwd(Ctx* c, K kern, const ILayout& L, const float* dense,
                           const float* pooled, int64_t B, float* out, int one_hot, int kid,
                           cudaStream_t s) {
  const int threads = L.nwarps * 32;
  const int grid = persistent_grid(c, kern, threads, L.cta_bytes, B);
  LaunchScope ls(c, kid, s);
  kern<<<grid, threads, L.cta_bytes, s>>>(c->p, L, dense, pooled, B, out, one_hot);
  return cudaGetLastError();
}

template <typename K>
static cudaError_t run_bwd(Ctx* c, K kern, const ILayout& L, const float* dout,
                           const float* dense, const float* pooled, int64_t B, float* ddense,
                           float* dpooled, int one_hot, int kid, cudaStream_t s) {
  const int threads = L.nwarps * 32;
  const int grid = persistent_grid(c, kern, threads, L.cta_bytes, B);
  LaunchScope ls(c, kid, s);
  kern<<<grid, threads, L.cta_bytes, s>>>(c->p, L, dout, dense, pooled, B, ddense, dpooled, one_hot);
  return cudaGetLastError();
}

cudaError_t launch_interact_fwd(Ctx* c, const float* dense, const float* pooled, int64_t B,
                                float* out, cudaStream_t s) {
  const ILayout L = make_layout(c->p.T, c->p.D, false, false);
  return run_fwd(c, k_interact_fwd<SRC_POOLED, false>, L, dense, pooled, B, out, 1,
                 K_INTERACT_FWD, s);
}

cudaError_t launch_interact_bwd(Ctx* c, const float* dout, const float* dense,
                                const float* pooled, int64_t B, float* ddense, float* dpooled,
                                cudaStream_t s) {
  const ILayout L = make_layout(c->p.T, c->p.D, true, false);
  return run_bwd(c, k_interact_bwd<SRC_POOLED, false>, L, dout, dense, pooled, B, ddense,
                 dpooled, 1, K_INTERACT_BWD, s);
}

cudaError_t launch_fused_fwd(Ctx* c, const float* dense, int64_t B, float* out, cudaStream_t s) {
  const bool tma = use_tma(c);
  const int one_hot = c->multi_hot ? 0 : 1;
  const ILayout L = make_layout(c->p.T, c->p.D, false, tma);
  if (tma)
    return run_fwd(c, k_interact_fwd<SRC_TMA, false>, L, dense, nullptr, B, out, one_hot,
                   K_FUSED_FWD, s);
  if (c->p.bf16)
    return run_fwd(c, k_interact_fwd<SRC_GATHER, true>, L, dense, nullptr, B, out, one_hot,
                   K_FUSED_FWD, s);
  return run_fwd(c, k_interact_fwd<SRC_GATHER, false>, L, dense, nullptr, B, out, one_hot,
                 K_FUSED_FWD, s);
}

cudaError_t launch_fused_bwd(Ctx* c, const float* dout, const float* dense, int64_t B,
                             float* ddense, cudaStream_t s) {
  const bool tma = use_tma(c);
  const int one_hot = c->multi_hot ? 0 : 1;
  const ILayout L = make_layout(c->p.T, c->p.D, true, tma);
  if (tma)
    return run_bwd(c, k_interact_bwd<SRC_TMA, false>, L, dout, dense, nullptr, B, ddense,
                   nullptr, one_hot, K_FUSED_BWD, s);
  if (c->p.bf16)
    return run_bwd(c, k_interact_bwd<SRC_GATHER, true>, L, dout, dense, nullptr, B, ddense,
                   nullptr, one_hot, K_FUSED_BWD, s);
  return run_bwd(c, k_interact_bwd<SRC_GATHER, false>, L, dout, dense, nullptr, B, ddense,
                 nullptr, one_hot, K_FUSED_BWD, s);
}

}  // namespace emb
