// Device helpers shared by the interaction kernels: the shared-memory layout of one sample's
// X, mbarrier / TMA bulk-copy primitives, the per-sample staging, and the forward and
// backward FMA micro-kernels.
//
// Layout of X (F = T+1 vectors of D floats): row i at slot(i) = i + i/4, row stride
// RS = (D/4)|1 float4 chunks (odd).  With it the chunks one instruction touches fall in
// distinct bank groups for every access pattern used: the forward reads x_{4I+r}[kc] for
// distinct I (slots 5I+r), the backward reads x_j[kc] with lane = kc, staging writes row
// chunks with lane = chunk, and TMA bulk copies land each 512-byte row 16-byte aligned.
#pragma once

#include <math.h>

#include "emb_internal.cuh"

namespace emb {

constexpr int kGStride = 48;      // floats per row of the backward coefficient table
constexpr int kRowsPerGroup = 9;  // dX rows per lane pass in the backward
constexpr int kMaxDoutPerLane = (128 + kMaxF * (kMaxF - 1) / 2 + 31) / 32;
constexpr int kMaxBlocks = 36;       // 4x4 blocks of the lower triangle for F <= 32
constexpr int kWaitLimit = 1 << 22;  // try_wait polls before a wait gives up

struct XShape {
  int F, Fpad, KC, RS, nslots, x_f4;
};

inline XShape make_xshape(int T, int D) {
  XShape X;
  X.F = T + 1;
  X.Fpad = (X.F + 3) & ~3;
  X.KC = D / 4;
  X.RS = X.KC | 1;
  X.nslots = (X.Fpad - 1) + ((X.Fpad - 1) >> 2) + 1;
  X.x_f4 = X.nslots * X.RS;
  return X;
}

__device__ __forceinline__ int xslot(int i) { return i + (i >> 2); }
__device__ __forceinline__ int gcol(int i) { return 12 * (i / kRowsPerGroup) + i % kRowsPerGroup; }

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

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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

// The same with a poll limit of `polls` (0: gives up at once, without polling).
__device__ __forceinline__ bool mbar_wait_polls(uint64_t* bar, uint32_t parity, uint32_t polls) {
  for (uint32_t n = 0; n < polls; ++n)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// ---- forward micro-kernel ----

// Sums over kc in [kc0, kc1) of 4x4 block (I, J): acc[r*4+c] = x_{4I+r} . x_{4J+c}.
__device__ __forceinline__ void fwd_block(const XShape& L, const float4* X, int I, int J, int kc0,
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

// ---- backward micro-kernels ----

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
__device__ __forceinline__ void bwd_group(const XShape& L, const float4* X, const float* Gs,
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
// 32m] for m % NW == w) and, when `with_inv`, the unique index of the lookup of feature
// `lane`.
__device__ __forceinline__ void load_dout(const Params& p, const float* dout, int64_t ss, int W,
                                          int T, bool with_inv, int lane, int w, int NW,
                                          float* dv, uint32_t& iv) {
  const float* drow = dout + ss * W;
#pragma unroll
  for (int m = 0; m < kMaxDoutPerLane; ++m) {
    const int e = lane + 32 * m;
    dv[m] = (m % NW == w && e < W) ? __ldg(drow + e) : 0.f;
  }
  if (with_inv && lane < T) iv = p.inv[ss * T + lane];
}

__device__ __forceinline__ int pair_code(int q) {
  int i = (int)((1.f + sqrtf(8.f * q + 1.f)) * 0.5f);
  while (i * (i - 1) / 2 > q) --i;
  while ((i + 1) * i / 2 <= q) ++i;
  const int j = q - i * (i - 1) / 2;
  return (i << 8) | j;
}

}  // namespace emb
