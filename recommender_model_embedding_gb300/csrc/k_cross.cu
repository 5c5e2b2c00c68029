// Cross interaction (one layer of a deep & cross network) over the concatenated feature
// vector of each sample.
//
// OneFlow OneEmbedding article, "operator optimisation": FusedCrossFeatureInteraction, with
// the cross layer of "Deep & Cross Network for Ad Click Predictions" (figure cited there):
// per sample, x_next = x0 * (xl . w) + b + xl, with x0, xl, w, b of width K.  Backward by
// the chain rule, with s = xl . w and t = x0 . dout per sample:
//   dxl = dout + w t,  dx0 = dout s,  dw = sum over samples of xl t,  db = sum of dout.
//
// Both directions are bound by HBM bandwidth (forward: x0 and xl in, out back, 12 K bytes
// per sample; backward: x0, xl, dout in, dx0 and dxl back, 20 K bytes), with w and b read
// from L2.  One warp per sample: a first pass over the row forms the dot product(s) with
// 16-byte loads (four in flight per lane and array), a warp reduction gives s (and t), and
// a second pass writes the outputs (the row is re-read from L1/L2).  The backward runs one
// or two CTAs of 16 warps per SM; dw and db are accumulated per CTA in shared memory (fp32
// partials of at most 32 samples folded into double sums) and added to the outputs with one
// fp32 atomic per column and CTA.
#include "emb_internal.cuh"

namespace emb {

constexpr int kCrossUnroll = 4;     // 16-byte chunks per lane and array in flight (forward)
constexpr int kCrossUnrollBwd = 2;  // the same for the backward's four arrays

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}

__global__ void __launch_bounds__(256) k_cross_fwd(const float4* x0, const float4* xl,
                                                   const float4* w, const float4* b, int64_t B,
                                                   int KC, float4* out) {
  const int lane = threadIdx.x & 31;
  const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t r = gwarp; r < B; r += nwarps) {
    const float4* xr = xl + r * KC;
    float s = 0.f;
    for (int c0 = 0; c0 < KC; c0 += 32 * kCrossUnroll) {
      float4 a[kCrossUnroll], v[kCrossUnroll];
#pragma unroll
      for (int u = 0; u < kCrossUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
        a[u] = c < KC ? xr[c] : make_float4(0.f, 0.f, 0.f, 0.f);
        v[u] = c < KC ? w[c] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kCrossUnroll; ++u) s += dot4(a[u], v[u]);
    }
    s = warp_sum(s);
    const float4* x0r = x0 + r * KC;
    float4* o = out + r * KC;
    for (int c0 = 0; c0 < KC; c0 += 32 * kCrossUnroll) {
      float4 a[kCrossUnroll], l[kCrossUnroll], bb[kCrossUnroll];
#pragma unroll
      for (int u = 0; u < kCrossUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < KC) {
          a[u] = x0r[c];
          l[u] = xr[c];
          bb[u] = b[c];
        }
      }
#pragma unroll
      for (int u = 0; u < kCrossUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < KC)
          o[c] = make_float4(fmaf(a[u].x, s, bb[u].x + l[u].x), fmaf(a[u].y, s, bb[u].y + l[u].y),
                             fmaf(a[u].z, s, bb[u].z + l[u].z), fmaf(a[u].w, s, bb[u].w + l[u].w));
      }
    }
  }
}

// Any width (one element per lane step).
__global__ void __launch_bounds__(256) k_cross_fwd_scalar(const float* x0, const float* xl,
                                                          const float* w, const float* b,
                                                          int64_t B, int K, float* out) {
  const int lane = threadIdx.x & 31;
  const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t r = gwarp; r < B; r += nwarps) {
    float s = 0.f;
    for (int k = lane; k < K; k += 32) s += xl[r * K + k] * w[k];
    s = warp_sum(s);
    for (int k = lane; k < K; k += 32) out[r * K + k] = fmaf(x0[r * K + k], s, b[k] + xl[r * K + k]);
  }
}

// dw and db: every warp adds its sample's terms into fp32 partials in shared memory
// (native shared-memory atomics); every two rounds (32 samples of the CTA) the partials are
// folded into double sums and cleared, so no fp32 partial holds more than 32 terms.
template <bool VEC>
__global__ void __launch_bounds__(512, 2) k_cross_bwd(const float* x0, const float* xl,
                                                      const float* w, const float* dout, int64_t B,
                                                      int K, float* dx0, float* dxl, float* dw,
                                                      float* db) {
  extern __shared__ double sacc[];  // [2][K] double sums, then [2][K] fp32 partials (dw, db)
  float* fdw = reinterpret_cast<float*>(sacc + 2 * K);
  float* fdb = fdw + K;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int k = threadIdx.x; k < 2 * K; k += blockDim.x) {
    sacc[k] = 0.0;
    fdw[k] = 0.f;
  }
  __syncthreads();
  auto fold = [&]() {
    __syncthreads();
    for (int k = threadIdx.x; k < 2 * K; k += blockDim.x) {
      sacc[k] += (double)fdw[k];
      fdw[k] = 0.f;
    }
    __syncthreads();
  };
  const int KC = K / 4;
  int round = 0;
  for (int64_t r0 = (int64_t)blockIdx.x * nw; r0 < B; r0 += (int64_t)gridDim.x * nw) {
    const int64_t r = r0 + warp;
    if (r < B) {
      float s = 0.f, t = 0.f;
      if (VEC) {
        const float4* a4 = reinterpret_cast<const float4*>(xl + r * K);
        const float4* b4 = reinterpret_cast<const float4*>(x0 + r * K);
        const float4* g4 = reinterpret_cast<const float4*>(dout + r * K);
        const float4* w4 = reinterpret_cast<const float4*>(w);
        for (int c0 = 0; c0 < KC; c0 += 32 * kCrossUnrollBwd) {
          float4 a[kCrossUnrollBwd], v[kCrossUnrollBwd], x[kCrossUnrollBwd], g[kCrossUnrollBwd];
#pragma unroll
          for (int u = 0; u < kCrossUnrollBwd; ++u) {
            const int c = c0 + u * 32 + lane;
            const bool in = c < KC;
            a[u] = in ? a4[c] : make_float4(0.f, 0.f, 0.f, 0.f);
            v[u] = in ? w4[c] : make_float4(0.f, 0.f, 0.f, 0.f);
            x[u] = in ? b4[c] : make_float4(0.f, 0.f, 0.f, 0.f);
            g[u] = in ? g4[c] : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < kCrossUnrollBwd; ++u) {
            s += dot4(a[u], v[u]);
            t += dot4(x[u], g[u]);
          }
        }
      } else {
        for (int k = lane; k < K; k += 32) {
          s += xl[r * K + k] * w[k];
          t += x0[r * K + k] * dout[r * K + k];
        }
      }
      s = warp_sum(s);
      t = warp_sum(t);
      if (VEC) {
        const float4* g4 = reinterpret_cast<const float4*>(dout + r * K);
        const float4* l4 = reinterpret_cast<const float4*>(xl + r * K);
        const float4* w4 = reinterpret_cast<const float4*>(w);
        float4* dl4 = reinterpret_cast<float4*>(dxl + r * K);
        float4* d04 = reinterpret_cast<float4*>(dx0 + r * K);
        for (int c0 = 0; c0 < KC; c0 += 32 * kCrossUnrollBwd) {
          float4 g[kCrossUnrollBwd], l[kCrossUnrollBwd], v[kCrossUnrollBwd];
#pragma unroll
          for (int u = 0; u < kCrossUnrollBwd; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < KC) {
              g[u] = g4[c];
              l[u] = l4[c];
              v[u] = w4[c];
            }
          }
#pragma unroll
          for (int u = 0; u < kCrossUnrollBwd; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < KC) {
              dl4[c] = make_float4(fmaf(v[u].x, t, g[u].x), fmaf(v[u].y, t, g[u].y),
                                   fmaf(v[u].z, t, g[u].z), fmaf(v[u].w, t, g[u].w));
              d04[c] = make_float4(g[u].x * s, g[u].y * s, g[u].z * s, g[u].w * s);
              const int k = 4 * c;
              atomicAdd(fdw + k, l[u].x * t);
              atomicAdd(fdw + k + 1, l[u].y * t);
              atomicAdd(fdw + k + 2, l[u].z * t);
              atomicAdd(fdw + k + 3, l[u].w * t);
              atomicAdd(fdb + k, g[u].x);
              atomicAdd(fdb + k + 1, g[u].y);
              atomicAdd(fdb + k + 2, g[u].z);
              atomicAdd(fdb + k + 3, g[u].w);
            }
          }
        }
      } else {
        for (int k = lane; k < K; k += 32) {
          const float g = dout[r * K + k], l = xl[r * K + k];
          dxl[r * K + k] = fmaf(w[k], t, g);
          dx0[r * K + k] = g * s;
          atomicAdd(fdw + k, l * t);
          atomicAdd(fdb + k, g);
        }
      }
    }
    if (++round == 2) {  // CTA-uniform: every warp runs the same rounds
      fold();
      round = 0;
    }
  }
  fold();
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    atomicAdd(dw + k, (float)sacc[k]);
    atomicAdd(db + k, (float)sacc[K + k]);
  }
}

static int cross_sms() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms < 1 ? 1 : sms;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

cudaError_t launch_cross_fwd(const float* x0, const float* xl, const float* w, const float* b,
                             int64_t B, int K, float* out, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  int64_t blocks = (B + 7) / 8;
  const int64_t cap = (int64_t)cross_sms() * 8;
  const int grid = (int)(blocks < cap ? blocks : cap);
  if (K % 4 == 0 && aligned16(x0) && aligned16(xl) && aligned16(w) && aligned16(b) && aligned16(out))
    k_cross_fwd<<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(x0),
                                     reinterpret_cast<const float4*>(xl),
                                     reinterpret_cast<const float4*>(w),
                                     reinterpret_cast<const float4*>(b), B, K / 4,
                                     reinterpret_cast<float4*>(out));
  else
    k_cross_fwd_scalar<<<grid, 256, 0, s>>>(x0, xl, w, b, B, K, out);
  return cudaGetLastError();
}

// dw and db are overwritten (zeroed here, then accumulated).
cudaError_t launch_cross_bwd(const float* x0, const float* xl, const float* w, const float* dout,
                             int64_t B, int K, float* dx0, float* dxl, float* dw, float* db,
                             cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(dw, 0, sizeof(float) * (size_t)K, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(db, 0, sizeof(float) * (size_t)K, s);
  if (e != cudaSuccess || B == 0) return e;
  const int smem = 2 * K * (int)(sizeof(double) + sizeof(float));
  // two CTAs of 16 warps per SM when both fit in shared memory (228 KB per SM), else one
  const int64_t cap = (int64_t)cross_sms() * (2 * (smem + 1024) <= 228 * 1024 ? 2 : 1);
  const int grid = (int)((B + 15) / 16 < cap ? (B + 15) / 16 : cap);
  const bool vec = K % 4 == 0 && aligned16(x0) && aligned16(xl) && aligned16(w) &&
                   aligned16(dout) && aligned16(dx0) && aligned16(dxl);
  if (vec) {
    e = cudaFuncSetAttribute(k_cross_bwd<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      k_cross_bwd<true><<<grid, 512, smem, s>>>(x0, xl, w, dout, B, K, dx0, dxl, dw, db);
  } else {
    e = cudaFuncSetAttribute(k_cross_bwd<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      k_cross_bwd<false><<<grid, 512, smem, s>>>(x0, xl, w, dout, B, K, dx0, dxl, dw, db);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace emb
