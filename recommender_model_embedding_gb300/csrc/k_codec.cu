// int8 row codec for the rows the layer exchanges (pooled rows and their gradients).
//
// Merlin Distributed Embeddings article, opening section: embedding rows are exchanged
// between GPUs in reduced precision; the format is not given.  Reading taken: symmetric
// per-row absmax scaling, scale = max|x| / 127, code = x / scale rounded to the nearest
// integer (ties to even) and clamped to [-127, 127]; a zero row has scale 0 and codes 0;
// decoding gives code * scale.  Every step is one IEEE fp32 operation (division,
// float-to-int conversion in round-to-nearest-even, multiplication), so the codes and the
// decoded values are fixed bit for bit.
//
// Both directions are bound by HBM bandwidth: per row of d floats, 4d bytes in and d + 4
// bytes out (encode), d + 4 in and 4d out (decode).  A group of G lanes holds one row in
// registers (16-byte loads, two or more chunks per lane, G a power of two of at most 32),
// the row maximum is a shuffle reduction within the group, and each lane stores its codes
// four at a time.  Widths that are not a multiple of 4 take a one-warp-per-row
// scalar path.
#include "emb_internal.cuh"

namespace emb {

constexpr int kCodecMaxChunks = 8;  // 16-byte chunks per lane: rows up to 32 * 8 * 4 floats

__device__ __forceinline__ int8_t encode1(float v, float s) {
  if (!(s > 0.f)) return 0;
  int c = __float2int_rn(__fdiv_rn(v, s));
  c = c > 127 ? 127 : (c < -127 ? -127 : c);
  return (int8_t)c;
}

// The next row's chunks are loaded before the current row is encoded (two rows per lane
// group in flight), so the loads of a warp overlap its reduction and divisions.
template <int NCH>
__global__ void __launch_bounds__(256) k_quantize_rows(const float* x, int64_t n, int d,
                                                       int8_t* q, float* scale, int G) {
  const int lane = threadIdx.x & 31, sub = lane % G, rpw = 32 / G;
  const int KC = d / 4;
  const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t step = nwarps * rpw;
  auto load = [&](int64_t row, float4 (&v)[NCH]) {
#pragma unroll
    for (int m = 0; m < NCH; ++m) {
      const int kc = sub + m * G;
      v[m] = (row < n && kc < KC) ? reinterpret_cast<const float4*>(x + row * d)[kc]
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  float4 v[NCH];
  load(gwarp * rpw + lane / G, v);
  for (int64_t r0 = gwarp * rpw; r0 < n; r0 += step) {
    const int64_t row = r0 + lane / G;
    float4 vn[NCH];
    load(row + step, vn);
    float amax = 0.f;
#pragma unroll
    for (int m = 0; m < NCH; ++m)
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[m].x), fabsf(v[m].y)), fmaxf(fabsf(v[m].z), fabsf(v[m].w))));
    for (int o = G / 2; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float s = __fdiv_rn(amax, 127.f);
    if (row < n) {
#pragma unroll
      for (int m = 0; m < NCH; ++m) {
        const int kc = sub + m * G;
        if (kc < KC) {
          char4 c;
          c.x = encode1(v[m].x, s);
          c.y = encode1(v[m].y, s);
          c.z = encode1(v[m].z, s);
          c.w = encode1(v[m].w, s);
          reinterpret_cast<char4*>(q + row * d)[kc] = c;
        }
      }
      if (sub == 0) scale[row] = s;
    }
#pragma unroll
    for (int m = 0; m < NCH; ++m) v[m] = vn[m];
  }
}

// any width: one warp per row
__global__ void __launch_bounds__(256) k_quantize_rows_scalar(const float* x, int64_t n, int d,
                                                              int8_t* q, float* scale) {
  const int lane = threadIdx.x & 31;
  const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t row = gwarp; row < n; row += nwarps) {
    const float* xr = x + row * d;
    float amax = 0.f;
    for (int c = lane; c < d; c += 32) amax = fmaxf(amax, fabsf(xr[c]));
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float s = __fdiv_rn(amax, 127.f);
    for (int c = lane; c < d; c += 32) q[row * d + c] = encode1(xr[c], s);
    if (lane == 0) scale[row] = s;
  }
}

template <int NCH>
__global__ void __launch_bounds__(256) k_dequantize_rows(const int8_t* q, const float* scale,
                                                         int64_t n, int d, float* x, int G) {
  const int lane = threadIdx.x & 31, sub = lane % G, rpw = 32 / G;
  const int KC = d / 4;
  const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t r0 = gwarp * rpw; r0 < n; r0 += nwarps * rpw) {
    const int64_t row = r0 + lane / G;
    if (row >= n) continue;
    const float s = scale[row];
    char4 c[NCH];
#pragma unroll
    for (int m = 0; m < NCH; ++m) {
      const int kc = sub + m * G;
      if (kc < KC) c[m] = reinterpret_cast<const char4*>(q + row * d)[kc];
    }
#pragma unroll
    for (int m = 0; m < NCH; ++m) {
      const int kc = sub + m * G;
      if (kc < KC)
        reinterpret_cast<float4*>(x + row * d)[kc] =
            make_float4(__fmul_rn((float)c[m].x, s), __fmul_rn((float)c[m].y, s),
                        __fmul_rn((float)c[m].z, s), __fmul_rn((float)c[m].w, s));
    }
  }
}

__global__ void __launch_bounds__(256) k_dequantize_rows_scalar(const int8_t* q, const float* scale,
                                                                int64_t n, int d, float* x) {
  const int lane = threadIdx.x & 31;
  const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t row = gwarp; row < n; row += nwarps) {
    const float s = scale[row];
    for (int c = lane; c < d; c += 32) x[row * d + c] = __fmul_rn((float)q[row * d + c], s);
  }
}

// lanes per row for the vectorised path: a power of two (<= 32) that gives each lane at
// least two 16-byte chunks where the row has four or more (more loads in flight per lane)
static int codec_lanes(int d) {
  const int KC = d / 4;
  int G = 1;
  while (2 * G < KC && G < 32) G <<= 1;
  return G;
}

static bool codec_vector_ok(int d, const void* a, const void* b) {
  return d % 4 == 0 && d / 4 <= 32 * kCodecMaxChunks &&
         (reinterpret_cast<uintptr_t>(a) & 15) == 0 && (reinterpret_cast<uintptr_t>(b) & 3) == 0;
}

static int codec_grid(int64_t rows_per_launch_unit) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms < 1) sms = 1;
  int64_t blocks = (rows_per_launch_unit + 7) / 8;  // 8 warps per block
  const int64_t cap = (int64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  return (int)(blocks < 1 ? 1 : blocks);
}

cudaError_t launch_quantize_rows(const float* x, int64_t n, int d, int8_t* q, float* scale,
                                 cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  if (!codec_vector_ok(d, x, q)) {
    k_quantize_rows_scalar<<<codec_grid(n), 256, 0, s>>>(x, n, d, q, scale);
    return cudaGetLastError();
  }
  const int G = codec_lanes(d), nch = (d / 4 + G - 1) / G;
  const int grid = codec_grid((n * G + 31) / 32);
  switch (nch) {
    case 1: k_quantize_rows<1><<<grid, 256, 0, s>>>(x, n, d, q, scale, G); break;
    case 2: k_quantize_rows<2><<<grid, 256, 0, s>>>(x, n, d, q, scale, G); break;
    case 3: case 4: k_quantize_rows<4><<<grid, 256, 0, s>>>(x, n, d, q, scale, G); break;
    default: k_quantize_rows<kCodecMaxChunks><<<grid, 256, 0, s>>>(x, n, d, q, scale, G); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_dequantize_rows(const int8_t* q, const float* scale, int64_t n, int d,
                                   float* x, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  if (!codec_vector_ok(d, x, q)) {
    k_dequantize_rows_scalar<<<codec_grid(n), 256, 0, s>>>(q, scale, n, d, x);
    return cudaGetLastError();
  }
  const int G = codec_lanes(d), nch = (d / 4 + G - 1) / G;
  const int grid = codec_grid((n * G + 31) / 32);
  switch (nch) {
    case 1: k_dequantize_rows<1><<<grid, 256, 0, s>>>(q, scale, n, d, x, G); break;
    case 2: k_dequantize_rows<2><<<grid, 256, 0, s>>>(q, scale, n, d, x, G); break;
    case 3: case 4: k_dequantize_rows<4><<<grid, 256, 0, s>>>(q, scale, n, d, x, G); break;
    default: k_dequantize_rows<kCodecMaxChunks><<<grid, 256, 0, s>>>(q, scale, n, d, x, G); break;
  }
  return cudaGetLastError();
}

}  // namespace emb
