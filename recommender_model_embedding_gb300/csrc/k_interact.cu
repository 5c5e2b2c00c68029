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
// Work split: one warp per sample.  X is staged in shared memory as float4 chunks of 4
// consecutive k, chunk-major: Xs[kc][pos(i)], pos(i) = i + i/4, row stride FS odd.  With
// that padding the chunks one instruction reads (x_{4I+r}[kc], distinct I) fall in
// distinct bank groups, and the staging writes (lane = kc, fixed i) do too.
//  - forward: lane -> one 4x4 block (I >= J) of the lower triangle of X X^T, accumulated
//    over all kc with fp32 FMAs (8 shared loads per 64 FMAs);
//  - backward: lane -> chunk kc of dX for 8 rows at a time: dX[i][kc] += G[i][j] x_j[kc].
// Fused variants gather the bag rows straight from the table into Xs (fp32 or bf16
// storage, fp32 sums) and, in the backward, add each dX row (scaled by 1/L for mean
// pooling) into the per-unique-row gradient buffer with vector reductions.
#include <math.h>

#include "emb_internal.cuh"

namespace emb {

struct ILayout {
  int F, Fpad, KC, FS;
  int xs_f4;   // float4 slots of Xs per warp
  int gs_f;    // floats of Gs per warp (backward)
};

static ILayout make_layout(int T, int D, bool bwd) {
  ILayout L;
  L.F = T + 1;
  L.Fpad = (L.F + 3) & ~3;
  L.KC = D / 4;
  const int last = (L.Fpad - 1) + ((L.Fpad - 1) >> 2);
  L.FS = (last + 1) | 1;
  L.xs_f4 = L.KC * L.FS;
  L.gs_f = bwd ? L.F * 32 : 0;
  return L;
}

__device__ __forceinline__ int xpos(int i) { return i + (i >> 2); }

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

// ---- staging X of one sample into shared memory ----

// MODE 0: pooled vectors from a [B][T][D] buffer; MODE 1: gather + pool from the table.
template <int MODE, bool BF16>
__device__ __forceinline__ void stage_x(const Params& p, const ILayout& L, float4* Xs,
                                        int64_t s, const float* dense, const float* pooled,
                                        int one_hot, int lane) {
  const int D = p.D, T = p.T, KC = L.KC, FS = L.FS;
  // x_0 = dense, rows F..Fpad-1 = 0
  for (int kc = lane; kc < KC; kc += 32) {
    Xs[kc * FS + xpos(0)] = __ldg(reinterpret_cast<const float4*>(dense + s * D) + kc);
    for (int i = L.F; i < L.Fpad; ++i) Xs[kc * FS + xpos(i)] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (MODE == 0) {
    for (int t = 0; t < T; ++t) {
      const float4* src = reinterpret_cast<const float4*>(pooled + (s * T + t) * D);
      for (int kc = lane; kc < KC; kc += 32) Xs[kc * FS + xpos(t + 1)] = __ldg(src + kc);
    }
    return;
  }
  constexpr int EPC = BF16 ? 8 : 4;
  const int nchunk = D / EPC;  // 16-byte chunks per row
  if (one_hot) {
    // eight bags at a time: row numbers first, then the row loads back to back
    for (int t0 = 0; t0 < T; t0 += 8) {
      uint32_t r[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) r[u] = (t0 + u < T) ? p.row_of[s * T + t0 + u] : kNoRow;
      for (int q = lane; q < nchunk; q += 32) {
        float4 v[8][BF16 ? 2 : 1];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (r[u] == kNoRow) {
            v[u][0] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (BF16) v[u][BF16 ? 1 : 0] = make_float4(0.f, 0.f, 0.f, 0.f);
          } else if (BF16) {
            ld_row8_bf16(reinterpret_cast<const __nv_bfloat16*>(p.table) + (int64_t)r[u] * D, q,
                         v[u][0], v[u][BF16 ? 1 : 0]);
          } else {
            v[u][0] = ld_row4_f32(reinterpret_cast<const float*>(p.table) + (int64_t)r[u] * D, q);
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (t0 + u >= T) continue;
          if (BF16) {
            Xs[(2 * q) * FS + xpos(t0 + u + 1)] = v[u][0];
            Xs[(2 * q + 1) * FS + xpos(t0 + u + 1)] = v[u][BF16 ? 1 : 0];
          } else {
            Xs[q * FS + xpos(t0 + u + 1)] = v[u][0];
          }
        }
      }
    }
    return;
  }
  // multi-hot bags
  for (int t = 0; t < T; ++t) {
    const int64_t bag = s * T + t;
    int64_t beg = p.offs[bag], end = p.offs[bag + 1];
    if (beg < 0 || end < beg || end > p.nnz) beg = end = 0;
    const float Lb = (float)(end - beg);
    for (int q = lane; q < nchunk; q += 32) {
      float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
      for (int64_t i = beg; i < end; ++i) {
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
        Xs[(2 * q) * FS + xpos(t + 1)] = a0;
        Xs[(2 * q + 1) * FS + xpos(t + 1)] = a1;
      } else {
        Xs[q * FS + xpos(t + 1)] = a0;
      }
    }
  }
}

// ---- forward ----

template <int MODE, bool BF16>
__global__ void __launch_bounds__(128) k_interact_fwd(Params p, ILayout L, const float* dense,
                                                      const float* pooled, int64_t B,
                                                      float* out, int one_hot) {
  extern __shared__ float4 smem[];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  float4* Xs = smem + wid * (L.xs_f4 + L.gs_f / 4);
  const int D = p.D, T = p.T, F = L.F, FS = L.FS;
  const int64_t W = D + (int64_t)F * (F - 1) / 2;
  const int R = L.Fpad / 4;
  const int nblk = R * (R + 1) / 2;
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t s = gw; s < B; s += nw) {
    __syncwarp();
    stage_x<MODE, BF16>(p, L, Xs, s, dense, pooled, one_hot, lane);
    if (MODE == 1) {
      // unique index of each lookup of this sample, for the fused backward
      int64_t q0 = one_hot ? s * T : p.offs[s * T];
      int64_t q1 = one_hot ? (s + 1) * T : p.offs[(s + 1) * T];
      q0 = q0 < 0 ? 0 : q0;  // malformed offsets are flagged; stay inside [0, nnz)
      q1 = q1 > p.nnz ? p.nnz : q1;
      for (int64_t q = q0 + lane; q < q1; q += 32) {
        const uint32_t sl = p.slot_of[q];
        p.inv[q] = (p.row_of[q] != kNoRow && sl != kEmpty32) ? p.set_vals[sl] : kNoRow;
      }
    }
    __syncwarp();
    float* orow = out + s * W;
    for (int k = lane; k < D; k += 32) orow[k] = __ldg(dense + s * D + k);
    for (int blk = lane; blk < nblk; blk += 32) {
      int I = (int)((sqrtf(8.f * blk + 1.f) - 1.f) * 0.5f);
      while (I * (I + 1) / 2 > blk) --I;
      while ((I + 1) * (I + 2) / 2 <= blk) ++I;
      const int J = blk - I * (I + 1) / 2;
      float acc[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e] = 0.f;
      const int pi = 5 * I, pj = 5 * J;  // xpos(4I + r) = 5I + r
      for (int kc = 0; kc < L.KC; ++kc) {
        const float4* row = Xs + kc * FS;
        float4 a[4], b[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) a[r] = row[pi + r];
#pragma unroll
        for (int c = 0; c < 4; ++c) b[c] = row[pj + c];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[r * 4 + c] += dot4(a[r], b[c]);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int i = 4 * I + r;
        if (i >= F) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int j = 4 * J + c;
          if (j < i) orow[D + i * (i - 1) / 2 + j] = acc[r * 4 + c];
        }
      }
    }
  }
}

// ---- backward ----

template <int MODE, bool BF16>
__global__ void __launch_bounds__(128) k_interact_bwd(Params p, ILayout L, const float* dout,
                                                      const float* dense, const float* pooled,
                                                      int64_t B, float* ddense, float* dpooled,
                                                      int one_hot) {
  extern __shared__ float4 smem[];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  float4* Xs = smem + wid * (L.xs_f4 + L.gs_f / 4);
  float* Gs = reinterpret_cast<float*>(Xs + L.xs_f4);  // [F][32]
  const int D = p.D, T = p.T, F = L.F, FS = L.FS;
  const int P = F * (F - 1) / 2;
  const int64_t W = D + P;
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int ngroups = (L.Fpad + 7) / 8;
  for (int64_t s = gw; s < B; s += nw) {
    __syncwarp();
    stage_x<MODE, BF16>(p, L, Xs, s, dense, pooled, one_hot, lane);
    const float* drow = dout + s * W;
    for (int e = lane; e < F * 32; e += 32) Gs[e] = 0.f;
    __syncwarp();
    for (int q = lane; q < P; q += 32) {
      int i = (int)((1.f + sqrtf(8.f * q + 1.f)) * 0.5f);
      while (i * (i - 1) / 2 > q) --i;
      while ((i + 1) * i / 2 <= q) ++i;
      const int j = q - i * (i - 1) / 2;
      const float gv = __ldg(drow + D + q);
      Gs[i * 32 + j] = gv;
      Gs[j * 32 + i] = gv;
    }
    __syncwarp();
    for (int kc = lane; kc < L.KC; kc += 32) {
      for (int g = 0; g < ngroups; ++g) {
        float4 acc[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < F; ++j) {
          const float4 x = Xs[kc * FS + xpos(j)];
          const float4 g0 = reinterpret_cast<const float4*>(Gs + j * 32 + 8 * g)[0];
          const float4 g1 = reinterpret_cast<const float4*>(Gs + j * 32 + 8 * g)[1];
          const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            acc[r].x = fmaf(gg[r], x.x, acc[r].x);
            acc[r].y = fmaf(gg[r], x.y, acc[r].y);
            acc[r].z = fmaf(gg[r], x.z, acc[r].z);
            acc[r].w = fmaf(gg[r], x.w, acc[r].w);
          }
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int i = 8 * g + r;
          if (i >= F) continue;
          float4 v = acc[r];
          if (i == 0) {
            const float* dsrc = drow + 4 * kc;  // dout rows are not 16-byte aligned
            v.x += __ldg(dsrc + 0);
            v.y += __ldg(dsrc + 1);
            v.z += __ldg(dsrc + 2);
            v.w += __ldg(dsrc + 3);
            reinterpret_cast<float4*>(ddense + s * D)[kc] = v;
          } else if (MODE == 0) {
            reinterpret_cast<float4*>(dpooled + (s * T + (i - 1)) * D)[kc] = v;
          } else {
            const int64_t bag = s * T + (i - 1);
            int64_t q0 = bag, q1 = bag + 1;
            if (!one_hot) {
              q0 = p.offs[bag];
              q1 = p.offs[bag + 1];
              if (q0 < 0 || q1 < q0 || q1 > p.nnz) q0 = q1 = 0;
            }
            if (p.mean && q1 > q0) v = f4_div(v, (float)(q1 - q0));
            for (int64_t q = q0; q < q1; ++q) {
              const uint32_t u = p.inv[q];
              if (u != kNoRow) red_add_f4(p.g + (int64_t)u * D + 4 * kc, v);
            }
          }
        }
      }
    }
  }
}

// ---- launchers ----

template <typename K>
static int blocks_for(Ctx* c, K kern, size_t smem, int64_t B) {
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 128, smem);
  if (per_sm < 1) per_sm = 1;
  int64_t want = (B + 3) / 4;
  int64_t cap = (int64_t)per_sm * c->num_sms;
  if (want > cap) want = cap;
  return (int)(want < 1 ? 1 : want);
}

cudaError_t launch_interact_fwd(Ctx* c, const float* dense, const float* pooled, int64_t B,
                                float* out, cudaStream_t s) {
  const ILayout L = make_layout(c->p.T, c->p.D, false);
  const size_t smem = (size_t)4 * (L.xs_f4 * 16 + L.gs_f * 4);
  auto kern = k_interact_fwd<0, false>;
  const int grid = blocks_for(c, kern, smem, B);
  LaunchScope ls(c, K_INTERACT_FWD, s);
  kern<<<grid, 128, smem, s>>>(c->p, L, dense, pooled, B, out, 1);
  return cudaGetLastError();
}

cudaError_t launch_interact_bwd(Ctx* c, const float* dout, const float* dense,
                                const float* pooled, int64_t B, float* ddense, float* dpooled,
                                cudaStream_t s) {
  const ILayout L = make_layout(c->p.T, c->p.D, true);
  const size_t smem = (size_t)4 * (L.xs_f4 * 16 + L.gs_f * 4);
  auto kern = k_interact_bwd<0, false>;
  const int grid = blocks_for(c, kern, smem, B);
  LaunchScope ls(c, K_INTERACT_BWD, s);
  kern<<<grid, 128, smem, s>>>(c->p, L, dout, dense, pooled, B, ddense, dpooled, 1);
  return cudaGetLastError();
}

cudaError_t launch_fused_fwd(Ctx* c, const float* dense, int64_t B, float* out, cudaStream_t s) {
  const ILayout L = make_layout(c->p.T, c->p.D, false);
  const size_t smem = (size_t)4 * (L.xs_f4 * 16 + L.gs_f * 4);
  auto kern = c->p.bf16 ? k_interact_fwd<1, true> : k_interact_fwd<1, false>;
  const int grid = blocks_for(c, kern, smem, B);
  LaunchScope ls(c, K_FUSED_FWD, s);
  kern<<<grid, 128, smem, s>>>(c->p, L, dense, nullptr, B, out, c->multi_hot ? 0 : 1);
  return cudaGetLastError();
}

cudaError_t launch_fused_bwd(Ctx* c, const float* dout, const float* dense, int64_t B,
                             float* ddense, cudaStream_t s) {
  const ILayout L = make_layout(c->p.T, c->p.D, true);
  const size_t smem = (size_t)4 * (L.xs_f4 * 16 + L.gs_f * 4);
  auto kern = c->p.bf16 ? k_interact_bwd<1, true> : k_interact_bwd<1, false>;
  const int grid = blocks_for(c, kern, smem, B);
  LaunchScope ls(c, K_FUSED_BWD, s);
  kern<<<grid, 128, smem, s>>>(c->p, L, dout, dense, nullptr, B, ddense, nullptr,
                               c->multi_hot ? 0 : 1);
  return cudaGetLastError();
}

}  // namespace emb
