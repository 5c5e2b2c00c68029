// Pairwise dot feature interaction, forward and backward: the standalone operator (pooled
// vectors in memory) and the fused variants that gather the rows themselves for multi-hot
// bags or bf16 storage.  The fp32 one-hot fused path has its own warp-specialised kernels
// (k_fused_ws.cu); this file dispatches to them.
//
// OneEmbedding article, "operator optimisation": DLRM's feature interaction as one fused
// operator (FusedDotFeatureInteraction); "usability": interaction(dense_fields, embedding).
//
// Per sample b: X = [x_0 = dense_b; x_1..x_T = pooled_b,0..T-1]  (F = T+1 vectors of D).
//   forward : out_b = [dense_b || x_i . x_j for i = 1..F-1, j = 0..i-1]
//   backward: G_ij = G_ji = dout_b[D + pair(i,j)], G_ii = 0; dX = G X;
//             d_dense = dX_0 + dout_b[0:D]; d_pooled[t] = dX_{t+1}.
//
// One CTA per sample at a time, a few warps sharing the sample's X in shared memory
// (layout in interact_common.cuh):
//  - forward: lane -> one 4x4 block (I >= J) of the lower triangle of X X^T; the warps of
//    the CTA split the k range and their partial blocks are summed through shared memory;
//  - backward: warp g -> dX rows 9g..9g+8, lane -> chunk kc.
// The fused multi-hot backward adds each dX row (scaled by 1/L for mean pooling) into the
// per-unique-row gradient buffer with vector reductions.
#include "interact_common.cuh"

namespace emb {

constexpr int kFwdWarps = 4;  // warps per CTA in the forward (split of the k range)

enum Src : int { SRC_POOLED = 0, SRC_GATHER = 1 };

struct ILayout {
  XShape x;
  int nblk;       // forward 4x4 blocks
  int nwarps;     // warps per CTA
  int p_f;        // floats of the forward partial sums (+ block coordinate table)
  int g_f;        // floats of the backward coefficient table
  int d_f;        // floats of the backward dense-gradient staging
  int cta_bytes;  // shared memory per CTA
};

static ILayout make_layout(int T, int D, bool bwd) {
  ILayout L;
  L.x = make_xshape(T, D);
  const int R = L.x.Fpad / 4;
  L.nblk = R * (R + 1) / 2;
  L.nwarps = bwd ? (L.x.F + kRowsPerGroup - 1) / kRowsPerGroup : kFwdWarps;
  L.p_f = bwd ? 0 : L.nwarps * 16 * L.nblk + kMaxBlocks;
  L.g_f = bwd ? L.x.F * kGStride : 0;
  L.d_f = bwd ? D : 0;
  const int bytes = L.x.x_f4 * 16 + L.p_f * 4 + L.g_f * 4 + L.d_f * 4 + (bwd ? 4 * 32 : 0);
  L.cta_bytes = (bytes + 15) & ~15;
  return L;
}

// Synchronous staging: lane = chunk; warp w of NW stages the rows i with i % NW == w.
template <int SRC, bool BF16>
__device__ __forceinline__ void stage_x(const Params& p, const XShape& L, float4* X, int64_t s,
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
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
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
      float4 a0 = z, a1 = z;
      int64_t i = beg;
      for (; i + 2 <= end; i += 2) {  // two rows in flight per lane
        const uint32_t r0 = p.row_of[i], r1 = p.row_of[i + 1];
        if (BF16) {
          float4 l0 = z, h0 = z, l1 = z, h1 = z;
          if (r0 != kNoRow)
            ld_row8_bf16(reinterpret_cast<const __nv_bfloat16*>(p.table) + (int64_t)r0 * D, q, l0, h0);
          if (r1 != kNoRow)
            ld_row8_bf16(reinterpret_cast<const __nv_bfloat16*>(p.table) + (int64_t)r1 * D, q, l1, h1);
          a0 = f4_add(a0, f4_add(l0, l1));
          a1 = f4_add(a1, f4_add(h0, h1));
        } else {
          const float* tb = reinterpret_cast<const float*>(p.table);
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

// Unique index of each lookup of sample s (fused forward), one warp.
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

__device__ __forceinline__ void zero_pad_rows(const XShape& L, float4* X) {
  const int n = (L.Fpad - L.F) * L.KC;
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int i = L.F + e / L.KC, kc = e % L.KC;
    X[xslot(i) * L.RS + kc] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// ---- forward ----

template <int SRC, bool BF16>
__global__ void __launch_bounds__(kFwdWarps * 32) k_interact_fwd(Params p, ILayout L,
                                                                 const float* dense,
                                                                 const float* pooled, int64_t B,
                                                                 float* out, int one_hot, int record_inv) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, NW = blockDim.x >> 5;
  float4* X = reinterpret_cast<float4*>(smem);
  float* Ps = reinterpret_cast<float*>(X + L.x.x_f4);       // [NW][16][nblk]
  int* Bij = reinterpret_cast<int*>(Ps + NW * 16 * L.nblk);  // (I << 8) | J per block
  const int D = p.D, F = L.x.F, nblk = L.nblk;
  const int64_t W = D + (int64_t)F * (F - 1) / 2;
  const int kc0 = (L.x.KC * w) / NW, kc1 = (L.x.KC * (w + 1)) / NW;
  zero_pad_rows(L.x, X);
  if (threadIdx.x == 0) {
    int blk = 0;
    for (int I = 0; I < L.x.Fpad / 4; ++I)
      for (int J = 0; J <= I; ++J) Bij[blk++] = (I << 8) | J;
  }
  __syncthreads();
  for (int64_t s = blockIdx.x; s < B; s += gridDim.x) {
    stage_x<SRC, BF16>(p, L.x, X, s, dense, pooled, one_hot, lane, w, NW);
    // the unique index of each lookup, unless the inverse kernel has produced it already
    if (SRC == SRC_GATHER && w == 0 && record_inv) record_inverse(p, s, one_hot, lane);
    __syncthreads();
    for (int blk = lane; blk < nblk; blk += 32) {
      float acc[16];
      const int ij = Bij[blk];
      fwd_block(L.x, X, ij >> 8, ij & 255, kc0, kc1, acc);
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

// ---- backward ----

template <int SRC, bool BF16>
__global__ void __launch_bounds__(128) k_interact_bwd(Params p, ILayout L, const float* dout,
                                                      const float* dense, const float* pooled,
                                                      int64_t B, float* ddense, float* dpooled,
                                                      int one_hot) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, NW = blockDim.x >> 5;
  float4* X = reinterpret_cast<float4*>(smem);
  float* Gs = reinterpret_cast<float*>(X + L.x.x_f4);
  float* Ds = Gs + L.g_f;
  const int D = p.D, T = p.T, F = L.x.F;
  const int W = D + F * (F - 1) / 2;
  const int g = w;  // dX rows 9g..9g+8
  zero_pad_rows(L.x, X);
  for (int e = threadIdx.x; e < L.g_f; e += blockDim.x) Gs[e] = 0.f;  // diagonal/padding stay 0
  int ptab[kMaxDoutPerLane];
#pragma unroll
  for (int m = 0; m < kMaxDoutPerLane; ++m) {
    const int e = lane + 32 * m;
    ptab[m] = (m % NW == w && e >= D && e < W) ? pair_code(e - D) : 0;
  }
  __syncthreads();
  float dv[kMaxDoutPerLane];
  uint32_t iv = kNoRow;
  for (int64_t s = blockIdx.x; s < B; s += gridDim.x) {
    load_dout(p, dout, s, W, T, false, lane, w, NW, dv, iv);
    stage_x<SRC, BF16>(p, L.x, X, s, dense, pooled, one_hot, lane, w, NW);
    build_g(Gs, Ds, dv, ptab, D, W, lane, w, NW);
    __syncthreads();
    for (int kc = lane; kc < L.x.KC; kc += 32) {
      float4 acc[kRowsPerGroup];
      bwd_group(L.x, X, Gs, g, kc, acc);
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
    __syncthreads();
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

template <int SRC, bool BF16>
static cudaError_t run_fwd(Ctx* c, const float* dense, const float* pooled, int64_t B,
                           float* out, int one_hot, int kid, cudaStream_t s) {
  const ILayout L = make_layout(c->p.T, c->p.D, false);
  auto kern = k_interact_fwd<SRC, BF16>;
  const int threads = L.nwarps * 32;
  const int grid = persistent_grid(c, kern, threads, L.cta_bytes, B);
  LaunchScope ls(c, kid, s);
  // the gather variant records the inverse only where no inverse kernel runs
  const int record_inv = (SRC == SRC_GATHER && fused_fwd_records_inverse(c)) ? 1 : 0;
  kern<<<grid, threads, L.cta_bytes, s>>>(c->p, L, dense, pooled, B, out, one_hot, record_inv);
  return cudaGetLastError();
}

template <int SRC, bool BF16>
static cudaError_t run_bwd(Ctx* c, const float* dout, const float* dense, const float* pooled,
                           int64_t B, float* ddense, float* dpooled, int one_hot, int kid,
                           cudaStream_t s) {
  const ILayout L = make_layout(c->p.T, c->p.D, true);
  auto kern = k_interact_bwd<SRC, BF16>;
  const int threads = L.nwarps * 32;
  const int grid = persistent_grid(c, kern, threads, L.cta_bytes, B);
  LaunchScope ls(c, kid, s);
  kern<<<grid, threads, L.cta_bytes, s>>>(c->p, L, dout, dense, pooled, B, ddense, dpooled,
                                          one_hot);
  return cudaGetLastError();
}

cudaError_t launch_interact_fwd(Ctx* c, const float* dense, const float* pooled, int64_t B,
                                float* out, cudaStream_t s) {
  return run_fwd<SRC_POOLED, false>(c, dense, pooled, B, out, 1, K_INTERACT_FWD, s);
}

cudaError_t launch_interact_bwd(Ctx* c, const float* dout, const float* dense,
                                const float* pooled, int64_t B, float* ddense, float* dpooled,
                                cudaStream_t s) {
  return run_bwd<SRC_POOLED, false>(c, dout, dense, pooled, B, ddense, dpooled, 1,
                                    K_INTERACT_BWD, s);
}

// The generic fused forward records the unique index of each lookup itself unless the
// inverse kernel runs: for the register-resident shapes and wherever the tensor-core
// backward runs (its steps may tag once rows).
// The generic forward records each lookup's unique index for the generic backward; the
// tensor-core and register-resident forwards leave that to the inverse kernel.
bool fused_fwd_records_inverse(const Ctx* c) {
  return !use_tc_fwd(c) && !reg_supported(c) && !use_tc_bwd(c);
}

cudaError_t launch_fused_fwd(Ctx* c, const float* dense, int64_t B, float* out, cudaStream_t s) {
  if (use_tc_fwd(c)) return launch_fused_fwd_tc(c, dense, B, out, s);
  if (reg_supported(c)) return launch_fused_fwd_reg(c, dense, B, out, s);
  const int one_hot = c->multi_hot ? 0 : 1;
  if (c->p.bf16) return run_fwd<SRC_GATHER, true>(c, dense, nullptr, B, out, one_hot, K_FUSED_FWD, s);
  return run_fwd<SRC_GATHER, false>(c, dense, nullptr, B, out, one_hot, K_FUSED_FWD, s);
}

cudaError_t launch_fused_bwd(Ctx* c, const float* dout, const float* dense, int64_t B,
                             float* ddense, cudaStream_t s) {
  if (use_tc_bwd(c)) return launch_fused_bwd_tc(c, dout, dense, B, ddense, s);
  if (reg_supported(c)) return launch_fused_bwd_reg(c, dout, dense, B, ddense, s);
  const int one_hot = c->multi_hot ? 0 : 1;
  if (c->p.bf16)
    return run_bwd<SRC_GATHER, true>(c, dout, dense, nullptr, B, ddense, nullptr, one_hot,
                                     K_FUSED_BWD, s);
  return run_bwd<SRC_GATHER, false>(c, dout, dense, nullptr, B, ddense, nullptr, one_hot,
                                    K_FUSED_BWD, s);
}

}  // namespace emb
