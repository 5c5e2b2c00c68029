// Fused interaction backward on the 5th-generation tensor cores (tcgen05 MMA, operands and
// accumulator in tensor memory) for fp32 one-hot tables with D = 128 and F = T+1 <= 32
// interaction vectors.
//
// Per sample the backward is a small dense contraction, dX_i[k] = sum_j G[i][j] x_j[k], with
// G the symmetric, zero-diagonal matrix of the upstream pair gradients.  Written as
// dX^T (128 x 32) = X^T (128 x 32) * G (32 x 32) it puts the embedding dimension on the
// M = 128 rows of one tcgen05 tile, so no MMA work is spent on cross-sample products.  fp32
// accuracy comes from three TF32 products, X_hi G_hi + X_hi G_lo + X_lo G_hi: the tensor core
// reads an fp32 operand as TF32 by dropping its 13 low mantissa bits, so hi = the value with
// those bits cleared (one AND) and lo = value - hi (exact in fp32, below 2^-10 of the value;
// the tensor core drops lo's own low bits in turn).  Each dropped part -- X_lo G_lo and the
// low bits of the two lo operands -- is below 2^-20 of |x||g|.
//
// One CTA (one warpgroup, 128 threads; thread k owns element k of the embedding dimension,
// which is TMEM lane k) works on one sample at a time:
//  1. thread k holds x_j[k] for the sample's F vectors (dense row, then one table row per
//     feature; 128-byte coalesced loads per warp, issued one sample ahead) and writes their
//     hi and lo TF32 parts into its own TMEM lane with tcgen05.st: the A operand never
//     passes through shared memory;
//  2. the pair gradients dout[D + q] are written as hi/lo into both (i,j) and (j,i) of the
//     B operand tiles in shared memory; diagonal and padding stay zero from the start;
//  3. after the TMEM stores complete, a CTA barrier, and one thread issues 12 MMAs (3 products
//     x 4 steps of K = 8) with A read from TMEM, into 32 TMEM accumulator columns, and commits
//     them to an mbarrier;
//  4. every warp waits on the mbarrier (bounded), reads its 32 TMEM lanes with tcgen05.ld
//     (thread k receives dX_i[k] for all i), writes d_dense = dX_0 + dout[0:D], and adds each
//     looked-up row's dX_i into the per-unique-row gradient buffer (coalesced 128-byte
//     reductions per warp).
//
// Steps that track once rows (rows that no other lookup of the batch shares; their inverse
// index carries kInvOnce) update such a row here instead of adding dX_i to the gradient
// buffer: dX_i is the row's whole gradient, the row's current values x_i[k] are still in
// TMEM (hi + lo is exact), and its Adagrad accumulator row has been copied into shared memory
// by a bulk copy issued one sample ahead.  The row then takes one accumulator read and two
// row writes instead of a reduction, a gradient read and a gradient clear in the update.
//
// TMEM columns of a CTA: [0, 32) accumulator dX^T, [32, 64) X_hi^T, [64, 96) X_lo^T (column
// j of lane k = x_j[k]).  B operand layout (K-major with the 128-byte swizzle): row n (the
// 32 tf32 values of K) is 128 bytes at n*128, its 16-byte chunk c stored at chunk position
// c ^ (n % 8); 8-row groups 1024 bytes apart (stride byte offset), the tile 1 KB-aligned.
// The swizzle spreads both the (i, j) and the (j, i) stores of a warp's pair gradients over
// the banks (the unswizzled layout put 4 to 8 of them in one bank).
#include <algorithm>

#include "interact_common.cuh"
#include "tc_common.cuh"

namespace emb {

constexpr int kTcThreads = 128;
constexpr int kTcN = 32;      // output columns i (F padded to 32)
constexpr int kTcK = 32;      // contraction index j (F padded to 32)
constexpr int kBRow = 128;    // B: bytes of one row (32 tf32 of K)
constexpr int kBSBO = 1024;   // B: bytes between 8-row groups in N
constexpr int kTileB = kTcN * kBRow;  // 4 KB: 32 x 32 tf32
constexpr int kTcDout = (128 + kMaxF * (kMaxF - 1) / 2 + kTcThreads - 1) / kTcThreads;
constexpr int kTcCols = 128;  // TMEM columns per CTA (96 used)
constexpr int kColD = 0, kColAhi = 32, kColAlo = 64;

// instruction descriptor: M = 128, N = 32, tf32 inputs, fp32 accumulator, B K-major
constexpr uint32_t kTcIdesc = idesc_tf32(128, kTcN);

constexpr int kOffBhi = 0;
constexpr int kOffBlo = kOffBhi + kTileB;
constexpr int kOffUs = kOffBlo + kTileB;  // [2][32] unique index of column i (double-buffered)
constexpr int kOffBar = kOffUs + 2 * 32 * 4;
constexpr int kOffTmem = kOffBar + 8;
constexpr int kTcLayout = kOffTmem + 8;
constexpr int kAlignSlack = 1024;  // the B tiles start on a 1 KB boundary (swizzle atoms)
constexpr int kTcSmem = kTcLayout + kAlignSlack;
// once-row variant: [2][32] table row of column i, two bulk-copy barriers, [2][32][128]
// accumulator rows (double-buffered by sample)
constexpr int kOffRs = kTcLayout;
constexpr int kOffAbar = kOffRs + 2 * 32 * 4;
constexpr int kOffOm = kOffAbar + 16;  // [2] once-column mask of the sample (bit i: column i)
constexpr int kOffAs = (kOffOm + 8 + 127) / 128 * 128;
constexpr int kTcSmemOnce = kOffAs + 2 * 32 * 128 * 4 + kAlignSlack;

// byte offset of B element (n, j)
__device__ __forceinline__ int b_off(int n, int j) {
  return n * kBRow + ((((j >> 2) ^ n) & 7) << 4) + (j & 3) * 4;
}

// the TF32 part of x the tensor core reads: x with its 13 low mantissa bits cleared
__device__ __forceinline__ float tf32_hi(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// one float from global memory when pred holds, zero otherwise (no branch)
__device__ __forceinline__ float ldg_if(const float* ptr, bool pred) {
  float v;
  asm("{\n .reg .pred p;\n setp.ne.b32 p, %2, 0;\n mov.f32 %0, 0f00000000;\n"
      " @p ld.global.nc.f32 %0, [%1];\n}"
      : "=f"(v)
      : "l"(ptr), "r"((uint32_t)pred));
  return v;
}

// *addr += v when u is a unique index to reduce into (bit 31 clear: neither kNoRow nor a
// lookup tagged kInvOnce); predicated, no branch
__device__ __forceinline__ void red_add_row(float* base, uint32_t u, float v) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .u64 a;\n setp.lt.u32 p, %1, 0x80000000;\n"
      " mad.wide.u32 a, %1, 512, %0;\n @p red.global.add.f32 [a], %2;\n}" ::"l"(base),
      "r"(u), "f"(v)
      : "memory");
}

// base[row * 128] = v when pred holds (a row of 128 fp32 values); predicated, no branch
__device__ __forceinline__ void st_row_if(float* base, uint32_t row, float v, uint32_t pred) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .u64 a;\n setp.ne.u32 p, %2, 0;\n"
      " mad.wide.u32 a, %1, 512, %0;\n @p st.global.f32 [a], %3;\n}" ::"l"(base),
      "r"(row), "r"(pred), "f"(v)
      : "memory");
}

// FT: the number of interaction vectors when known at compile time (27, the 26-table shape),
// else 0 (taken from p.T): the columns past F then cost no gathers, splits or reductions.
template <bool ONCE, int FT>
__global__ void __launch_bounds__(kTcThreads, 4) k_fused_bwd_tc(Params p, const float* dout,
                                                             const float* dense, int64_t B,
                                                             float* ddense) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // swizzle atoms: 1 KB
  const int k = threadIdx.x;
  const int lane = k & 31, warp = k >> 5;
  const int T = FT ? FT - 1 : p.T, F = FT ? FT : T + 1, D = 128;
  const int W = D + F * (F - 1) / 2;
  const float* table = reinterpret_cast<const float*>(p.table);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* Us = reinterpret_cast<uint32_t*>(smem + kOffUs);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);
  uint32_t* Rs = reinterpret_cast<uint32_t*>(smem + kOffRs);
  uint64_t* abar = reinterpret_cast<uint64_t*>(smem + kOffAbar);
  float* As = reinterpret_cast<float*>(smem + kOffAs);
  uint32_t* Om = reinterpret_cast<uint32_t*>(smem + kOffOm);
  const uint32_t sbase = smem_u32(smem);

  // B tiles start at zero; padding (i or j >= F) and the diagonal are never written
  for (int e = k; e < kOffUs / 16; e += kTcThreads)
    reinterpret_cast<float4*>(smem)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (k < 64) {  // column 0 (dense vector) and columns past F keep no row
    Us[k] = kNoRow;
    if (ONCE) Rs[k] = 0u;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "n"(kTcCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (k == 0) {
    mbar_init(bar, 1);
    if (ONCE) {
      mbar_init(abar, 1);
      mbar_init(abar + 1, 1);
    }
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tlane = tmem + ((uint32_t)(warp * 32) << 16);  // this warp's 32 lanes

  // operand offsets of (i,j) and (j,i) for the pair gradients this thread stages
  // (dout element k + 128 m, pair index q = element - D); -1 outside the pairs
  int off_ij[kTcDout], off_ji[kTcDout];
#pragma unroll
  for (int m = 0; m < kTcDout; ++m) {
    const int e = k + kTcThreads * m;
    off_ij[m] = off_ji[m] = -1;
    if (e >= D && e < W) {
      const int cd = pair_code(e - D), i = cd >> 8, j = cd & 255;
      off_ij[m] = b_off(i, j);
      off_ji[m] = b_off(j, i);
    }
  }

  const int64_t nb = gridDim.x;
  int64_t s = blockIdx.x;
  float x[kTcK];  // x_j[k] of the sample being staged
  float dn[kTcDout];
  // table rows and unique indices of the sample gathered next (lane t: feature t), loaded
  // one sample ahead; un / rcur hold those of the last gathered sample
  uint32_t rnext = (s < B && lane < T) ? p.row_of[s * T + lane] : kNoRow;
  uint32_t inext = (s < B && lane < T) ? p.inv[s * T + lane] : kNoRow;
  uint32_t un = kNoRow, rcur = kNoRow;
  auto gather = [&](int64_t ss) {
    rcur = rnext;
    un = inext;
    x[0] = __ldg(dense + ss * D + k);
#pragma unroll
    for (int j = 1; j < kTcK; ++j) {
      if (FT && j >= FT) {
        x[j] = 0.f;
        continue;
      }
      const uint32_t r = __shfl_sync(0xFFFFFFFFu, rcur, j - 1);
      x[j] = ldg_if(table + (int64_t)r * D + k, j < F && r != kNoRow);
    }
#pragma unroll
    for (int m = 0; m < kTcDout; ++m) {
      const int e = k + kTcThreads * m;
      dn[m] = e < W ? __ldg(dout + ss * W + e) : 0.f;
    }
    const int64_t s2 = ss + nb;
    rnext = (s2 < B && lane < T) ? p.row_of[s2 * T + lane] : kNoRow;
    inext = (s2 < B && lane < T) ? p.inv[s2 * T + lane] : kNoRow;
  };
  // Once-row variant, warp 1: bulk-copy the accumulator rows of the last gathered sample's
  // once rows into buffer b and record its rows; one arrival (with the byte count) per use.
  auto stage_once = [&](int b) {
    const bool once = lane < T && un != kNoRow && (un & kInvOnce);
    const unsigned m = __ballot_sync(0xFFFFFFFFu, once);
    if (lane == 0) mbar_arrive_expect_tx(abar + b, (uint32_t)__popc(m) * (uint32_t)(D * 4));
    __syncwarp();
    if (once)
      bulk_copy_g2s(As + (b * 32 + lane + 1) * D, p.acc + (int64_t)rcur * D, (uint32_t)(D * 4),
                    abar + b);
    if (lane < 31) Rs[b * 32 + lane + 1] = rcur;
  };
  if (s < B) {
    gather(s);
    if (ONCE && warp == 1) stage_once(0);
  }
  uint32_t phase = 0;
  bool ok = true;
  int it = 0;
  for (; s < B; s += nb, ++it) {
    // 1. A operand: hi and lo TF32 parts of x_j[k] into this thread's TMEM lane
    {
      float hi[kTcK];
#pragma unroll
      for (int j = 0; j < kTcK; ++j) {
        if (FT && j >= FT) {
          hi[j] = 0.f;  // padding column: zero in both parts
          continue;
        }
        hi[j] = tf32_hi(x[j]);
        x[j] -= hi[j];
      }
      tmem_st32(tlane + kColAhi, hi);
      tmem_st32(tlane + kColAlo, x);
    }
    // 2. B operands: G[i][j] = G[j][i] = dout[D + pair(i, j)]
#pragma unroll
    for (int m = 0; m < kTcDout; ++m) {
      if (off_ij[m] >= 0) {
        const float g = dn[m], h = tf32_hi(g), l = g - h;
        *reinterpret_cast<float*>(smem + kOffBhi + off_ij[m]) = h;
        *reinterpret_cast<float*>(smem + kOffBhi + off_ji[m]) = h;
        *reinterpret_cast<float*>(smem + kOffBlo + off_ij[m]) = l;
        *reinterpret_cast<float*>(smem + kOffBlo + off_ji[m]) = l;
      }
    }
    const float d0 = dn[0];  // dout[k]: the dense vector's direct gradient
    uint32_t* Ub = Us + 32 * (it & 1);
    if (warp == 0) {
      if (lane < 31) Ub[lane + 1] = un;  // column i = feature i-1
      if (ONCE) {  // the sample's once columns, for every thread's epilogue in one word
        const unsigned om = __ballot_sync(0xFFFFFFFFu, lane < 31 && un != kNoRow && (un & kInvOnce));
        if (lane == 0) Om[it & 1] = om << 1;
      }
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    if (s + nb < B) gather(s + nb);  // next sample's loads in flight over the MMA and epilogue
    fence_proxy_async();             // B stores visible to the tensor core
    tc_fence_before();
    __syncthreads();
    // every thread is past the previous epilogue: the other buffer is free for the next sample
    if (ONCE && warp == 1 && s + nb < B) stage_once((it + 1) & 1);
    // 3. one thread issues the MMAs
    if (k == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kTcK / 8; ++ks)  // K step ks: bytes 32 ks .. 32 ks + 31 of each row
        umma_tf32_ts(tmem + kColD, tmem + kColAhi + 8 * ks,
                     umma_desc_sw128(sbase + kOffBhi + ks * 32, kBSBO), kTcIdesc, ks);
#pragma unroll
      for (int ks = 0; ks < kTcK / 8; ++ks)
        umma_tf32_ts(tmem + kColD, tmem + kColAhi + 8 * ks,
                     umma_desc_sw128(sbase + kOffBlo + ks * 32, kBSBO), kTcIdesc, 1);
#pragma unroll
      for (int ks = 0; ks < kTcK / 8; ++ks)
        umma_tf32_ts(tmem + kColD, tmem + kColAlo + 8 * ks,
                     umma_desc_sw128(sbase + kOffBhi + ks * 32, kBSBO), kTcIdesc, 1);
      umma_commit(bar);
    }
    // 4. epilogue
    const int b = it & 1;
    bool done = mbar_wait_polls(bar, phase, p.first_wait_polls);
    if (ONCE) done = mbar_wait_bounded(abar + b, (uint32_t)(it >> 1) & 1u) && done;
    if (!__syncthreads_and(done)) {
      ok = false;
      break;
    }
    phase ^= 1u;
    tc_fence_after();
    float* grow = p.g + k;
    const uint32_t omask = ONCE ? Om[b] : 0u;
#pragma unroll
    for (int qc = 0; qc < 4; ++qc) {
      if (8 * qc < F) {
        float dx[8];
        tmem_ld8(tlane + kColD + 8 * qc, dx);
        if (qc == 0) ddense[s * D + k] = dx[0] + d0;
        uint32_t u[8];
        *reinterpret_cast<uint4*>(u) = reinterpret_cast<const uint4*>(Ub + 8 * qc)[0];
        *reinterpret_cast<uint4*>(u + 4) = reinterpret_cast<const uint4*>(Ub + 8 * qc)[1];
#pragma unroll
        for (int c = 0; c < 8; ++c)
          if (FT == 0 || 8 * qc + c < FT) red_add_row(grow, u[c], dx[c]);
        if (ONCE) {
          // once columns of this group (the same for every thread: branches and tcgen05.ld
          // stay uniform)
          const uint32_t om = (omask >> (8 * qc)) & 0xFFu;
          if (om) {
            float* wtab = reinterpret_cast<float*>(p.table) + k;
            float* atab = p.acc + k;
            if (__popc(om) >= 4) {
              // most of the group: all eight columns are computed (no per-column branch);
              // stores only for once columns (the others' staged values go unused)
              float hi[8], lo[8];
              tmem_ld8(tlane + kColAhi + 8 * qc, hi);
              tmem_ld8(tlane + kColAlo + 8 * qc, lo);
              const float* Ab = As + (b * 32 + 8 * qc) * D + k;
              uint32_t r[8];
              *reinterpret_cast<uint4*>(r) = reinterpret_cast<const uint4*>(Rs + b * 32 + 8 * qc)[0];
              *reinterpret_cast<uint4*>(r + 4) = reinterpret_cast<const uint4*>(Rs + b * 32 + 8 * qc)[1];
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                float w = hi[c] + lo[c], a = Ab[c * D];
                adagrad_elem(w, a, dx[c], p.lr, p.eps);
                st_row_if(atab, r[c], a, om & (1u << c));
                st_row_if(wtab, r[c], w, om & (1u << c));
              }
            } else {
              // a few once columns (Zipf batches: ~4 of 26 per sample): a loop over them,
              // the gradient and both parts of the row read back from tensor memory
              const float* Ab = As + (b * 32 + 8 * qc) * D + k;
              const uint32_t* Rb = Rs + b * 32 + 8 * qc;
              const uint32_t tq = tlane + 8 * qc;
              for (uint32_t mm = om; mm; mm &= mm - 1) {
                const int c = __ffs(mm) - 1;
                float g, hw, lw;
                tmem_ld1x3(tq + kColD + c, tq + kColAhi + c, tq + kColAlo + c, g, hw, lw);
                float w = hw + lw, a = Ab[c * D];
                adagrad_elem(w, a, g, p.lr, p.eps);
                const uint32_t row = Rb[c];
                st_row_if(atab, row, a, 1u);
                st_row_if(wtab, row, w, 1u);
              }
            }
          }
        }
      }
    }
    tc_fence_before();  // TMEM reads ordered before the next MMA (behind the next barrier)
  }
  if (!ok && k == 0) {
    raise_flag(p.counters, EMB_FLAG_WAIT_LIMIT);
    // one more bounded wait for the MMA, and for the bulk copies of this sample and of the
    // next, before TMEM and shared memory are given up
    mbar_wait_bounded(bar, phase);
    if (ONCE) {
      mbar_wait_bounded(abar + (it & 1), (uint32_t)(it >> 1) & 1u);
      if (s + nb < B) mbar_wait_bounded(abar + ((it + 1) & 1), (uint32_t)((it + 1) >> 1) & 1u);
    }
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "n"(kTcCols)
                 : "memory");
  }
}

bool tc_supported(const Ctx* c) {
  return !c->p.bf16 && !c->multi_hot && c->p.T + 1 <= kMaxF && c->p.D == 128;
}

// The tensor-core backward is the default where it applies; EMB_FUSED_BWD=simt at context
// creation selects the FMA-pipe kernels instead.
bool use_tc_bwd(const Ctx* c) { return tc_supported(c) && c->bwd_impl != 2; }

// Once rows take per-element Adagrad in the epilogue; the row-wise variant would need the
// squared norm of the whole row (all four warps) first, and stays with the update kernel.
// The mark of a row seen twice takes bit 31 of its dedup-set key: rows below 2^31 only.
// Admission (hashed tables) holds some rows' updates and Adagrad Decay discounts the
// accumulators; the epilogue does neither.
bool once_direct_ok(const Ctx* c) {
  return use_tc_bwd(c) && !c->p.rowwise && c->total_rows <= (int64_t)kSetMulti - 1 &&
         c->p.admit_min <= 1 && !c->p.decay;
}

template <bool ONCE, int FT>
static cudaError_t run_bwd_tc(Ctx* c, const float* dout, const float* dense, int64_t B,
                              float* ddense, cudaStream_t s) {
  const int smem = ONCE ? kTcSmemOnce : kTcSmem;
  // TMEM holds 512 columns per SM: with at most 4 resident CTAs an allocation never waits
  const int per_sm = std::max(
      1, std::min(resident_ctas(c, k_fused_bwd_tc<ONCE, FT>, kTcThreads, smem), 512 / kTcCols));
  int64_t grid = (int64_t)per_sm * c->num_sms;
  if (grid > B) grid = B;
  LaunchScope ls(c, K_FUSED_BWD, s);
  k_fused_bwd_tc<ONCE, FT><<<(int)grid, kTcThreads, smem, s>>>(c->p, dout, dense, B, ddense);
  return cudaGetLastError();
}

cudaError_t launch_fused_bwd_tc(Ctx* c, const float* dout, const float* dense, int64_t B,
                                float* ddense, cudaStream_t s) {
  // The 26-table shape with once rows has its own instantiation for batches whose rows are
  // mostly looked up more than once (fewer than one unique row per two lookups in the last
  // batch, from the host mirror): backward 0.365 -> 0.322 ms on the Criteo step.  On the
  // uniform shape (0.97) it measured 2.45 against 2.34 ms, and without once rows 2% slower,
  // so those keep the generic kernel.
  if (!c->once_step) return run_bwd_tc<false, 0>(c, dout, dense, B, ddense, s);
  const uint32_t u = c->h_unique ? *reinterpret_cast<volatile const uint32_t*>(c->h_unique) : 0u;
  if (c->p.T + 1 == 27 && 2.0 * u < (double)c->last_nnz)
    return run_bwd_tc<true, 27>(c, dout, dense, B, ddense, s);
  return run_bwd_tc<true, 0>(c, dout, dense, B, ddense, s);
}

}  // namespace emb
