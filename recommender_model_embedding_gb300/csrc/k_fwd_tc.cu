// Fused lookup + pooling + dot interaction (forward) on the 5th-generation tensor cores
// (tcgen05 MMA, A operand and accumulator in tensor memory) for fp32 one-hot tables with
// D = 128 and F = T+1 <= 32 interaction vectors.
//
// OneEmbedding article, "operator optimisation" (FusedDotFeatureInteraction): the pairwise
// dot products of the dense vector and the pooled embeddings, x_i . x_j for i > j.  HugeCTR
// interview, section 3 (5): pooling fused with its neighbour (one-hot pooling is the row
// itself, so the gathered rows are the interaction's inputs and are never written back).
//
// Per sample the forward is the strict lower triangle of the Gram matrix X X^T (X: F vectors
// x 128).  The output indices i, j are vectors, so they take the M and N sides of the MMA
// and the contraction runs over the embedding dimension (K = 128).  M is 128 rows at full
// rate, so one MMA group serves a pair of samples:
//   A (M = 128, in TMEM): rows [x(s0) | lo(s0) | x(s1) | lo(s1)], 32 rows each
//   B (N = 64, shared memory): rows [x(s0) | x(s1)], the gathered fp32 rows themselves
//   D (128 x 64, in TMEM) = A B^T over K = 128 (16 MMAs of K = 8).
// fp32 accuracy from TF32 inputs: the tensor core reads an fp32 operand as TF32 by dropping
// its 13 low mantissa bits, hi(x) = x with those bits cleared; lo(x) = x - hi(x) is exact
// in fp32.  Then x_i . x_j = hi_i.hi_j + lo_i.hi_j + hi_i.lo_j + lo_i.lo_j, and the last term
// is below 2^-20 of |x_i||x_j| per element.  D holds hi.hi (rows of x, columns of its own
// sample) and lo_i.hi_j (rows of lo); the third term is the transposed element,
// hi_i.lo_j = D[lo_j][hi_i], so the epilogue reads it across lanes through shared memory:
//   G_ij = D[x_i][x_j] + D[lo_i][x_j] + D[lo_j][x_i].
// The cross-sample quarter blocks of D are computed and never read.
//
// One CTA per SM, warp-specialised, every hand-off an mbarrier (all waits bounded):
//  - three producer warps fill a ring of six stages, one pair each, in turn: lane l of
//    the warp copies 16-byte chunk l of one row with cp.async straight into the B operand
//    layout (K-major, 128-byte swizzle); each lane's copies arrive on the stage's mbarrier
//    when they land (cp.async.mbarrier.arrive), so the producer never waits for data;
//  - two consumer warpgroups take alternate pairs.  Once a stage is full, each thread
//    orders the landed rows before the tensor core's reads (proxy fence); thread m of the
//    group reads row m of A's row set from the stage and writes it (x), or its lo part
//    (warps 1 and 3 of the group), into its own TMEM lane, and warps 0 and 2 copy the
//    dense rows to the output.  Then the group runs the epilogue of its previous pair while
//    the tensor core works on this one: each warp writes its 32 lanes of D (x rows: hi.hi,
//    lo rows: lo.hi) to shared memory, and every thread of the group forms its share of
//    the pairs, G_ij = H[i][j] + L[i][j] + L[j][i], storing them to the output coalesced;
//  - one thread issues each pair's 16 MMAs into the group's accumulator (two per group,
//    alternating) and commits them twice: the stage is free, the accumulator is full.
// Each consumer warpgroup owns 256 TMEM columns: A [0, 128), accumulators [128, 256).
// The stage's padding rows (vectors F..31) stay zero; a missing second sample (odd B)
// leaves its rows as they were, and only blocks that no output reads depend on them.
#include <algorithm>

#include "interact_common.cuh"
#include "tc_common.cuh"

namespace emb {

constexpr int kFtGroups = 2;                        // consumer warpgroups
constexpr int kFtProducers = 3;                     // producer warps
constexpr int kFtWarpMma = 4 * kFtGroups + kFtProducers;  // the MMA-issuing warp
constexpr int kFtThreads = 32 * (kFtWarpMma + 1);   // 384
constexpr int kFtStages = 6;                        // ring of pair stages
constexpr int kFtRowBytes = 128;                    // one swizzled row of an atom column
constexpr int kFtAtomCol = 64 * kFtRowBytes;        // 64 rows x 32 fp32 of K
constexpr int kFtStage = 4 * kFtAtomCol;            // 4 atom columns: K = 128 (32 KB)
constexpr int kFtColsGroup = 256;                   // per group: A [0,128), D [128,256)
constexpr int kFtColA = 0, kFtColD = 128;
constexpr int kFtCols = kFtGroups * kFtColsGroup;   // 512: the whole tensor memory
constexpr int kFtHs = 33;                           // floats per row of the D row buffers
constexpr int kFtHmat = 32 * kFtHs;                 // one 32 x 32 block of D
constexpr int kFtMaxPairs = kMaxF * (kMaxF - 1) / 2;
constexpr int kFtOutPerThread = (2 * kFtMaxPairs + 127) / 128;  // pair outputs per thread
constexpr uint32_t kFtIdesc = idesc_tf32(128, 64);

// per group: H [2 samples][32][33] (lanes of x rows: hi.hi) and L [2][32][33] (lo rows)
constexpr int kFtOffRows = kFtStages * kFtStage;
constexpr int kFtOffBar = kFtOffRows + kFtGroups * 4 * kFtHmat * 4;
// barriers: full[S], empty[S], aready[G], dfull[G][2], dempty[G][2]
constexpr int kFtNumBars = 2 * kFtStages + kFtGroups * 5;
constexpr int kFtOffAbort = kFtOffBar + 8 * kFtNumBars;
constexpr int kFtOffTmem = kFtOffAbort + 8;
constexpr int kFtSmem = kFtOffTmem + 8 + 1024;      // + slack to align the stages to 1 KB
static_assert(kFtSmem <= 232448, "shared memory of the tensor-core forward");

// Byte offset, inside a stage, of logical 16-byte chunk `l` (elements 4l..4l+3) of row n.
__device__ __forceinline__ uint32_t stage_off(int n, int l) {
  return (uint32_t)((l >> 3) * kFtAtomCol + n * kFtRowBytes + (((l & 7) ^ (n & 7)) << 4));
}

// FT: the number of interaction vectors when known at compile time (27, the 26-table shape),
// else 0 (taken from p.T): the producers then skip the padding slots' index shuffles and each
// consumer thread holds only the pair outputs that exist.
template <int FT>
__global__ void __launch_bounds__(kFtThreads, 1) k_fused_fwd_tc(Params p, const float* dense,
                                                             int64_t B, float* out) {
  constexpr int kOut = FT ? (FT * (FT - 1) + 127) / 128 : kFtOutPerThread;  // 2P / 128
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = FT ? FT - 1 : p.T, F = FT ? FT : T + 1, D = 128;
  const int P = F * (F - 1) / 2;
  const int W = D + P;
  const float* table = reinterpret_cast<const float*>(p.table);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kFtOffBar);
  uint64_t* full = bars;                            // [S] stage filled (producer lanes)
  uint64_t* empty = bars + kFtStages;               // [S] stage read by its MMAs (commit)
  uint64_t* aready = bars + 2 * kFtStages;          // [G] A written (128 threads)
  uint64_t* dfull = aready + kFtGroups;             // [G][2] accumulator written (commit)
  uint64_t* dempty = dfull + 2 * kFtGroups;         // [G][2] accumulator read (128 threads)
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kFtOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kFtOffTmem);

  for (int e = tid; e < kFtStages * kFtStage / 16; e += kFtThreads)
    reinterpret_cast<float4*>(smem)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (warp == 0) tmem_alloc<kFtCols>(tmem_slot);
  if (tid == 0) {
    for (int i = 0; i < kFtStages; ++i) {
      mbar_init(full + i, 32);
      mbar_init(empty + i, 1);
    }
    for (int g = 0; g < kFtGroups; ++g) {
      mbar_init(aready + g, 128);
      for (int d = 0; d < 2; ++d) {
        mbar_init(dfull + 2 * g + d, 1);
        mbar_init(dempty + 2 * g + d, 128);
      }
    }
    *abort_flag = 0u;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int64_t npairs = (B + 1) / 2;
  const int64_t nq = gridDim.x;
  const int64_t q0 = blockIdx.x;
  // number of pairs this CTA processes (pair it of the CTA is q0 + it * nq)
  const int64_t nit = q0 < npairs ? (npairs - 1 - q0) / nq + 1 : 0;

  if (warp >= 4 * kFtGroups && warp < kFtWarpMma) {
    // ---------------- producers: pairs it = pw, pw + 2, ...
    const int pw = warp - 4 * kFtGroups;
    // lane t < T: the table rows of feature t of the pair's two samples (loaded one own
    // pair ahead); kNoRow past the batch or for a rejected lookup (the zero row is copied)
    auto load_rows = [&](int64_t it, uint32_t& r0, uint32_t& r1) {
      const int64_t s0 = 2 * (q0 + it * nq);
      r0 = (it < nit && lane < T) ? p.row_of[s0 * T + lane] : kNoRow;
      r1 = (it < nit && s0 + 1 < B && lane < T) ? p.row_of[(s0 + 1) * T + lane] : kNoRow;
    };
    uint32_t r0, r1;
    load_rows(pw, r0, r1);
    for (int64_t it = pw; it < nit; it += kFtProducers) {
      const int st = (int)(it % kFtStages);
      bool ok = it < kFtStages || mbar_wait_bounded(empty + st, (uint32_t)((it / kFtStages - 1) & 1));
      if (!__all_sync(0xFFFFFFFFu, ok && *abort_flag == 0u)) {  // the warp decides together
        *abort_flag = 1u;
        break;
      }
      const uint32_t c0 = r0, c1 = r1;
      load_rows(it + kFtProducers, r0, r1);  // the next own pair's rows
      const int64_t s0 = 2 * (q0 + it * nq);
      const bool two = s0 + 1 < B;
      // stage row v (sample 0) and 32 + v (sample 1): chunk `lane` of vector v's row; the
      // loop over the 32 row slots is unrolled so that the index shuffles overlap
      const uint32_t sst = sbase + (uint32_t)(st * kFtStage) + (uint32_t)((lane >> 3) * kFtAtomCol);
      const float* z = p.zero_row + 4 * lane;
#pragma unroll
      for (int v = 0; v < (FT ? FT : kMaxF); ++v) {
        const uint32_t ra = __shfl_sync(0xFFFFFFFFu, c0, (v + 31) & 31);
        const uint32_t rb = __shfl_sync(0xFFFFFFFFu, c1, (v + 31) & 31);
        if (v < F) {
          const uint32_t off = (uint32_t)(v * kFtRowBytes + (((lane & 7) ^ (v & 7)) << 4));
          const float* sa = v == 0 ? dense + s0 * D + 4 * lane
                                   : (ra != kNoRow ? table + (size_t)ra * D + 4 * lane : z);
          cp_async16_s(sst + off, sa);
          if (two) {
            const float* sb = v == 0 ? dense + (s0 + 1) * D + 4 * lane
                                     : (rb != kNoRow ? table + (size_t)rb * D + 4 * lane : z);
            cp_async16_s(sst + 32 * kFtRowBytes + off, sb);
          }
        }
      }
      cp_async_arrive_noinc(full + st);  // this lane's copies of the pair, once they land
    }
    cp_async_wait_n<0>();
  } else if (warp == kFtWarpMma) {
    // ---------------- MMA issuer (one thread)
    if (lane == 0) {
      int64_t issued = 0;
      for (int64_t it = 0; it < nit; ++it) {
        const int g = (int)(it & 1);
        const int64_t j = it >> 1;
        const int d = (int)(j & 1);
        const int st = (int)(it % kFtStages);
        bool ok = mbar_wait_bounded(aready + g, (uint32_t)(j & 1));
        ok = ok && (j < 2 || mbar_wait_bounded(dempty + 2 * g + d, (uint32_t)(((j - 2) >> 1) & 1)));
        if (!ok || *abort_flag) {
          *abort_flag = 1u;
          break;
        }
        tc_fence_after();
        const uint32_t sst = sbase + (uint32_t)(st * kFtStage);
        const uint32_t tg = tmem + (uint32_t)(g * kFtColsGroup);
#pragma unroll
        for (int ks = 0; ks < 16; ++ks)
          umma_tf32_ts(tg + kFtColD + 64 * d, tg + kFtColA + 8 * ks,
                       umma_desc_sw128(sst + (uint32_t)((ks >> 2) * kFtAtomCol + (ks & 3) * 32),
                                       8 * kFtRowBytes),
                       kFtIdesc, ks > 0 ? 1u : 0u);
        umma_commit(empty + st);
        umma_commit(dfull + 2 * g + d);
        issued = it + 1;
      }
      // before tensor memory is given up: the last pair's MMAs have completed
      if (issued > 0) {
        const int64_t it = issued - 1;
        mbar_wait_bounded(dfull + 2 * (int)(it & 1) + (int)((it >> 1) & 1),
                          (uint32_t)(((it >> 1) >> 1) & 1));
      }
    }
  } else {
    // ---------------- consumer warpgroup g: pairs it = g, g + 2, ...
    const int g = warp >> 2, wq = warp & 3;          // lane quarter wq of the group's TMEM
    const int gt = tid - 128 * g;                    // thread index inside the group
    const uint32_t tg = tmem + (uint32_t)(g * kFtColsGroup) + ((uint32_t)(wq * 32) << 16);
    const int n = (wq >> 1) * 32 + lane;             // stage row this thread writes to TMEM
    const bool is_lo = (wq & 1) != 0;
    // D rows of the group's pair in shared memory: [H(s0), H(s1), L(s0), L(s1)]
    float* rows = reinterpret_cast<float*>(smem + kFtOffRows) + g * 4 * kFtHmat;
    float* myrow = rows + ((is_lo ? 2 : 0) + (wq >> 1)) * kFtHmat + lane * kFtHs;
    // this thread's pair outputs e = gt + 128 k of the pair's 2P: shared-memory offsets of
    // H[i][j] (also of L[i][j], one block pair further) and of L[j][i], and the output
    // offset from the pair's first row
    uint32_t o_ij[kOut], o_ji[kOut], o_out[kOut];
#pragma unroll
    for (int k = 0; k < kOut; ++k) {
      const int e = gt + 128 * k;
      const int ss = e >= P ? 1 : 0;
      const int q = e - ss * P;
      const int cd = pair_code(q < P ? q : 0), i = cd >> 8, j = cd & 255;
      o_ij[k] = (uint32_t)(ss * kFtHmat + i * kFtHs + j);
      o_ji[k] = (uint32_t)((2 + ss) * kFtHmat + j * kFtHs + i);
      o_out[k] = e < 2 * P ? (uint32_t)(ss * W + D + q) : 0xFFFFFFFFu;
    }
    const int nj = (int)((nit - g + 1) / 2 > 0 ? (nit - g + 1) / 2 : 0);  // pairs of the group
    // all 128 threads of the group take every give-up decision together (a barrier with an
    // AND reduction), so none is left waiting at a named barrier
    auto group_ok = [&](bool ok) -> bool {
      uint32_t r;
      asm volatile(
          "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, 128, p;\n"
          " selp.u32 %0, 1, 0, q;\n}"
          : "=r"(r)
          : "r"((uint32_t)ok), "r"(1 + g)
          : "memory");
      return r != 0;
    };
    for (int j = 0; j <= nj; ++j) {
      const bool have = j < nj;
      const int64_t it = 2 * (int64_t)j + g;
      // accumulator of the previous pair written: A is free, D can be read
      bool ok = j < 1 || mbar_wait_bounded(dfull + 2 * g + ((j - 1) & 1), (uint32_t)(((j - 1) >> 1) & 1));
      if (!group_ok(ok && *abort_flag == 0u)) {
        *abort_flag = 1u;
        break;
      }
      if (j >= 1) tc_fence_after();
      if (have) {
        const int st = (int)(it % kFtStages);
        if (!group_ok(mbar_wait_bounded(full + st, (uint32_t)((it / kFtStages) & 1)))) {
          *abort_flag = 1u;
          break;
        }
        fence_proxy_async();  // the landed rows, before the tensor core reads them
        const uint32_t sst = sbase + (uint32_t)(st * kFtStage);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v[32];
#pragma unroll
          for (int l = 0; l < 8; ++l) {
            const float4 f = lds4(sst + stage_off(n, 8 * c + l));
            v[4 * l + 0] = f.x;
            v[4 * l + 1] = f.y;
            v[4 * l + 2] = f.z;
            v[4 * l + 3] = f.w;
          }
          if (is_lo) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) lo_pair(v[e], v[e + 1]);
          }
          tmem_st32(tg + kFtColA + 32 * c, v);
        }
        if (!is_lo) {  // the dense row of this warp's sample (stage row 0 or 32) to the output
          const int64_t s = 2 * (q0 + it * nq) + (wq >> 1);
          if (s < B) {
            const float4 f = lds4(sst + (uint32_t)((lane >> 3) * kFtAtomCol +
                                                   32 * (wq >> 1) * kFtRowBytes + (lane & 7) * 16));
            float* o = out + s * W + 4 * lane;
            o[0] = f.x;
            o[1] = f.y;
            o[2] = f.z;
            o[3] = f.w;
          }
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        mbar_arrive(aready + g);
      }
      if (j >= 1) {
        // epilogue of the group's previous pair (its MMAs are done; this pair's may run)
        const int jp = j - 1;
        const int64_t q = q0 + (2 * (int64_t)jp + g) * nq;
        float d[32];
        tmem_ld32(tg + kFtColD + 64 * (jp & 1) + 32 * (wq >> 1), d);
        tc_fence_before();
        mbar_arrive(dempty + 2 * g + (jp & 1));
#pragma unroll
        for (int c = 0; c < (FT ? FT : 32); ++c) myrow[c] = d[c];  // columns past F: never read
        asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory");
        float* ob = out + 2 * q * W;
        const int nvalid = (2 * q + 1 < B) ? 2 * P : P;  // pair outputs of existing samples
#pragma unroll
        for (int k = 0; k < kOut; ++k) {
          if (gt + 128 * k < nvalid)
            ob[o_out[k]] = rows[o_ij[k]] + rows[o_ij[k] + 2 * kFtHmat] + rows[o_ji[k]];
        }
        asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory");  // row buffers free again
      }
    }
  }
  if (tid == 0 && *abort_flag) raise_flag(p.counters, EMB_FLAG_WAIT_LIMIT);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc<kFtCols>(tmem);
  }
}

bool tc_fwd_supported(const Ctx* c) {
  return !c->p.bf16 && !c->multi_hot && c->p.T + 1 <= kMaxF && c->p.D == 128;
}

bool use_tc_fwd(const Ctx* c) { return tc_fwd_supported(c) && c->fwd_impl != 2; }

cudaError_t launch_fused_fwd_tc(Ctx* c, const float* dense, int64_t B, float* out,
                                cudaStream_t s) {
  // one CTA per SM: it allocates all 512 TMEM columns, and its shared memory rules out a
  // second one
  auto kern = c->p.T + 1 == 27 ? k_fused_fwd_tc<27> : k_fused_fwd_tc<0>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kFtSmem);
  if (e != cudaSuccess) return e;
  const int64_t npairs = (B + 1) / 2;
  int64_t grid = c->num_sms;
  if (grid > npairs) grid = npairs;
  LaunchScope ls(c, K_FUSED_FWD, s);
  kern<<<(int)grid, kFtThreads, kFtSmem, s>>>(c->p, dense, B, out);
  return cudaGetLastError();
}

}  // namespace emb
