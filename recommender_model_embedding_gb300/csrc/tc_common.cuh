// tcgen05 (5th-generation tensor core) primitives shared by the tensor-core interaction
// kernels: the 128-byte-swizzled shared-memory matrix descriptor, the instruction
// descriptor of kind::tf32, the MMA with A in tensor memory, tensor-memory loads and
// stores, commit and fences.  Written from the field layouts of the PTX ISA (tcgen05 matrix
// and instruction descriptors).
#pragma once

#include "interact_common.cuh"

namespace emb {

// Descriptor of a K-major operand in the 128-byte swizzled layout: rows of 128 bytes (32
// fp32 along K), 8-row groups `sbo` bytes apart; inside each 1024-byte group the 16-byte
// chunk c of row r sits at chunk position c ^ (r % 8).  The swizzle follows address bits, so
// the group must start on a 1024-byte boundary; a K step inside the 128-byte row advances the
// start address.  The leading byte offset is not used by this layout (encoded as 1).
// Layout type 2 (bits 61-63) selects the 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)1 << 16) |
         ((uint64_t)(sbo >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::tf32: D fp32, A and B tf32, both K-major, no negation.
constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4)                       // D format fp32
         | (2u << 7)                     // A format tf32
         | (2u << 10)                    // B format tf32
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// D (TMEM) (+)= A (TMEM) * B (shared memory); accumulate = 0 overwrites D.
__device__ __forceinline__ void umma_tf32_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 consecutive 32-bit columns of the calling thread's TMEM lane from registers.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
      "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
      "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]),
      "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]),
      "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 8 consecutive fp32 columns of the calling thread's TMEM lane.
// The load and its wait form one asm statement: the outputs are defined only once the wait
// has returned, so the compiler cannot schedule a use of them in between.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive fp32 columns of the calling thread's TMEM lane (load and wait together).
// Columns a, b and c of this warp's 32 lanes (one value each), one wait for the three.
__device__ __forceinline__ void tmem_ld1x3(uint32_t ta, uint32_t tb, uint32_t tc, float& va,
                                           float& vb, float& vc) {
  uint32_t ra, rb, rc;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%3];\n"
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%1}, [%4];\n"
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%2}, [%5];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(ra), "=r"(rb), "=r"(rc)
      : "r"(ta), "r"(tb), "r"(tc)
      : "memory");
  va = __uint_as_float(ra);
  vb = __uint_as_float(rb);
  vc = __uint_as_float(rc);
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Tensor-memory allocation of `cols` columns (a power of two >= 32) by one whole warp; the
// base address is written to *slot in shared memory.
template <int kCols>
__device__ __forceinline__ void tmem_alloc(uint32_t* slot) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "n"(kCols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <int kCols>
__device__ __forceinline__ void tmem_dealloc(uint32_t base) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "n"(kCols)
               : "memory");
}

// ---- row staging: 16-byte cp.async copies, shared-memory loads, the TF32 remainder ----

__device__ __forceinline__ void cp_async16_s(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Arrive on the mbarrier once all of this thread's earlier cp.async copies have landed (the
// arrival is one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait_n() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float4 lds4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// lo(x) = x - hi(x) for two values at once: -hi(x) is x with the 13 low bits cleared and the
// sign flipped (one logic op), and the sum is exact.
__device__ __forceinline__ void lo_pair(float& a, float& b) {
  const float na = __uint_as_float((__float_as_uint(a) & 0xFFFFE000u) ^ 0x80000000u);
  const float nb = __uint_as_float((__float_as_uint(b) & 0xFFFFE000u) ^ 0x80000000u);
  uint64_t r;
  asm("{\n .reg .b64 x, y;\n mov.b64 x, {%1, %2};\n mov.b64 y, {%3, %4};\n"
      " add.rn.f32x2 %0, x, y;\n}"
      : "=l"(r)
      : "f"(a), "f"(b), "f"(na), "f"(nb));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}

}  // namespace emb
