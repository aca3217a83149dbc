// Thin inline-PTX wrappers for the sm_103a features the kernels use:
// mbarriers, TMA tensor copies, tcgen05 (TMEM allocation, MMA, loads/stores).
// Every wait is bounded: on expiry it records the site in the CTA's shared
// abort word, every role of the CTA unwinds, and the kernel copies the word to
// the device status word that the host reads (LAGA_ERR_TIMEOUT).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

namespace laga {

constexpr int kStatusTimeout = 5;
// A single wait on an mbarrier never legitimately takes this long.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// L2 prefetch of one tensor-map box (no shared memory, no completion signal):
// warms L2 for a box that a later cp.async.bulk.tensor load will read.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map), "r"(x), "r"(y),
               "r"(z)
               : "memory");
}

// Tensor-map store of one box shared -> global (bulk-group completion). Global
// writes outside the tensor are clipped; x must keep the 16-byte rule.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(map),
               "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most one committed bulk store group of this thread is still
// reading its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// Waits until at most N committed bulk stores of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read_n() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until every committed bulk store of this thread has completed (writes done).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Waits only until every committed bulk store of this thread has finished reading
// its shared-memory source: enough before that memory is reused or the CTA exits
// (the global writes still land before the grid completes).
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Plain (non-tensor) bulk copy global -> shared; both addresses 16-byte aligned,
// size a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Generic-proxy writes to shared memory become visible to the async proxy
// (tcgen05.mma operand reads, TMA stores).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle, 1024-byte aligned atoms.
// lbo/sbo in bytes. K-major: sbo = distance between 8-row groups, lbo unused.
// MN-major: lbo = distance between 64-element MN atoms, sbo = distance between
// 8-row K groups.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulation.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Warp-collective forms: every lane of a converged warp executes them and one
// lane (elect.sync) issues the instruction. Keeping the issuing loop warp-uniform
// lets descriptor arithmetic stay on the uniform datapath; a single lane running
// the loop alone issues MMAs markedly slower once softmax warps share its
// sub-partition.
__device__ __forceinline__ void mma_ss_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Blocks of two or four tcgen05.mma (kind::f16) on one accumulator, issued by one
// elected lane after a single elect.sync: the first MMA accumulates iff
// `accumulate` != 0, the others always accumulate. Measured on GB300: a warp that
// pays one elect.sync per MMA issues more slowly once busy compute warps share its
// SM sub-partition (the dK/dV step's MMAs 6% slower beside two of them); one per
// block of four keeps the tensor pipe fed.
__device__ __forceinline__ void mma2_ss_warp(uint32_t d_tmem, uint64_t a0, uint64_t a1, uint64_t b0, uint64_t b1,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "setp.eq.b32 t, %5, %5;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %3, %5, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %4, %5, t;\n\t}" ::"r"(d_tmem),
      "l"(a0), "l"(a1), "l"(b0), "l"(b1), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma4_ss_warp(uint32_t d_tmem, uint64_t a0, uint64_t a1, uint64_t a2, uint64_t a3,
                                             uint64_t b0, uint64_t b1, uint64_t b2, uint64_t b3, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %10, 0;\n\t"
      "setp.eq.b32 t, %9, %9;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %9, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %6, %9, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %9, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %8, %9, t;\n\t}" ::"r"(d_tmem),
      "l"(a0), "l"(a1), "l"(a2), "l"(a3), "l"(b0), "l"(b1), "l"(b2), "l"(b3), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma2_ts_warp(uint32_t d_tmem, uint32_t a0, uint32_t a1, uint64_t b0, uint64_t b1,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "setp.eq.b32 t, %5, %5;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %3, %5, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %4, %5, t;\n\t}" ::"r"(d_tmem),
      "r"(a0), "r"(a1), "l"(b0), "l"(b1), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma4_ts_warp(uint32_t d_tmem, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint64_t b0, uint64_t b1, uint64_t b2, uint64_t b3, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %10, 0;\n\t"
      "setp.eq.b32 t, %9, %9;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %5, %9, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %6, %9, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %7, %9, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %8, %9, t;\n\t}" ::"r"(d_tmem),
      "r"(a0), "r"(a1), "r"(a2), "r"(a3), "l"(b0), "l"(b1), "l"(b2), "l"(b3), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit_warp(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Arrive once on the mbarrier when every MMA issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp gets lane (base lane + t).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// ------------------------------------------------------------------ misc
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Two fp32 additions in one instruction: (a.x + b.x, a.y + b.y).
__device__ __forceinline__ float2 add_f32x2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 x, y, z;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 y, {%4, %5};\n\t"
      "add.rn.f32x2 z, x, y;\n\t"
      "mov.b64 {%0, %1}, z;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a 128-byte
// swizzled tile whose rows are 128 bytes (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B and the MMA reads with the 128B-swizzle descriptor).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// Byte offset of 16-byte chunk `chunk` (0..3) of row `row` inside a 64-byte
// swizzled tile whose rows are 64 bytes (CU_TENSOR_MAP_SWIZZLE_64B).
__device__ __forceinline__ uint32_t sw64_offset(uint32_t row, uint32_t chunk) {
  return row * 64u + ((chunk ^ ((row >> 1) & 3u)) << 4);
}

}  // namespace laga

namespace laga {
// Bounded wait that also gives up when another role of the CTA has set
// *abort_flag; on expiry it stores the timeout code and site in the flag.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                   int where) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > kWaitLimitNs) {
        *abort_flag = kStatusTimeout | (where << 8);
        return false;
      }
    }
  }
}

// Short bounded wait used only while unwinding after an abort.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > 200000000ull) return;  // 200 ms
  }
}
}  // namespace laga

namespace laga {
// Warp-uniform bounded wait: lane 0 waits, every lane gets its verdict.
__device__ __forceinline__ bool warp_wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                   int where) {
  bool w = true;
  if ((threadIdx.x & 31) == 0) w = mbar_wait_or_abort(bar, parity, abort_flag, where);
  const bool all = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
  __syncwarp();  // order lane 0's acquire before the other lanes' reads
  return all;
}

// Named barrier `id` over `nthreads` threads (a multiple of 32): every participant
// contributes `pred` and receives the AND of all contributions.
__device__ __forceinline__ bool bar_and(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Non-blocking test of an mbarrier phase (acquire on success). Meant to be issued
// by the MMA warp BEFORE a group of tcgen05.mma: a shared-memory access issued
// right after such a group waits behind it for well over 100 cycles, and a branch
// on its result leaves the tensor pipe idle for that long. The result is then
// consumed as a token by warp_wait_token after the group.
__device__ __forceinline__ uint32_t mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok;
}

// Warp-collective wait for a phase this lane already tested (token = that test's
// result): with a set token no memory is touched. The verdict is made uniform
// across the warp.
__device__ __forceinline__ bool warp_wait_token(uint64_t* bar, uint32_t parity, uint32_t token,
                                                volatile int* abort_flag, int where) {
  bool ok = true;
  if (!token) ok = mbar_wait_or_abort(bar, parity, abort_flag, where);
  return __all_sync(0xffffffffu, ok);
}

// Called by one thread after the CTA's final barrier: publish an abort.
__device__ __forceinline__ void publish_abort(volatile int* abort_flag, int* status) {
  const int a = *abort_flag;
  if (a != 0 && status != nullptr) atomicCAS(status, 0, a);
}
}  // namespace laga

// ------------------------------------------------------------------ debug trace
// Built only with -DLAGA_TRACE: kernels stamp the SM clock at chosen points of
// one CTA (blockIdx 0) into a per-file device array, slot
// (warp, step, tag), with plain stores; a debug export copies the array out.
// Release builds compile every trace point to nothing.
#ifdef LAGA_TRACE
#define LAGA_TRACE_WARPS 32
#define LAGA_TRACE_STEPS 512
#define LAGA_TRACE_TAGS 32
#define LAGA_TRACE_CAP (LAGA_TRACE_WARPS * LAGA_TRACE_STEPS * LAGA_TRACE_TAGS)
#define LAGA_TRACE_CTAS 32768
#ifndef LAGA_TRACE_BY
#define LAGA_TRACE_BY 0  // blockIdx.y of the CTA whose steps are stamped
#endif
#define LAGA_TRACE_DEFINE(name)                                                          \
  __device__ long long g_trace_##name[LAGA_TRACE_CAP];                                  \
  __device__ long long g_cta_##name[LAGA_TRACE_CTAS * 8];                               \
  __device__ long long g_stat_##name[LAGA_TRACE_CTAS * 8];                              \
  extern "C" int laga_debug_stat_##name(long long* host, int max) {                      \
    const int n = max < LAGA_TRACE_CTAS * 8 ? max : LAGA_TRACE_CTAS * 8;                 \
    cudaMemcpyFromSymbol(host, g_stat_##name, n * sizeof(long long));                   \
    return n;                                                                            \
  }                                                                                      \
  extern "C" int laga_debug_trace_##name(long long* host, int max) {                     \
    const int n = max < LAGA_TRACE_CAP ? max : LAGA_TRACE_CAP;                           \
    cudaMemcpyFromSymbol(host, g_trace_##name, n * sizeof(long long));                  \
    return n;                                                                            \
  }                                                                                      \
  extern "C" int laga_debug_cta_##name(long long* host, int max) {                       \
    const int n = max < LAGA_TRACE_CTAS * 8 ? max : LAGA_TRACE_CTAS * 8;                 \
    cudaMemcpyFromSymbol(host, g_cta_##name, n * sizeof(long long));                    \
    return n;                                                                            \
  }
#define LAGA_TRACE_POINT(name, tag, step)                                                \
  do {                                                                                   \
    if (blockIdx.x == 0 && blockIdx.y == LAGA_TRACE_BY && blockIdx.z == 0 && (step) >= 0 &&              \
        (step) < LAGA_TRACE_STEPS && (threadIdx.x >> 5) < LAGA_TRACE_WARPS)                               \
      g_trace_##name[((threadIdx.x >> 5) * LAGA_TRACE_STEPS + (step)) * LAGA_TRACE_TAGS + (tag)] = \
          clock64();                                                                     \
  } while (0)
// Per-CTA record (linear block index, SM id, entry and exit global time in ns,
// entry and exit SM clock), written by thread 0 at kernel entry (BEGIN) and
// after the final barrier (END).
#define LAGA_TRACE_CTA_BEGIN(name)                                                       \
  do {                                                                                   \
    const long long cta_ = blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z); \
    if (threadIdx.x == 0 && cta_ < LAGA_TRACE_CTAS) {                                    \
      uint32_t smid_;                                                                    \
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid_));                                 \
      g_cta_##name[cta_ * 8 + 0] = cta_;                                                 \
      g_cta_##name[cta_ * 8 + 1] = smid_;                                                \
      g_cta_##name[cta_ * 8 + 2] = (long long)global_ns();                               \
      g_cta_##name[cta_ * 8 + 4] = clock64();                                            \
    }                                                                                    \
  } while (0)
#define LAGA_TRACE_CTA_END(name)                                                         \
  do {                                                                                   \
    const long long cta_ = blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z); \
    if (threadIdx.x == 0 && cta_ < LAGA_TRACE_CTAS) {                                    \
      g_cta_##name[cta_ * 8 + 3] = (long long)global_ns();                               \
      g_cta_##name[cta_ * 8 + 5] = clock64();                                            \
    }                                                                                    \
  } while (0)
// Per-CTA counters (8 slots) kept in registers by one warp and written once.
#define LAGA_TRACE_STAT(name, slot, value)                                               \
  do {                                                                                   \
    const long long cta_ = blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z); \
    if (cta_ < LAGA_TRACE_CTAS) g_stat_##name[cta_ * 8 + (slot)] = (value);              \
  } while (0)
#else
#define LAGA_TRACE_DEFINE(name)
#define LAGA_TRACE_STAT(name, slot, value) \
  do {                                     \
  } while (0)
#define LAGA_TRACE_POINT(name, tag, step) \
  do {                                    \
  } while (0)
#define LAGA_TRACE_CTA_BEGIN(name) \
  do {                             \
  } while (0)
#define LAGA_TRACE_CTA_END(name) \
  do {                           \
  } while (0)
#endif
