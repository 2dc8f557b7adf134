// sm_103a building blocks for the tensor-core kernels: tcgen05 MMA with
// TMEM accumulators, shared-memory matrix descriptors, mbarriers with bounded
// waits, bulk-async (TMA) copies, and the canonical 128-byte-swizzled operand
// layouts for bf16.
//
// Layout conventions (bf16, 128-byte swizzle, every tile 1024-byte aligned):
//  * K-major operand with R rows (M or N) and K columns: K is split in blocks
//    of 64 elements (128 B); block kb occupies R*128 bytes; inside it rows are
//    128 B apart, 8-row groups 1024 B apart, and the 16-byte chunk c of row r
//    sits at chunk position c ^ (r % 8).  Descriptor: SBO = 1024, LBO unused.
//  * MN-major operand with MN extent R and K rows: MN is split in atoms of
//    64 elements (128 B) that are LBO = K*128 bytes apart; inside an atom the
//    K rows are 128 B apart, 8-row groups 1024 B apart, same chunk swizzle
//    (chunk from the MN offset, row from K).  Descriptor: LBO = K*128, SBO = 1024.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// byte offset of element (r, k) in a K-major tile of R rows
__device__ __forceinline__ uint32_t off_k(int r, int k, int R) {
  const int c = (k & 63) >> 3;
  return (uint32_t)((k >> 6) * R * 128 + (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4) +
                    (k & 7) * 2);
}
// byte offset of element (mn, k) in an MN-major tile with K rows
__device__ __forceinline__ uint32_t off_mn(int mn, int k, int K) {
  const int c = (mn & 63) >> 3;
  return (uint32_t)((mn >> 6) * K * 128 + (k >> 3) * 1024 + (k & 7) * 128 + ((c ^ (k & 7)) << 4) +
                    (mn & 7) * 2);
}

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;      // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;      // 128-byte swizzle
  return d;
}
// descriptor of k-step j (16 elements) of a K-major tile with R rows
__device__ __forceinline__ uint64_t desc_k(uint32_t base, int R, int j) {
  return desc_sw128(base + (uint32_t)((j >> 2) * R * 128 + (j & 3) * 32), 16, 1024);
}
// descriptor of k-step j (16 K rows) of an MN-major tile with K rows
__device__ __forceinline__ uint64_t desc_mn(uint32_t base, int K, int j) {
  return desc_sw128(base + (uint32_t)(j * 2048), (uint32_t)K * 128, 1024);
}

// instruction descriptor: bf16 x bf16 -> fp32, dense
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
      :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
// The same, executed by a whole converged warp: one elected lane (the lowest,
// so always the same one) issues.  Descriptors stay warp-uniform, which makes
// a run of issues several times cheaper than from a single-thread branch.
__device__ __forceinline__ void mma_w(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p, e; .reg .b32 r; elect.sync r|e, 0xffffffff; setp.ne.b32 p, %4, 0; "
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
      :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void mma_commit_w(uint32_t mbar) {
  asm volatile(
      "{ .reg .pred e; .reg .b32 r; elect.sync r|e, 0xffffffff; "
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0]; }"
      :: "r"(mbar) : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(mbar) : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// generic-proxy smem writes -> visible to the tensor core / bulk copies
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(slot_smem), "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols));
}

// 32 lanes x 16 / 32 consecutive 32-bit columns: each thread gets its lane's
// values.  The load and its wait sit in one asm statement: the destination
// registers of tcgen05.ld are only valid after tcgen05.wait::ld, and a separate
// wait would leave the compiler free to read (or copy) them before it.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr) : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr) : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ---- mbarriers -----------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(mbar), "r"(count));
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(mbar), "r"(bytes) : "memory");
}
// one arrival (release at CTA scope)
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(mbar) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t mbar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
  return done != 0;
}

// Device-side error word: bit 0 = an mbarrier wait gave up; bit 1 = a gate
// outside the chunked prefill's range [-10, 0] (or NaN) was read.  Read and
// cleared by the host through kda_device_errors(); one copy per translation
// unit that includes this header (the tensor-core kernels live in one).
constexpr int kDevErrWait = 1;
constexpr int kDevErrGate = 2;
static __device__ int g_kda_device_error = 0;

// Wait for phase `parity` of an mbarrier, giving up after about one second
// (2^31 SM clocks); on timeout raise the error word and return false.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity) {
  if (mbar_test(mbar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_test(mbar, parity)) {
    if (clock64() - t0 > (1LL << 31)) {
      atomicOr(&g_kda_device_error, kDevErrWait);
      return false;
    }
  }
  return true;
}

// bulk-async copy global -> shared (TMA engine), completion counted on mbar
__device__ __forceinline__ void bulk_g2s(uint32_t dst_smem, const void* src, uint32_t bytes, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(dst_smem), "l"(src), "r"(bytes), "r"(mbar) : "memory");
}

// 2-D tiled TMA load (tile mode) into shared memory, completion on mbar; x (the
// innermost coordinate) times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      :: "r"(dst), "l"(map), "r"(x), "r"(y), "r"(mbar) : "memory");
}

// Wait for phase `parity` of an mbarrier unless `abort_flag` becomes nonzero,
// giving up after about one second (2^31 SM clocks, which raises the error
// word).  Returns true only when the phase completed.
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t mbar, uint32_t parity, volatile int* abort_flag) {
  const long long t0 = clock64();
  while (!mbar_test(mbar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > (1LL << 31)) {
      atomicOr(&g_kda_device_error, kDevErrWait);
      return false;
    }
  }
  return true;
}

// shared -> global bulk copy tracked by bulk groups (16-byte aligned ends, size a multiple of 16)
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               :: "l"(dst), "r"(src_smem), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk groups have finished reading shared memory / have completed
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void st_bf16(unsigned char* base, uint32_t off, float x) {
  *reinterpret_cast<__nv_bfloat16*>(base + off) = __float2bfloat16_rn(x);
}

}  // namespace tc
}  // namespace kda
