// tc_ptx.cuh -- thin inline-PTX wrappers for the Blackwell (sm_103a) tensor-core
// path: TMEM allocation, tcgen05.mma (kind::f16, bf16 operands, fp32
// accumulators), tcgen05.ld/st, mbarriers with bounded waits, and TMA tiled
// loads. Nothing here is specific to the attention method.
//
// Shared-memory operand layout used throughout (no swizzle, "core matrices"):
// a core matrix is 8 rows x 16 bytes (8 bf16), stored as 128 contiguous bytes.
//   K-major operand  (MN index r, K index k):
//       byte(r, k) = (r/8)*SBO + (k/8)*LBO + (r%8)*16 + (k%8)*2
//   MN-major operand (MN index r, K index k):
//       byte(r, k) = (r/8)*SBO + (k/8)*LBO + (k%8)*16 + (r%8)*2
// i.e. with no swizzle the leading byte offset is always the stride between
// core matrices along K and the stride byte offset the stride between 8-row
// groups along M/N, whichever way the core matrix itself is oriented (checked
// against a host GEMM for both orientations and both group orders).
// One kind::f16 MMA consumes K = 16, i.e. two core matrices along K; the next
// K step starts 2*LBO bytes further.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include "debug_check.cuh"

// Timeline trace points. They expand to nothing unless a diagnostic build
// defines TSA_TRACE_DECL (declared once per kernel thread) and
// TSA_TRACE_EVENT(event, arg) before including this header.
#ifndef TSA_TRACE_DECL
#define TSA_TRACE_DECL
#define TSA_TRACE_EVENT(ev, a) ((void)0)
#endif

namespace tsa {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- descriptors ------------------------------------------------------------
// Shared-memory matrix descriptor (tcgen05): start address, leading and stride
// byte offsets (all >> 4), version 1 at bits 46-47, no swizzle, base offset 0.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo & 0x3FFFFu) >> 4) << 16;
  d |= (uint64_t)((sbo & 0x3FFFFu) >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// ---- checks of the debug build (debug_check.cuh) ------------------------------
#ifdef TSA_DEBUG
// The CTA's dynamic shared memory: [dyn_smem_lo, dyn_smem_lo + dyn_smem_size)
// (every extern shared array starts where the dynamic shared memory does).
__device__ __forceinline__ uint32_t dyn_smem_lo() {
  extern __shared__ __align__(16) uint8_t tsa_dynamic_smem[];
  return smem_u32(tsa_dynamic_smem);
}
__device__ __forceinline__ uint32_t dyn_smem_size() {
  uint32_t r;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
  return r;
}
// ncols columns from the address's column lie inside the 512 allocated
__device__ __forceinline__ bool chk_tmem_cols(uint32_t taddr, uint32_t ncols) {
  const uint32_t col = taddr & 0xFFFFu;
  return TSA_DCHECK(col + ncols <= 512u, dbg::kTmemColumns, col, ncols);
}
// a tcgen05.ld/st of this warp: its own 32-lane quarter, columns inside
__device__ __forceinline__ bool chk_tmem_warp(uint32_t taddr, uint32_t ncols) {
  const uint32_t lane = taddr >> 16, quarter = 32u * ((threadIdx.x >> 5) & 3u);
  return TSA_DCHECK(lane == quarter, dbg::kTmemLanes, lane, quarter) && chk_tmem_cols(taddr, ncols);
}
// an MMA accumulator or A operand in TMEM: lane 0, columns inside
__device__ __forceinline__ bool chk_tmem_mma(uint32_t taddr, uint32_t ncols) {
  return TSA_DCHECK((taddr >> 16) == 0u, dbg::kTmemLanes, taddr >> 16, 0) && chk_tmem_cols(taddr, ncols);
}
// the bytes of a no-swizzle operand of `rows` rows (M or N) and K = 16
__device__ __forceinline__ bool chk_smem_operand(uint64_t desc, uint32_t rows) {
  const uint32_t start = (uint32_t)(desc & 0x3FFFu) << 4;
  const uint32_t lbo = (uint32_t)((desc >> 16) & 0x3FFFu) << 4;
  const uint32_t sbo = (uint32_t)((desc >> 32) & 0x3FFFu) << 4;
  const uint32_t end = start + (rows / 8u - 1u) * sbo + lbo + 128u;
  // a descriptor holds the low 18 bits of the address; in a cluster the
  // shared-window address of the CTA's own memory carries its rank above them
  const uint32_t lo = dyn_smem_lo() & 0x3FFFFu, hi = lo + dyn_smem_size();
  return TSA_DCHECK(start >= lo && end <= hi, dbg::kSmemOperand, ((uint64_t)lo << 32) | start,
                    ((uint64_t)hi << 32) | end);
}
// a shared-memory address with `align`-byte alignment inside the CTA's
// dynamic shared memory, `bytes` of it
__device__ __forceinline__ bool chk_smem_range(uint32_t saddr, uint32_t bytes, uint32_t align) {
  const uint32_t lo = dyn_smem_lo(), hi = lo + dyn_smem_size();
  return TSA_DCHECK(saddr % align == 0u && saddr >= lo && saddr + bytes <= hi, dbg::kBulkCopy,
                    ((uint64_t)lo << 32) | saddr, ((uint64_t)hi << 32) | bytes);
}
#else
__device__ __forceinline__ bool chk_tmem_cols(uint32_t, uint32_t) { return true; }
__device__ __forceinline__ bool chk_tmem_warp(uint32_t, uint32_t) { return true; }
__device__ __forceinline__ bool chk_tmem_mma(uint32_t, uint32_t) { return true; }
__device__ __forceinline__ bool chk_smem_operand(uint64_t, uint32_t) { return true; }
__device__ __forceinline__ bool chk_smem_range(uint32_t, uint32_t, uint32_t) { return true; }
#endif

// Instruction descriptor of kind::f16 with bf16 A and B and an fp32 accumulator.
// a_mn / b_mn select MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---- TMEM -------------------------------------------------------------------
// Executed by one full warp. Writes the allocated base address to *dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy shared-memory writes -> visible to the async proxy (MMA, TMA).
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], issued by one elected lane of a converged
// warp: the operands stay warp-uniform (uniform registers), which keeps the
// issue cost per MMA low.
__device__ __forceinline__ void mma_bf16_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  if (dbg::kEnabled) {
    const uint32_t n = ((idesc >> 17) & 0x3Fu) << 3, m = ((idesc >> 24) & 0x1Fu) << 4;
    if (!(chk_tmem_mma(d_tmem, n) && chk_smem_operand(adesc, m) && chk_smem_operand(bdesc, n))) return;
  }
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}
// As mma_bf16_elect with A read from TMEM: row i of A at lane i, two bf16 per
// 32-bit column (element 2j in the low half of column j), K = 16 per MMA
// (8 columns), K-major.
__device__ __forceinline__ void mma_bf16_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                                  uint32_t idesc, uint32_t accumulate) {
  if (dbg::kEnabled) {
    const uint32_t n = ((idesc >> 17) & 0x3Fu) << 3;
    if (!(chk_tmem_mma(d_tmem, n) && chk_tmem_mma(a_tmem, 8u) && chk_smem_operand(bdesc, n))) return;
  }
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      :: "r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}
// Arrive once on the mbarrier when every MMA issued so far by the elected
// lane is done.
__device__ __forceinline__ void mma_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
      :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool elect_one() {
  uint32_t r;
  asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\tselp.u32 %0, 1, 0, e;\n\t}" : "=r"(r));
  return r != 0;
}

// 32 lanes x 16 columns of 32 bits: thread t of the warp gets lane (base + t).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  if (dbg::kEnabled && !chk_tmem_warp(taddr, 16u)) {
    for (int e = 0; e < 16; ++e) r[e] = 0u;
    return;
  }
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// 32 lanes x 32 columns of 32 bits in one load.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  if (dbg::kEnabled && !chk_tmem_warp(taddr, 32u)) {
    for (int e = 0; e < 32; ++e) r[e] = 0u;
    return;
  }
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  if (dbg::kEnabled && !chk_tmem_warp(taddr, 16u)) return;
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
         "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
         "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---- mbarriers --------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase with the given parity to complete, giving up after
// `limit_ns` nanoseconds. Returns false on time-out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// As mbar_wait, but also gives up as soon as *abort is set, and sets it on a
// time-out, so that every waiter of a CTA stops once one of them has given up.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                                   volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > limit_ns) {
      *abort = 1;
      return false;
    }
  }
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}

// ---- TMA --------------------------------------------------------------------
// 4-D tiled load of a box into shared memory, completing on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, uint64_t* bar, int c0, int c1,
                                            int c2, int c3) {
  if (dbg::kEnabled && !(TSA_DCHECK(c0 % 8 == 0, dbg::kTmaCoord, 0, c0) && chk_smem_range(smem_u32(dst), 16u, 16u) &&
                         chk_smem_range(smem_u32(bar), 8u, 8u)))
    return;
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5, %6}], [%2];"
      :: "r"(smem_u32(dst)), "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// Untiled bulk copy global -> shared (both 16-byte aligned, size a multiple
// of 16), completing on `bar` (tx bytes).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  if (dbg::kEnabled &&
      !(TSA_DCHECK(reinterpret_cast<uintptr_t>(src) % 16 == 0 && bytes % 16 == 0, dbg::kBulkCopy,
                   reinterpret_cast<uintptr_t>(src), bytes) &&
        chk_smem_range(smem_u32(dst), bytes, 16u)))
    return;
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// 4-D tiled store of a box from shared memory (bulk-group completion). The
// caller makes its shared-memory writes visible to the async proxy first.
__device__ __forceinline__ void tma_store_4d(const void* tmap, const void* src, int c0, int c1, int c2, int c3) {
  if (dbg::kEnabled &&
      !(TSA_DCHECK(c0 % 8 == 0, dbg::kTmaCoord, 0, c0) && TSA_DCHECK(c1 >= 0, dbg::kTmaCoord, 1, c1) &&
        TSA_DCHECK(c2 >= 0, dbg::kTmaCoord, 2, c2) && TSA_DCHECK(c3 >= 0, dbg::kTmaCoord, 3, c3) &&
        chk_smem_range(smem_u32(src), 16u, 16u)))
    return;
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];"
               :: "l"(tmap), "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk stores have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... and are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---- programmatic dependent launch ---------------------------------------------
// Wait until the grids this one depends on have completed and their writes are
// visible (returns at once when launched without a programmatic dependency).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next grid in the stream be launched now (its own grid_dep_wait
// still waits for this grid to complete).
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- thread-block clusters (distributed shared memory) -------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The address of this CTA's shared-memory location `saddr` in the shared
// memory of cluster CTA `rank` (the same offset there).
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
  return d;
}
__device__ __forceinline__ void st_cluster_f4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};"
               :: "r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
}
__device__ __forceinline__ void st_cluster_flag(uint32_t addr, uint32_t v) {
  asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster; this thread's earlier
// writes (to that CTA's shared memory too) are released at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(cluster_addr) : "memory");
}
// try_wait with acquire at cluster scope: the writes the arriving threads of
// the other CTA released are visible once it returns true.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// Every thread of every CTA of the cluster arrives, then waits.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---- packing ----------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace tc
}  // namespace tsa
