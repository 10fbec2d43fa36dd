// Inline-PTX wrappers for sm_103a: mbarrier, TMA (cp.async.bulk.tensor),
// tcgen05 (TMEM alloc, MMA, commit, ld) and fences.  Written from the PTX ISA
// descriptions of these instructions.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {
namespace ptx {

MOE_DEVICE uint32_t smem_addr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

MOE_DEVICE uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier ----
MOE_DEVICE void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

MOE_DEVICE void fence_barrier_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

MOE_DEVICE void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

MOE_DEVICE void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

MOE_DEVICE bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: spins until the phase with `parity` completed, or until
// `deadline` (globaltimer ns) passed or *abort is set.  Returns false on give-up.
MOE_DEVICE bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t deadline, volatile int* abort) {
    uint32_t n = 0;
    while (!mbar_try_wait(bar, parity)) {
        if ((++n & 1023u) == 0) {
            if (*abort) return false;
            if (globaltimer() > deadline) return false;
        }
    }
    return true;
}

// ---- TMA ----
MOE_DEVICE void prefetch_tmap(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

MOE_DEVICE uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

MOE_DEVICE uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

MOE_DEVICE void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t c0, int32_t c1,
                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// 16-byte global -> shared copy (cp.async, L2 only, with an L2 cache policy); src_bytes < 16 zero-fills the
// rest of the 16 bytes (0: no global read at all).  cp_async_wait_all waits for this thread's copies.
MOE_DEVICE void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes, uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst), "l"(src),
                 "r"(src_bytes), "l"(policy)
                 : "memory");
}

MOE_DEVICE void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Orders this thread's generic-proxy writes to shared memory before later async-proxy reads (tcgen05.mma
// operands, TMA stores) that are synchronised with it.
MOE_DEVICE void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

MOE_DEVICE void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t c0, int32_t c1, int32_t c2,
                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

MOE_DEVICE void tma_load_4d(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t c0, int32_t c1, int32_t c2,
                            int32_t c3, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

MOE_DEVICE void tma_load_5d(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t c0, int32_t c1, int32_t c2,
                            int32_t c3, int32_t c4, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_addr(bar)),
        "l"(policy)
        : "memory");
}

// ---- tcgen05 ----
MOE_DEVICE void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {   // whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

MOE_DEVICE void tmem_relinquish() {   // whole warp
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

MOE_DEVICE void tmem_dealloc(uint32_t taddr, uint32_t ncols) {   // whole warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

MOE_DEVICE void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_DEVICE void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= (A * 2^(SFA-127)) * (B * 2^(SFB-127))^T, kind::mxf8f6f4 with one E8M0 scale per 32 along K
// (scale_vec::1X): A and B E4M3 in shared memory (descriptors), K = 32 per instruction.  The scale factors
// sit in TMEM at sfa_tmem / sfb_tmem; the byte of each 32-bit column used by this instruction is the
// scale-factor id carried in idesc (bits 29-30 for A, 4-5 for B).
MOE_DEVICE void mma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t sfa_tmem,
                         uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}\n"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once all tcgen05.mma issued by this thread have completed.
MOE_DEVICE void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// Warp-wide issue: the whole warp runs the issue loop, so the addresses and descriptors stay warp-uniform,
// and only the lane with `issue` != 0 executes the instruction (predicated, no branch).  Always pass the same
// lane: a commit tracks the MMAs issued by its own thread.  On GB300 an M=128, K=16, N<=128 MMA issued this
// way took about 29 ns against 50 ns from a loop that only lane 0 runs.
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16/fp16 in, fp32 accumulate).
MOE_DEVICE void mma_f16_by(uint32_t issue, uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                           uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p, i;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 i, %5, 0;\n"
        " @i tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(issue)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16: A is M rows in TMEM lanes, K packed two
// 16-bit values per 32-bit column (8 columns per 16-element k step).
MOE_DEVICE void mma_f16_tmem_a_by(uint32_t issue, uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                  uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p, i;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 i, %5, 0;\n"
        " @i tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(issue)
        : "memory");
}

MOE_DEVICE void mma_commit_by(uint32_t issue, uint64_t* bar) {
    asm volatile(
        "{\n .reg .pred i;\n setp.ne.b32 i, %1, 0;\n"
        " @i tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(
            smem_addr(bar)),
        "r"(issue)
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i gets columns [col, col+32) of lane (base + i).
MOE_DEVICE void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

MOE_DEVICE void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

MOE_DEVICE void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Waits for this thread's tcgen05.ld and ties the 32 destination registers to the wait, so that no use of
// them can be scheduled before it (for loads issued ahead of their use).
MOE_DEVICE void tmem_ld_wait_regs(uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
          "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
          "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]),
          "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
          "+r"(r[30]), "+r"(r[31])
        :
        : "memory");
}

// As tmem_ld_wait_regs, for 16 destination registers.
MOE_DEVICE void tmem_ld_wait_regs16(uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
          "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
        :
        : "memory");
}

// 32 lanes x 4 consecutive 32-bit columns: thread i writes columns [col, col+4) of lane (base + i).
MOE_DEVICE void tmem_st_32x32b_x4(uint32_t taddr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r0), "r"(r1),
                 "r"(r2), "r"(r3)
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i writes columns [col, col+32) of lane (base + i).
MOE_DEVICE void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

MOE_DEVICE void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---- CTA pairs (clusters of 2 CTAs sharing one tcgen05 MMA: cta_group::2) ----
MOE_DEVICE uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

MOE_DEVICE uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

MOE_DEVICE uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// All threads of every CTA in the cluster (release / acquire at cluster scope).
MOE_DEVICE void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared::cluster address of the variable at `local` (a shared::cta address) in the CTA of rank `rank`.
MOE_DEVICE uint32_t map_to_rank(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

MOE_DEVICE uint32_t ld_shared_cluster_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Arrive on an mbarrier of another CTA of the cluster (address from map_to_rank).
MOE_DEVICE void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMA tile load into this CTA's shared memory whose completion is counted on an mbarrier that may sit in the
// peer CTA of the pair (`bar` is a shared::cluster address).
MOE_DEVICE void tma_load_2d_pair(void* dst, const CUtensorMap* m, uint32_t bar, int32_t c0, int32_t c1,
                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
        : "memory");
}

MOE_DEVICE void tma_load_3d_pair(void* dst, const CUtensorMap* m, uint32_t bar, int32_t c0, int32_t c1, int32_t c2,
                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
        : "memory");
}

MOE_DEVICE void tma_load_4d_pair(void* dst, const CUtensorMap* m, uint32_t bar, int32_t c0, int32_t c1, int32_t c2,
                                 int32_t c3, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar), "l"(policy)
        : "memory");
}

MOE_DEVICE void tma_load_5d_pair(void* dst, const CUtensorMap* m, uint32_t bar, int32_t c0, int32_t c1, int32_t c2,
                                 int32_t c3, int32_t c4, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar), "l"(policy)
        : "memory");
}

// TMEM allocation for a CTA pair: one warp of EACH CTA of the pair executes these together.
MOE_DEVICE void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

MOE_DEVICE void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

MOE_DEVICE void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Warp-wide pair forms (see mma_f16_by): every lane runs them, only the lane with `issue` != 0 executes.
// D[tmem] (+)= A * B^T over the CTA pair, kind::f16: A's M = 256 rows are 128 in each CTA's shared memory and
// B's N rows are N/2 in each, at the same offsets as the descriptors give in the issuing CTA; each CTA's TMEM
// holds its 128 rows of D.  Issued by one thread of the pair.
MOE_DEVICE void mma_f16_pair_by(uint32_t issue, uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p, i;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 i, %5, 0;\n"
        " @i tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(issue)
        : "memory");
}
// Arrive once on the mbarrier at the same shared-memory offset in every CTA of `cta_mask` when all tcgen05.mma
// issued by this thread have completed.
MOE_DEVICE void mma_commit_pair_by(uint32_t issue, uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "{\n .reg .pred i;\n setp.ne.b32 i, %2, 0;\n"
        " @i tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n}\n"
        ::"r"(smem_addr(bar)), "h"(cta_mask), "r"(issue)
        : "memory");
}

// Shared-memory matrix descriptor for a K-major operand staged by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row core groups 1024 bytes apart
// (stride byte offset), leading byte offset unused for this layout, fixed
// descriptor version 1 (bits 46-47), swizzle mode 2 = 128B (bits 61-63).
// The start address must sit in a 1024-byte aligned tile, plus k*32 bytes to
// select the k-th 16-element slice of the 64-element row.
MOE_DEVICE uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3FFFu);          // start address
    d |= uint64_t(1) << 16;                          // leading byte offset (16 B, ignored)
    d |= uint64_t(1024 >> 4) << 32;                  // stride byte offset
    d |= uint64_t(1) << 46;                          // version
    d |= uint64_t(2) << 61;                          // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16 with BF16 A and B, FP32 D, both K-major.
MOE_DEVICE constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4)                       // D format: f32
           | (1u << 7)                     // A format: bf16
           | (1u << 10)                    // B format: bf16
           | (uint32_t(N >> 3) << 17)      // N / 8
           | (uint32_t(M >> 4) << 24);     // M / 16
}

// Instruction descriptor, kind::mxf8f6f4 with E4M3 A and B, both K-major, E8M0 (UE8M0) scale factors, FP32 D;
// the scale-factor ids (bits 4-5 for B, 29-30 for A) are or-ed in per instruction.
MOE_DEVICE constexpr uint32_t idesc_mxf8(int M, int N) {
    return (0u << 7)                       // A format: E4M3
           | (0u << 10)                    // B format: E4M3
           | (uint32_t(N >> 3) << 17)      // N / 8
           | (1u << 23)                    // scale factor type: UE8M0
           | (uint32_t(M >> 4) << 24);     // M / 16
}

MOE_DEVICE constexpr uint32_t idesc_sf_ids(uint32_t a_id, uint32_t b_id) { return (a_id << 29) | (b_id << 4); }

}  // namespace ptx
}  // namespace moe
