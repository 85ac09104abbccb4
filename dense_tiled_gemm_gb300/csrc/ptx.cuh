// ptx.cuh: inline-PTX wrappers for the sm_100-family data path: mbarriers,
// tensor-memory-access (TMA) bulk copies, and the fifth-generation tensor
// core instructions (tcgen05: tensor-memory allocation, MMA, commit, loads).
//
// Each wrapper is a single instruction or a short fixed sequence, written
// from the PTX ISA's description of the instruction. Nothing here allocates
// or spins. The bounded waits built on mbar_try_wait live in the kernel.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace dtg {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%laneid;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ global flags
// Release store / acquire load of a 64-bit word at GPU scope: publish and
// observe data written by other CTAs of the same grid.
__device__ __forceinline__ void st_release_gpu(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// ------------------------------------------------------------------ cluster
__device__ __forceinline__ uint32_t cluster_cta_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory offset in CTA `cta` of this cluster.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t addr, uint32_t cta)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(cta));
    return r;
}

// ------------------------------------------------------------------ grid dependencies
// Programmatic dependent launch: block until the grids this one depends on
// (earlier work on the stream) have completed and their memory is visible.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Let the next grid on the stream be scheduled before this one finishes.
__device__ __forceinline__ void grid_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy and to the cluster.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_local(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrive on a barrier given by its shared::cluster address (possibly remote).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// One non-blocking probe: true once the phase with parity `parity` is complete.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Same probe with cluster-scope acquire, for barriers that CTAs of the
// cluster other than this one arrive on.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of one box into this CTA's shared memory; completion is
// counted in bytes on `bar` (this CTA's barrier).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t c0, int32_t c1)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
                 : "memory");
}

// 3-D tiled load (x innermost), completion on `bar` by transaction bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

// Paired-CTA form: the box lands in this CTA's shared memory while the
// completion is signalled on `bar_cluster`, a shared::cluster barrier address
// that may belong to the peer CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1)
{
    asm volatile("cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
                 : "memory");
}

// Paired-CTA multicast form: the box lands at the same shared-memory offset
// in every CTA of `cta_mask`, and each destination's bytes complete on the
// barrier at bar_cluster's offset in that destination's pair leader (the even
// CTA of its pair), whichever CTA issued the copy.
__device__ __forceinline__ void tma_load_2d_pair_mc(uint32_t dst, const CUtensorMap *map, uint32_t bar_cluster,
                                                    int32_t c0, int32_t c1, uint16_t cta_mask)
{
    asm volatile("cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
                 ".multicast::cluster [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "h"(cta_mask)
                 : "memory");
}

// 2-D tiled store of one box from this CTA's shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int32_t c0,
                                             int32_t c1)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}

// Same store with an L2 cache-policy hint (a policy from createpolicy).
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap *map, uint32_t src, int32_t c0,
                                                  int32_t c1, uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint"
                 " [%0, {%2, %3}], [%1], %4;" ::"l"(reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "l"(policy)
                 : "memory");
}

// L2 policy under which the accessed lines are the first to be evicted.
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    return policy;
}

__device__ __forceinline__ void bulk_commit_group()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until every committed bulk group has fully completed.
__device__ __forceinline__ void bulk_wait_group_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy reads (TMA store, tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05
template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    if constexpr (CG == 1)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                     "r"(ncols)
                     : "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_relinquish()
{
    if constexpr (CG == 1)
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    else
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    if constexpr (CG == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                     : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Operand kinds of the MMA:
//   KIND_F16   kind::f16,      FP16/BF16,          K = 16 per instruction
//   KIND_F8    kind::f8f6f4,   E4M3/E5M2,          K = 32
//   KIND_MXF8  kind::mxf8f6f4, E4M3/E5M2 + E8M0 scale per 32 K (scale_vec::1X), K = 32
//   KIND_MXF4  kind::mxf4,     packed E2M1 + E8M0 scale per 32 K (scale_vec::2X), K = 64
// Every instruction consumes 32 bytes of K from each operand row.
enum : int { KIND_F16 = 0, KIND_F8 = 1, KIND_MXF8 = 2, KIND_MXF4 = 3 };

__host__ __device__ constexpr bool kind_scaled(int kind) { return kind == KIND_MXF8 || kind == KIND_MXF4; }

// tcgen05.mma, tcgen05.cp and tcgen05.commit are each issued by one thread.
// The wrappers below are called by a whole converged warp: the warp computes
// the (warp-uniform) operands together, so that they stay in the uniform
// datapath, and the lane that elect.sync picks issues the instruction (the
// same lane every time, so its commits cover its products). Issued from a
// single divergent lane instead, every instruction first moves its operands
// there; with other warps of the same SM sub-partition competing for issue
// slots, that stretched a 64-cycle product (M128 N128 K16) to about 100
// cycles.
#define DTG_ELECT_PRED "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\t"

// D[tmem] (+)= A[smem] · B[smem] with an FP32 accumulator (unscaled kinds).
template <int CG, int KIND>
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                    uint32_t accumulate)
{
    static_assert(KIND == KIND_F16 || KIND == KIND_F8, "unscaled kinds only");
    if constexpr (CG == 1 && KIND == KIND_F16)
        asm volatile(DTG_ELECT_PRED "setp.ne.b32 p, %4, 0;\n\t"
                     "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
                     : "memory");
    else if constexpr (CG == 2 && KIND == KIND_F16)
        asm volatile(DTG_ELECT_PRED "setp.ne.b32 p, %4, 0;\n\t"
                     "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
                     : "memory");
    else if constexpr (CG == 1)
        asm volatile(DTG_ELECT_PRED "setp.ne.b32 p, %4, 0;\n\t"
                     "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
                     : "memory");
    else
        asm volatile(DTG_ELECT_PRED "setp.ne.b32 p, %4, 0;\n\t"
                     "@e tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
                     : "memory");
}

// D (+)= A * B with A read from tensor memory (one TMEM lane per row of A,
// two 16-bit elements per 32-bit column) and B from a shared-memory
// descriptor: kind::f16, one CTA.
__device__ __forceinline__ void mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(DTG_ELECT_PRED "setp.ne.b32 p, %4, 0;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Block-scaled MMA: D[tmem] (+)= (SFA ∘ A)·(SFB ∘ B). sfa_tmem / sfb_tmem are
// the tensor-memory addresses of the 32-bit columns that hold this
// instruction's E8M0 scales (one byte per row, picked by the scale-ID fields
// of idesc).
template <int CG, int KIND>
__device__ __forceinline__ void mma_scaled(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    static_assert(kind_scaled(KIND), "block-scaled kinds only");
    if constexpr (CG == 1 && KIND == KIND_MXF8)
        asm volatile(DTG_ELECT_PRED "setp.ne.b32 p, %6, 0;\n\t"
                     "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
                     "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
                     : "memory");
    else if constexpr (CG == 2 && KIND == KIND_MXF8)
        asm volatile(DTG_ELECT_PRED "setp.ne.b32 p, %6, 0;\n\t"
                     "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
                     "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
                     : "memory");
    else if constexpr (CG == 1)
        asm volatile(DTG_ELECT_PRED "setp.ne.b32 p, %6, 0;\n\t"
                     "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X "
                     "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
                     : "memory");
    else
        asm volatile(DTG_ELECT_PRED "setp.ne.b32 p, %6, 0;\n\t"
                     "@e tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X "
                     "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
                     : "memory");
}

// Copy 32 rows x 16 bytes from shared memory (matrix descriptor) into TMEM
// lanes 0-31 at 4 columns from taddr, replicated into each of the four lane
// quarters (.warpx4). With cta_group::2 the copy is made in both CTAs of the
// pair, each from its own shared memory into its own TMEM.
template <int CG>
__device__ __forceinline__ void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t s_desc)
{
    if constexpr (CG == 1)
        asm volatile(DTG_ELECT_PRED "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
                     "l"(s_desc)
                     : "memory");
    else
        asm volatile(DTG_ELECT_PRED "@e tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
                     "l"(s_desc)
                     : "memory");
}

// Arrive once on `bar` when every tcgen05 operation the elected lane issued
// before has completed. Single-CTA form.
__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile(DTG_ELECT_PRED
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

// Paired form: arrive on the barrier at the same offset in each CTA of
// `cta_mask` (bit i = cluster rank i).
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t cta_mask)
{
    asm volatile(DTG_ELECT_PRED
                 "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
                 " [%0], %1;\n\t}" ::"r"(bar),
                 "h"(cta_mask)
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t gets lane (base + t).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                 "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
                 "[%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// tcgen05.wait::ld that also names the registers of the load it completes as
// read-write operands, so that no computation on them can be placed before it
// (the load's register outputs are only valid after the wait).
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
                   "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                   "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// Store 32 lanes x 32 columns of 32-bit values (one row of 32 per thread of
// the warp) into tensor memory at taddr; warp-collective.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                 "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
                 "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
                   "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
                   "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
                   "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
                   "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor, 128-byte swizzle, sm_100-family format:
// start address >> 4 in bits 0-13, leading byte offset >> 4 in bits 16-29,
// stride byte offset >> 4 in bits 32-45, version 1 in bits 46-47, base
// offset 0 (tiles are 1024-byte aligned), swizzle mode 2 (128 B) in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Shared-memory matrix descriptor without swizzling: 8-row x 16-byte core
// matrices, SBO bytes between core matrices along the rows (LBO along K is
// unused for a single 16-byte column).
__device__ __forceinline__ uint64_t smem_desc_plain(uint32_t addr, uint32_t sbo)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    return d;   // layout type 0 (no swizzle) in bits 61-63
}

// Instruction descriptor for kind::f16 and kind::f8f6f4 with an FP32
// accumulator: D format bits 4-5 (1 = F32), A format bits 7-9 and B format
// bits 10-12, A major bit 15 (0 = K), B major bit 16 (1 = MN), N >> 3 in bits
// 17-22, M >> 4 in bits 24-28. The format code is 0 for F16 (kind::f16) or
// E4M3 (kind::f8f6f4), 1 for BF16 or E5M2.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t M, uint32_t N, uint32_t ab_format,
                                                  uint32_t b_mn_major)
{
    return (1u << 4) | (ab_format << 7) | (ab_format << 10) | (b_mn_major << 16) | ((N >> 3) << 17) |
           ((M >> 4) << 24);
}

// Instruction descriptor for the block-scaled kinds (kind::mxf8f6f4,
// kind::mxf4): B scale-factor ID bits 4-5, A format bits 7-9, B format bits
// 10-12, A and B K-major, N >> 3 in bits 17-22, scale type bit 23 (1 = E8M0),
// M >> 4 in bits 24-28, A scale-factor ID bits 29-30. The scale IDs (the
// byte of each 32-bit scale column an instruction starts at) are added per
// instruction: mx_sf_id(). Format codes: mxf8f6f4 E4M3 = 0, E5M2 = 1;
// mxf4 E2M1 = 1.
__host__ __device__ constexpr uint32_t make_idesc_mx(uint32_t M, uint32_t N, uint32_t ab_format)
{
    return (ab_format << 7) | (ab_format << 10) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24);
}

__host__ __device__ constexpr uint32_t mx_sf_id(uint32_t id) { return (id << 29) | (id << 4); }

} // namespace dtg
