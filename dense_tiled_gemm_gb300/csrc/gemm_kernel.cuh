// gemm_kernel.cuh: the persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
// C = A·B with FP16/BF16 or FP8 (E4M3/E5M2) operands, or the block-scaled
// (MX) C = (SFA ∘ A)·(SFB ∘ B) with MXFP8/MXFP4 operands, an FP32 accumulator
// in tensor memory (TMEM) and a cast on store. "Two Waves, One Stage Apart" (sections "Why the Matrix
// Pipeline Drains" and "Two Waves, One Stage Apart") keeps the matrix unit
// busy by holding data preparation one stage ahead of matrix work. Here that
// offset comes from fixed warp roles linked by shared-memory barriers, not
// from two wave groups taking turns:
//
//   warp 0     producer: one thread issues TMA loads of A and B k-blocks into
//              a ring of STAGES shared-memory slots;
//   warp 1     MMA issuer: the warp walks the job list together and one
//              elected lane issues tcgen05.mma on each filled slot and frees
//              it with tcgen05.commit; the warp owns the TMEM allocation;
//   warps 2-5  epilogue: tcgen05.ld of the accumulator, FP32 -> output cast,
//              swizzled staging in shared memory, TMA store.
//
// The dependency rule of that page's section "Dependencies Cross Groups and
// Iterations" (writes complete before the reader starts, reads finish before
// a slot is refilled) maps onto a full/empty barrier pair per ring slot, and
// a full/empty pair per TMEM accumulator. The page's section "Avoiding
// Unnecessary Waits" asks for one barrier per independent buffer, so that no
// false wait delays matrix work; each slot has its own pair here.
//
// Two accumulators of up to 256 FP32 columns each (TMEM columns 0 and 256)
// let the epilogue of one tile run under the main loop of the next. With
// CG = 2 a cluster of two CTAs shares each 256-row tile (tcgen05 cta_group::2):
// each CTA loads its own 128 rows of A and its half of B, and the even CTA
// issues the MMAs for both.
//
// Tails: TMA loads fill out-of-range rows/columns (ragged M, N and the last
// k-block of K) with zeros, and TMA stores clip at the matrix edge. The
// "Porting High-Performance HIP Kernels to FlyDSL" page (section "Buffer
// Resource Descriptors") relies on hardware range checks in the same way.
//
// Every wait is bounded (WaitCtx). Past the limit, a thread records the site
// in the library's device status word and stops: from then on it issues no
// work and no signal (no TMA, no MMA, no commit, no arrive), so it can never
// push a barrier out of step. The roles that depend on it then block in their
// own bounded waits, see the launch's timeout in the status word, and stop
// too. Only operations already in flight are drained, with bounded waits. The
// control flow is unchanged, so every CTA or cluster barrier is still reached
// and the kernel returns instead of hanging.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "ptx.cuh"
#include "schedule.cuh"

namespace dtg {

constexpr int SLAB_BYTES = 128;      // one K slab: one 128-byte swizzle row of every operand row
constexpr int BLOCK_M_CTA = 128;     // accumulator rows per CTA = TMEM lanes
constexpr int MMA_K_BYTES = 32;      // K bytes of one tcgen05.mma (K = 16 FP16/BF16, 32 FP8)
constexpr int SLAB_MMAS = SLAB_BYTES / MMA_K_BYTES;

// K elements in one slab: 64 for 16-bit operands, 128 for FP8, 256 for packed FP4.
__host__ __device__ constexpr int kind_slab_k(int kind) { return kind == KIND_F16 ? 64 : kind == KIND_MXF4 ? 256 : 128; }

// Block-scaled kinds. The E8M0 scales of up to 128 rows and 4 consecutive
// 32-K blocks form one 512-byte atom: byte m32 * 16 + m4 * 4 + k4 holds the
// scale of row m4 * 32 + m32, block k4. tcgen05.cp (32x128b.warpx4) turns
// an atom into 4 TMEM columns, lane m32 of every lane quarter, column m4,
// byte k4. A block-scaled MMA reads the scale of row m of A at column m / 32
// from its A-scale address (each CTA of a pair holds its own 128 rows), and
// the scale of column n of B at column n / 32 from its B-scale address, for
// all N columns of the instruction (each CTA of a pair holds all of them), in
// the byte its descriptor's scale-ID picks. A ring stage carries SF_GROUPS
// groups of 4 blocks: per group one atom of A and SFB_ATOMS atoms of B (the
// whole tile width). Before each K slab's MMAs the MMA warp copies that
// slab's groups into a TMEM scale buffer; tcgen05.cp and tcgen05.mma of one
// thread run in issue order. Consecutive slabs alternate between two
// buffers, at columns BN and BN + 256 (beside each accumulator), so a slab's
// copies never overwrite scales that the previous slab's MMAs may still read
// and the tensor pipe does not drain between slabs. Accumulators use columns
// [0, BN) and [256, 256 + BN), so block-scaled tiles are at most 224 wide.
constexpr int SF_ATOM_BYTES = 512;
constexpr int SF_ATOM_ROWS = 32;
constexpr int SF_ROW_BYTES = 16;
constexpr int MX_MAX_STAGES = 8;
constexpr int NUM_THREADS = 320;     // at most: producer warp, MMA warp, 8 epilogue warps
constexpr int EPI_WARP0 = 2;
// A launch runs 4 or 8 epilogue warps (192 or 320 threads): 8 shorten each
// tile's epilogue, which pays where a unit's last epilogue is a large share of
// its time (one or two tiles per unit), and cost a little in main loops that
// overlap an epilogue.
constexpr int EPI_WARPS_MAX = 8;
constexpr int TMEM_COLS = 512;       // two accumulators at columns 0 and 256
constexpr int ACC_STRIDE = 256;
constexpr int EPI_COLS = 32;         // accumulator columns per epilogue chunk
constexpr int MAX_STAGES = 8;
constexpr int SMEM_LIMIT = 232448;   // 227 KB of dynamic shared memory per CTA

enum : uint32_t { OUT_F16 = 0, OUT_BF16 = 1, OUT_F32 = 2 };

// Wait sites reported in the status detail: role << 8 | barrier kind.
enum : uint32_t {
    SITE_PRODUCER_EMPTY = 0x001,
    SITE_PRODUCER_DRAIN = 0x002,
    SITE_MMA_TMEM_EMPTY = 0x103,
    SITE_MMA_FULL = 0x104,
    SITE_MMA_DONE = 0x105,
    SITE_EPI_TMEM_FULL = 0x206,
    SITE_SELFTEST = 0x307,
    SITE_EPI_PARTIAL = 0x209,  // an owner waiting for another unit's partial sum
    SITE_SMEM_ALIGN = 0x008,   // dynamic shared memory not 1024-byte aligned: nothing ran
};

struct KernelParams {
    int32_t M, N, K;
    int32_t num_m_tiles, num_n_tiles, num_tiles, num_k_blocks, group_m;
    uint32_t idesc;
    uint32_t out_dtype;
    uint32_t b_mn_major;
    uint32_t direct_store;     // 1: write C with ordinary stores (unaligned C)
    uint32_t stages;           // ring depth (2 .. MAX_STAGES)
    uint32_t staging_bytes;    // one epilogue staging buffer: 32 rows x 32 columns of C
    uint32_t staging_bufs;     // staging buffers per TMEM lane quarter: 2 or 4, shared by its epilogue warps
    void *C;                   // used by the direct-store path
    int32_t sk_tiles;          // trailing tiles scheduled stream-K (0: all tiles data-parallel)
    float4 *partials;          // stream-K partial sums: one slot per CTA (128 rows x block_n FP32)
    unsigned long long *flags; // stream-K: per (CTA, epilogue warp), the id of the launch that filled it
    uint64_t timeout_ns;       // per-wait limit
    unsigned long long launch_id;
    unsigned long long *status;  // [0] first timed-out launch, [1] site, [2] last timed-out launch
    // Optional clock trace (null: off): CTA 0 writes %globaltimer (ns) and
    // clock64 (SM cycles) once global memory may be touched, [0] and [1], and
    // again after its teardown barrier, [2] and [3]. Their ratio is the SM
    // clock over the launch.
    unsigned long long *trace;
    // Self-test only (-1: off): unit 0's producer issues neither the
    // expect-tx arrive nor the loads of k-block `withhold_kb` of its first
    // job, so that stage never fills and the waits behind it run out.
    int32_t withhold_kb;
};

// KS = K slabs per ring stage, KIND = operand kind (KIND_F16, KIND_F8,
// KIND_MXF8, KIND_MXF4). One slab is a 128-byte-wide K strip of A and B in
// the 128-byte swizzle layout (64 K of 16-bit operands, 128 K of FP8, 256 K
// of packed FP4: 4 MMAs in every case). A stage holds KS slabs of A, KS slabs
// of B and, for the block-scaled kinds, the scale blocks of A and B, so one
// barrier wait on the MMA thread covers 4 x KS MMAs.
template <int CG, int BN, int KS, int KIND>
struct TileConfig {
    static_assert(CG == 1 || CG == 2, "cta_group is 1 or 2");
    static_assert(KS == 1 || KS == 2, "one or two K slabs per stage");
    static constexpr bool SCALED = kind_scaled(KIND);
    static constexpr int BN_CTA = BN / CG;   // B rows (K-major) or columns (MN-major) per CTA
    static_assert(BN % (16 * CG) == 0 && BN <= 256 && BN_CTA % 8 == 0, "invalid tile width");
    static_assert(!SCALED || (BN <= 224 && BN_CTA <= 128), "block-scaled tiles: <= 224 wide, <= 128 B rows per CTA");
    static constexpr int SLAB_K = kind_slab_k(KIND);
    static constexpr int A_SLAB = BLOCK_M_CTA * SLAB_BYTES;
    static constexpr int B_SLAB = BN_CTA * SLAB_BYTES;
    static constexpr int A_BYTES = KS * A_SLAB;
    static constexpr int AB_BYTES = KS * (A_SLAB + B_SLAB);
    static constexpr int STAGE_K = KS * SLAB_K;
    // scale groups per stage (4 blocks of 32 K each), B atoms per group (whole tile width)
    static constexpr int SF_GROUPS = SCALED ? STAGE_K / 128 : 0;
    static constexpr int SFB_ATOMS = (BN + 127) / 128;
    static constexpr int SFA_BYTES = SF_GROUPS * SF_ATOM_BYTES;
    static constexpr int SFB_BYTES = SF_GROUPS * SFB_ATOMS * SF_ATOM_BYTES;
    static constexpr int STAGE_TX = AB_BYTES + SFA_BYTES + SFB_BYTES;   // bytes TMA delivers per stage and CTA
    // distance between ring slots: the next 1024-byte boundary, so that every
    // slot's slabs keep the alignment of the 128-byte swizzle (one-slab MXFP8
    // stages carry 31.5 KB)
    static constexpr int STAGE_BYTES = (STAGE_TX + 1023) / 1024 * 1024;
    // TMEM scale buffers, one per K slab, alternating between SF_COL = BN and
    // SF_COL + 256: a slab's groups g < SLAB_SF_GROUPS, A at +4g, B at
    // +4 * SLAB_SF_GROUPS + 4 * (g * SFB_ATOMS + atom)
    static constexpr int SLAB_SF_GROUPS = SCALED ? SLAB_K / 128 : 0;
    static constexpr uint32_t SF_COL = SCALED ? static_cast<uint32_t>(BN) : 0u;
    static constexpr uint32_t SF_B_OFF = 4u * SLAB_SF_GROUPS;
    static_assert(!SCALED || (SLAB_SF_GROUPS >= 1 && SF_COL % 4u == 0 &&
                              SF_COL + SF_B_OFF + 4u * SLAB_SF_GROUPS * SFB_ATOMS <= 256u),
                  "a slab's TMEM scale buffer fits between the two accumulators");
    // TMA x coordinate units per slab: FP16/BF16 elements, or bytes for the 8- and 4-bit kinds
    static constexpr int SLAB_X = KIND == KIND_F16 ? 64 : 128;
    // K blocks of 32 per MMA: 2 for packed FP4 (K = 64), else 1 (K <= 32)
    static constexpr int MMA_SF_BLOCKS = KIND == KIND_MXF4 ? 2 : 1;
    static_assert(A_SLAB % 1024 == 0 && B_SLAB % 1024 == 0, "slabs must stay 1024-byte aligned");
};

// Dynamic shared memory, from a 1024-byte aligned base:
//   ring      stages x {KS slabs of A 128 x 128 B, KS slabs of B BN_CTA x 128 B} (128-byte swizzle)
//   staging   4 lane quarters x 2 or 4 buffers x staging_bytes (2 KB for 16-bit C, 4 KB for FP32 C),
//             split between a quarter's epilogue warps (one or two)
//   barriers  full[stages], empty[stages], tmem_full[2], tmem_empty[2], mma_done
//   TMEM base address written by tcgen05.alloc
__host__ __device__ constexpr uint32_t smem_bytes_for(uint32_t stage_bytes, uint32_t stages,
                                                      uint32_t staging_bytes, uint32_t staging_bufs)
{
    return stages * stage_bytes + 4u * staging_bufs * staging_bytes + (2u * stages + 5u) * 8u + 16u;
}

// ------------------------------------------------------------------ bounded waits
struct WaitCtx {
    uint64_t limit_ns;
    unsigned long long id;
    unsigned long long *status;
    bool aborted;
};

__device__ __forceinline__ void record_timeout(unsigned long long *status, unsigned long long id,
                                               uint32_t site)
{
    atomicCAS(&status[0], 0ull, id);
    atomicExch(&status[1], static_cast<unsigned long long>(site));
    atomicExch(&status[2], id);
    __threadfence();
}

template <bool CLUSTER>
__device__ __forceinline__ bool probe(uint32_t bar, uint32_t parity)
{
    return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
}

// Slow path of a wait: spin on `bar` until phase `parity` completes (returns
// true), until another thread of this launch has timed out (returns false),
// or until `limit_ns` passes (records the site and returns false).
template <bool CLUSTER>
__device__ __noinline__ bool wait_bounded_slow(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                               unsigned long long id, unsigned long long *status,
                                               uint32_t site)
{
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (probe<CLUSTER>(bar, parity))
            return true;
        if ((n & 63u) == 0) {
            const volatile unsigned long long *st = status;
            if (st[2] == id)
                return false;
            if (global_timer_ns() - t0 > limit_ns) {
                record_timeout(status, id, site);
                return false;
            }
        }
    }
}

// Wait for phase `parity` of `bar`. Returns false, without waiting, once this
// thread has seen the launch time out; the fast path is one probe.
template <bool CLUSTER>
__device__ __forceinline__ bool wait_bounded(WaitCtx &w, uint32_t bar, uint32_t parity,
                                             uint32_t site)
{
    if (w.aborted)
        return false;
    if (probe<CLUSTER>(bar, parity))
        return true;
    if (!wait_bounded_slow<CLUSTER>(bar, parity, w.limit_ns, w.id, w.status, site))
        w.aborted = true;
    return !w.aborted;
}

// Teardown wait: runs even after an abort (it only bounds how long copies or
// MMAs already in flight may take to land), and never waits past the limit.
template <bool CLUSTER>
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                        unsigned long long id, unsigned long long *status,
                                        uint32_t site)
{
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (probe<CLUSTER>(bar, parity))
            return;
        if ((n & 63u) == 0 && global_timer_ns() - t0 > limit_ns) {
            record_timeout(status, id, site);
            return;
        }
    }
}

// Wait until *flag == id (another CTA of this launch has published its
// partial sum). Returns false after a timeout of this or another thread of
// the launch, recording the site in the first case.
static __device__ __noinline__ bool wait_flag_slow(const unsigned long long *flag, uint64_t limit_ns,
                                            unsigned long long id, unsigned long long *status, uint32_t site)
{
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (ld_acquire_gpu(flag) == id)
            return true;
        if ((n & 15u) == 0) {
            const volatile unsigned long long *st = status;
            if (st[2] == id)
                return false;
            if (global_timer_ns() - t0 > limit_ns) {
                record_timeout(status, id, site);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait_flag_bounded(WaitCtx &w, const unsigned long long *flag, uint32_t site)
{
    if (w.aborted)
        return false;
    if (ld_acquire_gpu(flag) == w.id)
        return true;
    if (!wait_flag_slow(flag, w.limit_ns, w.id, w.status, site))
        w.aborted = true;
    return !w.aborted;
}

// Row of the packed scale tensor (16-byte rows) where the atoms of row block
// rb for ring stage kb start: blocks are row-block major, then stage, then
// atom, 32 rows of 16 bytes per atom.
__device__ __forceinline__ int sf_atom_row(int rb, int kb, int num_kb, int groups)
{
    return ((rb * num_kb + kb) * groups) * SF_ATOM_ROWS;
}

// ------------------------------------------------------------------ tile order
// Persistent tile t -> (m_blk, n_blk). Tiles run in groups of group_m tile
// rows. Inside a group, the tile row changes fastest, so tiles running at the
// same time share A row panels and B column panels in L2.
__device__ __forceinline__ void tile_coords(const KernelParams &p, int t, int &m_blk, int &n_blk)
{
    const int per_group = p.group_m * p.num_n_tiles;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int gm = min(p.num_m_tiles - first_m, p.group_m);
    const int r = t - g * per_group;
    m_blk = first_m + r % gm;
    n_blk = r / gm;
}

// ------------------------------------------------------------------ epilogue helpers
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint32_t pack2(uint32_t lo, uint32_t hi, uint32_t out_dtype)
{
    const float a = __uint_as_float(lo), b = __uint_as_float(hi);
    if (out_dtype == OUT_BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);   // .x (low half) = a
        return *reinterpret_cast<uint32_t *>(&v);
    }
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Write one accumulator row chunk (32 FP32 values of row `lane`) into a staging
// buffer in the layout the C tensor map's swizzle expects:
//   FP32 out: 128-byte rows, 16-byte unit j stored at j ^ (row % 8)        (128B swizzle)
//   16-bit out: 64-byte rows, 16-byte unit j stored at j ^ ((row / 2) % 4) (64B swizzle)
__device__ __forceinline__ void stage_row(uint32_t buf, uint32_t lane, const uint32_t (&v)[32],
                                          uint32_t out_dtype)
{
    if (out_dtype == OUT_F32) {
        const uint32_t row = buf + lane * 128u;
#pragma unroll
        for (uint32_t j = 0; j < 8; ++j)
            st_shared_v4(row + ((j ^ (lane & 7u)) << 4), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                         v[4 * j + 3]);
    } else {
        const uint32_t row = buf + lane * 64u;
#pragma unroll
        for (uint32_t j = 0; j < 4; ++j)
            st_shared_v4(row + ((j ^ ((lane >> 1) & 3u)) << 4), pack2(v[8 * j], v[8 * j + 1], out_dtype),
                         pack2(v[8 * j + 2], v[8 * j + 3], out_dtype),
                         pack2(v[8 * j + 4], v[8 * j + 5], out_dtype),
                         pack2(v[8 * j + 6], v[8 * j + 7], out_dtype));
    }
}

// Ordinary predicated stores of one row chunk, for a C whose base or row pitch
// cannot be described to the TMA engine.
__device__ __forceinline__ void store_row_direct(const KernelParams &p, int row, int col0,
                                                 const uint32_t (&v)[32])
{
    if (row >= p.M)
        return;
    const int64_t base = static_cast<int64_t>(row) * p.N;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int col = col0 + i;
        if (col >= p.N)
            break;
        const float f = __uint_as_float(v[i]);
        if (p.out_dtype == OUT_F32)
            static_cast<float *>(p.C)[base + col] = f;
        else if (p.out_dtype == OUT_F16)
            static_cast<__half *>(p.C)[base + col] = __float2half_rn(f);
        else
            static_cast<__nv_bfloat16 *>(p.C)[base + col] = __float2bfloat16_rn(f);
    }
}

// ------------------------------------------------------------------ the kernel
// MC = CTA pairs per cluster that share their A tiles (1 or 2; 2 needs CG = 2).
// With MC = 2 a cluster of four CTAs takes two tiles side by side in N: pair
// p (ranks 2p, 2p + 1) computes tile column 2 * n_unit + p, and both pairs
// use the same 256 rows of A. Each CTA loads 64 of its 128 A rows per slab
// and multicasts them to the CTA with the same row half in the other pair, so
// every A row is read from L2 once per cluster instead of once per pair. The
// completion of a multicast pair load lands on the barrier of each destination
// CTA's pair leader, so each leader still expects exactly the bytes its two
// CTAs receive; a ring slot is free again only when both pairs' products have
// read it (each pair's commit arrives on every CTA's empty barrier).
template <int CG, int BN, int KS, int KIND, int MC = 1>
__global__ void __launch_bounds__(NUM_THREADS, 1)
gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_c,
                    const __grid_constant__ CUtensorMap tmap_sfa,   // block-scaled kinds only
                    const __grid_constant__ CUtensorMap tmap_sfb, const KernelParams p)
{
    using Cfg = TileConfig<CG, BN, KS, KIND>;
    static_assert(MC == 1 || (MC == 2 && CG == 2 && !Cfg::SCALED), "A is shared by CTA pairs of plain products only");
    constexpr int CS = CG * MC;   // CTAs per cluster
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw);
    if (base & 1023u) {
        // 128-byte-swizzled tiles need a 1024-byte aligned base; report and run nothing
        if (threadIdx.x == 0)
            record_timeout(p.status, p.launch_id, SITE_SMEM_ALIGN);
        return;
    }
    uint8_t *smem = smem_raw;
    const uint32_t stages = p.stages;

    const uint32_t warp = threadIdx.x / 32u;
    const uint32_t lane = threadIdx.x % 32u;
    const uint32_t rank = (CS > 1) ? cluster_cta_rank() : 0u;
    const uint32_t half = rank % CG;      // this CTA's 128-row half of the pair's tile
    const uint32_t pair = rank / CG;      // the pair of the cluster (0 when MC = 1)
    const uint32_t leader = rank - half;  // the pair's even CTA: its barriers count both CTAs' bytes
    const int cluster_id = static_cast<int>(blockIdx.x) / CS;
    const int num_clusters = static_cast<int>(gridDim.x) / CS;

    const uint32_t staging_off = stages * Cfg::STAGE_BYTES;
    const uint32_t bar_off = staging_off + 4u * p.staging_bufs * p.staging_bytes;
    const uint32_t bar0 = base + bar_off;
    auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
    auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (stages + s); };
    auto tfull_bar = [&](uint32_t b) { return bar0 + 8u * (2u * stages + b); };
    auto tempty_bar = [&](uint32_t b) { return bar0 + 8u * (2u * stages + 2u + b); };
    const uint32_t done_bar = bar0 + 8u * (2u * stages + 4u);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + bar_off + 8u * (2u * stages + 5u));

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < stages; ++s) {
            mbar_init(full_bar(s), 1);    // producer's arrive.expect_tx (+ bytes of both CTAs)
            mbar_init(empty_bar(s), MC);  // one tcgen05.commit of every pair that reads or shares the slot
        }
        for (uint32_t b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);             // one tcgen05.commit
            mbar_init(tempty_bar(b), (blockDim.x / 32u - EPI_WARP0) * CG);   // every epilogue warp of the tile
        }
        mbar_init(done_bar, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(tmem_holder), TMEM_COLS);
        tmem_relinquish<CG>();
    }
    tc_fence_before_sync();
    if constexpr (CS > 1)
        cluster_sync();
    else
        __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_holder);
    // Launched with programmatic stream serialisation: the setup above may run
    // while the previous grid on the stream drains. Nothing in global memory is
    // read or written before that grid has completed.
    grid_dependency_wait();
    grid_launch_dependents();
    if (p.trace != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
        p.trace[0] = global_timer_ns();
        p.trace[1] = static_cast<unsigned long long>(clock64());
    }

    WaitCtx w{p.timeout_ns, p.launch_id, p.status, false};
    // This unit's jobs: whole tiles and, with stream-K, at most one writer and
    // one owner segment. Every role walks the same list.
    const UnitSchedule sch(cluster_id, num_clusters, p.num_tiles, p.num_k_blocks, p.sk_tiles);
    const int num_jobs = sch.num_jobs();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensor_map(&tmap_a);
            prefetch_tensor_map(&tmap_b);
            if constexpr (Cfg::SCALED) {
                prefetch_tensor_map(&tmap_sfa);
                prefetch_tensor_map(&tmap_sfb);
            }
            uint32_t s = 0, ph = 0, pend_mask = 0, pend_par = 0;
            // self-test: the k-block of the first job whose stage is never filled (-1: none)
            const int withhold = cluster_id == 0 ? p.withhold_kb : -1;
            for (int i = 0; i < num_jobs; ++i) {
                const Job jb = sch.job(i);
                int m_blk, n_blk;
                tile_coords(p, jb.tile, m_blk, n_blk);
                n_blk = n_blk * MC + static_cast<int>(pair);   // MC = 2: the pair's tile of the two
                const int a_row = m_blk * (BLOCK_M_CTA * CG) + static_cast<int>(half) * BLOCK_M_CTA;
                const int b_off = n_blk * BN + static_cast<int>(half) * Cfg::BN_CTA;
                for (int kb = jb.kb0; kb < jb.kb1; ++kb) {
                    wait_bounded<CG == 2>(w, empty_bar(s), ph ^ 1u, SITE_PRODUCER_EMPTY);
                    if (!w.aborted && !(i == 0 && kb == withhold)) {
                        const uint32_t a_dst = base + s * Cfg::STAGE_BYTES;
                        const uint32_t b_dst = a_dst + Cfg::A_BYTES;
                        const int x0 = kb * KS * Cfg::SLAB_X;
                        if constexpr (CG == 1) {
                            const uint32_t bar = full_bar(s);
                            mbar_arrive_expect_tx(bar, Cfg::STAGE_TX);
#pragma unroll
                            for (int j = 0; j < KS; ++j) {
                                const int kj = x0 + j * Cfg::SLAB_X;
                                tma_load_2d(a_dst + j * Cfg::A_SLAB, &tmap_a, bar, kj, a_row);
                                const uint32_t bj = b_dst + j * Cfg::B_SLAB;
                                if (KIND != KIND_F16 || !p.b_mn_major)
                                    tma_load_2d(bj, &tmap_b, bar, kj, b_off);
                                else
                                    for (int i = 0; i < Cfg::BN_CTA / 64; ++i)
                                        tma_load_2d(bj + i * 8192u, &tmap_b, bar, b_off + 64 * i, kj);
                            }
                            if constexpr (Cfg::SCALED) {
                                // this stage's scale atoms of the CTA's A and B row blocks
                                tma_load_2d(a_dst + Cfg::AB_BYTES, &tmap_sfa, bar, 0,
                                            sf_atom_row(a_row / BLOCK_M_CTA, kb, p.num_k_blocks, Cfg::SF_GROUPS));
                                tma_load_2d(a_dst + Cfg::AB_BYTES + Cfg::SFA_BYTES, &tmap_sfb, bar, 0,
                                            sf_atom_row(n_blk, kb, p.num_k_blocks, Cfg::SF_GROUPS * Cfg::SFB_ATOMS));
                            }
                        } else {
                            // both CTAs' boxes complete on the pair leader's full barrier
                            const uint32_t bar = map_to_cta(full_bar(s), leader);
                            if (half == 0)
                                mbar_arrive_expect_tx(full_bar(s), 2u * Cfg::STAGE_TX);
#pragma unroll
                            for (int j = 0; j < KS; ++j) {
                                const int kj = x0 + j * Cfg::SLAB_X;
                                if constexpr (MC == 1) {
                                    tma_load_2d_pair(a_dst + j * Cfg::A_SLAB, &tmap_a, bar, kj, a_row);
                                } else {
                                    // this CTA's 64-row share of the half's A rows, into the same
                                    // offset of both pairs' CTAs of this half (the A map's box is 64 rows)
                                    const uint16_t mask = static_cast<uint16_t>((1u << half) | (1u << (half + CG)));
                                    tma_load_2d_pair_mc(a_dst + j * Cfg::A_SLAB + pair * (Cfg::A_SLAB / 2), &tmap_a, bar,
                                                        kj, a_row + static_cast<int>(pair) * (BLOCK_M_CTA / 2), mask);
                                }
                                const uint32_t bj = b_dst + j * Cfg::B_SLAB;
                                if (KIND != KIND_F16 || !p.b_mn_major)
                                    tma_load_2d_pair(bj, &tmap_b, bar, kj, b_off);
                                else
                                    for (int i = 0; i < Cfg::BN_CTA / 64; ++i)
                                        tma_load_2d_pair(bj + i * 8192u, &tmap_b, bar, b_off + 64 * i, kj);
                            }
                            if constexpr (Cfg::SCALED) {
                                // both CTAs load the B scales of the whole tile width
                                tma_load_2d_pair(a_dst + Cfg::AB_BYTES, &tmap_sfa, bar, 0,
                                                 sf_atom_row(a_row / BLOCK_M_CTA, kb, p.num_k_blocks, Cfg::SF_GROUPS));
                                tma_load_2d_pair(a_dst + Cfg::AB_BYTES + Cfg::SFA_BYTES, &tmap_sfb, bar, 0,
                                                 sf_atom_row(n_blk, kb, p.num_k_blocks,
                                                             Cfg::SF_GROUPS * Cfg::SFB_ATOMS));
                            }
                        }
                        pend_mask |= 1u << s;
                        pend_par = (pend_par & ~(1u << s)) | (ph << s);
                    }
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // Leave no bulk copy into shared memory in flight: wait for the last
            // fill of every slot (the peer CTA's copies, and with MC = 2 the other
            // pair's shares of A, land on these barriers too).
            if (CG == 1 || half == 0)
                for (uint32_t s2 = 0; s2 < stages; ++s2)
                    if ((pend_mask >> s2) & 1u)
                        wait_drain<CG == 2>(full_bar(s2), (pend_par >> s2) & 1u, w.limit_ns, w.id, w.status,
                                           SITE_PRODUCER_DRAIN);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp walks the job list and waits; one elected lane issues
        // each product, copy and commit.
        if (CG == 1 || half == 0) {
            auto sync_abort = [&]() {
                __syncwarp();
                w.aborted = __any_sync(0xffffffffu, w.aborted);
            };
            // 8-bit and 4-bit operands are K-major only (the host rejects MN-major B for them).
            const bool b_mn = KIND == KIND_F16 && p.b_mn_major != 0;
            // K-major: rows of 128 B in 8-row groups 1024 B apart; one MMA step = 32 B.
            // MN-major (16-bit): 64-wide N atoms 8192 B apart (LBO), 8-row K groups
            // 1024 B apart (SBO); one K=16 step = 16 rows = 2048 B.
            const uint32_t b_lbo = b_mn ? 8192u : 16u;
            const uint32_t b_step = b_mn ? (2048u >> 4) : (32u >> 4);
            uint32_t s = 0, ph = 0, acc = 0, acc_ph = 0, sf_sel = 0;
            for (int i = 0; i < num_jobs; ++i) {
                const Job jb = sch.job(i);
                wait_bounded<CG == 2>(w, tempty_bar(acc), acc_ph ^ 1u, SITE_MMA_TMEM_EMPTY);
                sync_abort();
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * ACC_STRIDE;
                for (int kb = jb.kb0; kb < jb.kb1; ++kb) {
                    wait_bounded<CG == 2>(w, full_bar(s), ph, SITE_MMA_FULL);
                    sync_abort();
                    tc_fence_after_sync();
                    if (!w.aborted) {
                        const uint32_t a_addr = base + s * Cfg::STAGE_BYTES;
#pragma unroll
                        for (int j = 0; j < KS; ++j) {
                            // a slab wholly past K holds only TMA zero fill: skip its MMAs
                            if (j > 0 && kb * Cfg::STAGE_K + j * Cfg::SLAB_K >= p.K)
                                break;
                            // this slab's scale atoms (its groups of the stage's A atoms, then of
                            // its B atoms) into the next scale buffer; later MMAs of the issuing
                            // lane see them
                            const uint32_t sf_a = tmem_base + Cfg::SF_COL + 256u * sf_sel;
                            const uint32_t sf_b = sf_a + Cfg::SF_B_OFF;
                            if constexpr (Cfg::SCALED) {
                                sf_sel ^= 1u;
                                const uint32_t src_a = a_addr + Cfg::AB_BYTES, src_b = src_a + Cfg::SFA_BYTES;
#pragma unroll
                                for (int gi = 0; gi < Cfg::SLAB_SF_GROUPS; ++gi) {
                                    const int gs = j * Cfg::SLAB_SF_GROUPS + gi;
                                    tmem_cp_32x128b_warpx4<CG>(sf_a + 4u * gi,
                                                               smem_desc_plain(src_a + gs * SF_ATOM_BYTES, 128u));
#pragma unroll
                                    for (int at = 0; at < Cfg::SFB_ATOMS; ++at)
                                        tmem_cp_32x128b_warpx4<CG>(
                                            sf_b + 4u * (gi * Cfg::SFB_ATOMS + at),
                                            smem_desc_plain(src_b + (gs * Cfg::SFB_ATOMS + at) * SF_ATOM_BYTES, 128u));
                                }
                            }
                            const uint64_t a_desc = smem_desc_sw128(a_addr + j * Cfg::A_SLAB, 16u, 1024u);
                            const uint64_t b_desc = smem_desc_sw128(a_addr + Cfg::A_BYTES + j * Cfg::B_SLAB,
                                                                    b_lbo, 1024u);
#pragma unroll
                            for (uint32_t k = 0; k < SLAB_MMAS; ++k) {
                                const uint32_t acc_in = (kb > jb.kb0 || j > 0 || k > 0) ? 1u : 0u;
                                if constexpr (Cfg::SCALED) {
                                    // first 32-K block of this MMA within the slab: its scales
                                    // are byte blk % 4 of the slab's atom blk / 4 (4 TMEM columns)
                                    const uint32_t blk = k * Cfg::MMA_SF_BLOCKS;
                                    mma_scaled<CG, KIND>(d_tmem, a_desc + 2u * k, b_desc + b_step * k,
                                                         p.idesc | mx_sf_id(blk % 4u), sf_a + 4u * (blk / 4u),
                                                         sf_b + 4u * Cfg::SFB_ATOMS * (blk / 4u), acc_in);
                                } else {
                                    mma<CG, KIND>(d_tmem, a_desc + 2u * k, b_desc + b_step * k, p.idesc, acc_in);
                                }
                            }
                        }
                        if constexpr (CG == 1)
                            mma_commit(empty_bar(s));
                        else
                            mma_commit_pair(empty_bar(s), static_cast<uint16_t>((1u << CS) - 1u));   // every CTA of the cluster
                    }
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!w.aborted) {
                    if constexpr (CG == 1)
                        mma_commit(tfull_bar(acc));
                    else
                        mma_commit_pair(tfull_bar(acc), static_cast<uint16_t>(3u << leader));    // this pair
                }
                if (++acc == 2) {
                    acc = 0;
                    acc_ph ^= 1u;
                }
            }
            // No MMA may still be writing TMEM when it is freed.
            if constexpr (CG == 1)
                mma_commit(done_bar);
            else
                mma_commit_pair(done_bar, static_cast<uint16_t>(1u << leader));
            wait_drain<false>(done_bar, 0, w.limit_ns, w.id, w.status, SITE_MMA_DONE);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const uint32_t ew = warp - EPI_WARP0;                       // 0 .. epilogue warps - 1
        const uint32_t per_quarter = (blockDim.x / 32u - EPI_WARP0) / 4u;   // 1 or 2 warps
        const uint32_t quarter = warp & 3u;      // the TMEM lane quarter this warp may access
        // The quarter's warps split its staging buffers and its chunks: with two,
        // warps 2-5 take chunks [0, C_SPLIT) and warps 6-9 the rest.
        const uint32_t wbufs = p.staging_bufs / per_quarter;
        const uint32_t staging = base + staging_off + ew * wbufs * p.staging_bytes;
        const uint64_t c_policy = l2_evict_first_policy();   // C is written once: keep A and B in L2
        constexpr int CHUNKS = BN / EPI_COLS;
        constexpr int C_SPLIT = (CHUNKS + 1) / 2;
        const int c_begin = (per_quarter == 2u && ew >= 4u) ? C_SPLIT : 0;
        const int c_end = (per_quarter == 2u && ew < 4u) ? C_SPLIT : CHUNKS;
        // Stream-K partial slot of CTA `cta`, this warp's 32 rows, chunk c: 32 lanes x 8 float4,
        // laid out so that each float4 store or load of the warp covers 512 contiguous bytes.
        auto partial_chunk = [&](int cta, int c) {
            return p.partials + ((static_cast<size_t>(cta) * 4u + quarter) * CHUNKS + c) * 256u + lane;
        };
        uint32_t acc = 0, acc_ph = 0, sb = 0;
        for (int i = 0; i < num_jobs; ++i) {
            const Job jb = sch.job(i);
            int m_blk, n_blk;
            tile_coords(p, jb.tile, m_blk, n_blk);
            n_blk = n_blk * MC + static_cast<int>(pair);
            wait_bounded<CG == 2>(w, tfull_bar(acc), acc_ph, SITE_EPI_TMEM_FULL);
            // An owner needs every writer's partial for its rows first. The
            // writers did their segments at the start of their work lists.
            int w_first = cluster_id;
            // Which of the units cluster_id - 1, cluster_id - 2, ... (down to w_first)
            // left a partial: worked out once per owner job (each test takes two
            // 64-bit divisions), bit i for unit cluster_id - 1 - i; beyond 32 units
            // back (tiny problems spread over many units) the test is redone per use.
            uint32_t wmask = 0;
            auto wrote = [&](int u) {
                const int i = cluster_id - 1 - u;
                return i < 32 ? ((wmask >> i) & 1u) != 0 : sch.has_range(u);
            };
            if (jb.kind == JOB_OWNER && !w.aborted) {
                w_first = sch.first_writer();
                for (int i = 0; i < 32 && cluster_id - 1 - i >= w_first; ++i)
                    if (sch.has_range(cluster_id - 1 - i))
                        wmask |= 1u << i;
                if (lane == 0)
                    for (int v = cluster_id - 1; v >= w_first; --v)
                        if (wrote(v) &&
                            !wait_flag_bounded(w, &p.flags[(static_cast<size_t>(v) * CS + rank) * EPI_WARPS_MAX + ew],
                                               SITE_EPI_PARTIAL))
                            break;
                w.aborted = __shfl_sync(0xffffffffu, w.aborted ? 1 : 0, 0) != 0;
                __syncwarp();   // lane 0's acquire loads come before every lane's partial reads
            }
            const bool skip = __any_sync(0xffffffffu, w.aborted);   // warp-uniform
            w.aborted = skip;
            tc_fence_after_sync();
            const int row0 = m_blk * (BLOCK_M_CTA * CG) + static_cast<int>(half) * BLOCK_M_CTA +
                             static_cast<int>(quarter) * 32;
            const int col0 = n_blk * BN;
            const uint32_t t_row = tmem_base + ((quarter * 32u) << 16) + acc * ACC_STRIDE;
#pragma unroll 1
            for (int c = c_begin; c < c_end; ++c) {
                uint32_t v[32];
                if (!skip) {
                    tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * EPI_COLS), v);
                    tmem_ld_wait_regs(v);
                }
                if (c == c_end - 1 && i + 1 < num_jobs) {
                    // accumulator fully read: hand it back to the MMA issuer (after this
                    // unit's last tile nothing waits for it; teardown's cluster barrier
                    // orders the reads before TMEM is freed)
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0 && !skip) {
                        if constexpr (CG == 1)
                            mbar_arrive_local(tempty_bar(acc));
                        else
                            mbar_arrive_cluster(map_to_cta(tempty_bar(acc), leader));
                    }
                }
                const int gcol = col0 + c * EPI_COLS;
                if (skip || gcol >= p.N)
                    continue;
                if (jb.kind == JOB_WRITER) {
                    float4 *dst = partial_chunk(static_cast<int>(blockIdx.x), c);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4)
                        __stcg(dst + 32 * j4, make_float4(__uint_as_float(v[4 * j4]), __uint_as_float(v[4 * j4 + 1]),
                                                          __uint_as_float(v[4 * j4 + 2]),
                                                          __uint_as_float(v[4 * j4 + 3])));
                    continue;
                }
                if (jb.kind == JOB_OWNER) {
                    // add the writers' partial sums, nearest k-range first
                    for (int u = cluster_id - 1; u >= w_first; --u) {
                        if (!wrote(u))
                            continue;
                        const float4 *src = partial_chunk(u * CS + static_cast<int>(rank), c);
#pragma unroll
                        for (int j4 = 0; j4 < 8; ++j4) {
                            const float4 x = __ldcg(src + 32 * j4);
                            v[4 * j4] = __float_as_uint(__uint_as_float(v[4 * j4]) + x.x);
                            v[4 * j4 + 1] = __float_as_uint(__uint_as_float(v[4 * j4 + 1]) + x.y);
                            v[4 * j4 + 2] = __float_as_uint(__uint_as_float(v[4 * j4 + 2]) + x.z);
                            v[4 * j4 + 3] = __float_as_uint(__uint_as_float(v[4 * j4 + 3]) + x.w);
                        }
                    }
                }
                if (p.direct_store) {
                    store_row_direct(p, row0 + static_cast<int>(lane), gcol, v);
                    continue;
                }
                const uint32_t buf = staging + sb * p.staging_bytes;
                if (lane == 0) {
                    // the store that last used `buf` has read it
                    if (wbufs == 4)
                        bulk_wait_group_read<3>();
                    else if (wbufs == 2)
                        bulk_wait_group_read<1>();
                    else
                        bulk_wait_group_read<0>();
                }
                __syncwarp();
                stage_row(buf, lane, v, p.out_dtype);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && row0 < p.M) {
                    tma_store_2d_hint(&tmap_c, buf, gcol, row0, c_policy);
                    bulk_commit_group();
                }
                sb = (sb + 1u) & (wbufs - 1u);
            }
            if (jb.kind == JOB_WRITER && !skip) {
                // publish: every lane's partial stores, then the flag
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    st_release_gpu(&p.flags[static_cast<size_t>(blockIdx.x) * EPI_WARPS_MAX + ew], p.launch_id);
                }
            }
            if (jb.kind == JOB_OWNER && !skip) {
                // Every writer's partial has been read: clear the flags this owner
                // consumed (each has exactly one reader). A replay of the same
                // launch (a captured CUDA graph keeps its launch id and its
                // workspace) then cannot mistake the last replay's flags for new ones.
                __syncwarp();
                if (lane == 0)
                    for (int u = cluster_id - 1; u >= w_first; --u)
                        if (wrote(u))
                            p.flags[(static_cast<size_t>(u) * CS + rank) * EPI_WARPS_MAX + ew] = 0ull;
            }
            if (++acc == 2) {
                acc = 0;
                acc_ph ^= 1u;
            }
        }
        if (lane == 0)
            bulk_wait_group_all();
    }

    // ---------------------------------------------------------------- teardown
    __syncwarp();
    tc_fence_before_sync();
    if constexpr (CS > 1)
        cluster_sync();   // no other CTA of the cluster touches this CTA's barriers, ring or TMEM
    else
        __syncthreads();
    if (p.trace != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
        p.trace[2] = global_timer_ns();
        p.trace[3] = static_cast<unsigned long long>(clock64());
    }
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<CG>(tmem_base, TMEM_COLS);
    }
}

// One CTA waits, through the same bounded wait, on a barrier that nothing
// arrives at; it must record SITE_SELFTEST and return.
static __global__ void wait_selftest_kernel(uint64_t timeout_ns, unsigned long long launch_id,
                                     unsigned long long *status)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        WaitCtx w{timeout_ns, launch_id, status, false};
        wait_bounded<false>(w, smem_u32(&bar), 0, SITE_SELFTEST);
    }
}

// Repack E8M0 scales (rows x n_blocks bytes, row-major: one byte per 32 K)
// into the kernel's atoms: row blocks of R rows, and per row block and ring
// stage `groups` groups of 4 blocks, each group `atoms` atoms of 128 rows
// (see SF_ATOM_BYTES). Missing rows and blocks are zero. out has row_blocks x
// stages x groups x atoms x 32 rows of 16 bytes; each thread writes one such
// row. Consecutive threads take consecutive groups of 4 blocks of the same
// scale rows, so the reads (4-byte words when `words` is set: the scale
// rows and base are 4-byte aligned) are coalesced.
static __global__ void pack_scales_kernel(const uint8_t *__restrict__ sf, uint8_t *__restrict__ out, int64_t rows,
                                          int64_t n_blocks, int R, int64_t row_blocks, int64_t stages, int groups,
                                          int atoms, int words)
{
    const int64_t sg_count = stages * groups;   // groups of 4 blocks along K
    const int64_t total = row_blocks * atoms * SF_ATOM_ROWS * sg_count;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t sg = i % sg_count;
        int64_t t = i / sg_count;
        const int m32 = static_cast<int>(t % SF_ATOM_ROWS);
        t /= SF_ATOM_ROWS;
        const int a = static_cast<int>(t % atoms);
        const int64_t rb = t / atoms;
        const int64_t blk0 = sg * 4;
        uint32_t w[4] = {0, 0, 0, 0};
        for (int m4 = 0; m4 < 4; ++m4) {
            const int m = a * 128 + m4 * SF_ATOM_ROWS + m32;
            const int64_t row = rb * R + m;
            if (m >= R || row >= rows)
                continue;
            const uint8_t *src = sf + row * n_blocks + blk0;
            if (words && blk0 + 4 <= n_blocks) {
                w[m4] = *reinterpret_cast<const uint32_t *>(src);
            } else {
                for (int k4 = 0; k4 < 4; ++k4)
                    if (blk0 + k4 < n_blocks)
                        w[m4] |= static_cast<uint32_t>(src[k4]) << (8 * k4);
            }
        }
        const int64_t st = sg / groups, g = sg % groups;
        const int64_t o = (((rb * stages + st) * groups + g) * atoms + a) * SF_ATOM_ROWS + m32;
        reinterpret_cast<uint4 *>(out)[o] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Copy `rows` rows of `row_bytes` bytes each (source pitch row_bytes, densely
// packed) into a buffer whose row pitch `dst_pitch` is a multiple of 16 bytes
// (the library pads to 128) and whose base is 256-byte aligned, so the TMA
// engine can describe it. The
// bytes past row_bytes in each destination row are not written: the tensor
// map keeps the logical width, and TMA zero-fills past it.
//
// V is the widest word that divides the source base, row_bytes and hence
// every source row start (4 for a 4100-byte BF16 row), so every access is an
// aligned V-byte word inside the source or destination row. Each warp copies
// whole rows (grid-stride over rows): its lanes take consecutive words, and
// every lane keeps UNROLL loads in flight before it stores them (64 bytes per
// lane: 2 KB per warp, ~48 KB per SM at 3 blocks of 8 warps), enough to keep
// HBM busy although the words are small.
//
// Launched in plain stream order, so the previous grid has completed when it
// starts (its griddepcontrol.wait returns at once then, and guards a launch
// that lets it start early). It lets the GEMM that follows launch at once; that
// GEMM waits for this grid to complete before it reads.
template <int V>
__global__ void __launch_bounds__(256) realign_rows_kernel(const uint8_t *__restrict__ src,
                                                           uint8_t *__restrict__ dst, int64_t rows,
                                                           int64_t row_bytes, int64_t dst_pitch)
{
    using W = typename std::conditional<
        V == 16, uint4,
        typename std::conditional<V == 8, uint2,
                                  typename std::conditional<V == 4, uint32_t,
                                                            typename std::conditional<V == 2, uint16_t,
                                                                                      uint8_t>::type>::type>::type>::type;
    grid_dependency_wait();
    grid_launch_dependents();
    constexpr int UNROLL = V >= 4 ? 64 / V : 32;
    const int64_t words = row_bytes / V;
    const int lane = static_cast<int>(threadIdx.x % 32u);
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32u);
    for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x / 32u) + threadIdx.x / 32u; r < rows; r += warps) {
        const W *s = reinterpret_cast<const W *>(src + r * row_bytes);
        W *d = reinterpret_cast<W *>(dst + r * dst_pitch);
        for (int64_t i0 = lane; i0 < words; i0 += UNROLL * 32) {
            W v[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u)
                if (i0 + u * 32 < words)
                    v[u] = __ldg(s + i0 + u * 32);
#pragma unroll
            for (int u = 0; u < UNROLL; ++u)
                if (i0 + u * 32 < words)
                    d[i0 + u * 32] = v[u];
        }
    }
}

} // namespace dtg
