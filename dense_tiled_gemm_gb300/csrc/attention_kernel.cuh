// attention_kernel.cuh: attention forward, O = softmax(scale * Q K^T) V, for sm_103a.
//
// "Two Waves, One Stage Apart" (section "Beyond GEMM: FlashAttention")
// describes the FlashAttention inner loop: QK and PV products alternate with
// an online softmax over key/value blocks, and the matrix work of one wave
// group overlaps the softmax of the other. Here one CTA holds two query tiles
// (A: rows 0-127, B: rows 128-255 of its 256) with a softmax warp group each,
// so that while one group turns its scores into probabilities, the tensor
// core runs the other group's products:
//
//   warp 0     producer: one thread loads both Q tiles once, then K and V
//              blocks into two-slot rings (TMA, 128-byte swizzle);
//   warp 1     MMA issuer (the whole warp; one elected lane issues), per key
//              block j:
//                PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1)
//              (S_g = Q_g K^T into tile g's TMEM score buffer, O_g += P_g V
//              into tile g's FP32 accumulator, P_g read from TMEM); owns TMEM;
//   warps 2-5  softmax group A, warps 6-9 group B: one query row per thread.
//              Read S_g(j), keep the running row maximum m and sum l (base-2
//              exponent), and write P_g = exp2(s - m), rounded to the operand
//              type, over the first half of the score buffer it came from; at
//              the end divide by l and store O and the row log-sum-exp. The
//              maximum used for P is raised (and O and l rescaled by
//              exp2(m_old - m_new)) only when a row's maximum grows by more
//              than RESCALE_LOG2 = 8: until then P <= 2^8, which the operand
//              types hold, and O and l stay consistently scaled; l sums the
//              probabilities in FP32 before their rounding.
//
// The tensor core runs a CTA's products in issue order, so QK_g(j+1), issued
// after PV_g(j), overwrites P_g(j) only after PV_g(j) has read it, and the
// commit that signals S_g(j+1) also covers PV_g(j): a softmax group that holds
// S_g(j+1) may rescale O_g. The kernel is persistent: one CTA per SM walks
// row blocks (256 query rows of one head), one per round of gridDim.x; the
// K/V ring and every barrier phase carry over from one row block to the next,
// so the next block's Q load and first QK products overlap the current
// block's last softmax and its output. Blocks are 128 keys; the head
// dimension is 128.
// TMEM: score buffers at columns 0 (A) and 128 (B), accumulators at 256 (A)
// and 384 (B). Masked keys (past Lk, or after the causal diagonal, which is
// aligned to the last query row) score -inf. Every wait is bounded as in the
// GEMM kernel: past the limit a thread records the site and stops issuing
// work and signals.
#pragma once

#include "gemm_kernel.cuh"

namespace dtg {

constexpr int ATT_BM = 128;                       // query rows per tile
constexpr int ATT_TILES = 2;                      // query tiles per CTA
constexpr int ATT_ROWS = ATT_BM * ATT_TILES;      // query rows per CTA
constexpr int ATT_BN = 128;                       // keys per block
constexpr int ATT_D = 128;                        // head dimension
constexpr int ATT_TILE = ATT_BM * ATT_D * 2;      // 32 KB: one Q, K or V tile
constexpr int ATT_SLAB = ATT_TILE / 2;            // 64 columns of 16-bit data, 128-byte rows
constexpr int ATT_STAGES = 2;                     // K and V ring slots
constexpr uint32_t ATT_TMEM_COLS = 512;
constexpr uint32_t ATT_O_COL = 256;               // accumulator of tile g at 256 + 128 g
constexpr int ATT_THREADS = 64 + 32 * 4 * ATT_TILES;   // producer, MMA, 4 softmax warps per tile
constexpr float RESCALE_LOG2 = 8.0f;              // lazy rescaling threshold (base-2 exponent)

// shared memory: Q[2] | K[2] | V[2] | barriers | TMEM address
constexpr uint32_t ATT_Q_OFF = 0;
constexpr uint32_t ATT_K_OFF = ATT_TILES * ATT_TILE;
constexpr uint32_t ATT_V_OFF = ATT_K_OFF + ATT_STAGES * ATT_TILE;
constexpr uint32_t ATT_BAR_OFF = ATT_V_OFF + ATT_STAGES * ATT_TILE;
constexpr uint32_t ATT_NUM_BARS = 16;
constexpr uint32_t ATT_SMEM = ATT_BAR_OFF + ATT_NUM_BARS * 8 + 16;

enum : uint32_t {
    SITE_ATT_Q = 0x410,
    SITE_ATT_K_EMPTY = 0x411,
    SITE_ATT_V_EMPTY = 0x412,
    SITE_ATT_K_FULL = 0x413,
    SITE_ATT_P_FULL = 0x415,
    SITE_ATT_V_FULL = 0x416,
    SITE_ATT_S_FULL = 0x417,
    SITE_ATT_DRAIN = 0x419,
    SITE_ATT_DONE = 0x41A,
    SITE_ATT_Q_EMPTY = 0x41B,
};

struct AttParams {
    int32_t Lq, Lk;
    int32_t BH;                // batch x heads
    int32_t nq;                // row blocks of 256 per head
    uint32_t causal;
    uint32_t bf16;             // operand and output type: 1 BF16, 0 FP16
    float scale_log2;          // score scale times log2(e)
    uint32_t idesc_qk, idesc_pv;
    void *O;                   // [B][H][Lq][128], the operand type
    float *LSE;                // [B][H][Lq] natural-log row log-sum-exp, or null
    uint64_t timeout_ns;
    unsigned long long launch_id;
    unsigned long long *status;
};

// KV blocks the rows [q0, q0 + rows) need: all ceil(Lk / 128), or, when
// causal, those up to the block holding the last key their last row may see.
__host__ __device__ inline int att_num_blocks(int q0, int rows, int Lq, int Lk, bool causal)
{
    int n = (Lk + ATT_BN - 1) / ATT_BN;
    if (causal) {
        const int last_row = min(q0 + rows, Lq) - 1;
        const int last_key = last_row + (Lk - Lq);
        n = last_key < 0 ? 0 : min(n, last_key / ATT_BN + 1);
    }
    return n;
}

// 2^x by the PTX ex2 instruction (approximate, flushes subnormals; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction (three-input form, sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float y;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
    return y;
}

// Packed FP32 pairs (Blackwell f32x2 arithmetic): one instruction for two lanes of work.
__device__ __forceinline__ void ffma2(float &x0, float &x1, float a0, float a1, float b, float c)
{
    asm("{\n\t.reg .b64 pa, pb, pc, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "mov.b64 pb, {%4, %4};\n\t"
        "mov.b64 pc, {%5, %5};\n\t"
        "fma.rn.f32x2 pd, pa, pb, pc;\n\t"
        "mov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(x0), "=f"(x1)
        : "f"(a0), "f"(a1), "f"(b), "f"(c));
}

__device__ __forceinline__ void fadd2(float &s0, float &s1, float a0, float a1)
{
    asm("{\n\t.reg .b64 ps, pa;\n\t"
        "mov.b64 ps, {%0, %1};\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "add.rn.f32x2 ps, ps, pa;\n\t"
        "mov.b64 {%0, %1}, ps;\n\t}"
        : "+f"(s0), "+f"(s1)
        : "f"(a0), "f"(a1));
}

__device__ __forceinline__ uint32_t pack2_rn(float a, float b, bool bf16)
{
    if (bf16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&v);
    }
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

__global__ void __launch_bounds__(ATT_THREADS, 1)
attention_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const AttParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw);
    if (base & 1023u) {
        if (threadIdx.x == 0)
            record_timeout(p.status, p.launch_id, SITE_SMEM_ALIGN);
        return;
    }
    const uint32_t warp = threadIdx.x / 32u, lane = threadIdx.x % 32u;
    const int64_t num_items = static_cast<int64_t>(p.nq) * p.BH;
    // Row block L of the launch. Causal row blocks differ in work (a block
    // needs the key blocks up to its diagonal): they are taken in order of
    // decreasing work, longest first, so that the CTAs finish together.
    // Otherwise consecutive items are the row blocks of one head, which run
    // side by side and share its K and V in L2.
    // This CTA's k-th row block: rounds of gridDim.x row blocks, taken in
    // alternate directions (c, then gridDim.x - 1 - c, ...), so that under the
    // causal mask every CTA gets a heavy and a light block in turn. Returns
    // an index past the end when the last, partial round has none for it.
    auto item_index = [&](int64_t k) -> int64_t {
        const int64_t c = blockIdx.x, G = gridDim.x;
        return k * G + ((k & 1) ? G - 1 - c : c);
    };
    auto item = [&](int64_t L, int &qt, int &bh) {
        if (p.causal) {
            qt = p.nq - 1 - static_cast<int>(L / p.BH);
            bh = static_cast<int>(L % p.BH);
        } else {
            qt = static_cast<int>(L % p.nq);
            bh = static_cast<int>(L / p.nq);
        }
    };

    const uint32_t bar0 = base + ATT_BAR_OFF;
    const uint32_t q_full = bar0;
    auto k_full = [&](uint32_t s) { return bar0 + 8u * (1 + s); };
    auto k_empty = [&](uint32_t s) { return bar0 + 8u * (3 + s); };
    auto v_full = [&](uint32_t s) { return bar0 + 8u * (5 + s); };
    auto v_empty = [&](uint32_t s) { return bar0 + 8u * (7 + s); };
    auto s_full = [&](uint32_t g) { return bar0 + 8u * (9 + g); };
    auto p_full = [&](uint32_t g) { return bar0 + 8u * (11 + g); };
    auto done = [&](uint32_t g) { return bar0 + 8u * (13 + g); };   // tile g's last product of a row block
    const uint32_t q_empty = bar0 + 8u * 15;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem_raw + ATT_BAR_OFF + ATT_NUM_BARS * 8);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (uint32_t s = 0; s < ATT_STAGES; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), 1);
            mbar_init(v_full(s), 1);
            mbar_init(v_empty(s), 1);
        }
        for (uint32_t g = 0; g < ATT_TILES; ++g) {
            mbar_init(s_full(g), 1);    // one tcgen05.commit
            mbar_init(p_full(g), 4);    // the group's four warps
            mbar_init(done(g), 1);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(tmem_holder), ATT_TMEM_COLS);
        tmem_relinquish<1>();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_holder);
    grid_dependency_wait();
    grid_launch_dependents();

    WaitCtx w{p.timeout_ns, p.launch_id, p.status, false};

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensor_map(&tmap_q);
            prefetch_tensor_map(&tmap_k);
            prefetch_tensor_map(&tmap_v);
            uint32_t rb = 0, qi = 0, q_loads = 0;   // ring blocks, row blocks and Q loads so far
            uint32_t k_pend = 0, v_pend = 0, k_par = 0, v_par = 0;
            for (int64_t k = 0; k * gridDim.x < num_items; ++k) {
                const int64_t L = item_index(k);
                if (L >= num_items)
                    continue;
                int qt, bh;
                item(L, qt, bh);
                const int q0 = qt * ATT_ROWS;
                const int nkv = att_num_blocks(q0, ATT_ROWS, p.Lq, p.Lk, p.causal != 0);
                if (nkv == 0)
                    continue;
                // Q of both tiles, once the previous row block's last QK product is done with it
                if (qi > 0)
                    wait_bounded<false>(w, q_empty, (qi - 1) & 1, SITE_ATT_Q_EMPTY);
                if (!w.aborted) {
                    mbar_arrive_expect_tx(q_full, ATT_TILES * ATT_TILE);
                    for (int g = 0; g < ATT_TILES; ++g) {
                        const uint32_t dst = base + ATT_Q_OFF + g * ATT_TILE;
                        tma_load_3d(dst, &tmap_q, q_full, 0, q0 + g * ATT_BM, bh);
                        tma_load_3d(dst + ATT_SLAB, &tmap_q, q_full, 64, q0 + g * ATT_BM, bh);
                    }
                    ++q_loads;
                }
                ++qi;
                for (int j = 0; j < nkv; ++j, ++rb) {
                    const uint32_t s = rb % ATT_STAGES, ph = (rb / ATT_STAGES) & 1;
                    const int key0 = j * ATT_BN;
                    wait_bounded<false>(w, k_empty(s), ph ^ 1u, SITE_ATT_K_EMPTY);
                    if (!w.aborted) {
                        const uint32_t dst = base + ATT_K_OFF + s * ATT_TILE;
                        mbar_arrive_expect_tx(k_full(s), ATT_TILE);
                        tma_load_3d(dst, &tmap_k, k_full(s), 0, key0, bh);
                        tma_load_3d(dst + ATT_SLAB, &tmap_k, k_full(s), 64, key0, bh);
                        k_pend |= 1u << s;
                        k_par = (k_par & ~(1u << s)) | (ph << s);
                    }
                    wait_bounded<false>(w, v_empty(s), ph ^ 1u, SITE_ATT_V_EMPTY);
                    if (!w.aborted) {
                        // V serves as an N-contiguous B operand: per 64-key slab, two 64-wide d atoms
                        const uint32_t dst = base + ATT_V_OFF + s * ATT_TILE;
                        mbar_arrive_expect_tx(v_full(s), ATT_TILE);
                        for (int ks = 0; ks < 2; ++ks)
                            for (int na = 0; na < 2; ++na)
                                tma_load_3d(dst + ks * ATT_SLAB + na * 8192u, &tmap_v, v_full(s), 64 * na,
                                            key0 + 64 * ks, bh);
                        v_pend |= 1u << s;
                        v_par = (v_par & ~(1u << s)) | (ph << s);
                    }
                }
            }
            // leave no bulk copy in flight
            if (q_loads > 0)
                wait_drain<false>(q_full, (q_loads - 1) & 1, w.limit_ns, w.id, w.status, SITE_ATT_DRAIN);
            for (uint32_t s = 0; s < ATT_STAGES; ++s) {
                if ((k_pend >> s) & 1u)
                    wait_drain<false>(k_full(s), (k_par >> s) & 1u, w.limit_ns, w.id, w.status, SITE_ATT_DRAIN);
                if ((v_pend >> s) & 1u)
                    wait_drain<false>(v_full(s), (v_par >> s) & 1u, w.limit_ns, w.id, w.status, SITE_ATT_DRAIN);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp walks the schedule and waits; one elected lane issues
        // each product and commit.
        auto sync_abort = [&]() {
            __syncwarp();
            w.aborted = __any_sync(0xffffffffu, w.aborted);
        };
        uint32_t rb = 0, qi = 0;               // ring blocks and Q tiles consumed so far
        uint32_t pb[ATT_TILES] = {0u, 0u};     // blocks of each tile consumed so far (p_full phases)
        uint32_t nd = 0;                       // row blocks whose tile B signalled done
        for (int64_t k = 0; k * gridDim.x < num_items; ++k) {
            const int64_t L = item_index(k);
            if (L >= num_items)
                continue;
            int qt, bh;
            item(L, qt, bh);
            const int q0 = qt * ATT_ROWS;
            const int nkv_a = att_num_blocks(q0, ATT_BM, p.Lq, p.Lk, p.causal != 0);
            const int nkv = att_num_blocks(q0, ATT_ROWS, p.Lq, p.Lk, p.causal != 0);
            if (nkv == 0)
                continue;
            wait_bounded<false>(w, q_full, qi & 1, SITE_ATT_Q);
            ++qi;
            sync_abort();
            tc_fence_after_sync();
            // S_g(j) = Q_g K_j^T into tile g's score buffer; after tile B, K_j's slot
            // is free, and after tile B's last one, so is Q
            auto mma_qk = [&](int j, uint32_t g) {
                const uint32_t r = rb + j, s = r % ATT_STAGES;
                const uint32_t k_addr = base + ATT_K_OFF + s * ATT_TILE;
                const uint32_t q_addr = base + ATT_Q_OFF + g * ATT_TILE;
#pragma unroll
                for (int slab = 0; slab < 2; ++slab) {
                    const uint64_t a_desc = smem_desc_sw128(q_addr + slab * ATT_SLAB, 16u, 1024u);
                    const uint64_t b_desc = smem_desc_sw128(k_addr + slab * ATT_SLAB, 16u, 1024u);
#pragma unroll
                    for (uint32_t k = 0; k < 4; ++k)
                        mma<1, KIND_F16>(tmem_base + g * ATT_BN, a_desc + 2u * k, b_desc + 2u * k, p.idesc_qk,
                                         (slab > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(s_full(g));
                if (g == 1) {
                    mma_commit(k_empty(s));
                    if (j == nkv - 1)
                        mma_commit(q_empty);
                }
            };
            // O_g += P_g V_j, P_g from TMEM (16 products of 16 keys, 8 columns each);
            // after tile B, V_j's slot is free
            auto mma_pv = [&](int j, uint32_t g) {
                const uint32_t r = rb + j, s = r % ATT_STAGES;
                const uint32_t v_addr = base + ATT_V_OFF + s * ATT_TILE;
#pragma unroll
                for (int slab = 0; slab < 2; ++slab) {
                    // N-contiguous V: 64-wide d atoms 8192 B apart, 16 keys = 2048 B per MMA
                    const uint64_t b_desc = smem_desc_sw128(v_addr + slab * ATT_SLAB, 8192u, 1024u);
#pragma unroll
                    for (uint32_t k = 0; k < 4; ++k)
                        mma_tmem_a(tmem_base + ATT_O_COL + g * ATT_BN, tmem_base + g * ATT_BN + slab * 32 + k * 8,
                                   b_desc + (2048u >> 4) * k, p.idesc_pv, (j > 0 || slab > 0 || k > 0) ? 1u : 0u);
                }
                if (g == 1)
                    mma_commit(v_empty(s));
            };
            auto wait_k = [&](int j) {
                const uint32_t r = rb + j;
                wait_bounded<false>(w, k_full(r % ATT_STAGES), (r / ATT_STAGES) & 1, SITE_ATT_K_FULL);
            };
            auto wait_v = [&](int j) {
                const uint32_t r = rb + j;
                wait_bounded<false>(w, v_full(r % ATT_STAGES), (r / ATT_STAGES) & 1, SITE_ATT_V_FULL);
            };
            // Each step waits for its ring slots first (they fill well ahead) and
            // for the group's probabilities last, so that once those arrive the
            // products issue back to back.
            wait_k(0);
            sync_abort();
            tc_fence_after_sync();
            if (!w.aborted) {
                if (nkv_a > 0)
                    mma_qk(0, 0);
                mma_qk(0, 1);
            }
            for (int j = 0; j < nkv; ++j) {
                if (j < nkv_a) {
                    wait_v(j);
                    if (j + 1 < nkv_a)
                        wait_k(j + 1);
                    wait_bounded<false>(w, p_full(0), (pb[0] + j) & 1, SITE_ATT_P_FULL);
                    sync_abort();
                    tc_fence_after_sync();
                    if (!w.aborted) {
                        mma_pv(j, 0);
                        if (j + 1 == nkv_a)
                            mma_commit(done(0));   // tile A's output may be read
                        else
                            mma_qk(j + 1, 0);      // tile A's next scores while group B finishes block j
                    }
                }
                if (j >= nkv_a)
                    wait_v(j);
                if (j + 1 < nkv && j + 1 >= nkv_a)
                    wait_k(j + 1);
                wait_bounded<false>(w, p_full(1), (pb[1] + j) & 1, SITE_ATT_P_FULL);
                sync_abort();
                tc_fence_after_sync();
                if (!w.aborted) {
                    mma_pv(j, 1);
                    if (j + 1 < nkv)
                        mma_qk(j + 1, 1);
                }
            }
            mma_commit(done(1));
            ++nd;
            rb += nkv;
            pb[0] += nkv_a;
            pb[1] += nkv;
        }
        // no product may still be writing TMEM when it is freed (tile B's last
        // done follows every product of this warp)
        if (nd > 0)
            wait_drain<false>(done(1), (nd - 1) & 1, w.limit_ns, w.id, w.status, SITE_ATT_DONE);
    } else {
        // ------------------------------------------------------------ softmax and output
        const uint32_t g = (warp - EPI_WARP0) / 4u;            // the query tile of this warp group
        const uint32_t quarter = warp & 3u;                    // the TMEM lane quarter this warp may access
        const int r = static_cast<int>(quarter * 32u + lane);  // row within the tile (TMEM lane)
        const uint32_t t_lane = (quarter * 32u) << 16;
        const uint32_t s_col = g * ATT_BN, o_col = ATT_O_COL + g * ATT_BN;
        const bool bf16 = p.bf16 != 0;
        uint32_t sb = 0;   // score blocks of this tile consumed so far (s_full phases)
        uint32_t nd = 0;   // row blocks of this tile whose output was read (done phases)
        for (int64_t k = 0; k * gridDim.x < num_items; ++k) {
            const int64_t L = item_index(k);
            if (L >= num_items)
                continue;
            int qt, bh;
            item(L, qt, bh);
            const int q0 = qt * ATT_ROWS;
            const int qrow = q0 + static_cast<int>(g) * ATT_BM + r;
            const int nkv_g = att_num_blocks(q0, g == 0 ? ATT_BM : ATT_ROWS, p.Lq, p.Lk, p.causal != 0);
            const int key_end = p.causal ? min(p.Lk, qrow + (p.Lk - p.Lq) + 1) : p.Lk;
            float m = -INFINITY, l = 0.0f;
            for (int j = 0; j < nkv_g; ++j) {
                wait_bounded<false>(w, s_full(g), (sb + j) & 1, SITE_ATT_S_FULL);
                const bool skip = __any_sync(0xffffffffu, w.aborted);
                w.aborted = skip;
                if (skip)
                    break;
                tc_fence_after_sync();
                float sv[ATT_BN];
                {
                    uint32_t v[4][32];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        tmem_ld_32x32b_x32(tmem_base + t_lane + s_col + c * 32, v[c]);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            sv[c * 32 + i] = __uint_as_float(v[c][i]);
                }
                // mask (only blocks that reach past some row's last visible key),
                // then the running maximum over raw scores, scaled once (scale > 0)
                const int key0 = j * ATT_BN;
                if (__any_sync(0xffffffffu, key0 + ATT_BN > key_end)) {
#pragma unroll
                    for (int c = 0; c < ATT_BN; ++c)
                        sv[c] = (key0 + c < key_end) ? sv[c] : -INFINITY;
                }
                float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < ATT_BN; c += 2)
                    mx4[(c / 2) & 3] = fmax3(mx4[(c / 2) & 3], sv[c], sv[c + 1]);
                const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * p.scale_log2;
                // raise the maximum only when some row of the warp outgrew it by more
                // than the threshold (always on the first block with a visible key)
                const bool raise = __any_sync(0xffffffffu, mx > m + RESCALE_LOG2);
                const float m_new = raise ? fmaxf(m, mx) : m;
                const float m_use = m_new == -INFINITY ? 0.0f : m_new;
                const float alpha = raise ? ex2(m - m_use) : 1.0f;   // 0 while no key has been seen
                // probabilities p = 2^(s * scale_log2 - m): a packed FFMA per pair and one
                // ex2 each, rounded to the operand type, two per TMEM column over the
                // first 64 columns of the score buffer; l sums them in FP32 (packed
                // adds, two pairs of accumulators)
                float sum4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pk[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const int e = 64 * h + 2 * c;
                        float xa, xb;
                        ffma2(xa, xb, sv[e], sv[e + 1], p.scale_log2, -m_use);
                        const float pa = ex2(xa), pb = ex2(xb);
                        pk[c] = pack2_rn(pa, pb, bf16);
                        if (c & 1)
                            fadd2(sum4[2], sum4[3], pa, pb);
                        else
                            fadd2(sum4[0], sum4[1], pa, pb);
                    }
                    tmem_st_32x32b_x32(tmem_base + t_lane + s_col + h * 32, pk);
                }
                l = l * alpha + ((sum4[0] + sum4[1]) + (sum4[2] + sum4[3]));
                m = m_new;
                // rescale this tile's accumulator row when the warp raised its maximum
                // (PV_g(j-1) has completed: S_g(j)'s commit covers it)
                if (j > 0 && raise) {
#pragma unroll 1
                    for (int h = 0; h < 2; ++h) {
                        uint32_t v[2][32];
                        const uint32_t ta = tmem_base + t_lane + o_col + h * 64;
                        tmem_ld_32x32b_x32(ta, v[0]);
                        tmem_ld_32x32b_x32(ta + 32, v[1]);
                        tmem_ld_wait();
#pragma unroll
                        for (int c = 0; c < 2; ++c)
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                v[c][i] = __float_as_uint(__uint_as_float(v[c][i]) * alpha);
                        tmem_st_32x32b_x32(ta, v[0]);
                        tmem_st_32x32b_x32(ta + 32, v[1]);
                    }
                }
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_local(p_full(g));
            }
            sb += nkv_g;
            // ------------------------------------------------------ output
            // The group reads the accumulator in full before it signals its
            // first probabilities of the next row block, which PV_g(0) (the
            // product that overwrites the accumulator) waits for.
            bool skip = w.aborted;
            if (nkv_g > 0 && !skip) {
                wait_bounded<false>(w, done(g), nd & 1, SITE_ATT_DONE);
                skip = __any_sync(0xffffffffu, w.aborted);
                w.aborted = skip;
                tc_fence_after_sync();
            }
            if (nkv_g > 0)
                ++nd;
            if (skip)
                continue;
            const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
            uint8_t *orow = static_cast<uint8_t *>(p.O) + (static_cast<size_t>(bh) * p.Lq + qrow) * ATT_D * 2;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                if (nkv_g > 0) {
                    tmem_ld_32x32b_x32(tmem_base + t_lane + o_col + c * 32, v);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[i] = 0u;
                }
                if (qrow < p.Lq) {
                    uint32_t o[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        o[i] = pack2_rn(__uint_as_float(v[2 * i]) * inv_l, __uint_as_float(v[2 * i + 1]) * inv_l,
                                        bf16);
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 64);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                }
            }
            if (p.LSE && qrow < p.Lq)
                p.LSE[static_cast<size_t>(bh) * p.Lq + qrow] =
                    l > 0.0f ? m * 0.69314718055994531f + logf(l) : -INFINITY;
            tc_fence_before_sync();
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<1>(tmem_base, ATT_TMEM_COLS);
    }
}

} // namespace dtg
