// gemm.cu: host side of the C ABI declared in gemm.h.
//
// One call validates its arguments, picks a tile plan, builds the TMA tensor
// maps (A, B, C), optionally re-pitches an operand that the TMA engine cannot
// describe, and launches one persistent kernel on the caller's stream. Plans
// and tensor maps are cached per device, so a repeated call does neither the
// plan search nor the encoding. Stream-ordered scratch is taken only for a
// re-pitched operand, the stream-K partial sums and the MX scale repack. The
// launcher of "Porting High-Performance HIP Kernels to FlyDSL" (section
// "Structure of a FlyDSL Kernel") is the model for the interface: prebuilt
// code, caller's stream, no stream created per call, no per-call setup
// beyond the launch.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cstring>
#include <mutex>
#include <random>

#include "gemm.h"
#include "gemm_kernel.cuh"
#include "runtime.h"

using namespace dtg;

// Device status word of this library, one copy per device:
// [0] id of the first launch that timed out since the host last read it,
// [1] the wait site of the latest timeout, [2] id of the latest timed-out launch.
static __device__ unsigned long long g_status[4];

namespace {

constexpr int MAX_DEVICES = 64;
constexpr int STREAM_SCRATCH_ENTRIES = 8;
constexpr uint64_t DEFAULT_TIMEOUT_MS = 2000;
// K per ring stage, unless gemm_options_t.k_stage says otherwise: 128 for CTA
// pairs (8 MMAs per barrier wait; the MMA issuer's wait costs ~60-100 cycles
// of tensor idle, so fewer waits per MMA pay), 64 for single CTAs (a 128-deep
// stage leaves room for only two of them); one slab for the block-scaled kinds.
int default_k_slabs(int cg, int kind)
{
    // Pairs take stages of two 128-byte slabs (256 K of FP8), except the
    // block-scaled kinds: at 4096 x 4096 x 65536 one-slab stages (six in the
    // ring) measure 357 us against 376 us for two-slab ones (three in the ring)
    // with packed FP4, and 701-744 us against 782-792 us with MXFP8.
    return kind_scaled(kind) ? 1 : cg == 2 ? 2 : 1;
}

template <int CG, int BN, int KS, int KIND, int MC>
cudaError_t launch_variant(int grid_ctas, int threads, uint32_t smem, const CUtensorMap *maps,
                           const KernelParams &kp, cudaStream_t st);
using LaunchFn = cudaError_t (*)(int, int, uint32_t, const CUtensorMap *, const KernelParams &, cudaStream_t);

struct Variant {
    int cg;
    int mc;            // CTA pairs per cluster sharing A tiles (1 or 2)
    int bn;
    int ks;            // K slabs (128 bytes of K each) per ring stage
    int kind;          // KIND_F16, KIND_F8, KIND_MXF8 or KIND_MXF4
    int stage_bytes;   // one ring slot: A and B tiles (and scales) of one stage, per CTA
    const void *fn;
    LaunchFn launch;   // launch_variant of the same template arguments
    bool b_mn_ok;      // MN-major B needs 64-column TMA boxes per CTA (16-bit only)
};

template <int CG, int BN, int KS, int KIND, int MC = 1>
constexpr Variant variant(bool b_mn_ok)
{
    return {CG, MC, BN, KS, KIND, TileConfig<CG, BN, KS, KIND>::STAGE_BYTES,
            reinterpret_cast<const void *>(&gemm_tcgen05_kernel<CG, BN, KS, KIND, MC>),
            &launch_variant<CG, BN, KS, KIND, MC>, b_mn_ok};
}

const Variant kVariants[] = {
    variant<2, 256, 1, KIND_F16>(true),  variant<2, 224, 1, KIND_F16>(false), variant<1, 256, 1, KIND_F16>(true),
    variant<2, 256, 2, KIND_F16>(true),  variant<2, 224, 2, KIND_F16>(false), variant<1, 256, 2, KIND_F16>(true),
    variant<2, 256, 1, KIND_F8>(false),  variant<2, 224, 1, KIND_F8>(false),  variant<1, 256, 1, KIND_F8>(false),
    variant<2, 256, 2, KIND_F8>(false),  variant<2, 224, 2, KIND_F8>(false),  variant<1, 256, 2, KIND_F8>(false),
    variant<2, 224, 1, KIND_MXF8>(false), variant<2, 224, 2, KIND_MXF8>(false),
    variant<2, 224, 1, KIND_MXF4>(false), variant<2, 224, 2, KIND_MXF4>(false),
    // narrow single-CTA tiles: more units for problems of few tiles
    variant<1, 128, 1, KIND_F16>(true), variant<1, 64, 1, KIND_F16>(true),
    variant<1, 128, 1, KIND_F8>(false), variant<1, 64, 1, KIND_F8>(false),
    // two pairs per cluster sharing A (gemm_options_t.cluster_pairs = 2)
    variant<2, 256, 1, KIND_F16, 2>(true), variant<2, 256, 2, KIND_F16, 2>(true),
    variant<2, 256, 1, KIND_F8, 2>(false), variant<2, 256, 2, KIND_F8, 2>(false),
};
constexpr int NUM_VARIANTS = sizeof(kVariants) / sizeof(kVariants[0]);

// Shared-memory budget of one launch: the deepest ring that fits next to the
// epilogue staging buffers (2 KB each for a 16-bit C, 4 KB for an FP32 C).
struct Layout {
    uint32_t stages;
    uint32_t staging_bytes;
    uint32_t staging_bufs;
    uint32_t smem;
};

Layout layout_for(const Variant &v, int dtype_out)
{
    Layout l;
    l.staging_bytes = dtype_out == GEMM_F32 ? 4096u : 2048u;
    // block-scaled kinds keep one TMEM scale slot per ring stage (MX_MAX_STAGES of them)
    const uint32_t max_stages = kind_scaled(v.kind) ? MX_MAX_STAGES : MAX_STAGES;
    auto deepest = [&](uint32_t bufs) {
        uint32_t st = max_stages;
        while (st > 2 && smem_bytes_for(v.stage_bytes, st, l.staging_bytes, bufs) > SMEM_LIMIT)
            --st;
        return st;
    };
    // Four staging buffers per epilogue warp where they fit and cost no ring
    // stage: a chunk's TMA store then rarely waits for the store three chunks back.
    const uint32_t d4 = deepest(4);
    l.staging_bufs =
        (d4 == deepest(2) && smem_bytes_for(v.stage_bytes, d4, l.staging_bytes, 4u) <= SMEM_LIMIT) ? 4u : 2u;
    l.stages = deepest(l.staging_bufs);
    l.smem = smem_bytes_for(v.stage_bytes, l.stages, l.staging_bytes, l.staging_bufs);
    return l;
}

struct DeviceState {
    bool ready = false;
    int dev = 0;
    int sms = 0;
    unsigned long long *status = nullptr;
    int max_units[NUM_VARIANTS] = {};   // co-resident CTAs (cg 1) or CTA pairs (cg 2)
    // gemm_from_host(_async) staging: two slots of device copies of A, B and C, so
    // that one call's uploads (on h2d) overlap the previous call's product and
    // read-back (on the caller's stream)
    std::mutex ws_mu;
    struct HostSlot {
        void *ws = nullptr;
        size_t bytes = 0;
        cudaEvent_t uploaded = nullptr;   // A and B are on the device
        cudaEvent_t released = nullptr;   // the product and the read-back of C are done
        bool used = false;
    } slots[2];
    unsigned next_slot = 0;
    cudaStream_t h2d = nullptr;
    // Per-stream scratch for re-pitched operands, packed scales and stream-K
    // partial sums. A call reuses its stream's buffer, which stream order makes
    // safe, so no allocation (a stream operation that would stop the next
    // kernel from launching early) sits between two calls' kernels. Entries are
    // keyed by cudaStreamGetId, which no later stream reuses; a buffer grows
    // only on its own stream. Nothing is evicted: calls on further streams take
    // per-call scratch, and gemm_release_workspace frees every buffer.
    std::mutex scratch_mu;
    struct StreamScratch {
        unsigned long long stream_id = 0;
        bool used = false;
        void *ptr = nullptr;
        size_t bytes = 0;
    } scratch[STREAM_SCRATCH_ENTRIES];
};

std::mutex g_mu;
DeviceState g_dev[MAX_DEVICES];
std::atomic<uint64_t> g_launches{0};
// Launch ids start at a random 64-bit value. Stream-K flags are compared with
// the launch id, and a per-call workspace may hold any old bytes: a random
// start makes an accidental match with a stale word vanishingly unlikely
// (ids of this library's own earlier launches never match).
unsigned long long first_launch_id()
{
    std::random_device rd;
    unsigned long long v = (static_cast<unsigned long long>(rd()) << 32) ^ rd();
    return v ? v : 1;
}
std::atomic<unsigned long long> g_next_id{first_launch_id()};

unsigned long long next_launch_id()
{
    unsigned long long id;
    do
        id = g_next_id.fetch_add(1, std::memory_order_relaxed);
    while (id == 0);   // 0 means "no timeout" in the device status word
    return id;
}
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool is_fp8(int dtype) { return dtype == GEMM_E4M3 || dtype == GEMM_E5M2; }
int out_bytes(int dtype_out) { return dtype_out == GEMM_F32 ? 4 : 2; }

// The MMA kind for an input type, plain (gemm) or block-scaled (gemm_mx).
int kind_for(int dtype_in, bool scaled)
{
    if (dtype_in == GEMM_E2M1)
        return KIND_MXF4;
    if (is_fp8(dtype_in))
        return scaled ? KIND_MXF8 : KIND_F8;
    return KIND_F16;
}

// Bytes of one stored row of `elems` operand elements (packed FP4 rows are
// padded to whole bytes), and the TMA element size.
int64_t row_bytes(int kind, int64_t elems)
{
    return kind == KIND_F16 ? 2 * elems : kind == KIND_MXF4 ? (elems + 1) / 2 : elems;
}
int tma_elem_bytes(int kind) { return kind == KIND_F16 ? 2 : 1; }

// Row pitch, in TMA elements, of a re-pitched operand: the row of `cols` such
// elements rounded up to a multiple of 128 bytes. TMA needs 16; with rows that
// are only 16-byte aligned every 128-byte box row straddles two 128-byte lines,
// and the kernel runs up to a quarter slower (3000 x 5000 x 2056 BF16: 61 us,
// against 49 us at K = 2112, whose rows are 33 x 128 bytes).
int64_t padded_pitch(int64_t cols, int eb)
{
    const int64_t q = 128 / eb;
    return (cols + q - 1) / q * q;
}

gemm_status_t device_state(DeviceState **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_NO_DEVICE;
        }
        if (major != 10 || minor != 3)   // the library holds sm_103a code only
            return GEMM_ERR_NO_DEVICE;
        d.dev = dev;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return GEMM_ERR_CUDA;
        void *status = nullptr;
        if (cudaGetSymbolAddress(&status, g_status) != cudaSuccess)
            return GEMM_ERR_CUDA;
        d.status = static_cast<unsigned long long *>(status);
        for (int v = 0; v < NUM_VARIANTS; ++v) {
            const Variant &var = kVariants[v];
            if (cudaFuncSetAttribute(var.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT) !=
                cudaSuccess)
                return GEMM_ERR_CUDA;
            if (var.cg == 1) {
                int per_sm = 0;
                if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, var.fn, NUM_THREADS,
                                                                  SMEM_LIMIT) != cudaSuccess)
                    return GEMM_ERR_CUDA;
                d.max_units[v] = per_sm * d.sms;
            } else {
                cudaLaunchConfig_t cfg = {};
                const int cs = var.cg * var.mc;
                cfg.gridDim = dim3(static_cast<unsigned>(cs * d.sms));
                cfg.blockDim = dim3(NUM_THREADS);
                cfg.dynamicSmemBytes = SMEM_LIMIT;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                int clusters = 0;
                if (cudaOccupancyMaxActiveClusters(&clusters, var.fn, &cfg) != cudaSuccess)
                    return GEMM_ERR_CUDA;
                d.max_units[v] = clusters;
            }
        }
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                                 &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return GEMM_ERR_CUDA;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        d.ready = true;
    }
    *out = &d;
    return GEMM_OK;
}

gemm_status_t validate(const void *A, const void *B, const void *C, int64_t M, int64_t N, int64_t K,
                       int dtype_in, int dtype_out, int layoutA, int layoutB, const gemm_options_t *o,
                       bool scaled = false)
{
    if (!A || !B || !C)
        return GEMM_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1 || M > INT_MAX || N > INT_MAX || K > INT_MAX)
        return GEMM_ERR_INVALID_ARG;
    if (dtype_in != GEMM_F16 && dtype_in != GEMM_BF16 && !is_fp8(dtype_in) && dtype_in != GEMM_E2M1)
        return dtype_in == GEMM_F32 ? GEMM_ERR_UNSUPPORTED : GEMM_ERR_INVALID_ARG;
    // block-scaled products take 8- or 4-bit elements; packed FP4 only comes block-scaled
    if (scaled ? (!is_fp8(dtype_in) && dtype_in != GEMM_E2M1) : dtype_in == GEMM_E2M1)
        return GEMM_ERR_UNSUPPORTED;
    if (dtype_out != GEMM_F16 && dtype_out != GEMM_BF16 && dtype_out != GEMM_F32)
        return is_fp8(dtype_out) ? GEMM_ERR_UNSUPPORTED : GEMM_ERR_INVALID_ARG;
    if (layoutA != GEMM_K_MAJOR && layoutA != GEMM_MN_MAJOR)
        return GEMM_ERR_INVALID_ARG;
    if (layoutA == GEMM_MN_MAJOR)
        return GEMM_ERR_UNSUPPORTED;
    if (layoutB != GEMM_K_MAJOR && layoutB != GEMM_MN_MAJOR)
        return GEMM_ERR_INVALID_ARG;
    if ((is_fp8(dtype_in) || dtype_in == GEMM_E2M1) && layoutB == GEMM_MN_MAJOR)
        return GEMM_ERR_UNSUPPORTED;
    if (o) {
        if (o->cta_group < 0 || o->cta_group > 2 || o->max_clusters < 0 || o->group_m < 0 ||
            o->timeout_ms < 0 || o->block_n < 0)
            return GEMM_ERR_INVALID_ARG;
        if (o->block_n != 0 && o->block_n != 64 && o->block_n != 128 && o->block_n != 224 && o->block_n != 256)
            return GEMM_ERR_UNSUPPORTED;
        if (o->k_stage < 0 || o->stream_k < 0 || o->cluster_pairs < 0)
            return GEMM_ERR_INVALID_ARG;
        if (o->cluster_pairs > 2)
            return GEMM_ERR_UNSUPPORTED;
        if (o->epilogue_warps < 0 || o->reserved != 0)
            return GEMM_ERR_INVALID_ARG;
        if (o->epilogue_warps != 0 && o->epilogue_warps != 4 && o->epilogue_warps != 8)
            return GEMM_ERR_UNSUPPORTED;
        if (o->stream_k > 2)
            return GEMM_ERR_UNSUPPORTED;
        const int sk = kind_slab_k(kind_for(dtype_in, scaled));
        if (o->k_stage != 0 && o->k_stage != sk && o->k_stage != 2 * sk)
            return GEMM_ERR_UNSUPPORTED;
    }
    return GEMM_OK;
}

struct Plan {
    int variant;
    int num_m, num_n, num_tiles, num_kb;   // num_n, num_tiles: scheduling units (two tiles each with mc = 2)
    int grid_ctas;
    int group_m;
    int sk_tiles;          // trailing tiles split along K
    int epi_warps;         // epilogue warps of the launch: 4 or 8
    size_t ws_bytes;       // stream-K workspace: flags, then partial sums
    bool realign_a, realign_b, direct_store;
};

// ------------------------------------------------------------------ launch cache
// Per device, the plans and TMA tensor maps of the most recent launches, so
// that a repeated call skips the planner's variant search and the
// cuTensorMapEncodeTiled calls. Keys are compared bytewise (every key is
// zeroed before it is filled, padding included). Entries are replaced least
// recently used first. A tensor map holds only the numbers it was encoded
// from, so a cached one equals a fresh encoding of the same key.
struct PlanKey {
    int64_t M, N, K;
    int32_t dtype_in, dtype_out, layoutB, scaled;
    int32_t misalign;   // bit 0: A, bit 1: B, bit 2: C not describable to the TMA engine
    int32_t cta_group, block_n, max_clusters, group_m, k_stage, stream_k;
    int32_t cluster_pairs, epilogue_warps;
};

struct MapKey {
    PlanKey plan;
    int32_t variant, pad;
    const void *a, *b, *c, *sfa, *sfb;   // the addresses the maps describe
    int64_t lda, ldb;                    // their row pitches, in TMA elements
};

constexpr int CACHE_ENTRIES = GEMM_LAUNCH_CACHE_ENTRIES;

struct LaunchCache {
    std::mutex mu;
    uint64_t clock = 0;
    struct PlanEntry {
        PlanKey key;
        Plan plan;
        uint64_t used = 0;   // 0: empty
    } plans[CACHE_ENTRIES];
    struct MapEntry {
        MapKey key;
        CUtensorMap maps[5];
        uint64_t used = 0;
    } maps[CACHE_ENTRIES];

    template <typename E, typename Key>
    static E *find(E (&tab)[CACHE_ENTRIES], const Key &k)
    {
        for (E &e : tab)
            if (e.used && std::memcmp(&e.key, &k, sizeof(Key)) == 0)
                return &e;
        return nullptr;
    }
    template <typename E>
    static E *victim(E (&tab)[CACHE_ENTRIES])
    {
        E *v = &tab[0];
        for (E &e : tab)
            if (e.used < v->used)
                v = &e;
        return v;
    }
    void clear()
    {
        std::lock_guard<std::mutex> lock(mu);
        for (PlanEntry &e : plans)
            e.used = 0;
        for (MapEntry &e : maps)
            e.used = 0;
    }
};

LaunchCache g_cache[MAX_DEVICES];
std::atomic<uint64_t> g_plan_hits{0}, g_plan_misses{0}, g_map_hits{0}, g_map_misses{0};

// Stream-K workspace of a launch: one flag per (CTA, epilogue warp), then one
// partial-sum slot per CTA (128 rows x block_n FP32).
size_t sk_flag_bytes(int grid_ctas) { return (static_cast<size_t>(grid_ctas) * EPI_WARPS_MAX * 8 + 255) / 256 * 256; }
size_t sk_workspace_bytes(int grid_ctas, int bn)
{
    return sk_flag_bytes(grid_ctas) + static_cast<size_t>(grid_ctas) * BLOCK_M_CTA * bn * 4;
}

// Stream-K tiles for T tiles on U units: the last partial wave plus one full
// wave (so every tile is cut at most once while units >= tiles), or all
// tiles when there are fewer than two waves.
int sk_tiles_for(int64_t T, int64_t U) { return static_cast<int>(T < 2 * U ? T : U + T % U); }

// Predicted time of a plan in microseconds, fitted to CUDA-graph timings of
// every variant (128 x 64 to 256 x 256 tiles, each with and without stream-K)
// on 15 shapes from 512^3 to 2560^3 with K up to 16384, and of the planner's
// plan, data-parallel plans and 224-wide plans on 7 shapes from 3072^3 to
// 8192^3, at 1.7-1.9 GHz:
//  - one tile on one SM costs the larger of its products at 80% of the tensor
//    rate (block_n x K bytes / 64 cycles) and its operand bytes,
//    (128 / mc + block_n / cg) rows x K bytes, from L2 at ~55 bytes per SM
//    cycle for single CTAs and ~45 for CTA pairs: narrow tiles are bound by L2,
//    not by the tensor core, and 224-wide pair tiles do less work per byte
//    than 256-wide ones;
//  - a launch pays ~2.6 us (ring fill, teardown) plus its last tile's
//    epilogue, ~0.006 us per column, which nothing overlaps;
//  - a stream-K owner adds its writers' partial sums: in effect ~6 us plus
//    ~1.5 us per writer and 32-column chunk, more than the fix-up's own time
//    in a trace, as it also slows the main loop beside it. With one writer
//    and data-parallel tiles after it, the next tile's main loop hides up to
//    one tile time of that; otherwise (fewer tiles than two waves) the whole
//    fix-up adds to the launch.
struct Cost {
    double dp, sk;
    int sk_tiles;
};

Cost plan_cost(int64_t T, int64_t U, int64_t KB, int64_t k_bytes, int cg, int bn, int mc)
{
    constexpr double kMmaEff = 0.8, kCyclesPerUs = 1900.0;
    constexpr double kL2BytesPerCycleCta = 55.0, kL2BytesPerCyclePair = 45.0;
    constexpr double kLaunchUs = 2.6, kEpilogueUsPerCol = 0.006, kFixUs = 6.0, kFixChunkUs = 1.5;
    const double kb = static_cast<double>(k_bytes);
    const double mma = bn * kb / 64.0 / kMmaEff;
    const double l2 = (128.0 / mc + static_cast<double>(bn) / cg) * kb /
                      (cg == 1 ? kL2BytesPerCycleCta : kL2BytesPerCyclePair);
    const double tile = std::max(mma, l2) / kCyclesPerUs;
    const double fixed = kLaunchUs + kEpilogueUsPerCol * bn;
    Cost c;
    c.dp = static_cast<double>((T + U - 1) / U) * tile + fixed;
    const int64_t S = sk_tiles_for(T, U);
    c.sk_tiles = static_cast<int>(S);
    const int64_t L = (S * KB + U - 1) / U;                        // k-blocks per unit
    const int64_t writers = L >= KB ? 1 : (KB + L - 1) / L - 1;    // per split tile
    const double fix = kFixUs + static_cast<double>(writers * (bn / 32)) * kFixChunkUs;
    const int64_t dp_after = (T - S) / U;                          // whole tiles after the owner's
    c.sk = (static_cast<double>(dp_after) + static_cast<double>(L) / static_cast<double>(KB)) * tile + fixed +
           (dp_after >= 1 && writers == 1 ? std::max(0.0, fix - tile) : fix);
    return c;
}

bool misaligned(const void *p, int64_t row_elems, int elem_bytes)
{
    return (reinterpret_cast<uintptr_t>(p) % 16) != 0 || (row_elems * elem_bytes) % 16 != 0;
}

// Choose the variant (tile shape, CTA group) and schedule (data-parallel or
// stream-K) of least predicted time (plan_cost).
gemm_status_t make_plan(const DeviceState &d, int64_t M, int64_t N, int64_t K, int dtype_in,
                        int dtype_out, int layoutB, const void *A, const void *B, const void *C,
                        const gemm_options_t *o, Plan *pl, bool scaled = false)
{
    const bool b_mn = layoutB == GEMM_MN_MAJOR;
    const int kind = kind_for(dtype_in, scaled);
    const int sk_elems = kind_slab_k(kind);
    const int64_t k_bytes = row_bytes(kind, K);
    const int mode = o ? o->stream_k : 0;
    // pairs sharing A only on request: two pairs per cluster (cluster_pairs = 2)
    const int want_mc = (o && o->cluster_pairs) ? o->cluster_pairs : 1;
    int best = -1, best_sk = 0;
    double best_cost = 0;
    for (int v = 0; v < NUM_VARIANTS; ++v) {
        const Variant &var = kVariants[v];
        if (var.kind != kind)
            continue;
        if (o && o->cta_group && o->cta_group != var.cg)
            continue;
        if (o && o->block_n && o->block_n != var.bn)
            continue;
        if (var.ks != ((o && o->k_stage) ? o->k_stage / sk_elems : default_k_slabs(var.cg, var.kind)))
            continue;
        if (b_mn && !var.b_mn_ok)
            continue;
        if (var.mc != want_mc)
            continue;
        int units = d.max_units[v];
        if (o && o->max_clusters)
            units = std::min(units, static_cast<int>(o->max_clusters));
        if (units < 1)
            continue;
        // scheduling units: one tile, or with mc = 2 two tiles side by side in N
        const int64_t n_units = ((N + var.bn - 1) / var.bn + var.mc - 1) / var.mc;
        const int64_t tiles = ((M + 128 * var.cg - 1) / (128 * var.cg)) * n_units;
        const int64_t kb = (K + static_cast<int64_t>(sk_elems) * var.ks - 1) / (static_cast<int64_t>(sk_elems) * var.ks);
        const Cost c = plan_cost(tiles, units, kb, k_bytes, var.cg, var.bn, var.mc);
        // stream-K only where it saves more than 3%, or when asked for
        const bool sk = mode == 2 || (mode == 0 && tiles % units != 0 && c.sk < 0.97 * c.dp);
        const double cost = sk ? c.sk : c.dp;
        if (best < 0 || cost < best_cost) {
            best = v;
            best_cost = cost;
            best_sk = sk ? c.sk_tiles : 0;
        }
    }
    if (best < 0)
        return GEMM_ERR_UNSUPPORTED;
    const Variant &var = kVariants[best];
    int units = d.max_units[best];
    if (o && o->max_clusters)
        units = std::min(units, static_cast<int>(o->max_clusters));
    pl->variant = best;
    pl->num_m = static_cast<int>((M + 128 * var.cg - 1) / (128 * var.cg));
    pl->num_n = static_cast<int>(((N + var.bn - 1) / var.bn + var.mc - 1) / var.mc);
    const int64_t tiles = static_cast<int64_t>(pl->num_m) * pl->num_n;
    if (tiles > INT_MAX)
        return GEMM_ERR_UNSUPPORTED;
    pl->num_tiles = static_cast<int>(tiles);
    const int64_t stage_k = static_cast<int64_t>(sk_elems) * var.ks;
    pl->num_kb = static_cast<int>((K + stage_k - 1) / stage_k);
    pl->sk_tiles = best_sk;
    // Eight epilogue warps where a unit's last epilogue (which nothing overlaps)
    // is a large share of its time: work of at most two tiles (2048^3 measured
    // 5.8% faster, 1024^3 3.2%), or of at most four with a 16-bit C (4096^3 and
    // 4096 x 4096 x 8192: 0.5-0.7% faster in short runs, 0.7-1.8% under the
    // power cap). Four elsewhere: eight cost 0.5-1% at 8192^3 and beyond, and
    // with an FP32 C, which leaves each of the eight one staging buffer (1.1%
    // on the ragged 3000 x 5000 x 2050 workload).
    const double unit_tiles =
        best_sk ? static_cast<double>((tiles - best_sk) / units) +
                      static_cast<double>((static_cast<int64_t>(best_sk) * pl->num_kb + units - 1) / units) / pl->num_kb
                : static_cast<double>((tiles + units - 1) / units);
    const bool wide_epilogue = unit_tiles <= 2.0 || (unit_tiles <= 4.0 && dtype_out != GEMM_F32);
    pl->epi_warps = (o && o->epilogue_warps) ? o->epilogue_warps : (wide_epilogue ? 8 : 4);
    // with stream-K every unit takes a share; otherwise no more units than tiles
    pl->grid_ctas = static_cast<int>(best_sk ? units : std::min<int64_t>(tiles, units)) * var.cg * var.mc;
    pl->ws_bytes = best_sk ? sk_workspace_bytes(pl->grid_ctas, var.bn) : 0;
    pl->group_m = (o && o->group_m) ? o->group_m : 8;
    pl->realign_a = misaligned(A, row_bytes(kind, K), 1);
    pl->realign_b = misaligned(B, b_mn ? row_bytes(kind, N) : row_bytes(kind, K), 1);
    pl->direct_store = misaligned(C, N, out_bytes(dtype_out));
    return GEMM_OK;
}

PlanKey plan_key(int64_t M, int64_t N, int64_t K, int dtype_in, int dtype_out, int layoutB, bool scaled,
                 const void *A, const void *B, const void *C, const gemm_options_t *o)
{
    PlanKey k;
    std::memset(&k, 0, sizeof(k));
    k.M = M;
    k.N = N;
    k.K = K;
    k.dtype_in = dtype_in;
    k.dtype_out = dtype_out;
    k.layoutB = layoutB;
    k.scaled = scaled ? 1 : 0;
    const int kind = kind_for(dtype_in, scaled);
    const bool b_mn = layoutB == GEMM_MN_MAJOR;
    k.misalign = (misaligned(A, row_bytes(kind, K), 1) ? 1 : 0) |
                 (misaligned(B, b_mn ? row_bytes(kind, N) : row_bytes(kind, K), 1) ? 2 : 0) |
                 (misaligned(C, N, out_bytes(dtype_out)) ? 4 : 0);
    if (o) {   // the fields that steer the planner (not timeout_ms or clock_trace)
        k.cta_group = o->cta_group;
        k.block_n = o->block_n;
        k.max_clusters = o->max_clusters;
        k.group_m = o->group_m;
        k.k_stage = o->k_stage;
        k.stream_k = o->stream_k;
        k.cluster_pairs = o->cluster_pairs;
        k.epilogue_warps = o->epilogue_warps;
    }
    return k;
}

// make_plan through the device's launch cache. The plan depends only on the
// key: make_plan reads the operand pointers for their alignment alone.
gemm_status_t cached_plan(const DeviceState &d, const PlanKey &k, const void *A, const void *B, const void *C,
                          const gemm_options_t *o, Plan *pl)
{
    LaunchCache &c = g_cache[d.dev];
    {
        std::lock_guard<std::mutex> lock(c.mu);
        if (LaunchCache::PlanEntry *e = LaunchCache::find(c.plans, k)) {
            e->used = ++c.clock;
            *pl = e->plan;
            g_plan_hits.fetch_add(1, std::memory_order_relaxed);
            return GEMM_OK;
        }
    }
    g_plan_misses.fetch_add(1, std::memory_order_relaxed);
    const gemm_status_t rc =
        make_plan(d, k.M, k.N, k.K, k.dtype_in, k.dtype_out, k.layoutB, A, B, C, o, pl, k.scaled != 0);
    if (rc != GEMM_OK)
        return rc;
    std::lock_guard<std::mutex> lock(c.mu);
    LaunchCache::PlanEntry *e = LaunchCache::victim(c.plans);
    e->key = k;
    e->plan = *pl;
    e->used = ++c.clock;
    return GEMM_OK;
}

bool encode_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner,
               uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle)
{
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estride[2] = {1, 1};
    return g_encode(map, dt, 2, const_cast<void *>(base), dims, strides, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

CUtensorMapDataType tma_dtype(int dtype)
{
    switch (dtype) {
    case GEMM_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    case GEMM_F32: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    case GEMM_E4M3:
    case GEMM_E5M2:
    case GEMM_E2M1: return CU_TENSOR_MAP_DATA_TYPE_UINT8;   // bytes are moved, not converted
    default: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    }
}

// Copy a rows x cols matrix of eb-byte elements into `dst`, whose row pitch
// ld (elements) makes every row a multiple of 128 bytes. The pad is never
// read: the tensor map keeps the logical width `cols`, and TMA zero-fills
// past it.
gemm_status_t realign_into(const void *src, int64_t rows, int64_t cols, int64_t ld, int eb, int sms,
                           cudaStream_t st, void *dst)
{
    const int64_t row_bytes = cols * eb, pitch = ld * eb;
    // widest word (<= 16 bytes) dividing the source base and the row length, so
    // that every source row starts on a word boundary
    const uint64_t align = static_cast<uint64_t>(reinterpret_cast<uintptr_t>(src)) | static_cast<uint64_t>(row_bytes);
    const int v = (align % 16 == 0) ? 16 : (align % 8 == 0) ? 8 : (align % 4 == 0) ? 4 : (align % 2 == 0) ? 2 : 1;
    // one warp per row at a time, up to 3 blocks of 8 warps per SM
    const unsigned blocks = static_cast<unsigned>(
        std::max<int64_t>(std::min<int64_t>((rows + 7) / 8, static_cast<int64_t>(sms) * 3), 1));
    const uint8_t *s = static_cast<const uint8_t *>(src);
    uint8_t *d = static_cast<uint8_t *>(dst);
    // In plain stream order: launched early beside the previous GEMM (programmatic
    // stream serialisation), the copy measured 1.5 us slower per call back to back
    // on the ragged 3000 x 5000 x 2050 workload, and no faster in a CUDA graph.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cfg.numAttrs = 0;
    cudaError_t e;
    switch (v) {
    case 16: e = cudaLaunchKernelEx(&cfg, realign_rows_kernel<16>, s, d, rows, row_bytes, pitch); break;
    case 8: e = cudaLaunchKernelEx(&cfg, realign_rows_kernel<8>, s, d, rows, row_bytes, pitch); break;
    case 4: e = cudaLaunchKernelEx(&cfg, realign_rows_kernel<4>, s, d, rows, row_bytes, pitch); break;
    case 2: e = cudaLaunchKernelEx(&cfg, realign_rows_kernel<2>, s, d, rows, row_bytes, pitch); break;
    default: e = cudaLaunchKernelEx(&cfg, realign_rows_kernel<1>, s, d, rows, row_bytes, pitch); break;
    }
    if (e != cudaSuccess || cudaGetLastError() != cudaSuccess)
        return GEMM_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return GEMM_OK;
}

template <int CG, int BN, int KS, int KIND, int MC>
cudaError_t launch_variant(int grid_ctas, int threads, uint32_t smem, const CUtensorMap *maps,
                           const KernelParams &kp, cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid_ctas));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    // Programmatic stream serialisation lets this grid's CTAs start their setup
    // while the previous grid on the stream drains; the kernel waits
    // (griddepcontrol.wait) before touching global memory.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (CG * MC > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = CG * MC;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, gemm_tcgen05_kernel<CG, BN, KS, KIND, MC>, maps[0], maps[1], maps[2], maps[3],
                              maps[4], kp);
}

cudaError_t launch_any(const Variant &v, int grid_ctas, int epi_warps, uint32_t smem, const CUtensorMap *maps,
                       const KernelParams &kp, cudaStream_t st)
{
    return v.launch(grid_ctas, (EPI_WARP0 + epi_warps) * 32, smem, maps, kp, st);
}

// Packed-scale geometry of one operand: row blocks of R rows (128 for A, the
// CTA's B rows for B), `stages` ring stages along K, `groups` atoms per stage.
struct SfGeometry {
    int R;
    int64_t row_blocks, stages;
    int groups, atoms;   // groups of 4 blocks per stage, 128-row atoms per group
    int64_t atom_rows;   // 16-byte rows in the packed tensor
    int64_t bytes() const { return atom_rows * SF_ROW_BYTES; }
    int box_rows() const { return groups * atoms * SF_ATOM_ROWS; }
};

// A: row blocks of 128 rows (one CTA's rows), one atom per group. B: row
// blocks of the whole tile width (every CTA of a pair holds all of it).
SfGeometry sf_geometry(const Variant &var, const Plan &pl, int64_t rows, bool is_b)
{
    SfGeometry g;
    g.R = is_b ? var.bn : BLOCK_M_CTA;
    g.atoms = (g.R + 127) / 128;
    g.row_blocks = (rows + g.R - 1) / g.R;
    g.stages = pl.num_kb;
    g.groups = kind_slab_k(var.kind) * var.ks / 128;
    g.atom_rows = g.row_blocks * g.stages * g.groups * g.atoms * SF_ATOM_ROWS;
    return g;
}

// An operand ready for the tensor maps: base and row pitch in TMA elements
// (FP16/BF16 elements, or bytes for the 8- and 4-bit kinds).
struct Operand {
    const void *ptr;
    int64_t ld;
};

// Encode the plan's tensor maps (A, B, C and, block-scaled, the packed
// scales sfa/sfb) for operands already at TMA-describable addresses.
bool encode_maps(const Plan &pl, Operand a, Operand b, const void *sfa, const void *sfb, void *C, int64_t M,
                 int64_t N, int64_t K, int dtype_in, int dtype_out, bool b_mn, CUtensorMap *maps)
{
    const Variant &var = kVariants[pl.variant];
    const int eb = tma_elem_bytes(var.kind);
    const int64_t width = row_bytes(var.kind, K) / eb;   // K in TMA elements
    const uint32_t box_k = var.kind == KIND_F16 ? 64 : 128;
    std::memset(maps, 0, 5 * sizeof(CUtensorMap));
    const CUtensorMapDataType in_dt = tma_dtype(dtype_in);
    // with two pairs sharing A each CTA loads half of its 128 rows
    bool ok = encode_2d(&maps[0], in_dt, a.ptr, width, M, a.ld * eb, box_k, BLOCK_M_CTA / var.mc,
                        CU_TENSOR_MAP_SWIZZLE_128B);
    if (!b_mn)
        ok = ok && encode_2d(&maps[1], in_dt, b.ptr, width, N, b.ld * eb, box_k, var.bn / var.cg,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    else
        ok = ok && encode_2d(&maps[1], in_dt, b.ptr, N, K, b.ld * eb, 64, box_k, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!pl.direct_store)
        ok = ok && encode_2d(&maps[2], tma_dtype(dtype_out), C, N, M, N * out_bytes(dtype_out), EPI_COLS, 32,
                             dtype_out == GEMM_F32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
    if (kind_scaled(var.kind)) {
        // packed scales: 16-byte rows, one box = this stage's atoms of one row block
        const SfGeometry ga = sf_geometry(var, pl, M, false), gb = sf_geometry(var, pl, N, true);
        ok = ok && encode_2d(&maps[3], CU_TENSOR_MAP_DATA_TYPE_UINT8, sfa, SF_ROW_BYTES, ga.atom_rows, SF_ROW_BYTES,
                             SF_ROW_BYTES, ga.box_rows(), CU_TENSOR_MAP_SWIZZLE_NONE);
        ok = ok && encode_2d(&maps[4], CU_TENSOR_MAP_DATA_TYPE_UINT8, sfb, SF_ROW_BYTES, gb.atom_rows, SF_ROW_BYTES,
                             SF_ROW_BYTES, gb.box_rows(), CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    return ok;
}

// Per-launch extras: the clock trace words (gemm_options_t.clock_trace) and
// the self-test's withheld k-block (-1: none).
struct Extras {
    unsigned long long *trace = nullptr;
    int32_t withhold_kb = -1;
};

// Fetch the tensor maps from the launch cache (or encode and insert them),
// fill the kernel parameters and launch the plan's kernel on `st`. For the
// block-scaled kinds sfa/sfb are the packed scales (rows x num_kb x 16 bytes).
gemm_status_t encode_and_launch(const DeviceState &d, const PlanKey &pk, const Plan &pl, Operand a, Operand b,
                                const void *sfa, const void *sfb, void *C, int64_t M, int64_t N, int64_t K,
                                int dtype_in, int dtype_out, bool b_mn, uint64_t timeout_ms, void *workspace,
                                const Extras &x, cudaStream_t st)
{
    const Variant &var = kVariants[pl.variant];
    CUtensorMap maps[5];
    MapKey mk;
    std::memset(&mk, 0, sizeof(mk));
    mk.plan = pk;
    mk.variant = pl.variant;
    mk.a = a.ptr;
    mk.b = b.ptr;
    mk.c = C;
    mk.sfa = sfa;
    mk.sfb = sfb;
    mk.lda = a.ld;
    mk.ldb = b.ld;
    LaunchCache &cache = g_cache[d.dev];
    bool hit = false;
    {
        std::lock_guard<std::mutex> lock(cache.mu);
        if (LaunchCache::MapEntry *e = LaunchCache::find(cache.maps, mk)) {
            e->used = ++cache.clock;
            std::memcpy(maps, e->maps, sizeof(maps));
            hit = true;
        }
    }
    if (hit) {
        g_map_hits.fetch_add(1, std::memory_order_relaxed);
    } else {
        g_map_misses.fetch_add(1, std::memory_order_relaxed);
        if (!encode_maps(pl, a, b, sfa, sfb, C, M, N, K, dtype_in, dtype_out, b_mn, maps))
            return GEMM_ERR_CUDA;
        std::lock_guard<std::mutex> lock(cache.mu);
        LaunchCache::MapEntry *e = LaunchCache::victim(cache.maps);
        e->key = mk;
        std::memcpy(e->maps, maps, sizeof(maps));
        e->used = ++cache.clock;
    }

    KernelParams kp = {};
    kp.M = static_cast<int32_t>(M);
    kp.N = static_cast<int32_t>(N);
    kp.K = static_cast<int32_t>(K);
    kp.num_m_tiles = pl.num_m;
    kp.num_n_tiles = pl.num_n;
    kp.num_tiles = pl.num_tiles;
    kp.num_k_blocks = pl.num_kb;
    kp.group_m = pl.group_m;
    if (kind_scaled(var.kind)) {
        // mxf8f6f4: E4M3 = 0, E5M2 = 1; mxf4: E2M1 = 1
        const uint32_t fmt = (dtype_in == GEMM_E5M2 || dtype_in == GEMM_E2M1) ? 1u : 0u;
        kp.idesc = make_idesc_mx(128u * var.cg, static_cast<uint32_t>(var.bn), fmt);
    } else {
        const uint32_t fmt = (dtype_in == GEMM_BF16 || dtype_in == GEMM_E5M2) ? 1u : 0u;
        kp.idesc = make_idesc(128u * var.cg, static_cast<uint32_t>(var.bn), fmt, b_mn ? 1u : 0u);
    }
    kp.out_dtype = dtype_out == GEMM_F32 ? OUT_F32 : (dtype_out == GEMM_BF16 ? OUT_BF16 : OUT_F16);
    kp.b_mn_major = b_mn ? 1u : 0u;
    kp.direct_store = pl.direct_store ? 1u : 0u;
    const Layout lay = layout_for(var, dtype_out);
    kp.stages = lay.stages;
    kp.staging_bytes = lay.staging_bytes;
    kp.staging_bufs = lay.staging_bufs;
    kp.C = C;
    kp.sk_tiles = pl.sk_tiles;
    if (pl.sk_tiles) {
        kp.flags = static_cast<unsigned long long *>(workspace);
        kp.partials = reinterpret_cast<float4 *>(static_cast<char *>(workspace) + sk_flag_bytes(pl.grid_ctas));
    }
    kp.timeout_ns = timeout_ms * 1000000ull;
    kp.launch_id = next_launch_id();
    kp.status = d.status;
    kp.trace = x.trace;
    kp.withhold_kb = x.withhold_kb;

    if (launch_any(var, pl.grid_ctas, pl.epi_warps, lay.smem, maps, kp, st) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return GEMM_OK;
}

// Repack one operand's scales (rows x ceil(K/32) bytes) into the kernel's
// atoms (see pack_scales_kernel) at dst.
gemm_status_t pack_scales(const uint8_t *sf, int64_t rows, int64_t K, const SfGeometry &g, int sms,
                          cudaStream_t st, void *dst)
{
    const int64_t total = g.atom_rows;
    const unsigned blocks = static_cast<unsigned>(
        std::max<int64_t>(std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(sms) * 8), 1));
    const int64_t nb = (K + 31) / 32;
    const int words = (nb % 4 == 0 && reinterpret_cast<uintptr_t>(sf) % 4 == 0) ? 1 : 0;
    pack_scales_kernel<<<blocks, 256, 0, st>>>(sf, static_cast<uint8_t *>(dst), rows, nb, g.R, g.row_blocks,
                                               g.stages, g.groups, g.atoms, words);
    if (cudaGetLastError() != cudaSuccess)
        return GEMM_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return GEMM_OK;
}

// Scratch of `need` bytes for one call on `st`: the stream's cached buffer
// (grown, when too small, by a stream-ordered free and allocation on `st`), or,
// inside a stream capture or beyond STREAM_SCRATCH_ENTRIES streams, a
// stream-ordered allocation that the caller frees after its launch
// (*per_call = true; in a capture it becomes the graph's own memory).
gemm_status_t acquire_scratch(DeviceState &d, cudaStream_t st, size_t need, void **out, bool *per_call)
{
    *out = nullptr;
    *per_call = false;
    if (need == 0)
        return GEMM_OK;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    unsigned long long id = 0;
    const bool cacheable = cudaStreamIsCapturing(st, &cap) == cudaSuccess && cap == cudaStreamCaptureStatusNone &&
                           cudaStreamGetId(st, &id) == cudaSuccess;
    if (!cacheable)
        cudaGetLastError();
    if (cacheable) {
        std::lock_guard<std::mutex> lock(d.scratch_mu);
        DeviceState::StreamScratch *e = nullptr, *empty = nullptr;
        for (DeviceState::StreamScratch &x : d.scratch) {
            if (x.used && x.stream_id == id) {
                e = &x;
                break;
            }
            if (!x.used && !empty)
                empty = &x;
        }
        if (!e && empty) {
            e = empty;
            e->used = true;
            e->stream_id = id;
            e->ptr = nullptr;
            e->bytes = 0;
        }
        if (e) {
            if (e->bytes < need) {
                // grow by at least a quarter, in 2 MiB steps
                const size_t step = size_t(2) << 20;
                const size_t want = std::max(need, e->bytes + e->bytes / 4);
                const size_t bytes = (want + step - 1) / step * step;
                if (e->ptr)
                    cudaFreeAsync(e->ptr, st);   // after every earlier call on this stream
                e->ptr = nullptr;
                e->bytes = 0;
                if (cudaMallocAsync(&e->ptr, bytes, st) != cudaSuccess) {
                    cudaGetLastError();
                    e->ptr = nullptr;
                    return GEMM_ERR_OUT_OF_MEMORY;
                }
                e->bytes = bytes;
            }
            *out = e->ptr;
            return GEMM_OK;
        }
    }
    if (cudaMallocAsync(out, need, st) != cudaSuccess) {
        cudaGetLastError();
        *out = nullptr;
        return GEMM_ERR_OUT_OF_MEMORY;
    }
    *per_call = true;
    return GEMM_OK;
}

gemm_status_t run(const void *A, const void *B, const uint8_t *SFA, const uint8_t *SFB, void *C, int64_t M,
                  int64_t N, int64_t K, int dtype_in, int dtype_out, int layoutA, int layoutB,
                  const gemm_options_t *opts, cudaStream_t st, int32_t withhold_kb = -1)
{
    const bool scaled = SFA != nullptr;
    gemm_status_t rc = validate(A, B, C, M, N, K, dtype_in, dtype_out, layoutA, layoutB, opts, scaled);
    if (rc != GEMM_OK)
        return rc;
    DeviceState *d = nullptr;
    if ((rc = device_state(&d)) != GEMM_OK)
        return rc;
    const PlanKey pk = plan_key(M, N, K, dtype_in, dtype_out, layoutB, scaled, A, B, C, opts);
    Plan pl;
    if ((rc = cached_plan(*d, pk, A, B, C, opts, &pl)) != GEMM_OK)
        return rc;
    if (withhold_kb >= pl.num_kb)
        return GEMM_ERR_INVALID_ARG;
    Extras x;
    x.trace = opts ? reinterpret_cast<unsigned long long *>(opts->clock_trace) : nullptr;
    x.withhold_kb = withhold_kb;
    const Variant &var = kVariants[pl.variant];
    const bool b_mn = layoutB == GEMM_MN_MAJOR;
    const int eb = tma_elem_bytes(var.kind);
    const int64_t a_width = row_bytes(var.kind, K) / eb;
    const int64_t b_rows = b_mn ? K : N, b_width = b_mn ? N : a_width;

    // One scratch area per call: stream-K partial sums and flags, then the
    // re-pitched A and B, then the packed scales, each on a 256-byte boundary.
    auto up256 = [](size_t v) { return (v + 255) / 256 * 256; };
    const int64_t lda_pad = padded_pitch(a_width, eb), ldb_pad = padded_pitch(b_width, eb);
    const size_t a_off = up256(pl.ws_bytes);
    const size_t a_bytes = pl.realign_a ? static_cast<size_t>(M) * lda_pad * eb : 0;
    const size_t b_off = a_off + up256(a_bytes);
    const size_t b_bytes = pl.realign_b ? static_cast<size_t>(b_rows) * ldb_pad * eb : 0;
    const size_t sf_off = b_off + up256(b_bytes);
    SfGeometry ga{}, gb{};
    size_t sfa_bytes = 0, sfb_off = 0, sf_bytes = 0;
    if (scaled) {
        ga = sf_geometry(var, pl, M, false);
        gb = sf_geometry(var, pl, N, true);
        sfa_bytes = static_cast<size_t>(ga.bytes());
        sfb_off = up256(sfa_bytes);
        sf_bytes = sfb_off + static_cast<size_t>(gb.bytes());
    }
    const size_t need = scaled ? sf_off + sf_bytes : (b_bytes ? b_off + b_bytes : (a_bytes ? a_off + a_bytes : pl.ws_bytes));
    void *scratch = nullptr;
    bool per_call = false;
    if ((rc = acquire_scratch(*d, st, need, &scratch, &per_call)) != GEMM_OK)
        return rc;
    char *base = static_cast<char *>(scratch);
    auto release = [&]() {
        if (per_call)
            cudaFreeAsync(scratch, st);
    };

    Operand a{A, a_width}, b{B, b_width};
    void *ws = pl.ws_bytes ? base : nullptr;
    if (pl.realign_a) {
        if ((rc = realign_into(A, M, a_width, lda_pad, eb, d->sms, st, base + a_off)) != GEMM_OK) {
            release();
            return rc;
        }
        a = {base + a_off, lda_pad};
    }
    if (pl.realign_b) {
        if ((rc = realign_into(B, b_rows, b_width, ldb_pad, eb, d->sms, st, base + b_off)) != GEMM_OK) {
            release();
            return rc;
        }
        b = {base + b_off, ldb_pad};
    }
    const void *sfa = nullptr, *sfb = nullptr;
    if (scaled) {
        sfa = base + sf_off;
        sfb = base + sf_off + sfb_off;
        if ((rc = pack_scales(SFA, M, K, ga, d->sms, st, const_cast<void *>(sfa))) != GEMM_OK ||
            (rc = pack_scales(SFB, N, K, gb, d->sms, st, const_cast<void *>(sfb))) != GEMM_OK) {
            release();
            return rc;
        }
    }

    const uint64_t timeout_ms = opts && opts->timeout_ms ? static_cast<uint64_t>(opts->timeout_ms)
                                                         : DEFAULT_TIMEOUT_MS;
    rc = encode_and_launch(*d, pk, pl, a, b, sfa, sfb, C, M, N, K, dtype_in, dtype_out, b_mn, timeout_ms, ws, x,
                           st);
    release();
    return rc;
}

} // namespace

extern "C" {

gemm_status_t gemm(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype_in,
                   gemm_dtype_t dtype_out, gemm_layout_t layoutA, gemm_layout_t layoutB, void *stream)
{
    return run(A, B, nullptr, nullptr, C, M, N, K, dtype_in, dtype_out, layoutA, layoutB, nullptr,
               static_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_ex(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                      gemm_dtype_t dtype_in, gemm_dtype_t dtype_out, gemm_layout_t layoutA, gemm_layout_t layoutB,
                      const gemm_options_t *opts, void *stream)
{
    return run(A, B, nullptr, nullptr, C, M, N, K, dtype_in, dtype_out, layoutA, layoutB, opts,
               static_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_mx(const void *A, const void *B, const uint8_t *SFA, const uint8_t *SFB, void *C, int64_t M,
                      int64_t N, int64_t K, gemm_dtype_t dtype_in, gemm_dtype_t dtype_out, gemm_layout_t layoutA,
                      gemm_layout_t layoutB, void *stream)
{
    if (!SFA || !SFB)
        return GEMM_ERR_INVALID_ARG;
    return run(A, B, SFA, SFB, C, M, N, K, dtype_in, dtype_out, layoutA, layoutB, nullptr,
               static_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_mx_ex(const void *A, const void *B, const uint8_t *SFA, const uint8_t *SFB, void *C,
                         int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                         gemm_layout_t layoutA, gemm_layout_t layoutB, const gemm_options_t *opts, void *stream)
{
    if (!SFA || !SFB)
        return GEMM_ERR_INVALID_ARG;
    return run(A, B, SFA, SFB, C, M, N, K, dtype_in, dtype_out, layoutA, layoutB, opts,
               static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

gemm_status_t plan_query(int64_t M, int64_t N, int64_t K, int dtype_in, int dtype_out, int layoutA, int layoutB,
                         const void *A, const void *B, const void *C, const gemm_options_t *opts, gemm_plan_t *plan,
                         bool scaled)
{
    if (!plan)
        return GEMM_ERR_INVALID_ARG;
    gemm_status_t rc = validate(A, B, C, M, N, K, dtype_in, dtype_out, layoutA, layoutB, opts, scaled);
    if (rc != GEMM_OK)
        return rc;
    DeviceState *d = nullptr;
    if ((rc = device_state(&d)) != GEMM_OK)
        return rc;
    Plan pl;
    const PlanKey pk = plan_key(M, N, K, dtype_in, dtype_out, layoutB, scaled, A, B, C, opts);
    if ((rc = cached_plan(*d, pk, A, B, C, opts, &pl)) != GEMM_OK)
        return rc;
    const Variant &var = kVariants[pl.variant];
    std::memset(plan, 0, sizeof(*plan));
    plan->cta_group = var.cg;
    plan->block_m = 128 * var.cg;
    plan->block_n = var.bn;
    plan->block_k = kind_slab_k(var.kind) * var.ks;
    const Layout lay = layout_for(var, dtype_out);
    plan->stages = static_cast<int32_t>(lay.stages);
    plan->num_tiles = static_cast<int32_t>(static_cast<int64_t>(pl.num_m) * ((N + var.bn - 1) / var.bn));
    plan->grid_ctas = pl.grid_ctas;
    plan->group_m = pl.group_m;
    plan->realign_a = pl.realign_a;
    plan->realign_b = pl.realign_b;
    plan->direct_store = pl.direct_store;
    plan->smem_bytes = static_cast<int32_t>(lay.smem);
    plan->num_sms = d->sms;
    plan->sk_tiles = pl.sk_tiles;
    plan->workspace_bytes = static_cast<int32_t>(pl.ws_bytes);
    plan->cluster_pairs = var.mc;
    plan->epilogue_warps = pl.epi_warps;
    return GEMM_OK;
}

} // namespace

extern "C" {

gemm_status_t gemm_plan(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                        gemm_layout_t layoutA, gemm_layout_t layoutB, const void *A, const void *B, const void *C,
                        const gemm_options_t *opts, gemm_plan_t *plan)
{
    return plan_query(M, N, K, dtype_in, dtype_out, layoutA, layoutB, A, B, C, opts, plan, false);
}

gemm_status_t gemm_mx_plan(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                           gemm_layout_t layoutA, gemm_layout_t layoutB, const void *A, const void *B, const void *C,
                           const gemm_options_t *opts, gemm_plan_t *plan)
{
    return plan_query(M, N, K, dtype_in, dtype_out, layoutA, layoutB, A, B, C, opts, plan, true);
}

gemm_status_t gemm_from_host_async(const void *A_host, const void *B_host, void *C_host, int64_t M, int64_t N,
                                   int64_t K, gemm_dtype_t dtype_in, gemm_dtype_t dtype_out, gemm_layout_t layoutA,
                                   gemm_layout_t layoutB, void *stream)
{
    gemm_status_t rc = validate(A_host, B_host, C_host, M, N, K, dtype_in, dtype_out, layoutA, layoutB,
                                nullptr);
    if (rc != GEMM_OK)
        return rc;
    DeviceState *d = nullptr;
    if ((rc = device_state(&d)) != GEMM_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto up256 = [](size_t x) { return (x + 255) / 256 * 256; };
    const int kind = kind_for(dtype_in, false);
    const size_t a_bytes = static_cast<size_t>(M * row_bytes(kind, K));
    const size_t b_bytes = static_cast<size_t>(layoutB == GEMM_MN_MAJOR ? K * row_bytes(kind, N) : N * row_bytes(kind, K));
    const size_t c_bytes = static_cast<size_t>(M * N * out_bytes(dtype_out));
    const size_t need = up256(a_bytes) + up256(b_bytes) + up256(c_bytes);
    std::lock_guard<std::mutex> lock(d->ws_mu);
    auto cuda_failed = [](cudaError_t e) {
        if (e == cudaSuccess)
            return false;
        cudaGetLastError();
        return true;
    };
    if (!d->h2d && cuda_failed(cudaStreamCreateWithFlags(&d->h2d, cudaStreamNonBlocking)))
        return GEMM_ERR_CUDA;
    DeviceState::HostSlot &slot = d->slots[d->next_slot];
    if (!slot.uploaded && (cuda_failed(cudaEventCreateWithFlags(&slot.uploaded, cudaEventDisableTiming)) ||
                           cuda_failed(cudaEventCreateWithFlags(&slot.released, cudaEventDisableTiming))))
        return GEMM_ERR_CUDA;
    if (slot.bytes < need) {
        // the slot's previous call must be done with it before it is replaced
        if (slot.used && cuda_failed(cudaEventSynchronize(slot.released)))
            return GEMM_ERR_CUDA;
        if (slot.ws) {
            cudaFree(slot.ws);
            slot.ws = nullptr;
            slot.bytes = 0;
        }
        if (cudaMalloc(&slot.ws, need) != cudaSuccess) {
            cudaGetLastError();
            slot.ws = nullptr;
            return GEMM_ERR_OUT_OF_MEMORY;
        }
        slot.bytes = need;
        slot.used = false;
    }
    char *dA = static_cast<char *>(slot.ws);
    char *dB = dA + up256(a_bytes);
    char *dC = dB + up256(b_bytes);
    // uploads on the library's copy stream, once the slot's previous product and read-back are done
    if ((slot.used && cuda_failed(cudaStreamWaitEvent(d->h2d, slot.released, 0))) ||
        cuda_failed(cudaMemcpyAsync(dA, A_host, a_bytes, cudaMemcpyHostToDevice, d->h2d)) ||
        cuda_failed(cudaMemcpyAsync(dB, B_host, b_bytes, cudaMemcpyHostToDevice, d->h2d)) ||
        cuda_failed(cudaEventRecord(slot.uploaded, d->h2d)) || cuda_failed(cudaStreamWaitEvent(st, slot.uploaded, 0)))
        return GEMM_ERR_CUDA;
    // the product and the read-back on the caller's stream
    rc = run(dA, dB, nullptr, nullptr, dC, M, N, K, dtype_in, dtype_out, layoutA, layoutB, nullptr, st);
    if (rc != GEMM_OK)
        return rc;
    if (cuda_failed(cudaMemcpyAsync(C_host, dC, c_bytes, cudaMemcpyDeviceToHost, st)) ||
        cuda_failed(cudaEventRecord(slot.released, st)))
        return GEMM_ERR_CUDA;
    slot.used = true;
    d->next_slot ^= 1u;
    return GEMM_OK;
}

gemm_status_t gemm_from_host(const void *A_host, const void *B_host, void *C_host, int64_t M, int64_t N,
                             int64_t K, gemm_dtype_t dtype_in, gemm_dtype_t dtype_out, gemm_layout_t layoutA,
                             gemm_layout_t layoutB, void *stream)
{
    gemm_status_t rc = gemm_from_host_async(A_host, B_host, C_host, M, N, K, dtype_in, dtype_out, layoutA,
                                            layoutB, stream);
    if (rc != GEMM_OK)
        return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

gemm_status_t gemm_release_workspace(void)
{
    DeviceState *d = nullptr;
    gemm_status_t rc = device_state(&d);
    if (rc != GEMM_OK)
        return rc;
    std::lock_guard<std::mutex> lock(d->ws_mu);
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    for (DeviceState::HostSlot &slot : d->slots) {
        if (slot.ws && cudaFree(slot.ws) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        slot.ws = nullptr;
        slot.bytes = 0;
        slot.used = false;
    }
    {
        std::lock_guard<std::mutex> slock(d->scratch_mu);
        for (DeviceState::StreamScratch &e : d->scratch) {
            if (e.ptr && cudaFree(e.ptr) != cudaSuccess) {
                cudaGetLastError();
                return GEMM_ERR_CUDA;
            }
            e = DeviceState::StreamScratch{};
        }
    }
    g_cache[d->dev].clear();
    return GEMM_OK;
}

void gemm_cache_stats(uint64_t *plan_hits, uint64_t *plan_misses, uint64_t *map_hits, uint64_t *map_misses)
{
    if (plan_hits)
        *plan_hits = g_plan_hits.load(std::memory_order_relaxed);
    if (plan_misses)
        *plan_misses = g_plan_misses.load(std::memory_order_relaxed);
    if (map_hits)
        *map_hits = g_map_hits.load(std::memory_order_relaxed);
    if (map_misses)
        *map_misses = g_map_misses.load(std::memory_order_relaxed);
}

gemm_status_t gemm_cache_clear(void)
{
    DeviceState *d = nullptr;
    const gemm_status_t rc = device_state(&d);
    if (rc != GEMM_OK)
        return rc;
    g_cache[d->dev].clear();
    return GEMM_OK;
}

gemm_status_t gemm_last_device_status(void *stream, uint32_t *detail)
{
    if (detail)
        *detail = 0;
    DeviceState *d = nullptr;
    gemm_status_t rc = device_state(&d);
    if (rc != GEMM_OK)
        return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    unsigned long long h[4] = {0, 0, 0, 0};
    if (cudaMemcpyFromSymbol(h, g_status, sizeof(h)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (h[0] == 0)
        return GEMM_OK;
    const unsigned long long zero[4] = {0, 0, 0, 0};
    if (cudaMemcpyToSymbol(g_status, zero, sizeof(zero)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (detail)
        *detail = static_cast<uint32_t>(h[1]);
    return GEMM_ERR_TIMEOUT;
}

gemm_status_t gemm_selftest_wait_timeout(int32_t timeout_ms, void *stream)
{
    if (timeout_ms < 1 || timeout_ms > 10000)
        return GEMM_ERR_INVALID_ARG;
    DeviceState *d = nullptr;
    gemm_status_t rc = device_state(&d);
    if (rc != GEMM_OK)
        return rc;
    wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint64_t>(timeout_ms) * 1000000ull, next_launch_id(), d->status);
    if (cudaGetLastError() != cudaSuccess)
        return GEMM_ERR_CUDA;
    return GEMM_OK;
}

gemm_status_t gemm_selftest_withheld_load(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                                          gemm_dtype_t dtype_in, gemm_dtype_t dtype_out, gemm_layout_t layoutB,
                                          int32_t cta_group, int32_t withhold_kb, int32_t timeout_ms, void *stream)
{
    if (timeout_ms < 1 || timeout_ms > 10000 || withhold_kb < 0 || (cta_group != 1 && cta_group != 2))
        return GEMM_ERR_INVALID_ARG;
    gemm_options_t o = {};
    o.cta_group = cta_group;
    o.timeout_ms = timeout_ms;
    o.stream_k = 1;   // whole tiles: unit 0's first job is a full tile
    return run(A, B, nullptr, nullptr, C, M, N, K, dtype_in, dtype_out, GEMM_K_MAJOR, layoutB, &o,
               static_cast<cudaStream_t>(stream), withhold_kb);
}

const char *gemm_status_string(gemm_status_t status)
{
    switch (status) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
    case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
    case GEMM_ERR_NO_DEVICE: return "GEMM_ERR_NO_DEVICE";
    case GEMM_ERR_OUT_OF_MEMORY: return "GEMM_ERR_OUT_OF_MEMORY";
    default: return "GEMM_ERR_UNKNOWN";
    }
}

uint64_t gemm_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

gemm_status_t gemm_schedule_jobs(int32_t num_tiles, int32_t units, int32_t k_blocks, int32_t sk_tiles,
                                 int32_t unit, gemm_job_t *jobs, int32_t max_jobs, int32_t *n_jobs)
{
    if (num_tiles < 1 || units < 1 || unit < 0 || unit >= units || k_blocks < 1 || sk_tiles < 0 ||
        sk_tiles > num_tiles || (!jobs && max_jobs > 0) || !n_jobs)
        return GEMM_ERR_INVALID_ARG;
    const UnitSchedule sch(unit, units, num_tiles, k_blocks, sk_tiles);
    const int32_t n = sch.num_jobs();
    for (int32_t i = 0; i < n && i < max_jobs; ++i) {
        const Job j = sch.job(i);
        jobs[i] = {j.tile, j.kb0, j.kb1, j.kind};
    }
    *n_jobs = n;
    return GEMM_OK;
}

} // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point (gemm_no_alloc).
//
// For callers that cannot allocate device memory, for example a serving
// runtime that has given all of the GPU's memory to its own pool, or a
// latency-critical loop where cudaMalloc/cudaFree could synchronise the device
// or fail. gemm allocates stream-ordered scratch for the re-pitched copy of a
// misaligned A or B and for the stream-K partial sums and flags. Here both go
// into this fixed array, held on every GPU that loads the library until the
// process exits (or, when the partial sums do not fit, the plan keeps every
// tile whole). Host code must not use
// the name g_no_alloc_scratch as a device address: it stands for a host-side
// shadow. The device address comes from cudaGetSymbolAddress, looked up once
// per device with that device current.
static __device__ __align__(256) unsigned char g_no_alloc_scratch[GEMM_NO_ALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_no_alloc_mu;
void *g_no_alloc_ptr[MAX_DEVICES] = {};

// Device address of g_no_alloc_scratch on the current device (first call per
// device: cudaGetSymbolAddress, return code checked).
gemm_status_t no_alloc_scratch(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_no_alloc_mu);
    if (!g_no_alloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        g_no_alloc_ptr[dev] = p;
    }
    *out = g_no_alloc_ptr[dev];
    return GEMM_OK;
}

gemm_status_t run_no_alloc(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                           int dtype_in, int dtype_out, int layoutA, int layoutB, cudaStream_t st)
{
    gemm_status_t rc = validate(A, B, C, M, N, K, dtype_in, dtype_out, layoutA, layoutB, nullptr);
    if (rc != GEMM_OK)
        return rc;
    DeviceState *d = nullptr;
    if ((rc = device_state(&d)) != GEMM_OK)
        return rc;
    // the array's address is looked up on every device's first call, whether or
    // not that call needs it, so that a later call inside a stream capture never does
    void *scratch = nullptr;
    if ((rc = no_alloc_scratch(&scratch)) != GEMM_OK)
        return rc;
    PlanKey pk = plan_key(M, N, K, dtype_in, dtype_out, layoutB, false, A, B, C, nullptr);
    Plan pl;
    if ((rc = cached_plan(*d, pk, A, B, C, nullptr, &pl)) != GEMM_OK)
        return rc;
    const bool b_mn = layoutB == GEMM_MN_MAJOR;
    const int kind = kind_for(dtype_in, false);
    const int eb = tma_elem_bytes(kind);

    // Scratch layout: padded A at offset 0, padded B and then the stream-K
    // workspace, each at the next 256-byte boundary.
    const int64_t a_cols = row_bytes(kind, K) / eb;
    const int64_t b_rows = b_mn ? K : N, b_cols = b_mn ? N : a_cols;
    const int64_t lda_pad = padded_pitch(a_cols, eb), ldb_pad = padded_pitch(b_cols, eb);
    const uint64_t a_bytes = pl.realign_a ? static_cast<uint64_t>(M) * lda_pad * eb : 0;
    const uint64_t b_off = (a_bytes + 255) / 256 * 256;
    const uint64_t b_bytes = pl.realign_b ? static_cast<uint64_t>(b_rows) * ldb_pad * eb : 0;
    if (b_off + b_bytes > GEMM_NO_ALLOC_SCRATCH_BYTES)
        return GEMM_ERR_UNSUPPORTED;   // padded operands exceed the fixed scratch array
    const uint64_t ws_off = (b_off + b_bytes + 255) / 256 * 256;
    if (pl.sk_tiles && ws_off + pl.ws_bytes > GEMM_NO_ALLOC_SCRATCH_BYTES) {
        // no room for the partial sums: keep every tile whole
        gemm_options_t dp = {};
        dp.stream_k = 1;
        pk = plan_key(M, N, K, dtype_in, dtype_out, layoutB, false, A, B, C, &dp);
        if ((rc = cached_plan(*d, pk, A, B, C, &dp, &pl)) != GEMM_OK)
            return rc;
    }

    Operand a{A, a_cols}, b{B, b_cols};
    void *ws = nullptr;
    if (pl.realign_a || pl.realign_b || pl.sk_tiles) {
        char *base = static_cast<char *>(scratch);
        if (pl.sk_tiles)
            ws = base + ws_off;
        if (pl.realign_a) {
            if ((rc = realign_into(A, M, a_cols, lda_pad, eb, d->sms, st, base)) != GEMM_OK)
                return rc;
            a = {base, lda_pad};
        }
        if (pl.realign_b) {
            if ((rc = realign_into(B, b_rows, b_cols, ldb_pad, eb, d->sms, st, base + b_off)) != GEMM_OK)
                return rc;
            b = {base + b_off, ldb_pad};
        }
    }
    return encode_and_launch(*d, pk, pl, a, b, nullptr, nullptr, C, M, N, K, dtype_in, dtype_out, b_mn,
                             DEFAULT_TIMEOUT_MS, ws, Extras{}, st);
}

} // namespace

// ---------------------------------------------------------------------------
// Services for the library's other translation units (runtime.h).
namespace dtg {

gemm_status_t runtime_info(RuntimeInfo *out)
{
    DeviceState *d = nullptr;
    const gemm_status_t rc = device_state(&d);
    if (rc != GEMM_OK)
        return rc;
    out->status = d->status;
    out->sms = d->sms;
    return GEMM_OK;
}

unsigned long long runtime_next_launch_id() { return next_launch_id(); }

void runtime_count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

bool runtime_encode(CUtensorMap *map, CUtensorMapDataType dt, uint32_t rank, const void *base,
                    const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                    CUtensorMapSwizzle swizzle)
{
    if (!g_encode || rank < 1 || rank > 5)
        return false;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], es[5];
    for (uint32_t i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank)
            st[i] = strides_bytes[i];
    }
    return g_encode(map, dt, rank, const_cast<void *>(base), d, st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

} // namespace dtg

extern "C" gemm_status_t gemm_no_alloc(const void *A, const void *B, void *C, int64_t M, int64_t N,
                                       int64_t K, gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                                       gemm_layout_t layoutA, gemm_layout_t layoutB, void *stream)
{
    return run_no_alloc(A, B, C, M, N, K, dtype_in, dtype_out, layoutA, layoutB,
                        static_cast<cudaStream_t>(stream));
}

extern "C" gemm_status_t gemm_no_alloc_scratch(void **ptr, size_t *bytes)
{
    if (!ptr || !bytes)
        return GEMM_ERR_INVALID_ARG;
    *ptr = nullptr;
    *bytes = 0;
    void *p = nullptr;
    const gemm_status_t rc = no_alloc_scratch(&p);
    if (rc != GEMM_OK)
        return rc;
    *ptr = p;
    *bytes = GEMM_NO_ALLOC_SCRATCH_BYTES;
    return GEMM_OK;
}
