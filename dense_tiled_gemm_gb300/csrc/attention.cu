// attention.cu: host side of attention_fwd (include/attention.h).
//
// One launch of attention_fwd_kernel per call: a persistent grid of one CTA
// per SM (at most one per row block; ceil(Lq / 256) row blocks of two
// 128-row tiles per head), 320 threads and ~192 KB of shared memory per CTA,
// with programmatic stream serialisation like the GEMM. The tensor maps
// view Q, K and V as 3-D (d, rows, B * H) so that a tile never reads into
// the next head: rows past Lq or Lk come back as zeros.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "attention.h"
#include "attention_kernel.cuh"
#include "runtime.h"

using namespace dtg;

namespace {

constexpr uint64_t ATT_TIMEOUT_MS = 2000;

std::mutex g_att_mu;
bool g_att_ready[64] = {};

gemm_status_t prepare_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_att_mu);
    if (!g_att_ready[dev]) {
        if (cudaFuncSetAttribute(attention_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(ATT_SMEM)) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        g_att_ready[dev] = true;
    }
    return GEMM_OK;
}

bool map_3d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, int64_t rows, int64_t bh, uint32_t box_rows)
{
    const uint64_t dims[3] = {static_cast<uint64_t>(ATT_D), static_cast<uint64_t>(rows), static_cast<uint64_t>(bh)};
    const uint64_t strides[2] = {ATT_D * 2ull, static_cast<uint64_t>(rows) * ATT_D * 2ull};
    const uint32_t box[3] = {64u, box_rows, 1u};
    return runtime_encode(m, dt, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

} // namespace

extern "C" gemm_status_t attention_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
                                       int64_t B, int64_t H, int64_t Lq, int64_t Lk, int64_t d, int dtype,
                                       int causal, float scale, void *stream)
{
    return attention_fwd_ex(Q, K, V, O, LSE, B, H, Lq, Lk, d, dtype, causal, scale, 0, stream);
}

extern "C" gemm_status_t attention_fwd_ex(const void *Q, const void *K, const void *V, void *O, float *LSE,
                                          int64_t B, int64_t H, int64_t Lq, int64_t Lk, int64_t d, int dtype,
                                          int causal, float scale, int max_ctas, void *stream)
{
    if (!Q || !K || !V || !O)
        return GEMM_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || Lq < 1 || Lk < 1 || d < 1 || Lq > INT32_MAX / 2 || Lk > INT32_MAX / 2)
        return GEMM_ERR_INVALID_ARG;
    if (dtype != GEMM_F16 && dtype != GEMM_BF16)
        return dtype == GEMM_F32 ? GEMM_ERR_UNSUPPORTED : GEMM_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1)
        return GEMM_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.0f))
        return GEMM_ERR_INVALID_ARG;
    // heads index a 1-D persistent grid's row blocks and a tensor map dimension (int32)
    if (d != ATT_D || B > INT32_MAX || H > INT32_MAX || B * H > INT32_MAX)
        return GEMM_ERR_UNSUPPORTED;
    for (const void *ptr : {Q, K, V, const_cast<const void *>(O)})
        if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0)
            return GEMM_ERR_UNSUPPORTED;
    if (LSE && reinterpret_cast<uintptr_t>(LSE) % 4 != 0)
        return GEMM_ERR_INVALID_ARG;

    RuntimeInfo rt;
    gemm_status_t rc = runtime_info(&rt);
    if (rc != GEMM_OK)
        return rc;
    if ((rc = prepare_device()) != GEMM_OK)
        return rc;

    const int64_t bh = B * H;
    const CUtensorMapDataType dt = dtype == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    alignas(64) CUtensorMap tq, tk, tv;
    if (!map_3d(&tq, dt, Q, Lq, bh, ATT_BM) || !map_3d(&tk, dt, K, Lk, bh, ATT_BN) || !map_3d(&tv, dt, V, Lk, bh, 64))
        return GEMM_ERR_CUDA;

    AttParams p = {};
    p.Lq = static_cast<int32_t>(Lq);
    p.Lk = static_cast<int32_t>(Lk);
    p.BH = static_cast<int32_t>(bh);
    p.nq = static_cast<int32_t>((Lq + ATT_ROWS - 1) / ATT_ROWS);
    p.causal = static_cast<uint32_t>(causal);
    p.bf16 = dtype == GEMM_BF16 ? 1u : 0u;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);   // log2(e)
    const uint32_t fmt = p.bf16;
    p.idesc_qk = make_idesc(ATT_BM, ATT_BN, fmt, 0u);   // S = Q K^T: both K-major
    p.idesc_pv = make_idesc(ATT_BM, ATT_D, fmt, 1u);    // O += P V: V is N-contiguous
    p.O = O;
    p.LSE = LSE;
    p.timeout_ns = ATT_TIMEOUT_MS * 1000000ull;
    p.launch_id = runtime_next_launch_id();
    p.status = rt.status;

    cudaLaunchConfig_t cfg = {};
    // persistent: one CTA per SM, each walking row blocks blockIdx.x + k * gridDim.x
    int64_t ctas = std::min<int64_t>(static_cast<int64_t>(p.nq) * bh, rt.sms);
    if (max_ctas > 0)
        ctas = std::min<int64_t>(ctas, max_ctas);
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(ATT_THREADS);
    cfg.dynamicSmemBytes = ATT_SMEM;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, attention_fwd_kernel, tq, tk, tv, p) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    runtime_count_launch();
    return GEMM_OK;
}
