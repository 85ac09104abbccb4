// runtime.h: library-internal services shared by the translation units of
// libdtgemm.so (defined in gemm.cu): the per-device state, the device status
// word, launch ids and launch counting, and tensor-map encoding.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "gemm.h"

namespace dtg {

struct RuntimeInfo {
    unsigned long long *status;   // device status word of the current device
    int sms;                      // multiprocessors on the current device
};

// The current device's state (sm_103 check, status word, SM count).
gemm_status_t runtime_info(RuntimeInfo *out);

// A fresh launch id (never 0) for the device status word and stream-K flags.
unsigned long long runtime_next_launch_id();

// Count one kernel launch of this library (gemm_launch_count).
void runtime_count_launch();

// cuTensorMapEncodeTiled with interleave none, 256-byte L2 promotion and zero
// fill. dims/box have `rank` entries (innermost first); strides_bytes has
// rank - 1 entries. Returns false when the encoding is refused.
bool runtime_encode(CUtensorMap *map, CUtensorMapDataType dt, uint32_t rank, const void *base,
                    const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                    CUtensorMapSwizzle swizzle);

} // namespace dtg
