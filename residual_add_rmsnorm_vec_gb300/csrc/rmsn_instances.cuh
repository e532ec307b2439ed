// Explicit instantiations of the kernel templates for one (input, output)
// dtype pair.  Included by the per-pair translation units, which define
// RMSN_TI / RMSN_TO (types), RMSN_DTI / RMSN_DTO (DType codes) and
// RMSN_TABLE_FN (the table accessor declared in rmsn_registry.h).
#include "rmsn_kernels.cuh"

namespace rmsn {

#define RMSN_VEC(CH, WMAX, WR, RES, BIAS)                                                    \
    {RMSN_DTI, RMSN_DTO, (WR) ? kWarpRows : kBlockRow, CH, WMAX, 0, RES, BIAS,               \
     (const void*)&rmsn_vec_kernel<RMSN_TI, RMSN_TO, CH, WMAX, WR, RES, BIAS>}
#define RMSN_VEC4(CH, WMAX, WR)                                                              \
    RMSN_VEC(CH, WMAX, WR, false, false), RMSN_VEC(CH, WMAX, WR, true, false),               \
        RMSN_VEC(CH, WMAX, WR, false, true), RMSN_VEC(CH, WMAX, WR, true, true)
#define RMSN_BULK(CH, WMAX, RES, BIAS)                                                       \
    {RMSN_DTI, RMSN_DTO, kBulkRow, CH, WMAX, 0, RES, BIAS,                                   \
     (const void*)&rmsn_bulk_kernel<RMSN_TI, RMSN_TO, CH, WMAX, RES, BIAS>}
#define RMSN_BULK4(CH, WMAX)                                                                 \
    RMSN_BULK(CH, WMAX, false, false), RMSN_BULK(CH, WMAX, true, false),                     \
        RMSN_BULK(CH, WMAX, false, true), RMSN_BULK(CH, WMAX, true, true)
#define RMSN_GEN(RES)                                                                        \
    {RMSN_DTI, RMSN_DTO, kGeneric, 0, 8, 0, RES, -1,                                         \
     (const void*)&rmsn_generic_kernel<RMSN_TI, RMSN_TO, RES>}

static const KernelEntry kTable[] = {
    // decode: one warp per row; blocks of 1 or 4 warps
    RMSN_VEC4(1, 1, true), RMSN_VEC4(2, 1, true), RMSN_VEC4(4, 1, true), RMSN_VEC4(8, 1, true),
    RMSN_VEC4(1, 4, true), RMSN_VEC4(2, 4, true), RMSN_VEC4(4, 4, true), RMSN_VEC4(8, 4, true),
    // prefill: one block per row, up to WMAX warps
    RMSN_VEC4(1, 4, false), RMSN_VEC4(2, 4, false), RMSN_VEC4(4, 4, false),
    RMSN_VEC4(1, 8, false), RMSN_VEC4(2, 8, false), RMSN_VEC4(4, 8, false),
    RMSN_VEC4(1, 16, false), RMSN_VEC4(2, 16, false), RMSN_VEC4(4, 16, false),
    RMSN_VEC4(1, 32, false), RMSN_VEC4(2, 32, false),
    // prefill: rows streamed through shared memory by bulk async copies
    RMSN_BULK4(1, 8), RMSN_BULK4(2, 8), RMSN_BULK4(1, 16), RMSN_BULK4(2, 16),
    RMSN_BULK4(1, 32), RMSN_BULK4(2, 32),
#ifndef RMSN_NO_GENERIC
    // any shape
    RMSN_GEN(false), RMSN_GEN(true),
#endif
};

const KernelEntry* RMSN_TABLE_FN(int* n) {
    *n = (int)(sizeof(kTable) / sizeof(kTable[0]));
    return kTable;
}

}  // namespace rmsn
