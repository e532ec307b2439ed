// Explicit instantiations of the kernel templates for one (input, output)
// dtype pair.  Included by the per-pair translation units, which define
// RMSN_TI / RMSN_TO (types), RMSN_DTI / RMSN_DTO (DType codes) and
// RMSN_TABLE_FN (the table accessor declared in rmsn_registry.h).  For an
// fp32 residual stream under bf16 / fp16 activations they also define
// RMSN_TX (the activation type; RMSN_TI is then F32), RMSN_RF32 1 and
// RMSN_RES_ONLY.
#include "rmsn_kernels.cuh"

namespace rmsn {

#ifndef RMSN_TX
#define RMSN_TX RMSN_TI  // activations stored like the residual stream
#endif
#ifndef RMSN_RF32
#define RMSN_RF32 0
#endif

#define RMSN_VEC(CH, WMAX, WR, RES, BIAS)                                                    \
    {RMSN_DTI, RMSN_DTO, (WR) ? kWarpRows : kBlockRow, CH, WMAX, 0, RES, BIAS, RMSN_RF32,    \
     (const void*)&rmsn_vec_kernel<RMSN_TI, RMSN_TO, CH, WMAX, WR, RES, BIAS, RMSN_TX>}
#ifdef RMSN_RES_ONLY
#define RMSN_VEC4(CH, WMAX, WR) RMSN_VEC(CH, WMAX, WR, true, false), RMSN_VEC(CH, WMAX, WR, true, true)
#else
#define RMSN_VEC4(CH, WMAX, WR)                                                              \
    RMSN_VEC(CH, WMAX, WR, false, false), RMSN_VEC(CH, WMAX, WR, true, false),               \
        RMSN_VEC(CH, WMAX, WR, false, true), RMSN_VEC(CH, WMAX, WR, true, true)
#endif
#define RMSN_BULK(CH, WMAX, RES, BIAS)                                                       \
    {RMSN_DTI, RMSN_DTO, kBulkRow, CH, WMAX, 0, RES, BIAS, RMSN_RF32,                        \
     (const void*)&rmsn_bulk_kernel<RMSN_TI, RMSN_TO, CH, WMAX, RES, BIAS, RMSN_TX>}
#ifdef RMSN_RES_ONLY
#define RMSN_BULK4(CH, WMAX) RMSN_BULK(CH, WMAX, true, false), RMSN_BULK(CH, WMAX, true, true)
#else
#define RMSN_BULK4(CH, WMAX)                                                                 \
    RMSN_BULK(CH, WMAX, false, false), RMSN_BULK(CH, WMAX, true, false),                     \
        RMSN_BULK(CH, WMAX, false, true), RMSN_BULK(CH, WMAX, true, true)
#endif
#define RMSN_CLU(CH, K, RES, BIAS)                                                          \
    {RMSN_DTI, RMSN_DTO, kCluster, CH, K, 0, RES, BIAS, RMSN_RF32,                            \
     (const void*)&rmsn_cluster_kernel<RMSN_TI, RMSN_TO, CH, RES, BIAS>}
#define RMSN_CLU4(CH, K)                                                                     \
    RMSN_CLU(CH, K, false, false), RMSN_CLU(CH, K, true, false), RMSN_CLU(CH, K, false, true), \
        RMSN_CLU(CH, K, true, true)
#define RMSN_PIPE(CH, WMAX, RES, BIAS)                                                      \
    {RMSN_DTI, RMSN_DTO, kBulkPipe, CH, WMAX, 0, RES, BIAS, RMSN_RF32,                        \
     (const void*)&rmsn_bulk_kernel<RMSN_TI, RMSN_TO, CH, WMAX, RES, BIAS, RMSN_TX, true>}
#define RMSN_PIPE4(CH, WMAX)                                                                 \
    RMSN_PIPE(CH, WMAX, false, false), RMSN_PIPE(CH, WMAX, true, false),                     \
        RMSN_PIPE(CH, WMAX, false, true), RMSN_PIPE(CH, WMAX, true, true)
#define RMSN_GEN(RES)                                                                        \
    {RMSN_DTI, RMSN_DTO, kGeneric, 0, 8, 0, RES, -1, RMSN_RF32,                              \
     (const void*)&rmsn_generic_kernel<RMSN_TI, RMSN_TO, RES, RMSN_TX>}

static const KernelEntry kTable[] = {
    // decode: one warp per row; blocks of 1 or 4 warps
    RMSN_VEC4(1, 1, true), RMSN_VEC4(2, 1, true), RMSN_VEC4(4, 1, true), RMSN_VEC4(8, 1, true),
    RMSN_VEC4(1, 4, true), RMSN_VEC4(2, 4, true), RMSN_VEC4(4, 4, true), RMSN_VEC4(8, 4, true),
    // prefill: one block per row, up to WMAX warps
    RMSN_VEC4(1, 4, false), RMSN_VEC4(2, 4, false), RMSN_VEC4(4, 4, false),
    RMSN_VEC4(1, 8, false), RMSN_VEC4(2, 8, false), RMSN_VEC4(4, 8, false),
    RMSN_VEC4(1, 16, false), RMSN_VEC4(2, 16, false), RMSN_VEC4(4, 16, false),
    RMSN_VEC4(1, 32, false), RMSN_VEC4(2, 32, false),
#ifndef RMSN_NO_BULK
    // prefill: rows streamed through shared memory by bulk async copies
    RMSN_BULK4(1, 8), RMSN_BULK4(2, 8), RMSN_BULK4(1, 16), RMSN_BULK4(2, 16),
    RMSN_BULK4(1, 32), RMSN_BULK4(2, 32),
#endif
#ifdef RMSN_WITH_PIPE
    // prefill, per-token FP8 / NVFP4: the ring with two rows in flight per barrier
    RMSN_PIPE4(1, 8), RMSN_PIPE4(2, 8), RMSN_PIPE4(1, 16), RMSN_PIPE4(2, 16),
#endif
#ifdef RMSN_WITH_CLUSTER
    // decode: one row split over a cluster of K one-warp blocks
    RMSN_CLU4(1, 2), RMSN_CLU4(1, 4), RMSN_CLU4(1, 8), RMSN_CLU4(2, 2), RMSN_CLU4(2, 4),
    RMSN_CLU4(2, 8), RMSN_CLU4(4, 2), RMSN_CLU4(4, 4),
#endif
#ifndef RMSN_NO_GENERIC
    // any shape
#ifndef RMSN_RES_ONLY
    RMSN_GEN(false),
#endif
    RMSN_GEN(true),
#endif
};

const KernelEntry* RMSN_TABLE_FN(int* n) {
    *n = (int)(sizeof(kTable) / sizeof(kTable[0]));
    return kTable;
}

}  // namespace rmsn
