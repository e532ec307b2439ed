// Instantiations of the ragged-row kernel (rmsn_ragged_kernel) with a
// per-token FP8-E4M3 output: bf16, fp16 and fp32 rows, CH 16-byte vectors per
// thread (1, 2, 4, 8: up to 2048 vectors per row), with and without residual
// and bias.
#include "rmsn_kernels.cuh"

namespace rmsn {

#define RMSN_RAGQ(TI, DT, CH, RES, BIAS)                                     \
    {DT, kFP8, kRagged, CH, 8, 0, RES, BIAS, 0,                               \
     (const void*)&rmsn_ragged_kernel<TI, FP8, CH, RES, BIAS>}
#define RMSN_RAGQ4(TI, DT, CH)                                                        \
    RMSN_RAGQ(TI, DT, CH, false, false), RMSN_RAGQ(TI, DT, CH, true, false),           \
        RMSN_RAGQ(TI, DT, CH, false, true), RMSN_RAGQ(TI, DT, CH, true, true)
#define RMSN_RAGQ_ALL(TI, DT) \
    RMSN_RAGQ4(TI, DT, 1), RMSN_RAGQ4(TI, DT, 2), RMSN_RAGQ4(TI, DT, 4), RMSN_RAGQ4(TI, DT, 8)

static const KernelEntry kTable[] = {
    RMSN_RAGQ_ALL(BF16, kBF16),
    RMSN_RAGQ_ALL(F16, kF16),
    RMSN_RAGQ_ALL(F32, kF32),
};

const KernelEntry* kernels_ragged_fp8(int* n) {
    *n = (int)(sizeof(kTable) / sizeof(kTable[0]));
    return kTable;
}

}  // namespace rmsn
