// Instantiations of the ragged-row kernel (rmsn_ragged_kernel) whose output
// dtype differs from the rows': fp32 out from bf16 / fp16 rows, bf16 / fp16
// out from fp32 rows; CH 16-byte vectors per thread (1, 2, 4, 8), with and
// without residual and bias.
#include "rmsn_kernels.cuh"

namespace rmsn {

#define RMSN_RAGM(TI, DTI, TO, DTO, CH, RES, BIAS) \
    {DTI, DTO, kRagged, CH, 8, 0, RES, BIAS, 0, (const void*)&rmsn_ragged_kernel<TI, TO, CH, RES, BIAS>}
#define RMSN_RAGM4(TI, DTI, TO, DTO, CH)                                                       \
    RMSN_RAGM(TI, DTI, TO, DTO, CH, false, false), RMSN_RAGM(TI, DTI, TO, DTO, CH, true, false), \
        RMSN_RAGM(TI, DTI, TO, DTO, CH, false, true), RMSN_RAGM(TI, DTI, TO, DTO, CH, true, true)
#define RMSN_RAGM_ALL(TI, DTI, TO, DTO)                                               \
    RMSN_RAGM4(TI, DTI, TO, DTO, 1), RMSN_RAGM4(TI, DTI, TO, DTO, 2),                 \
        RMSN_RAGM4(TI, DTI, TO, DTO, 4), RMSN_RAGM4(TI, DTI, TO, DTO, 8)

static const KernelEntry kTable[] = {
    RMSN_RAGM_ALL(BF16, kBF16, F32, kF32),
    RMSN_RAGM_ALL(F16, kF16, F32, kF32),
    RMSN_RAGM_ALL(F32, kF32, BF16, kBF16),
    RMSN_RAGM_ALL(F32, kF32, F16, kF16),
};

const KernelEntry* kernels_ragged_mixed(int* n) {
    *n = (int)(sizeof(kTable) / sizeof(kTable[0]));
    return kTable;
}

}  // namespace rmsn
