// Instantiations of the ragged-row kernel (rmsn_ragged_kernel): bf16, fp16
// and fp32 rows, the same dtype in and out, CH 16-byte vectors per thread
// (1, 2, 4, 8: up to 2048 vectors per row), with and without residual and
// bias.
#include "rmsn_kernels.cuh"

namespace rmsn {

#define RMSN_RAG(TI, DT, CH, RES, BIAS) \
    {DT, DT, kRagged, CH, 8, 0, RES, BIAS, 0, (const void*)&rmsn_ragged_kernel<TI, TI, CH, RES, BIAS>}
#define RMSN_RAG4(TI, DT, CH)                                                        \
    RMSN_RAG(TI, DT, CH, false, false), RMSN_RAG(TI, DT, CH, true, false),           \
        RMSN_RAG(TI, DT, CH, false, true), RMSN_RAG(TI, DT, CH, true, true)
#define RMSN_RAG_ALL(TI, DT) \
    RMSN_RAG4(TI, DT, 1), RMSN_RAG4(TI, DT, 2), RMSN_RAG4(TI, DT, 4), RMSN_RAG4(TI, DT, 8)

static const KernelEntry kTable[] = {
    RMSN_RAG_ALL(BF16, kBF16),
    RMSN_RAG_ALL(F16, kF16),
    RMSN_RAG_ALL(F32, kF32),
};

const KernelEntry* kernels_ragged(int* n) {
    *n = (int)(sizeof(kTable) / sizeof(kTable[0]));
    return kTable;
}

}  // namespace rmsn
