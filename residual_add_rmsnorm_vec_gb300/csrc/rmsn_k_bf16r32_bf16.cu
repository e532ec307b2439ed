// Kernel instantiations: bf16 activations with an fp32 residual stream,
// bf16 output (register kernels, residual variants only).
#define RMSN_TI ::rmsn::F32
#define RMSN_TX ::rmsn::BF16
#define RMSN_TO ::rmsn::BF16
#define RMSN_DTI kBF16
#define RMSN_DTO kBF16
#define RMSN_RF32 1
#define RMSN_RES_ONLY
#define RMSN_TABLE_FN kernels_bf16r32_bf16
#include "rmsn_instances.cuh"
