// Kernel instantiations: f16 activations with an fp32 residual stream,
// f16 output (register kernels, residual variants only).
#define RMSN_TI ::rmsn::F32
#define RMSN_TX ::rmsn::F16
#define RMSN_TO ::rmsn::F16
#define RMSN_DTI kF16
#define RMSN_DTO kF16
#define RMSN_RF32 1
#define RMSN_RES_ONLY
#define RMSN_TABLE_FN kernels_f16r32_f16
#include "rmsn_instances.cuh"
