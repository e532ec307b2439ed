// Kernel instantiations: f32 input, bf16 output.
#define RMSN_TI ::rmsn::F32
#define RMSN_TO ::rmsn::BF16
#define RMSN_DTI kF32
#define RMSN_DTO kBF16
#define RMSN_TABLE_FN kernels_f32_bf16
#include "rmsn_instances.cuh"
