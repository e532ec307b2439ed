// Kernel instantiations: bf16 input, f32 output.
#define RMSN_TI ::rmsn::BF16
#define RMSN_TO ::rmsn::F32
#define RMSN_DTI kBF16
#define RMSN_DTO kF32
#define RMSN_TABLE_FN kernels_bf16_f32
#include "rmsn_instances.cuh"
