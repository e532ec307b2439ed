// Kernel instantiations: f32 input, f16 output.
#define RMSN_TI ::rmsn::F32
#define RMSN_TO ::rmsn::F16
#define RMSN_DTI kF32
#define RMSN_DTO kF16
#define RMSN_TABLE_FN kernels_f32_f16
#include "rmsn_instances.cuh"
