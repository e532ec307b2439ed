// Kernel instantiations: f16 input, f32 output.
#define RMSN_TI ::rmsn::F16
#define RMSN_TO ::rmsn::F32
#define RMSN_DTI kF16
#define RMSN_DTO kF32
#define RMSN_TABLE_FN kernels_f16_f32
#include "rmsn_instances.cuh"
