// Kernel instantiations: f32 input, f32 output.
#define RMSN_TI ::rmsn::F32
#define RMSN_TO ::rmsn::F32
#define RMSN_DTI kF32
#define RMSN_DTO kF32
#define RMSN_TABLE_FN kernels_f32_f32
#define RMSN_WITH_CLUSTER
#include "rmsn_instances.cuh"
