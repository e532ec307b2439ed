// Kernel instantiations: f32 input, fp8 output.
#define RMSN_TI ::rmsn::F32
#define RMSN_TO ::rmsn::FP8
#define RMSN_DTI kF32
#define RMSN_DTO kFP8
#define RMSN_TABLE_FN kernels_f32_fp8
#include "rmsn_instances.cuh"
