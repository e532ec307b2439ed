// Kernel instantiations: f16 input, fp8 output.
#define RMSN_TI ::rmsn::F16
#define RMSN_TO ::rmsn::FP8
#define RMSN_DTI kF16
#define RMSN_DTO kFP8
#define RMSN_TABLE_FN kernels_f16_fp8
#define RMSN_WITH_PIPE
#include "rmsn_instances.cuh"
