// Kernel instantiations: bf16 input, fp8 output.
#define RMSN_TI ::rmsn::BF16
#define RMSN_TO ::rmsn::FP8
#define RMSN_DTI kBF16
#define RMSN_DTO kFP8
#define RMSN_TABLE_FN kernels_bf16_fp8
#define RMSN_WITH_PIPE
#include "rmsn_instances.cuh"
