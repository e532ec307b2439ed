// Kernel instantiations: bf16 input, bf16 output.
#define RMSN_TI ::rmsn::BF16
#define RMSN_TO ::rmsn::BF16
#define RMSN_DTI kBF16
#define RMSN_DTO kBF16
#define RMSN_TABLE_FN kernels_bf16_bf16
#define RMSN_WITH_CLUSTER
#include "rmsn_instances.cuh"
