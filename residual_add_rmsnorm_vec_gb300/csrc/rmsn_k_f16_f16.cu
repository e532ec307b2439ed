// Kernel instantiations: f16 input, f16 output.
#define RMSN_TI ::rmsn::F16
#define RMSN_TO ::rmsn::F16
#define RMSN_DTI kF16
#define RMSN_DTO kF16
#define RMSN_TABLE_FN kernels_f16_f16
#define RMSN_WITH_CLUSTER
#include "rmsn_instances.cuh"
