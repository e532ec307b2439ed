// Kernel instantiations: bf16 input, NVFP4 block-scaled output
// (vector kernels only: the block formats need whole 32-byte vectors).
#define RMSN_TI ::rmsn::BF16
#define RMSN_TO ::rmsn::NVFP4
#define RMSN_DTI kBF16
#define RMSN_DTO kNVFP4
#define RMSN_TABLE_FN kernels_bf16_nvfp4
#define RMSN_NO_GENERIC
#define RMSN_WITH_PIPE
#include "rmsn_instances.cuh"
