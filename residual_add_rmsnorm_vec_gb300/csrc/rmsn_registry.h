// Kernel registry shared by the instantiation units and the C-ABI layer.
#pragma once

#include <stdint.h>

namespace rmsn {

// Kernel arguments (passed by value).  Pointers are device pointers; `b` is
// NULL when there is no bias; `nvec` = hidden / elements per 32-byte vector.
struct RmsnArgs {
    const void* x;
    const void* r;
    const void* w;
    const void* b;
    void* out;
    void* res_out;
    float* scale;   // per-token fp32 scale (FP8, NVFP4)
    void* bscale;   // block scales (MXFP8 / MXFP4: E8M0 per 32; NVFP4: E4M3 per 16)
    int64_t T;
    int32_t H;
    int32_t nvec;
    float eps;
    float woff;
    int32_t has_w;
    int32_t stages;      // shared-memory row buffers (bulk kernel)
    int32_t pdl;           // launched as a programmatic dependent
    int32_t early_params;  // weight / bias may be read before the prerequisite grid ends
    int32_t swz;           // bulk kernel: stages filled by 128-byte-swizzled tensor copies
    uint32_t* status;    // device status word: bit 0 = a bounded wait ran out
    int64_t wait_cycles;  // bound of the ring's row waits in clock cycles; < 0: probe the
                          // barrier once without waiting (tests of the expiry path)
};

// Default bound of a ring wait: about one second of SM clock cycles.
constexpr int64_t kDefaultWaitCycles = 2000000000LL;

enum DType : int32_t {
    kF32 = 0, kBF16 = 1, kFP8 = 2, kMXFP8 = 3, kMXFP4 = 4, kNVFP4 = 5, kF16 = 6
};

enum Variant : int32_t {
    kWarpRows = 0, kBlockRow = 1, kBulkRow = 2, kGeneric = 3, kRagged = 4, kCluster = 5,
    kBulkPipe = 6  // the ring kernel with its two-row pipeline (per-token FP8, NVFP4)
};

// One compiled kernel.  For kCluster, max_warps holds the cluster size (blocks
// of one warp per row).
struct KernelEntry {
    int32_t in_dt, out_dt, variant, chunks, max_warps, stages, res, bias;
    int32_t res_f32;  // fp32 residual stream under a bf16 / fp16 in_dt
    const void* fn;
};

// Each instantiation unit returns its table.
const KernelEntry* kernels_f32_f32(int* n);
const KernelEntry* kernels_f32_bf16(int* n);
const KernelEntry* kernels_f32_fp8(int* n);
const KernelEntry* kernels_bf16_f32(int* n);
const KernelEntry* kernels_bf16_bf16(int* n);
const KernelEntry* kernels_bf16_fp8(int* n);
const KernelEntry* kernels_f16_f16(int* n);
const KernelEntry* kernels_f16_f32(int* n);
const KernelEntry* kernels_f16_fp8(int* n);
const KernelEntry* kernels_f32_f16(int* n);
const KernelEntry* kernels_bf16r32_bf16(int* n);
const KernelEntry* kernels_bf16r32_fp8(int* n);
const KernelEntry* kernels_f16r32_f16(int* n);
const KernelEntry* kernels_f16r32_fp8(int* n);
const KernelEntry* kernels_bf16_mxfp8(int* n);
const KernelEntry* kernels_bf16_mxfp4(int* n);
const KernelEntry* kernels_bf16_nvfp4(int* n);
const KernelEntry* kernels_ragged(int* n);
const KernelEntry* kernels_ragged_fp8(int* n);
const KernelEntry* kernels_ragged_mixed(int* n);

}  // namespace rmsn
