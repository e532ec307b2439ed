// QK-norm kernel table shared by its instantiation unit and the C-ABI layer.
#pragma once

#include <stdint.h>

namespace rmsn {

// Kernel arguments (by value).  q / k: first element of token 0's first head;
// qs / ks: token strides in elements; weights [D] or NULL (1).
struct QkArgs {
    void* q;
    void* k;
    const void* qw;
    const void* kw;
    int64_t T;
    int64_t qs, ks;
    int32_t Hq, Hk, D;
    int32_t nvec;  // 32-byte vectors per head
    float eps;
    float woff;
    int32_t pdl;   // launched as a programmatic dependent
    uint32_t* status;  // device status word (bit 0: a bounded wait ran out; bit 1: a
                       // bounds check failed, checked build)
    float rcp_d;          // 1 / head_dim when head_dim is a power of two (exact), else 0
    int32_t stages;       // ring kernel: shared-memory token buffers
    int64_t wait_cycles;  // ring kernel: bound of a token wait (< 0: test once)
};

enum QkKind : int32_t { kQkDirect = 0, kQkBlockRing = 1 };

struct QkEntry {
    int32_t dt;    // DType of q, k and the weights
    int32_t tph;   // lanes per head
    int32_t kind;  // QkKind
    int32_t ch;    // block ring: vectors per thread; one-pass kernel: tokens per block
    const void* fn;
};

const QkEntry* qk_kernels(int* n);

}  // namespace rmsn
