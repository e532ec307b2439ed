// QK norm: per-head RMS norm of the query and key heads, in place (blog
// "CuTeDSL at Perplexity", section "QK norm").  Each head of head_dim
// elements is normalised on its own with the query or the key weight plus the
// scalar WEIGHT_BIAS, and written back in the element type.
//
// Layout on GB300: a head is held by TPH consecutive lanes, one 32-byte
// vector each (16 bf16 / 8 fp32; the blog uses 16-byte vectors on Hopper), so
// a warp carries 32 / TPH heads and the head's sum of squares needs only a
// butterfly over TPH lanes (log2(TPH) shuffles): no shared memory, no block
// barrier.  Query and key heads of all tokens form one index space, so one
// launch covers both.  q and k may live inside a fused qkv row (token stride
// larger than heads * head_dim); nothing outside the heads is touched.
#include "rmsn_kernels.cuh"
#include "rmsn_qk.h"

namespace rmsn {

template <class TI, int TPH>
__global__ void __launch_bounds__(256) rmsn_qk_kernel(const QkArgs a) {
    constexpr int VE = 32 / TI::kBytes;
    pdl_launch_dependents(a.pdl);
    pdl_wait(a.pdl);
    const int lane = threadIdx.x & 31;
    const int sub = lane % TPH;  // this lane's vector within its head
    const int64_t heads = a.Hq + a.Hk;
    const int64_t nh = a.T * heads;
    const int64_t step = (int64_t)gridDim.x * blockDim.x / TPH;
    // the warp's first head: the loop bound is uniform across the warp, so
    // every lane reaches every shuffle
    for (int64_t base = ((int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31)) / TPH;
         base < nh; base += step) {
        const int64_t head = base + lane / TPH;
        const bool valid = head < nh;
        const int64_t tok = valid ? head / heads : 0;
        const int hh = valid ? (int)(head % heads) : 0;
        const bool is_q = hh < a.Hq;
        void* row = is_q ? a.q : a.k;
        const int64_t e0 = is_q ? tok * a.qs + (int64_t)hh * a.D
                                : tok * a.ks + (int64_t)(hh - a.Hq) * a.D;
        const int64_t e = e0 + (int64_t)sub * VE;
        // elements of q (k) the heads span: (T - 1) * stride + heads * head_dim
        const int64_t ext = is_q ? (a.T - 1) * a.qs + (int64_t)a.Hq * a.D
                                 : (a.T - 1) * a.ks + (int64_t)a.Hk * a.D;
        const bool act = valid && sub < a.nvec &&
                         RMSN_CHECK(a.status, e >= 0 && e + VE <= ext &&
                                                  (sub + 1) * 32 <= a.D * TI::kBytes);
        V8 x;
        float acc = 0.f;
        if (act) {
            x = ld_stream32(static_cast<const char*>(row) + e * TI::kBytes);
#pragma unroll
            for (int k = 0; k < VE; ++k) {
                const float h = elem<TI>(x, k);
                acc = __fmaf_rn(h, h, acc);
            }
        }
#pragma unroll
        for (int o = TPH / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
        const float inv = inv_rms(acc, a.D, a.eps);
        if (act) {
            const void* w = is_q ? a.qw : a.kw;
            V8 wv;
            if (w) {
                wv = ld_keep32(static_cast<const char*>(w) + (int64_t)sub * 32);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) wv.u[k] = ones_word<TI>();
            }
            float y[VE];
#pragma unroll
            for (int k = 0; k < VE; ++k)
                y[k] = scale_elem<false>(elem<TI>(x, k), inv, elem<TI>(wv, k), a.woff, 0.f);
            store_out<TI, TI>(row, e, y, 0.f);
        }
    }
}

#define RMSN_QK(TI, DT, TPH) {DT, TPH, (const void*)&rmsn_qk_kernel<TI, TPH>}

static const QkEntry kQkTable[] = {
    RMSN_QK(BF16, kBF16, 1), RMSN_QK(BF16, kBF16, 2),  RMSN_QK(BF16, kBF16, 4),
    RMSN_QK(BF16, kBF16, 8), RMSN_QK(BF16, kBF16, 16), RMSN_QK(BF16, kBF16, 32),
    RMSN_QK(F32, kF32, 1),   RMSN_QK(F32, kF32, 2),    RMSN_QK(F32, kF32, 4),
    RMSN_QK(F32, kF32, 8),   RMSN_QK(F32, kF32, 16),   RMSN_QK(F32, kF32, 32),
    RMSN_QK(F16, kF16, 1),   RMSN_QK(F16, kF16, 2),    RMSN_QK(F16, kF16, 4),
    RMSN_QK(F16, kF16, 8),   RMSN_QK(F16, kF16, 16),   RMSN_QK(F16, kF16, 32),
};

const QkEntry* qk_kernels(int* n) {
    *n = (int)(sizeof(kQkTable) / sizeof(kQkTable[0]));
    return kQkTable;
}

}  // namespace rmsn
