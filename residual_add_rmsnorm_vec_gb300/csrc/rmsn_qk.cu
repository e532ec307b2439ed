// QK norm: per-head RMS norm of the query and key heads, in place (blog
// "CuTeDSL at Perplexity", section "QK norm").  Each head of head_dim
// elements is normalised on its own with the query or the key weight plus the
// scalar WEIGHT_BIAS, and written back in the element type.
//
// Layout on GB300: a head is held by TPH consecutive lanes, one 32-byte
// vector each (16 bf16 / 8 fp32; the blog uses 16-byte vectors on Hopper), so
// a warp carries 32 / TPH heads and the head's sum of squares needs only a
// butterfly over TPH lanes (log2(TPH) shuffles): no shared memory, no block
// barrier.  The query heads and then the key heads of a token are split into
// warps of 32 / TPH heads, so one launch covers both.  q and k may live inside
// a fused qkv row (token stride larger than heads * head_dim); nothing outside
// the heads is touched.
#include "rmsn_kernels.cuh"
#include "rmsn_qk.h"

namespace rmsn {

// rsqrt(sum / D + eps), the mean square correctly rounded.  For a power-of-two
// D, sum * (1 / D) is that same correctly rounded quotient (scaling by a power
// of two is exact), one multiply instead of a division.
__device__ __forceinline__ float qk_inv(float acc, const QkArgs& a) {
    const float ms = a.rcp_d > 0.f ? __fmul_rn(acc, a.rcp_d) : __fdiv_rn(acc, (float)a.D);
    return __frsqrt_rn(__fadd_rn(ms, a.eps));
}

// y = (w + woff) * (x * inv) for one vector.  Without an offset, 16-bit x and
// w: y = RN(p * inv) with p = x w formed exactly (one rounding, and the 16-bit
// lanes go straight into the FMAs); else the roundings of the listing, two
// lanes per instruction.
template <class TI>
__device__ __forceinline__ void qk_scale(const V8& x, const V8& w, float inv, float woff,
                                         float (&y)[32 / TI::kBytes]) {
    if constexpr (TI::kBytes == 2) {
        if (woff == 0.f) {
            const F2 inv2 = f2(inv, inv);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                f2split(mul2(mul16x2_exact<TI>(x.u[k], w.u[k]), inv2), y[2 * k], y[2 * k + 1]);
            return;
        }
    }
    float m = 0.f;
    scale_vec<TI, false>(x, w, w, inv, woff, y, m);
}

// This lane's sum of squares of one vector (fp32, in element order).
template <class TI>
__device__ __forceinline__ float qk_sumsq(const V8& x) {
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if constexpr (TI::kBytes == 2) {
            acc = sumsq16x2<TI>(x.u[k], acc);
        } else {
            const float h = __uint_as_float(x.u[k]);
            acc = __fmaf_rn(h, h, acc);
        }
    }
    return acc;
}

// Elements [e, e + n) inside the span of q (is_q) or k: (T - 1) * stride +
// heads * head_dim elements (the bounds-checked build's test).
__device__ __forceinline__ bool qk_in_span(const QkArgs& a, bool is_q, int64_t e, int n) {
    const int64_t ext = is_q ? (a.T - 1) * a.qs + (int64_t)a.Hq * a.D
                             : (a.T - 1) * a.ks + (int64_t)a.Hk * a.D;
    return e >= 0 && e + n <= ext;
}

// One block per U tokens and group of heads: warp w of block (b, g) holds
// heads (g W + w) NH .. + NH - 1 (NH = 32 / TPH, W warps per block) of tokens
// b U .. b U + U - 1, so a lane finds its head with a few multiply-adds, loads
// its U vectors and the weight's, and the block is done after one pass.  Many
// short blocks keep more reads in flight across the GPU than a persistent
// grid looping over heads (measured on GB300: 6.8 against 6.3 TB/s for an
// in-place pass over the same bytes); U = 2 puts two tokens' reads in flight
// per lane for long batches (at 16384 tokens of 32 + 8 heads x 128: 49.8
// against 53.5 us with one).  Tokens beyond the grid's x extent are taken by a
// stride loop (uniform across the warp, so every lane reaches every shuffle).
template <class TI, int TPH, int U>
__global__ void __launch_bounds__(512) rmsn_qk_kernel(const QkArgs a) {
    constexpr int VE = 32 / TI::kBytes;
    constexpr int NH = 32 / TPH;  // heads per warp
    pdl_launch_dependents(a.pdl);
    const int lane = threadIdx.x & 31;
    const int sub = lane % TPH;  // this lane's vector within its head
    const int hh = ((int)blockIdx.y * (int)(blockDim.x >> 5) + (int)(threadIdx.x >> 5)) * NH +
                   lane / TPH;  // head within the token
    const bool is_q = hh < a.Hq;
    const bool lane_on = hh < a.Hq + a.Hk && sub < a.nvec;
    void* row = is_q ? a.q : a.k;
    const int64_t ts = is_q ? a.qs : a.ks;
    const int64_t off = (int64_t)(is_q ? hh : hh - a.Hq) * a.D + (int64_t)sub * VE;
    const void* w = is_q ? a.qw : a.kw;
    pdl_wait(a.pdl);
    V8 wv;
    if (lane_on && w) {
        wv = ld_keep32(static_cast<const char*>(w) + (int64_t)sub * 32);
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) wv.u[k] = ones_word<TI>();
    }
    for (int64_t t0 = (int64_t)blockIdx.x * U; t0 < a.T; t0 += (int64_t)gridDim.x * U) {
        V8 x[U];
        bool act[U];
        float acc[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int64_t e = (t0 + j) * ts + off;
            act[j] = lane_on && t0 + j < a.T &&
                     RMSN_CHECK(a.status, qk_in_span(a, is_q, e, VE) &&
                                              (sub + 1) * 32 <= a.D * TI::kBytes);
            if (act[j]) x[j] = ld_stream32(static_cast<const char*>(row) + e * TI::kBytes);
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
            acc[j] = act[j] ? qk_sumsq<TI>(x[j]) : 0.f;
#pragma unroll
            for (int o = TPH / 2; o > 0; o >>= 1)
                acc[j] += __shfl_xor_sync(0xFFFFFFFFu, acc[j], o);
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
            if (act[j]) {
                float y[VE];
                qk_scale<TI>(x[j], wv, qk_inv(acc[j], a), a.woff, y);
                store_out<TI, TI>(row, (t0 + j) * ts + off, y, 0.f);
            }
        }
    }
}

// A 32-byte vector from shared memory, its halves read in the order that
// keeps a quarter warp's 16-byte loads on distinct banks (lanes 4-7 of each
// 8 start with the upper half).
__device__ __forceinline__ V8 ld_shared32_lanes(uint32_t addr) {
    const uint32_t sw = (threadIdx.x & 4u) << 2;  // 16 or 0
    uint32_t p[4], q[4];
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(p[0]), "=r"(p[1]), "=r"(p[2]), "=r"(p[3])
                 : "r"(addr + sw));
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3])
                 : "r"(addr + (sw ^ 16u)));
    V8 v;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        v.u[k] = sw ? q[k] : p[k];
        v.u[4 + k] = sw ? p[k] : q[k];
    }
    return v;
}

// ---------------------------------------------------------------- ring variant
//
// For long batches (opt-in, RMSN_QK_RING): persistent blocks, each taking
// tokens blockIdx.x + k * gridDim.x.  Thread 0 copies the query heads and
// the key heads of TPS consecutive tokens of the block (two 1-D bulk copies
// per token, TMA, completing on the stage's mbarrier) into one buffer of a
// ring of `stages` shared-memory buffers, up to `stages` buffers ahead;
// thread t holds the 32-byte vectors v = c * G + t (c < CH) of every token,
// so its weight vectors are the same for the whole launch and are loaded once
// into registers.  A head's TPH vectors sit on TPH neighbouring lanes (G is a
// multiple of 32 and TPH divides 32), so its sum of squares is a butterfly
// over those lanes; the normalised vectors are stored straight back in
// place.  Each lane reads its vector's two 16-byte halves in a lane-dependent
// order, so the 8 lanes of a quarter warp meet 32 different banks.  One block
// barrier per buffer (TPS = 2 tokens with one vector per thread) releases it,
// and thread 0 refills it.  Waits are bounded as in the row kernel's ring:
// one that runs out sets bit 0 of the status word, the block stops after the
// buffer's barrier, and thread 0 drains its copies in flight (default bound).

template <class TI, int TPH, int CH>
__global__ void __launch_bounds__(1024, 1) rmsn_qk_ring_kernel(const QkArgs a) {
    constexpr int VE = 32 / TI::kBytes;
    constexpr int TPS = CH == 1 ? 2 : 1;  // tokens per buffer
    extern __shared__ __align__(128) unsigned char qring[];
    __shared__ __align__(8) uint64_t full[kMaxStages];
    __shared__ int abort_flag;
    const int t = threadIdx.x;
    const int G = blockDim.x;
    const int S = a.stages;
    const int hv = a.nvec;                                // vectors per head
    const uint32_t qbytes = (uint32_t)a.Hq * a.D * TI::kBytes;
    const uint32_t kbytes = (uint32_t)a.Hk * a.D * TI::kBytes;
    const uint32_t tok_bytes = qbytes + kbytes;
    const uint32_t stage_bytes = TPS * tok_bytes;
    const int nvq = (int)(qbytes / 32), nv = (int)(tok_bytes / 32);
    const uint32_t ring0 = smem_u32(qring);
    const int64_t n_my = a.T > blockIdx.x ? (a.T - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int64_t n_buf = (n_my + TPS - 1) / TPS;  // buffers this block fills
    pdl_launch_dependents(a.pdl);
    if (t == 0) {
        abort_flag = 0;
        for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // this thread's weight vectors (query or key weight, vector index in the head)
    V8 wv[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const int v = c * G + t;
        const bool is_q = v < nvq;
        const void* w = is_q ? a.qw : a.kw;
        const int sub = (is_q ? v : v - nvq) % hv;
        if (v < nv && w) {
            wv[c] = ld_keep32(static_cast<const char*>(w) + (int64_t)sub * 32);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) wv[c].u[k] = ones_word<TI>();
        }
    }
    // thread 0: copy the tokens of buffer b (the block's tokens b * TPS ..)
    // into the stage at `dst`
    auto issue = [&](int64_t b, uint32_t dst, uint32_t bar) {
        const int64_t first = b * TPS;
        const int ntok = (int)(n_my - first < TPS ? n_my - first : TPS);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                     "r"((uint32_t)ntok * tok_bytes)
                     : "memory");
        for (int j = 0; j < ntok; ++j) {
            const int64_t tok = blockIdx.x + (first + j) * gridDim.x;
            const uint32_t d = dst + (uint32_t)j * tok_bytes;
            if (qbytes) {
                const char* src = static_cast<const char*>(a.q) + tok * a.qs * TI::kBytes;
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], "
                    "[%1], %2, [%3];" ::"r"(d), "l"(src), "r"(qbytes), "r"(bar)
                    : "memory");
            }
            if (kbytes) {
                const char* src = static_cast<const char*>(a.k) + tok * a.ks * TI::kBytes;
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], "
                    "[%1], %2, [%3];" ::"r"(d + qbytes), "l"(src), "r"(kbytes), "r"(bar)
                    : "memory");
            }
        }
    };
    pdl_wait(a.pdl);
    if (t == 0)
        for (int64_t b = 0; b < S && b < n_buf; ++b)
            issue(b, ring0 + (uint32_t)b * stage_bytes, smem_u32(&full[b]));
    __syncthreads();
    int64_t b_abort = 0;
    for (int64_t b = 0; b < n_buf; ++b) {
        const int s = (int)(b % S);
        const uint32_t phase = (uint32_t)((b / S) & 1);
        b_abort = b;
        if (!mbar_wait_bounded(smem_u32(&full[s]), phase, a.wait_cycles)) {
            atomicOr(a.status, 1u);
            abort_flag = 1;
        }
        const uint32_t base = ring0 + (uint32_t)s * stage_bytes;
        const int ntok = (int)(n_my - b * TPS < TPS ? n_my - b * TPS : TPS);
        V8 x[TPS][CH];
        float acc[TPS][CH];
#pragma unroll
        for (int j = 0; j < TPS; ++j) {
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const int v = c * G + t;
                acc[j][c] = 0.f;
                if (v < nv && j < ntok) {
                    x[j][c] = ld_shared32_lanes(base + (uint32_t)j * tok_bytes + (uint32_t)v * 32u);
                    acc[j][c] = qk_sumsq<TI>(x[j][c]);
                }
            }
        }
        // every thread has read the buffer: it may be refilled after this barrier
        __syncthreads();
        if (abort_flag) break;
        if (t == 0 && b + S < n_buf) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(b + S, base, smem_u32(&full[s]));
        }
#pragma unroll
        for (int j = 0; j < TPS; ++j) {
            const int64_t tok = blockIdx.x + (b * TPS + j) * gridDim.x;
#pragma unroll
            for (int c = 0; c < CH; ++c) {
#pragma unroll
                for (int o = TPH / 2; o > 0; o >>= 1)
                    acc[j][c] += __shfl_xor_sync(0xFFFFFFFFu, acc[j][c], o);
                const int v = c * G + t;
                if (v >= nv || j >= ntok) continue;
                const float inv = qk_inv(acc[j][c], a);
                const bool is_q = v < nvq;
                void* row = is_q ? a.q : a.k;
                const int64_t e = is_q ? tok * a.qs + (int64_t)v * VE
                                       : tok * a.ks + (int64_t)(v - nvq) * VE;
                if (!RMSN_CHECK(a.status, qk_in_span(a, is_q, e, VE))) continue;
                float y[VE];
                qk_scale<TI>(x[j][c], wv[c], inv, a.woff, y);
                store_out<TI, TI>(row, e, y, 0.f);
            }
        }
    }
    if (abort_flag && t == 0) {
        for (int64_t j = b_abort; j < b_abort + S && j < n_buf; ++j)
            mbar_wait_bounded(smem_u32(&full[j % S]), (uint32_t)((j / S) & 1),
                              kDefaultWaitCycles);
    }
}

#define RMSN_QK(TI, DT, TPH)                                            \
    {DT, TPH, kQkDirect, 1, (const void*)&rmsn_qk_kernel<TI, TPH, 1>}, \
        {DT, TPH, kQkDirect, 2, (const void*)&rmsn_qk_kernel<TI, TPH, 2>}
#define RMSN_QKR(TI, DT, TPH, CH) \
    {DT, TPH, kQkBlockRing, CH, (const void*)&rmsn_qk_ring_kernel<TI, TPH, CH>}

static const QkEntry kQkTable[] = {
    RMSN_QK(BF16, kBF16, 1), RMSN_QK(BF16, kBF16, 2),  RMSN_QK(BF16, kBF16, 4),
    RMSN_QK(BF16, kBF16, 8), RMSN_QK(BF16, kBF16, 16), RMSN_QK(BF16, kBF16, 32),
    RMSN_QK(F32, kF32, 1),   RMSN_QK(F32, kF32, 2),    RMSN_QK(F32, kF32, 4),
    RMSN_QK(F32, kF32, 8),   RMSN_QK(F32, kF32, 16),   RMSN_QK(F32, kF32, 32),
    RMSN_QK(F16, kF16, 1),   RMSN_QK(F16, kF16, 2),    RMSN_QK(F16, kF16, 4),
    RMSN_QK(F16, kF16, 8),   RMSN_QK(F16, kF16, 16),   RMSN_QK(F16, kF16, 32),
    // ring variant: head_dim 64 / 128 / 256 / 512 in 16-bit types, 32 .. 256 in fp32
    RMSN_QKR(BF16, kBF16, 4, 1),  RMSN_QKR(BF16, kBF16, 8, 1),  RMSN_QKR(BF16, kBF16, 16, 1),
    RMSN_QKR(BF16, kBF16, 32, 1), RMSN_QKR(BF16, kBF16, 4, 2),  RMSN_QKR(BF16, kBF16, 8, 2),
    RMSN_QKR(BF16, kBF16, 16, 2), RMSN_QKR(BF16, kBF16, 32, 2),
    RMSN_QKR(F16, kF16, 4, 1),    RMSN_QKR(F16, kF16, 8, 1),    RMSN_QKR(F16, kF16, 16, 1),
    RMSN_QKR(F16, kF16, 32, 1),   RMSN_QKR(F16, kF16, 4, 2),    RMSN_QKR(F16, kF16, 8, 2),
    RMSN_QKR(F16, kF16, 16, 2),   RMSN_QKR(F16, kF16, 32, 2),
    RMSN_QKR(F32, kF32, 4, 1),    RMSN_QKR(F32, kF32, 8, 1),    RMSN_QKR(F32, kF32, 16, 1),
    RMSN_QKR(F32, kF32, 32, 1),   RMSN_QKR(F32, kF32, 4, 2),    RMSN_QKR(F32, kF32, 8, 2),
    RMSN_QKR(F32, kF32, 16, 2),   RMSN_QKR(F32, kF32, 32, 2),
};

const QkEntry* qk_kernels(int* n) {
    *n = (int)(sizeof(kQkTable) / sizeof(kQkTable[0]));
    return kQkTable;
}

}  // namespace rmsn
