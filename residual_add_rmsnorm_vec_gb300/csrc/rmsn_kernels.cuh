// Device code of the fused residual-add + RMSNorm for sm_103a.
//
// The operation is the regular RMS norm of the blog "CuTeDSL at Perplexity"
// (section "QK norm": fp32 sum of squares, reciprocal square root of the mean
// square plus EPS, times the weight plus the scalar WEIGHT_BIAS, cast to the
// element type), fused with the residual add, an optional per-channel bias
// and an optional per-token FP8-E4M3 absmax output (section "Blackwell
// support").  Layout choices follow the same blog, section "Prefill and
// decode": the per-thread vector is picked for the widest load/store
// (256-bit on Blackwell), the warp count per block is a compile-time bound so
// the register allocation is known, decode rows go one warp per block to
// spread over as many SMs as possible, prefill rows go to multi-warp blocks.
//
// Kernels:
//   rmsn_vec_kernel     one row per warp (WARP_ROWS) or per block; each thread
//                       holds CH 32-byte vectors of the row in registers
//                       between the load and the store.  Launched with one
//                       unit (row, or WARP_ROWS rows) per block; a smaller
//                       grid loops over the rows.
//   rmsn_bulk_kernel    persistent blocks streaming whole rows into a ring of
//                       shared-memory buffers with TMA copies (swizzled 2-D
//                       tensor copies, or 1-D bulk copies).
//   rmsn_ragged_kernel  rows off the 32-byte grid: 16-byte vectors for the
//                       row's interior, single elements at its ends.
//   rmsn_generic_kernel any hidden size / alignment; element-wise, re-reads
//                       the row from the just-written residual_out.
#pragma once

#include <cuda.h>  // CUtensorMap (the bulk kernel's tensor-copy descriptors)
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "rmsn_registry.h"

namespace rmsn {

struct F32 {
    static constexpr int kBytes = 4;
};
struct BF16 {
    static constexpr int kBytes = 2;
};
struct F16 {
    static constexpr int kBytes = 2;
};
template <class T>
struct IsF16 {
    static constexpr bool value = false;
};
template <>
struct IsF16<F16> {
    static constexpr bool value = true;
};
struct FP8 {
    static constexpr int kBytes = 1;
};
// Block-scaled outputs (codes plus one scale per kBlock elements).
struct MXFP8 {
    static constexpr int kBytes = 1;
    static constexpr int kBlock = 32;
};
struct MXFP4 {
    static constexpr int kBytes = 1;
    static constexpr int kBlock = 32;
};
struct NVFP4 {
    static constexpr int kBytes = 1;
    static constexpr int kBlock = 16;
};
template <class T>
struct IsBlockFmt {
    static constexpr bool value = false;
};
template <>
struct IsBlockFmt<MXFP8> {
    static constexpr bool value = true;
};
template <>
struct IsBlockFmt<MXFP4> {
    static constexpr bool value = true;
};
template <>
struct IsBlockFmt<NVFP4> {
    static constexpr bool value = true;
};

// 32-byte register vector.
struct V8 {
    uint32_t u[8];
};

// ---------------------------------------------------------------- memory ops
// Streaming operands (x, residual) are read once: no L1 allocation.  Weight
// and bias are re-read by every row: default caching so they stay on chip.

__device__ __forceinline__ V8 ld_stream32(const void* p) {
    V8 v;
    asm volatile("ld.global.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.u[0]), "=r"(v.u[1]), "=r"(v.u[2]), "=r"(v.u[3]), "=r"(v.u[4]),
                   "=r"(v.u[5]), "=r"(v.u[6]), "=r"(v.u[7])
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_keep16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ V8 ld_keep32(const void* p) {
    V8 v;
    asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.u[0]), "=r"(v.u[1]), "=r"(v.u[2]), "=r"(v.u[3]), "=r"(v.u[4]),
                   "=r"(v.u[5]), "=r"(v.u[6]), "=r"(v.u[7])
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream32(void* p, const uint32_t* u) {
    asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p),
                 "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]),
                 "r"(u[7])
                 : "memory");
}

__device__ __forceinline__ void st_stream16(void* p, const uint32_t* u) {
    asm volatile("st.global.L1::no_allocate.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(u[0]),
                 "r"(u[1]), "r"(u[2]), "r"(u[3])
                 : "memory");
}

__device__ __forceinline__ void st_stream8(void* p, const uint32_t* u) {
    asm volatile("st.global.L1::no_allocate.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(u[0]), "r"(u[1])
                 : "memory");
}

// ---------------------------------------------------------------- conversions

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Round two floats to bf16 (nearest-even) and pack them, `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ float f16_to_f32(uint32_t bits) {
    float f;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"((uint16_t)(bits & 0xFFFFu)));
    return f;
}

// Round two floats to IEEE binary16 (nearest-even) and pack them, `lo` in the
// low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// The two 16-bit elements of a word of a 2-byte type T, and the reverse.
template <class T>
__device__ __forceinline__ float lo2(uint32_t u) {
    if constexpr (IsF16<T>::value) return f16_to_f32(u);
    else return bf16_lo(u);
}
template <class T>
__device__ __forceinline__ float hi2(uint32_t u) {
    if constexpr (IsF16<T>::value) return f16_to_f32(u >> 16);
    else return bf16_hi(u);
}
template <class T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (IsF16<T>::value) return pack_f16x2(lo, hi);
    else return pack_bf16x2(lo, hi);
}

// ---------------------------------------------------------------- packed arithmetic
//
// sm_100 and later run two fp32 lanes per instruction (the .f32x2 forms of
// add, mul and fma) and take 16-bit operands straight into fp32 adds and
// FMAs.  Every lane is rounded once, as the scalar operation rounds it, so
// these forms cut instructions without changing a single result.

// Two fp32 lanes in one 64-bit register pair.
struct F2 {
    uint64_t v;
};

__device__ __forceinline__ F2 f2(float lo, float hi) {
    F2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2split(F2 a, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
}

__device__ __forceinline__ F2 add2(F2 a, F2 b) {
    F2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}

__device__ __forceinline__ F2 mul2(F2 a, F2 b) {
    F2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}

__device__ __forceinline__ F2 fma2(F2 a, F2 b, F2 c) {
    F2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
    return r;
}

// The two 16-bit lanes of a word of T, widened to fp32 (exact).
template <class T>
__device__ __forceinline__ F2 widen2(uint32_t u) {
    return f2(lo2<T>(u), hi2<T>(u));
}

// acc + lo^2, then + hi^2, for the two lanes of u (type T): each step one
// fp32 rounding, as fmaf on the widened values (the square of a T value is
// exact in fp32).
template <class T>
__device__ __forceinline__ float sumsq16x2(uint32_t u, float acc) {
    float r;
    if constexpr (IsF16<T>::value)
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\t"
            "fma.rn.f32.f16 %0, l, l, %2;\n\tfma.rn.f32.f16 %0, h, h, %0;\n\t}"
            : "=f"(r)
            : "r"(u), "f"(acc));
    else
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\t"
            "fma.rn.f32.bf16 %0, l, l, %2;\n\tfma.rn.f32.bf16 %0, h, h, %0;\n\t}"
            : "=f"(r)
            : "r"(u), "f"(acc));
    return r;
}

// Both 16-bit lanes of u (type T) plus the fp32 c, each rounded once to fp32.
template <class T>
__device__ __forceinline__ F2 add16x2_f32(uint32_t u, float c) {
    float lo, hi;
    if constexpr (IsF16<T>::value)
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
            "add.rn.f32.f16 %0, l, %3;\n\tadd.rn.f32.f16 %1, h, %3;\n\t}"
            : "=f"(lo), "=f"(hi)
            : "r"(u), "f"(c));
    else
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
            "add.rn.f32.bf16 %0, l, %3;\n\tadd.rn.f32.bf16 %1, h, %3;\n\t}"
            : "=f"(lo), "=f"(hi)
            : "r"(u), "f"(c));
    return f2(lo, hi);
}

// The products h * w of the two 16-bit lanes of h and w (type T), exact: the
// product of two 8-bit (bf16) or 11-bit (fp16) significands fits fp32's 24
// bits, so the FMA with a -0 addend rounds nothing (and keeps the sign of a
// zero product).  Underflow below fp32's normal range is the only loss, at
// |h w| < 2^-126.
template <class T>
__device__ __forceinline__ F2 mul16x2_exact(uint32_t h, uint32_t w) {
    float lo, hi;
    if constexpr (IsF16<T>::value)
        asm("{\n\t.reg .b16 hl, hh, wl, wh;\n\tmov.b32 {hl, hh}, %2;\n\tmov.b32 {wl, wh}, %3;\n\t"
            "fma.rn.f32.f16 %0, hl, wl, 0f80000000;\n\tfma.rn.f32.f16 %1, hh, wh, 0f80000000;\n\t}"
            : "=f"(lo), "=f"(hi)
            : "r"(h), "r"(w));
    else
        asm("{\n\t.reg .b16 hl, hh, wl, wh;\n\tmov.b32 {hl, hh}, %2;\n\tmov.b32 {wl, wh}, %3;\n\t"
            "fma.rn.f32.bf16 %0, hl, wl, 0f80000000;\n\tfma.rn.f32.bf16 %1, hh, wh, 0f80000000;\n\t}"
            : "=f"(lo), "=f"(hi)
            : "r"(h), "r"(w));
    return f2(lo, hi);
}

// Both lanes of two packed 16-bit words of T added: the exact sum rounded
// once to T (nearest even), which is the residual's definition; the fp32 sum
// rounded to T gives the same value.
template <class T>
__device__ __forceinline__ uint32_t add16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    if constexpr (IsF16<T>::value) asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    else asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// max(m, |a|, |b|) in one three-input maximum.
__device__ __forceinline__ float absmax3(float m, float a, float b) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(m), "f"(fabsf(a)), "f"(fabsf(b)));
    return r;
}

// Round four floats to E4M3 (nearest-even, saturating to +-448), element 0
// in the lowest byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a0, float a1, float a2, float a3) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(a1), "f"(a0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(a3), "f"(a2));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Round two floats to FP4 E2M1 (nearest-even, saturating to +-6): element lo
// in bits 0-3, hi in bits 4-7 of the result.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
    uint16_t d;
    asm("{\n\t.reg .b8 q;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q, %1, %2;\n\t"
        "cvt.u16.u8 %0, q;\n\t}"
        : "=h"(d)
        : "f"(hi), "f"(lo));
    return (uint32_t)d & 0xFFu;
}

// Eight floats to E2M1, packed two per byte, element 0 in the lowest nibble.
__device__ __forceinline__ uint32_t pack_e2m1x8(float v0, float v1, float v2, float v3, float v4,
                                                float v5, float v6, float v7) {
    return cvt_e2m1x2(v0, v1) | (cvt_e2m1x2(v2, v3) << 8) | (cvt_e2m1x2(v4, v5) << 16) |
           (cvt_e2m1x2(v6, v7) << 24);
}

// Value of an E4M3 code (OCP FP8: bias 7, 3 mantissa bits), exact: every
// E4M3 value is a binary16 value, so the hardware widening is exact.  The
// code sits in the low byte, as cvt.rn.satfinite.e4m3x2.f32 writes its
// second operand.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)(c & 0xFFu)));
    return f16_to_f32(h2);
}

// Element k of a 32-byte vector of TI as float.
template <class TI>
__device__ __forceinline__ float elem(const V8& v, int k) {
    if constexpr (TI::kBytes == 2) {
        return (k & 1) ? hi2<TI>(v.u[k >> 1]) : lo2<TI>(v.u[k >> 1]);
    } else {
        return __uint_as_float(v.u[k]);
    }
}

// Make the compiler treat v as redefined here, so values unpacked from it are
// not hoisted out of the row loop (that would keep 2x the registers live).
__device__ __forceinline__ void opaque(V8& v) {
#pragma unroll
    for (int k = 0; k < 8; ++k) asm volatile("" : "+r"(v.u[k]));
}

// One vector of VE = 32 / TI::kBytes elements of a TX array starting at
// element `e`, as a TI vector.  TX == TI: one 32-byte access.  A 2-byte TX
// under an fp32 TI (bf16 / fp16 activations with an fp32 residual stream):
// one 16-byte access, widened exactly.
template <class TX, class TI, bool STREAM>
__device__ __forceinline__ V8 ld_vec(const void* base, int64_t e) {
    if constexpr (TX::kBytes == TI::kBytes) {
        const void* p = static_cast<const char*>(base) + e * TI::kBytes;
        return STREAM ? ld_stream32(p) : ld_keep32(p);
    } else {
        static_assert(TX::kBytes == 2 && TI::kBytes == 4, "2-byte values under fp32 only");
        const void* p = static_cast<const char*>(base) + e * 2;
        const uint4 w = STREAM ? ld_stream16(p) : ld_keep16(p);
        const uint32_t in[4] = {w.x, w.y, w.z, w.w};
        V8 v;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v.u[2 * k] = __float_as_uint(lo2<TX>(in[k]));
            v.u[2 * k + 1] = __float_as_uint(hi2<TX>(in[k]));
        }
        return v;
    }
}

template <class TI>
__device__ __forceinline__ uint32_t ones_word() {
    if constexpr (IsF16<TI>::value) return 0x3C003C00u;
    return TI::kBytes == 2 ? 0x3F803F80u : 0x3F800000u;
}

// ---------------------------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialization (a.pdl) may start
// before the preceding kernel in its stream has finished.  Such a kernel lets
// its own dependents start at once, and waits for its prerequisite grid (and
// that grid's memory) before its first global read of anything the caller
// did not declare constant (a.early_params: weight and bias may be read
// first).  Kernels launched the ordinary way skip both instructions.

__device__ __forceinline__ void pdl_launch_dependents(int pdl) {
    if (pdl) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait(int pdl) {
    if (pdl) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------- bounds-checked build
// Built with -DRMSNORM_BOUNDS_CHECK, every global access and ring copy below is
// first checked against the extent of its tensor; an access out of range is
// skipped (loads leave zeros) and sets bit 1 of the status word, so a wrong
// index shows up as a status bit instead of a fault.  In the normal build
// every check is the constant true and compiles away.

#ifdef RMSNORM_BOUNDS_CHECK
__device__ __forceinline__ bool check_ok(uint32_t* status, bool ok) {
    if (!ok) atomicOr(status, 2u);
    return ok;
}
#define RMSN_CHECK(status, cond) ::rmsn::check_ok((status), (cond))
#else
#define RMSN_CHECK(status, cond) true
#endif

// Elements [e, e + n) inside the [T, H] row tensors of a.
__device__ __forceinline__ bool rows_ok(const RmsnArgs& a, int64_t e, int64_t n) {
    return RMSN_CHECK(a.status, e >= 0 && e + n <= a.T * (int64_t)a.H);
}
// Elements [j, j + n) inside the [H] weight and bias.
__device__ __forceinline__ bool cols_ok(const RmsnArgs& a, int64_t j, int64_t n) {
    return RMSN_CHECK(a.status, j >= 0 && j + n <= (int64_t)a.H);
}
__device__ __forceinline__ bool row_ok(const RmsnArgs& a, int64_t row) {
    return RMSN_CHECK(a.status, row >= 0 && row < a.T);
}

// ---------------------------------------------------------------- reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Maximum over the warp of absolute maxima.  REDUX: every v is +0 or above
// and never NaN (they are maxima of |y| started from 0 with NaN-ignoring
// max), and such floats order as their bit patterns do as unsigned integers,
// so one redux.sync gives exactly the float maximum; else a butterfly.
template <bool REDUX = true>
__device__ __forceinline__ float warp_max(float v) {
    if constexpr (REDUX) {
        uint32_t r;
        asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(__float_as_uint(v)));
        return __uint_as_float(r);
    } else {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
        return v;
    }
}

// Sum (or max) over the warps of a block through shared memory.  `slot` is a
// [32] float array that alternates between calls so one barrier per call
// suffices; every thread adds the partials in the same order and so gets the
// same total.
template <bool MAX, bool REDUX = true>
__device__ __forceinline__ float block_allreduce(float v, float* slot) {
    v = MAX ? warp_max<REDUX>(v) : warp_sum(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) slot[warp] = v;
    __syncthreads();
    const int nw = blockDim.x >> 5;
    float t = slot[0];
    for (int i = 1; i < nw; ++i) t = MAX ? fmaxf(t, slot[i]) : __fadd_rn(t, slot[i]);
    return t;
}

__device__ __forceinline__ float inv_rms(float sumsq, int H, float eps) {
    return __frsqrt_rn(__fadd_rn(__fdiv_rn(sumsq, (float)H), eps));
}

// y = (w + w_off) * (h * inv) + b, with every rounding explicit so the two
// FP8 passes recompute identical values.
template <bool BIAS>
__device__ __forceinline__ float scale_elem(float h, float inv, float w, float woff, float b) {
    const float t = __fmul_rn(h, inv);
    const float wo = __fadd_rn(w, woff);
    return BIAS ? __fmaf_rn(wo, t, b) : __fmul_rn(wo, t);
}

// scale_elem over the VE elements of one vector; `m` takes the maximum of
// |y|.  PACK: two lanes per instruction (the same roundings, so the same
// values); else one element at a time.
template <class TI, bool BIAS, bool MAX = false, bool PACK = true>
__device__ __forceinline__ void scale_vec(const V8& h, const V8& w, const V8& b, float inv,
                                          float woff, float (&y)[32 / TI::kBytes], float& m) {
    const F2 inv2 = f2(inv, inv);
    if constexpr (!PACK) {
#pragma unroll
        for (int k = 0; k < 32 / TI::kBytes; ++k) {
            y[k] = scale_elem<BIAS>(elem<TI>(h, k), inv, elem<TI>(w, k), woff,
                                    BIAS ? elem<TI>(b, k) : 0.f);
            if constexpr (MAX) m = fmaxf(m, fabsf(y[k]));
        }
    } else if constexpr (TI::kBytes == 2) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const F2 t = mul2(widen2<TI>(h.u[k]), inv2);
            const F2 wo = add16x2_f32<TI>(w.u[k], woff);
            const F2 r = BIAS ? fma2(wo, t, widen2<TI>(b.u[k])) : mul2(wo, t);
            f2split(r, y[2 * k], y[2 * k + 1]);
            if constexpr (MAX) m = absmax3(m, y[2 * k], y[2 * k + 1]);
        }
    } else {
        const F2 woff2 = f2(woff, woff);
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            const F2 t = mul2(f2(__uint_as_float(h.u[k]), __uint_as_float(h.u[k + 1])), inv2);
            const F2 wo = add2(f2(__uint_as_float(w.u[k]), __uint_as_float(w.u[k + 1])), woff2);
            const F2 r = BIAS ? fma2(wo, t, f2(__uint_as_float(b.u[k]), __uint_as_float(b.u[k + 1])))
                              : mul2(wo, t);
            f2split(r, y[k], y[k + 1]);
            if constexpr (MAX) m = absmax3(m, y[k], y[k + 1]);
        }
    }
}

// y for the quantised outputs, whose codes and scales are taken from fp32 y.
// Without a weight offset (16-bit weights): y = RN(p * inv + b) with p = h w
// formed exactly, one rounding in all; the weight and h are used as packed
// 16-bit lanes, so nothing is unpacked but the bias.  With an offset (or an
// fp32 stream) the rounding sequence of scale_vec.
template <class TI, bool BIAS>
__device__ __forceinline__ void scale_vec_q(const V8& h, const V8& w, const V8& b, float inv,
                                            float woff, float (&y)[32 / TI::kBytes], float& m) {
    if constexpr (TI::kBytes == 2) {
        if (woff == 0.f) {
            const F2 inv2 = f2(inv, inv);
            float m2 = 0.f;  // a second maximum chain (the maximum is order-free)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const F2 p = mul16x2_exact<TI>(h.u[k], w.u[k]);
                const F2 r = BIAS ? fma2(p, inv2, widen2<TI>(b.u[k])) : mul2(p, inv2);
                f2split(r, y[2 * k], y[2 * k + 1]);
                if (k & 1) m2 = absmax3(m2, y[2 * k], y[2 * k + 1]);
                else m = absmax3(m, y[2 * k], y[2 * k + 1]);
            }
            m = fmaxf(m, m2);
            return;
        }
    }
    scale_vec<TI, BIAS, true, true>(h, w, b, inv, woff, y, m);
}

// Store the VE outputs of one input vector at element offset `e`.
template <class TI, class TO>
__device__ __forceinline__ void store_out(void* out, int64_t e, const float (&y)[32 / TI::kBytes],
                                          float qmul) {
    constexpr int VE = 32 / TI::kBytes;
    if constexpr (TO::kBytes == 4) {
        uint32_t u[VE];
#pragma unroll
        for (int k = 0; k < VE; ++k) u[k] = __float_as_uint(y[k]);
        float* o = reinterpret_cast<float*>(out) + e;
#pragma unroll
        for (int s = 0; s < VE / 8; ++s) st_stream32(o + 8 * s, u + 8 * s);
    } else if constexpr (TO::kBytes == 2) {
        uint32_t u[VE / 2];
#pragma unroll
        for (int k = 0; k < VE / 2; ++k) u[k] = pack2<TO>(y[2 * k], y[2 * k + 1]);
        uint16_t* o = reinterpret_cast<uint16_t*>(out) + e;
        if constexpr (VE == 16) st_stream32(o, u);
        else st_stream16(o, u);
    } else {
        uint32_t u[VE / 4];
        const F2 q2 = f2(qmul, qmul);
#pragma unroll
        for (int k = 0; k < VE / 4; ++k) {
            // y * qmul two lanes at a time (each lane rounded once, as __fmul_rn)
            float s0, s1, s2, s3;
            f2split(mul2(f2(y[4 * k], y[4 * k + 1]), q2), s0, s1);
            f2split(mul2(f2(y[4 * k + 2], y[4 * k + 3]), q2), s2, s3);
            u[k] = pack_e4m3x4(s0, s1, s2, s3);
        }
        uint8_t* o = reinterpret_cast<uint8_t*>(out) + e;
        if constexpr (VE == 16) st_stream16(o, u);
        else st_stream8(o, u);
    }
}

// Register budget: blocks of up to WMAX warps; at least 1024 resident threads
// per SM for CH <= 2 (64 registers / thread), 512 for CH = 4 (128) and 256
// for CH = 8 (255, one-warp decode rows).  With both a residual and a bias a
// thread holds four vectors per chunk (x, residual, weight, bias: 32
// registers), so from CH = 2 on the budget is doubled rather than spilled.
template <int WMAX, int CH, bool HEAVY = false>
struct Bounds {
    static constexpr int kThreads = WMAX * 32;
    static constexpr int kTarget = (CH <= 2 ? 1024 : (CH <= 4 ? 512 : 256)) /
                                   (HEAVY && CH >= 2 ? 2 : 1);
    static constexpr int kMinBlocks = kTarget / kThreads > 0 ? kTarget / kThreads : 1;
};

// ---------------------------------------------------------------- row body
//
// Shared by the register-streaming and the bulk-copy kernels.  A thread
// handles vectors v = c * G + t (c < CH, G = threads per row, t = thread
// within the row) of VE elements each, so a warp touches 1 KiB of contiguous
// memory per chunk.  hv holds x on entry (and rv the residual); on exit hv
// holds h = RN_in(x + r), which was also stored to residual_out.

template <class TX, class TI, int CH>
__device__ __forceinline__ void load_params(const RmsnArgs& a, int G, int t, V8 (&wv)[CH],
                                            V8* bv, bool bias) {
    constexpr int VE = 32 / TI::kBytes;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const int v = c * G + t;
        if (v < a.nvec && cols_ok(a, (int64_t)v * VE, VE)) {
            if (a.has_w) {
                wv[c] = ld_vec<TX, TI, false>(a.w, (int64_t)v * VE);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) wv[c].u[k] = ones_word<TI>();
            }
            if (bias) bv[c] = ld_vec<TX, TI, false>(a.b, (int64_t)v * VE);
        }
    }
}

// h = RN_in(x + r) (the sum formed in fp32), stored to residual_out; returns
// this thread's fp32 sum of h^2.  PADD: the packed 16-bit add (add.rn.bf16x2 /
// f16x2), the same h in an eighth of the instructions; measured on GB300 it
// made the 16-bit-output prefill ring ~15% slower, so only the quantised
// outputs, whose ring is bound by instruction issue, take it.  PACK: the
// squares take the 16-bit lanes straight into the FMA.
template <class TI, int CH, bool RES, bool PACK = true, bool PADD = false>
__device__ __forceinline__ float residual_sumsq(const RmsnArgs& a, int64_t rbase, int G, int t,
                                                V8 (&hv)[CH], const V8* rv) {
    constexpr int VE = 32 / TI::kBytes;
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const int v = c * G + t;
        if (v < a.nvec) {
            if constexpr (RES) {
                if constexpr (TI::kBytes == 2 && PADD) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) hv[c].u[k] = add16x2<TI>(hv[c].u[k], rv[c].u[k]);
                } else if constexpr (TI::kBytes == 2) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float lo = __fadd_rn(lo2<TI>(hv[c].u[k]), lo2<TI>(rv[c].u[k]));
                        const float hi = __fadd_rn(hi2<TI>(hv[c].u[k]), hi2<TI>(rv[c].u[k]));
                        hv[c].u[k] = pack2<TI>(lo, hi);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        hv[c].u[k] = __float_as_uint(__fadd_rn(__uint_as_float(hv[c].u[k]),
                                                               __uint_as_float(rv[c].u[k])));
                }
                const int64_t off = (rbase + (int64_t)v * VE) * TI::kBytes;
                if (rows_ok(a, rbase + (int64_t)v * VE, VE))
                    st_stream32(static_cast<char*>(a.res_out) + off, hv[c].u);
            }
            if constexpr (TI::kBytes == 2 && PACK && PADD) {
                // two interleaved chains, added at the end: half the dependent
                // latency for the quantised ring, whose rows are latency-bound
                float acc2 = 0.f;
#pragma unroll
                for (int k = 0; k < 8; k += 2) {
                    acc = sumsq16x2<TI>(hv[c].u[k], acc);
                    acc2 = sumsq16x2<TI>(hv[c].u[k + 1], acc2);
                }
                acc = __fadd_rn(acc, acc2);
            } else if constexpr (TI::kBytes == 2 && PACK) {
#pragma unroll
                for (int k = 0; k < 8; ++k) acc = sumsq16x2<TI>(hv[c].u[k], acc);
            } else {
#pragma unroll
                for (int k = 0; k < VE; ++k) {
                    const float h = elem<TI>(hv[c], k);
                    acc = __fmaf_rn(h, h, acc);
                }
            }
        }
    }
    return acc;
}

// Block-scaled outputs (blog section "Blackwell support": MXFP8 / MXFP4 /
// NVFP4 with the absolute maximum over 32 or 16 elements).  A block spans
// LPB = kBlock / VE neighbouring lanes (their vectors are adjacent), so the
// block maximum is a butterfly over LPB lanes.
//   MX:    scale 2^s, s = floor(log2 max|y|) - emax (8 for E4M3, 2 for E2M1),
//          clamped to [-127, 127], stored as E8M0 (s + 127); codes y * 2^-s.
//   NVFP4: per-token fp32 g = max|row| / (448 * 6) (the row max all-reduce),
//          block scale E4M3(max|block| * (1 / (6 g))), codes
//          E2M1(y * r_b) with r_b the hardware approximation of
//          1 / (scale * g); 1 / (6 g) is correctly rounded.
// All conversions round to nearest even and saturate.
// NVFP4's per-token scale g = max|row| / (448 * 6), stored for the row, and
// the correctly rounded 1 / (6 g) its block scales are formed with.
template <class TO>
__device__ __forceinline__ void nv_row_scale(const RmsnArgs& a, int64_t row, int t, float amax,
                                             float& g, float& rcp6g) {
    g = __fdiv_rn(amax, 2688.f);
    if (t == 0 && row_ok(a, row)) a.scale[row] = g;
    rcp6g = g > 0.f ? __frcp_rn(__fmul_rn(6.f, g)) : 0.f;  // one reciprocal per row
}

// One vector of y (element index e, vector v of the row) in a block format:
// its block scale from the block maximum bmax (NVFP4: with g and 1 / (6 g)),
// the codes of y under it, stored with the block scale (by the block's first
// lane).
template <class TI, class TO>
__device__ __forceinline__ void store_block_vec(const RmsnArgs& a, int64_t e, int v,
                                                float (&y)[32 / TI::kBytes], float bmax, float g,
                                                float rcp6g) {
    constexpr int VE = 32 / TI::kBytes;
    constexpr int LPB = TO::kBlock / VE;
    constexpr bool NV = TO::kBlock == 16;
    constexpr bool FP4 = !std::is_same<TO, MXFP8>::value;
    float mul;      // code = convert(y * mul)
    uint8_t sbyte;  // block scale code
    if constexpr (NV) {
        uint32_t sc = 0;
        if (g > 0.f) {
            uint16_t two;
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
                : "=h"(two)
                : "f"(0.f), "f"(__fmul_rn(bmax, rcp6g)));
            sc = two & 0xFFu;
        }
        const float s = __fmul_rn(e4m3_value(sc), g);
        // one reciprocal per block of 16, the hardware approximation (within
        // 1 ulp of 1/s): the codes are E2M1(RN(y * r)), which can differ by
        // one step from E2M1(y / s) where y / s lies within a few fp32 ulp of
        // a rounding midpoint of E2M1
        if (s > 0.f) asm("rcp.approx.f32 %0, %1;" : "=f"(mul) : "f"(s));
        else mul = 0.f;
        sbyte = (uint8_t)sc;
    } else {
        constexpr int emax = FP4 ? 2 : 8;
        const int ef = (int)((__float_as_uint(bmax) >> 23) & 0xFFu);
        int sx = ef == 0 ? -127 : ef - 127 - emax;  // zero / subnormal maxima clamp
        sx = sx < -127 ? -127 : (sx > 126 ? 126 : sx);
        mul = __uint_as_float((uint32_t)(127 - sx) << 23);  // 2^-s, exact
        sbyte = (uint8_t)(sx + 127);
    }
#pragma unroll
    for (int k = 0; k < VE; k += 2) f2split(mul2(f2(y[k], y[k + 1]), f2(mul, mul)), y[k], y[k + 1]);
    if (!rows_ok(a, e, VE)) return;
    if constexpr (FP4) {
        uint32_t u[VE / 8];
#pragma unroll
        for (int k = 0; k < VE / 8; ++k)
            u[k] = pack_e2m1x8(y[8 * k], y[8 * k + 1], y[8 * k + 2], y[8 * k + 3], y[8 * k + 4],
                               y[8 * k + 5], y[8 * k + 6], y[8 * k + 7]);
        uint8_t* o = reinterpret_cast<uint8_t*>(a.out) + e / 2;
        if constexpr (VE == 16) st_stream8(o, u);
        else asm volatile("st.global.b32 [%0], %1;" ::"l"(o), "r"(u[0]) : "memory");
    } else {
        uint32_t u[VE / 4];
#pragma unroll
        for (int k = 0; k < VE / 4; ++k)
            u[k] = pack_e4m3x4(y[4 * k], y[4 * k + 1], y[4 * k + 2], y[4 * k + 3]);
        uint8_t* o = reinterpret_cast<uint8_t*>(a.out) + e;
        if constexpr (VE == 16) st_stream16(o, u);
        else st_stream8(o, u);
    }
    if (v % LPB == 0) static_cast<uint8_t*>(a.bscale)[e / TO::kBlock] = sbyte;
}

template <class TI, class TO, int CH, bool BIAS, bool KEEP, bool QF, class ReduceMax>
__device__ __forceinline__ void scale_store_block(const RmsnArgs& a, int64_t row, int64_t rbase,
                                                  int G, int t, float inv, const V8 (&hv)[CH],
                                                  V8 (&wv)[CH], V8* bv, ReduceMax reduce_max) {
    constexpr int VE = 32 / TI::kBytes;
    constexpr int LPB = TO::kBlock / VE;
    constexpr bool NV = TO::kBlock == 16;
    constexpr bool HOLD = KEEP && NV;  // keep y between NVFP4's row-max and block passes
    static_assert(LPB >= 1 && LPB <= 4, "block spans 1..4 lanes");
    float ys[HOLD ? CH : 1][HOLD ? VE : 1];
    float bms[HOLD ? CH : 1];  // with HOLD: the lane's maximum of each vector
    float g = 0.f, rcp6g = 0.f;
    if constexpr (NV) {
        float amax = 0.f;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int v = c * G + t;
            if (v < a.nvec) {
                opaque(wv[c]);
                if constexpr (BIAS) opaque(bv[c]);
                float m = 0.f, y[VE];
                if constexpr (QF)
                    scale_vec_q<TI, BIAS>(hv[c], wv[c], bv[BIAS ? c : 0], inv, a.woff, y, m);
                else
                    scale_vec<TI, BIAS, true>(hv[c], wv[c], bv[BIAS ? c : 0], inv, a.woff, y, m);
                if constexpr (HOLD) {
#pragma unroll
                    for (int k = 0; k < VE; ++k) ys[c][k] = y[k];
                    bms[c] = m;
                }
                amax = fmaxf(amax, m);
            }
        }
        nv_row_scale<TO>(a, row, t, reduce_max(amax), g, rcp6g);
    }
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const int v = c * G + t;
        const bool valid = v < a.nvec;
        float y[VE];
        float bmax = 0.f;
        if (valid) {
            if constexpr (HOLD) {
#pragma unroll
                for (int k = 0; k < VE; ++k) y[k] = ys[c][k];
                bmax = bms[c];
            } else {
                opaque(wv[c]);
                if constexpr (BIAS) opaque(bv[c]);
                if constexpr (QF)
                    scale_vec_q<TI, BIAS>(hv[c], wv[c], bv[BIAS ? c : 0], inv, a.woff, y, bmax);
                else
                    scale_vec<TI, BIAS, true>(hv[c], wv[c], bv[BIAS ? c : 0], inv, a.woff, y,
                                              bmax);
            }
        }
        // every lane takes part; a block's lanes are all valid or all invalid
#pragma unroll
        for (int o = LPB / 2; o > 0; o >>= 1)
            bmax = fmaxf(bmax, __shfl_xor_sync(0xFFFFFFFFu, bmax, o));
        if (!valid) continue;
        store_block_vec<TI, TO>(a, rbase + (int64_t)v * VE, v, y, bmax, g, rcp6g);
    }
}

// Per-token FP8 of a held row of y: scale max|y| / 448, codes y * 448 / max|y|.
template <class TI, int CH>
__device__ __forceinline__ void store_fp8_held(const RmsnArgs& a, int64_t row, int64_t rbase,
                                               int G, int t, const float (&ys)[CH][32 / TI::kBytes],
                                               float amax) {
    constexpr int VE = 32 / TI::kBytes;
    const float qmul = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
    if (t == 0 && row_ok(a, row)) a.scale[row] = __fdiv_rn(amax, 448.f);
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const int v = c * G + t;
        if (v < a.nvec && rows_ok(a, rbase + (int64_t)v * VE, VE))
            store_out<TI, FP8>(a.out, rbase + (int64_t)v * VE, ys[c], qmul);
    }
}

// Scale, (FP8: absmax reduction and per-token scale) and store the row.
// `reduce_max` is the row-wide max all-reduce (only used for FP8 output).
// KEEP: hold the row's y in registers between the FP8 max pass and the
// quantising pass instead of recomputing it (for kernels with a large
// register budget).  QF: the quantised outputs take y from scale_vec_q (the
// exact product h w; fewer instructions), else from scale_vec.  The
// register kernels keep scale_vec: with two scale passes per row under a
// 64-register bound the second form spills.
template <class TI, class TO, int CH, bool BIAS, bool KEEP = false, bool QF = false,
          class ReduceMax>
__device__ __forceinline__ void scale_store(const RmsnArgs& a, int64_t row, int64_t rbase, int G,
                                            int t, float inv, const V8 (&hv)[CH], V8 (&wv)[CH],
                                            V8* bv, ReduceMax reduce_max) {
    if constexpr (IsBlockFmt<TO>::value) {
        scale_store_block<TI, TO, CH, BIAS, KEEP, QF>(a, row, rbase, G, t, inv, hv, wv, bv,
                                                      reduce_max);
        return;
    }
    constexpr int VE = 32 / TI::kBytes;
    constexpr bool HOLD = KEEP && TO::kBytes == 1;
    float ys[HOLD ? CH : 1][HOLD ? VE : 1];
    float qmul = 0.f;
    if constexpr (TO::kBytes == 1) {
        float amax = 0.f;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int v = c * G + t;
            if (v < a.nvec) {
                opaque(wv[c]);
                if constexpr (BIAS) opaque(bv[c]);
                float y[VE];
                if constexpr (QF)
                    scale_vec_q<TI, BIAS>(hv[c], wv[c], bv[BIAS ? c : 0], inv, a.woff, y, amax);
                else
                    scale_vec<TI, BIAS, true>(hv[c], wv[c], bv[BIAS ? c : 0], inv, a.woff, y,
                                              amax);
                if constexpr (HOLD) {
#pragma unroll
                    for (int k = 0; k < VE; ++k) ys[c][k] = y[k];
                }
            }
        }
        amax = reduce_max(amax);
        qmul = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
        if (t == 0 && row_ok(a, row)) a.scale[row] = __fdiv_rn(amax, 448.f);
    }
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const int v = c * G + t;
        if (v < a.nvec) {
            if (!rows_ok(a, rbase + (int64_t)v * VE, VE)) continue;
            if constexpr (HOLD) {
                store_out<TI, TO>(a.out, rbase + (int64_t)v * VE, ys[c], qmul);
            } else {
                opaque(wv[c]);
                if constexpr (BIAS) opaque(bv[c]);
                float y[VE], m = 0.f;
                if constexpr (QF && TO::kBytes == 1)
                    scale_vec_q<TI, BIAS>(hv[c], wv[c], bv[BIAS ? c : 0], inv, a.woff, y, m);
                else
                    scale_vec<TI, BIAS>(hv[c], wv[c], bv[BIAS ? c : 0], inv, a.woff, y, m);
                store_out<TI, TO>(a.out, rbase + (int64_t)v * VE, y, qmul);
            }
        }
    }
}

// ---------------------------------------------------------------- vector kernel
//
// WARP_ROWS: each warp owns one row (block = WMAX rows); else the block owns
// one row and has up to WMAX warps.  Each thread loads its CH vectors of x
// (and the residual) straight into registers; rows are visited grid-stride;
// weight and bias stay in registers across rows.
// TX: storage of x, weight and bias; TI: of the residual stream and h (TX
// unless an fp32 residual stream carries bf16 / fp16 activations).
template <class TI, class TO, int CH, int WMAX, bool WARP_ROWS, bool RES, bool BIAS,
          class TX = TI>
__global__ void __launch_bounds__(Bounds<WMAX, CH, RES && BIAS>::kThreads,
                                  Bounds<WMAX, CH, RES && BIAS>::kMinBlocks)
    rmsn_vec_kernel(const RmsnArgs a) {
    constexpr int VE = 32 / TI::kBytes;  // elements per 32-byte vector
    __shared__ float red[4][32];

    const int lane = threadIdx.x & 31;
    const int G = WARP_ROWS ? 32 : (int)blockDim.x;
    const int t = WARP_ROWS ? lane : (int)threadIdx.x;
    const int64_t rows_per_step = WARP_ROWS ? (int64_t)gridDim.x * (blockDim.x >> 5) : gridDim.x;
    int64_t row = WARP_ROWS ? (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)
                            : (int64_t)blockIdx.x;

    V8 hv[CH];
    V8 rv[RES ? CH : 1];
    auto load_row = [&](int64_t rw) {
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int v = c * G + t;
            const int64_t e = rw * (int64_t)a.H + (int64_t)v * VE;
            if (v < a.nvec && rows_ok(a, e, VE)) {
                hv[c] = ld_vec<TX, TI, true>(a.x, e);
                if constexpr (RES) rv[c] = ld_stream32(static_cast<const char*>(a.r) + e * TI::kBytes);
            }
        }
    };
    pdl_launch_dependents(a.pdl);
    V8 wv[CH];
    V8 bv[BIAS ? CH : 1];
    if (a.early_params) load_params<TX, TI, CH>(a, G, t, wv, bv, BIAS);
    pdl_wait(a.pdl);
    // without a bias the first row's loads go out before the weight's (a
    // single-row call then waits on the row, not on the weight behind it);
    // with one, the four vectors per chunk would all be live at once
    constexpr bool EARLY_ROW = !BIAS;
    const int64_t first = row;
    if (EARLY_ROW && row < a.T) load_row(row);
    if (!a.early_params) load_params<TX, TI, CH>(a, G, t, wv, bv, BIAS);

    int parity = 0;
    for (; row < a.T; row += rows_per_step) {
        const int64_t rbase = row * (int64_t)a.H;  // element offset of the row
        if (!EARLY_ROW || row != first) load_row(row);
        const float acc = residual_sumsq<TI, CH, RES>(a, rbase, G, t, hv, rv);
        const float sumsq = WARP_ROWS ? warp_sum(acc) : block_allreduce<false>(acc, red[parity]);
        const float inv = inv_rms(sumsq, a.H, a.eps);
        float* slot = red[2 + parity];
        scale_store<TI, TO, CH, BIAS>(a, row, rbase, G, t, inv, hv, wv, bv, [&](float m) {
            return WARP_ROWS ? warp_max(m) : block_allreduce<true>(m, slot);
        });
        parity ^= 1;
    }
}

// ---------------------------------------------------------------- bulk-copy kernel
//
// Persistent blocks (one row at a time, up to WMAX warps).  Whole rows of x
// and the residual are moved into a ring of `a.stages` shared-memory buffers
// by the TMA engine (cp.async.bulk.tensor with the 128-byte swizzle, or
// cp.async.bulk; completion counted on an mbarrier per buffer), issued by
// thread 0 up to `stages` rows ahead.  The
// threads copy their vectors from shared memory into registers, so a buffer
// is free again after the row's sum-of-squares barrier, where thread 0
// refills it with the row `stages` ahead.  Bytes in flight per SM are set by
// the ring size, not by the register file.
//
// Every mbarrier wait is bounded (a.wait_cycles, by default about one second
// of clock cycles).  A wait that runs out sets bit 0 of *a.status and a
// shared abort flag; the block still takes part in the row's barrier so no
// thread is left waiting, then stops, after thread 0 has waited (bounded by
// the default, whatever a.wait_cycles says) for its copies in flight, so no
// copy into the block's shared memory outlives the block.

constexpr int kMaxStages = 8;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete, for at most `limit`
// clock cycles; a negative limit tests the phase once and does not wait.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  long long limit) {
    if (limit < 0) return mbar_test_wait(bar, parity);
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) return false;
    }
    return true;
}

// Thread 0: expect the row's bytes on `bar`, then copy x (x_bytes) of `row`
// into `dst` and, with a residual, its residual row (r_bytes) right after it.
template <bool RES>
__device__ __forceinline__ void issue_row(const RmsnArgs& a, int64_t row, uint32_t dst,
                                          uint32_t bar, uint32_t x_bytes, uint32_t r_bytes) {
    const uint32_t bytes = RES ? x_bytes + r_bytes : x_bytes;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
    const char* src = static_cast<const char*>(a.x) + row * (int64_t)x_bytes;
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(x_bytes), "r"(bar)
        : "memory");
    if constexpr (RES) {
        const char* rsrc = static_cast<const char*>(a.r) + row * (int64_t)r_bytes;
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
            "[%3];" ::"r"(dst + x_bytes),
            "l"(rsrc), "r"(r_bytes), "r"(bar)
            : "memory");
    }
}

__device__ __forceinline__ V8 ld_shared32(uint32_t addr) {
    V8 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.u[0]), "=r"(v.u[1]), "=r"(v.u[2]), "=r"(v.u[3])
                 : "r"(addr));
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.u[4]), "=r"(v.u[5]), "=r"(v.u[6]), "=r"(v.u[7])
                 : "r"(addr + 16));
    return v;
}

// Stages filled by 2-D tensor copies with the 128-byte swizzle: the stage is
// a run of 128-byte lines starting on a 1024-byte boundary, and 16-byte
// chunk c of line l sits at chunk c ^ (l & 7).  A quarter warp reading 8
// neighbouring 32-byte vectors then meets every bank once per load.
__device__ __forceinline__ uint32_t swz128(uint32_t base, uint32_t off) {
    return base + (off ^ (((off >> 7) & 7u) << 4));
}

__device__ __forceinline__ V8 ld_shared32_swz(uint32_t base, uint32_t v) {
    V8 r;
    const uint32_t off = v * 32u;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.u[0]), "=r"(r.u[1]), "=r"(r.u[2]), "=r"(r.u[3])
                 : "r"(swz128(base, off)));
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.u[4]), "=r"(r.u[5]), "=r"(r.u[6]), "=r"(r.u[7])
                 : "r"(swz128(base, off + 16u)));
    return r;
}

// Thread 0: expect the row's bytes on `bar`, then copy x (and the residual
// right after it) of `row` as 2-D tensor boxes of `xl` (`rl`) 128-byte lines.
template <bool RES>
__device__ __forceinline__ void issue_row_tensor(const CUtensorMap* mx, const CUtensorMap* mr,
                                                 int64_t row, uint32_t dst, uint32_t bar,
                                                 uint32_t x_bytes, uint32_t r_bytes) {
    const uint32_t bytes = RES ? x_bytes + r_bytes : x_bytes;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(mx)), "r"(0), "r"((int)(row * (x_bytes / 128u))),
        "r"(bar)
        : "memory");
    if constexpr (RES) {
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
            "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst + x_bytes),
            "l"(reinterpret_cast<uint64_t>(mr)), "r"(0), "r"((int)(row * (r_bytes / 128u))),
            "r"(bar)
            : "memory");
    }
}

// One vector of VE = 32 / TI::kBytes elements from shared memory: 32 bytes,
// or 16 bytes of 2-byte values widened exactly to fp32 under an fp32 stream.
template <class TX, class TI>
__device__ __forceinline__ V8 ld_shared_vec(uint32_t addr) {
    if constexpr (TX::kBytes == TI::kBytes) {
        return ld_shared32(addr);
    } else {
        static_assert(TX::kBytes == 2 && TI::kBytes == 4, "2-byte values under fp32 only");
        uint32_t in[4];
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(in[0]), "=r"(in[1]), "=r"(in[2]), "=r"(in[3])
                     : "r"(addr));
        V8 v;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v.u[2 * k] = __float_as_uint(lo2<TX>(in[k]));
            v.u[2 * k + 1] = __float_as_uint(hi2<TX>(in[k]));
        }
        return v;
    }
}

template <class TX, class TI>
__device__ __forceinline__ V8 ld_shared_vec_swz(uint32_t base, uint32_t v) {
    if constexpr (TX::kBytes == TI::kBytes) {
        return ld_shared32_swz(base, v);
    } else {
        uint32_t in[4];
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(in[0]), "=r"(in[1]), "=r"(in[2]), "=r"(in[3])
                     : "r"(swz128(base, v * 16u)));
        V8 r;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            r.u[2 * k] = __float_as_uint(lo2<TX>(in[k]));
            r.u[2 * k + 1] = __float_as_uint(hi2<TX>(in[k]));
        }
        return r;
    }
}

// TX: storage of x, weight and bias, as in rmsn_vec_kernel; a stage holds
// the row of x followed by the row of the residual (TI).  With a.swz the
// stages are filled by swizzled 2-D tensor copies described by mx / mr (and
// start on 1024-byte boundaries), else by 1-D bulk copies.
// Sum and maximum over the warps of a block with one barrier: `slot` holds
// [64] floats (sums, then maxima) and alternates between calls.
__device__ __forceinline__ void block_allreduce_sum_max(float s, float m, float* slot, float& sum,
                                                        float& mx) {
    s = warp_sum(s);
    m = warp_max(m);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        slot[warp] = s;
        slot[32 + warp] = m;
    }
    __syncthreads();
    const int nw = blockDim.x >> 5;
    sum = slot[0];
    mx = slot[32];
    for (int i = 1; i < nw; ++i) {
        sum = __fadd_rn(sum, slot[i]);
        mx = fmaxf(mx, slot[32 + i]);
    }
}

// PIPE (per-token FP8 and NVFP4 outputs, whose rows need a second block
// reduction for the row maximum): a two-row software pipeline.  Iteration k
// takes row k - 1 through the scale pass and its maxima and row k through the
// residual add and its sum of squares; one barrier then reduces both (row k's
// sum, row k - 1's maximum), after which row k - 1 is quantised and stored.
// One barrier per row instead of two, and two independent dependency chains
// between barriers.
template <class TI, class TO, int CH, int WMAX, bool RES, bool BIAS, class TX = TI,
          bool PIPE = false>
__global__ void __launch_bounds__(WMAX * 32, 1)
    rmsn_bulk_kernel(const RmsnArgs a, const __grid_constant__ CUtensorMap mx,
                     const __grid_constant__ CUtensorMap mr) {
    constexpr int VE = 32 / TI::kBytes;
    constexpr int XVB = VE * TX::kBytes;  // bytes of one x vector
    // quantised outputs (per-token FP8, the block formats) are bound by
    // instruction issue here, not by DRAM: they take the packed 16-bit
    // residual add as well (the 16-bit outputs keep the fp32 add, measured
    // faster in this kernel)
    constexpr bool PADD = TO::kBytes == 1;
    // a quantised row's y stays in registers between its two passes where
    // the register budget allows it
    constexpr bool HOLD = WMAX <= 16 && CH * VE <= 32;
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[kMaxStages];
    __shared__ float red[PIPE ? 2 : 4][PIPE ? 64 : 32];
    __shared__ int abort_flag;

    const int G = blockDim.x;
    const int t = threadIdx.x;
    const int S = a.stages;
    const uint32_t x_bytes = (uint32_t)a.H * TX::kBytes;
    const uint32_t r_bytes = (uint32_t)a.H * TI::kBytes;
    const uint32_t stage_bytes = RES ? x_bytes + r_bytes : x_bytes;
    const uint32_t ring0 = a.swz ? (smem_u32(ring) + 1023u) & ~1023u : smem_u32(ring);
    // rows of this block: blockIdx.x + k * gridDim.x
    const int64_t n_my = a.T > blockIdx.x ? (a.T - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    pdl_launch_dependents(a.pdl);
    V8 wv[CH];
    V8 bv[BIAS ? CH : 1];
    if (t == 0) {
        // shared memory and the copy descriptors only: done before waiting for
        // the prerequisite grid
        abort_flag = 0;
        for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (a.swz) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mx))
                         : "memory");
            if (RES)
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mr))
                             : "memory");
        }
    }
    // thread 0: copy `row` into the stage at `dst`, completing on `bar` (a row
    // outside the tensor, in the bounds-checked build, is not copied: the
    // stage's phase completes on a plain arrival instead)
    auto issue = [&](int64_t row, uint32_t dst, uint32_t bar) {
        if (!row_ok(a, row)) {
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
            return;
        }
        if (a.swz)
            issue_row_tensor<RES>(&mx, &mr, row, dst, bar, x_bytes, r_bytes);
        else
            issue_row<RES>(a, row, dst, bar, x_bytes, r_bytes);
    };
    if (a.early_params) load_params<TX, TI, CH>(a, G, t, wv, bv, BIAS);
    pdl_wait(a.pdl);
    if (t == 0) {
        for (int64_t k = 0; k < S && k < n_my; ++k)
            issue(blockIdx.x + k * gridDim.x, ring0 + (uint32_t)k * stage_bytes,
                  smem_u32(&full[k]));
    }
    __syncthreads();
    if (!a.early_params) load_params<TX, TI, CH>(a, G, t, wv, bv, BIAS);

    int parity = 0;
    int64_t k_abort = 0;
    // the row of iteration k: x, residual -> registers (h), residual_out, and
    // this thread's sum of squares of h
    auto take_row = [&](int64_t k, V8 (&hv)[CH]) -> float {
        const int s = (int)(k % S);
        const uint32_t phase = (uint32_t)((k / S) & 1);
        const int64_t row = blockIdx.x + k * gridDim.x;
        if (!mbar_wait_bounded(smem_u32(&full[s]), phase, a.wait_cycles)) {
            atomicOr(a.status, 1u);
            abort_flag = 1;
        }
        const uint32_t base = ring0 + (uint32_t)s * stage_bytes;
        V8 rv[RES ? CH : 1];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int v = c * G + t;
            if (v < a.nvec && RMSN_CHECK(a.status, (uint32_t)(v + 1) * XVB <= x_bytes)) {
                if (a.swz) {
                    hv[c] = ld_shared_vec_swz<TX, TI>(base, (uint32_t)v);
                    if constexpr (RES) rv[c] = ld_shared32_swz(base + x_bytes, (uint32_t)v);
                } else {
                    hv[c] = ld_shared_vec<TX, TI>(base + (uint32_t)v * XVB);
                    if constexpr (RES) rv[c] = ld_shared32(base + x_bytes + (uint32_t)v * 32);
                }
            }
        }
        return residual_sumsq<TI, CH, RES, true, PADD>(a, row * (int64_t)a.H, G, t, hv, rv);
    };
    if constexpr (PIPE) {
        static_assert((std::is_same<TO, FP8>::value || std::is_same<TO, NVFP4>::value) &&
                          TX::kBytes == TI::kBytes,
                      "the two-row pipeline is built for per-token FP8 and NVFP4");
        constexpr bool NV = IsBlockFmt<TO>::value;
        V8 hp[CH];                // h of the previous row
        float ys[CH][VE];         // its y, held across the barrier
        float bms[NV ? CH : 1];   // NVFP4: the lane's maximum of each of its vectors
        float inv_p = 0.f;
        for (int64_t k = 0; k <= n_my; ++k) {
            const bool cur = k < n_my;
            V8 hv[CH];
            float acc = 0.f, amax = 0.f;
            if (k > 0) {
#pragma unroll
                for (int c = 0; c < CH; ++c) {
                    const int v = c * G + t;
                    if (v < a.nvec) {
                        opaque(wv[c]);
                        if constexpr (BIAS) opaque(bv[c]);
                        float m = 0.f;
                        scale_vec_q<TI, BIAS>(hp[c], wv[c], bv[BIAS ? c : 0], inv_p, a.woff,
                                              ys[c], m);
                        if constexpr (NV) bms[c] = m;
                        amax = fmaxf(amax, m);
                    }
                }
            }
            // row k after row k - 1's scale pass: the two h are not live together
            if (cur) {
                k_abort = k;
                acc = take_row(k, hv);
            }
            // one barrier: row k's sum of squares, row k - 1's maximum
            float sumsq, rmax;
            block_allreduce_sum_max(acc, amax, red[parity], sumsq, rmax);
            if (abort_flag) break;
            if (cur && t == 0 && k + S < n_my) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(blockIdx.x + (k + S) * gridDim.x, ring0 + (uint32_t)(k % S) * stage_bytes,
                      smem_u32(&full[k % S]));
            }
            if (k > 0) {
                const int64_t row_p = blockIdx.x + (k - 1) * gridDim.x;
                const int64_t rbase_p = row_p * (int64_t)a.H;
                if constexpr (NV) {
                    float g, rcp6g;
                    nv_row_scale<TO>(a, row_p, t, rmax, g, rcp6g);
#pragma unroll
                    for (int c = 0; c < CH; ++c) {
                        const int v = c * G + t;
                        if (v < a.nvec)
                            store_block_vec<TI, TO>(a, rbase_p + (int64_t)v * VE, v, ys[c],
                                                    bms[c], g, rcp6g);
                    }
                } else {
                    store_fp8_held<TI, CH>(a, row_p, rbase_p, G, t, ys, rmax);
                }
            }
            if (cur) {
                inv_p = inv_rms(sumsq, a.H, a.eps);
#pragma unroll
                for (int c = 0; c < CH; ++c) hp[c] = hv[c];
            }
            parity ^= 1;
        }
    } else
    for (int64_t k = 0; k < n_my; ++k) {
        const int s = (int)(k % S);
        const uint32_t phase = (uint32_t)((k / S) & 1);
        k_abort = k;
        const int64_t row = blockIdx.x + k * gridDim.x;
        const int64_t rbase = row * (int64_t)a.H;
        if (!mbar_wait_bounded(smem_u32(&full[s]), phase, a.wait_cycles)) {
            atomicOr(a.status, 1u);
            abort_flag = 1;
        }
        const uint32_t base = ring0 + (uint32_t)s * stage_bytes;
        V8 hv[CH];
        V8 rv[RES ? CH : 1];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int v = c * G + t;
            if (v < a.nvec && RMSN_CHECK(a.status, (uint32_t)(v + 1) * XVB <= x_bytes)) {
                if (a.swz) {
                    hv[c] = ld_shared_vec_swz<TX, TI>(base, (uint32_t)v);
                    if constexpr (RES) rv[c] = ld_shared32_swz(base + x_bytes, (uint32_t)v);
                } else {
                    hv[c] = ld_shared_vec<TX, TI>(base + (uint32_t)v * XVB);
                    if constexpr (RES) rv[c] = ld_shared32(base + x_bytes + (uint32_t)v * 32);
                }
            }
        }
        const float acc = residual_sumsq<TI, CH, RES, true, PADD>(a, rbase, G, t, hv, rv);
        const float sumsq = block_allreduce<false>(acc, red[parity]);
        // every thread has read buffer s: refill it with the row S ahead
        if (abort_flag) break;
        if (t == 0 && k + S < n_my) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(blockIdx.x + (k + S) * gridDim.x, base, smem_u32(&full[s]));
        }
        const float inv = inv_rms(sumsq, a.H, a.eps);
        float* slot = red[2 + parity];
        scale_store<TI, TO, CH, BIAS, HOLD, PADD && HOLD>(
            a, row, rbase, G, t, inv, hv, wv, bv,
            [&](float m) { return block_allreduce<true>(m, slot); });
        parity ^= 1;
    }
    if (abort_flag && t == 0) {
        // drain: rows k_abort .. k_abort + S - 1 may still have copies in
        // flight; wait (bounded) for each before the block's memory is reused
        for (int64_t j = k_abort; j < k_abort + S && j < n_my; ++j)
            mbar_wait_bounded(smem_u32(&full[j % S]), (uint32_t)((j / S) & 1),
                              kDefaultWaitCycles);
    }
}

// ---------------------------------------------------------------- split-row (cluster) kernel
//
// Decode-size rows split over a thread-block cluster (a split row for the
// blog's decode case, section "Prefill and decode", where the batch has too
// few rows to fill the SMs).  Each row goes to one cluster of K blocks of one
// warp; thread t = rank * 32 + lane of the row's K * 32 threads holds vectors
// v = c * 32K + t, c < CH, as in the register kernel.  The blocks exchange
// their partial sums of squares through distributed shared memory: lane j of
// each block sends the block's partial with an asynchronous store
// (st.async) into slot `rank` of block j, completing on block j's mbarrier,
// which expects 4 K bytes; each block waits (bounded) on its own mbarrier and
// adds the K partials in rank order, so all get the same total.  A relaxed
// cluster arrive at entry (after the mbarrier is initialised), waited for
// before the first remote store, ensures every block of the cluster has
// started and set up its mbarrier.  A block leaves only after all K partials
// have landed in its own shared memory, so no store into a block outlives it.
// 16-bit and fp32 outputs only (the quantised outputs would need a second
// exchange for the row maximum).

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_index() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Asynchronous store of v at the shared-memory location `local` (an address
// of this block's shared memory) in block `rank` of the cluster, completing 4
// transaction bytes on the mbarrier at `bar` (likewise this block's address)
// in that block.
__device__ __forceinline__ void st_async_cluster_f32(const void* local, const void* bar,
                                                     uint32_t rank, float v) {
    uint32_t rdst, rbar;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(rdst)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(local))), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(rbar)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar))), "r"(rank));
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(rdst),
        "r"(__float_as_uint(v)), "r"(rbar)
        : "memory");
}

constexpr int kMaxClusterBlocks = 8;

template <class TI, class TO, int CH, bool RES, bool BIAS>
__global__ void __launch_bounds__(32) rmsn_cluster_kernel(const RmsnArgs a) {
    static_assert(TO::kBytes >= 2, "16-bit and fp32 outputs only");
    __shared__ float part[kMaxClusterBlocks];
    __shared__ __align__(8) uint64_t got;  // completes when all K partials have landed
    const uint32_t rank = cluster_rank();
    const uint32_t K = cluster_size();
    const int lane = threadIdx.x;
    const int G = 32 * (int)K;
    const int t = (int)rank * 32 + lane;
    const int64_t row = cluster_index();
    if (lane == 0) {
        mbar_init(smem_u32(&got), 1);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                         smem_u32(&got)),
                     "r"(4u * K)
                     : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    cluster_arrive_relaxed();
    pdl_launch_dependents(a.pdl);
    V8 wv[CH];
    V8 bv[BIAS ? CH : 1];
    if (a.early_params) load_params<TI, TI, CH>(a, G, t, wv, bv, BIAS);
    pdl_wait(a.pdl);
    V8 hv[CH];
    V8 rv[RES ? CH : 1];
    const int64_t rbase = row * (int64_t)a.H;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const int v = c * G + t;
        const int64_t e = rbase + (int64_t)v * (32 / TI::kBytes);
        if (v < a.nvec && rows_ok(a, e, 32 / TI::kBytes)) {
            hv[c] = ld_stream32(static_cast<const char*>(a.x) + e * TI::kBytes);
            if constexpr (RES) rv[c] = ld_stream32(static_cast<const char*>(a.r) + e * TI::kBytes);
        }
    }
    if (!a.early_params) load_params<TI, TI, CH>(a, G, t, wv, bv, BIAS);
    const float acc = warp_sum(residual_sumsq<TI, CH, RES>(a, rbase, G, t, hv, rv));
    cluster_wait();  // every block of the cluster has started and set up `got`
    if (lane < (int)K) st_async_cluster_f32(&part[rank], &got, (uint32_t)lane, acc);
    if (!mbar_wait_bounded(smem_u32(&got), 0, kDefaultWaitCycles)) {
        // a partial did not arrive: report it, and wait for the stores into
        // this block once more before leaving (bounded again)
        atomicOr(a.status, 1u);
        mbar_wait_bounded(smem_u32(&got), 0, kDefaultWaitCycles);
        return;
    }
    float sumsq = part[0];
    for (uint32_t i = 1; i < K; ++i) sumsq = __fadd_rn(sumsq, part[i]);
    const float inv = inv_rms(sumsq, a.H, a.eps);
    scale_store<TI, TO, CH, BIAS>(a, row, rbase, G, t, inv, hv, wv, bv,
                                  [](float m) { return m; });
}

// ---------------------------------------------------------------- generic kernel
//
// Any hidden size and any pointer aligned to its element size.  One block per
// row (grid-stride), elements strided by the block: pass 1 forms h, stores
// residual_out and accumulates the squares; pass 2 re-reads h (from
// residual_out, written by the same thread) and writes the output; the FP8
// output takes an extra pass for the row's absmax.

template <class T>
__device__ __forceinline__ float ld_elem(const void* p, int64_t i) {
    if constexpr (T::kBytes == 2) {
        return lo2<T>((uint32_t)(static_cast<const uint16_t*>(p)[i]));
    } else {
        return static_cast<const float*>(p)[i];
    }
}

template <class T>
__device__ __forceinline__ float round_to(float v) {
    if constexpr (T::kBytes == 2) {
        return lo2<T>(pack2<T>(v, 0.f));
    } else {
        return v;
    }
}

template <class T>
__device__ __forceinline__ void st_elem(void* p, int64_t i, float v) {
    if constexpr (T::kBytes == 2) {
        static_cast<uint16_t*>(p)[i] = (uint16_t)(pack2<T>(v, 0.f) & 0xFFFFu);
    } else {
        static_cast<float*>(p)[i] = v;
    }
}

template <class TH, class TX>
__device__ __forceinline__ float generic_y(const RmsnArgs& a, const void* hsrc, int64_t base,
                                           int j, float inv) {
    if (!rows_ok(a, base + j, 1) || !cols_ok(a, j, 1)) return 0.f;
    const float h = ld_elem<TH>(hsrc, base + j);
    const float w = a.has_w ? ld_elem<TX>(a.w, j) : 1.f;
    if (a.b) return scale_elem<true>(h, inv, w, a.woff, ld_elem<TX>(a.b, j));
    return scale_elem<false>(h, inv, w, a.woff, 0.f);
}

// TX / TI as in rmsn_vec_kernel.
template <class TI, class TO, bool RES, class TX = TI>
__global__ void __launch_bounds__(256) rmsn_generic_kernel(const RmsnArgs a) {
    __shared__ float red[4][32];
    const int H = a.H;
    pdl_launch_dependents(a.pdl);
    pdl_wait(a.pdl);
    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.T; row += gridDim.x) {
        const int64_t base = row * (int64_t)H;
        float acc = 0.f;
        for (int j = threadIdx.x; j < H; j += blockDim.x) {
            if (!rows_ok(a, base + j, 1)) continue;
            float h = ld_elem<TX>(a.x, base + j);
            if constexpr (RES) {
                h = round_to<TI>(__fadd_rn(h, ld_elem<TI>(a.r, base + j)));
                st_elem<TI>(a.res_out, base + j, h);
            }
            acc = __fmaf_rn(h, h, acc);
        }
        const float inv = inv_rms(block_allreduce<false>(acc, red[parity]), H, a.eps);
        // h is re-read from residual_out (TI) or, without a residual, from x (TX == TI)
        using HSrc = TI;
        const void* hsrc = RES ? static_cast<const void*>(a.res_out) : a.x;
        float qmul = 0.f;
        if constexpr (TO::kBytes == 1) {
            float amax = 0.f;
            for (int j = threadIdx.x; j < H; j += blockDim.x) {
                amax = fmaxf(amax, fabsf(generic_y<HSrc, TX>(a, hsrc, base, j, inv)));
            }
            amax = block_allreduce<true>(amax, red[2 + parity]);
            qmul = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
            if (threadIdx.x == 0 && row_ok(a, row)) a.scale[row] = __fdiv_rn(amax, 448.f);
        }
        for (int j = threadIdx.x; j < H; j += blockDim.x) {
            if (!rows_ok(a, base + j, 1)) continue;
            const float y = generic_y<HSrc, TX>(a, hsrc, base, j, inv);
            if constexpr (TO::kBytes == 1) {
                uint16_t q;
                asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
                    : "=h"(q)
                    : "f"(0.f), "f"(__fmul_rn(y, qmul)));
                static_cast<uint8_t*>(a.out)[base + j] = (uint8_t)(q & 0xFF);
            } else {
                st_elem<TO>(a.out, base + j, y);
            }
        }
        parity ^= 1;
    }
}

// ---------------------------------------------------------------- ragged kernel
//
// Rows whose 32-byte vectors do not line up with the row (hidden not a
// multiple of the vector, or every pointer offset from a 32-byte boundary by
// the same amount): bf16, fp16 or fp32 in, and out in the same dtype, in
// fp32 / a 16-bit type (fp32 in), or as per-token FP8.  x, residual and
// residual_out share one alignment modulo 16 bytes, so each row splits the
// same way in all of them: a head (the elements before the row's first
// 16-byte boundary), an interior of 16-byte vectors, CH per thread, held in
// registers between the load and the store, and a tail.  Head and tail
// together hold at most 2 (16 / size - 1) elements, one per thread.  out is
// offset from a (16 / size) x (out size)-byte boundary by as many elements as
// x is from a 16-byte one, so each interior vector's outputs are one group on
// its own boundary.  An FP8 row takes a second pass over the registers for
// max|y| and a second block reduction.  Weight
// (plus the scalar offset) and bias are staged once per block in shared
// memory as fp32: their alignment relative to a row's vectors changes from
// row to row.  One block of 256 threads per row, rows grid-stride; the
// arithmetic (fp32 add rounded to the stream type, fp32 sum of squares,
// correctly rounded mean, reciprocal square root, scale; the FP8 scale
// max|y| / 448 and codes RN_E4M3(y * (448 / max|y|))) is that of the vector
// kernels.

template <class TI>
__device__ __forceinline__ float elem4(const uint32_t (&u)[4], int k) {
    if constexpr (TI::kBytes == 2) {
        return (k & 1) ? hi2<TI>(u[k >> 1]) : lo2<TI>(u[k >> 1]);
    } else {
        return __uint_as_float(u[k]);
    }
}

// Shared-memory slot of column j in the staged weight / bias rows: one pad
// word per 32 columns, so that the threads of a warp, whose vectors start
// 16 bytes of the row apart, read from 32 different banks.
__device__ __forceinline__ int ragged_slot(int j) { return j + (j >> 5); }

// One float as an E4M3 code (nearest-even, saturating).
__device__ __forceinline__ uint32_t e4m3_code(float v) {
    uint16_t q;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(q) : "f"(0.f), "f"(v));
    return q & 0xFFu;
}

template <class TI, class TO, int CH, bool RES, bool BIAS>
__global__ void __launch_bounds__(256, CH <= 2 ? 4 : (CH <= 4 ? 2 : 1))
    rmsn_ragged_kernel(const RmsnArgs a) {
    constexpr int S = TI::kBytes;
    constexpr int VE = 16 / S;  // elements per 16-byte vector
    constexpr bool Q = std::is_same<TO, FP8>::value;
    static_assert(Q || TO::kBytes == 2 || TO::kBytes == 4, "16-bit, fp32 or per-token FP8 out");
    // weight + offset, then bias, as fp32 in padded slots (ragged_slot)
    extern __shared__ __align__(16) float wsm[];
    __shared__ float red[4][32];
    const int H = a.H;
    const int t = threadIdx.x;
    const int G = blockDim.x;
    float* bsm = wsm + ragged_slot(H);
    pdl_launch_dependents(a.pdl);
    pdl_wait(a.pdl);
    for (int j = t; j < H; j += G) {
        if (!cols_ok(a, j, 1)) continue;
        wsm[ragged_slot(j)] = __fadd_rn(a.has_w ? ld_elem<TI>(a.w, j) : 1.f, a.woff);
        if constexpr (BIAS) bsm[ragged_slot(j)] = ld_elem<TI>(a.b, j);
    }
    __syncthreads();
    const char* xb = static_cast<const char*>(a.x);
    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.T; row += gridDim.x) {
        const int64_t e0 = row * (int64_t)H;
        const int mis = (int)(((reinterpret_cast<uintptr_t>(xb) + (uintptr_t)e0 * S) & 15u) / S);
        const int head = mis ? min(H, VE - mis) : 0;
        const int nv = (H - head) / VE;
        const int ne = H - nv * VE;  // head + tail elements
        // this thread's edge element (if any), as a column of the row
        const int je = t < head ? t : head + nv * VE + (t - head);
        uint32_t hu[CH][4];
        float he = 0.f;
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int v = c * G + t;
            const int64_t off = e0 + head + (int64_t)v * VE;
            if (v < nv && rows_ok(a, off, VE)) {
                const uint4 xw = ld_stream16(xb + off * S);
                hu[c][0] = xw.x;
                hu[c][1] = xw.y;
                hu[c][2] = xw.z;
                hu[c][3] = xw.w;
                if constexpr (RES) {
                    const uint4 rw = ld_stream16(static_cast<const char*>(a.r) + off * S);
                    const uint32_t ru[4] = {rw.x, rw.y, rw.z, rw.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        if constexpr (S == 2) {
                            hu[c][k] = pack2<TI>(__fadd_rn(lo2<TI>(hu[c][k]), lo2<TI>(ru[k])),
                                                 __fadd_rn(hi2<TI>(hu[c][k]), hi2<TI>(ru[k])));
                        } else {
                            hu[c][k] = __float_as_uint(
                                __fadd_rn(__uint_as_float(hu[c][k]), __uint_as_float(ru[k])));
                        }
                    }
                    st_stream16(static_cast<char*>(a.res_out) + off * S, hu[c]);
                }
#pragma unroll
                for (int k = 0; k < VE; ++k) {
                    const float h = elem4<TI>(hu[c], k);
                    acc = __fmaf_rn(h, h, acc);
                }
            }
        }
        if (t < ne && rows_ok(a, e0 + je, 1)) {
            he = ld_elem<TI>(a.x, e0 + je);
            if constexpr (RES) {
                he = round_to<TI>(__fadd_rn(he, ld_elem<TI>(a.r, e0 + je)));
                st_elem<TI>(a.res_out, e0 + je, he);
            }
            acc = __fmaf_rn(he, he, acc);
        }
        const float inv = inv_rms(block_allreduce<false>(acc, red[parity]), H, a.eps);
        // y of interior element k of chunk c (column col + k), and of the
        // edge element
        auto y_of = [&](int c, int col, int k) {
            const float tk = __fmul_rn(elem4<TI>(hu[c], k), inv);
            const int sl = ragged_slot(col + k);
            return BIAS ? __fmaf_rn(wsm[sl], tk, bsm[sl]) : __fmul_rn(wsm[sl], tk);
        };
        float ye = 0.f;
        if (t < ne && rows_ok(a, e0 + je, 1)) {
            const float tk = __fmul_rn(he, inv);
            const int sl = ragged_slot(je);
            ye = BIAS ? __fmaf_rn(wsm[sl], tk, bsm[sl]) : __fmul_rn(wsm[sl], tk);
        }
        float qmul = 0.f;
        if constexpr (Q) {
            // max|y| over the row: the interior recomputed from the registers
            float amax = fabsf(ye);
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const int v = c * G + t;
                if (v < nv && rows_ok(a, e0 + head + (int64_t)v * VE, VE)) {
#pragma unroll
                    for (int k = 0; k < VE; ++k)
                        amax = fmaxf(amax, fabsf(y_of(c, head + v * VE, k)));
                }
            }
            amax = block_allreduce<true>(amax, red[2 + parity]);
            qmul = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
            if (t == 0 && row_ok(a, row)) a.scale[row] = __fdiv_rn(amax, 448.f);
        }
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int v = c * G + t;
            if (v < nv && rows_ok(a, e0 + head + (int64_t)v * VE, VE)) {
                const int col = head + v * VE;
                float y[VE];
#pragma unroll
                for (int k = 0; k < VE; ++k) y[k] = y_of(c, col, k);
                if constexpr (Q) {
                    // VE codes on a VE-byte boundary: y * qmul, then E4M3
                    uint32_t u[VE / 4];
#pragma unroll
                    for (int k = 0; k < VE / 4; ++k)
                        u[k] = pack_e4m3x4(__fmul_rn(y[4 * k], qmul), __fmul_rn(y[4 * k + 1], qmul),
                                           __fmul_rn(y[4 * k + 2], qmul),
                                           __fmul_rn(y[4 * k + 3], qmul));
                    uint8_t* o = static_cast<uint8_t*>(a.out) + e0 + col;
                    if constexpr (VE == 8) st_stream8(o, u);
                    else asm volatile("st.global.b32 [%0], %1;" ::"l"(o), "r"(u[0]) : "memory");
                } else {
                    // VE outputs of TO: a VE * size-byte group on its own boundary
                    constexpr int OB = TO::kBytes;
                    char* o = static_cast<char*>(a.out) + (e0 + col) * OB;
                    if constexpr (OB == 2) {
                        uint32_t u[VE / 2];
#pragma unroll
                        for (int k = 0; k < VE / 2; ++k) u[k] = pack2<TO>(y[2 * k], y[2 * k + 1]);
                        if constexpr (VE == 8) st_stream16(o, u);
                        else st_stream8(o, u);
                    } else {
                        uint32_t u[VE];
#pragma unroll
                        for (int k = 0; k < VE; ++k) u[k] = __float_as_uint(y[k]);
                        if constexpr (VE == 8) st_stream32(o, u);
                        else st_stream16(o, u);
                    }
                }
            }
        }
        if (t < ne && rows_ok(a, e0 + je, 1)) {
            if constexpr (Q)
                static_cast<uint8_t*>(a.out)[e0 + je] = (uint8_t)e4m3_code(__fmul_rn(ye, qmul));
            else
                st_elem<TO>(a.out, e0 + je, ye);
        }
        parity ^= 1;
    }
}

}  // namespace rmsn
