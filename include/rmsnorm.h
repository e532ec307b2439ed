/*
 * rmsnorm.h -- C ABI of the GB300 (sm_103a) fused residual-add + RMSNorm.
 *
 * The operation (blog "CuTeDSL at Perplexity"; section "QK norm" defines the
 * regular RMS norm, section "Inference at Perplexity" the compile-time
 * weight-bias / dtype knobs, section "Blackwell support" the FP8 block-scaled
 * output), per token t of a row-major [n_tokens, hidden] activation:
 *
 *   h      = RN_in(x + residual)            (fp32 add, rounded to the input type;
 *                                            h = x when there is no residual)
 *   residual_out = h
 *   inv    = rsqrt(sum(h^2) / hidden + eps) (fp32 accumulation)
 *   y      = (weight + weight_offset) * (h * inv) + bias
 *   out    = RN_out(y)                      (f32 or bf16), or for FP8-E4M3:
 *            a = max|y|, out_scale[t] = a / 448,
 *            out = E4M3_RN_SATFINITE(y * 448 / a)   (all +0 when a == 0)
 *
 * weight_offset is the blog's scalar WEIGHT_BIAS added to every weight; bias is
 * a per-channel vector added after scaling.  The norm is taken on the ROUNDED
 * h, the value stored in residual_out.
 *
 * Ownership: every buffer belongs to the caller.  The library allocates no
 * device memory; it keeps per-device host-side caches (device attributes such
 * as the SM count, occupancy, and the launch chosen for each problem shape),
 * filled on first use and keyed exactly.  All calls are asynchronous
 * on `stream` (NULL = the legacy default stream) and thread-safe.
 *
 * Errors: argument errors are returned before anything is launched; a launch
 * failure returns RMSN_ECUDA (query cudaGetLastError for the cause).
 */
#ifndef RMSNORM_GB300_H
#define RMSNORM_GB300_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RMSN_OK = 0,
    RMSN_EINVAL = -1,       /* bad pointer / size / flag combination */
    RMSN_EALIGN = -2,       /* a pointer is not aligned to its element size */
    RMSN_EUNSUPPORTED = -3, /* a forced configuration that is not built */
    RMSN_ECUDA = -4         /* the CUDA runtime reported an error */
} rmsn_status;

/* flags: input dtype (x, residual, weight, bias, residual_out share it) */
#define RMSN_IN_F32 0x0u
#define RMSN_IN_BF16 0x1u
#define RMSN_IN_F16 0x2u
#define RMSN_IN_MASK 0x3u
/* output dtype of `out` */
#define RMSN_OUT_F32 0x0u
#define RMSN_OUT_BF16 0x4u
#define RMSN_OUT_FP8E4M3 0x8u
#define RMSN_OUT_F16 0xCu
#define RMSN_OUT_MASK 0xCu
/* optional operands; each must match a non-NULL pointer */
#define RMSN_HAS_RESIDUAL 0x10u /* residual and residual_out */
#define RMSN_HAS_WEIGHT 0x20u   /* weight (else 1) */
#define RMSN_HAS_BIAS 0x40u     /* bias (else 0) */
#define RMSN_RESIDUAL_F32 0x200u /* with RMSN_HAS_RESIDUAL and bf16 / fp16 input: residual
                                   and residual_out are fp32 (an fp32 residual stream);
                                   h = x + residual is kept in fp32, not rounded to the
                                   input type, and the norm is taken on it.  Built for
                                   outputs of the input dtype and FP8 (other outputs:
                                   RMSN_EUNSUPPORTED).  Vector kernels need
                                   hidden % 8 == 0, 16-byte aligned x / weight / bias
                                   and 32-byte aligned residuals. */
/* launch options (blog section "Grid synchronisation": programmatic dependent
 * launch cuts the launch overhead of chained kernels) */
#define RMSN_PDL 0x80u /* launch with programmatic stream serialization: the kernel
                          may start while the preceding kernel in the stream still
                          runs, and waits for it (and its memory) before reading
                          any input; it lets its own successor start at once */
#define RMSN_PDL_EARLY_PARAMS 0x100u /* with RMSN_PDL: weight and bias are not written
                                        by the preceding kernel and may be read
                                        before it ends */

/* kernel variants */
typedef enum {
    RMSN_VARIANT_WARP_ROWS = 0, /* decode: one warp per row, rows spread over SMs */
    RMSN_VARIANT_BLOCK_ROW = 1, /* prefill: one block (W warps) per row, register-resident */
    RMSN_VARIANT_BULK_ROW = 2,  /* prefill: persistent blocks; rows streamed into a ring of
                                   shared-memory buffers by TMA copies: 128-byte-swizzled 2-D
                                   tensor copies where a row is whole 1 KiB units of at most
                                   32 KiB, else 1-D bulk copies */
    RMSN_VARIANT_GENERIC = 3,   /* any hidden size / alignment (element-wise, three passes) */
    RMSN_VARIANT_RAGGED = 4,    /* rows off the 32-byte grid, same dtype in and out, all row
                                   pointers equally aligned mod 16 bytes: 16-byte vectors for
                                   the row's interior, single elements for head and tail */
    RMSN_VARIANT_CLUSTER = 5,   /* decode: each row split over a thread-block cluster of
                                   `cluster` one-warp blocks that exchange partial sums of
                                   squares through distributed shared memory (bf16 / fp16 /
                                   fp32 in with the same dtype out, not FP8) */
    RMSN_VARIANT_BULK_PIPE = 6  /* the bulk-copy ring with a two-row pipeline: one block
                                   barrier carries a row's sum of squares and the previous
                                   row's maximum (bf16 / fp16 in, per-token FP8 or NVFP4 out) */
} rmsn_variant;

/* One launch configuration. */
typedef struct {
    int32_t variant;         /* rmsn_variant */
    int32_t vec_bytes;       /* bytes per thread per access (32 = 256-bit) */
    int32_t warps_per_block; /* launched warps per block */
    int32_t warps_per_row;   /* warps that share one row */
    int32_t chunks;          /* vectors per thread per row (template) */
    int32_t max_warps;       /* template block-size bound (register budget) */
    int32_t stages;          /* shared-memory row buffers (bulk variants) */
    int32_t grid;            /* blocks launched */
    int32_t smem_bytes;      /* dynamic shared memory per block */
    int32_t num_sms;         /* SMs of the device the config was made for */
    int32_t ring_copy;       /* bulk variant: 2 = swizzled 2-D tensor copies, 1 = 1-D bulk
                                copies; 0 for the other variants (output only) */
    int32_t cluster;         /* cluster variant: blocks per row (its max_warps); else 0
                                (output only) */
} rmsn_config;

/*
 * Fused residual-add + RMSNorm over x[n_tokens, hidden].
 *
 *   x, residual, residual_out : [n_tokens, hidden] of the input dtype
 *   weight, bias               : [hidden] of the input dtype
 *   out                        : [n_tokens, hidden] of the output dtype
 *   out_scale                  : [n_tokens] float32, required iff FP8 output
 *   eps                        : added to the mean square inside the root
 *
 * All pointers are device (or device-resident managed) pointers, rows
 * contiguous (row stride = hidden); for rows in host memory use
 * rmsnorm_fwd_host.  Each pointer must be aligned to its
 * element size; the 256-bit vector kernels are used when hidden * element
 * size is a multiple of 32 bytes and every pointer is 32-byte aligned;
 * otherwise rows of bf16 / fp16 / fp32 (not over an fp32 residual stream)
 * take the ragged-row kernel (16-byte vectors plus single-element row ends)
 * when x, residual and residual_out are equally aligned modulo 16 bytes and
 * out, of the same dtype, per-token FP8, fp32 (16-bit rows) or 16-bit (fp32
 * rows), is offset from a (16 / input element size) x (output element
 * size)-byte boundary by as many elements as x is from a 16-byte one; the
 * rest take the generic kernel.
 * residual_out may be the same buffer as
 * residual, or as x when both have the same dtype; out may be the same
 * buffer as x or residual when their dtypes are equal; any other overlap is
 * undefined.  n_tokens == 0
 * is a no-op once the flags, hidden and eps have been checked (its pointers
 * may then be NULL).  Returns an rmsn_status.
 */
int rmsnorm_fwd(const void* x, const void* residual, const void* weight, const void* bias,
                void* out, void* residual_out, float* out_scale, int64_t n_tokens,
                int64_t hidden, float eps, uint32_t flags, cudaStream_t stream);

/*
 * rmsnorm_fwd with the scalar weight offset (the blog's WEIGHT_BIAS; 0 in
 * rmsnorm_fwd) and an optional forced configuration (`cfg` NULL = the
 * selector's choice).  A forced configuration must name a built variant;
 * its grid is used when > 0 (else the default grid for that variant).
 */
int rmsnorm_fwd_ex(const void* x, const void* residual, const void* weight, const void* bias,
                   void* out, void* residual_out, float* out_scale, int64_t n_tokens,
                   int64_t hidden, float eps, uint32_t flags, float weight_offset,
                   const rmsn_config* cfg, cudaStream_t stream);

/* block-scaled output formats of rmsnorm_fwd_blockscaled */
#define RMSN_FMT_MXFP8 1 /* E4M3 codes, one E8M0 scale per 32 elements */
#define RMSN_FMT_MXFP4 2 /* E2M1 codes (two per byte, low nibble first), E8M0 per 32 */
#define RMSN_FMT_NVFP4 3 /* E2M1 codes (packed), E4M3 scale per 16, fp32 scale per token */

/*
 * Fused residual-add + RMSNorm with a block-scaled quantised output (blog
 * section "Blackwell support": MXFP8 / MXFP4 / NVFP4, absolute maximum over
 * 32 or 16 elements).  The norm is that of rmsnorm_fwd; y is then encoded:
 *
 *   MXFP8 / MXFP4: per block of 32 elements, s = floor(log2(max|y|)) - emax
 *     (emax 8 for E4M3, 2 for E2M1) clamped to [-127, 127], stored as E8M0
 *     code s + 127 in block_scale[T, hidden/32]; codes RN_sat(y * 2^-s).
 *     An all-zero block stores code 0 and zero codes.
 *   NVFP4: token_scale[t] = g = max|row| / (448 * 6) (fp32); per block of 16
 *     elements E4M3 scale c_b = RN_sat(max|block| / (6 g)) in
 *     block_scale[T, hidden/16]; codes E2M1 RN_sat(y * r_b), where r_b is
 *     1 / (c_b g) to within 1 fp32 ulp (a hardware reciprocal), so a code can
 *     be one step from RN_sat(y / (c_b g)) when that quotient lies within a
 *     few fp32 ulp of an E2M1 rounding midpoint.
 *
 * out is [T, hidden] bytes (MXFP8) or [T, hidden/2] bytes (FP4, element 2j
 * in the low nibble).  Rounding is to nearest even with saturation.  flags
 * as for rmsnorm_fwd with the output-dtype bits 0; the input must be bf16,
 * hidden a multiple of 32 (MX) or 16 (NVFP4), and the vector-path
 * alignment of rmsnorm_fwd must hold (else RMSN_EUNSUPPORTED).  token_scale
 * is required iff NVFP4.  `cfg` as in rmsnorm_fwd_ex (NULL = selector).
 */
int rmsnorm_fwd_blockscaled(const void* x, const void* residual, const void* weight,
                            const void* bias, void* out, void* block_scale, float* token_scale,
                            void* residual_out, int64_t n_tokens, int64_t hidden, float eps,
                            uint32_t flags, int format, float weight_offset,
                            const rmsn_config* cfg, cudaStream_t stream);

/*
 * rmsnorm_fwd_ex on rows that live in HOST memory: the kernel itself reads x,
 * residual (and weight, bias) across the CPU-GPU link and writes out,
 * residual_out and out_scale back to host memory, with no staging buffer and
 * no allocation (on Grace-Blackwell the link is the coherent NVLink-C2C).
 *
 * Each pointer may be device memory of the current device, managed memory,
 * page-locked host memory (cudaHostAlloc, cudaMallocHost, cudaHostRegister,
 * torch pin_memory), or ordinary pageable host memory when the device
 * reports pageable-memory access (cudaDevAttrPageableMemoryAccess); any mix
 * is allowed.  A pointer the device cannot reach, including device memory of
 * another GPU, returns RMSN_EINVAL before any launch.  Only the
 * register-streaming kernels run here (plain loads and stores), shaped for
 * the link's latency: one block per row, one 32-byte vector per thread where
 * the row allows it.  The call is asynchronous on `stream`: host outputs are
 * complete once the stream has been synchronised.  The operation, aliasing
 * and alignment rules are those of rmsnorm_fwd.  Returns an rmsn_status.
 */
int rmsnorm_fwd_host(const void* x, const void* residual, const void* weight, const void* bias,
                     void* out, void* residual_out, float* out_scale, int64_t n_tokens,
                     int64_t hidden, float eps, uint32_t flags, float weight_offset,
                     cudaStream_t stream);

/*
 * QK norm (blog "CuTeDSL at Perplexity", section "QK norm"): per-head RMS
 * norm of query and key heads, IN PLACE.  Every head of head_dim elements is
 * normalised on its own:
 *
 *   inv = rsqrt(sum(x^2) / head_dim + eps);  x <- RN((w + weight_offset) * (x * inv))
 *
 * with w = q_weight[head_dim] for query heads and k_weight[head_dim] for key
 * heads (NULL = 1).  Token t's query heads start at element t * q_token_stride
 * of q (n_q_heads heads of head_dim elements, back to back); likewise k.  The
 * strides let q and k sit inside a fused qkv row; elements outside the heads
 * are not touched.  The q buffer must span (n_tokens - 1) * q_token_stride +
 * n_q_heads * head_dim elements (likewise k).  flags: RMSN_IN_F32,
 * RMSN_IN_BF16 or RMSN_IN_F16 (q, k and weights share it), optionally
 * RMSN_PDL, and at most one of RMSN_QK_RING / RMSN_QK_DIRECT.  One launch
 * covers both q and k, by a one-pass register kernel; RMSN_QK_RING asks for a
 * ring variant instead (heads of 4 to 32 whole 32-byte vectors, a power of
 * two, at most 2048 per token), in which persistent blocks stream each
 * token's query and key heads into shared memory with TMA bulk copies and hold
 * the weights in registers.  Without a weight offset the 16-bit kernels form
 * x * w exactly and round once more, for (x * w) * inv.  The fast path needs head_dim * element size to be a
 * multiple of 32 bytes and at most 1024 bytes (head_dim 64, 128, 256 in bf16
 * and fp32, 512 in bf16), 32-byte aligned pointers and token strides, and at
 * most 65535 x 16 warps' worth of heads per token (32 / lanes-per-head heads
 * a warp: over a million heads at head_dim 512 bf16); otherwise
 * RMSN_EUNSUPPORTED.  Returns an rmsn_status.
 */
#define RMSN_QK_RING 0x400u   /* rmsnorm_qk_fwd: take the ring variant whatever the batch
                                 (RMSN_EUNSUPPORTED where it does not apply); for tests
                                 and tuning */
#define RMSN_QK_DIRECT 0x800u /* rmsnorm_qk_fwd: take the one-pass register kernel */

int rmsnorm_qk_fwd(void* q, void* k, const void* q_weight, const void* k_weight,
                   int64_t n_tokens, int64_t n_q_heads, int64_t n_k_heads, int64_t head_dim,
                   int64_t q_token_stride, int64_t k_token_stride, float eps,
                   float weight_offset, uint32_t flags, cudaStream_t stream);

/*
 * The configuration rmsnorm_fwd would launch for this shape on the current
 * device, assuming 32-byte aligned pointers.  Returns an rmsn_status.
 */
int rmsnorm_query_config(int64_t n_tokens, int64_t hidden, uint32_t flags, rmsn_config* out);

/*
 * Every built configuration that can run this shape (for sweeps and tests).
 * Writes up to `capacity` entries; returns the total number available, or a
 * negative rmsn_status.
 */
int rmsnorm_list_configs(int64_t n_tokens, int64_t hidden, uint32_t flags, rmsn_config* out,
                         int capacity);

/*
 * Status word of the library's kernels on the current device.  Bit 0 is set
 * when a bounded wait inside a kernel (the bulk-copy variant waits about one
 * second at most for a row to arrive in shared memory) ran out; that kernel's
 * outputs are then incomplete.  Reads synchronously (the device's pending
 * work is not waited for beyond the copy's own ordering); `clear` != 0 resets
 * the word.  Returns an rmsn_status.
 */
int rmsnorm_read_status(uint32_t* status, int clear);

/*
 * Testing hook for the bounded waits of the bulk-copy variant (not needed in
 * normal use).  Sets, for launches that follow on the current device, how
 * many SM clock cycles a block waits for a row to arrive in shared memory
 * before it gives up: it then sets bit 0 of the status word, leaves the
 * remaining rows unwritten (the row it was waiting for may have a partly
 * written residual_out and no output), waits with the default bound for the
 * copies it has in flight, and returns.  0 restores the default (about one
 * second); a negative value makes each wait test the row's barrier once and
 * not wait at all, so that the give-up path runs on a healthy GPU.  Returns
 * an rmsn_status.
 */
int rmsnorm_set_wait_limit(int64_t cycles);

/* Human-readable name of an rmsn_status. */
const char* rmsnorm_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* RMSNORM_GB300_H */
