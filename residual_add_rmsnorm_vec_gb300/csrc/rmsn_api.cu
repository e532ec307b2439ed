// C ABI of the fused residual-add + RMSNorm: argument validation, the
// per-device attribute cache, the launch-configuration selector and the
// launch itself.  Declared in include/rmsnorm.h.
//
// Selector (blog "CuTeDSL at Perplexity", sections "Prefill and decode" and
// "Blackwell support"): pick the per-thread vector for the widest access
// (32 bytes = 16 bf16 / 8 fp32 on Blackwell), count the warps the whole
// problem needs, and if that is no more than the SM count use the decode
// shape (one warp per block, so the rows land on as many SMs as possible);
// otherwise use multi-warp blocks, with the warp count per hidden size taken
// from a table of measured bandwidth (rmsn_selector_table.inc) and a fixed
// rule where the table has no entry.  The SM count is queried from the
// device once, not compiled in.
#include <cuda_runtime.h>

#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "../../include/rmsnorm.h"
#include "rmsn_registry.h"

#define RMSN_API extern "C" __attribute__((visibility("default")))

namespace rmsn {
namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxHidden = int64_t(1) << 24;

struct DeviceInfo {
    std::once_flag once;
    int num_sms = 0;
    cudaError_t err = cudaSuccess;
};

DeviceInfo g_dev[kMaxDevices];

// SM count of the current device (queried once per device).
int device_sms(int* dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    DeviceInfo& d = g_dev[dev];
    std::call_once(d.once, [&] {
        int n = 0;
        d.err = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        d.num_sms = n;
    });
    if (dev_out) *dev_out = dev;
    return d.err == cudaSuccess ? d.num_sms : -1;
}

const std::vector<KernelEntry>& registry() {
    static const std::vector<KernelEntry> all = [] {
        std::vector<KernelEntry> v;
        const KernelEntry* (*fns[])(int*) = {kernels_f32_f32,  kernels_f32_bf16,  kernels_f32_fp8,
                                             kernels_bf16_f32, kernels_bf16_bf16, kernels_bf16_fp8};
        for (auto fn : fns) {
            int n = 0;
            const KernelEntry* t = fn(&n);
            v.insert(v.end(), t, t + n);
        }
        return v;
    }();
    return all;
}

struct Problem {
    int64_t T, H;
    int in_dt, out_dt;
    bool res, bias;
    int in_bytes, out_bytes;
    int ve;     // elements per 32-byte vector
    int nvec;   // vectors per row (valid when vec_ok)
    bool vec_ok;
};

int dtype_bytes(int dt) { return dt == kF32 ? 4 : (dt == kBF16 ? 2 : 1); }

bool aligned(const void* p, uintptr_t a) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int decode_flags(uint32_t flags, Problem* p) {
    const uint32_t known = RMSN_IN_MASK | RMSN_OUT_MASK | RMSN_HAS_RESIDUAL | RMSN_HAS_WEIGHT |
                           RMSN_HAS_BIAS;
    if (flags & ~known) return RMSN_EINVAL;
    const uint32_t in = flags & RMSN_IN_MASK, out = flags & RMSN_OUT_MASK;
    if (in == RMSN_IN_F32) p->in_dt = kF32;
    else if (in == RMSN_IN_BF16) p->in_dt = kBF16;
    else return RMSN_EINVAL;
    if (out == RMSN_OUT_F32) p->out_dt = kF32;
    else if (out == RMSN_OUT_BF16) p->out_dt = kBF16;
    else if (out == RMSN_OUT_FP8E4M3) p->out_dt = kFP8;
    else return RMSN_EINVAL;
    p->res = (flags & RMSN_HAS_RESIDUAL) != 0;
    p->bias = (flags & RMSN_HAS_BIAS) != 0;
    p->in_bytes = dtype_bytes(p->in_dt);
    p->out_bytes = dtype_bytes(p->out_dt);
    p->ve = 32 / p->in_bytes;
    return RMSN_OK;
}

int check_shape(int64_t T, int64_t H, Problem* p) {
    if (T < 0 || H < 1 || H > kMaxHidden) return RMSN_EINVAL;
    if (T > (INT64_MAX / 8) / H) return RMSN_EINVAL;
    p->T = T;
    p->H = H;
    return RMSN_OK;
}

// Can the 32-byte vector kernels run with these pointers?
bool vector_path_ok(const Problem& p, const void* const* ptrs, int n, const void* out) {
    if ((p.H * p.in_bytes) % 32 != 0) return false;
    for (int i = 0; i < n; ++i)
        if (!aligned(ptrs[i], 32)) return false;
    const int out_vec = p.ve * p.out_bytes;  // bytes stored per input vector
    return aligned(out, out_vec < 32 ? out_vec : 32);
}

const KernelEntry* find_kernel(const Problem& p, int variant, int ch, int wmax) {
    for (const KernelEntry& e : registry()) {
        if (e.in_dt != p.in_dt || e.out_dt != p.out_dt || e.variant != variant) continue;
        if (e.res != (p.res ? 1 : 0)) continue;
        if (variant == kGeneric) return &e;
        if (e.bias != (p.bias ? 1 : 0)) continue;
        if (e.chunks == ch && e.max_warps == wmax) return &e;
    }
    return nullptr;
}

int blocks_per_sm(const void* fn, int threads) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, 0) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    return n > 0 ? n : 1;
}

// Fill block shape, grid (persistent: at most one resident wave) for an entry.
bool shape_config(const Problem& p, const KernelEntry& e, int sms, int grid_req, rmsn_config* c) {
    memset(c, 0, sizeof(*c));
    c->variant = e.variant;
    c->chunks = e.chunks;
    c->max_warps = e.max_warps;
    c->num_sms = sms;
    int threads;
    int64_t units;  // rows handled per block-step
    if (e.variant == kGeneric) {
        c->vec_bytes = p.in_bytes;
        int w = (int)((p.H + 31) / 32);
        if (w > 8) w = 8;
        c->warps_per_block = w;
        c->warps_per_row = w;
        threads = w * 32;
        units = p.T;
    } else if (e.variant == kWarpRows) {
        if (p.nvec > 32 * e.chunks) return false;
        if (e.chunks > 1 && p.nvec <= 32 * (e.chunks / 2)) return false;  // a smaller CH fits
        c->vec_bytes = 32;
        c->warps_per_block = e.max_warps;
        c->warps_per_row = 1;
        threads = e.max_warps * 32;
        units = (p.T + e.max_warps - 1) / e.max_warps;
    } else {
        const int w = (int)((p.nvec + 32 * e.chunks - 1) / (32 * e.chunks));
        if (w > e.max_warps) return false;
        c->vec_bytes = 32;
        c->warps_per_block = w;
        c->warps_per_row = w;
        threads = w * 32;
        units = p.T;
    }
    const int64_t resident = (int64_t)sms * blocks_per_sm(e.fn, threads);
    int64_t grid = units < resident ? units : resident;
    if (grid_req > 0) grid = grid_req < units ? grid_req : units;
    if (grid < 1) grid = 1;
    c->grid = (int32_t)grid;
    return true;
}

#include "rmsn_selector_table.inc"

// The selector (see the file comment).
bool select(const Problem& p, int sms, rmsn_config* c) {
    if (!p.vec_ok) {
        const KernelEntry* e = find_kernel(p, kGeneric, 0, 0);
        return e && shape_config(p, *e, sms, 0, c);
    }
    const int64_t warps_needed = (p.T * p.nvec + 31) / 32;
    if (warps_needed <= sms && p.nvec <= 32 * 8) {
        // decode: one warp per block, CH = smallest power of two covering the row
        int ch = 1;
        while (32 * ch < p.nvec) ch *= 2;
        const KernelEntry* e = find_kernel(p, kWarpRows, ch, 1);
        if (e && shape_config(p, *e, sms, 0, c)) return true;
    }
    // measured table, then the fixed rule: fewest warps with CH <= 2 that fit
    int ch = 0, wmax = 0;
    if (!table_lookup(p.in_dt, p.out_dt, p.H, p.T, &ch, &wmax)) {
        const int cands[][2] = {{2, 4}, {2, 8}, {2, 16}, {2, 32}, {4, 16}};
        for (auto& cw : cands) {
            const int w = (int)((p.nvec + 32 * cw[0] - 1) / (32 * cw[0]));
            if (w <= cw[1]) {
                ch = cw[0];
                wmax = cw[1];
                break;
            }
        }
    }
    if (ch) {
        const KernelEntry* e = find_kernel(p, kBlockRow, ch, wmax);
        if (e && shape_config(p, *e, sms, 0, c)) return true;
    }
    const KernelEntry* e = find_kernel(p, kGeneric, 0, 0);
    return e && shape_config(p, *e, sms, 0, c);
}

}  // namespace
}  // namespace rmsn

using namespace rmsn;

RMSN_API const char* rmsnorm_status_string(int status) {
    switch (status) {
        case RMSN_OK: return "RMSN_OK";
        case RMSN_EINVAL: return "RMSN_EINVAL: invalid argument";
        case RMSN_EALIGN: return "RMSN_EALIGN: pointer not aligned to its element size";
        case RMSN_EUNSUPPORTED: return "RMSN_EUNSUPPORTED: configuration not built";
        case RMSN_ECUDA: return "RMSN_ECUDA: CUDA runtime error";
        default: return "unknown rmsn_status";
    }
}

RMSN_API int rmsnorm_fwd_ex(const void* x, const void* residual, const void* weight,
                            const void* bias, void* out, void* residual_out, float* out_scale,
                            int64_t n_tokens, int64_t hidden, float eps, uint32_t flags,
                            float weight_offset, const rmsn_config* cfg, cudaStream_t stream) {
    Problem p{};
    int st = decode_flags(flags, &p);
    if (st != RMSN_OK) return st;
    if ((st = check_shape(n_tokens, hidden, &p)) != RMSN_OK) return st;
    if (!(eps >= 0.f) || !isfinite(eps) || !isfinite(weight_offset)) return RMSN_EINVAL;
    // optional operands must match their flags exactly
    if (p.res != (residual != nullptr) || p.res != (residual_out != nullptr)) return RMSN_EINVAL;
    if (((flags & RMSN_HAS_WEIGHT) != 0) != (weight != nullptr)) return RMSN_EINVAL;
    if (p.bias != (bias != nullptr)) return RMSN_EINVAL;
    if ((p.out_dt == kFP8) != (out_scale != nullptr)) return RMSN_EINVAL;
    if (n_tokens == 0) return RMSN_OK;
    if (!x || !out) return RMSN_EINVAL;
    const void* ins[] = {x, residual, weight, bias, residual_out};
    for (const void* q : ins)
        if (!aligned(q, (uintptr_t)p.in_bytes)) return RMSN_EALIGN;
    if (!aligned(out, (uintptr_t)p.out_bytes) || !aligned(out_scale, 4)) return RMSN_EALIGN;
    p.vec_ok = vector_path_ok(p, ins, 5, out);
    p.nvec = p.vec_ok ? (int)(p.H / p.ve) : 0;

    const int sms = device_sms(nullptr);
    if (sms <= 0) return RMSN_ECUDA;
    rmsn_config c;
    const KernelEntry* e = nullptr;
    if (cfg) {
        if (cfg->variant != kGeneric && !p.vec_ok) return RMSN_EUNSUPPORTED;
        e = find_kernel(p, cfg->variant, cfg->chunks, cfg->max_warps);
        if (!e || !shape_config(p, *e, sms, cfg->grid, &c)) return RMSN_EUNSUPPORTED;
    } else {
        if (!select(p, sms, &c)) return RMSN_EUNSUPPORTED;
        e = find_kernel(p, c.variant, c.chunks, c.max_warps);
        if (!e) return RMSN_EUNSUPPORTED;
    }

    RmsnArgs a;
    a.x = x;
    a.r = residual;
    a.w = weight;
    a.b = bias;
    a.out = out;
    a.res_out = residual_out;
    a.scale = out_scale;
    a.T = p.T;
    a.H = (int32_t)p.H;
    a.nvec = p.nvec;
    a.eps = eps;
    a.woff = weight_offset;
    a.has_w = weight != nullptr;
    void* args[] = {&a};
    const cudaError_t err = cudaLaunchKernel(e->fn, dim3((unsigned)c.grid),
                                             dim3((unsigned)(c.warps_per_block * 32)), args,
                                             (size_t)c.smem_bytes, stream);
    return err == cudaSuccess ? RMSN_OK : RMSN_ECUDA;
}

RMSN_API int rmsnorm_fwd(const void* x, const void* residual, const void* weight,
                         const void* bias, void* out, void* residual_out, float* out_scale,
                         int64_t n_tokens, int64_t hidden, float eps, uint32_t flags,
                         cudaStream_t stream) {
    return rmsnorm_fwd_ex(x, residual, weight, bias, out, residual_out, out_scale, n_tokens,
                          hidden, eps, flags, 0.f, nullptr, stream);
}

static int query_problem(int64_t n_tokens, int64_t hidden, uint32_t flags, Problem* p) {
    int st = decode_flags(flags, p);
    if (st != RMSN_OK) return st;
    if ((st = check_shape(n_tokens, hidden, p)) != RMSN_OK) return st;
    p->vec_ok = (p->H * p->in_bytes) % 32 == 0;
    p->nvec = p->vec_ok ? (int)(p->H / p->ve) : 0;
    return RMSN_OK;
}

RMSN_API int rmsnorm_query_config(int64_t n_tokens, int64_t hidden, uint32_t flags,
                                  rmsn_config* out) {
    if (!out) return RMSN_EINVAL;
    Problem p{};
    int st = query_problem(n_tokens, hidden, flags, &p);
    if (st != RMSN_OK) return st;
    const int sms = device_sms(nullptr);
    if (sms <= 0) return RMSN_ECUDA;
    return select(p, sms, out) ? RMSN_OK : RMSN_EUNSUPPORTED;
}

RMSN_API int rmsnorm_list_configs(int64_t n_tokens, int64_t hidden, uint32_t flags,
                                  rmsn_config* out, int capacity) {
    if (capacity < 0 || (capacity > 0 && !out)) return RMSN_EINVAL;
    Problem p{};
    int st = query_problem(n_tokens, hidden, flags, &p);
    if (st != RMSN_OK) return st;
    const int sms = device_sms(nullptr);
    if (sms <= 0) return RMSN_ECUDA;
    int count = 0;
    for (const KernelEntry& e : registry()) {
        if (e.in_dt != p.in_dt || e.out_dt != p.out_dt || e.res != (p.res ? 1 : 0)) continue;
        if (e.variant != kGeneric && (e.bias != (p.bias ? 1 : 0) || !p.vec_ok)) continue;
        rmsn_config c;
        if (!shape_config(p, e, sms, 0, &c)) continue;
        if (count < capacity) out[count] = c;
        ++count;
    }
    return count;
}
