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
#include <cuda.h>
#include <cuda_runtime.h>

#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <unordered_map>
#include <utility>
#include <vector>

#include "../../include/rmsnorm.h"
#include "rmsn_qk.h"
#include "rmsn_registry.h"

#define RMSN_API extern "C" __attribute__((visibility("default")))

namespace rmsn {
namespace {

constexpr int kMaxDevices = 64;
// QK norm's ring variant is taken only when asked for (RMSN_QK_RING): measured
// on GB300 the one-pass register kernel finished sooner at every batch size.
// About this many bytes of token buffers per ring block.
constexpr int64_t kQkRingTokens = INT64_MAX;
constexpr int64_t kQkRingBytes = 96 * 1024;
// x extent of the one-pass QK grid (token groups); more tokens loop
constexpr int64_t kQkMaxGridX = int64_t(1) << 30;
constexpr int64_t kMaxHidden = int64_t(1) << 24;

// Status word of the kernels on each device (bit 0: a bounded wait ran out).
__device__ uint32_t g_status;

// Cache keys compared in full (a hash only picks the bucket): two problems
// that hash alike must never share a launch.
struct SelKey {
    int64_t T, H;
    uint32_t flags;
    int paths;  // bit 0: vector path, bit 1: ragged-row path
    int fmt;    // block-scaled output format (0: the output dtype of `flags`)
    bool operator==(const SelKey& o) const {
        return T == o.T && H == o.H && flags == o.flags && paths == o.paths && fmt == o.fmt;
    }
};
struct OccKey {
    const void* fn;
    int threads, smem;
    bool operator==(const OccKey& o) const {
        return fn == o.fn && threads == o.threads && smem == o.smem;
    }
};
inline uint64_t mix(uint64_t h, uint64_t v) {
    h ^= v + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
    return h;
}
struct SelKeyHash {
    size_t operator()(const SelKey& k) const {
        return (size_t)mix(mix(mix(mix((uint64_t)k.T, (uint64_t)k.H), k.flags), (uint64_t)k.paths),
                           (uint64_t)k.fmt);
    }
};
struct OccKeyHash {
    size_t operator()(const OccKey& k) const {
        return (size_t)mix(mix(reinterpret_cast<uintptr_t>(k.fn), (uint64_t)k.threads),
                           (uint64_t)k.smem);
    }
};

// A ring tensor map is a pure function of (base address, rows, row length,
// element size): a cached map is reused whenever all four match.
struct MapEntry {
    const void* base = nullptr;
    int64_t T = 0, H = 0;
    int bytes = 0;
    CUtensorMap map;  // the type carries its own alignment
};
constexpr int kMapCache = 32;

struct DeviceInfo {
    std::once_flag once;
    int num_sms = 0;
    int max_smem = 0;              // opt-in dynamic shared memory per block
    int pageable_access = 0;       // device can read and write pageable host memory
    uint32_t* status = nullptr;    // device address of g_status on this device
    std::atomic<int64_t> wait_cycles{kDefaultWaitCycles};  // ring wait bound (tests may lower it)
    cudaError_t err = cudaSuccess;
    std::mutex mu;
    std::vector<std::pair<const void*, int>> smem_set;  // kernel -> raised dynamic smem limit
    // occupancy results: (kernel, threads, smem) -> resident blocks per SM
    std::unordered_map<OccKey, int, OccKeyHash> occ_cache;
    // selector results: (tokens, hidden, flags, vector path) -> configuration
    std::unordered_map<SelKey, std::pair<rmsn_config, const KernelEntry*>, SelKeyHash> sel_cache;
    // tensor maps of the ring kernel's 2-D copies, replaced round-robin
    MapEntry maps[kMapCache];
    int map_next = 0;
};

DeviceInfo g_dev[kMaxDevices];

// Attributes of the current device (queried once per device).
DeviceInfo* device_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    DeviceInfo& d = g_dev[dev];
    std::call_once(d.once, [&] {
        int n = 0, sm = 0;
        d.err = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (d.err == cudaSuccess)
            d.err = cudaDeviceGetAttribute(&sm, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (d.err == cudaSuccess)
            d.err = cudaDeviceGetAttribute(&d.pageable_access, cudaDevAttrPageableMemoryAccess, dev);
        if (d.err == cudaSuccess) d.err = cudaGetSymbolAddress((void**)&d.status, g_status);
        d.num_sms = n;
        d.max_smem = sm;
    });
    if (d.err != cudaSuccess) return nullptr;
    return &d;
}

// Let a bulk kernel use the device's opt-in shared memory, less its static
// shared memory (once per device and kernel); returns the dynamic limit or 0.
int enable_smem(DeviceInfo* d, const void* fn) {
    std::lock_guard<std::mutex> lock(d->mu);
    for (const auto& f : d->smem_set)
        if (f.first == fn) return f.second;
    cudaFuncAttributes attr;
    if (cudaFuncGetAttributes(&attr, fn) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    const int limit = d->max_smem - (int)attr.sharedSizeBytes;
    if (limit <= 0 ||
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, limit) !=
            cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    d->smem_set.emplace_back(fn, limit);
    return limit;
}

const std::vector<KernelEntry>& registry() {
    static const std::vector<KernelEntry> all = [] {
        std::vector<KernelEntry> v;
        const KernelEntry* (*fns[])(int*) = {
            kernels_f32_f32,  kernels_f32_bf16,  kernels_f32_fp8,    kernels_f32_f16,
            kernels_bf16_f32, kernels_bf16_bf16, kernels_bf16_fp8,   kernels_f16_f16,
            kernels_f16_f32,  kernels_f16_fp8,   kernels_bf16_mxfp8, kernels_bf16_mxfp4,
            kernels_bf16_nvfp4, kernels_bf16r32_bf16, kernels_bf16r32_fp8, kernels_f16r32_f16,
            kernels_f16r32_fp8, kernels_ragged, kernels_ragged_fp8, kernels_ragged_mixed};
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
    bool pdl, early_params;  // launch options
    int in_bytes, out_bytes;
    bool res_f32;   // fp32 residual stream (residual, residual_out, h) under bf16 / fp16 x
    int res_bytes;  // element size of the residual stream
    int ve;     // elements per 32-byte vector
    int nvec;   // vectors per row (valid when vec_ok)
    bool vec_ok;
    bool ragged_ok;  // off the 32-byte grid, but the ragged-row kernel applies
};

int dtype_bytes(int dt) { return dt == kF32 ? 4 : ((dt == kBF16 || dt == kF16) ? 2 : 1); }

bool aligned(const void* p, uintptr_t a) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int decode_flags(uint32_t flags, Problem* p) {
    const uint32_t known = RMSN_IN_MASK | RMSN_OUT_MASK | RMSN_HAS_RESIDUAL | RMSN_HAS_WEIGHT |
                           RMSN_HAS_BIAS | RMSN_PDL | RMSN_PDL_EARLY_PARAMS | RMSN_RESIDUAL_F32;
    if (flags & ~known) return RMSN_EINVAL;
    const uint32_t in = flags & RMSN_IN_MASK, out = flags & RMSN_OUT_MASK;
    if (in == RMSN_IN_F32) p->in_dt = kF32;
    else if (in == RMSN_IN_BF16) p->in_dt = kBF16;
    else if (in == RMSN_IN_F16) p->in_dt = kF16;
    else return RMSN_EINVAL;
    if (out == RMSN_OUT_F32) p->out_dt = kF32;
    else if (out == RMSN_OUT_BF16) p->out_dt = kBF16;
    else if (out == RMSN_OUT_FP8E4M3) p->out_dt = kFP8;
    else p->out_dt = kF16;  // RMSN_OUT_F16
    if ((flags & RMSN_PDL_EARLY_PARAMS) && !(flags & RMSN_PDL)) return RMSN_EINVAL;
    p->pdl = (flags & RMSN_PDL) != 0;
    p->early_params = (flags & RMSN_PDL_EARLY_PARAMS) != 0;
    p->res = (flags & RMSN_HAS_RESIDUAL) != 0;
    p->bias = (flags & RMSN_HAS_BIAS) != 0;
    p->res_f32 = (flags & RMSN_RESIDUAL_F32) != 0;
    if (p->res_f32 && (!p->res || p->in_dt == kF32)) return RMSN_EINVAL;
    p->in_bytes = dtype_bytes(p->in_dt);
    p->res_bytes = p->res_f32 ? 4 : p->in_bytes;
    p->out_bytes = dtype_bytes(p->out_dt);
    p->ve = 32 / p->res_bytes;  // elements per 32-byte vector of the residual stream
    return RMSN_OK;
}

int check_shape(int64_t T, int64_t H, Problem* p) {
    if (T < 0 || H < 1 || H > kMaxHidden) return RMSN_EINVAL;
    if (T > (INT64_MAX / 8) / H) return RMSN_EINVAL;
    p->T = T;
    p->H = H;
    return RMSN_OK;
}

// Can the 32-byte vector kernels run with these pointers?  Each thread moves
// one 32-byte vector of the residual stream per chunk: ve elements, so
// ve * in_bytes bytes of x / weight / bias (32, or 16 under an fp32 stream).
bool vector_path_ok(const Problem& p, const void* x, const void* r, const void* w,
                    const void* b, const void* ro, const void* out) {
    const int xv = p.ve * p.in_bytes;
    if ((p.H * p.res_bytes) % 32 != 0 || (p.H * p.in_bytes) % xv != 0) return false;
    if (!aligned(x, xv) || !aligned(w, xv) || !aligned(b, xv)) return false;
    if (!aligned(r, 32) || !aligned(ro, 32)) return false;
    const int out_vec = p.ve * p.out_bytes;  // bytes stored per vector
    return aligned(out, out_vec < 32 ? out_vec : 32);
}

// The ragged-row kernel: the same 2- or 4-byte dtype in and out, no fp32
// stream, and every row pointer equally aligned modulo 16 bytes (so a row's
// 16-byte vectors sit at the same columns in all of them).
// The ragged-row kernel's dtype pairs: bf16 / fp16 / fp32 in; out in the
// same dtype, as per-token FP8, in fp32 from 16-bit rows or in a 16-bit type
// from fp32 rows.
bool ragged_dtypes_ok(const Problem& p) {
    const bool in16 = p.in_dt == kBF16 || p.in_dt == kF16;
    if (!(in16 || p.in_dt == kF32) || p.res_f32) return false;
    if (p.out_dt == p.in_dt || p.out_dt == kFP8) return true;
    return in16 ? p.out_dt == kF32 : (p.out_dt == kBF16 || p.out_dt == kF16);
}

// x, residual and residual_out equally aligned modulo 16 bytes; out offset
// from a (16 / in size) x (out size)-byte boundary by as many elements as x
// from its 16-byte boundary.
bool ragged_path_ok(const Problem& p, const void* x, const void* r, const void* ro,
                    const void* out) {
    if (!ragged_dtypes_ok(p)) return false;
    const uintptr_t m = reinterpret_cast<uintptr_t>(x) & 15u;
    const void* others[] = {r, ro};
    for (const void* o : others)
        if (o && (reinterpret_cast<uintptr_t>(o) & 15u) != m) return false;
    const uintptr_t si = (uintptr_t)p.in_bytes, so = (uintptr_t)p.out_bytes, ve = 16u / si;
    const uintptr_t ob = reinterpret_cast<uintptr_t>(out);
    return ob % so == 0 && (ob / so) % ve == m / si;
}

const KernelEntry* find_kernel(const Problem& p, int variant, int ch, int wmax) {
    for (const KernelEntry& e : registry()) {
        if (e.in_dt != p.in_dt || e.out_dt != p.out_dt || e.variant != variant) continue;
        if (e.res != (p.res ? 1 : 0) || e.res_f32 != (p.res_f32 ? 1 : 0)) continue;
        if (variant == kGeneric) return &e;
        if (e.bias != (p.bias ? 1 : 0)) continue;
        if (e.chunks == ch && e.max_warps == wmax) return &e;
    }
    return nullptr;
}

int blocks_per_sm(DeviceInfo* d, const void* fn, int threads, int smem) {
    const OccKey key{fn, threads, smem};
    {
        std::lock_guard<std::mutex> lock(d->mu);
        auto it = d->occ_cache.find(key);
        if (it != d->occ_cache.end()) return it->second;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(d->mu);
    d->occ_cache[key] = n;
    return n;
}

// Shared-memory row buffers of the bulk kernel: the requested count, else as
// many as fit in ~220 KB (one block per SM), at most kMaxStages.
constexpr int kMaxStages = 8;
constexpr int kBulkSmemTarget = 220 * 1024;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled();

// Ring stages filled by 128-byte-swizzled 2-D tensor copies: each row (of x
// and of the residual) must be whole 1024-byte units (the swizzle pattern
// repeats every 1024 bytes and every stage starts on such a boundary), at
// most 256 lines of 128 bytes (one tensor box), and the tensor's line index
// must fit the copy's signed 32-bit coordinate.
bool bulk_swizzle_ok(const Problem& p) {
    const int64_t xb = p.H * p.in_bytes, rb = p.H * p.res_bytes;
    if (xb % 1024 != 0 || xb > 256 * 128 || p.T * (xb / 128) >= (int64_t{1} << 31)) return false;
    if (p.res && (rb % 1024 != 0 || rb > 256 * 128 || p.T * (rb / 128) >= (int64_t{1} << 31)))
        return false;
    return true;
}

// One ring stage: the row of x, then (with a residual) the residual's row.
int bulk_stage_bytes(const Problem& p) {
    return (int)(p.H * p.in_bytes + (p.res ? p.H * p.res_bytes : 0));
}

// Fill block shape, grid (persistent: at most one resident wave) for an entry.
bool shape_config(const Problem& p, const KernelEntry& e, DeviceInfo* d, int grid_req,
                  int stages_req, rmsn_config* c) {
    const int sms = d->num_sms;
    memset(c, 0, sizeof(*c));
    c->variant = e.variant;
    c->chunks = e.chunks;
    c->max_warps = e.max_warps;
    c->num_sms = sms;
    int threads;
    int64_t units;  // rows handled per block-step
    if (e.variant == kRagged) {
        // at most ceil(H / (16 / size)) interior vectors: CH per thread x 256
        const int64_t vecs = (p.H * p.in_bytes + 15) / 16;
        if (vecs > (int64_t)e.chunks * 256) return false;
        // fp32 weight (and bias) rows with one pad word per 32 columns
        const int64_t smem = (p.H + p.H / 32) * 4 * (p.bias ? 2 : 1);
        if (smem > 48 * 1024 && smem > enable_smem(d, e.fn)) return false;
        c->vec_bytes = 16;
        c->warps_per_block = 8;
        c->warps_per_row = 8;
        c->smem_bytes = (int32_t)smem;
        threads = 256;
        units = p.T;
    } else if (e.variant == kGeneric) {
        c->vec_bytes = p.in_bytes;
        int w = (int)((p.H + 31) / 32);
        if (w > 8) w = 8;
        c->warps_per_block = w;
        c->warps_per_row = w;
        threads = w * 32;
        units = p.T;
    } else if (e.variant == kCluster) {
        // one row per cluster of K one-warp blocks; the row's vectors fill
        // CH chunks of K * 32 lanes (and would not fit half as many)
        const int K = e.max_warps;
        if (p.nvec > 32 * K * e.chunks) return false;
        if (e.chunks > 1 && p.nvec <= 32 * K * (e.chunks / 2)) return false;
        if (p.T > (int64_t)(INT32_MAX / K)) return false;
        c->vec_bytes = 32;
        c->warps_per_block = 1;
        c->warps_per_row = K;
        c->cluster = K;
        threads = 32;
        units = p.T * K;
        if (blocks_per_sm(d, e.fn, threads, 0) < 1) return false;
        c->grid = (int32_t)units;  // every row its own cluster, not limited to one wave
        return true;
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
        if (e.variant == kBulkRow || e.variant == kBulkPipe) {
            const int sb = bulk_stage_bytes(p);
            int st = stages_req > 0 ? stages_req : kBulkSmemTarget / sb;
            if (st > kMaxStages) st = kMaxStages;
            const int limit = enable_smem(d, e.fn);
            const int pad = bulk_swizzle_ok(p) ? 1024 : 0;
            if (stages_req <= 0)
                while (st > 2 && (int64_t)st * sb + pad > limit) --st;
            if (st < 2 || (int64_t)st * sb + pad > limit) return false;
            c->stages = st;
            // room to round the ring up to a 1024-byte boundary for the swizzle
            c->smem_bytes = st * sb + (bulk_swizzle_ok(p) ? 1024 : 0);
            c->ring_copy = bulk_swizzle_ok(p) && encode_tiled() ? 2 : 1;
        }
    }
    const int bps = blocks_per_sm(d, e.fn, threads, c->smem_bytes);
    if (bps < 1) return false;
    const int64_t resident = (int64_t)sms * bps;
    // the register kernels take one unit per block where a unit moves at
    // least 4 KiB of x: the block scheduler refills SMs as blocks finish,
    // which keeps more rows in flight than resident blocks looping over rows
    // (measured on GB300: 16384 x 16384 bf16 in 304 against 344 us, 16384 x
    // 8192 in 155 against 164 us); smaller units stay on a resident grid
    // (rows of 128 bf16 took twice as long as blocks of their own), and so
    // do the ring kernels (their copies run ahead of the rows)
    const int64_t unit_rows = e.variant == kWarpRows ? e.max_warps : 1;
    const bool one_pass = (e.variant == kBlockRow || e.variant == kWarpRows) &&
                          unit_rows * p.H * p.in_bytes >= 4096;
    const int64_t cap = one_pass ? (int64_t)INT32_MAX : resident;
    int64_t grid = units < cap ? units : cap;
    if (grid_req > 0) grid = grid_req < units ? grid_req : units;
    if (grid < 1) grid = 1;
    c->grid = (int32_t)grid;
    return true;
}

// Table keys of the input side: the DType of x, or one of these two for
// bf16 / fp16 activations over an fp32 residual stream, or the third for bf16
// rows measured as launches chained by programmatic dependent launch
// (RMSN_PDL; tried before the plain bf16 rows for calls with that flag).
constexpr int kTableBF16R32 = 7;
constexpr int kTableF16R32 = 8;
constexpr int kTableBF16PDL = 9;

#include "rmsn_selector_table.inc"

bool select_rules(const Problem& p, DeviceInfo* d, rmsn_config* c);

// Launch of a table row's shape for this problem, if it is built and fits.
bool table_shape(const Problem& p, DeviceInfo* d, int variant, int ch, int wmax, int stages,
                 rmsn_config* c) {
    const KernelEntry* e = find_kernel(p, variant, ch, wmax);
    return e && shape_config(p, *e, d, 0, stages, c);
}

// The selector (see the file comment): the measured table first (rows of this
// hidden size; else of the nearest measured hidden size within a factor of
// two, whose row lengths are of the same kind: a ring row only for rows its
// swizzled copies can take), then the decode rule (one warp per block while
// the whole problem needs no more warps than there are SMs), then the fixed
// prefill rule (fewest warps with CH <= 2).
bool select(const Problem& p, DeviceInfo* d, rmsn_config* c) {
    if (!p.vec_ok) {
        if (p.ragged_ok) {
            for (int ch = 1; ch <= 8; ch *= 2) {
                const KernelEntry* e = find_kernel(p, kRagged, ch, 8);
                if (e && shape_config(p, *e, d, 0, 0, c)) return true;
            }
        }
        const KernelEntry* e = find_kernel(p, kGeneric, 0, 0);
        return e && shape_config(p, *e, d, 0, 0, c);
    }
    int variant = 0, ch = 0, wmax = 0, stages = 0;
    const int res = p.res ? 1 : 0;
    // table keys to try: the rows measured with PDL for a PDL call, the
    // problem's own, then (fp16 moves the same bytes through the same kernels
    // as bf16) the bf16 rows for fp16
    int keys[3][2];
    int nkeys = 0;
    const int tin = p.res_f32 ? (p.in_dt == kF16 ? kTableF16R32 : kTableBF16R32) : p.in_dt;
    if (p.pdl && tin == kBF16) {
        keys[nkeys][0] = kTableBF16PDL;
        keys[nkeys++][1] = p.out_dt;
    }
    keys[nkeys][0] = tin;
    keys[nkeys++][1] = p.out_dt;
    if (tin == kF16 || tin == kTableF16R32) {
        keys[nkeys][0] = tin == kF16 ? kBF16 : kTableBF16R32;
        keys[nkeys++][1] = p.out_dt == kF16 ? kBF16 : p.out_dt;
    }
    for (int k = 0; k < nkeys; ++k) {
        if (table_lookup(keys[k][0], keys[k][1], p.H, p.T, res, &variant, &ch, &wmax, &stages))
            return table_shape(p, d, variant, ch, wmax, stages, c) ||
                   select_rules(p, d, c);
    }
    for (int k = 0; k < nkeys; ++k) {
        // the PDL rows stand for their own hidden sizes only
        if (keys[k][0] == kTableBF16PDL) continue;
        int64_t near[16];
        const int n = table_neighbours(keys[k][0], keys[k][1], p.H, near, 16);
        for (int i = 0; i < n; ++i) {
            if (!table_lookup(keys[k][0], keys[k][1], near[i], p.T, res, &variant, &ch, &wmax,
                              &stages))
                continue;
            if ((variant == kBulkRow || variant == kBulkPipe) && !bulk_swizzle_ok(p)) continue;
            if (table_shape(p, d, variant, ch, wmax, stages, c)) return true;
        }
    }
    return select_rules(p, d, c);
}

// The blog's decode rule, then the fixed prefill rule (shapes the table does
// not cover).
bool select_rules(const Problem& p, DeviceInfo* d, rmsn_config* c) {
    int ch = 0;
    const int64_t warps_needed = (p.T * p.nvec + 31) / 32;
    if (warps_needed <= d->num_sms && p.nvec <= 32 * 8) {
        ch = 1;
        while (32 * ch < p.nvec) ch *= 2;
        const KernelEntry* e = find_kernel(p, kWarpRows, ch, 1);
        if (e && shape_config(p, *e, d, 0, 0, c)) return true;
    }
    const int cands[][2] = {{2, 4}, {2, 8}, {2, 16}, {2, 32}, {4, 16}};
    for (auto& cw : cands) {
        const int w = (int)((p.nvec + 32 * cw[0] - 1) / (32 * cw[0]));
        if (w > cw[1]) continue;
        const KernelEntry* e = find_kernel(p, kBlockRow, cw[0], cw[1]);
        if (e && shape_config(p, *e, d, 0, 0, c)) return true;
        break;
    }
    const KernelEntry* e = find_kernel(p, kGeneric, 0, 0);
    return e && shape_config(p, *e, d, 0, 0, c);
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

namespace rmsn {
namespace {

// Argument checks shared by the entry points.  Fills `p` (including whether
// the 32-byte vector kernels can run with these pointers).  RMSN_OK with
// p->T == 0 means "nothing to do".
int validate(const void* x, const void* residual, const void* weight, const void* bias,
             const void* out, const void* residual_out, const float* out_scale,
             int64_t n_tokens, int64_t hidden, float eps, uint32_t flags, float weight_offset,
             Problem* p, int block_fmt = -1) {
    int st = decode_flags(flags, p);
    if (st != RMSN_OK) return st;
    if (block_fmt >= 0) {  // block-scaled output: byte codes, FP4 packed two per byte
        if (flags & RMSN_OUT_MASK) return RMSN_EINVAL;
        p->out_dt = block_fmt;
        p->out_bytes = 1;
    }
    if ((st = check_shape(n_tokens, hidden, p)) != RMSN_OK) return st;
    if (!(eps >= 0.f) || !isfinite(eps) || !isfinite(weight_offset)) return RMSN_EINVAL;
    // an empty batch touches nothing (its buffers may be NULL)
    if (n_tokens == 0) return RMSN_OK;
    // optional operands must match their flags exactly
    if (p->res != (residual != nullptr) || p->res != (residual_out != nullptr)) return RMSN_EINVAL;
    if (((flags & RMSN_HAS_WEIGHT) != 0) != (weight != nullptr)) return RMSN_EINVAL;
    if (p->bias != (bias != nullptr)) return RMSN_EINVAL;
    if ((p->out_dt == kFP8 || p->out_dt == kNVFP4) != (out_scale != nullptr)) return RMSN_EINVAL;
    if (!x || !out) return RMSN_EINVAL;
    const void* ins[] = {x, weight, bias};
    for (const void* q : ins)
        if (!aligned(q, (uintptr_t)p->in_bytes)) return RMSN_EALIGN;
    if (!aligned(residual, (uintptr_t)p->res_bytes) || !aligned(residual_out, (uintptr_t)p->res_bytes))
        return RMSN_EALIGN;
    if (!aligned(out, (uintptr_t)p->out_bytes) || !aligned(out_scale, 4)) return RMSN_EALIGN;
    p->vec_ok = vector_path_ok(*p, x, residual, weight, bias, residual_out, out);
    p->nvec = p->vec_ok ? (int)(p->H / p->ve) : 0;
    p->ragged_ok = !p->vec_ok && ragged_path_ok(*p, x, residual, residual_out, out);
    return RMSN_OK;
}

// cuTensorMapEncodeTiled from the driver, looked up once per process (no
// link-time dependency on the driver library); null where unavailable.
EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            f = nullptr;
        }
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// A [T, H] tensor of `bytes`-byte elements as 128-byte lines: a 2-D map of
// (128 / bytes) x (T H bytes / 128) elements whose box is one row's lines,
// copied with the 128-byte swizzle.
bool encode_rows(CUtensorMap* m, const void* base, int64_t T, int64_t H, int bytes) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)(128 / bytes), (cuuint64_t)(T * H * bytes / 128)};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / bytes), (cuuint32_t)(H * bytes / 128)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT32, 2,
              const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// encode_rows through the device's map cache.
bool cached_rows(DeviceInfo* d, CUtensorMap* m, const void* base, int64_t T, int64_t H,
                 int bytes) {
    {
        std::lock_guard<std::mutex> lock(d->mu);
        for (const MapEntry& e : d->maps) {
            if (e.base == base && e.T == T && e.H == H && e.bytes == bytes) {
                memcpy(m, &e.map, sizeof(*m));
                return true;
            }
        }
    }
    if (!encode_rows(m, base, T, H, bytes)) return false;
    std::lock_guard<std::mutex> lock(d->mu);
    MapEntry& e = d->maps[d->map_next];
    d->map_next = (d->map_next + 1) % kMapCache;
    e.base = base;
    e.T = T;
    e.H = H;
    e.bytes = bytes;
    memcpy(&e.map, m, sizeof(*m));
    return true;
}

int launch(const KernelEntry* e, const rmsn_config& c, DeviceInfo* d, const Problem& p,
           const void* x, const void* residual, const void* weight, const void* bias, void* out,
           void* residual_out, float* out_scale, float eps, float weight_offset,
           cudaStream_t stream, void* block_scale = nullptr) {
    RmsnArgs a;
    a.bscale = block_scale;
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
    a.stages = c.stages;
    a.pdl = p.pdl ? 1 : 0;
    a.early_params = p.early_params ? 1 : 0;
    a.status = d->status;
    a.wait_cycles = d->wait_cycles.load(std::memory_order_relaxed);
    // the bulk kernel also takes the tensor-copy descriptors of x and the
    // residual (zero and unused when its stages take 1-D copies)
    alignas(64) CUtensorMap mx;
    alignas(64) CUtensorMap mr;
    memset(&mx, 0, sizeof(mx));
    memset(&mr, 0, sizeof(mr));
    a.swz = 0;
    const bool ring = e->variant == kBulkRow || e->variant == kBulkPipe;
    if (ring && bulk_swizzle_ok(p) &&
        cached_rows(d, &mx, x, p.T, p.H, p.in_bytes) &&
        (!p.res || cached_rows(d, &mr, residual, p.T, p.H, p.res_bytes)))
        a.swz = 1;
    void* args_one[] = {&a};
    void* args_bulk[] = {&a, &mx, &mr};
    void** args = ring ? args_bulk : args_one;
    cudaError_t err;
    if (p.pdl || e->variant == kCluster) {
        // programmatic dependent launch: the kernel may start while the
        // preceding kernel in `stream` runs; it waits for it before reading.
        // The split-row kernel runs as clusters of c.cluster blocks.
        cudaLaunchAttribute attr[2];
        unsigned n = 0;
        if (p.pdl) {
            attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[n++].val.programmaticStreamSerializationAllowed = 1;
        }
        if (e->variant == kCluster) {
            attr[n].id = cudaLaunchAttributeClusterDimension;
            attr[n].val.clusterDim.x = (unsigned)c.cluster;
            attr[n].val.clusterDim.y = 1;
            attr[n++].val.clusterDim.z = 1;
        }
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3((unsigned)c.grid);
        lc.blockDim = dim3((unsigned)(c.warps_per_block * 32));
        lc.dynamicSmemBytes = (size_t)c.smem_bytes;
        lc.stream = stream;
        lc.attrs = attr;
        lc.numAttrs = n;
        err = cudaLaunchKernelExC(&lc, e->fn, args);
    } else {
        err = cudaLaunchKernel(e->fn, dim3((unsigned)c.grid),
                               dim3((unsigned)(c.warps_per_block * 32)), args,
                               (size_t)c.smem_bytes, stream);
    }
    return err == cudaSuccess ? RMSN_OK : RMSN_ECUDA;
}

// Device address at which the current device reaches `p`: device memory of
// this device and managed memory as is, page-locked host memory through its
// mapped address, other host memory only where the device can access
// pageable memory.  Device memory of another GPU is refused (without peer
// access a kernel reading it would fault, and whether peer access is on is
// not something the call can see without changing it).  Returns false when
// the device cannot reach `p`.
bool device_view(DeviceInfo* d, int dev_id, const void* p, const void** dev) {
    *dev = p;
    if (!p) return true;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        attr.type = cudaMemoryTypeUnregistered;
    }
    switch (attr.type) {
        case cudaMemoryTypeDevice:
            return attr.device == dev_id;
        case cudaMemoryTypeManaged:
            return true;
        case cudaMemoryTypeHost:
            if (!attr.devicePointer) return false;
            *dev = attr.devicePointer;
            return true;
        default:
            return d->pageable_access != 0;
    }
}

// Launch shape for rows that live in host memory: the register kernels only
// (plain loads and stores), one block per row with one 32-byte vector per
// thread where the row allows it, as many blocks as fit on the GPU, so the
// most requests are in flight across the CPU-GPU link.
bool select_host(const Problem& p, DeviceInfo* d, rmsn_config* c) {
    if (p.vec_ok) {
        const int shapes[][2] = {{1, 4}, {1, 8}, {1, 16}, {1, 32}, {2, 32}, {4, 16}};
        for (auto& s : shapes) {
            const int w = (int)((p.nvec + 32 * s[0] - 1) / (32 * s[0]));
            if (w > s[1]) continue;
            const KernelEntry* e = find_kernel(p, kBlockRow, s[0], s[1]);
            if (e && shape_config(p, *e, d, 0, 0, c)) return true;
        }
    } else if (p.ragged_ok) {
        for (int ch = 1; ch <= 8; ch *= 2) {
            const KernelEntry* e = find_kernel(p, kRagged, ch, 8);
            if (e && shape_config(p, *e, d, 0, 0, c)) return true;
        }
    }
    const KernelEntry* e = find_kernel(p, kGeneric, 0, 0);
    return e && shape_config(p, *e, d, 0, 0, c);
}

}  // namespace
}  // namespace rmsn

RMSN_API int rmsnorm_fwd_ex(const void* x, const void* residual, const void* weight,
                            const void* bias, void* out, void* residual_out, float* out_scale,
                            int64_t n_tokens, int64_t hidden, float eps, uint32_t flags,
                            float weight_offset, const rmsn_config* cfg, cudaStream_t stream) {
    Problem p{};
    int st = validate(x, residual, weight, bias, out, residual_out, out_scale, n_tokens, hidden,
                      eps, flags, weight_offset, &p);
    if (st != RMSN_OK || n_tokens == 0) return st;

    DeviceInfo* d = device_info();
    if (!d) return RMSN_ECUDA;
    rmsn_config c;
    const KernelEntry* e = nullptr;
    if (cfg) {
        if (cfg->variant == kRagged ? !p.ragged_ok : (cfg->variant != kGeneric && !p.vec_ok))
            return RMSN_EUNSUPPORTED;
        e = find_kernel(p, cfg->variant, cfg->chunks, cfg->max_warps);
        if (!e || !shape_config(p, *e, d, cfg->grid, cfg->stages, &c)) return RMSN_EUNSUPPORTED;
    } else {
        const SelKey key{p.T, p.H, flags, (p.vec_ok ? 1 : 0) | (p.ragged_ok ? 2 : 0), 0};
        bool hit = false;
        {
            std::lock_guard<std::mutex> lock(d->mu);
            auto it = d->sel_cache.find(key);
            if (it != d->sel_cache.end()) {
                c = it->second.first;
                e = it->second.second;
                hit = true;
            }
        }
        if (!hit) {
            if (!select(p, d, &c)) return RMSN_EUNSUPPORTED;
            e = find_kernel(p, c.variant, c.chunks, c.max_warps);
            if (!e) return RMSN_EUNSUPPORTED;
            std::lock_guard<std::mutex> lock(d->mu);
            if (d->sel_cache.size() > 4096) d->sel_cache.clear();
            d->sel_cache[key] = {c, e};
        }
    }
    return launch(e, c, d, p, x, residual, weight, bias, out, residual_out, out_scale, eps,
                  weight_offset, stream);
}

RMSN_API int rmsnorm_fwd_blockscaled(const void* x, const void* residual, const void* weight,
                                     const void* bias, void* out, void* block_scale,
                                     float* token_scale, void* residual_out, int64_t n_tokens,
                                     int64_t hidden, float eps, uint32_t flags, int format,
                                     float weight_offset, const rmsn_config* cfg,
                                     cudaStream_t stream) {
    int fmt, block;
    switch (format) {
        case RMSN_FMT_MXFP8: fmt = kMXFP8; block = 32; break;
        case RMSN_FMT_MXFP4: fmt = kMXFP4; block = 32; break;
        case RMSN_FMT_NVFP4: fmt = kNVFP4; block = 16; break;
        default: return RMSN_EINVAL;
    }
    Problem p{};
    int st = validate(x, residual, weight, bias, out, residual_out, token_scale, n_tokens, hidden,
                      eps, flags, weight_offset, &p, fmt);
    if (st != RMSN_OK || n_tokens == 0) return st;
    if (p.H % block != 0 || !block_scale) return RMSN_EINVAL;
    if (p.in_dt != kBF16 || !p.vec_ok) return RMSN_EUNSUPPORTED;
    DeviceInfo* d = device_info();
    if (!d) return RMSN_ECUDA;
    rmsn_config c;
    const KernelEntry* e = nullptr;
    if (cfg) {
        if (cfg->variant == kGeneric || cfg->variant == kRagged) return RMSN_EUNSUPPORTED;
        e = find_kernel(p, cfg->variant, cfg->chunks, cfg->max_warps);
        if (!e || !shape_config(p, *e, d, cfg->grid, cfg->stages, &c)) return RMSN_EUNSUPPORTED;
    } else {
        const SelKey key{p.T, p.H, flags, 1, format};
        bool hit = false;
        {
            std::lock_guard<std::mutex> lock(d->mu);
            auto it = d->sel_cache.find(key);
            if (it != d->sel_cache.end()) {
                c = it->second.first;
                e = it->second.second;
                hit = true;
            }
        }
        if (!hit) {
            if (!select(p, d, &c)) return RMSN_EUNSUPPORTED;
            e = find_kernel(p, c.variant, c.chunks, c.max_warps);
            if (!e) return RMSN_EUNSUPPORTED;
            std::lock_guard<std::mutex> lock(d->mu);
            if (d->sel_cache.size() > 4096) d->sel_cache.clear();
            d->sel_cache[key] = {c, e};
        }
    }
    return launch(e, c, d, p, x, residual, weight, bias, out, residual_out, token_scale, eps,
                  weight_offset, stream, block_scale);
}

RMSN_API int rmsnorm_fwd_host(const void* x, const void* residual, const void* weight,
                              const void* bias, void* out, void* residual_out, float* out_scale,
                              int64_t n_tokens, int64_t hidden, float eps, uint32_t flags,
                              float weight_offset, cudaStream_t stream) {
    Problem p{};
    int st = validate(x, residual, weight, bias, out, residual_out, out_scale, n_tokens, hidden,
                      eps, flags, weight_offset, &p);
    if (st != RMSN_OK || n_tokens == 0) return st;
    DeviceInfo* d = device_info();
    if (!d) return RMSN_ECUDA;
    int dev_id = 0;
    if (cudaGetDevice(&dev_id) != cudaSuccess) return RMSN_ECUDA;
    const void* dx;
    const void* dr;
    const void* dw;
    const void* db;
    const void* dout;
    const void* dres;
    const void* dscale;
    if (!device_view(d, dev_id, x, &dx) || !device_view(d, dev_id, residual, &dr) ||
        !device_view(d, dev_id, weight, &dw) || !device_view(d, dev_id, bias, &db) ||
        !device_view(d, dev_id, out, &dout) || !device_view(d, dev_id, residual_out, &dres) ||
        !device_view(d, dev_id, out_scale, &dscale))
        return RMSN_EINVAL;
    // the mapped addresses decide the vector path
    p.vec_ok = vector_path_ok(p, dx, dr, dw, db, dres, dout);
    p.nvec = p.vec_ok ? (int)(p.H / p.ve) : 0;
    p.ragged_ok = !p.vec_ok && ragged_path_ok(p, dx, dr, dres, dout);
    rmsn_config c;
    if (!select_host(p, d, &c)) return RMSN_EUNSUPPORTED;
    const KernelEntry* e = find_kernel(p, c.variant, c.chunks, c.max_warps);
    if (!e) return RMSN_EUNSUPPORTED;
    return launch(e, c, d, p, dx, dr, dw, db, const_cast<void*>(dout),
                  const_cast<void*>(dres), static_cast<float*>(const_cast<void*>(dscale)), eps,
                  weight_offset, stream);
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
    p->vec_ok = (p->H * p->res_bytes) % 32 == 0;
    p->nvec = p->vec_ok ? (int)(p->H / p->ve) : 0;
    p->ragged_ok = !p->vec_ok && ragged_dtypes_ok(*p);  // equally aligned buffers assumed
    return RMSN_OK;
}

RMSN_API int rmsnorm_query_config(int64_t n_tokens, int64_t hidden, uint32_t flags,
                                  rmsn_config* out) {
    if (!out) return RMSN_EINVAL;
    Problem p{};
    int st = query_problem(n_tokens, hidden, flags, &p);
    if (st != RMSN_OK) return st;
    DeviceInfo* d = device_info();
    if (!d) return RMSN_ECUDA;
    return select(p, d, out) ? RMSN_OK : RMSN_EUNSUPPORTED;
}

RMSN_API int rmsnorm_list_configs(int64_t n_tokens, int64_t hidden, uint32_t flags,
                                  rmsn_config* out, int capacity) {
    if (capacity < 0 || (capacity > 0 && !out)) return RMSN_EINVAL;
    Problem p{};
    int st = query_problem(n_tokens, hidden, flags, &p);
    if (st != RMSN_OK) return st;
    DeviceInfo* d = device_info();
    if (!d) return RMSN_ECUDA;
    int count = 0;
    for (const KernelEntry& e : registry()) {
        if (e.in_dt != p.in_dt || e.out_dt != p.out_dt || e.res != (p.res ? 1 : 0)) continue;
        if (e.res_f32 != (p.res_f32 ? 1 : 0)) continue;
        if (e.variant == kRagged) {
            if (e.bias != (p.bias ? 1 : 0) || !p.ragged_ok) continue;
        } else if (e.variant != kGeneric && (e.bias != (p.bias ? 1 : 0) || !p.vec_ok)) {
            continue;
        }
        // the bulk kernel is listed once per ring depth
        const int stage_opts[] = {0, 2, 3, 4, 6, 8};
        const bool ring = e.variant == kBulkRow || e.variant == kBulkPipe;
        const int n_opts = ring ? 6 : 1;
        for (int i = 0; i < n_opts; ++i) {
            if (ring && i == 0) continue;
            rmsn_config c;
            if (!shape_config(p, e, d, 0, stage_opts[i], &c)) continue;
            if (count < capacity) out[count] = c;
            ++count;
        }
    }
    return count;
}

RMSN_API int rmsnorm_read_status(uint32_t* status, int clear) {
    if (!status) return RMSN_EINVAL;
    DeviceInfo* d = device_info();
    if (!d) return RMSN_ECUDA;
    if (cudaMemcpy(status, d->status, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return RMSN_ECUDA;
    if (clear && *status) {
        if (cudaMemset(d->status, 0, sizeof(uint32_t)) != cudaSuccess) return RMSN_ECUDA;
    }
    return RMSN_OK;
}

RMSN_API int rmsnorm_set_wait_limit(int64_t cycles) {
    DeviceInfo* d = device_info();
    if (!d) return RMSN_ECUDA;
    d->wait_cycles.store(cycles == 0 ? kDefaultWaitCycles : cycles, std::memory_order_relaxed);
    return RMSN_OK;
}

RMSN_API int rmsnorm_qk_fwd(void* q, void* k, const void* q_weight, const void* k_weight,
                            int64_t n_tokens, int64_t n_q_heads, int64_t n_k_heads,
                            int64_t head_dim, int64_t q_token_stride, int64_t k_token_stride,
                            float eps, float weight_offset, uint32_t flags, cudaStream_t stream) {
    if (flags & ~(RMSN_IN_MASK | RMSN_PDL | RMSN_QK_RING | RMSN_QK_DIRECT)) return RMSN_EINVAL;
    if ((flags & RMSN_QK_RING) && (flags & RMSN_QK_DIRECT)) return RMSN_EINVAL;
    const uint32_t in = flags & RMSN_IN_MASK;
    if (in != RMSN_IN_F32 && in != RMSN_IN_BF16 && in != RMSN_IN_F16) return RMSN_EINVAL;
    const int dt = in == RMSN_IN_F32 ? kF32 : (in == RMSN_IN_BF16 ? kBF16 : kF16);
    const int64_t bytes = dt == kF32 ? 4 : 2;
    if (n_tokens < 0 || n_q_heads < 0 || n_k_heads < 0 || head_dim < 1 || head_dim > 4096)
        return RMSN_EINVAL;
    if (n_q_heads > (1 << 20) || n_k_heads > (1 << 20)) return RMSN_EINVAL;
    if (!(eps >= 0.f) || !isfinite(eps) || !isfinite(weight_offset)) return RMSN_EINVAL;
    if (n_q_heads && q_token_stride < n_q_heads * head_dim) return RMSN_EINVAL;
    if (n_k_heads && k_token_stride < n_k_heads * head_dim) return RMSN_EINVAL;
    const int64_t stride_max = q_token_stride > k_token_stride ? q_token_stride : k_token_stride;
    if (stride_max > 0 && n_tokens > (INT64_MAX / 8) / stride_max) return RMSN_EINVAL;
    if (n_tokens == 0 || n_q_heads + n_k_heads == 0) return RMSN_OK;
    if ((n_q_heads && !q) || (n_k_heads && !k)) return RMSN_EINVAL;
    const void* ptrs[] = {q, k, q_weight, k_weight};
    for (const void* p : ptrs)
        if (!aligned(p, (uintptr_t)bytes)) return RMSN_EALIGN;
    // every head must start on a 32-byte boundary and be whole 32-byte vectors
    if ((head_dim * bytes) % 32 != 0 || head_dim * bytes > 32 * 32) return RMSN_EUNSUPPORTED;
    for (const void* p : ptrs)
        if (!aligned(p, 32)) return RMSN_EUNSUPPORTED;
    if ((n_q_heads && (q_token_stride * bytes) % 32) || (n_k_heads && (k_token_stride * bytes) % 32))
        return RMSN_EUNSUPPORTED;

    DeviceInfo* d = device_info();
    if (!d) return RMSN_ECUDA;
    const int nvec = (int)(head_dim * bytes / 32);
    int tph = 1;
    while (tph < nvec) tph *= 2;
    const QkEntry* table = nullptr;
    int n = 0;
    table = qk_kernels(&n);
    // the ring variant: a token's heads are whole warps' worth of vectors
    // (vectors per head a power of two from 4 up), at most 2048 vectors per
    // token (two per thread), at least two token buffers in shared memory
    const int64_t tok_vecs = (n_q_heads + n_k_heads) * nvec;
    const int64_t tok_bytes = tok_vecs * 32;
    // a ring buffer holds two tokens with one vector per thread, else one
    const int64_t buf_bytes = (tok_vecs > 1024 ? 1 : 2) * tok_bytes;
    const bool ring_ok = tph == nvec && nvec >= 4 && tok_vecs <= 2048 &&
                         2 * buf_bytes <= d->max_smem - 1024;
    bool ring = ring_ok && n_tokens >= kQkRingTokens;
    if (flags & RMSN_QK_RING) {
        if (!ring_ok) return RMSN_EUNSUPPORTED;
        ring = true;
    }
    if (flags & RMSN_QK_DIRECT) ring = false;
    const int kind = ring ? kQkBlockRing : kQkDirect;
    // block ring: vectors per thread; one-pass kernel: tokens per block
    // (two tokens per block once there are at least two blocks per SM: more
    // bytes in flight per lane; measured on GB300 from 512 tokens on)
    const int ch = ring ? (tok_vecs > 1024 ? 2 : 1) : (n_tokens >= 2 * (int64_t)d->num_sms ? 2 : 1);
    const QkEntry* e = nullptr;
    for (int i = 0; i < n; ++i)
        if (table[i].dt == dt && table[i].tph == tph && table[i].kind == kind && table[i].ch == ch)
            e = &table[i];
    if (!e) return RMSN_EUNSUPPORTED;
    int threads = 256, stages = 0;
    size_t smem = 0;
    int64_t grid = 0;
    unsigned grid_y = 1;
    if (ring) {
        threads = (int)(((tok_vecs + ch - 1) / ch + 31) / 32 * 32);
        // about 96 KiB of token buffers per block (two blocks per SM), 2..8 of them
        stages = (int)(kQkRingBytes / buf_bytes);
        stages = stages < 2 ? 2 : (stages > kMaxStages ? kMaxStages : stages);
        smem = (size_t)stages * (size_t)buf_bytes;
        // the opt-in limit, always: the kernel's static shared memory counts too
        if ((int64_t)smem > enable_smem(d, e->fn)) return RMSN_EUNSUPPORTED;
        const int bps = blocks_per_sm(d, e->fn, threads, (int)smem);
        if (bps < 1) return RMSN_EUNSUPPORTED;
        const int64_t resident = (int64_t)d->num_sms * bps;
        grid = n_tokens < resident ? n_tokens : resident;
    } else {
        // one block per token and group of heads: W warps of 32 / tph heads,
        // W <= 16 chosen so the groups split evenly over the blocks
        const int64_t nh = 32 / tph;
        const int64_t warps = (n_q_heads + n_k_heads + nh - 1) / nh;
        const int64_t gy = (warps + 15) / 16;
        if (gy > 65535) return RMSN_EUNSUPPORTED;  // the grid's y extent
        threads = (int)((warps + gy - 1) / gy) * 32;
        const int64_t blocks = (n_tokens + ch - 1) / ch;
        grid = blocks < kQkMaxGridX ? blocks : kQkMaxGridX;
        grid_y = (unsigned)gy;
    }

    QkArgs a;
    a.q = q;
    a.k = k;
    a.qw = q_weight;
    a.kw = k_weight;
    a.T = n_tokens;
    a.qs = q_token_stride;
    a.ks = k_token_stride;
    a.Hq = (int32_t)n_q_heads;
    a.Hk = (int32_t)n_k_heads;
    a.D = (int32_t)head_dim;
    a.nvec = nvec;
    a.eps = eps;
    a.woff = weight_offset;
    a.pdl = (flags & RMSN_PDL) ? 1 : 0;
    a.status = d->status;
    a.rcp_d = (head_dim & (head_dim - 1)) == 0 ? 1.0f / (float)head_dim : 0.f;  // exact
    a.stages = stages;
    a.wait_cycles = d->wait_cycles.load(std::memory_order_relaxed);
    void* args[] = {&a};
    cudaError_t err;
    if (flags & RMSN_PDL) {
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3((unsigned)grid, grid_y);
        lc.blockDim = dim3(threads);
        lc.dynamicSmemBytes = smem;
        lc.stream = stream;
        lc.attrs = attr;
        lc.numAttrs = 1;
        err = cudaLaunchKernelExC(&lc, e->fn, args);
    } else {
        err = cudaLaunchKernel(e->fn, dim3((unsigned)grid, grid_y), dim3(threads), args, smem,
                               stream);
    }
    return err == cudaSuccess ? RMSN_OK : RMSN_ECUDA;
}
