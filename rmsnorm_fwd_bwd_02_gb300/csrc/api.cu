// api.cu -- the C ABI declared in include/rmsnorm.h: host-side argument
// checks, kernel choice, grid sizing and launches. No allocation, no
// synchronisation, no host copies; everything is enqueued on the caller's
// stream.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>
#include <initializer_list>
#include <utility>

#include "rmsnorm.h"
#include "context.h"
#include "params.h"
#include "bwd2.cuh"
#include "gemv.cuh"
#include "gemv_tma.cuh"
#include "gemv_tc.cuh"
#include "gemv_umma.cuh"
#include "reduce.cuh"
#include "registry.h"

using namespace rmsk;

namespace {

constexpr int kPathAuto = 0, kPathRows = 1, kPathSplit = 2, kPathScalar = 3, kPathStream = 4;
constexpr int kPathGemv = 5;           // RMSNorm fused with the GEMV: A in registers (5,
constexpr int kPathGemvTma = 6;        // reported only), by bulk copies (6), or the
constexpr int kPathGemvUmma = 7;       // product on tcgen05 (7); 6 and 7 also force it
constexpr int kPathGemvTc = 8;         // persistent tcgen05, y held per CTA (8; forces it)
constexpr int kGemvMaxRows = 64;
constexpr int64_t kGemvMaxSmem = 227 * 1024;
constexpr int kSplitMaxRows = 64;      // decode-sized batches ([P2 §3.2])
constexpr int kReduceCols = 32, kReduceRows = 16;

thread_local int t_last_cuda_error = 0;
thread_local int t_last_path = 0;
std::atomic<int> g_path_override{kPathAuto};
// Test hook for the streamed kernels' bounded waits (see rmsnorm.h).
std::atomic<unsigned> g_test_extra_tx{0}, g_test_wait_us{0};
std::atomic<int> g_test_tc_cluster{0};   // forced cluster size of the persistent projection

int cuda_fail(cudaError_t e)
{
    t_last_cuda_error = (int)e;
    return RMSNORM_ERR_CUDA;
}

size_t elem_size(int dtype) { return dtype == RMSNORM_F32 ? 4 : 2; }

bool aligned(const void *p, size_t a) { return p == nullptr || (uintptr_t)p % a == 0; }

// A tensor argument as the bytes it touches: `rows` rows of `row_bytes`
// bytes whose starts are `ld_bytes` apart (a flat buffer is one row).
struct Span {
    const void *p;
    int64_t rows, row_bytes, ld_bytes;
    bool empty() const { return p == nullptr || rows <= 0 || row_bytes <= 0; }
    uintptr_t begin() const { return (uintptr_t)p; }
    uintptr_t end() const { return (uintptr_t)p + (rows - 1) * ld_bytes + row_bytes; }
};

Span flat(const void *p, size_t n) { return {p, 1, (int64_t)n, (int64_t)n}; }

Span rows_span(const void *p, int64_t M, int64_t H, int64_t ld, size_t es)
{
    return {p, M, H * (int64_t)es, ld * (int64_t)es};
}

// Whether two arguments may share a byte. Exact for disjoint address
// ranges and for row windows of one stride that never meet (the rows of b
// fall, modulo the stride, after the end of a's rows and before the next
// row of a starts); any other pair whose ranges intersect counts as
// overlapping.
bool overlap(Span a, Span b)
{
    if (a.empty() || b.empty())
        return false;
    if (!(a.begin() < b.end() && b.begin() < a.end()))
        return false;
    if (a.ld_bytes == b.ld_bytes && a.ld_bytes > 0) {
        const int64_t ld = a.ld_bytes;
        const int64_t d = (int64_t)(b.begin() - a.begin());
        const int64_t s = ((d % ld) + ld) % ld;   // b's row offset within a's row frame
        if (s >= a.row_bytes && s + b.row_bytes <= ld)
            return false;
    }
    return true;
}

bool same(Span a, Span b)
{
    return a.p == b.p && a.rows == b.rows && a.row_bytes == b.row_bytes &&
           (a.rows == 1 || a.ld_bytes == b.ld_bytes);
}

// Allowed: the same tensor exactly (same start, shape and stride), or no
// shared byte at all.
bool same_or_disjoint(Span a, Span b) { return same(a, b) || !overlap(a, b); }

int check_common(int64_t M, int64_t H, float eps, int dtype)
{
    if (dtype != RMSNORM_F32 && dtype != RMSNORM_BF16 && dtype != RMSNORM_F16)
        return RMSNORM_ERR_BAD_DTYPE;
    if (M < 0 || H < 1)
        return RMSNORM_ERR_BAD_SHAPE;
    if (H > RMSNORM_MAX_H)
        return RMSNORM_ERR_UNSUPPORTED;
    if (M > INT64_MAX / 8 / H)
        return RMSNORM_ERR_BAD_SHAPE;
    if (!(eps >= 0.f) || !std::isfinite(eps))
        return RMSNORM_ERR_BAD_EPS;
    return RMSNORM_OK;
}

// A row stride is at least H and below 2^31 (the row kernels hold strides in
// 32 bits), and the tensor's last byte stays far below 2^63 (so every byte
// offset the kernels form fits an int64).
bool stride_ok(int64_t ld, int64_t M, int64_t H)
{
    if (ld < H || ld > INT32_MAX)
        return false;
    return M <= 1 || ld <= (INT64_MAX / 8 - H) / (M - 1);
}

// Row strides (elements) whose byte size is a multiple of `a`.
bool strides_multiple(size_t a, size_t es, std::initializer_list<int64_t> lds)
{
    for (int64_t ld : lds)
        if ((ld * (int64_t)es) % (int64_t)a != 0)
            return false;
    return true;
}

// ------------------------------------------------------- device properties
int current_device(int *dev)
{
    cudaError_t e = cudaGetDevice(dev);
    return e == cudaSuccess ? RMSNORM_OK : cuda_fail(e);
}

int sm_count(int dev, int *sms)
{
    cudaError_t e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
    return e == cudaSuccess ? RMSNORM_OK : cuda_fail(e);
}

// Resident CTAs per SM for a kernel launched with `smem` bytes of dynamic
// shared memory, cached per (kernel, device, smem). A kernel that needs more
// than the default 48 KB is opted in to the device's maximum (not to this
// size: a later call with more shared memory must still launch).
// Entries hold for the context they were made in (context.h).
int blocks_per_sm(const void *fn, int threads, int dev, int *out, int smem = 0)
{
    static std::mutex mu;
    static std::map<std::tuple<const void *, int, int, unsigned long long>, int> cache;
    const unsigned long long ctx = current_context_id();
    if (ctx != 0) {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(std::make_tuple(fn, dev, smem, ctx));
        if (it != cache.end()) {
            *out = it->second;
            return RMSNORM_OK;
        }
    }
    int n = 0;
    cudaError_t e = cudaSuccess;
    if (smem > 48 * 1024) {
        // the device's per-CTA maximum less the kernel's static shared memory
        int most = 0;
        cudaFuncAttributes fa;
        e = cudaDeviceGetAttribute(&most, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e == cudaSuccess)
            e = cudaFuncGetAttributes(&fa, fn);
        if (e == cudaSuccess) {
            most -= (int)fa.sharedSizeBytes;
            if (smem > most)
                return cuda_fail(cudaErrorInvalidValue);
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
        }
    }
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem);
    if (e != cudaSuccess)
        return cuda_fail(e);
    if (n < 1)
        return cuda_fail(cudaErrorInvalidConfiguration);
    // the context the attribute was set in (the calls above create the
    // primary context if none was current)
    const unsigned long long made_in = current_context_id();
    if (made_in != 0) {
        std::lock_guard<std::mutex> g(mu);
        cache[std::make_tuple(fn, dev, smem, made_in)] = n;
    }
    *out = n;
    return RMSNORM_OK;
}

// Clusters of `cs` CTAs of `fn` that can be resident at once on device
// `dev` (a cluster must fit within one GPC, so fewer CTAs than SMs x
// blocks_per_sm may run together).
int max_active_clusters(const void *fn, int threads, int smem, int cs, int dev, int *out)
{
    static std::mutex mu;
    static std::map<std::tuple<const void *, int, int, int, unsigned long long>, int> cache;
    const unsigned long long ctx = current_context_id();
    if (ctx != 0) {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(std::make_tuple(fn, dev, smem, cs, ctx));
        if (it != cache.end()) {
            *out = it->second;
            return RMSNORM_OK;
        }
    }
    int bps;
    int st = blocks_per_sm(fn, threads, dev, &bps, smem);     // sets the smem limit
    if (st)
        return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeClusterDimension;
    a.val.clusterDim.x = (unsigned)cs;
    a.val.clusterDim.y = 1;
    a.val.clusterDim.z = 1;
    cfg.attrs = &a;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
    if (e != cudaSuccess)
        return cuda_fail(e);
    if (n < 1)
        return cuda_fail(cudaErrorInvalidConfiguration);
    const unsigned long long made_in = current_context_id();
    if (made_in != 0) {
        std::lock_guard<std::mutex> g(mu);
        cache[std::make_tuple(fn, dev, smem, cs, made_in)] = n;
    }
    *out = n;
    return RMSNORM_OK;
}

// Persistent grid: no more CTAs than tiles, no more than fit at once.
int rows_grid(const RowShape &k, const void *fn, int64_t M, int64_t *grid)
{
    int dev, sms, bps, st;
    if ((st = current_device(&dev)) || (st = sm_count(dev, &sms)) ||
        (st = blocks_per_sm(fn, k.threads(), dev, &bps)))
        return st;
    const int64_t tiles = (M + k.tile_rows() - 1) / k.tile_rows();
    const int64_t cap = (int64_t)bps * sms;
    *grid = tiles < cap ? tiles : cap;
    return RMSNORM_OK;
}

// Streamed kernels: one group of NG rows in flight per CTA iteration.
int stream_grid(const StreamShape &k, const void *fn, int smem, int64_t M, int64_t *grid,
                int *dev_out)
{
    int dev, sms, bps, st;
    if ((st = current_device(&dev)) || (st = sm_count(dev, &sms)) ||
        (st = blocks_per_sm(fn, k.threads(), dev, &bps, smem)))
        return st;
    const int64_t tiles = (M + k.rows - 1) / k.rows;
    const int64_t cap = (int64_t)bps * sms;
    *grid = tiles < cap ? tiles : cap;
    *dev_out = dev;
    return RMSNORM_OK;
}

// Shapes with a streamed layout, and whether the automatic choice takes it
// (set from measurements on GB300: the faster kernel family per direction).
// At M = 32768 x 4096 the backward takes 116.6 us streamed against 132.9 us
// row-wise, the forward 85.5 us against 82.2 us; at 16384 x 5120 with the
// residual the backward takes 95.9 us against 128.3 us, the forward 106.6 us
// against 101.5 us; at 524288 x 128 the backward 62.6 us against 67.6 us,
// the forward 47.4 us against 43.0 us.
struct StreamPolicy {
    const StreamKernels *k;
    bool auto_fwd, auto_bwd;
};

// dense: every row stride equals H (the 128-wide kernels copy blocks of
// consecutive rows). fp16 takes the bf16 choices (same bytes, same layouts).
const StreamPolicy *pick_stream(int dtype, int64_t H, bool vec, bool dense)
{
    static const StreamPolicy b4096 = {&s_h4096, false, true};
    static const StreamPolicy b5120 = {&s_h5120, false, true};
    static const StreamPolicy b128 = {&s_h128, false, true};
    static const StreamPolicy h4096 = {&sh_h4096, false, true};
    static const StreamPolicy h5120 = {&sh_h5120, false, true};
    static const StreamPolicy h128 = {&sh_h128, false, true};
    if (dtype == RMSNORM_F32 || !vec)
        return nullptr;
    const bool b = dtype == RMSNORM_BF16;
    if (H == 128 && dense)
        return b ? &b128 : &h128;
    if (H == 4096)
        return b ? &b4096 : &h4096;
    if (H == 5120)
        return b ? &b5120 : &h5120;
    return nullptr;
}

cudaError_t launch2(const void *fn, dim3 grid, dim3 block, int smem, cudaStream_t s, void *a0,
                    void *a1)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    void *args[2] = {a0, a1};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// -------------------------------------------------------- kernel choice
// The row-wise layouts of one 16-bit format.
struct HalfSet {
    const RowKernels &s32, &s1024, &h128, &h128w, &h896, &h4096, &h4096w, &h5120, &h5120w,
        &g32, &g128, &g512;
};

const RowKernels &pick_half(const HalfSet &k, int64_t H, bool vec, bool wide)
{
    if (!vec)
        return H <= k.s32.max_cols() ? k.s32 : k.s1024;
    if (H == 128) return wide ? k.h128w : k.h128;
    if (H == 896) return k.h896;
    if (H == 4096) return wide ? k.h4096w : k.h4096;
    if (H == 5120) return wide ? k.h5120w : k.h5120;
    if (H <= k.g32.max_cols()) return k.g32;
    if (H <= k.g128.max_cols()) return k.g128;
    return k.g512;
}

// wide: every row start 32-byte aligned (pointers, H * element size and the
// row strides), so a forward with 32-byte packs may run.
const RowKernels &pick_rows(int dtype, int64_t H, bool vec, bool wide)
{
    static const HalfSet bf = {b_s32, b_s1024, b_h128, b_h128w, b_h896, b_h4096,
                               b_h4096w, b_h5120, b_h5120w, b_g32, b_g128, b_g512};
    static const HalfSet hf = {h_s32, h_s1024, h_h128, h_h128w, h_h896, h_h4096,
                               h_h4096w, h_h5120, h_h5120w, h_g32, h_g128, h_g512};
    if (dtype == RMSNORM_BF16)
        return pick_half(bf, H, vec, wide);
    if (dtype == RMSNORM_F16)
        return pick_half(hf, H, vec, wide);
    if (!vec)
        return H <= f_s32.max_cols() ? f_s32 : f_s1024;
    if (H == 896) return f_h896;
    if (H <= f_g32.max_cols()) return f_g32;
    if (H <= f_g128.max_cols()) return f_g128;
    return f_g512;
}

const SplitKernels &pick_split(int dtype, bool vec)
{
    if (dtype == RMSNORM_BF16)
        return vec ? split_bf16_v : split_bf16_s;
    if (dtype == RMSNORM_F16)
        return vec ? split_f16_v : split_f16_s;
    return vec ? split_f32_v : split_f32_s;
}

cudaError_t launch(const void *fn, dim3 grid, dim3 block, cudaStream_t s, void *arg,
                   bool pdl, unsigned cluster_x)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    unsigned n = 0;
    if (pdl) {
        attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_x) {
        attrs[n].id = cudaLaunchAttributeClusterDimension;
        attrs[n].val.clusterDim.x = cluster_x;
        attrs[n].val.clusterDim.y = 1;
        attrs[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = n;
    void *args[1] = {arg};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// ------------------------------------------------------------- forward
// Arguments already checked; ld* are row strides in elements (H if dense).
int fwd_impl(const void *x, int64_t ldx, const void *r, int64_t ldr, const void *w, void *y,
             int64_t ldy, void *h, int64_t ldh, float *rstd, int64_t M, int64_t H, float eps,
             int dtype, cudaStream_t stream)
{
    const bool res = r != nullptr;
    if (!res)
        ldr = ldh = H;
    const size_t es = elem_size(dtype);
    const bool vec16 = (H * (int64_t)es) % 16 == 0 && aligned(x, 16) && aligned(w, 16) &&
                       aligned(y, 16) && aligned(r, 16) && aligned(h, 16) &&
                       strides_multiple(16, es, {ldx, ldr, ldy, ldh});
    const int ov = g_path_override.load(std::memory_order_relaxed);
    const bool vec = vec16 && ov != kPathScalar;
    const bool wide = vec && (H * (int64_t)es) % 32 == 0 && aligned(x, 32) && aligned(w, 32) &&
                      aligned(y, 32) && aligned(r, 32) && aligned(h, 32) &&
                      strides_multiple(32, es, {ldx, ldr, ldy, ldh});
    const bool dense = ldx == H && ldr == H && ldy == H && ldh == H;
    const bool split = M <= 65535 && (ov == kPathSplit || (ov == kPathAuto && M <= kSplitMaxRows));

    if (split) {
        const SplitKernels &k = pick_split(dtype, vec);
        const int E = vec ? k.E : 1;
        const int NV = (int)(H / E);
        int K = (NV + 31) / 32;
        K = K < 2 ? 2 : (K > 8 ? 8 : K);
        const int SV = (NV + K - 1) / K;
        int NT = (SV + 31) / 32 * 32;
        NT = NT > 256 ? 256 : NT;
        const int V = (SV + NT - 1) / NT;   // <= 8 for H <= RMSNORM_MAX_H
        const void *fn = V == 1 ? (res ? k.v1_res : k.v1) : (res ? k.v8_res : k.v8);
        int dev;
        cudaError_t de = cudaGetDevice(&dev);
        if (de != cudaSuccess)
            return cuda_fail(de);
        unsigned int *tmo = stream_timeout_counter(dev);
        if (tmo == nullptr)
            return cuda_fail(cudaErrorInvalidSymbol);
        SplitParams p = {x, r, w, y, h, rstd, (int)H, NV, SV, eps, ldx, ldr, ldy, ldh, tmo,
                         g_test_extra_tx.load(std::memory_order_relaxed),
                         g_test_wait_us.load(std::memory_order_relaxed)};
        cudaError_t e = launch(fn, dim3(K, (unsigned)M), dim3(NT), stream, &p, true, K);
        if (e != cudaSuccess)
            return cuda_fail(e);
        t_last_path = kPathSplit;
        return RMSNORM_OK;
    }

    FwdParams p = {x, r, w, y, h, rstd, M, (int)H, eps, ldx, ldr, ldy, ldh, 0, 0};
    const StreamPolicy *sp = pick_stream(dtype, H, vec, dense);
    if (sp && (ov == kPathStream || (ov == kPathAuto && sp->auto_fwd))) {
        const StreamKernels &k = *sp->k;
        const void *fn = k.fwd[res ? 1 : 0];
        const int smem = k.fwd_smem[res ? 1 : 0];
        int64_t grid;
        int dev;
        int st = stream_grid(k.f, fn, smem, M, &grid, &dev);
        if (st)
            return st;
        unsigned int *tmo = stream_timeout_counter(dev);
        if (tmo == nullptr)
            return cuda_fail(cudaErrorInvalidSymbol);
        p.extra_tx = g_test_extra_tx.load(std::memory_order_relaxed);
        p.wait_limit_us = g_test_wait_us.load(std::memory_order_relaxed);
        cudaError_t e = launch2(fn, dim3((unsigned)grid), dim3(k.f.threads()), smem, stream, &p,
                                &tmo);
        if (e != cudaSuccess)
            return cuda_fail(e);
        t_last_path = kPathStream;
        return RMSNORM_OK;
    }

    const RowKernels &k = pick_rows(dtype, H, vec, wide);
    const void *fn = k.fwd[res ? 1 : 0];
    int64_t grid;
    int st = rows_grid(k.f, fn, M, &grid);
    if (st)
        return st;
    cudaError_t e = launch(fn, dim3((unsigned)grid), dim3(k.f.threads()), stream, &p, true, 0);
    if (e != cudaSuccess)
        return cuda_fail(e);
    t_last_path = vec ? kPathRows : kPathScalar;
    return RMSNORM_OK;
}

// Checks shared by the dense and strided forward entry points, then the
// launch. r and h are both NULL (plain) or both given (residual).
int fwd_checked(const void *x, int64_t ldx, const void *r, int64_t ldr, const void *w, void *y,
                int64_t ldy, void *h, int64_t ldh, float *rstd, int64_t M, int64_t H, float eps,
                int dtype, cudaStream_t stream)
{
    int st = check_common(M, H, eps, dtype);
    if (st)
        return st;
    const bool res = r != nullptr || h != nullptr;
    if (res && (r == nullptr || h == nullptr))
        return RMSNORM_ERR_NULLPTR;
    if (!stride_ok(ldx, M, H) || !stride_ok(ldy, M, H) ||
        (res && (!stride_ok(ldr, M, H) || !stride_ok(ldh, M, H))))
        return RMSNORM_ERR_BAD_STRIDE;
    if (M == 0)
        return RMSNORM_OK;
    if (!x || !w || !y)
        return RMSNORM_ERR_NULLPTR;
    const size_t es = elem_size(dtype);
    if (!aligned(x, es) || !aligned(r, es) || !aligned(w, es) || !aligned(h, es) ||
        !aligned(y, es) || !aligned(rstd, 4))
        return RMSNORM_ERR_MISALIGNED;
    const Span sx = rows_span(x, M, H, ldx, es), sw = flat(w, (size_t)H * es),
               sy = rows_span(y, M, H, ldy, es), ss = flat(rstd, (size_t)M * 4);
    if (!res) {
        if (!same_or_disjoint(sy, sx) || overlap(sy, sw) || overlap(ss, sx) ||
            overlap(ss, sw) || overlap(ss, sy))
            return RMSNORM_ERR_ALIAS;
    } else {
        const Span sr = rows_span(r, M, H, ldr, es), sh = rows_span(h, M, H, ldh, es);
        if (!same_or_disjoint(sh, sx) || !same_or_disjoint(sh, sr) || overlap(sh, sw) ||
            overlap(sh, ss))
            return RMSNORM_ERR_ALIAS;
        for (Span b : {sx, sr, sw, sh, ss})
            if (overlap(sy, b))
                return RMSNORM_ERR_ALIAS;
        for (Span b : {sx, sr, sw})
            if (overlap(ss, b))
                return RMSNORM_ERR_ALIAS;
    }
    return fwd_impl(x, ldx, r, ldr, w, y, ldy, h, ldh, rstd, M, H, eps, dtype, stream);
}

// ------------------------------------------------------------ backward
struct BwdPlan {
    const void *fn;
    int threads;
    int smem;
    int64_t grid;     // CTAs, and so partial dw rows
    bool stream;
    bool vec;
    unsigned int *timeouts;
};

// Kernel, grid (and so partial-row count) of the backward for these args.
int bwd_plan(int dtype, int64_t M, int64_t H, bool vec, bool dense, bool dh, bool have_rstd,
             int ov, BwdPlan *pl)
{
    const StreamPolicy *sp = pick_stream(dtype, H, vec, dense);
    pl->vec = vec;
    pl->timeouts = nullptr;
    if (sp && (ov == kPathStream || (ov == kPathAuto && sp->auto_bwd))) {
        const StreamKernels &k = *sp->k;
        pl->fn = k.bwd[dh ? 1 : 0][have_rstd ? 1 : 0];
        pl->threads = k.b.threads();
        pl->smem = k.bwd_smem[dh ? 1 : 0][have_rstd ? 1 : 0];
        pl->stream = true;
        if (M == 0) {
            pl->grid = 0;
            return RMSNORM_OK;
        }
        int dev;
        int st = stream_grid(k.b, pl->fn, pl->smem, M, &pl->grid, &dev);
        if (st)
            return st;
        pl->timeouts = stream_timeout_counter(dev);
        return pl->timeouts ? RMSNORM_OK : cuda_fail(cudaErrorInvalidSymbol);
    }
    const RowKernels &k = pick_rows(dtype, H, vec, false);   // 16-byte packs
    pl->fn = k.bwd[dh ? 1 : 0][have_rstd ? 1 : 0];
    pl->threads = k.b.threads();
    pl->smem = 0;
    pl->stream = false;
    if (M == 0) {
        pl->grid = 0;
        return RMSNORM_OK;
    }
    return rows_grid(k.b, pl->fn, M, &pl->grid);
}

// ld* are row strides in elements (H if dense); a NULL dh's stride is ignored.
int bwd_impl(const void *dy, int64_t lddy, const void *dh, int64_t lddh, const void *x,
             int64_t ldx, const void *w, const float *rstd, void *dx, int64_t lddx, float *dw,
             void *ws, size_t ws_bytes, int64_t M, int64_t H, float eps, int dtype,
             cudaStream_t stream, int flags = 0)
{
    int st = check_common(M, H, eps, dtype);
    if (st)
        return st;
    if (dh == nullptr)
        lddh = H;
    if (!stride_ok(lddy, M, H) || !stride_ok(lddh, M, H) || !stride_ok(ldx, M, H) ||
        !stride_ok(lddx, M, H))
        return RMSNORM_ERR_BAD_STRIDE;
    if (dw == nullptr)
        return RMSNORM_ERR_NULLPTR;
    if (M > 0 && (!dy || !x || !w || !dx))
        return RMSNORM_ERR_NULLPTR;
    const size_t es = elem_size(dtype);
    if (!aligned(dy, es) || !aligned(x, es) || !aligned(w, es) || !aligned(dx, es) ||
        !aligned(dh, es) || !aligned(rstd, 4) || !aligned(dw, 4) || !aligned(ws, 16))
        return RMSNORM_ERR_MISALIGNED;

    const Span sdy = rows_span(dy, M, H, lddy, es), sdh = rows_span(dh, M, H, lddh, es),
               sx = rows_span(x, M, H, ldx, es), sw = flat(w, (size_t)H * es),
               sr = flat(rstd, (size_t)M * 4), sdx = rows_span(dx, M, H, lddx, es),
               sdw = flat(dw, (size_t)H * 4);
    if (!same_or_disjoint(sdx, sdy) || !same_or_disjoint(sdx, sdh) || overlap(sdx, sx) ||
        overlap(sdx, sw) || overlap(sdx, sr) || overlap(sdx, sdw))
        return RMSNORM_ERR_ALIAS;
    for (Span b : {sdy, sdh, sx, sw, sr})
        if (overlap(sdw, b))
            return RMSNORM_ERR_ALIAS;

    const bool vec16 = (H * (int64_t)es) % 16 == 0 && aligned(dy, 16) && aligned(x, 16) &&
                       aligned(w, 16) && aligned(dx, 16) && aligned(dh, 16) &&
                       strides_multiple(16, es, {lddy, lddh, ldx, lddx});
    const bool dense = lddy == H && lddh == H && ldx == H && lddx == H;
    const int ov = g_path_override.load(std::memory_order_relaxed);
    const bool vec = vec16 && ov != kPathScalar;
    BwdPlan pl;
    if ((st = bwd_plan(dtype, M, H, vec, dense, dh != nullptr, rstd != nullptr, ov, &pl)))
        return st;
    const size_t need = (size_t)pl.grid * (size_t)H * sizeof(float);
    if (need > 0 && (ws == nullptr || ws_bytes < need))
        return RMSNORM_ERR_WORKSPACE;
    const Span sws = flat(ws, need);
    for (Span b : {sdy, sdh, sx, sw, sr, sdx, sdw})
        if (overlap(sws, b))
            return RMSNORM_ERR_ALIAS;

    if (M > 0) {
        BwdParams p = {dy,  x,        w,    rstd, dh,  dx,   static_cast<float *>(ws),
                       M,   (int)H,   eps,  lddy, ldx, lddh, lddx,
                       0,   0};
        if (pl.stream) {
            p.extra_tx = g_test_extra_tx.load(std::memory_order_relaxed);
            p.wait_limit_us = g_test_wait_us.load(std::memory_order_relaxed);
        }
        cudaError_t e =
            pl.stream ? launch2(pl.fn, dim3((unsigned)pl.grid), dim3(pl.threads), pl.smem, stream,
                                &p, &pl.timeouts)
                      : launch(pl.fn, dim3((unsigned)pl.grid), dim3(pl.threads), stream, &p,
                               true, 0);
        if (e != cudaSuccess)
            return cuda_fail(e);
    }
    const float *part = static_cast<const float *>(ws);
    int P = (int)pl.grid, Hi = (int)H, acc = (flags & RMSNORM_BWD_ACCUMULATE_DW) ? 1 : 0;
    struct {
        const float *part;
        int P, H;
        float *dw;
        int acc;
    } a = {part, P, Hi, dw, acc};
    void *args[5] = {&a.part, &a.P, &a.H, &a.dw, &a.acc};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((H + kReduceCols - 1) / kReduceCols));
    cfg.blockDim = dim3(kReduceCols * kReduceRows);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelExC(
        &cfg, (const void *)&dw_reduce<kReduceCols, kReduceRows>, args);
    if (e != cudaSuccess)
        return cuda_fail(e);
    t_last_path = M == 0 ? 0 : (pl.stream ? kPathStream : (vec ? kPathRows : kPathScalar));
    return RMSNORM_OK;
}

// ------------------------------------------------------- double backward
const Bwd2Kernel &pick_bwd2(int dtype, int64_t H, bool vec)
{
    struct Set {
        const Bwd2Kernel &g32, &g128, &h4096, &g512, &s1024;
    };
    static const Set bf = {b2_bf_g32, b2_bf_g128, b2_bf_h4096, b2_bf_g512, b2_bf_s1024};
    static const Set hf = {b2_h_g32, b2_h_g128, b2_h_h4096, b2_h_g512, b2_h_s1024};
    static const Set f3 = {b2_f_g32, b2_f_g128, b2_f_g128, b2_f_g512, b2_f_s1024};
    const Set &k = dtype == RMSNORM_BF16 ? bf : (dtype == RMSNORM_F16 ? hf : f3);
    if (!vec)
        return k.s1024;
    if (H == 4096 && dtype != RMSNORM_F32)
        return k.h4096;
    if (H <= k.g32.s.cols()) return k.g32;
    if (H <= k.g128.s.cols()) return k.g128;
    return k.g512;
}

// The double backward's kernel and grid (and so its partial-row count):
// streamed for the 16-bit feature counts with a streamed layout unless the
// row-wise family is forced, row-wise otherwise.
struct Bwd2Plan {
    const void *fn;
    int threads, smem;
    int64_t grid;
    bool stream;
    unsigned int *timeouts;
};

int bwd2_plan(int dtype, int64_t M, int64_t H, bool vec, bool have_rstd, int ov, Bwd2Plan *pl)
{
    const StreamPolicy *sp = pick_stream(dtype, H, vec, true);
    pl->timeouts = nullptr;
    if (sp && sp->k->bwd2[0] != nullptr && (ov == kPathAuto || ov == kPathStream)) {
        const StreamKernels &k = *sp->k;
        pl->fn = k.bwd2[have_rstd ? 1 : 0];
        pl->threads = k.d.threads();
        pl->smem = k.bwd2_smem[have_rstd ? 1 : 0];
        pl->stream = true;
        if (M == 0) {
            pl->grid = 0;
            return RMSNORM_OK;
        }
        int dev;
        int st = stream_grid(k.d, pl->fn, pl->smem, M, &pl->grid, &dev);
        if (st)
            return st;
        pl->timeouts = stream_timeout_counter(dev);
        return pl->timeouts ? RMSNORM_OK : cuda_fail(cudaErrorInvalidSymbol);
    }
    const Bwd2Kernel &k = pick_bwd2(dtype, H, vec);
    pl->fn = k.fn;
    pl->threads = k.s.threads();
    pl->smem = 0;
    pl->stream = false;
    if (M == 0) {
        pl->grid = 0;
        return RMSNORM_OK;
    }
    return rows_grid(k.s, k.fn, M, &pl->grid);
}

int bwd2_impl(const void *dy, const void *x, const void *w, const float *rstd, const void *gx,
              const float *gw, void *ddy, void *dx2, float *dw2, void *ws, size_t ws_bytes,
              int64_t M, int64_t H, float eps, int dtype, cudaStream_t stream)
{
    int st = check_common(M, H, eps, dtype);
    if (st)
        return st;
    if (dw2 == nullptr)
        return RMSNORM_ERR_NULLPTR;
    if (M > 0 && (!dy || !x || !w || !ddy || !dx2))
        return RMSNORM_ERR_NULLPTR;
    const size_t es = elem_size(dtype);
    if (!aligned(dy, es) || !aligned(x, es) || !aligned(w, es) || !aligned(gx, es) ||
        !aligned(ddy, es) || !aligned(dx2, es) || !aligned(rstd, 4) || !aligned(gw, 16) ||
        !aligned(dw2, 4) || !aligned(ws, 16))
        return RMSNORM_ERR_MISALIGNED;
    const size_t rows = (size_t)M * (size_t)H * es;
    const Span sdy = flat(dy, rows), sx = flat(x, rows), sw = flat(w, (size_t)H * es),
               sr = flat(rstd, (size_t)M * 4), sgx = flat(gx, rows), sgw = flat(gw, (size_t)H * 4),
               sddy = flat(ddy, rows), sdx2 = flat(dx2, rows), sdw2 = flat(dw2, (size_t)H * 4);
    for (Span o : {sddy, sdx2, sdw2})
        for (Span i : {sdy, sx, sw, sr, sgx, sgw})
            if (overlap(o, i))
                return RMSNORM_ERR_ALIAS;
    if (overlap(sddy, sdx2) || overlap(sddy, sdw2) || overlap(sdx2, sdw2))
        return RMSNORM_ERR_ALIAS;

    const bool vec16 = (H * (int64_t)es) % 16 == 0 && aligned(dy, 16) && aligned(x, 16) &&
                       aligned(w, 16) && aligned(gx, 16) && aligned(ddy, 16) && aligned(dx2, 16);
    const int ov = g_path_override.load(std::memory_order_relaxed);
    const bool vec = vec16 && ov != kPathScalar;
    Bwd2Plan pl;
    if ((st = bwd2_plan(dtype, M, H, vec, rstd != nullptr, ov, &pl)))
        return st;
    const int64_t grid = pl.grid;
    const size_t need = (size_t)grid * (size_t)H * sizeof(float);
    if (need > 0 && (ws == nullptr || ws_bytes < need))
        return RMSNORM_ERR_WORKSPACE;
    const Span sws = flat(ws, need);
    for (Span b : {sdy, sx, sw, sr, sgx, sgw, sddy, sdx2, sdw2})
        if (overlap(sws, b))
            return RMSNORM_ERR_ALIAS;

    if (M > 0) {
        Bwd2Params p = {dy, x, w, rstd, gx, gw, ddy, dx2, static_cast<float *>(ws), M,
                        (int)H, eps, 0, 0};
        cudaError_t e;
        if (pl.stream) {
            p.extra_tx = g_test_extra_tx.load(std::memory_order_relaxed);
            p.wait_limit_us = g_test_wait_us.load(std::memory_order_relaxed);
            e = launch2(pl.fn, dim3((unsigned)grid), dim3(pl.threads), pl.smem, stream, &p,
                        &pl.timeouts);
        } else {
            e = launch(pl.fn, dim3((unsigned)grid), dim3(pl.threads), stream, &p, true, 0);
        }
        if (e != cudaSuccess)
            return cuda_fail(e);
    }
    const float *part = static_cast<const float *>(ws);
    int P = (int)grid, Hi = (int)H, acc = 0;
    void *args[5] = {&part, &P, &Hi, &dw2, &acc};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((H + kReduceCols - 1) / kReduceCols));
    cfg.blockDim = dim3(kReduceCols * kReduceRows);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelExC(
        &cfg, (const void *)&dw_reduce<kReduceCols, kReduceRows>, args);
    if (e != cudaSuccess)
        return cuda_fail(e);
    t_last_path = M == 0 ? 0 : (pl.stream ? kPathStream : (vec ? kPathRows : kPathScalar));
    return RMSNORM_OK;
}

// ------------------------------------------------- norm + projection GEMV
// The bulk-copy fed kernel's plan: tiles per warp, K slice, ring stages,
// shared memory, or false when it does not fit (the register-fed kernel runs
// then).
// Rows above which the tcgen05 kernel is the automatic choice (at 1 to 8
// rows the bulk-copy kernel is faster: its 8-row MMA tile wastes less).
constexpr int64_t kGemvUmmaMinRows = 8;
constexpr int64_t kGemvTcMinH = 2048;     // rows wide enough for the persistent kernel

struct GemvTmaPlan {
    int TPW, KS, NSW, ctas, CS;
    bool stage_r;
    int64_t smem;
};

constexpr int64_t kGemvMinSliceTwoCtas = 256;
// cuTensorMapEncodeTiled, from the driver through the runtime's entry-point
// query (the library does not link the driver library itself); nullptr if
// the driver does not offer it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// cap: most CTAs that may run at once (0: SMs x CTAs per SM), for clusters
// the resident clusters x CS.
bool gemv_tma_plan(int64_t M, int64_t H, int64_t N, bool res, int sms, int64_t cap,
                   GemvTmaPlan *pl)
{
    const int MT = (int)((M + 15) / 16);
    const bool half = M <= 8;
    const int CS = MT > 1 ? kGemvCluster : 1;     // the norm shared by a cluster
    const int64_t tiles = (N + 7) / 8;
    for (int sr = res ? 1 : 0; sr >= 0; --sr) {
        const bool stage_r = sr != 0;
        const int64_t fixed = gemv_tma_fixed_bytes(MT, half, (int)M, (int)H, stage_r, CS);
        // Two CTAs per SM with half of its shared memory each when that
        // leaves room for a ring (one call's CTA and the next call's can then
        // share an SM), else one CTA per SM with all of it.
        for (int cps : {2, 1}) {
            const int64_t budget = cps == 2 ? (kGemvMaxSmem - 2048) / 2 : kGemvMaxSmem;
            // every warp with a tile, no more CTAs than fit at once (a whole
            // number of clusters)
            int64_t limit = (int64_t)cps * sms;
            if (cap > 0 && cap < limit)
                limit = cap;
            limit = limit / CS * CS;
            if (limit < CS)
                continue;
            int64_t ctas = (tiles + kGemvWarps - 1) / kGemvWarps;
            if (ctas > limit)
                ctas = limit;
            const int64_t TPW = (tiles + kGemvWarps * ctas - 1) / (kGemvWarps * ctas);
            ctas = (tiles + kGemvWarps * TPW - 1) / (kGemvWarps * TPW);
            ctas = (ctas + CS - 1) / CS * CS;        // whole clusters
            // whole rows first, in as many stages as there are tiles (<= 2)
            int NSW = TPW < 2 ? 1 : 2;
            int64_t bytes =
                gemv_tma_smem_bytes(MT, half, (int)M, (int)H, stage_r, CS, (int)H, NSW);
            int64_t KS = H;
            if (bytes > budget) {              // else K slices, double-buffered
                NSW = 2;
                const int64_t room = budget - fixed - kGemvWarps * NSW * 8;
                KS = (room / (kGemvWarps * NSW * 8) - 64) / 2;
                KS = KS / 32 * 32;
                // Two CTAs per SM only with slices of 256 columns or more:
                // narrower ones make every step a few short copies through a
                // two-stage ring (measured at 48 x 896 -> 9728: 64-column
                // slices, two CTAs per SM, 40 us; whole rows, one CTA per SM,
                // 18 us). One CTA per SM takes whatever fits, 64 at least.
                if (KS < (cps == 2 ? kGemvMinSliceTwoCtas : 64))
                    continue;
                bytes = gemv_tma_smem_bytes(MT, half, (int)M, (int)H, stage_r, CS, (int)KS, NSW);
            }
            *pl = {(int)TPW, (int)KS, NSW, (int)ctas, CS, stage_r, bytes};
            return true;
        }
    }
    return false;
}

// The tcgen05 kernel's plan (gemv_umma.cuh): KS CTAs per tile of 128
// features split K; among the cluster sizes whose shared memory fits and
// whose clusters are all resident at once, the fewest atoms per CTA, then
// the smallest cluster; if none is resident at once, the smallest that fits.
// KS = 0: none fits.
struct GemvUmmaPlan {
    int T, na, KS;
    int64_t tiles;
    UmmaLayout L;
    const void *fn;
};

// Whether some cluster of the tcgen05 kernel fits (M rows, H features).
bool gemv_umma_fits(int64_t M, int64_t H, bool res)
{
    const int T = (int)((M + 15) / 16 * 16);
    const int na = (int)((H + kUmmaKC - 1) / kUmmaKC);
    if (T > 64 || H % 16 != 0)
        return false;
    for (int ks = 1; ks <= kUmmaMaxCluster && ks <= na; ++ks)
        if ((int64_t)gemv_umma_layout(T, (int)H, ks, res).total <= kGemvMaxSmem)
            return true;
    return false;
}

int gemv_umma_plan(int64_t M, int64_t H, int64_t N, bool res, int dt, int dev, GemvUmmaPlan *pl)
{
    pl->T = (int)((M + 15) / 16 * 16);
    pl->na = (int)((H + kUmmaKC - 1) / kUmmaKC);
    pl->tiles = (N + kUmmaM - 1) / kUmmaM;
    pl->KS = 0;
    pl->fn = gemv_umma_kernels.fn[dt][res ? 1 : 0];
    if (pl->T > 64 || H % 16 != 0)
        return RMSNORM_OK;
    bool wave = false;
    for (int ks = 1; ks <= kUmmaMaxCluster && ks <= pl->na; ++ks) {
        const UmmaLayout L = gemv_umma_layout(pl->T, (int)H, ks, res);
        if ((int64_t)L.total > kGemvMaxSmem)
            continue;
        int maxc;
        const int st = max_active_clusters(pl->fn, kUmmaThreads, (int)L.total, ks, dev, &maxc);
        if (st)
            return st;
        const bool w1 = pl->tiles <= (int64_t)maxc;
        if (pl->KS == 0 || (w1 && (!wave || L.apc < pl->L.apc))) {
            pl->KS = ks;
            pl->L = L;
            wave = w1;
        }
    }
    return RMSNORM_OK;
}

// The persistent tcgen05 kernel's plan (gemv_tc.cuh): a cluster size KS
// from 1 to 8 that fits (at most the atoms of K, a ring of two stages beside
// the CTA's slice of y, w and the exchange blocks), with the deepest ring
// that fits. At 16 tokens the first of a fixed order, measured on GB300
// (residual, weights from HBM, per call): on rows of more than 1024 features
// clusters of 4 (4096 -> 6144: 17.7 us; against 39.1 alone, 20.3 in pairs,
// 27.4 in threes, 20.7 in fives, 21.6 in sixes, 24.6 in sevens, 21.8 in
// eights; 4096 -> 24576: 39.9 us in fours against 43.4 to 62.2 for the
// other sizes), then pairs, clusters of 8 and single CTAs; on narrower rows
// single CTAs first (896 -> 9728: 9.4 us alone, 12.0 in pairs, 13.0 in
// fours, 23.0 in eights), then 2, 4 and 8. Above 16 tokens the MMA thread's
// pace per atom grows with the tokens and the y slice shrinks the ring, so
// fewer atoms per CTA pay: there the plan takes the size with the least
// estimated time (gemv_tc_estimate_us): 4, 5 or 6 at 4096 features (4096
// -> 24576 at 32 tokens: 43.2 us in fives against 51.5 in fours; at 64
// tokens 65.7 in sixes against 79.5 in eights).
struct GemvTcPlan {
    int T, na, KS;
    int64_t clusters;
    TcLayout L;
};

// The deepest ring for one cluster size; false if no ring of two stages fits.
bool gemv_tc_layout_for(int T, int64_t H, int KS, TcLayout *out)
{
    bool found = false;
    for (int aps : {2, 1})
        for (int nst = 16; nst >= 2; --nst) {
            const TcLayout L = gemv_tc_layout(T, (int)H, KS, nst, aps);
            if ((int64_t)L.total > kGemvMaxSmem)
                continue;
            if (!found || L.NSt * L.APS > out->NSt * out->APS) {
                *out = L;
                found = true;
            }
            break;
        }
    return found;
}

bool gemv_tc_fits(int64_t M, int64_t H)
{
    const int T = (int)((M + 15) / 16 * 16);
    const int na = (int)((H + kUmmaKC - 1) / kUmmaKC);
    if (T > 64 || H % 16 != 0)
        return false;
    TcLayout L;
    for (int ks = 1; ks <= kTcMaxCluster; ++ks)
        if (ks <= na && gemv_tc_layout_for(T, H, ks, &L))
            return true;
    return false;
}

// Estimated microseconds of the persistent kernel's call with clusters of
// KS (above 16 tokens): the weight's atoms a CTA streams (ceil(tiles /
// clusters) tiles of its apc atoms) at the slowest of three rates (the MMA
// thread's pace, 0.1 + 0.1 T / 16 us an atom, 0.05 us more where each atom
// has its own stage and commit; the ring's bytes in flight over a 1.5 us
// round trip; the CTA's share of 7 TB/s of HBM), plus the norm of its slice
// (0.1 us an atom per 16 tokens) and each tile's exchange (0.2 us per peer).
// Fitted on GB300 to per-call times of every cluster size that fits, at 32,
// 48 and 64 tokens and 2048-5120 features (15 shapes): the pick is within
// 5 % of the best measured size in every case, within 1 % in 12.
static double gemv_tc_estimate_us(int T, int apc, const TcLayout &L, int64_t tiles,
                                  int64_t clusters, int KS)
{
    const double atom = (double)kTcAtom;
    const double t_atom = 0.1 + 0.1 * (double)T / 16.0 + (L.APS == 1 ? 0.05 : 0.0);
    const double ring = (double)L.NSt * (double)L.APS * atom;
    const double rate = std::min({atom / t_atom, ring / 1.5,
                                  7.0e6 / (double)(clusters * KS)});      // bytes per us
    const double rounds = (double)((tiles + clusters - 1) / clusters);
    return rounds * (double)apc * atom / rate + 0.1 * (double)apc * (double)T / 16.0 +
           0.2 * rounds * (double)(KS - 1);
}

// st != 0: a CUDA query failed; pl->KS == 0: nothing fits.
int gemv_tc_plan(int64_t M, int64_t H, int64_t N, const void *fn, int dev, int sms,
                 GemvTcPlan *pl)
{
    pl->T = (int)((M + 15) / 16 * 16);
    pl->na = (int)((H + kUmmaKC - 1) / kUmmaKC);
    pl->KS = 0;
    if (pl->T > 64 || H % 16 != 0)
        return RMSNORM_OK;
    const int64_t tiles = (N + kUmmaM - 1) / kUmmaM;
    // Clusters of KS resident at once, with the layout for KS; false if KS
    // does not fit.
    auto resident_for = [&](int ks, TcLayout *L, int64_t *resident) -> int {
        *resident = 0;
        if (ks > pl->na || !gemv_tc_layout_for(pl->T, H, ks, L))
            return RMSNORM_OK;
        if (ks == 1) {
            int bps;
            const int st = blocks_per_sm(fn, kTcThreads, dev, &bps, (int)L->total);
            if (st)
                return st;
            *resident = (int64_t)bps * sms;
        } else {
            int maxc;
            const int st = max_active_clusters(fn, kTcThreads, (int)L->total, ks, dev, &maxc);
            if (st)
                return st;
            *resident = maxc;
        }
        return RMSNORM_OK;
    };
    if (const int forced = g_test_tc_cluster.load(std::memory_order_relaxed)) {
        TcLayout L;
        int64_t resident;
        if (const int st = resident_for(forced, &L, &resident))
            return st;
        if (resident >= 1) {
            pl->KS = forced;
            pl->clusters = tiles < resident ? tiles : resident;
            pl->L = L;
        }
        return RMSNORM_OK;
    }
    if (pl->T == 16) {
        // 16 tokens: a fixed order, measured (the weight's copies, not the
        // MMAs, pace the call there)
        static const int wide[4] = {4, 2, 8, 1}, narrow[4] = {1, 2, 4, 8};
        const int *order = pl->na > 16 ? wide : narrow;
        for (int i = 0; i < 4 && pl->KS == 0; ++i) {
            TcLayout L;
            int64_t resident;
            if (const int st = resident_for(order[i], &L, &resident))
                return st;
            if (resident < 1)
                continue;
            pl->KS = order[i];
            pl->clusters = tiles < resident ? tiles : resident;
            pl->L = L;
        }
        return RMSNORM_OK;
    }
    // more tokens: the cluster size with the least estimated time (the
    // smaller one on a tie)
    double best = 0.0;
    for (int ks = 1; ks <= kTcMaxCluster; ++ks) {
        TcLayout L;
        int64_t resident;
        if (const int st = resident_for(ks, &L, &resident))
            return st;
        if (resident < 1)
            continue;
        const int64_t clusters = tiles < resident ? tiles : resident;
        const double est = gemv_tc_estimate_us(pl->T, L.apc, L, tiles, clusters, ks);
        if (pl->KS == 0 || est < best) {
            best = est;
            pl->KS = ks;
            pl->clusters = clusters;
            pl->L = L;
        }
    }
    return RMSNORM_OK;
}

int gemv_impl(const void *x, const void *r, const void *w, const void *A, void *out, void *h,
              void *y, float *rstd, int64_t M, int64_t H, int64_t N, float eps, int dtype,
              int flags, cudaStream_t stream)
{
    const int MT = (int)((M + 15) / 16);
    const bool half = M <= 8;
    const int ysr = (int)(H * 2 + 64);     // padded: the two rows a quarter-warp reads
                                           // fall in different halves of the banks
    const int dt = dtype == RMSNORM_F16 ? 1 : 0;
    const int ti = half ? 0 : MT;
    int dev, sms, st;
    if ((st = current_device(&dev)) || (st = sm_count(dev, &sms)))
        return st;
    const uint32_t static_w = (flags & RMSNORM_GEMV_STATIC_WEIGHTS) ? 1 : 0;
    const int ov = g_path_override.load(std::memory_order_relaxed);

    // The persistent tcgen05 kernel (gemv_tc.cuh): forced (override 8); or
    // automatic above kGemvUmmaMinRows rows on rows of at least kGemvTcMinH
    // features (measured faster there than the K-split kernel at every size
    // tried: 4096 -> 6144 at 16 / 48 rows 18.6 / 28.2 against 27.2 / 37.1
    // us, 4096 -> 24576 46 / 59 against 85 / 122 us); or automatic above
    // kGemvUmmaMinRows rows wherever the K-split kernel does not fit. At 896
    // features the K-split kernel is faster (896 -> 9728 at 16 rows: 8.0
    // against 9.4 us). launch_tc returns 1 when it did not take the call.
    auto launch_tc = [&]() -> int {
        PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
        const void *fn =
            gemv_tc_kernels.fn[dt][r != nullptr ? 1 : 0][(M + 15) / 16 * 16 <= 48 ? 1 : 0];
        GemvTcPlan tp;
        tp.KS = 0;
        if (encode != nullptr && (st = gemv_tc_plan(M, H, N, fn, dev, sms, &tp)))
            return st;
        if (encode != nullptr && tp.KS > 0) {
            const CUtensorMapDataType et =
                dt == 1 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
            // [rows][H] with the 128-byte swizzle, out-of-range reads zero:
            // A in boxes of 128 rows x 64 columns, x in boxes of T x 64
            auto make_map = [&](CUtensorMap *map, const void *base, int64_t rows,
                                uint32_t box_rows) {
                const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)rows};
                const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
                const cuuint32_t box[2] = {(cuuint32_t)kUmmaKC, (cuuint32_t)box_rows};
                const cuuint32_t estr[2] = {1, 1};
                return encode(map, et, 2, const_cast<void *>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            };
            CUtensorMap mapA, mapX;
            if (make_map(&mapA, A, N, kUmmaM) != CUDA_SUCCESS ||
                make_map(&mapX, x, M, (uint32_t)tp.T) != CUDA_SUCCESS)
                return cuda_fail(cudaErrorInvalidValue);
            unsigned int *tmo = stream_timeout_counter(dev);
            if (tmo == nullptr)
                return cuda_fail(cudaErrorInvalidSymbol);
            GemvTcParams p = {r,    w,     out,   h,    y,      rstd,
                              (int)M, (int)H, (int)N, tp.T, tp.na, tp.L,
                              eps,  (int)static_w,
                              g_test_extra_tx.load(std::memory_order_relaxed),
                              g_test_wait_us.load(std::memory_order_relaxed)};
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(tp.clusters * tp.KS));
            cfg.blockDim = dim3(kTcThreads);
            cfg.dynamicSmemBytes = (size_t)tp.L.total;
            cfg.stream = stream;
            cudaLaunchAttribute attrs[2];
            attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attrs[0].val.programmaticStreamSerializationAllowed = 1;
            attrs[1].id = cudaLaunchAttributeClusterDimension;
            attrs[1].val.clusterDim.x = (unsigned)tp.KS;
            attrs[1].val.clusterDim.y = 1;
            attrs[1].val.clusterDim.z = 1;
            cfg.attrs = attrs;
            cfg.numAttrs = tp.KS > 1 ? 2 : 1;
            void *args[4] = {&p, &mapA, &mapX, &tmo};
            const cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
            if (e != cudaSuccess)
                return cuda_fail(e);
            t_last_path = kPathGemvTc;
            return (int)RMSNORM_OK;
        }
        return 1;
    };
    if (ov == kPathGemvTc || (ov == kPathAuto && M > kGemvUmmaMinRows && H >= kGemvTcMinH)) {
        if ((st = launch_tc()) <= 0)
            return st;
    }

    // The product on tcgen05 with K split over a cluster: automatic above
    // kGemvUmmaMinRows rows where y is too large for one CTA (measured faster
    // there than the warp-level MMA kernels), or forced (override 7); where
    // no cluster size fits, the kernels below.
    if (ov == kPathGemvUmma || (ov == kPathAuto && M > kGemvUmmaMinRows)) {
        PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
        GemvUmmaPlan up;
        if (encode != nullptr) {
            if ((st = gemv_umma_plan(M, H, N, r != nullptr, dt, dev, &up)))
                return st;
        }
        if (encode != nullptr && up.KS > 0) {
            const CUtensorMapDataType et =
                dt == 1 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
            // 2-D tensors [rows][H columns], 128-byte swizzle, out-of-range
            // rows and columns read as zero: A in boxes of 128 rows x 64
            // columns, x and r in boxes of T rows x 64 columns
            auto make_map = [&](CUtensorMap *map, const void *base, int64_t rows,
                                uint32_t box_rows) {
                const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)rows};
                const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
                const cuuint32_t box[2] = {(cuuint32_t)kUmmaKC, (cuuint32_t)box_rows};
                const cuuint32_t estr[2] = {1, 1};
                return encode(map, et, 2, const_cast<void *>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            };
            CUtensorMap mapA, mapX, mapR;
            if (make_map(&mapA, A, N, kUmmaM) != CUDA_SUCCESS ||
                make_map(&mapX, x, M, (uint32_t)up.T) != CUDA_SUCCESS ||
                make_map(&mapR, r != nullptr ? r : x, M, (uint32_t)up.T) != CUDA_SUCCESS)
                return cuda_fail(cudaErrorInvalidValue);
            unsigned int *tmo = stream_timeout_counter(dev);
            if (tmo == nullptr)
                return cuda_fail(cudaErrorInvalidSymbol);
            GemvUmmaParams p = {w,       out,           h,   y,   rstd, (int)M, (int)H, (int)N,
                                up.T,    up.na,         up.L, eps, (int)static_w,
                                g_test_extra_tx.load(std::memory_order_relaxed),
                                g_test_wait_us.load(std::memory_order_relaxed)};
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(up.tiles * up.KS));
            cfg.blockDim = dim3(kUmmaThreads);
            cfg.dynamicSmemBytes = (size_t)up.L.total;
            cfg.stream = stream;
            cudaLaunchAttribute attrs[2];
            attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attrs[0].val.programmaticStreamSerializationAllowed = 1;
            attrs[1].id = cudaLaunchAttributeClusterDimension;
            attrs[1].val.clusterDim.x = (unsigned)up.KS;
            attrs[1].val.clusterDim.y = 1;
            attrs[1].val.clusterDim.z = 1;
            cfg.attrs = attrs;
            cfg.numAttrs = 2;
            void *args[5] = {&p, &mapA, &mapX, &mapR, &tmo};
            const cudaError_t e = cudaLaunchKernelExC(&cfg, up.fn, args);
            if (e != cudaSuccess)
                return cuda_fail(e);
            t_last_path = kPathGemvUmma;
            return RMSNORM_OK;
        }
    }

    // Above kGemvUmmaMinRows rows where no K-split cluster fits: the
    // persistent kernel, whose slices of y are smaller.
    if (ov == kPathAuto && M > kGemvUmmaMinRows &&
        gemv_smem_bytes(MT, half, (int)M, (int)H, false) > kGemvMaxSmem) {
        if ((st = launch_tc()) <= 0)
            return st;
    }

    // The warp-level MMA kernels need y (16-row tiles) and w in shared
    // memory: a call accepted for a tcgen05 kernel alone stops here when
    // none was taken (override 1 or 6, or no tensor-map encoder).
    if (gemv_smem_bytes(MT, half, (int)M, (int)H, false) > kGemvMaxSmem)
        return RMSNORM_ERR_UNSUPPORTED;
    GemvTmaPlan pl;
    bool tma = ov != kPathRows && gemv_tma_plan(M, H, N, r != nullptr, sms, 0, &pl);
    auto tma_fn = [&]() {
        return gemv_tma_kernels.fn[dt][ti][r == nullptr ? 0 : (pl.stage_r ? 2 : 1)];
    };
    // With clusters, plan again for the clusters that can be resident at
    // once: a grid of more would run a second wave.
    for (int pass = 0; tma && pl.CS > 1 && pass < 2; ++pass) {
        int maxc;
        if ((st = max_active_clusters(tma_fn(), kGemvWarps * 32, (int)pl.smem, pl.CS, dev,
                                      &maxc)))
            return st;
        if (pl.ctas <= (int64_t)maxc * pl.CS)
            break;
        tma = pass == 0 &&
              gemv_tma_plan(M, H, N, r != nullptr, sms, (int64_t)maxc * pl.CS, &pl);
    }
    if (tma) {
        const void *fn = tma_fn();
        int bps;
        if ((st = blocks_per_sm(fn, kGemvWarps * 32, dev, &bps, (int)pl.smem)))
            return st;
        if (pl.ctas <= bps * sms) {
            unsigned int *tmo = stream_timeout_counter(dev);
            if (tmo == nullptr)
                return cuda_fail(cudaErrorInvalidSymbol);
            GemvParams p = {x,      r,      w,      A,      out,     h,   y,
                            rstd,   (int)M, (int)H, (int)N, pl.TPW,  ysr, eps,
                            (int)static_w, pl.KS, pl.NSW,
                            g_test_extra_tx.load(std::memory_order_relaxed),
                            g_test_wait_us.load(std::memory_order_relaxed)};
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)pl.ctas);
            cfg.blockDim = dim3(kGemvWarps * 32);
            cfg.dynamicSmemBytes = (size_t)pl.smem;
            cfg.stream = stream;
            cudaLaunchAttribute attrs[2];
            attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attrs[0].val.programmaticStreamSerializationAllowed = 1;
            attrs[1].id = cudaLaunchAttributeClusterDimension;
            attrs[1].val.clusterDim.x = (unsigned)pl.CS;
            attrs[1].val.clusterDim.y = 1;
            attrs[1].val.clusterDim.z = 1;
            cfg.attrs = attrs;
            cfg.numAttrs = pl.CS > 1 ? 2 : 1;
            void *args[2] = {&p, &tmo};
            cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
            if (e != cudaSuccess)
                return cuda_fail(e);
            t_last_path = kPathGemvTma;
            return RMSNORM_OK;
        }
    }

    // A in registers: one 8-row tile per CTA at a time
    const void *const(&fns)[3] = gemv_kernels.fn[dt][ti];
    const int64_t tiles = (N + 7) / 8;
    // Tiles per CTA so that every CTA is resident at once, for a variant.
    auto plan = [&](int variant, int smem, int64_t *tn) {
        int bps;
        int s2 = blocks_per_sm(fns[variant], kGemvWarps * 32, dev, &bps, smem);
        if (s2)
            return s2;
        const int64_t cap = (int64_t)bps * sms;
        *tn = (tiles + cap - 1) / cap;
        return (int)RMSNORM_OK;
    };
    // r is staged in shared memory with x and w whenever it fits (measured:
    // staging beats reading r from L2 in the norm even when it costs the
    // grid a second round of tiles)
    const bool stage_r =
        r != nullptr && gemv_smem_bytes(MT, half, (int)M, (int)H, true) <= kGemvMaxSmem;
    const int variant = r == nullptr ? 0 : (stage_r ? 2 : 1);
    const int smem = (int)gemv_smem_bytes(MT, half, (int)M, (int)H, stage_r);
    int64_t TN;
    if ((st = plan(variant, smem, &TN)))
        return st;
    const void *fn = fns[variant];
    const int64_t grid = (tiles + TN - 1) / TN;
    GemvParams p = {x,      r,      w,      A,      out,     h,   y,
                    rstd,   (int)M, (int)H, (int)N, (int)TN, ysr, eps,
                    (int)static_w, 0, 0, 0, 0};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kGemvWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    void *args[1] = {&p};
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess)
        return cuda_fail(e);
    t_last_path = kPathGemv;
    return RMSNORM_OK;
}

} // namespace

// =================================================================== C ABI
extern "C" {

int rmsnorm_fwd(const void *x, const void *w, void *y, float *rstd, int64_t M, int64_t H,
                float eps, int dtype, void *stream)
{
    return fwd_checked(x, H, nullptr, H, w, y, H, nullptr, H, rstd, M, H, eps, dtype,
                       static_cast<cudaStream_t>(stream));
}

int rmsnorm_residual_fwd(const void *x, const void *r, const void *w, void *h, void *y,
                         float *rstd, int64_t M, int64_t H, float eps, int dtype, void *stream)
{
    if (check_common(M, H, eps, dtype) == RMSNORM_OK && M > 0 && (!r || !h))
        return RMSNORM_ERR_NULLPTR;
    return fwd_checked(x, H, r, H, w, y, H, h, H, rstd, M, H, eps, dtype,
                       static_cast<cudaStream_t>(stream));
}

int rmsnorm_fwd_strided(const void *x, int64_t ldx, const void *r, int64_t ldr, const void *w,
                        void *y, int64_t ldy, void *h, int64_t ldh, float *rstd, int64_t M,
                        int64_t H, float eps, int dtype, void *stream)
{
    return fwd_checked(x, ldx, r, ldr, w, y, ldy, h, ldh, rstd, M, H, eps, dtype,
                       static_cast<cudaStream_t>(stream));
}

int rmsnorm_bwd(const void *dy, const void *x, const void *w, const float *rstd, void *dx,
                float *dw, void *workspace, size_t workspace_bytes, int64_t M, int64_t H,
                float eps, int dtype, void *stream)
{
    return bwd_impl(dy, H, nullptr, H, x, H, w, rstd, dx, H, dw, workspace, workspace_bytes, M,
                    H, eps, dtype, static_cast<cudaStream_t>(stream));
}

int rmsnorm_residual_bwd(const void *dy, const void *dh_out, const void *h, const void *w,
                         const float *rstd, void *dx, float *dw, void *workspace,
                         size_t workspace_bytes, int64_t M, int64_t H, float eps, int dtype,
                         void *stream)
{
    return bwd_impl(dy, H, dh_out, H, h, H, w, rstd, dx, H, dw, workspace, workspace_bytes, M,
                    H, eps, dtype, static_cast<cudaStream_t>(stream));
}

int rmsnorm_bwd_ex(const void *dy, const void *dh_out, const void *x, const void *w,
                   const float *rstd, void *dx, float *dw, void *workspace,
                   size_t workspace_bytes, int64_t M, int64_t H, float eps, int dtype, int flags,
                   void *stream)
{
    if (flags & ~RMSNORM_BWD_ACCUMULATE_DW)
        return RMSNORM_ERR_BAD_FLAGS;
    return bwd_impl(dy, H, dh_out, H, x, H, w, rstd, dx, H, dw, workspace, workspace_bytes, M,
                    H, eps, dtype, static_cast<cudaStream_t>(stream), flags);
}

int rmsnorm_bwd_strided(const void *dy, int64_t lddy, const void *dh_out, int64_t lddh,
                        const void *x, int64_t ldx, const void *w, const float *rstd, void *dx,
                        int64_t lddx, float *dw, void *workspace, size_t workspace_bytes,
                        int64_t M, int64_t H, float eps, int dtype, int flags, void *stream)
{
    if (flags & ~RMSNORM_BWD_ACCUMULATE_DW)
        return RMSNORM_ERR_BAD_FLAGS;
    return bwd_impl(dy, lddy, dh_out, lddh, x, ldx, w, rstd, dx, lddx, dw, workspace,
                    workspace_bytes, M, H, eps, dtype, static_cast<cudaStream_t>(stream), flags);
}

int rmsnorm_gemv_fwd(const void *x, const void *r, const void *w, const void *A, void *out,
                     void *h, void *y, float *rstd, int64_t M, int64_t H, int64_t N, float eps,
                     int dtype, int flags, void *stream)
{
    if (flags & ~RMSNORM_GEMV_STATIC_WEIGHTS)
        return RMSNORM_ERR_BAD_FLAGS;
    int st = check_common(M, H, eps, dtype);
    if (st)
        return st;
    if (N < 1 || N > INT32_MAX / 2 || N * H > INT64_MAX / 8)
        return RMSNORM_ERR_BAD_SHAPE;
    if (dtype == RMSNORM_F32 || M > kGemvMaxRows || H % 32 != 0)
        return RMSNORM_ERR_UNSUPPORTED;
    // the warp-level MMA kernels fit, or above kGemvUmmaMinRows rows the
    // tcgen05 kernel does
    const int MT = (int)((M + 15) / 16);
    if (gemv_smem_bytes(MT > 0 ? MT : 1, false, (int)M, (int)H, false) > kGemvMaxSmem &&
        !(M > kGemvUmmaMinRows && (gemv_umma_fits(M, H, r != nullptr) || gemv_tc_fits(M, H))))
        return RMSNORM_ERR_UNSUPPORTED;
    if (h != nullptr && r == nullptr)
        return RMSNORM_ERR_NULLPTR;
    if (M == 0)
        return RMSNORM_OK;
    if (!x || !w || !A || !out)
        return RMSNORM_ERR_NULLPTR;
    if (!aligned(x, 16) || !aligned(r, 16) || !aligned(w, 16) || !aligned(A, 16) ||
        !aligned(h, 16) || !aligned(y, 16) || !aligned(out, 2) || !aligned(rstd, 4))
        return RMSNORM_ERR_MISALIGNED;
    const size_t es = 2;
    const Span sx = flat(x, (size_t)(M * H) * es), sr = flat(r, (size_t)(M * H) * es),
               sw = flat(w, (size_t)H * es), sA = flat(A, (size_t)(N * H) * es),
               so = flat(out, (size_t)(M * N) * es), sh = flat(h, (size_t)(M * H) * es),
               sy = flat(y, (size_t)(M * H) * es), ss = flat(rstd, (size_t)M * 4);
    // Every CTA reads x and r while CTA 0 writes h, y and rstd: no output may
    // share a byte with an input or with another output.
    for (Span o : {so, sh, sy, ss}) {
        for (Span i : {sx, sr, sw, sA})
            if (overlap(o, i))
                return RMSNORM_ERR_ALIAS;
    }
    if (overlap(so, sh) || overlap(so, sy) || overlap(so, ss) || overlap(sh, sy) ||
        overlap(sh, ss) || overlap(sy, ss))
        return RMSNORM_ERR_ALIAS;
    return gemv_impl(x, r, w, A, out, h, y, rstd, M, H, N, eps, dtype, flags,
                     static_cast<cudaStream_t>(stream));
}

int rmsnorm_bwd_bwd(const void *dy, const void *x, const void *w, const float *rstd,
                    const void *gdx, const float *gdw, void *ddy, void *dx2, float *dw2,
                    void *workspace, size_t workspace_bytes, int64_t M, int64_t H, float eps,
                    int dtype, void *stream)
{
    return bwd2_impl(dy, x, w, rstd, gdx, gdw, ddy, dx2, dw2, workspace, workspace_bytes, M, H,
                     eps, dtype, static_cast<cudaStream_t>(stream));
}

size_t rmsnorm_bwd_workspace_bytes(int64_t M, int64_t H, int dtype)
{
    if (check_common(M, H, 0.f, dtype) != RMSNORM_OK)
        return 0;
    size_t most = 0;
    for (int ov : {kPathAuto, kPathRows, kPathStream})
        for (int vec = 0; vec < 2; ++vec)
            for (int dh = 0; dh < 2; ++dh)
                for (int hr = 0; hr < 2; ++hr) {
                    BwdPlan pl;
                    if (bwd_plan(dtype, M, H, vec != 0, true, dh != 0, hr != 0, ov, &pl) !=
                        RMSNORM_OK)
                        return 0;
                    const size_t need = (size_t)pl.grid * (size_t)H * sizeof(float);
                    most = need > most ? need : most;
                }
    for (int ov : {kPathAuto, kPathRows})     // the double backward's grids too
        for (int vec = 0; vec < 2; ++vec)
            for (int hr = 0; hr < 2; ++hr) {
                Bwd2Plan pl;
                if (bwd2_plan(dtype, M, H, vec != 0, hr != 0, ov, &pl) != RMSNORM_OK)
                    return 0;
                const size_t need = (size_t)pl.grid * (size_t)H * sizeof(float);
                most = need > most ? need : most;
            }
    return most;
}

const char *rmsnorm_status_string(int status)
{
    switch (status) {
    case RMSNORM_OK: return "ok";
    case RMSNORM_ERR_NULLPTR: return "a required pointer is NULL";
    case RMSNORM_ERR_BAD_SHAPE: return "bad shape (M < 0, H < 1 or M*H too large)";
    case RMSNORM_ERR_BAD_DTYPE: return "dtype is not RMSNORM_F32, RMSNORM_BF16 or RMSNORM_F16";
    case RMSNORM_ERR_BAD_EPS: return "eps must be finite and >= 0";
    case RMSNORM_ERR_MISALIGNED: return "pointer not aligned to its element size (workspace: 16 bytes)";
    case RMSNORM_ERR_WORKSPACE: return "workspace missing or smaller than rmsnorm_bwd_workspace_bytes()";
    case RMSNORM_ERR_UNSUPPORTED: return "H exceeds RMSNORM_MAX_H, or the call is outside the limits of its entry point";
    case RMSNORM_ERR_CUDA: return "a CUDA runtime call failed (see rmsnorm_last_cuda_error)";
    case RMSNORM_ERR_ALIAS: return "output buffers overlap inputs or each other in a way not allowed";
    case RMSNORM_ERR_BAD_FLAGS: return "unknown bits in flags";
    case RMSNORM_ERR_BAD_STRIDE: return "a row stride is below H, above 2^31-1 or too large for the row count";
    case RMSNORM_ERR_SCRATCH_LIMIT:
        return "problem needs more scratch than RMSNORM_STATIC_SCRATCH_BYTES (use rmsnorm_bwd with a workspace)";
    default: return "unknown status";
    }
}

int rmsnorm_last_cuda_error(void) { return t_last_cuda_error; }

void rmsnorm_set_path_override(int path)
{
    const bool ok = (path >= kPathAuto && path <= kPathStream) || path == kPathGemvTma ||
                    path == kPathGemvUmma || path == kPathGemvTc;
    g_path_override.store(ok ? path : kPathAuto);
}

void rmsnorm_set_gemv_cluster_test(int cluster_size)
{
    g_test_tc_cluster.store(cluster_size >= 1 && cluster_size <= kTcMaxCluster ? cluster_size : 0);
}

void rmsnorm_set_stream_test_fault(unsigned int extra_tx_bytes, unsigned int wait_limit_us)
{
    g_test_extra_tx.store(extra_tx_bytes);
    g_test_wait_us.store(wait_limit_us);
}

int rmsnorm_wait_timeouts(unsigned int *count, int reset)
{
    if (count == nullptr)
        return RMSNORM_ERR_NULLPTR;
    int dev, st;
    if ((st = current_device(&dev)))
        return st;
    unsigned int *p = stream_timeout_counter(dev);
    if (p == nullptr)
        return cuda_fail(cudaErrorInvalidSymbol);
    cudaError_t e = cudaMemcpy(count, p, sizeof(unsigned int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && reset)
        e = cudaMemset(p, 0, sizeof(unsigned int));
    return e == cudaSuccess ? RMSNORM_OK : cuda_fail(e);
}

int rmsnorm_last_path(void) { return t_last_path; }

} // extern "C"

// ============================================ backward with built-in scratch
// For callers that cannot allocate device memory (see rmsnorm.h): the dw
// partial rows live in this file-scope device array instead of a
// caller-provided workspace. Host code must not use the array's name as a
// pointer (on the host it is only a stand-in); the device address comes
// from cudaGetSymbolAddress, looked up once per device (and again only if
// that device's context has been replaced, as by cudaDeviceReset).
namespace {

constexpr int kMaxDevices = 64;
static __device__ __align__(256) unsigned char g_static_scratch[RMSNORM_STATIC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};
// Test hook: a smaller usable size of the array (0: all of it).
std::atomic<size_t> g_scratch_test_limit{0};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

// Device address of g_static_scratch on the current device.
int static_scratch_address(void **out)
{
    int dev, st;
    if ((st = current_device(&dev)))
        return st;
    if (dev < 0 || dev >= kMaxDevices)
        return cuda_fail(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> g(g_scratch_mu);
    const unsigned long long ctx = current_context_id();
    if (g_scratch_addr[dev] == nullptr || ctx == 0 || g_scratch_ctx[dev] != ctx) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess)
            return cuda_fail(e);
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = current_context_id();
    }
    *out = g_scratch_addr[dev];
    return RMSNORM_OK;
}

} // namespace

extern "C" int rmsnorm_bwd_static_scratch(const void *dy, const void *x, const void *w,
                                          const float *rstd, void *dx, float *dw, int64_t M,
                                          int64_t H, float eps, int dtype, void *stream)
{
    int st = check_common(M, H, eps, dtype);
    if (st)
        return st;
    // The bound covers every kernel variant this call could take. (Without a
    // device the query gives 0 and the address lookup below reports it.)
    const size_t test_limit = g_scratch_test_limit.load(std::memory_order_relaxed);
    const size_t usable = test_limit != 0 && test_limit < RMSNORM_STATIC_SCRATCH_BYTES
                              ? test_limit
                              : RMSNORM_STATIC_SCRATCH_BYTES;
    if (rmsnorm_bwd_workspace_bytes(M, H, dtype) > usable)
        return RMSNORM_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    if ((st = static_scratch_address(&scratch)))
        return st;
    return bwd_impl(dy, H, nullptr, H, x, H, w, rstd, dx, H, dw, scratch,
                    RMSNORM_STATIC_SCRATCH_BYTES, M, H, eps, dtype,
                    static_cast<cudaStream_t>(stream));
}

extern "C" void rmsnorm_set_static_scratch_test_limit(size_t bytes)
{
    g_scratch_test_limit.store(bytes);
}
