// api.cu -- the C ABI declared in include/rmsnorm.h: host-side argument
// checks, kernel choice, grid sizing and launches. No allocation, no
// synchronisation, no host copies; everything is enqueued on the caller's
// stream.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "rmsnorm.h"
#include "params.h"
#include "reduce.cuh"
#include "registry.h"

using namespace rmsk;

namespace {

constexpr int kPathAuto = 0, kPathRows = 1, kPathSplit = 2, kPathScalar = 3, kPathStream = 4;
constexpr int kSplitMaxRows = 64;      // decode-sized batches ([P2 §3.2])
constexpr int kReduceCols = 32, kReduceRows = 16;

thread_local int t_last_cuda_error = 0;
thread_local int t_last_path = 0;
std::atomic<int> g_path_override{kPathAuto};
// Test hook for the streamed kernels' bounded waits (see rmsnorm.h).
std::atomic<unsigned> g_test_extra_tx{0}, g_test_wait_us{0};

int cuda_fail(cudaError_t e)
{
    t_last_cuda_error = (int)e;
    return RMSNORM_ERR_CUDA;
}

size_t elem_size(int dtype) { return dtype == RMSNORM_BF16 ? 2 : 4; }

bool aligned(const void *p, size_t a) { return p == nullptr || (uintptr_t)p % a == 0; }

struct Buf {
    const void *p;
    size_t n;
};

bool overlap(Buf a, Buf b)
{
    if (!a.p || !b.p || !a.n || !b.n)
        return false;
    const uintptr_t a0 = (uintptr_t)a.p, b0 = (uintptr_t)b.p;
    return a0 < b0 + b.n && b0 < a0 + a.n;
}

// Allowed: the same buffer exactly, or no overlap at all.
bool same_or_disjoint(Buf a, Buf b)
{
    return (a.p == b.p && a.n == b.n) || !overlap(a, b);
}

int check_common(int64_t M, int64_t H, float eps, int dtype)
{
    if (dtype != RMSNORM_F32 && dtype != RMSNORM_BF16)
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

// Resident CTAs per SM for a kernel, cached per (kernel, device). Kernels
// with dynamic shared memory above the default limit are opted in first.
int blocks_per_sm(const void *fn, int threads, int dev, int *out, int smem = 0)
{
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, int> cache;
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find({fn, dev});
        if (it != cache.end()) {
            *out = it->second;
            return RMSNORM_OK;
        }
    }
    int n = 0;
    cudaError_t e = cudaSuccess;
    if (smem > 48 * 1024)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem);
    if (e != cudaSuccess)
        return cuda_fail(e);
    if (n < 1)
        return cuda_fail(cudaErrorInvalidConfiguration);
    std::lock_guard<std::mutex> g(mu);
    cache[{fn, dev}] = n;
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

const StreamPolicy *pick_stream(int dtype, int64_t H, bool vec)
{
    static const StreamPolicy h4096 = {&s_h4096, false, true};
    static const StreamPolicy h5120 = {&s_h5120, false, true};
    static const StreamPolicy h128 = {&s_h128, false, true};
    if (dtype != RMSNORM_BF16 || !vec)
        return nullptr;
    if (H == 128)
        return &h128;
    if (H == 4096)
        return &h4096;
    if (H == 5120)
        return &h5120;
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
// wide: every row pointer 32-byte aligned and H * element size a multiple
// of 32, so a forward with 32-byte packs may run.
const RowKernels &pick_rows(int dtype, int64_t H, bool vec, bool wide)
{
    if (dtype == RMSNORM_BF16) {
        if (!vec)
            return H <= b_s32.max_cols() ? b_s32 : b_s1024;
        if (H == 128) return wide ? b_h128w : b_h128;
        if (H == 896) return b_h896;
        if (H == 4096) return wide ? b_h4096w : b_h4096;
        if (H == 5120) return wide ? b_h5120w : b_h5120;
        if (H <= b_g32.max_cols()) return b_g32;
        if (H <= b_g128.max_cols()) return b_g128;
        return b_g512;
    }
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
int fwd_impl(const void *x, const void *r, const void *w, void *y, void *h, float *rstd,
             int64_t M, int64_t H, float eps, int dtype, cudaStream_t stream)
{
    const bool res = r != nullptr;
    const size_t es = elem_size(dtype);
    const bool vec16 = (H * (int64_t)es) % 16 == 0 && aligned(x, 16) && aligned(w, 16) &&
                       aligned(y, 16) && aligned(r, 16) && aligned(h, 16);
    const int ov = g_path_override.load(std::memory_order_relaxed);
    const bool vec = vec16 && ov != kPathScalar;
    const bool wide = vec && (H * (int64_t)es) % 32 == 0 && aligned(x, 32) && aligned(w, 32) &&
                      aligned(y, 32) && aligned(r, 32) && aligned(h, 32);
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
        SplitParams p = {x, r, w, y, h, rstd, (int)H, NV, SV, eps};
        cudaError_t e = launch(fn, dim3(K, (unsigned)M), dim3(NT), stream, &p, true, K);
        if (e != cudaSuccess)
            return cuda_fail(e);
        t_last_path = kPathSplit;
        return RMSNORM_OK;
    }

    const StreamPolicy *sp = pick_stream(dtype, H, vec);
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
        FwdParams p = {x, r, w, y, h, rstd, M, (int)H, eps};
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
    FwdParams p = {x, r, w, y, h, rstd, M, (int)H, eps};
    cudaError_t e = launch(fn, dim3((unsigned)grid), dim3(k.f.threads()), stream, &p, true, 0);
    if (e != cudaSuccess)
        return cuda_fail(e);
    t_last_path = vec ? kPathRows : kPathScalar;
    return RMSNORM_OK;
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
int bwd_plan(int dtype, int64_t M, int64_t H, bool vec, bool dh, bool have_rstd, int ov,
             BwdPlan *pl)
{
    const StreamPolicy *sp = pick_stream(dtype, H, vec);
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

int bwd_impl(const void *dy, const void *dh, const void *x, const void *w, const float *rstd,
             void *dx, float *dw, void *ws, size_t ws_bytes, int64_t M, int64_t H, float eps,
             int dtype, cudaStream_t stream, int flags = 0)
{
    int st = check_common(M, H, eps, dtype);
    if (st)
        return st;
    if (dw == nullptr)
        return RMSNORM_ERR_NULLPTR;
    if (M > 0 && (!dy || !x || !w || !dx))
        return RMSNORM_ERR_NULLPTR;
    const size_t es = elem_size(dtype);
    if (!aligned(dy, es) || !aligned(x, es) || !aligned(w, es) || !aligned(dx, es) ||
        !aligned(dh, es) || !aligned(rstd, 4) || !aligned(dw, 4) || !aligned(ws, 16))
        return RMSNORM_ERR_MISALIGNED;

    const bool vec16 = (H * (int64_t)es) % 16 == 0 && aligned(dy, 16) && aligned(x, 16) &&
                       aligned(w, 16) && aligned(dx, 16) && aligned(dh, 16);
    const int ov = g_path_override.load(std::memory_order_relaxed);
    const bool vec = vec16 && ov != kPathScalar;
    BwdPlan pl;
    if ((st = bwd_plan(dtype, M, H, vec, dh != nullptr, rstd != nullptr, ov, &pl)))
        return st;
    const size_t need = (size_t)pl.grid * (size_t)H * sizeof(float);
    if (need > 0 && (ws == nullptr || ws_bytes < need))
        return RMSNORM_ERR_WORKSPACE;

    const size_t rows = (size_t)M * (size_t)H * es;
    const Buf bdy{dy, rows}, bdh{dh, rows}, bx{x, rows}, bw{w, (size_t)H * es},
        br{rstd, (size_t)M * 4}, bdx{dx, rows}, bdw{dw, (size_t)H * 4}, bws{ws, need};
    if (!same_or_disjoint(bdx, bdy) || !same_or_disjoint(bdx, bdh) || overlap(bdx, bx) ||
        overlap(bdx, bw) || overlap(bdx, br) || overlap(bdx, bdw) || overlap(bdx, bws))
        return RMSNORM_ERR_ALIAS;
    for (Buf b : {bdy, bdh, bx, bw, br, bws})
        if (overlap(bdw, b))
            return RMSNORM_ERR_ALIAS;
    for (Buf b : {bdy, bdh, bx, bw, br})
        if (overlap(bws, b))
            return RMSNORM_ERR_ALIAS;

    if (M > 0) {
        BwdParams p = {dy, x, w, rstd, dh, dx, static_cast<float *>(ws), M, (int)H, eps};
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

} // namespace

// =================================================================== C ABI
extern "C" {

int rmsnorm_fwd(const void *x, const void *w, void *y, float *rstd, int64_t M, int64_t H,
                float eps, int dtype, void *stream)
{
    int st = check_common(M, H, eps, dtype);
    if (st)
        return st;
    if (M == 0)
        return RMSNORM_OK;
    if (!x || !w || !y)
        return RMSNORM_ERR_NULLPTR;
    const size_t es = elem_size(dtype);
    if (!aligned(x, es) || !aligned(w, es) || !aligned(y, es) || !aligned(rstd, 4))
        return RMSNORM_ERR_MISALIGNED;
    const size_t rows = (size_t)M * (size_t)H * es;
    const Buf bx{x, rows}, bw{w, (size_t)H * es}, by{y, rows}, br{rstd, (size_t)M * 4};
    if (!same_or_disjoint(by, bx) || overlap(by, bw) || overlap(br, bx) || overlap(br, bw) ||
        overlap(br, by))
        return RMSNORM_ERR_ALIAS;
    return fwd_impl(x, nullptr, w, y, nullptr, rstd, M, H, eps, dtype,
                    static_cast<cudaStream_t>(stream));
}

int rmsnorm_residual_fwd(const void *x, const void *r, const void *w, void *h, void *y,
                         float *rstd, int64_t M, int64_t H, float eps, int dtype, void *stream)
{
    int st = check_common(M, H, eps, dtype);
    if (st)
        return st;
    if (M == 0)
        return RMSNORM_OK;
    if (!x || !r || !w || !h || !y)
        return RMSNORM_ERR_NULLPTR;
    const size_t es = elem_size(dtype);
    if (!aligned(x, es) || !aligned(r, es) || !aligned(w, es) || !aligned(h, es) ||
        !aligned(y, es) || !aligned(rstd, 4))
        return RMSNORM_ERR_MISALIGNED;
    const size_t rows = (size_t)M * (size_t)H * es;
    const Buf bx{x, rows}, br{r, rows}, bw{w, (size_t)H * es}, bh{h, rows}, by{y, rows},
        bs{rstd, (size_t)M * 4};
    if (!same_or_disjoint(bh, bx) || !same_or_disjoint(bh, br) || overlap(bh, bw) ||
        overlap(bh, bs))
        return RMSNORM_ERR_ALIAS;
    for (Buf b : {bx, br, bw, bh, bs})
        if (overlap(by, b))
            return RMSNORM_ERR_ALIAS;
    for (Buf b : {bx, br, bw})
        if (overlap(bs, b))
            return RMSNORM_ERR_ALIAS;
    return fwd_impl(x, r, w, y, h, rstd, M, H, eps, dtype, static_cast<cudaStream_t>(stream));
}

int rmsnorm_bwd(const void *dy, const void *x, const void *w, const float *rstd, void *dx,
                float *dw, void *workspace, size_t workspace_bytes, int64_t M, int64_t H,
                float eps, int dtype, void *stream)
{
    return bwd_impl(dy, nullptr, x, w, rstd, dx, dw, workspace, workspace_bytes, M, H, eps,
                    dtype, static_cast<cudaStream_t>(stream));
}

int rmsnorm_residual_bwd(const void *dy, const void *dh_out, const void *h, const void *w,
                         const float *rstd, void *dx, float *dw, void *workspace,
                         size_t workspace_bytes, int64_t M, int64_t H, float eps, int dtype,
                         void *stream)
{
    return bwd_impl(dy, dh_out, h, w, rstd, dx, dw, workspace, workspace_bytes, M, H, eps,
                    dtype, static_cast<cudaStream_t>(stream));
}

int rmsnorm_bwd_ex(const void *dy, const void *dh_out, const void *x, const void *w,
                   const float *rstd, void *dx, float *dw, void *workspace,
                   size_t workspace_bytes, int64_t M, int64_t H, float eps, int dtype, int flags,
                   void *stream)
{
    if (flags & ~RMSNORM_BWD_ACCUMULATE_DW)
        return RMSNORM_ERR_BAD_FLAGS;
    return bwd_impl(dy, dh_out, x, w, rstd, dx, dw, workspace, workspace_bytes, M, H, eps,
                    dtype, static_cast<cudaStream_t>(stream), flags);
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
                    if (bwd_plan(dtype, M, H, vec != 0, dh != 0, hr != 0, ov, &pl) != RMSNORM_OK)
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
    case RMSNORM_ERR_BAD_DTYPE: return "dtype is not RMSNORM_F32 or RMSNORM_BF16";
    case RMSNORM_ERR_BAD_EPS: return "eps must be finite and >= 0";
    case RMSNORM_ERR_MISALIGNED: return "pointer not aligned to its element size (workspace: 16 bytes)";
    case RMSNORM_ERR_WORKSPACE: return "workspace missing or smaller than rmsnorm_bwd_workspace_bytes()";
    case RMSNORM_ERR_UNSUPPORTED: return "H exceeds RMSNORM_MAX_H";
    case RMSNORM_ERR_CUDA: return "a CUDA runtime call failed (see rmsnorm_last_cuda_error)";
    case RMSNORM_ERR_ALIAS: return "output buffers overlap inputs or each other in a way not allowed";
    case RMSNORM_ERR_BAD_FLAGS: return "unknown bits in flags";
    case RMSNORM_ERR_SCRATCH_LIMIT:
        return "problem needs more scratch than RMSNORM_STATIC_SCRATCH_BYTES (use rmsnorm_bwd with a workspace)";
    default: return "unknown status";
    }
}

int rmsnorm_last_cuda_error(void) { return t_last_cuda_error; }

void rmsnorm_set_path_override(int path)
{
    g_path_override.store(path >= kPathAuto && path <= kPathStream ? path : kPathAuto);
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
// from cudaGetSymbolAddress, looked up once per device on first use.
namespace {

constexpr int kMaxDevices = 64;
static __device__ __align__(256) unsigned char g_static_scratch[RMSNORM_STATIC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device.
int static_scratch_address(void **out)
{
    int dev, st;
    if ((st = current_device(&dev)))
        return st;
    if (dev < 0 || dev >= kMaxDevices)
        return cuda_fail(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> g(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess)
            return cuda_fail(e);
        g_scratch_addr[dev] = p;
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
    if (rmsnorm_bwd_workspace_bytes(M, H, dtype) > RMSNORM_STATIC_SCRATCH_BYTES)
        return RMSNORM_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    if ((st = static_scratch_address(&scratch)))
        return st;
    return bwd_impl(dy, nullptr, x, w, rstd, dx, dw, scratch, RMSNORM_STATIC_SCRATCH_BYTES, M,
                    H, eps, dtype, static_cast<cudaStream_t>(stream));
}
