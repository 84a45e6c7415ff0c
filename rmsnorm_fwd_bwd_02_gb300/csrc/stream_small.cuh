// stream_small.cuh -- streamed kernels for short rows (H = 8 * NVP elements of
// a 16-bit format, NVP packs of 16 bytes per row, NVP a power of two <= 32),
// e.g. the 128-wide rows of Qwen3's QK-norm. Rows must be contiguous (row
// stride H in every tensor): one bulk copy moves a block of rows.
//
// Same arithmetic as rows.cuh ([P1] "训推加速 Qwen3 实战：从“调包”到手写 Triton
// Kernel（含 backward）" §4.1-4.2, §5.3-5.4). A row is NVP lanes, so a warp
// spans 32/NVP rows per instruction and every row sum is a butterfly over
// NVP lanes: no cross-warp reduction. Each warp therefore runs its own
// pipeline: a ring of NS shared-memory stages, each holding R = (32/NVP)*RPT
// consecutive rows of every staged tensor, filled by one cp.async.bulk per
// tensor (the rows are contiguous in memory) issued by lane 0 and completing
// on the stage's mbarrier. The warp works through a stage (lane = one pack of
// RPT rows), then refills it NS stages ahead. Waits are bounded as in
// stream.cuh; the dw accumulators (one pack of columns per lane) are folded
// over the warp's rows and then over the CTA's warps in a fixed order.
#pragma once

#include "stream.cuh"

namespace rmsk {

// Each warp's ring holds NS stages, or as many as fit in kBudget bytes for
// all warps (at least two).
template <int NVP, int RPT, int NW, int NS, int NTEN>
struct SmallSmem {
    static constexpr int kRows = (32 / NVP) * RPT;              // rows per stage
    static constexpr int kRowBytes = NVP * 16;
    static constexpr int kTenBytes = kRows * kRowBytes;           // one tensor
    static constexpr int kStageBytes = NTEN * kTenBytes;
    static constexpr int kBudget = 210 * 1024;
    static constexpr int kFit = kBudget / (NW * kStageBytes);
    static constexpr int kNS = NS * NW * kStageBytes <= kBudget ? NS : kFit;
    static constexpr int kStagesBytes = NW * kNS * kStageBytes;
    static constexpr int kBarOff = kStagesBytes;
    static constexpr int kBytes = kBarOff + NW * kNS * 8;
    static_assert(kBytes <= 227 * 1024, "shared memory per CTA");
    static_assert(kNS >= 2, "at least two stages");
};

// ------------------------------------------------------------------ forward
template <typename T, int NVP, int RPT, int NW, int NS, bool RES>
__global__ void __launch_bounds__(NW * 32, 1)
rms_fwd_stream_small(const FwdParams p, unsigned int *timeouts)
{
    using P = Pack<T, 8>;
    using X = Vals<8>;
    using F = float2;
    constexpr int NTEN = RES ? 2 : 1;
    using SM = SmallSmem<NVP, RPT, NW, NS, NTEN>;
    constexpr int RW = 32 / NVP;           // rows per warp instruction
    constexpr int NSE = SM::kNS;   // stages per warp
    extern __shared__ __align__(128) unsigned char smem[];

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int sub = lane / NVP;            // row of this lane within an instruction
    const int pk = lane % NVP;             // pack (column block) of this lane
    const uint32_t stage0 = smem_addr(smem) + warp * NSE * SM::kStageBytes;
    const uint32_t bar0 = smem_addr(smem) + SM::kBarOff + warp * NSE * 8;

    if (lane == 0)
        for (int s = 0; s < NSE; ++s)
            mbar_init(bar0 + 8 * s, 1);
    mbar_init_fence();
    __syncwarp();
    griddep_wait();
    const unsigned long long limit = wait_limit_ns(p.wait_limit_us);

    X wv;
    P::load_cached(p.w, pk).widen(wv);
    const float fH = (float)p.H;
    const int64_t wgid = (int64_t)blockIdx.x * NW + warp;
    const int64_t TW = (int64_t)gridDim.x * NW;
    const int64_t nblocks = (p.M + SM::kRows - 1) / SM::kRows;
    const int64_t nk = wgid < nblocks ? (nblocks - 1 - wgid) / TW + 1 : 0;

    auto issue = [&](int64_t k) {
        const int64_t row0 = (wgid + k * TW) * SM::kRows;
        const int64_t rows = p.M - row0 < SM::kRows ? p.M - row0 : SM::kRows;
        const uint32_t bytes = (uint32_t)(rows * SM::kRowBytes);
        const int s = (int)(k % NSE);
        const uint32_t st = stage0 + s * SM::kStageBytes;
        const uint32_t bar = bar0 + 8 * s;
        mbar_expect_tx(bar, NTEN * bytes + p.extra_tx);
        bulk_g2s(st, static_cast<const uint4 *>(p.x) + row0 * NVP, bytes, bar);
        if constexpr (RES)
            bulk_g2s(st + SM::kTenBytes, static_cast<const uint4 *>(p.r) + row0 * NVP, bytes,
                     bar);
    };
    if (lane == 0) {
        fence_proxy_async_smem();
        for (int64_t k = 0; k < NSE && k < nk; ++k)
            issue(k);
    }
    __syncwarp();

    int64_t k = 0;
    bool failed = false;
    for (; k < nk; ++k) {
        const int64_t row0 = (wgid + k * TW) * SM::kRows;
        const int s = (int)(k % NSE);
        const uint32_t st = stage0 + s * SM::kStageBytes;
        const bool ok = mbar_wait_bounded(bar0 + 8 * s, (uint32_t)((k / NSE) & 1), limit);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
            failed = true;
            break;
        }
        X a[RPT];
        float ss[RPT];
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int rs = j * RW + sub;
            as_pack<T>(lds128(st + rs * SM::kRowBytes + pk * 16)).widen(a[j]);
            if constexpr (RES) {
                X b;
                as_pack<T>(lds128(st + SM::kTenBytes + rs * SM::kRowBytes + pk * 16)).widen(b);
#pragma unroll
                for (int i = 0; i < X::N; ++i)
                    a[j].v[i] = vadd(a[j].v[i], b.v[i]);
                P::narrow(a[j]).widen(a[j]);   // h as stored
            }
            F acc = splat<F>(0.f);
#pragma unroll
            for (int i = 0; i < X::N; ++i)
                acc = vfma(a[j].v[i], a[j].v[i], acc);
            ss[j] = group_allreduce<NVP>(hsum(acc));
        }
        // every lane has its data in registers: release the stage
        __syncwarp();
        if (lane == 0 && k + NSE < nk) {
            fence_proxy_async_smem();
            issue(k + NSE);
        }
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int64_t row = row0 + j * RW + sub;
            if (row >= p.M)
                continue;
            const float r = rsqrtf(ss[j] / fH + p.eps);
            if (p.rstd != nullptr && pk == 0)
                p.rstd[row] = r;
            if constexpr (RES)
                P::narrow(a[j]).store(p.h, row * NVP + pk);
            const F r2 = splat<F>(r);
#pragma unroll
            for (int i = 0; i < X::N; ++i)
                a[j].v[i] = vmul(vmul(a[j].v[i], r2), wv.v[i]);
            P::narrow(a[j]).store(p.y, row * NVP + pk);
        }
    }
    if (failed && lane == 0) {
        atomicAdd(timeouts, 1u);
        for (int64_t q = k; q < k + NSE && q < nk; ++q)
            (void)mbar_wait_bounded(bar0 + 8 * (int)(q % NSE), (uint32_t)((q / NSE) & 1), limit);
    }
    griddep_launch_dependents();
}

// ----------------------------------------------------------------- backward
template <typename T, int NVP, int RPT, int NW, int NS, bool DH, bool LOADR>
__global__ void __launch_bounds__(NW * 32, 1)
rms_bwd_stream_small(const BwdParams p, unsigned int *timeouts)
{
    using P = Pack<T, 8>;
    using X = Vals<8>;
    using F = float2;
    constexpr int NTEN = DH ? 3 : 2;      // x, dy, [dh]
    using SM = SmallSmem<NVP, RPT, NW, NS, NTEN>;
    constexpr int RW = 32 / NVP;
    static_assert(NW * NVP * 8 * 4 <= SM::kStagesBytes, "dw combine reuses the stages");
    constexpr int NSE = SM::kNS;   // stages per warp
    extern __shared__ __align__(128) unsigned char smem[];

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int sub = lane / NVP;
    const int pk = lane % NVP;
    const uint32_t stage0 = smem_addr(smem) + warp * NSE * SM::kStageBytes;
    const uint32_t bar0 = smem_addr(smem) + SM::kBarOff + warp * NSE * 8;

    if (lane == 0)
        for (int s = 0; s < NSE; ++s)
            mbar_init(bar0 + 8 * s, 1);
    mbar_init_fence();
    __syncwarp();
    griddep_wait();
    const unsigned long long limit = wait_limit_ns(p.wait_limit_us);

    X wv, acc = X::zero();
    P::load_cached(p.w, pk).widen(wv);
    const float fH = (float)p.H;
    const int64_t wgid = (int64_t)blockIdx.x * NW + warp;
    const int64_t TW = (int64_t)gridDim.x * NW;
    const int64_t nblocks = (p.M + SM::kRows - 1) / SM::kRows;
    const int64_t nk = wgid < nblocks ? (nblocks - 1 - wgid) / TW + 1 : 0;

    auto issue = [&](int64_t k) {
        const int64_t row0 = (wgid + k * TW) * SM::kRows;
        const int64_t rows = p.M - row0 < SM::kRows ? p.M - row0 : SM::kRows;
        const uint32_t bytes = (uint32_t)(rows * SM::kRowBytes);
        const int s = (int)(k % NSE);
        const uint32_t st = stage0 + s * SM::kStageBytes;
        const uint32_t bar = bar0 + 8 * s;
        mbar_expect_tx(bar, NTEN * bytes + p.extra_tx);
        bulk_g2s(st, static_cast<const uint4 *>(p.x) + row0 * NVP, bytes, bar);
        bulk_g2s(st + SM::kTenBytes, static_cast<const uint4 *>(p.dy) + row0 * NVP, bytes, bar);
        if constexpr (DH)
            bulk_g2s(st + 2 * SM::kTenBytes, static_cast<const uint4 *>(p.dh) + row0 * NVP,
                     bytes, bar);
    };
    if (lane == 0) {
        fence_proxy_async_smem();
        for (int64_t k = 0; k < NSE && k < nk; ++k)
            issue(k);
    }
    __syncwarp();

    int64_t k = 0;
    bool failed = false;
    for (; k < nk; ++k) {
        const int64_t row0 = (wgid + k * TW) * SM::kRows;
        const int s = (int)(k % NSE);
        const uint32_t st = stage0 + s * SM::kStageBytes;
        float rs[RPT];
        if constexpr (LOADR) {
            // issued before the wait so their latency overlaps it
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
                const int64_t row = row0 + j * RW + sub;
                rs[j] = row < p.M ? p.rstd[row] : 0.f;
            }
        }
        const bool ok = mbar_wait_bounded(bar0 + 8 * s, (uint32_t)((k / NSE) & 1), limit);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
            failed = true;
            break;
        }
        P xv[RPT], dyv[RPT];
        float cs[RPT], ss[RPT];
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int rs_ = j * RW + sub;
            xv[j] = as_pack<T>(lds128(st + rs_ * SM::kRowBytes + pk * 16));
            dyv[j] = as_pack<T>(lds128(st + SM::kTenBytes + rs_ * SM::kRowBytes + pk * 16));
            X a, b;
            xv[j].widen(a);
            dyv[j].widen(b);
            F c2 = splat<F>(0.f), s2 = splat<F>(0.f);
#pragma unroll
            for (int i = 0; i < X::N; ++i) {
                c2 = vfma(vmul(wv.v[i], b.v[i]), a.v[i], c2);
                if constexpr (!LOADR)
                    s2 = vfma(a.v[i], a.v[i], s2);
            }
            cs[j] = group_allreduce<NVP>(hsum(c2));
            if constexpr (!LOADR)
                ss[j] = group_allreduce<NVP>(hsum(s2));
        }
        P dhv[DH ? RPT : 1];
        if constexpr (DH) {
#pragma unroll
            for (int j = 0; j < RPT; ++j)
                dhv[j] = as_pack<T>(lds128(st + 2 * SM::kTenBytes +
                                           (j * RW + sub) * SM::kRowBytes + pk * 16));
        }
        // every lane has its data in registers: release the stage
        __syncwarp();
        if (lane == 0 && k + NSE < nk) {
            fence_proxy_async_smem();
            issue(k + NSE);
        }
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int64_t row = row0 + j * RW + sub;
            if (row >= p.M)
                continue;
            float r;
            if constexpr (LOADR)
                r = rs[j];
            else
                r = rsqrtf(ss[j] / fH + p.eps);
            const float c = cs[j] / fH;
            const F r2 = splat<F>(r);
            const F negm = splat<F>(-(r * r * r * c));
            X a, b, o;
            xv[j].widen(a);
            dyv[j].widen(b);
#pragma unroll
            for (int i = 0; i < X::N; ++i) {
                o.v[i] = vfma(a.v[i], negm, vmul(r2, vmul(wv.v[i], b.v[i])));
                acc.v[i] = vfma(vmul(b.v[i], a.v[i]), r2, acc.v[i]);
            }
            if constexpr (DH) {
                X d;
                dhv[j].widen(d);
#pragma unroll
                for (int i = 0; i < X::N; ++i)
                    o.v[i] = vadd(o.v[i], d.v[i]);
            }
            P::narrow(o).store(p.dx, row * NVP + pk);
        }
    }
    if (failed && lane == 0) {
        atomicAdd(timeouts, 1u);
        for (int64_t q = k; q < k + NSE && q < nk; ++q)
            (void)mbar_wait_bounded(bar0 + 8 * (int)(q % NSE), (uint32_t)((q / NSE) & 1), limit);
    }
    griddep_launch_dependents();

    // lanes pk, pk + NVP, ... of a warp own the same columns: fold them, then
    // the CTA's warps in warp order, into one partial row.
#pragma unroll
    for (int i = 0; i < X::N; ++i)
#pragma unroll
        for (int o = NVP; o < 32; o <<= 1) {
            acc.v[i].x += __shfl_xor_sync(0xFFFFFFFFu, acc.v[i].x, o);
            acc.v[i].y += __shfl_xor_sync(0xFFFFFFFFu, acc.v[i].y, o);
        }
    __syncthreads();            // all warps done with their stages
    float *comb = reinterpret_cast<float *>(smem);
    if (lane < NVP) {
        float4 *d = reinterpret_cast<float4 *>(comb + (warp * NVP + pk) * 8);
        d[0] = make_float4(acc.v[0].x, acc.v[0].y, acc.v[1].x, acc.v[1].y);
        d[1] = make_float4(acc.v[2].x, acc.v[2].y, acc.v[3].x, acc.v[3].y);
    }
    __syncthreads();
    float *part = p.part + (int64_t)blockIdx.x * p.H;
    for (int c = threadIdx.x; c < NVP * 8; c += NW * 32) {
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < NW; ++q)
            v += comb[q * NVP * 8 + c];
        part[c] = v;
    }
}

} // namespace rmsk
