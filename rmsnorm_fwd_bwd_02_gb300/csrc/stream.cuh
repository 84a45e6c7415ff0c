// stream.cuh -- row kernels fed by bulk asynchronous copies (the TMA engine)
// for the feature counts with a shaped layout (H = 32 * GW * V * E).
//
// Same arithmetic as rows.cuh ([P1] "训推加速 Qwen3 实战：从“调包”到手写 Triton
// Kernel（含 backward）" §4.1-4.2 forward, §5.3-5.4 backward); what differs is
// how rows reach the SM. A CTA holds NG groups of GW warps. Each group owns
// a ring of NS shared-memory stages, one row per stage (x, plus r or dy and
// dh where the variant reads them). One elected thread of the group issues
// one cp.async.bulk per tensor and row, completing on the stage's mbarrier,
// NS rows ahead of the group's compute, so the bytes in flight per SM are set
// by shared memory (NG * NS stages) rather than by registers. The group
// reads a stage into registers (conflict-free 16-byte shared loads), reduces
// over its warps with one named barrier per row, and that barrier also
// releases the stage for the next copy. Outputs are stored from registers.
// Each tensor has its own row stride, a multiple of 8 elements, so every
// row copy starts on a 16-byte boundary.
//
// Every wait on an mbarrier is bounded in time (%globaltimer). A wait that
// runs out means a copy never landed: the group records it in a device
// counter, waits (again bounded) for its other copies in flight, skips its
// remaining rows and still joins the CTA-wide barriers, so the kernel ends.
#pragma once

#include "common.cuh"
#include "params.h"

namespace rmsk {

constexpr unsigned long long kStageWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ unsigned long long wait_limit_ns(uint32_t us)
{
    return us ? 1000ull * us : kStageWaitLimitNs;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Wait for the phase with this parity to complete; false if it has not
// within limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns)
            return false;
    return true;
}

// Order this thread's earlier generic-proxy accesses to shared memory before
// later async-proxy (bulk copy) writes to it.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bulk copy global -> shared of `bytes` (multiple of 16, both addresses
// 16-byte aligned), completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
                 "[%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// Named barrier over `count` threads that also ORs a predicate across them.
__device__ __forceinline__ bool bar_red_or(int id, int count, bool pred)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.or.pred q, %2, %3, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)pred), "r"(id), "r"(count)
                 : "memory");
    return r != 0;
}

// A 16-byte pack of a 16-bit format read from shared memory.
template <typename T>
__device__ __forceinline__ Pack<T, 8> as_pack(uint4 u)
{
    Pack<T, 8> p;
    p.u = u;
    return p;
}

// Shared-memory layout of one CTA. The stage ring of each group holds NS
// stages, or as many as fit in kBudget bytes for all groups (at least one).
template <int GW, int V, int NG, int NS, int NTEN, int NR>
struct StreamSmem {
    static constexpr int kRowBytes = 32 * GW * V * 16;        // one tensor row
    static constexpr int kStageBytes = NTEN * kRowBytes;
    static constexpr int kBudget = 210 * 1024;
    static constexpr int kFit = kBudget / (NG * kStageBytes);
    static constexpr int kNS = NS * NG * kStageBytes <= kBudget ? NS : (kFit > 0 ? kFit : 1);
    static constexpr int kStagesBytes = NG * kNS * kStageBytes;
    static constexpr int kBarOff = kStagesBytes;                 // NG*kNS mbarriers
    static constexpr int kRedOff = (kBarOff + NG * kNS * 8 + 15) / 16 * 16;  // [NG][2][GW][NR]
    static constexpr int kBytes = kRedOff + NG * 2 * GW * NR * 4;
    static_assert(kBytes <= 227 * 1024, "shared memory per CTA");
    static_assert(kNS >= 2, "a stage is refilled one iteration after use: two at least");
};

// The forward and backward read a stage twice (sums, then outputs) instead
// of holding the row in registers across the group barrier. A stage is refilled one
// iteration after it was consumed: the barrier of iteration k proves every
// thread of the group has finished iteration k-1, whose stage then takes the
// row NS-1 ahead. NS stages therefore keep NS-1 rows in flight per group.

// ------------------------------------------------------------------ forward
// Shaped rows of a 16-bit format (bf16 or fp16; 16-byte packs, E = 8).
template <typename T, int GW, int V, int NG, int NS, bool RES>
__global__ void __launch_bounds__(NG * GW * 32, 1)
rms_fwd_stream(const FwdParams p, unsigned int *timeouts)
{
    using P = Pack<T, 8>;
    using X = Vals<8>;
    using F = float2;
    constexpr int GT = GW * 32;
    constexpr int NV = GT * V;             // packs per row
    constexpr int NTEN = RES ? 2 : 1;
    using SM = StreamSmem<GW, V, NG, NS, NTEN, 1>;
    constexpr int NSE = SM::kNS;           // stages per group
    extern __shared__ __align__(128) unsigned char smem[];

    const int g = threadIdx.x / GT;
    const int t = threadIdx.x % GT;
    const int wg = t / 32;
    const uint32_t stage0 = smem_addr(smem) + g * NSE * SM::kStageBytes;
    const uint32_t bar0 = smem_addr(smem) + SM::kBarOff + g * NSE * 8;
    float *red = reinterpret_cast<float *>(smem + SM::kRedOff) + g * 2 * GW;   // [2][GW]

    if (t == 0)
        for (int s = 0; s < NSE; ++s)
            mbar_init(bar0 + 8 * s, 1);
    mbar_init_fence();
    __syncthreads();
    griddep_wait();
    const unsigned long long limit = wait_limit_ns(p.wait_limit_us);

    P wp[V];
#pragma unroll
    for (int j = 0; j < V; ++j)
        wp[j] = P::load_cached(p.w, t + j * GT);

    const int64_t gg = (int64_t)blockIdx.x * NG + g;
    const int64_t TG = (int64_t)gridDim.x * NG;
    const int64_t nk = gg < p.M ? (p.M - 1 - gg) / TG + 1 : 0;
    const float fH = (float)p.H;

    auto issue = [&](int64_t k) {
        const int64_t row = gg + k * TG;
        const int s = (int)(k % NSE);
        const uint32_t st = stage0 + s * SM::kStageBytes;
        const uint32_t bar = bar0 + 8 * s;
        mbar_expect_tx(bar, SM::kStageBytes + p.extra_tx);
        bulk_g2s(st, static_cast<const uint4 *>(p.x) + row * (p.ldx / 8), SM::kRowBytes, bar);
        if constexpr (RES)
            bulk_g2s(st + SM::kRowBytes, static_cast<const uint4 *>(p.r) + row * (p.ldr / 8),
                     SM::kRowBytes, bar);
    };
    // x (+ r) of pack j of the current stage, widened; with the residual,
    // rounded to the storage format first (h as stored).
    auto row_pack = [&](uint32_t st, int j, X &a) {
        if constexpr (RES) {
            X b;
            as_pack<T>(lds128(st + (t + j * GT) * 16)).widen(a);
            as_pack<T>(lds128(st + SM::kRowBytes + (t + j * GT) * 16)).widen(b);
#pragma unroll
            for (int i = 0; i < X::N; ++i)
                a.v[i] = vadd(a.v[i], b.v[i]);
            P::narrow(a).widen(a);
        } else {
            as_pack<T>(lds128(st + (t + j * GT) * 16)).widen(a);
        }
    };
    if (t == 0) {
        fence_proxy_async_smem();
        for (int64_t k = 0; k < NSE && k < nk; ++k)
            issue(k);
    }

    int64_t k = 0;
    bool failed = false;
    for (; k < nk; ++k) {
        const int64_t row = gg + k * TG;
        const uint32_t st = stage0 + (int)(k % NSE) * SM::kStageBytes;
        const bool ok = mbar_wait_bounded(bar0 + 8 * (int)(k % NSE), (uint32_t)((k / NSE) & 1), limit);

        F acc = splat<F>(0.f);
#pragma unroll
        for (int j = 0; j < V; ++j) {
            X a;
            row_pack(st, j, a);
#pragma unroll
            for (int i = 0; i < X::N; ++i)
                acc = vfma(a.v[i], a.v[i], acc);
        }
        float ss = group_allreduce<32>(hsum(acc));
        float *rb = red + (k & 1) * GW;   // double buffer
        if ((t & 31) == 0)
            rb[wg] = ss;
        // Every thread of the group has posted its sums and finished the
        // previous iteration (whose stage is refilled below).
        if (bar_red_or(1 + g, GT, !ok)) {
            failed = true;
            break;
        }
        if (t == 0 && k >= 1 && k - 1 + NSE < nk) {
            fence_proxy_async_smem();
            issue(k - 1 + NSE);
        }
        ss = 0.f;
#pragma unroll
        for (int q = 0; q < GW; ++q)
            ss += rb[q];
        const float r = rsqrtf(ss / fH + p.eps);
        if (p.rstd != nullptr && t == 0)
            p.rstd[row] = r;
        const F r2 = splat<F>(r);
#pragma unroll
        for (int j = 0; j < V; ++j) {
            X a, wv;
            row_pack(st, j, a);
            if constexpr (RES)
                P::narrow(a).store(p.h, row * (p.ldh / 8) + t + j * GT);
            wp[j].widen(wv);
#pragma unroll
            for (int i = 0; i < X::N; ++i)
                a.v[i] = vmul(vmul(a.v[i], r2), wv.v[i]);
            P::narrow(a).store(p.y, row * (p.ldy / 8) + t + j * GT);
        }
    }
    if (failed && t == 0) {
        atomicAdd(timeouts, 1u);
        // drain this group's copies still in flight (bounded):
        // issued and not consumed: rows k .. k+NSE-2, or all NSE of the
        // prologue when the first wait ran out
        const int64_t last = k == 0 ? NSE - 1 : k + NSE - 2;
        for (int64_t q = k; q <= last && q < nk; ++q)
            (void)mbar_wait_bounded(bar0 + 8 * (int)(q % NSE), (uint32_t)((q / NSE) & 1), limit);
    }
    griddep_launch_dependents();
}

// ----------------------------------------------------------------- backward
template <typename T, int GW, int V, int NG, int NS, bool DH, bool LOADR, bool HOLD = false>
__global__ void __launch_bounds__(NG * GW * 32, 1)
rms_bwd_stream(const BwdParams p, unsigned int *timeouts)
{
    // HOLD: the widened row stays in registers across the group barrier,
    // which then frees its stage at once (refilled NS rows ahead, not NS - 1)
    // and spares the second pass its shared-memory reads and conversions.
    constexpr int LAG = HOLD ? 0 : 1;
    using P = Pack<T, 8>;
    using X = Vals<8>;
    using F = float2;
    constexpr int GT = GW * 32;
    constexpr int NV = GT * V;
    constexpr int NTEN = DH ? 3 : 2;      // x, dy, [dh]
    constexpr int NR = LOADR ? 1 : 2;
    using SM = StreamSmem<GW, V, NG, NS, NTEN, NR>;
    constexpr int NSE = SM::kNS;          // stages per group
    static_assert(NG * NV * 8 * 4 <= SM::kStagesBytes, "dw combine reuses the stages");
    extern __shared__ __align__(128) unsigned char smem[];

    const int g = threadIdx.x / GT;
    const int t = threadIdx.x % GT;
    const int wg = t / 32;
    const uint32_t stage0 = smem_addr(smem) + g * NSE * SM::kStageBytes;
    const uint32_t bar0 = smem_addr(smem) + SM::kBarOff + g * NSE * 8;
    float *red = reinterpret_cast<float *>(smem + SM::kRedOff) + g * 2 * GW * NR;  // [2][GW][NR]

    if (t == 0)
        for (int s = 0; s < NSE; ++s)
            mbar_init(bar0 + 8 * s, 1);
    mbar_init_fence();
    __syncthreads();
    griddep_wait();
    const unsigned long long limit = wait_limit_ns(p.wait_limit_us);

    P wp[V];        // weight kept packed (registers are the constraint here)
    X acc[V];
#pragma unroll
    for (int j = 0; j < V; ++j) {
        wp[j] = P::load_cached(p.w, t + j * GT);
        acc[j] = X::zero();
    }

    const int64_t gg = (int64_t)blockIdx.x * NG + g;
    const int64_t TG = (int64_t)gridDim.x * NG;
    const int64_t nk = gg < p.M ? (p.M - 1 - gg) / TG + 1 : 0;
    const float fH = (float)p.H;

    auto issue = [&](int64_t k) {
        const int64_t row = gg + k * TG;
        const int s = (int)(k % NSE);
        const uint32_t st = stage0 + s * SM::kStageBytes;
        const uint32_t bar = bar0 + 8 * s;
        mbar_expect_tx(bar, SM::kStageBytes + p.extra_tx);
        bulk_g2s(st, static_cast<const uint4 *>(p.x) + row * (p.ldx / 8), SM::kRowBytes, bar);
        bulk_g2s(st + SM::kRowBytes, static_cast<const uint4 *>(p.dy) + row * (p.lddy / 8),
                 SM::kRowBytes, bar);
        if constexpr (DH)
            bulk_g2s(st + 2 * SM::kRowBytes, static_cast<const uint4 *>(p.dh) + row * (p.lddh / 8),
                     SM::kRowBytes, bar);
    };
    if (t == 0) {
        fence_proxy_async_smem();
        for (int64_t k = 0; k < NSE && k < nk; ++k)
            issue(k);
    }

    float r_next = 0.f;
    if constexpr (LOADR)
        r_next = nk > 0 ? p.rstd[gg] : 0.f;

    int64_t k = 0;
    bool failed = false;
    for (; k < nk; ++k) {
        const int64_t row = gg + k * TG;
        const uint32_t st = stage0 + (int)(k % NSE) * SM::kStageBytes;
        float r_cur = 0.f;
        if constexpr (LOADR) {
            r_cur = r_next;                 // loaded one row ahead
            if (k + 1 < nk)
                r_next = p.rstd[row + TG];
        }
        const bool ok = mbar_wait_bounded(bar0 + 8 * (int)(k % NSE), (uint32_t)((k / NSE) & 1), limit);

        F cs = splat<F>(0.f), ss = splat<F>(0.f);
        X hx[HOLD ? V : 1], hdy[HOLD ? V : 1], hdh[HOLD && DH ? V : 1];
#pragma unroll
        for (int j = 0; j < V; ++j) {
            X a, b, wv;
            as_pack<T>(lds128(st + (t + j * GT) * 16)).widen(a);
            as_pack<T>(lds128(st + SM::kRowBytes + (t + j * GT) * 16)).widen(b);
            if constexpr (HOLD) {
                hx[j] = a;
                hdy[j] = b;
                if constexpr (DH)
                    as_pack<T>(lds128(st + 2 * SM::kRowBytes + (t + j * GT) * 16)).widen(hdh[j]);
            }
            wp[j].widen(wv);
#pragma unroll
            for (int i = 0; i < X::N; ++i) {
                cs = vfma(vmul(wv.v[i], b.v[i]), a.v[i], cs);
                if constexpr (!LOADR)
                    ss = vfma(a.v[i], a.v[i], ss);
            }
        }
        float sums[NR];
        sums[0] = group_allreduce<32>(hsum(cs));
        if constexpr (!LOADR)
            sums[1] = group_allreduce<32>(hsum(ss));
        float *rb = red + (k & 1) * GW * NR;   // double buffer
        if ((t & 31) == 0)
#pragma unroll
            for (int i = 0; i < NR; ++i)
                rb[wg * NR + i] = sums[i];
        // Every thread of the group has posted its sums and finished the
        // previous iteration; with HOLD it has also read this row's stage.
        // The stage used LAG iterations ago is refilled below.
        if (bar_red_or(1 + g, GT, !ok)) {
            failed = true;
            break;
        }
        if (t == 0 && k >= LAG && k - LAG + NSE < nk) {
            fence_proxy_async_smem();
            issue(k - LAG + NSE);
        }
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            float v = 0.f;
#pragma unroll
            for (int q = 0; q < GW; ++q)
                v += rb[q * NR + i];
            sums[i] = v;
        }
        float r;
        if constexpr (LOADR)
            r = r_cur;
        else
            r = rsqrtf(sums[1] / fH + p.eps);
        const float c = sums[0] / fH;
        const F r2 = splat<F>(r);
        const F negm = splat<F>(-(r * r * r * c));
#pragma unroll
        for (int j = 0; j < V; ++j) {
            X a, b, o, wv;
            if constexpr (HOLD) {
                a = hx[j];
                b = hdy[j];
            } else {
                as_pack<T>(lds128(st + (t + j * GT) * 16)).widen(a);
                as_pack<T>(lds128(st + SM::kRowBytes + (t + j * GT) * 16)).widen(b);
            }
            wp[j].widen(wv);
#pragma unroll
            for (int i = 0; i < X::N; ++i) {
                o.v[i] = vfma(a.v[i], negm, vmul(r2, vmul(wv.v[i], b.v[i])));
                acc[j].v[i] = vfma(vmul(b.v[i], a.v[i]), r2, acc[j].v[i]);
            }
            if constexpr (DH) {
                X d;
                if constexpr (HOLD)
                    d = hdh[j];
                else
                    as_pack<T>(lds128(st + 2 * SM::kRowBytes + (t + j * GT) * 16)).widen(d);
#pragma unroll
                for (int i = 0; i < X::N; ++i)
                    o.v[i] = vadd(o.v[i], d.v[i]);
            }
            P::narrow(o).store(p.dx, row * (p.lddx / 8) + t + j * GT);
        }
    }
    if (failed && t == 0) {
        atomicAdd(timeouts, 1u);
        // issued and not consumed: rows k .. k+NSE-1-LAG, or all NSE of the
        // prologue when the first wait ran out
        const int64_t last = k == 0 ? NSE - 1 : k + NSE - 1 - LAG;
        for (int64_t q = k; q <= last && q < nk; ++q)
            (void)mbar_wait_bounded(bar0 + 8 * (int)(q % NSE), (uint32_t)((q / NSE) & 1), limit);
    }
    griddep_launch_dependents();

    // Fold the NG groups' dw accumulators (same columns) in group order into
    // one partial row; the stage memory is free now.
    __syncthreads();
    float *comb = reinterpret_cast<float *>(smem);
#pragma unroll
    for (int j = 0; j < V; ++j) {
        float4 *d = reinterpret_cast<float4 *>(comb + (size_t)g * NV * 8 + (t + j * GT) * 8);
        d[0] = make_float4(acc[j].v[0].x, acc[j].v[0].y, acc[j].v[1].x, acc[j].v[1].y);
        d[1] = make_float4(acc[j].v[2].x, acc[j].v[2].y, acc[j].v[3].x, acc[j].v[3].y);
    }
    __syncthreads();
    float *part = p.part + (int64_t)blockIdx.x * p.H;
    for (int c = threadIdx.x; c < NV * 8; c += NG * GT) {
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < NG; ++q)
            v += comb[q * NV * 8 + c];
        part[c] = v;
    }
}

// ---------------------------------------------------------- double backward
// Per-warp slots of the streamed double backward's reduction buffer: the
// four sums as one float4, plus a second float4 holding sum x^2 when rstd is
// recomputed (the registry sizes shared memory with the same count).
__host__ __device__ constexpr int bwd2_stream_slots(bool loadr)
{
    return loadr ? 4 : 8;
}

// The double backward of bwd2.cuh with rows staged like the backward above:
// a stage holds one row of x, dy and gx (gx's copy is skipped, and read as
// zero, when gx is absent); per row the four sums c = sum w dy x, A = sum
// gx w dy, B = sum gx x, D = sum gw dy x (and sum x^2 when rstd is not
// given) go through one group barrier, then ddy and dx2 are written and the
// dw2 accumulators updated. Unlike the kernels above, a thread keeps its
// packs of the row in registers (widened) across the barrier, so the barrier
// that completes row k also frees row k's stage: NS stages keep NS rows in
// flight, and a deep ring per group (one group of 8 warps, 8 stages at
// H = 4096) is what holds the copy engine at full rate with three tensors
// read per row. The four sums cross a warp in one spread reduction
// (warp_sum4_spread) and each warp posts them as one float4 slot (two when
// sum x^2 rides along).
template <typename T, int GW, int V, int NG, int NS, bool LOADR, int MINB = 1>
__global__ void __launch_bounds__(NG * GW * 32, MINB)
rms_bwd2_stream(const Bwd2Params p, unsigned int *timeouts)
{
    using P = Pack<T, 8>;
    using FP = Pack<float, 8>;
    using X = Vals<8>;
    using F = float2;
    constexpr int GT = GW * 32;
    constexpr int NV = GT * V;
    constexpr int NTEN = 3;               // x, dy, gx
    constexpr int NR = bwd2_stream_slots(LOADR);   // c, A, B, D, [sum x^2, pad]
    using SM = StreamSmem<GW, V, NG, NS, NTEN, NR>;
    constexpr int NSE = SM::kNS;
    static_assert(NG * NV * 8 * 4 <= SM::kStagesBytes, "dw combine reuses the stages");
    extern __shared__ __align__(128) unsigned char smem[];

    const int g = threadIdx.x / GT;
    const int t = threadIdx.x % GT;
    const int wg = t / 32;
    const uint32_t stage0 = smem_addr(smem) + g * NSE * SM::kStageBytes;
    const uint32_t bar0 = smem_addr(smem) + SM::kBarOff + g * NSE * 8;
    float *red = reinterpret_cast<float *>(smem + SM::kRedOff) + g * 2 * GW * NR;
    const bool has_gx = p.gx != nullptr;

    if (t == 0)
        for (int s = 0; s < NSE; ++s)
            mbar_init(bar0 + 8 * s, 1);
    mbar_init_fence();
    __syncthreads();
    griddep_wait();
    const unsigned long long limit = wait_limit_ns(p.wait_limit_us);

    P wp[V];        // the weight kept packed, gw widened, dw2 accumulators
    X gwv[V], acc[V];
#pragma unroll
    for (int j = 0; j < V; ++j) {
        wp[j] = P::load_cached(p.w, t + j * GT);
        if (p.gw != nullptr)
            FP::load_cached(p.gw, t + j * GT).widen(gwv[j]);
        else
            gwv[j] = X::zero();
        acc[j] = X::zero();
    }

    const int64_t gg = (int64_t)blockIdx.x * NG + g;
    const int64_t TG = (int64_t)gridDim.x * NG;
    const int64_t nk = gg < p.M ? (p.M - 1 - gg) / TG + 1 : 0;
    const float fH = (float)p.H;
    const int64_t NVr = p.H / 8;          // packs per row (dense rows)

    auto issue = [&](int64_t k) {
        const int64_t row = gg + k * TG;
        const int s = (int)(k % NSE);
        const uint32_t st = stage0 + s * SM::kStageBytes;
        const uint32_t bar = bar0 + 8 * s;
        mbar_expect_tx(bar, (has_gx ? 3 : 2) * SM::kRowBytes + p.extra_tx);
        bulk_g2s(st, static_cast<const uint4 *>(p.x) + row * NVr, SM::kRowBytes, bar);
        bulk_g2s(st + SM::kRowBytes, static_cast<const uint4 *>(p.dy) + row * NVr,
                 SM::kRowBytes, bar);
        if (has_gx)
            bulk_g2s(st + 2 * SM::kRowBytes, static_cast<const uint4 *>(p.gx) + row * NVr,
                     SM::kRowBytes, bar);
    };
    if (t == 0) {
        fence_proxy_async_smem();
        for (int64_t k = 0; k < NSE && k < nk; ++k)
            issue(k);
    }
    float r_next = 0.f;
    if constexpr (LOADR)
        r_next = nk > 0 ? p.rstd[gg] : 0.f;

    int64_t k = 0;
    bool failed = false;
    for (; k < nk; ++k) {
        const int64_t row = gg + k * TG;
        const uint32_t st = stage0 + (int)(k % NSE) * SM::kStageBytes;
        float r_cur = 0.f;
        if constexpr (LOADR) {
            r_cur = r_next;                 // loaded one row ahead
            if (k + 1 < nk)
                r_next = p.rstd[row + TG];
        }
        const bool ok = mbar_wait_bounded(bar0 + 8 * (int)(k % NSE), (uint32_t)((k / NSE) & 1), limit);

        // the row moves from the stage into registers, so the stage can be
        // refilled as soon as the group barrier below has passed
        X xa[V], dya[V], gxa[V];
        F s_c = splat<F>(0.f), s_a = splat<F>(0.f), s_b = splat<F>(0.f), s_d = splat<F>(0.f),
          s_xx = splat<F>(0.f);
#pragma unroll
        for (int j = 0; j < V; ++j) {
            X wv;
            as_pack<T>(lds128(st + (t + j * GT) * 16)).widen(xa[j]);
            as_pack<T>(lds128(st + SM::kRowBytes + (t + j * GT) * 16)).widen(dya[j]);
            if (has_gx)
                as_pack<T>(lds128(st + 2 * SM::kRowBytes + (t + j * GT) * 16)).widen(gxa[j]);
            else
                gxa[j] = X::zero();
            wp[j].widen(wv);
#pragma unroll
            for (int i = 0; i < X::N; ++i) {
                const F wdy = vmul(wv.v[i], dya[j].v[i]);
                s_c = vfma(wdy, xa[j].v[i], s_c);
                s_a = vfma(gxa[j].v[i], wdy, s_a);
                s_b = vfma(gxa[j].v[i], xa[j].v[i], s_b);
                s_d = vfma(vmul(gwv[j].v[i], dya[j].v[i]), xa[j].v[i], s_d);
                if constexpr (!LOADR)
                    s_xx = vfma(xa[j].v[i], xa[j].v[i], s_xx);
            }
        }
        // lane l holds the warp's total of sum (l >> 3) & 3: c, A, B, D
        const float tot = warp_sum4_spread(hsum(s_c), hsum(s_a), hsum(s_b), hsum(s_d));
        float *rb = red + (k & 1) * GW * NR;   // double buffer
        const int lane = t & 31;
        if ((lane & 7) == 0)
            rb[wg * NR + (lane >> 3)] = tot;
        if constexpr (!LOADR) {
            const float sxx = group_allreduce<32>(hsum(s_xx));
            if (lane == 0)
                rb[wg * NR + 4] = sxx;
        }
        // Every thread of the group has posted its sums and read this row's
        // stage (refilled below with the row NSE ahead); the slots of the
        // other buffer are free again.
        if (bar_red_or(1 + g, GT, !ok)) {
            failed = true;
            break;
        }
        if (t == 0 && k + NSE < nk) {
            fence_proxy_async_smem();
            issue(k + NSE);
        }
        // the warps' slots summed in warp order
        F cA = splat<F>(0.f), BD = splat<F>(0.f);
        float xx = 0.f;
#pragma unroll
        for (int q = 0; q < GW; ++q) {
            const float4 v = *reinterpret_cast<const float4 *>(rb + q * NR);
            cA = vadd(cA, make_float2(v.x, v.y));
            BD = vadd(BD, make_float2(v.z, v.w));
            if constexpr (!LOADR)
                xx += rb[q * NR + 4];
        }
        float r;
        if constexpr (LOADR)
            r = r_cur;
        else
            r = rsqrtf(xx / fH + p.eps);
        const float c = cA.x / fH;
        const float r3 = r * r * r;
        const float a2 = r3 * BD.x / fH;                                      // r^3 B / H
        const float a3 = r3 * c;                                              // r^3 c
        const float a1 = (r3 / fH) * (3.f * r * r * c * BD.x - cA.y - BD.y);
        const F r2 = splat<F>(r), A1 = splat<F>(a1), nA2 = splat<F>(-a2), nA3 = splat<F>(-a3);
#pragma unroll
        for (int j = 0; j < V; ++j) {
            X wv, o1, o2;
            wp[j].widen(wv);
#pragma unroll
            for (int i = 0; i < X::N; ++i) {
                // with u = r gx - a2 x and rgw = r gw:
                //   ddy = r w gx - a2 w x + r gw x    = w u + rgw x
                //   dx2 = a1 x - a2 w dy - a3 gx + r gw dy
                //       = a1 x - a3 gx + dy (rgw - a2 w)
                //   dw2 += r gx dy - a2 dy x          = dy u
                const F x = xa[j].v[i], dy = dya[j].v[i], gx = gxa[j].v[i];
                const F u = vfma(nA2, x, vmul(r2, gx));
                const F rgw = vmul(r2, gwv[j].v[i]);
                o1.v[i] = vfma(wv.v[i], u, vmul(rgw, x));
                o2.v[i] = vfma(dy, vfma(nA2, wv.v[i], rgw), vfma(nA3, gx, vmul(A1, x)));
                acc[j].v[i] = vfma(dy, u, acc[j].v[i]);
            }
            P::narrow(o1).store(p.ddy, row * NVr + t + j * GT);
            P::narrow(o2).store(p.dx2, row * NVr + t + j * GT);
        }
    }
    if (failed && t == 0) {
        atomicAdd(timeouts, 1u);
        // issued and not consumed: rows k .. k+NSE-1
        for (int64_t q = k; q < k + NSE && q < nk; ++q)
            (void)mbar_wait_bounded(bar0 + 8 * (int)(q % NSE), (uint32_t)((q / NSE) & 1), limit);
    }
    griddep_launch_dependents();

    // the NG groups' dw2 accumulators, in group order, into one partial row
    __syncthreads();
    float *comb = reinterpret_cast<float *>(smem);
#pragma unroll
    for (int j = 0; j < V; ++j) {
        float4 *d = reinterpret_cast<float4 *>(comb + (size_t)g * NV * 8 + (t + j * GT) * 8);
        d[0] = make_float4(acc[j].v[0].x, acc[j].v[0].y, acc[j].v[1].x, acc[j].v[1].y);
        d[1] = make_float4(acc[j].v[2].x, acc[j].v[2].y, acc[j].v[3].x, acc[j].v[3].y);
    }
    __syncthreads();
    float *part = p.part + (int64_t)blockIdx.x * p.H;
    for (int c = threadIdx.x; c < NV * 8; c += NG * GT) {
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < NG; ++q)
            v += comb[q * NV * 8 + c];
        part[c] = v;
    }
}

} // namespace rmsk
