// rows.cuh -- row-wise RMSNorm kernels: forward (optionally fused with the
// residual add) and backward (dx plus per-CTA partial dw rows).
//
// Sources: [P1] "训推加速 Qwen3 实战：从“调包”到手写 Triton Kernel（含 backward）"
// §4.1-4.2 (forward), §5.3-5.4 (backward); [P2] the 0.8B Qwen decode article
// (trdm.cn news/483216) §2.1 (residual add before the norm).
//
// Layout. A row is handled by a group of L lanes. Lane l of the group owns
// the packs l, l+L, ..., l+(V-1)L of the row (a pack = E elements moved by
// one memory instruction: 16 bytes for the vectorised kernels, one element
// for the scalar ones), so each memory instruction of a group covers L
// consecutive packs and the row stays in registers from load to store. A CTA
// holds S groups and walks tiles of S*G rows with a persistent grid-stride
// loop; every thread of a CTA runs the same number of iterations, rows past
// M are masked, so barriers and shuffles are always uniform.
//
// Arithmetic is fp32, two elements per FFMA2/FMUL2 instruction (Vals).
// Reductions: fp32 partials per lane, then a butterfly over the group's
// lanes (every lane ends with the same bits); groups wider than a warp add
// the per-warp sums from shared memory in warp order. The order is fixed, so
// results are reproducible run to run.
//
// dw. Every lane keeps fp32 accumulators for the columns it owns across all
// rows its CTA processes; at the end the CTA combines its groups in a fixed
// order and writes one partial row to the workspace. A second kernel
// (reduce.cuh) sums those rows in a fixed order ([P1 §5.4]: two passes, no
// atomics), with P = number of CTAs rows instead of M.
//
// Launch order. Every kernel is launched with programmatic stream
// serialization: it waits (griddep_wait) before its first global memory
// access until the previous kernel on the stream has completed, and lets the
// next kernel be scheduled once its own main loop is done.
#pragma once

#include "common.cuh"
#include "params.h"

// Tuning knob (measured on GB300): largest number of fp32 registers a lane
// spends on holding its weights widened.
#ifndef RMSK_WIDE_W_FLOATS
#define RMSK_WIDE_W_FLOATS 16
#endif

namespace rmsk {

template <int E, int L, int V, int G, int S>
struct RowLayout {
    static constexpr int kThreads = L * S;
    static constexpr int kRowWarps = L > 32 ? L / 32 : 1;
    static constexpr int kTileRows = S * G;
    static constexpr int kCols = L * V * E;
    // Column owners left after folding groups that share a warp.
    static constexpr int kColGroups = L < 32 ? kThreads / 32 : S;
    // Weight held widened to fp32 when that costs at most RMSK_WIDE_W_FLOATS
    // registers, else in its storage format (widened at each use).
    static constexpr bool kWideW = V * E <= RMSK_WIDE_W_FLOATS && E > 1;
    static_assert(kThreads % 32 == 0, "a CTA is whole warps");
    static_assert(L <= 32 ? (32 % L == 0) : (L % 32 == 0 && S == 1),
                  "a group is a power of two <= 32 lanes, or whole warps "
                  "with one group per CTA");
};

// Sum NR values over the L lanes of each row group; every lane of the group
// gets the same result. `red` is this iteration's [kRowWarps][NR] buffer.
template <int L, int NR>
__device__ __forceinline__ void row_allreduce(float (&v)[NR], float *red)
{
    if constexpr (L <= 32) {
#pragma unroll
        for (int i = 0; i < NR; ++i)
            v[i] = group_allreduce<L>(v[i]);
    } else {
        constexpr int NW = L / 32;
        const int warp = threadIdx.x / 32;
#pragma unroll
        for (int i = 0; i < NR; ++i)
            v[i] = group_allreduce<32>(v[i]);
        if ((threadIdx.x & 31) == 0) {
#pragma unroll
            for (int i = 0; i < NR; ++i)
                red[warp * NR + i] = v[i];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            float s = 0.f;
#pragma unroll
            for (int q = 0; q < NW; ++q)
                s += red[q * NR + i];
            v[i] = s;
        }
    }
}

// The weight of a lane's V packs: widened once, or kept packed, or (scalar
// kernels) re-read from L1 at each use.
template <typename T, int E, int L, int V, bool EXACT, bool WIDE>
struct LaneWeight {
    using P = Pack<T, E>;
    using X = Vals<E>;
    static constexpr bool kHold = E > 1;
    X wide[WIDE ? V : 1];
    P packed[(!WIDE && kHold) ? V : 1];
    const void *w;
    int lane, NV;

    __device__ __forceinline__ void init(const void *w_, int lane_, int NV_)
    {
        w = w_;
        lane = lane_;
        NV = NV_;
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int vi = lane + k * L;
            const bool ok = EXACT || vi < NV;
            if constexpr (WIDE) {
                if (ok)
                    P::load_cached(w, vi).widen(wide[k]);
                else
                    wide[k] = X::zero();
            } else if constexpr (kHold) {
                packed[k] = ok ? P::load_cached(w, vi) : P::zero();
            }
        }
    }
    __device__ __forceinline__ X get(int k) const
    {
        X r;
        if constexpr (WIDE) {
            r = wide[k];
        } else if constexpr (kHold) {
            packed[k].widen(r);
        } else {
            const int vi = lane + k * L;
            if (EXACT || vi < NV)
                P::load_cached(w, vi).widen(r);
            else
                r = X::zero();
        }
        return r;
    }
};

// ------------------------------------------------------------------ forward
template <typename T, int E, int L, int V, int G, int S, int MINB, bool EXACT, bool RES>
__global__ void __launch_bounds__(L * S, MINB)
rms_fwd_rows(const FwdParams p)
{
    using P = Pack<T, E>;
    using X = Vals<E>;
    using F = typename X::F;
    using Lay = RowLayout<E, L, V, G, S>;
    constexpr int NW = Lay::kRowWarps;
    // Two buffers: a warp can only reuse one after the barrier of the next
    // iteration, which every warp reaches only once it has read this one.
    __shared__ float red[2][NW * G];

    const int lane = threadIdx.x % L;
    const int grp = threadIdx.x / L;
    const int NV = p.H / E;                 // packs per row
    const float fH = (float)p.H;
    // row strides in packs (the host keeps strides below 2^31)
    const uint32_t sx = (uint32_t)p.ldx / E, sr = (uint32_t)p.ldr / E;
    const uint32_t sy = (uint32_t)p.ldy / E, sh = (uint32_t)p.ldh / E;

    griddep_wait();
    LaneWeight<T, E, L, V, EXACT, Lay::kWideW> wt;
    wt.init(p.w, lane, NV);

    const int64_t ntiles = (p.M + Lay::kTileRows - 1) / Lay::kTileRows;
    int buf = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int64_t row0 = t * Lay::kTileRows + (int64_t)grp * G;

        P xv[G][V];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int64_t row = row0 + g;
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const int vi = lane + k * L;
                const bool ok = row < p.M && (EXACT || vi < NV);
                xv[g][k] = ok ? P::load(p.x, row * sx + vi) : P::zero();
            }
        }
        if constexpr (RES) {
            P rv[G][V];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const int64_t row = row0 + g;
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    const int vi = lane + k * L;
                    const bool ok = row < p.M && (EXACT || vi < NV);
                    rv[g][k] = ok ? P::load(p.r, row * sr + vi) : P::zero();
                }
            }
            // h = round(x + r): the stored h is what the norm sees
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const int64_t row = row0 + g;
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    const int vi = lane + k * L;
                    X a, b;
                    xv[g][k].widen(a);
                    rv[g][k].widen(b);
#pragma unroll
                    for (int i = 0; i < X::N; ++i)
                        a.v[i] = vadd(a.v[i], b.v[i]);
                    xv[g][k] = P::narrow(a);
                    if (row < p.M && (EXACT || vi < NV))
                        xv[g][k].store(p.h, row * sh + vi);
                }
            }
        }

        float ss[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            F acc = splat<F>(0.f);
#pragma unroll
            for (int k = 0; k < V; ++k) {
                X a;
                xv[g][k].widen(a);
#pragma unroll
                for (int i = 0; i < X::N; ++i)
                    acc = vfma(a.v[i], a.v[i], acc);
            }
            ss[g] = hsum(acc);
        }
        row_allreduce<L, G>(ss, red[buf]);
        buf ^= 1;

#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int64_t row = row0 + g;
            if (row >= p.M)
                continue;
            const float r = rsqrtf(ss[g] / fH + p.eps);
            if (p.rstd != nullptr && lane == 0)
                p.rstd[row] = r;
            const F r2 = splat<F>(r);
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const int vi = lane + k * L;
                if (!(EXACT || vi < NV))
                    continue;
                X a;
                xv[g][k].widen(a);
                const X w = wt.get(k);
#pragma unroll
                for (int i = 0; i < X::N; ++i)
                    a.v[i] = vmul(vmul(a.v[i], r2), w.v[i]);
                P::narrow(a).store(p.y, row * sy + vi);
            }
        }
    }
    griddep_launch_dependents();
}

// ----------------------------------------------------------------- backward
// Store E fp32 values at dst (16-byte aligned when E is a multiple of 4).
template <int E>
__device__ __forceinline__ void store_vals(float *dst, const Vals<E> &v)
{
    if constexpr (E % 4 == 0) {
#pragma unroll
        for (int e = 0; e < E; e += 4)
            *reinterpret_cast<float4 *>(dst + e) =
                make_float4(v.get(e), v.get(e + 1), v.get(e + 2), v.get(e + 3));
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e)
            dst[e] = v.get(e);
    }
}

// The end of a backward CTA: the fp32 dw accumulators of the columns each
// lane owns, summed over the CTA's groups in a fixed order, become one
// partial row at `part` (H floats). Lanes of a warp that share columns
// (L < 32) fold first by butterfly; groups then meet in `comb` (shared
// memory, [kColGroups][kCols]) and are added in group order.
template <int E, int L, int V, int S, bool EXACT>
__device__ __forceinline__ void write_dw_partials(Vals<E> (&acc)[V], float *part, float *comb,
                                                  int H, int lane, int grp)
{
    using X = Vals<E>;
    using Lay = RowLayout<E, L, V, 1, S>;
    const int NV = H / E;
    if constexpr (Lay::kColGroups == 1) {
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int vi = lane + k * L;
            if (EXACT || vi < NV)
                store_vals<E>(part + (int64_t)vi * E, acc[k]);
        }
    } else {
        if constexpr (L < 32) {
            // lanes l, l+L, l+2L, ... of a warp own the same columns
#pragma unroll
            for (int k = 0; k < V; ++k)
#pragma unroll
                for (int i = 0; i < X::N; ++i)
#pragma unroll
                    for (int o = L; o < 32; o <<= 1) {
                        if constexpr (E % 2 == 0) {
                            acc[k].v[i].x += __shfl_xor_sync(0xFFFFFFFFu, acc[k].v[i].x, o);
                            acc[k].v[i].y += __shfl_xor_sync(0xFFFFFFFFu, acc[k].v[i].y, o);
                        } else {
                            acc[k].v[i] += __shfl_xor_sync(0xFFFFFFFFu, acc[k].v[i], o);
                        }
                    }
        }
        const int cg = L < 32 ? (int)(threadIdx.x / 32) : grp;
        if (L >= 32 || (threadIdx.x & 31) < L) {
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const int vi = lane + k * L;
                if (EXACT || vi < NV)
                    store_vals<E>(comb + cg * Lay::kCols + vi * E, acc[k]);
            }
        }
        __syncthreads();
        const int ncols = EXACT ? Lay::kCols : H;
        for (int c = threadIdx.x; c < ncols; c += Lay::kThreads) {
            float s = 0.f;
#pragma unroll
            for (int q = 0; q < Lay::kColGroups; ++q)
                s += comb[q * Lay::kCols + c];
            part[c] = s;
        }
    }
}

// LOADR: rstd is given (read it) instead of recomputed from x.
template <typename T, int E, int L, int V, int G, int S, int MINB, bool EXACT, bool DH,
          bool LOADR>
__global__ void __launch_bounds__(L * S, MINB)
rms_bwd_rows(const BwdParams p)
{
    using P = Pack<T, E>;
    using X = Vals<E>;
    using F = typename X::F;
    using Lay = RowLayout<E, L, V, G, S>;
    constexpr int NW = Lay::kRowWarps;
    constexpr int NR = LOADR ? G : 2 * G;      // values reduced per row group
    constexpr int kComb = Lay::kColGroups > 1 ? Lay::kColGroups * Lay::kCols : 1;
    static_assert(kComb * 4 + 2 * NW * NR * 4 <= 48 * 1024, "static shared memory");
    __shared__ float red[2][NW * NR];
    __shared__ __align__(16) float comb[kComb];

    const int lane = threadIdx.x % L;
    const int grp = threadIdx.x / L;
    const int NV = p.H / E;
    const float fH = (float)p.H;
    // row strides in packs (the host keeps strides below 2^31)
    const uint32_t sdy = (uint32_t)p.lddy / E, sx = (uint32_t)p.ldx / E;
    const uint32_t sdh = (uint32_t)p.lddh / E, sdx = (uint32_t)p.lddx / E;

    griddep_wait();
    LaneWeight<T, E, L, V, EXACT, Lay::kWideW> wt;
    wt.init(p.w, lane, NV);

    X acc[V];
#pragma unroll
    for (int k = 0; k < V; ++k)
        acc[k] = X::zero();

    const int64_t ntiles = (p.M + Lay::kTileRows - 1) / Lay::kTileRows;
    int buf = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int64_t row0 = t * Lay::kTileRows + (int64_t)grp * G;

        P xv[G][V], dyv[G][V];
        float rs[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int64_t row = row0 + g;
            if constexpr (LOADR)
                rs[g] = row < p.M ? p.rstd[row] : 0.f;
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const int vi = lane + k * L;
                const bool ok = row < p.M && (EXACT || vi < NV);
                xv[g][k] = ok ? P::load(p.x, row * sx + vi) : P::zero();
                dyv[g][k] = ok ? P::load(p.dy, row * sdy + vi) : P::zero();
            }
        }

        // [0, G): sum_j w_j dy_j x_j      [G, 2G): sum_j x_j^2 (recompute)
        float sums[NR];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            F cs = splat<F>(0.f), ss = splat<F>(0.f);
#pragma unroll
            for (int k = 0; k < V; ++k) {
                X a, b;
                xv[g][k].widen(a);
                dyv[g][k].widen(b);
                const X w = wt.get(k);
#pragma unroll
                for (int i = 0; i < X::N; ++i) {
                    cs = vfma(vmul(w.v[i], b.v[i]), a.v[i], cs);
                    if constexpr (!LOADR)
                        ss = vfma(a.v[i], a.v[i], ss);
                }
            }
            sums[g] = hsum(cs);
            if constexpr (!LOADR)
                sums[G + g] = hsum(ss);
        }
        row_allreduce<L, NR>(sums, red[buf]);
        buf ^= 1;

#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int64_t row = row0 + g;
            if (row >= p.M)
                continue;
            float r;
            if constexpr (LOADR)
                r = rs[g];
            else
                r = rsqrtf(sums[G + g] / fH + p.eps);
            const float c = sums[g] / fH;
            // dx = r (w dy - x r^2 c) = r (w dy) - x (r^3 c)
            const F r2 = splat<F>(r);
            const F negm = splat<F>(-(r * r * r * c));
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const int vi = lane + k * L;
                if (!(EXACT || vi < NV))
                    continue;
                X a, b, o;
                xv[g][k].widen(a);
                dyv[g][k].widen(b);
                const X w = wt.get(k);
#pragma unroll
                for (int i = 0; i < X::N; ++i) {
                    o.v[i] = vfma(a.v[i], negm, vmul(r2, vmul(w.v[i], b.v[i])));
                    acc[k].v[i] = vfma(vmul(b.v[i], a.v[i]), r2, acc[k].v[i]);
                }
                if constexpr (DH) {
                    X d;
                    P::load(p.dh, row * sdh + vi).widen(d);
#pragma unroll
                    for (int i = 0; i < X::N; ++i)
                        o.v[i] = vadd(o.v[i], d.v[i]);
                }
                P::narrow(o).store(p.dx, row * sdx + vi);
            }
        }
    }

    // The dw reduction kernel may be scheduled now; it waits for this grid
    // to finish before reading the partial rows.
    griddep_launch_dependents();

    write_dw_partials<E, L, V, S, EXACT>(acc, p.part + (int64_t)blockIdx.x * p.H, comb, p.H,
                                         lane, grp);
}

} // namespace rmsk
