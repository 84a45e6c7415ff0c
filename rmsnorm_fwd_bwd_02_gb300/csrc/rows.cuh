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
#pragma once

#include "common.cuh"
#include "params.h"

namespace rmsk {

template <int E, int L, int V, int G, int S>
struct RowLayout {
    static constexpr int kThreads = L * S;
    static constexpr int kRowWarps = L > 32 ? L / 32 : 1;
    static constexpr int kTileRows = S * G;
    static constexpr int kCols = L * V * E;
    // Column owners left after folding groups that share a warp.
    static constexpr int kColGroups = L < 32 ? kThreads / 32 : S;
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

// ------------------------------------------------------------------ forward
template <typename T, int E, int L, int V, int G, int S, int MINB, bool EXACT, bool RES>
__global__ void __launch_bounds__(L * S, MINB)
rms_fwd_rows(const FwdParams p)
{
    using P = Pack<T, E>;
    using Lay = RowLayout<E, L, V, G, S>;
    constexpr int NW = Lay::kRowWarps;
    // Two buffers: a warp can only reuse one after the barrier of the next
    // iteration, which every warp reaches only once it has read this one.
    __shared__ float red[2][NW * G];

    const int lane = threadIdx.x % L;
    const int grp = threadIdx.x / L;
    const int NV = p.H / E;                 // packs per row
    const float fH = (float)p.H;

    // The weight stays in registers in its storage format.
    P wp[V];
#pragma unroll
    for (int k = 0; k < V; ++k) {
        const int vi = lane + k * L;
        wp[k] = (EXACT || vi < NV) ? P::load_cached(p.w, vi) : P::zero();
    }

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
                xv[g][k] = ok ? P::load(p.x, row * NV + vi) : P::zero();
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
                    rv[g][k] = ok ? P::load(p.r, row * NV + vi) : P::zero();
                }
            }
            // h = round(x + r): the stored h is what the norm sees
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const int64_t row = row0 + g;
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    const int vi = lane + k * L;
                    float a[E], b[E];
                    xv[g][k].to_float(a);
                    rv[g][k].to_float(b);
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        a[e] += b[e];
                    xv[g][k] = P::from_float(a);
                    if (row < p.M && (EXACT || vi < NV))
                        xv[g][k].store(p.h, row * NV + vi);
                }
            }
        }

        float ss[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            ss[g] = 0.f;
#pragma unroll
            for (int k = 0; k < V; ++k) {
                float f[E];
                xv[g][k].to_float(f);
#pragma unroll
                for (int e = 0; e < E; ++e)
                    ss[g] = fmaf(f[e], f[e], ss[g]);
            }
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
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const int vi = lane + k * L;
                if (!(EXACT || vi < NV))
                    continue;
                float f[E], fw[E];
                xv[g][k].to_float(f);
                wp[k].to_float(fw);
#pragma unroll
                for (int e = 0; e < E; ++e)
                    f[e] = f[e] * r * fw[e];
                P::from_float(f).store(p.y, row * NV + vi);
            }
        }
    }
}

// ----------------------------------------------------------------- backward
// Store E fp32 values at dst (16-byte aligned when E is a multiple of 4).
template <int E>
__device__ __forceinline__ void store_f32(float *dst, const float (&v)[E])
{
    if constexpr (E % 4 == 0) {
#pragma unroll
        for (int e = 0; e < E; e += 4)
            *reinterpret_cast<float4 *>(dst + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e)
            dst[e] = v[e];
    }
}

template <typename T, int E, int L, int V, int G, int S, int MINB, bool EXACT, bool DH>
__global__ void __launch_bounds__(L * S, MINB)
rms_bwd_rows(const BwdParams p)
{
    using P = Pack<T, E>;
    using Lay = RowLayout<E, L, V, G, S>;
    constexpr int NW = Lay::kRowWarps;
    // The weight stays in registers in its storage format; the scalar
    // kernels re-read it from L1 instead.
    constexpr bool kWReg = E > 1;
    constexpr int kComb = Lay::kColGroups > 1 ? Lay::kColGroups * Lay::kCols : 1;
    static_assert(kComb * 4 + 2 * NW * 2 * G * 4 <= 48 * 1024, "static shared memory");
    __shared__ float red[2][NW * 2 * G];
    __shared__ __align__(16) float comb[kComb];

    const int lane = threadIdx.x % L;
    const int grp = threadIdx.x / L;
    const int NV = p.H / E;
    const float fH = (float)p.H;
    const bool have_rstd = p.rstd != nullptr;

    P wp[kWReg ? V : 1];
    if constexpr (kWReg) {
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int vi = lane + k * L;
            wp[k] = (EXACT || vi < NV) ? P::load_cached(p.w, vi) : P::zero();
        }
    }
    auto weight = [&](int k, float (&f)[E]) {
        if constexpr (kWReg) {
            wp[k].to_float(f);
        } else {
            const int vi = lane + k * L;
            if (EXACT || vi < NV) {
                P::load_cached(p.w, vi).to_float(f);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e)
                    f[e] = 0.f;
            }
        }
    };

    float acc[V][E];
#pragma unroll
    for (int k = 0; k < V; ++k)
#pragma unroll
        for (int e = 0; e < E; ++e)
            acc[k][e] = 0.f;

    const int64_t ntiles = (p.M + Lay::kTileRows - 1) / Lay::kTileRows;
    int buf = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int64_t row0 = t * Lay::kTileRows + (int64_t)grp * G;

        P xv[G][V], dyv[G][V];
        float rs[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int64_t row = row0 + g;
            rs[g] = (have_rstd && row < p.M) ? p.rstd[row] : 0.f;
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const int vi = lane + k * L;
                const bool ok = row < p.M && (EXACT || vi < NV);
                xv[g][k] = ok ? P::load(p.x, row * NV + vi) : P::zero();
                dyv[g][k] = ok ? P::load(p.dy, row * NV + vi) : P::zero();
            }
        }

        // [0, G): sum_j w_j dy_j x_j      [G, 2G): sum_j x_j^2
        float sums[2 * G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float cs = 0.f, ss = 0.f;
#pragma unroll
            for (int k = 0; k < V; ++k) {
                float fx[E], fdy[E], fw[E];
                xv[g][k].to_float(fx);
                dyv[g][k].to_float(fdy);
                weight(k, fw);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    cs = fmaf(fw[e] * fdy[e], fx[e], cs);
                    ss = fmaf(fx[e], fx[e], ss);
                }
            }
            sums[g] = cs;
            sums[G + g] = ss;
        }
        row_allreduce<L, 2 * G>(sums, red[buf]);
        buf ^= 1;

#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int64_t row = row0 + g;
            if (row >= p.M)
                continue;
            const float r = have_rstd ? rs[g] : rsqrtf(sums[G + g] / fH + p.eps);
            const float c = sums[g] / fH;
            const float coef = r * r * c;
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const int vi = lane + k * L;
                if (!(EXACT || vi < NV))
                    continue;
                float fx[E], fdy[E], fw[E], o[E];
                xv[g][k].to_float(fx);
                dyv[g][k].to_float(fdy);
                weight(k, fw);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    o[e] = r * (fw[e] * fdy[e] - fx[e] * coef);
                    acc[k][e] = fmaf(fdy[e] * fx[e], r, acc[k][e]);
                }
                if constexpr (DH) {
                    float fdh[E];
                    P::load(p.dh, row * NV + vi).to_float(fdh);
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        o[e] += fdh[e];
                }
                P::from_float(o).store(p.dx, row * NV + vi);
            }
        }
    }

    // The dw reduction kernel may be scheduled now; it waits for this grid
    // to finish before reading the partial rows.
    griddep_launch_dependents();

    float *part = p.part + (int64_t)blockIdx.x * p.H;
    if constexpr (Lay::kColGroups == 1) {
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int vi = lane + k * L;
            if (EXACT || vi < NV)
                store_f32<E>(part + (int64_t)vi * E, acc[k]);
        }
    } else {
        if constexpr (L < 32) {
            // lanes l, l+L, l+2L, ... of a warp own the same columns
#pragma unroll
            for (int k = 0; k < V; ++k)
#pragma unroll
                for (int e = 0; e < E; ++e)
#pragma unroll
                    for (int o = L; o < 32; o <<= 1)
                        acc[k][e] += __shfl_xor_sync(0xFFFFFFFFu, acc[k][e], o);
        }
        const int cg = L < 32 ? (int)(threadIdx.x / 32) : grp;
        if (L >= 32 || (threadIdx.x & 31) < L) {
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const int vi = lane + k * L;
                if (EXACT || vi < NV)
                    store_f32<E>(comb + cg * Lay::kCols + vi * E, acc[k]);
            }
        }
        __syncthreads();
        const int ncols = EXACT ? Lay::kCols : p.H;
        for (int c = threadIdx.x; c < ncols; c += Lay::kThreads) {
            float s = 0.f;
#pragma unroll
            for (int q = 0; q < Lay::kColGroups; ++q)
                s += comb[q * Lay::kCols + c];
            part[c] = s;
        }
    }
}

} // namespace rmsk
