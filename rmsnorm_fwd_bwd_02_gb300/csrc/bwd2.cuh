// bwd2.cuh -- double backward of the RMSNorm: given incoming gradients gx
// [M,H] on dx and gw [H] on dw, the gradients of sum(gx dx) + sum(gw dw)
// with respect to dy, x and w.
//
// [P1] "训推加速 Qwen3 实战：从“调包”到手写 Triton Kernel（含 backward）" §5.6
// asks an autograd wrapper to implement double backward or refuse it; the
// formulas come from differentiating the backward of §5.3 (dx = r w dy -
// r^3 c x, dw = sum dy x r) once more, with r a function of x. Per row, with
// c = (1/H) sum w dy x and the row sums A = sum gx w dy, B = sum gx x,
// D = sum gw dy x:
//   ddy = r w gx - (r^3 B / H) w x + r gw x
//   dx2 = (r^3 / H)(3 r^2 c B - A - D) x - (r^3 B / H) w dy - r^3 c gx + r gw dy
//   dw2 = sum over rows of r gx dy - (r^3 B / H) dy x
// The layout is that of the row-wise backward (rows.cuh) with one row per
// group: lanes of a group hold their packs of x, dy and gx in registers,
// the five row sums (and the sum of squares when rstd is not given) go
// through one group reduction, and the dw2 accumulators become one partial
// row per CTA, summed by dw_reduce in a fixed order.
#pragma once

#include "rows.cuh"

namespace rmsk {

template <typename T, int E, int L, int V, int S, int MINB, bool EXACT>
__global__ void __launch_bounds__(L * S, MINB)
rms_bwd2_rows(const Bwd2Params p)
{
    using P = Pack<T, E>;
    using X = Vals<E>;
    using F = typename X::F;
    using FP = Pack<float, E>;
    using Lay = RowLayout<E, L, V, 1, S>;
    constexpr int NW = Lay::kRowWarps;
    constexpr int NR = 5;                      // sum x^2, c, A, B, D
    constexpr int kComb = Lay::kColGroups > 1 ? Lay::kColGroups * Lay::kCols : 1;
    static_assert(kComb * 4 + 2 * NW * NR * 4 <= 48 * 1024, "static shared memory");
    __shared__ float red[2][NW * NR];
    __shared__ __align__(16) float comb[kComb];

    const int lane = threadIdx.x % L;
    const int grp = threadIdx.x / L;
    const int NV = p.H / E;
    const float fH = (float)p.H;
    const bool has_gx = p.gx != nullptr, has_gw = p.gw != nullptr;

    griddep_wait();
    LaneWeight<T, E, L, V, EXACT, Lay::kWideW> wt;
    wt.init(p.w, lane, NV);

    X acc[V];
#pragma unroll
    for (int k = 0; k < V; ++k)
        acc[k] = X::zero();

    auto gw_at = [&](int vi) {
        X g;
        if (has_gw)
            FP::load_cached(p.gw, vi).widen(g);
        else
            g = X::zero();
        return g;
    };

    const int64_t ntiles = (p.M + Lay::kTileRows - 1) / Lay::kTileRows;
    int buf = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int64_t row = t * Lay::kTileRows + grp;
        const bool rok = row < p.M;

        P xv[V], dyv[V], gv[V];
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int vi = lane + k * L;
            const bool ok = rok && (EXACT || vi < NV);
            xv[k] = ok ? P::load(p.x, row * NV + vi) : P::zero();
            dyv[k] = ok ? P::load(p.dy, row * NV + vi) : P::zero();
            gv[k] = (ok && has_gx) ? P::load(p.gx, row * NV + vi) : P::zero();
        }
        const float rs_given = (rok && p.rstd != nullptr) ? p.rstd[row] : 0.f;

        F s_xx = splat<F>(0.f), s_c = splat<F>(0.f), s_a = splat<F>(0.f), s_b = splat<F>(0.f),
          s_d = splat<F>(0.f);
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int vi = lane + k * L;
            X a, b, gg;
            xv[k].widen(a);
            dyv[k].widen(b);
            gv[k].widen(gg);
            const X w = wt.get(k);
            const X gwk = gw_at((EXACT || vi < NV) ? vi : 0);
#pragma unroll
            for (int i = 0; i < X::N; ++i) {
                const F wdy = vmul(w.v[i], b.v[i]);
                s_xx = vfma(a.v[i], a.v[i], s_xx);
                s_c = vfma(wdy, a.v[i], s_c);
                s_a = vfma(gg.v[i], wdy, s_a);
                s_b = vfma(gg.v[i], a.v[i], s_b);
                s_d = vfma(vmul(gwk.v[i], b.v[i]), a.v[i], s_d);
            }
        }
        float sums[NR] = {hsum(s_xx), hsum(s_c), hsum(s_a), hsum(s_b), hsum(s_d)};
        row_allreduce<L, NR>(sums, red[buf]);
        buf ^= 1;
        if (!rok)
            continue;                          // uniform over the group

        const float r = p.rstd != nullptr ? rs_given : rsqrtf(sums[0] / fH + p.eps);
        const float c = sums[1] / fH;
        const float r3 = r * r * r;
        const float a2 = r3 * sums[3] / fH;                                   // r^3 B / H
        const float a3 = r3 * c;                                              // r^3 c
        const float a1 = (r3 / fH) * (3.f * r * r * c * sums[3] - sums[2] - sums[4]);
        const F r2 = splat<F>(r), A1 = splat<F>(a1), nA2 = splat<F>(-a2), nA3 = splat<F>(-a3);
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int vi = lane + k * L;
            if (!(EXACT || vi < NV))
                continue;
            X a, b, gg, o1, o2;
            xv[k].widen(a);
            dyv[k].widen(b);
            gv[k].widen(gg);
            const X w = wt.get(k);
            const X gwk = gw_at(vi);
#pragma unroll
            for (int i = 0; i < X::N; ++i) {
                // with u = r gx - a2 x and rgw = r gw:
                //   ddy = r w gx - a2 w x + r gw x    = w u + rgw x
                //   dx2 = a1 x - a2 w dy - a3 gx + r gw dy
                //       = a1 x - a3 gx + dy (rgw - a2 w)
                //   dw2 += r gx dy - a2 dy x          = dy u
                const F u = vfma(nA2, a.v[i], vmul(r2, gg.v[i]));
                const F rgw = vmul(r2, gwk.v[i]);
                o1.v[i] = vfma(w.v[i], u, vmul(rgw, a.v[i]));
                o2.v[i] = vfma(b.v[i], vfma(nA2, w.v[i], rgw),
                               vfma(nA3, gg.v[i], vmul(A1, a.v[i])));
                acc[k].v[i] = vfma(b.v[i], u, acc[k].v[i]);
            }
            P::narrow(o1).store(p.ddy, row * NV + vi);
            P::narrow(o2).store(p.dx2, row * NV + vi);
        }
    }

    griddep_launch_dependents();
    write_dw_partials<E, L, V, S, EXACT>(acc, p.part + (int64_t)blockIdx.x * p.H, comb, p.H,
                                         lane, grp);
}

} // namespace rmsk
