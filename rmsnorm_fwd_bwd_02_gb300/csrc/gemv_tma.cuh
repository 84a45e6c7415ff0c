// gemv_tma.cuh -- RMSNorm fused with the projection GEMV, the weight fed by
// bulk asynchronous copies (the TMA engine) into per-warp shared-memory
// rings. Same result as rms_gemv (gemv.cuh): the chain of [P2] (the 0.8B
// Qwen decode article, trdm.cn news/483216) §2.1, §3.1, with y rounded to
// the dtype before out = y A^T, fp32 accumulation.
//
// Why a second kernel: with A held in registers (gemv.cuh) a CTA owns only
// one 8-row tile of A, so a wide projection needs many CTAs, and every CTA
// recomputes the norm of all M rows. Here a CTA has four warps, each owning
// whole 8-row tiles of A over all of K, and A reaches shared memory by bulk
// copies, so a few CTAs per SM keep the whole weight in flight and the norm
// is computed by few CTAs.
//
//  1. Lane 0 of each warp initialises the warp's ring of NSW stages (one
//     mbarrier each). A stage holds 8 rows x KS columns of A; a step of the
//     warp is one (tile, K slice), one 1-D bulk copy per row completing on
//     the stage's mbarrier. With static weights (nothing in flight writes w
//     or A) the first steps are issued before the wait on the previous
//     kernel, else right after it.
//  2. x (and r) rows and w reach shared memory by cp.async; the norm of all
//     rows is computed in place (row groups of threads, as in gemv.cuh).
//  3. Each warp walks its steps: a bounded wait on the stage's mbarrier,
//     then for each 32-wide K chunk one 16-byte shared load of A (row g,
//     k = 32c + 8q) and of y, and two m16n8k16 MMAs (k permuted the same way
//     on both operands, as in gemv.cuh); after the last K slice of a tile
//     the warp rounds and stores its outputs; the stage is refilled NSW
//     steps ahead once the warp has read it.
//  4. A wait that runs out (about one second, or the test limit) counts in
//     the device counter of streamed-kernel timeouts; the warp then waits,
//     bounded again, for its copies still in flight and stops.
//
// Many rows (CS > 1): the CTAs of a thread-block cluster of CS share the
// norm. Rank p stages, normalises and stores rows p, p + CS, ... and writes
// each finished y pack into its own shared memory and, through distributed
// shared memory, into every other CTA's of the cluster; one cluster barrier
// (release / acquire) then gives every CTA all of y. A first barrier phase,
// arrived at the start and waited on before the norm, makes sure every CTA
// of the cluster runs before its shared memory is written. Nothing touches
// another CTA's shared memory after the second barrier.

#pragma once

#include "gemv.cuh"
#include "split.cuh"
#include "stream.cuh"

namespace rmsk {

// 16 bytes into the shared memory of CTA `rank` of the cluster, at the
// offset `local` has in this CTA.
__device__ __forceinline__ void st_cluster_v4(const void *local, uint32_t rank, uint4 v)
{
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(local);
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(ra), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// CTAs of the cluster that share the norm when M > 16.
constexpr int kGemvCluster = 8;

// A ring stage: 8 rows of KS columns, each row padded by 64 bytes so that
// the rows a quarter-warp reads fall in different halves of the banks.
__host__ __device__ constexpr int gemv_tma_row_bytes(int KS) { return 2 * KS + 64; }
__host__ __device__ constexpr int gemv_tma_stage_bytes(int KS) { return 8 * gemv_tma_row_bytes(KS); }

// Bytes of the CTA's fixed shared memory (y, r, w, partial sums), then the
// rings, then the mbarriers.
// (With a cluster of CS, a CTA stages the r rows of its own (M + CS - 1) / CS
// rows only.)
__host__ __device__ constexpr int64_t gemv_tma_fixed_bytes(int MT, bool half, int M, int H,
                                                           bool stage_r, int CS)
{
    return (int64_t)gemv_y_rows(MT, half) * (2 * H + 64) +
           (stage_r ? (int64_t)((M + CS - 1) / CS) * 2 * H : 0) + 2 * H + 16;
}
__host__ __device__ constexpr int64_t gemv_tma_smem_bytes(int MT, bool half, int M, int H,
                                                          bool stage_r, int CS, int KS,
                                                          int NSW)
{
    return gemv_tma_fixed_bytes(MT, half, M, H, stage_r, CS) +
           (int64_t)kGemvWarps * NSW * gemv_tma_stage_bytes(KS) + kGemvWarps * NSW * 8;
}

template <typename T, int MT, bool HALF, bool RES, bool STAGER, int CS>
__global__ void __launch_bounds__(kGemvWarps * 32)
rms_gemv_tma(const GemvParams p, unsigned int *timeouts)
{
    using P = Pack<T, 8>;
    using X = Vals<8>;
    using F = float2;
    static_assert(!HALF || MT == 1, "the 8-row tile is one MMA tile");
    static_assert(RES || !STAGER, "r is staged only in the residual variant");
    constexpr int kYRows = gemv_y_rows(MT, HALF);
    extern __shared__ __align__(128) unsigned char smem[];
    const int rbytes = 2 * p.H;
    unsigned char *ys = smem;                                      // [kYRows][ysr]
    const uint32_t rank = CS > 1 ? cluster_ctarank() : 0;
    const int Mo = (p.M + CS - 1) / CS;                            // rows per rank
    unsigned char *rsm = ys + kYRows * p.ysr;                      // [Mo][2H] if STAGER
    unsigned char *wsm = rsm + (STAGER ? Mo * rbytes : 0);         // [2H]
    float *part = reinterpret_cast<float *>(wsm + rbytes);         // [4]
    const int stage_bytes = gemv_tma_stage_bytes(p.KS), asr = gemv_tma_row_bytes(p.KS);
    unsigned char *ring = reinterpret_cast<unsigned char *>(part + 4);   // [4][NSW][8][KS]
    const uint32_t bars = smem_addr(ring + kGemvWarps * p.NSW * stage_bytes);  // [4][NSW]

    const int tid = threadIdx.x;
    const int warp = tid / 32, lane = tid % 32;
    const int NP = p.H / 8;
    const int g = lane / 4, q = lane % 4;
    const int nslices = (p.H + p.KS - 1) / p.KS;

    // This warp's tiles: the CTA owns tiles [b 4 TPW, (b+1) 4 TPW); warp v
    // takes every fourth of them. Only tiles that start below N have steps.
    const int tile0 = blockIdx.x * kGemvWarps * p.TN + warp;
    int ntiles_w = 0;
    while (ntiles_w < p.TN && (tile0 + ntiles_w * kGemvWarps) * 8 < p.N)
        ++ntiles_w;
    const int steps = ntiles_w * nslices;
    unsigned char *myring = ring + warp * p.NSW * stage_bytes;
    const uint32_t mybar = bars + warp * p.NSW * 8;

    auto issue = [&](int step) {
        const int j = step / nslices, s = step - j * nslices;
        const int n0 = (tile0 + j * kGemvWarps) * 8;
        const int rows = min(8, p.N - n0);
        const int k0 = s * p.KS;
        const int kcols = min(p.KS, p.H - k0);
        const int st = step % p.NSW;
        const uint32_t bar = mybar + 8 * st;
        const uint32_t dst = smem_addr(myring + st * stage_bytes);
        mbar_expect_tx(bar, (uint32_t)(rows * kcols * 2) + p.extra_tx);
        for (int r = 0; r < rows; ++r)
            bulk_g2s(dst + r * asr,
                     static_cast<const T *>(p.A) + (size_t)(n0 + r) * p.H + k0,
                     (uint32_t)(kcols * 2), bar);
    };

    if (lane == 0)
        for (int s = 0; s < p.NSW; ++s)
            mbar_init(mybar + 8 * s, 1);
    mbar_init_fence();
    __syncwarp();
    // A CTA's shared memory may be written by its peers only once every CTA
    // of the cluster runs: arrive now, wait before the first such write.
    if constexpr (CS > 1)
        cluster_arrive_release();
    auto prologue = [&]() {
        if (lane == 0) {
            fence_proxy_async_smem();
            for (int k = 0; k < p.NSW && k < steps; ++k)
                issue(k);
        }
        __syncwarp();
    };
    if (p.static_w) {
        prologue();
        for (int j = tid; j < NP; j += kGemvWarps * 32)
            cp_async16(wsm + j * 16, static_cast<const uint4 *>(p.w) + j);
    }
    griddep_wait();
    if (!p.static_w) {
        prologue();
        for (int j = tid; j < NP; j += kGemvWarps * 32)
            cp_async16(wsm + j * 16, static_cast<const uint4 *>(p.w) + j);
    }

    // 2. x (and r) of this CTA's rows into shared memory; the norm of every
    //    row, in place (row i of this rank is row rank + i CS)
    for (int e = tid; e < Mo * NP; e += kGemvWarps * 32) {
        const int i = e / NP, j = e - i * NP;
        const int m = (int)rank + i * CS;
        if (m >= p.M)
            continue;
        const int64_t src = (int64_t)m * NP + j;
        cp_async16(ys + m * p.ysr + j * 16, static_cast<const uint4 *>(p.x) + src);
        if constexpr (STAGER)
            cp_async16(rsm + i * rbytes + j * 16, static_cast<const uint4 *>(p.r) + src);
    }
    for (int e = p.M * NP + tid; e < kYRows * NP; e += kGemvWarps * 32) {
        const int m = e / NP, j = e - m * NP;     // padding rows of y: zero
        *reinterpret_cast<uint4 *>(ys + m * p.ysr + j * 16) = make_uint4(0, 0, 0, 0);
    }
    if constexpr (RES && !STAGER) {
        for (int off = tid * 128; off < p.M * rbytes; off += kGemvWarps * 32 * 128)
            prefetch_l2(static_cast<const char *>(p.r) + off);
    }
    cp_async_wait_all();
    __syncthreads();

    if constexpr (CS > 1)
        cluster_wait_acquire();
    // the first cluster (or CTA) writes h, y and rstd of the rows it owns
    const bool writer = blockIdx.x < CS;
    int Mp = 1;
    while (Mp < Mo)
        Mp <<= 1;
    const int TPR = kGemvWarps * 32 / Mp;
    const int i_own = tid / TPR, sub = tid % TPR;
    const int m = (int)rank + i_own * CS;
    const bool row_ok = i_own < Mo && m < p.M;
    unsigned char *yrow = ys + m * p.ysr;
    const int64_t rb = (int64_t)m * NP;
    F acc = splat<F>(0.f);
    if (row_ok) {
        for (int j0 = sub; j0 < NP; j0 += kGemvIlp * TPR) {
#pragma unroll
            for (int u = 0; u < kGemvIlp; ++u) {
                const int j = j0 + u * TPR;
                if (j >= NP)
                    break;
                P xv;
                xv.u = lds_v4(yrow + j * 16);
                X a;
                if constexpr (RES) {
                    X b;
                    xv.widen(a);
                    if constexpr (STAGER) {
                        P rv;
                        rv.u = lds_v4(rsm + i_own * rbytes + j * 16);
                        rv.widen(b);
                    } else {
                        P::load_cached(p.r, rb + j).widen(b);
                    }
#pragma unroll
                    for (int i = 0; i < X::N; ++i)
                        a.v[i] = vadd(a.v[i], b.v[i]);
                    xv = P::narrow(a);           // h as stored
                    *reinterpret_cast<uint4 *>(yrow + j * 16) = xv.u;
                    if (writer && p.h != nullptr)
                        xv.store(p.h, rb + j);
                }
                xv.widen(a);
#pragma unroll
                for (int i = 0; i < X::N; ++i)
                    acc = vfma(a.v[i], a.v[i], acc);
            }
        }
    }
    float ss = hsum(acc);
    for (int o = (TPR < 32 ? TPR : 32) / 2; o > 0; o >>= 1)
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if (TPR > 32) {                           // uniform: M <= 2
        if (lane == 0)
            part[warp] = ss;
        __syncthreads();
        const int w0 = i_own * (TPR / 32);
        ss = 0.f;
        for (int v = 0; v < TPR / 32; ++v)
            ss += part[w0 + v];
    }
    if (row_ok) {
        const float rs = rsqrtf(ss / (float)p.H + p.eps);
        if (writer && sub == 0 && p.rstd != nullptr)
            p.rstd[m] = rs;
        const F r2 = splat<F>(rs);
        for (int j0 = sub; j0 < NP; j0 += kGemvIlp * TPR) {
#pragma unroll
            for (int u = 0; u < kGemvIlp; ++u) {
                const int j = j0 + u * TPR;
                if (j >= NP)
                    break;
                P hv, wp;
                hv.u = lds_v4(yrow + j * 16);
                wp.u = lds_v4(wsm + j * 16);
                X a, wv;
                hv.widen(a);
                wp.widen(wv);
#pragma unroll
                for (int i = 0; i < X::N; ++i)
                    a.v[i] = vmul(vmul(a.v[i], r2), wv.v[i]);
                const P yv = P::narrow(a);
                *reinterpret_cast<uint4 *>(yrow + j * 16) = yv.u;
                if constexpr (CS > 1) {
#pragma unroll
                    for (int d = 1; d < CS; ++d)
                        st_cluster_v4(yrow + j * 16, (rank + d) % CS, yv.u);
                }
                if (writer && p.y != nullptr)
                    yv.store(p.y, rb + j);
            }
        }
    }
    if constexpr (CS > 1) {
        // every CTA of the cluster has written its rows everywhere
        cluster_arrive_release();
        cluster_wait_acquire();
    } else {
        __syncthreads();
    }
    // every input but A is read: the next kernel may be scheduled
    griddep_launch_dependents();

    // 3. the warp's tiles, step by step through its ring
    const unsigned long long limit = wait_limit_ns(p.wait_limit_us);
    // two accumulators per m-tile, one per half of a 32-wide chunk, so the
    // two MMAs of a chunk do not wait on each other
    float c[MT][2][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
            c[mt][hh][0] = c[mt][hh][1] = c[mt][hh][2] = c[mt][hh][3] = 0.f;
    int k = 0;
    bool failed = false;
    for (; k < steps; ++k) {
        const int st = k % p.NSW;
        const bool ok = mbar_wait_bounded(mybar + 8 * st, (uint32_t)((k / p.NSW) & 1), limit);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
            failed = true;
            break;
        }
        const int j = k / nslices, s = k - j * nslices;
        const int k0 = s * p.KS;
        const int kcols = min(p.KS, p.H - k0);
        const unsigned char *stg = myring + st * stage_bytes + g * asr;
#pragma unroll 2
        for (int ch = 0; ch < kcols / 32; ++ch) {
            const uint4 bv = lds_v4(stg + (ch * 32 + q * 8) * 2);
            const int kb = (k0 + ch * 32 + q * 8) * 2;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const uint4 ya = lds_v4(ys + (mt * 16 + g) * p.ysr + kb);
                const uint4 yb = HALF ? make_uint4(0, 0, 0, 0)
                                      : lds_v4(ys + (mt * 16 + g + 8) * p.ysr + kb);
                MmaOp<T>::run(c[mt][0], ya.x, yb.x, ya.y, yb.y, bv.x, bv.y);
                MmaOp<T>::run(c[mt][1], ya.z, yb.z, ya.w, yb.w, bv.z, bv.w);
            }
        }
        // the warp is done reading this stage: refill it NSW steps ahead
        __syncwarp();
        if (lane == 0 && k + p.NSW < steps) {
            fence_proxy_async_smem();
            issue(k + p.NSW);
        }
        if (s == nslices - 1) {                   // the tile is complete
            const int n0 = (tile0 + j * kGemvWarps) * 8;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int mm = mt * 16 + g + (i >= 2 ? 8 : 0);
                    const int nn = n0 + 2 * q + (i & 1);
                    if (mm < p.M && nn < p.N) {
                        Vals<1> o;
                        o.v[0] = c[mt][0][i] + c[mt][1][i];
                        Pack<T, 1>::narrow(o).store(p.out, (int64_t)mm * p.N + nn);
                    }
                    c[mt][0][i] = c[mt][1][i] = 0.f;
                }
            }
        }
    }
    // 4. a wait ran out: record it and let the copies in flight land
    if (failed && lane == 0) {
        atomicAdd(timeouts, 1u);
        for (int qq = k; qq < k + p.NSW && qq < steps; ++qq)
            (void)mbar_wait_bounded(mybar + 8 * (qq % p.NSW), (uint32_t)((qq / p.NSW) & 1),
                                    limit);
    }
}

} // namespace rmsk
