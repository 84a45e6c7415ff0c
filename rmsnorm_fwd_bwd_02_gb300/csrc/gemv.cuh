// gemv.cuh -- RMSNorm fused with the projection that follows it in decode:
// out = round( round(RMSNorm(x) * w) A^T ) for a few rows x (M <= 64) and a
// row-major weight A of N rows of H (a linear layer's weight; q|k|v or
// gate|up stacked).
//
// [P2] (the 0.8B Qwen decode article, trdm.cn news/483216) §2.1 runs
// rms_norm and then the q/k/v (or gate/up) GEMVs as separate kernels, §3.1
// splits each GEMV's K = 896 over SPLIT_K programs plus a reduce kernel,
// and §6 names fusing the chain as the next step. Here the chain is one
// kernel, and its result is the chain's: the norm's output is rounded to
// the storage dtype before the product, as the separate rms_norm kernel
// would store it.
//
// Layout. CTA = 4 warps; it owns TN tiles of 8 consecutive rows of A.
//  1. Before waiting on the previous kernel it prefetches its rows of A into
//     L2 (L2 is the coherence point, so a prefetch never yields stale data).
//     After the wait it copies x (and r) rows and w into shared memory with
//     asynchronous copies issued all at once, then issues the first batch of
//     its A fragments, so the norm costs one memory round trip whatever M,
//     and the weight travels meanwhile. When the caller declares the weights
//     static (nothing in flight writes w or A), w and the first A batch are
//     fetched before the wait, overlapping the previous kernel entirely.
//  2. It computes the norm of all M rows from shared memory, in place (rows
//     are few; every CTA does the same fp32 arithmetic in the same order, so
//     all get the same bits) and keeps y, rounded, padded to whole 16-row
//     tiles (one 8-row tile when M <= 8; the MMA's rows 8..15 are then zero
//     registers). CTA 0 also writes h, y and rstd when they are wanted.
//     With every input but A read, it lets the next kernel be scheduled.
//  3. Each warp takes every fourth 32-wide chunk of K (the split of K that
//     [P2 §3.1] does across programs, done inside the CTA) and runs the
//     m16n8k16 tensor-core MMA with fp32 accumulation: lane (g = lane/4,
//     q = lane%4) loads 16 bytes of A row n0+g at k = 32c + 8q with one
//     instruction, and 16 bytes of y rows g and g+8 at the same k. The dot
//     product is a sum over k, so k may be permuted as long as both
//     operands use the same permutation: those 8 elements fill the k slots
//     {2q, 2q+1, 2q+8, 2q+9} of two consecutive MMAs.
//  4. The four warps' partial tiles are added in warp order through shared
//     memory (no atomics, reproducible) and rounded once into out.
//
// At decode sizes the kernel is bound by reading A from HBM (M flops per
// byte of A, M <= 64), so the warp-level MMA keeps the arithmetic far below
// the memory time.
#pragma once

#include "common.cuh"

namespace rmsk {

struct GemvParams {
    const void *x;    // [M,H]
    const void *r;    // [M,H] residual input, or unused
    const void *w;    // [H]
    const void *A;    // [N,H] row-major
    void *out;        // [M,N]
    void *h;          // [M,H] residual sum out, or nullptr
    void *y;          // [M,H] stored norm output, or nullptr
    float *rstd;      // [M] or nullptr
    int M, H, N;
    int TN;           // 8-row tiles of A per CTA (rms_gemv) or per warp (rms_gemv_tma)
    int ysr;          // shared-memory row stride of y in bytes
    float eps;
    int static_w;     // w and A are not written by work in flight before this
                      // kernel: they may be read before griddep_wait
    // rms_gemv_tma only: columns of A per ring stage, stages per warp, and
    // the test hook of the bounded waits (extra bytes a stage waits for,
    // wait limit in microseconds, 0 = about one second)
    int KS, NSW;
    uint32_t extra_tx, wait_limit_us;
};

// One m16n8k16 MMA, c += a b. Not volatile: it has no effect but its
// outputs, so the compiler may interleave independent MMAs and the shared
// loads that feed them.
template <typename T> struct MmaOp;

template <> struct MmaOp<bf16> {
    __device__ __forceinline__ static void run(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1)
    {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                     "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                     : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                     : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
};

template <> struct MmaOp<f16> {
    __device__ __forceinline__ static void run(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1)
    {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                     "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                     : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                     : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
};

__device__ __forceinline__ uint4 lds_v4(const unsigned char *p)
{
    return *reinterpret_cast<const uint4 *>(p);
}

constexpr int kGemvWarps = 4;
constexpr int kGemvBatch = 8;      // K chunks of A a lane holds in flight
constexpr int kGemvIlp = 8;        // independent packs per step of the norm
// Resident CTAs per SM the small-M (8-row) variants are built for: a
// register budget of 64 lets 8 CTAs share an SM, so the 8-row tiles of a
// wide projection (e.g. 1216 tiles for N = 9728) fit one wave on 152 SMs.
constexpr int kGemvHalfCtas = 8;

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)), "l"(gsrc)
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// Dynamic shared memory of one CTA, in this order: y (kYRows rows of ysr
// bytes; x is staged there and becomes h, then y, in place), r (M rows of
// 2H bytes, when staged), w (2H bytes), the four warps' partial tiles, the
// four warps' partial sums of squares.
__host__ __device__ constexpr int gemv_red_bytes(int MT) { return kGemvWarps * MT * 32 * 16; }
__host__ __device__ constexpr int gemv_y_rows(int MT, bool half) { return half ? 8 : MT * 16; }
__host__ __device__ constexpr int64_t gemv_smem_bytes(int MT, bool half, int M, int H,
                                                      bool stage_r)
{
    return (int64_t)gemv_y_rows(MT, half) * (2 * H + 64) + (stage_r ? (int64_t)M * 2 * H : 0) +
           2 * H + gemv_red_bytes(MT) + kGemvWarps * 4;
}

// MT: 16-row tiles of y (M <= 16 MT). HALF: M <= 8, y holds 8 rows and the
// MMA's rows 8..15 are zero registers. RES: residual add before the norm;
// STAGER: r staged in shared memory too (else read from L2 after a
// prefetch; for the largest M * H).
template <typename T, int MT, bool HALF, bool RES, bool STAGER>
__global__ void __launch_bounds__(kGemvWarps * 32, HALF ? kGemvHalfCtas : 1)
rms_gemv(const GemvParams p)
{
    using P = Pack<T, 8>;
    using X = Vals<8>;
    using F = float2;
    static_assert(!HALF || MT == 1, "the 8-row tile is one MMA tile");
    static_assert(RES || !STAGER, "r is staged only in the residual variant");
    constexpr int kYRows = gemv_y_rows(MT, HALF);
    extern __shared__ __align__(128) unsigned char smem[];
    const int rbytes = 2 * p.H;                                        // one row of T
    unsigned char *ys = smem;                                          // [kYRows][ysr]
    unsigned char *rsm = ys + kYRows * p.ysr;                          // [M][2H] if STAGER
    unsigned char *wsm = rsm + (STAGER ? p.M * rbytes : 0);            // [2H]
    float4 *red = reinterpret_cast<float4 *>(wsm + rbytes);            // [4][MT][32]
    float *part = reinterpret_cast<float *>(red + kGemvWarps * MT * 32);  // [4]

    const int tid = threadIdx.x;
    const int warp = tid / 32, lane = tid % 32;
    const int NP = p.H / 8;                  // 16-byte packs per row
    const int nchunks = p.H / 32;
    const int n_first = blockIdx.x * p.TN * 8;
    const int g = lane / 4, q = lane % 4;

    // 1. this CTA's rows of A (and an unstaged r) into L2 while the previous
    //    kernel finishes
    {
        const int n_end = min(p.N, n_first + p.TN * 8);
        if (n_end > n_first) {
            const char *a0 = static_cast<const char *>(p.A) + (size_t)n_first * p.H * sizeof(T);
            const size_t bytes = (size_t)(n_end - n_first) * p.H * sizeof(T);
            for (size_t off = (size_t)tid * 128; off < bytes; off += kGemvWarps * 32 * 128)
                prefetch_l2(a0 + off);
        }
        if constexpr (RES && !STAGER) {
            for (int off = tid * 128; off < p.M * rbytes; off += kGemvWarps * 32 * 128)
                prefetch_l2(static_cast<const char *>(p.r) + off);
        }
    }
    uint4 bf[kGemvBatch];
    auto load_batch = [&](int n0, int c0) {
        const int n = n0 + g;
        const bool nok = n < p.N;
        const uint4 *arow = reinterpret_cast<const uint4 *>(static_cast<const T *>(p.A) +
                                                            (size_t)(nok ? n : 0) * p.H);
#pragma unroll
        for (int b = 0; b < kGemvBatch; ++b) {
            const int ch = c0 + b * kGemvWarps;
            bf[b] = (nok && ch < nchunks) ? ld_row_v4(arow + ch * 4 + q) : make_uint4(0, 0, 0, 0);
        }
    };
    auto stage_w = [&]() {
        for (int j = tid; j < NP; j += kGemvWarps * 32)
            cp_async16(wsm + j * 16, static_cast<const uint4 *>(p.w) + j);
    };
    // Static weights: w and the first batch of A fragments are fetched while
    // the previous kernel still runs.
    if (p.static_w) {
        stage_w();
        if (n_first < p.N)
            load_batch(n_first, warp);
    }
    griddep_wait();

    // 2a. x (and r) rows and w into shared memory, all copies at once; then
    //     the first batch of A fragments, which travels meanwhile
    for (int e = tid; e < p.M * NP; e += kGemvWarps * 32) {
        const int m = e / NP, j = e - m * NP;
        cp_async16(ys + m * p.ysr + j * 16, static_cast<const uint4 *>(p.x) + e);
        if constexpr (STAGER)
            cp_async16(rsm + m * rbytes + j * 16, static_cast<const uint4 *>(p.r) + e);
    }
    if (!p.static_w)
        stage_w();
    for (int e = p.M * NP + tid; e < kYRows * NP; e += kGemvWarps * 32) {
        const int m = e / NP, j = e - m * NP;     // padding rows of y: zero
        *reinterpret_cast<uint4 *>(ys + m * p.ysr + j * 16) = make_uint4(0, 0, 0, 0);
    }

    if (!p.static_w && n_first < p.N)
        load_batch(n_first, warp);
    cp_async_wait_all();
    __syncthreads();

    // 2b. the norm of every row, from shared memory, in place: x -> h -> y.
    //     Rows run side by side: the CTA's threads form groups of TPR =
    //     128 / next_pow2(M) consecutive threads, group i owning row i, each
    //     thread every TPR-th pack of it. Sums: a butterfly over the group's
    //     lanes; a group wider than a warp (M <= 2) adds its warps' sums from
    //     shared memory in warp order.
    const bool writer = blockIdx.x == 0;
    int Mp = 1;
    while (Mp < p.M)
        Mp <<= 1;
    const int TPR = kGemvWarps * 32 / Mp;
    const int m = tid / TPR, sub = tid % TPR;
    const bool row_ok = m < p.M;
    unsigned char *yrow = ys + m * p.ysr;
    const int64_t rb = (int64_t)m * NP;
    F acc = splat<F>(0.f);
    // a thread's packs go in blocks of kGemvIlp independent iterations
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
                        rv.u = lds_v4(rsm + m * rbytes + j * 16);
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
        const int w0 = m * (TPR / 32);
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
                if (writer && p.y != nullptr)
                    yv.store(p.y, rb + j);
            }
        }
    }
    __syncthreads();
    // Every input but A is read: the next kernel may be scheduled and run up
    // to its own wait (its prefetch of its weights).
    griddep_launch_dependents();

    // 3./4. tiles of 8 rows of A
    for (int t = 0; t < p.TN; ++t) {
        const int n0 = n_first + t * 8;
        if (n0 >= p.N)
            break;                            // uniform over the CTA
        // two accumulators per m-tile, one per half of a 32-wide chunk, so
        // the two MMAs of a chunk do not wait on each other
        float c[MT][2][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
                c[mt][hh][0] = c[mt][hh][1] = c[mt][hh][2] = c[mt][hh][3] = 0.f;

        for (int c0 = warp; c0 < nchunks; c0 += kGemvWarps * kGemvBatch) {
            if (t > 0 || c0 != warp)
                load_batch(n0, c0);
#pragma unroll
            for (int b = 0; b < kGemvBatch; ++b) {
                const int ch = c0 + b * kGemvWarps;
                if (ch >= nchunks)
                    break;                    // uniform over the warp
                const int kb = (ch * 32 + q * 8) * (int)sizeof(T);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const uint4 ya = lds_v4(ys + (mt * 16 + g) * p.ysr + kb);
                    const uint4 yb = HALF ? make_uint4(0, 0, 0, 0)
                                          : lds_v4(ys + (mt * 16 + g + 8) * p.ysr + kb);
                    MmaOp<T>::run(c[mt][0], ya.x, yb.x, ya.y, yb.y, bf[b].x, bf[b].y);
                    MmaOp<T>::run(c[mt][1], ya.z, yb.z, ya.w, yb.w, bf[b].z, bf[b].w);
                }
            }
        }

#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
            red[(warp * MT + mt) * 32 + lane] =
                make_float4(c[mt][0][0] + c[mt][1][0], c[mt][0][1] + c[mt][1][1],
                            c[mt][0][2] + c[mt][1][2], c[mt][0][3] + c[mt][1][3]);
        __syncthreads();
        for (int e = tid; e < MT * 128; e += kGemvWarps * 32) {
            const int mt = e / 128, ln = (e % 128) / 4, i = e % 4;
            const int m = mt * 16 + ln / 4 + (i >= 2 ? 8 : 0);
            const int nn = n0 + 2 * (ln % 4) + (i & 1);
            if (m >= p.M || nn >= p.N)
                continue;
            float s = 0.f;
#pragma unroll
            for (int wv = 0; wv < kGemvWarps; ++wv) {
                const float4 v = red[(wv * MT + mt) * 32 + ln];
                s += i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
            }
            Vals<1> o;
            o.v[0] = s;
            Pack<T, 1>::narrow(o).store(p.out, (int64_t)m * p.N + nn);
        }
        __syncthreads();
    }
}

} // namespace rmsk
