// gemv_tc.cuh -- RMSNorm fused with the projection, persistent, the product
// on tcgen05 with four accumulators in tensor memory, K optionally split over
// a thread-block cluster. Same result as the other projection kernels: the
// chain of [P2] (the 0.8B Qwen decode article, trdm.cn news/483216) §2.1,
// §3.1 with y rounded to the dtype before out = y A^T, fp32 accumulation.
//
// A cluster of KS CTAs (KS = 1 to 8; one CTA per SM) normalises a
// decode batch once: CTA `rank` owns the 64-column atoms
// [rank na / KS, (rank + 1) na / KS) of the rows and keeps its slice of y
// (T tokens, T = M rounded up to 16) in shared memory. The cluster then
// takes the 128-feature tiles c, c + C, ... of A (c its index, C the
// clusters launched); each CTA streams its K slice of those tiles through
// one ring that runs on across tile boundaries, so the weight keeps
// flowing while tiles are finished. Splitting K keeps each CTA's y slice
// small and its ring deep (many bytes of A in flight per SM); the price is
// an exchange of partial products per tile.
//
// Roles (512 threads, 16 warps):
//  - warp 0, lane 0: the copies of A. Stage q of the ring (APS atoms of 128
//    features x 64 columns, 16 KB each, 128-byte swizzle) waits until the
//    MMAs that read its previous contents are complete (the `empty`
//    barrier, committed by the MMA thread), then is refilled, completing on
//    its `full` barrier. With static weights one stage starts before the
//    wait on the previous kernel and the rest once x's copies are issued
//    (an SM serves its tensor copies in order).
//  - warps 1-15 first normalise, all 480 threads: x arrives by tensor copies
//    (T x 64 per atom, rows past M and columns past H read as zero) into the
//    y area in the MMA's K-major layout; h = x + r (r read from global, a
//    batch of loads in flight per thread) is rounded and stored in place;
//    sums of h^2 per (4 tokens, atom) unit, reduced over the eight lanes
//    holding a row's chunks, then over the CTA's atoms in atom order; with
//    a cluster, each CTA stores its sums into every peer (asynchronous
//    stores counted on the peer's `sums` barrier, so no fence is waited
//    for) and, once all peers' sums have landed, adds the cluster's sums in
//    rank order; rstd; y = h rstd w in place. The first cluster stores h
//    and y (each CTA its columns), its rank 0 rstd.
//  - warp 1, lane 0 then issues the MMAs: per tile, into accumulator
//    (tile % 4), once the epilogue has released it; per stage, four MMAs
//    (m128 nT k16) an atom and one commit to the stage's `empty` barrier;
//    per tile one commit to the accumulator's `full` barrier.
//  - warps 4-11: the epilogue. Warp w reads lanes 32 (w % 4) .. + 31 of the
//    accumulator (features) for tokens 16 ((w - 4) / 4) + 32 j
//    (tcgen05.ld) and releases it. Without a cluster it rounds and stores
//    out[token][feature]. With one, feature f of the tile belongs to rank
//    f / ceil(128 / KS): a lane keeps its own features' partial sums in
//    registers and stores the others straight into the owner's receive
//    slot for this CTA (asynchronous 16-byte stores into distributed
//    shared memory, counted on the owner's `rx full` barrier; at 64
//    tokens it writes them into a send block per owner instead, which one
//    thread moves with one bulk copy); the owner adds the KS partials in
//    rank order, rounds and stores. Flow control per tile: an owner re-arms
//    its `rx full` barrier for the next tile and then releases its receive
//    slots by a remote arrival on each peer's `rx free` barrier, which a
//    sender waits for before its next stores or copies.
// So the MMAs of tiles j + 1 .. j + 3 run while the epilogue drains and
// exchanges tile j, and the copies of A run ahead of both.
//
// Every wait is bounded (about one second, or the test limit). One that
// runs out raises a flag in shared memory that every other wait also
// watches, so all roles stop; peers whose waits then run out stop too. The
// CTA waits (bounded) for its copies in flight, the MMAs and any partial
// products or sums still landing in it, counts one timeout, meets its peers
// at the final cluster barrier, frees the tensor memory and ends.
#pragma once

#include <cuda.h>

#include "gemv_umma.cuh"

namespace rmsk {

constexpr int kTcThreads = 512;
constexpr int kTcNormWarps = 15;              // warps 1..15
constexpr int kTcEpiWarp0 = 4, kTcEpiWarps = 8;
constexpr int kTcBatch = 8;                   // norm units whose r loads are in flight at once
constexpr int kTcMaxCluster = 8;
constexpr uint32_t kTcAtom = kUmmaAtomA;      // 128 x 64 of A: 16 KB
constexpr int kTcAcc = 4;                     // accumulators in tensor memory, used in turn

// Shared memory of one CTA, byte offsets from a 1024-byte aligned base: its
// slice of y (apc atoms of T x 128 bytes), the ring (NSt stages of APS
// atoms), its slice of w (apc x 128 bytes, zero past H), with a cluster the
// exchange blocks (receive: one slot per rank; send: one block per rank,
// used at 64 tokens and, at its start, for the cluster's sums of squares
// [KS][T]; the own ones unused; a block = ceil(128 / KS) features x xrow
// floats), the
// mbarriers (full[NSt], empty[NSt], acc_full[4], acc_empty[4], x landed,
// drain, x issued, sums published, rx full, rx free), eight words
// (tensor-memory address, failure flag, copies issued, copies consumed,
// partial products still expected), rstd[T], the CTA's sums of squares [T]
// and the per-atom partial sums [apc][T].
struct TcLayout {
    int NSt, APS, KS, apc, xrow;
    uint32_t ring, w, xch, xblock, bar, slots, total;   // total includes 1023 bytes of alignment
};

__host__ __device__ inline TcLayout gemv_tc_layout(int T, int H, int KS, int NSt, int APS)
{
    TcLayout L;
    const int na = (H + kUmmaKC - 1) / kUmmaKC;
    L.NSt = NSt;
    L.APS = APS;
    L.KS = KS;
    L.apc = (na + KS - 1) / KS;
    L.xrow = T + 4;                                        // conflict-free float4 rows
    L.ring = (uint32_t)L.apc * (uint32_t)T * 128u;
    L.w = L.ring + (uint32_t)NSt * (uint32_t)APS * kTcAtom;
    L.xch = L.w + (uint32_t)L.apc * 128u;
    L.xblock = (uint32_t)((kUmmaM + KS - 1) / KS) * (uint32_t)L.xrow * 4u;
    const uint32_t xbytes = KS > 1 ? 2u * (uint32_t)KS * L.xblock : 0u;
    L.bar = L.xch + xbytes;
    L.slots = L.bar + 8u * (uint32_t)(2 * NSt + 2 * kTcAcc + 6);
    L.total = L.slots + 32u + 8u * (uint32_t)T + 4u * (uint32_t)L.apc * (uint32_t)T + 1023u;
    return L;
}

struct GemvTcParams {
    const void *r;    // [M,H] residual, or nullptr
    const void *w;    // [H]
    void *out;        // [M,N]
    void *h;          // [M,H] residual sum out, or nullptr
    void *y;          // [M,H] stored norm output, or nullptr
    float *rstd;      // [M] or nullptr
    int M, H, N;
    int T;            // tokens as the MMA's N: M rounded up to 16 (<= 64)
    int na;           // atoms of K in a row: ceil(H / 64)
    TcLayout L;
    float eps;
    int static_w;     // w and A may be read before the wait on the previous kernel
    uint32_t extra_tx, wait_limit_us;   // test hook of the bounded waits (A's copies)
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrive on a peer's mbarrier with the default (CTA-scope) release: for
// handing back receive slots, where no data has to become visible to the
// peer. The slots' readers are done (their values were consumed before the
// named barrier that precedes this arrival) and the peer writes the slots
// again only by bulk copies it starts after observing the arrival. A
// release at cluster scope would also wait for this thread's outstanding
// memory traffic, which under the stream of A held an epilogue warp for
// microseconds per tile.
__device__ __forceinline__ void mbar_arrive_remote_cta(uint32_t cluster_bar)
{
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// Bounded wait that also gives up when another role has raised `fail`; a
// wait that runs out raises it. CLUSTER: acquire at cluster scope (for
// barriers that peers arrive on).
template <bool CLUSTER = false>
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, unsigned long long limit,
                                        volatile int *fail)
{
    auto test = [&]() {
        return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (test())
        return true;
    const unsigned long long t0 = global_ns();
    while (!test()) {
        if (*fail)
            return false;
        if (global_ns() - t0 > limit) {
            *fail = 1;
            return false;
        }
    }
    return true;
}

// grid = (clusters launched) x KS CTAs, cluster (KS, 1, 1) when KS > 1, 512
// threads, dynamic shared memory p.L.total.
// DIRECT: the partial products go to their owners by asynchronous stores
// (the host picks it up to 48 tokens), else by a send block and one bulk
// copy per owner.
template <typename T, bool RES, bool DIRECT>
__global__ void __launch_bounds__(kTcThreads, 1)
rms_gemv_tc(const GemvTcParams p, const __grid_constant__ CUtensorMap tmA,
            const __grid_constant__ CUtensorMap tmX, unsigned int *timeouts)
{
    using P = Pack<T, 8>;
    using X = Vals<8>;
    using F = float2;
    extern __shared__ __align__(1024) unsigned char tc_smem[];

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int H = p.H, NT = p.T, NP = H / 8, na = p.na;
    const TcLayout &L = p.L;
    const int NSt = L.NSt, APS = L.APS, KS = L.KS;
    const int rank = KS > 1 ? (int)cluster_ctarank() : 0;
    const int a0 = rank * na / KS;                            // this CTA's atoms of K
    const int nat = (rank + 1) * na / KS - a0;
    const int cid = (int)blockIdx.x / KS, ncl = (int)gridDim.x / KS;
    const uint32_t raw_s = smem_addr(tc_smem);
    unsigned char *base = tc_smem + (((raw_s + 1023u) & ~1023u) - raw_s);
    unsigned char *ysm = base, *wsm = base + L.w;
    const uint32_t y_s = smem_addr(ysm), ring_s = smem_addr(base + L.ring);
    unsigned char *recv = base + L.xch;                       // [KS] slots
    unsigned char *send = base + L.xch + (uint32_t)KS * L.xblock;
    const uint32_t recv_s = smem_addr(recv);
    const uint32_t full0 = smem_addr(base + L.bar), empty0 = full0 + 8u * (uint32_t)NSt;
    const uint32_t accf0 = empty0 + 8u * (uint32_t)NSt, acce0 = accf0 + 8u * kTcAcc;
    const uint32_t xbar = acce0 + 8u * kTcAcc, dbar = xbar + 8u, xiss = dbar + 8u;
    const uint32_t pready = xiss + 8u, rxfull = pready + 8u, rxfree = rxfull + 8u;
    int *slots = reinterpret_cast<int *>(base + L.slots);
    volatile int *fail = slots + 1;
    // slots[0]: tensor-memory address, [1]: a wait ran out, [2]: stages
    // issued, [3]: stages whose copies were consumed, [4]: phases of
    // partial products still expected
    float *rsv = reinterpret_cast<float *>(slots + 8);        // [T] rstd
    float *csum = rsv + NT;                                   // [T] this CTA's sums of h^2
    float *part = csum + NT;                                  // [apc][T] per atom
    const float *psum = reinterpret_cast<const float *>(send); // [KS][T] the cluster's sums
    const uint32_t atom = (uint32_t)NT * 128u;                // bytes of an atom of y
    const uint32_t ncols = gemv_umma_tmem_cols(NT);           // one accumulator
    const uint32_t stage = (uint32_t)APS * kTcAtom;
    const unsigned long long limit = wait_limit_ns(p.wait_limit_us);
    const int ntiles = (p.N + kUmmaM - 1) / kUmmaM;
    const int mt = cid < ntiles ? (ntiles - 1 - cid) / ncl + 1 : 0;
    const int ng = (nat + APS - 1) / APS;                     // stages per tile
    const int nq = mt * ng;                                   // stages of this CTA
    const bool writer = cid == 0;                             // stores h, y (and rstd)
    const int fpo = (kUmmaM + KS - 1) / KS;                   // features per owner (the last
                                                              // owner may hold fewer)
    // The partial products reach their owners by asynchronous 16-byte stores
    // straight from registers (DIRECT, up to 48 tokens); at 64 the stores'
    // count (four times that at 16 tokens) costs more than staging each
    // owner's block in shared memory and moving it with one bulk copy.
    constexpr bool direct = DIRECT;
    // expected per tile: every peer's partials of this CTA's features (T
    // tokens each when stored directly, whole slots when copied)
    const int nown = max(0, min(fpo, kUmmaM - rank * fpo));
    const uint32_t rx_bytes = direct ? (uint32_t)(KS - 1) * (uint32_t)nown * (uint32_t)NT * 4u
                                     : (uint32_t)(KS - 1) * L.xblock;

    // set-up: tensor memory (all accumulators), the barriers, the maps
    if (warp == 0) {
        tmem_alloc(smem_addr(slots), (uint32_t)kTcAcc * ncols);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int s = 0; s < NSt; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, 1);
        }
        for (int b = 0; b < kTcAcc; ++b) {
            mbar_init(accf0 + 8u * b, 1);
            mbar_init(acce0 + 8u * b, kTcEpiWarps);
        }
        mbar_init(xbar, 1);
        mbar_init(dbar, 1);
        mbar_init(xiss, 1);
        slots[4] = 0;
        if (KS > 1) {
            // the peers' sums of squares: (KS - 1) T words stored into this
            // CTA by the peers
            mbar_init(pready, 1);
            mbar_expect_tx(pready, (uint32_t)(KS - 1) * (uint32_t)NT * 4u);
            mbar_init(rxfull, 1);
            mbar_init(rxfree, (uint32_t)(KS - 1));
            if (mt > 0) {                       // the first tile's partial products
                mbar_expect_tx(rxfull, rx_bytes);
                slots[4] = 1;
            }
        }
        slots[1] = 0;
        slots[2] = 0;
        slots[3] = 0;
    }
    if (tid == 64) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmX);
    }
    mbar_init_fence();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (KS > 1) {               // every peer's barriers exist before any remote use
        cluster_arrive_release();
        cluster_wait_acquire();
    }
    const uint32_t tmem = static_cast<uint32_t>(slots[0]);
    int rx_done = 0;            // phases of partial products received (epilogue thread 0)

    if (warp == 0) {
        // ---------------------------------------------------- copies of A
        if (lane == 0) {
            if (!p.static_w)
                griddep_wait();
            int q = 0;
            for (; q < nq; ++q) {
                const int s = q % NSt, u = q / NSt;
                if (q == (p.static_w ? 1 : 0) && !tc_wait(xiss, 0, limit, fail))
                    break;
                if (u > 0 && !tc_wait(empty0 + 8u * s, (uint32_t)((u - 1) & 1), limit, fail))
                    break;
                if (*fail)
                    break;
                const int jt = q / ng, g = q % ng;
                const int f0 = (cid + jt * ncl) * kUmmaM;
                const int alo = g * APS, ahi = min(nat, alo + APS);
                const uint32_t bar = full0 + 8u * s;
                mbar_expect_tx(bar, (uint32_t)(ahi - alo) * (kTcAtom + p.extra_tx));
                for (int a = alo; a < ahi; ++a)
                    tma_load_2d(ring_s + (uint32_t)s * stage + (uint32_t)(a - alo) * kTcAtom, &tmA,
                                (a0 + a) * kUmmaKC, f0, bar);
                slots[2] = q + 1;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- the norm
        griddep_wait();
        const int nw = warp - 1;                              // 0..14
        if (warp == 1) {            // x: lane i copies atoms i, i + 32, ...
            if (lane == 0)
                mbar_expect_tx(xbar, atom * (uint32_t)nat);
            __syncwarp();
            for (int a = lane; a < nat; a += 32)
                tma_load_2d(y_s + (uint32_t)a * atom, &tmX, (a0 + a) * kUmmaKC, 0, xbar);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(xiss);                            // the weight's copies may follow
        }
        // this CTA's columns of w, zero past H (so y's padding is exact zeros)
        for (int j = tid - 32; j < nat * 8; j += kTcNormWarps * 32) {
            if (a0 * 8 + j < NP)
                cp_async16(wsm + j * 16, static_cast<const uint4 *>(p.w) + a0 * 8 + j);
            else
                *reinterpret_cast<uint4 *>(wsm + j * 16) = make_uint4(0, 0, 0, 0);
        }
        // Units of work: (row quad, atom), U = (T / 4) nat of them; norm warp
        // nw takes units nw, nw + 15, ...; in a unit, lane (c8 = lane % 8,
        // rq = lane / 8) takes the 16-byte chunk c8 of row 4 quad + rq
        // (a quarter-warp reads one row's 128 bytes: all banks once). r is
        // loaded kTcBatch units at a time, all loads first.
        const int c8 = lane & 7, rq = lane >> 3;
        const int RQ = NT / 4, U = RQ * nat;
        // unit u is (atom u / RQ, row quad u % RQ); a warp's units advance by
        // kTcNormWarps, so both are stepped by addition, not divided out
        const int dq = kTcNormWarps / RQ, dr = kTcNormWarps % RQ;
        auto step = [&](int &a, int &q) {
            q += dr;
            a += dq;
            if (q >= RQ) {
                q -= RQ;
                ++a;
            }
        };
        // warp-uniform (the units' shuffles need every lane of the warp)
        const bool ok = __all_sync(0xFFFFFFFFu, tc_wait(xbar, 0, limit, fail));
        int ab = nw / RQ, qb = nw % RQ;                       // unit u0's atom and quad
        for (int u0 = nw; ok && u0 < U; u0 += kTcNormWarps * kTcBatch) {
            uint4 rv[kTcBatch];
            if constexpr (RES) {
                int a = ab, q = qb;
#pragma unroll
                for (int k = 0; k < kTcBatch; ++k) {
                    const int u = u0 + k * kTcNormWarps;
                    const int row = 4 * q + rq, col8 = (a0 + a) * 8 + c8;
                    rv[k] = (u < U && row < p.M && col8 < NP)
                                ? ld_row_v4(static_cast<const uint4 *>(p.r) + (int64_t)row * NP + col8)
                                : make_uint4(0, 0, 0, 0);
                    step(a, q);
                }
            }
            int a = ab, q = qb;
#pragma unroll
            for (int k = 0; k < kTcBatch; ++k, step(a, q)) {
                const int u = u0 + k * kTcNormWarps;
                if (u >= U)                                   // warp-uniform
                    break;
                const int row = 4 * q + rq, col8 = (a0 + a) * 8 + c8;
                const uint32_t off = (uint32_t)a * atom + (uint32_t)row * 128u +
                                     ((uint32_t)(c8 ^ (row & 7)) << 4);
                F acc = splat<F>(0.f);
                if (row < p.M && col8 < NP) {
                    P hv;
                    hv.u = *reinterpret_cast<const uint4 *>(ysm + off);
                    if constexpr (RES) {
                        hv.u.x = add2_rn<T>(hv.u.x, rv[k].x);   // h as stored
                        hv.u.y = add2_rn<T>(hv.u.y, rv[k].y);
                        hv.u.z = add2_rn<T>(hv.u.z, rv[k].z);
                        hv.u.w = add2_rn<T>(hv.u.w, rv[k].w);
                        *reinterpret_cast<uint4 *>(ysm + off) = hv.u;
                        if (writer && p.h != nullptr)
                            hv.store(p.h, (int64_t)row * NP + col8);
                    }
                    X v;
                    hv.widen(v);
#pragma unroll
                    for (int e = 0; e < X::N; ++e)
                        acc = vfma(v.v[e], v.v[e], acc);
                }
                float sq = hsum(acc);
                sq += __shfl_xor_sync(0xFFFFFFFFu, sq, 1);
                sq += __shfl_xor_sync(0xFFFFFFFFu, sq, 2);
                sq += __shfl_xor_sync(0xFFFFFFFFu, sq, 4);
                if (c8 == 0)
                    part[a * NT + row] = sq;                  // atom a's share of row's sum
            }
#pragma unroll
            for (int k = 0; k < kTcBatch; ++k)
                step(ab, qb);
        }
        cp_async_wait_all_groups();                           // this thread's part of w
        named_bar_sync(1, kTcNormWarps * 32);
        // each token's sum over this CTA's atoms, in atom order
        if (ok && tid - 32 < NT) {
            float sq = 0.f;
            for (int a = 0; a < nat; ++a)
                sq += part[a * NT + (tid - 32)];
            csum[tid - 32] = sq;
        }
        named_bar_sync(1, kTcNormWarps * 32);
        // with a cluster: store the sums into every peer (psum[rank][row] of
        // its send area, unused until its epilogue), wait for theirs
        bool ok2 = ok;
        if (KS > 1) {
            if (ok && tid - 32 < NT) {
                const int row = tid - 32;
                const uint32_t at = smem_addr(psum + rank * NT + row);
                for (int q = 1; q < KS; ++q) {
                    const uint32_t peer = (uint32_t)((rank + q) % KS);
                    st_async_b32(cluster_map(at, peer), __float_as_uint(csum[row]),
                                 cluster_map(pready, peer));
                }
            }
            ok2 = ok && tc_wait<true>(pready, 0, limit, fail);
        }
        if (ok2 && tid - 32 < NT) {
            const int row = tid - 32;
            float sq;
            if (KS > 1) {
                sq = 0.f;
                for (int q = 0; q < KS; ++q)                  // rank order
                    sq += q == rank ? csum[row] : psum[q * NT + row];
            } else {
                sq = csum[row];
            }
            const float r = rsqrtf(sq / (float)H + p.eps);
            rsv[row] = r;
            if (writer && rank == 0 && p.rstd != nullptr && row < p.M)
                p.rstd[row] = r;
        }
        named_bar_sync(1, kTcNormWarps * 32);
        int a2 = nw / RQ, q2 = nw % RQ;
        for (int u = nw; ok2 && u < U; u += kTcNormWarps, step(a2, q2)) {
            const int a = a2, row = 4 * q2 + rq, col8 = (a0 + a) * 8 + c8;
            if (row >= p.M || col8 >= NP)
                continue;
            const uint32_t off = (uint32_t)a * atom + (uint32_t)row * 128u +
                                 ((uint32_t)(c8 ^ (row & 7)) << 4);
            const F r2 = splat<F>(rsv[row]);
            P h8, w8;
            h8.u = *reinterpret_cast<const uint4 *>(ysm + off);
            w8.u = *reinterpret_cast<const uint4 *>(wsm + (a * 8 + c8) * 16);
            X v, e8;
            h8.widen(v);
            w8.widen(e8);
#pragma unroll
            for (int e = 0; e < X::N; ++e)
                v.v[e] = vmul(vmul(v.v[e], r2), e8.v[e]);
            const P yv = P::narrow(v);
            *reinterpret_cast<uint4 *>(ysm + off) = yv.u;
            if (writer && p.y != nullptr)
                yv.store(p.y, (int64_t)row * NP + col8);
        }
        // every input but A is read; y is complete and, fenced, visible to
        // the tensor cores
        griddep_launch_dependents();
        fence_proxy_async_smem();
        named_bar_sync(1, kTcNormWarps * 32);

        if (tid == 32 && !*fail) {
            // ------------------------------------------------------ MMAs
            const uint32_t idesc = umma_idesc_f16(UmmaFormat<T>::value, kUmmaM, NT);
            const uint64_t dr0 = umma_desc_sw128(ring_s), dy0 = umma_desc_sw128(y_s);
            int q = 0;
            bool stop = false;
            for (int jt = 0; jt < mt && !stop; ++jt) {
                const int b = jt % kTcAcc;
                if (jt >= kTcAcc &&
                    !tc_wait(acce0 + 8u * b, (uint32_t)((jt / kTcAcc - 1) & 1), limit, fail))
                    break;
                tc_fence_after_sync();
                const uint32_t d = tmem + (uint32_t)b * ncols;
                for (int g = 0; g < ng; ++g, ++q) {
                    const int s = q % NSt;
                    if (!tc_wait(full0 + 8u * s, (uint32_t)((q / NSt) & 1), limit, fail)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after_sync();
                    const int alo = g * APS, ahi = min(nat, alo + APS);
                    const uint64_t ds = dr0 + (uint64_t)(s * (int)(stage >> 4));
                    for (int a = alo; a < ahi; ++a) {
                        const uint64_t da = ds + (uint64_t)((a - alo) * (int)(kTcAtom >> 4));
                        const uint64_t dy = dy0 + (uint64_t)(a * (int)(atom >> 4));
#pragma unroll
                        for (int k4 = 0; k4 < kUmmaKC / 16; ++k4)
                            umma_f16(d, da + 2 * k4, dy + 2 * k4, idesc, (a | k4) != 0 ? 1u : 0u);
                    }
                    umma_commit(empty0 + 8u * s);     // the stage is free once these are done
                    slots[3] = q + 1;
                }
                if (!stop)
                    umma_commit(accf0 + 8u * b);      // tile jt's accumulator is complete
            }
        } else if (warp >= kTcEpiWarp0 && warp < kTcEpiWarp0 + kTcEpiWarps) {
            // -------------------------------------------------- epilogue
            const int q4 = warp & 3, hh = (warp - kTcEpiWarp0) >> 2;
            const int ft = q4 * 32 + lane;                    // feature within the tile
            const int owner = ft / fpo, fl = ft % fpo;        // its owner, place there
            const bool mine = owner == rank;
            const uint32_t lanes = (uint32_t)(q4 * 32) << 16;
            const int etid = tid - kTcEpiWarp0 * 32;          // 0..255
            // Every decision to stop is uniform: across the warp without a
            // cluster, across the epilogue's warps with one (they meet at
            // named barriers, which must not be left by some and waited at
            // by others).
            for (int jt = 0; jt < mt; ++jt) {
                const int b = jt % kTcAcc;
                const bool okf = tc_wait(accf0 + 8u * b, (uint32_t)((jt / kTcAcc) & 1), limit, fail);
                if (KS > 1 ? bar_red_or(2, kTcEpiWarps * 32, !okf)
                           : !__all_sync(0xFFFFFFFFu, okf))
                    break;
                tc_fence_after_sync();
                const int f = (cid + jt * ncl) * kUmmaM + ft;
                float keep[2][16];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    if (16 * hh + 32 * j >= NT)
                        break;
                    const int t0 = 16 * hh + 32 * j;
                    uint32_t v[16];
                    tmem_ld16(tmem + (uint32_t)b * ncols + lanes + (uint32_t)t0, v);
                    if (KS == 1) {
                        if (f < p.N) {
#pragma unroll
                            for (int k = 0; k < 16; ++k) {
                                const int t = t0 + k;
                                if (t < p.M) {
                                    Vals<1> o;
                                    o.v[0] = __uint_as_float(v[k]);
                                    Pack<T, 1>::narrow(o).store(p.out, (int64_t)t * p.N + f);
                                }
                            }
                        }
                    } else if (mine || direct) {
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            keep[j][k] = __uint_as_float(v[k]);
                    } else {
                        float4 *dst = reinterpret_cast<float4 *>(
                            send + (uint32_t)owner * L.xblock + ((uint32_t)fl * L.xrow + t0) * 4u);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            dst[k] = make_float4(__uint_as_float(v[4 * k]),
                                                 __uint_as_float(v[4 * k + 1]),
                                                 __uint_as_float(v[4 * k + 2]),
                                                 __uint_as_float(v[4 * k + 3]));
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(acce0 + 8u * b);      // the accumulator may be reused
                if (KS == 1)
                    continue;
                // send this tile's partial products to their owners once each
                // owner has freed its slots after the previous tile: straight
                // from registers into the owner's receive slot for this CTA
                // (asynchronous stores counted on its `rx full` barrier), or
                // (64 tokens) one bulk copy of each owner's block
                if (!direct) {
                    fence_proxy_async_smem();
                    named_bar_sync(2, kTcEpiWarps * 32);
                    if (etid == 0 && !*fail &&
                        (jt == 0 || tc_wait<true>(rxfree, (uint32_t)((jt - 1) & 1), limit, fail))) {
                        for (int d1 = 1; d1 < KS; ++d1) {
                            const int o = (rank + d1) % KS;
                            bulk_s2s_cluster(
                                cluster_map(recv_s + (uint32_t)rank * L.xblock, (uint32_t)o),
                                smem_addr(send) + (uint32_t)o * L.xblock, L.xblock,
                                cluster_map(rxfull, (uint32_t)o));
                        }
                        bulk_wait_read_all();         // the send blocks are free again
                    }
                    if (bar_red_or(2, kTcEpiWarps * 32, *fail != 0))
                        break;
                } else {
                    const bool fr =
                        jt == 0 || tc_wait<true>(rxfree, (uint32_t)((jt - 1) & 1), limit, fail);
                    if (bar_red_or(2, kTcEpiWarps * 32, !fr || *fail != 0))
                        break;
                }
                if (direct && !mine) {
                    const uint32_t slot = cluster_map(recv_s + (uint32_t)rank * L.xblock, (uint32_t)owner);
                    const uint32_t rbar = cluster_map(rxfull, (uint32_t)owner);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        if (16 * hh + 32 * j >= NT)
                            break;
                        const int t0 = 16 * hh + 32 * j;
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4)
                            st_async_v4(slot + ((uint32_t)fl * L.xrow + t0 + 4 * k4) * 4u,
                                        make_float4(keep[j][4 * k4], keep[j][4 * k4 + 1],
                                                    keep[j][4 * k4 + 2], keep[j][4 * k4 + 3]),
                                        rbar);
                    }
                }
                // the peers' partial products for this CTA's features
                const bool got = tc_wait<true>(rxfull, (uint32_t)(jt & 1), limit, fail);
                if (bar_red_or(2, kTcEpiWarps * 32, !got))
                    break;
                if (etid == 0)
                    ++rx_done;
                if (mine && f < p.N) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        if (16 * hh + 32 * j >= NT)
                            break;
                        const int t0 = 16 * hh + 32 * j;
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4) {
                            float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
                            for (int q = 0; q < KS; ++q) {          // rank order
                                float4 pv;
                                if (q == rank)
                                    pv = make_float4(keep[j][4 * k4], keep[j][4 * k4 + 1],
                                                     keep[j][4 * k4 + 2], keep[j][4 * k4 + 3]);
                                else
                                    pv = *reinterpret_cast<const float4 *>(
                                        recv + (uint32_t)q * L.xblock +
                                        ((uint32_t)fl * L.xrow + t0 + 4 * k4) * 4u);
                                s4.x += pv.x;
                                s4.y += pv.y;
                                s4.z += pv.z;
                                s4.w += pv.w;
                            }
                            const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int t = t0 + 4 * k4 + e;
                                if (t < p.M) {
                                    Vals<1> o;
                                    o.v[0] = sv[e];
                                    Pack<T, 1>::narrow(o).store(p.out, (int64_t)t * p.N + f);
                                }
                            }
                        }
                    }
                }
                named_bar_sync(2, kTcEpiWarps * 32);         // done reading the receive slots
                if (etid == 0) {
                    if (jt + 1 < mt) {                        // the next tile's products
                        mbar_expect_tx(rxfull, rx_bytes);
                        slots[4] = slots[4] + 1;
                    }
                    for (int d1 = 1; d1 < KS; ++d1)           // the slots are free again
                        mbar_arrive_remote_cta(cluster_map(rxfree, (uint32_t)((rank + d1) % KS)));
                }
            }
        }
    }

    // every role has finished or given up
    __syncthreads();
    if (*fail) {
        if (tid == 0) {         // copies issued and not consumed: let them land
            for (int q = slots[3]; q < slots[2]; ++q)
                (void)mbar_wait_bounded(full0 + 8u * (q % NSt), (uint32_t)((q / NSt) & 1), limit);
            atomicAdd(timeouts, 1u);
        }
        if (tid == 32) {        // the MMAs issued are complete before the memory is freed
            umma_commit(dbar);
            (void)mbar_wait_bounded(dbar, 0, limit);
        }
        if (KS > 1 && tid == kTcEpiWarp0 * 32 && slots[4] > rx_done)
            // partial products a peer may still be copying into this CTA
            (void)mbar_wait_bounded(rxfull, (uint32_t)(rx_done & 1), limit);
        if (KS > 1 && tid == 64)   // sums of squares a peer may still be storing
            (void)mbar_wait_bounded(pready, 0, limit);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (KS > 1) {               // no CTA leaves while a peer may still use its memory
        cluster_arrive_release();
        cluster_wait_acquire();
    }
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, (uint32_t)kTcAcc * ncols);
    }
}

} // namespace rmsk
