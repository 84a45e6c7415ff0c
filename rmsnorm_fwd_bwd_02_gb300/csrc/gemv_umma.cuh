// gemv_umma.cuh -- RMSNorm fused with the projection, the product on the
// fifth-generation tensor cores (tcgen05, accumulators in tensor memory),
// K split over a thread-block cluster. Same result as rms_gemv and
// rms_gemv_tma: the chain of [P2] (the 0.8B Qwen decode article,
// trdm.cn news/483216) §2.1, §3.1 with y rounded to the dtype before
// out = y A^T, fp32 accumulation.
//
// Why this shape. In a decode batch of up to 64 tokens every CTA needs y
// for all of them, and the weight is the only large input. A CTA that
// normalised whole rows had to load all of x and r (229 KB at 64 x 896,
// as much as its share of the weight), and a warp-level MMA is bound by its
// issue rate from 16 rows on. Here a cluster of KS CTAs shares one tile of
// 128 output features and splits K between them: CTA `rank` owns the
// 64-column atoms [rank na / KS, (rank + 1) na / KS) of the row. It loads
// only those columns of x, r, w and of its 128 rows of A, so a grid of
// (N / 128) x KS CTAs reads every input once per cluster, and KS is chosen
// so that the grid fills the SMs.
//
// The product is laid out for a decode batch: the tile's 128 features are
// the MMA's M (rows of A), the tokens (M of the call rounded up to 16, T)
// its N, K = the CTA's columns. Operands are K-major in the 128-byte
// swizzled layout: an atom of R rows x 64 columns holds row i's 128 bytes at
// i 128, its 16-byte chunk c at position c ^ (i % 8), on a 1024-byte
// boundary. Tensor copies with the 128-byte swizzle write exactly this
// layout, for A and for x and r alike, so h and y are computed in place.
//
//  1. Warp 0 allocates the accumulator's tensor-memory columns, warp 1
//     initialises the mbarriers (A's atoms in two groups, one each; x and r;
//     the MMAs; the partial products received), warp 2 prefetches the three
//     tensor maps.
//  2. Tensor copies (the TMA engine, 128-byte swizzle), one per lane: x and
//     r (T rows x 64 columns per atom, rows past M and columns past H read
//     as zero) by warp 1 as soon as the previous kernel is complete, A's
//     atoms (128 rows x 64 columns, 16 KB) by warp 0 behind them. An SM
//     serves its tensor copies in order and the norm needs x and r first, so
//     with static weights only the first two atoms of A start before the
//     wait on the previous kernel. w by cp.async.
//  3. The norm: h = x + r (rounded, stored in place), the partial sums of
//     h^2 over the CTA's columns per token, published in shared memory; a
//     cluster barrier; each token's sum read from every CTA of the cluster
//     in rank order (distributed shared memory), rstd; y = h rstd w,
//     rounded, in place. The first cluster also stores h, y and rstd.
//  4. Thread 0 issues four MMAs (m128 nT k16) per atom, a group of atoms
//     once its copies have landed, and commits them to one mbarrier. Its
//     instruction stream is the cost here (some 120 cycles an MMA with the
//     descriptors built per MMA, about 200 per mbarrier wait even on a
//     completed phase), so the descriptors advance by additions and A's
//     atoms have two barriers, not one each.
//  5. The partial products: each warp reads 32 features x 16 tokens of the
//     accumulator at a time (tcgen05.ld); each group of 4 tokens belongs to
//     one CTA of the cluster (group g: rank g % KS). A CTA writes its own
//     groups into its receive area and stores the others straight into
//     their owner's receive area (asynchronous 16-byte stores into
//     distributed shared memory, counted on the owner's mbarrier: no
//     staging, no copy to issue). The owner adds the KS partials of its
//     groups in rank order (deterministic), rounds and stores
//     out[token][feature]. The tensor memory is freed as soon as it is
//     read.
//  6. A CTA leaves once the stores into it have landed and every CTA of
//     the cluster has read the partial sums it needed (a cluster barrier
//     arrived at right after that read and waited for only here).
//
// Every mbarrier wait is bounded (about one second, or the test limit); one
// that runs out counts in the streamed-kernel timeout counter, the CTA skips
// its remaining work but still takes part in both cluster barriers and in
// the exchange (sending zeros), waits (bounded again) for its copies in
// flight, and frees its tensor memory.
#pragma once

#include <cuda.h>

#include "gemv.cuh"
#include "split.cuh"
#include "stream.cuh"

namespace rmsk {

constexpr int kUmmaM = 128;        // output features per tile (the MMA's M)
constexpr int kUmmaKC = 64;        // K columns per atom: one swizzle span
constexpr int kUmmaThreads = 512;  // sixteen warps; warp w reads tensor-memory lanes
                                   // 32 (w % 4) .. 32 (w % 4) + 31
constexpr int kUmmaMaxCluster = 8; // CTAs splitting K (portable cluster size)
constexpr uint32_t kUmmaAtomA = kUmmaM * kUmmaKC * 2;   // 16 KB

// Shared-memory layout of one CTA, byte offsets from a 1024-byte aligned
// base: y (x copied in, h and y computed in place) at 0, r, the atoms of A,
// the partial products received (over r when r is large enough: r is
// consumed before any CTA sends), w, the mbarriers, the tensor-memory
// address, and the partial row sums and rstd of the T tokens. The receive
// area is [rank][feature][rs slots of 16 bytes].
struct UmmaLayout {
    int apc;             // most atoms per CTA: ceil(na / KS)
    int rs;              // 16-byte slots per feature and rank in the receive
                         // area (odd: conflict-free accesses)
    uint32_t r, a, recv, w, bar, total;   // total: with the 1023 bytes of alignment
};

__host__ __device__ inline UmmaLayout gemv_umma_layout(int T, int H, int KS, bool res)
{
    UmmaLayout L;
    const int na = (H + kUmmaKC - 1) / kUmmaKC;
    L.apc = (na + KS - 1) / KS;
    const int g4 = (T / 4 + KS - 1) / KS;                  // 4-token groups per owner, most
    L.rs = g4 | 1;
    const uint32_t atom = (uint32_t)T * 128u;               // one atom of x, r or y
    const uint32_t ybytes = (uint32_t)L.apc * atom;
    const uint32_t rbytes = res ? ybytes : 0u;
    const uint32_t recv = (uint32_t)KS * kUmmaM * (uint32_t)L.rs * 16u;
    const uint32_t abytes = (uint32_t)L.apc * kUmmaAtomA;
    L.r = ybytes;
    L.a = ybytes + rbytes;
    uint32_t end = L.a + abytes;
    if (rbytes >= recv) {
        L.recv = L.r;
    } else {
        L.recv = end;
        end += recv;
    }
    L.w = end;
    L.bar = L.w + (uint32_t)L.apc * kUmmaKC * 2;
    // mbarriers: apc + 3; then 4 words, then T partial sums and T rstd
    L.total = L.bar + 8u * (uint32_t)(L.apc + 3) + 16u + 8u * (uint32_t)T + 1023u;
    return L;
}

struct GemvUmmaParams {
    const void *w;    // [H]
    void *out;        // [M,N]
    void *h;          // [M,H] residual sum out, or nullptr
    void *y;          // [M,H] stored norm output, or nullptr
    float *rstd;      // [M] or nullptr
    int M, H, N;
    int T;            // tokens as the MMA's N: M rounded up to 16 (<= 64)
    int na;           // atoms of K in a row: ceil(H / 64)
    UmmaLayout L;     // for T, H, the cluster size and the residual
    float eps;
    int static_w;     // w and A may be read before the wait on the previous kernel
    // test hook of the bounded waits: bytes a copy of A is expected to bring
    // beyond what it does (0), and the wait limit in microseconds (0: about
    // one second)
    uint32_t extra_tx, wait_limit_us;
};

// Tensor-memory columns of a T-token accumulator (fp32, one column per
// token; a power of two, at least 32).
__host__ __device__ constexpr uint32_t gemv_umma_tmem_cols(int T)
{
    return T <= 32 ? 32u : (T <= 64 ? 64u : 128u);
}

// Instruction descriptor of kind::f16: D fp32 (bits 4-5 = 1), A and B of
// format `ab` (bits 7-9 and 10-12: 0 fp16, 1 bf16), both K-major (bits 15,
// 16 = 0), N / 8 in bits 17-22, M / 16 in bits 24-28.
__host__ __device__ constexpr uint32_t umma_idesc_f16(uint32_t ab, int M, int N)
{
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

template <typename T> struct UmmaFormat;
template <> struct UmmaFormat<bf16> { static constexpr uint32_t value = 1; };
template <> struct UmmaFormat<f16> { static constexpr uint32_t value = 0; };

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout: start address (16-byte units, bits 0-13), leading byte
// offset 16 bytes (unused by this layout; bits 16-29), stride byte offset
// 1024 bytes between 8-row groups (bits 32-45), descriptor version 1 (bits
// 46-47), base offset 0 (atoms on 1024-byte boundaries), layout type 2 =
// 128-byte swizzle (bits 61-63).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(16 >> 4) << 16) |
           ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D (tensor memory) = A B^T (+ D when accumulate != 0), kind::f16.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// The mbarrier completes a phase once every tcgen05 operation this thread
// issued before has.
__device__ __forceinline__ void umma_commit(uint32_t mbar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     mbar)
                 : "memory");
}

// 16 consecutive fp32 columns of the warp's 32 lanes (lane = this thread).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                   "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
                   "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Tiled tensor copy of the box at (x = column, y = row) of a 2-D tensor map
// into shared memory, completing its bytes on `bar`. x is a multiple of 64
// (whole atoms), so x * 2 bytes is a multiple of 16.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
                 "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all_groups()
{
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// Fetch a tensor map (a kernel parameter, by its generic address) into the
// descriptor cache ahead of its first copy.
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map))
                 : "memory");
}

// Bulk copy of `bytes` (a multiple of 16, 16-byte aligned) from this CTA's
// shared memory into another CTA's of the cluster, completing on that CTA's
// mbarrier (both given as cluster addresses).
__device__ __forceinline__ void bulk_s2s_cluster(uint32_t dst, uint32_t src, uint32_t bytes,
                                                 uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes "
                 "[%0], [%1], %2, [%3];" ::"r"(dst),
                 "r"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Barrier `id` (not 0: __syncthreads) over `count` threads, whole warps.
__device__ __forceinline__ void named_bar_sync(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// h = x + r on two packed elements, rounded to nearest even: for bf16 one
// packed bf16 addition (correctly rounded, so equal to adding in fp32 and
// rounding: the fp32 sum of two bf16 values is exact unless their exponents
// differ by more than 15, and then the smaller is far below half an ulp of
// the larger); fp16 goes through fp32 as the other kernels do.
template <typename T> __device__ __forceinline__ uint32_t add2_rn(uint32_t a, uint32_t b);
template <> __device__ __forceinline__ uint32_t add2_rn<bf16>(uint32_t a, uint32_t b)
{
    const __nv_bfloat162 s = __hadd2(*reinterpret_cast<const __nv_bfloat162 *>(&a),
                                     *reinterpret_cast<const __nv_bfloat162 *>(&b));
    return *reinterpret_cast<const uint32_t *>(&s);
}
template <> __device__ __forceinline__ uint32_t add2_rn<f16>(uint32_t a, uint32_t b)
{
    const float2 x = Half16<f16>::wide2(a), y = Half16<f16>::wide2(b);
    return Half16<f16>::narrow2(x.x + y.x, x.y + y.y);
}

// This thread's bulk copies issued so far have read their source.
__device__ __forceinline__ void bulk_wait_read_all()
{
    asm volatile("cp.async.bulk.commit_group;\ncp.async.bulk.wait_group.read 0;" ::: "memory");
}

// grid = (N / 128 rounded up) x KS CTAs, cluster = (KS, 1, 1), 256 threads,
// dynamic shared memory p.L.total.
template <typename T, bool RES>
__global__ void __launch_bounds__(kUmmaThreads, 1)
rms_gemv_umma(const GemvUmmaParams p, const __grid_constant__ CUtensorMap tmA,
              const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmR,
              unsigned int *timeouts)
{
    using P = Pack<T, 8>;
    using X = Vals<8>;
    using F = float2;
    constexpr int kB = 4;                                     // atoms per batch of loads
    constexpr int kEarly = 2;                                 // atoms of A before x and r
    extern __shared__ __align__(1024) unsigned char umma_smem[];

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int H = p.H, NT = p.T, NP = H / 8;                  // NT: tokens as the MMA's N
    const int KS = (int)cluster_nctarank(), rank = (int)cluster_ctarank();
    const int f0 = (int)(blockIdx.x / KS) * kUmmaM;           // the tile's first feature
    const int a0 = rank * p.na / KS;                          // this CTA's atoms of K
    const int nat = (rank + 1) * p.na / KS - a0;
    const bool writer = blockIdx.x < (unsigned)KS;            // the first cluster stores
                                                              // h, y and rstd
    const UmmaLayout &L = p.L;
    const uint32_t raw_s = smem_addr(umma_smem);
    unsigned char *base = umma_smem + (((raw_s + 1023u) & ~1023u) - raw_s);
    unsigned char *ysm = base, *rsm = base + L.r, *wsm = base + L.w;
    const float4 *recv = reinterpret_cast<const float4 *>(base + L.recv);
    const uint32_t y_s = smem_addr(ysm), r_s = smem_addr(rsm), a_s = smem_addr(base + L.a);
    const uint32_t recv_s = smem_addr(base + L.recv);
    // A's atoms land in two groups, each behind one mbarrier (a wait costs
    // some 200 cycles even when its phase is complete): [0, nh), [nh, nat)
    const uint32_t abar = smem_addr(base + L.bar);
    const uint32_t xbar = abar + 8u * (uint32_t)L.apc;        // x and r landed
    const uint32_t mbar = xbar + 8u, rbar = xbar + 16u;       // MMAs done; products received
    int *slots = reinterpret_cast<int *>(base + L.bar + 8 * (L.apc + 3));
    // slots[0]: tensor-memory address, [1]: a wait ran out, [2]: atoms multiplied
    float *part = reinterpret_cast<float *>(slots + 4);       // [T] sums of h^2, own columns
    float *rsv = part + NT;                                   // [T] rstd
    const uint32_t atom = (uint32_t)NT * 128u;                // bytes of an atom of x, r, y
    const uint32_t ncols = gemv_umma_tmem_cols(NT);
    const unsigned long long limit = wait_limit_ns(p.wait_limit_us);
    const int G4 = NT / 4;                                    // 4-token groups
    const int own = G4 > rank ? (G4 - 1 - rank) / KS + 1 : 0; // groups this CTA sums
    const int nh = (nat + 1) / 2;                             // atoms of A's first group
    constexpr int kWarps = kUmmaThreads / 32;

    // 1. descriptors, tensor memory and the barriers, by three warps at once
    if (tid == 64) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmX);
        if constexpr (RES)
            prefetch_tmap(&tmR);
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(slots), ncols);
        tmem_relinquish();
    }
    if (tid == 32) {
        mbar_init(abar, 1);
        if (nat > nh)
            mbar_init(abar + 8u, 1);
        mbar_init(xbar, 1);
        mbar_init(mbar, 1);
        mbar_init(rbar, 1);
        if (own > 0)     // every other CTA stores its partials of the owned groups
            mbar_expect_tx(rbar, (uint32_t)(KS - 1) * (uint32_t)kUmmaM * 16u * (uint32_t)own);
        slots[1] = 0;
        slots[2] = 0;
    }
    mbar_init_fence();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = static_cast<uint32_t>(slots[0]);

    // 2. copies. The tensor copies of one SM are served in order, and x and r
    //    (the norm's inputs, from L2) are needed first: ahead of them go
    //    only the atoms of A that static weights allow to start before the
    //    wait on the previous kernel (at most kEarly), the rest after them.
    const int c0 = a0 * kUmmaKC;                              // first column of this CTA
    const int c1 = min(H, (a0 + nat) * kUmmaKC);              // one past its last
    auto load_a = [&](int i0, int i1) {                       // warp 0, lane i: atom i
        const int i = i0 + lane;
        if (i < i1)
            tma_load_2d(a_s + (uint32_t)i * kUmmaAtomA, &tmA, (a0 + i) * kUmmaKC, f0,
                        abar + (i < nh ? 0u : 8u));
    };
    auto load_w = [&]() {
        for (int j = tid; j < (c1 - c0) / 8; j += kUmmaThreads)
            cp_async16(wsm + j * 16, static_cast<const uint4 *>(p.w) + c0 / 8 + j);
    };
    const int early = p.static_w ? min(nat, kEarly) : 0;
    if (warp == 0) {
        if (lane == 0) {        // each group's bytes, before any of its copies
            mbar_expect_tx(abar, (uint32_t)nh * (kUmmaAtomA + p.extra_tx));
            if (nat > nh)
                mbar_expect_tx(abar + 8u, (uint32_t)(nat - nh) * (kUmmaAtomA + p.extra_tx));
        }
        __syncwarp();
        load_a(0, early);
    }
    if (p.static_w)
        load_w();
    griddep_wait();
    // warp 1 copies x and r (lane i: atom i) and then lets warp 0 copy the
    // rest of A
    if (warp == 1) {
        if (lane == 0)
            mbar_expect_tx(xbar, atom * (uint32_t)nat * (RES ? 2u : 1u));
        __syncwarp();
        if (lane < nat) {
            tma_load_2d(y_s + (uint32_t)lane * atom, &tmX, (a0 + lane) * kUmmaKC, 0, xbar);
            if constexpr (RES)
                tma_load_2d(r_s + (uint32_t)lane * atom, &tmR, (a0 + lane) * kUmmaKC, 0, xbar);
        }
    }
    if (warp < 2)
        named_bar_sync(1, 64);
    if (warp == 0)
        load_a(early, nat);
    if (!p.static_w)
        load_w();

    // 3. the norm. Lane (c8 = lane % 8, rq = lane / 8) of warp w takes the
    //    16-byte chunk c8 of rows 4 (w + 16 m) + rq of every atom, so a
    //    quarter-warp reads one row's 128 bytes (all banks once); kB atoms'
    //    chunks are loaded before any is written back.
    const int c8 = lane & 7, rq = lane >> 3;
    const bool xfail = __syncthreads_or(!mbar_wait_bounded(xbar, 0, limit));
    {
        F acc[2] = {splat<F>(0.f), splat<F>(0.f)};
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int row = 4 * (warp + kWarps * m) + rq;
            if (xfail || 4 * (warp + kWarps * m) >= NT)            // warp-uniform
                break;
            const uint32_t roff = (uint32_t)row * 128u + ((uint32_t)(c8 ^ (row & 7)) << 4);
            for (int i0 = 0; i0 < nat; i0 += kB) {
                uint4 xv[kB], rv[kB];
#pragma unroll
                for (int b = 0; b < kB; ++b) {
                    const int i = i0 + b;
                    if (i < nat && (a0 + i) * 8 + c8 < NP) {  // zeros past H
                        xv[b] = *reinterpret_cast<const uint4 *>(ysm + i * atom + roff);
                        if constexpr (RES)
                            rv[b] = *reinterpret_cast<const uint4 *>(rsm + i * atom + roff);
                    }
                }
#pragma unroll
                for (int b = 0; b < kB; ++b) {
                    const int i = i0 + b, col8 = (a0 + i) * 8 + c8;
                    if (i >= nat || col8 >= NP)
                        continue;
                    P hv;
                    hv.u = xv[b];
                    X a;
                    if constexpr (RES) {
                        hv.u.x = add2_rn<T>(xv[b].x, rv[b].x);   // h as stored
                        hv.u.y = add2_rn<T>(xv[b].y, rv[b].y);
                        hv.u.z = add2_rn<T>(xv[b].z, rv[b].z);
                        hv.u.w = add2_rn<T>(xv[b].w, rv[b].w);
                        *reinterpret_cast<uint4 *>(ysm + i * atom + roff) = hv.u;
                        if (writer && p.h != nullptr && row < p.M)
                            hv.store(p.h, (int64_t)row * NP + col8);
                    }
                    hv.widen(a);
#pragma unroll
                    for (int e = 0; e < X::N; ++e)
                        acc[m] = vfma(a.v[e], a.v[e], acc[m]);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int row = 4 * (warp + kWarps * m) + rq;
            float s = hsum(acc[m]);
            s += __shfl_xor_sync(0xFFFFFFFFu, s, 1);
            s += __shfl_xor_sync(0xFFFFFFFFu, s, 2);
            s += __shfl_xor_sync(0xFFFFFFFFu, s, 4);
            if (c8 == 0 && row < NT)
                part[row] = s;
        }
    }
    // The partial sums are published, and this CTA is done with r's area
    // (the peers' copies of partial products may land there after the
    // barrier): order its accesses before the barrier, for both proxies.
    fence_proxy_async_smem();
    cluster_arrive_release();
    cluster_wait_acquire();
    if (tid < NT) {
        const float tot = sum_cluster_f32(part + tid, (uint32_t)KS);   // rank order
        const float rs = rsqrtf(tot / (float)H + p.eps);
        rsv[tid] = rs;
        if (writer && rank == 0 && p.rstd != nullptr && tid < p.M)
            p.rstd[tid] = rs;
    }
    // done with the peers' shared memory (the loads' values are used above):
    // a CTA waits for this arrival of every CTA only when it leaves
    cluster_arrive_relaxed();
    cp_async_wait_all_groups();                               // this thread's part of w
    __syncthreads();
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const int row = 4 * (warp + kWarps * m) + rq;
        if (xfail || 4 * (warp + kWarps * m) >= NT)
            break;
        const uint32_t roff = (uint32_t)row * 128u + ((uint32_t)(c8 ^ (row & 7)) << 4);
        const F r2 = splat<F>(rsv[row]);
        for (int i0 = 0; i0 < nat; i0 += kB) {
            uint4 hv[kB], wv[kB];
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                const int i = i0 + b;
                if (i < nat && (a0 + i) * 8 + c8 < NP) {
                    hv[b] = *reinterpret_cast<const uint4 *>(ysm + i * atom + roff);
                    wv[b] = *reinterpret_cast<const uint4 *>(wsm + (i * 8 + c8) * 16);
                }
            }
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                const int i = i0 + b, col8 = (a0 + i) * 8 + c8;
                if (i >= nat || col8 >= NP)
                    continue;
                P h8, w8;
                h8.u = hv[b];
                w8.u = wv[b];
                X a, e8;
                h8.widen(a);
                w8.widen(e8);
#pragma unroll
                for (int e = 0; e < X::N; ++e)
                    a.v[e] = vmul(vmul(a.v[e], r2), e8.v[e]);
                const P yv = P::narrow(a);
                *reinterpret_cast<uint4 *>(ysm + i * atom + roff) = yv.u;
                if (writer && p.y != nullptr && row < p.M)
                    yv.store(p.y, (int64_t)row * NP + col8);
            }
        }
    }
    // every input but A is read: the next kernel may be scheduled; y is
    // complete and, fenced, visible to the tensor cores
    griddep_launch_dependents();
    fence_proxy_async_smem();
    __syncthreads();

    // 4. thread 0: four MMAs per atom of A, a group of atoms once its copies
    //    have landed, one commit. The descriptors advance by adding to their
    //    start-address field (16-byte units): 32 bytes per 16-column step,
    //    an atom per atom.
    if (tid == 0) {
        const uint32_t idesc = umma_idesc_f16(UmmaFormat<T>::value, kUmmaM, NT);
        const uint64_t da0 = umma_desc_sw128(a_s), db0 = umma_desc_sw128(y_s);
        bool failed = xfail;
        int i = 0, gi = 0;
        for (; !failed && gi < 2; ++gi) {
            const int i1 = gi == 0 ? nh : nat;
            if (i >= i1)
                break;                                        // no second group
            if (!mbar_wait_bounded(abar + 8u * (uint32_t)gi, 0, limit)) {
                failed = true;
                break;
            }
            tc_fence_after_sync();
            for (; i < i1; ++i) {
                const uint64_t da = da0 + (uint64_t)(i * (int)(kUmmaAtomA >> 4));
                const uint64_t db = db0 + (uint64_t)(i * (int)(atom >> 4));
                if (H - (a0 + i) * kUmmaKC >= kUmmaKC) {
#pragma unroll
                    for (int k4 = 0; k4 < kUmmaKC / 16; ++k4)
                        umma_f16(tmem, da + 2 * k4, db + 2 * k4, idesc, (i | k4) != 0 ? 1u : 0u);
                } else {                                      // the last, partial atom
                    const int ksteps = (H - (a0 + i) * kUmmaKC) / 16;
                    for (int k4 = 0; k4 < ksteps; ++k4)
                        umma_f16(tmem, da + 2 * k4, db + 2 * k4, idesc, (i | k4) != 0 ? 1u : 0u);
                }
            }
        }
        if (i > 0)
            umma_commit(mbar);
        slots[1] = failed ? 1 : 0;
        slots[2] = i;                                         // atoms whose MMAs were issued
        if (failed)            // let the copies started and not waited for land
            for (int g = gi; g < (nat > nh ? 2 : 1); ++g)
                (void)mbar_wait_bounded(abar + 8u * (uint32_t)g, 0, limit);
    }
    __syncthreads();
    bool failed = slots[1] != 0;
    if (slots[2] > 0)
        failed = __syncthreads_or(!mbar_wait_bounded(mbar, 0, limit)) || failed;

    // 5. the partial products of each 4-token group g go to its owner, rank
    //    g % KS, slot g / KS: the own ones straight into this CTA's receive
    //    area, the others by asynchronous 16-byte stores into the owner's
    //    receive area, counted on its mbarrier (zeros when this CTA failed,
    //    so that no owner waits for them)
    tc_fence_after_sync();
    {
        float4 *recv_own = reinterpret_cast<float4 *>(base + L.recv);
        const int q4 = warp & 3;                              // lane quarter
        const int fl = q4 * 32 + lane;                        // feature within the tile
        const uint32_t tw = tmem + ((uint32_t)(q4 * 32) << 16);
        for (int t0 = 16 * (warp >> 2); t0 < NT; t0 += 16 * (kWarps / 4)) {   // token blocks
            uint32_t v[16];
            if (!failed) {
                tmem_ld16(tw + (uint32_t)t0, v);
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    v[e] = 0u;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int g = t0 / 4 + j;                     // 4-token group
                const int owner = g % KS, slot = g / KS;
                const float4 o = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                             __uint_as_float(v[4 * j + 2]),
                                             __uint_as_float(v[4 * j + 3]));
                const uint32_t at = (uint32_t)(((rank * kUmmaM + fl) * L.rs + slot) * 16);
                if (owner == rank)
                    recv_own[(rank * kUmmaM + fl) * L.rs + slot] = o;
                else
                    st_async_v4(cluster_map(recv_s + at, (uint32_t)owner), o,
                                cluster_map(rbar, (uint32_t)owner));
            }
        }
    }
    // the tensor memory is read: free it now
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, ncols);
    }
    bool got = true;
    if (own > 0)
        got = !__syncthreads_or(!mbar_wait_bounded(rbar, 0, limit));
    if (got && !failed) {
        // sum the KS partials of each owned group in rank order, round, store
        for (int idx = tid; idx < kUmmaM * own; idx += kUmmaThreads) {
            const int fl = idx % kUmmaM, slot = idx / kUmmaM;
            const int g = slot * KS + rank;
            float4 pv[kUmmaMaxCluster];
#pragma unroll
            for (int q = 0; q < kUmmaMaxCluster; ++q)
                if (q < KS)
                    pv[q] = recv[(q * kUmmaM + fl) * L.rs + slot];
            float4 s = pv[0];
#pragma unroll
            for (int q = 1; q < kUmmaMaxCluster; ++q)
                if (q < KS) {
                    s.x += pv[q].x;
                    s.y += pv[q].y;
                    s.z += pv[q].z;
                    s.w += pv[q].w;
                }
            const int f = f0 + fl;
            if (f < p.N) {
                const float sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = 4 * g + e;
                    if (t < p.M) {
                        Vals<1> o;
                        o.v[0] = sv[e];
                        Pack<T, 1>::narrow(o).store(p.out, (int64_t)t * p.N + f);
                    }
                }
            }
        }
    }
    if ((failed || !got) && tid == 0)
        atomicAdd(timeouts, 1u);

    // 6. the products this CTA waited for have landed (waited for again,
    //    bounded, if that wait ran out) and its own copies have read their
    //    source; no CTA leaves while a peer may still read its partial sums
    //    (the peers arrived after reading them)
    if (tid == 0) {
        if (!got)
            (void)mbar_wait_bounded(rbar, 0, limit);
        bulk_wait_read_all();
    }
    cluster_wait_acquire();
}

} // namespace rmsk
