// gemv_umma.cuh -- RMSNorm fused with the projection, the product on the
// fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
// Same result as rms_gemv and rms_gemv_tma: the chain of [P2] (the 0.8B
// Qwen decode article, trdm.cn news/483216) §2.1, §3.1 with y rounded to the
// dtype before out = y A^T, fp32 accumulation.
//
// Why a third kernel: the warp-level m16n8k16 MMA of the other two bounds
// them from 16 rows on (some 40 cycles per MMA per warp on this part). Here
// one thread per CTA issues tcgen05.mma on operands in shared memory, and
// the product runs on the tensor cores.
//
// The product is laid out for a decode batch: the CTA's 128 output
// features are the MMA's M (rows of A), the tokens its N (rows of y, M of
// the call rounded up to 16), K = H. Both operands are K-major in the
// 128-byte swizzled layout: K is cut into atoms of 64 columns; an atom of R
// rows holds row i's 128 bytes at i 128, its 16-byte chunk c at position
// c ^ (i % 8), and starts on a 1024-byte boundary. A descriptor names the
// atom (start address, advanced 32 bytes per 16-column MMA step), the next
// 8 rows 1024 bytes on, and the 128-byte swizzle.
//
//  1. Warp 0 allocates the tensor-memory columns of the accumulator (a power
//     of two >= 32 and >= the padded token count); thread 0 initialises a
//     "full" and an "empty" mbarrier per ring stage.
//  2. Thread 0 starts tensor copies (the TMA engine, 128-byte swizzle) of the
//     first NS K atoms of the CTA's 128 rows of A into the ring, 16 KB each,
//     rows past N filled with zeros; every thread copies its part of w by
//     cp.async. With static weights this happens before the wait on the
//     previous kernel.
//  3. The norm, one 8-row group of tokens at a time by all 256 threads:
//     lane (row % 8, pack % 4), warp w takes packs 4 w + lane / 8 + 32 u, so
//     a thread holds at most 8 packs (H <= 2048) and loads them all at once;
//     the row sums of the eight warps meet in shared memory in warp order.
//     Without a cluster a CTA normalises every group. With a cluster of 8
//     (32 tokens or more) rank p normalises groups p, p + 8, ... and sends
//     each group's 1024-byte block of every atom of y (8 rows of 128 bytes:
//     one whole swizzle block, valid as it is at the same offset in any
//     CTA) to the other seven by bulk copies that complete on their "y"
//     mbarrier; a first cluster barrier phase, arrived at the start, makes
//     sure every CTA runs before its shared memory is written. The first
//     CTA (the first cluster) also writes h, y and rstd.
//  4. Thread 0 alone walks the K atoms: wait for the atom's copy (full
//     barrier), issue four MMAs (m128 nT k16) and commit them to the stage's
//     empty barrier, then refill the stage of the atom three before once its
//     MMAs are done (the copies run NS - 3 atoms ahead; NS as deep as shared
//     memory allows, up to 12).
//  5. The commit of the last atom completes once every MMA has: warp w reads
//     lanes 32 (w % 4) .. +31 (its 32 features) of the accumulator, blocks
//     of 16 tokens alternating between warps w and w + 4, rounds them and
//     stores out[token][feature] (32 consecutive features per warp and
//     token).
//  6. Warp 0 frees the tensor memory.
//
// Every mbarrier wait is bounded (about one second, or the test limit); one
// that runs out counts in the streamed-kernel timeout counter, the CTA skips
// the rest of its work, waits (bounded again) for its copies and MMAs in
// flight, and still frees its tensor memory.
#pragma once

#include <cuda.h>

#include "gemv.cuh"
#include "split.cuh"
#include "stream.cuh"

namespace rmsk {

constexpr int kUmmaM = 128;        // output features per CTA (the MMA's M)
constexpr int kUmmaKC = 64;        // K columns per ring stage: one swizzle atom
constexpr int kUmmaThreads = 256;  // eight warps; warp w reads tensor-memory lanes
                                   // 32 (w % 4) .. 32 (w % 4) + 31
constexpr int kUmmaMaxH = 2048;    // the norm holds no row in registers; the
                                   // limit is shared memory (y beside the ring)
constexpr uint32_t kUmmaStageBytes = kUmmaM * kUmmaKC * 2;   // 16 KB
// Most ring stages: a deep ring keeps enough of A in flight per SM (the K
// loop is otherwise bound by it), as far as shared memory allows beside y;
// the refill lag of the K loop (see the kernel).
constexpr int kUmmaMaxStages = 12;
constexpr int kUmmaLag = 3;

struct GemvUmmaParams {
    const void *x;    // [M,H]
    const void *r;    // [M,H] residual input, or unused
    const void *w;    // [H]
    void *out;        // [M,N]
    void *h;          // [M,H] residual sum out, or nullptr
    void *y;          // [M,H] stored norm output, or nullptr
    float *rstd;      // [M] or nullptr
    int M, H, N;
    int T;            // tokens as the MMA's N: M rounded up to 16 (<= 64)
    int NS;           // ring stages (16 KB atoms of A), 2 .. kUmmaMaxStages
    float eps;
    int static_w;     // w and A may be read before the wait on the previous kernel
    // test hook of the bounded waits: bytes a copy of A is expected to bring
    // beyond what it does (0), and the wait limit in microseconds (0: about
    // one second)
    uint32_t extra_tx, wait_limit_us;
};

// Bytes of y in shared memory: one swizzle atom of T rows per 64 columns.
__host__ __device__ constexpr int64_t gemv_umma_y_bytes(int T, int H)
{
    return (int64_t)((H + 63) / 64) * T * 128;
}

// Bytes of w in shared memory (rounded up to 128).
__host__ __device__ constexpr int64_t gemv_umma_w_bytes(int H)
{
    return ((int64_t)H * 2 + 127) / 128 * 128;
}

// Bytes of shared memory: up to 1023 of alignment, y, NS ring stages, w,
// 2 NS mbarriers, three words (tensor-memory address, atoms multiplied, a
// wait ran out), the mbarrier of y's rows from the cluster and the [8][8]
// row sums of the shared norm.
__host__ __device__ constexpr int64_t gemv_umma_smem_bytes(int T, int H, int NS)
{
    return 1024 + gemv_umma_y_bytes(T, H) + (int64_t)NS * kUmmaStageBytes +
           gemv_umma_w_bytes(H) + 16 * NS + 16 + 16 + 256;
}

// CTAs of a cluster sharing the norm (each normalises the 8-row groups g
// with g % kUmmaCluster = its rank and sends them to the others).
constexpr int kUmmaCluster = 8;

// Tensor-memory columns of a T-token accumulator (fp32, one column per token).
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

// Byte offset of 16-byte chunk c8 (columns 8 c8 .. 8 c8 + 7) of row i in a
// swizzled K-major matrix of R rows.
__device__ __forceinline__ uint32_t sw128_offset(int R, int i, int c8)
{
    return (uint32_t)((c8 >> 3) * R * 128 + i * 128 + (((c8 & 7) ^ (i & 7)) << 4));
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

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
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

// This thread's bulk copies issued so far have read their source.
__device__ __forceinline__ void bulk_wait_read_all()
{
    asm volatile("cp.async.bulk.commit_group;\ncp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void cp_async_wait_all_groups()
{
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

template <typename T, bool RES, int CS>
__global__ void __launch_bounds__(kUmmaThreads, 1)
rms_gemv_umma(const GemvUmmaParams p, const __grid_constant__ CUtensorMap tmA,
              unsigned int *timeouts)
{
    static_assert(CS == 1 || CS == kUmmaCluster, "no cluster, or the norm shared by one");
    const int NS = p.NS;
    using P = Pack<T, 8>;
    using X = Vals<8>;
    using F = float2;
    // The stage of atom k is refilled with atom k + NS once the MMAs of atom
    // k are done, waited for after the MMAs of atom k + LAG are issued (LAG
    // at most NS - 1): the MMAs' completion overlaps LAG atoms, the copies
    // run NS - LAG atoms ahead. (A lag of 1 measured slower at 64 x 896 ->
    // 9728: 16.3 against 13.9 us.)
    const int LAG = NS > kUmmaLag ? kUmmaLag : NS - 1;
    extern __shared__ __align__(1024) unsigned char umma_smem[];

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int H = p.H, NP = H / 8, NT = p.T;                 // NT: tokens as the MMA's N
    const int f0 = blockIdx.x * kUmmaM;
    const int nk = (H + kUmmaKC - 1) / kUmmaKC;               // K atoms
    const uint32_t raw_s = smem_addr(umma_smem);
    unsigned char *ysm = umma_smem + (((raw_s + 1023u) & ~1023u) - raw_s);   // y atoms
    unsigned char *ring = ysm + gemv_umma_y_bytes(NT, H);     // NS stages of 16 KB
    unsigned char *wsm = ring + NS * kUmmaStageBytes;         // w [H]
    const uint32_t y_s = smem_addr(ysm), ring_s = smem_addr(ring);
    const uint32_t full0 = smem_addr(wsm + gemv_umma_w_bytes(H));   // NS "copy landed"
    const uint32_t empty0 = full0 + 8 * NS;                           // NS "MMAs done"
    int *slots = reinterpret_cast<int *>(wsm + gemv_umma_w_bytes(H) + 16 * NS);
    // slots[0]: tensor-memory address, [1]: atoms multiplied, [2]: a wait ran out
    const uint32_t ybar = smem_addr(slots) + 16;              // y's rows from the cluster
    float *red = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(slots) + 32);
    const uint32_t ncols = gemv_umma_tmem_cols(NT);
    const unsigned long long limit = wait_limit_ns(p.wait_limit_us);
    const bool has_a = f0 < p.N;                              // the grid may be padded to
                                                              // whole clusters
    // The shared norm: 8-row groups g of y, owned by rank g % CS; a CTA
    // receives every group it does not own, one 1024-byte block per atom.
    const int ngroups = NT / 8, na = (H + 63) / 64;
    const int rank = CS > 1 ? (int)cluster_ctarank() : 0;
    const int owned = ngroups > rank ? (ngroups - 1 - rank) / CS + 1 : 0;

    // 1. tensor memory and the stage barriers
    if (warp == 0) {
        tmem_alloc(smem_addr(slots), ncols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        if constexpr (CS > 1) {
            mbar_init(ybar, 1);
            mbar_expect_tx(ybar, (uint32_t)((ngroups - owned) * na * 1024));
        }
    }
    mbar_init_fence();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = static_cast<uint32_t>(slots[0]);
    // Peers write into this CTA's shared memory only once every CTA of the
    // cluster runs with its barriers initialised: arrive now, wait before
    // the first such write.
    if constexpr (CS > 1)
        cluster_arrive_release();

    // 2. copies of A (thread 0: atom kc into stage kc % NS) and of w
    auto issue = [&](int kc, int s) {                          // atom kc into stage s
        mbar_expect_tx(full0 + 8 * s, kUmmaStageBytes + p.extra_tx);
        tma_load_2d(ring_s + s * kUmmaStageBytes, &tmA, kc * kUmmaKC, f0, full0 + 8 * s);
    };
    const int first = nk < NS ? nk : NS;                      // atoms copied up front
    auto prologue = [&]() {
        if (tid == 0 && has_a)
            for (int kc = 0; kc < first; ++kc)
                issue(kc, kc);
        for (int j = tid; j < NP; j += kUmmaThreads)
            cp_async16(wsm + j * 16, static_cast<const uint4 *>(p.w) + j);
    };
    if (p.static_w)
        prologue();
    griddep_wait();
    if (!p.static_w)
        prologue();

    // 3. the norm
    {
        // The norm of this CTA's 8-row groups g = rank, rank + CS, ... (all of
        // them without a cluster): all 256 threads on one group: lane (row %
        // 8, pack % 4), warp w takes packs 4 w + (lane / 8) + 32 u; the row
        // sums of the eight warps meet in shared memory in warp order.
        const bool writer = blockIdx.x < CS;                  // the first cluster
        const int r8 = lane & 7, pj = warp * 4 + (lane >> 3);
        const float fH = (float)H;
        constexpr int kU = kUmmaMaxH / 8 / 32;                // packs per thread, at most
        for (int g = rank; g < ngroups; g += CS) {
            const int t = g * 8 + r8;
            const bool tok = t < p.M;
            const int64_t rb = (int64_t)t * NP;
            P hs[kU];
            F acc = splat<F>(0.f);
            {
                P xs[kU], rsv[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int j = pj + 32 * u;
                    xs[u] = P::zero();
                    rsv[u] = P::zero();
                    if (tok && j < NP) {
                        xs[u] = P::load(p.x, rb + j);
                        if constexpr (RES)
                            rsv[u] = P::load(p.r, rb + j);
                    }
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int j = pj + 32 * u;
                    hs[u] = xs[u];
                    if (tok && j < NP) {
                        X a;
                        if constexpr (RES) {
                            X b;
                            xs[u].widen(a);
                            rsv[u].widen(b);
#pragma unroll
                            for (int i = 0; i < X::N; ++i)
                                a.v[i] = vadd(a.v[i], b.v[i]);
                            hs[u] = P::narrow(a);             // h as stored
                            if (writer && p.h != nullptr)
                                hs[u].store(p.h, rb + j);
                        }
                        hs[u].widen(a);
#pragma unroll
                        for (int i = 0; i < X::N; ++i)
                            acc = vfma(a.v[i], a.v[i], acc);
                    }
                }
            }
            float ss = hsum(acc);
            ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 8);
            ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 16);
            if (lane < 8)
                red[warp * 8 + lane] = ss;
            if (g == rank) {       // w is in (every thread's copies of it)
                cp_async_wait_all_groups();
            }
            __syncthreads();
            float tot = 0.f;
#pragma unroll
            for (int q = 0; q < kUmmaThreads / 32; ++q)
                tot += red[q * 8 + r8];
            const float rs = rsqrtf(tot / fH + p.eps);
            if (tok && writer && pj == 0 && p.rstd != nullptr)
                p.rstd[t] = rs;
            const F r2 = splat<F>(rs);
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int j = pj + 32 * u;
                if (j >= NP)
                    break;
                P yv = P::zero();
                if (tok) {
                    P wp;
                    wp.u = *reinterpret_cast<const uint4 *>(wsm + j * 16);
                    X a, wv;
                    hs[u].widen(a);
                    wp.widen(wv);
#pragma unroll
                    for (int i = 0; i < X::N; ++i)
                        a.v[i] = vmul(vmul(a.v[i], r2), wv.v[i]);
                    yv = P::narrow(a);
                    if (writer && p.y != nullptr)
                        yv.store(p.y, rb + j);
                }
                *reinterpret_cast<uint4 *>(ysm + sw128_offset(NT, t, j)) = yv.u;
            }
            __syncthreads();       // the row sums' slots are reused by the next group
        }
        if (owned == 0) {          // w unused here, but its copies must land
            cp_async_wait_all_groups();
        }
    }
    // every input but A is read: the next kernel may be scheduled; this
    // CTA's part of y is complete (and, fenced, visible to the async proxy:
    // the tensor cores and the bulk copies)
    griddep_launch_dependents();
    fence_proxy_async_smem();
    __syncthreads();
    bool y_failed = false;
    if constexpr (CS > 1) {
        // send each owned group's block of every atom to the other CTAs,
        // then wait for theirs
        cluster_wait_acquire();
        const int ncopy = owned * na * (CS - 1);
        for (int i = tid; i < ncopy; i += kUmmaThreads) {
            const int d = 1 + i % (CS - 1), rest = i / (CS - 1);
            const int a = rest % na, g = rank + (rest / na) * CS;
            const uint32_t off = (uint32_t)(a * NT * 128 + g * 1024);
            const uint32_t peer = (uint32_t)((rank + d) % CS);
            bulk_s2s_cluster(cluster_map(y_s + off, peer), y_s + off, 1024,
                             cluster_map(ybar, peer));
        }
        const bool ok = mbar_wait_bounded(ybar, 0, limit);
        y_failed = __syncthreads_or(!ok);
    }

    // 4. thread 0 walks the K atoms: MMAs as each atom lands, the stage of
    //    the atom before refilled once its MMAs are done
    if (tid == 0) {
        const uint32_t idesc = umma_idesc_f16(UmmaFormat<T>::value, kUmmaM, NT);
        int loaded = has_a ? first : 0;                       // atoms whose copy started
        int kc = 0;
        bool failed = y_failed;
        tc_fence_after_sync();
        // stage and phase parity of atom kc, and of atom kc - LAG (the one
        // refilled), advanced without dividing
        int s = 0, ps = 0;
        uint32_t ph = 0, pph = 0;
        for (; has_a && !failed && kc < nk; ++kc) {
            if (!mbar_wait_bounded(full0 + 8 * s, ph, limit)) {
                failed = true;
                break;
            }
            tc_fence_after_sync();
            const int ksteps = min(kUmmaKC, H - kc * kUmmaKC) / 16;
            for (int k4 = 0; k4 < ksteps; ++k4) {
                const uint64_t ad = umma_desc_sw128(ring_s + s * kUmmaStageBytes + k4 * 32);
                const uint64_t bd = umma_desc_sw128(y_s + kc * NT * 128 + k4 * 32);
                umma_f16(tmem, ad, bd, idesc, (kc | k4) != 0 ? 1u : 0u);
            }
            umma_commit(empty0 + 8 * s);
            if (kc >= LAG) {
                if (kc - LAG + NS < nk) {
                    if (!mbar_wait_bounded(empty0 + 8 * ps, pph, limit)) {
                        failed = true;
                        ++kc;                                 // atom kc's MMAs were issued
                        break;
                    }
                    issue(kc - LAG + NS, ps);                 // the same stage
                    ++loaded;
                }
                if (++ps == NS) {
                    ps = 0;
                    pph ^= 1u;
                }
            }
            if (++s == NS) {
                s = 0;
                ph ^= 1u;
            }
        }
        slots[1] = kc;                                        // atoms whose MMAs were issued
        slots[2] = failed ? 1 : 0;
        if (failed)            // let the copies started and not waited for land
            for (int q = kc; q < loaded; ++q)
                (void)mbar_wait_bounded(full0 + 8 * (q % NS), (uint32_t)((q / NS) & 1), limit);
    }
    __syncthreads();
    const int issued = slots[1];
    const bool failed = slots[2] != 0;

    // 5. the accumulator, once the last issued atom's MMAs (and with them
    //    every earlier one) are complete
    bool done = true;
    if (issued > 0) {
        const int lc = issued - 1;
        const bool ok = mbar_wait_bounded(empty0 + 8 * (lc % NS), (uint32_t)((lc / NS) & 1), limit);
        done = !__syncthreads_or(!ok);
    }
    if (failed || !done) {
        if (tid == 0)
            atomicAdd(timeouts, 1u);
    } else {
        tc_fence_after_sync();
        const int q4 = warp & 3;                              // lane quarter
        const int f = f0 + q4 * 32 + lane;
        const uint32_t tw = tmem + ((uint32_t)(q4 * 32) << 16);
        for (int c0 = 16 * (warp >> 2); c0 < NT; c0 += 32) {  // token blocks by warp pair
            uint32_t v[16];
            tmem_ld16(tw + (uint32_t)c0, v);
            if (f < p.N) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int t = c0 + i;
                    if (t < p.M) {
                        Vals<1> o;
                        o.v[0] = __uint_as_float(v[i]);
                        Pack<T, 1>::narrow(o).store(p.out, (int64_t)t * p.N + f);
                    }
                }
            }
        }
    }

    // 6. with a cluster: this CTA's copies have read their source, the
    //    others' copies into it have landed (waited for again, bounded, if
    //    that wait ran out), and no CTA leaves before all are done
    if constexpr (CS > 1) {
        if (y_failed && tid == 0)
            (void)mbar_wait_bounded(ybar, 0, limit);
        bulk_wait_read_all();
        cluster_arrive_release();
        cluster_wait_acquire();
    }
    // free the tensor memory (every tcgen05 access of the CTA is ordered
    // before it by the barrier)
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, ncols);
    }
}

} // namespace rmsk
