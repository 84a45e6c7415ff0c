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
//  3. The norm of every token, by all eight warps in rounds of eight 8-row
//     groups; lane (row % 8, pack % 4) so that the 16-byte stores into the
//     swizzled layout of y hit 8 different chunk positions per quarter warp,
//     and a lane loads 16 packs of x (and r) before using any. Pass one adds
//     r, rounds h, stores it in place of y and sums the squares (the four
//     lanes of a row combine by shuffles); pass two scales the stored h by
//     rstd and w and rounds y. The first CTA also writes h, y and rstd.
//  4. Thread 0 alone walks the K atoms: wait for the atom's copy (full
//     barrier), issue four MMAs (m128 nT k16) and commit them to the stage's
//     empty barrier, then refill the stage the atom `lag` before used once
//     its MMAs are done.
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
#include "stream.cuh"

namespace rmsk {

constexpr int kUmmaM = 128;        // output features per CTA (the MMA's M)
constexpr int kUmmaKC = 64;        // K columns per ring stage: one swizzle atom
constexpr int kUmmaThreads = 256;  // eight warps; warp w reads tensor-memory lanes
                                   // 32 (w % 4) .. 32 (w % 4) + 31
constexpr int kUmmaMaxH = 2048;    // the norm holds no row in registers; the
                                   // limit is shared memory (y beside the ring)
constexpr uint32_t kUmmaStageBytes = kUmmaM * kUmmaKC * 2;   // 16 KB
// The stage of atom k is refilled (with atom k + NS) once the MMAs of atom
// k are done, waited for after the MMAs of atom k + lag are issued (lag =
// kUmmaLag, at most NS - 1): the MMAs' latency overlaps lag atoms, the
// copies run NS - lag atoms ahead.
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
// 2 NS mbarriers, the tensor-memory address.
__host__ __device__ constexpr int64_t gemv_umma_smem_bytes(int T, int H, int NS)
{
    return 1024 + gemv_umma_y_bytes(T, H) + (int64_t)NS * kUmmaStageBytes +
           gemv_umma_w_bytes(H) + 16 * NS + 16;
}

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

__device__ __forceinline__ void cp_async_wait_all_groups()
{
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

template <typename T, bool RES, int NS>
__global__ void __launch_bounds__(kUmmaThreads, 1)
rms_gemv_umma(const GemvUmmaParams p, const __grid_constant__ CUtensorMap tmA,
              unsigned int *timeouts)
{
    using P = Pack<T, 8>;
    using X = Vals<8>;
    using F = float2;
    static_assert(NS >= 2, "an atom is copied while the one before is multiplied");
    // the refill lag stays below the ring depth: atom k + NS goes into the
    // stage of atom k, and must be copied before the loop needs it
    constexpr int LAG = kUmmaLag < NS ? kUmmaLag : NS - 1;
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
    const uint32_t ncols = gemv_umma_tmem_cols(NT);
    const unsigned long long limit = wait_limit_ns(p.wait_limit_us);

    // 1. tensor memory and the stage barriers
    if (warp == 0) {
        tmem_alloc(smem_addr(slots), ncols);
        tmem_relinquish();
    }
    if (tid == 0)
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
    mbar_init_fence();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = static_cast<uint32_t>(slots[0]);

    // 2. copies of A (thread 0: atom kc into stage kc % NS) and of w
    auto issue = [&](int kc) {
        const int s = kc % NS;
        mbar_expect_tx(full0 + 8 * s, kUmmaStageBytes + p.extra_tx);
        tma_load_2d(ring_s + s * kUmmaStageBytes, &tmA, kc * kUmmaKC, f0, full0 + 8 * s);
    };
    const int first = nk < NS ? nk : NS;                      // atoms copied up front
    auto prologue = [&]() {
        if (tid == 0)
            for (int kc = 0; kc < first; ++kc)
                issue(kc);
        for (int j = tid; j < NP; j += kUmmaThreads)
            cp_async16(wsm + j * 16, static_cast<const uint4 *>(p.w) + j);
    };
    if (p.static_w)
        prologue();
    griddep_wait();
    if (!p.static_w)
        prologue();

    // 3. the norm, in rounds of four 8-row groups: warp `warp` takes group
    //    g0 + warp; lane = (row % 8) + 8 (pack % 4). A lane's packs of x (and
    //    r) are loaded kNormBatch at a time, so that many reads are in
    //    flight; w comes from shared memory (waited for once, after the first
    //    pass one).
    const bool writer = blockIdx.x == 0;
    const int r8 = lane & 7, jq = lane >> 3;
    const float fH = (float)H;
    constexpr int kNormBatch = 16, kScaleBatch = 8;   // packs in flight per lane
    for (int g0 = 0; g0 < NT / 8; g0 += kUmmaThreads / 32) {
        const int g = g0 + warp;
        const bool gv = g < NT / 8;
        const int t = g * 8 + r8;
        const bool tok = gv && t < p.M;
        const int64_t rb = (int64_t)t * NP;
        F acc = splat<F>(0.f);
        for (int j0 = jq; gv && j0 < NP; j0 += 4 * kNormBatch) {
            P xs[kNormBatch], rsv[kNormBatch];
#pragma unroll
            for (int u = 0; u < kNormBatch; ++u) {
                const int j = j0 + 4 * u;
                xs[u] = P::zero();
                rsv[u] = P::zero();
                if (tok && j < NP) {
                    xs[u] = P::load(p.x, rb + j);
                    if constexpr (RES)
                        rsv[u] = P::load(p.r, rb + j);
                }
            }
#pragma unroll
            for (int u = 0; u < kNormBatch; ++u) {
                const int j = j0 + 4 * u;
                if (j >= NP)
                    break;
                P hv = xs[u];
                if (tok) {
                    X a;
                    if constexpr (RES) {
                        X b;
                        xs[u].widen(a);
                        rsv[u].widen(b);
#pragma unroll
                        for (int i = 0; i < X::N; ++i)
                            a.v[i] = vadd(a.v[i], b.v[i]);
                        hv = P::narrow(a);                    // h as stored
                        if (writer && p.h != nullptr)
                            hv.store(p.h, rb + j);
                    }
                    hv.widen(a);
#pragma unroll
                    for (int i = 0; i < X::N; ++i)
                        acc = vfma(a.v[i], a.v[i], acc);
                }
                *reinterpret_cast<uint4 *>(ysm + sw128_offset(NT, t, j)) = hv.u;
            }
        }
        float ss = hsum(acc);
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 8);
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 16);
        const float rs = rsqrtf(ss / fH + p.eps);
        if (tok && writer && jq == 0 && p.rstd != nullptr)
            p.rstd[t] = rs;
        if (g0 == 0) {             // w is in (every thread's copies of it)
            cp_async_wait_all_groups();
            __syncthreads();
        }
        if (tok) {
            const F r2 = splat<F>(rs);
            for (int j0 = jq; j0 < NP; j0 += 4 * kScaleBatch) {
                P hs[kScaleBatch], ws[kScaleBatch];
#pragma unroll
                for (int u = 0; u < kScaleBatch; ++u) {
                    const int j = j0 + 4 * u;
                    if (j < NP) {
                        hs[u].u = *reinterpret_cast<const uint4 *>(ysm + sw128_offset(NT, t, j));
                        ws[u].u = *reinterpret_cast<const uint4 *>(wsm + j * 16);
                    }
                }
#pragma unroll
                for (int u = 0; u < kScaleBatch; ++u) {
                    const int j = j0 + 4 * u;
                    if (j >= NP)
                        break;
                    X a, wv;
                    hs[u].widen(a);
                    ws[u].widen(wv);
#pragma unroll
                    for (int i = 0; i < X::N; ++i)
                        a.v[i] = vmul(vmul(a.v[i], r2), wv.v[i]);
                    const P yv = P::narrow(a);
                    *reinterpret_cast<uint4 *>(ysm + sw128_offset(NT, t, j)) = yv.u;
                    if (writer && p.y != nullptr)
                        yv.store(p.y, rb + j);
                }
            }
        }
    }
    // every input but A is read: the next kernel may be scheduled; y is
    // complete (and, fenced, visible to the tensor cores' reads)
    griddep_launch_dependents();
    fence_proxy_async_smem();
    __syncthreads();

    // 4. thread 0 walks the K atoms: MMAs as each atom lands, the stage of
    //    the atom before refilled once its MMAs are done
    if (tid == 0) {
        const uint32_t idesc = umma_idesc_f16(UmmaFormat<T>::value, kUmmaM, NT);
        int loaded = first;                                   // atoms whose copy started
        int kc = 0;
        bool failed = false;
        tc_fence_after_sync();
        for (; kc < nk; ++kc) {
            const int s = kc % NS;
            if (!mbar_wait_bounded(full0 + 8 * s, (uint32_t)((kc / NS) & 1), limit)) {
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
            if (kc >= LAG && kc - LAG + NS < nk) {
                const int pc = kc - LAG;
                if (!mbar_wait_bounded(empty0 + 8 * (pc % NS), (uint32_t)((pc / NS) & 1),
                                       limit)) {
                    failed = true;
                    ++kc;                                     // atom kc's MMAs were issued
                    break;
                }
                issue(pc + NS);
                ++loaded;
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

    // 6. free the tensor memory (every tcgen05 access of the CTA is ordered
    //    before it by the barrier)
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, ncols);
    }
}

} // namespace rmsk
