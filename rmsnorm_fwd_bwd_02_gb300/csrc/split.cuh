// split.cuh -- split-row forward for decode-sized batches (M <= 64 rows).
//
// [P2] (the 0.8B Qwen decode article, trdm.cn news/483216) §3.2 spreads the
// sum of squares of one hidden-896 row over SPLIT_K programs, merges the
// fp32 partials in a one-block reduce kernel and scales in a third kernel;
// §3.3 keeps partials and merge in fp32 and avoids atomics. Here the same
// split runs as ONE kernel: a thread-block cluster of K CTAs per row. Each
// CTA loads its slice of the row into registers, reduces its partial sum of
// squares and stores it into every CTA of the cluster (asynchronous stores
// into distributed shared memory that complete on the receiver's mbarrier,
// so no cluster-wide barrier sits between the sums and the scaling); once
// the K - 1 words from its peers have landed, every CTA adds the K partials
// in rank order 0..K-1, so all CTAs of the row compute the same rstd bits.
// Then each CTA scales and stores its slice. One phase of the cluster
// barrier, arrived at after the set-up and waited for just before the
// stores, makes sure every CTA's mbarrier exists by then. The wait for the
// peers' words is bounded (about one second; one that runs out counts in
// the timeout counter). No TMA and no multicast are involved.
#pragma once

#include "common.cuh"
#include "params.h"
#include "stream.cuh"

namespace rmsk {

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on the cluster barrier without ordering memory accesses: for a
// phase that only says "this CTA got here" (for instance, done reading the
// peers' shared memory: loads whose values this thread has already used are
// complete). A release here would first wait for the thread's memory
// traffic still in flight.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

// Read a float that CTA `rank` of this cluster holds at the same shared
// memory offset as `local` does in this CTA.
__device__ __forceinline__ float ld_cluster_f32(const float *local, uint32_t rank)
{
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(local);
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}

// The sum over the n <= 8 CTAs of the cluster of the float each holds at
// `local`'s offset, added in rank order. All loads are issued before the
// first add, so the n remote round trips overlap.
__device__ __forceinline__ float sum_cluster_f32(const float *local, uint32_t n)
{
    float v[8];
#pragma unroll
    for (uint32_t q = 0; q < 8; ++q)
        if (q < n)
            v[q] = ld_cluster_f32(local, q);
    float s = 0.f;
#pragma unroll
    for (uint32_t q = 0; q < 8; ++q)
        if (q < n)
            s += v[q];
    return s;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// Store one 32-bit word into a peer's shared memory (cluster address) and
// count its 4 bytes on the peer's mbarrier (cluster address): the word is
// visible to the peer's threads once they see that barrier's phase complete.
__device__ __forceinline__ void st_async_b32(uint32_t cluster_addr, uint32_t v,
                                             uint32_t cluster_bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(
                     cluster_addr),
                 "r"(v), "r"(cluster_bar)
                 : "memory");
}

// Store 16 bytes (four floats) into a peer's shared memory (cluster
// address, 16-byte aligned) and count them on the peer's mbarrier.
__device__ __forceinline__ void st_async_v4(uint32_t cluster_addr, float4 v, uint32_t cluster_bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, "
                 "%4}, [%5];" ::"r"(cluster_addr),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(cluster_bar)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Bounded wait with acquire at cluster scope (for barriers that peers of the
// cluster complete); false if the phase has not completed within limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                          unsigned long long limit_ns)
{
    if (mbar_try_wait_cluster(bar, parity))
        return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait_cluster(bar, parity))
        if (global_ns() - t0 > limit_ns)
            return false;
    return true;
}

// grid = (K, M), cluster = (K, 1, 1), blockDim.x a multiple of 32 (<= 256).
template <typename T, int E, int V, bool RES>
__global__ void __launch_bounds__(256)
rms_fwd_split(const SplitParams p)
{
    using P = Pack<T, E>;
    __shared__ float warp_sum[8];
    __shared__ float sums[8];                          // each CTA's sum of squares, by rank
    __shared__ __align__(8) unsigned long long sbar;   // the peers' sums have landed

    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const uint32_t rank = cluster_ctarank();
    const uint32_t K = cluster_nctarank();
    const int64_t row = blockIdx.y;
    const int v0 = (int)rank * p.SV;
    const int v1 = min(v0 + p.SV, p.NV);
    // first pack of this row in each tensor
    const int64_t bx = row * (p.ldx / E), br = row * (p.ldr / E);
    const int64_t by = row * (p.ldy / E), bh = row * (p.ldh / E);
    const uint32_t sbar_s = (uint32_t)__cvta_generic_to_shared(&sbar);
    if (tid == 0) {
        mbar_init(sbar_s, 1);
        if (K > 1)                 // every other CTA of the cluster stores one word
            mbar_expect_tx(sbar_s, (K - 1) * 4u + p.extra_tx);
    }
    mbar_init_fence();
    __syncthreads();
    // this CTA's barrier exists; the peers store into it only after the
    // matching wait below, so this arrival is not waited for
    cluster_arrive_relaxed();

    griddep_wait();
    P xv[V];
#pragma unroll
    for (int k = 0; k < V; ++k) {
        const int vi = v0 + tid + k * nt;
        xv[k] = vi < v1 ? P::load(p.x, bx + vi) : P::zero();
    }
    if constexpr (RES) {
        P rv[V];
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int vi = v0 + tid + k * nt;
            rv[k] = vi < v1 ? P::load(p.r, br + vi) : P::zero();
        }
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int vi = v0 + tid + k * nt;
            float a[E], b[E];
            xv[k].to_float(a);
            rv[k].to_float(b);
#pragma unroll
            for (int e = 0; e < E; ++e)
                a[e] += b[e];
            xv[k] = P::from_float(a);
            if (vi < v1)
                xv[k].store(p.h, bh + vi);
        }
    }

    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < V; ++k) {
        float f[E];
        xv[k].to_float(f);
#pragma unroll
        for (int e = 0; e < E; ++e)
            ss = fmaf(f[e], f[e], ss);
    }
    ss = group_allreduce<32>(ss);
    if ((tid & 31) == 0)
        warp_sum[tid / 32] = ss;
    __syncthreads();
    cluster_wait_acquire();        // every peer's barrier exists
    if (tid == 0) {
        float s = 0.f;
        for (int q = 0; q < nt / 32; ++q)
            s += warp_sum[q];
        // this CTA's sum, here and in every peer (asynchronous stores that
        // complete on the peer's barrier)
        sums[rank] = s;
        const uint32_t at = (uint32_t)__cvta_generic_to_shared(&sums[rank]);
        for (uint32_t d = 1; d < K; ++d) {
            const uint32_t peer = (rank + d) % K;
            st_async_b32(cluster_map(at, peer), __float_as_uint(s), cluster_map(sbar_s, peer));
        }
        if (K > 1 && !mbar_wait_bounded_cluster(sbar_s, 0, wait_limit_ns(p.wait_limit_us)))
            atomicAdd(p.timeouts, 1u);
    }
    __syncthreads();
    griddep_launch_dependents();
    float total = 0.f;
    for (uint32_t q = 0; q < K; ++q)   // rank order
        total += sums[q];

    const float rs = rsqrtf(total / (float)p.H + p.eps);
    if (rank == 0 && tid == 0 && p.rstd != nullptr)
        p.rstd[row] = rs;
#pragma unroll
    for (int k = 0; k < V; ++k) {
        const int vi = v0 + tid + k * nt;
        if (vi >= v1)
            continue;
        float f[E], fw[E];
        xv[k].to_float(f);
        P::load_cached(p.w, vi).to_float(fw);
#pragma unroll
        for (int e = 0; e < E; ++e)
            f[e] = f[e] * rs * fw[e];
        P::from_float(f).store(p.y, by + vi);
    }
}

} // namespace rmsk
