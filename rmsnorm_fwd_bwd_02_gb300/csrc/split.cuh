// split.cuh -- split-row forward for decode-sized batches (M <= 64 rows).
//
// [P2] (the 0.8B Qwen decode article, trdm.cn news/483216) §3.2 spreads the
// sum of squares of one hidden-896 row over SPLIT_K programs, merges the
// fp32 partials in a one-block reduce kernel and scales in a third kernel;
// §3.3 keeps partials and merge in fp32 and avoids atomics. Here the same
// split runs as ONE kernel: a thread-block cluster of K CTAs per row. Each
// CTA loads its slice of the row into registers, reduces its partial sum of
// squares, publishes it in its own shared memory, and after a cluster
// barrier every CTA reads all K partials through distributed shared memory
// and adds them in rank order 0..K-1, so all CTAs of the row compute the
// same rstd bits. Then each CTA scales and stores its slice. No TMA and no
// multicast are involved; the waits are the hardware cluster barrier.
#pragma once

#include "common.cuh"
#include "params.h"

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

// grid = (K, M), cluster = (K, 1, 1), blockDim.x a multiple of 32 (<= 256).
template <typename T, int E, int V, bool RES>
__global__ void __launch_bounds__(256)
rms_fwd_split(const SplitParams p)
{
    using P = Pack<T, E>;
    __shared__ float warp_sum[8];
    __shared__ float cta_sum;

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
    if (tid == 0) {
        float s = 0.f;
        for (int q = 0; q < nt / 32; ++q)
            s += warp_sum[q];
        cta_sum = s;
    }

    cluster_arrive_release();   // publish cta_sum to the cluster
    cluster_wait_acquire();
    const float total = sum_cluster_f32(&cta_sum, K);   // rank order
    cluster_arrive_relaxed();   // this CTA is done reading the others
    griddep_launch_dependents();

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
    // Keep this CTA's shared memory alive until every CTA has read cta_sum.
    cluster_wait_acquire();
}

} // namespace rmsk
