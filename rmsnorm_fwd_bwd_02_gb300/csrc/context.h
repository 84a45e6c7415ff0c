// context.h -- the identity of the CUDA context current on the calling
// thread, for the library's per-device caches (device addresses of its
// __device__ variables, kernels' shared-memory attributes and occupancy).
// Those belong to a context: after cudaDeviceReset the runtime creates a new
// primary context, in which a cached address would dangle and a kernel's
// raised shared-memory limit is back at its default. Every cache entry is
// therefore stored with the context it was made in and used only while that
// context is current.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

namespace rmsk {

// Unique identifier (cuCtxGetId) of the current context, never reused
// within the process; 0 when no context is current yet or the driver does
// not offer the query (callers then look everything up afresh).
inline unsigned long long current_context_id()
{
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    });
    if (get_current == nullptr || get_id == nullptr)
        return 0;
    CUcontext c = nullptr;
    if (get_current(&c) != CUDA_SUCCESS || c == nullptr)
        return 0;
    unsigned long long id = 0;
    if (get_id(c, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

} // namespace rmsk
