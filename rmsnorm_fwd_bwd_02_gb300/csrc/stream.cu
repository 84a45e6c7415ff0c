// Streamed (bulk-copy fed) row kernels for the shaped bf16 feature counts,
// and the device counter of bounded waits that ran out (the fp16 kernels,
// in stream_f16.cu, count into the same one).
#include <cuda_runtime.h>

#include <mutex>

#include "context.h"
#include "registry.h"
#include "stream.cuh"
#include "stream_small.cuh"

namespace rmsk {

namespace {
__device__ unsigned int g_stream_timeouts;
std::mutex g_mu;
unsigned int *g_addr[64] = {};
unsigned long long g_ctx[64] = {};    // the context each address belongs to
} // namespace

// The counter's device address on device `dev` (current), looked up once
// per context (context.h).
unsigned int *stream_timeout_counter(int dev)
{
    if (dev < 0 || dev >= 64)
        return nullptr;
    std::lock_guard<std::mutex> g(g_mu);
    const unsigned long long ctx = current_context_id();
    if (g_addr[dev] == nullptr || ctx == 0 || g_ctx[dev] != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_stream_timeouts) != cudaSuccess)
            return nullptr;
        g_addr[dev] = static_cast<unsigned int *>(p);
        g_ctx[dev] = current_context_id();
    }
    return g_addr[dev];
}

// Stage counts are upper bounds: variants that stage more tensors per row get
// as many stages as fit in shared memory (StreamSmem).
// The double backward reads three tensors per row; it runs best with one
// group per CTA and a deep ring (8 stages of 24 KB at H = 4096, 6 of 30 KB at
// H = 5120: 206 and 204 us at 32768 x 4096 and 26214 x 5120 on GB300, against
// 234 us for two groups of 4 stages).
//           name    type   H     |-- forward: GW V NG NS --| |-- backward: GW V NG NS HOLD --| |-- double bwd --|
RMSK_STREAM(s_h4096, bf16, 4096,   4, 4, 4, 4,               8, 2, 2, 6, true,            8, 2, 1, 8)
RMSK_STREAM(s_h5120, bf16, 5120,   4, 5, 3, 3,              10, 2, 2, 3, false,          10, 2, 1, 6)

// 128-wide rows (QK-norm): warps with their own rings of row blocks.
//          name    type   H    |- forward: RPT NW NS -| |- backward: RPT NW NS -|
RMSK_SMALL(s_h128, bf16, 128,       4,   16,  4,              8,   8,  3)

} // namespace rmsk
