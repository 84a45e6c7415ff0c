// Streamed (bulk-copy fed) row kernels for fp16 rows of the shaped feature
// counts: the bf16 layouts of stream.cu with fp16 storage.
#include "registry.h"
#include "stream.cuh"
#include "stream_small.cuh"

namespace rmsk {
//           name      type  H     |-- forward: GW V NG NS --| |-- backward: GW V NG NS HOLD --| |-- double bwd --|
RMSK_STREAM(sh_h4096, f16, 4096,   4, 4, 4, 4,               8, 2, 2, 6, true,            8, 2, 1, 8)
RMSK_STREAM(sh_h5120, f16, 5120,   4, 5, 3, 3,              10, 2, 2, 3, false,          10, 2, 1, 6)

//          name     type  H    |- forward: RPT NW NS -| |- backward: RPT NW NS -|
RMSK_SMALL(sh_h128, f16, 128,       4,   16,  4,              8,   8,  3)
} // namespace rmsk
