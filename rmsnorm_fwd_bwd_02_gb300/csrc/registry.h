// registry.h -- the instantiated kernel configurations the C ABI dispatches
// to. Each RowKernels entry is one row layout (see rows.cuh) with its four
// kernels; each SplitKernels entry is one element type of the split-row
// forward (see split.cuh).
#pragma once

namespace rmsk {

struct RowKernels {
    const char *name;
    int E;       // elements per pack (8 bf16 / 4 fp32 vectorised, 1 scalar)
    int L;       // lanes per row group
    int V;       // packs per lane
    int G;       // rows per group per iteration
    int S;       // row groups per CTA
    bool exact;  // H == L * V * E (no column masking)
    const void *fwd, *fwd_res, *bwd, *bwd_dh;
    int threads() const { return L * S; }
    int tile_rows() const { return S * G; }
    long long max_cols() const { return (long long)L * V * E; }
};

struct SplitKernels {
    int E;
    const void *v1, *v1_res;   // one pack per thread
    const void *v8, *v8_res;   // up to eight packs per thread
};

// bf16, 16-byte packs. Named for the feature count they are shaped for
// (hNNN, exact) or the largest pack count per row they cover (gNNN lanes x 4).
extern const RowKernels b_h128, b_h896, b_h4096, b_h5120, b_g32, b_g128, b_g512;
// bf16, one element per access (rows not 16-byte aligned, odd H)
extern const RowKernels b_s32, b_s1024;
// fp32, 16-byte packs
extern const RowKernels f_h896, f_g32, f_g128, f_g512;
// fp32, one element per access
extern const RowKernels f_s32, f_s1024;

extern const SplitKernels split_bf16_v, split_bf16_s, split_f32_v, split_f32_s;

} // namespace rmsk

#define RMSK_ROWS(NAME, T, E, L, V, G, S, MINB, EXACT)                             \
    const RowKernels NAME = {                                                     \
        #NAME, E, L, V, G, S, EXACT,                                              \
        (const void *)&rms_fwd_rows<T, E, L, V, G, S, MINB, EXACT, false>,        \
        (const void *)&rms_fwd_rows<T, E, L, V, G, S, MINB, EXACT, true>,         \
        (const void *)&rms_bwd_rows<T, E, L, V, G, S, MINB, EXACT, false>,        \
        (const void *)&rms_bwd_rows<T, E, L, V, G, S, MINB, EXACT, true>};

#define RMSK_SPLIT(NAME, T, E)                                                    \
    const SplitKernels NAME = {                                                   \
        E,                                                                        \
        (const void *)&rms_fwd_split<T, E, 1, false>,                             \
        (const void *)&rms_fwd_split<T, E, 1, true>,                              \
        (const void *)&rms_fwd_split<T, E, 8, false>,                             \
        (const void *)&rms_fwd_split<T, E, 8, true>};
