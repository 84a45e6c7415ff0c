// registry.h -- the instantiated kernel configurations the C ABI dispatches
// to. A RowKernels entry pairs a forward layout and a backward layout (see
// rows.cuh; the best shapes differ) with their kernels; a SplitKernels
// entry is one element type of the split-row forward (see split.cuh).
#pragma once

namespace rmsk {

struct RowShape {
    int E;       // elements per pack (16/8 bf16 or 8/4 fp32 vectorised, 1 scalar)
    int L;       // lanes per row group
    int V;       // packs per lane
    int G;       // rows per group per iteration
    int S;       // row groups per CTA
    bool exact;  // H == L * V * E (no column masking)
    int threads() const { return L * S; }
    int tile_rows() const { return S * G; }
    long long cols() const { return (long long)L * V * E; }
};

struct RowKernels {
    const char *name;
    RowShape f, b;           // forward and backward layouts
    const void *fwd[2];      // [residual]
    const void *bwd[2][2];   // [dh_out given][rstd given]
    long long max_cols() const { return f.cols() < b.cols() ? f.cols() : b.cols(); }
    // bytes of one pack, for the alignment a call needs
    int align(int elem_bytes) const
    {
        const int a = f.E > b.E ? f.E : b.E;
        return a * elem_bytes;
    }
};

// A streamed (bulk-copy fed) layout, 16-bit formats only: the CTA's threads and the
// rows a CTA takes per round (stream.cuh: NG groups, one row each;
// stream_small.cuh: NW warps, one block of rows each).
struct StreamShape {
    int threads_;
    int rows;
    int threads() const { return threads_; }
};

struct StreamKernels {
    const char *name;
    int H;
    StreamShape f, b, d;       // forward, backward, double backward
    const void *fwd[2];        // [residual]
    int fwd_smem[2];
    const void *bwd[2][2];     // [dh_out given][rstd given]
    int bwd_smem[2][2];
    const void *bwd2[2];       // double backward [rstd given], or nullptr
    int bwd2_smem[2];
};

struct SplitKernels {
    int E;
    const void *v1, *v1_res;   // one pack per thread
    const void *v8, *v8_res;   // up to eight packs per thread
};

// bf16, 16-byte packs. Named for the feature count they are shaped for
// (hNNN, exact) or the lanes of their masked layouts (gNNN).
extern const RowKernels b_h128, b_h896, b_h4096, b_h5120, b_g32, b_g128, b_g512;
// bf16 shaped layouts whose forward moves 32-byte packs (rows 32-byte aligned)
extern const RowKernels b_h128w, b_h4096w, b_h5120w;
// bf16, one element per access (rows not 16-byte aligned, odd H)
extern const RowKernels b_s32, b_s1024;
// fp16: the same layouts as bf16
extern const RowKernels h_h128, h_h896, h_h4096, h_h5120, h_g32, h_g128, h_g512;
extern const RowKernels h_h128w, h_h4096w, h_h5120w;
extern const RowKernels h_s32, h_s1024;
// fp32, 16-byte packs
extern const RowKernels f_h896, f_g32, f_g128, f_g512;
// fp32, one element per access
extern const RowKernels f_s32, f_s1024;

extern const SplitKernels split_bf16_v, split_bf16_s, split_f32_v, split_f32_s;
extern const SplitKernels split_f16_v, split_f16_s;

// streamed layouts: bf16 (s_) and fp16 (sh_)
extern const StreamKernels s_h4096, s_h5120, s_h128;
extern const StreamKernels sh_h4096, sh_h5120, sh_h128;

// Double backward (bwd2.cuh): one layout and its kernel.
struct Bwd2Kernel {
    const char *name;
    RowShape s;
    const void *fn;
};
extern const Bwd2Kernel b2_bf_g32, b2_bf_g128, b2_bf_h4096, b2_bf_g512, b2_bf_s1024;
extern const Bwd2Kernel b2_h_g32, b2_h_g128, b2_h_h4096, b2_h_g512, b2_h_s1024;
extern const Bwd2Kernel b2_f_g32, b2_f_g128, b2_f_g512, b2_f_s1024;

// RMSNorm fused with the projection GEMV (gemv.cuh):
// fn[bf16 = 0, fp16 = 1][y tile: 0 = 8 rows (M <= 8), k = k 16-row tiles]
//   [0 plain, 1 residual (r from L2), 2 residual (r staged in shared memory)]
struct GemvKernels {
    const void *fn[2][5][3];
};
extern const GemvKernels gemv_kernels;       // A in registers (gemv.cuh)
extern const GemvKernels gemv_tma_kernels;   // A by bulk copies (gemv_tma.cuh)
// The product on tcgen05, K split over a cluster (gemv_umma.cuh):
// fn[bf16 = 0, fp16 = 1][residual]
struct GemvUmmaKernels {
    const void *fn[2][2];
};
extern const GemvUmmaKernels gemv_umma_kernels;
// Persistent, K optionally split over a cluster (gemv_tc.cuh):
// fn[bf16 = 0, fp16 = 1][residual][partials stored directly (<= 48 tokens)]
struct GemvTcKernels {
    const void *fn[2][2][2];
};
extern const GemvTcKernels gemv_tc_kernels;
// Device address of the counter of streamed-kernel waits that ran out.
unsigned int *stream_timeout_counter(int dev);

} // namespace rmsk

// RMSK_ROWS2(name, type, forward E L V G S MINB exact, backward E L V G S MINB exact)
#define RMSK_ROWS2(NAME, T, FE, FL, FV, FG, FS, FMB, FEX, BE, BL, BV, BG, BS, BMB, BEX)    \
    const RowKernels NAME = {                                                            \
        #NAME, {FE, FL, FV, FG, FS, FEX}, {BE, BL, BV, BG, BS, BEX},                     \
        {(const void *)&rms_fwd_rows<T, FE, FL, FV, FG, FS, FMB, FEX, false>,            \
         (const void *)&rms_fwd_rows<T, FE, FL, FV, FG, FS, FMB, FEX, true>},            \
        {{(const void *)&rms_bwd_rows<T, BE, BL, BV, BG, BS, BMB, BEX, false, false>,    \
          (const void *)&rms_bwd_rows<T, BE, BL, BV, BG, BS, BMB, BEX, false, true>},    \
         {(const void *)&rms_bwd_rows<T, BE, BL, BV, BG, BS, BMB, BEX, true, false>,     \
          (const void *)&rms_bwd_rows<T, BE, BL, BV, BG, BS, BMB, BEX, true, true>}}};

// Same pack width in both directions.
#define RMSK_ROWS(NAME, T, E, FL, FV, FG, FS, FMB, FEX, BL, BV, BG, BS, BMB, BEX)          \
    RMSK_ROWS2(NAME, T, E, FL, FV, FG, FS, FMB, FEX, E, BL, BV, BG, BS, BMB, BEX)

#define RMSK_STREAM(NAME, T, H, FGW, FV, FNG, FNS, BGW, BV, BNG, BNS, BH, DGW, DV, DNG, DNS) \
    static_assert(32 * FGW * FV * 8 == H && 32 * BGW * BV * 8 == H &&                    \
                      32 * DGW * DV * 8 == H,                                            \
                  "stream layout");                                                      \
    const StreamKernels NAME = {                                                         \
        #NAME, H, {FNG * FGW * 32, FNG}, {BNG * BGW * 32, BNG}, {DNG * DGW * 32, DNG},   \
        {(const void *)&rms_fwd_stream<T, FGW, FV, FNG, FNS, false>,                     \
         (const void *)&rms_fwd_stream<T, FGW, FV, FNG, FNS, true>},                     \
        {StreamSmem<FGW, FV, FNG, FNS, 1, 1>::kBytes,                                    \
         StreamSmem<FGW, FV, FNG, FNS, 2, 1>::kBytes},                                   \
        {{(const void *)&rms_bwd_stream<T, BGW, BV, BNG, BNS, false, false, BH>,         \
          (const void *)&rms_bwd_stream<T, BGW, BV, BNG, BNS, false, true, BH>},         \
         {(const void *)&rms_bwd_stream<T, BGW, BV, BNG, BNS, true, false, BH>,          \
          (const void *)&rms_bwd_stream<T, BGW, BV, BNG, BNS, true, true, BH>}},         \
        {{StreamSmem<BGW, BV, BNG, BNS, 2, 2>::kBytes,                                   \
          StreamSmem<BGW, BV, BNG, BNS, 2, 1>::kBytes},                                  \
         {StreamSmem<BGW, BV, BNG, BNS, 3, 2>::kBytes,                                   \
          StreamSmem<BGW, BV, BNG, BNS, 3, 1>::kBytes}},                                 \
        {(const void *)&rms_bwd2_stream<T, DGW, DV, DNG, DNS, false>,                    \
         (const void *)&rms_bwd2_stream<T, DGW, DV, DNG, DNS, true>},                    \
        {StreamSmem<DGW, DV, DNG, DNS, 3, bwd2_stream_slots(false)>::kBytes,              \
         StreamSmem<DGW, DV, DNG, DNS, 3, bwd2_stream_slots(true)>::kBytes}};

// Short rows (stream_small.cuh): H = 8 * NVP, NW warps, RPT rows per lane per stage.
// T is the 16-bit storage format.
#define RMSK_SMALL(NAME, T, H, FRPT, FNW, FNS, BRPT, BNW, BNS)                            \
    const StreamKernels NAME = {                                                         \
        #NAME, H, {FNW * 32, FNW * (256 / H) * FRPT}, {BNW * 32, BNW * (256 / H) * BRPT}, \
        {0, 0},                                                                          \
        {(const void *)&rms_fwd_stream_small<T, H / 8, FRPT, FNW, FNS, false>,           \
         (const void *)&rms_fwd_stream_small<T, H / 8, FRPT, FNW, FNS, true>},           \
        {SmallSmem<H / 8, FRPT, FNW, FNS, 1>::kBytes,                                    \
         SmallSmem<H / 8, FRPT, FNW, FNS, 2>::kBytes},                                   \
        {{(const void *)&rms_bwd_stream_small<T, H / 8, BRPT, BNW, BNS, false, false>,   \
          (const void *)&rms_bwd_stream_small<T, H / 8, BRPT, BNW, BNS, false, true>},   \
         {(const void *)&rms_bwd_stream_small<T, H / 8, BRPT, BNW, BNS, true, false>,    \
          (const void *)&rms_bwd_stream_small<T, H / 8, BRPT, BNW, BNS, true, true>}},   \
        {{SmallSmem<H / 8, BRPT, BNW, BNS, 2>::kBytes,                                   \
          SmallSmem<H / 8, BRPT, BNW, BNS, 2>::kBytes},                                  \
         {SmallSmem<H / 8, BRPT, BNW, BNS, 3>::kBytes,                                   \
          SmallSmem<H / 8, BRPT, BNW, BNS, 3>::kBytes}},                                 \
        {nullptr, nullptr},                                                              \
        {0, 0}};

#define RMSK_SPLIT(NAME, T, E)                                                    \
    const SplitKernels NAME = {                                                   \
        E,                                                                        \
        (const void *)&rms_fwd_split<T, E, 1, false>,                             \
        (const void *)&rms_fwd_split<T, E, 1, true>,                              \
        (const void *)&rms_fwd_split<T, E, 8, false>,                             \
        (const void *)&rms_fwd_split<T, E, 8, true>};
