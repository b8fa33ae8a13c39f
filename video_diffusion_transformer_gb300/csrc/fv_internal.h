// Internal declarations shared by the C-ABI layer and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdint>

#include "fv.h"

namespace fv {

// An NVTX range around one C-ABI call, named after the call, so a timeline
// profiler shows which launches each call enqueued.  Without a profiler
// attached the push and pop are calls to empty functions.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

// Device status word values (0 = no error).  A kernel that gives up on a
// bounded wait stores kDevTimeout | where, where names the wait.
constexpr int kDevTimeout = 0x7100;
// A per-token modality tag was >= the number of modalities; the row was skipped.
constexpr int kDevBadTag = 0x7200;
// Debug build only: an in-kernel index check failed (kDevCheck | where); the
// access it guarded was skipped.
constexpr int kDevCheck = 0x7300;

#ifndef FV_DEBUG_CHECKS
#define FV_DEBUG_CHECKS 0
#endif

// Debug build: true when `ok`; otherwise records kDevCheck | where in the
// status word (first error wins) and returns false, so the caller skips the
// access.  Release build: always true, compiled out.
__device__ __forceinline__ bool dev_check(bool ok, int *status, int where) {
#if FV_DEBUG_CHECKS
    if (!ok) atomicCAS(status, 0, kDevCheck | where);
    return ok;
#else
    (void)status;
    (void)where;
    return true;
#endif
}

// Compute capability check (10.3) and SM count of device `dev`; false if a
// runtime query fails.
bool probe_device(int dev, bool *supported, int *num_sms);

// The host-side argument checks every attention entry point makes (pointers,
// sizes, scale, 16-byte alignment, forbidden overlaps); FV_OK or the status
// the call returns without enqueueing anything.
fv_status check_attn_args(const void *Q, const void *K, const void *V, const void *O, int64_t N, int H, int D,
                          float scale, int head_group, const float *lse);

// The status a non-zero device status word stands for.
fv_status status_of_word(int word);

// The load index armed by fv_test_skip_load for `kernel` (an fv_test_kernel
// value), or -1; reading it disarms the hook.
int64_t take_test_skip_load(int kernel);

// cuTensorMapEncodeTiled, looked up once through the runtime (null if absent).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

struct AttnLaunch {
    const void *q, *k, *v;
    void *o;
    float *lse;
    int64_t n;
    int heads_total;   // H (row stride of Q/K/V/O is H * 128)
    int head_begin;    // first head of this launch
    int heads;         // heads in this launch
    float scale;
    int *status;       // device status word
    int num_sms;
    // windowed attention; frame_tokens == 0 selects dense attention
    int frame_tokens = 0, chunk_frames = 0, window_chunks = 0;
};

// Enqueue one head-group launch of the attention kernel.
fv_status launch_attn_fwd(const AttnLaunch &a, cudaStream_t stream);

fv_status launch_adaln_modulate(const void *x, void *y, bool y_fp32, int64_t n, int c, const float *shift_row,
                                const float *scale_row, float eps, int num_sms, cudaStream_t stream);

fv_status launch_gated_residual(const void *x, const void *a, void *out, int64_t n, int c, const float *gate_row,
                                int num_sms, cudaStream_t stream);

// Table rows chosen per token: token i reads row row_base + tags[i] of
// table0 (and table1), rows ld floats apart.
struct TaggedRows {
    const float *table0, *table1;
    int64_t ld;
    int row_base;
    const uint8_t *tags;
    int num_tags;
    int *status;
};

struct DeltaLaunch {
    const void *q, *k, *v;        // bf16 [n, heads * 128]
    const float *beta;            // [heads, n]
    const float *alpha;           // [heads, frames, 128]
    const float *text_state;      // [heads, 128, 128] or null
    int64_t n;
    int heads;
    int frame_tokens, chunk_frames, window_chunks;
    void *o;                      // bf16 [n, heads * 128]
    float *states;                // [2, heads, frames, 128, 128]
    float *workspace;             // [2, heads, frames, 128, 128]
    int *status;                  // device status word
    int num_sms;
};

// The per-frame sums I + A_t -> ws_m and B_t^T -> ws_c of frames 1 .. F-2 on
// the tensor cores (layout [heads, frames, 128, 128]).
fv_status launch_vda_stats_tc(const DeltaLaunch &a, float *ws_m, float *ws_c, cudaStream_t stream);
// The forward and reverse state scans S <- (S Diag(alpha_t) + B_t) M_t on the
// tensor cores (split-bf16 products); ws_m holds M_t = (I + A_t)^{-1} as hi/lo
// bf16 operand tiles (as the solve writes them), ws_c holds B_t^T.
fv_status launch_vda_scan_tc(const DeltaLaunch &a, const float *ws_m, const float *ws_c, cudaStream_t stream);
// o = (S_fwd[p] + S_rev[n]) q / |q| for every token, on the tensor cores;
// wsplit: scratch of heads * chunks * 2 * 128 * 128 bf16.
fv_status launch_vda_readout_tc(const DeltaLaunch &a, __nv_bfloat16 *wsplit, cudaStream_t stream);

// Enqueue the Video Delta Attention kernels (stats, solve, scan, readout).
fv_status launch_delta_attn(const DeltaLaunch &a, cudaStream_t stream);

struct VsaLaunch {
    const void *q, *k, *v;        // bf16 [n, heads * 128], tokens in (frame, row, column) raster order
    void *o;                      // bf16 [n, heads * 128]
    float *lse;                   // [heads, n] or null
    int32_t *selected;            // [heads, num_tiles, topk]
    int64_t n;
    int heads;
    int frames, height, width;    // latent grid, n = frames * height * width
    int topk;
    float scale;
    void *workspace;              // vsa_workspace_bytes(...) bytes
    int *status;
    int num_sms;
};

// Tiles of the (4, 4, 4) tiling of a latent grid.
int vsa_num_tiles(int frames, int height, int width);
// Bytes of scratch fv_vsa_attn needs (tile means, per-pair kept-tile lists).
int64_t vsa_workspace_bytes(int heads, int frames, int height, int width, int topk);
// Enqueue the VSA kernels (tile means, selection, block-sparse attention).
fv_status launch_vsa_attn(const VsaLaunch &a, cudaStream_t stream);

fv_status launch_adaln_modulate_tagged(const TaggedRows &t, const void *x, void *y, bool y_fp32, int64_t n, int c,
                                       float eps, int num_sms, cudaStream_t stream);

fv_status launch_gated_residual_tagged(const TaggedRows &t, const void *x, const void *a, void *out, int64_t n,
                                       int c, int num_sms, cudaStream_t stream);

}  // namespace fv
