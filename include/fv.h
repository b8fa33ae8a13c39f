/*
 * fv.h -- C ABI of the GB300 (sm_103a) dense video-token attention library.
 *
 * The library computes the hot path of one attention sub-layer of a
 * MiniMax-H3-shaped video diffusion transformer block:
 *
 *   fv_adaln_modulate   y = LN(x) * (1 + scale[step]) + shift[step]
 *   fv_attn_fwd         O = softmax(Q K^T * scale) V, full (unmasked), per head
 *   fv_gated_residual   out = x + gate[step] * a
 *
 * and the attention variants the pages describe for the same tensors:
 *
 *   fv_attn_fwd_window  the windowed softmax branch of Video DeltaNet
 *   fv_delta_attn       the linear (delta-rule) branch of Video DeltaNet
 *   fv_vsa_attn         VSA-style block-sparse attention over 3D tiles
 *   fv_adaln_modulate_tagged, fv_gated_residual_tagged
 *                       the table row chosen per token (step and modality)
 *   fv_attn_fwd_noalloc fv_attn_fwd for callers that cannot allocate
 *   fv_test_skip_load   test hook: make one bounded wait run out
 *
 * Sources ("FreeVideo: a 66 GB video transformer on an 8 GB card"):
 *   - section "What MiniMax H3 is, briefly": 56 heads of 128, Q/K/V 7168 wide,
 *     hidden size 5,376, tokens = latent frames x (H/32) x (W/32);
 *   - section "Why it does not fit: the arithmetic": the dense score matrix is
 *     never materialised, flash-style kernels stream it; attention is the
 *     time problem;
 *   - section "Cut one: 26 GB of AdaLN weights become 0.22 GB of tables":
 *     shift, scale and gate per step read from a stored table, and a call
 *     whose timestep is not the stored one is an error;
 *   - section "The rest is placement", item 1: attention runs on a group of
 *     4, 8 or 16 of the 56 heads at a time; a slice is tokens x heads x 128 x 2
 *     bytes.
 * And "FastH3 Preview v1", section "Lever two: VSA-H3 ...": one joint
 * bidirectional attention over the packed sequence (no causal mask).
 *
 * Conventions shared by every call:
 *   - Ownership: the caller owns every buffer.  Device pointers are plain CUDA
 *     device addresses (for example from torch).  The library allocates nothing
 *     per call; it keeps one small device status word per device, allocated on
 *     the first call that launches work on that device.
 *   - Execution: every compute call only enqueues work on `stream` (a
 *     cudaStream_t passed as void*; NULL is the legacy default stream) and
 *     returns without synchronising.  Argument errors are detected on the host
 *     before anything is enqueued.  Errors detected on the device (a bounded
 *     wait that ran out) are recorded in the status word and returned by
 *     fv_sync_status().
 *   - Errors: the return value is a status code.  The library never aborts,
 *     never exits and never traps a kernel.
 *   - bfloat16 data is IEEE-like 1-8-7; every float32 -> bfloat16 conversion
 *     rounds to nearest, ties to even.
 */
#ifndef FV_H
#define FV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FV_OK = 0,
    FV_ERR_NULL = -1,                /* a required pointer is NULL */
    FV_ERR_SHAPE = -2,               /* a size is out of range (N < 1, D != 128, C % 8 != 0, ...) */
    FV_ERR_ALIGN = -3,               /* a pointer or leading dimension breaks the 16-byte rule */
    FV_ERR_STEP = -4,                /* step not in [0, num_steps), or timestep off the ladder */
    FV_ERR_UNSUPPORTED_DEVICE = -5,  /* current device is not compute capability 10.3 */
    FV_ERR_LAUNCH = -6,              /* a CUDA call or kernel launch failed */
    FV_ERR_DEVICE_TIMEOUT = -7,      /* a bounded wait inside a kernel ran out */
    FV_ERR_ARG = -8,                 /* a scalar argument is invalid (scale < 0, eps < 0, NaN, ...) */
    FV_ERR_ALIAS = -9,               /* buffers overlap where the call forbids it */
    FV_ERR_DEVICE_CHECK = -10        /* debug build only: an in-kernel index check failed */
} fv_status;

/*
 * Dense bidirectional attention forward over the packed video tokens.
 *
 * For every head h in [0, H) and query row i in [0, N):
 *   s_ij = scale * q_i . k_j            (j = 0 .. N-1, no mask)
 *   o_i  = sum_j exp(s_ij - m_i) v_j / sum_j exp(s_ij - m_i),  m_i = max_j s_ij
 *   lse_i = m_i + ln sum_j exp(s_ij - m_i)
 * computed tile by tile with an online softmax; the N x N scores never exist.
 *
 * Q, K, V, O: device, bfloat16, [N, H*D] row-major (token-major, row stride
 *             H*D elements); head h occupies columns [h*D, h*D + D).  O must not
 *             overlap Q, K or V.  Each base address 16-byte aligned.
 * N:          tokens, >= 1 and < 2^31.
 * H:          heads, 1 .. 256.
 * D:          head dimension; must be 128.
 * scale:      softmax scale, finite and >= 0 (1/sqrt(128) for the model).
 * head_group: heads per launch, 1 .. H.  Heads run in groups of head_group
 *             (the last group holds H mod head_group heads when that is
 *             non-zero), one kernel launch per group, in order, on `stream`.
 * lse:        optional device float32 [H, N] (row h holds head h), natural-log
 *             log-sum-exp of each score row; NULL to skip.  4-byte aligned.
 * stream:     cudaStream_t as void*.
 * Compute: bf16 x bf16 products accumulated in float32 on the tensor cores;
 * softmax in float32; probabilities rounded to bf16 for the P.V product;
 * O normalised in float32 and rounded to bf16.
 */
fv_status fv_attn_fwd(const void *Q, const void *K, const void *V, void *O,
                      int64_t N, int H, int D, float scale, int head_group,
                      float *lse, void *stream);

/*
 * Windowed softmax attention: the softmax branch of Video DeltaNet
 * ("FreeVideo: a 66 GB video transformer on an 8 GB card", section "Where
 * Video DeltaNet comes in"): softmax attention stays exact but only within a
 * window; each query chunk of five latent frames (one VAE chunk) sees itself
 * and its two neighbours, every frame sees the first and the last latent
 * frame, and those two frames see everything.
 *
 * Tokens form latent frames of frame_tokens tokens (N must be a multiple of
 * frame_tokens; frames = N / frame_tokens); frames form chunks of
 * chunk_frames frames counted from frame 0 (the last chunk may be short).
 * Query i in frame f (chunk c = f / chunk_frames) sees key j in frame g when
 *   f is the first or the last frame, or g is the first or the last frame,
 *   or |g / chunk_frames - c| <= window_chunks,
 * and O is softmax attention over exactly those keys (same arithmetic and
 * output conventions as fv_attn_fwd; lse is over the admitted keys).
 * The kernel visits only the K/V tiles some row of a 256-row block may see.
 *
 * frame_tokens >= 1 with N % frame_tokens == 0; chunk_frames >= 1;
 * window_chunks >= 0; otherwise FV_ERR_SHAPE.  The model's values are
 * frame_tokens = (H/32)(W/32) (1,008 at 1344x768), chunk_frames = 5,
 * window_chunks = 1.  All other arguments as fv_attn_fwd.
 *
 * Memory: query blocks differ in cost (the anchors' see every key), so each
 * launch deals them to the CTAs from a table the library builds on the host
 * on the first call with a given geometry (N, frame_tokens, chunk_frames,
 * window_chunks, heads per launch, device), copies to a small device buffer
 * (grid x longest list ints, a few KB; cudaMalloc and a synchronous
 * cudaMemcpy) and keeps for the library's lifetime.  Later calls with the
 * same geometry allocate nothing.
 */
fv_status fv_attn_fwd_window(const void *Q, const void *K, const void *V, void *O,
                             int64_t N, int H, int D, float scale, int head_group,
                             int frame_tokens, int chunk_frames, int window_chunks,
                             float *lse, void *stream);

/*
 * Video Delta Attention: the linear branch of Video DeltaNet ("FreeVideo",
 * section "Where Video DeltaNet comes in").  Per head, q and k are
 * L2-normalised; frame t (frame_tokens tokens) has
 *   A_t = sum_u beta_u k_u k_u^T,   B_t = sum_u beta_u v_u k_u^T,
 * and the state after writing it is the closed form of the frame's joint
 * least-squares write,
 *   S_t = (S_{t-1} Diag(alpha_t) + B_t) (I + A_t)^{-1}.
 * Two scans run, forward over frames 1 .. F-2 and reverse over F-2 .. 1, each
 * seeded with text_state / 2; frames 0 and F-1 (the softmax branch's global
 * anchors) are not written.  A token of chunk c = frame / chunk_frames reads
 *   o = (S_fwd[p] + S_rev[n]) q,  p = max((c - window_chunks) chunk_frames - 1, 0),
 *                                n = min((c + window_chunks + 1) chunk_frames, F - 1),
 * the states just before and just after its softmax window (fv_attn_fwd_window).
 *
 * Q, K, V:      device bf16 [N, H*128], as fv_attn_fwd; O: device bf16 [N, H*128]
 *               (the linear branch's output, before its gate and projection).
 * beta:         device float32 [H, N], write strengths, >= 0.
 * alpha:        device float32 [H, F, 128], per-frame per-channel decay (entries
 *               of frames 0 and F-1 are not read).
 * text_state:   device float32 [H, 128, 128], or NULL for a zero state.
 * states:       device float32 [2, H, F, 128, 128]: written with the forward
 *               states (index 0) and reverse states (index 1) of every frame;
 *               S_fwd[0] = S_rev[F-1] = text_state / 2.
 * workspace:    device float32 [2, H, F, 128, 128], caller-owned scratch.
 * N = F * frame_tokens; F >= 1; chunk_frames >= 1; window_chunks >= 0; D = 128;
 * H 1 .. 256; all pointers 16-byte aligned; else FV_ERR_SHAPE / _NULL / _ALIGN.
 * Compute: the per-frame sums A_t, B_t, the state scans and the readout run on
 * the tensor cores with float32 accumulation; their operands (beta-weighted
 * normalised keys, values, the inverse (I + A_t)^{-1}, the scanned
 * S Diag(alpha) + B, the summed states) are split into bf16 hi + lo parts, so
 * the products keep close to float32 accuracy (states within ~2e-5 relative
 * of float64 over 72 frames).  The per-frame inversion (a symmetric sweep,
 * i.e. Gauss-Jordan elimination kept symmetric, on I + A_t, symmetric
 * positive definite) runs in float32.  O is rounded once
 * to bf16.
 */
fv_status fv_delta_attn(const void *Q, const void *K, const void *V, const float *beta,
                        const float *alpha, const float *text_state, int64_t N, int H, int D,
                        int frame_tokens, int chunk_frames, int window_chunks, void *O,
                        float *states, float *workspace, void *stream);

/*
 * VSA-style block-sparse attention ("FastH3 Preview v1", section "Lever two:
 * VSA-H3 makes each of the four calls cheaper").  The N = frames * height *
 * width video tokens form a latent grid in (frame, row, column) raster order
 * and are cut into 3D tiles of (4, 4, 4) tokens, numbered in raster order over
 * the tile grid; tiles on the far edges hold fewer tokens where a side is not
 * a multiple of 4.  Per head:
 *   1. coarse stage: score(b, c) = mean_{i in b} q_i . mean_{j in c} k_j for
 *      every query tile b and key tile c (float32);
 *   2. each query tile b keeps the topk key tiles with the highest scores,
 *      ties to the lower tile index;
 *   3. fine stage: o_i = softmax_j(scale q_i.k_j) v_j over the tokens j of the
 *      tiles b kept, for every token i of b (float32 softmax, bf16 P.V).
 * The page's count of kept tiles is fv_vsa_topk(num_tiles, sparsity).  The
 * learned compression branch is not part of this call (its gate needs
 * trained weights and starts at zero).
 *
 * Q, K, V, O:   device bf16 [N, H*128], as fv_attn_fwd.
 * frames, height, width: the latent grid, each >= 4; N must equal their
 *               product; at most 16,384 tiles.
 * topk:         1 .. fv_vsa_num_tiles(frames, height, width).
 * selected:     device int32 [H, num_tiles, topk], written: the kept tiles of
 *               every query tile, ascending.
 * workspace:    device scratch of at least fv_vsa_workspace_bytes(...) bytes
 *               (256-byte aligned), caller-owned; workspace_bytes is its size.
 *               It holds the tile means, the kept-tile lists and a tile-major
 *               copy of K and V (2 x H x tiles x 16 KB: 2.2 GB at 72 x 24 x 42
 *               with 56 heads).
 * lse:          nullable device float32 [H, N], as fv_attn_fwd.
 * Errors: FV_ERR_NULL, FV_ERR_SHAPE (grid, N, topk, tile count, D, H),
 * FV_ERR_ALIGN (16-byte Q/K/V/O, 4-byte selected and lse, 256-byte
 * workspace), FV_ERR_ARG (scale not finite and > 0, workspace too small),
 * FV_ERR_ALIAS (O or selected or workspace overlapping another buffer).
 * All heads run in one launch sequence on `stream`.
 */
fv_status fv_vsa_attn(const void *Q, const void *K, const void *V, void *O, int64_t N, int H, int D,
                      float scale, int frames, int height, int width, int topk, int32_t *selected,
                      void *workspace, int64_t workspace_bytes, float *lse, void *stream);

/* Number of (4, 4, 4) tiles of the grid; 0 for a side < 1, -1 above 16,384. */
int fv_vsa_num_tiles(int frames, int height, int width);

/* The page's count of kept tiles, max(1, min(ceil((1 - sparsity) * num_tiles),
 * num_tiles)), evaluated in double; 0 when num_tiles < 1 or sparsity is NaN. */
int fv_vsa_topk(int num_tiles, double sparsity);

/* Scratch bytes fv_vsa_attn needs for H heads, the grid and topk; -1 on bad sizes. */
int64_t fv_vsa_workspace_bytes(int H, int frames, int height, int width, int topk);

/*
 * Cached-AdaLN modulated LayerNorm of the residual stream for one schedule step:
 *   mu = mean_c x[i,c],  var = mean_c (x[i,c] - mu)^2   (biased)
 *   y[i,c] = (x[i,c] - mu) / sqrt(var + eps) * (1 + scale_table[step*ld + c])
 *            + shift_table[step*ld + c]
 * The LayerNorm has no learned affine of its own; the table supplies it.
 *
 * x:            device bfloat16 [N, C] row-major, 16-byte aligned.
 * y:            device [N, C]; float32 if y_is_fp32 != 0, else bfloat16.
 *               16-byte aligned; must not overlap x.
 * N:            rows (tokens), >= 1.   C: channels, 8 .. 8192, C % 8 == 0.
 * shift_table, scale_table: device float32 [num_steps, table_ld]; row `step`
 *               is read (each may be a strided view into a packed table of
 *               several vectors).  16-byte aligned, table_ld >= C and
 *               table_ld % 4 == 0.
 * num_steps:    rows in the tables (>= 1).   step: 0 .. num_steps-1, else
 *               FV_ERR_STEP (a timestep that is not on the stored schedule).
 * eps:          >= 0 and finite.
 */
fv_status fv_adaln_modulate(const void *x, void *y, int y_is_fp32, int64_t N, int C,
                            const float *shift_table, const float *scale_table,
                            int64_t table_ld, int num_steps, int step, float eps,
                            void *stream);

/*
 * Gated residual for one schedule step:
 *   out[i,c] = x[i,c] + gate_table[step*ld + c] * a[i,c]
 * computed as one float32 fused multiply-add, rounded once to bfloat16.
 *
 * x, a, out:  device bfloat16 [N, C] row-major, 16-byte aligned.  out may be
 *             exactly x (in place); any other overlap is FV_ERR_ALIAS.
 * gate_table: device float32 [num_steps, table_ld], 16-byte aligned,
 *             table_ld >= C, table_ld % 4 == 0.
 * N >= 1; C % 8 == 0, 8 .. 2^20; step in [0, num_steps) else FV_ERR_STEP.
 */
fv_status fv_gated_residual(const void *x, const void *a, void *out, int64_t N, int C,
                            const float *gate_table, int64_t table_ld, int num_steps,
                            int step, void *stream);

/*
 * Per-token modality rows ("FastH3 Preview v1", section "Update: consumer
 * GPUs and Trim": the six modulation vectors exist per modality, indexed
 * timestep_indices * 3 + token_tags).  The same two ops, but token i reads
 * table row step * num_modalities + token_tags[i], so a packed
 * [text | audio | video] sequence takes each token's own modality row.
 *
 * token_tags:     device uint8 [N], each in [0, num_modalities).  A tag out of
 *                 range is not detected on the host: the kernel leaves that
 *                 row's output unwritten and fv_sync_status() reports
 *                 FV_ERR_ARG.
 * num_modalities: 1 .. 255; tables hold num_steps * num_modalities rows.
 * step:           0 .. num_steps-1, else FV_ERR_STEP.
 * All other arguments, layouts and checks as the untagged calls.
 */
fv_status fv_adaln_modulate_tagged(const void *x, void *y, int y_is_fp32, int64_t N, int C,
                                   const float *shift_table, const float *scale_table,
                                   int64_t table_ld, int num_steps, int num_modalities, int step,
                                   const uint8_t *token_tags, float eps, void *stream);

fv_status fv_gated_residual_tagged(const void *x, const void *a, void *out, int64_t N, int C,
                                   const float *gate_table, int64_t table_ld, int num_steps,
                                   int num_modalities, int step, const uint8_t *token_tags,
                                   void *stream);

/*
 * Schedule cursor: the step whose stored timestep equals t exactly.
 * ladder: host float32 [num_steps].  Writes the first matching index to
 * *step_out and returns FV_OK, or returns FV_ERR_STEP if t is not on the
 * ladder (the tables were computed for other timesteps).  Host only.
 */
fv_status fv_step_for_timestep(const float *ladder, int num_steps, float t, int *step_out);

/*
 * Synchronise `stream`, then read and clear the current device's status word.
 * Returns FV_OK, FV_ERR_DEVICE_TIMEOUT if a kernel gave up on a bounded wait
 * since the last call, FV_ERR_ARG if a kernel met an out-of-range token tag,
 * FV_ERR_DEVICE_CHECK if (debug build only) an in-kernel index check failed,
 * or FV_ERR_LAUNCH if the stream reports a CUDA error.
 *
 * Debug build: the library compiled with FV_DEBUG_CHECKS=1 (libfv_debug.so,
 * made next to libfv.so by the package's build step) checks, inside the
 * attention kernels, every tile coordinate against N and the head range
 * and every tensor-memory column against the allocation before it is used;
 * a failed check records FV_ERR_DEVICE_CHECK here and skips the access
 * instead of trapping.  The release build compiles the checks out.
 */
fv_status fv_sync_status(void *stream);

/*
 * fv_attn_fwd for callers that must not allocate device memory.  The pages
 * have no counterpart: this is a property of the library, not of the method.
 *
 * fv_attn_fwd allocates (once per device, with cudaMalloc) the small status
 * word its kernels report into.  A caller whose device memory is owned by
 * someone else -- a framework's caching allocator, or a serving process that
 * budgets every byte of a fixed pool -- cannot let a library call cudaMalloc
 * behind its back, and cudaMalloc can also synchronise the whole device.
 * This variant computes exactly what fv_attn_fwd computes, with the same
 * arguments and checks, but keeps its scratch (one status word per
 * head-group launch) in an array compiled into the library: it calls no
 * cudaMalloc, cudaFree or other allocating routine.  The caller still passes
 * all inputs and outputs.
 *
 * Limits and sharing:
 *   - at most FV_NOALLOC_MAX_LAUNCHES head-group launches per call, i.e.
 *     ceil(H / head_group) <= 64; a call needing more returns FV_ERR_SHAPE
 *     before doing anything;
 *   - the scratch array is one per device and shared by every call on that
 *     device; each call clears the words it uses (on `stream`) before its
 *     launches.  Calls whose work overlaps on the GPU (different streams, or
 *     different host threads without ordering) race on it: order them;
 *   - the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 * device_status_out: NULL to return right after enqueueing (device-side
 *   timeouts then go unreported); otherwise the call synchronises `stream`,
 *   then writes FV_OK or FV_ERR_DEVICE_TIMEOUT (FV_ERR_DEVICE_CHECK from a
 *   failed index check of the debug build) to *device_status_out.
 */
#define FV_NOALLOC_MAX_LAUNCHES 64
fv_status fv_attn_fwd_noalloc(const void *Q, const void *K, const void *V, void *O,
                              int64_t N, int H, int D, float scale, int head_group,
                              float *lse, void *stream, int *device_status_out);

/*
 * Test hook for the failure path; not for production use.  The pages have no
 * counterpart.
 *
 * Every kernel that waits on a copy bounds that wait (about 2 s); a wait that
 * runs out records FV_ERR_DEVICE_TIMEOUT in the status word, the kernel
 * drains what it has in flight, releases its tensor memory and returns, and
 * the context stays usable.  This call arms that path without any fault:
 * the NEXT launch of the named kernel has its first CTA never issue the copy
 * numbered load_index (counted from 0 in the order that CTA issues them:
 * K/V tiles for FV_TEST_ATTN and FV_TEST_VSA_FINE, 64-token K/V stages for
 * FV_TEST_VDA_STATS, inverse tiles M_t for FV_TEST_VDA_SCAN, Q tiles for
 * FV_TEST_VDA_READOUT), so the wait for it runs out.  The hook is one-shot:
 * that launch disarms it.  load_index < 0 disarms it without a launch.  A
 * load_index the CTA never reaches leaves the launch unaffected.
 * Returns FV_ERR_ARG for an unknown kernel.  Host only; thread-safe.
 */
typedef enum {
    FV_TEST_ATTN = 0,         /* fv_attn_fwd, fv_attn_fwd_window, fv_attn_fwd_noalloc */
    FV_TEST_VSA_FINE = 1,     /* the fine (block-sparse attention) kernel of fv_vsa_attn */
    FV_TEST_VDA_STATS = 2,    /* the per-frame sums kernel of fv_delta_attn */
    FV_TEST_VDA_SCAN = 3,     /* the state-scan kernel of fv_delta_attn */
    FV_TEST_VDA_READOUT = 4   /* the readout kernel of fv_delta_attn */
} fv_test_kernel;
fv_status fv_test_skip_load(int kernel, int64_t load_index);

/* Static, human-readable name of a status code (never NULL). */
const char *fv_status_string(fv_status s);

/* Library version: major * 10000 + minor * 100 + patch. */
int fv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FV_H */
