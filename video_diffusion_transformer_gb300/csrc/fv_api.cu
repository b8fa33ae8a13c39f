// C ABI of the library (declared in include/fv.h): argument checks on the
// host, device checks, the per-device status word, and head-group launches.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fv.h"
#include "fv_internal.h"

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool probed = false;
    bool supported = false;
    int num_sms = 0;
    int *status = nullptr;  // device int, zeroed at allocation
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// fv_test_skip_load's armed load index per fv_test_kernel (-1: disarmed).
constexpr int kTestKernels = 5;
std::atomic<int64_t> g_test_skip[kTestKernels] = {{-1}, {-1}, {-1}, {-1}, {-1}};

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Current device's state; probes compute capability and SM count, and
// allocates the status word, on first use.
fv_status device_state(DeviceState **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FV_ERR_LAUNCH;
    std::lock_guard<std::mutex> g(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.probed) {
        if (!fv::probe_device(dev, &d.supported, &d.num_sms)) return FV_ERR_LAUNCH;
        d.probed = true;
    }
    if (!d.supported) return FV_ERR_UNSUPPORTED_DEVICE;
    if (d.status == nullptr) {
        void *p = nullptr;
        if (cudaMalloc(&p, 256) != cudaSuccess) return FV_ERR_LAUNCH;
        if (cudaMemset(p, 0, 256) != cudaSuccess) {
            cudaFree(p);
            return FV_ERR_LAUNCH;
        }
        d.status = static_cast<int *>(p);
    }
    *out = &d;
    return FV_OK;
}

// Shared by the dense and the windowed entry points: host checks, then one
// launch per head group.
fv_status attn_common(const void *Q, const void *K, const void *V, void *O, int64_t N, int H, int D, float scale,
                      int head_group, int frame_tokens, int chunk_frames, int window_chunks, float *lse,
                      void *stream) {
    fv_status st = fv::check_attn_args(Q, K, V, O, N, H, D, scale, head_group, lse);
    if (st != FV_OK) return st;
    DeviceState *d = nullptr;
    st = device_state(&d);
    if (st != FV_OK) return st;
    fv::AttnLaunch a;
    a.q = Q;
    a.k = K;
    a.v = V;
    a.o = O;
    a.lse = lse;
    a.n = N;
    a.heads_total = H;
    a.scale = scale;
    a.status = d->status;
    a.num_sms = d->num_sms;
    a.frame_tokens = frame_tokens;
    a.chunk_frames = chunk_frames;
    a.window_chunks = window_chunks;
    for (int h0 = 0; h0 < H; h0 += head_group) {
        a.head_begin = h0;
        a.heads = (H - h0) < head_group ? (H - h0) : head_group;
        st = fv::launch_attn_fwd(a, static_cast<cudaStream_t>(stream));
        if (st != FV_OK) return st;
    }
    return FV_OK;
}

}  // namespace

namespace fv {
bool probe_device(int dev, bool *supported, int *num_sms) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    *supported = (major == 10 && minor == 3);
    *num_sms = sms;
    return true;
}

fv_status check_attn_args(const void *Q, const void *K, const void *V, const void *O, int64_t N, int H, int D,
                          float scale, int head_group, const float *lse) {
    if (!Q || !K || !V || !O) return FV_ERR_NULL;
    if (D != 128 || N < 1 || N >= (int64_t(1) << 31) || H < 1 || H > 256 || head_group < 1 || head_group > H)
        return FV_ERR_SHAPE;
    if (!std::isfinite(scale) || scale < 0.0f) return FV_ERR_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || (lse && !aligned(lse, 4)))
        return FV_ERR_ALIGN;
    const size_t bytes = (size_t)N * (size_t)H * 128u * 2u;
    if (overlaps(O, bytes, Q, bytes) || overlaps(O, bytes, K, bytes) || overlaps(O, bytes, V, bytes))
        return FV_ERR_ALIAS;
    if (lse) {
        const size_t lb = (size_t)N * (size_t)H * 4u;
        if (overlaps(lse, lb, O, bytes) || overlaps(lse, lb, Q, bytes) || overlaps(lse, lb, K, bytes) ||
            overlaps(lse, lb, V, bytes))
            return FV_ERR_ALIAS;
    }
    return FV_OK;
}

fv_status status_of_word(int word) {
    if (word == 0) return FV_OK;
    if ((word & 0xFF00) == kDevBadTag) return FV_ERR_ARG;
    if ((word & 0xFF00) == kDevCheck) return FV_ERR_DEVICE_CHECK;
    return FV_ERR_DEVICE_TIMEOUT;
}

int64_t take_test_skip_load(int kernel) {
    if (kernel < 0 || kernel >= kTestKernels) return -1;
    // a plain load first: launches with the hook disarmed never write the atomic
    if (g_test_skip[kernel].load(std::memory_order_relaxed) < 0) return -1;
    return g_test_skip[kernel].exchange(-1);
}
}  // namespace fv

extern "C" {

fv_status fv_attn_fwd(const void *Q, const void *K, const void *V, void *O, int64_t N, int H, int D, float scale,
                      int head_group, float *lse, void *stream) {
    fv::NvtxRange nvtx("fv_attn_fwd");
    return attn_common(Q, K, V, O, N, H, D, scale, head_group, 0, 0, 0, lse, stream);
}

fv_status fv_attn_fwd_window(const void *Q, const void *K, const void *V, void *O, int64_t N, int H, int D,
                             float scale, int head_group, int frame_tokens, int chunk_frames, int window_chunks,
                             float *lse, void *stream) {
    fv::NvtxRange nvtx("fv_attn_fwd_window");
    if (frame_tokens < 1 || chunk_frames < 1 || window_chunks < 0 || N < 1 || (N % frame_tokens) != 0) {
        if (!Q || !K || !V || !O) return FV_ERR_NULL;
        return FV_ERR_SHAPE;
    }
    return attn_common(Q, K, V, O, N, H, D, scale, head_group, frame_tokens, chunk_frames, window_chunks, lse,
                       stream);
}

fv_status fv_delta_attn(const void *Q, const void *K, const void *V, const float *beta, const float *alpha,
                        const float *text_state, int64_t N, int H, int D, int frame_tokens, int chunk_frames,
                        int window_chunks, void *O, float *states, float *workspace, void *stream) {
    fv::NvtxRange nvtx("fv_delta_attn");
    if (!Q || !K || !V || !beta || !alpha || !O || !states || !workspace) return FV_ERR_NULL;
    if (D != 128 || N < 1 || N >= (int64_t(1) << 31) || H < 1 || H > 256 || frame_tokens < 1 ||
        (N % frame_tokens) != 0 || chunk_frames < 1 || window_chunks < 0)
        return FV_ERR_SHAPE;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(beta, 16) ||
        !aligned(alpha, 16) || !aligned(states, 16) || !aligned(workspace, 16) ||
        (text_state && !aligned(text_state, 16)))
        return FV_ERR_ALIGN;
    const size_t act = (size_t)N * (size_t)H * 128u * 2u;
    if (overlaps(O, act, Q, act) || overlaps(O, act, K, act) || overlaps(O, act, V, act)) return FV_ERR_ALIAS;
    const size_t st_bytes = (size_t)2 * H * (size_t)(N / frame_tokens) * 128u * 128u * 4u;
    if (overlaps(states, st_bytes, workspace, st_bytes)) return FV_ERR_ALIAS;
    DeviceState *d = nullptr;
    fv_status st = device_state(&d);
    if (st != FV_OK) return st;
    fv::DeltaLaunch a;
    a.q = Q;
    a.k = K;
    a.v = V;
    a.beta = beta;
    a.alpha = alpha;
    a.text_state = text_state;
    a.n = N;
    a.heads = H;
    a.frame_tokens = frame_tokens;
    a.chunk_frames = chunk_frames;
    a.window_chunks = window_chunks;
    a.o = O;
    a.states = states;
    a.workspace = workspace;
    a.status = d->status;
    a.num_sms = d->num_sms;
    return fv::launch_delta_attn(a, static_cast<cudaStream_t>(stream));
}

int fv_vsa_num_tiles(int frames, int height, int width) { return fv::vsa_num_tiles(frames, height, width); }

int fv_vsa_topk(int num_tiles, double sparsity) {
    if (num_tiles < 1 || std::isnan(sparsity)) return 0;
    const double want = std::ceil((1.0 - sparsity) * (double)num_tiles);
    if (!(want < (double)num_tiles)) return num_tiles;  // also +inf
    return want < 1.0 ? 1 : (int)want;
}

int64_t fv_vsa_workspace_bytes(int H, int frames, int height, int width, int topk) {
    const int nt = fv::vsa_num_tiles(frames, height, width);
    if (H < 1 || H > 256 || nt < 1 || topk < 1 || topk > nt) return -1;
    return fv::vsa_workspace_bytes(H, frames, height, width, topk);
}

fv_status fv_vsa_attn(const void *Q, const void *K, const void *V, void *O, int64_t N, int H, int D, float scale,
                      int frames, int height, int width, int topk, int32_t *selected, void *workspace,
                      int64_t workspace_bytes, float *lse, void *stream) {
    fv::NvtxRange nvtx("fv_vsa_attn");
    if (!Q || !K || !V || !O || !selected || !workspace) return FV_ERR_NULL;
    if (D != 128 || H < 1 || H > 256 || frames < 4 || height < 4 || width < 4 || N < 1 ||
        N >= (int64_t(1) << 31) || N != (int64_t)frames * height * width)
        return FV_ERR_SHAPE;
    const int nt = fv::vsa_num_tiles(frames, height, width);
    if (nt < 1 || topk < 1 || topk > nt) return FV_ERR_SHAPE;
    if (!std::isfinite(scale) || !(scale > 0.0f)) return FV_ERR_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(selected, 4) ||
        !aligned(workspace, 256) || (lse && !aligned(lse, 4)))
        return FV_ERR_ALIGN;
    const int64_t need = fv::vsa_workspace_bytes(H, frames, height, width, topk);
    if (workspace_bytes < need) return FV_ERR_ARG;
    const size_t act = (size_t)N * (size_t)H * 128u * 2u;
    const size_t selb = (size_t)H * (size_t)nt * (size_t)topk * 4u;
    const size_t lseb = (size_t)H * (size_t)N * 4u;
    const void *ins[3] = {Q, K, V};
    for (const void *in : ins) {
        if (overlaps(O, act, in, act) || overlaps(selected, selb, in, act) || overlaps(workspace, need, in, act) ||
            (lse && overlaps(lse, lseb, in, act)))
            return FV_ERR_ALIAS;
    }
    if (overlaps(O, act, selected, selb) || overlaps(O, act, workspace, need) ||
        overlaps(selected, selb, workspace, need) ||
        (lse && (overlaps(lse, lseb, O, act) || overlaps(lse, lseb, selected, selb) ||
                 overlaps(lse, lseb, workspace, need))))
        return FV_ERR_ALIAS;
    DeviceState *d = nullptr;
    fv_status st = device_state(&d);
    if (st != FV_OK) return st;
    fv::VsaLaunch a;
    a.q = Q;
    a.k = K;
    a.v = V;
    a.o = O;
    a.lse = lse;
    a.selected = selected;
    a.n = N;
    a.heads = H;
    a.frames = frames;
    a.height = height;
    a.width = width;
    a.topk = topk;
    a.scale = scale;
    a.workspace = workspace;
    a.status = d->status;
    a.num_sms = d->num_sms;
    return fv::launch_vsa_attn(a, static_cast<cudaStream_t>(stream));
}

fv_status fv_adaln_modulate(const void *x, void *y, int y_is_fp32, int64_t N, int C, const float *shift_table,
                            const float *scale_table, int64_t table_ld, int num_steps, int step, float eps,
                            void *stream) {
    fv::NvtxRange nvtx("fv_adaln_modulate");
    if (!x || !y || !shift_table || !scale_table) return FV_ERR_NULL;
    if (N < 1 || C < 8 || C > 8192 || (C % 8) != 0 || table_ld < C || num_steps < 1) return FV_ERR_SHAPE;
    if (step < 0 || step >= num_steps) return FV_ERR_STEP;
    if (!std::isfinite(eps) || eps < 0.0f) return FV_ERR_ARG;
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(shift_table, 16) || !aligned(scale_table, 16) ||
        (table_ld % 4) != 0)
        return FV_ERR_ALIGN;
    const size_t xb = (size_t)N * (size_t)C * 2u, yb = (size_t)N * (size_t)C * (y_is_fp32 ? 4u : 2u);
    if (overlaps(x, xb, y, yb)) return FV_ERR_ALIAS;
    DeviceState *d = nullptr;
    fv_status st = device_state(&d);
    if (st != FV_OK) return st;
    return fv::launch_adaln_modulate(x, y, y_is_fp32 != 0, N, C, shift_table + (int64_t)step * table_ld,
                                     scale_table + (int64_t)step * table_ld, eps, d->num_sms,
                                     static_cast<cudaStream_t>(stream));
}

fv_status fv_gated_residual(const void *x, const void *a, void *out, int64_t N, int C, const float *gate_table,
                            int64_t table_ld, int num_steps, int step, void *stream) {
    fv::NvtxRange nvtx("fv_gated_residual");
    if (!x || !a || !out || !gate_table) return FV_ERR_NULL;
    if (N < 1 || C < 8 || C > (1 << 20) || (C % 8) != 0 || table_ld < C || num_steps < 1) return FV_ERR_SHAPE;
    if (step < 0 || step >= num_steps) return FV_ERR_STEP;
    if (!aligned(x, 16) || !aligned(a, 16) || !aligned(out, 16) || !aligned(gate_table, 16) || (table_ld % 4) != 0)
        return FV_ERR_ALIGN;
    const size_t b = (size_t)N * (size_t)C * 2u;
    if (overlaps(out, b, a, b)) return FV_ERR_ALIAS;
    if (out != x && overlaps(out, b, x, b)) return FV_ERR_ALIAS;
    DeviceState *d = nullptr;
    fv_status st = device_state(&d);
    if (st != FV_OK) return st;
    return fv::launch_gated_residual(x, a, out, N, C, gate_table + (int64_t)step * table_ld, d->num_sms,
                                     static_cast<cudaStream_t>(stream));
}

fv_status fv_adaln_modulate_tagged(const void *x, void *y, int y_is_fp32, int64_t N, int C, const float *shift_table,
                                   const float *scale_table, int64_t table_ld, int num_steps, int num_modalities,
                                   int step, const uint8_t *token_tags, float eps, void *stream) {
    fv::NvtxRange nvtx("fv_adaln_modulate_tagged");
    if (!x || !y || !shift_table || !scale_table || !token_tags) return FV_ERR_NULL;
    if (N < 1 || C < 8 || C > 8192 || (C % 8) != 0 || table_ld < C || num_steps < 1 || num_modalities < 1 ||
        num_modalities > 255)
        return FV_ERR_SHAPE;
    if (step < 0 || step >= num_steps) return FV_ERR_STEP;
    if (!std::isfinite(eps) || eps < 0.0f) return FV_ERR_ARG;
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(shift_table, 16) || !aligned(scale_table, 16) ||
        (table_ld % 4) != 0)
        return FV_ERR_ALIGN;
    const size_t xb = (size_t)N * (size_t)C * 2u, yb = (size_t)N * (size_t)C * (y_is_fp32 ? 4u : 2u);
    if (overlaps(x, xb, y, yb)) return FV_ERR_ALIAS;
    DeviceState *d = nullptr;
    fv_status st = device_state(&d);
    if (st != FV_OK) return st;
    fv::TaggedRows t{shift_table, scale_table, table_ld, step * num_modalities, token_tags, num_modalities,
                     d->status};
    return fv::launch_adaln_modulate_tagged(t, x, y, y_is_fp32 != 0, N, C, eps, d->num_sms,
                                            static_cast<cudaStream_t>(stream));
}

fv_status fv_gated_residual_tagged(const void *x, const void *a, void *out, int64_t N, int C, const float *gate_table,
                                   int64_t table_ld, int num_steps, int num_modalities, int step,
                                   const uint8_t *token_tags, void *stream) {
    fv::NvtxRange nvtx("fv_gated_residual_tagged");
    if (!x || !a || !out || !gate_table || !token_tags) return FV_ERR_NULL;
    if (N < 1 || C < 8 || C > (1 << 20) || (C % 8) != 0 || table_ld < C || num_steps < 1 || num_modalities < 1 ||
        num_modalities > 255)
        return FV_ERR_SHAPE;
    if (step < 0 || step >= num_steps) return FV_ERR_STEP;
    if (!aligned(x, 16) || !aligned(a, 16) || !aligned(out, 16) || !aligned(gate_table, 16) || (table_ld % 4) != 0)
        return FV_ERR_ALIGN;
    const size_t b = (size_t)N * (size_t)C * 2u;
    if (overlaps(out, b, a, b)) return FV_ERR_ALIAS;
    if (out != x && overlaps(out, b, x, b)) return FV_ERR_ALIAS;
    DeviceState *d = nullptr;
    fv_status st = device_state(&d);
    if (st != FV_OK) return st;
    fv::TaggedRows t{gate_table, nullptr, table_ld, step * num_modalities, token_tags, num_modalities, d->status};
    return fv::launch_gated_residual_tagged(t, x, a, out, N, C, d->num_sms, static_cast<cudaStream_t>(stream));
}

fv_status fv_step_for_timestep(const float *ladder, int num_steps, float t, int *step_out) {
    if (!ladder || !step_out) return FV_ERR_NULL;
    if (num_steps < 1) return FV_ERR_SHAPE;
    for (int i = 0; i < num_steps; ++i) {
        if (ladder[i] == t) {
            *step_out = i;
            return FV_OK;
        }
    }
    return FV_ERR_STEP;
}

fv_status fv_sync_status(void *stream) {
    fv::NvtxRange nvtx("fv_sync_status");
    DeviceState *d = nullptr;
    fv_status st = device_state(&d);
    if (st != FV_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return FV_ERR_LAUNCH;
    int word = 0;
    if (cudaMemcpyAsync(&word, d->status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return FV_ERR_LAUNCH;
    if (word != 0) {
        if (cudaMemsetAsync(d->status, 0, sizeof(int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
            return FV_ERR_LAUNCH;
        return fv::status_of_word(word);
    }
    return FV_OK;
}

const char *fv_status_string(fv_status s) {
    switch (s) {
        case FV_OK: return "FV_OK";
        case FV_ERR_NULL: return "FV_ERR_NULL: a required pointer is NULL";
        case FV_ERR_SHAPE: return "FV_ERR_SHAPE: a size is out of range";
        case FV_ERR_ALIGN: return "FV_ERR_ALIGN: a pointer or leading dimension is not 16-byte aligned";
        case FV_ERR_STEP: return "FV_ERR_STEP: step/timestep is not on the stored schedule";
        case FV_ERR_UNSUPPORTED_DEVICE: return "FV_ERR_UNSUPPORTED_DEVICE: needs a compute capability 10.3 GPU";
        case FV_ERR_LAUNCH: return "FV_ERR_LAUNCH: a CUDA call or kernel launch failed";
        case FV_ERR_DEVICE_TIMEOUT: return "FV_ERR_DEVICE_TIMEOUT: a bounded wait inside a kernel ran out";
        case FV_ERR_ARG: return "FV_ERR_ARG: a scalar argument is invalid";
        case FV_ERR_ALIAS: return "FV_ERR_ALIAS: buffers overlap where the call forbids it";
        case FV_ERR_DEVICE_CHECK: return "FV_ERR_DEVICE_CHECK: an in-kernel index check of the debug build failed";
    }
    return "unknown fv_status";
}

fv_status fv_test_skip_load(int kernel, int64_t load_index) {
    if (kernel < 0 || kernel >= kTestKernels) return FV_ERR_ARG;
    g_test_skip[kernel].store(load_index < 0 ? -1 : load_index);
    return FV_OK;
}

int fv_version(void) { return 200; }

}  // extern "C"
