// Video Delta Attention: the linear branch of Video DeltaNet ("FreeVideo: a
// 66 GB video transformer on an 8 GB card", section "Where Video DeltaNet
// comes in").  Per head, with q and k L2-normalised:
//   frame t:  A_t = sum_u beta_u k_u k_u^T,  B_t = sum_u beta_u v_u k_u^T
//   state:    S_t = (S_{t-1} Diag(alpha_t) + B_t) (I + A_t)^{-1}
//             (the closed form of the frame's joint least-squares write)
//   scans:    forward over frames 1 .. F-2 and reverse over F-2 .. 1, each
//             seeded with half the text state (frames 0 and F-1 are the
//             softmax branch's global anchors and are not written)
//   readout:  a token of chunk c reads o = (S_fwd[p] + S_rev[n]) q with
//             p = (c - W) C - 1 (clamped to 0) the last frame before its
//             softmax window and n = (c + W + 1) C (clamped to F-1) the first
//             frame after it.
//
// Four kernels, float32 on the CUDA cores:
//   stats   (frame, head): I + A_t -> ws_m, B_t -> ws_c
//   solve   (frame, head): Cholesky of I + A_t in shared memory,
//                          M_t = (I + A_t)^{-1} -> ws_m, C_t = B_t M_t -> ws_c
//   scan    (head, direction): S <- (S Diag(alpha_t)) M_t + C_t, frame by frame
//   readout (frame, head): o = (S_fwd[p] + S_rev[n]) q_hat, rounded to bf16
// The scan is the only sequential part: 2 H chains of F - 2 128x128x128 steps.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fv_internal.h"

namespace fv {
namespace {

constexpr int kDv = 128;          // key and value dimension of a head
constexpr int kDThreads = 256;    // 16 x 16 threads, each an 8 x 8 block of a 128 x 128 result
constexpr int kTokBlock = 32;     // tokens staged per step of the statistics kernel
constexpr size_t kMat = (size_t)kDv * kDv;

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

// ------------------------------------------------------------------ stats
// I + A and B of frame t of head h.  Shared memory: normalised keys, beta
// times normalised keys, and values of kTokBlock tokens.
__global__ void __launch_bounds__(kDThreads, 1)
    vda_stats_kernel(const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
                     const float *__restrict__ beta, int64_t n, int ld, int frame_tokens, float *__restrict__ ws_m,
                     float *__restrict__ ws_c) {
    const int t = (int)blockIdx.x + 1;  // frames 1 .. F-2
    const int h = (int)blockIdx.y;
    const int frames = (int)(n / frame_tokens);
    __shared__ __align__(16) float kh[kTokBlock][kDv];
    __shared__ __align__(16) float bk[kTokBlock][kDv];
    __shared__ __align__(16) float vs[kTokBlock][kDv];
    const int tid = (int)threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ty = tid >> 4, tx = tid & 15;
    float acc_a[8][8], acc_b[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc_a[i][j] = acc_b[i][j] = 0.f;
    const int64_t tok0 = (int64_t)t * frame_tokens;
    for (int u0 = 0; u0 < frame_tokens; u0 += kTokBlock) {
        // stage: warp w normalises tokens w, w + 8, w + 16, w + 24 of the block
        for (int r = warp; r < kTokBlock; r += kDThreads / 32) {
            const int u = u0 + r;
            float kk[4], vv[4];
            float ss = 0.f, b = 0.f;
            if (u < frame_tokens) {
                const int64_t row = (tok0 + u) * (int64_t)ld + (int64_t)h * kDv + lane * 4;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    kk[e] = bf2f(k[row + e]);
                    vv[e] = bf2f(v[row + e]);
                    ss = fmaf(kk[e], kk[e], ss);
                }
                b = beta[(int64_t)h * n + tok0 + u];
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) kk[e] = vv[e] = 0.f;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float inv = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                kh[r][lane * 4 + e] = kk[e] * inv;
                bk[r][lane * 4 + e] = kk[e] * inv * b;
                vs[r][lane * 4 + e] = vv[e];
            }
        }
        __syncthreads();
#pragma unroll 2
        for (int r = 0; r < kTokBlock; ++r) {
            float ki[8], vi[8], bj[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                ki[i] = kh[r][ty * 8 + i];
                vi[i] = vs[r][ty * 8 + i];
                bj[i] = bk[r][tx * 8 + i];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    acc_a[i][j] = fmaf(ki[i], bj[j], acc_a[i][j]);
                    acc_b[i][j] = fmaf(vi[i], bj[j], acc_b[i][j]);
                }
        }
        __syncthreads();
    }
    const size_t base = ((size_t)h * frames + t) * kMat;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int r = ty * 8 + i, c = tx * 8 + j;
            ws_m[base + (size_t)r * kDv + c] = acc_a[i][j] + (r == c ? 1.0f : 0.0f);
            ws_c[base + (size_t)r * kDv + c] = acc_b[i][j];
        }
}

// ------------------------------------------------------------------ solve
// M = (I + A)^{-1} and C = B M for frame t of head h.  I + A is symmetric
// positive definite (A is a sum of beta-weighted outer products, beta >= 0),
// so a Cholesky factor L (lower, in place in g) gives M by two triangular
// solves against the identity.
constexpr int kLd = kDv + 1;  // padded row length of the factor

__global__ void __launch_bounds__(kDThreads, 1)
    vda_solve_kernel(int64_t n, int frame_tokens, float *__restrict__ ws_m, float *__restrict__ ws_c) {
    extern __shared__ float sh[];
    float *g = sh;                    // [kDv][kLd]  I + A, then its Cholesky factor
    float *y = sh + kDv * kLd;        // [kDv][kDv]  right-hand sides, then M
    const int t = (int)blockIdx.x + 1;
    const int h = (int)blockIdx.y;
    const int frames = (int)(n / frame_tokens);
    const size_t base = ((size_t)h * frames + t) * kMat;
    const int tid = (int)threadIdx.x;
    for (int e = tid; e < kDv * kDv; e += kDThreads) {
        g[(e / kDv) * kLd + (e % kDv)] = ws_m[base + e];
        y[e] = (e / kDv == e % kDv) ? 1.0f : 0.0f;
    }
    __syncthreads();
    // Cholesky, right-looking: column j, then the trailing lower triangle
    for (int j = 0; j < kDv; ++j) {
        const float d = sqrtf(g[j * kLd + j]);
        __syncthreads();
        for (int i = j + 1 + tid; i < kDv; i += kDThreads) g[i * kLd + j] /= d;
        if (tid == 0) g[j * kLd + j] = d;
        __syncthreads();
        const int m = kDv - 1 - j;  // trailing size
        for (int e = tid; e < m * m; e += kDThreads) {
            const int i = j + 1 + e / m, c = j + 1 + e % m;
            if (c <= i) g[i * kLd + c] = fmaf(-g[i * kLd + j], g[c * kLd + j], g[i * kLd + c]);
        }
        __syncthreads();
    }
    // L Y = I (forward), then L^T M = Y (backward); threads own columns of Y
    if (tid < kDv) {
        const int c = tid;
        for (int i = 0; i < kDv; ++i) {
            float s = y[i * kDv + c];
            for (int q = 0; q < i; ++q) s = fmaf(-g[i * kLd + q], y[q * kDv + c], s);
            y[i * kDv + c] = s / g[i * kLd + i];
        }
        for (int i = kDv - 1; i >= 0; --i) {
            float s = y[i * kDv + c];
            for (int q = i + 1; q < kDv; ++q) s = fmaf(-g[q * kLd + i], y[q * kDv + c], s);
            y[i * kDv + c] = s / g[i * kLd + i];
        }
    }
    __syncthreads();
    // C = B M, each thread an 8 x 8 block; B rows straight from global memory
    const int ty = tid >> 4, tx = tid & 15;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    for (int q = 0; q < kDv; ++q) {
        float bi[8], mj[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            bi[i] = ws_c[base + (size_t)(ty * 8 + i) * kDv + q];
            mj[i] = y[q * kDv + tx * 8 + i];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(bi[i], mj[j], acc[i][j]);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) ws_c[base + (size_t)(ty * 8 + i) * kDv + tx * 8 + j] = acc[i][j];
    for (int e = tid; e < kDv * kDv; e += kDThreads) ws_m[base + e] = y[e];
}

// ------------------------------------------------------------------- scan
// One head, one direction: S <- (S Diag(alpha_t)) M_t + C_t over the written
// frames, every state stored.  Shared memory: S and the frame's M_t.
__global__ void __launch_bounds__(kDThreads, 1)
    vda_scan_kernel(const float *__restrict__ alpha, const float *__restrict__ text_state, int frames,
                    const float *__restrict__ ws_m, const float *__restrict__ ws_c, float *__restrict__ states) {
    extern __shared__ float sh[];
    float *s = sh;               // [kDv][kDv]
    float *m = sh + kDv * kDv;   // [kDv][kDv]
    const int h = (int)blockIdx.x;
    const int dir = (int)blockIdx.y;  // 0 forward, 1 reverse
    const int H = (int)gridDim.x;
    const int tid = (int)threadIdx.x, ty = tid >> 4, tx = tid & 15;
    float *out = states + ((size_t)dir * H + h) * (size_t)frames * kMat;
    for (int e = tid; e < kDv * kDv; e += kDThreads)
        s[e] = text_state != nullptr ? 0.5f * text_state[(size_t)h * kMat + e] : 0.0f;
    __syncthreads();
    const int first = dir == 0 ? 0 : frames - 1;
    for (int e = tid; e < kDv * kDv; e += kDThreads) out[(size_t)first * kMat + e] = s[e];
    for (int step = 1; step <= frames - 2; ++step) {
        const int t = dir == 0 ? step : frames - 1 - step;
        const size_t base = ((size_t)h * frames + t) * kMat;
        const float *al = alpha + ((size_t)h * frames + t) * kDv;
        for (int e = tid; e < kDv * kDv; e += kDThreads) m[e] = ws_m[base + e] * al[e / kDv];
        __syncthreads();
        float acc[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = ws_c[base + (size_t)(ty * 8 + i) * kDv + tx * 8 + j];
        for (int q = 0; q < kDv; ++q) {
            float si[8], mj[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                si[i] = s[(ty * 8 + i) * kDv + q];
                mj[i] = m[q * kDv + tx * 8 + i];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(si[i], mj[j], acc[i][j]);
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = (ty * 8 + i) * kDv + tx * 8 + j;
                s[e] = acc[i][j];
                out[(size_t)t * kMat + e] = acc[i][j];
            }
        __syncthreads();
    }
    // the far anchor frame writes nothing: it carries the last written state
    if (frames >= 2) {
        const int last = dir == 0 ? frames - 1 : 0;
        for (int e = tid; e < kDv * kDv; e += kDThreads) out[(size_t)last * kMat + e] = s[e];
    }
}

// ---------------------------------------------------------------- readout
// o = (S_fwd[p] + S_rev[n]) q_hat for every token of frame t, head h.  The sum
// is held transposed in shared memory, so lane l reads the four outputs
// 4l .. 4l+3 of column q as one float4.
__global__ void __launch_bounds__(kDThreads)
    vda_readout_kernel(const __nv_bfloat16 *__restrict__ q, int64_t n, int ld, int frame_tokens, int chunk_frames,
                       int window_chunks, const float *__restrict__ states, __nv_bfloat16 *__restrict__ o) {
    extern __shared__ float sh[];
    float *wt = sh;                    // [kDv][kDv]  (S_fwd[p] + S_rev[n])^T
    float *qs = sh + kDv * kDv;        // [warps][kDv] normalised query of each warp
    const int t = (int)blockIdx.x;
    const int h = (int)blockIdx.y;
    const int H = (int)gridDim.y;
    const int frames = (int)(n / frame_tokens);
    const int tid = (int)threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = t / chunk_frames;
    int p = (c - window_chunks) * chunk_frames - 1;
    p = p < 0 ? 0 : p;
    int nx = (c + window_chunks + 1) * chunk_frames;
    nx = nx > frames - 1 ? frames - 1 : nx;
    const float *sf = states + ((size_t)h * frames + p) * kMat;
    const float *sr = states + (((size_t)H + h) * frames + nx) * kMat;
    for (int e = tid; e < kDv * kDv; e += kDThreads) {
        const int r = e / kDv, col = e % kDv;
        wt[col * kDv + r] = sf[e] + sr[e];
    }
    __syncthreads();
    float *qw = qs + warp * kDv;
    const int64_t tok0 = (int64_t)t * frame_tokens;
    for (int u = warp; u < frame_tokens; u += kDThreads / 32) {
        const int64_t row = (tok0 + u) * (int64_t)ld + (int64_t)h * kDv;
        float qq[4], ss = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            qq[e] = bf2f(q[row + lane * 4 + e]);
            ss = fmaf(qq[e], qq[e], ss);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float inv = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
#pragma unroll
        for (int e = 0; e < 4; ++e) qw[lane * 4 + e] = qq[e] * inv;
        __syncwarp();
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
        for (int k2 = 0; k2 < kDv; ++k2) {
            const float qk = qw[k2];
            const float4 w4 = *reinterpret_cast<const float4 *>(wt + k2 * kDv + lane * 4);
            acc[0] = fmaf(w4.x, qk, acc[0]);
            acc[1] = fmaf(w4.y, qk, acc[1]);
            acc[2] = fmaf(w4.z, qk, acc[2]);
            acc[3] = fmaf(w4.w, qk, acc[3]);
        }
        __syncwarp();
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0], acc[1]);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[2], acc[3]);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t *>(&lo);
        pk.y = *reinterpret_cast<uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(o + row + lane * 4) = pk;
    }
}

}  // namespace

fv_status launch_delta_attn(const DeltaLaunch &a, cudaStream_t stream) {
    const int frames = (int)(a.n / a.frame_tokens);
    const int ld = a.heads * kDv;
    const size_t solve_smem = (size_t)(kDv * kLd + kDv * kDv) * sizeof(float);
    const size_t scan_smem = (size_t)2 * kDv * kDv * sizeof(float);
    const size_t read_smem = (size_t)(kDv * kDv + (kDThreads / 32) * kDv) * sizeof(float);
    if (cudaFuncSetAttribute(vda_solve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)solve_smem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(vda_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)scan_smem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(vda_readout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)read_smem) !=
            cudaSuccess)
        return FV_ERR_LAUNCH;
    const auto *q = static_cast<const __nv_bfloat16 *>(a.q);
    const auto *k = static_cast<const __nv_bfloat16 *>(a.k);
    const auto *v = static_cast<const __nv_bfloat16 *>(a.v);
    float *ws_m = a.workspace;
    float *ws_c = a.workspace + (size_t)a.heads * frames * kMat;
    if (frames > 2) {
        const dim3 g(frames - 2, a.heads);
        vda_stats_kernel<<<g, kDThreads, 0, stream>>>(k, v, a.beta, a.n, ld, a.frame_tokens, ws_m, ws_c);
        vda_solve_kernel<<<g, kDThreads, solve_smem, stream>>>(a.n, a.frame_tokens, ws_m, ws_c);
    }
    vda_scan_kernel<<<dim3(a.heads, 2), kDThreads, scan_smem, stream>>>(a.alpha, a.text_state, frames, ws_m, ws_c,
                                                                       a.states);
    vda_readout_kernel<<<dim3(frames, a.heads), kDThreads, read_smem, stream>>>(
        q, a.n, ld, a.frame_tokens, a.chunk_frames, a.window_chunks, a.states,
        static_cast<__nv_bfloat16 *>(a.o));
    return cudaGetLastError() == cudaSuccess ? FV_OK : FV_ERR_LAUNCH;
}

}  // namespace fv
