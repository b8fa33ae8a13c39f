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
// Four kernels:
//   stats   (frame, head; tensor cores, delta_tc.cu): I + A_t -> ws_m, B_t -> ws_c
//   solve   (frame, head; float32): Gauss-Jordan on [I + A_t | B_t^T] in registers,
//                          M'_t = Diag(alpha_t) (I + A_t)^{-1} -> ws_m,
//                          C_t = B_t (I + A_t)^{-1} -> ws_c
//   scan    (head, direction; float32): S <- S M'_t + C_t, frame by frame
//   readout (chunk rows, head; tensor cores, delta_tc.cu): o = (S_fwd[p] + S_rev[n]) q_hat,
//           rounded to bf16
// The scan is the only sequential part: 2 H chains of F - 2 128x128x128 steps.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fv_internal.h"

namespace fv {
namespace {

constexpr int kDv = 128;          // key and value dimension of a head
constexpr int kDThreads = 256;    // 16 x 16 threads, each an 8 x 8 block of a 128 x 128 result
constexpr size_t kMat = (size_t)kDv * kDv;


// ------------------------------------------------------------------ solve
// Gauss-Jordan elimination on the 128 x 256 matrix [I + A | B^T] of frame t
// of head h: after the 128 pivot steps the left half holds M = (I + A)^{-1}
// and the right half X = M B^T, whose transpose is C = B M (M is symmetric).
// No pivoting is needed: I + A is symmetric positive definite with every
// Schur complement >= I (A is a sum of beta-weighted outer products,
// beta >= 0), so every pivot is >= 1.  The matrix lives in registers: thread
// (ty, tx) holds rows ty*8 .. ty*8+7 and columns tx*8 .. tx*8+7 of both
// halves.  Each step broadcasts the pivot row and pivot column through shared
// memory (two alternating buffers, one barrier per step).
// Written out: M' = Diag(alpha_t) M (the decay folded into the scan's
// multiplier, S_{t-1} Diag(alpha_t) M = S_{t-1} M') and C.
__global__ void __launch_bounds__(kDThreads, 1)
    vda_solve_kernel(const float *__restrict__ alpha, int frames, float *__restrict__ ws_m,
                     float *__restrict__ ws_c) {
    __shared__ __align__(16) float rowbuf[2][2 * kDv];
    __shared__ __align__(16) float colbuf[2][kDv];
    const int t = (int)blockIdx.x + 1;
    const int h = (int)blockIdx.y;
    const size_t base = ((size_t)h * frames + t) * kMat;
    const int tid = (int)threadIdx.x, ty = tid >> 4, tx = tid & 15;
    float g[8][8], x[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 *src = reinterpret_cast<const float4 *>(ws_m + base + (size_t)(ty * 8 + i) * kDv + tx * 8);
        const float4 a0 = src[0], a1 = src[1];
        g[i][0] = a0.x, g[i][1] = a0.y, g[i][2] = a0.z, g[i][3] = a0.w;
        g[i][4] = a1.x, g[i][5] = a1.y, g[i][6] = a1.z, g[i][7] = a1.w;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // X = B^T: x[i][j] = B[tx*8 + j][ty*8 + i]
        const float4 *src = reinterpret_cast<const float4 *>(ws_c + base + (size_t)(tx * 8 + j) * kDv + ty * 8);
        const float4 b0 = src[0], b1 = src[1];
        x[0][j] = b0.x, x[1][j] = b0.y, x[2][j] = b0.z, x[3][j] = b0.w;
        x[4][j] = b1.x, x[5][j] = b1.y, x[6][j] = b1.z, x[7][j] = b1.w;
    }
    for (int kb = 0; kb < kDv / 8; ++kb) {
        const bool own_row = ty == kb, own_col = tx == kb;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int k = kb * 8 + kk;
            float *rb = rowbuf[kk & 1];
            float *cb = colbuf[kk & 1];
            if (own_row) {
                float4 *dg = reinterpret_cast<float4 *>(rb + tx * 8);
                float4 *dx = reinterpret_cast<float4 *>(rb + kDv + tx * 8);
                dg[0] = make_float4(g[kk][0], g[kk][1], g[kk][2], g[kk][3]);
                dg[1] = make_float4(g[kk][4], g[kk][5], g[kk][6], g[kk][7]);
                dx[0] = make_float4(x[kk][0], x[kk][1], x[kk][2], x[kk][3]);
                dx[1] = make_float4(x[kk][4], x[kk][5], x[kk][6], x[kk][7]);
            }
            if (own_col) {
                float4 *dc = reinterpret_cast<float4 *>(cb + ty * 8);
                dc[0] = make_float4(g[0][kk], g[1][kk], g[2][kk], g[3][kk]);
                dc[1] = make_float4(g[4][kk], g[5][kk], g[6][kk], g[7][kk]);
            }
            __syncthreads();
            const float p = 1.0f / rb[k];
            float rg[8], rx[8], f[8];
            {
                const float4 *sg = reinterpret_cast<const float4 *>(rb + tx * 8);
                const float4 *sx = reinterpret_cast<const float4 *>(rb + kDv + tx * 8);
                const float4 *sc = reinterpret_cast<const float4 *>(cb + ty * 8);
                const float4 g0 = sg[0], g1 = sg[1], x0 = sx[0], x1 = sx[1], c0 = sc[0], c1 = sc[1];
                rg[0] = g0.x, rg[1] = g0.y, rg[2] = g0.z, rg[3] = g0.w;
                rg[4] = g1.x, rg[5] = g1.y, rg[6] = g1.z, rg[7] = g1.w;
                rx[0] = x0.x, rx[1] = x0.y, rx[2] = x0.z, rx[3] = x0.w;
                rx[4] = x1.x, rx[5] = x1.y, rx[6] = x1.z, rx[7] = x1.w;
                f[0] = c0.x, f[1] = c0.y, f[2] = c0.z, f[3] = c0.w;
                f[4] = c1.x, f[5] = c1.y, f[6] = c1.z, f[7] = c1.w;
            }
            // One update for every element: row i loses f_i times the pivot row
            // divided by the pivot, with f_k - 1 for the pivot row itself (so it
            // becomes the divided row), and the pivot column first set to the
            // identity's column (so it becomes column k of the inverse:
            // -f_i / pivot, and 1 / pivot on the diagonal).
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                rg[j] *= p;
                rx[j] *= p;
            }
            if (own_col) {
                rg[kk] = p;
#pragma unroll
                for (int i = 0; i < 8; ++i) g[i][kk] = (own_row && i == kk) ? 1.0f : 0.0f;
            }
            if (own_row) f[kk] -= 1.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    g[i][j] = fmaf(-f[i], rg[j], g[i][j]);
                    x[i][j] = fmaf(-f[i], rx[j], x[i][j]);
                }
            }
        }
    }
    const float *al = alpha + ((size_t)h * frames + t) * kDv;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float a = al[ty * 8 + i];
        float4 *dst = reinterpret_cast<float4 *>(ws_m + base + (size_t)(ty * 8 + i) * kDv + tx * 8);
        dst[0] = make_float4(a * g[i][0], a * g[i][1], a * g[i][2], a * g[i][3]);
        dst[1] = make_float4(a * g[i][4], a * g[i][5], a * g[i][6], a * g[i][7]);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // C[tx*8 + j][ty*8 + i] = X[ty*8 + i][tx*8 + j]
        float4 *dst = reinterpret_cast<float4 *>(ws_c + base + (size_t)(tx * 8 + j) * kDv + ty * 8);
        dst[0] = make_float4(x[0][j], x[1][j], x[2][j], x[3][j]);
        dst[1] = make_float4(x[4][j], x[5][j], x[6][j], x[7][j]);
    }
}

// ------------------------------------------------------------------- scan
// One head, one direction: S <- S M'_t + C_t over the written frames, every
// state stored.  The next frame's M' is copied into the other half of a
// double buffer (cp.async) while the current step computes.  S is kept
// transposed in shared memory with rows padded to kSLd floats, so both the
// reads of a column of S and the transposed writes stay free of bank
// conflicts.  Thread (ty, tx) computes rows {ty*4 + i, 64 + ty*4 + i} and
// columns {tx*4 + j, 64 + tx*4 + j} of the product.
constexpr int kSLd = kDv + 4;

__device__ __forceinline__ void cp_async_16(float *dst, const float *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void scan_prefetch(float *dst, const float *src, int tid) {
#pragma unroll
    for (int e = 0; e < (int)(kMat / 4 / kDThreads); ++e) {
        const int idx = (e * kDThreads + tid) * 4;
        cp_async_16(dst + idx, src + idx);
    }
    cp_async_commit();
}

__global__ void __launch_bounds__(kDThreads, 1)
    vda_scan_kernel(const float *__restrict__ text_state, int frames, const float *__restrict__ ws_m,
                    const float *__restrict__ ws_c, float *__restrict__ states) {
    extern __shared__ __align__(16) float sh[];
    float *st = sh;                    // [kDv][kSLd]  S transposed
    float *mb = sh + kDv * kSLd;       // [2][kDv][kDv] M' of this step and the next
    const int h = (int)blockIdx.x;
    const int dir = (int)blockIdx.y;  // 0 forward, 1 reverse
    const int H = (int)gridDim.x;
    const int tid = (int)threadIdx.x, ty = tid >> 4, tx = tid & 15;
    float *out = states + ((size_t)dir * H + h) * (size_t)frames * kMat;
    const int steps = frames - 2;
    auto frame_of = [&](int step) { return dir == 0 ? step : frames - 1 - step; };
    if (steps >= 1) scan_prefetch(mb, ws_m + ((size_t)h * frames + frame_of(1)) * kMat, tid);
    const int first = dir == 0 ? 0 : frames - 1;
    for (int e = tid; e < (int)kMat; e += kDThreads) {
        const float v = text_state != nullptr ? 0.5f * text_state[(size_t)h * kMat + e] : 0.0f;
        st[(e % kDv) * kSLd + e / kDv] = v;
        out[(size_t)first * kMat + e] = v;
    }
    int rows[8], cols[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        rows[i] = (i < 4 ? 0 : 64) + ty * 4 + (i & 3);
        cols[i] = (i < 4 ? 0 : 64) + tx * 4 + (i & 3);
    }
    for (int step = 1; step <= steps; ++step) {
        const int t = frame_of(step);
        const size_t base = ((size_t)h * frames + t) * kMat;
        const float *m = mb + (size_t)((step - 1) & 1) * kMat;
        cp_async_wait_all();
        __syncthreads();  // M'_t landed for every thread; the previous S is in st
        if (step < steps)
            scan_prefetch(mb + (size_t)(step & 1) * kMat, ws_m + ((size_t)h * frames + frame_of(step + 1)) * kMat,
                          tid);
        float cv[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 *src = reinterpret_cast<const float4 *>(ws_c + base + (size_t)rows[i] * kDv);
            const float4 c0 = src[tx], c1 = src[16 + tx];
            cv[i][0] = c0.x, cv[i][1] = c0.y, cv[i][2] = c0.z, cv[i][3] = c0.w;
            cv[i][4] = c1.x, cv[i][5] = c1.y, cv[i][6] = c1.z, cv[i][7] = c1.w;
        }
        float acc[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
#pragma unroll 4
        for (int q = 0; q < kDv; ++q) {
            const float4 s0 = *reinterpret_cast<const float4 *>(st + q * kSLd + ty * 4);
            const float4 s1 = *reinterpret_cast<const float4 *>(st + q * kSLd + 64 + ty * 4);
            const float4 m0 = *reinterpret_cast<const float4 *>(m + q * kDv + tx * 4);
            const float4 m1 = *reinterpret_cast<const float4 *>(m + q * kDv + 64 + tx * 4);
            const float si[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
            const float mj[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(si[i], mj[j], acc[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] += cv[i][j];
        __syncthreads();  // every read of the previous S is done
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float4 *dst = reinterpret_cast<float4 *>(out + (size_t)t * kMat + (size_t)rows[i] * kDv);
            dst[tx] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            dst[16 + tx] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            *reinterpret_cast<float4 *>(st + cols[j] * kSLd + ty * 4) =
                make_float4(acc[0][j], acc[1][j], acc[2][j], acc[3][j]);
            *reinterpret_cast<float4 *>(st + cols[j] * kSLd + 64 + ty * 4) =
                make_float4(acc[4][j], acc[5][j], acc[6][j], acc[7][j]);
        }
    }
    __syncthreads();
    // the far anchor frame writes nothing: it carries the last written state
    if (frames >= 2) {
        const int last = dir == 0 ? frames - 1 : 0;
        for (int e = tid; e < (int)kMat; e += kDThreads) out[(size_t)last * kMat + e] = st[(e % kDv) * kSLd + e / kDv];
    }
}

}  // namespace

fv_status launch_delta_attn(const DeltaLaunch &a, cudaStream_t stream) {
    const int frames = (int)(a.n / a.frame_tokens);
    const size_t scan_smem = (size_t)(kDv * kSLd + 2 * kDv * kDv) * sizeof(float);
    if (cudaFuncSetAttribute(vda_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)scan_smem) !=
        cudaSuccess)
        return FV_ERR_LAUNCH;
    float *ws_m = a.workspace;
    float *ws_c = a.workspace + (size_t)a.heads * frames * kMat;
    if (frames > 2) {
        const fv_status st = launch_vda_stats_tc(a, ws_m, ws_c, stream);
        if (st != FV_OK) return st;
        vda_solve_kernel<<<dim3(frames - 2, a.heads), kDThreads, 0, stream>>>(a.alpha, frames, ws_m, ws_c);
    }
    vda_scan_kernel<<<dim3(a.heads, 2), kDThreads, scan_smem, stream>>>(a.text_state, frames, ws_m, ws_c, a.states);
    if (cudaGetLastError() != cudaSuccess) return FV_ERR_LAUNCH;
    // the scan has consumed ws_m and ws_c: the readout's W splits reuse them
    return launch_vda_readout_tc(a, reinterpret_cast<__nv_bfloat16 *>(a.workspace), stream);
}

}  // namespace fv
