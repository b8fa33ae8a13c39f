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
// Five kernels:
//   stats   (frame, head; tensor cores, delta_tc.cu): I + A_t -> ws_m, B_t^T -> ws_c
//   solve   (frame, head; float32): Gauss-Jordan inversion of I + A_t in registers,
//           M_t = (I + A_t)^{-1} -> ws_m as bf16 hi/lo operand tiles
//   scan    (head, direction; tensor cores, delta_tc.cu): S <- U M_t with
//           U = S Diag(alpha_t) + B_t, frame by frame, split-bf16 products
//           with float32 accumulation
//   wsplit  (chunk, head; delta_tc.cu): W = S_fwd[p] + S_rev[n] as bf16 hi + lo
//   readout (chunk rows, head; tensor cores, delta_tc.cu): o = W q_hat, rounded
//           to bf16
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

// (c0, c1) = (a0, a1) * b + (c0, c1): one packed instruction (sm_100+), each
// lane rounded as a single fmaf.
__device__ __forceinline__ void fma2_acc(float &c0, float &c1, float a0, float a1, float b) {
    asm("{\n\t.reg .b64 a, b, c;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %4};\n\tmov.b64 c, {%0, %1};\n\t"
        "fma.rn.f32x2 c, a, b, c;\n\tmov.b64 {%0, %1}, c;\n\t}"
        : "+f"(c0), "+f"(c1)
        : "f"(a0), "f"(a1), "f"(b));
}


// ------------------------------------------------------------------ solve
// Gauss-Jordan inversion of G = I + A_t of frame t of head h in place:
// after the 128 pivot steps G holds M = (I + A_t)^{-1}.  No pivoting is
// needed: I + A is symmetric positive definite with every Schur complement
// >= I (A is a sum of beta-weighted outer products, beta >= 0), so every
// pivot is >= 1.  The matrix lives in registers: thread (ty, tx) holds rows
// ty*8 .. ty*8+7 and columns tx*8 .. tx*8+7.  Each step broadcasts the pivot
// row and pivot column through shared memory (two alternating buffers, one
// barrier per step) and applies one update to every element: row i loses f_i
// times the pivot row divided by the pivot, with f_k - 1 for the pivot row
// itself (so it becomes the divided row), and the pivot column first set to
// the identity's column (so it becomes column k of the inverse).
// Written out for the tensor-core scan as two bf16 operand tiles, hi and lo
// (M = hi + lo to 2^-17), each [2 column halves][128 rows][64 columns] in the
// 128-byte swizzled layout (16-byte chunk j of row q at chunk j ^ (q % 8)),
// in the frame's 64 KB of ws_m.
__global__ void __launch_bounds__(kDThreads, 2) vda_solve_kernel(int frames, float *__restrict__ ws_m) {
    __shared__ __align__(16) float rowbuf[2][kDv];
    __shared__ __align__(16) float colbuf[2][kDv];
    const int t = (int)blockIdx.x + 1;
    const int h = (int)blockIdx.y;
    const size_t base = ((size_t)h * frames + t) * kMat;
    const int tid = (int)threadIdx.x, ty = tid >> 4, tx = tid & 15;
    float g[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 *src = reinterpret_cast<const float4 *>(ws_m + base + (size_t)(ty * 8 + i) * kDv + tx * 8);
        const float4 a0 = src[0], a1 = src[1];
        g[i][0] = a0.x, g[i][1] = a0.y, g[i][2] = a0.z, g[i][3] = a0.w;
        g[i][4] = a1.x, g[i][5] = a1.y, g[i][6] = a1.z, g[i][7] = a1.w;
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
                dg[0] = make_float4(g[kk][0], g[kk][1], g[kk][2], g[kk][3]);
                dg[1] = make_float4(g[kk][4], g[kk][5], g[kk][6], g[kk][7]);
            }
            if (own_col) {
                float4 *dc = reinterpret_cast<float4 *>(cb + ty * 8);
                dc[0] = make_float4(g[0][kk], g[1][kk], g[2][kk], g[3][kk]);
                dc[1] = make_float4(g[4][kk], g[5][kk], g[6][kk], g[7][kk]);
            }
            __syncthreads();
            const float p = 1.0f / rb[k];
            float rg[8], f[8];
            {
                const float4 *sg = reinterpret_cast<const float4 *>(rb + tx * 8);
                const float4 *sc = reinterpret_cast<const float4 *>(cb + ty * 8);
                const float4 g0 = sg[0], g1 = sg[1], c0 = sc[0], c1 = sc[1];
                rg[0] = g0.x, rg[1] = g0.y, rg[2] = g0.z, rg[3] = g0.w;
                rg[4] = g1.x, rg[5] = g1.y, rg[6] = g1.z, rg[7] = g1.w;
                f[0] = c0.x, f[1] = c0.y, f[2] = c0.z, f[3] = c0.w;
                f[4] = c1.x, f[5] = c1.y, f[6] = c1.z, f[7] = c1.w;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) rg[j] *= p;
            if (own_col) {
                rg[kk] = p;
#pragma unroll
                for (int i = 0; i < 8; ++i) g[i][kk] = (own_row && i == kk) ? 1.0f : 0.0f;
            }
            if (own_row) f[kk] -= 1.0f;
            // two elements per packed fma (each lane rounds as fmaf would)
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; j += 2) fma2_acc(g[i][j], g[i][j + 1], rg[j], rg[j + 1], -f[i]);
        }
    }
    uint8_t *mo = reinterpret_cast<uint8_t *>(ws_m + base);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int q = ty * 8 + i;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float v0 = g[i][2 * e], v1 = g[i][2 * e + 1];
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(v0, v1);
            const float2 hf = __bfloat1622float2(h2);
            const __nv_bfloat162 l2 = __floats2bfloat162_rn(v0 - hf.x, v1 - hf.y);
            hi[e] = *reinterpret_cast<const uint32_t *>(&h2);
            lo[e] = *reinterpret_cast<const uint32_t *>(&l2);
        }
        const size_t off = (size_t)(tx >> 3) * 16384 + (size_t)q * 128 + (size_t)(((tx & 7) ^ (q & 7)) << 4);
        *reinterpret_cast<uint4 *>(mo + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(mo + 32768 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

}  // namespace

fv_status launch_delta_attn(const DeltaLaunch &a, cudaStream_t stream) {
    const int frames = (int)(a.n / a.frame_tokens);
    float *ws_m = a.workspace;
    float *ws_c = a.workspace + (size_t)a.heads * frames * kMat;
    if (frames > 2) {
        const fv_status st = launch_vda_stats_tc(a, ws_m, ws_c, stream);
        if (st != FV_OK) return st;
        vda_solve_kernel<<<dim3(frames - 2, a.heads), kDThreads, 0, stream>>>(frames, ws_m);
        if (cudaGetLastError() != cudaSuccess) return FV_ERR_LAUNCH;
    }
    const fv_status st = launch_vda_scan_tc(a, ws_m, ws_c, stream);
    if (st != FV_OK) return st;
    // the scan has consumed ws_m and ws_c: the readout's W splits reuse them
    return launch_vda_readout_tc(a, reinterpret_cast<__nv_bfloat16 *>(a.workspace), stream);
}

}  // namespace fv
