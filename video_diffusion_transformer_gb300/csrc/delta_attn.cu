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
//   solve   (frame, head; float32): symmetric sweep (Gauss-Jordan) inversion of
//           I + A_t over its upper triangle in registers,
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
// Inversion of G = I + A_t of frame t of head h by the symmetric sweep
// (Gauss-Jordan elimination that keeps the matrix symmetric): sweeping pivot
// k with d = g_kk maps
//   g_ij -> g_ij - g_ik g_kj / d   (i, j != k),
//   g_ik = g_ki -> g_ik / d        (i != k),
//   g_kk -> -1 / d,
// and after all 128 pivots G holds -(I + A_t)^{-1}.  No pivoting is needed:
// I + A is symmetric positive definite with every Schur complement >= I (A is
// a sum of beta-weighted outer products, beta >= 0), so every pivot is >= 1.
// As every step keeps G symmetric, only its upper triangle is swept, in the
// 136 blocks of 8 x 8 on or above the diagonal; a thread holds kSolveRows
// rows of one block in registers.  Step k broadcasts row k of G (its part
// right of the diagonal from block row k / 8, the rest from block column
// k / 8) and 1/d through shared memory (two alternating buffers, one barrier
// per step), and every element then takes one multiply-add g_ab -= u_a r_b
// with u = r / d for the thread's rows and r for its columns; the pivot row
// and column are cleared first and their entries of u and r set to -1/d and
// -1, so that the same multiply-add leaves r / d in them and -1/d on the
// diagonal.  1/d is the hardware reciprocal (rcp.approx, within 1 ulp).
// Written out negated, for the tensor-core scan, as two bf16 operand tiles,
// hi and lo (M = hi + lo to 2^-17), each [2 column halves][128 rows][64
// columns] in the 128-byte swizzled layout (16-byte chunk j of row q at chunk
// j ^ (q % 8)), in the frame's 64 KB of ws_m; an off-diagonal block is
// written at its place and transposed at the mirrored one.
constexpr int kSolveRows = 4;                                  // rows of a block a thread holds
constexpr int kSolveSplit = 8 / kSolveRows;                    // threads per 8 x 8 block
constexpr int kSweepBlocks = (kDv / 8) * (kDv / 8 + 1) / 2;   // 136 upper-triangle blocks
constexpr int kSolveThreads = kSweepBlocks * kSolveSplit;
constexpr int kSolveCtasPerSm = 3;

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// n = 4 or 8 values of row q of M, columns 8 cb + c0 .. 8 cb + c0 + n - 1, as hi
// and lo bf16 operand bytes.
template <int n>
__device__ __forceinline__ void store_m(uint8_t *mo, int q, int cb, int c0, const float (&v)[n]) {
    uint32_t hi[n / 2], lo[n / 2];
#pragma unroll
    for (int e = 0; e < n / 2; ++e) {
        const float v0 = -v[2 * e], v1 = -v[2 * e + 1];
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(v0, v1);
        const float2 hf = __bfloat1622float2(h2);
        const __nv_bfloat162 l2 = __floats2bfloat162_rn(v0 - hf.x, v1 - hf.y);
        hi[e] = *reinterpret_cast<const uint32_t *>(&h2);
        lo[e] = *reinterpret_cast<const uint32_t *>(&l2);
    }
    const size_t off =
        (size_t)(cb >> 3) * 16384 + (size_t)q * 128 + (size_t)(((cb & 7) ^ (q & 7)) << 4) + (size_t)(c0 * 2);
    if (n == 8) {
        *reinterpret_cast<uint4 *>(mo + off) = make_uint4(hi[0], hi[1], hi[2 % (n / 2)], hi[3 % (n / 2)]);
        *reinterpret_cast<uint4 *>(mo + 32768 + off) = make_uint4(lo[0], lo[1], lo[2 % (n / 2)], lo[3 % (n / 2)]);
    } else {
        *reinterpret_cast<uint2 *>(mo + off) = make_uint2(hi[0], hi[1]);
        *reinterpret_cast<uint2 *>(mo + 32768 + off) = make_uint2(lo[0], lo[1]);
    }
}

__global__ void __launch_bounds__(kSolveThreads, kSolveCtasPerSm) vda_solve_kernel(int frames, float *__restrict__ ws_m) {
    __shared__ __align__(16) float rowbuf[2][kDv];
    __shared__ float pbuf[2];
    const int t = (int)blockIdx.x + 1;
    const int h = (int)blockIdx.y;
    const size_t base = ((size_t)h * frames + t) * kMat;
    // thread -> (block (bi, bj) of the upper triangle, row by row; part hp of its rows)
    const int hp = (int)threadIdx.x % kSolveSplit;
    int bi = 0, rem = (int)threadIdx.x / kSolveSplit;
    while (rem >= kDv / 8 - bi) {
        rem -= kDv / 8 - bi;
        ++bi;
    }
    const int bj = bi + rem;
    const int row0 = bi * 8 + hp * kSolveRows;   // first row this thread holds
    float g[kSolveRows][8];
#pragma unroll
    for (int i = 0; i < kSolveRows; ++i) {
        const float4 *src = reinterpret_cast<const float4 *>(ws_m + base + (size_t)(row0 + i) * kDv + bj * 8);
        const float4 a0 = src[0], a1 = src[1];
        g[i][0] = a0.x, g[i][1] = a0.y, g[i][2] = a0.z, g[i][3] = a0.w;
        g[i][4] = a1.x, g[i][5] = a1.y, g[i][6] = a1.z, g[i][7] = a1.w;
    }
    for (int kb = 0; kb < kDv / 8; ++kb) {
        const bool own_col = bj == kb;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int kr = kk % kSolveRows;            // the pivot row's index among a holder's rows
            const bool own_row = bi == kb && hp == kk / kSolveRows;
            float *rb = rowbuf[kk & 1];
            if (own_row) {
                float4 *dg = reinterpret_cast<float4 *>(rb + bj * 8);
                dg[0] = make_float4(g[kr][0], g[kr][1], g[kr][2], g[kr][3]);
                dg[1] = make_float4(g[kr][4], g[kr][5], g[kr][6], g[kr][7]);
                if (own_col) pbuf[kk & 1] = rcp_approx(g[kr][kk]);
            } else if (own_col && bi != kb) {
                float *dc = rb + row0;
#pragma unroll
                for (int i = 0; i < kSolveRows; i += 4)
                    *reinterpret_cast<float4 *>(dc + i) = make_float4(g[i][kk], g[i + 1][kk], g[i + 2][kk], g[i + 3][kk]);
            }
            __syncthreads();
            const float p = pbuf[kk & 1];
            float u[kSolveRows], r[8];
            {
                const float4 *sr = reinterpret_cast<const float4 *>(rb + bj * 8);
                const float4 r0 = sr[0], r1 = sr[1];
                r[0] = r0.x, r[1] = r0.y, r[2] = r0.z, r[3] = r0.w;
                r[4] = r1.x, r[5] = r1.y, r[6] = r1.z, r[7] = r1.w;
#pragma unroll
                for (int i = 0; i < kSolveRows; i += 4) {
                    const float4 su = *reinterpret_cast<const float4 *>(rb + row0 + i);
                    u[i] = su.x, u[i + 1] = su.y, u[i + 2] = su.z, u[i + 3] = su.w;
                }
            }
#pragma unroll
            for (int i = 0; i < kSolveRows; ++i) u[i] *= -p;   // -(row k) / d at the thread's rows
            if (own_row) {
                u[kr] = p;
#pragma unroll
                for (int j = 0; j < 8; ++j) g[kr][j] = 0.0f;
            }
            if (own_col) {
                r[kk] = -1.0f;
#pragma unroll
                for (int i = 0; i < kSolveRows; ++i) g[i][kk] = 0.0f;
            }
            // two elements per packed fma (each lane rounds as fmaf would)
#pragma unroll
            for (int i = 0; i < kSolveRows; ++i)
#pragma unroll
                for (int j = 0; j < 8; j += 2) fma2_acc(g[i][j], g[i][j + 1], r[j], r[j + 1], u[i]);
        }
    }
    uint8_t *mo = reinterpret_cast<uint8_t *>(ws_m + base);
#pragma unroll
    for (int i = 0; i < kSolveRows; ++i) store_m<8>(mo, row0 + i, bj, 0, g[i]);
    if (bi != bj) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float col[kSolveRows];
#pragma unroll
            for (int i = 0; i < kSolveRows; ++i) col[i] = g[i][j];
            store_m<kSolveRows>(mo, bj * 8 + j, bi, hp * kSolveRows, col);
        }
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
        vda_solve_kernel<<<dim3(frames - 2, a.heads), kSolveThreads, 0, stream>>>(frames, ws_m);
        if (cudaGetLastError() != cudaSuccess) return FV_ERR_LAUNCH;
    }
    const fv_status st = launch_vda_scan_tc(a, ws_m, ws_c, stream);
    if (st != FV_OK) return st;
    // the scan has consumed ws_m and ws_c: the readout's W splits reuse them
    return launch_vda_readout_tc(a, reinterpret_cast<__nv_bfloat16 *>(a.workspace), stream);
}

}  // namespace fv
