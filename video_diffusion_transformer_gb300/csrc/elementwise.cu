// Bandwidth-bound ops around the attention: the cached-AdaLN modulated
// LayerNorm and the gated residual ("FreeVideo: a 66 GB video transformer on
// an 8 GB card", section "Cut one: 26 GB of AdaLN weights become 0.22 GB of
// tables": a shift, scale and gate per schedule step read from a stored table).
//
// Both kernels give one warp a whole row (5,376 channels = 21 chunks of 8 bf16
// per lane), so a row is read once and written once: the algorithmic traffic
// is the whole traffic.  Grids are persistent: a multiple of the SM count,
// warps striding over rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "fv_internal.h"

namespace fv {
namespace {

constexpr int kEwThreads = 256;
constexpr int kEwWarps = kEwThreads / 32;

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x); f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z); f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

// The same unpacking, but opaque to common-subexpression elimination: a row
// is unpacked afresh in each of its three passes, so only the packed row
// (4 registers per chunk) stays live between passes.
__device__ __forceinline__ void unpack8_fresh(const uint4 &v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t lo, hi;
        asm volatile("shl.b32 %0, %2, 16;\n\tand.b32 %1, %2, 0xffff0000;" : "=r"(lo), "=r"(hi) : "r"(w[i]));
        f[2 * i] = __uint_as_float(lo);
        f[2 * i + 1] = __uint_as_float(hi);
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Where modulate_row reads a row's table values: shift and 1 + scale for the
// 8 channels of chunk q.  Staged: both already in shared memory (1 + scale
// precomputed).  Cached: both rows in global memory, read through the
// read-only cache, 1 is added here (the same float32 sum as when staging).
struct StagedRows {
    const float4 *sh4, *sc4;
    __device__ __forceinline__ void get(int q, float (&sh)[8], float (&sc1)[8]) const {
        const float4 a0 = sh4[2 * q], a1 = sh4[2 * q + 1];
        const float4 b0 = sc4[2 * q], b1 = sc4[2 * q + 1];
        sh[0] = a0.x; sh[1] = a0.y; sh[2] = a0.z; sh[3] = a0.w; sh[4] = a1.x; sh[5] = a1.y; sh[6] = a1.z; sh[7] = a1.w;
        sc1[0] = b0.x; sc1[1] = b0.y; sc1[2] = b0.z; sc1[3] = b0.w;
        sc1[4] = b1.x; sc1[5] = b1.y; sc1[6] = b1.z; sc1[7] = b1.w;
    }
};

struct CachedRows {
    const float4 *sh4, *sc4;
    __device__ __forceinline__ void get(int q, float (&sh)[8], float (&sc1)[8]) const {
        const float4 a0 = __ldg(sh4 + 2 * q), a1 = __ldg(sh4 + 2 * q + 1);
        const float4 b0 = __ldg(sc4 + 2 * q), b1 = __ldg(sc4 + 2 * q + 1);
        sh[0] = a0.x; sh[1] = a0.y; sh[2] = a0.z; sh[3] = a0.w; sh[4] = a1.x; sh[5] = a1.y; sh[6] = a1.z; sh[7] = a1.w;
        const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) sc1[e] = 1.0f + b[e];
    }
};

// One row of modulate by one warp: LayerNorm statistics from the row held in
// registers, then y = (x - mu) rstd * sc1 + sh with sc1 = 1 + scale (both
// float32, from `rows`).  kChunks = 16-byte chunks per lane per row
// (ceil(C / 256)).
template <int kChunks, class Rows>
__device__ __forceinline__ void modulate_row(const uint4 *__restrict__ x, void *__restrict__ y, int y_fp32,
                                             int64_t row, int c, int lane, const Rows &rows, float eps) {
    const int cq = c >> 3;
    const uint4 *xr = x + row * cq;
    uint4 v[kChunks];
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
        const int q = lane + 32 * i;
        v[i] = q < cq ? __ldcs(xr + q) : make_uint4(0u, 0u, 0u, 0u);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
        float f[8];
        unpack8_fresh(v[i], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) s += f[e];
    }
    const float mu = warp_sum(s) / (float)c;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
        if (lane + 32 * i < cq) {
            float f[8];
            unpack8_fresh(v[i], f);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float d = f[e] - mu;
                ss = fmaf(d, d, ss);
            }
        }
    }
    const float rstd = 1.0f / sqrtf(warp_sum(ss) / (float)c + eps);
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
        const int q = lane + 32 * i;
        if (q < cq) {
            float f[8];
            unpack8_fresh(v[i], f);
            float sh[8], sc[8];
            rows.get(q, sh, sc);
            float r[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) r[e] = fmaf((f[e] - mu) * rstd, sc[e], sh[e]);
            if (y_fp32) {
                float4 *yr = reinterpret_cast<float4 *>(y) + row * (int64_t)(2 * cq) + 2 * q;
                __stcs(yr, make_float4(r[0], r[1], r[2], r[3]));
                __stcs(yr + 1, make_float4(r[4], r[5], r[6], r[7]));
            } else {
                uint4 w;
                w.x = pack_bf16x2(r[0], r[1]);
                w.y = pack_bf16x2(r[2], r[3]);
                w.z = pack_bf16x2(r[4], r[5]);
                w.w = pack_bf16x2(r[6], r[7]);
                __stcs(reinterpret_cast<uint4 *>(y) + row * cq + q, w);
            }
        }
    }
}

// y = LN(x) * (1 + scale_row) + shift_row.  kChunks = 16-byte chunks per lane
// per row (ceil(C / 256)); the packed bf16 row stays in registers between the
// two reductions (mean, then mean of squared deviations) and the output pass,
// which keeps the kernel at 125 registers: two 256-thread CTAs per SM.
// Shared memory holds the step's table rows: shift[C], then 1 + scale[C].
template <int kChunks>
__global__ void __launch_bounds__(kEwThreads, kChunks <= 21 ? 2 : 1)
    modulate_kernel(const uint4 *__restrict__ x, void *__restrict__ y, int y_fp32, int64_t n, int c,
                    const float *__restrict__ shift_row, const float *__restrict__ scale_row, float eps) {
    extern __shared__ float4 tab4[];
    float *tab = reinterpret_cast<float *>(tab4);
    for (int i = (int)threadIdx.x; i < c; i += kEwThreads) {
        tab[i] = shift_row[i];
        tab[c + i] = 1.0f + scale_row[i];
    }
    __syncthreads();
    const int lane = (int)(threadIdx.x & 31);
    const StagedRows rows{reinterpret_cast<const float4 *>(tab), reinterpret_cast<const float4 *>(tab + c)};
    for (int64_t row = (int64_t)blockIdx.x * kEwWarps + (threadIdx.x >> 5); row < n;
         row += (int64_t)gridDim.x * kEwWarps)
        modulate_row<kChunks>(x, y, y_fp32, row, c, lane, rows, eps);
}

// Modulate with per-token modality rows, every modality's rows staged in
// shared memory (num_tags x 2 x c floats, up to kTaggedSmemMax): one CTA of
// 512 threads per SM, 16 rows in flight as in the untagged kernel.  A tag >=
// num_tags skips the row and records kDevBadTag in the status word.
constexpr int kTaggedThreads = 512;
constexpr int kTaggedWarps = kTaggedThreads / 32;
constexpr size_t kTaggedSmemMax = 200 * 1024;

template <int kChunks>
__global__ void __launch_bounds__(kTaggedThreads, 1)
    modulate_tagged_smem_kernel(const uint4 *__restrict__ x, void *__restrict__ y, int y_fp32, int64_t n, int c,
                                const float *__restrict__ shift_base, const float *__restrict__ scale_base,
                                int64_t ld, int row_base, const uint8_t *__restrict__ tags, int num_tags, float eps,
                                int *status) {
    extern __shared__ float4 tab4[];
    float *tab = reinterpret_cast<float *>(tab4);  // [num_tags][shift, 1 + scale][c]
    for (int i = (int)threadIdx.x; i < num_tags * c; i += kTaggedThreads) {
        const int t = i / c, j = i - t * c;
        const int64_t src = (int64_t)(row_base + t) * ld + j;
        tab[(2 * t) * c + j] = shift_base[src];
        tab[(2 * t + 1) * c + j] = 1.0f + scale_base[src];
    }
    __syncthreads();
    const int lane = (int)(threadIdx.x & 31);
    for (int64_t row = (int64_t)blockIdx.x * kTaggedWarps + (threadIdx.x >> 5); row < n;
         row += (int64_t)gridDim.x * kTaggedWarps) {
        const int tag = (int)__ldg(tags + row);
        if (tag >= num_tags) {
            if (lane == 0) atomicCAS(status, 0, kDevBadTag);
            continue;
        }
        const StagedRows rows{reinterpret_cast<const float4 *>(tab + (size_t)(2 * tag) * c),
                              reinterpret_cast<const float4 *>(tab + (size_t)(2 * tag + 1) * c)};
        modulate_row<kChunks>(x, y, y_fp32, row, c, lane, rows, eps);
    }
}

// out = x + gate_row * a, one float32 FMA per element, rounded once to bf16.
// out may be x itself: every element is read and then written by one thread.
__global__ void __launch_bounds__(kEwThreads) gated_residual_kernel(const uint4 *x, const uint4 *__restrict__ a,
                                                                    uint4 *out, int64_t n, int cq,
                                                                    const float4 *__restrict__ gate) {
    constexpr int kBatch = 8;
    const int lane = (int)(threadIdx.x & 31);
    for (int64_t row = (int64_t)blockIdx.x * kEwWarps + (threadIdx.x >> 5); row < n;
         row += (int64_t)gridDim.x * kEwWarps) {
        const int64_t base = row * cq;
        for (int q0 = 0; q0 < cq; q0 += 32 * kBatch) {
            uint4 xv[kBatch], av[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const int q = q0 + lane + 32 * i;
                if (q < cq) {
                    xv[i] = __ldcs(x + base + q);
                    av[i] = __ldcs(a + base + q);
                }
            }
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const int q = q0 + lane + 32 * i;
                if (q < cq) {
                    float fx[8], fa[8];
                    unpack8(xv[i], fx);
                    unpack8(av[i], fa);
                    const float4 g0 = __ldg(gate + 2 * q), g1 = __ldg(gate + 2 * q + 1);
                    const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                    uint4 w;
                    w.x = pack_bf16x2(fmaf(g[0], fa[0], fx[0]), fmaf(g[1], fa[1], fx[1]));
                    w.y = pack_bf16x2(fmaf(g[2], fa[2], fx[2]), fmaf(g[3], fa[3], fx[3]));
                    w.z = pack_bf16x2(fmaf(g[4], fa[4], fx[4]), fmaf(g[5], fa[5], fx[5]));
                    w.w = pack_bf16x2(fmaf(g[6], fa[6], fx[6]), fmaf(g[7], fa[7], fx[7]));
                    __stcs(out + base + q, w);
                }
            }
        }
    }
}

// Per-token modality rows: token i reads table row row_base + tags[i] (the
// pages index the AdaLN table by timestep * 3 + token tag).  This version,
// for tables too large to stage, reads the rows through the read-only cache;
// a tag >= num_tags skips the row and records kDevBadTag in the status word.
template <int kChunks>
__global__ void __launch_bounds__(kEwThreads, kChunks <= 21 ? 2 : 1)
    modulate_tagged_kernel(const uint4 *__restrict__ x, void *__restrict__ y, int y_fp32, int64_t n, int c,
                           const float *__restrict__ shift_base, const float *__restrict__ scale_base, int64_t ld,
                           int row_base, const uint8_t *__restrict__ tags, int num_tags, float eps, int *status) {
    const int lane = (int)(threadIdx.x & 31);
    for (int64_t row = (int64_t)blockIdx.x * kEwWarps + (threadIdx.x >> 5); row < n;
         row += (int64_t)gridDim.x * kEwWarps) {
        const int tag = (int)__ldg(tags + row);
        if (tag >= num_tags) {
            if (lane == 0) atomicCAS(status, 0, kDevBadTag);
            continue;
        }
        const CachedRows rows{reinterpret_cast<const float4 *>(shift_base + (int64_t)(row_base + tag) * ld),
                              reinterpret_cast<const float4 *>(scale_base + (int64_t)(row_base + tag) * ld)};
        modulate_row<kChunks>(x, y, y_fp32, row, c, lane, rows, eps);
    }
}

__global__ void __launch_bounds__(kEwThreads)
    gated_residual_tagged_kernel(const uint4 *x, const uint4 *__restrict__ a, uint4 *out, int64_t n, int cq,
                                 const float *__restrict__ gate_base, int64_t ld, int row_base,
                                 const uint8_t *__restrict__ tags, int num_tags, int *status) {
    constexpr int kBatch = 8;
    const int lane = (int)(threadIdx.x & 31);
    for (int64_t row = (int64_t)blockIdx.x * kEwWarps + (threadIdx.x >> 5); row < n;
         row += (int64_t)gridDim.x * kEwWarps) {
        const int tag = (int)__ldg(tags + row);
        if (tag >= num_tags) {
            if (lane == 0) atomicCAS(status, 0, kDevBadTag);
            continue;
        }
        const float4 *gate = reinterpret_cast<const float4 *>(gate_base + (int64_t)(row_base + tag) * ld);
        const int64_t base = row * cq;
        for (int q0 = 0; q0 < cq; q0 += 32 * kBatch) {
            uint4 xv[kBatch], av[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const int q = q0 + lane + 32 * i;
                if (q < cq) {
                    xv[i] = __ldcs(x + base + q);
                    av[i] = __ldcs(a + base + q);
                }
            }
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const int q = q0 + lane + 32 * i;
                if (q < cq) {
                    float fx[8], fa[8];
                    unpack8(xv[i], fx);
                    unpack8(av[i], fa);
                    const float4 g0 = __ldg(gate + 2 * q), g1 = __ldg(gate + 2 * q + 1);
                    const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                    uint4 w;
                    w.x = pack_bf16x2(fmaf(g[0], fa[0], fx[0]), fmaf(g[1], fa[1], fx[1]));
                    w.y = pack_bf16x2(fmaf(g[2], fa[2], fx[2]), fmaf(g[3], fa[3], fx[3]));
                    w.z = pack_bf16x2(fmaf(g[4], fa[4], fx[4]), fmaf(g[5], fa[5], fx[5]));
                    w.w = pack_bf16x2(fmaf(g[6], fa[6], fx[6]), fmaf(g[7], fa[7], fx[7]));
                    __stcs(out + base + q, w);
                }
            }
        }
    }
}

template <int kChunks>
fv_status launch_modulate_t(const void *x, void *y, bool y_fp32, int64_t n, int c, const float *shift_row,
                            const float *scale_row, float eps, int num_sms, cudaStream_t stream) {
    const size_t smem = (size_t)2 * (size_t)c * sizeof(float);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(modulate_kernel<kChunks>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
        return FV_ERR_LAUNCH;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, modulate_kernel<kChunks>, kEwThreads, smem) !=
            cudaSuccess ||
        per_sm < 1)
        return FV_ERR_LAUNCH;
    const int64_t need = (n + kEwWarps - 1) / kEwWarps;
    const int64_t full = (int64_t)num_sms * per_sm;
    const int grid = (int)(need < full ? need : full);
    modulate_kernel<kChunks><<<grid, kEwThreads, smem, stream>>>(static_cast<const uint4 *>(x), y, y_fp32 ? 1 : 0, n,
                                                                 c, shift_row, scale_row, eps);
    return cudaGetLastError() == cudaSuccess ? FV_OK : FV_ERR_LAUNCH;
}

template <int kChunks>
fv_status launch_modulate_tagged_t(const TaggedRows &t, const void *x, void *y, bool y_fp32, int64_t n, int c,
                                   float eps, int num_sms, cudaStream_t stream) {
    // (rows wider than 21 chunks per lane would spill at 512 threads)
    const size_t staged = (size_t)t.num_tags * 2 * (size_t)c * sizeof(float);
    if constexpr (kChunks <= 21) {
        if (staged <= kTaggedSmemMax) {
            static std::mutex mu;
            static bool attr_set[64] = {};
            int dev = 0;
            if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FV_ERR_LAUNCH;
            {
                std::lock_guard<std::mutex> lk(mu);
                if (!attr_set[dev]) {
                    if (cudaFuncSetAttribute(modulate_tagged_smem_kernel<kChunks>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTaggedSmemMax) !=
                        cudaSuccess)
                        return FV_ERR_LAUNCH;
                    attr_set[dev] = true;
                }
            }
            const int64_t need = (n + kTaggedWarps - 1) / kTaggedWarps;
            const int grid = (int)(need < num_sms ? need : num_sms);
            modulate_tagged_smem_kernel<kChunks><<<grid, kTaggedThreads, staged, stream>>>(
                static_cast<const uint4 *>(x), y, y_fp32 ? 1 : 0, n, c, t.table0, t.table1, t.ld, t.row_base, t.tags,
                t.num_tags, eps, t.status);
            return cudaGetLastError() == cudaSuccess ? FV_OK : FV_ERR_LAUNCH;
        }
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, modulate_tagged_kernel<kChunks>, kEwThreads, 0) !=
            cudaSuccess ||
        per_sm < 1)
        return FV_ERR_LAUNCH;
    const int64_t need = (n + kEwWarps - 1) / kEwWarps;
    const int64_t full = (int64_t)num_sms * per_sm;
    const int grid = (int)(need < full ? need : full);
    modulate_tagged_kernel<kChunks><<<grid, kEwThreads, 0, stream>>>(
        static_cast<const uint4 *>(x), y, y_fp32 ? 1 : 0, n, c, t.table0, t.table1, t.ld, t.row_base, t.tags,
        t.num_tags, eps, t.status);
    return cudaGetLastError() == cudaSuccess ? FV_OK : FV_ERR_LAUNCH;
}

}  // namespace

fv_status launch_adaln_modulate_tagged(const TaggedRows &t, const void *x, void *y, bool y_fp32, int64_t n, int c,
                                       float eps, int num_sms, cudaStream_t stream) {
    const int chunks = (c / 8 + 31) / 32;
    if (chunks <= 4) return launch_modulate_tagged_t<4>(t, x, y, y_fp32, n, c, eps, num_sms, stream);
    if (chunks <= 8) return launch_modulate_tagged_t<8>(t, x, y, y_fp32, n, c, eps, num_sms, stream);
    if (chunks <= 16) return launch_modulate_tagged_t<16>(t, x, y, y_fp32, n, c, eps, num_sms, stream);
    if (chunks <= 21) return launch_modulate_tagged_t<21>(t, x, y, y_fp32, n, c, eps, num_sms, stream);
    if (chunks <= 32) return launch_modulate_tagged_t<32>(t, x, y, y_fp32, n, c, eps, num_sms, stream);
    return FV_ERR_SHAPE;
}

fv_status launch_gated_residual_tagged(const TaggedRows &t, const void *x, const void *a, void *out, int64_t n,
                                       int c, int num_sms, cudaStream_t stream) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gated_residual_tagged_kernel, kEwThreads, 0) !=
            cudaSuccess ||
        per_sm < 1)
        return FV_ERR_LAUNCH;
    const int64_t need = (n + kEwWarps - 1) / kEwWarps;
    const int64_t full = (int64_t)num_sms * per_sm;
    const int grid = (int)(need < full ? need : full);
    gated_residual_tagged_kernel<<<grid, kEwThreads, 0, stream>>>(
        static_cast<const uint4 *>(x), static_cast<const uint4 *>(a), static_cast<uint4 *>(out), n, c / 8, t.table0,
        t.ld, t.row_base, t.tags, t.num_tags, t.status);
    return cudaGetLastError() == cudaSuccess ? FV_OK : FV_ERR_LAUNCH;
}

fv_status launch_adaln_modulate(const void *x, void *y, bool y_fp32, int64_t n, int c, const float *shift_row,
                                const float *scale_row, float eps, int num_sms, cudaStream_t stream) {
    const int chunks = (c / 8 + 31) / 32;  // 16-byte chunks per lane
    if (chunks <= 4) return launch_modulate_t<4>(x, y, y_fp32, n, c, shift_row, scale_row, eps, num_sms, stream);
    if (chunks <= 8) return launch_modulate_t<8>(x, y, y_fp32, n, c, shift_row, scale_row, eps, num_sms, stream);
    if (chunks <= 16) return launch_modulate_t<16>(x, y, y_fp32, n, c, shift_row, scale_row, eps, num_sms, stream);
    if (chunks <= 21) return launch_modulate_t<21>(x, y, y_fp32, n, c, shift_row, scale_row, eps, num_sms, stream);
    if (chunks <= 32) return launch_modulate_t<32>(x, y, y_fp32, n, c, shift_row, scale_row, eps, num_sms, stream);
    return FV_ERR_SHAPE;
}

fv_status launch_gated_residual(const void *x, const void *a, void *out, int64_t n, int c, const float *gate_row,
                                int num_sms, cudaStream_t stream) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gated_residual_kernel, kEwThreads, 0) != cudaSuccess ||
        per_sm < 1)
        return FV_ERR_LAUNCH;
    const int64_t need = (n + kEwWarps - 1) / kEwWarps;
    const int64_t full = (int64_t)num_sms * per_sm;
    const int grid = (int)(need < full ? need : full);
    gated_residual_kernel<<<grid, kEwThreads, 0, stream>>>(static_cast<const uint4 *>(x),
                                                           static_cast<const uint4 *>(a), static_cast<uint4 *>(out), n,
                                                           c / 8, reinterpret_cast<const float4 *>(gate_row));
    return cudaGetLastError() == cudaSuccess ? FV_OK : FV_ERR_LAUNCH;
}

}  // namespace fv
