// VSA-style block-sparse attention over a video latent grid for sm_103a.
//
// "FastH3 Preview v1: four calls, one-tenth the attention, and what the 14x
// actually measures", section "Lever two: VSA-H3 makes each of the four calls
// cheaper": the video tokens of a (frames, height, width) latent grid are cut
// into 3D tiles of (4, 4, 4) = 64 tokens; a coarse stage scores every (query
// tile, key tile) pair from the tiles' mean query and mean key; each query
// tile keeps its top-k key tiles; every query then attends exactly, with the
// softmax, to the keys of its tile's kept tiles.  Tiles on the far edges of
// the grid hold fewer tokens; their means are over their own tokens and their
// missing tokens are masked.  Ties in the coarse score go to the lower tile.
//
// Three kernels:
//   vsa_pool    (tile): float32 means of q and k of every head over the tile;
//   vsa_select  (head, pair of query tiles 2p, 2p+1): coarse scores against
//               every key tile, the top-k of each of the two rows (a 32-step
//               search for the k-th largest score, ties to the lower index),
//               written as ascending tile lists, and the union of the two
//               lists with one owner bit per query tile, ordered so that a
//               K/V tile pairs a tile of one list only with a tile of the
//               other only (then the tiles both keep);
//   vsa_fine    (persistent, one CTA per SM): unit = (head, pair).  A 128-row
//               Q tile holds the pair's two query tiles (rows 0-63, 64-127),
//               each brought in by one 4D TMA box {64 channels, 4, 4, 4}
//               straight from the token-major tensor, so no permuted copy is
//               made; a K/V tile holds two key tiles of the union.  A warp's
//               32 rows all belong to one query tile, so which of the two key
//               tiles it sees is one warp-uniform bit each.  The two softmax
//               warpgroups split the K/V tiles of a unit (even / odd) and keep
//               their own running max, sum and O in tensor memory; at the end
//               of the unit they exchange (max, sum) through shared memory and
//               each writes half of the merged output columns.
// All waits are bounded; a wait that runs out records kDevTimeout | where.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "fv_internal.h"
#include "sm103_ptx.cuh"

namespace fv {
namespace {

constexpr int kD = 128;
constexpr int kTok = 64;                      // tokens of a tile
constexpr int kRows = 128;                    // rows of a Q tile, keys of a K/V tile
constexpr int kStages = 4;                    // K/V ring slots (5 or 6 measured no faster)
constexpr int kQSlots = 2;                    // Q tiles in flight
constexpr int kHalfBytes = kRows * 64 * 2;    // 128 rows x 64 channels (16 KB)
constexpr int kTileBytes = 2 * kHalfBytes;    // 32 KB
constexpr int kBoxBytes = kTok * 64 * 2;      // one tile x 64 channels (8 KB)
constexpr int kKeptBytes = 2 * kBoxBytes;     // one kept tile, both channel halves (16 KB)
constexpr uint32_t kGroupBytes = 2048;        // 8 rows x both channel halves of a K/V operand tile
constexpr int kThreads = 352;                 // warps 0-7 softmax, 8 TMA, 9-10 MMA
constexpr int kTmaWarp = 8, kMmaWarp = 9;     // MMA warp 9 + g issues group g's work
constexpr uint32_t kTmemCols = 512;
constexpr float kRedoSum = 1048576.0f;        // 2^20: largest half sum kept against the reference max
constexpr int kMaxTiles = 16384;              // tile index fits the low 16 bits of a list entry

// Load L of the K/V ring goes to slot L % kStages and completes on full
// barrier L % (2 kStages): with two MMA threads taking loads out of order a
// thread may wait on its load while the slot's previous use is still pending,
// and a period of twice the slot count keeps that wait from matching an older
// phase (see mma_issuer).
constexpr int kKvFullBars = 2 * kStages;
constexpr int kBarKvFull = 0;
constexpr int kBarKvEmpty = kBarKvFull + kKvFullBars;
constexpr int kBarQFull = kBarKvEmpty + kStages;
constexpr int kBarQEmpty = kBarQFull + kQSlots;
constexpr int kBarSFull = kBarQEmpty + kQSlots;
constexpr int kBarPFull = kBarSFull + 2;
constexpr int kBarOFull = kBarPFull + 2;
constexpr int kBarMlReady = kBarOFull + 2;
constexpr int kBarMerged = kBarMlReady + 1;
constexpr int kBarDrain = kBarMerged + 1;     // one per MMA issuer
constexpr int kNumBars = kBarDrain + 2;

constexpr int kSmemQ = 0;
constexpr int kSmemKV = kSmemQ + kQSlots * kTileBytes;
constexpr int kSmemMl = kSmemKV + kStages * kTileBytes;   // [2 units][2 groups][max, sum][128] float
constexpr int kSmemBar = kSmemMl + 2 * 2 * 2 * kRows * 4;
constexpr int kSmemMisc = kSmemBar + kNumBars * 8;
constexpr int kSmemBytes = kSmemMisc + 16 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

constexpr int kWhereQEmpty = 1, kWhereKvEmpty = 2, kWhereQFull = 3, kWhereKvFull = 4, kWherePFull = 5,
              kWhereSFull = 6, kWhereOFull = 7, kWhereDrain = 8, kWhereMl = 9, kWhereMerged = 10;

struct Geo {
    int frames, height, width;
    int tiles_h, tiles_w;  // tile grid along h and w
    int num_tiles;
};

struct TileCoord {
    int t0, h0, w0;  // first token of the tile along each axis
};

__host__ __device__ __forceinline__ TileCoord tile_coord(const Geo &g, int tile) {
    TileCoord c;
    c.w0 = 4 * (tile % g.tiles_w);
    c.h0 = 4 * ((tile / g.tiles_w) % g.tiles_h);
    c.t0 = 4 * (tile / (g.tiles_w * g.tiles_h));
    return c;
}

// Bit r of the result is set when row r = 16 lt + 4 lh + lw of the tile's
// box is a token of the grid.
__device__ __forceinline__ uint64_t tile_token_mask(const Geo &g, int tile) {
    const TileCoord c = tile_coord(g, tile);
    const int nw = min(4, g.width - c.w0), nh = min(4, g.height - c.h0), nt = min(4, g.frames - c.t0);
    const uint32_t row = (1u << nw) - 1u;
    uint32_t plane = 0;
    for (int i = 0; i < nh; ++i) plane |= row << (4 * i);
    uint64_t m = 0;
    for (int i = 0; i < nt; ++i) m |= (uint64_t)plane << (16 * i);
    return m;
}

// ----------------------------------------------------------------- pool
// Tile blockIdx.x: the means of q and k of every head over the tile's tokens,
// and a tile-major copy of K and V for the fine kernel.  Thread handles 8
// channels (16 bytes) of every head-row at a time, the tile's 64 box rows in
// raster order (rows outside the grid are copied as zeros).
//
// Copy layout: [heads, tiles, 8 row groups, 2 channel halves, 8 rows,
// 64 channels] bf16: each tile one contiguous 16 KB block, already in the
// 128-byte swizzled order the tensor core reads (16-byte chunk j of row r
// stored at chunk j ^ (r % 8)), so the fine kernel fetches a kept tile with
// one bulk copy and its operand descriptors step 2 KB per 8 rows.
__global__ void __launch_bounds__(256)
    vsa_pool_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                    const __nv_bfloat16 *__restrict__ v, Geo g, int heads, float *__restrict__ qbar,
                    float *__restrict__ kbar, __nv_bfloat16 *__restrict__ kp, __nv_bfloat16 *__restrict__ vp) {
    const int tile = (int)blockIdx.x;
    const TileCoord c = tile_coord(g, tile);
    const int nw = min(4, g.width - c.w0), nh = min(4, g.height - c.h0), nt = min(4, g.frames - c.t0);
    const int ld = heads * kD;
    const float count = (float)(nw * nh * nt);
    for (int ch = (int)threadIdx.x; ch < ld / 8; ch += (int)blockDim.x) {
        const int h = (ch * 8) / kD, half = ((ch * 8) % kD) / 64, j = ch & 7;
        const size_t blk = ((size_t)h * g.num_tiles + tile) * (size_t)(kKeptBytes / 2) + (size_t)half * 512;
        float sq[8], sk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) sq[e] = sk[e] = 0.f;
        // four tokens' loads in flight per thread (one at a time left HBM at 81 %)
#pragma unroll 4
        for (int r = 0; r < kTok; ++r) {
            const int lt = r >> 4, lh = (r >> 2) & 3, lw = r & 3;
            uint4 kk = make_uint4(0u, 0u, 0u, 0u), vv = make_uint4(0u, 0u, 0u, 0u);
            if (lt < nt && lh < nh && lw < nw) {
                const int64_t tok = ((int64_t)(c.t0 + lt) * g.height + (c.h0 + lh)) * g.width + (c.w0 + lw);
                const uint4 a = *reinterpret_cast<const uint4 *>(q + tok * ld + ch * 8);
                kk = *reinterpret_cast<const uint4 *>(k + tok * ld + ch * 8);
                vv = *reinterpret_cast<const uint4 *>(v + tok * ld + ch * 8);
                const __nv_bfloat162 *pa = reinterpret_cast<const __nv_bfloat162 *>(&a);
                const __nv_bfloat162 *pb = reinterpret_cast<const __nv_bfloat162 *>(&kk);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 fa = __bfloat1622float2(pa[e]), fb = __bfloat1622float2(pb[e]);
                    sq[2 * e] += fa.x;
                    sq[2 * e + 1] += fa.y;
                    sk[2 * e] += fb.x;
                    sk[2 * e + 1] += fb.y;
                }
            }
            const size_t off = blk + (size_t)(r >> 3) * 1024 + (size_t)(r & 7) * 64 + (size_t)((j ^ (r & 7)) * 8);
            *reinterpret_cast<uint4 *>(kp + off) = kk;
            *reinterpret_cast<uint4 *>(vp + off) = vv;
        }
        const int d = (ch * 8) % kD;
        float *dq = qbar + ((size_t)h * g.num_tiles + tile) * kD + d;
        float *dk = kbar + ((size_t)h * g.num_tiles + tile) * kD + d;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            dq[e] = sq[e] / count;
            dk[e] = sk[e] / count;
        }
    }
}

// --------------------------------------------------------------- select
// Order-preserving key of a float score (+0 and -0 map to the same key).
__device__ __forceinline__ uint32_t score_key(float f) {
    const uint32_t u = __float_as_uint(f + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The k-th largest key of keys[0, n), found bit by bit by one warp.  Each
// pass counts the keys at or above a candidate; the count runs four
// independent loads per lane at a time (one shared-memory load in flight per
// lane made every pass a chain of ~38 load latencies).
__device__ uint32_t kth_largest_key(const uint32_t *keys, int n, int k, int lane) {
    uint32_t t = 0;
    for (int b = 31; b >= 0; --b) {
        const uint32_t cand = t | (1u << b);
        int c0 = 0, c1 = 0, c2 = 0, c3 = 0;
        int i = lane;
        for (; i + 96 < n; i += 128) {
            const uint32_t k0 = keys[i], k1 = keys[i + 32], k2 = keys[i + 64], k3 = keys[i + 96];
            c0 += k0 >= cand ? 1 : 0;
            c1 += k1 >= cand ? 1 : 0;
            c2 += k2 >= cand ? 1 : 0;
            c3 += k3 >= cand ? 1 : 0;
        }
        for (; i < n; i += 32) c0 += keys[i] >= cand ? 1 : 0;
        const int cnt = (int)__reduce_add_sync(0xffffffffu, (unsigned)((c0 + c1) + (c2 + c3)));
        if (cnt >= k) t = cand;
    }
    return t;
}

// One CTA per (group of up to 8 pairs of query tiles, head): the coarse
// scores of the group's query tiles against every key tile (a thread scores
// whole key tiles, the query means in shared memory), then per query tile the
// top-k (one warp per row), then per pair the two ascending lists and their
// union (one warp per pair).
constexpr int kSelMaxRows = 16;
constexpr int kSelSmemBytes = 200 * 1024;

int select_pairs_per_cta(int num_tiles) {
    const int floats = kSelSmemBytes / 4 - kSelMaxRows * kD;
    const int rows = floats / num_tiles;
    const int pairs = rows / 2;
    return pairs < 1 ? 1 : (pairs > kSelMaxRows / 2 ? kSelMaxRows / 2 : pairs);
}

__global__ void __launch_bounds__(256, 1)
    vsa_select_kernel(const float *__restrict__ qbar, const float *__restrict__ kbar, Geo g, int pairs,
                      int pairs_per_cta, int topk, int32_t *__restrict__ selected, int32_t *__restrict__ lists,
                      int32_t *__restrict__ counts) {
    extern __shared__ uint32_t sh[];
    float *qs = reinterpret_cast<float *>(sh);  // [kSelMaxRows][128] query means
    uint32_t *keys = sh + kSelMaxRows * kD;     // [rows][num_tiles] score keys
    __shared__ uint32_t thr[kSelMaxRows];
    const int p0 = (int)blockIdx.x * pairs_per_cta, h = (int)blockIdx.y;
    const int np = min(pairs_per_cta, pairs - p0);
    const int nt = g.num_tiles;
    const int tid = (int)threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // rows past the group (or past the last tile) repeat the last tile; their
    // scores are never used
    for (int e = tid; e < kSelMaxRows * kD; e += (int)blockDim.x) {
        const int tile = min(2 * p0 + e / kD, nt - 1);
        qs[e] = qbar[((size_t)h * nt + tile) * kD + e % kD];
    }
    __syncthreads();
    const int rows = 2 * np;
    // a thread scores key tiles c and c + blockDim.x together, so each query
    // mean read from shared memory feeds both (the second tile repeats the
    // first past the end; its scores are not stored)
    for (int c = tid; c < nt; c += 2 * (int)blockDim.x) {
        const int c2 = c + (int)blockDim.x < nt ? c + (int)blockDim.x : c;
        const float4 *kr = reinterpret_cast<const float4 *>(kbar + ((size_t)h * nt + c) * kD);
        const float4 *kr2 = reinterpret_cast<const float4 *>(kbar + ((size_t)h * nt + c2) * kD);
        float acc[kSelMaxRows], acc2[kSelMaxRows];
#pragma unroll
        for (int r = 0; r < kSelMaxRows; ++r) acc[r] = 0.f, acc2[r] = 0.f;
#pragma unroll 2
        for (int d4 = 0; d4 < kD / 4; ++d4) {
            const float4 kk = kr[d4], kk2 = kr2[d4];
#pragma unroll
            for (int r = 0; r < kSelMaxRows; ++r) {
                const float4 qq = *reinterpret_cast<const float4 *>(qs + r * kD + 4 * d4);
                acc[r] = fmaf(qq.x, kk.x, fmaf(qq.y, kk.y, fmaf(qq.z, kk.z, fmaf(qq.w, kk.w, acc[r]))));
                acc2[r] = fmaf(qq.x, kk2.x, fmaf(qq.y, kk2.y, fmaf(qq.z, kk2.z, fmaf(qq.w, kk2.w, acc2[r]))));
            }
        }
#pragma unroll
        for (int r = 0; r < kSelMaxRows; ++r)
            if (r < rows) {
                keys[r * nt + c] = score_key(acc[r]);
                if (c2 != c) keys[r * nt + c2] = score_key(acc2[r]);
            }
    }
    __syncthreads();
    for (int r = warp; r < rows; r += 8) {
        const uint32_t t = kth_largest_key(keys + r * nt, nt, topk, lane);
        if (lane == 0) thr[r] = t;
    }
    __syncthreads();
    // One warp per pair walks the tiles in ascending order, 32 at a time: a
    // tile is kept when its key beats the threshold, or equals it and enough
    // lower tiles with the same key have not already filled the k slots.
    // The union is written so that K/V tile j (entries 2j, 2j+1) pairs a tile
    // only query tile a keeps with one only b keeps: every warp then has one
    // 64-key half to work on per K/V tile instead of zero or two.  Order:
    // a-only and b-only interleaved, the longer side's excess, then the tiles
    // both keep, each group ascending.  Two passes: the first counts.
    const uint32_t below = (1u << lane) - 1u;
    for (int pp = warp; pp < np; pp += 8) {
        const int p = p0 + pp;
        const uint32_t *ka_row = keys + (2 * pp) * nt, *kb_row = keys + (2 * pp + 1) * nt;
        const bool has_b = 2 * p + 1 < nt;
        const uint32_t ta = thr[2 * pp], tb = thr[2 * pp + 1];
        int gt_a = 0, gt_b = 0;
        for (int i = lane; i < nt; i += 32) {
            gt_a += ka_row[i] > ta ? 1 : 0;
            gt_b += kb_row[i] > tb ? 1 : 0;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            gt_a += __shfl_xor_sync(0xffffffffu, gt_a, o);
            gt_b += __shfl_xor_sync(0xffffffffu, gt_b, o);
        }
        const int eq_room_a = topk - gt_a, eq_room_b = topk - gt_b;
        // keep flags of tile base + lane; eq_a, eq_b count the tiles below base
        // whose key equals the threshold, and advance past this batch
        auto keeps = [&](int base, int &eq_a, int &eq_b, bool &keep_a, bool &keep_b) {
            const int c = base + lane;
            const bool in = c < nt;
            const uint32_t ka = in ? ka_row[c] : 0u, kb = in ? kb_row[c] : 0u;
            const uint32_t ea = __ballot_sync(0xffffffffu, in && ka == ta);
            const uint32_t eb = __ballot_sync(0xffffffffu, in && kb == tb);
            keep_a = in && (ka > ta || (ka == ta && eq_a + __popc(ea & below) < eq_room_a));
            keep_b = has_b && in && (kb > tb || (kb == tb && eq_b + __popc(eb & below) < eq_room_b));
            eq_a += __popc(ea);
            eq_b += __popc(eb);
        };
        int only_a = 0, only_b = 0;
        {
            int eq_a = 0, eq_b = 0;
            for (int base = 0; base < nt; base += 32) {
                bool keep_a, keep_b;
                keeps(base, eq_a, eq_b, keep_a, keep_b);
                only_a += __popc(__ballot_sync(0xffffffffu, keep_a && !keep_b));
                only_b += __popc(__ballot_sync(0xffffffffu, keep_b && !keep_a));
            }
        }
        const int mn = min(only_a, only_b), mx = max(only_a, only_b);
        int eq_a = 0, eq_b = 0, na = 0, nb = 0, ia = 0, ib = 0, is = 0;
        int32_t *sel_a = selected + ((size_t)h * nt + 2 * p) * topk;
        int32_t *sel_b = selected + ((size_t)h * nt + 2 * p + 1) * topk;
        int32_t *uni = lists + ((size_t)h * pairs + p) * 2 * topk;
        for (int base = 0; base < nt; base += 32) {
            const int c = base + lane;
            bool keep_a, keep_b;
            keeps(base, eq_a, eq_b, keep_a, keep_b);
            const uint32_t ba = __ballot_sync(0xffffffffu, keep_a);
            const uint32_t bb = __ballot_sync(0xffffffffu, keep_b);
            const uint32_t boa = __ballot_sync(0xffffffffu, keep_a && !keep_b);
            const uint32_t bob = __ballot_sync(0xffffffffu, keep_b && !keep_a);
            const uint32_t bs = ba & bb;
            if (keep_a) sel_a[na + __popc(ba & below)] = c;
            if (keep_b) sel_b[nb + __popc(bb & below)] = c;
            int pos = -1;
            if (keep_a && keep_b) {
                pos = mn + mx + is + __popc(bs & below);
            } else if (keep_a) {
                const int i = ia + __popc(boa & below);
                pos = i < mn ? 2 * i : mn + i;
            } else if (keep_b) {
                const int i = ib + __popc(bob & below);
                pos = i < mn ? 2 * i + 1 : mn + i;
            }
            if (pos >= 0) uni[pos] = c | (keep_a ? 1 << 16 : 0) | (keep_b ? 1 << 17 : 0);
            na += __popc(ba);
            nb += __popc(bb);
            ia += __popc(boa);
            ib += __popc(bob);
            is += __popc(bs);
        }
        const int nu = mn + mx + is;
        if (lane == 0) counts[(size_t)h * pairs + p] = nu;
    }
}

// ----------------------------------------------------------------- fine
// K/V tiles of a unit with `cnt` union entries: two kept tiles per K/V tile,
// at least two K/V tiles (an all-absent second one when the union has one or
// two tiles) so that each MMA issuer has work in every unit.
__device__ __forceinline__ int kv_tiles(int cnt) { return cnt > 2 ? (cnt + 1) / 2 : 2; }

struct Params {
    __nv_bfloat16 *o;
    float *lse;
    int *status;
    const int32_t *lists;   // [heads, pairs, list_ld] union entries: tile | owner bits << 16
    const int32_t *counts;  // [heads, pairs]
    const uint8_t *kp, *vp; // tile-major copies of K and V (16 KB per tile)
    const uint8_t *zero;    // 16 KB of zeros, stands in for an absent tile
    Geo g;
    int n, ld, pairs, num_units, list_ld;
    float scale_log2;
    int64_t skip_load;      // test hook: CTA 0 never issues its K/V load number skip_load (-1: off)
};

struct Smem {
    uint32_t q, kv, bar;
    float *ml;
    volatile int *abort_flag;
    __device__ uint32_t b(int i) const { return bar + 8u * (uint32_t)i; }
};

__device__ __forceinline__ bool wait_bar(const Smem &sm, int i, uint32_t parity, const Params &p, int where) {
    return ptx::mbar_wait(sm.b(i), parity, sm.abort_flag, p.status, kDevTimeout | where);
}

__device__ __forceinline__ void drain_bar(const Smem &sm, int i, uint32_t parity, const Params &p) {
    int never = 0;
    ptx::mbar_wait(sm.b(i), parity, &never, p.status, kDevTimeout | kWhereDrain);
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1, int c2,
                                            int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], "
        "[%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// Both channel halves of one tile into rows [64 half, 64 half + 64) of a
// 32 KB operand tile.  A tile index past the grid loads a box that lies wholly
// outside the tensor, which TMA fills with zeros.
__device__ __forceinline__ void load_tile(const CUtensorMap *map, const Params &p, uint32_t dst, int half, int tile,
                                          int x0, uint32_t bar) {
    TileCoord c{p.g.frames, 0, 0};
    if (tile < p.g.num_tiles) c = tile_coord(p.g, tile);
    const uint32_t d = dst + (uint32_t)(half * kBoxBytes);
    tma_load_4d(d, map, bar, x0, c.w0, c.h0, c.t0);
    tma_load_4d(d + kHalfBytes, map, bar, x0 + 64, c.w0, c.h0, c.t0);
}

// Kept tile `tile` of head `head` into rows [64 pos, 64 pos + 64) of a 32 KB
// K or V operand tile (8-row groups 2 KB apart, both channel halves in each):
// one 16 KB bulk copy from the tile-major copy (an absent tile, index >=
// tiles, copies zeros).
__device__ __forceinline__ void load_kv_tile(const uint8_t *src_base, const Params &p, uint32_t dst, int pos,
                                             int head, int tile, uint32_t bar) {
    const uint8_t *src =
        tile < p.g.num_tiles ? src_base + ((size_t)head * p.g.num_tiles + tile) * (size_t)kKeptBytes : p.zero;
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst + (uint32_t)(pos * kKeptBytes)),
        "l"(src), "n"(kKeptBytes), "r"(bar)
        : "memory");
}

// A softmax warp's view of one unit's list: for batches of 32 entries, one
// per lane, the 64-bit mask of the tile's columns this warp's query tile
// (owner bit 16 + qhalf) sees; the batch after next is already in flight.
// Read with shuffles, so the per-tile path has no global-memory load.  Every
// lane calls tile() with the same, never decreasing, index; entries past the
// count read as 0xFFFF (no tile, no owner).
struct MaskWindow {
    const int32_t *lst;
    const Geo *g;
    int cnt, lane, base, qhalf;
    uint32_t m0lo, m0hi, m1lo, m1hi;
    int raw2;
    __device__ __forceinline__ int ld(int batch) const {
        const int i = batch * 32 + lane;
        return i < cnt ? lst[i] : 0xFFFF;
    }
    __device__ __forceinline__ void masks(int e, uint32_t &lo, uint32_t &hi) const {
        const uint64_t m = ((e >> (16 + qhalf)) & 1) ? tile_token_mask(*g, e & 0xFFFF) : 0ull;
        lo = (uint32_t)m;
        hi = (uint32_t)(m >> 32);
    }
    __device__ __forceinline__ void init(const int32_t *l, int c, int ln, int qh, const Geo *geo) {
        lst = l;
        cnt = c;
        lane = ln;
        qhalf = qh;
        g = geo;
        base = 0;
        const int r0 = ld(0), r1 = ld(1);
        raw2 = ld(2);
        masks(r0, m0lo, m0hi);
        masks(r1, m1lo, m1hi);
    }
    // columns of K/V tile j: mk[0..1] from entry 2j, mk[2..3] from entry 2j+1
    __device__ __forceinline__ void tile(int j, uint32_t (&mk)[4]) {
        while (((2 * j) >> 5) - base >= 1) {
            m0lo = m1lo;
            m0hi = m1hi;
            masks(raw2, m1lo, m1hi);
            raw2 = ld(base + 3);
            ++base;
        }
        // entry 2j is in batch base; entry 2j + 1 is too (2j is even)
        const int src = (2 * j) & 31;
        mk[0] = __shfl_sync(0xffffffffu, m0lo, src);
        mk[1] = __shfl_sync(0xffffffffu, m0hi, src);
        mk[2] = __shfl_sync(0xffffffffu, m0lo, src + 1);
        mk[3] = __shfl_sync(0xffffffffu, m0hi, src + 1);
    }
};

// One thread (lane 0 of the TMA warp) issues every copy.
__device__ void producer(const CUtensorMap *tq, const Params &p, const Smem &sm, int lane) {
    if (lane != 0) return;
    uint32_t loads = 0, q_loads = 0;
    // Test hook: a load that is never issued, so that a consumer's bounded
    // wait runs out.  It must not be waited for in the drain below.
    const int64_t skipped = blockIdx.x == 0 ? p.skip_load : -1;
    bool ok = true;
    for (int unit = blockIdx.x; ok && unit < p.num_units; unit += gridDim.x) {
        const int head = unit / p.pairs, pr = unit % p.pairs;
        const int x0 = head * kD;
        const uint32_t qs = q_loads % kQSlots;
        ok = wait_bar(sm, kBarQEmpty + (int)qs, ((q_loads / kQSlots) & 1u) ^ 1u, p, kWhereQEmpty);
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(sm.b(kBarQFull + (int)qs), kTileBytes);
        const uint32_t qdst = sm.q + qs * (uint32_t)kTileBytes;
        load_tile(tq, p, qdst, 0, 2 * pr, x0, sm.b(kBarQFull + (int)qs));
        load_tile(tq, p, qdst, 1, 2 * pr + 1, x0, sm.b(kBarQFull + (int)qs));
        ++q_loads;
        const int32_t *lst = p.lists + ((size_t)head * p.pairs + pr) * p.list_ld;
        const int cnt = p.counts[(size_t)head * p.pairs + pr];
        const int nkv = kv_tiles(cnt);
        auto load_kv = [&](const uint8_t *m, int j) -> bool {
            const uint32_t s = loads % kStages, ph = (loads / kStages) & 1u;
            if (!wait_bar(sm, kBarKvEmpty + (int)s, ph ^ 1u, p, kWhereKvEmpty)) return false;
            const int e0 = 2 * j < cnt ? lst[2 * j] : 0xFFFF, e1 = 2 * j + 1 < cnt ? lst[2 * j + 1] : 0xFFFF;
            // debug build: every entry names a tile of the grid or no tile (0xFFFF)
            dev_check(((e0 & 0xFFFF) < p.g.num_tiles || (e0 & 0xFFFF) == 0xFFFF) &&
                          ((e1 & 0xFFFF) < p.g.num_tiles || (e1 & 0xFFFF) == 0xFFFF) && cnt <= p.list_ld,
                      p.status, 0x12);
            const uint32_t full = sm.b(kBarKvFull + (int)(loads % kKvFullBars));
            if ((int64_t)loads != skipped) {
                ptx::mbar_arrive_expect_tx(full, kTileBytes);
                const uint32_t dst = sm.kv + s * (uint32_t)kTileBytes;
                load_kv_tile(m, p, dst, 0, head, e0 & 0xFFFF, full);
                load_kv_tile(m, p, dst, 1, head, e1 & 0xFFFF, full);
            }
            ++loads;
            return true;
        };
        ok = load_kv(p.kp, 0);
        if (ok) ok = load_kv(p.kp, 1);
        for (int j = 0; ok && j < nkv; ++j) {
            ok = load_kv(p.vp, j);
            if (ok && j + 2 < nkv) ok = load_kv(p.kp, j + 2);
        }
    }
    // the last kKvFullBars loads each hold their own full barrier
    for (uint32_t l = loads > (uint32_t)kKvFullBars ? loads - kKvFullBars : 0u; l < loads; ++l)
        if ((int64_t)l != skipped) drain_bar(sm, kBarKvFull + (int)(l % kKvFullBars), (l / kKvFullBars) & 1u, p);
    for (uint32_t i = 0; i < (uint32_t)kQSlots && i < q_loads; ++i) {
        const uint32_t last = q_loads - 1u - i;
        drain_bar(sm, kBarQFull + (int)(last % kQSlots), (last / kQSlots) & 1u, p);
    }
}

constexpr uint64_t kDescTile = (uint64_t)(kTileBytes >> 4);

// S = Q K^T: Q in the TMA layout (channel halves 16 KB apart, 8-row groups
// 1 KB apart), K in the tile-major layout (halves 1 KB apart, groups 2 KB).
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc) {
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, 128, false, false);
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
        const uint64_t qoff = (uint64_t)(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
        const uint64_t koff = (uint64_t)(((kk >> 2) * 1024 + (kk & 3) * 32) >> 4);
        ptx::mma_ss(d_tmem, q_desc + qoff, k_desc + koff, idesc, kk > 0 ? 1u : 0u);
    }
}

// O += P V: V MN-major in the tile-major layout, 16 keys = two 2 KB groups.
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t v_desc, bool accumulate) {
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, 128, false, true);
#pragma unroll
    for (int kk = 0; kk < kRows / 16; ++kk) {
        const uint64_t off = (uint64_t)((kk * 2 * kGroupBytes) >> 4);
        ptx::mma_ts(d_tmem, p_tmem + (uint32_t)(kk * 8), v_desc + off, idesc, (accumulate || kk > 0) ? 1u : 0u);
    }
}

// Issuer of softmax group g's tensor work: S_g = Q K_j^T and O_g += P_g V_j
// for the unit's K/V tiles j = g, g + 2, ...  Two threads (one per group, in
// different warps) feed the tensor core, so one's waits and commits overlap
// the other's MMAs.  Each finds its tiles' K/V ring slots from the
// producer's fixed load order: K_0, K_1, then V_j, K_{j+2} for j = 0, 1, ...
// A thread waits on load L only after its own previous load L' >= L - 4
// completed (every unit has >= 2 K/V tiles, so each thread's loads are at
// most 3 apart); L' was issued after every load <= L' - 4 had been consumed,
// so load L - 8, the previous user of L's full barrier, is complete and the
// parity wait cannot match a stale phase.
__device__ void mma_issuer(const Params &p, const Smem &sm, uint32_t tmem, int g) {
    const uint64_t q0 = ptx::sdesc_sw128(sm.q, 16, 1024);
    const uint64_t kv0 = ptx::sdesc_sw128(sm.kv, 16, kGroupBytes);
    const uint64_t v0 = ptx::sdesc_sw128(sm.kv, 1024, kGroupBytes);
    const uint32_t t_s = tmem + 128u * (uint32_t)g, t_o = tmem + 256u + 128u * (uint32_t)g;
    uint32_t base = 0, uu = 0, ptile = 0;  // loads of the CTA's earlier units, units, P tiles seen
    bool ok = true;
    // wait for ring load `ld` (unit-relative) and return its slot
    auto kv_ready = [&](uint32_t ld, uint32_t &slot) -> bool {
        const uint32_t L = base + ld;
        slot = L % kStages;
        const bool r = wait_bar(sm, kBarKvFull + (int)(L % kKvFullBars), (L / kKvFullBars) & 1u, p, kWhereKvFull);
        if (r) ptx::tc_fence_after();
        return r;
    };
    for (int unit = blockIdx.x; ok && unit < p.num_units; unit += gridDim.x, ++uu) {
        const int head = unit / p.pairs, pr = unit % p.pairs;
        const uint32_t qs = uu % kQSlots;
        ok = wait_bar(sm, kBarQFull + (int)qs, (uu / kQSlots) & 1u, p, kWhereQFull);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint64_t qd = q0 + qs * kDescTile;
        const int nkv = kv_tiles(p.counts[(size_t)head * p.pairs + pr]);
        const int m = nkv - 2;  // K_{j+2} is loaded for j < m
        uint32_t s;
        ok = kv_ready((uint32_t)g, s);  // K_g
        if (!ok) break;
        issue_qk(t_s, qd, kv0 + s * kDescTile);
        ptx::tc_commit(sm.b(kBarSFull + g));
        ptx::tc_commit(sm.b(kBarKvEmpty + (int)s));
        // both groups must have read O_0 and O_1 of the previous unit
        if (uu > 0) {
            ok = wait_bar(sm, kBarMerged, (uu - 1u) & 1u, p, kWhereMerged);
            if (!ok) break;
            ptx::tc_fence_after();
        }
        for (int j = g; ok && j < nkv; j += 2) {
            const uint32_t lv = (uint32_t)(2 + j + (j < m ? j : m));  // V_j; K_{j+2} follows it
            ok = kv_ready(lv, s);
            if (!ok) break;
            ok = wait_bar(sm, kBarPFull + g, ptile & 1u, p, kWherePFull);
            if (!ok) break;
            ++ptile;
            ptx::tc_fence_after();
            issue_pv(t_o, t_s, v0 + s * kDescTile, j >= 2);
            ptx::tc_commit(sm.b(kBarKvEmpty + (int)s));
            if (j + 2 >= nkv) ptx::tc_commit(sm.b(kBarOFull + g));
            if (j + 2 < nkv) {
                ok = kv_ready(lv + 1u, s);
                if (!ok) break;
                issue_qk(t_s, qd, kv0 + s * kDescTile);
                ptx::tc_commit(sm.b(kBarSFull + g));
                ptx::tc_commit(sm.b(kBarKvEmpty + (int)s));
            }
        }
        if (!ok) break;
        ptx::tc_commit(sm.b(kBarQEmpty + (int)qs));
        base += 2u * (uint32_t)nkv;
    }
    ptx::tc_commit(sm.b(kBarDrain + g));
    drain_bar(sm, kBarDrain + g, 0u, p);
}

// -------------------------------------------------------------- softmax
__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// One 64-key half of a K/V tile: s[c][i] is the score of key 32 c + i of the
// half, visible to the warp when bit i of w[c] is set.  kMasked tests single
// keys (only tiles on the grid's edge, with missing tokens, need it).
template <bool kMasked>
__device__ __forceinline__ float half_max(const uint32_t (&s)[2][32], const uint32_t (&w)[2]) {
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        if (!kMasked) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                m0 = ptx::max3(m0, u2f(s[c][i]), u2f(s[c][i + 1]));
                m1 = ptx::max3(m1, u2f(s[c][i + 2]), u2f(s[c][i + 3]));
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if ((w[c] >> i) & 1u) m0 = fmaxf(m0, u2f(s[c][i]));
        }
    }
    return fmaxf(m0, m1);
}

// p = 2^(s * scale_log2 - m) for the half's 64 keys, as 32 packed bf16 pairs
// at TMEM address t_p; returns the float32 sum of p.
template <bool kMasked>
__device__ __forceinline__ float half_probs(const uint32_t (&s)[2][32], const uint32_t (&w)[2], float scale_log2,
                                            float m, uint32_t t_p) {
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
            float x0, x1, x2, x3;
            ptx::fma2(x0, x1, u2f(s[c][i]), u2f(s[c][i + 1]), scale_log2, -m);
            ptx::fma2(x2, x3, u2f(s[c][i + 2]), u2f(s[c][i + 3]), scale_log2, -m);
            float p0 = ptx::ex2_approx(x0), p1 = ptx::ex2_approx(x1);
            float p2 = ptx::ex2_approx(x2), p3 = ptx::ex2_approx(x3);
            if (kMasked) {
                p0 = ((w[c] >> i) & 1u) ? p0 : 0.f;
                p1 = ((w[c] >> (i + 1)) & 1u) ? p1 : 0.f;
                p2 = ((w[c] >> (i + 2)) & 1u) ? p2 : 0.f;
                p3 = ((w[c] >> (i + 3)) & 1u) ? p3 : 0.f;
            }
            ptx::add2(a0, a1, p0, p1);
            ptx::add2(b0, b1, p2, p3);
            pk[i / 2] = pack_bf16x2(p0, p1);
            pk[i / 2 + 1] = pack_bf16x2(p2, p3);
        }
        ptx::tmem_st_32x32b_x16(t_p + (uint32_t)(c * 16), pk);
    }
    return (a0 + a1) + (b0 + b1);
}

__device__ __forceinline__ void zero_half(uint32_t t_p) {
    uint32_t zero[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) zero[i] = 0u;
    ptx::tmem_st_32x32b_x16(t_p, zero);
    ptx::tmem_st_32x32b_x16(t_p + 16u, zero);
}

// Softmax warpgroup k (0 or 1); thread t owns row t of the Q tile.
__device__ void softmax_role(const Params &p, const Smem &sm, uint32_t tmem, int k, int t) {
    const uint32_t lane_base = (uint32_t)((t >> 5) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + 128u * (uint32_t)k;
    const uint32_t t_ok = tmem + lane_base + 256u + 128u * (uint32_t)k;
    const int qhalf = t >> 6;   // which query tile of the pair this row belongs to
    uint32_t seen = 0, uu = 0;
    bool ok = true;
    for (int unit = blockIdx.x; ok && unit < p.num_units; unit += gridDim.x, ++uu) {
        const int head = unit / p.pairs, pr = unit % p.pairs;
        const int32_t *lst = p.lists + ((size_t)head * p.pairs + pr) * p.list_ld;
        const int cnt = p.counts[(size_t)head * p.pairs + pr];
        const int nkv = kv_tiles(cnt);
        MaskWindow win;
        win.init(lst, cnt, t & 31, qhalf, &p.g);
        float m_used = -INFINITY, l = 0.f;
        for (int j = k; j < nkv; j += 2) {
            uint32_t mk[4];
            win.tile(j, mk);
            ok = __all_sync(0xffffffffu, wait_bar(sm, kBarSFull + k, seen & 1u, p, kWhereSFull));
            if (!ok) break;
            ++seen;
            ptx::tc_fence_after();
            // The two 64-key halves one after the other, each with only its own
            // scores in registers.  P (bf16 pairs) of half h goes to columns
            // [32 h, 32 h + 32) of S: half 1's P overwrites scores of half 0,
            // which by then are consumed; half 1's scores (columns 64-127) are
            // never overwritten.
            float factor = 1.f;  // rescale of O accumulated before this tile
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t w[2] = {mk[2 * h], mk[2 * h + 1]};
                const uint32_t t_p = t_s + 32u * (uint32_t)h;
                if ((w[0] | w[1]) == 0u) {
                    zero_half(t_p);
                    continue;
                }
                uint32_t sc[2][32];
                ptx::tmem_ld_32x32b_x32(t_s + 64u * (uint32_t)h, sc[0]);
                ptx::tmem_ld_32x32b_x32(t_s + 64u * (uint32_t)h + 32u, sc[1]);
                ptx::tmem_ld_wait();
                ptx::reg_fence(sc[0]);
                ptx::reg_fence(sc[1]);
                const bool full = (w[0] & w[1]) == 0xFFFFFFFFu;
                // The row's first visible half sets the reference maximum m_used;
                // later halves exponentiate against it directly and only a half
                // whose probabilities sum above 2^20 takes its own maximum and is
                // exponentiated again (the softmax does not depend on the
                // reference point; every p stays <= 2^20).
                float sum = 0.f;
                bool need_max = __any_sync(0xffffffffu, m_used == -INFINITY);
                if (!need_max) {
                    sum = full ? half_probs<false>(sc, w, p.scale_log2, m_used, t_p)
                               : half_probs<true>(sc, w, p.scale_log2, m_used, t_p);
                    need_max = __any_sync(0xffffffffu, !(sum <= kRedoSum));
                    if (need_max) ptx::tmem_st_wait();  // stored before it is overwritten
                }
                if (!need_max) {
                    l += sum;
                    continue;
                }
                const float mh = (full ? half_max<false>(sc, w) : half_max<true>(sc, w)) * p.scale_log2;
                float f = 1.f;
                if (mh > m_used) {
                    if (m_used != -INFINITY) f = ptx::ex2_approx(m_used - mh);
                    m_used = mh;
                }
                l *= f;
                factor *= f;
                // half 1 raised the maximum: half 0's P, already written with
                // the old one, takes the same factor (rare; warp-collective)
                if (h == 1 && (mk[0] | mk[1]) != 0u && __any_sync(0xffffffffu, f != 1.f)) {
                    uint32_t pp[32];
                    ptx::tmem_st_wait();
                    ptx::tmem_ld_32x32b_x32(t_s, pp);
                    ptx::tmem_ld_wait();
                    ptx::reg_fence(pp);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&pp[i]);
                        const float2 fv = __bfloat1622float2(v);
                        pp[i] = pack_bf16x2(fv.x * f, fv.y * f);
                    }
                    ptx::tmem_st_32x32b_x32(t_s, pp);
                }
                l += full ? half_probs<false>(sc, w, p.scale_log2, m_used, t_p)
                          : half_probs<true>(sc, w, p.scale_log2, m_used, t_p);
            }
            // O holds nothing of this unit before the group's first tile (and the
            // other group may still be reading the previous unit's O there)
            if (j != k && __any_sync(0xffffffffu, factor != 1.f)) {
#pragma unroll 1
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t o[32];
                    ptx::tmem_ld_32x32b_x32(t_ok + (uint32_t)(32 * c4), o);
                    ptx::tmem_ld_wait();
                    ptx::reg_fence(o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * factor);
                    ptx::tmem_st_32x32b_x32(t_ok + (uint32_t)(32 * c4), o);
                }
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(sm.b(kBarPFull + k));
        }
        if (!ok) break;
        ok = __all_sync(0xffffffffu, wait_bar(sm, kBarOFull + k, uu & 1u, p, kWhereOFull));
        if (!ok) break;
        ptx::tc_fence_after();
        // exchange the running max and sum with the other group
        float *ml = sm.ml + (uu & 1u) * 4 * kRows;
        ml[k * 2 * kRows + t] = m_used;
        ml[k * 2 * kRows + kRows + t] = l;
        ptx::mbar_arrive(sm.b(kBarMlReady));
        ok = __all_sync(0xffffffffu, wait_bar(sm, kBarMlReady, uu & 1u, p, kWhereMl));
        if (!ok) break;
        const float m0 = ml[t], l0 = ml[kRows + t];
        const float m1 = ml[2 * kRows + t], l1 = ml[3 * kRows + t];
        const float mx = fmaxf(m0, m1);
        const float a0 = l0 > 0.f ? ptx::ex2_approx(m0 - mx) : 0.f;
        const float a1 = l1 > 0.f ? ptx::ex2_approx(m1 - mx) : 0.f;
        const float sum = a0 * l0 + a1 * l1;
        const float inv = 1.0f / sum;
        // the row's token
        const int tile = 2 * pr + qhalf, r = t & 63;
        bool row_ok = tile < p.g.num_tiles;
        int64_t tok = 0;
        if (row_ok) {
            const TileCoord c = tile_coord(p.g, tile);
            const int tt = c.t0 + (r >> 4), hh = c.h0 + ((r >> 2) & 3), ww = c.w0 + (r & 3);
            row_ok = tt < p.g.frames && hh < p.g.height && ww < p.g.width;
            tok = ((int64_t)tt * p.g.height + hh) * p.g.width + ww;
        }
        uint4 *dst = reinterpret_cast<uint4 *>(p.o + (size_t)tok * (size_t)p.ld + (size_t)head * kD + 64 * k);
        const uint32_t t_o0 = tmem + lane_base + 256u + 64u * (uint32_t)k;
#pragma unroll 1
        for (int c2 = 0; c2 < 2; ++c2) {
            uint32_t x0[32], x1[32];
            ptx::tmem_ld_32x32b_x32(t_o0 + (uint32_t)(32 * c2), x0);
            ptx::tmem_ld_32x32b_x32(t_o0 + 128u + (uint32_t)(32 * c2), x1);
            ptx::tmem_ld_wait();
            ptx::reg_fence(x0);
            ptx::reg_fence(x1);
            if (row_ok) {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float y0 = l0 > 0.f ? a0 * u2f(x0[8 * v + e]) : 0.f;
                        const float y1 = l1 > 0.f ? a1 * u2f(x1[8 * v + e]) : 0.f;
                        f[e] = (y0 + y1) * inv;
                    }
                    uint4 w;
                    w.x = pack_bf16x2(f[0], f[1]);
                    w.y = pack_bf16x2(f[2], f[3]);
                    w.z = pack_bf16x2(f[4], f[5]);
                    w.w = pack_bf16x2(f[6], f[7]);
                    dst[c2 * 4 + v] = w;
                }
            }
        }
        if (k == 0 && row_ok && p.lse != nullptr)
            p.lse[(size_t)head * (size_t)p.n + (size_t)tok] = (mx + log2f(sum)) * 0.69314718055994531f;
        ptx::tc_fence_before();
        ptx::mbar_arrive(sm.b(kBarMerged));
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    vsa_fine_kernel(const __grid_constant__ CUtensorMap tm_q, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    Smem sm;
    sm.q = base + kSmemQ;
    sm.kv = base + kSmemKV;
    sm.bar = base + kSmemBar;
    sm.ml = reinterpret_cast<float *>(smem + kSmemMl);
    sm.abort_flag = reinterpret_cast<volatile int *>(smem + kSmemMisc + 4);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + kSmemMisc);
    const int warp = (int)(threadIdx.x >> 5), lane = (int)(threadIdx.x & 31);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kKvFullBars; ++s) ptx::mbar_init(sm.b(kBarKvFull + s), 1);
        for (int s = 0; s < kStages; ++s) ptx::mbar_init(sm.b(kBarKvEmpty + s), 1);
        for (int k = 0; k < kQSlots; ++k) {
            ptx::mbar_init(sm.b(kBarQFull + k), 1);
            ptx::mbar_init(sm.b(kBarQEmpty + k), 2);
        }
        for (int k = 0; k < 2; ++k) {
            ptx::mbar_init(sm.b(kBarSFull + k), 1);
            ptx::mbar_init(sm.b(kBarPFull + k), 128);
            ptx::mbar_init(sm.b(kBarOFull + k), 1);
        }
        ptx::mbar_init(sm.b(kBarMlReady), 256);
        ptx::mbar_init(sm.b(kBarMerged), 256);
        ptx::mbar_init(sm.b(kBarDrain), 1);
        ptx::mbar_init(sm.b(kBarDrain + 1), 1);
        *sm.abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == kTmaWarp && lane == 0) {
        ptx::prefetch_tensormap(&tm_q);
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_holder), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(tmem_holder);
    if (warp == kTmaWarp) {
        producer(&tm_q, p, sm, lane);
    } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
        if (lane == 0) mma_issuer(p, sm, tmem, warp - kMmaWarp);
    } else {
        softmax_role(p, sm, tmem, warp >> 2, (int)threadIdx.x & 127);
    }
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// [frames, height, width, heads * 128] bf16 viewed as a 4D tensor; boxes of
// one tile x 64 channels, 128-byte swizzle, zero fill outside the grid.
bool make_grid_map(CUtensorMap *m, const void *ptr, const Geo &g, int ld) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t row = (cuuint64_t)ld * 2u;
    const cuuint64_t dims[4] = {(cuuint64_t)ld, (cuuint64_t)g.width, (cuuint64_t)g.height, (cuuint64_t)g.frames};
    const cuuint64_t strides[3] = {row, row * (cuuint64_t)g.width, row * (cuuint64_t)g.width * (cuuint64_t)g.height};
    const cuuint32_t box[4] = {64u, 4u, 4u, 4u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

Geo make_geo(int frames, int height, int width) {
    Geo g;
    g.frames = frames;
    g.height = height;
    g.width = width;
    g.tiles_h = (height + 3) / 4;
    g.tiles_w = (width + 3) / 4;
    g.num_tiles = ((frames + 3) / 4) * g.tiles_h * g.tiles_w;
    return g;
}

size_t align256(size_t x) { return (x + 255u) & ~(size_t)255u; }

struct WsLayout {
    size_t qbar, kbar, lists, counts, kp, vp, zero, total;
};

WsLayout ws_layout(int heads, const Geo &g, int topk) {
    const int pairs = (g.num_tiles + 1) / 2;
    WsLayout w;
    const size_t means = align256((size_t)heads * g.num_tiles * kD * sizeof(float));
    w.qbar = 0;
    w.kbar = means;
    w.lists = 2 * means;
    w.counts = w.lists + align256((size_t)heads * pairs * 2 * topk * sizeof(int32_t));
    w.kp = w.counts + align256((size_t)heads * pairs * sizeof(int32_t));
    const size_t copy = align256((size_t)heads * g.num_tiles * kKeptBytes);
    w.vp = w.kp + copy;
    w.zero = w.vp + copy;
    w.total = w.zero + kKeptBytes;
    return w;
}

}  // namespace

int vsa_num_tiles(int frames, int height, int width) {
    if (frames < 1 || height < 1 || width < 1) return 0;
    const int64_t n = (int64_t)((frames + 3) / 4) * ((height + 3) / 4) * ((width + 3) / 4);
    return n > kMaxTiles ? -1 : (int)n;
}

int64_t vsa_workspace_bytes(int heads, int frames, int height, int width, int topk) {
    return (int64_t)ws_layout(heads, make_geo(frames, height, width), topk).total;
}

fv_status launch_vsa_attn(const VsaLaunch &a, cudaStream_t stream) {
    static std::mutex mu;
    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FV_ERR_LAUNCH;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!attr_set[dev]) {
            if (cudaFuncSetAttribute(vsa_fine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
                    cudaSuccess ||
                cudaFuncSetAttribute(vsa_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSelSmemBytes) != cudaSuccess)
                return FV_ERR_LAUNCH;
            attr_set[dev] = true;
        }
    }
    const Geo g = make_geo(a.frames, a.height, a.width);
    const int ld = a.heads * kD;
    const int pairs = (g.num_tiles + 1) / 2;
    const WsLayout w = ws_layout(a.heads, g, a.topk);
    uint8_t *ws = static_cast<uint8_t *>(a.workspace);
    float *qbar = reinterpret_cast<float *>(ws + w.qbar);
    float *kbar = reinterpret_cast<float *>(ws + w.kbar);
    int32_t *lists = reinterpret_cast<int32_t *>(ws + w.lists);
    int32_t *counts = reinterpret_cast<int32_t *>(ws + w.counts);
    CUtensorMap mq;
    if (!make_grid_map(&mq, a.q, g, ld)) return FV_ERR_LAUNCH;
    const auto *q = static_cast<const __nv_bfloat16 *>(a.q);
    const auto *k = static_cast<const __nv_bfloat16 *>(a.k);
    const auto *v = static_cast<const __nv_bfloat16 *>(a.v);
    if (cudaMemsetAsync(ws + w.zero, 0, kKeptBytes, stream) != cudaSuccess) return FV_ERR_LAUNCH;
    vsa_pool_kernel<<<g.num_tiles, 256, 0, stream>>>(q, k, v, g, a.heads, qbar, kbar,
                                                     reinterpret_cast<__nv_bfloat16 *>(ws + w.kp),
                                                     reinterpret_cast<__nv_bfloat16 *>(ws + w.vp));
    const int ppc = select_pairs_per_cta(g.num_tiles);
    const size_t sel_smem = ((size_t)kSelMaxRows * kD + (size_t)2 * ppc * g.num_tiles) * 4;
    vsa_select_kernel<<<dim3((pairs + ppc - 1) / ppc, a.heads), 256, sel_smem, stream>>>(
        qbar, kbar, g, pairs, ppc, a.topk, a.selected, lists, counts);
    Params p;
    p.o = static_cast<__nv_bfloat16 *>(a.o);
    p.lse = a.lse;
    p.status = a.status;
    p.lists = lists;
    p.counts = counts;
    p.kp = ws + w.kp;
    p.vp = ws + w.vp;
    p.zero = ws + w.zero;
    p.g = g;
    p.n = (int)a.n;
    p.ld = ld;
    p.pairs = pairs;
    p.num_units = a.heads * pairs;
    p.list_ld = 2 * a.topk;
    p.scale_log2 = (float)((double)a.scale * 1.4426950408889634);
    p.skip_load = take_test_skip_load(FV_TEST_VSA_FINE);
    const int grid = p.num_units < a.num_sms ? p.num_units : a.num_sms;
    vsa_fine_kernel<<<grid, kThreads, kSmemBytes, stream>>>(mq, p);
    return cudaGetLastError() == cudaSuccess ? FV_OK : FV_ERR_LAUNCH;
}

}  // namespace fv
