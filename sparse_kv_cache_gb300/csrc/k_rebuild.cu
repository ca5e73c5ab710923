// Sparse key reconstruction: K~ = RoPE(Gather(A, chunks) . B_h).
//
// ShadowKV (English summary, section 3.4, "Sparse KV Reconstruction and
// Overlapping Strategy": K_sparse = MatMul(Gather(A, I_miss), B), then RoPE at
// the tokens' own positions; Chinese digest section A2, Algorithm 2).  The
// same kernels serve Algorithm 1's pre-filling in "statistics" mode: instead
// of storing the keys they emit each chunk's mean (the landmark, summary
// section 3.4 "Landmark Construction") and the minimum cosine between a token
// key and that mean (Algorithm 1: CosineSimilarity, Min).
//
// A tile is 16 chunks = 128 token rows of one (batch, KV head) unit.
//  * bf16: a tcgen05 tile.  Once the tile is known to have work, one thread
//    issues the unit's B slice (stored transposed, [d][r], K-major) while the
//    chunk list is read, then sixteen threads issue the chunks' A rows (8 rows
//    each, from anywhere in A); all are 2-D TMA copies in 64-column (128-byte,
//    swizzled) blocks, and zero fill covers columns past r.  One elected
//    thread issues M=128, N=128, K=16 bf16 MMAs with an fp32 accumulator in
//    tensor memory; the four warps read their 32 rows back with tcgen05.ld.
//  * fp32: CUDA-core FMAs, one thread per row, B broadcast from shared memory
//    (tf32 tensor cores would not meet fp32 accuracy).
// Epilogue (both): the fp32 tile is staged in shared memory (the operand
// buffers, free once the MMAs retire), then RoPE runs one warp per row with
// angles composed from two tables, cos/sin(pos*theta) from the (pos & 255)
// and (pos >> 8)*256 entries built on the host in double precision, so every
// table read and key store is contiguous across the warp; then either the
// bf16/fp32 key rows go to their destination slot, or the statistics are
// formed in fp32.
//
// Also here: pre-filling from exact keys (the rows come from the caller's keys
// instead of A.B) and ShadowKV+'s projection of a generated token's key onto
// the rank-r basis.
#include <math_constants.h>

#include "skv_common.cuh"
#include "skv_internal.h"

namespace skv {

constexpr int kRows = kTileChunks * kC;   // 128
constexpr int kStagePitch = kD + 4;       // fp32 staging row pitch (floats)

struct TileInfo {
    int chunk;   // original chunk id, -1 if the row is not valid
    int dst;     // destination chunk slot
};

// Stage one row half (dims [32h, 32h+32) and [64+32h, +32)) of raw fp32 keys.
__device__ __forceinline__ void stage_half(float* stage, int row, int h, const float (&v0)[32], const float (&v1)[32]) {
    float* srow = stage + row * kStagePitch;
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
        *reinterpret_cast<float4*>(srow + 32 * h + i) = make_float4(v0[i], v0[i + 1], v0[i + 2], v0[i + 3]);
        *reinterpret_cast<float4*>(srow + kD / 2 + 32 * h + i) = make_float4(v1[i], v1[i + 1], v1[i + 2], v1[i + 3]);
    }
}

// RoPE over the staged tile.  Warp w owns chunks w, w+4, w+8, w+12; for a
// chunk it holds the (cos, sin) table entries of all 8 rows (one `hi` entry,
// shared by the chunk since 8-aligned chunks never straddle a 256 boundary,
// and 8 `lo` entries), fetched ahead with all loads in flight.  Lane l
// rotates the pairs (2l, 2l+64) and (2l+1, 2l+65), so table reads,
// shared-memory reads and the row stores are contiguous across the warp.  The
// angle of position pos is composed from the (pos & 255) and (pos >> 8)
// tables by the addition formulas.  Mode 0 stores the rotated rows into their
// slot; mode 1 writes them back into the staging tile for the statistics.
struct RopeRegs {
    float4 lo[kC];
    float4 hi;
};

__device__ __forceinline__ void rope_fetch(const RebuildParams& p, const TileInfo& t, RopeRegs& r) {
    const int lane = threadIdx.x & 31;
    if (t.chunk < 0) return;
    const int pos0 = t.chunk * kC;
    r.hi = reinterpret_cast<const float4*>(p.rope_hi + (pos0 >> 8) * (kD / 2))[lane];
#pragma unroll
    for (int i = 0; i < kC; ++i) r.lo[i] = reinterpret_cast<const float4*>(p.rope_lo + ((pos0 + i) & 255) * (kD / 2))[lane];
}

template <typename OutT>
__device__ __forceinline__ void rope_chunk(const RebuildParams& p, int u, int c, const TileInfo& t, const RopeRegs& r,
                                           float* stage) {
    const int lane = threadIdx.x & 31;
    if (t.chunk < 0) return;
#pragma unroll
    for (int i = 0; i < kC; ++i) {
        const int row = c * kC + i;
        const float4 lo = r.lo[i], hi = r.hi;
        const float c0 = hi.x * lo.x - hi.y * lo.y, s0 = hi.y * lo.x + hi.x * lo.y;
        const float c1 = hi.z * lo.z - hi.w * lo.w, s1 = hi.w * lo.z + hi.z * lo.w;
        float* srow = stage + row * kStagePitch;
        const float2 a = *reinterpret_cast<const float2*>(srow + 2 * lane);
        const float2 b = *reinterpret_cast<const float2*>(srow + kD / 2 + 2 * lane);
        const float2 ra = make_float2(a.x * c0 - b.x * s0, a.y * c1 - b.y * s1);
        const float2 rb = make_float2(a.x * s0 + b.x * c0, a.y * s1 + b.y * c1);
        if (p.mode == 0) {
            OutT* dst = static_cast<OutT*>(p.dst) + u * p.dst_us + (static_cast<int64_t>(t.dst) * kC + i) * kD;
            if constexpr (sizeof(OutT) == 2) {
                reinterpret_cast<uint32_t*>(dst)[lane] = pack_bf16x2(ra.x, ra.y);
                reinterpret_cast<uint32_t*>(dst + kD / 2)[lane] = pack_bf16x2(rb.x, rb.y);
            } else {
                reinterpret_cast<float2*>(dst)[lane] = ra;
                reinterpret_cast<float2*>(dst + kD / 2)[lane] = rb;
            }
        } else {
            *reinterpret_cast<float2*>(srow + 2 * lane) = ra;
            *reinterpret_cast<float2*>(srow + kD / 2 + 2 * lane) = rb;
        }
    }
}

// All chunks of the tile; `first` holds the prefetched entries of the warp's first chunk.
template <typename OutT>
__device__ void rope_tile(const RebuildParams& p, int u, const TileInfo* ti, float* stage, const RopeRegs& first) {
    const int warp = threadIdx.x >> 5;
    // the next chunk's table entries are in flight while the current chunk rotates
    RopeRegs cur = first;
    for (int c = warp; c < kTileChunks; c += 4) {
        RopeRegs nxt;
        if (c + 4 < kTileChunks) rope_fetch(p, ti[c + 4], nxt);
        rope_chunk<OutT>(p, u, c, ti[c], cur, stage);
        cur = nxt;
    }
}

// Landmarks and min-cos of the tile's chunks from the fp32 staging tile
// (needs all 128 threads; `smean` holds 16 x d floats).
__device__ void tile_stats(const RebuildParams& p, int u, const TileInfo* ti, const float* stage, float* smean) {
    const int tid = threadIdx.x;
    {
        const int c = tid >> 3, d0 = (tid & 7) * 16;
        const float* base = stage + c * kC * kStagePitch;
        float acc[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) acc[k] = 0.f;
#pragma unroll
        for (int t = 0; t < kC; ++t)
#pragma unroll
            for (int k = 0; k < 16; ++k) acc[k] += base[t * kStagePitch + d0 + k];
        float* lf = ti[c].chunk >= 0 ? p.Lfull + (u * p.stats_us + ti[c].chunk) * kD + d0 : nullptr;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float mval = acc[k] * (1.0f / kC);
            smean[c * kD + d0 + k] = mval;
            if (lf) lf[k] = mval;
        }
    }
    __syncthreads();
    const int row = tid, c = row >> 3;
    const float* x = stage + row * kStagePitch;
    const float* m = smean + c * kD;
    float dot = 0.f, nx = 0.f, nm = 0.f;
#pragma unroll 8
    for (int k = 0; k < kD; ++k) {
        const float a = x[k], b = m[k];
        dot = fmaf(a, b, dot);
        nx = fmaf(a, a, nx);
        nm = fmaf(b, b, nm);
    }
    float cosv = dot / fmaxf(sqrtf(nx) * sqrtf(nm), 1e-12f);
#pragma unroll
    for (int o = 1; o < kC; o <<= 1) cosv = fminf(cosv, __shfl_xor_sync(0xffffffffu, cosv, o));
    if ((row & 7) == 0 && ti[c].chunk >= 0) p.mcos[u * p.stats_us + ti[c].chunk] = cosv;
}

// Resolve the tile's chunk ids and destination slots; returns the number of
// chunks in this tile, or 0 if the CTA has nothing to do.
__device__ int load_tile_info(const RebuildParams& p, int u, int tile, TileInfo* ti) {
    int count = p.cnt ? p.cnt[u] : p.count_const;
    if (count < 0 || count > p.list_cap) {
        if (threadIdx.x == 0) set_err(p.err, DEV_ERR_BOUNDS, 401);
        count = 0;
    }
    const int first = tile * kTileChunks;
    if (first >= count) return 0;
    const int nch = min(kTileChunks, count - first);
    if (threadIdx.x < kTileChunks) {
        const int c = threadIdx.x;
        TileInfo t{-1, 0};
        if (c < nch) {
            const int idx = first + c;
            const int ch = p.list ? p.list[u * p.list_us + idx] : p.list_base + idx;
            const int dst = p.dst_idx ? p.dst_idx[u * p.list_us + idx] : idx;
            if (ch < 0 || ch >= p.nchunk || (p.mode == 0 && (dst < 0 || dst >= p.dst_cap)) ||
                (p.mode == 1 && ch >= p.stats_us)) {
                set_err(p.err, DEV_ERR_BOUNDS, 402);
            } else {
                t.chunk = ch;
                t.dst = dst;
            }
        }
        ti[c] = t;
    }
    return nch;
}

// ------------------------------------------------------------------ tcgen05 path
template <typename OutT>
__global__ void __launch_bounds__(128, 1) k_rebuild_tc(const __grid_constant__ CUtensorMap tmA,
                                                        const __grid_constant__ CUtensorMap tmB, RebuildParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar_tma, bar_mma;
    __shared__ uint32_t tmem_slot;
    __shared__ TileInfo ti[kTileChunks];
    __shared__ int s_fail;

    // units along x, tiles along y: the first tiles of every unit are dispatched before any
    // unit's later (often empty) ones
    const int u = blockIdx.x, tile = blockIdx.y, tid = threadIdx.x, warp = tid >> 5;
    // launched as a programmatic dependent of the selection: the list is its output
    pdl_wait();
    // the attention that follows (values in HBM) may be scheduled as this grid's CTAs finish; it
    // waits for the whole grid before it reads a key
    pdl_trigger();
    // the list entries are read in the same round trip as the count (in bounds up to list_cap)
    int ch_raw = 0, dst_raw = 0;
    const int first_idx = tile * kTileChunks;
    if (tid < kTileChunks && first_idx + tid < p.list_cap) {
        const int idx = first_idx + tid;
        ch_raw = p.list ? p.list[u * p.list_us + idx] : p.list_base + idx;
        dst_raw = p.dst_idx ? p.dst_idx[u * p.list_us + idx] : idx;
    }
    int count = p.cnt ? p.cnt[u] : p.count_const;
    if (count < 0 || count > p.list_cap) {
        if (tid == 0) set_err(p.err, DEV_ERR_BOUNDS, 401);
        count = 0;
    }
    if (first_idx >= count) return;   // uniform
    const int nch = min(kTileChunks, count - first_idx);
    const int nkb = p.nkb;
    uint8_t* sA = smem;                      // nkb x [128 rows][128 B]
    uint8_t* sB = smem + nkb * 16384;        // nkb x [128 rows][128 B]
    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        s_fail = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        // the unit's B slice does not depend on the chunk list: in flight while the list is read
        mbar_expect_tx(&bar_tma, static_cast<uint32_t>(nkb * 16384));
        for (int kb = 0; kb < nkb; ++kb) tma_load_2d(sB + kb * 16384, &tmB, kb * 64, u * kD, &bar_tma);
    }
    if (tid < kTileChunks) {
        TileInfo t{-1, 0};
        if (tid < nch) {
            const int ch = ch_raw, dst = dst_raw;
            if (ch < 0 || ch >= p.nchunk || (p.mode == 0 && (dst < 0 || dst >= p.dst_cap)) ||
                (p.mode == 1 && ch >= p.stats_us)) {
                set_err(p.err, DEV_ERR_BOUNDS, 402);
            } else {
                t.chunk = ch;
                t.dst = dst;
            }
        }
        ti[tid] = t;
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const int b = u / p.H;

    // A rows: the tile's nch x nkb boxes (8 rows x 64 columns of one chunk) spread over lanes
    // 0-15 of the four warps, one box per thread at a time: the copy instructions of different
    // warps issue side by side (measured: 21.1 against 22.7 us per layer at 128K b8 for one
    // thread per chunk issuing its nkb boxes)
    if ((tid & 31) < 16)
        for (int o = warp * 16 + (tid & 31); o < nch * nkb; o += 64) {
            const int c = o / nkb, kb = o - c * nkb;
            if (ti[c].chunk >= 0)
                tma_load_2d(sA + kb * 16384 + c * 1024, &tmA, kb * 64,
                            static_cast<int>(b * p.S + static_cast<int64_t>(ti[c].chunk) * kC), &bar_tma);
        }
    if (tid == 0) {
        int nvalid = 0;
        for (int c = 0; c < nch; ++c) nvalid += ti[c].chunk >= 0;
        mbar_arrive_expect_tx(&bar_tma, static_cast<uint32_t>(nkb * nvalid * 1024));
        if (!mbar_wait(&bar_tma, 0)) {
            set_err(p.err, DEV_ERR_TIMEOUT, 411);
            (void)mbar_wait(&bar_tma, 0);
            s_fail = 1;
        } else {
            tc_fence_after();
            constexpr uint32_t idesc = idesc_bf16_f32(128, kD);
            uint32_t acc = 0;
            for (int kb = 0; kb < nkb; ++kb) {
                const int ksteps = min(4, (p.r - kb * 64 + 15) / 16);
                for (int k = 0; k < ksteps; ++k) {
                    const uint64_t ad = smem_desc_sw128(smem_u32(sA + kb * 16384 + k * 32));
                    const uint64_t bd = smem_desc_sw128(smem_u32(sB + kb * 16384 + k * 32));
                    tc_mma_bf16(tmem, ad, bd, idesc, acc);
                    acc = 1;
                }
            }
            tc_commit(&bar_mma);
        }
    }
    __syncthreads();
    RopeRegs first;
    rope_fetch(p, ti[warp], first);   // table loads in flight while the MMAs run
    bool ok = !s_fail;
    if (ok && !mbar_wait(&bar_mma, 0)) {
        set_err(p.err, DEV_ERR_TIMEOUT, 412);
        (void)mbar_wait(&bar_mma, 0);
        ok = false;
    }
    ok = __syncthreads_and(ok);
    tc_fence_after();
    float* stage = reinterpret_cast<float*>(smem);            // reused once the MMAs are done
    float* smean = stage + kRows * kStagePitch;
    const int row = tid;
    if (ok) {
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
            float v0[32], v1[32];
            tmem_ld32(lane_base + 32 * h, v0);
            tmem_ld32(lane_base + kD / 2 + 32 * h, v1);
            tmem_ld_wait();
            stage_half(stage, row, h, v0, v1);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (ok) {
        rope_tile<OutT>(p, u, ti, stage, first);
        if (p.mode == 1) {
            __syncthreads();
            tile_stats(p, u, ti, stage, smean);
        }
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

// ------------------------------------------------------------------ fp32 CUDA-core path
__global__ void __launch_bounds__(128) k_rebuild_f32(RebuildParams p) {
    extern __shared__ __align__(16) uint8_t smem_f[];
    __shared__ TileInfo ti[kTileChunks];
    const int u = blockIdx.y, tile = blockIdx.x, tid = threadIdx.x;
    const int nch = load_tile_info(p, u, tile, ti);
    if (nch == 0) return;
    float* sB = reinterpret_cast<float*>(smem_f);                 // [r][d]
    float* stage = sB + p.r * kD;                                  // [128][pitch]
    float* smean = stage + kRows * kStagePitch;                    // [16][d]
    const float* B = static_cast<const float*>(p.B) + static_cast<int64_t>(u) * p.r * kD;
    for (int i = tid; i < p.r * kD / 4; i += 128)
        reinterpret_cast<float4*>(sB)[i] = reinterpret_cast<const float4*>(B)[i];
    __syncthreads();
    const int row = tid;
    const TileInfo mine = ti[row >> 3];
    const int b = u / p.H;
    float acc[kD];
#pragma unroll
    for (int k = 0; k < kD; ++k) acc[k] = 0.f;
    if (mine.chunk >= 0) {
        const float* arow = static_cast<const float*>(p.A) +
                            (b * p.S + static_cast<int64_t>(mine.chunk) * kC + (row & 7)) * p.r;
        for (int j = 0; j < p.r; ++j) {
            const float a = arow[j];
            const float4* brow = reinterpret_cast<const float4*>(sB + j * kD);
#pragma unroll
            for (int k = 0; k < kD / 4; ++k) {
                const float4 w = brow[k];
                acc[4 * k + 0] = fmaf(a, w.x, acc[4 * k + 0]);
                acc[4 * k + 1] = fmaf(a, w.y, acc[4 * k + 1]);
                acc[4 * k + 2] = fmaf(a, w.z, acc[4 * k + 2]);
                acc[4 * k + 3] = fmaf(a, w.w, acc[4 * k + 3]);
            }
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float v0[32], v1[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) { v0[i] = acc[32 * h + i]; v1[i] = acc[kD / 2 + 32 * h + i]; }
        stage_half(stage, row, h, v0, v1);
    }
    __syncthreads();
    RopeRegs first;
    rope_fetch(p, ti[threadIdx.x >> 5], first);
    rope_tile<float>(p, u, ti, stage, first);
    if (p.mode == 1) {
        __syncthreads();
        tile_stats(p, u, ti, stage, smean);
    }
}

// ------------------------------------------------------------------ exact keys (pre-filling)
// Algorithm 1 of the digest (section A2) takes the exact keys K and K_RoPE and
// builds the landmarks, the min-cosine test and the outlier keys from K_RoPE.
// When the caller has K, the tile's rows are the exact pre-RoPE keys, read
// straight into the fp32 staging tile (warp w loads rows w, w+4, ..., lane l
// dims [4l, 4l+4)); RoPE and the statistics follow as for rebuilt rows.
template <typename InT, typename OutT>
__global__ void __launch_bounds__(128) k_keys_exact(RebuildParams p) {
    extern __shared__ __align__(16) uint8_t smem_x[];
    __shared__ TileInfo ti[kTileChunks];
    const int u = blockIdx.y, tile = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nch = load_tile_info(p, u, tile, ti);
    if (nch == 0) return;
    float* stage = reinterpret_cast<float*>(smem_x);               // [128][pitch]
    float* smean = stage + kRows * kStagePitch;                    // [16][d]
    __syncthreads();
    const InT* K = static_cast<const InT*>(p.Kx) + static_cast<int64_t>(u) * p.S * kD;
    for (int row = warp; row < kRows; row += 4) {
        const TileInfo t = ti[row >> 3];
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t.chunk >= 0) {
            const InT* src = K + (static_cast<int64_t>(t.chunk) * kC + (row & 7)) * kD + 4 * lane;
            if constexpr (sizeof(InT) == 2) {
                const uint2 w = *reinterpret_cast<const uint2*>(src);
                const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
                const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
                v = make_float4(a.x, a.y, b.x, b.y);
            } else {
                v = *reinterpret_cast<const float4*>(src);
            }
        }
        *reinterpret_cast<float4*>(stage + row * kStagePitch + 4 * lane) = v;
    }
    __syncthreads();
    RopeRegs first;
    rope_fetch(p, ti[warp], first);
    rope_tile<OutT>(p, u, ti, stage, first);
    if (p.mode == 1) {
        __syncthreads();
        tile_stats(p, u, ti, stage, smean);
    }
}

int launch_keys_exact(const RebuildParams& p, int grid_x, bool out_bf16, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(kRows * kStagePitch + kTileChunks * kD) * sizeof(float);
    const dim3 grid(grid_x, p.U);
    cudaError_t e;
    if (p.kx_es == 2) {
        if (!out_bf16) return -1;
        auto k = k_keys_exact<__nv_bfloat16, __nv_bfloat16>;
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        k<<<grid, 128, smem, s>>>(p);
        e = cudaGetLastError();
    } else {
        if (out_bf16) return -1;
        auto k = k_keys_exact<float, float>;
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        k<<<grid, 128, smem, s>>>(p);
        e = cudaGetLastError();
    }
    return e == cudaSuccess ? 0 : -1;
}

// ------------------------------------------------------------------ ShadowKV+ append
// The rank-r state of a generated token (summary page, "The ShadowKV+ extension
// for generated tokens"): a[j] = sum over heads h and dims i of k'[h][i] * B[h][j][i],
// i.e. k' (the token's pre-RoPE key over the H heads) times Psi = B^T.  Block
// (b, j-group of 8), warp w -> j = 8*j-group + w; lane l covers dims [4l, 4l + 4)
// of every head, so each head's B row is read as one contiguous 256/512-byte line.
template <typename T>
__global__ void __launch_bounds__(256) k_project(const T* __restrict__ k_new, const T* __restrict__ B,
                                                 T* __restrict__ a_new, int H, int r, int64_t a_rows, int t) {
    const int b = blockIdx.x, lane = threadIdx.x & 31, j = blockIdx.y * 8 + (threadIdx.x >> 5);
    if (j >= r) return;
    float acc = 0.f;
    for (int h = 0; h < H; ++h) {
        const T* kr = k_new + (static_cast<int64_t>(b) * H + h) * kD + 4 * lane;
        const T* br = B + ((static_cast<int64_t>(b) * H + h) * r + j) * kD + 4 * lane;
        float kv[4], bv[4];
        if constexpr (sizeof(T) == 2) {
            const uint2 kw = *reinterpret_cast<const uint2*>(kr), bw = *reinterpret_cast<const uint2*>(br);
            const float2 k0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kw.x));
            const float2 k1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kw.y));
            const float2 b0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bw.x));
            const float2 b1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bw.y));
            kv[0] = k0.x; kv[1] = k0.y; kv[2] = k1.x; kv[3] = k1.y;
            bv[0] = b0.x; bv[1] = b0.y; bv[2] = b1.x; bv[3] = b1.y;
        } else {
            const float4 kw = *reinterpret_cast<const float4*>(kr), bw = *reinterpret_cast<const float4*>(br);
            kv[0] = kw.x; kv[1] = kw.y; kv[2] = kw.z; kv[3] = kw.w;
            bv[0] = bw.x; bv[1] = bw.y; bv[2] = bw.z; bv[3] = bw.w;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) acc = fmaf(kv[e], bv[e], acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) a_new[(static_cast<int64_t>(b) * a_rows + t) * r + j] = from_f<T>(acc);
}

int launch_project(int dtype, const void* k_new, const void* B, void* a_new, int batch, int H, int r,
                   int64_t a_rows, int t, cudaStream_t s) {
    const dim3 grid(batch, (r + 7) / 8);
    if (dtype == 0)
        k_project<float><<<grid, 256, 0, s>>>(static_cast<const float*>(k_new), static_cast<const float*>(B),
                                              static_cast<float*>(a_new), H, r, a_rows, t);
    else
        k_project<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(k_new),
                                                      static_cast<const __nv_bfloat16*>(B),
                                                      static_cast<__nv_bfloat16*>(a_new), H, r, a_rows, t);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// Then head h's key of the new token from the stored state: x = a . B_h, thread (g, c) summing
// rows j = g, g + 8, ... of column chunk c (eight dims), the 8 row groups summed in order, and
// RoPE at position pos with the angle composed from the (pos & 255) and (pos >> 8) tables.
// Small (128 threads, ~5 KB of shared memory) so that it fits beside the scorer.
template <typename T>
__global__ void __launch_bounds__(128) k_plus_key(PlusParams p) {
    extern __shared__ float sh_plus[];
    float* a_s = sh_plus;                         // [r]
    float* xp = a_s + p.r;                        // [8][d]
    const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const T* a = static_cast<const T*>(p.a_new) + (static_cast<int64_t>(b) * p.a_rows + p.t) * p.r;
    for (int j = tid; j < p.r; j += 128) a_s[j] = to_f(a[j]);
    __syncthreads();
    const int c = tid & 15, g = tid >> 4;
    const T* bh = static_cast<const T*>(p.B) + (static_cast<int64_t>(b) * p.H + h) * p.r * kD + 8 * c;
    float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int j = g; j < p.r; j += 8) {
        float v[8];
        load8(bh + static_cast<int64_t>(j) * kD, v);
        const float aj = a_s[j];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = fmaf(aj, v[e], x[e]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) xp[g * kD + 8 * c + e] = x[e];
    __syncthreads();
    if (tid < kD / 2) {
        float y1 = 0.f, y2 = 0.f;
        for (int gg = 0; gg < 8; ++gg) {
            y1 += xp[gg * kD + tid];
            y2 += xp[gg * kD + tid + kD / 2];
        }
        const int64_t pos = p.pos;
        const float2 lo = p.rope_lo[(pos & 255) * (kD / 2) + tid];
        const float2 hi = p.rope_hi[(pos >> 8) * (kD / 2) + tid];
        const float cs = hi.x * lo.x - hi.y * lo.y, sn = hi.y * lo.x + hi.x * lo.y;
        T* dst = static_cast<T*>(p.k_loc) + ((static_cast<int64_t>(b) * p.H + h) * p.loc_pitch + p.loc_row) * kD;
        dst[tid] = from_f<T>(y1 * cs - y2 * sn);
        dst[tid + kD / 2] = from_f<T>(y1 * sn + y2 * cs);
    }
}

int launch_plus_append(int dtype, const PlusParams& p, int batch, cudaStream_t s) {
    if (p.r > 256 || p.H < 1) return -1;
    if (launch_project(dtype, p.k_new, p.B, p.a_new, batch, p.H, p.r, p.a_rows, p.t, s)) return -1;
    const dim3 grid(batch, p.H);
    const size_t smem = static_cast<size_t>(p.r + 8 * kD) * sizeof(float);
    if (dtype == 0) k_plus_key<float><<<grid, 128, smem, s>>>(p);
    else k_plus_key<__nv_bfloat16><<<grid, 128, smem, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// ------------------------------------------------------------------ B transpose (bf16)
// Bt[u][n][k] = B[u][k][n]: the tensor-core B operand is K-major.
__global__ void k_transpose_B(const __nv_bfloat16* B, __nv_bfloat16* Bt, int r) {
    const int u = blockIdx.x;
    const __nv_bfloat16* src = B + static_cast<int64_t>(u) * r * kD;
    __nv_bfloat16* dst = Bt + static_cast<int64_t>(u) * r * kD;
    for (int i = threadIdx.x; i < r * kD; i += blockDim.x) {
        const int n = i / r, k = i % r;
        dst[i] = src[k * kD + n];
    }
}

static size_t tc_smem(const RebuildParams& p) {
    const size_t ops = static_cast<size_t>(p.nkb) * 2 * 16384;
    const size_t stats = static_cast<size_t>(kRows * kStagePitch + kTileChunks * kD) * 4;
    return (ops > stats ? ops : stats) + 1024;
}

int launch_rebuild_tc(const CUtensorMap* tmA, const CUtensorMap* tmB, const RebuildParams& p, int grid_x,
                      cudaStream_t s) {
    const size_t smem = tc_smem(p);
    auto fn = k_rebuild_tc<__nv_bfloat16>;
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (launch_pdl(fn, dim3(p.U, grid_x), dim3(128), smem, s, *tmA, *tmB, p) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return 0;
}

int launch_rebuild_f32(const RebuildParams& p, int grid_x, cudaStream_t s) {
    const size_t smem = (static_cast<size_t>(p.r) * kD + kRows * kStagePitch + kTileChunks * kD) * 4;
    cudaFuncSetAttribute(k_rebuild_f32, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    k_rebuild_f32<<<dim3(grid_x, p.U), 128, smem, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_transpose_B(const void* B, void* Bt, int U, int r, cudaStream_t s) {
    k_transpose_B<<<U, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(B), static_cast<__nv_bfloat16*>(Bt), r);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace skv
