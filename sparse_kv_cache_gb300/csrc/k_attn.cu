// Exact sparse attention over the assembled key/value set.
//
// ShadowKV (English summary, section 3.4, "Assembly of the final sparse KV
// cache": K = [K_outlier; RoPE(K_sparse); K_new], V likewise, then exact
// attention; Chinese digest section A2, Algorithm 2, and A7 "implementation
// details": attention itself was a library flash kernel on the A100).
//
// Split-K flash-decode.  Per (unit, split) one CTA takes 256 consecutive
// tokens of the virtual sequence [outliers | cache slots | local] and all G
// query heads of the unit: scores by half-warp dot products with a
// transpose-reduction, a block max and exp, then p.V with each half-warp
// owning 16 tokens and every lane 8 dims, reduced across half-warps in shared
// memory.  It writes (max, sum, acc[d]) per head; the CTA that finishes last
// for its unit (atomic ticket after a memory fence) merges the partials in
// fp32 and writes the output row.  Each key and value byte is read once.
#include <math_constants.h>

#include <cmath>
#include <mutex>

#include "shadowkv.h"
#include "skv_common.cuh"
#include "skv_internal.h"

namespace skv {

constexpr int kPartPitch = kD + 4;   // acc[d], max, sum, pad

// rows per unit of each region: the block pitch, or the region's own size when packed
__device__ __forceinline__ int64_t pitch_out(const AttnParams& p) { return p.unit_rows > 0 ? p.unit_rows : p.n_out; }
__device__ __forceinline__ int64_t pitch_c(const AttnParams& p) { return p.unit_rows > 0 ? p.unit_rows : p.n_cache; }
__device__ __forceinline__ int64_t pitch_loc(const AttnParams& p) { return p.unit_rows > 0 ? p.unit_rows : p.loc_cap; }

template <typename T>
__device__ __forceinline__ const T* row_ptr(const AttnParams& p, const void* out_b, const void* c_b,
                                            const void* loc_b, int u, int tau) {
    if (tau < p.n_out) return static_cast<const T*>(out_b) + (static_cast<int64_t>(u) * pitch_out(p) + tau) * kD;
    tau -= p.n_out;
    if (tau < p.n_cache) return static_cast<const T*>(c_b) + (static_cast<int64_t>(u) * pitch_c(p) + tau) * kD;
    tau -= p.n_cache;
    return static_cast<const T*>(loc_b) + (static_cast<int64_t>(u) * pitch_loc(p) + tau) * kD;
}

template <typename T, int G>
__global__ void __launch_bounds__(256) k_attn(AttnParams p) {
    extern __shared__ __align__(16) float sm[];
    float* sS = sm;                          // [256][G] scores, then probabilities
    float* sRed = sm + kAttnSeg * G;         // [16][G][d]
    __shared__ float red_m[8][G], red_l[8][G];
    __shared__ int s_last;

    const int u = blockIdx.y, split = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, hl = lane & 15, half = lane >> 4;
    const int ntot = p.n_out + p.n_cache + p.n_loc;
    const int seg0 = split * kAttnSeg;

    float qv[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) load8(static_cast<const T*>(p.q) + (static_cast<int64_t>(u) * G + g) * kD + hl * 8, qv[g]);

    // ---- scores
#pragma unroll
    for (int round = 0; round < 2; ++round) {
        const int tb = warp * 32 + round * 16 + half * 8;
        float acc[G][8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int tau = seg0 + tb + c;
            float v[8];
            if (tau < ntot) {
                load8(row_ptr<T>(p, p.k_out, p.k_c, p.k_loc, u, tau) + hl * 8, v);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) v[k] = 0.f;
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float a = 0.f;
#pragma unroll
                for (int k = 0; k < 8; ++k) a = fmaf(qv[g][k], v[k], a);
                acc[g][c] = a;
            }
        }
        float s[G];
#pragma unroll
        for (int g = 0; g < G; ++g) s[g] = transpose_reduce8(acc[g], hl) * p.scale;
        const int tl = tb + (hl >> 1);
        if ((hl & 1) == 0) {
            const bool valid = seg0 + tl < ntot;
#pragma unroll
            for (int g = 0; g < G; ++g) sS[tl * G + g] = valid ? s[g] : -CUDART_INF_F;
        }
    }
    __syncthreads();

    // ---- max and exp per head over the 256 tokens
    float M[G], Lsum[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float x = warp_max(sS[tid * G + g]);
        if (lane == 0) red_m[warp][g] = x;
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float x = red_m[0][g];
#pragma unroll
        for (int w = 1; w < 8; ++w) x = fmaxf(x, red_m[w][g]);
        M[g] = x;
        const float sv = sS[tid * G + g];
        const float pv = (sv == -CUDART_INF_F) ? 0.f : __expf(sv - x);
        sS[tid * G + g] = pv;
        const float ws = warp_sum(pv);
        if (lane == 0) red_l[warp][g] = ws;
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float x = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) x += red_l[w][g];
        Lsum[g] = x;
    }

    // ---- p . V
    const int hw = warp * 2 + half;
    float acc[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[g][k] = 0.f;
#pragma unroll 4
    for (int tl = hw; tl < kAttnSeg; tl += 16) {
        const int tau = seg0 + tl;
        if (tau >= ntot) break;
        float v[8];
        load8(row_ptr<T>(p, p.v_out, p.v_c, p.v_loc, u, tau) + hl * 8, v);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float pg = sS[tl * G + g];
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[g][k] = fmaf(pg, v[k], acc[g][k]);
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float* r = sRed + (hw * G + g) * kD + hl * 8;
        reinterpret_cast<float4*>(r)[0] = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
        reinterpret_cast<float4*>(r)[1] = make_float4(acc[g][4], acc[g][5], acc[g][6], acc[g][7]);
    }
    __syncthreads();
    float* mypart = p.part + (static_cast<int64_t>(u) * p.nsplit + split) * G * kPartPitch;
    for (int o = tid; o < G * kD; o += 256) {
        float x = 0.f;
#pragma unroll
        for (int h = 0; h < 16; ++h) x += sRed[h * G * kD + o];
        const int g = o / kD, dim = o % kD;
        mypart[g * kPartPitch + dim] = x;
        if (dim == 0) {
            mypart[g * kPartPitch + kD] = M[g];
            mypart[g * kPartPitch + kD + 1] = Lsum[g];
        }
    }

    // ---- the last CTA of this unit merges the partials
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(p.counter + u, 1) == p.nsplit - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const float* parts = p.part + static_cast<int64_t>(u) * p.nsplit * G * kPartPitch;
    for (int o = tid; o < G * kD; o += 256) {
        const int g = o / kD, dim = o % kD;
        float mx = -CUDART_INF_F;
        for (int s = 0; s < p.nsplit; ++s) mx = fmaxf(mx, __ldcg(parts + (s * G + g) * kPartPitch + kD));
        float ls = 0.f, a = 0.f;
        for (int s = 0; s < p.nsplit; ++s) {
            const float* ps = parts + (s * G + g) * kPartPitch;
            const float m = __ldcg(ps + kD);
            const float w = (m == -CUDART_INF_F) ? 0.f : __expf(m - mx);
            ls = fmaf(__ldcg(ps + kD + 1), w, ls);
            a = fmaf(__ldcg(ps + dim), w, a);
        }
        static_cast<T*>(p.out)[(static_cast<int64_t>(u) * G + g) * kD + dim] = from_f<T>(a / ls);
    }
    if (tid == 0) p.counter[u] = 0;
}

// ------------------------------------------------------------------ bf16: bulk-staged variant
// One thread issues 1-D bulk copies (TMA engine) of the CTA's key rows and
// value rows (at most three contiguous pieces: outliers, cache slots, local)
// into shared memory, completion counted on two mbarriers, so every byte of
// the CTA is in flight at once and the values arrive while the scores are
// being computed.  128 tokens per CTA, 4 warps, 3 CTAs per SM.
constexpr int kBSeg = 128;

template <int G>
__global__ void __launch_bounds__(128) k_attn_bulk(AttnParams p) {
    extern __shared__ __align__(128) uint8_t smb[];
    uint8_t* sK = smb;                                   // [128][128] bf16, then the reduction buffer
    uint8_t* sV = smb + kBSeg * kD * 2;                  // [128][128] bf16
    float* sS = reinterpret_cast<float*>(smb + 2 * kBSeg * kD * 2);   // [128][G]
    __shared__ uint64_t barK, barV;
    __shared__ float red_m[4][G], red_l[4][G];
    __shared__ int s_last, s_fail;

    const int u = blockIdx.y, split = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, hl = lane & 15, half = lane >> 4;
    const int ntot = p.n_out + p.n_cache + p.n_loc;
    const int seg0 = split * kBSeg;
    const int nseg = min(kBSeg, ntot - seg0);

    if (tid == 0) {
        mbar_init(&barK, 1);
        mbar_init(&barV, 1);
        s_fail = 0;
        fence_mbar_init();
        const uint32_t bytes = static_cast<uint32_t>(max(nseg, 0)) * kD * 2;
        mbar_arrive_expect_tx(&barK, bytes);
        mbar_arrive_expect_tx(&barV, bytes);
        // pieces of [seg0, seg0 + nseg) in the three regions
        const int bounds[4] = {0, p.n_out, p.n_out + p.n_cache, ntot};
        for (int r = 0; r < 3; ++r) {
            const int a = max(seg0, bounds[r]), b = min(seg0 + nseg, bounds[r + 1]);
            if (a >= b) continue;
            const __nv_bfloat16 *kb, *vb;
            if (r == 0) {
                kb = static_cast<const __nv_bfloat16*>(p.k_out) + (static_cast<int64_t>(u) * pitch_out(p) + a) * kD;
                vb = static_cast<const __nv_bfloat16*>(p.v_out) + (static_cast<int64_t>(u) * pitch_out(p) + a) * kD;
            } else if (r == 1) {
                kb = static_cast<const __nv_bfloat16*>(p.k_c) + (static_cast<int64_t>(u) * pitch_c(p) + a - bounds[1]) * kD;
                vb = static_cast<const __nv_bfloat16*>(p.v_c) + (static_cast<int64_t>(u) * pitch_c(p) + a - bounds[1]) * kD;
            } else {
                kb = static_cast<const __nv_bfloat16*>(p.k_loc) + (static_cast<int64_t>(u) * pitch_loc(p) + a - bounds[2]) * kD;
                vb = static_cast<const __nv_bfloat16*>(p.v_loc) + (static_cast<int64_t>(u) * pitch_loc(p) + a - bounds[2]) * kD;
            }
            const uint32_t nb = static_cast<uint32_t>(b - a) * kD * 2;
            bulk_g2s(sK + (a - seg0) * kD * 2, kb, nb, &barK);
            bulk_g2s(sV + (a - seg0) * kD * 2, vb, nb, &barV);
        }
    }
    float qv[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g)
        load8(static_cast<const __nv_bfloat16*>(p.q) + (static_cast<int64_t>(u) * G + g) * kD + hl * 8, qv[g]);
    __syncthreads();
    if (!mbar_wait(&barK, 0)) { set_err(p.err, DEV_ERR_TIMEOUT, 601); s_fail = 1; }

    // ---- scores: warp w owns tokens [32w, 32w+32), a half-warp per token row
#pragma unroll
    for (int round = 0; round < 2; ++round) {
        const int tb = warp * 32 + round * 16 + half * 8;
        float acc[G][8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float v[8];
            if (tb + c < nseg) {
                load8(reinterpret_cast<const __nv_bfloat16*>(sK + (tb + c) * kD * 2) + hl * 8, v);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) v[k] = 0.f;
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float a = 0.f;
#pragma unroll
                for (int k = 0; k < 8; ++k) a = fmaf(qv[g][k], v[k], a);
                acc[g][c] = a;
            }
        }
        float sc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) sc[g] = transpose_reduce8(acc[g], hl) * p.scale;
        const int tl = tb + (hl >> 1);
        if ((hl & 1) == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g) sS[tl * G + g] = tl < nseg ? sc[g] : -CUDART_INF_F;
        }
    }
    __syncthreads();
    float M[G], Lsum[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float x = warp_max(sS[tid * G + g]);
        if (lane == 0) red_m[warp][g] = x;
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float x = fmaxf(fmaxf(red_m[0][g], red_m[1][g]), fmaxf(red_m[2][g], red_m[3][g]));
        M[g] = x;
        const float sv = sS[tid * G + g];
        const float pv = (sv == -CUDART_INF_F) ? 0.f : __expf(sv - x);
        sS[tid * G + g] = pv;
        const float ws = warp_sum(pv);
        if (lane == 0) red_l[warp][g] = ws;
    }
    if (!mbar_wait(&barV, 0)) { set_err(p.err, DEV_ERR_TIMEOUT, 602); s_fail = 1; }
    __syncthreads();
    // A wait that ran out left shared memory incomplete: give the copies still in flight one
    // more bounded wait before the CTA may leave, and publish a NaN partial so that the unit's
    // output is NaN instead of a plausible wrong value (the error word says why).
    const bool failed = s_fail != 0;
    if (failed && tid == 0) {
        mbar_wait(&barK, 0);
        mbar_wait(&barV, 0);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) Lsum[g] = red_l[0][g] + red_l[1][g] + red_l[2][g] + red_l[3][g];

    // ---- p . V: 8 half-warps, 16 tokens each, lane owns 8 dims
    const int hw = warp * 2 + half;
    float acc[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[g][k] = 0.f;
#pragma unroll 4
    for (int tl = hw; tl < nseg; tl += 8) {
        float v[8];
        load8(reinterpret_cast<const __nv_bfloat16*>(sV + tl * kD * 2) + hl * 8, v);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float pg = sS[tl * G + g];
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[g][k] = fmaf(pg, v[k], acc[g][k]);
        }
    }
    float* sRed = reinterpret_cast<float*>(sK);          // keys are no longer needed
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float* r = sRed + (hw * G + g) * kD + hl * 8;
        reinterpret_cast<float4*>(r)[0] = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
        reinterpret_cast<float4*>(r)[1] = make_float4(acc[g][4], acc[g][5], acc[g][6], acc[g][7]);
    }
    __syncthreads();
    float* mypart = p.part + (static_cast<int64_t>(u) * p.nsplit + split) * G * kPartPitch;
    for (int o = tid; o < G * kD; o += 128) {
        float x = 0.f;
#pragma unroll
        for (int h = 0; h < 8; ++h) x += sRed[h * G * kD + o];
        const int g = o / kD, dim = o % kD;
        mypart[g * kPartPitch + dim] = failed ? CUDART_NAN_F : x;
        if (dim == 0) {
            mypart[g * kPartPitch + kD] = failed ? 0.f : M[g];
            mypart[g * kPartPitch + kD + 1] = failed ? 1.f : Lsum[g];
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(p.counter + u, 1) == p.nsplit - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // merge: (max, sum) of every split into shared memory, the weights once per
    // (split, head), then the accumulators with independent loads in flight
    const float* parts = p.part + static_cast<int64_t>(u) * p.nsplit * G * kPartPitch;
    float* sW = sS;                                   // [nsplit][G] weights (sS is free now)
    float* sMl = sS + p.nsplit * G;                   // [nsplit][G] (max, sum) pairs
    for (int i = tid; i < p.nsplit * G; i += 128) {
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(parts + i * kPartPitch + kD));
        sW[i] = ml.x;
        sMl[i] = ml.y;
    }
    __syncthreads();
    if (tid < G) {
        float mx = -CUDART_INF_F;
        for (int sp = 0; sp < p.nsplit; ++sp) mx = fmaxf(mx, sW[sp * G + tid]);
        float ls = 0.f;
        for (int sp = 0; sp < p.nsplit; ++sp) {
            const float m = sW[sp * G + tid];
            const float w = (m == -CUDART_INF_F) ? 0.f : __expf(m - mx);
            sW[sp * G + tid] = w;
            ls = fmaf(sMl[sp * G + tid], w, ls);
        }
        for (int sp = 0; sp < p.nsplit; ++sp) sW[sp * G + tid] /= ls;
    }
    __syncthreads();
    for (int o = tid; o < G * kD; o += 128) {
        const int g = o / kD, dim = o % kD;
        float a = 0.f;
#pragma unroll 8
        for (int sp = 0; sp < p.nsplit; ++sp) a = fmaf(__ldcg(parts + (sp * G + g) * kPartPitch + dim), sW[sp * G + g], a);
        static_cast<__nv_bfloat16*>(p.out)[(static_cast<int64_t>(u) * G + g) * kD + dim] = __float2bfloat16_rn(a);
    }
    if (tid == 0) p.counter[u] = 0;
}

template <int G>
static int launch_bulk(const AttnParams& p, cudaStream_t s) {
    const size_t scores = static_cast<size_t>(kBSeg) * G * 4;
    const size_t merge = static_cast<size_t>(2) * p.nsplit * G * 4;
    const size_t smem = static_cast<size_t>(2) * kBSeg * kD * 2 + (scores > merge ? scores : merge);
    cudaFuncSetAttribute(k_attn_bulk<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    k_attn_bulk<G><<<dim3(p.nsplit, p.U), 128, smem, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// ------------------------------------------------------------ persistent tensor-core form (bf16)
// The decode step's attention at full size: one CTA per SM walks a contiguous
// range of the flattened (unit, 128-token segment) sequence, as a pipeline of
// four roles over a ring of shared-memory stages:
//  * a producer warp loads each segment's key rows with two 2-D TMA copies
//    (128-row boxes, 128-byte swizzle) and its value rows with one 1-D bulk
//    copy -- a unit's outlier, cache and local rows are adjacent in its block --
//    and writes the unit's query rows;
//  * one thread issues q.K^T on the tensor cores (M = 128 rows, N = 16 >= G
//    query heads, K = 128) into a double-buffered accumulator in tensor memory;
//  * four score-reader warps turn the scores into probabilities against a
//    running max per head (one row per thread), keeping per-warp running sums;
//  * four value warps accumulate p.V on the CUDA cores one segment behind,
//    rescaling when the max moves.
// Where the range leaves a unit (or ends), a unit the CTA covers whole is
// normalised and written out; a unit shared with neighbouring CTAs is written
// as a partial at the slot of the CTA's first segment of it, and k_attn_merge,
// a programmatic dependent launch, merges those partials once the grid is done.
constexpr int kAWarps = 8;                          // score readers (warps 2..5) + value warps (6..9)
constexpr int kAKBytes = kBSeg * kD * 2;            // key tile: [2 halves][128 rows][128 B], swizzled
constexpr int kAQBytes = 4096;                      // query tile: [2 halves][16 rows][128 B], swizzled
constexpr int kAVBytes = kBSeg * kD * 2;            // value rows, plain
constexpr int kAStage = kAKBytes + kAQBytes + kAVBytes;
static_assert(kAStage % 1024 == 0, "stages keep the 1024-byte alignment of the swizzled tiles");
template <int G> struct AStages { static constexpr int value = G >= 8 ? 2 : 3; };


// 32-bit: the launcher checks that ncta * F fits
__device__ __forceinline__ int aseg_start(int c, int F, int ncta) { return c * F / ncta; }
// the CTA whose range holds flat segment f: the largest c with aseg_start(c) <= f
__device__ __forceinline__ int acta_of(int f, int F, int ncta) {
    int lo = 0, hi = ncta - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (aseg_start(mid, F, ncta) <= f) lo = mid; else hi = mid - 1;
    }
    return lo;
}
__device__ __forceinline__ void reader_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ void value_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

template <int G, int VB>   // VB: bytes of a value element, 2 (bf16) or 1 (e5m2)
__global__ void __launch_bounds__((kAWarps + 2) * 32, 1) k_attn_tc(const __grid_constant__ CUtensorMap tmK, AttnParams p) {
    constexpr int S = AStages<G>::value;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smb = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* sRed = reinterpret_cast<float*>(smb + S * kAStage);   // [4 value warps][G][kD]
    __shared__ uint64_t full[S], empty[S], accf[2], acce[2], pready[2], pfree[2], drain;
    __shared__ float sP[2][kBSeg * G];                 // probabilities of a segment
    __shared__ float red_m[2][4][G];                   // per-warp maxima of a segment
    __shared__ float sCorr[2][G], sMseg[2][G], sLw[2][4][G];   // rescale factor, running max, sums
    __shared__ uint32_t tmem_slot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntot = p.n_out + p.n_cache + p.n_loc;
    const int nsegu = p.nsplit;                       // segments per unit (= partial pitch)
    const int F = p.U * nsegu;
    const int ncta = gridDim.x;
    const int f0 = aseg_start(blockIdx.x, F, ncta), f1 = aseg_start(blockIdx.x + 1, F, ncta);
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 2);   // the copies (with their byte count), then the query rows
            mbar_init(&empty[i], 4);  // the value warps
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 4);
            mbar_init(&pready[b], 4);
            mbar_init(&pfree[b], 4);
        }
        mbar_init(&drain, 1);
        fence_mbar_init();
        prefetch_tensormap(&tmK);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_slot, 32);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    // launched as a programmatic dependent of the key rebuild (values in HBM): the prologue
    // above overlapped its tail; everything below reads what the earlier kernels wrote
    pdl_wait();
    // the merge kernel that follows may be scheduled beside this grid now; it waits for the
    // whole grid before it reads a partial
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        // ---------------------------------------------------------------- producer warp
        // The next segment's global reads (its cache slots' chunk ids, and the query rows when
        // it starts a new unit) are issued one segment ahead, so that their round trips overlap
        // the wait for a free stage and the current segment's copies.
        constexpr int QW = (G * 16 + 31) / 32;   // 16-byte words of the query rows per lane
        const uint64_t pol = l2_evict_first();   // read once per step
        const int ncs = p.n_cache / kC;          // cache slots per unit
        // chunk id of the cache slot lane `lane` copies for flat segment f (0: none)
        auto load_vch = [&](int f) -> int {
            if (!p.v_src || f >= f1) return 0;
            const int uu = f / nsegu, s0 = (f - uu * nsegu) * kBSeg;
            const int a0 = max(s0, p.n_out), a1 = min(s0 + min(kBSeg, ntot - s0), p.n_out + p.n_cache);
            const int nv = a1 > a0 ? (a1 - a0) / kC : 0;
            return lane < nv ? p.slot_chunk[static_cast<int64_t>(uu) * ncs + (a0 - p.n_out) / kC + lane] : 0;
        };
        auto load_q = [&](int uu, uint4 (&qw)[QW]) {
#pragma unroll
            for (int k = 0; k < QW; ++k) {
                const int w = lane + 32 * k, n = w >> 4, c16 = w & 15;
                qw[k] = n < G ? *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) +
                                                                (static_cast<int64_t>(uu) * G + n) * kD + c16 * 8)
                              : make_uint4(0, 0, 0, 0);
            }
        };
        int it = 0, u = f0 / nsegu, si = f0 - u * nsegu;
        uint4 qcur[QW], qnxt[QW];
#pragma unroll
        for (int k = 0; k < QW; ++k) qcur[k] = qnxt[k] = make_uint4(0, 0, 0, 0);
        if (f0 < f1) load_q(u, qcur);
        int vch_cur = load_vch(f0);
        for (int f = f0; f < f1; ++f, ++it) {
            const int vch_nxt = load_vch(f + 1);
            const bool unext = f + 1 < f1 && si + 1 == nsegu;   // segment f + 1 starts a new unit
            if (unext) load_q(u + 1, qnxt);
            const int st = it % S;
            const int okw = mbar_wait(&empty[st], ((it / S) & 1) ^ 1) ? 1 : 0;
            if (!__all_sync(0xffffffffu, okw)) {
                if (lane == 0) set_err(p.err, DEV_ERR_TIMEOUT, 621);
                break;
            }
            const int seg0 = si * kBSeg;
            const int ua = u;
            if (++si == nsegu) { si = 0; ++u; }
            const int nseg = min(kBSeg, ntot - seg0);
            uint8_t* sK = smb + st * kAStage;
            uint8_t* sQ = sK + kAKBytes;
            uint8_t* sV = sQ + kAQBytes;
            // cache rows of the segment whose values are read where they live (values in HBM):
            // lane i copies the rows of the segment's i-th cache slot from its chunk in V
            const int c0 = p.v_src ? max(seg0, p.n_out) : 0;
            const int c1 = p.v_src ? min(seg0 + nseg, p.n_out + p.n_cache) : 0;
            const int nvc = c1 > c0 ? (c1 - c0) / kC : 0;
            int vch = 0;
            if (lane < nvc) {
                vch = vch_cur;
                if (vch < 0 || vch >= p.nchunk) {
                    set_err(p.err, DEV_ERR_BOUNDS, 625);
                    vch = 0;   // read a valid chunk: the expected bytes still arrive
                }
            }
            if (lane == 0) {
                // the unit's block holds the segment's rows contiguously: two 128-row key boxes
                // (rows past the unit's tokens are read but scored -inf; past the last block the
                // copy fills zeros) and one bulk copy of the value rows (around the cache rows
                // when those are read from V)
                const int row = static_cast<int>(static_cast<int64_t>(ua) * p.unit_rows + seg0);
                mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(kAKBytes + nseg * kD * VB));
                tma_load_2d_hint(sK, &tmK, 0, row, &full[st], pol);
                tma_load_2d_hint(sK + 16384, &tmK, 64, row, &full[st], pol);
                const uint8_t* vb = static_cast<const uint8_t*>(p.v_out) + (static_cast<int64_t>(ua) * p.unit_rows + seg0) * kD * VB;
                if (nvc > 0) {
                    if (c0 > seg0)
                        bulk_g2s_hint(sV, vb, static_cast<uint32_t>(c0 - seg0) * kD * VB, &full[st], pol);
                    if (seg0 + nseg > c1)
                        bulk_g2s_hint(sV + (c1 - seg0) * kD * VB, vb + static_cast<int64_t>(c1 - seg0) * kD * VB,
                                      static_cast<uint32_t>(seg0 + nseg - c1) * kD * VB, &full[st], pol);
                } else {
                    bulk_g2s_hint(sV, vb, static_cast<uint32_t>(nseg) * kD * VB, &full[st], pol);
                }
            }
            __syncwarp();
            if (lane < nvc)
                bulk_g2s_hint(sV + (c0 - seg0 + lane * kC) * kD * VB,
                              static_cast<const uint8_t*>(p.v_src) + (static_cast<int64_t>(ua) * p.v_src_us +
                                                                      static_cast<int64_t>(vch) * kC * kD) * VB,
                              static_cast<uint32_t>(kC * kD * VB), &full[st], pol);
            // the unit's query rows g < G (the MMA's other columns are never read), written while
            // the copies are in flight; the second arrival publishes them
#pragma unroll
            for (int k = 0; k < QW; ++k) {
                const int w = lane + 32 * k, n = w >> 4, c16 = w & 15, kb = c16 >> 3, c = c16 & 7;
                if (n < G)
                    *reinterpret_cast<uint4*>(sQ + kb * 2048 + (n >> 3) * 1024 + (n & 7) * 128 + ((c ^ (n & 7)) << 4)) = qcur[k];
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[st]);
            vch_cur = vch_nxt;
            if (unext) {
#pragma unroll
                for (int k = 0; k < QW; ++k) qcur[k] = qnxt[k];
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        constexpr uint32_t idesc = idesc_bf16_f32(kBSeg, 16);
        int it = 0;
        for (int f = f0; f < f1; ++f, ++it) {
            const int st = it % S, b = it & 1;
            int ok = mbar_wait(&full[st], (it / S) & 1) ? 1 : 0;
            if (ok) ok = mbar_wait(&acce[b], ((it >> 1) & 1) ^ 1) ? 1 : 0;
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) set_err(p.err, DEV_ERR_TIMEOUT, 623);
                break;
            }
            if (lane == 0) {
                tc_fence_after();
                const uint8_t* sK = smb + st * kAStage;
                const uint8_t* sQ = sK + kAKBytes;
                uint32_t acc = 0;
                for (int kb = 0; kb < 2; ++kb)
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t ad = smem_desc_sw128(smem_u32(sK + kb * 16384 + k * 32));
                        const uint64_t bd = smem_desc_sw128(smem_u32(sQ + kb * 2048 + k * 32));
                        tc_mma_bf16(tmem + b * 16, ad, bd, idesc, acc);
                        acc = 1;
                    }
                tc_commit(&accf[b]);
            }
            __syncwarp();
        }
        if (lane == 0) tc_commit(&drain);
        __syncwarp();
        (void)mbar_wait(&drain, 0);
    } else if (warp < 2 + 4) {
        // ---------------------------------------------------------------- score readers
        // Four warps, one row (token) per thread: the segment's scores from the accumulator,
        // the running max per head across the unit's segments, the probabilities into
        // sP[buf], and per warp a running sum of them.  Segment i + 1 is worked here while the
        // value warps accumulate segment i.
        const int rw = warp - 2, quarter = warp & 3;     // TMEM lanes [32q, 32q + 32)
        const int tl = quarter * 32 + lane;
        bool ab = false;
        int cur_u = -1;
        float m_run[G], lw[G];
        int it = 0, u = f0 / nsegu, si = f0 - u * nsegu;
        for (int f = f0; f < f1; ++f, ++it) {
            const int buf = it & 1;
            const int seg0 = si * kBSeg;
            const int nseg = min(kBSeg, ntot - seg0);
            if (u != cur_u) {
                cur_u = u;
#pragma unroll
                for (int g = 0; g < G; ++g) { m_run[g] = -CUDART_INF_F; lw[g] = 0.f; }
            }
            if (!ab && !mbar_wait(&accf[buf], (it >> 1) & 1)) ab = true;
            tc_fence_after();
            float v[8];
            tmem_ld8(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + buf * 16, v);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[buf]);
            float sc[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                sc[g] = tl < nseg ? v[g] * p.scale : -CUDART_INF_F;
                const float x = warp_max(sc[g]);
                if (lane == 0) red_m[buf][rw][g] = x;
            }
            reader_sync();
            float corr[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float ms = fmaxf(fmaxf(red_m[buf][0][g], red_m[buf][1][g]), fmaxf(red_m[buf][2][g], red_m[buf][3][g]));
                const float mnew = fmaxf(m_run[g], ms);
                corr[g] = (m_run[g] == -CUDART_INF_F) ? 0.f : __expf(m_run[g] - mnew);
                m_run[g] = mnew;
            }
            // the value warps are done with this buffer (segment i - 2)
            if (!ab && !mbar_wait(&pfree[buf], ((it >> 1) & 1) ^ 1)) ab = true;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float pv = (sc[g] == -CUDART_INF_F) ? 0.f : __expf(sc[g] - m_run[g]);
                sP[buf][tl * G + g] = pv;
                lw[g] = lw[g] * corr[g] + warp_sum(pv);
            }
            if (lane == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    sLw[buf][rw][g] = lw[g];
                    if (rw == 0) {
                        sCorr[buf][g] = corr[g];
                        sMseg[buf][g] = m_run[g];
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&pready[buf]);
            if (++si == nsegu) { si = 0; ++u; }
        }
        if (ab && lane == 0) set_err(p.err, DEV_ERR_TIMEOUT, 624);
    } else {
        // ---------------------------------------------------------------- value warps
        // Four warps, eight half-warps, a lane 8 dims of every head: p . V over the segment's
        // rows, rescaled when the running max moves.  Where the range leaves a unit (or ends),
        // a unit this CTA covers whole is normalised and written out; otherwise the state is
        // written as the partial at the slot of the CTA's first segment of the unit, for
        // k_attn_merge.
        const int pt = tid - 192, pw = warp - 6;
        const int hl = lane & 15, half = lane >> 4, hw = pw * 2 + half;
        bool ab = false;
        int cur_u = -1, ubeg = 0;
        float acc[G][8];

        auto finish = [&](int u, int slot, int buf) {
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int k = 0; k < 8; ++k) acc[g][k] += __shfl_down_sync(0xffffffffu, acc[g][k], 16);
            if (half == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float* r = sRed + (pw * G + g) * kD + hl * 8;
                    reinterpret_cast<float4*>(r)[0] = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
                    reinterpret_cast<float4*>(r)[1] = make_float4(acc[g][4], acc[g][5], acc[g][6], acc[g][7]);
                }
            }
            value_sync();
            const bool whole = slot == 0 && f1 >= (u + 1) * nsegu;
            float* mypart = p.part + (static_cast<int64_t>(u) * nsegu + slot) * G * kPartPitch;
            for (int o = pt; o < G * kD; o += 128) {
                const int g = o / kD, dim = o % kD;
                const float l = sLw[buf][0][g] + sLw[buf][1][g] + sLw[buf][2][g] + sLw[buf][3][g];
                const float x = sRed[(0 * G + g) * kD + dim] + sRed[(1 * G + g) * kD + dim] +
                                sRed[(2 * G + g) * kD + dim] + sRed[(3 * G + g) * kD + dim];
                if (whole) {
                    static_cast<__nv_bfloat16*>(p.out)[(static_cast<int64_t>(u) * G + g) * kD + dim] = __float2bfloat16_rn(x / l);
                } else {
                    mypart[g * kPartPitch + dim] = x;
                    if (dim == 0) {
                        mypart[g * kPartPitch + kD] = sMseg[buf][g];
                        mypart[g * kPartPitch + kD + 1] = l;
                    }
                }
            }
            value_sync();   // sRed is free again
        };

        int it = 0, u = f0 / nsegu, si = f0 - u * nsegu;
        for (int f = f0; f < f1; ++f, ++it) {
            const int st = it % S, buf = it & 1;
            const int seg0 = si * kBSeg;
            const int nseg = min(kBSeg, ntot - seg0);
            if (u != cur_u) {
                cur_u = u;
                ubeg = f;
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int k = 0; k < 8; ++k) acc[g][k] = 0.f;
            }
            if (!ab && !mbar_wait(&full[st], (it / S) & 1)) ab = true;      // the value rows
            if (!ab && !mbar_wait(&pready[buf], (it >> 1) & 1)) ab = true;  // the probabilities
            const uint8_t* sV = smb + st * kAStage + kAKBytes + kAQBytes;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float c = sCorr[buf][g];
#pragma unroll
                for (int k = 0; k < 8; ++k) acc[g][k] *= c;
            }
#pragma unroll 4
            for (int r = hw; r < nseg; r += 8) {
                float v[8];
                if constexpr (VB == 1) load8_e5m2(sV + r * kD + hl * 8, v);
                else load8(reinterpret_cast<const __nv_bfloat16*>(sV + r * kD * 2) + hl * 8, v);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float pg = sP[buf][r * G + g];
#pragma unroll
                    for (int k = 0; k < 8; ++k) acc[g][k] = fmaf(pg, v[k], acc[g][k]);
                }
            }
            if (si == nsegu - 1 || f == f1 - 1) finish(u, ubeg - u * nsegu, buf);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&pfree[buf]);
                mbar_arrive(&empty[st]);
            }
            if (++si == nsegu) { si = 0; ++u; }
        }
        if (ab && lane == 0) set_err(p.err, DEV_ERR_TIMEOUT, 622);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 32);
    }
}

// Merges the partials of every unit shared by several CTAs of k_attn_tc (ncta CTAs):
// one CTA per unit, a thread per dimension.  The contributors' (max, sum, p.V) records of all
// heads come into shared memory by one bulk copy each, all in flight at once (measured: the
// attention phase with its merge 33.4 against 34.7 us per layer at 1M b1, where ~19 CTAs share
// a unit; 28.7 against 29.2 at 128K b8); past 96 KB of records they are loaded directly,
// eight contributors per round trip.  Launched as a programmatic dependent of k_attn_tc: its CTAs may
// become resident early and wait for the whole attention grid before reading.
// Combines contributors [0, ncon) of a unit in order, B at a time with all their loads in flight.
template <int G, int B>
__device__ __forceinline__ void merge_contribs(const float* parts, int cA, int ncon, int F, int ncta, int ubase,
                                               int dim, float (&M)[G], float (&L)[G], float (&A)[G]) {
    for (int c0 = 0; c0 < ncon; c0 += B) {
        float mm[B][G], ll[B][G], aa[B][G];
#pragma unroll
        for (int c = 0; c < B; ++c) {
            const bool on = c0 + c < ncon;
            const float* pc = parts;
            if (on) {
                const int st = aseg_start(cA + c0 + c, F, ncta) - ubase;
                pc = parts + static_cast<int64_t>(st > 0 ? st : 0) * G * kPartPitch;
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                mm[c][g] = on ? __ldcg(pc + g * kPartPitch + kD) : -CUDART_INF_F;
                ll[c][g] = on ? __ldcg(pc + g * kPartPitch + kD + 1) : 0.f;
                aa[c][g] = on ? __ldcg(pc + g * kPartPitch + dim) : 0.f;
            }
        }
#pragma unroll
        for (int c = 0; c < B; ++c)
#pragma unroll
            for (int g = 0; g < G; ++g) {
                if (mm[c][g] == -CUDART_INF_F) continue;
                if (mm[c][g] > M[g]) {
                    const float w = (M[g] == -CUDART_INF_F) ? 0.f : __expf(M[g] - mm[c][g]);
                    A[g] = A[g] * w + aa[c][g];
                    L[g] = L[g] * w + ll[c][g];
                    M[g] = mm[c][g];
                } else {
                    const float w = __expf(mm[c][g] - M[g]);
                    A[g] = fmaf(aa[c][g], w, A[g]);
                    L[g] = fmaf(ll[c][g], w, L[g]);
                }
            }
    }
}

template <int G>
__global__ void __launch_bounds__(kD) k_attn_merge(AttnParams p, int ncta, int stage_cap) {
    extern __shared__ __align__(16) uint8_t msm[];
    __shared__ uint64_t mbar;
    const int u = blockIdx.x, dim = threadIdx.x;
    const int nsegu = p.nsplit, F = p.U * nsegu;
    const int cA = acta_of(u * nsegu, F, ncta);
    const int ncon = acta_of((u + 1) * nsegu - 1, F, ncta) - cA + 1;
    // a unit with up to stage_cap contributors has their partials brought into shared memory by
    // one bulk copy each, all in flight at once
    const bool stg = ncon > 1 && ncon <= stage_cap;
    if (stg && dim == 0) {
        mbar_init(&mbar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (ncon <= 1) return;   // covered whole by one CTA, which wrote the output itself
    const float* parts = p.part + static_cast<int64_t>(u) * nsegu * G * kPartPitch;
    float M[G], L[G], A[G];
#pragma unroll
    for (int g = 0; g < G; ++g) { M[g] = -CUDART_INF_F; L[g] = 0.f; A[g] = 0.f; }
    if (stg) {
        constexpr uint32_t kBytes = G * kPartPitch * 4;   // one contributor's partial
        // one arrival with the byte count; the copies issued by lanes 0-7 of the four warps, so
        // that different warps' copy instructions issue side by side
        if (dim == 0) mbar_arrive_expect_tx(&mbar, static_cast<uint32_t>(ncon) * kBytes);
        if ((dim & 31) < 8)
            for (int c = (dim >> 5) * 8 + (dim & 31); c < ncon; c += 32) {
                const int st = aseg_start(cA + c, F, ncta) - u * nsegu;
                bulk_g2s(msm + c * kBytes, parts + static_cast<int64_t>(st > 0 ? st : 0) * G * kPartPitch, kBytes, &mbar);
            }
        if (!mbar_wait(&mbar, 0)) {
            if (dim == 0) set_err(p.err, DEV_ERR_TIMEOUT, 631);
            (void)mbar_wait(&mbar, 0);
        }
        const float* sp = reinterpret_cast<const float*>(msm);
        for (int c = 0; c < ncon; ++c)
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float* pc = sp + (c * G + g) * kPartPitch;
                const float mm = pc[kD], ll = pc[kD + 1], aa = pc[dim];
                if (mm == -CUDART_INF_F) continue;
                if (mm > M[g]) {
                    const float w = (M[g] == -CUDART_INF_F) ? 0.f : __expf(M[g] - mm);
                    A[g] = A[g] * w + aa;
                    L[g] = L[g] * w + ll;
                    M[g] = mm;
                } else {
                    const float w = __expf(mm - M[g]);
                    A[g] = fmaf(aa, w, A[g]);
                    L[g] = fmaf(ll, w, L[g]);
                }
            }
    } else if (ncon <= 4) {
        // a unit split over many CTAs (a long context at a small batch) takes eight
        // contributors per round trip; the usual two to four take two at a time
        merge_contribs<G, 2>(parts, cA, ncon, F, ncta, u * nsegu, dim, M, L, A);
    } else {
        merge_contribs<G, 8>(parts, cA, ncon, F, ncta, u * nsegu, dim, M, L, A);
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
        static_cast<__nv_bfloat16*>(p.out)[(static_cast<int64_t>(u) * G + g) * kD + dim] = __float2bfloat16_rn(A[g] / L[g]);
}

template <int G, int VB>
static int launch_tc(const CUtensorMap* tmK, const AttnParams& p, int nsm, cudaStream_t s) {
    const int ntot = p.n_out + p.n_cache + p.n_loc;
    if (!tmK || p.nsplit != (ntot + kBSeg - 1) / kBSeg || nsm <= 0) return -1;
    // the block layout, regions adjacent in each block
    const size_t rb = static_cast<size_t>(kD) * 2, rbv = static_cast<size_t>(kD) * VB;
    if (p.unit_rows < static_cast<int64_t>(p.n_out) + p.n_cache + p.n_loc ||
        static_cast<const uint8_t*>(p.k_c) != static_cast<const uint8_t*>(p.k_out) + p.n_out * rb ||
        static_cast<const uint8_t*>(p.k_loc) != static_cast<const uint8_t*>(p.k_c) + static_cast<size_t>(p.n_cache) * rb ||
        static_cast<const uint8_t*>(p.v_c) != static_cast<const uint8_t*>(p.v_out) + p.n_out * rbv ||
        static_cast<const uint8_t*>(p.v_loc) != static_cast<const uint8_t*>(p.v_c) + static_cast<size_t>(p.n_cache) * rbv)
        return -1;
    const int64_t F = static_cast<int64_t>(p.U) * p.nsplit;
    const int ncta = static_cast<int>(F < nsm ? F : nsm);
    if (ncta <= 0) return -1;
    if (F * (ncta + 1) > INT32_MAX || static_cast<int64_t>(p.U) * p.unit_rows > INT32_MAX) return -1;   // 32-bit indexing
    const size_t smem = static_cast<size_t>(AStages<G>::value) * kAStage + static_cast<size_t>(4) * G * kD * 4 + 1024;
    if (p.v_src && (!p.slot_chunk || p.n_cache % kC || p.nchunk <= 0)) return -1;
    cudaFuncSetAttribute(k_attn_tc<G, VB>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (p.pdl) {
        if (launch_pdl(k_attn_tc<G, VB>, dim3(ncta), dim3((kAWarps + 2) * 32), smem, s, *tmK, p) != cudaSuccess) {
            cudaGetLastError();
            return -1;
        }
    } else {
        k_attn_tc<G, VB><<<ncta, (kAWarps + 2) * 32, smem, s>>>(*tmK, p);
        if (cudaGetLastError() != cudaSuccess) return -1;
    }
    // contributors per unit at most: every CTA but the first and last of a unit's share holds at
    // least floor(F / ncta) of its segments
    const int64_t per_cta = F / ncta;
    const int64_t ncon_max = (p.nsplit - 1) / (per_cta > 0 ? per_cta : 1) + 2;
    const int64_t part_bytes = static_cast<int64_t>(G) * kPartPitch * 4;
    const int stage_cap = static_cast<int>(std::min<int64_t>(ncon_max, (96 << 10) / part_bytes));
    const size_t msmem = static_cast<size_t>(stage_cap) * part_bytes;
    if (msmem > 48 * 1024 &&
        cudaFuncSetAttribute(k_attn_merge<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(msmem)) != cudaSuccess)
        return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.U);
    cfg.blockDim = dim3(kD);
    cfg.dynamicSmemBytes = msmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k_attn_merge<G>, p, ncta, stage_cap) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return 2;   // the attention kernel and its merge
}

int launch_attn_tc(const CUtensorMap* k_all, const AttnParams& p, int nsm, cudaStream_t s) {
    switch (p.G) {
        case 1: return p.v_es == 1 ? launch_tc<1, 1>(k_all, p, nsm, s) : launch_tc<1, 2>(k_all, p, nsm, s);
        case 2: return p.v_es == 1 ? launch_tc<2, 1>(k_all, p, nsm, s) : launch_tc<2, 2>(k_all, p, nsm, s);
        case 4: return p.v_es == 1 ? launch_tc<4, 1>(k_all, p, nsm, s) : launch_tc<4, 2>(k_all, p, nsm, s);
        case 8: return p.v_es == 1 ? launch_tc<8, 1>(k_all, p, nsm, s) : launch_tc<8, 2>(k_all, p, nsm, s);
    }
    return -1;
}

int attn_segment(int dtype) { return dtype != 0 ? kBSeg : kAttnSeg; }

template <typename T, int G>
static int launch_t(const AttnParams& p, cudaStream_t s) {
    const size_t smem = (static_cast<size_t>(kAttnSeg) * G + 16 * G * kD) * 4;
    cudaFuncSetAttribute(k_attn<T, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    k_attn<T, G><<<dim3(p.nsplit, p.U), 256, smem, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_attn(int dtype, const AttnParams& p, cudaStream_t s) {
    if (dtype == 1) {
        switch (p.G) {
            case 1: return launch_bulk<1>(p, s);
            case 2: return launch_bulk<2>(p, s);
            case 4: return launch_bulk<4>(p, s);
            case 8: return launch_bulk<8>(p, s);
        }
    } else {
        switch (p.G) {
            case 1: return launch_t<float, 1>(p, s);
            case 2: return launch_t<float, 2>(p, s);
            case 4: return launch_t<float, 4>(p, s);
            case 8: return launch_t<float, 8>(p, s);
        }
    }
    return -1;
}

}  // namespace skv

// ---------------------------------------------------------------------------
// Sparse attention without any allocation.
//
// Some callers cannot allocate device memory while they run: an inference
// server that carves every byte of HBM out of one pool at start-up, code that
// runs under an allocator lock, or an integration that forbids cudaMalloc on
// its hot path because an allocation may synchronise the device.  This entry
// point serves them.  It runs k_attn_bulk, the bulk-copy split-K attention
// kernel above (the decode step itself runs the persistent tensor-core form,
// k_attn_tc, whose scratch lives with the layer), over key/value regions the
// caller provides, and keeps that kernel's scratch -- the per-split partial
// results, the per-unit merge tickets and an error word -- in one fixed array
// compiled into this library instead of memory allocated for a layer.  It
// calls no cudaMalloc, cudaFree or other allocating routine.
namespace skv {
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // whole array: 16 MiB
constexpr size_t kNoAllocTicketBytes = size_t(64) << 10;    // merge tickets of up to 16384 units
constexpr size_t kNoAllocErrBytes = 256;                    // error word (code, where), then padding
constexpr size_t kNoAllocPartOffset = kNoAllocTicketBytes + kNoAllocErrBytes;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Identifier of the calling thread's current context (0 if unknown): the array's address is
// resolved again when it changes, e.g. after cudaDeviceReset made a new primary context.
static unsigned long long current_ctx_id() {
    static CtxGetCurrentFn get_cur = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static bool looked = false;
    if (!looked) {
        looked = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
        cudaGetLastError();
    }
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (get_cur && get_id && get_cur(&c) == CUDA_SUCCESS && c && get_id(c, &id) == CUDA_SUCCESS) return id;
    return 0;
}

struct NoAllocDevice {
    void* addr = nullptr;              // the array's device address in that context
    unsigned long long ctx = 0;        // context the address belongs to
    int smem_limit = 0;                // dynamic shared memory a k_attn_bulk launch may ask for
    bool attr_set[4] = {false, false, false, false};   // G = 1, 2, 4, 8: the shared-memory cap set
};
static std::mutex g_noalloc_mu;
static NoAllocDevice g_noalloc_dev[256];

static int g_index(int G) { return G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3; }

template <int G>
static cudaError_t bulk_func_attrs(int* static_smem) {
    cudaFuncAttributes fa;
    const cudaError_t e = cudaFuncGetAttributes(&fa, k_attn_bulk<G>);
    *static_smem = e == cudaSuccess ? static_cast<int>(fa.sharedSizeBytes) : 0;
    return e;
}
template <int G>
static cudaError_t bulk_set_cap(int bytes) {
    return cudaFuncSetAttribute(k_attn_bulk<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// Per-device set-up, under g_noalloc_mu, with that device current: the array's address, the
// shared-memory limit, and the kernels' dynamic shared-memory cap (set once per device and G).
static int noalloc_setup(int dev, NoAllocDevice** out) {
    NoAllocDevice& d = g_noalloc_dev[dev];
    const unsigned long long ctx = current_ctx_id();
    if (!d.addr || (ctx != 0 && ctx != d.ctx)) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return SKV_ERR_CUDA;
        }
        d = NoAllocDevice{};
        d.addr = p;
        d.ctx = current_ctx_id();
        int optin = 0, st = 0, st_max = 0;
        if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            bulk_func_attrs<1>(&st) != cudaSuccess || (st_max = st, bulk_func_attrs<2>(&st)) != cudaSuccess ||
            (st_max = st > st_max ? st : st_max, bulk_func_attrs<4>(&st)) != cudaSuccess ||
            (st_max = st > st_max ? st : st_max, bulk_func_attrs<8>(&st)) != cudaSuccess) {
            cudaGetLastError();
            d = NoAllocDevice{};
            return SKV_ERR_CUDA;
        }
        st_max = st > st_max ? st : st_max;
        d.smem_limit = optin - st_max;
    }
    *out = &d;
    return SKV_OK;
}

// dynamic shared memory of one k_attn_bulk CTA: key and value rows, then the larger of the
// score buffer and the merge state (a weight and a (max, sum) value per split and head)
static int64_t bulk_smem_bytes(int64_t nsplit, int G) {
    const int64_t scores = static_cast<int64_t>(kBSeg) * G * 4;
    const int64_t merge = 2 * nsplit * G * 4;
    return static_cast<int64_t>(2) * kBSeg * kD * 2 + (scores > merge ? scores : merge);
}

template <int G>
static int launch_noalloc(const AttnParams& p, NoAllocDevice* d, int smem, cudaStream_t s) {
    const int gi = g_index(G);
    if (!d->attr_set[gi]) {
        // the cap is the device's limit, so any shape accepted by the size checks launches
        if (bulk_set_cap<G>(d->smem_limit) != cudaSuccess) {
            cudaGetLastError();
            return SKV_ERR_CUDA;
        }
        d->attr_set[gi] = true;
    }
    k_attn_bulk<G><<<dim3(p.nsplit, p.U), 128, smem, s>>>(p);
    if (cudaGetLastError() != cudaSuccess) return SKV_ERR_CUDA;
    return SKV_OK;
}

static bool is_device_mem(const void* ptr) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}
}  // namespace skv

extern "C" int shadowkv_sparse_attention_noalloc(const skv_attention_args* a, skv_stream stream) {
    using namespace skv;
    if (!a) return SKV_ERR_INVALID;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SKV_ERR_CUDA;
    }
    if (dev < 0 || dev >= 256) return SKV_ERR_UNSUPPORTED;
    if (a->units == 0) {   // set-up only
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        NoAllocDevice* d = nullptr;
        int rc = noalloc_setup(dev, &d);
        for (int G : {1, 2, 4, 8}) {
            if (rc) break;
            cudaError_t e = G == 1 ? bulk_set_cap<1>(d->smem_limit) : G == 2 ? bulk_set_cap<2>(d->smem_limit)
                          : G == 4 ? bulk_set_cap<4>(d->smem_limit) : bulk_set_cap<8>(d->smem_limit);
            if (e != cudaSuccess) {
                cudaGetLastError();
                rc = SKV_ERR_CUDA;
            } else {
                d->attr_set[g_index(G)] = true;
            }
        }
        return rc;
    }
    if (a->dtype != SKV_BF16) return SKV_ERR_UNSUPPORTED;
    const int G = a->group;
    if (a->units < 0 || (G != 1 && G != 2 && G != 4 && G != 8)) return SKV_ERR_INVALID;
    if (a->n_outlier_tokens < 0 || a->n_cache_tokens < 0 || a->n_local_tokens < 1 ||
        a->n_local_tokens > a->local_capacity)
        return SKV_ERR_INVALID;
    const void* ptrs[] = {a->q, a->k_outlier, a->v_outlier, a->k_cache, a->v_cache, a->k_local, a->v_local, a->out};
    for (const void* p : ptrs)
        if (reinterpret_cast<uintptr_t>(p) & 15) return SKV_ERR_INVALID;
    if (!a->q || !a->k_local || !a->v_local || !a->out) return SKV_ERR_INVALID;
    if ((a->n_outlier_tokens && (!a->k_outlier || !a->v_outlier)) || (a->n_cache_tokens && (!a->k_cache || !a->v_cache)))
        return SKV_ERR_INVALID;
    // every region the kernel reads or writes must be device memory (the bulk copies cannot
    // read pageable host memory); pointer queries allocate nothing
    if (!is_device_mem(a->q) || !is_device_mem(a->out) || !is_device_mem(a->k_local) || !is_device_mem(a->v_local) ||
        (a->n_outlier_tokens && (!is_device_mem(a->k_outlier) || !is_device_mem(a->v_outlier))) ||
        (a->n_cache_tokens && (!is_device_mem(a->k_cache) || !is_device_mem(a->v_cache))))
        return SKV_ERR_INVALID;
    const int64_t ntot = static_cast<int64_t>(a->n_outlier_tokens) + a->n_cache_tokens + a->n_local_tokens;
    const int64_t nsplit = (ntot + kBSeg - 1) / kBSeg;
    const int64_t part_bytes = static_cast<int64_t>(a->units) * nsplit * G * kPartPitch * 4;
    if (nsplit > (1 << 20) || static_cast<int64_t>(a->units) * 4 > static_cast<int64_t>(kNoAllocTicketBytes) ||
        part_bytes > static_cast<int64_t>(kNoAllocScratchBytes - kNoAllocPartOffset))
        return SKV_ERR_INVALID;   // the shape needs more scratch than the fixed array holds

    void* base = nullptr;
    NoAllocDevice* d = nullptr;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    int rc = noalloc_setup(dev, &d);
    if (rc) return rc;
    base = d->addr;
    const int64_t smem = bulk_smem_bytes(nsplit, G);
    if (smem > d->smem_limit) return SKV_ERR_INVALID;   // the merge state does not fit in shared memory
    // the merge tickets must start at zero; the partials are fully overwritten
    if (cudaMemsetAsync(base, 0, static_cast<size_t>(a->units) * 4, stream) != cudaSuccess) {
        cudaGetLastError();
        return SKV_ERR_CUDA;
    }
    AttnParams p{};
    p.q = a->q;
    p.k_out = a->k_outlier; p.v_out = a->v_outlier; p.n_out = a->n_outlier_tokens;
    p.k_c = a->k_cache; p.v_c = a->v_cache; p.n_cache = a->n_cache_tokens;
    p.k_loc = a->k_local; p.v_loc = a->v_local; p.n_loc = a->n_local_tokens; p.loc_cap = a->local_capacity;
    p.out = a->out;
    p.counter = static_cast<int*>(base);
    p.err = reinterpret_cast<int*>(static_cast<unsigned char*>(base) + kNoAllocTicketBytes);
    p.part = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kNoAllocPartOffset);
    p.nsplit = static_cast<int>(nsplit);
    p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(kD)));
    p.G = G; p.U = a->units;
    const int sm = static_cast<int>(smem);
    switch (G) {
        case 1: return launch_noalloc<1>(p, d, sm, stream);
        case 2: return launch_noalloc<2>(p, d, sm, stream);
        case 4: return launch_noalloc<4>(p, d, sm, stream);
        default: return launch_noalloc<8>(p, d, sm, stream);
    }
}

extern "C" int shadowkv_sparse_attention_noalloc_status(skv_stream stream) {
    using namespace skv;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SKV_ERR_CUDA;
    }
    if (dev < 0 || dev >= 256) return SKV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoAllocDevice* d = nullptr;
    int rc = noalloc_setup(dev, &d);
    if (rc) return rc;
    int e[2] = {0, 0};
    unsigned char* w = static_cast<unsigned char*>(d->addr) + kNoAllocTicketBytes;
    if (cudaStreamSynchronize(stream) != cudaSuccess ||
        cudaMemcpyAsync(e, w, sizeof(e), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaMemsetAsync(w, 0, sizeof(e), stream) != cudaSuccess || cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return SKV_ERR_CUDA;
    }
    if (e[0] == DEV_ERR_TIMEOUT) return SKV_ERR_TIMEOUT;
    if (e[0] != 0) return SKV_ERR_DEVICE_BOUNDS;
    return SKV_OK;
}
