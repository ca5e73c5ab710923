// Landmark scoring, P = q . L^T for the G query heads of each KV head.
//
// ShadowKV (Chinese digest, section A2, Algorithm 2: P = MatMul(Q, L.T),
// S = Softmax(P / sqrt(d))); English summary section 3.4, "Decoding-Time KV
// Selection", Step 1.  This is the largest HBM stream of a decode step: every
// selectable landmark row (d values) is read once per step.
//
// Work is cut into runs of kRunChunks landmarks of one unit.  Each run leaves,
// besides z = P / sqrt(d) as fp32 [U][n_c][G], one record per part (warp) and
// query head: the running (max z, sum exp(z - max)), from which the next
// kernel forms every head's log-sum-exp without a second pass over z.
//
// bf16 storage (k_score_tc): the contraction runs on the 5th-generation tensor
// cores so that the kernel is bound by the landmark stream alone.  A
// persistent CTA per SM claims runs from an atomic counter (fast SMs take more
// runs; the tail is one run).  One warp streams 128-landmark tiles (two
// 64-column, 128-byte-swizzled boxes, 32 KB) with 2-D TMA copies into a
// 6-stage shared-memory ring; one thread issues tcgen05 MMAs, M = 128
// landmarks x N = 16 (the unit's G <= 8 queries; the other columns are never
// read) x K = 128, into a double-buffered fp32 accumulator in tensor memory;
// four epilogue warps read one landmark row each per thread, scale, store z
// and keep the running (max, sum exp) per head.  Every stage carries its own
// copy of the run's query rows, written by the producer warp from registers,
// so runs of different units follow each other without any drain.
// fp32 storage (k_score): CUDA-core dot products, the query in registers, one
// half-warp per landmark row and a transpose-reduction of the partial sums;
// runs are dealt round-robin to the CTAs.
#include <math_constants.h>

#include "skv_common.cuh"
#include "skv_internal.h"

namespace skv {

// ------------------------------------------------------------------ CUDA-core path
template <typename T, int G>
__global__ void __launch_bounds__((kScoreWarps + 1) * 32) k_score(ScoreParams p) {
    constexpr int ROWB = kD * Elem<T>::bytes;
    constexpr int TILE = kScoreStageBytes / ROWB;
    static_assert(TILE <= kScoreWarps * 16, "tile larger than one pass of the consumer warps");
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t full[kScoreStages], empty[kScoreStages];
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kScoreStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kScoreWarps);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int64_t n_c = p.n_c;

    if (warp == kScoreWarps) {
        // ------------------------------------------------ producer (one lane)
        if (lane != 0) return;
        int it = 0;
        bool ok = true;
        for (int r = blockIdx.x; ok && r < p.total_runs; r += gridDim.x) {
            const int64_t u = r / p.nru;
            const int64_t a = u * n_c + static_cast<int64_t>(r % p.nru) * kRunChunks;
            const int64_t e = min(a + kRunChunks, (u + 1) * n_c);
            for (int64_t j = a; j < e; j += TILE, ++it) {
                const int nv = static_cast<int>(min(static_cast<int64_t>(TILE), e - j));
                const int s = it % kScoreStages;
                if (it >= kScoreStages && !mbar_wait(&empty[s], ((it / kScoreStages) - 1) & 1)) {
                    set_err(p.err, DEV_ERR_TIMEOUT, 101);
                    s_abort = 1;
                    ok = false;
                    break;
                }
                if (s_abort) { ok = false; break; }
                mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(nv * ROWB));
                bulk_g2s(smem + s * kScoreStageBytes, static_cast<const uint8_t*>(p.L) + j * ROWB,
                         static_cast<uint32_t>(nv * ROWB), &full[s]);
            }
        }
        if (!ok) {
            // leave no copy in flight: wait (bounded) for the stages issued last
            for (int k = max(0, it - kScoreStages); k < it; ++k)
                (void)mbar_wait(&full[k % kScoreStages], (k / kScoreStages) & 1);
        }
        return;
    }

    // ---------------------------------------------------- consumers
    const int hl = lane & 15, half = lane >> 4;
    float qv[G][8];
    int it = 0;
    bool ok = true;
    for (int r = blockIdx.x; ok && r < p.total_runs; r += gridDim.x) {
        const int64_t u = r / p.nru;
        const int64_t a = u * n_c + static_cast<int64_t>(r % p.nru) * kRunChunks;
        const int64_t e = min(a + kRunChunks, (u + 1) * n_c);
#pragma unroll
        for (int g = 0; g < G; ++g) load8(static_cast<const T*>(p.q) + (u * G + g) * kD + hl * 8, qv[g]);
        float m[G], sx[G];
#pragma unroll
        for (int g = 0; g < G; ++g) { m[g] = -CUDART_INF_F; sx[g] = 0.f; }

        for (int64_t j = a; ok && j < e; j += TILE, ++it) {
            const int nv = static_cast<int>(min(static_cast<int64_t>(TILE), e - j));
            const int s = it % kScoreStages;
            if (s_abort || !mbar_wait(&full[s], (it / kScoreStages) & 1)) {
                set_err(p.err, DEV_ERR_TIMEOUT, 102);
                s_abort = 1;
                ok = false;
                break;
            }
            const uint8_t* st = smem + s * kScoreStageBytes;
            const int cb = warp * 16 + half * 8;
            if (warp * 16 < nv) {
                float acc[G][8];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float v[8];
                    if (cb + c < nv) {
                        load8(reinterpret_cast<const T*>(st + (cb + c) * ROWB) + hl * 8, v);
                    } else {
#pragma unroll
                        for (int k = 0; k < 8; ++k) v[k] = 0.f;
                    }
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float acc1 = 0.f;
#pragma unroll
                        for (int k = 0; k < 8; ++k) acc1 = fmaf(qv[g][k], v[k], acc1);
                        acc[g][c] = acc1;
                    }
                }
                float z[G];
#pragma unroll
                for (int g = 0; g < G; ++g) z[g] = transpose_reduce8(acc[g], hl) * p.scale;
                const int cj = cb + (hl >> 1);
                if ((hl & 1) == 0 && cj < nv) {
                    float* dst = p.logits + (j + cj) * G;
#pragma unroll
                    for (int g = 0; g < G; ++g) dst[g] = z[g];
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        if (z[g] > m[g]) {
                            sx[g] = sx[g] * __expf(m[g] - z[g]) + 1.f;
                            m[g] = z[g];
                        } else {
                            sx[g] += __expf(z[g] - m[g]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        // merge the lanes' (max, sum) and publish this warp's record for run r
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float M = warp_max(m[g]);
            const float t = (m[g] == -CUDART_INF_F) ? 0.f : sx[g] * __expf(m[g] - M);
            const float S = warp_sum(t);
            if (lane == 0) p.part[(static_cast<int64_t>(r) * kScoreWarps + warp) * G + g] = make_float2(M, S);
        }
    }
}

// ------------------------------------------------------------------ tensor-core path
// What flows from the producer to the MMA thread (per stage) and from the MMA
// thread to the epilogue (per accumulator buffer).
struct ScTile {
    int run;        // -1: no more work
    int nv;         // valid landmarks in the tile
    int64_t j;      // flat index of the tile's first landmark
    int unit;
    int last;       // last tile of its run
};

template <int G>
__global__ void __launch_bounds__(192, 1) k_score_tc(const __grid_constant__ CUtensorMap tmL, ScoreParams p) {
    // stage s: [2 K-blocks][128 landmark rows][128 B] then [2 K-blocks][16 query rows][128 B]
    constexpr int kStage = 32768 + 4096;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[kScStages], empty[kScStages], accf[2], acce[2], drain;
    __shared__ ScTile stile[kScStages], atile[2];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n_c = p.n_c;
    if (tid == 0) {
        for (int s = 0; s < kScStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        // accf: the MMA commit (accumulator complete) + a release-arrive after the tile record is written
        for (int b = 0; b < 2; ++b) { mbar_init(&accf[b], 2); mbar_init(&acce[b], 4); }
        mbar_init(&drain, 1);
        s_abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmL);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_slot, 32);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    // the set-up above overlapped the previous kernel; everything below reads its results
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        // ------------------------------------------------ producer warp: claims runs, writes each
        // stage's query tile (rows g < G; the MMA's other columns are never read) and issues the
        // landmark copies
        constexpr int QW = (G * 16 + 31) / 32;   // 16-byte words of the query rows per lane
        const uint64_t pol = l2_evict_first();   // read once per step
        int it = 0;
        int next = (lane == 0) ? atomicAdd(p.sched, 1) : 0;
        next = __shfl_sync(0xffffffffu, next, 0);
        bool done = false;
        while (!done) {
            const int r = s_abort ? p.total_runs : next;
            int64_t a = 0, e = 0;
            int u = 0;
            if (r < p.total_runs) {
                u = r / p.nru;
                a = static_cast<int64_t>(u) * n_c + static_cast<int64_t>(r % p.nru) * kRunChunks;
                e = min(a + kRunChunks, static_cast<int64_t>(u + 1) * n_c);
                int nx = (lane == 0) ? atomicAdd(p.sched, 1) : 0;   // claim the next run early
                next = __shfl_sync(0xffffffffu, nx, 0);
            } else {
                done = true;
            }
            uint4 qw[QW];
#pragma unroll
            for (int k = 0; k < QW; ++k) {
                const int w = lane + 32 * k, n = w >> 4, c16 = w & 15;
                qw[k] = make_uint4(0, 0, 0, 0);
                if (!done && n < G)
                    qw[k] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) +
                                                            (static_cast<int64_t>(u) * G + n) * kD + c16 * 8);
            }
            for (int64_t j = a; done || j < e; j += kScTile, ++it) {
                const int s = it % kScStages;
                uint8_t* st = smem + s * kStage;
                const int okw = mbar_wait(&empty[s], ((it / kScStages) & 1) ^ 1) ? 1 : 0;
                if (!__all_sync(0xffffffffu, okw)) {
                    if (lane == 0) set_err(p.err, DEV_ERR_TIMEOUT, 111);
                    s_abort = 1;
                    done = true;
                }
                if (done) {   // end marker: a plain arrival completes the stage's phase
                    if (lane == 0) {
                        stile[s].run = -1;
                        mbar_arrive(&full[s]);
                    }
                    ++it;
                    break;
                }
#pragma unroll
                for (int k = 0; k < QW; ++k) {
                    const int w = lane + 32 * k, n = w >> 4, c16 = w & 15, kb = c16 >> 3, c = c16 & 7;
                    if (n < G)
                        *reinterpret_cast<uint4*>(st + 32768 + kb * 2048 + (n >> 3) * 1024 + (n & 7) * 128 +
                                                  ((c ^ (n & 7)) << 4)) = qw[k];
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ScTile t;
                    t.run = r;
                    t.j = j;
                    t.nv = static_cast<int>(min(static_cast<int64_t>(kScTile), e - j));
                    t.unit = u;
                    t.last = (j + kScTile >= e);
                    stile[s] = t;
                    mbar_arrive_expect_tx(&full[s], 32768);
                    tma_load_2d_hint(st, &tmL, 0, static_cast<int>(j), &full[s], pol);
                    tma_load_2d_hint(st + 16384, &tmL, 64, static_cast<int>(j), &full[s], pol);
                }
                __syncwarp();
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_bf16_f32(kScTile, kScN);
        int it = 0;
        while (true) {
            const int s = it % kScStages, b = it & 1;
            int ok = mbar_wait(&full[s], (it / kScStages) & 1) ? 1 : 0;
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) { if (lane == 0) set_err(p.err, DEV_ERR_TIMEOUT, 112); s_abort = 1; break; }
            const ScTile t = stile[s];
            // the accumulator buffer must be free before its record is replaced
            if (lane == 0) ok = mbar_wait(&acce[b], ((it >> 1) & 1) ^ 1) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) { if (lane == 0) set_err(p.err, DEV_ERR_TIMEOUT, 113); s_abort = 1; break; }
            if (t.run < 0) {
                if (lane == 0) { atile[b] = t; mbar_arrive_cnt(&accf[b], 2); }
                break;
            }
            if (lane == 0) {
                tc_fence_after();
                const uint8_t* st = smem + s * kStage;
                uint32_t acc = 0;
                for (int kb = 0; kb < 2; ++kb)
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t ad = smem_desc_sw128(smem_u32(st + kb * 16384 + k * 32));
                        const uint64_t bd = smem_desc_sw128(smem_u32(st + 32768 + kb * 2048 + k * 32));
                        tc_mma_bf16(tmem + b * kScN, ad, bd, idesc, acc);
                        acc = 1;
                    }
                tc_commit(&empty[s]);
                tc_commit(&accf[b]);
                atile[b] = t;
                mbar_arrive(&accf[b]);   // release: the record is visible once the phase completes
            }
            __syncwarp();
            ++it;
        }
        // every MMA retired before the accumulator is released
        if (lane == 0) tc_commit(&drain);
        __syncwarp();
        (void)mbar_wait(&drain, 0);
    } else {
        // ------------------------------------------------ epilogue: 4 warps, one landmark row per thread
        const int quarter = warp & 3;                     // TMEM lanes [32*quarter, +32)
        const int row = quarter * 32 + lane;
        const int ew = warp - 2;
        float m[G], sx[G];
#pragma unroll
        for (int g = 0; g < G; ++g) { m[g] = -CUDART_INF_F; sx[g] = 0.f; }
        for (int it = 0;; ++it) {
            const int b = it & 1;
            if (!mbar_wait(&accf[b], (it >> 1) & 1)) {
                set_err(p.err, DEV_ERR_TIMEOUT, 115);
                s_abort = 1;
                break;
            }
            const ScTile t = atile[b];
            if (t.run < 0) break;
            tc_fence_after();
            float v[8];
            tmem_ld8(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + b * kScN, v);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);
            if (row < t.nv) {
                float z[G];
#pragma unroll
                for (int g = 0; g < G; ++g) z[g] = v[g] * p.scale;
                float* dst = p.logits + (t.j + row) * G;
                if constexpr (G == 4) {
                    *reinterpret_cast<float4*>(dst) = make_float4(z[0], z[1], z[2], z[3]);
                } else {
#pragma unroll
                    for (int g = 0; g < G; ++g) dst[g] = z[g];
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    if (z[g] > m[g]) {
                        sx[g] = sx[g] * __expf(m[g] - z[g]) + 1.f;
                        m[g] = z[g];
                    } else {
                        sx[g] += __expf(z[g] - m[g]);
                    }
                }
            }
            if (t.last) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float M = warp_max(m[g]);
                    const float tt = (m[g] == -CUDART_INF_F) ? 0.f : sx[g] * __expf(m[g] - M);
                    const float S = warp_sum(tt);
                    if (lane == 0) p.part[(static_cast<int64_t>(t.run) * kScParts + ew) * G + g] = make_float2(M, S);
                    m[g] = -CUDART_INF_F;
                    sx[g] = 0.f;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 32);
    }
}

// ------------------------------------------------------------------ e5m2 landmarks (fp8 configuration)
// The same persistent pipeline over landmarks stored in e5m2: 256 landmarks per stage (two
// 128 x 128-byte TMA boxes, two M = 128 MMA halves) and kind::f8f6f4 MMAs (K = 32 per
// instruction).  The bf16 query enters as three e5m2
// terms per head, t1 = e5m2(x), t2 = e5m2(x - t1), t3 = e5m2(x - t1 - t2) of x = q * 2^s
// with 2^s the largest power of two keeping max|x| <= 2^14: each term carries the next three
// significant bits, so t1 + t2 + t3 = x exactly for every component down to max|q| * 2^-22,
// and the epilogue's (col_g + col_{G+g} + col_{2G+g}) * 2^-s is the bf16-query score.
struct ScTile8 {
    int run, nv;
    int64_t j;
    int unit, last;
    float inv[8];   // 2^-s of each head's query
};

template <int G>
__global__ void __launch_bounds__(320, 1) k_score_f8(const __grid_constant__ CUtensorMap tmL, ScoreParams p) {
    constexpr int NQ = (3 * G <= 16) ? 16 : 32;   // MMA N: the 3G term rows, padded
    constexpr int kQBytes = NQ * 128;
    constexpr int kT8 = 2 * kScTile;              // 256 landmarks per stage: two M = 128 halves
    constexpr int kStage = 32768 + kQBytes;
    constexpr int S = kScStages8;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[S], empty[S], accf[2], acce[2], drain;
    __shared__ ScTile8 stile[S], atile[2];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n_c = p.n_c;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int b = 0; b < 2; ++b) { mbar_init(&accf[b], 2); mbar_init(&acce[b], kScParts8); }
        mbar_init(&drain, 1);
        s_abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmL);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_slot, 4 * NQ);   // 2 buffers x 2 halves
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        // ------------------------------------------------ producer warp
        const uint64_t pol = l2_evict_first();   // read once per step
        int it = 0;
        int next = (lane == 0) ? atomicAdd(p.sched, 1) : 0;
        next = __shfl_sync(0xffffffffu, next, 0);
        bool done = false;
        while (!done) {
            const int r = s_abort ? p.total_runs : next;
            int64_t a = 0, e = 0;
            int u = 0;
            if (r < p.total_runs) {
                u = r / p.nru;
                a = static_cast<int64_t>(u) * n_c + static_cast<int64_t>(r % p.nru) * kRunChunks;
                e = min(a + kRunChunks, static_cast<int64_t>(u + 1) * n_c);
                int nx = (lane == 0) ? atomicAdd(p.sched, 1) : 0;   // claim the next run early
                next = __shfl_sync(0xffffffffu, nx, 0);
            } else {
                done = true;
            }
            // the run's query terms (formed once per step by k_qsplit): rows n = jt*G + g of
            // [3G][128 B]; lane l holds 16-byte words l, l + 32, ... and the heads' 2^-s
            constexpr int QW8 = (3 * G * 8 + 31) / 32;
            uint4 tq[QW8];
#pragma unroll
            for (int w = 0; w < QW8; ++w) {
                const int word = lane + 32 * w;
                tq[w] = make_uint4(0, 0, 0, 0);
                if (!done && word < 3 * G * 8) tq[w] = reinterpret_cast<const uint4*>(p.qt + static_cast<int64_t>(u) * 3 * G * 128)[word];
            }
            float inv[G];
#pragma unroll
            for (int g = 0; g < G; ++g) inv[g] = done ? 0.f : p.qinv[u * G + g];
            for (int64_t j = a; done || j < e; j += kT8, ++it) {
                const int s = it % S;
                uint8_t* st = smem + s * kStage;
                const int okw = mbar_wait(&empty[s], ((it / S) & 1) ^ 1) ? 1 : 0;
                if (!__all_sync(0xffffffffu, okw)) {
                    if (lane == 0) set_err(p.err, DEV_ERR_TIMEOUT, 131);
                    s_abort = 1;
                    done = true;
                }
                if (done) {   // end marker: a plain arrival completes the stage's phase
                    if (lane == 0) {
                        stile[s].run = -1;
                        mbar_arrive(&full[s]);
                    }
                    ++it;
                    break;
                }
                // term rows of the [NQ rows][128 B] swizzled query tile
                uint8_t* sq = st + 32768;
#pragma unroll
                for (int w = 0; w < QW8; ++w) {
                    const int word = lane + 32 * w, n = word >> 3, c = word & 7;
                    if (word < 3 * G * 8)
                        *reinterpret_cast<uint4*>(sq + (n >> 3) * 1024 + (n & 7) * 128 + ((c ^ (n & 7)) << 4)) = tq[w];
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ScTile8 t;
                    t.run = r;
                    t.j = j;
                    t.nv = static_cast<int>(min(static_cast<int64_t>(kT8), e - j));
                    t.unit = u;
                    t.last = (j + kT8 >= e);
#pragma unroll
                    for (int g = 0; g < 8; ++g) t.inv[g] = g < G ? inv[g] : 0.f;
                    stile[s] = t;
                    // rows past the tensor's end read as zeros; rows past the run are never scored
                    mbar_arrive_expect_tx(&full[s], 32768);
                    tma_load_2d_hint(st, &tmL, 0, static_cast<int>(j), &full[s], pol);
                    tma_load_2d_hint(st + 16384, &tmL, 0, static_cast<int>(j + kScTile), &full[s], pol);
                }
                __syncwarp();
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_e5m2_f32(kScTile, NQ);
        int it = 0;
        while (true) {
            const int s = it % S, b = it & 1;
            int ok = mbar_wait(&full[s], (it / S) & 1) ? 1 : 0;
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) { if (lane == 0) set_err(p.err, DEV_ERR_TIMEOUT, 132); s_abort = 1; break; }
            const ScTile8 t = stile[s];
            if (lane == 0) ok = mbar_wait(&acce[b], ((it >> 1) & 1) ^ 1) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) { if (lane == 0) set_err(p.err, DEV_ERR_TIMEOUT, 133); s_abort = 1; break; }
            if (t.run < 0) {
                if (lane == 0) { atile[b] = t; mbar_arrive_cnt(&accf[b], 2); }
                break;
            }
            if (lane == 0) {
                tc_fence_after();
                const uint8_t* st = smem + s * kStage;
                for (int h = 0; h < 2; ++h)
                    for (int k = 0; k < 4; ++k) {   // K = 128 bytes = 4 x 32 e5m2 values
                        const uint64_t ad = smem_desc_sw128(smem_u32(st + h * 16384 + k * 32));
                        const uint64_t bd = smem_desc_sw128(smem_u32(st + 32768 + k * 32));
                        tc_mma_f8(tmem + (2 * b + h) * NQ, ad, bd, idesc, k > 0 ? 1u : 0u);
                    }
                tc_commit(&empty[s]);
                tc_commit(&accf[b]);
                atile[b] = t;
                mbar_arrive(&accf[b]);   // release: the record is visible once the phase completes
            }
            __syncwarp();
            ++it;
        }
        if (lane == 0) tc_commit(&drain);
        __syncwarp();
        (void)mbar_wait(&drain, 0);
    } else {
        // ------------------------------------------------ epilogue: 8 warps, warp (h, quarter) scores
        // row 32*quarter + lane of half h of every stage
        const int quarter = warp & 3;                     // TMEM lanes [32*quarter, +32)
        const int ew = warp - 2;                          // 0..7
        const int h = ew >> 2;
        const int rr = h * kScTile + quarter * 32 + lane;
        float m[G], sx[G];
#pragma unroll
        for (int g = 0; g < G; ++g) { m[g] = -CUDART_INF_F; sx[g] = 0.f; }
        for (int it = 0;; ++it) {
            const int b = it & 1;
            if (!mbar_wait(&accf[b], (it >> 1) & 1)) {
                set_err(p.err, DEV_ERR_TIMEOUT, 135);
                s_abort = 1;
                break;
            }
            const ScTile8 t = atile[b];
            if (t.run < 0) break;
            tc_fence_after();
            constexpr int NC8 = (3 * G + 7) / 8;
            float v[NC8 * 8];
#pragma unroll
            for (int c8 = 0; c8 < NC8; ++c8) {
                float w[8];
                tmem_ld8(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + (2 * b + h) * NQ + 8 * c8, w);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) v[8 * c8 + kk] = w[kk];
            }
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);
            if (rr < t.nv) {
                float z[G];
#pragma unroll
                for (int g = 0; g < G; ++g) z[g] = (v[g] + v[G + g] + v[2 * G + g]) * t.inv[g] * p.scale;
                float* dst = p.logits + (t.j + rr) * G;
                if constexpr (G == 4) {
                    *reinterpret_cast<float4*>(dst) = make_float4(z[0], z[1], z[2], z[3]);
                } else {
#pragma unroll
                    for (int g = 0; g < G; ++g) dst[g] = z[g];
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    if (z[g] > m[g]) {
                        sx[g] = sx[g] * __expf(m[g] - z[g]) + 1.f;
                        m[g] = z[g];
                    } else {
                        sx[g] += __expf(z[g] - m[g]);
                    }
                }
            }
            if (t.last) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float M = warp_max(m[g]);
                    const float tt = (m[g] == -CUDART_INF_F) ? 0.f : sx[g] * __expf(m[g] - M);
                    const float Ssum = warp_sum(tt);
                    if (lane == 0) p.part[(static_cast<int64_t>(t.run) * kScParts8 + ew) * G + g] = make_float2(M, Ssum);
                    m[g] = -CUDART_INF_F;
                    sx[g] = 0.f;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 4 * NQ);
    }
}

// The query terms of the e5m2 scorer, once per step: block u, warp g = head, lane l = dims
// [4l, 4l + 4).  Per head the largest |q| over the 128 dimensions sets 2^s (largest power of two
// with max|q| * 2^s < 2^14), then x = q * 2^s gives t1 = e5m2(x), t2 = e5m2(x - t1),
// t3 = e5m2(x - t1 - t2) into rows jt*G + g of qt[u], and qinv[u][g] = 2^-s.
template <int G>
__global__ void __launch_bounds__(32 * G) k_qsplit(const __nv_bfloat16* __restrict__ q, uint8_t* __restrict__ qt,
                                                   float* __restrict__ qinv) {
    pdl_wait();
    pdl_trigger();
    const int u = blockIdx.x, g = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint2 raw = reinterpret_cast<const uint2*>(q + (static_cast<int64_t>(u) * G + g) * kD)[lane];
    const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
    float x[4];
    const float2 a = __bfloat1622float2(q2[0]), c = __bfloat1622float2(q2[1]);
    x[0] = a.x; x[1] = a.y; x[2] = c.x; x[3] = c.y;
    const float mx = warp_max(fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3]))));
    int sh = 0;
    if (mx > 0.f) {
        int ex;
        frexpf(mx, &ex);   // mx in [2^(ex-1), 2^ex)
        sh = max(-100, min(100, 14 - ex));
    }
    const float up = ldexpf(1.f, sh);
    uint32_t word[3] = {0u, 0u, 0u};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float r = x[e] * up;
#pragma unroll
        for (int jt = 0; jt < 3; ++jt) {
            const uint32_t b8 = from_f<__nv_fp8_e5m2>(r).__x & 0xffu;
            word[jt] |= b8 << (8 * e);
            r -= e5m2_to_f(b8);
        }
    }
    uint8_t* row = qt + static_cast<int64_t>(u) * 3 * G * kD;
#pragma unroll
    for (int jt = 0; jt < 3; ++jt) reinterpret_cast<uint32_t*>(row + (jt * G + g) * kD)[lane] = word[jt];
    if (lane == 0) qinv[u * G + g] = ldexpf(1.f, -sh);
}

int launch_qsplit(const void* q, void* qt, float* qinv, int U, int G, cudaStream_t s) {
    auto q16 = static_cast<const __nv_bfloat16*>(q);
    auto qt8 = static_cast<uint8_t*>(qt);
    cudaError_t e = cudaErrorInvalidValue;
    switch (G) {
        case 1: e = launch_pdl(k_qsplit<1>, dim3(U), dim3(32), 0, s, q16, qt8, qinv); break;
        case 2: e = launch_pdl(k_qsplit<2>, dim3(U), dim3(64), 0, s, q16, qt8, qinv); break;
        case 4: e = launch_pdl(k_qsplit<4>, dim3(U), dim3(128), 0, s, q16, qt8, qinv); break;
        case 8: e = launch_pdl(k_qsplit<8>, dim3(U), dim3(256), 0, s, q16, qt8, qinv); break;
        default: return -1;
    }
    if (e != cudaSuccess) { cudaGetLastError(); return -1; }
    return 0;
}

template <int G>
static int launch_f8(const CUtensorMap* tmL, const ScoreParams& p, int ncta, cudaStream_t s) {
    constexpr int NQ = (3 * G <= 16) ? 16 : 32;
    const int smem = kScStages8 * (32768 + NQ * 128) + 1024;
    cudaFuncSetAttribute(k_score_f8<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (launch_pdl(k_score_f8<G>, dim3(ncta), dim3(320), smem, s, *tmL, p) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return 0;
}

template <int G>
static int launch_tc(const CUtensorMap* tmL, const ScoreParams& p, int ncta, cudaStream_t s) {
    const int smem = kScStages * (32768 + 4096) + 1024;
    cudaFuncSetAttribute(k_score_tc<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (launch_pdl(k_score_tc<G>, dim3(ncta), dim3(192), smem, s, *tmL, p) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return 0;
}

template <typename T, int G>
static int launch_t(const ScoreParams& p, int ncta, cudaStream_t s) {
    const int smem = kScoreStages * kScoreStageBytes;
    cudaFuncSetAttribute(k_score<T, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    k_score<T, G><<<ncta, (kScoreWarps + 1) * 32, smem, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

template <typename T, int G>
static int occ_t() {
    const int smem = kScoreStages * kScoreStageBytes;
    cudaFuncSetAttribute(k_score<T, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_score<T, G>, (kScoreWarps + 1) * 32, smem) !=
        cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}

#define SKV_G_DISPATCH(G, CALL)                    \
    switch (G) {                                   \
        case 1: return CALL(1);                    \
        case 2: return CALL(2);                    \
        case 4: return CALL(4);                    \
        case 8: return CALL(8);                    \
        default: return -1;                        \
    }

int launch_score(int dtype, int G, const CUtensorMap* tmL, const ScoreParams& p, int ncta, cudaStream_t s) {
    if (dtype == 2) {
#define CALL8(g) launch_f8<g>(tmL, p, ncta, s)
        SKV_G_DISPATCH(G, CALL8)
#undef CALL8
    }
    if (dtype == 1) {
#define CALLB(g) launch_tc<g>(tmL, p, ncta, s)
        SKV_G_DISPATCH(G, CALLB)
#undef CALLB
    } else {
#define CALLF(g) launch_t<float, g>(p, ncta, s)
        SKV_G_DISPATCH(G, CALLF)
#undef CALLF
    }
}

int score_parts(int dtype) { return dtype == 2 ? kScParts8 : dtype != 0 ? kScParts : kScoreWarps; }

int score_ctas_per_sm(int dtype, int G) {
    if (dtype != 0) {
        (void)G;
        return 1;   // the tensor-core kernels hold most of the shared memory
    } else {
#define OCCF(g) occ_t<float, g>()
        SKV_G_DISPATCH(G, OCCF)
#undef OCCF
    }
}

}  // namespace skv
