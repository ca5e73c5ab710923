// Landmark scoring, P = q . L^T for the G query heads of each KV head.
//
// ShadowKV (Chinese digest, section A2, Algorithm 2: P = MatMul(Q, L.T),
// S = Softmax(P / sqrt(d))); English summary section 3.4, "Decoding-Time KV
// Selection", Step 1.  This is the largest HBM stream of a decode step: every
// selectable landmark row (d bf16 values) is read once per step.
//
// Design: one warp (the producer) streams landmark tiles of 32 KB into a
// three-stage shared-memory ring with 1-D bulk copies (the TMA engine), eight
// consumer warps read them.  Each half-warp owns one landmark row at a time;
// lane l holds dims [8l, 8l+8) of all G queries in registers, so a row costs
// 8*G FMAs per lane and one 16-byte shared load, and the 16 partial sums of 8
// rows are combined with a transpose-reduction (8 shuffles for 8 rows).
// Outputs: z = P / sqrt(d) as fp32 [U][n_c][G], and per (CTA, unit, warp, g)
// the running (max z, sum exp(z - max)) so the next kernel can form the
// log-sum-exp of every query head without re-reading z twice.
// The flat chunk range U*n_c is split evenly over at most (SMs x resident
// CTAs) CTAs, so every CTA is resident in one wave.
#include <math_constants.h>

#include "skv_common.cuh"
#include "skv_internal.h"

namespace skv {

template <typename T, int G>
__global__ void __launch_bounds__((kScoreWarps + 1) * 32) k_score(ScoreParams p) {
    constexpr int ROWB = kD * Elem<T>::bytes;
    constexpr int TILE = kScoreStageBytes / ROWB;
    static_assert(TILE <= kScoreWarps * 16, "tile larger than one pass of the consumer warps");
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t full[kScoreStages], empty[kScoreStages];
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * p.per;
    const int64_t c1 = min(c0 + p.per, p.total);
    if (tid == 0) {
        for (int s = 0; s < kScoreStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kScoreWarps);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (c0 >= c1) return;
    const int64_t n_c = p.n_c;

    if (warp == kScoreWarps) {
        // ------------------------------------------------ producer (one lane)
        if (lane != 0) return;
        int it = 0;
        bool ok = true;
        for (int64_t pos = c0; ok && pos < c1;) {
            const int64_t u = pos / n_c;
            const int64_t uend = min(c1, (u + 1) * n_c);
            for (int64_t j = pos; j < uend; j += TILE, ++it) {
                const int nv = static_cast<int>(min(static_cast<int64_t>(TILE), uend - j));
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
            pos = uend;
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
    int it = 0, slot = 0;
    bool ok = true;
    for (int64_t pos = c0; pos < c1; ++slot) {
        const int64_t u = pos / n_c;
        const int64_t uend = min(c1, (u + 1) * n_c);
#pragma unroll
        for (int g = 0; g < G; ++g) load8(static_cast<const T*>(p.q) + (u * G + g) * kD + hl * 8, qv[g]);
        float m[G], sx[G];
#pragma unroll
        for (int g = 0; g < G; ++g) { m[g] = -CUDART_INF_F; sx[g] = 0.f; }

        for (int64_t j = pos; ok && j < uend; j += TILE, ++it) {
            const int nv = static_cast<int>(min(static_cast<int64_t>(TILE), uend - j));
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
                        float a = 0.f;
#pragma unroll
                        for (int k = 0; k < 8; ++k) a = fmaf(qv[g][k], v[k], a);
                        acc[g][c] = a;
                    }
                }
                float z[G];
#pragma unroll
                for (int g = 0; g < G; ++g) z[g] = transpose_reduce8(acc[g], hl) * p.scale;
                const int cj = cb + (hl >> 1);
                if ((hl & 1) == 0 && cj < nv) {
                    float* dst = p.logits + (j + cj) * G;
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
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        // merge the lanes' (max, sum) and publish this warp's record for unit u
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float M = warp_max(m[g]);
            const float t = (m[g] == -CUDART_INF_F) ? 0.f : sx[g] * __expf(m[g] - M);
            const float S = warp_sum(t);
            if (lane == 0)
                p.part[((static_cast<int64_t>(blockIdx.x) * p.slots + slot) * kScoreWarps + warp) * G + g] =
                    make_float2(M, S);
        }
        pos = uend;
        if (!ok) break;
    }
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

int launch_score(int dtype, int G, const ScoreParams& p, int ncta, cudaStream_t s) {
    if (dtype == 1) {
#define CALLB(g) launch_t<__nv_bfloat16, g>(p, ncta, s)
        SKV_G_DISPATCH(G, CALLB)
#undef CALLB
    } else {
#define CALLF(g) launch_t<float, g>(p, ncta, s)
        SKV_G_DISPATCH(G, CALLF)
#undef CALLF
    }
}

int score_ctas_per_sm(int dtype, int G) {
    if (dtype == 1) {
#define OCCB(g) occ_t<__nv_bfloat16, g>()
        SKV_G_DISPATCH(G, OCCB)
#undef OCCB
    } else {
#define OCCF(g) occ_t<float, g>()
        SKV_G_DISPATCH(G, OCCF)
#undef OCCF
    }
}

}  // namespace skv
