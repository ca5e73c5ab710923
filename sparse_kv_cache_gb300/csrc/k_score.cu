// Landmark scoring, P = q . L^T for the G query heads of each KV head.
//
// ShadowKV (Chinese digest, section A2, Algorithm 2: P = MatMul(Q, L.T),
// S = Softmax(P / sqrt(d))); English summary section 3.4, "Decoding-Time KV
// Selection", Step 1.  This is the largest HBM stream of a decode step: every
// selectable landmark row (d values) is read once per step.
//
// bf16 storage (k_score_tc): the contraction runs on the 5th-generation tensor
// cores so that the kernel is bound by the landmark stream alone.  Per CTA one
// warp streams 128-landmark tiles (two 64-column, 128-byte-swizzled boxes,
// 32 KB) with 2-D TMA copies into a 6-stage shared-memory ring; one thread
// issues tcgen05 MMAs, M = 128 landmarks x N = 16 (the unit's G <= 8 queries,
// zero-padded) x K = 128, into a double-buffered fp32 accumulator in tensor
// memory; four epilogue warps read one landmark row each per thread, scale by
// 1/sqrt(d), store z and keep the running (max, sum exp) per query head.
// fp32 storage (k_score): CUDA-core dot products, the query in registers, one
// half-warp per landmark row and a transpose-reduction of the partial sums.
// Outputs: z = P / sqrt(d) as fp32 [U][n_c][G], and per (CTA, unit, part, g)
// the running (max z, sum exp(z - max)) so the next kernel can form the
// log-sum-exp of every query head.  The flat chunk range U*n_c is split evenly
// over at most (SMs x resident CTAs) CTAs, so every CTA is resident at once.
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
                p.part[((static_cast<int64_t>(blockIdx.x) * p.slots + slot) * p.nparts + warp) * G + g] =
                    make_float2(M, S);
        }
        pos = uend;
        if (!ok) break;
    }
}

// ------------------------------------------------------------------ tensor-core path
template <int G>
__global__ void __launch_bounds__(192, 1) k_score_tc(const __grid_constant__ CUtensorMap tmL, ScoreParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sL = smem;                                  // kScStages x (2 x [128 rows][128 B])
    uint8_t* sQ = smem + kScStages * 32768;              // 2 x [16 rows][128 B]
    __shared__ uint64_t full[kScStages], empty[kScStages], accf[2], acce[2], qdone;
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * p.per;
    const int64_t c1 = min(c0 + p.per, p.total);
    if (c0 >= c1) return;   // uniform
    const int64_t n_c = p.n_c;
    if (tid == 0) {
        for (int s = 0; s < kScStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int b = 0; b < 2; ++b) { mbar_init(&accf[b], 1); mbar_init(&acce[b], 4); }
        mbar_init(&qdone, 1);
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

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int it = 0;
            for (int64_t pos = c0; pos < c1 && !s_abort;) {
                const int64_t u = pos / n_c, uend = min(c1, (u + 1) * n_c);
                for (int64_t j = pos; j < uend; j += kScTile, ++it) {
                    const int s = it % kScStages;
                    if (!mbar_wait(&empty[s], ((it / kScStages) & 1) ^ 1)) {
                        set_err(p.err, DEV_ERR_TIMEOUT, 111);
                        s_abort = 1;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], 32768);
                    tma_load_2d(sL + s * 32768, &tmL, 0, static_cast<int>(j), &full[s]);
                    tma_load_2d(sL + s * 32768 + 16384, &tmL, 64, static_cast<int>(j), &full[s]);
                }
                pos = uend;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (whole warp writes the query tile)
        constexpr uint32_t idesc = idesc_bf16_f32(kScTile, kScN);
        int it = 0, qphase = 0;
        bool first = true;
        for (int64_t pos = c0; pos < c1 && !s_abort;) {
            const int64_t u = pos / n_c, uend = min(c1, (u + 1) * n_c);
            // the unit's queries as the B operand: rows g < G, zero rows up to 16
            if (!first) {
                if (lane == 0) tc_commit(&qdone);
                __syncwarp();
                if (!mbar_wait(&qdone, qphase & 1)) { set_err(p.err, DEV_ERR_TIMEOUT, 112); s_abort = 1; }
                ++qphase;
            }
            first = false;
            for (int e = lane; e < kScN * 16; e += 32) {
                const int n = e >> 4, c16 = e & 15, kb = c16 >> 3, c = c16 & 7;
                uint4 w = make_uint4(0, 0, 0, 0);
                if (n < G)
                    w = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) +
                                                        (u * G + n) * kD + kb * 64 + c * 8);
                *reinterpret_cast<uint4*>(sQ + kb * 2048 + (n >> 3) * 1024 + (n & 7) * 128 + ((c ^ (n & 7)) << 4)) = w;
            }
            fence_proxy_async_smem();
            __syncwarp();
            for (int64_t j = pos; j < uend; j += kScTile, ++it) {
                const int s = it % kScStages, b = it & 1;
                bool ok = true;
                if (lane == 0) {
                    ok = mbar_wait(&full[s], (it / kScStages) & 1) && mbar_wait(&acce[b], ((it >> 1) & 1) ^ 1);
                    if (ok) {
                        tc_fence_after();
                        uint32_t acc = 0;
                        for (int kb = 0; kb < 2; ++kb)
                            for (int k = 0; k < 4; ++k) {
                                const uint64_t ad = smem_desc_sw128(smem_u32(sL + s * 32768 + kb * 16384 + k * 32));
                                const uint64_t bd = smem_desc_sw128(smem_u32(sQ + kb * 2048 + k * 32));
                                tc_mma_bf16(tmem + b * kScN, ad, bd, idesc, acc);
                                acc = 1;
                            }
                        tc_commit(&empty[s]);
                        tc_commit(&accf[b]);
                    } else {
                        set_err(p.err, DEV_ERR_TIMEOUT, 113);
                        s_abort = 1;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0);
                if (!ok) break;
            }
            pos = uend;
        }
        // every MMA retired before the accumulator is released
        if (lane == 0) tc_commit(&qdone);
        __syncwarp();
        (void)mbar_wait(&qdone, qphase & 1);
    } else {
        // ------------------------------------------------ epilogue: 4 warps, one landmark row per thread
        const int quarter = warp & 3;                     // TMEM lanes [32*quarter, +32)
        const int row = quarter * 32 + lane;
        const int ew = warp - 2;
        int it = 0, slot = 0;
        for (int64_t pos = c0; pos < c1; ++slot) {
            const int64_t u = pos / n_c, uend = min(c1, (u + 1) * n_c);
            float m[G], sx[G];
#pragma unroll
            for (int g = 0; g < G; ++g) { m[g] = -CUDART_INF_F; sx[g] = 0.f; }
            for (int64_t j = pos; j < uend && !s_abort; j += kScTile, ++it) {
                const int b = it & 1;
                const int nv = static_cast<int>(min(static_cast<int64_t>(kScTile), uend - j));
                if (!mbar_wait(&accf[b], (it >> 1) & 1)) {
                    set_err(p.err, DEV_ERR_TIMEOUT, 114);
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                float v[8];
                tmem_ld8(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + b * kScN, v);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acce[b]);
                if (row < nv) {
                    float z[G];
#pragma unroll
                    for (int g = 0; g < G; ++g) z[g] = v[g] * p.scale;
                    float* dst = p.logits + (j + row) * G;
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
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float M = warp_max(m[g]);
                const float t = (m[g] == -CUDART_INF_F) ? 0.f : sx[g] * __expf(m[g] - M);
                const float S = warp_sum(t);
                if (lane == 0)
                    p.part[((static_cast<int64_t>(blockIdx.x) * p.slots + slot) * kScParts + ew) * G + g] =
                        make_float2(M, S);
            }
            pos = uend;
            if (s_abort) break;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 32);
    }
}

template <int G>
static int launch_tc(const CUtensorMap* tmL, const ScoreParams& p, int ncta, cudaStream_t s) {
    const int smem = kScStages * 32768 + 2 * 2048 + 1024;
    cudaFuncSetAttribute(k_score_tc<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    k_score_tc<G><<<ncta, 192, smem, s>>>(*tmL, p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
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

int score_parts(int dtype) { return dtype == 1 ? kScParts : kScoreWarps; }

int score_ctas_per_sm(int dtype, int G) {
    if (dtype == 1) {
        (void)G;
        return 1;   // the tensor-core kernel holds 133 KB of shared memory
    } else {
#define OCCF(g) occ_t<float, g>()
        SKV_G_DISPATCH(G, OCCF)
#undef OCCF
    }
}

}  // namespace skv
