// Value fetch and pre-filling gathers.
//
// ShadowKV (English summary, section 3.4, "Fetching values from the CPU": for
// each missed chunk the C value rows are transferred into the GPU cache;
// Chinese digest section A2, Algorithm 2: V_sparse = Gather(V_CPU, I)).  With
// values in page-locked Grace memory the GPU reads them in place over
// NVLink-C2C, on its own stream so that the transfer overlaps the key rebuild.
// A host read has a long latency, so bandwidth needs every missed chunk in
// flight at once: the decode step's k_gather2 gives each warp two chunks (2 KB
// each in bf16, all 16-byte loads of both issued before the first store), a
// grid covering every possible miss, no shared memory, and half the warps and
// registers that one chunk per warp would hold, so the rebuild's CTAs fit
// beside it (measured: 1045-1060 against 977-1033 tokens/s at 128K b8).  The
// pre-filling gathers use k_gather, one chunk per warp.
// The same kernel gathers the outlier chunks' and the local window's values
// during pre-filling (Algorithm 1: K_outlier, V_outlier = Gather(K_RoPE, V, I)).
//
// Pre-filling compaction: L = C \ Gather(C, I) (Algorithm 1, last line).  The
// landmark of candidate chunk j lands at position j - #{outliers < j}.
#include "skv_common.cuh"
#include "skv_internal.h"

namespace skv {

__global__ void __launch_bounds__(256) k_gather(GatherParams p) {
    const int u = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int idx = blockIdx.x * 8 + warp;
    int count = p.cnt ? p.cnt[u] : p.count_const;
    if (count < 0 || count > p.list_cap) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_err(p.err, DEV_ERR_BOUNDS, 501);
        return;
    }
    if (idx >= count) return;
    const int ch = p.list ? p.list[u * p.list_us + idx] : p.list_base + idx;
    const int dst = p.dst_idx ? p.dst_idx[u * p.list_us + idx] : idx;
    if (ch < 0 || ch >= p.nchunk || dst < 0 || dst >= p.dst_cap) {
        if (lane == 0) set_err(p.err, DEV_ERR_BOUNDS, 502);
        return;
    }
    const int64_t rowbytes = static_cast<int64_t>(kD) * p.es;
    const uint8_t* src = static_cast<const uint8_t*>(p.src) + (u * p.src_us + static_cast<int64_t>(ch) * kC * kD) * p.es;
    uint8_t* d = static_cast<uint8_t*>(p.dst) + (u * p.dst_us + static_cast<int64_t>(dst) * kC * kD) * p.es;
    const int n16 = static_cast<int>(kC * rowbytes / 16);   // 128 (bf16) or 256 (fp32) words
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(d);
    // issue every load of the chunk before the first store (bytes in flight)
    if (n16 == 128) {
        uint4 w0 = s4[lane], w1 = s4[lane + 32], w2 = s4[lane + 64], w3 = s4[lane + 96];
        d4[lane] = w0; d4[lane + 32] = w1; d4[lane + 64] = w2; d4[lane + 96] = w3;
    } else {
        for (int i = lane; i < n16; i += 32) d4[i] = s4[i];
    }
}

// The decode step's fetch with two chunks per warp: the same bytes in flight as one chunk per
// warp, from half the warps, so that the key rebuild's CTAs fit beside it on every SM.
template <int PER>   // 16-byte words per lane and chunk: 2 (e5m2), 4 (bf16), 8 (fp32)
__global__ void __launch_bounds__(256) k_gather2(GatherParams p) {
    const int u = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int idx0 = (blockIdx.x * 8 + warp) * 2;
    int count = p.cnt[u];
    if (count < 0 || count > p.list_cap) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_err(p.err, DEV_ERR_BOUNDS, 505);
        return;
    }
    if (idx0 >= count) return;
    const int n = min(2, count - idx0);
    const uint4* s4[2];
    uint4* d4[2];
    for (int c = 0; c < 2; ++c) {
        const int idx = idx0 + (c < n ? c : 0);
        const int ch = p.list[u * p.list_us + idx];
        const int dst = p.dst_idx[u * p.list_us + idx];
        if (ch < 0 || ch >= p.nchunk || dst < 0 || dst >= p.dst_cap) {
            if (lane == 0) set_err(p.err, DEV_ERR_BOUNDS, 506);
            return;
        }
        s4[c] = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.src) +
                                               (u * p.src_us + static_cast<int64_t>(ch) * kC * kD) * p.es);
        d4[c] = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.dst) +
                                         (u * p.dst_us + static_cast<int64_t>(dst) * kC * kD) * p.es);
    }
    uint4 v[2][PER];
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int k = 0; k < PER; ++k)
            if (c < n) v[c][k] = s4[c][lane + 32 * k];
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int k = 0; k < PER; ++k)
            if (c < n) d4[c][lane + 32 * k] = v[c][k];
}

int launch_fetch2(const GatherParams& p, int list_cap, cudaStream_t s) {
    if (!p.cnt || !p.list || !p.dst_idx || (p.es != 1 && p.es != 2 && p.es != 4)) return -1;
    const dim3 grid((list_cap + 15) / 16, p.U);
    if (p.es == 1) k_gather2<2><<<grid, 256, 0, s>>>(p);
    else if (p.es == 2) k_gather2<4><<<grid, 256, 0, s>>>(p);
    else k_gather2<8><<<grid, 256, 0, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_gather(const GatherParams& p, int grid_x, cudaStream_t s) {
    if (grid_x <= 0) return 0;
    k_gather<<<dim3(grid_x, p.U), 256, 0, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

template <typename T>
__global__ void __launch_bounds__(256) k_compact(CompactParams p) {
    const int u = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * 8 + warp;
    if (j >= p.ncand) return;
    const int32_t* oi = p.out_ids + static_cast<int64_t>(u) * p.O;
    int lo = 0, hi = p.O;   // outliers below j
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (oi[mid] < j) lo = mid + 1; else hi = mid;
    }
    if (lo < p.O && oi[lo] == j) return;
    const int64_t pos = j - lo;
    if (pos < 0 || pos >= p.n_c) {
        if (lane == 0) set_err(p.err, DEV_ERR_BOUNDS, 511);
        return;
    }
    if (lane == 0) p.ids[static_cast<int64_t>(u) * p.n_c + pos] = static_cast<int32_t>(j);
    const float* src = p.Lfull + (static_cast<int64_t>(u) * p.ncand + j) * kD;
    T* dst = static_cast<T*>(p.L) + (static_cast<int64_t>(u) * p.n_c + pos) * kD;
    for (int k = lane; k < kD; k += 32) dst[k] = from_f<T>(src[k]);
}

int launch_compact(const CompactParams& p, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>((p.ncand + 7) / 8), p.U);
    if (p.dtype == 1) k_compact<__nv_bfloat16><<<grid, 256, 0, s>>>(p);
    else if (p.dtype == 2) k_compact<__nv_fp8_e5m2><<<grid, 256, 0, s>>>(p);   // e5m2 landmarks
    else k_compact<float><<<grid, 256, 0, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace skv

// ---------------------------------------------------------------------------
// Measurement aid: the decode step's fetch kernel on a random chunk list.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "shadowkv.h"

extern "C" int shadowkv_fetch_probe(const void* src, size_t bytes, int64_t n_chunks, int chunk_bytes, uint64_t seed,
                                    int reps, int fresh, skv_stream stream, double* gbs_out) {
    using namespace skv;
    if (!src || !gbs_out || reps < 1 || n_chunks < 1 || n_chunks > (int64_t(1) << 24)) return SKV_ERR_INVALID;
    if (chunk_bytes != 1024 && chunk_bytes != 2048 && chunk_bytes != 4096) return SKV_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(src) & 15) return SKV_ERR_INVALID;
    const int64_t slots = static_cast<int64_t>(bytes / static_cast<size_t>(chunk_bytes));
    if (slots < 2 * n_chunks || slots > INT32_MAX) return SKV_ERR_INVALID;
    *gbs_out = 0.0;
    // distinct random chunk positions (splitmix64 stream), ascending: the decode step's address order
    uint64_t x = seed;
    auto next = [&x]() {
        uint64_t z = (x += 0x9E3779B97F4A7C15ull);
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        return z ^ (z >> 31);
    };
    const int32_t n = static_cast<int32_t>(n_chunks);
    auto draw = [&](std::vector<int32_t>& ids) {
        ids.clear();
        while (static_cast<int64_t>(ids.size()) < n_chunks) {
            const size_t need = static_cast<size_t>(n_chunks) - ids.size();
            for (size_t i = 0; i < need; ++i) ids.push_back(static_cast<int32_t>(next() % static_cast<uint64_t>(slots)));
            std::sort(ids.begin(), ids.end());
            ids.erase(std::unique(ids.begin(), ids.end()), ids.end());
        }
    };
    std::vector<int32_t> ids, dst_idx(static_cast<size_t>(n));
    for (int32_t i = 0; i < n; ++i) dst_idx[i] = i;
    draw(ids);
    int32_t *d_ids = nullptr, *d_dst = nullptr, *d_cnt = nullptr;
    int* d_err = nullptr;
    void* d_out = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    int rc = SKV_OK;
    if (cudaMalloc(&d_ids, n * sizeof(int32_t)) != cudaSuccess || cudaMalloc(&d_dst, n * sizeof(int32_t)) != cudaSuccess ||
        cudaMalloc(&d_cnt, sizeof(int32_t)) != cudaSuccess || cudaMalloc(&d_err, 4 * sizeof(int)) != cudaSuccess ||
        cudaMalloc(&d_out, static_cast<size_t>(n) * chunk_bytes) != cudaSuccess) {
        rc = SKV_ERR_OOM;
    } else if (cudaMemcpy(d_ids, ids.data(), n * sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess ||
               cudaMemcpy(d_dst, dst_idx.data(), n * sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess ||
               cudaMemcpy(d_cnt, &n, sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess ||
               cudaMemset(d_err, 0, 4 * sizeof(int)) != cudaSuccess ||
               cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        rc = SKV_ERR_CUDA;
    } else {
        GatherParams g{};
        g.src = src; g.src_us = 0; g.list = d_ids; g.list_us = n; g.list_cap = n; g.cnt = d_cnt;
        g.dst_idx = d_dst; g.dst_cap = n; g.dst = d_out; g.dst_us = 0; g.nchunk = static_cast<int>(slots);
        g.es = chunk_bytes / (kC * kD); g.U = 1; g.err = d_err;
        float best = 0.f;
        for (int r = 0; r <= reps && rc == SKV_OK; ++r) {
            if (fresh && r > 0) {
                draw(ids);
                if (cudaMemcpy(d_ids, ids.data(), n * sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess) {
                    rc = SKV_ERR_CUDA;
                    break;
                }
            }
            if (cudaEventRecord(e0, stream) != cudaSuccess || launch_fetch2(g, n, stream) ||
                cudaEventRecord(e1, stream) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess) {
                rc = SKV_ERR_CUDA;
                break;
            }
            float ms = 0.f;
            cudaEventElapsedTime(&ms, e0, e1);
            if (r > 0 && (best == 0.f || ms < best)) best = ms;   // the first run is a warm-up
        }
        int e[2] = {0, 0};
        if (rc == SKV_OK && cudaMemcpy(e, d_err, sizeof(e), cudaMemcpyDeviceToHost) != cudaSuccess) rc = SKV_ERR_CUDA;
        if (rc == SKV_OK && e[0] != 0) rc = SKV_ERR_DEVICE_BOUNDS;
        if (rc == SKV_OK && best > 0.f) *gbs_out = static_cast<double>(n) * chunk_bytes / (best * 1e-3) / 1e9;
    }
    if (stream) cudaStreamSynchronize(stream);
    cudaFree(d_ids); cudaFree(d_dst); cudaFree(d_cnt); cudaFree(d_err); cudaFree(d_out);
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    cudaGetLastError();
    return rc;
}
