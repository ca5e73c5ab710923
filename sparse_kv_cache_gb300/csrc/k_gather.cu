// Value fetch and pre-filling gathers.
//
// ShadowKV (English summary, section 3.4, "Fetching values from the CPU": for
// each missed chunk the C value rows are transferred into the GPU cache;
// Chinese digest section A2, Algorithm 2: V_sparse = Gather(V_CPU, I)).  With
// values in page-locked Grace memory the GPU reads them in place over
// NVLink-C2C, on its own stream so that the transfer overlaps the key rebuild.
// A host read has a long latency, so bandwidth needs every missed chunk in
// flight at once: one warp per chunk (2 KB in bf16, four 16-byte loads per
// lane issued before the first store), a grid covering every possible miss,
// no shared memory and few registers, so the rebuild's CTAs fit beside it.
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
