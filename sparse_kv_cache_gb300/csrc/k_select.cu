// Per-KV-head top-K selection, the temporal chunk cache's index scan and the
// append of the new token; and (prefill) the outlier choice.
//
// ShadowKV (Chinese digest, section A2, Algorithm 2): S = Softmax(P/sqrt(d)),
// S1 = sum over query tokens, S2 = max_kv_group(S1), I = ArgTopK(S2, k); the
// decoding text of the same section: an index scan finds the chunks missed
// against the previous step and only those are rebuilt and fetched.  English
// summary section 3.4, Steps 2-3 and "The temporal KV cache mechanism".
// Algorithm 1: I = ArgTopK(-Min(S, dim=-1), o) picks the outliers.
//
// One 1024-thread CTA per (batch, KV head) unit; a unit with more than 16K
// chunks, when SMs are left over, runs on a thread-block cluster of up to 16
// CTAs, each holding a contiguous slice of the unit's scores.  Each CTA
// streams its logits into two 64 KB shared-memory buffers by bulk copies
// issued as soon as the scores are complete, in flight while the log-sum-exp
// forms, so the score pass reads shared memory instead of waiting on L2 round
// trips (22.1 -> 20.9 us per layer at 128K b8; the cluster form at 1M b1:
// 245.7 -> 247.6 tokens/s).  The one-CTA form then brings the unit's position ->
// chunk id table into the first buffer the same way, in flight through the
// threshold and the compaction (2388 -> 2400 tokens/s at 128K b8, values in HBM).  Ordering by
// S2_j = max_g exp(z_gj - lse_g) equals ordering by v_j = max_g (z_gj - lse_g)
// (exp is increasing), so the kernel ranks v_j.  The exact K-th largest value
// T and the last index `jlast` taken among values equal to T are found with a
// 2048-bin histogram over [min v, max v] (monotone binning), then an exact
// rank among the <= 256 candidates of the boundary bin (or, for a crowded bin,
// an exact 4-pass radix select on the order-preserving integer image of the
// floats); the cluster form sums the range, the histogram and the radix
// counts over its CTAs through distributed shared memory.  The selection
// {v > T} U {v == T, j <= jlast} has exactly K members and gives equal scores
// to the lower index; it is written in ascending index order by a ballot-based
// compaction (per-warp counts of every row, one block-wide prefix sum, then each
// taken score goes to its rank).
#include <math_constants.h>

#include <algorithm>

#include "skv_common.cuh"
#include "skv_internal.h"

namespace skv {

constexpr int kBins = 2048;
constexpr int kSelStageBytes = 65536;   // one logits buffer of the staged one-CTA form
constexpr int kCand = 256;
constexpr int kWarps = kSelThreads / 32;

struct SelShared {
    int hist[kBins];
    float cand_v[kCand];
    int cand_j[kCand];
    int ncand;
    float red_f[kWarps];
    float red_f2[kWarps];
    int red_i[kWarps];
    int wpre[kWarps + 1];
    float lse[8];          // one-CTA form: log-sum-exp per query head
    float2 lse_part[16];   // cluster form: (max, sum) of the log-sum-exp per warp of the first 16
    float vmin, vmax, T;
    int jlast, bstar, above, total;
    float cl_lo, cl_hi;   // cluster form: this CTA's score range and counts, read by the others
    int cl_cnt;
};

__device__ __forceinline__ uint32_t ord_key(float x) {
    uint32_t b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
__device__ __forceinline__ int bin_of(float x, float vmin, float invw) {
    int b = static_cast<int>((x - vmin) * invw);
    return b < 0 ? 0 : (b >= kBins ? kBins - 1 : b);
}

// Block-wide exclusive prefix sum of one int per thread; *total gets the sum.
__device__ int block_exscan(int v, SelShared& sh, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh.red_i[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = sh.red_i[lane];
        int s = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        sh.wpre[lane] = s - w;
        if (lane == 31) sh.wpre[kWarps] = s;
    }
    __syncthreads();
    const int r = sh.wpre[warp] + x - v;
    if (total) *total = sh.wpre[kWarps];
    __syncthreads();
    return r;
}

// Sums of the int at `a` (and at `b`) over the first n CTAs of the cluster, the same offset in
// each CTA's shared memory; four ranks' loads are in flight at a time.
__device__ __forceinline__ int cluster_sum(const int* a, int n) {
    int s = 0;
    for (int r0 = 0; r0 < n; r0 += 4) {
        int v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = r0 + i < n ? ld_cluster_s32(cluster_addr(a, r0 + i)) : 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) s += v[i];
    }
    return s;
}
__device__ __forceinline__ void cluster_sum2(const int* a, const int* b, int n, int& sa, int& sb) {
    sa = 0;
    sb = 0;
    for (int r0 = 0; r0 < n; r0 += 4) {
        int va[4], vb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bool on = r0 + i < n;
            va[i] = on ? ld_cluster_s32(cluster_addr(a, r0 + i)) : 0;
            vb[i] = on ? ld_cluster_s32(cluster_addr(b, r0 + i)) : 0;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            sa += va[i];
            sb += vb[i];
        }
    }
}

// Exact threshold of the k largest of vals[0..n) (ties to the lower index).
// On return sh.T and sh.jlast describe the selection.
// lo/hi: this thread's partial min/max of the scores (from the pass that wrote them).
__device__ void topk_threshold(const float* vals, int n, int k, SelShared& sh, int* err, float lo, float hi) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    lo = warp_min(lo);
    hi = warp_max(hi);
    if (lane == 0) { sh.red_f[warp] = lo; sh.red_f2[warp] = hi; }
    for (int b = tid; b < kBins; b += kSelThreads) sh.hist[b] = 0;
    if (tid == 0) sh.ncand = 0;
    __syncthreads();
    if (warp == 0) {
        lo = warp_min(sh.red_f[lane]);
        hi = warp_max(sh.red_f2[lane]);
        if (lane == 0) { sh.vmin = lo; sh.vmax = hi; }
    }
    __syncthreads();
    const float vmin = sh.vmin, vmax = sh.vmax;
    if (!(vmax > vmin)) {
        // all scores equal (or not finite): the k lowest indices
        if (tid == 0) {
            sh.T = vmax;
            sh.jlast = k - 1;
            if (!(vmax == vmax) || isinf(vmax)) set_err(err, DEV_ERR_NUMERIC, 301);
        }
        __syncthreads();
        return;
    }
    float invw = static_cast<float>(kBins) / (vmax - vmin);
    if (!isfinite(invw)) invw = 0.f;
#pragma unroll 4
    for (int j = tid; j < n; j += kSelThreads) atomicAdd(&sh.hist[bin_of(vals[j], vmin, invw)], 1);
    __syncthreads();
    // the bin holding the k-th largest: thread t owns bins 2047-2t and 2046-2t (highest
    // first); a block-wide prefix sum gives the count in every higher bin
    static_assert(kBins == 2 * kSelThreads, "two bins per thread");
    {
        const int b0 = kBins - 1 - 2 * tid, b1 = b0 - 1;
        const int h0 = sh.hist[b0], h1 = sh.hist[b1];
        const int above = block_exscan(h0 + h1, sh, nullptr);
        if (above < k && k <= above + h0 + h1) {
            const bool first = above + h0 >= k;
            sh.bstar = first ? b0 : b1;
            sh.above = first ? above : above + h0;
        }
    }
    __syncthreads();
    const int bstar = sh.bstar, need = k - sh.above, cnt = sh.hist[bstar];
    if (cnt <= kCand) {
        for (int j = tid; j < n; j += kSelThreads) {
            const float x = vals[j];
            if (bin_of(x, vmin, invw) == bstar) {
                const int c = atomicAdd(&sh.ncand, 1);
                if (c < kCand) { sh.cand_v[c] = x; sh.cand_j[c] = j; }
            }
        }
        __syncthreads();
        const int nc = min(sh.ncand, kCand);
        if (tid < nc) {
            const float x = sh.cand_v[tid];
            const int jx = sh.cand_j[tid];
            int rank = 0;
            for (int m = 0; m < nc; ++m) {
                const float y = sh.cand_v[m];
                rank += (y > x) || (y == x && sh.cand_j[m] < jx);
            }
            if (rank == need - 1) { sh.T = x; sh.jlast = jx; }
        }
        __syncthreads();
        return;
    }
    // crowded boundary bin: exact radix select on the order-preserving keys
    uint32_t prefix = 0, mask = 0;
    int rem = need;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int b = tid; b < 256; b += kSelThreads) sh.hist[b] = 0;
        __syncthreads();
        for (int j = tid; j < n; j += kSelThreads) {
            const float x = vals[j];
            if (bin_of(x, vmin, invw) != bstar) continue;
            const uint32_t key = ord_key(x);
            if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & 255], 1);
        }
        __syncthreads();
        if (tid == 0) {
            int c = 0, d = 255;
            for (; d > 0; --d) {
                if (c + sh.hist[d] >= rem) break;
                c += sh.hist[d];
            }
            sh.above = c;
            sh.bstar = d;
        }
        __syncthreads();
        rem -= sh.above;
        prefix |= static_cast<uint32_t>(sh.bstar) << shift;
        mask |= 0xFFu << shift;
        __syncthreads();
    }
    const float T = key_to_float(prefix);
    // jlast: index of the rem-th score equal to T in index order
    const int seg = ((n + kWarps - 1) / kWarps + 31) & ~31;
    const int a = warp * seg, e = min(n, a + seg);
    int c = 0;
    for (int j = a + lane; j < a + seg; j += 32) {
        const bool eq = j < e && vals[j] == T;
        c += __popc(__ballot_sync(0xffffffffu, eq));
    }
    int tot2 = 0;
    const int wbase = block_exscan(lane == 0 ? c : 0, sh, &tot2);
    const int base0 = __shfl_sync(0xffffffffu, wbase, 0);
    int run = base0;
    for (int j = a + lane; j < a + seg; j += 32) {
        const bool eq = j < e && vals[j] == T;
        const unsigned bal = __ballot_sync(0xffffffffu, eq);
        const int r = run + __popc(bal & ((1u << lane) - 1u));
        if (eq && r == rem - 1) { sh.jlast = j; }
        run += __popc(bal);
    }
    if (tid == 0) sh.T = T;
    __syncthreads();
}

// The same threshold over a unit's scores split into C contiguous slices, one per CTA of a
// cluster (this CTA: rank `rank`, scores vals[0..nl) at global positions j0 + ...).  Every
// decision is taken on cluster-wide sums, so every CTA reaches the same T and jlast (global
// positions) as the one-CTA form: the score range, the histogram and each radix digit's
// counts are summed over the cluster; boundary candidates are gathered in the leader (rank 0),
// which ranks them; the jlast of a crowded bin is found by the CTA holding it.  All branches
// are uniform across the cluster, so every CTA passes every cluster barrier.
__device__ void topk_threshold_cl(const float* vals, int nl, int j0, int k, SelShared& sh, int* err, float lo, float hi,
                                  int C, int rank) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    lo = warp_min(lo);
    hi = warp_max(hi);
    if (lane == 0) { sh.red_f[warp] = lo; sh.red_f2[warp] = hi; }
    for (int b = tid; b < kBins; b += kSelThreads) sh.hist[b] = 0;
    if (tid == 0) sh.ncand = 0;
    __syncthreads();
    if (warp == 0) {
        lo = warp_min(sh.red_f[lane]);
        hi = warp_max(sh.red_f2[lane]);
        if (lane == 0) { sh.cl_lo = lo; sh.cl_hi = hi; }
    }
    cluster_sync_all();   // every CTA's range is published; every candidate counter is zero
    if (warp == 0) {
        // lane r reads rank r's range (C <= 32)
        float L = CUDART_INF_F, Hh = -CUDART_INF_F;
        if (lane < C) {
            L = ld_cluster_f32(cluster_addr(&sh.cl_lo, lane));
            Hh = ld_cluster_f32(cluster_addr(&sh.cl_hi, lane));
        }
        L = warp_min(L);
        Hh = warp_max(Hh);
        if (lane == 0) {
            sh.vmin = L;
            sh.vmax = Hh;
        }
    }
    __syncthreads();
    const float vmin = sh.vmin, vmax = sh.vmax;
    if (!(vmax > vmin)) {
        // all scores equal (or not finite): the k lowest positions
        if (tid == 0) {
            sh.T = vmax;
            sh.jlast = k - 1;
            if (rank == 0 && (!(vmax == vmax) || isinf(vmax))) set_err(err, DEV_ERR_NUMERIC, 301);
        }
        cluster_sync_all();   // nobody reads another CTA's range after this
        return;
    }
    float invw = static_cast<float>(kBins) / (vmax - vmin);
    if (!isfinite(invw)) invw = 0.f;
#pragma unroll 4
    for (int j = tid; j < nl; j += kSelThreads) atomicAdd(&sh.hist[bin_of(vals[j], vmin, invw)], 1);
    cluster_sync_all();   // every CTA's histogram is complete
    {
        const int b0 = kBins - 1 - 2 * tid, b1 = b0 - 1;
        int h0, h1;
        cluster_sum2(&sh.hist[b0], &sh.hist[b1], C, h0, h1);
        const int above = block_exscan(h0 + h1, sh, nullptr);
        if (above < k && k <= above + h0 + h1) {
            const bool first = above + h0 >= k;
            sh.bstar = first ? b0 : b1;
            sh.above = first ? above : above + h0;
            sh.total = first ? h0 : h1;   // the boundary bin's count over the cluster
        }
    }
    __syncthreads();
    const int bstar = sh.bstar, need = k - sh.above, cnt = sh.total;
    cluster_sync_all();   // every CTA has read the histograms
    if (cnt <= kCand) {
        // the boundary bin's members, gathered in the leader, ranked there
        const uint32_t lead_n = cluster_addr(&sh.ncand, 0);
        for (int j = tid; j < nl; j += kSelThreads) {
            const float x = vals[j];
            if (bin_of(x, vmin, invw) == bstar) {
                const int c = atom_cluster_add(lead_n, 1);
                if (c < kCand) {
                    st_cluster_f32(cluster_addr(&sh.cand_v[c], 0), x);
                    st_cluster_s32(cluster_addr(&sh.cand_j[c], 0), j0 + j);
                }
            }
        }
        cluster_sync_all();
        if (rank == 0) {
            const int nc = min(sh.ncand, kCand);
            if (tid < nc) {
                const float x = sh.cand_v[tid];
                const int jx = sh.cand_j[tid];
                int rnk = 0;
                for (int m = 0; m < nc; ++m) {
                    const float y = sh.cand_v[m];
                    rnk += (y > x) || (y == x && sh.cand_j[m] < jx);
                }
                if (rnk == need - 1) { sh.T = x; sh.jlast = jx; }
            }
        }
        cluster_sync_all();   // the leader's T and jlast are set
        if (tid == 0 && rank != 0) {
            sh.T = ld_cluster_f32(cluster_addr(&sh.T, 0));
            sh.jlast = ld_cluster_s32(cluster_addr(&sh.jlast, 0));
        }
        cluster_sync_all();   // nobody reads the leader after this
        return;
    }
    // crowded boundary bin: exact radix select on the order-preserving keys, digit counts summed
    uint32_t prefix = 0, mask = 0;
    int rem = need;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int b = tid; b < 256; b += kSelThreads) sh.hist[b] = 0;
        __syncthreads();
        for (int j = tid; j < nl; j += kSelThreads) {
            const float x = vals[j];
            if (bin_of(x, vmin, invw) != bstar) continue;
            const uint32_t key = ord_key(x);
            if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & 255], 1);
        }
        cluster_sync_all();   // every CTA's digit counts are complete
        // digit d's count over the cluster, one thread per digit (the candidate slots are free here)
        if (tid < 256) sh.cand_j[tid] = cluster_sum(&sh.hist[tid], C);
        __syncthreads();
        if (tid == 0) {
            int c = 0, d = 255;
            for (; d > 0; --d) {
                if (c + sh.cand_j[d] >= rem) break;
                c += sh.cand_j[d];
            }
            sh.above = c;
            sh.bstar = d;
        }
        cluster_sync_all();   // every CTA has read the counts before the next pass clears them
        rem -= sh.above;
        prefix |= static_cast<uint32_t>(sh.bstar) << shift;
        mask |= 0xFFu << shift;
    }
    const float T = key_to_float(prefix);
    // jlast: the rem-th score equal to T in position order; slices are in position order
    int c = 0;
    for (int j = tid; j < nl; j += kSelThreads) c += vals[j] == T;
    c = warp_sum_i(c);
    if (lane == 0) sh.red_i[warp] = c;
    __syncthreads();
    if (tid == 0) {
        int t = 0;
        for (int w = 0; w < kWarps; ++w) t += sh.red_i[w];
        sh.cl_cnt = t;
    }
    cluster_sync_all();   // every CTA's count of ties is published
    if (tid == 0) sh.above = cluster_sum(&sh.cl_cnt, rank);
    __syncthreads();
    const int base = sh.above;
    if (rem - 1 >= base && rem - 1 < base + sh.cl_cnt) {
        // this CTA holds it: warp-segmented scan of the slice in position order
        const int seg = ((nl + kWarps - 1) / kWarps + 31) & ~31;
        const int a = warp * seg, e = min(nl, a + seg);
        int cw = 0;
        for (int j = a + lane; j < a + seg; j += 32) {
            const bool eq = j < e && vals[j] == T;
            cw += __popc(__ballot_sync(0xffffffffu, eq));
        }
        int tot2 = 0;
        const int wbase = block_exscan(lane == 0 ? cw : 0, sh, &tot2);
        int run = base + __shfl_sync(0xffffffffu, wbase, 0);
        for (int j = a + lane; j < a + seg; j += 32) {
            const bool eq = j < e && vals[j] == T;
            const unsigned bal = __ballot_sync(0xffffffffu, eq);
            const int r = run + __popc(bal & ((1u << lane) - 1u));
            if (eq && r == rem - 1) st_cluster_s32(cluster_addr(&sh.jlast, 0), j0 + j);
            run += __popc(bal);
        }
    }
    cluster_sync_all();   // the leader's jlast is set
    if (tid == 0) {
        sh.T = T;
        if (rank != 0) sh.jlast = ld_cluster_s32(cluster_addr(&sh.jlast, 0));
    }
    cluster_sync_all();   // nobody reads the leader after this
}

// Writes the selected indices (ascending) via out_fn(pos, j); returns the count.
// Element j lives in row r = j / kSelThreads at thread j % kSelThreads, so a row
// is in index order across the block.  One read per element: warp w counts its
// takes in row r (a ballot), the (row, warp) counts are scanned in index order,
// and every taken element goes to its rank.  Up to 64 rows the counts fit in
// the histogram's storage; beyond, warps own contiguous segments (two passes).
template <class F>
__device__ int compact_selected(const float* vals, int n, float T, int jlast, SelShared& sh, F out_fn) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rows = (n + kSelThreads - 1) / kSelThreads;
    if (rows <= kBins / kWarps) {
        int* cnt = sh.hist;   // [rows][kWarps] counts, then their exclusive prefix
        const unsigned lt = (1u << lane) - 1u;
        for (int r = 0; r < rows; ++r) {
            const int j = r * kSelThreads + tid;
            bool take = false;
            if (j < n) { const float x = vals[j]; take = (x > T) || (x == T && j <= jlast); }
            const unsigned bal = __ballot_sync(0xffffffffu, take);
            if (lane == 0) cnt[r * kWarps + warp] = __popc(bal);
        }
        __syncthreads();
        const int ne = rows * kWarps;
        const int e0 = 2 * tid, e1 = e0 + 1;
        const int c0 = e0 < ne ? cnt[e0] : 0, c1 = e1 < ne ? cnt[e1] : 0;
        int total = 0;
        const int base = block_exscan(c0 + c1, sh, &total);
        if (e0 < ne) cnt[e0] = base;
        if (e1 < ne) cnt[e1] = base + c0;
        __syncthreads();
        for (int r = 0; r < rows; ++r) {
            const int j = r * kSelThreads + tid;
            bool take = false;
            if (j < n) { const float x = vals[j]; take = (x > T) || (x == T && j <= jlast); }
            const unsigned bal = __ballot_sync(0xffffffffu, take);
            if (take) out_fn(cnt[r * kWarps + warp] + __popc(bal & lt), j);
        }
        __syncthreads();
        return total;
    }
    const int seg = ((n + kWarps - 1) / kWarps + 31) & ~31;
    const int a = warp * seg, e = min(n, a + seg);
    int c = 0;
    for (int j = a + lane; j < a + seg; j += 32) {
        bool take = false;
        if (j < e) { const float x = vals[j]; take = (x > T) || (x == T && j <= jlast); }
        c += __popc(__ballot_sync(0xffffffffu, take));
    }
    int total = 0;
    const int wb = block_exscan(lane == 0 ? c : 0, sh, &total);
    int run = __shfl_sync(0xffffffffu, wb, 0);
    for (int j = a + lane; j < a + seg; j += 32) {
        bool take = false;
        if (j < e) { const float x = vals[j]; take = (x > T) || (x == T && j <= jlast); }
        const unsigned bal = __ballot_sync(0xffffffffu, take);
        if (take) out_fn(run + __popc(bal & ((1u << lane) - 1u)), j);
        run += __popc(bal);
    }
    __syncthreads();
    return total;
}

__device__ __forceinline__ int lower_bound(const int32_t* a, int n, int x) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] < x) lo = mid + 1; else hi = mid;
    }
    return lo;
}

// ----------------------------------------------------------------- decode
template <int G, bool CL>
__device__ __forceinline__ void select_decode(const SelectParams& p) {
    extern __shared__ __align__(16) uint8_t dsm[];
    __shared__ SelShared sh;
    // cluster form (CL): the unit's scores are split into C contiguous slices, one per CTA of a
    // cluster; the leader (rank 0) appends, gathers the selection and does the index scan
    const int C = CL ? p.cluster : 1;
    const int crank = CL ? static_cast<int>(cluster_ctarank()) : 0;
    const int u = blockIdx.x / C, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = p.n, K = p.k;
    const int j0 = static_cast<int>(static_cast<int64_t>(crank) * n / C);
    const int nl = static_cast<int>(static_cast<int64_t>(crank + 1) * n / C) - j0;
    const int nlmax = (n + C - 1) / C;
    pdl_wait();      // the scores of this step
    pdl_trigger();
    // staged one-CTA form: the unit's logits stream into two shared-memory buffers by bulk
    // copies issued now, in flight while the log-sum-exp forms; the score pass reads them there
    __shared__ uint64_t sbar[2];
    const bool stg = p.stage;
    const int sper = kSelStageBytes / (4 * G);             // scores per buffer
    const int nstg = stg ? (nl + sper - 1) / sper : 0;
    const bool ids_stg = !CL && stg && n % 4 == 0 && n * 4 <= kSelStageBytes;
    const float* z = p.logits + (static_cast<int64_t>(u) * n + j0) * G;   // this CTA's slice
    auto issue = [&](int c) {   // buffer c & 1 <- scores [c * sper, min(nl, (c + 1) * sper))
        const uint32_t bytes = static_cast<uint32_t>(min(sper, nl - c * sper)) * G * 4;
        mbar_arrive_expect_tx(&sbar[c & 1], bytes);
        bulk_g2s(dsm + p.stage_off + (c & 1) * kSelStageBytes, z + static_cast<int64_t>(c) * sper * G, bytes, &sbar[c & 1]);
    };
    if (stg && tid == 0) {
        mbar_init(&sbar[0], 1);
        mbar_init(&sbar[1], 1);
        fence_mbar_init();
        for (int c = 0; c < 2 && c < nstg; ++c) issue(c);
    }
    float* vals = (nlmax <= p.smem_cap) ? reinterpret_cast<float*>(dsm) : p.vbuf + static_cast<int64_t>(u) * n + j0;
    const int cap_f = (nlmax <= p.smem_cap) ? ((nlmax + 3) & ~3) : 0;
    int32_t* sSel = reinterpret_cast<int32_t*>(dsm) + cap_f;
    int32_t* sSlot = sSel + K;
    int32_t* sFree = sSlot + K;
    int32_t* sPid = sFree + K;       // previous step's selection (ascending) ...
    int32_t* sPslot = sPid + K;      // ... and its slots
    // log-sum-exp warps: one per query head in the one-CTA form; in the cluster form 16, kWpg
    // per head when the records need more than one round of loads
    constexpr int kLseWarps = CL ? 16 : G, kWpg = 16 / G;
    if (crank == 0 && warp >= kLseWarps) {
        // work with no dependency on the scores, done while the first warps form the log-sum-exp
        const int wt = tid - kLseWarps * 32, nt = kSelThreads - kLseWarps * 32;
        if (p.t > 0) {
            const int32_t* gp = p.prev_ids + static_cast<int64_t>(u) * K;
            const int32_t* gs = p.prev_slot + static_cast<int64_t>(u) * K;
            for (int i = wt; i < K; i += nt) { sPid[i] = gp[i]; sPslot[i] = gs[i]; }
        }
        // append the new token to the exact local set at row W + t
        const int row = p.W + p.t;
        const int n16 = kD * p.es / 16;
        if (row < p.loc_cap) {
            const int64_t off = (static_cast<int64_t>(u) * p.loc_pitch + row) * kD * p.es;
            const int64_t src = static_cast<int64_t>(u) * kD * p.es;
            if (wt < n16) {
                // no key here for generated keys kept at rank r: the rebuild writes it
                if (p.k_new)
                    copy_row16(static_cast<uint8_t*>(p.k_loc) + off, static_cast<const uint8_t*>(p.k_new) + src, n16,
                               wt, 1 << 30);
            } else if (p.es_v == 1) {
                // e5m2 value storage: 16 threads round 8 bf16 values each
                const int vt = wt - 64;
                if (vt >= 0 && vt < kD / 8) {
                    const __nv_bfloat16* vs = static_cast<const __nv_bfloat16*>(p.v_new) + static_cast<int64_t>(u) * kD + vt * 8;
                    uint8_t* vd = static_cast<uint8_t*>(p.v_loc) + (static_cast<int64_t>(u) * p.loc_pitch + row) * kD + vt * 8;
                    float f[8];
                    load8(vs, f);
                    uint32_t lo = 0, hi = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        lo |= static_cast<uint32_t>(from_f<__nv_fp8_e5m2>(f[i]).__x) << (8 * i);
                        hi |= static_cast<uint32_t>(from_f<__nv_fp8_e5m2>(f[4 + i]).__x) << (8 * i);
                    }
                    *reinterpret_cast<uint2*>(vd) = make_uint2(lo, hi);
                }
            } else if (wt >= 64 && wt < 64 + n16) {
                copy_row16(static_cast<uint8_t*>(p.v_loc) + off, static_cast<const uint8_t*>(p.v_new) + src, n16, wt - 64,
                           1 << 30);
            }
        } else if (wt == 0) {
            set_err(p.err, DEV_ERR_BOUNDS, 316);
        }
    }

    // 1. log-sum-exp of every query head from the scoring runs' records: wpg warps per head
    // (kWpg when the records need more than one round of loads), each over an interleaved share
    // of the records, combined after the barrier below
    const int nrec = p.nru * p.nparts;
    const int wpg = (CL && nrec > 4 * 32) ? kWpg : 1;
    if (warp < wpg * G) {
        const int g = warp % G, part = warp / G;
        const float2* rec = p.part + static_cast<int64_t>(u) * nrec * G;
        // running (max, sum) per lane over its records, four loads in flight at a time
        float m = -CUDART_INF_F, sx = 0.f;
        for (int r0 = part * 32 + lane; r0 < nrec; r0 += 4 * 32 * wpg) {
            float2 x[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = r0 + 32 * wpg * i;
                x[i] = r < nrec ? rec[r * G + g] : make_float2(-CUDART_INF_F, 0.f);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (x[i].x == -CUDART_INF_F) continue;
                if (x[i].x > m) {
                    sx = sx * __expf(m - x[i].x) + x[i].y;
                    m = x[i].x;
                } else {
                    sx += x[i].y * __expf(x[i].x - m);
                }
            }
        }
        const float M = warp_max(m);
        const float S = warp_sum(m == -CUDART_INF_F ? 0.f : sx * __expf(m - M));
        if (lane == 0) {
            if constexpr (CL) sh.lse_part[warp] = make_float2(M, S);
            else sh.lse[warp] = M + __logf(S);
        }
    }
    if (u == 0 && crank == 0 && tid == 0 && p.sched) *p.sched = 0;   // the scoring kernel of this step is done
    __syncthreads();
    // 2. v_j = max_g (z_gj - lse_g)
    float lse[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        if constexpr (!CL) {
            lse[g] = sh.lse[g];
            continue;
        }
        float M = sh.lse_part[g].x, S = sh.lse_part[g].y;
        if (wpg > 1) {
#pragma unroll
            for (int q = 1; q < kWpg; ++q) M = fmaxf(M, sh.lse_part[q * G + g].x);
            S = 0.f;
#pragma unroll
            for (int q = 0; q < kWpg; ++q) {
                const float2 e = sh.lse_part[q * G + g];
                if (e.x != -CUDART_INF_F) S += e.y * __expf(e.x - M);
            }
        }
        lse[g] = M + __logf(S);
    }
    float lo = CUDART_INF_F, hi = -CUDART_INF_F;
    if (stg) {
        bool ok = true;
        for (int c = 0; c < nstg; ++c) {
            const int b = c & 1;
            if (ok && !mbar_wait(&sbar[b], (c >> 1) & 1)) {
                if (tid == 0) set_err(p.err, DEV_ERR_TIMEOUT, 317);
                (void)mbar_wait(&sbar[b], (c >> 1) & 1);   // the copy may still be in flight
                ok = false;
            }
            const float* zs = reinterpret_cast<const float*>(dsm + p.stage_off + b * kSelStageBytes);
            const int e0 = c * sper, e1 = min(nl, e0 + sper);
            for (int j = e0 + tid; j < e1; j += kSelThreads) {
                float v;
                if constexpr (G == 4) {
                    const float4 zz = reinterpret_cast<const float4*>(zs)[j - e0];
                    v = fmaxf(fmaxf(zz.x - lse[0], zz.y - lse[1]), fmaxf(zz.z - lse[2], zz.w - lse[3]));
                } else {
                    v = -CUDART_INF_F;
#pragma unroll
                    for (int g = 0; g < G; ++g) v = fmaxf(v, zs[(j - e0) * G + g] - lse[g]);
                }
                vals[j] = v;
                lo = fminf(lo, v);
                hi = fmaxf(hi, v);
            }
            __syncthreads();   // buffer b is free again
            if (tid == 0 && ok && c + 2 < nstg) issue(c + 2);
        }
        // one-CTA form: the unit's position -> chunk id table, into buffer 0 once the scores are
        // read, in flight through the threshold and the compaction
        if (tid == 0 && ids_stg) {
            mbar_arrive_expect_tx(&sbar[0], static_cast<uint32_t>(n) * 4);
            bulk_g2s(dsm + p.stage_off, p.ids + static_cast<int64_t>(u) * n, static_cast<uint32_t>(n) * 4, &sbar[0]);
        }
    } else if constexpr (G == 4) {
        // four independent 16-byte loads in flight per thread
        const float4* z4 = reinterpret_cast<const float4*>(z);
        int j = tid;
        for (; j + 7 * kSelThreads < nl; j += 8 * kSelThreads) {
            float4 a[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) a[r] = __ldcg(z4 + j + r * kSelThreads);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float v = fmaxf(fmaxf(a[r].x - lse[0], a[r].y - lse[1]), fmaxf(a[r].z - lse[2], a[r].w - lse[3]));
                vals[j + r * kSelThreads] = v;
                lo = fminf(lo, v);
                hi = fmaxf(hi, v);
            }
        }
        for (; j < nl; j += kSelThreads) {
            const float4 zz = __ldcg(z4 + j);
            const float v = fmaxf(fmaxf(zz.x - lse[0], zz.y - lse[1]), fmaxf(zz.z - lse[2], zz.w - lse[3]));
            vals[j] = v;
            lo = fminf(lo, v);
            hi = fmaxf(hi, v);
        }
    } else {
#pragma unroll 4
        for (int j = tid; j < nl; j += kSelThreads) {
            float v = -CUDART_INF_F;
#pragma unroll
            for (int g = 0; g < G; ++g) v = fmaxf(v, z[static_cast<int64_t>(j) * G + g] - lse[g]);
            vals[j] = v;
            lo = fminf(lo, v);
            hi = fmaxf(hi, v);
        }
    }
    // 3. exact top-K threshold and ordered compaction into sSel (original chunk ids)
    if constexpr (CL) topk_threshold_cl(vals, nl, j0, K, sh, p.err, lo, hi, C, crank);
    else topk_threshold(vals, n, K, sh, p.err, lo, hi);
    const float T = sh.T;
    const int jlast = sh.jlast;
    const int32_t* ids = p.ids + static_cast<int64_t>(u) * n;
    const int got = compact_selected(vals, nl, T, jlast - j0, sh, [&](int pos, int j) {
        if (pos < K) sSel[pos] = j;
    });
    if constexpr (!CL) {
        if (got != K) {
            // only non-finite scores can break the count; keep downstream indices valid
            if (tid == 0) set_err(p.err, DEV_ERR_NUMERIC, 312);
            for (int i = tid; i < K; i += kSelThreads) sSel[i] = i;
            __syncthreads();
        }
        // positions -> original chunk ids, from the staged table or with every load in flight
        if (ids_stg) {
            const uint32_t par = static_cast<uint32_t>((nstg + 1) / 2) & 1u;   // buffer 0's next phase
            if (!mbar_wait(&sbar[0], par)) {
                if (tid == 0) set_err(p.err, DEV_ERR_TIMEOUT, 318);
                (void)mbar_wait(&sbar[0], par);
            }
            const int32_t* sids = reinterpret_cast<const int32_t*>(dsm + p.stage_off);
            for (int i = tid; i < K; i += kSelThreads) sSel[i] = sids[sSel[i]];
        } else {
            for (int i = tid; i < K; i += kSelThreads) sSel[i] = ids[sSel[i]];
        }
        __syncthreads();
    } else {
        // each CTA translates its slice's picks, then places them after the lower ranks' picks
        // in the leader's selection
        const int mine = min(got, K);
        for (int i = tid; i < mine; i += kSelThreads) sSel[i] = ids[j0 + sSel[i]];
        if (tid == 0) sh.cl_cnt = got;
        cluster_sync_all();
        if (tid == 0) sh.above = cluster_sum(&sh.cl_cnt, crank);
        if (tid == 32) sh.total = cluster_sum(&sh.cl_cnt, C);
        __syncthreads();
        const int base = sh.above;
        if (crank != 0)
            for (int i = tid; i < mine && base + i < K; i += kSelThreads)
                st_cluster_s32(cluster_addr(&sSel[base + i], 0), sSel[i]);
        cluster_sync_all();   // the leader's selection is complete; no CTA reads another after this
        if (crank != 0) return;
        if (sh.total != K) {
            if (tid == 0) set_err(p.err, DEV_ERR_NUMERIC, 312);
            for (int i = tid; i < K; i += kSelThreads) sSel[i] = ids[i];
        }
        __syncthreads();
    }
    // 4. index scan against the previous step's selection.  Entry i's thread looks
    // up sSel[i] among the previous ids (hit: keeps its slot) and the previous
    // entry i among the current ids (gone: its slot is freed), two independent
    // binary searches; misses are then numbered in order of i and freed slots in
    // order of their previous position, and the m-th miss takes the m-th freed slot.
    const int t = p.t;
    const int32_t* pids = sPid;
    const int32_t* pslot = sPslot;
    constexpr int PER = (4096 + kSelThreads - 1) / kSelThreads;   // K <= 4096
    const int per = (K + kSelThreads - 1) / kSelThreads;          // entries per thread (1 for K <= 1024)
    int mflag[PER], fflag[PER], mc = 0, fc = 0;
#pragma unroll
    for (int r = 0; r < PER; ++r) {
        const int i = tid * per + r;
        mflag[r] = fflag[r] = 0;
        if (r >= per || i >= K) continue;
        const int x = sSel[i];
        int slot = -1, fr = 1;
        if (t > 0) {
            const int y = pids[i];
            const int pidx = lower_bound(pids, K, x);
            const int q = lower_bound(sSel, K, y);
            if (pidx < K && pids[pidx] == x) {
                slot = pslot[pidx];
                if (slot < 0 || slot >= K) { set_err(p.err, DEV_ERR_BOUNDS, 313); slot = -1; }
            }
            fr = !(q < K && sSel[q] == y);
        }
        sSlot[i] = slot;
        mflag[r] = slot < 0;
        fflag[r] = fr;
        mc += mflag[r];
        fc += fr;
    }
    int both = 0;
    const int bb = block_exscan(mc | (fc << 16), sh, &both);
    int mbase = bb & 0xFFFF, fbase = bb >> 16;
    const int nmiss = both & 0xFFFF, nfree = both >> 16;
#pragma unroll
    for (int r = 0; r < PER; ++r) {
        const int i = tid * per + r;
        if (fflag[r]) sFree[fbase++] = (t == 0) ? i : pslot[i];
    }
    __syncthreads();
    if (nmiss != nfree && tid == 0) set_err(p.err, DEV_ERR_BOUNDS, 314);
    int32_t* cids = p.cur_ids + static_cast<int64_t>(u) * K;
    int32_t* cslot = p.cur_slot + static_cast<int64_t>(u) * K;
    int32_t* mch = p.miss_chunk + static_cast<int64_t>(u) * K;
    int32_t* msl = p.miss_slot + static_cast<int64_t>(u) * K;
#pragma unroll
    for (int r = 0; r < PER; ++r) {
        const int i = tid * per + r;
        if (r >= per || i >= K) continue;
        int slot = sSlot[i];
        if (mflag[r]) {
            const int m = mbase++;
            slot = (m < nfree) ? sFree[m] : 0;
            if (slot < 0 || slot >= K) { set_err(p.err, DEV_ERR_BOUNDS, 315); slot = 0; }
            mch[m] = sSel[i];
            msl[m] = slot;
        }
        cids[i] = sSel[i];
        cslot[i] = slot;
        if (p.slot_chunk) p.slot_chunk[static_cast<int64_t>(u) * K + slot] = sSel[i];
        if (p.sel_out_user) p.sel_out_user[static_cast<int64_t>(u) * K + i] = sSel[i];
    }
    if (tid == 0) {
        p.miss_count[u] = nmiss;
        atomicAdd(p.hits_step + t, K - nmiss);
    }
}

// One CTA per unit.
template <int G>
__global__ void __launch_bounds__(kSelThreads) k_select_decode(SelectParams p) {
    select_decode<G, false>(p);
}

// One cluster per unit (one CTA per SM: the full register file is available).
template <int G>
__global__ void __launch_bounds__(kSelThreads, 1) k_select_decode_cl(SelectParams p) {
    select_decode<G, true>(p);
}

// ----------------------------------------------------------------- outliers (prefill)
__global__ void __launch_bounds__(kSelThreads) k_select_outliers(SelectParams p) {
    extern __shared__ __align__(16) uint8_t dsm[];
    __shared__ SelShared sh;
    const int u = blockIdx.x, tid = threadIdx.x;
    const int n = p.n, k = p.k;
    float* vals = (n <= p.smem_cap) ? reinterpret_cast<float*>(dsm) : p.vbuf + static_cast<int64_t>(u) * n;
    const float* src = p.neg_src + static_cast<int64_t>(u) * n;
    float lo = CUDART_INF_F, hi = -CUDART_INF_F;
    for (int j = tid; j < n; j += kSelThreads) {
        const float v = -src[j];
        vals[j] = v;
        lo = fminf(lo, v);
        hi = fmaxf(hi, v);
    }
    topk_threshold(vals, n, k, sh, p.err, lo, hi);
    int32_t* out = p.sel_plain + static_cast<int64_t>(u) * k;
    const int got = compact_selected(vals, n, sh.T, sh.jlast, sh, [&](int pos, int j) {
        if (pos < k) out[pos] = j;
    });
    if (got != k) {
        if (tid == 0) set_err(p.err, DEV_ERR_NUMERIC, 321);
        for (int i = tid; i < k; i += kSelThreads) out[i] = i;
    }
}

constexpr int kSelMinPerCta = 4096;           // scores per CTA of a cluster, at least
constexpr int kSelOneCta = 16 * kSelThreads;    // up to this many scores a unit keeps one CTA

int launch_select_decode(int dtype, const SelectParams& p, cudaStream_t s) {
    (void)dtype;
    void (*fn)(SelectParams) = nullptr;    // one CTA per unit
    void (*fnc)(SelectParams) = nullptr;   // a cluster per unit
    switch (p.G) {
        case 1: fn = k_select_decode<1>; fnc = k_select_decode_cl<1>; break;
        case 2: fn = k_select_decode<2>; fnc = k_select_decode_cl<2>; break;
        case 4: fn = k_select_decode<4>; fnc = k_select_decode_cl<4>; break;
        case 8: fn = k_select_decode<8>; fnc = k_select_decode_cl<8>; break;
        default: return -1;
    }
    // A unit with more than kSelOneCta scores and SMs to spare is split over a cluster of C
    // CTAs: the largest C <= 16 that leaves every CTA at least kSelMinPerCta scores, fits a
    // slice in shared memory, and keeps all U clusters resident at once.
    static int max_clusters[4][17];   // per G, per cluster size; 0 = not queried
    const int gi = p.G == 1 ? 0 : p.G == 2 ? 1 : p.G == 4 ? 2 : 3;
    int C = 1;
    const int cmax = p.n > kSelOneCta ? std::min(16, p.nsm > 0 ? p.nsm / p.U : 1) : 1;
    if (cmax > 8) cudaFuncSetAttribute(fnc, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    for (int c = cmax; c >= 2 && C == 1; --c) {
        const int nlmax = (p.n + c - 1) / c;
        if (p.n / c < kSelMinPerCta || nlmax > p.smem_cap) continue;
        const size_t sm_c = static_cast<size_t>((nlmax + 3) & ~3) * 4 + static_cast<size_t>(p.k) * 4 * 5;
        if (max_clusters[gi][c] == 0) {
            cudaFuncSetAttribute(fnc, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm_c));
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(p.U * c);
            q.blockDim = dim3(kSelThreads);
            q.dynamicSmemBytes = sm_c;
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = c;
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            q.attrs = qa;
            q.numAttrs = 1;
            int nmax = 0;
            if (cudaOccupancyMaxActiveClusters(&nmax, fnc, &q) != cudaSuccess) {
                cudaGetLastError();
                nmax = 0;
            }
            max_clusters[gi][c] = nmax > 0 ? nmax : -1;
        }
        if (max_clusters[gi][c] >= p.U) C = c;
    }
    const int nlmax = (p.n + C - 1) / C;
    const int cap_f = (nlmax <= p.smem_cap) ? ((nlmax + 3) & ~3) : 0;
    size_t smem = static_cast<size_t>(cap_f) * 4 + static_cast<size_t>(p.k) * 4 * 5;
    // the staged form when the scores live in shared memory, every CTA's slice and buffer starts
    // on a 16-byte boundary, and the two buffers fit beside the scores
    static int smem_room = -1;   // opt-in shared memory per block minus the kernels' static use
    if (smem_room < 0) {
        int dev = 0, optin = 0;
        cudaFuncAttributes fa{}, fc{};
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
            cudaFuncGetAttributes(&fa, k_select_decode<8>) == cudaSuccess &&
            cudaFuncGetAttributes(&fc, k_select_decode_cl<8>) == cudaSuccess)
            smem_room = optin - static_cast<int>(std::max(fa.sharedSizeBytes, fc.sharedSizeBytes)) - 1024;
        else
            smem_room = 0;
        cudaGetLastError();
    }
    const size_t off = (smem + 127) & ~size_t(127);
    const bool aligned = C == 1 ? (static_cast<int64_t>(p.n) * p.G * 4) % 16 == 0 : (p.G * 4) % 16 == 0;
    const bool staged = cap_f > 0 && aligned && off + 2 * kSelStageBytes <= static_cast<size_t>(smem_room);
    if (staged) smem = off + 2 * kSelStageBytes;
    if (C == 1) {
        SelectParams ps = p;
        if (staged) {
            ps.stage = 1;
            ps.stage_off = static_cast<int>(off);
        }
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (launch_pdl(fn, dim3(p.U), dim3(kSelThreads), smem, s, ps) != cudaSuccess) {
            cudaGetLastError();
            return -1;
        }
        return 0;
    }
    SelectParams pc = p;
    pc.cluster = C;
    if (staged) {
        pc.stage = 1;
        pc.stage_off = static_cast<int>(off);
    }
    cudaFuncSetAttribute(fnc, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.U * C);
    cfg.blockDim = dim3(kSelThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = C;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, fnc, pc) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return 0;
}

int launch_select_outliers(const SelectParams& p, cudaStream_t s) {
    const size_t smem = (p.n <= p.smem_cap) ? static_cast<size_t>((p.n + 3) & ~3) * 4 : 0;
    cudaFuncSetAttribute(k_select_outliers, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    k_select_outliers<<<p.U, kSelThreads, smem, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace skv
