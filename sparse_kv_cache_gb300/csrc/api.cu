// Host side of the C ABI (include/shadowkv.h): config checks, library state
// in HBM, the pre-filling and decoding sequences of ShadowKV's Algorithms 1
// and 2 (Chinese digest, section A2), counters and the analytical models of
// the English summary (section 3.4, equivalent bandwidth; memory savings).
#include <cuda.h>
#include <cuda_runtime.h>

#include <errno.h>
#include <sys/mman.h>

#include <algorithm>
#include <array>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <chrono>
#include <mutex>
#include <new>
#include <thread>
#include <vector>


#include <nvtx3/nvToolsExt.h>

#include "shadowkv.h"
#include "skv_internal.h"

namespace {
// An NVTX range on the host timeline: one per library call and one per decode phase, so that a
// profiler shows where a step's launches come from and ncu can select a phase's kernels
// (--nvtx --nvtx-include).  A push and a pop cost a few nanoseconds when no tool listens.
struct NvtxRange {
    bool on = true;
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    void end() {
        if (on) nvtxRangePop();
        on = false;
    }
    ~NvtxRange() { end(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace

using namespace skv;

namespace {

constexpr int kVersion = 1 * 10000 + 0 * 100 + 0;

// ------------------------------------------------------------------ fault injection
// SHADOWKV_FAULT=oom[:N] makes the N-th device allocation of a pre-filling
// (1-based, default 1) fail, to exercise the clean-up path.
int g_alloc_counter = 0;
int fault_oom_at() {
    const char* e = std::getenv("SHADOWKV_FAULT");
    if (!e || std::strncmp(e, "oom", 3) != 0) return 0;
    if (e[3] == ':') return std::max(1, std::atoi(e + 4));
    return 1;
}

// huge-page host memory handed out by shadowkv_host_alloc_kind: (user pointer, mapping)
struct HostMap {
    void* user;       // the caller's pointer, aligned to the huge-page size
    size_t user_len;  // the caller's bytes, rounded up to whole huge pages
    void* raw;        // the whole mapping (with the alignment slack)
    size_t len;
};
std::mutex g_host_mu;
std::vector<HostMap> g_host_maps;

#ifndef MADV_COLLAPSE
#define MADV_COLLAPSE 25   // Linux 6.1+: collapse the range into transparent huge pages now
#endif

// Huge-page splits of the whole host (/proc/vmstat thp_split_pmd), or -1.
long host_thp_splits() {
    FILE* f = std::fopen("/proc/vmstat", "r");
    if (!f) return -1;
    char line[128];
    long v = -1;
    while (std::fgets(line, sizeof line, f))
        if (std::strncmp(line, "thp_split_pmd ", 14) == 0) {
            v = std::atol(line + 14);
            break;
        }
    std::fclose(f);
    return v;
}

// The keeper: a host thread that runs from the first decode step that reads huge-page values
// until the last such allocation is freed.  Every few milliseconds it reads the host kernel's
// count of huge-page splits; when the count moves, it collapses every huge-page allocation
// again (madvise MADV_COLLAPSE: a page that is whole costs nothing, a split one is copied into a
// fresh huge page, about 50 ms for 512 MiB), and then rests at least 50 ms.  A split page costs
// the fetch a translation per 64 KiB for the rest of the run.  It does not run while memory is
// filled and layers are pre-filled: a collapse needs a free huge page, the compaction that finds
// one can split other pages, and while pages are still being faulted in that feeds on itself
// (measured once: 86 splits and 104 collapses in one run).  Pre-filling repairs its own layer.
struct Keeper {
    std::thread th;
    std::atomic<bool> stop{false};
    bool running = false;
    std::mutex mu;   // start and halt; taken after g_host_mu when both are held
    ~Keeper() { halt(); }
    void halt() {
        std::lock_guard<std::mutex> lock(mu);
        if (!running) return;
        stop.store(true);
        th.join();
        running = false;
    }
    void start() {
        std::lock_guard<std::mutex> lock(mu);
        if (running) return;
        stop.store(false);
        th = std::thread([this] {
            long last = host_thp_splits();
            while (!stop.load()) {
                std::this_thread::sleep_for(std::chrono::milliseconds(5));
                const long now = host_thp_splits();
                if (now < 0 || now == last) continue;
                {
                    std::lock_guard<std::mutex> lock(g_host_mu);
                    for (const HostMap& m : g_host_maps) madvise(m.user, m.user_len, MADV_COLLAPSE);
                }
                last = host_thp_splits();   // splits the collapses themselves caused are not chased
                for (int i = 0; i < 10 && !stop.load(); ++i) std::this_thread::sleep_for(std::chrono::milliseconds(5));
            }
        });
        running = true;
    }
};
Keeper g_keeper;

// The huge-page host mapping holding [p, p + bytes), or nullptr.
const HostMap* find_host_map(const void* p, size_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    for (const HostMap& m : g_host_maps) {
        const uintptr_t b = reinterpret_cast<uintptr_t>(m.user);
        const uintptr_t e = b + m.user_len;
        if (a >= b && a < e && bytes <= e - a) return &m;
    }
    return nullptr;
}

// size of the host's transparent huge pages (512 MiB with 64 KiB base pages, 2 MiB with 4 KiB)
size_t host_huge_page_bytes() {
    size_t v = 0;
    if (FILE* f = std::fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
        unsigned long long x = 0;
        if (std::fscanf(f, "%llu", &x) == 1) v = static_cast<size_t>(x);
        std::fclose(f);
    }
    if (v < (size_t(2) << 20) || (v & (v - 1))) v = size_t(2) << 20;
    return v;
}

int es_of(int dtype) { return dtype == SKV_F32 ? 4 : 2; }   // A, B, q, keys, out
int es_l_of(int dtype) { return dtype == SKV_FP8 ? 1 : es_of(dtype); }   // landmarks
int es_v_of(int dtype) { return dtype == SKV_FP8 ? 1 : es_of(dtype); }   // values

}  // namespace

struct skv_layer {
    skv_config cfg{};
    int dev = 0, sm_count = 0;
    int U = 0, G = 0, H = 0, r = 0, K = 0, O = 0, W = 0, Tmax = 0, nchunk = 0, ncand = 0, n_c = 0;
    int es = 0, es_l = 0, es_v = 0, dtype = 0, nkb = 0, loc_cap = 0, nhi = 0;
    bool tc = false;   // bf16 keys and factors: the tensor-core kernels
    int64_t S = 0;
    const void* A = nullptr;
    const void* B = nullptr;
    const void* V = nullptr;
    const void* Vd = nullptr;
    std::vector<void*> allocs;
    void* L = nullptr;
    int32_t* ids = nullptr;
    int32_t* out_ids = nullptr;
    float* min_cos = nullptr;
    // keys and values of the attended set, one block of R rows per unit:
    // [O*C outlier rows | K*C cache rows (by slot) | loc_cap local rows]
    void *Kall = nullptr, *Vall = nullptr;
    int64_t R = 0;
    void *Kout = nullptr, *Vout = nullptr, *Kloc = nullptr, *Vloc = nullptr, *Kc = nullptr, *Vc = nullptr;
    int32_t* sel_ids[2] = {nullptr, nullptr};
    int32_t* sel_slot[2] = {nullptr, nullptr};
    int32_t *miss_chunk = nullptr, *miss_slot = nullptr, *miss_count = nullptr;
    int32_t* slot_chunk = nullptr;        // [U][K] chunk id of each cache slot
    bool v_direct = false;                // values in HBM read in place by attention (tensor-core path)
    bool v_huge = false;                  // values in a huge-page host allocation
    float* logits = nullptr;
    float2* score_part = nullptr;
    float* vbuf = nullptr;
    float* attn_part = nullptr;
    int32_t* attn_cnt = nullptr;
    void* Bt = nullptr;
    float2 *rope_lo = nullptr, *rope_hi = nullptr;
    int32_t* hits_step = nullptr;
    int* err = nullptr;
    CUtensorMap tmA{}, tmB{}, tmL{};
    CUtensorMap tmKall{};                 // the key blocks, [U*R][128], 128-row boxes (attention)
    int score_ncta = 0, score_nru = 0, score_nparts = 0, sel_smem_cap = 0;
    int32_t* sched = nullptr;
    int64_t launches = 0;                 // kernels launched by decode steps since the last reset
    int newkeys = SKV_NEWKEYS_EXACT;
    int Tpad = 0;                         // max_new_tokens rounded up to whole chunks
    void* Anew = nullptr;                 // ShadowKV+: rank-r states of generated tokens, [b][Tpad][r]
    uint8_t* qt = nullptr;                // e5m2 scorer: the query's three terms, [U][3G][d]
    float* qinv = nullptr;                // e5m2 scorer: 2^-s per head, [U][G]
    int64_t t = 0, t_reset = 0;
    cudaStream_t last_main = nullptr, last_side = nullptr;
    bool stepped = false;
    cudaEvent_t ev_sel = nullptr, ev_fetch = nullptr, ev_start = nullptr;
    cudaEvent_t user_sel = nullptr;       // the caller's event, recorded after each selection
    bool profiling = false;
    std::vector<std::array<cudaEvent_t, 8>> prof_pending, prof_free;
    double phase_ms[SKV_NPHASE] = {0};
    int64_t phase_n[SKV_NPHASE] = {0};
};

namespace {

int alloc(skv_layer* h, void** p, size_t bytes) {
    *p = nullptr;
    if (bytes == 0) bytes = 16;
    ++g_alloc_counter;
    const int f = fault_oom_at();
    if (f && g_alloc_counter == f) return SKV_ERR_OOM;
    if (cudaMalloc(p, bytes) != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        return SKV_ERR_OOM;
    }
    h->allocs.push_back(*p);
    return SKV_OK;
}
template <typename T>
int alloc_t(skv_layer* h, T** p, size_t count) {
    return alloc(h, reinterpret_cast<void**>(p), count * sizeof(T));
}

void free_all(skv_layer* h) {
    if (!h) return;
    for (void* p : h->allocs) cudaFree(p);
    h->allocs.clear();
    if (h->ev_sel) cudaEventDestroy(h->ev_sel);
    if (h->ev_fetch) cudaEventDestroy(h->ev_fetch);
    if (h->ev_start) cudaEventDestroy(h->ev_start);
    for (auto& a : h->prof_pending)
        for (auto e : a) cudaEventDestroy(e);
    for (auto& a : h->prof_free)
        for (auto e : a) cudaEventDestroy(e);
    h->prof_pending.clear();
    h->prof_free.clear();
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D byte tensor map (8-bit elements): rows of `cols` bytes, box = 128 bytes x box_rows,
// 128-byte swizzle.
int make_map_u8(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return SKV_ERR_CUDA;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SKV_OK : SKV_ERR_CUDA;
}

// 2-D bf16 tensor map: rows of `cols` elements, box = 64 columns x box_rows, 128-byte swizzle.
int make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return SKV_ERR_CUDA;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SKV_OK : SKV_ERR_CUDA;
}

bool is_device_ptr(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

int check_device_error(skv_layer* h) {
    int e[2] = {0, 0};
    if (cudaMemcpy(e, h->err, sizeof(e), cudaMemcpyDeviceToHost) != cudaSuccess) return SKV_ERR_CUDA;
    if (e[0] == DEV_ERR_TIMEOUT) return SKV_ERR_TIMEOUT;
    if (e[0] != 0) return SKV_ERR_DEVICE_BOUNDS;
    return SKV_OK;
}

// Algorithmic bytes of one decode step of one layer (every unit), given the
// number of missed chunks summed over units.
void step_bytes(const skv_config& c, int64_t t, double misses, double* hbm, double* link, double* scratch) {
    const double es = es_of(c.dtype), esl = es_l_of(c.dtype), esv = es_v_of(c.dtype);
    const double d = c.head_dim, r = c.rank, C = c.chunk, K = c.n_select, O = c.n_outlier;
    const double U = static_cast<double>(c.batch) * c.n_kv_heads, G = c.n_q_heads / c.n_kv_heads;
    const double n_c = static_cast<double>(c.seq_len) / C - O - c.local_window / C;
    const double loc = c.local_window + t + 1;
    // q and out, landmarks, the attended keys and values (outliers, cache, local), the append
    double h = U * d * (es * 2.0 * G + esl * n_c + (es + esv) * (O * C + K * C + loc + 1.0));
    h += misses * C * (es * r + es * d + esv * d);   // A rows read, K and V rows written into slots
    h += (misses > 0 ? U : 0.0) * es * r * d;        // B slices
    if (c.new_keys == SKV_NEWKEYS_LOWRANK) {
        // ShadowKV+: the projection reads k' instead of the append reading the key (no change)
        // and B (U r d) and writes a (b r); the new key reads a (U r) and B_h again (U r d)
        h += es * (2.0 * U * r * d + c.batch * r + U * r);
    }
    double l = misses * C * d * esv;                 // value rows over the host link
    if (c.v_place == SKV_V_HBM) {
        // values in HBM: the fp32 path copies missed rows into the value cache (one more read);
        // the tensor-core path's attention reads them in V, so no slot is written either
        if (c.dtype == SKV_F32) h += l;
        else h -= misses * C * esv * d;
        l = 0.0;
    }
    const double nsplit = std::ceil((O * C + K * C + loc) / attn_segment(c.dtype));
    *hbm = h;
    *link = l;
    *scratch = U * (2.0 * n_c * G * 4.0 + nsplit * G * (d + 4) * 4.0 * 2.0);
}

}  // namespace

extern "C" {

const char* shadowkv_strerror(int code) {
    switch (code) {
        case SKV_OK: return "ok";
        case SKV_ERR_INVALID: return "invalid argument or configuration";
        case SKV_ERR_OOM: return "device allocation failed";
        case SKV_ERR_NOT_PINNED: return "host values are not reachable by the GPU (not page-locked, no ATS)";
        case SKV_ERR_CUDA: return "CUDA call failed";
        case SKV_ERR_DEVICE_BOUNDS: return "a kernel met an out-of-range index";
        case SKV_ERR_TIMEOUT: return "a kernel wait timed out";
        case SKV_ERR_STEP_LIMIT: return "more decode steps than max_new_tokens";
        case SKV_ERR_UNSUPPORTED: return "unsupported on this device or shape";
        default: return "unknown error";
    }
}

int shadowkv_version(void) { return kVersion; }

int shadowkv_validate_config(const skv_config* c) {
    if (!c) return SKV_ERR_INVALID;
    if (c->batch < 1 || c->n_kv_heads < 1 || c->n_q_heads < 1) return SKV_ERR_INVALID;
    if (c->n_q_heads % c->n_kv_heads) return SKV_ERR_INVALID;
    const int G = c->n_q_heads / c->n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return SKV_ERR_INVALID;
    if (c->head_dim != kD || c->chunk != kC) return SKV_ERR_INVALID;
    if (c->rank < 8 || c->rank > 256 || c->rank % 8) return SKV_ERR_INVALID;
    if (c->seq_len < c->chunk || c->seq_len % c->chunk || c->seq_len > (int64_t(1) << 30)) return SKV_ERR_INVALID;
    if (c->local_window < 0 || c->local_window % c->chunk) return SKV_ERR_INVALID;
    if (c->n_outlier < 0 || c->n_select < 1 || c->n_select > 4096) return SKV_ERR_INVALID;
    if (c->max_new_tokens < 1 || c->max_new_tokens > (1 << 24)) return SKV_ERR_INVALID;
    const int64_t nchunk = c->seq_len / c->chunk;
    const int64_t n_c = nchunk - c->n_outlier - c->local_window / c->chunk;
    if (n_c < c->n_select) return SKV_ERR_INVALID;
    if (static_cast<int64_t>(c->batch) * c->seq_len > (int64_t(1) << 31) - 1) return SKV_ERR_INVALID;
    if (!(c->rope_base > 1.0) || !std::isfinite(c->rope_base)) return SKV_ERR_INVALID;
    if (c->dtype != SKV_F32 && c->dtype != SKV_BF16 && c->dtype != SKV_FP8) return SKV_ERR_INVALID;
    if (c->v_place != SKV_V_HBM && c->v_place != SKV_V_HOST) return SKV_ERR_INVALID;
    if (c->new_keys != SKV_NEWKEYS_EXACT && c->new_keys != SKV_NEWKEYS_LOWRANK) return SKV_ERR_INVALID;
    if (c->new_keys == SKV_NEWKEYS_LOWRANK && c->seq_len + c->max_new_tokens + kC > (int64_t(1) << 31) - 1)
        return SKV_ERR_INVALID;
    return SKV_OK;
}

int shadowkv_model(const skv_config* c, double alpha, int64_t t, double b_gpu_gbs, double b_link_gbs,
                   skv_model* out) {
    if (!out || shadowkv_validate_config(c) != SKV_OK) return SKV_ERR_INVALID;
    if (!(b_gpu_gbs > 0) || !(b_link_gbs > 0) || alpha < 0 || alpha > 1 || t < 0) return SKV_ERR_INVALID;
    const double S = static_cast<double>(c->seq_len), C = c->chunk, K = c->n_select, O = c->n_outlier;
    // M: width of one token's key across the KV heads (H d elements, 1024 for
    // Llama-3.1-8B) -- the reading under which the printed 7.08x is reproduced
    const double dall = static_cast<double>(c->head_dim) * c->n_kv_heads, r = c->rank, M = dall;
    out->eq_bandwidth_gbs =
        2.0 * S * b_gpu_gbs / (S / C + 2.0 * (K + O) * C + (1.0 - alpha) * K * C * b_gpu_gbs / b_link_gbs);
    out->memory_savings = 2.0 * S * M / (S * M / C + 2.0 * (K + O) * C + S * r + r * M);
    out->compression_ratio = S * dall / (r * (S + dall));
    const double U = static_cast<double>(c->batch) * c->n_kv_heads;
    double hbm, link, scratch;
    step_bytes(*c, t, (1.0 - alpha) * K * U, &hbm, &link, &scratch);
    out->hbm_bytes_per_step = hbm;
    out->link_bytes_per_step = link;
    out->t_pred_us = (hbm / (b_gpu_gbs * 1e9) + link / (b_link_gbs * 1e9)) * 1e6;
    return SKV_OK;
}

int shadowkv_prefill_index(const skv_config* cfg, const void* A, const void* B, const void* V, skv_stream stream,
                           skv_layer** out) {
    return shadowkv_prefill_index_keys(cfg, A, B, nullptr, V, stream, out);
}

int shadowkv_prefill_index_keys(const skv_config* cfg, const void* A, const void* B, const void* Kx, const void* V,
                                skv_stream stream, skv_layer** out) {
    NvtxRange call("shadowkv_prefill_index");
    if (!out) return SKV_ERR_INVALID;
    *out = nullptr;
    int rc = shadowkv_validate_config(cfg);
    if (rc) return rc;
    if (!A || !B || !V) return SKV_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(V) |
         reinterpret_cast<uintptr_t>(Kx)) & 15)
        return SKV_ERR_INVALID;
    cudaStream_t s = stream;
    skv_layer* h = new (std::nothrow) skv_layer();
    if (!h) return SKV_ERR_OOM;
    g_alloc_counter = 0;
    auto fail = [&](int code) {
        cudaStreamSynchronize(s);
        free_all(h);
        delete h;
        cudaGetLastError();
        return code;
    };
    const skv_config& c = *cfg;
    h->cfg = c;
    if (cudaGetDevice(&h->dev) != cudaSuccess) return fail(SKV_ERR_CUDA);
    int major = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, h->dev);
    cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->dev);
    if (major < 10) return fail(SKV_ERR_UNSUPPORTED);
    h->H = c.n_kv_heads;
    h->G = c.n_q_heads / c.n_kv_heads;
    h->U = c.batch * c.n_kv_heads;
    h->r = c.rank;
    h->K = c.n_select;
    h->O = c.n_outlier;
    h->W = c.local_window;
    h->Tmax = c.max_new_tokens;
    h->S = c.seq_len;
    h->nchunk = static_cast<int>(c.seq_len / kC);
    h->ncand = h->nchunk - h->W / kC;
    h->n_c = h->ncand - h->O;
    h->dtype = c.dtype;
    h->es = es_of(c.dtype);
    h->es_l = es_l_of(c.dtype);
    h->es_v = es_v_of(c.dtype);
    h->tc = c.dtype != SKV_F32;
    // with values in HBM the tensor-core attention reads a selected chunk's values where they
    // live: no copy into a value cache, and the attention follows the rebuild on one stream
    h->v_direct = h->tc && c.v_place == SKV_V_HBM;
    h->nkb = (h->r + 63) / 64;
    h->newkeys = c.new_keys;
    h->Tpad = (h->Tmax + kC - 1) / kC * kC;
    h->loc_cap = h->W + h->Tmax;
    // ShadowKV+ rotates generated keys at positions S .. S + max_new_tokens - 1 itself
    h->nhi = static_cast<int>((c.seq_len + (h->newkeys == SKV_NEWKEYS_LOWRANK ? h->Tmax : 0) + 255) / 256);
    h->A = A;
    h->B = B;
    h->V = V;
    if (!is_device_ptr(A) || !is_device_ptr(B) || (Kx && !is_device_ptr(Kx))) return fail(SKV_ERR_INVALID);
    if (c.v_place == SKV_V_HBM) {
        if (!is_device_ptr(V)) return fail(SKV_ERR_INVALID);
        h->Vd = V;
    } else {
        // page-locked host memory (mapped into the GPU's page tables), or, on
        // a device that reads pageable memory through the host's page tables
        // (Grace with NVLink-C2C), any system memory, e.g. shadowkv_host_alloc
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, V) != cudaSuccess) {
            cudaGetLastError();
            return fail(SKV_ERR_NOT_PINNED);
        }
        if (a.type == cudaMemoryTypeHost) {
            void* dp = nullptr;
            if (cudaHostGetDevicePointer(&dp, const_cast<void*>(V), 0) != cudaSuccess || !dp) {
                cudaGetLastError();
                return fail(SKV_ERR_NOT_PINNED);
            }
            h->Vd = dp;
        } else if (a.type == cudaMemoryTypeUnregistered) {
            int ats = 0;
            cudaDeviceGetAttribute(&ats, cudaDevAttrPageableMemoryAccessUsesHostPageTables, h->dev);
            if (!ats) return fail(SKV_ERR_NOT_PINNED);
            h->Vd = V;
        } else {
            return fail(SKV_ERR_NOT_PINNED);
        }
    }

    const int U = h->U, K = h->K, O = h->O, G = h->G, es = h->es;
    const size_t row = static_cast<size_t>(kD) * es;                 // a key (or bf16/fp32 value) row
    const size_t row_l = static_cast<size_t>(kD) * h->es_l;           // a landmark row
    const size_t row_v = static_cast<size_t>(kD) * h->es_v;           // a value row
    // scoring work: runs of kRunChunks landmarks of one unit; every CTA resident at once
    {
        h->score_nparts = score_parts(h->dtype);
        h->score_nru = (h->n_c + kRunChunks - 1) / kRunChunks;
        const int64_t runs = static_cast<int64_t>(U) * h->score_nru;
        const int cap = std::max(1, h->sm_count * score_ctas_per_sm(h->dtype, G));
        h->score_ncta = static_cast<int>(std::min<int64_t>(cap, runs));
    }
    h->sel_smem_cap = std::max(0, (200 * 1024 - 20 * K) / 4 - 4);

    const size_t nc = static_cast<size_t>(h->n_c);
    if ((rc = alloc(h, &h->L, U * nc * row_l)) || (rc = alloc_t(h, &h->ids, U * nc)) ||
        (rc = alloc_t(h, &h->out_ids, static_cast<size_t>(U) * std::max(O, 1))) ||
        (rc = alloc_t(h, &h->min_cos, static_cast<size_t>(U) * h->ncand)) ||
        (rc = alloc(h, &h->Kall, static_cast<size_t>(U) * (static_cast<size_t>(O + K) * kC + h->loc_cap) * row)) ||
        (rc = alloc(h, &h->Vall, static_cast<size_t>(U) * (static_cast<size_t>(O + K) * kC + h->loc_cap) * row_v)) ||
        (rc = alloc_t(h, &h->sel_ids[0], static_cast<size_t>(U) * K)) ||
        (rc = alloc_t(h, &h->sel_ids[1], static_cast<size_t>(U) * K)) ||
        (rc = alloc_t(h, &h->sel_slot[0], static_cast<size_t>(U) * K)) ||
        (rc = alloc_t(h, &h->sel_slot[1], static_cast<size_t>(U) * K)) ||
        (rc = alloc_t(h, &h->miss_chunk, static_cast<size_t>(U) * K)) ||
        (rc = alloc_t(h, &h->miss_slot, static_cast<size_t>(U) * K)) ||
        (rc = alloc_t(h, &h->miss_count, static_cast<size_t>(U))) ||
        (rc = alloc_t(h, &h->slot_chunk, static_cast<size_t>(U) * K)) ||
        (rc = alloc_t(h, &h->logits, U * nc * G)) ||
        (rc = alloc_t(h, &h->score_part, static_cast<size_t>(U) * h->score_nru * h->score_nparts * G)) ||
        (rc = alloc_t(h, &h->sched, 1)) ||
        (rc = alloc_t(h, &h->qt, static_cast<size_t>(U) * 3 * G * kD)) ||
        (h->newkeys == SKV_NEWKEYS_LOWRANK &&
         (rc = alloc(h, &h->Anew, static_cast<size_t>(c.batch) * h->Tpad * h->r * h->es))) ||
        (rc = alloc_t(h, &h->qinv, static_cast<size_t>(U) * G)) ||
        (rc = alloc_t(h, &h->vbuf, std::max(U * nc, static_cast<size_t>(U) * h->ncand))) ||
        (rc = alloc_t(h, &h->attn_cnt, static_cast<size_t>(U))) ||
        (rc = alloc_t(h, &h->rope_lo, static_cast<size_t>(256) * kD / 2)) ||
        (rc = alloc_t(h, &h->rope_hi, static_cast<size_t>(h->nhi) * kD / 2)) ||
        (rc = alloc_t(h, &h->hits_step, static_cast<size_t>(h->Tmax))) || (rc = alloc_t(h, &h->err, 4)))
        return fail(rc);
    h->R = static_cast<int64_t>(O + K) * kC + h->loc_cap;
    {
        uint8_t* kb = static_cast<uint8_t*>(h->Kall);
        uint8_t* vb = static_cast<uint8_t*>(h->Vall);
        const size_t c_rows = static_cast<size_t>(O) * kC, l_rows = static_cast<size_t>(O + K) * kC;
        h->Kout = kb; h->Kc = kb + c_rows * row; h->Kloc = kb + l_rows * row;
        h->Vout = vb; h->Vc = vb + c_rows * row_v; h->Vloc = vb + l_rows * row_v;
    }
    {
        const int ntot_max = O * kC + K * kC + h->loc_cap;
        const int seg = attn_segment(h->dtype);
        const int nsplit_max = (ntot_max + seg - 1) / seg;
        if ((rc = alloc_t(h, &h->attn_part, static_cast<size_t>(U) * nsplit_max * G * (kD + 4)))) return fail(rc);
    }
    void* Lfull = nullptr;
    if ((rc = alloc(h, &Lfull, static_cast<size_t>(U) * h->ncand * kD * 4))) return fail(rc);
    if (h->tc && (rc = alloc(h, &h->Bt, static_cast<size_t>(U) * h->r * kD * 2))) return fail(rc);
    if (cudaEventCreateWithFlags(&h->ev_sel, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_fetch, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_start, cudaEventDisableTiming) != cudaSuccess)
        return fail(SKV_ERR_CUDA);

    // RoPE tables in double precision: angle(pos) = (pos & 255)*theta + (pos >> 8)*256*theta
    {
        std::vector<float2> lo(256 * kD / 2), hi(static_cast<size_t>(h->nhi) * kD / 2);
        for (int i = 0; i < kD / 2; ++i) {
            const double th = std::pow(c.rope_base, -2.0 * i / kD);
            for (int p = 0; p < 256; ++p) {
                const double a = p * th;
                lo[p * (kD / 2) + i] = make_float2(static_cast<float>(std::cos(a)), static_cast<float>(std::sin(a)));
            }
            for (int q = 0; q < h->nhi; ++q) {
                const double a = (256.0 * q) * th;
                hi[static_cast<size_t>(q) * (kD / 2) + i] =
                    make_float2(static_cast<float>(std::cos(a)), static_cast<float>(std::sin(a)));
            }
        }
        if (cudaMemcpy(h->rope_lo, lo.data(), lo.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaMemcpy(h->rope_hi, hi.data(), hi.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess)
            return fail(SKV_ERR_CUDA);
    }
    cudaMemsetAsync(h->err, 0, 4 * sizeof(int), s);
    cudaMemsetAsync(h->attn_cnt, 0, U * sizeof(int32_t), s);
    cudaMemsetAsync(h->hits_step, 0, h->Tmax * sizeof(int32_t), s);
    cudaMemsetAsync(h->miss_count, 0, U * sizeof(int32_t), s);
    cudaMemsetAsync(h->sched, 0, sizeof(int32_t), s);
    if (h->Anew) cudaMemsetAsync(h->Anew, 0, static_cast<size_t>(c.batch) * h->Tpad * h->r * h->es, s);
    if (h->tc) {
        if (launch_transpose_B(B, h->Bt, U, h->r, s)) return fail(SKV_ERR_CUDA);
        if ((rc = make_map(&h->tmA, A, h->r, static_cast<uint64_t>(c.batch) * c.seq_len, 8)) ||
            (rc = make_map(&h->tmB, h->Bt, h->r, static_cast<uint64_t>(U) * kD, 128)) ||
            (rc = h->dtype == SKV_FP8 ? make_map_u8(&h->tmL, h->L, kD, static_cast<uint64_t>(U) * h->n_c, kScTile)
                                      : make_map(&h->tmL, h->L, kD, static_cast<uint64_t>(U) * h->n_c, kScTile)) ||
            (rc = make_map(&h->tmKall, h->Kall, kD, static_cast<uint64_t>(U) * h->R, 128)))
            return fail(rc);
    }

    // base parameters of the rebuild kernel
    RebuildParams rp{};
    rp.U = U; rp.H = h->H; rp.r = h->r; rp.nkb = h->nkb; rp.S = h->S; rp.nchunk = h->nchunk;
    rp.rope_lo = h->rope_lo; rp.rope_hi = h->rope_hi; rp.nhi = h->nhi;
    rp.A = A; rp.B = B; rp.err = h->err;
    rp.Kx = Kx; rp.kx_es = h->es;
    // K_RoPE: the exact keys' rotation when the caller has them, else the factors' keys
    auto rebuild = [&](const RebuildParams& p, int count_max) -> int {
        const int gx = (count_max + kTileChunks - 1) / kTileChunks;
        if (gx <= 0) return 0;
        if (Kx) return launch_keys_exact(p, gx, h->dtype != SKV_F32, s);
        return h->tc ? launch_rebuild_tc(&h->tmA, &h->tmB, p, gx, s) : launch_rebuild_f32(p, gx, s);
    };
    // 1. landmarks and min-cos of every candidate chunk (Algorithm 1: Reduce, CosineSimilarity, Min)
    {
        RebuildParams p = rp;
        p.mode = 1; p.list = nullptr; p.list_base = 0; p.list_cap = h->ncand; p.count_const = h->ncand;
        p.Lfull = static_cast<float*>(Lfull); p.mcos = h->min_cos; p.stats_us = h->ncand;
        if (rebuild(p, h->ncand)) return fail(SKV_ERR_CUDA);
    }
    // 2. outliers: the O lowest min-cos (ArgTopK(-Min(S), o)), ascending
    if (O > 0) {
        SelectParams sp{};
        sp.n = h->ncand; sp.k = O; sp.U = U; sp.H = h->H; sp.G = G;
        sp.neg_src = h->min_cos; sp.vbuf = h->vbuf; sp.smem_cap = h->sel_smem_cap; sp.sel_plain = h->out_ids;
        sp.err = h->err;
        if (launch_select_outliers(sp, s)) return fail(SKV_ERR_CUDA);
    }
    // 3. L = C \ Gather(C, I): compact the landmarks and their chunk ids
    {
        CompactParams cp{};
        cp.Lfull = static_cast<const float*>(Lfull); cp.ncand = h->ncand; cp.out_ids = h->out_ids; cp.O = O;
        cp.L = h->L; cp.ids = h->ids; cp.n_c = h->n_c; cp.U = U; cp.dtype = h->dtype; cp.err = h->err;
        if (launch_compact(cp, s)) return fail(SKV_ERR_CUDA);
    }
    // 4. K_outlier and the local window's keys, rebuilt; 5. their values, gathered
    {
        RebuildParams p = rp;
        p.mode = 0;
        if (O > 0) {
            p.list = h->out_ids; p.list_us = O; p.list_cap = O; p.count_const = O;
            p.dst = h->Kout; p.dst_cap = O; p.dst_us = h->R * kD;
            if (rebuild(p, O)) return fail(SKV_ERR_CUDA);
        }
        const int nloc = h->W / kC;
        if (nloc > 0) {
            p.list = nullptr; p.list_base = h->ncand; p.list_cap = nloc; p.count_const = nloc;
            p.dst = h->Kloc; p.dst_cap = h->loc_cap / kC; p.dst_us = h->R * kD;
            if (rebuild(p, nloc)) return fail(SKV_ERR_CUDA);
        }
        GatherParams g{};
        g.src = h->Vd; g.src_us = h->S * kD; g.nchunk = h->nchunk; g.es = h->es_v; g.U = U; g.err = h->err;
        if (O > 0) {
            GatherParams go = g;
            go.list = h->out_ids; go.list_us = O; go.list_cap = O; go.count_const = O; go.dst_cap = O;
            go.dst = h->Vout; go.dst_us = h->R * kD;
            if (launch_gather(go, (O + 7) / 8, s)) return fail(SKV_ERR_CUDA);
        }
        if (nloc > 0) {
            GatherParams gl = g;
            gl.list = nullptr; gl.list_base = h->ncand; gl.list_cap = nloc; gl.count_const = nloc;
            gl.dst = h->Vloc; gl.dst_cap = h->loc_cap / kC; gl.dst_us = h->R * kD;
            if (launch_gather(gl, (nloc + 7) / 8, s)) return fail(SKV_ERR_CUDA);
        }
    }
    if (cudaStreamSynchronize(s) != cudaSuccess) return fail(SKV_ERR_CUDA);
    if ((rc = check_device_error(h))) return fail(rc);
    if (c.v_place == SKV_V_HOST) {
        // values in a huge-page arena: pre-filling splits some of its huge pages (measured: about
        // ten of 128 over a 64 GiB arena, for reasons inside the host kernel and the driver);
        // put this layer's pages back together before the decode steps read them (best effort)
        const size_t vbytes = static_cast<size_t>(U) * static_cast<size_t>(c.seq_len) * kD * h->es_v;
        bool huge = false;
        {
            std::lock_guard<std::mutex> lock(g_host_mu);
            huge = find_host_map(V, vbytes) != nullptr;
        }
        if (huge) shadowkv_host_repair(const_cast<void*>(V), vbytes);
        h->v_huge = huge;
    }
    // the full landmark table is only needed during pre-filling
    cudaFree(Lfull);
    h->allocs.erase(std::find(h->allocs.begin(), h->allocs.end(), Lfull));
    *out = h;
    return SKV_OK;
}

int shadowkv_decode_step(skv_layer* h, const void* q, const void* k_new, const void* v_new, void* out,
                         int32_t* sel_out, skv_stream main, skv_stream side) {
    NvtxRange call("shadowkv_decode_step");
    if (!h || !q || !k_new || !v_new || !out) return SKV_ERR_INVALID;
    if (h->t >= h->Tmax) return SKV_ERR_STEP_LIMIT;
    if (h->v_huge && h->t == 0) {
        std::lock_guard<std::mutex> lock(g_host_mu);
        if (!g_host_maps.empty()) g_keeper.start();
    }
    cudaStream_t sm = main;
    cudaStream_t ss = (side == nullptr || side == main) ? main : side;
    h->last_main = sm;
    h->last_side = ss;
    h->stepped = true;
    const int t = static_cast<int>(h->t);
    const int U = h->U, K = h->K, G = h->G;
    std::array<cudaEvent_t, 8> ev{};
    if (h->profiling) {
        if (h->prof_free.empty()) {
            for (auto& e : ev) cudaEventCreate(&e);
        } else {
            ev = h->prof_free.back();
            h->prof_free.pop_back();
        }
        cudaEventRecord(ev[0], sm);
    }
    if (h->newkeys == SKV_NEWKEYS_LOWRANK) {
        // ShadowKV+: keep the new token as a = k'.Psi and write its key RoPE_{S+t}(a . B_h) into
        // local row W + t.  A generated token's key depends only on its fixed rank-r state, so
        // the rows of earlier generated tokens stay valid: the local rows cache the rebuilt
        // keys as the cache slots do for context chunks.  This needs only k_new, so it runs on
        // the side stream beside scoring and selection; attention waits for the side stream.
        if (ss != sm) {
            cudaEventRecord(h->ev_start, sm);
            cudaStreamWaitEvent(ss, h->ev_start, 0);
        }
        PlusParams pp{};
        pp.k_new = k_new; pp.B = h->B; pp.a_new = h->Anew; pp.k_loc = h->Kloc;
        pp.rope_lo = h->rope_lo; pp.rope_hi = h->rope_hi;
        pp.H = h->H; pp.r = h->r; pp.t = t;
        pp.a_rows = h->Tpad; pp.pos = h->S + t; pp.loc_pitch = h->R; pp.loc_row = h->W + t;
        if (launch_plus_append(h->dtype == SKV_F32 ? 0 : 1, pp, U / h->H, ss)) return SKV_ERR_CUDA;
    }
    NvtxRange ph_score("a2 landmark scoring");
    // a2: landmark scoring
    ScoreParams sp{};
    sp.L = h->L; sp.q = q; sp.logits = h->logits; sp.part = h->score_part; sp.n_c = h->n_c;
    sp.nru = h->score_nru; sp.total_runs = U * h->score_nru; sp.nparts = h->score_nparts; sp.sched = h->sched;
    sp.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(kD))); sp.err = h->err;
    sp.qt = h->qt; sp.qinv = h->qinv;
    if (h->dtype == SKV_FP8 && launch_qsplit(q, h->qt, h->qinv, U, G, sm)) return SKV_ERR_CUDA;
    if (launch_score(h->dtype, G, &h->tmL, sp, h->score_ncta, sm)) return SKV_ERR_CUDA;
    if (h->profiling) cudaEventRecord(ev[1], sm);
    ph_score.end();
    NvtxRange ph_select("a3-a4 selection, index scan, append");
    // a3 + a4 + a1: top-K, index scan, append
    SelectParams sel{};
    sel.n = h->n_c; sel.k = K; sel.U = U; sel.H = h->H; sel.G = G;
    sel.logits = h->logits; sel.part = h->score_part; sel.nru = h->score_nru; sel.nparts = h->score_nparts;
    sel.sched = h->sched; sel.vbuf = h->vbuf; sel.smem_cap = h->sel_smem_cap; sel.ids = h->ids;
    sel.nsm = h->sm_count;
    sel.sel_out_user = sel_out; sel.t = t;
    sel.prev_ids = h->sel_ids[t & 1]; sel.prev_slot = h->sel_slot[t & 1];
    sel.cur_ids = h->sel_ids[(t + 1) & 1]; sel.cur_slot = h->sel_slot[(t + 1) & 1];
    sel.miss_chunk = h->miss_chunk; sel.miss_slot = h->miss_slot; sel.miss_count = h->miss_count;
    sel.slot_chunk = h->slot_chunk;
    sel.hits_step = h->hits_step; sel.k_new = h->newkeys == SKV_NEWKEYS_LOWRANK ? nullptr : k_new; sel.v_new = v_new; sel.k_loc = h->Kloc; sel.v_loc = h->Vloc;
    sel.loc_cap = h->loc_cap; sel.loc_pitch = h->R; sel.W = h->W; sel.es = h->es; sel.es_v = h->es_v;
    sel.err = h->err;
    if (launch_select_decode(h->dtype, sel, sm)) return SKV_ERR_CUDA;
    if (h->user_sel && cudaEventRecord(h->user_sel, sm) != cudaSuccess) {
        cudaGetLastError();
        return SKV_ERR_CUDA;
    }
    if (h->profiling) cudaEventRecord(ev[2], sm);
    ph_select.end();
    NvtxRange ph_fetch("a6 value fetch");
    // a6 on the side stream: value rows of the missed chunks into their slots.  With values in
    // HBM on the tensor-core path there is nothing to move: attention reads them in V.
    // side_pending: the side stream holds work attention must wait for
    const bool side_pending = ss != sm && (!h->v_direct || h->newkeys == SKV_NEWKEYS_LOWRANK);
    if (!h->v_direct) {
        if (ss != sm) {
            cudaEventRecord(h->ev_sel, sm);
            cudaStreamWaitEvent(ss, h->ev_sel, 0);
        }
        if (h->profiling) cudaEventRecord(ev[5], ss);
        GatherParams g{};
        g.src = h->Vd; g.src_us = h->S * kD; g.list = h->miss_chunk; g.list_us = K; g.list_cap = K;
        g.cnt = h->miss_count; g.dst_idx = h->miss_slot; g.dst_cap = K; g.dst = h->Vc;
        g.dst_us = h->R * kD; g.nchunk = h->nchunk; g.es = h->es_v; g.U = U; g.err = h->err;
        const int frc = launch_fetch2(g, K, ss);
        if (frc) return SKV_ERR_CUDA;
        if (h->profiling) cudaEventRecord(ev[6], ss);
    }
    if (side_pending) cudaEventRecord(h->ev_fetch, ss);
    // values read in place and only ShadowKV+'s small new-key work on the side stream: wait for
    // it before the rebuild, so that the attention still follows the rebuild directly
    const bool wait_early = side_pending && h->v_direct;
    if (wait_early) cudaStreamWaitEvent(sm, h->ev_fetch, 0);
    ph_fetch.end();
    NvtxRange ph_rebuild("a5 key rebuild");
    // a5 on the main stream: rebuild + RoPE of the missed chunks' keys (timed from its own
    // launch, which with a single stream comes after the fetch)
    if (h->profiling) cudaEventRecord(ev[7], sm);
    RebuildParams rp{};
    rp.mode = 0; rp.U = U; rp.H = h->H; rp.r = h->r; rp.nkb = h->nkb; rp.S = h->S; rp.nchunk = h->nchunk;
    rp.list = h->miss_chunk; rp.list_us = K; rp.list_cap = K; rp.cnt = h->miss_count; rp.dst_idx = h->miss_slot;
    rp.dst_cap = K; rp.dst = h->Kc; rp.dst_us = h->R * kD;
    rp.rope_lo = h->rope_lo; rp.rope_hi = h->rope_hi; rp.nhi = h->nhi; rp.A = h->A; rp.B = h->B; rp.err = h->err;
    const int gx = (K + kTileChunks - 1) / kTileChunks;
    const int rc = h->tc ? launch_rebuild_tc(&h->tmA, &h->tmB, rp, gx, sm) : launch_rebuild_f32(rp, gx, sm);
    if (rc) return SKV_ERR_CUDA;
    if (h->profiling) cudaEventRecord(ev[3], sm);
    if (side_pending && !wait_early) cudaStreamWaitEvent(sm, h->ev_fetch, 0);
    ph_rebuild.end();
    NvtxRange ph_attn("a7 sparse attention");
    // a7: attention over outliers + cache + local, split-K with a dependent merge kernel
    AttnParams ap{};
    ap.q = q; ap.k_out = h->Kout; ap.v_out = h->Vout; ap.n_out = h->O * kC;
    ap.k_c = h->Kc; ap.v_c = h->Vc; ap.n_cache = K * kC;
    ap.k_loc = h->Kloc; ap.v_loc = h->Vloc; ap.n_loc = h->W + t + 1; ap.loc_cap = h->loc_cap;
    ap.unit_rows = h->R;
    ap.out = out; ap.part = h->attn_part; ap.counter = h->attn_cnt;
    const int seg = attn_segment(h->dtype);
    ap.nsplit = (ap.n_out + ap.n_cache + ap.n_loc + seg - 1) / seg;
    ap.scale = sp.scale; ap.G = G; ap.U = U; ap.err = h->err;
    ap.v_es = h->es_v;
    if (h->v_direct) {
        ap.v_src = h->Vd; ap.v_src_us = h->S * kD; ap.slot_chunk = h->slot_chunk; ap.nchunk = h->nchunk;
        ap.pdl = 1;   // a programmatic dependent of the rebuild, on one stream
    }
    const int na = h->tc ? launch_attn_tc(&h->tmKall, ap, h->sm_count, sm) : (launch_attn(h->dtype, ap, sm) ? -1 : 1);
    if (na < 0) return SKV_ERR_CUDA;
    // score, select, fetch (not with values read in place), rebuild, attention (+ its merge); the
    // e5m2 query split; ShadowKV+'s projection and new key
    h->launches += (h->v_direct ? 3 : 4) + na + (h->dtype == SKV_FP8 ? 1 : 0) +
                   (h->newkeys == SKV_NEWKEYS_LOWRANK ? 2 : 0);
    if (h->profiling) {
        cudaEventRecord(ev[4], sm);
        h->prof_pending.push_back(ev);
    }
    ++h->t;
    return SKV_OK;
}

int shadowkv_set_select_event(skv_layer* h, void* event) {
    if (!h) return SKV_ERR_INVALID;
    h->user_sel = static_cast<cudaEvent_t>(event);
    return SKV_OK;
}

int shadowkv_set_profiling(skv_layer* h, int enable) {
    if (!h) return SKV_ERR_INVALID;
    h->profiling = enable != 0;
    return SKV_OK;
}

int shadowkv_stats(skv_layer* h, skv_stats* out) {
    if (!h || !out) return SKV_ERR_INVALID;
    std::memset(out, 0, sizeof(*out));
    if (h->stepped) {
        cudaStreamSynchronize(h->last_main);
        if (h->last_side != h->last_main) cudaStreamSynchronize(h->last_side);
    }
    // phase times
    for (auto& ev : h->prof_pending) {
        float ms = 0.f;
        const int pairs[SKV_NPHASE][2] = {{0, 1}, {1, 2}, {7, 3}, {5, 6}, {3, 4}};
        for (int ph = 0; ph < SKV_NPHASE; ++ph) {
            if (cudaEventElapsedTime(&ms, ev[pairs[ph][0]], ev[pairs[ph][1]]) == cudaSuccess) {
                h->phase_ms[ph] += ms;
                h->phase_n[ph] += 1;
            } else {
                cudaGetLastError();
            }
        }
        h->prof_free.push_back(ev);
    }
    h->prof_pending.clear();
    std::vector<int32_t> hits(static_cast<size_t>(h->Tmax));
    if (cudaMemcpy(hits.data(), h->hits_step, hits.size() * sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SKV_ERR_CUDA;
    const double per_step = static_cast<double>(h->U) * h->K;
    out->steps = h->t - h->t_reset;
    out->units = h->U;
    out->n_select = h->K;
    double asum = 0.0;
    int64_t an = 0;
    for (int64_t t = h->t_reset; t < h->t; ++t) {
        const double hi = hits[static_cast<size_t>(t)];
        out->hits += static_cast<int64_t>(hi);
        out->misses += static_cast<int64_t>(per_step - hi);
        out->alpha_last = hi / per_step;
        if (t >= 1) { asum += hi / per_step; ++an; }
        double hb, lb, sb;
        step_bytes(h->cfg, t, per_step - hi, &hb, &lb, &sb);
        out->hbm_bytes += hb;
        out->link_bytes += lb;
        out->scratch_bytes += sb;
    }
    out->alpha_mean = an ? asum / an : 0.0;
    for (int ph = 0; ph < SKV_NPHASE; ++ph) {
        out->phase_ms[ph] = h->phase_ms[ph];
        out->phase_launches[ph] = h->phase_n[ph];
    }
    const int e = check_device_error(h);
    out->device_error = (e == SKV_ERR_DEVICE_BOUNDS || e == SKV_ERR_TIMEOUT) ? e : 0;
    out->kernel_launches = h->launches;
    return e;
}

int shadowkv_reset_stats(skv_layer* h) {
    if (!h) return SKV_ERR_INVALID;
    skv_stats tmp;
    shadowkv_stats(h, &tmp);
    h->t_reset = h->t;
    h->launches = 0;
    for (int ph = 0; ph < SKV_NPHASE; ++ph) { h->phase_ms[ph] = 0; h->phase_n[ph] = 0; }
    return SKV_OK;
}

int64_t shadowkv_export_size(const skv_layer* h, int field) {
    if (!h) return -1;
    const int64_t U = h->U, row = static_cast<int64_t>(kD) * h->es, row_v = static_cast<int64_t>(kD) * h->es_v;
    switch (field) {
        case SKV_F_LANDMARKS: return U * h->n_c * kD * h->es_l;
        case SKV_F_CHUNK_IDS: return U * h->n_c * 4;
        case SKV_F_OUTLIER_IDS: return U * h->O * 4;
        case SKV_F_MIN_COS: return U * h->ncand * 4;
        case SKV_F_K_OUTLIER: return U * h->O * kC * row;
        case SKV_F_V_OUTLIER: return U * h->O * kC * row_v;
        case SKV_F_K_LOCAL: return U * (h->W + h->Tmax) * row;
        case SKV_F_V_LOCAL: return U * (h->W + h->Tmax) * row_v;
        case SKV_F_K_CACHE: return U * h->K * kC * row;
        case SKV_F_V_CACHE: return U * h->K * kC * row_v;
        case SKV_F_SELECTION:
        case SKV_F_SLOT_OF_SEL: return U * h->K * 4;
        case SKV_F_MISS_COUNT: return U * 4;
        case SKV_F_HITS_PER_STEP: return static_cast<int64_t>(h->Tmax) * 4;
        case SKV_F_A_NEW:
            return h->Anew ? static_cast<int64_t>(U / h->H) * h->Tmax * h->r * h->es : 0;
        default: return -1;
    }
}

int shadowkv_export(skv_layer* h, int field, void* dst, size_t bytes, skv_stream stream) {
    const int64_t need = shadowkv_export_size(h, field);
    if (need < 0 || !dst || static_cast<int64_t>(bytes) < need) return SKV_ERR_INVALID;
    const void* src = nullptr;
    const int cur = static_cast<int>(h->t & 1);
    switch (field) {
        case SKV_F_LANDMARKS: src = h->L; break;
        case SKV_F_CHUNK_IDS: src = h->ids; break;
        case SKV_F_OUTLIER_IDS: src = h->out_ids; break;
        case SKV_F_MIN_COS: src = h->min_cos; break;
        case SKV_F_K_OUTLIER: src = h->Kout; break;
        case SKV_F_V_OUTLIER: src = h->Vout; break;
        case SKV_F_K_LOCAL: src = h->Kloc; break;
        case SKV_F_V_LOCAL: src = h->Vloc; break;
        case SKV_F_K_CACHE: src = h->Kc; break;
        case SKV_F_V_CACHE: src = h->Vc; break;
        case SKV_F_SELECTION: src = h->sel_ids[cur]; break;
        case SKV_F_SLOT_OF_SEL: src = h->sel_slot[cur]; break;
        case SKV_F_MISS_COUNT: src = h->miss_count; break;
        case SKV_F_HITS_PER_STEP: src = h->hits_step; break;
        case SKV_F_A_NEW: src = h->Anew; break;
    }
    if (need == 0) return SKV_OK;
    if (field == SKV_F_V_CACHE && h->v_direct) {
        // values read in place: the rows attention reads for each slot, gathered from V by the
        // slot's chunk
        if (!is_device_ptr(dst)) return SKV_ERR_INVALID;
        GatherParams g{};
        g.src = h->Vd; g.src_us = h->S * kD; g.list = h->slot_chunk; g.list_us = h->K; g.list_cap = h->K;
        g.cnt = nullptr; g.count_const = h->K; g.dst_idx = nullptr; g.dst_cap = h->K; g.dst = dst;
        g.dst_us = static_cast<int64_t>(h->K) * kC * kD; g.nchunk = h->nchunk; g.es = h->es_v; g.U = h->U;
        g.err = h->err;
        return launch_gather(g, (h->K + 7) / 8, stream) ? SKV_ERR_CUDA : SKV_OK;
    }
    // fields inside the per-unit key/value blocks: [U][rows][d] out of rows of pitch R
    int64_t rows = 0;
    switch (field) {
        case SKV_F_K_OUTLIER: case SKV_F_V_OUTLIER: rows = static_cast<int64_t>(h->O) * kC; break;
        case SKV_F_K_LOCAL: case SKV_F_V_LOCAL: rows = h->W + h->Tmax; break;
        case SKV_F_K_CACHE: case SKV_F_V_CACHE: rows = static_cast<int64_t>(h->K) * kC; break;
    }
    if (field == SKV_F_A_NEW) {   // [b][Tmax][r] out of [b][Tpad][r]
        const size_t rb = static_cast<size_t>(h->Tmax) * h->r * h->es;
        if (cudaMemcpy2DAsync(dst, rb, src, static_cast<size_t>(h->Tpad) * h->r * h->es, rb, h->U / h->H,
                              cudaMemcpyDefault, stream) != cudaSuccess) {
            cudaGetLastError();
            return SKV_ERR_CUDA;
        }
        return SKV_OK;
    }
    if (rows > 0) {
        const bool vfield = field == SKV_F_V_OUTLIER || field == SKV_F_V_LOCAL || field == SKV_F_V_CACHE;
        const size_t rb = static_cast<size_t>(kD) * (vfield ? h->es_v : h->es);
        if (cudaMemcpy2DAsync(dst, rows * rb, src, h->R * rb, rows * rb, h->U, cudaMemcpyDefault, stream) != cudaSuccess) {
            cudaGetLastError();
            return SKV_ERR_CUDA;
        }
        return SKV_OK;
    }
    if (cudaMemcpyAsync(dst, src, static_cast<size_t>(need), cudaMemcpyDefault, stream) != cudaSuccess) {
        cudaGetLastError();
        return SKV_ERR_CUDA;
    }
    return SKV_OK;
}

int shadowkv_host_alloc(size_t bytes, void** out) { return shadowkv_host_alloc_kind(bytes, SKV_HOST_PINNED, out); }

int shadowkv_host_alloc_kind(size_t bytes, int kind, void** out) {
    if (!out || bytes == 0) return SKV_ERR_INVALID;
    *out = nullptr;
    if (kind == SKV_HOST_PINNED) {
        void* p = nullptr;
        if (cudaHostAlloc(&p, bytes, cudaHostAllocPortable | cudaHostAllocMapped) != cudaSuccess || !p) {
            cudaGetLastError();
            return SKV_ERR_OOM;
        }
        *out = p;
        return SKV_OK;
    }
    if (kind != SKV_HOST_HUGE) return SKV_ERR_INVALID;
    // pageable memory in transparent huge pages, read by the GPU through the host's page
    // tables: needs a device that does that (Grace with NVLink-C2C)
    int dev = 0, ats = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&ats, cudaDevAttrPageableMemoryAccessUsesHostPageTables, dev) != cudaSuccess) {
        cudaGetLastError();
        return SKV_ERR_CUDA;
    }
    if (!ats) return SKV_ERR_UNSUPPORTED;
    const size_t hp = host_huge_page_bytes();
    if (bytes > SIZE_MAX - 2 * hp) return SKV_ERR_INVALID;
    const size_t len = (bytes + hp - 1) / hp * hp;
    void* raw = mmap(nullptr, len + hp, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS | MAP_NORESERVE, -1, 0);
    if (raw == MAP_FAILED) return SKV_ERR_OOM;
    void* p = reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(raw) + hp - 1) / hp * hp);
    // huge pages: one translation covers a whole page, so the fetch's scattered reads over a
    // span of tens of GiB keep their translations.  Preferred location host: the driver does
    // not migrate these pages toward the GPU on its access counts.  Measured on a 64 GiB arena
    // over 20 decode steps: with this hint alone no huge page split; adding "accessed by" the
    // device, or giving no hint, split 8-10 of the 128 pages and slowed the fetch.
    cudaMemLocation host{};
    host.type = cudaMemLocationTypeHost;
    host.id = 0;
    if (madvise(p, len, MADV_HUGEPAGE) != 0 ||
        cudaMemAdvise(p, len, cudaMemAdviseSetPreferredLocation, host) != cudaSuccess) {
        cudaGetLastError();
        munmap(raw, len + hp);
        return SKV_ERR_CUDA;
    }
    {
        std::lock_guard<std::mutex> lock(g_host_mu);
        g_host_maps.push_back({p, len, raw, len + hp});
    }
    *out = p;
    return SKV_OK;
}

int shadowkv_host_repair(void* p, size_t bytes) {
    if (!p || bytes == 0) return SKV_ERR_INVALID;
    uintptr_t a = 0, e = 0;
    {
        std::lock_guard<std::mutex> lock(g_host_mu);
        if (!find_host_map(p, bytes)) return SKV_ERR_INVALID;
        const size_t hp = host_huge_page_bytes();
        a = reinterpret_cast<uintptr_t>(p) / hp * hp;
        e = (reinterpret_cast<uintptr_t>(p) + bytes + hp - 1) / hp * hp;
    }
    if (madvise(reinterpret_cast<void*>(a), e - a, MADV_COLLAPSE) != 0) {
        if (errno == EINVAL) return SKV_ERR_UNSUPPORTED;
        return errno == ENOMEM || errno == EAGAIN ? SKV_ERR_OOM : SKV_ERR_INVALID;
    }
    return SKV_OK;
}

void shadowkv_host_free(void* p) {
    if (!p) return;
    bool last = false, found = false;
    {
        std::lock_guard<std::mutex> lock(g_host_mu);
        for (size_t i = 0; i < g_host_maps.size(); ++i)
            if (g_host_maps[i].user == p) {
                munmap(g_host_maps[i].raw, g_host_maps[i].len);
                g_host_maps.erase(g_host_maps.begin() + static_cast<long>(i));
                found = true;
                last = g_host_maps.empty();
                break;
            }
    }
    if (last) g_keeper.halt();   // outside the lock: the keeper takes it
    if (!found) cudaFreeHost(p);
}

void shadowkv_destroy(skv_layer* h) {
    if (!h) return;
    if (h->stepped) {
        cudaStreamSynchronize(h->last_main);
        if (h->last_side != h->last_main) cudaStreamSynchronize(h->last_side);
    }
    free_all(h);
    delete h;
}

}  // extern "C"
