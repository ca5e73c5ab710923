/*
 * shadowkv.h — C ABI of the ShadowKV decode-step sparse attention library
 * (libshadowkv.so, sm_103a / GB300).
 *
 * The method: "ShadowKV: KV Cache in Shadows for High-Throughput Long-Context
 * LLM Inference".  The calls map one to one onto the two algorithms of the
 * Chinese digest of that paper (section A2): Algorithm 1 (pre-filling) is
 * shadowkv_prefill_index, Algorithm 2 (decoding) is shadowkv_decode_step.
 * The analytical models (equivalent bandwidth, memory savings, compression
 * ratio) are those of the English summary, section 3.4 and the appendix A.2
 * memory-savings formula.
 *
 * Conventions for every call:
 *  - All tensors are dense row-major in the storage dtype of the config
 *    (float32 or bfloat16), 16-byte aligned.  "dev" marks device memory of the
 *    current CUDA device; "host" marks page-locked host memory.
 *  - Nothing throws across this ABI.  Every int-returning call returns
 *    SKV_OK (0) or one of the negative SKV_ERR_* codes below.
 *  - Calls that take streams enqueue work and return; they do not
 *    synchronise unless stated.  A handle must not be used from two host
 *    threads at once.
 *  - Kernels that index with chunk ids, slots or positions range-check them;
 *    a failed check sets a device error word and skips the access.  The word
 *    is read (with a synchronisation) by shadowkv_stats, which then returns
 *    SKV_ERR_DEVICE_BOUNDS or SKV_ERR_TIMEOUT.
 */
#ifndef SHADOWKV_H
#define SHADOWKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Error codes. */
#define SKV_OK                 0
#define SKV_ERR_INVALID       -1  /* bad config, null or misaligned pointer, bad handle */
#define SKV_ERR_OOM           -2  /* device allocation failed (all partial state freed) */
#define SKV_ERR_NOT_PINNED    -3  /* v_place = host but V is not page-locked host memory */
#define SKV_ERR_CUDA          -4  /* a CUDA runtime/driver call failed */
#define SKV_ERR_DEVICE_BOUNDS -5  /* a kernel met an out-of-range index (access skipped) */
#define SKV_ERR_TIMEOUT       -6  /* a kernel's bounded wait ran out (work abandoned) */
#define SKV_ERR_STEP_LIMIT    -7  /* more decode steps than max_new_tokens */
#define SKV_ERR_UNSUPPORTED   -8  /* valid for the method, not built for this device/shape */

/* A CUDA stream (cudaStream_t) without pulling in the CUDA headers. */
typedef struct CUstream_st* skv_stream;

/*
 * SKV_FP8: the configuration the summary page's precision study runs with
 * float8 e5m2 (section 5, "Precision sensitivity"): the landmarks the library
 * builds and the values V (handed in as e5m2 bytes) are stored in e5m2; A, B,
 * q, k_new, v_new, the keys and out stay bf16.  Scores stay bf16-exact (the
 * query is split into three e5m2 terms for the 8-bit tensor-core product).
 */
typedef enum { SKV_F32 = 0, SKV_BF16 = 1, SKV_FP8 = 2 } skv_dtype;
typedef enum { SKV_V_HBM = 0, SKV_V_HOST = 1 } skv_vplace;

/*
 * How the keys of generated tokens are kept.
 * SKV_NEWKEYS_EXACT: each decode step's k_new (post-RoPE) joins the exact local
 *   set as it is.
 * SKV_NEWKEYS_LOWRANK: ShadowKV+ (summary page, "The ShadowKV+ extension for
 *   generated tokens"; digest section A7 on newly generated tokens).  k_new is
 *   the PRE-RoPE key; the library keeps its rank-r state a = k'.Psi, where k'
 *   [H*d] is the token's key over the H heads of its batch element and
 *   Psi = B^T (B_b read as [r][H*d]), stored like A, and attends with the key
 *   rebuilt from the stored state, RoPE_{S+t}(a . B[b][h]) -- the same
 *   reconstruction as for context keys, made once when the token arrives and
 *   kept in the local rows as rebuilt context keys are kept in cache slots.
 *   For a true projection B_b's rows should be orthonormal (B = Psi^T from the
 *   SVD); the library does not check.
 */
typedef enum { SKV_NEWKEYS_EXACT = 0, SKV_NEWKEYS_LOWRANK = 1 } skv_newkeys;

/*
 * Sizes of one layer.  Notation of the pages: b batch, H KV heads, G = n_q/H
 * query heads per KV head, d head dim, r rank, C chunk, K selected chunks,
 * O outlier chunks, W local-window tokens, S context length.
 * Requirements: d = 128, C = 8, G in {1, 2, 4, 8}, n_q = G*H, S % C == 0,
 * W % C == 0, n_c = S/C - O - W/C >= K >= 1, O >= 0, 8 <= r <= 256 and
 * r % 8 == 0, max_new_tokens >= 1.
 */
typedef struct {
    int32_t batch;          /* b */
    int32_t n_kv_heads;     /* H */
    int32_t n_q_heads;      /* H*G */
    int32_t head_dim;       /* d */
    int32_t rank;           /* r, A is shared by the H heads of one batch element */
    int32_t chunk;          /* C */
    int32_t n_select;       /* K chunks selected per KV head and step */
    int32_t n_outlier;      /* O static outlier chunks per KV head */
    int32_t local_window;   /* W prefill tokens kept exact (plus every decode token) */
    int32_t max_new_tokens; /* decode steps the handle accepts */
    int64_t seq_len;        /* S */
    double  rope_base;      /* theta_i = rope_base^(-2i/d), half-split pairs (i, i+d/2) */
    int32_t dtype;          /* skv_dtype: storage of A, B, V, q, keys, landmarks, out (SKV_FP8: see above) */
    int32_t v_place;        /* skv_vplace of V */
    int32_t new_keys;       /* skv_newkeys */
} skv_config;

typedef struct skv_layer skv_layer;   /* opaque; one per layer */

/* Host-only check of a config against the requirements above.  No CUDA call. */
int shadowkv_validate_config(const skv_config* cfg);

/*
 * Algorithm 1 (pre-filling) for one layer: rebuilds K~ = RoPE(A.B) for every
 * context token, takes chunk means as landmarks, picks per (b, h) the O
 * chunks outside the local window with the lowest minimum cosine between a
 * token key and its chunk mean (lower chunk id first on ties), removes them
 * from the landmarks, and gathers the outlier chunks' K~/V and the local
 * window's K~/V to the GPU.
 *
 *   A  dev  [b][S][r]      low-rank token coordinates (borrowed)
 *   B  dev  [b][H][r][d]   per-head bases (borrowed)
 *   V  dev or host [b][H][S][d]  values (borrowed).  With v_place = SKV_V_HOST
 *      the GPU reads them in place over the host link: V must be page-locked
 *      (cudaHostAlloc / cudaHostRegister) or, on a device that reads pageable
 *      memory through the host's page tables (Grace + NVLink-C2C), any system
 *      memory.  Otherwise SKV_ERR_NOT_PINNED.  shadowkv_host_alloc provides
 *      suitable page-locked memory.
 *
 * A, B and V must stay valid until shadowkv_destroy: decode steps read A/B
 * rows and V rows of the chunks they miss.  The library owns everything else.
 * Runs on `stream` and synchronises it before returning.  On error *out is
 * NULL and nothing is leaked.
 */
int shadowkv_prefill_index(const skv_config* cfg, const void* A, const void* B, const void* V,
                           skv_stream stream, skv_layer** out);

/*
 * Algorithm 1 as the digest states it (section A2): its inputs are the exact
 * keys K and K_RoPE, and the landmarks, the min-cosine outlier test, the
 * outlier keys and the local window's keys are built from K_RoPE = RoPE(K),
 * while A and B (the SVD of K, computed by the caller) serve only the sparse
 * reconstruction at decode time.
 *
 *   K  dev [b][H][S][d]  exact pre-RoPE keys, storage dtype (bf16; fp32 for
 *      SKV_F32; bf16 for SKV_FP8), 16-byte aligned.  Read during this call
 *      only: the library keeps no reference to it.
 * Everything else as shadowkv_prefill_index; K = NULL is that call.
 */
int shadowkv_prefill_index_keys(const skv_config* cfg, const void* A, const void* B, const void* K,
                                const void* V, skv_stream stream, skv_layer** out);

/*
 * Algorithm 2 (decoding), one step of one layer:
 *   1. appends (k_new, v_new) to the exact local set;
 *   2. P = q.L^T for the G query heads of every KV head (q-head j belongs to
 *      KV head j / G); S2 = max over the group of softmax(P / sqrt(d)) over the
 *      n_c selectable chunks; I = ArgTopK(S2, K), lower chunk id first on ties;
 *   3. index scan against the previous step's I: hit chunks keep their cache
 *      slot, missed chunks take the freed slots;
 *   4. rebuilds the missed chunks' keys RoPE(A[rows].B[b][h]) into their slots
 *      (main stream) while their values are gathered from V (side stream); with
 *      values in HBM and bf16 or e5m2 storage nothing is gathered: attention
 *      reads every cache slot's values in V, and runs on `main` right after the
 *      rebuild;
 *   5. out = softmax(q.K^T / sqrt(d)).V over the O*C outlier tokens, the K*C
 *      cached tokens and the W + t + 1 local tokens (t = 0-based step).
 *
 *   q      dev [b][H*G][d]  post-RoPE queries at position S + t
 *   k_new  dev [b][H][d]    post-RoPE key of the new token (SKV_NEWKEYS_LOWRANK:
 *                           its pre-RoPE key; step 4 then stores a = k'.Psi and
 *                           the new token's key rebuilt from it)
 *   v_new  dev [b][H][d]
 *   out    dev [b][H*G][d]  written
 *   sel_out dev int32 [b][H][K] or NULL: I as original chunk ids, ascending
 *   main, side: streams; side may be NULL or equal to main (then all work runs
 *   on main).  The library orders the two with its own events; the step is
 *   complete when `main` reaches the end of the enqueued work.
 */
int shadowkv_decode_step(skv_layer* layer, const void* q, const void* k_new, const void* v_new,
                         void* out, int32_t* sel_out, skv_stream main, skv_stream side);

/*
 * Micro-batch pipelining.  A caller that splits its batch into independent
 * handles per layer (micro-batches on their own streams) can let one
 * micro-batch's value fetch overlap another's landmark scoring: the fetch
 * moves data over the host link, the scoring reads HBM.  `event` (a
 * cudaEvent_t the caller owns, or NULL to stop) is recorded on the main stream
 * of every later decode step of this layer right after its selection, when
 * the step's miss list is final; the caller makes the next micro-batch's
 * stream wait for it before that micro-batch's decode step.  The library
 * keeps no other reference to the event.
 */
int shadowkv_set_select_event(skv_layer* layer, void* event);

/* Phases timed when profiling is on (CUDA events on the launching stream). */
#define SKV_PH_SCORE   0
#define SKV_PH_SELECT  1
#define SKV_PH_REBUILD 2
#define SKV_PH_FETCH   3
#define SKV_PH_ATTN    4
#define SKV_NPHASE     5

typedef struct {
    int64_t steps;              /* decode steps taken */
    int64_t units;              /* b*H */
    int64_t n_select;           /* K */
    int64_t hits, misses;       /* summed over steps and units */
    double  alpha_last;         /* hit rate of the last step */
    double  alpha_mean;         /* mean hit rate over steps t >= 1 (0 if none) */
    double  hbm_bytes;          /* algorithmic HBM bytes, summed over steps */
    double  link_bytes;         /* algorithmic host-link bytes (v_place = host) */
    double  scratch_bytes;      /* implementation scratch traffic (logits, partials) */
    double  phase_ms[SKV_NPHASE];        /* summed event time per phase (profiling) */
    int64_t phase_launches[SKV_NPHASE];  /* launches timed per phase */
    int32_t device_error;       /* 0, SKV_ERR_DEVICE_BOUNDS or SKV_ERR_TIMEOUT */
    int64_t kernel_launches;    /* kernels the decode steps launched since the last reset */
} skv_stats;

/*
 * Synchronises the layer's streams, reads the device counters and the error
 * word, and fills *out.  Returns the device error (if any) after filling *out.
 */
int shadowkv_stats(skv_layer* layer, skv_stats* out);
int shadowkv_reset_stats(skv_layer* layer);

/* Per-phase CUDA-event timing on (1) or off (0, the default). */
int shadowkv_set_profiling(skv_layer* layer, int enable);

/*
 * Inspection: copies one internal buffer (device to device, on `stream`) into
 * caller memory `dst` of at least shadowkv_export_size(layer, field) bytes.
 */
#define SKV_F_LANDMARKS     0   /* [b*H][n_c][d] dtype, compacted (outliers removed) */
#define SKV_F_CHUNK_IDS     1   /* [b*H][n_c] int32: original chunk id of each landmark */
#define SKV_F_OUTLIER_IDS   2   /* [b*H][O] int32, ascending */
#define SKV_F_MIN_COS       3   /* [b*H][S/C - W/C] float32 */
#define SKV_F_K_OUTLIER     4   /* [b*H][O*C][d] dtype */
#define SKV_F_V_OUTLIER     5   /* [b*H][O*C][d] dtype */
#define SKV_F_K_LOCAL       6   /* [b*H][W + max_new_tokens][d] dtype */
#define SKV_F_V_LOCAL       7   /* [b*H][W + max_new_tokens][d] dtype */
#define SKV_F_K_CACHE       8   /* [b*H][K][C][d] dtype, by slot */
#define SKV_F_V_CACHE       9   /* [b*H][K][C][d] dtype, by slot (values in HBM, bf16 or e5m2: the
                                   rows attention reads in V for each slot, gathered by the export;
                                   dst must be device memory) */
#define SKV_F_SELECTION    10   /* [b*H][K] int32: current I, ascending chunk ids */
#define SKV_F_SLOT_OF_SEL  11   /* [b*H][K] int32: cache slot of each entry of I */
#define SKV_F_MISS_COUNT   12   /* [b*H] int32: misses of the last step */
#define SKV_F_HITS_PER_STEP 13  /* [max_new_tokens] int32: hits summed over units */
#define SKV_F_A_NEW        14   /* [b][max_new_tokens][r] (A's storage: bf16, fp32 for SKV_F32):
                                   rank-r states of generated tokens (SKV_NEWKEYS_LOWRANK;
                                   size 0 otherwise) */
#define SKV_NFIELD         14
int64_t shadowkv_export_size(const skv_layer* layer, int field);
int shadowkv_export(skv_layer* layer, int field, void* dst, size_t bytes, skv_stream stream);

/*
 * Analytical models of the pages, host only:
 *   eq_bandwidth_gbs = 2 S B_GPU / (S/C + 2(K+O)C + (1-alpha) K C B_GPU / B_link)
 *   memory_savings   = 2SM / (SM/C + 2(K+O)C + Sr + rM), literal, M = H d (the
 *                      key width of one token across the KV heads, in elements)
 *   compression      = S d' / (r (S + d')), d' = H d (A is shared by the heads)
 * plus the algorithmic bytes of one decode step of one layer at hit rate alpha
 * and step t, and the predicted step time of that layer
 *   t_pred = hbm_bytes / B_GPU + link_bytes / B_link.
 */
typedef struct {
    double eq_bandwidth_gbs;
    double memory_savings;
    double compression_ratio;
    double hbm_bytes_per_step;
    double link_bytes_per_step;
    double t_pred_us;
} skv_model;
int shadowkv_model(const skv_config* cfg, double alpha, int64_t t, double b_gpu_gbs,
                   double b_link_gbs, skv_model* out);

/*
 * Host memory for values read in place by the GPU (v_place = SKV_V_HOST).
 * Not from the pages: it serves the value offload of the summary page's
 * section 3.4 ("What gets offloaded to the CPU").  Returns page-locked host
 * memory mapped into the GPU's address space (cudaHostAlloc, portable).
 * Allocate the values of every layer in one call and hand out slices: the
 * GPU's translations of one large allocation cover far more memory than
 * those of many small ones, which keeps the random 2 KB chunk reads of the
 * value fetch near link speed (measured for 32 x 2 GiB of values: about
 * 130 GB/s from one allocation against 44 GB/s from one per layer).
 * shadowkv_host_free releases it.  SKV_ERR_INVALID for bytes == 0 or
 * out == NULL, SKV_ERR_OOM if the memory cannot be allocated and locked.
 */
int shadowkv_host_alloc(size_t bytes, void** out);

/*
 * The same with a choice of host memory kind:
 *   SKV_HOST_PINNED  page-locked memory (cudaHostAlloc); what shadowkv_host_alloc returns.
 *   SKV_HOST_HUGE    pageable memory in the host's transparent huge pages (512 MiB on a
 *                    kernel with 64 KiB base pages), which the GPU reads through the host's
 *                    own page tables (Grace with NVLink-C2C; SKV_ERR_UNSUPPORTED elsewhere).
 *                    The mapping is aligned to the huge-page size and advised for huge pages;
 *                    the CUDA driver is told that its preferred location is the host, so it
 *                    does not migrate the pages on the GPU's access counts.  Pages come into
 *                    being when first written (fill it before the first
 *                    shadowkv_prefill_index that reads it).  While its pages are whole, one
 *                    translation covers 512 MiB and the value fetch's scattered 2 KB reads
 *                    run at about 170 GB/s against 125 GB/s from page-locked memory (32 x
 *                    2 GiB of values; link copy peak about 210 GB/s).  But the host kernel
 *                    splits some of them -- measured: a few of 128 pages of a 64 GiB arena on
 *                    most runs, 40-86 on the first run on a freshly booted host -- and a split
 *                    page is read with a translation per 64 KiB; see shadowkv_host_repair.
 *                    SKV_HOST_PINNED is the steady choice.
 * SKV_ERR_INVALID for bytes == 0, out == NULL or an unknown kind; SKV_ERR_OOM if the memory
 * cannot be had.  shadowkv_host_free releases either kind.
 */
#define SKV_HOST_PINNED 0
#define SKV_HOST_HUGE   1
int shadowkv_host_alloc_kind(size_t bytes, int kind, void** out);

/*
 * Puts split huge pages of [p, p + bytes) -- inside one SKV_HOST_HUGE allocation -- back
 * together (madvise MADV_COLLAPSE, Linux 6.1+; a page that is whole costs nothing).  Measured
 * on a 64 GiB arena: about ten of its 128 pages split while the layers were pre-filled, and a
 * split page costs the fetch a translation per 64 KiB instead of per 512 MiB.
 * shadowkv_prefill_index repairs the layer's own values before it returns.  From the first
 * decode step that reads such memory until the last SKV_HOST_HUGE allocation is freed, a
 * library thread watches the host's split count (/proc/vmstat thp_split_pmd, every 5 ms) and
 * repairs every such allocation when it moves, resting 50 ms after each repair.  A caller may
 * also repair a range itself, e.g. after its warm-up.  Synchronous.
 * SKV_ERR_INVALID if the range is not inside such an allocation, SKV_ERR_UNSUPPORTED if the
 * host kernel lacks the call, SKV_ERR_OOM if no huge page could be had.
 */
int shadowkv_host_repair(void* p, size_t bytes);
void shadowkv_host_free(void* p);

/*
 * Sparse attention that allocates nothing.  The pages have no counterpart to
 * this call; it exists for callers that cannot allocate device memory while
 * they run -- a server that hands all of HBM to one pool at start-up, code
 * that runs under an allocator lock, or a hot path where an allocation (which
 * may synchronise the device) is forbidden.
 *
 * It computes what step 5 of shadowkv_decode_step computes -- for each unit u
 * (a batch element's KV head) and each of its G query heads,
 * out = softmax(q.K^T / sqrt(d)).V over the unit's outlier rows, then its
 * cache rows, then its first n_local_tokens local rows -- but with its own
 * kernel (k_attn_bulk: 128-token splits staged by bulk copies, merged by the
 * last CTA of each unit), not the decode step's persistent tensor-core kernel.
 * All bf16, d = 128, rows of a region contiguous per unit:
 *   q         dev [units*group][128]                    (post-RoPE)
 *   k/v_outlier dev [units][n_outlier_tokens][128]      (may be NULL if 0 rows)
 *   k/v_cache dev [units][n_cache_tokens][128]          (may be NULL if 0 rows)
 *   k/v_local dev [units][local_capacity][128]
 *   out       dev [units*group][128]                    written
 * The caller owns every buffer; each must be device memory (a host pointer is
 * refused with SKV_ERR_INVALID before anything runs).
 *
 * Scratch: the partial results of the splits, one merge ticket per unit and an
 * error word live in a fixed 16 MiB array compiled into the library, which
 * every GPU that loads the library holds until the process exits.  Refused
 * with SKV_ERR_INVALID: more than 16384 units; partials above
 * 16 MiB - 64.25 KiB (units * ceil(rows / 128) * group * 528 bytes); or a unit
 * whose merge state does not fit in one CTA's shared memory (64 KiB +
 * 8 * ceil(rows / 128) * group bytes above the device's per-block limit, e.g.
 * about 333K rows at group 8).  fp32 data: SKV_ERR_UNSUPPORTED.
 *
 * No cudaMalloc, cudaFree or other allocating call is made.  With CUDA's lazy
 * module loading, though, the array itself comes into being when this part of
 * the library is first used on a device -- by the first call here, or by the
 * first decode step, whose attention kernels live in the same module.  A
 * caller that gives all free HBM to a pool should therefore make a set-up call
 * first: args->units == 0 launches nothing and only loads the array, resolves
 * its device address for the current device and sets the kernel's
 * shared-memory limit.  The first call on a device (set-up or not) does that
 * set-up, with that device current; make it before any stream capture.  The
 * address is resolved again if the device's context changes (after
 * cudaDeviceReset).
 *
 * Every call shares the one array and clears the merge tickets itself
 * (asynchronously, on `stream`); calls that overlap on the GPU -- on different
 * streams, or from different threads -- race on it, so serialise them.
 *
 * Errors inside the kernel (a bounded wait for the staged rows that ran out,
 * after about one second) are not seen by the call, which has returned
 * already: the affected units' outputs are written as NaN, and the error is
 * kept in the array's error word until shadowkv_sparse_attention_noalloc_status
 * reads it.
 */
typedef struct {
    int32_t units;              /* b*H; 0: set-up only (see above) */
    int32_t group;              /* G in {1, 2, 4, 8} */
    int32_t dtype;              /* skv_dtype; only SKV_BF16 */
    int32_t n_outlier_tokens;   /* rows per unit in k/v_outlier */
    int32_t n_cache_tokens;     /* rows per unit in k/v_cache */
    int32_t n_local_tokens;     /* rows per unit used from k/v_local, >= 1 */
    int32_t local_capacity;     /* rows per unit allocated in k/v_local */
    const void* q;
    const void* k_outlier;
    const void* v_outlier;
    const void* k_cache;
    const void* v_cache;
    const void* k_local;
    const void* v_local;
    void* out;
} skv_attention_args;
int shadowkv_sparse_attention_noalloc(const skv_attention_args* args, skv_stream stream);

/*
 * Status of the no-allocation calls made so far on the current device:
 * synchronises `stream`, reads the error word of the fixed array and clears it.
 * Returns SKV_OK, SKV_ERR_TIMEOUT (a kernel's wait ran out; those units' outputs
 * are NaN), or SKV_ERR_CUDA.  Allocates nothing.  The pages have no counterpart.
 */
int shadowkv_sparse_attention_noalloc_status(skv_stream stream);

/*
 * Measurement aid, not from the pages: the rate of the decode step's value
 * fetch on its own.  Reads n_chunks distinct random chunks of chunk_bytes
 * (1024, 2048 or 4096: one chunk of C = 8 rows of e5m2, bf16 or fp32 values)
 * spread over [src, src + bytes) -- host memory the GPU reads in place, or
 * device memory -- into device scratch with the fetch kernel, in address
 * order as the decode step reads its miss lists, on `stream`, reps + 1 times
 * (the first untimed).  fresh = 0 reads the same chunks every time (the GPU's
 * translations of them are warm after the first); fresh = 1 draws new chunks
 * for every repetition, as successive layers' fetches do.  *gbs_out = chunk
 * bytes per second of the fastest timed repetition (CUDA events).  Allocates
 * and frees its own device scratch and synchronises `stream`.
 * SKV_ERR_INVALID for bad sizes or a null or misaligned src.
 */
int shadowkv_fetch_probe(const void* src, size_t bytes, int64_t n_chunks, int chunk_bytes, uint64_t seed,
                         int reps, int fresh, skv_stream stream, double* gbs_out);

void shadowkv_destroy(skv_layer* layer);   /* frees everything the handle owns; NULL ok */
const char* shadowkv_strerror(int code);
int shadowkv_version(void);                 /* major*10000 + minor*100 + patch */

#ifdef __cplusplus
}
#endif
#endif /* SHADOWKV_H */
