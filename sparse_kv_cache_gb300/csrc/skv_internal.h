// Internal types shared by the kernel translation units and the host API.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace skv {

constexpr int kD = 128;        // head dim
constexpr int kC = 8;          // chunk size
constexpr int kTileChunks = 16;   // chunks per tensor-core rebuild tile (128 rows)
constexpr int kSelThreads = 1024;
constexpr int kAttnSeg = 256;  // tokens per attention CTA
constexpr int kScoreWarps = 8; // consumer warps of the scoring kernel
constexpr int kScoreStages = 3;
constexpr int kScoreStageBytes = 32768;

// Device error word codes (err[0]); err[1] records where the error happened.
enum : int { DEV_ERR_BOUNDS = 1, DEV_ERR_TIMEOUT = 2, DEV_ERR_NUMERIC = 3 };

// ---------------------------------------------------------------- scoring
// tensor-core scoring (bf16): 128-chunk tiles, 6-stage TMA ring, 4 epilogue warps
constexpr int kScTile = 128;
constexpr int kScStages = 6;
constexpr int kScStages8 = 6;   // e5m2 scorer: 2 x 16 KB tiles + query terms per stage
constexpr int kScN = 16;          // MMA N: the G <= 8 query heads, zero-padded
constexpr int kScParts = 4;       // partial records per (CTA, unit): one per epilogue warp
constexpr int kScParts8 = 8;      // the e5m2 scorer's epilogue warps: two per TMEM lane quarter

constexpr int kRunChunks = 512;   // landmarks per unit of scheduled scoring work

struct ScoreParams {
    const uint8_t* qt; const float* qinv;   // e5m2 scorer: query terms [U][3G][d], 2^-s [U][G]
    const void* L;        // [U][n_c][d]
    const void* q;        // [U*G][d]
    float* logits;        // [U][n_c][G]  z = q.L / sqrt(d)
    float2* part;         // [U * nru][nparts][G] (max, sum exp(z - max)) per run
    int n_c;
    int nru;              // runs per unit: ceil(n_c / kRunChunks)
    int total_runs;       // U * nru
    int nparts;           // records per run
    int* sched;           // run counter (reset to 0 by the selection kernel)
    float scale;
    int* err;
};
// bf16: tcgen05 kernel through the tensor map of L; fp32: CUDA-core kernel
int launch_score(int dtype, int G, const CUtensorMap* tmL, const ScoreParams& p, int ncta, cudaStream_t s);
int launch_qsplit(const void* q, void* qt, float* qinv, int U, int G, cudaStream_t s);   // e5m2 query terms
int score_ctas_per_sm(int dtype, int G);
int score_parts(int dtype);

// ---------------------------------------------------------------- selection
struct SelectParams {
    // top-K over n scores per unit (ties to the lower index), output ascending
    int n;                // n_c (decode) or candidates (outliers)
    int k;                // K or O
    int U, H, G;
    // decode: scores from logits and score partials
    const float* logits; const float2* part;
    int nru; int nparts;
    int nsm;              // SMs of the device (decode: picks the cluster form)
    int cluster;          // set by the launcher: CTAs per unit (1: one CTA per unit)
    int* sched;           // scoring run counter, reset here for the next step
    // outlier mode: score = -src[u][j]
    const float* neg_src;
    float* vbuf;          // [U][n] global score buffer when n exceeds shared memory
    int smem_cap;         // scores that fit in shared memory
    // outputs
    const int32_t* ids;   // [U][n] original chunk id of position j (NULL: identity)
    int32_t* sel_out_user;   // [U][k] or NULL
    int32_t* sel_plain;   // [U][k] (outlier mode output)
    // hit/miss state (decode)
    int t;
    int32_t* prev_ids; int32_t* prev_slot;   // [U][K]
    int32_t* cur_ids; int32_t* cur_slot;     // [U][K]
    int32_t* miss_chunk; int32_t* miss_slot; int32_t* miss_count;  // [U][K], [U]
    int32_t* slot_chunk;  // [U][K] chunk id held by each cache slot, or NULL
    int32_t* hits_step;   // [max_new_tokens]
    // append of the new token
    const void* k_new; const void* v_new; void* k_loc; void* v_loc;
    int loc_cap; int64_t loc_pitch; int W; int es;   // local rows of unit u start at u * loc_pitch
    int es_v;             // bytes of a value element: 1 stores the new value in e5m2
    // one-CTA decode form: the logits stream through two shared-memory buffers of
    // kSelStageBytes by bulk copies (set by the launcher), starting at byte stage_off of the
    // dynamic shared memory
    int stage; int stage_off;
    int* err;
};
int launch_select_decode(int dtype, const SelectParams& p, cudaStream_t s);
int launch_select_outliers(const SelectParams& p, cudaStream_t s);

// ---------------------------------------------------------------- rebuild / gather
struct RebuildParams {
    int mode;                 // 0: store RoPE'd keys, 1: landmark + min-cos statistics
    int U, H, r, nkb;
    int64_t S;                // context length: rows of A per batch element
    int nchunk;               // S / C, bound on chunk ids
    const int32_t* list;      // [U][list_us] chunk ids, or NULL: chunk = list_base + index
    int64_t list_us; int list_base; int list_cap;
    const int32_t* cnt;       // [U] entries, or NULL: count_const
    int count_const;
    const int32_t* dst_idx;   // [U][list_us] destination chunk slot, or NULL: index
    int dst_cap;              // chunk slots per unit in dst
    void* dst; int64_t dst_us;   // elements per unit of dst
    float* Lfull; float* mcos; int64_t stats_us;   // [U][stats_us][d], [U][stats_us]
    const float2* rope_lo;    // [256][d/2] (cos, sin) of lo * theta_i
    const float2* rope_hi;    // [nhi][d/2] (cos, sin) of hi * 256 * theta_i
    int nhi;
    const void* Kx;           // exact pre-RoPE keys [U][S][d] (pre-filling from exact keys), or NULL
    int kx_es;                // their element size: 2 (bf16) or 4 (fp32)
    const void* A;            // fp32 path: [b][S][r]
    const void* B;            // fp32 path: [U][r][d]
    int* err;
};
int launch_rebuild_tc(const CUtensorMap* tmA, const CUtensorMap* tmB, const RebuildParams& p, int grid_x,
                      cudaStream_t s);
int launch_rebuild_f32(const RebuildParams& p, int grid_x, cudaStream_t s);
// the same outputs from exact pre-RoPE keys p.Kx instead of A.B (keys stored as bf16 when out_bf16)
int launch_keys_exact(const RebuildParams& p, int grid_x, bool out_bf16, cudaStream_t s);
int launch_transpose_B(const void* B, void* Bt, int U, int r, cudaStream_t s);
// ShadowKV+ append: a[b] = k'[b] . B_b^T (k' [b][H][d], B [b][H][r][d]) into row t of
// a_new [b][a_rows][r], and every head's key RoPE_pos(a . B_h) into local row loc_row of its
// unit (rows of loc_pitch per unit)
struct PlusParams {
    const void* k_new; const void* B; void* a_new; void* k_loc;
    const float2* rope_lo; const float2* rope_hi;
    int H, r, t;
    int64_t a_rows, pos, loc_pitch, loc_row;
};
int launch_plus_append(int dtype, const PlusParams& p, int batch, cudaStream_t s);

struct GatherParams {
    const void* src; int64_t src_us;   // rows of unit u start at src + u*src_us (elements)
    const int32_t* list; int64_t list_us; int list_base; int list_cap;
    const int32_t* cnt; int count_const;
    const int32_t* dst_idx; int dst_cap;
    void* dst; int64_t dst_us;
    int nchunk; int es; int U;
    int* err;
};
int launch_gather(const GatherParams& p, int grid_x, cudaStream_t s);
// the decode step's fetch, two chunks per warp (per-unit lists and counts required)
int launch_fetch2(const GatherParams& p, int list_cap, cudaStream_t s);

struct CompactParams {
    const float* Lfull; int64_t ncand;   // [U][ncand][d]
    const int32_t* out_ids; int O;       // [U][O] ascending
    void* L; int32_t* ids; int n_c;      // [U][n_c][d], [U][n_c]
    int U; int dtype; int* err;
};
int launch_compact(const CompactParams& p, cudaStream_t s);

// ---------------------------------------------------------------- attention
struct AttnParams {
    const void* q;                 // [U*G][d]
    const void* k_out; const void* v_out; int n_out;    // [U][n_out][d]
    const void* k_c; const void* v_c; int n_cache;      // [U][n_cache][d]
    const void* k_loc; const void* v_loc; int n_loc; int loc_cap;   // [U][loc_cap][d]
    // > 0: the three regions are slices of per-unit blocks of unit_rows rows (unit u's rows of
    // every region start at base + u * unit_rows); 0: each region is packed [U][its rows][d]
    int64_t unit_rows;
    int v_es;                      // bytes of a value element: 2 (bf16) or 1 (e5m2; tensor-core form only)
    // values of the cache rows read where they live (values in HBM; tensor-core form only): the
    // chunk of cache slot s of unit u is slot_chunk[u * n_cache / 8 + s], its rows start at
    // v_src + (u * v_src_us + chunk * 8) * 128 elements; NULL: the cache rows' values come from v_c
    const void* v_src; int64_t v_src_us; const int32_t* slot_chunk; int nchunk;
    int pdl;                       // launched as a programmatic dependent of the previous kernel
    void* out;                     // [U*G][d]
    float* part;                   // [U][nsplit][G][d + 4]
    int* counter;                  // [U]
    int nsplit; float scale; int G; int U;
    int* err;
};
int launch_attn(int dtype, const AttnParams& p, cudaStream_t s);
// bf16: persistent tensor-core form, one CTA per SM (nsm), nsplit = ceil(tokens / 128); needs the
// block layout (unit_rows > 0, regions adjacent in each block) and a tensor map over the key
// blocks, [U * unit_rows][128] (box 64 x 128, 128-byte swizzle)
int launch_attn_tc(const CUtensorMap* k_all, const AttnParams& p, int nsm, cudaStream_t s);   // kernels launched, or -1
int attn_segment(int dtype);   // tokens per attention CTA

}  // namespace skv
