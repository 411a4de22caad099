// fanout_internal.h -- types the kernels see: tile sizes, the work-unit
// record, kernel parameters and the launchers. Host-only planner and
// runtime declarations are in plan.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fanout {

constexpr int kBM = 128;      // query rows per tile (tcgen05 M)
constexpr int kBN = 128;      // keys per KV tile
constexpr int kHD = 128;      // the head dimension the kernels handle
constexpr int kNoCausal = 1 << 30;  // pos_base for units that need no causal mask

// One unit of split-KV work: the query rows of `n_tok` consecutive tokens
// (times the G query heads of KV head `kv_head`) against keys
// [key_begin, key_end) of branch `branch`'s logical sequence.
// Token r (global index) sits at absolute position pos_base + r, and key j
// is visible to it iff j < key_end and j <= pos_base + r.
// part >= 0: write the unnormalised partial (m, l, o) of the tile's rows into
// partial block `part` (128 * nq rows); part < 0: this unit covers every visible key
// of its rows, write the final out / lse.
struct Unit {
    int32_t kv_head;
    int32_t branch;
    int32_t tok_begin;
    int32_t n_tok;
    int32_t key_begin;
    int32_t key_end;
    int32_t pos_base;
    int32_t part;
};
static_assert(sizeof(Unit) == 32, "Unit is 8 int32");

struct MergeParams {
    const float* part_o;
    const float2* part_ml;
    const int32_t* merge_cnt;  // null: uniform parts (n_parts per output, part-major)
    const int2* merge_ent;     // [key][stride] {part, row base}
    const int32_t* merge_keys; // planned mode: keys to merge (null: every key)
    int32_t merge_stride;
    int32_t n_parts;           // uniform mode only
    int64_t n_out;             // rows to merge: R*H_q, |merge_keys|*G, or n (uniform mode)
    int32_t H_q, G;            // planned mode: out row n = token*H_q + kv_head*G + g
    int32_t rows_per_part;     // planned mode: rows of one partial block
    void* out;
    int32_t out_bf16;
    float* lse;
};

// Grid flags for the merge inside the attention kernel: one epoch word per CTA
// at the start of the plan's device scratch (so a re-laid-out plan never
// aliases them); a grid is at most this many CTAs when the merge is fused.
constexpr int kMaxFusedGrid = 1024;

struct SplitParams {
    const int32_t* page_table;
    const Unit* units;
    const int32_t* cta_first;
    float* part_o;    // [part][128 * nq rows][kHD]
    float* sink;      // kSinkBytes of scratch: the epilogue's dry-run stores
    float2* part_ml;  // [part][128 * nq rows]   (m in log2 units, l)
    void* out;        // [R][H_q][kHD] fp32 or bf16
    float* lse;       // [R][H_q] or null
    int32_t* err;     // device error word
    int32_t max_pages;
    int32_t num_pages;  // pool pages: clamps prefetch addresses of bad page ids
    int32_t R, H_q, H_kv, G, page_size, tpt;
    int32_t nq;        // query tiles per unit: selects the kernel instance
    int32_t out_bf16;
    float scale_log2;  // scale * log2(e)
    unsigned long long wait_limit_ns;
    // Merge inside the attention kernel (cooperative launch, all CTAs resident):
    // each CTA publishes `epoch` in flags[blockIdx.x] after its partials, waits
    // for every CTA's flag, then merges a slice of the output rows.
    int32_t fused_merge;
    uint32_t epoch;
    uint32_t* flags;
    MergeParams merge;
};

// Paged KV append: per-branch row offsets and current suffix lengths travel in
// the kernel parameters (no workspace).
constexpr int kMaxAppendBranches = 1024;
struct AppendParams {
    int32_t num_branches, R, H_kv, d, page_size, max_pages, num_pages, prefix_len;
    int32_t row_off[kMaxAppendBranches + 1];  // first row of each branch (+ total)
    int32_t suffix_len[kMaxAppendBranches];   // suffix length before the append
};

// Launchers (defined in the .cu files); return cudaError_t.
// cooperative: launch with all CTAs co-resident (required when p.fused_merge).
cudaError_t launch_split_attn(const SplitParams& p, const CUtensorMap& tm_q,
                              const CUtensorMap& tm_k, const CUtensorMap& tm_v, int grid,
                              bool cooperative, cudaStream_t stream);
cudaError_t launch_lse_merge(const MergeParams& p, cudaStream_t stream);
cudaError_t err_word_ptr(int32_t** ptr);
cudaError_t launch_copy_pages(void* k_pool, void* v_pool, const int32_t* pairs, int32_t n_pairs,
                              int32_t rows, int32_t H_kv, int32_t d, int32_t page_size,
                              int32_t num_pages, int32_t* err, cudaStream_t stream);
cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                             const int32_t* page_table, const AppendParams& p, int32_t* err,
                             cudaStream_t stream);
cudaError_t launch_wait_selftest(int32_t* err, unsigned long long limit_ns, cudaStream_t stream);

}  // namespace fanout
