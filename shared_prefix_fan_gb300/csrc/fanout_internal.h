// fanout_internal.h -- types shared by the host runtime and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

namespace fanout {

constexpr int kBM = 128;      // query rows per tile (tcgen05 M)
constexpr int kBN = 128;      // keys per KV tile
constexpr int kHD = 128;      // head dimension handled by this build
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

struct PlanInput {
    const int32_t* suffix_lens;
    const int32_t* q_rows;
    int32_t num_branches;
    int32_t prefix_len;
    int32_t H_q, H_kv, page_size;
    int32_t causal;
    int32_t num_sms;       // persistent CTAs: at most one per SM
    int32_t force_splits;  // >0: cut every key range into this many chunks
    int32_t tail_cuts = 1; // 0: never cut a direct range to even out the last wave
};

// A key range of the plan: the rows of n_tok tokens from tok_begin (one KV
// head) against keys [lo, hi) of a branch (branch 0 for the shared prefix).
struct PlanRange {
    int32_t kv_head, branch, tok_begin, n_tok, lo, hi, pos_base;
    bool complete;  // covers every visible key of its rows (no other range does)
};

struct Plan {
    std::vector<Unit> units;         // grouped by CTA: CTA c runs units [cta_first[c], cta_first[c+1])
    std::vector<int32_t> cta_first;  // n_cta + 1 entries
    std::vector<int32_t> merge_cnt;  // R*H_kv: partial entries of (token, KV head)
    std::vector<int32_t> merge_ent;  // [R*H_kv][merge_stride] pairs {part, first row of the token}
    // (token, KV head) keys that have partials, ascending; empty when every key
    // has (then the merge visits every output row)
    std::vector<int32_t> merge_keys;
    int32_t merge_stride = 0;
    int32_t n_parts = 0;             // partial blocks of 128 * nq rows
    int32_t R = 0;
    int32_t tpt = 0;                 // tokens per 128-row query tile
    int32_t nq = 1;                  // query tiles per unit (1 or 2)
    bool need_merge = false;
    std::vector<PlanRange> ranges;   // the key ranges the units were cut from
    std::vector<int32_t> unit_range; // per unit: its range
    int32_t n_cta() const { return cta_first.empty() ? 0 : static_cast<int32_t>(cta_first.size()) - 1; }
};

// Builds the work plan (host only). Returns a fanout_status code.
int build_plan(const PlanInput& in, Plan& plan);

// Carries `plan` over to a problem that differs from the one it was built
// for only in suffix lengths, when every key range keeps its number of
// 128-key tiles: the chunking, CTA assignment, partial blocks and merge index
// stay; each range's last unit gets the new range end and every unit the new
// causal position base. Returns false (plan untouched) otherwise.
bool patch_plan(const PlanInput& in, Plan& plan);

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


// One call: validated arguments (host) for the shared launch path.
struct CallArgs {
    const void* q;
    const void* k;
    const void* v;
    const int32_t* page_table;
    int32_t max_pages, num_pages, H_q, H_kv, page_size;
    int32_t out_bf16;
    float scale;
    void* out;
    float* lse;
    int64_t R;
    unsigned long long wait_limit_ns;
    int32_t fused_merge;  // 1: merge inside the attention kernel when the grid fits
    uint32_t epoch;       // this call's flag value (never 0; distinct from the last call's)
};

// Device layout of a plan inside one scratch buffer.
// Scratch the attention kernel's dry-run epilogue stores into (one row of O
// and its (m, l); written by every CTA, never read).
constexpr size_t kSinkBytes = 1024;

struct Layout {
    size_t flags, sink, units, cta, mcnt, ment, mkeys, ml, o, total;
};
Layout plan_layout(const Plan& pl);
// Copies the plan's tables into `base` (device) on `stream`.
cudaError_t upload_plan(const Plan& pl, const Layout& L, uint8_t* base, cudaStream_t stream);
// Tensor maps + split kernel (+ merge); events, when given, bracket the split kernel.
int launch_plan(const CallArgs& a, const Plan& pl, const Layout& L, uint8_t* base,
                cudaStream_t stream, cudaEvent_t ev_before, cudaEvent_t ev_after);
// The FANOUT_OPT_SPLITS setting (0 = planner's choice).
int32_t current_force_splits();
// The FANOUT_OPT_FUSED_MERGE setting.
int32_t current_fused_merge();
// Host-side argument checks shared by the entry points (fanout_status code).
int validate_shape(const int32_t* suffix_lens, const int32_t* q_rows, int32_t B, int32_t P,
                   int32_t H_q, int32_t H_kv, int32_t d, int32_t page_size, int32_t causal);
int validate_call(const void* q, const void* k, const void* v, const int32_t* page_table,
                  const int32_t* suffix_lens, int32_t B, int32_t P, int32_t max_pages,
                  int32_t num_pages, int32_t page_size, float scale, int32_t out_dtype,
                  const void* out);

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
