// plan.h -- host-only declarations: the work planner (plan.cpp), the
// device layout and upload of a plan, and the launch path (runtime.cpp).
#pragma once

#include <vector>

#include "fanout_internal.h"

namespace fanout {

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

}  // namespace fanout
