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
// slot >= 0: write the unnormalised partial (m, l, o) into partial slot `slot`;
// slot < 0: this unit covers every visible key of its rows, write final out/lse.
struct Unit {
    int32_t kv_head;
    int32_t branch;
    int32_t tok_begin;
    int32_t n_tok;
    int32_t key_begin;
    int32_t key_end;
    int32_t pos_base;
    int32_t slot;
};
static_assert(sizeof(Unit) == 32, "Unit is 8 int32");

struct PlanInput {
    const int32_t* suffix_lens;
    const int32_t* q_rows;
    int32_t num_branches;
    int32_t prefix_len;
    int32_t H_q, H_kv, page_size;
    int32_t causal;
    int32_t num_sms;
    int32_t force_splits;
};

struct Plan {
    std::vector<Unit> units;
    std::vector<int32_t> tok_slots;  // per token: partial slots to merge (0 = written directly)
    int32_t n_slots = 0;             // slots the partial buffer must hold
    int32_t R = 0;
    int32_t tpt = 0;                 // tokens per row tile
    bool need_merge = false;
};

// Builds the work plan (host only). Returns a fanout_status code.
int build_plan(const PlanInput& in, Plan& plan);

struct SplitParams {
    const int32_t* page_table;
    const Unit* units;
    float* part_o;    // [slot][R*H_q][kHD]
    float2* part_ml;  // [slot][R*H_q]   (m in log2 units, l)
    void* out;        // [R][H_q][kHD] fp32 or bf16
    float* lse;       // [R][H_q] or null
    int32_t* err;     // device error word
    int32_t n_units;
    int32_t max_pages;
    int32_t R, H_q, H_kv, G, page_size, tpt;
    int32_t out_bf16;
    float scale_log2;  // scale * log2(e)
    unsigned long long wait_limit_ns;
};

// Launchers (defined in the .cu files); return cudaError_t.
cudaError_t launch_split_attn(const SplitParams& p, const CUtensorMap& tm_q,
                              const CUtensorMap& tm_k, const CUtensorMap& tm_v, int grid,
                              cudaStream_t stream);
cudaError_t launch_lse_merge(const float* part_o, const float2* part_ml,
                             const int32_t* tok_slots, int32_t n_parts, int64_t n_out,
                             int32_t group, void* out, int32_t out_bf16, float* lse,
                             cudaStream_t stream);
cudaError_t err_word_ptr(int32_t** ptr);
cudaError_t launch_wait_selftest(int32_t* err, unsigned long long limit_ns, cudaStream_t stream);
int split_attn_smem_bytes();

}  // namespace fanout
