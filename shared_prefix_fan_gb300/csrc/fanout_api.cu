// fanout_api.cu -- the C ABI (include/fanout.h): the page-table fork, options,
// work-plan caching and the per-(device, stream) workspaces. The launch path
// itself (checks, tensor maps, kernels) is in runtime.cpp. No attention
// arithmetic happens here.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/fanout.h"
#include "plan.h"

using namespace fanout;

namespace {

std::mutex g_mu;
int64_t g_force_splits = 0;
int64_t g_validate_table = 0;
int64_t g_num_sms_override = 0;
int64_t g_fused_merge = 0;
unsigned long long g_wait_limit_ns = 1000000000ull;
cudaEvent_t g_ev_before = nullptr;
cudaEvent_t g_ev_after = nullptr;

// One per (device, stream). Its mutex serialises the calls on that stream's
// workspace (plan cache, buffer, upload, launch); calls on other streams only
// share g_mu for the map lookup and the option reads.
struct Workspace {
    std::mutex mu;
    void* buf = nullptr;
    size_t cap = 0;
    std::vector<int32_t> key;  // plan cache key
    Plan plan;
    Layout layout{};
    bool plan_ready = false;
    uint32_t epoch = 0;  // flag value of the last call (fused merge)
};
std::map<std::pair<int, cudaStream_t>, Workspace*> g_ws;

int status_from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return FANOUT_OK;
    if (e == cudaErrorMemoryAllocation) return FANOUT_ENOMEM;
    return FANOUT_ECUDA;
}

bool ok_align16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The host-only planning calls' default CTA count: a GB300's SMs.
constexpr int32_t kDefaultSms = 152;

int device_sms(int dev) {
    if (g_num_sms_override > 0) return static_cast<int>(g_num_sms_override);
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

}  // namespace

namespace fanout {
int32_t current_force_splits() {
    std::lock_guard<std::mutex> lk(g_mu);
    return static_cast<int32_t>(g_force_splits);
}
int32_t current_fused_merge() {
    std::lock_guard<std::mutex> lk(g_mu);
    return static_cast<int32_t>(g_fused_merge);
}
// read_floor.cu
cudaError_t launch_stream_read(const void* buf, int64_t bytes, uint32_t* xor_out,
                               cudaStream_t stream);
}  // namespace fanout

extern "C" {

const char* fanout_version(void) { return "0.2.0"; }

const char* fanout_strerror(int code) {
    switch (code) {
        case FANOUT_OK: return "ok";
        case FANOUT_EINVAL: return "invalid argument";
        case FANOUT_EUNSUPPORTED: return "problem outside what this library supports";
        case FANOUT_ECUDA: return "CUDA error";
        case FANOUT_ENOMEM: return "out of device memory";
        case FANOUT_ETIMEOUT: return "device-side wait timed out";
        default: return "unknown status";
    }
}

int fanout_fork(const int32_t* prefix_pages, int32_t n_prefix_pages, int32_t num_branches,
                const int32_t* suffix_lens, int32_t page_size, const int32_t* free_pages,
                int32_t n_free, int32_t* page_table, int32_t max_pages_per_branch) {
    if (n_prefix_pages < 0 || num_branches < 0 || page_size <= 0 || n_free < 0 ||
        max_pages_per_branch < 0)
        return FANOUT_EINVAL;
    if ((n_prefix_pages > 0 && !prefix_pages) || (num_branches > 0 && (!suffix_lens || !page_table)))
        return FANOUT_EINVAL;
    if (n_free > 0 && !free_pages) return FANOUT_EINVAL;
    int64_t cursor = 0;
    for (int32_t b = 0; b < num_branches; ++b) {
        if (suffix_lens[b] < 0) return FANOUT_EINVAL;
        const int64_t n_priv = (static_cast<int64_t>(suffix_lens[b]) + page_size - 1) / page_size;
        if (n_prefix_pages + n_priv > max_pages_per_branch) return FANOUT_EINVAL;
        if (cursor + n_priv > n_free) return FANOUT_EINVAL;
        int32_t* row = page_table + static_cast<int64_t>(b) * max_pages_per_branch;
        // shared prefix: the same physical ids in every branch, never copied
        std::copy(prefix_pages, prefix_pages + n_prefix_pages, row);
        std::copy(free_pages + cursor, free_pages + cursor + n_priv, row + n_prefix_pages);
        std::fill(row + n_prefix_pages + n_priv, row + max_pages_per_branch, -1);
        cursor += n_priv;
    }
    return FANOUT_OK;
}

int fanout_fork_cow(const int32_t* prefix_pages, int32_t prefix_len, int32_t num_branches,
                    const int32_t* suffix_lens, int32_t page_size, const int32_t* free_pages,
                    int32_t n_free, int32_t* page_table, int32_t max_pages_per_branch,
                    int32_t* cow_pairs, int32_t* n_used) {
    if (prefix_len < 0 || num_branches < 0 || page_size <= 0 || n_free < 0 ||
        max_pages_per_branch < 0)
        return FANOUT_EINVAL;
    const int64_t n_full = prefix_len / page_size;
    const bool partial = prefix_len % page_size != 0;
    const int64_t n_prefix_pages = n_full + (partial ? 1 : 0);
    if ((n_prefix_pages > 0 && !prefix_pages) || (num_branches > 0 && (!suffix_lens || !page_table)))
        return FANOUT_EINVAL;
    if (n_free > 0 && !free_pages) return FANOUT_EINVAL;
    int64_t cursor = 0;
    for (int32_t b = 0; b < num_branches; ++b) {  // check everything first
        if (suffix_lens[b] < 0) return FANOUT_EINVAL;
        const int64_t need =
            (static_cast<int64_t>(prefix_len) + suffix_lens[b] + page_size - 1) / page_size;
        if (std::max(need, n_prefix_pages) > max_pages_per_branch) return FANOUT_EINVAL;
        cursor += std::max<int64_t>(need, n_prefix_pages) - n_full;
        if (cursor > n_free) return FANOUT_EINVAL;
    }
    cursor = 0;
    for (int32_t b = 0; b < num_branches; ++b) {
        int32_t* row = page_table + static_cast<int64_t>(b) * max_pages_per_branch;
        const int64_t need = std::max<int64_t>(
            (static_cast<int64_t>(prefix_len) + suffix_lens[b] + page_size - 1) / page_size,
            n_prefix_pages);
        std::copy(prefix_pages, prefix_pages + n_full, row);  // whole pages: shared
        for (int64_t i = n_full; i < need; ++i) row[i] = free_pages[cursor++];  // own pages
        std::fill(row + need, row + max_pages_per_branch, -1);
        if (partial && cow_pairs) {  // the partial prefix page is copied into the branch's own
            cow_pairs[2 * b] = prefix_pages[n_full];
            cow_pairs[2 * b + 1] = row[n_full];
        }
    }
    if (n_used) *n_used = static_cast<int32_t>(cursor);
    return FANOUT_OK;
}

int fanout_copy_pages(void* k_pages, void* v_pages, const int32_t* pairs, int32_t n_pairs,
                      int32_t rows, int32_t num_pages, int32_t H_kv, int32_t d, int32_t page_size,
                      fanout_stream_t stream) {
    if (n_pairs < 0 || rows < 0 || rows > page_size || num_pages <= 0 || H_kv <= 0 || d <= 0 ||
        page_size <= 0)
        return FANOUT_EINVAL;
    if (d % 8 != 0) return FANOUT_EUNSUPPORTED;
    if (n_pairs == 0 || rows == 0) return FANOUT_OK;
    if (!k_pages || !v_pages || !pairs) return FANOUT_EINVAL;
    if (!ok_align16(k_pages) || !ok_align16(v_pages) || (reinterpret_cast<uintptr_t>(pairs) & 7u))
        return FANOUT_EINVAL;
    int32_t* err = nullptr;
    cudaError_t ce = err_word_ptr(&err);
    if (ce != cudaSuccess) return status_from_cuda(ce);
    return status_from_cuda(launch_copy_pages(k_pages, v_pages, pairs, n_pairs, rows, H_kv, d,
                                              page_size, num_pages, err,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

int fanout_extend(int32_t* page_table, int32_t num_branches, int32_t max_pages_per_branch,
                  int32_t prefix_len, const int32_t* suffix_lens, const int32_t* add_lens,
                  int32_t page_size, const int32_t* free_pages, int32_t n_free, int32_t* n_used) {
    if (num_branches < 0 || max_pages_per_branch < 0 || prefix_len < 0 || page_size <= 0 ||
        n_free < 0)
        return FANOUT_EINVAL;
    if (num_branches > 0 && (!page_table || !suffix_lens || !add_lens)) return FANOUT_EINVAL;
    if (n_free > 0 && !free_pages) return FANOUT_EINVAL;
    // Table entry i of a branch holds logical positions [i * page_size, (i+1) * page_size),
    // wherever the prefix ends: held = ceil(tokens / page_size) entries.
    auto entries = [&](int32_t b, bool grown) {
        const int64_t tokens = static_cast<int64_t>(prefix_len) + suffix_lens[b] +
                               (grown ? add_lens[b] : 0);
        return (tokens + page_size - 1) / page_size;
    };
    int64_t used = 0;
    for (int32_t b = 0; b < num_branches; ++b) {
        if (suffix_lens[b] < 0 || add_lens[b] < 0) return FANOUT_EINVAL;
        const int64_t need = entries(b, true);
        if (need > max_pages_per_branch) return FANOUT_EINVAL;
        used += need - entries(b, false);
        if (used > n_free) return FANOUT_EINVAL;
    }
    used = 0;
    for (int32_t b = 0; b < num_branches; ++b) {  // checked first: no partial update on error
        const int64_t need = entries(b, true);
        for (int64_t i = entries(b, false); i < need; ++i)
            page_table[static_cast<int64_t>(b) * max_pages_per_branch + i] = free_pages[used++];
    }
    if (n_used) *n_used = static_cast<int32_t>(used);
    return FANOUT_OK;
}

int fanout_kv_append(const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                     const int32_t* page_table, int32_t prefix_len, const int32_t* suffix_lens,
                     const int32_t* add_lens, int32_t num_branches, int32_t max_pages_per_branch,
                     int32_t num_pages, int32_t H_kv, int32_t d, int32_t page_size,
                     fanout_stream_t stream) {
    if (num_branches < 0 || prefix_len < 0 || H_kv <= 0 || d <= 0 || page_size <= 0 ||
        num_pages <= 0 || max_pages_per_branch <= 0)
        return FANOUT_EINVAL;
    if (num_branches > kMaxAppendBranches || d % 8 != 0 || d > 1024) return FANOUT_EUNSUPPORTED;
    if (num_branches > 0 && (!suffix_lens || !add_lens)) return FANOUT_EINVAL;
    AppendParams p;
    p.num_branches = num_branches;
    p.H_kv = H_kv;
    p.d = d;
    p.page_size = page_size;
    p.max_pages = max_pages_per_branch;
    p.num_pages = num_pages;
    p.prefix_len = prefix_len;
    int64_t R = 0;
    for (int32_t b = 0; b < num_branches; ++b) {
        if (suffix_lens[b] < 0 || add_lens[b] < 0) return FANOUT_EINVAL;
        const int64_t end = static_cast<int64_t>(prefix_len) + suffix_lens[b] + add_lens[b];
        if ((end + page_size - 1) / page_size > max_pages_per_branch) return FANOUT_EINVAL;
        p.row_off[b] = static_cast<int32_t>(R);
        p.suffix_len[b] = suffix_lens[b];
        R += add_lens[b];
    }
    if (R == 0) return FANOUT_OK;
    if (R * H_kv > (1LL << 31)) return FANOUT_EUNSUPPORTED;
    p.row_off[num_branches] = static_cast<int32_t>(R);
    p.R = static_cast<int32_t>(R);
    if (!k_new || !v_new || !k_pages || !v_pages || !page_table) return FANOUT_EINVAL;
    if (!ok_align16(k_new) || !ok_align16(v_new) || !ok_align16(k_pages) || !ok_align16(v_pages))
        return FANOUT_EINVAL;
    int32_t* err = nullptr;
    cudaError_t ce = err_word_ptr(&err);
    if (ce != cudaSuccess) return status_from_cuda(ce);
    return status_from_cuda(launch_kv_append(k_new, v_new, k_pages, v_pages, page_table, p, err,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int fanout_set_option(int32_t option, int64_t value) {
    std::lock_guard<std::mutex> lk(g_mu);
    switch (option) {
        case FANOUT_OPT_SPLITS:
            if (value < 0) return FANOUT_EINVAL;
            g_force_splits = value;  // part of every plan key: cached plans are not reused
            return FANOUT_OK;
        case FANOUT_OPT_VALIDATE_TABLE: g_validate_table = value; return FANOUT_OK;
        case FANOUT_OPT_WAIT_LIMIT_NS:
            if (value <= 0) return FANOUT_EINVAL;
            g_wait_limit_ns = static_cast<unsigned long long>(value);
            return FANOUT_OK;
        case FANOUT_OPT_NUM_SMS:
            if (value < 0) return FANOUT_EINVAL;
            g_num_sms_override = value;  // part of every plan key as well
            return FANOUT_OK;
        case FANOUT_OPT_FUSED_MERGE:
            if (value != 0 && value != 1) return FANOUT_EINVAL;
            g_fused_merge = value;
            return FANOUT_OK;
        default: return FANOUT_EINVAL;
    }
}

int fanout_set_profile_events(fanout_event_t before, fanout_event_t after) {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((before == nullptr) != (after == nullptr)) return FANOUT_EINVAL;
    g_ev_before = reinterpret_cast<cudaEvent_t>(before);
    g_ev_after = reinterpret_cast<cudaEvent_t>(after);
    return FANOUT_OK;
}

int fanout_plan(const int32_t* suffix_lens, const int32_t* q_rows_per_branch,
                int32_t num_branches, int32_t prefix_len, int32_t H_q, int32_t H_kv,
                int32_t page_size, int32_t causal, int32_t num_sms, int32_t* units, int32_t cap,
                int32_t* n_units, int32_t* cta_first, int32_t cta_cap, int32_t* n_ctas,
                int32_t* n_parts) {
    int st = validate_shape(suffix_lens, q_rows_per_branch, num_branches, prefix_len, H_q, H_kv,
                            kHD, page_size, causal);
    if (st != FANOUT_OK) return st;
    if (cap < 0 || (cap > 0 && !units) || cta_cap < 0 || (cta_cap > 0 && !cta_first))
        return FANOUT_EINVAL;
    PlanInput in{suffix_lens, q_rows_per_branch, num_branches, prefix_len, H_q, H_kv,
                 page_size, causal, num_sms > 0 ? num_sms : kDefaultSms, current_force_splits()};
    Plan plan;
    st = build_plan(in, plan);
    if (st != FANOUT_OK) return st;
    const int32_t n = static_cast<int32_t>(plan.units.size());
    if (n_units) *n_units = n;
    if (n_ctas) *n_ctas = plan.n_cta();
    if (n_parts) *n_parts = plan.n_parts;
    for (int32_t i = 0; i < std::min(n, cap); ++i)
        std::memcpy(units + 8 * static_cast<int64_t>(i), &plan.units[i], sizeof(Unit));
    for (int32_t i = 0; i < std::min<int32_t>(static_cast<int32_t>(plan.cta_first.size()), cta_cap); ++i)
        cta_first[i] = plan.cta_first[i];
    return FANOUT_OK;
}

int fanout_plan_step(const int32_t* prev_suffix_lens, const int32_t* suffix_lens,
                     const int32_t* q_rows_per_branch, int32_t num_branches, int32_t prefix_len,
                     int32_t H_q, int32_t H_kv, int32_t page_size, int32_t causal, int32_t num_sms,
                     int32_t* units, int32_t cap, int32_t* n_units, int32_t* cta_first,
                     int32_t cta_cap, int32_t* n_ctas, int32_t* n_parts, int32_t* reused) {
    int st = validate_shape(prev_suffix_lens, q_rows_per_branch, num_branches, prefix_len, H_q,
                            H_kv, kHD, page_size, causal);
    if (st != FANOUT_OK) return st;
    st = validate_shape(suffix_lens, q_rows_per_branch, num_branches, prefix_len, H_q, H_kv, kHD,
                        page_size, causal);
    if (st != FANOUT_OK) return st;
    if (cap < 0 || (cap > 0 && !units) || cta_cap < 0 || (cta_cap > 0 && !cta_first))
        return FANOUT_EINVAL;
    const int32_t sms = num_sms > 0 ? num_sms : kDefaultSms;
    const int32_t splits = current_force_splits();
    PlanInput prev{prev_suffix_lens, q_rows_per_branch, num_branches, prefix_len, H_q, H_kv,
                   page_size, causal, sms, splits};
    PlanInput in{suffix_lens, q_rows_per_branch, num_branches, prefix_len, H_q, H_kv,
                 page_size, causal, sms, splits};
    Plan plan;
    if ((st = build_plan(prev, plan)) != FANOUT_OK) return st;
    const bool kept = patch_plan(in, plan);
    if (!kept && (st = build_plan(in, plan)) != FANOUT_OK) return st;
    if (reused) *reused = kept ? 1 : 0;
    const int32_t n = static_cast<int32_t>(plan.units.size());
    if (n_units) *n_units = n;
    if (n_ctas) *n_ctas = plan.n_cta();
    if (n_parts) *n_parts = plan.n_parts;
    for (int32_t i = 0; i < std::min(n, cap); ++i)
        std::memcpy(units + 8 * static_cast<int64_t>(i), &plan.units[i], sizeof(Unit));
    for (int32_t i = 0; i < std::min<int32_t>(static_cast<int32_t>(plan.cta_first.size()), cta_cap); ++i)
        cta_first[i] = plan.cta_first[i];
    return FANOUT_OK;
}

int fanout_attn(const void* q, const void* k_pages, const void* v_pages,
                const int32_t* page_table, int32_t prefix_len, const int32_t* suffix_lens,
                const int32_t* q_rows_per_branch, int32_t num_branches,
                int32_t max_pages_per_branch, int32_t num_pages, int32_t H_q, int32_t H_kv,
                int32_t d, int32_t page_size, float scale, int32_t causal, void* out,
                int32_t out_dtype, float* lse, fanout_stream_t stream_) {
    int st = validate_shape(suffix_lens, q_rows_per_branch, num_branches, prefix_len, H_q, H_kv,
                            d, page_size, causal);
    if (st != FANOUT_OK) return st;
    if (out_dtype != FANOUT_OUT_F32 && out_dtype != FANOUT_OUT_BF16) return FANOUT_EINVAL;
    if (!(scale > 0.0f) || scale > 3.0e38f) return FANOUT_EINVAL;  // positive, finite
    int64_t R = 0;
    for (int32_t b = 0; b < num_branches; ++b) R += q_rows_per_branch[b];
    if (R == 0) return FANOUT_OK;
    st = validate_call(q, k_pages, v_pages, page_table, suffix_lens, num_branches, prefix_len,
                       max_pages_per_branch, num_pages, page_size, scale, out_dtype, out);
    if (st != FANOUT_OK) return st;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return status_from_cuda(ce);

    // Options and the workspace under the process-wide lock; everything after
    // under the workspace's own lock only.
    int64_t validate_table, fused_merge;
    int32_t splits;
    unsigned long long wait_limit_ns;
    cudaEvent_t ev_before, ev_after;
    int sms;
    Workspace* ws;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        validate_table = g_validate_table;
        fused_merge = g_fused_merge;
        splits = static_cast<int32_t>(g_force_splits);
        wait_limit_ns = g_wait_limit_ns;
        ev_before = g_ev_before;
        ev_after = g_ev_after;
        sms = device_sms(dev);
        Workspace*& slot = g_ws[{dev, stream}];
        if (!slot) slot = new Workspace();
        ws = slot;
    }
    std::lock_guard<std::mutex> wlk(ws->mu);

    if (validate_table) {
        std::vector<int32_t> tab(static_cast<size_t>(num_branches) * max_pages_per_branch);
        ce = cudaMemcpyAsync(tab.data(), page_table, tab.size() * sizeof(int32_t),
                             cudaMemcpyDeviceToHost, stream);
        if (ce == cudaSuccess) ce = cudaStreamSynchronize(stream);
        if (ce != cudaSuccess) return status_from_cuda(ce);
        const int32_t n_pre = prefix_len / page_size;
        for (int32_t b = 0; b < num_branches; ++b) {
            const int64_t n = (static_cast<int64_t>(prefix_len) + suffix_lens[b] + page_size - 1) / page_size;
            for (int64_t i = 0; i < n; ++i) {
                const int32_t v = tab[static_cast<size_t>(b) * max_pages_per_branch + i];
                if (v < 0 || v >= num_pages) return FANOUT_EINVAL;
                if (i < n_pre && v != tab[i]) return FANOUT_EINVAL;  // prefix must be shared
            }
        }
    }

    std::vector<int32_t> key = {prefix_len, num_branches, H_q, H_kv, page_size, causal, sms,
                                splits};
    key.insert(key.end(), suffix_lens, suffix_lens + num_branches);
    key.insert(key.end(), q_rows_per_branch, q_rows_per_branch + num_branches);
    // A call that differs from the cached plan's only in suffix lengths (a
    // decode step) keeps the plan when every key range keeps its tile count:
    // only the unit table moves (new range ends and causal positions).
    const size_t fixed = 8;  // key entries before the suffix lengths
    const PlanInput in{suffix_lens, q_rows_per_branch, num_branches, prefix_len, H_q, H_kv,
                       page_size, causal, sms, splits};
    bool patched = false;
    if (ws->plan_ready && key != ws->key && key.size() == ws->key.size() &&
        std::equal(key.begin(), key.begin() + fixed, ws->key.begin()) &&
        std::equal(key.begin() + fixed + num_branches, key.end(),
                   ws->key.begin() + fixed + num_branches)) {
        if (patch_plan(in, ws->plan)) {
            ce = cudaMemcpyAsync(static_cast<uint8_t*>(ws->buf) + ws->layout.units,
                                 ws->plan.units.data(), ws->plan.units.size() * sizeof(Unit),
                                 cudaMemcpyHostToDevice, stream);
            if (ce != cudaSuccess) {
                ws->plan_ready = false;
                return status_from_cuda(ce);
            }
            ws->key = key;
            patched = true;
        }
    }
    if (!patched && (!ws->plan_ready || key != ws->key)) {
        ws->plan_ready = false;
        if ((st = build_plan(in, ws->plan)) != FANOUT_OK) return st;
        ws->layout = plan_layout(ws->plan);
        if (ws->layout.total > ws->cap) {
            if (ws->buf) {
                cudaStreamSynchronize(stream);
                cudaFree(ws->buf);
                ws->buf = nullptr;
                ws->cap = 0;
            }
            ce = cudaMalloc(&ws->buf, ws->layout.total);
            if (ce != cudaSuccess) {
                ws->buf = nullptr;
                return status_from_cuda(ce);
            }
            ws->cap = ws->layout.total;
            // fused-merge flags start below every epoch a call can use
            ce = cudaMemsetAsync(static_cast<uint8_t*>(ws->buf) + ws->layout.flags, 0,
                                 kMaxFusedGrid * sizeof(uint32_t), stream);
            if (ce != cudaSuccess) return status_from_cuda(ce);
        }
        ce = upload_plan(ws->plan, ws->layout, static_cast<uint8_t*>(ws->buf), stream);
        if (ce != cudaSuccess) return status_from_cuda(ce);
        ws->key = key;
        ws->plan_ready = true;
    }
    if (++ws->epoch == 0) ws->epoch = 1;  // 0 is the flags' initial value
    CallArgs a{q, k_pages, v_pages, page_table, max_pages_per_branch, num_pages, H_q, H_kv,
               page_size, out_dtype == FANOUT_OUT_BF16, scale, out, lse, R, wait_limit_ns,
               static_cast<int32_t>(fused_merge), ws->epoch};
    return launch_plan(a, ws->plan, ws->layout, static_cast<uint8_t*>(ws->buf), stream,
                       ev_before, ev_after);
}

int fanout_lse_merge(const float* part_o, const float* part_ml, int32_t n_parts, int64_t n_out,
                     int32_t d, void* out, int32_t out_dtype, float* lse,
                     fanout_stream_t stream) {
    if (n_parts < 0 || n_out < 0) return FANOUT_EINVAL;
    if (d != kHD) return FANOUT_EUNSUPPORTED;
    if (out_dtype != FANOUT_OUT_F32 && out_dtype != FANOUT_OUT_BF16) return FANOUT_EINVAL;
    if (n_out == 0) return FANOUT_OK;
    if (n_parts == 0 || !part_o || !part_ml || !out) return FANOUT_EINVAL;
    if (!ok_align16(part_o) || !ok_align16(out) || (reinterpret_cast<uintptr_t>(part_ml) & 7u))
        return FANOUT_EINVAL;
    MergeParams m;
    m.part_o = part_o;
    m.part_ml = reinterpret_cast<const float2*>(part_ml);
    m.merge_cnt = nullptr;
    m.merge_keys = nullptr;
    m.merge_ent = nullptr;
    m.merge_stride = 0;
    m.n_parts = n_parts;
    m.n_out = n_out;
    m.H_q = 1;
    m.G = 1;
    m.rows_per_part = 0;
    m.out = out;
    m.out_bf16 = out_dtype == FANOUT_OUT_BF16;
    m.lse = lse;
    return status_from_cuda(launch_lse_merge(m, reinterpret_cast<cudaStream_t>(stream)));
}

int fanout_last_error_detail(fanout_stream_t stream, int32_t* site, int32_t* block) {
    cudaError_t ce = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (ce != cudaSuccess) return status_from_cuda(ce);
    int32_t* err = nullptr;
    if ((ce = err_word_ptr(&err)) != cudaSuccess) return status_from_cuda(ce);
    int32_t word[4] = {0, 0, 0, 0};
    ce = cudaMemcpy(word, err, sizeof(word), cudaMemcpyDeviceToHost);
    if (ce != cudaSuccess) return status_from_cuda(ce);
    if (site) *site = word[1];
    if (block) *block = word[2];
    if (word[0] != 0) {
        const int32_t zero[4] = {0, 0, 0, 0};
        cudaMemcpy(err, zero, sizeof(zero), cudaMemcpyHostToDevice);
        return word[0];
    }
    return FANOUT_OK;
}

int fanout_last_error(fanout_stream_t stream) {
    return fanout_last_error_detail(stream, nullptr, nullptr);
}

int fanout_selftest_wait_timeout(int64_t limit_ns, fanout_stream_t stream) {
    if (limit_ns <= 0 || limit_ns > 10000000000LL) return FANOUT_EINVAL;
    int32_t* err = nullptr;
    cudaError_t ce = err_word_ptr(&err);
    if (ce != cudaSuccess) return status_from_cuda(ce);
    ce = launch_wait_selftest(err, static_cast<unsigned long long>(limit_ns),
                              reinterpret_cast<cudaStream_t>(stream));
    if (ce != cudaSuccess) return status_from_cuda(ce);
    return fanout_last_error(stream);
}

int fanout_read_floor(const void* buf, int64_t bytes, uint32_t* xor_out,
                      fanout_stream_t stream) {
    if (buf == nullptr || xor_out == nullptr || bytes <= 0 || bytes % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(buf) & 15u) != 0 ||
        (reinterpret_cast<uintptr_t>(xor_out) & 3u) != 0)
        return FANOUT_EINVAL;
    return status_from_cuda(
        launch_stream_read(buf, bytes, xor_out, reinterpret_cast<cudaStream_t>(stream)));
}

int fanout_release(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    // The workspace records stay (a call on another thread may hold one between
    // the map lookup and its own lock); only their device buffers and plans go.
    for (auto& kv : g_ws) {
        Workspace* ws = kv.second;
        std::lock_guard<std::mutex> wlk(ws->mu);
        if (ws->buf) {
            cudaSetDevice(kv.first.first);
            cudaDeviceSynchronize();
            cudaFree(ws->buf);
        }
        ws->buf = nullptr;
        ws->cap = 0;
        ws->plan_ready = false;
        ws->key.clear();
    }
    cudaSetDevice(cur);
    return FANOUT_OK;
}

}  // extern "C"
