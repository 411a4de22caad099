// fanout_api.cu -- the C ABI (include/fanout.h): argument validation, the
// page-table fork, work-plan caching, per-(device, stream) workspaces, TMA
// tensor maps and kernel launches. No attention arithmetic happens here.
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
#include "fanout_internal.h"

using namespace fanout;

namespace {

std::mutex g_mu;
int64_t g_force_splits = 0;
int64_t g_validate_table = 0;
int64_t g_num_sms_override = 0;
unsigned long long g_wait_limit_ns = 1000000000ull;
cudaEvent_t g_ev_before = nullptr;
cudaEvent_t g_ev_after = nullptr;

struct Workspace {
    void* buf = nullptr;
    size_t cap = 0;
    std::vector<int32_t> key;  // plan cache key
    Plan plan;
    size_t off_units = 0, off_tok = 0, off_ml = 0, off_o = 0;
    bool plan_ready = false;
};
std::map<std::pair<int, cudaStream_t>, Workspace*> g_ws;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int status_from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return FANOUT_OK;
    if (e == cudaErrorMemoryAllocation) return FANOUT_ENOMEM;
    return FANOUT_ECUDA;
}

int get_encode() {
    if (g_encode) return FANOUT_OK;
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) return FANOUT_ECUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return FANOUT_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool ok_align16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-side checks shared by fanout_attn and fanout_plan.
int validate_shape(const int32_t* suffix_lens, const int32_t* q_rows, int32_t B, int32_t P,
                   int32_t H_q, int32_t H_kv, int32_t d, int32_t page_size, int32_t causal) {
    if (B < 0 || P < 0 || H_q <= 0 || H_kv <= 0 || d <= 0 || page_size <= 0) return FANOUT_EINVAL;
    if (B > 0 && (suffix_lens == nullptr || q_rows == nullptr)) return FANOUT_EINVAL;
    if (H_q % H_kv != 0) return FANOUT_EINVAL;
    if (d != kHD) return FANOUT_EUNSUPPORTED;
    if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128)
        return FANOUT_EUNSUPPORTED;
    if (H_q / H_kv > kBM) return FANOUT_EUNSUPPORTED;
    if (P % page_size != 0) return FANOUT_EUNSUPPORTED;
    int64_t R = 0;
    for (int32_t b = 0; b < B; ++b) {
        const int32_t S = suffix_lens[b], T = q_rows[b];
        if (S < 0 || T < 0) return FANOUT_EINVAL;
        if (static_cast<int64_t>(P) + S > (1 << 29)) return FANOUT_EUNSUPPORTED;
        if (causal && T > S) return FANOUT_EINVAL;     // new tokens are the suffix tail
        if (T > 0 && static_cast<int64_t>(P) + S == 0) return FANOUT_EINVAL;  // nothing to see
        R += T;
    }
    if (R * H_q > (static_cast<int64_t>(1) << 31) / kHD) return FANOUT_EUNSUPPORTED;
    return FANOUT_OK;
}

int encode_2d_pool(CUtensorMap* m, const void* base, int64_t rows, int32_t page_size) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHD), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHD) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(page_size)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FANOUT_OK : FANOUT_ECUDA;
}

int encode_q(CUtensorMap* m, const void* q, int64_t R, int32_t H_q, int32_t G, int32_t tpt) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHD), static_cast<cuuint64_t>(H_q),
                          static_cast<cuuint64_t>(R)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHD) * 2,
                             static_cast<cuuint64_t>(H_q) * kHD * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(tpt)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FANOUT_OK : FANOUT_ECUDA;
}

int device_sms(int dev) {
    if (g_num_sms_override > 0) return static_cast<int>(g_num_sms_override);
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

}  // namespace

extern "C" {

const char* fanout_version(void) { return "0.1.0"; }

const char* fanout_strerror(int code) {
    switch (code) {
        case FANOUT_OK: return "ok";
        case FANOUT_EINVAL: return "invalid argument";
        case FANOUT_EUNSUPPORTED: return "unsupported problem for this build";
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

int fanout_set_option(int32_t option, int64_t value) {
    std::lock_guard<std::mutex> lk(g_mu);
    switch (option) {
        case FANOUT_OPT_SPLITS:
            if (value < 0) return FANOUT_EINVAL;
            g_force_splits = value;
            for (auto& kv : g_ws) kv.second->plan_ready = false;
            return FANOUT_OK;
        case FANOUT_OPT_VALIDATE_TABLE: g_validate_table = value; return FANOUT_OK;
        case FANOUT_OPT_WAIT_LIMIT_NS:
            if (value <= 0) return FANOUT_EINVAL;
            g_wait_limit_ns = static_cast<unsigned long long>(value);
            return FANOUT_OK;
        case FANOUT_OPT_NUM_SMS:
            if (value < 0) return FANOUT_EINVAL;
            g_num_sms_override = value;
            for (auto& kv : g_ws) kv.second->plan_ready = false;
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
                int32_t* n_units, int32_t* n_slots, int32_t* tok_slots) {
    int st = validate_shape(suffix_lens, q_rows_per_branch, num_branches, prefix_len, H_q, H_kv,
                            kHD, page_size, causal);
    if (st != FANOUT_OK) return st;
    if (cap < 0 || (cap > 0 && !units)) return FANOUT_EINVAL;
    PlanInput in{suffix_lens, q_rows_per_branch, num_branches, prefix_len, H_q, H_kv,
                 page_size, causal, num_sms > 0 ? num_sms : 148,
                 static_cast<int32_t>(g_force_splits)};
    Plan plan;
    st = build_plan(in, plan);
    if (st != FANOUT_OK) return st;
    const int32_t n = static_cast<int32_t>(plan.units.size());
    if (n_units) *n_units = n;
    if (n_slots) *n_slots = plan.n_slots;
    for (int32_t i = 0; i < std::min(n, cap); ++i)
        std::memcpy(units + 8 * static_cast<int64_t>(i), &plan.units[i], sizeof(Unit));
    if (tok_slots) std::copy(plan.tok_slots.begin(), plan.tok_slots.end(), tok_slots);
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
    if (!(scale == scale) || scale == 0.0f) return FANOUT_EINVAL;
    int64_t R = 0;
    int64_t need_pages = 0;
    for (int32_t b = 0; b < num_branches; ++b) {
        R += q_rows_per_branch[b];
        need_pages = std::max<int64_t>(
            need_pages, (static_cast<int64_t>(prefix_len) + suffix_lens[b] + page_size - 1) / page_size);
    }
    if (R == 0) return FANOUT_OK;
    if (!q || !k_pages || !v_pages || !page_table || !out) return FANOUT_EINVAL;
    if (!ok_align16(q) || !ok_align16(k_pages) || !ok_align16(v_pages) || !ok_align16(out))
        return FANOUT_EINVAL;
    if (num_pages <= 0 || max_pages_per_branch < need_pages) return FANOUT_EINVAL;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

    std::lock_guard<std::mutex> lk(g_mu);
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return status_from_cuda(ce);
    if ((st = get_encode()) != FANOUT_OK) return st;

    if (g_validate_table) {
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

    const int sms = device_sms(dev);
    Workspace*& ws = g_ws[{dev, stream}];
    if (!ws) ws = new Workspace();
    std::vector<int32_t> key = {prefix_len, num_branches, H_q, H_kv, page_size, causal, sms,
                                static_cast<int32_t>(g_force_splits)};
    key.insert(key.end(), suffix_lens, suffix_lens + num_branches);
    key.insert(key.end(), q_rows_per_branch, q_rows_per_branch + num_branches);
    if (!ws->plan_ready || key != ws->key) {
        PlanInput in{suffix_lens, q_rows_per_branch, num_branches, prefix_len, H_q, H_kv,
                     page_size, causal, sms, static_cast<int32_t>(g_force_splits)};
        ws->plan_ready = false;
        if ((st = build_plan(in, ws->plan)) != FANOUT_OK) return st;
        const Plan& pl = ws->plan;
        size_t off = 0;
        ws->off_units = off;
        off = align_up(off + pl.units.size() * sizeof(Unit), 256);
        ws->off_tok = off;
        off = align_up(off + pl.tok_slots.size() * sizeof(int32_t), 256);
        ws->off_ml = off;
        off = align_up(off + static_cast<size_t>(pl.n_slots) * R * H_q * sizeof(float2), 256);
        ws->off_o = off;
        off = align_up(off + static_cast<size_t>(pl.n_slots) * R * H_q * kHD * sizeof(float), 256);
        if (off > ws->cap) {
            if (ws->buf) {
                cudaStreamSynchronize(stream);
                cudaFree(ws->buf);
                ws->buf = nullptr;
                ws->cap = 0;
            }
            ce = cudaMalloc(&ws->buf, off);
            if (ce != cudaSuccess) {
                ws->buf = nullptr;
                return status_from_cuda(ce);
            }
            ws->cap = off;
        }
        uint8_t* base = static_cast<uint8_t*>(ws->buf);
        ce = cudaMemcpyAsync(base + ws->off_units, pl.units.data(), pl.units.size() * sizeof(Unit),
                             cudaMemcpyHostToDevice, stream);
        if (ce == cudaSuccess)
            ce = cudaMemcpyAsync(base + ws->off_tok, pl.tok_slots.data(),
                                 pl.tok_slots.size() * sizeof(int32_t), cudaMemcpyHostToDevice,
                                 stream);
        if (ce != cudaSuccess) return status_from_cuda(ce);
        ws->key = key;
        ws->plan_ready = true;
    }
    const Plan& pl = ws->plan;
    uint8_t* base = static_cast<uint8_t*>(ws->buf);
    const int32_t G = H_q / H_kv;

    CUtensorMap tm_q, tm_k, tm_v;
    const int64_t pool_rows = static_cast<int64_t>(num_pages) * H_kv * page_size;
    if ((st = encode_q(&tm_q, q, R, H_q, G, pl.tpt)) != FANOUT_OK) return st;
    if ((st = encode_2d_pool(&tm_k, k_pages, pool_rows, page_size)) != FANOUT_OK) return st;
    if ((st = encode_2d_pool(&tm_v, v_pages, pool_rows, page_size)) != FANOUT_OK) return st;

    int32_t* err = nullptr;
    if ((ce = err_word_ptr(&err)) != cudaSuccess) return status_from_cuda(ce);

    SplitParams p;
    p.page_table = page_table;
    p.units = reinterpret_cast<const Unit*>(base + ws->off_units);
    p.part_o = reinterpret_cast<float*>(base + ws->off_o);
    p.part_ml = reinterpret_cast<float2*>(base + ws->off_ml);
    p.out = out;
    p.lse = lse;
    p.err = err;
    p.n_units = static_cast<int32_t>(pl.units.size());
    p.max_pages = max_pages_per_branch;
    p.R = static_cast<int32_t>(R);
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.G = G;
    p.page_size = page_size;
    p.tpt = pl.tpt;
    p.out_bf16 = out_dtype == FANOUT_OUT_BF16;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.wait_limit_ns = g_wait_limit_ns;

    if (g_ev_before) cudaEventRecord(g_ev_before, stream);
    ce = launch_split_attn(p, tm_q, tm_k, tm_v, p.n_units, stream);
    if (g_ev_after) cudaEventRecord(g_ev_after, stream);
    if (ce != cudaSuccess) return status_from_cuda(ce);
    if (pl.need_merge) {
        ce = launch_lse_merge(p.part_o, p.part_ml,
                              reinterpret_cast<const int32_t*>(base + ws->off_tok), pl.n_slots,
                              R * H_q, H_q, out, p.out_bf16, lse, stream);
        if (ce != cudaSuccess) return status_from_cuda(ce);
    }
    return FANOUT_OK;
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
    cudaError_t ce = launch_lse_merge(part_o, reinterpret_cast<const float2*>(part_ml), nullptr,
                                      n_parts, n_out, 1, out, out_dtype == FANOUT_OUT_BF16, lse,
                                      reinterpret_cast<cudaStream_t>(stream));
    return status_from_cuda(ce);
}

int fanout_last_error(fanout_stream_t stream) {
    cudaError_t ce = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (ce != cudaSuccess) return status_from_cuda(ce);
    int32_t* err = nullptr;
    if ((ce = err_word_ptr(&err)) != cudaSuccess) return status_from_cuda(ce);
    int32_t word[4] = {0, 0, 0, 0};
    ce = cudaMemcpy(word, err, sizeof(word), cudaMemcpyDeviceToHost);
    if (ce != cudaSuccess) return status_from_cuda(ce);
    if (word[0] != 0) {
        const int32_t zero[4] = {0, 0, 0, 0};
        cudaMemcpy(err, zero, sizeof(zero), cudaMemcpyHostToDevice);
        return word[0];
    }
    return FANOUT_OK;
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

int fanout_release(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto& kv : g_ws) {
        if (kv.second->buf) {
            cudaSetDevice(kv.first.first);
            cudaDeviceSynchronize();
            cudaFree(kv.second->buf);
        }
        delete kv.second;
    }
    g_ws.clear();
    cudaSetDevice(cur);
    return FANOUT_OK;
}

}  // extern "C"
