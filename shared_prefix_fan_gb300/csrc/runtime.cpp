// runtime.cpp -- the launch path shared by the entry points: argument checks,
// the device layout of a plan, its upload, the TMA tensor maps and the kernel
// launches. No attention arithmetic happens here.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "../../include/fanout.h"
#include "plan.h"

namespace fanout {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int status_of(cudaError_t e) {
    if (e == cudaSuccess) return FANOUT_OK;
    return e == cudaErrorMemoryAllocation ? FANOUT_ENOMEM : FANOUT_ECUDA;
}

// K / V page pool viewed as [num_pages * H_kv * page][128] bf16; a box is one
// page of one KV head, 64 columns (128 bytes, the swizzle span) wide.
int map_pool(CUtensorMap* m, const void* base, int64_t rows, int32_t box_rows) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHD), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHD) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t es[2] = {1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                       strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                       CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? FANOUT_OK
               : FANOUT_ECUDA;
}

// q viewed as [R][H_q][128] bf16; a box is 128/G tokens x the G heads of one
// KV head x 64 columns: one half of a 128-row tile, token-major.
int map_q(CUtensorMap* m, const void* q, int64_t R, int32_t H_q, int32_t G, int32_t tpt) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHD), static_cast<cuuint64_t>(H_q),
                          static_cast<cuuint64_t>(R)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHD) * 2,
                             static_cast<cuuint64_t>(H_q) * kHD * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(tpt)};
    cuuint32_t es[3] = {1, 1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims,
                       strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                       CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? FANOUT_OK
               : FANOUT_ECUDA;
}

}  // namespace

int validate_shape(const int32_t* suffix_lens, const int32_t* q_rows, int32_t B, int32_t P,
                   int32_t H_q, int32_t H_kv, int32_t d, int32_t page_size, int32_t causal) {
    if (B < 0 || P < 0 || H_q <= 0 || H_kv <= 0 || d <= 0 || page_size <= 0) return FANOUT_EINVAL;
    if (B > 0 && (suffix_lens == nullptr || q_rows == nullptr)) return FANOUT_EINVAL;
    if (H_q % H_kv != 0) return FANOUT_EINVAL;
    if (d != kHD) return FANOUT_EUNSUPPORTED;
    if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128)
        return FANOUT_EUNSUPPORTED;
    if (H_q / H_kv > kBM) return FANOUT_EUNSUPPORTED;
    int64_t R = 0;
    for (int32_t b = 0; b < B; ++b) {
        const int32_t S = suffix_lens[b], T = q_rows[b];
        if (S < 0 || T < 0) return FANOUT_EINVAL;
        if (static_cast<int64_t>(P) + S > (1 << 29)) return FANOUT_EUNSUPPORTED;
        if (causal && T > S) return FANOUT_EINVAL;  // new tokens are the suffix tail
        if (T > 0 && static_cast<int64_t>(P) + S == 0) return FANOUT_EINVAL;  // nothing to see
        R += T;
    }
    if (R * H_q > (static_cast<int64_t>(1) << 31) / kHD) return FANOUT_EUNSUPPORTED;
    return FANOUT_OK;
}

int validate_call(const void* q, const void* k, const void* v, const int32_t* page_table,
                  const int32_t* suffix_lens, int32_t B, int32_t P, int32_t max_pages,
                  int32_t num_pages, int32_t page_size, float scale, int32_t out_dtype,
                  const void* out) {
    if (out_dtype != FANOUT_OUT_F32 && out_dtype != FANOUT_OUT_BF16) return FANOUT_EINVAL;
    if (!(scale > 0.0f) || scale > 3.0e38f) return FANOUT_EINVAL;  // positive, finite
    if (!q || !k || !v || !page_table || !out) return FANOUT_EINVAL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return FANOUT_EINVAL;
    int64_t need_pages = 0;
    for (int32_t b = 0; b < B; ++b)
        need_pages = std::max<int64_t>(
            need_pages, (static_cast<int64_t>(P) + suffix_lens[b] + page_size - 1) / page_size);
    if (num_pages <= 0 || max_pages < need_pages) return FANOUT_EINVAL;
    return FANOUT_OK;
}

Layout plan_layout(const Plan& pl) {
    Layout L;
    size_t off = 0;
    L.flags = off;  // always first: epochs of the fused merge (zero when first allocated)
    off = align256(off + kMaxFusedGrid * sizeof(uint32_t));
    L.sink = off;
    off = align256(off + kSinkBytes);
    L.units = off;
    off = align256(off + pl.units.size() * sizeof(Unit));
    L.cta = off;
    off = align256(off + pl.cta_first.size() * sizeof(int32_t));
    L.mcnt = off;
    off = align256(off + pl.merge_cnt.size() * sizeof(int32_t));
    L.ment = off;
    off = align256(off + pl.merge_ent.size() * sizeof(int32_t));
    L.mkeys = off;
    off = align256(off + pl.merge_keys.size() * sizeof(int32_t));
    L.ml = off;
    const size_t rows = static_cast<size_t>(pl.n_parts) * kBM * pl.nq;
    off = align256(off + rows * sizeof(float2));
    L.o = off;
    off = align256(off + rows * kHD * sizeof(float));
    L.total = off;
    return L;
}

cudaError_t upload_plan(const Plan& pl, const Layout& L, uint8_t* base, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyAsync(base + L.units, pl.units.data(), pl.units.size() * sizeof(Unit),
                                    cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(base + L.cta, pl.cta_first.data(),
                            pl.cta_first.size() * sizeof(int32_t), cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && !pl.merge_cnt.empty())
        e = cudaMemcpyAsync(base + L.mcnt, pl.merge_cnt.data(),
                            pl.merge_cnt.size() * sizeof(int32_t), cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && !pl.merge_ent.empty())
        e = cudaMemcpyAsync(base + L.ment, pl.merge_ent.data(),
                            pl.merge_ent.size() * sizeof(int32_t), cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && !pl.merge_keys.empty())
        e = cudaMemcpyAsync(base + L.mkeys, pl.merge_keys.data(),
                            pl.merge_keys.size() * sizeof(int32_t), cudaMemcpyHostToDevice, stream);
    return e;
}

int launch_plan(const CallArgs& a, const Plan& pl, const Layout& L, uint8_t* base,
                cudaStream_t stream, cudaEvent_t ev_before, cudaEvent_t ev_after) {
    if (!encode_fn()) return FANOUT_ECUDA;
    const int32_t G = a.H_q / a.H_kv;
    CUtensorMap tm_q, tm_k, tm_v;
    const int64_t pool_rows = static_cast<int64_t>(a.num_pages) * a.H_kv * a.page_size;
    int st;
    if ((st = map_q(&tm_q, a.q, a.R, a.H_q, G, pl.tpt)) != FANOUT_OK) return st;
    if ((st = map_pool(&tm_k, a.k, pool_rows, a.page_size)) != FANOUT_OK) return st;
    if ((st = map_pool(&tm_v, a.v, pool_rows, a.page_size)) != FANOUT_OK) return st;
    int32_t* err = nullptr;
    cudaError_t ce = err_word_ptr(&err);
    if (ce != cudaSuccess) return status_of(ce);

    SplitParams p;
    p.page_table = a.page_table;
    p.units = reinterpret_cast<const Unit*>(base + L.units);
    p.cta_first = reinterpret_cast<const int32_t*>(base + L.cta);
    p.part_o = reinterpret_cast<float*>(base + L.o);
    p.part_ml = reinterpret_cast<float2*>(base + L.ml);
    p.sink = reinterpret_cast<float*>(base + L.sink);
    p.out = a.out;
    p.lse = a.lse;
    p.err = err;
    p.max_pages = a.max_pages;
    p.num_pages = a.num_pages;
    p.R = static_cast<int32_t>(a.R);
    p.H_q = a.H_q;
    p.H_kv = a.H_kv;
    p.G = G;
    p.page_size = a.page_size;
    p.tpt = pl.tpt;
    p.nq = pl.nq;
    p.out_bf16 = a.out_bf16;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.wait_limit_ns = a.wait_limit_ns;
    MergeParams& m = p.merge;
    m.part_o = p.part_o;
    m.part_ml = p.part_ml;
    m.merge_cnt = reinterpret_cast<const int32_t*>(base + L.mcnt);
    m.merge_ent = reinterpret_cast<const int2*>(base + L.ment);
    m.merge_keys = pl.merge_keys.empty() ? nullptr : reinterpret_cast<const int32_t*>(base + L.mkeys);
    m.merge_stride = pl.merge_stride;
    m.n_parts = 0;
    m.n_out = pl.merge_keys.empty() ? a.R * a.H_q : static_cast<int64_t>(pl.merge_keys.size()) * G;
    m.H_q = a.H_q;
    m.G = G;
    m.rows_per_part = kBM * pl.nq;
    m.out = a.out;
    m.out_bf16 = a.out_bf16;
    m.lse = a.lse;
    p.flags = reinterpret_cast<uint32_t*>(base + L.flags);
    p.epoch = a.epoch;
    // The merge runs inside the attention kernel when every CTA can be resident
    // at once (one per SM) and every output row has partials; otherwise, or if
    // the cooperative launch is refused, as a separate kernel.
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const bool fuse = pl.need_merge && a.fused_merge && pl.merge_keys.empty() &&
                      pl.n_cta() <= kMaxFusedGrid && pl.n_cta() <= sms;

    if (ev_before) cudaEventRecord(ev_before, stream);
    p.fused_merge = fuse ? 1 : 0;
    ce = launch_split_attn(p, tm_q, tm_k, tm_v, pl.n_cta(), fuse, stream);
    if (ce != cudaSuccess && fuse) {
        (void)cudaGetLastError();  // refused as a cooperative launch: merge separately
        p.fused_merge = 0;
        ce = launch_split_attn(p, tm_q, tm_k, tm_v, pl.n_cta(), false, stream);
    }
    if (ev_after) cudaEventRecord(ev_after, stream);
    if (ce != cudaSuccess) return status_of(ce);
    if (pl.need_merge && !p.fused_merge) {
        ce = launch_lse_merge(m, stream);
        if (ce != cudaSuccess) return status_of(ce);
    }
    return FANOUT_OK;
}

}  // namespace fanout
