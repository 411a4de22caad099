// merge_row.cuh -- the log-sum-exp merge of one output row's split-KV
// partials, shared by the stand-alone merge kernel and the merge tail of the
// attention kernel.
//
// ADR-0060 section 4 ("Reduction -- tree to the root") and "AHBM Agentic
// Runtime Architecture" section 3.4 ("Online softmax merge"): partial states
// of the SAME row from different key shards combine as
//   m = max(m_a, m_b); s_a = 2^(m_a - m); s_b = 2^(m_b - m);
//   l = l_a s_a + l_b s_b; o = o_a s_a + o_b s_b;  final out = o / l.
// The pages fold pairs up a tree of PEs over IPCQ links; on one GPU there are
// no links to save, so one warp folds all of a row's partials. It takes the
// overall max first and then sums in a fixed order (the merge is associative
// and commutative, so this is the same fold), so results are bitwise
// reproducible.
#pragma once

#include <cuda_bf16.h>

#include "fanout_internal.h"
#include "ptx_sm100.cuh"

namespace fanout {

// The merge index of the i-th row to merge: its output row n (a (token, query
// head) pair), partial count ne, head-in-group g, and the first 32 entries.
// Planned mode: fixed-stride entry lists {part, row base} per (token, KV head),
// partial row = base + g; the rows to merge are every output row, or the G
// rows of each listed key when only some keys have partials. Uniform mode
// (merge_cnt null): n_parts partials per row, part-major [n_parts][n_out].
// Plan data only, so it may be read before the partials exist.
struct MergeIdx {
    int32_t ne, g;
    int64_t key;
    int2 ent0;
    int64_t n;
};
__device__ __forceinline__ MergeIdx merge_index(const MergeParams& p, int64_t i, int lane) {
    MergeIdx ix{p.n_parts, 0, 0, make_int2(0, 0), i};
    if (p.merge_cnt != nullptr) {
        const int H_kv = p.H_q / p.G;
        if (p.merge_keys != nullptr) {
            ix.key = __ldcg(p.merge_keys + i / p.G);
            ix.g = static_cast<int32_t>(i % p.G);
            ix.n = (ix.key / H_kv) * p.H_q + (ix.key % H_kv) * p.G + ix.g;
        } else {
            const int64_t tok = i / p.H_q;
            const int32_t hq = static_cast<int32_t>(i % p.H_q);
            ix.key = tok * H_kv + hq / p.G;
            ix.g = hq % p.G;
        }
        if (lane < p.merge_stride) ix.ent0 = __ldcg(p.merge_ent + ix.key * p.merge_stride + lane);
        ix.ne = __ldcg(p.merge_cnt + ix.key);
    }
    return ix;
}

// One pass of a row's merge: up to kBatch of its partials, loaded in one
// memory round trip -- lane e holds entry e's (m, l), every lane its 4 columns
// of each partial's O vector. Slots past the row's count load a valid
// duplicate of its last partial and get weight 0, so all loads are issued
// unconditionally back to back (measured on GB300: predicating them on the
// count made a decode merge about 2.5x slower). Partials are read through L2
// (ld.global.cg): in the fused path they were written by other SMs of the
// same grid.
template <int kBatch>
struct MergePass {
    float4 o[kBatch];
    float2 ml;
    int32_t cnt;
};

template <int kBatch>
__device__ __forceinline__ void merge_load(const MergeParams& p, const MergeIdx& ix, int32_t c0,
                                           int lane, MergePass<kBatch>& r) {
    r.cnt = min(kBatch, ix.ne - c0);
    const int e = min(lane, r.cnt - 1);  // lanes past the count repeat the last entry
    int64_t my_row;
    if (p.merge_cnt != nullptr) {
        int2 en;
        if (c0 == 0) {  // the first entries are in the index already
            en.x = __shfl_sync(0xffffffffu, ix.ent0.x, e);
            en.y = __shfl_sync(0xffffffffu, ix.ent0.y, e);
        } else {
            en = __ldcg(p.merge_ent + ix.key * p.merge_stride + c0 + e);
        }
        my_row = static_cast<int64_t>(en.x) * p.rows_per_part + en.y + ix.g;
    } else {
        my_row = static_cast<int64_t>(c0 + e) * p.n_out + ix.n;
    }
    const float2 ml_raw = __ldcg(p.part_ml + my_row);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
        const int64_t row = __shfl_sync(0xffffffffu, my_row, u < r.cnt ? u : r.cnt - 1);
        r.o[u] = __ldcg(reinterpret_cast<const float4*>(p.part_o + row * kHD) + lane);
    }
    r.ml = (lane < r.cnt) ? ml_raw : make_float2(-INFINITY, 0.f);
}

// Folds a loaded pass into the row's running (max, sum, O), base-2 domain.
template <int kBatch>
__device__ __forceinline__ void merge_fold(const MergePass<kBatch>& r, float& M, float& L,
                                           float4& acc) {
    float mb = (r.ml.y > 0.f) ? r.ml.x : -INFINITY;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, s));
    const float m_new = fmaxf(M, mb);
    const float corr = (M == -INFINITY) ? 0.f : ptx::ex2(M - m_new);
    const float w = (r.ml.y > 0.f) ? ptx::ex2(r.ml.x - m_new) : 0.f;  // empty shard / padding: 0
    float lb = w * r.ml.y;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) lb += __shfl_xor_sync(0xffffffffu, lb, s);
    L = L * corr + lb;
    acc.x *= corr;
    acc.y *= corr;
    acc.z *= corr;
    acc.w *= corr;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
        const float wu = __shfl_sync(0xffffffffu, w, u);  // 0 for u >= cnt
        acc.x += wu * r.o[u].x;
        acc.y += wu * r.o[u].y;
        acc.z += wu * r.o[u].z;
        acc.w += wu * r.o[u].w;
    }
    M = m_new;
}

// Folds the row whose first pass is loaded in r (loading any further passes)
// and writes out / lse. dry: the same work with nothing written (the result
// only decides a store that cannot happen): run before the partials are
// final, it brings the code and the merge index into the caches.
template <int kBatch>
__device__ __forceinline__ void merge_finish(const MergeParams& p, const MergeIdx& ix,
                                             MergePass<kBatch>& r, int lane, bool dry) {
    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    merge_fold<kBatch>(r, M, L, acc);
    for (int32_t c0 = kBatch; c0 < ix.ne; c0 += kBatch) {
        merge_load<kBatch>(p, ix, c0, lane, r);
        merge_fold<kBatch>(r, M, L, acc);
    }
    const float inv = 1.f / L;
    if (dry) {
        __shared__ float dry_sink;  // keeps the dry computation; nothing reads it
        if (acc.x * inv == 1.2345e-30f) dry_sink = acc.y;
        return;
    }
    const int64_t n = ix.n;
    if (p.out_bf16) {
        uint2 v = make_uint2(ptx::pack_bf16x2(acc.x * inv, acc.y * inv),
                             ptx::pack_bf16x2(acc.z * inv, acc.w * inv));
        reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + n * kHD)[lane] = v;
    } else {
        reinterpret_cast<float4*>(static_cast<float*>(p.out) + n * kHD)[lane] =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
    if (p.lse && lane == 0) p.lse[n] = (M + __log2f(L)) * 0.69314718055994531f;
}

// One warp merges the row its index names (output row ix.n).
template <int kBatch>
__device__ __forceinline__ void merge_row_ix(const MergeParams& p, const MergeIdx& ix, int lane,
                                             bool dry = false) {
    if (ix.ne <= 0) return;  // written directly by the attention kernel
    MergePass<kBatch> r;
    merge_load<kBatch>(p, ix, 0, lane, r);
    merge_finish<kBatch>(p, ix, r, lane, dry);
}

template <int kBatch>
__device__ __forceinline__ void merge_row(const MergeParams& p, int64_t i, int lane) {
    merge_row_ix<kBatch>(p, merge_index(p, i, lane), lane);
}

}  // namespace fanout
