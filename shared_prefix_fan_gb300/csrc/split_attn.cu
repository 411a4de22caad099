// split_attn.cu -- split-KV fan-out attention kernel for sm_103a (GB300).
//
// What one CTA computes (per work unit, see Unit in fanout_internal.h):
//   the query rows of up to 128/G tokens x the G query heads of one KV head,
//   folded into the MMA M dimension (ADR-0060, TL;DR and section 5.2: "G folded
//   into M, no broadcast"), against one contiguous key range of one branch's
//   logical sequence, gathered page by page through the branch's page table
//   ("AHBM Agentic Runtime Architecture" section 3.1). The keys are swept in
//   128-key tiles with the FlashAttention online softmax (ADR-0060 section 3):
//     S = Q K_j^T ; m_new = max(m, rowmax S) ; P = exp(S - m_new) ;
//     corr = exp(m - m_new) ; l = l corr + rowsum P ; O = O corr + P V_j ,
//   done here in base 2 with the scale folded into log2(e). Causal tiles
//   entirely in the future are never produced (the planner trims the key
//   range), boundary tiles are masked per row (ADR-0060 section 5.4).
//   A unit covering a row's whole key range writes out = O / l and
//   lse = (m + log2 l) ln 2; otherwise it writes the partial (m, l, O) for the
//   log-sum-exp merge (ADR-0060 section 4).
//
// GB300 mapping:
//   warp 0      TMA producer: Q tile once per unit (3-D box over [R][H_q][d]),
//               K/V tiles page by page into a 4-stage ring (2-D boxes over the
//               page pool, 128-byte swizzle), stage released by MMA commits.
//   warp 1      TMEM owner + single-thread tcgen05 MMA issuer:
//               S(TMEM cols 0..127) = Q . K^T  (both K-major, smem),
//               O(TMEM cols 128..255) += P . V (P K-major smem, V MN-major smem).
//   warps 2..5  softmax warpgroup: thread i owns row i (TMEM lane i); reads S
//               from TMEM, masks, exponentiates, rescales O in TMEM when the
//               running max grows, writes P (bf16, swizzled) to smem, and runs
//               the epilogue.
// Every wait is bounded (mbar_wait); on expiry the CTA records
// FANOUT_ETIMEOUT, drains its own in-flight copies and MMAs, frees TMEM and
// returns.
#include <cuda_bf16.h>

#include "fanout_internal.h"
#include "ptx_sm100.cuh"

namespace fanout {
namespace {

constexpr int kStages = 4;
constexpr int kTileBytes = kBN * kHD * 2;   // one K or V tile, bf16
constexpr int kHalfBytes = kTileBytes / 2;  // 128 rows x 64 columns (128 B rows)
constexpr int kQBytes = kBM * kHD * 2;
constexpr int kPBytes = kBM * kBN * 2;

constexpr int kSmemQ = 0;
constexpr int kSmemRing = kSmemQ + kQBytes;
constexpr int kSmemP = kSmemRing + kStages * kTileBytes;
constexpr int kSmemBar = kSmemP + kPBytes;

enum : int {
    BAR_FULL = 0,
    BAR_EMPTY = kStages,
    BAR_QFULL = 2 * kStages,
    BAR_QFREE,
    BAR_SFULL,
    BAR_SFREE,
    BAR_PFULL,
    BAR_ODONE,
    BAR_OFREE,
    BAR_AUX,
    BAR_DRAIN,
    NUM_BARS
};
constexpr int kSmemMisc = kSmemBar + NUM_BARS * 8;
constexpr int kSmemTotal = kSmemMisc + 16;
constexpr int kSmemAlloc = kSmemTotal + 1024;  // slack to align the base to 1024 B

constexpr int kThreads = 192;
constexpr int kSoftmaxThreads = 128;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 128;

constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(kBM, kBN, false, false);
constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kBM, kHD, false, true);

constexpr int kErrTimeout = 5;  // FANOUT_ETIMEOUT

struct Smem {
    uint32_t base;  // shared-window address of the 1024-aligned base
    uint8_t* ptr;   // generic pointer to the same place
    __device__ uint32_t bar(int i) const { return base + kSmemBar + 8u * i; }
    __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(ptr + kSmemMisc); }
    __device__ volatile int* abort_flag() const {
        return reinterpret_cast<volatile int*>(ptr + kSmemMisc + 4);
    }
};

__device__ __forceinline__ void record_timeout(const SplitParams& p, const Smem& sm, int site) {
    *sm.abort_flag() = 1;
    if (atomicCAS(p.err, 0, kErrTimeout) == 0) {
        p.err[1] = site;
        p.err[2] = static_cast<int32_t>(blockIdx.x);
    }
}

// ------------------------------------------------------------------ producer
__device__ void producer_warp(const SplitParams& p, const Smem& sm, const CUtensorMap* tm_q,
                              const CUtensorMap* tm_k, const CUtensorMap* tm_v) {
    const int lane = threadIdx.x & 31;
    const uint64_t lim = p.wait_limit_ns;
    const volatile int* abort = sm.abort_flag();
    const int ps = p.page_size;
    const int box_rows = p.G * p.tpt;
    uint32_t it = 0;            // ring position
    uint32_t issued_mask = 0;   // stages ever loaded
    uint32_t issued_par = 0;    // parity of the last phase loaded per stage
    bool aux_pending = false;
    uint32_t aux_phase = 0;
    bool ok = true;
    int k = 0;
    for (int ui = blockIdx.x; ui < p.n_units && ok; ui += gridDim.x) {
        const Unit u = p.units[ui];
        const int n_tiles = (u.key_end - u.key_begin + kBN - 1) / kBN;
        if (n_tiles <= 0) continue;
        // Q tile: the Q buffer is free once the previous unit's last S MMA completed.
        if (k > 0) {
            bool w = true;
            if (lane == 0) w = ptx::mbar_wait(sm.bar(BAR_QFREE), (k - 1) & 1, lim, abort);
            if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; if (lane == 0) record_timeout(p, sm, 1); break; }
        }
        if (lane == 0) {
            const uint32_t qb = sm.bar(BAR_QFULL);
            ptx::mbar_arrive_expect_tx(qb, 2u * box_rows * 128u);
            const int y = u.kv_head * p.G;
            ptx::tma_load_3d(sm.base + kSmemQ, tm_q, qb, 0, y, u.tok_begin);
            ptx::tma_load_3d(sm.base + kSmemQ + kHalfBytes, tm_q, qb, 64, y, u.tok_begin);
        }
        const int32_t* prow = p.page_table + static_cast<int64_t>(u.branch) * p.max_pages;
        for (int j = 0; j < n_tiles && ok; ++j) {
            const int kt = u.key_begin + j * kBN;
            const int n_valid = min(kBN, u.key_end - kt);
            const int n_pg = (n_valid + ps - 1) / ps;
            const int pg0 = kt / ps;
            int my_page = (lane < n_pg) ? __ldg(prow + pg0 + lane) : 0;
            for (int kv = 0; kv < 2 && ok; ++kv, ++it) {
                const uint32_t stage = it % kStages;
                const uint32_t par = (it / kStages) & 1u;
                bool w = true;
                if (lane == 0) w = ptx::mbar_wait(sm.bar(BAR_EMPTY + stage), par ^ 1u, lim, abort);
                if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; if (lane == 0) record_timeout(p, sm, 2); break; }
                const uint32_t dst = sm.base + kSmemRing + stage * kTileBytes;
                const CUtensorMap* tm = kv == 0 ? tm_k : tm_v;
                const bool partial = n_valid < kBN;
                const uint32_t bar = partial ? sm.bar(BAR_AUX) : sm.bar(BAR_FULL + stage);
                if (lane == 0) ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n_pg * ps) * 256u);
                for (int pg = 0; pg < n_pg; ++pg) {
                    const int page = __shfl_sync(0xffffffffu, my_page, pg);
                    if (lane == 0) {
                        const int row = (page * p.H_kv + u.kv_head) * ps;
                        const uint32_t off = static_cast<uint32_t>(pg * ps) * 128u;
                        ptx::tma_load_2d(dst + off, tm, bar, 0, row);
                        ptx::tma_load_2d(dst + kHalfBytes + off, tm, bar, 64, row);
                    }
                }
                if (lane == 0) {
                    issued_mask |= 1u << stage;
                    issued_par = (issued_par & ~(1u << stage)) | (par << stage);
                }
                if (partial) {
                    // Tail tile: wait for the pages, then zero every row past the
                    // last valid key so no stale value reaches the MMAs.
                    aux_pending = true;
                    bool w2 = true;
                    if (lane == 0) w2 = ptx::mbar_wait(sm.bar(BAR_AUX), aux_phase, lim, abort);
                    if (!__shfl_sync(0xffffffffu, w2, 0)) { ok = false; if (lane == 0) record_timeout(p, sm, 3); break; }
                    aux_pending = false;
                    aux_phase ^= 1u;
                    const int n_zero = (kBN - n_valid) * 16;  // 16-byte chunks, both halves
                    for (int idx = lane; idx < n_zero; idx += 32) {
                        const int r = n_valid + (idx >> 4);
                        const int ch = idx & 15;
                        const uint32_t a = dst + (ch >> 3) * kHalfBytes + r * 128 + (ch & 7) * 16;
                        ptx::st_shared_v4(a, 0u, 0u, 0u, 0u);
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(sm.bar(BAR_FULL + stage));
                }
            }
        }
        ++k;
    }
    if (!ok && lane == 0) {
        // Drain: every copy this warp started must land before the CTA exits.
        for (int s = 0; s < kStages; ++s)
            if (issued_mask & (1u << s))
                ptx::mbar_wait(sm.bar(BAR_FULL + s), (issued_par >> s) & 1u, lim, nullptr);
        if (aux_pending) ptx::mbar_wait(sm.bar(BAR_AUX), aux_phase, lim, nullptr);
    }
}

// ------------------------------------------------------------------ MMA issuer
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile_base, int kk) {
    // K-major, 128-byte swizzle: 64-column halves 16 KB apart, 8-row groups 1 KB
    // apart; a 16-element K step advances 32 bytes inside the swizzle atom.
    return ptx::sdesc_sw128(tile_base + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t vmn_desc(uint32_t tile_base, int kk) {
    // V as the B operand of P.V: MN-major (d contiguous), 128-byte swizzle.
    // LBO = distance between 64-column halves, SBO = between 8-key groups;
    // a 16-key K step advances 16 rows = 2 KB.
    return ptx::sdesc_sw128(tile_base + kk * 2048, kHalfBytes, 1024);
}

__device__ void mma_thread(const SplitParams& p, const Smem& sm, uint32_t tmem) {
    const uint64_t lim = p.wait_limit_ns;
    const volatile int* abort = sm.abort_flag();
    const uint32_t tS = tmem + kColS, tO = tmem + kColO;
    uint32_t it0 = 0;  // ring position of this unit's K_0 (K_j at it0+2j, V_j at it0+2j+1)
    uint32_t jt = 0;   // tiles processed by this CTA before this unit
    bool ok = true;
    bool issued_any = false;
    int k = 0;
    for (int ui = blockIdx.x; ui < p.n_units && ok; ui += gridDim.x) {
        const Unit u = p.units[ui];
        const int n_tiles = (u.key_end - u.key_begin + kBN - 1) / kBN;
        if (n_tiles <= 0) continue;
        if (!ptx::mbar_wait(sm.bar(BAR_QFULL), k & 1, lim, abort)) { ok = false; record_timeout(p, sm, 10); break; }
        for (int j = 0; j <= n_tiles && ok; ++j) {
            if (j < n_tiles) {
                // S_j = Q K_j^T
                const uint32_t pos = it0 + 2u * j;
                const uint32_t st = pos % kStages, par = (pos / kStages) & 1u;
                if (!ptx::mbar_wait(sm.bar(BAR_FULL + st), par, lim, abort)) { ok = false; record_timeout(p, sm, 11); break; }
                if (jt + j > 0 && !ptx::mbar_wait(sm.bar(BAR_SFREE), (jt + j - 1) & 1u, lim, abort)) { ok = false; record_timeout(p, sm, 12); break; }
                ptx::tc_fence_after();
                const uint32_t kb = sm.base + kSmemRing + st * kTileBytes;
                const uint32_t qb = sm.base + kSmemQ;
#pragma unroll
                for (int kk = 0; kk < kHD / 16; ++kk)
                    ptx::mma_bf16_ss(tS, kmajor_desc(qb, kk), kmajor_desc(kb, kk), kIdescQK, kk > 0);
                issued_any = true;
                ptx::mma_commit(sm.bar(BAR_SFULL));
                ptx::mma_commit(sm.bar(BAR_EMPTY + st));
                if (j == n_tiles - 1) ptx::mma_commit(sm.bar(BAR_QFREE));
            }
            if (j > 0) {
                // O (+)= P_{j-1} V_{j-1}
                const int jj = j - 1;
                const uint32_t pos = it0 + 2u * jj + 1u;
                const uint32_t st = pos % kStages, par = (pos / kStages) & 1u;
                if (!ptx::mbar_wait(sm.bar(BAR_FULL + st), par, lim, abort)) { ok = false; record_timeout(p, sm, 13); break; }
                if (!ptx::mbar_wait(sm.bar(BAR_PFULL), (jt + jj) & 1u, lim, abort)) { ok = false; record_timeout(p, sm, 14); break; }
                if (jj == 0 && k > 0 && !ptx::mbar_wait(sm.bar(BAR_OFREE), (k - 1) & 1, lim, abort)) { ok = false; record_timeout(p, sm, 15); break; }
                ptx::tc_fence_after();
                const uint32_t vb = sm.base + kSmemRing + st * kTileBytes;
                const uint32_t pb = sm.base + kSmemP;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    ptx::mma_bf16_ss(tO, kmajor_desc(pb, kk), vmn_desc(vb, kk), kIdescPV,
                                     (jj > 0 || kk > 0) ? 1u : 0u);
                ptx::mma_commit(sm.bar(BAR_ODONE));
                ptx::mma_commit(sm.bar(BAR_EMPTY + st));
            }
        }
        it0 += 2u * n_tiles;
        jt += n_tiles;
        ++k;
    }
    if (!ok && issued_any) {
        ptx::mma_commit(sm.bar(BAR_DRAIN));
        ptx::mbar_wait(sm.bar(BAR_DRAIN), 0, lim, nullptr);
    }
}

// ------------------------------------------------------------------ softmax
// Thread i of the warpgroup owns query row i of the tile (TMEM lane i). A warp
// whose 32 rows are all padding follows the same barrier protocol but skips
// the TMEM traffic and the math, so arrivals always land in the right phase.
__device__ void softmax_warps(const SplitParams& p, const Smem& sm, uint32_t tmem) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint64_t lim = p.wait_limit_ns;
    const volatile int* abort = sm.abort_flag();
    const float sl2 = p.scale_log2;
    const uint32_t p_row = sm.base + kSmemP + row * 128;
    const int sw = row & 7;
    uint32_t jt = 0;
    bool ok = true;
    for (int ui = blockIdx.x; ui < p.n_units && ok; ui += gridDim.x) {
        const Unit u = p.units[ui];
        const int n_tiles = (u.key_end - u.key_begin + kBN - 1) / kBN;
        if (n_tiles <= 0) continue;
        const bool row_valid = row < u.n_tok * p.G;
        const bool active = __any_sync(0xffffffffu, row_valid);
        const int tok = u.tok_begin + row / p.G;
        const int hq = u.kv_head * p.G + row % p.G;
        const int vis_end = row_valid ? min(u.key_end, u.pos_base + tok + 1) : 0;
        float m_run = -INFINITY, l_run = 0.f;
        for (int j = 0; j < n_tiles; ++j, ++jt) {
            const int kt = u.key_begin + j * kBN;
            bool w = ptx::mbar_wait(sm.bar(BAR_SFULL), jt & 1u, lim, abort);
            if (!__all_sync(0xffffffffu, w)) { ok = false; record_timeout(p, sm, 20); break; }
            ptx::tc_fence_after();
            float x[kBN];
            if (active) {
                uint32_t r[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    ptx::tmem_ld32(lane_addr + kColS + 32 * c, r);
                    ptx::tmem_ld_wait(r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[32 * c + i] = __uint_as_float(r[i]);
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(sm.bar(BAR_SFREE));
            float corr = 1.f;
            if (active) {
                const int lim_c = vis_end - kt;  // visible columns of this tile for this row
                float mt = -INFINITY;
                if (lim_c >= kBN) {
#pragma unroll
                    for (int c = 0; c < kBN; ++c) {
                        x[c] *= sl2;
                        mt = fmaxf(mt, x[c]);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < kBN; ++c) {
                        x[c] = (c < lim_c) ? x[c] * sl2 : -INFINITY;
                        mt = fmaxf(mt, x[c]);
                    }
                }
                const float m_new = fmaxf(m_run, mt);
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                corr = (m_new == m_run) ? 1.f : ptx::ex2(m_run - m_use);
                float sum = 0.f;
#pragma unroll
                for (int c = 0; c < kBN; ++c) {
                    x[c] = ptx::ex2(x[c] - m_use);
                    sum += x[c];
                }
                l_run = l_run * corr + sum;
                m_run = m_new;
            }
            if (j > 0) {
                // PV of the previous tile done: O is stable and the P buffer is free.
                w = ptx::mbar_wait(sm.bar(BAR_ODONE), (jt - 1) & 1u, lim, abort);
                if (!__all_sync(0xffffffffu, w)) { ok = false; record_timeout(p, sm, 21); break; }
                ptx::tc_fence_after();
                if (active && __any_sync(0xffffffffu, corr != 1.f)) {
                    uint32_t r[32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        ptx::tmem_ld32(lane_addr + kColO + 32 * c, r);
                        ptx::tmem_ld_wait(r);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            r[i] = __float_as_uint(__uint_as_float(r[i]) * corr);
                        ptx::tmem_st32(lane_addr + kColO + 32 * c, r);
                    }
                    ptx::tmem_st_wait();
                }
            }
            // (At j == 0 the previous unit's epilogue already waited for its last
            // PV, so the P buffer is free and O will be overwritten.)
            if (active) {
                // P (bf16) into the K-major, 128-byte-swizzled A tile of P.V.
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint32_t a = p_row + (c >> 3) * kHalfBytes + (((c & 7) ^ sw) << 4);
                    ptx::st_shared_v4(a, ptx::pack_bf16x2(x[8 * c + 0], x[8 * c + 1]),
                                      ptx::pack_bf16x2(x[8 * c + 2], x[8 * c + 3]),
                                      ptx::pack_bf16x2(x[8 * c + 4], x[8 * c + 5]),
                                      ptx::pack_bf16x2(x[8 * c + 6], x[8 * c + 7]));
                }
                ptx::fence_proxy_async_smem();
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(sm.bar(BAR_PFULL));
        }
        if (!ok) break;
        // Epilogue: last PV done -> this row of O to global memory.
        bool w = ptx::mbar_wait(sm.bar(BAR_ODONE), (jt - 1) & 1u, lim, abort);
        if (!__all_sync(0xffffffffu, w)) { ok = false; record_timeout(p, sm, 22); break; }
        ptx::tc_fence_after();
        if (active) {
            const int64_t orow = static_cast<int64_t>(tok) * p.H_q + hq;
            const bool direct = u.slot < 0;
            const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                ptx::tmem_ld32(lane_addr + kColO + 32 * c, r);
                ptx::tmem_ld_wait(r);
                if (!row_valid) continue;
                if (direct && p.out_bf16) {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                                          orow * kHD + 32 * c);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_uint4(
                            ptx::pack_bf16x2(__uint_as_float(r[8 * i + 0]) * inv_l,
                                             __uint_as_float(r[8 * i + 1]) * inv_l),
                            ptx::pack_bf16x2(__uint_as_float(r[8 * i + 2]) * inv_l,
                                             __uint_as_float(r[8 * i + 3]) * inv_l),
                            ptx::pack_bf16x2(__uint_as_float(r[8 * i + 4]) * inv_l,
                                             __uint_as_float(r[8 * i + 5]) * inv_l),
                            ptx::pack_bf16x2(__uint_as_float(r[8 * i + 6]) * inv_l,
                                             __uint_as_float(r[8 * i + 7]) * inv_l));
                } else {
                    const float sc = direct ? inv_l : 1.f;
                    float* base = direct ? static_cast<float*>(p.out) + orow * kHD
                                         : p.part_o + (static_cast<int64_t>(u.slot) * p.R * p.H_q +
                                                       orow) * kHD;
                    float4* dst = reinterpret_cast<float4*>(base + 32 * c);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(r[4 * i + 0]) * sc,
                                             __uint_as_float(r[4 * i + 1]) * sc,
                                             __uint_as_float(r[4 * i + 2]) * sc,
                                             __uint_as_float(r[4 * i + 3]) * sc);
                }
            }
            if (row_valid) {
                if (direct) {
                    if (p.lse) p.lse[orow] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
                } else {
                    p.part_ml[static_cast<int64_t>(u.slot) * p.R * p.H_q + orow] =
                        make_float2(m_run, l_run);
                }
            }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(sm.bar(BAR_OFREE));
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    split_attn_kernel(const __grid_constant__ SplitParams p,
                      const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ uint8_t smem_raw[];
    Smem sm;
    {
        const uint32_t raw = ptx::smem_u32(smem_raw);
        const uint32_t aligned = (raw + 1023u) & ~1023u;
        sm.base = aligned;
        sm.ptr = smem_raw + (aligned - raw);
    }
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(sm.bar(BAR_FULL + s), 1);
            ptx::mbar_init(sm.bar(BAR_EMPTY + s), 1);
        }
        ptx::mbar_init(sm.bar(BAR_QFULL), 1);
        ptx::mbar_init(sm.bar(BAR_QFREE), 1);
        ptx::mbar_init(sm.bar(BAR_SFULL), 1);
        ptx::mbar_init(sm.bar(BAR_SFREE), kSoftmaxThreads);
        ptx::mbar_init(sm.bar(BAR_PFULL), kSoftmaxThreads);
        ptx::mbar_init(sm.bar(BAR_ODONE), 1);
        ptx::mbar_init(sm.bar(BAR_OFREE), kSoftmaxThreads);
        ptx::mbar_init(sm.bar(BAR_AUX), 1);
        ptx::mbar_init(sm.bar(BAR_DRAIN), 1);
        *sm.abort_flag() = 0;
        ptx::fence_barrier_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(sm.tmem_slot()), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *sm.tmem_slot();

    if (warp == 0) {
        producer_warp(p, sm, &tm_q, &tm_k, &tm_v);
    } else if (warp == 1) {
        if (lane == 0) mma_thread(p, sm, tmem);
        __syncwarp();
    } else {
        softmax_warps(p, sm, tmem);
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

int split_attn_smem_bytes() { return kSmemAlloc; }

cudaError_t launch_split_attn(const SplitParams& p, const CUtensorMap& tm_q,
                              const CUtensorMap& tm_k, const CUtensorMap& tm_v, int grid,
                              cudaStream_t stream) {
    static bool attr_set[64] = {};  // the attribute is set once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(split_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemAlloc);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    split_attn_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(p, tm_q, tm_k, tm_v);
    return cudaGetLastError();
}

}  // namespace fanout
