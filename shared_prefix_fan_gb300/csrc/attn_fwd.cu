// attn_fwd.cu -- split-KV fan-out attention kernel for sm_103a (GB300).
//
// A persistent CTA (at most one per SM) runs the list of work units the
// planner assigned to it, one after the other, with the K/V ring flowing
// across unit boundaries. A unit (see Unit) is the query rows of up to
// NQ*128/G tokens x the G query heads of one KV head -- G folded into the MMA
// M dimension (ADR-0060, TL;DR and section 5.2) -- against one contiguous key
// range of one branch's logical sequence, gathered page by page through the
// branch's page table ("AHBM Agentic Runtime Architecture" section 3.1).
// Keys are swept in 128-key tiles with the FlashAttention online softmax of
// ADR-0060 section 3, in base 2 with scale*log2(e) folded:
//   S = Q K_j^T ; raise the reference max m when needed ; P = 2^(S - m) ;
//   l = l corr + rowsum P ; O = O corr + P V_j .
// m is raised only when a tile's row max exceeds it by more than 2^8 (lazy
// rescaling): P then stays <= 256, O and l stay consistent with m, and the
// O rescale in TMEM is almost never needed. Causal tiles entirely in the
// future are never produced (the planner trims each unit's key range),
// boundary tiles are masked per row (ADR-0060 section 5.4). A unit covering
// all keys of its rows writes out = O / l and lse = (m + log2 l) ln 2;
// otherwise the partial (m, l, O) goes to the unit's partial block for the
// log-sum-exp merge (ADR-0060 section 4).
//
// GB300 mapping. NQ query tiles of 128 rows per unit (NQ = 1 for short row
// blocks such as decode, 2 for long ones):
//   warp 0     TMA producer: the unit's Q tiles (3-D boxes over [R][H_q][d]),
//              then K/V tiles page by page into a ring of 32 KB stages
//              (128-byte swizzle); page ids prefetched 32 at a time.
//   warp 1     TMEM owner + single-thread tcgen05 issuer:
//              S = Q K^T with Q and K from shared memory (both K-major);
//              O += P V with P from TMEM and V from shared memory (MN-major).
//   warps 2..  one softmax warpgroup per query tile: thread i owns row i
//              (TMEM lane i); reads S (tcgen05.ld), masks, exponentiates,
//              writes P as bf16 back over the first 64 columns of its S
//              (tcgen05.st), and runs the epilogue.
// TMEM (512 columns): NQ = 2: S_0 = 0, S_1 = 128, O_0 = 256, O_1 = 384;
//                     NQ = 1: S double-buffered at 0 / 128 by tile parity, O = 256.
// Issue order of the MMA thread per K/V tile j:
//   NQ = 2: S_0(j), P.V_1(j-1), S_1(j), P.V_0(j): while one softmax group
//           works, the tensor core runs the other group's products;
//   NQ = 1: S(j), P.V(j-1): S of the next tile overlaps the softmax; this
//           runs as one stream over all of the CTA's units.
// Since tcgen05 operations of one thread execute in order, an S that reuses
// the TMEM holding an earlier P is issued after the P.V that reads that P.
// Unit boundaries: the producer issues the next unit's first K/V tile before
// it waits for the Q buffer (one Q full/free barrier pair per query tile) and
// brings the next unit's Q into L2 one unit ahead; each softmax warp keeps its
// unit's output fields in a shared-memory slot, and each group runs its
// epilogue once dry before the first unit so that code is warm.
// The producer signals the dependent merge launch once it has issued its last
// copies. Every wait is bounded (mbar_wait); on expiry the CTA records
// FANOUT_ETIMEOUT, drains its own in-flight copies and MMAs, frees TMEM and
// returns.
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "fanout_internal.h"
#include "merge_row.cuh"
#include "ptx_sm100.cuh"

namespace fanout {
namespace {

constexpr int kTileBytes = kBN * kHD * 2;   // one K or V tile, bf16
constexpr int kHalfBytes = kTileBytes / 2;  // 128 rows x 64 columns (128 B rows)
constexpr int kQBytes = kBM * kHD * 2;
constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold (base-2 units)
constexpr int kErrTimeout = 5;        // FANOUT_ETIMEOUT

template <int NQ>
struct Cfg {
    static constexpr int kStages = NQ == 1 ? 6 : 5;
    static constexpr int kThreads = 64 + 128 * NQ;
    static constexpr int kSmemQ = 0;
    static constexpr int kSmemRing = kSmemQ + NQ * kQBytes;
    static constexpr int kSmemBar = kSmemRing + kStages * kTileBytes;
    // barriers: ring full/empty, Q full/free per query tile, aux, drain, then 5
    // per softmax group
    static constexpr int BAR_FULL = 0;
    static constexpr int BAR_EMPTY = kStages;
    static constexpr int BAR_QFULL = 2 * kStages;  // + x
    static constexpr int BAR_QFREE = BAR_QFULL + NQ;  // + x
    static constexpr int BAR_AUX = BAR_QFREE + NQ;
    static constexpr int BAR_DRAIN = BAR_AUX + 1;
    static constexpr int BAR_GROUP = BAR_DRAIN + 1;  // + 5 x + {SFULL, PFULL, ODONE, OFREE, SFREE}
    static constexpr int kNumBars = BAR_GROUP + 5 * NQ;
    static constexpr int kSmemMisc = kSmemBar + kNumBars * 8;
    // 16 bytes per warp (16-byte aligned for the vector accesses): the output
    // fields of a softmax warp's current unit
    static constexpr int kSmemWarp = (kSmemMisc + 16 + 15) & ~15;
    static constexpr int kSmemTotal = kSmemWarp + 16 * (kThreads / 32);
    static_assert(kSmemWarp % 16 == 0 && kSmemBar % 1024 == 0, "shared-memory alignment");
    static constexpr int kSmemAlloc = kSmemTotal + 1024;  // base aligned up to 1024 B
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColO = 256;
    static_assert(kSmemAlloc <= 232448, "shared memory per CTA");
};

enum { SFULL = 0, PFULL = 1, ODONE = 2, OFREE = 3, SFREE = 4 };

constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(kBM, kBN, false, false);
constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kBM, kHD, false, true);

// TMEM column of the S (and P) buffer group x uses for its t-th tile.
template <int NQ>
__device__ __forceinline__ uint32_t s_col(int x, uint32_t t) {
    return NQ == 2 ? 128u * x : 128u * (t & 1u);
}

template <int NQ>
struct Smem {
    using C = Cfg<NQ>;
    uint32_t base;  // shared-window address of the 1024-aligned base
    uint8_t* ptr;   // generic pointer to the same place
    __device__ uint32_t bar(int i) const { return base + C::kSmemBar + 8u * i; }
    __device__ uint32_t gbar(int x, int which) const { return bar(C::BAR_GROUP + 5 * x + which); }
    __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(ptr + C::kSmemMisc); }
    __device__ volatile int* abort_flag() const {
        return reinterpret_cast<volatile int*>(ptr + C::kSmemMisc + 4);
    }
    __device__ volatile int* merge_go() const {
        return reinterpret_cast<volatile int*>(ptr + C::kSmemMisc + 8);
    }
};

__device__ __forceinline__ void record_timeout(const SplitParams& p, volatile int* abort_flag,
                                               int site) {
    *abort_flag = 1;
    if (atomicCAS(p.err, 0, kErrTimeout) == 0) {
        p.err[1] = site;
        p.err[2] = static_cast<int32_t>(blockIdx.x);
    }
}

__device__ __forceinline__ int unit_tiles(const Unit& u) {
    return (u.key_end - u.key_begin + kBN - 1) / kBN;
}

// Query tiles of a unit that hold at least one row.
template <int NQ>
__device__ __forceinline__ int unit_nq(const Unit& u, int tpt) {
    return (NQ == 2 && u.n_tok > tpt) ? 2 : 1;
}

// ------------------------------------------------------------------ producer
// Q tile x of unit u into its buffer (lane 0 of the producer warp), once the
// buffer's previous contents were used by their last S MMA.
template <int NQ>
__device__ __forceinline__ bool load_q(const SplitParams& p, const Smem<NQ>& sm,
                                       const CUtensorMap* tm_q, const Unit& u, int x,
                                       uint32_t& loads) {
    using C = Cfg<NQ>;
    const int lane = threadIdx.x & 31;
    if (loads > 0) {
        bool w = true;
        if (lane == 0)
            w = ptx::mbar_wait(sm.bar(C::BAR_QFREE + x), (loads - 1) & 1u, p.wait_limit_ns,
                               sm.abort_flag());
        if (!__shfl_sync(0xffffffffu, w, 0)) {
            if (lane == 0) record_timeout(p, sm.abort_flag(), 1);
            return false;
        }
    }
    if (lane == 0) {
        const uint32_t qb = sm.bar(C::BAR_QFULL + x);
        const int box_bytes = p.G * p.tpt * 128;  // one half of one query tile
        ptx::mbar_arrive_expect_tx(qb, static_cast<uint32_t>(2 * box_bytes));
        const uint32_t dst = sm.base + C::kSmemQ + x * kQBytes;
        const int y = u.kv_head * p.G, z = u.tok_begin + x * p.tpt;
        ptx::tma_load_3d(dst, tm_q, qb, 0, y, z);
        ptx::tma_load_3d(dst + kHalfBytes, tm_q, qb, 64, y, z);
    }
    ++loads;
    return true;
}

template <int NQ>
__device__ void producer_warp(const SplitParams& p, const Smem<NQ>& sm, const CUtensorMap* tm_q,
                              const CUtensorMap* tm_k, const CUtensorMap* tm_v) {
    using C = Cfg<NQ>;
    const int lane = threadIdx.x & 31;
    const uint64_t lim = p.wait_limit_ns;
    volatile int* abort = sm.abort_flag();
    const int ps = p.page_size;
    uint32_t it = 0;            // ring position
    uint32_t issued_mask = 0;   // stages ever loaded
    uint32_t issued_par = 0;    // parity of the last phase loaded per stage
    bool aux_pending = false;
    uint32_t aux_phase = 0;
    uint32_t q_loads[NQ] = {};  // loads of each Q buffer so far
    bool ok = true;
    int k = 0;
    const int ui_end = p.cta_first[blockIdx.x + 1];
    for (int ui = p.cta_first[blockIdx.x]; ui < ui_end && ok; ++ui) {
        const Unit u = p.units[ui];
        const int n_tiles = unit_tiles(u);
        if (n_tiles <= 0) continue;
        const int nq = unit_nq<NQ>(u, p.tpt);
        // The CTA's first unit loads its Q tiles first. A later unit's Q waits
        // for the previous unit's last S MMAs, so its first K/V tile is issued
        // before (the ring keeps flowing across the boundary) and its Q is
        // brought into L2 one unit ahead (the load is then an L2 hit).
        if (k == 0) {
#pragma unroll
            for (int x = 0; x < NQ; ++x)
                if (ok && x < nq) ok = load_q<NQ>(p, sm, tm_q, u, x, q_loads[x]);
        }
        if (!ok) break;
        if (lane == 0 && ui + 1 < ui_end) {
            const Unit un = p.units[ui + 1];
            if (unit_tiles(un) > 0) {
                for (int x = 0; x < unit_nq<NQ>(un, p.tpt); ++x) {
                    const int y = un.kv_head * p.G, z = un.tok_begin + x * p.tpt;
                    ptx::tma_prefetch_3d(tm_q, 0, y, z);
                    ptx::tma_prefetch_3d(tm_q, 64, y, z);
                }
            }
        }
        // Page ids of the unit, 32 per window (lane l holds page l of the window),
        // loaded one window ahead so no tile waits on the page table.
        const int32_t* prow = p.page_table + static_cast<int64_t>(u.branch) * p.max_pages +
                              u.key_begin / ps;
        const int n_pages_unit = (u.key_end - u.key_begin + ps - 1) / ps;
        const int ppt = kBN / ps;  // pages per tile: 1, 2, 4 or 8 (divides 32)
        auto load_window = [&](int w) -> int {
            const int idx = w * 32 + lane;
            return idx < n_pages_unit ? __ldg(prow + idx) : 0;
        };
        int win = 0;
        int win_cur = load_window(0);
        int win_nxt = load_window(1);
        for (int j = 0; j < n_tiles && ok; ++j) {
            const int kt = u.key_begin + j * kBN;
            const int n_valid = min(kBN, u.key_end - kt);
            const int n_pg = (n_valid + ps - 1) / ps;
            const int rel = j * ppt;  // first page of the tile, relative to the unit
            if ((rel >> 5) != win) {
                win = rel >> 5;
                win_cur = win_nxt;
                win_nxt = load_window(win + 1);
            }
            const int pg_off = rel & 31;
            for (int kv = 0; kv < 2 && ok; ++kv, ++it) {
                const uint32_t stage = it % C::kStages;
                const uint32_t par = (it / C::kStages) & 1u;
                bool w = true;
                if (lane == 0) w = ptx::mbar_wait(sm.bar(C::BAR_EMPTY + stage), par ^ 1u, lim, abort);
                if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; if (lane == 0) record_timeout(p, abort, 2); break; }
                const uint32_t dst = sm.base + C::kSmemRing + stage * kTileBytes;
                const CUtensorMap* tm = kv == 0 ? tm_k : tm_v;
                const bool partial = n_valid < kBN;
                const uint32_t bar = partial ? sm.bar(C::BAR_AUX) : sm.bar(C::BAR_FULL + stage);
                if (lane == 0) ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n_pg * ps) * 256u);
                {
                    // one lane per page of the tile: the tile's copies go out in two
                    // warp instructions (lane pg holds window entry pg_off + pg)
                    const int page = __shfl_sync(0xffffffffu, win_cur, (pg_off + lane) & 31);
                    if (lane < n_pg) {
                        const int row = (page * p.H_kv + u.kv_head) * ps;
                        const uint32_t off = static_cast<uint32_t>(lane * ps) * 128u;
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
                    if (lane == 0) w2 = ptx::mbar_wait(sm.bar(C::BAR_AUX), aux_phase, lim, abort);
                    if (!__shfl_sync(0xffffffffu, w2, 0)) { ok = false; if (lane == 0) record_timeout(p, abort, 3); break; }
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
                    if (lane == 0) ptx::mbar_arrive(sm.bar(C::BAR_FULL + stage));
                }
            }
            if (k > 0 && j == 0) {
#pragma unroll
                for (int x = 0; x < NQ; ++x)
                    if (ok && x < nq) ok = load_q<NQ>(p, sm, tm_q, u, x, q_loads[x]);
            }
        }
        ++k;
    }
    // Every copy of this CTA is issued: the dependent merge grid may be
    // scheduled now (once every CTA got here or exited), a few tiles before this
    // CTA ends, so it is resident and has made its dry pass when the last CTA
    // finishes. Signalling at the kernel's start instead kept merge blocks
    // waiting beside the attention CTAs for the whole kernel, which measured
    // 3-4 % slower on a long prefill (they take issue slots from the softmax).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (!ok && lane == 0) {
        // Drain: every copy this warp started must land before the CTA exits.
        for (int s = 0; s < C::kStages; ++s)
            if (issued_mask & (1u << s))
                ptx::mbar_wait(sm.bar(C::BAR_FULL + s), (issued_par >> s) & 1u, lim, nullptr);
        if (aux_pending) ptx::mbar_wait(sm.bar(C::BAR_AUX), aux_phase, lim, nullptr);
#pragma unroll
        for (int x = 0; x < NQ; ++x)
            if (q_loads[x] > 0)
                ptx::mbar_wait(sm.bar(C::BAR_QFULL + x), (q_loads[x] - 1) & 1u, lim, nullptr);
    }
}

// ------------------------------------------------------------------ MMA issuer
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile_base, int kk) {
    // K-major, 128-byte swizzle: 64-column halves 16 KB apart, 8-row groups 1 KB
    // apart; a 16-element K step advances 32 bytes inside the swizzle atom.
    return ptx::sdesc_sw128(tile_base + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
}
// Start-address field increment of K step kk in a K-major tile: 64-column
// halves 16 KB (1024 units of 16 B) apart, 32 B (2 units) per step inside one.
__device__ __forceinline__ uint64_t kmajor_step(int kk) {
    return static_cast<uint64_t>((kk >> 2) * (kHalfBytes >> 4) + (kk & 3) * 2);
}
__device__ __forceinline__ uint64_t vmn_desc(uint32_t tile_base, int kk) {
    // V as the B operand of P.V: MN-major (d contiguous), 128-byte swizzle.
    // LBO = distance between 64-column halves, SBO = between 8-key groups;
    // a 16-key K step advances 16 rows = 2 KB.
    return ptx::sdesc_sw128(tile_base + kk * 2048, kHalfBytes, 1024);
}

// One P.V product: group x's P of its t-th tile (counted over the CTA) times
// the V tile at ring position pos. first: the unit's first product (O is
// overwritten, and the previous unit's O of group x must have been read out:
// kx = units group x finished before).
struct PvOp {
    int x;
    uint32_t t;
    bool first;
    int kx;
    uint32_t pos;
};

template <int NQ>
__device__ __forceinline__ void issue_s(const Smem<NQ>& sm, uint32_t tmem, int x, uint32_t t,
                                        uint32_t kb) {
    using C = Cfg<NQ>;
    // (the TMEM this S overwrites held a P whose P.V was issued earlier)
    ptx::tc_fence_after();
    const uint32_t qb = sm.base + C::kSmemQ + x * kQBytes;
    const uint32_t d = tmem + s_col<NQ>(x, t);
    // descriptors of the K step 0; a step only moves the start address field
    const uint64_t dq0 = kmajor_desc(qb, 0), dk0 = kmajor_desc(kb, 0);
#pragma unroll
    for (int kk = 0; kk < kHD / 16; ++kk)
        ptx::mma_bf16_ss(d, dq0 + kmajor_step(kk), dk0 + kmajor_step(kk), kIdescQK, kk > 0);
    ptx::mma_commit(sm.gbar(x, SFULL));
}

template <int NQ>
__device__ __forceinline__ bool issue_pv(const SplitParams& p, const Smem<NQ>& sm, uint32_t tmem,
                                         const PvOp& op, uint32_t vb) {
    using C = Cfg<NQ>;
    const uint64_t lim = p.wait_limit_ns;
    volatile int* abort = sm.abort_flag();
    // P of the tile written (and O rescaled) by softmax x; for the unit's first
    // product, the previous unit's O of group x read out.
    if (!ptx::mbar_wait(sm.gbar(op.x, PFULL), op.t & 1u, lim, abort)) { record_timeout(p, abort, 14); return false; }
    if (op.first && op.kx > 0 &&
        !ptx::mbar_wait(sm.gbar(op.x, OFREE), (op.kx - 1) & 1, lim, abort)) { record_timeout(p, abort, 15); return false; }
    ptx::tc_fence_after();
    const uint32_t a = tmem + s_col<NQ>(op.x, op.t);  // P: 64 columns of bf16 pairs
    const uint32_t d = tmem + C::kColO + 128u * op.x;
    const uint64_t dv0 = vmn_desc(vb, 0);  // a 16-key step adds 2 KB: 128 in the address field
#pragma unroll
    for (int kk = 0; kk < kBN / 16; ++kk)
        ptx::mma_bf16_ts(d, a + 8u * kk, dv0 + 128u * kk, kIdescPV, (!op.first || kk > 0) ? 1u : 0u);
    ptx::mma_commit(sm.gbar(op.x, ODONE));
    return true;
}

// The held P.V, if any (its V stage is released once it completes).
template <int NQ>
__device__ __forceinline__ bool issue_held(const SplitParams& p, const Smem<NQ>& sm, uint32_t tmem,
                                           const PvOp& op, bool& held) {
    using C = Cfg<NQ>;
    if (!held) return true;
    held = false;
    const uint32_t stage = op.pos % C::kStages;
    if (!ptx::mbar_wait(sm.bar(C::BAR_FULL + stage), (op.pos / C::kStages) & 1u, p.wait_limit_ns,
                        sm.abort_flag())) {
        record_timeout(p, sm.abort_flag(), 13);
        return false;
    }
    if (!issue_pv<NQ>(p, sm, tmem, op, sm.base + C::kSmemRing + stage * kTileBytes)) return false;
    ptx::mma_commit(sm.bar(C::BAR_EMPTY + stage));
    return true;
}

// The single tcgen05 issuer, two query tiles per unit: per K/V tile j the
// order S_0(j), P.V_1(j-1), S_1(j), P.V_0(j), so that one tile's softmax runs
// while the tensor core works on the other's products (ping-pong); the unit's
// last P.V_1 is issued before the next unit starts. Units with one query tile
// run S_0(j), P.V_0(j).
template <int NQ>
__device__ void mma_thread_pair(const SplitParams& p, const Smem<NQ>& sm, uint32_t tmem) {
    using C = Cfg<NQ>;
    const uint64_t lim = p.wait_limit_ns;
    volatile int* abort = sm.abort_flag();
    bool ok = true;
    bool issued_any = false;
    uint32_t it0 = 0;          // ring position of the unit's K_0 (K_j at it0+2j, V_j at it0+2j+1)
    uint32_t jt0 = 0, jt1 = 0;  // tiles each softmax group processed before this unit
    int kx0 = 0, kx1 = 0;      // units each softmax group processed before this unit
    uint32_t qu0 = 0, qu1 = 0;  // loads of each Q buffer consumed so far
    auto stage_of = [&](uint32_t pos) { return pos % C::kStages; };
    auto wait_full = [&](uint32_t pos, int site) -> bool {
        if (ptx::mbar_wait(sm.bar(C::BAR_FULL + stage_of(pos)), (pos / C::kStages) & 1u, lim, abort))
            return true;
        record_timeout(p, abort, site);
        return false;
    };
    auto ring = [&](uint32_t pos) { return sm.base + C::kSmemRing + stage_of(pos) * kTileBytes; };
    const int ui_end = p.cta_first[blockIdx.x + 1];
    for (int ui = p.cta_first[blockIdx.x]; ui < ui_end && ok; ++ui) {
        const Unit u = p.units[ui];
        const int n = unit_tiles(u);
        if (n <= 0) continue;
        const bool two = unit_nq<NQ>(u, p.tpt) == 2;
        if (!ptx::mbar_wait(sm.bar(C::BAR_QFULL), qu0 & 1u, lim, abort) ||
            (two && !ptx::mbar_wait(sm.bar(C::BAR_QFULL + 1), qu1 & 1u, lim, abort))) {
            ok = false;
            record_timeout(p, abort, 10);
            break;
        }
        for (int j = 0; j <= n && ok; ++j) {
            const uint32_t posK = it0 + 2u * j, posV = posK + 1u, posVp = posK - 1u;
            if (two) {
                if (j < n) {
                    if (!(ok = wait_full(posK, 11))) break;
                    issue_s<NQ>(sm, tmem, 0, jt0 + j, ring(posK));
                    issued_any = true;
                    if (j == n - 1) ptx::mma_commit(sm.bar(C::BAR_QFREE));
                }
                if (j > 0) {
                    const PvOp pv1{1, jt1 + j - 1, j == 1, kx1, posVp};
                    if (!(ok = issue_pv<NQ>(p, sm, tmem, pv1, ring(posVp)))) break;
                    ptx::mma_commit(sm.bar(C::BAR_EMPTY + stage_of(posVp)));
                }
                if (j < n) {
                    issue_s<NQ>(sm, tmem, 1, jt1 + j, ring(posK));
                    ptx::mma_commit(sm.bar(C::BAR_EMPTY + stage_of(posK)));
                    if (j == n - 1) ptx::mma_commit(sm.bar(C::BAR_QFREE + 1));
                    if (!(ok = wait_full(posV, 13))) break;
                    const PvOp pv0{0, jt0 + j, j == 0, kx0, posV};
                    if (!(ok = issue_pv<NQ>(p, sm, tmem, pv0, ring(posV)))) break;
                }
            } else if (j < n) {
                if (!(ok = wait_full(posK, 11))) break;
                issue_s<NQ>(sm, tmem, 0, jt0 + j, ring(posK));
                issued_any = true;
                ptx::mma_commit(sm.bar(C::BAR_EMPTY + stage_of(posK)));
                if (j == n - 1) ptx::mma_commit(sm.bar(C::BAR_QFREE));
                if (!(ok = wait_full(posV, 13))) break;
                const PvOp pv0{0, jt0 + j, j == 0, kx0, posV};
                if (!(ok = issue_pv<NQ>(p, sm, tmem, pv0, ring(posV)))) break;
                ptx::mma_commit(sm.bar(C::BAR_EMPTY + stage_of(posV)));
            }
        }
        if (!ok) break;
        it0 += 2u * n;
        jt0 += n;
        ++kx0;
        ++qu0;
        if (two) {
            jt1 += n;
            ++kx1;
            ++qu1;
        }
    }
    if (!ok && issued_any) {
        ptx::mma_commit(sm.bar(C::BAR_DRAIN));
        ptx::mbar_wait(sm.bar(C::BAR_DRAIN), 0, lim, nullptr);
    }
}

// The single tcgen05 issuer, one query tile per unit: S(t) into one of two S
// buffers, then P.V(t-1), as one stream over all of the CTA's units (t counts
// the CTA's tiles). A unit's last P.V is held back and issued after the next
// unit's first S, so the S double buffer stays full across the boundary; if
// that unit's Q has not landed yet the held P.V goes first.
template <int NQ>
__device__ void mma_thread_stream(const SplitParams& p, const Smem<NQ>& sm, uint32_t tmem) {
    using C = Cfg<NQ>;
    const uint64_t lim = p.wait_limit_ns;
    volatile int* abort = sm.abort_flag();
    bool ok = true;
    bool issued_any = false;
    uint32_t it0 = 0;   // ring position of the unit's K_0 (K_j at it0+2j, V_j at it0+2j+1)
    uint32_t jt = 0;    // tiles processed before this unit
    int kx = 0;         // units processed before this unit
    uint32_t qu = 0;    // Q loads consumed so far
    PvOp pend{0, 0, false, 0, 0};
    bool has_pend = false;
    const int ui_end = p.cta_first[blockIdx.x + 1];
    for (int ui = p.cta_first[blockIdx.x]; ui < ui_end && ok; ++ui) {
        const Unit u = p.units[ui];
        const int n = unit_tiles(u);
        if (n <= 0) continue;
        if (has_pend && !ptx::mbar_test_wait(sm.bar(C::BAR_QFULL), qu & 1u) &&
            !(ok = issue_held<NQ>(p, sm, tmem, pend, has_pend)))
            break;
        for (int j = 0; j < n && ok; ++j) {
            const uint32_t posK = it0 + 2u * j, t = jt + j;
            const uint32_t stage = posK % C::kStages;
            if (!ptx::mbar_wait(sm.bar(C::BAR_FULL + stage), (posK / C::kStages) & 1u, lim, abort)) {
                ok = false;
                record_timeout(p, abort, 11);
                break;
            }
            // S(t) waits until the softmax has read S(t-1), so S-full never runs
            // two phases ahead
            if (t > 0 && !ptx::mbar_wait(sm.gbar(0, SFREE), (t - 1) & 1u, lim, abort)) {
                ok = false;
                record_timeout(p, abort, 12);
                break;
            }
            if (j == 0 && !ptx::mbar_wait(sm.bar(C::BAR_QFULL), qu & 1u, lim, abort)) {
                ok = false;
                record_timeout(p, abort, 10);
                break;
            }
            issue_s<NQ>(sm, tmem, 0, t, sm.base + C::kSmemRing + stage * kTileBytes);
            issued_any = true;
            ptx::mma_commit(sm.bar(C::BAR_EMPTY + stage));
            if (j == n - 1) ptx::mma_commit(sm.bar(C::BAR_QFREE));
            if (!(ok = issue_held<NQ>(p, sm, tmem, pend, has_pend))) break;
            pend = PvOp{0, t, j == 0, kx, posK + 1u};
            has_pend = true;
        }
        if (!ok) break;
        it0 += 2u * n;
        jt += n;
        ++kx;
        ++qu;
    }
    if (ok) ok = issue_held<NQ>(p, sm, tmem, pend, has_pend);
    if (!ok && issued_any) {
        ptx::mma_commit(sm.bar(C::BAR_DRAIN));
        ptx::mbar_wait(sm.bar(C::BAR_DRAIN), 0, lim, nullptr);
    }
}

// ------------------------------------------------------------------ softmax
__device__ __forceinline__ float max8(const float (&a)[8]) {
    return fmaxf(fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3])),
                 fmaxf(fmaxf(a[4], a[5]), fmaxf(a[6], a[7])));
}
__device__ __forceinline__ float sum8(const float (&a)[8]) {
    return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
}

// Group x owns query tile x of every unit (rows 128x .. 128x+127); thread i
// owns row i of the tile (TMEM lane i). A warp whose 32 rows are all padding
// follows the barrier protocol but skips the TMEM traffic and the math.
template <int NQ>
__device__ void softmax_group(const SplitParams& p, const Smem<NQ>& sm, uint32_t tmem, int x) {
    using C = Cfg<NQ>;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t colO = C::kColO + 128u * x;
    const uint64_t lim = p.wait_limit_ns;
    volatile int* abort = sm.abort_flag();
    const float sl2 = p.scale_log2;
    const int rows_per_part = kBM * NQ;
    // the epilogue's fields of the current unit (token start, KV head, partial
    // block), kept in this warp's shared-memory slot rather than in registers
    // through the tile loop or re-read from global memory under load
    const uint32_t slot = sm.base + C::kSmemWarp + 16u * warp;
    uint32_t jt = 0;
    bool ok = true;
    // Before the first unit the group makes a dry run of the epilogue (no
    // tiles, no waits, one thread's stores into a scratch sink) while it waits
    // for its first K/V tile anyway: the epilogue code is otherwise first
    // fetched in the middle of the kernel, from a cold instruction cache, with
    // the memory system saturated by the other CTAs (measured: a unit's first
    // epilogue took 6-7 us in decode, a later one 0.8 us).
    const int ui_first = p.cta_first[blockIdx.x], ui_end = p.cta_first[blockIdx.x + 1];
    for (int ui = ui_first < ui_end ? ui_first - 1 : ui_first; ui < ui_end && ok; ++ui) {
        const bool dry = ui < ui_first;
        const Unit u = p.units[dry ? ui_first : ui];
        const int n_tiles = dry ? 0 : unit_tiles(u);
        if (!dry && (n_tiles <= 0 || x >= unit_nq<NQ>(u, p.tpt))) continue;
        const int urow = kBM * x + row;  // row within the unit
        const bool row_valid = dry ? (lane == 0 && quarter == 0) : urow < u.n_tok * p.G;
        if (lane == 0)
            ptx::st_shared_v4(slot, static_cast<uint32_t>(u.tok_begin), static_cast<uint32_t>(u.kv_head),
                              static_cast<uint32_t>(u.part), 0u);
        __syncwarp();
        const bool active = dry || __any_sync(0xffffffffu, row_valid);
        // Only the key start and this row's visible end stay live through the
        // tile loop (registers).
        const int key_begin = u.key_begin;
        const int vis_end = row_valid ? min(u.key_end, u.pos_base + u.tok_begin + urow / p.G + 1) : 0;
        float m_ref = -INFINITY, l_run = 0.f;
        for (int j = 0; j < n_tiles; ++j, ++jt) {
            const int kt = key_begin + j * kBN;
            bool w = ptx::mbar_wait(sm.gbar(x, SFULL), jt & 1u, lim, abort);
            if (!__all_sync(0xffffffffu, w)) { ok = false; record_timeout(p, abort, 20); break; }
            ptx::tc_fence_after();
            if (NQ == 1) {
                // S(jt) seen: the MMA may issue S(jt+1) into the other S buffer
                // (its S-full then cannot run two phases ahead of this wait).
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(sm.gbar(x, SFREE));
            }
            const uint32_t colS = s_col<NQ>(x, jt);
            float corr = 1.f;
            if (active) {
                const int lim_c = vis_end - kt;
                const bool full = __all_sync(0xffffffffu, lim_c >= kBN);
                uint32_t s[kBN];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t (&chunk)[32] = *reinterpret_cast<uint32_t (*)[32]>(&s[32 * c]);
                    ptx::tmem_ld32(lane_addr + colS + 32 * c, chunk);
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t (&chunk)[32] = *reinterpret_cast<uint32_t (*)[32]>(&s[32 * c]);
                    if (c == 0) ptx::tmem_ld_wait(chunk); else ptx::reg_touch(chunk);
                }
                if (!full) {
#pragma unroll
                    for (int c = 0; c < kBN; ++c)
                        if (c >= lim_c) s[c] = __float_as_uint(-INFINITY);
                }
                float mx[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) mx[q] = -INFINITY;
#pragma unroll
                for (int c = 0; c < kBN; c += 2)  // three-input max: two columns per step
                    mx[(c >> 1) & 7] = ptx::fmax3(mx[(c >> 1) & 7], __uint_as_float(s[c]),
                                                  __uint_as_float(s[c + 1]));
                const float mt = max8(mx) * sl2;  // scale > 0: max commutes with scaling
                if (mt > m_ref + kRescaleLog2) {
                    corr = (m_ref == -INFINITY) ? 0.f : ptx::ex2(m_ref - mt);
                    m_ref = mt;
                }
                const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
                // column pairs on the packed fp32x2 pipe: one FMA and one add per
                // two columns (the exponentials stay on the MUFU, one per column);
                // P is packed to bf16 pairs in place as the pairs are consumed
                uint64_t sm2[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) sm2[q] = 0ull;
                const uint64_t sl2p = ptx::f32x2(sl2, sl2), negm = ptx::f32x2(-m_use, -m_use);
#pragma unroll
                for (int c = 0; c < kBN; c += 2) {
                    const uint64_t t = ptx::fma_f32x2(ptx::f32x2(__uint_as_float(s[c]),
                                                                 __uint_as_float(s[c + 1])),
                                                      sl2p, negm);
                    const float e0 = ptx::ex2(ptx::lo_f32(t)), e1 = ptx::ex2(ptx::hi_f32(t));
                    sm2[(c >> 1) & 3] = ptx::add_f32x2(sm2[(c >> 1) & 3], ptx::f32x2(e0, e1));
                    s[c >> 1] = ptx::pack_bf16x2(e0, e1);
                }
                float sm8[8];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    sm8[2 * q] = ptx::lo_f32(sm2[q]);
                    sm8[2 * q + 1] = ptx::hi_f32(sm2[q]);
                }
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t (&chunk)[32] = *reinterpret_cast<uint32_t (*)[32]>(&s[32 * c]);
                    ptx::tmem_st32(lane_addr + colS + 32 * c, chunk);
                }
                l_run = l_run * corr + sum8(sm8);
                ptx::tmem_st_wait();
            }
            // The previous P.V must be done before O is rescaled in place. With one
            // query tile the wait comes every tile: it also keeps P-full from
            // running two phases ahead of the MMA thread (S of the next tile does
            // not wait for P.V). With two, S_x(j) is issued after P_x.V(j-1), so
            // S-full already implies that P.V completed: no wait is needed.
            const bool rescale = j > 0 && __any_sync(0xffffffffu, corr != 1.f);
            if (NQ == 1 && j > 0) {
                w = ptx::mbar_wait(sm.gbar(x, ODONE), (jt - 1) & 1u, lim, abort);
                if (!__all_sync(0xffffffffu, w)) { ok = false; record_timeout(p, abort, 21); break; }
                ptx::tc_fence_after();
            }
            if (rescale) {
                uint32_t r[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    ptx::tmem_ld32(lane_addr + colO + 32 * c, r);
                    ptx::tmem_ld_wait(r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * corr);
                    ptx::tmem_st32(lane_addr + colO + 32 * c, r);
                }
                ptx::tmem_st_wait();
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(sm.gbar(x, PFULL));
        }
        if (!ok) break;
        // Epilogue: the last P.V done -> this row of O to global memory (the
        // dry run: O's TMEM columns are not written before the first P.V, which
        // waits for this group; its stores go to the sink).
        if (!dry) {
            bool w = ptx::mbar_wait(sm.gbar(x, ODONE), (jt - 1) & 1u, lim, abort);
            if (!__all_sync(0xffffffffu, w)) { ok = false; record_timeout(p, abort, 22); break; }
        }
        ptx::tc_fence_after();
        if (active) {
            const uint4 f = ptx::ld_shared_v4(slot);
            const int e_part = static_cast<int>(f.z);
            const int tok = static_cast<int>(f.x) + urow / p.G;
            const int hq = static_cast<int>(f.y) * p.G + urow % p.G;
            const int64_t orow = dry ? 0 : static_cast<int64_t>(tok) * p.H_q + hq;
            const int64_t prow = dry ? 0 : static_cast<int64_t>(e_part) * rows_per_part + urow;
            void* const out_base = dry ? static_cast<void*>(p.sink) : p.out;
            float* const po_base = dry ? p.sink : p.part_o;
            float* const lse_base = dry ? p.sink : p.lse;
            float2* const ml_base = dry ? reinterpret_cast<float2*>(p.sink) : p.part_ml;
            const bool direct = e_part < 0;
            const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                __syncwarp();  // converged for the warp-collective TMEM load
                ptx::tmem_ld32(lane_addr + colO + 32 * c, r);
                ptx::tmem_ld_wait(r);
                if (!row_valid) {
                } else if (direct && p.out_bf16) {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out_base) +
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
                } else if (direct) {
                    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out_base) +
                                                            orow * kHD + 32 * c);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(r[4 * i + 0]) * inv_l,
                                             __uint_as_float(r[4 * i + 1]) * inv_l,
                                             __uint_as_float(r[4 * i + 2]) * inv_l,
                                             __uint_as_float(r[4 * i + 3]) * inv_l);
                } else {
                    // Partial O (unnormalised): each thread writes its own row, so a
                    // warp store touches 32 rows; 256-bit stores (whole sectors)
                    // halve the store instructions. The partial buffer is 256-byte
                    // aligned and rows are 512 bytes.
                    float* dst = po_base + prow * kHD + 32 * c;
#pragma unroll
                    for (int i = 0; i < 4; ++i) ptx::st_global_v8(dst + 8 * i, r + 8 * i);
                }
            }
            if (row_valid) {
                if (direct) {
                    if (lse_base) lse_base[orow] = (m_ref + __log2f(l_run)) * 0.69314718055994531f;
                } else {
                    ml_base[prow] = make_float2(m_ref, l_run);
                }
            }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0 && !dry) ptx::mbar_arrive(sm.gbar(x, OFREE));
    }
}

// ------------------------------------------------------------------ merge tail
// The log-sum-exp merge of the split-KV partials inside this grid (launched
// cooperatively, so every CTA is resident): each CTA publishes the call's
// epoch once its partials are written, waits (bounded) until every CTA has,
// then merges a contiguous slice of the output rows. This replaces the
// separate merge launch.
//
// The merge is latency bound, and this code runs once per launch from a cold
// instruction cache, so it is written as short rolled loops. Each warp takes
// its rows in chunks of up to kChunkRows: the chunk's merge index (plan data;
// the first chunk's read before the wait) costs two round trips, lane k
// reading row k's count and then every lane one entry; every partial O row of
// the chunk then comes into the warp's share of the idle Q + K/V ring by
// cp.async (16 B per lane, nothing held in registers) with the (m, l) pairs
// beside it, after one wait each row folds from shared memory in the passes
// and order of merge_row, so both paths give the same results. A row with more
// partials than the share holds falls back to merge_row.
constexpr int kChunkRows = 8;

template <int NQ>
struct MergeStage {
    using C = Cfg<NQ>;
    static constexpr int kWarps = C::kThreads / 32;
    static constexpr uint32_t kRegion = (C::kSmemBar / kWarps) & ~1023u;  // bytes per warp
    static constexpr uint32_t kTab = kChunkRows * 24;  // per row: key (8 B), ne, first, g
    static constexpr int kSlots = (kRegion - kTab) / (512 + 16);  // O + row index + (m, l)
    static_assert(kWarps * kRegion <= C::kSmemBar, "staging stays below the barriers");
};

// Reads the merge index of the chunk starting at row n (rows n, n + kWarps,
// ...), fills the warp's row table and slot list, returns the rows taken.
template <int NQ>
__device__ __noinline__ int merge_chunk_index(const MergeParams& mp, int64_t n, int64_t r1,
                                              uint8_t* region, int lane) {
    using M = MergeStage<NQ>;
    int64_t* tkey = reinterpret_cast<int64_t*>(region + M::kSlots * 528);
    int* tne = reinterpret_cast<int*>(tkey + kChunkRows);
    int* tfirst = tne + kChunkRows;
    int* tg = tfirst + kChunkRows;
    int64_t* sidx = reinterpret_cast<int64_t*>(region + M::kSlots * 512);
    const int64_t nk = n + static_cast<int64_t>(lane) * M::kWarps;
    const bool valid = lane < kChunkRows && nk < r1;
    const int H_kv = mp.H_q / mp.G;
    int cnt = 0, g = 0;
    int64_t key = 0;
    if (valid) {
        const int64_t tok = nk / mp.H_q;
        const int hq = static_cast<int>(nk % mp.H_q);
        key = tok * H_kv + hq / mp.G;
        g = hq % mp.G;
        cnt = __ldcg(mp.merge_cnt + key);
    }
    const int take = (cnt > 0 && cnt <= M::kSlots) ? cnt : 0;
    int incl = take;
    for (int d = 1; d < kChunkRows; d <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += t;
    }
    const unsigned fit = __ballot_sync(0xffffffffu, valid && incl <= M::kSlots);
    const int rows = __popc(fit);  // valid rows and fitting rows are both prefixes
    const int nslot = rows > 0 ? __shfl_sync(0xffffffffu, incl, rows - 1) : 0;
    if (lane < rows) {
        tkey[lane] = key;
        tne[lane] = (cnt > M::kSlots) ? -1 : max(cnt, 0);
        tfirst[lane] = incl - take;
        tg[lane] = g;
    }
    __syncwarp();
    for (int s = lane; s < nslot; s += 32) {
        int k = 0;
        while (k + 1 < rows && tfirst[k + 1] <= s) ++k;
        const int2 en = __ldcg(mp.merge_ent + tkey[k] * mp.merge_stride + (s - tfirst[k]));
        sidx[s] = static_cast<int64_t>(en.x) * mp.rows_per_part + en.y + tg[k];
    }
    __syncwarp();
    return rows;
}

// Pulls a warp's chunk of partials into its slots (cp.async for the O rows,
// every one in flight before the (m, l) loads), folds each row from shared
// memory and writes out / lse. dry: the same instructions, but the results stay
// in shared memory -- run while the other CTAs finish (reading partials that
// may not be final, which is harmless), it brings this code into the
// instruction cache: after an L2 flush a cold fetch of it costs microseconds
// on the critical path of the last CTA.
template <int NQ>
__device__ __noinline__ void merge_chunk_run(const MergeParams& mp, int64_t n, int rows,
                                             uint8_t* region, uint32_t region_s, int lane,
                                             bool dry) {
    using M = MergeStage<NQ>;
    float* so = reinterpret_cast<float*>(region);
    const int64_t* sidx = reinterpret_cast<const int64_t*>(region + M::kSlots * 512);
    float2* sml = reinterpret_cast<float2*>(region + M::kSlots * 520);
    const int* tne = reinterpret_cast<const int*>(region + M::kSlots * 528 + kChunkRows * 8);
    const int* tfirst = tne + kChunkRows;
    int nslot = 0;
    for (int k = 0; k < rows; ++k)
        if (tne[k] > 0) nslot = tfirst[k] + tne[k];
    for (int s2 = 0; s2 < nslot; ++s2)
        ptx::cp_async_16(region_s + s2 * 512 + lane * 16, mp.part_o + sidx[s2] * kHD + lane * 4);
    for (int s2 = lane; s2 < nslot; s2 += 32) {  // (m, l) through L2 into shared
        const float2 v = __ldcg(mp.part_ml + sidx[s2]);
        sml[s2] = v;
    }
    ptx::cp_async_wait_all();
    __syncwarp();
    const int kb = (mp.merge_stride <= 8) ? 8 : 24;  // the pass size merge_row uses
    for (int k = 0; k < rows; ++k) {
        const int64_t nk = n + static_cast<int64_t>(k) * M::kWarps;
        const int c = tne[k];
        if (c == 0) continue;
        if (c < 0) {
            if (!dry) merge_row<24>(mp, nk, lane);
            continue;
        }
        const int f = tfirst[k];
        float Mx = -INFINITY, L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c0 = 0; c0 < c; c0 += kb) {
            const int cnt = min(kb, c - c0);
            const float2 ml = (lane < cnt) ? sml[f + c0 + lane] : make_float2(-INFINITY, 0.f);
            float mb = (ml.y > 0.f) ? ml.x : -INFINITY;
            for (int s = 16; s > 0; s >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, s));
            const float m_new = fmaxf(Mx, mb);
            const float corr = (Mx == -INFINITY) ? 0.f : ptx::ex2(Mx - m_new);
            const float w = (ml.y > 0.f) ? ptx::ex2(ml.x - m_new) : 0.f;
            float lb = w * ml.y;
            for (int s = 16; s > 0; s >>= 1) lb += __shfl_xor_sync(0xffffffffu, lb, s);
            L = L * corr + lb;
            acc.x *= corr;
            acc.y *= corr;
            acc.z *= corr;
            acc.w *= corr;
            for (int u = 0; u < cnt; ++u) {
                const float wu = __shfl_sync(0xffffffffu, w, u);
                const float4 o = reinterpret_cast<const float4*>(so + (f + c0 + u) * kHD)[lane];
                acc.x += wu * o.x;
                acc.y += wu * o.y;
                acc.z += wu * o.z;
                acc.w += wu * o.w;
            }
            Mx = m_new;
        }
        const float inv = 1.f / L;
        if (dry) {
            reinterpret_cast<float4*>(so)[lane] =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, Mx + __log2f(L));
        } else if (mp.out_bf16) {
            uint2 v = make_uint2(ptx::pack_bf16x2(acc.x * inv, acc.y * inv),
                                 ptx::pack_bf16x2(acc.z * inv, acc.w * inv));
            reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(mp.out) + nk * kHD)[lane] = v;
        } else {
            reinterpret_cast<float4*>(static_cast<float*>(mp.out) + nk * kHD)[lane] =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
        if (!dry && mp.lse && lane == 0) mp.lse[nk] = (Mx + __log2f(L)) * 0.69314718055994531f;
    }
    __syncwarp();
}

template <int NQ>
__device__ __noinline__ void merge_tail(const SplitParams& p, const Smem<NQ>& sm) {
    using M = MergeStage<NQ>;
    const MergeParams& mp = p.merge;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // The __syncthreads before this call orders every partial store of the CTA
    // before thread 0's fence and release.
    if (threadIdx.x == 0) {
        __threadfence();
        ptx::st_release_gpu(p.flags + blockIdx.x, p.epoch);
    }
    const int64_t n_out = mp.n_out;
    const int64_t per = (n_out + gridDim.x - 1) / gridDim.x;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * per;
    const int64_t r1 = min(n_out, r0 + per);
    uint8_t* region = sm.ptr + warp * M::kRegion;
    const uint32_t region_s = sm.base + warp * M::kRegion;
    // Every role is done and every MMA / TMA of this CTA has completed: the
    // ring is free. Order its last async-proxy use before the writes below.
    ptx::fence_proxy_async_smem();
    int64_t n = r0 + warp;
    int rows = (n < r1) ? merge_chunk_index<NQ>(mp, n, r1, region, lane) : 0;
    // While other CTAs are still working, warp 1 makes a dry run of its first
    // chunk (instruction cache, and L2 for the CTAs that finish last); a CTA
    // that finds almost every flag set already skips it.
    if (warp == 1 && rows > 0) {
        int unset = 0;
        for (int c = lane; c < static_cast<int>(gridDim.x); c += 32)
            unset += ptx::ld_relaxed_gpu(p.flags + c) != p.epoch;
        for (int s = 16; s > 0; s >>= 1) unset += __shfl_xor_sync(0xffffffffu, unset, s);
        if (unset > 8) merge_chunk_run<NQ>(mp, n, rows, region, region_s, lane, true);
    }

    if (warp == 0) {
        bool all = false;
        const uint64_t t0 = ptx::globaltimer_ns();
        for (;;) {
            // all of this lane's flags in one round trip (relaxed loads; the
            // fence after the loop orders the reads that depend on them)
            bool mine = true;
            for (int c = lane; c < static_cast<int>(gridDim.x); c += 32)
                mine &= ptx::ld_relaxed_gpu(p.flags + c) == p.epoch;
            if (__all_sync(0xffffffffu, mine)) {
                all = true;
                break;
            }
            if (ptx::globaltimer_ns() - t0 > p.wait_limit_ns) break;
        }
        __threadfence();  // acquire side of the flags; the barrier below extends it to the CTA
        if (lane == 0) {
            if (!all && atomicCAS(p.err, 0, kErrTimeout) == 0) {
                p.err[1] = 30;
                p.err[2] = static_cast<int32_t>(blockIdx.x);
            }
            *sm.merge_go() = all ? 1 : 0;
        }
    }
    __syncthreads();
    if (!*sm.merge_go()) return;
    while (rows > 0) {
        merge_chunk_run<NQ>(mp, n, rows, region, region_s, lane, false);  // ends with __syncwarp
        n += static_cast<int64_t>(rows) * M::kWarps;
        rows = (n < r1) ? merge_chunk_index<NQ>(mp, n, r1, region, lane) : 0;
    }
}

template <int NQ>
__global__ void __launch_bounds__(Cfg<NQ>::kThreads, 1) __maxnreg__(NQ == 2 ? 200 : 255)
    attn_fwd_kernel(const __grid_constant__ SplitParams p,
                    const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v) {
    using C = Cfg<NQ>;
    extern __shared__ uint8_t smem_raw[];
    Smem<NQ> sm;
    {
        const uint32_t raw = ptx::smem_u32(smem_raw);
        const uint32_t aligned = (raw + 1023u) & ~1023u;
        sm.base = aligned;
        sm.ptr = smem_raw + (aligned - raw);
    }
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(sm.bar(C::BAR_FULL + s), 1);
            ptx::mbar_init(sm.bar(C::BAR_EMPTY + s), 1);
        }
        for (int x = 0; x < NQ; ++x) {
            ptx::mbar_init(sm.bar(C::BAR_QFULL + x), 1);
            ptx::mbar_init(sm.bar(C::BAR_QFREE + x), 1);
        }
        ptx::mbar_init(sm.bar(C::BAR_AUX), 1);
        ptx::mbar_init(sm.bar(C::BAR_DRAIN), 1);
        for (int x = 0; x < NQ; ++x) {
            ptx::mbar_init(sm.gbar(x, SFULL), 1);
            // P-full, O-free, S-free: one arrival per softmax warp (lane 0, after
            // the warp's own TMEM traffic and a warp barrier), not 128
            ptx::mbar_init(sm.gbar(x, PFULL), 4);
            ptx::mbar_init(sm.gbar(x, ODONE), 1);
            ptx::mbar_init(sm.gbar(x, OFREE), 4);
            ptx::mbar_init(sm.gbar(x, SFREE), 4);
        }
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
        ptx::tmem_alloc(ptx::smem_u32(sm.tmem_slot()), C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *sm.tmem_slot();

    if (warp == 0) {
        producer_warp<NQ>(p, sm, &tm_q, &tm_k, &tm_v);
    } else if (warp == 1) {
        if (lane == 0) {
            if (NQ == 2) mma_thread_pair<NQ>(p, sm, tmem);
            else mma_thread_stream<NQ>(p, sm, tmem);
        }
        __syncwarp();
    } else {
        softmax_group<NQ>(p, sm, tmem, (warp - 2) >> 2);
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
    if (p.fused_merge) merge_tail<NQ>(p, sm);
}

template <int NQ>
cudaError_t launch_nq(const SplitParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                      const CUtensorMap& tm_v, int grid, bool cooperative, cudaStream_t stream) {
    // The shared-memory attribute is set once per device (under a lock: calls
    // on several host threads may arrive here together).
    static std::atomic<bool> attr_set[64];
    static std::mutex attr_mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool known = dev >= 0 && dev < 64;
    if (!known || !attr_set[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(attr_mu);
        if (!known || !attr_set[dev].load(std::memory_order_relaxed)) {
            e = cudaFuncSetAttribute(attn_fwd_kernel<NQ>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Cfg<NQ>::kSmemAlloc);
            if (e != cudaSuccess) return e;
            if (known) attr_set[dev].store(true, std::memory_order_release);
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(Cfg<NQ>::kThreads);
    cfg.dynamicSmemBytes = Cfg<NQ>::kSmemAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cooperative ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, attn_fwd_kernel<NQ>, p, tm_q, tm_k, tm_v);
}

}  // namespace

cudaError_t launch_split_attn(const SplitParams& p, const CUtensorMap& tm_q,
                              const CUtensorMap& tm_k, const CUtensorMap& tm_v, int grid,
                              bool cooperative, cudaStream_t stream) {
    return p.nq == 2 ? launch_nq<2>(p, tm_q, tm_k, tm_v, grid, cooperative, stream)
                     : launch_nq<1>(p, tm_q, tm_k, tm_v, grid, cooperative, stream);
}

}  // namespace fanout
