// plan.cpp -- host work planner: packed query rows, split-KV units, partial slots.
//
// Rows ("AHBM Agentic Runtime Architecture" section 3.2, "Sub-agent query
// batching"; ADR-0060 TL;DR and section 5.2): per KV head, the query rows of a
// run of consecutive tokens times that head's G query heads form one 128-row
// tile (token-major, so a tile is 128/G tokens x G heads).
//
// Keys ("AHBM Agentic Runtime Architecture" sections 3.1 and 3.3):
//   * When at least two branches have new rows and the prefix is non-empty,
//     the shared prefix [0, P) is one key range for tiles packed across ALL
//     branches' rows (every new token sees the whole prefix), and each
//     branch's private suffix [P, P + S_b) is a key range for tiles of that
//     branch's rows only.
//   * Otherwise every branch's tiles take its whole context [0, P + S_b).
//   Causal: a tile's key range ends after the last key its last token sees;
//   tiles entirely in the future are never produced (ADR-0060 section 5.4).
// Split-KV (ADR-0060 section 4, FlashDecoding): each range is cut into chunks
// of whole 128-key tiles so the grid has about two units per SM; a row's
// chunks are its partial slots, merged later in ascending slot order.
#include <algorithm>
#include <cstdint>
#include <tuple>
#include <vector>

#include "fanout_internal.h"

namespace fanout {
namespace {

struct Range {
    int32_t branch, tok_begin, n_tok, lo, hi, pos_base;
    bool prefix;
};

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

int build_plan(const PlanInput& in, Plan& plan) {
    plan = Plan();
    const int32_t B = in.num_branches;
    const int32_t P = in.prefix_len;
    const int32_t G = in.H_q / in.H_kv;
    const int32_t tpt = kBM / G;
    plan.tpt = tpt;
    std::vector<int32_t> tok0(B + 1, 0);
    int active = 0;
    for (int32_t b = 0; b < B; ++b) {
        tok0[b + 1] = tok0[b] + in.q_rows[b];
        if (in.q_rows[b] > 0) ++active;
    }
    const int32_t R = tok0[B];
    plan.R = R;
    plan.tok_slots.assign(R, 0);
    if (R == 0) return 0;
    const bool shared = active >= 2 && P > 0;

    std::vector<Range> ranges;
    if (shared) {
        for (int32_t t = 0; t < R; t += tpt)
            ranges.push_back({0, t, std::min(tpt, R - t), 0, P, kNoCausal, true});
    }
    for (int32_t b = 0; b < B; ++b) {
        const int32_t T = in.q_rows[b], S = in.suffix_lens[b];
        for (int32_t t = tok0[b]; t < tok0[b + 1]; t += tpt) {
            const int32_t n = std::min(tpt, tok0[b + 1] - t);
            int32_t lo = shared ? P : 0;
            int32_t hi = P + S;
            int32_t pos_base = kNoCausal;
            if (in.causal) {
                pos_base = P + S - T - tok0[b];
                hi = std::min(hi, pos_base + t + n);  // last token's pos + 1
            }
            if (hi > lo) ranges.push_back({b, t, n, lo, hi, pos_base, false});
        }
    }

    // chunk size (in 128-key tiles) from the total work
    int64_t work = 0;
    for (const Range& r : ranges) work += cdiv(r.hi - r.lo, kBN);
    work *= in.H_kv;
    const int sms = std::max(1, in.num_sms);
    const int64_t chunk = std::max<int64_t>(4, cdiv(work, 2LL * sms));
    auto n_chunks = [&](const Range& r) -> int32_t {
        const int64_t nkt = cdiv(r.hi - r.lo, kBN);
        int64_t nch = in.force_splits > 0 ? in.force_splits : cdiv(nkt, chunk);
        return static_cast<int32_t>(std::max<int64_t>(1, std::min(nch, nkt)));
    };

    int32_t n_pre = 0;
    if (shared) n_pre = n_chunks(ranges.front());
    struct Keyed {
        int64_t work;
        int32_t chunk;
        Unit u;
    };
    std::vector<Keyed> all;
    for (const Range& r : ranges) {
        const int32_t nch = n_chunks(r);
        const int64_t nkt = cdiv(r.hi - r.lo, kBN);
        const bool direct = !shared && nch == 1;
        for (int32_t c = 0; c < nch; ++c) {
            const int32_t t_lo = static_cast<int32_t>(c * nkt / nch);
            const int32_t t_hi = static_cast<int32_t>((c + 1) * nkt / nch);
            const int32_t k_lo = r.lo + t_lo * kBN;
            const int32_t k_hi = std::min(r.hi, r.lo + t_hi * kBN);
            int32_t slot = direct ? -1 : (r.prefix ? c : n_pre + c);
            for (int32_t h = 0; h < in.H_kv; ++h)
                all.push_back({t_hi - t_lo, c,
                               Unit{h, r.branch, r.tok_begin, r.n_tok, k_lo, k_hi, r.pos_base,
                                    slot}});
        }
        if (!r.prefix) {
            const int32_t ns = direct ? 0 : n_pre + nch;
            for (int32_t t = r.tok_begin; t < r.tok_begin + r.n_tok; ++t) plan.tok_slots[t] = ns;
        }
    }
    if (shared) {
        // tokens without a private range still merge their prefix chunks
        for (int32_t t = 0; t < R; ++t)
            if (plan.tok_slots[t] == 0) plan.tok_slots[t] = n_pre;
    }
    // Longest units first; among equals, units reading the same key chunk of
    // the same KV head are adjacent so they run together and share it in L2.
    std::stable_sort(all.begin(), all.end(), [](const Keyed& a, const Keyed& b) {
        return std::make_tuple(-a.work, a.u.key_begin, a.u.kv_head, a.u.branch, a.u.tok_begin) <
               std::make_tuple(-b.work, b.u.key_begin, b.u.kv_head, b.u.branch, b.u.tok_begin);
    });
    plan.units.reserve(all.size());
    for (const Keyed& k : all) plan.units.push_back(k.u);
    int32_t ns = 0;
    for (int32_t t = 0; t < R; ++t) ns = std::max(ns, plan.tok_slots[t]);
    plan.n_slots = ns;
    plan.need_merge = ns > 0;
    return 0;
}

}  // namespace fanout
