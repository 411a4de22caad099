// plan.cpp -- host work planner: packed query rows, split-KV units, their
// assignment to persistent CTAs, and the merge index.
//
// Rows ("AHBM Agentic Runtime Architecture" section 3.2, "Sub-agent query
// batching"; ADR-0060 TL;DR and section 5.2): per KV head, the query rows of a
// run of consecutive tokens times that head's G query heads form a unit of
// one or two 128-row query tiles (token-major: 128/G tokens x G heads each).
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
//
// Split-KV (ADR-0060 section 4; "AHBM Agentic Runtime Architecture" 2.2/3.3):
// each range is cut into chunks of whole 128-key tiles. The chunk size comes
// from a small cost model -- the analogue of the pages' policy estimate
// T_A vs T_B ("AHBM Agentic Runtime Architecture" section 4.5) on one GPU:
//   time(C) = max over CTAs of sum(tiles + unit overhead)     (LPT assignment)
//           + partial-merge traffic spread over the CTAs + merge launch,
// evaluated for a ladder of chunk sizes C and for an exact-balance split
// (contiguous per-CTA quotas of tiles, Stream-K style); smallest estimate wins.
// Units are assigned to at most one persistent CTA per SM, longest first to
// the least-loaded CTA. Among equal units the order is (key chunk, KV head,
// row tile), so equal units land round-robin and the k-th units of all CTAs
// read the same key chunk at about the same time (shared through L2).
#include <algorithm>
#include <cstdint>
#include <functional>
#include <queue>
#include <tuple>
#include <vector>

#include "plan.h"

namespace fanout {
namespace {

using Range = PlanRange;

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Prologue + epilogue of a unit, in tile times: two query tiles per unit
// (tensor-bound tiles of ~1.8 us) and one (HBM-bound tiles of ~1.4 us, whose
// unit boundaries measured 3-5 us).
constexpr double kUnitOverhead2 = 2.0;
constexpr double kUnitOverhead1 = 3.0;
constexpr double kMergePerPart = 2.0;  // write + read of one 128-row partial, in tile times
constexpr double kMergeLaunch = 4.0;   // the extra merge launch, in tile times

struct Cand {
    std::vector<Unit> units;   // in assignment order
    std::vector<int64_t> work;
    std::vector<int32_t> cta_of;
    std::vector<int32_t> range_of;
    int32_t n_cta = 0;
    double cost = 0;
};

// Cut the ranges with chunk size `chunk` tiles (0 = whole ranges), sort, assign.
void make_candidate(const std::vector<Range>& ranges, int64_t chunk, int32_t force_splits,
                    int32_t max_cta, double unit_ovh, Cand& c) {
    struct Keyed {
        int64_t work;
        Unit u;
        bool whole;
        int32_t range;
    };
    std::vector<Keyed> all;
    for (size_t ri = 0; ri < ranges.size(); ++ri) {
        const Range& r = ranges[ri];
        const int64_t nkt = cdiv(r.hi - r.lo, kBN);
        int64_t nch = force_splits > 0 ? force_splits : (chunk > 0 ? cdiv(nkt, chunk) : 1);
        nch = std::max<int64_t>(1, std::min(nch, nkt));
        for (int64_t ch = 0; ch < nch; ++ch) {
            const int64_t t_lo = ch * nkt / nch, t_hi = (ch + 1) * nkt / nch;
            const int32_t k_lo = r.lo + static_cast<int32_t>(t_lo) * kBN;
            const int32_t k_hi = std::min<int32_t>(r.hi, r.lo + static_cast<int32_t>(t_hi) * kBN);
            all.push_back({t_hi - t_lo,
                           Unit{r.kv_head, r.branch, r.tok_begin, r.n_tok, k_lo, k_hi, r.pos_base,
                                0},
                           r.complete && nch == 1, static_cast<int32_t>(ri)});
        }
    }
    std::stable_sort(all.begin(), all.end(), [](const Keyed& a, const Keyed& b) {
        return std::make_tuple(-a.work, a.u.key_begin, a.u.kv_head, a.u.branch, a.u.tok_begin) <
               std::make_tuple(-b.work, b.u.key_begin, b.u.kv_head, b.u.branch, b.u.tok_begin);
    });
    c.n_cta = static_cast<int32_t>(std::min<int64_t>(max_cta, static_cast<int64_t>(all.size())));
    c.units.clear();
    c.work.clear();
    c.cta_of.clear();
    c.range_of.clear();
    using Slot = std::pair<double, int32_t>;
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
    for (int32_t i = 0; i < c.n_cta; ++i) heap.push({0.0, i});
    double makespan = 0;
    int64_t n_parts = 0;
    for (const Keyed& k : all) {
        Slot s = heap.top();
        heap.pop();
        s.first += static_cast<double>(k.work) + unit_ovh;
        makespan = std::max(makespan, s.first);
        heap.push(s);
        Unit u = k.u;
        u.part = k.whole ? -1 : 0;  // partial indices are numbered later
        if (!k.whole) ++n_parts;
        c.units.push_back(u);
        c.work.push_back(k.work);
        c.cta_of.push_back(s.second);
        c.range_of.push_back(k.range);
    }
    c.cost = makespan + (n_parts > 0 ? kMergeLaunch + kMergePerPart * n_parts / c.n_cta : 0.0);
}

// A lower bound of make_candidate's cost for chunk size `chunk` (whole-range
// chunking when 0), from the pieces' sizes alone: the busiest CTA carries at
// least the largest piece and at least the average load. A candidate whose
// bound cannot beat the best so far is skipped without being built.
double candidate_cost_bound(const std::vector<Range>& ranges, int64_t chunk, int32_t max_cta,
                            double unit_ovh) {
    int64_t n = 0, n_parts = 0, total = 0, max_w = 0;
    for (const Range& r : ranges) {
        const int64_t nkt = cdiv(r.hi - r.lo, kBN);
        int64_t nch = chunk > 0 ? cdiv(nkt, chunk) : 1;
        nch = std::max<int64_t>(1, std::min(nch, nkt));
        for (int64_t ch = 0; ch < nch; ++ch)
            max_w = std::max(max_w, (ch + 1) * nkt / nch - ch * nkt / nch);
        total += nkt;
        n += nch;
        if (!(r.complete && nch == 1)) n_parts += nch;
    }
    const int32_t n_cta = static_cast<int32_t>(std::min<int64_t>(max_cta, n));
    const double makespan =
        std::max(static_cast<double>(max_w) + unit_ovh,
                 (static_cast<double>(total) + unit_ovh * static_cast<double>(n)) / n_cta);
    return makespan + (n_parts > 0 ? kMergeLaunch + kMergePerPart * n_parts / n_cta : 0.0);
}

// Exact-balance candidate (Stream-K style): the ranges' tiles laid end to end
// and cut into one contiguous quota per CTA; a CTA's quota may end inside a
// range and the next CTA continues it.
void make_streamk(const std::vector<Range>& ranges, int32_t max_cta, double unit_ovh, Cand& c) {
    int64_t total = 0;
    for (const Range& r : ranges) total += cdiv(r.hi - r.lo, kBN);
    const int32_t n_cta = static_cast<int32_t>(std::min<int64_t>(max_cta, total));
    // per-CTA quota in tile times, counting one unit overhead per range and per
    // cut (about one cut per CTA)
    const double quota = (static_cast<double>(total) +
                          unit_ovh * static_cast<double>(ranges.size() + n_cta)) / n_cta;
    c.units.clear();
    c.work.clear();
    c.cta_of.clear();
    c.range_of.clear();
    std::vector<double> load(n_cta, 0.0);
    int32_t cta = 0;
    int64_t n_parts = 0;
    for (size_t ri = 0; ri < ranges.size(); ++ri) {
        const Range& r = ranges[ri];
        const int64_t nkt = cdiv(r.hi - r.lo, kBN);
        int64_t t = 0;
        while (t < nkt) {
            const double room = quota - load[cta] - unit_ovh;
            if (room < 0.5 && load[cta] > 0 && cta + 1 < n_cta) {
                ++cta;
                continue;
            }
            int64_t take = nkt - t;
            if (cta + 1 < n_cta)
                take = std::min<int64_t>(take, std::max<int64_t>(1, static_cast<int64_t>(room + 0.5)));
            const int32_t k_lo = r.lo + static_cast<int32_t>(t) * kBN;
            const int32_t k_hi = std::min<int32_t>(r.hi, r.lo + static_cast<int32_t>(t + take) * kBN);
            const bool whole = r.complete && take == nkt;
            c.units.push_back(Unit{r.kv_head, r.branch, r.tok_begin, r.n_tok, k_lo, k_hi, r.pos_base,
                                   whole ? -1 : 0});
            if (!whole) ++n_parts;
            c.work.push_back(take);
            c.cta_of.push_back(cta);
            c.range_of.push_back(static_cast<int32_t>(ri));
            load[cta] += static_cast<double>(take) + unit_ovh;
            t += take;
        }
    }
    c.n_cta = cta + 1;
    double makespan = 0;
    for (double l : load) makespan = std::max(makespan, l);
    c.cost = makespan + (n_parts > 0 ? kMergeLaunch + kMergePerPart * n_parts / c.n_cta : 0.0);
}

// Longest first with tail cuts: pieces go to the least-loaded CTA, largest
// first (as in make_candidate with whole ranges); a piece that would lift that
// CTA above the balanced load is cut there and its remainder goes back into
// the queue. The leading waves keep the lockstep order of the whole-range plan
// (the CTAs' first units read the same key chunks at about the same time) and
// only the cut pieces become partials.
void make_lpt_cut(const std::vector<Range>& ranges, int32_t max_cta, double unit_ovh, Cand& c) {
    struct Piece {
        int64_t work;
        int32_t range;
        int64_t t_lo;  // first tile of the piece within its range
        // the queue's order after the size: first key, KV head, branch, token
        int32_t k_lo, kv_head, branch, tok_begin;
    };
    int64_t total = 0;
    std::vector<int64_t> nkt(ranges.size());
    for (size_t i = 0; i < ranges.size(); ++i) {
        nkt[i] = cdiv(ranges[i].hi - ranges[i].lo, kBN);
        total += nkt[i];
    }
    const int32_t n_cta = static_cast<int32_t>(std::min<int64_t>(max_cta, total));
    const double target = (static_cast<double>(total) +
                           unit_ovh * static_cast<double>(ranges.size() + n_cta)) / n_cta;
    auto later = [](const Piece& a, const Piece& b) {
        return std::make_tuple(-b.work, b.k_lo, b.kv_head, b.branch, b.tok_begin) <
               std::make_tuple(-a.work, a.k_lo, a.kv_head, a.branch, a.tok_begin);
    };
    auto piece = [&](int64_t work, int32_t ri, int64_t t_lo) {
        const Range& r = ranges[ri];
        return Piece{work, ri, t_lo, r.lo + static_cast<int32_t>(t_lo) * kBN, r.kv_head, r.branch,
                     r.tok_begin};
    };
    std::priority_queue<Piece, std::vector<Piece>, decltype(later)> queue(later);
    for (size_t i = 0; i < ranges.size(); ++i)
        if (nkt[i] > 0) queue.push(piece(nkt[i], static_cast<int32_t>(i), 0));
    using Slot = std::pair<double, int32_t>;
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
    for (int32_t i = 0; i < n_cta; ++i) heap.push({0.0, i});
    c.units.clear();
    c.work.clear();
    c.cta_of.clear();
    c.range_of.clear();
    std::vector<bool> cut(ranges.size(), false);
    std::vector<int32_t>& range_of = c.range_of;
    double makespan = 0;
    while (!queue.empty()) {
        Piece pc = queue.top();
        queue.pop();
        Slot s = heap.top();
        heap.pop();
        int64_t take = pc.work;
        const double room = target - s.first - unit_ovh;
        if (s.first + unit_ovh + static_cast<double>(pc.work) > target + 0.5 && room >= 1.0 &&
            pc.work >= 2) {
            take = std::min<int64_t>(pc.work - 1, static_cast<int64_t>(room));
            queue.push(piece(pc.work - take, pc.range, pc.t_lo + take));
            cut[pc.range] = true;
        }
        const Range& r = ranges[pc.range];
        const int32_t k_lo = r.lo + static_cast<int32_t>(pc.t_lo) * kBN;
        const int32_t k_hi = std::min<int32_t>(r.hi, r.lo + static_cast<int32_t>(pc.t_lo + take) * kBN);
        c.units.push_back(Unit{r.kv_head, r.branch, r.tok_begin, r.n_tok, k_lo, k_hi, r.pos_base, 0});
        c.work.push_back(take);
        c.cta_of.push_back(s.second);
        range_of.push_back(pc.range);
        s.first += static_cast<double>(take) + unit_ovh;
        makespan = std::max(makespan, s.first);
        heap.push(s);
    }
    // CTAs that received nothing (fewer pieces than CTAs) are dropped
    std::vector<int32_t> renum(n_cta, -1);
    int32_t used = 0;
    for (int32_t& cta : c.cta_of) {
        if (renum[cta] < 0) renum[cta] = used++;
        cta = renum[cta];
    }
    // a range left whole that covers every visible key of its rows is written
    // directly; every other piece is a partial
    int64_t n_parts = 0;
    for (size_t i = 0; i < c.units.size(); ++i) {
        const int32_t ri = range_of[i];
        const bool whole = ranges[ri].complete && !cut[ri];
        c.units[i].part = whole ? -1 : 0;
        if (!whole) ++n_parts;
    }
    c.n_cta = used;
    c.cost = makespan + (n_parts > 0 ? kMergeLaunch + kMergePerPart * n_parts / c.n_cta : 0.0);
}

// The key ranges of a problem (rows x keys before any split-KV cut), and the
// row geometry: R tokens, nq query tiles per unit, tpt tokens per tile.
void make_ranges(const PlanInput& in, std::vector<Range>& ranges, int32_t& R, int32_t& nq,
                 int32_t& tpt_tile) {
    ranges.clear();
    const int32_t B = in.num_branches;
    // A prefix that ends inside a page: the whole pages are the shared range;
    // the tail of the last prefix page is read through each branch's own table
    // entry like its private keys (after a copy-on-write fork that entry is a
    // private copy). Positions do not change: P + S_b = P_al + (S_b + tail).
    const int32_t tail = in.prefix_len % in.page_size;
    const int32_t P = in.prefix_len - tail;
    std::vector<int32_t> S_eff(B);
    for (int32_t b = 0; b < B; ++b) S_eff[b] = in.suffix_lens[b] + tail;
    const int32_t G = in.H_q / in.H_kv;
    std::vector<int32_t> tok0(B + 1, 0);
    int active = 0;
    int32_t max_t = 0;
    for (int32_t b = 0; b < B; ++b) {
        tok0[b + 1] = tok0[b] + in.q_rows[b];
        if (in.q_rows[b] > 0) ++active;
        max_t = std::max(max_t, in.q_rows[b]);
    }
    R = tok0[B];
    const bool shared = active >= 2 && P > 0;
    // Two 128-row query tiles per unit when the row blocks are long enough to
    // fill them (they then share every K/V tile); one otherwise.
    const int64_t block_rows = static_cast<int64_t>(shared ? R : max_t) * G;
    nq = block_rows > kBM ? 2 : 1;
    tpt_tile = kBM / G;
    const int32_t tpt = tpt_tile * nq;  // tokens per unit
    for (int32_t h = 0; h < in.H_kv; ++h) {
        if (shared) {
            for (int32_t t = 0; t < R; t += tpt)
                ranges.push_back({h, 0, t, std::min(tpt, R - t), 0, P, kNoCausal, false});
        }
        for (int32_t b = 0; b < B; ++b) {
            const int32_t T = in.q_rows[b], S = S_eff[b];
            for (int32_t t = tok0[b]; t < tok0[b + 1]; t += tpt) {
                const int32_t n = std::min(tpt, tok0[b + 1] - t);
                const int32_t lo = shared ? P : 0;
                int32_t hi = P + S;
                int32_t pos_base = kNoCausal;
                if (in.causal) {
                    pos_base = P + S - T - tok0[b];
                    hi = std::min(hi, pos_base + t + n);  // last token's pos + 1
                }
                if (hi > lo) ranges.push_back({h, b, t, n, lo, hi, pos_base, !shared});
            }
        }
    }
}

}  // namespace

int build_plan(const PlanInput& in, Plan& plan) {
    plan = Plan();
    const int32_t B = in.num_branches;
    std::vector<Range> ranges;
    int32_t R = 0;
    make_ranges(in, ranges, R, plan.nq, plan.tpt);
    plan.R = R;
    if (R == 0) return 0;
    const int32_t G = in.H_q / in.H_kv;
    std::vector<int32_t> S_eff(B);
    const int32_t tail = in.prefix_len % in.page_size;
    const int32_t P = in.prefix_len - tail;
    for (int32_t b = 0; b < B; ++b) S_eff[b] = in.suffix_lens[b] + tail;

    // Chunk size from the cost model (or the forced split count).
    const int32_t max_cta = std::max(1, in.num_sms);
    const double ovh = plan.nq == 2 ? kUnitOverhead2 : kUnitOverhead1;
    Cand best, cand;
    if (in.force_splits > 0) {
        make_candidate(ranges, 0, in.force_splits, max_cta, ovh, best);
    } else {
        int64_t max_nkt = 1;
        for (const Range& r : ranges) max_nkt = std::max(max_nkt, cdiv(r.hi - r.lo, kBN));
        // keep the plan (and host planning time) bounded
        const int64_t max_units =
            std::max<int64_t>(16LL * max_cta, static_cast<int64_t>(ranges.size()));
        bool first = true;
        for (int64_t chunk : {0LL, 1024LL, 512LL, 384LL, 256LL, 192LL, 128LL, 96LL, 64LL, 48LL,
                              40LL, 32LL, 28LL, 24LL, 20LL, 18LL, 16LL, 14LL, 12LL, 10LL, 8LL, 6LL,
                              4LL, 3LL, 2LL}) {
            if (chunk > 0 && chunk >= max_nkt) continue;  // same as whole ranges
            if (chunk > 0) {
                int64_t n = 0;
                for (const Range& r : ranges) n += cdiv(cdiv(r.hi - r.lo, kBN), chunk);
                if (n > max_units) continue;
            }
            if (!first && candidate_cost_bound(ranges, chunk, max_cta, ovh) >= best.cost * 0.995)
                continue;  // could not replace the best
            make_candidate(ranges, chunk, 0, max_cta, ovh, cand);
            if (first || cand.cost < best.cost * 0.995) {
                std::swap(best, cand);
                first = false;
            }
        }
        // Tail cuts when every range is written directly (long prefill): the
        // cut pieces are then the only partials. With split ranges the
        // equal-chunk plans above already balance, and measured faster: the
        // cuts' remainders pile onto the CTAs that hold many short units.
        bool all_complete = true;
        for (const Range& r : ranges) all_complete = all_complete && r.complete;
        if (all_complete && in.tail_cuts) {
            make_lpt_cut(ranges, max_cta, ovh, cand);
            if (cand.cost < best.cost * 0.995) std::swap(best, cand);
        }
        // Exact balance scatters CTAs over different key offsets; use it only
        // when the whole KV fits in L2 (otherwise the lockstep waves of the
        // equal-chunk plan are what keeps a large shared prefix in L2).
        int64_t kv_tokens = P;
        for (int32_t b = 0; b < B; ++b) kv_tokens += S_eff[b];
        const int64_t kv_bytes = kv_tokens * in.H_kv * kHD * 2 * 2;
        if (kv_bytes <= (100LL << 20)) {
            make_streamk(ranges, max_cta, ovh, cand);
            if (cand.cost < best.cost * 0.97) std::swap(best, cand);
        }
    }

    // Group units by CTA (stable: each CTA keeps its assignment order) and
    // number the partials in that order.
    const int32_t n_cta = best.n_cta;
    plan.cta_first.assign(n_cta + 1, 0);
    for (int32_t c : best.cta_of) ++plan.cta_first[c + 1];
    for (int32_t c = 0; c < n_cta; ++c) plan.cta_first[c + 1] += plan.cta_first[c];
    std::vector<int32_t> fill(plan.cta_first.begin(), plan.cta_first.end() - 1);
    plan.units.resize(best.units.size());
    plan.unit_range.resize(best.units.size());
    for (size_t i = 0; i < best.units.size(); ++i) {
        const int32_t at = fill[best.cta_of[i]]++;
        plan.units[at] = best.units[i];
        plan.unit_range[at] = best.range_of[i];
    }
    plan.ranges = ranges;
    int32_t n_parts = 0;
    for (Unit& u : plan.units)
        if (u.part >= 0) u.part = n_parts++;
    plan.n_parts = n_parts;

    // Merge index: per (token, KV head), the partials covering it, in unit order,
    // as fixed-stride lists so a reader gets the count and the entries at once.
    if (n_parts > 0) {
        const size_t n_keys = static_cast<size_t>(R) * in.H_kv;
        plan.merge_cnt.assign(n_keys, 0);
        for (const Unit& u : plan.units)
            if (u.part >= 0)
                for (int32_t t = u.tok_begin; t < u.tok_begin + u.n_tok; ++t)
                    ++plan.merge_cnt[static_cast<size_t>(t) * in.H_kv + u.kv_head];
        int32_t stride = 1;
        for (int32_t c : plan.merge_cnt) stride = std::max(stride, c);
        plan.merge_stride = stride;
        plan.merge_ent.assign(n_keys * stride * 2, 0);
        std::vector<int32_t> fill_e(n_keys, 0);
        for (const Unit& u : plan.units)
            if (u.part >= 0)
                for (int32_t t = u.tok_begin; t < u.tok_begin + u.n_tok; ++t) {
                    const size_t key = static_cast<size_t>(t) * in.H_kv + u.kv_head;
                    const size_t e = key * stride + fill_e[key]++;
                    plan.merge_ent[2 * e] = u.part;
                    plan.merge_ent[2 * e + 1] = (t - u.tok_begin) * G;  // first row of t in u
                }
        // a (token, head) covered by a single direct unit has count 0; when
        // some are, the merge visits only the keys listed here
        bool sparse = false;
        for (int32_t c : plan.merge_cnt) sparse = sparse || c == 0;
        if (sparse)
            for (size_t k = 0; k < n_keys; ++k)
                if (plan.merge_cnt[k] > 0) plan.merge_keys.push_back(static_cast<int32_t>(k));
    }
    plan.need_merge = n_parts > 0;
    return 0;
}

bool patch_plan(const PlanInput& in, Plan& plan) {
    if (plan.units.empty() || plan.unit_range.size() != plan.units.size()) return false;
    std::vector<Range> ranges;
    int32_t R = 0, nq = 0, tpt = 0;
    make_ranges(in, ranges, R, nq, tpt);
    if (R != plan.R || nq != plan.nq || tpt != plan.tpt || ranges.size() != plan.ranges.size())
        return false;
    for (size_t i = 0; i < ranges.size(); ++i) {
        const Range& a = ranges[i];
        const Range& o = plan.ranges[i];
        if (a.kv_head != o.kv_head || a.branch != o.branch || a.tok_begin != o.tok_begin ||
            a.n_tok != o.n_tok || a.lo != o.lo || a.complete != o.complete ||
            (a.pos_base == kNoCausal) != (o.pos_base == kNoCausal) ||
            cdiv(a.hi - a.lo, kBN) != cdiv(o.hi - o.lo, kBN))
            return false;
    }
    for (size_t k = 0; k < plan.units.size(); ++k) {
        Unit& u = plan.units[k];
        const Range& o = plan.ranges[plan.unit_range[k]];
        const Range& a = ranges[plan.unit_range[k]];
        if (u.key_end == o.hi) u.key_end = a.hi;  // the range's last unit
        u.pos_base = a.pos_base;
    }
    plan.ranges = ranges;
    return true;
}

}  // namespace fanout
