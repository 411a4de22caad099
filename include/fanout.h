/*
 * fanout.h -- C ABI of the shared-prefix fan-out attention library
 * (libfanout.so, CUDA, sm_103a / GB300).
 *
 * The problem (from "AHBM Agentic Runtime Architecture"):
 *   section 3.1 "Fan-out context structure": a parent context is forked into
 *     branches by page table; every branch table is [shared prefix pages] +
 *     [private suffix pages]; shared pages are referenced, never copied.
 *   section 3.2 "Sub-agent query batching": the new query rows of all branches
 *     are concatenated along the row dimension (Q_combined) and run as one
 *     attention; each row stays independent.
 *   sections 3.3-3.5: every row's keys are split into sequence shards; each
 *     shard yields an online-softmax partial (m, l, o); partials of the same
 *     row are merged with the log-sum-exp rule.
 * and from "ADR-0060: AHBM GQA Fused Attention kernel (Llama3-70B)":
 *   TL;DR and section 5.2: per KV head, the G = H_q / H_kv query heads that
 *     share it are folded into the matrix M dimension (no K/V broadcast);
 *   section 3: FlashAttention tile sweep with online softmax;
 *   section 4: FlashDecoding split-KV partials merged by log-sum-exp;
 *   section 5.4: causal tile classification (all past / all future / partial);
 *   section 0.5.3: softmax_scale (1/sqrt(d) in the pages' use).
 *
 * Conventions for every call:
 *   - Tensors are plain pointers; the caller allocates and owns them. "dev"
 *     marks device memory of the current CUDA device, "host" host memory.
 *   - bf16 is IEEE bfloat16 stored in 16 bits.
 *   - A call returns FANOUT_OK or an error code; nothing is printed and no
 *     exception crosses the ABI. Argument errors are found on the host before
 *     any launch. Errors inside a kernel (a bounded wait that ran out) are
 *     recorded in a device word and reported by fanout_last_error().
 *   - Calls are asynchronous with respect to the host unless stated.
 */
#ifndef FANOUT_H
#define FANOUT_H

#include <stdint.h>

#if defined(__GNUC__)
#define FANOUT_API __attribute__((visibility("default")))
#else
#define FANOUT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *fanout_stream_t;
struct CUevent_st;
typedef struct CUevent_st *fanout_event_t;

enum fanout_status {
    FANOUT_OK = 0,
    FANOUT_EINVAL = 1,        /* invalid argument (null pointer, bad size, bad page id) */
    FANOUT_EUNSUPPORTED = 2,  /* valid problem outside what this library supports */
    FANOUT_ECUDA = 3,         /* a CUDA runtime/driver call failed */
    FANOUT_ENOMEM = 4,        /* workspace allocation failed */
    FANOUT_ETIMEOUT = 5       /* a bounded device-side wait ran out */
};

enum fanout_out_dtype { FANOUT_OUT_F32 = 0, FANOUT_OUT_BF16 = 1 };

/*
 * fanout_fork -- build branch page tables (host only, no device work).
 * "AHBM Agentic Runtime Architecture", section 3.1 "Fan-out context structure".
 *
 *   prefix_pages   host int32 [n_prefix_pages]: physical ids of the shared
 *                  prefix pages, in logical order.
 *   num_branches   B >= 0.
 *   suffix_lens    host int32 [B]: private suffix length of each branch, tokens.
 *   page_size      tokens per page (> 0).
 *   free_pages     host int32 [n_free]: physical ids available for private
 *                  pages; branch 0 takes the first ceil(S_0/page_size), branch
 *                  1 the next, and so on.
 *   page_table     host int32 [B][max_pages_per_branch], written: row b =
 *                  prefix ids, then branch b's private ids, then -1.
 * Returns FANOUT_EINVAL on a null pointer, a negative size, a free list too
 * short, or a row too narrow. On error page_table is left unspecified.
 */
FANOUT_API int fanout_fork(const int32_t *prefix_pages, int32_t n_prefix_pages, int32_t num_branches,
                const int32_t *suffix_lens, int32_t page_size, const int32_t *free_pages,
                int32_t n_free, int32_t *page_table, int32_t max_pages_per_branch);

/*
 * fanout_fork_cow -- fork when the prefix ends inside a page (host only).
 * "AHBM Agentic Runtime Architecture" section 3.1: shared pages are
 * referenced, never copied -- but a partially filled last prefix page cannot
 * be shared by branches that will each append after it, so every branch gets
 * its own copy of that one page (copy-on-write at fork time).
 *   prefix_pages  host int32 [ceil(prefix_len / page_size)] physical ids.
 *   page_table    host int32 [B][max_pages_per_branch], written: the whole
 *                 prefix pages (shared), then the branch's own pages -- first
 *                 the copy of the partial prefix page, if any, then its suffix
 *                 pages -- taken from free_pages in order, branch 0 first;
 *                 then -1.
 *   cow_pairs     host int32 [B][2] or NULL: {source page, branch's copy} per
 *                 branch when the prefix ends inside a page (unwritten
 *                 otherwise); copy them with fanout_copy_pages (rows =
 *                 prefix_len % page_size) before appending.
 *   n_used        out (may be NULL): free pages consumed.
 * With prefix_len a multiple of page_size this is fanout_fork. Returns
 * FANOUT_EINVAL (table untouched) when the free list or a row is too short.
 */
FANOUT_API int fanout_fork_cow(const int32_t *prefix_pages, int32_t prefix_len,
                int32_t num_branches, const int32_t *suffix_lens, int32_t page_size,
                const int32_t *free_pages, int32_t n_free, int32_t *page_table,
                int32_t max_pages_per_branch, int32_t *cow_pairs, int32_t *n_used);

/*
 * fanout_copy_pages -- copy token slots [0, rows) of page pairs[i][0] to page
 * pairs[i][1], every KV head, in both pools (device). The copy-on-write step
 * of fanout_fork_cow.
 *   pairs   dev int32 [n_pairs][2]; pools dev bf16 [num_pages][H_kv][page][d].
 * A page id outside [0, num_pages) is never used: the pair is skipped and
 * fanout_last_error() reports FANOUT_EINVAL.
 */
FANOUT_API int fanout_copy_pages(void *k_pages, void *v_pages, const int32_t *pairs,
                int32_t n_pairs, int32_t rows, int32_t num_pages, int32_t H_kv, int32_t d,
                int32_t page_size, fanout_stream_t stream);

/*
 * fanout_extend -- grow branch page tables for new tokens (host only).
 * "AHBM Agentic Runtime Architecture" section 3.1 (private suffix pages per
 * branch); ADR-0060 section 0.5.1 precondition P3 (the cache grows before
 * attention). Branch b's context grows from prefix_len + suffix_lens[b] to
 * prefix_len + suffix_lens[b] + add_lens[b] tokens; table entry i holds
 * logical positions [i * page_size, (i + 1) * page_size). The entries it now
 * needs beyond its current ceil((prefix_len + suffix_lens[b]) / page_size) are
 * taken from free_pages in order (branch 0 first).
 *   page_table   host int32 [B][max_pages_per_branch], updated in place.
 *   prefix_len   any value >= 0; a prefix ending inside a page must have been
 *                forked with fanout_fork_cow (its last page is then private).
 *   n_used       out (may be NULL): free pages consumed.
 * Returns FANOUT_EINVAL (table untouched) when a row is too narrow or the
 * free list too short.
 */
FANOUT_API int fanout_extend(int32_t *page_table, int32_t num_branches,
                int32_t max_pages_per_branch, int32_t prefix_len, const int32_t *suffix_lens,
                const int32_t *add_lens, int32_t page_size, const int32_t *free_pages,
                int32_t n_free, int32_t *n_used);

/*
 * fanout_kv_append -- write new K/V rows into the paged pools (device).
 * ADR-0060 section 0.5.1 precondition P3: the new tokens' post-RoPE K and V
 * are in the cache before attention runs. Row r of k_new / v_new is token t of
 * branch b (rows grouped by branch, branch b has add_lens[b] rows) and is
 * written, for every KV head h, to
 *   pool[page_table[b][pos / page_size]][h][pos % page_size][0..d-1],
 *   pos = prefix_len + suffix_lens[b] + t   (suffix_lens: BEFORE the append).
 *   k_new, v_new      dev bf16 [R][H_kv][d], 16-byte aligned, d % 8 == 0.
 *   k_pages, v_pages  dev bf16 [num_pages][H_kv][page_size][d], written.
 *   page_table        dev int32 [B][max_pages_per_branch] (grown already, e.g.
 *                     by fanout_extend then copied to the device).
 * num_branches <= 1024 and (sum of add_lens) * H_kv <= 2^31, else
 * FANOUT_EUNSUPPORTED; d % 8 == 0 and d <= 1024, else FANOUT_EUNSUPPORTED. An
 * out-of-range page id is never written through: the row is skipped and
 * fanout_last_error() reports FANOUT_EINVAL.
 */
FANOUT_API int fanout_kv_append(const void *k_new, const void *v_new, void *k_pages,
                void *v_pages, const int32_t *page_table, int32_t prefix_len,
                const int32_t *suffix_lens, const int32_t *add_lens, int32_t num_branches,
                int32_t max_pages_per_branch, int32_t num_pages, int32_t H_kv, int32_t d,
                int32_t page_size, fanout_stream_t stream);

/*
 * fanout_attn -- batched shared-prefix fan-out attention.
 * "AHBM Agentic Runtime Architecture" sections 3.2-3.5; "ADR-0060" TL;DR,
 * sections 3, 4, 5.2 and 5.4.
 *
 * Rows. R = sum_b q_rows_per_branch[b] query tokens, grouped by branch
 * (branch 0's T_0 tokens first). Token t of branch b sits at absolute position
 *   pos = prefix_len + suffix_lens[b] - q_rows_per_branch[b] + t,
 * i.e. the new tokens are the tail of the branch's private suffix, and their
 * K/V are already in the pool (the kernel is a pure read of the cache).
 * Keys. Branch b sees keys 0 .. prefix_len + suffix_lens[b] - 1 of its own
 * logical sequence; key j lives at
 *   k_pages[page_table[b][j / page_size]][h_kv][j % page_size][0..d-1].
 * With causal != 0 key j is visible to the token at pos iff j <= pos.
 * Query head h uses KV head h / (H_q / H_kv).
 *
 *   q                dev bf16 [R][H_q][d] (post-RoPE queries).
 *   k_pages, v_pages dev bf16 [num_pages][H_kv][page_size][d]. 16-byte aligned.
 *   page_table       dev int32 [num_branches][max_pages_per_branch]; every
 *                    entry a branch reads must be in [0, num_pages).
 *   prefix_len       tokens (>= 0). When it is not a multiple of page_size,
 *                    the whole pages are read as the shared prefix and the
 *                    rest of the last prefix page through each branch's own
 *                    table entry (a private copy after fanout_fork_cow).
 *   suffix_lens      HOST int32 [num_branches] (>= 0).
 *   q_rows_per_branch HOST int32 [num_branches] (>= 0); with causal != 0 each
 *                    must be <= suffix_lens[b].
 *   H_q, H_kv        H_q % H_kv == 0, G = H_q / H_kv <= 128.
 *   d                head dimension; the library supports d == 128.
 *   page_size        one of 16, 32, 64, 128.
 *   scale            softmax scale applied to q.k, finite and > 0 (the pages
 *                    use 1/sqrt(d)).
 *   out              dev [R][H_q][d], fp32 or bf16 per out_dtype:
 *                    out = softmax(scale q K^T) V, normalised.
 *   lse              dev fp32 [R][H_q] or NULL: natural-log log-sum-exp of the
 *                    scaled visible scores, m + ln(l).
 *   stream           stream the work is ordered on.
 * The shared prefix: entries [0, prefix_len / page_size) (whole pages) of
 * every row must be the same page ids; shared-prefix work reads them through
 * row 0. Host-side validation reads only host arrays; page-table entries are read by
 * the kernel (set option FANOUT_OPT_VALIDATE_TABLE to check them on the host
 * with a device-to-host copy first). R == 0 is a no-op returning FANOUT_OK.
 * Limits: prefix_len + suffix_lens[b] <= 2^29 keys and R * H_q <= 2^24
 * (FANOUT_EUNSUPPORTED otherwise); max_pages_per_branch must cover
 * ceil((prefix_len + suffix_lens[b]) / page_size) entries for every branch,
 * and a branch with query rows must have at least one key (FANOUT_EINVAL).
 * The library keeps a grow-only device workspace per (device, stream) for
 * split partials and the work plan; it is freed by fanout_release().
 */
FANOUT_API int fanout_attn(const void *q, const void *k_pages, const void *v_pages,
                const int32_t *page_table, int32_t prefix_len, const int32_t *suffix_lens,
                const int32_t *q_rows_per_branch, int32_t num_branches,
                int32_t max_pages_per_branch, int32_t num_pages, int32_t H_q, int32_t H_kv,
                int32_t d, int32_t page_size, float scale, int32_t causal, void *out,
                int32_t out_dtype, float *lse, fanout_stream_t stream);

/*
 * fanout_lse_merge -- the log-sum-exp merge of split partials on its own
 * (ADR-0060 section 4 "Reduction"; "AHBM Agentic Runtime Architecture"
 * section 3.4). For every output n (n < n_out) fold parts p = 0 .. n_parts-1
 * in ascending order:
 *   m_p   = part_ml[p][n].x  (running max, base-2 domain: max of scale*log2(e)*s)
 *   l_p   = part_ml[p][n].y  (sum of 2^(x - m_p))
 *   o_p   = part_o[p][n][0..d-1] (unnormalised)
 * out[n] = sum_p 2^(m_p - M) o_p / L,  L = sum_p 2^(m_p - M) l_p, M = max_p m_p;
 * lse[n] = (M + log2 L) * ln 2. A part with l_p == 0 (no visible key) weighs 0.
 *   part_o dev fp32 [n_parts][n_out][d]; part_ml dev fp32 [n_parts][n_out][2];
 *   out dev [n_out][d] (fp32/bf16), lse dev fp32 [n_out] or NULL.
 * This is the merge step fanout_attn runs internally, exposed for testing.
 */
FANOUT_API int fanout_lse_merge(const float *part_o, const float *part_ml, int32_t n_parts, int64_t n_out,
                     int32_t d, void *out, int32_t out_dtype, float *lse, fanout_stream_t stream);

/* Synchronises `stream`, then returns and clears the device error word of the
 * current device: FANOUT_OK, FANOUT_ETIMEOUT (a bounded wait ran out),
 * FANOUT_EINVAL (fanout_kv_append met a bad page id), or FANOUT_ECUDA when the
 * stream itself reports a CUDA error. */
FANOUT_API int fanout_last_error(fanout_stream_t stream);

/* fanout_last_error, also reporting where a device-side wait gave up: `site`
 * (an internal wait-site number of the kernel) and `block` (CTA index); both
 * may be NULL and are 0 when no error was recorded. */
FANOUT_API int fanout_last_error_detail(fanout_stream_t stream, int32_t *site, int32_t *block);

/* Static text for a status code (never NULL). */
FANOUT_API const char *fanout_strerror(int code);

/* Tuning / diagnostics options (process-wide; set before the calls they affect). */
enum fanout_option {
    FANOUT_OPT_SPLITS = 1,          /* >0: cut every key range into this many chunks; 0 = cost model */
    FANOUT_OPT_VALIDATE_TABLE = 2,  /* 1: check page-table entries on the host each call */
    FANOUT_OPT_WAIT_LIMIT_NS = 3,   /* bound of every device-side wait (default 1e9 ns) */
    FANOUT_OPT_NUM_SMS = 4,         /* >0: plan for this many SMs instead of the device's */
    FANOUT_OPT_FUSED_MERGE = 5      /* 0 (default): the log-sum-exp merge is a separate kernel,
                                       a programmatic dependent of the attention kernel; 1: it
                                       runs inside the attention kernel (cooperative launch)
                                       when every CTA fits on the device at once */
};
FANOUT_API int fanout_set_option(int32_t option, int64_t value);

/* Record `before` / `after` on the call's stream around the split-KV attention
 * kernel of every following fanout_attn call (NULL, NULL turns it off). Used to
 * time that kernel alone (it includes the merge when the merge is fused, see
 * FANOUT_OPT_FUSED_MERGE; a separate merge kernel falls outside the events). */
FANOUT_API int fanout_set_profile_events(fanout_event_t before, fanout_event_t after);

/* Host-side description of the work plan fanout_attn would run for a problem
 * (no device access), planned for `num_sms` persistent CTAs (<= 0: 152, a GB300's SM count).
 * Writes up to `cap` unit records of 8 int32 each, grouped by CTA:
 *   {kv_head, branch, tok_begin, n_tok, key_begin, key_end, pos_base, part}
 * (the query rows of n_tok tokens x the G heads of kv_head against keys
 * [key_begin, key_end) of the branch; token r is at position pos_base + r for
 * causal masking; part >= 0 is the unit's partial block, -1 a direct write),
 * and up to `cta_cap` entries of cta_first (CTA c runs units
 * [cta_first[c], cta_first[c+1])). Any output pointer may be NULL with a zero
 * capacity. Returns FANOUT_OK or an error code with the same validation as
 * fanout_attn. */
FANOUT_API int fanout_plan(const int32_t *suffix_lens, const int32_t *q_rows_per_branch,
                int32_t num_branches, int32_t prefix_len, int32_t H_q, int32_t H_kv,
                int32_t page_size, int32_t causal, int32_t num_sms, int32_t *units,
                int32_t cap, int32_t *n_units, int32_t *cta_first, int32_t cta_cap,
                int32_t *n_ctas, int32_t *n_parts);

/* The plan fanout_attn runs for a call whose previous call on the same stream
 * had the same arguments except the suffix lengths, prev_suffix_lens (a decode
 * step: each branch's suffix grew by the tokens just appended). When every key
 * range keeps its number of 128-key tiles, the previous plan is kept -- same
 * chunks, CTA assignment, partial blocks and merge index -- with each range's
 * last unit ending at the new range end and the new causal positions, and
 * *reused = 1 (fanout_attn then re-uploads only the unit table instead of
 * planning again); otherwise a new plan, *reused = 0. Outputs and errors as
 * fanout_plan; `reused` may be NULL. Host only. */
FANOUT_API int fanout_plan_step(const int32_t *prev_suffix_lens, const int32_t *suffix_lens,
                const int32_t *q_rows_per_branch, int32_t num_branches, int32_t prefix_len,
                int32_t H_q, int32_t H_kv, int32_t page_size, int32_t causal, int32_t num_sms,
                int32_t *units, int32_t cap, int32_t *n_units, int32_t *cta_first,
                int32_t cta_cap, int32_t *n_ctas, int32_t *n_parts, int32_t *reused);

/* Launches one tiny kernel whose single thread waits on a barrier nothing ever
 * completes, bounded by `limit_ns`; returns FANOUT_ETIMEOUT when the bound
 * fires and the kernel came back (the context stays usable), FANOUT_OK never
 * (a completed wait would be a bug). Tests the bounded-wait path. */
FANOUT_API int fanout_selftest_wait_timeout(int64_t limit_ns, fanout_stream_t stream);

/*
 * fanout_read_floor -- a calibration read; the pages have no counterpart.
 * One launch streams `bytes` of device memory at `buf` once from HBM with
 * plain 16-byte loads (four 512-thread CTAs per SM) and xors every 32-bit word
 * of it into *xor_out. Timed like a fanout_attn call (after an L2 flush, CUDA
 * events on `stream`), it is the shortest time one kernel that reads that many
 * bytes takes on this device, launch and ramp included: the floor under an
 * HBM-bound call, which a roofline at the steady copy bandwidth leaves out.
 *   buf      dev, 16-byte aligned, read only.
 *   bytes    > 0, a multiple of 16.
 *   xor_out  dev uint32, 4-byte aligned, updated in place (*xor_out ^= xor of
 *            the buffer's words); the caller sets it beforehand.
 * FANOUT_EINVAL, with nothing launched, for a null pointer or a size or
 * alignment outside these rules; FANOUT_ECUDA if the launch fails.
 * Asynchronous on `stream`.
 */
FANOUT_API int fanout_read_floor(const void *buf, int64_t bytes, uint32_t *xor_out,
                                 fanout_stream_t stream);

/*
 * fanout_attn_noalloc -- fanout_attn that allocates no device memory.
 * The pages have no counterpart: this entry exists for callers of this
 * library that must not allocate device memory during a call -- a serving
 * engine that has reserved the device's memory for its own pool, code that
 * cannot afford the device-wide synchronisation of cudaFree, or code running
 * where allocation is not allowed. fanout_attn obtains its workspace with
 * cudaMalloc; this entry instead keeps the work plan and the split-KV partials
 * in one fixed array of FANOUT_NOALLOC_SCRATCH_BYTES compiled into the library
 * (every GPU that loads the library holds it until the process exits).
 * Arguments, layouts and results are those of fanout_attn (same kernels, same
 * plan, so the same output); the caller still allocates q, the pools, the
 * page table, out and lse. Differences:
 *   - FANOUT_ENOMEM, before anything runs, when the problem's plan plus
 *     partials need more than FANOUT_NOALLOC_SCRATCH_BYTES;
 *   - the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture;
 *   - FANOUT_EUNSUPPORTED, with nothing done, when `stream` is capturing: each
 *     call copies its plan into the array from host memory that lives only
 *     for the call;
 *   - all calls share the one array, and it keeps the last call's contents.
 *     Nothing in it needs clearing (each call writes all it reads), but calls
 *     that overlap on the GPU (two streams, or a new call before the previous
 *     one finished) race on it and corrupt each other's results;
 *   - FANOUT_OPT_WAIT_LIMIT_NS and FANOUT_OPT_NUM_SMS do not apply (1 s bound,
 *     the device's own SM count); profile events are not recorded;
 *   - the last plan is kept per device (not per stream), and reused or
 *     carried over to new suffix lengths as fanout_plan_step describes.
 */
#define FANOUT_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
FANOUT_API int fanout_attn_noalloc(const void *q, const void *k_pages, const void *v_pages,
                const int32_t *page_table, int32_t prefix_len, const int32_t *suffix_lens,
                const int32_t *q_rows_per_branch, int32_t num_branches,
                int32_t max_pages_per_branch, int32_t num_pages, int32_t H_q, int32_t H_kv,
                int32_t d, int32_t page_size, float scale, int32_t causal, void *out,
                int32_t out_dtype, float *lse, fanout_stream_t stream);

/* Frees the workspace buffers and cached plans of every device and stream
 * (synchronising each device first); the next call on a stream allocates and
 * plans again. Safe while other threads call fanout_attn: a call in flight
 * finishes first (its workspace lock is taken before the buffer is freed). */
FANOUT_API int fanout_release(void);

/* Library version, "major.minor.patch". */
FANOUT_API const char *fanout_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FANOUT_H */
