// fanout_noalloc.cu -- fanout_attn_noalloc: the fan-out attention call without
// any device memory allocation by the library.
//
// Who needs it. fanout_attn keeps a grow-only workspace that it obtains with
// cudaMalloc the first time a problem needs more than it holds (and frees
// with cudaFree when it grows). Some callers cannot allow that: a serving
// engine that reserves nearly all device memory up front for its own pool and
// forbids any other allocation, code that must never trigger the device-wide
// synchronisation cudaFree implies, and callers running where allocation is
// not permitted at all. This entry point runs the same kernels (split-KV
// attention with its log-sum-exp merge) with their scratch -- the work plan and the
// split partials -- in one fixed array compiled into the library instead.
//
// The array. kScratchBytes (FANOUT_NOALLOC_SCRATCH_BYTES, 32 MiB) of device
// memory, a file-scope static __device__ array: every GPU that loads the
// library holds it until the process exits. A problem whose plan and
// partials need more is rejected with FANOUT_ENOMEM before anything runs.
// The host-side name of the array is only a stand-in, not a device address;
// the address is looked up with cudaGetSymbolAddress once per device, by the
// first call on that device (so make that first call before any stream
// capture). A call on a stream that is capturing is refused
// (FANOUT_EUNSUPPORTED, nothing done): the plan is copied from host memory
// that lives only for the call. All calls share the array and it keeps the last call's contents:
// nothing in it is read before the same call writes it (the plan is uploaded
// every call, and every partial slot the merge reads is written by one unit
// of the same call) except the fused merge's per-CTA flags at its start,
// which only ever hold 0 (the array's initial value) or an earlier call's
// epoch, never the current one -- so no clearing is needed. Calls that overlap on the GPU
// (different streams, or a second call before the first finished) race on the
// array and corrupt each other's results.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/fanout.h"
#include "plan.h"

using namespace fanout;

namespace {

constexpr size_t kScratchBytes = FANOUT_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};
uint32_t g_epoch[kMaxDevices] = {};  // fused-merge flag value of the last call per device

// The last plan per device (host memory; guarded by g_setup_mu), kept for a
// call with the same problem, or carried over to one whose suffix lengths
// alone changed (patch_plan), as fanout_attn does per stream.
struct PlanCache {
    std::vector<int32_t> key;
    Plan plan;
    bool ready = false;
};
PlanCache g_plan_cache[kMaxDevices];

// Once per device, with that device current: the device address of the array.
int scratch_for_device(int dev, uint8_t** out) {
    if (dev < 0 || dev >= kMaxDevices) return FANOUT_EUNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) return FANOUT_ECUDA;
        g_scratch_addr[dev] = p;
    }
    *out = static_cast<uint8_t*>(g_scratch_addr[dev]);
    return FANOUT_OK;
}

}  // namespace

extern "C" FANOUT_API int fanout_attn_noalloc(
    const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
    int32_t prefix_len, const int32_t* suffix_lens, const int32_t* q_rows_per_branch,
    int32_t num_branches, int32_t max_pages_per_branch, int32_t num_pages, int32_t H_q,
    int32_t H_kv, int32_t d, int32_t page_size, float scale, int32_t causal, void* out,
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
    // The plan is copied to the array from host memory that lives only for this
    // call; a captured copy would read it after it is gone. Refused, nothing done.
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &capture) != cudaSuccess) return FANOUT_ECUDA;
    if (capture != cudaStreamCaptureStatusNone) return FANOUT_EUNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FANOUT_ECUDA;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // The same plan fanout_attn builds (host memory only): the device's last
    // plan when the problem is the same or only its suffix lengths moved
    // within their tiles, else a new one.
    if (dev < 0 || dev >= kMaxDevices) return FANOUT_EUNSUPPORTED;
    PlanInput in{suffix_lens, q_rows_per_branch, num_branches, prefix_len, H_q, H_kv,
                 page_size, causal, sms > 0 ? sms : 1, current_force_splits()};
    std::vector<int32_t> key = {prefix_len, num_branches, H_q, H_kv, page_size, causal, in.num_sms,
                                in.force_splits};
    const size_t fixed = key.size();
    key.insert(key.end(), suffix_lens, suffix_lens + num_branches);
    key.insert(key.end(), q_rows_per_branch, q_rows_per_branch + num_branches);
    Plan plan;
    bool have = false;
    {
        std::lock_guard<std::mutex> lk(g_setup_mu);
        PlanCache& c = g_plan_cache[dev];
        if (c.ready && c.key == key) {
            plan = c.plan;
            have = true;
        } else if (c.ready && c.key.size() == key.size() &&
                   std::equal(key.begin(), key.begin() + fixed, c.key.begin()) &&
                   std::equal(key.begin() + fixed + num_branches, key.end(),
                              c.key.begin() + fixed + num_branches)) {
            plan = c.plan;
            have = patch_plan(in, plan);
        }
    }
    Layout L;
    if (have) {
        L = plan_layout(plan);
    } else {
        if ((st = build_plan(in, plan)) != FANOUT_OK) return st;
        L = plan_layout(plan);
        if (L.total > kScratchBytes) {
            // without the tail cuts a long prefill has no partials at all
            in.tail_cuts = 0;
            if ((st = build_plan(in, plan)) != FANOUT_OK) return st;
            L = plan_layout(plan);
        }
    }
    if (L.total > kScratchBytes) return FANOUT_ENOMEM;  // beyond the fixed array
    {
        std::lock_guard<std::mutex> lk(g_setup_mu);
        PlanCache& c = g_plan_cache[dev];
        c.key = key;
        c.plan = plan;
        c.ready = true;
    }

    uint8_t* scratch = nullptr;
    if ((st = scratch_for_device(dev, &scratch)) != FANOUT_OK) return st;
    if (upload_plan(plan, L, scratch, stream) != cudaSuccess) return FANOUT_ECUDA;
    uint32_t epoch;
    {
        std::lock_guard<std::mutex> lk(g_setup_mu);
        if (++g_epoch[dev] == 0) g_epoch[dev] = 1;
        epoch = g_epoch[dev];
    }
    CallArgs a{q, k_pages, v_pages, page_table, max_pages_per_branch, num_pages, H_q, H_kv,
               page_size, out_dtype == FANOUT_OUT_BF16, scale, out, lse, R, 1000000000ull,
               current_fused_merge(), epoch};
    return launch_plan(a, plan, L, scratch, stream, nullptr, nullptr);
}
