// fanout_noalloc.cu -- fanout_attn_noalloc: the fan-out attention call without
// any device memory allocation by the library.
//
// Who needs it. fanout_attn keeps a grow-only workspace that it obtains with
// cudaMalloc the first time a problem needs more than it holds (and frees
// with cudaFree when it grows). Some callers cannot allow that: a serving
// engine that reserves nearly all device memory up front for its own pool and
// forbids any other allocation, code that must never trigger the device-wide
// synchronisation cudaFree implies, and callers running where allocation is
// not permitted at all. This entry point runs the same two kernels (split-KV
// attention, log-sum-exp merge) with their scratch -- the work plan and the
// split partials -- in one fixed array compiled into the library instead.
//
// The array. kScratchBytes (FANOUT_NOALLOC_SCRATCH_BYTES, 32 MiB) of device
// memory, a file-scope static __device__ array: every GPU that loads the
// library holds it until the process exits. A problem whose plan and
// partials need more is rejected with FANOUT_ENOMEM before anything runs.
// The host-side name of the array is only a stand-in, not a device address;
// the address is looked up with cudaGetSymbolAddress once per device, by the
// first call on that device (so make that first call before any stream
// capture). All calls share the array and it keeps the last call's contents:
// nothing in it is read before the same call writes it (the plan is uploaded
// every call, and every partial slot the merge reads is written by one unit
// of the same call), so no clearing is needed. Calls that overlap on the GPU
// (different streams, or a second call before the first finished) race on the
// array and corrupt each other's results.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/fanout.h"
#include "fanout_internal.h"

using namespace fanout;

namespace {

constexpr size_t kScratchBytes = FANOUT_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode_fn = nullptr;

size_t round256(size_t x) { return (x + 255) / 256 * 256; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int to_status(cudaError_t e) { return e == cudaSuccess ? FANOUT_OK : FANOUT_ECUDA; }

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
    if (!g_encode_fn) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return FANOUT_ECUDA;
        g_encode_fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = static_cast<uint8_t*>(g_scratch_addr[dev]);
    return FANOUT_OK;
}

int map_pool(CUtensorMap* m, const void* base, int64_t rows, int32_t page_size) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHD), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHD) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(page_size)};
    cuuint32_t es[2] = {1, 1};
    return g_encode_fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                       strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? FANOUT_OK
               : FANOUT_ECUDA;
}

int map_q(CUtensorMap* m, const void* q, int64_t R, int32_t H_q, int32_t G, int32_t tpt) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHD), static_cast<cuuint64_t>(H_q),
                          static_cast<cuuint64_t>(R)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHD) * 2,
                             static_cast<cuuint64_t>(H_q) * kHD * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(tpt)};
    cuuint32_t es[3] = {1, 1, 1};
    return g_encode_fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                       box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? FANOUT_OK
               : FANOUT_ECUDA;
}

}  // namespace

extern "C" FANOUT_API int fanout_attn_noalloc(
    const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
    int32_t prefix_len, const int32_t* suffix_lens, const int32_t* q_rows_per_branch,
    int32_t num_branches, int32_t max_pages_per_branch, int32_t num_pages, int32_t H_q,
    int32_t H_kv, int32_t d, int32_t page_size, float scale, int32_t causal, void* out,
    int32_t out_dtype, float* lse, fanout_stream_t stream_) {
    if (out_dtype != FANOUT_OUT_F32 && out_dtype != FANOUT_OUT_BF16) return FANOUT_EINVAL;
    if (!(scale == scale) || scale == 0.0f) return FANOUT_EINVAL;
    if (d != kHD) return FANOUT_EUNSUPPORTED;
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return FANOUT_ECUDA;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // Shape validation and the work plan come from the host-only planner entry.
    int32_t n_units = 0, n_slots = 0;
    int64_t R = 0;
    for (int32_t b = 0; b < num_branches && suffix_lens && q_rows_per_branch; ++b)
        R += q_rows_per_branch[b] > 0 ? q_rows_per_branch[b] : 0;
    std::vector<int32_t> tok(static_cast<size_t>(R) + 1, 0);
    int st = fanout_plan(suffix_lens, q_rows_per_branch, num_branches, prefix_len, H_q, H_kv,
                         page_size, causal, sms, nullptr, 0, &n_units, &n_slots, tok.data());
    if (st != FANOUT_OK) return st;
    if (R == 0) return FANOUT_OK;
    if (!q || !k_pages || !v_pages || !page_table || !out) return FANOUT_EINVAL;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out))
        return FANOUT_EINVAL;
    int64_t need_pages = 0;
    for (int32_t b = 0; b < num_branches; ++b)
        need_pages = std::max<int64_t>(
            need_pages,
            (static_cast<int64_t>(prefix_len) + suffix_lens[b] + page_size - 1) / page_size);
    if (num_pages <= 0 || max_pages_per_branch < need_pages) return FANOUT_EINVAL;

    // Scratch layout: units | per-token slot counts | (m, l) partials | O partials.
    const size_t off_units = 0;
    const size_t off_tok = round256(off_units + static_cast<size_t>(n_units) * sizeof(Unit));
    const size_t off_ml = round256(off_tok + static_cast<size_t>(R) * sizeof(int32_t));
    const size_t rows = static_cast<size_t>(R) * H_q;
    const size_t off_o = round256(off_ml + static_cast<size_t>(n_slots) * rows * sizeof(float2));
    const size_t total = round256(off_o + static_cast<size_t>(n_slots) * rows * kHD * sizeof(float));
    if (total > kScratchBytes) return FANOUT_ENOMEM;  // beyond the fixed array

    std::vector<int32_t> units(static_cast<size_t>(n_units) * 8);
    st = fanout_plan(suffix_lens, q_rows_per_branch, num_branches, prefix_len, H_q, H_kv,
                     page_size, causal, sms, units.data(), n_units, &n_units, &n_slots,
                     tok.data());
    if (st != FANOUT_OK) return st;

    uint8_t* scratch = nullptr;
    if ((st = scratch_for_device(dev, &scratch)) != FANOUT_OK) return st;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    ce = cudaMemcpyAsync(scratch + off_units, units.data(), units.size() * sizeof(int32_t),
                         cudaMemcpyHostToDevice, stream);
    if (ce == cudaSuccess)
        ce = cudaMemcpyAsync(scratch + off_tok, tok.data(), static_cast<size_t>(R) * sizeof(int32_t),
                             cudaMemcpyHostToDevice, stream);
    if (ce != cudaSuccess) return to_status(ce);

    const int32_t G = H_q / H_kv;
    const int32_t tpt = kBM / G;
    CUtensorMap tm_q, tm_k, tm_v;
    const int64_t pool_rows = static_cast<int64_t>(num_pages) * H_kv * page_size;
    if ((st = map_q(&tm_q, q, R, H_q, G, tpt)) != FANOUT_OK) return st;
    if ((st = map_pool(&tm_k, k_pages, pool_rows, page_size)) != FANOUT_OK) return st;
    if ((st = map_pool(&tm_v, v_pages, pool_rows, page_size)) != FANOUT_OK) return st;
    int32_t* err = nullptr;
    if ((ce = err_word_ptr(&err)) != cudaSuccess) return to_status(ce);

    SplitParams p;
    p.page_table = page_table;
    p.units = reinterpret_cast<const Unit*>(scratch + off_units);
    p.part_o = reinterpret_cast<float*>(scratch + off_o);
    p.part_ml = reinterpret_cast<float2*>(scratch + off_ml);
    p.out = out;
    p.lse = lse;
    p.err = err;
    p.n_units = n_units;
    p.max_pages = max_pages_per_branch;
    p.R = static_cast<int32_t>(R);
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.G = G;
    p.page_size = page_size;
    p.tpt = tpt;
    p.out_bf16 = out_dtype == FANOUT_OUT_BF16;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.wait_limit_ns = 1000000000ull;
    if ((ce = launch_split_attn(p, tm_q, tm_k, tm_v, n_units, stream)) != cudaSuccess)
        return to_status(ce);
    if (n_slots > 0) {
        ce = launch_lse_merge(p.part_o, p.part_ml,
                              reinterpret_cast<const int32_t*>(scratch + off_tok), n_slots,
                              static_cast<int64_t>(rows), H_q, out, p.out_bf16, lse, stream);
        if (ce != cudaSuccess) return to_status(ce);
    }
    return FANOUT_OK;
}
