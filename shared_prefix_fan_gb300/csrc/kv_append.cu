// kv_append.cu -- the paged KV-cache append that precedes attention.
//
// ADR-0060 section 0.5.1 (precondition P3): the new step's K (post-RoPE) and
// V rows are written into the cache before the attention kernel runs, which
// is then a pure read. With fan-out ("AHBM Agentic Runtime Architecture"
// section 3.1) every branch appends to its own private suffix pages; the
// shared prefix pages are never written.
//
// Row r of k_new / v_new is token t of branch b (rows grouped by branch, as
// the query rows of fanout_attn) and goes to logical position
// prefix_len + suffix_len_b + t of branch b, i.e. to page
// page_table[b][pos / page], slot pos % page, for every KV head.
//
// Also the copy-on-write of a partially filled shared page (fork with a
// prefix that ends inside a page): each branch gets its own copy.
//
// HBM-bound scatter: one warp per (row, KV head) moves the K row with lanes
// 0..15 and the V row with lanes 16..31 in 16-byte pieces. The per-branch
// offsets travel in the kernel parameters, so the call needs no workspace.
#include <cuda_runtime.h>

#include <cstdint>

#include "fanout_internal.h"

namespace fanout {
namespace {

__global__ void __launch_bounds__(256)
    kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                     uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                     const int32_t* __restrict__ page_table, const __grid_constant__ AppendParams p,
                     int32_t* err) {
    const int lane = threadIdx.x & 31;
    const int64_t n_items = static_cast<int64_t>(p.R) * p.H_kv;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int chunks = p.d / 8;  // 16-byte pieces per row
    // Index arithmetic in 32 bits, and shifts for power-of-two head counts and
    // page sizes (warp-uniform branches): 64-bit divisions per item made this
    // scatter bound by instruction issue, not by memory.
    const bool hkv_pow2 = (p.H_kv & (p.H_kv - 1)) == 0;
    const int hkv_shift = __ffs(p.H_kv) - 1;
    const bool ps_pow2 = (p.page_size & (p.page_size - 1)) == 0;
    const int ps_shift = __ffs(p.page_size) - 1;
    for (int64_t item = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         item < n_items; item += warps) {
        const int32_t it = static_cast<int32_t>(item);  // R * H_kv <= 2^31 (host check)
        int32_t r, h;
        if (hkv_pow2) {
            r = it >> hkv_shift;
            h = it & (p.H_kv - 1);
        } else {
            r = it / p.H_kv;
            h = it - r * p.H_kv;
        }
        // branch of row r: largest b with row_off[b] <= r (binary search)
        int lo = 0, hi = p.num_branches - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.row_off[mid] <= r) lo = mid; else hi = mid - 1;
        }
        const int b = lo;
        const int64_t pos = static_cast<int64_t>(p.prefix_len) + p.suffix_len[b] + (r - p.row_off[b]);
        int64_t pidx, slot;
        if (ps_pow2) {
            pidx = pos >> ps_shift;
            slot = pos & (p.page_size - 1);
        } else {
            pidx = pos / p.page_size;
            slot = pos - pidx * p.page_size;
        }
        const int32_t page = page_table[static_cast<int64_t>(b) * p.max_pages + pidx];
        if (page < 0 || page >= p.num_pages) {  // never write through a bad page id
            if (lane == 0) atomicCAS(err, 0, 1);
            continue;
        }
        const int64_t dst = ((static_cast<int64_t>(page) * p.H_kv + h) * p.page_size + slot) *
                            chunks;
        const int64_t src = (static_cast<int64_t>(r) * p.H_kv + h) * chunks;
        const bool is_v = lane >= 16;
        const uint4* s = is_v ? v_new : k_new;
        uint4* d = is_v ? v_pool : k_pool;
        for (int c = lane & 15; c < chunks; c += 16) d[dst + c] = s[src + c];
    }
}

// Copy-on-write of partially filled pages: for every pair i, token slots
// [0, rows) of page src[i] -> page dst[i], all KV heads, K and V.
__global__ void __launch_bounds__(256)
    copy_pages_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                      const int2* __restrict__ pairs, int32_t n_pairs, int32_t rows, int32_t H_kv,
                      int32_t d, int32_t page_size, int32_t num_pages, int32_t* err) {
    const int lane = threadIdx.x & 31;
    const int chunks = d / 8;
    const int64_t n_items = static_cast<int64_t>(n_pairs) * H_kv * rows;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t item = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         item < n_items; item += warps) {
        const int32_t slot = static_cast<int32_t>(item % rows);
        const int32_t h = static_cast<int32_t>((item / rows) % H_kv);
        const int2 pr = pairs[item / (static_cast<int64_t>(rows) * H_kv)];
        if (pr.x < 0 || pr.x >= num_pages || pr.y < 0 || pr.y >= num_pages) {
            if (lane == 0) atomicCAS(err, 0, 1);
            continue;
        }
        const int64_t src = ((static_cast<int64_t>(pr.x) * H_kv + h) * page_size + slot) * chunks;
        const int64_t dst = ((static_cast<int64_t>(pr.y) * H_kv + h) * page_size + slot) * chunks;
        uint4* pool = lane >= 16 ? v_pool : k_pool;
        for (int c = lane & 15; c < chunks; c += 16) pool[dst + c] = pool[src + c];
    }
}

}  // namespace

cudaError_t launch_copy_pages(void* k_pool, void* v_pool, const int32_t* pairs, int32_t n_pairs,
                              int32_t rows, int32_t H_kv, int32_t d, int32_t page_size,
                              int32_t num_pages, int32_t* err, cudaStream_t stream) {
    const int64_t items = static_cast<int64_t>(n_pairs) * H_kv * rows;
    if (items <= 0) return cudaSuccess;
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t blocks = (items + 7) / 8;
    const int grid = static_cast<int>(blocks < 8LL * sms ? blocks : 8LL * sms);
    copy_pages_kernel<<<grid, 256, 0, stream>>>(
        static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool),
        reinterpret_cast<const int2*>(pairs), n_pairs, rows, H_kv, d, page_size, num_pages, err);
    return cudaGetLastError();
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                             const int32_t* page_table, const AppendParams& p, int32_t* err,
                             cudaStream_t stream) {
    const int64_t items = static_cast<int64_t>(p.R) * p.H_kv;
    if (items <= 0) return cudaSuccess;
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t blocks = (items + 7) / 8;
    const int grid = static_cast<int>(blocks < 8LL * sms ? blocks : 8LL * sms);
    kv_append_kernel<<<grid, 256, 0, stream>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
        static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), page_table, p, err);
    return cudaGetLastError();
}

}  // namespace fanout
