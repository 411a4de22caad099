// lse_merge.cu -- the stand-alone log-sum-exp merge kernel of split-KV
// partials (used when the merge cannot run inside the attention kernel, and
// by fanout_lse_merge), the device error word, and the bounded-wait self-test
// kernel. The per-row merge itself is merge_row (merge_row.cuh).
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "fanout_internal.h"
#include "merge_row.cuh"
#include "ptx_sm100.cuh"

namespace fanout {

// Device error word of this module: [0] status, [1] wait site, [2] block.
__device__ int32_t g_err_word[4];

namespace {

// One warp per output row at a time; kMergeBatch partials per pass: 24 for
// rows with many partials (decode), 8 when every row has few. Blocks of two
// warps: small enough to be resident beside an attention CTA (which leaves
// ~27 K registers and 2 KB of shared memory of an SM free), so part of the
// grid starts, and runs its dry pass, while the attention kernel is still
// working. The grid is at most what the device holds at once (the rest of it
// starts the moment the attention CTAs leave, in one wave), and warps loop
// over rows with the merge index read one row ahead, so after the wait a row
// costs one memory round trip (its partials).
constexpr int kMergeThreads = 64;
template <int kMergeBatch>
__global__ void __launch_bounds__(kMergeThreads, 1) lse_merge_kernel(const MergeParams p) {
    // Launched as a programmatic dependent of the attention kernel: this grid
    // is resident while that one runs. Before waiting for it to complete, each
    // warp reads the merge index of its first two rows and makes a dry run of
    // the first (instruction and data caches warm, nothing written).
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t n0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const MergeIdx none{0, 0, 0, make_int2(0, 0), 0};
    MergeIdx cur = n0 < p.n_out ? merge_index(p, n0, lane) : none;
    MergeIdx nxt = n0 + warps < p.n_out ? merge_index(p, n0 + warps, lane) : none;
    if (n0 < p.n_out) merge_row_ix<kMergeBatch>(p, cur, lane, true);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int64_t n = n0; n < p.n_out; n += warps) {
        const MergeIdx after = n + 2 * warps < p.n_out ? merge_index(p, n + 2 * warps, lane) : none;
        merge_row_ix<kMergeBatch>(p, cur, lane);
        cur = nxt;
        nxt = after;
    }
}

// Blocks of one merge kernel instance the device holds per SM (looked up once).
template <int kMergeBatch>
int merge_blocks_per_sm() {
    static std::atomic<int> cached{0};
    int v = cached.load(std::memory_order_relaxed);
    if (v > 0) return v;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, lse_merge_kernel<kMergeBatch>,
                                                      kMergeThreads, 0) != cudaSuccess || occ <= 0) {
        (void)cudaGetLastError();
        occ = 8;
    }
    cached.store(occ, std::memory_order_relaxed);
    return occ;
}

// One thread waits on a barrier that nothing will ever complete; the bounded
// wait must give up and report FANOUT_ETIMEOUT.
__global__ void wait_selftest_kernel(int32_t* err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = ptx::smem_u32(&bar);
    ptx::mbar_init(b, 1);
    ptx::fence_barrier_init();
    if (!ptx::mbar_wait(b, 0, limit_ns, nullptr)) {
        if (atomicCAS(err, 0, 5) == 0) err[1] = 99;
    }
}

}  // namespace

cudaError_t launch_lse_merge(const MergeParams& p, cudaStream_t stream) {
    if (p.n_out <= 0) return cudaSuccess;
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int32_t most = p.merge_cnt ? p.merge_stride : p.n_parts;  // partials of the fullest row
    const bool few = most <= 8;
    const int64_t rows_per_block = kMergeThreads / 32;
    const int64_t blocks_needed = (p.n_out + rows_per_block - 1) / rows_per_block;
    const int per_sm = few ? merge_blocks_per_sm<8>() : merge_blocks_per_sm<24>();
    const int grid = static_cast<int>(
        std::min<int64_t>(blocks_needed, static_cast<int64_t>(sms) * per_sm));
    // Programmatic dependent launch: the merge grid may start while the
    // attention kernel finishes; griddepcontrol.wait orders the reads.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (few) return cudaLaunchKernelEx(&cfg, lse_merge_kernel<8>, p);
    return cudaLaunchKernelEx(&cfg, lse_merge_kernel<24>, p);
}

// Device address of this device's error word (the symbol's host-side name is
// only a stand-in; the address must come from the runtime, per device).
// Looked up once per device (with that device current) and cached.
cudaError_t err_word_ptr(int32_t** ptr) {
    static std::atomic<int32_t*> cached[64];  // filled once per device, read lock-free
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool known = dev >= 0 && dev < 64;
    if (known) {
        int32_t* c = cached[dev].load(std::memory_order_acquire);
        if (c) {
            *ptr = c;
            return cudaSuccess;
        }
    }
    std::lock_guard<std::mutex> lk(mu);
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(ptr), g_err_word);
    if (e == cudaSuccess && known) cached[dev].store(*ptr, std::memory_order_release);
    return e;
}

cudaError_t launch_wait_selftest(int32_t* err, unsigned long long limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 1, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace fanout
