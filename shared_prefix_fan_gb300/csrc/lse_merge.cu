// lse_merge.cu -- log-sum-exp merge of split-KV partials, the device error
// word, and the bounded-wait self-test kernel.
//
// The merge is the reduction of ADR-0060 section 4 ("Reduction -- tree to the
// root") and "AHBM Agentic Runtime Architecture" section 3.4 ("Online softmax
// merge"): partial states of the SAME row from different key shards combine as
//   m = max(m_a, m_b); s_a = 2^(m_a - m); s_b = 2^(m_b - m);
//   l = l_a s_a + l_b s_b; o = o_a s_a + o_b s_b;  final out = o / l.
// The pages fold pairs up a tree of PEs over IPCQ links; on one GPU there are
// no links to save, so one warp folds all of a row's partials. It takes the
// overall max first and then sums in a fixed order (the merge is associative
// and commutative, so this is the same fold), so results are bitwise
// reproducible.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "fanout_internal.h"
#include "ptx_sm100.cuh"

namespace fanout {

// Device error word of this module: [0] status, [1] wait site, [2] block.
__device__ int32_t g_err_word[4];

namespace {

// One warp per output row n (a (token, query head) pair). Its partials are
// either listed in the merge index (planned mode: fixed-stride entry lists
// {part, row base} per (token, KV head), row = base + g) or uniform
// (part-major [n_parts][n_out]). The count and the first 32 entries of a row
// load together; then up to kMergeBatch partials per pass: lane e loads entry
// e's (m, l) while every lane loads its 4 columns of all the pass's O vectors,
// so a row of up to kMergeBatch partials costs two memory round trips.
// kMergeBatch partials per pass: 24 for rows with many partials (decode), 8 when
// every row has few (a smaller register footprint keeps three blocks per SM).
template <int kMergeBatch, int kMinBlocks>
__global__ void __launch_bounds__(256, kMinBlocks) lse_merge_kernel(const MergeParams p) {
    // Launched as a programmatic dependent of the attention kernel: wait until
    // that grid has completed and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const bool planned = p.merge_cnt != nullptr;
    const int H_kv = planned ? p.H_q / p.G : 1;
    for (int64_t n = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         n < p.n_out; n += warps) {
        int32_t ne = p.n_parts, g = 0;
        int64_t key = 0;
        int2 ent0 = make_int2(0, 0);
        if (planned) {
            const int64_t tok = n / p.H_q;
            const int32_t hq = static_cast<int32_t>(n % p.H_q);
            key = tok * H_kv + hq / p.G;
            g = hq % p.G;
            if (lane < p.merge_stride) ent0 = p.merge_ent[key * p.merge_stride + lane];
            ne = p.merge_cnt[key];
            if (ne <= 0) continue;  // written directly by the attention kernel
        }
        float M = -INFINITY, L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int32_t c0 = 0; c0 < ne; c0 += kMergeBatch) {
            const int32_t cnt = min(kMergeBatch, ne - c0);
            int64_t my_row = 0;
            if (lane < cnt) {
                if (planned) {
                    const int2 en = (c0 == 0) ? ent0 : p.merge_ent[key * p.merge_stride + c0 + lane];
                    my_row = static_cast<int64_t>(en.x) * p.rows_per_part + en.y + g;
                } else {
                    my_row = static_cast<int64_t>(c0 + lane) * p.n_out + n;
                }
            }
            float2 ml = make_float2(-INFINITY, 0.f);
            if (lane < cnt) ml = p.part_ml[my_row];
            float4 o[kMergeBatch];
#pragma unroll
            for (int u = 0; u < kMergeBatch; ++u) {
                const int64_t r = __shfl_sync(0xffffffffu, my_row, min(u, cnt - 1));
                o[u] = (u < cnt) ? reinterpret_cast<const float4*>(p.part_o + r * kHD)[lane]
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            // running (max, sum) over passes, in the base-2 domain
            float mb = (ml.y > 0.f) ? ml.x : -INFINITY;
#pragma unroll
            for (int s = 16; s > 0; s >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, s));
            const float m_new = fmaxf(M, mb);
            const float corr = (M == -INFINITY) ? 0.f : ptx::ex2(M - m_new);
            const float w = (ml.y > 0.f) ? ptx::ex2(ml.x - m_new) : 0.f;  // empty shard: 0
            float lb = w * ml.y;
#pragma unroll
            for (int s = 16; s > 0; s >>= 1) lb += __shfl_xor_sync(0xffffffffu, lb, s);
            L = L * corr + lb;
            acc.x *= corr;
            acc.y *= corr;
            acc.z *= corr;
            acc.w *= corr;
#pragma unroll
            for (int u = 0; u < kMergeBatch; ++u) {
                const float wu = __shfl_sync(0xffffffffu, w, u);  // 0 for u >= cnt
                acc.x += wu * o[u].x;
                acc.y += wu * o[u].y;
                acc.z += wu * o[u].z;
                acc.w += wu * o[u].w;
            }
            M = m_new;
        }
        const float inv = 1.f / L;
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
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t blocks_needed = (p.n_out + 7) / 8;
    const int grid =
        static_cast<int>(std::min<int64_t>(blocks_needed, static_cast<int64_t>(sms) * 16));
    // Programmatic dependent launch: the merge grid may start while the
    // attention kernel finishes; griddepcontrol.wait orders the reads.
    const int32_t most = p.merge_cnt ? p.merge_stride : p.n_parts;  // partials of the fullest row
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (most <= 8) return cudaLaunchKernelEx(&cfg, lse_merge_kernel<8, 3>, p);
    return cudaLaunchKernelEx(&cfg, lse_merge_kernel<24, 1>, p);
}

// Device address of this device's error word (the symbol's host-side name is
// only a stand-in; the address must come from the runtime, per device).
// Looked up once per device (with that device current) and cached.
cudaError_t err_word_ptr(int32_t** ptr) {
    static int32_t* cached[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && cached[dev]) {
        *ptr = cached[dev];
        return cudaSuccess;
    }
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(ptr), g_err_word);
    if (e == cudaSuccess && dev >= 0 && dev < 64) cached[dev] = *ptr;
    return e;
}

cudaError_t launch_wait_selftest(int32_t* err, unsigned long long limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 1, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace fanout
