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
// overall max first and then sums, in ascending slot order -- the same fold
// (the merge is associative and commutative) with a fixed order, so results
// are bitwise reproducible.
#include <cuda_bf16.h>

#include "fanout_internal.h"
#include "ptx_sm100.cuh"

namespace fanout {

// Device error word of this module: [0] status, [1] wait site, [2] block.
__device__ int32_t g_err_word[4];

namespace {

__global__ void __launch_bounds__(256)
    lse_merge_kernel(const float* __restrict__ part_o, const float2* __restrict__ part_ml,
                     const int32_t* __restrict__ tok_slots, int32_t n_parts, int64_t n_out,
                     int32_t group, void* __restrict__ out, int32_t out_bf16,
                     float* __restrict__ lse) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t n = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; n < n_out;
         n += warps) {
        const int32_t np = tok_slots ? tok_slots[n / group] : n_parts;
        if (np <= 0) continue;  // written directly by the attention kernel
        float M = -INFINITY;
        for (int32_t s = 0; s < np; ++s) {
            const float2 ml = part_ml[s * n_out + n];
            if (ml.y > 0.f) M = fmaxf(M, ml.x);
        }
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int32_t s = 0; s < np; ++s) {
            const float2 ml = part_ml[s * n_out + n];
            if (!(ml.y > 0.f)) continue;  // no visible key in this shard: weight 0
            const float w = ptx::ex2(ml.x - M);
            L += w * ml.y;
            const float4 o =
                reinterpret_cast<const float4*>(part_o + (s * n_out + n) * kHD)[lane];
            acc.x += w * o.x;
            acc.y += w * o.y;
            acc.z += w * o.z;
            acc.w += w * o.w;
        }
        const float inv = 1.f / L;
        if (out_bf16) {
            uint2 v = make_uint2(ptx::pack_bf16x2(acc.x * inv, acc.y * inv),
                                 ptx::pack_bf16x2(acc.z * inv, acc.w * inv));
            reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + n * kHD)[lane] = v;
        } else {
            reinterpret_cast<float4*>(static_cast<float*>(out) + n * kHD)[lane] =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
        if (lse && lane == 0) lse[n] = (M + __log2f(L)) * 0.69314718055994531f;
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

cudaError_t launch_lse_merge(const float* part_o, const float2* part_ml,
                             const int32_t* tok_slots, int32_t n_parts, int64_t n_out,
                             int32_t group, void* out, int32_t out_bf16, float* lse,
                             cudaStream_t stream) {
    if (n_out <= 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t blocks_needed = (n_out + 7) / 8;
    const int grid = static_cast<int>(std::min<int64_t>(blocks_needed, static_cast<int64_t>(sms) * 8));
    lse_merge_kernel<<<grid, 256, 0, stream>>>(part_o, part_ml, tok_slots, n_parts, n_out, group,
                                               out, out_bf16, lse);
    return cudaGetLastError();
}

// Device address of this device's error word (the symbol's host-side name is
// only a stand-in; the address must come from the runtime, per device).
cudaError_t err_word_ptr(int32_t** ptr) {
    return cudaGetSymbolAddress(reinterpret_cast<void**>(ptr), g_err_word);
}

cudaError_t launch_wait_selftest(int32_t* err, unsigned long long limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 1, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace fanout
