// read_floor.cu -- a calibration read with no counterpart in the method: one
// launch that streams a device buffer once from HBM with plain 16-byte loads
// and nothing else. Timed the way an attention call is timed (after an L2
// flush, CUDA events on the stream), it is the shortest time a single kernel
// that reads those bytes takes on this device, launch and ramp included: the
// floor under an HBM-bound call, which the copy-bandwidth roofline (a long
// steady stream) leaves out.
#include <cuda_runtime.h>

#include <cstdint>

namespace fanout {
namespace {

constexpr int kReadThreads = 512;
constexpr int kReadInFlight = 8;  // independent 16-byte loads per thread per step

// Grid-stride over the buffer; every thread keeps kReadInFlight loads in
// flight (evict-first: the data is read once). The xor of all words goes to
// *xor_out so that the loads are the kernel's result and a test can check
// that every byte was read.
__global__ void __launch_bounds__(kReadThreads) stream_read_kernel(const uint4* __restrict__ a,
                                                                   int64_t n16,
                                                                   uint32_t* xor_out) {
    uint32_t acc = 0;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + (kReadInFlight - 1) * stride < n16; i += kReadInFlight * stride) {
        uint4 v[kReadInFlight];
#pragma unroll
        for (int k = 0; k < kReadInFlight; ++k) v[k] = __ldcs(a + i + k * stride);
#pragma unroll
        for (int k = 0; k < kReadInFlight; ++k) acc ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
    }
    for (; i < n16; i += stride) {
        const uint4 v = __ldcs(a + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, s);
    if ((threadIdx.x & 31) == 0 && acc != 0u) atomicXor(xor_out, acc);
}

}  // namespace

// Four CTAs of 512 threads per SM: enough loads in flight to saturate HBM
// (a probe of 1, 2, 4 and 8 CTAs per SM: 2 and more read equally fast).
cudaError_t launch_stream_read(const void* buf, int64_t bytes, uint32_t* xor_out,
                               cudaStream_t stream) {
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    stream_read_kernel<<<4 * sms, kReadThreads, 0, stream>>>(static_cast<const uint4*>(buf),
                                                               bytes / 16, xor_out);
    return cudaGetLastError();
}

}  // namespace fanout
