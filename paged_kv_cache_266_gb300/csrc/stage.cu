// Kernel-driven staging copies for host-driven decode steps.
//
// A step whose inputs come from the host (the scheduler's block tables, slots and lengths, the
// new tokens' q/K/V) moves well under a few MB each way.  At that size a copy-engine transfer
// is dominated by its start-up, so the library offers a copy done by the SMs: every thread
// moves 16-byte vectors, four loads in flight, between any two addresses the device can reach
// (device memory, or pinned host memory through its mapped address).  The decode step's launch
// overhead is the part of a decode step "TensorRT-LLM 推理加速实战" §7.1 attacks with CUDA
// graphs; this copy goes into the same graph.
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kStageThreads = 256;
constexpr int kStageMaxBlocks = 1024;

__global__ void __launch_bounds__(kStageThreads) stage_copy_kernel(uint4* dst, const uint4* src, size_t n16) {
    const size_t stride = (size_t)gridDim.x * kStageThreads;
    size_t i = (size_t)blockIdx.x * kStageThreads + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = d;
    }
    for (; i < n16; i += stride) dst[i] = src[i];
}

// The address at which the current device reaches `p`: device memory of the current device,
// or registered (pinned) host memory mapped at the same address on the device (unified
// addressing); anything else (pageable host memory, another device's memory, a mapping at a
// different address) is refused.
pkv_status device_address(const void* p, int device, const void** out) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();  // the failed query leaves a (non-sticky) error behind
        return PKV_ERR_INVALID_ARG;
    }
    if (a.type == cudaMemoryTypeDevice) {
        if (a.device != device) return PKV_ERR_INVALID_ARG;
        *out = p;
        return PKV_OK;
    }
    if (a.type == cudaMemoryTypeHost && a.devicePointer && a.devicePointer == a.hostPointer) {
        *out = p;
        return PKV_OK;
    }
    return PKV_ERR_INVALID_ARG;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_stage_copy(void* dst, const void* src, size_t bytes, pkv_stream_t stream) {
    if (bytes == 0) return PKV_OK;
    if (!dst || !src || ((uintptr_t)dst | (uintptr_t)src | bytes) & 15u) return PKV_ERR_INVALID_ARG;
    const uintptr_t d0 = (uintptr_t)dst, s0 = (uintptr_t)src;
    if (d0 < s0 + bytes && s0 < d0 + bytes) return PKV_ERR_INVALID_ARG;  // overlapping ranges
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return PKV_ERR_CUDA;
    const void *dd = nullptr, *sd = nullptr;
    pkv_status st = pkv::device_address(dst, device, &dd);
    if (st != PKV_OK) return st;
    st = pkv::device_address(src, device, &sd);
    if (st != PKV_OK) return st;
    const size_t n16 = bytes / 16;
    const size_t want = (n16 + pkv::kStageThreads - 1) / pkv::kStageThreads;
    const unsigned blocks = (unsigned)(want < (size_t)pkv::kStageMaxBlocks ? want : (size_t)pkv::kStageMaxBlocks);
    pkv::stage_copy_kernel<<<blocks, pkv::kStageThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4*>(const_cast<void*>(dd)), static_cast<const uint4*>(sd), n16);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
