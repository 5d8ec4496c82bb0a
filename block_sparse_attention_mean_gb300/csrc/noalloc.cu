// noalloc.cu -- bsa_build_mask for callers that cannot allocate device memory.
//
// bsa_build_mask needs a caller-provided workspace. Some callers cannot call
// cudaMalloc: code running under a framework that owns every byte of device
// memory (a fixed pool carved out at start-up, with no allocation permitted
// afterwards), or a host process whose memory budget is frozen once it is
// serving. This entry point takes its scratch from a fixed array that lives in
// the library's own device memory instead: every GPU that loads the library
// holds the array until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace {

// Fixed scratch of every bsa_build_mask_noalloc call on a device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[BSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
bsa_status scratch_for_current_device(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return BSA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return BSA_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return BSA_OK;
}

}  // namespace

extern "C" bsa_status bsa_build_mask_noalloc(const void *Q, const void *K, int dt, int B, int H, int N, int d,
                                             int block, float density, const bsa_static_spec *spec,
                                             int32_t *row_ptr, int32_t *col_idx, int64_t col_capacity,
                                             uint32_t *bitmap, uint32_t *device_status, void *stream)
{
    // Every argument check runs first: a call that fails here has enqueued nothing,
    // so it neither clears the status word of an earlier call still in flight nor
    // leaves a stray node in a stream capture.
    bsa::MaskArgs a{};
    bsa_status s = bsa::prepare_build_mask(Q, K, dt, B, H, N, d, block, density, spec, row_ptr, col_idx,
                                           col_capacity, bitmap, &a);
    if (s != BSA_OK) return s;
    if (device_status != nullptr && reinterpret_cast<uintptr_t>(device_status) % 4 != 0) return BSA_ERR_INVALID_ARG;
    // A dynamic build pools Q and K into the scratch; a static one keeps only per-row
    // counts and one head's pattern there.
    if (bsa::mask_workspace_need(B, H, N, d, block, spec == nullptr) > BSA_NOALLOC_SCRATCH_BYTES)
        return BSA_ERR_WORKSPACE;  // problem larger than the fixed scratch
    s = bsa::current_sm_count(&a.sm_count);
    if (s != BSA_OK) return s;
    void *scratch = nullptr;
    s = scratch_for_current_device(&scratch);
    if (s != BSA_OK) return s;
    a.ws = static_cast<char *>(scratch);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents: the header (device status
    // word and the counters of last-CTA launches) must start at zero. Every other
    // byte the build reads is written by the same build first.
    if (cudaMemsetAsync(scratch, 0, bsa::kWsHeader, st) != cudaSuccess) return BSA_ERR_CUDA;
    s = bsa::launch_build_mask(a, st);
    if (s != BSA_OK) return s;
    if (device_status != nullptr &&
        cudaMemcpyAsync(device_status, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return BSA_ERR_CUDA;
    return BSA_OK;
}
