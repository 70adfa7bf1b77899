// static_ws.cu -- ssd_chunk_scan_static_ws: ssd_chunk_scan with its scratch
// in a fixed device array, for callers that cannot allocate device memory.
//
// The callers: code running inside a host program that owns every device
// allocation (a plugin of another runtime, which hands it tensors but no
// allocator), and serving loops that must keep cudaMalloc off their hot path
// because it can synchronise the device.  ssd_chunk_scan's tensor-core path
// with the conv fused needs a scratch buffer for the post-conv B|C columns
// of every row; here that buffer is g_scan_scratch, a file-scope array in
// this library's device image (SSD_STATIC_SCRATCH_BYTES on every GPU that
// loads the library, held until the process exits).  Nothing is allocated.
//
// In host code the name g_scan_scratch denotes a host-side shadow, not the
// device array, so the device address is looked up with
// cudaGetSymbolAddress, once per device with that device current, on the
// first call made on that device, and cached.
//
// No part of the array has to start at zero: the B|C conv kernel writes
// every scratch row the scan kernel reads, earlier on the same stream.  Every
// call on a GPU uses the same array, so calls that overlap on the GPU race.
#include "../../include/ssd.h"

#include <cuda_runtime.h>

#include <mutex>

namespace {

static __device__ __align__(256) unsigned char g_scan_scratch[SSD_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];  // device address of g_scan_scratch, per device
std::mutex g_scratch_mutex;

ssd_status scratch_address(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_scan_scratch) != cudaSuccess || ptr == nullptr)
            return SSD_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return SSD_OK;
}

}  // namespace

extern "C" ssd_status ssd_chunk_scan_static_ws(
    const ssd_dims* dims, ssd_dtype act, unsigned flags, const void* xbc, const float* conv_w,
    const float* conv_b, const void* conv_state_in, void* conv_state_out, const float* dt,
    const float* dt_bias, const float* A, const float* D, const void* z,
    const float* ssm_state_in, void* y, float* ssm_state_out, cudaStream_t stream)
{
    size_t need = 0;
    ssd_status s = ssd_chunk_scan_workspace_size(dims, act, flags, conv_w != nullptr, &need);
    if (s != SSD_OK) return s;
    if (need > SSD_STATIC_SCRATCH_BYTES) return SSD_ERR_UNSUPPORTED;  // larger than the array
    void* ws = nullptr;
    size_t ws_bytes = 0;
    if (need > 0) {
        s = scratch_address(&ws);
        if (s != SSD_OK) return s;
        ws_bytes = SSD_STATIC_SCRATCH_BYTES;
    }
    return ssd_chunk_scan(dims, act, flags, xbc, conv_w, conv_b, conv_state_in, conv_state_out,
                          dt, dt_bias, A, D, z, ssm_state_in, y, ssm_state_out, ws, ws_bytes,
                          stream);
}
