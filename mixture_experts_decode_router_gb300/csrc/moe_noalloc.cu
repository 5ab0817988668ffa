// moe_noalloc.cu -- moe_forward without a caller-supplied workspace.
//
// Some callers cannot allocate device memory: a plugin whose host application
// owns every allocation and hands it only input and output buffers, or code
// that is recording a CUDA graph, where cudaMalloc is not allowed.  For them
// this file keeps the layer's scratch in one file-scope device array,
// kStaticWorkspaceBytes (16 MiB) large, which every GPU that loads the library
// holds until the process exits.  The entry point allocates nothing and calls
// no allocating routine; it runs the same kernels as moe_forward.  All calls
// share the one array, so calls whose work overlaps on the GPU (two streams,
// or two host threads) race on it.
//
// Device-side failures of these calls (a bounded wait that gave up, or a
// refused dirty control block) are recorded in the array's control block, like
// a caller workspace's; moe_static_workspace_check reads and clears them.
#include <mutex>

#include "moe_launch.cuh"

namespace moe {
moe_status_t forward_with_workspace(const moe_config_t* cfg, const moe_weights_t* wts, const void* x,
                                    int32_t n, void* out, int32_t* idx, float* w, void* ws,
                                    size_t ws_bytes, moe_stream_t stream);
}

namespace {

constexpr size_t kStaticWorkspaceBytes = MOE_STATIC_WORKSPACE_BYTES;

// The scratch.  In host code this name is a host-side stand-in, not a device
// address: the set-up below asks the runtime for the device address.
__device__ __align__(256) uint8_t g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void* g_ws_ptr[kMaxDevices] = {};

bool capturing(cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return true;   // unknown: treat as capturing (refuse rather than break a capture)
    }
    return cs != cudaStreamCaptureStatusNone;
}

// Once per device, with that device current: the array's device address, and
// its control block cleared (the part of the workspace that must start at
// zero), on the caller's stream, which is then synchronised.  Runs on the
// first call made on each device; a first call made while `st` is being
// captured into a graph is refused (MOE_ERR_UNSUPPORTED), because the set-up
// synchronises.
moe_status_t static_workspace(cudaStream_t st, void** ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ws_ptr[dev]) {
        if (capturing(st)) return MOE_ERR_UNSUPPORTED;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return MOE_ERR_CUDA;
        if (cudaMemsetAsync(p, 0, sizeof(moe::Ctrl), st) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
        g_ws_ptr[dev] = p;
    }
    *ptr = g_ws_ptr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t moe_forward_static_ws(const moe_config_t* cfg, const moe_weights_t* wts, const void* x,
                                   int32_t n, void* out, int32_t* idx, float* w, moe_stream_t stream) {
    if (cfg && n > 0 && moe_workspace_bytes(cfg, n) > kStaticWorkspaceBytes) return MOE_ERR_WORKSPACE;
    void* ws = nullptr;
    const moe_status_t s = static_workspace(reinterpret_cast<cudaStream_t>(stream), &ws);
    if (s != MOE_OK) return s;
    return moe::forward_with_workspace(cfg, wts, x, n, out, idx, w, ws, kStaticWorkspaceBytes, stream);
}

moe_status_t moe_static_workspace_check(int32_t* device_error, void** workspace, moe_stream_t stream) {
    if (!device_error) return MOE_ERR_NULL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (capturing(st)) return MOE_ERR_UNSUPPORTED;   // it synchronises the stream
    void* ws = nullptr;
    const moe_status_t s = static_workspace(st, &ws);
    if (s != MOE_OK) return s;
    if (workspace) *workspace = ws;
    return moe_workspace_check(ws, kStaticWorkspaceBytes, device_error, stream);
}

}  // extern "C"
