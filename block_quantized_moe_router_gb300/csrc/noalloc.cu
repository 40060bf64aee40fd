// noalloc.cu -- moe_ffn_forward_noalloc: the expert FFN with a library-owned, statically sized
// workspace, for callers that cannot hand the library device memory.
//
// Who needs this: a host program that fixes its device memory plan at start-up and must not
// see another cudaMalloc afterwards (cudaMalloc may synchronise the device and changes the
// footprint the host budgeted for), or a plugin interface that passes tensors but no workspace
// and gives the plugin no allocator.  Such a caller still owns its inputs and outputs; only
// the scratch moves into the library.
//
// The scratch is one file-scope __device__ array of kNoAllocWorkspaceBytes, present on every
// GPU that loads this library until the process exits.  Host code cannot use the array's
// name as a device address (on the host it names a host-side shadow), so the first call on
// each device looks up the real address with cudaGetSymbolAddress while that device is
// current and caches it; that first call should therefore be made before any stream capture.
// Every call on a device shares the same array: calls whose kernels overlap on the GPU (two
// streams, or two host threads) race on it and must be serialised by the caller.  Nothing in
// the workspace needs to start at zero: each call's dispatch kernel rewrites every region the
// later kernels read, so the contents left by the previous call are never consumed.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kNoAllocWorkspaceBytes = size_t(8) << 20;  // 8 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_workspace[kNoAllocWorkspaceBytes];

std::mutex g_addr_mutex;
void* g_addr[kMaxDevices] = {};

// Device address of g_noalloc_workspace on the current device (looked up once per device).
moe_status_t workspace_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_addr_mutex);
    if (!g_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || !p) return MOE_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_ffn_forward_noalloc(const void* handle, int32_t T, int32_t act,
                                                float g_act1, float g_act2, const void* x_bf16,
                                                const int32_t* topk_ids, const float* topk_w,
                                                void* out_bf16, int32_t* dev_status,
                                                void* stream) {
    // T == 0 is a no-op and needs no workspace
    if (T == 0)
        return moe_ffn_forward(handle, T, act, g_act1, g_act2, x_bf16, topk_ids, topk_w, out_bf16,
                               nullptr, 0, dev_status, stream);
    void* ws = nullptr;
    const moe_status_t a = workspace_address(&ws);
    if (a != MOE_OK) return a;
    // moe_ffn_forward refuses (MOE_ERR_WORKSPACE, nothing launched) when this call's workspace
    // plan is larger than the static array
    return moe_ffn_forward(handle, T, act, g_act1, g_act2, x_bf16, topk_ids, topk_w, out_bf16, ws,
                           kNoAllocWorkspaceBytes, dev_status, stream);
}
