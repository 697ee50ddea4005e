// sb_static.cu -- sb_lmhead_project_static_scratch: the projection call for callers that
// cannot hand the library a workspace.
//
// Some callers cannot call cudaMalloc: a plug-in running inside a host engine that owns the
// whole device-memory pool (it pre-reserves HBM for its own caches and exposes no allocator
// hook), code on a latency-critical path where cudaMalloc's implicit device synchronisation
// is not allowed, or a foreign-function caller that links only this library and never sees
// the CUDA allocator.  For them this entry point takes its scratch (the per-tile records,
// the target logits and the device status word) from a fixed array compiled into the
// library instead of from the caller.
//
// The array below is a file-scope __device__ variable: every GPU that loads the library
// holds its kSbStaticScratchBytes until the process exits.  Host code cannot use the name
// `g_sb_scratch` as a device address (on the host it is only a stand-in symbol; passing it
// to a kernel would fault, or silently use the wrong memory where the GPU can reach host
// memory), so the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current, checks the result, caches it, and
// passes that pointer to the kernels.
#include <cstdint>
#include <mutex>

#include "sb.h"
#include "sb_internal.h"

namespace {

constexpr size_t kSbStaticScratchBytes = size_t(8) << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_sb_scratch[kSbStaticScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_sb_scratch on the current device, looked up once per device.
int32_t scratch_address(void **ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SB_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SB_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_sb_scratch) != cudaSuccess || p == nullptr)
            return SB_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return SB_OK;
}

}  // namespace

extern "C" int32_t sb_lmhead_project_static_scratch(const void *H, const void *W, int64_t M,
                                                    int64_t d, int64_t V, int32_t k,
                                                    int32_t surface, float temperature,
                                                    uint64_t seed, const sb_outputs *out,
                                                    void *stream) {
    if (!out) return SB_ERR_INVALID_ARG;
    const size_t need = sb_workspace_bytes(M, V, k, surface);
    if (need == 0) return SB_ERR_INVALID_ARG;
    if (need > kSbStaticScratchBytes) return SB_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    if (int32_t e = scratch_address(&scratch)) return e;
    sb_outputs o = *out;
    o.workspace = scratch;
    o.workspace_bytes = kSbStaticScratchBytes;
    return sb_lmhead_project(H, W, M, d, V, k, surface, temperature, seed, &o, stream);
}

// The device status of the last static-scratch call on the current device: its status
// word sits in the array's header, which the caller cannot address, so it is read here
// through the looked-up address, as sb_last_device_status reads a caller's workspace.
extern "C" int32_t sb_static_scratch_last_status(void) {
    void *scratch = nullptr;
    if (int32_t e = scratch_address(&scratch)) return e;
    sb_outputs o{};
    o.workspace = scratch;
    o.workspace_bytes = kSbStaticScratchBytes;
    return sb_last_device_status(&o);
}
