// Decode with library-owned scratch, for callers that cannot allocate.
//
// oxd_paged_decode_run needs a device workspace from its caller. Some callers
// cannot provide one: a serving process that reserves all of its HBM at
// start-up (weights, KV pages) and forbids later cudaMalloc, so that memory
// never fragments and no allocation ever stalls the device mid-decode; or a
// host that calls this library through a plugin interface that hands over
// only the input and output tensors and gives no access to an allocator.
// For them, oxd_paged_decode_run_static_workspace uses scratch that is part
// of the library itself: a file-scope device array, reserved once on every
// GPU that loads the library and kept until the process exits. It calls no
// cudaMalloc, no cudaFree and no allocating library routine.
#include <mutex>

#include "../../include/oxd.h"
#include "oxd_internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t{32} << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

// In host code this name is only a host-side stand-in for the device array;
// its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the array on `device`, which must be the calling thread's
// current device. Looked up once per device, on that device's first call.
cudaError_t static_workspace_address(int device, void** out) {
    if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_addr[device] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
        if (e != cudaSuccess) return e;
        g_addr[device] = p;
    }
    *out = g_addr[device];
    return cudaSuccess;
}

}  // namespace

extern "C" oxd_status oxd_paged_decode_run_static_workspace(
    oxd_plan plan, const void* q, const void* k_pages, const void* v_pages, const int32_t* indptr,
    const int32_t* indices, const int32_t* last_page_len, float sm_scale, void* out, float* lse,
    void* stream) {
    oxd_plan_info info;
    const oxd_status st = oxd_plan_get_info(plan, &info);
    if (st != OXD_OK) return st;
    if (info.workspace_bytes < 0 ||
        static_cast<size_t>(info.workspace_bytes) > kStaticWorkspaceBytes)
        return OXD_ERR_WORKSPACE_TOO_SMALL;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return OXD_ERR_CUDA;
    void* ws = nullptr;
    if (static_workspace_address(device, &ws) != cudaSuccess) return OXD_ERR_CUDA;
    // Nothing in the array has to start at zero: a run writes everything it
    // reads, and its status word is tagged with the run's epoch.
    return oxd_paged_decode_run(plan, q, k_pages, v_pages, indptr, indices, last_page_len,
                                sm_scale, out, lse, ws, kStaticWorkspaceBytes, stream);
}

extern "C" oxd_status oxd_read_static_workspace_status(void* stream, int32_t* code) {
    if (code == nullptr) return OXD_ERR_INVALID_ARGUMENT;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return OXD_ERR_CUDA;
    void* ws = nullptr;
    if (static_workspace_address(device, &ws) != cudaSuccess) return OXD_ERR_CUDA;
    // The status word sits where a caller-provided workspace keeps it, so the
    // regular reader applies (it synchronises the stream first).
    return oxd_read_device_status(ws, stream, code);
}
