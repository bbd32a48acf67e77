// wf_lmhead_argmax_noalloc: the LM-head argmax for callers that cannot hand
// the library a workspace.
//
// Some callers never get to allocate device memory: a plug-in that a host
// inference engine calls with nothing but its input and output buffers (the
// engine owns every byte of device memory and offers no allocator), or a
// latency-critical decode loop that may not call cudaMalloc because it
// synchronises the whole device.  For them this variant keeps its scratch -
// the control block and one packed key per verified row - in a fixed
// file-scope device array instead of a caller-provided workspace.
//
// Costs and limits:
// - every GPU that loads the library holds the array (WF_NOALLOC_MAX_ROWS * 8
//   + 256 bytes, about 128 KB) until the process exits;
// - P above WF_NOALLOC_MAX_ROWS is rejected with WF_ERR_INVALID_ARG;
// - every call on a device uses the same array: calls whose work overlaps on
//   the GPU (different streams, or concurrent host threads) race with each
//   other and must be serialised by the caller;
// - the first call on a device looks up the array's device address for that
//   device (host code cannot use the array's name as an address); make that
//   first call before any stream capture.
#include <mutex>

#include "wf_internal.cuh"

namespace wf {

wf_status launch_lmhead_argmax(const uint16_t* hidden, const uint16_t* W, int P, int d, int V, int32_t* ids,
                               float* maxlogit, void* ws, cudaStream_t s);

constexpr size_t NOALLOC_BYTES = sizeof(Control) + sizeof(uint64_t) * (size_t)WF_NOALLOC_MAX_ROWS;

static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_BYTES];

static std::mutex g_noalloc_mu;
static void* g_noalloc_addr[64];

// Device address of the scratch array on the current device (looked up once per device).
static wf_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return WF_ERR_CUDA;
    if (dev < 0 || dev >= 64) return WF_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return WF_ERR_CUDA;
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return WF_OK;
}

wf_status noalloc_lmhead_argmax(const uint16_t* hidden, const uint16_t* W, int P, int d, int V, int32_t* ids,
                                float* maxlogit, cudaStream_t s) {
    if (P > WF_NOALLOC_MAX_ROWS) return WF_ERR_INVALID_ARG;
    void* scratch = nullptr;
    const wf_status st = noalloc_scratch(&scratch);
    if (st != WF_OK) return st;
    // The array keeps whatever the previous call left; the keys and the
    // CTA counter must start at zero.
    if (cudaMemsetAsync(scratch, 0, sizeof(Control) + sizeof(uint64_t) * (size_t)P, s) != cudaSuccess)
        return WF_ERR_CUDA;
    return launch_lmhead_argmax(hidden, W, P, d, V, ids, maxlogit, scratch, s);
}

// The error word of the array's control block (a bounded wait that gave up
// records WF_ERR_TIMEOUT there): copied out after the work before it on the
// stream, optionally cleared.
wf_status noalloc_read_device_error(int* code, int* info, int clear, cudaStream_t s) {
    void* scratch = nullptr;
    const wf_status st = noalloc_scratch(&scratch);
    if (st != WF_OK) return st;
    uint32_t h[2] = {0, 0};
    if (cudaMemcpyAsync(h, scratch, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess) return WF_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return WF_ERR_CUDA;
    *code = (int)h[0];
    if (info) *info = (int)h[1];
    if (clear) {
        if (cudaMemsetAsync(scratch, 0, sizeof h, s) != cudaSuccess) return WF_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return WF_ERR_CUDA;
    }
    return WF_OK;
}

}  // namespace wf
