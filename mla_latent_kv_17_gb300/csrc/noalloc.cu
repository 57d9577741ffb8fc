// Dense decode for callers that cannot allocate device memory themselves.
//
// Some callers run where no allocation may happen at decode time: a host that has handed
// all device memory to a fixed arena up front, a real-time loop that must not call
// cudaMalloc (it can synchronise the device and take unbounded time), or a plugin whose
// host application owns every allocation.  They can still pass their inputs and outputs,
// but not a workspace.  mla_decode_static() gives them the plan + decode + merge with the
// workspace taken from a fixed array in this library's device image instead.
//
// The array is kStaticScratchBytes of device memory.  Each GPU that loads this library's
// module holds its own copy until the process exits.  On one device all calls share that
// copy: two calls whose work overlaps on the GPU (for example on two streams) race and
// corrupt each other's plan and partial results; calls on one stream run in order and are
// safe.  Each call rebuilds the plan and clears the status word before decoding, so
// nothing a previous call left in the array is read.
//
// The first call on a device looks up the array's device address (cudaGetSymbolAddress,
// which also loads this module on that device).  Make that first call before capturing a
// stream into a CUDA graph.
#include <cuda_runtime.h>

#include <mutex>

#include "mla_decode.h"
#include "plan.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(48) << 20;  // 48 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per device.  In host
// code `g_static_scratch` names a host-side stand-in, never the device memory itself.
mla_status scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();  // leave no pending error behind for the caller's next CUDA call
            return MLA_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MLA_OK;
}

}  // namespace

extern "C" mla_status mla_decode_static(const void *q_nope, const void *q_rope, const void *cache,
                                        mla_kv_dtype kv_dtype, int64_t num_pages,
                                        const int32_t *block_table, int max_pages,
                                        const int32_t *seq_lens, int B, int H,
                                        float softmax_scale, float *out, float *lse,
                                        int32_t *device_status, void *stream) {
    if (B < 1 || H < 1) return MLA_ERR_INVALID_ARG;
    if (H > mla::kMaxHeads) return MLA_ERR_UNSUPPORTED;
    const size_t need = mla_decode_workspace_size(B, H, 0);
    if (need == 0) return MLA_ERR_CUDA;
    if (need > kStaticScratchBytes) return MLA_ERR_WORKSPACE;  // B x H beyond the fixed array
    void *ws = nullptr;
    mla_status st = scratch_for_current_device(&ws);
    if (st != MLA_OK) return st;
    st = mla_decode_plan(seq_lens, B, H, 0, kv_dtype, 0, ws, kStaticScratchBytes, stream);
    if (st != MLA_OK) return st;
    st = mla_decode(ws, kStaticScratchBytes, q_nope, q_rope, cache, kv_dtype, num_pages,
                    block_table, max_pages, seq_lens, B, H, softmax_scale, out, lse, stream);
    if (st != MLA_OK) return st;
    if (device_status) {
        const unsigned char *status_word =
            static_cast<const unsigned char *>(ws) + mla::ws_layout(1, 1, 1).status;
        if (cudaMemcpyAsync(device_status, status_word, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                            static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return MLA_ERR_CUDA;
    }
    return MLA_OK;
}
