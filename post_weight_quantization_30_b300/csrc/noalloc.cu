// gptq_quantize_layer_noalloc: the whole-layer entry point for callers that
// must not allocate device memory.  Its workspace is a fixed array of device
// memory owned by this file instead of a caller-provided buffer.
//
// Who needs it: code that runs where cudaMalloc is unavailable or forbidden,
// for example a plugin inside a host application that owns all device memory
// through its own pool, a process that must never grow its footprint after
// start-up, or a caller in a real-time loop where a synchronizing allocation
// is not allowed.  Such a caller still allocates (or already owns) W, H and
// the outputs; only the scratch space moves into the library.
//
// The scratch is one file-scope __device__ array of kNoAllocScratchBytes.
// Every GPU on which this module is loaded holds it until the process exits.
// Host code cannot use the array's name as a device address (on the host it
// names a shadow variable), so the device address is looked up once per
// device with cudaGetSymbolAddress, with that device current, and passed on.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;  // 16 MiB
static_assert(kNoAllocScratchBytes == GQ_NOALLOC_SCRATCH_BYTES, "header and library disagree on the scratch size");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up on the
// first call for that device).  Returns nullptr on failure.
void *scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" gq_status gptq_quantize_layer_noalloc(const void *W, gq_dtype wt, int64_t rows, int64_t cols,
                                                 const float *H, int bits, int group, int block, float damp,
                                                 int32_t *qweight, float *scales, int32_t *qzeros, uint8_t *codes,
                                                 float *W_hat, float *row_err, gq_stream_t stream, int64_t *info) {
    const size_t need = gptq_quantize_layer_workspace_size(rows, cols, block);
    if (need == 0 || need > kNoAllocScratchBytes) {
        // Invalid sizes, or a layer too large for the fixed scratch.  Called with no
        // workspace, gptq_quantize_layer runs its own argument checks in its own
        // order and, when they pass, returns GQ_EWORKSPACE; it enqueues nothing
        // either way.  So a bad argument gets the status gptq_quantize_layer
        // would give it, whatever the layer's size.
        return gptq_quantize_layer(W, wt, rows, cols, H, bits, group, block, damp, qweight, scales, qzeros, codes,
                                   W_hat, row_err, nullptr, 0, stream, info);
    }
    void *ws = scratch_on_current_device();
    if (!ws) return GQ_ECUDA;
    // The wrapped call clears every part of the scratch that must start at zero
    // (the sweep's deferred-update buffer, the factor's status word) on `stream`
    // before using it, so what an earlier call left behind does not matter.
    return gptq_quantize_layer(W, wt, rows, cols, H, bits, group, block, damp, qweight, scales, qzeros, codes, W_hat,
                               row_err, ws, kNoAllocScratchBytes, stream, info);
}
