// decode_static_ws.cu -- attn_fwd_decode_static_ws: the decode entry point for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where they run
// attention: code that runs under a fixed memory budget set up once at start-up, plug-ins
// hosted inside another runtime that owns every device allocation, or real-time loops
// that must not enter the driver's allocator.  For them the split-KV scratch (partial
// outputs and their (max, sum) pairs) lives in one fixed array compiled into this library
// instead of a caller-provided workspace.
//
// The array is kDecodeStaticScratchBytes (64 MiB) of device memory on every GPU that
// loads the library, held until the process exits.  Calls whose scratch would exceed it
// are rejected with ATTN_ERR_WORKSPACE before anything is enqueued.  All calls share the
// array: two calls that overlap on the GPU (different streams, or different host threads
// without ordering) race on it.  Nothing in it needs to start at zero -- every partial the
// combine step reads is written earlier in the same call -- so it is never cleared.
//
// In host code the array's name is only a stand-in for the symbol, not a device address.
// Every call made while its stream is not being captured looks the real address up with
// cudaGetSymbolAddress (on the current device) and remembers it per device; a call made
// during a stream capture uses the remembered address, because the lookup may load the
// module, which a capture does not allow.  So the first call on each device should come
// before any stream capture begins.  A device reset (cudaDeviceReset) unloads the module
// and may move the array: the next call outside a capture picks up the new address, and
// graphs captured before the reset must be captured again.
#include <math.h>

#include <mutex>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr size_t kDecodeStaticScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_decode_static_scratch[kDecodeStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the static scratch on the current device: looked up afresh when the
// stream is not capturing, else the address remembered from an earlier call.
cudaError_t static_scratch_address(cudaStream_t stream, void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (cap == cudaStreamCaptureStatusNone) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    } else if (g_scratch_ptr[dev] == nullptr) {
        return cudaErrorStreamCaptureUnsupported;  // no lookup before the capture began
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace attn

extern "C" attn_status attn_fwd_decode_static_ws(
    const void* q, const void* k_cache, const void* v_cache, const uint32_t* block_table,
    const int32_t* cache_len, int b, int hq, int hkv, int d, int s_active, int page_size,
    int max_pages_per_seq, int num_pages, int max_cache_len, float scale, void* o, float* lse,
    attn_dtype o_dtype, int kv_chunk, void* stream) {
    const size_t need =
        attn_decode_workspace_bytes(b, hq, s_active, d, max_cache_len, kv_chunk);
    if (need == 0) {
        // invalid sizes: let the regular checks name the problem (no scratch is touched)
        return attn_fwd_decode(q, k_cache, v_cache, block_table, cache_len, b, hq, hkv, d,
                               s_active, page_size, max_pages_per_seq, num_pages, max_cache_len,
                               scale, o, lse, o_dtype, kv_chunk, nullptr, 0, stream);
    }
    if (need > attn::kDecodeStaticScratchBytes) return ATTN_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (attn::static_scratch_address(static_cast<cudaStream_t>(stream), &scratch) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    return attn_fwd_decode(q, k_cache, v_cache, block_table, cache_len, b, hq, hkv, d, s_active,
                           page_size, max_pages_per_seq, num_pages, max_cache_len, scale, o, lse,
                           o_dtype, kv_chunk, scratch, attn::kDecodeStaticScratchBytes, stream);
}
