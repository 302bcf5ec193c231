// attn_internal.h -- host-side interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Arguments reaching these functions are already validated.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "../../include/attn.h"

namespace attn {

// One-time setup of a kernel (its shared-memory limit, a register check) is per device:
// `done` holds one bit per device id.  needs_setup() is true until mark_setup() has run for
// the current device (device ids past 63 are set up on every call).
inline bool needs_setup(const std::atomic<unsigned long long>& done) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return true;
    }
    return dev < 0 || dev >= 64 || (done.load(std::memory_order_acquire) & (1ull << dev)) == 0;
}
inline void mark_setup(std::atomic<unsigned long long>& done) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    if (dev >= 0 && dev < 64) done.fetch_or(1ull << dev, std::memory_order_release);
}

// Bits of the per-translation-unit device error words (read and cleared by the host).
enum : unsigned {
    kDevErrPageOOB = 1u,   // a page-table entry >= num_pages was met (page not read)
    kDevErrTimeout = 2u,   // a pipeline wait ran past its limit (kernel gave up)
    kDevErrCacheLen = 4u,  // a cache_len outside [s_active, max_cache_len] (sequence skipped)
};

struct PrefillArgs {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;
    int b, hq, hkv, sq, skv, d;
    float scale;
    int causal, window;
    attn_dtype o_dtype;
    const float* sink;  // [hq] sink logits, or NULL
    const int32_t* cu_seqlens_q;  // packed sequences: [nseq + 1] offsets, or NULL
    const int32_t* cu_seqlens_k;
    int nseq;
    int* order;  // packed: scratch of one int per query tile for the work order, or NULL
};

struct DecodeArgs {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const uint32_t* block_table;  // NULL for a flat cache
    const int32_t* cache_len;
    int b, hq, hkv, d, s_active, page_size, max_pages_per_seq, num_pages, max_cache_len;
    float scale;
    void* o;
    float* lse;
    attn_dtype o_dtype;
    int kv_chunk;         // resolved (> 0)
    float* part_o;        // [b*hq*s_active][max_slots][d]: one partial per piece of a pair
    float* part_ml;       // [b*hq*s_active][max_slots][2]
    int* npieces;         // [b*hkv]: pieces written for each (sequence, kv head)
    int max_slots;        // partials a pair may need (kv_chunk bounds the piece count)
    const float* sink;    // [hq] sink logits, or NULL
    int kv_e4m3;          // the caches hold e4m3 bytes
    float k_scale, v_scale;  // their dequantisation scales (1 for bf16)
    int window;           // decode window (0 = none)
    int circular;         // flat cache used as a ring of max_cache_len rows
    const float* rope_inv_freq;  // [d/2] RoPE inverse frequencies of Q, or NULL
};

// The new tokens' K/V written into a bf16 cache (attn_append_kv).
struct AppendArgs {
    const void* k_new;
    const void* v_new;
    void* k_cache;
    void* v_cache;
    const uint32_t* block_table;  // NULL for a flat cache
    const int32_t* cache_len;
    int b, hkv, d, s_active, page_size, max_pages_per_seq, num_pages, max_cache_len, circular;
    const float* rope_inv_freq;  // [d/2], or NULL
};

// Tokens per tile of the decode kernels: splits cover whole tiles, and a window's first
// slot is rounded down to a tile boundary.
constexpr int kDecodeTile = 32;

// Tokens per split when the caller passes kv_chunk = 0: the largest power of two in
// [kMinDefaultKvChunk, kMaxDefaultKvChunk] that is at most b * max_cache_len / 128, i.e.
// about 128 splits across the batch for every kv head.  Long splits keep the per-split
// merge and the partial-output traffic small; short batches still get enough CTAs.
constexpr int kMinDefaultKvChunk = 256;
constexpr int kMaxDefaultKvChunk = 4096;
inline int default_kv_chunk(int b, int max_cache_len) {
    const long long per = (long long)b * max_cache_len / 128;
    int chunk = kMaxDefaultKvChunk;
    while (chunk > kMinDefaultKvChunk && chunk > per) chunk >>= 1;
    return chunk;
}

// cuTensorMapEncodeTiled, fetched once through the runtime (no link against libcuda).
typedef CUresult (*TensorMapEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                      const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                      const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                      CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
TensorMapEncodeFn tensor_map_encoder();

// bf16 tensor map of rank 2 or 3 (innermost dim first), 128-byte swizzle, zero OOB fill.
bool make_bf16_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                   const uint64_t* strides_bytes, const uint32_t* box);
// The same for a tensor of bytes (e4m3 values): dims and box in bytes.
bool make_u8_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box);

attn_status prefill_launch(const PrefillArgs& a, cudaStream_t stream);
attn_status decode_launch(const DecodeArgs& a, cudaStream_t stream);
attn_status append_launch(const AppendArgs& a, cudaStream_t stream);
attn_status wait_timeout_check_launch(long long wait_cycles, cudaStream_t stream);
attn_status gen_mask_launch(const int32_t* cache_len, int b, int hq, int s_active, int max_len,
                            uint8_t* mask, cudaStream_t stream);

// Read and clear each translation unit's device error word (bits of attn::kDevErr*).
unsigned prefill_take_error(cudaStream_t stream, cudaError_t* err);
unsigned decode_take_error(cudaStream_t stream, cudaError_t* err);

}  // namespace attn
