// api.cu -- the extern "C" entry points of attn.h: host-side argument checks, workspace
// carving, and dispatch to the kernel translation units.  Nothing here allocates device
// memory or touches tensor contents.
#include <math.h>
#include <algorithm>
#include <stdio.h>

#include "attn_internal.h"

namespace attn {

TensorMapEncodeFn tensor_map_encoder() {
    static TensorMapEncodeFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<TensorMapEncodeFn>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

namespace {

bool make_map(CUtensorMapDataType type, CUtensorMap* map, const void* base, int rank,
              const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box) {
    TensorMapEncodeFn enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t d[3], s[2];
    cuuint32_t bx[3], es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
    }
    for (int i = 0; i < rank - 1; ++i) s[i] = strides_bytes[i];
    return enc(map, type, (cuuint32_t)rank, const_cast<void*>(base), d, s, bx, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool make_bf16_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                   const uint64_t* strides_bytes, const uint32_t* box) {
    return make_map(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, map, base, rank, dims, strides_bytes, box);
}

bool make_u8_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box) {
    return make_map(CU_TENSOR_MAP_DATA_TYPE_UINT8, map, base, rank, dims, strides_bytes, box);
}

}  // namespace attn

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// The options of an _ex call (NULL = none set); returns false if a set option is invalid.
struct Opts {
    const float* sink = nullptr;
    bool e4m3 = false;
    float k_scale = 1.f, v_scale = 1.f;
    int window = 0;
    bool circular = false;
    const float* rope = nullptr;
    const int32_t* cu_q = nullptr;
    const int32_t* cu_k = nullptr;
    int nseq = 0;
    void* pws = nullptr;  // packed-prefill work-order scratch
    size_t pws_bytes = 0;
};

bool read_opts(const attn_opts* opts, Opts* o) {
    if (!opts) return true;
    o->sink = opts->sink;
    if (o->sink && !aligned4(o->sink)) return false;
    if (opts->kv_dtype != ATTN_KV_BF16 && opts->kv_dtype != ATTN_KV_E4M3) return false;
    o->e4m3 = opts->kv_dtype == ATTN_KV_E4M3;
    if (o->e4m3) {
        if (!isfinite(opts->k_scale) || !isfinite(opts->v_scale)) return false;
        o->k_scale = opts->k_scale;
        o->v_scale = opts->v_scale;
    }
    if (opts->window < 0 || (opts->circular != 0 && opts->circular != 1)) return false;
    o->window = opts->window;
    o->circular = opts->circular == 1;
    o->rope = opts->rope_inv_freq;
    if (o->rope && !aligned4(o->rope)) return false;
    o->cu_q = opts->cu_seqlens_q;
    o->cu_k = opts->cu_seqlens_k;
    o->nseq = opts->nseq;
    if (o->cu_q || o->cu_k) {
        if (!o->cu_q || !o->cu_k || !aligned4(o->cu_q) || !aligned4(o->cu_k) || o->nseq < 1)
            return false;
    }
    o->pws = opts->prefill_workspace;
    o->pws_bytes = opts->prefill_workspace_bytes;
    if (o->pws && !aligned4(o->pws)) return false;
    return true;
}

size_t prefill_ws_bytes(int sq) { return sq <= 0 ? 0 : (size_t)((sq + 127) / 128) * 4; }

// Paged-cache arguments shared by decode and append.
bool paged_args_ok(int page_size, int num_pages, int max_pages_per_seq, int max_cache_len) {
    if (page_size < 16 || page_size > 256 || (page_size & (page_size - 1)) != 0) return false;
    if (num_pages <= 0 || max_pages_per_seq <= 0) return false;
    return (long long)max_pages_per_seq * page_size >= max_cache_len;
}

bool head_dim_ok(int d) { return d == 64 || d == 128 || d == 256; }

int resolve_chunk(int kv_chunk, int b, int max_cache_len) {
    return kv_chunk == 0 ? attn::default_kv_chunk(b, max_cache_len) : kv_chunk;
}

// Split-KV scratch: partial outputs [rows][slots][d] fp32 (256-byte padded), their (m, l)
// pairs [rows][slots][2] (16-byte padded), then the piece count of every (sequence, kv
// head) pair (b * hq ints, as hkv <= hq).  A CTA of the split pass reads at least kv_chunk
// tokens unless it reads the last ones, so a pair of n tokens meets at most
// ceil(n / kv_chunk) + 1 CTAs: slots = ceil(max_cache_len / kv_chunk) + 1.
bool decode_scratch_sizes(int b, int hq, int s_active, int d, int max_cache_len, int kv_chunk,
                          size_t* o_bytes, size_t* ml_bytes, size_t* np_bytes, int* max_slots) {
    if (b <= 0 || hq <= 0 || s_active <= 0 || !head_dim_ok(d) || max_cache_len <= 0) return false;
    if (kv_chunk < 0 || (kv_chunk % 32) != 0) return false;
    const int chunk = resolve_chunk(kv_chunk, b, max_cache_len);
    const long long slots = (max_cache_len + (long long)chunk - 1) / chunk + 1;
    const long long rows = (long long)b * hq * s_active;
    *max_slots = (int)slots;
    *o_bytes = (size_t)(rows * slots * d * 4);
    *o_bytes = (*o_bytes + 255) & ~(size_t)255;
    *ml_bytes = (size_t)(rows * slots * 2 * 4);
    *ml_bytes = (*ml_bytes + 15) & ~(size_t)15;
    *np_bytes = (size_t)b * hq * 4;
    return true;
}

}  // namespace

extern "C" {

const char* attn_status_string(attn_status s) {
    switch (s) {
        case ATTN_OK: return "ATTN_OK";
        case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
        case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
        case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
        case ATTN_ERR_PAGE_OOB: return "ATTN_ERR_PAGE_OOB";
        case ATTN_ERR_DEVICE_TIMEOUT: return "ATTN_ERR_DEVICE_TIMEOUT";
        case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
        case ATTN_ERR_CACHE_LEN: return "ATTN_ERR_CACHE_LEN";
    }
    return "ATTN_ERR_UNKNOWN";
}

attn_status attn_fwd_prefill_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                                int b, int hq, int hkv, int sq, int skv, int d, float scale,
                                int causal, int window, attn_dtype o_dtype,
                                const attn_opts* opts, void* stream) {
    if (b <= 0 || hq <= 0 || hkv <= 0 || sq < 0 || skv < 0 || window < 0) return ATTN_ERR_INVALID_ARG;
    if (hq % hkv != 0 || !isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (o_dtype != ATTN_BF16 && o_dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
    if (!head_dim_ok(d)) return ATTN_ERR_UNSUPPORTED;
    if (window > 0 && !causal) return ATTN_ERR_UNSUPPORTED;  // the window is chained after causal
    Opts op;
    if (!read_opts(opts, &op)) return ATTN_ERR_INVALID_ARG;
    // prefill reads bf16 K and V and takes its window as an argument; RoPE and a circular
    // cache are decode options
    if (op.e4m3 || op.window != 0 || op.circular || op.rope) return ATTN_ERR_UNSUPPORTED;
    if (op.cu_q && b != 1) return ATTN_ERR_INVALID_ARG;  // packing is along one batch's rows
    if (op.pws && (!op.cu_q || op.pws_bytes < prefill_ws_bytes(sq))) return ATTN_ERR_INVALID_ARG;
    if (sq == 0) return ATTN_OK;
    if (!q || !o || (skv > 0 && (!k || !v))) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(o) || (skv > 0 && (!aligned16(k) || !aligned16(v))))
        return ATTN_ERR_INVALID_ARG;
    if ((long long)b * hq > 0x7fffffffLL || (long long)b * hkv > 0x7fffffffLL)
        return ATTN_ERR_UNSUPPORTED;
    attn::PrefillArgs a{q, k, v, o, lse, b, hq, hkv, sq, skv, d, scale, causal ? 1 : 0, window,
                        o_dtype, op.sink, op.cu_q, op.cu_k, op.nseq, static_cast<int*>(op.pws)};
    return attn::prefill_launch(a, static_cast<cudaStream_t>(stream));
}

attn_status attn_fwd_prefill(const void* q, const void* k, const void* v, void* o, float* lse,
                             int b, int hq, int hkv, int sq, int skv, int d, float scale,
                             int causal, int window, attn_dtype o_dtype, void* stream) {
    return attn_fwd_prefill_ex(q, k, v, o, lse, b, hq, hkv, sq, skv, d, scale, causal, window,
                               o_dtype, nullptr, stream);
}

size_t attn_prefill_workspace_bytes(int sq) { return prefill_ws_bytes(sq); }

size_t attn_decode_workspace_bytes(int b, int hq, int s_active, int d, int max_cache_len,
                                   int kv_chunk) {
    size_t ob, mlb, npb;
    int ms;
    if (!decode_scratch_sizes(b, hq, s_active, d, max_cache_len, kv_chunk, &ob, &mlb, &npb, &ms))
        return 0;
    return ob + mlb + npb;
}

attn_status attn_fwd_decode_ex(const void* q, const void* k_cache, const void* v_cache,
                               const uint32_t* block_table, const int32_t* cache_len, int b,
                               int hq, int hkv, int d, int s_active, int page_size,
                               int max_pages_per_seq, int num_pages, int max_cache_len,
                               float scale, void* o, float* lse, attn_dtype o_dtype, int kv_chunk,
                               const attn_opts* opts, void* workspace, size_t workspace_bytes,
                               void* stream) {
    if (b <= 0 || hq <= 0 || hkv <= 0 || s_active <= 0 || max_cache_len <= 0)
        return ATTN_ERR_INVALID_ARG;
    if (hq % hkv != 0 || !isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (o_dtype != ATTN_BF16 && o_dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
    if (kv_chunk < 0 || kv_chunk % 32 != 0) return ATTN_ERR_INVALID_ARG;
    if (!q || !k_cache || !v_cache || !cache_len || !o) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o))
        return ATTN_ERR_INVALID_ARG;
    if (!head_dim_ok(d)) return ATTN_ERR_UNSUPPORTED;
    if ((hq / hkv) * (long long)s_active > 16) return ATTN_ERR_UNSUPPORTED;
    Opts op;
    if (!read_opts(opts, &op)) return ATTN_ERR_INVALID_ARG;
    if (op.e4m3 && d == 64) return ATTN_ERR_UNSUPPORTED;  // half a 128-byte box per row
    if (op.cu_q || op.pws) return ATTN_ERR_UNSUPPORTED;  // prefill options
    // a circular cache is a flat ring that holds every new token's window
    if (op.circular && (block_table || op.window == 0 ||
                        (long long)op.window + s_active - 1 > max_cache_len || max_cache_len % 32 != 0))
        return ATTN_ERR_INVALID_ARG;
    if (block_table) {
        if (!paged_args_ok(page_size, num_pages, max_pages_per_seq, max_cache_len))
            return ATTN_ERR_INVALID_ARG;
        if ((long long)num_pages * hkv * page_size > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    } else if ((long long)b * hkv * max_cache_len > 0x7fffffffLL) {
        return ATTN_ERR_UNSUPPORTED;
    }
    size_t ob, mlb, npb;
    int max_slots;
    if (!decode_scratch_sizes(b, hq, s_active, d, max_cache_len, kv_chunk, &ob, &mlb, &npb,
                              &max_slots))
        return ATTN_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || workspace_bytes < ob + mlb + npb)
        return ATTN_ERR_WORKSPACE;
    int chunk = resolve_chunk(kv_chunk, b, max_cache_len);
    if (op.window > 0 && !op.circular) {
        // A window that does not wrap bounds the slots any sequence reads: its start is
        // rounded down to a whole tile, so at most window + s_active - 1 + (tile - 1)
        // slots, and no pair has more pieces than that span allows (the partials keep
        // the scratch's layout, with this smaller stride).  With the default kv_chunk the
        // least share of a CTA is the smallest one the scratch's slots still allow for that
        // span, so that short windows of a small batch spread over every CTA.
        const long long span = std::min<long long>(
            max_cache_len, (long long)op.window + s_active - 1 + (attn::kDecodeTile - 1));
        if (kv_chunk == 0) {
            const long long share = (span + max_slots - 2) / (max_slots - 1);  // max_slots >= 2
            chunk = (int)std::max<long long>(attn::kDecodeTile,
                                             (share + attn::kDecodeTile - 1) /
                                                 attn::kDecodeTile * attn::kDecodeTile);
        }
        max_slots = (int)std::min<long long>(max_slots, (span + chunk - 1) / chunk + 1);
    }
    attn::DecodeArgs a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_table = block_table;
    a.cache_len = cache_len;
    a.b = b;
    a.hq = hq;
    a.hkv = hkv;
    a.d = d;
    a.s_active = s_active;
    a.page_size = page_size;
    a.max_pages_per_seq = max_pages_per_seq;
    a.num_pages = num_pages;
    a.max_cache_len = max_cache_len;
    a.scale = scale;
    a.o = o;
    a.lse = lse;
    a.o_dtype = o_dtype;
    a.kv_chunk = chunk;
    a.part_o = static_cast<float*>(workspace);
    a.part_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + ob);
    a.npieces = reinterpret_cast<int*>(static_cast<char*>(workspace) + ob + mlb);
    a.max_slots = max_slots;
    a.sink = op.sink;
    a.kv_e4m3 = op.e4m3 ? 1 : 0;
    a.k_scale = op.k_scale;
    a.v_scale = op.v_scale;
    a.window = op.window;
    a.circular = op.circular ? 1 : 0;
    a.rope_inv_freq = op.rope;
    return attn::decode_launch(a, static_cast<cudaStream_t>(stream));
}

attn_status attn_fwd_decode(const void* q, const void* k_cache, const void* v_cache,
                            const uint32_t* block_table, const int32_t* cache_len, int b, int hq,
                            int hkv, int d, int s_active, int page_size, int max_pages_per_seq,
                            int num_pages, int max_cache_len, float scale, void* o, float* lse,
                            attn_dtype o_dtype, int kv_chunk, void* workspace,
                            size_t workspace_bytes, void* stream) {
    return attn_fwd_decode_ex(q, k_cache, v_cache, block_table, cache_len, b, hq, hkv, d, s_active,
                              page_size, max_pages_per_seq, num_pages, max_cache_len, scale, o,
                              lse, o_dtype, kv_chunk, nullptr, workspace, workspace_bytes, stream);
}

attn_status attn_append_kv(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                           const uint32_t* block_table, const int32_t* cache_len, int b, int hkv,
                           int d, int s_active, int page_size, int max_pages_per_seq,
                           int num_pages, int max_cache_len, const attn_opts* opts, void* stream) {
    if (b <= 0 || hkv <= 0 || s_active <= 0 || max_cache_len <= 0) return ATTN_ERR_INVALID_ARG;
    if (!k_new || !v_new || !k_cache || !v_cache || !cache_len) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return ATTN_ERR_INVALID_ARG;
    if (!head_dim_ok(d)) return ATTN_ERR_UNSUPPORTED;
    Opts op;
    if (!read_opts(opts, &op)) return ATTN_ERR_INVALID_ARG;
    if (op.e4m3) return ATTN_ERR_UNSUPPORTED;  // the append writes bf16 caches
    if (block_table) {
        if (op.circular || !paged_args_ok(page_size, num_pages, max_pages_per_seq, max_cache_len))
            return ATTN_ERR_INVALID_ARG;
        if ((long long)num_pages * hkv * page_size > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    } else if ((long long)b * hkv * max_cache_len > 0x7fffffffLL) {
        return ATTN_ERR_UNSUPPORTED;
    }
    attn::AppendArgs a{k_new, v_new, k_cache, v_cache, block_table, cache_len, b, hkv, d,
                       s_active, block_table ? page_size : 1, max_pages_per_seq, num_pages,
                       max_cache_len, op.circular ? 1 : 0, op.rope};
    return attn::append_launch(a, static_cast<cudaStream_t>(stream));
}

attn_status attn_gen_mask_decode(const int32_t* cache_len, int b, int hq, int s_active,
                                 int max_len, uint8_t* mask_out, void* stream) {
    if (b <= 0 || hq <= 0 || s_active <= 0 || max_len <= 0) return ATTN_ERR_INVALID_ARG;
    if (!cache_len || !mask_out) return ATTN_ERR_INVALID_ARG;
    return attn::gen_mask_launch(cache_len, b, hq, s_active, max_len, mask_out,
                                 static_cast<cudaStream_t>(stream));
}

attn_status attn_check_wait_timeout(long long wait_cycles, void* stream) {
    if (wait_cycles <= 0 || wait_cycles > (1ll << 33)) return ATTN_ERR_INVALID_ARG;
    return attn::wait_timeout_check_launch(wait_cycles, static_cast<cudaStream_t>(stream));
}

attn_status attn_get_device_error(void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e1 = cudaSuccess, e2 = cudaSuccess;
    const unsigned bits = attn::prefill_take_error(st, &e1) | attn::decode_take_error(st, &e2);
    if (e1 != cudaSuccess || e2 != cudaSuccess) return ATTN_ERR_CUDA;
    if (bits & attn::kDevErrTimeout) return ATTN_ERR_DEVICE_TIMEOUT;
    if (bits & attn::kDevErrPageOOB) return ATTN_ERR_PAGE_OOB;
    if (bits & attn::kDevErrCacheLen) return ATTN_ERR_CACHE_LEN;
    return ATTN_OK;
}

}  // extern "C"
