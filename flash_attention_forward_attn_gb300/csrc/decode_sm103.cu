// decode_sm103.cu -- memory-bound decode attention over a flat or paged bf16 KV cache.
//
// Method ("Flash-Attention: Decode (TKG)"): s_active new tokens per sequence attend the
// whole cache; the q-head group of one kv head is flattened into one tile of
// group * s_active <= 16 rows ("GQA / MQA grouped-query broadcast"), so every K/V byte
// is read once per kv head.  The cache axis is split into pieces, each keeping its own
// running max m, sum l and unnormalised output (the online softmax recurrence of
// "Flash-Attention: Context (CTE)", "The online-softmax recurrence"); a second kernel
// merges the pieces by log-sum-exp, i.e. the deferred normalise of the TKG flash path.
//
// GB300 design: one wave of persistent CTAs (as many as the SMs hold) shares the KV tiles
// of all (sequence, kv head) pairs evenly, as one stream; a CTA's run is cut into pieces
// where it crosses from one pair to the next.  One producer thread streams 32-token K and
// V tiles with TMA (128-byte swizzle) into a shared-memory ring under mbarriers, fetching
// each page through the block table ("Paged / block cache"), and prepares each piece's Q
// ahead of it; four consumer warps take alternate tiles, each with its own (m, l, O)
// state, and merge through shared memory at the end of each piece.  The 16-row
// contractions run on the warp MMA (m16n8k16, bf16 in, fp32 accumulate): with 16 rows an
// fp32 FMA path would need more arithmetic than the CUDA cores deliver at HBM speed.
// Slots past cache_len may hold anything: their scores are replaced by -inf (select, so
// NaN never propagates) and their V rows are zeroed in registers before the P.V product.
#include <type_traits>

#include "attn_internal.h"
#include "attn_ptx.cuh"

namespace attn {
namespace {

__device__ unsigned g_decode_error;

constexpr int kConsumers = 4;    // consumer warps
constexpr int kThreads = (kConsumers + 1) * 32;
// Consumer warp w takes tiles w, w + kConsumers, ... and waits on slot i % kStages at the
// phase of tile i; that phase accounting holds only when every slot belongs to one warp.
// So kStages is a multiple of kConsumers: slot s then only ever holds tiles of warp s % kConsumers.
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// The decode mask (TKG "gen_mask_tkg"): type A keeps j < cache_len; type C gives the
// s_active new tokens (the last s_active slots) a lower-triangular block, so new token t
// sees slot j iff j <= cache_len - s_active + t.  Shared by the decode kernel and the
// mask materialiser.
__device__ __forceinline__ bool decode_allowed(int j, int len, int s_active, int t) {
    return j < len && j <= len - s_active + t;
}

// With a window W > 0 new token t also needs j >= q_pos - W + 1 (the prefill window band,
// AGENTS "Sliding window"; TKG "gen_mask_tkg" type B is that band at the cache end).
__device__ __forceinline__ bool decode_allowed_w(int j, int len, int s_active, int t, int window) {
    return decode_allowed(j, len, s_active, t) && (window == 0 || j >= len - s_active + t - window + 1);
}

// Cache slots of a sequence and the first one any new token may read.  A flat or paged
// cache keeps logical position j in slot j.  A circular flat cache of max_cache_len rows
// keeps it in row j mod max_cache_len, so only min(len, max_cache_len) slots were ever
// written and every one is read (the window covers nearly all of them).  Otherwise tiles
// before the earliest window start are skipped (the start is rounded down to a whole tile
// of gran tokens, the kernel's tile: a power of two).
__device__ __forceinline__ int decode_nslots(int len, int circular, int max_cache_len) {
    return circular ? min(len, max_cache_len) : len;
}
__device__ __forceinline__ int decode_first_slot(int len, int s_active, int window, int circular,
                                                 int gran) {
    return (window > 0 && !circular) ? (max(0, len - s_active - window + 1) & ~(gran - 1)) : 0;
}

// Programmatic dependent launch: a grid lets its stream successor (launched with
// programmatic stream serialisation) start, and that successor waits for its predecessor
// grid to complete, with its memory visible, before it reads the predecessor's output.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Logical position held by slot r of a circular cache of cap rows whose newest position
// is len - 1 (r < min(len, cap)).
__device__ __forceinline__ int circular_pos(int r, int len, int cap) {
    return r + cap * ((len - 1 - r) / cap);
}

// RoPE of the element pairs (i, i + d/2) and (i + 1, i + 1 + d/2) held as bf16 pairs
// lo = (x_i, x_i+1) and hi = (x_i+d/2, x_i+1+d/2), at position pos, half-split form
// ("Flash-Attention: Decode (TKG)", "Algorithm", step 0): theta = pos * inv_freq[i],
//   x_i' = x_i cos theta - x_{i+d/2} sin theta,  x_{i+d/2}' = x_{i+d/2} cos theta + x_i sin theta.
// theta is reduced modulo 2 pi in fp32 by Cody and Waite's additive reduction: pos * f
// is held exactly as hi + lo (an FMA gives the product's rounding error; pos < 2^24 is
// exact in fp32), and 2 pi is taken off k times in two pieces, the first with 8
// significant bits so that k * piece is exact while |k| < 2^16.  The error stays near
// 1e-5 rad.  Larger angles (beyond 2^18 rad, rare) are reduced in double.  The reduced
// angle (|r| <= pi + 1e-5) goes to the hardware sine and cosine (__sincosf, absolute error
// about 5e-7 there).
__device__ __forceinline__ void rope_sincos(int pos, float f, float& sn, float& cs) {
    const float x = (float)pos;
    const float hi = x * f;
    if (fabsf(hi) < 262144.f && pos < (1 << 24)) {
        const float lo = fmaf(x, f, -hi);
        constexpr float kInvTwoPi = 0.15915494309189535f;
        constexpr float kC1 = 6.28125f;               // 201 / 32
        constexpr float kC2 = 1.9353071795864769e-3f;  // 2 pi - kC1
        const float k = rintf(hi * kInvTwoPi);
        const float r = (fmaf(-k, kC1, hi) - k * kC2) + lo;
        __sincosf(r, &sn, &cs);
        return;
    }
    constexpr double kTwoPi = 6.283185307179586;
    double th = (double)pos * (double)f;
    th -= kTwoPi * rint(th * (1.0 / kTwoPi));
    __sincosf((float)th, &sn, &cs);
}
// The rotation of two pairs by the angles (s0, c0) and (s1, c1).
__device__ __forceinline__ void rope_apply(uint32_t& lo, uint32_t& hi, float s0, float c0,
                                           float s1, float c1) {
    const float a0 = __uint_as_float(lo << 16), a1 = __uint_as_float(lo & 0xffff0000u);
    const float b0 = __uint_as_float(hi << 16), b1 = __uint_as_float(hi & 0xffff0000u);
    lo = pack_bf16(a0 * c0 - b0 * s0, a1 * c1 - b1 * s1);
    hi = pack_bf16(b0 * c0 + a0 * s0, b1 * c1 + a1 * s1);
}

// Rows a (position pa) and b (position pb) of a lane, elements i and i + 1 of each:
// the angles are computed once when the two rows share a position.  inv_freq is the
// CTA's shared-memory copy of the inverse frequencies.
__device__ __forceinline__ void rope_rows(uint32_t& alo, uint32_t& ahi, uint32_t& blo,
                                          uint32_t& bhi, int i, int pa, int pb,
                                          const float* inv_freq) {
    const float f0 = inv_freq[i], f1 = inv_freq[i + 1];
    float s0, c0, s1, c1;
    rope_sincos(pa, f0, s0, c0);
    rope_sincos(pa, f1, s1, c1);
    rope_apply(alo, ahi, s0, c0, s1, c1);
    if (pb != pa) {
        rope_sincos(pb, f0, s0, c0);
        rope_sincos(pb, f1, s1, c1);
    }
    rope_apply(blo, bhi, s0, c0, s1, c1);
}

// A K (or V) tile of a slot is kBoxes column boxes of kBT rows x 128 bytes (64 bf16 or 128
// e4m3 head dims per box), each written by TMA with the 128-byte swizzle.
template <int D, bool kE4M3>
struct DecodeLayout {
    // Tokens per tile.  (64-token e4m3 tiles, one 16 KB slot per consumer warp, measured
    // 0.67x the rate of 32-token tiles in two 8 KB slots: a warp then cannot compute one tile
    // while the next one loads.)
    static constexpr int kBT = kDecodeTile;
    // Ring slots.  A CTA keeps kStages tiles in flight; with two CTAs per SM (registers) the
    // bf16 ring of 4 x 16 KB keeps HBM near its copy rate, and the e4m3 ring, with tiles half
    // as large, takes 8 slots (two per consumer warp) to keep the same bytes in flight.
    static constexpr int kStages = kE4M3 ? 8 : 4;
    static_assert(kStages % kConsumers == 0, "each ring slot belongs to one consumer warp");
    static constexpr int kElemBytes = kE4M3 ? 1 : 2;
    static constexpr int kBoxBytes = kBT * 128;
    static constexpr int kBoxElems = 128 / kElemBytes;
    static constexpr int kBoxes = D * kElemBytes / 128;
    static_assert(kBoxes >= 1 && D * kElemBytes == kBoxes * 128, "whole 128-byte box columns");
    static constexpr int kHalf = kBoxes * kBoxBytes;    // K (or V) tile of one slot
    static constexpr int kSlot = 2 * kHalf;
    static constexpr int kPipe = kStages * kSlot;
    // The Q fragments of a piece (identical in every consumer warp) live in shared memory,
    // 16 bytes per lane and k-step, read back per k-step, instead of D/4 registers per
    // thread: with head_dim 256 they would not fit beside the 16 x 256 O, and with head_dim
    // <= 128 the freed registers let three CTAs share an SM (measured on the 1- and 4-token
    // decodes of 64 sequences: bf16 6436 -> 6750 and 6141 -> 6391 GB/s, e4m3 4725 -> 5505
    // and 4394 -> 5041 GB/s, against two CTAs per SM with Q in registers).  Two slots: the
    // producer prepares the next piece's Q while the consumers work on this one, and a
    // finished piece's slot (32 D bytes, half of one warp's O) carries the piece's merge.
    static constexpr int kQSmem = (D / 16) * 32 * 16;
    static constexpr int kDynBytes = kPipe + 2 * kQSmem + 1024;  // + alignment slack
    static constexpr int kMinCtas = D > 128 ? 1 : 3;  // CTAs per SM the registers are fitted to
    // dynamic + static (barriers, piece records, merge maxima, inverse frequencies: under
    // 1.5 KB) + the 1 KB the SM reserves per CTA, within the SM's 228 KB
    static_assert(kMinCtas * (kDynBytes + 1536 + 1024) <= 233472, "shared memory of kMinCtas CTAs");
};

struct DecodeParams {
    const __nv_bfloat16* q;
    const uint32_t* table;
    const int32_t* cache_len;
    float* part_o;   // [b*hq*s_active][max_slots][d]: one partial per piece of a pair
    float* part_ml;  // [b*hq*s_active][max_slots][2]
    int* npieces;    // [b*hkv]: pieces written for each (sequence, kv head)
    int b, hq, hkv, s_active, page_size, max_pages, num_pages, max_cache_len;
    int group, rows, min_tiles, max_slots, paged, box_rows;
    int window, circular;    // decode window (0 = none); circular flat cache
    const float* rope_inv_freq;  // [d/2] RoPE inverse frequencies of Q, or NULL
    float c;        // scale * log2(e) (* k_scale for an e4m3 cache)
    float v_scale;  // V dequantisation scale of an e4m3 cache (1 for bf16)
};

__device__ __forceinline__ bool mbar_wait_plain(uint64_t* bar, uint32_t parity,
                                                long long limit) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > limit) return false;
    return true;
}

// Tiles that every kv head of sequence b reads: 0 for a cache_len out of range (the merge
// reports it).
__device__ __forceinline__ int pair_tiles(const DecodeParams& p, int b) {
    const int len = __ldg(p.cache_len + b);
    if (len < p.s_active || (!p.circular && len > p.max_cache_len)) return 0;
    const int first = decode_first_slot(len, p.s_active, p.window, p.circular, kDecodeTile);
    return (decode_nslots(len, p.circular, p.max_cache_len) - first + kDecodeTile - 1) /
           kDecodeTile;
}

// True in every consumer thread when pred holds in any of them (a barrier of the consumer
// warps with an OR reduction: they all take the same branch after it).
__device__ __forceinline__ bool consumers_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
        " bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((uint32_t)pred), "n"(kConsumers * 32)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
}

// One piece: the tiles of one (sequence, kv head) pair that a CTA reads, handed from the
// producer to the consumers with the piece's Q fragments.
struct PieceInfo {
    int b, g, len, nslots, first;  // sequence, kv head, cache length, slots [first, nslots)
    int t_off;  // the pair's tile index of the piece's first tile
    int npc;    // tiles in the piece; 0 ends the CTA's work
    int i0;     // ring index of the piece's first tile
    int k;      // the piece's index within its pair: its partial slot
    float c_row[16];  // softmax scale of each row (log2 units)
};

// kE4M3: the cache holds e4m3 bytes.  k_scale is folded into p.c and v_scale applied to the
// piece's output, so the products run on the exact e4m3 values, converted to f16 (one
// instruction per pair): Q.K^T with Q in f16 and P.V with P in f16.  Each Q row is scaled by
// a power of two that puts its largest |element| in [2^13, 2^14) before it is rounded to
// f16 (the factor comes back out of the row's softmax scale), so the f16 row holds every
// bf16 element exactly unless it is below 2^-27 of the row's largest.
//
// Work split: the KV tiles of all (sequence, kv head) pairs, sequence-major, form one
// stream of NT tiles; CTA c of the grid takes tiles [c tpc, (c + 1) tpc) with
// tpc = max(ceil(NT / gridDim.x), min_tiles).  The grid is one wave (the CTAs the SMs hold),
// so every CTA streams the same number of bytes and pays its start-up once.  The run of a
// CTA is cut into pieces at pair boundaries; each piece keeps its own (m, l, O) and writes
// one partial.  A pair of n tiles meets at most ceil(n / min_tiles) + 1 CTAs, which bounds
// the partial slots a pair needs.
template <int D, bool kE4M3>
__global__ void __launch_bounds__(kThreads, DecodeLayout<D, kE4M3>::kMinCtas) decode_split_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const DecodeParams p) {
    using L = DecodeLayout<D, kE4M3>;
    constexpr int kStages = L::kStages;
    constexpr int kBT = L::kBT;
    constexpr int kQWords = (D / 16) * 32;  // uint4 words of one Q slot
    extern __shared__ uint8_t dyn_smem[];
    uint8_t* pipe = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    uint4* const qslots = reinterpret_cast<uint4*>(pipe + L::kPipe);  // [2][kQWords]
    __shared__ uint64_t full_bar[kStages], empty_bar[kStages], q_full[2], q_empty[2];
    __shared__ PieceInfo info[2];
    __shared__ float m_sh[kConsumers][16], l_sh[kConsumers][16];
    __shared__ float inv_freq[D / 2];  // RoPE inverse frequencies (producer only)
    // head_dim 256: row r's new token (r mod s_active), which the masked tiles read here
    // rather than keep in registers; the consumers sit at the 255-register ceiling there, and
    // this is what keeps them from spilling (8 bytes with the tokens in registers)
    __shared__ int row_tok[16];
    __shared__ int abort_flag;

    // The merge kernel is launched as this grid's programmatic dependent: it may take free
    // slots once every CTA here has started (or exited), and waits for this grid to finish
    // before it reads a partial.
    griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, qd = lane & 3;
    const int r0 = gq, r1 = gq + 8;
    const bool v0 = r0 < p.rows, v1 = r1 < p.rows;
    const int t0 = r0 % p.s_active, t1 = r1 % p.s_active;

    if constexpr (D > 128)
        if (threadIdx.x < 16) row_tok[threadIdx.x] = (int)threadIdx.x % p.s_active;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&q_full[s], 1);
            mbar_init(&q_empty[s], kConsumers);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // ------------------------------------------------------------------ producer
    if (warp == kConsumers) {
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
        }
        // the inverse frequencies once per CTA: each piece's RoPE then waits on no global load
        if (p.rope_inv_freq != nullptr)
            for (int i = lane; i < D / 2; i += 32) inv_freq[i] = __ldg(p.rope_inv_freq + i);
        __syncwarp();
        const int nbox = kBT / p.box_rows;
        const uint32_t box_bytes = (uint32_t)p.box_rows * 128u;
        int issued = 0;
        bool ok = true;

        // Tiles [x0, x1) of a piece of pair (b, g) whose first tile is the pair's tile
        // t_off, at ring index i0 + x.  The rows of 32 tiles are found at once, one tile per
        // lane (a paged cache costs a dependent block-table load per tile, which one thread
        // would pay tile after tile); lane 0 then issues the tiles in order.
        auto issue = [&](int b, int g, int first, int nslots, int t_off, int i0, int x0,
                         int x1) {
            for (int xb = x0; ok && xb < x1; xb += 32) {
                int rl[kBT / 16];  // lane's tile xb + lane: cache row of each box, -1 = not read
#pragma unroll
                for (int bx = 0; bx < kBT / 16; ++bx) {
                    rl[bx] = -1;
                    const int jb = first + (t_off + xb + lane) * kBT + bx * p.box_rows;
                    // a box wholly past the cache end is not read
                    if (bx >= nbox || xb + lane >= x1 || jb >= nslots) continue;
                    if (p.paged) {
                        const uint32_t pg =
                            __ldg(p.table + (size_t)b * p.max_pages + jb / p.page_size);
                        if (pg >= (uint32_t)p.num_pages) {
                            atomicOr(&g_decode_error, kDevErrPageOOB);
                            continue;  // never dereference an out-of-range page
                        }
                        rl[bx] = (int)(((long long)pg * p.hkv + g) * p.page_size + jb % p.page_size);
                    } else {
                        rl[bx] = (int)(((long long)b * p.hkv + g) * p.max_cache_len + jb);
                    }
                }
                const int n = min(32, x1 - xb);
                for (int t = 0; t < n; ++t) {
                    int rows[kBT / 16];
#pragma unroll
                    for (int bx = 0; bx < kBT / 16; ++bx) rows[bx] = __shfl_sync(0xffffffffu, rl[bx], t);
                    if (lane == 0) {
                        const int i = i0 + xb + t;
                        const int s = i % kStages;
                        if (i >= kStages &&
                            !mbar_wait(&empty_bar[s], ((i / kStages) - 1) & 1, &abort_flag)) {
                            ok = false;
                        } else {
                            uint32_t bytes = 0;
#pragma unroll
                            for (int bx = 0; bx < kBT / 16; ++bx)
                                if (bx < nbox && rows[bx] >= 0) bytes += 2u * (uint32_t)L::kBoxes * box_bytes;
                            uint8_t* kdst = pipe + s * L::kSlot;
                            uint8_t* vdst = kdst + L::kHalf;
                            mbar_arrive_expect_tx(&full_bar[s], bytes);
#pragma unroll
                            for (int bx = 0; bx < kBT / 16; ++bx) {
                                if (bx >= nbox || rows[bx] < 0) continue;
#pragma unroll
                                for (int dc = 0; dc < L::kBoxes; ++dc) {
                                    tma_load_2d(kdst + dc * L::kBoxBytes + bx * box_bytes, &tm_k,
                                                dc * L::kBoxElems, rows[bx], &full_bar[s]);
                                    tma_load_2d(vdst + dc * L::kBoxBytes + bx * box_bytes, &tm_v,
                                                dc * L::kBoxElems, rows[bx], &full_bar[s]);
                                }
                            }
                            issued = i + 1;
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                }
            }
        };

        // Q slot j % 2 may be refilled once the consumers have merged piece j - 2.
        auto q_slot_free = [&](int j) {
            if (j < 2) return;
            bool w = true;
            if (lane == 0) w = mbar_wait(&q_empty[j & 1], ((j >> 1) - 1) & 1, &abort_flag);
            ok = ok && __shfl_sync(0xffffffffu, w, 0);
        };

        // The Q fragments of pair (b, g) in the consumers' lane layout (16 bytes per lane and
        // k-step), and each row's softmax scale.
        auto prep_q = [&](int b, int g, int len, uint4* qs, float* c_row) {
            const int qpos0 = len - p.s_active + t0, qpos1 = len - p.s_active + t1;  // RoPE positions
            const __nv_bfloat16* q0 = nullptr;
            const __nv_bfloat16* q1 = nullptr;
            if (v0) q0 = p.q + ((size_t)(b * p.hq + g * p.group + r0 / p.s_active) * p.s_active + t0) * D;
            if (v1) q1 = p.q + ((size_t)(b * p.hq + g * p.group + r1 / p.s_active) * p.s_active + t1) * D;
            uint32_t qf[D / 16][4];
            float c_row0 = p.c, c_row1 = p.c;
            if constexpr (kE4M3) {
                // The k index of k-step ks maps 2qd, 2qd+1 to head dims 16 ks + 4 qd + {0, 1} and
                // 2qd+8, 2qd+9 to 16 ks + 4 qd + {2, 3} (a dot product does not depend on the
                // order of its terms): one 32-bit shared load then gives a lane the four K bytes
                // of its k-step.
                uint2 qa[D / 16], qb[D / 16];
                float mx_a = 0.f, mx_b = 0.f;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int c = ks * 16 + 4 * qd;
                    qa[ks] = v0 ? __ldg(reinterpret_cast<const uint2*>(q0 + c)) : make_uint2(0u, 0u);
                    qb[ks] = v1 ? __ldg(reinterpret_cast<const uint2*>(q1 + c)) : make_uint2(0u, 0u);
                }
                if (p.rope_inv_freq != nullptr) {  // element i of k-step ks pairs with k-step ks + D/32
#pragma unroll
                    for (int ks = 0; ks < D / 32; ++ks) {
                        const int c = ks * 16 + 4 * qd;
                        rope_rows(qa[ks].x, qa[ks + D / 32].x, qb[ks].x, qb[ks + D / 32].x, c, qpos0,
                                  qpos1, inv_freq);
                        rope_rows(qa[ks].y, qa[ks + D / 32].y, qb[ks].y, qb[ks + D / 32].y, c + 2,
                                  qpos0, qpos1, inv_freq);
                    }
                }
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t wa[2] = {qa[ks].x, qa[ks].y}, wb[2] = {qb[ks].x, qb[ks].y};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const uint32_t ba = (h & 1) ? (wa[h >> 1] & 0xffff0000u) : (wa[h >> 1] << 16);
                        const uint32_t bb = (h & 1) ? (wb[h >> 1] & 0xffff0000u) : (wb[h >> 1] << 16);
                        mx_a = fmaxf(mx_a, fabsf(__uint_as_float(ba)));
                        mx_b = fmaxf(mx_b, fabsf(__uint_as_float(bb)));
                    }
                }
                mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
                mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
                // power-of-two row factors 2^sa, 2^sb: the largest |q| lands in [2^13, 2^14)
                int ea = 0, eb = 0;
                if (mx_a > 0.f) frexpf(mx_a, &ea);  // mx in [2^(ea-1), 2^ea)
                if (mx_b > 0.f) frexpf(mx_b, &eb);
                const int sa = mx_a > 0.f ? 14 - ea : 0, sb = mx_b > 0.f ? 14 - eb : 0;
                c_row0 = ldexpf(p.c, -sa);
                c_row1 = ldexpf(p.c, -sb);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t wa[2] = {qa[ks].x, qa[ks].y}, wb[2] = {qb[ks].x, qb[ks].y};
                    uint32_t fa[2], fb[2];
#pragma unroll
                    for (int w2 = 0; w2 < 2; ++w2) {
                        fa[w2] = pack_f16(ldexpf(__uint_as_float(wa[w2] << 16), sa),
                                          ldexpf(__uint_as_float(wa[w2] & 0xffff0000u), sa));
                        fb[w2] = pack_f16(ldexpf(__uint_as_float(wb[w2] << 16), sb),
                                          ldexpf(__uint_as_float(wb[w2] & 0xffff0000u), sb));
                    }
                    qf[ks][0] = fa[0];
                    qf[ks][2] = fa[1];
                    qf[ks][1] = fb[0];
                    qf[ks][3] = fb[1];
                }
            } else {
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int c = ks * 16 + 2 * qd;
                    qf[ks][0] = v0 ? __ldg(reinterpret_cast<const uint32_t*>(q0 + c)) : 0u;
                    qf[ks][1] = v1 ? __ldg(reinterpret_cast<const uint32_t*>(q1 + c)) : 0u;
                    qf[ks][2] = v0 ? __ldg(reinterpret_cast<const uint32_t*>(q0 + c + 8)) : 0u;
                    qf[ks][3] = v1 ? __ldg(reinterpret_cast<const uint32_t*>(q1 + c + 8)) : 0u;
                }
                if (p.rope_inv_freq != nullptr) {  // element i of k-step ks pairs with k-step ks + D/32
#pragma unroll
                    for (int ks = 0; ks < D / 32; ++ks) {
                        const int c = ks * 16 + 2 * qd;
                        rope_rows(qf[ks][0], qf[ks + D / 32][0], qf[ks][1], qf[ks + D / 32][1], c,
                                  qpos0, qpos1, inv_freq);
                        rope_rows(qf[ks][2], qf[ks + D / 32][2], qf[ks][3], qf[ks + D / 32][3], c + 8,
                                  qpos0, qpos1, inv_freq);
                    }
                }
            }
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                qs[ks * 32 + lane] = make_uint4(qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
            if (qd == 0) {
                c_row[r0] = c_row0;
                c_row[r1] = c_row1;
            }
        };

        // NT, the tiles of every pair, and this CTA's run [lo, hi) of them
        long long cnt = 0;
        for (int bb = lane; bb < p.b; bb += 32) cnt += pair_tiles(p, bb);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        const long long nt_all = cnt * p.hkv;
        const long long tpc =
            max((nt_all + gridDim.x - 1) / (long long)gridDim.x, (long long)p.min_tiles);
        const long long lo = (long long)blockIdx.x * tpc;
        const long long hi = min(nt_all, lo + tpc);
        int j = 0;  // pieces handed to the consumers
        if (lo < hi) {
            // the sequence holding tile lo: 32 sequences at a time, by a prefix sum over lanes
            int bcur = -1;
            long long bstart = 0, base = 0;
            for (int bb0 = 0; bb0 < p.b; bb0 += 32) {
                const int bb = bb0 + lane;
                const long long t = bb < p.b ? (long long)pair_tiles(p, bb) * p.hkv : 0;
                long long incl = t;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const long long y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                const long long excl = incl - t;
                const unsigned hit =
                    __ballot_sync(0xffffffffu, t > 0 && lo >= base + excl && lo < base + incl);
                if (hit != 0u) {
                    const int l0 = __ffs(hit) - 1;
                    bcur = bb0 + l0;
                    bstart = base + __shfl_sync(0xffffffffu, excl, l0);
                    break;
                }
                base += __shfl_sync(0xffffffffu, incl, 31);
            }
            int nt_b = bcur >= 0 ? pair_tiles(p, bcur) : 0;
            if (nt_b <= 0) ok = false;  // cannot happen: lo < NT lies in some sequence
            int gcur = ok ? (int)((lo - bstart) / nt_b) : 0;
            int t_off = ok ? (int)((lo - bstart) % nt_b) : 0;
            long long pstart = bstart + (long long)gcur * nt_b;  // stream index of the pair's first tile
            int i = 0;  // ring index of the next tile
            const int total = (int)(hi - lo);
            while (ok && i < total) {
                const int npc = min(nt_b - t_off, total - i);
                const int k = (int)(blockIdx.x - pstart / tpc);
                const int len = __ldg(p.cache_len + bcur);
                const int nslots = decode_nslots(len, p.circular, p.max_cache_len);
                const int first = decode_first_slot(len, p.s_active, p.window, p.circular, kBT);
                // The first piece's tiles start loading before its Q is prepared; later
                // pieces are prepared while the ring still holds the previous piece.
                const int pre = (j == 0) ? min(npc, kStages) : 0;
                issue(bcur, gcur, first, nslots, t_off, i, 0, pre);
                q_slot_free(j);
                if (!ok) break;
                PieceInfo& pi = info[j & 1];
                prep_q(bcur, gcur, len, qslots + (j & 1) * kQWords, pi.c_row);
                if (lane == 0) {
                    pi.b = bcur;
                    pi.g = gcur;
                    pi.len = len;
                    pi.nslots = nslots;
                    pi.first = first;
                    pi.t_off = t_off;
                    pi.npc = npc;
                    pi.i0 = i;
                    pi.k = k;
                    // the CTA that reads a pair's last tile records how many pieces it has
                    if (t_off + npc == nt_b) p.npieces[(size_t)bcur * p.hkv + gcur] = k + 1;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&q_full[j & 1]);
                issue(bcur, gcur, first, nslots, t_off, i, pre, npc);
                i += npc;
                ++j;
                t_off = 0;  // the next pair
                pstart += nt_b;
                if (++gcur == p.hkv) {
                    gcur = 0;
                    nt_b = 0;
                    while (nt_b == 0 && ++bcur < p.b) nt_b = pair_tiles(p, bcur);
                    if (nt_b == 0 && i < total) ok = false;  // cannot happen: tiles remain
                }
            }
        }
        // the end of this CTA's work
        if (ok) q_slot_free(j);
        if (ok) {
            if (lane == 0) info[j & 1].npc = 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_full[j & 1]);
        } else if (lane == 0) {
            abort_flag = 1;  // the consumers stop at their next wait
        }
        if (lane == 0 && abort_flag) {  // let copies already in flight land before the CTA exits
            for (int i = max(0, issued - kStages); i < issued; ++i)
                mbar_wait_plain(&full_bar[i % kStages], (i / kStages) & 1, kWaitLimitCycles);
            atomicOr(&g_decode_error, kDevErrTimeout);
        }
    } else {
        // -------------------------------------------------------------- consumers
        constexpr int kNT = kBT / 8;  // 8-token n-tiles of S per tile
        for (int j = 0;; ++j) {
            const int qsl = j & 1;
            const bool got = __all_sync(0xffffffffu, mbar_wait(&q_full[qsl], (j >> 1) & 1, &abort_flag));
            if (consumers_any(!got || abort_flag != 0)) break;
            const PieceInfo& pi = info[qsl];
            const int npc = pi.npc;
            if (npc == 0) break;  // the same value in every consumer warp
            const int len = pi.len, nslots = pi.nslots, first = pi.first;
            const int t_off = pi.t_off, i0 = pi.i0;
            const float c_row0 = pi.c_row[r0], c_row1 = pi.c_row[r1];
            const uint4* const qs = qslots + qsl * kQWords;
            auto qfrag = [&](int ks, uint32_t* f) {
                const uint4 x = qs[ks * 32 + lane];
                f[0] = x.x;
                f[1] = x.y;
                f[2] = x.z;
                f[3] = x.w;
            };
            float o[D / 8][4];
#pragma unroll
            for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
            float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

            // this warp's tiles of the piece: ring indices i = warp (mod kConsumers)
            for (int i = i0 + (warp - i0 % kConsumers + kConsumers) % kConsumers; i < i0 + npc;
                 i += kConsumers) {
                const int s = i % kStages;
                if (!__all_sync(0xffffffffu, mbar_wait(&full_bar[s], (i / kStages) & 1, &abort_flag)))
                    break;
                const uint32_t kbase = smem_u32(pipe + s * L::kSlot);
                const uint32_t vbase = kbase + L::kHalf;
                // S = Q K^T for 16 rows x kBT tokens
                float sc[kNT][4];
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
                if constexpr (kE4M3) {
                    // token nt*8 + gq, head dims 16 ks + 4 qd .. +3 (chunk ks of its 128-byte row)
                    const uint8_t* kt = pipe + s * L::kSlot;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        uint32_t qk[4];
                        qfrag(ks, qk);
#pragma unroll
                        for (int nt = 0; nt < kNT; ++nt) {
                            const int tok = nt * 8 + gq;
                            const uint32_t w = *reinterpret_cast<const uint32_t*>(
                                kt + (ks >> 3) * L::kBoxBytes + sw128_off(tok, ks & 7) + 4 * qd);
                            mma_f16_16816(sc[nt], qk, e4m3x2_to_f16x2(w & 0xffffu),
                                          e4m3x2_to_f16x2(w >> 16));
                        }
                    }
                } else {
#pragma unroll
                    for (int kp = 0; kp < D / 32; ++kp) {
                        uint32_t qa[4], qb[4];
                        qfrag(2 * kp, qa);
                        qfrag(2 * kp + 1, qb);
#pragma unroll
                        for (int nt = 0; nt < kNT; ++nt) {
                            const uint32_t tok = nt * 8 + (lane & 7);
                            const uint32_t cg = 4 * kp + (lane >> 3);
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4(kbase + (cg >> 3) * L::kBoxBytes + sw128_off(tok, cg & 7), b0, b1, b2, b3);
                            mma_bf16_16816(sc[nt], qa, b0, b1);
                            mma_bf16_16816(sc[nt], qb, b2, b3);
                        }
                    }
                }
                const int j0 = first + (t_off + (i - i0)) * kBT;  // first slot of the tile
                // tiles that touch the new tokens, the cache end or a window start are masked;
                // every tile of a circular cache is (its slots hold positions of two laps)
                const bool edge = p.circular || j0 + kBT > len - p.s_active ||
                                  (p.window > 0 && j0 < len - p.window);
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float x0 = sc[nt][e] * c_row0, x1 = sc[nt][2 + e] * c_row1;
                        if (edge) {
                            const int r = j0 + nt * 8 + 2 * qd + e;  // slot
                            const int j = p.circular ? circular_pos(r, len, p.max_cache_len) : r;
                            const bool in = r < nslots;
                            const int u0 = D > 128 ? row_tok[r0] : t0, u1 = D > 128 ? row_tok[r1] : t1;
                            if (!(v0 && in && decode_allowed_w(j, len, p.s_active, u0, p.window))) x0 = -INFINITY;
                            if (!(v1 && in && decode_allowed_w(j, len, p.s_active, u1, p.window))) x1 = -INFINITY;
                        }
                        sc[nt][e] = x0;
                        sc[nt][2 + e] = x1;
                        mx0 = fmaxf(mx0, x0);
                        mx1 = fmaxf(mx1, x1);
                    }
                }
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
                // a row with nothing allowed yet keeps exponent base 0: exp2(-inf - 0) = 0
                const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0;
                const float mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
                const float a0 = ex2(m_run[0] - mu0), a1 = ex2(m_run[1] - mu1);
                m_run[0] = mn0;
                m_run[1] = mn1;
                l_run[0] *= a0;
                l_run[1] *= a1;
#pragma unroll
                for (int n = 0; n < D / 8; ++n) {
                    o[n][0] *= a0;
                    o[n][1] *= a0;
                    o[n][2] *= a1;
                    o[n][3] *= a1;
                }
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt) {
                    sc[nt][0] = ex2(sc[nt][0] - mu0);
                    sc[nt][1] = ex2(sc[nt][1] - mu0);
                    sc[nt][2] = ex2(sc[nt][2] - mu1);
                    sc[nt][3] = ex2(sc[nt][3] - mu1);
                    l_run[0] += sc[nt][0] + sc[nt][1];
                    l_run[1] += sc[nt][2] + sc[nt][3];
                }
                // O += P V (P from the score accumulators)
#pragma unroll
                for (int ks = 0; ks < kBT / 16; ++ks) {
                    uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;
                    if (edge) {  // zero V rows of slots past the cache end (they may hold NaN)
                        const int jl = j0 + ks * 16 + 2 * qd;
                        keep_lo = (jl < nslots ? 0x0000ffffu : 0u) | (jl + 1 < nslots ? 0xffff0000u : 0u);
                        keep_hi = (jl + 8 < nslots ? 0x0000ffffu : 0u) | (jl + 9 < nslots ? 0xffff0000u : 0u);
                    }
                    uint32_t pa[4];
                    if constexpr (kE4M3) {
                        // P in f16, V converted to f16.  The n index of n-tile np maps n to head
                        // dim (D/8) n + np, so a lane (n = gq) reads D/8 consecutive bytes of each
                        // of its four tokens (k = 2qd, 2qd+1, 2qd+8, 2qd+9) and pairs them bytewise.
                        pa[0] = pack_f16(sc[2 * ks][0], sc[2 * ks][1]);
                        pa[1] = pack_f16(sc[2 * ks][2], sc[2 * ks][3]);
                        pa[2] = pack_f16(sc[2 * ks + 1][0], sc[2 * ks + 1][1]);
                        pa[3] = pack_f16(sc[2 * ks + 1][2], sc[2 * ks + 1][3]);
                        constexpr int kW = D / 32;  // 32-bit words of a lane's bytes per token
                        const uint8_t* vt = pipe + s * L::kSlot + L::kHalf;
                        const int ta = ks * 16 + 2 * qd;
                        uint32_t vw[4][kW];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const int tok = ta + (r & 1) + (r >> 1) * 8;
#pragma unroll
                            for (int c = 0; c < kW / 4; ++c) {
                                const int ch = (D / 128) * gq + c;  // 16-byte chunk along the row
                                const uint4 x = *reinterpret_cast<const uint4*>(
                                    vt + (ch >> 3) * L::kBoxBytes + sw128_off(tok, ch & 7));
                                vw[r][4 * c] = x.x;
                                vw[r][4 * c + 1] = x.y;
                                vw[r][4 * c + 2] = x.z;
                                vw[r][4 * c + 3] = x.w;
                            }
                        }
                        // the keep masks only bite on edge tiles (the choice is per tile, so
                        // warp-uniform): other tiles skip the 64 ANDs
                        auto pv = [&](auto masked) {
#pragma unroll
                            for (int wd = 0; wd < kW; ++wd) {
                                const uint32_t ab0 = __byte_perm(vw[0][wd], vw[1][wd], 0x5140);
                                const uint32_t ab1 = __byte_perm(vw[0][wd], vw[1][wd], 0x7362);
                                const uint32_t cd0 = __byte_perm(vw[2][wd], vw[3][wd], 0x5140);
                                const uint32_t cd1 = __byte_perm(vw[2][wd], vw[3][wd], 0x7362);
                                const uint32_t pairs[4][2] = {{ab0 & 0xffffu, cd0 & 0xffffu},
                                                              {ab0 >> 16, cd0 >> 16},
                                                              {ab1 & 0xffffu, cd1 & 0xffffu},
                                                              {ab1 >> 16, cd1 >> 16}};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    uint32_t b0 = e4m3x2_to_f16x2(pairs[e][0]);
                                    uint32_t b1 = e4m3x2_to_f16x2(pairs[e][1]);
                                    if constexpr (decltype(masked)::value) {
                                        b0 &= keep_lo;
                                        b1 &= keep_hi;
                                    }
                                    mma_f16_16816(o[4 * wd + e], pa, b0, b1);
                                }
                            }
                        };
                        if (edge) pv(std::true_type{});
                        else pv(std::false_type{});
                        continue;
                    }
                    // bf16: V through transposed ldmatrix
                    pa[0] = pack_bf16(sc[2 * ks][0], sc[2 * ks][1]);
                    pa[1] = pack_bf16(sc[2 * ks][2], sc[2 * ks][3]);
                    pa[2] = pack_bf16(sc[2 * ks + 1][0], sc[2 * ks + 1][1]);
                    pa[3] = pack_bf16(sc[2 * ks + 1][2], sc[2 * ks + 1][3]);
#pragma unroll
                    for (int np = 0; np < D / 16; ++np) {
                        const uint32_t mi = lane >> 3;
                        const uint32_t tok = ks * 16 + (mi & 1) * 8 + (lane & 7);
                        const uint32_t cg = 2 * np + (mi >> 1);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(vbase + (cg >> 3) * L::kBoxBytes + sw128_off(tok, cg & 7), b0, b1, b2, b3);
                        b0 &= keep_lo;
                        b2 &= keep_lo;
                        b1 &= keep_hi;
                        b3 &= keep_hi;
                        mma_bf16_16816(o[2 * np], pa, b0, b1);
                        mma_bf16_16816(o[2 * np + 1], pa, b2, b3);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty_bar[s]);
            }
            l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 1);
            l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 2);
            l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 1);
            l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 2);

            // ------------------------------------------------------ the piece's merge
            // Warp 0 gathers the other warps' (m, l, O) through the finished piece's Q slot
            // (32 D bytes: half of one warp's O), one half of one warp at a time, and writes
            // the piece's partial.
            if (qd == 0) {
                m_sh[warp][r0] = m_run[0];
                l_sh[warp][r0] = l_run[0];
                m_sh[warp][r1] = m_run[1];
                l_sh[warp][r1] = l_run[1];
            }
            consumers_sync();
            // merged row maxima (warp 0); a row with nothing allowed keeps exponent base 0
            float mu0 = 0.f, mu1 = 0.f;
            if (warp == 0) {
                float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
                for (int w = 0; w < kConsumers; ++w) {
                    M0 = fmaxf(M0, m_sh[w][r0]);
                    M1 = fmaxf(M1, m_sh[w][r1]);
                }
                mu0 = (M0 == -INFINITY) ? 0.f : M0;
                mu1 = (M1 == -INFINITY) ? 0.f : M1;
                const float w0 = ex2(m_sh[0][r0] - mu0), w1 = ex2(m_sh[0][r1] - mu1);
#pragma unroll
                for (int n = 0; n < D / 8; ++n) {
                    o[n][0] *= w0;
                    o[n][1] *= w0;
                    o[n][2] *= w1;
                    o[n][3] *= w1;
                }
            }
            float* const xb = reinterpret_cast<float*>(qslots + qsl * kQWords);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int w = 1; w < kConsumers; ++w) {
                    if (warp == w) {
#pragma unroll
                        for (int nn = 0; nn < D / 16; ++nn)
#pragma unroll
                            for (int e = 0; e < 4; ++e) xb[(nn * 4 + e) * 32 + lane] = o[h * (D / 16) + nn][e];
                    }
                    consumers_sync();
                    if (warp == 0) {
                        const float w0 = ex2(m_sh[w][r0] - mu0), w1 = ex2(m_sh[w][r1] - mu1);
#pragma unroll
                        for (int nn = 0; nn < D / 16; ++nn)
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                o[h * (D / 16) + nn][e] += (e < 2 ? w0 : w1) * xb[(nn * 4 + e) * 32 + lane];
                    }
                    consumers_sync();
                }
            }
            // the piece's pair and slot, read before the producer may reuse the record
            const int b = pi.b, g = pi.g, k = pi.k;
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_empty[qsl]);  // Q slot, record and merge buffer are free
            if (warp == 0) {
                if (k < 0 || k >= p.max_slots) {
                    // cannot happen while the scratch holds max_slots partials per row: never
                    // write past it
                    if (lane == 0) atomicOr(&g_decode_error, kDevErrTimeout);
                } else {
                    const float vs = kE4M3 ? p.v_scale : 1.f;
                    const size_t row0 = ((size_t)b * p.hq + g * p.group + r0 / p.s_active) * p.s_active + t0;
                    const size_t row1 = ((size_t)b * p.hq + g * p.group + r1 / p.s_active) * p.s_active + t1;
                    float* const po0 = p.part_o + (row0 * p.max_slots + k) * D;
                    float* const po1 = p.part_o + (row1 * p.max_slots + k) * D;
#pragma unroll
                    for (int n = 0; n < D / 8; ++n) {
                        if constexpr (kE4M3) {  // n-tile n holds head dims (D/8) * {2qd, 2qd+1} + n
                            const int d0 = (D / 8) * 2 * qd + n, d1 = d0 + D / 8;
                            if (v0) {
                                po0[d0] = o[n][0] * vs;
                                po0[d1] = o[n][1] * vs;
                            }
                            if (v1) {
                                po1[d0] = o[n][2] * vs;
                                po1[d1] = o[n][3] * vs;
                            }
                        } else {
                            const int col = n * 8 + 2 * qd;
                            if (v0) *reinterpret_cast<float2*>(po0 + col) = make_float2(o[n][0], o[n][1]);
                            if (v1) *reinterpret_cast<float2*>(po1 + col) = make_float2(o[n][2], o[n][3]);
                        }
                    }
                    if (qd == 0) {
                        // (max, sum) of the piece; m_sh is rewritten only after the next
                        // piece's first barrier, which this warp has not reached
                        float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f;
#pragma unroll
                        for (int w = 0; w < kConsumers; ++w) {
                            M0 = fmaxf(M0, m_sh[w][r0]);
                            M1 = fmaxf(M1, m_sh[w][r1]);
                            L0 += ex2(m_sh[w][r0] - mu0) * l_sh[w][r0];
                            L1 += ex2(m_sh[w][r1] - mu1) * l_sh[w][r1];
                        }
                        if (v0) {
                            p.part_ml[(row0 * p.max_slots + k) * 2 + 0] = M0;
                            p.part_ml[(row0 * p.max_slots + k) * 2 + 1] = L0;
                        }
                        if (v1) {
                            p.part_ml[(row1 * p.max_slots + k) * 2 + 0] = M1;
                            p.part_ml[(row1 * p.max_slots + k) * 2 + 1] = L1;
                        }
                    }
                }
            }
        }
    }
}

// Merge the pieces of each (sequence, head, new token) row by log-sum-exp:
//   M = max_i m_i,  L = sum_i 2^(m_i - M) l_i,  O = sum_i 2^(m_i - M) O_i / L,
//   LSE = (M + log2 L) ln 2   (m_i are in log2 units of the scaled scores);
// with a sink, the merged row is finished by finish_row (the sink joins M and L).  One CTA
// per (sequence, kv head): its group * s_active rows share the piece count, and each thread
// merges four columns of a row at a time (16-byte loads of the partials).  The rows of a
// sequence whose cache_len is out of range get O = 0, LSE = -inf and are reported.
constexpr int kMergeThreads = 256;

template <int D, typename OutT>
__global__ void __launch_bounds__(kMergeThreads) decode_combine_kernel(
    const int32_t* __restrict__ cache_len, const float* __restrict__ part_o,
    const float* __restrict__ part_ml, const int* __restrict__ npieces,
    const float* __restrict__ sink, OutT* __restrict__ o, float* lse, int hq, int hkv,
    int s_active, int max_slots, int max_cache_len, int circular) {
    const int pair = blockIdx.x;  // b * hkv + g
    const int b = pair / hkv, g = pair % hkv;
    const int group = hq / hkv, rows = group * s_active;
    const int len = cache_len[b];  // not written by the split kernel
    griddep_wait();                // the split kernel's partials are complete and visible
    const bool valid = len >= s_active && (circular || len <= max_cache_len);
    int ns = 0;
    if (valid) {
        ns = npieces[pair];
        if (ns < 1 || ns > max_slots) {  // cannot happen: never read past the slots
            if (threadIdx.x == 0) atomicOr(&g_decode_error, kDevErrTimeout);
            ns = 0;
        }
    } else if (threadIdx.x == 0 && g == 0) {
        atomicOr(&g_decode_error, kDevErrCacheLen);
    }
    constexpr int kQ = D / 4;  // 16-byte column groups of a row
    for (int c = threadIdx.x; c < rows * kQ; c += kMergeThreads) {
        const int r = c / kQ, x4 = c % kQ;
        const int h = g * group + r / s_active, t = r % s_active;
        const size_t rowid = ((size_t)b * hq + h) * s_active + t;
        const float* ml = part_ml + rowid * max_slots * 2;
        float M = -INFINITY;
        for (int s = 0; s < ns; ++s) M = fmaxf(M, ml[2 * s]);
        float4 out = make_float4(0.f, 0.f, 0.f, 0.f);
        float lse_v = -INFINITY;
        if (M != -INFINITY) {
            float Lsum = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            const float4* po = reinterpret_cast<const float4*>(part_o + rowid * max_slots * D) + x4;
            for (int s = 0; s < ns; ++s) {
                const float wt = ex2(ml[2 * s] - M);
                const float4 v = po[(size_t)s * kQ];
                Lsum += wt * ml[2 * s + 1];
                acc.x += wt * v.x;
                acc.y += wt * v.y;
                acc.z += wt * v.z;
                acc.w += wt * v.w;
            }
            if (sink == nullptr) {
                out = make_float4(acc.x / Lsum, acc.y / Lsum, acc.z / Lsum, acc.w / Lsum);
                lse_v = (M + __log2f(Lsum)) * kLn2;
            } else {
                float inv;
                finish_row(true, M, Lsum, sink[h], inv, lse_v);
                out = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            }
        } else if (valid && sink != nullptr) {  // nothing allowed: the sink alone (O = 0, LSE = sink)
            float inv;
            finish_row(false, 0.f, 0.f, sink[h], inv, lse_v);
        }
        if constexpr (sizeof(OutT) == 2) {
            uint2 w;
            w.x = pack_bf16(out.x, out.y);
            w.y = pack_bf16(out.z, out.w);
            *reinterpret_cast<uint2*>(o + rowid * D + 4 * x4) = w;
        } else {
            *reinterpret_cast<float4*>(o + rowid * D + 4 * x4) = out;
        }
        if (lse != nullptr && x4 == 0) lse[rowid] = lse_v;
    }
}

// The new tokens' K and V written into a bf16 cache ("Flash-Attention: Decode (TKG)",
// "New-token K/V append": the persistent store of the RoPE'd K).  One CTA per (new token,
// kv head, sequence), thread i handles head dims i and i + d/2: new token t sits at logical
// position len - s_active + t, which is its RoPE position (inv_freq != NULL) and its cache
// slot (through the block table, or row j mod max_cache_len of a circular flat cache).
__global__ void append_kv_kernel(const __nv_bfloat16* __restrict__ k_new,
                                 const __nv_bfloat16* __restrict__ v_new,
                                 __nv_bfloat16* __restrict__ k_cache,
                                 __nv_bfloat16* __restrict__ v_cache, AppendArgs a) {
    const int t = blockIdx.x, g = blockIdx.y, b = blockIdx.z, i = threadIdx.x;
    const int h = a.d / 2;
    const int len = a.cache_len[b];
    if (len < a.s_active || (!a.circular && len > a.max_cache_len)) {
        if (i == 0 && t == 0 && g == 0) atomicOr(&g_decode_error, kDevErrCacheLen);
        return;
    }
    const int j = len - a.s_active + t;
    size_t row;
    if (a.block_table != nullptr) {
        const uint32_t pg = __ldg(a.block_table + (size_t)b * a.max_pages_per_seq + j / a.page_size);
        if (pg >= (uint32_t)a.num_pages) {
            if (i == 0) atomicOr(&g_decode_error, kDevErrPageOOB);
            return;  // never write an out-of-range page
        }
        row = ((size_t)pg * a.hkv + g) * a.page_size + (size_t)(j % a.page_size);
    } else {
        row = ((size_t)b * a.hkv + g) * (size_t)a.max_cache_len +
              (size_t)(a.circular ? j % a.max_cache_len : j);
    }
    const size_t src = (((size_t)b * a.hkv + g) * a.s_active + t) * a.d;
    float k0 = __bfloat162float(k_new[src + i]), k1 = __bfloat162float(k_new[src + i + h]);
    if (a.rope_inv_freq != nullptr) {
        float sn, cs;
        rope_sincos(j, __ldg(a.rope_inv_freq + i), sn, cs);
        const float r0 = k0 * cs - k1 * sn, r1 = k1 * cs + k0 * sn;
        k0 = r0;
        k1 = r1;
    }
    k_cache[row * a.d + i] = __float2bfloat16_rn(k0);
    k_cache[row * a.d + i + h] = __float2bfloat16_rn(k1);
    v_cache[row * a.d + i] = v_new[src + i];
    v_cache[row * a.d + i + h] = v_new[src + i + h];
}

// A check of the failure path: one thread waits, with the kernels' bounded wait, on an
// mbarrier phase that nothing completes.  After wait_cycles it gives up, sets the device
// timeout word like a stalled pipeline would, and returns; the context stays usable.
__global__ void wait_timeout_check_kernel(long long wait_cycles) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, &abort_flag, wait_cycles)) atomicOr(&g_decode_error, kDevErrTimeout);
}

// The 0/1 decode mask, one byte per (sequence, head, new token, cache position).
__global__ void gen_mask_kernel(const int32_t* __restrict__ cache_len, int hq, int s_active,
                                int max_len, uint8_t* __restrict__ mask, long long total) {
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long row = idx / max_len;
        const int j = (int)(idx - row * max_len);
        const int t = (int)(row % s_active);
        const int b = (int)(row / ((long long)hq * s_active));
        const int len = cache_len[b];
        uint8_t v = 0;
        if (len < s_active || len > max_len) {
            if (j == 0) atomicOr(&g_decode_error, kDevErrCacheLen);
        } else {
            v = decode_allowed(j, len, s_active, t) ? 1 : 0;
        }
        mask[idx] = v;
    }
}

// SMs of the current device (looked up once per device).
int device_sms() {
    constexpr int kMaxDevices = 64;
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return 0;
    }
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

template <int D, bool kE4M3>
attn_status decode_launch_d(const DecodeArgs& a, cudaStream_t stream) {
    using L = DecodeLayout<D, kE4M3>;
    const bool paged = a.block_table != nullptr;
    constexpr int kBT = L::kBT;
    const int box_rows = paged ? (a.page_size < kBT ? a.page_size : kBT) : kBT;
    CUtensorMap tk, tv;
    uint64_t rows = paged ? (uint64_t)a.num_pages * a.hkv * a.page_size
                          : (uint64_t)a.b * a.hkv * a.max_cache_len;
    uint64_t dims[2] = {(uint64_t)D, rows};
    uint64_t strides[1] = {(uint64_t)D * L::kElemBytes};
    uint32_t box[2] = {(uint32_t)L::kBoxElems, (uint32_t)box_rows};
    const auto make = kE4M3 ? make_u8_map : make_bf16_map;
    if (!make(&tk, a.k_cache, 2, dims, strides, box) || !make(&tv, a.v_cache, 2, dims, strides, box))
        return ATTN_ERR_CUDA;
    DecodeParams p;
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.table = a.block_table;
    p.cache_len = a.cache_len;
    p.part_o = a.part_o;
    p.part_ml = a.part_ml;
    p.npieces = a.npieces;
    p.b = a.b;
    p.hq = a.hq;
    p.hkv = a.hkv;
    p.s_active = a.s_active;
    p.page_size = paged ? a.page_size : 1;
    p.max_pages = a.max_pages_per_seq;
    p.num_pages = a.num_pages;
    p.max_cache_len = a.max_cache_len;
    p.group = a.hq / a.hkv;
    p.rows = p.group * a.s_active;
    p.min_tiles = a.kv_chunk / kBT;
    p.max_slots = a.max_slots;
    p.paged = paged ? 1 : 0;
    p.box_rows = box_rows;
    p.c = kE4M3 ? a.scale * a.k_scale * kLog2e : a.scale * kLog2e;
    p.v_scale = kE4M3 ? a.v_scale : 1.0f;
    p.window = a.window;
    p.circular = a.circular;
    p.rope_inv_freq = a.rope_inv_freq;

    static std::atomic<unsigned long long> attr_done{0};  // setting it twice is harmless
    if (needs_setup(attr_done)) {
        if (cudaFuncSetAttribute(decode_split_kernel<D, kE4M3>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynBytes) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        mark_setup(attr_done);
    }
    // one wave: the CTAs every SM holds at once
    const int sms = device_sms();
    if (sms <= 0) return ATTN_ERR_CUDA;
    decode_split_kernel<D, kE4M3><<<sms * L::kMinCtas, kThreads, L::kDynBytes, stream>>>(tk, tv, p);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    // The merge launches as a programmatic dependent of the split pass, so its launch overlaps
    // the split pass's last CTAs.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((size_t)a.b * a.hkv));
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    const float* po = a.part_o;
    const float* pml = a.part_ml;
    const int* np = a.npieces;
    if (a.o_dtype == ATTN_BF16)
        e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<D, __nv_bfloat16>, a.cache_len, po, pml,
                               np, a.sink, static_cast<__nv_bfloat16*>(a.o), a.lse, a.hq, a.hkv,
                               a.s_active, a.max_slots, a.max_cache_len, a.circular);
    else
        e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<D, float>, a.cache_len, po, pml, np,
                               a.sink, static_cast<float*>(a.o), a.lse, a.hq, a.hkv, a.s_active,
                               a.max_slots, a.max_cache_len, a.circular);
    if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

}  // namespace

attn_status decode_launch(const DecodeArgs& a, cudaStream_t stream) {
    if (a.kv_e4m3) {
        switch (a.d) {  // a 64-dim e4m3 row is half a 128-byte box: not supported
            case 128: return decode_launch_d<128, true>(a, stream);
            case 256: return decode_launch_d<256, true>(a, stream);
            default: return ATTN_ERR_UNSUPPORTED;
        }
    }
    switch (a.d) {
        case 64: return decode_launch_d<64, false>(a, stream);
        case 128: return decode_launch_d<128, false>(a, stream);
        case 256: return decode_launch_d<256, false>(a, stream);
        default: return ATTN_ERR_UNSUPPORTED;
    }
}

attn_status append_launch(const AppendArgs& a, cudaStream_t stream) {
    dim3 grid(a.s_active, a.hkv, a.b);
    append_kv_kernel<<<grid, a.d / 2, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(a.k_new), static_cast<const __nv_bfloat16*>(a.v_new),
        static_cast<__nv_bfloat16*>(a.k_cache), static_cast<__nv_bfloat16*>(a.v_cache), a);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

attn_status wait_timeout_check_launch(long long wait_cycles, cudaStream_t stream) {
    wait_timeout_check_kernel<<<1, 32, 0, stream>>>(wait_cycles);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

attn_status gen_mask_launch(const int32_t* cache_len, int b, int hq, int s_active, int max_len,
                            uint8_t* mask, cudaStream_t stream) {
    const long long total = (long long)b * hq * s_active * max_len;
    if (total == 0) return ATTN_OK;
    long long blocks = (total + 255) / 256;
    if (blocks > 152ll * 64) blocks = 152ll * 64;
    gen_mask_kernel<<<(unsigned)blocks, 256, 0, stream>>>(cache_len, hq, s_active, max_len, mask,
                                                          total);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

unsigned decode_take_error(cudaStream_t stream, cudaError_t* err) {
    unsigned v = 0, zero = 0;
    *err = cudaMemcpyFromSymbolAsync(&v, g_decode_error, sizeof v, 0, cudaMemcpyDeviceToHost, stream);
    if (*err == cudaSuccess)
        *err = cudaMemcpyToSymbolAsync(g_decode_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice,
                                       stream);
    if (*err == cudaSuccess) *err = cudaStreamSynchronize(stream);
    if (*err != cudaSuccess) cudaGetLastError();
    return v;
}

}  // namespace attn
