// prefill_sm103.cu -- fused attention forward (prefill) on the 5th-generation tensor cores.
//
// Method: the flash-attention online-softmax recurrence ("Flash-Attention: Context (CTE)",
// "The online-softmax recurrence"; minfer "03 - 8n", section 2.1): for each query row a
// running max m, a running sum l and an output accumulator O are carried across K/V
// tiles, O and l are rescaled by alpha = exp(m_old - m_new), and O is divided by l at
// the end.  Q stays resident while K/V stream ("CTE", "Tile shapes and residency"); tiles
// wholly outside the causal / window band are never loaded ("CTE", "Algorithm -
// compute-skip"; optimum-neuron AGENTS.md, "Sliding window": large-tile filtering), and
// the element mask runs only on tiles that cross a band edge ("CTE", "The diagonal
// affine_select mask").  GQA maps query head h to kv head h / (hq / hkv) ("CTE", "GQA
// and multi-head"); head_dim 256 simply widens the MMA contraction, the role the pages
// give to d-tiling (optimum-neuron AGENTS.md, "flash_fwd_large_d").
//
// GB300 design.  Two kernels share the method: for head_dim 64 and 128 a CTA owns two
// 128-row query tiles that share every K/V tile (the two-q-tile kernel below); for
// head_dim 256 the two accumulators would not fit TMEM, so a CTA owns one tile (the
// one-q-tile kernel).  The common structure, per CTA:
//   warp 0    TMA producer: Q once, then K and V tiles through two 2-deep rings.
//   warp 1    MMA issuer (one thread): S = Q K^T into one of two TMEM buffers, then
//             O += P V into a TMEM accumulator that lives for the whole KV pass.  S(j+2)
//             is issued as soon as the softmax has copied S(j) out of TMEM, so the tensor
//             pipe holds the next scores while the softmax of tile j runs.
//   warp 2    owns the TMEM allocation.
//   softmax   one warpgroup per TMEM accumulator; thread = query row = TMEM lane.  With
//             head_dim <= 128 two warpgroups take alternate KV tiles, each with its own
//             running max, sum and O accumulator (S0, S1, O0, O1 fill the 512 TMEM columns),
//             and the two partial results are merged once in the epilogue -- the
//             split-KV identity of the online softmax, applied inside the CTA.  With
//             head_dim 256 one warpgroup takes every tile.  Each thread reads its S row from
//             TMEM, masks it if the tile crosses a band edge, folds scale*log2(e) into the
//             exponent, writes P (bf16) into a 128-byte-swizzled shared-memory tile for the
//             second MMA, and rescales its O in TMEM only when the row max has grown by more
//             than 2^8 since the last rescale (the stale max is used consistently for P and
//             l, so O / l is unchanged).
// The accumulators never leave TMEM until the epilogue, so no O round trip through HBM
// (the pages' sectioned design) is needed at any sequence length.
#include <float.h>

#include "attn_internal.h"
#include "attn_ptx.cuh"

namespace attn {
namespace {

__device__ unsigned g_prefill_error;

constexpr int kBM = 128;           // query rows per tile (= TMEM lanes)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale threshold, log2 units
// Registers after re-balancing: the TMA/MMA warpgroup gives up registers to the softmax
// warpgroups.  128 * kRegsLow + 256 * kRegsHigh == 384 * kRegsLaunch3 (the launch budget).
constexpr int kRegsLaunch3 = 168;
constexpr int kRegsLow = 96;
constexpr int kRegsHigh = 200;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= 384 * kRegsLaunch3, "register split");

struct PrefillParams {
    void* o;
    float* lse;
    const float* sink;  // [hq] sink logits of the query heads, or NULL
    // packed sequences: offsets [nseq + 1] along the query and key rows, or NULL
    const int* cu_q;
    const int* cu_k;
    int nseq;
    const int* order;  // packed: the work order of the query units (unit_order_kernel), or NULL
    int* unit_counter; // packed, head_dim <= 128: units handed out at run time from this, or NULL
    int hq, hkv, sq, skv, group, nqt, window, causal, o_f32;
    int nbh;     // b * hq
    int nunits;  // work units of the persistent kernel
    float c;     // scale * log2(e)
};

// Persistent schedule.  Units are numbered heaviest first (for a causal mask the last
// query tiles see the most keys), and CTA c of G takes units c, 2G-1-c, 2G+c, 4G-1-c, ...
// (a zig-zag over the sorted list), so heavy and light units pair up on every CTA.
__device__ __forceinline__ int zigzag_unit(int cta, int round, int grid) {
    return (round & 1) ? round * grid + (grid - 1 - cta) : round * grid + cta;
}

// The same units of CTA c, lightest round first (INT_MAX past the last).  The last rounds
// hold the lightest units, of a different length on each CTA, so the CTAs' unit boundaries
// (each with a Q tile load from DRAM) no longer fall together: head_dim-256 window prefill
// 1267 -> 1286 TFLOP/s with bit-identical results, each CTA's total work unchanged.
__device__ __forceinline__ int zigzag_unit_rev(int cta, int round, int grid, int nunits) {
    int rounds = nunits / grid;
    if (rounds * grid + ((rounds & 1) ? grid - 1 - cta : cta) < nunits) ++rounds;
    return round < rounds ? zigzag_unit(cta, rounds - 1 - round, grid) : INT_MAX;
}

// Shared-memory descriptors advance along a tile by adding the byte offset / 16 to the
// address field in the low bits (tiles never straddle the 256 KB field range).
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t byte_off) { return d + (byte_off >> 4); }

// Packed sequences: the sequence of query row i (the last s with cu_q[s] <= i).
__device__ __forceinline__ int row_sequence(const PrefillParams& p, int i) {
    int a = 0, b = p.nseq - 1;
    while (a < b) {
        const int m = (a + b + 1) >> 1;
        if (__ldg(p.cu_q + m) <= i) a = m;
        else b = m - 1;
    }
    return a;
}

// Packed sequences: key rows [lo, hi] that query row i of sequence s may attend (hi < lo:
// none).  The sequence's keys are rows [cu_k[s], cu_k[s+1]), its queries sit at the tail of
// them, and the causal and window bands apply inside it ("Flash-Attention: Context (CTE)",
// "Algorithm - the dynamic range_select family": per-row key bounds for sequence packing
// and a dynamic prefix length).
__device__ __forceinline__ void row_key_bounds(const PrefillParams& p, int i, int s, int& lo,
                                               int& hi) {
    const int q0 = __ldg(p.cu_q + s), k0 = __ldg(p.cu_k + s);
    const int nk = __ldg(p.cu_k + s + 1) - k0;
    const int qpos = (i - q0) + nk - (__ldg(p.cu_q + s + 1) - q0);
    hi = k0 + (p.causal ? min(qpos, nk - 1) : nk - 1);
    lo = k0 + (p.window > 0 ? max(0, qpos - p.window + 1) : 0);
}

// A query tile and its KV-tile range [kt0, kt0 + n).  One problem per (batch, head): the
// queries sit at the tail of the keys (q_pos = i + skv - sq).  Packed sequences (kPacked):
// [all_lo, all_hi] holds the keys every row of the tile may attend (tiles wholly inside
// need no mask).  Bounds grow with the row inside one sequence, so its first and last rows
// give them; a tile that spans sequences is masked everywhere, and its range reaches at
// least to the start of its last sequence (a causal sequence with more queries than keys
// has leading rows with no key at all).  kPacked is a template parameter so that the
// unpacked kernels keep their own code.
struct TileRange {
    int q0, rows, qpos_lo, qpos_hi, kt0, n, all_lo, all_hi;
};

template <int BN, bool kPacked>
__device__ __forceinline__ TileRange tile_range(const PrefillParams& p, int qt) {
    TileRange r;
    r.q0 = qt * kBM;
    r.rows = min(kBM, p.sq - r.q0);
    const int off = p.skv - p.sq;  // queries sit at the tail of the keys
    r.qpos_lo = r.q0 + off;
    r.qpos_hi = r.q0 + r.rows - 1 + off;
    r.all_lo = INT_MAX;
    r.all_hi = INT_MIN;
    if (r.rows <= 0) {  // a query tile past the end of the sequence
        r.kt0 = 0;
        r.n = 0;
        return r;
    }
    int k_end, k_begin;
    if constexpr (kPacked) {
        const int last = r.q0 + r.rows - 1;
        const int s0 = row_sequence(p, r.q0), s1 = row_sequence(p, last);
        int lo0, hi0, lo1, hi1;
        row_key_bounds(p, r.q0, s0, lo0, hi0);
        row_key_bounds(p, last, s1, lo1, hi1);
        k_end = min(p.skv, hi1 + 1);
        k_begin = max(0, lo0);
        if (s0 == s1) {
            r.all_lo = lo1;
            r.all_hi = hi0;
        } else {
            k_end = max(k_end, min(p.skv, __ldg(p.cu_k + s1)));
        }
    } else {
        k_end = p.causal ? min(p.skv, r.qpos_hi + 1) : p.skv;
        k_begin = p.window > 0 ? max(0, r.qpos_lo - p.window + 1) : 0;
    }
    if (k_end <= k_begin) {
        r.kt0 = 0;
        r.n = 0;
    } else {
        r.kt0 = k_begin / BN;
        r.n = (k_end + BN - 1) / BN - r.kt0;
    }
    return r;
}

// Packed sequences: the work order of the query units (a 128-row tile, or a pair of them).
// One CTA; the 64-bit keys are sorted by a bitonic network in shared memory, and the unit
// index is the low 32 bits of each key.
//  * Static schedule (head_dim 256): KV-tile count, most first, ties by index.  The
//    persistent kernel's zig-zag then pairs heavy with light units on every CTA as it does
//    for one causal problem, where the index order already is the order of the work.
//  * Units handed out at run time (head_dim <= 128, `counter` set): sequence first, then
//    KV-tile count, most first.  The CTAs draw units from the counter, which this pass
//    resets, so the units in flight are always a window of this list: the K/V of one or two
//    sequences, which stays in L2 while their query tiles pass, and the CTAs stay balanced
//    without a static pairing.  (Against the count order with the zig-zag, on 16 packed
//    sequences: the count order runs units of every sequence at once, whose K/V (177 MB)
//    exceed the L2, and read 1.8x the algorithmic bytes.)
constexpr int kOrderMax = 8192;  // units sorted in one CTA (64 KB of keys)
constexpr int kOrderThreads = 1024;

template <int BN, int kTilesPerUnit>
__global__ void __launch_bounds__(kOrderThreads) unit_order_kernel(const PrefillParams p, int nu,
                                                                   int* order, int* counter) {
    extern __shared__ unsigned long long keys[];
    int n2 = 1;
    while (n2 < nu) n2 <<= 1;
    for (int u = threadIdx.x; u < n2; u += blockDim.x) {
        unsigned long long key = ~0ull;  // padding sorts last
        if (u < nu) {
            int cost = 0;
            for (int x = 0; x < kTilesPerUnit; ++x) cost += tile_range<BN, true>(p, kTilesPerUnit * u + x).n;
            if (counter != nullptr) {
                const int seq = row_sequence(p, min(kTilesPerUnit * u * kBM, p.sq - 1));
                key = ((unsigned long long)min(seq, 0xffff) << 48) |
                      ((unsigned long long)(0xffff - min(cost, 0xffff)) << 32) | (unsigned)u;
            } else {
                key = ((unsigned long long)(0x7fffffff - cost) << 32) | (unsigned)u;
            }
        }
        keys[u] = key;
    }
    __syncthreads();
    for (int k = 2; k <= n2; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n2; i += blockDim.x) {
                const int l = i ^ j;
                if (l > i) {
                    const unsigned long long a = keys[i], b = keys[l];
                    if ((a > b) == ((i & k) == 0)) {  // ascending where bit k of i is clear
                        keys[i] = b;
                        keys[l] = a;
                    }
                }
            }
            __syncthreads();
        }
    for (int u = threadIdx.x; u < nu; u += blockDim.x) order[u] = (int)(keys[u] & 0xffffffffu);
    if (counter != nullptr && threadIdx.x == 0) *counter = 0;
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, int* abort_flag) {
    return mbar_wait(bar, parity, reinterpret_cast<volatile int*>(abort_flag));
}

__device__ __forceinline__ void wait_bounded(uint64_t* bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitLimitCycles) return;
}

// =========================================================================== head_dim 256
// Shared-memory / TMEM plan of the head_dim-256 kernel (BN = 64).  Shared memory: the Q
// tile (64 KB), a 3-slot K ring and a 2-slot V ring (32 KB slots).  TMEM:
//   S0..S3 [i BN, (i+1) BN)  O [256, 256 + D)
// The softmax writes P(T) over the first BN/2 columns of S buffer T % 4, and S(T+4) takes
// that buffer once PV(T) is done.  Four buffers keep the S chain (S issue, softmax read)
// from waiting on its own latency, and let the softmax run four tiles ahead of P.V, which
// covers the wait of a unit's first P.V for the epilogue to read O out.
template <int D>
struct CfgW {
    static constexpr int BN = 64;
    static constexpr int kQBytes = D * kBM * 2;
    static constexpr int kSlotBytes = D * BN * 2;
    static constexpr int kKSlots = 3;
    static constexpr int kVSlots = 2;
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQBytes;
    static constexpr int kVOff = kKOff + kKSlots * kSlotBytes;
    static constexpr int kSmem = kVOff + kVSlots * kSlotBytes;
    static constexpr int kDynBytes = kSmem + 1024;
    static constexpr int kTmemCols = 512;
    static constexpr int kSBufs = 4;        // S buffers, each also holding its P
    static constexpr uint32_t kColO = 256;  // O at [256, 256 + D)
    static constexpr int kThreads = 512;
    static_assert(kSBufs * BN <= (int)kColO && kColO + D <= kTmemCols, "TMEM budget");
    static_assert(kDynBytes + 512 <= 232448, "shared memory budget");
};

// Persistent: each CTA loops over work units (one 128-row query tile of one head, heaviest
// first, zig-zag over CTAs).  Roles:
//   warp 0: Q and K producer      warp 2: V producer (and TMEM owner)
//   warps 1 / 4: S issuers of the even / odd KV tiles   S(T) = Q K(T)^T into buffer T % 4
//   warp 3: PV issuer  O += P(T) V(T)
//   warps 8-11: softmax (thread = query row = TMEM lane)
//   warps 12-15: epilogue -- normalise O, write it and the LSE out
// An S tile of head_dim 256 takes 16 products of N = BN, more than one thread issues in
// the time the pipe runs them, so two issuers take alternate tiles.  At the end of a unit
// the softmax hands its (max, sum) per row to the epilogue warps through shared memory and
// goes on with the next unit's tiles; the next unit's first PV waits until the epilogue
// has read O out of TMEM.  That read-out is bound by the latency of the TMEM loads, so it
// takes 64 columns per load.  Register split per warpgroup: roles kRegsRole, softmax
// kRegsSoftmax, epilogue the launch budget.
constexpr int kRegsLaunch4 = 128;  // 512 threads
constexpr int kRegsRole = 96;
constexpr int kRegsSoftmax = 160;
static_assert(256 * kRegsRole + 128 * kRegsSoftmax + 128 * kRegsLaunch4 <= 512 * kRegsLaunch4,
              "register split");

template <int D, bool kPacked>
__global__ void __launch_bounds__(CfgW<D>::kThreads, 1) prefill_wide_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
    using C = CfgW<D>;
    constexpr int BN = C::BN;
    constexpr int NK = C::kKSlots;
    constexpr int NV = C::kVSlots;
    constexpr int NS = C::kSBufs;
    extern __shared__ uint8_t dyn_smem[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t q_full, q_empty, k_full[NK], k_empty[NK], v_full[NV], v_empty[NV];
    __shared__ uint64_t s_full[NS], p_full[NS], p_free[NS];
    // o_free[h]: the epilogue has read O's columns [h D/2, (h+1) D/2)
    __shared__ uint64_t o_done, o_free[2], mma_drain, stats_full, stats_free;
    __shared__ uint64_t turn[2];   // S issue turns of the even and odd tiles
    __shared__ float2 stats[kBM];  // per row: the unit's running max and sum, for the epilogue
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, cta = blockIdx.x;

    // unit w -> (query tile, batch*head, kv batch*head) and its KV tile range
    auto unit_at = [&](int w, int& bh, int& kvz) -> TileRange {
        int qt = p.nqt - 1 - w / p.nbh;
        if constexpr (kPacked)
            if (p.order) {
                qt = __ldg(p.order + w / p.nbh);
                if (qt < 0 || qt >= p.nqt) qt = p.nqt;  // never trust an index: past sq = no work
            }
        bh = w % p.nbh;
        const int bidx = bh / p.hq, h = bh % p.hq;
        kvz = bidx * p.hkv + h / p.group;
        return tile_range<BN, kPacked>(p, qt);
    };

    if (threadIdx.x == 0) {
        mbar_init(&q_full, 1);
        mbar_init(&q_empty, 2);  // both S issuers, after their last product of the unit
        for (int i = 0; i < NK; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < NS; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 128);
            mbar_init(&p_free[i], 1);
        }
        mbar_init(&o_done, 1);
        mbar_init(&o_free[0], 128);
        mbar_init(&o_free[1], 128);
        mbar_init(&mma_drain, 3);
        mbar_init(&turn[0], 1);
        mbar_init(&turn[1], 1);
        mbar_arrive(&turn[0]);  // the even issuer takes the first turn
        mbar_init(&stats_full, 128);
        mbar_init(&stats_free, 128);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(&tmem_base_sh, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp < 8) {
        regs_dec<kRegsRole>();
        if ((warp == 0 || warp == 2) && lane == 0) {
            // -------------------------------------------- Q + K producer / V producer
            const bool is_k = warp == 0;
            uint64_t* full = is_k ? k_full : v_full;
            uint64_t* empty = is_k ? k_empty : v_empty;
            const int ns = is_k ? NK : NV;
            const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
            uint8_t* ring = sm + (is_k ? C::kKOff : C::kVOff);
            tma_prefetch_desc(tm);
            if (is_k) tma_prefetch_desc(&tm_q);
            int L = 0;   // tiles issued into this ring
            int rq = 0;  // Q tiles issued
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int w = zigzag_unit_rev(cta, r, G, p.nunits);
                if (w >= p.nunits) break;
                int bh, kvz;
                const TileRange t = unit_at(w, bh, kvz);
                if (t.n == 0) continue;
                if (is_k) {
                    // the Q tile is free once every S product of the previous unit is done
                    if (rq > 0 && !wait_or_abort(&q_empty, (rq - 1) & 1, &abort_flag)) break;
                    ++rq;
                    mbar_arrive_expect_tx(&q_full, C::kQBytes);
#pragma unroll
                    for (int dc = 0; dc < D / 64; ++dc)
                        tma_load_3d(sm + C::kQOff + dc * (kBM * 128), &tm_q, dc * 64, t.q0, bh, &q_full);
                }
                for (int i = 0; i < t.n; ++i, ++L) {
                    const int slot = L % ns;
                    if (L >= ns && !wait_or_abort(&empty[slot], ((L / ns) - 1) & 1, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[slot], C::kSlotBytes);
#pragma unroll
                    for (int dc = 0; dc < D / 64; ++dc)
                        tma_load_3d(ring + slot * C::kSlotBytes + dc * (BN * 128), tm, dc * 64,
                                    (t.kt0 + i) * BN, kvz, &full[slot]);
                }
            }
            if (abort_flag) {  // let copies in flight land before the CTA exits
                for (int i = max(0, L - ns); i < L; ++i) wait_bounded(&full[i % ns], (i / ns) & 1);
                if (rq > 0) wait_bounded(&q_full, (rq - 1) & 1);
            }
        } else if (warp == 1 || warp == 4) {
            // --------------------------------------------- S issuers (even / odd tiles)
            // A turn passes from tile T's issuer to tile T+1's once T's waits are done and
            // before its products are issued, so the two issue at once while every wait runs
            // in tile order.  That order matters for the K ring: the wait for K(T) on slot
            // T % NK reads the slot's phase by parity, which is only sound once K(T - NK),
            // the other issuer's tile when NK is odd, is known to have landed.  Four S
            // buffers let the issuers drift apart, so nothing else ensures it.  The whole
            // warp runs the issuing code, waits included, and one elected lane issues (see
            // the two-q-tile kernel): 8K window 1201 -> 1238 TFLOP/s.
            const int par = warp == 1 ? 0 : 1;
            constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, BN, 0, 0);
            const uint64_t qd = sw128_desc(smem_u32(sm + C::kQOff), 16, 1024);
            const uint64_t kd0 = sw128_desc(smem_u32(sm + C::kKOff), 16, 1024);
            int T = 0;      // tiles of all units so far (= K ring index)
            int uq = 0;     // units with tiles so far (phase of q_full)
            int turns = 0;  // turns taken so far (phase of turn[par])
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int w = zigzag_unit_rev(cta, r, G, p.nunits);
                if (w >= p.nunits) break;
                int bh, kvz;
                const TileRange t = unit_at(w, bh, kvz);
                if (t.n == 0) continue;
                if (!__all_sync(0xffffffffu, wait_or_abort(&q_full, uq & 1, &abort_flag))) break;
                ++uq;
                tc_fence_after();
                for (int i = 0; i < t.n; ++i, ++T) {
                    if ((T & 1) != par) continue;
                    const int b = T % NS, slot = T % NK;
                    // S buffer b is free once PV(T - NS) has read P(T - NS) out of it
                    bool okw = wait_or_abort(&turn[par], turns & 1, &abort_flag);
                    if (okw && T >= NS) okw = wait_or_abort(&p_free[b], ((T / NS) - 1) & 1, &abort_flag);
                    if (okw) okw = wait_or_abort(&k_full[slot], (T / NK) & 1, &abort_flag);
                    ok = __all_sync(0xffffffffu, okw);
                    if (!ok) break;
                    ++turns;
                    mbar_arrive_w(&turn[par ^ 1]);  // tile T+1's issuer may do its waits
                    tc_fence_after();
                    const uint64_t kd = desc_add(kd0, (uint32_t)(slot * C::kSlotBytes));
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off_a = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
                        const uint32_t off_b = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
                        tc_mma_ss_w(tmem + b * BN, desc_add(qd, off_a), desc_add(kd, off_b),
                                    idesc_s, kk > 0 ? 1u : 0u);
                    }
                    tc_commit_w(&s_full[b]);
                    tc_commit_w(&k_empty[slot]);  // K(T) consumed once this product is done
                }
                if (ok) tc_commit_w(&q_empty);  // this issuer's products of the unit read Q no more
            }
            tc_commit_w(&mma_drain);
            wait_bounded(&mma_drain, 0);
        } else if (warp == 3) {
            // ----------------------------------------------------------- PV issuer
            // (warp-collective like the S issuers)
            // P.V in two N = D/2 halves (the same products, column by column)
            constexpr uint32_t idesc_oh = idesc_bf16_f32(kBM, D / 2, 0, 1);
            const uint64_t vd0 = sw128_desc(smem_u32(sm + C::kVOff), BN * 128, 1024);
            int T = 0;
            int uo = 0;  // units with tiles so far (o_free completes once per such unit)
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int w = zigzag_unit_rev(cta, r, G, p.nunits);
                if (w >= p.nunits) break;
                int bh, kvz;
                const TileRange t = unit_at(w, bh, kvz);
                if (t.n == 0) continue;
                // the previous unit's epilogue must have read each half of O before that
                // half is overwritten: the first tile's products wait for each half apart
                bool oko = true;
                if (uo > 0) oko = wait_or_abort(&o_free[0], (uo - 1) & 1, &abort_flag);
                if (!__all_sync(0xffffffffu, oko)) break;
                const uint32_t ofph = (uo - 1) & 1;
                const bool wait_hi = uo > 0;
                ++uo;
                for (int i = 0; i < t.n; ++i, ++T) {
                    const int b = T % NS, slot = T % NV;
                    const bool okw = wait_or_abort(&p_full[b], (T / NS) & 1, &abort_flag) &&
                                     wait_or_abort(&v_full[slot], (T / NV) & 1, &abort_flag);
                    ok = __all_sync(0xffffffffu, okw);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t vd = desc_add(vd0, (uint32_t)(slot * C::kSlotBytes));
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        tc_mma_ts_w(tmem + C::kColO, tmem + b * BN + kk * 8,
                                    desc_add(vd, kk * 16 * 128), idesc_oh, (i > 0 || kk > 0) ? 1u : 0u);
                    if (i == 0 && wait_hi) {
                        ok = __all_sync(0xffffffffu, wait_or_abort(&o_free[1], ofph, &abort_flag));
                        if (!ok) break;
                        tc_fence_after();
                    }
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        tc_mma_ts_w(tmem + C::kColO + D / 2, tmem + b * BN + kk * 8,
                                    desc_add(vd, (D / 2) / 64 * (BN * 128) + kk * 16 * 128), idesc_oh,
                                    (i > 0 || kk > 0) ? 1u : 0u);
                    tc_commit_w(&p_free[b]);      // S buffer b may be rewritten; O holds PV(T)
                    tc_commit_w(&v_empty[slot]);  // V(T) consumed
                    if (i == t.n - 1) tc_commit_w(&o_done);
                }
            }
            tc_commit_w(&mma_drain);
            wait_bounded(&mma_drain, 0);
        }
    } else if (warp < 12) {
        // ------------------------------------------------------------------ softmax
        regs_inc<kRegsSoftmax>();
        const int row = (warp & 3) * 32 + lane;
        const uint32_t tm_row = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t tm_o = tm_row + C::kColO;
        const float c = p.c;
        const bool c_pos = c > 0.f;
        const float cm = c_pos ? c : 1.0f;  // exponent = x * cm - m
        int T = 0;   // S tiles consumed so far (across units)
        int su = 0;  // units with tiles so far (phase of stats_full / stats_free)
        bool ok = true;
        // Waits end with a warp-uniform verdict, so that a wait given up on never leaves
        // part of a warp ahead of a warp-collective tcgen05 access.
        auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, wait_or_abort(bar, parity, &abort_flag));
        };
        for (int r = 0;; ++r) {
            const int w = zigzag_unit_rev(cta, r, G, p.nunits);
            if (w >= p.nunits) break;
            int bh, kvz;
            const TileRange t = unit_at(w, bh, kvz);
            int key_lo, key_hi;
            if constexpr (kPacked) {
                const int qrow = min(t.q0 + row, p.sq - 1);  // rows past sq are never stored
                row_key_bounds(p, qrow, row_sequence(p, qrow), key_lo, key_hi);
            } else {
                const int qpos = t.qpos_lo + row;
                key_lo = p.window > 0 ? qpos - p.window + 1 : INT_MIN;
                key_hi = p.causal ? min(qpos, p.skv - 1) : p.skv - 1;
            }
            float m_used = -INFINITY, l_sum = 0.f;
            for (int i = 0; ok && i < t.n; ++i, ++T) {
                const int b = T % NS;
                if (!wait_warp(&s_full[b], (T / NS) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tm_s = tm_row + b * BN;
                const int k0 = (t.kt0 + i) * BN;
                const bool edge =
                    kPacked ? (k0 < t.all_lo || k0 + BN - 1 > t.all_hi)
                            : ((p.causal && k0 + BN - 1 > t.qpos_lo) || (k0 + BN > p.skv) ||
                               (p.window > 0 && k0 < t.qpos_hi - p.window + 1));
                // the S row from TMEM, scaled for scale <= 0, then masked (edge tiles; a
                // masked key is -inf whatever the sign of the scale)
                auto load_s = [&](float* v) {
                    uint32_t rr[BN];
                    tmem_ld64(tm_s, rr);
#pragma unroll
                    for (int e = 0; e < BN; ++e) v[e] = __uint_as_float(rr[e]);
                    if (!c_pos) {
#pragma unroll
                        for (int e = 0; e < BN; ++e) v[e] *= c;
                    }
                    if (edge) {
#pragma unroll
                        for (int e = 0; e < BN; ++e) {
                            const int key = k0 + e;
                            if (key < key_lo || key > key_hi) v[e] = -INFINITY;
                        }
                    }
                };
                // P = 2^(v * cm - m_e) packed to bf16 pairs; returns its sum, and the packed
                // maximum through pmax
                auto exps = [&](const float* v, float m_e, uint32_t* pk, uint32_t& pmax) -> float {
                    float ls[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) ls[e] = 0.f;
                    pmax = 0u;
#pragma unroll
                    for (int e = 0; e < BN / 2; ++e) {
                        float a0, a1;
                        ffma2(a0, a1, v[2 * e], v[2 * e + 1], cm, cm, -m_e, -m_e);
                        const float p0 = ex2(a0), p1 = ex2(a1);
                        fadd2(ls[(2 * e) & 7], ls[(2 * e + 1) & 7], ls[(2 * e) & 7], ls[(2 * e + 1) & 7], p0, p1);
                        pk[e] = pack_bf16(p0, p1);
                        pmax = __vmaxu2(pmax, pk[e]);
                    }
                    return ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
                };
                uint32_t pk[BN / 2];
                float l_tile = 0.f;
                // Common case: one pass of exponents against the running max m_used.  The
                // row's max grew by more than 2^kRescaleLog2 exactly when an exponent exceeds
                // 2^kRescaleLog2, read off the packed bf16 values (an unsigned 16-bit max
                // orders non-negative bf16 values by size).  A row without a finite max yet
                // takes the exact path; decided per warp, as the TMEM loads are collective.
                bool redo = __any_sync(0xffffffffu, m_used == -INFINITY);
                if (!redo) {
                    float v[BN];
                    load_s(v);
                    uint32_t pmax;
                    l_tile = exps(v, m_used, pk, pmax);
                    constexpr uint32_t kTwoPow8 = 0x4380u;  // bf16 bits of 2^kRescaleLog2 = 256
                    redo = __any_sync(0xffffffffu,
                                      (pmax & 0xFFFFu) > kTwoPow8 || (pmax >> 16) > kTwoPow8);
                }
                if (redo) {
                    // Exact path: the tile max (S(T) is still in TMEM), O and l rescaled where
                    // the max moves, the exponents recomputed.
                    float v[BN];
                    load_s(v);
                    float mx[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
#pragma unroll
                    for (int e = 0; e < BN; ++e) mx[e & 7] = fmaxf(mx[e & 7], v[e]);
                    float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                    if (c_pos) tmax *= c;  // -inf stays -inf
                    const float m_new = fmaxf(m_used, tmax);
                    const bool need = (m_used != -INFINITY) && (m_new > m_used + kRescaleLog2);
                    if (__any_sync(0xffffffffu, need)) {
                        // O holds the unit's products up to PV(T-1): let it land, then scale
                        // it in place
                        if (!wait_warp(&p_free[(T - 1) % NS], ((T - 1) / NS) & 1)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const float alpha = need ? ex2(m_used - m_new) : 1.0f;
#pragma unroll 1
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t rr[32];
                            tmem_ld32(tm_o + c0, rr);
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
                            tmem_st32(tm_o + c0, rr);
                        }
                        tmem_wait_st();
                        if (need) l_sum *= alpha;
                    }
                    if (m_used == -INFINITY || need) m_used = m_new;  // nothing accumulated yet
                    uint32_t pmax;
                    l_tile = exps(v, (m_used == -INFINITY) ? 0.f : m_used, pk, pmax);
                }
                l_sum += l_tile;
                // P(T) over the first BN/2 columns of S buffer b (S(T) has been read)
                tmem_st32(tm_s, pk);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&p_full[b]);
            }
            if (t.n > 0) {
                // hand the unit's (max, sum) to the epilogue warps once they have taken the
                // previous unit's
                if (su > 0) ok = wait_warp(&stats_free, (su - 1) & 1) && ok;
                stats[row] = make_float2(m_used, l_sum);
                mbar_arrive(&stats_full);
                ++su;
            }
        }
    } else {
        // ----------------------------------------------------------------- epilogue
        const int row = (warp & 3) * 32 + lane;
        const uint32_t tm_o = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + C::kColO;
        int ue = 0;  // units with tiles so far (phase of o_done and stats_full)
        auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, wait_or_abort(bar, parity, &abort_flag));
        };
        for (int r = 0;; ++r) {
            const int w = zigzag_unit_rev(cta, r, G, p.nunits);
            if (w >= p.nunits) break;
            int bh, kvz;
            const TileRange t = unit_at(w, bh, kvz);
            const int q_row = t.q0 + row;
            bool have_o = false;
            float m_used = -INFINITY, l_sum = 0.f;
            if (t.n > 0) {
                have_o = wait_warp(&o_done, ue & 1);
                tc_fence_after();
                have_o = wait_warp(&stats_full, ue & 1) && have_o;
                const float2 st = stats[row];
                m_used = st.x;
                l_sum = st.y;
                mbar_arrive(&stats_free);
                ++ue;
            }
            const bool row_valid = t.rows > 0 && row < t.rows;
            const bool live = have_o && l_sum > 0.f;
            float inv, lse_v;
            finish_row(live, m_used, l_sum, p.sink ? p.sink[bh % p.hq] : -INFINITY, inv, lse_v);
            const size_t orow = (size_t)bh * p.sq + q_row;
            if (row_valid && p.lse != nullptr) p.lse[orow] = lse_v;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 64) {
                uint32_t rr[64];
                if (t.n > 0) {
                    tmem_ld64(tm_o + c0, rr);
                } else {
#pragma unroll
                    for (int e = 0; e < 64; ++e) rr[e] = 0u;
                }
                if ((c0 + 64 == D / 2 || c0 + 64 == D) && t.n > 0) {
                    tc_fence_before();
                    mbar_arrive(&o_free[c0 + 64 == D]);  // this half of O has been read
                }
                if (row_valid) {
                    if (p.o_f32) {
                        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow * D + c0);
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            dst[e] = make_float4(__uint_as_float(rr[4 * e]) * inv, __uint_as_float(rr[4 * e + 1]) * inv,
                                                 __uint_as_float(rr[4 * e + 2]) * inv, __uint_as_float(rr[4 * e + 3]) * inv);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + orow * D + c0);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            dst[e] = make_uint4(
                                pack_bf16(__uint_as_float(rr[8 * e]) * inv, __uint_as_float(rr[8 * e + 1]) * inv),
                                pack_bf16(__uint_as_float(rr[8 * e + 2]) * inv, __uint_as_float(rr[8 * e + 3]) * inv),
                                pack_bf16(__uint_as_float(rr[8 * e + 4]) * inv, __uint_as_float(rr[8 * e + 5]) * inv),
                                pack_bf16(__uint_as_float(rr[8 * e + 6]) * inv, __uint_as_float(rr[8 * e + 7]) * inv));
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0 && abort_flag) atomicOr(&g_prefill_error, kDevErrTimeout);
    if (warp == 2) tmem_dealloc(tmem, C::kTmemCols);
}

// =========================================================================== two q-tiles
// Shared-memory / TMEM plan of the two-q-tile kernel (head_dim 64 or 128, BN = 128):
// Q_A, Q_B stay resident; K and V tiles stream through their own rings, each fed by its
// own producer thread; S_A, S_B, O_A, O_B fill the 512 TMEM columns and P_X is written
// back into the first BN/2 columns of S_X as packed bf16 pairs.  A bf16 output tile is
// staged in shared memory and written back with one TMA store per 64 columns.
template <int D, bool kQRing = false>
struct Cfg2Q {
    static constexpr int BN = 128;
    static constexpr int kQBytes = D * kBM * 2;
    static constexpr int kSlotBytes = D * BN * 2;
    static constexpr int kKSlots = (D == 128) ? 2 : 5;
    static constexpr int kVSlots = (D == 128) ? 2 : 3;
    // Q_A and Q_B; with the Q ring also the next unit's Q_A, in the place of the bf16 O
    // staging tile (O is then stored from registers)
    static constexpr int kQSlots = kQRing ? 3 : 2;
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQSlots * kQBytes;
    static constexpr int kVOff = kKOff + kKSlots * kSlotBytes;
    static constexpr int kOStOff = kVOff + kVSlots * kSlotBytes;  // bf16 O staging tile
    static constexpr int kOStBytes = kQRing ? 0 : kBM * D * 2;
    static constexpr int kSmem = kOStOff + kOStBytes;
    static constexpr int kDynBytes = kSmem + 1024;
    static constexpr int kTmemCols = 512;
    static constexpr int kThreads = 384;
    static_assert(2 * BN + 2 * D <= kTmemCols, "TMEM budget");
    static_assert(kDynBytes + 512 <= 232448, "shared memory budget");
};

// Persistent: each CTA loops over work units; a unit = query rows [256 p, 256 p + 256) of
// one head, as tiles A (first 128 rows) and B.  TMEM and the barriers are set up once.
// Warp 0: K producer; warp 2 (also the TMEM owner): Q and V producer (the next unit's
// Q_A, Q_B once the current unit's last S products are done, and every unit's V tiles);
// warps 1 / 3: MMA issuers of tile A / B; warps 4-7 / 8-11: softmax of tile A / B
// (thread = row = TMEM lane), which also run the unit's epilogue.  Packed sequences take
// the Q tiles through a three-slot ring instead, loaded by the K producer (below).  Per KV tile j the
// issuer of tile X runs  O_X += P_X(j-1) V(j-1)  then  S_X = Q_X K(j)^T, so while one
// softmax warpgroup works on its scores the tensor pipe holds the other tile's products.
// P_X(j-1) lives in S_X's TMEM columns; the product that reads it is issued before the one
// that overwrites S_X by the same thread, and one thread's products run in issue order on
// the tensor pipe.  The first PV of a unit into O_X waits until the previous unit's
// epilogue has read O_X out of TMEM.
template <int D, bool kPacked>
__global__ void __launch_bounds__(384, 1) prefill2q_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_out,
    const PrefillParams p) {
    constexpr bool kRing = kPacked;  // the three-slot Q ring
    using C = Cfg2Q<D, kRing>;
    constexpr int BN = C::BN;
    constexpr int NK = C::kKSlots;
    constexpr int NV = C::kVSlots;
    constexpr int NQ = C::kQSlots;
    extern __shared__ uint8_t dyn_smem[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t q_full[NQ], q_empty[NQ], k_full[NK], k_empty[NK], v_full[NV], v_empty[NV];
    __shared__ uint64_t s_full[2], p_full[2], o_done[2], o_free[2], mma_drain, stage_free;
    __shared__ uint64_t turn[2];  // MMA issue turns of tiles A and B
    __shared__ uint64_t unit_full[4], unit_empty[4];  // the ring of units drawn at run time
    __shared__ int unit_ring[4];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int npairs = (p.nqt + 1) / 2;
    const int G = gridDim.x, cta = blockIdx.x;

    // The units of this CTA, in order.  Fixed: the zig-zag over the work list.  Drawn at run
    // time (packed sequences with a counter): warp 0 (the K producer, which runs furthest
    // ahead) takes the next unit from the counter and passes it to the other eleven warps
    // through a 4-slot ring, which they read in the same order.  A wait that gives up returns
    // INT_MAX with ok cleared.
    const bool drawn = kPacked && p.unit_counter != nullptr;
    auto draw_unit = [&](int r, bool& ok) -> int {  // warp 0, lane 0
        if (!drawn) return zigzag_unit(cta, r, G);
        const int slot = r & 3;
        if (r >= 4 && !mbar_wait(&unit_empty[slot], ((r >> 2) - 1) & 1,
                                 reinterpret_cast<volatile int*>(&abort_flag))) {
            ok = false;
            return INT_MAX;
        }
        const int w = atomicAdd(p.unit_counter, 1);
        unit_ring[slot] = w;
        mbar_arrive(&unit_full[slot]);
        return w;
    };
    auto read_unit = [&](int r, bool one_lane, bool& ok) -> int {  // the other warps
        if (!drawn) return zigzag_unit(cta, r, G);
        const int slot = r & 3;
        bool got = mbar_wait(&unit_full[slot], (r >> 2) & 1, reinterpret_cast<volatile int*>(&abort_flag));
        if (!one_lane) got = __all_sync(0xffffffffu, got);
        if (!got) {
            ok = false;
            return INT_MAX;
        }
        const int w = unit_ring[slot];
        if (!one_lane) __syncwarp();
        if (one_lane || lane == 0) mbar_arrive(&unit_empty[slot]);
        return w;
    };

    struct Unit {
        int bh, kvz, u0, u1;
        bool has_b;
        TileRange t[2];
    };
    auto unit_at = [&](int w) -> Unit {
        Unit u;
        int pair = npairs - 1 - w / p.nbh;
        if constexpr (kPacked)
            if (p.order) {
                pair = __ldg(p.order + w / p.nbh);
                if (pair < 0 || pair >= npairs) pair = npairs;  // never trust an index: no work
            }
        u.bh = w % p.nbh;
        const int bidx = u.bh / p.hq, h = u.bh % p.hq;
        u.kvz = bidx * p.hkv + h / p.group;
        u.t[0] = tile_range<BN, kPacked>(p, 2 * pair);
        u.t[1] = tile_range<BN, kPacked>(p, 2 * pair + 1);  // rows <= 0 (past sq) gives n = 0
        u.has_b = u.t[1].rows > 0;
        u.u0 = INT_MAX;
        u.u1 = INT_MIN;
        for (int x = 0; x < 2; ++x)
            if (u.t[x].n > 0) {
                u.u0 = min(u.u0, u.t[x].kt0);
                u.u1 = max(u.u1, u.t[x].kt0 + u.t[x].n);
            }
        if (u.u1 <= u.u0) u.u0 = u.u1 = 0;
        return u;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < NQ; ++i) {
            mbar_init(&q_full[i], 1);   // the slot's Q tile (Q_A / Q_B without the ring) landed
            mbar_init(&q_empty[i], 1);  // its tile's last S product of the unit done
        }
        for (int i = 0; i < NK; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 2);
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 2);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 128);
            mbar_init(&o_done[i], 1);
            mbar_init(&o_free[i], 128);
        }
        mbar_init(&mma_drain, 2);
        mbar_init(&stage_free, 1);
        mbar_init(&turn[0], 1);
        mbar_init(&turn[1], 1);
        mbar_arrive(&turn[0]);  // tile A takes the first turn
        for (int i = 0; i < 4; ++i) {
            mbar_init(&unit_full[i], 1);    // warp 0 wrote the slot
            mbar_init(&unit_empty[i], 11);  // warps 1-11 read it
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(&tmem_base_sh, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp < 4) {
        regs_dec<kRegsLow>();
        if ((warp == 0 || warp == 2) && lane == 0) {
            // ---------------------------------------------- K producer / Q + V producer
            // K(j) streams through its own ring so it never waits behind a V slot; the V
            // producer also loads each unit's Q tiles once every S of the previous unit is
            // done (V(u0) is needed only after S(u0) and its softmax, so it can wait).
            // With the Q ring (packed sequences) the K producer loads them, before the
            // unit's K tiles, in load order Q_A, Q_B of each unit: load n waits only until
            // load n - 3's tile has had its last S product, so the next unit's Q_A lands
            // while the current unit still has K tiles to go.  Packed units are short and
            // many: 972 -> 999 TFLOP/s on 16 sequences (A/B, bit-identical); the 32K causal
            // prefill lost 1 % with the ring, so the fixed-head kernel keeps two slots.
            // Only tiles with KV tiles get a Q load.  An issuer waits on a ring slot by
            // phase parity, which is sound only once the slot's previous load has landed;
            // when that load was the other tile's, the turns both issuers take in its unit
            // order this wait after the other issuer's, and a unit takes turns only when
            // one of its tiles has products.
            const bool is_k = warp == 0;
            const bool loads_q = kRing ? is_k : !is_k;
            const int ns = is_k ? NK : NV;
            uint64_t* full = is_k ? k_full : v_full;
            uint64_t* empty = is_k ? k_empty : v_empty;
            const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
            uint8_t* ring = sm + (is_k ? C::kKOff : C::kVOff);
            tma_prefetch_desc(tm);
            if (loads_q) tma_prefetch_desc(&tm_q);
            int L = 0;           // tiles issued so far into this ring
            int nq[2] = {0, 0};  // Q_A / Q_B loads issued (two slots)
            int nql = 0;         // Q tiles issued (the ring)
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int w = is_k ? draw_unit(r, ok) : read_unit(r, true, ok);
                if (!ok || w >= p.nunits) break;
                const Unit u = unit_at(w);
                if (loads_q) {
                    if constexpr (kRing) {
                        for (int x = 0; x < (u.has_b ? 2 : 1); ++x) {
                            if (u.t[x].n == 0) continue;  // no product reads this tile's Q
                            const int qs = nql % NQ;
                            if (nql >= NQ && !wait_or_abort(&q_empty[qs], ((nql / NQ) - 1) & 1, &abort_flag)) {
                                ok = false;
                                break;
                            }
                            mbar_arrive_expect_tx(&q_full[qs], C::kQBytes);
#pragma unroll
                            for (int dc = 0; dc < D / 64; ++dc)
                                tma_load_3d(sm + C::kQOff + qs * C::kQBytes + dc * (kBM * 128), &tm_q,
                                            dc * 64, u.t[x].q0, u.bh, &q_full[qs]);
                            ++nql;
                        }
                    } else {
                        // Q_X is reloaded as soon as tile X's last S of the previous unit is
                        // done (tile A's KV range ends a tile before B's, so Q_A comes back first)
                        for (int x = 0; ok && x < (u.has_b ? 2 : 1); ++x) {
                            if (nq[x] > 0 && !wait_or_abort(&q_empty[x], (nq[x] - 1) & 1, &abort_flag)) {
                                ok = false;
                                break;
                            }
                            ++nq[x];
                            mbar_arrive_expect_tx(&q_full[x], C::kQBytes);
#pragma unroll
                            for (int dc = 0; dc < D / 64; ++dc)
                                tma_load_3d(sm + C::kQOff + x * C::kQBytes + dc * (kBM * 128), &tm_q,
                                            dc * 64, u.t[x].q0, u.bh, &q_full[x]);
                        }
                    }
                    if (!ok) break;
                }
                for (int j = u.u0; j < u.u1; ++j, ++L) {
                    const int slot = L % ns;
                    if (L >= ns && !wait_or_abort(&empty[slot], ((L / ns) - 1) & 1, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[slot], C::kSlotBytes);
#pragma unroll
                    for (int dc = 0; dc < D / 64; ++dc)
                        tma_load_3d(ring + slot * C::kSlotBytes + dc * (BN * 128), tm, dc * 64, j * BN,
                                    u.kvz, &full[slot]);
                }
            }
            if (abort_flag) {  // let copies in flight land before the CTA exits
                for (int i = max(0, L - ns); i < L; ++i) wait_bounded(&full[i % ns], (i / ns) & 1);
                for (int x = 0; x < 2; ++x)
                    if (nq[x] > 0) wait_bounded(&q_full[x], (nq[x] - 1) & 1);
                for (int i = max(0, nql - NQ); i < nql; ++i) wait_bounded(&q_full[i % NQ], (i / NQ) & 1);
            }
        } else if (warp == 1 || warp == 3) {
            // ------------------------------------------------ MMA issuers, one per Q tile
            // Tile A's products come from warp 1 and tile B's from warp 3, taking turns per KV
            // tile (a token passed through the turn barriers keeps the pipe order
            // PV_A S_A | PV_B S_B | ...): each issuer does its waits while the other one
            // issues, then its turn's products back to back.  The whole warp runs this code,
            // waits included, and one elected lane issues (the warp-collective forms of
            // attn_ptx.cuh), so the issue keeps the pipe's rate while the softmax warps on the
            // same sub-partitions run.  (Waits polled by lane 0 alone, with the verdict passed
            // on by shuffle, made the kernel 2-3x slower in this form; every lane polling
            // gave 2K 731 -> 760 and 32K 1474 -> 1553 TFLOP/s against the lane-0 issuer.)
            // K and V slots are released once both issuers have arrived (count-2 barriers).
            const int x = warp == 1 ? 0 : 1;
            constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, BN, 0, 0);
            constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, D, 0, 1);
            const uint64_t qd0 = sw128_desc(smem_u32(sm + C::kQOff), 16, 1024);
            const uint64_t kd0 = sw128_desc(smem_u32(sm + C::kKOff), 16, 1024);
            const uint64_t vd0 = sw128_desc(smem_u32(sm + C::kVOff), BN * 128, 1024);
            const uint32_t tm_sx = tmem + (x ? (uint32_t)BN : 0u);
            const uint32_t tm_ox = tmem + (uint32_t)(2 * BN) + (x ? (uint32_t)D : 0u);
            uint64_t* const sfull = &s_full[x];
            uint64_t* const pfull = &p_full[x];
            int Lbase = 0;  // ring index (K and V alike) of the unit's first tile
            int cnt = 0;    // S products of this tile issued so far (phase of s/p_full)
            int turns = 0;  // turns taken so far (phase of turn[x])
            int nq = 0;     // units with a tile X so far (phase of q_full[x], two slots)
            int nql = 0;    // Q loads of earlier units (the ring's load order: A, then B)
            int uo = 0;     // units in which tile X had products so far (phase of o_free[x])
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int w = read_unit(r, false, ok);
                if (!ok || w >= p.nunits) break;
                const Unit u = unit_at(w);
                const TileRange t = x ? u.t[1] : u.t[0];
                const bool has_x = x == 0 || u.has_b;  // tile X exists in this unit
                int qs = x, qpar = nq & 1;              // Q_X's slot and its phase
                bool wait_q = has_x;                    // Q_X has a load to wait for
                if constexpr (kRing) {
                    // the ring loads Q only for tiles with KV tiles
                    const bool load_a = u.t[0].n > 0, load_b = u.has_b && u.t[1].n > 0;
                    const int nqx = nql + ((x == 1 && load_a) ? 1 : 0);
                    qs = nqx % NQ;
                    qpar = (nqx / NQ) & 1;
                    wait_q = x ? load_b : load_a;
                    nql += (load_a ? 1 : 0) + (load_b ? 1 : 0);
                }
                const uint64_t qd = desc_add(qd0, (uint32_t)(qs * C::kQBytes));
                if (wait_q) {
                    if (!__all_sync(0xffffffffu, wait_or_abort(&q_full[qs], qpar, &abort_flag))) break;
                    ++nq;
                    if (!kRing && t.n == 0) tc_commit_w(&q_empty[qs]);  // no product will read Q_X
                }
                // O_X may be overwritten once the epilogue has read out the previous unit
                // in which tile X had products (o_free completes once per such unit, so it
                // can never run two phases ahead of this wait)
                bool freed = uo == 0;
                const int cbase = cnt;
                const int nu = u.u1 - u.u0;
                for (int j = u.u0; ok && j <= u.u1 && nu > 0; ++j) {
                    const int Lk = Lbase + (j - u.u0), Lv = Lk - 1;  // K(j), V(j-1)
                    const bool have_k = j < u.u1, have_v = j > u.u0;
                    const bool in_k = have_k && j >= t.kt0 && j < t.kt0 + t.n;
                    const bool in_v = have_v && j - 1 >= t.kt0 && j - 1 < t.kt0 + t.n;
                    const int ks = Lk % NK, vs = (Lv + NV) % NV;
                    const int i = (j - 1) - t.kt0;  // index of V(j-1) within this tile's range
                    // everything this turn's products need, before taking the turn; P_X(j-1),
                    // which the softmax finishes last, is waited for last, so that the turn
                    // starts one barrier round trip after it
                    bool okw = true;
                    if (have_v) okw = wait_or_abort(&v_full[vs], (Lv / NV) & 1, &abort_flag);
                    if (okw && in_v && !freed) okw = wait_or_abort(&o_free[x], (uo - 1) & 1, &abort_flag);
                    if (okw && have_k) okw = wait_or_abort(&k_full[ks], (Lk / NK) & 1, &abort_flag);
                    if (okw) okw = wait_or_abort(&turn[x], turns & 1, &abort_flag);
                    if (okw && in_v) okw = wait_or_abort(pfull, (cbase + i) & 1, &abort_flag);
                    ok = __all_sync(0xffffffffu, okw);
                    if (!ok) break;
                    if (in_v) freed = true;
                    ++turns;
                    tc_fence_after();
                    if (in_v) {
                        // O_X += P_X(j-1) V(j-1)
                        const uint64_t vd = desc_add(vd0, (uint32_t)(vs * C::kSlotBytes));
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk)
                            tc_mma_ts_w(tm_ox, tm_sx + kk * 8, desc_add(vd, kk * 16 * 128),
                                        idesc_o, (i > 0 || kk > 0) ? 1u : 0u);
                    }
                    if (in_k) {
                        // S_X = Q_X K(j)^T
                        const uint64_t kd = desc_add(kd0, (uint32_t)(ks * C::kSlotBytes));
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off_a = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
                            const uint32_t off_b = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
                            tc_mma_ss_w(tm_sx, desc_add(qd, off_a), desc_add(kd, off_b),
                                        idesc_s, kk > 0 ? 1u : 0u);
                        }
                    }
                    mbar_arrive_w(&turn[x ^ 1]);  // the other tile's turn
                    if (in_k) {
                        tc_commit_w(sfull);
                        ++cnt;
                    }
                    if (in_v && i == t.n - 1) tc_commit_w(&o_done[x]);  // the unit's last into O_X
                    // this tile is done with V(j-1) and K(j) once the products above finish
                    // (or at once if it never reads them)
                    if (have_v) {
                        if (in_v) tc_commit_w(&v_empty[vs]);
                        else mbar_arrive_w(&v_empty[vs]);
                    }
                    if (have_k) {
                        if (in_k) tc_commit_w(&k_empty[ks]);
                        else mbar_arrive_w(&k_empty[ks]);
                    }
                    if (in_k && j == t.kt0 + t.n - 1) tc_commit_w(&q_empty[qs]);  // last S of tile X
                }
                if (t.n > 0) ++uo;
                Lbase += nu;
            }
            tc_commit_w(&mma_drain);
            wait_bounded(&mma_drain, 0);
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        regs_inc<kRegsHigh>();
        const int x = (warp >> 2) - 1;  // 0: tile A, 1: tile B
        const int row = (warp & 3) * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tm_s = tmem + lane_off + (x ? (uint32_t)BN : 0u);
        const uint32_t tm_o = tmem + lane_off + (uint32_t)(2 * BN) + (x ? (uint32_t)D : 0u);
        uint64_t* sfull = x ? &s_full[1] : &s_full[0];
        uint64_t* pfull = x ? &p_full[1] : &p_full[0];
        uint64_t* odone = x ? &o_done[1] : &o_done[0];
        uint64_t* ofree = x ? &o_free[1] : &o_free[0];
        const float c = p.c;
        const bool c_pos = c > 0.f;
        const float cm = c_pos ? c : 1.0f;  // exponent = x * cm - m
        int cnt = 0;   // S tiles consumed so far (phase of s_full)
        int ocnt = 0;  // units with at least one product into O_X (phase of o_done)
        int ebase = 0; // staged output tiles of earlier units (order: A then B per unit)
        const bool store_thread = (warp & 3) == 0 && lane == 0;
        bool ok = true;
        for (int r = 0;; ++r) {
            const int w = read_unit(r, false, ok);
            if (!ok || w >= p.nunits) break;
            const Unit u = unit_at(w);
            const TileRange t = x ? u.t[1] : u.t[0];
            // this tile's position in the CTA's sequence of staged output tiles
            const int eidx = ebase + ((x == 1 && u.t[0].rows > 0) ? 1 : 0);
            ebase += (u.t[0].rows > 0 ? 1 : 0) + (u.t[1].rows > 0 ? 1 : 0);
            const int q_row = t.q0 + row;
            int key_lo, key_hi;
            if constexpr (kPacked) {
                const int qrow = min(q_row, p.sq - 1);  // rows past sq are never stored
                row_key_bounds(p, qrow, row_sequence(p, qrow), key_lo, key_hi);
            } else {
                const int qpos = t.qpos_lo + row;
                key_lo = p.window > 0 ? qpos - p.window + 1 : INT_MIN;
                key_hi = p.causal ? min(qpos, p.skv - 1) : p.skv - 1;
            }
            float m_used = -INFINITY, l_sum = 0.f;
            for (int i = 0; ok && i < t.n; ++i, ++cnt) {
                if (!wait_or_abort(sfull, cnt & 1, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int k0 = (t.kt0 + i) * BN;
                const bool edge =
                    kPacked ? (k0 < t.all_lo || k0 + BN - 1 > t.all_hi)
                            : ((p.causal && k0 + BN - 1 > t.qpos_lo) || (k0 + BN > p.skv) ||
                               (p.window > 0 && k0 < t.qpos_hi - p.window + 1));
                // S row of this tile from TMEM, scaled for scale <= 0, then masked (edge tiles;
                // a masked key is -inf whatever the sign of the scale)
                auto load_s = [&](float* v) {
                    uint32_t rr[BN];
                    tmem_ld128(tm_s, rr);
#pragma unroll
                    for (int e = 0; e < BN; ++e) v[e] = __uint_as_float(rr[e]);
                    if (!c_pos) {
#pragma unroll
                        for (int e = 0; e < BN; ++e) v[e] *= c;
                    }
                    if (edge) {
#pragma unroll
                        for (int e = 0; e < BN; ++e) {
                            const int key = k0 + e;
                            if (key < key_lo || key > key_hi) v[e] = -INFINITY;
                        }
                    }
                };
                // P = 2^(v * cm - m_e) packed to bf16 pairs; returns its row sum
                auto exps = [&](const float* v, float m_e, uint32_t* pk) -> float {
                    float ls[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) ls[e] = 0.f;
#pragma unroll
                    for (int e = 0; e < BN / 2; ++e) {
                        float a0, a1;
                        ffma2(a0, a1, v[2 * e], v[2 * e + 1], cm, cm, -m_e, -m_e);
                        const float p0 = ex2(a0), p1 = ex2(a1);
                        fadd2(ls[(2 * e) & 7], ls[(2 * e + 1) & 7], ls[(2 * e) & 7], ls[(2 * e + 1) & 7], p0, p1);
                        pk[e] = pack_bf16(p0, p1);
                    }
                    return ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
                };
                auto reduce8 = [](const float* mx) {
                    return fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                };
                // O_X *= alpha in TMEM (the unit's previous PVs have finished: S_X(i) was
                // issued after them)
                auto rescale_o = [&](float alpha) {
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t rr[32];
                        tmem_ld32(tm_o + c0, rr);
#pragma unroll
                        for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
                        tmem_st32(tm_o + c0, rr);
                    }
                };
                uint32_t pk[BN / 2];
                float l_tile = 0.f;
                bool redo = __any_sync(0xffffffffu, m_used == -INFINITY);
                if (!redo) {
                    // Common case: one pass of exponents against the running max m_used.  The
                    // row's max grew by more than 2^kRescaleLog2 exactly when some exponent
                    // exceeds 2^kRescaleLog2, which is read off the packed bf16 values (an
                    // unsigned 16-bit max orders non-negative bf16 values by size).
                    float v[BN];
                    load_s(v);
                    float ls[8];
                    uint32_t pmax = 0u;
#pragma unroll
                    for (int e = 0; e < 8; ++e) ls[e] = 0.f;
#pragma unroll
                    for (int e = 0; e < BN / 2; ++e) {
                        float a0, a1;
                        ffma2(a0, a1, v[2 * e], v[2 * e + 1], cm, cm, -m_used, -m_used);
                        const float p0 = ex2(a0), p1 = ex2(a1);
                        fadd2(ls[(2 * e) & 7], ls[(2 * e + 1) & 7], ls[(2 * e) & 7], ls[(2 * e + 1) & 7], p0, p1);
                        pk[e] = pack_bf16(p0, p1);
                        pmax = __vmaxu2(pmax, pk[e]);
                    }
                    l_tile = ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
                    constexpr uint32_t kTwoPow8 = 0x4380u;  // bf16 bits of 2^kRescaleLog2 = 256
                    const bool big = (pmax & 0xFFFFu) > kTwoPow8 || (pmax >> 16) > kTwoPow8;
                    redo = __any_sync(0xffffffffu, big);
                }
                if (redo) {
                    // First tile of a row, or its max grew by more than 2^kRescaleLog2: take the
                    // exact tile max from S (still in TMEM: P has not been written over it),
                    // rescale O and l where the max moved, and recompute the exponents.
                    float v[BN];
                    load_s(v);
                    float mx[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
#pragma unroll
                    for (int e = 0; e < BN; ++e) mx[e & 7] = fmaxf(mx[e & 7], v[e]);
                    float tmax = reduce8(mx);
                    if (c_pos) tmax *= c;  // -inf stays -inf
                    const float m_new = fmaxf(m_used, tmax);
                    const bool need = (m_used != -INFINITY) && (m_new > m_used + kRescaleLog2);
                    if (__any_sync(0xffffffffu, need)) {
                        const float alpha = need ? ex2(m_used - m_new) : 1.0f;
                        rescale_o(alpha);
                        if (need) l_sum *= alpha;
                    }
                    if (m_used == -INFINITY || need) m_used = m_new;  // nothing accumulated yet
                    l_tile = exps(v, (m_used == -INFINITY) ? 0.f : m_used, pk);
                }
                l_sum += l_tile;
                tmem_st64(tm_s, pk);  // P_X over the first BN/2 columns of S_X
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(pfull);
            }
            // ------------------------------------------------------------ epilogue
            bool have_o = false;
            if (t.n > 0) {
                have_o = ok && wait_or_abort(odone, ocnt & 1, &abort_flag);
                ++ocnt;
                tc_fence_after();
            }
            const bool row_valid = t.rows > 0 && row < t.rows;
            const bool live = have_o && l_sum > 0.f;
            float inv, lse_v;
            finish_row(live, m_used, l_sum, p.sink ? p.sink[u.bh % p.hq] : -INFINITY, inv, lse_v);
            const size_t orow = (size_t)u.bh * p.sq + q_row;
            if (row_valid && p.lse != nullptr) p.lse[orow] = lse_v;
            if (!p.o_f32) {
                // bf16: O_X -> registers (then O_X is free), scale, stage in shared memory in
                // the 128-byte-swizzled box layout, and one thread stores the boxes with TMA
                // (rows past sq are clipped by the store).  With the Q ring there is no
                // staging tile: each thread stores its row (rows past sq are not stored).
                uint32_t ob[D / 2];
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t rr[32];
                    if (t.n > 0) {
                        tmem_ld32(tm_o + c0, rr);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) rr[e] = 0u;
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        ob[c0 / 2 + e] = pack_bf16(__uint_as_float(rr[2 * e]) * inv,
                                                   __uint_as_float(rr[2 * e + 1]) * inv);
                }
                tc_fence_before();
                if (t.n > 0) mbar_arrive(ofree);  // O_X read out: the next unit may overwrite it
                if constexpr (kRing) {
                    if (row_valid) {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + orow * D);
#pragma unroll
                        for (int ch = 0; ch < D / 8; ++ch)
                            dst[ch] = make_uint4(ob[4 * ch], ob[4 * ch + 1], ob[4 * ch + 2], ob[4 * ch + 3]);
                    }
                } else if (t.rows > 0) {
                    if (eidx > 0) ok = wait_or_abort(&stage_free, (eidx - 1) & 1, &abort_flag) && ok;
                    uint8_t* st = sm + C::kOStOff;
#pragma unroll
                    for (int ch = 0; ch < D / 8; ++ch) {
                        const uint32_t off = (ch >> 3) * (kBM * 128) + sw128_off(row, ch & 7);
                        *reinterpret_cast<uint4*>(st + off) =
                            make_uint4(ob[4 * ch], ob[4 * ch + 1], ob[4 * ch + 2], ob[4 * ch + 3]);
                    }
                    fence_proxy_async_smem();
                    if (x == 0)
                        asm volatile("bar.sync 1, 128;" ::: "memory");
                    else
                        asm volatile("bar.sync 2, 128;" ::: "memory");
                    if (store_thread) {
#pragma unroll
                        for (int dc = 0; dc < D / 64; ++dc)
                            tma_store_3d(&tm_out, st + dc * (kBM * 128), dc * 64, t.q0, u.bh);
                        bulk_commit();
                        bulk_wait_read0();  // the staging tile may be reused once read
                        mbar_arrive(&stage_free);
                    }
                }
            } else {
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t rr[32];
                    if (t.n > 0) {
                        tmem_ld32(tm_o + c0, rr);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) rr[e] = 0u;
                    }
                    if (!row_valid) continue;
                    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow * D + c0);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[e] = make_float4(__uint_as_float(rr[4 * e]) * inv, __uint_as_float(rr[4 * e + 1]) * inv,
                                             __uint_as_float(rr[4 * e + 2]) * inv, __uint_as_float(rr[4 * e + 3]) * inv);
                }
                tc_fence_before();
                if (t.n > 0) mbar_arrive(ofree);  // O_X read out: the next unit may overwrite it
            }
        }
        if (store_thread) bulk_wait0();  // every staged tile has reached global memory
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0 && abort_flag) atomicOr(&g_prefill_error, kDevErrTimeout);
    if (warp == 2) tmem_dealloc(tmem, C::kTmemCols);
}

// Streaming multiprocessors of the current device (cached per device).
int num_sms() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 148;
    }
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 148;
        }
        cached[dev] = n;
    }
    return cached[dev];
}

// Writes the packed work order into `order` (nu <= kOrderMax ints) on the stream.
template <int BN, int kTilesPerUnit>
bool unit_order_launch(const PrefillParams& p, int nu, int* order, int* counter,
                       cudaStream_t stream) {
    static std::atomic<unsigned long long> attr_done{0};
    if (needs_setup(attr_done)) {
        if (cudaFuncSetAttribute(unit_order_kernel<BN, kTilesPerUnit>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kOrderMax * (int)sizeof(unsigned long long)) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        mark_setup(attr_done);
    }
    int n2 = 1;
    while (n2 < nu) n2 <<= 1;
    unit_order_kernel<BN, kTilesPerUnit><<<1, kOrderThreads, n2 * sizeof(unsigned long long), stream>>>(
        p, nu, order, counter);
    return cudaGetLastError() == cudaSuccess;
}

template <int D, bool kPacked>
attn_status prefill_wide_launch(const PrefillArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const PrefillParams& p, cudaStream_t stream) {
    using C = CfgW<D>;
    static std::atomic<unsigned long long> attr_done{0};
    if (needs_setup(attr_done)) {
        if (cudaFuncSetAttribute(prefill_wide_kernel<D, kPacked>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kDynBytes) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        // setmaxnreg.inc waits until the launch's register pool can serve it; the split is
        // sized for exactly kRegsLaunch4 registers per thread at launch.
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, prefill_wide_kernel<D, kPacked>) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        if (fa.numRegs != kRegsLaunch4) return ATTN_ERR_UNSUPPORTED;
        mark_setup(attr_done);
    }
    const long long units = (long long)p.nqt * a.b * a.hq;
    if (units > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    PrefillParams pp = p;
    pp.nunits = (int)units;
    if constexpr (kPacked) {
        if (a.order && p.nqt <= kOrderMax) {
            if (!unit_order_launch<C::BN, 1>(p, p.nqt, a.order, nullptr, stream)) return ATTN_ERR_CUDA;
            pp.order = a.order;
        }
    }
    const int grid = (int)(units < num_sms() ? units : num_sms());
    prefill_wide_kernel<D, kPacked><<<grid, C::kThreads, C::kDynBytes, stream>>>(tq, tk, tv, pp);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

template <int D, bool kPacked>
attn_status prefill2q_launch(const PrefillArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                             const CUtensorMap& tv, const PrefillParams& p, cudaStream_t stream) {
    using C = Cfg2Q<D, kPacked>;
    static std::atomic<unsigned long long> attr_done{0};
    if (needs_setup(attr_done)) {
        if (cudaFuncSetAttribute(prefill2q_kernel<D, kPacked>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kDynBytes) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        // setmaxnreg.inc waits until the launch's register pool can serve it; the split is
        // sized for exactly kRegsLaunch3 registers per thread at launch.
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, prefill2q_kernel<D, kPacked>) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        if (fa.numRegs != kRegsLaunch3) return ATTN_ERR_UNSUPPORTED;
        mark_setup(attr_done);
    }
    const long long units = (long long)((p.nqt + 1) / 2) * a.b * a.hq;
    if (units > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    PrefillParams pp = p;
    pp.nunits = (int)units;
    if constexpr (kPacked) {
        const int npairs = (p.nqt + 1) / 2;
        if (a.order && npairs <= kOrderMax) {
            // the counter sits after the order (the scratch holds one int per query tile)
            int* counter = p.nqt >= npairs + 1 ? a.order + npairs : nullptr;
            if (!unit_order_launch<C::BN, 2>(p, npairs, a.order, counter, stream)) return ATTN_ERR_CUDA;
            pp.order = a.order;
            pp.unit_counter = counter;
        }
    }
    const int grid = (int)(units < num_sms() ? units : num_sms());
    CUtensorMap to;  // bf16 O for the TMA stores (unused, never dereferenced, for fp32 O)
    if (a.o_dtype == ATTN_BF16) {
        uint64_t od[3] = {(uint64_t)D, (uint64_t)a.sq, (uint64_t)a.b * a.hq};
        uint64_t os[2] = {(uint64_t)D * 2, (uint64_t)a.sq * D * 2};
        uint32_t ob[3] = {64u, (uint32_t)kBM, 1u};
        if (!make_bf16_map(&to, a.o, 3, od, os, ob)) return ATTN_ERR_CUDA;
    } else {
        to = tq;
    }
    prefill2q_kernel<D, kPacked><<<grid, C::kThreads, C::kDynBytes, stream>>>(tq, tk, tv, to, pp);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

template <int D>
attn_status prefill_launch_d(const PrefillArgs& a, cudaStream_t stream) {
    constexpr int BN = (D <= 128) ? Cfg2Q<(D <= 128 ? D : 128)>::BN : CfgW<(D > 128 ? D : 256)>::BN;
    CUtensorMap tq, tk, tv;
    const uint64_t skv = a.skv > 0 ? (uint64_t)a.skv : 1u;
    uint64_t qd[3] = {(uint64_t)D, (uint64_t)a.sq, (uint64_t)a.b * a.hq};
    uint64_t qs[2] = {(uint64_t)D * 2, (uint64_t)a.sq * D * 2};
    uint32_t qb[3] = {64u, (uint32_t)kBM, 1u};
    uint64_t kd[3] = {(uint64_t)D, skv, (uint64_t)a.b * a.hkv};
    uint64_t ks[2] = {(uint64_t)D * 2, skv * D * 2};
    uint32_t kb[3] = {64u, (uint32_t)BN, 1u};
    const void* kp = a.skv > 0 ? a.k : a.q;  // never read when skv == 0
    const void* vp = a.skv > 0 ? a.v : a.q;
    if (!make_bf16_map(&tq, a.q, 3, qd, qs, qb) || !make_bf16_map(&tk, kp, 3, kd, ks, kb) ||
        !make_bf16_map(&tv, vp, 3, kd, ks, kb))
        return ATTN_ERR_CUDA;
    PrefillParams p;
    p.o = a.o;
    p.lse = a.lse;
    p.sink = a.sink;
    p.cu_q = a.cu_seqlens_q;
    p.cu_k = a.cu_seqlens_k;
    p.nseq = a.nseq;
    p.order = nullptr;
    p.unit_counter = nullptr;
    p.hq = a.hq;
    p.hkv = a.hkv;
    p.sq = a.sq;
    p.skv = a.skv;
    p.group = a.hq / a.hkv;
    p.nqt = (a.sq + kBM - 1) / kBM;
    p.window = a.window;
    p.causal = a.causal;
    p.o_f32 = a.o_dtype == ATTN_F32 ? 1 : 0;
    p.c = a.scale * kLog2e;
    p.nbh = a.b * a.hq;
    p.nunits = 0;
    if constexpr (D <= 128)
        return p.cu_q ? prefill2q_launch<D, true>(a, tq, tk, tv, p, stream)
                      : prefill2q_launch<D, false>(a, tq, tk, tv, p, stream);
    else
        return p.cu_q ? prefill_wide_launch<D, true>(a, tq, tk, tv, p, stream)
                      : prefill_wide_launch<D, false>(a, tq, tk, tv, p, stream);
}

}  // namespace

attn_status prefill_launch(const PrefillArgs& a, cudaStream_t stream) {
    switch (a.d) {
        case 64: return prefill_launch_d<64>(a, stream);
        case 128: return prefill_launch_d<128>(a, stream);
        case 256: return prefill_launch_d<256>(a, stream);
        default: return ATTN_ERR_UNSUPPORTED;
    }
}

unsigned prefill_take_error(cudaStream_t stream, cudaError_t* err) {
    unsigned v = 0, zero = 0;
    *err = cudaMemcpyFromSymbolAsync(&v, g_prefill_error, sizeof v, 0, cudaMemcpyDeviceToHost, stream);
    if (*err == cudaSuccess)
        *err = cudaMemcpyToSymbolAsync(g_prefill_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice,
                                       stream);
    if (*err == cudaSuccess) *err = cudaStreamSynchronize(stream);
    if (*err != cudaSuccess) cudaGetLastError();
    return v;
}

}  // namespace attn
