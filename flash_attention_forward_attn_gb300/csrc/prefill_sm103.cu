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
// GB300 design (one CTA per 128-row query tile of one head, 8 warps):
//   warp 0    TMA producer: Q once, then K and V tiles through two 2-deep rings.
//   warp 1    MMA issuer (one thread): S = Q K^T into TMEM (double-buffered), then
//             O += P V into a TMEM accumulator that lives for the whole KV pass.
//   warp 2    owns the TMEM allocation.
//   warps 4-7 softmax: thread = query row = TMEM lane.  Reads its S row from TMEM,
//             masks it if the tile crosses a band edge, folds scale*log2(e) into the
//             exponent, writes P (bf16) into a 128-byte-swizzled shared-memory tile for
//             the second MMA, and rescales O in TMEM only when the row max has grown by
//             more than 2^8 since the last rescale (the stale max is used consistently
//             for P and l, so O / l is unchanged).
// The accumulator never leaves TMEM until the epilogue, so no O round trip through HBM
// (the pages' sectioned design) is needed at any sequence length.
#include <float.h>

#include "attn_internal.h"
#include "attn_ptx.cuh"

namespace attn {
namespace {

__device__ unsigned g_prefill_error;

constexpr int kThreads = 256;
constexpr int kBM = 128;           // query rows per tile (= TMEM lanes)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale threshold, log2 units

template <int D>
struct PrefillCfg {
    static constexpr int BN = (D == 256) ? 64 : 128;   // keys per tile
    static constexpr int kQBytes = D * kBM * 2;        // D/64 boxes of 128 rows x 128 B
    static constexpr int kKVBytes = D * BN * 2;        // D/64 boxes of BN rows x 128 B
    static constexpr int kPBytes = BN * kBM * 2;       // BN/64 boxes of 128 rows x 128 B
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + kQBytes;
    static constexpr int kVOff = kKOff + 2 * kKVBytes;
    static constexpr int kPOff = kVOff + 2 * kKVBytes;
    static constexpr int kSmem = kPOff + 2 * kPBytes;
    static constexpr int kDynBytes = kSmem + 1024;
    static constexpr int kTmemCols = 512;
    static constexpr int kSCol = 0;                    // S buffers at columns [0, 2 BN)
    static constexpr int kOCol = 2 * BN;               // O at [2 BN, 2 BN + D)
    static_assert(2 * BN + D <= kTmemCols, "TMEM budget");
    static_assert(kDynBytes <= 232448, "shared memory budget");
};

struct PrefillParams {
    void* o;
    float* lse;
    int hq, hkv, sq, skv, group, nqt, window, causal, o_f32;
    float c;  // scale * log2(e)
};

struct TileRange {
    int q0, rows, qpos_lo, qpos_hi, kt0, n;
};

template <int BN>
__device__ __forceinline__ TileRange tile_range(const PrefillParams& p, int qt) {
    TileRange r;
    r.q0 = qt * kBM;
    r.rows = min(kBM, p.sq - r.q0);
    const int off = p.skv - p.sq;  // queries sit at the tail of the keys
    r.qpos_lo = r.q0 + off;
    r.qpos_hi = r.q0 + r.rows - 1 + off;
    const int k_end = p.causal ? min(p.skv, r.qpos_hi + 1) : p.skv;
    const int k_begin = p.window > 0 ? max(0, r.qpos_lo - p.window + 1) : 0;
    if (k_end <= k_begin) {
        r.kt0 = 0;
        r.n = 0;
    } else {
        r.kt0 = k_begin / BN;
        r.n = (k_end + BN - 1) / BN - r.kt0;
    }
    return r;
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, int* abort_flag) {
    return mbar_wait(bar, parity, reinterpret_cast<volatile int*>(abort_flag));
}

__device__ __forceinline__ void wait_bounded(uint64_t* bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitLimitCycles) return;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
    using C = PrefillCfg<D>;
    constexpr int BN = C::BN;
    extern __shared__ uint8_t dyn_smem[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t q_full, k_full[2], k_empty[2], v_full[2], v_empty[2];
    __shared__ uint64_t s_full[2], p_full[2], o_done[2], mma_drain;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nbh = gridDim.x / p.nqt;
    const int qt = p.nqt - 1 - (int)(blockIdx.x / nbh);  // heaviest causal tiles first
    const int bh = (int)(blockIdx.x % nbh);
    const int bidx = bh / p.hq, h = bh % p.hq;
    const int kvz = bidx * p.hkv + h / p.group;
    const TileRange tr = tile_range<BN>(p, qt);

    if (threadIdx.x == 0) {
        mbar_init(&q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 128);
            mbar_init(&o_done[i], 1);
        }
        mbar_init(&mma_drain, 1);
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
    const int n = tr.n;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && n > 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            mbar_arrive_expect_tx(&q_full, C::kQBytes);
#pragma unroll
            for (int dc = 0; dc < D / 64; ++dc)
                tma_load_3d(sm + C::kQOff + dc * (kBM * 128), &tm_q, dc * 64, tr.q0, bh, &q_full);
            int issued = 0;
            for (int j = 0; j < n; ++j) {
                const int s = j & 1;
                const int k0 = (tr.kt0 + j) * BN;
                if (j >= 2 && !wait_or_abort(&k_empty[s], ((j >> 1) - 1) & 1, &abort_flag)) break;
                mbar_arrive_expect_tx(&k_full[s], C::kKVBytes);
#pragma unroll
                for (int dc = 0; dc < D / 64; ++dc)
                    tma_load_3d(sm + C::kKOff + s * C::kKVBytes + dc * (BN * 128), &tm_k, dc * 64,
                                k0, kvz, &k_full[s]);
                if (j >= 2 && !wait_or_abort(&v_empty[s], ((j >> 1) - 1) & 1, &abort_flag)) {
                    issued = -(j + 1);  // K of tile j issued, V not
                    break;
                }
                mbar_arrive_expect_tx(&v_full[s], C::kKVBytes);
#pragma unroll
                for (int dc = 0; dc < D / 64; ++dc)
                    tma_load_3d(sm + C::kVOff + s * C::kKVBytes + dc * (BN * 128), &tm_v, dc * 64,
                                k0, kvz, &v_full[s]);
                issued = j + 1;
            }
            if (abort_flag) {  // let copies in flight land before the CTA exits
                wait_bounded(&q_full, 0);
                const int kdone = issued < 0 ? -issued : issued;
                const int vdone = issued < 0 ? -issued - 1 : issued;
                for (int j = max(0, kdone - 2); j < kdone; ++j) wait_bounded(&k_full[j & 1], (j >> 1) & 1);
                for (int j = max(0, vdone - 2); j < vdone; ++j) wait_bounded(&v_full[j & 1], (j >> 1) & 1);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n > 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, BN, 0, 0);
            constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, D, 0, 1);
            const uint32_t q_base = smem_u32(sm + C::kQOff);
            const uint32_t tm_o = tmem + C::kOCol;
            bool ok = wait_or_abort(&q_full, 0, &abort_flag);
            tc_fence_after();
            auto issue_s = [&](int t) -> bool {
                const int s = t & 1;
                if (!wait_or_abort(&k_full[s], (t >> 1) & 1, &abort_flag)) return false;
                tc_fence_after();
                const uint32_t k_base = smem_u32(sm + C::kKOff + s * C::kKVBytes);
                const uint32_t tm_s = tmem + C::kSCol + s * BN;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t a = sw128_desc(q_base + (kk >> 2) * (kBM * 128) + (kk & 3) * 32, 16, 1024);
                    const uint64_t b = sw128_desc(k_base + (kk >> 2) * (BN * 128) + (kk & 3) * 32, 16, 1024);
                    tc_mma_ss(tm_s, a, b, idesc_s, kk > 0 ? 1u : 0u);
                }
                tc_commit(&s_full[s]);
                tc_commit(&k_empty[s]);
                return true;
            };
            if (ok) ok = issue_s(0);
            if (ok && n > 1) ok = issue_s(1);
            for (int j = 0; ok && j < n; ++j) {
                const int s = j & 1;
                if (!wait_or_abort(&p_full[s], (j >> 1) & 1, &abort_flag)) break;
                if (!wait_or_abort(&v_full[s], (j >> 1) & 1, &abort_flag)) break;
                tc_fence_after();
                const uint32_t p_base = smem_u32(sm + C::kPOff + s * C::kPBytes);
                const uint32_t v_base = smem_u32(sm + C::kVOff + s * C::kKVBytes);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t a = sw128_desc(p_base + (kk >> 2) * (kBM * 128) + (kk & 3) * 32, 16, 1024);
                    const uint64_t b = sw128_desc(v_base + kk * (16 * 128), BN * 128, 1024);
                    tc_mma_ss(tm_o, a, b, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&o_done[s]);
                tc_commit(&v_empty[s]);
                if (j + 2 < n) ok = issue_s(j + 2);
            }
            tc_commit(&mma_drain);
            wait_bounded(&mma_drain, 0);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax
        const int row = (warp & 3) * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const int q_row = tr.q0 + row;
        const int qpos = tr.qpos_lo + row;
        const int key_lo = p.window > 0 ? qpos - p.window + 1 : INT_MIN;
        const int key_hi = p.causal ? min(qpos, p.skv - 1) : p.skv - 1;
        const float c = p.c;
        const bool c_pos = c > 0.f;
        float m_used = -INFINITY, l_sum = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const int s = j & 1;
            if (!wait_or_abort(&s_full[s], (j >> 1) & 1, &abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float x[BN];
            {
                uint32_t r[BN];
                if constexpr (BN == 128)
                    tmem_ld128(tmem + lane_off + C::kSCol + s * BN, r);
                else
                    tmem_ld64(tmem + lane_off + C::kSCol + s * BN, r);
#pragma unroll
                for (int i = 0; i < BN; ++i) x[i] = __uint_as_float(r[i]);
            }
            const int k0 = (tr.kt0 + j) * BN;
            const bool edge = (p.causal && k0 + BN - 1 > tr.qpos_lo) || (k0 + BN > p.skv) ||
                              (p.window > 0 && k0 < tr.qpos_hi - p.window + 1);
            if (edge) {
#pragma unroll
                for (int i = 0; i < BN; ++i) {
                    const int key = k0 + i;
                    if (key < key_lo || key > key_hi) x[i] = -INFINITY;
                }
            }
            // row max with 8 independent chains (a single chain is latency-bound)
            float mx[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) mx[u] = -INFINITY;
            if (!c_pos) {
#pragma unroll
                for (int i = 0; i < BN; ++i) x[i] *= c;
            }
#pragma unroll
            for (int i = 0; i < BN; ++i) mx[i & 7] = fmaxf(mx[i & 7], x[i]);
            float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
            if (c_pos) tmax *= c;  // -inf stays -inf
            // x holds raw scores when c > 0 (exponent = x*c - m), scaled scores otherwise
            const float m_new = fmaxf(m_used, tmax);
            const bool need = (m_used != -INFINITY) && (m_new > m_used + kRescaleLog2);
            if (m_used == -INFINITY) m_used = m_new;  // nothing accumulated yet for this row
            if (__any_sync(0xffffffffu, need)) {
                // O holds PV of the previous tile only after that MMA is done
                if (!wait_or_abort(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float alpha = need ? ex2(m_used - m_new) : 1.0f;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_off + C::kOCol + c0, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                    tmem_st32(tmem + lane_off + C::kOCol + c0, r);
                }
                tmem_wait_st();
                if (need) {
                    l_sum *= alpha;
                    m_used = m_new;
                }
            }
            const float m_e = (m_used == -INFINITY) ? 0.f : m_used;
            const float cm = c_pos ? c : 1.0f;  // exponent = x * cm - m_e
            uint8_t* pbuf = sm + C::kPOff + s * C::kPBytes;
            float ls[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) ls[u] = 0.f;
#pragma unroll
            for (int ch = 0; ch < BN / 8; ++ch) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p0 = ex2(fmaf(x[ch * 8 + 2 * e], cm, -m_e));
                    const float p1 = ex2(fmaf(x[ch * 8 + 2 * e + 1], cm, -m_e));
                    ls[2 * e] += p0;
                    ls[2 * e + 1] += p1;
                    pk[e] = pack_bf16(p0, p1);
                }
                const uint32_t off = (ch >> 3) * (kBM * 128) + sw128_off(row, ch & 7);
                *reinterpret_cast<uint4*>(pbuf + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            l_sum += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&p_full[s]);
        }
        // ------------------------------------------------------------ epilogue
        bool have_o = false;
        if (ok && n > 0) {
            have_o = wait_or_abort(&o_done[(n - 1) & 1], ((n - 1) >> 1) & 1, &abort_flag);
            tc_fence_after();
        }
        const bool row_valid = q_row < p.sq;
        const bool live = have_o && l_sum > 0.f;
        const float inv = live ? 1.0f / l_sum : 0.f;
        const size_t orow = (size_t)bh * p.sq + q_row;
        if (row_valid && p.lse != nullptr)
            p.lse[orow] = live ? (m_used + __log2f(l_sum)) * kLn2 : -INFINITY;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t r[32];
            if (have_o) {
                tmem_ld32(tmem + lane_off + C::kOCol + c0, r);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = 0u;
            }
            if (!row_valid) continue;
            if (p.o_f32) {
                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow * D + c0);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    dst[i] = make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                                         __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv);
            } else {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + orow * D + c0);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    dst[i] = make_uint4(
                        pack_bf16(__uint_as_float(r[8 * i]) * inv, __uint_as_float(r[8 * i + 1]) * inv),
                        pack_bf16(__uint_as_float(r[8 * i + 2]) * inv, __uint_as_float(r[8 * i + 3]) * inv),
                        pack_bf16(__uint_as_float(r[8 * i + 4]) * inv, __uint_as_float(r[8 * i + 5]) * inv),
                        pack_bf16(__uint_as_float(r[8 * i + 6]) * inv, __uint_as_float(r[8 * i + 7]) * inv));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0 && abort_flag) atomicOr(&g_prefill_error, kDevErrTimeout);
    if (warp == 2) tmem_dealloc(tmem, C::kTmemCols);
}

template <int D>
attn_status prefill_launch_d(const PrefillArgs& a, cudaStream_t stream) {
    using C = PrefillCfg<D>;
    CUtensorMap tq, tk, tv;
    const uint64_t skv = a.skv > 0 ? (uint64_t)a.skv : 1u;
    uint64_t qd[3] = {(uint64_t)D, (uint64_t)a.sq, (uint64_t)a.b * a.hq};
    uint64_t qs[2] = {(uint64_t)D * 2, (uint64_t)a.sq * D * 2};
    uint32_t qb[3] = {64u, (uint32_t)kBM, 1u};
    uint64_t kd[3] = {(uint64_t)D, skv, (uint64_t)a.b * a.hkv};
    uint64_t ks[2] = {(uint64_t)D * 2, skv * D * 2};
    uint32_t kb[3] = {64u, (uint32_t)C::BN, 1u};
    const void* kp = a.skv > 0 ? a.k : a.q;  // never read when skv == 0
    const void* vp = a.skv > 0 ? a.v : a.q;
    if (!make_bf16_map(&tq, a.q, 3, qd, qs, qb) || !make_bf16_map(&tk, kp, 3, kd, ks, kb) ||
        !make_bf16_map(&tv, vp, 3, kd, ks, kb))
        return ATTN_ERR_CUDA;
    PrefillParams p;
    p.o = a.o;
    p.lse = a.lse;
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
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kDynBytes) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        attr_set = true;
    }
    const long long grid = (long long)p.nqt * a.b * a.hq;
    if (grid > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    prefill_kernel<D><<<(unsigned)grid, kThreads, C::kDynBytes, stream>>>(tq, tk, tv, p);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
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
