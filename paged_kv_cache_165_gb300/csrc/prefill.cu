// prefill.cu -- varlen causal attention over packed prompts (cu_seqlens).
//
// Sequence b owns tokens [cu_seqlens[b], cu_seqlens[b+1]) of q/k/v (0539edu.com
// "从KV cache共享到批量调度…" §3.3).  Token t of a sequence attends to tokens 0..t of
// the same sequence (causal prefill, zwjcode.cn "KV Cache 的增量解码" §05; the mask is
// aligned so that a query at position t sees keys 0..t, §13), with query head i reading
// KV head floor(i/m) (limoncc.com "大语言模型研究15——注意力机制优化之KV缓存" §3.3).
//
// Tensor-core path (bf16, d in {64, 128}): 5th-generation tensor cores (tcgen05).  One
// CTA per (query head, 128-query tile, sequence): TMA brings the Q tile once and 64-key
// K/V tiles through a multi-stage ring (128-byte swizzle, mbarrier completion with bounded
// waits); one thread issues S = Q K^T into tensor memory (double-buffered) and O += P V
// into a tensor-memory accumulator; four warps own one query row per thread for the online
// softmax (running max and sum, plumephp.com "KV Cache 优化与注意力机制加速" §2.2-§2.3) and
// hand P back through shared memory as bf16 hi + lo parts, so the weights keep ~16 bits.
// Only key tiles at or below the diagonal are visited.
// CUDA-core path (fp32 or other d): one warp per (query row, head).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned kFull = 0xffffffffu;

struct PrefillKParams {
    float *out;
    float *lse;
    const int32_t *cu;
    unsigned *err;
    int B, T, max_seqlen, Hq, Hkv, m;
    float scale_log2;
};

// Validated [start, start+len) of sequence b; false if cu_seqlens is inconsistent.
__device__ __forceinline__ bool seq_range(const PrefillKParams &p, int b, int &start, int &len,
                                          bool report) {
    const int c0 = __ldg(p.cu + b), c1 = __ldg(p.cu + b + 1);
    if (c0 < 0 || c1 < c0 || c1 > p.T || (b == 0 && c0 != 0) || (b == p.B - 1 && c1 != p.T)) {
        if (report) raise_error(p.err, PKV_DEVERR_CU_SEQLENS);
        return false;
    }
    start = c0;
    len = c1 - c0;
    if (len > p.max_seqlen && report) raise_error(p.err, PKV_DEVERR_CU_SEQLENS);
    return true;
}

// ============================================================ tcgen05 path

// Tiles of the tcgen05 prefill: two 128-row query tiles per CTA, 64-key K/V tiles.
template <int D>
struct TcPrefillCfg {
    static constexpr int kBM = 128, kBN = 64, kGroups = 2;
    static constexpr int kStages = D == 64 ? 6 : 3;    // K/V ring depth
    static constexpr int kQBytes = kBM * D * 2;        // one Q tile: D/64 panels of [128][128 B]
    static constexpr int kKVBytes = kBN * D * 2;       // one K or V tile: D/64 panels of [64][128 B]
    static constexpr int kPBytes = kBM * kBN * 2;      // P (bf16) [128][64]: one panel
    static constexpr int kOffKV = kGroups * kQBytes;   // stage s: K, then V
    static constexpr int kOffP = kOffKV + kStages * 2 * kKVBytes;   // per group: P_hi, P_lo
    static constexpr int kOffBar = kOffP + kGroups * 2 * kPBytes;
    static constexpr int kNumBars = 1 + 2 * kStages + kGroups * 6;
    static constexpr int kSmemBytes = 1024 + kOffBar + kNumBars * 8 + 16;
    static constexpr int kTmemCols = 512;              // per group: S 2 x 64 columns, O D columns
    static constexpr int kGroupCols = 256;
    static constexpr int kSCol = 0, kOCol = 2 * kBN;
    static_assert(kOCol + D <= kGroupCols, "tensor memory budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// mbarrier slots: Q; K/V full and K/V free per stage; per group S full x2, S free x2,
// P full, O done
template <int NS>
struct PrefillBars {
    static constexpr int kQ = 0, kKvFull = 1, kKvFree = 1 + NS, kGroup0 = 1 + 2 * NS;
    static constexpr int s_full(int g, int b) { return kGroup0 + g * 6 + b; }
    static constexpr int s_free(int g, int b) { return kGroup0 + g * 6 + 2 + b; }
    static constexpr int p_full(int g) { return kGroup0 + g * 6 + 4; }
    static constexpr int o_done(int g) { return kGroup0 + g * 6 + 5; }
};

// One CTA per (query head, pair of 128-query tiles, sequence); ten warps.
//   warp 9 (one lane): TMA loads of both Q tiles and of a K/V ring shared by the two tiles;
//     a stage is refilled as soon as the MMAs of its previous tile are done.
//   warp 8 (one lane): every tcgen05.mma: per tile g and key tile j, S_g = Q_g K_j^T into one of
//     two tensor-memory S buffers of g, and O_g += P_g V_j (P as bf16 hi + lo, two MMA
//     chains) into g's tensor-memory accumulator.  Issue order alternates between the
//     tiles, so the tensor core works on one tile while the other tile's rows are in the
//     softmax.
//   warps 4g .. 4g+3: one query row of tile g per thread.  Per key tile: read the row of
//     S from tensor memory, apply the causal mask (key <= query) on diagonal tiles, update
//     the running max and sum (online softmax), rescale the O row in tensor memory when
//     the reference max grew by more than 2^8 (exponentials stay <= 256 otherwise, and O
//     and l share the same reference), and write the row of P_hi and P_lo to shared memory
//     in the 128-byte-swizzled K-major layout the MMA reads.  At the end: O / l and lse.
template <int D>
__global__ void __launch_bounds__(320, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const PrefillKParams p) {
    using Cfg = TcPrefillCfg<D>;
    constexpr int BM = Cfg::kBM, BN = Cfg::kBN, PANELS = D / 64, NS = Cfg::kStages, G = Cfg::kGroups;
    using Bars = PrefillBars<NS>;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + Cfg::kNumBars);
    volatile int *abort = reinterpret_cast<volatile int *>(tslot + 1);
    auto bar = [&](int k) { return smem_addr(&bars[k]); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x, b = blockIdx.z;
    int start = 0, len = 0;
    if (!seq_range(p, b, start, len, threadIdx.x == 0 && blockIdx.y == 0 && i == 0)) return;
    const int npairs = (p.max_seqlen + G * BM - 1) / (G * BM);
    const int q0 = (npairs - 1 - static_cast<int>(blockIdx.y)) * G * BM;   // longest first
    if (q0 >= len) return;
    const int kvh = i / p.m;
    int n_kt[G];   // key tiles up to the diagonal, per query tile (0: tile past the end)
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const int qg = q0 + g * BM;
        n_kt[g] = qg < len ? (min(qg + BM, len) - 1) / BN + 1 : 0;
    }
    const int n_all = max(n_kt[0], n_kt[1]);

    if (threadIdx.x == 0) {
        mbar_init(bar(Bars::kQ), 1);
        for (int st = 0; st < NS; ++st) {
            mbar_init(bar(Bars::kKvFull + st), 1);
            mbar_init(bar(Bars::kKvFree + st), 1);
        }
        for (int g = 0; g < G; ++g) {
            for (int sb = 0; sb < 2; ++sb) {
                mbar_init(bar(Bars::s_full(g, sb)), 1);
                mbar_init(bar(Bars::s_free(g, sb)), 4);
            }
            mbar_init(bar(Bars::p_full(g)), 4);
            mbar_init(bar(Bars::o_done(g)), 1);
        }
        *abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(smem_addr(tslot), Cfg::kTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;
    auto sQ = [&](int g) { return smem_addr(smem + g * Cfg::kQBytes); };
    auto sK = [&](int st) { return smem_addr(smem + Cfg::kOffKV + st * 2 * Cfg::kKVBytes); };
    auto sV = [&](int st) { return sK(st) + Cfg::kKVBytes; };
    auto sP = [&](int g) { return smem_addr(smem + Cfg::kOffP + g * 2 * Cfg::kPBytes); };   // hi; lo after

    if (warp == 2 * 4) {
        if (lane == 0) {
            const uint32_t idesc_s = umma_idesc_bf16(BM, BN, 0);
            const uint32_t idesc_o = umma_idesc_bf16(BM, D, 1);
            auto issue_s = [&](int g, int j) {   // S_g[j & 1] = Q_g K_j^T
                const int st = j % NS, sb = j & 1;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t ad = umma_desc_sw128(sQ(g) + (kk / 4) * BM * 128 + (kk % 4) * 32, 16, 1024);
                    const uint64_t bd = umma_desc_sw128(sK(st) + (kk / 4) * BN * 128 + (kk % 4) * 32, 16, 1024);
                    umma_bf16(tmem + g * Cfg::kGroupCols + Cfg::kSCol + sb * BN, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
                }
                umma_commit(bar(Bars::s_full(g, sb)));
            };
            auto issue_pv = [&](int g, int j) {  // O_g += P_g,hi V_j + P_g,lo V_j
                const int st = j % NS;
#pragma unroll
                for (int half = 0; half < 2; ++half)
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        const uint64_t ad = umma_desc_sw128(sP(g) + half * Cfg::kPBytes + kk * 32, 16, 1024);
                        const uint64_t bd = umma_desc_sw128(sV(st) + kk * 16 * 128, BN * 128, 1024);
                        umma_bf16(tmem + g * Cfg::kGroupCols + Cfg::kOCol, ad, bd, idesc_o,
                                  (j > 0 || half > 0 || kk > 0) ? 1u : 0u);
                    }
                umma_commit(bar(Bars::o_done(g)));
            };
            int j = 0;
            if (wait_or_abort(bar(Bars::kQ), 0, abort, p.err) &&
                wait_or_abort(bar(Bars::kKvFull), 0, abort, p.err)) {
                tc_fence_after_sync();
                for (int g = 0; g < G; ++g)
                    if (n_kt[g] > 0) issue_s(g, 0);
                bool alive = true;
                for (; j < n_all && alive; ++j) {
                    const int t = j + 1;
                    if (t < n_all) {
                        alive = wait_or_abort(bar(Bars::kKvFull + t % NS), (t / NS) & 1, abort, p.err);
                        for (int g = 0; g < G && alive; ++g) {
                            if (t >= n_kt[g]) continue;
                            if (t >= 2)
                                alive = wait_or_abort(bar(Bars::s_free(g, t & 1)), ((t >> 1) - 1) & 1, abort, p.err);
                            if (!alive) break;
                            tc_fence_after_sync();
                            issue_s(g, t);
                        }
                    }
                    for (int g = 0; g < G && alive; ++g) {
                        if (j >= n_kt[g]) continue;
                        alive = wait_or_abort(bar(Bars::p_full(g)), j & 1, abort, p.err);
                        if (!alive) break;
                        tc_fence_after_sync();
                        issue_pv(g, j);
                    }
                    if (!alive) break;
                    umma_commit(bar(Bars::kKvFree + j % NS));   // stage j % NS is free after these MMAs
                }
            }
            if (*abort && j > 0) {
                // let the MMAs already issued finish (bounded) before teardown
                umma_commit(bar(Bars::kKvFree + j % NS));
                mbar_wait_bounded(bar(Bars::kKvFree + j % NS), (j / NS) & 1);
            }
        }
    } else if (warp == 2 * 4 + 1) {
        if (lane == 0) {
            // loader: both Q tiles, then K/V tile t into stage t % NS as soon as the MMAs of
            // tile t - NS (the stage's previous tile) are done
            mbar_arrive_expect_tx(bar(Bars::kQ), G * Cfg::kQBytes);
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int pn = 0; pn < PANELS; ++pn)
                    tma_load_3d(sQ(g) + pn * BM * 128, &tm_q, pn * 64, i, start + q0 + g * BM, bar(Bars::kQ));
            int t = 0;
            for (; t < n_all; ++t) {
                if (t >= NS && !wait_or_abort(bar(Bars::kKvFree + t % NS), ((t - NS) / NS) & 1, abort, p.err))
                    break;
                const int st = t % NS;
                mbar_arrive_expect_tx(bar(Bars::kKvFull + st), 2 * Cfg::kKVBytes);
#pragma unroll
                for (int pn = 0; pn < PANELS; ++pn) {
                    tma_load_3d(sK(st) + pn * BN * 128, &tm_k, pn * 64, kvh, start + t * BN, bar(Bars::kKvFull + st));
                    tma_load_3d(sV(st) + pn * BN * 128, &tm_v, pn * 64, kvh, start + t * BN, bar(Bars::kKvFull + st));
                }
            }
            // before teardown, every copy issued must have landed (bounded)
            mbar_wait_bounded(bar(Bars::kQ), 0);
            for (int u = max(0, t - NS); u < t; ++u)
                mbar_wait_bounded(bar(Bars::kKvFull + u % NS), (u / NS) & 1);
        }
    } else {
        const int g = warp >> 2;                 // query tile of this warp
        const int r = (warp & 3) * 32 + lane;    // its row in the tile
        const int qg0 = q0 + g * BM;
        const int qpos = qg0 + r;
        const int nk = n_kt[g];
        const uint32_t lane_base = tmem + g * Cfg::kGroupCols + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        uint8_t *pbuf = smem + Cfg::kOffP + g * 2 * Cfg::kPBytes;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = nk > 0;
        for (int j = 0; j < nk && ok; ++j) {
            const int sb = j & 1;
            ok = wait_or_abort(bar(Bars::s_full(g, sb)), (j >> 1) & 1, abort, p.err);
            if (!ok) break;
            tc_fence_after_sync();
            uint32_t sr[BN];
            tmem_ld32(lane_base + Cfg::kSCol + sb * BN, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
            tmem_ld32(lane_base + Cfg::kSCol + sb * BN + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
            tmem_ld_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Bars::s_free(g, sb)));

            // causal mask (diagonal tiles only), tile max, reference max (moved only when it
            // grows by more than 2^8); scores stay raw and the scale enters one FMA
            const int key0 = j * BN;
            float sc[BN];
#pragma unroll
            for (int c = 0; c < BN; ++c) sc[c] = __uint_as_float(sr[c]);
            if (key0 + BN - 1 > qg0) {
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (key0 + c > qpos) sc[c] = -INFINITY;
            }
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < BN; ++c) mx4[c & 3] = fmaxf(mx4[c & 3], sc[c]);
            const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * p.scale_log2;
            const float m_new = mx > m_ref + 8.f ? mx : m_ref;
            const float alpha = ex2_approx(m_ref - m_new);
            m_ref = m_new;
            const float neg_m = -m_ref;
            float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < BN; ++c) {
                sc[c] = ex2_approx(fmaf(sc[c], p.scale_log2, neg_m));
                l4[c & 3] += sc[c];
            }
            l = l * alpha + ((l4[0] + l4[1]) + (l4[2] + l4[3]));
            // the previous P.V of this tile must be done: P is free and O is current
            if (j > 0) {
                ok = wait_or_abort(bar(Bars::o_done(g)), (j - 1) & 1, abort, p.err);
                if (!ok) break;
                tc_fence_after_sync();
                if (__any_sync(kFull, alpha != 1.f)) {
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t ov[32];
                        tmem_ld32(lane_base + Cfg::kOCol + cc * 32, ov);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                        tmem_st32(lane_base + Cfg::kOCol + cc * 32, ov);
                    }
                    tmem_st_wait();
                }
            }
            // row r of P_hi and P_lo: 8 chunks of 8 keys, 128-byte swizzle
#pragma unroll
            for (int c16 = 0; c16 < BN / 8; ++c16) {
                uint32_t h[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    split_bf16x2(sc[c16 * 8 + 2 * e], sc[c16 * 8 + 2 * e + 1], h[e], lo[e]);
                const uint32_t off = r * 128 + ((c16 ^ (r & 7)) << 4);
                *reinterpret_cast<uint4 *>(pbuf + off) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4 *>(pbuf + Cfg::kPBytes + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Bars::p_full(g)));
        }
        if (ok) ok = wait_or_abort(bar(Bars::o_done(g)), (nk - 1) & 1, abort, p.err);
        if (ok) {
            tc_fence_after_sync();
            const float inv_l = 1.f / l;
            const bool row_ok = qpos < len;
            float *dst = p.out + (static_cast<size_t>(start + qpos) * p.Hq + i) * D;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t ov[32];
                tmem_ld32(lane_base + Cfg::kOCol + cc * 32, ov);
                tmem_ld_wait();
                if (row_ok) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(dst + cc * 32 + e) =
                            make_float4(__uint_as_float(ov[e]) * inv_l, __uint_as_float(ov[e + 1]) * inv_l,
                                        __uint_as_float(ov[e + 2]) * inv_l, __uint_as_float(ov[e + 3]) * inv_l);
                }
            }
            if (row_ok && p.lse != nullptr)
                p.lse[static_cast<size_t>(start + qpos) * p.Hq + i] = (m_ref + log2f(l)) * kLn2;
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, Cfg::kTmemCols);
}

// ============================================================== CUDA-core path

template <typename T>
__device__ __forceinline__ float ld(const T *p);
template <>
__device__ __forceinline__ float ld<float>(const float *p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}

// One warp per (query row t, head i, sequence b); lanes own elements lane + 32*j.
template <typename T, int J>
__global__ void __launch_bounds__(32)
    prefill_simt_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                        const PrefillKParams p, int d) {
    const int lane = threadIdx.x;
    const int t = blockIdx.x, i = blockIdx.y, b = blockIdx.z;
    int start = 0, len = 0;
    if (!seq_range(p, b, start, len, lane == 0 && t == 0 && i == 0)) return;
    if (t >= len) return;
    const int kvh = i / p.m;
    const size_t qrow = (static_cast<size_t>(start + t) * p.Hq + i) * d;
    float qv[J], acc[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        qv[j] = e < d ? ld(q + qrow + e) : 0.f;
        acc[j] = 0.f;
    }
    float m_run = -INFINITY, l_run = 0.f;
    for (int u = 0; u <= t; ++u) {
        const size_t krow = (static_cast<size_t>(start + u) * p.Hkv + kvh) * d;
        float dot = 0.f;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int e = lane + 32 * j;
            if (e < d) dot += qv[j] * ld(k + krow + e);
        }
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) dot += __shfl_xor_sync(kFull, dot, sh);
        const float s = dot * p.scale_log2;
        const float m_new = fmaxf(m_run, s);
        const float alpha = exp2f(m_run - m_new);
        const float w = exp2f(s - m_new);
        l_run = l_run * alpha + w;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int e = lane + 32 * j;
            acc[j] = acc[j] * alpha + (e < d ? w * ld(v + krow + e) : 0.f);
        }
        m_run = m_new;
    }
    const size_t orow = (static_cast<size_t>(start + t) * p.Hq + i) * d;
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        if (e < d) p.out[orow + e] = acc[j] / l_run;
    }
    if (lane == 0 && p.lse != nullptr)
        p.lse[static_cast<size_t>(start + t) * p.Hq + i] = (m_run + log2f(l_run)) * kLn2;
}

template <int D>
cudaError_t launch_prefill_tc(const PrefillArgs &a, const PrefillKParams &kp, cudaStream_t stream) {
    using Cfg = TcPrefillCfg<D>;
    CUtensorMap tq, tk, tv;
    const uint64_t dq[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.Hq),
                            static_cast<uint64_t>(a.T)};
    const uint64_t sq[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(a.Hq) * D * 2};
    const uint64_t dk[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.Hkv),
                            static_cast<uint64_t>(a.T)};
    const uint64_t sk[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(a.Hkv) * D * 2};
    const uint32_t qbox[3] = {64, 1, static_cast<uint32_t>(Cfg::kBM)};
    const uint32_t kvbox[3] = {64, 1, static_cast<uint32_t>(Cfg::kBN)};
    if (!encode_map_bf16(&tq, a.q, 3, dq, sq, qbox) || !encode_map_bf16(&tk, a.k, 3, dk, sk, kvbox) ||
        !encode_map_bf16(&tv, a.v, 3, dk, sk, kvbox))
        return cudaErrorInvalidValue;
    auto kernel = prefill_tc_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int pair = Cfg::kGroups * Cfg::kBM;
    const dim3 grid(a.Hq, (a.max_seqlen + pair - 1) / pair, a.B);
    kernel<<<grid, 320, Cfg::kSmemBytes, stream>>>(tq, tk, tv, kp);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_prefill_simt(const PrefillArgs &a, const PrefillKParams &kp,
                                cudaStream_t stream) {
    const T *q = static_cast<const T *>(a.q);
    const T *k = static_cast<const T *>(a.k);
    const T *v = static_cast<const T *>(a.v);
    const dim3 grid(a.max_seqlen, a.Hq, a.B);
    switch ((a.d + 31) / 32) {
#define PKV_CASE(n)                                                               \
    case n:                                                                       \
        prefill_simt_kernel<T, n><<<grid, 32, 0, stream>>>(q, k, v, kp, a.d);     \
        break;
        PKV_CASE(1)
        PKV_CASE(2)
        PKV_CASE(3)
        PKV_CASE(4)
        PKV_CASE(5)
        PKV_CASE(6)
        PKV_CASE(7)
        PKV_CASE(8)
#undef PKV_CASE
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

bool prefill_tensor_core_ok(pkv_dtype dt, int d, const void *q, const void *k, const void *v,
                            int T, int Hq, int Hkv) {
    auto a16 = [](const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
    return dt == PKV_BF16 && (d == 64 || d == 128) && a16(q) && a16(k) && a16(v) && T > 0 &&
           static_cast<long long>(T) < (1ll << 31) && Hq > 0 && Hkv > 0;
}

cudaError_t launch_prefill(const PrefillArgs &a, pkv_dtype dt, cudaStream_t stream) {
    if (a.B == 0 || a.T == 0 || a.max_seqlen == 0) return cudaSuccess;
    PrefillKParams kp{};
    kp.out = a.out;
    kp.lse = a.lse;
    kp.cu = a.cu_seqlens;
    kp.err = a.err;
    kp.B = a.B;
    kp.T = a.T;
    kp.max_seqlen = a.max_seqlen;
    kp.Hq = a.Hq;
    kp.Hkv = a.Hkv;
    kp.m = a.Hq / a.Hkv;
    kp.scale_log2 = a.scale * kLog2e;
    if (prefill_tensor_core_ok(dt, a.d, a.q, a.k, a.v, a.T, a.Hq, a.Hkv))
        return a.d == 64 ? launch_prefill_tc<64>(a, kp, stream) : launch_prefill_tc<128>(a, kp, stream);
    return dt == PKV_F32 ? launch_prefill_simt<float>(a, kp, stream)
                         : launch_prefill_simt<__nv_bfloat16>(a, kp, stream);
}

}  // namespace pkv
