// prefill.cu -- varlen causal attention over packed prompts (cu_seqlens).
//
// Sequence b owns tokens [cu_seqlens[b], cu_seqlens[b+1]) of q/k/v (0539edu.com
// "从KV cache共享到批量调度…" §3.3).  Token t of a sequence attends to tokens 0..t of
// the same sequence (causal prefill, zwjcode.cn "KV Cache 的增量解码" §05; the mask is
// aligned so that a query at position t sees keys 0..t, §13), with query head i reading
// KV head floor(i/m) (limoncc.com "大语言模型研究15——注意力机制优化之KV缓存" §3.3).
//
// Tensor-core path (bf16, d in {64, 128}): 5th-generation tensor cores (tcgen05), one
// persistent CTA per SM walking the 128-query tiles of the launch, longest first.  TMA
// brings each Q tile and 128-key K/V tiles through two rings (128-byte swizzle, mbarrier
// completion with bounded waits); one thread issues S = Q K^T into one of three
// tensor-memory buffers, another O += P V into a tensor-memory accumulator with P read
// from the same buffer; eight warps, four threads per query row of one warp, run the online
// softmax (running max and sum, plumephp.com "KV Cache 优化与注意力机制加速" §2.2-§2.3) and
// write P over the scores as bf16 hi + lo parts, so the weights keep ~16 bits; four warps
// write the output while the softmax goes on with the next tile (details at
// prefill_tc_kernel).
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

// Tiles of the tcgen05 prefill: 128-row query tiles of one head, 128-key K/V tiles.  One
// CTA per SM works through the query tiles of the launch.
template <int D>
struct TcPrefillCfg {
    static constexpr int kBM = 128, kTK = 128;
    static constexpr int PANELS = D / 64;
    static constexpr int NK = D == 64 ? 6 : 3, NV = D == 64 ? 5 : 2;   // K and V ring slots
    static constexpr int NSP = 3;                      // S / P buffers in tensor memory
    static constexpr int kQBytes = kBM * D * 2;        // the Q tile: D/64 panels of [128][128 B]
    static constexpr int kSlotBytes = kTK * D * 2;     // one K or V tile: D/64 panels of [128][128 B]
    static constexpr int kOffK = kQBytes;
    static constexpr int kOffV = kOffK + NK * kSlotBytes;
    // output staging of the epilogue warps: [warp][32 rows][32 columns + 4] floats
    static constexpr int kPitch = 36;
    static constexpr int kOffStage = kOffV + NV * kSlotBytes;
    // row statistics handed to the epilogue warps, double-buffered by query tile:
    // [buffer][m, l][128 rows] floats
    static constexpr int kOffStats = kOffStage + 4 * 32 * kPitch * 4;
    static constexpr int kOffBar = kOffStats + 2 * 2 * kBM * 4;
    // barriers: Q loaded, Q free (a query tile's scores all computed); K full / free per
    // slot; V full / free per slot; per S/P buffer: S full, P full, P consumed (its P.V
    // done); O done (a query tile's last P.V), O free (read by the epilogue warps); per
    // statistics buffer: full, free; drain x2 (one per MMA-issuing thread)
    static constexpr int kQ = 0, kQFree = 1, kKFull = 2, kKFree = 2 + NK, kVFull = 2 + 2 * NK,
                         kVFree = 2 + 2 * NK + NV, kSFull = 2 + 2 * NK + 2 * NV, kPFull = kSFull + NSP,
                         kPFree = kPFull + NSP, kODone = kPFree + NSP, kOFree = kODone + 1,
                         kStFull = kOFree + 1, kStFree = kStFull + 2, kDrain = kStFree + 2,
                         kNumBars = kDrain + 2;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;   // TMEM slot, abort flag
    static constexpr int kSmemBytes = 1024 + kOffMisc + 16;
    // tensor memory: NSP S buffers of 128 columns, then O.  The weights of a key tile
    // overwrite its scores: P_hi of keys 2e, 2e + 1 (one bf16 pair) in column e of the
    // buffer, P_lo in column 64 + e.
    static constexpr int kTmemCols = 512;
    static constexpr int kSCol = 0, kOCol = NSP * kTK;
    static constexpr int kThreads = 512;
    static_assert(kOCol + D <= kTmemCols, "tensor memory budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// A query tile: 128 query rows of one head of one sequence.
struct PrefillItem {
    int b, head, q0, start, len, ntiles;
};

// The query tiles of the launch, in the order largest start first, then sequence, then
// head (tiles past a sequence's end, and sequences with inconsistent offsets, are not in
// it).  CTA c of G takes tile k = r G + c of round r when r is even and k = r G + G - 1 - c
// when r is odd ("snake" order), so that every CTA gets a similar share of long and short
// tiles.  Each role of a CTA walks the same tiles with its own walker; the walk only moves
// forward, so finding a tile's band (its start) is amortised over the walk.
struct PrefillWalk {
    const PrefillKParams *p;
    int nqt, total;        // 128-row bands of starts; query tiles of the launch
    int r = 0;             // next round
    int z = 0, base = 0;   // band z (start (nqt - 1 - z) 128) holds tiles base .. base + band - 1
    int band = 0;

    __device__ __forceinline__ int len_of(int b) const {
        int s0, l0;
        return seq_range(*p, b, s0, l0, false) ? l0 : 0;
    }
    __device__ __forceinline__ int band_size(int zz) const {
        const int q0 = (nqt - 1 - zz) * 128;
        int n = 0;
        for (int b = 0; b < p->B; ++b) n += len_of(b) > q0 ? 1 : 0;
        return n * p->Hq;
    }
    __device__ __forceinline__ void init(const PrefillKParams &pp) {
        p = &pp;
        nqt = (pp.max_seqlen + 127) / 128;
        total = 0;   // a sequence longer than max_seqlen (flagged) has only nqt tiles
        for (int b = 0; b < pp.B; ++b) total += min((len_of(b) + 127) / 128, nqt) * pp.Hq;
        band = band_size(0);
    }
    // the CTA's next query tile; false when it has none left
    __device__ __forceinline__ bool next(PrefillItem &w) {
        const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
        const int k = r * G + ((r & 1) ? G - 1 - c : c);
        ++r;
        if (k >= total) return false;
        while (k >= base + band) {
            base += band;
            ++z;
            band = band_size(z);
        }
        const int idx = k - base, rank = idx / p->Hq;
        w.b = 0;
        w.start = 0;
        w.len = 0;
        w.head = idx % p->Hq;
        w.q0 = (nqt - 1 - z) * 128;
        int seen = 0;
        for (int b = 0; b < p->B; ++b) {
            int s0, l0;
            if (!seq_range(*p, b, s0, l0, false) || l0 <= w.q0) continue;
            if (seen++ == rank) {
                w.b = b;
                w.start = s0;
                w.len = l0;
                break;
            }
        }
        w.ntiles = w.len > w.q0 ? (min(w.q0 + 128, w.len) - 1) / 128 + 1 : 0;   // key tiles up to the diagonal
        return true;
    }
};

// One CTA per SM, taking the query tiles of the launch in snake order (PrefillWalk), the
// longest first.  Sixteen warps, each role walking the same tiles:
//   warps 9 and 10 (TMA): the K and the V tiles into two rings of tile slots, one
//     {64, 1, 16} box (16 rows of one 64-column panel) per lane, so that sixteen threads
//     issue copies at once; a K slot is free once its scores are computed, a V slot once its
//     P.V is.  The rings run on across query tiles, so the next tile's copies start while
//     the current one is being finished.
//   warps 11 and 8 (one lane each issues tcgen05.mma): S = Q K_j^T (N = 128 keys) into
//     tensor-memory buffer g % 3 (g counts key tiles over all query tiles), once K_j has
//     landed and the P.V three key tiles back (which read that buffer) is done; and
//     O += P_hi V_j + P_lo V_j (N = d) with P_hi and P_lo read from the same buffer, the
//     first product of a query tile once the epilogue warps have read the previous O.
//     The score issuer also brings each Q tile, once the previous query tile's scores
//     have all been computed (it has nothing else to issue until then).
//   warps 0-7 (softmax): row r of the query tile is tensor-memory lane r; warp w reads
//     lanes 32 (w % 4) + 16 (w / 4) .. + 15 with the 16-lane shapes, thread t taking rows
//     t / 4 and t / 4 + 8 of them and, of each key tile, the key pairs 4k + t % 4 (keys
//     8k + 2 (t % 4), + 1; k = 0 .. 15): the four threads of a row are lanes of one warp and
//     share its maximum and sum by shuffles, and the eight warps run independently.  Per
//     key tile: read the rows of S, apply the causal mask (key <= query) on the diagonal
//     tile, update the running maximum and sum (online softmax), rescale the O rows in
//     tensor memory when the reference maximum grew by more than 2^8 (exponentials stay
//     <= 256 otherwise, and O and l share the reference), and write P as bf16 hi and lo
//     parts (P = P_hi + P_lo to about 2^-16 relative) over the scores.  At the end of a
//     query tile the rows' maxima and sums go to the epilogue warps, and the softmax warps
//     go on with the next query tile.
//   warps 12-15 (epilogue): once a query tile's last P.V is done, thread (w, lane) reads O
//     row 32 (w % 4) + lane 32 columns at a time, frees O for the next query tile, and
//     writes O / l (staged in shared memory, so that each store writes whole 128-byte row
//     segments) and the log-sum-exp.
// Every wait is bounded and shares an abort flag: on a timeout the block drains its copies
// and MMAs, frees tensor memory and returns with PKV_DEVERR_TIMEOUT.
template <int D>
__global__ void __launch_bounds__(512, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const PrefillKParams p) {
    using Cfg = TcPrefillCfg<D>;
    constexpr int BM = Cfg::kBM, TK = Cfg::kTK, PANELS = Cfg::PANELS, NK = Cfg::NK, NV = Cfg::NV,
                  NSP = Cfg::NSP;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 4);
    float *stats = reinterpret_cast<float *>(smem + Cfg::kOffStats);
    auto bar = [&](int k) { return smem_addr(&bars[k]); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    PrefillWalk walk;
    walk.init(p);

    if (threadIdx.x == 0) {
        if (blockIdx.x == 0)   // inconsistent offsets are reported once; their tiles are skipped
            for (int b = 0; b < p.B; ++b) {
                int s0, l0;
                seq_range(p, b, s0, l0, true);
            }
        mbar_init(bar(Cfg::kQ), 1);
        mbar_init(bar(Cfg::kQFree), 1);
        for (int s = 0; s < NK; ++s) {
            mbar_init(bar(Cfg::kKFull + s), 1);
            mbar_init(bar(Cfg::kKFree + s), 1);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(bar(Cfg::kVFull + s), 1);
            mbar_init(bar(Cfg::kVFree + s), 1);
        }
        for (int u = 0; u < NSP; ++u) {
            mbar_init(bar(Cfg::kSFull + u), 1);
            mbar_init(bar(Cfg::kPFull + u), 8);
            mbar_init(bar(Cfg::kPFree + u), 1);
        }
        mbar_init(bar(Cfg::kODone), 1);
        mbar_init(bar(Cfg::kOFree), 4);
        for (int u = 0; u < 2; ++u) {
            mbar_init(bar(Cfg::kStFull + u), 8);
            mbar_init(bar(Cfg::kStFree + u), 4);
        }
        mbar_init(bar(Cfg::kDrain), 1);
        mbar_init(bar(Cfg::kDrain + 1), 1);
        *abort = 0;
        fence_barrier_init();
        tma_prefetch_map(&tm_q);
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_v);
    }
    if (warp == 0) tmem_alloc(smem_addr(tslot), Cfg::kTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t sQ = smem_addr(smem);
    auto sK = [&](int s) { return smem_addr(smem + Cfg::kOffK + s * Cfg::kSlotBytes); };
    auto sV = [&](int s) { return smem_addr(smem + Cfg::kOffV + s * Cfg::kSlotBytes); };

    if (warp == 9 || warp == 10) {
        // ---- TMA loaders: warp 9 the K tiles, warp 10 the V tiles.  Key tile g (counted over
        // all query tiles) goes to slot g % N once the slot's previous tile is consumed.  Lane
        // l < 8 * PANELS copies rows 16 (l / PANELS) .. + 15 of panel l % PANELS.
        const bool is_k = warp == 9;
        const int N = is_k ? NK : NV;
        const int full0 = is_k ? Cfg::kKFull : Cfg::kVFull, free0 = is_k ? Cfg::kKFree : Cfg::kVFree;
        const CUtensorMap *map = is_k ? &tm_k : &tm_v;
        const int chunk = lane / PANELS, pn = lane % PANELS;
        int t = 0;   // key tiles copied
        bool alive = true;
        PrefillItem w;
        while (alive && walk.next(w)) {
            const int kvh = w.head / p.m;
            for (int j = 0; j < w.ntiles; ++j) {
                bool fr = true;
                if (lane == 0 && t >= N) fr = wait_or_abort(bar(free0 + t % N), ((t - N) / N) & 1, abort, p.err);
                if (!__shfl_sync(kFull, fr ? 1 : 0, 0)) {
                    alive = false;
                    break;
                }
                const int s = t % N;
                if (lane == 0) mbar_arrive_expect_tx(bar(full0 + s), Cfg::kSlotBytes);
                __syncwarp();
                if (lane < 8 * PANELS) {
                    const uint32_t dst = (is_k ? sK(s) : sV(s)) + pn * TK * 128 + chunk * 16 * 128;
                    tma_load_3d(dst, map, pn * 64, kvh, w.start + j * TK + chunk * 16, bar(full0 + s));
                }
                ++t;
            }
        }
        // before teardown every copy issued must have landed (bounded)
        if (lane == 0) {
            for (int u = max(0, t - N); u < t; ++u)
                if (!mbar_wait_bounded(bar(full0 + u % N), (u / N) & 1)) raise_error(p.err, PKV_DEVERR_TIMEOUT);
        }
    } else if (warp == 8 || warp == 11) {
        // ---- MMA issue, one lane each: warp 11 the scores, warp 8 the products with V.
        // tcgen05.commit covers the committing thread's MMAs: warp 11 signals S full, K free
        // and, after a query tile's last scores, Q free (waited by itself before it copies the
        // next Q tile); warp 8 P consumed, V free and, after a query tile's last P.V, O done.
        // Buffer g % 3's barriers complete once per use, no use starts before the previous
        // one is consumed, and a query tile's barriers complete once per query tile with the
        // next one waiting for this one's consumer, so each wait's phase is unambiguous.
        if (lane == 0) {
            const bool is_s = warp == 11;
            bool issued = false, alive = true;
            int g = 0, cnt = 0;   // key tiles and query tiles done
            if (is_s) {
                const uint32_t idesc_s = umma_idesc_bf16(BM, TK, 0);
                bool q_in_flight = false;
                PrefillItem w;
                while (alive && walk.next(w)) {
                    // the Q tile, over the previous one once its scores have all been computed
                    if (cnt > 0) alive = wait_or_abort(bar(Cfg::kQFree), (cnt - 1) & 1, abort, p.err);
                    if (!alive) break;
                    mbar_arrive_expect_tx(bar(Cfg::kQ), Cfg::kQBytes);
#pragma unroll
                    for (int k = 0; k < PANELS; ++k)
                        tma_load_3d(sQ + k * BM * 128, &tm_q, k * 64, w.head, w.start + w.q0, bar(Cfg::kQ));
                    q_in_flight = true;
                    alive = wait_or_abort(bar(Cfg::kQ), cnt & 1, abort, p.err);
                    if (!alive) break;
                    q_in_flight = false;
                    for (int j = 0; j < w.ntiles && alive; ++j) {
                        const int sb = g % NSP;
                        if (g >= NSP) alive = wait_or_abort(bar(Cfg::kPFree + sb), ((g - NSP) / NSP) & 1, abort, p.err);
                        alive = alive && wait_or_abort(bar(Cfg::kKFull + g % NK), (g / NK) & 1, abort, p.err);
                        if (!alive) break;
                        tc_fence_after_sync();
                        const int s = g % NK;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint64_t ad = umma_desc_sw128(sQ + (kk / 4) * BM * 128 + (kk % 4) * 32, 16, 1024);
                            const uint64_t bd = umma_desc_sw128(sK(s) + (kk / 4) * TK * 128 + (kk % 4) * 32, 16, 1024);
                            umma_bf16(tmem + Cfg::kSCol + sb * TK, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
                        }
                        umma_commit(bar(Cfg::kSFull + sb));
                        umma_commit(bar(Cfg::kKFree + s));
                        issued = true;
                        ++g;
                    }
                    if (!alive) break;
                    umma_commit(bar(Cfg::kQFree));
                    ++cnt;
                }
                // a Q copy whose wait gave up must still land before teardown (bounded)
                if (q_in_flight && !mbar_wait_bounded(bar(Cfg::kQ), cnt & 1)) raise_error(p.err, PKV_DEVERR_TIMEOUT);
            } else {
                const uint32_t idesc_o = umma_idesc_bf16(BM, D, 1);
                PrefillItem w;
                while (alive && walk.next(w)) {
                    for (int j = 0; j < w.ntiles && alive; ++j) {
                        const int sb = g % NSP;
                        alive = wait_or_abort(bar(Cfg::kPFull + sb), (g / NSP) & 1, abort, p.err) &&
                                wait_or_abort(bar(Cfg::kVFull + g % NV), (g / NV) & 1, abort, p.err);
                        // the first product of a query tile overwrites O: the previous one read
                        if (alive && j == 0 && cnt > 0)
                            alive = wait_or_abort(bar(Cfg::kOFree), (cnt - 1) & 1, abort, p.err);
                        if (!alive) break;
                        tc_fence_after_sync();
                        const int s = g % NV;
#pragma unroll
                        for (int half = 0; half < 2; ++half)
#pragma unroll
                            for (int kk = 0; kk < TK / 16; ++kk) {
                                // keys 16 kk .. 16 kk + 15: the pairs 8 kk .. 8 kk + 7 of P_hi (half 0) or P_lo
                                const uint32_t pcol = Cfg::kSCol + sb * TK + half * 64 + kk * 8;
                                const uint64_t bd = umma_desc_sw128(sV(s) + kk * 16 * 128, TK * 128, 1024);
                                umma_bf16_ts(tmem + Cfg::kOCol, tmem + pcol, bd, idesc_o,
                                             (j > 0 || half > 0 || kk > 0) ? 1u : 0u);
                            }
                        umma_commit(bar(Cfg::kPFree + sb));
                        umma_commit(bar(Cfg::kVFree + s));
                        issued = true;
                        ++g;
                    }
                    if (!alive) break;
                    umma_commit(bar(Cfg::kODone));
                    ++cnt;
                }
            }
            if (*abort && issued) {
                // let this thread's MMAs finish (bounded) before teardown
                const int drain = is_s ? Cfg::kDrain + 1 : Cfg::kDrain;
                umma_commit(bar(drain));
                if (!mbar_wait_bounded(bar(drain), 0)) raise_error(p.err, PKV_DEVERR_TIMEOUT);
            }
        }
    } else if (warp < 8) {
        // ---- softmax: thread (w, t) owns rows ra = 32 (w % 4) + 16 (w / 4) + t / 4 and rb =
        // ra + 8 of the query tile, and of each key tile the key pairs 4k + c4 (c4 = t % 4)
        const int c4 = lane & 3;
        const int ra = 32 * (warp & 3) + 16 * (warp >> 2) + (lane >> 2), rb = ra + 8;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * (warp & 3) + 16 * (warp >> 2)) << 16);
        const uint32_t ocol = lane_base + Cfg::kOCol;
        // ok is warp-uniform; a failed wait skips the remaining work of this warp
        bool ok = true;
        int g = 0, cnt = 0;
        PrefillItem w;
        while (walk.next(w)) {
            const int qa = w.q0 + ra, qb = w.q0 + rb;   // the rows' positions
            float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
            for (int j = 0; j < w.ntiles; ++j, ++g) {
                const int pb = g % NSP;            // S / P buffer
                const uint32_t scol = lane_base + Cfg::kSCol + pb * TK;
                if (ok) ok = __all_sync(kFull, wait_or_abort(bar(Cfg::kSFull + pb), (g / NSP) & 1, abort, p.err));
                if (!ok) continue;
                tc_fence_after_sync();
                // sc[4k + e]: row a, key 8k + 2 c4 + e; sc[4k + 2 + e]: row b, the same key
                float sc[64];
                {
                    uint32_t s0[32], s1[32];
                    tmem_ld_16x256b_x8(scol, s0);
                    tmem_ld_16x256b_x8(scol + 64, s1);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        sc[c] = __uint_as_float(s0[c]);
                        sc[32 + c] = __uint_as_float(s1[c]);
                    }
                }
                // causal mask on the diagonal tile: key <= query
                const int key0 = j * TK + 2 * c4;
                if (j * TK + TK - 1 > w.q0) {
#pragma unroll
                    for (int k = 0; k < 16; ++k)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            if (key0 + 8 * k + e > qa) sc[4 * k + e] = -INFINITY;
                            if (key0 + 8 * k + e > qb) sc[4 * k + 2 + e] = -INFINITY;
                        }
                }
                // the rows' maxima over the four threads of each row
                float xa0 = -INFINITY, xa1 = -INFINITY, xb0 = -INFINITY, xb1 = -INFINITY;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    xa0 = fmaxf(xa0, sc[4 * k]);
                    xa1 = fmaxf(xa1, sc[4 * k + 1]);
                    xb0 = fmaxf(xb0, sc[4 * k + 2]);
                    xb1 = fmaxf(xb1, sc[4 * k + 3]);
                }
                float mxa = fmaxf(xa0, xa1), mxb = fmaxf(xb0, xb1);
                mxa = fmaxf(mxa, __shfl_xor_sync(kFull, mxa, 1));
                mxb = fmaxf(mxb, __shfl_xor_sync(kFull, mxb, 1));
                mxa = fmaxf(mxa, __shfl_xor_sync(kFull, mxa, 2)) * p.scale_log2;
                mxb = fmaxf(mxb, __shfl_xor_sync(kFull, mxb, 2)) * p.scale_log2;
                // key 0 is always visible, so the row maxima are finite from the first tile on
                const float mna = mxa > m_a + 8.f ? mxa : m_a, mnb = mxb > m_b + 8.f ? mxb : m_b;
                const float alpha_a = ex2_approx(m_a - mna), alpha_b = ex2_approx(m_b - mnb);
                m_a = mna;
                m_b = mnb;
                // the key pairs of a row as packed fp32 pairs: one FMA and one add a pair
                const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
                const float2 nma = make_float2(-m_a, -m_a), nmb = make_float2(-m_b, -m_b);
                float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    float2 xa = fma2(make_float2(sc[4 * k], sc[4 * k + 1]), sl2, nma);
                    float2 xb = fma2(make_float2(sc[4 * k + 2], sc[4 * k + 3]), sl2, nmb);
                    xa.x = ex2_approx(xa.x);
                    xa.y = ex2_approx(xa.y);
                    xb.x = ex2_approx(xb.x);
                    xb.y = ex2_approx(xb.y);
                    la = add2(la, xa);
                    lb = add2(lb, xb);
                    sc[4 * k] = xa.x;
                    sc[4 * k + 1] = xa.y;
                    sc[4 * k + 2] = xb.x;
                    sc[4 * k + 3] = xb.y;
                }
                l_a = l_a * alpha_a + (la.x + la.y);
                l_b = l_b * alpha_b + (lb.x + lb.y);
                // the weights over the scores (all of them in registers by now): pair 4k + c4
                // of P_hi in column 4k + c4, of P_lo in column 64 + 4k + c4, 64 keys at a time
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t ph[16], pl[16];
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const int k = 8 * q + kk;
                        split_bf16x2_p(sc[4 * k], sc[4 * k + 1], ph[2 * kk], pl[2 * kk]);
                        split_bf16x2_p(sc[4 * k + 2], sc[4 * k + 3], ph[2 * kk + 1], pl[2 * kk + 1]);
                    }
                    tmem_st_16x128b_x8(scol + 32 * q, ph);
                    tmem_st_16x128b_x8(scol + 64 + 32 * q, pl);
                }
                // a rescale of O waits for the previous P.V of this query tile (and so every
                // earlier one): O is then current, and this tile's P.V waits for its P
                if (j > 0 && __any_sync(kFull, alpha_a != 1.f || alpha_b != 1.f)) {
                    const int qb2 = (g - 1) % NSP;
                    ok = __all_sync(kFull, wait_or_abort(bar(Cfg::kPFree + qb2), ((g - 1) / NSP) & 1, abort, p.err));
                    if (!ok) continue;
                    tc_fence_after_sync();
#pragma unroll
                    for (int cc = 0; cc < D / 64; ++cc) {
                        uint32_t ov[32];
                        tmem_ld_16x256b_x8(ocol + cc * 64, ov);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            ov[4 * k] = __float_as_uint(__uint_as_float(ov[4 * k]) * alpha_a);
                            ov[4 * k + 1] = __float_as_uint(__uint_as_float(ov[4 * k + 1]) * alpha_a);
                            ov[4 * k + 2] = __float_as_uint(__uint_as_float(ov[4 * k + 2]) * alpha_b);
                            ov[4 * k + 3] = __float_as_uint(__uint_as_float(ov[4 * k + 3]) * alpha_b);
                        }
                        tmem_st_16x256b_x8(ocol + cc * 64, ov);
                    }
                }
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(Cfg::kPFull + pb));
            }
            // the rows' sums over their four threads, and the maxima, for the epilogue warps
            // (the buffer was read by them two query tiles ago)
            l_a += __shfl_xor_sync(kFull, l_a, 1);
            l_b += __shfl_xor_sync(kFull, l_b, 1);
            l_a += __shfl_xor_sync(kFull, l_a, 2);
            l_b += __shfl_xor_sync(kFull, l_b, 2);
            const int sbuf = cnt & 1;
            if (ok && cnt >= 2)
                ok = __all_sync(kFull, wait_or_abort(bar(Cfg::kStFree + sbuf), ((cnt - 2) >> 1) & 1, abort, p.err));
            if (ok) {
                if (c4 == 0) {
                    stats[(sbuf * 2) * BM + ra] = m_a;
                    stats[(sbuf * 2 + 1) * BM + ra] = l_a;
                    stats[(sbuf * 2) * BM + rb] = m_b;
                    stats[(sbuf * 2 + 1) * BM + rb] = l_b;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(Cfg::kStFull + sbuf));
            }
            ++cnt;
        }
    } else {
        // ---- epilogue: thread (w, lane) writes query row r = 32 (w % 4) + lane
        const int r = ((warp & 3) << 5) | lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        float *stage = reinterpret_cast<float *>(smem + Cfg::kOffStage) + (warp & 3) * 32 * Cfg::kPitch;
        bool ok = true;
        int cnt = 0;
        PrefillItem w;
        while (ok && walk.next(w)) {
            const int sbuf = cnt & 1;
            ok = __all_sync(kFull, wait_or_abort(bar(Cfg::kStFull + sbuf), (cnt >> 1) & 1, abort, p.err)) &&
                 __all_sync(kFull, wait_or_abort(bar(Cfg::kODone), cnt & 1, abort, p.err));
            if (!ok) break;
            tc_fence_after_sync();
            const float m = stats[(sbuf * 2) * BM + r];
            const float lr = stats[(sbuf * 2 + 1) * BM + r];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Cfg::kStFree + sbuf));
            const float inv_l = 1.f / lr;
            const int wrow0 = w.q0 + ((warp & 3) << 5);
            const int nrows = min(32, w.len - wrow0);   // rows of the warp inside the sequence
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t ov[32];
                tmem_ld32(lane_base + Cfg::kOCol + c * 32, ov);
                tmem_ld_wait();
                if (c == D / 32 - 1) {
                    // O has been read: the next query tile's first P.V may overwrite it
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(Cfg::kOFree));
                }
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4 *>(stage + lane * Cfg::kPitch + e) =
                        make_float4(__uint_as_float(ov[e]) * inv_l, __uint_as_float(ov[e + 1]) * inv_l,
                                    __uint_as_float(ov[e + 2]) * inv_l, __uint_as_float(ov[e + 3]) * inv_l);
                __syncwarp();
                // four rows a store: lane l writes columns 4 (l % 8) .. + 3 of row 4 i + l / 8
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int rr = 4 * i + (lane >> 3);
                    if (rr < nrows)
                        *reinterpret_cast<float4 *>(p.out + (static_cast<size_t>(w.start + wrow0 + rr) * p.Hq + w.head) * D +
                                                    c * 32 + (lane & 7) * 4) =
                            *reinterpret_cast<const float4 *>(stage + rr * Cfg::kPitch + (lane & 7) * 4);
                }
                __syncwarp();
            }
            if (w.q0 + r < w.len && p.lse != nullptr)
                p.lse[static_cast<size_t>(w.start + w.q0 + r) * p.Hq + w.head] = (m + log2f(lr)) * kLn2;
            ++cnt;
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
    const uint32_t kvbox[3] = {64, 1, 16};   // 16 rows of one panel: one box per loader lane
    if (!encode_map_bf16(&tq, a.q, 3, dq, sq, qbox) || !encode_map_bf16(&tk, a.k, 3, dk, sk, kvbox) ||
        !encode_map_bf16(&tv, a.v, 3, dk, sk, kvbox))
        return cudaErrorInvalidValue;
    auto kernel = prefill_tc_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    // one CTA per SM (at most one per query tile)
    const long long n_items = static_cast<long long>((a.max_seqlen + Cfg::kBM - 1) / Cfg::kBM) * a.B * a.Hq;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(min(static_cast<long long>(sms), n_items));
    kernel<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(tq, tk, tv, kp);
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
    // the tcgen05 kernel numbers the query tiles of the launch with an int
    // the tcgen05 kernel writes out in 8-byte pieces
    if (prefill_tensor_core_ok(dt, a.d, a.q, a.k, a.v, a.T, a.Hq, a.Hkv) &&
        reinterpret_cast<uintptr_t>(a.out) % 8 == 0 &&
        static_cast<long long>((a.max_seqlen + 127) / 128) * a.B * a.Hq < (1ll << 31))
        return a.d == 64 ? launch_prefill_tc<64>(a, kp, stream) : launch_prefill_tc<128>(a, kp, stream);
    return dt == PKV_F32 ? launch_prefill_simt<float>(a, kp, stream)
                         : launch_prefill_simt<__nv_bfloat16>(a, kp, stream);
}

}  // namespace pkv
