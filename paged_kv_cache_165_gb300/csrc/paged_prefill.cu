// paged_prefill.cu -- chunked prefill over a paged cache: many new query rows of each
// sequence against everything the cache holds for it (a prefix-cache hit: only the new
// suffix is prefilled, limoncc.com "大语言模型研究15——注意力机制优化之KV缓存" §5).
//
// What is computed is pkv_paged_attention with query rows: the nq rows of sequence b are
// its last nq positions, P0 .. P0 + nq - 1 with P0 = L - nq (their K/V already appended),
// and row r sees the keys at positions 0 .. P0 + r of the sequence -- causal, aligned to
// the end of the cache (zwjcode.cn "KV Cache 的增量解码" §13) -- read through block_table[b]
// (plumephp.com "KV Cache 优化与注意力机制加速" §4.2-§4.3), with query head i reading KV
// head floor(i/m) (limoncc.com §3.3) and the online softmax of plumephp.com §2.2-§2.3.
//
// The design follows the prefill kernel's (prefill.cu): one CTA per SM walking the work
// tiles (128 query rows of one head of one sequence), 128-key tiles, sixteen warps.  What
// differs:
//   - the queries are fp32: the epilogue warps split each into bf16 hi + lo parts and store
//     them, 128-byte swizzled, as two shared-memory operand tiles; S = Q_hi K^T + Q_lo K^T
//     (two passes over the head dimension) carries q to about 2^-16 relative.
//   - K and V come from the paged cache: one {64, bs} TMA box per page and 64-column panel,
//     pages found through the block table, one box per loader lane.
//   - the causal mask is bottom-right: row r sees keys up to P0 + r, so only the last key
//     tiles of a row tile are masked; rows past nq see nothing and are not stored.
//   - the last page may end inside its block: its V rows past the end are zeroed in shared
//     memory before P.V (NaN or Inf in unwritten slots stay invisible).
// Every wait is bounded and shares an abort flag: on a timeout the block drains its copies
// and MMAs, frees tensor memory and returns with PKV_DEVERR_TIMEOUT.
#include <math.h>

#include "common.cuh"
#include "decode_kparams.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr unsigned kFull = 0xffffffffu;

template <int D, int BS>
struct PagedPrefillCfg {
    static constexpr int kBM = 128, kTK = 128, kPPT = kTK / BS;   // pages per key tile
    static constexpr int PANELS = D / 64;
    static constexpr int NK = D == 64 ? 5 : 2, NV = D == 64 ? 5 : 2;   // K and V ring slots
    static constexpr int NSP = 3;                      // S / P buffers in tensor memory
    static constexpr int kQBytes = kBM * D * 2;        // one Q part: D/64 panels of [128][128 B]
    static constexpr int kSlotBytes = kTK * D * 2;     // one K or V tile
    static constexpr int kOffQHi = 0, kOffQLo = kQBytes;
    static constexpr int kOffK = 2 * kQBytes;
    static constexpr int kOffV = kOffK + NK * kSlotBytes;
    // output staging of the epilogue warps: [warp][32 rows][32 columns + 4] floats
    static constexpr int kPitch = 36;
    static constexpr int kOffStage = kOffV + NV * kSlotBytes;
    // row statistics handed to the epilogue warps, double-buffered by work tile:
    // [buffer][m, l of half 0, l of half 1][128 rows] floats
    static constexpr int kOffStats = kOffStage + 4 * 32 * kPitch * 4;
    // row-maximum exchange of the two softmax warps of a row, double-buffered by key tile:
    // [buffer][value, ok][half][128 rows] floats
    static constexpr int kOffXch = kOffStats + 2 * 3 * kBM * 4;
    static constexpr int kOffBar = kOffXch + 2 * 2 * 2 * kBM * 4;
    // barriers: Q written, Q free (a work tile's scores all computed); K full / free per
    // slot; V full / free per slot; per S/P buffer: S full, P full, P consumed (its P.V
    // done); O done (a work tile's last P.V), O free (read by the epilogue warps); per
    // statistics buffer: full, free; drain x2 (one per MMA-issuing thread)
    static constexpr int kQ = 0, kQFree = 1, kKFull = 2, kKFree = 2 + NK, kVFull = 2 + 2 * NK,
                         kVFree = 2 + 2 * NK + NV, kSFull = 2 + 2 * NK + 2 * NV, kPFull = kSFull + NSP,
                         kPFree = kPFull + NSP, kODone = kPFree + NSP, kOFree = kODone + 1,
                         kStFull = kOFree + 1, kStFree = kStFull + 2, kDrain = kStFree + 2,
                         kNumBars = kDrain + 2;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;   // TMEM slot, abort flag
    static constexpr int kSmemBytes = 1024 + kOffMisc + 16;
    // tensor memory: NSP S buffers of 128 columns, then O.  The weights of a key tile
    // overwrite its scores: the thread that read S columns 64h .. 64h + 63 of a row writes
    // P_hi of those keys to columns 64h .. 64h + 31 of the buffer and P_lo to 64h + 32 ..
    // 64h + 63.
    static constexpr int kTmemCols = 512;
    static constexpr int kSCol = 0, kOCol = NSP * kTK;
    static constexpr int kThreads = 512;
    static_assert(D == 64 || D == 128, "head size");
    static_assert(BS == 16 || BS == 32, "block size");
    static_assert(kOCol + D <= kTmemCols, "tensor memory budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kPPT * PANELS <= 32 && 32 % kPPT == 0, "one box per loader lane; tiles within 32 pages");
};

// A work tile: 128 rows against key tiles kt0 .. kt0 + ntiles - 1.
//   chunked prefill (tile (qt, head, b) of the launch): rows r0 = 128 qt .. r0 + nrows - 1 of
//     sequence b's nq query rows, head `head`, row r at position P0 + r seeing keys 0 ..
//     P0 + r (pages from block_table[b]);
//   shared prefix (tile (ks, kvh, g rtiles + rt)): rows rho = 128 rt .. of group g's
//     (member, head) pairs, rho = mu m + hh for member mu and head kvh m + hh, all seeing the
//     group's prefix keys of split ks (pages from the first member's row).
// kind: kWork, or a tile with no attention to compute: kEmpty (a split with no prefix key:
// empty partials), kBadRows (inconsistent query rows: out = 0, lse = -inf), kNone.
enum { kWork = 0, kEmpty = 1, kBadRows = 2, kNone = 3 };
struct PPItem {
    int kind, b, head, kvh, c0, r0, nrows, nq, P0, key_end, npages, ntiles, kt0, gs, ks;
    const int32_t *tbl_row;
};

template <int BS, bool kShared>
__device__ __forceinline__ PPItem pp_item(const DecodeKParams &p, int it, int gx, int gy, bool report) {
    constexpr int BM = 128, TK = 128;
    PPItem w{};
    w.kind = kNone;
    const int x = it % gx, y = (it / gx) % gy, z = it / (gx * gy);
    if constexpr (kShared) {
        w.ks = x;
        w.kvh = y;
        const int g = z / p.prefix_rtiles, rt = z % p.prefix_rtiles;
        w.gs = __ldg(p.cu_q + g);
        const int nmem = __ldg(p.cu_q + g + 1) - w.gs;
        if (w.gs < 0 || nmem < 0 || w.gs + nmem > p.n_members ||
            static_cast<long long>(nmem) * p.m > static_cast<long long>(p.prefix_rtiles) * BM) {
            // offsets outside the member list, or a group larger than the declared maximum
            if (report) raise_error(p.err, PKV_DEVERR_PREFIX);
            return w;
        }
        w.r0 = rt * BM;
        w.nrows = min(BM, nmem * p.m - w.r0);
        if (w.nrows <= 0) return w;
        const int first = __ldg(p.group_seqs + w.gs);
        if (first < 0 || first >= p.B) {
            if (report) raise_error(p.err, PKV_DEVERR_PREFIX);
            return w;
        }
        int P = __ldg(p.kv_start + first);
        if (P < 0 || P % BS != 0 || P > p.MBS * BS) P = 0;   // flagged by the merge
        const int KT = (P + TK - 1) / TK;
        const int kps = (KT + p.prefix_splits - 1) / p.prefix_splits;
        w.kt0 = w.ks * kps;
        w.ntiles = min(KT, w.kt0 + kps) - w.kt0;
        w.key_end = P;
        w.npages = P / BS;
        w.tbl_row = p.block_table + static_cast<size_t>(first) * p.MBS;
        w.kind = w.ntiles > 0 ? kWork : kEmpty;
    } else {
        const int qt = x;
        w.head = y;
        w.b = z;
        const int L = checked_len(p, w.b, BS, report);
        w.c0 = __ldg(p.cu_q + w.b);
        w.nq = __ldg(p.cu_q + w.b + 1) - w.c0;
        w.r0 = qt * BM;                     // the tile's first query row
        if (w.nq < 0 || w.nq > L) {
            if (report) raise_error(p.err, PKV_DEVERR_CU_SEQLENS);
            if (w.r0 == 0) w.kind = kBadRows;
            return w;
        }
        if (w.r0 >= w.nq) return w;
        w.nrows = min(BM, w.nq - w.r0);     // rows of this tile
        w.P0 = L - w.nq + w.r0;             // position of the tile's first row
        w.key_end = w.P0 + w.nrows;         // one past the last key any row of the tile sees
        w.npages = (w.key_end + BS - 1) / BS;
        w.ntiles = (w.key_end + TK - 1) / TK;
        w.kvh = w.head / p.m;
        w.tbl_row = p.block_table + static_cast<size_t>(w.b) * p.MBS;
        w.kind = kWork;
    }
    return w;
}

// The (sequence, head) pair that row rr of work tile w is; shared prefix: member mu of the group.
template <bool kShared>
__device__ __forceinline__ void pp_row(const DecodeKParams &p, const PPItem &w, int rr, int &bq, int &hq,
                                       size_t &member) {
    if constexpr (kShared) {
        const int rho = w.r0 + rr;
        member = static_cast<size_t>(w.gs + rho / p.m);
        bq = __ldg(p.group_seqs + member);
        if (bq < 0 || bq >= p.B) bq = 0;   // flagged by the merge; never read out of range
        hq = w.kvh * p.m + rho % p.m;
    } else {
        member = 0;
        bq = w.c0 + w.r0 + rr;   // the query row
        hq = w.head;
    }
}

// One CTA per SM; CTA c takes work tiles c, c + G, c + 2G, .. of the launch (tile (x, y, z)
// of the grid the work is cut into is number x + gx (y + gy z)).  Sixteen warps, each role
// walking the same tiles:
//   warps 9 and 10 (TMA): the K and the V tiles into two rings, one {64, bs} box (one page,
//     one panel) per lane; a K slot is free once its scores are computed, a V slot once
//     its P.V is.  A page past the keys any row sees is placed outside the cache, where TMA
//     fills zeros.  The rings run on across work tiles.
//   warps 11 and 8 (one lane each issues): S = Q_hi K_j^T + Q_lo K_j^T (N = 128 keys) into
//     tensor-memory buffer g % 3 (g counts key tiles over all work tiles), once K_j has
//     landed and the P.V three key tiles back (which read that buffer) is done; O += P_hi
//     V_j + P_lo V_j (N = d), P read from the same buffer, the first product of a work tile
//     once the epilogue warps have read the previous O.
//   warps 0-7 (softmax): per key tile the online softmax for row r = 32 (w % 4) + lane over
//     keys 64h .. 64h + 63 of the tile (h = w / 4; the two warps of a row share its maximum
//     through shared memory), with the bottom-right causal mask; at the end of a work tile
//     the row's maximum and partial sums go to the epilogue warps, and the softmax warps go
//     on with the next tile.  (The prefill kernel's softmax on the 16-lane shapes measured
//     slower here: this kernel's two query passes keep the tensor pipe the busier unit.)
//   warps 12-15 (queries and epilogue): thread (w, lane) loads row r = 32 (w % 4) + lane of
//     the next work tile's fp32 queries once the current tile's scores have all been
//     computed, splits them into bf16 hi and lo parts and stores both as row r of the two
//     swizzled operand tiles (zeros for rows past the tile's rows); then, once the previous
//     tile's last P.V is done, it reads that tile's O row 32 columns at a time, frees O, and
//     writes O / l (staged in shared memory, four rows a vector store) and the log-sum-exp
//     (chunked prefill: the output rows; shared prefix: this split's normalised partials).
//     They also write the empty results of tiles with nothing to compute.
// Every wait is bounded and shares an abort flag: on a timeout the block drains its copies
// and MMAs, frees tensor memory and returns with PKV_DEVERR_TIMEOUT.
template <int D, int BS, bool kShared>
__global__ void __launch_bounds__(512, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const DecodeKParams p, int gx, int gy, int n_items) {
    using Cfg = PagedPrefillCfg<D, BS>;
    constexpr int BM = Cfg::kBM, TK = Cfg::kTK, PPT = Cfg::kPPT, PANELS = Cfg::PANELS, NK = Cfg::NK,
                  NV = Cfg::NV, NSP = Cfg::NSP;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 4);
    float *xch = reinterpret_cast<float *>(smem + Cfg::kOffXch);
    float *stats = reinterpret_cast<float *>(smem + Cfg::kOffStats);
    auto bar = [&](int k) { return smem_addr(&bars[k]); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        mbar_init(bar(Cfg::kQ), 4);
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
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_v);
    }
    if (warp == 0) tmem_alloc(smem_addr(tslot), Cfg::kTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t sQHi = smem_addr(smem + Cfg::kOffQHi), sQLo = smem_addr(smem + Cfg::kOffQLo);
    auto sK = [&](int s) { return smem_addr(smem + Cfg::kOffK + s * Cfg::kSlotBytes); };
    auto sV = [&](int s) { return smem_addr(smem + Cfg::kOffV + s * Cfg::kSlotBytes); };

    if (warp == 9 || warp == 10) {
        // ---- TMA loaders: warp 9 the K tiles, warp 10 the V tiles.  Key tile t (counted over
        // all work tiles) goes to slot t % N once the slot's previous tile is consumed.  Lane
        // i < PPT * PANELS copies panel i % PANELS of page i / PANELS of the tile; the
        // block-table entries come 32 at a time.
        const bool is_k = warp == 9;
        const int N = is_k ? NK : NV;
        const int full0 = is_k ? Cfg::kKFull : Cfg::kVFull, free0 = is_k ? Cfg::kKFree : Cfg::kVFree;
        const CUtensorMap *map = is_k ? &tm_k : &tm_v;
        const int oob_row = p.NB * p.Hkv * BS;
        const int pg = lane / PANELS, pn = lane % PANELS;
        int t = 0;
        bool alive = true;
        for (int it = blockIdx.x; it < n_items && alive; it += G) {
            const PPItem w = pp_item<BS, kShared>(p, it, gx, gy, false);
            if (w.kind != kWork) continue;
            const int pbase = w.kt0 * PPT;              // the first page read
            const int npg = w.npages - pbase;            // pages from there to the last key
            const int32_t *tbl = w.tbl_row + pbase;
            int tcur = lane < npg ? __ldg(tbl + lane) : -1;
            int tbase = 0;
            for (int j = 0; j < w.ntiles; ++j) {
                bool fr = true;
                if (lane == 0 && t >= N) fr = wait_or_abort(bar(free0 + t % N), ((t - N) / N) & 1, abort, p.err);
                if (!__shfl_sync(kFull, fr ? 1 : 0, 0)) {
                    alive = false;
                    break;
                }
                const int s = t % N;
                if (j * PPT >= tbase + 32) {   // a tile never straddles 32 pages (32 % PPT == 0)
                    tbase += 32;
                    tcur = tbase + lane < npg ? __ldg(tbl + tbase + lane) : -1;
                }
                const int k = j * PPT + pg;
                const int phys = __shfl_sync(kFull, tcur, k & 31);
                if (lane == 0) mbar_arrive_expect_tx(bar(full0 + s), Cfg::kSlotBytes);
                __syncwarp();
                if (lane < PPT * PANELS) {
                    int row = oob_row;
                    if (k < npg) {
                        if (phys < 0 || phys >= p.NB) {
                            if (is_k && pn == 0) raise_error(p.err, PKV_DEVERR_BLOCK);
                        } else {
                            row = (phys * p.Hkv + w.kvh) * BS;
                        }
                    }
                    const uint32_t dst = (is_k ? sK(s) : sV(s)) + pn * TK * 128 + pg * BS * 128;
                    tma_load_2d(dst, map, pn * 64, row, bar(full0 + s));
                }
                ++t;
            }
        }
        // before teardown every copy issued must have landed (bounded)
        if (lane == 0)
            for (int u = max(0, t - N); u < t; ++u)
                if (!mbar_wait_bounded(bar(full0 + u % N), (u / N) & 1)) raise_error(p.err, PKV_DEVERR_TIMEOUT);
    } else if (warp == 8 || warp == 11) {
        // ---- MMA issue, one lane each: warp 11 the scores, warp 8 the products with V.
        // tcgen05.commit covers the committing thread's MMAs: warp 11 signals S full, K free
        // and, after a work tile's last scores, Q free; warp 8 P consumed, V free and, after
        // a work tile's last P.V, O done.  Buffer g % 3's barriers complete once per use, no
        // use starts before the previous one is consumed, and a work tile's barriers complete
        // once per work tile with the next one waiting for this one's consumer, so each
        // wait's phase is unambiguous.
        if (lane == 0) {
            const bool is_s = warp == 11;
            bool issued = false, alive = true;
            int g = 0, cnt = 0;   // key tiles and work tiles done
            if (is_s) {
                const uint32_t idesc_s = umma_idesc_bf16(BM, TK, 0);
                for (int it = blockIdx.x; it < n_items && alive; it += G) {
                    const PPItem w = pp_item<BS, kShared>(p, it, gx, gy, false);
                    if (w.kind != kWork) continue;
                    alive = wait_or_abort(bar(Cfg::kQ), cnt & 1, abort, p.err);
                    for (int j = 0; j < w.ntiles && alive; ++j) {
                        const int sb = g % NSP;
                        if (g >= NSP) alive = wait_or_abort(bar(Cfg::kPFree + sb), ((g - NSP) / NSP) & 1, abort, p.err);
                        alive = alive && wait_or_abort(bar(Cfg::kKFull + g % NK), (g / NK) & 1, abort, p.err);
                        if (!alive) break;
                        tc_fence_after_sync();
                        const int s = g % NK;
#pragma unroll
                        for (int part = 0; part < 2; ++part)
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint64_t ad = umma_desc_sw128((part ? sQLo : sQHi) + (kk / 4) * BM * 128 +
                                                                        (kk % 4) * 32, 16, 1024);
                                const uint64_t bd =
                                    umma_desc_sw128(sK(s) + (kk / 4) * TK * 128 + (kk % 4) * 32, 16, 1024);
                                umma_bf16(tmem + Cfg::kSCol + sb * TK, ad, bd, idesc_s, (part > 0 || kk > 0) ? 1u : 0u);
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
            } else {
                const uint32_t idesc_o = umma_idesc_bf16(BM, D, 1);
                for (int it = blockIdx.x; it < n_items && alive; it += G) {
                    const PPItem w = pp_item<BS, kShared>(p, it, gx, gy, false);
                    if (w.kind != kWork) continue;
                    for (int j = 0; j < w.ntiles && alive; ++j) {
                        const int sb = g % NSP;
                        alive = wait_or_abort(bar(Cfg::kPFull + sb), (g / NSP) & 1, abort, p.err) &&
                                wait_or_abort(bar(Cfg::kVFull + g % NV), (g / NV) & 1, abort, p.err);
                        // the first product of a work tile overwrites O: the previous one read
                        if (alive && j == 0 && cnt > 0)
                            alive = wait_or_abort(bar(Cfg::kOFree), (cnt - 1) & 1, abort, p.err);
                        if (!alive) break;
                        tc_fence_after_sync();
                        const int s = g % NV;
#pragma unroll
                        for (int half = 0; half < 2; ++half)
#pragma unroll
                            for (int kk = 0; kk < TK / 16; ++kk) {
                                // keys 16 kk .. 16 kk + 15: P_hi (half 0) or P_lo of the keys' 64-key half
                                const uint32_t pcol = Cfg::kSCol + sb * TK + (kk / 4) * 64 + half * 32 + (kk % 4) * 8;
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
        // ---- softmax: thread (w, lane) owns row r = 32 (w % 4) + lane (tensor-memory lane r)
        // and keys 64h .. 64h + 63 of each key tile (h = w / 4)
        const int h = warp >> 2;
        const int r = ((warp & 3) << 5) | lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const int pair_bar = 1 + (warp & 3);   // named barrier of warps w and w + 4
        auto xs = [&](int buf, int kind, int hh) { return xch + ((buf * 2 + kind) * 2 + hh) * BM + r; };
        // ok is warp-uniform, and after each key tile's exchange the same in both warps of a
        // row: a failed wait skips the remaining work but never a named barrier (the warps
        // walk every key tile of every work tile either way)
        bool ok = true;
        int g = 0, cnt = 0;
        for (int it = blockIdx.x; it < n_items; it += G) {
            const PPItem w = pp_item<BS, kShared>(p, it, gx, gy, false);
            if (w.kind != kWork) continue;
            const bool row_ok = r < w.nrows;
            const int qpos = w.P0 + r;   // chunked prefill: this row's position, keys 0 .. qpos
            // The last page may end inside its block: V rows past the last key are zeroed
            const int tail_valid = w.key_end - (w.npages - 1) * BS;   // 1..BS tokens (BS for a prefix)
            const int tail_tile = (w.npages - 1) / PPT - w.kt0;
            const int tail_row0 = ((w.npages - 1) % PPT) * BS + tail_valid;
            const int tail_rows = BS - tail_valid;
            float m_ref = -INFINITY, l = 0.f;
            for (int j = 0; j < w.ntiles; ++j, ++g) {
                const int sb = g & 1;              // exchange buffer
                const int pb = g % NSP;            // S / P buffer
                const uint32_t scol = lane_base + Cfg::kSCol + pb * TK + h * 64;
                if (ok) ok = __all_sync(kFull, wait_or_abort(bar(Cfg::kSFull + pb), (g / NSP) & 1, abort, p.err));
                float sc[64];
                if (ok) {
                    tc_fence_after_sync();
                    uint32_t s0[32], s1[32];
                    tmem_ld32(scol, s0);
                    tmem_ld32(scol + 32, s1);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        sc[c] = __uint_as_float(s0[c]);
                        sc[32 + c] = __uint_as_float(s1[c]);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 64; ++c) sc[c] = -INFINITY;
                }
                if (ok && j == tail_tile && tail_rows > 0) {
                    // once the V copies of this tile have landed
                    ok = __all_sync(kFull, wait_or_abort(bar(Cfg::kVFull + g % NV), (g / NV) & 1, abort, p.err));
                    if (ok) {
                        uint8_t *vt = smem + Cfg::kOffV + (g % NV) * Cfg::kSlotBytes;
                        for (int idx = threadIdx.x; idx < tail_rows * PANELS * 8; idx += 256) {
                            const int row = tail_row0 + idx / (PANELS * 8), rem = idx % (PANELS * 8);
                            *reinterpret_cast<uint4 *>(vt + (rem >> 3) * TK * 128 + row * 128 + (rem & 7) * 16) =
                                make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                    }
                }
                const int key0 = (w.kt0 + j) * TK + h * 64;
                if constexpr (kShared) {
                    // every row sees every prefix key; keys past the prefix and rows past the
                    // group's pairs see nothing
                    if (key0 + 63 >= w.key_end || !row_ok) {
#pragma unroll
                        for (int c = 0; c < 64; ++c)
                            if (key0 + c >= w.key_end || !row_ok) sc[c] = -INFINITY;
                    }
                } else {
                    // bottom-right causal mask: key <= this row's position; a row past nq sees nothing
                    if (key0 + 63 > w.P0 || !row_ok) {
#pragma unroll
                        for (int c = 0; c < 64; ++c)
                            if (key0 + c > qpos || !row_ok) sc[c] = -INFINITY;
                    }
                }
                float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < 64; ++c) mx4[c & 3] = fmaxf(mx4[c & 3], sc[c]);
                float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
                // the other half's maximum of this row, and whether it is still ok; the
                // exchange buffer alternates with the key tile, so one barrier a tile suffices
                *xs(sb, 0, h) = mx;
                *xs(sb, 1, h) = ok ? 1.f : 0.f;
                named_barrier(pair_bar, 64);
                mx = fmaxf(mx, *xs(sb, 0, 1 - h)) * p.scale_log2;
                ok = ok && *xs(sb, 1, 1 - h) != 0.f;
                if (!ok) continue;
                // a row that has seen no key yet (one past nq) keeps m = -inf and weight 0
                const float m_new = mx > m_ref + 8.f ? mx : m_ref;
                const float alpha = m_new == m_ref ? 1.f : ex2_approx(m_ref - m_new);
                m_ref = m_new;
                const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
                // the keys as packed fp32 pairs: one FMA and one add a pair
                const float2 sl2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(neg_m, neg_m);
                float2 l2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    float2 x = fma2(make_float2(sc[2 * c], sc[2 * c + 1]), sl2, nm2);
                    x.x = ex2_approx(x.x);
                    x.y = ex2_approx(x.y);
                    l2[c & 1] = add2(l2[c & 1], x);
                    sc[2 * c] = x.x;
                    sc[2 * c + 1] = x.y;
                }
                l = l * alpha + ((l2[0].x + l2[0].y) + (l2[1].x + l2[1].y));
                // the weights over this thread's own scores (already in registers), 32 keys at
                // a time: P_hi of keys 2e, 2e + 1 in column e, P_lo in column 32 + e
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t phi[16], plo[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        split_bf16x2_p(sc[32 * q + 2 * e], sc[32 * q + 2 * e + 1], phi[e], plo[e]);
                    tmem_st16(scol + 16 * q, phi);
                    tmem_st16(scol + 32 + 16 * q, plo);
                }
                // a rescale of O waits for the previous P.V of this work tile (and so every
                // earlier one): O is then current, and this tile's P.V waits for its P
                if (j > 0 && __any_sync(kFull, alpha != 1.f)) {
                    const int qb = (g - 1) % NSP;
                    ok = __all_sync(kFull, wait_or_abort(bar(Cfg::kPFree + qb), ((g - 1) / NSP) & 1, abort, p.err));
                    if (!ok) continue;
                    tc_fence_after_sync();
                    // this half rescales columns D/2 h .. D/2 h + D/2 - 1 of its rows
#pragma unroll
                    for (int cc = 0; cc < D / 64; ++cc) {
                        uint32_t ov[32];
                        tmem_ld32(lane_base + Cfg::kOCol + h * (D / 2) + cc * 32, ov);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                        tmem_st32(lane_base + Cfg::kOCol + h * (D / 2) + cc * 32, ov);
                    }
                }
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(Cfg::kPFull + pb));
            }
            // the row's maximum and this half's sum for the epilogue warps (the buffer was
            // read by them two work tiles ago)
            const int sbuf = cnt & 1;
            if (ok && cnt >= 2)
                ok = __all_sync(kFull, wait_or_abort(bar(Cfg::kStFree + sbuf), ((cnt - 2) >> 1) & 1, abort, p.err));
            if (ok) {
                if (h == 0) stats[(sbuf * 3) * BM + r] = m_ref;
                stats[(sbuf * 3 + 1 + h) * BM + r] = l;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(Cfg::kStFull + sbuf));
            }
            ++cnt;
        }
    } else {
        // ---- queries and epilogue: thread (w, lane) handles row r = 32 (w % 4) + lane
        const int r = ((warp & 3) << 5) | lane;
        const int et = threadIdx.x - 12 * 32;   // 0 .. 127
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        float *stage = reinterpret_cast<float *>(smem + Cfg::kOffStage) + (warp & 3) * 32 * Cfg::kPitch;
        bool ok = true;
        int qcnt = 0, ocnt = 0;   // Q tiles written, outputs written
        PPItem prev{};
        bool have_prev = false;
        // O / l and the log-sum-exp of work tile w (its ocnt-th)
        auto output = [&](const PPItem &w) {
            const int sbuf = ocnt & 1;
            ok = ok && __all_sync(kFull, wait_or_abort(bar(Cfg::kStFull + sbuf), (ocnt >> 1) & 1, abort, p.err)) &&
                 __all_sync(kFull, wait_or_abort(bar(Cfg::kODone), ocnt & 1, abort, p.err));
            if (!ok) return;
            tc_fence_after_sync();
            const float m = stats[(sbuf * 3) * BM + r];
            const float lr = stats[(sbuf * 3 + 1) * BM + r] + stats[(sbuf * 3 + 2) * BM + r];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Cfg::kStFree + sbuf));
            const float inv_l = lr > 0.f ? 1.f / lr : 0.f;
            const int wrow0 = (warp & 3) << 5;
            const int wrows = min(32, w.nrows - wrow0);   // rows of the warp inside the tile
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t ov[32];
                tmem_ld32(lane_base + Cfg::kOCol + c * 32, ov);
                tmem_ld_wait();
                if (c == D / 32 - 1) {
                    // O has been read: the next work tile's first P.V may overwrite it
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
                    if (rr < wrows) {
                        int bq, hq;
                        size_t member;
                        pp_row<kShared>(p, w, wrow0 + rr, bq, hq, member);
                        // chunked prefill: the output row; shared prefix: this split's normalised partial
                        float *dst = kShared ? p.ws_o + ((member * p.Hq + hq) * p.prefix_splits + w.ks) * D
                                             : p.out + (static_cast<size_t>(bq) * p.Hq + hq) * D;
                        *reinterpret_cast<float4 *>(dst + c * 32 + (lane & 7) * 4) =
                            *reinterpret_cast<const float4 *>(stage + rr * Cfg::kPitch + (lane & 7) * 4);
                    }
                }
                __syncwarp();
            }
            if (r < w.nrows) {
                int bq, hq;
                size_t member;
                pp_row<kShared>(p, w, r, bq, hq, member);
                const float lse2 = m == -INFINITY ? -INFINITY : m + log2f(lr);
                if constexpr (kShared)
                    p.ws_lse[(member * p.Hq + hq) * p.prefix_splits + w.ks] = lse2;
                else if (p.lse != nullptr)
                    p.lse[static_cast<size_t>(bq) * p.Hq + hq] = lse2 * kDecLn2;
            }
            ++ocnt;
        };
        for (int it = blockIdx.x; it < n_items && ok; it += G) {
            const PPItem w = pp_item<BS, kShared>(p, it, gx, gy, warp == 12 && lane == 0);
            if (w.kind == kEmpty) {
                // no prefix key in this split: empty partials
                for (int idx = et; idx < w.nrows * D; idx += 128) {
                    const int rho = w.r0 + idx / D;
                    const size_t slot = (static_cast<size_t>(w.gs + rho / p.m) * p.Hq + w.kvh * p.m + rho % p.m) *
                                            p.prefix_splits + w.ks;
                    p.ws_o[slot * D + idx % D] = 0.f;
                    if (idx % D == 0) p.ws_lse[slot] = -INFINITY;
                }
                continue;
            }
            if (w.kind == kBadRows) {
                // inconsistent rows: out = 0, lse = -inf (as the other query-row kernels)
                for (int idx = et; idx < min(max(w.nq, 0), BM) * D; idx += 128) {
                    const size_t bi = static_cast<size_t>(w.c0 + idx / D) * p.Hq + w.head;
                    p.out[bi * D + idx % D] = 0.f;
                    if (idx % D == 0 && p.lse != nullptr) p.lse[bi] = -INFINITY;
                }
                continue;
            }
            if (w.kind != kWork) continue;
            // this work tile's queries, over the previous tile's once its scores are computed
            if (qcnt > 0) ok = __all_sync(kFull, wait_or_abort(bar(Cfg::kQFree), (qcnt - 1) & 1, abort, p.err));
            if (!ok) break;
            {
                const bool row_ok = r < w.nrows;
                int bq, hq;
                size_t member;
                pp_row<kShared>(p, w, row_ok ? r : 0, bq, hq, member);
                const float *qrow = p.q + (static_cast<size_t>(bq) * p.Hq + hq) * D;
#pragma unroll 4
                for (int c8 = 0; c8 < D / 8; ++c8) {   // 8 columns (16 bytes of each part) at a time
                    float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
                    if (row_ok) {
                        x0 = __ldg(reinterpret_cast<const float4 *>(qrow + 8 * c8));
                        x1 = __ldg(reinterpret_cast<const float4 *>(qrow + 8 * c8 + 4));
                    }
                    uint4 hi, lo;
                    split_bf16x2(x0.x, x0.y, hi.x, lo.x);
                    split_bf16x2(x0.z, x0.w, hi.y, lo.y);
                    split_bf16x2(x1.x, x1.y, hi.z, lo.z);
                    split_bf16x2(x1.z, x1.w, hi.w, lo.w);
                    const uint32_t off = swz128(BM, r, 8 * c8);
                    *reinterpret_cast<uint4 *>(smem + Cfg::kOffQHi + off) = hi;
                    *reinterpret_cast<uint4 *>(smem + Cfg::kOffQLo + off) = lo;
                }
                fence_proxy_async_smem();   // the tensor core reads these through the async proxy
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(Cfg::kQ));
                ++qcnt;
            }
            // the previous work tile's output
            if (have_prev) output(prev);
            prev = w;
            have_prev = true;
        }
        if (ok && have_prev) output(prev);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, Cfg::kTmemCols);
}

template <int D, int BS, bool kShared>
cudaError_t launch_pp(const DecodeKParams &kp, const CUtensorMap &tk, const CUtensorMap &tv, dim3 grid,
                      cudaStream_t stream) {
    using Cfg = PagedPrefillCfg<D, BS>;
    auto kernel = paged_prefill_kernel<D, BS, kShared>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    // the work tiles of `grid`, walked by one CTA per SM
    const long long n_items = static_cast<long long>(grid.x) * grid.y * grid.z;
    if (n_items == 0) return cudaSuccess;
    if (n_items >= (1ll << 31)) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const unsigned ctas = static_cast<unsigned>(min(static_cast<long long>(sms), n_items));
    kernel<<<ctas, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(tk, tv, kp, static_cast<int>(grid.x),
                                                             static_cast<int>(grid.y), static_cast<int>(n_items));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_paged_prefill(const DecodeKParams &kp, const CUtensorMap &tk, const CUtensorMap &tv, int d,
                                 int bs, dim3 grid, cudaStream_t stream) {
    if (d == 128) return bs == 16 ? launch_pp<128, 16, false>(kp, tk, tv, grid, stream)
                                  : launch_pp<128, 32, false>(kp, tk, tv, grid, stream);
    if (d == 64) return bs == 16 ? launch_pp<64, 16, false>(kp, tk, tv, grid, stream)
                                 : launch_pp<64, 32, false>(kp, tk, tv, grid, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_shared_prefix(const DecodeKParams &kp, const CUtensorMap &tk, const CUtensorMap &tv, int d,
                                 int bs, dim3 grid, cudaStream_t stream) {
    if (d == 128) return bs == 16 ? launch_pp<128, 16, true>(kp, tk, tv, grid, stream)
                                  : launch_pp<128, 32, true>(kp, tk, tv, grid, stream);
    if (d == 64) return bs == 16 ? launch_pp<64, 16, true>(kp, tk, tv, grid, stream)
                                 : launch_pp<64, 32, true>(kp, tk, tv, grid, stream);
    return cudaErrorInvalidValue;
}

namespace {

// One warp per (member, query head): sequence b's attention over its group's prefix (the
// prefix kernel's partials, lse in base 2) and over its own keys after the prefix (the
// decode's result in out, its natural-log lse in suffix_lse) merge by log-sum-exp --
// lse = log2 sum 2^{lse_k}, out = sum 2^{lse_k - lse} o_k (plumephp.com "KV Cache 优化与注意
// 力机制加速" §2.2-§2.3 applied to the two key sets).  The head-0 warp of each member checks
// that the member's prefix matches the group's first member (same length, a whole number
// of blocks below the member's last position, the same physical blocks) and raises
// PKV_DEVERR_PREFIX otherwise.
template <int D>
__global__ void __launch_bounds__(256)
    shared_prefix_merge_kernel(const DecodeKParams p, const float *suffix_lse, int bs, int n_groups, int n_members) {
    const int lane = threadIdx.x & 31;
    const long long wid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (wid >= static_cast<long long>(n_members) * p.Hq) return;
    const int member = static_cast<int>(wid / p.Hq), hq = static_cast<int>(wid % p.Hq);
    const int b = __ldg(p.group_seqs + member);
    if (b < 0 || b >= p.B) {   // a member that is no sequence of the batch: flagged, skipped
        if (hq == 0 && lane == 0) raise_error(p.err, PKV_DEVERR_PREFIX);
        return;
    }
    if (hq == 0) {
        int lo = 0, hi = n_groups;   // the group: cu_q[g] <= member < cu_q[g + 1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(p.cu_q + mid) <= member) lo = mid;
            else hi = mid;
        }
        const int g0 = __ldg(p.cu_q + lo);
        int first = g0 >= 0 && g0 < n_members ? __ldg(p.group_seqs + g0) : -1;
        if (first < 0 || first >= p.B) first = b;   // (flagged below: the offsets or ids are bad)
        const int P = __ldg(p.kv_start + b), len = __ldg(p.context_lens + b);
        const bool good = g0 >= 0 && g0 < n_members && __ldg(p.group_seqs + g0) == first &&
                          P == __ldg(p.kv_start + first) && P >= 0 && P % bs == 0 && P <= len - 1 &&
                          len <= p.MBS * bs;
        // the leading blocks, compared without a test between loads so that they are in flight together
        const int nb = good ? P / bs : 0;
        const int32_t *tb = p.block_table + static_cast<size_t>(b) * p.MBS;
        const int32_t *tf = p.block_table + static_cast<size_t>(first) * p.MBS;
        int diff = 0;
#pragma unroll 4
        for (int j = lane; j < nb; j += 32) diff |= __ldg(tb + j) ^ __ldg(tf + j);
        if (!__all_sync(kFull, good && diff == 0) && lane == 0) raise_error(p.err, PKV_DEVERR_PREFIX);
    }
    const size_t row = static_cast<size_t>(b) * p.Hq + hq;
    const size_t part = (static_cast<size_t>(member) * p.Hq + hq) * p.prefix_splits;
    const int S = p.prefix_splits;
    const float ls = __ldg(suffix_lse + row) * kDecLog2e;   // base 2
    float M = ls;
    for (int k = lane; k < S; k += 32) M = fmaxf(M, __ldcg(p.ws_lse + part + k));
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, sh));
    constexpr int CPL = D / 32;   // columns per lane
    float acc[CPL];
    const float ws = M == -INFINITY ? 0.f : ex2_approx(ls - M);
    float L = ws;
#pragma unroll
    for (int e = 0; e < CPL; ++e) acc[e] = ws * p.out[row * D + lane * CPL + e];
    // four partials at a time: their loads are in flight together
    for (int k0 = 0; k0 < S; k0 += 4) {
        float lk[4], v[4][CPL];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int k = min(k0 + u, S - 1);
            lk[u] = k0 + u < S ? __ldcg(p.ws_lse + part + k) : -INFINITY;
            const float *po = p.ws_o + (part + k) * D + lane * CPL;
            if constexpr (CPL == 4) {
                const float4 x = __ldcg(reinterpret_cast<const float4 *>(po));
                v[u][0] = x.x;
                v[u][1] = x.y;
                v[u][2] = x.z;
                v[u][3] = x.w;
            } else {
                const float2 x = __ldcg(reinterpret_cast<const float2 *>(po));
                v[u][0] = x.x;
                v[u][1] = x.y;
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float w = M == -INFINITY ? 0.f : ex2_approx(lk[u] - M);   // 0 past the last partial
            L += w;
#pragma unroll
            for (int e = 0; e < CPL; ++e) acc[e] += w * v[u][e];
        }
    }
    const float il = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int e = 0; e < CPL; ++e) p.out[row * D + lane * CPL + e] = acc[e] * il;
    if (lane == 0 && p.lse != nullptr) p.lse[row] = L > 0.f ? (M + log2f(L)) * kDecLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_shared_prefix_merge(const DecodeKParams &kp, const float *suffix_lse, int d, int bs,
                                       int n_groups, int n_members, cudaStream_t stream) {
    const long long warps = static_cast<long long>(n_members) * kp.Hq;
    if (warps == 0) return cudaSuccess;
    const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);
    if (d == 128) shared_prefix_merge_kernel<128><<<blocks, 256, 0, stream>>>(kp, suffix_lse, bs, n_groups, n_members);
    else if (d == 64) shared_prefix_merge_kernel<64><<<blocks, 256, 0, stream>>>(kp, suffix_lse, bs, n_groups, n_members);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace pkv
