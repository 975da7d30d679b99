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
// The tile is the prefill kernel's (prefill.cu): one CTA per (128 query rows of one head,
// head, sequence), 128-key tiles, twelve warps.  What differs:
//   - the queries are fp32: the softmax warps split each into bf16 hi + lo parts and store
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
    static constexpr int kQBytes = kBM * D * 2;        // one Q part: D/64 panels of [128][128 B]
    static constexpr int kSlotBytes = kTK * D * 2;     // one K or V tile
    static constexpr int kOffQHi = 0, kOffQLo = kQBytes;
    static constexpr int kOffK = 2 * kQBytes;
    static constexpr int kOffV = kOffK + NK * kSlotBytes;
    static constexpr int kOffBar = kOffV + NV * kSlotBytes;
    static constexpr int NSP = 3;                       // S / P buffers in tensor memory
    // barriers: Q written; K full / free per slot; V full / free per slot; per S/P buffer: S
    // full, P full, P consumed (its P.V done); all MMAs done; drain x2 (one per MMA-issuing
    // thread)
    static constexpr int kQ = 0, kKFull = 1, kKFree = 1 + NK, kVFull = 1 + 2 * NK, kVFree = 1 + 2 * NK + NV,
                         kSFull = 1 + 2 * NK + 2 * NV, kPFull = kSFull + NSP, kPFree = kPFull + NSP,
                         kDone = kPFree + NSP, kDrain = kDone + 1, kNumBars = kDrain + 2;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;          // TMEM slot, abort flag
    // row exchange of the two warps of a row, double-buffered by tile parity:
    // [buffer][value, ok][half][128 rows] floats
    static constexpr int kOffXch = (kOffMisc + 16 + 15) / 16 * 16;
    static constexpr int kSmemBytes = 1024 + kOffXch + 2 * 2 * 2 * kBM * 4;
    // tensor memory: NSP S buffers of 128 columns, then O.  The weights of tile j overwrite
    // its scores: the thread that read S columns 64h .. 64h + 63 of a row writes P_hi of
    // those keys to columns 64h .. 64h + 31 of the buffer and P_lo to 64h + 32 .. 64h + 63.
    static constexpr int kTmemCols = 512;
    static constexpr int kSCol = 0, kOCol = NSP * kTK;
    static constexpr int kThreads = 384;
    static_assert(D == 64 || D == 128, "head size");
    static_assert(BS == 16 || BS == 32, "block size");
    static_assert(kOCol + D <= kTmemCols, "tensor memory budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kPPT * PANELS <= 32 && 32 % kPPT == 0, "one box per loader lane; tiles within 32 pages");
    static_assert(8 * 32 * (D / 2 + 4) * 4 <= (NK + NV) * kSlotBytes, "the output staging fits the K/V rings");
};

// One CTA per (query tile, query head, sequence); twelve warps:
//   warps 9 and 10 (TMA): the K and the V tiles into two rings, one {64, bs} box (one page,
//     one panel) per lane; a K slot is free once its scores are computed, a V slot once
//     its P.V is.  A page past the keys any row sees is placed outside the cache, where TMA
//     fills zeros.
//   warps 11 and 8 (one lane each issues): S_j = Q_hi K_j^T + Q_lo K_j^T (N = 128 keys)
//     into tensor-memory buffer j % 3, once K_j has landed and, for j >= 3, P_{j-3} V_{j-3}
//     (which read that buffer) is done; O += P_hi V_j + P_lo V_j (N = d), P read from the
//     same buffer.  With three buffers the softmax of tile j never waits for a P.V unless
//     it rescales O, and the scores of the next tiles are computed while it runs.
//   warps 0-7 (softmax): first the queries -- thread (w, lane) loads row r = 32 (w % 4) +
//     lane, columns D/2 h .. D/2 h + D/2 - 1 (h = w / 4), splits them and stores both parts;
//     then per key tile the prefill kernel's online softmax for row r over keys 64h ..
//     64h + 63 of the tile, with the bottom-right causal mask.
template <int D, int BS, bool kShared>
__global__ void __launch_bounds__(384, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const DecodeKParams p) {
    using Cfg = PagedPrefillCfg<D, BS>;
    constexpr int BM = Cfg::kBM, TK = Cfg::kTK, PPT = Cfg::kPPT, PANELS = Cfg::PANELS, NK = Cfg::NK,
                  NV = Cfg::NV;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 4);
    float *xch = reinterpret_cast<float *>(smem + Cfg::kOffXch);
    auto bar = [&](int k) { return smem_addr(&bars[k]); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The rows of the tile and the keys they see.
    //   chunked prefill: rows r0 .. r0 + nrows - 1 of sequence b's nq query rows, head `head`,
    //     row r at position P0 + r seeing keys 0 .. P0 + r (pages from block_table[b]);
    //   shared prefix: rows rho = 128 rt .. of the group's (member, head) pairs, rho = mu m + hh
    //     for member mu and head kvh m + hh, all seeing the group's prefix keys of this split:
    //     key tiles kt0 .. kt0 + ntiles - 1 of the prefix (pages from the first member's row).
    int b = 0, head = 0, kvh = 0, c0 = 0, r0 = 0, nrows = 0, P0 = 0, key_end = 0, npages = 0, ntiles = 0;
    int kt0 = 0, gs = 0, ks = 0;
    const int32_t *tbl_row = nullptr;
    if constexpr (kShared) {
        ks = blockIdx.x;
        kvh = blockIdx.y;
        const int g = blockIdx.z / p.prefix_rtiles, rt = blockIdx.z % p.prefix_rtiles;
        gs = __ldg(p.cu_q + g);
        const int nmem = __ldg(p.cu_q + g + 1) - gs;
        if (gs < 0 || nmem < 0 || gs + nmem > p.n_members ||
            static_cast<long long>(nmem) * p.m > static_cast<long long>(p.prefix_rtiles) * BM) {
            // offsets outside the member list, or a group larger than the declared maximum
            if (threadIdx.x == 0 && ks == 0 && kvh == 0 && rt == 0) raise_error(p.err, PKV_DEVERR_PREFIX);
            return;
        }
        r0 = rt * BM;
        nrows = min(BM, nmem * p.m - r0);
        if (nrows <= 0) return;
        const int first = __ldg(p.group_seqs + gs);
        if (first < 0 || first >= p.B) {
            if (threadIdx.x == 0 && ks == 0 && kvh == 0 && rt == 0) raise_error(p.err, PKV_DEVERR_PREFIX);
            return;
        }
        int P = __ldg(p.kv_start + first);
        if (P < 0 || P % BS != 0 || P > p.MBS * BS) P = 0;   // flagged by the merge
        const int KT = (P + TK - 1) / TK;
        const int kps = (KT + p.prefix_splits - 1) / p.prefix_splits;
        kt0 = ks * kps;
        ntiles = min(KT, kt0 + kps) - kt0;
        key_end = P;
        npages = P / BS;
        tbl_row = p.block_table + static_cast<size_t>(first) * p.MBS;
        if (ntiles <= 0) {   // no prefix key in this split: empty partials
            for (int idx = threadIdx.x; idx < nrows * D; idx += blockDim.x) {
                const int rho = r0 + idx / D;
                const size_t slot = (static_cast<size_t>(gs + rho / p.m) * p.Hq + kvh * p.m + rho % p.m) *
                                        p.prefix_splits + ks;
                p.ws_o[slot * D + idx % D] = 0.f;
                if (idx % D == 0) p.ws_lse[slot] = -INFINITY;
            }
            return;
        }
    } else {
        const int qt = blockIdx.x;
        head = blockIdx.y;
        b = blockIdx.z;
        const bool report = threadIdx.x == 0 && qt == 0 && head == 0;
        const int L = checked_len(p, b, BS, report);
        c0 = __ldg(p.cu_q + b);
        const int nq = __ldg(p.cu_q + b + 1) - c0;
        r0 = qt * BM;                     // the tile's first query row
        if (nq < 0 || nq > L) {
            if (report) raise_error(p.err, PKV_DEVERR_CU_SEQLENS);
            // inconsistent rows: out = 0, lse = -inf (as the other query-row kernels)
            if (r0 == 0)
                for (int rr = 0; rr < min(max(nq, 0), BM); ++rr) {
                    const size_t bi = static_cast<size_t>(c0 + rr) * p.Hq + head;
                    for (int e = threadIdx.x; e < D; e += blockDim.x) p.out[bi * D + e] = 0.f;
                    if (threadIdx.x == 0 && p.lse != nullptr) p.lse[bi] = -INFINITY;
                }
            return;
        }
        if (r0 >= nq) return;
        nrows = min(BM, nq - r0);         // rows of this tile
        P0 = L - nq + r0;                 // position of the tile's first row
        key_end = P0 + nrows;             // one past the last key any row of the tile sees
        npages = (key_end + BS - 1) / BS;
        ntiles = (key_end + TK - 1) / TK;
        kvh = head / p.m;
        tbl_row = p.block_table + static_cast<size_t>(b) * p.MBS;
    }
    const int pbase = kt0 * PPT;                 // the first page read
    const int npg = npages - pbase;              // pages from there to the last key

    if (threadIdx.x == 0) {
        mbar_init(bar(Cfg::kQ), 8);
        for (int s = 0; s < NK; ++s) {
            mbar_init(bar(Cfg::kKFull + s), 1);
            mbar_init(bar(Cfg::kKFree + s), 1);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(bar(Cfg::kVFull + s), 1);
            mbar_init(bar(Cfg::kVFree + s), 1);
        }
        for (int u = 0; u < Cfg::NSP; ++u) {
            mbar_init(bar(Cfg::kSFull + u), 1);
            mbar_init(bar(Cfg::kPFull + u), 8);
            mbar_init(bar(Cfg::kPFree + u), 1);
        }
        mbar_init(bar(Cfg::kDone), 1);
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
        // ---- TMA loaders: warp 9 the K tiles, warp 10 the V tiles.  Tile t goes to slot
        // t % N once the slot's previous tile is consumed.  Lane i < PPT * PANELS copies panel
        // i % PANELS of page i / PANELS of the tile; the block-table entries come 32 at a time.
        const bool is_k = warp == 9;
        const int N = is_k ? NK : NV;
        const int full0 = is_k ? Cfg::kKFull : Cfg::kVFull, free0 = is_k ? Cfg::kKFree : Cfg::kVFree;
        const CUtensorMap *map = is_k ? &tm_k : &tm_v;
        const int32_t *tbl = tbl_row + pbase;
        int tcur = lane < npg ? __ldg(tbl + lane) : -1;
        int tbase = 0;
        const int oob_row = p.NB * p.Hkv * BS;
        const int pg = lane / PANELS, pn = lane % PANELS;
        int t = 0;
        for (; t < ntiles; ++t) {
            bool fr = true;
            if (lane == 0 && t >= N) fr = wait_or_abort(bar(free0 + t % N), ((t - N) / N) & 1, abort, p.err);
            if (!__shfl_sync(kFull, fr ? 1 : 0, 0)) break;
            const int s = t % N;
            if (t * PPT >= tbase + 32) {   // a tile never straddles 32 pages (32 % PPT == 0)
                tbase += 32;
                tcur = tbase + lane < npg ? __ldg(tbl + tbase + lane) : -1;
            }
            const int k = t * PPT + pg;
            const int phys = __shfl_sync(kFull, tcur, k & 31);
            if (lane == 0) mbar_arrive_expect_tx(bar(full0 + s), Cfg::kSlotBytes);
            __syncwarp();
            if (lane < PPT * PANELS) {
                int row = oob_row;
                if (k < npg) {
                    if (phys < 0 || phys >= p.NB) {
                        if (is_k && pn == 0) raise_error(p.err, PKV_DEVERR_BLOCK);
                    } else {
                        row = (phys * p.Hkv + kvh) * BS;
                    }
                }
                const uint32_t dst = (is_k ? sK(s) : sV(s)) + pn * TK * 128 + pg * BS * 128;
                tma_load_2d(dst, map, pn * 64, row, bar(full0 + s));
            }
        }
        // before teardown every copy issued must have landed (bounded)
        if (lane == 0)
            for (int u = max(0, t - N); u < t; ++u)
                if (!mbar_wait_bounded(bar(full0 + u % N), (u / N) & 1)) raise_error(p.err, PKV_DEVERR_TIMEOUT);
    } else if (warp == 8 || warp == 11) {
        // ---- MMA issue, one lane each: warp 11 the scores, warp 8 the products with V.
        // tcgen05.commit covers the committing thread's MMAs: warp 11 signals S full and K
        // free, warp 8 P consumed, V free and, after the last P.V (which follows every S),
        // all MMAs done.  Buffer j % 3's barriers complete once per use (tiles j, j + 3, ..),
        // and no use starts before the previous one is consumed, so each wait's phase is
        // unambiguous.
        if (lane == 0) {
            const bool is_s = warp == 11;
            bool issued = false, alive = true;
            if (is_s) {
                const uint32_t idesc_s = umma_idesc_bf16(BM, TK, 0);
                alive = wait_or_abort(bar(Cfg::kQ), 0, abort, p.err);
                for (int t = 0; t < ntiles && alive; ++t) {
                    const int sb = t % Cfg::NSP;
                    if (t >= Cfg::NSP)
                        alive = wait_or_abort(bar(Cfg::kPFree + sb), ((t - Cfg::NSP) / Cfg::NSP) & 1, abort, p.err);
                    alive = alive && wait_or_abort(bar(Cfg::kKFull + t % NK), (t / NK) & 1, abort, p.err);
                    if (!alive) break;
                    tc_fence_after_sync();
                    const int s = t % NK;
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
                }
            } else {
                const uint32_t idesc_o = umma_idesc_bf16(BM, D, 1);
                for (int j = 0; j < ntiles && alive; ++j) {
                    const int sb = j % Cfg::NSP;
                    alive = wait_or_abort(bar(Cfg::kPFull + sb), (j / Cfg::NSP) & 1, abort, p.err) &&
                            wait_or_abort(bar(Cfg::kVFull + j % NV), (j / NV) & 1, abort, p.err);
                    if (!alive) break;
                    tc_fence_after_sync();
                    const int s = j % NV;
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
                }
                if (alive) umma_commit(bar(Cfg::kDone));
            }
            if (*abort && issued) {
                // let this thread's MMAs finish (bounded) before teardown
                const int drain = is_s ? Cfg::kDrain + 1 : Cfg::kDrain;
                umma_commit(bar(drain));
                if (!mbar_wait_bounded(bar(drain), 0)) raise_error(p.err, PKV_DEVERR_TIMEOUT);
            }
        }
    } else {
        // ---- softmax: thread (w, lane) owns query row r = 32 (w % 4) + lane (tensor-memory
        // lane r) and keys 64h .. 64h + 63 of each key tile (h = w / 4)
        const int h = warp >> 2;
        const int r = ((warp & 3) << 5) | lane;
        const bool row_ok = r < nrows;
        const int qpos = P0 + r;                  // chunked prefill: this row's position, keys 0 .. qpos
        // the (sequence, head) pair this row is: shared prefix, member mu of the group
        auto row_seq_head = [&](int rr, int &bq, int &hq, size_t &member) {
            if constexpr (kShared) {
                const int rho = r0 + rr;
                member = static_cast<size_t>(gs + rho / p.m);
                bq = __ldg(p.group_seqs + member);
                if (bq < 0 || bq >= p.B) bq = 0;   // flagged by the merge; never read out of range
                hq = kvh * p.m + rho % p.m;
            } else {
                member = 0;
                bq = c0 + r0 + rr;   // the query row
                hq = head;
            }
        };
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const int pair_bar = 1 + (warp & 3);   // named barrier of warps w and w + 4
        auto xs = [&](int buf, int kind, int hh) { return xch + ((buf * 2 + kind) * 2 + hh) * BM + r; };

        // the query row's columns D/2 h .. D/2 h + D/2 - 1, split into bf16 hi and lo parts
        // and stored as row r of the two swizzled operand tiles (zeros for rows past nq)
        {
            int bq, hq;
            size_t member;
            row_seq_head(row_ok ? r : 0, bq, hq, member);
            const float *qrow = p.q + (static_cast<size_t>(bq) * p.Hq + hq) * D + h * (D / 2);
#pragma unroll
            for (int c8 = 0; c8 < D / 16; ++c8) {   // 8 columns (16 bytes of each part) at a time
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
                const uint32_t off = swz128(BM, r, h * (D / 2) + 8 * c8);
                *reinterpret_cast<uint4 *>(smem + Cfg::kOffQHi + off) = hi;
                *reinterpret_cast<uint4 *>(smem + Cfg::kOffQLo + off) = lo;
            }
            fence_proxy_async_smem();   // the tensor core reads these through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Cfg::kQ));
        }

        // The last page may end inside its block: V rows past the last key are zeroed
        const int tail_valid = key_end - (npages - 1) * BS;   // 1..BS tokens (BS for a prefix)
        const int tail_tile = (npages - 1) / PPT - kt0;
        const int tail_row0 = ((npages - 1) % PPT) * BS + tail_valid;
        const int tail_rows = BS - tail_valid;
        float m_ref = -INFINITY, l = 0.f;
        // ok is warp-uniform, and after each tile's exchange the same in both warps of a
        // row: a failed wait skips the remaining work but never a named barrier
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int sb = j & 1;              // exchange buffer
            const int pb = j % Cfg::NSP;       // S / P buffer
            const uint32_t scol = lane_base + Cfg::kSCol + pb * TK + h * 64;
            if (ok)
                ok = __all_sync(kFull, wait_or_abort(bar(Cfg::kSFull + pb), (j / Cfg::NSP) & 1, abort, p.err));
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
                ok = __all_sync(kFull, wait_or_abort(bar(Cfg::kVFull + j % NV), (j / NV) & 1, abort, p.err));
                if (ok) {
                    uint8_t *vt = smem + Cfg::kOffV + (j % NV) * Cfg::kSlotBytes;
                    for (int idx = threadIdx.x; idx < tail_rows * PANELS * 8; idx += 256) {
                        const int row = tail_row0 + idx / (PANELS * 8), rem = idx % (PANELS * 8);
                        *reinterpret_cast<uint4 *>(vt + (rem >> 3) * TK * 128 + row * 128 + (rem & 7) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
            }
            const int key0 = (kt0 + j) * TK + h * 64;
            if constexpr (kShared) {
                // every row sees every prefix key; keys past the prefix and rows past the
                // group's pairs see nothing
                if (key0 + 63 >= key_end || !row_ok) {
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (key0 + c >= key_end || !row_ok) sc[c] = -INFINITY;
                }
            } else {
                // bottom-right causal mask: key <= this row's position; a row past nq sees nothing
                if (key0 + 63 > P0 || !row_ok) {
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (key0 + c > qpos || !row_ok) sc[c] = -INFINITY;
                }
            }
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < 64; ++c) mx4[c & 3] = fmaxf(mx4[c & 3], sc[c]);
            float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
            // the other half's maximum of this row, and whether it is still ok; the exchange
            // buffer alternates with the tile, so one barrier a tile suffices
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
            float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                sc[c] = ex2_approx(fmaf(sc[c], p.scale_log2, neg_m));
                l4[c & 3] += sc[c];
            }
            l = l * alpha + ((l4[0] + l4[1]) + (l4[2] + l4[3]));
            uint32_t phi[32], plo[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) split_bf16x2(sc[2 * e], sc[2 * e + 1], phi[e], plo[e]);
            // a rescale of O waits for P_{j-1} V_{j-1} (and so every earlier P.V): O is then
            // current, and P_j V_j has not started, as it waits for this tile's P
            if (j > 0 && __any_sync(kFull, alpha != 1.f)) {
                const int qb = (j - 1) % Cfg::NSP;
                ok = __all_sync(kFull, wait_or_abort(bar(Cfg::kPFree + qb), ((j - 1) / Cfg::NSP) & 1, abort, p.err));
                if (!ok) continue;
                tc_fence_after_sync();
                {
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
            }
            // the weights over this thread's own scores (already in registers)
            tmem_st32(scol, phi);
            tmem_st32(scol + 32, plo);
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Cfg::kPFull + pb));
        }
        if (ok) ok = __all_sync(kFull, wait_or_abort(bar(Cfg::kDone), 0, abort, p.err));

        // ---- the row's sum over its two threads, through the exchange buffer the last tile
        // did not use; O / l and the log-sum-exp
        const int fb = ntiles & 1;
        *xs(fb, 0, h) = l;
        named_barrier(pair_bar, 64);
        const float lr = l + *xs(fb, 0, 1 - h);
        if (ok) {
            tc_fence_after_sync();
            const float inv_l = lr > 0.f ? 1.f / lr : 0.f;
            // O / l of the warp's 32 rows x D/2 columns, staged in the K/V rings (every MMA
            // and copy has completed, so they are free) so that each store writes whole row
            // segments; the pitch spreads the rows over the banks
            constexpr int HW = D / 2, PITCH = HW + 4;
            float *stage = reinterpret_cast<float *>(smem + Cfg::kOffK) + warp * 32 * PITCH;
            fence_proxy_async_smem();
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                uint32_t ov[32];
                tmem_ld32(lane_base + Cfg::kOCol + h * HW + cc * 32, ov);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4 *>(stage + lane * PITCH + cc * 32 + e) =
                        make_float4(__uint_as_float(ov[e]) * inv_l, __uint_as_float(ov[e + 1]) * inv_l,
                                    __uint_as_float(ov[e + 2]) * inv_l, __uint_as_float(ov[e + 3]) * inv_l);
            }
            __syncwarp();
            const int wrow0 = (warp & 3) << 5;
            const int wrows = min(32, nrows - wrow0);   // rows of the warp inside the tile
            for (int rr = 0; rr < wrows; ++rr) {
                int bq, hq;
                size_t member;
                row_seq_head(wrow0 + rr, bq, hq, member);
                // chunked prefill: the output row; shared prefix: this split's normalised partial
                float *dst = kShared ? p.ws_o + ((member * p.Hq + hq) * p.prefix_splits + ks) * D + h * HW
                                     : p.out + (static_cast<size_t>(bq) * p.Hq + hq) * D + h * HW;
                if constexpr (HW == 64)
                    *reinterpret_cast<float2 *>(dst + 2 * lane) =
                        *reinterpret_cast<const float2 *>(stage + rr * PITCH + 2 * lane);
                else
                    dst[lane] = stage[rr * PITCH + lane];
            }
            if (row_ok && h == 0) {
                int bq, hq;
                size_t member;
                row_seq_head(r, bq, hq, member);
                const float lse2 = m_ref == -INFINITY ? -INFINITY : m_ref + log2f(lr);
                if constexpr (kShared)
                    p.ws_lse[(member * p.Hq + hq) * p.prefix_splits + ks] = lse2;
                else if (p.lse != nullptr)
                    p.lse[static_cast<size_t>(bq) * p.Hq + hq] = lse2 * kDecLn2;
            }
        }
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
    kernel<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(tk, tv, kp);
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
        bool good = g0 >= 0 && g0 < n_members && __ldg(p.group_seqs + g0) == first &&
                    P == __ldg(p.kv_start + first) && P >= 0 && P % bs == 0 && P <= len - 1 && len <= p.MBS * bs;
        for (int j = lane; good && j < P / bs; j += 32)
            if (__ldg(p.block_table + static_cast<size_t>(b) * p.MBS + j) !=
                __ldg(p.block_table + static_cast<size_t>(first) * p.MBS + j))
                good = false;
        if (!__all_sync(kFull, good) && lane == 0) raise_error(p.err, PKV_DEVERR_PREFIX);
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
