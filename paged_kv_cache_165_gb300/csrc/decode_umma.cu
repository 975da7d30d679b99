// decode_umma.cu -- paged decode attention for large GQA groups (9..64 query heads per
// KV head; MQA is m = Hq) on the 5th-generation tensor cores (tcgen05).
//
// What is computed is the decode attention of decode.cu: for sequence b and query head
// i reading KV head j = floor(i/m), out = softmax_t(scale * q . K_t) V_t over the
// cached tokens gathered through block_table[b] (limoncc.com "大语言模型研究15——注意力
// 机制优化之KV缓存" §3.1, §3.3; plumephp.com "KV Cache 优化与注意力机制加速" §4.2-§4.3),
// with the online softmax of plumephp.com §2.2-§2.3 and log-sum-exp partials per chunk.
//
// With m heads sharing every K/V page the page math is a real contraction: S = Q K^T
// with M = 2m rows.  One CTA per (sequence, KV head, chunk of blocks) and SM, 11 warps:
//   warps 9 and 10 (TMA): warp 9 first the group's fp32 queries (one bulk copy), then the
//     K pages of each 64-key tile into a ring of shared stages; warp 10 the V pages into a
//     second ring (one {64, bs} box per page and 64-column panel, 128-byte swizzle, one
//     lane per page).  A K stage is free once its scores are computed, a V stage once its
//     P.V is, so K runs ahead of V by the two tiles in softmax.  A page past the chunk
//     is placed outside the cache, where TMA fills zeros.
//   warp 8 (one lane issues): S_j = Q K_j^T (M = 128, N = 64) into tensor memory, and
//     O += P_j V_j (M = 128, N = d) into a tensor-memory O.
//   warps 0-3 and 4-7: two softmax groups taking the tiles in turn (tile j goes to group
//     j % 2), each with its own S buffers, P buffer, O and online-softmax state, so one
//     group's exponentials overlap the other's hand-offs with the tensor core.  Thread r
//     of a group owns row r of the 128-row tile.  Row 2h holds the bf16 rounding of head
//     h's fp32 query ("hi"), row 2h+1 the bf16 rounding of the remainder ("lo"), so
//     s = S[2h] + S[2h+1] carries q to about 2^-16 relative.  The two rows sit in lanes
//     2h and 2h+1 of one warp: each lane takes half of the tile's 64 keys, receives the
//     partner row's values for its half by one shuffle per key, and runs the online
//     softmax for its half (the running max is shared by one more shuffle).  The weights
//     P go back to shared memory as hi (row 2h) and lo (row 2h+1) bf16 parts, so
//     O[2h] + O[2h+1] = sum_t P_t V_t to about 2^-16 relative as well.  O rows are
//     rescaled in tensor memory only when the running max grew by more than 2^8.
// At the end the two groups' (max, sum, O) merge by log-sum-exp inside the CTA; a chunk
// then writes a normalised partial and its base-2 log-sum-exp into the workspace, merged
// by the merge kernel of decode.cu.  Every wait is bounded and shares an abort flag: on a
// timeout the block drains the copies and MMAs it issued, frees tensor memory and returns
// with PKV_DEVERR_TIMEOUT.
#include <math.h>

#include "common.cuh"
#include "decode_kparams.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr unsigned kFullMask = 0xffffffffu;

template <int D, int BS, int NK, int NV>
struct UmmaDecodeCfg {
    static constexpr int kBM = 128, kBN = kUmmaDecodeKeys, kPPT = kBN / BS;   // pages per tile
    static constexpr int PANELS = D / 64;
    static constexpr int kQBytes = kBM * D * 2;     // Q hi/lo rows: D/64 panels of [128][128 B]
    static constexpr int kKVBytes = kBN * D * 2;    // one K or V tile: D/64 panels of [64][128 B]
    static constexpr int kPBytes = kBM * kBN * 2;   // P hi/lo rows [128][64] bf16: one panel
    static constexpr int kOffK = kQBytes;           // K ring, NK stages
    static constexpr int kOffV = kOffK + NK * kKVBytes;        // V ring, NV stages
    static constexpr int kOffP = kOffV + NV * kKVBytes;        // P of group g; first the raw fp32 q
    static constexpr int kOffBar = kOffP + 2 * kPBytes;
    // barriers: raw q; Q; K full / free per K stage; V full / free per V stage; per group:
    // S full x2, S free x2, P full, O done
    static constexpr int kQRaw = 0, kQ = 1, kKFull = 2, kKFree = 2 + NK, kVFull = 2 + 2 * NK,
                         kVFree = 2 + 2 * NK + NV, kGroup0 = 2 + 2 * NK + 2 * NV;
    static constexpr int kDrain = kGroup0 + 12;   // completes once every MMA issued is done
    static constexpr int kNumBars = kGroup0 + 13;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;     // TMEM slot, abort flag
    static constexpr int kOffXch = (kOffMisc + 16 + 15) / 16 * 16;   // [group][m, l, ok][128]
    static constexpr int kSmemBytes = 1024 + kOffXch + 2 * 3 * kBM * 4;
    static constexpr int kTmemCols = 512;           // per group: S 2 x 64 columns, O D columns
    static constexpr int kGroupCols = 256;
    static constexpr int kSCol = 0, kOCol = 2 * kBN;
    static constexpr int kStageRow = D + 4;         // fp32 row stride of the O staging area
    static constexpr int kThreads = 352;
    static constexpr int s_full(int g, int b) { return kGroup0 + g * 6 + b; }
    static constexpr int s_free(int g, int b) { return kGroup0 + g * 6 + 2 + b; }
    static constexpr int p_full(int g) { return kGroup0 + g * 6 + 4; }
    static constexpr int o_done(int g) { return kGroup0 + g * 6 + 5; }
    static_assert(D == 64 || D == 128, "head size");
    static_assert(BS == 16 || BS == 32, "block size");
    static_assert(kOCol + D <= kGroupCols, "tensor memory budget");
    static_assert(64 * D * 4 <= 2 * kPBytes, "raw queries fit the P buffers");
    static_assert(kBM * kStageRow * 4 <= NK * kKVBytes, "O staging fits the K ring");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

template <int D, int BS, int NK, int NV>
__global__ void __launch_bounds__(352, 1)
    decode_umma_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const DecodeKParams p) {
    using Cfg = UmmaDecodeCfg<D, BS, NK, NV>;
    constexpr int BM = Cfg::kBM, BN = Cfg::kBN, PPT = Cfg::kPPT, PANELS = Cfg::PANELS;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 4);
    float *xch = reinterpret_cast<float *>(smem + Cfg::kOffXch);
    auto bar = [&](int k) { return smem_addr(&bars[k]); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, kvh = blockIdx.y;
    const int b = blockIdx.z / p.qtiles, qt = blockIdx.z % p.qtiles;
    const bool report = threadIdx.x == 0 && split == 0 && kvh == 0 && qt == 0;
    // the sequence's query rows c0 .. c0+nq-1 (decode: row b) sit at positions L-nq ..
    // L-1; this block takes rows q0 .. q0+nqt-1 of them, slot = (row - q0) * m + head
    const int L = checked_len(p, b, BS, report);
    int c0 = b, nq = 1;
    bool rows_ok = true;
    if (p.cu_q != nullptr) {
        c0 = __ldg(p.cu_q + b);
        nq = __ldg(p.cu_q + b + 1) - c0;
        if (nq < 0 || nq > L) {
            if (report) raise_error(p.err, PKV_DEVERR_CU_SEQLENS);
            rows_ok = false;
        }
    }
    const int q0 = qt * p.q_per_tile;
    const int nqt = max(0, min(p.q_per_tile, nq - q0));
    const int slots = nqt * p.m;   // 1..64 query rows x heads
    const int P0 = L - nq + q0;    // position of the tile's first query
    // keys the whole sequence's rows see (chunk boundaries) and this tile's rows see
    const int lo_seq = p.window > 0 ? max(0, L - nq + 1 - p.window) : 0;
    const int cpfirst = lo_seq / BS, cnpages = L > 0 ? (L + BS - 1) / BS - cpfirst : 0;
    const int nc = (cnpages + p.chunk_pages - 1) / p.chunk_pages;
    const int lo_tile = p.window > 0 ? max(0, P0 + 1 - p.window) : 0;    // first query's window
    const int lo_last = p.window > 0 ? max(0, P0 + nqt - p.window) : 0;   // last query's window
    const int hi_tile = P0 + nqt;                                         // one past the last query
    const int cp0 = cpfirst + split * p.chunk_pages;                      // this chunk's pages
    const int cp1 = min(cpfirst + cnpages, cp0 + p.chunk_pages);
    const int apg0 = max(cp0, lo_tile / BS);                              // ... that the tile sees
    const int apg1 = min(cp1, (hi_tile + BS - 1) / BS);
    auto row_of = [&](int slot) { return static_cast<size_t>(c0 + q0 + slot / p.m) * p.Hq + kvh * p.m + slot % p.m; };
    if (nqt <= 0) return;
    if (!rows_ok || cp0 >= cp1) {
        if (split == 0) {   // an empty sequence or inconsistent rows: out = 0, lse = -inf
            for (int idx = threadIdx.x; idx < slots * D; idx += blockDim.x) p.out[row_of(idx / D) * D + idx % D] = 0.f;
            if (p.lse != nullptr)
                for (int sl = threadIdx.x; sl < slots; sl += blockDim.x) p.lse[row_of(sl)] = -INFINITY;
        }
        return;
    }
    if (apg0 >= apg1) {     // none of the tile's keys in this chunk: empty partials
        for (int idx = threadIdx.x; idx < slots * D; idx += blockDim.x)
            p.ws_o[(row_of(idx / D) * p.splits + split) * D + idx % D] = 0.f;
        for (int sl = threadIdx.x; sl < slots; sl += blockDim.x) p.ws_lse[row_of(sl) * p.splits + split] = -INFINITY;
        return;
    }
    const int len = L;
    const int pfirst = apg0, pages = apg1 - apg0;
    const int ntiles = (pages + PPT - 1) / PPT;
    const int tok0 = pfirst * BS;                        // first token of the pages read
    const int tok_lo = max(tok0, lo_tile);               // first key any row sees
    const int tok_end = min(hi_tile, apg1 * BS);         // one past the last key any row sees

    if (threadIdx.x == 0) {
        mbar_init(bar(Cfg::kQRaw), 1);
        mbar_init(bar(Cfg::kQ), 8);
        mbar_init(bar(Cfg::kDrain), 1);
        for (int st = 0; st < NK; ++st) {
            mbar_init(bar(Cfg::kKFull + st), 1);
            mbar_init(bar(Cfg::kKFree + st), 1);
        }
        for (int st = 0; st < NV; ++st) {
            mbar_init(bar(Cfg::kVFull + st), 1);
            mbar_init(bar(Cfg::kVFree + st), 1);
        }
        for (int g = 0; g < 2; ++g) {
            for (int sb = 0; sb < 2; ++sb) {
                mbar_init(bar(Cfg::s_full(g, sb)), 1);
                mbar_init(bar(Cfg::s_free(g, sb)), 4);
            }
            mbar_init(bar(Cfg::p_full(g)), 4);
            mbar_init(bar(Cfg::o_done(g)), 1);
        }
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
    const uint32_t sQ = smem_addr(smem);
    auto sK = [&](int st) { return smem_addr(smem + Cfg::kOffK + st * Cfg::kKVBytes); };
    auto sV = [&](int st) { return smem_addr(smem + Cfg::kOffV + st * Cfg::kKVBytes); };
    auto sP = [&](int g) { return smem_addr(smem + Cfg::kOffP + g * Cfg::kPBytes); };

    if (warp >= 9) {
        // ---- TMA loaders: warp 9 the raw queries and the K tiles, warp 10 the V tiles.
        // Tile t (pages pfirst + t*PPT ...) goes to stage t % N of its ring once the stage's
        // previous tile is consumed (K: by S_{t-NK}; V: by P_{t-NV} V).
        const bool is_k = warp == 9;
        const int N = is_k ? NK : NV;
        const int full0 = is_k ? Cfg::kKFull : Cfg::kVFull, free0 = is_k ? Cfg::kKFree : Cfg::kVFree;
        const CUtensorMap *map = is_k ? &tm_k : &tm_v;
        if (is_k && lane == 0) {
            // the m heads of one query row are contiguous: one copy per row of the tile
            const uint32_t row_bytes = static_cast<uint32_t>(p.m) * D * 4;
            mbar_arrive_expect_tx(bar(Cfg::kQRaw), row_bytes * nqt);
            for (int qi = 0; qi < nqt; ++qi)
                bulk_load(sP(0) + qi * row_bytes, p.q + row_of(qi * p.m) * D, row_bytes, bar(Cfg::kQRaw));
        }
        const int32_t *tbl = p.block_table + static_cast<size_t>(b) * p.MBS + pfirst;
        int tcur = lane < pages ? __ldg(tbl + lane) : -1;
        int tbase = 0;
        const int oob_row = p.NB * p.Hkv * BS;
        int t = 0;
        for (; t < ntiles; ++t) {
            bool fr = true;
            if (lane == 0 && t >= N)
                fr = wait_or_abort(bar(free0 + t % N), ((t - N) / N) & 1, abort, p.err);
            if (!__shfl_sync(kFullMask, fr ? 1 : 0, 0)) break;
            const int st = t % N;
            if (t * PPT >= tbase + 32) {   // a tile never straddles 32 pages (32 % PPT == 0)
                tbase += 32;
                tcur = tbase + lane < pages ? __ldg(tbl + tbase + lane) : -1;
            }
            // lane i < PPT issues the copies of the tile's page i
            const int k = t * PPT + lane;
            const int phys = __shfl_sync(kFullMask, tcur, k & 31);
            if (lane == 0) mbar_arrive_expect_tx(bar(full0 + st), Cfg::kKVBytes);
            __syncwarp();
            if (lane < PPT) {
                int row = oob_row;
                if (k < pages) {
                    if (phys < 0 || phys >= p.NB) {
                        if (is_k) raise_error(p.err, PKV_DEVERR_BLOCK);
                    } else {
                        row = (phys * p.Hkv + kvh) * BS;
                    }
                }
                const uint32_t dst = (is_k ? sK(st) : sV(st)) + lane * BS * 128;
#pragma unroll
                for (int pn = 0; pn < PANELS; ++pn) tma_load_2d(dst + pn * BN * 128, map, pn * 64, row, bar(full0 + st));
            }
        }
        // before teardown every copy issued must have landed (bounded)
        if (lane == 0) {
            if (is_k) mbar_wait_bounded(bar(Cfg::kQRaw), 0);
            for (int u = max(0, t - N); u < t; ++u) mbar_wait_bounded(bar(full0 + u % N), (u / N) & 1);
        }
    } else if (warp == 8) {
        // ---- MMA issue.  Tile j belongs to group j % 2 (its (j/2)-th tile); S_{j+2} goes
        // out before P_j V_j, so the next tile of a group is scored while it is in softmax.
        if (lane == 0) {
            const uint32_t idesc_s = umma_idesc_bf16(BM, BN, 0);
            const uint32_t idesc_o = umma_idesc_bf16(BM, D, 1);
            auto issue_s = [&](int j) {
                const int st = j % NK, g = j & 1, sb = (j >> 1) & 1;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t ad = umma_desc_sw128(sQ + (kk / 4) * BM * 128 + (kk % 4) * 32, 16, 1024);
                    const uint64_t bd = umma_desc_sw128(sK(st) + (kk / 4) * BN * 128 + (kk % 4) * 32, 16, 1024);
                    umma_bf16(tmem + g * Cfg::kGroupCols + Cfg::kSCol + sb * BN, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
                }
                umma_commit(bar(Cfg::s_full(g, sb)));
                umma_commit(bar(Cfg::kKFree + st));
            };
            auto issue_pv = [&](int j) {
                const int st = j % NV, g = j & 1;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t ad = umma_desc_sw128(sP(g) + kk * 32, 16, 1024);
                    const uint64_t bd = umma_desc_sw128(sV(st) + kk * 16 * 128, BN * 128, 1024);
                    umma_bf16(tmem + g * Cfg::kGroupCols + Cfg::kOCol, ad, bd, idesc_o,
                              (j > 1 || kk > 0) ? 1u : 0u);
                }
                umma_commit(bar(Cfg::o_done(g)));
                umma_commit(bar(Cfg::kVFree + st));
            };
            // Tile j belongs to group j % 2 (its (j/2)-th tile).  S_{j+2} goes out before
            // P_j V_j, so a group's next tile is scored while the group is in softmax.
            int j = 0;
            bool issued = false, alive = wait_or_abort(bar(Cfg::kQ), 0, abort, p.err);
            for (int t = 0; t < 2 && t < ntiles && alive; ++t) {
                alive = wait_or_abort(bar(Cfg::kKFull + t), 0, abort, p.err);
                if (!alive) break;
                tc_fence_after_sync();
                issue_s(t);
                issued = true;
            }
            for (; j < ntiles && alive; ++j) {
                const int g = j & 1, t = j + 2;
                if (t < ntiles) {
                    alive = wait_or_abort(bar(Cfg::kKFull + t % NK), (t / NK) & 1, abort, p.err);
                    const int tt = t >> 1;   // the group's tile index of t
                    if (alive && tt >= 2)
                        alive = wait_or_abort(bar(Cfg::s_free(g, tt & 1)), ((tt >> 1) - 1) & 1, abort, p.err);
                    if (!alive) break;
                    tc_fence_after_sync();
                    issue_s(t);
                }
                alive = wait_or_abort(bar(Cfg::p_full(g)), (j >> 1) & 1, abort, p.err) &&
                        wait_or_abort(bar(Cfg::kVFull + j % NV), (j / NV) & 1, abort, p.err);
                if (!alive) break;
                tc_fence_after_sync();
                issue_pv(j);
            }
            if (*abort && issued) {
                // let the MMAs already issued finish (bounded) before teardown
                umma_commit(bar(Cfg::kDrain));
                mbar_wait_bounded(bar(Cfg::kDrain), 0);
            }
        }
    } else {
        // ---- softmax group g: thread r owns row r of the tile (TMEM lane r)
        const int g = warp >> 2;
        const int r = threadIdx.x & 127;
        const int slot = r >> 1, part = r & 1;
        const bool slot_ok = slot < slots;
        // this row's query position and visible keys [lo_r, hi_r)
        const int pos_r = P0 + (slot_ok ? slot / p.m : 0);
        const int lo_r = p.window > 0 ? max(0, pos_r + 1 - p.window) : 0;
        const int hi_r = min(pos_r + 1, apg1 * BS);
        const uint32_t lane_base = tmem + g * Cfg::kGroupCols + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const int njj = (ntiles - g + 1) / 2;   // tiles of this group
        bool ok = __all_sync(kFullMask, wait_or_abort(bar(Cfg::kQRaw), 0, abort, p.err));

        // Q rows from the raw queries: group g writes panels g, g+2, ...; row 2s = rn(q_s),
        // row 2s+1 = rn(q_s - rn(q_s)) for slot s, 128-byte swizzle.  Reads are rotated by
        // s so that the rows read by a quarter warp fall in distinct banks.
        if (ok) {
            const float *qraw = reinterpret_cast<const float *>(smem + Cfg::kOffP) + (slot_ok ? slot : 0) * D;
            for (int pn = g; pn < PANELS; pn += 2) {
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const int cc = (c8 + slot) & 7;
                    float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
                    if (slot_ok) {
                        x0 = *reinterpret_cast<const float4 *>(qraw + pn * 64 + cc * 8);
                        x1 = *reinterpret_cast<const float4 *>(qraw + pn * 64 + cc * 8 + 4);
                    }
                    uint32_t w[4], hi, lo;
                    split_bf16x2(x0.x, x0.y, hi, lo);
                    w[0] = part ? lo : hi;
                    split_bf16x2(x0.z, x0.w, hi, lo);
                    w[1] = part ? lo : hi;
                    split_bf16x2(x1.x, x1.y, hi, lo);
                    w[2] = part ? lo : hi;
                    split_bf16x2(x1.z, x1.w, hi, lo);
                    w[3] = part ? lo : hi;
                    *reinterpret_cast<uint4 *>(smem + pn * BM * 128 + r * 128 + ((cc ^ (r & 7)) << 4)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(Cfg::kQ));

        uint8_t *pbuf = smem + Cfg::kOffP + g * Cfg::kPBytes;
        const int r_hi = r & ~1, r_lo = r | 1;
        // The chunk's last page may end inside the sequence's last block: its V rows past
        // the end hold whatever the slots hold (NaN, Inf) and must be zero for P.V.
        const int tail_valid = tok_end - (apg1 - 1) * BS;   // 1..BS tokens
        const int tail_tile = (pages - 1) / PPT;
        const int tail_row0 = ((pages - 1) % PPT) * BS + tail_valid;
        const int tail_rows = BS - tail_valid;
        float m_ref = -INFINITY, l = 0.f;
        for (int jj = 0; jj < njj && ok; ++jj) {
            const int j = 2 * jj + g, sb = jj & 1;
            ok = __all_sync(kFullMask, wait_or_abort(bar(Cfg::s_full(g, sb)), (jj >> 1) & 1, abort, p.err));
            if (!ok) break;
            tc_fence_after_sync();
            uint32_t sr[BN];
            tmem_ld32(lane_base + Cfg::kSCol + sb * BN, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
            tmem_ld32(lane_base + Cfg::kSCol + sb * BN + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
            tmem_ld_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Cfg::s_free(g, sb)));
            if (j == tail_tile && tail_rows > 0) {
                // once the V copies of this tile have landed
                ok = __all_sync(kFullMask, wait_or_abort(bar(Cfg::kVFull + j % NV), (j / NV) & 1, abort, p.err));
                if (!ok) break;
                uint8_t *vt = smem + Cfg::kOffV + (j % NV) * Cfg::kKVBytes;
                for (int idx = r; idx < tail_rows * PANELS * 8; idx += BM) {
                    const int row = tail_row0 + idx / (PANELS * 8), rem = idx % (PANELS * 8);
                    *reinterpret_cast<uint4 *>(vt + (rem >> 3) * BN * 128 + row * 128 + (rem & 7) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
            }

            // keys part*32 .. part*32+31 of the tile: own row plus the partner row
            float sc[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float mine = __uint_as_float(part ? sr[32 + c] : sr[c]);
                const float send = __uint_as_float(part ? sr[c] : sr[32 + c]);
                sc[c] = mine + __shfl_xor_sync(kFullMask, send, 1);
            }
            const int key0 = tok0 + j * BN + part * 32;
            if (tok0 + j * BN < lo_r || tok0 + (j + 1) * BN > hi_r) {
                // keys outside this row's [lo_r, hi_r): before its window, after its own
                // position (causal), or past the end of the chunk
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if (key0 + c < lo_r || key0 + c >= hi_r) sc[c] = -INFINITY;
            }
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < 32; ++c) mx4[c & 3] = fmaxf(mx4[c & 3], sc[c]);
            float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
            mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 1)) * p.scale_log2;
            // a row that has seen no key yet keeps m = -inf and weight 0
            const float m_new = mx > m_ref + 8.f ? mx : m_ref;
            const float alpha = m_new == m_ref ? 1.f : ex2_approx(m_ref - m_new);
            m_ref = m_new;
            const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
            float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                sc[c] = ex2_approx(fmaf(sc[c], p.scale_log2, neg_m));
                l4[c & 3] += sc[c];
            }
            l = l * alpha + ((l4[0] + l4[1]) + (l4[2] + l4[3]));
            uint32_t phi[16], plo[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) split_bf16x2(sc[2 * e], sc[2 * e + 1], phi[e], plo[e]);
            // P.V of the group's previous tile must be done: P is free and O is current
            if (jj > 0) {
                ok = __all_sync(kFullMask, wait_or_abort(bar(Cfg::o_done(g)), (jj - 1) & 1, abort, p.err));
                if (!ok) break;
                tc_fence_after_sync();
                if (__any_sync(kFullMask, alpha != 1.f)) {
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
            // P_hi into row 2h, P_lo into row 2h+1, keys part*32 .. part*32+31
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const int c16 = part * 4 + q4;
                *reinterpret_cast<uint4 *>(pbuf + r_hi * 128 + ((c16 ^ (r_hi & 7)) << 4)) =
                    make_uint4(phi[4 * q4], phi[4 * q4 + 1], phi[4 * q4 + 2], phi[4 * q4 + 3]);
                *reinterpret_cast<uint4 *>(pbuf + r_lo * 128 + ((c16 ^ (r_lo & 7)) << 4)) =
                    make_uint4(plo[4 * q4], plo[4 * q4 + 1], plo[4 * q4 + 2], plo[4 * q4 + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Cfg::p_full(g)));
        }
        if (ok && njj > 0)
            ok = __all_sync(kFullMask, wait_or_abort(bar(Cfg::o_done(g)), (njj - 1) & 1, abort, p.err));

        // ---- merge the two groups: rows r of both groups hold the same query row
        const float l_pair = l + __shfl_xor_sync(kFullMask, l, 1);   // the head's sum in this group
        xch[(g * 3 + 0) * BM + r] = m_ref;
        xch[(g * 3 + 1) * BM + r] = l_pair;
        xch[(g * 3 + 2) * BM + r] = ok ? 1.f : 0.f;
        named_barrier(1, 256);
        const int o = 1 - g;
        const bool good = ok && xch[(o * 3 + 2) * BM + r] != 0.f;   // warp-uniform
        const float m_o = xch[(o * 3 + 0) * BM + r], l_o = xch[(o * 3 + 1) * BM + r];
        // M = -inf: the row sees no key of this chunk (an empty partial)
        const float M = fmaxf(m_ref, m_o);
        const bool empty = M == -INFINITY;
        const float f = empty ? 0.f : ex2_approx(m_ref - M), f_o = empty ? 0.f : ex2_approx(m_o - M);
        const float L = f * l_pair + f_o * l_o;
        const float scale = empty ? 0.f : f / L;
        float *stage = reinterpret_cast<float *>(smem + Cfg::kOffK) + r * Cfg::kStageRow;
        const int njj1 = ntiles / 2;
        if (g == 1 && good && njj1 > 0) {
            // every MMA is done (both groups saw their last O), so the K ring is free
            tc_fence_after_sync();
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t ov[32];
                tmem_ld32(lane_base + Cfg::kOCol + cc * 32, ov);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4 *>(stage + cc * 32 + e) =
                        make_float4(__uint_as_float(ov[e]) * scale, __uint_as_float(ov[e + 1]) * scale,
                                    __uint_as_float(ov[e + 2]) * scale, __uint_as_float(ov[e + 3]) * scale);
            }
        }
        named_barrier(1, 256);
        if (g == 0 && good) {
            tc_fence_after_sync();
            const size_t bi = row_of(slot_ok ? slot : 0);
            float *dst = nc == 1 ? p.out + bi * D : p.ws_o + (bi * p.splits + split) * D;
            // O[2s] + O[2s+1] over both groups; lane 2s writes the first half of the
            // columns, 2s+1 the second
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t ov[32];
                tmem_ld32(lane_base + Cfg::kOCol + cc * 32, ov);
                tmem_ld_wait();
                float sum[32];
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    float4 s1 = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (njj1 > 0) s1 = *reinterpret_cast<const float4 *>(stage + cc * 32 + e);
                    sum[e] = __uint_as_float(ov[e]) * scale + s1.x;
                    sum[e + 1] = __uint_as_float(ov[e + 1]) * scale + s1.y;
                    sum[e + 2] = __uint_as_float(ov[e + 2]) * scale + s1.z;
                    sum[e + 3] = __uint_as_float(ov[e + 3]) * scale + s1.w;
                }
#pragma unroll
                for (int e = 0; e < 32; ++e) sum[e] += __shfl_xor_sync(kFullMask, sum[e], 1);
                if (slot_ok && (cc < D / 64) == (part == 0)) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(dst + cc * 32 + e) =
                            make_float4(sum[e], sum[e + 1], sum[e + 2], sum[e + 3]);
                }
            }
            if (slot_ok && part == 0) {
                const float lse2 = empty ? -INFINITY : M + log2f(L);
                if (nc == 1) {
                    if (p.lse != nullptr) p.lse[bi] = lse2 * kDecLn2;
                } else {
                    p.ws_lse[bi * p.splits + split] = lse2;
                }
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, Cfg::kTmemCols);
}

template <int D, int BS, int NK, int NV>
cudaError_t launch_umma(const DecodeKParams &kp, const CUtensorMap &tk, const CUtensorMap &tv, dim3 grid,
                        cudaStream_t stream) {
    using Cfg = UmmaDecodeCfg<D, BS, NK, NV>;
    auto kernel = decode_umma_kernel<D, BS, NK, NV>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    kernel<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(tk, tv, kp);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_umma(const DecodeKParams &kp, const CUtensorMap &tk, const CUtensorMap &tv,
                               int d, int bs, dim3 grid, cudaStream_t stream) {
    if (d == 128) return bs == 16 ? launch_umma<128, 16, 5, 4>(kp, tk, tv, grid, stream)
                                  : launch_umma<128, 32, 5, 4>(kp, tk, tv, grid, stream);
    if (d == 64) return bs == 16 ? launch_umma<64, 16, 8, 8>(kp, tk, tv, grid, stream)
                                 : launch_umma<64, 32, 8, 8>(kp, tk, tv, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
