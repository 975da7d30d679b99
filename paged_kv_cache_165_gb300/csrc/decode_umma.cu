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
// with M = 2m rows.  One CTA per (sequence, KV head, chunk of blocks) and SM, 12 warps,
// key tiles of 128 tokens:
//   warps 9 and 10 (TMA): the K and the V pages of each tile into two rings of tile
//     slots (one {64, bs} box per page and 64-column panel, 128-byte swizzle, one box per
//     lane: copies issued by different threads proceed in parallel, one thread's copies
//     largely one after another).  A K slot is free once its scores are computed, a V
//     slot once its P.V is.  A page past the chunk is placed outside the cache, where TMA
//     fills zeros.
//   warps 11 and 8 (one lane each issues): S_t = Q K_t^T (M = 128, N = 128) into one of two
//     tensor-memory S buffers, and O += P_j V_j (N = d) into a tensor-memory O.  Q and P
//     are the A operands and live in tensor memory; K and V are read from shared memory.
//     S_t goes into the buffer S_{t-2} leaves once P_{t-2} is written (S_{t-2} has been
//     read), so the tensor core computes the next scores while the softmax runs; with one
//     issuer per kind, the waits of one overlap the MMAs of the other.
//   warps 0-7 (softmax): row r of the 128-row tile is tensor-memory lane r.  Query slot
//     s = 8g + i (g = 0 .. 7, i = 0 .. 7) has two rows in lane group g (lanes 16g .. 16g +
//     15): row 16g + i holds the bf16 rounding of the query ("hi"), row 16g + 8 + i the bf16
//     rounding of the remainder ("lo"), so s = S_hi + S_lo carries q to about 2^-16
//     relative.  Warp w reads lane group 2 (w % 4) + w / 4 with the 16-lane shapes: thread
//     t holds both rows of slot 8g + t / 4 and, of each key tile, the key pairs 4k + t % 4
//     (keys 8k + 2 (t % 4), + 1), so it adds the two parts itself; the four threads of a
//     slot share its maximum and sum by two shuffles, and the warps run independently.  The
//     weights go back to tensor memory as hi (the hi row) and lo (the lo row) bf16 parts,
//     so O_hi + O_lo = sum_t P_t V_t to about 2^-16 relative as well.  O rows are rescaled
//     in tensor memory only when the running maximum grew by more than 2^8.
// A chunk writes a normalised partial and its base-2 log-sum-exp into the workspace,
// merged by the merge kernel of decode.cu (or, for a single chunk, the output).  Every wait
// is bounded and shares an abort flag: on a timeout the block drains the copies and MMAs
// it issued, frees tensor memory and returns with PKV_DEVERR_TIMEOUT.
#include <math.h>

#include "common.cuh"
#include "decode_kparams.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr unsigned kFullMask = 0xffffffffu;

template <int D, int BS, int NKT, int NVT>
struct UmmaDecodeCfg {
    static constexpr int kBM = 128, kTK = kUmmaDecodeKeys, kPPT = kTK / BS;   // pages per tile
    static constexpr int PANELS = D / 64;
    static constexpr int kSlotBytes = kTK * D * 2;   // one K or V tile: D/64 panels of [128][128 B]
    static constexpr int kOffK = 0;                  // K ring, NKT tile slots
    static constexpr int kOffV = kOffK + NKT * kSlotBytes;    // V ring, NVT tile slots
    static constexpr int kOffBar = kOffV + NVT * kSlotBytes;
    // barriers: Q built; K full / free per slot; V full / free per slot; S full x2; P full;
    // O done (after each P.V); all MMAs done; drain x2 (one per MMA-issuing thread)
    static constexpr int kQ = 0, kKFull = 1, kKFree = 1 + NKT, kVFull = 1 + 2 * NKT, kVFree = 1 + 2 * NKT + NVT,
                         kSFull = 1 + 2 * NKT + 2 * NVT, kPFull = kSFull + 2, kODone = kPFull + 1,
                         kDone = kODone + 1, kDrain = kDone + 1, kNumBars = kDrain + 2;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;          // TMEM slot, abort flag
    static constexpr int kSmemBytes = 1024 + kOffMisc + 16;
    // tensor memory: two S buffers, O, P, Q
    static constexpr int kTmemCols = 512;
    static constexpr int kSCol = 0, kOCol = 2 * kTK, kPCol = kOCol + D, kQCol = kPCol + kTK / 2;
    static constexpr int kThreads = 384;
    static_assert(D == 64 || D == 128, "head size");
    static_assert(BS == 16 || BS == 32, "block size");
    static_assert(kQCol + D / 2 <= kTmemCols, "tensor memory budget");
    static_assert(kPPT * PANELS <= 32 && 32 % kPPT == 0, "one box per loader lane; tiles within 32 pages");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

template <int D, int BS, int NKT, int NVT>
__global__ void __launch_bounds__(384, 1)
    decode_umma_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const DecodeKParams p) {
    using Cfg = UmmaDecodeCfg<D, BS, NKT, NVT>;
    constexpr int BM = Cfg::kBM, TK = Cfg::kTK, PPT = Cfg::kPPT, PANELS = Cfg::PANELS;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 4);
    auto bar = [&](int k) { return smem_addr(&bars[k]); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, kvh = blockIdx.y;
    const int qt = blockIdx.z % p.qtiles;
    int b = blockIdx.z / p.qtiles;
    // Decode in launch order (one query, no window, no shared prefix): the chunk's pages start
    // at split * chunk_pages whatever the sequence's length, so the loader warps load their
    // first block-table entries now, while the block sets up
    const bool early_table = !p.longest_first && p.cu_q == nullptr && p.window <= 0 && p.kv_start == nullptr &&
                             (warp == 9 || warp == 10);
    const int early_page0 = split * p.chunk_pages;
    int early_tcur = -1;
    if (early_table && early_page0 + lane < p.MBS)
        early_tcur = __ldg(p.block_table + static_cast<size_t>(b) * p.MBS + early_page0 + lane);
    if (p.longest_first) {
        // grid z ranks the sequences by length, longest first (ties: lower index first), so
        // that with lengths that differ the long blocks start first and the short ones fill
        // the end of the launch; the K ring is free scratch until the first copies
        int *len_s = reinterpret_cast<int *>(smem + Cfg::kOffK);
        for (int x = threadIdx.x; x < p.B; x += blockDim.x) len_s[x] = checked_len(p, x, BS, false);
        __syncthreads();
        for (int x = threadIdx.x; x < p.B; x += blockDim.x) {
            const int lx = len_s[x];
            int rank = 0;
            for (int y = 0; y < p.B; ++y) {
                const int ly = len_s[y];
                rank += (ly > lx || (ly == lx && y < x)) ? 1 : 0;
            }
            if (rank == b) len_s[p.B] = x;   // ranks are a permutation: exactly one x
        }
        __syncthreads();
        b = len_s[p.B];
        fence_proxy_async_smem();   // the copies that will land here come after these reads
        __syncthreads();
    }
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
    // a shared prefix attended elsewhere (decode only): keys from kv_start[b] on, the last kept
    const int kv0 = p.kv_start != nullptr && p.cu_q == nullptr && L > 0 ? min(__ldg(p.kv_start + b), L - 1) : 0;
    const int lo_seq = max(kv0, p.window > 0 ? max(0, L - nq + 1 - p.window) : 0);
    const int cpfirst = lo_seq / BS, cnpages = L > 0 ? (L + BS - 1) / BS - cpfirst : 0;
    const int nc = (cnpages + p.chunk_pages - 1) / p.chunk_pages;
    const int lo_tile = max(kv0, p.window > 0 ? max(0, P0 + 1 - p.window) : 0);   // first query's window
    const int hi_tile = P0 + nqt;                                         // one past the last query
    const int cp0 = cpfirst + split * p.chunk_pages;                      // this chunk's pages
    const int cp1 = min(cpfirst + cnpages, cp0 + p.chunk_pages);
    const int apg0 = max(cp0, lo_tile / BS);                              // ... that the tile sees
    const int apg1 = min(cp1, (hi_tile + BS - 1) / BS);
    auto row_of = [&](int slot) { return static_cast<size_t>(c0 + q0 + slot / p.m) * p.Hq + kvh * p.m + slot % p.m; };
    if (nqt <= 0) return;
    if (!rows_ok || cp0 >= cp1) {
        // a new token for a sequence that holds none has no position: flagged, not written
        if (p.new_slots != nullptr && split == 0 && threadIdx.x == 0 && L == 0 && __ldg(p.new_slots + b) >= 0)
            raise_error(p.err, PKV_DEVERR_SLOT);
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
    const int pfirst = apg0, pages = apg1 - apg0;
    const int ntiles = (pages + PPT - 1) / PPT;
    const int tok0 = pfirst * BS;                        // first token of the pages read
    const int tok_end = min(hi_tile, apg1 * BS);         // one past the last key any row sees

    // The step's new token (pkv_decode_step, one query per sequence): the block that reads
    // the sequence's last page writes it there before any copy (the barrier below orders
    // the writes before the loaders' copies)
    const bool writes_token = p.new_slots != nullptr && cp1 == cpfirst + cnpages;
    if (writes_token && warp == 1) {
        write_new_token<D, BS>(p, b, kvh, L, lane);
        fence_proxy_async_global();
    }
    if (threadIdx.x == 0) {
        mbar_init(bar(Cfg::kQ), 8);
        for (int s = 0; s < NKT; ++s) {
            mbar_init(bar(Cfg::kKFull + s), 1);
            mbar_init(bar(Cfg::kKFree + s), 1);
        }
        for (int s = 0; s < NVT; ++s) {
            mbar_init(bar(Cfg::kVFull + s), 1);
            mbar_init(bar(Cfg::kVFree + s), 1);
        }
        mbar_init(bar(Cfg::kSFull), 1);
        mbar_init(bar(Cfg::kSFull + 1), 1);
        mbar_init(bar(Cfg::kPFull), 8);
        mbar_init(bar(Cfg::kODone), 1);
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
    pdl_launch_dependents();   // the merge kernel may be scheduled; it waits for this grid
    const uint32_t tmem = *tslot;
    auto sK = [&](int s) { return smem_addr(smem + Cfg::kOffK + s * Cfg::kSlotBytes); };
    auto sV = [&](int s) { return smem_addr(smem + Cfg::kOffV + s * Cfg::kSlotBytes); };

    if (warp == 9 || warp == 10) {
        if (writes_token) fence_proxy_async_global();
        // ---- TMA loaders: warp 9 the K tiles, warp 10 the V tiles.  Tile t goes to slot
        // t % N of its ring once the slot's previous tile is consumed (K: by S_{t-N}; V: by
        // P_{t-N} V).  Lane i < PPT * PANELS copies panel i % PANELS of page i / PANELS.
        const bool is_k = warp == 9;
        const int N = is_k ? NKT : NVT;
        const int full0 = is_k ? Cfg::kKFull : Cfg::kVFull, free0 = is_k ? Cfg::kKFree : Cfg::kVFree;
        const CUtensorMap *map = is_k ? &tm_k : &tm_v;
        const int32_t *tbl = p.block_table + static_cast<size_t>(b) * p.MBS + pfirst;
        int tcur = early_table && pfirst == early_page0 ? (lane < pages ? early_tcur : -1)
                                                        : (lane < pages ? __ldg(tbl + lane) : -1);
        int tbase = 0;
        const int oob_row = p.NB * p.Hkv * BS;
        const int pg = lane / PANELS, pn = lane % PANELS;
        int t = 0;
        for (; t < ntiles; ++t) {
            bool fr = true;
            if (lane == 0 && t >= N)
                fr = wait_or_abort(bar(free0 + t % N), ((t - N) / N) & 1, abort, p.err);
            if (!__shfl_sync(kFullMask, fr ? 1 : 0, 0)) break;
            const int s = t % N;
            if (t * PPT >= tbase + 32) {   // a tile never straddles 32 pages (32 % PPT == 0)
                tbase += 32;
                tcur = tbase + lane < pages ? __ldg(tbl + tbase + lane) : -1;
            }
            const int k = t * PPT + pg;
            const int phys = __shfl_sync(kFullMask, tcur, k & 31);
            if (lane == 0) mbar_arrive_expect_tx(bar(full0 + s), Cfg::kSlotBytes);
            __syncwarp();
            if (lane < PPT * PANELS) {
                int row = oob_row;
                if (k < pages) {
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
        // ---- MMA issue, one lane of each of two warps: warp 11 the scores S_t (once K_t has
        // landed and, for t >= 2, P_{t-2} is written, i.e. S_{t-2} has been read from the
        // buffer S_t goes to), warp 8 the products P_j V_j.  Each waits only for its own
        // inputs, so one issuer's waits overlap the other's MMAs.  tcgen05.commit covers
        // the committing thread's MMAs: warp 11 signals S full and K free, warp 8 O done,
        // V free and, after the last P.V (which follows every S), all MMAs done.
        if (lane == 0) {
            const bool is_s = warp == 11;
            bool issued = false, alive = true;
            if (is_s) {
                const uint32_t idesc_s = umma_idesc_bf16(BM, TK, 0);
                alive = wait_or_abort(bar(Cfg::kQ), 0, abort, p.err);
                for (int t = 0; t < ntiles && alive; ++t) {
                    if (t >= 2) alive = wait_or_abort(bar(Cfg::kPFull), (t - 2) & 1, abort, p.err);
                    alive = alive && wait_or_abort(bar(Cfg::kKFull + t % NKT), (t / NKT) & 1, abort, p.err);
                    if (!alive) break;
                    tc_fence_after_sync();
                    const int s = t % NKT;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t bd = umma_desc_sw128(sK(s) + (kk / 4) * TK * 128 + (kk % 4) * 32, 16, 1024);
                        umma_bf16_ts(tmem + Cfg::kSCol + (t & 1) * TK, tmem + Cfg::kQCol + kk * 8, bd, idesc_s,
                                     kk > 0 ? 1u : 0u);
                    }
                    umma_commit(bar(Cfg::kSFull + (t & 1)));
                    umma_commit(bar(Cfg::kKFree + s));
                    issued = true;
                }
            } else {
                const uint32_t idesc_o = umma_idesc_bf16(BM, D, 1);
                for (int j = 0; j < ntiles && alive; ++j) {
                    alive = wait_or_abort(bar(Cfg::kPFull), j & 1, abort, p.err) &&
                            wait_or_abort(bar(Cfg::kVFull + j % NVT), (j / NVT) & 1, abort, p.err);
                    if (!alive) break;
                    tc_fence_after_sync();
                    const int s = j % NVT;
#pragma unroll
                    for (int kk = 0; kk < TK / 16; ++kk) {
                        const uint64_t bd = umma_desc_sw128(sV(s) + kk * 16 * 128, TK * 128, 1024);
                        umma_bf16_ts(tmem + Cfg::kOCol, tmem + Cfg::kPCol + kk * 8, bd, idesc_o,
                                     (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(bar(Cfg::kODone));
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
        // ---- softmax.  First the queries: thread (w, lane) writes tensor-memory lane r =
        // 32 (w % 4) + lane (the hi or lo row of one query slot), columns D/4 h .. D/4 h +
        // D/4 - 1 (two values a column) of it for h = w / 4
        {
            const int h = warp >> 2;
            const int r = ((warp & 3) << 5) | lane;
            const int qslot = 8 * (r >> 4) + (r & 7), qpart = (r >> 3) & 1;
            const bool qok = qslot < slots;
            const uint32_t qbase = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
            const float *qrow = p.q + row_of(qok ? qslot : 0) * D + h * (D / 2);
            uint32_t w[D / 4];
#pragma unroll
            for (int e = 0; e < D / 8; ++e) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (qok) x = __ldg(reinterpret_cast<const float4 *>(qrow + 4 * e));
                uint32_t hi, lo;
                split_bf16x2(x.x, x.y, hi, lo);
                w[2 * e] = qpart ? lo : hi;
                split_bf16x2(x.z, x.w, hi, lo);
                w[2 * e + 1] = qpart ? lo : hi;
            }
            if constexpr (D == 128) tmem_st32(qbase + Cfg::kQCol + h * (D / 4), w);
            else tmem_st16(qbase + Cfg::kQCol + h * (D / 4), w);
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Cfg::kQ));
        }

        // Then per key tile: thread t of warp w owns slot `slot` = 8 g + t / 4 of lane group
        // g = 2 (w % 4) + w / 4 (its hi row is lane 16 g + t / 4 of the group's base, its lo
        // row 8 lanes further) and the key pairs 4k + c4 (c4 = t % 4) of the tile
        const int c4 = lane & 3;
        const int grp = 2 * (warp & 3) + (warp >> 2);
        const int slot = 8 * grp + (lane >> 2);
        const bool slot_ok = slot < slots;
        // this slot's query position and visible keys [lo_r, hi_r)
        const int pos_r = P0 + (slot_ok ? slot / p.m : 0);
        const int lo_r = max(kv0, p.window > 0 ? max(0, pos_r + 1 - p.window) : 0);
        const int hi_r = min(pos_r + 1, apg1 * BS);
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(16 * grp) << 16);

        // The chunk's last page may end inside the sequence's last block: its V rows past
        // the end hold whatever the slots hold (NaN, Inf) and must be zero for P.V.
        const int tail_valid = tok_end - (apg1 - 1) * BS;   // 1..BS tokens
        const int tail_tile = (pages - 1) / PPT;
        const int tail_row0 = ((pages - 1) % PPT) * BS + tail_valid;
        const int tail_rows = BS - tail_valid;
        float m_ref = -INFINITY, l = 0.f;
        // ok is warp-uniform; a failed wait skips the remaining work of this warp
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int sb = j & 1;
            if (ok) ok = __all_sync(kFullMask, wait_or_abort(bar(Cfg::kSFull + sb), (j >> 1) & 1, abort, p.err));
            if (ok && j == tail_tile && tail_rows > 0) {
                // once the V copies of this tile have landed (each softmax warp zeroes its
                // share of the rows, so each waits)
                ok = __all_sync(kFullMask, wait_or_abort(bar(Cfg::kVFull + j % NVT), (j / NVT) & 1, abort, p.err));
                if (ok) {
                    uint8_t *vt = smem + Cfg::kOffV + (j % NVT) * Cfg::kSlotBytes;
                    for (int idx = threadIdx.x; idx < tail_rows * PANELS * 8; idx += 256) {
                        const int row = tail_row0 + idx / (PANELS * 8), rem = idx % (PANELS * 8);
                        *reinterpret_cast<uint4 *>(vt + (rem >> 3) * TK * 128 + row * 128 + (rem & 7) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
            }
            if (!ok) continue;
            tc_fence_after_sync();
            // sc[2k + e]: the slot's score of key 8k + 2 c4 + e of the tile (hi + lo rows)
            float sc[32];
            {
                uint32_t s0[32], s1[32];
                tmem_ld_16x256b_x8(lane_base + Cfg::kSCol + sb * TK, s0);
                tmem_ld_16x256b_x8(lane_base + Cfg::kSCol + sb * TK + 64, s1);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float2 a = add2(make_float2(__uint_as_float(s0[4 * k]), __uint_as_float(s0[4 * k + 1])),
                                          make_float2(__uint_as_float(s0[4 * k + 2]), __uint_as_float(s0[4 * k + 3])));
                    const float2 c = add2(make_float2(__uint_as_float(s1[4 * k]), __uint_as_float(s1[4 * k + 1])),
                                          make_float2(__uint_as_float(s1[4 * k + 2]), __uint_as_float(s1[4 * k + 3])));
                    sc[2 * k] = a.x;
                    sc[2 * k + 1] = a.y;
                    sc[16 + 2 * k] = c.x;
                    sc[16 + 2 * k + 1] = c.y;
                }
            }
            const int key0 = tok0 + j * TK + 2 * c4;
            if (tok0 + j * TK < lo_r || tok0 + (j + 1) * TK > hi_r) {
                // keys outside this slot's [lo_r, hi_r): before its window, after its own
                // position (causal), or past the end of the chunk
#pragma unroll
                for (int k = 0; k < 16; ++k)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        if (key0 + 8 * k + e < lo_r || key0 + 8 * k + e >= hi_r) sc[2 * k + e] = -INFINITY;
            }
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < 32; ++c) mx4[c & 3] = fmaxf(mx4[c & 3], sc[c]);
            float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
            mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 2)) * p.scale_log2;
            // a slot that has seen no key yet keeps m = -inf and weight 0
            const float m_new = mx > m_ref + 8.f ? mx : m_ref;
            const float alpha = m_new == m_ref ? 1.f : ex2_approx(m_ref - m_new);
            m_ref = m_new;
            const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
            // the key pairs as packed fp32 pairs: one FMA and one add a pair
            const float2 sl2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(neg_m, neg_m);
            float2 l2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                float2 x = fma2(make_float2(sc[2 * k], sc[2 * k + 1]), sl2, nm2);
                x.x = ex2_approx(x.x);
                x.y = ex2_approx(x.y);
                l2[k & 1] = add2(l2[k & 1], x);
                sc[2 * k] = x.x;
                sc[2 * k + 1] = x.y;
            }
            l = l * alpha + ((l2[0].x + l2[0].y) + (l2[1].x + l2[1].y));
            // pair 4k + c4 of the weights: P_hi for the hi row, P_lo for the lo row
            uint32_t pw[2][16];
#pragma unroll
            for (int k = 0; k < 16; ++k)
                split_bf16x2_p(sc[2 * k], sc[2 * k + 1], pw[k >> 3][2 * (k & 7)], pw[k >> 3][2 * (k & 7) + 1]);
            // P_{j-1} V_{j-1} must be done: the P columns are free and O is current
            if (j > 0) {
                ok = __all_sync(kFullMask, wait_or_abort(bar(Cfg::kODone), (j - 1) & 1, abort, p.err));
                if (!ok) continue;
                tc_fence_after_sync();
                if (__any_sync(kFullMask, alpha != 1.f)) {
                    // both rows of the slot, D columns in 64-column pieces
#pragma unroll
                    for (int cc = 0; cc < D / 64; ++cc) {
                        uint32_t ov[32];
                        tmem_ld_16x256b_x8(lane_base + Cfg::kOCol + cc * 64, ov);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                        tmem_st_16x256b_x8(lane_base + Cfg::kOCol + cc * 64, ov);
                    }
                }
            }
            // pair e of the hi and lo rows in column e: the 64 pairs in two 32-column stores
            tmem_st_16x128b_x8(lane_base + Cfg::kPCol, pw[0]);
            tmem_st_16x128b_x8(lane_base + Cfg::kPCol + 32, pw[1]);
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Cfg::kPFull));
        }
        if (ok) ok = __all_sync(kFullMask, wait_or_abort(bar(Cfg::kDone), 0, abort, p.err));

        // ---- the slot's sum over its four threads; O_hi + O_lo normalised
        float lr = l + __shfl_xor_sync(kFullMask, l, 1);
        lr += __shfl_xor_sync(kFullMask, lr, 2);
        // m = -inf: the slot sees no key of this chunk (an empty partial)
        const bool empty = m_ref == -INFINITY;
        const float scale = empty ? 0.f : 1.f / lr;
        if (ok) {
            tc_fence_after_sync();
            const size_t bi = row_of(slot_ok ? slot : 0);
            float *dst = nc == 1 ? p.out + bi * D : p.ws_o + (bi * p.splits + split) * D;
            // columns 8k + 2 c4, + 1 of each 64-column piece: the four threads of a slot
            // write 32 contiguous bytes a step
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                uint32_t ov[32];
                tmem_ld_16x256b_x8(lane_base + Cfg::kOCol + cc * 64, ov);
                tmem_ld_wait();
                if (slot_ok) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        *reinterpret_cast<float2 *>(dst + cc * 64 + 8 * k + 2 * c4) =
                            make_float2((__uint_as_float(ov[4 * k]) + __uint_as_float(ov[4 * k + 2])) * scale,
                                        (__uint_as_float(ov[4 * k + 1]) + __uint_as_float(ov[4 * k + 3])) * scale);
                }
            }
            if (slot_ok && c4 == 0) {
                const float lse2 = empty ? -INFINITY : m_ref + log2f(lr);
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

template <int D, int BS, int NKT, int NVT>
cudaError_t launch_umma(const DecodeKParams &kp, const CUtensorMap &tk, const CUtensorMap &tv, dim3 grid,
                        cudaStream_t stream) {
    using Cfg = UmmaDecodeCfg<D, BS, NKT, NVT>;
    auto kernel = decode_umma_kernel<D, BS, NKT, NVT>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    kernel<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(tk, tv, kp);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_umma(const DecodeKParams &kp, const CUtensorMap &tk, const CUtensorMap &tv,
                               int d, int bs, dim3 grid, cudaStream_t stream) {
    if (d == 128) return bs == 16 ? launch_umma<128, 16, 3, 3>(kp, tk, tv, grid, stream)
                                  : launch_umma<128, 32, 3, 3>(kp, tk, tv, grid, stream);
    if (d == 64) return bs == 16 ? launch_umma<64, 16, 6, 6>(kp, tk, tv, grid, stream)
                                 : launch_umma<64, 32, 6, 6>(kp, tk, tv, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
