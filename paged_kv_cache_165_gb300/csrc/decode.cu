// decode.cu -- paged decode attention: one query per sequence against its cached K/V.
//
// What is computed (for sequence b, query head i, KV head j = floor(i/m)):
//   out[b][i] = softmax_t(scale * q[b][i] . K_t) V_t over the context_lens[b] cached
//   tokens, gathered through block_table[b] (limoncc.com "大语言模型研究15——注意力机制
//   优化之KV缓存" §3.1, §3.3; plumephp.com "KV Cache 优化与注意力机制加速" §4.2-§4.3).
// The softmax is taken online, block by block, keeping a running max m and running sum
// l (plumephp.com §2.2, online_softmax_update); any stretch of blocks yields the
// log-sum-exp statistic m + log l (§2.3) by which partial results merge (split-K).
//
// Tensor-core page math (bf16 cache, d in {64,128,256}, bs in {16,32}), shared by two
// kernels.  One warp consumes one block page (bs tokens x d of K, then of V) that TMA
// brought into a 128-byte-swizzled shared-memory stage.  The m query heads of a GQA group
// share every K/V tile read from HBM: scores are m16n8k16 bf16 MMAs whose 16 A rows are
// the group's (up to 8) heads twice -- rows 0-7 the bf16 rounding of q ("hi"), rows
// 8-15 the bf16 rounding of the remainder q - hi ("lo") -- so the fp32 query enters the
// tensor core to about 2^-16 relative and the two rows of a head, held by the same
// thread, add in fp32.  The softmax weights P are split the same way for P.V.
//
// decode_chunked_kernel: one CTA per (sequence, KV-head group, chunk of blocks), whose
//   warps take the chunk's blocks round-robin, each warp with a private TMA ring (d 128,
//   bs 16: two stages, three CTAs per SM, so one CTA starting a chunk overlaps two streaming).  Chunks
//   of a unit write normalised partials; the last chunk to finish (an arrival counter, no
//   waiting) merges them by log-sum-exp.  Many short-lived CTAs let the hardware scheduler
//   balance SMs whose memory paths differ in speed (an equal static split of the pages
//   over persistent warps measured a 137-209 us spread of per-warp finish times).
// CUDA-core path (fp32 caches, other head sizes): one warp per (sequence, head, chunk),
//   chunks merged by decode_merge_kernel.
#include <algorithm>
#include <atomic>
#include <cuda_fp8.h>
#include <math.h>

#include "common.cuh"
#include "decode_epilogue.cuh"
#include "decode_kparams.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr float kLog2e = kDecLog2e;
constexpr float kLn2 = kDecLn2;
constexpr unsigned kFull = 0xffffffffu;

// ============================================================ tensor-core page math

template <int D, int BS>
struct TcPage {
    static constexpr int NT = BS / 8;    // 8-token score tiles per block
    static constexpr int KT = BS / 16;   // 16-token k-steps of P.V per block
    static constexpr int KS = D / 16;    // 16-wide k-steps of q.K
    static constexpr int ONT = D / 8;    // 8-wide output tiles
    static constexpr int PANELS = D / 64;
    static constexpr int kPageBytes = BS * D * 2;        // one K (or V) tile of a block
    static constexpr int kStageBytes = 2 * kPageBytes;   // K tile then V tile
    static_assert(D % 64 == 0 && BS % 16 == 0, "tile shape");

    // A fragments of q (16 rows x D): row g = hi part of head head0+g, row g+8 = its lo
    // remainder; rows of heads outside the group (g >= nheads) are zero.
    __device__ static void load_q(uint32_t (&qa)[KS][4], const float *q_group, int nheads,
                                  int lane) {
        const int g = lane >> 2, t4 = lane & 3;
        const bool row_ok = g < nheads;
        const float *qrow = q_group + (row_ok ? g : 0) * D;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            float2 x0 = make_float2(0.f, 0.f), x1 = make_float2(0.f, 0.f);
            if (row_ok) {
                x0 = *reinterpret_cast<const float2 *>(qrow + kk * 16 + 2 * t4);
                x1 = *reinterpret_cast<const float2 *>(qrow + kk * 16 + 8 + 2 * t4);
            }
            split_bf16x2(x0.x, x0.y, qa[kk][0], qa[kk][1]);
            split_bf16x2(x1.x, x1.y, qa[kk][2], qa[kk][3]);
        }
    }

    // Lane 0: copy the K and V tiles whose first row is `row` into stage `dst`.
    __device__ static void issue(uint32_t dst, uint32_t bar, const CUtensorMap *tm_k,
                                 const CUtensorMap *tm_v, int row) {
        mbar_arrive_expect_tx(bar, kStageBytes);
#pragma unroll
        for (int pn = 0; pn < PANELS; ++pn) {
            tma_load_2d(dst + pn * BS * 128, tm_k, pn * 64, row, bar);
            tma_load_2d(dst + kPageBytes + pn * BS * 128, tm_v, pn * 64, row, bar);
        }
    }

    __device__ static void reset(float (&o)[ONT][4], float &m_run, float &l_run) {
#pragma unroll
        for (int nt = 0; nt < ONT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
        m_run = -INFINITY;
        l_run = 0.f;
    }

    // Consume one page: its tokens first .. valid-1 (0 <= first < valid <= BS) are
    // visible.  Updates this lane's running max (head g), partial sum and output
    // fragments.
    __device__ static void page(uint8_t *stage, int first, int valid, const uint32_t (&qa)[KS][4],
                                float (&o)[ONT][4], float &m_run, float &l_run,
                                float scale_log2, int lane) {
        const int t4 = lane & 3;
        if (valid < BS) {
            // V rows past the end of the sequence may hold anything (NaN, Inf): zero them
            // so that their zero weights contribute exactly zero.
            for (int idx = lane; idx < (BS - valid) * (D / 8); idx += 32) {
                const int r = valid + idx / (D / 8), c16 = idx % (D / 8);
                *reinterpret_cast<uint4 *>(stage + kPageBytes + (c16 >> 3) * BS * 128 + r * 128 +
                                           (c16 & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
        }
        const uint32_t k_s = smem_addr(stage), v_s = k_s + kPageBytes;

        // scores S^T: (2 x group heads) x BS tokens, fp32 accumulate
        float s[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                const int mi = lane >> 3, r8 = lane & 7;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(k_s + swz128(BS, np * 16 + (mi >> 1) * 8 + r8, kk * 16 + (mi & 1) * 8),
                        b0, b1, b2, b3);
                mma_bf16_16816(s[2 * np], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                mma_bf16_16816(s[2 * np + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
            }
        }

        // online softmax (base 2) for head g: rows g (hi) + g+8 (lo) of each tile
        float sc[NT][2];
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int tok = nt * 8 + 2 * t4 + e;
                const float v = (s[nt][e] + s[nt][2 + e]) * scale_log2;
                sc[nt][e] = tok < valid && tok >= first ? v : -INFINITY;
                mx = fmaxf(mx, sc[nt][e]);
            }
        }
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
        const float m_new = fmaxf(m_run, mx);   // finite: every page holds a valid token
        const float alpha = exp2f(m_run - m_new);
        float psum = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                sc[nt][e] = exp2f(sc[nt][e] - m_new);
                psum += sc[nt][e];
            }
        }
        l_run = l_run * alpha + psum;
        m_run = m_new;
        if (__any_sync(kFull, alpha != 1.f)) {   // only when a running max moved
#pragma unroll
            for (int nt = 0; nt < ONT; ++nt) {
                o[nt][0] *= alpha;
                o[nt][1] *= alpha;
                o[nt][2] *= alpha;
                o[nt][3] *= alpha;
            }
        }

        // O += P V with P = P_hi (rows 0-7) + P_lo (rows 8-15)
#pragma unroll
        for (int kt = 0; kt < KT; ++kt) {
            uint32_t a0, a1, a2, a3;
            split_bf16x2(sc[2 * kt][0], sc[2 * kt][1], a0, a1);
            split_bf16x2(sc[2 * kt + 1][0], sc[2 * kt + 1][1], a2, a3);
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
                const int mi = lane >> 3, r8 = lane & 7;
                uint32_t b0, b1, b2, b3;
                ldsm_x4_trans(v_s + swz128(BS, kt * 16 + (mi & 1) * 8 + r8, np * 16 + (mi >> 1) * 8),
                              b0, b1, b2, b3);
                mma_bf16_16816(o[2 * np], a0, a1, a2, a3, b0, b1);
                mma_bf16_16816(o[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        __syncwarp();
    }
};

template <int D, int BS, int NW, int ST>
struct MmaCfg {
    using PG = TcPage<D, BS>;
    static constexpr int kStagesBytes = NW * ST * PG::kStageBytes;
    static constexpr int kMergeBytes = NW * (16 + 8 * D) * 4;
    static constexpr int kSmemBytes = 1024 + kStagesBytes + NW * ST * 8;
    static_assert(kMergeBytes <= kStagesBytes, "merge scratch reuses the stage buffers");
};

// Shared-memory stages of a block, aligned to the 1024-byte swizzle atom.
__device__ __forceinline__ uint8_t *aligned_smem(uint8_t *raw) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
}

// ================================================================ chunked kernel

template <int D, int BS, int NW, int ST>
__global__ void __launch_bounds__(NW * 32)
    decode_chunked_kernel(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const DecodeKParams p) {
    using PG = TcPage<D, BS>;
    using Cfg = MmaCfg<D, BS, NW, ST>;
    constexpr int KS = PG::KS, ONT = PG::ONT;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = aligned_smem(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kStagesBytes);

    pdl_launch_dependents();   // a merge kernel after this one waits for the whole grid
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    // grid: x = (chunk, head tile) with the tile fastest, y = KV head, z = sequence.  The
    // head tiles of one KV head read the same pages, so they run side by side and share
    // them in L2; chunks of one stream come next; the KV heads of one block, whose pages
    // sit side by side in HBM, are far apart in launch order.
    const int tile = blockIdx.x % p.head_tiles;
    const int split = blockIdx.x / p.head_tiles;
    const int kvh = blockIdx.y;
    const int b = blockIdx.z;
    const int g_unit = kvh * p.head_tiles + tile;
    const int head0 = kvh * p.m + tile * 8;
    const int nheads = min(8, (kvh + 1) * p.m - head0);

    const SeqSpan sp = seq_span(p, b, BS, threadIdx.x == 0 && split == 0 && g_unit == 0);
    const int len = sp.len;
    const int n_pages = sp.npages;
    const int pg0 = split * p.chunk_pages;   // pages relative to sp.pfirst
    const int pg1 = min(n_pages, pg0 + p.chunk_pages);
    if (pg0 >= pg1) {
        // Nothing to read.  Chunk 0 of an empty sequence writes out = 0, lse = -inf; any
        // other empty chunk is simply absent (the merge counts chunks from the length).
        if (split == 0) {
            // a new token for a sequence that holds none has no position: flagged, not written
            if (p.new_slots != nullptr && threadIdx.x == 0 && len == 0 && __ldg(p.new_slots + b) >= 0)
                raise_error(p.err, PKV_DEVERR_SLOT);
            for (int idx = threadIdx.x; idx < nheads * D; idx += NW * 32)
                p.out[(static_cast<size_t>(b) * p.Hq + head0 + idx / D) * D + idx % D] = 0.f;
            if (p.lse != nullptr && threadIdx.x < nheads)
                p.lse[static_cast<size_t>(b) * p.Hq + head0 + threadIdx.x] = -INFINITY;
        }
        return;
    }

    if (p.new_slots != nullptr && pg1 == n_pages) {
        // The step's new token (the append fused into this launch): the block that reads
        // the sequence's last page writes the token's K and V rows of its KV head there,
        // before any copy of the page.  The slot must be that of the last position
        // len - 1; another slot is flagged and not written.
        if (warp == 0) {
            write_new_token<D, BS>(p, b, kvh, len, lane);
            fence_proxy_async_global();   // the page's copies come after these writes
        }
        __syncthreads();
        fence_proxy_async_global();
    }

    if (lane == 0) {
        for (int s = 0; s < ST; ++s) mbar_init(smem_addr(&bars[warp * ST + s]), 1);
        fence_barrier_init();
    }
    if (threadIdx.x == 0) {
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_v);
    }
    __syncwarp();

    uint32_t qa[KS][4];
    PG::load_q(qa, p.q + (static_cast<size_t>(b) * p.Hq + head0) * D, nheads, lane);

    // This warp's blocks: pg0 + warp + NW*k, k = 0 .. n_my-1.  Block-table entries are
    // fetched 32 at a time (one per lane) ahead of the copies that need them.
    const int pages = pg1 - pg0;
    const int n_my = pages > warp ? (pages - warp + NW - 1) / NW : 0;
    const int32_t *tbl = p.block_table + static_cast<size_t>(b) * p.MBS + sp.pfirst + pg0 + warp;
    int tcur = lane < n_my ? __ldg(tbl + static_cast<size_t>(lane) * NW) : 0;
    int tnext = 32 + lane < n_my ? __ldg(tbl + static_cast<size_t>(32 + lane) * NW) : 0;
    int tbase = 0;
    const int oob_row = p.NB * p.Hkv * BS;   // a row past the end: TMA fills zeros

    auto issue = [&](int k) {   // whole warp (shuffle); lane 0 issues the copies
        while (k >= tbase + 32) {
            tcur = tnext;
            tbase += 32;
            const int kn = tbase + 32 + lane;
            tnext = kn < n_my ? __ldg(tbl + static_cast<size_t>(kn) * NW) : 0;
        }
        const int phys = __shfl_sync(kFull, tcur, k & 31);
        if (lane == 0) {
            int row;
            if (phys < 0 || phys >= p.NB) {
                raise_error(p.err, PKV_DEVERR_BLOCK);
                row = oob_row;
            } else {
                row = (phys * p.Hkv + kvh) * BS;
            }
            const int st = warp * ST + k % ST;
            PG::issue(smem_addr(smem + static_cast<size_t>(st) * PG::kStageBytes),
                      smem_addr(&bars[st]), &tm_k, &tm_v, row);
        }
    };

    float o[ONT][4];
    float m_run, l_run;
    PG::reset(o, m_run, l_run);

    int issued = min(ST, n_my);
    for (int k = 0; k < issued; ++k) issue(k);

    int k = 0;
    for (; k < n_my; ++k) {
        const int st = warp * ST + k % ST;
        const bool arrived = mbar_wait_bounded(smem_addr(&bars[st]), (k / ST) & 1);
        if (!__all_sync(kFull, arrived)) {
            if (lane == 0) raise_error(p.err, PKV_DEVERR_TIMEOUT);
            break;
        }
        const int pg = sp.pfirst + pg0 + warp + k * NW;
        PG::page(smem + static_cast<size_t>(st) * PG::kStageBytes, max(0, sp.lo - pg * BS),
                 min(BS, len - pg * BS), qa, o, m_run, l_run, p.scale_log2, lane);
        if (k + ST < n_my) {
            issue(k + ST);
            issued = k + ST + 1;
        }
    }
    if (k < n_my) {
        // A copy did not arrive in time: wait (bounded) for the copies still in flight
        // so that none lands after the block exits.
        for (int kk = k; kk < issued; ++kk)
            mbar_wait_bounded(smem_addr(&bars[warp * ST + kk % ST]), (kk / ST) & 1);
    }

    l_run += __shfl_xor_sync(kFull, l_run, 1);
    l_run += __shfl_xor_sync(kFull, l_run, 2);

    // ---- merge the warps' (m, l, O) through shared memory (stage buffers are free now)
    __syncthreads();
    float *mw = reinterpret_cast<float *>(smem);
    float *lw = mw + NW * 8;
    float *ow = lw + NW * 8;
    if (t4 == 0) {
        mw[warp * 8 + g] = m_run;
        lw[warp * 8 + g] = l_run;
    }
#pragma unroll
    for (int nt = 0; nt < ONT; ++nt) {
        float2 v = make_float2(o[nt][0] + o[nt][2], o[nt][1] + o[nt][3]);
        *reinterpret_cast<float2 *>(ow + (warp * 8 + g) * D + nt * 8 + 2 * t4) = v;
    }
    __syncthreads();
    finish_chunk<D, NW>(smem, p, b, kvh, tile, head0, nheads, split,
                        (n_pages + p.chunk_pages - 1) / p.chunk_pages);
}

// ============================================================ large-group kernel

// For m > 8 query heads per KV head (MQA is m = Hq): one CTA per (sequence, KV head,
// chunk) holds every head tile of the group.  A producer warp streams each block page of
// the chunk once into a shared ring (TMA, "full" mbarrier per stage); one consumer warp
// per 8-head tile reads every page from shared memory and releases the stage on an
// "empty" mbarrier that counts the consumer warps.  Each page thus leaves L2 once per CTA
// instead of once per head tile.
template <int D, int BS, int ST>
struct GroupCfg {
    using PG = TcPage<D, BS>;
    static constexpr int kMaxTiles = 8;   // m <= 64
    static constexpr int kStagesBytes = ST * PG::kStageBytes;
    static constexpr int kSmemBytes = 1024 + kStagesBytes + 2 * ST * 8;
};

template <int D, int BS, int ST>
__global__ void __launch_bounds__((GroupCfg<D, BS, ST>::kMaxTiles + 1) * 32, 1)
    decode_group_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeKParams p) {
    using PG = TcPage<D, BS>;
    using Cfg = GroupCfg<D, BS, ST>;
    constexpr int KS = PG::KS, ONT = PG::ONT;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = aligned_smem(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::kStagesBytes);
    uint64_t *empty = full + ST;

    pdl_launch_dependents();   // the merge kernel after this one waits for the whole grid
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int tiles = p.head_tiles;          // consumer warps; warp `tiles` is the producer
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;

    const SeqSpan sp = seq_span(p, b, BS, threadIdx.x == 0 && split == 0 && kvh == 0);
    const int len = sp.len;
    const int n_pages = sp.npages;
    const int pg0 = split * p.chunk_pages;   // pages relative to sp.pfirst
    const int pg1 = min(n_pages, pg0 + p.chunk_pages);
    const size_t bi_group = static_cast<size_t>(b) * p.Hq + static_cast<size_t>(kvh) * p.m;
    if (pg0 >= pg1) {
        if (split == 0) {   // an empty sequence: out = 0, lse = -inf for the whole group
            for (int idx = threadIdx.x; idx < p.m * D; idx += blockDim.x) p.out[bi_group * D + idx] = 0.f;
            if (p.lse != nullptr)
                for (int h = threadIdx.x; h < p.m; h += blockDim.x) p.lse[bi_group + h] = -INFINITY;
        }
        return;
    }
    const int pages = pg1 - pg0;
    __shared__ int s_issued;
    if (threadIdx.x == 0) {
        s_issued = 0;
        for (int s = 0; s < ST; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), tiles);
        }
        fence_barrier_init();
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_v);
    }
    __syncthreads();

    bool ok = true;
    if (warp == tiles) {
        // ---- producer: page k goes to stage k % ST once the consumers released it
        const int32_t *tbl = p.block_table + static_cast<size_t>(b) * p.MBS + sp.pfirst + pg0;
        int tcur = lane < pages ? __ldg(tbl + lane) : 0;
        int tnext = 32 + lane < pages ? __ldg(tbl + 32 + lane) : 0;
        int tbase = 0;
        const int oob_row = p.NB * p.Hkv * BS;
        for (int k = 0; k < pages; ++k) {
            while (k >= tbase + 32) {
                tcur = tnext;
                tbase += 32;
                tnext = tbase + 32 + lane < pages ? __ldg(tbl + tbase + 32 + lane) : 0;
            }
            const int phys = __shfl_sync(kFull, tcur, k & 31);
            const int st = k % ST;
            bool free_ = true;
            if (lane == 0 && k >= ST)
                free_ = mbar_wait_bounded(smem_addr(&empty[st]), ((k / ST) - 1) & 1);
            if (!__shfl_sync(kFull, free_ ? 1 : 0, 0)) {
                if (lane == 0) raise_error(p.err, PKV_DEVERR_TIMEOUT);
                ok = false;
                break;
            }
            if (lane == 0) {
                int row = oob_row;
                if (phys < 0 || phys >= p.NB) raise_error(p.err, PKV_DEVERR_BLOCK);
                else row = (phys * p.Hkv + kvh) * BS;
                PG::issue(smem_addr(smem + static_cast<size_t>(st) * PG::kStageBytes),
                          smem_addr(&full[st]), &tm_k, &tm_v, row);
                s_issued = k + 1;
            }
            __syncwarp();
        }
    } else {
        // ---- consumer warp: heads head0 .. head0 + nheads - 1 of the group
        const int head0 = warp * 8;
        const int nheads = min(8, p.m - head0);
        uint32_t qa[KS][4];
        PG::load_q(qa, p.q + (bi_group + head0) * D, nheads, lane);
        float o[ONT][4];
        float m_run, l_run;
        PG::reset(o, m_run, l_run);
        int k = 0;
        for (; k < pages; ++k) {
            const int st = k % ST;
            const bool arrived = mbar_wait_bounded(smem_addr(&full[st]), (k / ST) & 1);
            if (!__all_sync(kFull, arrived)) {
                if (lane == 0) raise_error(p.err, PKV_DEVERR_TIMEOUT);
                ok = false;
                break;
            }
            const int pg = sp.pfirst + pg0 + k;
            PG::page(smem + static_cast<size_t>(st) * PG::kStageBytes, max(0, sp.lo - pg * BS),
                     min(BS, len - pg * BS), qa, o, m_run, l_run, p.scale_log2, lane);
            if (lane == 0) mbar_arrive(smem_addr(&empty[st]));
        }
        l_run += __shfl_xor_sync(kFull, l_run, 1);
        l_run += __shfl_xor_sync(kFull, l_run, 2);
        const int nc = (n_pages + p.chunk_pages - 1) / p.chunk_pages;
        if (ok && g < nheads) {
            const float inv_l = 1.f / l_run;
            const size_t bi = bi_group + head0 + g;
            float *dst = nc == 1 ? p.out + bi * D : p.ws_o + (bi * p.splits + split) * D;
#pragma unroll
            for (int nt = 0; nt < ONT; ++nt)
                *reinterpret_cast<float2 *>(dst + nt * 8 + 2 * t4) =
                    make_float2((o[nt][0] + o[nt][2]) * inv_l, (o[nt][1] + o[nt][3]) * inv_l);
            if (t4 == 0) {
                const float lse2 = m_run + log2f(l_run);
                if (nc == 1) {
                    if (p.lse != nullptr) p.lse[bi] = lse2 * kLn2;
                } else {
                    p.ws_lse[bi * p.splits + split] = lse2;
                }
            }
        }
    }
    if (__syncthreads_or(!ok)) {
        // a wait gave up: let the last copies issued land (bounded) before the block exits
        if (threadIdx.x == 0)
            for (int k = max(0, s_issued - ST); k < s_issued; ++k)
                mbar_wait_bounded(smem_addr(&full[k % ST]), (k / ST) & 1);
        return;
    }
    const int nc = (n_pages + p.chunk_pages - 1) / p.chunk_pages;
    if (nc == 1 || p.counters == nullptr) return;

    // ---- the last chunk of this (sequence, KV head) to finish merges the chunks
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned *ctr = p.counters + static_cast<size_t>(b) * p.Hkv + kvh;
        const unsigned prev = atomicAdd(ctr, 1u);
        s_last = prev + 1 == static_cast<unsigned>(nc);
        if (s_last) *ctr = 0u;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int nw = blockDim.x >> 5;
    for (int h = warp; h < p.m; h += nw) {
        const size_t bi = bi_group + h;
        const float *ls = p.ws_lse + bi * p.splits;
        float M = -INFINITY;
        for (int c = lane; c < nc; c += 32) M = fmaxf(M, __ldcg(ls + c));
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, sh));
        float L = 0.f;
        for (int c = lane; c < nc; c += 32) L += exp2f(__ldcg(ls + c) - M);
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) L += __shfl_xor_sync(kFull, L, sh);
        const float il = 1.f / L;
        for (int c4 = lane * 4; c4 < D; c4 += 128) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (int c = 0; c < nc; ++c) {
                const float w = exp2f(__ldcg(ls + c) - M);
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                    p.ws_o + (bi * p.splits + c) * D + c4));
                acc.x += w * v.x;
                acc.y += w * v.y;
                acc.z += w * v.z;
                acc.w += w * v.w;
            }
            *reinterpret_cast<float4 *>(p.out + bi * D + c4) =
                make_float4(acc.x * il, acc.y * il, acc.z * il, acc.w * il);
        }
        if (lane == 0 && p.lse != nullptr) p.lse[bi] = (M + log2f(L)) * kLn2;
    }
}

// ================================================================ CUDA-core path

template <typename T>
__device__ __forceinline__ float load_f32(const T *p);
template <>
__device__ __forceinline__ float load_f32<float>(const float *p) { return __ldg(p); }
template <>
__device__ __forceinline__ float load_f32<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}
// an E4M3 code (its row scale is applied by the caller)
template <>
__device__ __forceinline__ float load_f32<uint8_t>(const uint8_t *p) {
    return __half2float(__half(__nv_cvt_fp8_to_halfraw(*p, __NV_E4M3)));
}

// One warp per (query row, query head, chunk); lanes own head-dim elements lane + 32*j.
// A row is a sequence (decode) or one of the query rows of a sequence (cu_q).
template <typename T, int J>
__global__ void __launch_bounds__(32)
    decode_simt_kernel(const T *__restrict__ kc, const T *__restrict__ vc, const DecodeKParams p,
                       int d, int bs) {
    pdl_launch_dependents();   // the merge kernel after this one waits for the whole grid
    const int lane = threadIdx.x;
    const int row = blockIdx.x, i = blockIdx.y, split = blockIdx.z;
    const int kvh = i / p.m;
    const SeqSpan sp = row_span(p, row, bs, lane == 0 && split == 0 && i == 0);
    const int b = sp.b;
    const int len = sp.len;
    const int nc = (sp.cnpages + p.chunk_pages - 1) / p.chunk_pages;   // the sequence's chunks
    const int c0 = sp.cpfirst + split * p.chunk_pages;                  // this chunk's pages
    const int c1 = min(sp.cpfirst + sp.cnpages, c0 + p.chunk_pages);
    const int pg0 = max(c0, sp.pfirst);                                 // ... that this row sees
    const int pg1 = min(c1, sp.pfirst + sp.npages);
    const size_t bi = static_cast<size_t>(row) * p.Hq + i;
    if (c0 >= c1) {
        if (split == 0) {   // an empty sequence: out = 0, lse = -inf
            for (int e = lane; e < d; e += 32) p.out[bi * d + e] = 0.f;
            if (lane == 0 && p.lse != nullptr) p.lse[bi] = -INFINITY;
        }
        return;
    }
    if (pg0 >= pg1) {   // the chunk holds none of this row's keys: an empty partial
        for (int e = lane; e < d; e += 32) p.ws_o[(bi * p.splits + split) * d + e] = 0.f;
        if (lane == 0) p.ws_lse[bi * p.splits + split] = -INFINITY;
        return;
    }
    float qv[J], acc[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        qv[j] = e < d ? p.q[bi * d + e] : 0.f;
        acc[j] = 0.f;
    }
    float m_run = -INFINITY, l_run = 0.f;
    for (int pg = pg0; pg < pg1; ++pg) {
        const int phys = __ldg(p.block_table + static_cast<size_t>(b) * p.MBS + pg);
        const bool bad = phys < 0 || phys >= p.NB;
        if (bad && lane == 0) raise_error(p.err, PKV_DEVERR_BLOCK);
        const int valid = min(bs, len - pg * bs);
        for (int off = max(0, sp.lo - pg * bs); off < valid; ++off) {
            const size_t srow = bad ? 0 : (static_cast<size_t>(phys) * p.Hkv + kvh) * bs + off;
            const size_t base = srow * d;
            float dot = 0.f;
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int e = lane + 32 * j;
                if (e < d && !bad) dot += qv[j] * load_f32(kc + base + e);
            }
#pragma unroll
            for (int sh = 16; sh > 0; sh >>= 1) dot += __shfl_xor_sync(kFull, dot, sh);
            if (p.k_scale != nullptr && !bad) dot *= __ldg(p.k_scale + srow);   // FP8 rows
            const float s = dot * p.scale_log2;
            const float m_new = fmaxf(m_run, s);
            const float alpha = exp2f(m_run - m_new);
            const float w = exp2f(s - m_new);
            l_run = l_run * alpha + w;
            const float wv = p.v_scale != nullptr && !bad ? w * __ldg(p.v_scale + srow) : w;
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int e = lane + 32 * j;
                const float v = (e < d && !bad) ? load_f32(vc + base + e) : 0.f;
                acc[j] = acc[j] * alpha + wv * v;
            }
            m_run = m_new;
        }
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        if (e >= d) continue;
        if (nc == 1)
            p.out[bi * d + e] = acc[j] / l_run;
        else
            p.ws_o[(bi * p.splits + split) * d + e] = acc[j] / l_run;
    }
    if (lane == 0) {
        if (nc == 1) {
            if (p.lse != nullptr) p.lse[bi] = (m_run + log2f(l_run)) * kLn2;
        } else {
            p.ws_lse[bi * p.splits + split] = m_run + log2f(l_run);
        }
    }
}

// ==================================================================== LSE merge

// One block of 256 threads per (sequence, query head): lse = log2 sum_c 2^{lse_c} and
// out = sum_c 2^{lse_c - lse} o_c over the chunks that hold tokens.  The chunk weights
// are computed in parallel into shared memory.  The threads then form G groups of d/4
// (d/1 when d is not a multiple of 4) threads; group k sums chunks k, k+G, ... of its
// columns, so each thread has nc/G independent row loads in flight rather than a chain
// of nc/4, and the G partial sums are added through shared memory.  Sequences with at
// most one chunk were written directly by the attention kernel.
constexpr int kMergeThreads = 256;
constexpr int kMergeMaxChunks = 4096;
constexpr int kMergePrefetch = 6;   // even: the prefetched chunks keep the two sums' order

__global__ void __launch_bounds__(kMergeThreads)
    decode_merge_kernel(const DecodeKParams p, int d, int bs) {
    __shared__ float w[kMergeMaxChunks];
    __shared__ float red[kMergeThreads / 32];
    __shared__ __align__(16) float part[4 * kMergeThreads];   // G x d partial sums, G * d <= 1024
    // Every block waits for the attention kernel before it (launched as its programmatic
    // dependent) to complete, also one that has nothing to merge: the grid must not end
    // before that kernel, which work queued after it relies on.
    pdl_wait();
    const size_t bi = blockIdx.x;
    const int b = static_cast<int>(bi / p.Hq);
    const int n_pages = row_span(p, b, bs, false).cnpages;
    const int nc = (n_pages + p.chunk_pages - 1) / p.chunk_pages;
    if (nc <= 1) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float *ls = p.ws_lse + bi * p.splits;
    const float *po = p.ws_o + bi * p.splits * d;
    const bool vec = d % 4 == 0 && (reinterpret_cast<uintptr_t>(p.ws_o) & 15) == 0;
    const int width = vec ? d / 4 : d;          // threads per group (d <= 256)
    const int G = kMergeThreads / width;        // groups
    const int grp = tid / width, col = tid % width;
    // the rows of this thread's first kMergePrefetch chunks, loaded before the weights are
    // known so that their latency overlaps the weights' reductions
    float4 pre[kMergePrefetch];
    if (vec && grp < G) {
#pragma unroll
        for (int i = 0; i < kMergePrefetch; ++i) {
            const int c = grp + i * G;
            pre[i] = c < nc ? *reinterpret_cast<const float4 *>(po + static_cast<size_t>(c) * d + 4 * col)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    float M = -INFINITY;
    for (int c = tid; c < nc; c += kMergeThreads) {
        w[c] = ls[c];
        M = fmaxf(M, w[c]);
    }
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, sh));
    if (lane == 0) red[warp] = M;
    __syncthreads();
    M = red[0];
#pragma unroll
    for (int i = 1; i < kMergeThreads / 32; ++i) M = fmaxf(M, red[i]);
    __syncthreads();
    float L = 0.f;
    for (int c = tid; c < nc; c += kMergeThreads) {
        w[c] = exp2f(w[c] - M);
        L += w[c];
    }
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) L += __shfl_xor_sync(kFull, L, sh);
    if (lane == 0) red[warp] = L;
    __syncthreads();
    L = 0.f;
#pragma unroll
    for (int i = 0; i < kMergeThreads / 32; ++i) L += red[i];
    const float il = 1.f / L;
    if (grp < G) {
        if (vec) {
            float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
            // chunks grp + iG alternate between the two sums, as in the loop below
#pragma unroll
            for (int i = 0; i < kMergePrefetch; ++i) {
                const int c = grp + i * G;
                if (c < nc) {
                    const float wx = w[c];
                    float4 &a = (i & 1) ? a1 : a0;
                    a.x += wx * pre[i].x; a.y += wx * pre[i].y; a.z += wx * pre[i].z; a.w += wx * pre[i].w;
                }
            }
            int c = grp + kMergePrefetch * G;
            for (; c + G < nc; c += 2 * G) {
                const float4 x = *reinterpret_cast<const float4 *>(po + static_cast<size_t>(c) * d + 4 * col);
                const float4 y = *reinterpret_cast<const float4 *>(po + static_cast<size_t>(c + G) * d + 4 * col);
                const float wx = w[c], wy = w[c + G];
                a0.x += wx * x.x; a0.y += wx * x.y; a0.z += wx * x.z; a0.w += wx * x.w;
                a1.x += wy * y.x; a1.y += wy * y.y; a1.z += wy * y.z; a1.w += wy * y.w;
            }
            if (c < nc) {
                const float4 x = *reinterpret_cast<const float4 *>(po + static_cast<size_t>(c) * d + 4 * col);
                const float wx = w[c];
                a0.x += wx * x.x; a0.y += wx * x.y; a0.z += wx * x.z; a0.w += wx * x.w;
            }
            *reinterpret_cast<float4 *>(part + grp * d + 4 * col) =
                make_float4(a0.x + a1.x, a0.y + a1.y, a0.z + a1.z, a0.w + a1.w);
        } else {
            float a0 = 0.f, a1 = 0.f;
            int c = grp;
            for (; c + G < nc; c += 2 * G) {
                a0 += w[c] * po[static_cast<size_t>(c) * d + col];
                a1 += w[c + G] * po[static_cast<size_t>(c + G) * d + col];
            }
            if (c < nc) a0 += w[c] * po[static_cast<size_t>(c) * d + col];
            part[grp * d + col] = a0 + a1;
        }
    }
    __syncthreads();
    for (int e = tid; e < d; e += kMergeThreads) {
        float acc = 0.f;
        for (int k = 0; k < G; ++k) acc += part[k * d + e];
        p.out[bi * d + e] = acc * il;
    }
    if (tid == 0 && p.lse != nullptr) p.lse[bi] = (M + log2f(L)) * kLn2;
}

// The merge as a programmatic dependent of the attention kernel just launched on `stream`:
// its blocks may be scheduled while the attention kernel drains and wait in pdl_wait().
cudaError_t launch_merge(const DecodeKParams &kp, int d, int bs, unsigned rows_x_heads, cudaStream_t stream) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(rows_x_heads);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_merge_kernel, kp, d, bs);
}

// ====================================================================== launch

template <typename Kernel>
cudaError_t set_smem_once(Kernel kernel, int bytes, std::atomic<unsigned long long> &done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(done.load() & bit)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        done.fetch_or(bit);
    }
    return cudaSuccess;
}

template <int D, int BS, int NW, int ST>
cudaError_t launch_tc(const DecodeKParams &kp, const CUtensorMap &tk, const CUtensorMap &tv,
                      dim3 grid, cudaStream_t stream) {
    using Cfg = MmaCfg<D, BS, NW, ST>;
    static std::atomic<unsigned long long> done{0};
    auto kernel = decode_chunked_kernel<D, BS, NW, ST>;
    cudaError_t e = set_smem_once(kernel, Cfg::kSmemBytes, done);
    if (e != cudaSuccess) return e;
    kernel<<<grid, NW * 32, Cfg::kSmemBytes, stream>>>(tk, tv, kp);
    return cudaGetLastError();
}

template <int D, int BS, int ST>
cudaError_t launch_group(const DecodeKParams &kp, const CUtensorMap &tk, const CUtensorMap &tv,
                         dim3 grid, cudaStream_t stream) {
    using Cfg = GroupCfg<D, BS, ST>;
    static std::atomic<unsigned long long> done{0};
    auto kernel = decode_group_kernel<D, BS, ST>;
    cudaError_t e = set_smem_once(kernel, Cfg::kSmemBytes, done);
    if (e != cudaSuccess) return e;
    kernel<<<grid, (kp.head_tiles + 1) * 32, Cfg::kSmemBytes, stream>>>(tk, tv, kp);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_simt(const DecodeArgs &a, const DecodeKParams &kp, dim3 grid,
                        cudaStream_t stream) {
    const T *kc = static_cast<const T *>(a.k_cache);
    const T *vc = static_cast<const T *>(a.v_cache);
    const int J = (a.d + 31) / 32;
    switch (J) {
#define PKV_SIMT_CASE(n)                                                                  \
    case n:                                                                               \
        decode_simt_kernel<T, n><<<grid, 32, 0, stream>>>(kc, vc, kp, a.d, a.bs);          \
        break;
        PKV_SIMT_CASE(1)
        PKV_SIMT_CASE(2)
        PKV_SIMT_CASE(3)
        PKV_SIMT_CASE(4)
        PKV_SIMT_CASE(5)
        PKV_SIMT_CASE(6)
        PKV_SIMT_CASE(7)
        PKV_SIMT_CASE(8)
#undef PKV_SIMT_CASE
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// Units with at most this many chunks merge inside the attention kernel.
constexpr int kFusedMergeMaxChunks = 8;

// Chunk plan: a chunk size, the chunk count per sequence and the workspace layout --
// arrival counters (a fixed-size region, so that a workspace zeroed once stays valid for
// any later shape), then o partials [B*Hq][splits][d], then lse partials [B*Hq][splits].
void chunk_plan(DecodePlan &plan, int B, int Hq, int Hkv, int d, int bs, int MBS, int num_splits,
                int sm_count, int rows = -1) {
    if (rows < 0) rows = B;   // query rows (partials are per row and head)
    const int m = Hq / Hkv;
    const long long units = static_cast<long long>(B) * Hkv * ((m + 7) / 8);
    const long long max_counters = PKV_DECODE_COUNTER_BYTES / sizeof(unsigned);
    int chunk = MBS;
    if (num_splits == 1) {
        chunk = MBS;
    } else if (num_splits > 1) {
        chunk = (MBS + num_splits - 1) / num_splits;
    } else {
        // enough (sequence, head-group, chunk) units for several waves of the CTAs an SM holds,
        // without making chunks shorter than 16 blocks
        const long long target = 8ll * std::max(sm_count, 1);
        while (chunk > 16 && units * ((MBS + chunk - 1) / chunk) < target)
            chunk = (chunk + 1) / 2;
        // and no chunk longer than 8192 tokens (equal chunks): a long sequence among short
        // ones then spreads over several blocks instead of running alone at the end of the
        // launch (a ragged batch with one chunk per sequence ran 1.4x slower)
        const int cap = std::max(16, 8192 / bs);
        if (chunk > cap) {
            const int parts = (MBS + cap - 1) / cap;
            chunk = (MBS + parts - 1) / parts;
        }
    }
    chunk = std::max(chunk, (MBS + kMergeMaxChunks - 1) / kMergeMaxChunks);   // merge capacity
    chunk = std::max(chunk, 1);
    if (plan.umma) {
        // one CTA per (sequence, KV head, chunk) and SM, one wave: the start of a block
        // (queries, first copies) and its end are paid once per SM; chunks of whole
        // 128-key tiles
        const int ppt = kUmmaDecodeKeys / bs;
        if (num_splits == 0) {
            const long long gunits = static_cast<long long>(B) * Hkv * plan.qtiles;
            const long long per_unit = std::max(1ll, (std::max(sm_count, 1) + gunits - 1) / gunits);
            chunk = static_cast<int>((MBS + per_unit - 1) / per_unit);
        }
        chunk = std::max(chunk, (MBS + kMergeMaxChunks - 1) / kMergeMaxChunks);
        chunk = (chunk + ppt - 1) / ppt * ppt;
    } else if (plan.group && num_splits == 0) {
        // one CTA per (sequence, KV head, chunk) with up to 9 warps: about four waves
        chunk = MBS;
        const long long gunits = static_cast<long long>(B) * Hkv;
        const long long target = 2ll * std::max(sm_count, 1);
        while (chunk > 16 && gunits * ((MBS + chunk - 1) / chunk) < target) chunk = (chunk + 1) / 2;
    }
    // the grid's x holds chunks x head tiles
    const int tiles = (m + 7) / 8;
    chunk = std::max(chunk, static_cast<int>((static_cast<long long>(MBS) * tiles + 0x7ffffffell - 1) / 0x7ffffffell));
    plan.chunk_pages = chunk;
    plan.splits = (MBS + chunk - 1) / chunk;
    plan.workspace_bytes = plan.splits > 1 ? PKV_DECODE_COUNTER_BYTES +
                                                 static_cast<size_t>(rows) * Hq * plan.splits *
                                                     (static_cast<size_t>(d) + 1) * sizeof(float)
                                           : 0;
    // The last chunk merges in place when a unit has few chunks; many chunks (long
    // contexts, the group kernel) merge in a separate kernel, many blocks at once.
    plan.fused_merge = plan.tensor_core && !plan.group && plan.splits > 1 &&
                       plan.splits <= kFusedMergeMaxChunks && units <= max_counters;
    plan.counter_bytes = plan.fused_merge ? static_cast<size_t>(units) * sizeof(unsigned) : 0;
}

}  // namespace

// The chunked bf16 kernel with one head tile per KV head (m <= 8), and the tcgen05 kernel
// with one query tile per sequence, write the step's new tokens themselves: exactly one
// block reads the page that holds a sequence's last position for each KV head.  The
// 16-byte row copies need 16-byte aligned new rows.  The FP8 kernel (m <= 8 as well)
// quantises bf16 new rows there.
bool decode_fuses_append(const DecodePlan &plan, pkv_dtype dt, pkv_dtype new_dt, int Hq, int Hkv,
                         const void *k_new, const void *v_new) {
    if (!plan.tensor_core || new_dt != PKV_BF16) return false;
    if (dt == PKV_FP8_E4M3)
        return Hq / Hkv <= 8 && reinterpret_cast<uintptr_t>(k_new) % 2 == 0 &&
               reinterpret_cast<uintptr_t>(v_new) % 2 == 0;
    const bool kernel_ok = (!plan.group && !plan.umma && Hq / Hkv <= 8) || (plan.umma && plan.qtiles == 1);
    return dt == PKV_BF16 && kernel_ok && reinterpret_cast<uintptr_t>(k_new) % 16 == 0 &&
           reinterpret_cast<uintptr_t>(v_new) % 16 == 0;
}

DecodePlan plan_decode(int B, int Hq, int Hkv, int d, int bs, int MBS, int NB, pkv_dtype dt,
                       int num_splits, int sm_count, bool caches_aligned, bool q_aligned) {
    DecodePlan plan{};
    plan.sm_count = sm_count;
    const int tiles = (Hq / Hkv + 7) / 8;
    if (dt == PKV_FP8_E4M3) {
        // E4M3 codes: the tensor-core kernel takes d = 128 and one head tile per KV head
        plan.tensor_core = d == 128 && (bs == 16 || bs == 32) && tiles == 1 && caches_aligned &&
                           static_cast<long long>(NB + 1) * Hkv * bs < (1ll << 31);
        chunk_plan(plan, B, Hq, Hkv, d, bs, MBS, num_splits, sm_count);
        return plan;
    }
    plan.tensor_core = dt == PKV_BF16 && (d == 64 || d == 128 || d == 256) &&
                       (bs == 16 || bs == 32) && caches_aligned &&
                       static_cast<long long>(NB + 1) * Hkv * bs < (1ll << 31);
    plan.group = plan.tensor_core && tiles >= 2 && tiles <= 8;
    plan.umma = plan.group && (d == 64 || d == 128) && q_aligned;
    chunk_plan(plan, B, Hq, Hkv, d, bs, MBS, num_splits, sm_count);
    return plan;
}

DecodePlan plan_attention_rows(int B, int Tq, int max_q, int Hq, int Hkv, int d, int bs, int MBS, int NB,
                               pkv_dtype dt, int window, int num_splits, int sm_count, bool caches_aligned,
                               bool q_aligned) {
    DecodePlan plan{};
    plan.sm_count = sm_count;
    const int m = Hq / Hkv;
    if (dt == PKV_BF16 && (d == 64 || d == 128) && (bs == 16 || bs == 32) && caches_aligned && q_aligned &&
        window == 0 && max_q >= kPagedPrefillMinRows && static_cast<long long>(NB + 1) * Hkv * bs < (1ll << 31)) {
        // a chunk of new tokens per sequence over its cached prefix: 128 query rows of one
        // head per block over all of the sequence's keys, in one pass
        plan.paged_prefill = plan.tensor_core = true;
        plan.qtiles = (max_q + 127) / 128;
        plan.splits = 1;
        plan.chunk_pages = MBS;
        plan.workspace_bytes = 0;
        plan.fused_merge = false;
        return plan;
    }
    plan.umma = dt == PKV_BF16 && (d == 64 || d == 128) && (bs == 16 || bs == 32) && caches_aligned &&
                q_aligned && m <= 64 && static_cast<long long>(NB + 1) * Hkv * bs < (1ll << 31);
    if (plan.umma) {
        plan.q_per_tile = 64 / m;
        plan.qtiles = (max_q + plan.q_per_tile - 1) / plan.q_per_tile;
        plan.umma = static_cast<long long>(B) * plan.qtiles <= 65535;
    }
    if (!plan.umma) plan.q_per_tile = plan.qtiles = 1;
    plan.tensor_core = plan.group = plan.umma;
    chunk_plan(plan, B, Hq, Hkv, d, bs, MBS, num_splits, sm_count, Tq);
    return plan;
}

size_t decode_workspace_upper_bound(int B, int Hq, int Hkv, int d, int bs, int MBS,
                                    int num_splits, int sm_count) {
    // the query knows neither the element type nor the alignment: cover both paths
    DecodePlan tc{}, umma{}, other{};
    tc.tensor_core = true;
    const int tiles = (Hq / Hkv + 7) / 8;
    tc.group = tiles >= 2 && tiles <= 8;
    umma = tc;
    umma.umma = tc.group && (d == 64 || d == 128) && (bs == 16 || bs == 32);
    chunk_plan(tc, B, Hq, Hkv, d, bs, MBS, num_splits, sm_count);
    chunk_plan(umma, B, Hq, Hkv, d, bs, MBS, num_splits, sm_count);
    chunk_plan(other, B, Hq, Hkv, d, bs, MBS, num_splits, sm_count);
    return std::max({tc.workspace_bytes, umma.workspace_bytes, other.workspace_bytes});
}

cudaError_t launch_decode(const DecodeArgs &a, const DecodePlan &plan, pkv_dtype dt,
                          cudaStream_t stream) {
    const int rows = a.rows >= 0 ? a.rows : a.B;
    if (a.B == 0 || rows == 0) return cudaSuccess;
    if (a.cu_q != nullptr && plan.tensor_core && !plan.umma && !plan.paged_prefill) return cudaErrorInvalidValue;
    DecodeKParams kp{};
    kp.out = a.out;
    kp.lse = a.lse;
    kp.q = a.q;
    kp.block_table = a.block_table;
    kp.context_lens = a.context_lens;
    kp.err = a.err;
    kp.B = a.B;
    kp.Hq = a.Hq;
    kp.Hkv = a.Hkv;
    kp.m = a.Hq / a.Hkv;
    kp.MBS = a.MBS;
    kp.NB = a.NB;
    kp.head_tiles = (kp.m + 7) / 8;
    kp.chunk_pages = plan.chunk_pages;
    kp.splits = plan.splits;
    kp.scale_log2 = a.scale * kLog2e;
    kp.window = a.window;
    kp.cu_q = a.cu_q;
    kp.k_scale = a.k_scale;
    kp.v_scale = a.v_scale;
    kp.q_per_tile = plan.q_per_tile;
    kp.qtiles = plan.qtiles;
    kp.kv_start = a.kv_start;
    if (a.new_slots != nullptr && decode_fuses_append(plan, dt, PKV_BF16, a.Hq, a.Hkv, a.k_new, a.v_new)) {
        kp.k_new = a.k_new;
        kp.v_new = a.v_new;
        kp.new_slots = a.new_slots;
        kp.k_cache_w = const_cast<void *>(a.k_cache);
        kp.v_cache_w = const_cast<void *>(a.v_cache);
        kp.k_scale_w = const_cast<float *>(a.k_scale);
        kp.v_scale_w = const_cast<float *>(a.v_scale);
    }
    // the tcgen05 kernel with one query tile per sequence (decode, verification): each block
    // takes a whole chunk for a long time, so start the long sequences first (a block ranks
    // up to 256 lengths at its start; a 4-token verification step on ragged lengths: 4.7%
    // faster).  With many query tiles per sequence the blocks are fine-grained already and
    // the ranking cost 1%.
    // ... but only when the grid has more blocks than one wave: in a single wave every block
    // starts at once and the ranking (a load of every length at the block's start) only delays
    // the first copies
    kp.longest_first = plan.umma && plan.qtiles == 1 && a.B <= 256 &&
                               static_cast<long long>(plan.splits) * a.Hkv * a.B > plan.sm_count
                           ? 1
                           : 0;
    if (plan.splits > 1) {
        uint8_t *ws = static_cast<uint8_t *>(a.workspace);
        kp.counters = plan.fused_merge ? reinterpret_cast<unsigned *>(ws) : nullptr;
        kp.ws_o = reinterpret_cast<float *>(ws + PKV_DECODE_COUNTER_BYTES);
        kp.ws_lse = kp.ws_o + static_cast<size_t>(rows) * a.Hq * plan.splits * a.d;
    }

    cudaError_t e;
    if (plan.paged_prefill) {
        CUtensorMap tk, tv;
        const uint64_t dims[2] = {static_cast<uint64_t>(a.d), static_cast<uint64_t>(a.NB) * a.Hkv * a.bs};
        const uint64_t strides[1] = {static_cast<uint64_t>(a.d) * 2};
        const uint32_t box[2] = {64, static_cast<uint32_t>(a.bs)};
        if (a.cu_q == nullptr || !encode_map_bf16(&tk, a.k_cache, 2, dims, strides, box) ||
            !encode_map_bf16(&tv, a.v_cache, 2, dims, strides, box))
            return cudaErrorInvalidValue;
        return launch_paged_prefill(kp, tk, tv, a.d, a.bs, dim3(plan.qtiles, a.Hq, a.B), stream);
    }
    if (dt == PKV_FP8_E4M3 && plan.tensor_core) {
        CUtensorMap tk, tv;
        const uint64_t dims[2] = {static_cast<uint64_t>(a.d), static_cast<uint64_t>(a.NB) * a.Hkv * a.bs};
        const uint64_t strides[1] = {static_cast<uint64_t>(a.d)};
        const uint32_t box[2] = {128, static_cast<uint32_t>(a.bs)};
        if (!encode_map_u8(&tk, a.k_cache, 2, dims, strides, box) ||
            !encode_map_u8(&tv, a.v_cache, 2, dims, strides, box))
            return cudaErrorInvalidValue;
        e = launch_decode_fp8(kp, tk, tv, a.bs, dim3(static_cast<unsigned>(plan.splits) * kp.head_tiles, a.Hkv, a.B),
                              stream);
        if (e != cudaSuccess || plan.splits == 1 || plan.fused_merge) return e;
    } else if (plan.tensor_core) {
        CUtensorMap tk, tv;
        const uint64_t dims[2] = {static_cast<uint64_t>(a.d),
                                  static_cast<uint64_t>(a.NB) * a.Hkv * a.bs};
        const uint64_t strides[1] = {static_cast<uint64_t>(a.d) * 2};
        const uint32_t box[2] = {64, static_cast<uint32_t>(a.bs)};
        if (!encode_map_bf16(&tk, a.k_cache, 2, dims, strides, box) ||
            !encode_map_bf16(&tv, a.v_cache, 2, dims, strides, box))
            return cudaErrorInvalidValue;
        if (plan.umma) {
            e = launch_decode_umma(kp, tk, tv, a.d, a.bs, dim3(plan.splits, a.Hkv, a.B * plan.qtiles), stream);
            if (e != cudaSuccess || plan.splits == 1) return e;
            return launch_merge(kp, a.d, a.bs, static_cast<unsigned>(rows * a.Hq), stream);
        }
        if (plan.group) {
            const dim3 ggrid(plan.splits, a.Hkv, a.B);
            if (a.bs == 16) {
                if (a.d == 64) e = launch_group<64, 16, 16>(kp, tk, tv, ggrid, stream);
                else if (a.d == 128) e = launch_group<128, 16, 12>(kp, tk, tv, ggrid, stream);
                else e = launch_group<256, 16, 6>(kp, tk, tv, ggrid, stream);
            } else {
                if (a.d == 64) e = launch_group<64, 32, 12>(kp, tk, tv, ggrid, stream);
                else if (a.d == 128) e = launch_group<128, 32, 6>(kp, tk, tv, ggrid, stream);
                else e = launch_group<256, 32, 3>(kp, tk, tv, ggrid, stream);
            }
            if (e != cudaSuccess || plan.splits == 1) return e;
            return launch_merge(kp, a.d, a.bs, static_cast<unsigned>(a.B * a.Hq), stream);
        }
        const dim3 grid(static_cast<unsigned>(plan.splits) * kp.head_tiles, a.Hkv, a.B);
        if (a.bs == 16) {
            if (a.d == 64) e = launch_tc<64, 16, 4, 6>(kp, tk, tv, grid, stream);
            else if (a.d == 128) e = launch_tc<128, 16, 4, 2>(kp, tk, tv, grid, stream);
            else e = launch_tc<256, 16, 4, 2>(kp, tk, tv, grid, stream);
        } else {
            if (a.d == 64) e = launch_tc<64, 32, 4, 3>(kp, tk, tv, grid, stream);
            else if (a.d == 128) e = launch_tc<128, 32, 2, 2>(kp, tk, tv, grid, stream);
            else e = launch_tc<256, 32, 2, 2>(kp, tk, tv, grid, stream);
        }
        if (e != cudaSuccess || plan.splits == 1 || plan.fused_merge) return e;
    } else {
        const dim3 grid(rows, a.Hq, plan.splits);
        e = dt == PKV_F32    ? launch_simt<float>(a, kp, grid, stream)
            : dt == PKV_BF16 ? launch_simt<__nv_bfloat16>(a, kp, grid, stream)
                             : launch_simt<uint8_t>(a, kp, grid, stream);
        if (e != cudaSuccess || plan.splits == 1) return e;
    }
    return launch_merge(kp, a.d, a.bs, static_cast<unsigned>(rows * a.Hq), stream);
}

}  // namespace pkv
