// decode_fp8.cu -- paged decode attention over an FP8 (E4M3) cache with one fp32 scale
// per cached row (token slot x KV head): the cached value is code * scale.
//
// What is computed is the decode attention of decode.cu over those values (limoncc.com
// "大语言模型研究15——注意力机制优化之KV缓存" §3.1, §3.3; online softmax, plumephp.com
// "KV Cache 优化与注意力机制加速" §2.2-§2.3); the low-bit cache is the trade-off of
// zwjcode.cn "KV Cache 的增量解码" §14 (half the bytes of bf16).  The scales factor out
// of the products: s_t = scale * k_scale[t] * (q . codes_t) and
// o = sum_t (p_t * v_scale[t]) codes_t / sum_t p_t, so the tensor cores see the codes,
// which are exact in f16, and the fp32 query and weights enter as f16 hi + lo pairs
// (about 2^-22 relative).
//
// decode_fp8_kernel (d = 128, bs 16 or 32, up to 8 query heads per KV head): the block
// layout of decode_chunked_kernel -- one CTA per (sequence, KV head, chunk of blocks),
// four warps taking the chunk's blocks in turn, each with a private TMA ring (up to four
// blocks per SM: the MMA chains are short and need the warps to hide their latency); a stage
// holds a block's K and V codes (128-byte rows, 128-byte swizzle) and its two rows of
// scales.  Per block and warp, with m16n8k16 f16 MMAs:
//   scores S^T (16 rows: the heads' hi and lo query parts; 8 keys per tile): the
//     head dimension is taken in a permuted order so that lane (g, t4) reads the 32
//     contiguous code bytes 32*t4 .. 32*t4+31 of key g -- k-step kk covers dimensions
//     32*t4 + 4*kk + {0..3} -- and the query is loaded in the same order;
//   output O^T = V^T P^T: V^T is the A operand (16 dimensions x 16 keys), read as four
//     16-byte rows per lane and paired across keys with byte permutes; P^T is the B
//     operand, which is exactly the softmax weights the lane already holds for its head.
#include <cuda_fp16.h>

#include "common.cuh"
#include "decode_epilogue.cuh"
#include "decode_kparams.cuh"
#include "fp8_codes.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr unsigned kFullMask = 0xffffffffu;

// Four E4M3 codes (byte i = code i) to two f16x2: lo = codes 0, 1; hi = codes 2, 3 (exact).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(four));
}

// x ~= hi + lo with hi = rn_f16(x), lo = rn_f16(x - hi); the low half holds x0.
__device__ __forceinline__ void split_f16x2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(x0, x1);
    const __half2 l = __floats2half2_rn(x0 - __low2float(h), x1 - __high2float(h));
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// D = A(16x16, f16, row) * B(16x8, f16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int BS, int ST>
struct Fp8Cfg {
    static constexpr int D = 128, NW = 4;
    static constexpr int NT = BS / 8;              // 8-key score tiles per block
    static constexpr int KT = BS / 16;             // 16-key steps of P.V per block
    static constexpr int kPageBytes = BS * D;      // the codes of one K or V block
    static constexpr int kStageBytes = 2 * kPageBytes;          // K codes, then V codes
    static constexpr int kScaleBytes = 2 * BS * 4;               // K scales, then V scales
    static constexpr int kStagesBytes = NW * ST * kStageBytes;
    static constexpr int kScalesOff = kStagesBytes;
    static constexpr int kBarOff = kScalesOff + NW * ST * kScaleBytes;
    static constexpr int kMergeBytes = NW * (16 + 8 * D) * 4;
    static constexpr int kSmemBytes = 1024 + kBarOff + NW * ST * 8;
    static_assert(kMergeBytes <= kStagesBytes, "merge scratch reuses the stage buffers");
};

// The step's new token into the FP8 cache (pkv_decode_step_fp8 with the append inside this
// launch): warp 0 quantises and writes the K row of KV head kvh, warp 1 the V row, from
// k_new / v_new [B][Hkv][128] (bf16) into the slot of position len - 1, with the codes and
// the scale that kv_append_fp8 writes for the same row.  A slot that is not that
// position's is flagged (once, by warp 0) and not written.  The caller fences the writes
// for the asynchronous proxy and syncs the block before the page's copies.
template <int BS>
__device__ __forceinline__ void write_new_token_fp8(const DecodeKParams &p, int b, int kvh, int len, int warp,
                                                    int lane) {
    constexpr int D = 128, J = D / 32;
    const long long slot = __ldg(p.new_slots + b);
    if (slot < 0) return;                                  // no new token this step
    const int pos = len - 1;
    const int phys = pos >= 0 ? __ldg(p.block_table + static_cast<size_t>(b) * p.MBS + pos / BS) : -1;
    if (phys < 0 || phys >= p.NB || slot != static_cast<long long>(phys) * BS + pos % BS) {
        if (warp == 0 && lane == 0) raise_error(p.err, PKV_DEVERR_SLOT);
        return;
    }
    const bool is_v = warp == 1;
    const __nv_bfloat16 *src =
        static_cast<const __nv_bfloat16 *>(is_v ? p.v_new : p.k_new) + (static_cast<size_t>(b) * p.Hkv + kvh) * D;
    float x[J];
#pragma unroll
    for (int j = 0; j < J; ++j) x[j] = __bfloat162float(src[lane + 32 * j]);
    uint8_t code[J];
    const float scale = e4m3_quantise_row<J>(x, code);
    const size_t row = (static_cast<size_t>(phys) * p.Hkv + kvh) * BS + pos % BS;
    uint8_t *dst = static_cast<uint8_t *>(is_v ? p.v_cache_w : p.k_cache_w) + row * D;
#pragma unroll
    for (int j = 0; j < J; ++j) dst[lane + 32 * j] = code[j];
    if (lane == 0) (is_v ? p.v_scale_w : p.k_scale_w)[row] = scale;
}

template <int BS, int ST>
__global__ void __launch_bounds__(128, 4)
    decode_fp8_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const DecodeKParams p) {
    using Cfg = Fp8Cfg<BS, ST>;
    constexpr int D = Cfg::D, NW = Cfg::NW, NT = Cfg::NT, KT = Cfg::KT;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kBarOff);

    pdl_launch_dependents();   // a merge kernel after this one waits for the whole grid
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int tile = blockIdx.x % p.head_tiles;
    const int split = blockIdx.x / p.head_tiles;
    const int kvh = blockIdx.y;
    const int b = blockIdx.z;
    const int head0 = kvh * p.m + tile * 8;
    const int nheads = min(8, (kvh + 1) * p.m - head0);

    const SeqSpan sp = seq_span(p, b, BS, threadIdx.x == 0 && split == 0 && kvh == 0 && tile == 0);
    const int len = sp.len;
    const int n_pages = sp.npages;
    const int pg0 = split * p.chunk_pages;   // pages relative to sp.pfirst
    const int pg1 = min(n_pages, pg0 + p.chunk_pages);
    if (pg0 >= pg1) {
        if (split == 0) {   // an empty sequence: out = 0, lse = -inf
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
        // the step's new token: the block that reads the sequence's last page writes its K
        // and V rows there (codes and scales) before any copy of the page
        if (warp < 2) {
            write_new_token_fp8<BS>(p, b, kvh, len, warp, lane);
            fence_proxy_async_global();
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

    // query fragments: k-step kk covers dimensions d0 = 32*t4 + 4*kk .. d0+3; rows g (hi)
    // and g+8 (lo) of head head0 + g
    uint32_t qa[8][4];
    {
        const bool row_ok = g < nheads;
        const float *qrow = p.q + (static_cast<size_t>(b) * p.Hq + head0 + (row_ok ? g : 0)) * D + 32 * t4;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            float2 x0 = make_float2(0.f, 0.f), x1 = x0;
            if (row_ok) {
                x0 = *reinterpret_cast<const float2 *>(qrow + 4 * kk);
                x1 = *reinterpret_cast<const float2 *>(qrow + 4 * kk + 2);
            }
            split_f16x2(x0.x, x0.y, qa[kk][0], qa[kk][1]);
            split_f16x2(x1.x, x1.y, qa[kk][2], qa[kk][3]);
        }
    }

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
        const int phys = __shfl_sync(kFullMask, tcur, k & 31);
        if (lane == 0) {
            int row, srow;
            if (phys < 0 || phys >= p.NB) {
                raise_error(p.err, PKV_DEVERR_BLOCK);
                row = oob_row;
                srow = 0;            // any valid scales: the codes read as zeros
            } else {
                row = (phys * p.Hkv + kvh) * BS;
                srow = row;
            }
            const int st = warp * ST + k % ST;
            const uint32_t bar = smem_addr(&bars[st]);
            const uint32_t dst = smem_addr(smem + static_cast<size_t>(st) * Cfg::kStageBytes);
            const uint32_t sdst = smem_addr(smem + Cfg::kScalesOff + static_cast<size_t>(st) * Cfg::kScaleBytes);
            mbar_arrive_expect_tx(bar, Cfg::kStageBytes + Cfg::kScaleBytes);
            tma_load_2d(dst, &tm_k, 0, row, bar);
            tma_load_2d(dst + Cfg::kPageBytes, &tm_v, 0, row, bar);
            bulk_load(sdst, p.k_scale + srow, BS * 4, bar);
            bulk_load(sdst + BS * 4, p.v_scale + srow, BS * 4, bar);
        }
    };

    // this lane's state: running max and sum of head g (base 2); O^T accumulators for
    // heads 2*t4 and 2*t4+1 at dimensions 16*g + 2*mt (+1)
    float oT[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) oT[mt][0] = oT[mt][1] = oT[mt][2] = oT[mt][3] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;

    int issued = min(ST, n_my);
    for (int k = 0; k < issued; ++k) issue(k);

    int k = 0;
    for (; k < n_my; ++k) {
        const int st = warp * ST + k % ST;
        const bool arrived = mbar_wait_bounded(smem_addr(&bars[st]), (k / ST) & 1);
        if (!__all_sync(kFullMask, arrived)) {
            if (lane == 0) raise_error(p.err, PKV_DEVERR_TIMEOUT);
            break;
        }
        const int pg = sp.pfirst + pg0 + warp + k * NW;
        const int first = max(0, sp.lo - pg * BS), valid = min(BS, len - pg * BS);
        uint8_t *kpage = smem + static_cast<size_t>(st) * Cfg::kStageBytes;
        uint8_t *vpage = kpage + Cfg::kPageBytes;
        const float *ksc = reinterpret_cast<const float *>(smem + Cfg::kScalesOff + static_cast<size_t>(st) * Cfg::kScaleBytes);
        const float *vsc = ksc + BS;
        if (valid < BS) {
            // codes past the end of the sequence may be anything (an E4M3 NaN among
            // them): zero those V rows so that their zero weights contribute zero
            for (int idx = lane; idx < (BS - valid) * 8; idx += 32)
                *reinterpret_cast<uint4 *>(vpage + (valid + idx / 8) * 128 + (idx % 8) * 16) = make_uint4(0, 0, 0, 0);
            __syncwarp();
        }

        // ---- scores of head g (rows g: hi, g+8: lo) for keys 8*nt + 2*t4 + {0, 1}; the
        // k-steps of a tile accumulate in two halves (independent MMA chains)
        float s[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float s2[4] = {0.f, 0.f, 0.f, 0.f};
            s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
            const int row = nt * 8 + g;
            const uint8_t *krow = kpage + row * 128;
            const uint4 c0 = *reinterpret_cast<const uint4 *>(krow + (((2 * t4) ^ (row & 7)) << 4));
            const uint4 c1 = *reinterpret_cast<const uint4 *>(krow + (((2 * t4 + 1) ^ (row & 7)) << 4));
            const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
            for (int kk = 0; kk < 8; kk += 2) {
                uint32_t b0, b1, b2, b3;
                e4m3x4_to_f16x2x2(w[kk], b0, b1);
                e4m3x4_to_f16x2x2(w[kk + 1], b2, b3);
                mma_f16_16816(s[nt], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                mma_f16_16816(s2, qa[kk + 1][0], qa[kk + 1][1], qa[kk + 1][2], qa[kk + 1][3], b2, b3);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) s[nt][e] += s2[e];
        }

        // ---- online softmax (base 2) of head g
        float sc[NT][2];
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int tok = nt * 8 + 2 * t4 + e;
                const bool vis = tok >= first && tok < valid;
                sc[nt][e] = vis ? (s[nt][e] + s[nt][2 + e]) * (ksc[tok] * p.scale_log2) : -INFINITY;
                mx = fmaxf(mx, sc[nt][e]);
            }
        }
        mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 2));
        const float m_new = fmaxf(m_run, mx);   // finite: every block holds a visible key
        const float alpha = ex2_approx(m_run - m_new);
        float psum = 0.f;
        float pv[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int tok = nt * 8 + 2 * t4 + e;
                const float w = ex2_approx(sc[nt][e] - m_new);
                psum += w;
                pv[nt][e] = tok >= first && tok < valid ? w * vsc[tok] : 0.f;
            }
        }
        l_run = l_run * alpha + psum;
        m_run = m_new;
        // rescale O^T when a running max moved: its heads are 2*t4 and 2*t4+1, whose
        // states live in lanes 8*t4 + x
        if (__any_sync(kFullMask, alpha != 1.f)) {
            const float alpha_a = __shfl_sync(kFullMask, alpha, 8 * t4);
            const float alpha_b = __shfl_sync(kFullMask, alpha, 8 * t4 + 4);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                oT[mt][0] *= alpha_a;
                oT[mt][1] *= alpha_b;
                oT[mt][2] *= alpha_a;
                oT[mt][3] *= alpha_b;
            }
        }

        // ---- O^T += V^T P^T, 16 keys per step
#pragma unroll
        for (int kt = 0; kt < KT; ++kt) {
            uint32_t bh0, bl0, bh1, bl1;
            split_f16x2(pv[2 * kt][0], pv[2 * kt][1], bh0, bl0);
            split_f16x2(pv[2 * kt + 1][0], pv[2 * kt + 1][1], bh1, bl1);
            const int r0 = kt * 16 + 2 * t4;
            uint4 R[4];
            const int rows[4] = {r0, r0 + 1, r0 + 8, r0 + 9};
#pragma unroll
            for (int i = 0; i < 4; ++i)
                R[i] = *reinterpret_cast<const uint4 *>(vpage + rows[i] * 128 + ((g ^ (rows[i] & 7)) << 4));
            const uint32_t w0[4] = {R[0].x, R[0].y, R[0].z, R[0].w}, w1[4] = {R[1].x, R[1].y, R[1].z, R[1].w};
            const uint32_t w2[4] = {R[2].x, R[2].y, R[2].z, R[2].w}, w3[4] = {R[3].x, R[3].y, R[3].z, R[3].w};
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                // bytes 2*mt and 2*mt+1 of each row: dimensions 16g + 2mt (+1)
                const int wi = mt >> 1, bi = 2 * (mt & 1);
                const uint32_t sel = bi | ((4 + bi) << 4) | ((bi + 1) << 8) | ((5 + bi) << 12);
                uint32_t a0, a1, a2, a3;
                e4m3x4_to_f16x2x2(__byte_perm(w0[wi], w1[wi], sel), a0, a1);
                e4m3x4_to_f16x2x2(__byte_perm(w2[wi], w3[wi], sel), a2, a3);
                mma_f16_16816(oT[mt], a0, a1, a2, a3, bh0, bh1);
                mma_f16_16816(oT[mt], a0, a1, a2, a3, bl0, bl1);
            }
        }
        __syncwarp();
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

    l_run += __shfl_xor_sync(kFullMask, l_run, 1);
    l_run += __shfl_xor_sync(kFullMask, l_run, 2);

    // ---- the warps' (m, l, O) through shared memory (stage buffers are free now)
    __syncthreads();
    float *mw = reinterpret_cast<float *>(smem);
    float *lw = mw + NW * 8;
    float *ow = lw + NW * 8;
    if (t4 == 0) {
        mw[warp * 8 + g] = m_run;
        lw[warp * 8 + g] = l_run;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const int dcol = 16 * g + 2 * mt;
        *reinterpret_cast<float2 *>(ow + (warp * 8 + 2 * t4) * D + dcol) = make_float2(oT[mt][0], oT[mt][2]);
        *reinterpret_cast<float2 *>(ow + (warp * 8 + 2 * t4 + 1) * D + dcol) = make_float2(oT[mt][1], oT[mt][3]);
    }
    __syncthreads();
    finish_chunk<D, NW>(smem, p, b, kvh, tile, head0, nheads, split, (n_pages + p.chunk_pages - 1) / p.chunk_pages);
}

template <int BS, int ST>
cudaError_t launch_fp8(const DecodeKParams &kp, const CUtensorMap &tk, const CUtensorMap &tv, dim3 grid,
                       cudaStream_t stream) {
    using Cfg = Fp8Cfg<BS, ST>;
    auto kernel = decode_fp8_kernel<BS, ST>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    kernel<<<grid, Cfg::NW * 32, Cfg::kSmemBytes, stream>>>(tk, tv, kp);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_fp8(const DecodeKParams &kp, const CUtensorMap &tk, const CUtensorMap &tv, int bs,
                              dim3 grid, cudaStream_t stream) {
    // 12 KB (bs 16) or 16 KB (bs 32) of copies in flight per warp; four (three) blocks per SM
    return bs == 16 ? launch_fp8<16, 3>(kp, tk, tv, grid, stream) : launch_fp8<32, 2>(kp, tk, tv, grid, stream);
}

}  // namespace pkv
