// decode_epilogue.cuh -- end of a decode block that holds up to 8 query heads of one KV
// head: the warps' online-softmax states merge, the chunk's result is written, and the
// last chunk of a (sequence, head tile) merges all chunks by log-sum-exp (not part of
// the ABI).
#pragma once

#include "common.cuh"
#include "decode_kparams.cuh"

namespace pkv {

// Shared memory holds, from `smem`, the NW warps' running max and sum per head (base 2,
// [NW][8] each) and their unnormalised outputs [NW][8][D]; the caller has synchronised.
// A sequence with a single chunk writes out / lse directly; otherwise the chunk's
// normalised partial (o_c, lse_c in base 2) goes to the workspace, and when the
// workspace carries arrival counters the block that completes the unit merges
// lse = log2 sum_c 2^{lse_c}, out = sum_c 2^{lse_c - lse} o_c (plumephp.com
// "KV Cache 优化与注意力机制加速" §2.2-§2.3 applied to whole chunks).
template <int D, int NW>
__device__ __forceinline__ void finish_chunk(uint8_t *smem, const DecodeKParams &p, int b, int kvh, int tile,
                                             int head0, int nheads, int split, int nc) {
    constexpr unsigned kFull = 0xffffffffu;
    constexpr float kLn2 = kDecLn2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *mw = reinterpret_cast<float *>(smem);
    float *lw = mw + NW * 8;
    float *ow = lw + NW * 8;
    // A sequence with a single chunk writes its result directly; otherwise this chunk's
    // normalised partial (o_c, lse_c in base 2) goes to the workspace.
    const size_t bi0 = static_cast<size_t>(b) * p.Hq + head0;
    for (int idx = threadIdx.x; idx < nheads * D; idx += NW * 32) {
        const int h = idx / D, c = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, mw[w * 8 + h]);
        float L = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float f = exp2f(mw[w * 8 + h] - M);
            L += lw[w * 8 + h] * f;
            acc += ow[(w * 8 + h) * D + c] * f;
        }
        const size_t bi = bi0 + h;
        if (nc == 1) {
            p.out[bi * D + c] = acc / L;
            if (c == 0 && p.lse != nullptr) p.lse[bi] = (M + log2f(L)) * kLn2;
        } else {
            p.ws_o[(bi * p.splits + split) * D + c] = acc / L;
            if (c == 0) p.ws_lse[bi * p.splits + split] = M + log2f(L);
        }
    }
    if (nc == 1 || p.counters == nullptr) return;

    // ---- the last chunk to finish merges all chunks of this (sequence, head group):
    // partials are published (fence) before the arrival is counted; the CTA that sees
    // the count reach nc resets the counter for the next call and reads them back.
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned *ctr = p.counters + (static_cast<size_t>(b) * p.Hkv + kvh) * p.head_tiles + tile;
        const unsigned prev = atomicAdd(ctr, 1u);
        s_last = prev + 1 == static_cast<unsigned>(nc);
        if (s_last) *ctr = 0u;   // every chunk of this call has arrived
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // per-head chunk weights 2^{lse_c - M} and their sum, in shared memory (stage area)
    float *wts = reinterpret_cast<float *>(smem);              // [8][nc]
    float *inv_l = wts + 8 * nc;                                // [8]
    float *lse_h = inv_l + 8;                                   // [8]
    for (int h = warp; h < nheads; h += NW) {
        const float *ls = p.ws_lse + (bi0 + h) * p.splits;
        float M = -INFINITY;
        for (int c = lane; c < nc; c += 32) M = fmaxf(M, __ldcg(ls + c));
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, sh));
        float L = 0.f;
        for (int c = lane; c < nc; c += 32) {
            const float w = exp2f(__ldcg(ls + c) - M);
            wts[h * nc + c] = w;
            L += w;
        }
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) L += __shfl_xor_sync(kFull, L, sh);
        if (lane == 0) {
            inv_l[h] = 1.f / L;
            lse_h[h] = M + log2f(L);
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < nheads * (D / 4); idx += NW * 32) {
        const int h = idx / (D / 4), c4 = (idx % (D / 4)) * 4;
        const float *po = p.ws_o + (bi0 + h) * p.splits * D + c4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int c = 0; c < nc; ++c) {
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(po + static_cast<size_t>(c) * D));
            const float w = wts[h * nc + c];
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
        const float il = inv_l[h];
        *reinterpret_cast<float4 *>(p.out + (bi0 + h) * D + c4) =
            make_float4(acc.x * il, acc.y * il, acc.z * il, acc.w * il);
        if (c4 == 0 && p.lse != nullptr) p.lse[bi0 + h] = lse_h[h] * kLn2;
    }
}

}  // namespace pkv
