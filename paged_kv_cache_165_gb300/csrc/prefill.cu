// prefill.cu -- varlen causal attention over packed prompts (cu_seqlens).
//
// Sequence b owns tokens [cu_seqlens[b], cu_seqlens[b+1]) of q/k/v (0539edu.com
// "从KV cache共享到批量调度…" §3.3).  Token t of a sequence attends to tokens 0..t of
// the same sequence (causal prefill, zwjcode.cn "KV Cache 的增量解码" §05; the mask is
// aligned so that a query at position t sees keys 0..t, §13), with query head i reading
// KV head floor(i/m) (limoncc.com "大语言模型研究15——注意力机制优化之KV缓存" §3.3).
//
// Tensor-core path (bf16, d in {64, 128}): one CTA of 4 warps per (64-query tile, query
// head, sequence).  TMA brings the Q tile once and 64-key K/V tiles through a two-stage
// ring (128-byte swizzle, mbarrier completion with a bounded wait).  Each warp owns 16
// query rows: S = Q K^T on m16n8k16 bf16 MMAs, an online softmax per row (running max
// and sum, plumephp.com "KV Cache 优化与注意力机制加速" §2.2-§2.3), and O += P V with
// P split into bf16 hi + lo parts (two MMAs) so the weights keep ~16 bits.  Only key
// tiles at or below the diagonal are visited.
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

// ============================================================ tensor-core path

template <int D>
struct PrefillCfg {
    static constexpr int kBM = 64, kBN = 64;
    static constexpr int kTileBytes = 64 * D * 2;
    static constexpr int kSmemBytes = 1024 + 5 * kTileBytes + 3 * 8;   // Q + 2 x (K, V) + bars
};

template <int D>
__global__ void __launch_bounds__(128)
    prefill_mma_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const PrefillKParams p) {
    using Cfg = PrefillCfg<D>;
    constexpr int BN = Cfg::kBN, BM = Cfg::kBM, TB = Cfg::kTileBytes;
    constexpr int KS = D / 16, ONT = D / 8, PANELS = D / 64;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *q_s = smem;                       // Q tile
    uint8_t *kv_s = smem + TB;                 // stage s: K at kv_s + 2*s*TB, V at + TB
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 5 * TB);   // [0] Q, [1..2] K/V stages

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int qt = blockIdx.x, i = blockIdx.y, b = blockIdx.z;
    const int kvh = i / p.m;
    int start = 0, len = 0;
    if (!seq_range(p, b, start, len, threadIdx.x == 0 && qt == 0 && i == 0)) return;
    const int q0 = qt * BM;
    if (q0 >= len) return;
    const int n_kt = (min(q0 + BM, len) - 1) / BN + 1;   // key tiles at or below the diagonal

    if (threadIdx.x == 0) {
        for (int s = 0; s < 3; ++s) mbar_init(smem_addr(&bars[s]), 1);
        fence_barrier_init();
    }
    __syncthreads();

    auto issue_kv = [&](int kt) {   // thread 0 only
        const int s = kt & 1;
        const uint32_t bar = smem_addr(&bars[1 + s]);
        const uint32_t dk = smem_addr(kv_s + 2 * s * TB), dv = dk + TB;
        mbar_arrive_expect_tx(bar, 2 * TB);
#pragma unroll
        for (int pn = 0; pn < PANELS; ++pn) {
            tma_load_3d(dk + pn * BN * 128, &tm_k, pn * 64, kvh, start + kt * BN, bar);
            tma_load_3d(dv + pn * BN * 128, &tm_v, pn * 64, kvh, start + kt * BN, bar);
        }
    };
    if (threadIdx.x == 0) {
        const uint32_t bar = smem_addr(&bars[0]);
        mbar_arrive_expect_tx(bar, TB);
#pragma unroll
        for (int pn = 0; pn < PANELS; ++pn)
            tma_load_3d(smem_addr(q_s) + pn * BM * 128, &tm_q, pn * 64, i, start + q0, bar);
        issue_kv(0);
        if (n_kt > 1) issue_kv(1);
    }

    bool ok = __syncthreads_and(mbar_wait_bounded(smem_addr(&bars[0]), 0)) != 0;
    uint32_t qa[KS][4];
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
        const int mi = lane >> 3, r8 = lane & 7;
        ldsm_x4(smem_addr(q_s) + swz128(BM, warp * 16 + (mi & 1) * 8 + r8, kk * 16 + (mi >> 1) * 8),
                qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
    }

    const int row0 = q0 + warp * 16 + g;   // this thread's rows: row0 and row0 + 8
    float o[ONT][4];
#pragma unroll
    for (int nt = 0; nt < ONT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    int kt = 0;
    for (; kt < n_kt && ok; ++kt) {
        const int s = kt & 1;
        const bool arrived = mbar_wait_bounded(smem_addr(&bars[1 + s]), (kt >> 1) & 1);
        if (!__syncthreads_and(arrived)) {
            ok = false;
            break;
        }
        uint8_t *k_tile = kv_s + 2 * s * TB;
        uint8_t *v_tile = k_tile + TB;
        const int key0 = kt * BN;
        if (key0 + BN > len) {
            // V rows past the sequence end hold other sequences' data or TMA's zero fill;
            // zero them so that their zero weights contribute exactly zero.
            const int valid = len - key0;
            for (int idx = threadIdx.x; idx < (BN - valid) * (D / 8); idx += 128) {
                const int r = valid + idx / (D / 8), c16 = idx % (D / 8);
                *reinterpret_cast<uint4 *>(v_tile + (c16 >> 3) * BN * 128 + r * 128 +
                                           (c16 & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncthreads();
        }
        const uint32_t k_a = smem_addr(k_tile), v_a = smem_addr(v_tile);

        float sacc[BN / 8][4];
#pragma unroll
        for (int nt = 0; nt < BN / 8; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
            for (int np = 0; np < BN / 16; ++np) {
                const int mi = lane >> 3, r8 = lane & 7;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(k_a + swz128(BN, np * 16 + (mi >> 1) * 8 + r8, kk * 16 + (mi & 1) * 8), b0,
                        b1, b2, b3);
                mma_bf16_16816(sacc[2 * np], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                mma_bf16_16816(sacc[2 * np + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
            }
        }

        // online softmax per row (base 2): rows row0 (c0, c1) and row0 + 8 (c2, c3)
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < BN / 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = key0 + nt * 8 + 2 * t4 + (e & 1);
                const int row = row0 + (e >> 1) * 8;
                const float v = sacc[nt][e] * p.scale_log2;
                sacc[nt][e] = key <= row ? v : -INFINITY;
                mx[e >> 1] = fmaxf(mx[e >> 1], sacc[nt][e]);
            }
        }
        float alpha[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(kFull, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(kFull, mx[r], 2));
            const float m_new = fmaxf(m_run[r], mx[r]);
            // a row can only be fully masked in a tile after it already saw key 0
            alpha[r] = m_new == -INFINITY ? 1.f : exp2f(m_run[r] - m_new);
            m_run[r] = m_new;
        }
        float psum[2] = {0.f, 0.f};
#pragma unroll
        for (int nt = 0; nt < BN / 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float mr = m_run[e >> 1];
                sacc[nt][e] = mr == -INFINITY ? 0.f : exp2f(sacc[nt][e] - mr);
                psum[e >> 1] += sacc[nt][e];
            }
        }
        l_run[0] = l_run[0] * alpha[0] + psum[0];
        l_run[1] = l_run[1] * alpha[1] + psum[1];
#pragma unroll
        for (int nt = 0; nt < ONT; ++nt) {
            o[nt][0] *= alpha[0];
            o[nt][1] *= alpha[0];
            o[nt][2] *= alpha[1];
            o[nt][3] *= alpha[1];
        }

        // O += (P_hi + P_lo) V
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
            uint32_t h0, l0, h1, l1, h2, l2, h3, l3;
            split_bf16x2(sacc[2 * ks][0], sacc[2 * ks][1], h0, l0);          // row g, keys 2t..
            split_bf16x2(sacc[2 * ks][2], sacc[2 * ks][3], h1, l1);          // row g+8
            split_bf16x2(sacc[2 * ks + 1][0], sacc[2 * ks + 1][1], h2, l2);  // row g, keys 2t+8..
            split_bf16x2(sacc[2 * ks + 1][2], sacc[2 * ks + 1][3], h3, l3);  // row g+8
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
                const int mi = lane >> 3, r8 = lane & 7;
                uint32_t b0, b1, b2, b3;
                ldsm_x4_trans(v_a + swz128(BN, ks * 16 + (mi & 1) * 8 + r8, np * 16 + (mi >> 1) * 8),
                              b0, b1, b2, b3);
                mma_bf16_16816(o[2 * np], h0, h1, h2, h3, b0, b1);
                mma_bf16_16816(o[2 * np], l0, l1, l2, l3, b0, b1);
                mma_bf16_16816(o[2 * np + 1], h0, h1, h2, h3, b2, b3);
                mma_bf16_16816(o[2 * np + 1], l0, l1, l2, l3, b2, b3);
            }
        }
        __syncthreads();   // every warp is done with this stage
        if (threadIdx.x == 0 && kt + 2 < n_kt) issue_kv(kt + 2);
    }
    if (!ok) {
        if (threadIdx.x == 0) {
            raise_error(p.err, PKV_DEVERR_TIMEOUT);
            // let the copies still in flight land before the block exits
            mbar_wait_bounded(smem_addr(&bars[0]), 0);
            for (int k2 = kt; k2 < min(n_kt, kt + 2); ++k2)
                mbar_wait_bounded(smem_addr(&bars[1 + (k2 & 1)]), (k2 >> 1) & 1);
        }
        return;
    }

#pragma unroll
    for (int r = 0; r < 2; ++r) {
        l_run[r] += __shfl_xor_sync(kFull, l_run[r], 1);
        l_run[r] += __shfl_xor_sync(kFull, l_run[r], 2);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int row = row0 + r * 8;
        if (row >= len) continue;
        const size_t tok = static_cast<size_t>(start + row);
        float *dst = p.out + (tok * p.Hq + i) * D;
        const float inv = 1.f / l_run[r];
#pragma unroll
        for (int nt = 0; nt < ONT; ++nt)
            *reinterpret_cast<float2 *>(dst + nt * 8 + 2 * t4) =
                make_float2(o[nt][2 * r] * inv, o[nt][2 * r + 1] * inv);
        if (t4 == 0 && p.lse != nullptr) p.lse[tok * p.Hq + i] = (m_run[r] + log2f(l_run[r])) * kLn2;
    }
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
cudaError_t launch_prefill_mma(const PrefillArgs &a, const PrefillKParams &kp,
                               cudaStream_t stream) {
    using Cfg = PrefillCfg<D>;
    CUtensorMap tq, tk, tv;
    const uint64_t dq[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.Hq),
                            static_cast<uint64_t>(a.T)};
    const uint64_t sq[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(a.Hq) * D * 2};
    const uint64_t dk[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.Hkv),
                            static_cast<uint64_t>(a.T)};
    const uint64_t sk[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(a.Hkv) * D * 2};
    const uint32_t box[3] = {64, 1, 64};
    if (!encode_map_bf16(&tq, a.q, 3, dq, sq, box) || !encode_map_bf16(&tk, a.k, 3, dk, sk, box) ||
        !encode_map_bf16(&tv, a.v, 3, dk, sk, box))
        return cudaErrorInvalidValue;
    auto kernel = prefill_mma_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    const dim3 grid((a.max_seqlen + Cfg::kBM - 1) / Cfg::kBM, a.Hq, a.B);
    kernel<<<grid, 128, Cfg::kSmemBytes, stream>>>(tq, tk, tv, kp);
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
        return a.d == 64 ? launch_prefill_mma<64>(a, kp, stream)
                         : launch_prefill_mma<128>(a, kp, stream);
    return dt == PKV_F32 ? launch_prefill_simt<float>(a, kp, stream)
                         : launch_prefill_simt<__nv_bfloat16>(a, kp, stream);
}

}  // namespace pkv
