// cache_ops.cu -- writes into the paged KV cache: token scatter and whole-block copy.
//
// kv_append: each new token's K and V rows go to the slot slot_mapping[t] names
//   (limoncc.com "大语言模型研究15——注意力机制优化之KV缓存" §2: compute only the new
//   token's K/V and add it to the cache; zwjcode.cn "KV Cache 的增量解码" §10: write a
//   preallocated slot instead of re-concatenating the cache).
// kv_block_copy: copy-on-write duplicates a whole physical block before a sequence
//   writes into a block it shares (plumephp.com "KV Cache 优化与注意力机制加速" §4.3;
//   0539edu.com "从KV cache共享到批量调度…" §3.2).
//
// Both are pure byte copies, so they move the widest unit (16, 8, 4 or 2 bytes) that
// divides the row (or block) size and the pointers, in a grid-stride loop sized to
// the SM count.  Both are HBM-bound and tiny next to the attention read.
// kv_append_fp8: the same scatter into an FP8 (E4M3) cache with one fp32 scale per row
//   (token slot x KV head): scale = amax(row) / 448, code = E4M3(x / scale) rounded to
//   nearest even and saturated (both divisions in fp32); a row of zeros stores scale 0
//   and codes 0.  The low-bit cache is the trade-off of zwjcode.cn "KV Cache 的增量解码"
//   §14.  One warp per row.
#include <algorithm>
#include <initializer_list>

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "fp8_codes.cuh"
#include "internal.h"

namespace pkv {
namespace {

// One unit = `U` bytes. row_units units per (token, head) row.
template <typename U>
__global__ void __launch_bounds__(256)
    kv_append_kernel(const U *__restrict__ k_new, const U *__restrict__ v_new, U *__restrict__ kc,
                     U *__restrict__ vc, const int64_t *__restrict__ slots, int T, int Hkv,
                     int row_units, int bs, long long n_slots, unsigned *err) {
    const long long total = static_cast<long long>(T) * Hkv * row_units;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int u = static_cast<int>(idx % row_units);
        const long long th = idx / row_units;           // t * Hkv + h
        const int h = static_cast<int>(th % Hkv);
        const int t = static_cast<int>(th / Hkv);
        const long long slot = __ldg(slots + t);
        if (slot < 0) continue;                          // padding token
        if (slot >= n_slots) {
            if (h == 0 && u == 0) raise_error(err, PKV_DEVERR_SLOT);
            continue;
        }
        const long long dst = (((slot / bs) * Hkv + h) * bs + slot % bs) * row_units + u;
        kc[dst] = k_new[idx];
        vc[dst] = v_new[idx];
    }
}

template <typename U>
__global__ void __launch_bounds__(256)
    kv_block_copy_kernel(U *__restrict__ kc, U *__restrict__ vc, const int32_t *__restrict__ pairs,
                         int n, long long block_units, int NB, unsigned *err) {
    for (int pair = blockIdx.y; pair < n; pair += gridDim.y) {
        const int src = __ldg(pairs + 2 * pair), dst = __ldg(pairs + 2 * pair + 1);
        if (src < 0 || src >= NB || dst < 0 || dst >= NB) {
            if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(err, PKV_DEVERR_PAIR);
            continue;
        }
        const U *ks = kc + src * block_units;
        const U *vs = vc + src * block_units;
        U *kd = kc + dst * block_units;
        U *vd = vc + dst * block_units;
        for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
             i < block_units; i += static_cast<long long>(gridDim.x) * blockDim.x) {
            kd[i] = ks[i];
            vd[i] = vs[i];
        }
    }
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// Rows r = (t * Hkv + h) * 2 + {0: K, 1: V}, one warp each; lanes own elements lane + 32*j.
template <typename T, int J>
__global__ void __launch_bounds__(256)
    kv_append_fp8_kernel(const T *__restrict__ k_new, const T *__restrict__ v_new, uint8_t *__restrict__ kc,
                         uint8_t *__restrict__ vc, float *__restrict__ ks, float *__restrict__ vs,
                         const int64_t *__restrict__ slots, int T_, int Hkv, int d, int bs, long long n_slots,
                         unsigned *err) {
    const int lane = threadIdx.x & 31;
    const long long rows = static_cast<long long>(T_) * Hkv * 2;
    for (long long r = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5; r < rows;
         r += (static_cast<long long>(gridDim.x) * blockDim.x) >> 5) {
        const bool is_v = r & 1;
        const long long th = r >> 1;                     // t * Hkv + h
        const int h = static_cast<int>(th % Hkv);
        const int t = static_cast<int>(th / Hkv);
        const long long slot = __ldg(slots + t);
        if (slot < 0) continue;                          // padding token
        if (slot >= n_slots) {
            if (h == 0 && !is_v && lane == 0) raise_error(err, PKV_DEVERR_SLOT);
            continue;
        }
        const T *src = (is_v ? v_new : k_new) + th * d;
        float x[J];
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int e = lane + 32 * j;
            x[j] = e < d ? to_f32(src[e]) : 0.f;
        }
        uint8_t code[J];
        const float scale = e4m3_quantise_row<J>(x, code);
        const long long row = ((slot / bs) * Hkv + h) * bs + slot % bs;
        uint8_t *dst = (is_v ? vc : kc) + row * d;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int e = lane + 32 * j;
            if (e < d) dst[e] = code[j];
        }
        if (lane == 0) (is_v ? vs : ks)[row] = scale;
    }
}

int unit_bytes(size_t row_bytes, std::initializer_list<const void *> ptrs) {
    for (int u : {16, 8, 4, 2}) {
        bool ok = row_bytes % u == 0;
        for (const void *p : ptrs) ok = ok && (reinterpret_cast<uintptr_t>(p) % u == 0);
        if (ok) return u;
    }
    return 1;
}

int sm_count_current() {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

}  // namespace

cudaError_t launch_kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                             int elem_bytes, const int64_t *slot_mapping, int T, int Hkv, int d,
                             int bs, int NB, unsigned *err, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const size_t row_bytes = static_cast<size_t>(d) * elem_bytes;
    const int u = unit_bytes(row_bytes, {k_new, v_new, k_cache, v_cache});
    const int row_units = static_cast<int>(row_bytes / u);
    const long long total = static_cast<long long>(T) * Hkv * row_units;
    const long long want = (total + 255) / 256;
    const int grid = static_cast<int>(std::min<long long>(want, 8ll * sm_count_current()));
    const long long n_slots = static_cast<long long>(NB) * bs;
#define PKV_APPEND(UT)                                                                        \
    kv_append_kernel<UT><<<grid, 256, 0, stream>>>(                                           \
        static_cast<const UT *>(k_new), static_cast<const UT *>(v_new), static_cast<UT *>(k_cache), \
        static_cast<UT *>(v_cache), slot_mapping, T, Hkv, row_units, bs, n_slots, err)
    switch (u) {
        case 16: PKV_APPEND(uint4); break;
        case 8: PKV_APPEND(uint2); break;
        case 4: PKV_APPEND(uint32_t); break;
        case 2: PKV_APPEND(uint16_t); break;
        default: PKV_APPEND(uint8_t); break;
    }
#undef PKV_APPEND
    return cudaGetLastError();
}

cudaError_t launch_kv_append_fp8(const void *k_new, const void *v_new, pkv_dtype new_dt, uint8_t *k_codes,
                                 uint8_t *v_codes, float *k_scale, float *v_scale,
                                 const int64_t *slot_mapping, int T, int Hkv, int d, int bs, int NB,
                                 unsigned *err, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const long long rows = static_cast<long long>(T) * Hkv * 2;
    const int grid = static_cast<int>(std::min<long long>((rows + 7) / 8, 8ll * sm_count_current()));
    const long long n_slots = static_cast<long long>(NB) * bs;
    const int J = (d + 31) / 32;
#define PKV_FP8(TT, JJ)                                                                              \
    kv_append_fp8_kernel<TT, JJ><<<grid, 256, 0, stream>>>(                                         \
        static_cast<const TT *>(k_new), static_cast<const TT *>(v_new), k_codes, v_codes, k_scale, \
        v_scale, slot_mapping, T, Hkv, d, bs, n_slots, err)
#define PKV_FP8_J(TT)                   \
    switch (J) {                        \
        case 1: PKV_FP8(TT, 1); break;  \
        case 2: PKV_FP8(TT, 2); break;  \
        case 3: PKV_FP8(TT, 3); break;  \
        case 4: PKV_FP8(TT, 4); break;  \
        case 5: PKV_FP8(TT, 5); break;  \
        case 6: PKV_FP8(TT, 6); break;  \
        case 7: PKV_FP8(TT, 7); break;  \
        case 8: PKV_FP8(TT, 8); break;  \
        default: return cudaErrorInvalidValue; \
    }
    if (new_dt == PKV_BF16) {
        PKV_FP8_J(__nv_bfloat16)
    } else {
        PKV_FP8_J(float)
    }
#undef PKV_FP8_J
#undef PKV_FP8
    return cudaGetLastError();
}

cudaError_t launch_kv_block_copy(void *k_cache, void *v_cache, int elem_bytes,
                                 const int32_t *pairs, int n, int Hkv, int d, int bs, int NB,
                                 unsigned *err, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    const size_t block_bytes = static_cast<size_t>(Hkv) * bs * d * elem_bytes;
    const int u = unit_bytes(block_bytes, {k_cache, v_cache});
    const long long block_units = static_cast<long long>(block_bytes / u);
    const int gx = static_cast<int>(std::min<long long>((block_units + 255) / 256, 16));
    const dim3 grid(gx, std::min(n, 65535));
#define PKV_COPY(UT)                                                                          \
    kv_block_copy_kernel<UT><<<grid, 256, 0, stream>>>(static_cast<UT *>(k_cache),           \
                                                        static_cast<UT *>(v_cache), pairs, n, \
                                                        block_units, NB, err)
    switch (u) {
        case 16: PKV_COPY(uint4); break;
        case 8: PKV_COPY(uint2); break;
        case 4: PKV_COPY(uint32_t); break;
        case 2: PKV_COPY(uint16_t); break;
        default: PKV_COPY(uint8_t); break;
    }
#undef PKV_COPY
    return cudaGetLastError();
}

}  // namespace pkv
