// E4M3 row quantisation shared by every kernel that writes an FP8 cache row (kv_append_fp8
// and the decode step that writes its new token inside the attention launch), so that one
// row gets the same codes and scale whichever kernel writes it.
//
// The low-bit cache trade-off of zwjcode.cn "KV Cache 的增量解码" §14, as this library stores
// it: a cached value is an E4M3 code times an fp32 scale, one scale per row (token slot x
// KV head), chosen so that the row's largest magnitude maps to E4M3's largest finite
// value, 448.
#pragma once

#include <cuda_fp8.h>
#include <cstdint>

namespace pkv {

// One row held by a whole warp, lane owning elements lane + 32*j (elements past the row's end
// passed as 0).  Returns scale = amax / 448 and sets code[j] = E4M3(x[j] / scale) (IEEE fp32
// division, round to nearest even, saturating at +-448); a row of zeros gets scale 0 and
// codes 0.  All 32 lanes must call it together.
template <int J>
__device__ __forceinline__ float e4m3_quantise_row(const float (&x)[J], uint8_t (&code)[J]) {
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < J; ++j) amax = fmaxf(amax, fabsf(x[j]));
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, sh));
    const float scale = amax / 448.f;
#pragma unroll
    for (int j = 0; j < J; ++j)
        code[j] = amax > 0.f ? static_cast<uint8_t>(__nv_cvt_float_to_fp8(x[j] / scale, __NV_SATFINITE, __NV_E4M3))
                             : uint8_t{0};
    return scale;
}

}  // namespace pkv
