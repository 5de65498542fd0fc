// e4m3.cuh -- exact E4M3FN -> FP16 decode used by the kernels and by the debug export.
//
// Every E4M3FN value (OCP 8-bit floating point: bias 7, 3 mantissa bits, largest finite 448,
// smallest subnormal 2^-9) is exactly representable in FP16 (bias 15, 10 mantissa bits, largest
// 65504, smallest subnormal 2^-24), so the decode is exact. The hardware conversion
// cvt.rn.f16x2.e4m3x2 turns two codes into two FP16 values per instruction; on this GPU it runs
// about three times faster than an integer bit-placement decode (measured), so the kernels use it.
// The NaN codes S.1111.111 decode to FP16 NaN.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace dflash {

// Two codes (byte 0 = first element) -> FP16x2 (low half = first element).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two_codes) {
    uint32_t out;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(two_codes));
    return out;
}

// Four codes packed in a word (code k in bits 8k..8k+7) -> two FP16x2 words:
// lo = (code 0, code 1), hi = (code 2, code 3).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t x, uint32_t& lo, uint32_t& hi) {
    lo = e4m3x2_to_f16x2(static_cast<uint16_t>(x & 0xFFFFu));
    hi = e4m3x2_to_f16x2(static_cast<uint16_t>(x >> 16));
}

// One code -> its exact value as FP32.
__device__ __forceinline__ float e4m3_to_float(uint32_t code) {
    const uint32_t h2 = e4m3x2_to_f16x2(static_cast<uint16_t>(code & 0xFFu));
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

}  // namespace dflash
