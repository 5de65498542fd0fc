// e4m3.cuh -- exact E4M3FN -> FP16 decode used by every kernel and by the debug export.
//
// E4M3FN (OCP 8-bit floating point) and FP16 share the sign / exponent / mantissa order, so
// moving the code's low seven bits up by seven places puts its 4-bit exponent in the low bits of
// FP16's 5-bit exponent and its 3-bit mantissa in FP16's top mantissa bits. The FP16 number that
// results equals the E4M3 value times 2^-8 exactly, subnormals included (FP16 exponent bias 15
// vs E4M3 bias 7). Callers fold the 2^8 into a scale. The NaN codes S.1111.111 come out as
// +-480 * 2^-8; the encoder that fills a KV cache never produces them.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace dflash {

// Four codes packed in x (code k in bits 8k..8k+7) -> two FP16x2 words, values * 2^-8.
// even holds codes 0 and 2 (low, high half), odd holds codes 1 and 3.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t x, uint32_t& even, uint32_t& odd) {
    odd = ((x & 0x7F007F00u) >> 1) | (x & 0x80008000u);
    const uint32_t xe = x << 8;
    even = ((xe & 0x7F007F00u) >> 1) | (xe & 0x80008000u);
}

// One code -> its exact value as FP32 (through the same bit placement).
__device__ __forceinline__ float e4m3_to_float(uint32_t code) {
    const uint32_t h = ((code & 0x7Fu) << 7) | ((code & 0x80u) << 8);
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h))) * 256.0f;
}

}  // namespace dflash
