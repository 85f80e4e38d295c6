// Power-of-two block scales of the second e4m3 recipe (MOE_FP8_E4M3_POW2).
//
// "7.13 Serving Mixture-of-Experts", DeepEP section (FP8 dispatch: e4m3 payloads with block
// scales) fixes the payload format and the fp32 scales, not the scale values. This recipe
// keeps the 1x128 activation and 128x128 weight blocks and takes each scale as the smallest
// power of two 2^e with amax <= 448 * 2^e, -126 <= e <= 127 (1 for an all-zero block): then
// value / scale is exact, and the tensor core can apply the scale itself (its UE8M0 scale
// bytes hold the biased exponent e + 127).
#pragma once

#include <cstdint>

namespace moe {

// With amax = m * 2^ea, m in [1, 2), and 448 = 1.75 * 2^8: amax <= 448 * 2^e holds for
// e >= ea - 8 when m <= 1.75 (mantissa field at most 0x600000), else for e >= ea - 7.
// Integer operations on the bits, exact. An fp32-subnormal amax takes the floor 2^-126.
__device__ __forceinline__ float pow2_block_scale(float amax) {
  if (!(amax > 0.0f)) return 1.0f;
  const uint32_t b = __float_as_uint(amax);
  const int ebits = static_cast<int>((b >> 23) & 0xFFu);
  int e = ebits == 0 ? -126 : ebits - 127 - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  e = e < -126 ? -126 : (e > 127 ? 127 : e);
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// The scale-factor byte (UE8M0: 2^(byte - 127)) of an fp32 power-of-two scale: its exponent
// field. ok is cleared when the scale is not a positive normal power of two.
__device__ __forceinline__ uint32_t ue8m0_of(float scale, bool& ok) {
  const uint32_t b = __float_as_uint(scale);
  const uint32_t ebits = (b >> 23) & 0xFFu;
  if ((b & 0x807FFFFFu) != 0u || ebits == 0u || ebits == 0xFFu) ok = false;
  return ebits;
}

}  // namespace moe
