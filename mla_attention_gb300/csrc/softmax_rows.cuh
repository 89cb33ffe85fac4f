// Score-row helpers shared by the attention kernels: masking a 32-column piece of a row of
// raw scores read from tensor memory, and its extreme.
//
// kUp: the softmax scale is >= 0, so the row's largest scaled score belongs to its largest raw
// score (else to its smallest).  Keys of a piece past the visible limit get the raw score -inf
// (+inf when the scale is negative), so one mask-free body serves every piece: the extreme
// ignores them and 2^(s * scale_log2 - m) is 0 for them.  A zero scale is run as a tiny
// positive one, so no infinite score is ever multiplied by 0.
#pragma once
#include <cstdint>
#include <math_constants.h>

#include "sm103_ptx.cuh"

namespace mla {

// keys lim .. 31 of the piece are hidden (nothing when lim >= 32)
template <bool kUp>
__device__ __forceinline__ void mask_piece(uint32_t (&sr)[32], int lim) {
  if (lim < 32) {
    const uint32_t hide = __float_as_uint(kUp ? -CUDART_INF_F : CUDART_INF_F);
#pragma unroll
    for (int c = 0; c < 32; ++c) sr[c] = (c < lim) ? sr[c] : hide;
  }
}

// the same with the piece's visible keys given as bits (bit c: key c is visible)
template <bool kUp>
__device__ __forceinline__ void mask_bits(uint32_t (&sr)[32], uint32_t bits) {
  if (bits != 0xffffffffu) {
    const uint32_t hide = __float_as_uint(kUp ? -CUDART_INF_F : CUDART_INF_F);
#pragma unroll
    for (int c = 0; c < 32; ++c) sr[c] = ((bits >> c) & 1u) ? sr[c] : hide;
  }
}

// extreme of the piece's raw scores folded into four running partial extremes (three-input
// max / min: two scores per instruction)
template <bool kUp>
__device__ __forceinline__ void row_extreme(const uint32_t (&sr)[32], float (&eq)[4]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float v0 = __uint_as_float(sr[2 * i]), v1 = __uint_as_float(sr[2 * i + 1]);
    eq[i & 3] = kUp ? max3f(eq[i & 3], v0, v1) : min3f(eq[i & 3], v0, v1);
  }
}

template <bool kUp>
__device__ __forceinline__ float extreme4(const float (&eq)[4]) {
  return kUp ? fmaxf(fmaxf(eq[0], eq[1]), fmaxf(eq[2], eq[3])) : fminf(fminf(eq[0], eq[1]), fminf(eq[2], eq[3]));
}

}  // namespace mla
