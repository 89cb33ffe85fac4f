// One decode step before attention: RoPE on the new token's q_pe and k_pe, and the append of
// its latent-cache row [c_kv | rotated k_pe] into the paged cache (TensorRT-LLM "mla.py",
// forward_absorption_generation: apply_rope on q's RoPE slice and on k_pe, the rotated q_pe
// written into the fused query, the latent cache row appended by mla_rope_generation /
// mla_rope_append_paged_kv_assign_q; RotaryEmbedding(head_dim=qk_rope_head_dim, is_neox)).
//
// One CTA per request.  Pair i of a 64-value RoPE vector is (x[2i], x[2i+1]) or, with is_neox,
// (x[i], x[i+32]); it turns by the angle whose cosine and sine are cos_sin[pos][i] and
// cos_sin[pos][32 + i]: (a, b) -> (a cos - b sin, a sin + b cos), in fp32, rounded to bf16.
// Every access is a 16-byte vector.  HBM-bound and tiny (a few KB per request).
#include <cuda_bf16.h>

#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

constexpr int kR = 64;      // RoPE width
constexpr int kPairs = 32;

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// Rotates the 64 values at src into dst (both 16-byte aligned) with `unit` in [0, 8): the
// unit's share of the vector (interleaved: values 8u .. 8u + 7, four pairs; halves: for u < 4
// values 8u .. 8u + 7 and their partners 32 + 8u .., eight pairs; units 4-7 idle).
__device__ __forceinline__ void rotate_unit(const __nv_bfloat16* src, __nv_bfloat16* dst, int unit, bool neox,
                                            const float* cs) {
  if (!neox) {
    float x[8];
    unpack8(*reinterpret_cast<const uint4*>(src + 8 * unit), x);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = 4 * unit + k;
      const float c = cs[i], s = cs[kPairs + i];
      const float a = x[2 * k], b = x[2 * k + 1];
      x[2 * k] = a * c - b * s;
      x[2 * k + 1] = a * s + b * c;
    }
    *reinterpret_cast<uint4*>(dst + 8 * unit) = pack8(x);
  } else if (unit < 4) {
    float lo[8], hi[8];
    unpack8(*reinterpret_cast<const uint4*>(src + 8 * unit), lo);
    unpack8(*reinterpret_cast<const uint4*>(src + kPairs + 8 * unit), hi);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = 8 * unit + k;
      const float c = cs[i], s = cs[kPairs + i];
      const float a = lo[k], b = hi[k];
      lo[k] = a * c - b * s;
      hi[k] = a * s + b * c;
    }
    *reinterpret_cast<uint4*>(dst + 8 * unit) = pack8(lo);
    *reinterpret_cast<uint4*>(dst + kPairs + 8 * unit) = pack8(hi);
  }
}

__global__ void __launch_bounds__(256) rope_append_kernel(const RopeAppendParams p) {
  const int b = blockIdx.x;
  __shared__ float cs[kR];
  __shared__ int64_t row_s;
  __shared__ int ok_s, pos_s;
  // guarded build: every plain access is checked against the extent its sizes give (guard_span)
  const uint64_t ext_cache = (uint64_t)p.num_pages * p.page_size * kDk * 2;
  if (threadIdx.x == 0) {
    const int pos = guard_span(p.err, G_POS, p.positions + b, 4, p.positions, (uint64_t)p.B * 4) ? p.positions[b] : -1;
    const int64_t cap = (int64_t)p.max_pages * p.page_size;
    bool ok = pos >= 0 && pos < p.max_pos && pos < cap;
    int64_t row = 0;
    if (ok) {
      const int32_t* e = p.block_table + (int64_t)b * p.max_pages + pos / p.page_size;
      const int32_t pg =
          guard_span(p.err, G_BLOCK_TABLE, e, 4, p.block_table, (uint64_t)p.B * p.max_pages * 4) ? *e : -1;
      ok = pg >= 0 && pg < p.num_pages;
      row = (int64_t)pg * p.page_size + pos % p.page_size;
    }
    if (!ok) record_error(p.err, DEV_RANGE_BASE | 0x60);
    ok_s = ok && guard_span(p.err, G_ROPE_OUT, p.cache + row * kDk, kDk * 2, p.cache, ext_cache) &&
           guard_span(p.err, G_ROPE_IN, p.cos_sin + (int64_t)pos * kR, kR * 4, p.cos_sin, (uint64_t)p.max_pos * kR * 4);
    row_s = row;
    pos_s = pos;
  }
  __syncthreads();
  if (!ok_s) return;
  if (threadIdx.x < kR) cs[threadIdx.x] = p.cos_sin[(int64_t)pos_s * kR + threadIdx.x];
  __syncthreads();
  const bool neox = p.is_neox != 0;
  // q: H rows of 64 values, 8 units each
  for (int u = threadIdx.x; u < p.H * 8; u += blockDim.x) {
    const int h = u >> 3;
    const __nv_bfloat16* src = p.q_pe + ((int64_t)b * p.H + h) * kR;
    __nv_bfloat16* dst = p.q_out + ((int64_t)b * p.H + h) * kDk + kLatent;
    if (guard_span(p.err, G_ROPE_IN, src, kR * 2, p.q_pe, (uint64_t)p.B * p.H * kR * 2) &&
        guard_span(p.err, G_ROPE_OUT, dst, kR * 2, p.q_out, (uint64_t)p.B * p.H * kDk * 2))
      rotate_unit(src, dst, u & 7, neox, cs);
  }
  // the cache row: 512 latent values copied, 64 RoPE values rotated
  __nv_bfloat16* crow = p.cache + row_s * kDk;
  const int t = threadIdx.x;
  if (t < kLatent / 8) {
    const __nv_bfloat16* src = p.c_kv + (int64_t)b * kLatent;
    if (guard_span(p.err, G_ROPE_IN, src, kLatent * 2, p.c_kv, (uint64_t)p.B * kLatent * 2))
      reinterpret_cast<uint4*>(crow)[t] = reinterpret_cast<const uint4*>(src)[t];
  } else if (t < kLatent / 8 + 8) {
    const __nv_bfloat16* src = p.k_pe + (int64_t)b * kR;
    if (guard_span(p.err, G_ROPE_IN, src, kR * 2, p.k_pe, (uint64_t)p.B * kR * 2))
      rotate_unit(src, crow + kLatent, t - kLatent / 8, neox, cs);
  }
}

}  // namespace

cudaError_t launch_rope_append(const RopeAppendParams& p, cudaStream_t stream) {
  if (p.B <= 0) return cudaSuccess;
  rope_append_kernel<<<p.B, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
