// LSE merge of two partial attention results, and the split-K reduction of
// the decode path.  Both are HBM-bound streaming kernels on CUDA cores.
//
// Algebra (TensorRT-LLM "mla.py", merge_attention_for_mla inside
// forward_context_with_chunked_prefill; Ascend "RingMLAOperation", prevOut /
// prevLse; Mojo "mha_single_batch_pipelined", split-K reduction):
//   m = max(lse_a, lse_b); w_a = e^(lse_a - m); w_b = e^(lse_b - m)
//   out = (w_a out_a + w_b out_b) / (w_a + w_b); lse = m + ln(w_a + w_b)
// A side with lse = -inf has weight 0; two such sides give (0, -inf).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "mla_internal.h"

namespace mla {

namespace {

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ uint4 f32_to_bf16x8(const float (&f)[8]) {
  uint4 v;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return v;
}

// one warp per (row, head); lanes stride over dv in 8-element (16-byte) chunks.  out / lse may
// be the same buffers as out_a / lse_a or out_b / lse_b (an in-place merge), so no pointer is
// declared __restrict__: every element is read before the same lane writes it.
__global__ void __launch_bounds__(256) merge_kernel(const __nv_bfloat16* out_a, const float* lse_a,
                                                    const __nv_bfloat16* out_b, const float* lse_b,
                                                    __nv_bfloat16* out, float* lse, int64_t rows, int H, int dv) {
  const int lane = threadIdx.x & 31;
  const int64_t nitems = rows * (int64_t)H;
  const int64_t warp0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t it = warp0; it < nitems; it += nwarps) {
    const int64_t r = it / H;
    const int h = (int)(it - r * H);
    const float la = lse_a[(int64_t)h * rows + r];
    const float lb = lse_b[(int64_t)h * rows + r];
    const float m = fmaxf(la, lb);
    float wa = 0.f, wb = 0.f;
    if (m != -CUDART_INF_F) {
      wa = (la == -CUDART_INF_F) ? 0.f : expf(la - m);
      wb = (lb == -CUDART_INF_F) ? 0.f : expf(lb - m);
    }
    const float wsum = wa + wb;
    const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
    const float ca = wa * inv, cb = wb * inv;
    const uint4* pa = reinterpret_cast<const uint4*>(out_a + it * dv);
    const uint4* pb = reinterpret_cast<const uint4*>(out_b + it * dv);
    uint4* po = reinterpret_cast<uint4*>(out + it * dv);
    for (int c = lane; c < dv / 8; c += 32) {
      float fa[8], fb[8], fo[8];
      uint4 va = pa[c], vb = pb[c];
      bf16x8_to_f32(va, fa);
      bf16x8_to_f32(vb, fb);
#pragma unroll
      for (int i = 0; i < 8; ++i) fo[i] = (wsum > 0.f) ? (ca * fa[i] + cb * fb[i]) : 0.f;
      po[c] = f32_to_bf16x8(fo);
    }
    __syncwarp();  // every lane has read lse_a / lse_b of this item before lse (maybe the same word) is written
    if (lane == 0) lse[(int64_t)h * rows + r] = (wsum > 0.f) ? m + logf(wsum) : -CUDART_INF_F;
  }
}

// Decode split-K reduction: query group b, head h merges the partials of the CTA
// pairs whose key ranges overlapped group b (slot = b + pair).  With sinks, head h's sink
// logit joins the softmax denominator as one more term that carries no value (Modular Mojo
// "mha_single_batch_pipelined", sink / sink_weights): out = sum_j e^{s_j} v_j / (e^{sink_h} +
// sum_j e^{s_j}), lse = ln(e^{sink_h} + sum_j e^{s_j}).
__global__ void __launch_bounds__(256) decode_reduce_kernel(const __grid_constant__ CoreParams prm, __nv_bfloat16* out,
                                                            float* lse) {
  const float* __restrict__ part_o = prm.part_o;
  const float* __restrict__ part_lse = prm.part_lse;
  const int32_t* __restrict__ tile_prefix = prm.tile_prefix;
  const float* __restrict__ sinks = prm.sinks;
  const int B = prm.B, H = prm.H, num_pairs = prm.num_pairs;
  uint32_t* err = prm.err;
  // guarded build: every plain access below is checked against its buffer (see guard_span)
  auto prefix = [&](int64_t i) -> int64_t {
    return guard_span(err, G_TILE_PREFIX, tile_prefix + i, 4, tile_prefix, prm.ext_tile_prefix) ? tile_prefix[i] : 0;
  };
  auto plse = [&](int64_t slot) -> float {
    return guard_span(err, G_PART_LSE, part_lse + slot, 4, part_lse, prm.ext_part_lse) ? part_lse[slot] : -CUDART_INF_F;
  };
  const int lane = threadIdx.x & 31;
  const int64_t nitems = (int64_t)B * H;
  const int64_t warp0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t total = prefix(B);
  for (int64_t it = warp0; it < nitems; it += nwarps) {
    const int b = (int)(it / H);
    const int h = (int)(it - (int64_t)b * H);
    const int64_t t0 = prefix(b), t1 = prefix(b + 1);
    __nv_bfloat16* orow = out + it * kLatent;
    if (!guard_span(err, G_OUT, orow, kLatent * 2, out, prm.ext_out)) continue;
    float* lse_it = (lse && guard_span(err, G_LSE, lse + it, 4, lse, prm.ext_lse)) ? lse + it : nullptr;
    const float sink = (sinks && guard_span(err, G_SINKS, sinks + h, 4, sinks, prm.ext_sinks)) ? sinks[h] : -CUDART_INF_F;
    if (t1 <= t0) {  // no key: out = 0, lse = -inf (or the sink's logit)
      for (int c = lane; c < kLatent / 8; c += 32) reinterpret_cast<uint4*>(orow)[c] = make_uint4(0, 0, 0, 0);
      if (lane == 0 && lse_it) *lse_it = sink;
      continue;
    }
    // pair owning tile t: the largest p with floor(p * total / P) <= t
    const int p_first = (int)(((t0 + 1) * (int64_t)num_pairs - 1) / total);
    const int p_last = (int)(((t1) * (int64_t)num_pairs - 1) / total);
    // a pair whose share of the tiles is empty wrote no partial: skip it
    auto owns = [&](int p) { return (int64_t)p * total / num_pairs < (int64_t)(p + 1) * total / num_pairs; };
    float m = sink;
    for (int p = p_first; p <= p_last; ++p)
      if (owns(p)) m = fmaxf(m, plse((int64_t)(b + p) * H + h));
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
    float wsum = (sink == -CUDART_INF_F) ? 0.f : expf(sink - m);
    if (m != -CUDART_INF_F) {
      for (int p = p_first; p <= p_last; ++p) {
        if (!owns(p)) continue;
        const int64_t slot = (int64_t)(b + p) * H + h;
        const float l = plse(slot);
        if (l == -CUDART_INF_F) continue;
        if (!guard_span(err, G_PART_O, part_o + slot * kLatent, kLatent * 4, part_o, prm.ext_part_o)) continue;
        const float w = expf(l - m);
        wsum += w;
        const float4* src = reinterpret_cast<const float4*>(part_o + slot * kLatent);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float4 v = src[lane + 32 * k];
          acc[4 * k + 0] += w * v.x;
          acc[4 * k + 1] += w * v.y;
          acc[4 * k + 2] += w * v.z;
          acc[4 * k + 3] += w * v.w;
        }
      }
    }
    const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc[4 * k] * inv, acc[4 * k + 1] * inv);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc[4 * k + 2] * inv, acc[4 * k + 3] * inv);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(orow)[lane + 32 * k] = pk;
    }
    if (lane == 0 && lse_it) *lse_it = (wsum > 0.f) ? m + logf(wsum) : -CUDART_INF_F;
  }
}

int grid_for(int64_t warps_needed) {
  const int sms = device_sm_count();
  int64_t blocks = (warps_needed + 7) / 8;
  int64_t cap = (int64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

}  // namespace

cudaError_t launch_merge(const __nv_bfloat16* out_a, const float* lse_a, const __nv_bfloat16* out_b,
                         const float* lse_b, __nv_bfloat16* out, float* lse, int64_t rows, int H, int dv,
                         cudaStream_t stream) {
  const int64_t items = rows * (int64_t)H;
  if (items == 0) return cudaSuccess;
  merge_kernel<<<grid_for(items), 256, 0, stream>>>(out_a, lse_a, out_b, lse_b, out, lse, rows, H, dv);
  return cudaGetLastError();
}

cudaError_t launch_decode_reduce(const CoreParams& p, __nv_bfloat16* out, float* lse, cudaStream_t stream) {
  const int64_t items = (int64_t)p.B * p.H;
  if (items == 0) return cudaSuccess;
  decode_reduce_kernel<<<grid_for(items), 256, 0, stream>>>(p, out, lse);
  return cudaGetLastError();
}

}  // namespace mla
