// Non-absorbed MLA prefill on the split layout (Huawei Ascend
// "RingMLAOperation": querySplit1/keySplit1 = 128 no-PE columns,
// querySplit2/keySplit2 = 64 RoPE columns, value = 128 columns, BSND,
// seqLen [batch] or [2, batch], kvHeadNum for grouped heads, qkScale,
// maskType NO_MASK / TRIU, prevOut / prevLse merged into the output).
//
// One CTA per (128-query tile of one sequence, head).  The scores use both
// column groups: S = Q_nope K_nope^T + Q_pe K_pe^T, one contraction of depth
// 192 over the two tensors' boxes.  Tensor memory holds two S buffers (128
// columns each) and O (128 x 128 fp32).  P is written back over its own S
// buffer as bf16 and consumed from tensor memory by the P V MMA, so shared
// memory only holds Q and the K/V stages.
//
//   warp 4: TMA (Q once; K_nope, K_pe, V per 128-key tile, two stages)
//   warp 5: MMA issue in the order S0, S1, PV0, S2, PV1, ...
//   warps 0-3: one query row per thread: mask, online softmax with lazy
//              rescale (threshold 2^8), P -> TMEM, epilogue with prev merge
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "mla_internal.h"
#include "mma_seq.cuh"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads = 192;
constexpr int kTile = 128;                 // queries per tile = keys per KV tile
constexpr int kBox = kTile * 128;          // one 128-row x 64-col box: 16 KB
constexpr int kQBytes = 3 * kBox;          // nope (2 boxes) + pe (1 box)
constexpr int kKBytes = 3 * kBox;
constexpr int kVBytes = 2 * kBox;
constexpr int kStageBytes = kKBytes + kVBytes;  // 80 KB
constexpr int kStages = 2;
constexpr int kOffQ = 0;
constexpr int kOffStage = kQBytes;
constexpr int kOffBars = kOffStage + kStages * kStageBytes;
constexpr int kSmemAlloc = kOffBars + 256 + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory over the sm_103a limit");

constexpr uint32_t kTmemS = 0;     // two S buffers: [0,128), [128,256)
constexpr uint32_t kTmemO = 256;   // O: [256, 384)
constexpr float kRescaleLog2 = 8.0f;

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kStages], k_empty[kStages];  // K part of stage s (freed by the S MMA)
  uint64_t v_full[kStages], v_empty[kStages];  // V part of stage s (freed by the P V MMA)
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];  // pv_done[b]: the P V that read P from S buffer b is complete
  uint64_t stall;  // fault injection: never arrived on
  uint64_t drain;  // abort: one commit of the MMA issuer lands here
  uint32_t tmem_base;
  uint32_t abort_flag;
};

static_assert(sizeof(Bars) <= 256, "barrier block larger than its shared-memory slot");

enum : uint32_t { W_QFULL = 0x20, W_KVEMPTY, W_KVFULL, W_SFULL, W_PFULL, W_ODONE, W_STALL };

struct TileInfo {
  int seq, tile, h, hk;
  int q0, ql, kv0, kl;  // token offsets and lengths of the sequence
  int J;                // KV tiles
};

__device__ __forceinline__ int keys_for_query(const SplitParams& p, int ql, int kl, int i) {
  if (!p.causal) return kl;
  int n = kl - ql + i + 1;
  if (n > kl) n = kl;
  return n < 0 ? 0 : n;
}

__device__ __forceinline__ TileInfo tile_info(const SplitParams& p, int block) {
  TileInfo t;
  // Head-major: the CTAs running at one time work on one or a few heads, so those heads' K/V
  // stay in L2 while every query tile of the head reads them (head-minor order had ~150 heads'
  // K/V in flight at once and re-read them from HBM for every query tile).  Within a head the
  // tiles go longest first.
  const int per_head = p.total_q_tiles;
  const int gt = per_head - 1 - block % per_head;
  t.h = block / per_head;
  t.hk = t.h / (p.H / p.Hkv);
  int s = 0;
  while (s + 1 < p.batch && p.tile_off[s + 1] <= gt) ++s;
  t.seq = s;
  t.tile = gt - p.tile_off[s];
  t.q0 = p.q_off[s];
  t.ql = p.q_off[s + 1] - p.q_off[s];
  t.kv0 = p.kv_off[s];
  t.kl = p.kv_off[s + 1] - p.kv_off[s];
  int last = t.tile * kTile + kTile - 1;
  if (last > t.ql - 1) last = t.ql - 1;
  const int n = keys_for_query(p, t.ql, t.kl, last);
  t.J = (n + kTile - 1) / kTile;
  return t;
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_split_kernel(const __grid_constant__ SplitParams p, const __grid_constant__ CUtensorMap mq_nope,
                     const __grid_constant__ CUtensorMap mq_pe, const __grid_constant__ CUtensorMap mk_nope,
                     const __grid_constant__ CUtensorMap mk_pe, const __grid_constant__ CUtensorMap mv) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars& bars = *reinterpret_cast<Bars*>(smem + kOffBars);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t lim = p.spin_limit;
  uint32_t* err = p.err;
  const TileInfo ti = tile_info(p, blockIdx.x);

  if (tid == 0) {
    mbar_init(&bars.q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], kTile);
    }
    mbar_init(&bars.pv_done[0], 1);
    mbar_init(&bars.pv_done[1], 1);
    mbar_init(&bars.stall, 1);
    mbar_init(&bars.drain, 1);
    bars.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars.tmem_base;
  volatile uint32_t* abort_flag = &bars.abort_flag;
  // Every wait is made by a whole warp and its outcome is warp-uniform, so no
  // warp reaches a warp-collective tcgen05 instruction with some lanes gone.
  auto waitb = [&](uint64_t* bar, uint32_t parity, uint32_t site) -> bool {
    bool ok = (*abort_flag == 0) && mbar_wait_inline(bar, parity, err, site, lim);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) *abort_flag = 1;
    return ok;
  };
  const int qz = ti.q0 + ti.tile * kTile;  // first query token of the tile
  if (p.debug_stall && warp == 5) waitb(&bars.stall, 0, W_STALL);  // runs out: injected fault

  // abort drain: the last barrier phase this thread's TMA loads were counted on
  uint64_t* drain_bar = nullptr;
  uint32_t drain_par = 0;
  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (ti.J > 0) {
      drain_bar = &bars.q_full;
      drain_par = 0;
    }
    if (ti.J > 0) {
      const uint32_t sq = smem_u32(smem + kOffQ);
      if (lane == 0) mbar_arrive_expect_tx(&bars.q_full, kQBytes);
      __syncwarp();
      if (lane < 3) tma_load_3d(sq + lane * kBox, lane < 2 ? &mq_nope : &mq_pe, lane == 1 ? 64 : 0, ti.h, qz, &bars.q_full);
    }
    // K of a stage goes back to the producer once its S MMA is done, V once its P V MMA is done,
    // so K runs one tile ahead of V.  The boxes of a part go out from separate lanes at once: one
    // thread issues a TMA box only every few hundred cycles, lanes of a warp overlap theirs.
    auto load_k = [&](int j) -> bool {
      const int s = j % kStages;
      if (!waitb(&bars.k_empty[s], ((j / kStages) & 1) ^ 1, W_KVEMPTY)) return false;
      const uint32_t st = smem_u32(smem + kOffStage + s * kStageBytes);
      if (lane == 0) mbar_arrive_expect_tx(&bars.k_full[s], kKBytes);
      __syncwarp();
      if (lane < 3) tma_load_3d(st + lane * kBox, lane < 2 ? &mk_nope : &mk_pe, lane == 1 ? 64 : 0, ti.hk,
                                ti.kv0 + j * kTile, &bars.k_full[s]);
      drain_bar = &bars.k_full[s];
      drain_par = (j / kStages) & 1;
      __syncwarp();
      return true;
    };
    auto load_v = [&](int j) -> bool {
      const int s = j % kStages;
      if (!waitb(&bars.v_empty[s], ((j / kStages) & 1) ^ 1, W_KVEMPTY)) return false;
      const uint32_t st = smem_u32(smem + kOffStage + s * kStageBytes + kKBytes);
      if (lane == 0) mbar_arrive_expect_tx(&bars.v_full[s], kVBytes);
      __syncwarp();
      if (lane < 2) tma_load_3d(st + lane * kBox, &mv, 64 * lane, ti.hk, ti.kv0 + j * kTile, &bars.v_full[s]);
      drain_bar = &bars.v_full[s];
      drain_par = (j / kStages) & 1;
      __syncwarp();
      return true;
    };
    bool ok = ti.J == 0 || load_k(0);
    for (int j = 0; ok && j < ti.J; ++j) {
      if (j + 1 < ti.J && !load_k(j + 1)) break;
      ok = load_v(j);
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc_s = idesc_bf16_f32(kTile, kTile, false, false);
    const uint32_t idesc_o = idesc_bf16_f32(kTile, 128, false, true);
    const uint32_t sq = smem_u32(smem + kOffQ);
    auto issue_s = [&](int j) -> bool {
      const int s = j % kStages;
      if (!waitb(&bars.k_full[s], (j / kStages) & 1, W_KVFULL)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t st = smem_u32(smem + kOffStage + s * kStageBytes);
        mma_s_k192_n128(tbase + kTmemS + (j & 1) * kTile, sdesc_sw128(sq, 16, 1024), sdesc_sw128(st, 16, 1024),
                        idesc_s);
        mma_commit(&bars.k_empty[s]);
        mma_commit(&bars.s_full[j & 1]);
      }
      __syncwarp();
      return true;
    };
    bool live = ti.J == 0 ? true : waitb(&bars.q_full, 0, W_QFULL);
    if (live && ti.J > 0) live = issue_s(0);
    for (int j = 0; live && j < ti.J; ++j) {
      if (j + 1 < ti.J && !issue_s(j + 1)) break;
      if (!waitb(&bars.p_full[j & 1], (j >> 1) & 1, W_PFULL)) break;
      if (!waitb(&bars.v_full[j % kStages], (j / kStages) & 1, W_KVFULL)) break;
      tc_fence_after();
      if (lane == 0) {
        const int s = j % kStages;
        const uint32_t vst = smem_u32(smem + kOffStage + s * kStageBytes + kKBytes);
        mma_pv_tmem_k128_n128(tbase + kTmemO, tbase + kTmemS + (j & 1) * kTile, sdesc_sw128(vst, kBox, 1024), idesc_o,
                              j > 0 ? 1u : 0u);
        mma_commit(&bars.v_empty[s]);
        mma_commit(&bars.pv_done[j & 1]);
      }
      __syncwarp();
    }
  } else {
    // ---------------- rows: softmax and epilogue ----------------
    const int r = tid;
    const int i = ti.tile * kTile + r;  // query index within the sequence
    const bool row_ok = i < ti.ql;
    const int nkeys = row_ok ? keys_for_query(p, ti.ql, ti.kl, i) : 0;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float m_used = -CUDART_INF_F, l = 0.f;
    bool live = true;
    for (int j = 0; j < ti.J; ++j) {
      const int sb = j & 1;
      if (!waitb(&bars.s_full[sb], (j >> 1) & 1, W_SFULL)) { live = false; break; }
      tc_fence_after();
      const uint32_t sa = tbase + lane_base + kTmemS + sb * kTile;
      float x[128];
      float mt = -CUDART_INF_F;
      int nv = nkeys - j * kTile;
      nv = nv < 0 ? 0 : (nv > kTile ? kTile : nv);
#pragma unroll
      for (int c0 = 0; c0 < kTile; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(sa + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c0 + c] = (c0 + c < nv) ? __uint_as_float(v[c]) * p.scale_log2 : -CUDART_INF_F;
          mt = fmaxf(mt, x[c0 + c]);
        }
      }
      float a = 1.f;
      if (mt > m_used + kRescaleLog2) {
        if (l > 0.f) a = ex2_approx(m_used - mt);
        l *= a;
        m_used = mt;
      }
      // tcgen05.ld/st are warp-collective: rescale when any row of the warp needs it
      if (__any_sync(0xffffffffu, a != 1.f)) {
        // O must hold P V of every earlier tile before it is rescaled: PV(j-1) is
        // use (j-1)/2 of buffer (j-1)%2 and the next use of that buffer needs P(j+1)
        if (!waitb(&bars.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, W_ODONE)) { live = false; break; }
        tc_fence_after();
        const uint32_t oa = tbase + lane_base + kTmemO;
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(oa + c0, v);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * a);
          tmem_st32(oa + c0, v);
        }
      }
      const float msub = (m_used == -CUDART_INF_F) ? 0.f : m_used;
      float rs = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < kTile; c0 += 32) {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float e0 = ex2_approx(x[c0 + 2 * c] - msub);
          const float e1 = ex2_approx(x[c0 + 2 * c + 1] - msub);
          rs += e0 + e1;
          pk[c] = pack_bf16x2(e0, e1);
        }
        tmem_st16(sa + (c0 >> 1), pk);  // P (bf16 pairs) over the first 64 columns of S
      }
      l += rs;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars.p_full[sb]);
    }
    // ---- epilogue ----
    if (live && ti.J > 0) {
      live = waitb(&bars.pv_done[(ti.J - 1) & 1], ((ti.J - 1) >> 1) & 1, W_ODONE);
      tc_fence_after();
    }
    if (live) {
      const int64_t tok = (int64_t)ti.q0 + (row_ok ? i : 0);
      const bool has = (ti.J > 0) && (l > 0.f);
      const float lse_new = has ? (m_used + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
      float wn = has ? 1.f : 0.f, wp = 0.f, lse_out = lse_new;
      const __nv_bfloat16* prow = nullptr;
      // guarded build: rows checked against the [Nq, H, 128] / [H, Nq] extents (guard_span)
      const uint64_t ext_rows = (uint64_t)p.Nq * p.H * 128 * 2, ext_lse = (uint64_t)p.H * p.Nq * 4;
      if (p.prev_out && row_ok && guard_span(p.err, G_PREV_OUT, p.prev_out + (tok * p.H + ti.h) * 128, 256, p.prev_out, ext_rows) &&
          guard_span(p.err, G_PREV_LSE, p.prev_lse + (int64_t)ti.h * p.Nq + tok, 4, p.prev_lse, ext_lse)) {
        prow = p.prev_out + (tok * p.H + ti.h) * 128;
        const float pl = p.prev_lse[(int64_t)ti.h * p.Nq + tok];
        const float m = fmaxf(pl, lse_new);
        if (m == -CUDART_INF_F) {
          wn = wp = 0.f;
          lse_out = -CUDART_INF_F;
        } else {
          wp = (pl == -CUDART_INF_F) ? 0.f : expf(pl - m);
          wn = has ? expf(lse_new - m) : 0.f;
          const float ws = wp + wn;
          lse_out = m + logf(ws);
          wp /= ws;
          wn /= ws;
        }
      }
      const float cn = has ? wn / l : 0.f;
      __nv_bfloat16* orow = p.out + (tok * p.H + ti.h) * 128;
      const bool out_ok = guard_span(p.err, G_OUT, orow, 256, p.out, ext_rows) &&
                          guard_span(p.err, G_LSE, p.lse + (int64_t)ti.h * p.Nq + tok, 4, p.lse, ext_lse);
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 32) {
        float o[32];
        if (ti.J > 0) {  // uniform over the CTA: every lane takes part in the TMEM load
          uint32_t v[32];
          tmem_ld32(tbase + lane_base + kTmemO + c0, v);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __uint_as_float(v[c]) * cn;
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = 0.f;
        }
        if (!row_ok || !out_ok) continue;
        if (prow && wp > 0.f) {
          const uint4* pr = reinterpret_cast<const uint4*>(prow + c0);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 xv = pr[u];
            const __nv_bfloat162* hx = reinterpret_cast<const __nv_bfloat162*>(&xv);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              float2 f2 = __bfloat1622float2(hx[k]);
              o[8 * u + 2 * k] += wp * f2.x;
              o[8 * u + 2 * k + 1] += wp * f2.y;
            }
          }
        }
        uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          dst[u] = make_uint4(pack_bf16x2(o[8 * u], o[8 * u + 1]), pack_bf16x2(o[8 * u + 2], o[8 * u + 3]),
                              pack_bf16x2(o[8 * u + 4], o[8 * u + 5]), pack_bf16x2(o[8 * u + 6], o[8 * u + 7]));
      }
      if (row_ok && out_ok) p.lse[(int64_t)ti.h * p.Nq + tok] = lse_out;
    }
  }

  __syncwarp();
  if (*abort_flag) {
    // let what this thread issued land before the CTA leaves: its MMAs (one more commit, which
    // arrives once they are all done) and its TMA loads (their last full barrier phase)
    if (warp == 5 && lane == 0) {
      mma_commit(&bars.drain);
      mbar_drain(&bars.drain, 0);
    }
    mbar_drain(drain_bar, drain_par);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) tmem_dealloc(tbase, 512);
}

}  // namespace

cudaError_t launch_split(const SplitParams& p, const CUtensorMap& mq_nope, const CUtensorMap& mq_pe,
                         const CUtensorMap& mk_nope, const CUtensorMap& mk_pe, const CUtensorMap& mv,
                         cudaStream_t stream) {
  static PerDeviceOnce attrs;
  cudaError_t e = attrs.run(
      [] { return cudaFuncSetAttribute(mla_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc); });
  if (e != cudaSuccess) return e;
  const int64_t blocks = (int64_t)p.total_q_tiles * p.H;
  if (blocks == 0) return cudaSuccess;
  mla_split_kernel<<<dim3((unsigned)blocks), dim3(kThreads), kSmemAlloc, stream>>>(p, mq_nope, mq_pe, mk_nope, mk_pe,
                                                                                   mv);
  return cudaGetLastError();
}

}  // namespace mla
