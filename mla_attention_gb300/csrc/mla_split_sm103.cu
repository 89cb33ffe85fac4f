// Non-absorbed MLA prefill on the split layout (Huawei Ascend
// "RingMLAOperation": querySplit1/keySplit1 = 128 no-PE columns,
// querySplit2/keySplit2 = 64 RoPE columns, value = 128 columns, BSND,
// seqLen [batch] or [2, batch], kvHeadNum for grouped heads, qkScale,
// maskType NO_MASK / TRIU, prevOut / prevLse merged into the output).
//
// Work items are (128-query tile of one sequence, head) pairs, in head-major order (the
// items running at one time share one or a few heads, whose K/V stays in L2) and longest
// first within a head.  The kernel is persistent: one CTA per SM claims the next item from a
// counter in the workspace whenever it starts one, so the items in flight stay a window of
// consecutive items (a fixed share per CTA lets CTAs drift apart by many heads and their K/V
// out of L2); the claiming warp hands the item to the others through a small queue in
// shared memory.  The scores use both column groups: S = Q_nope K_nope^T +
// Q_pe K_pe^T, one contraction of depth 192 over the two tensors' boxes.  Tensor memory
// holds two S buffers (128 columns each) and two O buffers (128 x 128 fp32 each, one per
// item in flight).  P is written back over its own S buffer as bf16 and consumed from
// tensor memory by the P V MMA, so shared memory only holds Q and the K/V stages.
//
//   warp 4: claims items; TMA (Q per item once the previous item's S MMAs are done; K_nope,
//           K_pe, V per 128-key tile, two stages; an L2 prefetch of the next item's Q)
//   warp 5: MMA issue in the order S0, S1, PV0, S2, PV1, ... across items (the first S of
//           an item goes out before the last P V of the previous one)
//   warps 0-3: one query row per thread: mask, online softmax with lazy rescale (threshold
//           2^8), P -> TMEM; an item's epilogue (O / l, prev merge, store) runs in four
//           32-column pieces, one after each of the next item's first tiles, so the tensor
//           pipe keeps working through it
//
// A row's 128 scores of a tile are read from tensor memory in one go (four 32-column loads,
// one wait); its extreme is taken on the raw scores and 2^(s * scale_log2 - m) with one
// packed two-wide FMA per pair of scores (the sign of the scale picks the instantiation:
// the extreme of the raw scores is their maximum for a scale >= 0, their minimum below).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "mla_internal.h"
#include "mma_seq.cuh"
#include "sm103_ptx.cuh"
#include "softmax_rows.cuh"

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
constexpr uint32_t kTmemO = 256;   // two O buffers: [256,384), [384,512)
constexpr float kRescaleLog2 = 8.0f;
constexpr int kEpiPieces = 4;      // 32-column pieces of an item's epilogue
constexpr int kRing = 4;           // claimed items handed from the TMA warp to the others

struct Bars {
  uint64_t q_full;
  uint64_t q_empty;  // every S MMA of the item that holds Q is done (one commit per item)
  uint64_t k_full[kStages], k_empty[kStages];  // K part of stage s (freed by the S MMA)
  uint64_t v_full[kStages], v_empty[kStages];  // V part of stage s (freed by the P V MMA)
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];  // pv_done[b]: the P V that read P from S buffer b is complete
  uint64_t o_free[2];   // the rows read O buffer b out (its item's epilogue is done)
  uint64_t item_full[kRing], item_empty[kRing];  // the queue of claimed items (empty: 5 readers)
  uint64_t stall;  // fault injection: never arrived on
  uint64_t drain;  // abort: one commit of the MMA issuer lands here
  uint32_t tmem_base;
  uint32_t abort_flag;
  int32_t ring[kRing];  // item index, -1: no item left
};

static_assert(sizeof(Bars) <= 256, "barrier block larger than its shared-memory slot");

enum : uint32_t { W_QFULL = 0x20, W_KVEMPTY, W_KVFULL, W_SFULL, W_PFULL, W_ODONE, W_STALL, W_QEMPTY, W_OFREE, W_ITEM };

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

__device__ __forceinline__ TileInfo tile_info(const SplitParams& p, int64_t item) {
  TileInfo t;
  // Head-major: the CTAs running at one time work on one or a few heads, so those heads' K/V
  // stay in L2 while every query tile of the head reads them (head-minor order had ~150 heads'
  // K/V in flight at once and re-read them from HBM for every query tile).  Within a head the
  // tiles go longest first.
  const int per_head = p.total_q_tiles;
  const int gt = per_head - 1 - (int)(item % per_head);
  t.h = (int)(item / per_head);
  t.hk = t.h / (p.H / p.Hkv);
  // the sequence: the largest s with tile_off[s] <= gt (a sequence without query tiles shares
  // its offset with the next one and is passed over)
  int lo = 0, hi = p.batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.tile_off[mid] <= gt) lo = mid;
    else hi = mid - 1;
  }
  const int s = lo;
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

// One row's epilogue still to write: its item's output row, the softmax statistics and the
// merge with the previous output, written out in 32-column pieces.
struct RowEpilogue {
  int64_t tok;        // the row's token (the sequence's first when the row is past its end)
  int h;
  bool row_ok;        // the row is a query of the sequence
  bool tm;            // O is in tensor memory (the item has KV tiles)
  uint32_t item;      // the item's O buffer is item & 1
  uint32_t g_last;    // the item's last KV tile: its P V completes O
  float m_used, l;    // log2-domain offset and row sum
  // set by the first piece
  const __nv_bfloat16* prow;
  __nv_bfloat16* orow;
  float cn, wp, lse_out;
  int piece;          // next piece to write; kEpiPieces: nothing pending
};

template <bool kUp>
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
  const int64_t n_items = (int64_t)p.total_q_tiles * p.H;

  if (tid == 0) {
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.q_empty, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], 4);  // one arrival per row warp
      mbar_init(&bars.pv_done[i], 1);
      mbar_init(&bars.o_free[i], 4);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&bars.item_full[i], 1);
      mbar_init(&bars.item_empty[i], 5);  // the MMA warp and the four row warps
    }
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
  if (p.debug_stall && warp == 5) waitb(&bars.stall, 0, W_STALL);  // runs out: injected fault
  // the next claimed item from the queue (warps 0-3 and 5); -1 once none is left
  uint32_t n_popped = 0;
  auto pop_item = [&](int64_t& w) -> bool {
    const int k = n_popped % kRing;
    if (!waitb(&bars.item_full[k], (n_popped / kRing) & 1, W_ITEM)) return false;
    w = *reinterpret_cast<volatile int32_t*>(&bars.ring[k]);
    warp_arrive(&bars.item_empty[k]);
    ++n_popped;
    return true;
  };

  // abort drain: the last barrier phase this thread's TMA loads were counted on
  uint64_t* drain_bar = nullptr;
  uint32_t drain_par = 0;
  if (warp == 4) {
    // ---------------- TMA producer ----------------
    // K of a stage goes back to the producer once its S MMA is done, V once its P V MMA is done,
    // so K runs one tile ahead of V.  The boxes of a part go out from separate lanes at once: one
    // thread issues a TMA box only every few hundred cycles, lanes of a warp overlap theirs.
    // Counters run over the CTA's items: gk / gv KV tiles whose K / V went out, nq Q loads.
    uint32_t gk = 0, gv = 0, nq = 0;
    auto load_k = [&](const TileInfo& ti, int j) -> bool {
      const int s = gk % kStages;
      if (!waitb(&bars.k_empty[s], ((gk / kStages) & 1) ^ 1, W_KVEMPTY)) return false;
      const uint32_t st = smem_u32(smem + kOffStage + s * kStageBytes);
      if (lane == 0) mbar_arrive_expect_tx(&bars.k_full[s], kKBytes);
      __syncwarp();
      if (lane < 3) tma_load_3d(st + lane * kBox, lane < 2 ? &mk_nope : &mk_pe, lane == 1 ? 64 : 0, ti.hk,
                                ti.kv0 + j * kTile, &bars.k_full[s]);
      drain_bar = &bars.k_full[s];
      drain_par = (gk / kStages) & 1;
      ++gk;
      __syncwarp();
      return true;
    };
    auto load_v = [&](const TileInfo& ti, int j) -> bool {
      const int s = gv % kStages;
      if (!waitb(&bars.v_empty[s], ((gv / kStages) & 1) ^ 1, W_KVEMPTY)) return false;
      const uint32_t st = smem_u32(smem + kOffStage + s * kStageBytes + kKBytes);
      if (lane == 0) mbar_arrive_expect_tx(&bars.v_full[s], kVBytes);
      __syncwarp();
      if (lane < 2) tma_load_3d(st + lane * kBox, &mv, 64 * lane, ti.hk, ti.kv0 + j * kTile, &bars.v_full[s]);
      drain_bar = &bars.v_full[s];
      drain_par = (gv / kStages) & 1;
      ++gv;
      __syncwarp();
      return true;
    };
    auto claim = [&]() -> int64_t {
      uint32_t v = 0;
      if (lane == 0) v = atomicAdd(p.ticket, 1u);
      v = __shfl_sync(0xffffffffu, v, 0);
      return (int64_t)v < n_items ? (int64_t)v : -1;
    };
    uint32_t n_pushed = 0;
    auto push_item = [&](int64_t w) -> bool {
      const int k = n_pushed % kRing;
      if (!waitb(&bars.item_empty[k], ((n_pushed / kRing) & 1) ^ 1, W_ITEM)) return false;
      if (lane == 0) {
        bars.ring[k] = (int32_t)w;
        mbar_arrive(&bars.item_full[k]);  // release: the readers see the entry
      }
      __syncwarp();
      ++n_pushed;
      return true;
    };
    bool ok = true;
    int64_t w = claim();
    while (ok) {
      if (!push_item(w) || w < 0) break;
      const int64_t wn = claim();  // claimed now: its Q is prefetched while this item runs
      const TileInfo ti = tile_info(p, w);
      w = wn;
      if (ti.J == 0) continue;
      // Q: the single buffer is free once every S MMA of the previous item is done
      if (nq > 0 && !waitb(&bars.q_empty, (nq - 1) & 1, W_QEMPTY)) break;
      const int qz = ti.q0 + ti.tile * kTile;  // first query token of the tile
      const uint32_t sq = smem_u32(smem + kOffQ);
      if (lane == 0) mbar_arrive_expect_tx(&bars.q_full, kQBytes);
      __syncwarp();
      if (lane < 3) tma_load_3d(sq + lane * kBox, lane < 2 ? &mq_nope : &mq_pe, lane == 1 ? 64 : 0, ti.h, qz, &bars.q_full);
      drain_bar = &bars.q_full;
      drain_par = nq & 1;
      ++nq;
      // the next item's Q into L2 while this item runs (its load then waits on L2, not HBM)
      if (wn >= 0) {
        const TileInfo tn = tile_info(p, wn);
        const int qn = tn.q0 + tn.tile * kTile;
        if (lane < 3) tma_prefetch_3d(lane < 2 ? &mq_nope : &mq_pe, lane == 1 ? 64 : 0, tn.h, qn);
      }
      __syncwarp();
      ok = load_k(ti, 0);
      for (int j = 0; ok && j < ti.J; ++j) {
        if (j + 1 < ti.J && !load_k(ti, j + 1)) { ok = false; break; }
        ok = load_v(ti, j);
      }
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    // S(g) goes out as soon as K(g) has landed; the P V of the tile before it then waits for
    // its P.  Across items the order is the same: the next item's first S is issued before the
    // last P V of the previous item, so the tensor pipe works while the rows finish that P.
    const uint32_t idesc_s = idesc_bf16_f32(kTile, kTile, false, false);
    const uint32_t idesc_o = idesc_bf16_f32(kTile, 128, false, true);
    const uint32_t sq = smem_u32(smem + kOffQ);
    uint32_t g = 0;      // KV tiles whose S went out
    uint32_t items = 0;  // items with KV tiles started
    // the P V still to issue: its tile, its item (O buffer item & 1), first of its item
    bool pend = false, pfirst = false;
    uint32_t pg = 0, pitem = 0;
    auto issue_pv = [&]() -> bool {
      if (!waitb(&bars.p_full[pg & 1], (pg >> 1) & 1, W_PFULL)) return false;
      const int s = pg % kStages;
      if (!waitb(&bars.v_full[s], (pg / kStages) & 1, W_KVFULL)) return false;
      // the first P V of an item overwrites its O buffer: the rows must have read out the item
      // that used the buffer before (item - 2)
      if (pfirst && pitem >= 2 && !waitb(&bars.o_free[pitem & 1], ((pitem >> 1) & 1) ^ 1, W_OFREE)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t vst = smem_u32(smem + kOffStage + s * kStageBytes + kKBytes);
        mma_pv_tmem_k128_n128(tbase + kTmemO + (pitem & 1) * 128, tbase + kTmemS + (pg & 1) * kTile,
                              sdesc_sw128(vst, kBox, 1024), idesc_o, pfirst ? 0u : 1u);
        mma_commit(&bars.v_empty[s]);
        mma_commit(&bars.pv_done[pg & 1]);
      }
      __syncwarp();
      pend = false;
      return true;
    };
    bool live = true;
    while (live) {
      int64_t w;
      if (!pop_item(w)) { live = false; break; }
      if (w < 0) break;
      const TileInfo ti = tile_info(p, w);
      if (ti.J == 0) continue;
      if (!waitb(&bars.q_full, items & 1, W_QFULL)) { live = false; break; }
      for (int j = 0; j < ti.J; ++j, ++g) {
        const int s = g % kStages;
        if (!waitb(&bars.k_full[s], (g / kStages) & 1, W_KVFULL)) { live = false; break; }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t st = smem_u32(smem + kOffStage + s * kStageBytes);
          mma_s_k192_n128(tbase + kTmemS + (g & 1) * kTile, sdesc_sw128(sq, 16, 1024), sdesc_sw128(st, 16, 1024),
                          idesc_s);
          mma_commit(&bars.k_empty[s]);
          mma_commit(&bars.s_full[g & 1]);
          if (j + 1 == ti.J) mma_commit(&bars.q_empty);  // the item's last read of Q
        }
        __syncwarp();
        if (pend && !issue_pv()) { live = false; break; }
        pend = true;
        pg = g;
        pitem = items;
        pfirst = (j == 0);
      }
      ++items;
    }
    if (live && pend) issue_pv();
  } else {
    // ---------------- rows: softmax and epilogue ----------------
    const int r = tid;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float sl2 = (p.scale_log2 == 0.f) ? 1e-30f : p.scale_log2;  // see softmax_rows.cuh
    const uint64_t sl2x2 = f32x2(sl2, sl2);
    // guarded build: rows checked against the [Nq, H, 128] / [H, Nq] extents (guard_span)
    const uint64_t ext_rows = (uint64_t)p.Nq * p.H * 128 * 2, ext_lse = (uint64_t)p.H * p.Nq * 4;
    auto epi_begin = [&](RowEpilogue& e, int64_t tok, int h, bool row_ok, bool tm, uint32_t item, uint32_t g_last,
                         float m_used, float l) {
      e.tok = tok;
      e.h = h;
      e.row_ok = row_ok;
      e.tm = tm;
      e.item = item;
      e.g_last = g_last;
      e.m_used = m_used;
      e.l = l;
      e.piece = 0;
    };
    // One 32-column piece of an epilogue; the first waits for the item's last P V and works
    // out the weights.  The TMEM load is warp-collective: e.tm is uniform over the CTA.
    auto epi_piece = [&](RowEpilogue& e) -> bool {
      const int c0 = 32 * e.piece;
      if (e.piece == 0) {
        if (e.tm) {
          if (!waitb(&bars.pv_done[e.g_last & 1], (e.g_last >> 1) & 1, W_ODONE)) return false;
          tc_fence_after();
        }
        const bool has = e.tm && (e.l > 0.f);
        const float lse_new = has ? (e.m_used + log2f(e.l)) * 0.69314718055994531f : -CUDART_INF_F;
        float wn = has ? 1.f : 0.f, wp = 0.f, lse_out = lse_new;
        e.prow = nullptr;
        if (p.prev_out && e.row_ok &&
            guard_span(p.err, G_PREV_OUT, p.prev_out + (e.tok * p.H + e.h) * 128, 256, p.prev_out, ext_rows) &&
            guard_span(p.err, G_PREV_LSE, p.prev_lse + (int64_t)e.h * p.Nq + e.tok, 4, p.prev_lse, ext_lse)) {
          e.prow = p.prev_out + (e.tok * p.H + e.h) * 128;
          const float pl = p.prev_lse[(int64_t)e.h * p.Nq + e.tok];
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
        e.cn = has ? wn / e.l : 0.f;
        e.wp = wp;
        e.lse_out = lse_out;
        __nv_bfloat16* orow = p.out + (e.tok * p.H + e.h) * 128;
        const bool out_ok = e.row_ok && guard_span(p.err, G_OUT, orow, 256, p.out, ext_rows) &&
                            guard_span(p.err, G_LSE, p.lse + (int64_t)e.h * p.Nq + e.tok, 4, p.lse, ext_lse);
        e.orow = out_ok ? orow : nullptr;
      }
      float o[32];
      if (e.tm) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_base + kTmemO + (e.item & 1) * 128 + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) o[c] = __uint_as_float(v[c]) * e.cn;
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) o[c] = 0.f;
      }
      if (e.orow) {
        if (e.prow && e.wp > 0.f) {
          const uint4* pr = reinterpret_cast<const uint4*>(e.prow + c0);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 xv = pr[u];
            const __nv_bfloat162* hx = reinterpret_cast<const __nv_bfloat162*>(&xv);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              float2 f2 = __bfloat1622float2(hx[k]);
              o[8 * u + 2 * k] += e.wp * f2.x;
              o[8 * u + 2 * k + 1] += e.wp * f2.y;
            }
          }
        }
        uint4* dst = reinterpret_cast<uint4*>(e.orow + c0);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          dst[u] = make_uint4(pack_bf16x2(o[8 * u], o[8 * u + 1]), pack_bf16x2(o[8 * u + 2], o[8 * u + 3]),
                              pack_bf16x2(o[8 * u + 4], o[8 * u + 5]), pack_bf16x2(o[8 * u + 6], o[8 * u + 7]));
      }
      if (++e.piece == kEpiPieces) {
        if (e.orow) p.lse[(int64_t)e.h * p.Nq + e.tok] = e.lse_out;
        if (e.tm) {  // O buffer item & 1 is read out: the item two on may overwrite it
          tc_fence_before();
          warp_arrive(&bars.o_free[e.item & 1]);
        }
      }
      return true;
    };

    RowEpilogue ep;  // the previous item's epilogue, written during this item's first tiles
    ep.piece = kEpiPieces;
    uint32_t g = 0, items = 0;  // KV tiles and items with KV tiles so far (as the MMA warp counts)
    bool live = true;
    while (live) {
      int64_t w;
      if (!pop_item(w)) { live = false; break; }
      if (w < 0) break;
      const TileInfo ti = tile_info(p, w);
      const int i = ti.tile * kTile + r;  // query index within the sequence
      const bool row_ok = i < ti.ql;
      const int nkeys = row_ok ? keys_for_query(p, ti.ql, ti.kl, i) : 0;
      const int64_t tok = (int64_t)ti.q0 + (row_ok ? i : 0);
      if (p.prev_out && row_ok) {  // the previous output row into L2 for this item's epilogue
        const __nv_bfloat16* pr = p.prev_out + (tok * p.H + ti.h) * 128;
        if (guard_span(p.err, G_PREV_OUT, pr, 256, p.prev_out, ext_rows)) {
          prefetch_l2(pr);
          prefetch_l2(pr + 64);
        }
      }
      if (ti.J == 0) {  // no key: O is zero and the previous output passes through
        RowEpilogue z;
        epi_begin(z, tok, ti.h, row_ok, false, 0, 0, -CUDART_INF_F, 0.f);
        while (z.piece < kEpiPieces) epi_piece(z);  // no wait without TMEM
        continue;
      }
      float m_used = -CUDART_INF_F, l = 0.f;
      for (int j = 0; j < ti.J; ++j, ++g) {
        const int sb = g & 1;
        if (!waitb(&bars.s_full[sb], (g >> 1) & 1, W_SFULL)) { live = false; break; }
        tc_fence_after();
        const uint32_t sa = tbase + lane_base + kTmemS + sb * kTile;
        uint32_t sr[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(sa + 32 * q, sr[q]);
        tmem_wait_ld();
        int nv = nkeys - j * kTile;
        nv = nv < 0 ? 0 : (nv > kTile ? kTile : nv);
        float eq[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) eq[k] = kUp ? -CUDART_INF_F : CUDART_INF_F;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          mask_piece<kUp>(sr[q], nv - 32 * q);
          row_extreme<kUp>(sr[q], eq);
        }
        const float mt = (nv == 0) ? -CUDART_INF_F : extreme4<kUp>(eq) * sl2;
        float a = 1.f;
        if (mt > m_used + kRescaleLog2) {
          if (l > 0.f) a = ex2_approx(m_used - mt);
          l *= a;
          m_used = mt;
        }
        // tcgen05.ld/st are warp-collective: rescale when any row of the warp needs it (never on
        // an item's first tile, where l is 0 and the first P V overwrites O)
        if (__any_sync(0xffffffffu, a != 1.f)) {
          // O must hold P V of every earlier tile of the item before it is rescaled
          if (!waitb(&bars.pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, W_ODONE)) { live = false; break; }
          tc_fence_after();
          const uint32_t oa = tbase + lane_base + kTmemO + (items & 1) * 128;
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
        const uint64_t nmsub2 = f32x2(-msub, -msub);
        uint64_t rsq[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t pk[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            float x0, x1;
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(sr[q][2 * u]), __uint_as_float(sr[q][2 * u + 1])), sl2x2,
                                  nmsub2),
                        x0, x1);
            const float e0 = ex2_approx(x0);
            const float e1 = ex2_approx(x1);
            rsq[u & 1] = add_f32x2(rsq[u & 1], f32x2(e0, e1));
            pk[u] = pack_bf16x2(e0, e1);
          }
          tmem_st16(sa + 16 * q, pk);  // P (bf16 pairs) over the first 64 columns of S
        }
        {
          float q0, q1, q2, q3;
          f32x2_split(rsq[0], q0, q1);
          f32x2_split(rsq[1], q2, q3);
          l += (q0 + q1) + (q2 + q3);
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(&bars.p_full[sb]);
        // a piece of the previous item's epilogue while the tensor pipe runs this tile's P V
        if (ep.piece < kEpiPieces && !epi_piece(ep)) { live = false; break; }
      }
      if (!live) break;
      while (live && ep.piece < kEpiPieces) live = epi_piece(ep);  // the item had fewer tiles than pieces
      if (!live) break;
      epi_begin(ep, tok, ti.h, row_ok, true, items, g - 1, m_used, l);
      ++items;
    }
    while (live && ep.piece < kEpiPieces) live = epi_piece(ep);
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
  cudaError_t e = attrs.run([] {
    cudaError_t r = cudaFuncSetAttribute(mla_split_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (r != cudaSuccess) return r;
    return cudaFuncSetAttribute(mla_split_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  });
  if (e != cudaSuccess) return e;
  const int64_t items = (int64_t)p.total_q_tiles * p.H;
  if (items == 0) return cudaSuccess;
  const int64_t sms = device_sm_count();
  const int64_t blocks = items < sms ? items : sms;
  auto kern = p.scale_log2 >= 0.f ? mla_split_kernel<true> : mla_split_kernel<false>;
  kern<<<dim3((unsigned)blocks), dim3(kThreads), kSmemAlloc, stream>>>(p, mq_nope, mq_pe, mk_nope, mk_pe, mv);
  return cudaGetLastError();
}

}  // namespace mla
