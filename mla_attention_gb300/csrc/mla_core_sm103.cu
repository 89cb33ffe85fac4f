// Absorbed MLA tile engine for sm_103a: one shared KV head whose rows are
// [512 latent | 64 RoPE]; QK^T over all 576 columns; V = the first 512
// columns of the same rows (Tenstorrent "ttnn.transformer.ring_mla": "QK uses
// the full KV head dimension and QKT@V uses the first head_dim_v columns").
//
// One tile = 128 query rows against the KV rows in tiles of 64 keys.  An
// fp32 O tile of 128 x 512 fills the whole 512-column tensor memory of one
// SM, so each tile is handled by a cluster of two CTAs on two SMs:
//
//   S-CTA (cluster rank 0)                 O-CTA (cluster rank 1)
//   TMEM: Q [128 x 576 bf16] (288 cols)    TMEM: O [128 x 512 fp32] (512 cols)
//         S double buffer (2 x 64 cols)
//   warp 4: TMA K tiles (9 col boxes)      warp 4: TMA V tiles (8 col boxes)
//   warp 5: S = Q K^T (A from TMEM)        warp 5: O += P V (P, V from smem)
//   warps 0-3: online softmax, one row     warps 0-3: lazy O rescale, epilogue
//     per thread; P (bf16) and the           (normalise, prev merge)
//     rescale factor into shared memory
//   warp 6: one bulk copy of P and the factors into the O-CTA per tile
//
// The two CTAs hand P over through distributed shared memory with cluster-
// scope mbarrier arrivals.  The online softmax keeps a stale row maximum and
// only rescales O when the maximum grows by more than 2^8, so O rescales are
// rare.  Every wait is bounded; on a timeout a CTA records the wait site in
// the device status word, stops issuing work, lets in-flight copies and MMAs
// drain, and exits through the same cluster barrier as the normal path.
//
// Three sources of KV tiles share the engine:
//   prefill - dense [Tkv, 576] rows (TMA tile boxes); causal by global position
//   decode  - a paged latent cache; split-K: each CTA pair owns an equal share
//             of all requests' key tiles and writes per-request partials that
//             a reduction kernel merges (Mojo "mha_single_batch_pipelined")
//   sparse  - the top-k rows of each query, gathered with 16-byte cp.async into the
//             layout the TMA boxes give (AWS NKI "MLA Sparse Attention CTE Kernel
//             API Reference"); the c_kv and k_pe tensor maps are still encoded
//             (which validates the tensors) but no load uses them
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "mla_internal.h"
#include "mma_seq.cuh"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

// warps 0-3 rows, warp 4 TMA; S-CTA: warps 5 and 7 issue the S MMAs of even and odd tiles,
// warp 6 copies P out, and on the sparse path warp 9 copies half of each K tile's gathered
// rows (warp 8 has no role: warp 9 sits on another scheduler than warp 4).  O-CTA: warp 5
// issues P V.
constexpr int kThreadsDense = 256;
constexpr int kThreadsSparse = 320;
constexpr int kGatherWarp2 = 9;
constexpr int kStagesS = 2;  // stage g % 2 pairs with S buffer g % 2
constexpr int kStagesO = 3;
constexpr int kBoxBytes = kKeys * 128;                 // 64 rows x 128 B
constexpr int kStageBytesS = kKBoxes * kBoxBytes;      // 73728
constexpr int kStageBytesO = kVBoxes * kBoxBytes;      // 65536
constexpr int kPBytes = kRows * kKeys * 2;             // 16384

// shared memory map (offsets from a 1024-aligned base; identical in both CTAs)
constexpr int kOffStages = 0;
constexpr int kOffPS = kStagesS * kStageBytesS;        // S-CTA: P buffers (147456)
constexpr int kOffAlpha = kOffPS + 2 * kPBytes;        // S-CTA: rescale factors [2][128]
constexpr int kOffStats = kOffAlpha + 2 * kRows * 4;   // S-CTA: (m, l) [128][2]
constexpr int kOffPO = kStagesO * kStageBytesO;        // O-CTA: local P buffers (196608)
constexpr int kOffAlphaO = kOffPO + 2 * kPBytes;       // O-CTA: rescale factors [2][128] (229376)
constexpr int kOffBars = kOffAlphaO + 2 * kRows * 4;   // both: barriers (230400)
constexpr int kSmemUsed = kOffBars + 512;
constexpr int kSmemAlloc = kSmemUsed + 1024;
static_assert(kOffStats + kRows * 8 <= kOffBars, "S-CTA layout overlaps the barriers");
static_assert(kSmemAlloc <= 232448, "shared memory over the sm_103a limit");

constexpr uint32_t kTmemQ = 0;          // S-CTA: Q columns [0, 288)
constexpr uint32_t kTmemS = 288;        // S-CTA: S buffers [288, 416)
constexpr float kRescaleLog2 = 8.0f;    // rescale O only when the max grows by > 2^8

struct Bars {
  // S-CTA
  // s_go[b]: K tile g (b = g % 2) landed AND every row read S tile g-2 out of buffer b
  // (one arrival per row warp + the producer's expect_tx), so the MMA warp waits once per tile.
  // s_full[b]: the S MMA of tile g is done: S is ready, and stage b may be refilled.
  uint64_t s_go[2];
  uint64_t s_full[2];
  uint64_t q_full;
  uint64_t q_taken;         // both S issuers passed q_full of the current item (count 2)
  uint64_t stats_free;      // arrived remotely by the O-CTA rows
  uint64_t pwritten[2];     // S-CTA: all 128 rows wrote P tile b into the local buffer
  uint64_t pbuf_free[2];    // S-CTA: the bulk copy out of local P buffer b has been read
  // O-CTA
  uint64_t o_kv_full[kStagesO], o_kv_empty[kStagesO];
  uint64_t p_full[2];       // O-CTA: P tile b landed (bulk copy from the S-CTA, with its tx bytes)
  uint64_t p_ready[2];
  // both CTAs: pb_free[b] completes when the P V that read the O-CTA's P buffer b is
  // done (one multicast commit arrives on both copies; the S-CTA's copy gates the next
  // bulk copy into that buffer)
  uint64_t pb_free[2];
  uint64_t stats_full;      // arrived remotely by the S-CTA rows
  uint64_t o_free;
  uint64_t ep_half[2];      // O-CTA: both warps of an epilogue half staged their rows (count 2)
  uint64_t stall;           // fault injection: never arrived on
  uint64_t drain[2];        // abort: one commit of each MMA issuer lands here
  uint32_t tmem_base;
  uint32_t abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barrier block too large");

// wait-site ids (device status word detail)
enum : uint32_t {
  W_S_KV_EMPTY = 1, W_S_KV_FULL, W_S_SFREE, W_S_QFULL, W_S_SFULL, W_S_PFREE, W_S_STATSFREE, W_S_PWRITTEN,
  W_S_PBOFREE,
  W_O_KV_EMPTY, W_O_KV_FULL, W_O_PREADY, W_O_PFULL, W_O_PBFREE, W_O_PVDONE, W_O_STATSFULL, W_O_OFREE, W_STALL,
  W_O_EPHALF,
  R_PAGE = 0x40, R_LEN = 0x41,
};

// ---------------------------------------------------------------------------
// the work list of one CTA pair
// ---------------------------------------------------------------------------
struct Item {
  int id;          // prefill: row tile; decode: request; sparse: token
  int J;           // KV tiles
  int64_t k0;      // decode: first key (within the request) of this segment
  int64_t k1;      // decode: end key of this segment
  int slot;        // decode: partial slot
};

__device__ __forceinline__ int64_t prefill_keys_for_token(const CoreParams& p, int64_t t) {
  int64_t n = p.kv_valid;
  if (p.causal) {
    int64_t c = p.q_pos0 + t - p.kv_pos0 + 1;
    if (c < n) n = c;
  }
  return n < 0 ? 0 : n;
}

// keys seen by decode query group b (one query token of a request; see decode_group_len)
__device__ __forceinline__ int decode_len(const CoreParams& p, int b) { return decode_group_len(p, b); }

struct ItemIter {
  const CoreParams* p;
  int pair;
  int64_t k;        // prefill / sparse: running index
  // decode state
  int b;
  int64_t pre;
  int64_t lo, hi;

  __device__ void init(const CoreParams& prm, int pair_id) {
    p = &prm;
    pair = pair_id;
    k = pair_id;
    b = 0;
    pre = 0;
    if (prm.mode == MODE_DECODE) {
      int64_t tot = 0;
      for (int i = 0; i < prm.B; ++i) tot += (decode_len(prm, i) + kKeys - 1) / kKeys;
      lo = tot * pair_id / prm.num_pairs;
      hi = tot * (pair_id + 1) / prm.num_pairs;
    }
  }

  __device__ bool next(Item& it) {
    const CoreParams& P = *p;
    if (P.mode == MODE_PREFILL) {
      const int64_t rows = (int64_t)P.T * P.H;
      const int64_t n_items = (rows + kRows - 1) / kRows;
      if (k >= n_items) return false;
      const int64_t id = n_items - 1 - k;  // longest causal rows first
      k += P.num_pairs;
      int64_t last = id * kRows + kRows - 1;
      if (last >= rows) last = rows - 1;
      const int64_t n = prefill_keys_for_token(P, last / P.H);
      it.id = (int)id;
      it.J = (int)((n + kKeys - 1) / kKeys);
      // In place, a row that sees no key keeps its previous (out, lse) exactly; J only
      // falls along this order (causal) or is constant, so the rest of the list is done.
      if (it.J == 0 && P.prev_out && (const void*)P.prev_out == (const void*)P.out &&
          (const void*)P.prev_lse == (const void*)P.lse)
        return false;
      return true;
    }
    if (P.mode == MODE_SPARSE) {
      if (k >= P.T) return false;
      it.id = (int)k;
      it.J = (P.K + kKeys - 1) / kKeys;
      k += P.num_pairs;
      return true;
    }
    // decode: segments of requests overlapping [lo, hi); an empty share has none
    if (hi <= lo) return false;
    while (b < P.B) {
      const int len = decode_len(P, b);
      const int64_t nt = (len + kKeys - 1) / kKeys;
      const int64_t s = pre, e = pre + nt;
      const int cur = b;
      pre = e;
      ++b;
      if (nt == 0 || e <= lo) continue;  // no key, or wholly before this pair's share
      if (s >= hi) {
        b = P.B;
        return false;
      }
      const int64_t t0 = (s > lo ? s : lo) - s, t1 = (e < hi ? e : hi) - s;
      if (t1 <= t0) continue;
      it.id = cur;
      it.J = (int)(t1 - t0);
      it.k0 = t0 * kKeys;
      it.k1 = t1 * kKeys < len ? t1 * kKeys : len;
      it.slot = cur + pair;
      return true;
    }
    return false;
  }
};

constexpr int kRowWarps = kRows / 32;  // row barriers count warps (see warp_arrive)

// The query row (and for sparse its RoPE part) that row r of item `it` reads.
__device__ __forceinline__ bool query_row(const CoreParams& p, const Item& it, int r, const __nv_bfloat16*& qrow,
                                          const __nv_bfloat16*& qpe, int64_t& nkeys) {
  qrow = nullptr;
  qpe = nullptr;
  nkeys = 0;
  if (p.mode == MODE_PREFILL) {
    const int64_t f = (int64_t)it.id * kRows + r;
    if (f >= (int64_t)p.T * p.H) return false;
    const int64_t t = f / p.H, h = f - t * p.H;
    qrow = p.q + t * p.q_stride_t + h * p.q_stride_h;
    nkeys = prefill_keys_for_token(p, t);
    return true;
  }
  if (r >= p.H) return false;
  if (p.mode == MODE_DECODE) {
    qrow = p.q + ((int64_t)it.id * p.H + r) * kDk;
  } else {
    qrow = p.q + ((int64_t)it.id * p.H + r) * kLatent;
    qpe = p.q_pe + ((int64_t)it.id * p.H + r) * kRope;
  }
  return true;
}

// ---------------------------------------------------------------------------
// KV tile loaders (producer warp).  `dst` is a stage base; boxes [b0, b1).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void gather4(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y0, int32_t y1,
                                        int32_t y2, int32_t y3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(smem_u32(bar))
      : "memory");
}

// rows[i] for i in 0..63 held by lanes: lane l holds rows 2l and 2l+1.  Column
// boxes 0..7 come from map_lat at x = 64*box; box 8 (the RoPE columns) from
// map_pe at x = pe_x (512 on a [rows, 576] cache, 0 on a separate [rows, 64] tensor).
__device__ __forceinline__ void issue_gather_tile(uint32_t dst, const CUtensorMap* map_lat, const CUtensorMap* map_pe,
                                                  int32_t pe_x, int nboxes, int32_t r_even, int32_t r_odd,
                                                  uint64_t* bar) {
  const int lane = threadIdx.x & 31;
  // lane g (0..15) issues rows 4g..4g+3 = lanes 2g, 2g+1 (even/odd each)
  const int32_t a0 = __shfl_sync(0xffffffffu, r_even, (2 * lane) & 31);
  const int32_t a1 = __shfl_sync(0xffffffffu, r_odd, (2 * lane) & 31);
  const int32_t a2 = __shfl_sync(0xffffffffu, r_even, (2 * lane + 1) & 31);
  const int32_t a3 = __shfl_sync(0xffffffffu, r_odd, (2 * lane + 1) & 31);
  if (lane < 16) {
    for (int bx = 0; bx < nboxes; ++bx) {
      const CUtensorMap* m = (bx < kVBoxes) ? map_lat : map_pe;
      const int32_t x = (bx < kVBoxes) ? bx * kBoxCols : pe_x;
      gather4(dst + bx * kBoxBytes + lane * 512, m, x, a0, a1, a2, a3, bar);
    }
  }
}

// Raw top-k entries of tile j that lane l gathers (rows 2l and 2l+1 of the tile); -1 past K.
// Loaded a tile before their use, so the range check waits for that use (sparse_row).
__device__ __forceinline__ void sparse_tile_idx(const CoreParams& p, int id, int j, int32_t& re, int32_t& ro) {
  const int lane = threadIdx.x & 31;
  const int32_t* tk = p.topk + (int64_t)id * p.K;
  const int c0 = j * kKeys + 2 * lane;
  re = (c0 < p.K && guard_span(p.err, G_TOPK, tk + c0, 4, p.topk, p.ext_topk)) ? __ldg(tk + c0) : -1;
  ro = (c0 + 1 < p.K && guard_span(p.err, G_TOPK, tk + c0 + 1, 4, p.topk, p.ext_topk)) ? __ldg(tk + c0 + 1) : -1;
}

// A top-k entry outside [0, S_kv) is padding: no row (-1 gathers zeros).
__device__ __forceinline__ int32_t sparse_row(const CoreParams& p, int32_t r) {
  return (r < 0 || r >= p.S_kv) ? -1 : r;
}

// Gathered rows 8*q0 .. 8*q1-1 of a 64-row tile with 16-byte cp.async, in the layout of the
// SW128 boxes a tiled TMA load gives: the 512 latent columns (eight boxes) and, when k_pe is
// given, the 64 RoPE columns (the ninth).  A TMA gather moves one 128-byte row piece per
// request and runs at a fraction of the tiled rate on scattered rows; here each warp
// instruction moves 512 contiguous bytes of one latent row, or four 128-byte RoPE rows.
// Rows as in issue_gather_tile (lane l: rows 2l, 2l+1; -1 gives a zero row).  Every lane
// arrives on `bar` (noinc) once its copies have landed; the reader of the stage orders them
// before its async-proxy reads with a proxy fence.
__device__ __forceinline__ void lsu_gather_rows(uint32_t dst, const __nv_bfloat16* c_kv, const __nv_bfloat16* k_pe,
                                                int32_t r_even, int32_t r_odd, uint64_t* bar, int q0, int q1,
                                                const CoreParams& p) {
  const int lane = threadIdx.x & 31;
  // latent: lane copies pieces `lane` and `lane + 32` of each 1024-byte row: boxes lane/8 and
  // lane/8 + 4, 16-byte column lane % 8 (XOR the row's swizzle phase)
  const char* base = reinterpret_cast<const char*>(c_kv) + lane * 16;
  const uint32_t lp0 = (uint32_t)(lane >> 3) * kBoxBytes + ((uint32_t)(lane & 7) << 4);
  const uint32_t lp1 = lp0 + 4u * kBoxBytes;
#pragma unroll 1
  for (int q = q0; q < q1; ++q) {  // rows 8q..8q+7, held by lanes 4q..4q+3
    const uint32_t rb = dst + (uint32_t)q * 1024u;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      int32_t ri = __shfl_sync(0xffffffffu, (k & 1) ? r_odd : r_even, 4 * q + (k >> 1));
      if (ri >= 0 && !guard_span(p.err, G_C_KV, c_kv + (int64_t)ri * kLatent, kLatent * 2, p.c_kv, p.ext_c_kv)) ri = -1;
      const uint32_t n = ri >= 0 ? 16u : 0u;
      const char* src = base + (int64_t)(ri >= 0 ? ri : 0) * (kLatent * 2);
      cp_async16_zfill(rb + k * 128 + (lp0 ^ ((uint32_t)k << 4)), src, n);
      cp_async16_zfill(rb + k * 128 + (lp1 ^ ((uint32_t)k << 4)), src + 512, n);
    }
  }
  if (k_pe != nullptr) {
    // RoPE: lane copies piece lane % 8 of row 4i + lane / 8, for row groups i of these rows
    const int rr = lane >> 3, c = lane & 7;
    const char* pbase = reinterpret_cast<const char*>(k_pe) + c * 16;
    const uint32_t box = dst + (uint32_t)kVBoxes * kBoxBytes;
#pragma unroll 1
    for (int i = 2 * q0; i < 2 * q1; ++i) {
      const int row = 4 * i + rr;
      const int32_t ae = __shfl_sync(0xffffffffu, r_even, 2 * i + (rr >> 1));
      const int32_t ao = __shfl_sync(0xffffffffu, r_odd, 2 * i + (rr >> 1));
      int32_t ri = (rr & 1) ? ao : ae;
      if (ri >= 0 && !guard_span(p.err, G_K_PE, k_pe + (int64_t)ri * kRope, kRope * 2, p.k_pe, p.ext_k_pe)) ri = -1;
      cp_async16_zfill(box + (uint32_t)row * 128u + ((uint32_t)(c ^ (row & 7)) << 4),
                       pbase + (int64_t)(ri >= 0 ? ri : 0) * (kRope * 2), ri >= 0 ? 16u : 0u);
    }
  }
  cp_async_arrive_noinc(bar);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// One instantiation for the sparse path and one for prefill and decode: each carries only
// its own loaders (the shared code is sensitive to instruction-cache footprint).
template <bool kSparse>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kSparse ? kThreadsSparse : kThreadsDense, 1)
    mla_core_kernel(const __grid_constant__ CoreParams p, const __grid_constant__ CoreMaps maps) {
  const CUtensorMap& map_kv = maps.kv;
  const CUtensorMap& map_row = maps.row;
  const CUtensorMap& map_pe = maps.pe;
  const CUtensorMap& map_out = maps.out;
  const CUtensorMap& map_prev = maps.prev;
  // Prefill (128 flat rows per tile) and sparse with H a multiple of 64 stage
  // their output (and the previous output) through two V stages and TMA; decode
  // writes fp32 partials directly, and other head counts write bf16 rows directly.
  const bool staged = kSparse ? (p.H % 64) == 0 : p.mode == MODE_PREFILL;
  const int rows_per_item = (p.mode == MODE_PREFILL) ? kRows : p.H;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars& bars = *reinterpret_cast<Bars*>(smem + kOffBars);
  const uint32_t rank = cluster_ctarank();
  const bool is_s = (rank == 0);
  const int pair = blockIdx.x >> 1;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t lim = p.spin_limit;
  uint32_t* err = p.err;
  const uint32_t peer = rank ^ 1u;

  // ---- setup ----
  if (tid == 0) {
    if (is_s) {
      // sparse: one noinc arrival per lane of the two gathering warps instead of the
      // producer's expect-tx arrival
      for (int i = 0; i < 2; ++i) {
        mbar_init(&bars.s_go[i], kRowWarps + (kSparse ? 64 : 1));
        mbar_init(&bars.s_full[i], 1);
        mbar_init(&bars.pb_free[i], 1);
      }
      mbar_init(&bars.q_full, kRowWarps);
      mbar_init(&bars.q_taken, 2);
      mbar_init(&bars.stats_free, kRowWarps);
      for (int i = 0; i < 2; ++i) {
        mbar_init(&bars.pwritten[i], kRowWarps);
        mbar_init(&bars.pbuf_free[i], 1);
      }
    } else {
      for (int i = 0; i < kStagesO; ++i) {
        mbar_init(&bars.o_kv_full[i], 1 + (kSparse ? 32 : 0));
        mbar_init(&bars.o_kv_empty[i], 1);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(&bars.p_full[i], 1);
        mbar_init(&bars.pb_free[i], 1);
        mbar_init(&bars.p_ready[i], kRowWarps);
      }
      mbar_init(&bars.stats_full, kRowWarps);
      mbar_init(&bars.o_free, kRowWarps);
      mbar_init(&bars.ep_half[0], 2);
      mbar_init(&bars.ep_half[1], 2);
    }
    mbar_init(&bars.stall, 1);
    mbar_init(&bars.drain[0], 1);
    mbar_init(&bars.drain[1], 1);
    bars.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&map_kv);
    tma_prefetch_desc(&map_row);
    tma_prefetch_desc(&map_pe);
    if (staged) tma_prefetch_desc(&map_out);
    if (staged && p.prev_out) tma_prefetch_desc(&map_prev);
  }
  // decode: publish the per-request tile prefix for the reduction kernel
  if (p.mode == MODE_DECODE && blockIdx.x == 0 && warp == 0) {
    int64_t run = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + lane;
      int n = 0;
      if (b < p.B) {
        const int32_t* lp = p.lens + decode_request(p, b);
        const int raw = guard_span(err, G_LENS, lp, 4, p.lens, p.ext_lens) ? *lp : 0;
        const int64_t cap = (int64_t)p.max_pages * p.page_size;
        if (raw < 0 || raw > cap) record_error(err, DEV_RANGE_BASE | R_LEN);
        n = (decode_len(p, b) + kKeys - 1) / kKeys;
      }
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (b < p.B && guard_span(err, G_TILE_PREFIX, p.tile_prefix + b, 4, p.tile_prefix, p.ext_tile_prefix))
        p.tile_prefix[b] = (int32_t)(run + incl - n);
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0 && guard_span(err, G_TILE_PREFIX, p.tile_prefix + p.B, 4, p.tile_prefix, p.ext_tile_prefix))
      p.tile_prefix[p.B] = (int32_t)run;
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised before any remote arrive
  tc_fence_after();
  const uint32_t tbase = bars.tmem_base;
  volatile uint32_t* abort_flag = &bars.abort_flag;
  // Every wait is made by a whole warp and its outcome is warp-uniform, so no
  // warp reaches a warp-collective tcgen05 instruction with some lanes gone.
  auto waitb = [&](uint64_t* bar, uint32_t parity, uint32_t site, bool cl) -> bool {
    bool ok = (*abort_flag == 0) && mbar_wait(bar, parity, err, site, lim, cl);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) *abort_flag = 1;
    return ok;
  };

  ItemIter iter;
  iter.init(p, pair);
  Item it;
  // abort drain: the last barrier phase this thread's TMA loads were counted on
  uint64_t* drain_bar = nullptr;
  uint32_t drain_par = 0;
  if (p.debug_stall && warp == 5) waitb(&bars.stall, 0, W_STALL, false);  // runs out: injected fault

  if (is_s) {
    // =====================================================================
    // S-CTA
    // =====================================================================
    if (warp == 4 || (kSparse && warp == kGatherWarp2)) {
      // ---------------- TMA producer: K tiles (all 576 columns) ----------------
      uint32_t g = 0;
      bool live = true;
      while (live && iter.next(it)) {
        int32_t nre = -1, nro = -1;  // sparse: top-k entries of the next tile, loaded a tile ahead
        if (kSparse && it.J > 0) sparse_tile_idx(p, it.id, 0, nre, nro);
        // decode with pages of whole tiles: block-table entry of the next tile, loaded a tile ahead
        const bool whole_pages = !kSparse && p.mode == MODE_DECODE && p.page_size % kKeys == 0;
        int32_t npg = -1;
        if (whole_pages && it.J > 0)
          npg = bt_entry(p, p.block_table + (int64_t)decode_request(p, it.id) * p.max_pages + it.k0 / p.page_size);
        for (int j = 0; j < it.J && live; ++j, ++g) {
          const int s = g & 1;
          // stage s was last read by the S MMA of tile g-2
          if (!waitb(&bars.s_full[s], ((g >> 1) & 1) ^ 1, W_S_KV_EMPTY, false)) { live = false; break; }
          const uint32_t dst = smem_u32(smem + kOffStages + s * kStageBytesS);
          if (!kSparse && p.mode == MODE_PREFILL) {
            if (lane == 0) {
              mbar_arrive_expect_tx(&bars.s_go[s], kStageBytesS);
              for (int bx = 0; bx < kKBoxes; ++bx)
                tma_load_2d(dst + bx * kBoxBytes, &map_kv, bx * kBoxCols, j * kKeys, &bars.s_go[s]);
            }
            drain_bar = &bars.s_go[s];
            drain_par = (g >> 1) & 1;
          } else {
            int32_t re = -1, ro = -1;
            bool tiled = false;
            int32_t ytile = 0;
            if constexpr (!kSparse) {
              const int64_t kb = it.k0 + (int64_t)j * kKeys;  // first key of the tile
              const int len = decode_len(p, it.id);
              const int32_t* bt = p.block_table + (int64_t)decode_request(p, it.id) * p.max_pages;
              auto row_of = [&](int64_t key) -> int32_t {
                if (key >= len) return -1;
                const int32_t pg = bt_entry(p, bt + key / p.page_size);
                if (pg < 0 || pg >= p.num_pages) {
                  record_error(err, DEV_RANGE_BASE | R_PAGE);
                  return -1;
                }
                return (int32_t)(pg * (int64_t)p.page_size + key % p.page_size);
              };
              // pages that hold whole tiles: this tile's entry was loaded a tile ago
              const int32_t pg = npg;
              if (whole_pages && j + 1 < it.J) npg = bt_entry(p, bt + (kb + kKeys) / p.page_size);
              if (whole_pages && kb + kKeys <= len && pg >= 0 && pg < p.num_pages) {
                tiled = true;
                ytile = (int32_t)(pg * (int64_t)p.page_size + kb % p.page_size);
              } else {
                re = row_of(kb + 2 * lane);
                ro = row_of(kb + 2 * lane + 1);
              }
            } else {
              re = sparse_row(p, nre);
              ro = sparse_row(p, nro);
              if (j + 1 < it.J) sparse_tile_idx(p, it.id, j + 1, nre, nro);  // lands during this gather
            }
            if constexpr (kSparse) {
              // all 576 columns by 16-byte copies: warp 4 copies rows 0-31, warp 9 rows 32-63
              const int q0 = (warp == 4) ? 0 : kKeys / 16;
              lsu_gather_rows(dst, p.c_kv, p.k_pe, re, ro, &bars.s_go[s], q0, q0 + kKeys / 16, p);
            } else {
              if (lane == 0) mbar_arrive_expect_tx(&bars.s_go[s], kStageBytesS);
              __syncwarp();
              drain_bar = &bars.s_go[s];
              drain_par = (g >> 1) & 1;
              if (tiled) {
                if (lane == 0)
                  for (int bx = 0; bx < kKBoxes; ++bx)
                    tma_load_2d(dst + bx * kBoxBytes, &map_kv, bx * kBoxCols, ytile, &bars.s_go[s]);
              } else {
                issue_gather_tile(dst, &map_row, &map_pe, kLatent, kKBoxes, re, ro, &bars.s_go[s]);
              }
            }
          }
          __syncwarp();
        }
      }
      if (kSparse) cp_async_wait_all();  // no copy into this CTA outlives it
    } else if (warp == 5 || warp == 7) {
      // ---------------- MMA issuers: S = Q K^T ----------------
      // Two warps take turns, warp 5 the even tiles and warp 7 the odd ones; each owns one K
      // stage and one S buffer (index g % 2).  A barrier wait by the thread that issued MMAs
      // stalls until its queued MMAs drain, so with one issuer the tensor pipe idles at every
      // tile boundary; the second issuer's queued tile covers that gap.  One thread per warp
      // runs the loop (these warps issue no warp-collective tcgen05 instruction here).
      if (lane == 0) {
        const uint32_t b = (warp == 5) ? 0u : 1u;
        const uint32_t idesc = idesc_bf16_f32(kRows, kKeys, false, false);
        auto wait1 = [&](uint64_t* bar, uint32_t parity, uint32_t site) -> bool {
          const bool ok = (*abort_flag == 0) && mbar_wait(bar, parity, err, site, lim, false);
          if (!ok) *abort_flag = 1;
          return ok;
        };
        const uint32_t stage = smem_u32(smem + kOffStages + b * kStageBytesS);
        const uint64_t bdesc = sdesc_sw128(stage, 16, 1024);
        const uint32_t d_tmem = tbase + kTmemS + b * kKeys;
        uint32_t g = 0, i = 0;  // i counts items that have KV tiles
        bool live = true;
        while (live && iter.next(it)) {
          if (it.J == 0) continue;  // no key: the O-CTA writes these rows on its own
          // every item's Q is waited for by both issuers, so neither can read q_full a phase
          // ahead: the rows write the next item's Q only after both have arrived on q_taken
          if (!wait1(&bars.q_full, i & 1, W_S_QFULL)) break;
          mbar_arrive(&bars.q_taken);
          for (int j = 0; j < it.J; ++j, ++g) {
            if ((g & 1u) != b) continue;
            if (!wait1(&bars.s_go[b], (g >> 1) & 1, W_S_KV_FULL)) {
              live = false;
              break;
            }
            if (kSparse) fence_proxy_async_smem();  // cp.async rows, read by the MMA
            tc_fence_after();
            mma_s_q576_n64(d_tmem, tbase + kTmemQ, bdesc, idesc);
            mma_commit(&bars.s_full[b]);
          }
          ++i;
        }
      }
      __syncwarp();
    } else if (warp == 6) {
      // ---------------- P hand-over: one bulk copy per tile into the O-CTA ----------------
      // Kept off the softmax warps: waiting for a copy to be read would otherwise delay
      // one row warp, and every S tile waits for all 128 rows.
      uint8_t* pbuf = smem + kOffPS;
      float* alpha = reinterpret_cast<float*>(smem + kOffAlpha);
      const uint32_t rem_p_full0 = map_to_rank(smem_u32(&bars.p_full[0]), peer);
      const uint32_t rem_p_full1 = map_to_rank(smem_u32(&bars.p_full[1]), peer);
      const uint32_t rem_p_o = map_to_rank(smem_u32(smem + kOffPO), peer);          // O-CTA P buffers
      const uint32_t rem_alpha_o = map_to_rank(smem_u32(smem + kOffAlphaO), peer);  // O-CTA factors
      uint32_t g = 0;
      bool live = true;
      while (live && iter.next(it)) {
        for (int j = 0; j < it.J; ++j, ++g) {
          const int sb = g & 1;
          // every row wrote P tile g, and the O-CTA's buffer sb is free (its P V of tile g-2 is done)
          if (!waitb(&bars.pwritten[sb], (g >> 1) & 1, W_S_PWRITTEN, false) ||
              !waitb(&bars.pb_free[sb], ((g >> 1) & 1) ^ 1, W_S_PBOFREE, true)) {
            live = false;
            break;
          }
          if (lane == 0) {
            const uint32_t bar = sb ? rem_p_full1 : rem_p_full0;
            mbar_arrive_expect_tx_remote(bar, kPBytes + kRows * 4);
            bulk_copy_to_peer(rem_p_o + sb * kPBytes, smem_u32(pbuf + sb * kPBytes), kPBytes, bar);
            bulk_copy_to_peer(rem_alpha_o + sb * kRows * 4, smem_u32(alpha + sb * kRows), kRows * 4, bar);
            bulk_commit();
            // two copies in flight: once every group but this one has been read, the local
            // buffer of tile g-1 is free
            bulk_wait_read_le1();
            if (g > 0) mbar_arrive(&bars.pbuf_free[sb ^ 1]);
          }
          __syncwarp();
        }
      }
      if (lane == 0) {
        bulk_wait_all();  // our shared memory is read until the copies end
        if (g > 0) mbar_arrive(&bars.pbuf_free[(g - 1) & 1]);
      }
    } else if (warp < 4) {
      // ---------------- rows: Q load, online softmax, P hand-over ----------------
      const int r = tid;  // row within the tile = TMEM lane
      const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
      uint8_t* pbuf = smem + kOffPS;
      float* alpha = reinterpret_cast<float*>(smem + kOffAlpha);
      float* stats = reinterpret_cast<float*>(smem + kOffStats);
      const uint32_t rem_stats_full = map_to_rank(smem_u32(&bars.stats_full), peer);
      uint32_t g = 0, i = 0;  // i counts items that have KV tiles
      bool live = true;
      // both S buffers start free (the row arrivals of tiles 0 and 1)
      warp_arrive(&bars.s_go[0]);
      warp_arrive(&bars.s_go[1]);
      while (live && iter.next(it)) {
        if (it.J == 0) continue;  // no key: the O-CTA writes these rows on its own
        // ---- this row's query and key limit ----
        const __nv_bfloat16* qrow;
        const __nv_bfloat16* qpe;
        int64_t nkeys;  // prefill: keys visible to the row
        const bool row_ok = query_row(p, it, r, qrow, qpe, nkeys);
        // warm L2 with the next item's query row while this item runs
        {
          ItemIter peek = iter;
          Item nx;
          bool found = false;
          while (peek.next(nx)) {
            if (nx.J > 0) {
              found = true;
              break;
            }
          }
          const __nv_bfloat16 *nq, *npe;
          int64_t nk;
          if (found && query_row(p, nx, r, nq, npe, nk)) {
            const char* b = reinterpret_cast<const char*>(nq);
            const int nbytes = kSparse ? kLatent * 2 : kDk * 2;
            for (int o = 0; o < nbytes; o += 128) prefetch_l2(b + o);
            if (npe) prefetch_l2(npe);
          }
        }
        // ---- Q -> TMEM (bf16 pairs, K-contiguous): 9 chunks of 64 columns, 3 in flight ----
        // (both issuers took the previous item's Q signal; its MMAs are done, since every S
        // tile of that item has been read)
        if (i > 0 && !waitb(&bars.q_taken, (i - 1) & 1, W_S_QFULL, false)) break;
#pragma unroll 1
        for (int c0 = 0; c0 < kDk / 64; c0 += 3) {
          uint4 x[3][8];
#pragma unroll
          for (int cc = 0; cc < 3; ++cc) {
            const int c = c0 + cc;
            const uint4* src = nullptr;
            if (row_ok) {
              if (kSparse)
                src = (c < 8) ? reinterpret_cast<const uint4*>(qrow + c * 64) : reinterpret_cast<const uint4*>(qpe);
              else
                src = reinterpret_cast<const uint4*>(qrow + c * 64);
              const bool pe_part = kSparse && c >= 8;
              if (!guard_span(err, pe_part ? G_Q_PE : G_Q, src, 128, pe_part ? (const void*)p.q_pe : (const void*)p.q,
                              pe_part ? p.ext_q_pe : p.ext_q))
                src = nullptr;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) x[cc][u] = src ? __ldg(src + u) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int cc = 0; cc < 3; ++cc) {
            uint32_t v[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              v[4 * u + 0] = x[cc][u].x;
              v[4 * u + 1] = x[cc][u].y;
              v[4 * u + 2] = x[cc][u].z;
              v[4 * u + 3] = x[cc][u].w;
            }
            tmem_st32(tbase + lane_base + kTmemQ + (c0 + cc) * 32, v);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(&bars.q_full);

        float m_used = -CUDART_INF_F;  // log2-domain offset of the exponentials
        float l = 0.f;                 // running row sum (relative to m_used)
        for (int j = 0; j < it.J; ++j, ++g) {
          const int sb = g & 1;
          // ---- per-tile key validity mask ----
          uint64_t vmask;
          if (!kSparse && p.mode == MODE_PREFILL) {
            int64_t nv = nkeys - (int64_t)j * kKeys;
            nv = nv < 0 ? 0 : (nv > 64 ? 64 : nv);
            vmask = (nv == 64) ? ~0ull : ((1ull << nv) - 1ull);
          } else if (!kSparse) {
            int64_t nv = it.k1 - (it.k0 + (int64_t)j * kKeys);
            nv = nv < 0 ? 0 : (nv > 64 ? 64 : nv);
            vmask = (nv == 64) ? ~0ull : ((1ull << nv) - 1ull);
          } else {
            const int32_t* tk = p.topk + (int64_t)it.id * p.K;
            const int c0 = j * kKeys + lane, c1 = c0 + 32;
            const int32_t i0 = (c0 < p.K && guard_span(err, G_TOPK, tk + c0, 4, p.topk, p.ext_topk)) ? tk[c0] : -1;
            const int32_t i1 = (c1 < p.K && guard_span(err, G_TOPK, tk + c1, 4, p.topk, p.ext_topk)) ? tk[c1] : -1;
            const uint32_t lo = __ballot_sync(0xffffffffu, i0 >= 0 && i0 < p.S_kv);
            const uint32_t hi = __ballot_sync(0xffffffffu, i1 >= 0 && i1 < p.S_kv);
            vmask = ((uint64_t)hi << 32) | lo;
          }
          if (!row_ok) vmask = 0;

          if (!waitb(&bars.s_full[sb], (g >> 1) & 1, W_S_SFULL, false)) { live = false; break; }
          tc_fence_after();
          // Scores in the log2 domain: t = s * scale * log2(e); the row maximum is taken on the
          // raw dot products (their largest, or their smallest when the scale is negative).
          // Two passes over the tile in 32-column pieces read from TMEM, each a rolled loop:
          // fully unrolled 64-column loops made the row loop too large for the instruction
          // cache, which slowed these warps several times over.
          const uint32_t scol = tbase + lane_base + kTmemS + sb * kKeys;
          const float sl2 = p.scale_log2;
          const bool up = sl2 >= 0.f;
          float eq[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) eq[k] = up ? -CUDART_INF_F : CUDART_INF_F;
#pragma unroll 1
          for (int p32 = 0; p32 < kKeys / 32; ++p32) {
            uint32_t sr[32];
            tmem_ld32(scol + 32 * p32, sr);
            tmem_wait_ld();
            const uint32_t vm = (uint32_t)(vmask >> (32 * p32));
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const float v = __uint_as_float(sr[c]);
              const bool ok = (vm >> c) & 1u;
              eq[c & 3] = !ok ? eq[c & 3] : (up ? fmaxf(eq[c & 3], v) : fminf(eq[c & 3], v));
            }
          }
          const float ext = up ? fmaxf(fmaxf(eq[0], eq[1]), fmaxf(eq[2], eq[3]))
                               : fminf(fminf(eq[0], eq[1]), fminf(eq[2], eq[3]));
          const float mt = (vmask == 0ull) ? -CUDART_INF_F : ext * sl2;
          float a = 1.f;
          if (mt > m_used + kRescaleLog2) {
            if (l > 0.f) a = ex2_approx(m_used - mt);
            l *= a;
            m_used = mt;
          }
          if (j == 0) a = 1.f;  // the first P V overwrites O
          const float msub = (m_used == -CUDART_INF_F) ? 0.f : m_used;

          // ---- P into the local buffer (the copy warp hands it to the O-CTA) ----
          // local buffer sb was last read by the copy of tile g-2
          if (!waitb(&bars.pbuf_free[sb], ((g >> 1) & 1) ^ 1, W_S_PFREE, false)) { live = false; break; }
          uint8_t* prow = pbuf + sb * kPBytes + r * 128;
          float rsq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
          for (int p32 = 0; p32 < kKeys / 32; ++p32) {
            uint32_t sr[32];
            tmem_ld32(scol + 32 * p32, sr);
            tmem_wait_ld();
            const uint32_t vm = (uint32_t)(vmask >> (32 * p32));
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {  // 8 keys -> one 16-byte chunk of P
              uint32_t w[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int c = 8 * c8 + 2 * u;
                float e0 = ex2_approx(fmaf(__uint_as_float(sr[c]), sl2, -msub));
                float e1 = ex2_approx(fmaf(__uint_as_float(sr[c + 1]), sl2, -msub));
                e0 = ((vm >> c) & 1u) ? e0 : 0.f;
                e1 = ((vm >> (c + 1)) & 1u) ? e1 : 0.f;
                rsq[u] += e0 + e1;
                w[u] = pack_bf16x2(e0, e1);
              }
              const int kc = 4 * p32 + c8;
              *reinterpret_cast<uint4*>(prow + ((kc ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
          tc_fence_before();
          warp_arrive(&bars.s_go[sb]);  // S buffer sb has been read: it may take tile g+2
          l += (rsq[0] + rsq[1]) + (rsq[2] + rsq[3]);
          alpha[sb * kRows + r] = a;
          fence_proxy_async_smem();  // the bulk copy reads through the async proxy
          warp_arrive(&bars.pwritten[sb]);
        }
        if (!live) break;
        // ---- row statistics for the epilogue ----
        if (!waitb(&bars.stats_free, (i & 1) ^ 1, W_S_STATSFREE, true)) break;
        stats[2 * r] = m_used;
        stats[2 * r + 1] = l;
        warp_arrive_remote(rem_stats_full);
        ++i;
      }
    }
  } else {
    // =====================================================================
    // O-CTA
    // =====================================================================
    if (warp == 4) {
      // ---------------- TMA producer: V tiles (first 512 columns) ----------------
      uint32_t g = 0;  // position in the stage ring
      bool live = true;
      while (live && iter.next(it)) {
        int32_t nre = -1, nro = -1;  // sparse: top-k entries of the next tile, loaded a tile ahead
        if (kSparse && it.J > 0) sparse_tile_idx(p, it.id, 0, nre, nro);
        // decode with pages of whole tiles: block-table entry of the next tile, loaded a tile ahead
        const bool whole_pages = !kSparse && p.mode == MODE_DECODE && p.page_size % kKeys == 0;
        int32_t npg = -1;
        if (whole_pages && it.J > 0)
          npg = bt_entry(p, p.block_table + (int64_t)decode_request(p, it.id) * p.max_pages + it.k0 / p.page_size);
        for (int j = 0; j < it.J && live; ++j, ++g) {
          const int s = g % kStagesO;
          if (!waitb(&bars.o_kv_empty[s], ((g / kStagesO) & 1) ^ 1, W_O_KV_EMPTY, false)) { live = false; break; }
          const uint32_t dst = smem_u32(smem + kOffStages + s * kStageBytesO);
          if (!kSparse && p.mode == MODE_PREFILL) {
            if (lane == 0) {
              mbar_arrive_expect_tx(&bars.o_kv_full[s], kStageBytesO);
              for (int bx = 0; bx < kVBoxes; ++bx)
                tma_load_2d(dst + bx * kBoxBytes, &map_kv, bx * kBoxCols, j * kKeys, &bars.o_kv_full[s]);
            }
            drain_bar = &bars.o_kv_full[s];
            drain_par = (g / kStagesO) & 1;
          } else {
            int32_t re = -1, ro = -1;
            bool tiled = false;
            int32_t ytile = 0;
            if constexpr (!kSparse) {
              const int64_t kb = it.k0 + (int64_t)j * kKeys;
              const int len = decode_len(p, it.id);
              const int32_t* bt = p.block_table + (int64_t)decode_request(p, it.id) * p.max_pages;
              auto row_of = [&](int64_t key) -> int32_t {
                if (key >= len) return -1;
                const int32_t pg = bt_entry(p, bt + key / p.page_size);
                if (pg < 0 || pg >= p.num_pages) return -1;
                return (int32_t)(pg * (int64_t)p.page_size + key % p.page_size);
              };
              // pages that hold whole tiles: this tile's entry was loaded a tile ago
              const int32_t pg = npg;
              if (whole_pages && j + 1 < it.J) npg = bt_entry(p, bt + (kb + kKeys) / p.page_size);
              if (whole_pages && kb + kKeys <= len && pg >= 0 && pg < p.num_pages) {
                tiled = true;
                ytile = (int32_t)(pg * (int64_t)p.page_size + kb % p.page_size);
              } else {
                re = row_of(kb + 2 * lane);
                ro = row_of(kb + 2 * lane + 1);
              }
            } else {
              re = sparse_row(p, nre);
              ro = sparse_row(p, nro);
              if (j + 1 < it.J) sparse_tile_idx(p, it.id, j + 1, nre, nro);  // lands during this gather
            }
            if constexpr (kSparse) {
              if (lane == 0) mbar_arrive(&bars.o_kv_full[s]);
              lsu_gather_rows(dst, p.c_kv, nullptr, re, ro, &bars.o_kv_full[s], 0, kKeys / 8, p);
            } else {
              if (lane == 0) mbar_arrive_expect_tx(&bars.o_kv_full[s], kStageBytesO);
              __syncwarp();
              drain_bar = &bars.o_kv_full[s];
              drain_par = (g / kStagesO) & 1;
              if (tiled) {
                if (lane == 0)
                  for (int bx = 0; bx < kVBoxes; ++bx)
                    tma_load_2d(dst + bx * kBoxBytes, &map_kv, bx * kBoxCols, ytile, &bars.o_kv_full[s]);
              } else {
                issue_gather_tile(dst, &map_row, &map_pe, 0, kVBoxes, re, ro, &bars.o_kv_full[s]);
              }
            }
          }
          __syncwarp();
        }
        // two more ring stages stage the epilogue of this item: rows 0-63 and 64-127,
        // holding the previous output when there is one
        if (staged && it.J > 0) {
          for (int hh = 0; hh < 2 && live; ++hh, ++g) {
            const int s = g % kStagesO;
            if (!waitb(&bars.o_kv_empty[s], ((g / kStagesO) & 1) ^ 1, W_O_KV_EMPTY, false)) { live = false; break; }
            if (lane == 0) {
              const int64_t row0 = (int64_t)it.id * kRows + hh * 64;
              if (p.prev_out && row0 < (int64_t)p.T * p.H) {
                const uint32_t dst = smem_u32(smem + kOffStages + s * kStageBytesO);
                mbar_arrive_expect_tx(&bars.o_kv_full[s], kStageBytesO);
                for (int bx = 0; bx < kVBoxes; ++bx)
                  tma_load_2d(dst + bx * kBoxBytes, &map_prev, bx * kBoxCols, (int32_t)row0, &bars.o_kv_full[s]);
                drain_bar = &bars.o_kv_full[s];
                drain_par = (g / kStagesO) & 1;
              } else {
                mbar_arrive(&bars.o_kv_full[s]);
              }
            }
            if (kSparse) mbar_arrive(&bars.o_kv_full[s]);  // the lanes' share of the count
            __syncwarp();
          }
        }
      }
      if (kSparse) cp_async_wait_all();  // no copy into this CTA outlives it
    } else if (warp == 5) {
      // ---------------- MMA issuer: O += P V ----------------
      const uint32_t idesc = idesc_bf16_f32(kRows, 256, false, true);
      uint32_t g = 0, gs = 0, i = 0;  // P tiles, stage ring position, items that have KV tiles
      bool live = true;
      while (live && iter.next(it)) {
        if (it.J == 0) continue;
        if (i > 0 && !waitb(&bars.o_free, (i - 1) & 1, W_O_OFREE, false)) break;
        for (int j = 0; j < it.J; ++j, ++g, ++gs) {
          const int s = gs % kStagesO;
          const int pb = g & 1;
          if (!waitb(&bars.o_kv_full[s], (gs / kStagesO) & 1, W_O_KV_FULL, false) ||
              !waitb(&bars.p_ready[pb], (g >> 1) & 1, W_O_PREADY, false)) {
            live = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
            if (kSparse) fence_proxy_async_smem();  // cp.async rows, read by the MMA
            const uint32_t vst = smem_u32(smem + kOffStages + s * kStageBytesO);
            const uint32_t pst = smem_u32(smem + kOffPO + pb * kPBytes);
            mma_pv_k64_n512(tbase, tbase + 256, sdesc_sw128(pst, 16, 1024), sdesc_sw128(vst, kBoxBytes, 1024),
                            sdesc_sw128(vst + 4 * kBoxBytes, kBoxBytes, 1024), idesc, j > 0 ? 1u : 0u);
            mma_commit(&bars.o_kv_empty[s]);
            mma_commit_multicast(&bars.pb_free[pb], 0x3);  // this CTA and the S-CTA
          }
          __syncwarp();
        }
        if (staged) gs += 2;  // the epilogue's two stages
        ++i;
      }
    } else if (warp < 4) {
      // ---------------- rows: lazy rescale, epilogue ----------------
      const int r = tid;
      const int half = r >> 6;   // warps 0-1: rows 0-63, warps 2-3: rows 64-127
      const int rr = r & 63;
      const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
      const uint32_t rem_stats = map_to_rank(smem_u32(smem + kOffStats), peer);
      const uint32_t rem_stats_free = map_to_rank(smem_u32(&bars.stats_free), peer);
      const float* alpha_o = reinterpret_cast<const float*>(smem + kOffAlphaO);
      uint32_t g = 0, gs = 0, i = 0;  // P tiles, stage ring position, items that have KV tiles
      uint32_t ep_phase = 0;          // staged epilogues done (phase of ep_half)
      bool live = true;
      bool stored = false;            // this thread issued TMA stores that must finish before exit
      while (live && iter.next(it)) {
        // ---- destination of this row ----
        bool row_ok = false;
        float prev_l = -CUDART_INF_F;
        const __nv_bfloat16* prev_row = nullptr;
        __nv_bfloat16* orow = nullptr;
        float* orow_f = nullptr;
        float* lse_dst = nullptr;
        if (!kSparse && p.mode == MODE_PREFILL) {
          const int64_t f = (int64_t)it.id * kRows + r;
          if (f < (int64_t)p.T * p.H) {
            const int64_t t = f / p.H, h = f - t * p.H;
            row_ok = true;
            orow = p.out + f * kLatent;
            lse_dst = p.lse + h * (p.lse_stride ? p.lse_stride : (int64_t)p.T) + t;
            if (p.prev_out) {
              prev_row = p.prev_out + f * kLatent;
              const float* pl = p.prev_lse + h * (p.lse_stride ? p.lse_stride : (int64_t)p.T) + t;
              prev_l = guard_span(err, G_PREV_LSE, pl, 4, p.prev_lse, p.ext_prev_lse) ? *pl : -CUDART_INF_F;
            }
          }
        } else if (!kSparse) {
          if (r < p.H) {
            row_ok = true;
            orow_f = p.part_o + ((int64_t)it.slot * p.H + r) * kLatent;
            lse_dst = p.part_lse + (int64_t)it.slot * p.H + r;
          }
        } else {
          if (r < p.H) {
            row_ok = true;
            orow = p.out + ((int64_t)it.id * p.H + r) * kLatent;
            lse_dst = p.lse ? p.lse + (int64_t)it.id * p.H + r : nullptr;
          }
        }

        // guarded build: a row outside its buffer is not written (or read) at all
        if (orow && !guard_span(err, G_OUT, orow, kLatent * 2, p.out, p.ext_out)) orow = nullptr;
        if (orow_f && !guard_span(err, G_PART_O, orow_f, kLatent * 4, p.part_o, p.ext_part_o)) orow_f = nullptr;
        if (prev_row && !guard_span(err, G_PREV_OUT, prev_row, kLatent * 2, p.prev_out, p.ext_prev_out)) prev_row = nullptr;
        if (lse_dst) {
          const bool part = !kSparse && p.mode != MODE_PREFILL;
          if (!guard_span(err, part ? G_PART_LSE : G_LSE, lse_dst, 4, part ? (const void*)p.part_lse : (const void*)p.lse,
                          part ? p.ext_part_lse : p.ext_lse))
            lse_dst = nullptr;
        }
        if (it.J == 0) {
          // no key reaches these rows: out = prev (or 0), lse = prev_lse (or -inf).
          // Only prefill and sparse produce such items; decode segments always hold keys.
          if (row_ok && orow) {
            for (int c = 0; c < kLatent; c += 8) {
              uint4 v = prev_row ? *reinterpret_cast<const uint4*>(prev_row + c) : make_uint4(0, 0, 0, 0);
              *reinterpret_cast<uint4*>(orow + c) = v;
            }
            if (lse_dst) *lse_dst = prev_row ? prev_l : -CUDART_INF_F;
          }
          continue;
        }

        for (int j = 0; j < it.J; ++j, ++g, ++gs) {
          const int pb = g & 1;
          // P tile g and its rescale factors landed in the local buffer pb (bulk copy)
          if (!waitb(&bars.p_full[pb], (g >> 1) & 1, W_O_PFULL, true)) {
            live = false;
            break;
          }
          const float a = alpha_o[pb * kRows + r];
          // tcgen05.ld/st are warp-collective: rescale when any row of the warp needs it
          if (__any_sync(0xffffffffu, a != 1.f)) {
            // O must hold every earlier P V before it is rescaled: PV(g-1) is use
            // (g-1)/2 of P buffer (g-1)%2, and no later use of that buffer can start yet
            if (!waitb(&bars.pb_free[(g - 1) & 1], ((g - 1) >> 1) & 1, W_O_PVDONE, false)) { live = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < kLatent; c0 += 32) {
              uint32_t v[32];
              tmem_ld32(tbase + lane_base + c0, v);
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * a);
              tmem_st32(tbase + lane_base + c0, v);
            }
            tmem_wait_st();
          }
          tc_fence_before();
          warp_arrive(&bars.p_ready[pb]);
        }
        if (!live) break;

        // ---- epilogue ----
        if (!waitb(&bars.stats_full, i & 1, W_O_STATSFULL, true)) break;
        float m_used, l;
        asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(m_used) : "r"(rem_stats + r * 8));
        asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(l) : "r"(rem_stats + r * 8 + 4));
        warp_arrive_remote(rem_stats_free);
        // the last P V of the item: use (g-1)/2 of P buffer (g-1)%2
        if (!waitb(&bars.pb_free[(g - 1) & 1], ((g - 1) >> 1) & 1, W_O_PVDONE, false)) break;
        tc_fence_after();
        const bool has = l > 0.f;
        const float inv_l = has ? 1.f / l : 0.f;
        const float lse_new = has ? (m_used + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
        // merge weights with the previous pair (weight 0 for an empty side)
        float wn = has ? 1.f : 0.f, wp = 0.f, lse_out = lse_new;
        if (row_ok && prev_row) {
          const float m = fmaxf(prev_l, lse_new);
          if (m == -CUDART_INF_F) {
            wn = 0.f;
            wp = 0.f;
            lse_out = -CUDART_INF_F;
          } else {
            wp = (prev_l == -CUDART_INF_F) ? 0.f : expf(prev_l - m);
            wn = has ? expf(lse_new - m) : 0.f;
            const float ws = wp + wn;
            lse_out = m + logf(ws);
            wp /= ws;
            wn /= ws;
          }
        }
        const float cn = wn * inv_l;

        if (staged) {
          // rows of this half live in ring stage gs + half, [8 column boxes][64 rows][128 B] swizzled
          const uint32_t sidx = gs + half;
          const int s = sidx % kStagesO;
          if (!waitb(&bars.o_kv_full[s], (sidx / kStagesO) & 1, W_O_KV_FULL, false)) break;
          uint8_t* stage = smem + kOffStages + s * kStageBytesO;
          const bool use_prev = (prev_row != nullptr) && wp > 0.f;
#pragma unroll 1
          for (int c0 = 0; c0 < kLatent; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tbase + lane_base + c0, v);
            tmem_wait_ld();
            uint8_t* rowp = stage + (c0 >> 6) * kBoxBytes + rr * 128;
            const int g0 = (c0 & 63) >> 3;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              uint4* cell = reinterpret_cast<uint4*>(rowp + (((g0 + u) ^ (rr & 7)) << 4));
              float o[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) o[k] = __uint_as_float(v[8 * u + k]) * cn;
              if (use_prev) {
                const uint4 x = *cell;
                const __nv_bfloat162* hx = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const float2 f2 = __bfloat1622float2(hx[k]);
                  o[2 * k] += wp * f2.x;
                  o[2 * k + 1] += wp * f2.y;
                }
              }
              *cell = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                                 pack_bf16x2(o[6], o[7]));
            }
          }
          // O has been read: the next item's P V may start
          tc_fence_before();
          warp_arrive(&bars.o_free);
          if (row_ok && lse_dst) *lse_dst = lse_out;
          // the 64 rows of this half go out with TMA (rows past the end are clipped)
          fence_proxy_async_smem();
          // both warps of this half staged their rows (a bounded wait: a named barrier would
          // hang if the other warp left on an abort)
          warp_arrive(&bars.ep_half[half]);
          if (!waitb(&bars.ep_half[half], ep_phase & 1, W_O_EPHALF, false)) break;
          ++ep_phase;
          if (rr == 0) {
            if (half * 64 < rows_per_item) {
              const int32_t row0 = it.id * rows_per_item + half * 64;
              const uint32_t sbase = smem_u32(stage);
              for (int bx = 0; bx < kVBoxes; ++bx)
                tma_store_2d(&map_out, bx * kBoxCols, row0, sbase + bx * kBoxBytes);
              bulk_commit();
              bulk_wait_read_all();
              stored = true;
            }
            mbar_arrive(&bars.o_kv_empty[s]);
          }
          gs += 2;
        } else {
          // decode: fp32 partial rows to the workspace; sparse with other head counts: bf16 rows
#pragma unroll 1
          for (int c0 = 0; c0 < kLatent; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tbase + lane_base + c0, v);
            tmem_wait_ld();
            if (!row_ok) continue;
            if (orow_f) {
              float4* dst = reinterpret_cast<float4*>(orow_f + c0);
#pragma unroll
              for (int u = 0; u < 8; ++u)
                dst[u] = make_float4(__uint_as_float(v[4 * u]) * cn, __uint_as_float(v[4 * u + 1]) * cn,
                                     __uint_as_float(v[4 * u + 2]) * cn, __uint_as_float(v[4 * u + 3]) * cn);
            } else if (orow) {
              uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                dst[u] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * u]) * cn, __uint_as_float(v[8 * u + 1]) * cn),
                                    pack_bf16x2(__uint_as_float(v[8 * u + 2]) * cn, __uint_as_float(v[8 * u + 3]) * cn),
                                    pack_bf16x2(__uint_as_float(v[8 * u + 4]) * cn, __uint_as_float(v[8 * u + 5]) * cn),
                                    pack_bf16x2(__uint_as_float(v[8 * u + 6]) * cn, __uint_as_float(v[8 * u + 7]) * cn));
              }
            }
          }
          tc_fence_before();
          warp_arrive(&bars.o_free);
          if (row_ok && lse_dst) *lse_dst = lse_out;
        }
        ++i;
      }
      if (stored) bulk_wait_all();
    }
  }

  // ---- teardown: drain on abort, then leave together ----
  __syncwarp();
  if (*abort_flag) {
    // let what this thread issued land before the CTA leaves: its MMAs (one more commit, which
    // arrives once they are all done) and its TMA loads (their last full barrier phase)
    const bool mma_thread = lane == 0 && (is_s ? (warp == 5 || warp == 7) : warp == 5);
    if (mma_thread) {
      uint64_t* db = &bars.drain[(is_s && warp == 7) ? 1 : 0];
      mma_commit(db);
      mbar_drain(db, 0);
    }
    mbar_drain(drain_bar, drain_par);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 5) tmem_dealloc(tbase, 512);
}

}  // namespace

size_t core_smem_bytes() { return kSmemAlloc; }

cudaError_t launch_core(const CoreParams& p, const CoreMaps& maps, cudaStream_t stream) {
  static PerDeviceOnce attrs;
  cudaError_t e = attrs.run([] {
    cudaError_t r = cudaFuncSetAttribute(mla_core_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemAlloc);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(mla_core_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    return r;
  });
  if (e != cudaSuccess) return e;
  if (p.num_pairs <= 0) return cudaSuccess;
  if (p.mode == MODE_SPARSE)
    mla_core_kernel<true><<<dim3(2 * p.num_pairs), dim3(kThreadsSparse), kSmemAlloc, stream>>>(p, maps);
  else
    mla_core_kernel<false><<<dim3(2 * p.num_pairs), dim3(kThreadsDense), kSmemAlloc, stream>>>(p, maps);
  return cudaGetLastError();
}

}  // namespace mla
