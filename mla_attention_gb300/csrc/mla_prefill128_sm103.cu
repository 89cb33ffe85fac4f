// Absorbed MLA prefill and paged decode with 128-key score tiles (sm_103a: tcgen05, TMEM,
// TMA).  Decode is the pages' seqlen-1 form: the 128 heads of one query token are the 128
// rows of an item, the request's keys are split into segments of whole tiles over the CTA
// pairs (split-K), each pair writes an fp32 partial (O / l, LSE) and decode_reduce_kernel
// merges the partials by LSE.
//
// What it computes is the prefill of mla_core_kernel (pages: Tenstorrent ring_mla and
// Ascend RingMLA "prefill" sections -- scores over all 576 columns of the shared KV row,
// V = its first 512 columns, causal mask by global position, output plus natural-log LSE,
// merged with (prev_out, prev_lse) when given).  The tiling differs: a score tile is
// 128 query rows x 128 keys, which the tensor core runs at about 90% of its N=256 rate
// where the 64-key tile of mla_core_kernel runs at about 55%.
//
// Cluster of two CTAs per 128-row item, as in mla_core_kernel (an fp32 O tile of
// 128 x 512 fills one SM's TMEM); 13 warps per CTA:
//   S-CTA  TMEM: Q latent part (512 bf16 = 256 columns) + two S buffers of 128 columns.
//          smem: K ring of three 48 KB groups (64-column boxes 0-2, 3-5, 6-8 of 128 rows),
//          Q RoPE part (128 x 64, SW128), two local P buffers (128 x 128 bf16) and factors.
//          warps 0-3: softmax, one row per thread (the scores of a tile read from TMEM in
//          32-column pieces); warps 4, 8-12: K producers, one per (group, 64-key half);
//          warps 5, 6: S MMAs of even / odd tiles; warp 7: P copies.
//   O-CTA  TMEM: O (512 columns).  smem: V ring of two 64-key halves (64 KB each), two P
//          buffers and factors, the row statistics.
//          warps 0-3: rescale and epilogue rows; warps 4, 8: V producers, one per half
//          (FP8 cache: warps 4, 6-12, four per half); warp 5: P V MMAs.
// Every wait is bounded (see mbar_wait); a timeout sets the abort flag, the CTA lets its
// copies and MMAs land and leaves through the cluster barrier.
#include <math_constants.h>

#include "mla_internal.h"
#include "mma_seq.cuh"
#include "sm103_ptx.cuh"
#include "softmax_rows.cuh"

namespace mla {
namespace {

constexpr int kThreadsT = 416;  // 13 warps: see the role table above
constexpr int kKeysT = 128;                           // keys per score tile
constexpr int kGroups = 3;                            // K groups per tile
constexpr int kBoxBytesK = kKeysT * 128;              // 128 rows x 128 B
constexpr int kGroupBytes = 3 * kBoxBytesK;           // 49152
constexpr int kBoxBytesV = 64 * 128;                  // 64 rows x 128 B
constexpr int kHalfBytesV = kVBoxes * kBoxBytesV;     // 65536: 64 keys x 512 columns
constexpr int kPBytesT = kRows * kKeysT * 2;          // 32768
constexpr int kPBoxBytes = kRows * 128;               // 16384: P for 64 keys
constexpr int kRowWarpsS = 4;
constexpr int kRowWarpsO = 4;

// shared memory (offsets from the dynamic base, which is 1024-byte aligned; the barrier
// block sits at the same offset in both CTAs)
constexpr int kOffK = 0;                              // S: 3 K groups
constexpr int kOffQpe = kGroups * kGroupBytes;        // S: Q RoPE part (147456)
constexpr int kOffPS = kOffQpe + kRows * 128;         // S: P buffers (163840)
constexpr int kOffAlphaS = kOffPS + 2 * kPBytesT;     // S: factors [2][128] (229376)
constexpr int kOffV = 0;                              // O: 2 V halves
constexpr int kOffPO = 2 * kHalfBytesV;               // O: P buffers (131072)
constexpr int kOffAlphaO = kOffPO + 2 * kPBytesT;     // O: factors [2][128] (196608)
constexpr int kOffStatsO = kOffAlphaO + 2 * kRows * 4;  // O: (m, l) [128][2] from the S-CTA (197632)
constexpr int kOffBarsT = kOffAlphaS + 2 * kRows * 4;   // both (230400)
constexpr int kSmemT = kOffBarsT + 512;               // 231936
static_assert(kOffStatsO + kRows * 8 <= kOffBarsT, "O-CTA layout overlaps the barriers");
static_assert(kSmemT <= 232448, "shared memory over the sm_103a limit");
static_assert(kOffPS % 1024 == 0 && kOffPO % 1024 == 0 && kOffQpe % 1024 == 0, "SW128 operands need 1 KB");

constexpr uint32_t kTmemQ = 0;      // S: Q latent part [0, 256)
constexpr uint32_t kTmemS = 256;    // S: S buffers [256, 384), [384, 512)
constexpr float kRescaleLog2 = 8.0f;
constexpr int kPrefetchTiles = 4;   // decode: L2 prefetch distance of the O-CTA's V producers
// decode: L2 eviction priorities of the cache stream (see l2_policy).  Every cache row is read
// twice, by the K load (576 columns) and a tile or two later by the V load (512 columns): the K
// load marks its lines evict-last so that they survive until the V load, which marks them
// evict-first (their last use).  Measured on the 64 x U[4096, 32768] decode: DRAM reads 1.62 ->
// 1.46 GB for 1.37 GB of cache, 3813 -> 3888 GB/s.
constexpr int kHintPf = kL2Plain;
constexpr int kHintK = kL2Keep;
constexpr int kHintV = kL2Done;

struct BarsT {
  // S-CTA
  uint64_t kfull[kGroups][2];  // group k of tile t landed (index t % 2: one consumer per barrier)
  uint64_t kempty[kGroups];    // the MMAs of group k of the last tile are done
  uint64_t s_full[2];          // S tile of issuer b done
  uint64_t s_free[2];          // every row warp read S buffer b
  uint64_t q_full;             // Q of the item in TMEM / smem (prefill, sparse: latent pieces 0-5, the producers' part)
  uint64_t q_tail;             // prefill, sparse: latent pieces 6-7 and the RoPE part (the rows' part)
  uint64_t q_taken;            // both issuers passed q_full (count 2)
  uint64_t q_free;             // every S MMA of the item is done: Q may be replaced (one commit per issuer)
  uint64_t pwritten[2];        // rows wrote local P buffer b
  uint64_t pbuf_free[2];       // the copy out of local P buffer b has been read
  uint64_t stats_free;         // the O-CTA read the row statistics (remote)
  // O-CTA
  uint64_t vfull[2], vempty[2];
  uint64_t p_full[2];          // P tile and factors landed (bulk copy with its tx bytes); sparse: box 0 of P
                               // (keys 0-63) and the factors
  uint64_t p_full1[2];         // sparse: box 1 of P tile b (keys 64-127) landed
  uint64_t p_ready[2];         // rows rescaled O for P tile b
  uint64_t stats_full;         // row statistics stored here by the S-CTA (remote)
  uint64_t o_free;             // the epilogue read O
  uint64_t ep_half[2];         // both warps of an epilogue half staged their rows (count 2)
  // both
  uint64_t pb_free[2];         // P V of O-CTA buffer b done (multicast commit)
  uint64_t stall;              // fault injection: never arrived on
  uint64_t drain[2];           // abort: one commit of each MMA issuer lands here
  uint64_t raw[16];            // FP8: producer warp q's staged e4m3 boxes landed (S-CTA: q < 6, O-CTA: 8 + q)
  uint32_t tmem_base;
  uint32_t abort_flag;
};
static_assert(sizeof(BarsT) <= 512, "barrier block too large");

enum : uint32_t {
  X_K_EMPTY = 0x40, X_K_FULL, X_S_FREE, X_S_FULL, X_Q_FULL, X_Q_TAKEN, X_P_WRITTEN, X_PBUF_FREE, X_PB_FREE,
  X_STATS_FREE, X_V_EMPTY, X_V_FULL, X_P_FULL, X_P_READY, X_PV_DONE, X_STATS_FULL, X_O_FREE, X_STALL, X_EP_HALF,
  X_Q_FREE, X_RAW,
  X_ALIGN = 0x4F, X_PAGE = 0x50, X_LEN = 0x51,
};

// Optional wait-time trace (built only with -DMLA_TRACE): cycles each warp spends in
// each wait site, summed over the launch, and each warp's total cycles.
#ifdef MLA_TRACE
__device__ unsigned long long g_trace_wait[2][16][32];
__device__ unsigned long long g_trace_total[2][16];
#define MLA_TRACE_ONLY(...) __VA_ARGS__
#else
#define MLA_TRACE_ONLY(...)
#endif

struct ItemT {
  int id;        // prefill: row tile; decode: request
  int J;         // 128-key tiles
  int64_t k0;    // decode: first key of this segment (within the request)
  int64_t k1;    // decode: end key of this segment
  int slot;      // decode: partial slot (request + pair)
};

// keys seen by decode query group b (one query token of a request; see decode_group_len)
__device__ __forceinline__ int decode_len_t(const CoreParams& p, int b) { return decode_group_len(p, b); }

__device__ __forceinline__ int64_t keys_for_token(const CoreParams& p, int64_t t) {
  int64_t n = p.kv_valid;
  if (p.causal) {
    const int64_t c = p.q_pos0 + t - p.kv_pos0 + 1;
    if (c < n) n = c;
  }
  return n < 0 ? 0 : n;
}

// Row tiles in longest-first order, dealt round robin to the CTA pairs.  In place, a row
// that sees no key keeps its previous (out, lse); J only falls along this order (causal)
// or is constant, so the first key-less item ends the list.
// Decode: the key tiles of all requests, in request order, are split into equal shares, one
// per CTA pair; an item is the part of one request inside this pair's share (an empty
// share has none).
template <bool kDec, bool kSp = false>
struct ItemIterT {
  const CoreParams* p;
  int pair;
  int64_t k;
  int b;
  int64_t pre, lo, hi;
  __device__ void init(const CoreParams& prm, int pair_id) {
    p = &prm;
    pair = pair_id;
    k = pair_id;
    b = 0;
    pre = 0;
    lo = hi = 0;
    if constexpr (kDec) {
      int64_t tot = 0;
      for (int i = 0; i < prm.B; ++i) tot += (decode_len_t(prm, i) + kKeysT - 1) / kKeysT;
      lo = tot * pair_id / prm.num_pairs;
      hi = tot * (pair_id + 1) / prm.num_pairs;
    }
  }
  __device__ bool next(ItemT& it) {
    const CoreParams& P = *p;
    if constexpr (kDec) {
      if (hi <= lo) return false;
      while (b < P.B) {
        const int len = decode_len_t(P, b);
        const int64_t nt = (len + kKeysT - 1) / kKeysT;
        const int64_t s0 = pre, e0 = pre + nt;
        const int cur = b;
        pre = e0;
        ++b;
        if (nt == 0 || e0 <= lo) continue;
        if (s0 >= hi) {
          b = P.B;
          return false;
        }
        const int64_t t0 = (s0 > lo ? s0 : lo) - s0, t1 = (e0 < hi ? e0 : hi) - s0;
        if (t1 <= t0) continue;
        it.id = cur;
        it.J = (int)(t1 - t0);
        it.k0 = t0 * kKeysT;
        it.k1 = t1 * kKeysT < len ? t1 * kKeysT : len;
        it.slot = cur + pair;
        return true;
      }
      return false;
    } else if constexpr (kSp) {  // one query token (all its heads) per item, every top-k tile
      if (k >= P.T) return false;
      it.id = (int)k;
      it.J = (P.K + kKeysT - 1) / kKeysT;
      it.k0 = 0;
      it.k1 = P.K;
      k += P.num_pairs;
      return true;
    } else {
    const int64_t rows = (int64_t)P.T * P.H;
    const int64_t n_items = (rows + kRows - 1) / kRows;
    if (k >= n_items) return false;
    const int64_t id = n_items - 1 - k;
    k += P.num_pairs;
    int64_t last = id * kRows + kRows - 1;
    if (last >= rows) last = rows - 1;
    const int64_t n = keys_for_token(P, last / P.H);
    it.id = (int)id;
    it.J = (int)((n + kKeysT - 1) / kKeysT);
    if (it.J == 0 && P.prev_out && (const void*)P.prev_out == (const void*)P.out &&
        (const void*)P.prev_lse == (const void*)P.lse)
      return false;
    return true;
    }
  }
};

__device__ __forceinline__ void st_cluster_f32x2(uint32_t addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}

// ---- decode: where the 64 keys [kh, kh + 64) of a tile half come from ----
// A whole half inside one valid page is one tiled TMA box per 64 columns; otherwise its
// rows are gathered four at a time (tile::gather4), keys past the request's length and
// rows of an out-of-range page as -1 (zero fill; the page is reported).
// The block-table entries are read a tile ahead (load_half_ids) and used only when the
// tile is issued (issue_half), so the producer never waits on them.
struct HalfIds {
  int32_t pe, po;              // page ids of keys kh + 2 lane, kh + 2 lane + 1 (0 past the length: unused)
};
__device__ __forceinline__ HalfIds load_half_ids(const CoreParams& p, int req, int len, int64_t kh) {
  const int lane = threadIdx.x & 31;
  const int32_t* bt = p.block_table + (int64_t)decode_request(p, req) * p.max_pages;
  const int64_t ke = kh + 2 * lane, ko = ke + 1;
  HalfIds ids;
  const int32_t* be = bt + ke / p.page_size;
  const int32_t* bo = bt + ko / p.page_size;
  ids.pe = (ke < len && guard_span(p.err, G_BLOCK_TABLE, be, 4, p.block_table, p.ext_block_table)) ? __ldg(be) : 0;
  ids.po = (ko < len && guard_span(p.err, G_BLOCK_TABLE, bo, 4, p.block_table, p.ext_block_table)) ? __ldg(bo) : 0;
  return ids;
}
// Rows of a half that is not one tiled box per column block (the last half of a request,
// pages of 16 or 32 tokens, a bad page): lane l < 16 gathers rows 4 l .. 4 l + 3 of every
// column block (tile::gather4), keys past the length and rows of an out-of-range page as -1
// (zero fill; the page is reported).  Rare, so kept out of line: the producers' hot loop
// stays small for the instruction cache.
static __device__ __noinline__ void gather_half(uint32_t dst, uint32_t box_stride, int32_t x0, int nbox,
                                                const CUtensorMap* row_map, int page_size, int64_t num_pages,
                                                int len, int64_t kh, int32_t pe, int32_t po, uint64_t* bar,
                                                uint32_t* err) {
  const int lane = threadIdx.x & 31;
  auto row_of = [&](int32_t pg, int64_t key) -> int32_t {
    if (key >= len) return -1;
    if (pg < 0 || pg >= num_pages) {
      record_error(err, DEV_RANGE_BASE | X_PAGE);
      return -1;
    }
    return (int32_t)(pg * (int64_t)page_size + key % page_size);
  };
  const int32_t re = row_of(pe, kh + 2 * lane);
  const int32_t ro = row_of(po, kh + 2 * lane + 1);
  const int32_t a0 = __shfl_sync(0xffffffffu, re, (2 * lane) & 31);
  const int32_t a1 = __shfl_sync(0xffffffffu, ro, (2 * lane) & 31);
  const int32_t a2 = __shfl_sync(0xffffffffu, re, (2 * lane + 1) & 31);
  const int32_t a3 = __shfl_sync(0xffffffffu, ro, (2 * lane + 1) & 31);
  if (lane < 16)
    for (int i = 0; i < nbox; ++i) tma_gather4(dst + i * box_stride + lane * 512, row_map, x0 + i * kBoxCols, a0, a1, a2, a3, bar);
}

// Issues the 64-row boxes of one tile half [kh, kh + 64): nbox (<= 32) column blocks starting
// at column x0, landing box_stride bytes apart from dst.  A half inside one valid page is one
// tiled box per column block, lane i issuing block i.  Warp-uniform.
template <int kHint>
__device__ __forceinline__ void issue_half(uint32_t dst, uint32_t box_stride, int32_t x0, int nbox, const CoreParams& p,
                                           const CoreMaps& maps, int len, int64_t kh, const HalfIds& ids,
                                           uint64_t* bar, uint32_t* err) {
  const int32_t pg0 = __shfl_sync(0xffffffffu, ids.pe, 0);  // page of key kh
  if (p.page_size % 64 == 0 && kh + 64 <= len && pg0 >= 0 && pg0 < p.num_pages) {
    const int lane = threadIdx.x & 31;  // one box per lane: lanes overlap their TMA issues
    if (lane < nbox) {
      const int32_t y = (int32_t)(pg0 * (int64_t)p.page_size + kh % p.page_size);
      tma_load_2d_hint<kHint>(dst + lane * box_stride, &maps.kv, x0 + lane * kBoxCols, y, bar);
    }
  } else {
    gather_half(dst, box_stride, x0, nbox, &maps.row, p.page_size, p.num_pages, len, kh, ids.pe, ids.po, bar, err);
  }
}

// ---- sparse: the top-k rows of a tile half ----
// Raw top-k entries of keys kh + 2 lane and kh + 2 lane + 1 of token `id` (-1 past K), read a
// tile ahead and range-checked where they are used: an entry outside [0, S_kv) is padding.
__device__ __forceinline__ HalfIds sparse_half_ids(const CoreParams& p, int id, int64_t kh) {
  const int lane = threadIdx.x & 31;
  const int32_t* tk = p.topk + (int64_t)id * p.K;
  const int64_t c0 = kh + 2 * lane;
  HalfIds ids;
  ids.pe = (c0 < p.K && guard_span(p.err, G_TOPK, tk + c0, 4, p.topk, p.ext_topk)) ? __ldg(tk + c0) : -1;
  ids.po = (c0 + 1 < p.K && guard_span(p.err, G_TOPK, tk + c0 + 1, 4, p.topk, p.ext_topk)) ? __ldg(tk + c0 + 1) : -1;
  return ids;
}
// Gathers the 64 rows of a tile half listed in ids, column boxes cb0 .. cb0 + kBox - 1 (boxes 0-7
// from c_kv, box 8 = the RoPE columns from k_pe), into 64-row SW128 boxes box_stride bytes
// apart from dst, with 16-byte cp.async.  Each warp instruction moves one 128-byte box row of
// four rows (lane / 8: which of the four, lane % 8: the 16-byte chunk), so the warp reads four
// whole 128-byte lines.  Padding rows are zero-filled (source size 0).  Every lane then arrives
// (noinc) on bar once its copies have landed; the reader of the stage orders them before its
// async-proxy reads with a proxy fence.
template <int kBox>
__device__ __forceinline__ void gather_half_sparse(uint32_t dst, uint32_t box_stride, int cb0, const CoreParams& p,
                                                   const HalfIds& ids, uint64_t* bar) {
  uint32_t* err = p.err;
  const int lane = threadIdx.x & 31;
  const int rq = lane >> 3, c = lane & 7;
#pragma unroll 2
  for (int i = 0; i < 16; ++i) {
    const int rr = 4 * i + rq;  // row of the half
    const int32_t ae = __shfl_sync(0xffffffffu, ids.pe, rr >> 1);
    const int32_t ao = __shfl_sync(0xffffffffu, ids.po, rr >> 1);
    const int32_t raw = (rr & 1) ? ao : ae;
    const bool ok = raw >= 0 && raw < p.S_kv;
    const int64_t row = ok ? raw : 0;
    const uint32_t line = dst + (uint32_t)rr * 128u + ((uint32_t)(c ^ (rr & 7)) << 4);
#pragma unroll
    for (int b = 0; b < kBox; ++b) {
      const int gb = cb0 + b;
      const __nv_bfloat16* src = (gb < kVBoxes) ? p.c_kv + row * kLatent + gb * kBoxCols + c * 8
                                                : p.k_pe + row * kRope + c * 8;
      const bool in = ok && ((gb < kVBoxes) ? guard_span(err, G_C_KV, src, 16, p.c_kv, p.ext_c_kv)
                                            : guard_span(err, G_K_PE, src, 16, p.k_pe, p.ext_k_pe));
      cp_async16_zfill(line + b * box_stride, (kGuarded && !in) ? p.c_kv : src, in ? 16u : 0u);
    }
  }
  cp_async_arrive_noinc(bar);
}

// FP8 decode: rows [kh, kh + 64) of column blocks cb0 .. cb0 + kBlk - 1 (64 values each) of the
// e4m3 cache, converted to f16 (exactly) into 64-row SW128 boxes box_stride bytes apart from dst.
// Lane l converts whole 64-value row pieces (units l, l + 32, ...: four 16-byte loads, eight
// 16-byte chunks), the loads of kBlk units in flight together.  Keys past len and rows of an
// out-of-range page give zero rows (the page is reported).  The caller fences the async proxy
// and arrives once every lane has stored.  The cache rows are normally in L2 already: the
// O-CTA's producers prefetch each page a few tiles ahead.
template <int kBlk>
__device__ __forceinline__ void fill_half_fp8(uint8_t* dst, uint32_t box_stride, int cb0, const CoreParams& p,
                                              int len, int64_t kh, const HalfIds& ids, uint32_t* err) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int batch = 0; batch < 2; ++batch) {
    uint4 v[kBlk][4];
    int rows[kBlk];
#pragma unroll
    for (int i = 0; i < kBlk; ++i) {
      // 64 * kBlk units (box b, row r), 2 * kBlk per lane; consecutive lanes take consecutive rows
      // of one box, so each quarter-warp's swizzled 16-byte stores fall in distinct banks
      const int u = lane + 32 * (batch * kBlk + i);
      const int r = u & 63, b = u >> 6;
      rows[i] = r;
      const int32_t pe = __shfl_sync(0xffffffffu, ids.pe, r >> 1);
      const int32_t po = __shfl_sync(0xffffffffu, ids.po, r >> 1);
      const int32_t pg = (r & 1) ? po : pe;
      const int64_t key = kh + r;
      const bool in_len = key < len;
      const bool ok = in_len && pg >= 0 && pg < p.num_pages;
      if (in_len && !ok) record_error(err, DEV_RANGE_BASE | X_PAGE);
      const uint4* src = reinterpret_cast<const uint4*>(
          p.cache8 + ((int64_t)pg * p.page_size + key % p.page_size) * kDk + (cb0 + b) * 64);
      const bool in = ok && guard_span(err, G_CACHE8, src, 64, p.cache8, p.ext_cache8);
#pragma unroll
      for (int w = 0; w < 4; ++w) v[i][w] = in ? __ldg(src + w) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kBlk; ++i) {
      const int u = lane + 32 * (batch * kBlk + i);
      const int r = rows[i], b = u >> 6;
      uint8_t* line = dst + b * box_stride + r * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {  // chunk c: values 8c .. 8c + 7 = bytes 8c .. 8c + 7 of the piece
        const uint4& q = v[i][c >> 1];
        const uint32_t w0 = (c & 1) ? q.z : q.x, w1 = (c & 1) ? q.w : q.y;
        *reinterpret_cast<uint4*>(line + ((c ^ (r & 7)) << 4)) =
            make_uint4(e4m3x2_to_f16x2((uint16_t)(w0 & 0xFFFFu)), e4m3x2_to_f16x2((uint16_t)(w0 >> 16)),
                       e4m3x2_to_f16x2((uint16_t)(w1 & 0xFFFFu)), e4m3x2_to_f16x2((uint16_t)(w1 >> 16)));
      }
    }
  }
}

// ---- Q of an item: latent part -> TMEM (256 columns), RoPE part -> smem (SW128 K-major) ----
// Pieces [c_begin, c_end) of 64 latent columns of this thread's query row go to TMEM columns
// 32 c .. 32 c + 31 of its lane (tq: the lane's TMEM address of the Q region); two pieces'
// loads are in flight together.  Warp-uniform (tcgen05.st is warp-collective).  The row warps
// and four producer warps (one per TMEM lane quadrant) split the pieces, so the next item's
// Q is in place sooner.  FP8 decode: the MMAs take f16 operands.
template <bool kF16>
__device__ __forceinline__ void load_q_pieces(uint32_t tq, const __nv_bfloat16* qrow, int c_begin, int c_end,
                                              const CoreParams& p) {
#pragma unroll 1
  for (int c0 = c_begin; c0 < c_end; c0 += 2) {
    const bool two = c0 + 1 < c_end;
    uint4 x[2][8];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const uint4* src = (qrow && (cc == 0 || two)) ? reinterpret_cast<const uint4*>(qrow + 64 * (c0 + cc)) : nullptr;
      if (src && !guard_span(p.err, G_Q, src, 128, p.q, p.ext_q)) src = nullptr;
#pragma unroll
      for (int u = 0; u < 8; ++u) x[cc][u] = src ? __ldg(src + u) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      if (cc == 1 && !two) break;
      uint32_t v[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        v[4 * u + 0] = x[cc][u].x;
        v[4 * u + 1] = x[cc][u].y;
        v[4 * u + 2] = x[cc][u].z;
        v[4 * u + 3] = x[cc][u].w;
      }
      if constexpr (kF16) {
#pragma unroll
        for (int u = 0; u < 32; ++u) v[u] = bf16x2_to_f16x2(v[u]);
      }
      tmem_st32(tq + 32 * (c0 + cc), v);
    }
  }
}
template <bool kF16>
__device__ __forceinline__ void load_q_rope(uint8_t* qpe_row, const __nv_bfloat16* qpe, int r, uint32_t* err,
                                            const void* base, uint64_t extent) {
  const uint4* src = reinterpret_cast<const uint4*>(qpe);
  if (src && !guard_span(err, G_Q_PE, src, 128, base, extent)) src = nullptr;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint4 v = src ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
    if constexpr (kF16)
      v = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
    *reinterpret_cast<uint4*>(qpe_row + ((c ^ (r & 7)) << 4)) = v;
  }
  fence_proxy_async_smem();  // read by the MMA through the async proxy
}
// Prefill and sparse: producer warps 8-11 load latent pieces 0-5 of the next item's Q (K groups 0
// and 1 of the S MMA) as soon as the previous item's MMAs are done; the row warps, which first
// finish the previous item's last softmax, load pieces 6-7 and the RoPE part (group 2).  The
// first tile's groups 0-1 run on the producers' part while the rows load theirs.
constexpr int kQProdPieces = 6;

// FP8 decode, staged path: a 64-row box of the e4m3 cache (64 bytes a row) that TMA wrote into
// the upper half of its own 8 KB f16 chunk is converted in place into 64 SW128 rows of 128 B.
// Rows 0-31 land below the staged bytes; rows 32-63 overwrite them, so each half's staged
// bytes are all loaded before any lane stores that half (the warp synchronises in between).
// Each staged load covers 512 contiguous bytes (lane l: row 8 i + l / 4, bytes 16 (l % 4) ..),
// so it has no bank conflict; the two 16-byte f16 chunks a lane then stores (chunks 2 (l % 4)
// and the next, swizzled by row) fall in distinct banks across each quarter-warp.  The caller
// fences the async proxy and arrives once every lane has stored.
__device__ __forceinline__ void convert_box_in_place(uint8_t* chunk) {
  const int lane = threadIdx.x & 31;
  const uint8_t* raw = chunk + 4096;
  const int c0 = 2 * (lane & 3);  // first f16 chunk of the lane's 16 values
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = reinterpret_cast<const uint4*>(raw + half * 2048 + i * 512)[lane];
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 32 * half + 8 * i + (lane >> 2);
      uint8_t* line = chunk + r * 128;
      *reinterpret_cast<uint4*>(line + ((c0 ^ (r & 7)) << 4)) =
          make_uint4(e4m3x2_to_f16x2((uint16_t)(v[i].x & 0xFFFFu)), e4m3x2_to_f16x2((uint16_t)(v[i].x >> 16)),
                     e4m3x2_to_f16x2((uint16_t)(v[i].y & 0xFFFFu)), e4m3x2_to_f16x2((uint16_t)(v[i].y >> 16)));
      *reinterpret_cast<uint4*>(line + (((c0 + 1) ^ (r & 7)) << 4)) =
          make_uint4(e4m3x2_to_f16x2((uint16_t)(v[i].z & 0xFFFFu)), e4m3x2_to_f16x2((uint16_t)(v[i].z >> 16)),
                     e4m3x2_to_f16x2((uint16_t)(v[i].w & 0xFFFFu)), e4m3x2_to_f16x2((uint16_t)(v[i].w >> 16)));
    }
  }
}

// ---- softmax rows: one 32-column piece of a score row ----
// Sparse: raw top-k entries of tile j of token id, key 32 q + lane in e[q] (-1 past K).
__device__ __forceinline__ void sparse_tile_entries(const CoreParams& p, int id, int j, int32_t (&e)[4]) {
  const int lane = threadIdx.x & 31;
  const int32_t* tk = p.topk + (int64_t)id * p.K;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int c = j * kKeysT + 32 * q + lane;
    e[q] = (c < p.K && guard_span(p.err, G_TOPK, tk + c, 4, p.topk, p.ext_topk)) ? __ldg(tk + c) : -1;
  }
}
// p = 2^(s * scale_log2 - msub) of a piece as bf16 into four 16-byte chunks (chunk0 .. chunk0 + 3
// of the row's 128-byte line of the piece's 64-key P box, swizzled), row sums into rsq (two
// pairs of partial sums), and the extreme of the raw scores into eq.  Scores go through the
// scale in pairs (packed fp32).
template <bool kUp, bool kF16>
__device__ __forceinline__ void row_exp(const uint32_t (&sr)[32], uint64_t sl2x2, uint64_t nmsub2, uint8_t* pline,
                                        int chunk0, int r, uint64_t (&rsq)[2], float (&eq)[4]) {
#pragma unroll
  for (int c8 = 0; c8 < 4; ++c8) {  // 8 keys -> one 16-byte chunk of P
    uint32_t w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = 8 * c8 + 2 * u;
      const float v0 = __uint_as_float(sr[c]), v1 = __uint_as_float(sr[c + 1]);
      eq[u] = kUp ? max3f(eq[u], v0, v1) : min3f(eq[u], v0, v1);
      float x0, x1;
      f32x2_split(fma_f32x2(f32x2(v0, v1), sl2x2, nmsub2), x0, x1);
      const float e0 = ex2_approx(x0);
      const float e1 = ex2_approx(x1);
      rsq[u & 1] = add_f32x2(rsq[u & 1], f32x2(e0, e1));
      w[u] = kF16 ? pack_f16x2(e0, e1) : pack_bf16x2(e0, e1);
    }
    *reinterpret_cast<uint4*>(pline + (((chunk0 + c8) ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// kUp: the scale is >= 0, so the row extreme of the raw scores is their maximum (else
// their minimum).  kDecode: paged decode (else prefill).  kFp8 (decode only): the cache is
// e4m3 with a per-tensor scale; producers convert its rows to f16 (exact) into the K and V
// rings with ordinary loads, Q and P are f16, and both MMAs take f16 operands.  One
// instantiation per combination keeps the choices out of the loops: the loop bodies must stay
// small for the instruction cache.
template <bool kUp, bool kDecode, bool kFp8, bool kSparse>
__device__ __forceinline__ void prefill128_body(const CoreParams& p, const CoreMaps& maps) {
  extern __shared__ __align__(1024) uint8_t smem[];
  BarsT& bars = *reinterpret_cast<BarsT*>(smem + kOffBarsT);
  const uint32_t rank = cluster_ctarank();
  const bool is_s = (rank == 0);
  const uint32_t peer = rank ^ 1u;
  const int pair = blockIdx.x >> 1;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t lim = p.spin_limit;
  uint32_t* err = p.err;
  constexpr bool decode = kDecode;
  // prefill stages its epilogue (prev in, out) through the V ring; sparse when an item's 128 rows
  // are 128 consecutive output rows (H = 128), else its rows store themselves
  const bool staged = kSparse ? (p.H == kRows) : !kDecode;
  // The layout assumes a 1 KB aligned dynamic base (true when the kernel has no static
  // shared memory); anything else is refused before any barrier is touched.
  if (smem_u32(smem) & 1023u) {
    if (tid == 0) record_error(err, DEV_RANGE_BASE | X_ALIGN);
    return;
  }

  // ---- setup ----
  if (tid == 0) {
    if (is_s) {
      for (int k = 0; k < kGroups; ++k) {
        // the two producers of group k (one per 64-row half); sparse: every lane of both (noinc
        // arrivals of its row copies)
        mbar_init(&bars.kfull[k][0], kSparse ? 64 : 2);
        mbar_init(&bars.kfull[k][1], kSparse ? 64 : 2);
        mbar_init(&bars.kempty[k], 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(&bars.s_full[b], 1);
        mbar_init(&bars.s_free[b], kRowWarpsS);
        mbar_init(&bars.pwritten[b], kRowWarpsS);
        mbar_init(&bars.pbuf_free[b], 1);
        mbar_init(&bars.pb_free[b], 1);
      }
      mbar_init(&bars.q_full, 4);  // decode: the row warps; prefill, sparse: producer warps 8-11
      mbar_init(&bars.q_tail, kRowWarpsS);
      mbar_init(&bars.q_taken, 2);
      mbar_init(&bars.q_free, 2);
      mbar_init(&bars.stats_free, kRowWarpsO);
    } else {
      for (int b = 0; b < 2; ++b) {
        // FP8: the four warps that fill half b; sparse: every lane of those four
        mbar_init(&bars.vfull[b], kSparse ? 128 : (kFp8 ? 4 : 1));
        mbar_init(&bars.vempty[b], 1);
        mbar_init(&bars.p_full[b], 1);
        mbar_init(&bars.p_full1[b], 1);
        mbar_init(&bars.p_ready[b], kRowWarpsO);
        mbar_init(&bars.pb_free[b], 1);
      }
      mbar_init(&bars.stats_full, kRowWarpsS);
      mbar_init(&bars.o_free, kRowWarpsO);
      mbar_init(&bars.ep_half[0], 2);
      mbar_init(&bars.ep_half[1], 2);
    }
    mbar_init(&bars.stall, 1);
    for (int q = 0; q < 16; ++q) mbar_init(&bars.raw[q], 1);
    mbar_init(&bars.drain[0], 1);
    mbar_init(&bars.drain[1], 1);
    bars.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  if (!kFp8 && warp == 4 && lane == 0) {  // (FP8 decode and sparse read the cache without TMA)
    if (!kSparse) {
      tma_prefetch_desc(&maps.kv);
      tma_prefetch_desc(&maps.row);
    }
    if (staged) tma_prefetch_desc(&maps.out);
    if (staged && p.prev_out) tma_prefetch_desc(&maps.prev);
  }
  // decode: publish the per-request count of 128-key tiles (prefix sums) for the reduction
  if (decode && blockIdx.x == 0 && warp == 0) {
    int64_t run = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + lane;
      int n = 0;
      if (b < p.B) {
        const int32_t* lp = p.lens + decode_request(p, b);
        const int raw = guard_span(err, G_LENS, lp, 4, p.lens, p.ext_lens) ? *lp : 0;
        const int64_t cap = (int64_t)p.max_pages * p.page_size;
        if (raw < 0 || raw > cap) record_error(err, DEV_RANGE_BASE | X_LEN);
        n = (decode_len_t(p, b) + kKeysT - 1) / kKeysT;
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
  cluster_sync();
  tc_fence_after();
  const uint32_t tbase = bars.tmem_base;
  volatile uint32_t* abort_flag = &bars.abort_flag;
  MLA_TRACE_ONLY(unsigned long long trace_wait[32] = {}; const long long trace_t0 = clock64();)
  auto waitb = [&](uint64_t* bar, uint32_t parity, uint32_t site, bool cl) -> bool {
    MLA_TRACE_ONLY(const long long tw = clock64();)
    bool ok = (*abort_flag == 0) && mbar_wait(bar, parity, err, site, lim, cl);
    MLA_TRACE_ONLY(trace_wait[site & 31] += clock64() - tw;)
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) *abort_flag = 1;
    return ok;
  };
  // single-thread wait for the MMA issuers (no warp-collective tcgen05 instruction follows)
  auto wait1 = [&](uint64_t* bar, uint32_t parity, uint32_t site, bool cl) -> bool {
    MLA_TRACE_ONLY(const long long tw = clock64();)
    const bool ok = (*abort_flag == 0) && mbar_wait(bar, parity, err, site, lim, cl);
    MLA_TRACE_ONLY(trace_wait[site & 31] += clock64() - tw;)
    if (!ok) *abort_flag = 1;
    return ok;
  };
  if (p.debug_stall && warp == 5) waitb(&bars.stall, 0, X_STALL, false);  // runs out: injected fault

  ItemIterT<kDecode, kSparse> iter;
  // The query row of row r of an item: its latent part (512 columns) and RoPE part (64), or
  // null for a row past the item's end.
  auto q_row_ptrs = [&](const ItemT& itm, int r, const __nv_bfloat16*& qr, const __nv_bfloat16*& qp) {
    qr = nullptr;
    qp = nullptr;
    if constexpr (decode) {
      if (r < p.H) {
        qr = p.q + ((int64_t)itm.id * p.H + r) * kDk;
        qp = qr + kLatent;
      }
    } else if constexpr (kSparse) {  // q_lift and q_pe rows of head r of token itm.id
      if (r < p.H) {
        qr = p.q + ((int64_t)itm.id * p.H + r) * kLatent;
        qp = p.q_pe + ((int64_t)itm.id * p.H + r) * kRope;
      }
    } else {
      const int64_t f = (int64_t)itm.id * kRows + r;
      if (f < (int64_t)p.T * p.H) {
        const int64_t tt = f / p.H, hh = f - tt * p.H;
        qr = p.q + tt * p.q_stride_t + hh * p.q_stride_h;
        qp = qr + kLatent;
      }
    }
  };
  iter.init(p, pair);
  ItemT it;
  // abort drain: the last barrier phase this thread's TMA loads were counted on
  uint64_t* drain_bar = nullptr;
  uint32_t drain_par = 0;
  const CUtensorMap& map_v = maps.kv;    // V rows, box {64, 64}

  if (is_s) {
    // =====================================================================
    // S-CTA
    // =====================================================================
    if (warp == 4 || warp >= 8) {
      // ---------------- TMA producers: rows 64 h .. 64 h + 63 of K group k ----------------
      // Six warps (4, 8, 9, 10, 11, 12), one per (group k, half h).  Group k of every tile
      // goes to slot k once the MMAs of group k of the previous tile are done; its landing
      // barrier alternates with the tile's parity, so each issuer waits only on the barriers
      // of its own tiles.  A thread issues a TMA box every few hundred cycles whatever the
      // memory does, so the ring is fed by many threads, each with few boxes per tile.
      const int q = (warp == 4) ? 0 : warp - 7;
      const int k = q % kGroups, h = q / kGroups;
      const uint32_t dst = smem_u32(smem + kOffK + k * kGroupBytes + h * kBoxBytesV);
      // prefill and sparse: one per TMEM lane quadrant, they load most of each item's Q (decode has
      // few, long items: its rows load Q alone)
      const bool q_helper = !kDecode && warp >= 8 && warp <= 11;
      uint32_t t = 0, items = 0, n_raw = 0;
      bool live = true;
      while (live && iter.next(it)) {
        const int len = decode ? decode_len_t(p, it.id) : 0;
        HalfIds ids;
        if constexpr (decode) ids = load_half_ids(p, it.id, len, it.k0 + 64 * h);
        if constexpr (kSparse) ids = sparse_half_ids(p, it.id, 64 * h);
        for (int j = 0; j < it.J && live; ++j, ++t) {
          const uint32_t par = t & 1;
          const int64_t kh = it.k0 + (int64_t)j * kKeysT + 64 * h;
          HalfIds cur;
          if constexpr (decode) {
            cur = ids;
            if (j + 1 < it.J) ids = load_half_ids(p, it.id, len, kh + kKeysT);  // read while this tile is issued
          }
          if constexpr (kSparse) {
            cur = ids;
            if (j + 1 < it.J) ids = sparse_half_ids(p, it.id, kh + kKeysT);  // lands during this gather
          }
          if (!waitb(&bars.kempty[k], par ^ 1, X_K_EMPTY, false)) { live = false; break; }
          uint64_t* fb = &bars.kfull[k][par];
          if constexpr (kSparse) {  // the listed rows by cp.async; each lane arrives (noinc) once they land
            gather_half_sparse<3>(dst, kBoxBytesK, 3 * k, p, cur, fb);
          } else if constexpr (kFp8) {
            // a half inside one valid page: its three e4m3 boxes by TMA into the upper halves of their
            // f16 chunks, converted in place; else ordinary loads converted into the slot
            uint8_t* chunk0 = smem + kOffK + k * kGroupBytes + h * kBoxBytesV;
            const int32_t pg0 = __shfl_sync(0xffffffffu, cur.pe, 0);
            if (p.page_size % 64 == 0 && kh + 64 <= len && pg0 >= 0 && pg0 < p.num_pages) {
              uint64_t* rb = &bars.raw[q];
              if (lane == 0) mbar_arrive_expect_tx(rb, 3 * 4096);
              __syncwarp();
              const int32_t y = (int32_t)(pg0 * (int64_t)p.page_size + kh % p.page_size);
              if (lane < 3)
                tma_load_2d_hint<kHintK>(smem_u32(chunk0 + lane * kBoxBytesK + 4096), &maps.kv, (3 * k + lane) * 64, y, rb);
              drain_bar = rb;
              drain_par = n_raw & 1;
              if (!waitb(rb, n_raw & 1, X_RAW, false)) { live = false; break; }
              ++n_raw;
#pragma unroll 1
              for (int b = 0; b < 3; ++b) convert_box_in_place(chunk0 + b * kBoxBytesK);
            } else {
              fill_half_fp8<3>(chunk0, kBoxBytesK, 3 * k, p, len, kh, cur, err);
            }
            fence_proxy_async_smem();  // the MMA reads the slot through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(fb);
          } else {
            if (lane == 0) mbar_arrive_expect_tx(fb, kGroupBytes / 2);
            drain_bar = fb;
            drain_par = (t >> 1) & 1;
            __syncwarp();
            if constexpr (!decode) {  // one box per lane: lanes overlap their TMA issues
              if (lane < 3) tma_load_2d(dst + lane * kBoxBytesK, &map_v, (3 * k + lane) * kBoxCols, j * kKeysT + 64 * h, fb);
            } else {
              issue_half<kHintK>(dst, kBoxBytesK, 3 * k * kBoxCols, 3, p, maps, len, kh, cur, fb, err);
            }
            __syncwarp();
          }
          if (q_helper && j == 0) {
            // This item's Q: latent pieces 0 .. kQProdPieces - 1 of the rows of this warp's TMEM lane
            // quadrant, once every S MMA of the previous item is done (both issuers commit to q_free
            // after their last tile of an item), so the Q region and the RoPE box are free.
            if (items > 0 && !waitb(&bars.q_free, (items - 1) & 1, X_Q_FREE, false)) { live = false; break; }
            const int rq = (warp & 3) * 32 + lane;
            const __nv_bfloat16 *qr, *qp;
            q_row_ptrs(it, rq, qr, qp);
            load_q_pieces<kFp8>(tbase + ((uint32_t)((warp & 3) * 32) << 16) + kTmemQ, qr, 0, kQProdPieces, p);
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(&bars.q_full);
          }
        }
        if (it.J > 0) ++items;
      }
      if constexpr (kSparse) cp_async_wait_all();  // no copy into this CTA outlives it
    } else if (warp == 5 || warp == 6) {
      // ---------------- S MMA issuers: even tiles (warp 5), odd tiles (warp 6) ----------------
      // A barrier wait by the thread that issued MMAs stalls until its queued MMAs drain;
      // the other issuer's queued tile keeps the tensor pipe busy meanwhile.
      if (lane == 0) {
        const uint32_t b = (uint32_t)(warp - 5);
        const uint32_t idesc = kFp8 ? idesc_f16_f32(kRows, kKeysT, false, false) : idesc_bf16_f32(kRows, kKeysT, false, false);
        const uint64_t a_rope = sdesc_sw128(smem_u32(smem + kOffQpe), 16, 1024);
        const uint32_t d_tmem = tbase + kTmemS + b * kKeysT;
        uint32_t t = 0, i = 0, nb = 0;  // all tiles, items with keys, this issuer's tiles
        bool live = true;
        while (live && iter.next(it)) {
          if (it.J == 0) continue;
          if (!wait1(&bars.q_full, i & 1, X_Q_FULL, false)) break;
          // prefill, sparse: group 2 of the first tile waits for the rows' part of Q (q_tail)
          bool tail = kDecode;
          auto take_tail = [&]() -> bool {
            if (tail) return true;
            if (!wait1(&bars.q_tail, i & 1, X_Q_FULL, false)) return false;
            tail = true;
            mbar_arrive(&bars.q_taken);
            return true;
          };
          if (kDecode) mbar_arrive(&bars.q_taken);
          for (int j = 0; j < it.J && live; ++j, ++t) {
            if ((t & 1u) != b) continue;
            // S buffer b was read by the rows (this issuer's previous tile)
            if (!wait1(&bars.s_free[b], (nb & 1) ^ 1, X_S_FREE, false)) { live = false; break; }
            // Nothing of this issuer is queued now, so testing the later groups costs no drain:
            // when all three have landed the tile goes out as one block of 36 MMAs; otherwise
            // group by group, waiting for each.
            if (!wait1(&bars.kfull[0][b], nb & 1, X_K_FULL, false)) { live = false; break; }
            const bool all = tail && mbar_try_wait(smem_u32(&bars.kfull[1][b]), nb & 1) &&
                             mbar_try_wait(smem_u32(&bars.kfull[2][b]), nb & 1);
            if (all) {
              tc_fence_after();
              if constexpr (kSparse) fence_proxy_async_smem();  // cp.async rows, read by the MMA
              mma_s_tile_n128(d_tmem, tbase + kTmemQ, sdesc_sw128(smem_u32(smem + kOffK), 16, 1024), a_rope, idesc,
                              smem_u32(&bars.kempty[0]), smem_u32(&bars.kempty[1]), smem_u32(&bars.kempty[2]));
            } else {
              for (int k = 0; k < kGroups; ++k) {
                if (k > 0 && !wait1(&bars.kfull[k][b], nb & 1, X_K_FULL, false)) { live = false; break; }
                if (k == 2 && !take_tail()) { live = false; break; }
                tc_fence_after();
                if constexpr (kSparse) fence_proxy_async_smem();
                const uint64_t bd = sdesc_sw128(smem_u32(smem + kOffK + k * kGroupBytes), 16, 1024);
                if (k < 2) mma_s_grp3_n128(d_tmem, tbase + kTmemQ + 96 * k, bd, idesc, (uint32_t)k);
                else mma_s_grp2r_n128(d_tmem, tbase + kTmemQ + 192, bd, a_rope, idesc);
                mma_commit(&bars.kempty[k]);
              }
              if (!live) break;
            }
            mma_commit(&bars.s_full[b]);
            ++nb;
          }
          if (!live || !take_tail()) break;  // an issuer with no tile in the item consumes q_tail too
          if (!kDecode) mma_commit(&bars.q_free);  // arrives once this issuer's MMAs of the item (reading Q) are done
          ++i;
        }
      }
      __syncwarp();
    } else if (warp == 7) {
      // ---------------- P copies into the O-CTA ----------------
      const uint8_t* pbuf = smem + kOffPS;
      const float* alpha = reinterpret_cast<const float*>(smem + kOffAlphaS);
      const uint32_t rem_p_full0 = map_to_rank(smem_u32(&bars.p_full[0]), peer);
      const uint32_t rem_p_full1 = map_to_rank(smem_u32(&bars.p_full[1]), peer);

      const uint32_t rem_p_o = map_to_rank(smem_u32(smem + kOffPO), peer);
      const uint32_t rem_alpha_o = map_to_rank(smem_u32(smem + kOffAlphaO), peer);
      uint32_t t = 0;
      bool live = true;
      while (live && iter.next(it)) {
        for (int j = 0; j < it.J; ++j, ++t) {
          const int sb = t & 1;
          if (!waitb(&bars.pwritten[sb], (t >> 1) & 1, X_P_WRITTEN, false) ||
              !waitb(&bars.pb_free[sb], ((t >> 1) & 1) ^ 1, X_PB_FREE, true)) {
            live = false;
            break;
          }
          if (lane == 0) {
            const uint32_t bar = sb ? rem_p_full1 : rem_p_full0;
            if constexpr (kSparse) {
              // two boxes on two barriers: P V of keys 0-63 starts once the first has landed
              mbar_arrive_expect_tx_remote(bar, kPBoxBytes + kRows * 4);
              bulk_copy_to_peer(rem_alpha_o + sb * kRows * 4, smem_u32(alpha + sb * kRows), kRows * 4, bar);
              bulk_copy_to_peer(rem_p_o + sb * kPBytesT, smem_u32(pbuf + sb * kPBytesT), kPBoxBytes, bar);
              const uint32_t bar1 = map_to_rank(smem_u32(&bars.p_full1[sb]), peer);
              mbar_arrive_expect_tx_remote(bar1, kPBoxBytes);
              bulk_copy_to_peer(rem_p_o + sb * kPBytesT + kPBoxBytes, smem_u32(pbuf + sb * kPBytesT + kPBoxBytes),
                                kPBoxBytes, bar1);
            } else {
              mbar_arrive_expect_tx_remote(bar, kPBytesT + kRows * 4);
              bulk_copy_to_peer(rem_p_o + sb * kPBytesT, smem_u32(pbuf + sb * kPBytesT), kPBytesT, bar);
              bulk_copy_to_peer(rem_alpha_o + sb * kRows * 4, smem_u32(alpha + sb * kRows), kRows * 4, bar);
            }
            bulk_commit();
            bulk_wait_read_all();  // this copy has read local buffer sb: the rows may refill it
            mbar_arrive(&bars.pbuf_free[sb]);
          }
          __syncwarp();
        }
      }
      if (lane == 0) bulk_wait_all();
    } else if (warp < kRowWarpsS) {
      // ---------------- rows: Q load, online softmax, one row per thread ----------------
      const int r = tid;  // row within the item = TMEM lane
      const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
      float* alpha = reinterpret_cast<float*>(smem + kOffAlphaS);
      const uint32_t rem_stats = map_to_rank(smem_u32(smem + kOffStatsO), peer);
      const uint32_t rem_stats_full = map_to_rank(smem_u32(&bars.stats_full), peer);
      const float sl2 = (p.scale_log2 == 0.f) ? 1e-30f : p.scale_log2;  // see mask_piece
      uint32_t t = 0, i = 0;
      bool live = true;
      while (live && iter.next(it)) {
        if (it.J == 0) continue;  // no key: the O-CTA writes these rows on its own
        // this row's query and the keys it sees from the item's first tile on
        const __nv_bfloat16 *qrow, *qpe;
        q_row_ptrs(it, r, qrow, qpe);
        const bool row_ok = qrow != nullptr;
        int64_t nkeys = 0;  // keys the row sees from the item's first tile on (prefill, decode)
        if (row_ok) {
          if constexpr (decode) nkeys = it.k1 - it.k0;
          else if constexpr (!kSparse) nkeys = keys_for_token(p, ((int64_t)it.id * kRows + r) / p.H);
        }
        // warm L2 with the next item's query row while this item runs (its Q load then
        // does not wait on HBM at the item boundary)
        {
          ItemIterT<kDecode, kSparse> peek = iter;
          ItemT nx;
          if (peek.next(nx) && nx.J > 0) {
            const __nv_bfloat16 *nq, *np;
            q_row_ptrs(nx, r, nq, np);
            if (nq) {
              const char* b = reinterpret_cast<const char*>(nq);
              for (int o = 0; o < kLatent * 2; o += 128) prefetch_l2(b + o);
              prefetch_l2(np);
            }
          }
        }
        MLA_TRACE_ONLY(long long tq = clock64();)
        // ---- Q: latent part -> TMEM (256 columns), RoPE part -> smem (SW128 K-major) ----
        if (i > 0 && !waitb(&bars.q_taken, (i - 1) & 1, X_Q_TAKEN, false)) break;
        load_q_pieces<kFp8>(tbase + lane_base + kTmemQ, row_ok ? qrow : nullptr, kDecode ? 0 : kQProdPieces, 8, p);
        load_q_rope<kFp8>(smem + kOffQpe + r * 128, row_ok ? qpe : nullptr, r, err,
                          kSparse ? (const void*)p.q_pe : (const void*)p.q, kSparse ? p.ext_q_pe : p.ext_q);
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(kDecode ? &bars.q_full : &bars.q_tail);

        MLA_TRACE_ONLY(trace_wait[24] += clock64() - tq;)
        float m_used = -CUDART_INF_F;  // log2-domain offset of the exponentials
        float l = 0.f;                 // running row sum (relative to m_used)
        int32_t nidx[4];               // sparse: raw top-k entries of the next tile (key 32 q + lane)
        if constexpr (kSparse) sparse_tile_entries(p, it.id, 0, nidx);
        for (int j = 0; j < it.J; ++j, ++t) {
          const int sb = t & 1;
          int nv;                              // keys of this tile visible to the row (sparse: 0 or 128)
          uint64_t vlo = ~0ull, vhi = ~0ull;   // sparse: which of keys 0-63 / 64-127 are listed
          if constexpr (kSparse) {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) w[q] = __ballot_sync(0xffffffffu, nidx[q] >= 0 && nidx[q] < p.S_kv);
            vlo = row_ok ? (w[0] | ((uint64_t)w[1] << 32)) : 0ull;
            vhi = row_ok ? (w[2] | ((uint64_t)w[3] << 32)) : 0ull;
            nv = (vlo | vhi) ? kKeysT : 0;
            if (j + 1 < it.J) sparse_tile_entries(p, it.id, j + 1, nidx);  // lands during this tile
          } else {
            const int64_t nv64 = nkeys - (int64_t)j * kKeysT;
            nv = (int)(nv64 < 0 ? 0 : (nv64 > kKeysT ? kKeysT : nv64));
          }

          if (!waitb(&bars.s_full[sb], (t >> 1) & 1, X_S_FULL, false)) { live = false; break; }
          tc_fence_after();
          MLA_TRACE_ONLY(long long tp = clock64();)
          // The exponentials are taken against the running offset m_used in one pass over the
          // tile's 128 scores (32-column pieces read from TMEM), which also finds the tile's
          // extreme.  Only when that extreme passes m_used by more than 2^8 (rare after a row's
          // first tile) does the row move m_used and take the pass again.  A row that has seen
          // no key yet finds the extreme first.
          const uint32_t scol = tbase + lane_base + kTmemS + sb * kKeysT;
          auto tile_offset = [&](const float (&eq)[4]) -> float {
            return (nv == 0) ? -CUDART_INF_F : extreme4<kUp>(eq) * sl2;
          };
          float a = 1.f;  // factor on the O accumulated so far
          // (tcgen05.ld is warp-collective: every branch around one is taken by the whole warp;
          // rows that need nothing from it recompute what they already have)
          if (__any_sync(0xffffffffu, m_used == -CUDART_INF_F)) {
            float eq[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) eq[k] = kUp ? -CUDART_INF_F : CUDART_INF_F;
#pragma unroll 1
            for (int pp = 0; pp < kKeysT / 32; pp += 2) {
              uint32_t s0[32], s1[32];
              tmem_ld32(scol + 32 * pp, s0);
              tmem_ld32(scol + 32 * pp + 32, s1);
              tmem_wait_ld();
              if constexpr (kSparse) {
                const uint64_t w = pp == 0 ? vlo : vhi;
                mask_bits<kUp>(s0, (uint32_t)w);
                mask_bits<kUp>(s1, (uint32_t)(w >> 32));
              } else {
                mask_piece<kUp>(s0, nv - 32 * pp);
                mask_piece<kUp>(s1, nv - 32 * pp - 32);
              }
              row_extreme<kUp>(s0, eq);
              row_extreme<kUp>(s1, eq);
            }
            if (m_used == -CUDART_INF_F) m_used = tile_offset(eq);  // still -inf when the tile shows no key
          }
          MLA_TRACE_ONLY(trace_wait[25] += clock64() - tp;)

          // ---- P (two K-major boxes of 64 keys) and the rescale factor ----
          if (!waitb(&bars.pbuf_free[sb], ((t >> 1) & 1) ^ 1, X_PBUF_FREE, false)) { live = false; break; }
          MLA_TRACE_ONLY(tp = clock64();)
          uint8_t* prow = smem + kOffPS + sb * kPBytesT + r * 128;
          uint64_t rsq[2];
          const uint64_t sl2x2 = f32x2(sl2, sl2);
          for (int pass = 0;; ++pass) {  // at most two passes: the second finds no larger extreme
            const float msub = (m_used == -CUDART_INF_F) ? 0.f : m_used;
            const uint64_t nmsub2 = f32x2(-msub, -msub);
            rsq[0] = rsq[1] = f32x2(0.f, 0.f);
            float eq[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) eq[k] = kUp ? -CUDART_INF_F : CUDART_INF_F;
#pragma unroll 1
            for (int p32 = 0; p32 < kKeysT / 32; ++p32) {
              uint32_t sr[32];
              tmem_ld32(scol + 32 * p32, sr);
              tmem_wait_ld();
              if constexpr (kSparse) mask_bits<kUp>(sr, (uint32_t)((p32 < 2 ? vlo : vhi) >> (32 * (p32 & 1))));
              else mask_piece<kUp>(sr, nv - 32 * p32);
              row_exp<kUp, kFp8>(sr, sl2x2, nmsub2, prow + (p32 >> 1) * kPBoxBytes, (4 * p32) & 7, r, rsq, eq);
            }
            const float mt = tile_offset(eq);
            const bool move = mt > m_used + kRescaleLog2;
            if (move) {  // the pass again, against the tile's own extreme
              const float an = ex2_approx(m_used - mt);
              a *= an;
              l *= an;
              m_used = mt;
            }
            if (!__any_sync(0xffffffffu, move) || pass == 1) break;
          }
          tc_fence_before();
          warp_arrive(&bars.s_free[sb]);  // every score of the tile is read: S buffer sb is free
          MLA_TRACE_ONLY(trace_wait[27] += clock64() - tp;)
          {
            float q0, q1, q2, q3;
            f32x2_split(rsq[0], q0, q1);
            f32x2_split(rsq[1], q2, q3);
            l += (q0 + q1) + (q2 + q3);
          }
          if (j == 0) a = 1.f;  // the first P V overwrites O
          alpha[sb * kRows + r] = a;
          fence_proxy_async_smem();  // the bulk copy reads through the async proxy
          warp_arrive(&bars.pwritten[sb]);
        }
        if (!live) break;
        // ---- row statistics into the O-CTA ----
        if (!waitb(&bars.stats_free, (i & 1) ^ 1, X_STATS_FREE, false)) break;
        st_cluster_f32x2(rem_stats + r * 8, m_used, l);
        warp_arrive_remote(rem_stats_full);
        ++i;
      }
    }
  } else {
    // =====================================================================
    // O-CTA
    // =====================================================================
    if ((kFp8 || kSparse) ? (warp == 4 || warp >= 6) : (warp == 4 || warp == 8)) {
      // ---------------- TMA producers: V halves (64 keys x 512 columns), epilogue stages ----------------
      // Ring slot h holds key half h of every tile (and then rows 64 h .. 64 h + 63 of the
      // epilogue); warp 4 fills slot 0 and warp 8 slot 1, each at its own issue rate.
      // Decode: the same warp also brings half h of tile j + kPrefetchTiles into L2 (one bulk
      // prefetch of its 64 contiguous cache rows when they lie in one page), so the S-CTA's K
      // loads of that tile hit L2: its one-tile K ring cannot cover the latency of HBM.
      // FP8 and sparse: eight warps fill the slots, four per half, two column boxes each (warp
      // 4 and warps 6-12 in order: half = index / 4, boxes 2 (index % 4) and the next).
      constexpr bool kEight = kFp8 || kSparse;
      const int vq = (warp == 4) ? 0 : warp - 5;
      const int h = kEight ? (vq >> 2) : ((warp == 4) ? 0 : 1);
      const int qq = kEight ? (vq & 3) : 0;
      const uint32_t dst = smem_u32(smem + kOffV + h * kHalfBytesV);
      uint32_t m = 0;      // uses of this slot
      uint32_t n_raw = 0;  // FP8: staged loads of this warp
      bool live = true;
      while (live && iter.next(it)) {
        const int len = decode ? decode_len_t(p, it.id) : 0;
        const int32_t* bt = decode ? p.block_table + (int64_t)decode_request(p, it.id) * p.max_pages : nullptr;
        const bool pf_ok = decode && p.page_size % 64 == 0;
        HalfIds ids;
        int32_t pf_pg = -1;  // page under half h of tile j + kPrefetchTiles (read a tile ahead)
        if constexpr (decode) {
          ids = load_half_ids(p, it.id, len, it.k0 + 64 * h);
          const int64_t kp = it.k0 + (int64_t)kPrefetchTiles * kKeysT + 64 * h;
          if (pf_ok && kp + 64 <= len && guard_span(err, G_BLOCK_TABLE, bt + kp / p.page_size, 4, p.block_table,
                                                    p.ext_block_table))
            pf_pg = __ldg(bt + kp / p.page_size);
        }
        if constexpr (kSparse) ids = sparse_half_ids(p, it.id, 64 * h);
        for (int j = 0; j < it.J && live; ++j, ++m) {
          const int64_t kh = it.k0 + (int64_t)j * kKeysT + 64 * h;
          HalfIds cur;
          if constexpr (kSparse) {
            cur = ids;
            if (j + 1 < it.J) ids = sparse_half_ids(p, it.id, kh + kKeysT);
          }
          if constexpr (decode) {
            cur = ids;
            if (j + 1 < it.J) ids = load_half_ids(p, it.id, len, kh + kKeysT);
            const int64_t kp = kh + (int64_t)kPrefetchTiles * kKeysT;
            if (lane == 0 && qq == 0 && pf_pg >= 0 && pf_pg < p.num_pages) {
              const int64_t row = pf_pg * (int64_t)p.page_size + kp % p.page_size;
              if constexpr (kFp8) bulk_prefetch_l2_hint<kHintPf>(p.cache8 + row * kDk, 64 * kDk);
              else bulk_prefetch_l2_hint<kHintPf>(p.cache + row * kDk, 64 * kDk * 2);
            }
            pf_pg = (pf_ok && kp + kKeysT + 64 <= len &&
                     guard_span(err, G_BLOCK_TABLE, bt + (kp + kKeysT) / p.page_size, 4, p.block_table,
                                p.ext_block_table))
                        ? __ldg(bt + (kp + kKeysT) / p.page_size)
                        : -1;
          }
          if (!waitb(&bars.vempty[h], (m & 1) ^ 1, X_V_EMPTY, false)) { live = false; break; }
          if constexpr (kSparse) {  // each lane arrives (noinc) once its row copies land
            gather_half_sparse<2>(dst + 2 * qq * kBoxBytesV, kBoxBytesV, 2 * qq, p, cur, &bars.vfull[h]);
            continue;
          }
          if constexpr (kFp8) {
            // as the K producers: two staged e4m3 boxes converted in place, or ordinary loads
            uint8_t* chunk0 = smem + kOffV + h * kHalfBytesV + 2 * qq * kBoxBytesV;
            const int32_t pg0 = __shfl_sync(0xffffffffu, cur.pe, 0);
            if (p.page_size % 64 == 0 && kh + 64 <= len && pg0 >= 0 && pg0 < p.num_pages) {
              uint64_t* rb = &bars.raw[8 + vq];
              if (lane == 0) mbar_arrive_expect_tx(rb, 2 * 4096);
              __syncwarp();
              const int32_t y = (int32_t)(pg0 * (int64_t)p.page_size + kh % p.page_size);
              if (lane < 2)
                tma_load_2d_hint<kHintV>(smem_u32(chunk0 + lane * kBoxBytesV + 4096), &maps.kv, (2 * qq + lane) * 64, y,
                                         rb);
              drain_bar = rb;
              drain_par = n_raw & 1;
              if (!waitb(rb, n_raw & 1, X_RAW, false)) { live = false; break; }
              ++n_raw;
#pragma unroll 1
              for (int b = 0; b < 2; ++b) convert_box_in_place(chunk0 + b * kBoxBytesV);
            } else {
              fill_half_fp8<2>(chunk0, kBoxBytesV, 2 * qq, p, len, kh, cur, err);
            }
            fence_proxy_async_smem();  // the MMA reads the slot through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.vfull[h]);
            continue;
          }
          if (lane == 0) mbar_arrive_expect_tx(&bars.vfull[h], kHalfBytesV);
          drain_bar = &bars.vfull[h];
          drain_par = m & 1;
          __syncwarp();
          if constexpr (!decode) {  // one box per lane
            if (lane < kVBoxes)
              tma_load_2d(dst + lane * kBoxBytesV, &map_v, lane * kBoxCols, j * kKeysT + 64 * h, &bars.vfull[h]);
          } else {
            issue_half<kHintV>(dst, kBoxBytesV, 0, kVBoxes, p, maps, len, kh, cur, &bars.vfull[h], err);
          }
          __syncwarp();
        }
        // the slot then stages the epilogue rows 64 h .. 64 h + 63 (with prev)
        if (staged && it.J > 0 && live) {
          if (!waitb(&bars.vempty[h], (m & 1) ^ 1, X_V_EMPTY, false)) { live = false; break; }
          const int64_t row0 = (int64_t)it.id * kRows + h * 64;
          if (kSparse) {  // no prev: every lane of the half's four warps arrives
            mbar_arrive(&bars.vfull[h]);
          } else if (p.prev_out && row0 < (int64_t)p.T * p.H) {
            if (lane == 0) mbar_arrive_expect_tx(&bars.vfull[h], kHalfBytesV);
            __syncwarp();
            if (lane < kVBoxes)
              tma_load_2d(dst + lane * kBoxBytesV, &maps.prev, lane * kBoxCols, (int32_t)row0, &bars.vfull[h]);
            drain_bar = &bars.vfull[h];
            drain_par = m & 1;
          } else if (lane == 0) {
            mbar_arrive(&bars.vfull[h]);
          }
          __syncwarp();
          ++m;
        }
      }
      if constexpr (kSparse) cp_async_wait_all();  // no copy into this CTA outlives it
    } else if (warp == 5) {
      // ---------------- P V issuer ----------------
      if (lane == 0) {
        const uint32_t idesc = kFp8 ? idesc_f16_f32(kRows, 256, false, true) : idesc_bf16_f32(kRows, 256, false, true);
        uint32_t t = 0, u = 0, i = 0;
        bool live = true;
        while (live && iter.next(it)) {
          if (it.J == 0) continue;
          if (i > 0 && !wait1(&bars.o_free, (i - 1) & 1, X_O_FREE, false)) break;
          for (int j = 0; j < it.J && live; ++j, ++t) {
            const int pb = t & 1;
            if (!wait1(&bars.p_ready[pb], (t >> 1) & 1, X_P_READY, false)) { live = false; break; }
            for (int h = 0; h < 2; ++h, ++u) {
              const int s = u & 1;
              if (!wait1(&bars.vfull[s], (u >> 1) & 1, X_V_FULL, false)) { live = false; break; }
              if (kSparse && h == 1 && !wait1(&bars.p_full1[pb], (t >> 1) & 1, X_P_FULL, true)) { live = false; break; }
              tc_fence_after();
              if constexpr (kSparse) fence_proxy_async_smem();  // cp.async rows, read by the MMA
              const uint32_t vst = smem_u32(smem + kOffV + s * kHalfBytesV);
              const uint32_t pst = smem_u32(smem + kOffPO + pb * kPBytesT + h * kPBoxBytes);
              mma_pv_k64_n512(tbase, tbase + 256, sdesc_sw128(pst, 16, 1024), sdesc_sw128(vst, kBoxBytesV, 1024),
                              sdesc_sw128(vst + 4 * kBoxBytesV, kBoxBytesV, 1024), idesc,
                              (j > 0 || h > 0) ? 1u : 0u);
              mma_commit(&bars.vempty[s]);
            }
            if (!live) break;
            mma_commit_multicast(&bars.pb_free[pb], 0x3);  // this CTA and the S-CTA
          }
          if (staged) u += 2;  // the epilogue's stages
          ++i;
        }
      }
      __syncwarp();
    } else if (warp < kRowWarpsO) {
      // ---------------- rows: lazy rescale, epilogue ----------------
      const int r = tid;
      const int half = r >> 6;
      const int rr = r & 63;
      const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
      const uint32_t rem_stats_free = map_to_rank(smem_u32(&bars.stats_free), peer);
      const float* alpha_o = reinterpret_cast<const float*>(smem + kOffAlphaO);
      const float* stats = reinterpret_cast<const float*>(smem + kOffStatsO);
      uint32_t t = 0, u = 0, i = 0;
      bool live = true;
      bool stored = false;
      while (live && iter.next(it)) {
        bool row_ok;
        float prev_l = -CUDART_INF_F;
        const __nv_bfloat16* prev_row = nullptr;
        __nv_bfloat16* orow = nullptr;
        float* orow_f = nullptr;   // decode: fp32 partial row in the workspace
        float* lse_dst = nullptr;
        if constexpr (decode) {
          row_ok = r < p.H;
          if (row_ok) {
            orow_f = p.part_o + ((int64_t)it.slot * p.H + r) * kLatent;
            lse_dst = p.part_lse + (int64_t)it.slot * p.H + r;
          }
        } else if constexpr (kSparse) {  // out [S, H * 512] = rows (t, h); lse [S, H] (nullable)
          row_ok = r < p.H;
          if (row_ok) {
            const int64_t f = (int64_t)it.id * p.H + r;
            orow = p.out + f * kLatent;
            if (p.lse) lse_dst = p.lse + f;
          }
        } else {
          const int64_t f = (int64_t)it.id * kRows + r;
          row_ok = f < (int64_t)p.T * p.H;
          if (row_ok) {
            const int64_t tt = f / p.H, hh = f - tt * p.H;
            orow = p.out + f * kLatent;
            lse_dst = p.lse + hh * (p.lse_stride ? p.lse_stride : (int64_t)p.T) + tt;
            if (p.prev_out) {
              prev_row = p.prev_out + f * kLatent;
              const float* pl = p.prev_lse + hh * (p.lse_stride ? p.lse_stride : (int64_t)p.T) + tt;
              prev_l = guard_span(err, G_PREV_LSE, pl, 4, p.prev_lse, p.ext_prev_lse) ? *pl : -CUDART_INF_F;
            }
          }
        }
        // guarded build: a row outside its buffer is not written (or read) at all
        if (orow && !guard_span(err, G_OUT, orow, kLatent * 2, p.out, p.ext_out)) orow = nullptr;
        if (orow_f && !guard_span(err, G_PART_O, orow_f, kLatent * 4, p.part_o, p.ext_part_o)) orow_f = nullptr;
        if (prev_row && !guard_span(err, G_PREV_OUT, prev_row, kLatent * 2, p.prev_out, p.ext_prev_out)) prev_row = nullptr;
        if (lse_dst && !guard_span(err, decode ? G_PART_LSE : G_LSE, lse_dst, 4, decode ? (const void*)p.part_lse : (const void*)p.lse,
                                   decode ? p.ext_part_lse : p.ext_lse))
          lse_dst = nullptr;
        if (it.J == 0) {
          // no key reaches these rows: out = prev (or 0), lse = prev_lse (or -inf); only
          // prefill has such items (decode segments always hold keys)
          if (row_ok && orow) {
            for (int c = 0; c < kLatent; c += 8) {
              uint4 v = prev_row ? *reinterpret_cast<const uint4*>(prev_row + c) : make_uint4(0, 0, 0, 0);
              *reinterpret_cast<uint4*>(orow + c) = v;
            }
            if (lse_dst) *lse_dst = prev_row ? prev_l : -CUDART_INF_F;
          }
          continue;
        }
        for (int j = 0; j < it.J; ++j, ++t) {
          const int pb = t & 1;
          if (!waitb(&bars.p_full[pb], (t >> 1) & 1, X_P_FULL, true)) { live = false; break; }
          const float a = alpha_o[pb * kRows + r];
          if (__any_sync(0xffffffffu, a != 1.f)) {
            // O holds every earlier P V before it is rescaled (P V of tile t-1 is done)
            if (!waitb(&bars.pb_free[(t - 1) & 1], ((t - 1) >> 1) & 1, X_PV_DONE, false)) { live = false; break; }
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
        u += 2 * it.J;

        // ---- epilogue ----
        if (!waitb(&bars.stats_full, i & 1, X_STATS_FULL, true)) break;
        const float m_used = stats[2 * r];
        const float l = stats[2 * r + 1];
        warp_arrive_remote(rem_stats_free);
        if (!waitb(&bars.pb_free[(t - 1) & 1], ((t - 1) >> 1) & 1, X_PV_DONE, false)) break;
        tc_fence_after();
        const bool has = l > 0.f;
        const float inv_l = has ? 1.f / l : 0.f;
        const float lse_new = has ? (m_used + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
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
        const float cn = wn * inv_l * (kFp8 ? p.kv_scale : 1.f);  // FP8: one e4m3 unit of V is kv_scale
        if constexpr (decode) {
          // fp32 partial rows (O / l) and their LSE for the split-K reduction
#pragma unroll 1
          for (int c0 = 0; c0 < kLatent; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tbase + lane_base + c0, v);
            tmem_wait_ld();
            if (row_ok && orow_f) {
              float4* dst = reinterpret_cast<float4*>(orow_f + c0);
#pragma unroll
              for (int q = 0; q < 8; ++q)
                dst[q] = make_float4(__uint_as_float(v[4 * q]) * cn, __uint_as_float(v[4 * q + 1]) * cn,
                                     __uint_as_float(v[4 * q + 2]) * cn, __uint_as_float(v[4 * q + 3]) * cn);
            }
          }
          tc_fence_before();
          warp_arrive(&bars.o_free);  // O has been read: the next item's P V may start
          if (row_ok && lse_dst) *lse_dst = lse_out;
          ++i;
          continue;
        }
        if (!staged) {
          // sparse with H < 128: each row stores its own bf16 row
#pragma unroll 1
          for (int c0 = 0; c0 < kLatent; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tbase + lane_base + c0, v);
            tmem_wait_ld();
            if (row_ok && orow) {
              uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
              for (int q = 0; q < 4; ++q)
                dst[q] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * q]) * cn, __uint_as_float(v[8 * q + 1]) * cn),
                                    pack_bf16x2(__uint_as_float(v[8 * q + 2]) * cn, __uint_as_float(v[8 * q + 3]) * cn),
                                    pack_bf16x2(__uint_as_float(v[8 * q + 4]) * cn, __uint_as_float(v[8 * q + 5]) * cn),
                                    pack_bf16x2(__uint_as_float(v[8 * q + 6]) * cn, __uint_as_float(v[8 * q + 7]) * cn));
            }
          }
          tc_fence_before();
          warp_arrive(&bars.o_free);
          if (row_ok && lse_dst) *lse_dst = lse_out;
          ++i;
          continue;
        }
        // rows of this half live in ring slot (u + half), [8 column boxes][64 rows][128 B] swizzled
        const uint32_t sidx = u + half;
        const int s = sidx & 1;
        if (!waitb(&bars.vfull[s], (sidx >> 1) & 1, X_V_FULL, false)) break;
        uint8_t* stage = smem + kOffV + s * kHalfBytesV;
        const bool use_prev = (prev_row != nullptr) && wp > 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < kLatent; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_base + c0, v);
          tmem_wait_ld();
          uint8_t* rowp = stage + (c0 >> 6) * kBoxBytesV + rr * 128;
          const int g0 = (c0 & 63) >> 3;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4* cell = reinterpret_cast<uint4*>(rowp + (((g0 + q) ^ (rr & 7)) << 4));
            float o[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) o[k] = __uint_as_float(v[8 * q + k]) * cn;
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
        tc_fence_before();
        warp_arrive(&bars.o_free);  // O has been read: the next item's P V may start
        if (row_ok && lse_dst) *lse_dst = lse_out;
        fence_proxy_async_smem();
        // both warps of this half staged their rows (a bounded wait, unlike a named barrier)
        warp_arrive(&bars.ep_half[half]);
        if (!waitb(&bars.ep_half[half], i & 1, X_EP_HALF, false)) break;
        if (rr == 0) {
          const int32_t row0 = it.id * kRows + half * 64;
          const uint32_t sbase = smem_u32(stage);
          for (int bx = 0; bx < kVBoxes; ++bx) tma_store_2d(&maps.out, bx * kBoxCols, row0, sbase + bx * kBoxBytesV);
          bulk_commit();
          bulk_wait_read_all();
          stored = true;
          mbar_arrive(&bars.vempty[s]);
        }
        u += 2;
        ++i;
      }
      if (stored) bulk_wait_all();
    }
  }

  // ---- teardown: drain on abort, then leave together ----
  __syncwarp();
  MLA_TRACE_ONLY(if (lane == 0) {
    for (int q = 0; q < 32; ++q) atomicAdd(&g_trace_wait[is_s ? 0 : 1][warp][q], trace_wait[q]);
    atomicAdd(&g_trace_total[is_s ? 0 : 1][warp], (unsigned long long)(clock64() - trace_t0));
  })
  if (*abort_flag) {
    // let what this thread issued land before the CTA leaves: its MMAs (one more commit, which
    // arrives once they are all done) and its TMA loads (their last full barrier phase)
    const bool mma_thread = lane == 0 && (is_s ? (warp == 5 || warp == 6) : warp == 5);
    if (mma_thread) {
      uint64_t* db = &bars.drain[is_s ? warp - 5 : 0];
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

template <bool kUp, bool kDecode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreadsT, 1)
    mla_prefill128_kernel(const __grid_constant__ CoreParams p, const __grid_constant__ CoreMaps maps) {
  prefill128_body<kUp, kDecode, false, false>(p, maps);
}

// Decode over the e4m3 cache.
template <bool kUp>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreadsT, 1)
    mla_prefill128_fp8_kernel(const __grid_constant__ CoreParams p, const __grid_constant__ CoreMaps maps) {
  prefill128_body<kUp, true, true, false>(p, maps);
}

// Top-k sparse attention (the scale is positive).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreadsT, 1)
    mla_prefill128_sparse_kernel(const __grid_constant__ CoreParams p, const __grid_constant__ CoreMaps maps) {
  prefill128_body<true, false, false, true>(p, maps);
}

}  // namespace

#ifdef MLA_TRACE
// copies the trace (2 x 16 x 32 wait sums, then 2 x 16 totals) to host and clears it
extern "C" int mla_trace_read(unsigned long long* host) {
  static unsigned long long zero[2 * 16 * 32] = {};
  if (cudaMemcpyFromSymbol(host, g_trace_wait, sizeof(g_trace_wait)) != cudaSuccess) return 1;
  if (cudaMemcpyFromSymbol(host + 1024, g_trace_total, sizeof(g_trace_total)) != cudaSuccess) return 1;
  if (cudaMemcpyToSymbol(g_trace_wait, zero, sizeof(g_trace_wait)) != cudaSuccess) return 1;
  if (cudaMemcpyToSymbol(g_trace_total, zero, sizeof(g_trace_total)) != cudaSuccess) return 1;
  return 0;
}
#endif

cudaError_t launch_prefill128(const CoreParams& p, const CoreMaps& maps, cudaStream_t stream) {
  static PerDeviceOnce attrs;
  cudaError_t e = attrs.run([] {
    cudaError_t r = cudaSuccess;
    auto set = [&](const void* fn) {
      if (r == cudaSuccess) r = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemT);
    };
    set((const void*)mla_prefill128_kernel<true, false>);
    set((const void*)mla_prefill128_kernel<false, false>);
    set((const void*)mla_prefill128_kernel<true, true>);
    set((const void*)mla_prefill128_kernel<false, true>);
    set((const void*)mla_prefill128_fp8_kernel<true>);
    set((const void*)mla_prefill128_fp8_kernel<false>);
    set((const void*)mla_prefill128_sparse_kernel);
    return r;
  });
  if (e != cudaSuccess) return e;
  if (p.num_pairs <= 0) return cudaSuccess;
  const dim3 grid(2 * p.num_pairs), block(kThreadsT);
  const bool up = p.scale_log2 >= 0.f;
  if (p.mode == MODE_SPARSE) {
    mla_prefill128_sparse_kernel<<<grid, block, kSmemT, stream>>>(p, maps);
  } else if (p.mode == MODE_DECODE && p.cache8) {
    if (up) mla_prefill128_fp8_kernel<true><<<grid, block, kSmemT, stream>>>(p, maps);
    else mla_prefill128_fp8_kernel<false><<<grid, block, kSmemT, stream>>>(p, maps);
  } else if (p.mode == MODE_DECODE) {
    if (up) mla_prefill128_kernel<true, true><<<grid, block, kSmemT, stream>>>(p, maps);
    else mla_prefill128_kernel<false, true><<<grid, block, kSmemT, stream>>>(p, maps);
  } else {
    if (up) mla_prefill128_kernel<true, false><<<grid, block, kSmemT, stream>>>(p, maps);
    else mla_prefill128_kernel<false, false><<<grid, block, kSmemT, stream>>>(p, maps);
  }
  return cudaGetLastError();
}

}  // namespace mla
