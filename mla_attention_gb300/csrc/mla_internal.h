// Internal interfaces between the C-ABI layer (mla_api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "../../include/mla.h"
#include "mla_device_status.h"

namespace mla {

// ---------------------------------------------------------------------------
// geometry of the absorbed (latent) path
// ---------------------------------------------------------------------------
constexpr int kLatent = 512;            // V width = latent width
constexpr int kRope = 64;               // RoPE columns
constexpr int kDk = kLatent + kRope;    // 576
constexpr int kRows = 128;              // query rows per tile (MMA M)
constexpr int kKeys = 64;               // keys per KV tile (MMA N of QK^T, K of PV)
constexpr int kBoxCols = 64;            // 64 bf16 = 128 B: one 128B-swizzle row
constexpr int kKBoxes = kDk / kBoxCols;       // 9 column boxes for K (576 columns)
constexpr int kVBoxes = kLatent / kBoxCols;   // 8 column boxes for V (512 columns)

// ---------------------------------------------------------------------------
// workspace layout (shared by every call): a 256-byte header first
// ---------------------------------------------------------------------------
constexpr size_t kWsHeader = 256;       // [0]: device status word
constexpr size_t kWsTicket = 64;        // split kernel: next work item to claim (zeroed before each launch)
constexpr uint32_t kDefaultSpinLimit = 1u << 25;

uint32_t spin_limit();                  // process-wide bound for device waits
uint32_t debug_stall();                 // 1: kernels wait on a barrier nothing arrives on (tests)

// kinds of work the absorbed tile engine runs
enum CoreMode : int { MODE_PREFILL = 0, MODE_DECODE = 1, MODE_SPARSE = 2 };

struct CoreParams {
  int mode;
  int num_pairs;          // CTA pairs in the grid (cluster of 2 per pair)
  float scale_log2;       // scale * log2(e)
  uint32_t spin_limit;
  uint32_t debug_stall;   // tests: the MMA warps wait on a barrier that is never arrived on
  uint32_t* err;          // device status word

  // ---- query rows ----
  const __nv_bfloat16* q;        // prefill / decode: [.., 576] rows; sparse: q_lift [.., 512]
  const __nv_bfloat16* q_pe;     // sparse: q_pe [.., 64]
  int64_t q_stride_t;            // prefill: token stride (elements)
  int64_t q_stride_h;            // prefill: head stride (elements)
  int T;                         // prefill: tokens; sparse: S
  int H;                         // heads

  // ---- prefill ----
  int64_t q_pos0, kv_pos0;
  int kv_valid;
  int causal;
  const __nv_bfloat16* prev_out; // [T,H,512] or null
  const float* prev_lse;         // [H,T] or null
  __nv_bfloat16* out;            // prefill: [T,H,512]; sparse: [S,H*512]
  float* lse;                    // prefill: [H,T]; sparse: [S,H] (nullable)
  int64_t lse_stride;            // prefill: head stride of lse / prev_lse (0 = T)

  // ---- decode ----
  const int32_t* block_table;    // [B, max_pages]
  const int32_t* lens;           // [B]
  int B;
  int max_pages;
  int page_size;
  int64_t num_pages;
  const __nv_bfloat16* cache;    // [num_pages * page_size, 576] rows (L2 prefetch addresses)
  const uint8_t* cache8;         // FP8 decode: e4m3 rows [num_pages * page_size, 576] (else null)
  float kv_scale;                // FP8 decode: value of one e4m3 unit (the epilogue scales O by it)
  int q_per_req;                 // query tokens per request (B above counts B_req * q_per_req groups)
  const float* sinks;            // [H] per-head sink logit, or null (used by the reduction)
  int32_t* tile_prefix;          // ws: [B+1] tiles before request b (written by CTA 0)
  float* part_o;                 // ws: [slots, H, 512]
  float* part_lse;               // ws: [slots, H]

  // ---- sparse ----
  const int32_t* topk;           // [S, K]
  const __nv_bfloat16* c_kv;     // [S_kv, 512] rows, read with 16-byte copies
  const __nv_bfloat16* k_pe;     // [S_kv, 64] rows, read with 16-byte copies
  int K;
  int S_kv;

  // ---- byte extents of the buffers above from their base pointers (the guarded build checks
  // every plain access against them; 0 where a buffer is unused) ----
  uint64_t ext_q, ext_q_pe, ext_out, ext_prev_out, ext_lse, ext_prev_lse;
  uint64_t ext_block_table, ext_lens, ext_cache8, ext_sinks;
  uint64_t ext_tile_prefix, ext_part_o, ext_part_lse;
  uint64_t ext_topk, ext_c_kv, ext_k_pe;
};

// Decode query groups: group g is query token g % q_per_req of request g / q_per_req.  Token i of a
// request of len keys sits at position len - q_per_req + i and sees keys 0 .. len - q_per_req + i
// (causal among the request's query tokens; with one token it sees all len keys).
__device__ __forceinline__ int decode_request(const CoreParams& p, int g) {
  return p.q_per_req > 1 ? g / p.q_per_req : g;
}
__device__ __forceinline__ int decode_group_len(const CoreParams& p, int g) {
  const int64_t cap = (int64_t)p.max_pages * p.page_size;
  int64_t n;
  if (p.q_per_req <= 1) {  // one token per request: it sees all len keys
    n = guard_span(p.err, G_LENS, p.lens + g, 4, p.lens, p.ext_lens) ? p.lens[g] : 0;
    if (n > cap) n = cap;
  } else {
    const int s = p.q_per_req;
    const int b = g / s;
    int64_t len = guard_span(p.err, G_LENS, p.lens + b, 4, p.lens, p.ext_lens) ? p.lens[b] : 0;
    if (len > cap) len = cap;
    n = len - s + 1 + (g - (int64_t)b * s);
  }
  return (int)(n < 0 ? 0 : n);
}

// An entry of the block table (guarded build: an entry outside the table's extent reads as -1, an
// invalid page, and is recorded).
__device__ __forceinline__ int32_t bt_entry(const CoreParams& p, const int32_t* e) {
  return guard_span(p.err, G_BLOCK_TABLE, e, 4, p.block_table, p.ext_block_table) ? *e : -1;
}

// TMA descriptors of one launch of the absorbed engine
struct CoreMaps {
  CUtensorMap kv;    // K/V rows [rows, 576] (prefill: the chunk; decode: the cache), box {64, 64 or page};
                     // FP8 decode: the e4m3 cache as bytes, box {64 bytes, 64 rows}, no swizzle
  CUtensorMap row;   // gather rows, box {64, 1} (decode: the cache; sparse: c_kv [S_kv, 512])
  CUtensorMap pe;    // sparse: k_pe [S_kv, 64], box {64, 1}
  CUtensorMap out;   // prefill / sparse output rows [rows, 512], box {64, 64}
  CUtensorMap prev;  // prefill previous output rows [rows, 512], box {64, 64}
};

// Runs a set-up step (the kernels' shared-memory attributes) once on each device that launches
// the kernel, from any number of host threads: the attribute belongs to the device that is
// current when it is set, so a process that drives several GPUs sets it on each.
class PerDeviceOnce {
 public:
  template <class F>
  cudaError_t run(F&& setup) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (done_[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    e = setup();
    if (e == cudaSuccess) done_[dev].store(true, std::memory_order_release);
    return e;
  }

 private:
  static constexpr int kMaxDevices = 64;
  std::mutex mu_;
  std::atomic<bool> done_[kMaxDevices] = {};
};

// decode step: RoPE on q_pe / k_pe and the paged latent-cache append
struct RopeAppendParams {
  const __nv_bfloat16* q_pe;     // [B, H, 64]
  const __nv_bfloat16* c_kv;     // [B, 512]
  const __nv_bfloat16* k_pe;     // [B, 64]
  const int32_t* positions;      // [B]
  const float* cos_sin;          // [max_pos, 64]
  const int32_t* block_table;    // [B, max_pages]
  __nv_bfloat16* cache;          // [num_pages * page_size, 576] rows
  __nv_bfloat16* q_out;          // [B, H, 576] (columns 512..575 written)
  uint32_t* err;
  int64_t num_pages;
  int max_pos, is_neox, page_size, max_pages, B, H;
};
cudaError_t launch_rope_append(const RopeAppendParams& p, cudaStream_t stream);

// absorption BMMs: D[t, n] = sum_k A[t, k] B[h][n, k] per head, bf16 out with token/head strides
struct BmmParams {
  __nv_bfloat16* out;
  int64_t out_stride_t, out_stride_h;  // elements
  int T, H, N;                         // tokens, heads, columns of D (512 for q_lift, 128 for the output)
  uint32_t* err;
  uint32_t spin_limit;
};
// A map: 3-D {K, H, T} box {64, 1, 128}; B map: 2-D {K, H * N} box {64, 256 (q_lift) / 128 (output)}
// (output map: 3-D {N, H, T} with the output strides, box {64, 1, 128})
cudaError_t launch_absorb_q(const BmmParams& p, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo,
                            cudaStream_t stream);
cudaError_t launch_project_out(const BmmParams& p, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo,
                               cudaStream_t stream);

// kernels' host launchers (return cudaError_t of the launch)
cudaError_t launch_core(const CoreParams& p, const CoreMaps& maps, cudaStream_t stream);
// prefill and decode with 128-key score tiles.  Prefill: maps.row holds the K rows with box
// {64, 128}, maps.kv the V rows with box {64, 64}.  Decode: maps.kv the cache rows with box
// {64, 64} (whole pages), maps.row the cache rows with box {64, 1} (gathers).
cudaError_t launch_prefill128(const CoreParams& p, const CoreMaps& maps, cudaStream_t stream);
size_t core_smem_bytes();

cudaError_t launch_merge(const __nv_bfloat16* out_a, const float* lse_a, const __nv_bfloat16* out_b,
                         const float* lse_b, __nv_bfloat16* out, float* lse, int64_t rows, int H, int dv,
                         cudaStream_t stream);

cudaError_t launch_decode_reduce(const CoreParams& p, __nv_bfloat16* out, float* lse, cudaStream_t stream);

// non-absorbed split layout
struct SplitParams {
  int batch;
  int H, Hkv;
  int Nq, Nkv;
  float scale_log2;
  int causal;
  uint32_t spin_limit;
  uint32_t debug_stall;
  uint32_t* err;
  int total_q_tiles;           // sum over sequences of ceil(q_len / 128)
  uint32_t* ticket;            // ws: work items claimed so far (0 at launch)
  const __nv_bfloat16* prev_out;
  const float* prev_lse;
  __nv_bfloat16* out;
  float* lse;
  // per-sequence tables (kernel parameters; batch <= kMaxBatch)
  int q_off[257];
  int kv_off[257];
  int tile_off[257];
};
constexpr int kSplitMaxBatch = 256;

cudaError_t launch_split(const SplitParams& p, const CUtensorMap& mq_nope, const CUtensorMap& mq_pe,
                         const CUtensorMap& mk_nope, const CUtensorMap& mk_pe, const CUtensorMap& mv,
                         cudaStream_t stream);

// ---------------------------------------------------------------------------
// host helpers
// ---------------------------------------------------------------------------
// cuTensorMapEncodeTiled through the runtime's driver entry point
CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swizzle);

int device_sm_count();

// Record `msg` as the calling thread's last error and return `s`.
mla_status set_last_error(mla_status s, const char* msg);

}  // namespace mla
