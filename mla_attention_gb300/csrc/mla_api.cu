// The C ABI of libmla: argument validation, workspace checks, TMA tensor
// maps and kernel launches.  Nothing here computes attention; every step of
// the path runs in the kernels of this directory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "mla_internal.h"

namespace mla {

namespace {

thread_local char g_err[512] = {0};
std::atomic<uint32_t> g_spin_limit{kDefaultSpinLimit};
std::atomic<uint32_t> g_debug_stall{0};

mla_status fail(mla_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

mla_status ok() {
  g_err[0] = 0;
  return MLA_OK;
}

mla_status cuda_fail(cudaError_t e, const char* where) {
  return fail(MLA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define MLA_REQUIRE(cond, ...)                            \
  do {                                                    \
    if (!(cond)) return fail(MLA_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

}  // namespace

uint32_t spin_limit() { return g_spin_limit.load(std::memory_order_relaxed); }
uint32_t debug_stall() { return g_debug_stall.load(std::memory_order_relaxed); }

mla_status set_last_error(mla_status s, const char* msg) { return fail(s, "%s", msg); }

CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t d[5];
  cuuint64_t s[4];
  cuuint32_t b[5], e[5];
  for (uint32_t i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  return g_encode(map, dtype, rank, const_cast<void*>(base), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

int device_sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  static int cached[64] = {0};
  if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n <= 0) n = 1;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

namespace {

// 2-D bf16 map [rows, cols] (cols contiguous), 128B swizzle, box {64 cols, box_rows}
mla_status map2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t row_stride_elems,
                 uint32_t box_rows, const char* what) {
  uint64_t dims[2] = {cols, rows};
  uint64_t strides[1] = {row_stride_elems * 2};
  uint32_t box[2] = {64, box_rows};
  CUresult r = encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box,
                            CU_TENSOR_MAP_SWIZZLE_128B);
  if (r != CUDA_SUCCESS) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", what, (int)r);
  return MLA_OK;
}

uint32_t* ws_err(void* ws) { return reinterpret_cast<uint32_t*>(ws); }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Keys per score tile of prefill (and sparse) and of decode: 128 (mla_prefill128_kernel) or 64
// (mla_core_kernel); set with mla_set_tile_keys.
constexpr int kDefaultPrefillKeys = 128, kDefaultDecodeKeys = 128;
std::atomic<int> g_prefill_keys{kDefaultPrefillKeys};
std::atomic<int> g_decode_keys{kDefaultDecodeKeys};

int default_pairs() {
  int p = device_sm_count() / 2;
  return p < 1 ? 1 : p;
}

}  // namespace
}  // namespace mla

using namespace mla;

// ---------------------------------------------------------------------------
namespace {
// 3-D bf16 map over rows of one head: {K columns, H heads, T tokens}, box {64, 1, 128}, SW128
mla_status map_head_rows(CUtensorMap* m, const void* base, uint64_t K, uint64_t H, uint64_t T, int64_t stride_h,
                         int64_t stride_t, const char* what) {
  uint64_t dims[3] = {K, H, T};
  uint64_t strides[2] = {(uint64_t)stride_h * 2, (uint64_t)stride_t * 2};
  uint32_t box[3] = {64, 1, 128};
  CUresult r = encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box,
                            CU_TENSOR_MAP_SWIZZLE_128B);
  if (r != CUDA_SUCCESS) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", what, (int)r);
  return MLA_OK;
}

mla_status run_bmm(bool lift, const void* a, int64_t a_st, int64_t a_sh, const void* w, int T, int H, void* out,
                   int64_t o_st, int64_t o_sh, void* workspace, size_t workspace_bytes, void* stream,
                   const char* name) {
  const int K = lift ? 128 : kLatent, N = lift ? kLatent : 128;
  MLA_REQUIRE(T >= 0 && H >= 1, "%s: need T >= 0, H >= 1", name);
  if (!workspace || workspace_bytes < kWsHeader)
    return fail(MLA_ERR_WORKSPACE, "%s: workspace must hold %zu bytes", name, (size_t)kWsHeader);
  if (T == 0) return ok();
  MLA_REQUIRE(a && w && out, "%s: every tensor is required", name);
  MLA_REQUIRE(aligned16(a) && aligned16(w) && aligned16(out), "%s: tensors must be 16-byte aligned", name);
  MLA_REQUIRE(a_sh >= K && a_st >= (int64_t)H * a_sh && (a_sh * 2) % 16 == 0 && (a_st * 2) % 16 == 0,
              "%s: input rows need head stride >= %d and token stride >= H x head stride, multiples of 8 elements",
              name, K);
  MLA_REQUIRE(o_sh >= N && o_st >= (int64_t)H * o_sh && o_sh % 8 == 0 && o_st % 8 == 0,
              "%s: output rows need head stride >= %d, token stride >= H x head stride, multiples of 8", name, N);
  CUtensorMap ma, mb, mo;
  mla_status s = map_head_rows(&ma, a, K, H, T, a_sh, a_st, "bmm rows");
  if (s == MLA_OK) s = map_head_rows(&mo, out, N, H, T, o_sh, o_st, "bmm output rows");
  if (s != MLA_OK) return s;
  s = map2d(&mb, w, K, (uint64_t)H * N, K, lift ? 256 : 128, "bmm weights");
  if (s != MLA_OK) return s;
  BmmParams p;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.out_stride_t = o_st;
  p.out_stride_h = o_sh;
  p.T = T;
  p.H = H;
  p.N = N;
  p.err = ws_err(workspace);
  p.spin_limit = spin_limit();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = lift ? launch_absorb_q(p, ma, mb, mo, st) : launch_project_out(p, ma, mb, mo, st);
  if (e != cudaSuccess) return cuda_fail(e, name);
  return ok();
}
}  // namespace

namespace {
mla_status prefill_one(const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* kv, int64_t kv_stride,
                       int T, int H, int Tkv, int dk, int dv, float scale, int causal, int64_t q_pos0,
                       int64_t kv_pos0, int kv_valid, const void* prev_out, const float* prev_lse, void* out,
                       float* lse, int64_t lse_stride, void* workspace, size_t workspace_bytes, void* stream) {
  MLA_REQUIRE(T >= 0 && H >= 1 && Tkv >= 0, "mla_prefill: need T >= 0, H >= 1, Tkv >= 0 (T=%d H=%d Tkv=%d)", T, H,
              Tkv);
  MLA_REQUIRE(dk > dv && dv > 0, "mla_prefill: V must be narrower than K (dk=%d dv=%d)", dk, dv);
  if (dk != kDk || dv != kLatent)
    return fail(MLA_ERR_UNSUPPORTED, "mla_prefill: only dk=576, dv=512 is built (got %d, %d)", dk, dv);
  MLA_REQUIRE(std::isfinite(scale), "mla_prefill: scale must be finite");
  MLA_REQUIRE((prev_out == nullptr) == (prev_lse == nullptr), "mla_prefill: prev_out and prev_lse go together");
  if (kv_valid < 0) kv_valid = Tkv;
  MLA_REQUIRE(kv_valid <= Tkv, "mla_prefill: kv_valid (%d) > Tkv (%d)", kv_valid, Tkv);
  if (!workspace || workspace_bytes < mla_prefill_workspace_size(T, H))
    return fail(MLA_ERR_WORKSPACE, "mla_prefill: workspace must hold %zu bytes", mla_prefill_workspace_size(T, H));
  if (T == 0) return ok();
  MLA_REQUIRE(q && out && lse, "mla_prefill: q, out and lse are required");
  MLA_REQUIRE(aligned16(q) && aligned16(out) && (!prev_out || aligned16(prev_out)),
              "mla_prefill: q, out, prev_out must be 16-byte aligned");
  MLA_REQUIRE(q_stride_h >= kDk && q_stride_t >= 0 && (q_stride_h % 8) == 0 && (q_stride_t % 8) == 0,
              "mla_prefill: q strides must be multiples of 8 elements with q_stride_h >= 576");
  if (kv_valid > 0) {
    MLA_REQUIRE(kv != nullptr, "mla_prefill: kv is NULL");
    MLA_REQUIRE(aligned16(kv) && (kv_stride % 8) == 0 && kv_stride >= kDk,
                "mla_prefill: kv must be 16-byte aligned with kv_stride a multiple of 8 and >= 576");
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  CoreMaps maps;
  memset(&maps, 0, sizeof(maps));
  const bool tile128 = g_prefill_keys.load() == 128;
  if (kv_valid > 0) {
    mla_status s = map2d(&maps.kv, kv, kDk, (uint64_t)kv_valid, (uint64_t)kv_stride, kKeys, "kv");
    if (s == MLA_OK && tile128) s = map2d(&maps.row, kv, kDk, (uint64_t)kv_valid, (uint64_t)kv_stride, 128, "kv");
    if (s != MLA_OK) return s;
  }
  {
    const uint64_t rows = (uint64_t)T * (uint64_t)H;  // output rows are 32-bit signed tensor-map coordinates
    MLA_REQUIRE(rows <= (uint64_t)INT32_MAX, "mla_prefill: T * H must be below 2^31");
    mla_status s = map2d(&maps.out, out, kLatent, rows, kLatent, 64, "out");
    if (s == MLA_OK && prev_out) s = map2d(&maps.prev, prev_out, kLatent, rows, kLatent, 64, "prev_out");
    if (s != MLA_OK) return s;
  }
  CoreParams p;
  memset(&p, 0, sizeof(p));
  p.mode = MODE_PREFILL;
  p.num_pairs = default_pairs();
  p.scale_log2 = scale * 1.4426950408889634f;
  p.spin_limit = spin_limit();
  p.debug_stall = debug_stall();
  p.err = ws_err(workspace);
  p.q = reinterpret_cast<const __nv_bfloat16*>(q);
  p.q_stride_t = q_stride_t;
  p.q_stride_h = q_stride_h;
  p.T = T;
  p.H = H;
  p.q_pos0 = q_pos0;
  p.kv_pos0 = kv_pos0;
  p.kv_valid = kv_valid;
  p.causal = causal ? 1 : 0;
  p.prev_out = reinterpret_cast<const __nv_bfloat16*>(prev_out);
  p.prev_lse = prev_lse;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.lse_stride = lse_stride;
  {
    const uint64_t hs = (uint64_t)(lse_stride ? lse_stride : (int64_t)T);  // head stride of lse / prev_lse
    p.ext_q = ((uint64_t)(T - 1) * (uint64_t)q_stride_t + (uint64_t)(H - 1) * (uint64_t)q_stride_h + kDk) * 2;
    p.ext_out = (uint64_t)T * H * kLatent * 2;
    p.ext_prev_out = prev_out ? p.ext_out : 0;
    p.ext_lse = ((uint64_t)(H - 1) * hs + (uint64_t)T) * 4;
    p.ext_prev_lse = prev_lse ? p.ext_lse : 0;
  }
  const int64_t items = ((int64_t)T * H + kRows - 1) / kRows;
  if (items < p.num_pairs) p.num_pairs = (int)items;
  cudaError_t e = tile128 ? launch_prefill128(p, maps, st) : launch_core(p, maps, st);
  if (e != cudaSuccess) return cuda_fail(e, "mla_prefill launch");
  return ok();
}
}  // namespace

namespace {
mla_status decode_impl(const void* q, int q_per_req, const void* kv_cache, bool fp8, float kv_scale, int64_t num_pages,
                       int page_size, const int32_t* block_table, int max_pages, const int32_t* lens, int B, int H,
                       float scale, const float* sinks, int num_splits, void* out, float* lse, void* workspace,
                       size_t workspace_bytes, void* stream) {
  MLA_REQUIRE(B >= 0 && H >= 1 && num_pages >= 0 && max_pages >= 0 && num_splits >= 0,
              "mla_decode: need B >= 0, H >= 1, num_pages >= 0, max_pages >= 0, num_splits >= 0");
  MLA_REQUIRE(q_per_req >= 1 && (int64_t)B * q_per_req <= (int64_t)1 << 24,
              "mla_decode: q_per_req >= 1 and B * q_per_req <= 2^24 (got %d, %d)", q_per_req, B);
  const int G = B * q_per_req;  // query groups: one query token of one request each
  if (H > kRows) return fail(MLA_ERR_UNSUPPORTED, "mla_decode: H <= 128 (got %d)", H);
  MLA_REQUIRE(page_size == 16 || page_size == 32 || (page_size > 0 && page_size % 64 == 0),
              "mla_decode: page_size must be 16, 32 or a multiple of 64 (got %d)", page_size);
  MLA_REQUIRE(std::isfinite(scale), "mla_decode: scale must be finite");
  const size_t need = mla_decode_workspace_size(G, H, num_splits);
  if (!workspace || workspace_bytes < need)
    return fail(MLA_ERR_WORKSPACE, "mla_decode: workspace must hold %zu bytes", need);
  if (B == 0) return ok();
  MLA_REQUIRE(q && kv_cache && block_table && lens && out, "mla_decode: q, kv_cache, block_table, lens, out required");
  MLA_REQUIRE(aligned16(q) && aligned16(kv_cache) && aligned16(out), "mla_decode: q, kv_cache, out 16-byte aligned");
  MLA_REQUIRE(num_pages >= 1 && max_pages >= 1, "mla_decode: need at least one page");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  CoreMaps maps;
  memset(&maps, 0, sizeof(maps));
  const uint64_t rows = (uint64_t)num_pages * (uint64_t)page_size;
  // cache rows are 32-bit signed tensor-map coordinates
  MLA_REQUIRE(rows <= (uint64_t)INT32_MAX, "mla_decode: num_pages * page_size must be below 2^31");
  if (!fp8) {
    mla_status s = map2d(&maps.kv, kv_cache, kDk, rows, kDk, page_size >= kKeys ? kKeys : (uint32_t)page_size, "cache");
    if (s != MLA_OK) return s;
    s = map2d(&maps.row, kv_cache, kDk, rows, kDk, 1, "cache rows");
    if (s != MLA_OK) return s;
    maps.pe = maps.row;
  } else {
    // the e4m3 cache as bytes [rows, 576], boxes of 64 bytes x 64 rows with no swizzle: the kernel
    // stages them and converts in place (ordinary loads where a 64-key half spans pages)
    const uint64_t dims[2] = {(uint64_t)kDk, rows};
    const uint64_t strides[1] = {(uint64_t)kDk};
    const uint32_t box[2] = {64, 64};
    CUresult r = encode_tiled(&maps.kv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, kv_cache, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_NONE);
    if (r != CUDA_SUCCESS) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled(e4m3 cache) failed: %d", (int)r);
  }
  CoreParams p;
  memset(&p, 0, sizeof(p));
  p.mode = MODE_DECODE;
  p.num_pairs = num_splits > 0 ? num_splits : default_pairs();
  p.scale_log2 = scale * (fp8 ? kv_scale : 1.f) * 1.4426950408889634f;  // FP8: scores of e4m3 units
  p.spin_limit = spin_limit();
  p.debug_stall = debug_stall();
  p.err = ws_err(workspace);
  p.q = reinterpret_cast<const __nv_bfloat16*>(q);
  p.H = H;
  p.block_table = block_table;
  p.lens = lens;
  p.B = G;
  p.q_per_req = q_per_req;
  p.sinks = sinks;
  p.max_pages = max_pages;
  p.page_size = page_size;
  p.num_pages = num_pages;
  p.cache = fp8 ? nullptr : reinterpret_cast<const __nv_bfloat16*>(kv_cache);
  p.cache8 = fp8 ? reinterpret_cast<const uint8_t*>(kv_cache) : nullptr;
  p.kv_scale = kv_scale;
  char* w = reinterpret_cast<char*>(workspace) + kWsHeader;
  const size_t slots = (size_t)G + (size_t)p.num_pairs;
  p.tile_prefix = reinterpret_cast<int32_t*>(w);
  w += align_up(sizeof(int32_t) * ((size_t)G + 1), 256);
  p.part_lse = reinterpret_cast<float*>(w);
  w += align_up(sizeof(float) * slots * (size_t)H, 256);
  p.part_o = reinterpret_cast<float*>(w);
  p.ext_q = (uint64_t)G * H * kDk * 2;
  p.ext_out = (uint64_t)G * H * kLatent * 2;
  p.ext_lse = lse ? (uint64_t)G * H * 4 : 0;
  p.ext_block_table = (uint64_t)B * max_pages * 4;
  p.ext_lens = (uint64_t)B * 4;
  p.ext_cache8 = fp8 ? rows * kDk : 0;
  p.ext_sinks = sinks ? (uint64_t)H * 4 : 0;
  p.ext_tile_prefix = ((uint64_t)G + 1) * 4;
  p.ext_part_lse = slots * H * 4;
  p.ext_part_o = slots * H * kLatent * 4;
  // FP8 runs on the 128-key engine only
  cudaError_t e = (fp8 || g_decode_keys.load() == 128) ? launch_prefill128(p, maps, st) : launch_core(p, maps, st);
  if (e != cudaSuccess) return cuda_fail(e, "mla_decode launch");
  e = launch_decode_reduce(p, reinterpret_cast<__nv_bfloat16*>(out), lse, st);
  if (e != cudaSuccess) return cuda_fail(e, "mla_decode reduce launch");
  return ok();
}
}  // namespace

extern "C" {

int mla_version(void) { return 100; }

const char* mla_last_error_string(void) { return g_err; }

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    case MLA_ERR_DEVICE_RANGE: return "MLA_ERR_DEVICE_RANGE";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
  }
  return "MLA_UNKNOWN";
}

void mla_set_spin_limit(uint32_t limit) { g_spin_limit.store(limit ? limit : kDefaultSpinLimit); }

void mla_set_tile_keys(int prefill_keys, int decode_keys) {
  if (prefill_keys == 0) prefill_keys = kDefaultPrefillKeys;
  if (decode_keys == 0) decode_keys = kDefaultDecodeKeys;
  if (prefill_keys == 64 || prefill_keys == 128) g_prefill_keys.store(prefill_keys);
  if (decode_keys == 64 || decode_keys == 128) g_decode_keys.store(decode_keys);
}

void mla_debug_inject_stall(int enable) { g_debug_stall.store(enable ? 1u : 0u); }

mla_status mla_check_device_status(void* workspace, void* stream, uint32_t* detail) {
  if (!workspace) return fail(MLA_ERR_INVALID_ARG, "mla_check_device_status: workspace is NULL");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(word), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "mla_check_device_status");
  if (detail) *detail = word;
  if (word == 0) return ok();
  if ((word & 0xF000u) == DEV_TIMEOUT_BASE)
    return fail(MLA_ERR_TIMEOUT, "a device wait ran out of its spin bound (site 0x%x)", word & 0xFFFu);
  if ((word & 0xF000u) == DEV_GUARD_BASE)
    return fail(MLA_ERR_DEVICE_RANGE, "guarded build: an access left its buffer (site %u)", word & 0xFFFu);
  return fail(MLA_ERR_DEVICE_RANGE, "a kernel met an out-of-range index (site 0x%x)", word & 0xFFFu);
}

// ---------------------------------------------------------------------------
size_t mla_prefill_workspace_size(int T, int H) {
  (void)T;
  (void)H;
  return kWsHeader;
}

mla_status mla_prefill(const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* kv, int64_t kv_stride,
                       int T, int H, int Tkv, int dk, int dv, float scale, int causal, int64_t q_pos0,
                       int64_t kv_pos0, int kv_valid, const void* prev_out, const float* prev_lse, void* out,
                       float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  return prefill_one(q, q_stride_t, q_stride_h, kv, kv_stride, T, H, Tkv, dk, dv, scale, causal, q_pos0, kv_pos0,
                     kv_valid, prev_out, prev_lse, out, lse, 0, workspace, workspace_bytes, stream);
}

size_t mla_prefill_varlen_workspace_size(int total_q, int H) { return mla_prefill_workspace_size(total_q, H); }

mla_status mla_prefill_varlen(const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* kv,
                              int64_t kv_stride, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, int batch,
                              int H, int dk, int dv, float scale, int causal, const void* prev_out,
                              const float* prev_lse, void* out, float* lse, void* workspace, size_t workspace_bytes,
                              void* stream) {
  MLA_REQUIRE(batch >= 0 && cu_seqlens_q && cu_seqlens_kv, "mla_prefill_varlen: batch >= 0 and host cu_seqlens");
  MLA_REQUIRE(cu_seqlens_q[0] == 0 && cu_seqlens_kv[0] == 0, "mla_prefill_varlen: cu_seqlens start at 0");
  for (int b = 0; b < batch; ++b)
    MLA_REQUIRE(cu_seqlens_q[b + 1] >= cu_seqlens_q[b] && cu_seqlens_kv[b + 1] >= cu_seqlens_kv[b],
                "mla_prefill_varlen: cu_seqlens must not decrease (sequence %d)", b);
  const int64_t total_q = cu_seqlens_q[batch];
  MLA_REQUIRE((prev_out == nullptr) == (prev_lse == nullptr), "mla_prefill_varlen: prev_out and prev_lse go together");
  if (!workspace || workspace_bytes < mla_prefill_varlen_workspace_size((int)total_q, H))
    return fail(MLA_ERR_WORKSPACE, "mla_prefill_varlen: workspace must hold %zu bytes",
                mla_prefill_varlen_workspace_size((int)total_q, H));
  const char* bq = reinterpret_cast<const char*>(q);
  const char* bkv = reinterpret_cast<const char*>(kv);
  for (int b = 0; b < batch; ++b) {
    const int q0 = cu_seqlens_q[b], ql = cu_seqlens_q[b + 1] - q0;
    const int k0 = cu_seqlens_kv[b], kl = cu_seqlens_kv[b + 1] - k0;
    if (ql == 0) continue;
    // one sequence: the cached prefix precedes its queries (query i sees keys j <= kl - ql + i)
    const int64_t row0 = (int64_t)q0 * H;  // first (token, head) row of the sequence
    mla_status s = prefill_one(
        bq + 2 * (int64_t)q0 * q_stride_t, q_stride_t, q_stride_h, kl ? bkv + 2 * (int64_t)k0 * kv_stride : nullptr,
        kv_stride, ql, H, kl, dk, dv, scale, causal, (int64_t)kl - ql, 0, kl,
        prev_out ? reinterpret_cast<const char*>(prev_out) + 2 * row0 * dv : nullptr,
        prev_lse ? prev_lse + q0 : nullptr, reinterpret_cast<char*>(out) + 2 * row0 * dv, lse + q0, total_q,
        workspace, workspace_bytes, stream);
    if (s != MLA_OK) return s;
  }
  return ok();
}

// ---------------------------------------------------------------------------
size_t mla_decode_workspace_size(int B, int H, int num_splits) {
  const int P = num_splits > 0 ? num_splits : default_pairs();
  const size_t slots = (size_t)B + (size_t)P;
  size_t sz = kWsHeader;
  sz += align_up(sizeof(int32_t) * ((size_t)B + 1), 256);    // tile prefix
  sz += align_up(sizeof(float) * slots * (size_t)H, 256);    // partial lse
  sz += align_up(sizeof(float) * slots * (size_t)H * kLatent, 256);  // partial out
  return sz;
}

size_t mla_decode_ex_workspace_size(int B, int q_per_req, int H, int num_splits) {
  return mla_decode_workspace_size(B * (q_per_req > 0 ? q_per_req : 1), H, num_splits);
}

mla_status mla_decode(const void* q, const void* kv_cache, int64_t num_pages, int page_size,
                      const int32_t* block_table, int max_pages, const int32_t* lens, int B, int H, float scale,
                      int num_splits, void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  return mla_decode_ex(q, 1, kv_cache, num_pages, page_size, block_table, max_pages, lens, B, H, scale, nullptr,
                       num_splits, out, lse, workspace, workspace_bytes, stream);
}

mla_status mla_decode_ex(const void* q, int q_per_req, const void* kv_cache, int64_t num_pages, int page_size,
                         const int32_t* block_table, int max_pages, const int32_t* lens, int B, int H, float scale,
                         const float* sinks, int num_splits, void* out, float* lse, void* workspace,
                         size_t workspace_bytes, void* stream) {
  return decode_impl(q, q_per_req, kv_cache, false, 1.f, num_pages, page_size, block_table, max_pages, lens, B, H,
                     scale, sinks, num_splits, out, lse, workspace, workspace_bytes, stream);
}

size_t mla_decode_fp8_workspace_size(int B, int q_per_req, int H, int num_splits) {
  return mla_decode_ex_workspace_size(B, q_per_req, H, num_splits);
}

mla_status mla_decode_fp8(const void* q, int q_per_req, const void* kv_cache_e4m3, float kv_scale, int64_t num_pages,
                          int page_size, const int32_t* block_table, int max_pages, const int32_t* lens, int B, int H,
                          float scale, const float* sinks, int num_splits, void* out, float* lse, void* workspace,
                          size_t workspace_bytes, void* stream) {
  MLA_REQUIRE(std::isfinite(kv_scale) && kv_scale > 0.f, "mla_decode_fp8: kv_scale must be finite and > 0");
  return decode_impl(q, q_per_req, kv_cache_e4m3, true, kv_scale, num_pages, page_size, block_table, max_pages, lens,
                     B, H, scale, sinks, num_splits, out, lse, workspace, workspace_bytes, stream);
}


// ---------------------------------------------------------------------------
size_t mla_sparse_workspace_size(int S, int H) {
  (void)S;
  (void)H;
  return kWsHeader;
}

mla_status mla_sparse(const void* q_lift, const void* q_pe, const void* c_kv, const void* k_pe, const int32_t* topk,
                      int B, int S, int S_kv, int H, int K, float softmax_scale, void* out, float* lse,
                      void* workspace, size_t workspace_bytes, void* stream) {
  MLA_REQUIRE(B == 1, "mla_sparse: B must be 1 (got %d)", B);
  MLA_REQUIRE(S >= 0 && S_kv >= 1 && H >= 1 && K >= 1, "mla_sparse: need S >= 0, S_kv >= 1, H >= 1, K >= 1");
  if (H > kRows) return fail(MLA_ERR_UNSUPPORTED, "mla_sparse: H <= 128 (got %d)", H);
  MLA_REQUIRE(softmax_scale > 0.f && std::isfinite(softmax_scale), "mla_sparse: softmax_scale must be positive");
  if (!workspace || workspace_bytes < mla_sparse_workspace_size(S, H))
    return fail(MLA_ERR_WORKSPACE, "mla_sparse: workspace must hold %zu bytes", mla_sparse_workspace_size(S, H));
  if (S == 0) return ok();
  MLA_REQUIRE(q_lift && q_pe && c_kv && k_pe && topk && out, "mla_sparse: tensors must be non-NULL");
  MLA_REQUIRE(aligned16(q_lift) && aligned16(q_pe) && aligned16(c_kv) && aligned16(k_pe) && aligned16(out),
              "mla_sparse: tensors must be 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  CoreMaps maps;
  memset(&maps, 0, sizeof(maps));
  mla_status s = map2d(&maps.row, c_kv, kLatent, (uint64_t)S_kv, kLatent, 1, "c_kv");
  if (s != MLA_OK) return s;
  s = map2d(&maps.pe, k_pe, kRope, (uint64_t)S_kv, kRope, 1, "k_pe");
  if (s != MLA_OK) return s;
  s = map2d(&maps.out, out, kLatent, (uint64_t)S * (uint64_t)H, kLatent, 64, "out");
  if (s != MLA_OK) return s;
  maps.kv = maps.row;
  CoreParams p;
  memset(&p, 0, sizeof(p));
  p.mode = MODE_SPARSE;
  p.num_pairs = default_pairs();
  if (S < p.num_pairs) p.num_pairs = S;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.spin_limit = spin_limit();
  p.debug_stall = debug_stall();
  p.err = ws_err(workspace);
  p.q = reinterpret_cast<const __nv_bfloat16*>(q_lift);
  p.q_pe = reinterpret_cast<const __nv_bfloat16*>(q_pe);
  p.T = S;
  p.H = H;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.topk = topk;
  p.c_kv = reinterpret_cast<const __nv_bfloat16*>(c_kv);
  p.k_pe = reinterpret_cast<const __nv_bfloat16*>(k_pe);
  p.K = K;
  p.S_kv = S_kv;
  p.ext_q = (uint64_t)S * H * kLatent * 2;
  p.ext_q_pe = (uint64_t)S * H * kRope * 2;
  p.ext_out = (uint64_t)S * H * kLatent * 2;
  p.ext_lse = lse ? (uint64_t)S * H * 4 : 0;
  p.ext_topk = (uint64_t)S * K * 4;
  p.ext_c_kv = (uint64_t)S_kv * kLatent * 2;
  p.ext_k_pe = (uint64_t)S_kv * kRope * 2;
  // the prefill engine choice applies to sparse as well (both are context-phase attention)
  cudaError_t e = g_prefill_keys.load() == 128 ? launch_prefill128(p, maps, st) : launch_core(p, maps, st);
  if (e != cudaSuccess) return cuda_fail(e, "mla_sparse launch");
  return ok();
}

// ---------------------------------------------------------------------------
size_t mla_prefill_split_workspace_size(int Nq, int H) {
  (void)Nq;
  (void)H;
  return kWsHeader;
}

mla_status mla_prefill_split(const void* q_nope, const void* q_pe, const void* k_nope, const void* k_pe,
                             const void* v, const int32_t* seq_len_host, int seq_len_rows, int batch, int head_num,
                             int kv_head_num, float qk_scale, int mask_type, const void* prev_out,
                             const float* prev_lse, void* out, float* lse, void* workspace, size_t workspace_bytes,
                             void* stream) {
  MLA_REQUIRE(batch >= 1 && batch <= kSplitMaxBatch, "mla_prefill_split: 1 <= batch <= %d (got %d)", kSplitMaxBatch,
              batch);
  MLA_REQUIRE(seq_len_host != nullptr && (seq_len_rows == 1 || seq_len_rows == 2),
              "mla_prefill_split: seq_len_host [batch] or [2, batch] (seq_len_rows 1 or 2)");
  MLA_REQUIRE(head_num >= 1 && kv_head_num >= 0, "mla_prefill_split: head_num >= 1, kv_head_num >= 0");
  const int Hkv = kv_head_num ? kv_head_num : head_num;
  MLA_REQUIRE(head_num % Hkv == 0, "mla_prefill_split: head_num %% kv_head_num must be 0 (%d, %d)", head_num, Hkv);
  MLA_REQUIRE(mask_type == 0 || mask_type == 1, "mla_prefill_split: mask_type 0 (NO_MASK) or 1 (TRIU)");
  MLA_REQUIRE(std::isfinite(qk_scale), "mla_prefill_split: qk_scale must be finite");
  MLA_REQUIRE((prev_out == nullptr) == (prev_lse == nullptr), "mla_prefill_split: prev_out and prev_lse go together");
  SplitParams p;
  memset(&p, 0, sizeof(p));
  int64_t nq = 0, nkv = 0, tiles = 0;
  for (int b = 0; b < batch; ++b) {
    const int ql = seq_len_host[b];
    const int kl = seq_len_rows == 2 ? seq_len_host[batch + b] : ql;
    MLA_REQUIRE(ql >= 0 && kl >= 0, "mla_prefill_split: negative sequence length at %d", b);
    p.q_off[b] = (int)nq;
    p.kv_off[b] = (int)nkv;
    p.tile_off[b] = (int)tiles;
    nq += ql;
    nkv += kl;
    tiles += (ql + kRows - 1) / kRows;
    MLA_REQUIRE(nq < (1ll << 31) && nkv < (1ll << 31), "mla_prefill_split: too many tokens");
  }
  MLA_REQUIRE(tiles * head_num < (1ll << 31), "mla_prefill_split: too many (query tile, head) items");
  p.q_off[batch] = (int)nq;
  p.kv_off[batch] = (int)nkv;
  p.tile_off[batch] = (int)tiles;
  if (!workspace || workspace_bytes < mla_prefill_split_workspace_size((int)nq, head_num))
    return fail(MLA_ERR_WORKSPACE, "mla_prefill_split: workspace must hold %zu bytes",
                mla_prefill_split_workspace_size((int)nq, head_num));
  if (nq == 0) return ok();
  MLA_REQUIRE(q_nope && q_pe && out && lse, "mla_prefill_split: q_nope, q_pe, out, lse required");
  MLA_REQUIRE(nkv == 0 || (k_nope && k_pe && v), "mla_prefill_split: k_nope, k_pe, v required");
  MLA_REQUIRE(aligned16(q_nope) && aligned16(q_pe) && aligned16(out) && (!prev_out || aligned16(prev_out)) &&
                  (nkv == 0 || (aligned16(k_nope) && aligned16(k_pe) && aligned16(v))),
              "mla_prefill_split: tensors must be 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // 3-D maps [tokens][heads][cols]: box {64 cols, 1 head, 128 tokens}
  CUtensorMap m[5];
  memset(m, 0, sizeof(m));
  struct Spec {
    const void* base;
    uint64_t cols, heads, tokens;
  } specs[5] = {{q_nope, 128, (uint64_t)head_num, (uint64_t)nq},
                {q_pe, 64, (uint64_t)head_num, (uint64_t)nq},
                {k_nope, 128, (uint64_t)Hkv, (uint64_t)nkv},
                {k_pe, 64, (uint64_t)Hkv, (uint64_t)nkv},
                {v, 128, (uint64_t)Hkv, (uint64_t)nkv}};
  for (int i = 0; i < 5; ++i) {
    if (specs[i].tokens == 0) continue;
    uint64_t dims[3] = {specs[i].cols, specs[i].heads, specs[i].tokens};
    uint64_t strides[2] = {specs[i].cols * 2, specs[i].cols * specs[i].heads * 2};
    uint32_t box[3] = {64, 1, (uint32_t)kRows};
    CUresult r = encode_tiled(&m[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, specs[i].base, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled(split %d) failed: %d", i, (int)r);
  }
  p.batch = batch;
  p.H = head_num;
  p.Hkv = Hkv;
  p.Nq = (int)nq;
  p.Nkv = (int)nkv;
  p.scale_log2 = qk_scale * 1.4426950408889634f;
  p.causal = mask_type;
  p.spin_limit = spin_limit();
  p.debug_stall = debug_stall();
  p.err = ws_err(workspace);
  p.total_q_tiles = (int)tiles;
  p.prev_out = reinterpret_cast<const __nv_bfloat16*>(prev_out);
  p.prev_lse = prev_lse;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.ticket = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(workspace) + kWsTicket);
  cudaError_t e = cudaMemsetAsync(p.ticket, 0, sizeof(uint32_t), st);  // the kernel's CTAs claim items from 0
  if (e != cudaSuccess) return cuda_fail(e, "mla_prefill_split ticket reset");
  e = launch_split(p, m[0], m[1], m[2], m[3], m[4], st);
  if (e != cudaSuccess) return cuda_fail(e, "mla_prefill_split launch");
  return ok();
}


mla_status mla_absorb_q(const void* q_nope, int64_t q_nope_stride_t, int64_t q_nope_stride_h,
                        const void* k_b_proj_trans, int T, int H, void* q_out, int64_t q_out_stride_t,
                        int64_t q_out_stride_h, void* workspace, size_t workspace_bytes, void* stream) {
  return run_bmm(true, q_nope, q_nope_stride_t, q_nope_stride_h, k_b_proj_trans, T, H, q_out, q_out_stride_t,
                 q_out_stride_h, workspace, workspace_bytes, stream, "mla_absorb_q");
}

mla_status mla_project_out(const void* o_latent, const void* v_b_proj, int T, int H, void* out,
                           int64_t out_stride_t, int64_t out_stride_h, void* workspace, size_t workspace_bytes,
                           void* stream) {
  return run_bmm(false, o_latent, (int64_t)H * kLatent, kLatent, v_b_proj, T, H, out, out_stride_t, out_stride_h,
                 workspace, workspace_bytes, stream, "mla_project_out");
}

// ---------------------------------------------------------------------------
size_t mla_rope_append_workspace_size(int B) {
  (void)B;
  return kWsHeader;
}

mla_status mla_rope_append(const void* q_pe, const void* c_kv, const void* k_pe, const int32_t* positions,
                           const float* cos_sin, int max_pos, int is_neox, void* kv_cache, int64_t num_pages,
                           int page_size, const int32_t* block_table, int max_pages, int B, int H, void* q_out,
                           void* workspace, size_t workspace_bytes, void* stream) {
  MLA_REQUIRE(B >= 0 && H >= 1 && max_pos >= 1 && num_pages >= 0 && page_size >= 1 && max_pages >= 0,
              "mla_rope_append: need B >= 0, H >= 1, max_pos >= 1, num_pages >= 0, page_size >= 1, max_pages >= 0");
  MLA_REQUIRE(is_neox == 0 || is_neox == 1, "mla_rope_append: is_neox must be 0 or 1");
  if (!workspace || workspace_bytes < mla_rope_append_workspace_size(B))
    return fail(MLA_ERR_WORKSPACE, "mla_rope_append: workspace must hold %zu bytes", mla_rope_append_workspace_size(B));
  if (B == 0) return ok();
  MLA_REQUIRE(q_pe && c_kv && k_pe && positions && cos_sin && kv_cache && block_table && q_out,
              "mla_rope_append: every tensor is required");
  MLA_REQUIRE(aligned16(q_pe) && aligned16(c_kv) && aligned16(k_pe) && aligned16(kv_cache) && aligned16(q_out),
              "mla_rope_append: bf16 tensors must be 16-byte aligned");
  RopeAppendParams p;
  p.q_pe = reinterpret_cast<const __nv_bfloat16*>(q_pe);
  p.c_kv = reinterpret_cast<const __nv_bfloat16*>(c_kv);
  p.k_pe = reinterpret_cast<const __nv_bfloat16*>(k_pe);
  p.positions = positions;
  p.cos_sin = cos_sin;
  p.block_table = block_table;
  p.cache = reinterpret_cast<__nv_bfloat16*>(kv_cache);
  p.q_out = reinterpret_cast<__nv_bfloat16*>(q_out);
  p.err = ws_err(workspace);
  p.num_pages = num_pages;
  p.max_pos = max_pos;
  p.is_neox = is_neox;
  p.page_size = page_size;
  p.max_pages = max_pages;
  p.B = B;
  p.H = H;
  cudaError_t e = launch_rope_append(p, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_rope_append launch");
  return ok();
}

// ---------------------------------------------------------------------------
mla_status mla_merge_lse(const void* out_a, const float* lse_a, const void* out_b, const float* lse_b, void* out,
                         float* lse, int64_t rows, int H, int dv, void* stream) {
  MLA_REQUIRE(rows >= 0 && H >= 1 && dv >= 8 && dv % 8 == 0, "mla_merge_lse: rows >= 0, H >= 1, dv %% 8 == 0");
  if (rows == 0) return ok();
  MLA_REQUIRE(out_a && lse_a && out_b && lse_b && out && lse, "mla_merge_lse: all tensors required");
  MLA_REQUIRE(aligned16(out_a) && aligned16(out_b) && aligned16(out), "mla_merge_lse: outputs 16-byte aligned");
  cudaError_t e = launch_merge(reinterpret_cast<const __nv_bfloat16*>(out_a), lse_a,
                               reinterpret_cast<const __nv_bfloat16*>(out_b), lse_b,
                               reinterpret_cast<__nv_bfloat16*>(out), lse, rows, H, dv,
                               reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_merge_lse launch");
  return ok();
}

}  // extern "C"
