// The absorption BMMs around the latent attention (TensorRT-LLM "mla.py",
// forward_absorption_generation): per head h,
//   q_lift[t, h, :] = q_nope[t, h, :] x k_b_proj_trans[h]^T   ([T, 128] x [128, 512]), written
//                     into the latent part of the fused query [T, H, 576];
//   out[t, h, :]    = O[t, h, :] x v_b_proj[h]^T              ([T, 512] x [512, 128]).
// Both are D[t, n] = sum_k A[t, k] B[n, k] with A rows of one head (strided in memory) and B
// the head's weight, K-major: one tcgen05 kernel serves both.
//
// Persistent: one CTA per SM walks a contiguous range of items (128-token tile, head, kN-column
// slice of D; the slices of one tile and head are neighbours, so their shared A rows are read
// from HBM once and from L2 after).  Warp 0 streams A and B through a ring of TMA stages (A: a
// 3-D box {64 columns, 1 head, 128 tokens} -> 128 rows x 128 B, SW128; B: a 2-D box of kN weight
// rows), warp 1 issues M128 x kN x K16 MMAs (both operands from shared memory) into one of two
// TMEM accumulators of kN columns, and warps 2-5 (one per TMEM lane quadrant) read an item's
// accumulator back into bf16 rows staged in shared memory, which TMA stores write out.  The
// two accumulators let an item's epilogue run while the next item's MMAs do, and the ring
// keeps loading meanwhile.
#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

constexpr int kRowsM = 128;              // tokens per tile
constexpr int kChunk = 64;               // K columns per stage (one 128-byte swizzled row)
constexpr int kABytes = kRowsM * 128;    // 16 KB
constexpr int kBmmThreads = 192;         // warps: 0 TMA, 1 MMA, 2-5 epilogue

enum : uint32_t { B_FULL = 0x70, B_EMPTY, B_ACC_FULL, B_ACC_EMPTY, B_STAGE_FULL, B_STAGE_FREE };

struct BmmBars {
  uint64_t full[8], empty[8];
  uint64_t acc_full[2], acc_empty[2];  // accumulator b holds an item / was read out
  uint64_t stage_full, stage_free;     // epilogue staging written (4 warps) / read by its TMA stores
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
};

template <int kN, int kK, int kStages>
__global__ void __launch_bounds__(kBmmThreads, 1)
    absorb_bmm_kernel(const __grid_constant__ BmmParams p, const __grid_constant__ CUtensorMap ma,
                      const __grid_constant__ CUtensorMap mb, const __grid_constant__ CUtensorMap mo) {
  constexpr int kBBytes = kN * 128;
  constexpr int kStageBytes = kABytes + kBBytes;
  constexpr int kChunks = kK / kChunk;
  constexpr int kOffStage = kStages * kStageBytes;  // the staged output tile: kN / 64 boxes of 16 KB
  static_assert(kStages <= 8 && kN <= 256 && kN % 64 == 0 && kK % kChunk == 0, "tile shape");
  extern __shared__ __align__(1024) uint8_t smem[];
  BmmBars& bars = *reinterpret_cast<BmmBars*>(smem + kOffStage + (kN / 64) * kABytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* err = p.err;
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) record_error(err, DEV_RANGE_BASE | 0x7F);
    return;
  }
  // this CTA's items: a contiguous share of (token tile, head, slice), slices fastest
  const int n_slices = p.N / kN;
  const int64_t n_items = (int64_t)((p.T + kRowsM - 1) / kRowsM) * p.H * n_slices;
  const int64_t i0 = n_items * blockIdx.x / gridDim.x, i1 = n_items * (blockIdx.x + 1) / gridDim.x;
  auto item = [&](int64_t i, int& t0, int& h, int& n0) {
    n0 = (int)(i % n_slices) * kN;
    const int64_t th = i / n_slices;
    h = (int)(th % p.H);
    t0 = (int)(th / p.H) * kRowsM;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.acc_full[b], 1);
      mbar_init(&bars.acc_empty[b], 4);
    }
    mbar_init(&bars.stage_full, 4);
    mbar_init(&bars.stage_free, 1);
    mbar_init(&bars.drain, 1);
    bars.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars.tmem_base, 2 * kN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars.tmem_base;
  volatile uint32_t* abort_flag = &bars.abort_flag;
  auto wait1 = [&](uint64_t* bar, uint32_t parity, uint32_t site) -> bool {
    const bool ok = (*abort_flag == 0) && mbar_wait(bar, parity, err, site, p.spin_limit);
    if (!ok) *abort_flag = 1;
    return ok;
  };
  auto waitw = [&](uint64_t* bar, uint32_t parity, uint32_t site) -> bool {  // warp-uniform
    bool ok = (*abort_flag == 0) && mbar_wait(bar, parity, err, site, p.spin_limit);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) *abort_flag = 1;
    return ok;
  };
  uint64_t* drain_bar = nullptr;
  uint32_t drain_par = 0;
  bool stored = false;

  if (warp == 0) {
    // ---- TMA producer: lane 0 issues the A box of each stage and lane 1 the B box (a thread
    // issues a box only every few hundred cycles, so the two overlap) ----
    uint32_t g = 0;  // chunks issued
    for (int64_t i = i0; i < i1; ++i) {
      int t0, h, n0;
      item(i, t0, h, n0);
      bool live = true;
      for (int c = 0; c < kChunks; ++c, ++g) {
        const int s = g % kStages;
        if (!waitw(&bars.empty[s], ((g / kStages) & 1) ^ 1, B_EMPTY)) { live = false; break; }
        const uint32_t st = smem_u32(smem + s * kStageBytes);
        if (lane == 0) mbar_arrive_expect_tx(&bars.full[s], kStageBytes);
        __syncwarp();
        if (lane == 0) tma_load_3d(st, &ma, c * kChunk, h, t0, &bars.full[s]);
        if (lane == 1) tma_load_2d(st + kABytes, &mb, c * kChunk, h * p.N + n0, &bars.full[s]);
        drain_bar = &bars.full[s];
        drain_par = (g / kStages) & 1;
      }
      if (!live) break;
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer: item u into accumulator u % 2 ----
    const uint32_t idesc = idesc_bf16_f32(kRowsM, kN, false, false);
    uint32_t g = 0, u = 0;
    for (int64_t i = i0; i < i1; ++i, ++u) {
      const uint32_t b = u & 1;
      if (!wait1(&bars.acc_empty[b], ((u >> 1) & 1) ^ 1, B_ACC_EMPTY)) break;
      tc_fence_after();
      bool live = true;
      for (int c = 0; c < kChunks; ++c, ++g) {
        const int s = g % kStages;
        if (!wait1(&bars.full[s], (g / kStages) & 1, B_FULL)) { live = false; break; }
        tc_fence_after();
        const uint32_t st = smem_u32(smem + s * kStageBytes);
#pragma unroll
        for (int k16 = 0; k16 < kChunk / 16; ++k16)
          mma_ss(tbase + b * kN, sdesc_sw128(st + 32 * k16, 16, 1024), sdesc_sw128(st + kABytes + 32 * k16, 16, 1024),
                 idesc, (c | k16) != 0 ? 1u : 0u);
        mma_commit(&bars.empty[s]);
      }
      if (!live) break;
      mma_commit(&bars.acc_full[b]);
    }
  } else if (warp >= 2) {
    // ---- epilogue: token row (warp % 4) * 32 + lane of an item, kN columns -> bf16 rows staged as
    // 64-column SW128 boxes, then TMA stores (rows past T are clipped) ----
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    uint8_t* stage = smem + kOffStage;
    uint32_t u = 0;
    for (int64_t i = i0; i < i1; ++i, ++u) {
      int t0, h, n0;
      item(i, t0, h, n0);
      const uint32_t b = u & 1;
      if (!waitw(&bars.acc_full[b], (u >> 1) & 1, B_ACC_FULL)) break;
      // the previous item's TMA stores have read the staging buffer
      if (u > 0 && !waitw(&bars.stage_free, (u - 1) & 1, B_STAGE_FREE)) break;
      tc_fence_after();
#pragma unroll 1
      for (int c0 = 0; c0 < kN; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_base + b * kN + c0, v);
        tmem_wait_ld();
        uint8_t* line = stage + (c0 >> 6) * kABytes + r * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk = ((c0 & 63) >> 3) + q;
          *reinterpret_cast<uint4*>(line + ((chunk ^ (r & 7)) << 4)) =
              make_uint4(pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                         pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                         pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                         pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
        }
      }
      tc_fence_before();
      warp_arrive(&bars.acc_empty[b]);  // accumulator b has been read: the MMA may reuse it
      fence_proxy_async_smem();         // the TMA stores read the staged rows through the async proxy
      warp_arrive(&bars.stage_full);
      if (warp == 2) {
        if (!waitw(&bars.stage_full, u & 1, B_STAGE_FULL)) break;
        if (lane == 0) {
          for (int c = 0; c < kN / 64; ++c) tma_store_3d(&mo, n0 + 64 * c, h, t0, smem_u32(stage + c * kABytes));
          bulk_commit();
          bulk_wait_read_all();  // staging may be rewritten once the stores have read it
          stored = true;
          mbar_arrive(&bars.stage_free);
        }
        __syncwarp();
      }
    }
    if (warp == 2 && lane == 0 && stored) bulk_wait_all();
  }
  __syncwarp();

  // ---- teardown: on abort, let this thread's MMAs and TMA loads land first ----
  if (*abort_flag) {
    if (warp == 1 && lane == 0) {
      mma_commit(&bars.drain);
      mbar_drain(&bars.drain, 0);
    }
    mbar_drain(drain_bar, drain_par);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 2 * kN);
}

template <int kN, int kK, int kStages>
constexpr int bmm_smem() {
  return kStages * (kABytes + kN * 128) + (kN / 64) * kABytes + (int)sizeof(BmmBars) + 1024;
}

template <int kN, int kK, int kStages>
cudaError_t launch_bmm(const BmmParams& p, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo,
                       cudaStream_t stream) {
  constexpr int smem = bmm_smem<kN, kK, kStages>();
  static_assert(smem <= 232448, "shared memory over the sm_103a limit");
  static PerDeviceOnce attrs;
  cudaError_t e = attrs.run([] {
    return cudaFuncSetAttribute(absorb_bmm_kernel<kN, kK, kStages>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem);
  });
  if (e != cudaSuccess) return e;
  const int64_t items = (int64_t)((p.T + kRowsM - 1) / kRowsM) * p.H * (p.N / kN);
  int grid = device_sm_count();
  if (items < grid) grid = (int)items;
  if (grid < 1) grid = 1;
  absorb_bmm_kernel<kN, kK, kStages><<<grid, kBmmThreads, smem, stream>>>(p, ma, mb, mo);
  return cudaGetLastError();
}

}  // namespace

// q_lift: K = 128 (q_nope), N = 512 in slices of 256 columns; project_out: K = 512 (latent),
// N = 128.  One persistent CTA per SM.
cudaError_t launch_absorb_q(const BmmParams& p, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo,
                            cudaStream_t stream) {
  if (p.T <= 0) return cudaSuccess;
  return launch_bmm<256, 128, 3>(p, ma, mb, mo, stream);
}
cudaError_t launch_project_out(const BmmParams& p, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo,
                               cudaStream_t stream) {
  if (p.T <= 0) return cudaSuccess;
  return launch_bmm<128, 512, 6>(p, ma, mb, mo, stream);
}

}  // namespace mla
