// The absorption BMMs around the latent attention (TensorRT-LLM "mla.py",
// forward_absorption_generation): per head h,
//   q_lift[t, h, :] = q_nope[t, h, :] x k_b_proj_trans[h]^T   ([T, 128] x [128, 512]), written
//                     into the latent part of the fused query [T, H, 576];
//   out[t, h, :]    = O[t, h, :] x v_b_proj[h]^T              ([T, 512] x [512, 128]).
// Both are D[t, n] = sum_k A[t, k] B[n, k] with A rows of one head (strided in memory) and B
// the head's weight, K-major: one tcgen05 kernel serves both.
//
// One CTA per (128-token tile, head, kN-column slice of D): A and B stream through a ring of
// TMA stages (A: a 3-D box {64 columns, 1 head, 128 tokens} -> 128 rows x 128 B, SW128; B: a
// 2-D box of kN weight rows), one thread issues M128 x kN x K16 MMAs (both operands from
// shared memory) into a TMEM accumulator of kN columns, and the four warps read it back (one
// token row per thread) into bf16 rows staged in shared memory, which TMA stores write out.
// kN <= 256 columns of TMEM and a ring of at most ~100 KB keep two CTAs on an SM, so one CTA's
// epilogue overlaps the other's loads.
#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

constexpr int kRowsM = 128;              // tokens per tile
constexpr int kChunk = 64;               // K columns per stage (one 128-byte swizzled row)
constexpr int kABytes = kRowsM * 128;    // 16 KB

enum : uint32_t { B_FULL = 0x70, B_EMPTY, B_DONE };

struct BmmBars {
  uint64_t full[8], empty[8], done, drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
};

template <int kN, int kK, int kStages>
__global__ void __launch_bounds__(128, 2)
    absorb_bmm_kernel(const __grid_constant__ BmmParams p, const __grid_constant__ CUtensorMap ma,
                      const __grid_constant__ CUtensorMap mb, const __grid_constant__ CUtensorMap mo) {
  constexpr int kBBytes = kN * 128;
  constexpr int kStageBytes = kABytes + kBBytes;
  constexpr int kChunks = kK / kChunk;
  constexpr int kNmma = kN < 256 ? kN : 256;
  static_assert(kStages <= 8 && kN % kNmma == 0 && kK % kChunk == 0, "tile shape");
  extern __shared__ __align__(1024) uint8_t smem[];
  BmmBars& bars = *reinterpret_cast<BmmBars*>(smem + kStages * kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRowsM, h = blockIdx.y, n0 = blockIdx.z * kN;
  uint32_t* err = p.err;
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) record_error(err, DEV_RANGE_BASE | 0x7F);
    return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], 1);
    }
    mbar_init(&bars.done, 1);
    mbar_init(&bars.drain, 1);
    bars.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars.tmem_base, kN);
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
  uint64_t* drain_bar = nullptr;
  uint32_t drain_par = 0;

  if (warp == 0 && lane == 0) {
    // ---- TMA producer ----
    for (int c = 0; c < kChunks; ++c) {
      const int s = c % kStages;
      if (!wait1(&bars.empty[s], ((c / kStages) & 1) ^ 1, B_EMPTY)) break;
      const uint32_t st = smem_u32(smem + s * kStageBytes);
      mbar_arrive_expect_tx(&bars.full[s], kStageBytes);
      tma_load_3d(st, &ma, c * kChunk, h, t0, &bars.full[s]);
      for (int nb = 0; nb < kN / kNmma; ++nb)
        tma_load_2d(st + kABytes + nb * kNmma * 128, &mb, c * kChunk, h * p.N + n0 + nb * kNmma, &bars.full[s]);
      drain_bar = &bars.full[s];
      drain_par = (c / kStages) & 1;
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    const uint32_t idesc = idesc_bf16_f32(kRowsM, kNmma, false, false);
    bool live = true;
    for (int c = 0; c < kChunks && live; ++c) {
      const int s = c % kStages;
      if (!wait1(&bars.full[s], (c / kStages) & 1, B_FULL)) { live = false; break; }
      tc_fence_after();
      const uint32_t st = smem_u32(smem + s * kStageBytes);
#pragma unroll
      for (int k16 = 0; k16 < kChunk / 16; ++k16) {
        const uint64_t ad = sdesc_sw128(st + 32 * k16, 16, 1024);
#pragma unroll
        for (int nb = 0; nb < kN / kNmma; ++nb) {
          const uint64_t bd = sdesc_sw128(st + kABytes + nb * kNmma * 128 + 32 * k16, 16, 1024);
          mma_ss(tbase + nb * kNmma, ad, bd, idesc, (c | k16) != 0 ? 1u : 0u);
        }
      }
      mma_commit(&bars.empty[s]);
    }
    if (live) mma_commit(&bars.done);
  }
  __syncwarp();

  // ---- epilogue: token row (warp * 32 + lane) of the tile, kN columns -> bf16 rows staged in the
  // (now idle) ring as 64-column SW128 boxes, then TMA stores (rows past T are clipped) ----
  bool stored = false;
  if (wait1(&bars.done, 0, B_DONE)) {
    tc_fence_after();
    const int r = warp * 32 + lane;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
#pragma unroll 1
    for (int c0 = 0; c0 < kN; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(tbase + lane_base + c0, v);
      tmem_wait_ld();
      uint8_t* line = smem + (c0 >> 6) * kABytes + r * 128;
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
    fence_proxy_async_smem();  // the TMA stores read the staged rows through the async proxy
    stored = true;
  }
  __syncthreads();
  if (stored && threadIdx.x == 0) {
    for (int c = 0; c < kN / 64; ++c) tma_store_3d(&mo, n0 + 64 * c, h, t0, smem_u32(smem + c * kABytes));
    bulk_commit();
    bulk_wait_all();
  }

  // ---- teardown: on abort, let this thread's MMAs and TMA loads land first ----
  __syncwarp();
  if (*abort_flag) {
    if (warp == 1 && lane == 0) {
      mma_commit(&bars.drain);
      mbar_drain(&bars.drain, 0);
    }
    mbar_drain(drain_bar, drain_par);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, kN);
}

template <int kN, int kK, int kStages>
constexpr int bmm_smem() {
  return kStages * (kABytes + kN * 128) + (int)sizeof(BmmBars) + 1024;
}

template <int kN, int kK, int kStages>
cudaError_t launch_bmm(const BmmParams& p, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo,
                       cudaStream_t stream) {
  static_assert(kStages * (kABytes + kN * 128) >= (kN / 64) * kABytes, "the ring holds the staged output tile");
  constexpr int smem = bmm_smem<kN, kK, kStages>();
  static_assert(2 * smem <= 232448, "two CTAs per SM");
  static PerDeviceOnce attrs;
  cudaError_t e = attrs.run([] {
    return cudaFuncSetAttribute(absorb_bmm_kernel<kN, kK, kStages>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem);
  });
  if (e != cudaSuccess) return e;
  const dim3 grid((p.T + kRowsM - 1) / kRowsM, p.H, p.N / kN);
  absorb_bmm_kernel<kN, kK, kStages><<<grid, 128, smem, stream>>>(p, ma, mb, mo);
  return cudaGetLastError();
}

}  // namespace

// q_lift: K = 128 (q_nope), N = 512 in two CTAs of 256 columns; project_out: K = 512 (latent),
// N = 128.
cudaError_t launch_absorb_q(const BmmParams& p, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo,
                            cudaStream_t stream) {
  if (p.T <= 0) return cudaSuccess;
  return launch_bmm<256, 128, 2>(p, ma, mb, mo, stream);
}
cudaError_t launch_project_out(const BmmParams& p, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo,
                               cudaStream_t stream) {
  if (p.T <= 0) return cudaSuccess;
  return launch_bmm<128, 512, 3>(p, ma, mb, mo, stream);
}

}  // namespace mla
