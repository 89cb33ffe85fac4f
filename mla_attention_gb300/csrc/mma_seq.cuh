// Fixed sequences of tcgen05.mma (kind::f16, bf16 in, fp32 accumulate) issued
// from one asm block each.  One thread issues every MMA of a tile; with the
// descriptors advanced by plain adds inside the block the tensor core receives
// instructions as fast as it executes them, whereas rebuilding descriptors in
// a C++ loop limited issue to about one instruction per 130 cycles.
//
// Shared-memory descriptor low bits hold (address >> 4): +2 moves 32 bytes (one
// K16 step inside a 128-byte swizzled row); a 64-column box of R rows spans
// R * 128 / 16 = 8 * R units.  A tensor-memory A operand advances 8 columns
// (16 bf16) per K16 step.
#pragma once
#include <cstdint>

namespace mla {

#define MLA_TS(P, BINC) \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, " P ";\n\tadd.u32 at, at, 8;\n\tadd.s64 bd, bd, " #BINC ";\n\t"
// four K16 steps inside one 64-column box of 64 rows, then on to the next box (64 rows: 512 units)
#define MLA_TS_BOX64(P0) MLA_TS(P0, 2) MLA_TS("pt", 2) MLA_TS("pt", 2) MLA_TS("pt", 506)

// S[128 x 64] = Q[128 x 576] (TMEM, 288 columns from a_tmem) * K^T, K = 9 boxes [64 rows x 64 cols].
__device__ __forceinline__ void mma_s_q576_n64(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b64 bd;\n\t.reg .b32 at;\n\t"
      "setp.ne.u32 pf, %3, %3;\n\tsetp.eq.u32 pt, %3, %3;\n\t"
      "mov.b64 bd, %2;\n\tmov.b32 at, %1;\n\t"
      MLA_TS_BOX64("pf") MLA_TS_BOX64("pt") MLA_TS_BOX64("pt") MLA_TS_BOX64("pt") MLA_TS_BOX64("pt")
      MLA_TS_BOX64("pt") MLA_TS_BOX64("pt") MLA_TS_BOX64("pt") MLA_TS_BOX64("pt")
      "}" ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc)
      : "memory");
}

// ---- 128-key score tiles: M128 N128, K streamed in groups of three 64-column boxes of
// 128 rows (16 KB each, 1024 units) ----
#define MLA_TS128(P, BINC) \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, " P ";\n\tadd.u32 at, at, 8;\n\tadd.s64 bd, bd, " #BINC ";\n\t"
#define MLA_TS128_BOX(P0) MLA_TS128(P0, 2) MLA_TS128("pt", 2) MLA_TS128("pt", 2) MLA_TS128("pt", 1018)
#define MLA_SS128(P) \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, " P ";\n\tadd.s64 ad, ad, 2;\n\tadd.s64 bd, bd, 2;\n\t"

// S[128 x 128] (+)= Q[:, three latent boxes] (TMEM, 96 columns from a_tmem) * K_group^T.
// accumulate = 0 overwrites S (the first group of a tile).
__device__ __forceinline__ void mma_s_grp3_n128(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pa, pt;\n\t.reg .b64 bd;\n\t.reg .b32 at;\n\t"
      "setp.ne.u32 pa, %4, 0;\n\tsetp.eq.u32 pt, %3, %3;\n\tmov.b64 bd, %2;\n\tmov.b32 at, %1;\n\t"
      MLA_TS128_BOX("pa") MLA_TS128_BOX("pt") MLA_TS128_BOX("pt")
      "}" ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// S[128 x 128] += Q[:, two latent boxes] (TMEM) * K_group[boxes 0, 1]^T + Q_rope (smem, 128 x 64)
// * K_group[box 2]^T.
__device__ __forceinline__ void mma_s_grp2r_n128(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                 uint64_t a_rope_desc, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred pt;\n\t.reg .b64 bd, ad;\n\t.reg .b32 at;\n\t"
      "setp.eq.u32 pt, %3, %3;\n\tmov.b64 bd, %2;\n\tmov.b32 at, %1;\n\tmov.b64 ad, %4;\n\t"
      MLA_TS128_BOX("pt") MLA_TS128_BOX("pt")
      MLA_SS128("pt") MLA_SS128("pt") MLA_SS128("pt") MLA_SS128("pt")
      "}" ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "l"(a_rope_desc)
      : "memory");
}

// S[128 x 128] = Q * K^T for a whole 128-key tile whose three K groups (boxes 0-2, 3-5,
// 6-8 of 128 rows, contiguous in smem) have all landed: 32 TS MMAs over the latent boxes
// and 4 SS MMAs over the RoPE box, with the group release commits in between.
__device__ __forceinline__ void mma_s_tile_n128(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint64_t a_rope_desc, uint32_t idesc, uint32_t empty0,
                                                uint32_t empty1, uint32_t empty2) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b64 bd, ad;\n\t.reg .b32 at;\n\t"
      "setp.ne.u32 pf, %3, %3;\n\tsetp.eq.u32 pt, %3, %3;\n\tmov.b64 bd, %2;\n\tmov.b32 at, %1;\n\tmov.b64 ad, %4;\n\t"
      MLA_TS128_BOX("pf") MLA_TS128_BOX("pt") MLA_TS128_BOX("pt")
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t"
      MLA_TS128_BOX("pt") MLA_TS128_BOX("pt") MLA_TS128_BOX("pt")
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t"
      MLA_TS128_BOX("pt") MLA_TS128_BOX("pt")
      MLA_SS128("pt") MLA_SS128("pt") MLA_SS128("pt") MLA_SS128("pt")
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%7];\n\t"
      "}" ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "l"(a_rope_desc), "r"(empty0), "r"(empty1),
      "r"(empty2)
      : "memory");
}

#define MLA_PV256(ACC) \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd0, %4, " ACC ";\n\t" \
  "tcgen05.mma.cta_group::1.kind::f16 [%1], ad, bd1, %4, " ACC ";\n\t" \
  "add.s64 ad, ad, 2;\n\tadd.s64 bd0, bd0, 128;\n\tadd.s64 bd1, bd1, 128;\n\t"

// O[128 x 512] (+)= P[128 x 64] (smem, K-major) * V[64 x 512] (smem, MN-major, two N=256 halves).
// K16 step: P +32 bytes, V +16 rows (2048 bytes).  accumulate = 0 overwrites O.
__device__ __forceinline__ void mma_pv_k64_n512(uint32_t d0, uint32_t d1, uint64_t a_desc, uint64_t b_desc0,
                                                uint64_t b_desc1, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pa, pt;\n\t.reg .b64 ad, bd0, bd1;\n\t"
      "setp.ne.u32 pa, %5, 0;\n\tsetp.eq.u32 pt, %4, %4;\n\t"
      "mov.b64 ad, %2;\n\tmov.b64 bd0, %3;\n\tmov.b64 bd1, %6;\n\t"
      MLA_PV256("pa") MLA_PV256("pt") MLA_PV256("pt") MLA_PV256("pt")
      "}" ::"r"(d0), "r"(d1), "l"(a_desc), "l"(b_desc0), "r"(idesc), "r"(accumulate), "l"(b_desc1)
      : "memory");
}

#define MLA_SS(P, INC) \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, " P ";\n\tadd.s64 ad, ad, " #INC ";\n\tadd.s64 bd, bd, " #INC ";\n\t"
// four K16 steps in a box of 128 rows, then the next box (128 rows: 1024 units)
#define MLA_SS_BOX128(P0) MLA_SS(P0, 2) MLA_SS("pt", 2) MLA_SS("pt", 2) MLA_SS("pt", 1018)

// S[128 x 128] = Q[128 x 192] * K[128 x 192]^T, both 3 boxes [128 rows x 64 cols] in smem.
__device__ __forceinline__ void mma_s_k192_n128(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b64 ad, bd;\n\t"
      "setp.ne.u32 pf, %3, %3;\n\tsetp.eq.u32 pt, %3, %3;\n\t"
      "mov.b64 ad, %1;\n\tmov.b64 bd, %2;\n\t"
      MLA_SS_BOX128("pf") MLA_SS_BOX128("pt") MLA_SS_BOX128("pt")
      "}" ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc)
      : "memory");
}

#define MLA_TSV(P) \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, " P ";\n\tadd.u32 at, at, 8;\n\tadd.s64 bd, bd, 128;\n\t"

// O[128 x 128] (+)= P[128 x 128] (TMEM, 64 columns from a_tmem) * V[128 x 128] (smem, MN-major).
__device__ __forceinline__ void mma_pv_tmem_k128_n128(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                      uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pa, pt;\n\t.reg .b64 bd;\n\t.reg .b32 at;\n\t"
      "setp.ne.u32 pa, %4, 0;\n\tsetp.eq.u32 pt, %3, %3;\n\t"
      "mov.b64 bd, %2;\n\tmov.b32 at, %1;\n\t"
      MLA_TSV("pa") MLA_TSV("pt") MLA_TSV("pt") MLA_TSV("pt") MLA_TSV("pt") MLA_TSV("pt") MLA_TSV("pt") MLA_TSV("pt")
      "}" ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

#undef MLA_TS
#undef MLA_TS_BOX64
#undef MLA_PV256
#undef MLA_SS
#undef MLA_SS_BOX128
#undef MLA_TSV
#undef MLA_TS128
#undef MLA_TS128_BOX
#undef MLA_SS128

}  // namespace mla
