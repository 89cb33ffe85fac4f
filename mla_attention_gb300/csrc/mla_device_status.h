// Codes written into the device status word (the first 4 bytes of a workspace).
#pragma once
#include <cstdint>

namespace mla {
enum : uint32_t {
  DEV_OK = 0,
  DEV_TIMEOUT_BASE = 0x1000,   // | wait-site id: a bounded wait ran out
  DEV_RANGE_BASE = 0x2000,     // | check-site id: an index was out of range
  DEV_GUARD_BASE = 0x3000,     // | guard-site id: guarded build only, an access left its buffer
};

// The first fault of a launch wins: later ones leave the word as it is.
__device__ __forceinline__ void record_error(uint32_t* err, uint32_t code) {
  if (err) atomicCAS(err, 0u, code);
}

// Guarded build (compiled with -DMLA_GUARD; the checks compile to nothing otherwise): every plain
// global load and store of the kernels first asks whether its bytes [ptr, ptr + n) lie inside
// the buffer they belong to, [base, base + bytes) with the extent the host derived from the call's
// sizes.  An access outside is skipped (a load gives zero) and recorded as DEV_GUARD_BASE | site
// in the status word (the first one stays).  TMA copies need no check: the hardware clips them
// to their tensor maps.
#ifdef MLA_GUARD
constexpr bool kGuarded = true;
#else
constexpr bool kGuarded = false;
#endif
__device__ __forceinline__ bool guard_span(uint32_t* err, uint32_t site, const void* ptr, uint32_t n,
                                           const void* base, uint64_t bytes) {
  if constexpr (!kGuarded) {
    return true;
  } else {
    const uint64_t a = reinterpret_cast<uint64_t>(ptr), b = reinterpret_cast<uint64_t>(base);
    const bool ok = base != nullptr && a >= b && a + n <= b + bytes;
    if (!ok) record_error(err, DEV_GUARD_BASE | site);
    return ok;
  }
}

// Sites of the guarded build's checks (the low bits of DEV_GUARD_BASE codes).
enum : uint32_t {
  G_BLOCK_TABLE = 1, G_LENS, G_TOPK, G_CACHE8, G_Q, G_Q_PE, G_OUT, G_PREV_OUT, G_LSE, G_PREV_LSE, G_TILE_PREFIX,
  G_PART_O, G_PART_LSE, G_C_KV, G_K_PE, G_SINKS, G_MERGE_IN, G_MERGE_OUT, G_ROPE_IN, G_ROPE_OUT, G_POS,
};
}  // namespace mla
