// Codes written into the device status word (the first 4 bytes of a workspace).
#pragma once
#include <cstdint>

namespace mla {
enum : uint32_t {
  DEV_OK = 0,
  DEV_TIMEOUT_BASE = 0x1000,   // | wait-site id: a bounded wait ran out
  DEV_RANGE_BASE = 0x2000,     // | check-site id: an index was out of range
};
}  // namespace mla
