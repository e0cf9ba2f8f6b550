// Bits of the library's device status word (see fa_get_device_status).
#pragma once

namespace fa {
constexpr unsigned kStatusTimeoutBit = 1u << 0;   // a bounded pipeline wait gave up
constexpr unsigned kStatusBadTableBit = 1u << 1;  // a block-table entry was out of range
constexpr unsigned kStatusLaunchBit = 1u << 2;    // a kernel could not set up its shared memory
constexpr unsigned kStatusBadArgBit = 1u << 3;    // device-side argument check failed (e.g. max_seqlen too small)
constexpr unsigned kStatusBoundsBit = 1u << 4;    // FA_DEBUG builds: an index outside its buffer (access skipped)
}  // namespace fa
