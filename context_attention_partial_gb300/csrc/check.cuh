// check.cuh -- optional device-side bounds checks.
//
// A build with -DCPATTN_CHECK (libcpattn_check.so, a debugging aid) tests
// every global store and load of the kernels against the extent of the
// buffer the host described, in bytes from the buffer's base pointer.  An
// access outside it is skipped and kErrBounds is ORed into the device error
// word, so the caller sees CPATTN_ERR_BOUNDS from cpattn_last_device_status;
// nothing traps.  Normal builds compile every check to `true`: the kernels
// are unchanged.
#pragma once
#include <cstdint>

namespace cpattn {

constexpr unsigned kErrBounds = 0x100u;

// Extent of one buffer for the checks: base pointer and byte count.
struct Span {
  const void* base;
  uint64_t bytes;
};

#ifdef CPATTN_CHECK
__device__ __forceinline__ bool in_span(const Span& s, const void* p, unsigned bytes,
                                        unsigned int* err) {
  // (an address below the base wraps to a huge offset)
  const uint64_t off = static_cast<uint64_t>(static_cast<const char*>(p) -
                                             static_cast<const char*>(s.base));
  if (off <= s.bytes && bytes <= s.bytes - off) return true;
  atomicOr(err, kErrBounds);
  return false;
}
#define CPATTN_IN(span, ptr, bytes, err) ::cpattn::in_span((span), (ptr), (bytes), (err))
#else
#define CPATTN_IN(span, ptr, bytes, err) true
#endif

}  // namespace cpattn
