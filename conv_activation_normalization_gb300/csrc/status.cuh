// Device-side error bits.  Kernels never trap: a failed check sets a bit in
// the library's device status word (passed to every kernel as a pointer) and
// the kernel unwinds; gf_device_status() reads and clears the word.
#pragma once

#include <cstdint>

namespace gf {

enum : uint32_t {
  GF_DEV_WAIT_TIMEOUT = 1u,  // an mbarrier wait ran past its time limit
  GF_DEV_BAD_LAUNCH = 2u,    // a kernel was launched with a shape it cannot run
};

__device__ __forceinline__ void record_error(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

}  // namespace gf
