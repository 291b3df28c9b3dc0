// Status codes and device-side error slots shared by the host library and the
// kernels (the public values are repeated in include/fattn.h).
#pragma once

namespace fattn {

enum Status : int {
  kOk = 0,
  kErrInvalidArg = -1,
  kErrUnsupported = -2,
  kErrMisaligned = -3,
  kErrTooLarge = -4,
  kErrLaunch = -5,
  kErrPipelineTimeout = -6,
  kErrCuda = -7,
};

// Device status block, one per device: word 0 holds the first error code a
// kernel raised (0 = none), word 1 where it was raised (role << 8 | barrier),
// word 2 the block index, word 3 is reserved.
constexpr int kStatusWords = 4;

// Roles and barrier ids recorded in status word 1.
enum Role : int { kRoleLoad = 1, kRoleMma = 2, kRoleSoftmax = 3, kRoleCorrection = 4 };
// (5 and 6 are the cache kernels' roles.)  The bounded-wait check kernel:
constexpr int kRoleWaitCheck = 7;

}  // namespace fattn
