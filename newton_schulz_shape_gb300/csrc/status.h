// Device status-word bits written by the kernels (atomicOr) and read back by
// ns_check_status(). Host and device share this header.
#pragma once

#define NS_DEV_TIMEOUT 0x1u        // a bounded wait ran out; the kernel unwound
#define NS_DEV_BAD_INDEX 0x2u      // a kernel skipped an access outside its buffers
#define NS_DEV_BAD_LAUNCH 0x4u     // launch shape did not match the kernel's role layout
