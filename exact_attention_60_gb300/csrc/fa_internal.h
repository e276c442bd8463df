// fa_internal.h -- links between the forward (fa_fwd.cu) and backward (fa_bwd.cu)
// translation units of libfa.so.  Not part of the C ABI.
#pragma once

// Read and clear the backward kernels' device status word (0 or an fa_status code in
// bits 0..7 and a wait site in bits 8..15); FA_ERR_CUDA if it cannot be read.
unsigned fa_bwd_take_device_status();

// The wait limit set with fa_debug_set (0 = the default of one second).
unsigned long long fa_internal_wait_limit_ns();

// The test-hook flags set with fa_debug_set.
unsigned fa_internal_debug_flags();
