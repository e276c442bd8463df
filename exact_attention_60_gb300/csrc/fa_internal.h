// fa_internal.h -- links between the forward (fa_fwd.cu) and backward (fa_bwd.cu)
// translation units of libfa.so.  Not part of the C ABI.
#pragma once

#include <stddef.h>

#include <algorithm>
#include <utility>

// Read and clear the backward kernels' device status word (0 or an fa_status code in
// bits 0..7 and a wait site in bits 8..15); FA_ERR_CUDA if it cannot be read.
unsigned fa_bwd_take_device_status();

// The wait limit set with fa_debug_set (0 = the default of one second).
unsigned long long fa_internal_wait_limit_ns();

// The test-hook flags set with fa_debug_set.
unsigned fa_internal_debug_flags();

// Checks of strided [B,H,L,D] layouts (element strides {batch, head, row}, features
// contiguous), shared by the forward and backward entry points.
namespace fa_layout {

// Byte span [lo, lo + bytes) that a [B,H,L,D] tensor with element strides st touches.
inline size_t span_bytes(long long B, long long H, long long L, int D, const long long* st) {
  const long long last = (B - 1) * st[0] + (H - 1) * st[1] + (L - 1) * st[2] + D;
  return static_cast<size_t>(last) * 2;
}

// Strides of one tensor: non-negative multiples of 8 elements (16 bytes, the tensor-memory-
// access unit's rule) for every dimension of size > 1, and byte offsets below 2^40.
inline bool strides_ok(long long B, long long H, long long L, int D, const long long* st) {
  const long long size[3] = {B, H, L};
  for (int i = 0; i < 3; ++i) {
    if (size[i] <= 1) continue;
    if (st[i] < 0 || (st[i] & 7) || st[i] >= (1ll << 39)) return false;
  }
  return span_bytes(B, H, L, D, st) < (1ull << 40);
}

// No two elements of the tensor share an address: with the dimensions of size > 1 ordered
// by stride (features innermost, stride 1, extent D), each stride covers the extent of the
// dimension inside it.
inline bool no_self_overlap(long long B, long long H, long long L, int D, const long long* st) {
  std::pair<long long, long long> dims[4] = {{1, D}};   // (stride, extent)
  int n = 1;
  const long long size[3] = {B, H, L};
  for (int i = 0; i < 3; ++i)
    if (size[i] > 1) dims[n++] = {st[i], size[i]};
  std::sort(dims, dims + n);
  for (int i = 1; i < n; ++i)
    if (dims[i].first < dims[i - 1].first * dims[i - 1].second) return false;
  return true;
}

}  // namespace fa_layout
