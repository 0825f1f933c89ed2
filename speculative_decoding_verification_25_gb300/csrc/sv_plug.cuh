// The plug step: append each row's emitted tokens to its sequence buffer and
// advance its length on the device, so the next decode step can be launched
// without reading the accepted lengths back to the host (the page
// "Accelerating Sonar through speculation", single-token MTP schedule: once
// the target's input tokens are shifted, a kernel plugs the next target
// tokens into their places).
#pragma once

#include <stdint.h>

namespace sv {

constexpr unsigned kDevPlugClipped = 16u;
constexpr unsigned kDevBadLength = 32u;

struct PlugArgs {
  const int32_t* accepted_len;   // [B]
  const int32_t* out_tokens;     // [B, K+1]
  int B, K, max_len;
  int32_t* tokens;               // [B, max_len]
  int32_t* seq_len;              // [B]
  int32_t* last_token;           // [B] or nullptr
  unsigned* flags;               // or nullptr
};

// One warp per row: lane i writes emitted token i at position L + i.
__global__ void __launch_bounds__(256) sv_plug_kernel(PlugArgs a) {
  const int lane = threadIdx.x & 31;
  const long long b = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (b >= a.B) return;
  const int n = a.accepted_len[b];
  if (n < 0) return;   // error row
  const int L = a.seq_len[b];
  if (L < 0 || L > a.max_len) {
    if (lane == 0 && a.flags) atomicOr(a.flags, kDevBadLength);
    return;
  }
  const int32_t* src = a.out_tokens + b * (a.K + 1);
  int32_t* dst = a.tokens + b * a.max_len;
  for (int i = lane; i <= n; i += 32)
    if (L + i < a.max_len) dst[L + i] = src[i];
  if (lane == 0) {
    const bool clipped = L + n + 1 > a.max_len;
    a.seq_len[b] = clipped ? a.max_len : L + n + 1;
    if (a.last_token) a.last_token[b] = src[n];
    if (clipped && a.flags) atomicOr(a.flags, kDevPlugClipped);
  }
}

}  // namespace sv
