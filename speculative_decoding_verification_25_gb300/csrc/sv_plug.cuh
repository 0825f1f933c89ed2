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

// Plug one row with one warp.  Lane i (i <= n) holds emitted token i in
// `tok`; n = accepted_len, so n + 1 <= SV_MAX_K + 1 <= 32 tokens.  An error
// row (n < 0) and a length outside [0, max_len] leave the row unchanged (the
// latter flags kDevBadLength); tokens past max_len are dropped and the
// length stops at max_len (kDevPlugClipped).  Every lane of the warp calls it.
__device__ __forceinline__ void plug_row(int lane, int n, int32_t tok, int32_t* seq_row,
                                         int32_t* seq_len_b, int max_len, int32_t* last_token_b,
                                         unsigned* flags) {
  if (n < 0) return;
  const int L = *seq_len_b;
  if (L < 0 || L > max_len) {
    if (lane == 0 && flags) atomicOr(flags, kDevBadLength);
    return;
  }
  if (lane <= n && L + lane < max_len) seq_row[L + lane] = tok;
  const int32_t last = __shfl_sync(0xffffffffu, tok, n);
  if (lane == 0) {
    const bool clipped = L + n + 1 > max_len;
    *seq_len_b = clipped ? max_len : L + n + 1;
    if (last_token_b) *last_token_b = last;
    if (clipped && flags) atomicOr(flags, kDevPlugClipped);
  }
}

// One warp per row.
__global__ void __launch_bounds__(256) sv_plug_kernel(PlugArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the verify step's outputs, before any access
  const int lane = threadIdx.x & 31;
  const long long b = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (b >= a.B) return;
  const int n = a.accepted_len[b];
  if (n > a.K) {   // not a length spec_verify writes: the row is left unchanged
    if (lane == 0 && a.flags) atomicOr(a.flags, kDevBadLength);
    return;
  }
  const int32_t tok = (n >= 0 && lane <= n) ? a.out_tokens[b * (a.K + 1) + lane] : -1;
  plug_row(lane, n, tok, a.tokens + b * a.max_len, a.seq_len + b, a.max_len,
           a.last_token ? a.last_token + b : nullptr, a.flags);
}

}  // namespace sv
