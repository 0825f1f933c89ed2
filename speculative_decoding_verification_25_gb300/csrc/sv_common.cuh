// Device helpers shared by the two spec_verify kernels: 16-byte streaming
// loads, bf16 unpacking, warp reductions, and unevaluated float32 pairs
// ("double-float": value = hi + lo) used where float32 alone is not accurate
// enough for the sampling step.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "exp2_table.inc"

namespace sv {

#define SV_NEG_INF (-__int_as_float(0x7f800000))
constexpr float kFltMin = 1.17549435e-38f;

// The checked build (compiled with -DSV_CHECKED): every global index the
// verify kernel forms is tested against its buffer's extent before the
// access; a failed test skips the access and sets kDevOutOfBounds in the
// device flags instead of faulting.  The plain build compiles the tests
// away.
#ifdef SV_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif
constexpr unsigned kDevOutOfBounds = 256u;

// ----------------------------------------------------------------- element types
// A "vector" is 16 bytes of one logit row held as four 32-bit words:
// 8 bf16 (two per word, element 2i in the low half) or 4 float32.
struct Bf16 {
  static constexpr int kVec = 8;
  static constexpr int kBytes = 2;
  // -inf in both halves: the fill value of masked elements
  static constexpr uint32_t kFillWord = 0xff80ff80u;
  __device__ __forceinline__ static float elem(const uint32_t (&w)[4], int k) {
    const uint32_t word = (k & 4) ? ((k & 2) ? w[3] : w[2]) : ((k & 2) ? w[1] : w[0]);
    return __uint_as_float((k & 1) ? (word & 0xffff0000u) : (word << 16));
  }
  __device__ __forceinline__ static float load_scalar(const void* base, long long i) {
    unsigned short h;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(h) : "l"((const unsigned short*)base + i));
    return __uint_as_float(((uint32_t)h) << 16);
  }
  // a float32 value cut to a bf16 one (toward zero)
  __device__ __forceinline__ static float round_logit(float v) {
    return __uint_as_float(__float_as_uint(v) & 0xffff0000u);
  }
};

struct F32 {
  static constexpr int kVec = 4;
  static constexpr int kBytes = 4;
  static constexpr uint32_t kFillWord = 0xff800000u;
  __device__ __forceinline__ static float elem(const uint32_t (&w)[4], int k) {
    return __uint_as_float((k & 2) ? ((k & 1) ? w[3] : w[2]) : ((k & 1) ? w[1] : w[0]));
  }
  __device__ __forceinline__ static float load_scalar(const void* base, long long i) {
    float f;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(f) : "l"((const float*)base + i));
    return f;
  }
  __device__ __forceinline__ static float round_logit(float v) { return v; }
};

// 16-byte read-only streaming load that does not allocate in L1.
__device__ __forceinline__ void ldg_stream16(const void* p, uint32_t (&w)[4]) {
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "l"(p));
}

// Load vector `v` (elements v*kVec .. v*kVec+kVec-1) of a row of V elements.
// kAligned: the row base is 16-byte aligned and V*kBytes % 16 == 0, so every
// in-range vector is full and one 16-byte load fetches it.  Otherwise the
// elements are fetched one by one.  Elements at or beyond V read as -inf.
template <typename E, bool kAligned>
__device__ __forceinline__ void load_vec(const void* row, long long v, int V, uint32_t (&w)[4]) {
  const long long e0 = v * E::kVec;
  if (kAligned) {
    if (e0 < V) {
      ldg_stream16((const char*)row + e0 * E::kBytes, w);
    } else {
      w[0] = w[1] = w[2] = w[3] = E::kFillWord;
    }
  } else {
    if constexpr (E::kBytes == 2) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const long long e = e0 + 2 * i;
        const float a = (e < V) ? E::load_scalar(row, e) : SV_NEG_INF;
        const float b = (e + 1 < V) ? E::load_scalar(row, e + 1) : SV_NEG_INF;
        w[i] = (__float_as_uint(a) >> 16) | (__float_as_uint(b) & 0xffff0000u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const long long e = e0 + i;
        w[i] = __float_as_uint((e < V) ? E::load_scalar(row, e) : SV_NEG_INF);
      }
    }
  }
}

// ----------------------------------------------------------------- packed float32 pairs
// Two float32 lanes in one 64-bit register (add and fma .f32x2 on sm_100+).
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// max of two packed bf16 pairs
__device__ __forceinline__ uint32_t bf2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Wait until the preceding kernel on the stream has completed and its
// writes are visible.  A kernel launched as a programmatic dependent may
// start while that kernel's last CTAs drain; one launched without the
// attribute returns from this at once.
__device__ __forceinline__ void wait_for_preceding_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Let the next kernel on the stream (launched as a programmatic dependent)
// be scheduled as this grid's CTAs exit, instead of after the last one: its
// CTAs take the freed slots and run up to their own griddepcontrol.wait,
// which still returns only once this grid has completed.
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ----------------------------------------------------------------- warp reductions
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_min_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ----------------------------------------------------------------- double-float
// Error-free transformations (Knuth two-sum, Dekker fast-two-sum, FMA-based
// two-product).  The explicit _rn intrinsics keep the compiler from fusing
// or reassociating them.
struct DF {
  float hi, lo;
};

__device__ __forceinline__ DF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}
// requires |a| >= |b| (or a == 0)
__device__ __forceinline__ DF fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ DF df_add(DF x, DF y) {
  const DF s = two_sum(x.hi, y.hi);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo)));
}
__device__ __forceinline__ DF df_add_f(DF x, float y) {
  const DF s = two_sum(x.hi, y);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, x.lo));
}
__device__ __forceinline__ DF df_neg(DF x) { return {-x.hi, -x.lo}; }
__device__ __forceinline__ DF df_sub(DF x, DF y) { return df_add(x, df_neg(y)); }
__device__ __forceinline__ DF df_mul_f(DF a, float b) {
  const float p = __fmul_rn(a.hi, b);
  float e = __fmaf_rn(a.hi, b, -p);
  e = __fmaf_rn(a.lo, b, e);
  return fast_two_sum(p, e);
}
__device__ __forceinline__ DF df_mul(DF a, DF b) {
  const float p = __fmul_rn(a.hi, b.hi);
  float e = __fmaf_rn(a.hi, b.hi, -p);
  e = __fmaf_rn(a.hi, b.lo, e);
  e = __fmaf_rn(a.lo, b.hi, e);
  return fast_two_sum(p, e);
}
// a / b for b > 0: one correction step on the float32 quotient
__device__ __forceinline__ DF df_div(DF a, DF b) {
  const float q1 = __fdiv_rn(a.hi, b.hi);
  const DF r = df_sub(a, df_mul_f(b, q1));
  const float q2 = __fdiv_rn(r.hi, b.hi);
  return fast_two_sum(q1, q2);
}
// sign of x (x normalised: |lo| <= ulp(hi)/2, so hi carries the sign unless x == 0)
__device__ __forceinline__ bool df_pos(DF x) { return x.hi > 0.f || (x.hi == 0.f && x.lo > 0.f); }
__device__ __forceinline__ bool df_lt(DF x, DF y) { return df_pos(df_sub(y, x)); }

__device__ __forceinline__ DF df_shfl_xor(DF v, int o) {
  return {__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ DF df_shfl_up(DF v, int o) {
  return {__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ DF warp_sum_df(DF v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = df_add(v, df_shfl_xor(v, o));
  return v;
}
// Warp sums of four double-floats at once: after the call lanes 0-7 hold
// the sum of v0, lanes 8-15 of v1, 16-23 of v2, 24-31 of v3.  Every lane
// exchanges and adds only what its half (then quarter) of the warp keeps.
__device__ __forceinline__ DF warp_sum4_df(DF v0, DF v1, DF v2, DF v3) {
  const int lane = threadIdx.x & 31;
  const bool hi16 = (lane & 16) != 0, hi8 = (lane & 8) != 0;
  DF a0 = hi16 ? v2 : v0, a1 = hi16 ? v3 : v1;   // kept
  const DF b0 = hi16 ? v0 : v2, b1 = hi16 ? v1 : v3;   // given to lane ^ 16
  a0 = df_add(a0, df_shfl_xor(b0, 16));
  a1 = df_add(a1, df_shfl_xor(b1, 16));
  DF c = hi8 ? a1 : a0;
  const DF d = hi8 ? a0 : a1;   // given to lane ^ 8
  c = df_add(c, df_shfl_xor(d, 8));
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) c = df_add(c, df_shfl_xor(c, o));
  return c;
}

// log2(e) / T as a double-float: the float32 quotient plus the correctly
// signed remainder divided by T.
__device__ __forceinline__ DF log2e_over(float T) {
  const float h = __fdiv_rn(kLog2eHi, T);
  const float r = __fmaf_rn(-h, T, kLog2eHi);          // exact remainder
  const float l = __fdiv_rn(__fadd_rn(r, kLog2eLo), T);
  return fast_two_sum(h, l);
}

// 2^(yh + yl) to ~1e-13 relative, for yh in [-126, 0]; the caller guarantees
// yl is tiny against yh.  Method: y = n/256 + f with |f| <= 1/512 (exact
// split), 2^(n/256) = 2^floor(n/256) * tab[n mod 256] from the double-float
// table, and 2^f = e^g with g = f ln 2 by its Taylor series to g^5 (|g| <
// 1.4e-3, so the first omitted term is below 1e-20).
__device__ __forceinline__ DF exp2_df(float yh, float yl, const float2* tab) {
  if (!(yh > -126.f)) return DF{0.f, 0.f};   // underflow, -inf and NaN
  const float n = rintf(__fmul_rn(yh, 256.f));
  const float f = __fsub_rn(yh, __fmul_rn(n, 1.f / 256.f));  // exact
  const DF s = two_sum(f, yl);
  const float gh = __fmul_rn(s.hi, kLn2Hi);
  float gl = __fmaf_rn(s.hi, kLn2Hi, -gh);
  gl = __fmaf_rn(s.hi, kLn2Lo, gl);
  gl = __fmaf_rn(s.lo, kLn2Hi, gl);
  const float tail =
      gh * gh * (0.5f + gh * (1.f / 6.f + gh * (1.f / 24.f + gh * (1.f / 120.f))));
  DF e = fast_two_sum(1.f, gh);
  e = fast_two_sum(e.hi, __fadd_rn(e.lo, __fadd_rn(gl, tail)));
  const int ni = (int)n;
  const int k = ni >> 8;             // floor(n / 256)
  const float2 t = tab[ni & 255];
  const DF r = df_mul(e, DF{t.x, t.y});
  const float scale = __int_as_float((k + 127) << 23);
  return DF{r.hi * scale, r.lo * scale};
}

// e^((x - m) / T) = 2^((x - m) * L) with L = log2(e)/T as a double-float;
// (x - m) is formed exactly with two-sum.
__device__ __forceinline__ DF exp_df(float x, float m, DF L, const float2* tab) {
  const DF d = two_sum(x, -m);
  const float yh = __fmul_rn(d.hi, L.hi);
  float yl = __fmaf_rn(d.hi, L.hi, -yh);
  yl = __fmaf_rn(d.hi, L.lo, yl);
  yl = __fmaf_rn(d.lo, L.hi, yl);
  const DF y = fast_two_sum(yh, yl);
  return exp2_df(y.hi, y.lo, tab);
}

__device__ __forceinline__ bool valid_temperature(float T) {
  // 0 (greedy) or a finite value >= FLT_MIN; NaN fails every comparison
  return T == 0.f || (T >= kFltMin && T <= 3.4028235e38f);
}

}  // namespace sv
