// Device helpers shared by the layer's kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8moe {

// Bits of the context's device error flag.
enum : int {
  DEV_ERR_TIMEOUT = 1,    // a bounded wait gave up
  DEV_ERR_NONFINITE = 2,  // a router logit was NaN or infinite
  DEV_ERR_BOUNDS = 4,     // an index failed a consistency check
};

__device__ __forceinline__ void set_error(int *flag, int bit) { atomicOr(flag, bit); }

// Programmatic dependent launch: wait until the preceding kernel of the
// stream has completed and its writes are visible (a no-op when the kernel
// was launched without the programmatic-serialization attribute), and let
// the next kernel of the stream start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// 16-byte global load that bypasses L1 (weights are streamed once).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 16-byte read-only global load through L1 (activations, reused).
__device__ __forceinline__ uint4 ld_ro16(const void *p) {
  return __ldg(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ uint32_t u4_word(const uint4 &v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Two e4m3 codes (low byte first) -> f16x2 (low half first).  Exact: every
// e4m3 value is an f16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_bytes & 0xffffu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t v) {
  __half2 h = *reinterpret_cast<__half2 *>(&v);
  return __half22float2(h);
}

// D = A(16x16, f16, row) * B(16x8, f16, col) + D, f32 accumulate.
__device__ __forceinline__ void mma_16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// silu(z) * u with silu(z) = z / (1 + e^-z).  The fast division (about two
// ulps) stays far below the precision at which h is kept, and has no slow
// path for large or non-finite operands.
__device__ __forceinline__ float swiglu(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

// Exact power of two 2^e for |e| < 127.
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// v * 2^e as two multiplications by representable powers of two (|e| <= 252):
// exact whenever the result is a normal float, without a per-value ldexpf.
struct Pow2 {
  float f1, f2;
  __device__ __forceinline__ float operator()(float v) const { return v * f1 * f2; }
};
__device__ __forceinline__ Pow2 pow2_factors(int e) {
  const int a = e / 2;
  return Pow2{exp2i(a), exp2i(e - a)};
}

// Power-of-two exponent that brings a non-negative magnitude m to at most
// 2^14 (the f16 conversion range used by the tensor-core GEMV); 0 if it
// already fits.  Scaling by 2^-e is exact.
__device__ __forceinline__ int f16_range_shift(float m) {
  if (!(m > 16384.0f)) return 0;
  int e;
  frexpf(m, &e);     // m in [2^(e-1), 2^e)
  int s = e - 14;    // m * 2^-s < 2^14
  return s > 120 ? 120 : s;
}

}  // namespace fp8moe

namespace fp8moe {

// Exponent e of the power-of-two block scale 2^e for a block whose largest
// magnitude is amax: the smallest e with amax / 2^e <= 448 (the largest e4m3
// value), so scaling is exact and the block's values land in [-448, 448].
// 0 for an all-zero block.
__device__ __forceinline__ int e4m3_block_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  int q;
  const float m = frexpf(amax / 448.f, &q);  // amax / 448 = m 2^q, m in [0.5, 1)
  return m > 0.5f ? q : q - 1;
}

// Multi-term e4m3 encoding of values already divided by their power-of-two
// block scale (|v| <= 448): v ~= t0 + t1 + ... with t0 = e4m3(v),
// t1 = e4m3(v - t0), ..., each rounded to nearest even and saturated
// (cvt.rn.satfinite).  Each term carries 4 significant bits, so two terms
// hold a bf16 value exactly (down to 2^-10 of the block scale) and three
// terms keep about 12 bits of an f32 value.  Codes of (v0, v1), first value
// in the low byte, one 16-bit pair per term.
template <int NT>
__device__ __forceinline__ void e4m3_terms(float v0, float v1, uint32_t (&codes)[NT]) {
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(make_float2(v0, v1), __NV_SATFINITE, __NV_E4M3);
    codes[t] = c;
    if (t + 1 < NT) {
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(c, __NV_E4M3);
      const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
      v0 -= f.x;
      v1 -= f.y;
    }
  }
}

}  // namespace fp8moe
