// Device helpers shared by the layer's kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// ---------------------------------------------------------------- packed conversions
// Four bytes, each holding two e2m1 codes (low nibble = lower column), to four
// f16x2 registers (low half = lower column).  Exact: every e2m1 value is an f16.
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Four bytes, each an e2m3 code in its low 6 bits, to two f16x2 registers
// (byte 0 -> low half of h[0], byte 1 -> high half of h[0], ...).  Exact.
__device__ __forceinline__ void e2m3x4_to_f16x4(uint32_t w, uint32_t (&h)[2]) {
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e2m3x2 %0, lo;\n\t"
      "cvt.rn.f16x2.e2m3x2 %1, hi;\n\t}"
      : "=r"(h[0]), "=r"(h[1])
      : "r"(w));
}

// Two e4m3 bytes (low 16 bits of v) to f16x2 (byte 0 -> low half).  Exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  uint32_t h;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
      : "=r"(h)
      : "r"(v));
  return h;
}

// fp32 >= 0 to an e4m3 byte, round to nearest even, saturating at 448 (both
// halves of the packed result hold the same byte, so its order does not matter).
__device__ __forceinline__ uint32_t f32_to_e4m3_satfinite(float v) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 t, %1, %1;\n\t"
      "cvt.u32.u16 %0, t;\n\t}"
      : "=r"(r)
      : "f"(v));
  return r & 0xFFu;
}

// Status word values the kernels record (the negative moe_status codes).
constexpr int kStatusInvalid = -1;  // MOE_EINVAL: a bad expert id or work entry
constexpr int kStatusTimeout = -5;  // MOE_ETIMEOUT: a bounded wait gave up
constexpr int kStatusRange = -6;    // MOE_ERANGE: a value outside f16's finite range

// True when an f16 (either half of an f16x2 word) is infinite or NaN.
__device__ __forceinline__ bool f16_nonfinite(uint32_t h) { return (h & 0x7C00u) == 0x7C00u; }
__device__ __forceinline__ bool f16x2_nonfinite(uint32_t h) {
  return f16_nonfinite(h) || f16_nonfinite(h >> 16);
}

// The SwiGLU output a as f16 bits (round to nearest even).  The f16 copy is
// exact to 11 bits for |a| in [2^-14, 65504]; larger values (and non-finite
// ones) record MOE_ERANGE in the status word.
__device__ __forceinline__ uint16_t a_to_f16(float a, int* status) {
  const uint16_t h = __half_as_ushort(__float2half_rn(a));
  if (f16_nonfinite(h)) *status = kStatusRange;
  return h;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// f16x2 with both halves equal to the low (or high) half of v
__device__ __forceinline__ uint32_t dup_lo(uint32_t v) { return (v & 0xFFFFu) | (v << 16); }
__device__ __forceinline__ uint32_t dup_hi(uint32_t v) { return (v >> 16) | (v & 0xFFFF0000u); }

// ---------------------------------------------------------------- tensor-core MMA (register operands)
// D = A * B + D, m16n8k16, A row-major f16, B col-major f16, fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- memory
// Streaming loads of data that no kernel writes while it runs (packed weights,
// router weights): read-only path, not kept in L1.  Not volatile, so the
// compiler may hoist them ahead of the math that consumes earlier loads.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_stream_u32(const void* p) {
  uint32_t v;
  asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// ---------------------------------------------------------------- programmatic dependent launch
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// fire-and-forget request to bring a line into L2
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ uint32_t u4get(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

}  // namespace moe
