// Device helpers shared by the W4A16 kernels (sm_103a).
//
// Packed format (see include/w4a16.h): a word holds 8 consecutive k of one
// column; nibble p holds k-offset rev3(p), i.e. nibbles 0..7 hold k-offsets
// 0 4 2 6 1 5 3 7, so one mask on the word (or on the word shifted by 8)
// pulls a pair of consecutive k-offsets into the two fp16 halves of a
// register: (0,1) and (4,5) from the word, (2,3) and (6,7) from word >> 8,
// the second pair of each one nibble higher.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "w4a16.h"

namespace w4a16 {

constexpr int kStripCols = 16;   // columns per strip
constexpr int kAtomK = 64;       // k per atom
constexpr int kAtomWords = 128;  // 32-bit words per atom (16 * 64 / 8)

// ------------------------------------------------------------------ checked build
// Compiled with -DW4A16_CHECKED (build(checked=True)), every global and
// shared-memory access of the kernels is tested against its buffer's extent
// first; an access outside sets kErrBounds in the library's device error
// word and is skipped (a load reads the buffer's first element instead), so
// nothing faults and w4a16_device_status reports it. In the normal build the
// tests compile away.
constexpr int kErrBounds = 64;

#ifdef W4A16_CHECKED
constexpr bool kCheckedBuild = true;
#else
constexpr bool kCheckedBuild = false;
#endif

// p lies in [base, base + n): true; else (checked build) records kErrBounds.
template <class T>
__device__ __forceinline__ bool in_buf(const T* p, const T* base, size_t n, int* err) {
  if (!kCheckedBuild) return true;
  if (p >= base && p < base + n) return true;
  atomicOr(err, kErrBounds);
  return false;
}

// The address to load element p from: p if it lies in [base, base + n), else
// base (and kErrBounds).
template <class T>
__device__ __forceinline__ const T* ld_at(const T* p, const T* base, size_t n, int* err) {
  return in_buf(p, base, n, err) ? p : base;
}

// [addr, addr + bytes) lies in this CTA's dynamic shared memory, which starts
// at shared address `dyn_base`: true; else (checked build) records kErrBounds.
__device__ __forceinline__ bool in_smem(uint32_t addr, uint32_t bytes, uint32_t dyn_base, int* err) {
  if (!kCheckedBuild) return true;
  uint32_t dyn;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
  if (addr >= dyn_base && addr + bytes <= dyn_base + dyn) return true;
  atomicOr(err, kErrBounds);
  return false;
}

// Tensor-memory columns [col, col + ncols) lie in an allocation of `cols`.
__device__ __forceinline__ bool in_tmem(uint32_t col, uint32_t ncols, uint32_t cols, int* err) {
  if (!kCheckedBuild) return true;
  if (col + ncols <= cols) return true;
  atomicOr(err, kErrBounds);
  return false;
}

// ------------------------------------------------------------------ fp16x2

__device__ __forceinline__ uint32_t hsub2_rn(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hmul2_rn(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hfma2_rn(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Per (group, column) constants of the dequantization of one column.
struct DeqConst {
  uint32_t zb;    // fp16x2 (1024 + z): subtracted from (1024 + q)
  uint32_t nzb4;  // fp16x2 -(64 + z): added to (1024 + 16 q)/16
  uint32_t s2;    // fp16x2 (s, s)
};

__device__ __forceinline__ DeqConst make_deq_const(uint32_t z, uint16_t s_bits) {
  DeqConst c;
  c.zb = (0x6400u + z) * 0x00010001u;           // 1024 + z, exact (ulp 1)
  c.nzb4 = (0xD400u + 16u * z) * 0x00010001u;   // -(64 + z), exact (ulp 1/16)
  c.s2 = (uint32_t)s_bits * 0x00010001u;
  return c;
}

// One packed word -> four fp16x2 values out[p] = (deq[2p], deq[2p+1]) with
// deq = RNE_fp16((q - z) * s). The subtraction is exact (integers below
// 2048 in fp16, or an fma whose exact result is the integer q - z), so the
// multiply by s is the only rounding, as in the definition.
__device__ __forceinline__ void dequant_word(uint32_t w, const DeqConst& c, uint32_t out[4]) {
  const uint32_t kMagic = 0x64006400u;      // fp16x2 (1024, 1024)
  const uint32_t kSixteenth = 0x2C002C00u;  // fp16x2 (1/16, 1/16)
  const uint32_t w8 = w >> 8;
  const uint32_t x0 = (w & 0x000F000Fu) | kMagic;    // 1024 + q0,    1024 + q1
  const uint32_t x1 = (w8 & 0x000F000Fu) | kMagic;   // 1024 + q2,    1024 + q3
  const uint32_t x2 = (w & 0x00F000F0u) | kMagic;    // 1024 + 16 q4, 1024 + 16 q5
  const uint32_t x3 = (w8 & 0x00F000F0u) | kMagic;   // 1024 + 16 q6, 1024 + 16 q7
  out[0] = hmul2_rn(hsub2_rn(x0, c.zb), c.s2);
  out[1] = hmul2_rn(hsub2_rn(x1, c.zb), c.s2);
  out[2] = hmul2_rn(hfma2_rn(x2, kSixteenth, c.nzb4), c.s2);
  out[3] = hmul2_rn(hfma2_rn(x3, kSixteenth, c.nzb4), c.s2);
}

// Per (group, column) constants of the bf16 dequantization of one column.
struct DeqConstBf16 {
  float s;    // the fp16 scale, exact in fp32
  float nzs;  // -(128 + z) * s, exact (8 x 11 significant bits)
};

__device__ __forceinline__ DeqConstBf16 make_deq_const_bf16(uint32_t z, uint16_t s_bits) {
  DeqConstBf16 c;
  c.s = __half2float(__ushort_as_half(s_bits));
  c.nzs = -(float)(128u + z) * c.s;
  return c;
}

// One packed word -> four bf16x2 values out[p] = (deq[2p], deq[2p+1]) with
// deq = RNE_bf16((q - z) * s). Each code becomes the fp32 128 + q: byte
// permutes put a byte 0x0q (the nibbles masked apart: even nibbles in place,
// odd ones shifted down) under the bytes 0x43 and 0x00 of 128.0's bit
// pattern, where its unit bit is bit 16. Then (128 + q) s - (128 + z) s is
// one fma of exact operands whose exact result, (q - z) s with at most 15
// significant bits, is representable: the fma returns it unrounded, and the
// conversion to bf16 is the only rounding.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void dequant_word_bf16(uint32_t w, const DeqConstBf16& c, uint32_t out[4]) {
  const uint32_t t = w & 0x0F0F0F0Fu;         // bytes: nibbles 0 2 4 6 = k 0 2 1 3
  const uint32_t u = (w >> 4) & 0x0F0F0F0Fu;  // bytes: nibbles 1 3 5 7 = k 4 6 5 7
  constexpr uint32_t kHi = 0x00000043u;       // byte 4 = 0x43, bytes 5..7 = 0
  auto f = [&](uint32_t x, uint32_t sel) { return fmaf(__uint_as_float(__byte_perm(x, kHi, sel)), c.s, c.nzs); };
  // selector: result bytes (0, 0, byte b of x, 0x43) = 0x4b55
  out[0] = bf16x2_rn(f(t, 0x4055), f(t, 0x4255));  // k 0, 1
  out[1] = bf16x2_rn(f(t, 0x4155), f(t, 0x4355));  // k 2, 3
  out[2] = bf16x2_rn(f(u, 0x4055), f(u, 0x4255));  // k 4, 5
  out[3] = bf16x2_rn(f(u, 0x4155), f(u, 0x4355));  // k 6, 7
}

// ------------------------------------------------------------------ loads

// Streaming 16-byte load of packed weights: read once, keep out of L1.
__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// 16-byte load of activations, cached in L1 (shared by the CTA's warps).
__device__ __forceinline__ uint4 ldg_keep(const void* p) {
  uint4 v;
  asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// ------------------------------------------------------------------ mma.sync

// D (16x8 f32) += A (16x16 f16, row) * B (16x8 f16, col).
__device__ __forceinline__ void mma_16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace w4a16
