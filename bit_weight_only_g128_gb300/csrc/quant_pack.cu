// Offline weight preparation on the GPU: quantize (fp32 -> int4 codes,
// fp16 scales, int4 zero points), pack into the device layout, unpack, and
// dequantize from the packed layout (for checks).
//
// The quantization rule is the asymmetric one that compressed-tensors PR #269
// "Some fixes for AWQ" aligns with AutoAWQ's pseudo_quantize_tensor:
// s = (max - min)/15, z = round(-min/s), q = clamp(round(w/s) + z, 0, 15),
// per group of `group` consecutive k of one column.
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

__device__ __forceinline__ float clamp_0_15(float v) {
  if (!(v >= 0.0f)) return 0.0f;  // also maps NaN to 0
  if (v > 15.0f) return 15.0f;
  return v;
}

// One thread per (group, column); columns fastest so that the k loop reads
// coalesced rows of W.
__global__ void quantize_kernel(const float* __restrict__ W, int K, int N, int group,
                                uint8_t* __restrict__ q, uint16_t* __restrict__ s,
                                uint8_t* __restrict__ z, int* err) {
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int G = K / group;
  if (idx >= (size_t)G * N) return;
  const size_t KN = (size_t)K * N;
  const int n = (int)(idx % N);
  const int grp = (int)(idx / N);
  const size_t k0 = (size_t)grp * group;
  // min and max over the group
  float mn = *ld_at(W + k0 * N + n, W, KN, err), mx = mn;
  for (int k = 0; k < group; ++k) {
    const float w = *ld_at(W + (k0 + k) * N + n, W, KN, err);
    if (w < mn) mn = w;
    if (w > mx) mx = w;
  }
  // s = (max - min)/15 in fp32, stored as fp16; the stored value is used below
  const float s32 = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
  __half sh = __float2half_rn(s32);
  if ((__half_as_ushort(sh) & 0x7fffu) == 0) sh = __float2half_rn(1e-5f);
  const float sf = __half2float(sh);
  // z = clamp(round(-min/s), 0, 15); q = clamp(round(w/s) + z, 0, 15)
  const float zf = clamp_0_15(rintf(__fdiv_rn(-mn, sf)));
  for (int k = 0; k < group; ++k) {
    const float w = *ld_at(W + (k0 + k) * N + n, W, KN, err);
    uint8_t* d = q + (k0 + k) * N + n;
    if (in_buf(d, q, KN, err)) *d = (uint8_t)clamp_0_15(__fadd_rn(rintf(__fdiv_rn(w, sf)), zf));
  }
  if (in_buf(s + idx, s, (size_t)G * N, err)) s[idx] = __half_as_ushort(sh);
  if (in_buf(z + idx, z, (size_t)G * N, err)) z[idx] = (uint8_t)zf;
}

// Position of packed word `widx`: column n and first k of its octet.
__device__ __forceinline__ void word_position(size_t widx, int K, int* n, int* k0) {
  const size_t strip_words = (size_t)(K / kAtomK) * kAtomWords;
  const int j = (int)(widx / strip_words);
  const size_t rem = widx % strip_words;
  const int a = (int)(rem / kAtomWords);
  const int wi = (int)(rem % kAtomWords);
  const int L = wi >> 2, i = wi & 3;
  const int g = L >> 2, t = L & 3, sh = i >> 1, r = i & 1;
  *n = kStripCols * j + g + 8 * r;
  *k0 = kAtomK * a + 32 * sh + 8 * t;
}

// Nibble position of k-offset e within a word: the 3-bit reversal of e.
__device__ __forceinline__ int nibble_of(int e) { return ((e & 1) << 2) | (e & 2) | (e >> 2); }

__global__ void pack_weights_kernel(const uint8_t* __restrict__ q, int K, int N,
                                    uint32_t* __restrict__ Wq, int* err) {
  const size_t widx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (widx >= (size_t)K * N / 8) return;
  int n, k0;
  word_position(widx, K, &n, &k0);
  uint32_t word = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e)
    word |= (uint32_t)(*ld_at(q + (size_t)(k0 + e) * N + n, q, (size_t)K * N, err) & 15u) << (4 * nibble_of(e));
  if (in_buf(Wq + widx, Wq, (size_t)K * N / 8, err)) Wq[widx] = word;
}

// One thread per (strip, group, half h): the 8 scales of columns 16j+8h+c
// (interleaved with the other half), and zero-point word h, whose bytes
// 4h..4h+3 pair the zero points of columns 16j+c and 16j+8+c.
__global__ void pack_meta_kernel(const uint16_t* __restrict__ s, const uint8_t* __restrict__ z,
                                 int K, int N, int group, uint16_t* __restrict__ Sp,
                                 uint32_t* __restrict__ Zp, int* err) {
  const int G = K / group;
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;  // (j*G + grp)*2 + h
  if (idx >= (size_t)(N / kStripCols) * G * 2) return;
  const int h = (int)(idx & 1);
  const size_t jg = idx >> 1;
  const int grp = (int)(jg % G);
  const int j = (int)(jg / G);
  uint32_t word = 0;
  for (int c = 0; c < 8; ++c) {
    const int n = kStripCols * j + 8 * h + c;
    const uint16_t v = *ld_at(s + (size_t)grp * N + n, s, (size_t)G * N, err);
    if (in_buf(Sp + jg * 16 + 2 * c + h, Sp, (size_t)G * N, err)) Sp[jg * 16 + 2 * c + h] = v;
  }
  for (int b = 0; b < 4; ++b) {
    const int c = 4 * h + b;  // byte c of the record
    const uint32_t lo = *ld_at(z + (size_t)grp * N + kStripCols * j + c, z, (size_t)G * N, err) & 15u;
    const uint32_t hi = *ld_at(z + (size_t)grp * N + kStripCols * j + 8 + c, z, (size_t)G * N, err) & 15u;
    word |= (lo | (hi << 4)) << (8 * b);
  }
  if (in_buf(Zp + idx, Zp, (size_t)G * N / 8, err)) Zp[idx] = word;
}

__global__ void unpack_weights_kernel(const uint32_t* __restrict__ Wq, int K, int N,
                                      uint8_t* __restrict__ q, int* err) {
  const size_t widx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (widx >= (size_t)K * N / 8) return;
  int n, k0;
  word_position(widx, K, &n, &k0);
  const uint32_t word = *ld_at(Wq + widx, Wq, (size_t)K * N / 8, err);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    uint8_t* d = q + (size_t)(k0 + e) * N + n;
    if (in_buf(d, q, (size_t)K * N, err)) *d = (uint8_t)((word >> (4 * nibble_of(e))) & 15u);
  }
}

__global__ void unpack_meta_kernel(const uint16_t* __restrict__ Sp, const uint32_t* __restrict__ Zp,
                                   int K, int N, int group, uint16_t* __restrict__ s,
                                   uint8_t* __restrict__ z, int* err) {
  const int G = K / group;
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (size_t)(N / kStripCols) * G * 2) return;
  const int h = (int)(idx & 1);
  const size_t jg = idx >> 1;
  const int grp = (int)(jg % G);
  const int j = (int)(jg / G);
  const size_t GN = (size_t)G * N;
  const uint32_t word = *ld_at(Zp + idx, Zp, GN / 8, err);
  for (int c = 0; c < 8; ++c) {
    const int n = kStripCols * j + 8 * h + c;
    const uint16_t v = *ld_at(Sp + jg * 16 + 2 * c + h, Sp, GN, err);
    if (in_buf(s + (size_t)grp * N + n, s, GN, err)) s[(size_t)grp * N + n] = v;
  }
  for (int b = 0; b < 4; ++b) {
    const int c = 4 * h + b;
    const uint32_t byte = (word >> (8 * b)) & 0xffu;
    uint8_t* d0 = z + (size_t)grp * N + kStripCols * j + c;
    if (in_buf(d0, z, GN, err)) *d0 = (uint8_t)(byte & 15u);
    if (in_buf(d0 + 8, z, GN, err)) d0[8] = (uint8_t)(byte >> 4);
  }
}

// deq [K][N] from the packed buffers, through dequant_word (kB: the bf16
// routine dequant_word_bf16), the tensor-core GEMM's routines.
template <bool kB>
__global__ void dequantize_kernel(const uint32_t* __restrict__ Wq, const uint16_t* __restrict__ Sp,
                                  const uint32_t* __restrict__ Zp, int K, int N, int group,
                                  uint16_t* __restrict__ deq, int* err) {
  const size_t widx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (widx >= (size_t)K * N / 8) return;
  int n, k0;
  word_position(widx, K, &n, &k0);
  const int G = K / group;
  const int j = n / kStripCols, c = n % kStripCols;
  const int grp = k0 / group;
  const size_t jg = (size_t)j * G + grp;
  const size_t GN = (size_t)G * N, KN = (size_t)K * N;
  const uint8_t* zp = reinterpret_cast<const uint8_t*>(Zp);
  const uint32_t zbyte = *ld_at(zp + jg * 8 + (c & 7), zp, GN / 2, err);
  const uint32_t zc = (zbyte >> (4 * (c >> 3))) & 15u;
  const uint16_t sc = *ld_at(Sp + jg * 16 + 2 * (c & 7) + (c >> 3), Sp, GN, err);
  const uint32_t word = *ld_at(Wq + widx, Wq, KN / 8, err);
  uint32_t pairs[4];
  if (kB)
    dequant_word_bf16(word, make_deq_const_bf16(zc, sc), pairs);
  else
    dequant_word(word, make_deq_const(zc, sc), pairs);
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    uint16_t* d = deq + (size_t)(k0 + 2 * p) * N + n;
    if (in_buf(d, deq, KN, err)) *d = (uint16_t)(pairs[p] & 0xffffu);
    if (in_buf(d + N, deq, KN, err)) d[N] = (uint16_t)(pairs[p] >> 16);
  }
}

inline unsigned blocks_for(size_t n, int threads) { return (unsigned)((n + threads - 1) / threads); }

}  // namespace

cudaError_t launch_quantize(const float* W, int K, int N, int group, uint8_t* q, uint16_t* s,
                            uint8_t* z, cudaStream_t stream) {
  int* err = nullptr;
  cudaError_t e = device_error_word(&err);
  if (e != cudaSuccess) return e;
  const size_t n = (size_t)(K / group) * N;
  quantize_kernel<<<blocks_for(n, 256), 256, 0, stream>>>(W, K, N, group, q, s, z, err);
  return cudaGetLastError();
}

cudaError_t launch_pack(const uint8_t* q, const uint16_t* s, const uint8_t* z, int K, int N,
                        int group, uint32_t* Wq, uint16_t* Sp, uint32_t* Zp, cudaStream_t stream) {
  int* err = nullptr;
  cudaError_t e = device_error_word(&err);
  if (e != cudaSuccess) return e;
  const size_t words = (size_t)K * N / 8;
  pack_weights_kernel<<<blocks_for(words, 256), 256, 0, stream>>>(q, K, N, Wq, err);
  const size_t meta = (size_t)(N / kStripCols) * (K / group) * 2;
  pack_meta_kernel<<<blocks_for(meta, 256), 256, 0, stream>>>(s, z, K, N, group, Sp, Zp, err);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint32_t* Wq, const uint16_t* Sp, const uint32_t* Zp, int K,
                          int N, int group, uint8_t* q, uint16_t* s, uint8_t* z,
                          cudaStream_t stream) {
  int* err = nullptr;
  cudaError_t e = device_error_word(&err);
  if (e != cudaSuccess) return e;
  const size_t words = (size_t)K * N / 8;
  unpack_weights_kernel<<<blocks_for(words, 256), 256, 0, stream>>>(Wq, K, N, q, err);
  const size_t meta = (size_t)(N / kStripCols) * (K / group) * 2;
  unpack_meta_kernel<<<blocks_for(meta, 256), 256, 0, stream>>>(Sp, Zp, K, N, group, s, z, err);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint32_t* Wq, const uint16_t* Sp, const uint32_t* Zp, int K,
                              int N, int group, uint16_t* deq, bool bf16, cudaStream_t stream) {
  int* err = nullptr;
  cudaError_t e = device_error_word(&err);
  if (e != cudaSuccess) return e;
  const size_t words = (size_t)K * N / 8;
  if (bf16)
    dequantize_kernel<true><<<blocks_for(words, 256), 256, 0, stream>>>(Wq, Sp, Zp, K, N, group, deq, err);
  else
    dequantize_kernel<false><<<blocks_for(words, 256), 256, 0, stream>>>(Wq, Sp, Zp, K, N, group, deq, err);
  return cudaGetLastError();
}

}  // namespace w4a16
