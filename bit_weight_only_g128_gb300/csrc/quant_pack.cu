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
                                uint8_t* __restrict__ z) {
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int G = K / group;
  if (idx >= (size_t)G * N) return;
  const int n = (int)(idx % N);
  const int grp = (int)(idx / N);
  const size_t k0 = (size_t)grp * group;
  // min and max over the group
  float mn = W[k0 * N + n], mx = mn;
  for (int k = 0; k < group; ++k) {
    const float w = W[(k0 + k) * N + n];
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
    const float w = W[(k0 + k) * N + n];
    q[(k0 + k) * N + n] = (uint8_t)clamp_0_15(__fadd_rn(rintf(__fdiv_rn(w, sf)), zf));
  }
  s[idx] = __half_as_ushort(sh);
  z[idx] = (uint8_t)zf;
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
                                    uint32_t* __restrict__ Wq) {
  const size_t widx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (widx >= (size_t)K * N / 8) return;
  int n, k0;
  word_position(widx, K, &n, &k0);
  uint32_t word = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e)
    word |= (uint32_t)(q[(size_t)(k0 + e) * N + n] & 15u) << (4 * nibble_of(e));
  Wq[widx] = word;
}

// One thread per (strip, group, half h): the 8 scales of columns 16j+8h+c
// (interleaved with the other half), and zero-point word h, whose bytes
// 4h..4h+3 pair the zero points of columns 16j+c and 16j+8+c.
__global__ void pack_meta_kernel(const uint16_t* __restrict__ s, const uint8_t* __restrict__ z,
                                 int K, int N, int group, uint16_t* __restrict__ Sp,
                                 uint32_t* __restrict__ Zp) {
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
    Sp[jg * 16 + 2 * c + h] = s[(size_t)grp * N + n];
  }
  for (int b = 0; b < 4; ++b) {
    const int c = 4 * h + b;  // byte c of the record
    const uint32_t lo = z[(size_t)grp * N + kStripCols * j + c] & 15u;
    const uint32_t hi = z[(size_t)grp * N + kStripCols * j + 8 + c] & 15u;
    word |= (lo | (hi << 4)) << (8 * b);
  }
  Zp[idx] = word;
}

__global__ void unpack_weights_kernel(const uint32_t* __restrict__ Wq, int K, int N,
                                      uint8_t* __restrict__ q) {
  const size_t widx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (widx >= (size_t)K * N / 8) return;
  int n, k0;
  word_position(widx, K, &n, &k0);
  const uint32_t word = Wq[widx];
#pragma unroll
  for (int e = 0; e < 8; ++e)
    q[(size_t)(k0 + e) * N + n] = (uint8_t)((word >> (4 * nibble_of(e))) & 15u);
}

__global__ void unpack_meta_kernel(const uint16_t* __restrict__ Sp, const uint32_t* __restrict__ Zp,
                                   int K, int N, int group, uint16_t* __restrict__ s,
                                   uint8_t* __restrict__ z) {
  const int G = K / group;
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (size_t)(N / kStripCols) * G * 2) return;
  const int h = (int)(idx & 1);
  const size_t jg = idx >> 1;
  const int grp = (int)(jg % G);
  const int j = (int)(jg / G);
  const uint32_t word = Zp[idx];
  for (int c = 0; c < 8; ++c) {
    const int n = kStripCols * j + 8 * h + c;
    s[(size_t)grp * N + n] = Sp[jg * 16 + 2 * c + h];
  }
  for (int b = 0; b < 4; ++b) {
    const int c = 4 * h + b;
    const uint32_t byte = (word >> (8 * b)) & 0xffu;
    z[(size_t)grp * N + kStripCols * j + c] = (uint8_t)(byte & 15u);
    z[(size_t)grp * N + kStripCols * j + 8 + c] = (uint8_t)(byte >> 4);
  }
}

// deq [K][N] from the packed buffers, through dequant_word (kB: the bf16
// routine dequant_word_bf16), the tensor-core GEMM's routines.
template <bool kB>
__global__ void dequantize_kernel(const uint32_t* __restrict__ Wq, const uint16_t* __restrict__ Sp,
                                  const uint32_t* __restrict__ Zp, int K, int N, int group,
                                  uint16_t* __restrict__ deq) {
  const size_t widx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (widx >= (size_t)K * N / 8) return;
  int n, k0;
  word_position(widx, K, &n, &k0);
  const int G = K / group;
  const int j = n / kStripCols, c = n % kStripCols;
  const int grp = k0 / group;
  const size_t jg = (size_t)j * G + grp;
  const uint32_t zbyte = reinterpret_cast<const uint8_t*>(Zp)[jg * 8 + (c & 7)];
  const uint32_t zc = (zbyte >> (4 * (c >> 3))) & 15u;
  const uint16_t sc = Sp[jg * 16 + 2 * (c & 7) + (c >> 3)];
  uint32_t pairs[4];
  if (kB)
    dequant_word_bf16(Wq[widx], make_deq_const_bf16(zc, sc), pairs);
  else
    dequant_word(Wq[widx], make_deq_const(zc, sc), pairs);
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    deq[(size_t)(k0 + 2 * p) * N + n] = (uint16_t)(pairs[p] & 0xffffu);
    deq[(size_t)(k0 + 2 * p + 1) * N + n] = (uint16_t)(pairs[p] >> 16);
  }
}

inline unsigned blocks_for(size_t n, int threads) { return (unsigned)((n + threads - 1) / threads); }

}  // namespace

cudaError_t launch_quantize(const float* W, int K, int N, int group, uint8_t* q, uint16_t* s,
                            uint8_t* z, cudaStream_t stream) {
  const size_t n = (size_t)(K / group) * N;
  quantize_kernel<<<blocks_for(n, 256), 256, 0, stream>>>(W, K, N, group, q, s, z);
  return cudaGetLastError();
}

cudaError_t launch_pack(const uint8_t* q, const uint16_t* s, const uint8_t* z, int K, int N,
                        int group, uint32_t* Wq, uint16_t* Sp, uint32_t* Zp, cudaStream_t stream) {
  const size_t words = (size_t)K * N / 8;
  pack_weights_kernel<<<blocks_for(words, 256), 256, 0, stream>>>(q, K, N, Wq);
  const size_t meta = (size_t)(N / kStripCols) * (K / group) * 2;
  pack_meta_kernel<<<blocks_for(meta, 256), 256, 0, stream>>>(s, z, K, N, group, Sp, Zp);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint32_t* Wq, const uint16_t* Sp, const uint32_t* Zp, int K,
                          int N, int group, uint8_t* q, uint16_t* s, uint8_t* z,
                          cudaStream_t stream) {
  const size_t words = (size_t)K * N / 8;
  unpack_weights_kernel<<<blocks_for(words, 256), 256, 0, stream>>>(Wq, K, N, q);
  const size_t meta = (size_t)(N / kStripCols) * (K / group) * 2;
  unpack_meta_kernel<<<blocks_for(meta, 256), 256, 0, stream>>>(Sp, Zp, K, N, group, s, z);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint32_t* Wq, const uint16_t* Sp, const uint32_t* Zp, int K,
                              int N, int group, uint16_t* deq, bool bf16, cudaStream_t stream) {
  const size_t words = (size_t)K * N / 8;
  if (bf16)
    dequantize_kernel<true><<<blocks_for(words, 256), 256, 0, stream>>>(Wq, Sp, Zp, K, N, group, deq);
  else
    dequantize_kernel<false><<<blocks_for(words, 256), 256, 0, stream>>>(Wq, Sp, Zp, K, N, group, deq);
  return cudaGetLastError();
}

}  // namespace w4a16
