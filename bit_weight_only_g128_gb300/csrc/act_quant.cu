// W4A8: the dynamic per-token quantization of the activations to 8 bits
// (compressed-tensors PR #269, the Arm example: 16-bit activations in, 8-bit
// activations inside the operation; lmdeploy issue #2274: W4A8 with online
// activation quantization). Per row m: amax = max_k |a|, s_a = amax / 127
// (1 for a row of zeros), a_q = clamp(round(a / s_a), -127, 127), in IEEE
// fp32 with round-half-to-even, so the codes do not depend on compiler
// flags (the scale's division is __fdiv_rn).
//
// The codes need round(RN(a / s_a)), not the quotient itself. t = a * RN(1/s_a)
// differs from the exact quotient a / s_a by under 2 ulps of t (two
// roundings), and so does RN(a / s_a); where the exact quotient is farther
// than that from a midpoint k + 1/2, both round to the same integer. So t
// decides unless it lies within 2^-14 (at least 4 ulps, |t| < 128) of a
// midpoint, and there the code is taken from the correctly rounded quotient.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

constexpr int kQThreads = 256;

template <bool kIn>
__device__ __forceinline__ float act_value(uint32_t bits16) {
  return kIn ? __bfloat162float(__ushort_as_bfloat16((unsigned short)bits16))
             : __half2float(__ushort_as_half((unsigned short)bits16));
}

__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void wait_for_previous_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// One CTA per row. The row is read once from global memory, 16 bytes per
// thread at a time, into shared memory (K * 2 bytes) while its largest
// magnitude is found; the codes are then formed from shared memory. Launched
// as a plain launch (fully after the previous kernel, fully before the GEMM):
// measured on the 7B decode step, letting the GEMM start early (programmatic
// serialization) helped at one row but delayed the GEMM's CTAs on the SMs
// this kernel holds at 8 and 16 rows, and the step lost 3%. (The grid-
// dependency instructions below are then no-ops.)
// kIn: bf16 input; kCodes: the codes as bf16 (else fp16) integer values.
template <bool kIn, bool kCodes>
__global__ void __launch_bounds__(kQThreads) quantize_act_kernel(const uint16_t* __restrict__ A, int K,
                                                                 int8_t* __restrict__ aq,
                                                                 uint16_t* __restrict__ codes,
                                                                 float* __restrict__ s_a, int M,
                                                                 int* err) {
  extern __shared__ uint4 srow[];
  __shared__ float wmax[kQThreads / 32];
  allow_dependents();
  wait_for_previous_grid();
  const int m = blockIdx.x;
  const uint4* row = reinterpret_cast<const uint4*>(A + (size_t)m * K);
  const int nv = K / 8;
  float amax = 0.f;
  const uint4* Av = reinterpret_cast<const uint4*>(A);
  uint32_t dyn;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
  for (int i = threadIdx.x; i < nv; i += kQThreads) {
    const uint4 v = *ld_at(row + i, Av, (size_t)M * nv, err);
    if (!kCheckedBuild || in_buf(srow + i, srow, dyn / 16, err)) srow[i] = v;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      amax = fmaxf(amax, fabsf(act_value<kIn>(w[j] & 0xffffu)));
      amax = fmaxf(amax, fabsf(act_value<kIn>(w[j] >> 16)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = wmax[0];
#pragma unroll
  for (int i = 1; i < kQThreads / 32; ++i) amax = fmaxf(amax, wmax[i]);
  const float s = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 1.0f;
  const float inv = __frcp_rn(s);
  if (threadIdx.x == 0 && in_buf(s_a + m, s_a, (size_t)M, err)) s_a[m] = s;
  auto code = [&](float a) {
    const float t = a * inv;
    float r = rintf(t);
    if (fabsf(fabsf(t - r) - 0.5f) < 6.103515625e-05f)  // within 2^-14 of a midpoint
      r = rintf(__fdiv_rn(a, s));
    return fminf(fmaxf(r, -127.f), 127.f);
  };
  for (int i = threadIdx.x; i < nv; i += kQThreads) {
    const uint4 v = *ld_at(srow + i, srow, kCheckedBuild ? dyn / 16 : (size_t)nv, err);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float r[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      r[2 * j] = act_value<kIn>(w[j] & 0xffffu);
      r[2 * j + 1] = act_value<kIn>(w[j] >> 16);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) r[j] = code(r[j]);
    if (aq) {
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        lo |= ((uint32_t)(int)r[j] & 0xffu) << (8 * j);
        hi |= ((uint32_t)(int)r[4 + j] & 0xffu) << (8 * j);
      }
      uint2* d = reinterpret_cast<uint2*>(aq + (size_t)m * K) + i;
      if (in_buf(d, reinterpret_cast<uint2*>(aq), (size_t)M * nv, err)) *d = make_uint2(lo, hi);
    }
    if (codes) {
      uint32_t c[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (kCodes) {
          const __nv_bfloat162 b = __floats2bfloat162_rn(r[2 * j], r[2 * j + 1]);
          c[j] = *reinterpret_cast<const uint32_t*>(&b);
        } else {
          const __half2 h = __floats2half2_rn(r[2 * j], r[2 * j + 1]);
          c[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
      }
      uint4* d = reinterpret_cast<uint4*>(codes + (size_t)m * K) + i;
      if (in_buf(d, reinterpret_cast<uint4*>(codes), (size_t)M * nv, err)) *d = make_uint4(c[0], c[1], c[2], c[3]);
    }
  }
}

template <bool kIn, bool kCodes>
cudaError_t launch_q(const uint16_t* A, int M, int K, int8_t* aq, uint16_t* codes, float* s_a,
                     cudaStream_t stream) {
  auto kern = quantize_act_kernel<kIn, kCodes>;
  const size_t smem = (size_t)K * 2;
  if (smem > 48 * 1024) {
    cudaError_t e = set_max_smem_once(reinterpret_cast<const void*>(kern), (int)smem);
    if (e != cudaSuccess) return e;
  }
  int* err = nullptr;
  cudaError_t e = device_error_word(&err);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(M);
  cfg.blockDim = dim3(kQThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kern, A, K, aq, codes, s_a, M, err);
}

}  // namespace

// K up to 2^16 (128 KiB of shared memory for the row).
cudaError_t launch_quantize_act(const uint16_t* A, int M, int K, bool in_bf16, int8_t* aq,
                                uint16_t* codes, bool codes_bf16, float* s_a, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  if (K > 65536) return cudaErrorInvalidValue;
  if (in_bf16)
    return codes_bf16 ? launch_q<true, true>(A, M, K, aq, codes, s_a, stream)
                      : launch_q<true, false>(A, M, K, aq, codes, s_a, stream);
  return codes_bf16 ? launch_q<false, true>(A, M, K, aq, codes, s_a, stream)
                    : launch_q<false, false>(A, M, K, aq, codes, s_a, stream);
}

}  // namespace w4a16
