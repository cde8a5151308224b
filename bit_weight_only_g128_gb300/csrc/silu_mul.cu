// The fused gate/up epilogue as a separate pass, for the paths that do not
// fuse it into the GEMM (stream-K decode, tensor core): the product of the
// fused [gate | up] weight, rounded to fp16, is read back and
// Y = silu(gate) * up is formed in fp32 and rounded once (lmdeploy issue
// #2274, "Modification": gate and up fused into one weight, SiLU fused with
// the kernels around the GEMM).
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

// Two adjacent output columns per thread (N/2 is a multiple of 16); T is
// __half2 or __nv_bfloat162.
__device__ __forceinline__ float2 to_float2(__half2 v) { return __half22float2(v); }
__device__ __forceinline__ float2 to_float2(__nv_bfloat162 v) { return __bfloat1622float2(v); }
__device__ __forceinline__ void from_float2(float lo, float hi, __half2* d) { *d = __floats2half2_rn(lo, hi); }
__device__ __forceinline__ void from_float2(float lo, float hi, __nv_bfloat162* d) {
  *d = __floats2bfloat162_rn(lo, hi);
}

template <typename T>
__global__ void silu_mul_kernel(const T* __restrict__ yfull, int M, int N, T* __restrict__ y) {
  const int hp = N / 4;  // column pairs of one half
  const long total = (long)M * hp;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
       i += (long)gridDim.x * blockDim.x) {
    const long m = i / hp, j = i - m * hp;
    const float2 g = to_float2(yfull[m * (N / 2) + j]);
    const float2 u = to_float2(yfull[m * (N / 2) + hp + j]);
    const float lo = g.x / (1.0f + expf(-g.x)) * u.x;
    const float hi = g.y / (1.0f + expf(-g.y)) * u.y;
    from_float2(lo, hi, y + m * hp + j);
  }
}

}  // namespace

cudaError_t launch_silu_mul(const uint16_t* Yfull, int M, int N, uint16_t* Y, bool bf16,
                            cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  const long pairs = (long)M * (N / 4);
  int blocks = (int)((pairs + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  if (bf16)
    silu_mul_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const __nv_bfloat162*>(Yfull), M, N,
                                                reinterpret_cast<__nv_bfloat162*>(Y));
  else
    silu_mul_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const __half2*>(Yfull), M, N,
                                                reinterpret_cast<__half2*>(Y));
  return cudaGetLastError();
}

}  // namespace w4a16
