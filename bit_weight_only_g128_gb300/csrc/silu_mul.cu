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

// Eight adjacent output columns per thread (16-byte loads and stores; N/2 is
// a multiple of 16). silu(g) = g / (1 + e^-g) with the fast exponential and
// division intrinsics: their relative error (a few fp32 ulps) is far inside
// the epilogue's share of the bound (2^-10 of the result, which also covers
// the final rounding). kB: bf16 values, else fp16.
template <bool kB>
__device__ __forceinline__ float2 to_float2(uint32_t v) {
  if (kB) return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}
template <bool kB>
__device__ __forceinline__ uint32_t from_float2(float lo, float hi) {
  if (kB) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&b);
  }
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float silu_times(float g, float u) {
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

template <bool kB>
__global__ void __launch_bounds__(256) silu_mul_kernel(const uint4* __restrict__ yfull, int M, int N,
                                                       uint4* __restrict__ y, int* err) {
  // launched with programmatic serialization: scheduled while the GEMM that
  // writes the product drains, it waits for that grid before reading it
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int hv = N / 16;  // 16-byte vectors of one half of a row
  const long total = (long)M * hv;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
       i += (long)gridDim.x * blockDim.x) {
    const long m = i / hv, j = i - m * hv;
    const size_t nin = (size_t)M * (N / 8);
    const uint4 g = *ld_at(yfull + m * (N / 8) + j, yfull, nin, err);
    const uint4 u = *ld_at(yfull + m * (N / 8) + hv + j, yfull, nin, err);
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 gf = to_float2<kB>(gw[k]), uf = to_float2<kB>(uw[k]);
      o[k] = from_float2<kB>(silu_times(gf.x, uf.x), silu_times(gf.y, uf.y));
    }
    if (in_buf(y + m * hv + j, y, (size_t)total, err)) y[m * hv + j] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

cudaError_t launch_silu_mul(const uint16_t* Yfull, int M, int N, uint16_t* Y, bool bf16,
                            cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  int* err = nullptr;
  cudaError_t e = device_error_word(&err);
  if (e != cudaSuccess) return e;
  const long vecs = (long)M * (N / 16);
  int blocks = (int)((vecs + 255) / 256);
  if (blocks > 152 * 16) blocks = 152 * 16;
  const uint4* in = reinterpret_cast<const uint4*>(Yfull);
  uint4* out = reinterpret_cast<uint4*>(Y);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return bf16 ? cudaLaunchKernelEx(&cfg, silu_mul_kernel<true>, in, M, N, out, err)
              : cudaLaunchKernelEx(&cfg, silu_mul_kernel<false>, in, M, N, out, err);
}

}  // namespace w4a16
