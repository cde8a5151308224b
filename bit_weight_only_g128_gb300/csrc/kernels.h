// Launchers of the W4A16 kernels (host side). Arguments are validated by the
// C ABI layer (api.cu) before any of these is called.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace w4a16 {

cudaError_t launch_quantize(const float* W, int K, int N, int group, uint8_t* q, uint16_t* s,
                            uint8_t* z, cudaStream_t stream);
cudaError_t launch_pack(const uint8_t* q, const uint16_t* s, const uint8_t* z, int K, int N,
                        int group, uint32_t* Wq, uint16_t* Sp, uint32_t* Zp, cudaStream_t stream);
cudaError_t launch_unpack(const uint32_t* Wq, const uint16_t* Sp, const uint32_t* Zp, int K,
                          int N, int group, uint8_t* q, uint16_t* s, uint8_t* z,
                          cudaStream_t stream);
cudaError_t launch_dequantize(const uint32_t* Wq, const uint16_t* Sp, const uint32_t* Zp, int K,
                              int N, int group, uint16_t* deq, cudaStream_t stream);

// Split-K register-dequant GEMV for M <= 16 rows of A (one launch); `split`
// CTAs of one thread-block cluster share each block of 128 output columns.
cudaError_t launch_decode(const uint16_t* A, const uint32_t* Wq, const uint16_t* Sp,
                          const uint32_t* Zp, uint16_t* Y, int M, int N, int K, int group,
                          int split, cudaStream_t stream);

// Largest split the decode kernel accepts (cluster size).
constexpr int kDecodeMaxSplit = 8;
// Output columns per decode CTA.
constexpr int kDecodeBlockCols = 128;

}  // namespace w4a16
