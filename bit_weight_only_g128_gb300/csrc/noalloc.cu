// w4a16_gemm_noalloc: the decode-path GEMM for callers that cannot allocate
// device memory. The pages have no counterpart of this entry point.
//
// Who needs it: code that is not allowed to allocate on the device once it is
// running (a serving process with a fixed memory budget, a plugin hosted by a
// framework whose allocator it cannot reach, a latency-critical loop that must
// not pay for an allocation), but still wants the split-work decode kernel,
// which combines partial sums through scratch memory.
//
// The scratch lives in one file-scope device array below: every GPU that
// loads the library reserves it (32 KiB of flags plus 8 MiB of partial
// tiles) until the process exits. Host code cannot pass the array's name to
// a kernel (on the host it only stands for the symbol); its device address is
// looked up once per device, on the first call made with that device current,
// and kept for the life of the process (a device reset would make it stale:
// no call may follow one).
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

constexpr size_t kCounterBytes = 32768;       // room for 2^20 / 128 column blocks
constexpr size_t kTileBytes = 8u << 20;       // fp32 partial tiles
constexpr size_t kScratchBytes = kCounterBytes + kTileBytes;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on device `dev` (current), looked up
// once per device.
cudaError_t scratch_address(int dev, void** addr) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = ptr;
  }
  *addr = g_scratch_addr[dev];
  return cudaSuccess;
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int fail_fmt(int code, const char* fmt, long a = 0, long b = 0) {
  char msg[256];
  snprintf(msg, sizeof(msg), fmt, a, b);
  return report_error(code, msg);
}

}  // namespace
}  // namespace w4a16

using namespace w4a16;

extern "C" int w4a16_gemm_noalloc(const uint16_t* A, const uint32_t* Wq, const uint16_t* scales,
                                  const uint32_t* zeros, int M, int N, int K, int group,
                                  uint16_t* Y, void* stream) {
  if (M < 0 || K <= 0 || N <= 0 || group <= 0)
    return fail_fmt(W4A16_ERR_INVALID_ARG, "M, N, K, group must be positive (M may be 0)");
  if (M > (1 << 20) || K > (1 << 20) || N > (1 << 20))
    return fail_fmt(W4A16_ERR_UNSUPPORTED_SHAPE, "M, N or K above 2^20");
  if (N % kStripCols || K % kAtomK || group % kAtomK || K % group)
    return fail_fmt(W4A16_ERR_UNSUPPORTED_SHAPE,
                    "shape rules: N %% 16, K %% 64, group %% 64 and K %% group must be 0");
  const long units = decode_units(N, K, group);
  if (units <= 0)
    return fail_fmt(W4A16_ERR_UNSUPPORTED_SHAPE, "group=%ld must be K or 64 times a power of two",
                    group);
  if (M == 0) return report_ok();
  if (!A || !Wq || !scales || !zeros || !Y) return fail_fmt(W4A16_ERR_INVALID_ARG, "null pointer");
  if (!aligned_to(A, 16) || !aligned_to(Wq, 16) || !aligned_to(scales, 16) || !aligned_to(Y, 16) ||
      !aligned_to(zeros, 8))
    return fail_fmt(W4A16_ERR_MISALIGNED, "alignment: A, Wq, scales, Y need 16 bytes and zeros 8");

  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess && (dev < 0 || dev >= kMaxDevices)) e = cudaErrorInvalidDevice;
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // the kernels run on the stream's device with this device's scratch address:
  // the two must be the same device
  int stream_dev = dev;
  if (e == cudaSuccess) e = cudaStreamGetDevice((cudaStream_t)stream, &stream_dev);
  if (e == cudaSuccess && stream_dev != dev) {
    char msg[256];
    snprintf(msg, sizeof(msg), "the stream belongs to device %d, the current device is %d",
             stream_dev, dev);
    return report_error(W4A16_ERR_INVALID_ARG, msg);
  }
  void* scratch = nullptr;
  if (e == cudaSuccess) e = scratch_address(dev, &scratch);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "scratch set-up: %s", cudaGetErrorString(e));
    return report_error(W4A16_ERR_CUDA, msg);
  }
  // one CTA per resident slot, as w4a16_gemm chooses, if the scratch holds its tiles
  const int rows = M < 16 ? M : 16;
  long ctas = (long)sms * decode_ctas_per_sm(rows);
  if (ctas > units) ctas = units;
  if (ctas > kDecodeMaxCtas) ctas = kDecodeMaxCtas;
  const size_t need = decode_workspace_bytes(rows, N, (int)ctas);
  if (need > kScratchBytes)
    return fail_fmt(W4A16_ERR_UNSUPPORTED_SHAPE,
                    "needs %ld scratch bytes, above the %ld this entry point holds", (long)need,
                    (long)kScratchBytes);
  // the per-CTA flags must start at zero (the kernel leaves them at zero)
  e = cudaMemsetAsync(scratch, 0, (size_t)ctas * sizeof(int), (cudaStream_t)stream);
  for (int r0 = 0; e == cudaSuccess && r0 < M; r0 += 16) {
    const int r = M - r0 < 16 ? M - r0 : 16;
    e = launch_decode(A + (size_t)r0 * K, Wq, scales, zeros, Y + (size_t)r0 * N, r, N, K, group,
                      (int)ctas, scratch, false, false, nullptr, (cudaStream_t)stream);
  }
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "decode kernel launch: %s", cudaGetErrorString(e));
    return report_error(W4A16_ERR_CUDA, msg);
  }
  return report_ok();
}
