// Decode path of the W4A16 linear layer: host side (shapes, layouts,
// launches) and the fp16-activation instantiations of the kernels in
// decode_impl.cuh.
#include <atomic>

#include "decode_impl.cuh"

namespace w4a16 {
namespace {

// Atoms per group as the kernel template sees it (1, 2, 4, or 8 for >= 8
// atoms or a single group per column) and the group shift; false if the
// group size is not supported.
bool group_shape(int K, int group, int* apg_t, int* gshift) {
  const int apg = group / kAtomK;
  const bool pow2 = apg > 0 && (apg & (apg - 1)) == 0;
  if (pow2) {
    int sh = 0;
    while ((1 << sh) < apg) ++sh;
    *gshift = sh;
    *apg_t = apg < 8 ? apg : 8;
    return true;
  }
  if (group == K) {  // one group per column
    *apg_t = 8;
    *gshift = 30;
    return true;
  }
  return false;
}

}  // namespace

// CTAs of the decode kernel that fit on one SM (occupancy query, M <= 8 or
// 9..16 rows, for the variant with the most shared memory: groups of 64),
// cached per device; concurrent first calls may both run the query, and
// store the same value.
int decode_ctas_per_sm(int M) {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices][2];
  const int v = M <= 8 ? 0 : 1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = -1;
  if (dev >= 0) {
    const int c = cache[dev][v].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  cudaError_t e;
  if (v == 0) {
    e = set_max_smem_once(reinterpret_cast<const void*>(decode_kernel<1, 1, false>), Smem<1, 8>::kTotal);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<1, 1, false>, kThreads, Smem<1, 8>::kTotal);
  } else {
    e = set_max_smem_once(reinterpret_cast<const void*>(decode_kernel<2, 1, false>), Smem<2, 8>::kTotal);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<2, 1, false>, kThreads, Smem<2, 8>::kTotal);
  }
  if (e != cudaSuccess || n <= 0) return 1;
  if (dev >= 0) cache[dev][v].store(n, std::memory_order_relaxed);
  return n;
}

// Atoms per split granule: runs start at group boundaries (a group's atoms,
// 8 for groups of 8 atoms or more) or anywhere with one group per column.
int split_granule(int apg_t, int gshift) { return gshift == 30 ? 1 : apg_t; }

// Split granules of a problem (the most CTAs a launch can use); 0 if the
// group size is not supported by the decode kernel.
long decode_units(int N, int K, int group) {
  int apg_t, gshift;
  if (!group_shape(K, group, &apg_t, &gshift)) return 0;
  const long natoms = K / kAtomK;
  return (long)((N + kDecodeBlockCols - 1) / kDecodeBlockCols) * natoms / split_granule(apg_t, gshift);
}

// The flag area has room for the most CTAs a launch may have (8192), whatever
// this call's shape: a workspace can then serve calls of any shape in turn.
size_t decode_counter_bytes(int N) {
  (void)N;
  return (size_t)kDecodeMaxCtas * sizeof(int);
}

// Flags, then one fp32 partial tile (M rows padded to 8 or 16 x 128 columns)
// per CTA.
size_t decode_workspace_bytes(int M, int N, int ctas) {
  const int mt = M <= 8 ? 1 : 2;
  const size_t tile_bytes = (size_t)mt * 8 * kDecodeBlockCols * sizeof(float);
  return decode_counter_bytes(N) + (size_t)ctas * tile_bytes;
}

cudaError_t launch_decode(const uint16_t* A, const uint32_t* Wq, const uint16_t* Sp,
                          const uint32_t* Zp, uint16_t* Y, int M, int N, int K, int group,
                          int ctas, void* workspace, bool early_weights, bool bf16,
                          const float* row_scale, cudaStream_t stream) {
  DecodeArgs args = {};
  args.row_scale = row_scale;
  int apg_t = 0;
  if (!group_shape(K, group, &apg_t, &args.gshift)) return cudaErrorInvalidValue;
  args.A = A;
  args.Wq = reinterpret_cast<const uint4*>(Wq);
  args.Sp2 = reinterpret_cast<const uint32_t*>(Sp);
  args.Zp = reinterpret_cast<const uint8_t*>(Zp);
  args.Y = Y;
  args.flags = static_cast<int*>(workspace);
  args.tiles = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + decode_counter_bytes(N));
  args.tile_floats = (decode_workspace_bytes(M, N, ctas) - decode_counter_bytes(N)) / sizeof(float);
  args.granule = split_granule(apg_t, args.gshift);
  cudaError_t e = device_error_word(&args.err);
  if (e != cudaSuccess) return e;
  args.M = M;
  args.N = N;
  args.K = K;
  args.early_weights = early_weights ? 1 : 0;
  const int mt = M <= 8 ? 1 : 2;
  return bf16 ? decode_dispatch_streamk_bf16(args, mt, apg_t, ctas, stream)
              : dispatch_streamk<false>(args, mt, apg_t, ctas, stream);
}

namespace {

// The resident variant's shape for a launch: 8 warps and two CTAs per SM
// (113 KiB each) or 16 warps and one CTA per SM (227 KiB; the same warps per
// SM, the activations staged once per SM). Measured on the Llama shapes, 16
// warps are faster from 4 rows up and 8 warps below, so that order is tried
// first. `requested` CTAs, else one per resident slot, clamped to the strips
// and to 8192. With `automatic`, staged activations above 160 KiB count as
// not fitting unless the strips spread over the CTAs at least 90% evenly
// (S / (C ceil(S / C))): measured, the stream-K variant was faster at 8 rows
// of K = 11008 over 256 strips (84%) and 16 rows of K = 5120 over 320 strips
// (70%), slower at 16 rows of K = 5120 over 960 and 1728 strips (90%, 95%).
// Returns the CTA count (0: no fit) and sets the warps per CTA.
int resident_shape(int M, int N, int K, int gshift, int requested, int sms, bool automatic,
                   bool silu, int* nw, DecodeArgs* args, int* bytes) {
  // units of work: strips, or with the fused gate/up epilogue strip pairs
  const int units = silu ? N / kStripCols / 2 : N / kStripCols;
  const long act_bytes = (M + 1L) * (2L * K + 64);
  for (int i = 0; i < 2; ++i) {
    const int w = (M >= 4) == (i == 0) ? 16 : 8;
    long c = requested > 0 ? requested : (w == 8 ? 2L : 1L) * sms;
    if (c > units) c = units;
    if (c > kDecodeMaxCtas) c = kDecodeMaxCtas;
    if (c >= 1 && strip_layout(M, N, K, gshift, (int)c, w, w == 8 ? kTwoCtaSmem : kOneCtaSmem, silu,
                               args, bytes)) {
      if (automatic && act_bytes > 160L * 1024) {
        const long most = (units + c - 1) / c;  // units of the busiest CTA
        if (10L * units < 9L * c * most) return 0;
      }
      *nw = w;
      return (int)c;
    }
  }
  return 0;
}

}  // namespace

int decode_resident_ctas(int M, int N, int K, int group, int requested, int sms, bool automatic,
                         bool silu) {
  int apg_t = 0, gshift = 0, nw = 0, bytes = 0;
  if (M < 1 || M > 16 || !group_shape(K, group, &apg_t, &gshift)) return 0;
  if (silu && (N / kStripCols) % 2 != 0) return 0;
  DecodeArgs args;
  return resident_shape(M, N, K, gshift, requested, sms, automatic, silu, &nw, &args, &bytes);
}

namespace {

__device__ int g_selftest_flag;  // never set: the self-test waits on it

// Self-test of the stream-K fix-up's bounded wait: one thread waits, with
// the kernel's own routine and limit, for a flag that nothing sets; the wait
// gives up, the thread records kDecodeWaitTimedOut in the error word and the
// kernel returns.
__global__ void selftest_flag_kernel(int* err) {
  if (threadIdx.x == 0 && !wait_flag(&g_selftest_flag)) atomicOr(err, kDecodeWaitTimedOut);
}

}  // namespace

cudaError_t launch_selftest_flag_wait(cudaStream_t stream) {
  int* err = nullptr;
  cudaError_t e = device_error_word(&err);
  if (e != cudaSuccess) return e;
  selftest_flag_kernel<<<1, 32, 0, stream>>>(err);
  return cudaGetLastError();
}

cudaError_t launch_decode_resident(const uint16_t* A, const uint32_t* Wq, const uint16_t* Sp,
                                   const uint32_t* Zp, uint16_t* Y, int M, int N, int K, int group,
                                   int ctas, int sms, bool automatic, bool silu,
                                   bool early_weights, bool bf16, const float* row_scale,
                                   cudaStream_t stream) {
  DecodeArgs args = {};
  int apg_t = 0, bytes = 0, nw = 0;
  if (!group_shape(K, group, &apg_t, &args.gshift)) return cudaErrorInvalidValue;
  if (silu && (N / kStripCols) % 2 != 0) return cudaErrorInvalidValue;
  if (ctas < 1 ||
      resident_shape(M, N, K, args.gshift, ctas, sms, automatic, silu, &nw, &args, &bytes) != ctas)
    return cudaErrorInvalidValue;
  args.A = A;
  args.Wq = reinterpret_cast<const uint4*>(Wq);
  args.Sp2 = reinterpret_cast<const uint32_t*>(Sp);
  args.Zp = reinterpret_cast<const uint8_t*>(Zp);
  args.Y = Y;
  args.granule = split_granule(apg_t, args.gshift);
  args.M = M;
  args.N = N;
  args.K = K;
  args.early_weights = early_weights ? 1 : 0;
  args.row_scale = row_scale;
  const int mt = M <= 8 ? 1 : 2;
  return bf16 ? decode_dispatch_resident_bf16(args, mt, nw, apg_t, ctas, bytes, stream)
              : dispatch_resident<false>(args, mt, nw, apg_t, ctas, bytes, stream);
}

}  // namespace w4a16
