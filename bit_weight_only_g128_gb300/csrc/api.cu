// C ABI of the W4A16 library: argument checks, path choice, launches.
// Declarations and the contract of every entry point: include/w4a16.h.
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

thread_local std::string t_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return code;
}

int ok() {
  t_last_error.clear();
  return W4A16_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(W4A16_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int kMaxDim = 1 << 20;

// Shape rules shared by every entry point that takes K, N, group.
int check_kn(int K, int N, int group) {
  if (K <= 0 || N <= 0 || group <= 0)
    return fail(W4A16_ERR_INVALID_ARG, "K=%d, N=%d, group=%d must be positive", K, N, group);
  if (K > kMaxDim || N > kMaxDim)
    return fail(W4A16_ERR_UNSUPPORTED_SHAPE, "K=%d or N=%d above %d", K, N, kMaxDim);
  if (N % kStripCols)
    return fail(W4A16_ERR_UNSUPPORTED_SHAPE, "N=%d is not a multiple of 16", N);
  if (K % kAtomK) return fail(W4A16_ERR_UNSUPPORTED_SHAPE, "K=%d is not a multiple of 64", K);
  if (group % kAtomK)
    return fail(W4A16_ERR_UNSUPPORTED_SHAPE, "group=%d is not a multiple of 64", group);
  if (K % group) return fail(W4A16_ERR_UNSUPPORTED_SHAPE, "group=%d does not divide K=%d", group, K);
  return W4A16_OK;
}

// SM count of the current device (cached per device; 148 if unknown).
int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return 148;
  if (dev < 64) cache[dev] = sms;
  return sms;
}

// Persistent CTAs of the decode kernel: every resident slot of the device,
// but never more than the work units (each CTA must own at least one).
int decode_ctas(int M, int N, int K, int group, int requested) {
  const long T = decode_units(N, K, group);
  if (T <= 0) return 0;
  long c = requested > 0 ? requested : (long)sm_count() * decode_ctas_per_sm(M);
  if (c > T) c = T;
  if (c > kDecodeMaxCtas) c = kDecodeMaxCtas;
  return (int)c;
}

// The path for M rows, from measurements on GB300 (CUDA graphs of 20 launches
// over weight copies larger than L2; the full tables are kept with the design
// notes).
// Decode GEMV up to 16 rows; on wide layers (N >= 16384) of at most 2^28
// weights up to 24 rows (two 16-row passes over the weights) (us, decode /
// one-SM tensor cores):
//   7B gate_up (4096 x 22016):  16 rows 16.3 / 27.3, 24 rows 26.8 / 28.0, 32 rows 32.2 / 28.1
//   13B gate_up (5120 x 27648): 16 rows 22.7 / 40.7, 24 rows 38.2 / 39.7, 32 rows 44.7 / 39.4
//   70B gate_up (8192 x 57344): 16 rows 77.9 / 110.0, 20 rows 116.1 / 108.6
//   13B o_proj (5120 x 5120):   16 rows 11.7 / 11.8, 20 rows 18.6 / 12.1
// Above, the tensor cores: a CTA pair per 256-column tile (tcgen05.mma
// cta_group::2) from 256 rows where the pairs' CTAs make at least 80 (they
// have no K split), else one SM per tile (TFLOP/s, one SM / pair):
//   256 rows: 70B gate_up 1629 / 1775, 70B qkv 898 / 1003, 70B o_proj 1068 / 818
//   512 rows: 70B down 1476 / 1724, 13B o_proj 888 / 893, 7B o_proj 775 / 710
//   4096 rows: 70B gate_up 1452 / 1583, 7B o_proj 1275 / 1398, 7B qkv 1390 / 1545
//   128 rows: 13B qkv 778 / 680, 70B qkv 587 / 513, 7B qkv 488 / 530
// and, on wide layers of at most 2^28 weights, from 65 to 128 rows (us, one
// SM / pair): 7B gate_up 80 rows 45.4 / 41.6, 128 rows 47.7 / 41.8; 13B
// gate_up 80 rows 53.2 / 51.1, 128 rows 55.7 / 51.2; 70B gate_up (above 2^28)
// 128 rows 114.0 / 118.3; 13B qkv (narrower) 128 rows 25.7 / 29.4; and on
// wide layers from 193 to 255 rows: 7B gate_up 208 rows 48.6 / 44.5, 13B
// gate_up 224 rows 60.0 / 54.6, 70B gate_up 240 rows 147.7 / 137.6
int choose_path(int M, int N, int K, int group) {
  const long long nk = (long long)N * K;
  // (group sizes the decode kernel does not take go to the tensor cores)
  const bool wide = N >= 16384;
  if ((M <= 16 || (wide && M <= 24 && nk <= (1LL << 28))) &&
      decode_units(N, K, group) > 0)
    return W4A16_PATH_DECODE;
  const long long pair_ctas = 2LL * ((N + 255) / 256) * ((M + 255) / 256);
  if (M >= 256 && pair_ctas >= 80) return W4A16_PATH_TENSOR_PAIR;
  // wide layers of at most 2^28 weights at 65-128 rows: pairs of 128-token tiles
  if (M > 64 && M <= 128 && wide && nk <= (1LL << 28)) return W4A16_PATH_TENSOR_PAIR;
  // wide layers at 193-255 rows, where the one-SM kernel's 208-256-token
  // tiles leave room for two dequant groups only
  if (M > 192 && M < 256 && wide) return W4A16_PATH_TENSOR_PAIR;
  return W4A16_PATH_TENSOR;
}

bool is_tensor(int path) { return path == W4A16_PATH_TENSOR || path == W4A16_PATH_TENSOR_PAIR; }

bool is_decode(int path) {
  return path == W4A16_PATH_DECODE || path == W4A16_PATH_DECODE_RESIDENT ||
         path == W4A16_PATH_DECODE_STREAMK;
}

// The decode variant for one launch of `rows` rows: activations resident in
// shared memory when they fit (with the CTA count `parts` asks for), else
// stream-K. Returns the variant and its CTA count.
int decode_variant(int path, int rows, int N, int K, int group, int parts, bool silu, int* ctas) {
  if (path != W4A16_PATH_DECODE_STREAMK) {
    const int c = decode_resident_ctas(rows, N, K, group, parts, sm_count(),
                                       path == W4A16_PATH_DECODE, silu);
    if (c > 0 || path == W4A16_PATH_DECODE_RESIDENT) {
      *ctas = c;
      return W4A16_PATH_DECODE_RESIDENT;
    }
  }
  *ctas = decode_ctas(rows, N, K, group, parts);
  return W4A16_PATH_DECODE_STREAMK;
}

// Scratch bytes of a (path, parts) choice: the decode path's counters and
// partial tiles (16-row chunks share one workspace); none for tensor cores.
// K split of the tensor-core path (requested, else chosen from the tiles).
int tc_split(int M, int N, int K, int group, int requested) {
  const int nk = K / (kAtomK * tc_stage_atoms(M, K, group));  // pipeline stages
  int s = requested > 0 ? requested : tc_choose_split(M, N, K, group, sm_count());
  if (s > nk) s = nk;
  return s < 1 ? 1 : s;
}

// Workspace of a call: the path's own scratch first (the decode path's size
// covers either variant, so that it does not depend on which one a device
// picks; the resident one uses none). Then, never inside the 32 KiB
// flag/counter area that every call must leave zero-filled (a launch without
// a K split has no scratch of its own, but a later call may use the area),
// each at a 256-byte boundary:
//   - with the fused gate/up epilogue on a path that does not fuse it
//     (stream-K, tensor cores), the fp16 product of the rows of one launch
//     ([rows][N]; all M rows for tensor cores, 16 for the decode path);
//   - with W4A8, the activations' codes as 16-bit integer values [M][K] and
//     their per-row scales [M] (fp32).
constexpr size_t kFlagAreaBytes = 32768;
size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }
size_t product_offset(size_t base) { return align256(base > kFlagAreaBytes ? base : kFlagAreaBytes); }

struct WsLayout {
  size_t base;    // the path's own scratch
  size_t prod;    // fused epilogue's product (0: none)
  size_t codes;   // W4A8 codes (0: none)
  size_t scales;  // W4A8 row scales
  size_t total;
};

WsLayout ws_layout(int M, int N, int K, int group, int path, bool silu, bool a8, int parts) {
  WsLayout l = {0, 0, 0, 0, 0};
  if (M == 0) return l;
  int prod_rows = 0;
  if (path == W4A16_PATH_TENSOR) {
    l.base = tc_workspace_bytes(M, N, tc_split(M, N, K, group, parts));
    prod_rows = M;
  } else if (path == W4A16_PATH_TENSOR_PAIR) {
    prod_rows = M;  // no K split: no scratch of its own
  } else if (is_decode(path) && path != W4A16_PATH_DECODE_RESIDENT) {
    const int rows = M < 16 ? M : 16;
    const int c = decode_ctas(rows, N, K, group, parts);
    l.base = c > 0 ? decode_workspace_bytes(rows, N, c) : 0;
    prod_rows = rows;
  }
  size_t end = l.base;
  if (silu && prod_rows > 0) {
    l.prod = product_offset(end);
    end = l.prod + (size_t)prod_rows * N * 2;
  }
  if (a8) {
    l.codes = product_offset(end);
    l.scales = align256(l.codes + (size_t)M * K * 2);
    end = l.scales + (size_t)M * sizeof(float);
  }
  l.total = end;
  return l;
}

size_t workspace_for(int M, int N, int K, int group, int path, int parts, bool silu, bool a8 = false) {
  return ws_layout(M, N, K, group, path, silu, a8, parts).total;
}

int gemm_impl(const uint16_t* A, const uint32_t* Wq, const uint16_t* scales,
              const uint32_t* zeros, int M, int N, int K, int group, uint16_t* Y,
              void* workspace, size_t workspace_bytes, int path, int parts,
              cudaStream_t stream) {
  if (M < 0) return fail(W4A16_ERR_INVALID_ARG, "M=%d is negative", M);
  if (M > kMaxDim) return fail(W4A16_ERR_UNSUPPORTED_SHAPE, "M=%d above %d", M, kMaxDim);
  if (int rc = check_kn(K, N, group)) return rc;
  if (M == 0) return ok();
  if (!A || !Wq || !scales || !zeros || !Y)
    return fail(W4A16_ERR_INVALID_ARG, "null pointer (A=%p Wq=%p scales=%p zeros=%p Y=%p)", A, Wq,
                scales, zeros, Y);
  if (!aligned(A, 16) || !aligned(Wq, 16) || !aligned(scales, 16) || !aligned(Y, 16) ||
      !aligned(zeros, 8))
    return fail(W4A16_ERR_MISALIGNED,
                "alignment: A, Wq, scales, Y need 16 bytes and zeros 8 bytes");
  const bool static_weights = (path & W4A16_STATIC_WEIGHTS) != 0;
  const bool silu = (path & W4A16_SILU_MUL) != 0;
  const bool bf16 = (path & W4A16_BF16) != 0;
  const bool a8 = (path & W4A16_ACT_A8) != 0;
  path &= ~(W4A16_STATIC_WEIGHTS | W4A16_SILU_MUL | W4A16_BF16 | W4A16_ACT_A8);
  if (path == W4A16_PATH_AUTO) path = choose_path(M, N, K, group);
  if (!is_decode(path) && !is_tensor(path))
    return fail(W4A16_ERR_INVALID_ARG, "unknown path %d", path);
  if (parts < 0) return fail(W4A16_ERR_INVALID_ARG, "parts=%d is negative", parts);
  if (a8 && K > 65536)
    return fail(W4A16_ERR_UNSUPPORTED_SHAPE, "W4A8: K=%d above 65536 (a row must fit shared memory)", K);
  // W4A8: quantize the activations into the workspace, then multiply the
  // codes and scale each row of the result (launched once the workspace is
  // checked, below)
  const float* row_scale = nullptr;
  auto quantize_activations = [&](const WsLayout& l) -> cudaError_t {
    uint16_t* codes = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + l.codes);
    float* sc = reinterpret_cast<float*>(static_cast<char*>(workspace) + l.scales);
    cudaError_t e = launch_quantize_act(A, M, K, bf16, nullptr, codes, bf16, sc, stream);
    A = codes;
    row_scale = sc;
    return e;
  };
  if (silu && N % 32 != 0)
    return fail(W4A16_ERR_UNSUPPORTED_SHAPE,
                "fused gate/up epilogue: N=%d is not two halves of 16-column strips "
                "(a multiple of 32)", N);
  const int ycols = silu ? N / 2 : N;  // columns of Y
  if (is_tensor(path)) {
    const bool pair = path == W4A16_PATH_TENSOR_PAIR;
    const int split = pair ? 1 : tc_split(M, N, K, group, parts);
    const WsLayout l = ws_layout(M, N, K, group, path, silu, a8, parts);
    const size_t need = l.total;
    if (need > 0 && (!workspace || workspace_bytes < need))
      return fail(W4A16_ERR_WORKSPACE_TOO_SMALL,
                  "tensor-core path (K split %d) needs a workspace of %zu bytes (got %zu)", split,
                  need, workspace ? workspace_bytes : (size_t)0);
    if (need > 0 && !aligned(workspace, 256))
      return fail(W4A16_ERR_MISALIGNED, "workspace needs 256-byte alignment");
    cudaError_t e = a8 ? quantize_activations(l) : cudaSuccess;
    if (e != cudaSuccess) return cuda_fail(e, "activation quantization launch");
    // with the fused epilogue the product goes to the workspace first
    uint16_t* prod = silu ? reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + l.prod) : Y;
    e = pair ? launch_tc_pair(A, Wq, scales, zeros, prod, M, N, K, group, static_weights, bf16,
                              row_scale, stream)
             : launch_tc_gemm(A, Wq, scales, zeros, prod, M, N, K, group, split,
                              l.base > 0 ? workspace : nullptr, static_weights, bf16, row_scale,
                              stream);
    if (e != cudaSuccess) return cuda_fail(e, "tensor-core kernel launch");
    if (silu && (e = launch_silu_mul(prod, M, N, Y, bf16, stream)) != cudaSuccess)
      return cuda_fail(e, "gate/up epilogue launch");
    return ok();
  }
  if (decode_units(N, K, group) <= 0)
    return fail(W4A16_ERR_UNSUPPORTED_SHAPE,
                "decode path: group=%d must be K or 64 times a power of two", group);
  // 16 rows per launch; larger M re-streams the weights once per 16 rows
  int ctas = 0;
  for (int r0 = 0; r0 < M; r0 += 16) {
    const int rows = M - r0 < 16 ? M - r0 : 16;
    if (decode_variant(path, rows, N, K, group, parts, silu, &ctas) ==
            W4A16_PATH_DECODE_RESIDENT &&
        ctas == 0)
      return fail(W4A16_ERR_UNSUPPORTED_SHAPE,
                  "resident decode variant: %d rows of K=%d (with the strips of N=%d over %d "
                  "CTAs) do not fit a CTA's shared memory",
                  rows, K, N, parts > 0 ? parts : 2 * sm_count());
  }
  const WsLayout l = ws_layout(M, N, K, group, path, silu, a8, parts);
  const size_t need = l.total;
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(W4A16_ERR_WORKSPACE_TOO_SMALL, "decode path needs a workspace of %zu bytes (got %zu)",
                need, workspace ? workspace_bytes : (size_t)0);
  if (need > 0 && !aligned(workspace, 256))
    return fail(W4A16_ERR_MISALIGNED, "workspace needs 256-byte alignment");
  if (a8) {
    cudaError_t e = quantize_activations(l);
    if (e != cudaSuccess) return cuda_fail(e, "activation quantization launch");
  }
  // the stream-K variant's product, with the fused epilogue, before silu * up
  uint16_t* prod = l.prod ? reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + l.prod) : nullptr;
  for (int r0 = 0; r0 < M; r0 += 16) {
    const int rows = M - r0 < 16 ? M - r0 : 16;
    const uint16_t* Ar = A + (size_t)r0 * K;
    uint16_t* Yr = Y + (size_t)r0 * ycols;
    const float* rs = row_scale ? row_scale + r0 : nullptr;
    cudaError_t e;
    if (decode_variant(path, rows, N, K, group, parts, silu, &ctas) == W4A16_PATH_DECODE_RESIDENT) {
      e = launch_decode_resident(Ar, Wq, scales, zeros, Yr, rows, N, K, group, ctas, sm_count(),
                                 path == W4A16_PATH_DECODE, silu, static_weights, bf16, rs, stream);
    } else {
      e = launch_decode(Ar, Wq, scales, zeros, silu ? prod : Yr, rows, N, K, group, ctas, workspace,
                        static_weights, bf16, rs, stream);
      if (e == cudaSuccess && silu) e = launch_silu_mul(prod, rows, N, Yr, bf16, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
  }
  return ok();
}

}  // namespace

cudaError_t set_max_smem_once(const void* kernel, int bytes) {
  struct Entry {
    const void* kernel;
    int device, bytes;
  };
  static std::mutex mu;
  static std::vector<Entry> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& d : done)
    if (d.kernel == kernel && d.device == dev && d.bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.push_back({kernel, dev, bytes});
  return e;
}

// Record an error (or success) for w4a16_last_error from other translation
// units of the library.
int report_error(int code, const char* message) { return fail(code, "%s", message); }
int report_ok() { return ok(); }

}  // namespace w4a16

using namespace w4a16;

extern "C" {

const char* w4a16_last_error(void) { return t_last_error.c_str(); }

int w4a16_version(void) { return 100; }

int w4a16_packed_sizes(int K, int N, int group, size_t* wq_bytes, size_t* sp_bytes,
                       size_t* zp_bytes) {
  if (int rc = check_kn(K, N, group)) return rc;
  if (!wq_bytes || !sp_bytes || !zp_bytes) return fail(W4A16_ERR_INVALID_ARG, "null output pointer");
  const size_t G = (size_t)(K / group);
  *wq_bytes = (size_t)K * N / 2;
  *sp_bytes = 2 * G * N;
  *zp_bytes = G * N / 2;
  return ok();
}

int w4a16_quantize(const float* W, int K, int N, int group, uint8_t* q, uint16_t* s, uint8_t* z,
                   void* stream) {
  if (int rc = check_kn(K, N, group)) return rc;
  if (!W || !q || !s || !z) return fail(W4A16_ERR_INVALID_ARG, "null pointer");
  cudaError_t e = launch_quantize(W, K, N, group, q, s, z, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "quantize kernel launch");
  return ok();
}

int w4a16_pack(const uint8_t* q, const uint16_t* s, const uint8_t* z, int K, int N, int group,
               uint32_t* Wq, uint16_t* Sp, uint32_t* Zp, void* stream) {
  if (int rc = check_kn(K, N, group)) return rc;
  if (!q || !s || !z || !Wq || !Sp || !Zp) return fail(W4A16_ERR_INVALID_ARG, "null pointer");
  if (!aligned(Wq, 16) || !aligned(Sp, 16) || !aligned(Zp, 8))
    return fail(W4A16_ERR_MISALIGNED, "alignment: Wq, Sp need 16 bytes and Zp 8 bytes");
  cudaError_t e = launch_pack(q, s, z, K, N, group, Wq, Sp, Zp, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "pack kernel launch");
  return ok();
}

int w4a16_unpack(const uint32_t* Wq, const uint16_t* Sp, const uint32_t* Zp, int K, int N,
                 int group, uint8_t* q, uint16_t* s, uint8_t* z, void* stream) {
  if (int rc = check_kn(K, N, group)) return rc;
  if (!q || !s || !z || !Wq || !Sp || !Zp) return fail(W4A16_ERR_INVALID_ARG, "null pointer");
  cudaError_t e = launch_unpack(Wq, Sp, Zp, K, N, group, q, s, z, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "unpack kernel launch");
  return ok();
}

int w4a16_dequantize(const uint32_t* Wq, const uint16_t* Sp, const uint32_t* Zp, int K, int N,
                     int group, uint16_t* deq, void* stream) {
  if (int rc = check_kn(K, N, group)) return rc;
  if (!Wq || !Sp || !Zp || !deq) return fail(W4A16_ERR_INVALID_ARG, "null pointer");
  cudaError_t e = launch_dequantize(Wq, Sp, Zp, K, N, group, deq, false, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "dequantize kernel launch");
  return ok();
}

int w4a16_quantize_act(const uint16_t* A, int M, int K, int flags, int8_t* aq, float* s_a,
                       void* stream) {
  if (M < 0 || K < 0) return fail(W4A16_ERR_INVALID_ARG, "M=%d, K=%d: negative", M, K);
  if (flags & ~W4A16_BF16) return fail(W4A16_ERR_INVALID_ARG, "flags=0x%x: only W4A16_BF16", flags);
  if (K % 8 != 0 || K > 65536)
    return fail(W4A16_ERR_UNSUPPORTED_SHAPE, "K=%d is not a multiple of 8 up to 65536", K);
  if (M == 0) return ok();
  if (!A || !aq || !s_a) return fail(W4A16_ERR_INVALID_ARG, "null pointer");
  if (!aligned(A, 16) || !aligned(aq, 16) || !aligned(s_a, 4))
    return fail(W4A16_ERR_MISALIGNED, "alignment: A and aq need 16 bytes, s_a 4");
  cudaError_t e = launch_quantize_act(A, M, K, (flags & W4A16_BF16) != 0, aq, nullptr, false, s_a,
                                      (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "activation quantization launch");
  return ok();
}

int w4a16_dequantize_bf16(const uint32_t* Wq, const uint16_t* Sp, const uint32_t* Zp, int K, int N,
                          int group, uint16_t* deq, void* stream) {
  if (int rc = check_kn(K, N, group)) return rc;
  if (!Wq || !Sp || !Zp || !deq) return fail(W4A16_ERR_INVALID_ARG, "null pointer");
  cudaError_t e = launch_dequantize(Wq, Sp, Zp, K, N, group, deq, true, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "dequantize kernel launch");
  return ok();
}

int w4a16_workspace_size(int M, int N, int K, int group, size_t* bytes) {
  return w4a16_workspace_size_ex(M, N, K, group, W4A16_PATH_AUTO, 0, bytes);
}

int w4a16_workspace_size_ex(int M, int N, int K, int group, int path, int parts, size_t* bytes) {
  if (M < 0) return fail(W4A16_ERR_INVALID_ARG, "M=%d is negative", M);
  if (parts < 0) return fail(W4A16_ERR_INVALID_ARG, "parts=%d is negative", parts);
  if (int rc = check_kn(K, N, group)) return rc;
  if (!bytes) return fail(W4A16_ERR_INVALID_ARG, "null output pointer");
  const bool silu = (path & W4A16_SILU_MUL) != 0;
  const bool a8 = (path & W4A16_ACT_A8) != 0;
  path &= ~(W4A16_STATIC_WEIGHTS | W4A16_SILU_MUL | W4A16_BF16 | W4A16_ACT_A8);
  if (path == W4A16_PATH_AUTO) path = choose_path(M, N, K, group);
  if (!is_decode(path) && !is_tensor(path))
    return fail(W4A16_ERR_INVALID_ARG, "unknown path %d", path);
  if (silu && N % 32 != 0)
    return fail(W4A16_ERR_UNSUPPORTED_SHAPE, "fused gate/up epilogue: N=%d is not a multiple of 32", N);
  *bytes = workspace_for(M, N, K, group, path, parts, silu, a8);
  return ok();
}

int w4a16_gemm(const uint16_t* A, const uint32_t* Wq, const uint16_t* scales, const uint32_t* zeros,
               int M, int N, int K, int group, uint16_t* Y, void* workspace,
               size_t workspace_bytes, void* stream) {
  return gemm_impl(A, Wq, scales, zeros, M, N, K, group, Y, workspace, workspace_bytes,
                   W4A16_PATH_AUTO, 0, (cudaStream_t)stream);
}

int w4a16_gemm_ex(const uint16_t* A, const uint32_t* Wq, const uint16_t* scales,
                  const uint32_t* zeros, int M, int N, int K, int group, uint16_t* Y,
                  void* workspace, size_t workspace_bytes, int path, int parts, void* stream) {
  return gemm_impl(A, Wq, scales, zeros, M, N, K, group, Y, workspace, workspace_bytes, path,
                   parts, (cudaStream_t)stream);
}

int w4a16_plan(int M, int N, int K, int group, int* path, int* parts) {
  if (M < 0) return fail(W4A16_ERR_INVALID_ARG, "M=%d is negative", M);
  if (int rc = check_kn(K, N, group)) return rc;
  if (!path || !parts) return fail(W4A16_ERR_INVALID_ARG, "null output pointer");
  *path = choose_path(M, N, K, group);
  const int rows = M < 16 ? (M > 0 ? M : 1) : 16;
  if (*path == W4A16_PATH_DECODE)
    *path = decode_variant(W4A16_PATH_DECODE, rows, N, K, group, 0, false, parts);
  else if (*path == W4A16_PATH_TENSOR_PAIR)
    *parts = 1;
  else
    *parts = tc_split(M, N, K, group, 0);
  return ok();
}

int w4a16_tc_config(int M, int K, int group, int* out, int n) {
  if (M < 1) return fail(W4A16_ERR_INVALID_ARG, "M=%d must be positive", M);
  if (!out || n < 8) return fail(W4A16_ERR_INVALID_ARG, "out must hold 8 values (n=%d)", n);
  if (int rc = check_kn(K, 16, group)) return rc;
  int cfg[15];
  if (!tc_config(M, K, group, cfg))
    return fail(W4A16_ERR_UNSUPPORTED_SHAPE, "no valid tensor-core configuration for M=%d K=%d", M, K);
  if (n >= 15 && !tc_pair_config(M, K, group, cfg + 8))
    return fail(W4A16_ERR_UNSUPPORTED_SHAPE, "no valid CTA-pair configuration for M=%d K=%d", M, K);
  for (int i = 0; i < (n >= 15 ? 15 : 8); ++i) out[i] = cfg[i];
  return ok();
}

int w4a16_selftest_wait(int which, void* stream) {
  cudaError_t e;
  if (which == 0)
    e = launch_selftest_flag_wait((cudaStream_t)stream);
  else if (which == 1)
    e = launch_selftest_mbar_wait((cudaStream_t)stream);
  else
    return fail(W4A16_ERR_INVALID_ARG, "which=%d: 0 (flag wait) or 1 (mbarrier wait)", which);
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return ok();
}

int w4a16_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int flag = 0;
  e = read_and_clear_device_error(&flag);
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  if (flag != 0)
    return fail(W4A16_ERR_DEVICE_CHECK,
                "device error word = 0x%x (bits: 1 producer, 2 MMA, 4 dequant, 8 epilogue waits "
                "timed out; 16 drain timed out; 32 decode fix-up wait timed out; 64 access out of "
                "bounds, bounds-checked build)",
                flag);
  return ok();
}

}  // extern "C"
