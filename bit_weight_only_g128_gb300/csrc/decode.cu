// Decode path of the W4A16 linear layer: M <= 16 rows of activations, where
// the layer is bound by streaming the packed weights from HBM (vLLM PR #1032
// thread: the AWQ kernel is "fastest below batch size 8"; the same thread
// calls dequantization "the most tricky part ... the rest is normal FP16
// operations").
//
// Design (sm_103a):
//   * One warp owns one 16-column strip and a contiguous range of 64-k atoms.
//     Each lane streams its four words of an atom with one 16-byte load
//     (L1 bypassed); U atoms are kept in flight per warp, refilled as they are
//     consumed.
//   * Dequantization happens in registers (LOP3 + exact fp16 subtract + one
//     fp16 multiply per pair of codes) and feeds mma.sync m16n8k16 with the
//     weights as the 16-row operand (output columns) and up to 8 tokens as the
//     8-column operand. k inside each MMA is permuted identically on both
//     operands (a lane holds 4 consecutive k), which the sum is invariant to.
//   * A CTA is 8 warps = 128 columns over one K range; `split` CTAs of a
//     thread-block cluster cover the K ranges of the same columns, and their
//     fp32 partials are summed in a fixed order through distributed shared
//     memory (deterministic, no global scratch).
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace w4a16 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRedStride = kDecodeBlockCols + 4;  // padded row of the partial tile
constexpr int kPrefetch = 8;                      // weight atoms in flight per warp

// Activation atoms staged per chunk (1024 or 2048 k), and the bytes of one
// staged row. The extra 64 bytes put consecutive rows in opposite halves of
// the 32 banks, so the 16-byte fragment loads of a quarter-warp (two rows x
// 64 bytes) never collide.
template <int MT>
__host__ __device__ constexpr int chunk_atoms() { return MT == 1 ? 32 : 16; }
template <int MT>
__host__ __device__ constexpr int act_row_bytes() { return chunk_atoms<MT>() * kAtomK * 2 + 64; }
template <int MT>
__host__ __device__ constexpr int act_buffer_bytes() { return MT * 8 * act_row_bytes<MT>(); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Copy the activations of atoms [a0, a1) (rows 0..M-1) into a chunk buffer.
template <int MT>
__device__ __forceinline__ void stage_activations(uint32_t buf, const uint16_t* __restrict__ A,
                                                  int M, int K, int a0, int a1) {
  const int units = (a1 - a0) * (kAtomK / 8);  // 16-byte units per row
  for (int idx = threadIdx.x; idx < M * units; idx += kThreads) {
    const int row = idx / units, u = idx % units;
    cp_async16(buf + row * act_row_bytes<MT>() + u * 16,
               A + (size_t)row * K + (size_t)a0 * kAtomK + u * 8);
  }
}

// MT: token octets (1: M <= 8, 2: M <= 16).
template <int MT>
__global__ void __launch_bounds__(kThreads, 2)
decode_kernel(const uint16_t* __restrict__ A, const uint4* __restrict__ Wq,
              const uint32_t* __restrict__ Sp2, const uint2* __restrict__ Zp,
              uint16_t* __restrict__ Y, int M, int N, int K, int group, int split) {
  constexpr int U = kPrefetch;
  constexpr int CH = chunk_atoms<MT>();
  constexpr int kRow = act_row_bytes<MT>();
  constexpr int kBuf = act_buffer_bytes<MT>();
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, t = lane & 3;  // mma groupID / thread-in-group
  const int nstrips = N / kStripCols;
  const int strip = blockIdx.y * kWarps + warp;
  const bool active = strip < nstrips;
  const int natoms = K / kAtomK;
  const int a_begin = (int)(((long long)blockIdx.x * natoms) / split);
  const int a_end = (int)(((long long)(blockIdx.x + 1) * natoms) / split);
  const int G = K / group;
  const int apg = group / kAtomK;  // atoms per group

  const uint4* wp = Wq + (size_t)(active ? strip : 0) * natoms * 32 + lane;
  const uint32_t* sp = Sp2 + (size_t)(active ? strip : 0) * G * 8 + gq;  // (s[gq], s[gq+8])
  const uint2* zp = Zp + (size_t)(active ? strip : 0) * G;

  // Slot u holds the atom a with (a - a_begin) % U == u: its weights, and the
  // scale pair / zero words of its group when it is the first atom of a group
  // (or of the range). The load stream runs U atoms ahead of consumption.
  uint4 w[U];
  uint32_t ms[U];
  uint2 mz[U];
  int l_atom = a_begin, l_grp = a_begin / apg, l_rem = a_begin % apg;
  if (active) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (l_atom < a_end) {
        w[u] = ldg_stream(wp + (size_t)l_atom * 32);
        if (u == 0 || l_rem == 0) {
          ms[u] = __ldg(sp + (size_t)l_grp * 8);
          mz[u] = __ldg(zp + l_grp);
        }
        ++l_atom;
        if (++l_rem == apg) { l_rem = 0; ++l_grp; }
      }
    }
  }
  int c_rem = a_begin % apg;  // position of the consumed atom inside its group
  DeqConst d0 = {}, d1 = {};

  float acc[2][MT][4];
#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int o = 0; o < MT; ++o) acc[s][o][0] = acc[s][o][1] = acc[s][o][2] = acc[s][o][3] = 0.f;

  const int nchunks = (a_end - a_begin + CH - 1) / CH;
  stage_activations<MT>(sbase, A, M, K, a_begin, min(a_end, a_begin + CH));
  cp_async_commit();
  for (int c = 0; c < nchunks; ++c) {
    const int c0 = a_begin + c * CH;
    const int c1 = min(a_end, c0 + CH);
    if (c + 1 < nchunks) {  // next chunk into the other buffer
      stage_activations<MT>(sbase + ((c + 1) & 1) * kBuf, A, M, K, c1, min(a_end, c1 + CH));
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    // lane's fragment row and column inside the chunk buffer
    const uint32_t abuf = sbase + (c & 1) * kBuf + gq * kRow + 16 * t;
    if (active) {
      for (int a = c0; a < c1; a += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int au = a + u;
          if (au < c1) {  // warp-uniform; false only in the last batch of the range
            const uint4 cw = w[u];
            if (c_rem == 0 || au == a_begin) {  // first atom of a group: new constants
              const uint32_t z0 = (mz[u].x >> (4 * gq)) & 15u, z1 = (mz[u].y >> (4 * gq)) & 15u;
              d0 = make_deq_const(z0, (uint16_t)(ms[u] & 0xffffu));
              d1 = make_deq_const(z1, (uint16_t)(ms[u] >> 16));
            }
            if (++c_rem == apg) c_rem = 0;
            if (l_atom < a_end) {  // refill this slot with the atom U ahead
              w[u] = ldg_stream(wp + (size_t)l_atom * 32);
              if (l_rem == 0) {
                ms[u] = __ldg(sp + (size_t)l_grp * 8);
                mz[u] = __ldg(zp + l_grp);
              }
              ++l_atom;
              if (++l_rem == apg) { l_rem = 0; ++l_grp; }
            }
            // B fragments: token 8o+gq, k = 64au + 32s + 8t .. +7
            uint4 act[2][MT];
#pragma unroll
            for (int o = 0; o < MT; ++o)
#pragma unroll
              for (int s = 0; s < 2; ++s)
                act[s][o] = lds128(abuf + o * 8 * kRow + ((au - c0) * kAtomK + 32 * s) * 2);
            uint32_t p[4][4];
            dequant_word(cw.x, d0, p[0]);  // k-half 0, column gq
            dequant_word(cw.y, d1, p[1]);  // k-half 0, column gq + 8
            dequant_word(cw.z, d0, p[2]);  // k-half 1, column gq
            dequant_word(cw.w, d1, p[3]);  // k-half 1, column gq + 8
#pragma unroll
            for (int o = 0; o < MT; ++o) {
#pragma unroll
              for (int s = 0; s < 2; ++s) {
                const uint32_t* lo = p[2 * s];
                const uint32_t* hi = p[2 * s + 1];
                mma_16816(acc[s][o], lo[0], hi[0], lo[1], hi[1], act[s][o].x, act[s][o].y);
                mma_16816(acc[s][o], lo[2], hi[2], lo[3], hi[3], act[s][o].z, act[s][o].w);
              }
            }
          }
        }
      }
    }
    __syncthreads();  // buffer (c & 1) is refilled by the copies issued next iteration
  }

  // partial tile [token][column] (reuses activation buffer 0)
  float* red = reinterpret_cast<float*>(smem);
  if (active) {
#pragma unroll
    for (int o = 0; o < MT; ++o) {
      const int tok = 8 * o + 2 * t;
      const int col = kStripCols * warp + gq;
      red[tok * kRedStride + col] = acc[0][o][0] + acc[1][o][0];
      red[(tok + 1) * kRedStride + col] = acc[0][o][1] + acc[1][o][1];
      red[tok * kRedStride + col + 8] = acc[0][o][2] + acc[1][o][2];
      red[(tok + 1) * kRedStride + col + 8] = acc[0][o][3] + acc[1][o][3];
    }
  }

  const int col0 = blockIdx.y * kDecodeBlockCols;
  const int total = M * kDecodeBlockCols;
  if (split == 1) {
    __syncthreads();
    for (int e = threadIdx.x; e < total; e += kThreads) {
      const int tok = e / kDecodeBlockCols, col = e % kDecodeBlockCols;
      if (col0 + col < N)
        Y[(size_t)tok * N + col0 + col] = __half_as_ushort(__float2half_rn(red[tok * kRedStride + col]));
    }
  } else {
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();  // every CTA's partial tile is in its shared memory
    const int rank = (int)cluster.block_rank();
    const int per = (total + split - 1) / split;
    const int beg = rank * per;
    const int end = min(total, beg + per);
    for (int e = beg + threadIdx.x; e < end; e += kThreads) {
      const int tok = e / kDecodeBlockCols, col = e % kDecodeBlockCols;
      if (col0 + col < N) {
        float sum = 0.f;
        for (int r = 0; r < split; ++r)  // fixed order: deterministic
          sum += cluster.map_shared_rank(red, r)[tok * kRedStride + col];
        Y[(size_t)tok * N + col0 + col] = __half_as_ushort(__float2half_rn(sum));
      }
    }
    cluster.sync();  // keep shared memory alive until every remote read is done
  }
}

}  // namespace

namespace {

// Opt both kernel variants into their dynamic shared memory (once per process).
cudaError_t prepare_decode_kernels() {
  static cudaError_t state = cudaErrorNotReady;
  if (state == cudaErrorNotReady) {
    state = cudaFuncSetAttribute(decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 2 * act_buffer_bytes<1>());
    if (state == cudaSuccess)
      state = cudaFuncSetAttribute(decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   2 * act_buffer_bytes<2>());
  }
  return state;
}

}  // namespace

// CTAs of the decode kernel variant for M rows that fit on one SM.
int decode_ctas_per_sm(int M) {
  static int cache[2] = {0, 0};
  const int v = M <= 8 ? 0 : 1;
  if (cache[v] == 0) {
    int n = 0;
    if (prepare_decode_kernels() != cudaSuccess) return 2;
    cudaError_t e = v == 0 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                 &n, decode_kernel<1>, kThreads, 2 * act_buffer_bytes<1>())
                           : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                 &n, decode_kernel<2>, kThreads, 2 * act_buffer_bytes<2>());
    if (e != cudaSuccess || n <= 0) return 2;
    cache[v] = n;
  }
  return cache[v];
}

namespace {

template <int MT>
cudaError_t launch_mt(const uint16_t* A, const uint32_t* Wq, const uint16_t* Sp,
                      const uint32_t* Zp, uint16_t* Y, int M, int N, int K, int group, int split,
                      cudaStream_t stream) {
  constexpr int smem_bytes = 2 * act_buffer_bytes<MT>();
  static_assert(MT * 8 * kRedStride * 4 <= act_buffer_bytes<MT>(), "partial tile must fit");
  const cudaError_t prep = prepare_decode_kernels();
  if (prep != cudaSuccess) return prep;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)split, (unsigned)((N + kDecodeBlockCols - 1) / kDecodeBlockCols), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<MT>, A, reinterpret_cast<const uint4*>(Wq),
                            reinterpret_cast<const uint32_t*>(Sp),
                            reinterpret_cast<const uint2*>(Zp), Y, M, N, K, group, split);
}

}  // namespace

cudaError_t launch_decode(const uint16_t* A, const uint32_t* Wq, const uint16_t* Sp,
                          const uint32_t* Zp, uint16_t* Y, int M, int N, int K, int group,
                          int split, cudaStream_t stream) {
  if (M <= 8) return launch_mt<1>(A, Wq, Sp, Zp, Y, M, N, K, group, split, stream);
  return launch_mt<2>(A, Wq, Sp, Zp, Y, M, N, K, group, split, stream);
}

}  // namespace w4a16
