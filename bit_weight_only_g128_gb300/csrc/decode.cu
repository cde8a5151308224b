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

// MT: token octets (1: M <= 8, 2: M <= 16). U: atoms in flight per warp.
template <int MT, int U>
__global__ void __launch_bounds__(kThreads)
decode_kernel(const uint16_t* __restrict__ A, const uint4* __restrict__ Wq,
              const uint16_t* __restrict__ Sp, const uint2* __restrict__ Zp,
              uint16_t* __restrict__ Y, int M, int N, int K, int group, int split) {
  __shared__ float red[MT * 8 * kRedStride];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, t = lane & 3;  // mma groupID / thread-in-group
  const int nstrips = N / kStripCols;
  const int strip = blockIdx.y * kWarps + warp;
  const int natoms = K / kAtomK;
  const int a_begin = (int)(((long long)blockIdx.x * natoms) / split);
  const int a_end = (int)(((long long)(blockIdx.x + 1) * natoms) / split);
  const int G = K / group;
  const int apg = group / kAtomK;  // atoms per group

  float acc[MT][4];
#pragma unroll
  for (int o = 0; o < MT; ++o) acc[o][0] = acc[o][1] = acc[o][2] = acc[o][3] = 0.f;

  if (strip < nstrips) {
    const uint4* wp = Wq + (size_t)strip * natoms * 32 + lane;
    const uint16_t* sp = Sp + (size_t)strip * G * 16 + gq;
    const uint2* zp = Zp + (size_t)strip * G;
    const uint16_t* arow[MT];
    bool aval[MT];
#pragma unroll
    for (int o = 0; o < MT; ++o) {
      const int m = 8 * o + gq;
      aval[o] = m < M;
      arow[o] = A + (size_t)(aval[o] ? m : 0) * K + 8 * t;
    }

    // weights and per-group constants of the atoms in flight
    uint4 w[U];
    uint32_t sv[U];
    uint2 zv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int au = a_begin + u;
      if (au < a_end) {
        const int grp = au / apg;
        w[u] = ldg_stream(wp + (size_t)au * 32);
        sv[u] = (uint32_t)sp[grp * 16] | ((uint32_t)sp[grp * 16 + 8] << 16);
        zv[u] = zp[grp];
      }
    }

    for (int a = a_begin; a < a_end; a += U) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int au = a + u;
        if (au < a_end) {
          const uint4 cw = w[u];
          const uint32_t cs = sv[u];
          const uint2 cz = zv[u];
          const int nx = au + U;
          if (nx < a_end) {  // refill this slot with the atom U ahead
            const int grp = nx / apg;
            w[u] = ldg_stream(wp + (size_t)nx * 32);
            sv[u] = (uint32_t)sp[grp * 16] | ((uint32_t)sp[grp * 16 + 8] << 16);
            zv[u] = zp[grp];
          }
          // activations of this atom: lane holds k = 64au + 32s + 8t .. +7 of token 8o+gq
          uint4 act[2][MT];
#pragma unroll
          for (int o = 0; o < MT; ++o) {
#pragma unroll
            for (int s = 0; s < 2; ++s)
              act[s][o] = aval[o] ? ldg_keep(arow[o] + (size_t)au * kAtomK + 32 * s)
                                  : make_uint4(0u, 0u, 0u, 0u);
          }
          const DeqConst d0 = make_deq_const((cz.x >> (4 * gq)) & 15u, (uint16_t)(cs & 0xffffu));
          const DeqConst d1 = make_deq_const((cz.y >> (4 * gq)) & 15u, (uint16_t)(cs >> 16));
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
              mma_16816(acc[o], lo[0], hi[0], lo[1], hi[1], act[s][o].x, act[s][o].y);
              mma_16816(acc[o], lo[2], hi[2], lo[3], hi[3], act[s][o].z, act[s][o].w);
            }
          }
        }
      }
    }

    // accumulator fragment: rows = columns gq / gq+8 of the strip, cols = tokens 2t, 2t+1
#pragma unroll
    for (int o = 0; o < MT; ++o) {
      const int tok = 8 * o + 2 * t;
      const int col = kStripCols * warp + gq;
      red[tok * kRedStride + col] = acc[o][0];
      red[(tok + 1) * kRedStride + col] = acc[o][1];
      red[tok * kRedStride + col + 8] = acc[o][2];
      red[(tok + 1) * kRedStride + col + 8] = acc[o][3];
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

template <int MT>
cudaError_t launch_mt(const uint16_t* A, const uint32_t* Wq, const uint16_t* Sp,
                      const uint32_t* Zp, uint16_t* Y, int M, int N, int K, int group, int split,
                      cudaStream_t stream) {
  constexpr int U = 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)split, (unsigned)((N + kDecodeBlockCols - 1) / kDecodeBlockCols), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<MT, U>, A, reinterpret_cast<const uint4*>(Wq), Sp,
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
