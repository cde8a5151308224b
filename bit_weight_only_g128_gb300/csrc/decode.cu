// Decode path of the W4A16 linear layer: up to 16 rows of activations. Here
// the layer streams every packed weight from HBM once and does little math per
// byte; the vLLM PR #1032 thread reports the AWQ kernel ahead of FP16 only for
// batches below about 8, and names dequantization as the hard part. On GB300
// the HBM delivers about 22 bytes per SM clock, i.e. 44 int4 weights, so the
// kernel is as much bound by instruction issue as by memory: every
// instruction per weight counts.
//
// Design (sm_103a):
//   * Grid (split, N/128): a CTA is 8 warps = 8 strips of 16 columns (one
//     128-column block) over one K range; `split` ranges per block, chosen on
//     the host to fill the resident CTA slots in whole waves.
//   * A warp walks its strip's range in batches of 8 atoms (64 k each). Each
//     lane streams its four words of an atom with one 16-byte load (L1
//     bypassed); the next batch is loaded while the current one is computed,
//     so 8 atoms (4 KiB per warp) are always in flight. The scale / zero-point
//     pairs of the groups of the next batch are fetched with it.
//   * Group boundaries fall at fixed positions of a batch (the range starts on
//     a group boundary and groups are 1, 2, 4 or >= 8 atoms), so the code that
//     rebuilds the dequantization constants is placed at compile time.
//   * Dequantization in registers (LOP3 + exact fp16 subtract + one fp16
//     multiply per pair of codes) feeds mma.sync m16n8k16 with the weights as
//     the 16-row operand (output columns) and up to 8 tokens as the 8-column
//     operand. k inside each MMA is permuted identically on both operands (a
//     lane holds 4 consecutive k), which leaves the sum unchanged. The 8
//     warps read the same activations, which therefore stay in L1.
//   * With split > 1, each CTA writes its fp32 partial tile to the workspace
//     and bumps the block's counter; the CTA that completes the count sums the
//     tiles in split order (deterministic), writes Y and resets the counter to
//     zero. No CTA ever waits for another.
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRedStride = kDecodeBlockCols + 4;  // padded row of the partial tile
constexpr int kBatch = 8;                         // atoms per batch (in flight per warp)

// 16-byte activation load, kept in L1: the 8 warps of a CTA read the same
// activations (same atoms, different strips).
__device__ __forceinline__ uint4 ldg_act(const uint16_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

struct DecodeArgs {
  const uint16_t* A;
  const uint4* Wq;
  const uint32_t* Sp2;  // scale pairs (s[c], s[c+8])
  const uint8_t* Zp;    // zero-point pairs z[c] | z[c+8] << 4
  uint16_t* Y;
  int* counters;
  float* tiles;
  int M, N, K;
  int gran;    // K ranges are multiples of this many atoms
  int gshift;  // group of atom a is a >> gshift (30: a single group per column)
};

// One atom: dequantize the lane's 4 words and run the MMAs on the activation
// fragments of token octets 0..MT-1.
template <int MT>
__device__ __forceinline__ void atom_mma(float (&acc)[2][MT][4], const uint4& cw, const DeqConst& d0,
                                         const DeqConst& d1, const uint4 (&act)[2][MT]) {
  uint32_t q[4][4];
  dequant_word(cw.x, d0, q[0]);  // k-half 0, column gq
  dequant_word(cw.y, d1, q[1]);  // k-half 0, column gq + 8
  dequant_word(cw.z, d0, q[2]);  // k-half 1, column gq
  dequant_word(cw.w, d1, q[3]);  // k-half 1, column gq + 8
#pragma unroll
  for (int o = 0; o < MT; ++o) {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const uint32_t* lo = q[2 * s];
      const uint32_t* hi = q[2 * s + 1];
      mma_16816(acc[s][o], lo[0], hi[0], lo[1], hi[1], act[s][o].x, act[s][o].y);
      mma_16816(acc[s][o], lo[2], hi[2], lo[3], hi[3], act[s][o].z, act[s][o].w);
    }
  }
}

// MT: token octets (1: M <= 8, 2: M <= 16). APG: atoms per group, 1, 2 or 4;
// 8 stands for groups of 8 or more atoms (or one group per column), whose
// boundaries fall on batch starts.
template <int MT, int APG>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const DecodeArgs p) {
  constexpr int NG = kBatch / APG;  // groups per batch
  __shared__ float red[MT * 8 * kRedStride];
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, t = lane & 3;  // mma groupID / thread-in-group
  const int N = p.N, K = p.K, M = p.M;
  const int natoms = K / kAtomK;
  const int split = gridDim.x, sidx = blockIdx.x, b = blockIdx.y;
  const int ngran = natoms / p.gran;
  const int a0 = (int)((long long)sidx * ngran / split) * p.gran;
  const int a1 = (int)((long long)(sidx + 1) * ngran / split) * p.gran;
  const int n = a1 - a0;
  const int strip = b * kWarps + warp;
  const bool active = strip < N / kStripCols;
  const int groups = (natoms + (1 << p.gshift) - 1) >> p.gshift;

  float acc[2][MT][4];
#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int o = 0; o < MT; ++o) acc[s][o][0] = acc[s][o][1] = acc[s][o][2] = acc[s][o][3] = 0.f;

  if (active && n > 0) {
    const uint4* wp = p.Wq + ((size_t)strip * natoms + a0) * 32 + lane;
    const uint32_t* sp = p.Sp2 + (size_t)strip * groups * 8 + gq;
    const uint8_t* zp = p.Zp + (size_t)strip * groups * 8 + gq;
    const uint16_t* ap[MT];
#pragma unroll
    for (int o = 0; o < MT; ++o)  // rows >= M read row M-1; those columns are never stored
      ap[o] = p.A + (size_t)min(8 * o + gq, M - 1) * K + (size_t)a0 * kAtomK + 8 * t;

    // batch 0: weights and the group pairs of its groups
    uint4 w[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (u < n) w[u] = ldg_stream(wp + u * 32);
    uint32_t ms[NG], mz[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const int grp = (a0 + g * APG) >> p.gshift;
      if (g * APG < n) {
        ms[g] = __ldg(sp + (size_t)grp * 8);
        mz[g] = __ldg(zp + (size_t)grp * 8);
      }
    }
    DeqConst d0 = {}, d1 = {};

    for (int i = 0; i * kBatch < n; ++i) {
      const int base = i * kBatch;       // first atom of this batch (relative to a0)
      const int nb = base + kBatch;      // first atom of the next batch
      // group pairs of the next batch
      uint32_t nms[NG], nmz[NG];
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        if (nb + g * APG < n) {
          const int grp = (a0 + nb + g * APG) >> p.gshift;
          nms[g] = __ldg(sp + (size_t)grp * 8);
          nmz[g] = __ldg(zp + (size_t)grp * 8);
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (base + u < n) {  // warp-uniform; false only in a short last batch
          const uint4 cw = w[u];
          if (nb + u < n) w[u] = ldg_stream(wp + (nb + u) * 32);  // same slot, next batch
          if (u % APG == 0) {  // first atom of a group
            const uint32_t zz = mz[u / APG], ss = ms[u / APG];
            d0 = make_deq_const(zz & 15u, (uint16_t)(ss & 0xffffu));
            d1 = make_deq_const((zz >> 4) & 15u, (uint16_t)(ss >> 16));
          }
          uint4 act[2][MT];
#pragma unroll
          for (int o = 0; o < MT; ++o)
#pragma unroll
            for (int s = 0; s < 2; ++s)
              act[s][o] = ldg_act(ap[o] + (size_t)(base + u) * kAtomK + 32 * s);
          atom_mma<MT>(acc, cw, d0, d1, act);
        }
      }
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        ms[g] = nms[g];
        mz[g] = nmz[g];
      }
    }
  }

  // partial tile [token][column] of this CTA
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
  __syncthreads();
  const int col0 = b * kDecodeBlockCols;
  const int total = M * kDecodeBlockCols;
  if (split == 1) {
    for (int e = threadIdx.x; e < total; e += kThreads) {
      const int tok = e / kDecodeBlockCols, col = e % kDecodeBlockCols;
      if (col0 + col < N)
        p.Y[(size_t)tok * N + col0 + col] = __half_as_ushort(__float2half_rn(red[tok * kRedStride + col]));
    }
    return;
  }
  // publish the partial tile, then count this CTA in
  constexpr int kTileFloats = MT * 8 * kDecodeBlockCols;
  float* my = p.tiles + ((size_t)b * split + sidx) * kTileFloats;
  for (int e = threadIdx.x; e < total; e += kThreads) {
    const int tok = e / kDecodeBlockCols, col = e % kDecodeBlockCols;
    my[e] = red[tok * kRedStride + col];
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(p.counters + b, 1) == split - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();  // every other split of this block has published its tile
  const float* tb = p.tiles + (size_t)b * split * kTileFloats;
  for (int e = threadIdx.x; e < total; e += kThreads) {
    const int col = e % kDecodeBlockCols;
    if (col0 + col >= N) continue;
    float sum = 0.f;
    for (int r = 0; r < split; ++r) sum += __ldcg(tb + (size_t)r * kTileFloats + e);  // fixed order
    p.Y[(size_t)(e / kDecodeBlockCols) * N + col0 + col] = __half_as_ushort(__float2half_rn(sum));
  }
  if (threadIdx.x == 0) p.counters[b] = 0;  // ready for the next call
}

template <int MT, int APG>
cudaError_t launch_variant(const DecodeArgs& args, int split, cudaStream_t stream) {
  const dim3 grid((unsigned)split, (unsigned)((args.N + kDecodeBlockCols - 1) / kDecodeBlockCols), 1);
  decode_kernel<MT, APG><<<grid, kThreads, 0, stream>>>(args);
  return cudaGetLastError();
}

template <int MT>
cudaError_t launch_mt(const DecodeArgs& args, int apg_t, int split, cudaStream_t stream) {
  switch (apg_t) {
    case 1: return launch_variant<MT, 1>(args, split, stream);
    case 2: return launch_variant<MT, 2>(args, split, stream);
    case 4: return launch_variant<MT, 4>(args, split, stream);
    default: return launch_variant<MT, 8>(args, split, stream);
  }
}

// Atoms per group as the kernel template sees it (1, 2, 4, or 8 for >= 8 or
// a single group), the K-range granularity, and the group shift; false if
// the group size is not supported.
bool group_shape(int K, int group, int* apg_t, int* gran, int* gshift) {
  const int natoms = K / kAtomK;
  const int apg = group / kAtomK;
  if (group == K) {  // one group per column: any range, any batch position
    *apg_t = 8;
    *gran = 1;
    *gshift = 30;
    if (apg > 0 && (apg & (apg - 1)) == 0 && apg < 8) {  // also a small power of two
      *apg_t = apg;
      *gran = apg;
      *gshift = apg == 1 ? 0 : (apg == 2 ? 1 : 2);
    }
    return natoms > 0;
  }
  if (apg <= 0 || (apg & (apg - 1)) != 0) return false;
  int sh = 0;
  while ((1 << sh) < apg) ++sh;
  *gshift = sh;
  *apg_t = apg < 8 ? apg : 8;
  *gran = apg < 8 ? apg : 8;
  return true;
}

}  // namespace

// CTAs of the decode kernel that fit on one SM (occupancy query, M <= 8 or
// 9..16 rows; group size does not change the resources).
int decode_ctas_per_sm(int M) {
  static int cache[2] = {0, 0};
  const int v = M <= 8 ? 0 : 1;
  if (cache[v] == 0) {
    int n = 0;
    cudaError_t e = v == 0 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<1, 2>, kThreads, 0)
                           : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<2, 2>, kThreads, 0);
    if (e != cudaSuccess || n <= 0) return 1;
    cache[v] = n;
  }
  return cache[v];
}

// Number of K ranges (granules of `gran` atoms) the decode kernel can split
// K into; 0 if the group size is not supported.
int decode_max_split(int K, int group) {
  int apg_t, gran, gshift;
  if (!group_shape(K, group, &apg_t, &gran, &gshift)) return 0;
  return (K / kAtomK) / gran;
}

// The counter area has room for the largest legal N (2^20 columns = 8192
// blocks), whatever N this call has: a workspace can then serve calls of any
// shape in turn, since no call's partial tiles ever land on another call's
// counters.
size_t decode_counter_bytes(int N) {
  (void)N;
  return (size_t)((1 << 20) / kDecodeBlockCols) * sizeof(int);
}

size_t decode_workspace_bytes(int M, int N, int split) {
  if (split <= 1) return 0;
  const int mt = M <= 8 ? 1 : 2;
  const size_t nblk = (size_t)((N + kDecodeBlockCols - 1) / kDecodeBlockCols);
  const size_t tile_bytes = (size_t)mt * 8 * kDecodeBlockCols * sizeof(float);
  return decode_counter_bytes(N) + nblk * (size_t)split * tile_bytes;
}

cudaError_t launch_decode(const uint16_t* A, const uint32_t* Wq, const uint16_t* Sp,
                          const uint32_t* Zp, uint16_t* Y, int M, int N, int K, int group,
                          int split, void* workspace, cudaStream_t stream) {
  DecodeArgs args;
  int apg_t = 0;
  if (!group_shape(K, group, &apg_t, &args.gran, &args.gshift)) return cudaErrorInvalidValue;
  args.A = A;
  args.Wq = reinterpret_cast<const uint4*>(Wq);
  args.Sp2 = reinterpret_cast<const uint32_t*>(Sp);
  args.Zp = reinterpret_cast<const uint8_t*>(Zp);
  args.Y = Y;
  args.counters = static_cast<int*>(workspace);
  args.tiles = workspace ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                                    decode_counter_bytes(N))
                         : nullptr;
  args.M = M;
  args.N = N;
  args.K = K;
  if (M <= 8) return launch_mt<1>(args, apg_t, split, stream);
  return launch_mt<2>(args, apg_t, split, stream);
}

}  // namespace w4a16
