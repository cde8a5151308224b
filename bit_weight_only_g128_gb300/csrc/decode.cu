// Decode path of the W4A16 linear layer: up to 16 rows of activations. Here
// the layer streams every packed weight from HBM once and does little math per
// byte; the vLLM PR #1032 thread reports the AWQ kernel ahead of FP16 only for
// batches below about 8, and names dequantization as the hard part. On GB300
// the HBM delivers about 22 bytes per SM clock, i.e. 44 int4 weights, so the
// kernel is as much bound by instruction issue as by memory: every
// instruction per weight counts.
//
// Design (sm_103a):
//   * Work unit: one 128-column block (8 strips of 16 columns) x one batch of
//     8 atoms (512 k; the last batch of a block may be shorter). Units are
//     ordered block-major; the grid is persistent and CTA c takes the run
//     [c*T/C, (c+1)*T/C) of the T units (stream-K), so every CTA streams the
//     same number of bytes in one long, uninterrupted pass.
//   * Warp w handles strip w of each unit's block. Each lane streams its four
//     words of an atom with one 16-byte load (L1 bypassed); the next unit's
//     atoms are loaded while the current one is computed (8 atoms, 4 KiB per
//     warp, always in flight), across block boundaries too. The next unit's
//     activations are copied into a two-slot shared-memory ring (cp.async)
//     meanwhile, one CTA barrier per unit.
//   * Group boundaries fall at fixed positions of a unit (groups are 1, 2, 4
//     or >= 8 atoms and units start at multiples of 8 atoms), so the code that
//     rebuilds the dequantization constants is placed at compile time.
//   * Dequantization in registers (LOP3 + exact fp16 subtract + one fp16
//     multiply per pair of codes) feeds mma.sync m16n8k16 with the weights as
//     the 16-row operand (output columns) and up to 8 tokens as the 8-column
//     operand. k inside each MMA is permuted identically on both operands (a
//     lane holds 4 consecutive k), which leaves the sum unchanged.
//   * A run's piece of one block ("segment") that covers the whole block
//     writes Y directly. A block shared by several CTAs is finished by the
//     last of them to arrive: each writes its fp32 partial tile to the
//     workspace, then bumps the block's counter; the one that completes the
//     count sums the tiles in CTA order (deterministic), writes Y and resets
//     the counter to zero. No CTA ever waits for another.
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRedStride = kDecodeBlockCols + 4;  // padded row of the partial tile
constexpr int kBatch = 8;                         // atoms per unit
// One staged activation row of a unit: 8 atoms x 64 k x 2 bytes, padded by
// 64 bytes so that consecutive rows fall in opposite halves of the 32 banks
// (a quarter-warp's 16-byte fragment loads cover two rows x 64 bytes).
constexpr int kActRow = kBatch * kAtomK * 2 + 64;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// atomicAdd with acquire-release semantics at device scope: the caller's
// earlier stores (and those it observed through a CTA barrier) are visible to
// whoever observes the new value, and the caller observes everything that
// the earlier adders released.
__device__ __forceinline__ int atomic_add_acq_rel(int* addr, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
  return old;
}

// CTA that owns unit u when T units are split among C CTAs.
__device__ __forceinline__ int owner_cta(long long u, long long T, int C) {
  return (int)(((u + 1) * C - 1) / T);
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
  int gshift;  // group of atom a is a >> gshift (30: a single group per column)
};

// Where one unit's data lives for this warp/lane.
struct Unit {
  int blk;       // 128-column block
  int a0;        // first atom
  int n;         // atoms in the unit (1..8)
  bool active;   // this warp's strip exists (N tail)
  const uint4* wp;
  const uint32_t* sp;
  const uint8_t* zp;
};

__device__ __forceinline__ Unit unit_at(const DecodeArgs& p, int x, int natoms, int nbb, int groups,
                                        int warp, int lane, int gq) {
  Unit u;
  u.blk = x / nbb;
  u.a0 = (x - u.blk * nbb) * kBatch;
  u.n = min(kBatch, natoms - u.a0);
  const int strip = u.blk * kWarps + warp;
  u.active = strip < p.N / kStripCols;
  const int st = u.active ? strip : 0;
  u.wp = p.Wq + ((size_t)st * natoms + u.a0) * 32 + lane;
  u.sp = p.Sp2 + (size_t)st * groups * 8 + gq;
  u.zp = p.Zp + (size_t)st * groups * 8 + gq;
  return u;
}

// Activations of a unit (rows 0..M-1, atoms a0..a0+n-1) into a ring slot.
__device__ __forceinline__ void stage_act(uint32_t slot, const uint16_t* __restrict__ A, int M,
                                          int K, int a0, int n) {
  const int units = n * (kAtomK / 8);  // 16-byte pieces per row
  for (int idx = threadIdx.x; idx < M * units; idx += kThreads) {
    const int row = idx / units, c = idx - row * units;
    cp_async16(slot + row * kActRow + c * 16, A + (size_t)row * K + (size_t)a0 * kAtomK + c * 8);
  }
}

// MT: token octets (1: M <= 8, 2: M <= 16). APG: atoms per group, 1, 2 or 4;
// 8 stands for groups of 8 or more atoms (or one group per column), whose
// boundaries fall on unit starts.
template <int MT, int APG>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const DecodeArgs p) {
  constexpr int NG = kBatch / APG;  // groups per unit
  __shared__ __align__(16) uint8_t act_ring[2][MT * 8 * kActRow];
  __shared__ float red[MT * 8 * kRedStride];
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, t = lane & 3;  // mma groupID / thread-in-group
  const int N = p.N, K = p.K, M = p.M;
  const int natoms = K / kAtomK;
  const int nbb = (natoms + kBatch - 1) / kBatch;  // units per block
  const int nblk = (N + kDecodeBlockCols - 1) / kDecodeBlockCols;
  const int groups = (natoms + (1 << p.gshift) - 1) >> p.gshift;
  const int C = gridDim.x;
  const int T = nblk * nbb;
  const int u_begin = (int)((long long)blockIdx.x * T / C);
  const int u_end = (int)((long long)(blockIdx.x + 1) * T / C);
  const int first_blk = u_begin / nbb;
  const uint32_t ring = (uint32_t)__cvta_generic_to_shared(&act_ring[0][0]);
  constexpr uint32_t kSlot = MT * 8 * kActRow;
  // this lane's B-fragment position inside a ring slot: row gq, k-octet t
  const uint32_t frag = (uint32_t)gq * kActRow + 16u * t;

  // ---- first unit: weights, group pairs, activations
  Unit cu = unit_at(p, u_begin, natoms, nbb, groups, warp, lane, gq);
  uint4 w[kBatch];
  uint32_t ms[NG], mz[NG];
  if (cu.active) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (u < cu.n) w[u] = ldg_stream(cu.wp + u * 32);
#pragma unroll
    for (int g = 0; g < NG; ++g)
      if (g * APG < cu.n) {
        const int grp = (cu.a0 + g * APG) >> p.gshift;
        ms[g] = __ldg(cu.sp + (size_t)grp * 8);
        mz[g] = __ldg(cu.zp + (size_t)grp * 8);
      }
  }
  stage_act(ring, p.A, M, K, cu.a0, cu.n);
  cp_async_commit();

  float acc[2][MT][4];
#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int o = 0; o < MT; ++o) acc[s][o][0] = acc[s][o][1] = acc[s][o][2] = acc[s][o][3] = 0.f;
  int seg_a0 = cu.a0;  // first atom of the current segment
  DeqConst d0 = {}, d1 = {};

  for (int x = u_begin; x < u_end; ++x) {
    const int i = x - u_begin;
    const bool has_next = x + 1 < u_end;
    const Unit nu = unit_at(p, has_next ? x + 1 : x, natoms, nbb, groups, warp, lane, gq);
    cp_async_wait_all();
    __syncthreads();  // unit x's activations landed; everyone is done with unit x-1's slot
    if (has_next) stage_act(ring + ((i + 1) & 1) * kSlot, p.A, M, K, nu.a0, nu.n);
    cp_async_commit();
    const uint32_t abuf = ring + (i & 1) * kSlot + frag;

    // group pairs of the next unit
    uint32_t nms[NG], nmz[NG];
    if (has_next && nu.active) {
#pragma unroll
      for (int g = 0; g < NG; ++g)
        if (g * APG < nu.n) {
          const int grp = (nu.a0 + g * APG) >> p.gshift;
          nms[g] = __ldg(nu.sp + (size_t)grp * 8);
          nmz[g] = __ldg(nu.zp + (size_t)grp * 8);
        }
    }
    const bool refill = has_next && nu.active;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const uint4 cw = w[u];
      if (refill && u < nu.n) w[u] = ldg_stream(nu.wp + u * 32);  // same slot, next unit
      if (cu.active && u < cu.n) {  // warp-uniform
        if (u % APG == 0) {  // first atom of a group
          const uint32_t zz = mz[u / APG], ss = ms[u / APG];
          d0 = make_deq_const(zz & 15u, (uint16_t)(ss & 0xffffu));
          d1 = make_deq_const((zz >> 4) & 15u, (uint16_t)(ss >> 16));
        }
        uint4 act[2][MT];
#pragma unroll
        for (int o = 0; o < MT; ++o)
#pragma unroll
          for (int s = 0; s < 2; ++s) act[s][o] = lds128(abuf + o * 8 * kActRow + (u * kAtomK + 32 * s) * 2);
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
    }
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      ms[g] = nms[g];
      mz[g] = nmz[g];
    }

    if (!has_next || nu.blk != cu.blk) {
      // ---- end of a segment: atoms [seg_a0, cu.a0 + cu.n) of block cu.blk
      const int b = cu.blk;
      const bool whole = seg_a0 == 0 && cu.a0 + cu.n == natoms;
      if (cu.active) {
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
#pragma unroll
      for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int o = 0; o < MT; ++o) acc[s][o][0] = acc[s][o][1] = acc[s][o][2] = acc[s][o][3] = 0.f;
      __syncthreads();
      const int col0 = b * kDecodeBlockCols;
      const int total = M * kDecodeBlockCols;
      if (whole) {
        for (int e = threadIdx.x; e < total; e += kThreads) {
          const int tok = e / kDecodeBlockCols, col = e - tok * kDecodeBlockCols;
          if (col0 + col < N)
            p.Y[(size_t)tok * N + col0 + col] =
                __half_as_ushort(__float2half_rn(red[tok * kRedStride + col]));
        }
      } else {
        // publish the partial tile, then count this CTA in (one release
        // atomic after the CTA barrier covers every thread's tile stores)
        constexpr int kTileFloats = MT * 8 * kDecodeBlockCols;
        constexpr int kPerThread = (kTileFloats + kThreads - 1) / kThreads;
        const int slot = 2 * blockIdx.x + (b == first_blk ? 0 : 1);
        float* my = p.tiles + (size_t)slot * kTileFloats;
        for (int e = threadIdx.x; e < total; e += kThreads) {
          const int tok = e / kDecodeBlockCols, col = e - tok * kDecodeBlockCols;
          my[e] = red[tok * kRedStride + col];
        }
        __syncthreads();
        const int c_first = owner_cta((long long)b * nbb, T, C);
        const int c_last = owner_cta((long long)b * nbb + nbb - 1, T, C);
        if (threadIdx.x == 0) s_last = (atomic_add_acq_rel(p.counters + b, 1) == c_last - c_first);
        __syncthreads();
        if (s_last) {  // every other contributor has published: finish the block
          // sum the contributors' tiles in CTA order (deterministic); every
          // thread keeps its elements' sums in registers and issues the loads
          // of one contributor at once
          float sum[kPerThread];
#pragma unroll
          for (int k = 0; k < kPerThread; ++k) sum[k] = 0.f;
          for (int c = c_first; c <= c_last; ++c) {
            const int cfirst_blk = (int)(((long long)c * T / C) / nbb);
            const float* tile = p.tiles + (size_t)(2 * c + (b == cfirst_blk ? 0 : 1)) * kTileFloats;
#pragma unroll
            for (int k = 0; k < kPerThread; ++k) {
              const int e = threadIdx.x + k * kThreads;
              if (e < total) sum[k] += __ldcg(tile + e);
            }
          }
#pragma unroll
          for (int k = 0; k < kPerThread; ++k) {
            const int e = threadIdx.x + k * kThreads;
            const int col = e % kDecodeBlockCols;
            if (e < total && col0 + col < N)
              p.Y[(size_t)(e / kDecodeBlockCols) * N + col0 + col] = __half_as_ushort(__float2half_rn(sum[k]));
          }
          if (threadIdx.x == 0) p.counters[b] = 0;  // ready for the next call
        }
      }
      __syncthreads();  // the partial tile buffer is reused by the next segment
      seg_a0 = nu.a0;
    }
    cu = nu;
  }
}

template <int MT, int APG>
cudaError_t launch_variant(const DecodeArgs& args, int ctas, cudaStream_t stream) {
  decode_kernel<MT, APG><<<ctas, kThreads, 0, stream>>>(args);
  return cudaGetLastError();
}

template <int MT>
cudaError_t launch_mt(const DecodeArgs& args, int apg_t, int ctas, cudaStream_t stream) {
  switch (apg_t) {
    case 1: return launch_variant<MT, 1>(args, ctas, stream);
    case 2: return launch_variant<MT, 2>(args, ctas, stream);
    case 4: return launch_variant<MT, 4>(args, ctas, stream);
    default: return launch_variant<MT, 8>(args, ctas, stream);
  }
}

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
// 9..16 rows; the group size does not change the resources).
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

// Work units (128 columns x 8 atoms) of a problem; 0 if the group size is not
// supported by the decode kernel.
long decode_units(int N, int K, int group) {
  int apg_t, gshift;
  if (!group_shape(K, group, &apg_t, &gshift)) return 0;
  const long natoms = K / kAtomK;
  return (long)((N + kDecodeBlockCols - 1) / kDecodeBlockCols) * ((natoms + kBatch - 1) / kBatch);
}

// The counter area has room for the largest legal N (2^20 columns = 8192
// blocks), whatever N this call has: a workspace can then serve calls of any
// shape in turn, since no call's partial tiles ever land on another call's
// counters.
size_t decode_counter_bytes(int N) {
  (void)N;
  return (size_t)((1 << 20) / kDecodeBlockCols) * sizeof(int);
}

size_t decode_workspace_bytes(int M, int N, int ctas) {
  const int mt = M <= 8 ? 1 : 2;
  const size_t tile_bytes = (size_t)mt * 8 * kDecodeBlockCols * sizeof(float);
  return decode_counter_bytes(N) + 2 * (size_t)ctas * tile_bytes;
}

cudaError_t launch_decode(const uint16_t* A, const uint32_t* Wq, const uint16_t* Sp,
                          const uint32_t* Zp, uint16_t* Y, int M, int N, int K, int group,
                          int ctas, void* workspace, cudaStream_t stream) {
  DecodeArgs args;
  int apg_t = 0;
  if (!group_shape(K, group, &apg_t, &args.gshift)) return cudaErrorInvalidValue;
  args.A = A;
  args.Wq = reinterpret_cast<const uint4*>(Wq);
  args.Sp2 = reinterpret_cast<const uint32_t*>(Sp);
  args.Zp = reinterpret_cast<const uint8_t*>(Zp);
  args.Y = Y;
  args.counters = static_cast<int*>(workspace);
  args.tiles = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + decode_counter_bytes(N));
  args.M = M;
  args.N = N;
  args.K = K;
  if (M <= 8) return launch_mt<1>(args, apg_t, ctas, stream);
  return launch_mt<2>(args, apg_t, ctas, stream);
}

}  // namespace w4a16
