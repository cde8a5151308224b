// Decode path of the W4A16 linear layer: up to 16 rows of activations. Here
// the layer streams every packed weight from HBM once and does little math per
// byte; the vLLM PR #1032 thread reports the AWQ kernel ahead of FP16 only for
// batches below about 8, and names dequantization as the hard part.
//
// Design (sm_103a):
//   * Work unit: one 128-column block (8 strips of 16 columns) x one 64-k atom
//     (4 KiB of packed codes). The units are ordered block-major and the grid
//     is persistent (one or two CTAs per SM): CTA c takes the contiguous run
//     [c*T/C, (c+1)*T/C) of the T units (stream-K), so every CTA streams the
//     same number of bytes and runs long enough to keep 8 atoms per warp in
//     flight. A run covers a few "segments": pieces of consecutive blocks.
//   * Inside a segment, warp w owns strip w of the block. Each lane streams its
//     four words of an atom with one 16-byte load (L1 bypassed), 8 atoms ahead
//     of use; the activations of the segment's k-range are staged in shared
//     memory in chunks (cp.async, double buffered) and shared by the 8 warps.
//   * Dequantization in registers (LOP3 + exact fp16 subtract + one fp16
//     multiply per pair of codes) feeds mma.sync m16n8k16 with the weights as
//     the 16-row operand (output columns) and up to 8 tokens as the 8-column
//     operand. k inside each MMA is permuted identically on both operands (a
//     lane holds 4 consecutive k), which leaves the sum unchanged.
//   * A segment that covers a whole block writes Y directly. A block split
//     between CTAs is finished by the last of them to arrive: each writes its
//     fp32 partial tile to the workspace, then bumps the block's counter; the
//     one that completes the count sums the partial tiles in CTA order
//     (deterministic), writes Y and resets the counter to zero. No CTA ever
//     waits for another.
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRedStride = kDecodeBlockCols + 4;  // padded row of the partial tile

// Weight atoms in flight per warp (even: activations use a 2-deep ring).
template <int MT>
__host__ __device__ constexpr int prefetch_atoms() { return MT == 1 ? 8 : 4; }
template <int MT>
__host__ __device__ constexpr int smem_bytes() { return MT * 8 * kRedStride * 4; }

// 16-byte activation load, kept in L1: the 8 warps of a CTA read the same
// activations (same atoms, different strips).
__device__ __forceinline__ uint4 ldg_act(const uint16_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
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
  int gshift;  // group index of atom a is a >> gshift
};

// MT: token octets (1: M <= 8, 2: M <= 16).
template <int MT>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const DecodeArgs p) {
  constexpr int U = prefetch_atoms<MT>();
  extern __shared__ __align__(16) float red[];  // partial tile [token][column]
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, t = lane & 3;  // mma groupID / thread-in-group
  const int N = p.N, K = p.K, M = p.M;
  const int nstrips = N / kStripCols;
  const int nblk = (N + kDecodeBlockCols - 1) / kDecodeBlockCols;
  const int natoms = K / kAtomK;
  const int gshift = p.gshift;
  const int gmask = (1 << gshift) - 1;
  const int groups = (natoms + gmask) >> gshift;  // groups per strip (1 when per-channel)
  const int C = gridDim.x;
  const int T = nblk * natoms;  // < 2^27 for legal shapes
  const int u_begin = (int)((long long)blockIdx.x * T / C);
  const int u_end = (int)((long long)(blockIdx.x + 1) * T / C);
  const int first_blk = u_begin / natoms;
  constexpr int kTileFloats = MT * 8 * kDecodeBlockCols;  // one partial tile in the workspace

  // activation rows of this lane's fragment (rows >= M read row M-1; their
  // products land in accumulator columns that are never stored)
  const uint16_t* arow[MT];
#pragma unroll
  for (int o = 0; o < MT; ++o) arow[o] = p.A + (size_t)min(8 * o + gq, M - 1) * K + 8 * t;

  // ---- load stream: units u_begin.. in order, U units ahead of consumption
  int l_unit = u_begin;
  int l_blk = first_blk;
  int l_atom = u_begin - first_blk * natoms;
  int l_strip = l_blk * kWarps + warp;
  bool l_active = l_strip < nstrips;
  const uint4* l_ptr = p.Wq + ((size_t)(l_active ? l_strip : 0) * natoms + l_atom) * 32 + lane;
  const uint32_t* l_sp = p.Sp2 + (size_t)(l_active ? l_strip : 0) * groups * 8 + gq;
  const uint8_t* l_zp = p.Zp + (size_t)(l_active ? l_strip : 0) * groups * 8 + gq;

  uint4 w[U];
  uint32_t ms[U];
  uint32_t mz[U];
  // advance the load stream by one unit into slot `u`; group constants are
  // fetched at group starts and for the first unit of the run
  auto refill = [&](int u, bool first) {
    if (l_unit < u_end) {
      if (l_active) {
        w[u] = ldg_stream(l_ptr);
        if (first || (l_atom & gmask) == 0) {
          const int g = l_atom >> gshift;
          ms[u] = __ldg(l_sp + (size_t)g * 8);
          mz[u] = __ldg(l_zp + (size_t)g * 8);
        }
      }
      ++l_unit;
      l_ptr += 32;
      if (++l_atom == natoms) {  // next block: strip `warp` of it
        l_atom = 0;
        ++l_blk;
        l_strip = l_blk * kWarps + warp;
        l_active = l_strip < nstrips;
        l_ptr = p.Wq + (size_t)(l_active ? l_strip : 0) * natoms * 32 + lane;
        l_sp = p.Sp2 + (size_t)(l_active ? l_strip : 0) * groups * 8 + gq;
        l_zp = p.Zp + (size_t)(l_active ? l_strip : 0) * groups * 8 + gq;
      }
    }
  };
#pragma unroll
  for (int u = 0; u < U; ++u) refill(u, u == 0);

  // ---- activation ring: unit x uses act[(x - u_begin) & 1]; 2 units ahead
  uint4 act[2][2][MT];
  auto load_act = [&](int slot, int atom) {
#pragma unroll
    for (int o = 0; o < MT; ++o)
#pragma unroll
      for (int s = 0; s < 2; ++s) act[slot][s][o] = ldg_act(arow[o] + (size_t)atom * kAtomK + 32 * s);
  };
  {
    const int a0 = u_begin - first_blk * natoms;
    load_act(0, a0);
    if (u_begin + 1 < u_end) load_act(1, a0 + 1 < natoms ? a0 + 1 : 0);
  }

  for (int s0 = u_begin; s0 < u_end;) {
    // segment [s0, s1): atoms [a0, a1) of block b
    const int b = s0 / natoms;
    const int a0 = s0 - b * natoms;
    const int s1 = min(u_end, (b + 1) * natoms);
    const int a1 = s1 - b * natoms;
    const bool active = b * kWarps + warp < nstrips;

    float acc[2][MT][4];
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int o = 0; o < MT; ++o) acc[s][o][0] = acc[s][o][1] = acc[s][o][2] = acc[s][o][3] = 0.f;
    int cur_grp = -1;
    DeqConst d0 = {}, d1 = {};
    int c_atom = a0;  // atom of the unit being consumed

    // batches aligned to the run start keep slot indices compile-time constants
    for (int ub = u_begin + (s0 - u_begin) / U * U; ub < s1; ub += U) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int x = ub + u;
        if (x >= s0 && x < s1) {  // warp-uniform
          const uint4 cw = w[u];
          const uint32_t cms = ms[u];
          const uint32_t cmz = mz[u];
          refill(u, false);
          uint4 ca[2][MT];
#pragma unroll
          for (int o = 0; o < MT; ++o) {
            ca[0][o] = act[u & 1][0][o];
            ca[1][o] = act[u & 1][1][o];
          }
          if (x + 2 < u_end) {  // atom of unit x + 2 (the run may wrap into the next block)
            int na = c_atom + 2;
            if (na >= natoms) na -= natoms;
            if (na >= natoms) na -= natoms;  // K = 64: one atom per block
            load_act(u & 1, na);
          }
          if (active) {
            const int grp = c_atom >> gshift;
            if (grp != cur_grp) {  // first atom of a group (or of the segment)
              cur_grp = grp;
              d0 = make_deq_const(cmz & 15u, (uint16_t)(cms & 0xffffu));
              d1 = make_deq_const((cmz >> 4) & 15u, (uint16_t)(cms >> 16));
            }
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
                mma_16816(acc[s][o], lo[0], hi[0], lo[1], hi[1], ca[s][o].x, ca[s][o].y);
                mma_16816(acc[s][o], lo[2], hi[2], lo[3], hi[3], ca[s][o].z, ca[s][o].w);
              }
            }
          }
          ++c_atom;
        }
      }
    }

    // ---- segment epilogue: partial tile [token][column] in shared memory
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
    if (a0 == 0 && a1 == natoms) {  // the whole block is ours
      for (int e = threadIdx.x; e < total; e += kThreads) {
        const int tok = e / kDecodeBlockCols, col = e % kDecodeBlockCols;
        if (col0 + col < N)
          p.Y[(size_t)tok * N + col0 + col] =
              __half_as_ushort(__float2half_rn(red[tok * kRedStride + col]));
      }
    } else {
      // publish the partial tile, then count this CTA in
      const int slot = 2 * blockIdx.x + (b == first_blk ? 0 : 1);
      float* my = p.tiles + (size_t)slot * kTileFloats;
      for (int e = threadIdx.x; e < total; e += kThreads) {
        const int tok = e / kDecodeBlockCols, col = e % kDecodeBlockCols;
        my[e] = red[tok * kRedStride + col];
      }
      __threadfence();
      __syncthreads();
      const int c_first = owner_cta((long long)b * natoms, T, C);
      const int c_last = owner_cta((long long)b * natoms + natoms - 1, T, C);
      if (threadIdx.x == 0) {
        const int old = atomicAdd(p.counters + b, 1);
        s_last = (old == c_last - c_first);
      }
      __syncthreads();
      if (s_last) {  // every other contributor has published: finish the block
        __threadfence();
        for (int e = threadIdx.x; e < total; e += kThreads) {
          const int col = e % kDecodeBlockCols;
          if (col0 + col >= N) continue;
          float sum = 0.f;
          for (int c = c_first; c <= c_last; ++c) {  // fixed order: deterministic
            const int cfirst_blk = (int)(((long long)c * T / C) / natoms);
            const int cslot = 2 * c + (b == cfirst_blk ? 0 : 1);
            sum += __ldcg(p.tiles + (size_t)cslot * kTileFloats + e);
          }
          const int tok = e / kDecodeBlockCols;
          p.Y[(size_t)tok * N + col0 + col] = __half_as_ushort(__float2half_rn(sum));
        }
        if (threadIdx.x == 0) p.counters[b] = 0;  // ready for the next call
      }
    }
    __syncthreads();  // the partial tile buffer is reused by the next segment
    s0 = s1;
  }
}

// Opt both kernel variants into their dynamic shared memory (once per process).
cudaError_t prepare_decode_kernels() {
  static cudaError_t state = cudaErrorNotReady;
  if (state == cudaErrorNotReady) {
    state = cudaFuncSetAttribute(decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_bytes<1>());
    if (state == cudaSuccess)
      state = cudaFuncSetAttribute(decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   smem_bytes<2>());
    if (state == cudaSuccess)
      state = cudaFuncSetAttribute(decode_kernel<1>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   cudaSharedmemCarveoutMaxL1);
    if (state == cudaSuccess)
      state = cudaFuncSetAttribute(decode_kernel<2>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   cudaSharedmemCarveoutMaxL1);
  }
  return state;
}

template <int MT>
cudaError_t launch_mt(const DecodeArgs& args, int ctas, cudaStream_t stream) {
  const cudaError_t prep = prepare_decode_kernels();
  if (prep != cudaSuccess) return prep;
  decode_kernel<MT><<<ctas, kThreads, smem_bytes<MT>(), stream>>>(args);
  return cudaGetLastError();
}

}  // namespace

// CTAs of the decode kernel variant for M rows that fit on one SM.
int decode_ctas_per_sm(int M) {
  static int cache[2] = {0, 0};
  const int v = M <= 8 ? 0 : 1;
  if (cache[v] == 0) {
    int n = 0;
    if (prepare_decode_kernels() != cudaSuccess) return 1;
    cudaError_t e = v == 0 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                 &n, decode_kernel<1>, kThreads, smem_bytes<1>())
                           : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                 &n, decode_kernel<2>, kThreads, smem_bytes<2>());
    if (e != cudaSuccess || n <= 0) return 1;
    cache[v] = n;
  }
  return cache[v];
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
  args.gshift = decode_group_shift(K, group);
  if (args.gshift < 0) return cudaErrorInvalidValue;
  if (M <= 8) return launch_mt<1>(args, ctas, stream);
  return launch_mt<2>(args, ctas, stream);
}

// Group index of atom a is a >> shift: log2(group/64) for power-of-two
// groups, 30 (always group 0) for one group per column; -1 otherwise.
int decode_group_shift(int K, int group) {
  const int apg = group / kAtomK;
  if (apg > 0 && (apg & (apg - 1)) == 0) {
    int sh = 0;
    while ((1 << sh) < apg) ++sh;
    return sh;
  }
  return group == K ? 30 : -1;
}

}  // namespace w4a16
