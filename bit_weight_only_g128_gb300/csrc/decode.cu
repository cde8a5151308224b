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
constexpr int kPrefetch = 8;                      // weight atoms in flight per warp

// Activation atoms staged per chunk (2048 or 1024 k), and the bytes of one
// staged row. The extra 64 bytes put consecutive rows in opposite halves of
// the 32 banks, so the 16-byte fragment loads of a quarter-warp (two rows x
// 64 bytes) never collide.
template <int MT>
__host__ __device__ constexpr int chunk_atoms() { return MT == 1 ? 32 : 16; }
template <int MT>
__host__ __device__ constexpr int act_row_bytes() { return chunk_atoms<MT>() * kAtomK * 2 + 64; }
template <int MT>
__host__ __device__ constexpr int act_buffer_bytes() { return MT * 8 * act_row_bytes<MT>(); }
template <int MT>
__host__ __device__ constexpr int red_bytes() { return MT * 8 * kRedStride * 4; }
template <int MT>
__host__ __device__ constexpr int smem_bytes() { return 2 * act_buffer_bytes<MT>() + red_bytes<MT>(); }

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

// CTA that owns unit u when T units are split among C CTAs.
__device__ __forceinline__ int owner_cta(long long u, long long T, int C) {
  return (int)(((u + 1) * C - 1) / T);
}

// Partial sums of strip `strip` over atoms [a_begin, a_end) for this lane's
// fragment: acc[s][o] (two independent accumulator chains, s = k-half).
template <int MT>
__device__ __forceinline__ void segment_mainloop(
    float (&acc)[2][MT][4], const uint16_t* __restrict__ A, const uint4* __restrict__ Wq,
    const uint32_t* __restrict__ Sp2, const uint2* __restrict__ Zp, int M, int K, int group,
    int strip, bool active, int a_begin, int a_end, uint32_t sbase) {
  constexpr int U = kPrefetch;
  constexpr int CH = chunk_atoms<MT>();
  constexpr int kRow = act_row_bytes<MT>();
  constexpr int kBuf = act_buffer_bytes<MT>();
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2, t = lane & 3;  // mma groupID / thread-in-group
  const int natoms = K / kAtomK;
  const int G = K / group;
  const int apg = group / kAtomK;  // atoms per group

  const uint4* wp = Wq + (size_t)(active ? strip : 0) * natoms * 32 + lane;
  const uint32_t* sp = Sp2 + (size_t)(active ? strip : 0) * G * 8 + gq;  // (s[gq], s[gq+8])
  const uint2* zp = Zp + (size_t)(active ? strip : 0) * G;

#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int o = 0; o < MT; ++o) acc[s][o][0] = acc[s][o][1] = acc[s][o][2] = acc[s][o][3] = 0.f;

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
        if (++l_rem == apg) {
          l_rem = 0;
          ++l_grp;
        }
      }
    }
  }
  int c_rem = a_begin % apg;  // position of the consumed atom inside its group
  DeqConst d0 = {}, d1 = {};

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
              if (++l_rem == apg) {
                l_rem = 0;
                ++l_grp;
              }
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
}

// MT: token octets (1: M <= 8, 2: M <= 16).
template <int MT>
__global__ void __launch_bounds__(kThreads, 2)
decode_kernel(const uint16_t* __restrict__ A, const uint4* __restrict__ Wq,
              const uint32_t* __restrict__ Sp2, const uint2* __restrict__ Zp,
              uint16_t* __restrict__ Y, int M, int N, int K, int group, int* __restrict__ counters,
              float* __restrict__ tiles) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem);
  float* red = reinterpret_cast<float*>(smem + 2 * act_buffer_bytes<MT>());
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, t = lane & 3;
  const int nstrips = N / kStripCols;
  const int nblk = (N + kDecodeBlockCols - 1) / kDecodeBlockCols;
  const int natoms = K / kAtomK;
  const int C = gridDim.x;
  const long long T = (long long)nblk * natoms;
  const long long u_begin = (long long)blockIdx.x * T / C;
  const long long u_end = (long long)(blockIdx.x + 1) * T / C;
  const int first_blk = (int)(u_begin / natoms);
  constexpr int kTileFloats = MT * 8 * kDecodeBlockCols;  // one partial tile in the workspace

  for (long long u = u_begin; u < u_end;) {
    const int b = (int)(u / natoms);
    const int a0 = (int)(u - (long long)b * natoms);
    const int a1 = (int)min((long long)natoms, u_end - (long long)b * natoms);
    u = (long long)(b + 1) * natoms;

    const int strip = b * kWarps + warp;
    const bool active = strip < nstrips;
    float acc[2][MT][4];
    segment_mainloop<MT>(acc, A, Wq, Sp2, Zp, M, K, group, strip, active, a0, a1, sbase);

    // partial tile [token][column] of this segment
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
          Y[(size_t)tok * N + col0 + col] =
              __half_as_ushort(__float2half_rn(red[tok * kRedStride + col]));
      }
    } else {
      // publish the partial tile, then count this CTA in
      const int slot = 2 * blockIdx.x + (b == first_blk ? 0 : 1);
      float* my = tiles + (size_t)slot * kTileFloats;
      for (int e = threadIdx.x; e < total; e += kThreads) {
        const int tok = e / kDecodeBlockCols, col = e % kDecodeBlockCols;
        my[e] = red[tok * kRedStride + col];
      }
      __threadfence();
      __syncthreads();
      const int c_first = owner_cta((long long)b * natoms, T, C);
      const int c_last = owner_cta((long long)b * natoms + natoms - 1, T, C);
      if (threadIdx.x == 0) {
        const int old = atomicAdd(counters + b, 1);
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
            sum += __ldcg(tiles + (size_t)cslot * kTileFloats + e);
          }
          const int tok = e / kDecodeBlockCols;
          Y[(size_t)tok * N + col0 + col] = __half_as_ushort(__float2half_rn(sum));
        }
        if (threadIdx.x == 0) counters[b] = 0;  // ready for the next call
      }
    }
    __syncthreads();  // the partial tile buffer is reused by the next segment
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
  }
  return state;
}

template <int MT>
cudaError_t launch_mt(const uint16_t* A, const uint32_t* Wq, const uint16_t* Sp,
                      const uint32_t* Zp, uint16_t* Y, int M, int N, int K, int group, int ctas,
                      int* counters, float* tiles, cudaStream_t stream) {
  const cudaError_t prep = prepare_decode_kernels();
  if (prep != cudaSuccess) return prep;
  decode_kernel<MT><<<ctas, kThreads, smem_bytes<MT>(), stream>>>(
      A, reinterpret_cast<const uint4*>(Wq), reinterpret_cast<const uint32_t*>(Sp),
      reinterpret_cast<const uint2*>(Zp), Y, M, N, K, group, counters, tiles);
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
  int* counters = static_cast<int*>(workspace);
  float* tiles =
      reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + decode_counter_bytes(N));
  if (M <= 8) return launch_mt<1>(A, Wq, Sp, Zp, Y, M, N, K, group, ctas, counters, tiles, stream);
  return launch_mt<2>(A, Wq, Sp, Zp, Y, M, N, K, group, ctas, counters, tiles, stream);
}

}  // namespace w4a16
