// Decode path of the W4A16 linear layer (device code, shared by the
// translation units that instantiate it for fp16 and bf16 activations): up to 16 rows of activations. Here
// the layer streams every packed weight from HBM once and does little math per
// byte; the vLLM PR #1032 thread reports the AWQ kernel ahead of FP16 only for
// batches below about 8, and names dequantization as the hard part. On GB300
// the HBM delivers about 22 bytes per SM clock, i.e. 44 int4 weights, so the
// kernel is as much bound by instruction issue as by memory: every
// instruction per weight counts.
//
// Design (sm_103a):
//   * Work: the atoms (64 k) of every 128-column block (8 strips of 16
//     columns), block-major, are split among the persistent CTAs in equal
//     runs (stream-K). Runs start at group boundaries (multiples of a
//     group's atoms, up to 8; any atom with one group per column), so every
//     CTA streams the same number of bytes, to within one group. A run is
//     walked in units of up to 8 atoms, a unit never crossing a block.
//   * Warp w handles strip w of each unit's block. Each lane streams its four
//     words of an atom with one 16-byte load (L1 bypassed); the next unit's
//     atoms are loaded while the current one is computed, across block
//     boundaries too. Activations and the units' scale and zero-point pairs
//     go through a four-slot shared-memory ring (cp.async), three units
//     ahead, with one CTA barrier per unit; a unit's copies have two units of
//     compute to land.
//   * Codes enter the tensor core as they are. A 4-bit code q masked into the
//     low nibble of an fp16 half is the subnormal q * 2^-24, exact; masked
//     one nibble higher it is 16 q * 2^-24. So one AND per pair of codes
//     feeds mma.sync m16n8k16 (weights as the 16-row operand, tokens as the
//     8 columns), with the "low nibble" and "high nibble" pairs accumulated
//     separately (fp32) and the latter divided by 16 at the group's end. k
//     inside each MMA is permuted identically on both operands, which leaves
//     the sum unchanged.
//   * Scale and zero point are applied once per group in fp32: with
//     P = sum_k q_k a_k over the group and S = sum_k a_k (per token, from one
//     extra MMA per atom against a ones operand, computed once per CTA), the
//     group adds s * (P - z * S) = sum_k (q_k - z) s a_k. The product of a
//     code and an activation is exact, so the only roundings are fp32 ones;
//     the fp16 rounding of each dequantized weight that a dequantize-then-
//     multiply kernel performs is not made (the result moves by at most
//     2^-11 sum |a w|, a quarter of the accuracy bound).
//   * A run's piece of one block ("segment") that covers the whole block
//     writes Y directly. Otherwise the block is shared: a run that starts
//     inside a block contributes its first segment as an fp32 partial tile
//     (workspace slot of the CTA) and raises the CTA's flag; the CTA holding
//     the block's first atom, whose segment of it ends its run, waits for the
//     flags of the later contributors (raised at the start of their runs, so
//     the wait is normally over at once; bounded, with an error bit when it
//     runs out), adds their tiles to its own partial in CTA order
//     (deterministic), writes Y and lowers the flags for the next call.
//   * Launched with programmatic stream serialization: the grid may start
//     while the previous kernel on the stream drains. Everything that grid
//     may write (A, Y, the workspace) is touched only after the grid-
//     dependency wait; on request the first units' weights, scales and zero
//     points are read before it (weights that the preceding work does not
//     write).
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace w4a16 {

struct DecodeArgs {
  const uint16_t* A;
  const uint4* Wq;
  const uint32_t* Sp2;  // scale pairs (s[c], s[c+8])
  const uint8_t* Zp;    // zero-point pairs z[c] | z[c+8] << 4
  uint16_t* Y;
  int* flags;   // one per CTA: its partial tile is published
  float* tiles;  // one partial tile per CTA
  int* err;      // device error word
  int M, N, K;
  int gshift;         // group of atom a is a >> gshift (30: a single group per column)
  int granule;        // atoms per split granule (runs start at multiples of it)
  int early_weights;  // read the first units' weights before the grid-dependency wait
  // strip variant: shared-memory layout (bytes)
  int act_row, sums_off, meta_off, zp_off, red_off;
  // resident variant, fused gate/up epilogue: the N columns are [gate | up]
  // and Y (N/2 columns) = silu(gate) * up; the CTA's finished fp32 strips
  // at ytile_off, ytile_stride floats apart. They overlay the scale records
  // (each strip's own, which only the warp that finishes a whole strip
  // reads, and nobody once every warp has left the main loop) when those
  // are large enough; else the activation rows, dead after the main loop,
  // when the CTA has no more strips than warps (whole_in_red: every warp
  // then has at most two segments, and finished strips go through the
  // warps' partial slots too); else a region of their own
  int silu, ytile_off, ytile_stride, whole_in_red;
  // W4A8: per-row factors of the result (the activations' scales), or null
  const float* row_scale;
  size_t tile_floats;  // extent of `tiles` (for the checked build)
};

// The row factor of token `tok` (1 without one).
__device__ __forceinline__ float row_factor(const float* rs, int tok) { return rs ? rs[tok] : 1.0f; }

// The decode kernels' global accesses, tested against the buffers' extents
// in the checked build (see common.cuh): packed weights, activation rows,
// scale and zero-point pairs, results, flags and partial tiles.
__device__ __forceinline__ const uint4* wq_at(const DecodeArgs& p, const uint4* ptr) {
  return ld_at(ptr, p.Wq, (size_t)p.N * p.K / 32, p.err);
}
__device__ __forceinline__ const uint16_t* a_at(const DecodeArgs& p, const uint16_t* ptr) {
  return ld_at(ptr, p.A, (size_t)p.M * p.K - 7, p.err);  // 16-byte copies
}
__device__ __forceinline__ const uint4* sp_at(const DecodeArgs& p, const uint4* ptr, int group_count) {
  return ld_at(ptr, reinterpret_cast<const uint4*>(p.Sp2), (size_t)group_count * p.N / 8, p.err);
}
__device__ __forceinline__ const uint2* zp_at(const DecodeArgs& p, const uint2* ptr, int group_count) {
  return ld_at(ptr, reinterpret_cast<const uint2*>(p.Zp), (size_t)group_count * p.N / 16, p.err);
}
__device__ __forceinline__ bool y_ok(const DecodeArgs& p, const uint16_t* ptr, size_t n) {
  return in_buf(ptr, static_cast<const uint16_t*>(p.Y), n, p.err);
}
__device__ __forceinline__ float row_factor_at(const DecodeArgs& p, int tok) {
  return p.row_scale ? *ld_at(p.row_scale + tok, p.row_scale, (size_t)p.M, p.err) : 1.0f;
}
__device__ __forceinline__ bool flag_ok(const DecodeArgs& p, const int* f) {
  return in_buf(f, static_cast<const int*>(p.flags), (size_t)kDecodeMaxCtas, p.err);
}
__device__ __forceinline__ bool tile_ok(const DecodeArgs& p, const float* t) {
  return in_buf(t, static_cast<const float*>(p.tiles), p.tile_floats, p.err);
}

// The bf16-activation instantiations live in their own translation unit.
cudaError_t decode_dispatch_resident_bf16(const DecodeArgs& args, int mt, int nw, int apg_t, int ctas,
                                          int bytes, cudaStream_t stream);
cudaError_t decode_dispatch_streamk_bf16(const DecodeArgs& args, int mt, int apg_t, int ctas,
                                         cudaStream_t stream);

namespace {


constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRedStride = kDecodeBlockCols + 4;  // padded row of the partial tile
constexpr int kBatch = 8;                         // atoms per unit
constexpr int kSlots = 4;                         // activation ring slots
constexpr int kDecodeWaitTimedOut = 32;           // device error bit
// One staged activation row of a unit: 8 atoms x 64 k x 2 bytes, padded by
// 64 bytes so that consecutive rows fall in opposite halves of the 32 banks
// (a quarter-warp's 16-byte fragment loads cover two rows x 64 bytes).
constexpr int kActRow = kBatch * kAtomK * 2 + 64;
constexpr int kActRowVec = kActRow / 16;  // the same in 16-byte vectors

// Dynamic shared memory of the kernel for MT token octets and NG groups per
// unit. A ring slot holds one unit's activations (MT*8 rows) and the scale and
// zero-point pairs of its 8 strips.
template <int MT, int NG>
struct Smem {
  static constexpr int kActVecs = MT * 8 * kActRowVec;
  static constexpr int kSpVecs = kWarps * NG * 2;         // 32 bytes per (strip, group)
  static constexpr int kZpVecs = (kWarps * NG + 1) / 2;   // 8 bytes per (strip, group)
  static constexpr int kSlotVecs = kActVecs + kSpVecs + kZpVecs;
  static constexpr int kRingBytes = kSlots * kSlotVecs * 16;
  static constexpr int kSumFloats = kBatch * MT * 8;  // one buffer: [atom][token]
  static constexpr int kSumBytes = 2 * kSumFloats * 4;
  static constexpr int kRedBytes = MT * 8 * kRedStride * 4;
  static constexpr int kTotal = kRingBytes + kSumBytes + kRedBytes;
};

__device__ __forceinline__ void cp_async16(const void* dst_smem, const void* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst_smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(const void* dst_smem, const void* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst_smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// all but the most recently committed group of this thread's copies landed
__device__ __forceinline__ void cp_async_wait_prior() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Programmatic dependent launch: let the next grid on the stream be
// scheduled, and wait until the previous grid has completed and its writes
// are visible (a no-op when the launch had no programmatic dependency).
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits (at most about a second) until *flag is non-zero; false if it never
// became so.
__device__ __forceinline__ bool wait_flag(const int* flag) {
  if (ld_acquire(flag) != 0) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    __nanosleep(64);
    if (ld_acquire(flag) != 0) return true;
    if (global_ns() - t0 > 1000000000ull) return false;
  }
}

// D (16x8 f32) += A (16x16) * B (16x8), and the same with D = A * B; kB:
// both operands bf16, else both fp16.
template <bool kB>
__device__ __forceinline__ void mma_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  if (kB)
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
template <bool kB>
__device__ __forceinline__ void mma_first(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  if (kB)
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
  else
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// The four code pairs of one packed word (nibble p holds k-offset rev3(p)).
// fp16: as fp16x2 subnormals, c[0] = (k 0,1) and c[1] = (k 2,3) hold
// q * 2^-24, c[2] = (k 4,5) and c[3] = (k 6,7) hold 16 q * 2^-24. bf16 (kB):
// as bf16x2 normals 128 + q, every pair alike: a byte 0x0q under a high
// byte 0x43 is the bf16 128 + q (the low 4 of its 7 fraction bits count
// units at exponent 2^7). The even nibbles (one mask) and the odd ones (a
// shift and a mask) are paired with the 0x43 bytes by byte permutes; the
// offset 128 is taken out with the group's sums. (Written as shifts, masks
// and ORs, the same extraction measured 13-35% slower on the 7B decode
// layers.)
template <bool kB>
__device__ __forceinline__ void code_pairs(uint32_t w, uint32_t (&c)[4]) {
  if (kB) {
    const uint32_t t = w & 0x0F0F0F0Fu;         // nibbles 0 2 4 6 (k 0 2 1 3)
    const uint32_t u = (w >> 4) & 0x0F0F0F0Fu;  // nibbles 1 3 5 7 (k 4 6 5 7)
    c[0] = __byte_perm(t, 0x43434343u, 0x4240);  // (k 0, k 1)
    c[1] = __byte_perm(t, 0x43434343u, 0x4341);  // (k 2, k 3)
    c[2] = __byte_perm(u, 0x43434343u, 0x4240);  // (k 4, k 5)
    c[3] = __byte_perm(u, 0x43434343u, 0x4341);  // (k 6, k 7)
  } else {
    const uint32_t w8 = w >> 8;
    c[0] = w & 0x000F000Fu;
    c[1] = w8 & 0x000F000Fu;
    c[2] = w & 0x00F000F0u;
    c[3] = w8 & 0x00F000F0u;
  }
}

// The ones operand of the per-atom activation sums: fp16 2^-24 (the scale of
// the fp16 codes) or bf16 1.0.
template <bool kB>
__device__ __forceinline__ constexpr uint32_t ones_pair() { return kB ? 0x3F803F80u : 0x00010001u; }

// Factor from the accumulators to the product: 2^24 for the fp16 codes
// (q * 2^-24), 1 for the bf16 ones.
template <bool kB>
__device__ __forceinline__ constexpr float unscale() { return kB ? 1.0f : 16777216.0f; }

// fp32 -> the activation type's bits, round to nearest even.
template <bool kB>
__device__ __forceinline__ uint16_t to_act(float v) {
  if (kB) return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  return __half_as_ushort(__float2half_rn(v));
}

// A small non-negative integer as fp32 (exact, no conversion unit).
__device__ __forceinline__ float small_int_float(uint32_t v) {
  return __uint_as_float(0x4B000000u | v) - 8388608.0f;
}

// CTA whose run holds granule u when T granules are split among C CTAs
// (CTA c takes granules [floor(c T / C), floor((c + 1) T / C))).
__device__ __forceinline__ int owner_cta(long long u, long long T, int C) {
  return (int)(((u + 1) * C - 1) / T);
}


// Where one unit's data lives for this warp/lane.
struct Unit {
  int blk;       // 128-column block
  int a0;        // first atom
  int n;         // atoms in the unit (1..8)
  bool active;   // this warp's strip exists (N tail)
  const uint4* wp;
};

__device__ __forceinline__ Unit make_unit(const DecodeArgs& p, int blk, int a0, int n, int natoms,
                                          int nstrips, int warp, int lane) {
  Unit u;
  u.blk = blk;
  u.a0 = a0;
  u.n = n;
  const int strip = blk * kWarps + warp;
  u.active = strip < nstrips;
  const int st = u.active ? strip : 0;
  u.wp = p.Wq + ((size_t)st * natoms + a0) * 32 + lane;
  return u;
}

// Position of a unit: block, first atom, global atom index (blk * natoms + a0).
struct Pos {
  int blk, a0, g;
};

// Atoms of the unit starting at q: up to 8, within the block and the run.
__device__ __forceinline__ int unit_len(const Pos& q, int natoms, int run_end) {
  return min(kBatch, min(natoms - q.a0, run_end - q.g));
}

__device__ __forceinline__ void step(Pos& q, int n, int natoms) {
  q.g += n;
  q.a0 += n;
  if (q.a0 == natoms) {
    q.a0 = 0;
    ++q.blk;
  }
}

// Activations of a unit (rows 0..M-1, atoms a0..a0+n-1) into a ring slot.
__device__ __forceinline__ void stage_act(uint4* slot, const DecodeArgs& p, int a0, int n) {
  const int pieces = n * (kAtomK / 8);  // 16-byte pieces per row
  for (int idx = threadIdx.x; idx < p.M * (kBatch * kAtomK / 8); idx += kThreads) {
    const int row = idx >> 6, c = idx & 63;
    if (c < pieces)
      cp_async16(slot + row * kActRowVec + c, a_at(p, p.A + (size_t)row * p.K + (size_t)a0 * kAtomK + c * 8));
  }
}

// The scale pairs and zero-point pairs of the groups a unit touches, for the
// block's existing strips, into the ring slot after the activations.
template <int MT, int NG, int APG>
__device__ __forceinline__ void stage_meta(uint4* slot, const DecodeArgs& p, int blk, int a0, int n,
                                           int nstrips, int groups) {
  using SM = Smem<MT, NG>;
  const int ng = APG < kBatch ? n / APG : 1;  // groups present in the unit
  const int grp0 = a0 >> p.gshift;
  const int strips = min(kWarps, nstrips - blk * kWarps);
  const uint4* sp_src = reinterpret_cast<const uint4*>(p.Sp2);
  const uint2* zp_src = reinterpret_cast<const uint2*>(p.Zp);
  uint4* sp_dst = slot + SM::kActVecs;
  uint2* zp_dst = reinterpret_cast<uint2*>(slot + SM::kActVecs + SM::kSpVecs);
  for (int idx = threadIdx.x; idx < strips * NG * 3; idx += kThreads) {
    const int w = idx / (NG * 3), r = idx - w * (NG * 3);
    const size_t base = (size_t)(blk * kWarps + w) * groups + grp0;
    if (r < 2 * NG) {  // scale pairs: two 16-byte pieces per group
      if ((r >> 1) < ng) cp_async16(sp_dst + w * NG * 2 + r, sp_at(p, sp_src + base * 2 + r, groups));
    } else {           // zero-point pairs: 8 bytes per group
      const int g = r - 2 * NG;
      if (g < ng) cp_async8(zp_dst + w * NG + g, zp_at(p, zp_src + base + g, groups));
    }
  }
}

// sum_k a[k] over one atom of a staged unit, per token, into the sum buffer,
// at the codes' scale (times 2^-24 for fp16, the subnormal ones operand).
template <int MT, bool kB>
__device__ __forceinline__ void atom_sums(const uint4* slot, float* sb, int atom, int gq, int t) {
  constexpr uint32_t kOnes = ones_pair<kB>();
#pragma unroll
  for (int o = 0; o < MT; ++o) {
    const uint4* f = slot + (8 * o + gq) * kActRowVec + atom * 8 + t;
    const uint4 b0 = f[0], b1 = f[4];
    float d[4];
    mma_first<kB>(d, kOnes, kOnes, kOnes, kOnes, b0.x, b0.y);
    mma_acc<kB>(d, kOnes, kOnes, kOnes, kOnes, b0.z, b0.w);
    mma_acc<kB>(d, kOnes, kOnes, kOnes, kOnes, b1.x, b1.y);
    mma_acc<kB>(d, kOnes, kOnes, kOnes, kOnes, b1.z, b1.w);
    if (gq == 0) *reinterpret_cast<float2*>(sb + atom * MT * 8 + 8 * o + 2 * t) = make_float2(d[0], d[1]);
  }
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// One atom: the code pairs of the lane's four words (x, y: columns gq and
// gq + 8 in the first 32 k; z, v: the same columns in the last 32 k) against
// the staged activations at shared address `frag` (row gq, k-octet t of the
// atom). pe collects the q * 2^-24 pairs, po the 16 q * 2^-24 ones; each
// MMA's B operand is one adjacent register pair of a 16-byte fragment load.
// The fragment loads are volatile: they stay next to their MMAs instead of
// being hoisted a whole unit ahead into registers.
template <int MT, bool kFirst, bool kB>
__device__ __forceinline__ void atom_mma(float (&pe)[MT][4], float (&po)[MT][4],
                                         const uint32_t (&x)[4], const uint32_t (&y)[4],
                                         const uint32_t (&z)[4], const uint32_t (&v)[4],
                                         uint32_t frag) {
#pragma unroll
  for (int o = 0; o < MT; ++o) {
    const uint4 b = lds128(frag + o * 8 * kActRow);
    if (kFirst) {
      mma_first<kB>(pe[o], x[0], y[0], x[1], y[1], b.x, b.y);
      mma_first<kB>(po[o], x[2], y[2], x[3], y[3], b.z, b.w);
    } else {
      mma_acc<kB>(pe[o], x[0], y[0], x[1], y[1], b.x, b.y);
      mma_acc<kB>(po[o], x[2], y[2], x[3], y[3], b.z, b.w);
    }
  }
#pragma unroll
  for (int o = 0; o < MT; ++o) {
    const uint4 b = lds128(frag + o * 8 * kActRow + 64);
    mma_acc<kB>(pe[o], z[0], v[0], z[1], v[1], b.x, b.y);
    mma_acc<kB>(po[o], z[2], v[2], z[3], v[3], b.z, b.w);
  }
}

// End of a group of `na` atoms starting at atom a: acc += s * (P - z * S),
// with the group's scale pair sp (s[c], s[c+8]) and zero-point pair zp. For
// bf16 codes P holds 128 S more, taken out with the zero point.
template <int MT, bool kB>
__device__ __forceinline__ void apply_group(float (&acc)[MT][4], const float (&pe)[MT][4],
                                            const float (&po)[MT][4], uint32_t sp, uint32_t zp,
                                            const float* sb, int a, int na, int t) {
  const float s0 = __half2float(__ushort_as_half((unsigned short)(sp & 0xffffu)));
  const float s1 = __half2float(__ushort_as_half((unsigned short)(sp >> 16)));
  constexpr uint32_t kOff = kB ? 128u : 0u;
  const float nsz0 = -s0 * small_int_float(kOff + (zp & 15u));
  const float nsz1 = -s1 * small_int_float(kOff + ((zp >> 4) & 15u));
  constexpr float kHi = kB ? 1.0f : 0.0625f;  // weight of the po pairs
#pragma unroll
  for (int o = 0; o < MT; ++o) {
    const float* col = sb + a * MT * 8 + 8 * o + 2 * t;
    float2 S = *reinterpret_cast<const float2*>(col);
#pragma unroll
    for (int j = 1; j < kBatch; ++j)
      if (j < na) {
        const float2 v = *reinterpret_cast<const float2*>(col + j * MT * 8);
        S.x += v.x;
        S.y += v.y;
      }
    const float p0 = fmaf(po[o][0], kHi, pe[o][0]);
    const float p1 = fmaf(po[o][1], kHi, pe[o][1]);
    const float p2 = fmaf(po[o][2], kHi, pe[o][2]);
    const float p3 = fmaf(po[o][3], kHi, pe[o][3]);
    acc[o][0] = fmaf(nsz0, S.x, fmaf(s0, p0, acc[o][0]));  // column gq,     token 2t
    acc[o][1] = fmaf(nsz0, S.y, fmaf(s0, p1, acc[o][1]));  // column gq,     token 2t+1
    acc[o][2] = fmaf(nsz1, S.x, fmaf(s1, p2, acc[o][2]));  // column gq + 8, token 2t
    acc[o][3] = fmaf(nsz1, S.y, fmaf(s1, p3, acc[o][3]));  // column gq + 8, token 2t+1
  }
}

// One unit of this warp's strip, from ring slot `slot` (activations, group
// pairs) and the unit's atom sums `sb`. kFull: all 8 atoms present, the strip
// exists and the next unit (if refilled) is full too, so nothing is
// predicated; otherwise atoms past cu.n are skipped and the refill loads
// only the next unit's atoms.
template <int MT, int APG, bool kFull, bool kB>
__device__ __forceinline__ void unit_compute(const DecodeArgs& p, float (&acc)[MT][4], uint4 (&w)[kBatch],
                                             const Unit& cu, const Unit& nu, bool refill,
                                             const uint4* slot, const float* sb, int warp,
                                             int gq, int t) {
  constexpr int NG = kBatch / APG;
  using SM = Smem<MT, NG>;
  // B fragments: row gq, k-octet t
  const uint32_t frag = (uint32_t)__cvta_generic_to_shared(slot + gq * kActRowVec + t);
  const uint32_t* sps = reinterpret_cast<const uint32_t*>(slot + SM::kActVecs) + warp * NG * 8 + gq;
  const uint8_t* zps = reinterpret_cast<const uint8_t*>(slot + SM::kActVecs + SM::kSpVecs) + warp * NG * 8 + gq;
  float pe[MT][4], po[MT][4];
  const bool compute = kFull || cu.active;
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    // the codes leave w[u] before the next unit's atom u is loaded into it
    uint32_t x[4], y[4], z[4], v[4];
    code_pairs<kB>(w[u].x, x);
    code_pairs<kB>(w[u].y, y);
    code_pairs<kB>(w[u].z, z);
    code_pairs<kB>(w[u].w, v);
    if (refill && (kFull || u < nu.n)) w[u] = ldg_stream(wq_at(p, nu.wp + u * 32));
    if (compute && (kFull || u < cu.n)) {
      if (u % APG == 0)
        atom_mma<MT, true, kB>(pe, po, x, y, z, v, frag + u * 128);
      else
        atom_mma<MT, false, kB>(pe, po, x, y, z, v, frag + u * 128);
      if (APG < kBatch) {
        if (u % APG == APG - 1)
          apply_group<MT, kB>(acc, pe, po, sps[(u / APG) * 8], zps[(u / APG) * 8], sb, u + 1 - APG, APG, t);
      } else if (kFull ? u == kBatch - 1 : u == cu.n - 1) {
        apply_group<MT, kB>(acc, pe, po, sps[0], zps[0], sb, 0, kFull ? kBatch : cu.n, t);
      }
    }
  }
}

// MT: token octets (1: M <= 8, 2: M <= 16). APG: atoms per group, 1, 2 or 4;
// 8 stands for groups of 8 or more atoms (or one group per column), whose
// boundaries fall on unit starts.
template <int MT, int APG, bool kB>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const DecodeArgs p) {
  constexpr int NG = kBatch / APG;  // groups per unit
  using SM = Smem<MT, NG>;
  extern __shared__ __align__(16) uint8_t smem[];
  uint4* ring = reinterpret_cast<uint4*>(smem);
  float* sums = reinterpret_cast<float*>(smem + SM::kRingBytes);
  float* red = reinterpret_cast<float*>(smem + SM::kRingBytes + SM::kSumBytes);

  allow_dependent_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, t = lane & 3;  // mma groupID / thread-in-group
  const int N = p.N, K = p.K, M = p.M;
  const int natoms = K / kAtomK;
  const int nstrips = N / kStripCols;
  const int nblk = (N + kDecodeBlockCols - 1) / kDecodeBlockCols;
  const int groups = (natoms + (1 << p.gshift) - 1) >> p.gshift;
  const int C = gridDim.x;
  const int gr = p.granule;
  const long long T = (long long)nblk * natoms / gr;  // granules
  const int run_begin = (int)((long long)blockIdx.x * T / C) * gr;
  const int run_end = (int)((long long)(blockIdx.x + 1) * T / C) * gr;

  // unit cursors: the current unit, the next one (weights), and the one two
  // ahead (activation staging)
  Pos sq;
  sq.blk = run_begin / natoms;
  sq.a0 = run_begin - sq.blk * natoms;
  sq.g = run_begin;
  Pos nq = sq;
  Unit cu = make_unit(p, sq.blk, sq.a0, unit_len(sq, natoms, run_end), natoms, nstrips, warp, lane);
  step(nq, cu.n, natoms);
  const bool two = nq.g < run_end;  // the run has a second unit
  const int n1 = two ? unit_len(nq, natoms, run_end) : 0;
  uint4 w[kBatch];
  auto load_first = [&]() {
    if (cu.active) {
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (u < cu.n) w[u] = ldg_stream(wq_at(p, cu.wp + u * 32));
    }
    stage_meta<MT, NG, APG>(ring, p, sq.blk, sq.a0, cu.n, nstrips, groups);
    if (two) stage_meta<MT, NG, APG>(ring + SM::kSlotVecs, p, nq.blk, nq.a0, n1, nstrips, groups);
  };
  if (p.early_weights) load_first();
  grid_dependency_wait();
  if (!p.early_weights) load_first();

  // token rows past M stay zero (never staged)
  if (M < MT * 8) {
    const int per = (MT * 8 - M) * kActRowVec;
    for (int idx = threadIdx.x; idx < kSlots * per; idx += kThreads) {
      const int s = idx / per, r = idx - s * per;
      ring[s * SM::kSlotVecs + M * kActRowVec + r] = make_uint4(0, 0, 0, 0);
    }
  }
  stage_act(ring, p, sq.a0, cu.n);
  if (two) stage_act(ring + SM::kSlotVecs, p, nq.a0, n1);
  cp_async_commit();
  step(sq, cu.n, natoms);
  if (two) step(sq, n1, natoms);
  // the third unit in a group of its own, left in flight
  if (sq.g < run_end) {
    const int n2 = unit_len(sq, natoms, run_end);
    stage_meta<MT, NG, APG>(ring + 2 * SM::kSlotVecs, p, sq.blk, sq.a0, n2, nstrips, groups);
    stage_act(ring + 2 * SM::kSlotVecs, p, sq.a0, n2);
    step(sq, n2, natoms);
  }
  cp_async_commit();  // sq: three units ahead of the current one
  cp_async_wait_prior();
  __syncthreads();
  if (warp < cu.n) atom_sums<MT, kB>(ring, sums, warp, gq, t);

  float acc[MT][4];
#pragma unroll
  for (int o = 0; o < MT; ++o) acc[o][0] = acc[o][1] = acc[o][2] = acc[o][3] = 0.f;
  int seg_a0 = cu.a0;  // first atom of the current segment
  int slot = 0;        // ring slot of the current unit

  for (int i = 0;; ++i) {
    const bool has_next = nq.g < run_end;
    const Unit nu = has_next ? make_unit(p, nq.blk, nq.a0, unit_len(nq, natoms, run_end), natoms,
                                         nstrips, warp, lane)
                             : cu;
    const int slot1 = (slot + 1) & (kSlots - 1);
    const int slot3 = (slot + 3) & (kSlots - 1);
    // the next unit's copies (committed two units ago) landed; the copies
    // committed one unit ago may still be in flight
    cp_async_wait_prior();
    __syncthreads();  // the next unit's slot and this unit's sums are visible; slot i-1 is free
    if (sq.g < run_end) {
      const int n3 = unit_len(sq, natoms, run_end);
      stage_meta<MT, NG, APG>(ring + slot3 * SM::kSlotVecs, p, sq.blk, sq.a0, n3, nstrips, groups);
      stage_act(ring + slot3 * SM::kSlotVecs, p, sq.a0, n3);
      step(sq, n3, natoms);
    }
    cp_async_commit();
    if (has_next && warp < nu.n)
      atom_sums<MT, kB>(ring + slot1 * SM::kSlotVecs, sums + ((i + 1) & 1) * SM::kSumFloats, warp, gq, t);

    const bool refill = has_next && nu.active;
    const uint4* cur = ring + slot * SM::kSlotVecs;
    const float* sb = sums + (i & 1) * SM::kSumFloats;
    if (cu.active && cu.n == kBatch && refill && nu.n == kBatch)
      unit_compute<MT, APG, true, kB>(p, acc, w, cu, nu, true, cur, sb, warp, gq, t);
    else
      unit_compute<MT, APG, false, kB>(p, acc, w, cu, nu, refill, cur, sb, warp, gq, t);

    if (!has_next || nu.blk != cu.blk) {
      // ---- end of a segment: atoms [seg_a0, cu.a0 + cu.n) of block cu.blk
      const int b = cu.blk;
      const bool head = seg_a0 == 0;  // holds the block's first atom
      const bool whole = head && cu.a0 + cu.n == natoms;
      if (cu.active) {
        constexpr float kUnscale = unscale<kB>();
#pragma unroll
        for (int o = 0; o < MT; ++o) {
          const int tok = 8 * o + 2 * t;
          const int col = kStripCols * warp + gq;
          red[tok * kRedStride + col] = acc[o][0] * kUnscale;
          red[(tok + 1) * kRedStride + col] = acc[o][1] * kUnscale;
          red[tok * kRedStride + col + 8] = acc[o][2] * kUnscale;
          red[(tok + 1) * kRedStride + col + 8] = acc[o][3] * kUnscale;
        }
      }
#pragma unroll
      for (int o = 0; o < MT; ++o) acc[o][0] = acc[o][1] = acc[o][2] = acc[o][3] = 0.f;
      constexpr int kTileFloats = MT * 8 * kDecodeBlockCols;
      const int col0 = b * kDecodeBlockCols;
      const int total = M * kDecodeBlockCols;
      if (whole) {
        __syncthreads();
        for (int e = threadIdx.x; e < total; e += kThreads) {
          const int tok = e >> 7, col = e & (kDecodeBlockCols - 1);
          if (col0 + col < N && y_ok(p, p.Y + (size_t)tok * N + col0 + col, (size_t)M * N))
            p.Y[(size_t)tok * N + col0 + col] =
                to_act<kB>(red[tok * kRedStride + col] * row_factor_at(p, tok));
        }
      } else if (head) {
        // finish the block: the later contributors' tiles, in CTA order
        const int c_last = owner_cta(((long long)(b + 1) * natoms - 1) / gr, T, C);
        const int others = c_last - (int)blockIdx.x;
        bool ok = true;
        for (int j = threadIdx.x; j < others; j += kThreads) {
          int* f = p.flags + blockIdx.x + 1 + j;
          if (!flag_ok(p, f))
            ok = false;
          else if (wait_flag(f))
            *f = 0;  // lowered for the next call
          else
            ok = false;
        }
        if (!ok) atomicOr(p.err, kDecodeWaitTimedOut);
        __syncthreads();  // (acquire by the waiting threads, then the barrier)
        // own partial first, then the tiles in CTA order (deterministic); the
        // values of kAhead contributors are loaded at a time
        constexpr int kPerThread = (kTileFloats + kThreads - 1) / kThreads;
        constexpr int kAhead = 4 / MT;
        float v[kPerThread];
#pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
          const int e = threadIdx.x + k * kThreads;
          v[k] = e < total ? red[(e >> 7) * kRedStride + (e & (kDecodeBlockCols - 1))] : 0.f;
        }
        for (int j0 = 1; j0 <= others; j0 += kAhead) {
          float tv[kAhead][kPerThread];
#pragma unroll
          for (int jj = 0; jj < kAhead; ++jj) {
            const float* tile = p.tiles + (size_t)(blockIdx.x + j0 + jj) * kTileFloats;
#pragma unroll
            for (int k = 0; k < kPerThread; ++k) {
              const int e = threadIdx.x + k * kThreads;
              tv[jj][k] = (j0 + jj <= others && e < total && tile_ok(p, tile + e)) ? __ldcg(tile + e) : 0.f;
            }
          }
#pragma unroll
          for (int jj = 0; jj < kAhead; ++jj)
            if (j0 + jj <= others)
#pragma unroll
              for (int k = 0; k < kPerThread; ++k) v[k] += tv[jj][k];
        }
#pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
          const int e = threadIdx.x + k * kThreads;
          const int col = e & (kDecodeBlockCols - 1);
          if (e < total && col0 + col < N && y_ok(p, p.Y + (size_t)(e >> 7) * N + col0 + col, (size_t)M * N))
            p.Y[(size_t)(e >> 7) * N + col0 + col] = to_act<kB>(v[k] * row_factor_at(p, e >> 7));
        }
      } else {
        // a run that starts inside block b: publish the partial tile, then
        // raise the flag (release after the CTA barrier covers every
        // thread's tile stores)
        __syncthreads();
        float* my = p.tiles + (size_t)blockIdx.x * kTileFloats;
        for (int e = threadIdx.x; e < total; e += kThreads) {
          const int tok = e >> 7, col = e & (kDecodeBlockCols - 1);
          if (tile_ok(p, my + e)) my[e] = red[tok * kRedStride + col];
        }
        __syncthreads();
        if (threadIdx.x == 0 && flag_ok(p, p.flags + blockIdx.x)) st_release(p.flags + blockIdx.x, 1);
      }
      __syncthreads();  // the partial tile buffer is reused by the next segment
      seg_a0 = nu.a0;
    }
    if (!has_next) break;
    cu = nu;
    slot = slot1;
    step(nq, cu.n, natoms);
  }
}

// ---------------------------------------------------------------------------
// Strip variant, for problems whose activations (M x K) fit in shared memory.
// CTA c owns whole strips [c S / C, (c + 1) S / C) of the S strips, over all
// of K, so no output column is shared between CTAs: no workspace, no flags,
// no cross-CTA fix-up. The CTA's atoms, strip-major (a contiguous range of
// Wq), are split among its 8 warps in equal ranges that start at group
// boundaries; each warp streams its range through registers (one unit of up
// to 8 atoms ahead) with no CTA barrier. A strip that a warp covers whole goes
// to Y from registers; a strip shared by warps is summed after the CTA's one
// final barrier, in warp order, from the warps' partials in shared memory.
// A (with a zero row for tokens past M), the per-token sums of every atom and
// the group pairs of the CTA's strips are staged once.

// One atom against resident activations: as atom_mma, with the fragments of
// token octet 0 at shared address fa and of octet 1 at fb.
template <int MT, bool kFirst, bool kB>
__device__ __forceinline__ void atom_mma_rows(float (&pe)[MT][4], float (&po)[MT][4],
                                              const uint32_t (&x)[4], const uint32_t (&y)[4],
                                              const uint32_t (&z)[4], const uint32_t (&v)[4],
                                              uint32_t fa, uint32_t fb) {
#pragma unroll
  for (int o = 0; o < MT; ++o) {
    const uint4 b = lds128(o == 0 ? fa : fb);
    if (kFirst) {
      mma_first<kB>(pe[o], x[0], y[0], x[1], y[1], b.x, b.y);
      mma_first<kB>(po[o], x[2], y[2], x[3], y[3], b.z, b.w);
    } else {
      mma_acc<kB>(pe[o], x[0], y[0], x[1], y[1], b.x, b.y);
      mma_acc<kB>(po[o], x[2], y[2], x[3], y[3], b.z, b.w);
    }
  }
#pragma unroll
  for (int o = 0; o < MT; ++o) {
    const uint4 b = lds128((o == 0 ? fa : fb) + 64);
    mma_acc<kB>(pe[o], z[0], v[0], z[1], v[1], b.x, b.y);
    mma_acc<kB>(po[o], z[2], v[2], z[3], v[3], b.z, b.w);
  }
}

// One unit of n atoms (a group boundary at its start) of the warp's strip,
// activations resident: fa/fb address the unit's first atom, sps/zps its
// first group's pairs, sb its first atom's sums. The next unit's nn atoms are
// loaded from nwp into w as the codes leave it (when refill).
template <int MT, int APG, bool kFull, bool kB>
__device__ __forceinline__ void resident_unit(const DecodeArgs& p, float (&acc)[MT][4], uint4 (&w)[kBatch], int n, int nn,
                                           const uint4* nwp, bool refill, uint32_t fa, uint32_t fb,
                                           const uint32_t* sps, const uint8_t* zps, const float* sb,
                                           int t) {
  float pe[MT][4], po[MT][4];
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    uint32_t x[4], y[4], z[4], v[4];
    code_pairs<kB>(w[u].x, x);
    code_pairs<kB>(w[u].y, y);
    code_pairs<kB>(w[u].z, z);
    code_pairs<kB>(w[u].w, v);
    if (refill && (kFull || u < nn)) w[u] = ldg_stream(wq_at(p, nwp + u * 32));
    if (kFull || u < n) {
      if (u % APG == 0)
        atom_mma_rows<MT, true, kB>(pe, po, x, y, z, v, fa + u * 128, fb + u * 128);
      else
        atom_mma_rows<MT, false, kB>(pe, po, x, y, z, v, fa + u * 128, fb + u * 128);
      if (APG < kBatch) {
        if (u % APG == APG - 1)
          apply_group<MT, kB>(acc, pe, po, sps[(u / APG) * 8], zps[(u / APG) * 8], sb, u + 1 - APG, APG, t);
      } else if (kFull ? u == kBatch - 1 : u == n - 1) {
        apply_group<MT, kB>(acc, pe, po, sps[0], zps[0], sb, 0, kFull ? kBatch : n, t);
      }
    }
  }
}

template <int MT, int APG, int NW, bool kSilu, bool kB>
__global__ void __launch_bounds__(NW * 32, 16 / NW) decode_resident_kernel(const DecodeArgs p) {
  constexpr int kSeg = MT * 8 * kStripCols;  // floats of one partial strip
  extern __shared__ __align__(16) uint8_t smem[];
  float* sums = reinterpret_cast<float*>(smem + p.sums_off);
  const uint32_t* meta_sp = reinterpret_cast<const uint32_t*>(smem + p.meta_off);
  const uint8_t* meta_zp = smem + p.zp_off;
  float* red = reinterpret_cast<float*>(smem + p.red_off);  // [warp][2][kSeg]

  allow_dependent_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, t = lane & 3;
  const int M = p.M, K = p.K, N = p.N;
  const int natoms = K / kAtomK;
  const int nstrips = N / kStripCols;
  const int G = (natoms + (1 << p.gshift) - 1) >> p.gshift;  // groups per strip
  const int gr = p.granule;
  // this CTA's strips: units [u0, u1) of the S strips, or with the fused
  // gate/up epilogue of the S/2 strip pairs (pair q: gate strip q and up
  // strip S/2 + q). Its nv "virtual" strips v (the unit strips in order; for
  // pairs the gate strips, then the up strips) hold virtual atoms
  // [0, nv natoms), split into NW warp ranges of whole granules; warp w
  // starts at wbeg(w). Virtual strip v is strip gstrip(v) of Wq and Y.
  const int C = gridDim.x;
  const int units = kSilu ? nstrips / 2 : nstrips;
  const int u0 = (int)((long long)blockIdx.x * units / C);
  const int u1 = (int)((long long)(blockIdx.x + 1) * units / C);
  const int nu = u1 - u0, nv = kSilu ? 2 * nu : nu;
  auto gstrip = [&](int v) { return kSilu && v >= nu ? nstrips / 2 + u0 + (v - nu) : u0 + v; };
  const int Lg = nv * (natoms / gr);
  auto wbeg = [&](int w) { return gr * (int)((long long)w * Lg / NW); };
  const int run_begin = wbeg(warp), run_end = wbeg(warp + 1);

  int strip = run_begin / natoms, a = run_begin - strip * natoms, g = run_begin;
  int n = g < run_end ? min(kBatch - (a & (kBatch - 1)), min(natoms - a, run_end - g)) : 0;
  // the lane's word of virtual strip v, atom a
  auto wptr = [&](int v, int a_) { return p.Wq + ((size_t)gstrip(v) * natoms + a_) * 32 + lane; };
  const uint4* wp = wptr(strip, a);
  // consecutive virtual strips are consecutive in Wq (strip-major, atoms in
  // order), except from the last gate strip to the first up strip
  const int jump_v = kSilu ? nu : -1;
  const int jump = (nstrips / 2 - nu) * natoms * 32;
  uint4 w[kBatch];
  auto prefetch = [&]() {
    if (g < run_end) {
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (u < n) w[u] = ldg_stream(wq_at(p, wp + u * 32));
    }
    // group pairs of the CTA's strips, in virtual strip order: record
    // v G + grp of the stage is record gstrip(v) G + grp of Sp/Zp
    const int nrec = nv * G;
    const uint4* sp_src = reinterpret_cast<const uint4*>(p.Sp2);
    const uint2* zp_src = reinterpret_cast<const uint2*>(p.Zp);
    for (int i = threadIdx.x; i < 3 * nrec; i += (NW * 32)) {
      const int r = i < 2 * nrec ? i >> 1 : i - 2 * nrec;  // staged record
      const int v = r / G;
      const size_t rg = (size_t)gstrip(v) * G + (r - v * G);  // its record in Sp/Zp
      if (i < 2 * nrec)
        cp_async16(reinterpret_cast<uint4*>(smem + p.meta_off) + i, sp_at(p, sp_src + rg * 2 + (i & 1), G));
      else
        cp_async8(reinterpret_cast<uint2*>(smem + p.zp_off) + r, zp_at(p, zp_src + rg, G));
    }
  };
  if (p.early_weights) prefetch();
  grid_dependency_wait();
  if (!p.early_weights) prefetch();

  // activation rows 0..M-1, then the zero row M (token rows past M read it)
  {
    uint4* act = reinterpret_cast<uint4*>(smem);
    const int row_vecs = p.act_row / 16, per_row = K / 8;
    for (int i = threadIdx.x; i < M * per_row; i += (NW * 32)) {
      const int row = i / per_row, c = i - row * per_row;
      cp_async16(act + row * row_vecs + c, a_at(p, p.A + (size_t)row * K + c * 8));
    }
    for (int c = threadIdx.x; c < row_vecs; c += (NW * 32)) act[M * row_vecs + c] = make_uint4(0, 0, 0, 0);
  }
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();
  const uint32_t act_s = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t fa0 = act_s + (uint32_t)((gq < M ? gq : M) * p.act_row + 16 * t);
  const uint32_t fb0 = act_s + (uint32_t)((8 + gq < M ? 8 + gq : M) * p.act_row + 16 * t);
  // per-token sums of every atom, sum_k 2^-24 a[k]: row sums of the staged
  // rows against a ones B operand (fp16 2^-24). One MMA chain sums a block of
  // 16 atoms of one token; lane (gq, t) loads atoms gq and gq + 8 of the
  // block as A fragments (the order of k within a row does not matter to a
  // sum). Atoms past K read the zero row.
  {
    constexpr uint32_t kOnes = ones_pair<kB>();
    const int nab = (natoms + 15) >> 4;  // atom blocks per token
    const uint32_t zero_row = act_s + (uint32_t)(M * p.act_row + 16 * t);
    for (int b = warp; b < M * nab; b += NW) {
      const int tok = b / nab, at = (b - tok * nab) * 16 + gq;
      const uint32_t row = act_s + (uint32_t)(tok * p.act_row + 16 * t);
      // lanes of odd gq read the atom's second 64 bytes first: the two rows of
      // a quarter-warp then fall in opposite halves of the banks
      const uint32_t first = (gq & 1) * 64, second = 64 - first;
      const uint32_t lo = at < natoms ? row + at * 128 : zero_row;
      const uint32_t hi = at + 8 < natoms ? row + (at + 8) * 128 : zero_row;
      const uint4 l0 = lds128(lo + first), h0 = lds128(hi + first);
      const uint4 l1 = lds128(lo + second), h1 = lds128(hi + second);
      float d[4], e[4];
      mma_first<kB>(d, l0.x, h0.x, l0.y, h0.y, kOnes, kOnes);
      mma_first<kB>(e, l0.z, h0.z, l0.w, h0.w, kOnes, kOnes);
      mma_acc<kB>(d, l1.x, h1.x, l1.y, h1.y, kOnes, kOnes);
      mma_acc<kB>(e, l1.z, h1.z, l1.w, h1.w, kOnes, kOnes);
      if (t == 0) {
        if (at < natoms) sums[at * MT * 8 + tok] = d[0] + e[0];
        if (at + 8 < natoms) sums[(at + 8) * MT * 8 + tok] = d[2] + e[2];
      }
    }
  }
  __syncthreads();
  // the first unit's codes are not taken apart before this point, so the
  // staging and sums above overlap its loads
#pragma unroll
  for (int u = 0; u < kBatch; ++u) asm volatile("" : "+r"(w[u].x), "+r"(w[u].y), "+r"(w[u].z), "+r"(w[u].w));

  // element j of token octet o of this lane: token 8o + 2t + (j & 1), column gq + 8 (j >> 1)
  auto elem = [&](int o, int j) { return (8 * o + 2 * t + (j & 1)) * kStripCols + gq + 8 * (j >> 1); };
  // the finished virtual strip s: to Y, or with the fused epilogue to the
  // CTA's fp32 tile ([virtual strip][token][column])
  float* ytile = reinterpret_cast<float*>(smem + p.ytile_off);
  auto store_y = [&](const float (&v)[MT][4], int s, float scale) {
#pragma unroll
    for (int o = 0; o < MT; ++o)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tok = 8 * o + 2 * t + (j & 1);
        if (tok >= M) continue;  // rows past M hold nothing (the zero row)
        const float val = v[o][j] * scale * row_factor_at(p, tok);
        if (kSilu)
          ytile[s * p.ytile_stride + tok * kStripCols + gq + 8 * (j >> 1)] = val;
        else if (y_ok(p, p.Y + (size_t)tok * N + gstrip(s) * kStripCols + gq + 8 * (j >> 1), (size_t)M * N))
          p.Y[(size_t)tok * N + gstrip(s) * kStripCols + gq + 8 * (j >> 1)] = to_act<kB>(val);
      }
  };
  constexpr float kUnscale = unscale<kB>();
  float acc[MT][4];
#pragma unroll
  for (int o = 0; o < MT; ++o) acc[o][0] = acc[o][1] = acc[o][2] = acc[o][3] = 0.f;
  const int first_strip = strip;
  int seg_a0 = a;
  bool first_seg = true;
  int heads = 0;  // bit s: the segment in red slot s starts its strip
  while (g < run_end) {
    int s2 = strip, a2 = a + n;
    if (a2 == natoms) {
      a2 = 0;
      ++s2;
    }
    const int g2 = g + n;
    const bool has_next = g2 < run_end;
    const int n2 = has_next ? min(kBatch - (a2 & (kBatch - 1)), min(natoms - a2, run_end - g2)) : 0;
    const uint4* wp2 = has_next ? wp + n * 32 + (s2 == jump_v && s2 != strip ? jump : 0) : wp;
    const int rec = strip * G + (a >> p.gshift);
    const uint32_t* sps = meta_sp + rec * 8 + gq;
    const uint8_t* zps = meta_zp + rec * 8 + gq;
    const float* sb = sums + a * MT * 8;
    const uint32_t fa = fa0 + a * 128, fb = fb0 + a * 128;
    if (n == kBatch && n2 == kBatch)
      resident_unit<MT, APG, true, kB>(p, acc, w, n, n2, wp2, true, fa, fb, sps, zps, sb, t);
    else
      resident_unit<MT, APG, false, kB>(p, acc, w, n, n2, wp2, has_next, fa, fb, sps, zps, sb, t);
    if (!has_next || s2 != strip) {
      // ---- end of a segment: atoms [seg_a0, a + n) of `strip`
      if (seg_a0 == 0 && a + n == natoms && !(kSilu && p.whole_in_red)) {
        store_y(acc, strip, kUnscale);  // the whole strip
      } else {
        const int rs = first_seg ? 0 : 1;
        float* dst = red + (warp * 2 + rs) * kSeg;
#pragma unroll
        for (int o = 0; o < MT; ++o)
#pragma unroll
          for (int j = 0; j < 4; ++j) dst[elem(o, j)] = acc[o][j] * kUnscale;
        if (seg_a0 == 0) heads |= 1 << rs;
      }
#pragma unroll
      for (int o = 0; o < MT; ++o) acc[o][0] = acc[o][1] = acc[o][2] = acc[o][3] = 0.f;
      seg_a0 = a2;
      first_seg = false;
    }
    strip = s2;
    a = a2;
    g = g2;
    n = n2;
    wp = wp2;
  }
  __syncthreads();
#pragma unroll 1
  for (int rs = 0; rs < 2; ++rs) {
    if (!(heads >> rs & 1)) continue;
    // this warp's segment in red slot rs starts strip s; the rest of the
    // strip is the first segment of each following warp that starts inside it
    const int s = rs == 0 ? first_strip : (run_end - 1) / natoms;
    const int strip_end = (s + 1) * natoms;
    float v[MT][4];
    const float* own = red + (warp * 2 + rs) * kSeg;
#pragma unroll
    for (int o = 0; o < MT; ++o)
#pragma unroll
      for (int j = 0; j < 4; ++j) v[o][j] = own[elem(o, j)];
    for (int w2 = warp + 1; w2 < NW && wbeg(w2) < strip_end; ++w2) {
      if (wbeg(w2) == wbeg(w2 + 1)) continue;  // an empty range
      const float* part = red + (w2 * 2) * kSeg;
#pragma unroll
      for (int o = 0; o < MT; ++o)
#pragma unroll
        for (int j = 0; j < 4; ++j) v[o][j] += part[elem(o, j)];
    }
    store_y(v, s, 1.f);
  }
  if (kSilu) {
    // Y[tok][16 (u0 + q) + c] = silu(gate) * up for the CTA's pairs q
    __syncthreads();
    const int half = N / 2;
    for (int e = threadIdx.x; e < nu * M * kStripCols; e += NW * 32) {
      const int q = e / (M * kStripCols), r = e - q * (M * kStripCols);
      const int tok = r / kStripCols, c = r - tok * kStripCols;
      const float gv = ytile[q * p.ytile_stride + tok * kStripCols + c];
      const float uv = ytile[(nu + q) * p.ytile_stride + tok * kStripCols + c];
      if (y_ok(p, p.Y + (size_t)tok * half + (u0 + q) * kStripCols + c, (size_t)M * half))
        p.Y[(size_t)tok * half + (u0 + q) * kStripCols + c] = to_act<kB>(gv / (1.0f + expf(-gv)) * uv);
    }
  }
}

// Shared memory one CTA may use with two CTAs per SM (228 KiB per SM, 1 KiB
// of it reserved per CTA), and the most one CTA may use.
constexpr int kTwoCtaSmem = 113 * 1024;
constexpr int kOneCtaSmem = 227 * 1024;

// Layout of the strip variant's shared memory for `ctas` CTAs of `nw` warps:
// A (rows 0..M), the atom sums, the scale and zero-point pairs of a CTA's
// strips and the warps' partial strips; with the fused gate/up epilogue also
// the CTA's finished strips (placed as DecodeArgs describes). False if it
// exceeds `limit` bytes.
bool strip_layout(int M, int N, int K, int gshift, int ctas, int nw, int limit, bool silu,
                  DecodeArgs* a, int* bytes) {
  const long mt = M <= 8 ? 1 : 2;
  const long natoms = K / kAtomK;
  const long nstrips = N / kStripCols;
  const long G = (natoms + (1L << gshift) - 1) >> gshift;
  // strips of the busiest CTA (with the fused gate/up epilogue: both strips
  // of its pairs)
  const long strips_max = silu ? 2 * ((nstrips / 2 + ctas - 1) / ctas) : (nstrips + ctas - 1) / ctas;
  const long act_row = 2L * K + 64;
  // the fused epilogue's finished strips: over their own scale records, else
  // over the activation rows, else apart
  const long slot = mt * 8 * kStripCols * 4;
  const bool on_meta = silu && G * 32 >= slot;
  const bool on_rows = silu && !on_meta && strips_max <= nw;
  const long ytile_bytes = silu ? strips_max * slot : 0;
  const long act_bytes = (M + 1) * act_row;
  const long sums_off = ((on_rows && ytile_bytes > act_bytes ? ytile_bytes : act_bytes) + 15) & ~15L;
  const long meta_off = sums_off + ((natoms * mt * 8 * 4 + 15) & ~15L);
  const long zp_off = meta_off + strips_max * G * 32;
  const long red_off = zp_off + ((strips_max * G * 8 + 15) & ~15L);
  const long red_end = red_off + (long)nw * 2 * mt * 8 * kStripCols * 4;
  const long ytile_off = on_meta ? meta_off : on_rows ? 0 : red_end;
  const long total = silu && !on_meta && !on_rows ? red_end + ytile_bytes : red_end;
  if (total > limit) return false;
  a->silu = silu ? 1 : 0;
  a->ytile_off = (int)ytile_off;
  a->ytile_stride = (int)((on_meta ? G * 32 : slot) / 4);
  a->whole_in_red = on_rows ? 1 : 0;
  a->act_row = (int)act_row;
  a->sums_off = (int)sums_off;
  a->meta_off = (int)meta_off;
  a->zp_off = (int)zp_off;
  a->red_off = (int)red_off;
  *bytes = (int)total;
  return true;
}

template <int MT, int APG, int NW, bool kB>
cudaError_t launch_strip(const DecodeArgs& args, int ctas, int bytes, cudaStream_t stream) {
  auto kern = args.silu ? decode_resident_kernel<MT, APG, NW, true, kB>
                        : decode_resident_kernel<MT, APG, NW, false, kB>;
  cudaError_t e = set_max_smem_once(reinterpret_cast<const void*>(kern),
                                    NW == 8 ? kTwoCtaSmem : kOneCtaSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = (size_t)bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args);
}

template <int MT, int NW, bool kB>
cudaError_t launch_strip_mt(const DecodeArgs& args, int apg_t, int ctas, int bytes,
                            cudaStream_t stream) {
  switch (apg_t) {
    case 1: return launch_strip<MT, 1, NW, kB>(args, ctas, bytes, stream);
    case 2: return launch_strip<MT, 2, NW, kB>(args, ctas, bytes, stream);
    case 4: return launch_strip<MT, 4, NW, kB>(args, ctas, bytes, stream);
    default: return launch_strip<MT, 8, NW, kB>(args, ctas, bytes, stream);
  }
}

// The resident variant for `mt` token octets and `nw` warps per CTA.
template <bool kB>
cudaError_t dispatch_resident(const DecodeArgs& args, int mt, int nw, int apg_t, int ctas, int bytes,
                              cudaStream_t stream) {
  if (nw == 8)
    return mt == 1 ? launch_strip_mt<1, 8, kB>(args, apg_t, ctas, bytes, stream)
                   : launch_strip_mt<2, 8, kB>(args, apg_t, ctas, bytes, stream);
  return mt == 1 ? launch_strip_mt<1, 16, kB>(args, apg_t, ctas, bytes, stream)
                 : launch_strip_mt<2, 16, kB>(args, apg_t, ctas, bytes, stream);
}

template <int MT, int APG, bool kB>
cudaError_t launch_variant(const DecodeArgs& args, int ctas, cudaStream_t stream) {
  auto kern = decode_kernel<MT, APG, kB>;
  constexpr int kSmem = Smem<MT, kBatch / APG>::kTotal;
  cudaError_t e = set_max_smem_once(reinterpret_cast<const void*>(kern), kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args);
}

template <int MT, bool kB>
cudaError_t launch_mt(const DecodeArgs& args, int apg_t, int ctas, cudaStream_t stream) {
  switch (apg_t) {
    case 1: return launch_variant<MT, 1, kB>(args, ctas, stream);
    case 2: return launch_variant<MT, 2, kB>(args, ctas, stream);
    case 4: return launch_variant<MT, 4, kB>(args, ctas, stream);
    default: return launch_variant<MT, 8, kB>(args, ctas, stream);
  }
}

// The stream-K variant for `mt` token octets.
template <bool kB>
cudaError_t dispatch_streamk(const DecodeArgs& args, int mt, int apg_t, int ctas, cudaStream_t stream) {
  return mt == 1 ? launch_mt<1, kB>(args, apg_t, ctas, stream) : launch_mt<2, kB>(args, apg_t, ctas, stream);
}

}  // namespace
}  // namespace w4a16
