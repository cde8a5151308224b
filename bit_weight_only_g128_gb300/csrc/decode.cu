// Decode path of the W4A16 linear layer: up to 16 rows of activations. Here
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
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
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

// D (16x8 f32) += A (16x16 f16) * B (16x8 f16), and the same with D = A * B.
__device__ __forceinline__ void mma_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_first(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// The four code pairs of one packed word (nibble p holds k-offset rev3(p)) as
// fp16x2 subnormals: c[0] = (k 0,1) and c[1] = (k 2,3) hold q * 2^-24,
// c[2] = (k 4,5) and c[3] = (k 6,7) hold 16 q * 2^-24.
__device__ __forceinline__ void code_pairs(uint32_t w, uint32_t (&c)[4]) {
  const uint32_t w8 = w >> 8;
  c[0] = w & 0x000F000Fu;
  c[1] = w8 & 0x000F000Fu;
  c[2] = w & 0x00F000F0u;
  c[3] = w8 & 0x00F000F0u;
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
};

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
      cp_async16(slot + row * kActRowVec + c, p.A + (size_t)row * p.K + (size_t)a0 * kAtomK + c * 8);
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
      if ((r >> 1) < ng) cp_async16(sp_dst + w * NG * 2 + r, sp_src + base * 2 + r);
    } else {           // zero-point pairs: 8 bytes per group
      const int g = r - 2 * NG;
      if (g < ng) cp_async8(zp_dst + w * NG + g, zp_src + base + g);
    }
  }
}

// sum_k 2^-24 a[k] over one atom of a staged unit, per token, into the sum
// buffer (the ones operand is the fp16 subnormal 2^-24).
template <int MT>
__device__ __forceinline__ void atom_sums(const uint4* slot, float* sb, int atom, int gq, int t) {
  constexpr uint32_t kOnes = 0x00010001u;
#pragma unroll
  for (int o = 0; o < MT; ++o) {
    const uint4* f = slot + (8 * o + gq) * kActRowVec + atom * 8 + t;
    const uint4 b0 = f[0], b1 = f[4];
    float d[4];
    mma_first(d, kOnes, kOnes, kOnes, kOnes, b0.x, b0.y);
    mma_acc(d, kOnes, kOnes, kOnes, kOnes, b0.z, b0.w);
    mma_acc(d, kOnes, kOnes, kOnes, kOnes, b1.x, b1.y);
    mma_acc(d, kOnes, kOnes, kOnes, kOnes, b1.z, b1.w);
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
template <int MT, bool kFirst>
__device__ __forceinline__ void atom_mma(float (&pe)[MT][4], float (&po)[MT][4],
                                         const uint32_t (&x)[4], const uint32_t (&y)[4],
                                         const uint32_t (&z)[4], const uint32_t (&v)[4],
                                         uint32_t frag) {
#pragma unroll
  for (int o = 0; o < MT; ++o) {
    const uint4 b = lds128(frag + o * 8 * kActRow);
    if (kFirst) {
      mma_first(pe[o], x[0], y[0], x[1], y[1], b.x, b.y);
      mma_first(po[o], x[2], y[2], x[3], y[3], b.z, b.w);
    } else {
      mma_acc(pe[o], x[0], y[0], x[1], y[1], b.x, b.y);
      mma_acc(po[o], x[2], y[2], x[3], y[3], b.z, b.w);
    }
  }
#pragma unroll
  for (int o = 0; o < MT; ++o) {
    const uint4 b = lds128(frag + o * 8 * kActRow + 64);
    mma_acc(pe[o], z[0], v[0], z[1], v[1], b.x, b.y);
    mma_acc(po[o], z[2], v[2], z[3], v[3], b.z, b.w);
  }
}

// End of a group of `na` atoms starting at atom a: acc += s * (P - z * S),
// with the group's scale pair sp (s[c], s[c+8]) and zero-point pair zp.
template <int MT>
__device__ __forceinline__ void apply_group(float (&acc)[MT][4], const float (&pe)[MT][4],
                                            const float (&po)[MT][4], uint32_t sp, uint32_t zp,
                                            const float* sb, int a, int na, int t) {
  const float s0 = __half2float(__ushort_as_half((unsigned short)(sp & 0xffffu)));
  const float s1 = __half2float(__ushort_as_half((unsigned short)(sp >> 16)));
  const float nsz0 = -s0 * small_int_float(zp & 15u);
  const float nsz1 = -s1 * small_int_float((zp >> 4) & 15u);
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
    const float p0 = fmaf(po[o][0], 0.0625f, pe[o][0]);
    const float p1 = fmaf(po[o][1], 0.0625f, pe[o][1]);
    const float p2 = fmaf(po[o][2], 0.0625f, pe[o][2]);
    const float p3 = fmaf(po[o][3], 0.0625f, pe[o][3]);
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
template <int MT, int APG, bool kFull>
__device__ __forceinline__ void unit_compute(float (&acc)[MT][4], uint4 (&w)[kBatch],
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
    code_pairs(w[u].x, x);
    code_pairs(w[u].y, y);
    code_pairs(w[u].z, z);
    code_pairs(w[u].w, v);
    if (refill && (kFull || u < nu.n)) w[u] = ldg_stream(nu.wp + u * 32);
    if (compute && (kFull || u < cu.n)) {
      if (u % APG == 0)
        atom_mma<MT, true>(pe, po, x, y, z, v, frag + u * 128);
      else
        atom_mma<MT, false>(pe, po, x, y, z, v, frag + u * 128);
      if (APG < kBatch) {
        if (u % APG == APG - 1)
          apply_group<MT>(acc, pe, po, sps[(u / APG) * 8], zps[(u / APG) * 8], sb, u + 1 - APG, APG, t);
      } else if (kFull ? u == kBatch - 1 : u == cu.n - 1) {
        apply_group<MT>(acc, pe, po, sps[0], zps[0], sb, 0, kFull ? kBatch : cu.n, t);
      }
    }
  }
}

// MT: token octets (1: M <= 8, 2: M <= 16). APG: atoms per group, 1, 2 or 4;
// 8 stands for groups of 8 or more atoms (or one group per column), whose
// boundaries fall on unit starts.
template <int MT, int APG>
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
        if (u < cu.n) w[u] = ldg_stream(cu.wp + u * 32);
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
  if (warp < cu.n) atom_sums<MT>(ring, sums, warp, gq, t);

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
      atom_sums<MT>(ring + slot1 * SM::kSlotVecs, sums + ((i + 1) & 1) * SM::kSumFloats, warp, gq, t);

    const bool refill = has_next && nu.active;
    const uint4* cur = ring + slot * SM::kSlotVecs;
    const float* sb = sums + (i & 1) * SM::kSumFloats;
    if (cu.active && cu.n == kBatch && refill && nu.n == kBatch)
      unit_compute<MT, APG, true>(acc, w, cu, nu, true, cur, sb, warp, gq, t);
    else
      unit_compute<MT, APG, false>(acc, w, cu, nu, refill, cur, sb, warp, gq, t);

    if (!has_next || nu.blk != cu.blk) {
      // ---- end of a segment: atoms [seg_a0, cu.a0 + cu.n) of block cu.blk
      const int b = cu.blk;
      const bool head = seg_a0 == 0;  // holds the block's first atom
      const bool whole = head && cu.a0 + cu.n == natoms;
      if (cu.active) {
        constexpr float kUnscale = 16777216.0f;  // 2^24: codes entered as q * 2^-24
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
          if (col0 + col < N)
            p.Y[(size_t)tok * N + col0 + col] =
                __half_as_ushort(__float2half_rn(red[tok * kRedStride + col]));
        }
      } else if (head) {
        // finish the block: the later contributors' tiles, in CTA order
        const int c_last = owner_cta(((long long)(b + 1) * natoms - 1) / gr, T, C);
        const int others = c_last - (int)blockIdx.x;
        bool ok = true;
        for (int j = threadIdx.x; j < others; j += kThreads) {
          int* f = p.flags + blockIdx.x + 1 + j;
          if (wait_flag(f))
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
              tv[jj][k] = (j0 + jj <= others && e < total) ? __ldcg(tile + e) : 0.f;
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
          if (e < total && col0 + col < N)
            p.Y[(size_t)(e >> 7) * N + col0 + col] = __half_as_ushort(__float2half_rn(v[k]));
        }
      } else {
        // a run that starts inside block b: publish the partial tile, then
        // raise the flag (release after the CTA barrier covers every
        // thread's tile stores)
        __syncthreads();
        float* my = p.tiles + (size_t)blockIdx.x * kTileFloats;
        for (int e = threadIdx.x; e < total; e += kThreads) {
          const int tok = e >> 7, col = e & (kDecodeBlockCols - 1);
          my[e] = red[tok * kRedStride + col];
        }
        __syncthreads();
        if (threadIdx.x == 0) st_release(p.flags + blockIdx.x, 1);
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

template <int MT, int APG>
cudaError_t launch_variant(const DecodeArgs& args, int ctas, cudaStream_t stream) {
  auto kern = decode_kernel<MT, APG>;
  constexpr int kSmem = Smem<MT, kBatch / APG>::kTotal;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
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
// 9..16 rows, for the variant with the most shared memory: groups of 64).
int decode_ctas_per_sm(int M) {
  static int cache[2] = {0, 0};
  const int v = M <= 8 ? 0 : 1;
  if (cache[v] == 0) {
    int n = 0;
    cudaError_t e;
    if (v == 0) {
      e = cudaFuncSetAttribute(decode_kernel<1, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<1, 8>::kTotal);
      if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<1, 1>, kThreads, Smem<1, 8>::kTotal);
    } else {
      e = cudaFuncSetAttribute(decode_kernel<2, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<2, 8>::kTotal);
      if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<2, 1>, kThreads, Smem<2, 8>::kTotal);
    }
    if (e != cudaSuccess || n <= 0) return 1;
    cache[v] = n;
  }
  return cache[v];
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
                          int ctas, void* workspace, bool early_weights, cudaStream_t stream) {
  DecodeArgs args;
  int apg_t = 0;
  if (!group_shape(K, group, &apg_t, &args.gshift)) return cudaErrorInvalidValue;
  args.A = A;
  args.Wq = reinterpret_cast<const uint4*>(Wq);
  args.Sp2 = reinterpret_cast<const uint32_t*>(Sp);
  args.Zp = reinterpret_cast<const uint8_t*>(Zp);
  args.Y = Y;
  args.flags = static_cast<int*>(workspace);
  args.tiles = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + decode_counter_bytes(N));
  args.granule = split_granule(apg_t, args.gshift);
  cudaError_t e = device_error_word(&args.err);
  if (e != cudaSuccess) return e;
  args.M = M;
  args.N = N;
  args.K = K;
  args.early_weights = early_weights ? 1 : 0;
  if (M <= 8) return launch_mt<1>(args, apg_t, ctas, stream);
  return launch_mt<2>(args, apg_t, ctas, stream);
}

}  // namespace w4a16
