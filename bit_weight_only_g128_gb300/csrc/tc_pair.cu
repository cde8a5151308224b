// Two-SM tensor-core path of the W4A16 linear layer for large M (sm_103a:
// tcgen05.mma.cta_group::2, tensor memory, TMA).
//
// Once the int4 weights are dequantized the layer is an ordinary fp16 matrix
// product (the point made in the vLLM PR #1032 "Implement AWQ quantization
// support for LLaMA" thread), so at large M the work is the tensor cores'.
// Here a cluster of two CTAs, on the two SMs of a TPC, computes one output
// tile of 256 weight columns x BT tokens (BT = 128 or 256) with 256 x BT x 16
// MMAs issued by one thread of the first CTA:
//   - each CTA dequantizes its own 128 weight columns (the MMA's A operand,
//     M = 256 over the pair) into its shared memory, exactly as the one-CTA
//     kernel does: RNE_fp16((q - z) s) per weight;
//   - each CTA stages half of the tile's tokens (the B operand, split along
//     N between the pair); the MMA reads both halves and each CTA's tensor
//     memory receives its 128 columns x all BT tokens.
// Against a 128 x BT tile on one SM, every SM reads half the activation bytes
// from L2 and from its shared memory per MMA, which leaves room for deep
// rings: the pipeline's round trip (copy, dequantization, MMA, commit) takes
// several times an MMA stage, and a ring must hold that many stages.
//
// CTA roles (both CTAs of the pair):
//   warp 0      TMA producer: its half of the tile's tokens [BT/2 x 64] per
//               64-k atom (128B swizzle), and the packed codes of its 8
//               strips, which run two stages ahead;
//   warp 1      tensor-memory allocation (both CTAs, together); in the first
//               CTA one thread issues the MMAs;
//   warps 2..9  dequantize into the ring of 128B-swizzled K-major operand
//               tiles, then run the epilogue (tensor memory -> Y).
// Three rings, each deep enough for its own round trip: activations
// (act_full: the CTA's copy landed), dequantized weights (dq_full, in the
// first CTA: a group's warps of both CTAs arrived, each after its own CTA's
// activations of the stage landed) and packed codes (code_full, code_empty).
// stage_empty (both CTAs) completes when a stage's MMAs have: it frees the
// stage's activation slot and its dequantized-operand slot, and the MMA
// thread signals it to both CTAs with one multicast commit per stage. So per
// stage the MMA thread tests one barrier and commits once: each of those
// costs it about as long as an MMA of 256 tokens takes the tensor core, and
// the tensor core idles whenever its short queue of issued MMAs drains.
// Arrivals on the other CTA's barriers use mbarrier.arrive's default
// (CTA-scope) release: a cluster-scope release is a memory fence that waits
// for the thread's outstanding loads, and the dequantizing warps always have
// the next stages' scale loads in flight. Waits on barriers that the other
// CTA completes poll with test_wait: a thread suspended in try_wait resumes
// late when the phase is completed from the other SM. Every wait is bounded;
// a wait that gives up sets the library's error word and its CTA drains and
// leaves through the same final cluster barrier as a normal run.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace w4a16 {
namespace {

using namespace tc;

constexpr int kCols = 128;                          // weight columns per CTA (256 per pair)
constexpr int kStageK = 64;                         // k per stage: one 128-byte swizzle row
constexpr int kDqWarps = 8;
constexpr int kThreads = 64 + 32 * kDqWarps;
constexpr int kWdqBytes = kCols * kStageK * 2;      // 16 KiB dequantized operand
constexpr int kCodeBytes = kCols * kStageK / 2;     // 4 KiB packed codes
constexpr int kCodeLead = 2;  // stages by which the codes' copies run ahead of the activations'
constexpr int kSmemLimit = 227 * 1024;

struct PairParams {
  const uint16_t* Sp;
  const uint32_t* Zp;
  uint16_t* Y;
  int M, N, K, group;
  int bt;         // tokens per tile (MMA N over the pair): 128 or 256
  int act_slots;  // activation ring depth (stages), a multiple of dq_slots
  int dq_slots;   // dequantized-operand ring depth, a multiple of dq_groups
  int code_slots; // packed-code ring depth
  int dq_groups;  // dequant warp groups (4, 2 or 1)
  int early_weights;       // static weights: first codes and scales before the grid wait
  const float* row_scale;  // W4A8: per-row factors of the result, or null
  int* err;                // the library's error word
};

// ------------------------------------------------------------------ cluster PTX

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of both CTAs arrives, then waits for all of them.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The address in CTA `rank`'s shared memory of this CTA's shared address `a`.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

// Arrive on an mbarrier in either CTA of the pair (`cluster_bar` from
// cluster_addr), with the default release semantics of mbarrier.arrive.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// Bounded wait (as mbar_wait) that polls with test_wait instead of suspending
// in try_wait: for barriers completed by the other CTA (its arrivals, or the
// pair's multicast commits), where a thread suspended in try_wait was measured
// to resume about 0.45 us after the phase completed.
__device__ __forceinline__ bool mbar_wait_poll(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, int code, int* err) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicOr(err, code);
        return false;
      }
    }
  }
}

// Tensor memory of the pair: one warp of each CTA allocates (and frees)
// together; every tcgen05 instruction of the kernel uses cta_group::2.
__device__ __forceinline__ void pair_tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void pair_tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void pair_tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D (256 x N over the pair, fp32 in tensor memory) (+)= A (256 x 16: each
// CTA's 128 rows at the same shared address) * B (16 x N: each CTA's N/2
// columns at the same shared address).
__device__ __forceinline__ void pair_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the mbarrier at shared address `bar` of BOTH CTAs when every
// MMA this thread issued before has completed.
__device__ __forceinline__ void pair_commit_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}

// ------------------------------------------------------------------ kernel

// SA: 64-k atoms per pipeline stage (2 when K and the group are multiples of
// 128, else 1). Per stage the MMA thread tests one barrier, issues 4 * SA
// MMAs and commits once: a barrier test or a commit costs the issuing thread
// about as long as an MMA of 256 tokens takes the tensor core, so the fewer
// per MMA, the less the tensor core waits for its next instruction.
template <int SA, bool kB>
__global__ void __launch_bounds__(kThreads, 1)
tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
               const PairParams p) {
  extern __shared__ uint8_t smem_raw[];
  // the same offsets in both CTAs: the MMA's descriptors, given by the first
  // CTA, address the second CTA's operands at the same shared addresses
  const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const int bt = p.bt, half = bt / 2, nact = p.act_slots, ndq = p.dq_slots, ncode = p.code_slots;
  const uint32_t atom_act = (uint32_t)half * 128u;  // this CTA's tokens of one 64-k atom
  const uint32_t act_bytes = SA * atom_act;         // one slot of each ring
  const uint32_t dq_bytes = SA * kWdqBytes;
  const uint32_t code_bytes = SA * kCodeBytes;
  // [activation ring | dequantized-operand ring | code ring | barriers],
  // 1024-aligned slots (atoms inside a slot too)
  const uint32_t dq_base = base + (uint32_t)nact * act_bytes;
  const uint32_t code_base = dq_base + (uint32_t)ndq * dq_bytes;
  const uint32_t bars = code_base + (uint32_t)ncode * code_bytes;
  auto act_full = [&](int a) { return bars + 8u * a; };
  auto stage_empty = [&](int a) { return bars + 8u * (nact + a); };
  auto dq_full = [&](int w) { return bars + 8u * (2 * nact + w); };
  auto code_full = [&](int c) { return bars + 8u * (2 * nact + ndq + c); };
  auto code_empty = [&](int c) { return bars + 8u * (2 * nact + ndq + ncode + c); };
  const uint32_t accum_bar = bars + 8u * (2 * nact + ndq + 2 * ncode);
  const uint32_t tmem_slot = accum_bar + 8u;
  uint8_t* gen_base = smem_raw + (base - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gen_base + (tmem_slot + 4u - base));

  const uint32_t rank = cluster_rank();  // 0: the CTA that issues the MMAs
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // grid: x = 2 * token tile + column half (the pair: two consecutive x; token
  // tiles fastest, so the token tiles of one column pair run together and its
  // weights are read from DRAM once), y = column pair
  const int n0 = (2 * blockIdx.y + (blockIdx.x & 1)) * kCols;  // this CTA's 128 weight columns
  const int m0 = (blockIdx.x >> 1) * bt;                        // the pair's tokens
  const int nk = p.K / (kStageK * SA);   // stages
  const int groups = p.dq_groups;
  const int wpg = kDqWarps / groups;     // dequant warps per group

  if (threadIdx.x == 0) {
    for (int a = 0; a < nact; ++a) {
      mbar_init(act_full(a), 1);
      // the stage in activation slot a completed its MMAs: frees the slot, and
      // the dequantized-operand slot of the same stage
      mbar_init(stage_empty(a), 1);
    }
    for (int w = 0; w < ndq; ++w)
      mbar_init(dq_full(w), 2 * wpg);  // used in the first CTA: a group's warps of both CTAs
    for (int c = 0; c < ncode; ++c) {
      mbar_init(code_full(c), 1);
      mbar_init(code_empty(c), wpg);  // the warps of the group that converts the stage
    }
    mbar_init(accum_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    pair_tmem_alloc(tmem_slot, (uint32_t)bt);
    pair_tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers initialized, tensor memory allocated
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(gen_base + (tmem_slot - base));
  allow_dependent_launch();

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    // the packed codes of stage kb + kCodeLead go out before the activations of
    // stage kb: the dequantizing warps run ahead of the MMAs
    if (lane == 0) {
      const int tok0 = m0 + (int)rank * half;  // this CTA's half of the tile's tokens
      auto issue_codes = [&](int kb) -> bool {
        const int c = kb % ncode;
        if (!mbar_wait_poll(code_empty(c), ((uint32_t)(kb / ncode) & 1u) ^ 1u, abort_flag,
                            kErrProducer, p.err))
          return false;
        mbar_expect_tx(code_full(c), code_bytes);
        tma_load_2d(code_base + (uint32_t)c * code_bytes, &tmW, kb * SA * kAtomWords,
                    n0 / kStripCols, code_full(c));
        return true;
      };
      bool ok = true;
      int codes_issued = 0, act_issued = 0;
      // static weights: the first codes before the wait for the previous grid
      const int lead = nk < kCodeLead ? nk : kCodeLead;
      if (p.early_weights)
        for (; codes_issued < lead && ok; ++codes_issued) ok = issue_codes(codes_issued);
      grid_dependency_wait();
      for (; codes_issued < lead && ok; ++codes_issued) ok = issue_codes(codes_issued);
      for (int kb = 0; kb < nk && ok; ++kb) {
        if (codes_issued < nk) {
          if (!(ok = issue_codes(codes_issued))) break;
          ++codes_issued;
        }
        const int a = kb % nact;
        if (!(ok = mbar_wait_poll(stage_empty(a), ((uint32_t)(kb / nact) & 1u) ^ 1u, abort_flag,
                                  kErrProducer, p.err)))
          break;
        const uint32_t st = base + (uint32_t)a * act_bytes;
        mbar_expect_tx(act_full(a), act_bytes);
#pragma unroll
        for (int u = 0; u < SA; ++u)
          tma_load_2d(st + u * atom_act, &tmA, (kb * SA + u) * kStageK, tok0, act_full(a));
        ++act_issued;
      }
      if (*abort_flag) {
        // let the copies already issued land before the CTA leaves
        for (int kb = (act_issued > nact ? act_issued - nact : 0); kb < act_issued; ++kb)
          mbar_drain(act_full(kb % nact), (uint32_t)(kb / nact) & 1u, p.err);
        for (int kb = (codes_issued > ncode ? codes_issued - ncode : 0); kb < codes_issued; ++kb)
          mbar_drain(code_full(kb % ncode), (uint32_t)(kb / ncode) & 1u, p.err);
      } else {
        // the pair's last commits have reached this CTA: none is still on its way
        for (int kb = (nk > nact ? nk - nact : 0); kb < nk; ++kb)
          if (!mbar_wait_poll(stage_empty(kb % nact), (uint32_t)(kb / nact) & 1u, abort_flag,
                              kErrProducer, p.err))
            break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------------------- MMA issuer (first CTA)
      // dq_full completes when the stage's dequantizing warps of both CTAs
      // have arrived, each after its own CTA's activation copy of the stage
      // landed: one test covers both operands of both CTAs. The next stage's
      // barrier is tested between this stage's MMAs, while the tensor core
      // works through the queued ones.
      const uint32_t idesc = f16_idesc(2 * kCols, bt, kB);
      int a = 0, w = 0;
      uint32_t pw = 0;
      bool ok = mbar_wait_poll(dq_full(0), 0, abort_flag, kErrMma, p.err);
      for (int kb = 0; kb < nk && ok; ++kb) {
        tc_fence_after();
        const uint32_t bst = base + (uint32_t)a * act_bytes;
        const uint32_t ast = dq_base + (uint32_t)w * dq_bytes;
        const int w2 = w + 1 == ndq ? 0 : w + 1;
        const uint32_t pw2 = w2 == 0 ? pw ^ 1u : pw;
        bool ready = true;
#pragma unroll
        for (int u = 0; u < SA; ++u) {
          const uint64_t bdesc = sw128_kmajor_desc(bst + u * atom_act);
          const uint64_t adesc = sw128_kmajor_desc(ast + u * kWdqBytes);
#pragma unroll
          for (int kk = 0; kk < kStageK / 16; ++kk) {  // +32 bytes of k per MMA
            pair_mma_f16(tmem_base, adesc + 2u * kk, bdesc + 2u * kk, idesc, (kb | u | kk) != 0);
            if (u == 0 && kk == 1 && kb + 1 < nk) ready = mbar_test(dq_full(w2), pw2);
          }
        }
        pair_commit_both(stage_empty(a));
        a = a + 1 == nact ? 0 : a + 1;
        w = w2;
        pw = pw2;
        if (kb + 1 < nk && !ready) ok = mbar_wait_poll(dq_full(w), pw, abort_flag, kErrMma, p.err);
      }
      pair_commit_both(accum_bar);  // fires once every MMA issued above has completed
      if (!ok) mbar_drain(accum_bar, 0, p.err);  // no MMA may run past the release of tensor memory
    }
  } else {
    // ---------------------------------------------------------- dequant + epilogue
    // `groups` groups of warps; group g converts the stages kb = g, g + groups,
    // ... into dequantized-operand slot kb % dq_slots (dq_slots is a multiple
    // of groups: a slot is always converted by the same group); within a stage
    // each of its warps converts `groups` strips of this CTA's 8. Scales and
    // zero points are loaded into registers two of the group's stages ahead.
    const int dw = warp - 2;
    const int dg = dw / wpg, sub = dw % wpg;
    const int gq = lane >> 2, t = lane & 3;
    const int nstrips = p.N / kStripCols;
    const int G = p.K / p.group;
    const uint32_t* sp2 = reinterpret_cast<const uint32_t*>(p.Sp);
    const uint8_t* zpb = reinterpret_cast<const uint8_t*>(p.Zp);
    const uint32_t flip = (uint32_t)(gq & 1);  // odd rows take the other k-half first (banks)
    struct Meta {
      uint32_t ms[4];  // (s[gq], s[gq + 8]) of each strip
      uint32_t mz[4];  // (z[gq] | z[gq + 8] << 4) of each strip
    };
    auto load = [&](int kb, Meta& d) {
      if (kb >= nk) return;
      const int grp = (int)((long long)kb * SA * kStageK / p.group);  // one group per stage
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int strip = n0 / kStripCols + groups * sub + i;
        d.ms[i] = 0;
        d.mz[i] = 0;
        if (i < groups && strip < nstrips) {
          const size_t off = ((size_t)strip * G + grp) * 8 + gq;
          d.ms[i] = sp2[off];
          d.mz[i] = zpb[off];
        }
      }
    };
    const uint32_t dq_remote0 = cluster_addr(dq_full(0), 0);  // the first CTA's dq_full(0)
    // one stage: wait for its codes and its slot, dequantize this warp's
    // strips, release the codes, wait for the stage's activations, arrive
    auto stage = [&](int kb, const Meta& d) -> bool {
      const int w = kb % ndq, c = kb % ncode, a = kb % nact;
      if (!mbar_wait(code_full(c), (uint32_t)(kb / ncode) & 1u, abort_flag, kErrDequant, p.err))
        return false;
      // the slot's previous stage (kb - dq_slots) has completed its MMAs
      if (kb >= ndq) {
        const int prev = kb - ndq;
        if (!mbar_wait_poll(stage_empty(prev % nact), (uint32_t)(prev / nact) & 1u, abort_flag,
                            kErrDequant, p.err))
          return false;
      }
      const uint32_t wdq = dq_base + (uint32_t)w * dq_bytes;
      const uint32_t codes = code_base + (uint32_t)c * code_bytes;
      uint4 v[4][SA];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int u = 0; u < SA; ++u)
          if (i < groups) v[i][u] = lds128(codes + (groups * sub + i) * (SA * 512) + u * 512 + lane * 16);
      __syncwarp();
      if (lane == 0) mbar_arrive(code_empty(c));  // the codes are in registers
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int ls = groups * sub + i;  // strip within the CTA's 8
        if (i < groups && n0 / kStripCols + ls < nstrips) {
          const uint32_t z0 = d.mz[i] & 15u, z1 = (d.mz[i] >> 4) & 15u;
          const uint16_t s0 = (uint16_t)(d.ms[i] & 0xffffu), s1 = (uint16_t)(d.ms[i] >> 16);
#pragma unroll
          for (int u = 0; u < SA; ++u) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t ks = (uint32_t)(j >> 1) ^ flip;  // k-half of this word
              const uint32_t r = (uint32_t)(j & 1);           // column gq or gq + 8
              const uint4 vv = v[i][u];
              const uint32_t word = ks ? (r ? vv.w : vv.z) : (r ? vv.y : vv.x);
              uint32_t o[4];
              if (kB)
                dequant_word_bf16(word, make_deq_const_bf16(r ? z1 : z0, r ? s1 : s0), o);
              else
                dequant_word(word, make_deq_const(r ? z1 : z0, r ? s1 : s0), o);
              // row n = 16 ls + gq + 8 r of the operand, 16-byte chunk kw = 4 ks + t
              const uint32_t row = 16u * ls + gq + 8u * r;
              const uint32_t kw = 4u * ks + t;
              sts128(wdq + u * kWdqBytes + (row >> 3) * 1024u + (row & 7u) * 128u +
                         ((kw ^ (row & 7u)) << 4),
                     o[0], o[1], o[2], o[3]);
            }
          }
        }
      }
      fence_async_shared();  // this thread's generic-proxy stores -> visible to the tensor core
      // this CTA's activations of the stage have landed (the MMAs read them too)
      if (!mbar_wait(act_full(a), (uint32_t)(kb / nact) & 1u, abort_flag, kErrDequant, p.err))
        return false;
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(dq_remote0 + 8u * w);
      return true;
    };
    // scales and zero points: three register sets in rotation, each loaded two
    // of this group's stages before its own (no stage waits for its loads)
    Meta m0s, m1s, m2s;
    const int gs = groups;
    if (p.early_weights) {
      load(dg, m0s);
      load(dg + gs, m1s);
    }
    grid_dependency_wait();
    if (!p.early_weights) {
      load(dg, m0s);
      load(dg + gs, m1s);
    }
    for (int kb = dg; kb < nk; kb += 3 * gs) {
      load(kb + 2 * gs, m2s);
      if (!stage(kb, m0s) || kb + gs >= nk) break;
      load(kb + 3 * gs, m0s);
      if (!stage(kb + gs, m1s) || kb + 2 * gs >= nk) break;
      load(kb + 4 * gs, m1s);
      if (!stage(kb + 2 * gs, m2s)) break;
    }

    // epilogue: tensor-memory lanes 32q..32q+31 are this CTA's columns, its
    // columns are the pair's BT tokens (the first CTA's half, then the second's)
    const bool have_accum = mbar_wait(accum_bar, 0, abort_flag, kErrEpilogue, p.err);
    __syncwarp();
    if (__all_sync(0xffffffffu, have_accum)) {  // warp-uniform: tcgen05.ld is .aligned
      tc_fence_after();
      const int q = warp & 3;
      const int hsel = dw >> 2;  // two warpgroups split the token chunks
      const int n = n0 + 32 * q + lane;
      for (int c = hsel; c < bt / 16; c += 2) {
        uint32_t r[16];
        tmem_ld16(tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(16 * c), r);
        tmem_wait_ld();
        if (n < p.N) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int tok = m0 + 16 * c + j;
            if (tok < p.M)
              p.Y[(size_t)tok * p.N + n] =
                  to_out<kB>(__uint_as_float(r[j]) * (p.row_scale ? p.row_scale[tok] : 1.0f));
          }
        }
      }
    }
  }

  // an epilogue that gave up still lets the pair's last commit land here
  // before the CTA can leave (immediate in a normal run)
  if (threadIdx.x == 64) mbar_drain(accum_bar, 0, p.err);
  __syncwarp();
  tc_fence_before();
  cluster_sync();  // both CTAs done with the tensor memory and each other's barriers
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    pair_tmem_dealloc(tmem_base, (uint32_t)bt);
  }
}

// ------------------------------------------------------------------ host

template <int SA, bool kB>
cudaError_t launch_pair_kernel(const CUtensorMap& tmA, const CUtensorMap& tmW, const PairParams& prm,
                               dim3 grid, size_t smem, cudaStream_t stream) {
  cudaError_t e = set_max_smem_once(reinterpret_cast<const void*>(tc_pair_kernel<SA, kB>), kSmemLimit);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, tc_pair_kernel<SA, kB>, tmA, tmW, prm);
}

}  // namespace

int tc_pair_token_tile(int M) { return M > 128 ? 256 : 128; }

int tc_pair_stage_atoms(int K, int group) { return K % 128 == 0 && group % 128 == 0 ? 2 : 1; }

// Ring depths, counted in 64-k atoms of the pair's shared memory: 8 atoms of
// activations, 4 of dequantized weights (8 for 128-token tiles, whose
// activation slots are half as large) and 8 of packed codes; in stages of SA
// atoms. The dequantized-operand slots of a stage are freed with its
// activation slot (one commit per stage), which needs the activation ring to
// be a multiple of the dequantized one and of the two dequant groups.
size_t tc_pair_smem_bytes(int bt, int sa, int* act_slots, int* dq_slots, int* code_slots) {
  const size_t atom_act = (size_t)(bt / 2) * 128;
  const int a = 8 / sa, w = (bt > 128 ? 4 : 8) / sa, c = 8 / sa;
  if (act_slots) *act_slots = a;
  if (dq_slots) *dq_slots = w;
  if (code_slots) *code_slots = c;
  return (size_t)sa * (a * atom_act + (size_t)w * kWdqBytes + (size_t)c * kCodeBytes) + 1024 + 512;
}

cudaError_t launch_tc_pair(const uint16_t* A, const uint32_t* Wq, const uint16_t* Sp,
                           const uint32_t* Zp, uint16_t* Y, int M, int N, int K, int group,
                           bool early_weights, bool bf16, const float* row_scale,
                           cudaStream_t stream) {
  const int bt = tc_pair_token_tile(M);
  const int sa = tc_pair_stage_atoms(K, group);
  CUtensorMap tmA, tmW;
  if (!cached_tensor_map(&tmA, A, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                         2, (uint64_t)K, (uint64_t)M, 64, (uint32_t)(bt / 2), CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // packed weights viewed as [N/16 strips][K/64 atoms * 128 words] of uint32
  if (!cached_tensor_map(&tmW, Wq, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, (uint64_t)(K / kAtomK) * kAtomWords,
                         (uint64_t)(N / kStripCols), (uint32_t)(kAtomWords * sa), kCols / kStripCols,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  PairParams prm;
  prm.Sp = Sp;
  prm.Zp = Zp;
  prm.Y = Y;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.group = group;
  prm.bt = bt;
  prm.early_weights = early_weights ? 1 : 0;
  prm.row_scale = row_scale;
  cudaError_t e = device_error_word(&prm.err);
  if (e != cudaSuccess) return e;
  const size_t smem = tc_pair_smem_bytes(bt, sa, &prm.act_slots, &prm.dq_slots, &prm.code_slots);
  prm.dq_groups = 2;
  const dim3 grid((unsigned)(2 * ((M + bt - 1) / bt)), (unsigned)((N + 2 * kCols - 1) / (2 * kCols)), 1);
  if (bf16)
    return sa == 2 ? launch_pair_kernel<2, true>(tmA, tmW, prm, grid, smem, stream)
                   : launch_pair_kernel<1, true>(tmA, tmW, prm, grid, smem, stream);
  return sa == 2 ? launch_pair_kernel<2, false>(tmA, tmW, prm, grid, smem, stream)
                 : launch_pair_kernel<1, false>(tmA, tmW, prm, grid, smem, stream);
}

}  // namespace w4a16
