// Two-SM tensor-core path of the W4A16 linear layer for large M (sm_103a:
// tcgen05.mma.cta_group::2, tensor memory, TMA).
//
// Once the int4 weights are dequantized the layer is an ordinary fp16 matrix
// product (the point made in the vLLM PR #1032 "Implement AWQ quantization
// support for LLaMA" thread), so at large M the work is the tensor cores'.
// Here a cluster of two CTAs, on the two SMs of a TPC, computes one output
// tile of 256 weight columns x BT tokens (BT = 128 or 256) with 256 x BT x 16
// MMAs issued by one thread of the first CTA:
//   - each CTA dequantizes its own 128 weight columns straight into its
//     tensor memory (the MMA's A operand, 128 of the 256 rows per CTA), as
//     the one-SM kernel does: RNE_fp16((q - z) s) per weight, one column per
//     thread, 32-bit cells of two k each (tcgen05.st 32x32b);
//   - each CTA stages half of the tile's tokens (the B operand, split along
//     N between the pair); the MMA reads both halves and each CTA's tensor
//     memory receives its 128 columns x all BT tokens.
// Against a 128 x BT tile on one SM, every SM reads half the activation bytes
// from L2 (and DRAM, once they no longer fit L2) per MMA.
//
// CTA roles (both CTAs of the pair):
//   warp 0      TMA producer (one thread, polling the slots of both rings):
//               the packed codes of its 8 strips (3-D map, 128-byte swizzle)
//               and its half of the tile's tokens [BT/2 x 64] per atom
//               (128-byte swizzle);
//   warp 1      tensor-memory allocation (both CTAs, together); in the first
//               CTA one thread issues the MMAs (A from tensor memory);
//   warps 2..   two or four groups of four warps (one per tensor-memory lane
//               quarter) convert the stages g, g + groups, ... of this CTA's
//               128 columns, then run the epilogue (tensor memory -> Y).
// Rings (per CTA): activations (act_full), packed codes (code_full,
// code_empty), dequantized operand in tensor memory. dq_full, in the first
// CTA, completes when the stage's group of both CTAs has arrived, each warp
// after its tensor-memory stores completed and its own CTA's activations of
// the stage landed. stage_done (both CTAs) completes when a stage's MMAs
// have: it frees the stage's activation slot and its tensor-memory slot; the
// MMA thread signals it to both CTAs with one multicast commit per stage.
// Ring depths obey the one-SM kernel's invariants (code slots a multiple of
// the groups; activation slots at least the groups and the dequantized
// slots), which keep every parity wait within one phase of its barrier.
// Arrivals on the other CTA's barriers use mbarrier.arrive's default
// (CTA-scope) release: a cluster-scope release is a memory fence that waits
// for the thread's outstanding loads. Waits on barriers that the other CTA
// completes poll with test_wait: a thread suspended in try_wait resumes late
// when the phase is completed from the other SM. Every wait is bounded; a
// wait that gives up sets the library's error word and its CTA drains and
// leaves through the same final cluster barrier as a normal run.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace w4a16 {
namespace {

using namespace tc;

constexpr int kCols = 128;                       // weight columns per CTA (256 per pair)
constexpr int kStageK = 64;                      // k per atom
constexpr int kCodeAtomBytes = kCols * kStageK / 2;  // 4 KiB: 8 strips x 512 B
constexpr int kAtomCols = kStageK / 2;           // tensor-memory columns of one atom of A
constexpr int kSmemLimit = 227 * 1024;
constexpr int kBarBytes = 1024;

template <int NG>
struct PairWarps {
  static constexpr int kThreads = 64 + 128 * NG;
};

struct PairParams {
  const uint16_t* Sp;
  const uint32_t* Zp;
  uint16_t* Y;
  int M, N, K, group;
  int bt;          // tokens per tile (MMA N over the pair): 128 or 256
  int act_slots;   // activation ring depth (stages)
  int code_slots;  // packed-code ring depth (stages)
  int dq_slots;    // dequantized-operand ring depth (stages), at most act_slots
  int dq_col0;     // first tensor-memory column of the dequantized-operand ring
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
// D (256 x N over the pair, fp32 in tensor memory) (+)= A (256 x 16 in tensor
// memory: each CTA's 128 rows at the same address) * B (16 x N: each CTA's
// N/2 columns at the same shared address).
__device__ __forceinline__ void pair_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
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
// 128, else 1); NG: dequant groups.
template <int SA, bool kB, int NG>
__global__ void __launch_bounds__(PairWarps<NG>::kThreads, 1)
tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
               const PairParams p) {
  extern __shared__ uint8_t smem_raw[];
  // the same offsets in both CTAs: the MMA's descriptors, given by the first
  // CTA, address the second CTA's operands at the same shared addresses
  const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const int bt = p.bt, half = bt / 2, nact = p.act_slots, ncode = p.code_slots, ndq = p.dq_slots;
  const uint32_t atom_act = (uint32_t)half * 128u;  // this CTA's tokens of one 64-k atom
  const uint32_t act_bytes = SA * atom_act;
  const uint32_t code_bytes = SA * kCodeAtomBytes;
  // [activation ring | code ring | barriers], 1024-aligned slots
  const uint32_t code_base = base + (uint32_t)nact * act_bytes;
  const uint32_t bars = code_base + (uint32_t)ncode * code_bytes;
  auto act_full = [&](int a) { return bars + 8u * a; };
  auto stage_done = [&](int a) { return bars + 8u * (nact + a); };
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
  const int nk = p.K / (kStageK * SA);                          // stages

  if (threadIdx.x == 0) {
    for (int a = 0; a < nact; ++a) {
      mbar_init(act_full(a), 1);
      mbar_init(stage_done(a), 1);
    }
    for (int w = 0; w < ndq; ++w) mbar_init(dq_full(w), 8);  // used in the first CTA: a group of both CTAs
    for (int c = 0; c < ncode; ++c) {
      mbar_init(code_full(c), 1);
      mbar_init(code_empty(c), 4);
    }
    mbar_init(accum_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    pair_tmem_alloc(tmem_slot, 512);
    pair_tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers initialized, tensor memory allocated
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(gen_base + (tmem_slot - base));
  allow_dependent_launch();

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    // One thread keeps both rings full: it polls the slot of the next copy of
    // each ring and issues whichever is free.
    if (lane == 0) {
      const int tok0 = m0 + (int)rank * half;  // this CTA's half of the tile's tokens
      auto codes = [&](int kb) {
        const int c = kb % ncode;
        if (!in_smem(code_base + (uint32_t)c * code_bytes, code_bytes, raw, p.err)) return;
        mbar_expect_tx(code_full(c), code_bytes);
        tma_load_3d(code_base + (uint32_t)c * code_bytes, &tmW, 0, kb * SA * 4, n0 / kStripCols,
                    code_full(c));
      };
      auto acts = [&](int kb) {
        const int a = kb % nact;
        const uint32_t st = base + (uint32_t)a * act_bytes;
        if (!in_smem(st, act_bytes, raw, p.err)) return;
        mbar_expect_tx(act_full(a), act_bytes);
#pragma unroll
        for (int u = 0; u < SA; ++u)
          tma_load_2d(st + u * atom_act, &tmA, (kb * SA + u) * kStageK, tok0, act_full(a));
      };
      int ci = 0, ai = 0;
      // static weights: the first ring of codes before the wait for the
      // previous grid (the slots are free: nothing has used them yet)
      if (p.early_weights)
        for (; ci < nk && ci < ncode; ++ci) codes(ci);
      grid_dependency_wait();
      uint64_t t0 = globaltimer();
      uint32_t idle = 0;
      while (ci < nk || ai < nk) {
        bool progress = false;
        if (ci < nk && mbar_test(code_empty(ci % ncode), ((uint32_t)(ci / ncode) & 1u) ^ 1u)) {
          codes(ci++);
          progress = true;
        }
        if (ai < nk && mbar_test(stage_done(ai % nact), ((uint32_t)(ai / nact) & 1u) ^ 1u)) {
          acts(ai++);
          progress = true;
        }
        if (progress) {
          idle = 0;
        } else if ((++idle & 63u) == 0) {
          if (*abort_flag) break;
          const uint64_t t = globaltimer();
          if (idle == 64) t0 = t;  // first check of this idle spell
          else if (t - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(p.err, kErrProducer);
            break;
          }
        }
      }
      if (*abort_flag) {
        // let the copies already issued land before the CTA leaves
        for (int kb = (ai > nact ? ai - nact : 0); kb < ai; ++kb)
          mbar_drain(act_full(kb % nact), (uint32_t)(kb / nact) & 1u, p.err);
        for (int kb = (ci > ncode ? ci - ncode : 0); kb < ci; ++kb)
          mbar_drain(code_full(kb % ncode), (uint32_t)(kb / ncode) & 1u, p.err);
      } else {
        // the pair's last commits have reached this CTA: none is still on its way
        for (int kb = (nk > nact ? nk - nact : 0); kb < nk; ++kb)
          if (!mbar_wait_poll(stage_done(kb % nact), (uint32_t)(kb / nact) & 1u, abort_flag,
                              kErrProducer, p.err))
            break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------------------- MMA issuer (first CTA)
      // dq_full completes when the stage's group of both CTAs has arrived, each
      // warp after its tensor-memory stores completed and its own CTA's
      // activations of the stage landed: one test covers both operands of
      // both CTAs. The next stage's barrier is tested between this stage's
      // MMAs, while the tensor core works through the queued ones.
      const uint32_t idesc = f16_idesc(2 * kCols, bt, kB);
      int a = 0, w = 0;
      uint32_t pw = 0;
      bool ok = nk > 0 && in_tmem(0, (uint32_t)bt, 512, p.err) &&
                mbar_wait_poll(dq_full(0), 0, abort_flag, kErrMma, p.err);
      for (int kb = 0; kb < nk && ok; ++kb) {
        tc_fence_after();
        const uint32_t bst = base + (uint32_t)a * act_bytes;
        const uint32_t acol = tmem_base + (uint32_t)(p.dq_col0 + w * SA * kAtomCols);
        if (!in_smem(bst, act_bytes, raw, p.err) ||
            !in_tmem((uint32_t)(p.dq_col0 + w * SA * kAtomCols), SA * kAtomCols, 512, p.err)) {
          ok = false;
          break;
        }
        const int w2 = w + 1 == ndq ? 0 : w + 1;
        const uint32_t pw2 = w2 == 0 ? pw ^ 1u : pw;
        bool ready = true;
#pragma unroll
        for (int u = 0; u < SA; ++u) {
          const uint64_t bdesc = sw128_kmajor_desc(bst + u * atom_act);
#pragma unroll
          for (int kk = 0; kk < kStageK / 16; ++kk) {  // 16 k per MMA: 8 columns of A, 32 bytes of B
            pair_mma_f16_ts(tmem_base, acol + (uint32_t)(u * kAtomCols + 8 * kk), bdesc + 2u * kk, idesc,
                            (kb | u | kk) != 0);
            if (u == 0 && kk == 1 && kb + 1 < nk) ready = mbar_test(dq_full(w2), pw2);
          }
        }
        pair_commit_both(stage_done(a));
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
    // NG groups of four warps; group g converts the stages g, g + NG, ...
    // Thread (lane quarter q, lane) owns weight column 32 q + lane of this
    // CTA's 128: tensor-memory lane 32 q + lane, strip 2 q + lane / 16,
    // column c = lane % 16 of the strip. In the packed format the 16 bytes at
    // 64 (c % 8) + 16 l (l = 0..3) of a strip's atom hold the words of
    // k-octets l and 4 + l of columns c % 8 (words 0, 2) and c % 8 + 8 (words
    // 1, 3).
    const int dw = warp - 2;
    const int grp_id = dw >> 2;
    const int q = warp & 3;
    const int ls = 2 * q + (lane >> 4);
    const int c = lane & 15, cp = c & 7;
    const bool hi = c >= 8;
    const int strip = n0 / kStripCols + ls;
    const bool live = strip < p.N / kStripCols;
    const int G = p.K / p.group;
    const uint32_t tlane = (uint32_t)(32 * q) << 16;
    // scale bits (low half) and zero point (bits 16..19) of this column for a
    // stage (one group per stage)
    auto load_meta = [&](int kb) -> uint32_t {
      if (kb >= nk || !live) return 0u;
      const int grp = (int)((long long)kb * SA * kStageK / p.group);
      const size_t pg = (size_t)strip * G + grp;
      const uint8_t* zp = reinterpret_cast<const uint8_t*>(p.Zp);
      const uint32_t sb = *ld_at(p.Sp + pg * 16 + 2 * cp + (hi ? 1 : 0), p.Sp, (size_t)G * p.N, p.err);
      const uint32_t zb = *ld_at(zp + pg * 8 + cp, zp, (size_t)G * p.N / 2, p.err);
      return sb | (((zb >> (hi ? 4 : 0)) & 15u) << 16);
    };
    const uint32_t dq_remote0 = cluster_addr(dq_full(0), 0);  // the first CTA's dq_full(0)
    // a wait that every lane of the warp passes or every lane gives up on:
    // the tensor-memory stores that follow are .sync.aligned
    auto warp_wait = [&](uint32_t bar, uint32_t parity, bool poll) -> bool {
      const bool ok = poll ? mbar_wait_poll(bar, parity, abort_flag, kErrDequant, p.err)
                           : mbar_wait(bar, parity, abort_flag, kErrDequant, p.err);
      return __all_sync(0xffffffffu, ok);
    };
    // one stage: wait for its codes, read this column's words, release the
    // codes; wait for the tensor-memory slot (its previous stage's MMAs, a
    // commit from the first CTA); dequantize and store; wait for this CTA's
    // activations of the stage; arrive on the first CTA's dq_full
    auto stage = [&](int kb, uint32_t meta) -> bool {
      const int cs = kb % ncode, a = kb % nact, w = kb % ndq;
      if (!warp_wait(code_full(cs), (uint32_t)(kb / ncode) & 1u, false)) return false;
      const uint32_t cb = code_base + (uint32_t)cs * code_bytes;
      uint32_t wl[SA][4], wh[SA][4];  // k-octets l and 4 + l of each atom
#pragma unroll
      for (int u = 0; u < SA; ++u) {
        const uint32_t row = (uint32_t)(ls * 4 * SA + 4 * u + (cp >> 1));  // 128-byte row of the tile
#pragma unroll
        for (int l = 0; l < 4; ++l) {
          const uint32_t chunk = ((uint32_t)(4 * (cp & 1) + l)) ^ (row & 7u);  // 128-byte swizzle
          const uint32_t at = cb + row * 128u + (chunk << 4);
          const uint4 v = lds128(in_smem(at, 16, raw, p.err) ? at : cb);
          wl[u][l] = hi ? v.y : v.x;
          wh[u][l] = hi ? v.w : v.z;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(code_empty(cs));  // the codes are in registers
      if (kb >= ndq) {
        const int prev = kb - ndq;
        if (!warp_wait(stage_done(prev % nact), (uint32_t)(prev / nact) & 1u, true)) return false;
        tc_fence_after();
      }
      const uint32_t z = (meta >> 16) & 15u;
      const uint16_t s = (uint16_t)(meta & 0xffffu);
      const uint32_t tcol = tmem_base + tlane + (uint32_t)(p.dq_col0 + w * SA * kAtomCols);
#pragma unroll
      for (int u = 0; u < SA; ++u) {
        uint32_t r[32];  // cell j = (deq[2j], deq[2j + 1]): k-octet o fills cells 4o..4o+3
#pragma unroll
        for (int l = 0; l < 4; ++l) {
          uint32_t o0[4], o1[4];
          if (kB) {
            const DeqConstBf16 dc = make_deq_const_bf16(z, s);
            dequant_word_bf16(wl[u][l], dc, o0);
            dequant_word_bf16(wh[u][l], dc, o1);
          } else {
            const DeqConst dc = make_deq_const(z, s);
            dequant_word(wl[u][l], dc, o0);
            dequant_word(wh[u][l], dc, o1);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            r[4 * l + j] = o0[j];
            r[16 + 4 * l + j] = o1[j];
          }
        }
        if (in_tmem((uint32_t)(p.dq_col0 + w * SA * kAtomCols + u * kAtomCols), kAtomCols, 512, p.err))
          tmem_st32(tcol + (uint32_t)(u * kAtomCols), r);
      }
      tmem_wait_st();
      // this CTA's activations of the stage have landed (the MMAs read them too)
      if (!warp_wait(act_full(a), (uint32_t)(kb / nact) & 1u, false)) return false;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(dq_remote0 + 8u * w);
      return true;
    };
    // scales and zero points: three register sets in rotation, each loaded two
    // of this group's stages before its own (no stage waits for its loads).
    // They are weights: with static weights the first sets are read before the
    // wait for the previous grid (which orders this warp's stores of Y)
    uint32_t m0s = 0, m1s = 0, m2s = 0;
    if (p.early_weights) {
      m0s = load_meta(grp_id);
      m1s = load_meta(grp_id + NG);
    }
    grid_dependency_wait();
    if (!p.early_weights) {
      m0s = load_meta(grp_id);
      m1s = load_meta(grp_id + NG);
    }
    for (int kb = grp_id; kb < nk; kb += 3 * NG) {
      m2s = load_meta(kb + 2 * NG);
      if (!stage(kb, m0s) || kb + NG >= nk) break;
      m0s = load_meta(kb + 3 * NG);
      if (!stage(kb + NG, m1s) || kb + 2 * NG >= nk) break;
      m1s = load_meta(kb + 4 * NG);
      if (!stage(kb + 2 * NG, m2s)) break;
    }

    // epilogue: tensor-memory lanes 32q..32q+31 are this CTA's columns, its
    // columns are the pair's BT tokens (the first CTA's half, then the second's)
    const bool have_accum = mbar_wait_poll(accum_bar, 0, abort_flag, kErrEpilogue, p.err);
    __syncwarp();
    if (__all_sync(0xffffffffu, have_accum)) {  // warp-uniform: tcgen05.ld is .aligned
      tc_fence_after();
      const int n = n0 + 32 * q + lane;
      for (int ch = grp_id; ch < bt / 16; ch += NG) {
        uint32_t r[16];
        tmem_ld16(tmem_base + tlane + (uint32_t)(16 * ch), r);
        tmem_wait_ld();
        if (n < p.N) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int tok = m0 + 16 * ch + j;
            uint16_t* d = p.Y + (size_t)tok * p.N + n;
            if (tok < p.M && in_buf(d, p.Y, (size_t)p.M * p.N, p.err))
              *d = to_out<kB>(__uint_as_float(r[j]) *
                              (p.row_scale ? *ld_at(p.row_scale + tok, p.row_scale, (size_t)p.M, p.err) : 1.0f));
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
    pair_tmem_dealloc(tmem_base, 512);
  }
}

// ------------------------------------------------------------------ host

struct PairRings {
  int act, code, dq, groups, dq_col0;
  size_t smem;
};

// Ring depths per CTA (stages of SA atoms): codes 16 atoms (64 KiB), the
// activations as deep as the rest of the shared memory allows (at most 16
// atoms), the dequantized operand in the tensor memory the accumulator (BT
// columns) leaves (at most 16 atoms, no deeper than the activation ring);
// four dequant groups where four activation slots fit, else two.
PairRings pair_rings(int bt, int sa) {
  PairRings r;
  const size_t budget = (size_t)kSmemLimit - 1024 - kBarBytes;
  r.code = 16 / sa;
  const size_t act_slot = (size_t)sa * (bt / 2) * 128;
  const size_t code_slot = (size_t)sa * kCodeAtomBytes;
  const int act = (int)((budget - (size_t)r.code * code_slot) / act_slot);
  r.act = act > 16 / sa ? 16 / sa : act;
  r.groups = r.act >= 4 ? 4 : 2;
  r.dq_col0 = bt;
  int dq = (512 - bt) / (sa * kAtomCols);
  if (dq > 16 / sa) dq = 16 / sa;
  r.dq = dq > r.act ? r.act : dq;
  r.smem = (size_t)r.act * act_slot + (size_t)r.code * code_slot + 1024 + kBarBytes;
  return r;
}

bool pair_rings_valid(const PairRings& r) {
  return r.dq >= 1 && r.dq <= r.act && r.act >= r.groups && r.code % r.groups == 0;
}

template <int SA, bool kB, int NG>
cudaError_t launch_pair_kernel(const CUtensorMap& tmA, const CUtensorMap& tmW, const PairParams& prm,
                               dim3 grid, size_t smem, cudaStream_t stream) {
  cudaError_t e =
      set_max_smem_once(reinterpret_cast<const void*>(tc_pair_kernel<SA, kB, NG>), kSmemLimit);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(PairWarps<NG>::kThreads);
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
  return cudaLaunchKernelEx(&cfg, tc_pair_kernel<SA, kB, NG>, tmA, tmW, prm);
}

template <bool kB>
cudaError_t launch_pair_sa(int sa, int ng, const CUtensorMap& tmA, const CUtensorMap& tmW,
                           const PairParams& prm, dim3 grid, size_t smem, cudaStream_t stream) {
  if (ng == 4)
    return sa == 2 ? launch_pair_kernel<2, kB, 4>(tmA, tmW, prm, grid, smem, stream)
                   : launch_pair_kernel<1, kB, 4>(tmA, tmW, prm, grid, smem, stream);
  return sa == 2 ? launch_pair_kernel<2, kB, 2>(tmA, tmW, prm, grid, smem, stream)
                 : launch_pair_kernel<1, kB, 2>(tmA, tmW, prm, grid, smem, stream);
}

}  // namespace

int tc_pair_token_tile(int M) { return M > 128 ? 256 : 128; }

int tc_pair_stage_atoms(int K, int group) { return K % 128 == 0 && group % 128 == 0 ? 2 : 1; }

size_t tc_pair_smem_bytes(int bt, int sa, int* act_slots, int* dq_slots, int* code_slots) {
  const PairRings r = pair_rings(bt, sa);
  if (act_slots) *act_slots = r.act;
  if (dq_slots) *dq_slots = r.dq;
  if (code_slots) *code_slots = r.code;
  return r.smem;
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
  if (!cached_code_map(&tmW, Wq, N, K, sa)) return cudaErrorInvalidValue;
  const PairRings rings = pair_rings(bt, sa);
  if (!pair_rings_valid(rings)) return cudaErrorInvalidValue;
  PairParams prm;
  prm.Sp = Sp;
  prm.Zp = Zp;
  prm.Y = Y;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.group = group;
  prm.bt = bt;
  prm.act_slots = rings.act;
  prm.code_slots = rings.code;
  prm.dq_slots = rings.dq;
  prm.dq_col0 = rings.dq_col0;
  prm.early_weights = early_weights ? 1 : 0;
  prm.row_scale = row_scale;
  cudaError_t e = device_error_word(&prm.err);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)(2 * ((M + bt - 1) / bt)), (unsigned)((N + 2 * kCols - 1) / (2 * kCols)), 1);
  return bf16 ? launch_pair_sa<true>(sa, rings.groups, tmA, tmW, prm, grid, rings.smem, stream)
              : launch_pair_sa<false>(sa, rings.groups, tmA, tmW, prm, grid, rings.smem, stream);
}

}  // namespace w4a16
