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

#include <mutex>
#include <vector>

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

// Stage s of a cluster's sequence as (its tile's index in the sequence,
// stage kb of that tile), stepped forward without a division.
struct SeqPos {
  int kb, tile;
  __device__ __forceinline__ void step(int d, int nk) {
    kb += d;
    while (kb >= nk) {
      kb -= nk;
      ++tile;
    }
  }
};

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
  int tiles;       // output tiles of the launch: column pairs x token tiles
  int tiles_m;     // token tiles (the fastest index of a tile)
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
//
// Persistent: the grid is one cluster per TPC (at most), and cluster c takes
// the tiles c, c + clusters, ... in raster order (token tiles fastest). The
// rings run on across tiles: stage s of the cluster's sequence is stage
// s % nk of its tile s / nk, so the copies and conversions of a tile's first
// stages proceed while the previous tile's last MMAs and epilogue run. The
// single accumulator is handed over with two more barriers: accum_full (both
// CTAs; committed after a tile's last MMA) and accum_empty (first CTA; every
// dequant warp of both CTAs arrives once it has stored its part of the tile);
// the MMA thread waits for accum_empty before the next tile's first MMA.
// A group stores its part of tile i right after converting its first stage of
// a later tile (whose operands then wait in the rings), or at its end.
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
  const uint32_t accum_full = bars + 8u * (2 * nact + ndq + 2 * ncode);
  const uint32_t accum_empty = accum_full + 8u;  // used in the first CTA
  const uint32_t drain_bar = accum_empty + 8u;   // the MMAs issued before an abort completed
  const uint32_t tmem_slot = drain_bar + 8u;
  uint8_t* gen_base = smem_raw + (base - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gen_base + (tmem_slot + 4u - base));

  const uint32_t rank = cluster_rank();  // 0: the CTA that issues the MMAs
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cluster = blockIdx.x >> 1, clusters = gridDim.x >> 1;
  const int nk = p.K / (kStageK * SA);  // stages of one tile
  // this cluster's tiles: cluster, cluster + clusters, ...
  const int ntl = cluster < p.tiles ? (p.tiles - 1 - cluster) / clusters + 1 : 0;
  const int total = ntl * nk;  // stages of the cluster's sequence
  // tile i of the sequence: this CTA's 128 weight columns and the pair's tokens
  auto tile_n0 = [&](int i) {
    const int t = cluster + i * clusters;
    return (2 * (t / p.tiles_m) + (int)rank) * kCols;
  };
  auto tile_m0 = [&](int i) {
    const int t = cluster + i * clusters;
    return (t % p.tiles_m) * bt;
  };

  if (threadIdx.x == 0) {
    for (int a = 0; a < nact; ++a) {
      mbar_init(act_full(a), 1);
      mbar_init(stage_done(a), 1);
    }
    for (int w = 0; w < ndq; ++w) mbar_init(dq_full(w), 8);  // used in the first CTA: a group of both CTAs
    for (int c = 0; c < ncode; ++c) {
      mbar_init(code_full(c), 1);
      mbar_init(code_empty(c), 4);  // the warps of the group that converts the stage
    }
    mbar_init(accum_full, 1);
    mbar_init(accum_empty, 2 * 4 * NG);  // every dequant warp of both CTAs
    mbar_init(drain_bar, 1);
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
      // the next copy of each ring: its stage, tile position, ring slot and
      // the tile's strip (codes) or this CTA's first token (activations)
      int ci = 0, ai = 0;
      SeqPos cseq{0, 0}, aseq{0, 0};
      RingPos cpos{0, 0u}, apos{0, 0u};
      int cstrip = tile_n0(0) / kStripCols;
      int atok = tile_m0(0) + (int)rank * half;  // this CTA's half of the tile's tokens
      auto codes = [&]() {
        const int c = cpos.slot;
        if (in_smem(code_base + (uint32_t)c * code_bytes, code_bytes, raw, p.err)) {
          mbar_expect_tx(code_full(c), code_bytes);
          tma_load_3d(code_base + (uint32_t)c * code_bytes, &tmW, 0, cseq.kb * SA * 4, cstrip, code_full(c));
        }
        ++ci;
        cpos.step(1, ncode);
        const int tl = cseq.tile;
        cseq.step(1, nk);
        if (cseq.tile != tl && ci < total) cstrip = tile_n0(cseq.tile) / kStripCols;
      };
      auto acts = [&]() {
        const int a = apos.slot;
        const uint32_t st = base + (uint32_t)a * act_bytes;
        if (in_smem(st, act_bytes, raw, p.err)) {
          mbar_expect_tx(act_full(a), act_bytes);
#pragma unroll
          for (int u = 0; u < SA; ++u)
            tma_load_2d(st + u * atom_act, &tmA, (aseq.kb * SA + u) * kStageK, atok, act_full(a));
        }
        ++ai;
        apos.step(1, nact);
        const int tl = aseq.tile;
        aseq.step(1, nk);
        if (aseq.tile != tl && ai < total) atok = tile_m0(aseq.tile) + (int)rank * half;
      };
      // static weights: the first ring of codes before the wait for the
      // previous grid (the slots are free: nothing has used them yet)
      if (p.early_weights)
        while (ci < total && ci < ncode) codes();
      grid_dependency_wait();
      uint64_t t0 = globaltimer();
      uint32_t idle = 0;
      while (ci < total || ai < total) {
        bool progress = false;
        if (ci < total && mbar_test(code_empty(cpos.slot), cpos.phase ^ 1u)) {
          codes();
          progress = true;
        }
        if (ai < total && mbar_test(stage_done(apos.slot), apos.phase ^ 1u)) {
          acts();
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
        for (int s = (ai > nact ? ai - nact : 0); s < ai; ++s)
          mbar_drain(act_full(s % nact), (uint32_t)(s / nact) & 1u, p.err);
        for (int s = (ci > ncode ? ci - ncode : 0); s < ci; ++s)
          mbar_drain(code_full(s % ncode), (uint32_t)(s / ncode) & 1u, p.err);
      } else {
        // the pair's last commits have reached this CTA: none is still on its way
        for (int s = (total > nact ? total - nact : 0); s < total; ++s)
          if (!mbar_wait_poll(stage_done(s % nact), (uint32_t)(s / nact) & 1u, abort_flag,
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
      // MMAs, while the tensor core works through the queued ones. A tile's
      // first MMA waits for the previous tile's accumulator to be stored.
      const uint32_t idesc = f16_idesc(2 * kCols, bt, kB);
      int a = 0, w = 0;
      uint32_t pw = 0;
      bool ok = total > 0 && in_tmem(0, (uint32_t)bt, 512, p.err) &&
                mbar_wait_poll(dq_full(0), 0, abort_flag, kErrMma, p.err);
      // one loop per tile: the hand-over of the accumulator stays out of the
      // loop that issues the MMAs (a branch there cost about 10% of the stage
      // rate: this thread's issue is on the critical path)
      for (int tl = 0; tl < ntl && ok; ++tl) {
        if (tl > 0 && !(ok = mbar_wait_poll(accum_empty, (uint32_t)(tl - 1) & 1u, abort_flag, kErrMma, p.err)))
          break;
        const bool more = tl + 1 < ntl;  // another tile's stages follow this tile's last
        for (int kb = 0; kb < nk && ok; ++kb) {
          tc_fence_after();
          const uint32_t bst = base + (uint32_t)a * act_bytes;
          const uint32_t acol = tmem_base + (uint32_t)(p.dq_col0 + w * SA * kAtomCols);
          if (!in_smem(bst, act_bytes, raw, p.err) ||
              !in_tmem((uint32_t)(p.dq_col0 + w * SA * kAtomCols), SA * kAtomCols, 512, p.err)) {
            ok = false;
            break;
          }
          const bool next = kb + 1 < nk || more;
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
              if (u == 0 && kk == 1 && next) ready = mbar_test(dq_full(w2), pw2);
            }
          }
          pair_commit_both(stage_done(a));
          a = a + 1 == nact ? 0 : a + 1;
          w = w2;
          pw = pw2;
          if (next && !ready) ok = mbar_wait_poll(dq_full(w), pw, abort_flag, kErrMma, p.err);
        }
        if (ok) pair_commit_both(accum_full);  // the tile's accumulator is complete
      }
      if (!ok) {
        // no MMA may run past the release of tensor memory: one more commit,
        // to both CTAs' drain barriers, fires once every MMA issued has completed
        pair_commit_both(drain_bar);
        mbar_drain(drain_bar, 0, p.err);
      }
    }
  } else {
    // ---------------------------------------------------------- dequant + epilogue
    // NG groups of four warps; group g converts the stages g, g + NG, ... of
    // the cluster's sequence. Thread (lane quarter q, lane) owns weight column
    // 32 q + lane of this CTA's 128: tensor-memory lane 32 q + lane, strip
    // 2 q + lane / 16, column c = lane % 16 of the strip. In the packed format
    // the 16 bytes at 64 (c % 8) + 16 l (l = 0..3) of a strip's atom hold the
    // words of k-octets l and 4 + l of columns c % 8 (words 0, 2) and c % 8 + 8
    // (words 1, 3).
    const int dw = warp - 2;
    const int grp_id = dw >> 2;
    const int q = warp & 3;
    const int ls = 2 * q + (lane >> 4);
    const int c = lane & 15, cp = c & 7;
    const bool hi = c >= 8;
    const int G = p.K / p.group;
    const uint32_t tlane = (uint32_t)(32 * q) << 16;
    // scale bits (low half) and zero point (bits 16..19) of this column for a
    // stage (one group per stage). The stages' meta are loaded in order, NG
    // stages apart; the stage's tile, strip and group are followed without a
    // division (mgend: the k where the group after the stage's group starts).
    int mi = grp_id;  // stage of the sequence whose meta loads next
    SeqPos mseq{grp_id, 0};
    mseq.step(0, nk);
    int mstrip = tile_n0(mseq.tile) / kStripCols + ls;
    int mgrp = mseq.kb * SA * kStageK / p.group;
    int mgend = (mgrp + 1) * p.group;
    auto load_meta = [&]() -> uint32_t {
      uint32_t v = 0u;
      if (mi < total && mstrip < p.N / kStripCols) {
        const size_t pg = (size_t)mstrip * G + mgrp;
        const uint8_t* zp = reinterpret_cast<const uint8_t*>(p.Zp);
        const uint32_t sb = *ld_at(p.Sp + pg * 16 + 2 * cp + (hi ? 1 : 0), p.Sp, (size_t)G * p.N, p.err);
        const uint32_t zb = *ld_at(zp + pg * 8 + cp, zp, (size_t)G * p.N / 2, p.err);
        v = sb | (((zb >> (hi ? 4 : 0)) & 15u) << 16);
      }
      mi += NG;
      const int tl = mseq.tile;
      mseq.step(NG, nk);
      if (mseq.tile != tl) {
        if (mi < total) mstrip = tile_n0(mseq.tile) / kStripCols + ls;
        mgrp = 0;
        mgend = p.group;
      }
      while (mseq.kb * SA * kStageK >= mgend) {
        ++mgrp;
        mgend += p.group;
      }
      return v;
    };
    const uint32_t dq_remote0 = cluster_addr(dq_full(0), 0);          // the first CTA's dq_full(0)
    const uint32_t empty_remote = cluster_addr(accum_empty, 0);       // the first CTA's accum_empty
    // a wait that every lane of the warp passes or every lane gives up on:
    // the tensor-memory stores and loads that follow are .sync.aligned
    auto warp_wait = [&](uint32_t bar, uint32_t parity, bool poll, int code) -> bool {
      const bool ok = poll ? mbar_wait_poll(bar, parity, abort_flag, code, p.err)
                           : mbar_wait(bar, parity, abort_flag, code, p.err);
      return __all_sync(0xffffffffu, ok);
    };
    // one stage: wait for its codes, read this column's words, release the
    // codes; wait for the tensor-memory slot (its previous stage's MMAs, a
    // commit from the first CTA); dequantize and store; wait for this CTA's
    // activations of the stage; arrive on the first CTA's dq_full
    // ring positions and tile of this group's next stage (its stages are NG
    // apart); stile: the tile of the stage converted last
    RingPos spos_code, spos_act;
    spos_code.init(grp_id, ncode);
    spos_act.init(grp_id, nact);
    int sw = grp_id % ndq;
    SeqPos sseq{grp_id, 0};
    sseq.step(0, nk);
    int stile = 0;
    auto stage = [&](int s, uint32_t meta) -> bool {
      const int cs = spos_code.slot, a = spos_act.slot, w = sw;
      const uint32_t code_par = spos_code.phase, act_par = spos_act.phase;
      const RingPos prev = spos_act.before(ndq, nact);  // stage s - dq_slots (dq_slots <= act_slots)
      stile = sseq.tile;
      spos_code.step(NG, ncode);
      spos_act.step(NG, nact);
      sw += NG;
      while (sw >= ndq) sw -= ndq;
      sseq.step(NG, nk);
      if (!warp_wait(code_full(cs), code_par, false, kErrDequant)) return false;
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
      if (s >= ndq) {
        if (!warp_wait(stage_done(prev.slot), prev.phase, true, kErrDequant)) return false;
        tc_fence_after();
      }
      const uint32_t z = (meta >> 16) & 15u;
      const uint16_t sc = (uint16_t)(meta & 0xffffu);
      const uint32_t tcol = tmem_base + tlane + (uint32_t)(p.dq_col0 + w * SA * kAtomCols);
#pragma unroll
      for (int u = 0; u < SA; ++u) {
        uint32_t r[32];  // cell j = (deq[2j], deq[2j + 1]): k-octet o fills cells 4o..4o+3
#pragma unroll
        for (int l = 0; l < 4; ++l) {
          uint32_t o0[4], o1[4];
          if (kB) {
            const DeqConstBf16 dc = make_deq_const_bf16(z, sc);
            dequant_word_bf16(wl[u][l], dc, o0);
            dequant_word_bf16(wh[u][l], dc, o1);
          } else {
            const DeqConst dc = make_deq_const(z, sc);
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
      if (!warp_wait(act_full(a), act_par, false, kErrDequant)) return false;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(dq_remote0 + 8u * w);
      return true;
    };
    // this warp's part of tile i's epilogue: tensor-memory lanes 32q..32q+31
    // are this CTA's columns, its columns the pair's BT tokens (the first
    // CTA's half, then the second's); then the accumulator is free for the
    // first CTA's next tile
    auto epilogue = [&](int i) -> bool {
      if (!warp_wait(accum_full, (uint32_t)i & 1u, true, kErrEpilogue)) return false;
      tc_fence_after();
      const int n = tile_n0(i) + 32 * q + lane, m0 = tile_m0(i);
      for (int ch = grp_id; ch < bt / 16; ch += NG) {
        uint32_t r[16];
        if (in_tmem((uint32_t)(16 * ch), 16, 512, p.err)) tmem_ld16(tmem_base + tlane + (uint32_t)(16 * ch), r);
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
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(empty_remote);
      return true;
    };
    // scales and zero points, loaded two of this group's stages before their
    // own (m0s: this stage's, m1s: the next one's). They are weights: with
    // static weights the first ones are read before the wait for the previous
    // grid (which orders this warp's stores of Y)
    uint32_t m0s = 0, m1s = 0;
    if (p.early_weights) {
      m0s = load_meta();  // stage grp_id
      m1s = load_meta();  // stage grp_id + NG
    }
    grid_dependency_wait();
    if (!p.early_weights) {
      m0s = load_meta();
      m1s = load_meta();
    }
    // the tiles whose epilogue this warp has done: [0, done). One call site
    // each for the stage and the epilogue keeps the loop's code small.
    int done = 0;
    bool ok = true;
    for (int s = grp_id; s < total && ok; s += NG) {
      const uint32_t m2s = load_meta();  // stage s + 2 NG
      ok = stage(s, m0s);
      // the epilogues of the tiles before the converted stage's tile
      for (; ok && done < stile; ++done) ok = epilogue(done);
      m0s = m1s;
      m1s = m2s;
    }
    // the remaining epilogues (normally the last tile's)
    for (; ok && done < ntl; ++done) ok = epilogue(done);
  }

  // the pair's last commit has landed here before the CTA can leave: the last
  // tile's accumulator commit in a normal run (already waited for by the
  // epilogue), the drain commit after an abort
  if (threadIdx.x == 64) {
    if (*abort_flag == 0) mbar_drain(accum_full, (uint32_t)(ntl - 1) & 1u, p.err);
    else mbar_drain(drain_bar, 0, p.err);
  }
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

// Besides the one-SM kernel's invariants, the dequantized slots are at least
// the groups: a group's conversion of a stage then waits only for MMAs of
// tiles whose accumulator it has already stored (its previous stage came at
// most `groups` stages earlier), so a tile's epilogue never waits for itself.
bool pair_rings_valid(const PairRings& r) {
  return r.dq >= r.groups && r.dq <= r.act && r.act >= r.groups && r.code % r.groups == 0;
}

// Clusters of a kernel and launch shape that are resident at once
// (cudaOccupancyMaxActiveClusters, kept per kernel, device and shared-memory
// size). A cluster's two CTAs sit on the two SMs of one TPC within one GPC,
// so GPCs with an odd number of usable SMs leave an SM out and the count can
// be below SMs / 2; a persistent grid larger than it would run its last
// clusters after the others, each with its whole share of the tiles.
cudaError_t max_active_clusters(const void* kernel, const cudaLaunchConfig_t& cfg, int* out) {
  struct Entry {
    const void* kernel;
    int device;
    size_t smem;
    int clusters;
  };
  static std::mutex mu;
  static std::vector<Entry> known;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& k : known)
      if (k.kernel == kernel && k.device == dev && k.smem == cfg.dynamicSmemBytes) {
        *out = k.clusters;
        return cudaSuccess;
      }
  }
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  std::lock_guard<std::mutex> lock(mu);
  known.push_back({kernel, dev, cfg.dynamicSmemBytes, n});
  *out = n;
  return cudaSuccess;
}

template <int SA, bool kB, int NG>
cudaError_t launch_pair_kernel(const CUtensorMap& tmA, const CUtensorMap& tmW, const PairParams& prm,
                               size_t smem, cudaStream_t stream) {
  const void* kern = reinterpret_cast<const void*>(tc_pair_kernel<SA, kB, NG>);
  cudaError_t e = set_max_smem_once(kern, kSmemLimit);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
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
  cfg.numAttrs = 1;           // the occupancy query takes the cluster shape only
  cfg.gridDim = dim3(2, 1, 1);  // and a grid of whole clusters
  int resident = 0;
  e = max_active_clusters(kern, cfg, &resident);
  if (e != cudaSuccess) return e;
  // persistent: as many clusters as are resident at once (at most one per
  // tile), each taking every clusters-th tile
  const int clusters = prm.tiles < resident ? prm.tiles : resident;
  cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, tc_pair_kernel<SA, kB, NG>, tmA, tmW, prm);
}

template <bool kB>
cudaError_t launch_pair_sa(int sa, int ng, const CUtensorMap& tmA, const CUtensorMap& tmW,
                           const PairParams& prm, size_t smem, cudaStream_t stream) {
  if (ng == 4)
    return sa == 2 ? launch_pair_kernel<2, kB, 4>(tmA, tmW, prm, smem, stream)
                   : launch_pair_kernel<1, kB, 4>(tmA, tmW, prm, smem, stream);
  return sa == 2 ? launch_pair_kernel<2, kB, 2>(tmA, tmW, prm, smem, stream)
                 : launch_pair_kernel<1, kB, 2>(tmA, tmW, prm, smem, stream);
}

}  // namespace

int tc_pair_token_tile(int M) { return M > 128 ? 256 : 128; }

int tc_pair_stage_atoms(int K, int group) { return K % 128 == 0 && group % 128 == 0 ? 2 : 1; }

bool tc_pair_config(int M, int K, int group, int out[7]) {
  const int bt = tc_pair_token_tile(M);
  const int sa = tc_pair_stage_atoms(K, group);
  const PairRings r = pair_rings(bt, sa);
  out[0] = bt;
  out[1] = sa;
  out[2] = r.act;
  out[3] = r.code;
  out[4] = r.dq;
  out[5] = r.groups;
  out[6] = (int)r.smem;
  return pair_rings_valid(r);
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
  prm.tiles_m = (M + bt - 1) / bt;
  prm.tiles = prm.tiles_m * ((N + 2 * kCols - 1) / (2 * kCols));
  return bf16 ? launch_pair_sa<true>(sa, rings.groups, tmA, tmW, prm, rings.smem, stream)
              : launch_pair_sa<false>(sa, rings.groups, tmA, tmW, prm, rings.smem, stream);
}

}  // namespace w4a16
