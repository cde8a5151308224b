// Tensor-core path of the W4A16 linear layer (sm_103a, tcgen05 + TMEM + TMA).
//
// At large M the layer is a dense contraction: once the weights are
// dequantized, what remains is an ordinary fp16 matrix product (the point made
// in the vLLM PR #1032 thread). Here CUDA cores dequantize the int4 weights
// straight into tensor memory, which tcgen05.mma kind::f16 reads as its A
// operand; the activations are the B operand, in shared memory; the fp32
// accumulators are in tensor memory too.
//
// Orientation: D[n][m] = sum_k Wdeq[n][k] * A[m][k]: weight column n is
// tensor-memory lane n of the 128-row A operand and of the accumulator, the
// tokens are the MMA's N dimension (16..256). Each dequantized weight serves
// up to 256 tokens.
//
// Shared memory per SM carries only the copies of the packed codes and of the
// activations and their reads; the dequantized operand (16 KiB per 64 k of a
// 128-column tile) never passes through it, which leaves room for rings deep
// enough to cover a DRAM round trip.
//
// CTA (one output tile of 128 columns x BT tokens over one K range):
//   warp 0      TMA producer (one thread, polling): the packed codes of the
//               tile's 8 strips (a 3-D map with the 128-byte swizzle, so that
//               the dequantizing threads' 16-byte reads of one column each
//               fall on distinct banks) up to the code ring's depth ahead,
//               and the activations [BT x 64 k] per atom (128-byte swizzle)
//               up to the activation ring's depth ahead;
//   warp 1      tensor-memory allocation; one thread issues 4 MMAs per 64 k
//               of a stage, A from tensor memory;
//   warps 2..9  two groups of four warps, one warp per lane quarter; group g
//               converts the stages g, g + 2, ...: each thread dequantizes
//               one weight column's k of the stage into 32-bit tensor-memory
//               cells of its own lane (tcgen05.st 32x32b); then the epilogue
//               (tensor memory -> Y).
// Rings and their barriers: activations (act_full; stage_done when the
// stage's MMAs completed, which also frees the stage's dequantized slot),
// packed codes (code_full, code_empty once the converting warps hold them in
// registers), dequantized operand in tensor memory (dq_full, after the
// converting warps' stores and the stage's activations landed).
// Every wait is bounded; a wait that gives up sets the library's device error
// word and the CTA drains and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace w4a16 {

__device__ int g_device_error = 0;

namespace {

constexpr int kTileN = 128;        // output columns per CTA (MMA M)
constexpr int kStageK = 64;        // k per atom (one 128-byte swizzle row of activations)
// NG groups of four dequantizing warps (one warp per tensor-memory lane
// quarter): 2 at two CTAs per SM, 4 at one
template <int NG>
struct Warps {
  static constexpr int kDqThreads = 128 * NG;
  static constexpr int kThreads = 64 + kDqThreads;
};
constexpr int kCodeAtomBytes = kTileN * kStageK / 2;  // 4 KiB: 8 strips x 512 B
constexpr int kAtomCols = kStageK / 2;  // tensor-memory columns of one atom's A operand
constexpr size_t kTcCounterBytes = 32768;  // tile counters of a K-split launch
constexpr int kBarBytes = 1024;            // barriers and flags after the rings

using namespace tc;

// ------------------------------------------------------------------ kernel

struct TcParams {
  const uint16_t* Sp;
  const uint32_t* Zp;
  uint16_t* Y;
  int* counters;  // split > 1: one per output tile, zero between calls
  float* tiles;   // split > 1: fp32 partial tiles [tile][split][bt][128]
  size_t tile_floats;  // extent of `tiles` (for the checked build)
  int M, N, K, group;
  int bt;          // token tile (MMA N): multiple of 16, 16..256
  int act_slots;   // activation ring depth (stages)
  int code_slots;  // packed-code ring depth (stages)
  int dq_slots;    // dequantized-operand ring depth (stages), at most act_slots
  int dq_col0;     // first tensor-memory column of the dequantized-operand ring
  int tmem_cols;
  int split;       // K ranges per output tile (grid z)
  int early_weights;  // weights are static: read the first stages' codes and
                      // scales before the grid-dependency wait
  const float* row_scale;  // W4A8: per-row factors of the result, or null
  int* err;                // the library's error word
};

// named barrier of the dequant/epilogue warps
template <int NT>
__device__ __forceinline__ void epilogue_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

// SA: atoms (64 k) per pipeline stage, 1 or 2. Larger stages cut the
// barrier hand-offs per weight byte; SA = 2 needs K and the group to be
// multiples of 128 (one scale and zero point per stage). NG: dequant groups.
template <int SA, bool kB, int NG>
__global__ void __launch_bounds__(Warps<NG>::kThreads, NG == 2 ? 2 : 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
               const TcParams p) {
  static_assert(SA == 1 || SA == 2, "stages of one or two 64-k atoms");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const int bt = p.bt, nact = p.act_slots, ncode = p.code_slots, ndq = p.dq_slots;
  const uint32_t atom_act = (uint32_t)bt * 128u;  // one atom of activations
  const uint32_t act_bytes = SA * atom_act;
  const uint32_t code_bytes = SA * kCodeAtomBytes;
  // [activation ring | code ring | barriers], slots 1024-aligned
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
  volatile int* last_flag = reinterpret_cast<volatile int*>(gen_base + (tmem_slot + 8u - base));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // grid: x = token tiles (fastest, so the token tiles of one column tile run
  // together and its weights are read from DRAM once), y = column tiles, z = K
  // ranges
  const int n0 = blockIdx.y * kTileN;
  const int m0 = blockIdx.x * bt;
  // this CTA's K range: stages [kb0, kb0 + nk)
  const int nk_all = p.K / (kStageK * SA);
  const int kb0 = (int)((long long)blockIdx.z * nk_all / p.split);
  const int nk = (int)((long long)(blockIdx.z + 1) * nk_all / p.split) - kb0;

  if (threadIdx.x == 0) {
    for (int a = 0; a < nact; ++a) {
      mbar_init(act_full(a), 1);
      mbar_init(stage_done(a), 1);
    }
    for (int w = 0; w < ndq; ++w) mbar_init(dq_full(w), 4);  // the group's four warps
    for (int c = 0; c < ncode; ++c) {
      mbar_init(code_full(c), 1);
      mbar_init(code_empty(c), 4);
    }
    mbar_init(accum_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(gen_base + (tmem_slot - base));
  // the next grid may be scheduled now: its CTAs land on SMs as this grid's
  // CTAs leave them, and it waits for this grid before it touches memory
  allow_dependent_launch();

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    // One thread keeps both rings full: it polls the slot of the next copy of
    // each ring and issues whichever is free, so that neither ring waits for
    // the other's slots.
    if (lane == 0) {
      auto codes = [&](int kb, int c) {
        if (!in_smem(code_base + (uint32_t)c * code_bytes, code_bytes, raw, p.err)) return;
        mbar_expect_tx(code_full(c), code_bytes);
        tma_load_3d(code_base + (uint32_t)c * code_bytes, &tmW, 0, (kb0 + kb) * SA * 4,
                    n0 / kStripCols, code_full(c));
      };
      auto acts = [&](int kb, int a) {
        const uint32_t st = base + (uint32_t)a * act_bytes;
        if (!in_smem(st, act_bytes, raw, p.err)) return;
        mbar_expect_tx(act_full(a), act_bytes);
#pragma unroll
        for (int u = 0; u < SA; ++u)
          tma_load_2d(st + u * atom_act, &tmA, ((kb0 + kb) * SA + u) * kStageK, m0, act_full(a));
      };
      int ci = 0, ai = 0;
      RingPos cpos{0, 0u}, apos{0, 0u};  // ring positions of stages ci and ai
      // static weights: the first ring of codes goes out before the wait for
      // the previous grid (the slots are free: nothing has used them yet)
      if (p.early_weights)
        for (; ci < nk && ci < ncode; ++ci, cpos.step(1, ncode)) codes(ci, cpos.slot);
      grid_dependency_wait();
      uint64_t t0 = globaltimer();
      uint32_t idle = 0;
      while (ci < nk || ai < nk) {
        bool progress = false;
        if (ci < nk && mbar_test(code_empty(cpos.slot), cpos.phase ^ 1u)) {
          codes(ci++, cpos.slot);
          cpos.step(1, ncode);
          progress = true;
        }
        if (ai < nk && mbar_test(stage_done(apos.slot), apos.phase ^ 1u)) {
          acts(ai++, apos.slot);
          apos.step(1, nact);
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
        // let the copies already issued land before the CTA exits
        for (int kb = (ai > nact ? ai - nact : 0); kb < ai; ++kb)
          mbar_drain(act_full(kb % nact), (uint32_t)(kb / nact) & 1u, p.err);
        for (int kb = (ci > ncode ? ci - ncode : 0); kb < ci; ++kb)
          mbar_drain(code_full(kb % ncode), (uint32_t)(kb / ncode) & 1u, p.err);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // dq_full completes when the stage's four converting warps have arrived,
    // each after its tensor-memory stores completed and the stage's
    // activations landed: one test covers both operands. The next stage's
    // barrier is tested between this stage's MMAs, while the tensor core
    // works through the queued ones.
    if (lane == 0) {
      const uint32_t idesc = f16_idesc(kTileN, bt, kB);
      int a = 0, w = 0;
      uint32_t pw = 0;
      bool ok = nk > 0 && in_tmem(0, (uint32_t)bt, (uint32_t)p.tmem_cols, p.err) &&
                mbar_wait(dq_full(0), 0, abort_flag, kErrMma, p.err);
      for (int kb = 0; kb < nk && ok; ++kb) {
        tc_fence_after();
        const uint32_t bst = base + (uint32_t)a * act_bytes;
        const uint32_t acol = tmem_base + (uint32_t)(p.dq_col0 + w * SA * kAtomCols);
        if (!in_smem(bst, act_bytes, raw, p.err) ||
            !in_tmem((uint32_t)(p.dq_col0 + w * SA * kAtomCols), SA * kAtomCols, (uint32_t)p.tmem_cols, p.err)) {
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
            tc_mma_f16_ts(tmem_base, acol + (uint32_t)(u * kAtomCols + 8 * kk), bdesc + 2u * kk, idesc,
                          (kb | u | kk) != 0);
            if (u == 0 && kk == 1 && kb + 1 < nk) ready = mbar_test(dq_full(w2), pw2);
          }
        }
        tc_commit(stage_done(a));
        a = a + 1 == nact ? 0 : a + 1;
        w = w2;
        pw = pw2;
        if (kb + 1 < nk && !ready) ok = mbar_wait(dq_full(w), pw, abort_flag, kErrMma, p.err);
      }
      tc_commit(accum_bar);  // fires once every MMA issued above has completed
      if (!ok) mbar_drain(accum_bar, 0, p.err);  // no MMA may run past the TMEM release
    }
  } else {
    // ---------------------------------------------------------- dequant + epilogue
    // NG groups of four warps; group g converts the stages g, g + NG, ...
    // Thread (lane quarter q, lane) owns weight column 32 q + lane of the
    // tile: tensor-memory lane 32 q + lane, strip 2 q + lane / 16, column c =
    // lane % 16 of the strip. In the packed format the 16 bytes at 64 (c % 8)
    // + 16 l (l = 0..3) of a strip's atom hold the words of k-octets l and
    // 4 + l of columns c % 8 (words 0, 2) and c % 8 + 8 (words 1, 3).
    const int dw = warp - 2;
    const int grp_id = dw >> 2;  // this warp's group
    const int q = warp & 3;      // lane quarter
    const int ls = 2 * q + (lane >> 4);
    const int c = lane & 15, cp = c & 7;
    const bool hi = c >= 8;
    const int strip = n0 / kStripCols + ls;
    const bool live = strip < p.N / kStripCols;
    const int G = p.K / p.group;
    const uint32_t tlane = (uint32_t)(32 * q) << 16;
    // scale bits (low half) and zero point (bits 16..19) of this column for
    // each 128 k of a stage (one group: SA >= 2 needs groups of 128 or more)
    constexpr int MH = SA >= 2 ? SA / 2 : 1;
    struct Meta {
      uint32_t v[MH];
    };
    // the stages' meta are loaded in order, NG stages apart: the group of
    // stage mkb is followed without a division (gk = k of the stage's first
    // atom, gend = k where the group after the stage's group starts)
    int mkb = grp_id, mgrp = 0, mgend = p.group;
    auto meta_step = [&]() {
      mkb += NG;
      const int gk = (kb0 + mkb) * SA * kStageK;
      while (gk >= mgend) {
        ++mgrp;
        mgend += p.group;
      }
    };
    {
      const int gk = (kb0 + mkb) * SA * kStageK;
      mgrp = gk / p.group;
      mgend = (mgrp + 1) * p.group;
    }
    // loads the meta of stage mkb into m and steps to the group's next stage
    auto load_meta = [&](Meta& m) {
#pragma unroll
      for (int h = 0; h < MH; ++h) {
        m.v[h] = 0u;
        if (mkb < nk && live) {
          // SA >= 2: groups of 128 k or more, and the second 128 k of a stage
          // starts a new group exactly when it reaches gend
          const int grp = mgrp + ((h > 0 && (kb0 + mkb) * SA * kStageK + h * 128 >= mgend) ? 1 : 0);
          const size_t pg = (size_t)strip * G + grp;
          const uint8_t* zp = reinterpret_cast<const uint8_t*>(p.Zp);
          const uint32_t sb = *ld_at(p.Sp + pg * 16 + 2 * cp + (hi ? 1 : 0), p.Sp, (size_t)G * p.N, p.err);
          const uint32_t zb = *ld_at(zp + pg * 8 + cp, zp, (size_t)G * p.N / 2, p.err);
          m.v[h] = sb | (((zb >> (hi ? 4 : 0)) & 15u) << 16);
        }
      }
      meta_step();
    };
    // one stage: wait for its codes, read this column's words, release the
    // codes; wait for the tensor-memory slot; dequantize and store; wait for
    // the stage's activations; arrive
    // ring positions of this group's next stage kb (its stages are NG apart)
    RingPos spos_code, spos_act;
    spos_code.init(grp_id, ncode);
    spos_act.init(grp_id, nact);
    int sw = grp_id % ndq;
    auto stage = [&](int kb, const Meta& meta) -> bool {
      const int cs = spos_code.slot, a = spos_act.slot, w = sw;
      const uint32_t code_par = spos_code.phase, act_par = spos_act.phase;
      const RingPos prev = spos_act.before(ndq, nact);  // stage kb - dq_slots (dq_slots <= act_slots)
      spos_code.step(NG, ncode);
      spos_act.step(NG, nact);
      sw += NG;
      while (sw >= ndq) sw -= ndq;
      if (!mbar_wait(code_full(cs), code_par, abort_flag, kErrDequant, p.err))
        return false;
      const uint32_t cb = code_base + (uint32_t)cs * code_bytes;
      // the slot's previous stage (kb - dq_slots) has completed its MMAs
      auto wait_slot = [&]() -> bool {
        if (kb < ndq) return true;
        if (!mbar_wait(stage_done(prev.slot), prev.phase, abort_flag, kErrDequant, p.err))
          return false;
        tc_fence_after();
        return true;
      };
      // atoms are read and converted CA at a time (four atoms of words would
      // not fit the registers of 18 warps); the codes are released once the
      // last ones are in registers
      constexpr int CA = SA > 2 ? 2 : SA;
      if (SA > CA && !wait_slot()) return false;
      const uint32_t tcol = tmem_base + tlane + (uint32_t)(p.dq_col0 + w * SA * kAtomCols);
#pragma unroll
      for (int u0 = 0; u0 < SA; u0 += CA) {
        uint32_t wl[CA][4], wh[CA][4];  // k-octets l and 4 + l of each atom
#pragma unroll
        for (int u = 0; u < CA; ++u) {
          const uint32_t row = (uint32_t)(ls * 4 * SA + 4 * (u0 + u) + (cp >> 1));  // 128-byte row of the tile
#pragma unroll
          for (int l = 0; l < 4; ++l) {
            const uint32_t chunk = ((uint32_t)(4 * (cp & 1) + l)) ^ (row & 7u);  // 128-byte swizzle
            const uint32_t at = cb + row * 128u + (chunk << 4);
            const uint4 v = lds128(in_smem(at, 16, raw, p.err) ? at : cb);
            wl[u][l] = hi ? v.y : v.x;
            wh[u][l] = hi ? v.w : v.z;
          }
        }
        if (u0 + CA == SA) {
          __syncwarp();
          if (lane == 0) mbar_arrive(code_empty(cs));  // the codes are in registers
          if (SA == CA && !wait_slot()) return false;
        }
#pragma unroll
        for (int u = 0; u < CA; ++u) {
          const uint32_t mv = meta.v[(u0 + u) / 2 < MH ? (u0 + u) / 2 : 0];
          const uint32_t z = (mv >> 16) & 15u;
          const uint16_t s = (uint16_t)(mv & 0xffffu);
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
          if (in_tmem((uint32_t)(p.dq_col0 + w * SA * kAtomCols + (u0 + u) * kAtomCols), kAtomCols,
                      (uint32_t)p.tmem_cols, p.err))
            tmem_st32(tcol + (uint32_t)((u0 + u) * kAtomCols), r);
        }
      }
      tmem_wait_st();
      // the stage's activations have landed (the MMAs read them too)
      if (!mbar_wait(act_full(a), act_par, abort_flag, kErrDequant, p.err))
        return false;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_full(w));
      return true;
    };
    // scales and zero points: three register sets in rotation, each loaded two
    // of this group's stages before its own (no stage waits for its loads).
    // They are weights: with static weights the first sets are read before the
    // wait for the previous grid (which orders this warp's stores of Y)
    Meta m0s, m1s, m2s;
    if (p.early_weights) {
      load_meta(m0s);  // stage grp_id
      load_meta(m1s);  // stage grp_id + NG
    }
    grid_dependency_wait();
    if (!p.early_weights) {
      load_meta(m0s);
      load_meta(m1s);
    }
    for (int kb = grp_id; kb < nk; kb += 3 * NG) {
      load_meta(m2s);  // stage kb + 2 NG
      if (!stage(kb, m0s) || kb + NG >= nk) break;
      load_meta(m0s);  // kb + 3 NG
      if (!stage(kb + NG, m1s) || kb + 2 * NG >= nk) break;
      load_meta(m1s);  // kb + 4 NG
      if (!stage(kb + 2 * NG, m2s)) break;
    }

    // epilogue: TMEM lanes 32q..32q+31 are output columns, TMEM columns are tokens
    const bool have_accum = mbar_wait(accum_bar, 0, abort_flag, kErrEpilogue, p.err);
    __syncwarp();
    if (__all_sync(0xffffffffu, have_accum)) {  // warp-uniform: tcgen05.ld is .aligned
      tc_fence_after();
      const int half = dw >> 2;  // the NG warpgroups split the token chunks
      const int n = n0 + 32 * q + lane;
      float* part = p.tiles + (((size_t)blockIdx.y * gridDim.x + blockIdx.x) * p.split + blockIdx.z) *
                                  (size_t)bt * kTileN;
      for (int ch = half; ch < bt / 16; ch += NG) {
        uint32_t r[16];
        tmem_ld16(tmem_base + tlane + (uint32_t)(16 * ch), r);
        tmem_wait_ld();
        if (p.split > 1) {  // fp32 partial tile [token][column]
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float* d = part + (16 * ch + j) * kTileN + 32 * q + lane;
            if (in_buf(d, p.tiles, p.tile_floats, p.err)) *d = __uint_as_float(r[j]);
          }
        } else if (n < p.N) {
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
    if (p.split > 1) {
      // K split: the last of the tile's CTAs to arrive sums the partial tiles in
      // split order (deterministic), writes Y and resets the tile's counter
      const int tile = blockIdx.y * gridDim.x + blockIdx.x;
      epilogue_bar<Warps<NG>::kDqThreads>();  // every partial store issued; one release atomic covers them
      if (dw == 0 && lane == 0) {
        int old = 0;
        if (*abort_flag == 0 && in_buf(p.counters + tile, p.counters, kTcCounterBytes / sizeof(int), p.err))
          asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                       : "=r"(old)
                       : "l"(p.counters + tile)
                       : "memory");
        *last_flag = (*abort_flag == 0) && old == p.split - 1;
      }
      epilogue_bar<Warps<NG>::kDqThreads>();
      if (*last_flag) {
        // 4 columns per float4, 8 float4 per thread and round: the loads of
        // one partial tile for the round are all in flight together, and the
        // partial tiles are added in split order
        const float4* tb = reinterpret_cast<const float4*>(p.tiles + (size_t)tile * p.split * bt * kTileN);
        const int n4 = bt * kTileN / 4;
        constexpr int kRound = 8;
        for (int e0 = dw * 32 + lane; e0 < n4; e0 += kRound * Warps<NG>::kDqThreads) {
          float4 acc[kRound];
#pragma unroll
          for (int u = 0; u < kRound; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int z = 0; z < p.split; ++z) {
            float4 v[kRound];
#pragma unroll
            for (int u = 0; u < kRound; ++u) {
              const int e = e0 + u * Warps<NG>::kDqThreads;
              const float4* src = tb + (size_t)z * (n4) + e;
              v[u] = e < n4 ? __ldcg(ld_at(src, reinterpret_cast<const float4*>(p.tiles), p.tile_floats / 4, p.err))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kRound; ++u) {
              acc[u].x += v[u].x;
              acc[u].y += v[u].y;
              acc[u].z += v[u].z;
              acc[u].w += v[u].w;
            }
          }
#pragma unroll
          for (int u = 0; u < kRound; ++u) {
            const int e = e0 + u * Warps<NG>::kDqThreads;
            const int tok = m0 + e / (kTileN / 4), n = n0 + (e % (kTileN / 4)) * 4;
            if (e < n4 && tok < p.M && n < p.N) {
              const float f = p.row_scale ? *ld_at(p.row_scale + tok, p.row_scale, (size_t)p.M, p.err) : 1.0f;
              uint2 o;
              o.x = to_out2<kB>(acc[u].x * f, acc[u].y * f);
              o.y = to_out2<kB>(acc[u].z * f, acc[u].w * f);
              uint16_t* d = p.Y + (size_t)tok * p.N + n;
              if (in_buf(d, p.Y, (size_t)p.M * p.N - 3, p.err)) *reinterpret_cast<uint2*>(d) = o;
            }
          }
        }
        if (dw == 0 && lane == 0 && in_buf(p.counters + tile, p.counters, kTcCounterBytes / sizeof(int), p.err))
          p.counters[tile] = 0;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, (uint32_t)p.tmem_cols);
  }
}

// ------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    return nullptr;
  }();
  return fn;
}


}  // namespace

int tc_token_tile(int M) {
  if (M >= 256) return 256;
  return (M + 15) / 16 * 16;
}

// CTAs per SM the tensor-core kernel is sized for: two when the token tile is
// at most 64 (the middle band of M: few output tiles, which a K split then
// spreads over both CTA slots of every SM; measured at 64 tokens, 2 CTAs
// against 1: 70B qkv 37.2 -> 31.3 us, 13B gate_up 56.4 -> 48.0, 13B down
// 28.0 -> 25.7, 13B qkv 28.2 -> 28.4), else one.
int tc_ctas_per_sm(int bt) { return bt <= 64 ? 2 : 1; }

namespace {

struct TcRings {
  int act, code, dq;  // ring depths in stages
  int groups;         // dequant groups (2 or 4)
  int dq_col0, tmem_cols;
  size_t smem;
};

// Ring depths of a token tile. Codes: 16 atoms (64 KiB), 8 at two CTAs per
// SM or for tiles of 192 tokens and more (whose activation slots are large).
// Activations: as deep as the rest of the shared memory allows, at most 16
// atoms. Dequantized operand: in the tensor memory the accumulator leaves, at
// most 16 atoms and no deeper than the activation ring. Dequant groups: four
// where one CTA per SM has at least four activation slots, else two.
//
// A parity wait is unambiguous only while its barrier is at most one phase
// away from the awaited one. Group g waits for stage kb's codes, for the MMAs
// of stage kb - dq (its slot) and for stage kb's activations; it has already
// seen its own previous stage kb - groups through the same three waits. So:
//   - code slots are a multiple of the groups: the previous stage in stage
//     kb's code slot is one of this group's own, whose codes have landed;
//   - activation slots (which index stage_done) are at least the groups and
//     at least the dequantized slots: the previous phase of the awaited
//     stage_done, stage kb - dq - act, is no later than kb - groups - dq,
//     whose MMAs the group saw complete (MMAs complete in order), and the
//     previous phase of stage kb's act_full, stage kb - act, is no later than
//     kb - dq, whose MMAs read those activations.
TcRings tc_rings(int bt, int sa) {
  TcRings r;
  const bool two = tc_ctas_per_sm(bt) == 2;
  const size_t budget = (size_t)(two ? 113 : 227) * 1024 - 1024 - kBarBytes;
  r.code = ((two || bt >= 192) ? 8 : 16) / sa;
  const size_t act_slot = (size_t)sa * bt * 128;
  const size_t code_slot = (size_t)sa * kCodeAtomBytes;
  int act = (int)((budget - (size_t)r.code * code_slot) / act_slot);
  // one CTA per SM: a shorter code ring (down to 4 slots) where it buys the
  // fourth activation slot, and with it four dequant groups instead of two
  // (176-token tiles: 5-18% faster on the Llama layers)
  while (!two && act < 4 && r.code > 4 &&
         (int)((budget - (size_t)(r.code / 2) * code_slot) / act_slot) >= 4) {
    r.code /= 2;
    act = (int)((budget - (size_t)r.code * code_slot) / act_slot);
  }
  r.act = act > 16 / sa ? 16 / sa : act;
  r.groups = !two && r.act >= 4 ? 4 : 2;
  r.tmem_cols = two ? 256 : 512;
  r.dq_col0 = (bt + 31) / 32 * 32;
  int dq = (r.tmem_cols - r.dq_col0) / (sa * kAtomCols);
  if (dq > 16 / sa) dq = 16 / sa;
  r.dq = dq > r.act ? r.act : dq;
  r.smem = (size_t)r.act * act_slot + (size_t)r.code * code_slot + 1024 + kBarBytes;
  return r;
}

bool tc_rings_valid(const TcRings& r) {
  return r.dq >= 1 && r.dq <= r.act && r.act >= r.groups && r.code % r.groups == 0;
}

}  // namespace

// Atoms per stage: two when K and the group are multiples of 128 (one scale
// and zero point per stage), else one.
int tc_stage_atoms(int M, int K, int group) {
  (void)M;
  return K % 128 == 0 && group % 128 == 0 ? 2 : 1;
}

bool tc_config(int M, int K, int group, int out[8]) {
  const int bt = tc_token_tile(M);
  const int sa = tc_stage_atoms(M, K, group);
  const TcRings r = tc_rings(bt, sa);
  out[0] = bt;
  out[1] = sa;
  out[2] = r.act;
  out[3] = r.code;
  out[4] = r.dq;
  out[5] = r.groups;
  out[6] = (int)r.smem;
  out[7] = tc_ctas_per_sm(bt);
  return tc_rings_valid(r);
}

size_t tc_workspace_bytes(int M, int N, int split) {
  if (split <= 1) return 0;
  const int bt = tc_token_tile(M);
  const size_t tiles = (size_t)((N + kTileN - 1) / kTileN) * ((M + bt - 1) / bt);
  return kTcCounterBytes + tiles * (size_t)split * bt * kTileN * sizeof(float);
}

// K split of the tensor-core GEMM.
// Token tiles of 64..256 (one CTA per SM): a CTA streams its K range at a rate
// per 64-k stage that does not depend on the split, so a launch takes about
// waves x (stages per CTA + the fix-up of a split tile by its last CTA, about
// 2 + split stages, 12 + split for 256-token tiles whose 128 KiB partial
// tiles cost HBM time); the split minimizes that, keeping at least 8 stages
// per CTA (measured on the Llama middle band: 13B gate_up at 64 rows 68.9 ->
// 62.3 us with 2 ranges, 70B down at 64 rows 108 -> 95 us with 7; 70B qkv at
// 512 rows, 160 tiles on 152 SMs, 126 -> 120 us with 3).
// Other tiles: only when the output tiles cannot fill the SMs; among splits
// that keep >= 8 stages per CTA, the score is the wave efficiency times the
// share of weight bytes in the traffic once the fp32 partial tiles (written
// and read back) are counted.
int tc_choose_split(int M, int N, int K, int group, int sms) {
  const int bt = tc_token_tile(M);
  const long tiles = (long)((N + kTileN - 1) / kTileN) * ((M + bt - 1) / bt);
  const long slots = (long)sms * tc_ctas_per_sm(bt);
  if (tiles > (long)(kTcCounterBytes / sizeof(int))) return 1;
  const int sa = tc_stage_atoms(M, K, group);
  const long stages = K / (kStageK * sa);  // pipeline stages of the whole K
  const long nk = K / kStageK;             // atoms (costs are counted in atoms)
  if (bt >= 64) {
    const long fixup = bt > 128 ? 12 : 2;
    int best = 1;
    long best_cost = -1;
    for (int split = 1; split <= 16 && split <= stages && (split == 1 || nk / split >= 8); ++split) {
      const long waves = (tiles * split + slots - 1) / slots;
      const long cost = waves * ((stages + split - 1) / split * sa + (split > 1 ? fixup + split : 0));
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        best = split;
      }
    }
    return best;
  }
  if (tiles >= slots) return 1;
  const double wbytes = (double)K * N / 2 + 2.0 * M * K;
  int best = 1;
  double best_score = -1.0;
  for (int split = 1; split <= 16 && split <= stages && nk / split >= 8; ++split) {
    const long total = tiles * split;
    const long waves = (total + slots - 1) / slots;
    const double eff = (double)total / (double)(waves * slots);
    const double part = split > 1 ? 2.0 * tiles * split * bt * kTileN * 4.0 : 0.0;
    const double score = eff * wbytes / (wbytes + part);
    if (score > best_score + 0.01) {
      best_score = score;
      best = split;
    }
  }
  return best;
}

namespace {

template <int SA, bool kB, int NG>
cudaError_t launch_kernel(const CUtensorMap& tmA, const CUtensorMap& tmW, const TcParams& prm,
                          dim3 grid, size_t smem, cudaStream_t stream) {
  cudaError_t e = set_max_smem_once(reinterpret_cast<const void*>(tc_gemm_kernel<SA, kB, NG>), 227 * 1024);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(Warps<NG>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<SA, kB, NG>, tmA, tmW, prm);
}

template <bool kB>
cudaError_t launch_sa(int sa, int ng, const CUtensorMap& tmA, const CUtensorMap& tmW, const TcParams& prm,
                      dim3 grid, size_t smem, cudaStream_t stream) {
  if (ng == 2)
    return sa == 2 ? launch_kernel<2, kB, 2>(tmA, tmW, prm, grid, smem, stream)
                   : launch_kernel<1, kB, 2>(tmA, tmW, prm, grid, smem, stream);
  return sa == 2 ? launch_kernel<2, kB, 4>(tmA, tmW, prm, grid, smem, stream)
                 : launch_kernel<1, kB, 4>(tmA, tmW, prm, grid, smem, stream);
}

}  // namespace

// Encoded tensor maps of recent calls, keyed by what they encode: encoding
// one costs a driver call, and a layer calls with the same pointers and
// shapes every step. A small table per process, replaced round-robin.
namespace {

struct MapKey {
  const void* ptr;
  uint64_t dims[3];
  uint32_t box[3];
  int dtype, rank, swizzle;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && dims[0] == o.dims[0] && dims[1] == o.dims[1] && dims[2] == o.dims[2] &&
           box[0] == o.box[0] && box[1] == o.box[1] && box[2] == o.box[2] && dtype == o.dtype &&
           rank == o.rank && swizzle == o.swizzle;
  }
};
constexpr int kMapCache = 64;
std::mutex g_map_mutex;
MapKey g_map_keys[kMapCache];
CUtensorMap g_maps[kMapCache];
int g_map_used = 0, g_map_next = 0;

// A densely packed row-major array of rank 2 or 3 (dims[0] innermost).
bool cached_map(CUtensorMap* out, const void* ptr, CUtensorMapDataType dt, int esize, int rank,
                const uint64_t (&dims)[3], const uint32_t (&box)[3], CUtensorMapSwizzle swizzle) {
  const MapKey key = {ptr, {dims[0], dims[1], dims[2]}, {box[0], box[1], box[2]}, (int)dt, rank,
                      (int)swizzle};
  {
    std::lock_guard<std::mutex> lock(g_map_mutex);
    for (int i = 0; i < g_map_used; ++i)
      if (g_map_keys[i] == key) {
        *out = g_maps[i];
        return true;
      }
  }
  PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
  if (!encode) return false;
  const cuuint64_t gdims[3] = {(cuuint64_t)dims[0], (cuuint64_t)dims[1], (cuuint64_t)dims[2]};
  const cuuint64_t strides[2] = {(cuuint64_t)dims[0] * esize, (cuuint64_t)dims[0] * dims[1] * esize};
  const cuuint32_t gbox[3] = {box[0], box[1], box[2]};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (encode(out, dt, (cuuint32_t)rank, const_cast<void*>(ptr), gdims, strides, gbox, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lock(g_map_mutex);
  const int slot = g_map_used < kMapCache ? g_map_used++ : (g_map_next++ % kMapCache);
  g_map_keys[slot] = key;
  g_maps[slot] = *out;
  return true;
}

}  // namespace

bool cached_tensor_map(CUtensorMap* out, const void* ptr, CUtensorMapDataType dt, int esize,
                       uint64_t dims0, uint64_t dims1, uint32_t box0, uint32_t box1,
                       CUtensorMapSwizzle swizzle) {
  return cached_map(out, ptr, dt, esize, 2, {dims0, dims1, 1}, {box0, box1, 1}, swizzle);
}

bool cached_code_map(CUtensorMap* out, const uint32_t* Wq, int N, int K, int sa) {
  return cached_map(out, Wq, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, 3,
                    {32, (uint64_t)(K / kAtomK) * 4, (uint64_t)(N / kStripCols)},
                    {32, (uint32_t)(4 * sa), (uint32_t)(kTileN / kStripCols)}, CU_TENSOR_MAP_SWIZZLE_128B);
}

cudaError_t launch_tc_gemm(const uint16_t* A, const uint32_t* Wq, const uint16_t* Sp,
                           const uint32_t* Zp, uint16_t* Y, int M, int N, int K, int group,
                           int split, void* workspace, bool early_weights, bool bf16,
                           const float* row_scale, cudaStream_t stream) {
  const int bt = tc_token_tile(M);
  const int sa = tc_stage_atoms(M, K, group);
  CUtensorMap tmA, tmW;
  if (!cached_tensor_map(&tmA, A, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  2, (uint64_t)K, (uint64_t)M, 64, (uint32_t)bt, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // packed weights viewed as [N/16 strips][K/64 atoms * 4 rows][32 words] of
  // uint32: a box is the stage's SA atoms of the tile's 8 strips, 128-byte rows
  // swizzled
  if (!cached_code_map(&tmW, Wq, N, K, sa)) return cudaErrorInvalidValue;
  TcParams prm;
  prm.Sp = Sp;
  prm.Zp = Zp;
  prm.Y = Y;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.group = group;
  prm.bt = bt;
  prm.split = split < 1 ? 1 : split;
  prm.row_scale = row_scale;
  prm.early_weights = early_weights ? 1 : 0;
  cudaError_t e = device_error_word(&prm.err);
  if (e != cudaSuccess) return e;
  prm.counters = static_cast<int*>(workspace);
  prm.tiles = workspace ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kTcCounterBytes)
                        : nullptr;
  prm.tile_floats = workspace ? (tc_workspace_bytes(M, N, prm.split) - kTcCounterBytes) / sizeof(float) : 0;
  const TcRings rings = tc_rings(bt, sa);
  prm.act_slots = rings.act;
  prm.code_slots = rings.code;
  prm.dq_slots = rings.dq;
  prm.dq_col0 = rings.dq_col0;
  prm.tmem_cols = rings.tmem_cols;
  const size_t smem = rings.smem;
  const dim3 grid((unsigned)((M + bt - 1) / bt), (unsigned)((N + kTileN - 1) / kTileN),
                  (unsigned)prm.split);
  const int ng = rings.groups;
  if (!tc_rings_valid(rings)) return cudaErrorInvalidValue;
  return bf16 ? launch_sa<true>(sa, ng, tmA, tmW, prm, grid, smem, stream)
              : launch_sa<false>(sa, ng, tmA, tmW, prm, grid, smem, stream);
}

namespace {

// Self-test of the pipeline's bounded wait: one thread initializes an
// mbarrier that nothing ever arrives on and waits for its first phase with
// the kernel's own wait routine and limit. The wait gives up, records
// kErrMma in the error word, and the kernel returns.
__global__ void selftest_mbar_kernel(int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  const uint32_t b = (uint32_t)__cvta_generic_to_shared(&bar);
  mbar_init(b, 1);
  abort_flag = 0;
  fence_barrier_init();
  mbar_wait(b, 0, &abort_flag, kErrMma, err);
}

}  // namespace

cudaError_t launch_selftest_mbar_wait(cudaStream_t stream) {
  int* err = nullptr;
  cudaError_t e = device_error_word(&err);
  if (e != cudaSuccess) return e;
  selftest_mbar_kernel<<<1, 32, 0, stream>>>(err);
  return cudaGetLastError();
}

cudaError_t device_error_word(int** ptr) {
  static int* cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && cache[dev]) {
    *ptr = cache[dev];
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_device_error);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) cache[dev] = static_cast<int*>(p);
  *ptr = static_cast<int*>(p);
  return cudaSuccess;
}

cudaError_t read_and_clear_device_error(int* flag) {
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_device_error, sizeof(int));
  if (e != cudaSuccess || *flag == 0) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

}  // namespace w4a16
