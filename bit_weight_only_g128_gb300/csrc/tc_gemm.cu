// Tensor-core path of the W4A16 linear layer (sm_103a, tcgen05 + TMEM + TMA).
//
// At large M the layer is a dense contraction: once the weights are
// dequantized, what remains is an ordinary fp16 matrix product (the point made
// in the vLLM PR #1032 thread). So the int4 weights are dequantized into
// shared memory and fed to tcgen05.mma kind::f16 with fp32 accumulation in
// tensor memory.
//
// Orientation: D[n][m] = sum_k Wdeq[n][k] * A[m][k] (the weight tile is the
// 128-row MMA operand, the tokens are the MMA's N dimension). Each
// dequantized weight then serves up to 256 tokens, which halves the dequant
// work per FLOP compared with putting the tokens on the 128-row side, and
// token tiles of 16..256 cover the middle band of M as well.
//
// CTA (one output tile: 128 columns x BT tokens, full K):
//   warp 0      TMA producer: activations tile [BT x 64] (128B swizzle) and
//               the packed int4 atoms of 8 strips [8 x 512 B] per k-stage;
//   warp 1      TMEM allocation; one thread issues 4 MMAs (K=16) per stage;
//   warps 2..9  dequantize the packed atoms into the 128B-swizzled K-major
//               operand tile (usually 4 pairs of warps, each pair on every
//               4th stage, so 4 stages are converted concurrently), then run
//               the epilogue (TMEM -> fp16 Y).
// Stages form a ring guarded by mbarriers: full_tma (TMA bytes landed),
// full_dq (the stage's dequant group done), empty (MMAs of the stage
// completed).
// Every wait is bounded; a wait that gives up sets the library's device
// error word and the CTA drains and exits.
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
constexpr int kStageK = 64;        // k per atom of a pipeline stage (one 128-byte swizzle row)
constexpr int kDqWarps = 8;
constexpr int kDqThreads = kDqWarps * 32;
constexpr int kThreads = 64 + kDqThreads;
constexpr int kWdqBytes = kTileN * kStageK * 2;   // 16 KiB dequantized operand
constexpr int kPackedBytes = kTileN * kStageK / 2;  // 4 KiB packed codes
constexpr size_t kTcCounterBytes = 32768;          // tile counters of a K-split launch

using namespace tc;

// ------------------------------------------------------------------ kernel

struct TcParams {
  const uint16_t* Sp;
  const uint32_t* Zp;
  uint16_t* Y;
  int* counters;  // split > 1: one per output tile, zero between calls
  float* tiles;   // split > 1: fp32 partial tiles [tile][split][bt][128]
  int M, N, K, group;
  int bt;         // token tile (MMA N): multiple of 16, 16..256
  int stages;     // pipeline depth
  int tmem_cols;
  int split;      // K ranges per output tile (grid z)
  int dq_groups;  // dequant warp groups (4, 2 or 1), dividing `stages`
  int early_weights;  // weights are static: read the first stages' codes and
                      // scales before the grid-dependency wait
  const float* row_scale;  // W4A8: per-row factors of the result, or null
  int* err;                // the library's error word
};


// named barrier of the 8 dequant/epilogue warps
__device__ __forceinline__ void epilogue_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// SA: atoms (64 k) per pipeline stage, 1 or 2. A stage of two atoms halves
// the barrier hand-offs per weight byte; it needs an even number of atoms
// and groups of at least 128 (one scale and zero point per stage).
template <int SA, bool kB>
__global__ void __launch_bounds__(kThreads, 2)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
               const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const int bt = p.bt, stages = p.stages;
  const uint32_t act_bytes = (uint32_t)bt * 128u;  // one atom of activations
  const uint32_t stage_bytes = SA * (act_bytes + kWdqBytes + kPackedBytes);
  // stage s: [activations of atom 0..SA-1 | dequantized weights of atom
  // 0..SA-1 | packed codes of the SA atoms], each piece 1024-aligned
  const uint32_t wdq_off = SA * act_bytes, packed_off = SA * (act_bytes + kWdqBytes);
  const uint32_t bars = base + (uint32_t)stages * stage_bytes;
  auto full_tma = [&](int s) { return bars + 8u * s; };
  auto full_dq = [&](int s) { return bars + 8u * (stages + s); };
  auto empty = [&](int s) { return bars + 8u * (2 * stages + s); };
  const uint32_t accum_bar = bars + 8u * (3 * stages);
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
    for (int s = 0; s < stages; ++s) {
      mbar_init(full_tma(s), 1);
      mbar_init(full_dq(s), kDqWarps / p.dq_groups);  // one arrival per warp of the group
      mbar_init(empty(s), 1);
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
    if (lane == 0) {
      auto load_codes = [&](int kb, uint32_t st, int s) {
        tma_load_2d(st + packed_off, &tmW, (kb0 + kb) * SA * kAtomWords, n0 / kStripCols,
                    full_tma(s));
      };
      auto load_act = [&](int kb, uint32_t st, int s) {
#pragma unroll
        for (int u = 0; u < SA; ++u)
          tma_load_2d(st + u * act_bytes, &tmA, ((kb0 + kb) * SA + u) * kStageK, m0, full_tma(s));
      };
      // static weights: the first ring's codes go out before the wait for the
      // previous grid (the slots are free: nothing has used them yet)
      const int pre = p.early_weights ? (nk < stages ? nk : stages) : 0;
      for (int kb = 0; kb < pre; ++kb) {
        mbar_expect_tx(full_tma(kb), SA * (act_bytes + kPackedBytes));
        load_codes(kb, base + (uint32_t)kb * stage_bytes, kb);
      }
      grid_dependency_wait();
      for (int kb = 0; kb < pre; ++kb) load_act(kb, base + (uint32_t)kb * stage_bytes, kb);
      int issued = pre;
      for (int kb = pre; kb < nk; ++kb) {
        const int s = kb % stages;
        const uint32_t ph = (uint32_t)(kb / stages) & 1u;
        if (!mbar_wait(empty(s), ph ^ 1u, abort_flag, kErrProducer, p.err)) break;
        const uint32_t st = base + (uint32_t)s * stage_bytes;
        mbar_expect_tx(full_tma(s), SA * (act_bytes + kPackedBytes));
        load_act(kb, st, s);
        load_codes(kb, st, s);
        ++issued;
      }
      if (*abort_flag) {
        // let the copies already issued land before the CTA exits
        for (int kb = (issued > stages ? issued - stages : 0); kb < issued; ++kb)
          mbar_drain(full_tma(kb % stages), (uint32_t)(kb / stages) & 1u, p.err);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = f16_idesc(kTileN, bt, kB);
      bool ok = true;
      int s = 0;
      uint32_t ph = 0;
      // descriptors of stage 0, atom 0; stage s adds s * stage_bytes >> 4,
      // atom u adds u * act_bytes >> 4 (activations) or u * kWdqBytes >> 4
      const uint64_t bdesc0 = sw128_kmajor_desc(base);
      const uint64_t adesc0 = sw128_kmajor_desc(base + wdq_off);
      for (int kb = 0; kb < nk && ok; ++kb) {
        // The dequant group arrives on full_dq only after its own wait on the
        // stage's full_tma phase: acquiring full_dq orders these MMAs after the
        // stage's TMA bytes (activations and codes) as well, so full_tma needs
        // no wait of its own here.
        ok = mbar_wait(full_dq(s), ph, abort_flag, kErrMma, p.err);
        if (!ok) break;
        tc_fence_after();
        const uint64_t soff = (uint64_t)((uint32_t)s * (stage_bytes >> 4));
#pragma unroll
        for (int u = 0; u < SA; ++u)
#pragma unroll
          for (int kk = 0; kk < kStageK / 16; ++kk)  // +32 bytes of k per MMA
            tc_mma_f16(tmem_base, adesc0 + soff + (uint64_t)(u * (kWdqBytes >> 4)) + 2u * kk,
                       bdesc0 + soff + (uint64_t)(u * (act_bytes >> 4)) + 2u * kk, idesc,
                       (kb | u | kk) != 0);
        tc_commit(empty(s));
        if (++s == stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      tc_commit(accum_bar);  // fires once every MMA issued above has completed
      if (!ok) mbar_drain(accum_bar, 0, p.err);  // no MMA may run past the TMEM release
    }
  } else {
    // ---------------------------------------------------------- dequant + epilogue
    // The 8 warps form `groups` groups (4, 2 or 1); group g dequantizes the
    // stages kb = g, g + groups, ... so several stages are converted at once;
    // within a stage each of the group's warps converts `groups` strips.
    // `stages` is a multiple of `groups`, so a ring slot is always converted
    // by the same group, which has waited for the slot's previous round: a
    // parity wait can then never run more than one phase ahead of its
    // barrier (where it would take an older phase for the awaited one).
    const int groups = p.dq_groups;
    const int wpg = kDqWarps / groups;  // warps per group
    const int dw = warp - 2;
    const int dg = dw / wpg, sub = dw % wpg;
    const int gq = lane >> 2, t = lane & 3;
    const int nstrips = p.N / kStripCols;
    const int G = p.K / p.group;
    const uint32_t* sp2 = reinterpret_cast<const uint32_t*>(p.Sp);
    const uint8_t* zpb = reinterpret_cast<const uint8_t*>(p.Zp);
    // process the lane's words in an order that keeps the 16-byte stores of
    // each quarter-warp on distinct banks (odd rows take the other k-half first)
    const uint32_t flip = (uint32_t)(gq & 1);
    // (s[gq], s[gq+8]) and zero-point pairs of this warp's strips for a stage
    auto load_meta = [&](int kb, uint32_t (&ms)[4], uint32_t (&mz)[4]) {
      const int grp = (int)((long long)(kb0 + kb) * SA * kStageK / p.group);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int strip = n0 / kStripCols + groups * sub + i;
        ms[i] = 0;
        mz[i] = 0;
        if (i < groups && strip < nstrips) {
          const size_t off = ((size_t)strip * G + grp) * 8 + gq;
          ms[i] = sp2[off];
          mz[i] = zpb[off];
        }
      }
    };
    // one stage of this group: wait for its copies, dequantize this warp's
    // strips with the stage's scales and zero points (ms, mz), arrive
    auto stage = [&](int kb, const uint32_t (&ms)[4], const uint32_t (&mz)[4]) -> bool {
      const int s = kb % stages;
      const uint32_t ph = (uint32_t)(kb / stages) & 1u;
      if (!mbar_wait(full_tma(s), ph, abort_flag, kErrDequant, p.err)) return false;
      const uint32_t st = base + (uint32_t)s * stage_bytes;
      // the next strip's codes are loaded while this strip is converted (the
      // loop is unrolled: no register copies)
      uint4 v[2][SA];
      auto load_codes = [&](int i, uint4 (&d)[SA]) {
#pragma unroll
        for (int u = 0; u < SA; ++u)
          d[u] = lds128(st + packed_off + (groups * sub + i) * (SA * 512) + u * 512 + lane * 16);
      };
      load_codes(0, v[0]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (i + 1 < 4 && i + 1 < groups) load_codes(i + 1, v[(i + 1) & 1]);
        const int ls = groups * sub + i;  // strip within the tile
        if (i < groups && n0 / kStripCols + ls < nstrips) {
          const uint32_t z0 = mz[i] & 15u, z1 = (mz[i] >> 4) & 15u;
          const uint16_t s0 = (uint16_t)(ms[i] & 0xffffu), s1 = (uint16_t)(ms[i] >> 16);
#pragma unroll
          for (int u = 0; u < SA; ++u) {
            const uint32_t wdq = st + wdq_off + u * kWdqBytes;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t ks = (uint32_t)(j >> 1) ^ flip;  // k-half of this word
              const uint32_t r = (uint32_t)(j & 1);           // column gq or gq + 8
              const uint4 vv = v[i & 1][u];
              const uint32_t word = ks ? (r ? vv.w : vv.z) : (r ? vv.y : vv.x);
              uint32_t o[4];
              if (kB)
                dequant_word_bf16(word, make_deq_const_bf16(r ? z1 : z0, r ? s1 : s0), o);
              else
                dequant_word(word, make_deq_const(r ? z1 : z0, r ? s1 : s0), o);
              // row n = 16 ls + gq + 8 r of the operand, 16-byte chunk kw = 4 ks + t
              const uint32_t row = 16u * ls + gq + 8u * r;
              const uint32_t kw = 4u * ks + t;
              sts128(wdq + (row >> 3) * 1024u + (row & 7u) * 128u + ((kw ^ (row & 7u)) << 4),
                     o[0], o[1], o[2], o[3]);
            }
          }
        }
      }
      fence_async_shared();  // this thread's generic-proxy stores -> visible to the tensor core
      __syncwarp();          // every lane of the warp has fenced its stores
      if (lane == 0) mbar_arrive(full_dq(s));
      return true;
    };
    // two register sets of scales and zero points, alternating between this
    // group's stages: each set is loaded one stage ahead and read only by its
    // own stage, so no stage waits for the next stage's loads. Scales and
    // zero points are weights: with static weights the first set is read
    // before the wait for the previous grid (which orders this warp's stores
    // of Y)
    uint32_t ma[4], za[4], mb[4], zb[4];
    if (p.early_weights && dg < nk) load_meta(dg, ma, za);
    grid_dependency_wait();
    if (!p.early_weights && dg < nk) load_meta(dg, ma, za);
    for (int kb = dg; kb < nk; kb += 2 * groups) {
      if (kb + groups < nk) load_meta(kb + groups, mb, zb);
      if (!stage(kb, ma, za) || kb + groups >= nk) break;
      if (kb + 2 * groups < nk) load_meta(kb + 2 * groups, ma, za);
      if (!stage(kb + groups, mb, zb)) break;
    }

    // epilogue: TMEM lanes 32q..32q+31 are output columns, TMEM columns are tokens
    const bool have_accum = mbar_wait(accum_bar, 0, abort_flag, kErrEpilogue, p.err);
    __syncwarp();
    if (__all_sync(0xffffffffu, have_accum)) {  // warp-uniform: tcgen05.ld is .aligned
      tc_fence_after();
      const int q = warp & 3;
      const int half = dw >> 2;  // two warpgroups split the token chunks
      const int n = n0 + 32 * q + lane;
      float* part = p.tiles + (((size_t)blockIdx.y * gridDim.x + blockIdx.x) * p.split + blockIdx.z) *
                                  (size_t)bt * kTileN;
      for (int c = half; c < bt / 16; c += 2) {
        uint32_t r[16];
        tmem_ld16(tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(16 * c), r);
        tmem_wait_ld();
        if (p.split > 1) {  // fp32 partial tile [token][column]
#pragma unroll
          for (int j = 0; j < 16; ++j) part[(16 * c + j) * kTileN + 32 * q + lane] = __uint_as_float(r[j]);
        } else if (n < p.N) {
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
    if (p.split > 1) {
      // K split: the last of the tile's CTAs to arrive sums the partial tiles in
      // split order (deterministic), writes Y and resets the tile's counter
      const int tile = blockIdx.y * gridDim.x + blockIdx.x;
      epilogue_bar();  // every partial store issued; one release atomic covers them
      if (dw == 0 && lane == 0) {
        int old = 0;
        if (*abort_flag == 0)
          asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                       : "=r"(old)
                       : "l"(p.counters + tile)
                       : "memory");
        *last_flag = (*abort_flag == 0) && old == p.split - 1;
      }
      epilogue_bar();
      if (*last_flag) {
        // 4 columns per float4, 8 float4 per thread and round: the loads of
        // one partial tile for the round are all in flight together, and the
        // partial tiles are added in split order
        const float4* tb = reinterpret_cast<const float4*>(p.tiles + (size_t)tile * p.split * bt * kTileN);
        const int n4 = bt * kTileN / 4;
        constexpr int kRound = 8;
        for (int e0 = dw * 32 + lane; e0 < n4; e0 += kRound * kDqThreads) {
          float4 acc[kRound];
#pragma unroll
          for (int u = 0; u < kRound; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int z = 0; z < p.split; ++z) {
            float4 v[kRound];
#pragma unroll
            for (int u = 0; u < kRound; ++u) {
              const int e = e0 + u * kDqThreads;
              v[u] = e < n4 ? __ldcg(tb + (size_t)z * (n4) + e) : make_float4(0.f, 0.f, 0.f, 0.f);
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
            const int e = e0 + u * kDqThreads;
            const int tok = m0 + e / (kTileN / 4), n = n0 + (e % (kTileN / 4)) * 4;
            if (e < n4 && tok < p.M && n < p.N) {
              const float f = p.row_scale ? p.row_scale[tok] : 1.0f;
              uint2 o;
              o.x = to_out2<kB>(acc[u].x * f, acc[u].y * f);
              o.y = to_out2<kB>(acc[u].z * f, acc[u].w * f);
              *reinterpret_cast<uint2*>(p.Y + (size_t)tok * p.N + n) = o;
            }
          }
        }
        if (dw == 0 && lane == 0) p.counters[tile] = 0;
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

int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

}  // namespace

int tc_token_tile(int M) {
  if (M >= 256) return 256;
  return (M + 15) / 16 * 16;
}

// CTAs per SM the tensor-core kernel is sized for: two when the token tile is
// at most 48 (four stages still fit in half the shared memory; more CTAs for
// the small tile counts of the middle band of M), else one with the deepest
// pipeline that fits.
int tc_ctas_per_sm(int bt) { return bt <= 48 ? 2 : 1; }

size_t tc_smem_bytes(int bt, int sa, int* stages_out) {
  const size_t stage = (size_t)sa * ((size_t)bt * 128 + kWdqBytes + kPackedBytes);
  const size_t budget = (tc_ctas_per_sm(bt) == 2 ? 113 * 1024 : 227 * 1024) - 1024 - 256;
  int stages = (int)(budget / stage);
  if (stages > 8) stages = 8;
  if (stages >= 4) stages &= ~3;  // a multiple of the 4 dequant groups
  else if (stages == 3) stages = 2;  // of 2 groups
  if (stages_out) *stages_out = stages;
  return (size_t)stages * stage + 1024 + 256;
}

// Two-atom stages halve the hand-offs per weight byte but need a ring of at
// least 4 of them to pay: measured, 64-token tiles (4 stages) gained 15-22%
// and 128- or 256-token tiles (2 stages) lost 5-10%.
int tc_stage_atoms(int M, int K, int group) {
  if (K % 128 != 0 || group % 128 != 0) return 1;
  int stages = 0;
  tc_smem_bytes(tc_token_tile(M), 2, &stages);
  return stages >= 4 ? 2 : 1;
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

template <int SA, bool kB>
cudaError_t launch_kernel(const CUtensorMap& tmA, const CUtensorMap& tmW, const TcParams& prm,
                          dim3 grid, size_t smem, cudaStream_t stream) {
  cudaError_t e = set_max_smem_once(reinterpret_cast<const void*>(tc_gemm_kernel<SA, kB>), 227 * 1024);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<SA, kB>, tmA, tmW, prm);
}

}  // namespace

// Encoded tensor maps of recent calls, keyed by what they encode: encoding
// one costs a driver call, and a layer calls with the same pointers and
// shapes every step. A small table per process, replaced round-robin.
namespace {

struct MapKey {
  const void* ptr;
  uint64_t dims0, dims1;
  uint32_t box0, box1;
  int dtype;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && dims0 == o.dims0 && dims1 == o.dims1 && box0 == o.box0 &&
           box1 == o.box1 && dtype == o.dtype;
  }
};
constexpr int kMapCache = 64;
std::mutex g_map_mutex;
MapKey g_map_keys[kMapCache];
CUtensorMap g_maps[kMapCache];
int g_map_used = 0, g_map_next = 0;

}  // namespace

bool cached_tensor_map(CUtensorMap* out, const void* ptr, CUtensorMapDataType dt, int esize,
                       uint64_t dims0, uint64_t dims1, uint32_t box0, uint32_t box1,
                       CUtensorMapSwizzle swizzle) {
  const MapKey key = {ptr, dims0, dims1, box0, box1, (int)dt};
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
  const cuuint64_t dims[2] = {(cuuint64_t)dims0, (cuuint64_t)dims1};
  const cuuint64_t strides[1] = {(cuuint64_t)dims0 * esize};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(out, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lock(g_map_mutex);
  const int slot = g_map_used < kMapCache ? g_map_used++ : (g_map_next++ % kMapCache);
  g_map_keys[slot] = key;
  g_maps[slot] = *out;
  return true;
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
  // packed weights viewed as [N/16 strips][K/64 atoms * 128 words] of uint32
  if (!cached_tensor_map(&tmW, Wq, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, (uint64_t)(K / kAtomK) * kAtomWords,
                  (uint64_t)(N / kStripCols), (uint32_t)(kAtomWords * sa), kTileN / kStripCols,
                  CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
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
  const size_t smem = tc_smem_bytes(bt, sa, &prm.stages);
  prm.tmem_cols = pow2_at_least(bt);
  prm.dq_groups = prm.stages % 4 == 0 ? 4 : (prm.stages % 2 == 0 ? 2 : 1);
  const dim3 grid((unsigned)((M + bt - 1) / bt), (unsigned)((N + kTileN - 1) / kTileN),
                  (unsigned)prm.split);
  if (bf16)
    return sa == 2 ? launch_kernel<2, true>(tmA, tmW, prm, grid, smem, stream)
                   : launch_kernel<1, true>(tmA, tmW, prm, grid, smem, stream);
  return sa == 2 ? launch_kernel<2, false>(tmA, tmW, prm, grid, smem, stream)
                 : launch_kernel<1, false>(tmA, tmW, prm, grid, smem, stream);
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
