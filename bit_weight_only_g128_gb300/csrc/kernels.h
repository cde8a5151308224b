// Launchers of the W4A16 kernels (host side). Arguments are validated by the
// C ABI layer (api.cu) before any of these is called. Activations and
// results are 16-bit floats: fp16, or bf16 where a launcher takes `bf16`.
// GEMM launchers take `row_scale`: per-row factors applied to the fp32
// result before its rounding (W4A8: the activations' scales), or null.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace w4a16 {

cudaError_t launch_quantize(const float* W, int K, int N, int group, uint8_t* q, uint16_t* s,
                            uint8_t* z, cudaStream_t stream);
cudaError_t launch_pack(const uint8_t* q, const uint16_t* s, const uint8_t* z, int K, int N,
                        int group, uint32_t* Wq, uint16_t* Sp, uint32_t* Zp, cudaStream_t stream);
cudaError_t launch_unpack(const uint32_t* Wq, const uint16_t* Sp, const uint32_t* Zp, int K,
                          int N, int group, uint8_t* q, uint16_t* s, uint8_t* z,
                          cudaStream_t stream);
// deq = RNE((q - z) * s) in fp16, or in bf16 with `bf16`.
cudaError_t launch_dequantize(const uint32_t* Wq, const uint16_t* Sp, const uint32_t* Zp, int K,
                              int N, int group, uint16_t* deq, bool bf16, cudaStream_t stream);

// Stream-K register-dequant GEMV for M <= 16 rows of A (one launch of `ctas`
// persistent CTAs, 1 <= ctas <= min(decode_units, kDecodeMaxCtas)).
// `workspace` holds the per-CTA flags (zero before the first call, left zero
// by every call) followed by the partial tiles; see decode_workspace_bytes.
// With early_weights the first weights are read before the grid-dependency
// wait.
cudaError_t launch_decode(const uint16_t* A, const uint32_t* Wq, const uint16_t* Sp,
                          const uint32_t* Zp, uint16_t* Y, int M, int N, int K, int group,
                          int ctas, void* workspace, bool early_weights, bool bf16,
                          const float* row_scale, cudaStream_t stream);
size_t decode_workspace_bytes(int M, int N, int ctas);

// Register-dequant GEMV with the activations resident in shared memory, for
// M <= 16 rows: `ctas` CTAs (as decode_resident_ctas returned for the same
// `sms`, `automatic` and `silu`) each own whole 16-column strips over all of
// K; no workspace. With `silu` the N columns are [gate | up], each CTA owns
// pairs of strips (q, N/32 + q), and Y is M x N/2 = silu(gate) * up.
cudaError_t launch_decode_resident(const uint16_t* A, const uint32_t* Wq, const uint16_t* Sp,
                                   const uint32_t* Zp, uint16_t* Y, int M, int N, int K, int group,
                                   int ctas, int sms, bool automatic, bool silu,
                                   bool early_weights, bool bf16, const float* row_scale,
                                   cudaStream_t stream);
// CTAs of that kernel (`requested`, else one per resident slot of `sms` SMs:
// two 8-warp CTAs or one 16-warp CTA per SM; clamped to the strips and to
// 8192), or 0 when the problem's activations, sums and group pairs do not fit
// a CTA's shared memory at that count (with `automatic`, also when the
// staged activations exceed 160 KiB) or the group is unsupported.
int decode_resident_ctas(int M, int N, int K, int group, int requested, int sms, bool automatic,
                         bool silu);
// Y [M][N/2] = silu(Yfull[:, :N/2]) * Yfull[:, N/2:] for a 16-bit product
// Yfull [M][N] (row stride N): the fused gate/up epilogue as a separate pass.
cudaError_t launch_silu_mul(const uint16_t* Yfull, int M, int N, uint16_t* Y, bool bf16,
                            cudaStream_t stream);
// W4A8: per row, s_a = max|a| / 127 (1 for a zero row) and the codes
// clamp(round(a / s_a), -127, 127), IEEE fp32. A [M][K] is fp16 (bf16 with
// in_bf16); K a multiple of 8 and A 16-byte aligned. Writes the codes as int8
// to aq and/or as 16-bit integer values (bf16 with codes_bf16) to `codes`,
// either may be null; s_a [M].
cudaError_t launch_quantize_act(const uint16_t* A, int M, int K, bool in_bf16, int8_t* aq,
                                uint16_t* codes, bool codes_bf16, float* s_a, cudaStream_t stream);
// Bytes of the counter area at the start of the decode workspace.
size_t decode_counter_bytes(int N);
// Split granules (128 columns x a group's atoms, at most 8) of a problem: the
// most CTAs a decode launch can use; 0 if the group size is not supported.
long decode_units(int N, int K, int group);
// CTAs of the decode kernel for M rows that fit on one SM (occupancy query).
int decode_ctas_per_sm(int M);

// tcgen05/TMEM tensor-core GEMM: one CTA per 128 output columns x token tile
// x K range (`split` ranges; with split > 1 the workspace holds the tile
// counters, zero between calls, and the fp32 partial tiles).
// With early_weights (static weights) the first stages' codes, scales and
// zero points are read before the wait for the previous grid.
cudaError_t launch_tc_gemm(const uint16_t* A, const uint32_t* Wq, const uint16_t* Sp,
                           const uint32_t* Zp, uint16_t* Y, int M, int N, int K, int group,
                           int split, void* workspace, bool early_weights, bool bf16,
                           const float* row_scale, cudaStream_t stream);
size_t tc_workspace_bytes(int M, int N, int split);
// Two-SM tensor-core GEMM for large M: persistent clusters of two CTAs (as
// many as are resident at once), each pair taking output tiles of 256
// columns x tc_pair_token_tile(M) tokens over all of K in turn, the rings
// running on across tiles (tcgen05.mma.cta_group::2); no workspace.
cudaError_t launch_tc_pair(const uint16_t* A, const uint32_t* Wq, const uint16_t* Sp,
                           const uint32_t* Zp, uint16_t* Y, int M, int N, int K, int group,
                           bool early_weights, bool bf16, const float* row_scale,
                           cudaStream_t stream);
int tc_pair_token_tile(int M);
int tc_pair_stage_atoms(int K, int group);
// The CTA-pair kernel's configuration for M rows (w4a16_tc_config's
// out[8..14]); false if its rings would break the kernel's barrier invariants.
bool tc_pair_config(int M, int K, int group, int out[7]);
// 2-D tensor map of a row-major [dims1][dims0] array of `esize`-byte elements
// with box [box1][box0], from a per-process cache keyed by pointer, shape,
// box and type (encoding one costs a driver call); false if it cannot be
// encoded.
bool cached_tensor_map(CUtensorMap* out, const void* ptr, CUtensorMapDataType dt, int esize,
                       uint64_t dims0, uint64_t dims1, uint32_t box0, uint32_t box1,
                       CUtensorMapSwizzle swizzle);
// 3-D tensor map of the packed weights as [N/16 strips][K/64 atoms x 4 rows]
// [32 words] with the 128-byte swizzle; a box is `sa` atoms of 8 strips (128
// columns). From the same cache.
bool cached_code_map(CUtensorMap* out, const uint32_t* Wq, int N, int K, int sa);
int tc_choose_split(int M, int N, int K, int group, int sms);
// 64-k atoms per pipeline stage of the tensor-core GEMM (2 when K and the
// group are multiples of 128, else 1).
int tc_stage_atoms(int M, int K, int group);
// Token tile (MMA N) used for M rows.
int tc_token_tile(int M);
// The one-SM kernel's configuration for M rows (w4a16_tc_config's out[0..7]);
// false if its rings would break the kernel's barrier invariants.
bool tc_config(int M, int K, int group, int out[8]);

// Self-tests of the bounded waits (a flag wait of the stream-K decode
// kernel's kind, an mbarrier wait of the tensor-core pipeline's kind): each
// waits about a second for something that never happens, then records its
// error bit and returns.
cudaError_t launch_selftest_flag_wait(cudaStream_t stream);
cudaError_t launch_selftest_mbar_wait(cudaStream_t stream);

// Reads the device error word (bounded waits that gave up, self-checks) and
// clears it if set.
cudaError_t read_and_clear_device_error(int* flag);

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device): the attribute is per device, and setting
// it on every launch costs a driver call.
cudaError_t set_max_smem_once(const void* kernel, int bytes);

// Set (or clear) the calling thread's w4a16_last_error message; returns code.
int report_error(int code, const char* message);
int report_ok();

// Output columns per decode CTA.
constexpr int kDecodeBlockCols = 128;
// Most CTAs of one decode launch (the size of its flag area).
constexpr int kDecodeMaxCtas = 8192;

// Device address of the library's error word (bits set by kernels whose
// bounded waits ran out), for kernels that take it as an argument.
cudaError_t device_error_word(int** ptr);

}  // namespace w4a16
