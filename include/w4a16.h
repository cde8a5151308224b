/*
 * w4a16.h - C ABI of the GB300 (sm_103a) W4A16 group-quantized linear layer.
 *
 * The operation (compressed-tensors PR #269 "Some fixes for AWQ", the reply
 * defining w4a16): fp16 activations are multiplied by int4-quantized weights
 * to give fp16 outputs. Weights are quantized asymmetrically per group of
 * `group` consecutive input channels (128 in the "w4-g128" / "AWQ-g128"
 * checkpoints of vLLM PR #1032 "Implement AWQ quantization support for LLaMA"
 * and the lmdeploy issue #2274 tables; group == K is the per-channel variant)
 * with the rule that PR #269 aligns with AutoAWQ's pseudo_quantize_tensor:
 *     s = (max - min)/15,  z = round(-min/s),  q = clamp(round(w/s) + z, 0, 15),
 * and are dequantized inside the kernels as (q - z)*s, rounded once to fp16.
 * Products accumulate in fp32; Y is rounded to fp16 (ties to even).
 * Variants, chosen per call by flags of w4a16_gemm_ex (below): bf16
 * activations and results (W4A16_BF16), the fused gate/up epilogue
 * silu(gate)*up (W4A16_SILU_MUL), and W4A8, the activations quantized to
 * 8 bits inside the call (W4A16_ACT_A8). All use the same packed weights.
 *
 * Conventions for every entry point:
 *   - Every pointer argument is a DEVICE pointer on the current CUDA device,
 *     owned by the caller. The library never allocates, frees or keeps device
 *     memory (apart from its static device arrays: a 4-byte error word, and
 *     the scratch of w4a16_gemm_noalloc), and never synchronizes (apart from
 *     w4a16_device_status): work is enqueued on `stream` (a cudaStream_t
 *     passed as void*; NULL is the legacy default stream), which must belong
 *     to the current device.
 *   - The library keeps per-device state for the life of the process (the
 *     error word's address, kernel attributes, encoded tensor maps keyed by
 *     pointer and shape): make no call after a reset of the device
 *     (cudaDeviceReset) in the same process.
 *   - fp16 values are passed as uint16_t bit patterns (IEEE binary16).
 *   - Return value: W4A16_OK (0) or a negative W4A16_ERR_* code. On error no
 *     kernel has been launched (except W4A16_ERR_CUDA, which reports a failed
 *     launch), and w4a16_last_error() returns a message for the calling
 *     thread. No C++ exception crosses this interface.
 *   - Shapes: N % 16 == 0, K % 64 == 0, group % 64 == 0 and K % group == 0;
 *     M >= 0 (M == 0 is a no-op). Other shapes return
 *     W4A16_ERR_UNSUPPORTED_SHAPE. 1 <= N, K <= 1<<20 and M <= 1<<20.
 *
 * Interchange (logical) layouts, as in the transposed AWQ format quoted in
 * vLLM PR #1032 (the Triton variant: qw (K/pack, N), scales (K/group, N),
 * qzeros (K/group/pack, N)), unpacked to one byte per code here:
 *     q     uint8  [K][N]   codes 0..15 (row k, column n)
 *     s     fp16   [G][N]   scales, G = K / group
 *     z     uint8  [G][N]   zero points 0..15
 *     A     fp16   [M][K]   activations, row-major
 *     Y     fp16   [M][N]   outputs, row-major
 *
 * Packed device layout (this library's own format; built by w4a16_pack):
 *   Wq: uint32 words, K*N/8 of them, 8 codes per word. Columns form strips
 *     of 16 (strip j = columns 16j..16j+15); K forms atoms of 64 (atom a =
 *     k in [64a, 64a+64)). The word at offset (j*(K/64) + a)*128 + 4*L + i,
 *     L in [0,32), i in [0,4), with g = L>>2, t = L&3, s = i>>1, r = i&1,
 *     holds column n = 16j + g + 8r at k = 64a + 32s + 8t + e, e = 0..7;
 *     code e sits in nibble p (bits 4p..4p+3), p = the 3-bit reversal of e
 *     (e = 4 e2 + 2 e1 + e0 -> p = 4 e0 + 2 e1 + e2: nibbles 0..7 hold
 *     k-offsets 0 4 2 6 1 5 3 7). So (word >> 4p) & 0x000F000F holds the
 *     codes of k-offsets (0,1), (4,5), (2,3), (6,7) for p = 0, 1, 2, 3 in its
 *     two 16-bit halves, and each lane L of a warp reads its four words of an
 *     atom with one 16-byte load.
 *   Sp: fp16, N*G of them; offset (j*G + grp)*16 + 2c + h is the scale of
 *     column 16j + 8h + c (c in [0,8), h in {0,1}) in group grp, so the two
 *     columns g and g + 8 that one lane dequantizes share one 32-bit word.
 *   Zp: bytes, N*G/2 of them (addressed as uint32 words); byte
 *     (j*G + grp)*8 + c holds the zero point of column 16j + c in its low
 *     nibble and that of column 16j + 8 + c in its high nibble (c in [0,8)),
 *     again the two columns one lane dequantizes.
 *   Sizes: w4a16_packed_sizes(). Alignment: Wq, Sp, A and Y 16-byte aligned,
 *   Zp 8-byte aligned (W4A16_ERR_MISALIGNED otherwise).
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define W4A16_OK 0
#define W4A16_ERR_INVALID_ARG (-1)         /* null pointer, negative size  */
#define W4A16_ERR_UNSUPPORTED_SHAPE (-2)   /* shape rules above violated   */
#define W4A16_ERR_MISALIGNED (-3)          /* pointer alignment violated   */
#define W4A16_ERR_WORKSPACE_TOO_SMALL (-4) /* workspace below the size query */
#define W4A16_ERR_CUDA (-5)                /* CUDA runtime/launch failure  */
#define W4A16_ERR_DEVICE_CHECK (-6)        /* a kernel reported an error   */

/* Paths for w4a16_gemm_ex. */
#define W4A16_PATH_AUTO 0
#define W4A16_PATH_DECODE 1   /* register-dequant GEMV, variant below chosen
                                 per launch: resident when it fits    */
#define W4A16_PATH_TENSOR 2   /* tcgen05/TMEM tensor-core GEMM          */
/* The two variants of the decode GEMV, forced. RESIDENT: each CTA owns whole
 * 16-column strips over all of K and keeps the launch's activation rows in
 * shared memory (two 8-warp CTAs per SM, or one 16-warp CTA for larger rows);
 * it needs no workspace, and shapes whose rows (16 rows per launch at most)
 * do not fit give W4A16_ERR_UNSUPPORTED_SHAPE (about (M+1)*K <= 110 Ki
 * elements: K = 4096 up to 16 rows, K = 11008 up to 8). W4A16_PATH_DECODE
 * takes it up to 160 KiB of staged rows, and beyond that only when the
 * strips spread over the CTAs at least 90% evenly. STREAMK: the
 * weights of 128-column blocks are split across CTAs in equal runs of
 * groups, the activations are streamed through shared memory with them, and
 * blocks split between CTAs are combined through the workspace; any shape
 * the decode path takes. */
#define W4A16_PATH_DECODE_RESIDENT 3
#define W4A16_PATH_DECODE_STREAMK 4
/* The tensor-core GEMM on pairs of SMs (tcgen05.mma.cta_group::2): clusters
 * of two CTAs, as many as are resident at once, each taking output tiles of
 * 256 columns x 256 tokens (128 when M <= 128) over all of K in turn; each
 * CTA dequantizes its 128 columns into its tensor memory (the MMA's A
 * operand) and stages half of the tokens, and the pair's MMAs read both
 * halves. The same
 * arithmetic as W4A16_PATH_TENSOR (RNE_fp16((q - z) s) operands, fp32
 * accumulation); no K split and no workspace of its own. */
#define W4A16_PATH_TENSOR_PAIR 5
/* Flag OR-ed into the path of w4a16_gemm_ex: the weights (Wq, scales, zeros)
 * are not written by the work queued just before this call on the stream, so
 * the kernel may read them while that work drains. The GEMM kernels (both
 * decode variants and the tensor-core GEMM) and the fused epilogue's
 * separate pass are launched with programmatic stream serialization: a grid
 * may be scheduled while the previous one drains, and touches A, Y and the
 * workspace only after the previous grid has completed. (The W4A8
 * activation-quantization kernel is a plain launch.) With this flag the
 * decode kernels also load their first weights before that point, and the
 * tensor-core kernel its first ring of packed codes and its first scales and
 * zero points, which hides the gap between back-to-back layers. Without it
 * every read of the weights also waits for the previous grid. */
#define W4A16_STATIC_WEIGHTS 0x100
/* Flag OR-ed into the path of w4a16_gemm_ex and w4a16_workspace_size_ex: the
 * fused gate/up epilogue of a gated MLP (lmdeploy issue #2274 "[Feature]
 * support qqq(w4a8) for lmdeploy", section "Modification": the gate and up
 * projections fused into one weight, SiLU fused into the GEMM). The N
 * columns of the weight are [gate | up], two halves of N/2 (N a multiple of
 * 32, else W4A16_ERR_UNSUPPORTED_SHAPE), and the output is
 * Y [M][N/2] = silu(A.W[:, :N/2]) * (A.W[:, N/2:]), silu(g) = g/(1+exp(-g)),
 * formed in fp32 and rounded to fp16 once. The resident decode variant
 * forms it from the fp32 accumulators inside the GEMM kernel (each CTA owns
 * both strips of its column pairs; no workspace). The stream-K variant and
 * the tensor-core path write the fp16 product [rows][N] to the workspace
 * (after their own scratch and at least after its 32 KiB flag/counter area,
 * at a 256-byte boundary; 16 rows per decode launch, all M rows for tensor
 * cores) and a second kernel forms Y from it;
 * w4a16_workspace_size_ex with this flag counts those bytes. */
#define W4A16_SILU_MUL 0x200
/* Flag OR-ed into the path of w4a16_gemm_ex (and accepted, with no effect on
 * the sizes, by w4a16_workspace_size_ex): A and Y hold bfloat16 instead of
 * fp16 (compressed-tensors PR #269 "Some fixes for AWQ": W4A16 keeps the
 * activations as unquantized 16-bit floats, and a reply names an API taking
 * fp32, bf16 or fp16 activations). The quantized weights are the same
 * buffers (fp16 scales). The tensor-core path multiplies bf16 activations by
 * RNE_bf16((q - z) * s) (w4a16_dequantize_bf16 gives the same values); the
 * decode path takes the codes exactly and applies s and z per group in fp32;
 * both accumulate in fp32 and round the result once to bf16. Accuracy
 * contract: |y - y_ref| <= 2^-6 * sum_k |a_k w_kn| + 1e-3 against the fp64
 * product of the same bf16 activations and bf16-dequantized weights (four
 * units of bf16 rounding, as the fp16 bound is four of fp16). Combines with
 * the other flags; w4a16_gemm_noalloc has no bf16 form. */
#define W4A16_BF16 0x400
/* Flag OR-ed into the path of w4a16_gemm_ex and w4a16_workspace_size_ex:
 * W4A8. The 16-bit activations A are quantized to 8 bits inside the call
 * and the product is 8-bit activations by 4-bit weights (compressed-tensors
 * PR #269, the Arm example: fp16 in, 8-bit activations inside the
 * operation, fp16 out; lmdeploy issue #2274: W4A8 with online activation
 * quantization). Per row m, in IEEE fp32: s_a = max_k |a| / 127 (1 for a row
 * of zeros) and a_q = clamp(round(a / s_a), -127, 127), ties to even (what
 * w4a16_quantize_act writes). Then y = s_a * sum_k a_q (q - z) s, with s_a
 * scaling the fp32 result before its one rounding; the codes enter the
 * tensor cores as exact 16-bit integer values. On the decode path each
 * integer product a_q (q - z) and each group's sum is exact in fp32 and the
 * group's sum is multiplied by s; on the tensor-core path the codes multiply
 * the same dequantized operand RNE_fp16((q - z) s) (RNE_bf16 with
 * W4A16_BF16) that 16-bit activations use, so each product carries that
 * weight's one rounding. The workspace holds the
 * codes ([M][K], 16-bit) and the scales after the path's own scratch (and
 * after the fused epilogue's product), so w4a16_workspace_size_ex must be
 * asked with the same flags. Accuracy contract: the 16-bit bound of the
 * result's type with sum |a w| read as s_a * sum |a_q (q - z) s|. Combines
 * with the other flags. */
#define W4A16_ACT_A8 0x800

/* Message for the last error returned on the calling thread ("" if none). */
const char* w4a16_last_error(void);

/* Library version, as MAJOR*10000 + MINOR*100 + PATCH. */
int w4a16_version(void);

/* Byte sizes of the packed buffers for a K x N weight with group `group`:
 * Wq = K*N/2, Sp = 2*N*(K/group), Zp = N*(K/group)/2. Host-only. */
int w4a16_packed_sizes(int K, int N, int group,
                       size_t* wq_bytes, size_t* sp_bytes, size_t* zp_bytes);

/* Offline step: quantize fp32 W [K][N] per group along K with the rule
 * above (R-eps: a scale that rounds to zero in fp16 is replaced by
 * RNE_fp16(1e-5)). q/z must use the stored fp16 scale, all divisions and
 * roundings are IEEE fp32 round-to-nearest-even. W must be finite.
 * Outputs: q [K][N], s [G][N] (fp16 bits), z [G][N]. */
int w4a16_quantize(const float* W, int K, int N, int group,
                   uint8_t* q, uint16_t* s, uint8_t* z, void* stream);

/* Offline step: interchange (q, s, z) -> packed (Wq, Sp, Zp), layout above.
 * Codes and zero points above 15 keep only their low 4 bits. */
int w4a16_pack(const uint8_t* q, const uint16_t* s, const uint8_t* z,
               int K, int N, int group,
               uint32_t* Wq, uint16_t* Sp, uint32_t* Zp, void* stream);

/* Inverse of w4a16_pack (for checks and debugging). */
int w4a16_unpack(const uint32_t* Wq, const uint16_t* Sp, const uint32_t* Zp,
                 int K, int N, int group,
                 uint8_t* q, uint16_t* s, uint8_t* z, void* stream);

/* deq [K][N] fp16 = RNE_fp16((q - z)*s) computed from the packed buffers
 * with the same device routine the GEMM kernels use (for checks). */
int w4a16_dequantize(const uint32_t* Wq, const uint16_t* Sp, const uint32_t* Zp,
                     int K, int N, int group, uint16_t* deq, void* stream);

/* W4A8 activation quantization (the rule under W4A16_ACT_A8): A [M][K]
 * 16-bit (fp16, or bf16 with flags = W4A16_BF16) -> aq [M][K] int8 and s_a
 * [M] fp32. K a multiple of 8, at most 65536 (the same limit applies to
 * W4A16_ACT_A8); A and aq 16-byte aligned. */
int w4a16_quantize_act(const uint16_t* A, int M, int K, int flags, int8_t* aq, float* s_a,
                       void* stream);

/* As w4a16_dequantize with deq in bfloat16: RNE_bf16((q - z)*s), the
 * operand the tensor-core path builds for bf16 activations (W4A16_BF16). */
int w4a16_dequantize_bf16(const uint32_t* Wq, const uint16_t* Sp, const uint32_t* Zp,
                          int K, int N, int group, uint16_t* deq, void* stream);

/* Scratch bytes w4a16_gemm needs for this problem on the current device
 * (0 when none). Work split across CTAs is combined through it: the decode
 * path's stream-K variant (M <= 16 rows per launch) shares 128-column blocks
 * between CTAs, and the tensor-core path splits K when its output tiles
 * cannot fill the SMs. For W4A16_PATH_DECODE the size is that of the
 * stream-K variant whichever variant the device then runs.
 * Layout: a 32 KiB flag/counter area followed by fp32 partial tiles. That
 * area must be zero-filled before the first use; every call leaves it
 * zero-filled again, so one buffer serves any number of calls, of any shape
 * that fits, that run one after another. Calls that may run concurrently
 * (other streams) need separate workspaces. After W4A16_ERR_DEVICE_CHECK,
 * zero it again. Host-only. */
int w4a16_workspace_size(int M, int N, int K, int group, size_t* bytes);

/* As w4a16_workspace_size for a forced path and work partition (see
 * w4a16_gemm_ex); `path` may carry the flags w4a16_gemm_ex takes
 * (W4A16_SILU_MUL adds the fp16 product's bytes). Host-only. */
int w4a16_workspace_size_ex(int M, int N, int K, int group, int path, int parts,
                            size_t* bytes);

/* Y [M][N] = A [M][K] . dequant(Wq, scales, zeros) with fp32 accumulation.
 * The path and its grid are chosen from M, N, K, the group and the device's
 * SM count, by rules measured on GB300: the decode GEMV for M <= 16 (for
 * layers with N >= 16384 and N*K <= 2^28 up to 24 rows, in two passes over
 * the weights), else the tensor-core GEMM, on SM pairs
 * (W4A16_PATH_TENSOR_PAIR) for M >= 256 when the pairs make at least 80
 * CTAs (2 x ceil(N/256) x ceil(M/256)), for 64 < M <= 128 on layers with
 * N >= 16384 and N*K <= 2^28, and for 192 < M < 256 on layers with
 * N >= 16384, on single SMs otherwise; group sizes
 * the decode kernel does not take always go to the tensor cores. `workspace` (256-byte
 * aligned, zero-filled before first use) may be NULL when
 * w4a16_workspace_size reports 0; W4A16_ERR_WORKSPACE_TOO_SMALL otherwise.
 * Y must not overlap the inputs. */
int w4a16_gemm(const uint16_t* A, const uint32_t* Wq, const uint16_t* scales,
               const uint32_t* zeros, int M, int N, int K, int group,
               uint16_t* Y, void* workspace, size_t workspace_bytes, void* stream);

/* As w4a16_gemm with the path forced (W4A16_PATH_AUTO = automatic) and the
 * work partition forced (`parts`, 0 = automatic): for the decode path the
 * number of CTAs. The resident variant clamps it to N/16 strips (and checks
 * the fit at that count); the stream-K variant clamps it to 8192 and to the
 * split granules: 128-column blocks x groups of K, a group counted as at most
 * 512 k and K split anywhere on 64-k boundaries when group == K),
 * for the tensor-core path the number of K ranges per output tile (clamped to
 * the pipeline stages of K: K/64, or K/128 when K and the group are multiples
 * of 128). The decode path handles any M in launches of 16 rows (it streams the
 * weights once per launch) and needs group == K or group = 64 * 2^j
 * (W4A16_ERR_UNSUPPORTED_SHAPE otherwise). `path` may carry
 * W4A16_STATIC_WEIGHTS, W4A16_SILU_MUL, W4A16_BF16 and W4A16_ACT_A8 (see
 * above; with W4A16_SILU_MUL Y is [M][N/2]); any other bit is
 * W4A16_ERR_INVALID_ARG. */
int w4a16_gemm_ex(const uint16_t* A, const uint32_t* Wq, const uint16_t* scales,
                  const uint32_t* zeros, int M, int N, int K, int group,
                  uint16_t* Y, void* workspace, size_t workspace_bytes,
                  int path, int parts, void* stream);

/* The path and work partition w4a16_gemm would use on the current device:
 * for the decode path the variant (W4A16_PATH_DECODE_RESIDENT or
 * W4A16_PATH_DECODE_STREAMK) of a launch of min(M, 16) rows and its CTAs;
 * for the tensor-core paths W4A16_PATH_TENSOR and its K ranges, or
 * W4A16_PATH_TENSOR_PAIR and 1. Host-only. */
int w4a16_plan(int M, int N, int K, int group, int* path, int* parts);

/* The configuration of the one-SM tensor-core kernel (W4A16_PATH_TENSOR) for
 * M rows of a K x N layer with the given group: out[0] token tile (the MMA's
 * N), out[1] 64-k atoms per pipeline stage, out[2] activation ring slots,
 * out[3] packed-code ring slots, out[4] dequantized-operand ring slots (in
 * tensor memory), out[5] dequantizing warp groups, out[6] dynamic shared
 * memory bytes, out[7] CTAs per SM. With n >= 15, out[8..14] hold the same
 * for the CTA-pair kernel (W4A16_PATH_TENSOR_PAIR), per CTA: token tile of
 * the pair (the MMA's N), atoms per stage, activation, code and dequantized
 * ring slots, dequantizing warp groups, dynamic shared memory bytes.
 * `n` is the length of `out` (at least 8).
 * Host-only (no device is touched); W4A16_ERR_INVALID_ARG for M < 1, a null
 * `out` or n < 8, and the shape errors of w4a16_gemm. */
int w4a16_tc_config(int M, int K, int group, int* out, int n);

/* The decode-path GEMM (same kernel, same results as w4a16_gemm_ex with
 * W4A16_PATH_DECODE_STREAMK and the automatic CTA count) for callers that cannot
 * allocate device memory: code that must not allocate once running (a fixed
 * memory budget), plugins without access to their host's allocator, or loops
 * that cannot afford an allocation. The pages have no counterpart of it.
 * It takes no workspace: its scratch is a device array inside the library,
 * 32 KiB of flags plus 8 MiB of partial tiles, which every GPU that loads
 * the library holds until the process exits. Shapes whose partial tiles do
 * not fit (more than 1024 CTAs for 9..16 rows, 2048 for up to 8) are rejected
 * with W4A16_ERR_UNSUPPORTED_SHAPE; the decode path's group rule applies.
 * The first call on each device looks up the array's device address (with
 * that device current) and keeps it for the life of the process; make that
 * first call before any stream capture, and make no call after a reset of
 * the device (cudaDeviceReset), which would leave the kept address stale.
 * `stream` must belong to the current device (W4A16_ERR_INVALID_ARG
 * otherwise).
 * Every call on a device shares the one array: calls that overlap on the GPU
 * (other streams, other host threads) race and give wrong results. Each call
 * clears the flags it uses before its kernels run. Any M is taken, in
 * launches of 16 rows. */
int w4a16_gemm_noalloc(const uint16_t* A, const uint32_t* Wq, const uint16_t* scales,
                       const uint32_t* zeros, int M, int N, int K, int group,
                       uint16_t* Y, void* stream);

/* Synchronizes `stream`, then reads and clears the library's device error
 * word (set by a kernel that gave up a bounded wait or failed a self-check;
 * in the bounds-checked build of the library, compiled with -DW4A16_CHECKED,
 * also by any global or shared-memory access outside its buffer, which the
 * kernel then skips: bit 64).
 * Returns W4A16_OK or W4A16_ERR_DEVICE_CHECK (message: which check, where). */
int w4a16_device_status(void* stream);

/* Self-test of the failure path of the kernels' bounded waits, for tests:
 * launches on `stream` one kernel whose wait can never be satisfied, with
 * the kernels' own wait routine and limit (about a second): which = 0, a
 * flag that nothing sets (the stream-K decode fix-up's kind of wait; error
 * bit 32); which = 1, an mbarrier that nothing arrives on (the tensor-core
 * pipeline's kind; error bit 2). The wait gives up, records its bit in the
 * device error word and the kernel returns: nothing faults, and the next
 * w4a16_device_status returns W4A16_ERR_DEVICE_CHECK (and clears the word).
 * Other `which`: W4A16_ERR_INVALID_ARG. */
int w4a16_selftest_wait(int which, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
