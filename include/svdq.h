/*
 * svdq.h -- C ABI of the GB300 (sm_103a) SVDQuant W4A4 linear-layer operator.
 *
 *     y = scaled_mma(act4, wgt4) * wcscale + bias + lora_act_in @ lora_up
 *
 * The operator, its tensors and their dtypes are those of "SVDQuant W4A4 on
 * Blackwell" §2; the NVFP4 format (two E2M1 nibbles per byte, one FP8-E4M3
 * scale per 16 K elements, single-level scaling) is §3.1 of the same page.
 * The calling convention (argument order, NULL meanings, status codes) is
 * this library's own: the page defines no ABI.
 *
 * All functions are plain C.  Pointers named "device" are CUDA device
 * pointers owned by the caller; the library never frees or retains them.
 * Nothing in this header uses torch or any C++ type.
 */
#ifndef SVDQ_H
#define SVDQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  Every entry point returns one of these synchronously; an
 * execution fault inside the kernel surfaces, as usual with CUDA, at the
 * caller's next synchronising call. */
#define SVDQ_OK 0
#define SVDQ_ERR_INVALID_ARG -1        /* NULL required pointer, negative size, K == 0 */
#define SVDQ_ERR_UNSUPPORTED_SHAPE -2  /* M,N not multiples of 16, K not a multiple of 64,
                                          R > 128, or a size beyond the limits below   */
#define SVDQ_ERR_MISALIGNED -3         /* a tensor pointer not 16-byte aligned          */
#define SVDQ_ERR_UNSUPPORTED_DEVICE -4 /* current device is not compute capability 10.3 */
#define SVDQ_ERR_LAUNCH -5             /* the kernel launch was rejected                */
#define SVDQ_ERR_CUDA -6               /* another CUDA runtime/driver call failed       */
#define SVDQ_ERR_TIMEOUT -7            /* device status only: a bounded wait expired     */
#define SVDQ_ERR_BAD_OPTION -8         /* an svdq_options_t field is out of range       */
#define SVDQ_ERR_WORKSPACE -9          /* split-K needs a workspace: missing, smaller than
                                          svdq_workspace_size, or not 256-byte aligned  */
#define SVDQ_ERR_SCRATCH_LIMIT -10     /* the plan needs more scratch than the library's
                                          fixed SVDQ_NOALLOC_SCRATCH_BYTES              */
#define SVDQ_ERR_WCSCALE_ZERO -11      /* device status only: R > 0 and wcscale[n] == 0 for
                                          a column n (reported as the status site): the
                                          LoRA term of that column was dropped, the rest
                                          of out is computed                            */
#define SVDQ_ERR_LU_OVERFLOW -12       /* device status only: lora_up[n][r] / wcscale[n]
                                          is beyond the 16-bit I/O type's range (or not
                                          finite) for a column n (the site): that
                                          column's LoRA term is not finite, the rest of
                                          out is computed                               */

/* Size of the library's own scratch array (svdq_w4a4_gemm_split_noalloc). */
#define SVDQ_NOALLOC_SCRATCH_BYTES (16LL << 20)

/* Size limits: M, N <= 2^24 and K <= 2^20 (elements). */
#define SVDQ_MAX_MN (1LL << 24)
#define SVDQ_MAX_K (1LL << 20)
#define SVDQ_MAX_RANK 128

/* 16-bit I/O types (svdq_options_t.io_dtype). */
#define SVDQ_IO_BF16 0
#define SVDQ_IO_FP16 1

/*
 * svdq_w4a4_gemm -- y = scaled_mma(act4, wgt4) * wcscale + bias + lora_act_in @ lora_up
 * ("SVDQuant W4A4 on Blackwell" §2, §3.1, and the fused epilogue of §6.6).
 *
 * act         device, uint8 [M, K/2] row-major: element (m, k) is the E2M1 code
 *             in the low nibble of byte act[m][k/2] for even k, the high nibble
 *             for odd k.
 * wgt         device, uint8 [N, K/2], same packing (K-major; y uses act . wgt^T).
 * ascales     device, uint8 [K/16, M] FP8-E4M3, M contiguous: ascales[g][m]
 *             scales act[m][16g .. 16g+15].  Scales must be finite and
 *             non-negative (the tensor core reads them as unsigned E4M3).
 * wscales     device, uint8 [K/16, N] FP8-E4M3, likewise for wgt.
 * lora_act_in device, fp32 [M, R] row-major; NULL if and only if R == 0.
 * lora_up     device, bf16 [N, R] row-major; NULL if and only if R == 0.
 * wcscale     device, bf16 [N]; NULL means 1.  With R > 0 every wcscale[n]
 *             must be finite and non-zero, and lora_up[n][r] / wcscale[n]
 *             must fit the 16-bit type: the LoRA operand is pre-divided by
 *             wcscale so that LoRA and the main product share one
 *             accumulator.  A column that breaks this gets a wrong LoRA term
 *             (none for a zero wcscale[n], an infinite one on overflow; in
 *             fp16 that is |lora_up / wcscale| > 65504) and the launch records
 *             SVDQ_ERR_WCSCALE_ZERO or SVDQ_ERR_LU_OVERFLOW with the column in
 *             the device status word (svdq_read_device_status); every other
 *             column is unaffected.
 * bias        device, bf16 [N]; NULL means 0.
 * out         device, bf16 [M, N] row-major; every element is written.
 * M, N        multiples of 16 (the scale tensors' rows must be 16-byte
 *             strided); M == 0 or N == 0 is an empty product and returns
 *             SVDQ_OK without launching.
 * K           a positive multiple of 64.
 * R           LoRA rank, 0 <= R <= 128 (any value; padded internally).
 * stream      a cudaStream_t (0 = the legacy default stream).
 *
 * Every pointer must be 16-byte aligned.
 *
 * The computation is asynchronous on `stream`; the call never synchronises
 * and allocates no device memory.  Inputs must not be modified and `out`
 * must not be read until the stream reaches the call.  `out` must not
 * overlap any input.  Accumulation is fp32 in tensor memory; the result is
 * rounded to bf16 once, and the same call on the same inputs and device gives
 * the same bits (see svdq_options_t.relaxed_order).  The call is thread-safe;
 * concurrent calls on different streams are independent.
 */
int svdq_w4a4_gemm(const void* act, const void* wgt, const void* ascales, const void* wscales,
                   const float* lora_act_in, const void* lora_up, const void* wcscale,
                   const void* bias, void* out, int64_t M, int64_t N, int64_t K, int64_t R,
                   void* stream);

/* Optional knobs.  Zero-initialise and set only what is needed; a NULL
 * options pointer equals all zeros. */
typedef struct svdq_options {
    int32_t tile_n;      /* 0 = planner's choice; else 128 or 256                  */
    int32_t stages;      /* 0 = pipeline-depth solver's choice; else forced (2..8)  */
    int32_t max_ctas;    /* 0 = one persistent CTA per SM; else cap on the grid    */
    int32_t timeout_ms;  /* bounded-wait limit inside the kernel; 0 = 2000 ms       */
    int32_t debug_fault; /* tests only: 1 makes the MMA issuers wait on a barrier
                            no role arrives on, so the kernel must time out and
                            report SVDQ_ERR_TIMEOUT instead of hanging             */
    int32_t cta_group;   /* 0 = planner's choice; 1 = one CTA per MMA, 2 = a CTA pair
                            issuing 256-row MMAs (tile_n must then be 256)           */
    int32_t io_dtype;    /* 16-bit I/O type of lora_up, wcscale, bias and out:
                            SVDQ_IO_BF16 (0, default) or SVDQ_IO_FP16 (1, IEEE
                            binary16; LoRA operands are then rounded to fp16) */
    int32_t k_splits;    /* split-K: 0 = default (none on entry points without a
                            workspace, the planner's choice on svdq_w4a4_gemm_split);
                            -1 = the planner's choice; 1 = none; 2..8 = that many K
                            splits per tile (svdq_w4a4_gemm_split only)           */
    int32_t act_scales_packed; /* 0 = ascales as uint8 [K/16, M] (default); 1 = the
                            same scales as uint32 words [K/64, M], word (s, m) byte g
                            = ascales[4s + g][m] (svdq_pack_scales' layout): an
                            activation quantiser that writes them this way saves
                            the kernel's per-call transpose                      */
    int32_t relaxed_order; /* 0 = bit-reproducible (default): the two MMA issuer
                            threads take turns, so ring items reach the tensor core
                            in a fixed order and every call on the same inputs gives
                            the same bits; 1 = the issuers run freely, so the fp32
                            accumulation order (and the last bits of out, always
                            within the stated tolerance) may change from call to
                            call, for a few percent more speed when scales arrive
                            packed                                               */
    int32_t lora_act_16bit; /* 0 = lora_act_in is fp32 [M, R] (default); 1 = it holds
                            the 16-bit values [M, R] in the I/O type (bf16, or fp16
                            with io_dtype fp16; pass the buffer's address cast to
                            const float*): the LoRA operand the tensor cores take,
                            which the kernel otherwise rounds from fp32 (RNE), as an
                            activation quantiser can write it.  The operator then
                            carries 64 ranks per LoRA ring item instead of 32
                            (half the ring slots at R = 128).  Needs R a multiple
                            of 8 (SVDQ_ERR_BAD_OPTION otherwise); results equal
                            the fp32 route's on the rounded values, bit for bit */
} svdq_options_t;

/* svdq_w4a4_gemm with options; identical semantics otherwise.  With
 * io_dtype = SVDQ_IO_FP16, lora_up, wcscale, bias and out hold IEEE fp16 in
 * the same shapes (the fp16 variant "SVDQuant W4A4 on Blackwell" §8 also
 * measures): y is rounded to fp16 (RNE) and the LoRA operands LA' = f16(LA),
 * LU' = f16(LU / wcscale) are fp16 on the tensor cores. */
int svdq_w4a4_gemm_ex(const void* act, const void* wgt, const void* ascales, const void* wscales,
                      const float* lora_act_in, const void* lora_up, const void* wcscale,
                      const void* bias, void* out, int64_t M, int64_t N, int64_t K, int64_t R,
                      const svdq_options_t* options, void* stream);

/*
 * svdq_prepack_weights -- the weight-side operands in the form the kernel
 * consumes them, built once per weight load ("SVDQuant W4A4 on Blackwell"
 * §3.1: the tensor core takes the four group scales of one 64-wide K step
 * as one 32-bit word per row; §6.3: the LoRA up-projection shares the main
 * accumulator, so it is pre-divided by wcscale).  Weights are static, so
 * neither the per-call scale transpose nor the divide needs to be repeated.
 *
 * wscales        device, uint8 [K/16, N] FP8-E4M3 (as for svdq_w4a4_gemm).
 * lora_up        device, 16-bit [N, R]; NULL if and only if R == 0.
 * wcscale        device, 16-bit [N]; NULL means 1.
 * N, K, R        as for svdq_w4a4_gemm (N a multiple of 16, K of 64, R <= 128).
 * io_dtype       SVDQ_IO_BF16 or SVDQ_IO_FP16: the type of lora_up, wcscale
 *                and lora_up_packed.
 * wscales_packed device, uint32 [K/64, N] (K*N/16 bytes, the same size as
 *                wscales): word (s, n) holds byte g (bits 8g..8g+7) =
 *                wscales[4s + g][n], g < 4.
 * lora_up_packed device, 16-bit [N, R]: LU'[n][r] = round16(fp32(lora_up[n][r])
 *                * rcp(wcscale[n])) with the correctly rounded fp32 reciprocal,
 *                one fp32 product and round-to-nearest-even into io_dtype;
 *                0 where wcscale[n] == 0, lora_up itself when wcscale is NULL.
 *                Ignored (may be NULL) when R == 0.
 * stream         a cudaStream_t.
 *
 * Every pointer must be 16-byte aligned; outputs must not overlap inputs.
 * Asynchronous on `stream`, allocates nothing.  Returns SVDQ_OK for N == 0.
 */
int svdq_prepack_weights(const void* wscales, const void* lora_up, const void* wcscale,
                         int64_t N, int64_t K, int64_t R, int32_t io_dtype, void* wscales_packed,
                         void* lora_up_packed, void* stream);

/*
 * svdq_pack_scales -- any FP8-E4M3 scale tensor [K/16, rows] (activation or
 * weight scales) into the word layout the kernel feeds to the tensor core
 * ("SVDQuant W4A4 on Blackwell" §3.1: one 32-bit word of four group scales
 * per row and 64-wide K step): uint32 [K/64, rows], word (s, r) byte g =
 * scales[4s + g][r].  The words are what svdq_options_t.act_scales_packed
 * expects for ascales and what svdq_prepack_weights writes for wscales.
 * rows a multiple of 16, K of 64; 16-byte aligned pointers; asynchronous on
 * `stream`, allocates nothing.  Returns SVDQ_OK for rows == 0.
 */
int svdq_pack_scales(const void* scales, int64_t rows, int64_t K, void* packed, void* stream);

/*
 * svdq_quantize_act -- the operator's activation inputs from 16-bit
 * activations, in one pass over x ("SVDQuant W4A4 on Blackwell" §1: the W4A4
 * operator is the compute-bound half of SVDQuant, fed by an activation
 * quantiser; §2: act, ascales and lora_act_in, in the formats of §3.1; §3.3:
 * LA is the LoRA-down activation).  The page names this producer but does not
 * define it; the library takes the plain NVFP4 reading, per group of 16
 * consecutive k in a row m (single-level scaling, as everywhere here):
 *
 *     amax             = max |x[m, k]| over the group
 *     ascales[g][m]    = E4M3(amax / 6), rounded to nearest even, saturating
 *                        at 448; the scale s is that byte's value
 *     code(m, k)       = E2M1(x[m, k] / s), rounded to nearest even (ties to
 *                        the even code), saturating at +-6; every code of the
 *                        group is 0 when s == 0; a code of magnitude 0 is +0
 *     lora_act_in[m,r] = sum_k x[m, k] * lora_down[r, k]   (fp32 result)
 *
 * The rounding decisions are those of the exact quotients amax / 6 and x / s
 * (the kernel's fp32 arithmetic reaches the same codes for 16-bit x).
 *
 * x             device, 16-bit [M, K] row-major (io_dtype: bf16 or fp16), finite.
 * lora_down     device, same 16-bit type [R, K] row-major; NULL iff R == 0.
 * M, K, R       M a multiple of 16, K a positive multiple of 64, 0 <= R <= 128,
 *               within the size limits above.  M == 0 returns SVDQ_OK without
 *               touching any pointer (which may then be NULL).
 * io_dtype      SVDQ_IO_BF16 or SVDQ_IO_FP16.
 * scales_packed 0: ascales is uint8 [K/16, M] (svdq_w4a4_gemm's layout);
 *               1: uint32 [K/64, M] words, word (s, m) byte g = scale of group
 *               4s + g (svdq_pack_scales' layout, for act_scales_packed).
 * lora_act_16bit 0: lora_act_in is fp32; 1: it is written in x's 16-bit type,
 *               rounded to nearest even from the fp32 sum (the operand the
 *               operator's lora_act_16bit option takes).
 * act           device, uint8 [M, K/2]: low nibble = even k.
 * ascales       device, as selected by scales_packed.
 * lora_act_in   device, fp32 (or 16-bit) [M, R]; NULL iff R == 0.  Accumulated in fp32 on
 *               the tensor cores from the 16-bit products; with several CTAs
 *               per 128-row tile their fp32 partials are added in a fixed
 *               order, so the same call gives the same bits every time.
 * stream        a cudaStream_t.
 *
 * Every pointer must be 16-byte aligned; outputs must not overlap inputs or
 * each other.  Asynchronous on `stream`, allocates nothing, never
 * synchronises.  A bounded wait that expires records SVDQ_ERR_TIMEOUT in the
 * device status word.
 */
int svdq_quantize_act(const void* x, const void* lora_down, int64_t M, int64_t K, int64_t R,
                      int32_t io_dtype, int32_t scales_packed, int32_t lora_act_16bit, void* act,
                      void* ascales, void* lora_act_in, void* stream);

/* The launch svdq_quantize_act would make (host only; touches no device when
 * sm_count > 0): CTAs per 128-row tile along K (*splits, 1, 2, 4 or 8: a
 * cluster that adds its LoRA-down partials in distributed shared memory),
 * total CTAs, ring stages and dynamic shared memory per CTA.  Any output
 * pointer may be NULL.  sm_count <= 0 plans for the current device. */
int svdq_quantize_query(int64_t M, int64_t K, int64_t R, int32_t sm_count, int32_t* splits,
                        int32_t* grid, int32_t* stages, int32_t* smem_bytes);

/*
 * svdq_w4a4_linear -- the whole layer from 16-bit activations ("SVDQuant W4A4
 * on Blackwell" §1: the activation quantiser feeding the W4A4 operator of §2):
 *
 *     y = scaled_mma(quant(x), wgt4) * wcscale + bias + (x @ lora_down^T) @ lora_up
 *
 * as svdq_quantize_act (packed activation scales; the LoRA-down product in x's
 * 16-bit type when R is a multiple of 8, else in fp32) followed by
 * svdq_w4a4_gemm_prepacked with act_scales_packed (and lora_act_16bit when the
 * product is 16-bit), both on `stream`; act, the scale words and lora_act_in
 * live in `workspace` between the two launches.  The result is that of those
 * two calls, bit for bit.
 *
 * x, lora_down   as for svdq_quantize_act; their 16-bit type is options->io_dtype.
 * wgt, wscales_packed, lora_up_packed, wcscale, bias, out
 *                as for svdq_w4a4_gemm_prepacked (weights from svdq_prepack_weights).
 * M, N, K, R     as for svdq_w4a4_gemm.
 * options        as for svdq_w4a4_gemm_ex (NULL: defaults); act_scales_packed and
 *                lora_act_16bit are set by this call.
 * workspace      device, 256-byte aligned, at least svdq_linear_workspace_size(M, K, R)
 *                bytes (NULL when that is 0); SVDQ_ERR_WORKSPACE otherwise.
 *
 * Returns the first non-OK status of the two steps; if the operator step
 * rejects its arguments, the quantiser may already be in the stream (it
 * writes only the workspace).  Asynchronous, allocates nothing.
 */
int svdq_w4a4_linear(const void* x, const void* lora_down, const void* wgt,
                     const void* wscales_packed, const void* lora_up_packed, const void* wcscale,
                     const void* bias, void* out, int64_t M, int64_t N, int64_t K, int64_t R,
                     const svdq_options_t* options, void* workspace, int64_t workspace_bytes,
                     void* stream);

/* Workspace bytes svdq_w4a4_linear needs (host only): act, the packed
 * activation scales and lora_act_in, each padded to 256 bytes; a negative
 * status for arguments svdq_w4a4_linear would reject by shape. */
int64_t svdq_linear_workspace_size(int64_t M, int64_t K, int64_t R);

/*
 * svdq_w4a4_gemm_prepacked -- svdq_w4a4_gemm_ex on prepacked weights: the
 * same operator and result, with wscales_packed and lora_up_packed from
 * svdq_prepack_weights in place of wscales and lora_up.  wcscale must be the
 * one the LoRA operand was packed with (the epilogue still multiplies by it);
 * bias, options and every other argument are as for svdq_w4a4_gemm_ex
 * (options->io_dtype must match the packing).
 */
int svdq_w4a4_gemm_prepacked(const void* act, const void* wgt, const void* ascales,
                             const void* wscales_packed, const float* lora_act_in,
                             const void* lora_up_packed, const void* wcscale, const void* bias,
                             void* out, int64_t M, int64_t N, int64_t K, int64_t R,
                             const svdq_options_t* options, void* stream);

/*
 * svdq_w4a4_gemm_split -- the operator with split-K: each output tile's K
 * range is divided into k_splits parts that run on different SMs at once;
 * every part but the last writes an fp32 partial tile into `workspace`, the
 * last adds them to its own accumulator and applies the epilogue.  This is
 * for shapes whose tiles leave most SMs idle (few rows, e.g. M = 256) and
 * whose K is long: the planner splits only when the tiles fill at most half
 * of the co-resident clusters, gives every part a cluster of its own and
 * keeps at least eight 256-wide K blocks per part (a split costs about as
 * much as ten K blocks of tensor-core work).  Forced splits (k_splits 2..8)
 * need at least one K block per part.  "SVDQuant W4A4 on Blackwell" §4 names the small-M
 * case; the split itself is this library's.
 *
 * Arguments are those of svdq_w4a4_gemm_ex (or svdq_w4a4_gemm_prepacked when
 * weights_prepacked == 1), plus:
 * workspace        device, at least svdq_workspace_size(...) bytes, 256-byte
 *                  aligned, zero-filled before its first use; owned by the
 *                  caller and reused across calls.  Every completed call
 *                  leaves its flags at zero again (a part raises its flag when
 *                  its partial is stored, the last part lowers it once it has
 *                  added the partial), so the same workspace serves any later
 *                  call, including launches replayed from a CUDA graph.  After
 *                  a launch that recorded SVDQ_ERR_TIMEOUT the flags may be
 *                  left raised: zero the workspace again before reusing it.
 *                  Calls that share a workspace must not overlap on the GPU
 *                  (they would race on its contents).
 * workspace_bytes  its size.
 * When the plan has no split the workspace is not touched.  The summation
 * order of the K parts differs from the unsplit kernel (fp32 partials), so
 * results agree with it within the operator's tolerance, not bit for bit.
 * The last part of a tile waits (bounded) for the other parts, which the
 * planner places on clusters of their own so that all parts of a launch are
 * resident at once.  That holds while the launch has the GPU's SMs to itself:
 * a split launch running concurrently with other kernels that occupy many
 * SMs (another stream) may not get all of its parts scheduled in time and
 * then ends with SVDQ_ERR_TIMEOUT in the device status word instead of a
 * result.  Run split launches alone on the device, or stream-ordered.
 * Returns SVDQ_ERR_WORKSPACE if the workspace is missing or too small.
 */
int svdq_w4a4_gemm_split(const void* act, const void* wgt, const void* ascales,
                         const void* wscales, const float* lora_act_in, const void* lora_up,
                         const void* wcscale, const void* bias, void* out, int64_t M, int64_t N,
                         int64_t K, int64_t R, const svdq_options_t* options,
                         int32_t weights_prepacked, void* workspace, int64_t workspace_bytes,
                         void* stream);

/*
 * svdq_w4a4_gemm_split_noalloc -- svdq_w4a4_gemm_split for callers that cannot
 * allocate device memory: code that runs while a serving engine has reserved
 * the whole device for its own memory pool, or inside a runtime that forbids
 * cudaMalloc after start-up, and so has no workspace to pass.  (The paper has
 * no counterpart; it is this library's own.)  The split-K partial tiles and
 * flags live in a scratch array built into the library,
 * SVDQ_NOALLOC_SCRATCH_BYTES (16 MiB) per GPU that loads it, held until the
 * process exits; nothing is allocated per call, by this function or by
 * anything it calls.
 *
 * Arguments are those of svdq_w4a4_gemm_split without the workspace.  Plans
 * needing more than SVDQ_NOALLOC_SCRATCH_BYTES (svdq_workspace_size) return
 * SVDQ_ERR_SCRATCH_LIMIT before anything is launched.  The first call on a
 * device looks up the array's device address (one cudaGetSymbolAddress per
 * device, under the library's lock).  Every call on a device
 * shares the one array: calls that overlap on the GPU (other streams, other
 * threads) race on it and must be serialised by the caller.  The array
 * starts zero-filled and every completed call leaves its flags at zero, so
 * nothing needs clearing between calls; after a launch that recorded
 * SVDQ_ERR_TIMEOUT, svdq_read_device_status with clear != 0 zero-fills the
 * array again (synchronously) along with the status word.
 */
int svdq_w4a4_gemm_split_noalloc(const void* act, const void* wgt, const void* ascales,
                                 const void* wscales, const float* lora_act_in,
                                 const void* lora_up, const void* wcscale, const void* bias,
                                 void* out, int64_t M, int64_t N, int64_t K, int64_t R,
                                 const svdq_options_t* options, int32_t weights_prepacked,
                                 void* stream);

/* Workspace bytes svdq_w4a4_gemm_split needs for this shape and options
 * (0 when the plan does not split), or a negative status.  sm_count <= 0
 * plans exactly as a launch on the current device does; sm_count > 0 plans
 * for that many SMs without touching a device. */
int64_t svdq_workspace_size(int64_t M, int64_t N, int64_t K, int64_t R,
                            const svdq_options_t* options, int32_t sm_count);

/* The launch plan the library would use (host only; touches no device when
 * sm_count > 0).  Shared-memory accounting follows "SVDQuant W4A4 on
 * Blackwell" §7 (pipeline depth solved from the per-SM budget after every
 * other buffer; operands split across a CTA pair are counted per CTA). */
typedef struct svdq_plan {
    int32_t tile_m, tile_n, tile_k;  /* output tile per cluster and K per ring item  */
    int32_t cta_group;               /* CTAs sharing one MMA (1 or 2)                */
    int32_t num_ab_stage;            /* ring depth (stages in flight)                */
    int32_t num_acc_stage;           /* accumulator buffers in tensor memory         */
    int32_t stage_bytes;             /* shared-memory bytes per ring stage, per CTA  */
    int32_t lora_block_bytes;        /* LoRA operand bytes per ring item, per CTA    */
    int32_t lora_blocks;             /* LoRA ring items per tile (32 ranks each)     */
    int32_t k_blocks;                /* 256-wide K blocks per tile                   */
    int32_t smem_bytes;              /* dynamic shared memory per CTA                */
    int32_t tmem_cols;               /* tensor-memory columns allocated per CTA      */
    int32_t tmem_cols_used;          /* of which used                                */
    int32_t threads;                 /* threads per CTA                              */
    int64_t num_tiles;               /* output tiles                                 */
    int32_t grid;                    /* persistent CTAs launched                     */
    int32_t sm_count;                /* SMs the grid was sized for                   */
    int32_t kblocks_per_stage;       /* 256-wide K blocks carried by one ring stage  */
    int32_t k_splits;                /* K splits per tile (1: none)                  */
    int64_t num_units;               /* work units: num_tiles * k_splits             */
    int64_t workspace_bytes;         /* split-K workspace the launch needs (0: none) */
} svdq_plan_t;

/* Fill *plan for the given shape.  sm_count <= 0 queries the current device
 * (SVDQ_ERR_UNSUPPORTED_DEVICE if none); sm_count > 0 plans for that many
 * SMs with GB300 limits (227 KB shared memory per block, 512 TMEM columns)
 * and touches no device.  With options->k_splits == 0 the plan is that of the
 * entry points without a workspace (no split-K); -1 or 2..8 plans split-K as
 * svdq_w4a4_gemm_split would. */
int svdq_query_plan(int64_t M, int64_t N, int64_t K, int64_t R, const svdq_options_t* options,
                    int32_t sm_count, svdq_plan_t* plan);

/* Per-CTA LoRA prologue bytes of one pipeline stage when an A-side operand
 * [tile_m, R] and a B-side operand [tile_n, R] of elem_bytes each are split
 * across cta_group CTAs: A along M, B along N, so BOTH are divided by
 * cta_group ("SVDQuant W4A4 on Blackwell" §7.1-7.5).  Writes the two parts
 * to *la_bytes / *lu_bytes (either may be NULL) and returns their sum, or a
 * negative status for bad arguments. */
int64_t svdq_lora_stage_bytes(int64_t tile_m, int64_t tile_n, int64_t R, int64_t elem_bytes,
                              int64_t cta_group, int64_t* la_bytes, int64_t* lu_bytes);

/* Read (and if clear != 0, reset) the library's device status word for the
 * current device.  *code is SVDQ_OK, SVDQ_ERR_TIMEOUT (*site identifies the
 * wait that expired), SVDQ_ERR_WCSCALE_ZERO or SVDQ_ERR_LU_OVERFLOW (*site is
 * the column); *block is the CTA that recorded it.  The first condition
 * recorded since the last reset is kept.  Clearing a SVDQ_ERR_TIMEOUT also
 * zero-fills the scratch array of svdq_w4a4_gemm_split_noalloc, if that entry
 * point has been used on this device (a timed-out split launch can leave its
 * flags raised).  Synchronises the device.  Any of the output pointers may
 * be NULL. */
int svdq_read_device_status(int32_t* code, int32_t* site, int32_t* block, int clear);

/* Human-readable name of a status code (static storage, never NULL). */
const char* svdq_status_string(int status);

/* Library ABI version (major * 10000 + minor * 100 + patch).  The structs
 * above grow only at their end; a caller built against a header with another
 * major.minor (SVDQ_ABI_VERSION / 100) must not pass them to this library. */
#define SVDQ_ABI_VERSION 701
int svdq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SVDQ_H */
