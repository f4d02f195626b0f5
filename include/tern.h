/*
 * tern.h -- C ABI of libtern, the ternary-weight linear layer for one
 * NVIDIA GB300 GPU (sm_103a).
 *
 * The layer computes Y[M,N] = X[M,K] . W^T with W[n,k] = t[n,k] * s[n, k/128]:
 * ternary weights t in {-1,0,+1}, one FP16 scale per 128 consecutive weights
 * along K, BF16 activations X, fp32 accumulation and fp32 output Y.
 *
 * Sources (web pages, cited by a short name, address and section):
 *   [EMB] "Ternary embedding model in vLLM", 2kiu.com/news/5082861
 *         §1.1 ternary weights with a shared FP16 scale per 128 weights;
 *         §2.2 the packed weight tensor is [out_features, in_features/4]
 *              uint8; fused QKV tensors are cut by offsets, and the scales
 *              must be cut the same way;
 *         §3.1 the packing rule (2-bit codes 00->0, 01->+1, 10->-1,
 *              11->reserved read as 0; four codes per byte, little-endian,
 *              first weight in the lowest bits; scale blocks cut
 *              contiguously along K);
 *         §3   disk layout and GPU layout must be reconciled;
 *         §4.2 the op: x [M,K], packed w [N,K/4], scale [N,K/128] -> y [M,N];
 *              signs accumulated inside a 128-block, scale applied once at
 *              the block boundary; the page's kernel takes half-precision
 *              activations and writes a half-precision output;
 *         §4.4 inputs are reshaped to a 2-D contiguous [tokens, hidden].
 *   [B27] "Porting ternary Bonsai 2 27B to vLLM", m.xxqk.cn/news/594847
 *         §5.2 FP16 scales are stored little-endian.
 *
 * Conventions for every call
 *   - Pointers named d_* or documented as "device" are device pointers on
 *     the current CUDA device; arrays documented as "host" live in host
 *     memory.  The caller owns and allocates every buffer, including the
 *     workspace; the library allocates no memory and keeps no state.
 *   - `stream` is a cudaStream_t passed as void* (NULL: the legacy default
 *     stream).  Calls only enqueue work and return; results are ready when
 *     the stream reaches them.
 *   - Argument problems (null pointers, bad shapes, misalignment, small
 *     buffers) return an error code before anything is enqueued.  Launch
 *     failures return TERN_ERR_CUDA.  Data problems (values outside the
 *     format) never stop a call; where a `d_err` counter is given, the
 *     kernel adds their count to it with an atomic add.
 *   - No call throws; no call synchronises the device.
 *   - Sizes are int64_t elements unless named *_bytes.
 */
#ifndef TERN_H
#define TERN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of activations (x_type) and outputs (out_type). */
typedef enum { TERN_X_BF16 = 0, TERN_X_F16 = 1 } tern_x_type;
typedef enum { TERN_OUT_F32 = 0, TERN_OUT_BF16 = 1, TERN_OUT_F16 = 2 } tern_out_type;

typedef enum {
    TERN_OK = 0,
    TERN_ERR_NULL = 1,        /* a required pointer is NULL */
    TERN_ERR_SHAPE = 2,       /* bad dimension: negative, K not a multiple of 128, ... */
    TERN_ERR_ALIGN = 3,       /* a pointer or leading dimension breaks an alignment rule */
    TERN_ERR_SIZE = 4,        /* a buffer given with its size is too small */
    TERN_ERR_UNSUPPORTED = 5, /* valid request this build cannot serve (e.g. no GPU) */
    TERN_ERR_CUDA = 6         /* a CUDA runtime call or kernel launch failed */
} tern_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* tern_status_string(int status);

/* Library ABI version: major*10000 + minor*100 + patch. */
int tern_version(void);

/* ------------------------------------------------------------------------
 * On-disk format ([EMB] §2.2, §3.1)
 *   packed : uint8 [N, K/4], row-major.  Weight (n,k) is in byte
 *            n*(K/4) + k/4 at bits 2*(k%4)..2*(k%4)+1.  Codes: 00 -> 0,
 *            01 -> +1, 10 -> -1, 11 -> reserved, read as 0.
 *   scales : raw IEEE FP16 bits, uint16 [N, K/128], row-major,
 *            little-endian ([B27] §5.2); scale (n,g) covers k in
 *            [128g, 128g+128).
 * ---------------------------------------------------------------------- */

/* Pack ternary values into 2-bit codes ([EMB] §3.1).
 *   d_t      device int8 [N, K] row-major, values in {-1, 0, +1}
 *   d_packed device uint8 [N, K/4] output
 *   d_err    optional device int32: incremented by the number of entries of
 *            d_t outside {-1,0,+1}; those are written as code 00 (weight 0).
 * Requires N >= 0, K >= 0, K % 4 == 0.  N*K == 0 is a no-op. */
tern_status tern_pack(const int8_t* d_t, int64_t N, int64_t K, uint8_t* d_packed,
                      int32_t* d_err, void* stream);

/* Unpack 2-bit codes into ternary values ([EMB] §3.1, the unpack routine).
 *   d_packed device uint8 [N, K/4];  d_t device int8 [N, K] output.
 *   d_err    optional: incremented by the number of reserved code-11
 *            entries, which unpack to 0.
 * Requires N >= 0, K >= 0, K % 4 == 0. */
tern_status tern_unpack(const uint8_t* d_packed, int64_t N, int64_t K, int8_t* d_t,
                        int32_t* d_err, void* stream);

/* ------------------------------------------------------------------------
 * GPU tile layout ("tiled"): this library's own format, built by
 * tern_repack from the on-disk pair.  The pages give no GPU layout; they
 * only ask that it be reconciled with the disk layout ([EMB] §3).
 *
 * Rows are padded to Np = 128*ceil(N/128) with weight 0 and scale 0.  With
 * G = K/128 scale groups and R = Np/128 row tiles, a unit is one 128-row x
 * 128-weight block:
 *   codes : R*G units of 4096 bytes; unit (b,g) at byte (b*G + g)*4096.
 *           Half h (0,1) at byte 2048*h of the unit; row r (0..127) of the
 *           tile at 16*r within the half; the row's 16 bytes are four
 *           little-endian uint32 words, word q covering the weights
 *           k0..k0+15 with k0 = 128g + 64h + 16q.  In a word, weight k0+2i
 *           is at bits 2i..2i+1 and weight k0+2i+1 at bits 16+2i..17+2i
 *           (i = 0..7).  The value stored is the biased code v = t + 1 in
 *           {0,1,2}.
 *   scales: R*G units of 256 bytes starting at byte R*G*4096; unit (b,g)
 *           at R*G*4096 + (b*G + g)*256 holds the FP16 scales s[128b+r][g]
 *           for r = 0..127 (little-endian).
 * A unit is one contiguous 4 KB stream element; one thread per row reads
 * its own two 16-byte runs, and each 16-weight word decodes to the eight
 * bf16 pairs of one tensor-core K-step.
 * ---------------------------------------------------------------------- */

/* Bytes of the tiled layout for an N x K weight: 4352 * ceil(N/128) * (K/128).
 * Returns 0 for invalid shapes (N < 0, K <= 0 or K % 128 != 0). */
size_t tern_tiled_bytes(int64_t N, int64_t K);

/* On-disk (packed, scales) -> tiled.  Reserved code 11 is stored as weight
 * 0 and counted in d_err.  Requires K > 0, K % 128 == 0, N >= 0,
 * d_packed 4-byte aligned, d_tiled 16-byte aligned,
 * tiled_bytes >= tern_tiled_bytes(N, K). */
tern_status tern_repack(const uint8_t* d_packed, const uint16_t* d_scales, int64_t N, int64_t K,
                        void* d_tiled, size_t tiled_bytes, int32_t* d_err, void* stream);

/* Several independent repacks in one launch (a library convenience, with no
 * counterpart in the pages: a loader converting many weights at once shares
 * the fixed costs of a launch).  Repack i is tern_repack(d_packed[i],
 * d_scales[i], Ns[i], Ks[i], d_tiled[i], tiled_bytes[i]); every array is a
 * HOST array of `count` entries (1 <= count <= TERN_MAX_GROUP) and the
 * pointers in them follow tern_repack's rules.  Repacks with Ns[i] == 0 are
 * skipped; invalid codes of all of them add up in *d_err.  The tiled
 * buffers must not overlap one another or any source. */
tern_status tern_repack_grouped(int count, const uint8_t* const* d_packed, const uint16_t* const* d_scales,
                                const int64_t* Ns, const int64_t* Ks, void* const* d_tiled,
                                const size_t* tiled_bytes, int32_t* d_err, void* stream);

/* tiled -> on-disk (packed, scales), rows < N only; the inverse of
 * tern_repack on valid data (code 11 comes back as 00).  A stored value of
 * 3 (never written by tern_repack) unpacks to weight 0 and is counted in
 * d_err.  Requires the same shapes and alignments as tern_repack, and
 * d_packed 4-byte aligned. */
tern_status tern_unrepack(const void* d_tiled, int64_t N, int64_t K, uint8_t* d_packed,
                          uint16_t* d_scales, int32_t* d_err, void* stream);

/* ------------------------------------------------------------------------
 * The linear layer ([EMB] §4.2).
 *
 *   Y[m, n] = sum_k X[m, k] * t[n, k] * s[n, k/128]
 *
 * computed as: per 128-wide group, an fp32 partial of exact products
 * x * t; the FP16 scale (converted exactly to fp32) multiplies the partial
 * once per group; the scaled partials are summed in fp32.  The result
 * satisfies |Y - Y_exact| <= 1e-4 * sum_k |X[m,k] * W[n,k]| per output.
 *
 *   d_X      device bf16 bits [M, ldx] row-major; 16-byte aligned,
 *            ldx % 8 == 0, ldx >= K
 *   d_tiled  device tiled weights for N x K (tern_repack); 16-byte aligned
 *   d_Y      device fp32 [M, ldy] row-major output, ldy >= N; 4-byte aligned
 *   d_ws     device workspace of ws_bytes >= tern_workspace_bytes(M, N, K),
 *            256-byte aligned.  It must be zero-filled before its first
 *            use; every completed call leaves its counters at zero again,
 *            so one workspace can serve a sequence of calls on one stream.
 *            Calls that may overlap in time need separate workspaces.  Its
 *            first 32-bit word is an error word: the kernel sets it non-zero
 *            (and returns early, leaving Y incomplete) only if a pipeline
 *            wait timed out (2 s), which correct inputs never cause.  Read
 *            it with tern_workspace_error.  A call that ended that way may
 *            also leave tile counters and partial sums behind: clear the
 *            whole workspace (tern_workspace_reset) before it serves again.
 * M == 0 or N == 0 is a no-op.  K must be a positive multiple of 128.
 * X is read after any preceding kernel on the stream completes; kernels
 * launched with programmatic dependent launch may begin streaming weights
 * earlier. */
size_t tern_workspace_bytes(int64_t M, int64_t N, int64_t K);

tern_status tern_linear(const uint16_t* d_X, int64_t ldx, const void* d_tiled,
                        int64_t M, int64_t N, int64_t K,
                        float* d_Y, int64_t ldy, void* d_ws, size_t ws_bytes, void* stream);

/* Multi-output variant for fused projections (QKV, gate+up; [EMB] §2.2):
 * one weight stream over the concatenated rows, N = sum(n_sizes), with
 * output rows [off_j, off_j + n_sizes[j]) written to d_Ys[j] (row stride
 * ldys[j] >= n_sizes[j]).  Each scale travels with its own row, so the
 * cut applies to weights and scales alike.  n_sizes, d_Ys and ldys are
 * HOST arrays of n_out entries (1 <= n_out <= 4); d_Ys[j] are device
 * pointers.  Other arguments as tern_linear; the workspace size is
 * tern_workspace_bytes(M, N, K) for the total N. */
tern_status tern_linear_multi(const uint16_t* d_X, int64_t ldx, const void* d_tiled,
                              int64_t M, int64_t K, int n_out, const int64_t* n_sizes,
                              float* const* d_Ys, const int64_t* ldys,
                              void* d_ws, size_t ws_bytes, void* stream);

/* tern_linear for callers that cannot allocate device memory, e.g. code
 * running while a CUDA graph is being captured (where cudaMalloc is not
 * allowed) or a plug-in whose device memory belongs to a host framework's
 * allocator.  The source pages have no counterpart: this is a library
 * convenience.  Arguments and results are those of tern_linear; instead of a
 * caller workspace the call uses a scratch array built into the library
 * (16 MiB per device, held by every GPU that loads the library until the
 * process exits).  It allocates nothing.
 *   - Problems whose tern_workspace_bytes(M, N, K) exceeds 16 MiB return
 *     TERN_ERR_SIZE before anything is enqueued.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address and may load the library's GPU code; make that
 *     first call before any stream capture.
 *   - Each call clears the part of the array it uses (an asynchronous
 *     memset on `stream`) before its kernels run.  All calls share the one
 *     array, so calls that may overlap in time on the GPU race; serialise
 *     them (one stream) or use tern_linear with separate workspaces. */
tern_status tern_linear_noalloc(const uint16_t* d_X, int64_t ldx, const void* d_tiled,
                                int64_t M, int64_t N, int64_t K, float* d_Y, int64_t ldy,
                                void* stream);

/* The general form of tern_linear_multi ([EMB] §4.2 half-precision
 * activations and output; §2.2 fused projections):
 *   d_X      device [M, ldx] of bf16 (x_type TERN_X_BF16) or fp16
 *            (TERN_X_F16) bits; alignment as tern_linear.  fp16 and bf16
 *            inputs are used exactly (the weights are exact in both
 *            formats and products accumulate in fp32).
 *   d_Ys[j]  device [M, ldys[j]] outputs of out_type: fp32, or bf16 / fp16
 *            rounded to nearest even from the fp32 result (4-byte aligned
 *            for fp32, 2-byte otherwise).
 * Other arguments as tern_linear_multi; unknown x_type or out_type values
 * return TERN_ERR_SHAPE. */
tern_status tern_linear_ex(const void* d_X, int x_type, int64_t ldx, const void* d_tiled,
                           int64_t M, int64_t K, int n_out, const int64_t* n_sizes,
                           void* const* d_Ys, const int64_t* ldys, int out_type,
                           void* d_ws, size_t ws_bytes, void* stream);

/* A group of independent linears in one launch.  The source pages have no
 * counterpart: this is a library convenience for problems that do not feed
 * one another (projections of different sequences or experts, or layers
 * whose inputs are all known), so that small linears share the fixed costs
 * of a launch.  Problem i computes
 *   Y_i[m, n] = sum_k X_i[m, k] * t_i[n, k] * s_i[n, k/128]
 * exactly as tern_linear_ex with one output: X_i = d_Xs[i] [M, ldxs[i]]
 * (x_type for all), weights d_tiled[i] for Ns[i] x Ks[i] (plain tiled
 * layout), output d_Ys[i] [M, ldys[i]] of out_type.  d_Xs, ldxs, d_tiled,
 * Ns, Ks, d_Ys and ldys are HOST arrays of `count` entries
 * (1 <= count <= TERN_MAX_GROUP); the pointers in them are device pointers
 * with the alignment rules of tern_linear_ex.  Problems with Ns[i] == 0 are
 * skipped; M == 0 is a no-op.  Each result meets the bound of tern_linear;
 * it may differ from a separate call's in the last bits, as the CTAs split a
 * problem's groups differently and fp32 partial sums then add in another
 * order (a given group is still deterministic).  M <= 16 runs as one
 * streaming launch; larger M as one tensor-core GEMM launch over all the
 * problems' tiles (after one activation conversion, and followed by one
 * reduction of the problems whose K is split).  The outputs must not overlap
 * one another or any input.  The workspace is sized by
 * tern_grouped_workspace_bytes (0 for invalid shapes) and follows the rules
 * of tern_linear. */
#define TERN_MAX_GROUP 8
size_t tern_grouped_workspace_bytes(int64_t M, int count, const int64_t* Ns, const int64_t* Ks);

tern_status tern_linear_grouped(int x_type, int64_t M, int count, const void* const* d_Xs,
                                const int64_t* ldxs, const void* const* d_tiled, const int64_t* Ns,
                                const int64_t* Ks, void* const* d_Ys, const int64_t* ldys, int out_type,
                                void* d_ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Fused gate+up projection with SwiGLU ([EMB] §2.2: gate and up are one
 * fused tensor cut by offsets):
 *   h[m, i] = silu(gate[m, i]) * up[m, i],  silu(g) = g / (1 + exp(-g)),
 * with gate and up each the linear layer above over their I rows.
 *
 * GLU tile layout: the tiled layout of a 2*ceil(I/16)*16-row weight whose
 * row n is gate row 16*(n/32) + n%32 when n%32 < 16 and up row
 * 16*(n/32) + n%32 - 16 otherwise (blocks of 16 rows alternating; rows
 * past I are zero).  Paired rows then meet in one warp of the epilogue.
 * ---------------------------------------------------------------------- */

/* Bytes of the GLU tile layout: tern_tiled_bytes(2*ceil(I/16)*16, K). */
size_t tern_tiled_glu_bytes(int64_t I, int64_t K);

/* (gate, up) on-disk pairs -> GLU tile layout.  Each of the two sources is
 * an on-disk pair as for tern_repack with I rows; a fused [2I, K/4] tensor
 * passes d_packed_up = d_packed_gate + I*K/4 (and likewise the scales).
 * Alignments, errors and d_err as tern_repack. */
tern_status tern_repack_glu(const uint8_t* d_packed_gate, const uint16_t* d_scales_gate,
                            const uint8_t* d_packed_up, const uint16_t* d_scales_up,
                            int64_t I, int64_t K, void* d_tiled, size_t tiled_bytes,
                            int32_t* d_err, void* stream);

/* Workspace bytes of tern_linear_swiglu. */
size_t tern_swiglu_workspace_bytes(int64_t M, int64_t I, int64_t K);

/* h = silu(X . gate^T) * (X . up^T) in one pass over the GLU tile layout.
 *   d_H  device [M, ldh] of out_type, ldh >= I.
 * gate and up are computed as by tern_linear (fp32, same error bound) and
 * combined in fp32 before the output conversion.  Other arguments as
 * tern_linear_ex. */
tern_status tern_linear_swiglu(const void* d_X, int x_type, int64_t ldx, const void* d_tiled_glu,
                               int64_t M, int64_t I, int64_t K, void* d_H, int64_t ldh,
                               int out_type, void* d_ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Zero-block skipping ([EMB] §6, outlook: skip blocks that are all zero
 * with a sparse mask).  A unit (128 rows x 128 weights of the tiled
 * layout) whose weights are all 0 contributes nothing: with its flag set
 * the linear kernels neither copy, decode nor multiply it.
 * ---------------------------------------------------------------------- */

/* Units of the tiled layout: ceil(N/128) * (K/128); unit (b, g) has index b*G + g. */
size_t tern_unit_count(int64_t N, int64_t K);

/* d_flags[u] (device uint8, tern_unit_count entries) = 1 if every weight of
 * unit u is 0, else 0.  Reads only the code units, so it serves the plain,
 * GLU and INT8-scale layouts alike. */
tern_status tern_zero_units(const void* d_tiled, int64_t N, int64_t K, uint8_t* d_flags, void* stream);

/* tern_linear_ex (plain tiled layout) skipping the units flagged in d_flags
 * (as written by tern_zero_units; a flag set on a unit that is not all
 * zero drops that unit's contribution). */
tern_status tern_linear_sparse(const void* d_X, int x_type, int64_t ldx, const void* d_tiled,
                               const uint8_t* d_flags, int64_t M, int64_t K, int n_out,
                               const int64_t* n_sizes, void* const* d_Ys, const int64_t* ldys,
                               int out_type, void* d_ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * INT8 group scales ([EMB] §6, outlook: compress the FP16 scales to INT8).
 * The page gives no format; this library's reading: one fp32 factor per
 * row and one int8 per group,
 *   s8[n, g] = q8[n, g] * f[n],   f[n] = max_g |s[n,g]| / 127,
 *   q8[n, g] = rint(s[n,g] * (127 / max_g |s[n,g]|))  (fp32, ties to even)
 * and the layer becomes Y = X . (s8 (.) T)^T with the same error bound.
 *
 * INT8-scale tile layout: the codes of the tiled layout (R*G units of 4096
 * bytes), then per unit (b, g) the 128 int8 q8[128b + r][g] (r = 0..127),
 * then per row tile b the 128 fp32 factors f[128b + r] (0 for padding).
 * ---------------------------------------------------------------------- */

/* Bytes of the INT8-scale layout: ceil(N/128) * (K/128) * 4224 + ceil(N/128) * 512. */
size_t tern_tiled_s8_bytes(int64_t N, int64_t K);

/* FP16 scales [N, K/128] -> d_q8 int8 [N, K/128] and d_f fp32 [N] (device).
 * A row of zero scales gives f = 0, q8 = 0. */
tern_status tern_quantize_scales(const uint16_t* d_scales, int64_t N, int64_t K, int8_t* d_q8,
                                 float* d_f, void* stream);

/* (packed [N, K/4], q8, f) -> INT8-scale tile layout; otherwise as tern_repack. */
tern_status tern_repack_s8(const uint8_t* d_packed, const int8_t* d_q8, const float* d_f,
                           int64_t N, int64_t K, void* d_tiled, size_t tiled_bytes,
                           int32_t* d_err, void* stream);

/* tern_linear_ex over INT8-scale weights (workspace: tern_workspace_bytes). */
tern_status tern_linear_s8(const void* d_X, int x_type, int64_t ldx, const void* d_tiled_s8,
                           int64_t M, int64_t K, int n_out, const int64_t* n_sizes,
                           void* const* d_Ys, const int64_t* ldys, int out_type,
                           void* d_ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * int8-activation variant ([EMB] §4.1-§4.3: the page's third route, signs
 * accumulated as integers inside each 128-wide group and the float scale
 * applied once at the group boundary).  The page does not define how the
 * activations become integers; this library quantises per token:
 *   a[m]    = max_k |x[m,k]| / 127                         (fp32)
 *   q[m,k]  = rint(x[m,k] * (127 / max_k |x[m,k]|))        (fp32, ties to
 *             even), within [-127, 127]; a zero row gives a = 0, q = 0
 *   Y[m,n]  = a[m] * sum_g s[n,g] * I[m,n,g],  I = sum_{k in g} t[n,k] q[m,k]
 * I is an exact int32.  The result satisfies
 * |Y - Y_exact| <= 1e-4 * sum_k |a[m] q[m,k] W[n,k]| per output.
 * ---------------------------------------------------------------------- */

/* Bytes of the quantised activations of M x K (tern_quantize_x output). */
size_t tern_xq_bytes(int64_t M, int64_t K);

/* X (bf16 or fp16 bits, [M, ldx], 2-byte aligned) -> d_xq (device,
 * tern_xq_bytes(M, K) bytes, 16-byte aligned: q in this library's order,
 * within each row and each run of 16 weights k0..k0+15 first the even
 * then the odd k) and d_a (device fp32 [M]).  K a positive multiple of 128. */
tern_status tern_quantize_x(const void* d_X, int x_type, int64_t ldx, int64_t M, int64_t K,
                            void* d_xq, float* d_a, void* stream);

/* Workspace bytes of tern_linear_i8 (256-byte aligned, zero-filled before
 * first use; its first word is the error word as for tern_linear). */
size_t tern_i8_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* Y = the int8-activation layer above, from tern_quantize_x's (d_xq, d_a)
 * and the tiled weights; d_Y [M, ldy] of out_type.  Deterministic. */
tern_status tern_linear_i8(const void* d_xq, const float* d_a, const void* d_tiled, int64_t M,
                           int64_t N, int64_t K, void* d_Y, int64_t ldy, int out_type,
                           void* d_ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Workspace maintenance (library conveniences; the pages have none).
 * ---------------------------------------------------------------------- */

/* Copy the workspace's error word to *h_err (host) and wait for `stream`
 * to reach that point -- the one call in this header that synchronises
 * (the stream only).  Non-zero: a call that used the workspace gave up
 * after a pipeline wait timed out; its outputs are incomplete. */
tern_status tern_workspace_error(const void* d_ws, int32_t* h_err, void* stream);

/* Zero ws_bytes of the workspace on `stream` (the state a workspace must be
 * in before its first use, and again after an error). */
tern_status tern_workspace_reset(void* d_ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TERN_H */
