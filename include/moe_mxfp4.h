/*
 * moe_mxfp4.h — C ABI of a GB300 (sm_103a) mixture-of-experts layer with
 * MXFP4 expert weights, for decode (T = 1 .. 64 tokens) and prefill.
 *
 * What is computed (page "3 ways to speed up MoE inference on NVIDIA DGX
 * Spark", §2: every MoE layer sends each token to 8 of 512 routed experts plus
 * one shared expert; §3: moe_intermediate_size 768; §1: at batch 1, decode is
 * bound by reading weights). Per token t with activations x (bf16, width d):
 *
 *   l[e]   = sum_j x[j] * Wr[e][j]                      router logits (fp32)
 *   key[e] = l[e] + bias[e]                             fp32 add; bias optional
 *   S      = the k experts with the largest key; equal keys -> lower index
 *   w[j]   = exp(key[S_j] - key[S_0]) / sum_i exp(key[S_i] - key[S_0])
 *   h_e    = silu(Wg_e x) * (Wu_e x)                    SwiGLU, fp32
 *   y      = sum_j w[j] * Wd_{S_j} h_{S_j}  +  Wd_sh (silu(Wg_sh x) * (Wu_sh x))
 *
 * Routed experts are stored in MXFP4 (OCP Microscaling v1.0): E2M1 codes
 * (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6, sign bit), one E8M0 scale
 * 2^(s-127) per 32 consecutive elements along K. Router and shared expert
 * are bf16. Accumulation is fp32; y is bf16.
 *
 * Conventions for every entry point
 *   - Pointers ending in a device buffer are device pointers owned by the
 *     caller; the library allocates no device memory. The one piece of
 *     mutable global state is the fixed scratch array behind
 *     moe_forward_static_scratch. Host pointers are marked "host".
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream). Nothing synchronises the host.
 *   - Return value: MOE_OK (0) or a negative moe_status. Arguments are
 *     checked before anything is enqueued; on error nothing is enqueued.
 *   - Conditions only a kernel can see are OR-ed into *dev_status (a device
 *     int the caller zeroes and reads after synchronising), as moe_dev_status
 *     bits. dev_status may be NULL where noted.
 *   - There is no CPU fallback and no alternate backend: an unsupported
 *     shape is an error, never a silent slow path.
 *   - Calls are reentrant; concurrent calls must not share output or
 *     workspace buffers.
 */
#ifndef MOE_MXFP4_H
#define MOE_MXFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* == cudaStream_t */

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,        /* null pointer, negative size, bad enum */
  MOE_ERR_UNSUPPORTED_SHAPE = -2,  /* e.g. K % 32 != 0, N % 16 != 0, k > E */
  MOE_ERR_BAD_DESCRIPTOR = -3,     /* packed-weight descriptor does not match */
  MOE_ERR_WORKSPACE_TOO_SMALL = -4,
  MOE_ERR_BUFFER_TOO_SMALL = -5,   /* packed buffer smaller than required */
  MOE_ERR_CUDA = -6,               /* a CUDA runtime call failed */
  MOE_ERR_NO_DEVICE = -7           /* current device is not sm_103 */
} moe_status;

/* Bits OR-ed into *dev_status by kernels. */
typedef enum moe_dev_status {
  MOE_DEV_NONFINITE_INPUT = 1,  /* pack: a block held inf/NaN (its scale byte is 255) */
  MOE_DEV_SCALE_RANGE = 2,      /* pack: a scale byte above 248 (|w| >= 2^122); the
                                   expert kernels cannot represent it */
  MOE_DEV_INDEX_OOB = 4,        /* a routing index outside [0, E) reached a kernel */
  MOE_DEV_TIMEOUT = 8           /* a bounded wait in a kernel gave up */
} moe_dev_status;

/* Packed layouts (byte formats of moe_pack_mxfp4's output).
 *
 * MOE_LAYOUT_TILE16: matrix W [N][K] (N % 16 == 0, K % 32 == 0) is cut into
 *   row tiles of 16 rows. For tile r (rows 16r..16r+15) and K-block b
 *   (columns 32b..32b+31) a 272-byte unit sits at byte (r*K/32 + b) * 272:
 *     bytes [0, 256): the 512 E2M1 codes, row-major: bytes [16i, 16i+16)
 *       hold row 16r+i, columns 32b..32b+31, column 32b+2j in the low nibble
 *       of byte j and 32b+2j+1 in its high nibble (the canonical MXFP4 byte
 *       order). Each 8-byte half-row (16 codes) is the low half of one
 *       16-byte chunk of the tensor cores' E2M1 operand form, and the
 *       even/odd nibbles of a 4-byte word re-encode with two logic
 *       operations as E4M3 bytes worth 2^-6 times the E2M1 value.
 *     bytes [256, 272): scale bytes, row g at 256 + 2g, row g+8 at 257 + 2g
 *       (g = 0..7).
 *   A tile's units over all K are contiguous, and a matrix's tiles too.
 *   Bytes per matrix: N*K/2 + N*K/32 (exactly the MXFP4 payload).
 * MOE_LAYOUT_TILE16_GATEUP: the input matrix is a fused [2I][K] gate/up
 *   projection (rows 0..I-1 gate, I..2I-1 up, I % 8 == 0). Packed tile r
 *   holds gate rows 8r..8r+7 as its rows 0..7 and up rows 8r..8r+7 as its
 *   rows 8..15; otherwise as MOE_LAYOUT_TILE16.
 */
typedef enum moe_layout {
  MOE_LAYOUT_TILE16 = 1,
  MOE_LAYOUT_TILE16_GATEUP = 2
} moe_layout;

#define MOE_PACK_MAGIC 0x3446584Du /* "MXF4" */
#define MOE_PACK_VERSION 2u

/* Host-side descriptor of a packed weight buffer. moe_pack_mxfp4 fills it;
 * moe_forward refuses buffers whose descriptor does not match the layer
 * shape (MOE_ERR_BAD_DESCRIPTOR) instead of reinterpreting them. */
typedef struct moe_packed_desc {
  uint32_t magic;        /* MOE_PACK_MAGIC */
  uint32_t version;      /* MOE_PACK_VERSION */
  int32_t layout;        /* moe_layout */
  int32_t n_mat;         /* number of matrices (experts) */
  int32_t N, K;          /* rows, reduction length of each matrix */
  uint64_t bytes_per_mat;
  uint64_t total_bytes;
} moe_packed_desc;

typedef struct moe_shape {
  int32_t d_model;    /* d: hidden width (multiple of 256) */
  int32_t d_ff;       /* I: expert intermediate width (multiple of 32) */
  int32_t n_experts;  /* E: routed experts (1 .. 1024) */
  int32_t top_k;      /* k: experts per token (1 .. min(E, 32)) */
  int32_t has_shared; /* 1: one bf16 shared expert, 0: none */
} moe_shape;

/* A layer's weights (all device pointers, caller-owned, read-only). */
typedef struct moe_layer {
  moe_shape shape;
  const void* router_w;        /* bf16 [E][d] row-major */
  const void* gate_up;         /* packed, MOE_LAYOUT_TILE16_GATEUP, n_mat=E, N=2I, K=d */
  moe_packed_desc gate_up_desc;
  const void* down;            /* packed, MOE_LAYOUT_TILE16, n_mat=E, N=d, K=I */
  moe_packed_desc down_desc;
  const void* shared_gate;     /* bf16 [I][d]  (unused if has_shared == 0) */
  const void* shared_up;       /* bf16 [I][d] */
  const void* shared_down;     /* bf16 [d][I] */
} moe_layer;

/* Kernel paths moe_forward can take (moe_query_path). */
typedef enum moe_path {
  MOE_PATH_DECODE_MMA = 1,   /* T <= 4 where the single-launch kernel does not
                                apply (e.g. E > 512): per-stage kernels: router
                                GEMV, top-k + sort, MXFP4 expert GEMVs on e4m3
                                mma.sync, combine */
  MOE_PATH_DECODE_FUSED = 2, /* T <= 4: one cooperative persistent kernel per
                                call (router, top-k, shared and routed experts,
                                combine), one CTA per SM */
  MOE_PATH_PREFILL_TC = 3    /* T >= 5: per-stage kernels with the routed
                                experts as grouped GEMMs on block-scaled tcgen05
                                MMAs (MXFP4 weights as E4M3 codes with E8M0
                                scales, activations as E4M3 terms with E8M0
                                scales, fp32 accumulators in tensor memory) */
} moe_path;

/* ---- packing ------------------------------------------------------------ */

/* Bytes of a packed buffer for n_mat matrices [N][K] in `layout`; 0 if the
 * shape or layout is unsupported. */
size_t moe_packed_bytes(int n_mat, int N, int K, int layout);

/* Fill *out (host) with the descriptor of a packed buffer of that shape
 * (for buffers packed earlier and stored). */
int moe_describe_packed(int n_mat, int N, int K, int layout, moe_packed_desc* out);

/* Quantise fp32 weights to MXFP4 and write them in `layout`.
 * Source: page "3 ways to speed up MoE inference on NVIDIA DGX Spark", §2
 * (the routed experts of Ling-3.0-flash are served in MXFP4, the baseline
 * running FlashInfer's MXFP4 MoE kernel); the pages do not define the format,
 * so the element, scale and rounding rule are those of the OCP Microscaling
 * Formats (MX) v1.0 specification, §5 (E2M1 elements, E8M0 scale per 32) and
 * §6.3 (conversion). The call is an offline step, done once per weight set.
 *   w_dev       fp32 [n_mat][N][K] row-major (device)
 *   packed_dev  output, packed_bytes >= moe_packed_bytes(...) (device, 16-B aligned)
 *   desc_out    host, may be NULL
 *   dev_status  device int, may be NULL; MOE_DEV_NONFINITE_INPUT,
 *               MOE_DEV_SCALE_RANGE
 * Rule (OCP MX v1.0, §6.3): per 32-block, s = clamp(floor(log2 amax) - 2 +
 * 127, 0, 254) (amax = 0 -> 0); codes = RNE(v * 2^(127-s)) onto the E2M1
 * grid, ties to even mantissa, saturating at 6, sign kept (-0 -> code 8).
 * A block with inf/NaN gets scale 255, its non-finite elements code 0.
 * Errors: MOE_ERR_INVALID_ARG (null pointer, bad layout),
 * MOE_ERR_UNSUPPORTED_SHAPE (N % 16, K % 32), MOE_ERR_BUFFER_TOO_SMALL. */
int moe_pack_mxfp4(const float* w_dev, int n_mat, int N, int K, int layout,
                   void* packed_dev, size_t packed_bytes, moe_packed_desc* desc_out,
                   int* dev_status, moe_stream_t stream);

/* Inverse permutation of a packed buffer into the canonical MXFP4 layout
 * (test aid): codes [n_mat][N][K/2] (element 2j in the low nibble of byte j),
 * scales [n_mat][N][K/32], rows in the order of moe_pack_mxfp4's input. */
int moe_unpack_mxfp4(const void* packed_dev, const moe_packed_desc* desc,
                     uint8_t* codes_dev, uint8_t* scales_dev, moe_stream_t stream);

/* ---- routing ------------------------------------------------------------ */

/* Top-k selection and renormalised softmax weights from fp32 logits.
 * Source: page "3 ways to speed up MoE inference on NVIDIA DGX Spark", §2
 * (each MoE layer sends a token to 8 of its 512 routed experts) and page
 * "NVIDIA three-layer optimisation speeds up MoE inference on DGX Spark by
 * 42.5%", its background section on sparse activation (a gating network
 * scores every expert and only the top-k highest-scoring ones run). The
 * pages give neither the tie rule nor the weight normalisation; the reading
 * here is a softmax over the k selected keys, equal keys to the lower index.
 *   logits_dev      fp32 [T][E] (device)
 *   bias_dev        fp32, NULL for none; bias_row_stride 0: one row [E]
 *                   for all tokens, >= E: row t at bias_dev + t*stride
 *   idx_dev         int32 [T][k], slots in descending key order (device)
 *   w_dev           fp32 [T][k] (device)
 * Keys are logit + bias in fp32 (round-to-nearest-even); -0 ranks as +0, NaN
 * ranks as -inf; equal keys go to the lower expert index. E <= 1024, k <= 32.
 * Errors: MOE_ERR_INVALID_ARG (null pointer, T < 1, stride in (0, E)),
 * MOE_ERR_UNSUPPORTED_SHAPE (E > 1024, k > 32 or k > E). */
int moe_route_topk(const float* logits_dev, int T, int E, int k,
                   const float* bias_dev, int bias_row_stride,
                   int32_t* idx_dev, float* w_dev, moe_stream_t stream);

/* Group (token, slot) pairs by expert, stable in p = t*k + j (page "MoE-SpeQ
 * ...", §4.2: sort the verify tokens' expert assignments by expert id so each
 * expert runs once over all its tokens).
 *   idx_dev      int32 [T][k], values in [0, E)
 *   counts_dev   int32 [E]; offsets_dev int32 [E+1] (exclusive scan)
 *   perm_dev     int32 [T*k]: sorted position -> p;  inv_dev: p -> position
 *   active_dev   int32 [E]: the D experts with count > 0, ascending
 *   n_active_dev int32 [1]: D
 *   workspace    >= moe_sort_workspace_bytes(T, k, E) bytes (device)
 * An index outside [0, E) sets MOE_DEV_INDEX_OOB in dev_status (may be NULL);
 * that pair is left out of every list (its inv entry is -1 and offsets[E]
 * counts only the pairs kept). */
size_t moe_sort_workspace_bytes(int T, int k, int E);
int moe_sort_by_expert(const int32_t* idx_dev, int T, int k, int E,
                       int32_t* counts_dev, int32_t* offsets_dev, int32_t* perm_dev,
                       int32_t* inv_dev, int32_t* active_dev, int32_t* n_active_dev,
                       void* workspace_dev, size_t workspace_bytes, int* dev_status,
                       moe_stream_t stream);

/* ---- the layer ---------------------------------------------------------- */

/* Device workspace moe_forward needs for T tokens (256-B aligned base).
 * The first bytes hold synchronisation counters that carry over from one call
 * to the next: zero-fill a workspace once before its first moe_forward, and
 * do not share one workspace between calls that may run concurrently. After
 * a call that reported MOE_DEV_TIMEOUT, zero it again. */
size_t moe_workspace_bytes(const moe_shape* shape, int T);

/* Which moe_path moe_forward takes for this shape and T on the current
 * device; negative status if unsupported (MOE_ERR_NO_DEVICE without an
 * sm_103 device, since the choice depends on its SM count and shared memory). */
int moe_query_path(const moe_shape* shape, int T);

/* The layer over T tokens.
 * Source: page "3 ways to speed up MoE inference on NVIDIA DGX Spark", §1
 * (at batch 1, decode is bound by reading weights), §2 (8 of 512 routed
 * experts plus one shared expert per token), §3 (moe_intermediate_size 768)
 * and §5 (a 4-token verify window touches up to 32 distinct experts); the
 * per-token formula is the one at the top of this file.
 *   L             host struct with device weight pointers and descriptors
 *   x_dev         bf16 [T][d] (device, 16-B aligned);  y_dev bf16 [T][d]
 *                 (device; may not alias x)
 *   bias_dev      fp32 router bias as in moe_route_topk (NULL: none)
 *   logits_out    fp32 [T][E] router logits before bias (NULL: not returned)
 *   idx_out       int32 [T][k]; w_out fp32 [T][k] (NULL: not returned)
 *   workspace_dev >= moe_workspace_bytes(&L->shape, T) bytes (device, 256-B
 *                 aligned), zero-filled before its first use (see
 *                 moe_workspace_bytes)
 *   dev_status    device int (may be NULL)
 * Activations must satisfy |x| < 2^100 and expert outputs stay finite.
 * Errors (nothing enqueued): MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED_SHAPE,
 * MOE_ERR_BAD_DESCRIPTOR (a packed buffer's descriptor does not match the
 * shape: refused, never reinterpreted), MOE_ERR_WORKSPACE_TOO_SMALL,
 * MOE_ERR_NO_DEVICE; MOE_ERR_CUDA if a launch fails. */
int moe_forward(const moe_layer* L, const void* x_dev, int T, void* y_dev,
                const float* bias_dev, int bias_row_stride,
                float* logits_out, int32_t* idx_out, float* w_out,
                void* workspace_dev, size_t workspace_bytes, int* dev_status,
                moe_stream_t stream);

/* Profiling hook: moe_forward that also records caller-created CUDA events
 * at the boundaries of its stages, for per-stage timing. Same arguments and
 * result as moe_forward, plus
 *   stage_events  host array of n_stage_events cudaEvent_t handles: event 0
 *                 is recorded on `stream` before the first kernel and event i
 *                 after stage i (stages listed by moe_stage_names); extra
 *                 events are left untouched. Under stream capture the records
 *                 become external event nodes, so graph replays time them.
 * The kernels launched are exactly moe_forward's. */
int moe_forward_profiled(const moe_layer* L, const void* x_dev, int T, void* y_dev,
                         const float* bias_dev, int bias_row_stride,
                         float* logits_out, int32_t* idx_out, float* w_out,
                         void* workspace_dev, size_t workspace_bytes, int* dev_status,
                         void* const* stage_events, int n_stage_events,
                         moe_stream_t stream);

/* The layer with 8-bit activations (W4A8): before each routed-expert GEMM the
 * activations (x for gate/up, h for down) are quantised to MXFP8 - E4M3
 * elements with one E8M0 scale per 32, OCP MX v1.0 rule s = floor(log2 amax)
 * - 8 + 127, round to nearest even, saturate at 448 - and the GEMMs run on
 * block-scaled tcgen05 MMAs. Router and shared expert stay bf16.
 * Source: page "3 ways to speed up MoE inference on NVIDIA DGX Spark", §2
 * (the baseline runs the W4A8 configuration of the FlashInfer MXFP4 MoE
 * kernel). The pages do not define the 8-bit format; MXFP8 E4M3 is the reading.
 * Arguments, workspace and errors as moe_forward; any T >= 1 (the call always
 * takes the per-stage tcgen05 path, MOE_PATH_PREFILL_TC). */
int moe_forward_w4a8(const moe_layer* L, const void* x_dev, int T, void* y_dev,
                     const float* bias_dev, int bias_row_stride,
                     float* logits_out, int32_t* idx_out, float* w_out,
                     void* workspace_dev, size_t workspace_bytes, int* dev_status,
                     moe_stream_t stream);

/* Quantise activation rows to MXFP8, the operation moe_forward_w4a8 applies
 * to x and to h: per row and 32-element block, s = clamp(floor(log2 amax) - 8
 * + 127, 0, 254) (amax = 0 -> 0), elements RNE(v * 2^(127 - s)) to E4M3,
 * saturating at 448 (OCP MX v1.0, §6.3, with E4M3's emax 8).
 * Source: page "3 ways to speed up MoE inference on NVIDIA DGX Spark", §2
 * (W4A8: 8-bit activations against 4-bit weights).
 *   src_dev      bf16 (src_is_bf16 = 1) or fp32 (0) [rows][K] (device, 16-B aligned)
 *   codes_dev    uint8 [rows][K] E4M3 codes (device, 16-B aligned)
 *   scales_dev   uint8 [rows][K/32] E8M0 scale bytes (device)
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED_SHAPE (K % 32 != 0). */
int moe_quant_mxfp8(const void* src_dev, int src_is_bf16, int rows, int K, uint8_t* codes_dev,
                    uint8_t* scales_dev, moe_stream_t stream);

/* ---- FP8 LM head ------------------------------------------------------------ */

/* Quantise a bf16 LM head to FP8 once (online, at load time): per output row
 * v, s_v = fp32(amax_v / 448) (1 for a zero row) and codes = E4M3 round to
 * nearest even of fp32(w / s_v), saturating at 448.
 * Source: page "3 ways to speed up MoE inference on NVIDIA DGX Spark", §4 (the
 * BF16 LM head, 2,560 -> 157,184, is quantised to FP8 when it is built, which
 * halves the bytes each decode step reads); the pages do not give the FP8
 * recipe, and this per-row scale is the reading.
 *   w_dev       bf16 [V][d] (device)
 *   codes_dev   uint8 [V][d] E4M3 (device, 2-B aligned); scales_dev fp32 [V]
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED_SHAPE (d odd). */
int moe_lmhead_pack_fp8(const void* w_dev, int V, int d, uint8_t* codes_dev, float* scales_dev,
                        moe_stream_t stream);

/* logits[t][v] = s_v * sum_j x[t][j] * codes[v][j] for T <= 8 tokens; the
 * codes are read once from HBM, the activations enter exactly (bf16 split into
 * e4m3 terms), fp32 accumulation. Same source as moe_lmhead_pack_fp8.
 *   codes_dev, scales_dev  as written by moe_lmhead_pack_fp8 (device, 8-B aligned codes)
 *   x_dev       bf16 [T][d] (device, 16-B aligned)
 *   logits_dev  fp32 [T][V] (device); overwritten (zeroed on `stream` first)
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED_SHAPE (V % 16, d % 64, T > 8). */
int moe_lmhead_fp8(const uint8_t* codes_dev, const float* scales_dev, int V, int d, const void* x_dev, int T,
                   float* logits_dev, moe_stream_t stream);

/* Size in bytes of the scratch array inside the library that
 * moe_forward_static_scratch uses instead of a caller's workspace. */
#define MOE_STATIC_SCRATCH_BYTES (4u * 1024u * 1024u)

/* moe_forward for callers that cannot allocate device memory.
 *
 * Source: none. The paper has no counterpart to this call; it is a library
 * service, and the layer it computes is exactly moe_forward's.
 *
 * Who needs it: code that runs inside a host program whose memory manager
 * has already reserved the device memory (a further cudaMalloc fails, or
 * escapes that manager's accounting), and latency-critical loops that cannot
 * afford the device-wide synchronisation cudaMalloc and cudaFree may cause.
 * Such callers have no way to provide moe_forward's workspace.
 *
 * Instead of a workspace this call uses a MOE_STATIC_SCRATCH_BYTES array that
 * is part of the library's device image (one per device). It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 * Arguments are those of moe_forward without the workspace. Every check of
 * moe_forward is made before anything is enqueued: a call that returns an
 * error has enqueued nothing.
 *
 *   - Set-up: the first call on each device, with that device current, looks
 *     up the array's device address (cudaGetSymbolAddress) and keeps it.
 *     Make that first call before any stream capture begins on the device.
 *   - Each call first clears, on `stream`, the counters at the head of the
 *     array that must read zero when its kernels start. No earlier call has to
 *     have finished cleanly.
 *   - All calls on one device share the array. Calls that can overlap in
 *     time (on different streams, or from host threads with no ordering
 *     between them) race on it and corrupt each other's results: put them on
 *     one stream or order them with events.
 *   - Returns MOE_ERR_WORKSPACE_TOO_SMALL, with nothing enqueued, when
 *     moe_workspace_bytes(&L->shape, T) > MOE_STATIC_SCRATCH_BYTES (at
 *     d = 2560, I = 768, E = 512, k = 8 that is T > 26). Larger calls need
 *     moe_forward with a workspace of their own. */
int moe_forward_static_scratch(const moe_layer* L, const void* x_dev, int T, void* y_dev,
                               const float* bias_dev, int bias_row_stride,
                               float* logits_out, int32_t* idx_out, float* w_out,
                               int* dev_status, moe_stream_t stream);

/* Comma-separated names of the stages of `path` in launch order (the
 * boundaries moe_forward's stage_events mark); NULL for an unknown path. */
const char* moe_stage_names(int path);

/* Failure-detection self-test: one GPU thread waits for *flag_dev == want with
 * the bounded spin the kernels use for every cross-CTA wait (acquire loads,
 * clock64 budget of budget_cycles, at most the kernels' own budget). If the
 * flag never takes that value, MOE_DEV_TIMEOUT is OR-ed into *dev_status and
 * the kernel returns; nothing hangs or faults. flag_dev: device uint32. */
int moe_selftest_bounded_wait(const uint32_t* flag_dev, uint32_t want, long long budget_cycles,
                              int* dev_status, moe_stream_t stream);

/* Static text for a moe_status value. */
const char* moe_status_string(int status);

/* Library version, e.g. "moe_mxfp4 1.2 sm_103a". */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_MXFP4_H */
