/*
 * qlin -- skinny W4A8 / W6A8 quantized linear for GB300 (sm_103a).
 *
 *   y[M, N] = s_m * sum_g sw[n, g] * sum_{k in group g} q[m, k] * level[n, k]
 *
 * for M = 1..8 rows (one decoded token plus up to seven multi-token-prediction
 * drafts), with level = code - 2^(b-1) from b = 4 or 6 bit weight codes, fp32
 * group scales sw, and q = per-row int8 quantisation of the activation, which
 * is x itself, RMSNorm(x) or silu(gate) * up.
 *
 * Sources (page title, section):
 *  [LIN]  "Doubling the LLM token rate in ComfyUI", section "Optimising the
 *         linear kernel": skinny GEMV for M = 1 and thin MTP verification M;
 *         weights and per-group scales interleaved in the order the kernel
 *         reads them, rearranged once per model load in place in VRAM; the M
 *         rows mapped onto the 8-wide side of a tensor-core MMA so that up to
 *         eight rows cost about what one row costs; the activation
 *         quantisation absorbs the RMSNorm or SwiGLU in front of it.
 *  [BOT]  same page, section "What is the bottleneck?": every token reads
 *         every weight once, so decode speed is VRAM read speed.
 *  [MTP]  same page, section "Adaptive-tree MTP": verification carries at
 *         most eight rows (one committed token plus seven drafts).
 *  [FMT]  "Comfy Quantization Formats", section "Weight formats": N output
 *         width, K input width, G group size, FP32 scales.
 *  [OPT]  same page, section "Format options": asym_w4a8_int8 (uniform levels
 *         without a codebook) and w6a8_int8; symmetric weights; grouped W4A8
 *         needs K % 16 == 0, K % G == 0, G >= 4 and (16 % G == 0 or
 *         G % 16 == 0); W6A8 needs K % 32 == 0 and G % 16 == 0; backends may
 *         restrict shapes further.
 *  [ACT]  same page, section "Activations and smoothing": integer formats take
 *         float activations and quantise them inside the kernel; no stored
 *         input scale.
 *
 * Conventions for every entry point:
 *  - All buffer pointers are DEVICE pointers owned by the caller; the library
 *    never allocates, frees or synchronises (except qlin_read_device_status).
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream) on the current device.
 *  - Argument and shape errors are returned before anything is enqueued.
 *    Launch failures return QLIN_ERR_CUDA.  A device-side bounded wait that
 *    expires writes QLIN_ERR_DEVICE_TIMEOUT into the workspace status word,
 *    read back by qlin_read_device_status; the kernel returns instead of
 *    hanging.
 *  - fmt is QLIN_W4A8 or QLIN_W6A8; b = 4 or 6 bits per code.
 *  - Backend limits beyond [OPT] (QLIN_ERR_UNSUPPORTED): G in {4, 8, 16, 32,
 *    64, 128, 256} (4 and 8 for 4-bit codes, as the format allows),
 *    K % 32 == 0, N % 16 == 0, K <= 65536 (K <= 57344 for G = 4, whose
 *    per-group start values fill the shared memory of 16 CTAs first), M <= 8.
 */
#ifndef QLIN_H_
#define QLIN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QLIN_OK = 0,
  QLIN_ERR_INVALID_ARG = 1,    /* bad pointer, alignment, size, or a shape [OPT] forbids */
  QLIN_ERR_UNSUPPORTED = 2,    /* legal per [OPT] but outside this backend's limits */
  QLIN_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed */
  QLIN_ERR_DEVICE_TIMEOUT = 4, /* a device-side bounded wait expired (status word) */
  QLIN_ERR_WORKSPACE = 5       /* workspace smaller than the size query returned */
} qlin_status;

typedef enum { QLIN_W4A8 = 0, QLIN_W6A8 = 1 } qlin_format;

typedef enum {
  QLIN_PROLOGUE_NONE = 0,    /* a = x */
  QLIN_PROLOGUE_RMSNORM = 1, /* a = x * gamma / sqrt(mean(x^2) + eps) */
  QLIN_PROLOGUE_SWIGLU = 2   /* a = gate / (1 + exp(-gate)) * up */
} qlin_prologue;

/* qlin_forward flags. */
#define QLIN_FLAG_PDL 1u /* Launch with programmatic dependent launch: the kernel may start
                            streaming `packed` and reading `gamma` while earlier kernels in
                            `stream` still run.  The caller asserts that neither was written
                            by any kernel still in flight in `stream` (true for model
                            weights repacked at load time and for norm weights).
                            Activations, y and the workspace are still touched only after
                            earlier kernels complete. */

/* Library version string. */
const char* qlin_version(void);

/* Human-readable name of a status code (static storage). */
const char* qlin_status_string(qlin_status s);

/* Validate a weight shape against [OPT] and the backend limits.  Host only.
 * Returns QLIN_OK, QLIN_ERR_INVALID_ARG or QLIN_ERR_UNSUPPORTED. */
qlin_status qlin_check_shape(int fmt, int64_t N, int64_t K, int64_t G);

/* Bytes of one quantized weight, in either layout: N*K*b/8 code bytes plus
 * N*(K/G)*4 scale bytes [FMT].  0 when qlin_check_shape fails. */
size_t qlin_packed_bytes(int fmt, int64_t N, int64_t K, int64_t G);

/*
 * In-place repack [LIN]: rewrites `buf` from the checkpoint layout into the
 * kernel-order stream that qlin_forward reads.  Same size in and out
 * (qlin_packed_bytes).  One call per weight, once per load; calling it twice
 * does not give the same bytes as calling it once.
 *
 * Checkpoint layout (input): codes, then scales.
 *   4-bit: uint8 [N, K/2], low nibble = even k.  6-bit: uint8 [N, 3K/4], each 3
 *   bytes a little-endian 24-bit word holding 4 codes, code i at bits 6i..6i+5.
 *   Scales: fp32 [N, K/G] row-major, little-endian, right after the codes.
 * Stream layout (output), KB = max(128, G):
 *   tiles of 128 output rows (the last may hold fewer, a multiple of 16), in
 *   order; inside a tile, units of KB input columns (the last may be
 *   narrower), in order; a unit of R rows and W columns is
 *     scale block  R*(W/G) fp32: for each group of the unit, for each 16-row
 *                  slab, for p = 0..7: sw[row p], sw[row p + 8];
 *     code block   for each slab, for each pair of 16-wide k-steps:
 *                  4-bit plane: 32 lanes x {word for step A, word for step B};
 *                  6-bit codes only, then the 2-bit plane: 32 lanes x 1 word.
 *   A lane (g, t) = (lane / 4, lane % 4) holds the A operand of a 16x16 fp16
 *   tensor-core tile: register i in 0..3 holds (row g, k 2t..2t+1),
 *   (row g+8, k 2t..2t+1), (row g, k 2t+8..2t+9), (row g+8, k 2t+8..2t+9).  In
 *   a 4-bit plane word, register i's two elements sit at bits 4i..4i+3 and
 *   16+4i..16+4i+3 (the low 4 bits of the code).  In the 2-bit plane word the
 *   top 2 bits of register i of step s (0 = A, 1 = B) sit at bits
 *   8s + 2*(i / 2) + 4*(i % 2) and 16 above that (odd k).  So a row-g field
 *   and its row-g+8 partner are 4 bits apart in both planes, and one shift of
 *   the 2-bit word lines a pair up with its nibbles.  Codes are stored
 *   unsigned (not offset).
 *
 * buf: device, 16-byte aligned, qlin_packed_bytes(fmt, N, K, G) bytes.
 * ws : device scratch, 256-byte aligned, at least *min_bytes from
 *      qlin_repack_workspace_bytes; larger means fewer, bigger copy waves.
 *      Strictly zero extra memory is not possible because codes and scales sit
 *      in separate regions of the input; the scratch holds all scales plus one
 *      wave of 128-row code tiles.
 */
qlin_status qlin_repack_workspace_bytes(int fmt, int64_t N, int64_t K, int64_t G,
                                        size_t* min_bytes, size_t* recommended_bytes);
qlin_status qlin_repack(int fmt, int64_t N, int64_t K, int64_t G, void* buf,
                        void* ws, size_t ws_bytes, void* stream);

/*
 * Forward workspace: one status word (plus reserved bytes) that a device-side
 * wait which expires sets to QLIN_ERR_DEVICE_TIMEOUT.  Zero it once with
 * qlin_workspace_init; one workspace may serve every call of a model.  The
 * forward keeps everything else (the quantised activations, the split-K
 * partial sums) in on-chip shared memory.
 */
/*
 * qlin_repack for a W4A8 weight whose levels come from a codebook
 * (qlin_forward_codebook): the same stream, except that in a 4-bit plane
 * word A-register i's two codes sit in byte i (even k at bits 8i..8i+3, odd
 * k at 8i+4..8i+7), so that one table lookup yields one register.  Same
 * arguments, sizes and errors as qlin_repack with fmt = QLIN_W4A8.  A buffer
 * repacked this way is for qlin_forward_codebook only.
 */
qlin_status qlin_repack_codebook(int64_t N, int64_t K, int64_t G, void* buf, void* ws, size_t ws_bytes,
                                 void* stream);

qlin_status qlin_forward_workspace_bytes(int fmt, int64_t N, int64_t K, int64_t G, size_t* bytes);
qlin_status qlin_workspace_init(void* ws, size_t ws_bytes, void* stream);

/*
 * y = packed-weight x quantised activation [LIN], [ACT], [MTP].
 *   fmt, prologue : qlin_format, qlin_prologue.
 *   M             : rows, 1..8 (M = 0 or N = 0 enqueues nothing; with M = 0
 *                   the activation and output pointers are not read and may
 *                   be null).
 *   packed        : device, repacked stream (qlin_repack), 16-byte aligned.
 *   x             : bf16 [M, K] row-major, 16-byte aligned (NONE, RMSNORM).
 *   gate, up      : bf16 [M, K] row-major, 16-byte aligned (SWIGLU).
 *   gamma         : fp32 [K], 16-byte aligned (RMSNORM); eps >= 0 (RMSNORM).
 *   y             : fp32 [M, N] row-major, 4-byte aligned; fully overwritten.
 *   ws, ws_bytes  : forward workspace (see above), 256-byte aligned.
 *   flags         : 0 or QLIN_FLAG_PDL.
 * Numerics: the prologue and the scale s_m = amax/127 are computed in fp32,
 * q = clamp(round-half-even(a / s_m), -127, 127) (s_m = 0, q = 0 for an
 * all-zero row; with no prologue a / s_m is the IEEE fp32 quotient, with a
 * prologue a * c, c = rstd * 127 / amax from fast fp32 reciprocals, which the
 * method's tolerance allows); group sums are exact integers; y is accumulated
 * in fp32 in a fixed order that depends on (N, K, G) and the device, never on
 * M or on the other rows, so row m of an 8-row call equals the same row run
 * alone: the split of K over the CTAs of a cluster is planned for 8 rows
 * whatever M is, and M changes only how deep the weight ring is.  One kernel
 * is enqueued: a cluster of CTAs per 256 output rows
 * splits K, computes the prologue and the row statistics in shared memory,
 * streams the weights through the tensor cores and reduces its split-K
 * partial sums through distributed shared memory.
 */
qlin_status qlin_forward(int fmt, int prologue, int M, int64_t N, int64_t K, int64_t G,
                         const void* packed, const void* x, const void* gate, const void* up,
                         const float* gamma, float eps, float* y,
                         void* ws, size_t ws_bytes, unsigned flags, void* stream);

/*
 * Several weights that read the same activation, in one launch [LIN], [ACT]:
 * y[l] = packed[l] x quantised activation for l = 0..n-1, e.g. the q, k and v
 * projections after one RMSNorm, or gate and up.  The prologue and the
 * activation quantisation are computed for the shared input only; fusing the
 * steps that share an input follows "Doubling the LLM token rate in
 * ComfyUI", section "Optimising the linear kernel" (the prologue is absorbed
 * into the quantisation and the launches between them disappear).
 *   n             : 1..QLIN_MAX_MULTI weights.
 *   N             : host array [n] of output rows (each N[l] obeys the rules
 *                   of qlin_forward; N[l] = 0 skips weight l).
 *   packed        : host array [n] of device pointers, each a repacked stream
 *                   of shape (N[l], K, G), 16-byte aligned.
 *   y             : host array [n] of device pointers, fp32 [M, N[l]]
 *                   row-major, 4-byte aligned; fully overwritten.
 *   bias          : NULL, or a host array [n] of device pointers (each NULL or
 *                   fp32 [N[l]], 4-byte aligned): y[l][m][n] gets bias[l][n]
 *                   added once, unscaled ("Comfy Quantization Formats",
 *                   sections "Checkpoint layout" and "Activations and
 *                   smoothing": a layer's bias stays floating point).
 *   All other arguments, the numerics and the errors are those of
 *   qlin_forward; the host arrays are read during the call only.  Each y[l]
 *   equals qlin_forward on weight l within the output tolerance; the
 *   split-K order may differ because the cluster size is chosen for the
 *   whole launch.
 */
#define QLIN_MAX_MULTI 8

/*
 * Expert bank (MoE) [MOE]: y[m][j][:] = expert ids[m][j] applied to the
 * quantised activation of token m.  "Comfy Quantization Formats", section
 * "Embeddings and MoE": a grouped W4A8 / W6A8 bank stores its experts with
 * the expert and output rows flattened to E * N, and an optional [E, N] bias.
 *   bank   : device, the bank repacked as one weight of E * N rows
 *            (qlin_repack with N = E * N), 16-byte aligned.
 *   E, N   : experts (1..4096) and rows per expert (a multiple of 128 here,
 *            so that every expert starts on a stream tile).  G >= 32 here.
 *   ids    : device int32 [M, topk], topk in 1..8: the expert of each token
 *            and slot.  It may be written by the previous kernel in the
 *            stream: it is read after the dependency wait.  An id outside
 *            [0, E) routes nowhere and its output row is not written; a token
 *            may name one expert in several slots.
 *   bias   : device fp32 [E, N], or NULL.
 *   y      : device fp32 [M, topk, N] row-major; every routed (m, j) row is
 *            fully overwritten.  No routing weights are applied.
 *   Other arguments, numerics and errors as qlin_forward.  One launch is
 *   sized for min(E, M * topk) experts; the experts actually routed take its
 *   row blocks in increasing id order, the remaining blocks return at once.
 *   The split of K is planned for min(E, 8 * topk) experts, so for a given
 *   bank (E, N, K, G) and topk, token m's output does not depend on M or on
 *   the other tokens' routing.
 *   Under QLIN_FLAG_PDL the weights are not streamed before the previous
 *   kernel completes (the routing decides which weights).
 */
#define QLIN_MOE_MAX_E 4096
#define QLIN_MOE_MAX_TOPK 8
qlin_status qlin_forward_moe(int fmt, int prologue, int M, int E, int64_t N, int64_t K, int64_t G, const void* bank,
                             const int32_t* ids, int topk, const void* x, const void* gate, const void* up,
                             const float* gamma, float eps, const float* bias, float* y, void* ws, size_t ws_bytes,
                             unsigned flags, void* stream);
/*
 * 4-bit codes with a codebook [FMT]: "Comfy Quantization Formats", section
 * "Format options" -- a W4A8 weight may carry a float [16] codebook that
 * replaces the uniform levels (code - 8); W6A8 has none.  Here the level of
 * code c is codebook[c], scaled per group by the weight scale as usual:
 *   y[m][n] = s_m * sum_g sw[n][g] * sum_{k in g} q[m][k] * codebook[code[n][k]]
 *             (+ bias[n]).
 *   fmt      : QLIN_W4A8 only (else QLIN_ERR_INVALID_ARG); G >= 32 here.
 *   packed   : the stream written by qlin_repack_codebook (the codebook
 *              layout of the 4-bit plane), 16-byte aligned.
 *   codebook : device fp32 [16], 4-byte aligned.  It is read like `packed`
 *              (before the dependency wait under QLIN_FLAG_PDL).
 *   bias     : device fp32 [N], or NULL.
 *   Other arguments, numerics and errors as qlin_forward, except that the
 *   group sums are not exact integers: the table is scaled by the power of
 *   two that puts its largest magnitude in [2^14, 2^15) and rounded to fp16
 *   (11 significant bits, relative error <= 2^-12 per level), products and
 *   sums in fp32, the power of two removed exactly afterwards.
 */
qlin_status qlin_forward_codebook(int fmt, int prologue, int M, int64_t N, int64_t K, int64_t G, const void* packed,
                                  const float* codebook, const void* x, const void* gate, const void* up,
                                  const float* gamma, float eps, const float* bias, float* y, void* ws,
                                  size_t ws_bytes, unsigned flags, void* stream);
qlin_status qlin_forward_multi(int fmt, int prologue, int M, int n, const int64_t* N, int64_t K, int64_t G,
                               const void* const* packed, const void* x, const void* gate, const void* up,
                               const float* gamma, float eps, float* const* y, const float* const* bias, void* ws,
                               size_t ws_bytes, unsigned flags, void* stream);

/* Launch shape of qlin_forward's GEMV on the current device: CTAs, stream
 * units (128 rows x KB columns) and bytes of `packed` read per call.  The
 * CTAs are the same for every M (the split of K does not depend on M). */
qlin_status qlin_forward_launch_info(int fmt, int64_t N, int64_t K, int64_t G,
                                     int64_t* ctas, int64_t* units, int64_t* stream_bytes);

/* Synchronises `stream`, then returns the workspace status word (QLIN_OK when
 * no device-side wait has expired since qlin_workspace_init).  For tests. */
qlin_status qlin_read_device_status(const void* ws, void* stream);

/*
 * Test export: qlin_forward with extra outputs (device pointers, each may be
 * NULL): y fp32 [M, N]; acc int32 [M, N, K/G], the exact per-group integer
 * sums sum_k q[m,k] * level[n,k]; q int8 [M, K], the activation codes; s fp32
 * [M], the row scales.  It runs a build of the forward kernel that carries
 * these exports (the production kernels do not), with the same arithmetic:
 * its y equals qlin_forward's bit for bit.
 */
qlin_status qlin_debug_forward(int fmt, int prologue, int M, int64_t N, int64_t K, int64_t G,
                               const void* packed, const void* x, const void* gate, const void* up,
                               const float* gamma, float eps, float* y, int32_t* acc, int8_t* q, float* s,
                               void* ws, size_t ws_bytes, void* stream);

/*
 * Test export for failure detection: qlin_forward, except that the first CTA
 * of the launch never issues the weight copy of its local unit `unit` (0 is
 * its first unit and always exists).  Its consumers' bounded wait on that
 * unit expires after about a second; the kernel writes
 * QLIN_ERR_DEVICE_TIMEOUT into the workspace status word, waits (bounded) for
 * the copies it did issue, and returns, leaving the context usable.  y is
 * unspecified afterwards.  Nothing faults.
 */
qlin_status qlin_debug_forward_fault(int fmt, int prologue, int M, int64_t N, int64_t K, int64_t G,
                                     const void* packed, const void* x, const void* gate, const void* up,
                                     const float* gamma, float eps, float* y, void* ws, size_t ws_bytes,
                                     int64_t unit, void* stream);

/*
 * Test export: the plan qlin_forward uses on the current device for a weight
 * of N rows, K columns and group size G at M rows: *cluster = CTAs that split
 * K for one 256-row block (the same for every M), *stages = ring stages per
 * CTA (more for fewer rows, whose activation operand is smaller).
 */
qlin_status qlin_debug_plan(int fmt, int M, int64_t N, int64_t K, int64_t G, int* cluster, int* stages);

/*
 * Test exports of the second main loop, on the 5th-generation tensor cores
 * (tcgen05.mma with the fp16 weight operand in tensor memory, accumulators in
 * tensor memory), kept to measure it against qlin_forward's warp-level MMA
 * loop; it computes the same results ("Doubling the LLM token rate in
 * ComfyUI", section "Optimising the linear kernel": the M <= 8 activation
 * rows on the narrow side of the tensor-core product).  It is slower on this
 * path: every 4-bit code is unpacked on the CUDA cores either way, and the
 * tensor-memory stores, the hand-offs between warps and the MMA issue (one
 * 128 x 16 step per instruction) cost more than the warp-level MMAs they
 * replace.
 *
 * qlin_debug_repack_tcgen05: qlin_repack into the row layout this loop reads
 *   (G >= 32): per unit of R rows and W columns,
 *     scale block  R*(W/G) fp32, [group][row];
 *     4-bit plane  for each 32-wide k chunk c, for each row: 4 words, word j
 *                  holding the low 4 bits of the codes of k = 32c + 8j + i at
 *                  bits 4i (i = 0..7);
 *     6-bit codes only, then the 2-bit plane: for each chunk, for each row: 2
 *                  words; word h holds the top 2 bits of the codes of words
 *                  2h (at offset 0) and 2h+1 (at offset 2), code i of a word
 *                  at bit P(i) + offset, P = (4, 8, 0, 12, 20, 24, 16, 28).
 *   Arguments and errors as qlin_repack; QLIN_ERR_UNSUPPORTED for G < 32.
 * qlin_debug_forward_tcgen05: qlin_debug_forward on a weight repacked by
 *   qlin_debug_repack_tcgen05 (y required; acc, q, s may be NULL), with
 *   qlin_forward's flags.  Its split of K is planned for its own shared-memory
 *   operand, so y may differ from qlin_forward's in the last bits (the order
 *   of the fp32 partial sums); the group sums are the same exact integers.
 */
qlin_status qlin_debug_repack_tcgen05(int fmt, int64_t N, int64_t K, int64_t G, void* buf, void* ws,
                                      size_t ws_bytes, void* stream);
qlin_status qlin_debug_forward_tcgen05(int fmt, int prologue, int M, int64_t N, int64_t K, int64_t G,
                                       const void* packed, const void* x, const void* gate, const void* up,
                                       const float* gamma, float eps, float* y, int32_t* acc, int8_t* q, float* s,
                                       void* ws, size_t ws_bytes, unsigned flags, void* stream);

/*
 * qlin_forward without a caller workspace.  The method has no counterpart: this
 * is for callers that cannot allocate device memory where they run the layer
 * (a host whose memory pool owns the whole device and forbids cudaMalloc, code
 * that must avoid cudaMalloc's implicit synchronisation, a fixed-footprint
 * deployment).  The call allocates nothing; it uses a 64 KiB device array
 * inside the library instead, which every GPU that loads the library holds
 * until the process exits.
 *  - Arguments are those of qlin_forward without ws/ws_bytes.
 *  - Returns QLIN_ERR_WORKSPACE when the shape's workspace
 *    (qlin_forward_workspace_bytes) exceeds 64 KiB; nothing is enqueued then.
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any CUDA
 *    stream capture.
 *  - All calls share the one array, which keeps the previous call's contents.
 *    The forward kernel keeps nothing there that must start at zero: the
 *    array holds only the status word, written only when a wait expires.
 *    Calls that overlap on the GPU (different streams, or unordered work)
 *    race on it: order them on one stream.
 *  - A device-side wait that expires is recorded in the array's status word,
 *    which this entry point does not read back; the kernel still returns
 *    instead of hanging.
 */
qlin_status qlin_forward_noalloc(int fmt, int prologue, int M, int64_t N, int64_t K, int64_t G,
                                 const void* packed, const void* x, const void* gate, const void* up,
                                 const float* gamma, float eps, float* y, unsigned flags, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* QLIN_H_ */
