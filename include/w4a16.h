/*
 * w4a16.h -- C ABI of the GB300 (sm_103a) group-wise INT4 weight-only linear
 * layer library (W4A16).
 *
 * The operation (forum.sourcefind.cn thread "vLLM on Hygon Z100", section 四
 * "W4A16"; haowenji.com V100 decode article, paragraph on "groupwise-int"):
 * weights are 4-bit integers q with one fp16 scale s and one 4-bit zero z per
 * group of 128 consecutive inputs; the layer restores w = (q - z) * s and
 * multiplies it with fp16 activations, accumulating in fp32:
 *
 *     y[m, n] = sum_k x[m, k] * (q[n, k] - z[n, k / 128]) * s[n, k / 128]
 *
 * for m < M (tokens: 1 for plain decode, 4..8 for a speculative verify pass of
 * 1 + 3 .. 1 + 7 tokens that reads the weights once; section 五 of the same
 * thread, "M = 2, 4, 8"), n < N (outputs) and k < K (inputs).
 *
 * Data layout (all row-major, all little-endian):
 *   x       [M, K]            fp16 (passed as uint16_t bit patterns)
 *   qweight [N, K/8]          uint32; element k of row n is bits
 *                             4*(k%8) .. 4*(k%8)+3 of word k/8 (the thread's
 *                             "[N,K/8] int32" packed INT4 layout, section 四;
 *                             the nibble order within a word is this library's
 *                             reading: the pages do not state one)
 *   scales  [N, K/128]        fp16
 *   zeros   [N, ceil(G/8)]    uint32, G = K/128; group g of row n is nibble
 *                             g%8 of word g/8; nibbles past G are ignored
 *   y       [M, N]            fp16, fully overwritten, round-to-nearest-even
 *
 * Conventions shared by every entry point:
 *   - Pointers are DEVICE pointers unless a parameter says "host".  The caller
 *     owns every buffer; the library never frees or keeps caller pointers past
 *     the call (a captured graph keeps them, see w4a16_round_graph_create).
 *   - One exception: the output y of w4a16_linear, w4a16_linear_noalloc,
 *     w4a16_linear_epilogue, w4a16_linear_ex and of a decode round's
 *     descriptors may be page-locked host memory that the device addresses at
 *     the same pointer (cudaHostAlloc / cudaMallocHost, on a system with
 *     unified addressing).  The kernels then store y straight into host memory
 *     (on a Grace-Blackwell part, over the NVLink-C2C link), and the result is
 *     on the host once the stream has passed the call: no copy back.  Every
 *     other pointer stays device memory, so such a y can be neither a residual
 *     nor another linear's x.  The library does not inspect pointer kinds: a
 *     host y that the device cannot address faults like any bad pointer.
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *     default stream.  Work is enqueued asynchronously; nothing synchronises.
 *   - Arguments are validated on the host before anything is enqueued.  A
 *     nonzero status means nothing was launched.  A device fault inside a
 *     kernel surfaces, as usual for CUDA, at the caller's next synchronisation.
 *   - group must be 128 (W4A16_ERR_UNSUPPORTED otherwise); K must be a
 *     positive multiple of 128, at most 2^22; 1 <= N < 2^31; 1 <= M <= 65535.
 *   - x, qweight and y must be 16-byte aligned, scales 2-byte, zeros 4-byte
 *     (W4A16_ERR_MISALIGNED).  x and y must not overlap (INVALID_ARG).
 *   - w4a16_linear and w4a16_decode_round allocate nothing, free nothing and
 *     never synchronise the device, so they may be captured into a CUDA graph.  They need
 *     w4a16_init first (the split-K workspace and the kernel attributes).
 *   - The split-K workspace is shared by every call: calls that may use it must
 *     be ordered on one stream (or otherwise serialised).  Two such calls that
 *     overlap on the GPU race on it.
 *
 * Functions return an int status (w4a16_status) unless stated otherwise.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4A16_OK = 0,
    W4A16_ERR_INVALID_ARG = 1,     /* null pointer, bad size, overlap, bad rung */
    W4A16_ERR_UNSUPPORTED = 2,     /* group != 128, or a forced rung that cannot run the shape */
    W4A16_ERR_MISALIGNED = 3,      /* pointer alignment below the stated minimum */
    W4A16_ERR_WORKSPACE = 4,       /* the shape needs more split-K workspace than w4a16_init reserved */
    W4A16_ERR_NOT_INITIALIZED = 5, /* w4a16_init has not succeeded */
    W4A16_ERR_CUDA = 6,            /* a CUDA runtime call failed; see w4a16_last_cuda_error */
    W4A16_ERR_DEVICE = 7           /* a kernel gave up a bounded wait; see w4a16_device_status */
} w4a16_status;

/* Kernel rungs chosen by the dispatch table (w4a16_select_rung).  Every launch
 * increments the rung's probe counter (w4a16_probe_counts). */
typedef enum {
    W4A16_RUNG_AUTO = -1,
    W4A16_RUNG_GEMV = 0,        /* CUDA cores: warp per output row, whole K per CTA */
    W4A16_RUNG_GEMV_SPLITK = 1, /* CUDA cores: K split across CTAs, fixed-order fp32 reduce */
    W4A16_RUNG_TC = 2,          /* tcgen05 dequant-GEMM, tokens as the MMA N dimension */
    W4A16_RUNG_TC_SPLITK = 3,   /* tcgen05 dequant-GEMM, CTAs take equal runs of (tile, K stage) work */
    W4A16_RUNG_MMA = 4,         /* warp MMA (m16n8k16), A = weights dequantised in registers, M <= 8 */
    W4A16_RUNG_MMA_SPLITK = 5,  /* the same with K split across CTAs */
    W4A16_NUM_RUNGS = 6
} w4a16_rung;

/* Select `device`, reserve `workspace_bytes` of split-K workspace (0: 64 MiB)
 * plus the reducer's arrival counters, set kernel attributes, and read the
 * environment once: W4A16_FORCE_RUNG=<name|id> pins a rung, W4A16_LOG=1
 * prints each dispatch decision to stderr.  Allocates; must not run inside a
 * stream capture.  Calling it again re-initialises (after w4a16_shutdown's
 * implicit device synchronisation). */
int w4a16_init(int device, size_t workspace_bytes);

/* Synchronise the device, free the workspace and drop the library state. */
int w4a16_shutdown(void);

/* Bytes of split-K workspace the current dispatch needs for this shape (0 if
 * the selected rung splits nothing).  Pure host query. */
size_t w4a16_workspace_bytes(int M, int N, int K, int group);

/* Pack 4-bit values into the layout above (load time, before any capture: the
 * thread's section 四 notes that persistent packed tensors built lazily inside
 * graph capture were charged to the graph's memory pool).
 *   q [N, K] uint8 and z [N, K/group] uint8, device; only the low 4 bits of
 *   each byte are used.  Writes qweight [N, K/8] and zeros [N, ceil(G/8)]
 *   (pad nibbles 0).  q must be 16-byte aligned; qweight 16-byte; z, zeros
 *   4-byte. */
int w4a16_pack(const uint8_t *q, const uint8_t *z, int N, int K, int group,
               uint32_t *qweight, uint32_t *zeros, void *stream);

/* Inverse of w4a16_pack: q [N, K] and z [N, G] bytes 0..15. */
int w4a16_unpack(const uint32_t *qweight, const uint32_t *zeros, int N, int K, int group,
                 uint8_t *q, uint8_t *z, void *stream);

/* Restore the weights: w_f32[n, k] = (q - z) * s exactly (the product has at
 * most 15 significant bits, so fp32 holds it exactly), and w_f16 = that value
 * rounded once to fp16 (nearest, ties to even).  Either output may be NULL,
 * not both.  Outputs [N, K], 16-byte aligned. */
int w4a16_dequant(const uint32_t *qweight, const uint16_t *scales, const uint32_t *zeros,
                  int N, int K, int group, float *w_f32, uint16_t *w_f16, void *stream);

/* Load-time repack of a checkpoint whose INT4 layout is transposed (the Z100
 * thread, section 四: checkpoint layouts are transposed and repacked at load
 * time, nibble by nibble in 8 x 8 blocks, with no full int32 copy of the
 * matrix).  Transposes a packed 4-bit matrix A [rows, cols]:
 *   src [rows, cols/8] uint32, packed along cols: element (r, c) is nibble
 *       ((src_order >> 4*(c%8)) & 7) of word src[r][c/8].  src_order lists, in
 *       nibble j, the position holding element j of each word's eight;
 *       0x76543210 is this library's sequential order.  It must name each
 *       position 0..7 once (INVALID_ARG otherwise).
 *   dst [cols, ceil(rows/8)] uint32, packed along rows in sequential order;
 *       pad nibbles past `rows` are 0.
 * cols a multiple of 8; 1 <= rows, cols <= 2^24; src and dst 4-byte aligned
 * and apart.  A checkpoint with qweight [K, N/8] and zeros [G, N/8] (packed
 * along N) gives this library's qweight = repack(qweight, K, N) and zeros =
 * repack(zeros, G, N); its scales [G, N] go through w4a16_transpose_f16. */
int w4a16_repack_transpose(const uint32_t *src, int rows, int cols, uint32_t src_order,
                           uint32_t *dst, void *stream);

/* dst [cols, rows] = src [rows, cols]^T for 16-bit elements (fp16 bit patterns);
 * 1 <= rows, cols <= 2^24, 2-byte aligned, apart. */
int w4a16_transpose_f16(const uint16_t *src, int rows, int cols, uint16_t *dst, void *stream);

/* y = x @ W^T for one W4A16 linear layer (the operation at the top of this
 * file).  Enqueues one kernel for the rung w4a16_select_rung picks (the
 * split-K rungs reduce inside the same kernel); the CUDA-core rungs enqueue one
 * kernel per tile of up to 8 tokens. */
int w4a16_linear(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                 const uint32_t *zeros, int M, int N, int K, int group, uint16_t *y,
                 void *stream);

/* What w4a16_linear_epilogue (and a decode round's linear) does with the
 * linear's fp32 result h = x @ W^T before the single fp16 rounding of y.  The
 * steps that follow the linear in a decoder layer, done in the same kernel so
 * that h never goes to memory: the residual add after an output projection
 * (haowenji.com V100 decode article, its third round of changes, which merged
 * the add-back of the layer input into the matmul's output stage) and the
 * SiLU-and-mul after a fused gate+up projection (forum.sourcefind.cn thread
 * "vLLM on Hygon Z100", section 二, which names it among the MLP operators). */
typedef enum {
    W4A16_EPILOGUE_NONE = 0,     /* y[M, N] = h */
    W4A16_EPILOGUE_RESIDUAL = 1, /* y[M, N] = h + residual[M, N] (fp16, read as fp32) */
    W4A16_EPILOGUE_SILU_MUL = 2  /* y[M, N/2] = silu(h[:, :N/2]) * h[:, N/2:] with
                                    silu(g) = g / (1 + e^-g): the weight's first N/2 rows are
                                    the gate projection, the last N/2 the up projection; N must
                                    be a multiple of 32 */
} w4a16_epilogue;

/* The 16-bit type of x, scales, y and the residual.  The pages name fp16 or
 * bf16 activations; a bf16 layer keeps its scales in bf16 too.  Weights and
 * zeros are 4-bit either way; accumulation is fp32 either way. */
typedef enum {
    W4A16_DTYPE_F16 = 0,  /* IEEE binary16 */
    W4A16_DTYPE_BF16 = 1  /* bfloat16 (the top half of an IEEE binary32) */
} w4a16_dtype;

/* One linear of a decode round.  x is [M, K] and y [M, N] ([M, N/2] with
 * SiLU-and-mul); `group` must be 128.  `epilogue` is a w4a16_epilogue;
 * `residual` is [M, N] for W4A16_EPILOGUE_RESIDUAL and NULL otherwise;
 * `dtype` is a w4a16_dtype (0: fp16). */
typedef struct {
    const uint16_t *x;
    const uint32_t *qweight;
    const uint16_t *scales;
    const uint32_t *zeros;
    uint16_t *y;
    int N;
    int K;
    int group;
    int epilogue;
    const uint16_t *residual;
    int dtype;
} w4a16_linear_desc;

/* y = epilogue(x @ W^T): w4a16_linear followed, in the same kernel, by the
 * step `epilogue` names (w4a16_epilogue).  W4A16_EPILOGUE_NONE is exactly
 * w4a16_linear.  The other epilogues run on the warp-MMA rungs (up to 8
 * tokens) and on the tcgen05 rungs (more than 8 tokens: one reading of the
 * weights for up to 64; a SiLU-and-mul tile holds 64 outputs' gate and up
 * rows), not on the CUDA-core rungs (a forced one: W4A16_ERR_UNSUPPORTED).
 *   residual  [M, N] fp16, 2-byte aligned, for W4A16_EPILOGUE_RESIDUAL (NULL
 *             otherwise: INVALID_ARG); it may be y itself (y += x @ W^T) but
 *             must not otherwise overlap y.
 *   y         [M, N], or [M, N/2] with W4A16_EPILOGUE_SILU_MUL (N a multiple
 *             of 32: W4A16_ERR_UNSUPPORTED otherwise).
 * With split K the partial sums of h are reduced first and the epilogue applied
 * once to each output.  SiLU-and-mul always passes h through the split-K
 * workspace (on the warp-MMA rungs S x M x N fp32, S >= 1 K slices, and one
 * arrival counter per block of rows; on the tcgen05 rungs two 128-row slots
 * per CTA) and applies the epilogue where an output's gate and up sums meet:
 * W4A16_ERR_WORKSPACE if w4a16_init reserved too little. */
int w4a16_linear_epilogue(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                          const uint32_t *zeros, int M, int N, int K, int group, int epilogue,
                          const uint16_t *residual, uint16_t *y, void *stream);

/* w4a16_linear_epilogue with the 16-bit type `dtype` (w4a16_dtype) of x,
 * scales, residual and y.  bf16 runs on the warp-MMA and tcgen05 rungs, not on
 * the CUDA-core rungs.  On the warp-MMA rungs (up to 8 tokens) each token's
 * slice of x is staged as fp16 scaled by a power of two chosen from its
 * largest exponent (so any bf16 magnitude fits; bf16's 8 significant bits fit
 * fp16's 11, so the staged values are exact but for those 2^29 below the
 * token's largest), the fp16 tensor-core path runs unchanged, and the scale
 * is removed in fp32 before the one rounding of y to bf16.  On the tcgen05
 * rungs (more than 8 tokens) each weight is restored to bf16 ((q - z) * s,
 * rounded once) and multiplied with the bf16 activations on the tensor cores
 * (fp32 sums).  W4A16_DTYPE_F16 is exactly w4a16_linear_epilogue.  An invalid
 * dtype is INVALID_ARG. */
int w4a16_linear_ex(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                    const uint32_t *zeros, int M, int N, int K, int group, int dtype,
                    int epilogue, const uint16_t *residual, uint16_t *y, void *stream);

/* A decode round: the linears of `descs` (a HOST array of n_descs entries,
 * e.g. 64 layers x {qkv, o, gate+up, down}) run on `stream`, all at the same
 * M, each reading its weights once (haowenji.com V100 decode article: one
 * round reads every weight once).  All descriptors are validated before
 * anything is launched.
 *
 * The results are those of running the linears one after another in array
 * order.  Without a forced rung, a round of M <= 64 tokens is ONE kernel
 * launch: M <= 8 on the warp-MMA kernel (each linear gets its own part of the
 * split-K workspace), 9 <= M <= 64 on the tcgen05 kernel (one stream-K
 * sequence over every linear's tiles; two partial-sum slots per CTA shared by
 * all linears, one arrival counter per tile).  The weights of all linears
 * stream without a break, and a linear that reads an earlier linear's
 * output, writes an earlier linear's input or output (overlapping device
 * ranges) waits inside the kernel for that linear to complete.  Such a round
 * needs n_descs <= 4096, one 16-bit type for all its linears, and workspace
 * for its partial sums and counters (W4A16_ERR_WORKSPACE otherwise).  Its
 * descriptors are copied to device memory on `stream` when they differ from
 * the previous round's (the copy may briefly block the calling thread while
 * it stages them).  Other rounds, and every round enqueued on a stream that is
 * being captured, launch linear by linear; w4a16_round_graph_create captures
 * the fused form. */
int w4a16_decode_round(const w4a16_linear_desc *descs, int n_descs, int M, void *stream);
/* Each linear of a round applies its own epilogue and 16-bit type, with the
 * rules of w4a16_linear_ex; a linear's residual counts as one of its inputs for
 * the ordering above.  A round whose linears mix fp16 and bf16 launches linear
 * by linear. */

/* Capture a decode round into an instantiated CUDA graph (an opaque handle in
 * *graph).  Allocates (the graph's own copy of a fused round's descriptors)
 * and captures on an internal stream: call after w4a16_init, outside any other
 * capture.  The graph keeps the descriptors' device pointers and the dispatch
 * decisions made at capture time. */
int w4a16_round_graph_create(const w4a16_linear_desc *descs, int n_descs, int M,
                             void **graph);
/* Replay a captured round on `stream`. */
int w4a16_round_graph_launch(void *graph, void *stream);
/* Destroy a captured round (after its last replay has finished). */
int w4a16_round_graph_destroy(void *graph);

/* y = x @ W^T like w4a16_linear, for M <= 8 on the warp-MMA rungs, with no
 * allocation and no w4a16_init.  The pages have no counterpart: this serves
 * callers that cannot allocate device memory (a process whose memory a
 * caching allocator has wholly reserved, a serving loop that must not call
 * cudaMalloc, which synchronises the device).  Its split-K scratch is a
 * statically sized device array of the library, which every GPU that loads
 * the library holds until the process exits: 4 MiB of fp32 partial sums and
 * 4096 block counters.  That covers every M <= 8 linear of a 27B-class decode
 * layer (qkv 5120 x 8192, o 6144 x 5120, gate+up 5120 x 34816, down
 * 17408 x 5120, K x N); shapes whose split needs more return
 * W4A16_ERR_WORKSPACE before anything is launched, and M > 8 returns
 * W4A16_ERR_UNSUPPORTED.  The first call on a device (the current device at
 * the call) sets up that device: it looks up the scratch's device address,
 * zeroes its counters and sets the kernel attributes; make that first call
 * before any stream capture.  Every call shares the one scratch array: calls
 * that overlap on the GPU race on it.  Bounded-wait errors of its kernel are
 * recorded in a status word of the scratch, which w4a16_device_status reads
 * (that read also re-zeroes the scratch's counters when the word is set).
 * Each call counts one launch and one linear of its rung in the probes.
 * Argument rules as for w4a16_linear. */
int w4a16_linear_noalloc(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                         const uint32_t *zeros, int M, int N, int K, int group, uint16_t *y,
                         void *stream);

/* Dense 16-bit linear y [M, N] = x [M, K] @ w [N, K]^T for weights already
 * dequantised to fp16 or bf16 (the Z100 thread, section 六: FP8 weights
 * dequantised at load time to FP16/BF16 run through a large-K, small-M GEMV
 * with fp32 products and sums).  x, w and y share the 16-bit type `dtype`
 * (w4a16_dtype); accumulation is fp32, y rounded once (nearest even).
 * Streams w once per tile of up to 8 tokens on the warp MMA (split K through
 * the w4a16_init workspace when the plan splits; W4A16_ERR_WORKSPACE if it is
 * too small).  K a multiple of 128 (128..2^22), 1 <= N < 2^31, 1 <= M <=
 * 65535; x, w, y 16-byte aligned; y apart from x and w.  Needs w4a16_init. */
int w4a16_dense_linear(const uint16_t *x, const uint16_t *w, int M, int N, int K, int dtype,
                       uint16_t *y, void *stream);

/* ---- mixture of experts (the Z100 thread, section 七: a router picks k of E
 * experts per token; the tokens are regrouped by expert; a W4A16 small-M GEMV
 * runs over the packed INT4 experts; each token's expert outputs are summed
 * with the router's weights).  Token t's j-th choice is slot s = t*k + j.
 * The router itself (its linear, softmax and top-k) is the caller's.
 *
 * w4a16_moe_align: topk_ids [n_slots] int32 (device) -> the slots grouped by
 * expert, stable in slot order: offsets [E+1] (first sorted position of each
 * expert; offsets[E] = the slots with a valid id), sorted [n_slots] (slot at
 * each position), pos [n_slots] (position of each slot).  An id outside
 * [0, E) gives its slot pos = -1 (left out of every expert and of the sum) and
 * sets a bit that w4a16_device_status reports.  E <= 1024.  Needs w4a16_init. */
int w4a16_moe_align(const int32_t *topk_ids, int n_slots, int E, int32_t *sorted, int32_t *pos,
                    int32_t *offsets, void *stream);

/* An expert layer: E experts stacked, qweight [E, N, K/8], scales [E, N, G],
 * zeros [E, N, ceil(G/8)], each expert in this library's layout.  `epilogue`
 * is W4A16_EPILOGUE_NONE or W4A16_EPILOGUE_SILU_MUL (the experts' fused
 * gate+up); `dtype` the 16-bit type of activations, scales and outputs.
 * max_slots bounds n_slots of later calls.  Allocates (call after w4a16_init,
 * outside any capture); the weights must outlive the handle.  One plan serves
 * every call: it assumes min(max_slots, E) experts in use side by side. */
int w4a16_moe_create(int E, int N, int K, int group, const uint32_t *qweight,
                     const uint16_t *scales, const uint32_t *zeros, int epilogue, int dtype,
                     int max_slots, void **moe);
int w4a16_moe_destroy(void *moe);

/* y [n_slots, N] (N/2 with SiLU-and-mul), in sorted order (row p = slot
 * sorted[p]): each slot's expert linear.  x is by token, [n_slots/gather_k, K]
 * (slot s reads token s / gather_k, gathered on the device), when gather_k > 0;
 * by sorted position, [n_slots, K] (e.g. the y of an earlier expert linear),
 * when gather_k == 0.  sorted and offsets come from w4a16_moe_align.  Two
 * kernels: the tile descriptors (and the gather), then every expert tile of up
 * to 8 slots in one launch of the warp-MMA kernel.  Calls on one handle must
 * not overlap on the GPU (it holds the descriptors and gathered rows). */
int w4a16_moe_linear(void *moe, const uint16_t *x, int gather_k, const int32_t *sorted,
                     const int32_t *offsets, int n_slots, uint16_t *y, void *stream);

/* An expert MLP: gate+up (usually with SiLU-and-mul) then down over the same
 * routing, made of two handles from w4a16_moe_create (down's K = gate+up's
 * output columns, down's N = gate+up's K, same E and dtype, down without an
 * epilogue).  Holds the chain's buffers for up to max_tokens tokens of k
 * choices (max_tokens * k must not exceed either handle's max_slots).
 * Allocates: call after w4a16_init, outside any capture.  Both split-K spaces
 * must fit the workspace at once (W4A16_ERR_WORKSPACE). */
int w4a16_moe_mlp_create(void *gate_up, void *down, int max_tokens, int k, void **mlp);
int w4a16_moe_mlp_destroy(void *mlp);

/* out [T, N_down] = sum_j weights[t, j] * down_e(gate_up_e(x[t])) with e the
 * token's j-th expert.  x [T, K] by token; topk_ids [T, k] int32; weights
 * [T, k] fp32 (device).  Two paths (w4a16_moe_path):
 *   chain: align, then one kernel preparing both linears' tiles (and
 *     gathering x), then ONE launch of the warp-MMA kernel over the gate+up
 *     tiles and the down tiles (a down tile waits inside the kernel for its
 *     gate+up tile), then the weighted sum;
 *   decode: ONE launch for the whole MLP (routing in every CTA, gate+up with
 *     SiLU-and-mul, down, and the weighted sum), for gate+up with
 *     SiLU-and-mul, K and down's K multiples of 128, down's N a multiple of
 *     128, T <= 8, T * k <= 128 and activation rows that fit on chip.
 * The intermediate and each expert's output are rounded to the 16-bit type
 * on both paths, and the sum runs over j in order in fp32.  Calls on one
 * handle must not overlap on the GPU. */
int w4a16_moe_mlp(void *mlp, const uint16_t *x, const int32_t *topk_ids, const float *weights,
                  int T, uint16_t *out, void *stream);

typedef enum {
    W4A16_MOE_PATH_AUTO = 0,   /* decode when the call fits it, else chain */
    W4A16_MOE_PATH_CHAIN = 1,
    W4A16_MOE_PATH_DECODE = 2  /* calls that do not fit return W4A16_ERR_UNSUPPORTED */
} w4a16_moe_path;

/* Choose the path of later w4a16_moe_mlp calls on this handle (host state;
 * a graph captured earlier keeps its launches). */
int w4a16_moe_mlp_set_path(void *mlp, int path);

/* The path (W4A16_MOE_PATH_CHAIN or _DECODE) a call with T tokens takes, in
 * *path; W4A16_ERR_UNSUPPORTED when the forced decode path cannot take T. */
int w4a16_moe_mlp_path(void *mlp, int T, int *path);

/* Device pointers to the handle's intermediate rows h [max_tokens * k, K_down]
 * and expert outputs o [max_tokens * k, N_down] (16-bit), which every
 * w4a16_moe_mlp call on either path writes in sorted order (the expert-major,
 * slot-stable order of w4a16_moe_align; row p belongs to the slot at sorted
 * position p).  Valid until w4a16_moe_mlp_destroy; for inspection and tests. */
int w4a16_moe_mlp_buffers(void *mlp, uint16_t **h, uint16_t **o);

/* out [T, N] = sum_j weights[t*k + j] * y_sorted[pos[t*k + j]], fp32
 * accumulation in j order, one rounding; weights fp32 [T, k]; y_sorted and
 * out of type dtype. */
int w4a16_moe_sum(const uint16_t *y_sorted, const int32_t *pos, const float *weights, int T,
                  int k, int N, int dtype, uint16_t *out, void *stream);

/* The rung the dispatch table picks for a shape (honouring a forced rung), or
 * -1 for an invalid shape.  Pure host query.  Unforced: M <= 8 takes the warp
 * MMA rungs, except small fp16 linears without an epilogue, which take the
 * CUDA-core rungs (where the lighter launch wins: up to 24 Mi weights N*K at
 * M <= 2, 16 Mi at M <= 4, 8 Mi at M <= 8); M >= 9 takes the tcgen05 rungs.
 * The _SPLITK variant is the plan's choice for the shape. */
int w4a16_select_rung(int M, int N, int K, int group);

/* The plan of the first tile of a linear (of up to 8 tokens on the mma and
 * gemv rungs, 64 on the tc rungs) as w4a16_linear_ex / w4a16_linear_epilogue
 * would launch it now (honouring a forced rung): info[0] the rung, info[1]
 * threads per CTA (the warp-MMA kernel: 256 = 8 warps, two CTAs per SM, or
 * 512 = 16 warps, one CTA per SM), info[2] K slices (the tc rungs: 1 = whole
 * tiles, 2 = stream-K), info[3] CTAs in the launch.  Pure host query; before
 * w4a16_init it assumes 152 SMs.  Returns INVALID_ARG for a bad shape,
 * epilogue or dtype (or a null info), UNSUPPORTED if a forced rung cannot run
 * the shape. */
int w4a16_plan_info(int M, int N, int K, int group, int epilogue, int dtype, int32_t *info);

/* Force a rung for later calls (W4A16_RUNG_AUTO restores the table).  A forced
 * rung that cannot run a shape makes that call return W4A16_ERR_UNSUPPORTED.
 * Returns the previous setting, or -2 for an invalid rung.  Host state only:
 * graphs captured earlier keep their rungs. */
int w4a16_set_forced_rung(int rung);

/* Copy min(n, W4A16_NUM_RUNGS) per-rung counts into counts (host); returns
 * the number written.  A rung's count grows by one for every linear (every
 * tile of up to its token limit) it computes: a fused decode round counts each
 * of its linears under the rung that computes it.  Counts are host-side
 * dispatch decisions (a graph replay does not re-count). */
int w4a16_probe_counts(uint64_t *counts, int n);
/* Kernels this library has launched (host count, all entry points, since the
 * last w4a16_probe_reset; a graph replay does not re-count). */
uint64_t w4a16_kernel_launches(void);
void w4a16_probe_reset(void);

/* Static strings; "?" for unknown values. */
const char *w4a16_rung_name(int rung);
const char *w4a16_status_string(int status);

/* Kernels that wait on on-chip barriers (the tensor-core rungs) bound every
 * wait by a timer; if one expires the kernel ORs a code into a device status
 * word, drains its in-flight copies, frees its tensor memory and exits, so the
 * CUDA context stays usable.  This call synchronises `stream`, returns
 * W4A16_ERR_DEVICE with the accumulated code in *code (may be NULL) if any
 * kernel reported one since the last call, and clears the word.  It also
 * reads the status word of w4a16_linear_noalloc's scratch on the current
 * device (once a call has set that device up) and ORs it in; when that word
 * is set it re-zeroes the scratch's block counters and scheduling words too,
 * since a launch cut short by an expired wait can leave them nonzero (call it
 * with no w4a16_linear_noalloc call in flight).  W4A16_ERR_NOT_INITIALIZED
 * when neither w4a16_init nor a w4a16_linear_noalloc call has run. */
int w4a16_device_status(void *stream, int *code);

/* Exercise the expired-wait report: one thread runs the library's bounded
 * waits on a completion counter that nothing increments and on an mbarrier
 * that nothing arrives at; each gives up after its limit (200 ms) and ORs a
 * bit into the device status word (4096: the counter wait, 8192: the
 * mbarrier wait), which the next w4a16_device_status returns.  When a
 * w4a16_linear_noalloc call has set up the current device, a second probe
 * does the same on that scratch's status word after incrementing its first
 * block counter, as a split-K launch cut short can leave it.  Nothing faults
 * or hangs; the stream is busy for about 0.4 s per probe.  For tests of the
 * error path.  Needs w4a16_init. */
int w4a16_wait_probe(void *stream);

/* The cudaError_t behind the calling thread's last W4A16_ERR_CUDA (0 if none). */
int w4a16_last_cuda_error(void);

/* Number of streaming multiprocessors of the initialised device (0 before init). */
int w4a16_device_sm_count(void);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
