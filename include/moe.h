/*
 * moe.h - C ABI of libmoe: the hot path of one expert-parallel MoE layer on one GB300 GPU.
 *
 * The layer (router -> dispatch -> grouped SwiGLU expert GEMMs + shared expert -> combine) is
 * the one described in "7.13 Serving Mixture-of-Experts: Expert Parallelism & All-to-All
 * Inference" (llm-stack-book), section "Expert Parallelism Mechanics: Dispatch, Compute,
 * Combine", with the DeepSeek-V3 router of "Mixture-of-experts serving" (learn-kernels),
 * paragraphs 1 and 3, and the receive-buffer design of "One-Sided Expert-Parallel All-to-All
 * for Mixture-of-Experts Inference over NVLink" (abstract): every source pushes its rows into
 * rank-major buffers with no metadata exchange first, and the grouped GEMMs read those buffers
 * in place. The expert-parallel ranks are logical: R partitions of this GPU's memory.
 *
 * Conventions for every entry point
 *  - All array pointers are DEVICE pointers, allocated and owned by the caller. The library
 *    allocates nothing and keeps no state between calls except cached kernel attributes and
 *    the driver entry point it uses to encode TMA tensor maps.
 *  - Work is enqueued on `stream` and the call returns at once (asynchronous). No call
 *    synchronises with the host or copies device memory to the host, except
 *    moe_read_status, which says so.
 *  - Arrays are dense and row-major with the shapes given. bf16 is IEEE bfloat16, e4m3 is the
 *    8-bit float with 4 exponent bits (bias 7) and 3 mantissa bits (largest finite 448).
 *    Device pointers must be 16-byte aligned.
 *  - Return value: MOE_OK, or an MOE_ERR_* code describing the first failed check; nothing
 *    is enqueued when a check fails. moe_strerror() names the code.
 *  - Errors found on the device (a wait that ran out, a bounds check) are OR-ed into a status
 *    word at the start of the workspace `ws`; read it with moe_read_status().
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 3

/* Return codes */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1  /* a shape constraint failed or a required pointer is NULL */
#define MOE_ERR_UNSUPPORTED 2  /* valid MoE shape outside what these kernels implement */
#define MOE_ERR_MISALIGNED 3   /* a device pointer is not 16-byte aligned */
#define MOE_ERR_CUDA 4         /* a CUDA runtime/driver call or a kernel launch failed */

/* Device status bits (moe_read_status) */
#define MOE_DEV_TIMEOUT 1u     /* a bounded wait inside a kernel gave up; outputs invalid */
#define MOE_DEV_BOUNDS 2u      /* an index read from device memory was out of range */
#define MOE_DEV_SCALE 4u       /* MOE_FP8_E4M3_POW2: a weight block scale is not a power of two
                                  (not positive, not finite, or with mantissa bits); the GEMM
                                  applied 2^(its exponent field - 127) in its place */

/* Element formats */
#define MOE_BF16 0
#define MOE_FP8_E4M3 1       /* e4m3 with fp32 block scales: 1x128 for activations (scale =
                                amax / 448), 128x128 for weights (any positive scales) */
#define MOE_FP8_E4M3_POW2 2  /* e4m3 with power-of-two fp32 block scales: the same blocks, each
                                activation scale the smallest power of two 2^e with
                                amax <= 448 * 2^e (e in [-126, 127], 1 for an all-zero block);
                                the weight scales must be powers of two too. The grouped GEMMs
                                apply the scales in the tensor core (block-scaled MMA) instead
                                of promoting each 128-K block's partial sums. These kernels
                                take d % 256 == 0, d <= 8192 and d_ff <= 8192 in this format
                                (MOE_ERR_UNSUPPORTED otherwise). */

/* Number of events moe_layer records when given an event array (see moe_layer). */
#define MOE_LAYER_EVENTS 7

/* Shape of one MoE layer. Notation of the pages: T tokens of width d, E routed experts, top-k
 * routing with n_group groups of which topk_group are kept, SwiGLU experts of width d_ff,
 * one shared expert of width d_ff_shared, R logical expert-parallel ranks. */
typedef struct moe_cfg {
  int32_t T;            /* tokens in the batch, all logical ranks together; T % R == 0 */
  int32_t d;            /* model width; d % 128 == 0 */
  int32_t E;            /* routed experts; E % R == 0, E % n_group == 0, E <= 1024 */
  int32_t k;            /* experts per token; 1 <= k <= min(32, topk_group * E / n_group) */
  int32_t n_group;      /* expert groups (contiguous blocks of E/n_group experts), <= 64 */
  int32_t topk_group;   /* groups kept per token; 1 <= topk_group <= n_group */
  int32_t d_ff;         /* routed expert SwiGLU width; d_ff % 128 == 0 */
  int32_t d_ff_shared;  /* shared expert width; 0 = no shared expert, else % 128 == 0 */
  int32_t R;            /* logical ranks; expert e lives on rank e / (E/R), token t is sent by
                           rank t / (T/R); R <= 64 */
  float route_scale;    /* factor applied to the renormalised gate weights */
  int32_t act_dtype;    /* dispatched activations: MOE_BF16, MOE_FP8_E4M3 or MOE_FP8_E4M3_POW2 */
  int32_t w_dtype;      /* expert weights: must equal act_dtype */
} moe_cfg;

/* Buffer sizes the caller allocates for a configuration. */
typedef struct moe_sizes {
  int64_t recv_rows;        /* R * R * cap rows in the receive buffer */
  int32_t cap;              /* rows per (destination rank, source rank) segment:
                               (T/R) * min(k, E/R), the most one source can send one rank */
  size_t recv_bytes;        /* recv: [R][R][cap][d], bf16 (2 B) or e4m3 (1 B) elements */
  size_t recv_scale_bytes;  /* e4m3 only: recv_scales fp32, block-major [d/128][recv_rows]
                               (scale of block b of row j at b * recv_rows + j); else 0 */
  size_t ebuf_bytes;        /* ebuf: expert outputs, bf16 [R][R][cap][d] (same rows as recv) */
  size_t ws_bytes;          /* ws: scratch workspace (status word, router partials, tile
                               schedule, SwiGLU intermediates) */
} moe_sizes;

/* Expert weights, K-major (the reduction dimension is contiguous).
 *  w13  [E][2*d_ff][d]: rows 0..d_ff-1 are the gate projection, d_ff..2*d_ff-1 the up one.
 *  w2   [E][d][d_ff]:   down projection.
 *  ws13 [2*d_ff_shared][d], ws2 [d][d_ff_shared]: the shared expert (NULL if none).
 *  e4m3 weights carry one fp32 scale per 128x128 block: w13_scales [E][2*d_ff/128][d/128],
 *  w2_scales [E][d/128][d_ff/128], ws13_scales [2*d_ff_shared/128][d/128],
 *  ws2_scales [d/128][d_ff_shared/128]; all scale pointers are NULL for bf16. */
typedef struct moe_weights {
  const void* w13;
  const float* w13_scales;
  const void* w2;
  const float* w2_scales;
  const void* ws13;
  const float* ws13_scales;
  const void* ws2;
  const float* ws2_scales;
} moe_weights;

/* Checks a configuration. Returns MOE_OK, MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED. */
int moe_validate(const moe_cfg* cfg);

/* Fills *out with the buffer sizes for cfg. Same return codes as moe_validate. */
int moe_query_sizes(const moe_cfg* cfg, moe_sizes* out);

/* Router ("Mixture-of-experts serving", paragraphs 1 and 3; "Serving Mixture-of-Experts",
 * Expert Parallelism Mechanics, router step). For every token t:
 *   z[e] = x[t] . w_gate[e] in fp32, summed in a fixed order: d in 16 equal chunks, each a
 *          sequential fused multiply-add chain, the 16 partials added by a pairwise tree;
 *   s[e] = 1 / (1 + exp(-z[e])) (exp by Cody-Waite reduction and a degree-7 Taylor series);
 *   v[e] = s[e] + bias[e]   (the bias steers selection only);
 *   group score = sum of the two largest v in the group; the topk_group best groups are kept;
 *   the k best experts of the kept groups by v are chosen (ties: lower index first);
 *   topk_w[t][i] = s[e_i] / (s[e_0] + ... + s[e_{k-1}]) * route_scale.
 * x bf16 [T][d]; w_gate fp32 [E][d]; bias fp32 [E]; outputs topk_idx int32 [T][k] in
 * selection order and topk_w fp32 [T][k]. ws: workspace of moe_sizes.ws_bytes. */
int moe_route(const moe_cfg* cfg, const void* x, const float* w_gate, const float* bias,
              int32_t* topk_idx, float* topk_w, void* ws, cudaStream_t stream);

/* The router of moe_route for callers that cannot give the library any device memory beyond
 * their inputs and outputs: a plugin inside another framework with no access to its
 * allocator, a deployment whose device memory is fully planned at start-up, or a hot path that
 * must not enter the driver allocator (cudaMalloc/cudaFree can synchronise the device). It
 * needs no ws: its scratch (16 partial dot products per token and expert) is a fixed 8 MiB
 * device array inside the library, which every device that loads the library holds until the
 * process exits. The pages have no counterpart to this entry point; it exists for such
 * callers only. Arguments and results are those of moe_route. Limits and behaviour:
 *  - returns MOE_ERR_UNSUPPORTED when 16 * T * E exceeds 2^21 floats (T*E > 131072, e.g. more
 *    than 512 tokens at 256 experts); nothing is enqueued then;
 *  - the first call in each device context looks up the array's device address with that
 *    device current (cudaGetSymbolAddress) and caches it under the context's ID; make that
 *    first call before any stream capture (a context made after a device reset looks it up
 *    again on its own first call);
 *  - it allocates nothing (no cudaMalloc, no cudaFree, no allocating library call);
 *  - every call shares the array and leaves its contents behind; each call writes every entry
 *    it reads, so nothing needs clearing, but calls whose kernels overlap on the GPU (other
 *    streams, other host threads on the same device) race on it: serialise them. */
int moe_route_noalloc(const moe_cfg* cfg, const void* x, const float* w_gate, const float* bias,
                      int32_t* topk_idx, float* topk_w, cudaStream_t stream);

/* Dispatch ("Serving Mixture-of-Experts", Expert Parallelism Mechanics, dispatch step;
 * "One-Sided Expert-Parallel All-to-All...", abstract; "Serving Mixture-of-Experts", DeepEP,
 * FP8 dispatch and fixed-size buffers). Each logical source rank s (tokens s*T/R ..) counts
 * its rows per expert, takes exclusive sums of those counts inside each destination rank, and
 * writes one row per (token, chosen expert) into segment (r = rank(e), s) of the receive
 * buffer: row (r*R + s)*cap + [sum of counts[s][e'] for e' on rank r, e' < e] + [number of
 * earlier tokens of s that chose e]. No count is exchanged before the rows are written.
 * bf16: recv[row] = x[t]. e4m3: x[t] is quantised once per 128-column block (scale =
 * amax/448, or 1 if amax is 0; code = e4m3(x/scale), nearest even, saturating) and written to
 * each of its rows; the block scales are block-major, recv_scales[b * recv_rows + row], so the
 * expert GEMMs read one K block's scales for consecutive rows from consecutive addresses.
 * Inputs x bf16 [T][d], topk_idx int32 [T][k] (entries in [0, E), distinct per token).
 * Outputs recv (see moe_sizes), recv_scales (e4m3 only, else NULL), counts int32 [R][E],
 * row_of int32 [T][k] (receive row of each choice), src_tok int32 [recv_rows] (token of each
 * row, -1 for empty rows; NULL to skip). Receive rows that get no token are not written.
 * status: NULL, or a device uint32 (for instance the workspace's status word: pass ws) into
 * which MOE_DEV_BOUNDS is OR-ed when topk_idx breaks its contract. A choice whose expert is
 * outside [0, E), or repeats an earlier choice of the same token, is skipped: its row_of is
 * -1, it is not counted, and nothing is written for it. With distinct experts no segment can
 * overflow; every receive row written lies inside recv. moe_route never produces either. */
int moe_dispatch(const moe_cfg* cfg, const void* x, const int32_t* topk_idx, void* recv,
                 float* recv_scales, int32_t* counts, int32_t* row_of, int32_t* src_tok,
                 uint32_t* status, cudaStream_t stream);

/* Expert FFNs ("Serving Mixture-of-Experts", Expert Parallelism Mechanics, expert compute: a
 * grouped GEMM over the rows each expert received; Hot-Expert Skew section and
 * "Mixture-of-experts serving" paragraph 1: the always-on shared expert). For every filled
 * receive row of expert e, read in place from recv:
 *   h = silu(row . Wgate_e^T) * (row . Wup_e^T), rounded to the activation format
 *       (e4m3: re-quantised per 128 columns like the dispatch);
 *   ebuf[row] = bf16(h . Wdown_e^T).
 * The shared expert does the same for every token of x: shared_out[t] (bf16 [T][d]).
 * counts: the dispatch's counts [R][E] (the only metadata; rows are located from it).
 * x: bf16 [T][d], the shared expert's input (NULL when d_ff_shared == 0). For e4m3 the shared
 * input is quantised here with the dispatch's rule. Rows of ebuf that hold no token are not
 * written. ws: workspace (holds the tile schedule and the SwiGLU intermediates). The two
 * GEMMs follow this call's own schedule kernels with programmatic launches (see moe_layer). */
int moe_expert_ffn(const moe_cfg* cfg, const void* recv, const float* recv_scales,
                   const int32_t* counts, const void* x, const moe_weights* w, void* ebuf,
                   void* shared_out, void* ws, cudaStream_t stream);

/* Combine ("Serving Mixture-of-Experts", Expert Parallelism Mechanics, combine step: the k
 * partial results of a token weighted-summed by its gate weights; DeepEP section: BF16
 * combine). y[t] = bf16( sum_i topk_w[t][i] * ebuf[row_of[t][i]] + shared_out[t] ), summed in
 * fp32 in selection order. ebuf bf16 [recv_rows][d]; row_of int32 [T][k]; topk_w fp32
 * [T][k]; shared_out bf16 [T][d] or NULL; y bf16 [T][d]. Passing the receive buffer as ebuf
 * (bf16) gives route_scale * x: the identity-expert check of the dispatch/combine pair.
 * Negative entries of row_of are skipped (a choice the dispatch skipped). Entries at or past
 * recv_rows are skipped too and reported: MOE_DEV_BOUNDS is OR-ed into status (NULL, or a
 * device uint32 such as the workspace's status word). Nothing outside ebuf is read.
 * moe_dispatch's row_of holds only valid rows and -1. */
int moe_combine(const moe_cfg* cfg, const void* ebuf, const int32_t* row_of,
                const float* topk_w, const void* shared_out, void* y, uint32_t* status,
                cudaStream_t stream);

/* The whole layer on one stream: moe_route, moe_dispatch, moe_expert_ffn, moe_combine.
 * Buffers as in those calls (src_tok is not produced). events: NULL, or MOE_LAYER_EVENTS
 * created events that are recorded on `stream` before the router, after the router, after
 * the dispatch, after the FFN set-up (schedule and shared-input quantisation), after the
 * gate/up GEMM, after the down GEMM, and after the combine.
 * With events == NULL every kernel after the first is launched with programmatic stream
 * serialisation: it may become resident while the previous kernel runs, and waits for that
 * kernel to finish before it touches memory. The first kernel (the router's) starts after the
 * work already on `stream`, as any launch. With events, the stages are launched one after
 * another so that the events time them. With a shared expert, the router's selection kernel
 * also starts prefetching w->ws13 into L2 (reads only; the gate/up GEMM reads it first). */
int moe_layer(const moe_cfg* cfg, const void* x, const float* w_gate, const float* bias,
              const moe_weights* w, int32_t* topk_idx, float* topk_w, void* recv,
              float* recv_scales, int32_t* counts, int32_t* row_of, void* ebuf,
              void* shared_out, void* y, void* ws, cudaStream_t stream,
              const cudaEvent_t* events);

/* ---------------------------------------------------------------------------------------
 * Variants of the layer ("next" steps of the method, each optional)
 * ------------------------------------------------------------------------------------- */

/* Gather mode. The dispatch writes only the indices (counts, row_of and the token of each
 * receive row); the gate/up GEMM reads each routed row straight from x by token instead of
 * from a receive-buffer copy, so the copy pass and its Tk*d bytes of writes and reads are
 * skipped. The grouped GEMMs reading pushed rows in place is the design of "One-Sided
 * Expert-Parallel All-to-All ..." (abstract); "DeepSeek MoE Serving: Where Expert-Parallel
 * All-to-All Time Goes" (groundy) counts the extra pass of a two-sided scheme as HBM traffic.
 * On one GPU the source rank's own x is the pushed buffer, read in place. e4m3: x is
 * quantised once per token (not once per (token, expert) row) with the dispatch's rule. The
 * expert outputs still land in ebuf at the receive rows, so the combine is unchanged and every
 * output equals moe_layer's. recv and recv_scales are not used (may be NULL). */
#define MOE_OPT_GATHER_X 1u
/* Shared expert on a second stream ("Serving Mixture-of-Experts", Hot-Expert Skew: the shared
 * expert's FFN needs no all-to-all, so it is free work to overlap with the dispatch; DeepEP
 * section: hook-based overlap). Its GEMMs depend only on x: they are enqueued on side_stream
 * after fork_event (recorded on `stream` at the start of the layer), limited to side_ctas CTAs
 * (one per SM, leaving the other SMs to the router and dispatch), and the combine waits on
 * join_event (recorded on side_stream after them). On one GPU this partitions the SMs between
 * the two streams. The events are created by the caller (cudaEventDisableTiming is enough). */
#define MOE_OPT_SHARED_SIDE_STREAM 2u
/* Fused expert stage (bf16 only): the gate/up GEMM, the down GEMM and the combine run in one
 * persistent cooperative launch ("DeepSeek MoE Serving: Where Expert-Parallel All-to-All Time
 * Goes" (groundy), regimes table and the paragraph after it: a fused MoE kernel against
 * separate kernels). A down unit starts as soon as the gate/up units of its own token tile
 * have published their rows (device-side counters in ws, every wait bounded), so SMs that run
 * out of gate/up units do not idle until the whole stage ends; the combine follows in the same
 * launch. Not with MOE_OPT_SHARED_SIDE_STREAM (MOE_ERR_INVALID_ARG) or e4m3
 * (MOE_ERR_UNSUPPORTED). Stage events 4..6 are all recorded after the launch. */
#define MOE_OPT_FUSED_FFN 4u

/* Redundant experts ("Serving Mixture-of-Experts", Hot-Expert Skew: place extra copies of the
 * busiest experts on under-loaded ranks and let the dispatch split their tokens across the
 * copies; exercise 5: each copy takes an equal share of its expert's load, copies assigned
 * largest first to the least-loaded rank). Each of the R logical ranks has slots_per_rank
 * expert slots, G = R * slots_per_rank >= E in all; slot p lives on rank p / slots_per_rank.
 * The dispatch sends source s's j-th row of expert e (in token order) to copy
 * (j + s) mod n_copies[e]: every source splits its own rows of an expert evenly over the
 * copies without exchanging counts. All arrays are DEVICE int32 arrays owned by the caller,
 * normally filled from moe_place_experts:
 *  slot_expert [G]: the expert each slot holds; n_copies [E]: copies of each expert (>= 1);
 *  copy_slot [E][max_copies]: the slots of each expert's copies in ascending order.
 * With a placement the receive layout and counts are over the G slots (counts [R][G],
 * cap = (T/R) * min(k, slots_per_rank); moe_query_sizes_placed gives the sizes). The expert
 * GEMMs take the rows of all copies of an expert through its weights together (one GPU holds
 * one set of weights per expert), so the output equals moe_layer's bit for bit. */
typedef struct moe_placement {
  int32_t slots_per_rank;
  int32_t max_copies;
  const int32_t* slot_expert;
  const int32_t* n_copies;
  const int32_t* copy_slot;
} moe_placement;

typedef struct moe_layer_opts {
  uint32_t flags;           /* MOE_OPT_* bits; 0 = moe_layer */
  cudaStream_t side_stream; /* MOE_OPT_SHARED_SIDE_STREAM: the shared expert's stream */
  cudaEvent_t fork_event;   /* recorded on `stream`, waited on by side_stream */
  cudaEvent_t join_event;   /* recorded on side_stream, waited on by `stream` */
  int32_t side_ctas;        /* CTAs of each shared-expert GEMM; 0 = 16 */
  const moe_placement* placement; /* NULL, or redundant experts placed on slots (above) */
} moe_layer_opts;

/* Placement of E experts on R ranks of slots_per_rank slots from estimated loads (host
 * function, no GPU; load: host double [E], e.g. a moving average of past counts). The
 * R*slots_per_rank - E spare slots take one more copy at a time of the expert with the largest
 * load per copy (ties: lower expert). Each copy carries load/copies; copies are placed largest
 * first (ties: lower expert, then lower copy) on the least-loaded rank that has a free slot
 * (ties: lower rank); a rank's slots are ordered by (expert, copy). Outputs (host int32):
 * slot_expert [R*slots_per_rank], n_copies [E], copy_slot [E][max_copies] (-1 past a copy
 * count). Returns MOE_ERR_INVALID_ARG for a NULL pointer, non-positive sizes, a negative or
 * non-finite load, R*slots_per_rank < E, or an expert needing more than max_copies copies. */
int moe_place_experts(int32_t E, int32_t R, int32_t slots_per_rank, const double* load,
                      int32_t max_copies, int32_t* slot_expert, int32_t* n_copies,
                      int32_t* copy_slot);

/* moe_query_sizes for a layer whose experts are placed on R*slots_per_rank slots. */
int moe_query_sizes_placed(const moe_cfg* cfg, int32_t slots_per_rank, moe_sizes* out);

/* moe_layer with the variants selected by opts (NULL = moe_layer). Arguments as in moe_layer;
 * with MOE_OPT_GATHER_X, recv and recv_scales may be NULL. With MOE_OPT_SHARED_SIDE_STREAM and
 * a shared expert, side_stream, fork_event and join_event must be valid (else
 * MOE_ERR_INVALID_ARG); stage events are recorded on `stream` only, so the FFN stages then
 * time the routed experts alone. With a placement, recv, counts, ebuf and ws are sized by
 * moe_query_sizes_placed and counts is [R][G] over the slots; a slot whose expert lies outside
 * [0, E) is reported (MOE_DEV_BOUNDS) and computed with expert 0's weights. The layer output
 * y is moe_layer's in every mode, bit for bit. */
int moe_layer_ex(const moe_cfg* cfg, const moe_layer_opts* opts, const void* x,
                 const float* w_gate, const float* bias, const moe_weights* w, int32_t* topk_idx,
                 float* topk_w, void* recv, float* recv_scales, int32_t* counts, int32_t* row_of,
                 void* ebuf, void* shared_out, void* y, void* ws, cudaStream_t stream,
                 const cudaEvent_t* events);

/* The index pass of moe_dispatch alone (gather mode): counts, row_of and src_tok exactly as
 * moe_dispatch writes them (src_tok required here; receive rows that get no token hold -1),
 * with no payload copied. status as in moe_dispatch. */
int moe_dispatch_index(const moe_cfg* cfg, const int32_t* topk_idx, int32_t* counts,
                       int32_t* row_of, int32_t* src_tok, uint32_t* status,
                       cudaStream_t stream);

/* moe_expert_ffn in gather mode: the routed rows are read from x by token through src_tok
 * (from moe_dispatch_index) instead of from a receive buffer. x: bf16 [T][d], required. The
 * outputs (ebuf at the receive rows, shared_out) equal moe_expert_ffn's. */
int moe_expert_ffn_gather(const moe_cfg* cfg, const void* x, const int32_t* counts,
                          const int32_t* src_tok, const moe_weights* w, void* ebuf,
                          void* shared_out, void* ws, cudaStream_t stream);

/* Sets the device status word in ws to 0 (enqueued on stream). */
int moe_clear_status(void* ws, cudaStream_t stream);

/* Synchronises `stream`, then copies the device status word of ws into *status (MOE_DEV_*
 * bits). This is the one call that blocks the host. */
int moe_read_status(const void* ws, uint32_t* status, cudaStream_t stream);

/* Diagnostic of the device-side failure handling (the pages have no counterpart; it serves
 * callers and tests that must see a kernel give up instead of hang). Launches one CTA in which
 * one thread waits on a barrier that nothing ever completes, bounded by limit_ns, while a
 * second thread waits on another such barrier with a limit three times as long. When the first
 * wait runs out it ORs MOE_DEV_TIMEOUT into the status word of ws and raises the CTA's abort
 * flag, on which the second wait returns at once; the kernel then ends (after about limit_ns,
 * well before 3 x limit_ns) and the context stays usable. ws: any workspace of this library
 * (only its status word is written). limit_ns: 1 us .. 10 s, else MOE_ERR_INVALID_ARG. */
int moe_selftest_wait(void* ws, int64_t limit_ns, cudaStream_t stream);

/* Static name of a return code. */
const char* moe_strerror(int code);

/* MOE_ABI_VERSION of the library. */
int moe_abi_version(void);

/* The cudaError_t value behind the last MOE_ERR_CUDA returned on this host thread (0 if
 * none). */
int moe_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
