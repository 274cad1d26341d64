/*
 * kosmos.h -- C ABI of the GB300 (sm_103a) self-scheduling persistent kernels.
 *
 * The method: "KOSMOS: Self-scheduling Persistent Kernels for
 * Communication-Compute Overlap" (arXiv 2611.07477, abstract), explained on
 * learnaivisually.com ("KOSMOS -- Self-scheduling persistent kernels -- What
 * does it mean?").  Each fused operator is ONE persistent launch with one CTA
 * resident per SM; CTAs take work by atomically claiming the next entry of a
 * shared queue ("rail") that is ordered by consumer demand, and switch role
 * (mover / builder / reducer) when their own work runs out (explainer,
 * paragraphs "KOSMOS removes the manager" and "Role switching only works").
 *
 * Emulated ranks.  On one GPU the P "ranks" are P shard buffers in the same
 * HBM; a transfer between ranks is a device-to-device copy made by mover CTAs
 * inside the persistent kernel.  Nothing here talks to a second GPU.
 *
 * Conventions for every entry point:
 *   - All tensors are row-major, caller-owned DEVICE memory; every pointer must
 *     be 16-byte aligned.  bf16 = IEEE bfloat16 bit patterns (uint16).
 *   - `stream` is a cudaStream_t passed as void*; NULL = legacy default stream.
 *     Calls are stream-ordered and asynchronous: a KOSMOS_OK return means the
 *     arguments were accepted and the work was enqueued.
 *   - Argument errors are detected on the host, return synchronously and
 *     launch nothing.  Errors found on the device (a bounded wait that ran
 *     out, a device-side check) are written to the workspace status word and
 *     read back with kosmos_status_sync().
 *   - The library allocates no memory and keeps no state between calls other
 *     than cached device attributes and driver entry points.  The workspace
 *     holds ticket counters, readiness flags, the status word, the optional
 *     role trace and (GEMM+RS only) the per-rank partial products.  One
 *     workspace serves one stream at a time; it must be zeroed once with
 *     kosmos_workspace_init() before first use and again after any call whose
 *     status was not KOSMOS_OK.  Successful calls leave it ready for the next.
 */
#ifndef KOSMOS_H
#define KOSMOS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KOSMOS_MAX_P 8

#if defined(__GNUC__)
#define KOSMOS_API __attribute__((visibility("default")))
#else
#define KOSMOS_API
#endif

typedef enum kosmos_status {
    KOSMOS_OK = 0,
    KOSMOS_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, bad shape, P out of range */
    KOSMOS_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement */
    KOSMOS_ERR_WORKSPACE = 3,    /* workspace missing or smaller than kosmos_workspace_bytes() */
    KOSMOS_ERR_CUDA = 4,         /* a CUDA runtime call failed (launch, attribute, copy) */
    KOSMOS_ERR_TIMEOUT = 5,      /* device: a readiness wait exceeded opts.wait_limit_ns */
    KOSMOS_ERR_DEVICE = 6        /* device: an internal pipeline wait or check failed */
} kosmos_status;

typedef enum kosmos_dtype {
    KOSMOS_BF16 = 0,
    KOSMOS_MXFP8_E4M3 = 1        /* E4M3 bytes + one E8M0 scale byte per 32 K-elements */
} kosmos_dtype;

typedef enum kosmos_op {
    KOSMOS_OP_AG_GEMM = 0,
    KOSMOS_OP_GEMM_RS = 1,
    KOSMOS_OP_MOE_FWD = 2
} kosmos_op;

/* Scheduling policy.  SELF is the method; FIXED and UNFUSED are the two
 * baselines the explainer contrasts it with (paragraph "Picture a restaurant
 * kitchen": a manager fixes the mover/builder split at launch; paragraph
 * "Start with the problem": transfer, then multiply). */
enum {
    KOSMOS_SCHED_SELF = 0,     /* one-way role switching driven by readiness */
    KOSMOS_SCHED_FIXED = 1,    /* static partition: movers/reducers never switch */
    KOSMOS_SCHED_UNFUSED = 2   /* separate copy (or reduce) launch and GEMM launch */
};

/* Output order of the reduce-scatter tile rails (explainer, "Role switching
 * only works": band by band across every rank's chunk; the row-by-row order
 * is the ablation). */
enum { KOSMOS_ORDER_BAND = 0, KOSMOS_ORDER_ROW = 1 };

/* Fault injection bits for tests (host-set; the failure is a flag that is
 * never released, so the waiting side's bounded wait runs out). */
#define KOSMOS_INJECT_DROP_TRANSFER 0x1ull  /* AG: transfer ticket (inject >> 32) never releases its flag */
#define KOSMOS_INJECT_DROP_PARTIAL  0x2ull  /* RS: rank (inject >> 32) never signals its partial tiles */
#define KOSMOS_INJECT_DROP_DISPATCH 0x8ull  /* MoE forward: the DISPATCH entry of main-rail ticket (inject >> 32)
                                               copies its rows but never counts them as arrived */
#define KOSMOS_INJECT_DROP_ARRIVAL  0x10ull /* AG host-input call: shard (inject >> 32) is copied to the device
                                               but its arrival words are never written */
/* MoE debug mode: every expert is the identity map (no expert GEMMs; the
 * pushed rows are the dispatched token rows), which isolates router,
 * dispatch, push and fold.  Not a fault: the output is x * sum of gates. */
#define KOSMOS_INJECT_IDENTITY_EXPERTS 0x4ull

typedef struct kosmos_opts {
    int32_t sched;            /* KOSMOS_SCHED_* */
    int32_t n_comm0;          /* CTAs that start as movers (AG) / first reducers per rank (RS: self-scheduled,
                                 they build until their rank has a ready reduce entry); -1 = default */
    int32_t fixed_comm_ctas;  /* FIXED: size of the static mover / reducer crew (per rank for RS); -1 = n_comm0 */
    int32_t order;            /* KOSMOS_ORDER_* (GEMM+RS) */
    int32_t num_ctas;         /* -1 = one CTA per SM */
    int32_t trace;            /* nonzero: record a per-entry role trace in the workspace */
    int32_t cta_pair;         /* AG (bf16, MXFP8) / RS tiles: 1 = 256x256 per SM pair (tcgen05 cta_group::2),
                                 0 = 128x256 per SM; -1 = default (pairs) */
    int32_t plain_launch;     /* 0 = cooperative launch (the driver guarantees every CTA is resident);
                                 1 = the same grid as a plain launch, for profilers that cannot replay
                                 cooperative cluster launches.  The grid never exceeds the occupancy
                                 limit, so on an otherwise idle GPU every CTA is resident; if one is
                                 not, the others' bounded waits run out and the call reports
                                 KOSMOS_ERR_TIMEOUT. */
    uint64_t wait_limit_ns;   /* bound on every readiness wait; 0 = 2e9 (2 s) */
    uint64_t inject;          /* KOSMOS_INJECT_* bits | (argument << 32); 0 = none */
    int64_t tail_split;       /* bf16 AG: the last tail_split tiles of the tile rail run as two K halves
                                 each (two entries whose fp32 partials are added through the
                                 workspace); 0 = none; -1 = one wave (the number of tile engines,
                                 i.e. SM pairs or SMs, that build).  At most 256; needs k >= 128.
                                 The workspace holds 256 KB per split tile. */
    int64_t link_gbs;         /* emulated link bandwidth in GB/s (1e9 bytes/s) for the bytes that would
                                 cross GPU-to-GPU links (all-gather: remote shard pieces; GEMM+RS: the
                                 partial tiles of other ranks).  One link for the emulated traffic: a
                                 transfer is released no earlier than a pipe of this rate, busy from
                                 the launch's first link transfer on, would have delivered it.
                                 0 = uncapped; else 1..1000000.  MoE: must be 0. */
} kosmos_opts;

/* Fills *opts with the defaults (SELF, band order, all SMs, no trace). */
KOSMOS_API void kosmos_default_opts(kosmos_opts *opts);

/* Number of SMs of the current device (the persistent grid size), or -1. */
KOSMOS_API int kosmos_num_sms(void);

/* Workspace size in bytes for one call of `op` with these sizes (same
 * meaning as the op's own arguments; MoE: m = tokens, n = hidden, k = inter,
 * P = EP ranks).  opts may be NULL.  Returns 0 for invalid sizes. */
KOSMOS_API size_t kosmos_workspace_bytes(int op, int P, int64_t m, int64_t n, int64_t k, int dtype,
                              const kosmos_opts *opts);

/* Zeroes the workspace (stream-ordered). */
KOSMOS_API kosmos_status kosmos_workspace_init(void *ws, size_t ws_bytes, void *stream);

/*
 * All-gather + GEMM  (explainer, "Start with the problem": gather the input
 * pieces from the other ranks before the multiplication; "Role switching only
 * works": builders start on the local shard while movers fetch the remote
 * shards in the order the multiplication consumes them).
 *
 *   Y = concat_{r=0..P-1}(X_r) . W          computed from rank 0's view
 *
 *   x_shards[r]  : P pointers, X_r [m_per_shard, k]; x_shards[0] is the local shard.
 *                  BF16: bf16.  MXFP8: E4M3 bytes.
 *   x_scales[r]  : MXFP8 only: E8M0 scales of X_r (one per row and 32
 *                  consecutive K-elements) in the MMA-tiled layout below; else NULL.
 *   w            : [k, n] (BF16: bf16; MXFP8: E4M3 bytes).
 *   w_scales     : MXFP8 only: E8M0 scales of W (one per column and 32
 *                  consecutive K-elements), MMA-tiled with the columns of W as
 *                  scale rows; else NULL.
 *   MMA-tiled scale layout: for R scale rows and K, the scale of (row r,
 *   K-block b = k/32) is at byte ((r/128)*(K/128) + b/4)*512 + (r%32)*16 +
 *   ((r/32)%4)*4 + b%4; size ceil(R/128)*128*K/32 bytes.  kosmos_mxfp8_quantize
 *   writes it.  The MXFP8 workspace also holds the gathered scale blocks.
 *   x_gathered   : out, [P*m_per_shard, k], same element type as X: the
 *                  gathered input (kept for the backward pass).
 *   y            : out, [P*m_per_shard, n] bf16, fp32 accumulation, one
 *                  round-to-nearest-even per element.
 *   Requirements: 1 <= P <= 8, m_per_shard >= 1, k % 64 == 0, n % 8 == 0
 *   (MXFP8: k % 128 == 0, n % 16 == 0).
 */
KOSMOS_API kosmos_status kosmos_ag_gemm(const void *const *x_shards, const void *const *x_scales, int P,
                             int64_t m_per_shard, int64_t k, int64_t n,
                             const void *w, const void *w_scales, int dtype,
                             void *x_gathered, void *y, void *ws, size_t ws_bytes,
                             const kosmos_opts *opts, void *stream);

/* The tile-rail split (number of trailing tiles run as two K halves) and
 * the tile height (256: SM pairs, 128: one SM per tile) that kosmos_ag_gemm
 * would use for these sizes and options on the current device; the values
 * to pass to kosmos_rail_decode.  Returns 0, or -1 for invalid arguments. */
KOSMOS_API int kosmos_ag_tile_plan(int P, int64_t m_per_shard, int64_t k, int64_t n, int dtype,
                                   const kosmos_opts *opts, int64_t *tail_split, int *tile_m);

/*
 * All-gather + GEMM with the shards in host memory (BF16): the copies to the
 * device run on h2d_stream, shard by shard (the local shard first), each into
 * its slot of x_gathered and followed by a 4-byte copy that sets its arrival
 * word (from a pinned word the library allocates once); the kernel's tiles
 * read a shard as soon as its word is set, so the copies overlap the
 * multiplication, and its movers copy each shard on into x_dev[r] beside the
 * tiles.  Each shard's output rows go back on d2h_stream in two groups of
 * tile rows, each as soon as its tiles are written (a stream wait on the
 * group's tile count).  The kernel is enqueued before the copies.  Same
 * result as kosmos_ag_gemm on x_dev (Y and x_gathered bit for bit).
 *   x_host[r]     : X_r [m_per_shard, k] bf16 in pinned host memory.
 *   x_dev[r]      : out, device buffers [m_per_shard, k] that receive X_r.
 *   y_dev, y_host : [P * m_per_shard, n] bf16, device and pinned host.
 *   stream        : the kernel's stream; on return, work enqueued on it
 *                   waits for both copy streams, so its completion means the
 *                   whole call (copies included) is done.
 *   h2d_stream, d2h_stream : two further streams, distinct from `stream`.
 *   Requirements as kosmos_ag_gemm (BF16); opts.tail_split is ignored.  If
 *   the kernel fails, the output waits are released (the status tells).
 */
KOSMOS_API kosmos_status kosmos_ag_gemm_host(const void *const *x_host, void *const *x_dev, int P,
                             int64_t m_per_shard, int64_t k, int64_t n, const void *w, void *x_gathered,
                             void *y_dev, void *y_host, void *ws, size_t ws_bytes, const kosmos_opts *opts,
                             void *stream, void *h2d_stream, void *d2h_stream);

/*
 * GEMM + reduce-scatter  (explainer, "Start with the problem": scatter and
 * add the partial results; "KOSMOS removes the manager": builders join the
 * reduction when the multiplication tiles run out).
 *
 *   Y = sum_{r=0..P-1} X_r . W_r,  chunk c = rows [c*m/P, (c+1)*m/P) of Y
 *
 *   x_shards[r]  : X_r [m, k_per_rank]; BF16: bf16; MXFP8: E4M3 bytes.
 *   x_scales[r]  : MXFP8 only: E8M0 scales of X_r (one per row and 32 K),
 *                  MMA-tiled as for kosmos_ag_gemm; else NULL.
 *   w_shards[r]  : W_r [k_per_rank, n]; BF16: bf16; MXFP8: E4M3 bytes.
 *   w_scales[r]  : MXFP8 only: E8M0 scales of W_r (one per column and 32 K),
 *                  MMA-tiled with the columns as scale rows; else NULL.
 *   y_chunks[c]  : out, [m/P, n] bf16: each rank's partial (fp32 accumulation)
 *                  rounded once to bf16, the P partials summed in fp32 in rank
 *                  order 0..P-1, the sum rounded once to bf16.
 *   Requirements: 1 <= P <= 8, m % P == 0, k_per_rank % 64 == 0, n % 8 == 0;
 *   MXFP8: SM-pair tiles only (cta_pair != 0), (m/P) % 128 == 0,
 *   k_per_rank % 128 == 0, n % 16 == 0.
 */
KOSMOS_API kosmos_status kosmos_gemm_rs(const void *const *x_shards, const void *const *x_scales,
                             const void *const *w_shards, const void *const *w_scales, int P,
                             int64_t m, int64_t k_per_rank, int64_t n, int dtype,
                             void *const *y_chunks, void *ws, size_t ws_bytes,
                             const kosmos_opts *opts, void *stream);

/*
 * MoE expert layer forward in one launch  (abstract: "runs an entire expert
 * layer, from router to fold, in one launch per direction"; explainer,
 * "KOSMOS removes the manager": in the combine step a CTA pushes any ready
 * result and otherwise builds a tile).
 *
 *   x_shards[q]   : EP rank q's tokens [tokens/P, hidden] bf16 (token t lives on
 *                   rank t / (tokens/P)).
 *   w_router      : [hidden, n_experts] bf16 (the router is bf16 for both dtypes).
 *   w_gate[q], w_up[q] : rank q's experts [n_experts/P, hidden, inter]; BF16: bf16,
 *                   MXFP8: E4M3 bytes.
 *   w_down[q]     : [n_experts/P, inter, hidden]; bf16 or E4M3 bytes.
 *   w_*_scales[q] : MXFP8 only (else NULL): the E8M0 scales of rank q's experts,
 *                   one after the other, each expert's matrix quantised along its
 *                   K dimension (hidden for gate/up, inter for down; one scale per
 *                   column and 32 K) and MMA-tiled with the columns as scale rows
 *                   (kosmos_mxfp8_quantize with along_cols = 0 per expert):
 *                   inter*hidden/32 bytes per expert.
 *   dtype         : KOSMOS_BF16 or KOSMOS_MXFP8_E4M3.  MXFP8 quantises the token
 *                   rows (along hidden) and the SwiGLU activations h (along
 *                   inter) inside the launch with the rule of kosmos_mxfp8_quantize
 *                   (h from its fp32 value); the expert GEMMs are block-scaled
 *                   with fp32 accumulation.
 *   y_shards[q]   : out, [tokens/P, hidden] bf16.
 *   topk_idx      : out, [tokens, topk] int32, descending router score, ties to the lower index.
 *   topk_gate     : out, [tokens, topk] fp32, softmax probabilities renormalised over the top-k.
 *   expert_counts : out, [n_experts] int32.
 *   dispatch_pos  : out, [tokens, topk] int32: row of (t, k) in the expert-ordered
 *                   receive buffer (experts ascending, then tokens ascending),
 *                   counted without padding (MXFP8 stores each expert's rows
 *                   from a 128-row boundary: physical row = dispatch_pos -
 *                   unpadded offset of the expert + padded offset).
 *   Requirements: P in {1..8}, n_experts % P == 0, n_experts % 64 == 0,
 *   n_experts <= 256, 1 <= topk <= 8, topk <= n_experts, tokens % P == 0,
 *   hidden % 256 == 0, inter % 128 == 0.  MXFP8: no identity-expert
 *   injection (KOSMOS_ERR_UNSUPPORTED).  Workspace: kosmos_moe_workspace_bytes.
 */
KOSMOS_API kosmos_status kosmos_moe_fwd(const void *const *x_shards, const void *w_router, int P,
                             int64_t tokens, int64_t hidden, int n_experts, int topk, int64_t inter,
                             const void *const *w_gate, const void *const *w_gate_scales,
                             const void *const *w_up, const void *const *w_up_scales,
                             const void *const *w_down, const void *const *w_down_scales, int dtype,
                             void *const *y_shards,
                             int32_t *topk_idx, float *topk_gate, int32_t *expert_counts,
                             int32_t *dispatch_pos, void *ws, size_t ws_bytes,
                             const kosmos_opts *opts, void *stream);

/* Workspace size in bytes for kosmos_moe_fwd with these sizes and dtype (opts
 * may be NULL).  Returns 0 for invalid sizes or dtype. */
KOSMOS_API size_t kosmos_moe_workspace_bytes(int P, int64_t tokens, int64_t hidden, int n_experts, int topk,
                                             int64_t inter, int dtype, const kosmos_opts *opts);

/* Device views into a MoE workspace after a call (for checks and tools).
 * R = tokens*topk rows (BF16) or the padded row capacity (MXFP8: each expert's
 * rows from a 128-row boundary, row order as in the receive buffer):
 *   what 0: router logits [tokens, n_experts] fp32 (as the kernel computed them)
 *        1: receive buffer [R, hidden], bf16 or E4M3 bytes, expert-ordered rows
 *        2: SwiGLU activations h [R, inter], bf16 or E4M3 bytes, same row order
 *        3: expert outputs [R, hidden] bf16, same row order
 *        4: pushed slots [tokens, topk, hidden] bf16
 *        5: expert offsets [n_experts + 1] int32 (MXFP8: padded)
 *        6: role trace records (only for a workspace sized with opts.trace)
 *        7: MXFP8: receive-row scales, MMA-tiled (K = hidden)
 *        8: MXFP8: quantised tokens [tokens, hidden] E4M3 bytes
 *        9: MXFP8: their scales [tokens, hidden/32], row-major
 * Returns KOSMOS_OK and sets *ptr / *bytes, or KOSMOS_ERR_INVALID_ARG. */
KOSMOS_API kosmos_status kosmos_moe_debug_view(int what, int P, int64_t tokens, int64_t hidden, int n_experts,
                                               int topk, int64_t inter, int dtype, void *ws, void **ptr,
                                               int64_t *bytes);

/*
 * MoE expert layer backward in one launch  (abstract: "one launch per
 * direction").  Gradients of a BF16 kosmos_moe_fwd call with its top-K
 * routing held fixed (L = <dout, out>):
 *   dgate[t][k] = <dout_t, y[t][k]>, dy[t][k] = gate[t][k] dout_t,
 *   dh = dy W_down^T, dg = dh * u * silu'(g), du = dh * silu(g),
 *   dx_t = sum_k (dg W_gate^T + du W_up^T) + dl_t W_router^T,
 *   dl = softmax backward of the renormalised top-K gates,
 *   dW_gate[e] = x^T dg, dW_up[e] = x^T du, dW_down[e] = h^T dy (sums over
 *   the slots routed to e), dW_router = x^T dl (all tokens).
 *   Arguments as for kosmos_moe_fwd, plus:
 *   topk_idx, topk_gate : the forward's outputs.
 *   fwd_ws        : the forward's workspace, untouched since that call (it
 *                   holds the saved context: expert-ordered token rows, g, u,
 *                   h, the per-slot outputs, logits, dispatch tables).
 *   dy_shards[q]  : dout of rank q's tokens [tokens/P, hidden] bf16.
 *   dx_shards[q]  : out, [tokens/P, hidden] bf16: the expert and router parts
 *                   summed in fp32 (slots in k order, then the router part),
 *                   one rounding.
 *   dw_router     : out, [hidden, n_experts] fp32.
 *   dw_gate[q], dw_up[q] : out, [n_experts/P, hidden, inter] bf16;
 *   dw_down[q]    : out, [n_experts/P, inter, hidden] bf16 (fp32 sums over
 *                   each expert's rows, one rounding).
 *   Intermediates dy, dg, du, dl and the slot gradients are bf16.
 *   Requirements: those of kosmos_moe_fwd, inter % 256 == 0 and
 *   (tokens/P) % 64 == 0; SELF schedule, no link cap, no injection.
 *   Workspace: kosmos_moe_bwd_workspace_bytes.
 */
KOSMOS_API kosmos_status kosmos_moe_bwd(const void *const *x_shards, const void *w_router, int P,
                             int64_t tokens, int64_t hidden, int n_experts, int topk, int64_t inter,
                             const void *const *w_gate, const void *const *w_up,
                             const void *const *w_down, const int32_t *topk_idx,
                             const float *topk_gate, const void *fwd_ws, size_t fwd_ws_bytes,
                             const void *const *dy_shards, void *const *dx_shards, float *dw_router,
                             void *const *dw_gate, void *const *dw_up, void *const *dw_down,
                             void *ws, size_t ws_bytes, const kosmos_opts *opts, void *stream);

/* Workspace size in bytes for kosmos_moe_bwd (opts may be NULL); 0 for invalid sizes. */
KOSMOS_API size_t kosmos_moe_bwd_workspace_bytes(int P, int64_t tokens, int64_t hidden, int n_experts, int topk,
                                                 int64_t inter, const kosmos_opts *opts);

/* Device views into a backward workspace after a call (R = the padded row
 * capacity: each expert's rows from a 16-row boundary, experts ascending):
 *   what 0: dy [R, hidden] bf16   1: dg [R, inter] bf16   2: du [R, inter] bf16
 *        3: dx of the expert rows [R, hidden] bf16   4: dx slots [tokens, topk, hidden] bf16
 *        5: dgate [tokens, topk] fp32   6: dl [tokens, n_experts] bf16
 *        7: dx of the router path [tokens, hidden] fp32
 *        8: role trace records (only for a workspace sized with opts.trace)
 * Returns KOSMOS_OK and sets *ptr / *bytes, or KOSMOS_ERR_INVALID_ARG. */
KOSMOS_API kosmos_status kosmos_moe_bwd_debug_view(int what, int P, int64_t tokens, int64_t hidden, int n_experts,
                                                   int topk, int64_t inter, void *ws, void **ptr,
                                                   int64_t *bytes);

/*
 * MXFP8 quantiser for the MXFP8 all-gather+GEMM operands.  For each block of
 * 32 consecutive K-elements: e = smallest integer with blockmax <= 448 * 2^e
 * (clamped to [-127, 127]; an all-zero block takes e = 0), scale byte e + 127,
 * element byte = E4M3(x / 2^e) rounded to nearest even.
 *   along_cols = 1: x [rows, cols], blocks along a row (activations X[m, k]);
 *                   scale rows = rows, K = cols.
 *   along_cols = 0: x [rows, cols], blocks along a column (weights W[k, n]);
 *                   scale rows = cols, K = rows.
 *   q keeps x's [rows, cols] layout; scales are written in the MMA-tiled
 *   layout described at kosmos_ag_gemm (ceil(R/128)*128*K/32 bytes; padding
 *   rows get the scale byte 127).  Requirements: K % 128 == 0.
 */
KOSMOS_API kosmos_status kosmos_mxfp8_quantize(const void *x, int64_t rows, int64_t cols, int along_cols,
                                    void *q, void *scales, void *stream);

/* Size in bytes of the scratch array that kosmos_ag_gemm_noalloc uses. */
#define KOSMOS_STATIC_WS_BYTES 65536

/*
 * All-gather + GEMM without a workspace, for callers that cannot allocate
 * device memory (a plugin behind an operator interface with no scratch
 * argument, or code that must not call the device allocator while it runs).
 * The KOSMOS pages have no counterpart to this entry point: it is a
 * packaging variant of kosmos_ag_gemm with the same arguments, minus ws and
 * ws_bytes, and the same results.
 *
 * Scratch: a file-scope __device__ array of KOSMOS_STATIC_WS_BYTES (64 KiB)
 * inside the library, which every GPU that loads the library holds until the
 * process exits.  Calls whose workspace would exceed it (see
 * kosmos_workspace_bytes) return KOSMOS_ERR_WORKSPACE; opts.trace is not
 * supported (KOSMOS_ERR_UNSUPPORTED).  The 8-rank 1024 x 8192 x 3584 call
 * needs 1536 bytes.
 * Set-up: every call looks up the array's device address in the current
 * device's context (cudaGetSymbolAddress; nothing is cached, so a reset device
 * or a new context is picked up).  The first lookup in a context loads the
 * module, so make the first call on a device before any stream capture.
 * Every call shares the one array per device: each call first clears the part
 * it uses on `stream`, so calls that overlap on the GPU (different streams,
 * or different host threads without ordering) race and give wrong results.
 * Device-side wait failures are written to the array's status word like a
 * workspace's: read them with kosmos_noalloc_status_sync() before the next
 * call on the device clears the array.  Allocates no memory: no cudaMalloc,
 * cudaFree or allocating library routine.
 */
KOSMOS_API kosmos_status kosmos_ag_gemm_noalloc(const void *const *x_shards, const void *const *x_scales, int P,
                                                int64_t m_per_shard, int64_t k, int64_t n,
                                                const void *w, const void *w_scales, int dtype,
                                                void *x_gathered, void *y, const kosmos_opts *opts,
                                                void *stream);

/* Synchronises `stream`, then returns the device status of the last call
 * that used `ws` (KOSMOS_OK, KOSMOS_ERR_TIMEOUT or KOSMOS_ERR_DEVICE) and,
 * if failing_entry is not NULL, the ticket of the entry that failed (-1 if
 * none). */
KOSMOS_API kosmos_status kosmos_status_sync(void *ws, void *stream, int64_t *failing_entry);

/* kosmos_status_sync for kosmos_ag_gemm_noalloc: synchronises `stream`, then
 * returns the device status of the last no-allocation call on the current
 * device (KOSMOS_OK, KOSMOS_ERR_TIMEOUT or KOSMOS_ERR_DEVICE) and, if
 * failing_entry is not NULL, the ticket of the entry that failed (-1 if none).
 * Valid until the next kosmos_ag_gemm_noalloc call on the device, which
 * clears the status; KOSMOS_ERR_CUDA if the library's array cannot be found
 * in the current context.  Allocates no memory. */
KOSMOS_API kosmos_status kosmos_noalloc_status_sync(void *stream, int64_t *failing_entry);

/* Role trace.  When opts.trace is set, every claimed entry appends one record
 * to its CTA's ring in the workspace:
 *   int64 t_claim, t_ready, t_done  (%globaltimer, ns)
 *   int32 kind (1 TRANSFER, 2 TILE, 3 REDUCE, 4 ROUTE, 5 DISPATCH, 6 TILE_GU,
 *               7 TILE_D, 8 PUSH, 9 FOLD), ticket, cta, pad.
 * kosmos_trace_info() gives the ring's device address, the per-CTA capacity
 * and the CTA count for the workspace of a call with these sizes. */
typedef struct kosmos_trace_rec {
    int64_t t_claim, t_ready, t_done;
    int32_t kind, ticket, cta, pad;
} kosmos_trace_rec;

KOSMOS_API kosmos_status kosmos_trace_info(int op, int P, int64_t m, int64_t n, int64_t k, int dtype,
                                const kosmos_opts *opts, void *ws, void **records,
                                int32_t *per_cta_capacity, int32_t *num_ctas);

/* Rail decode, for checking ticket order against an independent rail
 * builder.  Writes 4 int32 {kind, a, b, c} per ticket of one rail:
 *   op AG_GEMM: rail 0 = transfers {1, shard, piece, part} (128-row pieces in
 *               32-row parts); rail 1 = tiles {2, shard, tile_row, tile_col}.
 *               args: m = m_per_shard.
 *   op GEMM_RS: rail 0 = the tile rail shared by all ranks
 *               {2, q * P + chunk, band, tile_col} (rank q's partial);
 *               rail 1 = reductions of rank `rank` {3, rank, band, tile_col}.
 * tile_m = tile (band) height in rows: 128 (one SM per tile) or 256 (SM pairs).
 * split = AG tile rail only: trailing tiles run as two K halves (entries
 * {10, shard, tile-row, 2 * tile-col + half}); ignored for GEMM+RS.
 * out is HOST memory of max_entries*4 int32; returns the rail length or -1.
 * Runs the same decode functions the kernels use, compiled for the host. */
KOSMOS_API int64_t kosmos_rail_decode(int op, int P, int64_t m, int64_t n, int order, int rank, int rail,
                           int tile_m, int64_t split, int32_t *out, int64_t max_entries);

/* Same decode executed by a device kernel (out is DEVICE memory). */
KOSMOS_API int64_t kosmos_rail_decode_device(int op, int P, int64_t m, int64_t n, int order, int rank,
                                  int rail, int tile_m, int64_t split, int32_t *out, int64_t max_entries,
                                  void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KOSMOS_H */
