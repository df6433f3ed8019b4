/*
 * moe.h -- C ABI of the GB300 (sm_103a) MegaMoE expert path, expert parallelism 1.
 *
 * The MegaMoE guide (Primus technical guide "MegaMoE") describes the layer as a
 * fused router (score function + group-limited top-k + aux score) followed by
 * dispatch_grouped_gemm -> SwiGLU -> grouped_gemm_combine, with weights
 * w1 [g, 2I, H] (gate rows, then up rows) and w2 [g, H, I] (section "Design:
 * two stages + weight modules"), and names the one-shot op
 * fused_mega_moe(x, topk_idx, topk_weights, w1, w2, group). On one GPU the
 * dispatch / combine all-to-all becomes a local row gather and a weighted sum,
 * and g = E (all experts are local).
 *
 * Conventions for every entry point:
 *   - Pointers named x, w_r, ..., y and ws are DEVICE pointers owned by the
 *     caller; the library never allocates, frees or keeps them. Tensors are
 *     dense row-major and 16-byte aligned. bf16 means IEEE bfloat16 storage.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Calls only
 *     enqueue work on it and return; they never synchronise the device, except
 *     moe_get_device_error, which waits for `stream`.
 *   - Argument errors are reported synchronously by the return value, before
 *     anything is enqueued. Data errors found on the device (an expert index
 *     outside [0, E), a wait that ran out of time) set bits in the error word
 *     of the workspace; read them with moe_get_device_error.
 *   - Limits: H and I multiples of 8; 1 <= k <= 32; k <= E <= 1024; T*k < 2^31.
 *     Outside them a call returns MOE_ERR_UNSUPPORTED. The device must be an
 *     sm_103 GPU.
 *   - The workspace `ws` (moe_workspace_size bytes, 256-byte aligned) holds the
 *     routing metadata and intermediates. Zero its first 256 bytes once before
 *     first use (moe_workspace_init). Calls that share a workspace must be
 *     ordered on one stream; stages read what earlier stages left there.
 *   - Training: a shape with flags = MOE_SHAPE_TRAINING sizes the workspace
 *     for the backward as well. The backward entry points read the routing
 *     metadata the forward left in the workspace, so a training step runs its
 *     forward and backward on one workspace, in order, on one stream.
 */
#ifndef MOE_GB300_MOE_H
#define MOE_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,      /* null / misaligned pointer, bad size or config */
    MOE_ERR_UNSUPPORTED = 2,      /* outside the limits above, or not an sm_103 device */
    MOE_ERR_CUDA = 3,             /* a CUDA runtime call failed */
    MOE_ERR_WORKSPACE = 4,        /* ws_bytes smaller than moe_workspace_size */
    MOE_ERR_DEVICE_FLAGGED = 5    /* moe_get_device_error found a non-zero error word */
} moe_status_t;

/* Bits of the device error word. */
#define MOE_DEVERR_BAD_EXPERT_INDEX 0x1  /* a topk_idx entry outside [0, E): that slot was dropped */
#define MOE_DEVERR_WAIT_TIMEOUT     0x2  /* a pipeline wait ran out of time: outputs are invalid */
#define MOE_DEVERR_CAPACITY         0x4  /* expert parallelism: a routed row beyond a block's capacity was dropped */

typedef struct moe_shape {
    int64_t T;   /* tokens */
    int64_t H;   /* hidden size */
    int64_t I;   /* expert intermediate size (w1 has 2I rows per expert) */
    int64_t E;   /* experts */
    int32_t k;   /* experts per token */
    int32_t flags;  /* 0, or an OR of the MOE_SHAPE_* flags below */
} moe_shape_t;

/* moe_shape_t.flags: the workspace also holds the backward's intermediates. */
#define MOE_SHAPE_TRAINING 0x1
/* moe_shape_t.flags: the workspace also holds the MXFP8 path's quantized x and a. */
#define MOE_SHAPE_MXFP8 0x2
/* moe_shape_t.flags: the w1 / w2 pointers given to moe_dispatch_gemm1,
 * moe_swiglu_gemm2_combine and moe_forward are in the tile-packed layout of
 * moe_pack_weights (bf16 forward only: not with MOE_SHAPE_TRAINING or
 * MOE_SHAPE_MXFP8, which return MOE_ERR_UNSUPPORTED). */
#define MOE_SHAPE_PACKED_WEIGHTS 0x4

#define MOE_SCORE_SOFTMAX 0
#define MOE_SCORE_SIGMOID 1

typedef struct moe_router_cfg {
    int32_t score_fn;    /* MOE_SCORE_SOFTMAX or MOE_SCORE_SIGMOID */
    int32_t normalize;   /* 1: divide the k weights by their score sum */
    float scale;         /* multiply the k weights (1.0 for none) */
    int32_t n_group;     /* 1: no group limit; else E % n_group == 0 and n_group <= 32 */
    int32_t topk_group;  /* groups kept per token (1 <= topk_group <= n_group) */
    int32_t group_topn;  /* largest selection scores summed per group score (>= 1) */
} moe_router_cfg_t;

/* Byte offsets of the regions inside the workspace (for inspection and tests). */
typedef struct moe_ws_layout {
    size_t err;        /* int32 error word (first 4 bytes) */
    size_t counts;     /* int32 [E]   rows routed to each expert */
    size_t offsets;    /* int32 [E+1] exclusive prefix sum of counts */
    size_t mt_prefix;  /* int32 [E+1] prefix sum of ceil(counts/256) (row tiles) */
    size_t perm_slot;  /* int32 [T*k] flat slot t*k+j of each routed row */
    size_t row_of;     /* int32 [T*k] routed row of each slot, -1 if dropped */
    size_t meta;       /* int32 [ceil(T*k/1024), E] per-chunk expert histograms (scratch) */
    size_t router;     /* router scratch: fp32 split-K partial logits [s,T,E], bf16 split of w_r [3,E,H], sums, counts */
    size_t a;          /* bf16 [T*k, I] SwiGLU activations (moe_forward only) */
    size_t obuf;       /* bf16 [T*k, H] weighted expert outputs in routed-row order;
                          before stage 2 writes them, stage 1 (outside training)
                          holds x's rows dispatched into routed order here; the
                          backward's dX rows (unweighted, routed order) reuse it */
    size_t combine;    /* int32 [T, ceil(H/256)] counters of stage 2's fused k-way sum, used
                          when T*k <= 64 E (set by moe_routing_metadata) */
    /* training workspaces only (flags = MOE_SHAPE_TRAINING), else equal to total: */
    size_t dh;         /* bf16 [T*k, 2I] gradient of h = [gate | up], routed order */
    size_t aw;         /* bf16 [T*k, I] routing weight times a, routed order */
    size_t dtw_part;   /* fp32 [ceil(I/256), T*k] partial routing-weight gradients */
    size_t dlogits;    /* fp32 [T, E] gradient of the router logits */
    size_t xp;         /* bf16 [T*k, H] x rows in routed order (training stage 1's dispatch) */
    size_t dyp;        /* bf16 [T*k, H] dY rows in routed order (the backward's dispatch) */
    size_t dwr_part;   /* fp32 [8, E, H] partial sums of the router weight gradient */
    /* MXFP8 workspaces only (flags & MOE_SHAPE_MXFP8), else equal to total: */
    size_t x_codes;    /* E4M3 [T*k, H] quantized x rows in routed order (the MXFP8 dispatch) */
    size_t x_scales;   /* E8M0, k-block-major over T*k rows (rows4(T*k)*H/32 bytes) */
    size_t a_codes;    /* E4M3 [T*k, I] quantized SwiGLU output, routed order (moe_forward_mx) */
    size_t a_scales;   /* E8M0, k-block-major over T*k rows (rows4(T*k)*I/32 bytes) */
    /* training + MXFP8 workspaces only, else equal to total: */
    size_t mx_wgrad;   /* the MXFP8 weight gradients' operands, quantized along the routed rows */
    size_t total;      /* == moe_workspace_size */
} moe_ws_layout_t;

/* Bytes of workspace needed for `shape`. Host-only; touches no device. */
moe_status_t moe_workspace_size(const moe_shape_t *shape, size_t *bytes);

/* Region offsets of the workspace for `shape`. Host-only. */
moe_status_t moe_workspace_layout(const moe_shape_t *shape, moe_ws_layout_t *layout);

/* Zero the workspace header (error word and counters) on `stream`. */
moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, void *stream);

/*
 * Fused router (MegaMoE guide, opening section: score function + group-limited
 * top-k + aux score; the aux load-balance value is computed and returned).
 *
 *   l[t,e]   = sum_h x[t,h] * w_r[e,h] (+ logit_offset[e]), fp32
 *   s[t,:]   = softmax(l[t,:]) or sigmoid(l[t,:])
 *   sel[t,e] = s[t,e] + sel_bias[e]          (selection only, never the weights)
 *   groups   = (n_group > 1) keep the topk_group groups with the largest sum of
 *              their group_topn best sel values; other experts are ineligible
 *   topk_idx = the k eligible experts with the largest sel, best first; ties go
 *              to the lower expert (and group) index
 *   topk_w   = s of those experts, / their sum if normalize, * scale
 *   aux      = E * sum_e (c_e / (T k)) * (1/T) sum_t s[t,e]   (c_e = rows of e)
 *
 * x bf16 [T,H]; w_r fp32 [E,H]; logit_offset, sel_bias fp32 [E] or NULL;
 * topk_idx int32 [T,k], topk_w fp32 [T,k], aux fp32 [1] or NULL (outputs).
 * topk_idx and topk_w are the same bits on every call with the same inputs;
 * the per-expert score sums of aux are float atomics whose order varies, so
 * aux can differ from call to call in its last bits.
 */
moe_status_t moe_router(const void *x, const float *w_r, const float *logit_offset,
                        const float *sel_bias, const moe_shape_t *shape,
                        const moe_router_cfg_t *cfg, int32_t *topk_idx, float *topk_w,
                        float *aux, void *ws, size_t ws_bytes, void *stream);

/*
 * The router's selection from given fp32 logits l [T,E] instead of x . w_r^T:
 * scores, selection bias, group limit, top-k, weights and aux exactly as in
 * moe_router (logit_offset is added to l first). This is the guide's
 * force-load-balancing mode `uniform` (section "Router force load
 * balancing": the logits are replaced with random values before routing, so
 * per-expert counts are balanced only statistically and vary from step to
 * step) when the caller fills `logits` with random values; the random values
 * are an input, drawn by the caller.
 */
moe_status_t moe_route_logits(const float *logits, const float *logit_offset, const float *sel_bias,
                              const moe_shape_t *shape, const moe_router_cfg_t *cfg, int32_t *topk_idx,
                              float *topk_w, float *aux, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_router_noalloc: the same router as moe_router, for callers that cannot
 * allocate device memory. The pages have no counterpart to this entry point.
 *
 * Who needs it: a plug-in running inside a host runtime that owns all device
 * memory (for example an inference engine with a fixed memory pool) must not
 * call cudaMalloc, because the host accounts for every byte itself, and it may
 * have no spare buffer to pass as a workspace. This call takes no workspace:
 * the router's scratch (the bf16 split of w_r, the split-K partial logits and
 * the aux accumulators) lives in a static array of 10 MiB + 9 KiB inside the
 * library, which every GPU that loads the library keeps until the process
 * exits. It allocates nothing.
 *
 * Limits: T * E <= 1048576 and E * H <= 1048576 (the scratch must fit the
 * static array); larger shapes return MOE_ERR_UNSUPPORTED. All other arguments,
 * limits and results are those of moe_router, except that the split-K factor
 * may be lower, which can change the last bits of the fp32 logits.
 *
 * The first call on each device looks up the array's device address (set-up
 * once per device); make that first call before any stream capture. All calls
 * on a device share the one array: calls whose kernels may run at the same
 * time on the GPU (unordered streams) race on it and give wrong results.
 * Each call clears the accumulators it needs before using them.
 */
moe_status_t moe_router_noalloc(const void *x, const float *w_r, const float *logit_offset,
                                const float *sel_bias, const moe_shape_t *shape,
                                const moe_router_cfg_t *cfg, int32_t *topk_idx, float *topk_w,
                                float *aux, void *stream);

/*
 * The device error word of moe_router_noalloc (it has no workspace to hold
 * one): wait for `stream`, then read and clear the word kept in the last bytes
 * of the static array of the current device. Bits as for moe_get_device_error
 * (MOE_DEVERR_WAIT_TIMEOUT: a pipeline wait of the router's GEMM ran out of
 * time and that call's routing is invalid). Returns MOE_ERR_DEVICE_FLAGGED
 * when it was non-zero, MOE_OK when it was zero. The word is shared by every
 * moe_router_noalloc call on the device, so a flag stays until it is read here.
 * Not for the hot path (it synchronises the stream).
 */
moe_status_t moe_router_noalloc_get_error(int32_t *code, void *stream);

/*
 * Routing metadata: the local stand-in for the dispatch all-to-all (MegaMoE
 * guide, opening section, dispatch_grouped_gemm; section "Router force load
 * balancing": ragged per-expert counts absorbed without padding or host sync).
 * From topk_idx int32 [T,k] it writes into ws the per-expert counts, their
 * exclusive prefix sum, the row-tile prefix, and the stable permutation: rows
 * of expert e are offsets[e] .. offsets[e+1]-1 in increasing flat slot order.
 * Slots with an index outside [0, E) are dropped and flag the error word.
 */
moe_status_t moe_routing_metadata(const int32_t *topk_idx, const moe_shape_t *shape,
                                  void *ws, size_t ws_bytes, void *stream);

/*
 * dispatch_grouped_gemm with the SwiGLU fused into its epilogue (MegaMoE
 * guide, opening section and section "Design: two stages", stage 1):
 *
 *   for routed row r of expert e, token t = perm_slot[r] / k:
 *     h = x[t,:] . w1[e]^T  (2I values, fp32 accumulate)
 *     a[r, i] = silu(h[i]) * h[I + i],  i < I   (rounded to bf16)
 *
 * x bf16 [T,H]; w1 bf16 [E,2I,H]; a bf16 [T*k, I] (caller-owned, rows in the
 * metadata's routed order; rows past offsets[E] are left untouched). Needs the
 * metadata of moe_routing_metadata in ws.
 */
moe_status_t moe_dispatch_gemm1(const void *x, const void *w1, const moe_shape_t *shape,
                                void *a, void *ws, size_t ws_bytes, void *stream);

/*
 * grouped_gemm_combine (MegaMoE guide, opening section and section "Design:
 * two stages", stage 2). The SwiGLU already ran in stage 1's epilogue, so the
 * input is a:
 *
 *   o[r,:] = a[r,:] . w2[e]^T   (H values, fp32 accumulate)
 *   y[t,:] = sum_j topk_w[t,j] * o[row_of[t*k+j], :]   (fp32 sum, bf16 out)
 *
 * a bf16 [T*k, I] (routed order, from moe_dispatch_gemm1); topk_w fp32 [T,k];
 * w2 bf16 [E,H,I]; y bf16 [T,H] is fully overwritten (tokens whose slots were
 * all dropped get zeros). Needs the metadata of moe_routing_metadata in ws.
 */
moe_status_t moe_swiglu_gemm2_combine(const void *a, const float *topk_w, const void *w2,
                                      const moe_shape_t *shape, void *y, void *ws,
                                      size_t ws_bytes, void *stream);

/*
 * One-shot expert path, the single-device counterpart of the guide's
 * fused_mega_moe(x, topk_idx, topk_weights, w1, w2, group) without the process
 * group: routing metadata, then stage 1, then stage 2, with `a` kept in ws.
 */
moe_status_t moe_forward(const void *x, const int32_t *topk_idx, const float *topk_w,
                         const void *w1, const void *w2, const moe_shape_t *shape, void *y,
                         void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------ expert parallelism
 *
 * Across devices the guide fuses the dispatch all-to-all into
 * dispatch_grouped_gemm and the combine all-to-all into grouped_gemm_combine
 * (opening section). These two calls are the device-side halves of that
 * exchange when the caller moves the rows with its own collective: routed rows
 * are expert-major, so the rows bound for the device that owns experts
 * [e0, e1) are the contiguous rows offsets[e0] .. offsets[e1]-1.
 */

/*
 * Dispatch send buffer: rows[r, :] = x[perm_slot[r] / k, :] for every routed row
 * r < offsets[E] (rows of dropped slots are not written), and, when row_weight is
 * not NULL, row_weight[r] = topk_w[perm_slot[r]]. x bf16 [T,H]; rows bf16
 * [T*k, H]; topk_w fp32 [T,k]; row_weight fp32 [T*k]. Needs the metadata of
 * moe_routing_metadata in ws.
 */
moe_status_t moe_dispatch_rows(const void *x, const float *topk_w, const moe_shape_t *shape, void *rows,
                               float *row_weight, void *ws, size_t ws_bytes, void *stream);

/*
 * Combine of returned rows: y[t, :] = sum_j rows[row_of[t*k + j], :] (rows already
 * weighted, in this device's routed order; dropped slots skipped; fp32 sum,
 * bf16 y [T,H], fully written). Needs the metadata of moe_routing_metadata in ws.
 */
moe_status_t moe_combine_rows(const void *rows, const moe_shape_t *shape, void *y, void *ws, size_t ws_bytes,
                              void *stream);

/*
 * Expert parallelism without host synchronisation (the guide's "Example 2"
 * runs the whole layer under one CUDA graph). P ranks, rank q owning experts
 * [q E_loc, (q+1) E_loc), E = P E_loc. Every rank sends every rank a block of
 * `capacity` rows (C), so the caller's collective (an all-to-all with equal
 * splits) needs no per-step sizes from the device; C = T k can never drop a
 * row. A step on rank p:
 *   1. moe_routing_metadata of its tokens, then moe_ep_pack: send_rows [P*C, H]
 *      (block q: the rows of rank q's experts in routed order, from place 0),
 *      send_w [P*C] their routing weights, send_counts [P, E_loc] the rows of
 *      each expert that were sent.
 *   2. the caller exchanges the counts, rows and weights (equal splits).
 *   3. moe_ep_receive_metadata on a second workspace, shaped (T = P*C, k = 1,
 *      E = E_loc, H, I), from the received counts; then moe_dispatch_gemm1 and
 *      moe_swiglu_gemm2_combine on the received rows with the received weights
 *      as topk_w [P*C, 1]: y_recv [P*C, H] holds each received row's weighted
 *      output at the place it arrived (zero where nothing arrived).
 *   4. the caller returns y_recv (equal splits), and moe_ep_combine sums each
 *      token's returned rows into y.
 * Places not filled by a sender are never read as rows of a token.
 */

/* Step 1 (sender). x bf16 [T,H], topk_w fp32 [T,k]; the metadata of
 * moe_routing_metadata for `shape` in ws. Rows past `capacity` in a block are
 * dropped and flag MOE_DEVERR_CAPACITY. n_ranks must divide E. */
moe_status_t moe_ep_pack(const void *x, const float *topk_w, const moe_shape_t *shape, int32_t n_ranks,
                         int64_t capacity, void *send_rows, float *send_w, int32_t *send_counts, void *ws,
                         size_t ws_bytes, void *stream);

/* Step 3 (receiver): the routing metadata of the received rows, from
 * recv_counts int32 [n_ranks, E_loc] (row p: what source p sent), into ws for
 * recv_shape = (T = n_ranks * capacity, k = 1, E = E_loc, H, I). Received row
 * p*C + i is a token with one slot; the routed order is expert-major, then
 * source, then place (the order moe_routing_metadata gives for those slots). */
moe_status_t moe_ep_receive_metadata(const int32_t *recv_counts, int32_t n_ranks, int64_t capacity,
                                     const moe_shape_t *recv_shape, void *ws, size_t ws_bytes, void *stream);

/* Step 4 (sender): y[t] = sum over the token's slots of back_rows[place of the
 * slot's row] (fp32 in slot order, bf16 y [T,H], fully written). back_rows
 * bf16 [n_ranks*capacity, H]; the metadata of step 1 in ws. */
moe_status_t moe_ep_combine(const void *back_rows, const moe_shape_t *shape, int32_t n_ranks, int64_t capacity,
                            void *y, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------ training
 *
 * The backward of the expert path and the router (MegaMoE guide, section
 * "Design: two stages": stage 2's backward yields dW2, then stage 1's backward
 * yields dW1). The loss gradient enters as dY bf16 [T,H]. All GEMMs accumulate
 * in fp32; gradients of bf16 tensors are written in bf16. The selection (top-k,
 * groups, selection bias) passes no gradient; the aux value is not
 * differentiated. All calls below need a workspace sized with
 * flags = MOE_SHAPE_TRAINING.
 */

/*
 * moe_router with the fp32 logits l[t,e] (logit_offset included, selection
 * bias not) also written to `logits` [T,E], for moe_router_backward.
 */
moe_status_t moe_router_train(const void *x, const float *w_r, const float *logit_offset,
                              const float *sel_bias, const moe_shape_t *shape,
                              const moe_router_cfg_t *cfg, int32_t *topk_idx, float *topk_w,
                              float *aux, float *logits, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_dispatch_gemm1 that also stores the pre-activation h [T*k, 2I] bf16 in
 * routed order (columns [0,I) the gate, [I,2I) the up projection), which the
 * backward's SwiGLU needs. h is caller-owned and must be kept until
 * moe_backward_stage2_data has run.
 */
moe_status_t moe_dispatch_gemm1_train(const void *x, const void *w1, const moe_shape_t *shape,
                                      void *a, void *h, void *ws, size_t ws_bytes, void *stream);

/*
 * Stage 2 backward, data part (grouped_gemm_combine and the SwiGLU):
 *
 *   for routed row r of expert e, token t, slot s, weight w = topk_w[s]:
 *     dA_u[r,:] = dY[t,:] . w2[e]                      (I values)
 *     dtopk_w[s] = sum_i dA_u[r,i] a[r,i]              (= <dY[t], o[r]>)
 *     dA = w dA_u;  dU = dA silu(g);  dG = dA u silu'(g)   with [g | u] = h[r]
 *
 * dy bf16 [T,H]; topk_w fp32 [T,k]; w2 bf16 [E,H,I]; h from
 * moe_dispatch_gemm1_train; dtopk_w fp32 [T,k] (output, 0 for dropped slots)
 * or NULL. dY's rows are first copied into routed order (workspace region
 * dyp); they, dH = [dG | dU] and w a stay in the workspace for the other
 * backward calls.
 */
moe_status_t moe_backward_stage2_data(const void *dy, const float *topk_w, const void *w2, const void *h,
                                      const moe_shape_t *shape, float *dtopk_w, void *ws, size_t ws_bytes,
                                      void *stream);

/*
 * Stage 2 backward, weight part: dW2[e] = sum over e's rows of dY[t]^T (w a)[r]
 * into dw2 bf16 [E,H,I] (every expert written; experts without rows get 0).
 * Needs moe_backward_stage2_data on this workspace: the dY rows are read from
 * the routed-order copy that call made, so dy must be the tensor given there
 * (it is only checked for NULL and alignment).
 */
moe_status_t moe_backward_stage2_weight(const void *dy, const moe_shape_t *shape, void *dw2, void *ws,
                                        size_t ws_bytes, void *stream);

/*
 * Router backward: the logit gradient from dtopk_w (softmax or sigmoid,
 * normalised over the chosen experts or not, times scale), kept in the
 * workspace for moe_backward_stage1_data's dX term, and
 *   dW_r[e,:] = sum_t dl[t,e] x[t,:]   (fp32 [E,H], output).
 * logits from moe_router_train; topk_idx, topk_w from the same router call.
 */
moe_status_t moe_router_backward(const void *x, const float *logits, const int32_t *topk_idx,
                                 const float *topk_w, const float *dtopk_w, const moe_shape_t *shape,
                                 const moe_router_cfg_t *cfg, float *dw_r, void *ws, size_t ws_bytes,
                                 void *stream);

/*
 * Stage 1 backward, data part (dispatch_grouped_gemm):
 *
 *   dX[t,:] = sum over t's slots of dH[r,:] . w1[e]  (+ sum_e dl[t,e] w_r[e,:]
 *             when w_r is not NULL: the router's term, from moe_router_backward)
 *
 * w1 bf16 [E,2I,H]; w_r fp32 [E,H] or NULL; with w_r, topk_idx and cfg are
 * those of the router call (they tell which logit gradients can be non-zero);
 * dx bf16 [T,H] is the output: a sum of rows rounded to bf16 per slot plus the
 * fp32 router term, rounded to bf16 once. Needs moe_backward_stage2_data (and,
 * with w_r, moe_router_backward) on this workspace.
 */
moe_status_t moe_backward_stage1_data(const void *w1, const float *w_r, const int32_t *topk_idx,
                                      const moe_router_cfg_t *cfg, const moe_shape_t *shape, void *dx,
                                      void *ws, size_t ws_bytes, void *stream);

/*
 * Stage 1 backward, weight part: dW1[e] = sum over e's rows of dH[r]^T x[t]
 * into dw1 bf16 [E,2I,H] (every expert written; experts without rows get 0).
 * x bf16 [T,H]. Needs moe_dispatch_gemm1_train and moe_backward_stage2_data on
 * this workspace: the x rows are read from the routed-order copy that the
 * training forward made, so x must be the tensor given there (it is only
 * checked for NULL and alignment).
 */
moe_status_t moe_backward_stage1_weight(const void *x, const moe_shape_t *shape, void *dw1, void *ws,
                                        size_t ws_bytes, void *stream);

/*
 * The whole backward, in the guide's order: stage 2 (data, weight), the router
 * (skipped when w_r is NULL; then dw_r is not written and logits may be NULL),
 * stage 1 (data, weight). With w_r, the arguments logits, cfg, dw_r, topk_idx and
 * dtopk_w (fp32 [T,k]: the routing-weight gradient, written by stage 2 and read by
 * the router backward) are all required, else MOE_ERR_INVALID_ARG; without w_r,
 * dtopk_w may be NULL.
 */
moe_status_t moe_backward(const void *x, const float *w_r, const float *logits,
                          const int32_t *topk_idx, const float *topk_w, const void *w1,
                          const void *w2, const void *h, const void *dy, const moe_shape_t *shape,
                          const moe_router_cfg_t *cfg, void *dx, void *dw1, void *dw2, float *dw_r,
                          float *dtopk_w, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------ packed weights
 *
 * The forward GEMMs read one weight slab per pipeline stage: 256 rows x 64
 * K-elements of one expert (stage 1: 128 gate rows and the matching 128 up
 * rows; stage 2: 256 rows of w2[e]). Packed, each slab is one contiguous 32 KB
 * block already in the 128-byte-swizzled shared-memory image, fetched with one
 * bulk copy instead of 256 strided 128-byte pieces. Pack once per weight
 * update (the layout is a pure permutation plus zero padding; the values are
 * unchanged, so results are identical) and pass the packed buffers with
 * flags |= MOE_SHAPE_PACKED_WEIGHTS.
 *
 *   w1p: 32 KB tiles (e, n, kb), n < ceil(I/128), kb < ceil(H/64), in that
 *        order; tile row r < 128 = w1[e][128 n + r], row 128 + r =
 *        w1[e][I + 128 n + r] (zero where 128 n + r >= I), columns
 *        [64 kb, 64 kb + 64) (zero past H); 16-byte chunk c of row r at byte
 *        128 r + 16 (c XOR (r mod 8)).
 *   w2p: tiles (e, n, kb), n < ceil(H/256), kb < ceil(I/64); row r =
 *        w2[e][256 n + r] (zero past H), columns [64 kb, 64 kb + 64) (zero
 *        past I); same chunk order.
 */

/* Bytes of the packed w1 and w2 for `shape` (either pointer may be NULL). Host-only. */
moe_status_t moe_packed_weights_size(const moe_shape_t *shape, size_t *w1p_bytes, size_t *w2p_bytes);

/* Pack w1 [E,2I,H] into w1p and w2 [E,H,I] into w2p (bf16, 16-byte aligned,
 * caller-owned; a pair of NULL src/dst pointers skips that tensor). Enqueued
 * on `stream`. */
moe_status_t moe_pack_weights(const void *w1, const void *w2, const moe_shape_t *shape, void *w1p, void *w2p,
                              void *stream);

/* ------------------------------------------------------------------ MXFP8
 *
 * The guide's second expert precision (section "Expert precision": mxfp8 runs
 * the two expert stages in MXFP8; parameters stay bf16). MXFP8 is the OCP
 * Microscaling format: blocks of 32 consecutive elements along a GEMM's
 * reduction dimension share a power-of-two scale 2^(floor(log2 max|v|) - 8),
 * stored as E8M0 (one byte, bias 127); elements are FP8 E4M3 (one byte),
 * rounded to nearest even and saturated to +-448. A matrix [rows, cols] is
 * stored as codes uint8 [rows, cols], row-major, and scales in k-block-major
 * order: 32-bit words [cols/128][rows4], rows4 = rows rounded up to a multiple
 * of 4, byte j (j = 0..3, little-endian) of word [kb][r] being the scale of
 * elements r, 128 kb + 32 j .. 128 kb + 32 j + 31 (rows4*cols/32 bytes; the
 * words of rows rows..rows4-1 are padding, never written or read). A word is
 * one row's scales for one 128-deep k-block of the block-scaled MMA; the GEMMs
 * copy the words of a unit's rows for each k-block into shared memory with
 * TMA, next to its operand tiles.
 * The MXFP8 calls need H and I multiples of 128 (else MOE_ERR_UNSUPPORTED).
 */

/*
 * Quantize a bf16 [rows, cols] matrix (cols a multiple of 128) along its rows:
 * codes uint8 [rows, cols] (E4M3) and k-block-major scales (E8M0, words
 * [cols/128][rows4], layout above). in, codes and scales 16-byte aligned.
 * For the weights, quantize w1 as [E*2I, H] and w2 as [E*H, I] once per weight
 * update and keep the result (the guide's weight-quant cache); x is quantized
 * every step (moe_forward_mx does it).
 */
moe_status_t moe_mx_quantize(const void *in, int64_t rows, int64_t cols, void *codes, void *scales,
                             void *stream);

/*
 * The dispatch of the MXFP8 path, fused into the quantization of x: routed row
 * r of the metadata (token t = perm_slot[r] / k) gets MXFP8 codes and scales of
 * x[t,:] in the workspace (x_codes [T*k, H]; x_scales words [H/128][rows4(T*k)];
 * routed order), so stage 1 reads whole tiles. x bf16 [T,H]. Needs the metadata of
 * moe_routing_metadata in ws and flags containing MOE_SHAPE_MXFP8. Each token's
 * row is read and quantized once and written to its k routed rows; the scales
 * pass through the workspace's obuf region (idle until stage 2), which this call
 * overwrites.
 */
moe_status_t moe_mx_quantize_dispatch(const void *x, const moe_shape_t *shape, void *ws, size_t ws_bytes,
                                      void *stream);

/*
 * Stage 1 in MXFP8 over the dispatched rows of moe_mx_quantize_dispatch: for
 * routed row r of expert e,
 *   h = X(x)[r,:] . X(w1)[e]^T (fp32 accumulate from E4M3 products scaled per block)
 *   a[r, i] = silu(h[i]) * h[I + i], then quantized per 32 columns of i
 * w1_codes [E,2I,H] with w1_scales words [H/128][E*2I] (moe_mx_quantize of w1
 * as [E*2I, H]); outputs a_codes [T*k, I] and a_scales words
 * [I/128][rows4(T*k)] (routed order; rows4(T*k)*I/32 bytes).
 */
moe_status_t moe_dispatch_gemm1_mx(const void *w1_codes, const void *w1_scales, const moe_shape_t *shape,
                                   void *a_codes, void *a_scales, void *ws, size_t ws_bytes, void *stream);

/*
 * Stage 2 in MXFP8: o[r,:] = X(a)[r,:] . X(w2)[e]^T, y[t,:] = sum_j topk_w[t,j] o[row_of[t*k+j],:]
 * (bf16 y, fp32 sum). a_codes / a_scales as stage 1 writes them; w2_codes
 * [E,H,I] with w2_scales words [I/128][E*H] (moe_mx_quantize of w2 as [E*H, I]).
 */
moe_status_t moe_swiglu_gemm2_combine_mx(const void *a_codes, const void *a_scales, const float *topk_w,
                                         const void *w2_codes, const void *w2_scales,
                                         const moe_shape_t *shape, void *y, void *ws, size_t ws_bytes,
                                         void *stream);

/*
 * One-shot MXFP8 expert path: routing metadata, the quantizing dispatch of x,
 * stage 1, stage 2. Needs a workspace sized with flags containing MOE_SHAPE_MXFP8.
 */
moe_status_t moe_forward_mx(const void *x, const int32_t *topk_idx, const float *topk_w,
                            const void *w1_codes, const void *w1_scales, const void *w2_codes,
                            const void *w2_scales, const moe_shape_t *shape, void *y, void *ws,
                            size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------ MXFP8 training
 *
 * The guide's mxfp8 also runs the dW1 / dW2 weight gradients in MXFP8
 * (section "Expert precision"). A training step in MXFP8 runs, on one
 * workspace sized with flags = MOE_SHAPE_TRAINING | MOE_SHAPE_MXFP8:
 * moe_router_train, moe_routing_metadata, moe_mx_quantize_dispatch,
 * moe_dispatch_gemm1_mx_train, moe_swiglu_gemm2_combine_mx, then
 * moe_backward_stage2_data (bf16 w2), moe_backward_stage2_weight_mx,
 * moe_router_backward, moe_backward_stage1_data (bf16 w1) and
 * moe_backward_stage1_weight_mx. The data gradients are those of the bf16
 * backward at the MXFP8 forward's pre-activation h (quantization passes the
 * gradient through); the weight gradients quantize both operands to MXFP8
 * along their reduction dimension, the expert's routed rows: blocks of 32
 * consecutive routed rows of the expert from its first row (the last block
 * zero-padded), with the routing weight on the activation side:
 *   dW2[e] = Q(dY rows)^T Q(w a rows),   dW1[e] = Q(dH rows)^T Q(x rows).
 * H and I must be multiples of 128.
 */

/*
 * moe_dispatch_gemm1_mx that also stores the pre-activation h [T*k, 2I] bf16
 * (routed order; the fp32 accumulator of the MXFP8 GEMM rounded to bf16) for
 * moe_backward_stage2_data.
 */
moe_status_t moe_dispatch_gemm1_mx_train(const void *w1_codes, const void *w1_scales, const moe_shape_t *shape,
                                         void *a_codes, void *a_scales, void *h, void *ws, size_t ws_bytes,
                                         void *stream);

/*
 * dW2[e] = Q(dY rows of e)^T Q(w a rows of e) into dw2 bf16 [E,H,I] (experts
 * without rows get 0), fp32 accumulation of the block-scaled products. Needs
 * moe_backward_stage2_data on this workspace (its routed-order dY rows and w a);
 * dy is only checked for NULL and alignment.
 */
moe_status_t moe_backward_stage2_weight_mx(const void *dy, const moe_shape_t *shape, void *dw2, void *ws,
                                           size_t ws_bytes, void *stream);

/*
 * dW1[e] = Q(dH rows of e)^T Q(x rows of e) into dw1 bf16 [E,2I,H]. x bf16
 * [T,H] (the tensor of the forward); needs moe_backward_stage2_data on this
 * workspace (dH).
 */
moe_status_t moe_backward_stage1_weight_mx(const void *x, const moe_shape_t *shape, void *dw1, void *ws,
                                           size_t ws_bytes, void *stream);

/*
 * Wait for `stream`, then read and clear the workspace error word into *code.
 * Returns MOE_ERR_DEVICE_FLAGGED when it was non-zero. Not for the hot path.
 */
moe_status_t moe_get_device_error(void *ws, int32_t *code, void *stream);

/* Static description of a status code. */
const char *moe_status_string(moe_status_t status);

/* Number of kernels this library has launched in this process (statistics). */
uint64_t moe_kernel_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_MOE_H */
