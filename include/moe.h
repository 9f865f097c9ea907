/*
 * moe.h -- C ABI of the B300 (sm_103a) DeepSeekMoE feed-forward layer.
 *
 * The layer (DeepSeek-V3 technical report; ai.flicky.cc "06 - DeepSeek-V3
 * reading" section 2.1.2 and xyznot.com "DeepSeek-V3 technical report"
 * Method 2):
 *
 *   h'_t    = u_t + sum_{s<N_s} FFN^(s)_s(u_t) + sum_{i<N_r} g_{i,t} FFN^(r)_i(u_t)
 *   s_{i,t} = sigmoid(u_t^T e_i)
 *   g'_{i,t}= s_{i,t} if s_{i,t} + b_i is among the K_r largest of {s_{j,t} + b_j}, else 0
 *   g_{i,t} = g'_{i,t} / sum_j g'_{j,t}
 *   FFN(x)  = W2 (SiLU(W1 x) * (W3 x))       (SwiGLU expert of three d x I matrices)
 *
 * and the auxiliary-loss-free bias update between steps (same section):
 * b_i decreases by gamma when expert i is overloaded, increases when it is
 * underloaded.  FP8 variant (ai.flicky.cc section 3.3): E4M3 operands for the
 * expert GEMMs, activations scaled per 1 x 128 tile, weights per 128 x 128
 * block, partial sums promoted to FP32 every 128 elements of K; the router
 * stays bf16 with fp32 accumulation.
 *
 * Conventions shared by every call
 *   Memory     Every pointer is DEVICE memory owned by the caller, unless a
 *              parameter says otherwise.  The library allocates nothing and
 *              keeps no mutable global state (the one exception is the fixed
 *              scratch array of moe_route_noalloc); each call only enqueues work.
 *              Base pointers must be 16-byte aligned.
 *   Streams    `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *              default stream).  Calls are asynchronous on that stream.
 *   bf16       bf16 tensors are passed as uint16_t bit patterns.
 *   Layouts    Row-major.  Weights are K-major (nn.Linear: [out, in]).
 *   Errors     Argument and shape errors are returned at once and enqueue
 *              nothing.  Errors found on the device (an out-of-range expert
 *              index, a bounded wait that ran out) are written to a status
 *              word at the start of the workspace; moe_read_device_status()
 *              returns it.  Every call that takes a workspace clears that word
 *              first, so it reports the most recent such call.
 *   Limits     1 <= k <= min(E, 32); E <= 1024; d and I multiples of 128;
 *              T >= 0 (T == 0 enqueues nothing and succeeds).
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer, bad shape, k > E, misaligned pointer */
  MOE_ERR_UNSUPPORTED = 2,  /* shape outside the limits above */
  MOE_ERR_WORKSPACE = 3,    /* workspace smaller than moe_workspace_size() */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime call failed (launch, attribute, ...), or the FP8 GEMM
                               was compiled to another register count than its warpgroup register
                               split assumes (a build problem: nothing is launched) */
  MOE_ERR_TIMEOUT = 5,      /* device: a bounded wait inside a kernel ran out */
  MOE_ERR_BAD_INDEX = 6,    /* device: an expert index outside [0, E) */
  MOE_ERR_OUT_OF_RANGE = 7  /* device, range-checked build only (-DMOE_CHECK): a computed index outside
                               its buffer; the access was skipped */
} moe_status;

/* Precision of the expert GEMMs.  MOE_FP8_UE8M0: the FP8 scheme with UE8M0
 * scales -- the scheme DeepSeek-V3.1 moved to (ai.flicky.cc, continuation of
 * section 3.5): every scale a power of two (an 8-bit exponent, no mantissa),
 * taken as amax/448 rounded up to the next power of two, so that no element
 * of a group exceeds 448 after scaling; everything else as MOE_FP8_E4M3 (the
 * weights must be quantised with power-of-two scales too, see
 * moe_quantize_fp8_blocks). */
typedef enum { MOE_BF16 = 0, MOE_FP8_E4M3 = 1, MOE_FP8_UE8M0 = 2 } moe_precision;

/* Layer shape.  T tokens, hidden size d, E routed experts, k of them per
 * token, n_shared shared experts, SwiGLU intermediate size inter (= I) of
 * every expert, prec the precision of the expert GEMMs.
 * Node-limited routing (ai.flicky.cc 2.1.2: a token is sent to at most 4
 * nodes): route_groups > 0 places the experts on route_groups nodes of
 * E / route_groups consecutive experts, and a token's k experts span at most
 * route_group_limit of them -- the k best experts (biased score) on the
 * route_group_limit nodes whose best expert scores highest.  0 and 0: no
 * limit.  Requires E % route_groups == 0, route_groups <= 32,
 * 1 <= route_group_limit <= route_groups and route_group_limit * E /
 * route_groups >= k. */
typedef struct {
  int32_t T, d, E, k, n_shared, inter;
  int32_t prec; /* moe_precision */
  int32_t route_groups, route_group_limit;
} moe_dims;

/*
 * Expert weights of one layer.
 *   w13  routed gate/up weights [E, 2I, d]: for j = 0 .. I/128-1, rows
 *        [256j, 256j+128) are W1 rows [128j, 128j+128) and rows
 *        [256j+128, 256j+256) are W3 rows [128j, 128j+128).  (One 256-row
 *        tile then holds matching gate and up features; moe_pack_gate_up
 *        builds this layout.)  bf16, or E4M3 bytes when prec is FP8.
 *   w2   routed down weights [E, d, I].
 *   w13_scale, w2_scale  FP8 only: fp32 scale of every 128 x 128 block,
 *        [E, 2I/128, d/128] and [E, d/128, I/128]; NULL for bf16.
 *   ws13, ws2, ws13_scale, ws2_scale  the same for the n_shared shared experts.
 *   centroids  router centroids e_i, [E, d] bf16 (the router is never FP8).
 */
typedef struct {
  const void* w13;
  const float* w13_scale;
  const void* w2;
  const float* w2_scale;
  const void* ws13;
  const float* ws13_scale;
  const void* ws2;
  const float* ws2_scale;
  const uint16_t* centroids;
} moe_weights;

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status s);

/* Bytes of workspace moe_forward (and every call below that takes `ws`) needs
 * for these dimensions.  The workspace is caller-owned device memory, 256-byte
 * aligned, with no required initial content. */
moe_status moe_workspace_size(const moe_dims* dims, size_t* bytes);

/*
 * Router: s = sigmoid(u e^T), top-k of s + b, gates normalised over the
 * selected unbiased affinities (ai.flicky.cc 2.1.2, the s_{i,t} and g'_{i,t}
 * equations; xyznot.com Method 2, the normalisation of g').
 *   u          [T, d] bf16 layer input.
 *   centroids  [E, d] bf16.
 *   bias       [E] fp32 selection bias (read only).
 *   topk_idx   out [T, k] int32: the selected experts of each token, by biased
 *              score descending (exact ties: lower index first).
 *   topk_gate  out [T, k] fp32: g of each selected expert (sums to 1 per token).
 *   counts     out [E] int32: tokens routed to each expert (the load).
 * Logits are a bf16 x bf16 -> fp32 tensor-core GEMM.  A NaN score ranks
 * below every number.
 */
moe_status moe_route(const moe_dims* dims, const uint16_t* u, const uint16_t* centroids,
                     const float* bias, int32_t* topk_idx, float* topk_gate, int32_t* counts,
                     void* ws, size_t ws_bytes, void* stream);

/*
 * moe_route for callers that cannot allocate device memory.  (A library
 * addition with no counterpart in the paper.)
 *
 * Who needs it: code that may not call cudaMalloc -- for example a plugin
 * running inside a host engine that owns all device memory through its own
 * pool, or a serving process that reserves every byte at start-up and must
 * not allocate on the request path, where cudaMalloc can stall the device and
 * can fail under memory pressure.  Such a caller has no way to obtain the
 * workspace moe_route wants.
 *
 * This variant does the same work with the same kernels and results, but its
 * scratch (the [T, E] fp32 router logits) lives in a fixed array inside the
 * library (a `static __device__` array of MOE_ROUTE_NOALLOC_MAX_LOGITS floats,
 * 8 MiB, 256-byte aligned).  The CUDA runtime places that array on every
 * device that loads the library and keeps it until the process exits.  The
 * call itself allocates nothing and calls no allocating routine.
 *
 *   u, centroids, bias, topk_idx, topk_gate, counts  as in moe_route.
 *   device_status  optional [1] int32 device word (NULL: not reported): set to
 *                  MOE_OK by the call, MOE_ERR_TIMEOUT if a bounded wait in
 *                  the logits GEMM ran out.
 * Limits: T * E <= MOE_ROUTE_NOALLOC_MAX_LOGITS, else MOE_ERR_UNSUPPORTED is
 * returned and nothing is enqueued; other limits as moe_route.
 * Set-up: the first call on a device (the current device) looks up the
 * device address of the array with cudaGetSymbolAddress and caches it with
 * the id of the device's current context; make that first call on each device
 * before any stream capture begins.  If the context changes (cudaDeviceReset,
 * or a context the caller made current), the next call on that device looks
 * the address up again, so it is a set-up call too.
 * Sharing: every call on a device uses the same array, whose content is
 * whatever the last call left (every logit read is first written by the same
 * call).  Calls whose work overlaps on the GPU -- on different streams, or
 * from different host threads -- race on the array: serialise them.
 */
#define MOE_ROUTE_NOALLOC_MAX_LOGITS (1 << 21)
moe_status moe_route_noalloc(const moe_dims* dims, const uint16_t* u, const uint16_t* centroids,
                             const float* bias, int32_t* topk_idx, float* topk_gate, int32_t* counts,
                             int32_t* device_status, void* stream);

/*
 * Dropless dispatch (ai.flicky.cc 2.1.2: no token is dropped): groups the
 * T*k (token, expert) pairs by expert, tokens ascending within an expert.
 *   topk_idx  [T, k] int32 (as from moe_route); entries outside [0, E) raise
 *             MOE_ERR_BAD_INDEX on the device and are skipped.
 *   u         [T, d] bf16.
 *   offsets   out [E+1] int32: rows of expert e are [offsets[e], offsets[e+1]).
 *   perm      out [T*k] int32: token of every permuted row.
 *   slot      out [T, k] int32: permuted row of pair (t, j).
 *   x_perm    out [T*k, d]: x_perm[r] = u[perm[r]] as bf16, or (FP8) as E4M3
 *             codes of u quantised per 1 x 128 tile.
 *   x_scale   FP8: out [d/128, T*k] fp32 tile scales (amax/448, column-major
 *             by row so a 128-row tile's scales are contiguous); NULL for bf16.
 */
moe_status moe_permute(const moe_dims* dims, const int32_t* topk_idx, const uint16_t* u,
                       int32_t* offsets, int32_t* perm, int32_t* slot, void* x_perm, float* x_scale,
                       void* ws, size_t ws_bytes, void* stream);

/*
 * Grouped SwiGLU experts: for g < n_groups, rows [offsets[g], offsets[g+1])
 * of x go through expert g: y = W2_g (SiLU(W1_g x) * (W3_g x)) -- an expert
 * is three d x I matrices (ai.flicky.cc practice section "Практика:
 * перепроверяем числа статьи"), FFN_i of the layer equation (ai.flicky.cc
 * 2.1.2); FP8: the fine-grained scheme of ai.flicky.cc 3.3 items 2-3.
 *   rows      rows allocated in x and y (offsets[n_groups] <= rows).
 *   offsets   [n_groups+1] int32 device array, non-decreasing, offsets[0] = 0.
 *   x         [rows, d] bf16, or E4M3 codes with x_scale [d/128, rows] fp32.
 *   w13, w2   weights of the n_groups experts in the moe_weights layout
 *             (with their block scales for FP8).
 *   y         out [rows, d] bf16.
 *   group_expert  NULL: group g uses the weights of expert g (the weight
 *             arrays hold n_groups experts).  Otherwise [n_groups] int32
 *             device array: group g uses the weights of expert
 *             group_expert[g] < n_weight_experts, the number of experts the
 *             weight arrays hold.  Several groups may share one expert's
 *             weights: the copies of a replicated hot expert (ai.flicky.cc
 *             3.5: popular experts are duplicated), or the rows an
 *             expert-parallel rank receives for one expert from each sender
 *             (ai.flicky.cc 3.4, EP with all-to-all).  An entry outside
 *             [0, n_weight_experts) raises MOE_ERR_BAD_INDEX on the device and
 *             uses expert 0.
 * Limits: n_groups <= dims->E + dims->n_shared (the workspace's group tables
 * are sized by dims), rows <= dims->T * dims->k.
 * The gate/up product and SiLU(g)*u are one fused tcgen05 GEMM; FP8 also
 * quantises h per 1 x 128 tile inside that GEMM before the down product.
 */
moe_status moe_grouped_ffn(const moe_dims* dims, int32_t n_groups, int32_t rows, const int32_t* offsets,
                           const int32_t* group_expert, int32_t n_weight_experts, const void* x,
                           const float* x_scale, const void* w13, const float* w13_scale, const void* w2,
                           const float* w2_scale, uint16_t* y, void* ws, size_t ws_bytes, void* stream);

/*
 * Combine (the layer equation of ai.flicky.cc 2.1.2):
 *   out_t = u_t + sum_{s<N_s} shared_y[s, t] + sum_{j<k} topk_gate[t, j] * y_perm[slot[t, j]]
 * summed in fp32 in that order, rounded once to bf16.
 *   shared_y  [n_shared, T, d] bf16, or NULL when n_shared == 0.
 *   y_perm    [T*k, d] bf16;  slot [T, k] int32;  topk_gate [T, k] fp32.
 *   out       out [T, d] bf16.
 * A slot outside [0, T*k) contributes nothing (its term is skipped).
 */
moe_status moe_combine(const moe_dims* dims, const uint16_t* u, const uint16_t* shared_y,
                       const uint16_t* y_perm, const int32_t* slot, const float* topk_gate,
                       uint16_t* out, void* stream);

/*
 * Auxiliary-loss-free bias update (ai.flicky.cc 2.1.2; xyznot.com Method 2,
 * gamma = 0.001): in fp32, b_i <- b_i + gamma * sign(T*k/E - counts_i), so an
 * overloaded expert loses gamma, an underloaded one gains gamma, and one
 * exactly at the mean load keeps its bias.
 *   counts  [E] int32 loads of the step;  bias  [E] fp32, updated in place.
 */
moe_status moe_bias_update(int32_t E, int32_t T, int32_t k, const int32_t* counts, float gamma,
                           float* bias, void* stream);

/*
 * The whole layer (the layer equation of ai.flicky.cc 2.1.2 and xyznot.com
 * Method 2; FP8 per ai.flicky.cc 3.3): route, dispatch, routed and shared
 * SwiGLU experts, combine.  bias is read only (moe_bias_update is its only
 * writer).
 *   u           [T, d] bf16.
 *   out         out [T, d] bf16 (h').
 *   counts_out  out [E] int32 per-expert loads of this step, or NULL.
 * The call enqueues its kernels and returns; it never waits on the device.
 */
moe_status moe_forward(const moe_dims* dims, const moe_weights* w, const uint16_t* u, const float* bias,
                       uint16_t* out, int32_t* counts_out, void* ws, size_t ws_bytes, void* stream);

/*
 * Redundant experts (ai.flicky.cc 3.5: popular experts are duplicated to even
 * out the load).  A plan gives expert e replica_count[e] >= 1 copies, the
 * physical slots replica_first[e] .. replica_first[e] + replica_count[e] - 1,
 * and slot_expert[p] names the expert whose weights slot p uses; P = E +
 * n_extra slots in all.  The copies share the expert's weights (nothing is
 * duplicated in memory on one GPU; in an expert-parallel deployment each copy
 * would live on another device).
 *
 * moe_plan_replicas: HOST function (all pointers host memory, no GPU work):
 *   counts  [E] the experts' loads (e.g. the previous step's counts_out).
 *   Each of the n_extra copies goes to the expert with the highest load per
 *   copy, counts[e] / replica_count[e] (ties: lower index); then slots are
 *   numbered expert by expert.  Outputs replica_first [E], replica_count [E],
 *   slot_expert [E + n_extra].  Limits: 1 <= E <= 1024, 0 <= n_extra <= 1024.
 *
 * moe_forward_replicated: moe_forward with the plan (device copies of the
 *   three tables; n_slots = P).  A token's pair (t, j) with expert e goes to
 *   copy t mod replica_count[e]; the grouped GEMMs run one group per physical
 *   slot on the shared weights.  h' is that of moe_forward; counts_out holds
 *   the experts' (not the slots') loads.  The workspace must be at least
 *   moe_workspace_size of dims with E replaced by n_slots (the per-expert
 *   tables hold the slots).  A bad plan entry raises MOE_ERR_BAD_INDEX on the
 *   device and the pair is left out.
 */
moe_status moe_plan_replicas(int32_t E, const int32_t* counts, int32_t n_extra, int32_t* replica_first,
                             int32_t* replica_count, int32_t* slot_expert);
moe_status moe_forward_replicated(const moe_dims* dims, const moe_weights* w, const uint16_t* u, const float* bias,
                                  const int32_t* replica_first, const int32_t* replica_count,
                                  const int32_t* slot_expert, int32_t n_slots, uint16_t* out, int32_t* counts_out,
                                  void* ws, size_t ws_bytes, void* stream);

/*
 * Backward pass of the layer, bf16 or in the FP8 scheme (prec MOE_FP8_E4M3 or
 * MOE_FP8_UE8M0).  Given dL/dh' (dout), the gradients of the layer equation of
 * ai.flicky.cc 2.1.2 (xyznot.com Method 2) with respect to its input u, the
 * router centroids and every expert weight.  The selection is held fixed --
 * the gradient flows through the gate values g = s / sum s, not through the
 * top-k choice -- and the bias, which the pages update by the sign rule
 * (moe_bias_update), gets no gradient.  Weight and centroid gradients are
 * fp32 (ai.flicky.cc 3.3 item 1: weight gradients are kept in higher
 * precision); activations inside are bf16, as in the forward.
 *
 * The data-gradient products run on transposed weights, prepared once by
 * moe_transpose_expert_weights:
 *   w13t [n, d, 2I] = w13 [n, 2I, d] transposed per expert (the w13 row
 *   interleave becomes the column order), w2t [n, I, d] = w2 [n, d, I]
 *   transposed.  n = E for the routed experts, n_shared for the shared ones.
 *   inter and d must be multiples of 128 (else MOE_ERR_INVALID_ARG).
 *   FP8: moe_quantize_fp8_blocks of the transposed bf16 weights (a 128 x 128
 *   block has the same scale either way round) gives the codes and the
 *   w13t_scale [n, d/128, 2I/128] / w2t_scale [n, I/128, d/128] grids.
 *
 * moe_backward recomputes the forward's routing, dispatch and expert
 * activations (the same kernels), then:
 *   dy = g G (routed rows), dg = G . y (bf16 layers: as (dh . h) / g, the
 *   same in exact arithmetic since dh = g G W2, so y is not recomputed),
 *   ds = (dg - sum g dg) / S,
 *   dz = ds s (1 - s);  dh = dy W2;  da, db from the SwiGLU derivative;
 *   dx = [da db] W13;  du = G + sum_j dx_j + sum_s dx_s + sum_j dz_j c_{e_j};
 *   dW2 = dy^T h, dW13 = [da db]^T x per expert (fp32 GEMMs over the expert's
 *   tokens), dcentroids_e = sum over its tokens of dz u.
 * FP8 (ai.flicky.cc 3.3 items 1-4: forward, data-gradient and weight-gradient
 * GEMMs in E4M3, weights in 128 x 128 blocks, activations and gradients in
 * 1 x 128 tiles along each GEMM's contraction axis):
 *   forward  as moe_forward in FP8 (a, b kept as bf16; h quantised along I);
 *   dgrad    dh = Q(dy) Q(W2), dx = Q([da db]) Q(W13): the FP8 expert GEMM,
 *            dy and [da db] quantised per 1 x 128 tile along their rows;
 *   wgrad    dW2 = Q_t(dy)^T Q_t(h), dW13 = Q_t([da db])^T Q_t(u): every
 *            operand quantised to E4M3 in 1 x 128 tiles along the tokens of
 *            its expert (blocks from the expert's first token), then the
 *            product of the dequantised values on the bf16 tensor cores with
 *            fp32 accumulation (each dequantised value rounded to bf16: exact
 *            for UE8M0 scales, within 2^-9 relative otherwise).
 *   dout   [T, d] bf16 dL/dh'.
 *   grads  outputs, all fp32 device memory: du [T, d]; dcentroids [E, d];
 *          dw13 [E, 2I, d] and dw2 [E, d, I] in the layout of w13 and w2 (an
 *          expert no token chose gets zeros); dws13, dws2 the same for the
 *          shared experts (unused when n_shared == 0).  du and the weight
 *          gradients must be 16-byte aligned (else MOE_ERR_INVALID_ARG).  With
 *          T == 0, u, dout and du may be NULL and the other gradients are
 *          zeroed.
 *   ws     at least moe_backward_workspace_size bytes.
 */
typedef struct {
  const void* w13t;          /* [E, d, 2I] bf16, or E4M3 codes (FP8) */
  const void* w2t;           /* [E, I, d] */
  const void* ws13t;         /* [n_shared, d, 2I] */
  const void* ws2t;          /* [n_shared, I, d] */
  const float* w13t_scale;   /* FP8 only: [E, d/128, 2I/128] block scales; NULL for bf16 */
  const float* w2t_scale;    /* FP8 only: [E, I/128, d/128] */
  const float* ws13t_scale;  /* FP8 only: [n_shared, d/128, 2I/128] */
  const float* ws2t_scale;   /* FP8 only: [n_shared, I/128, d/128] */
} moe_weights_t;

typedef struct {
  float* du;
  float* dcentroids;
  float* dw13;
  float* dw2;
  float* dws13;
  float* dws2;
} moe_grads;

moe_status moe_backward_workspace_size(const moe_dims* dims, size_t* bytes);
moe_status moe_transpose_expert_weights(int32_t n_experts, int32_t inter, int32_t d, const uint16_t* w13,
                                        const uint16_t* w2, uint16_t* w13t, uint16_t* w2t, void* stream);
/*
 * FP8 weights transposed for the backward: the E4M3 codes of w13 [n, 2I, d] /
 * w2 [n, d, I] and their block-scale grids [n, 2I/128, d/128] / [n, d/128,
 * I/128] become w13t [n, d, 2I] / w2t [n, I, d] with w13t_scale [n, d/128,
 * 2I/128] / w2t_scale [n, I/128, d/128].  A 128 x 128 block keeps its codes
 * and its scale when transposed, so this equals moe_quantize_fp8_blocks of the
 * transposed bf16 weights.  inter and d multiples of 128, 16-byte aligned
 * codes (else MOE_ERR_INVALID_ARG).  Asynchronous on `stream`.
 */
moe_status moe_transpose_expert_weights_fp8(int32_t n_experts, int32_t inter, int32_t d, const uint8_t* w13,
                                            const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                                            uint8_t* w13t, float* w13t_scale, uint8_t* w2t, float* w2t_scale,
                                            void* stream);
moe_status moe_backward(const moe_dims* dims, const moe_weights* w, const moe_weights_t* wt, const uint16_t* u,
                        const float* bias, const uint16_t* dout, const moe_grads* grads, void* ws, size_t ws_bytes,
                        void* stream);

/*
 * moe_forward with stage timing.  `events` holds n_events >= MOE_PROFILE_EVENTS
 * cudaEvent_t handles (passed as void*) created by the caller; the call
 * records events[0] on `stream` before its first kernel and events[i] after
 * stage i: 1 router logits GEMM, 2 top-k, 3 expert scan + tile plan,
 * 4 row gather (and FP8 quantisation), 5 routed gate/up + SwiGLU GEMM,
 * 6 routed down GEMM, 7 shared gate/up GEMM, 8 shared down GEMM, 9 combine
 * (stages 7 and 8 are empty when n_shared == 0).  The device work is that of
 * moe_forward.
 */
#define MOE_PROFILE_EVENTS 10
moe_status moe_forward_profiled(const moe_dims* dims, const moe_weights* w, const uint16_t* u, const float* bias,
                                uint16_t* out, int32_t* counts_out, void* ws, size_t ws_bytes, void* stream,
                                void* const* events, int32_t n_events);

/*
 * Offline weight preparation (not part of the timed layer).
 * moe_pack_gate_up: w13[e] = interleave of w1[e], w3[e] ([E, I, d] bf16 each)
 *   in 128-row blocks, the layout moe_weights.w13 describes (a layout of this
 *   library: the pages name the three matrices, not their storage).
 * moe_quantize_fp8_blocks: w [rows, cols] bf16 -> q [rows, cols] E4M3 codes and
 *   scale [rows/128, cols/128] fp32 with scale = amax/448 of each 128 x 128 block
 *   (1 for an all-zero block), q = round-to-nearest-even, saturating, of w/scale
 *   (ai.flicky.cc 3.3 item 2).  rows and cols multiples of 128.  pow2_scales
 *   != 0: the scale rounded up to a power of two (UE8M0, MOE_FP8_UE8M0).
 */
moe_status moe_pack_gate_up(const uint16_t* w1, const uint16_t* w3, int32_t E, int32_t inter, int32_t d,
                            uint16_t* w13, void* stream);
moe_status moe_quantize_fp8_blocks(const uint16_t* w, int64_t rows, int32_t cols, uint8_t* q, float* scale,
                                   int32_t pow2_scales, void* stream);

/* Synchronises `stream` and returns the device status word of workspace `ws`
 * (MOE_OK, MOE_ERR_TIMEOUT, MOE_ERR_BAD_INDEX), or MOE_ERR_CUDA if the stream
 * itself reports an error. */
moe_status moe_read_device_status(const void* ws, void* stream);

/*
 * Self-test of the bounded waits: launches one CTA that waits on an mbarrier
 * nothing ever arrives on, with a limit of timeout_us microseconds.  The
 * kernel then gives up, records MOE_ERR_TIMEOUT in the status word of `ws`
 * and returns normally, leaving the context usable.  Every wait inside the
 * library's kernels is bounded the same way (with a limit of seconds).
 */
moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes, int32_t timeout_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
