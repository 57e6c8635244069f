/*
 * moe_route_sort.h -- C ABI of the GB300 (sm_103a) MoE route-sort library.
 *
 * Route-sort turns router logits into the expert-grouped dispatch metadata a grouped MoE
 * GEMM consumes.  Source of the operation: "perf(flydsl): Kimi-K3 B1 route-sort +
 * prepared-MoE handoff (stack)", Summary -- one kernel converts the logits to FP32, applies
 * the correction bias, runs grouped top-k and both sort phases, and its prepared metadata
 * is consumed by the MoE GEMMs with no second top-k or sort.  Sort-phase contracts (dropped
 * routes, caller-owned integer capacity): "Summary -- general gfx1250 ordinary-TP route
 * optimization" (ROCm/aiter pull 7095), section "Dispatch and contracts".
 *
 * Notation: T tokens, E experts, G = n_group groups of g = E/G consecutive experts,
 * Kg = topk_group kept groups, K = topk experts per token, R = routed_scale,
 * B = block_m, N = T*K routes.
 *
 * What is computed, per token t (all fp32, IEEE expf, IEEE division, no fast-math):
 *   x_e   = float(bf16 logit)                       (exact)
 *   s_e   = 1 / (1 + expf(-x_e))                    sigmoid score
 *   key_e = s_e + bias_e                            selection key (bias steers selection only)
 *   group score of group j = the sum of its two largest keys (its one key when g == 1)
 *   kept groups = the Kg best group scores (equal scores: lower group index first)
 *   topk_ids[t,0..K) = the K best keys among experts of kept groups, best first
 *                      (equal keys: lower expert index first)
 *   topk_weights[t,k] = (s_{id_k} / (s_{id_0} + ... + s_{id_{K-1}})) * R  (sum in slot order)
 * Sort, over the routes r = t*K + k in token-then-slot order:
 *   cnt_e = routes of expert e; pad_e = ceil(cnt_e / B) * B; off_e = sum of pad over
 *   experts below e; num_tokens_post_pad = npp = sum of pad_e;
 *   sorted_token_ids[off_e + i] = the i-th route of expert e (its flat index r),
 *   rows [off_e + cnt_e, off_e + pad_e) = sentinel N with sorted_weights 0,
 *   sorted_weights[p] = topk_weights of the route at row p,
 *   expert_ids[b] = the expert owning rows [b*B, (b+1)*B), for b < npp / B.
 * Entries of sorted_token_ids / sorted_weights at or past npp, and of expert_ids at or
 * past npp / B, are not written.
 *
 * Layouts and ownership: every pointer is DEVICE memory owned by the caller, row-major and
 * contiguous.  logits_bf16: [T, E] bf16 (16-byte aligned base); bias: [E] fp32;
 * topk_ids, topk_weights: [T, K]; sorted_token_ids, sorted_weights:
 * [moe_sort_max_padded(T,E,K,B)]; expert_ids: [moe_sort_max_blocks(T,E,K,B)];
 * num_tokens_post_pad: [1].  "Device memory" includes pinned host memory mapped into the
 * device's address space (zero-copy): pass the address moe_route_sort_map_host returns for it.
 * The kernels then read the logits from, and write the outputs to, host memory over the host
 * link, with no copy enqueued, and the host may read the outputs once the stream has passed the
 * call.  The workspace must be ordinary device memory.  The library allocates nothing, and
 * between calls it keeps on the device only the word that records its proxy check (below)
 * and the scratch of moe_route_sort_noalloc; inputs are never written.  The operations that
 * take a workspace argument only enqueue work on `stream` (no host synchronisation), so they
 * can be captured in a CUDA graph once the first call on the current device has been made
 * outside capture (that call caches device attributes and enqueues the proxy check).
 *
 * Limits: 1 <= E <= 4096, 1 <= G <= 64, E % G == 0, 1 <= Kg <= G, 1 <= K <= 32,
 * K <= Kg * g, B a power of two in [1, 1024], T >= 0, N and the padded length fit in
 * int32.  Logits must be finite (NaN logits give unspecified selections).
 *
 * Errors: every entry point returns MOE_RS_OK (0) or a negative status and, on a negative
 * status, writes nothing and launches nothing (except MOE_RS_ERR_LAUNCH, raised when the
 * CUDA runtime refuses a launch).  Problems only the device can see are reported in the
 * workspace's status word (the first int32 of the workspace, MOE_RS_DEVICE_* bits), valid
 * once the call has completed on the stream; read it with cudaMemcpyAsync if wanted.
 *
 * Devices: a call runs on the CUDA device current in the calling thread, and every pointer
 * must be memory that device can address (its own, or mapped host memory).
 *
 * Exactness of the pruned selection: the multi-CTA route kernels discard experts with a cheap
 * score whose error bound is a property of the GPU's tanh approximation.  The first such call
 * in each device context (made outside stream capture) enqueues an exhaustive check of that
 * bound over all bf16 inputs ahead of its own kernels (one 1024-thread block, once); the
 * kernels prune only where the check has passed and otherwise evaluate every expert exactly
 * (same results, slower).  moe_route_sort_proxy_state reports the outcome.
 */
#ifndef MOE_ROUTE_SORT_H_
#define MOE_ROUTE_SORT_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Host-side status codes (return values). */
#define MOE_RS_OK 0
#define MOE_RS_ERR_NULL_POINTER (-1)      /* a required pointer is NULL (with T > 0)        */
#define MOE_RS_ERR_BAD_EXPERTS (-2)       /* E outside [1, 4096]                           */
#define MOE_RS_ERR_BAD_GROUPS (-3)        /* G outside [1, 64], E % G != 0, Kg outside [1,G] */
#define MOE_RS_ERR_BAD_TOPK (-4)          /* K outside [1, 32] or K > Kg * g               */
#define MOE_RS_ERR_BAD_BLOCK_M (-5)       /* B not a power of two in [1, 1024]             */
#define MOE_RS_ERR_BAD_TOKENS (-6)        /* T < 0 (or T > 8 for moe_gate_route_sort)      */
#define MOE_RS_ERR_OVERFLOW (-7)          /* N or the padded length does not fit in int32  */
#define MOE_RS_ERR_MISALIGNED (-8)        /* logits not 16-byte aligned, or another buffer
                                             not aligned to its element size (workspace: 16) */
#define MOE_RS_ERR_ALIAS (-9)             /* an output overlaps an input or another output */
#define MOE_RS_ERR_WORKSPACE (-10)        /* workspace NULL or smaller than required       */
#define MOE_RS_ERR_BAD_SCALE (-11)        /* routed_scale not finite                       */
#define MOE_RS_ERR_LAUNCH (-12)           /* the CUDA runtime rejected a kernel launch     */
#define MOE_RS_ERR_TOO_LARGE (-13)        /* shape needs more than the static scratch of
                                             moe_route_sort_noalloc                        */
#define MOE_RS_ERR_BAD_HIDDEN (-14)       /* H not a multiple of 8 in [8, 8192]            */
#define MOE_RS_ERR_NOT_MAPPED (-15)       /* host memory not mapped into the device space  */
#define MOE_RS_ERR_BAD_DEBUG_KNOB (-16)   /* moe_route_sort_debug_set: unknown knob         */

/* Device-side status bits, written to the first int32 of the workspace by every call. */
#define MOE_RS_DEVICE_BAD_EXPERT_ID 0x1   /* moe_sort saw an id >= E; those routes dropped */
#define MOE_RS_DEVICE_WAIT_TIMEOUT 0x2    /* a bounded device-side wait gave up (an input copy
                                             did not complete in time); outputs are invalid */

/* ---------------------------------------------------------------- size queries */

/* Worst-case padded length: N + min(E, N) * (B - 1) (each nonempty expert pads by at most
 * B - 1 rows).  Length of sorted_token_ids and sorted_weights.  0 for invalid arguments. */
size_t moe_sort_max_padded(int T, int E, int topk, int block_m);

/* Worst-case number of blocks: floor(moe_sort_max_padded / B).  Length of expert_ids. */
size_t moe_sort_max_blocks(int T, int E, int topk, int block_m);

/* Bytes of device workspace that moe_route_sort and moe_sort need for this shape (16-byte
 * aligned, any contents; the library overwrites what it uses).  One workspace must not be
 * used by two calls that can run at the same time. */
size_t moe_route_sort_workspace_bytes(int T, int E, int topk, int block_m);

/* Device address of pinned host memory, for passing host buffers to the operations below
 * without copies (zero-copy): `host_ptr` must lie in memory allocated with cudaHostAlloc /
 * cudaMallocHost, or registered with cudaHostRegister and the mapped flag.  On systems with
 * unified addressing the address is host_ptr itself.  Writes it to *device_ptr and returns
 * MOE_RS_OK, or MOE_RS_ERR_NOT_MAPPED (host memory the device cannot address) or
 * MOE_RS_ERR_NULL_POINTER.  A host-side query: it enqueues nothing. */
int moe_route_sort_map_host(const void* host_ptr, void** device_ptr);

/* Static text for a status code (host codes above). */
const char* moe_route_sort_strerror(int status);

/* ------------------------------------------------------------------ operations */

/* The whole path: route step (scores, grouped top-k, weights) then sort step.
 * Source: "perf(flydsl): Kimi-K3 B1 route-sort + prepared-MoE handoff (stack)", Summary.
 * Outputs: topk_ids/topk_weights [T,K]; sorted metadata as described above. */
int moe_route_sort(const void* logits_bf16, const float* bias, int T, int E, int n_group,
                   int topk_group, int topk, float routed_scale, int block_m,
                   int32_t* topk_ids, float* topk_weights, int32_t* sorted_token_ids,
                   float* sorted_weights, int32_t* expert_ids,
                   int32_t* num_tokens_post_pad, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream);

/* The whole path with softmax scoring, for MoE families that route on a softmax without a
 * correction bias or expert groups.  The source pages define only the sigmoid + bias scoring
 * above; this is its plain generalisation to the other scoring, over the expert counts and
 * top-k widths that "Summary -- general gfx1250 ordinary-TP route optimization" (ROCm/aiter
 * pull 7095), Generality and negative results, sweeps.  Per token t:
 *   x_e = float(bf16 logit); topk_ids[t,0..K) = the K largest x_e, best first (equal logits:
 *   lower expert index first; -0 and +0 are equal);
 *   m = x of slot 0; q_k = expf(x_{id_k} - m); topk_weights[t,k] = (q_k / (q_0 + ... +
 *   q_{K-1})) * R (sum in slot order) -- the softmax over all E experts restricted to the
 *   selected ones and renormalised, whose normaliser over all E cancels.
 * The sort step, outputs, layouts, workspace, limits (with n_group = topk_group = 1, so
 * 1 <= K <= min(32, E)) and errors are those of moe_route_sort; there is no bias argument. */
int moe_route_sort_softmax(const void* logits_bf16, int T, int E, int topk, float routed_scale,
                           int block_m, int32_t* topk_ids, float* topk_weights,
                           int32_t* sorted_token_ids, float* sorted_weights,
                           int32_t* expert_ids, int32_t* num_tokens_post_pad,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* The router gate projection fused ahead of the whole path, for batch-one decode and other
 * calls of up to 8 tokens ("perf(flydsl): Kimi-K3 B1 route-sort + prepared-MoE handoff
 * (stack)", Summary: the stack specialises the Kimi-K3 B1 gate projection whose logits the
 * route-sort consumes).  First
 *   logits[t,e] = bf16 nearest (ties to even) to sum over h of hidden[t,h] * w_gate[e,h],
 * with the sum accumulated in fp32 in a fixed order (so the same inputs always give the same
 * logits; the rounding is exactly that of the true dot product whenever the fp32 partial
 * sums are exact, for example on coarse value grids), then moe_route_sort on those logits.
 * hidden_bf16: [T,H] bf16, w_gate_bf16: [E,H] bf16 (one row per expert, the layout of a
 * linear layer's weight), both 16-byte aligned device memory, read only; logits_bf16: [T,E]
 * bf16 device output owned by the caller (16-byte aligned), also the path's input.  The
 * projection reads the gate matrix once (E*H*2 bytes); at T <= 8 it is bound by that read, and
 * its arithmetic runs as m16n8k16 bf16 tensor-core MMAs with fp32 accumulation (tokens on the
 * N side).  The route kernels start while it runs and wait for its results on the device, so
 * the call is one stream-ordered sequence.
 * Limits: those of moe_route_sort, plus 0 <= T <= 8 and H a multiple of 8 in [8, 8192].
 * Errors: those of moe_route_sort, plus MOE_RS_ERR_BAD_HIDDEN, MOE_RS_ERR_BAD_TOKENS for
 * T > 8, MOE_RS_ERR_NULL_POINTER / MOE_RS_ERR_MISALIGNED for hidden, w_gate or logits, and
 * MOE_RS_ERR_ALIAS if hidden, w_gate or bias overlaps any output (the logits included) or
 * the workspace. */
int moe_gate_route_sort(const void* hidden_bf16, const void* w_gate_bf16, const float* bias,
                        int T, int E, int H, int n_group, int topk_group, int topk,
                        float routed_scale, int block_m, void* logits_bf16, int32_t* topk_ids,
                        float* topk_weights, int32_t* sorted_token_ids, float* sorted_weights,
                        int32_t* expert_ids, int32_t* num_tokens_post_pad, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream);

/* Route step only ("grouped top-k" of the same Summary): topk_ids/topk_weights [T,K]. */
int moe_topk(const void* logits_bf16, const float* bias, int T, int E, int n_group,
             int topk_group, int topk, float routed_scale, int32_t* topk_ids,
             float* topk_weights, cudaStream_t stream);

/* Sort step only ("both sort phases" of the same Summary) from caller-given routes.
 * topk_ids [T,K] int32: an id < 0 is a dropped route (no slot, not counted: "Summary --
 * general gfx1250 ordinary-TP route optimization", Dispatch and contracts); an id >= E is
 * invalid, dropped, and sets MOE_RS_DEVICE_BAD_EXPERT_ID.  Ids may repeat within a token.
 * topk_weights [T,K] fp32 are copied to the sorted rows. */
int moe_sort(const int32_t* topk_ids, const float* topk_weights, int T, int E, int topk,
             int block_m, int32_t* sorted_token_ids, float* sorted_weights,
             int32_t* expert_ids, int32_t* num_tokens_post_pad, void* workspace,
             size_t workspace_bytes, cudaStream_t stream);

/* Sort step with atomic slot reservation: the arguments, contracts, npp, expert_ids and
 * padding rows of moe_sort, but the rows of one expert's segment hold its routes in an order
 * that depends on how the device's atomics happen to run (no token-then-slot guarantee; two
 * calls may differ).  Per-block shared-memory counts, one global atomic interval reservation
 * per nonempty (expert, block), block-local atomic ranks: the scheme of "Summary -- general
 * gfx1250 ordinary-TP route optimization", Capacity and dispatch.  It exists to measure what
 * moe_sort's deterministic order costs.  Uses the workspace of moe_route_sort_workspace_bytes;
 * zeroes part of it with one cudaMemsetAsync on `stream`. */
int moe_sort_atomic(const int32_t* topk_ids, const float* topk_weights, int T, int E, int topk,
                    int block_m, int32_t* sorted_token_ids, float* sorted_weights,
                    int32_t* expert_ids, int32_t* num_tokens_post_pad, void* workspace,
                    size_t workspace_bytes, cudaStream_t stream);

/* moe_route_sort for callers whose logits live in host memory, as one enqueued sequence on
 * `stream`: copy the T x E bf16 logits from `logits_host` (pinned host memory, for an
 * asynchronous copy) into `logits_dev`, run moe_route_sort on them with the other device
 * arguments, then copy `result_bytes` bytes from `result_dev` (device memory holding the
 * outputs the caller wants back, for example one block containing all of them) to
 * `result_host`.  Returns MOE_RS_ERR_NULL_POINTER for a missing copy pointer, the codes of
 * moe_route_sort, or MOE_RS_ERR_LAUNCH if a copy cannot be enqueued.  Nothing waits: the
 * host results are valid once the stream has reached the end of this sequence. */
int moe_route_sort_from_host(const void* logits_host, void* logits_dev, const float* bias,
                             int T, int E, int n_group, int topk_group, int topk,
                             float routed_scale, int block_m, int32_t* topk_ids,
                             float* topk_weights, int32_t* sorted_token_ids,
                             float* sorted_weights, int32_t* expert_ids,
                             int32_t* num_tokens_post_pad, void* workspace,
                             size_t workspace_bytes, const void* result_dev, void* result_host,
                             size_t result_bytes, cudaStream_t stream);

/* ------------------------------------------------------- allocation-free variant */

/* Bytes of the scratch array that moe_route_sort_noalloc keeps in the library itself. */
#define MOE_RS_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* moe_route_sort without a workspace argument.  (This entry point has no counterpart in the
 * source pages; it exists for callers, not for the method.)
 *
 * Some callers cannot hand the library scratch memory: a plugin invoked by an inference
 * runtime that passes it only its input and output pointers and owns all device memory
 * itself; code that must not call cudaMalloc on the serving path because it synchronises
 * the device and is not stream-ordered; or an engine whose memory budget is fully reserved
 * up front.  For them the scratch lives in a fixed 32 MiB array compiled into the library
 * (MOE_RS_NOALLOC_SCRATCH_BYTES), so this call allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.  Every GPU that loads the library holds those
 * 32 MiB until the process exits.
 *
 * Arguments, outputs, results and errors are those of moe_route_sort, plus
 * MOE_RS_ERR_TOO_LARGE when moe_route_sort_workspace_bytes(T, E, topk, block_m) exceeds
 * MOE_RS_NOALLOC_SCRATCH_BYTES (for example 16384 tokens x 4096 experts x top-8 needs about
 * 9.3 MiB and is accepted); shapes are checked before that, and a rejected call touches
 * nothing.  The first call on each device context looks up the array's device address with
 * that device current and caches it (a context created again, for example after
 * cudaDeviceReset, gets a fresh lookup).
 * All calls on a device share the one array and it keeps whatever the previous call left in
 * it (the path needs no zeroed scratch); two calls that can run on the GPU at the same time
 * (different streams, or graphs replayed concurrently) race on it and give wrong results.
 * The status word of moe_route_sort lands in that shared array: read it with
 * moe_route_sort_noalloc_status. */
int moe_route_sort_noalloc(const void* logits_bf16, const float* bias, int T, int E,
                           int n_group, int topk_group, int topk, float routed_scale,
                           int block_m, int32_t* topk_ids, float* topk_weights,
                           int32_t* sorted_token_ids, float* sorted_weights,
                           int32_t* expert_ids, int32_t* num_tokens_post_pad,
                           cudaStream_t stream);

/* Copies the device status word (MOE_RS_DEVICE_* bits) of the last moe_route_sort_noalloc
 * call on the current device into dst[0] (device memory or mapped pinned host memory, one
 * int32, caller-owned), as a copy enqueued on `stream`: the value is that of the last such
 * call ordered before the copy, valid once the stream reaches it.  It has no counterpart in
 * the source pages.  Returns MOE_RS_OK, MOE_RS_ERR_NULL_POINTER, MOE_RS_ERR_MISALIGNED or
 * MOE_RS_ERR_LAUNCH; it allocates nothing. */
int moe_route_sort_noalloc_status(int32_t* dst, cudaStream_t stream);

/* ------------------------------------------------------------------ diagnostics */

/* Exhaustive check of the bound behind the route kernels' pruning (not an operation of the
 * path; it has no counterpart in the source pages).  The multi-CTA route kernels discard an
 * expert only when a cheap score 0.5 * tanh.approx(0.5 x) + 0.5 proves it cannot be
 * selected; that proof assumes |cheap - exact sigmoid| <= bound for every bf16 x.  Writes
 * out2[0] = the largest difference over all finite bf16 inputs on this device and
 * out2[1] = the bound assumed (device memory, 2 floats, caller-owned; valid after the
 * stream reaches this call).  Selection stays exact only if out2[0] <= out2[1]; the library
 * runs the same check itself (see "Exactness of the pruned selection" above). */
int moe_route_sort_proxy_selftest(float* out2, cudaStream_t stream);

/* The library's own record of that check on the current device: copies into dst[0] (device
 * memory or mapped pinned host memory, one int32) 0 if no check has run in this context yet,
 * 1 if the bound held (the route kernels prune), 2 if it failed (they evaluate every expert
 * exactly).  Enqueued on `stream`; valid once the stream reaches it. */
int moe_route_sort_proxy_state(int32_t* dst, cudaStream_t stream);

/* Test hooks (process-wide settings read when later calls launch; no counterpart in the source
 * pages).  They exist so that the failure paths can be exercised on a healthy GPU:
 *   MOE_RS_DEBUG_WAIT_LIMIT_NS     every bounded device wait of the multi-CTA path (row copies,
 *                                  the sort step's look-back) gives up after `value` ns;
 *                                  0 gives up at once without waiting, which makes those calls
 *                                  report MOE_RS_DEVICE_WAIT_TIMEOUT (outputs invalid, every
 *                                  write still inside the caller's buffers); a negative value
 *                                  restores the default of 200 ms.  Copies already in flight
 *                                  are still waited for (with the default bound) before a CTA
 *                                  exits.
 *   MOE_RS_DEBUG_FORCE_PROXY_FAIL  `value` != 0: the in-library proxy check reports a failure
 *                                  (it runs again in each context on the next call that would
 *                                  prune), so the route kernels evaluate every expert exactly;
 *                                  0 restores the real check.
 *   MOE_RS_DEBUG_CLUSTER_TOKENS    largest T that moe_route_sort and moe_route_sort_softmax run
 *                                  as one thread-block cluster (route step and both sort
 *                                  phases in one launch) instead of the three-kernel multi-CTA
 *                                  path, and moe_sort likewise, whatever the sizes; 0 turns
 *                                  the cluster paths off, a negative value restores the
 *                                  default reach (moe_route_sort: T <= 256 and at most 512 KiB
 *                                  of logits, for shapes the segment route kernel takes;
 *                                  moe_sort: at most 8192 routes; both: a worst-case padded
 *                                  length of at most 65536 rows).
 *   MOE_RS_DEBUG_GRID_TOKENS       largest T that moe_route_sort and moe_route_sort_softmax run
 *                                  on a cooperative grid with one CTA per token (taken before
 *                                  every other multi-token path but the warp-per-token grid;
 *                                  2 <= T <= min(320, value));
 *                                  0 turns it off, a negative value restores the default
 *                                  (5 <= T <= 320, when the grid's shared memory fits).
 *   MOE_RS_DEBUG_WARP_GRID_TOKENS  moe_route_sort and moe_route_sort_softmax run calls of
 *                                  more than `value` tokens (and at least 2) on a cooperative
 *                                  grid with one warp per token and up to 16 tokens per CTA
 *                                  (taken before every other multi-token path, while
 *                                  ceil(T / #SMs) <= 16 and its shared memory fits); a negative
 *                                  value restores the default (128 < T <= 2048).
 *                                  The paths give the same outputs; these hooks let tests
 *                                  compare them on one shape.
 * Returns MOE_RS_OK or MOE_RS_ERR_BAD_DEBUG_KNOB. */
#define MOE_RS_DEBUG_WAIT_LIMIT_NS 1
#define MOE_RS_DEBUG_FORCE_PROXY_FAIL 2
#define MOE_RS_DEBUG_CLUSTER_TOKENS 3
#define MOE_RS_DEBUG_GRID_TOKENS 4
#define MOE_RS_DEBUG_WARP_GRID_TOKENS 5
int moe_route_sort_debug_set(int knob, long long value);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTE_SORT_H_ */
