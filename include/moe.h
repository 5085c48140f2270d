/*
 * moe.h -- C ABI of libmoe, the GB300 (sm_103a) routed-expert MoE layer.
 *
 * The layer, as the Hebrus "Agent Field Notes" state it:
 *   router logits -> float32 softmax over the selected experts, top-k in rank
 *   order -> token rows grouped by expert -> per expert SwiGLU
 *   (gate and up together, then down) -> weighted sum in route-rank order;
 *   plus deduplication of repeated routes across a verifier block.
 *
 * Conventions shared by every call:
 *  - Every pointer is a DEVICE pointer owned by the caller, except where a
 *    comment says otherwise.  The library allocates no device memory: where a
 *    call needs scratch space the caller passes it in (see *_workspace_size).
 *  - bf16 values travel as uint16_t bit patterns; all arrays are dense and
 *    row-major with the shapes given in brackets.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and the calls return before it completes.
 *  - Arguments are checked on the host BEFORE anything is enqueued.  A call
 *    that returns anything but MOE_OK has enqueued nothing and written
 *    nothing: the rule of AFN-010 "One bank flip is enough: make the whole
 *    inference chunk transactional", section "The publication model" (output
 *    remains caller-private while work is fallible), applied to rejection.
 *  - Errors seen on the device (an expert ID outside [0,E), a non-finite
 *    output, a bounded wait that ran out) are OR-ed into *dev_status as
 *    MOE_DEV_* bits; the caller reads it after synchronising.  No kernel
 *    traps.  dev_status may be NULL where a call says so.
 *  - Supported geometry (anything else returns MOE_ENOTSUP):
 *      1 <= k <= 32, k <= E <= 1024, H % 128 == 0, I % 64 == 0,
 *      T * k < 2^31, 16-byte aligned pointers for every bf16/f32 array.
 *    T == 0 is accepted and enqueues nothing.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_EINVAL = 1,          /* null pointer, misaligned pointer, bad enum       */
  MOE_ESHAPE = 2,          /* inconsistent or non-positive sizes               */
  MOE_ERANGE = 3,          /* reserved: device-side range errors use dev_status */
  MOE_ECUDA = 4,           /* a CUDA runtime/driver call failed                */
  MOE_ENOTSUP = 5,         /* geometry outside the supported envelope          */
  MOE_EDEVICE_TIMEOUT = 6, /* reserved: device-side timeouts use dev_status    */
  MOE_EWORKSPACE = 7       /* workspace pointer null or smaller than required  */
} moe_status;

/* Bits OR-ed into *dev_status by kernels. */
#define MOE_DEV_BAD_EXPERT 0x1 /* an expert ID outside [0, E) was seen       */
#define MOE_DEV_NONFINITE 0x2  /* a layer output was NaN or infinite         */
#define MOE_DEV_TIMEOUT 0x4    /* a bounded pipeline wait ran out            */
#define MOE_DEV_CACHE_FULL 0x8 /* routed experts did not fit the expert cache */

typedef enum moe_wfmt {
  MOE_W_BF16 = 0,          /* bf16 weights, plain record layout                  */
  MOE_W_INT4_G64 = 1,      /* int4 codes + bf16 scale per 64 inputs, plain layout
                              (input of moe_pack_experts only)                   */
  MOE_W_BF16_TILED = 2,    /* bf16 weights packed by moe_pack_experts            */
  MOE_W_INT4_G64_TILED = 3 /* int4 g64 weights packed by moe_pack_experts        */
} moe_wfmt;

/* ABI version of this header (major * 100 + minor). */
MOE_API int moe_abi_version(void);

/* Human-readable name of a status code (static storage; never NULL). */
MOE_API const char *moe_status_str(moe_status s);

/* Number of streaming multiprocessors of the current device, or -1. */
MOE_API int moe_device_sm_count(void);

/* ---------------------------------------------------------------------------
 * moe_route -- router logits, top-k in rank order, renormalised weights.
 *
 * Source: AFN-001 "Porting Qwen3.8-Flash-Next to Hebrus: evidence before
 * execution", section "Phase 1: separate math from acceleration" (float32
 * router softmax and normalized top-10 selection); AFN-021 "Replay decode as
 * prefill", section "The key equivalence -- and where it breaks" (IDs and
 * their rank order are the label; weights compared within a tolerance).
 *
 *   L[t,e]  = sum_h x[t,h] * w_router[e,h] + bias[e]      (fp32 accumulate)
 *   ids[t]  = the k experts with the largest L[t,:], ordered by logit
 *             descending, ties broken by the lower expert ID
 *   w[t,j]  = exp(L[t,ids_j] - L[t,ids_0]) / sum_j' exp(L[t,ids_j'] - L[t,ids_0])
 *   gap[t]  = L(k-th) - L((k+1)-th), +inf when k == E
 *
 *   x          [T,H] bf16          w_router [E,H] bf16
 *   bias       [E] f32, or NULL    topk_ids [T,k] int32 (out)
 *   topk_w     [T,k] f32 (out)     gap      [T] f32 (out) or NULL
 *   workspace  >= moe_route_workspace_size(T,E) bytes, 256-byte aligned;
 *              contents need no initialisation and are clobbered.
 * ------------------------------------------------------------------------- */
MOE_API size_t moe_route_workspace_size(int T, int E);
MOE_API moe_status moe_route(const uint16_t *x, const uint16_t *w_router, const float *bias, int T, int H,
                     int E, int k, int32_t *topk_ids, float *topk_w, float *gap, void *workspace,
                     size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * moe_route_noalloc -- moe_route for callers that cannot allocate device
 * memory.  The pages have no counterpart to this entry point; it exists for
 * callers that are handed their inputs and outputs but have no way to
 * allocate a workspace (a host framework that owns every device buffer, or a
 * path on which allocating is not allowed).
 *
 * Same arguments and results as moe_route, without the workspace: the
 * [T,E] fp32 logits scratch lives in a fixed 256 KB array inside the library
 * (held by every GPU that loads it, until exit).  Limits: T <= 64 and
 * E <= 1024.  T > 64 returns MOE_EWORKSPACE; E > 1024 is beyond the router's
 * own limit and returns MOE_ENOTSUP; either way nothing is enqueued.  Every
 * call looks up the array's device address for the current device (a host
 * lookup, so a reset device never gets a stale address); the first call on a
 * device may load the library's device code, so make it before any stream
 * capture.  All
 * calls share the array: calls that overlap on the GPU (e.g. on two streams)
 * race.  Nothing in the array needs to start at zero.  No allocation of any
 * kind is made.
 * ------------------------------------------------------------------------- */
MOE_API moe_status moe_route_noalloc(const uint16_t *x, const uint16_t *w_router, const float *bias, int T,
                                     int H, int E, int k, int32_t *topk_ids, float *topk_w, float *gap,
                                     void *stream);

/* ---------------------------------------------------------------------------
 * moe_permute -- group token rows by expert (count, exclusive scan, stable
 * scatter), optionally gathering the rows of x into expert order.
 *
 * Source: AFN-019 "Hide SSD misses before the router knows they exist",
 * section "Why overlap alone cannot defeat the byte roofline" (grouping token
 * rows by expert as a byte owner).
 *
 * With R = T*k and flat route index r = t*k + j:
 *   counts[e]   = #{r : topk_ids[r] == e}                       [E] int32 (out)
 *   offsets[e]  = sum_{e' < e} counts[e'], offsets[E] = R       [E+1] int32 (out)
 *   perm[s]     = the route stored in slot s; the slots of expert e are
 *                 offsets[e] .. offsets[e+1]-1 in ascending r    [R] int32 (out)
 *   inv_perm[r] = the slot of route r (perm[inv_perm[r]] == r)   [R] int32 (out)
 *   x_perm[s,:] = x[perm[s] / k, :]  if x_perm != NULL          [R,H] bf16 (out)
 * x may be NULL only when x_perm is NULL.  An ID outside [0,E) sets
 * MOE_DEV_BAD_EXPERT in *dev_status (required, 4 bytes) and the kernel then
 * writes none of counts/offsets/perm/inv_perm/x_perm.  The row gather also
 * writes nothing while *dev_status holds MOE_DEV_BAD_EXPERT from an earlier
 * call (the word is sticky until the caller clears it).
 * ------------------------------------------------------------------------- */
MOE_API moe_status moe_permute(const int32_t *topk_ids, int T, int k, int E, const uint16_t *x, int H,
                       int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv_perm,
                       uint16_t *x_perm, int32_t *dev_status, void *stream);

/* ---------------------------------------------------------------------------
 * moe_permute_ws -- moe_permute for large route counts, on many CTAs.
 *
 * Source: as moe_permute.  Arguments, outputs, dev_status and the result are
 * exactly those of moe_permute (bit for bit: the slot order is fixed by the
 * definition).  The routes are cut into chunks of 2,048; one launch counts
 * each chunk's routes per expert, one CTA scans the counts into offsets and
 * each chunk's per-expert start, and one launch scatters every chunk.
 * workspace: device, 16-byte aligned, at least moe_permute_workspace_size(T,
 * k, E) bytes, owned by the caller, contents on entry do not matter; it must
 * not be used by another call in flight at the same time.  NULL or too small:
 * MOE_EWORKSPACE; misaligned: MOE_EINVAL.  An ID outside [0,E) sets
 * MOE_DEV_BAD_EXPERT and then none of counts/offsets/perm/inv_perm/x_perm
 * is written.
 * ------------------------------------------------------------------------- */
MOE_API size_t moe_permute_workspace_size(int T, int k, int E);
MOE_API moe_status moe_permute_ws(const int32_t *topk_ids, int T, int k, int E, const uint16_t *x, int H,
                                  int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv_perm,
                                  uint16_t *x_perm, void *workspace, size_t workspace_bytes,
                                  int32_t *dev_status, void *stream);

/* ---------------------------------------------------------------------------
 * moe_route_permute -- moe_route followed by moe_permute (without the row
 * gather) for a decode block of T <= 16 tokens, in one launch.
 *
 * Sources: as moe_route and moe_permute.  Outputs: topk_ids, topk_w, gap as
 * moe_route; counts, offsets, perm, inv_perm as moe_permute.  The selection
 * rule and the grouping are the same; the logits are summed in a different
 * (fixed) order than moe_route's, so a route whose 10th and 11th logits are
 * within rounding of each other may differ between the two entry points.
 * Runs as one 16-CTA thread-block cluster; returns MOE_ENOTSUP for T > 16 or
 * on a device that cannot run such a cluster (use moe_route + moe_permute).
 * On GB300 it is slower than moe_route + moe_permute issued back to back with
 * programmatic launch (16 SMs pull the whole router matrix); it serves callers
 * that want a single launch.
 * No workspace.  dev_status (required) gets MOE_DEV_BAD_EXPERT as moe_permute.
 * ------------------------------------------------------------------------- */
MOE_API moe_status moe_route_permute(const uint16_t *x, const uint16_t *w_router, const float *bias, int T, int H,
                                     int E, int k, int32_t *topk_ids, float *topk_w, float *gap, int32_t *counts,
                                     int32_t *offsets, int32_t *perm, int32_t *inv_perm, int32_t *dev_status,
                                     void *stream);

/* ---------------------------------------------------------------------------
 * Expert contractions (tensor cores: tcgen05 MMA, TMEM accumulators, TMA).
 *
 * Source: AFN-019, section "Why overlap alone cannot defeat the byte roofline"
 * (one expert = gate [I,H] + up [I,H] + down [H,I]) and section "Hypothesis
 * H4: ExpertMajor should stream as a wavefront, not a barrier" (gate and up
 * are used together; down only once the SwiGLU intermediate exists).
 *
 * Expert weight record layout (one contiguous record per expert):
 *   MOE_W_BF16:     w_gateup [E, 2I, H] bf16: rows 0..I-1 gate, I..2I-1 up
 *                   w_down   [E, H, I]  bf16
 *                   s_gateup = s_down = NULL
 *   MOE_W_BF16_TILED, MOE_W_INT4_G64_TILED: the records as moe_pack_experts
 *                   writes them (w_* its output, s_* NULL).
 *   MOE_W_INT4_G64 (plain; accepted by moe_pack_experts only):
 *                   w_gateup [E, 2I, H/2] uint8, w_down [E, H, I/2] uint8,
 *                   two signed 4-bit codes per byte (two's complement, -8..7),
 *                   even input index in the low nibble; s_gateup [E, 2I, H/64]
 *                   and s_down [E, H, I/64] bf16, one scale per 64 consecutive
 *                   inputs of a row; w = scale * code.  (AFN-001, section
 *                   "Phase 2": affine4 with group size 64, read as symmetric
 *                   codes with one bf16 scale per group.)  Decode-sized
 *                   launches (up to 320 slots, K <= 2560) multiply the exact
 *                   codes with the token values rounded to fp16 (exact inside
 *                   fp16's normal range; magnitudes of 65,520 and more become
 *                   infinite) and apply the scale in fp32; larger launches
 *                   give the tensor cores w = bf16(scale * code).
 *
 * moe_expert_gateup:  for every slot s of expert e (offsets from moe_permute)
 *     g = Wgate_e . x_perm[s],  u = Wup_e . x_perm[s]      (fp32 accumulate)
 *     h[s,i] = bf16( silu(g_i) * u_i ),  silu(z) = z / (1 + exp(-z))
 *   x_perm [R,H] bf16, offsets [E+1] int32, h [R,I] bf16 (out)
 *
 * moe_expert_down:  y_perm[s,:] = Wdown_e . h[s]           (fp32 accumulate)
 *   h [R,I] bf16, offsets [E+1] int32, y_perm [R,H] f32 (out)
 *
 * moe_grouped_swiglu: moe_expert_gateup then moe_expert_down on one stream;
 *   h is caller-owned scratch of R*I bf16.
 *
 * R is T*k of the routing call; slots past offsets[E] are not touched.
 * dev_status (4 bytes, required) gets MOE_DEV_TIMEOUT if a bounded pipeline
 * wait ran out (the kernel then stops early; outputs are incomplete).
 *
 * Launch overlap (decode-sized int4 launches over resident records): a
 * gate/up call issued right after moe_permute's row gather, and a down
 * call issued right after a gate/up call, over the same offsets on the same
 * stream, start streaming their weights before the call in front of them
 * has finished; they wait for it only where they read its output (x_perm
 * or h).  The library decides this from its own launch order on the
 * stream, so any other order is safe and simply waits: it needs no action
 * from the caller.  Calls that share a stream are issued from one host
 * thread at a time, as their order on the stream requires anyway.
 * ------------------------------------------------------------------------- */
MOE_API moe_status moe_expert_gateup(const uint16_t *x_perm, const int32_t *offsets, int R, int E, int H,
                             int I, int fmt, const void *w_gateup, const uint16_t *s_gateup,
                             uint16_t *h, int32_t *dev_status, void *stream);
MOE_API moe_status moe_expert_down(const uint16_t *h, const int32_t *offsets, int R, int E, int H, int I,
                           int fmt, const void *w_down, const uint16_t *s_down, float *y_perm,
                           int32_t *dev_status, void *stream);
MOE_API moe_status moe_grouped_swiglu(const uint16_t *x_perm, const int32_t *offsets, int R, int E, int H,
                              int I, int fmt, const void *w_gateup, const uint16_t *s_gateup,
                              const void *w_down, const uint16_t *s_down, uint16_t *h,
                              float *y_perm, int32_t *dev_status, void *stream);

/* ---------------------------------------------------------------------------
 * moe_expert_swiglu_fused -- moe_grouped_swiglu in one persistent launch for
 * tile-packed bf16 records (fmt = MOE_W_BF16_TILED): the down tiles of an
 * expert start as soon as that expert's gate/up tiles have stored h, so the
 * two contractions share the GPU instead of meeting at a kernel boundary.
 * Optionally the launch also does moe_permute's row gather first.
 *
 * Same arithmetic and outputs (h, y_perm) as moe_grouped_swiglu, plus
 *   x        [R/k, H] bf16 or NULL.  If given, the launch first writes
 *            x_perm[s,:] = x[perm[s] / k, :] for every slot (perm [R] int32
 *            from moe_permute, k the routes per token, R % k == 0), exactly
 *            what moe_permute's gather writes; if NULL, x_perm is an input
 *            holding those rows and k, perm are ignored.
 *   sync_ws  [E+3] int32 scratch, zero-filled before its first use; a call
 *            that completes leaves it zero-filled again.  After a call whose
 *            dev_status shows MOE_DEV_TIMEOUT, zero it again.  Calls that
 *            share one sync_ws must not overlap on the GPU.
 * The launch is persistent (one CTA per SM) and its CTAs wait on one another
 * (bounded): do not run it beside work that could keep some of its CTAs from
 * becoming resident.
 * ------------------------------------------------------------------------- */
MOE_API moe_status moe_expert_swiglu_fused(const uint16_t *x, int k, const int32_t *perm, uint16_t *x_perm,
                                           const int32_t *offsets, int R, int E, int H, int I, int fmt,
                                           const void *w_gateup, const void *w_down, uint16_t *h, float *y_perm,
                                           int32_t *sync_ws, int32_t *dev_status, void *stream);

/* ---------------------------------------------------------------------------
 * moe_expert_swiglu_fused_weighted -- moe_expert_swiglu_fused with the route
 * weight applied inside the launch and bf16 expert outputs: for every slot s
 * with route weight w_s = topk_w[perm[s]],
 *   h[s,:]       = bf16( w_s * silu(g) * u )        [R,I] bf16 (out)
 *   yw_perm[s,:] = bf16( W_down h[s,:] )            [R,H] bf16 (out)
 * in place of the fp32 y_perm (W_down is linear, so yw_perm carries the
 * route weight).  For prefill-sized calls this halves the bytes of the expert
 * outputs, written here and read again by the combine (moe_combine_weighted),
 * at the cost of one bf16 rounding per route term.
 * Source: AFN-019, section "Hypothesis H4" (results of ready experts go to
 * separate slots; the weighted sum follows route-rank order).
 *   perm    [R] int32 from moe_permute (required), k the routes per token,
 *           R % k == 0;  topk_w [T*k] f32, the route weights of moe_route.
 * A perm entry outside [0,R) sets MOE_DEV_BAD_EXPERT and leaves that slot's
 * row unwritten.  Everything else (x, x_perm, h, sync_ws, the persistent
 * launch) is as moe_expert_swiglu_fused.
 * ------------------------------------------------------------------------- */
MOE_API moe_status moe_expert_swiglu_fused_weighted(const uint16_t *x, int k, const int32_t *perm,
                                                    uint16_t *x_perm, const int32_t *offsets, int R, int E, int H,
                                                    int I, int fmt, const void *w_gateup, const void *w_down,
                                                    const float *topk_w, uint16_t *h, uint16_t *yw_perm,
                                                    int32_t *sync_ws, int32_t *dev_status, void *stream);

/* ---------------------------------------------------------------------------
 * Expert records in host memory, served through an HBM slot cache.
 *
 * Source: AFN-019 "Hide SSD misses before the router knows they exist",
 * sections "Why overlap alone cannot defeat the byte roofline" (the routed
 * records fetched from the slower tier are the first-order cost) and
 * "Hypothesis H4" (gate/up and down records of one expert, fetched whole).
 * On GB300 the slower tier is Grace memory behind NVLink-C2C: the packed
 * records (moe_pack_experts output) of all E experts live in pinned host
 * memory that the GPU reads directly; S slots of HBM hold recent experts.
 *
 * moe_cache_plan -- one CTA.  State (device, caller-owned, persistent across
 *   calls): slot_of [E] int32 (slot of each expert or -1), expert_of [S]
 *   int32 (expert in each slot or -1), hand [2] int32 {FIFO hand, call
 *   counter}; initialise to -1, -1, {0, 0}.  From counts [E] (moe_permute):
 *   routed experts with a slot are hits, the others misses (expert order).
 *   Slots holding an expert routed in this call are pinned; the others are
 *   victims in the order of `policy`, ties to the lower slot:
 *     MOE_CACHE_FIFO  rotation order from the hand;
 *     MOE_CACHE_LRU   empty slots, then least recent use; needs last_use [S]
 *                     int32 (initialise to -1);
 *     MOE_CACHE_SCORE empty slots, then lowest score(record) (AFN-019, "Two
 *                     storage workloads, not one": P(use before eviction) x
 *                     expected exposed latency avoided / resident bytes;
 *                     whole records of one size, so the order is that of
 *                     P(use), estimated per expert as f <- decay * f +
 *                     [routed in this call], one fp32 fused multiply-add);
 *                     needs score [E] fp32 (initialise to 0), 0 <= decay < 1
 *                     (MOE_ERANGE otherwise).
 *   Miss m takes the m-th victim.  Writes miss_list [S] (experts to fetch),
 *   miss_slot [S] (their slots), stats[0..1] = {hits, misses} of this call,
 *   adds them to the running totals stats[2..3] (the caller zeroes those),
 *   and updates the state.  If the misses do not fit (more routed experts
 *   than unpinned slots), sets MOE_DEV_CACHE_FULL, counts the call as
 *   {hits, 0} and leaves the slots unchanged (the call counter and the use
 *   rates still advance).  S <= 1024, E <= 1024.
 * moe_cache_fetch -- copies the planned misses' records from host memory
 *   (host_gateup / host_down, E records of rec_* bytes, 16-byte aligned) into
 *   the pools (S records each); reads the miss count from stats on the
 *   device, so the plan and the fetch need no host round trip.
 * ------------------------------------------------------------------------- */
#define MOE_CACHE_FIFO 0
#define MOE_CACHE_LRU 1
#define MOE_CACHE_SCORE 2
MOE_API moe_status moe_cache_plan(const int32_t *counts, int E, int32_t *slot_of, int32_t *expert_of, int S,
                                  int32_t *hand, int policy, float decay, float *score, int32_t *last_use,
                                  int32_t *miss_list, int32_t *miss_slot, int32_t *stats, int32_t *dev_status,
                                  void *stream);
MOE_API moe_status moe_cache_fetch(const void *host_gateup, const void *host_down, size_t rec_gateup,
                                   size_t rec_down, const int32_t *miss_list, const int32_t *miss_slot,
                                   const int32_t *stats, void *pool_gateup, void *pool_down, void *stream);

/* ---------------------------------------------------------------------------
 * Route sidecar forward pass.
 *
 * Source: AFN-021 "Replay decode as prefill: a training flywheel for
 * predictive MoE I/O", section "What feature should the sidecar see?": an
 * opaque feature vector goes through a low-rank trunk shared by all layers,
 * the target layer's embedding is added, scores against expert-head
 * embeddings shared by all layers give one score per expert, and the ranked
 * experts are the prefetch candidates.  Readings: no nonlinearity (the
 * pages name none), bf16 weights, fp32 arithmetic.
 *
 * moe_sidecar_prepare -- head_bias [L, E] fp32 = w_head [E, r] bf16 .
 *   layer_emb [L, r] bf16, once per weight set.
 * moe_sidecar_forward -- for feat [T, F] bf16 (the feature of each
 *   position): z [T, r] fp32 = feat . w_trunk^T (w_trunk [r, F] bf16), then
 *   for every layer l the scores w_head (z + layer_emb[l]), computed as
 *   w_head z + head_bias[l], and the N best experts in rank order
 *   (ties to the lower expert ID): cand [T, L, N] int32, cand_score [T, L, N]
 *   fp32.  F % 128 == 0, r % 8 == 0, r <= 1024, E <= 1024, N <= 32, N <= E.
 *   A non-finite score sets MOE_DEV_NONFINITE.
 * ------------------------------------------------------------------------- */
MOE_API moe_status moe_sidecar_prepare(const uint16_t *w_head, const uint16_t *layer_emb, int E, int r, int L,
                                       float *head_bias, void *stream);
MOE_API moe_status moe_sidecar_forward(const uint16_t *feat, const uint16_t *w_trunk, const uint16_t *w_head,
                                       const float *head_bias, int T, int F, int r, int E, int L, int N, float *z,
                                       int32_t *cand, float *cand_score, int32_t *dev_status, void *stream);

/* ---------------------------------------------------------------------------
 * Selected records or the whole layer.
 *
 * Source: AFN-019, section "Hypothesis H5: prefill and decode need different
 * streaming modes": decode and small blocks read the selected records; a
 * large prefill tile routes to most experts, where one sequential layer
 * extent may cost less than sparse reads; macro prefill streams layer l+1
 * into a two-layer ring while layer l computes; the crossover is measured
 * from the unique-record fraction and sustained bandwidth, not guessed from
 * the prompt length.
 *
 * moe_layer_stream -- host -> device copy of a whole layer's packed records
 *   (bytes_* each a multiple of 16, 16-byte aligned), one copy-engine copy
 *   per component on `stream`: the ring fill of macro prefill.
 * moe_stream_mode -- host only: the cheaper way to bring a call's U distinct
 *   records (of E, record_bytes each) to the device, from measured rates:
 *   t_selected = overhead + U * record_bytes / selected_gbs (0 when U = 0),
 *   t_layer = E * record_bytes / layer_gbs (times in microseconds, rates in
 *   GB/s).  Returns MOE_STREAM_LAYER if t_layer < t_selected, else
 *   MOE_STREAM_SELECTED; -1 on an argument out of range.  Writes the two
 *   times when the pointers are not NULL.
 * ------------------------------------------------------------------------- */
#define MOE_STREAM_SELECTED 0
#define MOE_STREAM_LAYER 1
MOE_API moe_status moe_layer_stream(const void *host_gateup, const void *host_down, size_t bytes_gateup,
                                    size_t bytes_down, void *dev_gateup, void *dev_down, void *stream);
MOE_API int moe_stream_mode(int U, int E, double record_bytes, double selected_gbs, double layer_gbs,
                            double selected_overhead_us, double *t_selected_us, double *t_layer_us);

/* moe_expert_int4_slots -- moe_expert_gateup (kind 0) or moe_expert_down
 *   (kind 1) for int4 g64 records held in an HBM slot cache: pool holds S
 *   tile-packed int4 records of that component (MOE_W_INT4_G64_TILED layout,
 *   one expert each, 2,611,200 B per expert at the Qwen4Exp shape against
 *   9,830,400 B in bf16) and expert e's record is record slot_of[e]
 *   (moe_cache_plan; the misses copied by moe_cache_fetch with the int4
 *   record sizes).  rows: x_perm [R,H] bf16 (kind 0) or h [R,I] bf16
 *   (kind 1); out: h [R,I] bf16 (kind 0) or y_perm [R,H] f32 (kind 1).  Same
 *   arithmetic as the resident int4 path, so the same bits.  A routed expert
 *   whose slot_of entry is outside [0, S) is read from slot 0 and flags
 *   MOE_DEV_CACHE_FULL.  Decode-sized launches only (R <= 320 routes, K <=
 *   2,560 inputs): MOE_ENOTSUP otherwise. */
MOE_API moe_status moe_expert_int4_slots(int kind, const uint16_t *rows, const int32_t *offsets, int R, int E,
                                         int H, int I, const void *pool, int S, const int32_t *slot_of, void *out,
                                         int32_t *dev_status, void *stream);

/* moe_expert_int4_fetch -- moe_expert_int4_slots(kind 0, gate/up) that also
 *   fetches the plan of moe_cache_plan (miss_list, miss_slot, stats) from the
 *   host records (host_gateup / host_down: E tile-packed int4 records each,
 *   pinned host memory the device can read, 16-byte aligned) into the slot
 *   pools pool_gateup / pool_down: two extra warps per CTA copy the misses'
 *   gate/up records, then their down records, over the CPU-GPU link while the
 *   resident experts compute (their tiles come first); a fetched expert's
 *   tiles start once their 128-row blocks have landed.  The down launch that
 *   follows (moe_expert_int4_slots, kind 1) finds every down record in place.
 *   Source: AFN-019, section "Hypothesis H4" (gate and up of an expert
 *   together, down once h exists; ready experts compute at once).
 *   sync_ws: [2 + E * I/64] int32, zero before the first call; every launch
 *   leaves it zero again (after a launch that flagged MOE_DEV_TIMEOUT, zero
 *   it).  The CTAs wait on one another's copies (bounded).  Decode-sized
 *   launches only (MOE_ENOTSUP otherwise). */
MOE_API moe_status moe_expert_int4_fetch(const uint16_t *x_perm, const int32_t *offsets, int R, int E, int H, int I,
                                         void *pool_gateup, void *pool_down, int S, const int32_t *slot_of,
                                         const void *host_gateup, const void *host_down, const int32_t *miss_list,
                                         const int32_t *miss_slot, const int32_t *stats, uint16_t *h,
                                         int32_t *sync_ws, int32_t *dev_status, void *stream);

/* moe_expert_swiglu_cached -- moe_expert_swiglu_fused over slot pools:
 *   pool_gateup / pool_down hold S tile-packed bf16 records (MOE_W_BF16_TILED
 *   layout, one expert each) and expert e's records are record slot_of[e].
 *   A routed expert whose slot_of entry is outside [0, S) is read from slot 0
 *   and flags MOE_DEV_CACHE_FULL.
 *   host_gateup == NULL: the slots are already filled (moe_cache_fetch).
 *   host_gateup != NULL: the launch fetches the plan of moe_cache_plan itself
 *   (miss_list, miss_slot, stats) from the host records (host_gateup /
 *   host_down, E records each, pinned host memory the device can read, 16-byte
 *   aligned): extra warps copy the records over the CPU-GPU link in 32 KiB
 *   pieces while the experts already resident compute, and the tiles of each
 *   missing expert start once its record has landed.  Order of the copies: the
 *   wave order of AFN-019 "Hypothesis H4" with `wave` experts per wave (gate/up
 *   of wave 0; then per wave w the gate/up records of wave w and the down
 *   records of wave w-1; then the last down records); wave >= the number of
 *   misses copies every gate/up record before any down record.  The combine
 *   that follows stays in route-rank order.  Needs H/64 and I/64 even
 *   (MOE_ENOTSUP otherwise).
 *   sync_ws: [E * (1 + I/64 + H/128) + 4] int32 (per-expert readiness, and a
 *   landed-piece counter per weight block), zero before the first call;
 *   every launch leaves it zero again. */
MOE_API moe_status moe_expert_swiglu_cached(const uint16_t *x, int k, const int32_t *perm, uint16_t *x_perm,
                                            const int32_t *offsets, int R, int E, int H, int I, int fmt,
                                            void *pool_gateup, void *pool_down, int S, const int32_t *slot_of,
                                            const void *host_gateup, const void *host_down,
                                            const int32_t *miss_list, const int32_t *miss_slot,
                                            const int32_t *stats, int wave, uint16_t *h, float *y_perm,
                                            int32_t *sync_ws, int32_t *dev_status, void *stream);

/* ---------------------------------------------------------------------------
 * moe_pack_experts -- reorder one component of every expert record into the
 * tile order the contraction streams (done once, like loading a checkpoint).
 *
 * Source: AFN-019, section "Hypothesis H4" (ExpertMajor: one contiguous record
 * per expert with explicit component extents).  Each expert's component stays
 * contiguous; inside it, bytes are ordered by (128-row weight block, 64-input
 * step) so that every pipeline stage is one contiguous chunk:
 *   MOE_W_BF16 in -> MOE_W_BF16_TILED out: 16,384-byte chunks, the 128-byte-
 *     swizzled image of a 128 x 64 bf16 tile;
 *   MOE_W_INT4_G64 in -> MOE_W_INT4_G64_TILED out: 4,352-byte chunks, 128 rows
 *     x 32 code bytes followed by the 128 rows' bf16 scales of that group; in
 *     each 32-bit word the eight codes are stored offset by +8, nibble j
 *     holding element 0,2,4,6,1,3,5,7 of the word's eight inputs.
 * which = 0: gate/up (w [E,2I,H] or codes [E,2I,H/2] + s [E,2I,H/64]); gate/up
 *   tiles hold 16 gate rows then the 16 matching up rows, four times.
 * which = 1: down (w [E,H,I] or codes [E,H,I/2] + s [E,H,I/64]).
 * out must hold moe_pack_size(...) bytes, 16-byte aligned, and must not
 * overlap the input.
 * ------------------------------------------------------------------------- */
MOE_API size_t moe_pack_size(int fmt_in, int E, int H, int I, int which);
MOE_API moe_status moe_pack_experts(int fmt_in, const void *w, const uint16_t *s, int E, int H, int I,
                                    int which, void *out, size_t out_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * moe_combine -- weighted sum of expert outputs in route-rank order.
 *
 * Source: AFN-019, section "Hypothesis H4" (the final weighted sum follows a
 * deterministic route-rank order).
 *
 *   acc[t,:] = sum_{j=0}^{k-1} topk_w[t,j] * y_perm[inv_perm[t*k+j], :]
 *              (fp32, accumulated in j order)
 *   out_f32[t,:] = acc + residual[t,:]   (residual [T,H] f32 or NULL -> 0)
 *   out_bf16[t,:] = bf16(out_f32[t,:])
 * At least one of out_bf16 / out_f32 must be non-NULL; residual may be the
 * same buffer as out_f32 (an in-place residual stream).  A non-finite result
 * sets MOE_DEV_NONFINITE in *dev_status (may be NULL to skip the check).
 * ------------------------------------------------------------------------- */
MOE_API moe_status moe_combine(const float *y_perm, const int32_t *inv_perm, const float *topk_w, int T,
                       int k, int H, const float *residual, uint16_t *out_bf16, float *out_f32,
                       int32_t *dev_status, void *stream);

/* ---------------------------------------------------------------------------
 * moe_combine_weighted -- moe_combine over expert outputs that already carry
 * their route weights (yw_perm [T*k,H] bf16 from
 * moe_expert_swiglu_fused_weighted).  Source as moe_combine.
 *
 *   acc[t,:] = sum_{j=0}^{k-1} float(yw_perm[inv_perm[t*k+j], :])
 *              (fp32, accumulated in j order)
 *   out_f32 / out_bf16 / residual / dev_status as in moe_combine.
 * ------------------------------------------------------------------------- */
MOE_API moe_status moe_combine_weighted(const uint16_t *yw_perm, const int32_t *inv_perm, int T, int k, int H,
                                        const float *residual, uint16_t *out_bf16, float *out_f32,
                                        int32_t *dev_status, void *stream);

/* ---------------------------------------------------------------------------
 * route_block_dedup -- unique experts per (layer, verifier block) and the
 * exact routed bytes each block needs.
 *
 * Source: AFN-019, section "Why overlap alone cannot defeat the byte roofline"
 * (deduplication of repeated routes across a verifier block; ideal payload at
 * two and four bits) and section "Hypothesis H7: DFlash block size must follow
 * I/O cost" (48 * U_B * record bytes per block; break-even U_B < 10 tau(B)).
 *
 *   ids     [L, T_tot, k] int32; block b holds tokens [b*block, (b+1)*block)
 *           (the last block may be shorter); nb = ceil(T_tot / block)
 *   mask    [L, nb, ceil(E/32)] uint32 (out): bit e set iff expert e is routed
 *   U       [L, nb] int32 (out): popcount of the mask
 *   bytes2  [nb] int64 (out): sum_l U[l,b] * 3*H*I * 2 / 8
 *   bytes4  [nb] int64 (out): sum_l U[l,b] * 3*H*I * 4 / 8
 * An ID outside [0,E) sets MOE_DEV_BAD_EXPERT in *dev_status (required);
 * that block's outputs are then not written.
 * ------------------------------------------------------------------------- */
MOE_API moe_status route_block_dedup(const int32_t *ids, int L, int T_tot, int k, int E, int block, int H,
                             int I, uint32_t *mask, int32_t *U, int64_t *bytes2, int64_t *bytes4,
                             int32_t *dev_status, void *stream);

/* ---------------------------------------------------------------------------
 * moe_rmsnorm -- zero-centred RMS normalisation feeding the router and the
 * experts of a residual stack layer  x <- x + MoE(RMSNorm(x)).
 *
 * Source: AFN-001, section "Phase 1: separate math from acceleration"
 * (zero-centred RMS normalisation: the gain is 1 + gamma).
 *
 *   out[t,h] = bf16( x[t,h] / sqrt(mean_h x[t,:]^2 + eps) * (1 + gamma[h]) )
 *   raw_bf16[t,h] = bf16( x[t,h] )  if raw_bf16 != NULL (the representation
 *                   before normalisation, read by a route predictor)
 *   x [T,H] f32, gamma [H] f32 or NULL (-> 0), out / raw_bf16 [T,H] bf16
 * ------------------------------------------------------------------------- */
MOE_API moe_status moe_rmsnorm(const float *x, const float *gamma, float eps, int T, int H, uint16_t *out,
                               uint16_t *raw_bf16, void *stream);

/* ---------------------------------------------------------------------------
 * moe_route_recall -- how many of a token's native experts a predicted route
 * names.
 *
 * Source: AFN-019, section "Hypothesis H2: predict expert routes before
 * attention, not after it" (a pre-attention predictor may move bytes but
 * never chooses experts; zero-training controls: the previous token's
 * same-layer route, the native router on an earlier representation).
 *
 *   hits[t] = | {pred_ids[t,:]} intersect {ref_ids[t,:]} |   (0..k)
 *   pred_ids, ref_ids [T,k] int32, each row k distinct IDs; hits [T] int32.
 *   recall = hits / k; exact top-k set match = (hits == k).
 * ------------------------------------------------------------------------- */
MOE_API moe_status moe_route_recall(const int32_t *pred_ids, const int32_t *ref_ids, int T, int k,
                                    int32_t *hits, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
