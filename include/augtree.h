/*
 * augtree.h - C ABI of exact, differentiable shared-prompt tree attention on one GPU.
 *
 * Method: AugTree, "Splitting Prompt Prefill from Response Replay for
 * Context-Parallel Long-Context LLM Post-Training".
 *   - Sec. 2.1 / 3.1: a replay tree T = (P, {R_i}, i = 1..G): one shared prompt and
 *     G sibling response branches.  A batch holds several trees ("groups").
 *   - Sec. 2.2: attention O = softmax(Q K^T / sqrt(D_h) + M) V, tiled over Q and KV
 *     blocks with an online softmax state.
 *   - Sec. 3.2, Eq. 1: a response token t of branch i sees all prompt keys and the
 *     keys of its own branch up to and including itself; never a sibling's keys.
 *     Prompt tokens see earlier prompt tokens (causal prefill) and no response keys.
 *   - Sec. 3.2, Eq. 2: the prompt K/V gradient is the sum over all G branches,
 *     accumulated and then propagated through the prompt-prefill graph.
 *   - Sec. 3.3: partial online-softmax states merge associatively.
 *   - Sec. 3.4: replay units with work weights, balanced largest-first.
 *
 * Data layout ("THD", row-major, contiguous, all tensors on the current device):
 *   prompt  Q, O, dQ, dO : [total_prompt, Hq,  D]     prompt  K, V, dK, dV : [total_prompt, Hkv, D]
 *   response Q, O, dQ, dO: [total_resp,   Hq,  D]     response K, V, dK, dV: [total_resp,   Hkv, D]
 *   lse (log-sum-exp of the scaled scores, natural log, fp32): [Hq, tokens]
 * Groups are contiguous in the prompt arrays and in the response arrays; the
 * branches of one group are contiguous in the response arrays.  Query head h uses
 * KV head floor(h / (Hq / Hkv)).  Element type: all of Q, K, V, O, dO, dQ, dK, dV
 * have the plan's dtype (fp32 or bf16); lse, the prompt-gradient sums and every
 * workspace are fp32.  Computation is fp32 accumulation in both modes.
 *
 * Ownership: the caller owns every tensor and every workspace.  A plan owns only its
 * device copies of the descriptors and work queues (allocated by augtree_plan_create,
 * freed by augtree_plan_destroy).  The compute calls allocate nothing.
 *
 * Execution: compute calls are asynchronous on the given stream (0 = legacy default
 * stream) of the plan's device.  They validate arguments on the host and return an
 * error code; no exception, abort or device trap is ever raised.  A CUDA launch
 * failure is reported as AUGTREE_ERR_CUDA.  Calls that use one plan must be ordered on
 * the GPU (one stream, or events between streams): the plan's device memory holds its
 * error word and the work counters of the forward kernels, which take their items in
 * queue order through a counter that each launch leaves at zero.
 */
#ifndef AUGTREE_H
#define AUGTREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  AUGTREE_OK = 0,
  AUGTREE_ERR_INVALID_ARG = 1,          /* null pointer, bad offsets, bad sizes            */
  AUGTREE_ERR_UNSUPPORTED = 2,          /* dtype, head_dim not in {64,128}, Hq % Hkv != 0,
                                           tensor cores asked for other than bf16, D=128 */
  AUGTREE_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes below augtree_plan_workspace_bytes    */
  AUGTREE_ERR_CUDA = 4,                 /* a CUDA runtime call or launch failed           */
  AUGTREE_ERR_DEVICE_CHECK = 5,         /* a kernel reported a failed internal check      */
  AUGTREE_ERR_TIMEOUT = 6,              /* a bounded device-side wait gave up             */
  AUGTREE_ERR_CAPACITY = 7              /* an output buffer is too small (schedule export)*/
} augtree_status;

typedef enum { AUGTREE_FP32 = 0, AUGTREE_BF16 = 1 } augtree_dtype;

/* Kernel family: SIMT fp32-FMA kernels (any dtype; the only family for fp32) or the
 * tcgen05 tensor-core kernels (bf16 with head_dim 128 only).  AUTO picks tensor
 * cores for bf16 with head_dim 128, SIMT otherwise. */
typedef enum { AUGTREE_KERNEL_AUTO = 0, AUGTREE_KERNEL_SIMT = 1, AUGTREE_KERNEL_TC = 2 } augtree_kernel;

/* Scheduling of the tensor-core kernels' work units (augtree_config.schedule).
 *   QUEUE       units taken in queue order as SMs free up (the dynamic largest-first
 *               greedy; the default): the forward runs one persistent thread block per
 *               SM that takes units one after the other through a counter in the plan's
 *               device memory and overlaps consecutive units; the backward kernels run
 *               one thread block per unit, dispatched by the hardware in queue order.
 *   PERSISTENT  every tensor-core kernel runs one persistent thread block per lane
 *               (num_sms lanes), each walking a fixed list of units: AssignGrid (Sec.
 *               3.4, Eq. 6; augtree_assign_grid) places the queue's units on lanes,
 *               exactly when a queue has at most AUGTREE_LANES_EXACT_UNITS units, by the
 *               largest-first greedy otherwise (augtree_schedule_lanes exports the
 *               placement).  The SIMT kernels ignore it.  Measured slower than QUEUE on
 *               every configuration; an option, not the default. */
typedef enum { AUGTREE_SCHED_QUEUE = 0, AUGTREE_SCHED_PERSISTENT = 1 } augtree_schedule;
#define AUGTREE_LANES_EXACT_UNITS 12

/* Operations, used to select a work queue or a workspace size. */
typedef enum {
  AUGTREE_OP_PREFILL_FWD = 0,
  AUGTREE_OP_REPLAY_FWD = 1,
  AUGTREE_OP_REPLAY_BWD = 2,
  AUGTREE_OP_PREFILL_BWD = 3,
  AUGTREE_OP_TREE_BWD = 4   /* the whole backward in one call (augtree_tree_bwd) */
} augtree_op;

/* Ragged group / branch descriptors (host memory, read during plan creation only).
 *   prompt_off  [n_groups+1]   prompt token offsets; group g owns prompt rows
 *                              [prompt_off[g], prompt_off[g+1]); prompt_off[0] = 0.
 *   branch_begin[n_groups+1]   group g owns branches [branch_begin[g], branch_begin[g+1]);
 *                              branch_begin[0] = 0, branch_begin[n_groups] = n_branches.
 *   resp_off    [n_branches+1] response token offsets; branch b owns response rows
 *                              [resp_off[b], resp_off[b+1]); resp_off[0] = 0.
 * All three must be non-decreasing.  Empty prompts, empty branches and groups
 * without branches are allowed. */
typedef struct {
  const int32_t* prompt_off;
  const int32_t* branch_begin;
  const int32_t* resp_off;
  int32_t n_groups;
  int32_t n_branches;
} augtree_desc;

typedef struct {
  int32_t hq;            /* query heads                                         */
  int32_t hkv;           /* key/value heads; hq % hkv == 0 (MHA, GQA, MQA)       */
  int32_t head_dim;      /* 64 or 128                                           */
  int32_t dtype;         /* augtree_dtype                                       */
  float softmax_scale;   /* 0 => 1/sqrt(head_dim) (Sec. 2.2)                    */
  int32_t num_sms;       /* balancing width of the work queues; 0 => device SMs */
  int32_t kernel;        /* augtree_kernel                                      */
  int32_t schedule;      /* augtree_schedule (0: one block per unit)             */
} augtree_config;

typedef struct augtree_plan augtree_plan;

/* ---- Work queues ------------------------------------------------------------------
 * Every compute call walks a queue of work items, AUGTREE_ITEM_WORDS int32 each:
 *   [0] kind   [1] group   [2] tile   [3] head   [4] split   [5] cost   [6] a   [7] b
 * Tile sizes: BM query rows per query tile, BN keys per KV tile (augtree_tile_sizes).
 * Let, for group g, L_P its prompt length, p0 its first prompt row, L_R the total
 * length of its branches, r0 their first response row, r = Hq/Hkv.
 *
 *  kind 0 PREFILL_Q (prefill_fwd): query tile `tile` of the prompt, rows
 *    [p0 + tile*BM, min(p0 + (tile+1)*BM, p0 + L_P)), query head `head`.
 *    a = number of prompt KV tiles = ceil((row_end - p0) / BN), b = 0, cost = a.
 *  kind 1 REPLAY_Q (replay_fwd): query tile `tile` of the group's concatenated
 *    branches, rows [r0 + tile*BM, min(r0 + (tile+1)*BM, r0 + L_R)) (a tile may span
 *    branches), query head `head`.  a = ceil(L_P / BN) prompt KV tiles (dense);
 *    b = ceil((row_end - branch_start(first row)) / BN) own KV tiles starting at the
 *    first row's branch start; the tile's KV walk is the a prompt tiles, then the b
 *    own tiles.  Unsplit: split = 0, cost = a + b.  Split-KV (tensor-core kernels,
 *    rule below): the tile has s items per head; item `split` = k walks tiles
 *    [k*C, min((k+1)*C, a + b)) of the walk, C = ceil((a + b) / s), cost = that count.
 *
 * Split-KV rule (replay_fwd with the tensor-core kernels; Sec. 3.3: partial softmax
 * states over disjoint key ranges merge exactly): let n = (number of replay query
 * tiles) * Hq.  If n >= 2 * num_sms nothing is split.  Otherwise a tile of cost c gets
 * s(c, T) = ceil(c / ceil(c / min(64, max(1, ceil(c / T))))) splits for the chunk T
 * chosen among ceil(c_max / k), k = 1..64 (c_max the largest tile cost; T >= 4 for
 * k > 1; the split tiles, s > 1, holding at most 4096 partial states, tiles x Hq x s)
 * with the least ceil(B / num_sms) * (max_tile ceil(c / s) + 2), B = Hq times the sum
 * over tiles of s (one thread block per split and head); the largest T on ties.
 * The replay forward then needs a workspace for the partial states and merges them in
 * split order; the replay query-side backward (same items) writes fp32 dQ partials and
 * sums them in split order.  The SIMT kernels never split.
 *  kind 2 PROMPT_KV (replay_bwd): prompt KV tile `tile` (keys [p0 + tile*BN, ...)),
 *    KV head `head`, split `split`: response query tiles [a, b) of the group, each
 *    for the r query heads of the KV head.  cost = (b - a) * r.
 *  kind 3 RESP_KV (replay_bwd): response KV tile `tile` (keys [r0 + tile*BN, ...)),
 *    KV head `head`: response query tiles [a, b) where a = floor(tile*BN/BM) and b
 *    covers the end of the branch holding the tile's last key.  cost = (b - a) * r.
 *  kind 4 PREFILL_KV (prefill_bwd): prompt KV tile `tile`, KV head `head`: prompt
 *    query tiles [a, b) = [floor(tile*BN/BM), ceil(L_P/BM)).  cost = (b - a) * r.
 *  kind 5 TREE_PROMPT_KV (tree_bwd): prompt KV tile `tile`, KV head `head`, split
 *    `split`: response query tiles [a, b) of the group as in PROMPT_KV and, for split
 *    0 only, also the prompt query tiles [floor(tile*BN/BM), ceil(L_P/BM)) as in
 *    PREFILL_KV.  cost = (b - a + (split == 0 ? ceil(L_P/BM) - floor(tile*BN/BM) : 0)) * r.
 *    The tree_bwd queue holds: for every prompt KV tile and KV head of a group with
 *    L_P > 0, one kind-5 item per split of the replay_bwd split rule below (one item,
 *    a = b = 0, when the group has no response rows); and the RESP_KV items of
 *    replay_bwd.
 *
 * Split rule (replay_bwd, atomic-free split-K of the prompt dK/dV, Eq. 2): let
 * U = sum of the costs of all replay_bwd items before splitting, T = max(r,
 * ceil(U / (2 * num_sms))), nq = ceil(L_R / BM).  A group with L_P > 0 and L_R > 0
 * gets s = min(64, max(1, ceil(nq*r / T))) splits of C = ceil(nq / s) query tiles
 * (then s = ceil(nq / C)); split k covers query tiles [k*C, min((k+1)*C, nq)).
 *
 * Order: items start in queue order.  Every item walks the tiles of one stream: a
 * forward item (kinds 0, 1) the K/V of its group's KV head (head / r); a key-side item
 * the query tiles of its group for its KV head (kinds 2, 4, 5) or of the branch holding
 * the tile's first key (kind 3).  The items of a stream are contiguous; streams come by
 * total cost descending, then (group, KV head, branch) ascending with -1 for a
 * group-wide stream.  Within a stream, replay forward items (kind 1) form sub-streams by
 * the branch of their query tile's first row (whose own-branch keys they read): the
 * items of a sub-stream are contiguous, sub-streams come by total cost descending, then
 * branch ascending; every other item is its stream's only sub-stream.  Within a
 * sub-stream items come by cost descending, then (tile, kind, split, head) ascending -
 * the largest-first greedy balancing of replay units (Sec. 3.4) within each sub-stream.
 * Blocks that run side by side then walk the same tiles, which L2 holds once for all of
 * them.
 */
#define AUGTREE_ITEM_WORDS 8

/* Tile sizes BM (query rows) and BN (keys) the plan's kernels use for an op. */
augtree_status augtree_tile_sizes(const augtree_config* cfg, int32_t op, int32_t* bm, int32_t* bn);

/* Host-only schedule build, no GPU needed: writes the work queue of `op` for the
 * given descriptors and config (cfg->num_sms must be > 0) into out[cap_items *
 * AUGTREE_ITEM_WORDS]; *n_items receives the item count.  Returns
 * AUGTREE_ERR_CAPACITY (with *n_items set) when cap_items is too small. */
augtree_status augtree_schedule_build(const augtree_desc* desc, const augtree_config* cfg,
                                      int32_t op, int32_t* out, size_t cap_items,
                                      size_t* n_items);

/* Host-only, no GPU needed: the persistent schedule's placement of a kernel's work
 * units on lanes (cfg->schedule is ignored; cfg->num_sms lanes, must be > 0).
 * kernel_id selects the kernel: AUGTREE_KID_BWD_QUERY_SIDE (op 0 or 1, the forward queue
 * the query side walks) or AUGTREE_KID_BWD_KEY_SIDE (op 2, 3 or 4); a unit is one queue
 * item.  Unit weights are the items' costs; AssignGrid
 * places U units on L = min(num_sms, U) lanes of ceil(U / L) rounds, exactly when U <=
 * AUGTREE_LANES_EXACT_UNITS, else by its largest-first greedy.  Out (CSR): lane l runs
 * units[lane_off[l] .. lane_off[l+1]) in round order; lane_off needs n_lanes + 1 entries
 * (cap_lanes), units n_units (cap_units).  AUGTREE_ERR_CAPACITY (with *n_lanes, *n_units
 * set) when a buffer is too small. */
augtree_status augtree_schedule_lanes(const augtree_desc* desc, const augtree_config* cfg, int32_t op,
                                      int32_t kernel_id, int32_t* lane_off, size_t cap_lanes, int32_t* units,
                                      size_t cap_units, size_t* n_lanes, size_t* n_units);

/* AssignGrid (Sec. 3.4, Eq. 6), host only, no GPU needed: places n_units replay units
 * with work estimates w[n_units] (>= 0) on a grid of `rounds` x `lanes` cells, at most
 * one unit per cell (a lane runs its rounds one after another), minimising the
 * largest lane total max_j sum_{k on lane j} w[k].  With n_units <= u_max the
 * placement is exact (subset dynamic program over lanes; u_max <= 16, cost about
 * lanes * 3^n_units / 2 steps); otherwise it is the largest-first greedy: units in
 * order of weight descending (index ascending on ties), each to the lane with the
 * smallest total among those with a free round (lowest lane on ties).  u_max = 0
 * always takes the greedy.  Within a lane, rounds follow the same largest-first order.
 * Out: round_out[k] in [0, rounds), lane_out[k] in [0, lanes), *makespan_out = the
 * largest lane total, *exact_out (nullable) = 1 if the dynamic program ran.  Errors:
 * AUGTREE_ERR_INVALID_ARG for null pointers, a negative weight, rounds or lanes < 1,
 * u_max outside [0, 16] or n_units > rounds * lanes. */
augtree_status augtree_assign_grid(const int64_t* w, int32_t n_units, int32_t rounds, int32_t lanes,
                                   int32_t u_max, int32_t* round_out, int32_t* lane_out,
                                   int64_t* makespan_out, int32_t* exact_out);

/* ---- Plans ------------------------------------------------------------------------ */

/* Validates the descriptors and config, builds all four work queues on the host and
 * copies them with the descriptors to the current device (synchronously).
 * *out receives the plan; free it with augtree_plan_destroy. */
augtree_status augtree_plan_create(const augtree_desc* desc, const augtree_config* cfg,
                                   augtree_plan** out);
augtree_status augtree_plan_destroy(augtree_plan* plan);

/* Workspace bytes each compute call needs (0 allowed: pass ws = NULL).  A workspace is
 * device memory owned by the caller, 16-byte aligned (AUGTREE_ERR_INVALID_ARG
 * otherwise), and its contents on entry do not matter.  The prefill
 * forward needs none; the replay forward needs one only when its queue is split-KV
 * (n_parts partial states: 64 KiB of fp32 O plus 512 bytes of lse each, 256-byte
 * aligned); the replay and fused backward add 64 KiB of fp32 dQ per partial state. */
augtree_status augtree_plan_workspace_bytes(const augtree_plan* plan, int32_t op, size_t* bytes);

/* Copy of the plan's work queue for `op` to host memory (for bit-exact checks). */
augtree_status augtree_schedule_export(const augtree_plan* plan, int32_t op, int32_t* host_out,
                                       size_t cap_items, size_t* n_items);

/* ---- Compute (device pointers; stream = cudaStream_t) ----------------------------- */

/* Prompt prefill (Sec. 3.2): causal self-attention of every group's prompt.
 * In: qp [P,Hq,D], kp/vp [P,Hkv,D].  Out: op [P,Hq,D], lse_p [Hq,P]. */
augtree_status augtree_prefill_fwd(const augtree_plan* plan, const void* qp, const void* kp,
                                   const void* vp, void* op, float* lse_p, void* ws,
                                   size_t ws_bytes, void* stream);

/* Response replay (Sec. 3.2-3.3, Eq. 1): each response row attends to all prompt keys
 * of its group (dense) and to its own branch's keys up to itself (causal); the two
 * partial states are merged in one online softmax.  With a split-KV queue (a queue
 * with too few blocks for the GPU, rule above) each split writes its partial state
 * (O / l in fp32, lse) to ws, and a second kernel merges a row's states in split order
 * (the n-way form of augtree_lse_merge) into or_ and lse_r: ws_bytes must then be at
 * least augtree_plan_workspace_bytes(AUGTREE_OP_REPLAY_FWD), else
 * AUGTREE_ERR_WORKSPACE_TOO_SMALL.
 * In: qr [R,Hq,D], kp/vp [P,Hkv,D], kr/vr [R,Hkv,D].  Out: or_ [R,Hq,D], lse_r [Hq,R]. */
augtree_status augtree_replay_fwd(const augtree_plan* plan, const void* qr, const void* kp,
                                  const void* vp, const void* kr, const void* vr, void* or_,
                                  float* lse_r, void* ws, size_t ws_bytes, void* stream);

/* Replay backward.  In: forward inputs, or_, lse_r, dor [R,Hq,D].
 * Out: dqr [R,Hq,D], dkr/dvr [R,Hkv,D] (plan dtype), and the fp32 prompt-gradient sums
 * over all branches dkp_sum/dvp_sum [P,Hkv,D] (Eq. 2; overwritten, not accumulated).
 * Split-K partials of the prompt sums are reduced in a fixed order (no atomics). */
augtree_status augtree_replay_bwd(const augtree_plan* plan, const void* qr, const void* kp,
                                  const void* vp, const void* kr, const void* vr,
                                  const void* or_, const float* lse_r, const void* dor,
                                  void* dqr, void* dkr, void* dvr, float* dkp_sum,
                                  float* dvp_sum, void* ws, size_t ws_bytes, void* stream);

/* Prefill backward: causal backward of the prompt with dop [P,Hq,D], plus the replay
 * sums: dkp = dK_prefill + dkp_acc, dvp = dV_prefill + dvp_acc (dkp_acc / dvp_acc
 * nullable => 0).  Out: dqp [P,Hq,D], dkp/dvp [P,Hkv,D] in the plan dtype. */
augtree_status augtree_prefill_bwd(const augtree_plan* plan, const void* qp, const void* kp,
                                   const void* vp, const void* op, const float* lse_p,
                                   const void* dop, const float* dkp_acc, const float* dvp_acc,
                                   void* dqp, void* dkp, void* dvp, void* ws, size_t ws_bytes,
                                   void* stream);

/* The whole backward in one call (Sec. 3.2, Eq. 2: the prompt K/V gradient is the sum
 * over branches of the replay gradients plus the prompt's own causal gradient).  The
 * results equal augtree_replay_bwd followed by augtree_prefill_bwd with the replay sums
 * (up to fp32 summation order), without the fp32 sums in memory: with the tensor-core
 * kernels each prompt KV tile accumulates the prompt's own causal query tiles and all
 * branches' query tiles in one pass (work queue AUGTREE_OP_TREE_BWD; split-K partials,
 * reduced in a fixed order, only for groups split by the replay_bwd split rule); the
 * SIMT family runs the two calls.
 * In: the prefill inputs qp, kp, vp, op, lse_p, dop and the replay inputs qr, kr, vr,
 * or_, lse_r, dor (layouts as above).  Out: dqp, dkp, dvp, dqr, dkr, dvr (plan dtype).
 * Workspace: augtree_plan_workspace_bytes(AUGTREE_OP_TREE_BWD). */
augtree_status augtree_tree_bwd(const augtree_plan* plan, const void* qp, const void* kp,
                                const void* vp, const void* op, const float* lse_p,
                                const void* dop, const void* qr, const void* kr, const void* vr,
                                const void* or_, const float* lse_r, const void* dor, void* dqp,
                                void* dkp, void* dvp, void* dqr, void* dkr, void* dvr, void* ws,
                                size_t ws_bytes, void* stream);

/* Prefill backward that allocates nothing and takes no workspace.  The paper has no
 * counterpart: this is a convenience for callers that cannot allocate device memory
 * while they run (a caching-allocator or memory-pool callback, where allocating would
 * recurse; a real-time step that must not take the driver's allocation lock or meet an
 * out-of-memory error; a host framework that only lends its own buffers).  Arguments
 * and results are those of augtree_prefill_bwd; the plan must already exist (creating
 * it allocates).
 * Scratch: a 64 MiB array defined by the library.  augtree_plan_create looks up its
 * device address on the plan's device (loading the library module that holds it, which
 * reserves the 64 MiB on that device until the process exits), so this call does no
 * lookup and no allocation.  Per prompt row and query head the array holds 40 bytes
 * with the tensor-core kernels (row statistics and extra-MMA rows) plus 32 MiB of dK/dV
 * flush slots overall, so prompt rows x query heads up to about 838,000; with the SIMT
 * kernels 4 + 4 * head_dim bytes (Delta and the fp32 dQ accumulator), up to about
 * 130,000 at head_dim 128.  A plan whose prefill-backward workspace
 * (augtree_plan_workspace_bytes) exceeds 64 MiB is rejected with
 * AUGTREE_ERR_WORKSPACE_TOO_SMALL before any work is queued; AUGTREE_ERR_CUDA if the
 * lookup at plan creation failed.  Every call shares the array and re-initializes what
 * it reads, so results do not depend on earlier calls, but calls that may overlap on
 * the GPU (unordered streams) race on it. */
augtree_status augtree_prefill_bwd_static(const augtree_plan* plan, const void* qp, const void* kp,
                                          const void* vp, const void* op, const float* lse_p,
                                          const void* dop, const float* dkp_acc,
                                          const float* dvp_acc, void* dqp, void* dkp, void* dvp,
                                          void* stream);

/* State merge (+) of Sec. 3.3 in (O, lse) form, fp32:
 *   lse = log(exp(lse_a) + exp(lse_b)),  o = exp(lse_a - lse) oa + exp(lse_b - lse) ob.
 * oa/ob/o [rows, h, d], lse_a/lse_b/lse [h, rows].  (0, -inf) is the identity; two
 * -inf inputs give o = 0, lse = -inf.  o may alias oa or ob; lse may alias lse_a or
 * lse_b. */
augtree_status augtree_lse_merge(int64_t rows, int32_t h, int32_t d, const float* oa,
                                 const float* lse_a, const float* ob, const float* lse_b,
                                 float* o, float* lse, void* stream);

/* Backward of augtree_lse_merge (same layouts), fp32.  Given the upstream gradient
 * dout [rows, h, d] of the merged o and, optionally, dlse [h, rows] of the merged lse
 * (NULL: zero), writes the gradients with respect to the inputs:
 *   w_a = exp(lse_a - lse), w_b = exp(lse_b - lse)  (lse recomputed from lse_a, lse_b),
 *   doa = w_a dout,  dob = w_b dout,
 *   dlse_a = w_a w_b <dout, oa - ob> + w_a dlse,  dlse_b = w_a w_b <dout, ob - oa> + w_b dlse.
 * An input with lse = -inf has weight 0 and receives zero gradients.  Outputs must not
 * alias inputs.  It makes the merge of Sec. 3.3 usable as a differentiable operator
 * (the pages' MoveQ reduction is a custom autograd operator). */
augtree_status augtree_lse_merge_bwd(int64_t rows, int32_t h, int32_t d, const float* oa,
                                     const float* lse_a, const float* ob, const float* lse_b,
                                     const float* dout, const float* dlse, float* doa, float* dlse_a,
                                     float* dob, float* dlse_b, void* stream);

/* Sets how long a device-side wait of this plan's kernels on another warp's work (a
 * tile landing, a product finishing, a softmax handing over P) may last before the
 * kernel gives up: ns nanoseconds, 2 s by default, 1 ns to 60 s.  A kernel that gives
 * up records AUGTREE_ERR_TIMEOUT for augtree_plan_check, skips the rest of its work
 * item (its outputs are then unspecified), waits for its own bulk copies and MMAs to
 * finish (those waits keep a fixed 2 s limit, since they always end on their own),
 * frees its tensor memory and exits; the device stays usable.  No limit is part of the
 * paper's method: this bounds a wait that a fault elsewhere would make endless.  The
 * value lives in device memory and is written synchronously (cudaMemcpy); it applies to
 * kernels launched after the call.  Errors: AUGTREE_ERR_INVALID_ARG outside the range
 * or on another device's plan. */
augtree_status augtree_plan_set_wait_limit(augtree_plan* plan, uint64_t ns);

/* Synchronizes `stream`, then reads and clears the plan's device error word.  Returns
 * AUGTREE_ERR_TIMEOUT if a kernel launched with this plan gave up on a bounded
 * device-side wait (it then skipped the rest of its work item and exited cleanly),
 * AUGTREE_ERR_DEVICE_CHECK for any other recorded device-side failure, else OK. */
augtree_status augtree_plan_check(const augtree_plan* plan, void* stream);

/* ---- Per-kernel timing (tracing aid; not part of the paper's method) -------------------
 * Off by default.  When enabled, every compute call of the plan records CUDA events on
 * its stream before each kernel it launches and after the last one, in a ring that
 * keeps the last AUGTREE_TIMING_RING calls of each op.  The cost is a few event
 * records per call; nothing else changes.  A call launches at most seven kernels
 * (augtree_tree_bwd with split-K and split-KV); with the SIMT family, augtree_tree_bwd records its two internal
 * calls under AUGTREE_OP_REPLAY_BWD and AUGTREE_OP_PREFILL_BWD.  Kernel kinds
 * (augtree_plan_kernel_times): */
typedef enum {
  AUGTREE_KID_FWD_TC = 1,        /* tensor-core forward (prefill or replay)             */
  AUGTREE_KID_FWD_SIMT = 2,      /* SIMT forward                                        */
  AUGTREE_KID_PREPROCESS = 3,    /* backward preprocess (Delta, row statistics)         */
  AUGTREE_KID_BWD_KEY_SIDE = 4,  /* tensor-core backward, key side (dK, dV)             */
  AUGTREE_KID_SPLIT_REDUCE = 5,  /* fixed-order reduction of prompt dK/dV partials      */
  AUGTREE_KID_BWD_QUERY_SIDE = 6,/* tensor-core backward, query side (dQ)               */
  AUGTREE_KID_DQ_CONVERT = 7,    /* fp32 dQ accumulator to the output dtype (SIMT)      */
  AUGTREE_KID_BWD_SIMT = 8,      /* SIMT backward                                       */
  AUGTREE_KID_FWD_MERGE = 9,     /* merge of the replay forward's split-KV partials     */
  AUGTREE_KID_DQ_REDUCE = 10     /* sum of the replay query side's split-KV dQ partials */
} augtree_kernel_id;
#define AUGTREE_TIMING_RING 64

/* Turns per-kernel timing on (enable != 0) or off.  Turning it on creates the events
 * (on the plan's device); turning it off keeps them until the plan is destroyed. */
augtree_status augtree_plan_set_timing(augtree_plan* plan, int32_t enable);

/* Durations of the kernels of the `back`-th most recent timed call of `op` (back = 0:
 * the last one), in launch order: kind[i] (augtree_kernel_id) and ms[i] for
 * i < *n <= cap.  Waits for that call's events.  AUGTREE_ERR_INVALID_ARG if timing is
 * off, op is not an AUGTREE_OP_*, back >= AUGTREE_TIMING_RING or fewer than back + 1
 * timed calls of op were made. */
augtree_status augtree_plan_kernel_times(const augtree_plan* plan, int32_t op, int32_t back, int32_t* kind,
                                         float* ms, int32_t cap, int32_t* n);

const char* augtree_status_string(augtree_status s);

/* Library version, major*10000 + minor*100 + patch. */
int32_t augtree_version(void);

#ifdef __cplusplus
}
#endif
#endif /* AUGTREE_H */
