/*
 * kvevict -- per-decode-step KV-cache eviction engine for one GB300 GPU.
 *
 * C ABI.  Every pointer argument documented "device" is a CUDA device address
 * owned by the caller; the library never allocates device memory.  Every call
 * that takes a stream is asynchronous on that stream (a cudaStream_t passed
 * as void*; NULL = the legacy default stream): its outputs are valid once the
 * stream has progressed past it.  A call returns KVEVICT_OK after enqueueing
 * its work; argument errors are returned synchronously before anything is
 * enqueued.  Faults found on the device (pool exhausted, a table index out of
 * range, a bounded wait that gave up) set bits in a status word that
 * kvevict_last_error reads and clears.
 *
 * Terms.  A lane is one (sequence b, KV head h) of one layer: lane = b * Hkv + h.
 * Eviction is decided per lane (H2O Guide, "The Dual-Pool Budget
 * Partitioning": a budget per layer and head; FAQ on GQA: the scores of a KV
 * head sum its query heads).  Every lane keeps a token table: its kept
 * tokens in ascending position, each with a physical slot (vToken review,
 * Sec. 3.2), slot = block * 16 + offset (Eq. (2)).  Blocks hold 16 tokens of
 * one lane and come from one pool per layer.
 *
 * Layouts (row-major, C order; L layers, B sequences, Hq query heads, Hkv KV
 * heads, g = Hq / Hkv, d = head_dim, P = blocks_per_pool, C = max_tokens):
 *   k_pool, v_pool  [L][P][16][d]   kv_dtype (bf16 or fp32)
 *   positions       [L][B*Hkv][C]   int32, ascending within a lane
 *   slots           [L][B*Hkv][C]   int32
 *   counts          [L][B*Hkv]      int32, kept tokens per lane
 *   scores          [L][B*Hkv][C]   fp32, H2O cumulative scores
 *   ring            [L][P][16][obs_window] fp32 (SnapKV, and DropKV with
 *                   obs_window >= 1; else NULL): a kept token's history row
 *                   sits at its slot and moves with its K/V rows, so that
 *                   removing a token from a table moves no history
 *   ring_slot       [L][B*Hkv]      int32
 *   block_owner     [L][P]          int32, owning lane or -1 when free
 *   block_mask      [L][P]          int32, bit o set = offset o holds a live token
 *   lane_blocks     [L][B*Hkv][C]   int32, the lane's blocks (unordered)
 *   lane_nblocks    [L][B*Hkv]      int32
 *   stats           [L][KVEVICT_NSTATS] int64 cumulative counters
 *   workspace       kvevict_workspace_size() bytes, 256-byte aligned
 */
#ifndef KVEVICT_H
#define KVEVICT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVEVICT_OK = 0,
  KVEVICT_E_INVALID_ARG = 1,       /* NULL pointer, bad shape, layer out of range */
  KVEVICT_E_POOL_KERNEL_EVEN = 2,  /* SnapKV "Parameters": poolKernel must be odd */
  KVEVICT_E_RECENT_GE_BUDGET = 3,  /* SnapKV "Parameters": recentWindow >= budget is refused */
  KVEVICT_E_OBS_WINDOW_ZERO = 4,   /* SnapKV "Parameters": obsWindow of zero is refused */
  KVEVICT_E_NO_BLOCKS = 5,         /* the pool cannot hold the request */
  KVEVICT_E_DTYPE = 6,             /* unsupported kv or key dtype / head_dim */
  KVEVICT_E_CUDA = 7,              /* a CUDA runtime call failed */
  KVEVICT_E_TIMEOUT = 8,           /* a device-side bounded wait gave up */
  KVEVICT_E_DEVICE = 9,            /* the device status word has fault bits set */
  KVEVICT_E_SCRATCH_LIMIT = 10     /* kvevict_attend_static: the layer needs more scratch
                                      than KVEVICT_STATIC_SCRATCH_BYTES */
} kvevict_status;

typedef enum { KVEVICT_H2O = 0, KVEVICT_SNAPKV = 1, KVEVICT_DROPKV = 2 } kvevict_policy;
typedef enum { KVEVICT_BF16 = 0, KVEVICT_F32 = 1 } kvevict_dtype;
typedef enum { KVEVICT_KEY_F32 = 0, KVEVICT_KEY_F64 = 1 } kvevict_key_dtype;

/* Cumulative per-layer counters written into buffers.stats and returned by
 * kvevict_stats (the last four are computed at the time of the call). */
enum {
  KVEVICT_STAT_STEPS = 0,          /* decode steps run */
  KVEVICT_STAT_VICTIMS = 1,        /* tokens evicted */
  KVEVICT_STAT_ADMIT_NEW_BLOCK = 2,/* admissions that needed a fresh block */
  KVEVICT_STAT_FREED_DEAD = 3,     /* blocks released because every token died */
  KVEVICT_STAT_FREED_RELOC = 4,    /* source blocks released by relocation */
  KVEVICT_STAT_MOVED = 5,          /* tokens relocated */
  KVEVICT_STAT_PLANS = 6,          /* relocation plans run */
  KVEVICT_STAT_DEFERRED = 7,       /* calls whose plans were deferred (pool short) */
  KVEVICT_STAT_NAN_KEYS = 8,       /* NaN eviction keys seen (kept, never evicted first) */
  KVEVICT_STAT_BLOCKS = 9,         /* now: allocated blocks N */
  KVEVICT_STAT_LIVE = 10,          /* now: live tokens (sum of n_b) */
  KVEVICT_STAT_HALF_EMPTY = 11,    /* now: blocks with n_b <= 8 (<= 50% utilisation) */
  KVEVICT_STAT_LANES = 12,         /* now: lanes of the layer */
  KVEVICT_NSTATS = 13
};

/* Engine configuration.  Refusals (kvevict_validate, kvevict_create):
 *   pool_kernel even or < 1          -> KVEVICT_E_POOL_KERNEL_EVEN
 *   recent_window >= budget          -> KVEVICT_E_RECENT_GE_BUDGET
 *   SnapKV with obs_window == 0      -> KVEVICT_E_OBS_WINDOW_ZERO
 *   block_size != 16, recent_window < 1, Hq % Hkv != 0, g > 16,
 *   obs_window > 64, pool_kernel > 31, max_tokens < 2, batch*Hkv > 1024,
 *   max_window < 0, g * max_window > 512 -> KVEVICT_E_INVALID_ARG
 *   head_dim not 64 or 128, kv_dtype not bf16/fp32 -> KVEVICT_E_DTYPE
 * theta_f is the relocation trigger on a lane's waste ratio (vToken review,
 * Sec. 3.3 Stage 2; 0.25 there). */
typedef struct {
  int32_t policy;          /* kvevict_policy */
  int32_t num_layers;
  int32_t batch;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;        /* 64 or 128 */
  int32_t kv_dtype;        /* kvevict_dtype */
  int32_t block_size;      /* must be 16 */
  int32_t blocks_per_pool; /* P: blocks in each layer's pool */
  int32_t max_tokens;      /* C: token-table capacity per lane */
  int32_t budget;          /* tokens kept per lane after each step */
  int32_t recent_window;   /* the newest recent_window positions are never evicted */
  int32_t obs_window;      /* history ring length: SnapKV (>= 1), DropKV decode (0 = no
                              decode steps), ignored for H2O */
  int32_t pool_kernel;     /* SnapKV max-pool width, odd; 1 disables pooling */
  float theta_f;           /* relocation trigger on the lane's waste ratio */
  int32_t max_window;      /* DropKV scoring: largest w passed to kvevict_score
                              (sizes the workspace; 0 if kvevict_score is unused) */
} kvevict_config;

/* Caller-owned device buffers (layouts above). */
typedef struct {
  void* k_pool;
  void* v_pool;
  int32_t* positions;
  int32_t* slots;
  int32_t* counts;
  float* scores;
  float* ring;
  int32_t* ring_slot;
  int32_t* block_owner;
  int32_t* block_mask;
  int32_t* lane_blocks;
  int32_t* lane_nblocks;
  int64_t* stats;
  void* workspace;
} kvevict_buffers;

typedef enum {
  KVEVICT_BUF_K_POOL = 0, KVEVICT_BUF_V_POOL, KVEVICT_BUF_POSITIONS, KVEVICT_BUF_SLOTS,
  KVEVICT_BUF_COUNTS, KVEVICT_BUF_SCORES, KVEVICT_BUF_RING, KVEVICT_BUF_RING_SLOT,
  KVEVICT_BUF_BLOCK_OWNER, KVEVICT_BUF_BLOCK_MASK, KVEVICT_BUF_LANE_BLOCKS,
  KVEVICT_BUF_LANE_NBLOCKS, KVEVICT_BUF_STATS, KVEVICT_BUF_WORKSPACE, KVEVICT_NBUF
} kvevict_buffer_id;

typedef struct kvevict_ctx kvevict_ctx;

/* Host only.  Checks the configuration against the refusals above. */
kvevict_status kvevict_validate(const kvevict_config* cfg);

/* Host only.  Bytes the caller must provide for buffer `which`
 * (kvevict_buffer_id); 0 for an invalid configuration or a buffer the
 * policy does not use (the SnapKV ring outside SnapKV). */
size_t kvevict_buffer_size(const kvevict_config* cfg, int which);

/* Host only.  Bytes of library scratch (== kvevict_buffer_size(cfg,
 * KVEVICT_BUF_WORKSPACE)). */
size_t kvevict_workspace_size(const kvevict_config* cfg);

/* Validates cfg, records the buffer pointers (no copy, no allocation) and
 * queries the current CUDA device.  k_pool and v_pool must be 16-byte aligned
 * and the workspace 256-byte aligned (KVEVICT_E_INVALID_ARG otherwise).  With
 * a scoring window (max_window > 0, bf16, head_dim 128) it also encodes, on
 * the host, TMA tensor maps over every layer's K and V pool for the window
 * scoring's row gathers (KVEVICT_E_CUDA if the driver refuses).  *out is
 * NULL on failure. */
kvevict_status kvevict_create(const kvevict_config* cfg, const kvevict_buffers* bufs,
                              kvevict_ctx** out);
void kvevict_destroy(kvevict_ctx* ctx);

/* Empties every layer: all blocks free, all tables empty, counters zero,
 * status word zero. */
kvevict_status kvevict_reset(kvevict_ctx* ctx, void* stream);

/* Per-layer budget (H2O Guide, "Asymmetric Layer Allocation": early layers
 * want larger recent windows and fewer heavy hitters, deep layers larger
 * heavy-hitter pools).  Sets the budget and recent window that later decode
 * steps of `layer` use (the configuration's values until then); a host-side
 * setting, read when a step is enqueued, so steps already enqueued (or
 * captured in a CUDA graph) keep the values they were launched with.  Pool
 * capacity stays the caller's sizing.  Refuses recent_window >= budget
 * (KVEVICT_E_RECENT_GE_BUDGET, as create does), recent_window < 1 or a
 * layer out of range (KVEVICT_E_INVALID_ARG).  kvevict_reset keeps it. */
kvevict_status kvevict_set_layer_budget(kvevict_ctx* ctx, int layer, int32_t budget,
                                        int32_t recent_window);

/* Prompt admission (vToken review, Sec. 3.2 sync_new_tokens) for one layer:
 * every lane gets positions 0..n-1 with k_ctx/v_ctx [B][Hkv][n][d]
 * (kv_dtype, device), stored in ceil(n/16) blocks taken lowest-id first in
 * ascending lane order, token i at (block i/16, offset i%16); scores and
 * histories start at zero.  The layer's tables must be empty (after
 * kvevict_reset).  KVEVICT_E_NO_BLOCKS (device status) if the pool is short. */
kvevict_status kvevict_prefill(kvevict_ctx* ctx, int layer, const void* k_ctx, const void* v_ctx,
                               int32_t n, void* stream);

/* One decode step of one layer (H2O Guide, "Step-by-Step Eviction
 * Lifecycle"; vToken review, Algorithm 1), for every lane:
 *   attend   the g query heads q[B][Hq][d] (kv_dtype, device) attend the kept
 *            tokens and the new token (k_new/v_new [B][Hkv][d], device) at
 *            position new_pos; out [B][Hq][d] fp32 and lse [B][Hq] fp32
 *            (natural log of the softmax denominator) are written;
 *   score    H2O: score_j += sum over the group of p_hj for every kept j
 *            ("Formulating Cumulative Attention Scores"); SnapKV: the
 *            group's weights go into ring slot ring_slot, which then advances
 *            (SnapKV, "How it works"); DropKV (decode variant, obs_window
 *            >= 1): each kept token's residual-output score of this step,
 *            sum over the group's heads h of p_hj / (1 - p_hj) * ||a_h - v_j||
 *            with a_h the head's output (+inf where 1 - p_hj <= 0; DropKV
 *            explainer, Lemma 1, with the window reduced to the current
 *            query), goes into the ring the same way;
 *   keys     H2O: the scores; SnapKV and DropKV: max over kept neighbours
 *            i-r..i+r (r = (pool_kernel-1)/2, clamped) of the float64 window
 *            sums taken in slot order 0 upward; the new token has key 0;
 *   select   k = max(0, counts+1 - budget) victims among tokens with
 *            position < new_pos - recent_window + 1, smallest (key,
 *            position) first (SnapKV, "Tie-breaking"); written ascending to
 *            victims[lane][0..k) (victims is [B*Hkv][max_tokens] int32,
 *            device) with k in n_victims[lane] (int32, device);
 *   evict    victims leave the token table; a block with no live token left
 *            returns to the pool (vToken review, Sec. 3.2 evict_token);
 *   admit    the new token takes the lowest free slot among its lane's
 *            blocks (H2O Guide, "PagedAttention Memory Integration"), else
 *            a new block (lowest free id, ascending lanes);
 *   reclaim  a lane whose waste ratio F (vToken Eq. (1)) exceeds theta_f
 *            packs the live tokens of its partially filled blocks into
 *            ceil(T_live/16) fresh blocks in ascending position when that
 *            frees strictly more blocks than it takes (Sec. 3.3 Stage 3).
 * q == NULL is inert for the scores and the ring (SnapKV, "How it works":
 * a null attention vector writes nothing and does not advance the ring);
 * out/lse are then not written; admission and eviction still run.
 * new_pos must exceed every kept position of every lane (ST_POSITION).
 * DropKV without a ring (obs_window 0) is refused (KVEVICT_E_INVALID_ARG). */
kvevict_status kvevict_decode_step(kvevict_ctx* ctx, int layer, const void* q, const void* k_new,
                                   const void* v_new, int32_t new_pos, float* out, float* lse,
                                   int32_t* victims, int32_t* n_victims, void* stream);

/* The two halves of kvevict_decode_step, for callers that schedule or time
 * them separately: decode_step(...) == attend(...) then finish_step(...) on
 * the same stream with the same arguments.  kvevict_attend runs the split-K
 * attention kernel only (it writes library scratch, no engine state, so it
 * may be repeated); kvevict_finish_step runs the rest of the step (combine,
 * scores, keys, select, evict, admit, reclaim).  With q == NULL, attend does
 * nothing and finish_step is the inert step described above. */
kvevict_status kvevict_attend(kvevict_ctx* ctx, int layer, const void* q, const void* k_new,
                              const void* v_new, void* stream);
kvevict_status kvevict_finish_step(kvevict_ctx* ctx, int layer, const void* q, const void* k_new,
                                   const void* v_new, int32_t new_pos, float* out, float* lse,
                                   int32_t* victims, int32_t* n_victims, void* stream);

/* DropKV prefill-window scoring of one layer (DropKV explainer: Lemma 1 and
 * the fused scoring paragraph).  q_win [B][Hq][w][d] (kv_dtype, device) are
 * the last w prompt queries at positions q_pos[w] (int32, device); every
 * query row attends the lane's kept tokens at positions <= its own (causal).
 * Writes lse [B][Hq][w] (fp32, natural log), a_out [B][Hq][w][d] (fp32 attention
 * outputs) and scores[lane][j] (fp32, [B*Hkv][max_tokens], kept order) =
 * sum over the group's rows of p/(1-p) * ||a - v_j|| (+inf where 1-p <= 0).
 * q_win and a_out must be 16-byte aligned (KVEVICT_E_INVALID_ARG otherwise).
 * q_win == NULL is inert: nothing is written. */
kvevict_status kvevict_score(kvevict_ctx* ctx, int layer, const void* q_win, int32_t w,
                             const int32_t* q_pos, float* lse, float* a_out, float* scores,
                             void* stream);

/* Prefill-window attention mass of one layer: how much attention the last w
 * prompt queries pay to each kept token, values unused.  q_win [B][Hq][w][d]
 * (kv_dtype, device, 16-byte aligned) at positions q_pos[w] (int32, device);
 * every row attends the lane's kept tokens at positions <= its own (causal
 * softmax, p_ij = exp(s_ij - LSE_i)).  Writes lse [B][Hq][w] (fp32, natural
 * log) and, per lane, scores[lane][j] (fp32, [B*Hkv][max_tokens], kept
 * order):
 *   KVEVICT_MASS_SNAPKV  (SnapKV, "On the adaptation": the paper compresses a
 *       prompt once from the attention its last few queries pay to each key,
 *       then pools and selects; "How it works" for the pooling)
 *       sums_j = sum over the group's rows with key position <= row position
 *       of p_ij, then scores_j = max of sums over kept indices [j-r, j+r]
 *       clamped to the lane, r = (pool_kernel - 1) / 2 from the config
 *       (a NaN sum wins the max);
 *   KVEVICT_MASS_H2O  (H2O Guide, "Formulating Cumulative Attention Scores":
 *       S_j sums the rows t >= j + 1) scores_j = sum over the rows with key
 *       position < row position of p_ij, no pooling.  With every prompt
 *       position in the window this is the causal-prefill S_j; passing the
 *       layer's slice of the score table as `scores` starts H2O decoding from
 *       it.
 * Sums are fp32 in an unspecified order.  Keep budget tokens with
 * kvevict_select on these keys and kvevict_compact.  q_win == NULL is inert:
 * nothing is written.  Needs kv_dtype bf16, head_dim 128 and
 * g * w <= g * max_window (KVEVICT_E_DTYPE / KVEVICT_E_INVALID_ARG). */
typedef enum { KVEVICT_MASS_SNAPKV = 0, KVEVICT_MASS_H2O = 1 } kvevict_mass_kind;
kvevict_status kvevict_score_mass(kvevict_ctx* ctx, int layer, const void* q_win, int32_t w,
                                  const int32_t* q_pos, int32_t kind, float* lse, float* scores,
                                  void* stream);

/* Bottom-k selection on given keys.  keys [n_lanes][stride] (fp32 or fp64,
 * device), positions [n_lanes][stride] ascending (int32, device), counts
 * [n_lanes] (int32, device).  Per lane: newest = positions[counts-1];
 * k = max(0, counts - budget); candidates have position < newest -
 * recent_window + 1; the k smallest (key, position) candidates (-0 = +0;
 * NaN after +inf) are written ascending to victims[lane][0..k) ([n_lanes]
 * [stride]) and k (or the number of candidates, if fewer) to n_victims. */
kvevict_status kvevict_select(kvevict_ctx* ctx, const void* keys, int32_t key_dtype,
                              const int32_t* positions, const int32_t* counts, int32_t n_lanes,
                              int32_t stride, int32_t budget, int32_t recent_window,
                              int32_t* victims, int32_t* n_victims, void* stream);

/* Forced compaction of one layer (vToken review, Sec. 3.3 Stages 1 and 3,
 * invariants I1, I2, I4): evict victims[lane][0..n_victims[lane]) (positions
 * ascending, [B*Hkv][max_tokens] int32, device), release emptied blocks, then
 * for every lane whose plan frees blocks, pack the live tokens of its
 * partially filled blocks into fresh blocks (no theta_f gate).  Outputs
 * (device, may be NULL): freed [P] block ids released by this call,
 * ascending, n_freed [1]; moves [m][6] = (lane, position, src_block,
 * src_offset, dst_block, dst_offset) grouped by ascending lane, ascending
 * position within a lane, n_moves [1].  If the pool cannot supply every
 * destination, all plans of the call are deferred (KVEVICT_STAT_DEFERRED). */
kvevict_status kvevict_compact(kvevict_ctx* ctx, int layer, const int32_t* victims,
                               const int32_t* n_victims, int32_t* freed, int32_t* n_freed,
                               int32_t* moves, int32_t* n_moves, void* stream);

/* Asynchronous reclamation (vToken review, Sec. 3.3 Stage 4: the relocation
 * copy runs on its own stream after the step's forward pass, and the next
 * step's attention waits on an event, not the host).
 * kvevict_defer_relocation(ctx, 1): later decode steps evict and admit as
 * before but plan no relocation (their Eq. (1) test is skipped); 0 restores
 * in-step relocation.  A host-side setting read when a step is enqueued.
 * kvevict_relocate(ctx, layer, ...): the relocation a decode step of `layer`
 * would have run, now: every lane whose waste ratio F (Eq. (1)) exceeds
 * theta_f and whose plan strictly lowers its block count (I4) packs the live
 * tokens of its partly filled blocks into fresh lowest-id blocks (Stages 1
 * and 3), in ascending position; outputs as kvevict_compact (freed [P]
 * ascending, n_freed [1], moves [m][6], n_moves [1]; each may be NULL).  It
 * has its own scratch, so it may run on another stream while decode steps
 * of OTHER layers run; the caller orders it after the layer's last step
 * (record an event on the step's stream, cudaStreamWaitEvent on the
 * relocation stream) and makes that layer's next step wait for it (an event
 * recorded after kvevict_relocate, waited on by the step's stream).  Two
 * kvevict_relocate calls, or one and a kvevict_compact, must not overlap. */
kvevict_status kvevict_defer_relocation(kvevict_ctx* ctx, int32_t deferred);
kvevict_status kvevict_relocate(kvevict_ctx* ctx, int layer, int32_t* freed, int32_t* n_freed,
                                int32_t* moves, int32_t* n_moves, void* stream);

/* Attention output and log-sum-exp of one layer without any scratch from the
 * caller.  The pages have no counterpart to this call; it exists for callers
 * that cannot allocate device memory: code running during CUDA-graph stream
 * capture (cudaMalloc cannot be captured), hosts whose own allocator owns all
 * device memory, and serving loops that ban allocation on the hot path
 * because cudaMalloc synchronises the device.
 * Computes, for every lane, what kvevict_decode_step writes to out
 * [B][Hq][d] (fp32) and lse [B][Hq] (fp32) for the same q [B][Hq][d] and new
 * token k_new/v_new [B][Hkv][d] (kv_dtype, all device pointers), and changes
 * no engine state (no scores, no eviction, no admission).  Its scratch is
 * one array of KVEVICT_STATIC_SCRATCH_BYTES compiled into the library, held
 * on every GPU that loads the library until the process exits; a layer
 * needing more returns KVEVICT_E_SCRATCH_LIMIT before anything is enqueued.
 * It calls no cudaMalloc and no allocating routine.  The first call on a
 * device looks up that array's device address (cudaGetSymbolAddress) with
 * the device current; make that first call before any stream capture.  The
 * address is kept with the CUDA context it belongs to and looked up again
 * when another context is current (after cudaDeviceReset, for example).
 * Every call shares the array and it keeps the last call's contents (no
 * part of it needs to start at zero); calls that overlap on the GPU race. */
#define KVEVICT_STATIC_SCRATCH_BYTES (16u << 20)
kvevict_status kvevict_attend_static(kvevict_ctx* ctx, int layer, const void* q, const void* k_new,
                                     const void* v_new, float* out, float* lse, void* stream);

/* Kernels one kvevict_decode_step with a query launches: 2 (attention, then
 * one epilogue: the small one that runs beside the next layer's attention
 * when it fits on the SMs the attention leaves free, or the larger one that
 * also applies admissions into fresh blocks and relocations when all its
 * one-CTA-per-lane grid fits on the device at once) or 3 (an apply kernel
 * follows); 0 for a NULL context. */
int32_t kvevict_kernels_per_decode_step(const kvevict_ctx* ctx);

/* Writes KVEVICT_NSTATS int64 counters of one layer to out (device). */
kvevict_status kvevict_stats(kvevict_ctx* ctx, int layer, int64_t* out, void* stream);

/* Self-check of the timeout reporting (no counterpart in the pages): one
 * thread waits on a barrier that nothing completes, gives up after `polls`
 * polls (1 .. 2^22; KVEVICT_E_INVALID_ARG otherwise) and sets the timeout
 * bit, exactly as the library's own bounded waits do when a producer never
 * arrives; the next kvevict_last_error then returns KVEVICT_E_TIMEOUT and
 * the context stays usable.  Nothing faults or hangs. */
kvevict_status kvevict_check_wait_timeout(kvevict_ctx* ctx, int32_t polls, void* stream);

/* Synchronises the device, reads and clears the status word.  Returns
 * KVEVICT_OK if no fault bit was set, else KVEVICT_E_DEVICE (or
 * KVEVICT_E_TIMEOUT for a bounded wait) and a description in buf. */
kvevict_status kvevict_last_error(kvevict_ctx* ctx, char* buf, size_t len);

#ifdef __cplusplus
}
#endif
#endif /* KVEVICT_H */
