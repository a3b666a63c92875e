// Internal declarations of the eviction engine: data layout, workspace
// layout, status bits, PTX helpers and block-level primitives shared by the
// kernels.  Not part of the public C ABI (include/kvevict.h).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>           // CUtensorMap (the type only; encoding goes through the runtime's driver entry point)
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/kvevict.h"

namespace kve {

constexpr int kBlock = 16;          // tokens per paged block (vToken review, Sec. 4.5 default)
constexpr int kMaxSeg = 64;         // split-K segments per lane in the decode kernel
constexpr int kMaxW = 64;           // largest SnapKV obsWindow supported
constexpr int kMaxG = 16;           // largest GQA group
constexpr int kAttendWarps = 4;     // warps per CTA of the decode kernel
constexpr int kStages = 3;          // copy stages per warp of the decode kernel
constexpr int kScratchBufs = 3;     // copies of the decode split-K scratch (layer l uses copy l % 3)

// device status bits (read and cleared by kvevict_last_error)
enum : uint32_t {
  ST_NO_BLOCKS = 1u << 0,     // a mandatory admission found no free block
  ST_BAD_INDEX = 1u << 1,     // an index read from the tables was out of range
  ST_TIMEOUT = 1u << 2,       // a bounded wait gave up
  ST_CAPACITY = 1u << 3,      // a lane's token table is full
  ST_POSITION = 1u << 4,      // the new position is not after the lane's last
};

// per-layer cumulative counters (int64), index into stats[layer][...]
enum : int {
  SC_STEPS = 0, SC_VICTIMS, SC_ADMIT_NEW_BLOCK, SC_FREED_DEAD, SC_FREED_RELOC,
  SC_MOVED, SC_PLANS, SC_DEFERRED, SC_NAN_KEYS, SC_NCOUNTERS
};

struct Dims {
  int policy, L, B, Hq, Hkv, g, d, dtype, P, cap, lanes, W, budget, R, pool_kernel;
  float theta_f;
  int lcap;          // logits row capacity (cap + 1 rounded up to 16)
  int max_window;    // DropKV window queries per head the workspace holds
};

// One layer's slice of the engine state.
struct LayerState {
  void* k_pool; void* v_pool;      // [P][16][d]
  int32_t* pos; int32_t* slot;     // [lanes][cap]
  int32_t* count;                  // [lanes]
  float* score;                    // [lanes][cap]
  float* ring;                     // [lanes][cap][W] or null
  int32_t* ring_slot;              // [lanes]
  int32_t* owner; int32_t* mask;   // [P]
  int32_t* lane_blocks;            // [lanes][cap]
  int32_t* lane_nblocks;           // [lanes]
  long long* stats;                // [SC_NCOUNTERS]
};

// Library scratch, carved out of the caller's workspace.
constexpr int kFreedRanges = 256;   // most CTAs the freed-list kernels use

struct Workspace {
  uint32_t* status;                // 1 word
  int32_t* work_flag;              // 1 word: any lane needs the allocator this call
  // split-K scratch, kScratchBufs copies: layer l uses copy l % kScratchBufs,
  // so the attention of layer l+1 may run beside the epilogues of layers l and
  // l-1.  reads_done[c] counts the epilogue CTAs that have finished with copy
  // c (monotonic, wrapping); an attention writes copy c only once every
  // epilogue launched on it before has finished.
  float* logits_buf[kScratchBufs];       // [lanes][g][lcap] base-2 scaled logits
  float* part_o_buf[kScratchBufs];       // [lanes][kMaxSeg][g][d]
  float* part_ml_buf[kScratchBufs];      // [lanes][kMaxSeg][g][2]  (max, sum), base 2
  int32_t* lane_nseg_buf[kScratchBufs];  // [lanes]
  uint32_t* reads_done;                  // [kScratchBufs]
  unsigned long long* keys64;      // [lanes][cap]  window sums (monotone images), when not in shared memory
  unsigned long long* pooled64;    // [lanes][cap]  pooled keys (monotone images), several victims
  int32_t* need_admit;             // [lanes]
  int32_t* want_dst;               // [lanes]
  int32_t* admit_block;            // [lanes]
  int32_t* dst_begin;              // [lanes]  index into alloc_ids
  int32_t* move_begin;             // [lanes]  index into the moves output
  int32_t* plan_tlive;             // [lanes]  tokens a relocation plan moves
  int32_t* alloc_ids;              // [P]
  int32_t* freed_flag;             // [P]  1 = released during this call
  int32_t* blk_tag;                // [P]  1 = source block of a running plan
  int32_t* counters;               // [16] per-call scalars
  int32_t* freed_part;             // [kFreedRanges] freed blocks per range of the pool (freed list)
  int32_t* epi_done;               // 1 word: epilogue CTAs finished this call
  int32_t* apply_list;             // [lanes]  lanes left with an admission or a relocation to apply
  // DropKV prefill-window scorer
  float* d3_part;                  // [lanes][chunks][rows_cap][d + 2]
  __nv_bfloat16* d3_ahi;           // [lanes][rows][d]
  __nv_bfloat16* d3_alo;           // [lanes][rows][d]
  float* d3_rowc;                  // [lanes][rows][2]  (lse2, |a|^2)
  float* d3_score_part;            // [2][lanes][cap]
  float* d3_vn;                    // [lanes][cap]  |v|^2 of each kept key (scoring pass 1 -> pass 2)
  int32_t* cmp_pos;                // [lanes][cap]  forced compaction: survivors of each CTA's range,
  int32_t* cmp_slot;               //               compacted at the range start
  float* cmp_score;                // [lanes][cap]
  int32_t* cmp_cnt;                // [lanes][cmp_ctas_per_lane + 1]  survivors per CTA, entries before
};

struct Ctx {
  kvevict_config cfg;
  kvevict_buffers buf;
  Dims dims;
  Workspace ws;
  int sm_count;
  int device;
  size_t ws_bytes;
  int attend_ctas_per_sm;
  // One CTA of the lean H2O epilogue fits on an SM beside attend_ctas_per_sm
  // CTAs of the attention kernel (registers, shared memory, threads).
  bool lean_coresident;
  // Launch history for programmatic dependent launch: the most recent launch
  // (kLaunch*, its layer), and per scratch copy the number of decode
  // epilogues launched on it (wrapping), whose CTAs the next attention on
  // that copy waits for (Workspace::reads_done).
  int last_layer;
  int last_kind;
  uint32_t epi_launches[kScratchBufs];
  // TMA tensor maps over each layer's K and V pool ([P * 16 rows][d], bf16,
  // 128-byte swizzle, boxes of one 64-element half row x 1, 16 or 64 rows),
  // kTmapsPerLayer per layer, for the window scoring's row copies; null when
  // the configuration has no scoring window.
  CUtensorMap* tmaps;
  // Per-layer budget and recent window ([L] each, host memory; the
  // configuration's values until kvevict_set_layer_budget changes a layer).
  // Only the decode epilogue reads them, from its launch arguments.
  int* layer_budget;
  int* layer_recent;
  // Relocation deferred to kvevict_relocate (decode steps then plan none).
  bool defer_reloc;
  // The compaction and allocator scratch of kvevict_relocate: a second copy
  // of those workspace fields (the rest alias ws), so a relocation on
  // another stream shares no scratch with decode steps of other layers.
  Workspace ws_reloc;
  int32_t* no_victims;   // [lanes] zeros: kvevict_relocate removes nothing
  // Every CTA of the decode epilogue fits on the device at once (one per
  // lane): the epilogue then also applies its lane's admission and
  // relocation after the layer allocator, and no apply kernel is launched.
  bool epi_applies;
  // The lean H2O epilogue (one small CTA per lane, beside the attention
  // kernel's CTAs) can serve this configuration.
  bool lean_epi;
  // Ring policies: a cluster of four CTAs per lane runs the lane's step (all
  // of them resident at once, one per SM).
  bool ring_cluster;
  // Per layer [L] (host): every lane of the layer holds at most its budget,
  // so a decode step evicts at most one token per lane and the lean
  // epilogue is the right kernel.  A performance hint only: both epilogue
  // kernels handle every case.
  bool* layer_steady;
};

enum : int { kLaunchOther = 0, kLaunchAttend = 1, kLaunchEpilogue = 2, kLaunchApply = 3 };

// Launch-history rules (host).  An attention kernel checks on the device,
// before it writes anything, that every decode epilogue launched earlier on
// its scratch copy has finished (which also covers every earlier epilogue of
// its own layer, which uses the same copy), so it may start early after any
// kernel but a separate apply kernel, which rewrites a layer's tables after
// its epilogue has finished.  The epilogue starts early only right after its
// layer's attention launch.
inline bool attend_early_ok(const Ctx& c) { return c.last_kind != kLaunchApply; }
inline void note_attend(Ctx& c, int layer) {
  c.last_kind = kLaunchAttend;
  c.last_layer = layer;
}
inline void note_epilogue(Ctx& c, int layer) {
  c.epi_launches[layer % kScratchBufs] += 1u;
  c.last_kind = kLaunchEpilogue;
  c.last_layer = layer;
}
inline void note_apply(Ctx& c) { c.last_kind = kLaunchApply; }
// Kernels launched without early start (they never let a successor start
// before they complete).
inline void note_other(Ctx& c) { c.last_kind = kLaunchOther; }

// workspace layout (host)
bool has_ring(const kvevict_config& c);
size_t workspace_layout(const kvevict_config& c, Workspace* ws, char* base, Workspace* ws_reloc = nullptr,
                        int32_t** no_victims = nullptr);
Dims make_dims(const kvevict_config& c);
LayerState layer_state(const Ctx& ctx, int layer);
int d3_chunks(const Dims& dm, int sm_count);
int d3_rows_max(const Dims& dm);
// CTAs per lane of the forced compaction's removal (each takes at most
// kCmpPerCta table entries).
constexpr int kCmpPerCta = 4096;
inline int cmp_ctas_per_lane(const Dims& dm) { return (dm.cap + kCmpPerCta - 1) / kCmpPerCta; }
// tensor maps per layer: {K, V} x {1-row gather box, 16-row box, 64-row box}
constexpr int kTmapsPerLayer = 6;
// Encodes ctx.tmaps (host); cudaSuccess when the configuration needs none.
cudaError_t prepare_tensor_maps(Ctx& ctx);

// kernel launchers (host)
cudaError_t launch_reset(const Ctx&, cudaStream_t);
cudaError_t launch_prefill(const Ctx&, int layer, const void* k, const void* v, int n, cudaStream_t);
cudaError_t launch_decode(Ctx&, int layer, const void* q, const void* k_new, const void* v_new,
                          int new_pos, float* out, float* lse, int32_t* victims, int32_t* n_victims,
                          cudaStream_t);
cudaError_t launch_select(const Ctx&, const void* keys, int key_dtype, const int32_t* positions,
                          const int32_t* counts, int n_lanes, int stride, int budget, int recent,
                          int32_t* victims, int32_t* n_victims, cudaStream_t);
cudaError_t launch_compact(const Ctx&, const Workspace& ws, int layer, const int32_t* victims,
                           const int32_t* n_victims, bool gated, int32_t* freed, int32_t* n_freed,
                           int32_t* moves, int32_t* n_moves, cudaStream_t);
cudaError_t launch_score(const Ctx&, int layer, const void* q_win, int w, const int32_t* q_pos,
                         float* lse, float* a_out, float* scores, cudaStream_t);
cudaError_t launch_score_mass(const Ctx&, int layer, const void* q_win, int w, const int32_t* q_pos,
                              bool later, int pool_r, float* lse, float* scores, cudaStream_t);
cudaError_t launch_stats(const Ctx&, int layer, long long* out, cudaStream_t);
cudaError_t launch_wait_check(const Ctx&, int polls, cudaStream_t);
cudaError_t launch_attend_into(const Ctx&, int layer, const void* q, const void* k_new, const void* v_new,
                               float* logits, float* part_o, float* part_ml, int32_t* lane_nseg, cudaStream_t);
cudaError_t prepare_epilogue();     // one-time attributes of the epilogue kernels
int epilogue_ctas_per_sm();         // co-resident decode-epilogue CTAs per SM (the large kernel)
int lean_epilogue_ctas_per_sm();    // the same for the lean H2O epilogue
int ring_cluster_ctas();             // CTAs of a ring policy's cluster epilogue per lane (0: unavailable)
cudaError_t lean_epilogue_attributes(cudaFuncAttributes*, int* threads);
cudaError_t prepare_select();       // one-time attributes of the selection kernels
cudaError_t prepare_dropkv();       // one-time attributes of the window-scoring kernels
cudaError_t prepare_kernels(Ctx&);   // one-time kernel attributes and occupancy (not stream work)
// early_trigger: the successor in the stream is this layer's decode
// epilogue, which may be scheduled as soon as the attention starts.
cudaError_t launch_attend(const Ctx&, int layer, const void* q, const void* k_new, const void* v_new,
                          cudaStream_t, bool early_trigger);
cudaError_t launch_epilogue(const Ctx&, int layer, bool has_q, int new_pos, const void* k_new,
                            const void* v_new, float* out, float* lse, int32_t* victims,
                            int32_t* n_victims, cudaStream_t, bool* used_apply_kernel = nullptr);
cudaError_t launch_allocate(const Ctx&, const Workspace& ws, int layer, cudaStream_t);
cudaError_t launch_allocate_apply(const Ctx&, int layer, const void* k_new, const void* v_new,
                                  bool mark_freed, int32_t* moves, cudaStream_t, bool with_allocate);

// Kernel launch with programmatic dependent launch allowed (the kernel may
// start before its predecessor in the stream completes; it orders itself
// with griddepcontrol.wait where it consumes the predecessor's results).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void set_status(uint32_t* st, uint32_t bits) { atomicOr(st, bits); }

// 4-byte asynchronous global -> shared copies (completion: cp_async_wait_all)
__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// mbarrier and bulk-copy (TMA, untiled) primitives
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for phase `parity` of the barrier; gives up after a bounded number
// of polls (each try_wait itself suspends for a while), records ST_TIMEOUT
// and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t* status,
                                                  int max_polls = 1 << 22) {
  for (int spins = 0; spins < max_polls; ++spins)
    if (mbar_try_wait(bar, parity)) return true;
  set_status(status, ST_TIMEOUT);
  return false;
}
// global -> shared bulk copy completing on `bar`; dst, src and bytes are
// multiples of 16 bytes
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// atomicAdd with release semantics at device scope: the writes ordered
// before it (this thread's, and the CTA's through a preceding barrier) are
// visible to a reader that observes the result and then acquires.
__device__ __forceinline__ int atomic_add_release(int* p, int v) {
  int old;
  asm volatile("atom.release.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Waits until *p differs from `old` (acquire), with a bounded number of polls
// (about a second); on giving up records ST_TIMEOUT and returns false.
__device__ __forceinline__ bool wait_changed_bounded(const int* p, int old, uint32_t* status) {
  for (int polls = 0; polls < (1 << 20); ++polls) {
    if (ld_acquire_gpu(p) != old) return true;
    __nanosleep(64);
  }
  set_status(status, ST_TIMEOUT);
  return false;
}

// Pulls the 128-byte line holding p into L2 (no registers, no completion).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Monotone unsigned images of float keys: a < b  <=>  mono(a) < mono(b).
// -0.0 maps to +0.0; every NaN maps above +inf (a NaN-scored token is the
// last to be evicted).
__device__ __forceinline__ unsigned long long mono_key(float x) {
  if (x == 0.0f) x = 0.0f;
  uint32_t u = __float_as_uint(x);
  if (x != x) return 0xFFFFFFFFull;
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return u;
}
__device__ __forceinline__ unsigned long long mono_key(double x) {
  if (x == 0.0) x = 0.0;
  unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(x));
  if (x != x) return 0xFFFFFFFFFFFFFFFFull;
  u = (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
  return u;
}

// warp/block reductions and scans
__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Block-wide exclusive scan of one int per thread; returns the exclusive
// prefix and writes the block total.  sh must hold 33 ints.  All threads of
// the block must call it.
__device__ __forceinline__ int block_excl_scan(int v, int* sh, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int inc = warp_incl_scan(v);
  if (lane == 31) sh[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    int x = lane < nw ? sh[lane] : 0;
    int xs = warp_incl_scan(x);
    if (lane < nw) sh[lane] = xs - x;
    if (lane == nw - 1) sh[32] = xs;
  }
  __syncthreads();
  int r = sh[wid] + inc - v;
  *total = sh[32];
  __syncthreads();
  return r;
}

template <typename T>
__device__ __forceinline__ T warp_max(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
template <typename T>
__device__ __forceinline__ T warp_min(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// Bottom-k selection over one lane (one CTA): the k candidates with the
// smallest (key, position), found by an MSB-first radix descent over the
// composite key (monotone key bits, then the position).  The result is a
// threshold such that a candidate is a victim iff its composite, restricted
// to the resolved bits, is below the prefix (or equal to it when inclusive).
// ---------------------------------------------------------------------------
struct SelectResult {
  unsigned long long key_prefix, key_mask;
  uint32_t pos_prefix, pos_mask;
  int inclusive;   // candidates equal to the prefix on the resolved bits are victims
  int k;           // number of victims (0 = none)
};

__device__ __forceinline__ bool select_is_victim(const SelectResult& r, unsigned long long key,
                                                 uint32_t pos) {
  if (r.k <= 0) return false;
  unsigned long long kk = key & r.key_mask;
  if (kk != r.key_prefix) return kk < r.key_prefix;
  uint32_t pp = pos & r.pos_mask;
  if (pp != r.pos_prefix) return pp < r.pos_prefix;
  return r.inclusive != 0;
}

// KeyFn(i) -> unsigned long long monotone key of entry i; PosFn(i) -> uint32
// position; CandFn(i) -> bool.  key_bits = 32 or 64.  sh_hist: 256 ints,
// 8-byte aligned (it also holds 64-bit keys), sh_misc: 40 ints (blockDim <= 1024).  Returns the same SelectResult in
// every thread.  k == 1 (the steady state of a full cache) takes one pass.
template <typename KeyFn, typename PosFn, typename CandFn>
__device__ SelectResult block_bottom_k(int n, int k, int key_bits, KeyFn keyf, PosFn posf,
                                       CandFn candf, int* sh_hist, int* sh_misc) {
  SelectResult r;
  r.key_prefix = 0; r.key_mask = 0; r.pos_prefix = 0; r.pos_mask = 0; r.inclusive = 0; r.k = k;
  if (k <= 0) { r.k = 0; return r; }
  if (k == 1) {
    // a single victim: block-wide minimum of (key, position)
    unsigned long long bk = ~0ull;
    uint32_t bp = 0xFFFFFFFFu;
    int any = 0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      if (!candf(i)) continue;
      const unsigned long long kk = keyf(i);
      const uint32_t pp = posf(i);
      any = 1;
      if (kk < bk || (kk == bk && pp < bp)) { bk = kk; bp = pp; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long ok = __shfl_xor_sync(0xffffffffu, bk, o);
      const uint32_t op = __shfl_xor_sync(0xffffffffu, bp, o);
      any |= __shfl_xor_sync(0xffffffffu, any, o);
      if (ok < bk || (ok == bk && op < bp)) { bk = ok; bp = op; }
    }
    unsigned long long* shk = reinterpret_cast<unsigned long long*>(sh_hist);   // 32 x 8 bytes
    uint32_t* shp = reinterpret_cast<uint32_t*>(sh_hist + 64);
    const int wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if ((threadIdx.x & 31) == 0) { shk[wid] = bk; shp[wid] = bp; sh_misc[wid] = any; }
    __syncthreads();
    bk = ~0ull; bp = 0xFFFFFFFFu; any = 0;
    for (int w = 0; w < nw; ++w) {
      any |= sh_misc[w];
      if (shk[w] < bk || (shk[w] == bk && shp[w] < bp)) { bk = shk[w]; bp = shp[w]; }
    }
    __syncthreads();
    if (!any) { r.k = 0; return r; }
    r.key_prefix = bk; r.key_mask = ~0ull; r.pos_prefix = bp; r.pos_mask = 0xFFFFFFFFu; r.inclusive = 1;
    return r;
  }
  const int total_bits = key_bits + 32;
  int k_rem = k;
  for (int shift = total_bits - 8; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) sh_hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      if (!candf(i)) continue;
      unsigned long long key = keyf(i);
      uint32_t pos = posf(i);
      if ((key & r.key_mask) != r.key_prefix || (pos & r.pos_mask) != r.pos_prefix) continue;
      int digit = shift >= 32 ? (int)((key >> (shift - 32)) & 0xFF) : (int)((pos >> shift) & 0xFF);
      atomicAdd(&sh_hist[digit], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // find the bucket where the cumulative count reaches k_rem
      const int lane = threadIdx.x;
      int c[8];
      int s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) { c[j] = sh_hist[lane * 8 + j]; s += c[j]; }
      int inc = warp_incl_scan(s);
      int exc = inc - s;
      int found = -1, below = 0, cnt = 0;
      if (exc < k_rem && inc >= k_rem) {
        int acc = exc;
        for (int j = 0; j < 8; ++j) {
          if (acc + c[j] >= k_rem) { found = lane * 8 + j; below = acc; cnt = c[j]; break; }
          acc += c[j];
        }
      }
      unsigned ball = __ballot_sync(0xffffffffu, found >= 0);
      int src = ball ? __ffs(ball) - 1 : 0;
      found = __shfl_sync(0xffffffffu, found, src);
      below = __shfl_sync(0xffffffffu, below, src);
      cnt = __shfl_sync(0xffffffffu, cnt, src);
      if (lane == 0) { sh_misc[0] = ball ? found : -1; sh_misc[1] = below; sh_misc[2] = cnt; }
    }
    __syncthreads();
    int b = sh_misc[0], below = sh_misc[1], cnt = sh_misc[2];
    __syncthreads();
    if (b < 0) {   // fewer candidates than k: everything matching the prefix is a victim
      r.inclusive = 1;
      return r;
    }
    if (shift >= 32) {
      r.key_prefix |= (unsigned long long)b << (shift - 32);
      r.key_mask |= 0xFFull << (shift - 32);
    } else {
      r.pos_prefix |= (uint32_t)b << shift;
      r.pos_mask |= 0xFFu << shift;
    }
    k_rem -= below;
    if (cnt == k_rem) { r.inclusive = 1; return r; }
  }
  r.inclusive = 1;   // fully resolved: exactly one entry equals the prefix
  return r;
}

}  // namespace kve

// The opaque handle of the C ABI.
struct kvevict_ctx {
  kve::Ctx c;
};
