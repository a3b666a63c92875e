// Host side of the C ABI declared in include/kvevict.h: configuration checks,
// buffer and workspace sizing, the context, and argument validation before
// each call enqueues its kernels.  No device memory is allocated here.
#include <cstdio>
#include <cstring>
#include <new>

#include <nvtx3/nvToolsExt.h>

#include "kvevict_internal.cuh"

namespace {
// An NVTX range around a call's launches, named after the call, for
// profilers and tracers (inert and nearly free when none is attached).
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};
}  // namespace

namespace kve {

namespace {
constexpr size_t kAlign = 256;
inline size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
inline size_t es_of(int dtype) { return dtype == KVEVICT_BF16 ? 2 : 4; }
}  // namespace

// A history ring per kept token: SnapKV always, DropKV (decode variant) when
// obs_window >= 1.
bool has_ring(const kvevict_config& c) {
  return c.policy == KVEVICT_SNAPKV || (c.policy == KVEVICT_DROPKV && c.obs_window >= 1);
}

Dims make_dims(const kvevict_config& c) {
  Dims d;
  d.policy = c.policy;
  d.L = c.num_layers;
  d.B = c.batch;
  d.Hq = c.num_q_heads;
  d.Hkv = c.num_kv_heads;
  d.g = c.num_kv_heads > 0 ? c.num_q_heads / c.num_kv_heads : 0;
  d.d = c.head_dim;
  d.dtype = c.kv_dtype;
  d.P = c.blocks_per_pool;
  d.cap = c.max_tokens;
  d.lanes = c.batch * c.num_kv_heads;
  d.W = has_ring(c) ? c.obs_window : 1;
  d.budget = c.budget;
  d.R = c.recent_window;
  d.pool_kernel = c.pool_kernel;
  d.theta_f = c.theta_f;
  d.lcap = (c.max_tokens + 1 + 15) / 16 * 16;
  d.max_window = c.max_window;
  return d;
}

// Carves the workspace; with base == nullptr only sizes it.
size_t workspace_layout(const kvevict_config& c, Workspace* ws, char* base, Workspace* ws_reloc,
                        int32_t** no_victims) {
  const Dims dm = make_dims(c);
  size_t off = 0;
  auto take = [&](size_t bytes) -> char* {
    char* p = base ? base + off : nullptr;
    off += up(bytes);
    return p;
  };
  const size_t lanes = dm.lanes, cap = dm.cap, P = dm.P, g = dm.g, d = dm.d;
  Workspace w;
  w.status = reinterpret_cast<uint32_t*>(take(4));
  w.work_flag = reinterpret_cast<int32_t*>(take(4));
  for (int c = 0; c < kScratchBufs; ++c) {
    w.logits_buf[c] = reinterpret_cast<float*>(take(lanes * g * dm.lcap * 4));
    w.part_o_buf[c] = reinterpret_cast<float*>(take(lanes * kMaxSeg * g * d * 4));
    w.part_ml_buf[c] = reinterpret_cast<float*>(take(lanes * kMaxSeg * g * 2 * 4));
    w.lane_nseg_buf[c] = reinterpret_cast<int32_t*>(take(lanes * 4));
  }
  const bool snap = has_ring(c);
  w.keys64 = snap ? reinterpret_cast<unsigned long long*>(take(lanes * cap * 8)) : nullptr;
  w.pooled64 = snap ? reinterpret_cast<unsigned long long*>(take(lanes * cap * 8)) : nullptr;
  w.need_admit = reinterpret_cast<int32_t*>(take(lanes * 4));
  w.want_dst = reinterpret_cast<int32_t*>(take(lanes * 4));
  w.admit_block = reinterpret_cast<int32_t*>(take(lanes * 4));
  w.dst_begin = reinterpret_cast<int32_t*>(take(lanes * 4));
  w.move_begin = reinterpret_cast<int32_t*>(take(lanes * 4));
  w.plan_tlive = reinterpret_cast<int32_t*>(take(lanes * 4));
  w.alloc_ids = reinterpret_cast<int32_t*>(take(P * 4));
  w.freed_flag = reinterpret_cast<int32_t*>(take(P * 4));
  w.blk_tag = reinterpret_cast<int32_t*>(take(P * 4));
  w.counters = reinterpret_cast<int32_t*>(take(64));
  w.freed_part = reinterpret_cast<int32_t*>(take(kFreedRanges * 4));
  w.cmp_pos = reinterpret_cast<int32_t*>(take(lanes * cap * 4));
  w.cmp_slot = reinterpret_cast<int32_t*>(take(lanes * cap * 4));
  w.cmp_score = reinterpret_cast<float*>(take(lanes * cap * 4));
  w.cmp_cnt = reinterpret_cast<int32_t*>(take(lanes * static_cast<size_t>(cmp_ctas_per_lane(dm) + 1) * 4));
  w.epi_done = reinterpret_cast<int32_t*>(take(4));
  w.reads_done = reinterpret_cast<uint32_t*>(take(kScratchBufs * 4));
  w.apply_list = reinterpret_cast<int32_t*>(take(lanes * 4));
  if (dm.max_window > 0 && dm.dtype == KVEVICT_BF16 && dm.d == 128) {
    const size_t rows = static_cast<size_t>(d3_rows_max(dm));
    const size_t chunks = static_cast<size_t>(d3_chunks(dm, 0));
    w.d3_part = reinterpret_cast<float*>(take(lanes * chunks * rows * (d + 2) * 4));
    w.d3_ahi = reinterpret_cast<__nv_bfloat16*>(take(lanes * rows * d * 2));
    w.d3_alo = reinterpret_cast<__nv_bfloat16*>(take(lanes * rows * d * 2));
    w.d3_rowc = reinterpret_cast<float*>(take(lanes * rows * 2 * 4));
    w.d3_score_part = reinterpret_cast<float*>(take(4 * lanes * cap * 4));
    w.d3_vn = reinterpret_cast<float*>(take(lanes * cap * 4));
  } else {
    w.d3_part = nullptr; w.d3_ahi = nullptr; w.d3_alo = nullptr; w.d3_rowc = nullptr; w.d3_score_part = nullptr;
    w.d3_vn = nullptr;
  }
  // kvevict_relocate's own compaction and allocator scratch
  Workspace r = w;
  r.work_flag = reinterpret_cast<int32_t*>(take(4));
  r.need_admit = reinterpret_cast<int32_t*>(take(lanes * 4));
  r.want_dst = reinterpret_cast<int32_t*>(take(lanes * 4));
  r.admit_block = reinterpret_cast<int32_t*>(take(lanes * 4));
  r.dst_begin = reinterpret_cast<int32_t*>(take(lanes * 4));
  r.move_begin = reinterpret_cast<int32_t*>(take(lanes * 4));
  r.plan_tlive = reinterpret_cast<int32_t*>(take(lanes * 4));
  r.alloc_ids = reinterpret_cast<int32_t*>(take(P * 4));
  r.freed_flag = reinterpret_cast<int32_t*>(take(P * 4));
  r.blk_tag = reinterpret_cast<int32_t*>(take(P * 4));
  r.counters = reinterpret_cast<int32_t*>(take(64));
  r.freed_part = reinterpret_cast<int32_t*>(take(kFreedRanges * 4));
  r.cmp_pos = reinterpret_cast<int32_t*>(take(lanes * cap * 4));
  r.cmp_slot = reinterpret_cast<int32_t*>(take(lanes * cap * 4));
  r.cmp_score = reinterpret_cast<float*>(take(lanes * cap * 4));
  r.cmp_cnt = reinterpret_cast<int32_t*>(take(lanes * static_cast<size_t>(cmp_ctas_per_lane(dm) + 1) * 4));
  r.epi_done = reinterpret_cast<int32_t*>(take(4));
  r.apply_list = reinterpret_cast<int32_t*>(take(lanes * 4));
  int32_t* nv = reinterpret_cast<int32_t*>(take(lanes * 4));
  if (ws) *ws = w;
  if (ws_reloc) *ws_reloc = r;
  if (no_victims) *no_victims = nv;
  return off;
}

LayerState layer_state(const Ctx& ctx, int layer) {
  const Dims& dm = ctx.dims;
  const kvevict_buffers& b = ctx.buf;
  const size_t L = static_cast<size_t>(layer);
  const size_t lanes = dm.lanes, cap = dm.cap, P = dm.P;
  LayerState s;
  const size_t pool = P * kBlock * dm.d * es_of(dm.dtype);
  s.k_pool = static_cast<char*>(b.k_pool) + L * pool;
  s.v_pool = static_cast<char*>(b.v_pool) + L * pool;
  s.pos = b.positions + L * lanes * cap;
  s.slot = b.slots + L * lanes * cap;
  s.count = b.counts + L * lanes;
  s.score = b.scores + L * lanes * cap;
  s.ring = (has_ring(ctx.cfg) && b.ring) ? b.ring + L * P * kBlock * dm.W : nullptr;
  s.ring_slot = b.ring_slot + L * lanes;
  s.owner = b.block_owner + L * P;
  s.mask = b.block_mask + L * P;
  s.lane_blocks = b.lane_blocks + L * lanes * cap;
  s.lane_nblocks = b.lane_nblocks + L * lanes;
  s.stats = reinterpret_cast<long long*>(b.stats) + L * KVEVICT_NSTATS;
  return s;
}

cudaError_t launch_reset(const Ctx& ctx, cudaStream_t st) {
  const kvevict_config& c = ctx.cfg;
  const kvevict_buffers& b = ctx.buf;
  auto sz = [&](int which) { return kvevict_buffer_size(&c, which); };
  cudaError_t e = cudaSuccess;
  auto ms = [&](void* p, int v, size_t n) {
    if (e == cudaSuccess && p && n) e = cudaMemsetAsync(p, v, n, st);
  };
  ms(b.positions, 0, sz(KVEVICT_BUF_POSITIONS));
  ms(b.slots, 0xFF, sz(KVEVICT_BUF_SLOTS));
  ms(b.counts, 0, sz(KVEVICT_BUF_COUNTS));
  ms(b.scores, 0, sz(KVEVICT_BUF_SCORES));
  if (has_ring(c)) ms(b.ring, 0, sz(KVEVICT_BUF_RING));
  ms(b.ring_slot, 0, sz(KVEVICT_BUF_RING_SLOT));
  ms(b.block_owner, 0xFF, sz(KVEVICT_BUF_BLOCK_OWNER));
  ms(b.block_mask, 0, sz(KVEVICT_BUF_BLOCK_MASK));
  ms(b.lane_blocks, 0xFF, sz(KVEVICT_BUF_LANE_BLOCKS));
  ms(b.lane_nblocks, 0, sz(KVEVICT_BUF_LANE_NBLOCKS));
  ms(b.stats, 0, sz(KVEVICT_BUF_STATS));
  const Workspace& w = ctx.ws;
  const size_t lanes = ctx.dims.lanes, P = ctx.dims.P;
  ms(w.status, 0, 4);
  ms(w.work_flag, 0, 4);
  ms(w.need_admit, 0, lanes * 4);
  ms(w.want_dst, 0, lanes * 4);
  ms(w.plan_tlive, 0, lanes * 4);
  ms(w.freed_flag, 0, P * 4);
  ms(w.blk_tag, 0, P * 4);
  ms(w.counters, 0, 64);
  ms(w.epi_done, 0, 4);
  ms(w.reads_done, 0, kScratchBufs * 4);
  const Workspace& r = ctx.ws_reloc;
  ms(r.work_flag, 0, 4);
  ms(r.need_admit, 0, lanes * 4);
  ms(r.want_dst, 0, lanes * 4);
  ms(r.plan_tlive, 0, lanes * 4);
  ms(r.freed_flag, 0, P * 4);
  ms(r.blk_tag, 0, P * 4);
  ms(r.counters, 0, 64);
  ms(r.epi_done, 0, 4);
  ms(ctx.no_victims, 0, lanes * 4);
  return e;
}

}  // namespace kve

using kve::Ctx;

extern "C" {

kvevict_status kvevict_validate(const kvevict_config* c) {
  if (!c) return KVEVICT_E_INVALID_ARG;
  if (c->pool_kernel < 1 || c->pool_kernel % 2 == 0) return KVEVICT_E_POOL_KERNEL_EVEN;
  if (c->recent_window >= c->budget) return KVEVICT_E_RECENT_GE_BUDGET;
  if (c->policy == KVEVICT_SNAPKV && c->obs_window == 0) return KVEVICT_E_OBS_WINDOW_ZERO;
  if (c->policy < 0 || c->policy > 2) return KVEVICT_E_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return KVEVICT_E_DTYPE;
  if (c->kv_dtype != KVEVICT_BF16 && c->kv_dtype != KVEVICT_F32) return KVEVICT_E_DTYPE;
  if (c->block_size != 16 || c->recent_window < 1 || c->num_layers < 1 || c->batch < 1 ||
      c->num_kv_heads < 1 || c->num_q_heads < 1 || c->num_q_heads % c->num_kv_heads != 0 ||
      c->num_q_heads / c->num_kv_heads > kve::kMaxG || c->blocks_per_pool < 1 || c->max_tokens < 2 ||
      c->batch * c->num_kv_heads > 1024 || c->pool_kernel > 31 || c->max_window < 0 ||
      (c->num_q_heads / c->num_kv_heads) * c->max_window > 512 || !(c->theta_f >= 0.0f))
    return KVEVICT_E_INVALID_ARG;
  if (c->policy == KVEVICT_SNAPKV && (c->obs_window < 1 || c->obs_window > kve::kMaxW ))
    return KVEVICT_E_INVALID_ARG;
  if (c->policy == KVEVICT_DROPKV && (c->obs_window < 0 || c->obs_window > kve::kMaxW))
    return KVEVICT_E_INVALID_ARG;
  // 16-token blocks are addressed with int32 slots
  if (static_cast<long long>(c->blocks_per_pool) * 16 >= (1ll << 31)) return KVEVICT_E_INVALID_ARG;
  return KVEVICT_OK;
}

size_t kvevict_buffer_size(const kvevict_config* c, int which) {
  if (kvevict_validate(c) != KVEVICT_OK) return 0;
  const size_t L = c->num_layers, lanes = static_cast<size_t>(c->batch) * c->num_kv_heads;
  const size_t cap = c->max_tokens, P = c->blocks_per_pool, d = c->head_dim;
  const size_t es = c->kv_dtype == KVEVICT_BF16 ? 2 : 4;
  switch (which) {
    case KVEVICT_BUF_K_POOL:
    case KVEVICT_BUF_V_POOL: return L * P * 16 * d * es;
    case KVEVICT_BUF_POSITIONS:
    case KVEVICT_BUF_SLOTS:
    case KVEVICT_BUF_SCORES:
    case KVEVICT_BUF_LANE_BLOCKS: return L * lanes * cap * 4;
    case KVEVICT_BUF_COUNTS:
    case KVEVICT_BUF_RING_SLOT:
    case KVEVICT_BUF_LANE_NBLOCKS: return L * lanes * 4;
    case KVEVICT_BUF_RING:
      return kve::has_ring(*c) ? L * P * kve::kBlock * static_cast<size_t>(c->obs_window) * 4 : 0;
    case KVEVICT_BUF_BLOCK_OWNER:
    case KVEVICT_BUF_BLOCK_MASK: return L * P * 4;
    case KVEVICT_BUF_STATS: return L * KVEVICT_NSTATS * 8;
    case KVEVICT_BUF_WORKSPACE: return kve::workspace_layout(*c, nullptr, nullptr);
    default: return 0;
  }
}

size_t kvevict_workspace_size(const kvevict_config* c) {
  return kvevict_buffer_size(c, KVEVICT_BUF_WORKSPACE);
}

kvevict_status kvevict_create(const kvevict_config* cfg, const kvevict_buffers* bufs, kvevict_ctx** out) {
  if (!out) return KVEVICT_E_INVALID_ARG;
  *out = nullptr;
  const kvevict_status v = kvevict_validate(cfg);
  if (v != KVEVICT_OK) return v;
  if (!bufs || !bufs->k_pool || !bufs->v_pool || !bufs->positions || !bufs->slots || !bufs->counts ||
      !bufs->scores || !bufs->ring_slot || !bufs->block_owner || !bufs->block_mask || !bufs->lane_blocks ||
      !bufs->lane_nblocks || !bufs->stats || !bufs->workspace ||
      (kve::has_ring(*cfg) && !bufs->ring))
    return KVEVICT_E_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(bufs->workspace) % 256 != 0 || reinterpret_cast<uintptr_t>(bufs->k_pool) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(bufs->v_pool) % 16 != 0)
    return KVEVICT_E_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVEVICT_E_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KVEVICT_E_CUDA;
  kvevict_ctx* ctx = new (std::nothrow) kvevict_ctx;
  if (!ctx) return KVEVICT_E_INVALID_ARG;
  ctx->c.cfg = *cfg;
  ctx->c.buf = *bufs;
  ctx->c.dims = kve::make_dims(*cfg);
  ctx->c.sm_count = sms;
  ctx->c.device = dev;
  ctx->c.last_layer = -1;
  ctx->c.last_kind = kve::kLaunchOther;
  for (int c = 0; c < kve::kScratchBufs; ++c) ctx->c.epi_launches[c] = 0u;
  ctx->c.tmaps = nullptr;
  ctx->c.layer_budget = new (std::nothrow) int[cfg->num_layers];
  ctx->c.layer_recent = new (std::nothrow) int[cfg->num_layers];
  ctx->c.layer_steady = new (std::nothrow) bool[cfg->num_layers];
  if (!ctx->c.layer_budget || !ctx->c.layer_recent || !ctx->c.layer_steady) {
    delete[] ctx->c.layer_budget;
    delete[] ctx->c.layer_recent;
    delete[] ctx->c.layer_steady;
    delete ctx;
    return KVEVICT_E_INVALID_ARG;
  }
  for (int l = 0; l < cfg->num_layers; ++l) {
    ctx->c.layer_budget[l] = cfg->budget;
    ctx->c.layer_recent[l] = cfg->recent_window;
    // unknown contents (the buffers may hold a saved state): the large
    // epilogue until a decode step or a reset says otherwise
    ctx->c.layer_steady[l] = false;
  }
  ctx->c.defer_reloc = false;
  ctx->c.ws_bytes = kve::workspace_layout(*cfg, &ctx->c.ws, static_cast<char*>(bufs->workspace), &ctx->c.ws_reloc,
                                          &ctx->c.no_victims);
  const bool ok = kve::prepare_kernels(ctx->c) == cudaSuccess && ctx->c.attend_ctas_per_sm >= 1 &&
                  kve::prepare_select() == cudaSuccess && kve::prepare_tensor_maps(ctx->c) == cudaSuccess;
  // the epilogue applies admissions and relocations itself when all its
  // CTAs (one per lane) are resident at once
  ctx->c.epi_applies = ok && static_cast<long long>(kve::epilogue_ctas_per_sm()) * sms >= ctx->c.dims.lanes;
  // the lean H2O epilogue: bf16 pools, groups of at most 8 heads, at most one
  // lane per SM (one lean CTA fits beside the attention kernel's CTAs)
  ctx->c.lean_epi = ok && cfg->policy == KVEVICT_H2O && cfg->kv_dtype == KVEVICT_BF16 && ctx->c.dims.g <= 8 &&
                    ctx->c.dims.lanes <= sms && ctx->c.lean_coresident && kve::lean_epilogue_ctas_per_sm() >= 1;
  // ring policies: the cluster epilogue when every lane's cluster is resident at once
  const int rcc = ok && cfg->policy != KVEVICT_H2O ? kve::ring_cluster_ctas() : 0;
  ctx->c.ring_cluster = rcc > 0 && static_cast<long long>(ctx->c.dims.lanes) * rcc <= sms;
  if (!ok) {
    delete[] ctx->c.tmaps;
    delete[] ctx->c.layer_budget;
    delete[] ctx->c.layer_recent;
    delete[] ctx->c.layer_steady;
    delete ctx;
    return KVEVICT_E_CUDA;
  }
  *out = ctx;
  return KVEVICT_OK;
}

void kvevict_destroy(kvevict_ctx* ctx) {
  if (!ctx) return;
  delete[] ctx->c.tmaps;
  delete[] ctx->c.layer_budget;
  delete[] ctx->c.layer_recent;
  delete[] ctx->c.layer_steady;
  delete ctx;
}

static kvevict_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVEVICT_OK : KVEVICT_E_CUDA; }

kvevict_status kvevict_set_layer_budget(kvevict_ctx* ctx, int layer, int32_t budget, int32_t recent_window) {
  if (!ctx || layer < 0 || layer >= ctx->c.dims.L || recent_window < 1) return KVEVICT_E_INVALID_ARG;
  if (recent_window >= budget) return KVEVICT_E_RECENT_GE_BUDGET;
  // a smaller budget: the next step may evict more than one token per lane
  if (budget < ctx->c.layer_budget[layer]) ctx->c.layer_steady[layer] = false;
  ctx->c.layer_budget[layer] = budget;
  ctx->c.layer_recent[layer] = recent_window;
  return KVEVICT_OK;
}

kvevict_status kvevict_defer_relocation(kvevict_ctx* ctx, int32_t deferred) {
  if (!ctx) return KVEVICT_E_INVALID_ARG;
  ctx->c.defer_reloc = deferred != 0;
  return KVEVICT_OK;
}

kvevict_status kvevict_relocate(kvevict_ctx* ctx, int layer, int32_t* freed, int32_t* n_freed, int32_t* moves,
                                int32_t* n_moves, void* stream) {
  const CallRange range("kvevict_relocate");
  if (!ctx || layer < 0 || layer >= ctx->c.dims.L) return KVEVICT_E_INVALID_ARG;
  kve::note_other(ctx->c);
  return cuda_status(kve::launch_compact(ctx->c, ctx->c.ws_reloc, layer, ctx->c.no_victims, ctx->c.no_victims, true,
                                         freed, n_freed, moves, n_moves, static_cast<cudaStream_t>(stream)));
}

kvevict_status kvevict_reset(kvevict_ctx* ctx, void* stream) {
  if (!ctx) return KVEVICT_E_INVALID_ARG;
  kve::note_other(ctx->c);
  for (int l = 0; l < ctx->c.dims.L; ++l) ctx->c.layer_steady[l] = true;   // every lane empty
  // the reset zeroes the epilogue counts of the scratch copies
  for (int c = 0; c < kve::kScratchBufs; ++c) ctx->c.epi_launches[c] = 0u;
  return cuda_status(kve::launch_reset(ctx->c, static_cast<cudaStream_t>(stream)));
}

kvevict_status kvevict_prefill(kvevict_ctx* ctx, int layer, const void* k_ctx, const void* v_ctx, int32_t n,
                               void* stream) {
  const CallRange range("kvevict_prefill");
  if (!ctx || !k_ctx || !v_ctx || layer < 0 || layer >= ctx->c.dims.L || n < 1 || n > ctx->c.dims.cap - 1)
    return KVEVICT_E_INVALID_ARG;
  kve::note_other(ctx->c);
  ctx->c.layer_steady[layer] = ctx->c.layer_steady[layer] && n <= ctx->c.layer_budget[layer];
  return cuda_status(kve::launch_prefill(ctx->c, layer, k_ctx, v_ctx, n, static_cast<cudaStream_t>(stream)));
}

kvevict_status kvevict_decode_step(kvevict_ctx* ctx, int layer, const void* q, const void* k_new, const void* v_new,
                                   int32_t new_pos, float* out, float* lse, int32_t* victims, int32_t* n_victims,
                                   void* stream) {
  const CallRange range("kvevict_decode_step");
  if (!ctx || layer < 0 || layer >= ctx->c.dims.L || !k_new || !v_new || !victims || !n_victims || new_pos < 0)
    return KVEVICT_E_INVALID_ARG;
  if (q && (!out || !lse)) return KVEVICT_E_INVALID_ARG;
  if (ctx->c.dims.policy == KVEVICT_DROPKV && !kve::has_ring(ctx->c.cfg)) return KVEVICT_E_INVALID_ARG;
  const cudaError_t e = kve::launch_decode(ctx->c, layer, q, k_new, v_new, new_pos, out, lse, victims, n_victims,
                                           static_cast<cudaStream_t>(stream));
  return cuda_status(e);
}

kvevict_status kvevict_attend(kvevict_ctx* ctx, int layer, const void* q, const void* k_new, const void* v_new,
                              void* stream) {
  const CallRange range("kvevict_attend");
  if (!ctx || layer < 0 || layer >= ctx->c.dims.L || !k_new || !v_new) return KVEVICT_E_INVALID_ARG;
  if (ctx->c.dims.policy == KVEVICT_DROPKV && !kve::has_ring(ctx->c.cfg)) return KVEVICT_E_INVALID_ARG;
  if (!q) return KVEVICT_OK;
  const cudaError_t e = kve::launch_attend(ctx->c, layer, q, k_new, v_new, static_cast<cudaStream_t>(stream), false);
  if (e == cudaSuccess) kve::note_attend(ctx->c, layer);
  return cuda_status(e);
}

kvevict_status kvevict_finish_step(kvevict_ctx* ctx, int layer, const void* q, const void* k_new, const void* v_new,
                                   int32_t new_pos, float* out, float* lse, int32_t* victims, int32_t* n_victims,
                                   void* stream) {
  const CallRange range("kvevict_finish_step");
  if (!ctx || layer < 0 || layer >= ctx->c.dims.L || !k_new || !v_new || !victims || !n_victims || new_pos < 0)
    return KVEVICT_E_INVALID_ARG;
  if (q && (!out || !lse)) return KVEVICT_E_INVALID_ARG;
  if (ctx->c.dims.policy == KVEVICT_DROPKV && !kve::has_ring(ctx->c.cfg)) return KVEVICT_E_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  bool apply_kernel = false;
  cudaError_t e = kve::launch_epilogue(ctx->c, layer, q != nullptr, new_pos, k_new, v_new, out, lse, victims,
                                       n_victims, st, &apply_kernel);
  if (e == cudaSuccess) {
    kve::note_epilogue(ctx->c, layer);
    ctx->c.layer_steady[layer] = true;
  }
  if (e == cudaSuccess && apply_kernel) {
    e = kve::launch_allocate_apply(ctx->c, layer, k_new, v_new, false, nullptr, st, false);
    kve::note_apply(ctx->c);
  }
  return cuda_status(e);
}

kvevict_status kvevict_score(kvevict_ctx* ctx, int layer, const void* q_win, int32_t w, const int32_t* q_pos,
                             float* lse, float* a_out, float* scores, void* stream) {
  const CallRange range("kvevict_score");
  if (!ctx || layer < 0 || layer >= ctx->c.dims.L) return KVEVICT_E_INVALID_ARG;
  if (!q_win) return KVEVICT_OK;   // null attention is inert
  if (w < 1 || w > ctx->c.dims.max_window || !q_pos || !lse || !a_out || !scores) return KVEVICT_E_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(q_win) % 16 || reinterpret_cast<uintptr_t>(a_out) % 16)
    return KVEVICT_E_INVALID_ARG;   // 16-byte row copies and stores
  if (ctx->c.dims.dtype != KVEVICT_BF16 || ctx->c.dims.d != 128) return KVEVICT_E_DTYPE;
  kve::note_other(ctx->c);
  return cuda_status(kve::launch_score(ctx->c, layer, q_win, w, q_pos, lse, a_out, scores,
                                       static_cast<cudaStream_t>(stream)));
}

kvevict_status kvevict_score_mass(kvevict_ctx* ctx, int layer, const void* q_win, int32_t w, const int32_t* q_pos,
                                  int32_t kind, float* lse, float* scores, void* stream) {
  const CallRange range("kvevict_score_mass");
  if (!ctx || layer < 0 || layer >= ctx->c.dims.L) return KVEVICT_E_INVALID_ARG;
  if (kind != KVEVICT_MASS_SNAPKV && kind != KVEVICT_MASS_H2O) return KVEVICT_E_INVALID_ARG;
  if (!q_win) return KVEVICT_OK;   // null attention is inert
  if (w < 1 || w > ctx->c.dims.max_window || !q_pos || !lse || !scores) return KVEVICT_E_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(q_win) % 16) return KVEVICT_E_INVALID_ARG;   // 16-byte row copies
  if (ctx->c.dims.dtype != KVEVICT_BF16 || ctx->c.dims.d != 128) return KVEVICT_E_DTYPE;
  const int pk = ctx->c.cfg.pool_kernel;
  if (kind == KVEVICT_MASS_SNAPKV && (pk < 1 || pk % 2 == 0)) return KVEVICT_E_POOL_KERNEL_EVEN;
  const int pool_r = kind == KVEVICT_MASS_SNAPKV && pk > 1 ? (pk - 1) / 2 : -1;
  kve::note_other(ctx->c);
  return cuda_status(kve::launch_score_mass(ctx->c, layer, q_win, w, q_pos, kind == KVEVICT_MASS_H2O, pool_r, lse,
                                            scores, static_cast<cudaStream_t>(stream)));
}

kvevict_status kvevict_select(kvevict_ctx* ctx, const void* keys, int32_t key_dtype, const int32_t* positions,
                              const int32_t* counts, int32_t n_lanes, int32_t stride, int32_t budget,
                              int32_t recent_window, int32_t* victims, int32_t* n_victims, void* stream) {
  const CallRange range("kvevict_select");
  if (!ctx || !keys || !positions || !counts || !victims || !n_victims || n_lanes < 0 || stride < 1 ||
      recent_window < 1 || budget < 0)
    return KVEVICT_E_INVALID_ARG;
  if (key_dtype != KVEVICT_KEY_F32 && key_dtype != KVEVICT_KEY_F64) return KVEVICT_E_DTYPE;
  if (n_lanes == 0) return KVEVICT_OK;
  kve::note_other(ctx->c);
  return cuda_status(kve::launch_select(ctx->c, keys, key_dtype, positions, counts, n_lanes, stride, budget,
                                        recent_window, victims, n_victims, static_cast<cudaStream_t>(stream)));
}

kvevict_status kvevict_compact(kvevict_ctx* ctx, int layer, const int32_t* victims, const int32_t* n_victims,
                               int32_t* freed, int32_t* n_freed, int32_t* moves, int32_t* n_moves, void* stream) {
  const CallRange range("kvevict_compact");
  if (!ctx || layer < 0 || layer >= ctx->c.dims.L || !victims || !n_victims) return KVEVICT_E_INVALID_ARG;
  kve::note_other(ctx->c);
  return cuda_status(kve::launch_compact(ctx->c, ctx->c.ws, layer, victims, n_victims, false, freed, n_freed, moves,
                                         n_moves,
                                         static_cast<cudaStream_t>(stream)));
}

kvevict_status kvevict_stats(kvevict_ctx* ctx, int layer, int64_t* out, void* stream) {
  if (!ctx || !out || layer < 0 || layer >= ctx->c.dims.L) return KVEVICT_E_INVALID_ARG;
  kve::note_other(ctx->c);
  return cuda_status(kve::launch_stats(ctx->c, layer, reinterpret_cast<long long*>(out),
                                       static_cast<cudaStream_t>(stream)));
}

int32_t kvevict_kernels_per_decode_step(const kvevict_ctx* ctx) {
  if (!ctx) return 0;
  return (ctx->c.epi_applies || ctx->c.lean_epi) ? 2 : 3;
}

kvevict_status kvevict_check_wait_timeout(kvevict_ctx* ctx, int32_t polls, void* stream) {
  if (!ctx || polls < 1 || polls > (1 << 22)) return KVEVICT_E_INVALID_ARG;
  kve::note_other(ctx->c);
  return cuda_status(kve::launch_wait_check(ctx->c, polls, static_cast<cudaStream_t>(stream)));
}

kvevict_status kvevict_last_error(kvevict_ctx* ctx, char* buf, size_t len) {
  if (!ctx) return KVEVICT_E_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  uint32_t st = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&st, ctx->c.ws.status, 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(ctx->c.ws.status, 0, 4);
  if (e != cudaSuccess) {
    if (buf && len) snprintf(buf, len, "CUDA error: %s", cudaGetErrorString(e));
    return KVEVICT_E_CUDA;
  }
  if (buf && len) {
    snprintf(buf, len, "%s%s%s%s%s", st == 0 ? "ok" : "",
             (st & kve::ST_NO_BLOCKS) ? "pool exhausted; " : "", (st & kve::ST_BAD_INDEX) ? "table index out of range; " : "",
             (st & kve::ST_TIMEOUT) ? "bounded wait gave up; " : "",
             (st & (kve::ST_CAPACITY | kve::ST_POSITION)) ? "token table full or position not increasing; " : "");
  }
  if (st & kve::ST_TIMEOUT) return KVEVICT_E_TIMEOUT;
  return st ? KVEVICT_E_DEVICE : KVEVICT_OK;
}

}  // extern "C"
