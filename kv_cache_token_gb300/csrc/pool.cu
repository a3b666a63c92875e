// Pool management: reset, prompt admission, standalone bottom-k selection,
// forced compaction with its freed-block / move outputs, and the layer
// metrics (vToken review, Eq. (1) and Fig. 1's share of blocks at <= 50%
// utilisation).
#include <cooperative_groups.h>

#include "lane_ops.cuh"

namespace kve {
namespace {

constexpr int kThreads = 512;
constexpr int kSelThreads = 1024;

// ---------------------------------------------------------------------------
// prompt admission
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) prefill_alloc_kernel(LayerState ls, Workspace ws, Dims dm, int n) {
  __shared__ int sh_scan[40];
  __shared__ int sh_bad;
  const int tid = threadIdx.x;
  const int need = (n + kBlock - 1) / kBlock;
  const int total = need * dm.lanes;
  if (tid == 0) sh_bad = 0;
  __syncthreads();
  for (int l = tid; l < dm.lanes; l += blockDim.x)
    if (ls.count[l] != 0) sh_bad = 1;
  __syncthreads();
  if (sh_bad || n > dm.cap - 1) {
    if (tid == 0) { ws.counters[4] = 0; set_status(ws.status, ST_CAPACITY); }
    return;
  }
  int found = 0;
  for (int base = 0; base < dm.P && found < total; base += blockDim.x) {
    const int blk = base + tid;
    const int fr = (blk < dm.P && ls.owner[blk] < 0) ? 1 : 0;
    int tot;
    const int ex = block_excl_scan(fr, sh_scan, &tot);
    if (fr && found + ex < total) ws.alloc_ids[found + ex] = blk;
    found += tot;
  }
  __syncthreads();
  if (found < total) {
    if (tid == 0) { ws.counters[4] = 0; set_status(ws.status, ST_NO_BLOCKS); }
    return;
  }
  for (int j = tid; j < total; j += blockDim.x) {
    const int blk = ws.alloc_ids[j];
    const int l = j / need, jb = j % need;
    ls.owner[blk] = l;
    const int filled = min(kBlock, n - jb * kBlock);
    ls.mask[blk] = filled >= kBlock ? 0xFFFF : ((1 << filled) - 1);
    ls.lane_blocks[static_cast<size_t>(l) * dm.cap + jb] = blk;
  }
  for (int l = tid; l < dm.lanes; l += blockDim.x) {
    ls.lane_nblocks[l] = need;
    ls.count[l] = n;
    ls.ring_slot[l] = 0;
  }
  if (tid == 0) ws.counters[4] = 1;
}

// grid (token chunks, lanes): table entries and K/V rows (16-byte pieces)
template <typename KT>
__global__ void __launch_bounds__(kThreads) prefill_fill_kernel(LayerState ls, Workspace ws, Dims dm, int n,
                                                               const KT* kc, const KT* vc) {
  if (ws.counters[4] == 0) return;
  const int l = blockIdx.y;
  const int need = (n + kBlock - 1) / kBlock;
  const int per = 256;   // tokens per CTA
  const int t0 = blockIdx.x * per;
  if (t0 >= n) return;
  const int t1 = min(n, t0 + per);
  const size_t lo = static_cast<size_t>(l) * dm.cap;
  for (int i = t0 + threadIdx.x; i < t1; i += blockDim.x) {
    const int blk = ws.alloc_ids[l * need + i / kBlock];
    ls.pos[lo + i] = i;
    ls.slot[lo + i] = blk * kBlock + (i % kBlock);
    if (ls.score) ls.score[lo + i] = 0.f;
  }
  if (ls.ring) {
    float* r = ls.ring + lo * dm.W;
    for (size_t e = static_cast<size_t>(t0) * dm.W + threadIdx.x; e < static_cast<size_t>(t1) * dm.W; e += blockDim.x)
      r[e] = 0.f;
  }
  const int vec = 16 / sizeof(KT);               // elements per 16-byte piece
  const int per_row = dm.d / vec;
  const size_t src_lane = static_cast<size_t>(l) * n * dm.d;
  const uint4* ks = reinterpret_cast<const uint4*>(kc + src_lane);
  const uint4* vs = reinterpret_cast<const uint4*>(vc + src_lane);
  uint4* kd = reinterpret_cast<uint4*>(ls.k_pool);
  uint4* vd = reinterpret_cast<uint4*>(ls.v_pool);
  for (int e = threadIdx.x; e < (t1 - t0) * per_row; e += blockDim.x) {
    const int i = t0 + e / per_row, c = e % per_row;
    const int blk = ws.alloc_ids[l * need + i / kBlock];
    const size_t slot = static_cast<size_t>(blk) * kBlock + (i % kBlock);
    kd[slot * per_row + c] = ks[static_cast<size_t>(i) * per_row + c];
    vd[slot * per_row + c] = vs[static_cast<size_t>(i) * per_row + c];
  }
}

// ---------------------------------------------------------------------------
// standalone selection
// ---------------------------------------------------------------------------
template <typename KeyT>
__global__ void __launch_bounds__(kSelThreads) select_kernel(const KeyT* keys, const int32_t* positions,
                                                            const int32_t* counts, int stride, int budget, int R,
                                                            int32_t* victims, int32_t* n_victims) {
  __shared__ __align__(16) int sh_hist[256];   // also read as 64-bit words
  __shared__ int sh_misc[40];
  __shared__ int sh_scan[40];
  const int l = blockIdx.x;
  const int n = max(0, min(counts[l], stride));
  const KeyT* kk = keys + static_cast<size_t>(l) * stride;
  const int32_t* pp = positions + static_cast<size_t>(l) * stride;
  if (n == 0) {
    if (threadIdx.x == 0) n_victims[l] = 0;
    return;
  }
  const int newest = pp[n - 1];
  const int cut = newest - R + 1;
  const int k = max(0, n - budget);
  auto candf = [&](int i) { return pp[i] < cut; };
  auto posf = [&](int i) { return static_cast<uint32_t>(pp[i]); };
  auto keyf = [&](int i) { return mono_key(kk[i]); };
  const SelectResult sel = block_bottom_k(n, k, sizeof(KeyT) * 8, keyf, posf, candf, sh_hist, sh_misc);
  int total = 0;
  int32_t* vo = victims + static_cast<size_t>(l) * stride;
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const bool v = i < n && candf(i) && select_is_victim(sel, keyf(i), posf(i));
    int tot;
    const int ex = block_excl_scan(v ? 1 : 0, sh_scan, &tot);
    if (v) vo[total + ex] = pp[i];
    total += tot;
  }
  if (threadIdx.x == 0) n_victims[l] = total;
}

// Selection by a cluster of kSelCluster CTAs per lane: each CTA takes a
// contiguous slice of the lane's entries; every radix pass merges the CTAs'
// 256-bin histograms into the leader CTA's shared memory (distributed shared
// memory atomics) and the leader's bucket choice is read back by all; the
// victims are written ascending, each CTA at the offset of the lower ranks'
// counts.  Same result as select_kernel.
constexpr int kSelCluster = 8;
constexpr int kSelClThreads = 1024;

struct SelState {
  unsigned long long key_prefix, key_mask;
  uint32_t pos_prefix, pos_mask;
  int k_rem, done, inclusive;
};

template <typename KeyT>
__global__ void __cluster_dims__(kSelCluster, 1, 1) __launch_bounds__(kSelClThreads)
    select_cluster_kernel(const KeyT* keys, const int32_t* positions, const int32_t* counts, int stride,
                          int budget, int R, int32_t* victims, int32_t* n_victims) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ int sh_hist[256];       // leader: merged histogram
  __shared__ int sh_local[256];      // this CTA's histogram
  __shared__ SelState sh_state;      // leader: the descent so far
  __shared__ int sh_count;           // this CTA's number of victims
  __shared__ int sh_scan[40];
  const int rank = static_cast<int>(cluster.block_rank());
  const int l = blockIdx.x / kSelCluster;
  const int tid = threadIdx.x;
  const int n = max(0, min(counts[l], stride));
  const int k = max(0, n - budget);
  if (n == 0 || k == 0) {               // uniform over the cluster
    if (rank == 0 && tid == 0) n_victims[l] = 0;
    return;
  }
  const KeyT* kk = keys + static_cast<size_t>(l) * stride;
  const int32_t* pp = positions + static_cast<size_t>(l) * stride;
  const int cut = pp[n - 1] - R + 1;
  const int chunk = (n + kSelCluster - 1) / kSelCluster;
  const int i_begin = min(n, rank * chunk), i_end = min(n, i_begin + chunk);
  int* lead_hist = cluster.map_shared_rank(sh_hist, 0);
  SelState* lead = cluster.map_shared_rank(&sh_state, 0);
  if (rank == 0 && tid == 0) {
    sh_state.key_prefix = 0; sh_state.key_mask = 0; sh_state.pos_prefix = 0; sh_state.pos_mask = 0;
    sh_state.k_rem = k; sh_state.done = 0; sh_state.inclusive = 0;
  }
  const int key_bits = static_cast<int>(sizeof(KeyT)) * 8;
  SelectResult r;
  r.key_prefix = 0; r.key_mask = 0; r.pos_prefix = 0; r.pos_mask = 0; r.inclusive = 0; r.k = k;
  if (rank == 0 && tid < 256) sh_hist[tid] = 0;
  cluster.sync();
  for (int shift = key_bits + 32 - 8; shift >= 0; shift -= 8) {
    if (tid < 256) sh_local[tid] = 0;
    __syncthreads();
    for (int i = i_begin + tid; i < i_end; i += blockDim.x) {
      const int p = pp[i];
      if (p >= cut) continue;
      const unsigned long long key = mono_key(kk[i]);
      if ((key & r.key_mask) != r.key_prefix || (static_cast<uint32_t>(p) & r.pos_mask) != r.pos_prefix) continue;
      const int digit = shift >= 32 ? static_cast<int>((key >> (shift - 32)) & 0xFF)
                                    : static_cast<int>((static_cast<uint32_t>(p) >> shift) & 0xFF);
      atomicAdd(&sh_local[digit], 1);
    }
    __syncthreads();
    if (tid < 256 && sh_local[tid]) atomicAdd(&lead_hist[tid], sh_local[tid]);
    cluster.sync();
    if (rank == 0 && tid < 32) {
      // the bucket where the cumulative count reaches k_rem
      const int k_rem = sh_state.k_rem;
      int c[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) { c[j] = sh_hist[tid * 8 + j]; sum += c[j]; }
      const int inc = warp_incl_scan(sum), exc = inc - sum;
      int found = -1, below = 0, cnt = 0;
      if (exc < k_rem && inc >= k_rem) {
        int acc = exc;
        for (int j = 0; j < 8; ++j) {
          if (acc + c[j] >= k_rem) { found = tid * 8 + j; below = acc; cnt = c[j]; break; }
          acc += c[j];
        }
      }
      const unsigned ball = __ballot_sync(0xffffffffu, found >= 0);
      const int src = ball ? __ffs(ball) - 1 : 0;
      found = __shfl_sync(0xffffffffu, found, src);
      below = __shfl_sync(0xffffffffu, below, src);
      cnt = __shfl_sync(0xffffffffu, cnt, src);
#pragma unroll
      for (int j = 0; j < 8; ++j) sh_hist[tid * 8 + j] = 0;   // ready for the next pass
      if (tid == 0) {
        if (!ball) {
          sh_state.done = 1; sh_state.inclusive = 1;    // fewer candidates than k: all matching are victims
        } else {
          if (shift >= 32) {
            sh_state.key_prefix |= static_cast<unsigned long long>(found) << (shift - 32);
            sh_state.key_mask |= 0xFFull << (shift - 32);
          } else {
            sh_state.pos_prefix |= static_cast<uint32_t>(found) << shift;
            sh_state.pos_mask |= 0xFFu << shift;
          }
          sh_state.k_rem = k_rem - below;
          if (cnt == k_rem - below || shift == 0) { sh_state.done = 1; sh_state.inclusive = 1; }
        }
      }
    }
    cluster.sync();
    const SelState st = *lead;
    r.key_prefix = st.key_prefix; r.key_mask = st.key_mask;
    r.pos_prefix = st.pos_prefix; r.pos_mask = st.pos_mask; r.inclusive = st.inclusive;
    if (st.done) break;
  }
  // victims of this CTA's slice, counted, then written at the cluster offset
  int mine = 0;
  for (int i = i_begin + tid; i < i_end; i += blockDim.x) {
    const int p = pp[i];
    mine += (p < cut && select_is_victim(r, mono_key(kk[i]), static_cast<uint32_t>(p))) ? 1 : 0;
  }
  int tot;
  (void)block_excl_scan(mine, sh_scan, &tot);
  if (tid == 0) sh_count = tot;
  cluster.sync();
  int offset = 0, all = 0;
  for (int q = 0; q < kSelCluster; ++q) {
    const int cq = *cluster.map_shared_rank(&sh_count, q);
    if (q < rank) offset += cq;
    all += cq;
  }
  int32_t* vo = victims + static_cast<size_t>(l) * stride;
  for (int base = i_begin; base < i_end; base += blockDim.x) {
    const int i = base + tid;
    bool v = false;
    int p = 0;
    if (i < i_end) {
      p = pp[i];
      v = p < cut && select_is_victim(r, mono_key(kk[i]), static_cast<uint32_t>(p));
    }
    int t2;
    const int ex = block_excl_scan(v ? 1 : 0, sh_scan, &t2);
    if (v) vo[offset + ex] = p;
    offset += t2;
  }
  if (rank == 0 && tid == 0) n_victims[l] = all;
  cluster.sync();    // no CTA leaves while another may still read its shared memory
}

// ---------------------------------------------------------------------------
// forced compaction
// ---------------------------------------------------------------------------
// Victim test against an ascending victim list: per chunk of table entries
// the list's slice that can match (it starts at the first victim position
// not below the chunk's first position) is staged in shared memory, and
// each entry is looked up there.  The slice start only moves forward.
struct SegVictims {
  const int32_t* vl;
  int k;
  const int32_t* pos;
  int* seg;
  int* sh_len;
  int start, len;
  __device__ void prepare(int base) {
    if (base > 0) {
      // drop the slice entries below this chunk's first position
      const int p0 = pos[base];
      for (;;) {
        const int c = __syncthreads_count(static_cast<int>(threadIdx.x) < len && seg[threadIdx.x] < p0);
        start += c;
        if (c < len || start >= k) break;
        // the whole slice was below p0 (victims not in the table): next slice
        len = min(static_cast<int>(blockDim.x), k - start);
        if (static_cast<int>(threadIdx.x) < len) seg[threadIdx.x] = vl[start + threadIdx.x];
        __syncthreads();
      }
    }
    len = min(static_cast<int>(blockDim.x), max(0, k - start));
    __syncthreads();
    if (static_cast<int>(threadIdx.x) < len) seg[threadIdx.x] = vl[start + threadIdx.x];
    __syncthreads();
  }
  __device__ bool operator()(int i) const {
    const int p = pos[i];
    int lo = 0, hi = len;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (seg[mid] < p) lo = mid + 1; else hi = mid;
    }
    return lo < len && seg[lo] == p;
  }
};

__global__ void __launch_bounds__(kThreads) compact_evict_kernel(LayerState ls, Workspace ws, Dims dm,
                                                                const int32_t* victims,
                                                                const int32_t* n_victims) {
  __shared__ int sh_scan[40];
  __shared__ int sh_seg[kThreads];
  __shared__ int sh_seg_len;
  __shared__ int sh_idx[kThreads];
  __shared__ __align__(16) float sh_rows[128 * kMaxW];
  const int l = blockIdx.x, tid = threadIdx.x;
  LaneRefs L = lane_refs(ls, dm, l);
  const int n = ls.count[l];
  if (n < 0 || n > dm.cap) {
    if (tid == 0) { set_status(ws.status, ST_BAD_INDEX); ws.want_dst[l] = 0; ws.need_admit[l] = 0; }
    return;
  }
  const int k = max(0, min(n_victims[l], n));
  SegVictims isv;
  isv.vl = victims + static_cast<size_t>(l) * dm.cap;
  isv.k = k;
  isv.pos = L.pos;
  isv.seg = sh_seg;
  isv.sh_len = &sh_seg_len;
  isv.start = 0;
  isv.len = 0;
  int dead = 0;
  const int vcount = lane_remove(L, n, isv, nullptr, ws.freed_flag, &dead, dm.P, ws.status, sh_scan, sh_idx,
                                 sh_rows);
  const int m = n - vcount;
  if (tid == 0) ls.count[l] = m;
  const int nb = lane_prune_blocks(L, l, sh_scan);
  int t_live = 0;
  const int ndst = lane_plan(L, nb, m, true, dm.theta_f, false, &t_live, sh_scan);
  if (tid == 0) {
    ws.need_admit[l] = 0;
    ws.want_dst[l] = ndst;
    ws.plan_tlive[l] = t_live;
    if (ndst > 0) atomicOr(ws.work_flag, 1);
    atomicAdd(reinterpret_cast<unsigned long long*>(&ls.stats[SC_VICTIMS]), (unsigned long long)vcount);
    if (dead) atomicAdd(reinterpret_cast<unsigned long long*>(&ls.stats[SC_FREED_DEAD]), (unsigned long long)dead);
  }
}

__global__ void __launch_bounds__(1024) compact_finalize_kernel(Workspace ws, Dims dm, int32_t* freed,
                                                               int32_t* n_freed, int32_t* n_moves) {
  __shared__ int sh_scan[40];
  int total = 0;
  for (int base = 0; base < dm.P; base += blockDim.x) {
    const int blk = base + threadIdx.x;
    const int f = (blk < dm.P && ws.freed_flag[blk]) ? 1 : 0;
    int tot;
    const int ex = block_excl_scan(f, sh_scan, &tot);
    if (f) {
      if (freed) freed[total + ex] = blk;
      ws.freed_flag[blk] = 0;
    }
    total += tot;
  }
  if (threadIdx.x == 0) {
    if (n_freed) *n_freed = total;
    if (n_moves) *n_moves = ws.counters[1] ? ws.counters[2] : 0;
  }
}

// ---------------------------------------------------------------------------
// metrics
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) stats_kernel(LayerState ls, Dims dm, long long* out) {
  __shared__ unsigned long long sh[3][32];
  unsigned long long N = 0, live = 0, half = 0;
  for (int blk = threadIdx.x; blk < dm.P; blk += blockDim.x) {
    if (ls.owner[blk] >= 0) {
      const int c = __popc(ls.mask[blk] & 0xFFFF);
      ++N;
      live += c;
      if (c <= kBlock / 2) ++half;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    N += __shfl_xor_sync(0xffffffffu, N, o);
    live += __shfl_xor_sync(0xffffffffu, live, o);
    half += __shfl_xor_sync(0xffffffffu, half, o);
  }
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) { sh[0][w] = N; sh[1][w] = live; sh[2][w] = half; }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long a = 0, b = 0, c = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) { a += sh[0][i]; b += sh[1][i]; c += sh[2][i]; }
    for (int i = 0; i < SC_NCOUNTERS; ++i) out[i] = ls.stats[i];
    out[KVEVICT_STAT_BLOCKS] = (long long)a;
    out[KVEVICT_STAT_LIVE] = (long long)b;
    out[KVEVICT_STAT_HALF_EMPTY] = (long long)c;
    out[KVEVICT_STAT_LANES] = dm.lanes;
  }
}

}  // namespace

cudaError_t launch_prefill(const Ctx& ctx, int layer, const void* k, const void* v, int n, cudaStream_t stream) {
  LayerState ls = layer_state(ctx, layer);
  prefill_alloc_kernel<<<1, 1024, 0, stream>>>(ls, ctx.ws, ctx.dims, n);
  dim3 grid((n + 255) / 256, ctx.dims.lanes);
  if (ctx.dims.dtype == KVEVICT_BF16)
    prefill_fill_kernel<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(
        ls, ctx.ws, ctx.dims, n, static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v));
  else
    prefill_fill_kernel<float><<<grid, kThreads, 0, stream>>>(ls, ctx.ws, ctx.dims, n,
                                                             static_cast<const float*>(k),
                                                             static_cast<const float*>(v));
  return cudaGetLastError();
}

cudaError_t launch_select(const Ctx& ctx, const void* keys, int key_dtype, const int32_t* positions,
                          const int32_t* counts, int n_lanes, int stride, int budget, int recent,
                          int32_t* victims, int32_t* n_victims, cudaStream_t stream) {
  (void)ctx;
  if (n_lanes <= 0) return cudaSuccess;
  if (key_dtype == KVEVICT_KEY_F64)
    select_cluster_kernel<double><<<n_lanes * kSelCluster, kSelClThreads, 0, stream>>>(
        static_cast<const double*>(keys), positions, counts, stride, budget, recent, victims, n_victims);
  else
    select_cluster_kernel<float><<<n_lanes * kSelCluster, kSelClThreads, 0, stream>>>(
        static_cast<const float*>(keys), positions, counts, stride, budget, recent, victims, n_victims);
  return cudaGetLastError();
}

cudaError_t launch_compact(const Ctx& ctx, int layer, const int32_t* victims, const int32_t* n_victims,
                           int32_t* freed, int32_t* n_freed, int32_t* moves, int32_t* n_moves,
                           cudaStream_t stream) {
  LayerState ls = layer_state(ctx, layer);
  compact_evict_kernel<<<ctx.dims.lanes, kThreads, 0, stream>>>(ls, ctx.ws, ctx.dims, victims, n_victims);
  cudaError_t e = launch_allocate_apply(ctx, layer, nullptr, nullptr, true, moves, stream, true);
  if (e != cudaSuccess) return e;
  compact_finalize_kernel<<<1, 1024, 0, stream>>>(ctx.ws, ctx.dims, freed, n_freed, n_moves);
  return cudaGetLastError();
}

cudaError_t launch_stats(const Ctx& ctx, int layer, long long* out, cudaStream_t stream) {
  LayerState ls = layer_state(ctx, layer);
  stats_kernel<<<1, 1024, 0, stream>>>(ls, ctx.dims, out);
  return cudaGetLastError();
}

cudaError_t launch_decode(const Ctx& ctx, int layer, const void* q, const void* k_new, const void* v_new,
                          int new_pos, float* out, float* lse, int32_t* victims, int32_t* n_victims,
                          cudaStream_t stream) {
  cudaError_t e;
  if (q) {
    e = launch_attend(ctx, layer, q, k_new, v_new, stream);
    if (e != cudaSuccess) return e;
  }
  e = launch_epilogue(ctx, layer, q != nullptr, new_pos, k_new, v_new, out, lse, victims, n_victims, stream);
  if (e != cudaSuccess) return e;
  return launch_allocate_apply(ctx, layer, k_new, v_new, false, nullptr, stream, false);
}

}  // namespace kve
