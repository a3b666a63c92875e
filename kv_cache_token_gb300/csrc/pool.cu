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
    // empty histories, at the tokens' slots
    for (int e = threadIdx.x; e < (t1 - t0) * dm.W; e += blockDim.x) {
      const int i = t0 + e / dm.W, t = e % dm.W;
      const int blk = ws.alloc_ids[l * need + i / kBlock];
      ls.ring[(static_cast<size_t>(blk) * kBlock + i % kBlock) * dm.W + t] = 0.f;
    }
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

// Selection by a cluster of kCl CTAs per lane (8, or 16 for tables of at
// least kSelWideFrom entries, where the wider split measured faster): each CTA takes a
// contiguous slice of the lane's entries; every radix pass merges the CTAs'
// 256-bin histograms into the leader CTA's shared memory (distributed shared
// memory atomics) and the leader's bucket choice is read back by all; the
// victims are written ascending, each CTA at the offset of the lower ranks'
// counts.  Same result as select_kernel.
constexpr int kSelCluster = 8;        // CTAs per lane below kSelWideFrom entries
constexpr int kSelClusterWide = 16;   // at or above (a non-portable cluster size)
constexpr int kSelWideFrom = 1 << 16;
constexpr int kSelClThreads = 1024;

struct SelState {
  unsigned long long key_prefix, key_mask;
  uint32_t pos_prefix, pos_mask;
  int k_rem, done, inclusive;
};

template <typename KeyT, int kCl>
__global__ void __launch_bounds__(kSelClThreads)
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
  const int l = blockIdx.x / kCl;
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
  const int chunk = (n + kCl - 1) / kCl;
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
  for (int q = 0; q < kCl; ++q) {
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
// Removal, cmp_ctas_per_lane CTAs per lane
// over contiguous ranges of the table (one wave at 128K instead of one CTA
// per lane).  compact_remove_kernel: each CTA finds the slice of the
// ascending victim list that can match its range (positions between its
// first and last entry; extra positions match nothing, as in the oracle's
// membership test), stages it in shared memory when it fits, tests each
// entry by binary search, clears the victims' live bits and writes its
// survivors, in order, to
// scratch at the range start, with their count.
// compact_place_kernel: each CTA copies its survivors to their final index
// (the counts of the lane's earlier CTAs before it; the lane's entry count
// before the removal comes from scratch).
constexpr int kCmpThreads = 512;
constexpr int kCmpStage = 4096;     // victim-slice entries staged in shared memory

// cmp_cnt per lane: cpl survivor counts, then the entry count before the
// removal (-1 for a count out of range)

// First index of the ascending a[0..k) whose value is >= x (strict: > x),
// by one warp: 32 probes per round narrow the interval 32-fold, so a
// search costs a few dependent loads instead of one per halving.
template <bool kStrict>
__device__ __forceinline__ int warp_lower_bound(const int32_t* a, int k, int x) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = k;   // the answer lies in [lo, hi]
  while (hi - lo > 32) {
    const int step = (hi - lo + 31) / 32;
    const int idx = lo + lane * step;
    const int v = idx < hi ? a[idx] : 0x7FFFFFFF;
    const bool ge = idx >= hi || (kStrict ? v > x : v >= x);
    const unsigned bal = __ballot_sync(0xffffffffu, ge);
    const int f = __ffs(bal) - 1;        // first probe at or past the answer (lane 31 at worst... or none)
    if (bal == 0u) {
      lo = lo + 31 * step + 1;
    } else {
      const int nhi = min(hi, lo + f * step);
      lo = f == 0 ? lo : lo + (f - 1) * step + 1;
      hi = nhi;
    }
  }
  const int idx = lo + lane;
  const bool ge = idx >= hi || (kStrict ? a[idx] > x : a[idx] >= x);
  const unsigned bal = __ballot_sync(0xffffffffu, ge);
  return bal ? lo + __ffs(bal) - 1 : hi;
}

__global__ void __launch_bounds__(kCmpThreads) compact_remove_kernel(LayerState ls, Workspace ws, Dims dm,
                                                                    const int32_t* victims,
                                                                    const int32_t* n_victims, int cpl) {
  __shared__ int sh_vic[kCmpStage];
  __shared__ int sh_scan[40];
  __shared__ int sh_v0, sh_v1;
  const int l = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  LaneRefs L = lane_refs(ls, dm, l);
  const int n = ls.count[l];
  const bool lane_ok = n >= 0 && n <= dm.cap;
  if (c == 0 && tid == 0) ws.cmp_cnt[static_cast<size_t>(l) * (cpl + 1) + cpl] = lane_ok ? n : -1;
  if (!lane_ok) return;
  const int per = (n + cpl - 1) / cpl;
  const int s = min(n, c * per), e = min(n, s + per);
  const int k = max(0, min(n_victims[l], n));
  const int32_t* vl = victims + static_cast<size_t>(l) * dm.cap;
  // the victims between the range's first and last position: warp 0 finds
  // the first >= the first position, warp 1 the first > the last
  if (tid < 64) {
    int v = 0;
    if (s < e && k > 0) {
      v = tid < 32 ? warp_lower_bound<false>(vl, k, L.pos[s]) : warp_lower_bound<true>(vl, k, L.pos[e - 1]);
    }
    if ((tid & 31) == 0) {
      if (tid == 0) sh_v0 = v; else sh_v1 = v;
    }
  }
  __syncthreads();
  const int v0 = sh_v0, len = sh_v1 - sh_v0;
  const bool staged = len <= kCmpStage;
  if (staged)
    for (int i = tid; i < len; i += blockDim.x) sh_vic[i] = vl[v0 + i];
  __syncthreads();
  const int* slice = staged ? sh_vic : vl + v0;
  const size_t lo_off = static_cast<size_t>(l) * dm.cap;
  int kept_total = 0, vict_total = 0;
  for (int base = s; base < e; base += blockDim.x) {
    const int i = base + tid;
    int p = 0, sl = 0;
    float sc = 0.f;
    bool isv = false, keep = false;
    if (i < e) {
      p = L.pos[i];
      sl = L.slot[i];
      if (L.score) sc = L.score[i];
      int lo = 0, hi = len;
      while (lo < hi) { const int mid = (lo + hi) >> 1; if (slice[mid] < p) lo = mid + 1; else hi = mid; }
      isv = lo < len && slice[lo] == p;
      keep = !isv;
    }
    int tot2;
    const int ex2 = block_excl_scan((keep ? 1 : 0) | (isv ? 0x10000 : 0), sh_scan, &tot2);
    if (keep) {
      const size_t o = lo_off + s + kept_total + (ex2 & 0xFFFF);
      ws.cmp_pos[o] = p;
      ws.cmp_slot[o] = sl;
      ws.cmp_score[o] = sc;
    }
    if (isv) {
      if (sl >= 0 && sl < dm.P * kBlock) {
        atomicAnd(&L.mask[sl >> 4], ~(1 << (sl & 15)));
      } else if (sl >= 0) {
        set_status(ws.status, ST_BAD_INDEX);
      }
    }
    kept_total += tot2 & 0xFFFF;
    vict_total += tot2 >> 16;
  }
  if (tid == 0) {
    ws.cmp_cnt[static_cast<size_t>(l) * (cpl + 1) + c] = kept_total;
    if (vict_total) atomicAdd(reinterpret_cast<unsigned long long*>(&ls.stats[SC_VICTIMS]), (unsigned long long)vict_total);
  }
}

__global__ void __launch_bounds__(kCmpThreads) compact_place_kernel(LayerState ls, Workspace ws, Dims dm, int cpl) {
  __shared__ int sh_off;
  const int l = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  LaneRefs L = lane_refs(ls, dm, l);
  const int32_t* cnt = ws.cmp_cnt + static_cast<size_t>(l) * (cpl + 1);
  const int n = cnt[cpl];
  if (n < 0) {
    if (c == 0 && tid == 0) { set_status(ws.status, ST_BAD_INDEX); ws.want_dst[l] = 0; ws.need_admit[l] = 0; }
    return;
  }
  const int per = (n + cpl - 1) / cpl;
  const int s = min(n, c * per);
  if (tid < 32) {
    int before = 0;
    for (int j = tid; j < c; j += 32) before += cnt[j];
    for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
    if (tid == 0) sh_off = before;
  }
  __syncthreads();
  const int off = sh_off, mine = cnt[c];
  const size_t lo_off = static_cast<size_t>(l) * dm.cap;
  for (int j = tid; j < mine; j += blockDim.x) {
    L.pos[off + j] = ws.cmp_pos[lo_off + s + j];
    L.slot[off + j] = ws.cmp_slot[lo_off + s + j];
    if (L.score) L.score[off + j] = ws.cmp_score[lo_off + s + j];
  }
}

// One CTA per lane after the removal, kBlkPer consecutive entries of the
// lane's block list per thread, all loads of a pass issued together: sets
// the count, releases the blocks the removal emptied (every live bit was
// cleared by the removal kernel), drops them from the list (stably), and
// sizes the forced relocation plan from the remaining blocks' live counts
// (vToken review, Sec. 3.3 Stage 1).
constexpr int kBlkPer = 8;

__global__ void __launch_bounds__(1024) compact_blocks_kernel(LayerState ls, Workspace ws, Dims dm, int cpl,
                                                              int gated) {
  __shared__ int sh_scan[40];
  __shared__ int sh_m;
  const int l = blockIdx.x, tid = threadIdx.x;
  LaneRefs L = lane_refs(ls, dm, l);
  const int32_t* cnt = ws.cmp_cnt + static_cast<size_t>(l) * (cpl + 1);
  if (cnt[cpl] < 0) {
    if (tid == 0) { set_status(ws.status, ST_BAD_INDEX); ws.want_dst[l] = 0; ws.need_admit[l] = 0; }
    return;
  }
  if (tid < 32) {
    int all = 0;
    for (int j = tid; j < cpl; j += 32) all += cnt[j];
    for (int o = 16; o > 0; o >>= 1) all += __shfl_xor_sync(0xffffffffu, all, o);
    if (tid == 0) sh_m = all;
  }
  const int nb = *L.nblocks;
  int out = 0, dead_tot = 0, src_tot = 0, tl_tot = 0;
  for (int base = 0; base < nb; base += blockDim.x * kBlkPer) {
    const int j0 = base + tid * kBlkPer;
    int b[kBlkPer], mk[kBlkPer], ow[kBlkPer];
#pragma unroll
    for (int u = 0; u < kBlkPer; ++u) {
      b[u] = j0 + u < nb ? L.blocks[j0 + u] : -1;
      if (b[u] >= dm.P) b[u] = -1;
    }
#pragma unroll
    for (int u = 0; u < kBlkPer; ++u) {
      mk[u] = b[u] >= 0 ? (__ldcg(L.mask + b[u]) & 0xFFFF) : 0;
      ow[u] = b[u] >= 0 ? L.owner[b[u]] : -1;
    }
    int keep = 0, dead = 0, src = 0, tl = 0;
#pragma unroll
    for (int u = 0; u < kBlkPer; ++u) {
      if (b[u] < 0) continue;
      if (mk[u] == 0) {
        if (ow[u] >= 0) {
          L.owner[b[u]] = -1;
          ws.freed_flag[b[u]] = 1;
          ++dead;
        }
      } else if (ow[u] == l) {
        ++keep;
        const int c = __popc(mk[u]);
        if (c < kBlock) { ++src; tl += c; }
      }
    }
    int tot;
    int ex = block_excl_scan(keep, sh_scan, &tot);
    int tot2, tot3;
    (void)block_excl_scan(dead | (src << 16), sh_scan, &tot2);
    (void)block_excl_scan(tl, sh_scan, &tot3);
    // every read of this pass precedes the scans' barriers; writes go below
    // the next pass's entries
#pragma unroll
    for (int u = 0; u < kBlkPer; ++u)
      if (b[u] >= 0 && mk[u] != 0 && ow[u] == l) L.blocks[out + ex++] = b[u];
    out += tot;
    dead_tot += tot2 & 0xFFFF;
    src_tot += tot2 >> 16;
    tl_tot += tot3;
  }
  __syncthreads();
  if (tid == 0) {
    const int m = sh_m;
    *L.nblocks = out;
    ls.count[l] = m;
    const int ndst = (tl_tot + kBlock - 1) / kBlock;
    const bool over = !gated || (out > 0 && frag_over(m, out, dm.theta_f));
    const int plan = (out > 0 && over && src_tot > ndst) ? ndst : 0;
    ws.need_admit[l] = 0;
    ws.want_dst[l] = plan;
    ws.plan_tlive[l] = plan ? tl_tot : 0;
    if (plan > 0) atomicOr(ws.work_flag, 1);
    if (dead_tot)
      atomicAdd(reinterpret_cast<unsigned long long*>(&ls.stats[SC_FREED_DEAD]), (unsigned long long)dead_tot);
  }
}

// Relocation of the forced compaction (vToken review, Sec. 3.3 Stage 3),
// cmp_ctas_per_lane CTAs per lane over contiguous ranges of the table.  A
// token moves when its block holds between 1 and 15 live tokens (a source;
// the live masks are final after the removal and untouched until
// compact_reloc_finish_kernel); the q-th moving token of the lane in table
// order goes to destination q / 16, offset q % 16.  count: sources per
// range.  move: each CTA ranks its sources after the lane's earlier CTAs,
// points their table slots at the destinations, writes the move tuples and
// copies the K and V rows (eight 16-byte loads in flight per thread).
// finish (one CTA per lane): releases the sources, sets the destinations'
// masks, rebuilds the block list.
__device__ __forceinline__ bool reloc_src(const LaneRefs& L, int old, int P) {
  if (old < 0 || old >= P * kBlock) return false;
  const int c = __popc(__ldcg(L.mask + (old >> 4)) & 0xFFFF);
  return c > 0 && c < kBlock;
}

__global__ void __launch_bounds__(kCmpThreads) compact_reloc_count_kernel(LayerState ls, Workspace ws, Dims dm,
                                                                         int cpl) {
  __shared__ int sh_scan[40];
  const int l = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  if (__ldcg(ws.counters + 1) == 0 || __ldcg(ws.want_dst + l) <= 0) return;
  LaneRefs L = lane_refs(ls, dm, l);
  const int m = min(max(__ldcg(ls.count + l), 0), dm.cap);
  const int per = (m + cpl - 1) / cpl;
  const int s = min(m, c * per), e = min(m, s + per);
  int cnt = 0;
  for (int i = s + tid; i < e; i += blockDim.x) cnt += reloc_src(L, L.slot[i], dm.P) ? 1 : 0;
  int tot;
  (void)block_excl_scan(cnt, sh_scan, &tot);
  if (tid == 0) ws.cmp_cnt[static_cast<size_t>(l) * (cpl + 1) + c] = tot;
}

template <typename KT>
__global__ void __launch_bounds__(kCmpThreads, 1) compact_reloc_move_kernel(LayerState ls, Workspace ws, Dims dm,
                                                                        int cpl, int32_t* moves) {
  constexpr int kBatch = 8;
  __shared__ int sh_scan[40];
  __shared__ int sh_off;
  __shared__ int sh_src[kCmpThreads], sh_dst[kCmpThreads];
  const int l = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  const int ndst = __ldcg(ws.want_dst + l);
  if (__ldcg(ws.counters + 1) == 0 || ndst <= 0) return;
  LaneRefs L = lane_refs(ls, dm, l);
  const int m = min(max(__ldcg(ls.count + l), 0), dm.cap);
  const int per = (m + cpl - 1) / cpl;
  const int s = min(m, c * per), e = min(m, s + per);
  const int32_t* cnt = ws.cmp_cnt + static_cast<size_t>(l) * (cpl + 1);
  if (tid < 32) {
    int before = 0;
    for (int j = tid; j < c; j += 32) before += cnt[j];
    for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
    if (tid == 0) sh_off = before;
  }
  __syncthreads();
  const int dbeg = ws.dst_begin[l], mbeg = ws.move_begin[l];
  const int d = dm.d;
  const int cpr = d * static_cast<int>(sizeof(KT)) / 16;     // 16-byte pieces per K or V row
  const size_t row_bytes = static_cast<size_t>(d) * sizeof(KT);
  unsigned char* kpb = static_cast<unsigned char*>(ls.k_pool);
  unsigned char* vpb = static_cast<unsigned char*>(ls.v_pool);
  int q_run = sh_off;
  for (int base = s; base < e; base += blockDim.x) {
    const int i = base + tid;
    int old = -1;
    bool src = false;
    if (i < e) {
      old = L.slot[i];
      src = reloc_src(L, old, dm.P);
    }
    int tot;
    const int ex = block_excl_scan(src ? 1 : 0, sh_scan, &tot);
    if (src) {
      const int q = q_run + ex;
      if (q / kBlock >= ndst) {
        set_status(ws.status, ST_BAD_INDEX);   // plan and tables disagree: leave the token in place
        sh_src[ex] = -1;
      } else {
        const int db = ws.alloc_ids[dbeg + q / kBlock];
        const int dof = q % kBlock;
        const int ns = db * kBlock + dof;
        sh_src[ex] = old;
        sh_dst[ex] = ns;
        L.slot[i] = ns;
        if (moves) {
          int32_t* mv = moves + static_cast<size_t>(mbeg + q) * 6;
          mv[0] = l; mv[1] = L.pos[i]; mv[2] = old >> 4; mv[3] = old & 15; mv[4] = db; mv[5] = dof;
        }
      }
    }
    __syncthreads();
    const int npieces = tot * 2 * cpr;
    for (int e0 = tid; e0 < npieces; e0 += blockDim.x * kBatch) {
      uint4 v[kBatch];
      unsigned char* dst[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int pe = e0 + u * static_cast<int>(blockDim.x);
        dst[u] = nullptr;
        if (pe < npieces) {
          const int mvi = pe / (2 * cpr), rem = pe - mvi * 2 * cpr;
          const int so = sh_src[mvi];
          if (so >= 0) {
            unsigned char* pool = rem < cpr ? kpb : vpb;
            const size_t c16 = static_cast<size_t>(rem < cpr ? rem : rem - cpr) * 16;
            v[u] = *reinterpret_cast<const uint4*>(pool + static_cast<size_t>(so) * row_bytes + c16);
            dst[u] = pool + static_cast<size_t>(sh_dst[mvi]) * row_bytes + c16;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (dst[u]) *reinterpret_cast<uint4*>(dst[u]) = v[u];
    }
    if (L.ring) move_history_rows(L.ring, L.W, sh_src, sh_dst, tot);
    __syncthreads();
    q_run += tot;
  }
}

__global__ void __launch_bounds__(1024) compact_reloc_finish_kernel(LayerState ls, Workspace ws, Dims dm, int cpl) {
  __shared__ int sh_scan[40];
  __shared__ int sh_moved;
  const int l = blockIdx.x, tid = threadIdx.x;
  const int ndst = __ldcg(ws.want_dst + l);
  if (__ldcg(ws.counters + 1) == 0 || ndst <= 0) return;
  LaneRefs L = lane_refs(ls, dm, l);
  if (tid < 32) {
    int all = 0;
    for (int j = tid; j < cpl; j += 32) all += ws.cmp_cnt[static_cast<size_t>(l) * (cpl + 1) + j];
    for (int o = 16; o > 0; o >>= 1) all += __shfl_xor_sync(0xffffffffu, all, o);
    if (tid == 0) sh_moved = all;
  }
  const int dbeg = ws.dst_begin[l];
  // sources (1 to 15 live tokens) are released; the full blocks stay, in order
  const int nb = *L.nblocks;
  int out = 0, nsrc_tot = 0;
  for (int base = 0; base < nb; base += blockDim.x * kBlkPer) {
    const int j0 = base + tid * kBlkPer;
    int b[kBlkPer], c[kBlkPer], ow[kBlkPer];
#pragma unroll
    for (int u = 0; u < kBlkPer; ++u) {
      b[u] = j0 + u < nb ? L.blocks[j0 + u] : -1;
      if (b[u] >= dm.P) b[u] = -1;
    }
#pragma unroll
    for (int u = 0; u < kBlkPer; ++u) {
      c[u] = b[u] >= 0 ? __popc(L.mask[b[u]] & 0xFFFF) : 0;
      ow[u] = b[u] >= 0 ? L.owner[b[u]] : -1;
    }
    int keep = 0, nsrc = 0;
#pragma unroll
    for (int u = 0; u < kBlkPer; ++u) {
      if (b[u] < 0) continue;
      if (c[u] > 0 && c[u] < kBlock) {
        L.mask[b[u]] = 0;
        L.owner[b[u]] = -1;
        ws.freed_flag[b[u]] = 1;
        ++nsrc;
      } else if (c[u] > 0 && ow[u] == l) {
        ++keep;
      }
    }
    int tot, tot2;
    int ex = block_excl_scan(keep, sh_scan, &tot);
    (void)block_excl_scan(nsrc, sh_scan, &tot2);
#pragma unroll
    for (int u = 0; u < kBlkPer; ++u)
      if (b[u] >= 0 && c[u] == kBlock && ow[u] == l) L.blocks[out + ex++] = b[u];
    out += tot;
    nsrc_tot += tot2;
  }
  __syncthreads();
  const int moved = min(sh_moved, ndst * kBlock);
  for (int j = tid; j < ndst; j += blockDim.x) {
    const int db = ws.alloc_ids[dbeg + j];
    const int filled = min(kBlock, moved - j * kBlock);
    L.mask[db] = filled >= kBlock ? 0xFFFF : (filled > 0 ? (1 << filled) - 1 : 0);
    L.blocks[out + j] = db;
  }
  if (tid == 0) {
    *L.nblocks = out + ndst;
    ws.want_dst[l] = 0;
    atomicAdd(reinterpret_cast<unsigned long long*>(&ls.stats[SC_PLANS]), 1ull);
    atomicAdd(reinterpret_cast<unsigned long long*>(&ls.stats[SC_MOVED]), (unsigned long long)sh_moved);
    atomicAdd(reinterpret_cast<unsigned long long*>(&ls.stats[SC_FREED_RELOC]), (unsigned long long)nsrc_tot);
  }
}

// The freed list: block ids with a set flag, ascending, in two launches over
// ranges of the pool (`span` flags per CTA, walked kFreedChunk at a time):
// count the set flags of each range, then each range writes its ids after
// the earlier ranges' counts, by warp ballots (32 flags per coalesced load),
// and clears them.
constexpr int kFreedPer = 8;                           // flags a thread takes per chunk
constexpr int kFreedChunk = 1024 * kFreedPer;          // flags per CTA per chunk
__global__ void __launch_bounds__(1024) freed_count_kernel(Workspace ws, Dims dm, int span) {
  __shared__ int sh_scan[40];
  const int b0 = blockIdx.x * span, b1 = min(dm.P, b0 + span);
  int c = 0;
  for (int base = b0; base < b1; base += kFreedChunk) {
#pragma unroll
    for (int u = 0; u < kFreedPer; ++u) {
      const int idx = base + u * 1024 + threadIdx.x;
      c += (idx < b1 && ws.freed_flag[idx] != 0) ? 1 : 0;
    }
  }
  int tot;
  (void)block_excl_scan(c, sh_scan, &tot);
  if (threadIdx.x == 0) ws.freed_part[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(1024) freed_write_kernel(Workspace ws, Dims dm, int span, int32_t* freed,
                                                           int32_t* n_freed, int32_t* n_moves) {
  __shared__ int sh_scan[40];
  __shared__ int sh_off;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt = (1u << lane) - 1u;
  if (warp == 0) {
    // this range's offset (and, in CTA 0, the total) from the range counts
    int off = 0, all = 0;
    for (int r = lane; r < static_cast<int>(gridDim.x); r += 32) {
      const int c = ws.freed_part[r];
      if (r < static_cast<int>(blockIdx.x)) off += c;
      all += c;
    }
    for (int o = 16; o > 0; o >>= 1) {
      off += __shfl_xor_sync(0xffffffffu, off, o);
      all += __shfl_xor_sync(0xffffffffu, all, o);
    }
    if (lane == 0) {
      sh_off = off;
      if (blockIdx.x == 0) {
        if (n_freed) *n_freed = all;
        if (n_moves) *n_moves = ws.counters[1] ? ws.counters[2] : 0;
      }
    }
  }
  __syncthreads();
  const int b0 = blockIdx.x * span, b1 = min(dm.P, b0 + span);
  int off = sh_off;
  for (int base = b0; base < b1; base += kFreedChunk) {
    // each warp: 32 * kFreedPer consecutive flags of the chunk
    const int wb = base + warp * 32 * kFreedPer;
    unsigned bal[kFreedPer];
    int wtot = 0;
#pragma unroll
    for (int u = 0; u < kFreedPer; ++u) {
      const int idx = wb + u * 32 + lane;
      bal[u] = __ballot_sync(0xffffffffu, idx < b1 && ws.freed_flag[idx] != 0);
      wtot += __popc(bal[u]);
    }
    int tot;
    const int wex = block_excl_scan(lane == 0 ? wtot : 0, sh_scan, &tot);
    int o = off + __shfl_sync(0xffffffffu, wex, 0);
#pragma unroll
    for (int u = 0; u < kFreedPer; ++u) {
      if ((bal[u] >> lane) & 1u) {
        const int idx = wb + u * 32 + lane;
        if (freed) freed[o + __popc(bal[u] & lt)] = idx;
        ws.freed_flag[idx] = 0;
      }
      o += __popc(bal[u]);
    }
    off += tot;
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

// The bounded-wait path on its own: one thread waits on a shared-memory
// mbarrier that expects one arrival and gets none, gives up after `polls`
// polls, and records ST_TIMEOUT in the status word, as every wait of the
// library does when its producer never arrives.
__global__ void wait_check_kernel(uint32_t* status, int polls) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  (void)mbar_wait_bounded(&bar, 0, status, polls);
}

}  // namespace

cudaError_t launch_wait_check(const Ctx& ctx, int polls, cudaStream_t stream) {
  wait_check_kernel<<<1, 32, 0, stream>>>(ctx.ws.status, polls);
  return cudaGetLastError();
}

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

// One cluster of kCl CTAs per lane (thread-block cluster launch attribute;
// sizes above 8 need the non-portable opt-in).
template <typename KeyT, int kCl>
static cudaError_t launch_sel(int n_lanes, cudaStream_t stream, const KeyT* keys, const int32_t* positions,
                              const int32_t* counts, int stride, int budget, int recent, int32_t* victims,
                              int32_t* n_victims) {
  const auto fn = select_cluster_kernel<KeyT, kCl>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_lanes * kCl);
  cfg.blockDim = dim3(kSelClThreads);
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kCl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, keys, positions, counts, stride, budget, recent, victims, n_victims);
}

// Opt-in to the non-portable cluster size of the wide selection (once per
// context creation).
cudaError_t prepare_select() {
  cudaError_t e = cudaFuncSetAttribute(select_cluster_kernel<float, kSelClusterWide>,
                                       cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(select_cluster_kernel<double, kSelClusterWide>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

cudaError_t launch_select(const Ctx& ctx, const void* keys, int key_dtype, const int32_t* positions,
                          const int32_t* counts, int n_lanes, int stride, int budget, int recent,
                          int32_t* victims, int32_t* n_victims, cudaStream_t stream) {
  (void)ctx;
  if (n_lanes <= 0) return cudaSuccess;
  if (key_dtype == KVEVICT_KEY_F64)
    return stride >= kSelWideFrom
               ? launch_sel<double, kSelClusterWide>(n_lanes, stream, static_cast<const double*>(keys), positions,
                                                     counts, stride, budget, recent, victims, n_victims)
               : launch_sel<double, kSelCluster>(n_lanes, stream, static_cast<const double*>(keys), positions, counts,
                                                 stride, budget, recent, victims, n_victims);
  return stride >= kSelWideFrom
             ? launch_sel<float, kSelClusterWide>(n_lanes, stream, static_cast<const float*>(keys), positions, counts,
                                                  stride, budget, recent, victims, n_victims)
             : launch_sel<float, kSelCluster>(n_lanes, stream, static_cast<const float*>(keys), positions, counts,
                                              stride, budget, recent, victims, n_victims);
}

// gated: plan only lanes whose Eq. (1) waste ratio exceeds theta_f (the
// relocation a decode step would have run); otherwise every lane whose plan
// frees blocks (forced).
cudaError_t launch_compact(const Ctx& ctx, const Workspace& ws, int layer, const int32_t* victims,
                           const int32_t* n_victims, bool gated, int32_t* freed, int32_t* n_freed,
                           int32_t* moves, int32_t* n_moves, cudaStream_t stream) {
  LayerState ls = layer_state(ctx, layer);
  {
    const int cpl = cmp_ctas_per_lane(ctx.dims);
    const dim3 grid(cpl, ctx.dims.lanes);
    compact_remove_kernel<<<grid, kCmpThreads, 0, stream>>>(ls, ws, ctx.dims, victims, n_victims, cpl);
    compact_place_kernel<<<grid, kCmpThreads, 0, stream>>>(ls, ws, ctx.dims, cpl);
    compact_blocks_kernel<<<ctx.dims.lanes, 1024, 0, stream>>>(ls, ws, ctx.dims, cpl, gated ? 1 : 0);
  }
  cudaError_t e = launch_allocate(ctx, ws, layer, stream);
  if (e != cudaSuccess) return e;
  {
    const int cpl = cmp_ctas_per_lane(ctx.dims);
    const dim3 grid(cpl, ctx.dims.lanes);
    compact_reloc_count_kernel<<<grid, kCmpThreads, 0, stream>>>(ls, ws, ctx.dims, cpl);
    if (ctx.dims.dtype == KVEVICT_BF16)
      compact_reloc_move_kernel<__nv_bfloat16><<<grid, kCmpThreads, 0, stream>>>(ls, ws, ctx.dims, cpl, moves);
    else
      compact_reloc_move_kernel<float><<<grid, kCmpThreads, 0, stream>>>(ls, ws, ctx.dims, cpl, moves);
    compact_reloc_finish_kernel<<<ctx.dims.lanes, 1024, 0, stream>>>(ls, ws, ctx.dims, cpl);
  }
  const int chunks = (ctx.dims.P + kFreedChunk - 1) / kFreedChunk;
  const int ranges = chunks < kFreedRanges ? chunks : kFreedRanges;
  const int span = (chunks + ranges - 1) / ranges * kFreedChunk;
  freed_count_kernel<<<ranges, 1024, 0, stream>>>(ws, ctx.dims, span);
  freed_write_kernel<<<ranges, 1024, 0, stream>>>(ws, ctx.dims, span, freed, n_freed, n_moves);
  return cudaGetLastError();
}

cudaError_t launch_stats(const Ctx& ctx, int layer, long long* out, cudaStream_t stream) {
  LayerState ls = layer_state(ctx, layer);
  stats_kernel<<<1, 1024, 0, stream>>>(ls, ctx.dims, out);
  return cudaGetLastError();
}

cudaError_t launch_decode(Ctx& ctx, int layer, const void* q, const void* k_new, const void* v_new,
                          int new_pos, float* out, float* lse, int32_t* victims, int32_t* n_victims,
                          cudaStream_t stream) {
  cudaError_t e;
  if (q) {
    e = launch_attend(ctx, layer, q, k_new, v_new, stream, true);
    if (e != cudaSuccess) return e;
    note_attend(ctx, layer);
  }
  bool apply_kernel = false;
  e = launch_epilogue(ctx, layer, q != nullptr, new_pos, k_new, v_new, out, lse, victims, n_victims, stream,
                      &apply_kernel);
  if (e != cudaSuccess) return e;
  note_epilogue(ctx, layer);
  // every lane of the layer is now within its budget
  ctx.layer_steady[layer] = true;
  if (!apply_kernel) return e;
  e = launch_allocate_apply(ctx, layer, k_new, v_new, false, nullptr, stream, false);
  note_apply(ctx);
  return e;
}

}  // namespace kve
