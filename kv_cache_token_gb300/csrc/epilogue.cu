// Decode-step epilogue (one CTA per lane) and the layer allocator.
//
// epilogue: combines the split-K partials into the lane's log-sum-exp and
// output; turns every kept token's logits into its group weight
// w_j = sum_h exp(s_hj - LSE_h) and writes it straight into the policy's
// score state (H2O: S_j += w_j; SnapKV: history[j][slot] = w_j); builds the
// eviction keys (SnapKV: float64 window sums in slot order 0 upward, then a
// warp-shuffle sliding max over kept neighbours, clamped); selects the
// budgeted bottom-k outside the recent window (radix descent on (key,
// position)); removes the victims from the token table in place; admits the
// new token into the lowest free slot of the lane's blocks; and sizes the
// lane's relocation plan.
// allocate: one CTA hands out the lowest free block ids, ascending lanes,
// first to admissions that found no slot, then to relocation destinations.
// apply: one CTA per lane writes those admissions and runs the relocation
// (vToken review, Sec. 3.3 Stage 3: fill each destination completely, in
// ascending position, and release the sources).
#include "lane_ops.cuh"

namespace kve {
namespace {

constexpr int kEpiThreads = 512;
constexpr int kFastPer = 7;     // tokens per thread on the one-victim H2O path
constexpr int kFastN = kFastPer * kEpiThreads;   // tokens a lane may hold on that path
constexpr int kPoSeg = 16;      // split-K partial outputs staged in shared memory on that path
constexpr int kWorkShift = 16;  // done counter: arrivals below, lanes asking for blocks above
constexpr int kWorkUnit = 1 << kWorkShift;
// dynamic shared memory of the epilogue: the fast path's logits [8][kFastN]
// and partial outputs [kPoSeg][8][128]; the general path's row buffer
constexpr size_t kEpiDynSmem = (static_cast<size_t>(8) * kFastN + static_cast<size_t>(kPoSeg) * 8 * 128) * 4;
static_assert(kEpiDynSmem >= static_cast<size_t>(128) * kMaxW * 4, "row buffer fits");
constexpr int kApplyThreads = 512;
constexpr int kCopyBatch = 8;   // relocation: 16-byte loads in flight per thread
constexpr float kLn2 = 0.6931471805599453f;

struct EpiArgs {
  LayerState ls;
  Workspace ws;
  Dims dm;
  int has_q, new_pos, layer;
  const void* k_new; const void* v_new;
  float* out; float* lse; int32_t* victims; int32_t* n_victims;
};

template <typename KT>
__device__ __forceinline__ void copy_row(KT* dst, const KT* src, int d) {
  for (int e = threadIdx.x; e < d; e += blockDim.x) dst[e] = src[e];
}

template <typename KT>
__device__ __forceinline__ void lane_step(const EpiArgs& A, const LaneRefs& L, const int n, unsigned char* dsm,
                                          int* sh_work);
__device__ void allocate_layer(const LayerState& ls, const Workspace& ws, const Dims& dm, int* sh_scan,
                               int* sh_flag);

// 2^x by the hardware approximation (PTX ex2.approx.ftz, relative error
// about 2^-22; results below 2^-126 flush to zero).
__device__ __forceinline__ float hw_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// DropKV decode variant: this step's residual-output score of one kept
// token, sum over the group's heads h of p / (1 - p) * ||a_h - v|| (DropKV
// explainer, Lemma 1, with the window reduced to the current query of each
// head).  a [g][d] are the heads' outputs (shared memory), v the token's V
// row; the distance is taken directly in fp32 (no expansion, so no
// cancellation when a_h is close to v), 1 - p from expm1 when p > 1/2, and
// the term is +inf where 1 - p <= 0.  lg: the token's base-2 scaled logits,
// one per head, lcap apart.  Out of line, so the token loop that SnapKV and
// H2O run stays small.
template <typename KT>
__device__ __noinline__ float dropkv_step_score(const float* a, const KT* v, int g, int d, const float* lg,
                                                   int lcap, const float* lse2) {
  float dist[kMaxG];
#pragma unroll
  for (int h = 0; h < kMaxG; ++h) dist[h] = 0.f;
  constexpr int kPer = 16 / static_cast<int>(sizeof(KT));    // elements per 16-byte load
  for (int e0 = 0; e0 < d; e0 += kPer) {
    const uint4 raw = *reinterpret_cast<const uint4*>(v + e0);
    const KT* pv = reinterpret_cast<const KT*>(&raw);
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const float x = static_cast<float>(pv[u]);
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) {
        if (h < g) {
          const float df = a[h * d + e0 + u] - x;
          dist[h] = fmaf(df, df, dist[h]);
        }
      }
    }
  }
  float sc = 0.f;
#pragma unroll
  for (int h = 0; h < kMaxG; ++h) {
    if (h < g) {
      const float x = lg[static_cast<size_t>(h) * lcap] - lse2[h];
      const float p = exp2f(x);
      if (p > 0.f) {
        const float om = p > 0.5f ? -expm1f(x * kLn2) : 1.f - p;
        sc += om > 0.f ? p / om * sqrtf(dist[h]) : INFINITY;
      }
    }
  }
  return sc;
}

// Marks this lane's epilogue done (thread 0 only).  The per-lane requests
// the allocator reads (need_admit, want_dst, plan_tlive, count, released
// block owners) are written before (by any thread of the CTA, ordered by a
// barrier before this call); the release makes them visible to the last CTA.  The done counter carries the number of lanes asking for blocks
// in its upper bits, so the common no-work case needs no further atomic.
__device__ __forceinline__ void signal_done(const Workspace& ws, bool work, int* sh_last, int* sh_flag) {
  const int old = atomic_add_release(ws.epi_done, 1 + (work ? kWorkUnit : 0));
  *sh_last = (old & (kWorkUnit - 1)) == static_cast<int>(gridDim.x) - 1;
  *sh_flag = (old >> kWorkShift) + (work ? 1 : 0);
}

// H2O with at most one victim (the steady state of a full cache), all
// threads of the CTA.  Before the dependency wait: the lane's token table
// (kFastPer tokens a thread), its block list with the live masks (kFastPer
// blocks a thread) and the new token's K/V row, none of which the attention
// kernel writes; from the masks, each warp's lowest free slot.  After it:
// logits and split-K partial outputs by bulk copy into shared memory,
// split-K statistics by plain loads.  The minimum (key, position) and its
// slot come from three warp reductions and one barrier; the holder of the
// victim's block decides from the mask it already holds whether the block
// empties.  The fragmentation test of Eq. (1) is evaluated before the wait
// for each of the eight outcomes the scoring can have (double division is
// slow on this part).  The allocator's requests and the done counter go out
// before the table is rewritten, so the counter's release does not wait for
// those stores, and the counter's old value is read only at the end.
template <typename KT>
__device__ __forceinline__ void h2o_fast_step(const EpiArgs& A, const LaneRefs& L, const int n, unsigned char* dsm,
                                              int* sh_sig, int* sh_last, int* sh_flag) {
  __shared__ float sh_rL[8], sh_lse2[8];
  __shared__ __align__(16) float sh_scale[8][kMaxSeg];   // per head, per split-K segment
  __shared__ unsigned sh_over;
  __shared__ unsigned sh_wkey[kEpiThreads / 32], sh_wpos[kEpiThreads / 32], sh_wslot[kEpiThreads / 32];
  __shared__ unsigned sh_wfree[kEpiThreads / 32];
  __shared__ int sh_nan, sh_dead, sh_tail;
  __shared__ int sh_scan2[40];
  __shared__ uint64_t sh_bar;
  constexpr unsigned kNone = 0xFFFFFFFFu;
  const Dims& dm = A.dm;
  const int l = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = l / dm.Hkv, kh = l % dm.Hkv, g = dm.g, d = dm.d;
  const int cbuf = A.layer & 1;
  const int k = max(0, n + 1 - dm.budget);          // 0 or 1
  const int cut = A.new_pos - dm.R + 1;

  // ---- before the dependency wait -----------------------------------------------
  float sc[kFastPer];
  int ps[kFastPer], sl[kFastPer];
#pragma unroll
  for (int j = 0; j < kFastPer; ++j) {
    const int i = tid + j * kEpiThreads;
    const bool ok = i < n;
    sc[j] = ok ? __ldcg(L.score + i) : 0.f;
    ps[j] = ok ? __ldcg(L.pos + i) : 0x7FFFFFFF;
    sl[j] = ok ? __ldcg(L.slot + i) : -1;
  }
  KT knv{}, vnv{};
  if (tid < d) {
    knv = static_cast<const KT*>(A.k_new)[static_cast<size_t>(l) * d + tid];
    vnv = static_cast<const KT*>(A.v_new)[static_cast<size_t>(l) * d + tid];
  }
  const int nb = min(__ldcg(L.nblocks), kFastN);   // every block holds a live token, so nb <= n
  int bk[kFastPer], bm[kFastPer];
#pragma unroll
  for (int j = 0; j < kFastPer; ++j) {
    const int jj = tid + j * kEpiThreads;
    bk[j] = jj < nb ? __ldcg(L.blocks + jj) : -1;
  }
  bool bad_blk = false;
#pragma unroll
  for (int j = 0; j < kFastPer; ++j) {
    if (bk[j] >= dm.P) { bad_blk = true; bk[j] = -1; }
    bm[j] = bk[j] >= 0 ? (__ldcg(L.mask + bk[j]) & 0xFFFF) : 0xFFFF;
  }
  if (bad_blk) set_status(A.ws.status, ST_BAD_INDEX);
  // a request of this lane left non-zero (the invariant is that none is)
  const bool stale_req = tid == 0 && (__ldcg(A.ws.need_admit + l) | __ldcg(A.ws.want_dst + l)) != 0;
  if (tid == 0) {
    sh_nan = 0;
    sh_dead = -1;
    mbar_init(&sh_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  {
    // lowest free slot of the lane's blocks before this step's eviction
    unsigned fr = kNone;
#pragma unroll
    for (int j = 0; j < kFastPer; ++j)
      if (bk[j] >= 0 && bm[j] != 0xFFFF) fr = min(fr, static_cast<unsigned>(bk[j] * kBlock + (__ffs(~bm[j]) - 1)));
    fr = __reduce_min_sync(0xffffffffu, fr);
    if (lane == 0) sh_wfree[warp] = fr;
  }
  // Eq. (1)'s test for each outcome the scoring has yet to decide: a victim
  // or none (bit 0), its block emptied or not (bit 1), the new token waiting
  // for a fresh block or not (bit 2); one lane per outcome
  if (warp == 0) {
    const int vc = lane & 1, dead = (lane >> 1) & 1, fresh = (lane >> 2) & 1;
    const int N = nb - dead + fresh;
    const bool o = lane < 8 && N > 0 && frag_over(n - vc + 1, N, dm.theta_f);
    const unsigned bits = __ballot_sync(0xffffffffu, o);
    if (lane == 0) sh_over = bits;
  }
  // the last kept token must precede the new one
  bool late = false;
#pragma unroll
  for (int j = 0; j < kFastPer; ++j) late |= (tid + j * kEpiThreads == n - 1) && ps[j] >= A.new_pos;

  grid_dep_wait();      // the attention kernel's results are complete and visible
  grid_dep_launch();

  // split-K statistics of all kMaxSeg segments (in bounds), masked below
  const float2* ml = reinterpret_cast<const float2*>(A.ws.part_ml_buf[cbuf]) + static_cast<size_t>(l) * kMaxSeg * g;
  float2 m0 = make_float2(-INFINITY, 0.f), m1 = make_float2(-INFINITY, 0.f);
  if (A.has_q && warp < g) {
    m0 = __ldcg(ml + lane * g + warp);
    m1 = __ldcg(ml + (lane + 32) * g + warp);
  }
  const int nseg = A.has_q ? min(__ldcg(A.ws.lane_nseg_buf[cbuf] + l), kMaxSeg) : 0;
  if (__syncthreads_or(late)) {
    if (tid == 0) {
      set_status(A.ws.status, ST_POSITION);
      A.n_victims[l] = 0; A.ws.need_admit[l] = 0; A.ws.want_dst[l] = 0; A.ws.plan_tlive[l] = 0;
    }
    return;
  }
  float* lg_s = reinterpret_cast<float*>(dsm);                 // [g][kFastN]
  float* po_s = lg_s + 8 * kFastN;                             // [kPoSeg][g][d]
  const float* po = A.ws.part_o_buf[cbuf] + static_cast<size_t>(l) * kMaxSeg * g * d;
  if (A.has_q && tid == 0) {
    const float* lg = A.ws.logits_buf[cbuf] + static_cast<size_t>(l) * g * dm.lcap;
    const uint32_t row = static_cast<uint32_t>((n + 3) & ~3) * 4u;   // 16-byte multiple, inside lcap
    const uint32_t pob = static_cast<uint32_t>(kPoSeg * g * d) * 4u;
    mbar_arrive_expect_tx(&sh_bar, row * g + pob);
    if (row)
      for (int h = 0; h < g; ++h) bulk_g2s(lg_s + h * kFastN, lg + static_cast<size_t>(h) * dm.lcap, row, &sh_bar);
    bulk_g2s(po_s, po, pob, &sh_bar);
  }
  // per-head log-sum-exp of the split-K segments (one warp per head)
  if (A.has_q && warp < g) {
    const int h = warp;
    if (lane >= nseg) m0 = make_float2(-INFINITY, 0.f);
    if (lane + 32 >= nseg) m1 = make_float2(-INFINITY, 0.f);
    const float M = warp_max(fmaxf(m0.x, m1.x));
    const float s0 = m0.x == -INFINITY ? 0.f : exp2f(m0.x - M);
    const float s1 = m1.x == -INFINITY ? 0.f : exp2f(m1.x - M);
    sh_scale[h][lane] = s0;
    sh_scale[h][lane + 32] = s1;
    float Ls = m0.y * s0 + m1.y * s1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
    if (lane == 0) {
      sh_rL[h] = 1.f / Ls;
      const float lse2 = M + log2f(Ls);
      sh_lse2[h] = lse2;
      A.lse[static_cast<size_t>(b) * dm.Hq + kh * g + h] = lse2 * kLn2;
    }
  }
  __syncthreads();
  unsigned pre_free = lane < kEpiThreads / 32 ? sh_wfree[lane] : kNone;
  pre_free = __reduce_min_sync(0xffffffffu, pre_free);
  if (A.has_q && !mbar_wait_bounded(&sh_bar, 0, A.ws.status)) (void)mbar_wait_bounded(&sh_bar, 0, A.ws.status);

  // ---- weights -> scores; candidate minimum (key, position) -------------------------
  if (A.has_q) {
    float w[kFastPer];
#pragma unroll
    for (int j = 0; j < kFastPer; ++j) w[j] = 0.f;
    if (g == 8) {
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float lse2 = sh_lse2[h];
        const float* row = lg_s + h * kFastN + tid;
#pragma unroll
        for (int j = 0; j < kFastPer; ++j) w[j] += hw_exp2(row[j * kEpiThreads] - lse2);
      }
    } else {
      for (int h = 0; h < g; ++h) {
        const float lse2 = sh_lse2[h];
        const float* row = lg_s + h * kFastN + tid;
#pragma unroll
        for (int j = 0; j < kFastPer; ++j) w[j] += hw_exp2(row[j * kEpiThreads] - lse2);
      }
    }
#pragma unroll
    for (int j = 0; j < kFastPer; ++j) sc[j] += w[j];
  }
  unsigned ck = kNone, cp = kNone;
  int cs = -1, nan_count = 0;
#pragma unroll
  for (int j = 0; j < kFastPer; ++j) {
    const int i = tid + j * kEpiThreads;
    if (i < n) {
      if (sc[j] != sc[j]) ++nan_count;
      if (k == 1 && ps[j] < cut) {
        const unsigned kk = static_cast<unsigned>(mono_key(sc[j]));
        const unsigned pp = static_cast<unsigned>(ps[j]);
        if (kk < ck || (kk == ck && pp < cp)) { ck = kk; cp = pp; cs = sl[j]; }
      }
    }
  }
  {
    const unsigned wk = __reduce_min_sync(0xffffffffu, ck);
    const unsigned wp = __reduce_min_sync(0xffffffffu, ck == wk ? cp : kNone);
    const unsigned ws = __reduce_min_sync(0xffffffffu, (ck == wk && cp == wp) ? static_cast<unsigned>(cs) : kNone);
    if (lane == 0) { sh_wkey[warp] = wk; sh_wpos[warp] = wp; sh_wslot[warp] = ws; }
  }
  if (nan_count) atomicAdd(&sh_nan, nan_count);
  __syncthreads();
  unsigned vkey, vpos, vslot_u;
  {
    const bool in = lane < kEpiThreads / 32;
    const unsigned k1 = in ? sh_wkey[lane] : kNone, p1 = in ? sh_wpos[lane] : kNone;
    const unsigned s1 = in ? sh_wslot[lane] : kNone;
    vkey = __reduce_min_sync(0xffffffffu, k1);
    vpos = __reduce_min_sync(0xffffffffu, k1 == vkey ? p1 : kNone);
    vslot_u = __reduce_min_sync(0xffffffffu, (k1 == vkey && p1 == vpos) ? s1 : kNone);
  }
  const bool has_victim = k == 1 && vpos != kNone;   // positions are below 2^31
  const int vslot = static_cast<int>(vslot_u);
  const int vcount = has_victim ? 1 : 0;
  // ---- eviction: the victim's slot is released; an emptied block is freed ---------
  bool vslot_ok = false;
  if (has_victim) {
    if (vslot >= 0 && vslot < dm.P * kBlock) {
      vslot_ok = true;
      const int vb = vslot >> 4, vbit = 1 << (vslot & 15);
#pragma unroll
      for (int j = 0; j < kFastPer; ++j) {
        if (bk[j] == vb) {
          atomicAnd(&L.mask[vb], ~vbit);
          if ((bm[j] & ~vbit) == 0) {
            L.owner[vb] = -1;
            sh_dead = tid + j * kEpiThreads;     // index of the block in the lane's list
          }
        }
      }
    } else if (vslot >= 0 && tid == 0) {
      set_status(A.ws.status, ST_BAD_INDEX);
    }
  }
  __syncthreads();
  const int dead_j = sh_dead;
  int nb2 = nb;
  unsigned best;
  if (dead_j < 0) {
    // the victim's slot is now free too
    best = min(pre_free, vslot_ok ? static_cast<unsigned>(vslot) : kNone);
  } else {
    // rare: the victim emptied its block; drop it from the list (the last
    // entry moves into its place) and look for a free slot in the others
    const int vb = vslot >> 4;
    if (tid == 0) sh_tail = __ldcg(L.blocks + nb - 1);
    unsigned fr = kNone;
#pragma unroll
    for (int j = 0; j < kFastPer; ++j)
      if (bk[j] >= 0 && bk[j] != vb && bm[j] != 0xFFFF)
        fr = min(fr, static_cast<unsigned>(bk[j] * kBlock + (__ffs(~bm[j]) - 1)));
    fr = __reduce_min_sync(0xffffffffu, fr);
    if (lane == 0) sh_wfree[warp] = fr;
    __syncthreads();
    if (tid == 0) {
      L.blocks[dead_j] = sh_tail;
      *L.nblocks = nb - 1;
    }
    best = lane < kEpiThreads / 32 ? sh_wfree[lane] : kNone;
    best = __reduce_min_sync(0xffffffffu, best);
    nb2 = nb - 1;
    __syncthreads();
  }
  const bool need = best == kNone;
  const int m = n - vcount;
  // ---- admission into the lowest free slot; relocation plan --------------------------
  if (!need && tid == 0) atomicOr(&L.mask[best >> 4], 1 << (best & 15));
  __syncthreads();
  int t_live = 0;
  const int outcome = vcount | (dead_j >= 0 ? 2 : 0) | (need ? 4 : 0);
  const int ndst = lane_plan_given(L, nb2, ((sh_over >> outcome) & 1u) != 0, false, need, &t_live, sh_scan2);
  const bool work = need || ndst > 0;
  // the done counter's old value is only needed at the end: its round trip
  // overlaps the table rewrite and the output combine
  int done_old = 0;
  if (tid == 0) {
    A.ls.count[l] = m + 1;
    if (m + 1 >= dm.cap) set_status(A.ws.status, ST_CAPACITY);
    // The allocator reads a lane's requests (and its count) only when they
    // are non-zero; between steps they hold zero (the apply kernel clears
    // what it consumed).  A lane that asks for blocks, released a block or
    // clears a request left over publishes with release semantics; the
    // writes of the others are of no concern to the allocator.
    const bool publish = work || dead_j >= 0 || stale_req;
    if (work || stale_req) {
      A.ws.need_admit[l] = need ? 1 : 0;
      A.ws.want_dst[l] = ndst;
      A.ws.plan_tlive[l] = t_live;
    }
    if (work) atomicOr(A.ws.work_flag, 1);
    const int inc = 1 + (work ? kWorkUnit : 0);
    done_old = publish ? atomic_add_release(A.ws.epi_done, inc) : atomicAdd(A.ws.epi_done, inc);
  }
  // ---- the table: survivors shift over the victim; the new token goes last -----------
#pragma unroll
  for (int j = 0; j < kFastPer; ++j) {
    const int i = tid + j * kEpiThreads;
    if (i < n) {
      const unsigned pp = static_cast<unsigned>(ps[j]);
      if (has_victim && pp == vpos) {
        A.victims[static_cast<size_t>(l) * dm.cap] = ps[j];
      } else {
        const int ni = (has_victim && pp > vpos) ? i - 1 : i;
        if (ni != i) {
          L.pos[ni] = ps[j];
          L.slot[ni] = sl[j];
        }
        L.score[ni] = sc[j];
      }
    }
  }
  if (!need && tid < d) {
    static_cast<KT*>(A.ls.k_pool)[static_cast<size_t>(best) * d + tid] = knv;
    static_cast<KT*>(A.ls.v_pool)[static_cast<size_t>(best) * d + tid] = vnv;
  }
  if (tid == 0) {
    L.pos[m] = A.new_pos;
    L.slot[m] = need ? -1 : static_cast<int>(best);
    L.score[m] = 0.f;
    A.n_victims[l] = vcount;
    if (vcount) atomicAdd(reinterpret_cast<unsigned long long*>(&A.ls.stats[SC_VICTIMS]), 1ull);
    if (dead_j >= 0) atomicAdd(reinterpret_cast<unsigned long long*>(&A.ls.stats[SC_FREED_DEAD]), 1ull);
    if (sh_nan) atomicAdd(reinterpret_cast<unsigned long long*>(&A.ls.stats[SC_NAN_KEYS]), (unsigned long long)sh_nan);
    if (l == 0) atomicAdd(reinterpret_cast<unsigned long long*>(&A.ls.stats[SC_STEPS]), 1ull);
  }
  // ---- output: combine the split-K partial outputs (the first kPoSeg from
  // shared memory); a thread owns two adjacent elements of one head, so the
  // segment scales are warp-uniform and read four at a time -------------------------
  if (A.has_q) {
    const int ns = min(nseg, kPoSeg);
    const bool out8 = (reinterpret_cast<uintptr_t>(A.out) & 7) == 0;
    for (int q2 = tid; q2 < (g * d) >> 1; q2 += kEpiThreads) {
      const int he = q2 * 2, h = he / d, e = he - h * d;
      const float4* sc4 = reinterpret_cast<const float4*>(sh_scale[h]);
      float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int s4 = 0; s4 < kPoSeg / 4; ++s4) {
        const float4 c4 = sc4[s4];
        const float cs[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int s2 = s4 * 4 + u;
          if (s2 < ns) {
            const float2 pv = *reinterpret_cast<const float2*>(po_s + (s2 * g + h) * d + e);
            float2& a = (u & 1) ? a1 : a0;
            a.x = fmaf(pv.x, cs[u], a.x);
            a.y = fmaf(pv.y, cs[u], a.y);
          }
        }
      }
      for (int s2 = kPoSeg; s2 < nseg; ++s2) {
        const float2 pv = __ldcg(reinterpret_cast<const float2*>(po + (static_cast<size_t>(s2) * g + h) * d + e));
        a0.x = fmaf(pv.x, sh_scale[h][s2], a0.x);
        a0.y = fmaf(pv.y, sh_scale[h][s2], a0.y);
      }
      const float r = sh_rL[h];
      float* o = A.out + (static_cast<size_t>(b) * dm.Hq + kh * g + h) * d + e;
      if (out8) {
        *reinterpret_cast<float2*>(o) = make_float2((a0.x + a1.x) * r, (a0.y + a1.y) * r);
      } else {
        o[0] = (a0.x + a1.x) * r;
        o[1] = (a0.y + a1.y) * r;
      }
    }
  }
  if (tid == 0) {
    *sh_last = (done_old & (kWorkUnit - 1)) == static_cast<int>(gridDim.x) - 1;
    *sh_flag = (done_old >> kWorkShift) + (work ? 1 : 0);
    *sh_sig = 1;
  }
}

template <typename KT>
__global__ void __launch_bounds__(kEpiThreads, 1) decode_epilogue_kernel(EpiArgs A) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ int sh_scan[40];
  __shared__ int sh_work, sh_last, sh_flag, sh_sig;
  const Dims& dm = A.dm;
  const int l = blockIdx.x, tid = threadIdx.x;
  LaneRefs L = lane_refs(A.ls, dm, l);
  // The token count (and, on the fast path, the token table and the block
  // list) is not written by the attention kernel: it is read before the
  // dependency wait, while the attention kernel drains.
  const int n = __ldcg(A.ls.count + l);
  if (tid == 0) { sh_work = 0; sh_sig = 0; }
  if (n < 0 || n >= dm.cap) {
    grid_dep_wait();
    grid_dep_launch();
    if (tid == 0) {
      set_status(A.ws.status, ST_CAPACITY);
      A.n_victims[l] = 0; A.ws.need_admit[l] = 0; A.ws.want_dst[l] = 0; A.ws.plan_tlive[l] = 0;
    }
  } else if (dm.policy == KVEVICT_H2O && n + 1 - dm.budget <= 1 && n <= kFastN && dm.g <= 8 && dm.d <= 128 &&
             (dm.d & 1) == 0) {
    h2o_fast_step<KT>(A, L, n, dsm, &sh_sig, &sh_last, &sh_flag);
  } else {
    lane_step<KT>(A, L, n, dsm, &sh_work);
  }
  __syncthreads();
  if (!sh_sig) {
    if (tid == 0) signal_done(A.ws, sh_work != 0, &sh_last, &sh_flag);
    __syncthreads();
  }
  // The last CTA of the grid to finish runs the layer allocator, if any lane
  // asked for blocks.
  if (sh_last) {
    if (sh_flag == 0) {
      if (tid == 0) { *A.ws.epi_done = 0; A.ws.counters[1] = 0; A.ws.counters[2] = 0; }
    } else {
      if (tid == 0) *A.ws.epi_done = 0;
      __threadfence();
      allocate_layer(A.ls, A.ws, dm, sh_scan, &sh_flag);
    }
  }
}

// One lane's step after the attention kernel (all threads of the CTA).
template <typename KT>
__device__ __forceinline__ void lane_step(const EpiArgs& A, const LaneRefs& L, const int n, unsigned char* dsm,
                                          int* sh_work) {
  __shared__ float sh_M[kMaxG], sh_L[kMaxG], sh_lse2[kMaxG];
  __shared__ __align__(16) int sh_hist[256];   // also read as 64-bit words
  __shared__ int sh_misc[40];
  __shared__ int sh_scan[40];
  __shared__ int sh_idx[kEpiThreads];
  __shared__ unsigned sh_min[32];
  __shared__ int sh_nan;
  __shared__ float sh_scale[kMaxSeg][kMaxG];
  float* sh_rows = reinterpret_cast<float*>(dsm);      // general path: 128 * kMaxW floats
  const Dims& dm = A.dm;
  const int l = blockIdx.x, tid = threadIdx.x;
  const int b = l / dm.Hkv, kh = l % dm.Hkv, g = dm.g, d = dm.d;
  const int cbuf = A.layer & 1;

  // ---- general path ------------------------------------------------------------
  grid_dep_wait();      // the attention kernel's results are complete and visible
  grid_dep_launch();
  if (tid == 0) sh_nan = 0;
  if (n > 0 && L.pos[n - 1] >= A.new_pos) {
    if (tid == 0) {
      set_status(A.ws.status, ST_POSITION);
      A.n_victims[l] = 0; A.ws.need_admit[l] = 0; A.ws.want_dst[l] = 0; A.ws.plan_tlive[l] = 0;
    }
    return;
  }

  // ---- combine the split-K partials --------------------------------------
  if (A.has_q) {
    const int nseg = min(A.ws.lane_nseg_buf[cbuf][l], kMaxSeg);
    const float2* ml = reinterpret_cast<const float2*>(A.ws.part_ml_buf[cbuf]) + static_cast<size_t>(l) * kMaxSeg * g;
    const int warp = tid >> 5, lane = tid & 31;
    if (warp < g) {
      // one warp per head; lanes hold segments lane and lane + 32
      const int h = warp;
      const float2 v0 = lane < nseg ? ml[lane * g + h] : make_float2(-INFINITY, 0.f);
      const float2 v1 = lane + 32 < nseg ? ml[(lane + 32) * g + h] : make_float2(-INFINITY, 0.f);
      const float M = warp_max(fmaxf(v0.x, v1.x));
      const float s0 = v0.x == -INFINITY ? 0.f : exp2f(v0.x - M);
      const float s1 = v1.x == -INFINITY ? 0.f : exp2f(v1.x - M);
      if (lane < nseg) sh_scale[lane][h] = s0;
      if (lane + 32 < nseg) sh_scale[lane + 32][h] = s1;
      float Ls = v0.y * s0 + v1.y * s1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
      if (lane == 0) {
        sh_M[h] = M;
        sh_L[h] = Ls;
        const float lse2 = M + log2f(Ls);
        sh_lse2[h] = lse2;
        A.lse[static_cast<size_t>(b) * dm.Hq + kh * g + h] = lse2 * kLn2;
      }
    }
    __syncthreads();
    const float* po = A.ws.part_o_buf[cbuf] + static_cast<size_t>(l) * kMaxSeg * g * d;
    for (int he = tid; he < g * d; he += blockDim.x) {
      const int h = he / d, e = he - h * d;
      float acc = 0.f;
#pragma unroll 8
      for (int s = 0; s < nseg; ++s) acc = fmaf(po[(static_cast<size_t>(s) * g + h) * d + e], sh_scale[s][h], acc);
      const float o = acc / sh_L[h];
      A.out[(static_cast<size_t>(b) * dm.Hq + kh * g + h) * d + e] = o;
      sh_rows[he] = o;    // the heads' outputs, for the DropKV scores below
    }
    __syncthreads();
  }

  // ---- weights -> score state; SnapKV window sums ----------------------------
  const int policy = dm.policy;
  const bool ringp = policy != KVEVICT_H2O;   // SnapKV, DropKV decode variant: history ring keys
  const int W = dm.W;
  const int rs = ringp ? A.ls.ring_slot[l] : 0;
  double* keys64 = A.ws.keys64 ? A.ws.keys64 + static_cast<size_t>(l) * dm.cap : nullptr;
  double* pooled64 = A.ws.pooled64 ? A.ws.pooled64 + static_cast<size_t>(l) * dm.cap : nullptr;
  const float* lg = A.ws.logits_buf[cbuf] + static_cast<size_t>(l) * g * dm.lcap;
  const int k = max(0, n + 1 - dm.budget);
  const int cut = A.new_pos - dm.R + 1;
  // k == 1 (a full cache in steady state): the minimum candidate (key,
  // position) is tracked in the same pass that produces the keys.
  unsigned long long best_k = ~0ull;
  uint32_t best_p = 0xFFFFFFFFu;
  int best_i = -1;
  int nan_count = 0;
  for (int i = tid; i < n; i += blockDim.x) {
    float w = 0.f;
    if (A.has_q) {
      if (policy == KVEVICT_DROPKV) {
        const int s = L.slot[i];
        if (s >= 0 && s < dm.P * kBlock) {
          w = dropkv_step_score<KT>(sh_rows, static_cast<const KT*>(A.ls.v_pool) + static_cast<size_t>(s) * d, g, d,
                                    lg + i, dm.lcap, sh_lse2);
        } else {
          set_status(A.ws.status, ST_BAD_INDEX);
        }
      } else {
        for (int h = 0; h < g; ++h) w += exp2f(lg[static_cast<size_t>(h) * dm.lcap + i] - sh_lse2[h]);
      }
    }
    if (ringp) {
      float* row = L.ring + static_cast<size_t>(i) * W;
      if (A.has_q) row[rs] = w;
      double sum = 0.0;
      for (int t = 0; t < W; ++t) sum += static_cast<double>((A.has_q && t == rs) ? w : row[t]);
      keys64[i] = sum;
      if (sum != sum) ++nan_count;
    } else {
      float sc = L.score[i];
      if (A.has_q) {
        sc += w;
        L.score[i] = sc;
      }
      if (sc != sc) ++nan_count;
      if (k == 1) {
        const int p = L.pos[i];
        const unsigned long long kk = mono_key(sc);
        if (p < cut && (kk < best_k || (kk == best_k && static_cast<uint32_t>(p) < best_p))) {
          best_k = kk; best_p = static_cast<uint32_t>(p); best_i = i;
        }
      }
    }
  }
  if (ringp && tid == 0) keys64[n] = 0.0;
  __syncthreads();
  if (ringp) {
    if (A.has_q && tid == 0) A.ls.ring_slot[l] = (rs + 1) % W;
    // sliding max over kept neighbours [i-r, i+r], clamped to [0, n]
    const int r = (dm.pool_kernel - 1) / 2;
    const int span = 32 - 2 * r;
    const int lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const int nn = n + 1;
    for (int base = warp * span; base < nn; base += nwarps * span) {
      const int idx = base - r + lane;
      const double v = (idx >= 0 && idx < nn) ? keys64[idx] : -INFINITY;
      double m = v;
      for (int o = 1; o <= r; ++o) {
        m = fmax(m, __shfl_down_sync(0xffffffffu, v, o));
        m = fmax(m, __shfl_up_sync(0xffffffffu, v, o));
      }
      if (lane >= r && lane < 32 - r && idx >= 0 && idx < nn) {
        pooled64[idx] = m;
        if (k == 1 && idx < n) {
          const int p = L.pos[idx];
          const unsigned long long kk = mono_key(m);
          if (p < cut && (kk < best_k || (kk == best_k && static_cast<uint32_t>(p) < best_p))) {
            best_k = kk; best_p = static_cast<uint32_t>(p); best_i = idx;
          }
        }
      }
    }
    __syncthreads();
  }

  // ---- bottom-k selection and eviction ------------------------------------------
  auto candf = [&](int i) { return L.pos[i] < cut; };
  auto posf = [&](int i) { return static_cast<uint32_t>(L.pos[i]); };
  int vcount = 0, dead = 0;
  int32_t* vout = A.victims + static_cast<size_t>(l) * dm.cap;
  if (k == 1) {
    const int v = block_argmin3(best_k, best_p, best_i, sh_hist, sh_misc);
    if (v >= 0) {
      vcount = 1;
      dead = lane_remove_one(L, n, v, vout, dm.P, A.ws.status, sh_misc, sh_rows);
    }
  } else if (k > 1) {
    SelectResult sel;
    if (ringp) {
      auto keyf = [&](int i) { return mono_key(pooled64[i]); };
      sel = block_bottom_k(n, k, 64, keyf, posf, candf, sh_hist, sh_misc);
      auto isv = [&](int i) { return candf(i) && select_is_victim(sel, keyf(i), posf(i)); };
      vcount = lane_remove(L, n, plain_victims(isv), vout, nullptr, &dead, dm.P, A.ws.status, sh_scan, sh_idx,
                           sh_rows);
    } else {
      auto keyf = [&](int i) { return mono_key(L.score[i]); };
      sel = block_bottom_k(n, k, 32, keyf, posf, candf, sh_hist, sh_misc);
      auto isv = [&](int i) { return candf(i) && select_is_victim(sel, keyf(i), posf(i)); };
      vcount = lane_remove(L, n, plain_victims(isv), vout, nullptr, &dead, dm.P, A.ws.status, sh_scan, sh_idx,
                           sh_rows);
    }
  }
  const int m = n - vcount;
  const int nb = (k > 1 && dead > 0) ? lane_prune_blocks(L, l, sh_scan) : *L.nblocks;

  // ---- admission: lowest free slot among the lane's blocks --------------------
  unsigned best = 0xFFFFFFFFu;
  for (int j = tid; j < nb; j += blockDim.x) {
    const int blk = L.blocks[j];
    const int mk = L.mask[blk] & 0xFFFF;
    if (mk != 0xFFFF) best = min(best, static_cast<unsigned>(blk * kBlock + (__ffs(~mk) - 1)));
  }
  best = warp_min(best);
  if ((tid & 31) == 0) sh_min[tid >> 5] = best;
  __syncthreads();
  best = 0xFFFFFFFFu;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) best = min(best, sh_min[w]);
  const bool need = best == 0xFFFFFFFFu;
  if (!need) {
    KT* kp = static_cast<KT*>(A.ls.k_pool);
    KT* vp = static_cast<KT*>(A.ls.v_pool);
    copy_row(kp + static_cast<size_t>(best) * d, static_cast<const KT*>(A.k_new) + static_cast<size_t>(l) * d, d);
    copy_row(vp + static_cast<size_t>(best) * d, static_cast<const KT*>(A.v_new) + static_cast<size_t>(l) * d, d);
    if (tid == 0) atomicOr(&L.mask[best >> 4], 1 << (best & 15));
  }
  if (tid == 0) {
    L.pos[m] = A.new_pos;
    L.slot[m] = need ? -1 : static_cast<int>(best);
    if (L.score) L.score[m] = 0.f;
    A.ls.count[l] = m + 1;
    if (m + 1 >= dm.cap) set_status(A.ws.status, ST_CAPACITY);
    A.n_victims[l] = vcount;
  }
  if (L.ring)
    for (int t = tid; t < W; t += blockDim.x) L.ring[static_cast<size_t>(m) * W + t] = 0.f;
  __syncthreads();

  // ---- relocation plan ---------------------------------------------------------
  int t_live = 0;
  const int ndst = lane_plan(L, nb, m + 1, false, dm.theta_f, need, &t_live, sh_scan);
  if (nan_count) atomicAdd(&sh_nan, nan_count);
  __syncthreads();
  const int nan_tot = sh_nan;
  if (tid == 0) {
    A.ws.need_admit[l] = need ? 1 : 0;
    A.ws.want_dst[l] = ndst;
    A.ws.plan_tlive[l] = t_live;
    if (need || ndst > 0) {
      atomicOr(A.ws.work_flag, 1);
      *sh_work = 1;
    }
    atomicAdd(reinterpret_cast<unsigned long long*>(&A.ls.stats[SC_VICTIMS]), (unsigned long long)vcount);
    if (dead) atomicAdd(reinterpret_cast<unsigned long long*>(&A.ls.stats[SC_FREED_DEAD]), (unsigned long long)dead);
    if (nan_tot) atomicAdd(reinterpret_cast<unsigned long long*>(&A.ls.stats[SC_NAN_KEYS]), (unsigned long long)nan_tot);
    if (l == 0) atomicAdd(reinterpret_cast<unsigned long long*>(&A.ls.stats[SC_STEPS]), 1ull);
  }
}

// ---------------------------------------------------------------------------
// allocator: run by one CTA (the last epilogue CTA of a decode step, or its
// own launch in the forced compaction).  Per-lane requests written by other
// CTAs of the same grid are read with ld.global.cg (L2), after their
// __threadfence().
// ---------------------------------------------------------------------------
__device__ void allocate_layer(const LayerState& ls, const Workspace& ws, const Dims& dm, int* sh_scan,
                               int* sh_flag) {
  const int tid = threadIdx.x;
  if (tid == 0) {
    *sh_flag = atomicExch(ws.work_flag, 0);
  }
  __syncthreads();
  if (*sh_flag == 0) {
    if (tid == 0) { ws.counters[1] = 0; ws.counters[2] = 0; }
    return;
  }
  // exclusive prefixes over lanes: admissions, destinations, moved tokens
  int totA = 0, totD = 0, totM = 0;
  for (int base = 0; base < dm.lanes; base += blockDim.x) {
    const int l = base + tid;
    const int a = l < dm.lanes ? __ldcg(ws.need_admit + l) : 0;
    const int dd = l < dm.lanes ? __ldcg(ws.want_dst + l) : 0;
    const int mm = (l < dm.lanes && dd > 0) ? __ldcg(ws.plan_tlive + l) : 0;
    int ta, td, tm;
    const int ea = block_excl_scan(a, sh_scan, &ta);
    const int ed = block_excl_scan(dd, sh_scan, &td);
    const int em = block_excl_scan(mm, sh_scan, &tm);
    if (l < dm.lanes) {
      ws.admit_block[l] = totA + ea;
      ws.dst_begin[l] = totD + ed;
      ws.move_begin[l] = totM + em;
    }
    totA += ta; totD += td; totM += tm;
  }
  const int need_total = totA + totD;
  // the lowest free block ids, ascending
  int found = 0;
  for (int base = 0; base < dm.P && found < need_total; base += blockDim.x) {
    const int blk = base + tid;
    const int fr = (blk < dm.P && __ldcg(ls.owner + blk) < 0) ? 1 : 0;
    int tot;
    const int ex = block_excl_scan(fr, sh_scan, &tot);
    if (fr && found + ex < need_total) ws.alloc_ids[found + ex] = blk;
    found += tot;
  }
  found = min(found, need_total);
  __syncthreads();
  const int gotA = min(found, totA);
  const bool deferred = totD > found - gotA;
  for (int l = tid; l < dm.lanes; l += blockDim.x) {
    if (__ldcg(ws.need_admit + l)) {
      const int idx = ws.admit_block[l];
      if (idx < gotA) {
        const int blk = ws.alloc_ids[idx];
        ws.admit_block[l] = blk;
        ls.owner[blk] = l;
      } else {
        // no block: the new token is not stored (its table entry is dropped)
        ws.admit_block[l] = -1;
        ws.need_admit[l] = 0;
        ls.count[l] = __ldcg(ls.count + l) - 1;
        set_status(ws.status, ST_NO_BLOCKS);
      }
    }
    const int nd = __ldcg(ws.want_dst + l);
    if (deferred) {
      if (nd > 0) ws.want_dst[l] = 0;
    } else {
      ws.dst_begin[l] = totA + ws.dst_begin[l];
    }
  }
  if (!deferred && totD > 0) {
    // destination q belongs to the last lane whose first destination is at
    // or before it (lanes without destinations share the next one's start)
    __syncthreads();
    for (int q = tid; q < totD; q += blockDim.x) {
      int lo = 0, hi = dm.lanes;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldcg(ws.dst_begin + mid) <= totA + q) lo = mid + 1; else hi = mid;
      }
      ls.owner[ws.alloc_ids[totA + q]] = lo - 1;
    }
  }
  if (tid == 0) {
    ws.counters[1] = 1;
    ws.counters[2] = deferred ? 0 : totM;
    if (deferred && totD > 0)
      atomicAdd(reinterpret_cast<unsigned long long*>(&ls.stats[SC_DEFERRED]), 1ull);
  }
}

__global__ void __launch_bounds__(1024) allocate_kernel(LayerState ls, Workspace ws, Dims dm) {
  __shared__ int sh_scan[40];
  __shared__ int sh_flag;
  allocate_layer(ls, ws, dm, sh_scan, &sh_flag);
}

// ---------------------------------------------------------------------------
// apply: one CTA per lane
// ---------------------------------------------------------------------------
template <typename KT>
__global__ void __launch_bounds__(kApplyThreads) apply_kernel(LayerState ls, Workspace ws, Dims dm,
                                                           const void* k_new, const void* v_new,
                                                           int mark_freed, int32_t* moves) {
  __shared__ int sh_scan[40];
  __shared__ int sh_mv_src[kApplyThreads], sh_mv_dst[kApplyThreads];
  grid_dep_launch();    // the next layer's attention may start (it touches other state)
  grid_dep_wait();      // the epilogue and its allocator are complete
  const int l = blockIdx.x, tid = threadIdx.x;
  if (ws.counters[1] == 0) return;
  const int need = ws.need_admit[l];
  const int ndst = ws.want_dst[l];
  if (!need && ndst == 0) return;
  LaneRefs L = lane_refs(ls, dm, l);
  const int d = dm.d;
  KT* kp = static_cast<KT*>(ls.k_pool);
  KT* vp = static_cast<KT*>(ls.v_pool);
  const int m = ls.count[l];
  if (need) {
    const int blk = ws.admit_block[l];
    const size_t s = static_cast<size_t>(blk) * kBlock;
    copy_row(kp + s * d, static_cast<const KT*>(k_new) + static_cast<size_t>(l) * d, d);
    copy_row(vp + s * d, static_cast<const KT*>(v_new) + static_cast<size_t>(l) * d, d);
    if (tid == 0) {
      L.mask[blk] = 1;
      L.slot[m - 1] = blk * kBlock;
      const int nb = *L.nblocks;
      L.blocks[nb] = blk;
      *L.nblocks = nb + 1;
      ws.need_admit[l] = 0;
      atomicAdd(reinterpret_cast<unsigned long long*>(&ls.stats[SC_ADMIT_NEW_BLOCK]), 1ull);
    }
    __syncthreads();
  }
  if (ndst > 0) {
    const int nb = *L.nblocks;
    int nsrc = 0;
    for (int j = tid; j < nb; j += blockDim.x) {
      const int blk = L.blocks[j];
      const int c = __popc(L.mask[blk] & 0xFFFF);
      if (c > 0 && c < kBlock) { ws.blk_tag[blk] = 1; ++nsrc; }
    }
    int nsrc_tot;
    (void)block_excl_scan(nsrc, sh_scan, &nsrc_tot);
    const int dbeg = ws.dst_begin[l];
    const int mbeg = ws.move_begin[l];
    const int cpr = d * static_cast<int>(sizeof(KT)) / 16;     // 16-byte pieces per K or V row
    const size_t row_bytes = static_cast<size_t>(d) * sizeof(KT);
    unsigned char* kpb = reinterpret_cast<unsigned char*>(kp);
    unsigned char* vpb = reinterpret_cast<unsigned char*>(vp);
    int q_total = 0;
    for (int base = 0; base < m; base += blockDim.x) {
      const int i = base + tid;
      int old = -1;
      bool src = false;
      if (i < m) {
        old = L.slot[i];
        src = old >= 0 && ws.blk_tag[old >> 4] == 1;
      }
      int tot;
      const int ex = block_excl_scan(src ? 1 : 0, sh_scan, &tot);
      if (src && (q_total + ex) / kBlock >= ndst) {
        set_status(ws.status, ST_BAD_INDEX);   // plan and tables disagree: leave the token in place
        sh_mv_src[ex] = -1;
      } else if (src) {
        const int q = q_total + ex;
        const int db = ws.alloc_ids[dbeg + q / kBlock];
        const int dof = q % kBlock;
        const int ns = db * kBlock + dof;
        sh_mv_src[ex] = old;
        sh_mv_dst[ex] = ns;
        L.slot[i] = ns;
        if (moves) {
          int32_t* mv = moves + static_cast<size_t>(mbeg + q) * 6;
          mv[0] = l; mv[1] = L.pos[i]; mv[2] = old >> 4; mv[3] = old & 15; mv[4] = db; mv[5] = dof;
        }
      }
      __syncthreads();
      // the chunk's K and V rows in 16-byte pieces, eight loads in flight per
      // thread before their stores (destinations are fresh blocks, never a
      // source of the same plan)
      const int npieces = tot * 2 * cpr;
      for (int e0 = tid; e0 < npieces; e0 += blockDim.x * kCopyBatch) {
        uint4 v[kCopyBatch];
        unsigned char* dst[kCopyBatch];
#pragma unroll
        for (int u = 0; u < kCopyBatch; ++u) {
          const int e = e0 + u * static_cast<int>(blockDim.x);
          dst[u] = nullptr;
          if (e < npieces) {
            const int mvi = e / (2 * cpr), rem = e - mvi * 2 * cpr;
            const int so = sh_mv_src[mvi];
            if (so >= 0) {
              unsigned char* base = rem < cpr ? kpb : vpb;
              const size_t c16 = static_cast<size_t>(rem < cpr ? rem : rem - cpr) * 16;
              v[u] = *reinterpret_cast<const uint4*>(base + static_cast<size_t>(so) * row_bytes + c16);
              dst[u] = base + static_cast<size_t>(sh_mv_dst[mvi]) * row_bytes + c16;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kCopyBatch; ++u)
          if (dst[u]) *reinterpret_cast<uint4*>(dst[u]) = v[u];
      }
      __syncthreads();
      q_total += tot;
    }
    __syncthreads();
    for (int j = tid; j < ndst; j += blockDim.x) {
      const int db = ws.alloc_ids[dbeg + j];
      const int filled = min(kBlock, q_total - j * kBlock);
      L.mask[db] = filled >= kBlock ? 0xFFFF : ((1 << filled) - 1);
    }
    for (int j = tid; j < nb; j += blockDim.x) {
      const int blk = L.blocks[j];
      if (ws.blk_tag[blk] == 1) {
        ws.blk_tag[blk] = 0;
        L.mask[blk] = 0;
        L.owner[blk] = -1;
        if (mark_freed) ws.freed_flag[blk] = 1;
      }
    }
    __syncthreads();
    const int nb2 = lane_prune_blocks(L, l, sh_scan);
    for (int j = tid; j < ndst; j += blockDim.x) L.blocks[nb2 + j] = ws.alloc_ids[dbeg + j];
    __syncthreads();
    if (tid == 0) {
      *L.nblocks = nb2 + ndst;
      ws.want_dst[l] = 0;
      atomicAdd(reinterpret_cast<unsigned long long*>(&ls.stats[SC_PLANS]), 1ull);
      atomicAdd(reinterpret_cast<unsigned long long*>(&ls.stats[SC_MOVED]), (unsigned long long)q_total);
      atomicAdd(reinterpret_cast<unsigned long long*>(&ls.stats[SC_FREED_RELOC]), (unsigned long long)nsrc_tot);
    }
  }
}

}  // namespace

cudaError_t launch_epilogue(const Ctx& ctx, int layer, bool has_q, int new_pos, const void* k_new,
                            const void* v_new, float* out, float* lse, int32_t* victims,
                            int32_t* n_victims, cudaStream_t stream) {
  EpiArgs A;
  A.ls = layer_state(ctx, layer);
  A.ws = ctx.ws;
  A.dm = ctx.dims;
  A.has_q = has_q ? 1 : 0;
  A.new_pos = new_pos;
  A.layer = layer;
  A.k_new = k_new; A.v_new = v_new;
  A.out = out; A.lse = lse; A.victims = victims; A.n_victims = n_victims;
  // After this layer's attention launch the predecessor triggers only once
  // its own predecessors are complete; without one, the predecessor may be
  // the last step's apply, whose epilogue may still be writing that layer's
  // tables, which this kernel reads before its dependency wait.
  const bool pdl = has_q || ctx.last_layer != layer;
  if (ctx.dims.dtype == KVEVICT_BF16)
    return launch_k(decode_epilogue_kernel<__nv_bfloat16>, dim3(ctx.dims.lanes), dim3(kEpiThreads), kEpiDynSmem,
                    stream, pdl, A);
  return launch_k(decode_epilogue_kernel<float>, dim3(ctx.dims.lanes), dim3(kEpiThreads), kEpiDynSmem, stream,
                  pdl, A);
}

cudaError_t prepare_epilogue() {
  cudaError_t e = cudaFuncSetAttribute(decode_epilogue_kernel<__nv_bfloat16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kEpiDynSmem));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_epilogue_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kEpiDynSmem));
  return e;
}

cudaError_t launch_allocate(const Ctx& ctx, int layer, cudaStream_t stream) {
  allocate_kernel<<<1, 1024, 0, stream>>>(layer_state(ctx, layer), ctx.ws, ctx.dims);
  return cudaGetLastError();
}

cudaError_t launch_allocate_apply(const Ctx& ctx, int layer, const void* k_new, const void* v_new,
                                  bool mark_freed, int32_t* moves, cudaStream_t stream, bool with_allocate) {
  LayerState ls = layer_state(ctx, layer);
  if (with_allocate) allocate_kernel<<<1, 1024, 0, stream>>>(ls, ctx.ws, ctx.dims);
  const bool pdl = !with_allocate;   // in a decode step apply follows the epilogue directly
  const int mf = mark_freed ? 1 : 0;
  if (ctx.dims.dtype == KVEVICT_BF16)
    return launch_k(apply_kernel<__nv_bfloat16>, dim3(ctx.dims.lanes), dim3(kApplyThreads), 0, stream, pdl, ls,
                    ctx.ws, ctx.dims, k_new, v_new, mf, moves);
  return launch_k(apply_kernel<float>, dim3(ctx.dims.lanes), dim3(kApplyThreads), 0, stream, pdl, ls, ctx.ws,
                  ctx.dims, k_new, v_new, mf, moves);
}

}  // namespace kve
