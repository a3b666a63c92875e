// D1: split-K GQA decode attention over a paged, token-table-indexed KV pool.
//
// For every lane (sequence b, KV head h) the g query heads of the group
// attend the lane's kept tokens (read through their slots, vToken review
// Eq. (2)) and the new token (read from the call's k_new/v_new).  The work
// is the concatenation of every lane's 16-token tiles, cut into equal
// contiguous ranges, one per warp of a persistent grid (stream-K), so every
// warp streams the same number of bytes whatever the lanes' lengths.  A warp
// writes, per lane segment it covers, the running max / sum / unnormalised
// output of the segment (split-K partials) and, for every token, its base-2
// scaled logits, which the epilogue turns into weights once the lane's
// log-sum-exp is known (H2O Guide, "Formulating Cumulative Attention
// Scores": the weights are the ones the attention pass already computes).
//
// bf16: K/V rows move HBM -> shared memory with one cp.async.bulk per row,
// completing on a per-stage mbarrier (3 stages per warp, L2 evict_first);
// QK^T and PV run on the tensor cores with the warp-level bf16 MMA
// (m16n8k16; the 16 M rows are the group's query heads), fp32 accumulation;
// P enters the PV product as a hi + lo pair of bf16 values so the output
// keeps ~16 bits of weight precision.
// fp32: one thread per token on the CUDA cores (small heads only).
#include "kvevict_internal.cuh"

namespace kve {

namespace {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// p -> (hi, lo) bf16 pairs with hi + lo == p to ~16 significant bits
__device__ __forceinline__ void split_bf16(float p0, float p1, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
  float2 hf = __bfloat1622float2(h);
  __nv_bfloat162 l = __floats2bfloat162_rn(p0 - hf.x, p1 - hf.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}

struct AttendArgs {
  const void* k_pool; const void* v_pool;
  const int32_t* slot; const int32_t* count;
  const void* q; const void* k_new; const void* v_new;
  float* logits; float* part_o; float* part_ml; int32_t* lane_nseg;
  uint32_t* status;
  int lanes, g, Hkv, Hq, cap, lcap, P;
  float scale2;   // log2(e) / sqrt(d)
  int early_trigger;   // let the successor (the decode epilogue) be scheduled at once
  // Before writing its scratch copy the kernel waits (acquire) until
  // *reads_done has reached reads_expect (wrapping): every epilogue launched
  // on the copy before has finished with it.  Null: no such wait.
  const uint32_t* reads_done;
  uint32_t reads_expect;
};

constexpr int kMaxLanesSmem = 1024;   // lanes per layer (validated at create)

// The layer's T tiles are cut into one contiguous range per warp, skewed:
// warp gw of W starts at floor(T (x + c x (1 - x))), x = gw / W (fp32, exact
// at both ends), so early warps take more tiles than late ones.  Every warp issues its first
// copy stages at launch, and the copy engine serves that burst roughly in
// launch order: a warp of the last CTAs receives its first tile several
// microseconds after one of the first CTAs, and with equal ranges finishes
// that much later.  c is chosen so the skew is about kSkewTiles tiles between
// the first and the last warp (the stages in flight at launch, times the
// ratio of streaming to burst bandwidth, measured on the 70B-shaped layer),
// and no smaller than a lane's split-K segment bound allows.  Consecutive
// starts are at least two tiles apart, so the fp32 rounding (T 2^-23 at most)
// cannot reorder them below 2^23 tiles per layer.
constexpr int kSkewTiles = 2;

struct Split {
  int T, W;
  int tp;          // > 0: equal ranges of tp tiles (small layers), no skew
  float c, rW;
  __device__ __forceinline__ int begin(int gw) const {
    if (gw >= W) return T;
    if (tp > 0) return min(T, gw * tp);
    const float x = static_cast<float>(gw) * rW;
    return min(T, __float2int_rd(static_cast<float>(T) * fmaf(c * x, 1.f - x, x)));
  }
  // the warp whose range holds tile t (the last warp starting at or before
  // it): the quadratic inverted in fp32, then corrected against begin()
  __device__ __forceinline__ int warp_of(int t) const {
    if (tp > 0) return min(W - 1, t / tp);
    const float y = static_cast<float>(t) / static_cast<float>(T);
    float x = y;
    if (c > 0.f) {
      const float b = 1.f + c;
      x = (b - sqrtf(fmaxf(0.f, b * b - 4.f * c * y))) / (2.f * c);
    }
    int g = min(W - 1, max(0, __float2int_rd(x * static_cast<float>(W))));
    while (g + 1 < W && begin(g + 1) <= t) ++g;
    while (g > 0 && begin(g) > t) --g;
    return g;
  }
};

// ---------------------------------------------------------------------------
// bf16 tensor-core kernel
//
// Per 16-token tile a warp computes S^T = K Q^T (M = 16 tokens, N = 8 query
// heads of the group, K = d) and O^T += V^T P^T (M = 16 rows of d, N = 8
// heads, K = 16 tokens), so a group of 8 heads fills the MMA with no padding.
// P^T reaches the B operand through a shared-memory transpose (stmatrix.trans
// then ldmatrix), as a hi + lo pair of bf16 values.
// ---------------------------------------------------------------------------
constexpr int kAttStages = 2;      // copy stages per warp
constexpr float kRescaleLog2 = 8.f;  // lazy-rescale threshold (log2 units)

template <int D, int NT>
struct Bf16Cfg {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kRowStride = kRowBytes + 16;            // +16 B: conflict-free ldmatrix
  static constexpr int kStageBytes = 2 * 16 * kRowStride;      // K rows then V rows
  static constexpr int kPBytes = NT * 2 * 8 * 32;              // [NT][hi, lo][8 heads][16 tokens] bf16
  static constexpr int kWarpBytes = kAttStages * kStageBytes + kPBytes;
  static constexpr int kSmem = kAttendWarps * kWarpBytes;      // warp buffers; the lane prefix follows
  // dynamic shared memory of a launch over `lanes` lanes: the warp buffers,
  // then the lanes' tile prefix (lanes + 1 ints)
  static constexpr int smem_for(int lanes) { return kSmem + ((lanes + 1) * 4 + 15) / 16 * 16; }
  static constexpr int kKs = D / 16;                           // k-steps over d (QK^T)
  static constexpr int kDt = D / 16;                           // 16-row tiles of d (PV)
};

__device__ __forceinline__ void stsm_x2_t(uint32_t addr, uint32_t r0, uint32_t r1) {
  asm volatile("stmatrix.sync.aligned.m8n8.x2.trans.shared.b16 [%0], {%1, %2};" ::"r"(addr), "r"(r0), "r"(r1)
               : "memory");
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16a(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  mma_bf16(c, a[0], a[1], a[2], a[3], b0, b1);
}

template <int D, int NT>
__device__ __forceinline__ bool attend_warp(const AttendArgs& a, const int* sh_prefix, const Split& sp, const int gw,
                                            const int t_begin, const int t_end, unsigned char* wbuf,
                                            uint64_t* bars);

// With one head tile, three CTAs of this kernel (12 warps) fill an SM's
// register file only to three quarters (128 registers a thread), and their
// shared memory leaves about 12 KB: one CTA of the lean decode epilogue fits
// beside them, so the epilogue of one layer runs on the same SMs while the
// next layer streams.  (Two head tiles need more registers.)
template <int D, int NT>
__global__ void __launch_bounds__(kAttendWarps * 32, NT == 1 ? 4 : 3) attend_bf16_kernel(AttendArgs a) {
  using C = Bf16Cfg<D, NT>;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int sh_scan[40];
  __shared__ uint64_t sh_bar[kAttendWarps][kAttStages];

  const int tid = threadIdx.x, lane_id = tid & 31, warp = tid >> 5;
  const int lanes = a.lanes;
  int* sh_prefix = reinterpret_cast<int*>(smem + C::kSmem);   // [lanes + 1]
  // The kernel may have started before earlier kernels in the stream
  // finished: it touches nothing until every epilogue launched before on its
  // scratch copy has finished (which orders every earlier epilogue of its
  // layer, and everything each of those waited for, before it).  Thread 0
  // polls, bounded; past the bound the dependency wait covers it instead.
  if (a.reads_done) {
    if (tid == 0) {
      int ok = 0;
      for (int polls = 0; polls < (1 << 14); ++polls) {
        if (static_cast<int>(static_cast<uint32_t>(ld_acquire_gpu(reinterpret_cast<const int*>(a.reads_done))) -
                             a.reads_expect) >= 0) {
          ok = 1;
          break;
        }
        __nanosleep(128);
      }
      sh_scan[0] = ok;
    }
    __syncthreads();
    const int ok = sh_scan[0];
    __syncthreads();
    if (!ok) grid_dep_wait();
  }
  // Inside a decode step the kernel that consumes these results (the decode
  // epilogue) may be scheduled from now on: it reads only what this kernel
  // does not write before its own dependency wait, which returns once this
  // grid is complete.  Otherwise the successor is unknown and starts only
  // once every CTA of this grid is at its end.
  if (a.early_trigger) grid_dep_launch();

  // --- lane tile prefix (every CTA computes the same table) ---------------
  int my_max = 0;
  {
    int carry = 0;
    for (int base = 0; base < lanes; base += blockDim.x) {
      int l = base + tid;
      int t = 0;
      if (l < lanes) {
        int n = a.count[l];
        if (n < 0 || n >= a.cap) { set_status(a.status, ST_BAD_INDEX); n = n < 0 ? 0 : a.cap - 1; }
        t = (n + 1 + 15) >> 4;
      }
      my_max = max(my_max, t);
      int tot;
      int ex = block_excl_scan(t, sh_scan, &tot);
      if (l < lanes) sh_prefix[l] = carry + ex;
      carry += tot;
    }
    if (tid == 0) sh_prefix[lanes] = carry;
  }
  my_max = warp_max(my_max);
  if (lane_id == 0) sh_scan[warp] = my_max;
  __syncthreads();
  int max_tiles = 0;
  for (int w = 0; w < kAttendWarps; ++w) max_tiles = max(max_tiles, sh_scan[w]);
  const int total = sh_prefix[lanes];
  // warps in use: every warp's range must hold at least `need` tiles, so a
  // lane spans at most kMaxSeg - 1 ranges (plus one for a partial start)
  const int need = max(1, (max_tiles + kMaxSeg - 2) / (kMaxSeg - 1));
  const int warps_total = gridDim.x * kAttendWarps;
  Split sp;
  sp.T = total;
  if (total < (need + 2) * warps_total) {
    // a small layer: equal ranges of at least `need` tiles, integer
    // boundaries, no skew
    sp.tp = max(need, (total + warps_total - 1) / warps_total);
    sp.W = (total + sp.tp - 1) / sp.tp;
    sp.rW = 0.f;
    sp.c = 0.f;
  } else {
    // every warp; the mean range is at least need + 2 tiles, so fp32
    // rounding keeps every skewed range at or above need
    sp.tp = 0;
    sp.W = warps_total;
    sp.rW = 1.f / static_cast<float>(sp.W);
    // skew: about kSkewTiles tiles first to last, while the smallest range,
    // mean (1 - c), keeps at least need + 1 tiles; c <= 1/2
    const float mean = static_cast<float>(total) * sp.rW;
    const float cmax = mean > static_cast<float>(need + 1) ? 1.f - static_cast<float>(need + 1) / mean : 0.f;
    sp.c = fmaxf(0.f, fminf(fminf(static_cast<float>(kSkewTiles) / mean, cmax), 0.5f));
  }
  // the split-K segment count of each lane, by the CTA with the fewest tiles
  if (blockIdx.x == gridDim.x - 1) {
    for (int l = tid; l < lanes; l += blockDim.x) {
      const int s = sh_prefix[l], e = sh_prefix[l + 1];
      a.lane_nseg[l] = sp.warp_of(e - 1) - sp.warp_of(s) + 1;
    }
  }

  const int gw = blockIdx.x * kAttendWarps + warp;
  const int t_begin = gw < sp.W ? sp.begin(gw) : total;
  const int t_end = gw < sp.W ? sp.begin(gw + 1) : total;
  if (t_begin < t_end)
    (void)attend_warp<D, NT>(a, sh_prefix, sp, gw, t_begin, t_end, smem + warp * C::kWarpBytes, sh_bar[warp]);
  // this grid completes only after its predecessor did (so completion
  // orders everything before it)
  grid_dep_wait();
  if (!a.early_trigger) grid_dep_launch();
}

// One warp's range of tiles [t_begin, t_end) (stream-K split of the layer);
// false if a bounded wait gave up.
template <int D, int NT>
__device__ __forceinline__ bool attend_warp(const AttendArgs& a, const int* sh_prefix, const Split& sp, const int gw,
                                            const int t_begin, const int t_end, unsigned char* wbuf,
                                            uint64_t* bars) {
  using C = Bf16Cfg<D, NT>;
  const int lane_id = threadIdx.x & 31;
  unsigned char* pbuf = wbuf + kAttStages * C::kStageBytes;
  if (lane_id == 0) {
    for (int s = 0; s < kAttStages; ++s) mbar_init(&bars[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  const uint64_t pol = policy_evict_first();

  const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(a.k_pool);
  const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(a.v_pool);
  const __nv_bfloat16* kn = static_cast<const __nv_bfloat16*>(a.k_new);
  const __nv_bfloat16* vn = static_cast<const __nv_bfloat16*>(a.v_new);
  const int pool_rows = a.P * kBlock;
  const int r = lane_id & 15;          // the row (token) this thread copies
  const bool isv = lane_id >= 16;      // K row (lanes 0-15) or V row (16-31)

  // --- producer: slot indices are fetched one issue ahead -----------------
  int pf_lane = 0, pf_n = 0;
  {
    int l = 0;
    while (sh_prefix[l + 1] <= t_begin) ++l;
    pf_lane = l;
    pf_n = min(max(a.count[l], 0), a.cap - 1);
  }
  int iss_lane = pf_lane, iss_n = pf_n;
  auto fetch_slot = [&](int t) -> int {
    if (t >= t_end) return -1;
    while (sh_prefix[pf_lane + 1] <= t) {
      ++pf_lane;
      pf_n = min(max(a.count[pf_lane], 0), a.cap - 1);
    }
    const int i = (t - sh_prefix[pf_lane]) * 16 + r;
    return i < pf_n ? a.slot[static_cast<size_t>(pf_lane) * a.cap + i] : -1;
  };
  // --- query fragments -------------------------------------------------------
  // qb holds the query of the lane being consumed; with one head tile, qn
  // receives the next lane's query as soon as the copy of that lane's first
  // tile is issued, so a lane change does not wait on a global load.
  const int gq = lane_id >> 2, cq = lane_id & 3;
  constexpr bool kQAhead = NT == 1;
  uint32_t qb[NT][C::kKs][2];
  uint32_t qn[kQAhead ? NT : 1][kQAhead ? C::kKs : 1][2];
  auto fetch_q = [&](int l, uint32_t (*dst)[C::kKs][2]) {
    const int b = l / a.Hkv, kh = l % a.Hkv;
    const __nv_bfloat16* qbase = static_cast<const __nv_bfloat16*>(a.q) +
                                 (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(kh) * a.g) * D;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h = nt * 8 + gq;
      const bool ok = h < a.g;
#pragma unroll
      for (int ks = 0; ks < C::kKs; ++ks) {
        const int c0 = ks * 16 + cq * 2;
        dst[nt][ks][0] = ok ? *reinterpret_cast<const uint32_t*>(qbase + h * D + c0) : 0u;
        dst[nt][ks][1] = ok ? *reinterpret_cast<const uint32_t*>(qbase + h * D + c0 + 8) : 0u;
      }
    }
  };

  auto issue = [&](int t, int st, int slot) {
    while (sh_prefix[iss_lane + 1] <= t) {
      ++iss_lane;
      iss_n = min(max(a.count[iss_lane], 0), a.cap - 1);
      if constexpr (kQAhead) fetch_q(iss_lane, reinterpret_cast<uint32_t (*)[C::kKs][2]>(qn));
    }
    const int l = iss_lane, n = iss_n;
    const int i0 = (t - sh_prefix[l]) * 16;
    const int valid = min(16, n + 1 - i0);
    unsigned char* sbuf = wbuf + st * C::kStageBytes;
    fence_proxy_async();
    if (lane_id == 0) mbar_arrive_expect_tx(&bars[st], static_cast<uint32_t>(valid * 2 * C::kRowBytes));
    __syncwarp();
    unsigned char* dst = sbuf + (isv ? 16 * C::kRowStride : 0) + r * C::kRowStride;
    const int i = i0 + r;
    if (r < valid) {
      const __nv_bfloat16* src;
      if (i < n) {
        int s = slot;
        if (s < 0 || s >= pool_rows) { set_status(a.status, ST_BAD_INDEX); s = 0; }
        src = (isv ? vp : kp) + static_cast<size_t>(s) * D;
      } else {
        src = (isv ? vn : kn) + static_cast<size_t>(l) * D;
      }
      bulk_g2s(dst, src, C::kRowBytes, &bars[st], pol);
    } else {
      const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int o = 0; o < C::kRowBytes; o += 16) *reinterpret_cast<uint4*>(dst + o) = z;
    }
  };

  // --- consumer state -------------------------------------------------------
  float o_acc[NT][C::kDt][4];
  float m_run[NT][2], l_run[NT][2];
  int cur_lane = -1, seg = 0, cur_n = 0;

  auto reset_acc = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int dt = 0; dt < C::kDt; ++dt) o_acc[nt][dt][0] = o_acc[nt][dt][1] = o_acc[nt][dt][2] = o_acc[nt][dt][3] = 0.f;
      m_run[nt][0] = m_run[nt][1] = -INFINITY;
      l_run[nt][0] = l_run[nt][1] = 0.f;
    }
  };

  auto flush = [&]() {
    const size_t base = (static_cast<size_t>(cur_lane) * kMaxSeg + seg) * a.g;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float s = l_run[nt][e];
        s += __shfl_xor_sync(0xffffffffu, s, 4);
        s += __shfl_xor_sync(0xffffffffu, s, 8);
        s += __shfl_xor_sync(0xffffffffu, s, 16);
        const int h = nt * 8 + cq * 2 + e;
        if (h < a.g) {
          float* po = a.part_o + (base + h) * D;
#pragma unroll
          for (int dt = 0; dt < C::kDt; ++dt) {
            po[dt * 16 + gq] = o_acc[nt][dt][e];
            po[dt * 16 + gq + 8] = o_acc[nt][dt][2 + e];
          }
          if (gq == 0) *reinterpret_cast<float2*>(a.part_ml + (base + h) * 2) = make_float2(m_run[nt][e], s);
        }
      }
    }
  };

  // --- pipeline ---------------------------------------------------------------
  int next_slot = fetch_slot(t_begin);
  fetch_q(iss_lane, qb);
  issue(t_begin, 0, next_slot);
  next_slot = fetch_slot(t_begin + 1);

  // smem lane addresses
  const int ktok = (lane_id & 7) + (((lane_id >> 3) & 1) << 3);
  const int kcol = (lane_id >> 4) * 16;                  // bytes
  const int vtok = (lane_id & 7) + ((lane_id >> 4) << 3);
  const int vcol = ((lane_id >> 3) & 1) * 16;            // bytes
  const int prow = (lane_id & 7) * 32 + ((lane_id >> 3) & 1) * 16;   // stmatrix / ldmatrix.x2 rows

  int cons_lane = 0;
  while (sh_prefix[cons_lane + 1] <= t_begin) ++cons_lane;
  for (int t = t_begin, u = 0; t < t_end; ++t, ++u) {
    // lane change of the consumer first: issuing tile t + 1 may refill qn
    while (sh_prefix[cons_lane + 1] <= t) ++cons_lane;
    if (cons_lane != cur_lane) {
      if (cur_lane >= 0) {
        flush();
        if constexpr (kQAhead) {
#pragma unroll
          for (int ks = 0; ks < C::kKs; ++ks) {
            qb[0][ks][0] = qn[0][ks][0];
            qb[0][ks][1] = qn[0][ks][1];
          }
        } else {
          fetch_q(cons_lane, qb);
        }
      }
      cur_lane = cons_lane;
      seg = gw - sp.warp_of(sh_prefix[cur_lane]);
      cur_n = min(max(a.count[cur_lane], 0), a.cap - 1);
      reset_acc();
    }
    if (t + 1 < t_end) {
      issue(t + 1, (u + 1) % kAttStages, next_slot);
      next_slot = fetch_slot(t + 2);
    }
    const int st = u % kAttStages;
    const uint32_t par = (u / kAttStages) & 1;
    {
      int spins = 0;
      while (!mbar_try_wait(&bars[st], par)) {
        if (++spins > (1 << 22)) { set_status(a.status, ST_TIMEOUT); return false; }
      }
    }
    __syncwarp();
    const int i0 = (t - sh_prefix[cur_lane]) * 16;
    const unsigned char* kb = wbuf + st * C::kStageBytes;
    const unsigned char* vb = kb + 16 * C::kRowStride;

    // S^T = K Q^T : kSAcc independent accumulators per head tile (k-steps
    // round robin), summed at the end, to keep the dependent MMA chain short
    constexpr int kSAcc = C::kKs >= 4 ? 4 : C::kKs;
    float sacc[kSAcc][NT][4];
#pragma unroll
    for (int c = 0; c < kSAcc; ++c)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[c][nt][e] = 0.f;
    {
      const uint32_t addr = smem_u32(kb + ktok * C::kRowStride + kcol);
#pragma unroll
      for (int ks = 0; ks < C::kKs; ++ks) {
        uint32_t af[4];
        ldsm_x4(addr + ks * 32, af[0], af[1], af[2], af[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16a(sacc[ks % kSAcc][nt], af, qb[nt][ks][0], qb[nt][ks][1]);
      }
    }
    const bool ok0 = i0 + gq <= cur_n, ok1 = i0 + gq + 8 <= cur_n;
    uint32_t ph[NT][2], pl[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float sv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool ok = (e < 2) ? ok0 : ok1;
        float acc = sacc[0][nt][e];
#pragma unroll
        for (int c = 1; c < kSAcc; ++c) acc += sacc[c][nt][e];
        sv[e] = ok ? acc * a.scale2 : -INFINITY;
      }
      // logits of the valid heads: [lane][head][token]
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = nt * 8 + cq * 2 + e;
        if (h < a.g) {
          float* lrow = a.logits + (static_cast<size_t>(cur_lane) * a.g + h) * a.lcap + i0;
          lrow[gq] = sv[e];
          lrow[gq + 8] = sv[2 + e];
        }
      }
      // Lazy rescaling: the running max m_run only moves when some logit
      // of the tile exceeds it by more than kRescaleLog2 (a warp vote), so
      // the cross-lane max and the rescale of o_acc are skipped on most
      // tiles.  Weights are then at most 2^kRescaleLog2, far inside fp32;
      // (m_run, l_run) stay a consistent pair for the split-K combine.
      bool grow = false;
#pragma unroll
      for (int e = 0; e < 2; ++e) grow |= fmaxf(sv[e], sv[2 + e]) > m_run[nt][e] + kRescaleLog2;
      if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float tm = fmaxf(sv[e], sv[2 + e]);
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 4));
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 8));
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
          const float mo = m_run[nt][e];
          const float mn = fmaxf(mo, tm);
          const float corr = (mo == -INFINITY) ? 0.f : exp2f(mo - mn);
          m_run[nt][e] = mn;
          l_run[nt][e] *= corr;
#pragma unroll
          for (int dt = 0; dt < C::kDt; ++dt) {
            o_acc[nt][dt][e] *= corr;
            o_acc[nt][dt][2 + e] *= corr;
          }
        }
      }
      float pv[4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        pv[e] = exp2f(sv[e] - m_run[nt][e]);
        pv[2 + e] = exp2f(sv[2 + e] - m_run[nt][e]);
        l_run[nt][e] += pv[e] + pv[2 + e];
      }
      split_bf16(pv[0], pv[1], ph[nt][0], pl[nt][0]);   // token gq,     heads 2c, 2c+1
      split_bf16(pv[2], pv[3], ph[nt][1], pl[nt][1]);   // token gq + 8
    }
    // P -> [head][token] in shared memory (transposed store), then B fragments
    uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      unsigned char* pb = pbuf + nt * 2 * 8 * 32;
      stsm_x2_t(smem_u32(pb + prow), ph[nt][0], ph[nt][1]);
      stsm_x2_t(smem_u32(pb + 256 + prow), pl[nt][0], pl[nt][1]);
    }
    __syncwarp();
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const unsigned char* pb = pbuf + nt * 2 * 8 * 32;
      ldsm_x2(smem_u32(pb + prow), bh[nt][0], bh[nt][1]);
      ldsm_x2(smem_u32(pb + 256 + prow), bl[nt][0], bl[nt][1]);
    }
    // O^T += V^T P^T
    {
      const uint32_t addr = smem_u32(vb + vtok * C::kRowStride + vcol);
#pragma unroll
      for (int dt = 0; dt < C::kDt; ++dt) {
        uint32_t af[4];
        ldsm_x4_t(addr + dt * 32, af[0], af[1], af[2], af[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_bf16a(o_acc[nt][dt], af, bh[nt][0], bh[nt][1]);
          mma_bf16a(o_acc[nt][dt], af, bl[nt][0], bl[nt][1]);
        }
      }
    }
    __syncwarp();
  }
  flush();
  return true;
}

// ---------------------------------------------------------------------------
// fp32 CUDA-core kernel: grid (chunks, lanes), one thread per token
// ---------------------------------------------------------------------------
constexpr int kF32Chunk = 128;

__global__ void __launch_bounds__(kF32Chunk) attend_f32_kernel(AttendArgs a, int D) {
  extern __shared__ float fsm[];
  float* sq = fsm;                       // [g][D]
  float* sp = sq + a.g * D;              // [g][kF32Chunk]
  float* sred = sp + a.g * kF32Chunk;    // [g][2]
  const int l = blockIdx.y, chunk = blockIdx.x, tid = threadIdx.x;
  int n = a.count[l];
  if (n < 0 || n >= a.cap) { if (tid == 0) set_status(a.status, ST_BAD_INDEX); n = max(0, min(n, a.cap - 1)); }
  const int nchunks = (n + 1 + kF32Chunk - 1) / kF32Chunk;
  if (chunk == 0 && tid == 0) a.lane_nseg[l] = nchunks;
  if (chunk >= nchunks) {
    grid_dep_wait();
    return;
  }
  const int b = l / a.Hkv, kh = l % a.Hkv;
  const float* qb = static_cast<const float*>(a.q) + (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(kh) * a.g) * D;
  for (int i = tid; i < a.g * D; i += blockDim.x) sq[i] = qb[i];
  __syncthreads();
  const int i = chunk * kF32Chunk + tid;
  const bool ok = i <= n;
  const float* krow = nullptr;
  const size_t pool_rows = static_cast<size_t>(a.P) * kBlock;
  // the chunk's pool rows, read once (-1: the new token, whose rows come
  // with the call), so the P V loop below has no dependent global loads
  __shared__ int sh_slot[kF32Chunk];
  if (ok) {
    if (i < n) {
      int s = a.slot[static_cast<size_t>(l) * a.cap + i];
      if (s < 0 || static_cast<size_t>(s) >= pool_rows) { set_status(a.status, ST_BAD_INDEX); s = 0; }
      krow = static_cast<const float*>(a.k_pool) + static_cast<size_t>(s) * D;
      sh_slot[tid] = s;
    } else {
      krow = static_cast<const float*>(a.k_new) + static_cast<size_t>(l) * D;
      sh_slot[tid] = -1;
    }
  }
  // pool rows are 16-byte aligned (D floats, base checked at create); the
  // caller's new row may not be
  const bool k_vec = ok && (reinterpret_cast<uintptr_t>(krow) & 15) == 0;
  __shared__ float swarp[kF32Chunk / 32];
  for (int h = 0; h < a.g; ++h) {
    float s = -INFINITY;
    if (ok) {
      float acc = 0.f;
      if (k_vec) {
        const float4* k4 = reinterpret_cast<const float4*>(krow);
        const float4* q4 = reinterpret_cast<const float4*>(sq + h * D);
        float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
#pragma unroll 4
        for (int e4 = 0; e4 < D / 4; ++e4) {
          const float4 kv = k4[e4], qv = q4[e4];
          c0 = fmaf(qv.x, kv.x, c0);
          c1 = fmaf(qv.y, kv.y, c1);
          c2 = fmaf(qv.z, kv.z, c2);
          c3 = fmaf(qv.w, kv.w, c3);
        }
        acc = (c0 + c1) + (c2 + c3);
      } else {
        for (int e = 0; e < D; ++e) acc = fmaf(sq[h * D + e], krow[e], acc);
      }
      s = acc * a.scale2;
      a.logits[(static_cast<size_t>(l) * a.g + h) * a.lcap + i] = s;
    }
    float m = warp_max(s);
    if ((tid & 31) == 0) swarp[tid >> 5] = m;
    __syncthreads();
    m = swarp[0];
    for (int w = 1; w < kF32Chunk / 32; ++w) m = fmaxf(m, swarp[w]);
    __syncthreads();
    const float pv = ok ? exp2f(s - m) : 0.f;
    sp[h * kF32Chunk + tid] = pv;
    float ps = pv;
    for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
    if ((tid & 31) == 0) swarp[tid >> 5] = ps;
    __syncthreads();
    if (tid == 0) {
      float tot = 0.f;
      for (int w = 0; w < kF32Chunk / 32; ++w) tot += swarp[w];
      sred[h * 2 + 0] = m;
      sred[h * 2 + 1] = tot;
    }
    __syncthreads();
  }
  // O[h][e] = sum_i p[h][i] v_i[e]: consecutive threads read consecutive
  // elements of one value row; the rows' addresses come from shared memory,
  // so the unrolled loads of several tokens are in flight together
  const size_t base = (static_cast<size_t>(l) * kMaxSeg + chunk) * a.g;
  const int cnt = min(kF32Chunk, n + 1 - chunk * kF32Chunk);
  const float* vpool = static_cast<const float*>(a.v_pool);
  const float* vnew = static_cast<const float*>(a.v_new) + static_cast<size_t>(l) * D;
  for (int he = tid; he < a.g * D; he += blockDim.x) {
    const int h = he / D, e = he % D;
    float acc0 = 0.f, acc1 = 0.f;
    int t = 0;
#pragma unroll 8
    for (; t + 1 < cnt; t += 2) {
      const int s0 = sh_slot[t], s1 = sh_slot[t + 1];
      const float v0 = s0 >= 0 ? vpool[static_cast<size_t>(s0) * D + e] : vnew[e];
      const float v1 = s1 >= 0 ? vpool[static_cast<size_t>(s1) * D + e] : vnew[e];
      acc0 = fmaf(sp[h * kF32Chunk + t], v0, acc0);
      acc1 = fmaf(sp[h * kF32Chunk + t + 1], v1, acc1);
    }
    if (t < cnt) {
      const int s0 = sh_slot[t];
      acc0 = fmaf(sp[h * kF32Chunk + t], s0 >= 0 ? vpool[static_cast<size_t>(s0) * D + e] : vnew[e], acc0);
    }
    a.part_o[(base + h) * D + e] = acc0 + acc1;
  }
  if (tid < a.g) {
    a.part_ml[(base + tid) * 2 + 0] = sred[tid * 2 + 0];
    a.part_ml[(base + tid) * 2 + 1] = sred[tid * 2 + 1];
  }
  grid_dep_wait();
  grid_dep_launch();
}

}  // namespace

template <int D, int NT>
static cudaError_t set_attr() {
  cudaError_t e = cudaFuncSetAttribute(attend_bf16_kernel<D, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Bf16Cfg<D, NT>::smem_for(kMaxLanesSmem));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attend_bf16_kernel<D, NT>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  return e;
}

template <int D, int NT>
static int ctas_per_sm(int lanes) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attend_bf16_kernel<D, NT>, kAttendWarps * 32,
                                                    Bf16Cfg<D, NT>::smem_for(lanes)) != cudaSuccess)
    return 0;
  return n;
}

// Whether one CTA of the lean H2O epilogue fits on an SM beside `n` CTAs of
// this attention kernel launched over `lanes` lanes.
template <int D, int NT>
static bool lean_fits_beside(int dev, int n, int lanes) {
  cudaFuncAttributes fa, fl;
  int lean_threads = 0;
  if (cudaFuncGetAttributes(&fa, attend_bf16_kernel<D, NT>) != cudaSuccess) return false;
  if (lean_epilogue_attributes(&fl, &lean_threads) != cudaSuccess) return false;
  int smem_sm = 0, reserved = 0, regs_sm = 0, threads_sm = 0;
  if (cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) != cudaSuccess)
    return false;
  // registers are granted per warp, in units of 8 a thread
  auto regs = [](const cudaFuncAttributes& f, int threads) { return (f.numRegs + 7) / 8 * 8 * threads; };
  const long long smem = static_cast<long long>(n) *
                             (static_cast<long long>(fa.sharedSizeBytes) + Bf16Cfg<D, NT>::smem_for(lanes) + reserved) +
                         static_cast<long long>(fl.sharedSizeBytes) + reserved;
  const long long r = static_cast<long long>(n) * regs(fa, kAttendWarps * 32) + regs(fl, lean_threads);
  const int threads = n * kAttendWarps * 32 + lean_threads;
  return smem <= smem_sm && r <= regs_sm && threads <= threads_sm;
}

cudaError_t prepare_kernels(Ctx& ctx) {
  cudaError_t e = set_attr<128, 1>();
  if (e == cudaSuccess) e = set_attr<128, 2>();
  if (e == cudaSuccess) e = set_attr<64, 1>();
  if (e == cudaSuccess) e = set_attr<64, 2>();
  if (e == cudaSuccess) e = prepare_epilogue();
  if (e == cudaSuccess) e = prepare_dropkv();
  if (e != cudaSuccess) return e;
  const Dims& dm = ctx.dims;
  const int nt = dm.g > 8 ? 2 : 1;
  ctx.attend_ctas_per_sm = 1;
  if (dm.dtype == KVEVICT_BF16) {
    if (dm.d == 128) ctx.attend_ctas_per_sm = nt == 1 ? ctas_per_sm<128, 1>(dm.lanes) : ctas_per_sm<128, 2>(dm.lanes);
    else ctx.attend_ctas_per_sm = nt == 1 ? ctas_per_sm<64, 1>(dm.lanes) : ctas_per_sm<64, 2>(dm.lanes);
  }
  ctx.lean_coresident = false;
  if (dm.dtype == KVEVICT_BF16 && ctx.attend_ctas_per_sm >= 1) {
    const int n = ctx.attend_ctas_per_sm;
    if (dm.d == 128)
      ctx.lean_coresident = nt == 1 ? lean_fits_beside<128, 1>(ctx.device, n, dm.lanes)
                                    : lean_fits_beside<128, 2>(ctx.device, n, dm.lanes);
    else
      ctx.lean_coresident = nt == 1 ? lean_fits_beside<64, 1>(ctx.device, n, dm.lanes)
                                    : lean_fits_beside<64, 2>(ctx.device, n, dm.lanes);
  }
  return cudaGetLastError();
}

cudaError_t launch_attend(const Ctx& ctx, int layer, const void* q, const void* k_new, const void* v_new,
                          cudaStream_t stream, bool early_trigger) {
  const Dims& dm = ctx.dims;
  LayerState ls = layer_state(ctx, layer);
  AttendArgs a;
  a.k_pool = ls.k_pool; a.v_pool = ls.v_pool; a.slot = ls.slot; a.count = ls.count;
  a.q = q; a.k_new = k_new; a.v_new = v_new;
  const int c = layer % kScratchBufs;
  a.logits = ctx.ws.logits_buf[c]; a.part_o = ctx.ws.part_o_buf[c]; a.part_ml = ctx.ws.part_ml_buf[c];
  a.lane_nseg = ctx.ws.lane_nseg_buf[c]; a.status = ctx.ws.status;
  a.reads_done = ctx.ws.reads_done + c;
  a.reads_expect = ctx.epi_launches[c] * static_cast<uint32_t>(dm.lanes);
  a.lanes = dm.lanes; a.g = dm.g; a.Hkv = dm.Hkv; a.Hq = dm.Hq; a.cap = dm.cap; a.lcap = dm.lcap;
  a.P = dm.P;
  a.scale2 = 1.4426950408889634f / sqrtf(static_cast<float>(dm.d));
  a.early_trigger = early_trigger ? 1 : 0;
  // early start: see attend_early_ok (the kernel guards itself)
  const bool pdl = attend_early_ok(ctx);
  if (dm.dtype == KVEVICT_BF16) {
    if (dm.lanes > kMaxLanesSmem) return cudaErrorInvalidValue;
    const int grid = ctx.sm_count * ctx.attend_ctas_per_sm;
    const int nt = dm.g > 8 ? 2 : 1;
    const dim3 blk(kAttendWarps * 32);
    if (dm.d == 128 && nt == 1)
      return launch_k(attend_bf16_kernel<128, 1>, dim3(grid), blk, Bf16Cfg<128, 1>::smem_for(dm.lanes), stream, pdl, a);
    else if (dm.d == 128)
      return launch_k(attend_bf16_kernel<128, 2>, dim3(grid), blk, Bf16Cfg<128, 2>::smem_for(dm.lanes), stream, pdl, a);
    else if (nt == 1)
      return launch_k(attend_bf16_kernel<64, 1>, dim3(grid), blk, Bf16Cfg<64, 1>::smem_for(dm.lanes), stream, pdl, a);
    else
      return launch_k(attend_bf16_kernel<64, 2>, dim3(grid), blk, Bf16Cfg<64, 2>::smem_for(dm.lanes), stream, pdl, a);
  } else {
    const int chunks = (dm.cap + kF32Chunk) / kF32Chunk;   // enough for n = cap - 1 plus the new token
    if (chunks > kMaxSeg) return cudaErrorInvalidValue;
    dim3 grid(chunks, dm.lanes);
    const size_t sm = (static_cast<size_t>(dm.g) * dm.d + dm.g * kF32Chunk + 2 * dm.g) * sizeof(float);
    return launch_k(attend_f32_kernel, grid, dim3(kF32Chunk), sm, stream, pdl, a, dm.d);
  }
  return cudaGetLastError();
}

// The same attention kernels writing their split-K scratch to caller-chosen
// buffers (used by the entry point that allocates nothing); ordinary launch.
cudaError_t launch_attend_into(const Ctx& ctx, int layer, const void* q, const void* k_new, const void* v_new,
                               float* logits, float* part_o, float* part_ml, int32_t* lane_nseg,
                               cudaStream_t stream) {
  const Dims& dm = ctx.dims;
  LayerState ls = layer_state(ctx, layer);
  AttendArgs a;
  a.k_pool = ls.k_pool; a.v_pool = ls.v_pool; a.slot = ls.slot; a.count = ls.count;
  a.q = q; a.k_new = k_new; a.v_new = v_new;
  a.logits = logits; a.part_o = part_o; a.part_ml = part_ml; a.lane_nseg = lane_nseg;
  a.status = ctx.ws.status;
  a.lanes = dm.lanes; a.g = dm.g; a.Hkv = dm.Hkv; a.Hq = dm.Hq; a.cap = dm.cap; a.lcap = dm.lcap;
  a.P = dm.P;
  a.scale2 = 1.4426950408889634f / sqrtf(static_cast<float>(dm.d));
  a.early_trigger = 0;
  a.reads_done = nullptr;   // its own scratch, launched without early start
  a.reads_expect = 0u;
  if (dm.dtype == KVEVICT_BF16) {
    if (dm.lanes > kMaxLanesSmem) return cudaErrorInvalidValue;
    const int grid = ctx.sm_count * ctx.attend_ctas_per_sm;
    const int nt = dm.g > 8 ? 2 : 1;
    const dim3 blk(kAttendWarps * 32);
    if (dm.d == 128 && nt == 1)
      return launch_k(attend_bf16_kernel<128, 1>, dim3(grid), blk, Bf16Cfg<128, 1>::smem_for(dm.lanes), stream, false, a);
    else if (dm.d == 128)
      return launch_k(attend_bf16_kernel<128, 2>, dim3(grid), blk, Bf16Cfg<128, 2>::smem_for(dm.lanes), stream, false, a);
    else if (nt == 1)
      return launch_k(attend_bf16_kernel<64, 1>, dim3(grid), blk, Bf16Cfg<64, 1>::smem_for(dm.lanes), stream, false, a);
    return launch_k(attend_bf16_kernel<64, 2>, dim3(grid), blk, Bf16Cfg<64, 2>::smem_for(dm.lanes), stream, false, a);
  }
  const int chunks = (dm.cap + kF32Chunk) / kF32Chunk;
  if (chunks > kMaxSeg) return cudaErrorInvalidValue;
  const size_t sm = (static_cast<size_t>(dm.g) * dm.d + dm.g * kF32Chunk + 2 * dm.g) * sizeof(float);
  return launch_k(attend_f32_kernel, dim3(chunks, dm.lanes), dim3(kF32Chunk), sm, stream, false, a, dm.d);
}

}  // namespace kve
