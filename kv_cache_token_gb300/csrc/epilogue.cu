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
// apply: the admissions and relocations of the lanes that asked for blocks
// (vToken review, Sec. 3.3 Stage 3: fill each destination completely, in
// ascending position, and release the sources), claimed lane by lane by the
// epilogue's CTAs once the allocator has published its result, or one CTA per
// lane in a separate kernel.
// Two epilogue kernels: a large one (512 threads, 180 KB of shared memory)
// for every policy and step, and a lean H2O one (128 threads, no dynamic
// shared memory) that fits on an SM beside three CTAs of the attention
// kernel, so the epilogue of one layer runs while the next layer streams.
#include "lane_ops.cuh"

#include <cooperative_groups.h>

namespace kve {
namespace {
namespace cg = cooperative_groups;

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
  int applies;   // admission and relocation done here (no apply kernel follows)
  const void* k_new; const void* v_new;
  float* out; float* lse; int32_t* victims; int32_t* n_victims;
};

constexpr int kGenCounter = 7;   // ws.counters slot: allocator results published (one increment per call)
constexpr int kApplyCount = 8;   // ws.counters slot: lanes in ws.apply_list this call
constexpr int kApplyClaim = 9;   // ws.counters slot: next entry of ws.apply_list to claim
constexpr int kLeanThreads = 128;   // lean H2O epilogue: threads per CTA (one lane)
constexpr int kLeanWarps = kLeanThreads / 32;
constexpr int kLeanU = 4;           // lean H2O epilogue: tokens a thread has in flight in the weight pass
constexpr int kShiftU = 8;          // lean H2O epilogue: table entries a thread moves per round of the shift

template <typename KT>
__device__ void apply_lane(const LayerState& ls, const Workspace& ws, const Dims& dm, const int l,
                           const void* k_new, const void* v_new, int mark_freed, int32_t* moves, int* sh_scan,
                           int* sh_mv_src, int* sh_mv_dst);

template <typename KT>
__device__ __forceinline__ void copy_row(KT* dst, const KT* src, int d) {
  for (int e = threadIdx.x; e < d; e += blockDim.x) dst[e] = src[e];
}

template <typename KT, bool kRing>
__device__ __forceinline__ void lane_step(const EpiArgs& A, const LaneRefs& L, const int l, const int n,
                                          unsigned char* dsm, int* sh_work, int* sh_gen);
__device__ void allocate_layer(const LayerState& ls, const Workspace& ws, const Dims& dm, int* sh_scan,
                               int* sh_flag);

// 2^x by the hardware approximation (PTX ex2.approx.ftz, relative error
// about 2^-22; results below 2^-126 flush to zero).
__device__ __forceinline__ float hw_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// DropKV decode variant: this step's residual-output score of every kept
// token, written to column rs of its history-ring row: the sum over the
// group's heads of p / (1 - p) * ||a_h - v|| (DropKV explainer, Lemma 1, with
// the window reduced to the current query of each head), 1 - p from expm1
// when p > 1/2, +inf where 1 - p <= 0, no term where p = 0.  sh_a holds the
// heads' outputs a_h (g x d floats), lg the base-2 scaled logits (one row of
// lcap per head).  The ring row of a token is the one at its slot; hrows
// (if not null) holds the kept tokens' rows in shared memory, ld apart, and
// gets the scores too.
//
// Eight lanes share a token: each loads CPL 16-byte pieces of its V row
// (lanes side by side, so a group reads 128 contiguous bytes per load) and
// the group keeps kU tokens' rows in flight before any arithmetic.  The
// distances are taken directly in fp32 (no expansion, so no cancellation when
// a_h is close to v), four heads at a time, summed across the group; the
// p / (1 - p) factors of a token's four heads are spread over its lanes.
// The monotone image (mono_key) of +0.0.
constexpr unsigned long long kKeyZero = 0x8000000000000000ull;

// The window sum of one history row (column rs replaced by w when rs >= 0),
// as its monotone key: the float64 sum in slot order 0 upward (SnapKV, "How
// it works").  When the row's nonzero entries are finite, normal and their
// exponents lie within `spread` of each other (spread + 24 + log2 W <= 53),
// every partial sum of that order is exact in float64, so the sum is the
// exact one; it is then taken in 64-bit integer arithmetic (significands
// aligned to the smallest exponent) and converted once, exactly.  Other rows
// are summed in float64.
template <int kW>   // kW > 0: the row length at compile time; 0: W at run time
__device__ __forceinline__ unsigned long long window_key(const float* row, const int Wr, const int rs, const float w,
                                                        const int spread) {
  const int W = kW > 0 ? kW : Wr;
  unsigned umax = 0u, umin1 = 0xFFFFFFFFu;     // umin1: smallest nonzero bit pattern minus 1
#pragma unroll
  for (int t = 0; t < W; ++t) {
    const unsigned u = __float_as_uint(t == rs ? w : row[t]);
    umax = max(umax, u);
    umin1 = min(umin1, u - 1u);
  }
  if (umax == 0u) return kKeyZero;
  const int emax = static_cast<int>(umax >> 23), emin = static_cast<int>((umin1 + 1u) >> 23);
  if (umax < 0x7F800000u && emin >= 1 && emax - emin <= spread) {
    unsigned long long acc = 0ull;
#pragma unroll
    for (int t = 0; t < W; ++t) {
      const unsigned u = __float_as_uint(t == rs ? w : row[t]);
      const unsigned long long m = u != 0u ? static_cast<unsigned long long>((u & 0x7FFFFFu) | 0x800000u) : 0ull;
      acc += m << max(static_cast<int>(u >> 23) - emin, 0);
    }
    // acc < 2^53: exact as a double; the scale 2^(emin - 150) is a normal power of two
    const double v = static_cast<double>(acc) * __longlong_as_double(static_cast<long long>(emin - 150 + 1023) << 52);
    return static_cast<unsigned long long>(__double_as_longlong(v)) | kKeyZero;
  }
  double sum = 0.0;
  for (int t = 0; t < W; ++t) sum += static_cast<double>(t == rs ? w : row[t]);
  return mono_key(sum);
}

// Starts asynchronous copies of the history rows of a lane's n kept tokens
// (at their slots; W a multiple of 4) to rows[i * ld + t], t < W, in 16-byte
// pieces, consecutive lanes on consecutive pieces; a row whose slot is out
// of range is zero.  The slots go through sh_slot (n ints) first, so no copy
// waits on a slot load.  All threads of the CTA take part.
__device__ __forceinline__ void stage_history_async(const LaneRefs& L, const int n, const int W, const int ld,
                                                    const int nslot, float* rows, int* sh_slot) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int s = L.slot[i];
    sh_slot[i] = (s >= 0 && s < nslot) ? s : -1;
  }
  __syncthreads();
  const int pr = W / 4;     // pieces per row
  for (int e = threadIdx.x; e < n * pr; e += blockDim.x) {
    const int i = e / pr, c = (e - i * pr) * 4;
    const int s = sh_slot[i];
    float* dst = rows + i * ld + c;
    if (s >= 0) {
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)),
                   "l"(L.ring + static_cast<size_t>(s) * W + c) : "memory");
    } else {
      *reinterpret_cast<float4*>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  cp_async_commit();
}

// window_key of a 16-byte aligned row with W a multiple of 4 (no column
// replaced), read four floats at a time.
template <int kW>
__device__ __forceinline__ unsigned long long window_key4(const float* row, const int Wr, const int spread) {
  const int W4 = (kW > 0 ? kW : Wr) / 4;
  const uint4* r4 = reinterpret_cast<const uint4*>(row);
  unsigned umax = 0u, umin1 = 0xFFFFFFFFu;
#pragma unroll
  for (int q = 0; q < W4; ++q) {
    const uint4 v = r4[q];
    umax = max(max(umax, max(v.x, v.y)), max(v.z, v.w));
    umin1 = min(min(umin1, min(v.x - 1u, v.y - 1u)), min(v.z - 1u, v.w - 1u));
  }
  if (umax == 0u) return kKeyZero;
  const int emax = static_cast<int>(umax >> 23), emin = static_cast<int>((umin1 + 1u) >> 23);
  if (umax < 0x7F800000u && emin >= 1 && emax - emin <= spread) {
    unsigned long long acc = 0ull;
    auto add = [&](const unsigned u) {
      const unsigned long long m = u != 0u ? static_cast<unsigned long long>((u & 0x7FFFFFu) | 0x800000u) : 0ull;
      acc += m << max(static_cast<int>(u >> 23) - emin, 0);
    };
#pragma unroll
    for (int q = 0; q < W4; ++q) {
      const uint4 v = r4[q];
      add(v.x); add(v.y); add(v.z); add(v.w);
    }
    const double v = static_cast<double>(acc) * __longlong_as_double(static_cast<long long>(emin - 150 + 1023) << 52);
    return static_cast<unsigned long long>(__double_as_longlong(v)) | kKeyZero;
  }
  double sum = 0.0;
  for (int t = 0; t < 4 * W4; ++t) sum += static_cast<double>(row[t]);
  return mono_key(sum);
}

// window_key in two parts, for a row whose column rs changes last: the
// part over the other columns (before the new value is known), then the key
// once it is (merge).  merge returns exactly window_key(row with column rs
// = w): the exact-sum condition of the whole row implies the others' one,
// so their aligned integer sum is valid and re-aligns exactly to the
// row's smallest exponent; otherwise it sums the row in float64 in slot
// order as window_key does.
struct WindowPart {
  unsigned long long acc;   // the others' significands aligned to their smallest exponent (valid when the row's test passes)
  unsigned umax, umin1;     // largest bit pattern, smallest nonzero one minus 1, over the other columns
};
__device__ __forceinline__ WindowPart window_part(const float* row, const int W, const int rs, const int spread) {
  WindowPart p;
  p.umax = 0u;
  p.umin1 = 0xFFFFFFFFu;
  for (int t = 0; t < W; ++t) {
    if (t == rs) continue;
    const unsigned u = __float_as_uint(row[t]);
    p.umax = max(p.umax, u);
    p.umin1 = min(p.umin1, u - 1u);
  }
  p.acc = 0ull;
  if (p.umax == 0u) return p;
  const int emax = static_cast<int>(p.umax >> 23), emin = static_cast<int>((p.umin1 + 1u) >> 23);
  if (p.umax < 0x7F800000u && emin >= 1 && emax - emin <= spread) {
    for (int t = 0; t < W; ++t) {
      if (t == rs) continue;
      const unsigned u = __float_as_uint(row[t]);
      const unsigned long long m = u != 0u ? static_cast<unsigned long long>((u & 0x7FFFFFu) | 0x800000u) : 0ull;
      p.acc += m << max(static_cast<int>(u >> 23) - emin, 0);
    }
  }
  return p;
}
__device__ __forceinline__ unsigned long long window_merge(const WindowPart& p, const float w, const float* row,
                                                           const int W, const int rs, const int spread) {
  const unsigned uw = __float_as_uint(w);
  const unsigned umax = max(p.umax, uw), umin1 = min(p.umin1, uw - 1u);
  if (umax == 0u) return kKeyZero;
  const int emax = static_cast<int>(umax >> 23), emin = static_cast<int>((umin1 + 1u) >> 23);
  if (umax < 0x7F800000u && emin >= 1 && emax - emin <= spread) {
    unsigned long long acc = 0ull;
    if (p.umax != 0u) acc = p.acc << (static_cast<int>((p.umin1 + 1u) >> 23) - emin);
    if (uw != 0u) acc += static_cast<unsigned long long>((uw & 0x7FFFFFu) | 0x800000u) << (static_cast<int>(uw >> 23) - emin);
    const double v = static_cast<double>(acc) * __longlong_as_double(static_cast<long long>(emin - 150 + 1023) << 52);
    return static_cast<unsigned long long>(__double_as_longlong(v)) | kKeyZero;
  }
  double sum = 0.0;
  for (int t = 0; t < W; ++t) sum += static_cast<double>(t == rs ? w : row[t]);
  return mono_key(sum);
}

// One 16-byte piece of a K or V row as floats (8 bf16 or 4 fp32).
template <typename KT>
__device__ __forceinline__ void piece_to_float(const uint4 w, float* x);
template <>
__device__ __forceinline__ void piece_to_float<__nv_bfloat16>(const uint4 w, float* x) {
  const unsigned u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = __uint_as_float(u[k] << 16);
    x[2 * k + 1] = __uint_as_float(u[k] & 0xFFFF0000u);
  }
}
template <>
__device__ __forceinline__ void piece_to_float<float>(const uint4 w, float* x) {
  x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y); x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
}

// Tokens i_lo .. i_hi - 1: the score goes to ring column rs of the tokens in
// [own_lo, own_hi) and to row i - i_lo of hrows (if given) for all of them.
template <typename KT, int CPL>
__device__ __forceinline__ void dropkv_ring_scores(const EpiArgs& A, const LaneRefs& L, const int i_lo, const int i_hi,
                                                const int own_lo, const int own_hi, const float* sh_a,
                                                const float* lg, const float* sh_lse2, const int W, const int rs,
                                                float* hrows, const int ld) {
  constexpr int kEpc = 16 / static_cast<int>(sizeof(KT));   // elements per 16-byte piece
  constexpr int kU = 8 / CPL;                                // tokens per group and pass
  constexpr int kPairs = kU / 2;                             // (token, head) terms per lane
  constexpr int kTokLanes = 4 / kPairs;                      // lanes holding one token's terms
  const Dims& dm = A.dm;
  const int g = dm.g, d = dm.d;
  const int tid = threadIdx.x, sub = tid & 7, grp = tid >> 3, ngrp = blockDim.x >> 3;
  const uint4* vp = static_cast<const uint4*>(A.ls.v_pool);
  const int rowc = d / kEpc;
  const int nslot = dm.P * kBlock;
  const int stride = ngrp * kU;
  const int n = i_hi;
  const int npass = (i_hi - i_lo + stride - 1) / stride;    // the same for every thread (shuffles below)
  for (int ps = 0; ps < npass; ++ps) {
    const int base = i_lo + ps * stride + grp;
    uint4 v[kU][CPL];
    int sl[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = base + u * ngrp;
      int s = -1;
      if (i < n) {
        s = L.slot[i];
        if (s < 0 || s >= nslot) {
          if (sub == 0) set_status(A.ws.status, ST_BAD_INDEX);
          s = -1;
        }
      }
      sl[u] = s;
#pragma unroll
      for (int c = 0; c < CPL; ++c)
        v[u][c] = s >= 0 ? vp[static_cast<size_t>(s) * rowc + sub + 8 * c] : make_uint4(0u, 0u, 0u, 0u);
    }
    float sc = 0.f;
    for (int h0 = 0; h0 < g; h0 += 4) {
      // this lane's factors p / (1 - p), loaded before the distance arithmetic
      float f[kPairs];
#pragma unroll
      for (int j = 0; j < kPairs; ++j) {
        const int q = sub * kPairs + j, h = h0 + (q & 3), i = base + (q >> 2) * ngrp;
        f[j] = 0.f;
        if (h < g && i < n) {
          const float x = lg[static_cast<size_t>(h) * dm.lcap + i] - sh_lse2[h];
          const float p = exp2f(x);
          if (p > 0.f) {
            const float om = p > 0.5f ? -expm1f(x * kLn2) : 1.f - p;
            f[j] = om > 0.f ? p / om : INFINITY;
          }
        }
      }
      float dist[kU][4];
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int hq = 0; hq < 4; ++hq) dist[u][hq] = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const int e0 = (sub + 8 * c) * kEpc;
#pragma unroll
        for (int hq = 0; hq < 4; ++hq) {
          if (h0 + hq < g) {
            float a[kEpc];
            const float4* ap = reinterpret_cast<const float4*>(sh_a + (h0 + hq) * d + e0);
#pragma unroll
            for (int e = 0; e < kEpc / 4; ++e) {
              const float4 t = ap[e];
              a[4 * e] = t.x; a[4 * e + 1] = t.y; a[4 * e + 2] = t.z; a[4 * e + 3] = t.w;
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
              float x[kEpc];
              piece_to_float<KT>(v[u][c], x);
#pragma unroll
              for (int e = 0; e < kEpc; ++e) {
                const float df = a[e] - x[e];
                dist[u][hq] = fmaf(df, df, dist[u][hq]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int hq = 0; hq < 4; ++hq)
#pragma unroll
          for (int o = 1; o < 8; o <<= 1) dist[u][hq] += __shfl_xor_sync(0xffffffffu, dist[u][hq], o);
      float t = 0.f;
#pragma unroll
      for (int j = 0; j < kPairs; ++j) {
        const int q = sub * kPairs + j;
        float dd = 0.f;
#pragma unroll
        for (int qq = 0; qq < kU * 4; ++qq)
          if (qq == q) dd = dist[qq >> 2][qq & 3];
        if (f[j] != 0.f) t += f[j] == INFINITY ? INFINITY : f[j] * sqrtf(dd);
      }
#pragma unroll
      for (int o = 1; o < kTokLanes; o <<= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      sc += t;
    }
    int s = -1;
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (u == sub / kTokLanes) s = sl[u];
    const int it = base + (sub / kTokLanes) * ngrp;
    if (sub % kTokLanes == 0 && it < n) {
      if (s >= 0 && it >= own_lo && it < own_hi) L.ring[static_cast<size_t>(s) * W + rs] = sc;
      if (hrows) hrows[(it - i_lo) * ld + rs] = sc;
    }
  }
}

// Marks this lane's epilogue done (thread 0 only; nsig CTAs signal, one a lane).  The per-lane requests
// the allocator reads (need_admit, want_dst, plan_tlive, count, released
// block owners) are written before (by any thread of the CTA, ordered by a
// barrier before this call); the release makes them visible to the last CTA.  The done counter carries the number of lanes asking for blocks
// in its upper bits, so the common no-work case needs no further atomic.
__device__ __forceinline__ void signal_done(const Workspace& ws, bool work, int* sh_last, int* sh_flag, int nsig) {
  const int old = atomic_add_release(ws.epi_done, 1 + (work ? kWorkUnit : 0));
  *sh_last = (old & (kWorkUnit - 1)) == nsig - 1;
  *sh_flag = (old >> kWorkShift) + (work ? 1 : 0);
}

// Right after the dependency wait (thread 0): the allocator-result
// generation before this CTA signals (it changes only after every CTA of the
// grid has signalled, and the previous layer's epilogue, which also
// publishes one, is complete by now).
__device__ __forceinline__ void read_generation(const EpiArgs& A, int* sh_gen) {
  if (threadIdx.x == 0) *sh_gen = A.applies ? __ldcg(A.ws.counters + kGenCounter) : 0;
}

// H2O with at most one victim (the steady state of a full cache), all
// threads of the CTA.  Before the dependency wait: the lane's token table
// (kFastPer tokens a thread), its block list with the live masks (kFastPer
// blocks a thread) and the new token's K/V row, none of which the attention
// kernel or another layer's epilogue writes; from the masks, each warp's
// lowest free slot.  After it: logits and split-K partial outputs by bulk
// copy into shared memory, split-K statistics by plain loads.  The minimum
// (key, position) and its slot come from three warp reductions and one
// barrier; the holder of the victim's block decides from the mask it already
// holds whether the block empties.  The fragmentation test of Eq. (1) is
// evaluated before the wait for each of the eight outcomes the scoring can
// have (double division is slow on this part).  The done counter goes out
// (release) once the table is rewritten: another CTA may apply this lane's
// admission or relocation, which reads the table.
template <typename KT>
__device__ __forceinline__ void h2o_fast_step(const EpiArgs& A, const LaneRefs& L, const int n, unsigned char* dsm,
                                              int* sh_sig, int* sh_last, int* sh_flag, int* sh_gen,
                                              int* sh_work) {
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
  const int cbuf = A.layer % kScratchBufs;
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
  read_generation(A, sh_gen);
  // a request of this lane left non-zero (the invariant is that none is)
  const bool stale_req = tid == 0 && (__ldcg(A.ws.need_admit + l) | __ldcg(A.ws.want_dst + l)) != 0;

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
  // The allocator reads a lane's requests (and its count) only when they are
  // non-zero; between steps they hold zero (applying them clears what was
  // consumed).  A lane that asks for blocks, released a block or clears a
  // request left over signals with release semantics once its table is
  // rewritten; the writes of the others are of no concern to the allocator.
  const bool publish = work || dead_j >= 0 || stale_req;
  if (tid == 0) {
    A.ls.count[l] = m + 1;
    if (m + 1 >= dm.cap) set_status(A.ws.status, ST_CAPACITY);
    if (work || stale_req) {
      A.ws.need_admit[l] = need ? 1 : 0;
      A.ws.want_dst[l] = ndst;
      A.ws.plan_tlive[l] = t_live;
    }
    if (work) atomicOr(A.ws.work_flag, 1);
    *sh_work = work ? 1 : 0;
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
  // the done counter, once every thread's table writes are ordered before it;
  // its old value is only needed at the end, so its round trip overlaps the
  // output combine
  __syncthreads();
  int done_old = 0;
  if (tid == 0) {
    const int inc = 1 + (work ? kWorkUnit : 0);
    done_old = publish ? atomic_add_release(A.ws.epi_done, inc) : atomicAdd(A.ws.epi_done, inc);
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

// Waits until *p differs from `old` (acquire), for a bounded number of polls;
// false if it did not change (not an error: see epilogue_tail).
__device__ __forceinline__ bool wait_changed_quiet(const int* p, int old) {
  for (int polls = 0; polls < (1 << 20); ++polls) {
    if (ld_acquire_gpu(p) != old) return true;
    __nanosleep(64);
  }
  return false;
}

// Applies lanes of ws.apply_list until none is left unclaimed (all threads of
// the CTA; the list and its count are published).
template <typename KT>
__device__ __forceinline__ void apply_claimed(const EpiArgs& A, int* sh_scan, int* mv_src, int* mv_dst) {
  __shared__ int sh_claim;
  const int total = __ldcg(A.ws.counters + kApplyCount);
  for (;;) {
    if (threadIdx.x == 0) sh_claim = atomicAdd(A.ws.counters + kApplyClaim, 1);
    __syncthreads();
    const int c = sh_claim;
    __syncthreads();
    if (c >= total) break;
    apply_lane<KT>(A.ls, A.ws, A.dm, __ldcg(A.ws.apply_list + c), A.k_new, A.v_new, 0, nullptr, sh_scan, mv_src,
                   mv_dst);
    __syncthreads();
  }
}

// The end of every epilogue CTA (all threads), after its lane's step.  The
// last CTA of the grid to finish runs the layer allocator, if any lane asked
// for blocks.  With A.applies, admissions into fresh blocks and relocations
// are applied here instead of in an apply kernel: the last CTA publishes the
// allocator's result (a release store of the generation counter), then
// claims the listed lanes one by one; a CTA whose own lane asked for blocks
// waits for that result (bounded) and claims lanes too.  A waiter that gives
// up simply leaves: whatever nobody else claims, the last CTA applies, so no
// lane is left half-applied whatever else occupies the GPU.
template <typename KT>
__device__ __forceinline__ void epilogue_tail(const EpiArgs& A, int* sh_scan, int* sh_work, int* sh_last,
                                              int* sh_flag, const int* sh_sig, const int* sh_gen, int* mv_src,
                                              int* mv_dst, int nsig) {
  __shared__ int sh_go;
  const int tid = threadIdx.x;
  __syncthreads();
  if (!*sh_sig) {
    if (tid == 0) signal_done(A.ws, *sh_work != 0, sh_last, sh_flag, nsig);
    __syncthreads();
  }
  if (*sh_last) {
    if (*sh_flag == 0) {
      if (tid == 0) {
        *A.ws.epi_done = 0;
        A.ws.counters[1] = 0; A.ws.counters[2] = 0; A.ws.counters[kApplyCount] = 0;
      }
    } else {
      if (tid == 0) *A.ws.epi_done = 0;
      __threadfence();
      allocate_layer(A.ls, A.ws, A.dm, sh_scan, sh_flag);
    }
  }
  if (!A.applies) return;
  if (*sh_last) {
    __syncthreads();   // the allocator's stores by every thread of this CTA
    if (tid == 0) {
      __threadfence();
      st_release_gpu(A.ws.counters + kGenCounter, *sh_gen + 1);
    }
    apply_claimed<KT>(A, sh_scan, mv_src, mv_dst);
    return;
  }
  if (tid == 0) sh_go = *sh_work != 0 && wait_changed_quiet(A.ws.counters + kGenCounter, *sh_gen);
  __syncthreads();
  if (sh_go) apply_claimed<KT>(A, sh_scan, mv_src, mv_dst);
}

// The end of an epilogue CTA: it is done with its scratch copy and with its
// layer's tables (release, after every thread's last access), for the
// attention kernels that guard themselves on the copy's count.
__device__ __forceinline__ void scratch_released(const EpiArgs& A) {
  __syncthreads();
  if (threadIdx.x == 0) (void)atomic_add_release(reinterpret_cast<int*>(A.ws.reads_done) + A.layer % kScratchBufs, 1);
}

// kRing: the policy keeps a history ring (SnapKV, DropKV decode variant);
// the H2O instantiation carries none of that code.
template <typename KT, bool kRing>
__global__ void __launch_bounds__(kEpiThreads, 1) decode_epilogue_kernel(EpiArgs A) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ int sh_scan[40];
  __shared__ int sh_work, sh_last, sh_flag, sh_sig, sh_gen;
  const Dims& dm = A.dm;
  const int l = blockIdx.x, tid = threadIdx.x;
  LaneRefs L = lane_refs(A.ls, dm, l);
  // The token count (and, on the fast path, the token table and the block
  // list) is not written by the attention kernel: it is read before the
  // dependency wait, while the attention kernel drains.
  const int n = __ldcg(A.ls.count + l);
  if (tid == 0) { sh_work = 0; sh_sig = 0; sh_gen = 0; }
  if (n < 0 || n >= dm.cap) {
    grid_dep_wait();
    grid_dep_launch();
    read_generation(A, &sh_gen);
    if (tid == 0) {
      set_status(A.ws.status, ST_CAPACITY);
      A.n_victims[l] = 0; A.ws.need_admit[l] = 0; A.ws.want_dst[l] = 0; A.ws.plan_tlive[l] = 0;
    }
  } else if (!kRing && n + 1 - dm.budget <= 1 && n <= kFastN && dm.g <= 8 && dm.d <= 128 && (dm.d & 1) == 0) {
    h2o_fast_step<KT>(A, L, n, dsm, &sh_sig, &sh_last, &sh_flag, &sh_gen, &sh_work);
  } else {
    lane_step<KT, kRing>(A, L, l, n, dsm, &sh_work, &sh_gen);
  }
  // the step is done with the dynamic shared memory: the relocation's move
  // lists go there
  int* mv = reinterpret_cast<int*>(dsm);
  epilogue_tail<KT>(A, sh_scan, &sh_work, &sh_last, &sh_flag, &sh_sig, &sh_gen, mv, mv + kApplyThreads,
                    static_cast<int>(gridDim.x));
  scratch_released(A);
}

// H2O with at most one victim (the steady state of a full cache) in a CTA of
// kLeanThreads threads with no dynamic shared memory (the lean epilogue).
// Before the dependency wait it reads only what neither the attention kernel
// nor another layer's epilogue writes: the lane's
// scores (kLeanPer a thread, in registers), its positions (the candidates
// outside the recent window are a prefix of the table, since positions
// ascend: it counts them), its block list and live masks (each warp's lowest
// free slot), the new token's K/V row; and it pulls the lane's slots into L2.
// After it: the split-K statistics give each head's log-sum-exp; one pass
// reads each token's logits from L2 (kLeanU tokens a thread in flight), adds
// its group weight to its score (written in place) and keeps the minimum
// candidate (key, index: the index orders like the position); the victim's
// live bit is cleared (an emptied block is released and dropped from the
// list); the new token takes the lowest free slot; the entries after the
// victim move down one place; the done counter goes out (release) once the
// table is written; then the split-K output combine, 8 elements of one head
// a thread, eight segments in flight.  The same results as h2o_fast_step.
constexpr int kLeanPer = 32;   // tokens a thread holds: lanes of up to kLeanPer * kLeanThreads tokens
template <typename KT>
__device__ __forceinline__ void h2o_lean_step(const EpiArgs& A, const LaneRefs& L, const int n, int* sh_sig,
                                              int* sh_last, int* sh_flag, int* sh_gen, int* sh_work) {
  __shared__ float sh_rL[8], sh_lse2[8];
  __shared__ float sh_scale[8][kMaxSeg];   // per head, per split-K segment
  __shared__ unsigned sh_over;
  __shared__ unsigned sh_wkey[kLeanWarps], sh_widx[kLeanWarps];
  __shared__ unsigned sh_wfree[kLeanWarps], sh_wfree2[kLeanWarps];
  __shared__ int sh_ncand[kLeanWarps];
  __shared__ int sh_nan, sh_late, sh_dead, sh_dead_j, sh_vpos, sh_vslot;
  __shared__ int sh_scan2[40];
  constexpr unsigned kNone = 0xFFFFFFFFu;
  const Dims& dm = A.dm;
  const int l = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = l / dm.Hkv, kh = l % dm.Hkv, g = dm.g, d = dm.d;
  const int cbuf = A.layer % kScratchBufs;
  const int k = max(0, n + 1 - dm.budget);          // 0 or 1
  const int cut = A.new_pos - dm.R + 1;

  // ---- before the dependency wait -----------------------------------------------
  if (tid == 0) { sh_nan = 0; sh_late = 0; sh_dead = -1; sh_dead_j = -1; }
  float sc[kLeanPer];
  int ncand = 0;
#pragma unroll
  for (int j = 0; j < kLeanPer; ++j) {
    const int i = tid + j * kLeanThreads;
    sc[j] = 0.f;
    if (i < n) {
      sc[j] = __ldcg(L.score + i);
      ncand += __ldcg(L.pos + i) < cut ? 1 : 0;
      if (lane == 0 || lane == 31) prefetch_l2(L.slot + i);
    }
  }
  ncand = warp_sum(ncand);
  if (lane == 0) sh_ncand[warp] = ncand;
  const int nb = min(max(__ldcg(L.nblocks), 0), dm.cap);
  {
    // lowest free slot of the lane's blocks before this step's eviction
    unsigned fr = kNone;
    bool bad_blk = false;
    for (int j = tid; j < nb; j += kLeanThreads) {
      const int blk = __ldcg(L.blocks + j);
      if (blk < 0 || blk >= dm.P) { bad_blk = true; continue; }
      const int mk = __ldcg(L.mask + blk) & 0xFFFF;
      if (mk != 0xFFFF) fr = min(fr, static_cast<unsigned>(blk * kBlock + (__ffs(~mk) - 1)));
    }
    if (bad_blk) set_status(A.ws.status, ST_BAD_INDEX);
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
  KT knv{}, vnv{};
  if (tid < d) {
    knv = static_cast<const KT*>(A.k_new)[static_cast<size_t>(l) * d + tid];
    vnv = static_cast<const KT*>(A.v_new)[static_cast<size_t>(l) * d + tid];
  }
  // the last kept token must precede the new one
  const bool late = tid == 0 && n > 0 && __ldcg(L.pos + n - 1) >= A.new_pos;

  grid_dep_wait();      // the attention kernel's results are complete and visible
  grid_dep_launch();
  read_generation(A, sh_gen);
  // a request of this lane left non-zero (the invariant is that none is)
  const bool stale_req = tid == 0 && (__ldcg(A.ws.need_admit + l) | __ldcg(A.ws.want_dst + l)) != 0;
  // split-K statistics of all kMaxSeg segments (in bounds), masked below
  const float2* ml = reinterpret_cast<const float2*>(A.ws.part_ml_buf[cbuf]) + static_cast<size_t>(l) * kMaxSeg * g;
  float2 m0[2], m1[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int h = warp + r * kLeanWarps;
    m0[r] = (A.has_q && h < g) ? __ldcg(ml + lane * g + h) : make_float2(-INFINITY, 0.f);
    m1[r] = (A.has_q && h < g) ? __ldcg(ml + (lane + 32) * g + h) : make_float2(-INFINITY, 0.f);
  }
  const int nseg = A.has_q ? min(__ldcg(A.ws.lane_nseg_buf[cbuf] + l), kMaxSeg) : 0;
  // the first round of logits goes out with the statistics (it does not need
  // the log-sum-exp)
  const float* lg = A.ws.logits_buf[cbuf] + static_cast<size_t>(l) * g * dm.lcap;
  float lv0[kLeanU][8];
#pragma unroll
  for (int u = 0; u < kLeanU; ++u) {
    const int i = tid + u * kLeanThreads;
#pragma unroll
    for (int h = 0; h < 8; ++h)
      lv0[u][h] = (A.has_q && h < g && i < n) ? __ldcg(lg + static_cast<size_t>(h) * dm.lcap + i) : 0.f;
  }
  if (__syncthreads_or(late)) {
    if (tid == 0) {
      set_status(A.ws.status, ST_POSITION);
      A.n_victims[l] = 0; A.ws.need_admit[l] = 0; A.ws.want_dst[l] = 0; A.ws.plan_tlive[l] = 0;
    }
    return;
  }
  ncand = 0;
#pragma unroll
  for (int w = 0; w < kLeanWarps; ++w) ncand += sh_ncand[w];
  // ---- per-head log-sum-exp of the split-K segments (a warp per head) ------------
  if (A.has_q) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int h = warp + r * kLeanWarps;
      if (h < g) {
        if (lane >= nseg) m0[r] = make_float2(-INFINITY, 0.f);
        if (lane + 32 >= nseg) m1[r] = make_float2(-INFINITY, 0.f);
        const float M = warp_max(fmaxf(m0[r].x, m1[r].x));
        const float s0 = m0[r].x == -INFINITY ? 0.f : exp2f(m0[r].x - M);
        const float s1 = m1[r].x == -INFINITY ? 0.f : exp2f(m1[r].x - M);
        sh_scale[h][lane] = s0;
        sh_scale[h][lane + 32] = s1;
        float Ls = m0[r].y * s0 + m1[r].y * s1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
        if (lane == 0) {
          sh_rL[h] = 1.f / Ls;
          const float lse2 = M + log2f(Ls);
          sh_lse2[h] = lse2;
          A.lse[static_cast<size_t>(b) * dm.Hq + kh * g + h] = lse2 * kLn2;
        }
      }
    }
  }
  __syncthreads();

  // ---- weights -> scores (in place); candidate minimum (key, index) ---------------
  unsigned ck = kNone, ci = kNone;
  int nan_count = 0;
#pragma unroll
  for (int j0 = 0; j0 < kLeanPer; j0 += kLeanU) {
    if (tid + j0 * kLeanThreads < n) {
      float lv[kLeanU][8];
#pragma unroll
      for (int u = 0; u < kLeanU; ++u) {
        const int i = tid + (j0 + u) * kLeanThreads;
#pragma unroll
        for (int h = 0; h < 8; ++h)
          lv[u][h] = j0 == 0 ? lv0[u][h]
                             : (A.has_q && h < g && i < n) ? __ldcg(lg + static_cast<size_t>(h) * dm.lcap + i) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kLeanU; ++u) {
        const int i = tid + (j0 + u) * kLeanThreads;
        if (i < n) {
          float s = sc[j0 + u];
          if (A.has_q) {
            float w = 0.f;
#pragma unroll
            for (int h = 0; h < 8; ++h)
              if (h < g) w += hw_exp2(lv[u][h] - sh_lse2[h]);
            s += w;
            L.score[i] = s;
          }
          if (s != s) ++nan_count;
          if (k == 1 && i < ncand) {
            const unsigned kk = static_cast<unsigned>(mono_key(s));
            if (kk < ck) { ck = kk; ci = static_cast<unsigned>(i); }   // ascending i: ties keep the lower index
          }
        }
      }
    }
  }
  {
    const unsigned wk = __reduce_min_sync(0xffffffffu, ck);
    const unsigned wi = __reduce_min_sync(0xffffffffu, ck == wk ? ci : kNone);
    if (lane == 0) { sh_wkey[warp] = wk; sh_widx[warp] = wi; }
  }
  nan_count = warp_sum(nan_count);
  if (lane == 0 && nan_count) atomicAdd(&sh_nan, nan_count);
  __syncthreads();
  unsigned vidx;
  {
    const bool in = lane < kLeanWarps;
    const unsigned k1 = in ? sh_wkey[lane] : kNone;
    const unsigned vkey = __reduce_min_sync(0xffffffffu, k1);
    vidx = __reduce_min_sync(0xffffffffu, (in && k1 == vkey) ? sh_widx[lane] : kNone);
  }
  const bool has_victim = k == 1 && vidx != kNone;
  const int vi = static_cast<int>(vidx);
  // the first round of the table shift (entries after the victim) goes out
  // before the eviction's round trips
  int sp[kShiftU], ssl[kShiftU];
  float ssc[kShiftU];
#pragma unroll
  for (int u = 0; u < kShiftU; ++u) {
    const int i = vi + 1 + u * kLeanThreads + tid;
    if (has_victim && i < n) { sp[u] = __ldcg(L.pos + i); ssl[u] = __ldcg(L.slot + i); ssc[u] = L.score[i]; }
  }
  // ---- eviction: the victim's slot is released; an emptied block is freed ---------
  if (tid == 0) {
    int vslot = -1, vpos = -1;
    if (has_victim) {
      vpos = __ldcg(L.pos + vi);
      vslot = __ldcg(L.slot + vi);
      if (vslot >= 0 && vslot < dm.P * kBlock) {
        const int vb = vslot >> 4, vbit = 1 << (vslot & 15);
        const int old = atomicAnd(&L.mask[vb], ~vbit);
        if (((old & 0xFFFF) & ~vbit) == 0) {
          L.owner[vb] = -1;
          sh_dead = vb;
        }
      } else if (vslot >= 0) {
        set_status(A.ws.status, ST_BAD_INDEX);
      }
    }
    sh_vpos = vpos;
    sh_vslot = vslot;
  }
  __syncthreads();
  const int dead_blk = sh_dead;
  const int vslot = sh_vslot;
  const bool vslot_ok = has_victim && vslot >= 0 && vslot < dm.P * kBlock;
  const int vcount = has_victim ? 1 : 0;
  int nb2 = nb;
  unsigned best;
  if (dead_blk < 0) {
    // the victim's slot is now free too
    unsigned pre = lane < kLeanWarps ? sh_wfree[lane] : kNone;
    pre = __reduce_min_sync(0xffffffffu, pre);
    best = min(pre, vslot_ok ? static_cast<unsigned>(vslot) : kNone);
  } else {
    // rare: the victim emptied its block; drop it from the list (the last
    // entry moves into its place) and look for a free slot in the others
    unsigned fr = kNone;
    for (int j = tid; j < nb; j += kLeanThreads) {
      const int blk = __ldcg(L.blocks + j);
      if (blk == dead_blk) {
        sh_dead_j = j;
      } else if (blk >= 0 && blk < dm.P) {
        const int mk = __ldcg(L.mask + blk) & 0xFFFF;
        if (mk != 0xFFFF) fr = min(fr, static_cast<unsigned>(blk * kBlock + (__ffs(~mk) - 1)));
      }
    }
    fr = __reduce_min_sync(0xffffffffu, fr);
    if (lane == 0) sh_wfree2[warp] = fr;
    __syncthreads();
    if (tid == 0 && sh_dead_j >= 0) {
      L.blocks[sh_dead_j] = __ldcg(L.blocks + nb - 1);
      *L.nblocks = nb - 1;
    }
    best = lane < kLeanWarps ? sh_wfree2[lane] : kNone;
    best = __reduce_min_sync(0xffffffffu, best);
    nb2 = sh_dead_j >= 0 ? nb - 1 : nb;
    __syncthreads();
  }
  const bool need = best == kNone;
  const int m = n - vcount;
  // ---- admission into the lowest free slot; relocation plan --------------------------
  if (!need && tid == 0) atomicOr(&L.mask[best >> 4], 1 << (best & 15));
  __syncthreads();
  int t_live = 0;
  const int outcome = vcount | (dead_blk >= 0 ? 2 : 0) | (need ? 4 : 0);
  const int ndst = lane_plan_given(L, nb2, ((sh_over >> outcome) & 1u) != 0, false, need, &t_live, sh_scan2);
  const bool work = need || ndst > 0;
  // the allocator reads a lane's requests only when they are non-zero (see
  // h2o_fast_step)
  const bool publish = work || dead_blk >= 0 || stale_req;
  if (tid == 0) {
    A.ls.count[l] = m + 1;
    if (m + 1 >= dm.cap) set_status(A.ws.status, ST_CAPACITY);
    if (work || stale_req) {
      A.ws.need_admit[l] = need ? 1 : 0;
      A.ws.want_dst[l] = ndst;
      A.ws.plan_tlive[l] = t_live;
    }
    if (work) atomicOr(A.ws.work_flag, 1);
    *sh_work = work ? 1 : 0;
  }
  // ---- the table: entries after the victim move down one place; every read of a
  // round precedes its barrier, the round's writes (one index lower) follow it -------
  if (has_victim) {
    if (tid == 0) A.victims[static_cast<size_t>(l) * dm.cap] = sh_vpos;
    // round 0 was read before the eviction's barriers
#pragma unroll
    for (int u = 0; u < kShiftU; ++u) {
      const int i = vi + 1 + u * kLeanThreads + tid;
      if (i < n) { L.pos[i - 1] = sp[u]; L.slot[i - 1] = ssl[u]; L.score[i - 1] = ssc[u]; }
    }
    for (int base = vi + 1 + kLeanThreads * kShiftU; base < n; base += kLeanThreads * kShiftU) {
#pragma unroll
      for (int u = 0; u < kShiftU; ++u) {
        const int i = base + u * kLeanThreads + tid;
        if (i < n) { sp[u] = __ldcg(L.pos + i); ssl[u] = __ldcg(L.slot + i); ssc[u] = L.score[i]; }
      }
      __syncthreads();
#pragma unroll
      for (int u = 0; u < kShiftU; ++u) {
        const int i = base + u * kLeanThreads + tid;
        if (i < n) { L.pos[i - 1] = sp[u]; L.slot[i - 1] = ssl[u]; L.score[i - 1] = ssc[u]; }
      }
    }
  }
  __syncthreads();
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
    if (dead_blk >= 0) atomicAdd(reinterpret_cast<unsigned long long*>(&A.ls.stats[SC_FREED_DEAD]), 1ull);
    if (sh_nan) atomicAdd(reinterpret_cast<unsigned long long*>(&A.ls.stats[SC_NAN_KEYS]), (unsigned long long)sh_nan);
    if (l == 0) atomicAdd(reinterpret_cast<unsigned long long*>(&A.ls.stats[SC_STEPS]), 1ull);
  }
  // the done counter, once every thread's table writes are ordered before it
  __syncthreads();
  int done_old = 0;
  if (tid == 0) {
    const int inc = 1 + (work ? kWorkUnit : 0);
    done_old = publish ? atomic_add_release(A.ws.epi_done, inc) : atomicAdd(A.ws.epi_done, inc);
  }
  // ---- output: combine the split-K partial outputs; a thread owns 8 adjacent
  // elements of one head, four segments' loads in flight ----------------------------
  if (A.has_q) {
    const float* po = A.ws.part_o_buf[cbuf] + static_cast<size_t>(l) * kMaxSeg * g * d;
    const bool out16 = (reinterpret_cast<uintptr_t>(A.out) & 15) == 0;
    for (int q8 = tid; q8 < (g * d) >> 3; q8 += kLeanThreads) {
      const int he = q8 * 8, h = he / d, e = he - h * d;
      float acc[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) acc[t] = 0.f;
      for (int s0 = 0; s0 < nseg; s0 += 8) {
        float4 x[8][2];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int s2 = s0 + u;
          const float4* src = reinterpret_cast<const float4*>(po + (static_cast<size_t>(s2) * g + h) * d + e);
          x[u][0] = s2 < nseg ? __ldcg(src) : make_float4(0.f, 0.f, 0.f, 0.f);
          x[u][1] = s2 < nseg ? __ldcg(src + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float c = s0 + u < nseg ? sh_scale[h][s0 + u] : 0.f;
          acc[0] = fmaf(x[u][0].x, c, acc[0]); acc[1] = fmaf(x[u][0].y, c, acc[1]);
          acc[2] = fmaf(x[u][0].z, c, acc[2]); acc[3] = fmaf(x[u][0].w, c, acc[3]);
          acc[4] = fmaf(x[u][1].x, c, acc[4]); acc[5] = fmaf(x[u][1].y, c, acc[5]);
          acc[6] = fmaf(x[u][1].z, c, acc[6]); acc[7] = fmaf(x[u][1].w, c, acc[7]);
        }
      }
      const float r = sh_rL[h];
      float* o = A.out + (static_cast<size_t>(b) * dm.Hq + kh * g + h) * d + e;
      if (out16) {
        reinterpret_cast<float4*>(o)[0] = make_float4(acc[0] * r, acc[1] * r, acc[2] * r, acc[3] * r);
        reinterpret_cast<float4*>(o)[1] = make_float4(acc[4] * r, acc[5] * r, acc[6] * r, acc[7] * r);
      } else {
#pragma unroll
        for (int t = 0; t < 8; ++t) o[t] = acc[t] * r;
      }
    }
  }
  if (tid == 0) {
    *sh_last = (done_old & (kWorkUnit - 1)) == static_cast<int>(gridDim.x) - 1;
    *sh_flag = (done_old >> kWorkShift) + (work ? 1 : 0);
    *sh_sig = 1;
  }
}

// The lean H2O epilogue: one CTA of kLeanThreads threads per lane, at most
// 128 registers a thread and no dynamic shared memory, so that one of its
// CTAs shares an SM with three CTAs of the attention kernel (which lets it
// be scheduled from its start): the epilogue of a layer then runs while the
// next layer's attention streams.  Lanes with more than one victim take the
// general step (correct, slower with fewer threads).
template <typename KT>
__global__ void __launch_bounds__(kLeanThreads, 4) decode_epilogue_lean_kernel(EpiArgs A) {
  __shared__ int sh_scan[40];
  __shared__ int sh_work, sh_last, sh_flag, sh_sig, sh_gen;
  __shared__ int sh_mv[2 * kLeanThreads];
  const Dims& dm = A.dm;
  const int l = blockIdx.x, tid = threadIdx.x;
  // The next layer's attention may start now: it works on another layer and
  // another scratch copy, and guards its copy itself.
  grid_dep_launch();
  LaneRefs L = lane_refs(A.ls, dm, l);
  const int n = __ldcg(A.ls.count + l);
  if (tid == 0) { sh_work = 0; sh_sig = 0; sh_gen = 0; }
  if (n < 0 || n >= dm.cap) {
    grid_dep_wait();
    grid_dep_launch();
    read_generation(A, &sh_gen);
    if (tid == 0) {
      set_status(A.ws.status, ST_CAPACITY);
      A.n_victims[l] = 0; A.ws.need_admit[l] = 0; A.ws.want_dst[l] = 0; A.ws.plan_tlive[l] = 0;
    }
  } else if (n + 1 - dm.budget <= 1 && n <= kLeanPer * kLeanThreads && dm.g <= 8 && dm.d <= kLeanThreads &&
             (dm.d & 7) == 0) {
    h2o_lean_step<KT>(A, L, n, &sh_sig, &sh_last, &sh_flag, &sh_gen, &sh_work);
  } else {
    lane_step<KT, false>(A, L, l, n, nullptr, &sh_work, &sh_gen);
  }
  epilogue_tail<KT>(A, sh_scan, &sh_work, &sh_last, &sh_flag, &sh_sig, &sh_gen, sh_mv, sh_mv + kLeanThreads,
                    static_cast<int>(gridDim.x));
  scratch_released(A);
}

// One lane's step after the attention kernel (all threads of the CTA).  dsm
// (the ring policies' row buffer, kEpiDynSmem bytes) is used only with kRing.
// The lane's block list, live masks and new K/V row as read before the
// dependency wait (nothing running writes them), and what the step's single
// eviction changed since: the victim's slot (its live bit is clear now) and
// the block it released (-1: none; that block left the list).
template <typename KT>
struct LanePrefetch {
  const int* blocks;
  const int* masks;
  int nb;
  int victim_slot;
  int dead_blk;
  const KT* k_new;
  const KT* v_new;
};

// After the victims are out (vcount of them; dead: blocks their removal
// released): admission of the new token into the lowest free slot of the
// lane's blocks, the table's new tail, the relocation plan and the
// per-lane requests and statistics (all threads of the CTA owning the lane).
// pf (optional): the block state and new row read ahead (one victim at most).
template <typename KT>
__device__ __forceinline__ void lane_finish(const EpiArgs& A, const LaneRefs& L, const int l, const int n,
                                            const int k, const int vcount, const int dead, const int nan_count,
                                            int* sh_work, int* sh_scan, const LanePrefetch<KT>* pf = nullptr) {
  __shared__ unsigned sh_min[32];
  __shared__ int sh_nan;
  const Dims& dm = A.dm;
  const int tid = threadIdx.x, d = dm.d, W = dm.W;
  if (tid == 0) sh_nan = 0;
  const int m = n - vcount;
  const int nb = (k > 1 && dead > 0) ? lane_prune_blocks(L, l, sh_scan) : *L.nblocks;

  // ---- admission: lowest free slot among the lane's blocks --------------------
  unsigned best = 0xFFFFFFFFu;
  if (pf) {
    for (int j = tid; j < pf->nb; j += blockDim.x) {
      const int blk = pf->blocks[j];
      if (blk == pf->dead_blk) continue;
      int mk = pf->masks[j] & 0xFFFF;
      if (pf->victim_slot >= 0 && (pf->victim_slot >> 4) == blk) mk &= ~(1 << (pf->victim_slot & 15));
      if (mk != 0xFFFF) best = min(best, static_cast<unsigned>(blk * kBlock + (__ffs(~mk) - 1)));
    }
  } else {
    for (int j = tid; j < nb; j += blockDim.x) {
      const int blk = L.blocks[j];
      const int mk = L.mask[blk] & 0xFFFF;
      if (mk != 0xFFFF) best = min(best, static_cast<unsigned>(blk * kBlock + (__ffs(~mk) - 1)));
    }
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
    copy_row(kp + static_cast<size_t>(best) * d,
             pf ? pf->k_new : static_cast<const KT*>(A.k_new) + static_cast<size_t>(l) * d, d);
    copy_row(vp + static_cast<size_t>(best) * d,
             pf ? pf->v_new : static_cast<const KT*>(A.v_new) + static_cast<size_t>(l) * d, d);
    if (L.ring)
      for (int t = tid; t < W; t += blockDim.x) L.ring[static_cast<size_t>(best) * W + t] = 0.f;
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

template <typename KT, bool kRing>
__device__ __forceinline__ void lane_step(const EpiArgs& A, const LaneRefs& L, const int l, const int n,
                                          unsigned char* dsm, int* sh_work, int* sh_gen) {
  __shared__ float sh_M[kMaxG], sh_L[kMaxG], sh_lse2[kMaxG];
  __shared__ __align__(16) int sh_hist[256];   // also read as 64-bit words
  __shared__ int sh_misc[40];
  __shared__ int sh_scan[40];
  __shared__ int sh_ncand;
  __shared__ float sh_scale[kMaxSeg][kMaxG];
  float* sh_rows = reinterpret_cast<float*>(dsm);      // general path: 128 * kMaxW floats
  const Dims& dm = A.dm;
  const int tid = threadIdx.x;
  const int b = l / dm.Hkv, kh = l % dm.Hkv, g = dm.g, d = dm.d;
  const int cbuf = A.layer % kScratchBufs;
  const int policy = dm.policy;
  constexpr bool ringp = kRing;   // SnapKV, DropKV decode variant: history ring keys
  const int W = dm.W;
  // history rows staged whole in shared memory: ld = 4 (mod 32) floats, so
  // the 16-byte reads of eight lanes on eight consecutive rows hit distinct banks
  const int ld = ((W + 27) / 32) * 32 + 4;

  // ---- history rows, before the dependency wait ---------------------------------
  // The ring is not written by the attention kernel, and every kernel before
  // it is complete once it lets this one start, so the rows of all kept
  // tokens are copied to shared memory (when they fit beside the heads'
  // outputs and the keys) while the attention kernel drains.
  float* hrows = kRing ? sh_rows + kMaxG * 128 : nullptr;
  const size_t hkeys_off = ((static_cast<size_t>(kMaxG) * 128 + static_cast<size_t>(n) * ld) * 4 + 7) & ~static_cast<size_t>(7);
  const bool staged_all = ringp && n > 0 && (W & 3) == 0 && hkeys_off + static_cast<size_t>(n + 1) * 8 <= kEpiDynSmem;
  if (staged_all) stage_history_async(L, n, W, ld, dm.P * kBlock, hrows, reinterpret_cast<int*>(dsm + hkeys_off));

  // ---- general path ------------------------------------------------------------
  grid_dep_wait();      // the attention kernel's results are complete and visible
  grid_dep_launch();
  read_generation(A, sh_gen);
  if (tid == 0) sh_ncand = 0;
  if (n > 0 && L.pos[n - 1] >= A.new_pos) {
    if (staged_all) cp_async_wait_all();
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
      if constexpr (kRing) sh_rows[he] = o;    // the heads' outputs, for the DropKV scores below
    }
    __syncthreads();
  }

  // ---- weights -> score state; SnapKV window sums ----------------------------
  if (staged_all) {
    cp_async_wait_all();
    __syncthreads();
  }
  const int rs = ringp ? A.ls.ring_slot[l] : 0;
  unsigned long long* kbuf = A.ws.keys64 ? A.ws.keys64 + static_cast<size_t>(l) * dm.cap : nullptr;
  unsigned long long* pooled = A.ws.pooled64 ? A.ws.pooled64 + static_cast<size_t>(l) * dm.cap : nullptr;
  const float* lg = A.ws.logits_buf[cbuf] + static_cast<size_t>(l) * g * dm.lcap;
  const int k = max(0, n + 1 - dm.budget);
  const int cut = A.new_pos - dm.R + 1;
  // k == 1 (a full cache in steady state): the minimum candidate (key,
  // position) is tracked in the same pass that produces the keys.
  unsigned long long best_k = ~0ull;
  uint32_t best_p = 0xFFFFFFFFu;
  int best_i = -1;
  int nan_count = 0;
  if (ringp && policy == KVEVICT_DROPKV && A.has_q) {
    // this step's residual-output scores straight into ring column rs
    constexpr int kEpc = 16 / static_cast<int>(sizeof(KT));
    float* hr = staged_all ? hrows : nullptr;
    if (d == 128) dropkv_ring_scores<KT, 128 / kEpc / 8>(A, L, 0, n, 0, n, sh_rows, lg, sh_lse2, W, rs, hr, ld);
    else dropkv_ring_scores<KT, 64 / kEpc / 8>(A, L, 0, n, 0, n, sh_rows, lg, sh_lse2, W, rs, hr, ld);
    __syncthreads();
  }
  int lw = 0;
  while ((1 << lw) < W) ++lw;
  const int spread = 29 - lw;    // exact-sum bound: spread + 24 + log2(W) <= 53
  if (staged_all) {
    // every row is in shared memory: a thread per token; SnapKV's new weight
    // goes into column rs of the staged row and of the ring (the DropKV
    // variant's scores are already in both)
    kbuf = reinterpret_cast<unsigned long long*>(dsm + hkeys_off);
    const bool fresh = A.has_q && policy == KVEVICT_SNAPKV;
    int ncand = 0;
    for (int i = tid; i < n; i += blockDim.x) {
      float* row = hrows + i * ld;
      if (fresh) {
        float w = 0.f;
        for (int h = 0; h < g; ++h) w += exp2f(lg[static_cast<size_t>(h) * dm.lcap + i] - sh_lse2[h]);
        row[rs] = w;
        const int s = L.slot[i];
        if (s >= 0 && s < dm.P * kBlock) L.ring[static_cast<size_t>(s) * W + rs] = w;
        else set_status(A.ws.status, ST_BAD_INDEX);
      }
      const unsigned long long key = W == 32 ? window_key4<32>(row, 32, spread) : window_key4<0>(row, W, spread);
      kbuf[i] = key;
      if (key == ~0ull) ++nan_count;
      ncand += L.pos[i] < cut ? 1 : 0;
    }
    ncand = warp_sum(ncand);
    if ((tid & 31) == 0 && ncand) atomicAdd(&sh_ncand, ncand);
  } else if (ringp) {
    // window sums: each warp stages 32 tokens' history rows in shared memory
    // (one row per load instruction, coalesced), then each lane takes its own
    // token's sum (window_key); SnapKV's new weight enters the sum (and the
    // ring) at column rs
    const int lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int ld = W + 1;    // padded row: the lanes' row reads hit distinct banks
    float* stg = sh_rows + kMaxG * 128 + warp * 32 * ld;
    const bool fresh = A.has_q && policy == KVEVICT_SNAPKV;
    // the keys stay in shared memory when they fit beside the staging rows
    const size_t used = (static_cast<size_t>(kMaxG) * 128 + static_cast<size_t>(nw) * 32 * ld) * 4;
    if (used + static_cast<size_t>(n + 1) * 8 <= kEpiDynSmem) kbuf = reinterpret_cast<unsigned long long*>(dsm + used);
    // slots one chunk ahead; a chunk's position, weight and row loads are
    // all issued before its arithmetic (the ring write of column rs comes
    // after the row loads: the sums take w for that column anyway)
    int ncand = 0;     // this thread's candidates (positions below the cut: a prefix of the table)
    int s_next = warp * 32 + lane < n ? L.slot[warp * 32 + lane] : -1;
    for (int base = warp * 32; base < n; base += nw * 32) {
      const int i = base + lane;
      int s = s_next;
      if (i < n && (s < 0 || s >= dm.P * kBlock)) {
        set_status(A.ws.status, ST_BAD_INDEX);
        s = -1;
      }
      const int inext = i + nw * 32;
      s_next = inext < n ? L.slot[inext] : -1;
      const int p = i < n ? L.pos[i] : 0;
      float lgv[kMaxG];
#pragma unroll
      for (int h = 0; h < kMaxG; ++h)
        lgv[h] = (fresh && h < g && i < n) ? lg[static_cast<size_t>(h) * dm.lcap + i] : 0.f;
      for (int c = lane; c - lane < W; c += 32) {
        float x[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) {
          const int sr = __shfl_sync(0xffffffffu, s, r);
          x[r] = (sr >= 0 && c < W) ? L.ring[static_cast<size_t>(sr) * W + c] : 0.f;
        }
        if (c < W) {
#pragma unroll
          for (int r = 0; r < 32; ++r) stg[r * ld + c] = x[r];
        }
      }
      float w = 0.f;
      if (fresh) {
#pragma unroll
        for (int h = 0; h < kMaxG; ++h)
          if (h < g) w += exp2f(lgv[h] - sh_lse2[h]);
        if (s >= 0) L.ring[static_cast<size_t>(s) * W + rs] = w;
      }
      ncand += (i < n && p < cut) ? 1 : 0;
      __syncwarp();
      if (i < n) {
        const unsigned long long key = W == 32 ? window_key<32>(stg + lane * ld, 32, fresh ? rs : -1, w, spread)
                                               : window_key<0>(stg + lane * ld, W, fresh ? rs : -1, w, spread);
        kbuf[i] = key;
        if (key == ~0ull) ++nan_count;
      }
      __syncwarp();
    }
    ncand = warp_sum(ncand);
    if (lane == 0 && ncand) atomicAdd(&sh_ncand, ncand);
  } else {
    for (int i = tid; i < n; i += blockDim.x) {
      float w = 0.f;
      if (A.has_q)
        for (int h = 0; h < g; ++h) w += exp2f(lg[static_cast<size_t>(h) * dm.lcap + i] - sh_lse2[h]);
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
  if (ringp && tid == 0) kbuf[n] = kKeyZero;     // the new token's sum
  __syncthreads();
  if (ringp) {
    if (A.has_q && tid == 0) A.ls.ring_slot[l] = (rs + 1) % W;
    // max over kept neighbours [i-r, i+r], clamped to [0, n], on the keys'
    // monotone images (a NaN sum, the largest image, wins the max); each
    // thread takes a run of consecutive entries
    // (candidates are the first ncand entries; positions ascend with the
    // index, so the index breaks ties in the position's place)
    const int r = (dm.pool_kernel - 1) / 2;
    const int nn = n + 1;
    const int ncand = sh_ncand;
    const int per = (nn + static_cast<int>(blockDim.x) - 1) / static_cast<int>(blockDim.x);
    const int j1 = min(nn, (tid + 1) * per);
    for (int j = tid * per; j < j1; ++j) {
      unsigned long long m = 0;
      const int qa = max(0, j - r), qb = min(nn - 1, j + r);
      for (int q = qa; q <= qb; ++q) m = max(m, kbuf[q]);
      if (k > 1) pooled[j] = m;
      if (k == 1 && j < ncand && (m < best_k || (m == best_k && static_cast<uint32_t>(j) < best_p))) {
        best_k = m; best_p = static_cast<uint32_t>(j); best_i = j;
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
      dead = lane_remove_one(L, n, v, vout, dm.P, A.ws.status, sh_misc);
    }
  } else if (k > 1) {
    SelectResult sel;
    if (ringp) {
      auto keyf = [&](int i) { return pooled[i]; };
      sel = block_bottom_k(n, k, 64, keyf, posf, candf, sh_hist, sh_misc);
      auto isv = [&](int i) { return candf(i) && select_is_victim(sel, keyf(i), posf(i)); };
      vcount = lane_remove(L, n, plain_victims(isv), vout, nullptr, &dead, dm.P, A.ws.status, sh_scan);
    } else {
      auto keyf = [&](int i) { return mono_key(L.score[i]); };
      sel = block_bottom_k(n, k, 32, keyf, posf, candf, sh_hist, sh_misc);
      auto isv = [&](int i) { return candf(i) && select_is_victim(sel, keyf(i), posf(i)); };
      vcount = lane_remove(L, n, plain_victims(isv), vout, nullptr, &dead, dm.P, A.ws.status, sh_scan);
    }
  }
  lane_finish<KT>(A, L, l, n, k, vcount, dead, nan_count, sh_work, sh_scan);
}

// ---------------------------------------------------------------------------
// Ring policies (SnapKV, DropKV decode variant) with one lane per cluster of
// kRingCluster CTAs, each owning a quarter of the lane's tokens: the lane's
// step has few lanes to spread over the GPU otherwise (one CTA a lane left
// most SMs idle).  Before the dependency wait each rank stages the history
// rows of its tokens and of a pooling halo (pool radius on each side).
// After it: every rank derives the heads' log-sum-exp; each combines a
// quarter of the split-K outputs (the DropKV scores need all of them: the
// ranks read one another's quarter from distributed shared memory); each
// scores and keys its range, writing the ring's new column only for the
// tokens it owns; each pools and takes the minimum candidate over the
// tokens it owns, and the lane's minimum is the smallest (key, index) over
// the ranks.  The table shift after the victim is split over the ranks
// (every read before a cluster barrier, the writes after it).  Rank 0 then
// does the rest (the victim's live bit, admission, the relocation plan, the
// per-lane requests).  Several victims (k > 1): the ranks publish their
// pooled keys and rank 0 selects and removes them.
// ---------------------------------------------------------------------------
constexpr int kRingCluster = 4;
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// History rows of tokens lo .. hi - 1 to rows[(i - lo) * ld + t] (W a
// multiple of 4), as stage_history_async; their raw slots and positions to
// sh_slot and sh_pos (hi - lo ints each).
__device__ __forceinline__ void stage_history_range_async(const LaneRefs& L, const int lo, const int hi, const int W,
                                                          const int ld, const int nslot, float* rows, int* sh_slot,
                                                          int* sh_pos) {
  for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) {
    sh_slot[i - lo] = L.slot[i];
    sh_pos[i - lo] = L.pos[i];
  }
  __syncthreads();
  const int pr = W / 4;
  for (int e = threadIdx.x; e < (hi - lo) * pr; e += blockDim.x) {
    const int i = e / pr, c = (e - i * pr) * 4;
    const int s = sh_slot[i] >= 0 && sh_slot[i] < nslot ? sh_slot[i] : -1;
    float* dst = rows + i * ld + c;
    if (s >= 0) {
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)),
                   "l"(L.ring + static_cast<size_t>(s) * W + c) : "memory");
    } else {
      *reinterpret_cast<float4*>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  cp_async_commit();
}

// Layout of the dynamic shared memory of one rank: the heads' outputs, the
// staged rows, their slots, the keys.  Returns the bytes needed (the caller
// checks them against kEpiDynSmem).
constexpr int kPfBlocks = kEpiThreads;   // block list entries rank 0 reads ahead (more: read at admission)
struct RingClusterSmem {
  float* sh_a;
  float* rows;
  int* slots;        // raw slots of tokens lo .. hi - 1
  int* pos;          // their positions
  unsigned long long* keys;
  WindowPart* parts; // window sums of tokens lo .. hi - 1 without column rs (before the wait)
  int* pf_blocks;    // rank 0: the lane's block list and live masks, the new K/V row
  int* pf_masks;
  unsigned char* pf_row;
  size_t bytes;
};
__device__ __forceinline__ size_t ring_cluster_bytes(int span, int ld) {
  size_t off = static_cast<size_t>(kMaxG) * 128 * 4 + static_cast<size_t>(span) * ld * 4;
  off += 2 * ((static_cast<size_t>(span) * 4 + 7) & ~static_cast<size_t>(7));
  off += static_cast<size_t>(span + 1) * 8;
  off += static_cast<size_t>(span) * sizeof(WindowPart);
  off += 2 * static_cast<size_t>(kPfBlocks) * 4 + 2 * 128 * 4;
  return off;
}
__device__ __forceinline__ RingClusterSmem ring_cluster_smem(unsigned char* dsm, int span, int ld) {
  RingClusterSmem m;
  size_t off = 0;
  m.sh_a = reinterpret_cast<float*>(dsm + off);
  off += static_cast<size_t>(kMaxG) * 128 * 4;
  m.rows = reinterpret_cast<float*>(dsm + off);
  off += static_cast<size_t>(span) * ld * 4;
  m.slots = reinterpret_cast<int*>(dsm + off);
  off += (static_cast<size_t>(span) * 4 + 7) & ~static_cast<size_t>(7);
  m.pos = reinterpret_cast<int*>(dsm + off);
  off += (static_cast<size_t>(span) * 4 + 7) & ~static_cast<size_t>(7);
  m.keys = reinterpret_cast<unsigned long long*>(dsm + off);
  off += static_cast<size_t>(span + 1) * 8;
  m.parts = reinterpret_cast<WindowPart*>(dsm + off);
  off += static_cast<size_t>(span) * sizeof(WindowPart);
  m.pf_blocks = reinterpret_cast<int*>(dsm + off);
  off += static_cast<size_t>(kPfBlocks) * 4;
  m.pf_masks = reinterpret_cast<int*>(dsm + off);
  off += static_cast<size_t>(kPfBlocks) * 4;
  m.pf_row = dsm + off;
  off += 2 * 128 * 4;
  m.bytes = off;
  return m;
}

// The largest range (owned tokens and halo) any rank of a lane of n tokens
// stages, and whether the cluster step applies (every rank's owned tokens
// within one pass of the CTA's threads, W a multiple of 4, the staging in
// shared memory).  The same answer on every rank.
__device__ __forceinline__ bool ring_cluster_fits(const Dims& dm, const int n) {
  const int R = (dm.pool_kernel - 1) / 2;
  const int own = (n + kRingCluster - 1) / kRingCluster;
  const int span = own + 2 * R;
  const int ld = ((dm.W + 27) / 32) * 32 + 4;
  const size_t bytes = ring_cluster_bytes(span, ld);
  return n > 0 && (dm.W & 3) == 0 && own <= kEpiThreads && dm.g <= kMaxG && dm.d <= 128 && bytes <= kEpiDynSmem;
}

template <typename KT>
__device__ __forceinline__ void lane_step_cluster(const EpiArgs& A, const LaneRefs& L, const int l, const int rank,
                                                  const int n, unsigned char* dsm, int* sh_work, int* sh_gen) {
  __shared__ float sh_L[kMaxG], sh_lse2[kMaxG];
  __shared__ float sh_scale[kMaxSeg][kMaxG];
  __shared__ __align__(16) int sh_hist[256];
  __shared__ int sh_misc[40];
  __shared__ int sh_scan[40];
  __shared__ unsigned long long sh_bk;   // this rank's minimum candidate key, and its index (-1: none)
  __shared__ int sh_bi, sh_nanr;
  __shared__ int sh_vslot, sh_dead;     // rank 0: the victim's raw slot and the block it released
  __shared__ int sh_vpos;               // rank 0: the victim's position (from its owner)
  __shared__ int sh_pfnb;
  __shared__ unsigned long long sh_ck[kRingCluster];   // every rank's minimum candidate (pushed by each rank)
  __shared__ int sh_ci[kRingCluster], sh_cn[kRingCluster];   // its index (-1: none), its NaN count
  cg::cluster_group cluster = cg::this_cluster();
  const Dims& dm = A.dm;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = l / dm.Hkv, kh = l % dm.Hkv, g = dm.g, d = dm.d, W = dm.W;
  const int cbuf = A.layer % kScratchBufs;
  const int policy = dm.policy;
  const int R = (dm.pool_kernel - 1) / 2;
  const int i0 = (n * rank) / kRingCluster, i1 = (n * (rank + 1)) / kRingCluster;   // owned tokens
  const int lo = max(0, i0 - R), hi = min(n, i1 + R);                              // with the halo
  const int ld = ((W + 27) / 32) * 32 + 4;
  const RingClusterSmem sm = ring_cluster_smem(dsm, hi - lo, ld);

  // ---- before the dependency wait: history rows, slots and positions of the
  // range; rank 0 also the lane's block list with its live masks and the new
  // token's K/V row (none of which the attention kernel writes)
  if (tid == 0) { sh_vslot = -1; sh_dead = -1; }
  const int rs = A.ls.ring_slot[l];   // written by this layer's previous epilogue only
  stage_history_range_async(L, lo, hi, W, ld, dm.P * kBlock, sm.rows, sm.slots, sm.pos);
  if (rank == 0) {
    const int nb0 = *L.nblocks;
    if (tid == 0) sh_pfnb = nb0;
    if (nb0 <= kPfBlocks) {
      for (int j = tid; j < nb0; j += blockDim.x) {
        const int blk = L.blocks[j];
        sm.pf_blocks[j] = blk;
        sm.pf_masks[j] = L.mask[blk];
      }
    }
    // element by element: the new rows carry no alignment promise
    KT* row = reinterpret_cast<KT*>(sm.pf_row);
    for (int e = tid; e < 2 * d; e += blockDim.x)
      row[e] = e < d ? static_cast<const KT*>(A.k_new)[static_cast<size_t>(l) * d + e]
                     : static_cast<const KT*>(A.v_new)[static_cast<size_t>(l) * d + e - d];
  }
  int lw = 0;
  while ((1 << lw) < W) ++lw;
  const int spread = 29 - lw;    // exact-sum bound: spread + 24 + log2(W) <= 53
  // the window sums without column rs, while the attention kernel drains
  // (column rs takes this step's value after the wait)
  cp_async_wait_all();
  __syncthreads();
  for (int i = lo + tid; i < hi; i += blockDim.x) sm.parts[i - lo] = window_part(sm.rows + (i - lo) * ld, W, A.has_q ? rs : -1, spread);
  grid_dep_wait();      // the attention kernel's results are complete and visible
  grid_dep_launch();
  if (rank == 0) read_generation(A, sh_gen);
  if (tid == 0) { sh_bi = -1; sh_bk = ~0ull; sh_nanr = 0; }
  if (L.pos[n - 1] >= A.new_pos) {
    cp_async_wait_all();
    if (rank == 0 && tid == 0) {
      set_status(A.ws.status, ST_POSITION);
      A.n_victims[l] = 0; A.ws.need_admit[l] = 0; A.ws.want_dst[l] = 0; A.ws.plan_tlive[l] = 0;
    }
    return;
  }

  // ---- combine the split-K partials: a quarter of the outputs per rank -----------
  if (A.has_q) {
    const int nseg = min(A.ws.lane_nseg_buf[cbuf][l], kMaxSeg);
    const float2* ml = reinterpret_cast<const float2*>(A.ws.part_ml_buf[cbuf]) + static_cast<size_t>(l) * kMaxSeg * g;
    if (warp < g) {
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
        sh_L[h] = Ls;
        const float lse2 = M + log2f(Ls);
        sh_lse2[h] = lse2;
        if (rank == 0) A.lse[static_cast<size_t>(b) * dm.Hq + kh * g + h] = lse2 * kLn2;
      }
    }
    __syncthreads();
  }
  // The split-K output combine of outputs e0 .. e0 + cnt - 1 (all threads):
  // four threads per output, each a quarter of the segments (fewer loads in a
  // chain), their sums added by two shuffles.  The DropKV scores need every
  // output first (a quarter per rank, then exchanged); SnapKV's step does
  // not, so ranks 1..3 combine a third each after the eviction, while rank 0
  // finishes the lane.
  const int ghd = g * d;
  auto combine = [&](const int e0, const int cnt) {
    const int nseg = min(A.ws.lane_nseg_buf[cbuf][l], kMaxSeg);
    const float* po = A.ws.part_o_buf[cbuf] + static_cast<size_t>(l) * kMaxSeg * g * d;
    for (int base = 0; base < 4 * cnt; base += blockDim.x) {
      const int x = base + tid, q = x & 3;
      const bool act = x < 4 * cnt;
      const int he = e0 + (x >> 2);
      const int h = act ? he / d : 0, e = act ? he - h * d : 0;
      float acc = 0.f;
      if (act) {
#pragma unroll 4
        for (int s = q; s < nseg; s += 4) acc = fmaf(po[(static_cast<size_t>(s) * g + h) * d + e], sh_scale[s][h], acc);
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      if (act && q == 0) {
        const float o = acc / sh_L[h];
        A.out[(static_cast<size_t>(b) * dm.Hq + kh * g + h) * d + e] = o;
        sm.sh_a[he] = o;
      }
    }
  };
  if (A.has_q && policy == KVEVICT_DROPKV) {
    const int per = (ghd + kRingCluster - 1) / kRingCluster;
    combine(rank * per, max(0, min(ghd, rank * per + per) - rank * per));
    {
      cluster.sync();   // every rank's quarter of the outputs is in its shared memory
      for (int rr = 0; rr < kRingCluster; ++rr) {
        if (rr == rank) continue;
        const float* ra = cluster.map_shared_rank(sm.sh_a, rr);
        for (int he = rr * per + tid; he < min(ghd, (rr + 1) * per); he += blockDim.x) sm.sh_a[he] = ra[he];
      }
    }
    __syncthreads();
  }

  // ---- scores of this step into the ring, window-sum keys of lo .. hi - 1 --------
  const float* lg = A.ws.logits_buf[cbuf] + static_cast<size_t>(l) * g * dm.lcap;
  const int k = max(0, n + 1 - dm.budget);
  const int cut = A.new_pos - dm.R + 1;
  if (policy == KVEVICT_DROPKV && A.has_q) {
    constexpr int kEpc = 16 / static_cast<int>(sizeof(KT));
    if (d == 128) dropkv_ring_scores<KT, 128 / kEpc / 8>(A, L, lo, hi, i0, i1, sm.sh_a, lg, sh_lse2, W, rs, sm.rows, ld);
    else dropkv_ring_scores<KT, 64 / kEpc / 8>(A, L, lo, hi, i0, i1, sm.sh_a, lg, sh_lse2, W, rs, sm.rows, ld);
    __syncthreads();
  }
  const bool fresh = A.has_q && policy == KVEVICT_SNAPKV;
  int nan_count = 0;
  for (int i = lo + tid; i < hi; i += blockDim.x) {
    float* row = sm.rows + (i - lo) * ld;
    const bool own = i >= i0 && i < i1;
    if (fresh) {
      float w = 0.f;
      for (int h = 0; h < g; ++h) w += exp2f(lg[static_cast<size_t>(h) * dm.lcap + i] - sh_lse2[h]);
      row[rs] = w;
      if (own) {
        const int s = sm.slots[i - lo];
        if (s >= 0 && s < dm.P * kBlock) L.ring[static_cast<size_t>(s) * W + rs] = w;
        else set_status(A.ws.status, ST_BAD_INDEX);
      }
    }
    // this step's column rs joins the sum taken before the wait
    const unsigned long long key = window_merge(sm.parts[i - lo], A.has_q ? row[rs] : 0.f, row, W,
                                                A.has_q ? rs : -1, spread);
    sm.keys[i - lo] = key;
    if (own && key == ~0ull) ++nan_count;
  }
  if (tid == 0 && hi == n) sm.keys[n - lo] = kKeyZero;     // the new token's sum
  if (nan_count) atomicAdd(&sh_nanr, nan_count);
  __syncthreads();

  // ---- max-pool over kept neighbours, minimum candidate of the owned tokens -------
  unsigned long long* pooled = A.ws.pooled64 ? A.ws.pooled64 + static_cast<size_t>(l) * dm.cap : nullptr;
  unsigned long long best_k = ~0ull;
  uint32_t best_p = 0xFFFFFFFFu;
  int best_i = -1;
  for (int j = i0 + tid; j < i1; j += blockDim.x) {
    unsigned long long m = 0;
    const int qa = max(0, j - R), qb = min(n, j + R);
    for (int q = qa; q <= qb; ++q) m = max(m, sm.keys[q - lo]);
    if (k > 1) pooled[j] = m;
    if (k == 1 && sm.pos[j - lo] < cut && (m < best_k || (m == best_k && static_cast<uint32_t>(j) < best_p))) {
      best_k = m; best_p = static_cast<uint32_t>(j); best_i = j;
    }
  }
  int vcount = 0, dead = 0;
  int32_t* vout = A.victims + static_cast<size_t>(l) * dm.cap;
  if (k == 1) {
    const int v_local = block_argmin3(best_k, best_p, best_i, sh_hist, sh_misc);
    // each rank pushes its minimum (and NaN count) into every rank's shared
    // memory: after the barrier every rank reads them locally
    if (tid < kRingCluster) {
      unsigned long long m = ~0ull;
      if (v_local >= 0) {
        m = 0;
        const int qa = max(0, v_local - R), qb = min(n, v_local + R);
        for (int q = qa; q <= qb; ++q) m = max(m, sm.keys[q - lo]);
      }
      cluster.map_shared_rank(sh_ck, tid)[rank] = m;
      cluster.map_shared_rank(sh_ci, tid)[rank] = v_local;
      cluster.map_shared_rank(sh_cn, tid)[rank] = sh_nanr;
    }
    cluster.sync();   // every rank's minimum and NaN count is in every rank's shared memory
    unsigned long long gk = ~0ull;
    int v = -1;
    int nan_all = 0;
    for (int rr = 0; rr < kRingCluster; ++rr) {
      const int ri = sh_ci[rr];
      const unsigned long long rk = sh_ck[rr];
      if (ri >= 0 && (v < 0 || rk < gk || (rk == gk && ri < v))) { gk = rk; v = ri; }
      nan_all += sh_cn[rr];
    }
    if (v >= 0) {
      // the rank owning the victim pushes its slot and position to rank 0;
      // every rank reads the entries it moves down one place
      if (v >= i0 && v < i1 && tid == 0) {
        *cluster.map_shared_rank(&sh_vslot, 0) = sm.slots[v - lo];
        *cluster.map_shared_rank(&sh_vpos, 0) = sm.pos[v - lo];
      }
      const int i = max(i0, v + 1) + tid;
      const bool mv = i < i1;
      int p = 0, s = 0;
      float sc = 0.f;
      if (mv) {
        p = sm.pos[i - lo];
        s = sm.slots[i - lo];
        if (L.score) sc = L.score[i];
      }
      cluster.sync();   // every read is done: no rank touches another's shared memory after this
      if (mv) {
        L.pos[i - 1] = p;
        L.slot[i - 1] = s;
        if (L.score) L.score[i - 1] = sc;
      }
      vcount = 1;
      if (rank == 0) {
        if (tid == 0) vout[0] = sh_vpos;
        // the victim's live bit (an emptied block is released and leaves the
        // list), from the live masks read ahead when the list fitted
        const int vs = sh_vslot;
        if (vs >= 0 && vs < dm.P * kBlock) {
          const int blk = vs >> 4, bit = 1 << (vs & 15);
          if (sh_pfnb <= kPfBlocks) {
            for (int j = tid; j < sh_pfnb; j += blockDim.x) {
              if (sm.pf_blocks[j] == blk) {
                const int old = sm.pf_masks[j];
                atomicAnd(&L.mask[blk], ~bit);
                if ((old & ~bit) == 0 && (old & bit)) {
                  L.owner[blk] = -1;
                  sh_dead = blk;
                }
              }
            }
          } else if (tid == 0) {
            const int old = atomicAnd(&L.mask[blk], ~bit);
            if ((old & ~bit) == 0 && (old & bit)) {
              L.owner[blk] = -1;
              sh_dead = blk;
            }
          }
        } else if (vs >= 0 && tid == 0) {
          set_status(A.ws.status, ST_BAD_INDEX);
        }
        __syncthreads();
        const int dead_blk = sh_dead;
        if (dead_blk >= 0) {
          const int nb = *L.nblocks;
          for (int j = tid; j < nb; j += blockDim.x) {
            if (L.blocks[j] == dead_blk) {
              L.blocks[j] = L.blocks[nb - 1];
              *L.nblocks = nb - 1;
            }
          }
          dead = 1;
        }
        __syncthreads();
      }
    } else {
      cluster.sync();   // no rank touches another's shared memory after this
    }
    if (A.has_q && policy != KVEVICT_DROPKV && rank != 0) {
      const int per3 = (ghd + kRingCluster - 2) / (kRingCluster - 1);
      const int e0 = (rank - 1) * per3;
      combine(e0, max(0, min(ghd, e0 + per3) - e0));
    }
    // the table writes (and outputs) of every rank are done before rank 0
    // signals for the lane (arrive here, wait before the signal)
    cluster_arrive();
    if (rank != 0) {
      cluster_wait();
      return;
    }
    if (A.has_q && tid == 0) A.ls.ring_slot[l] = (rs + 1) % W;
    LanePrefetch<KT> pf;
    pf.blocks = sm.pf_blocks;
    pf.masks = sm.pf_masks;
    pf.nb = sh_pfnb;
    pf.victim_slot = vcount == 1 ? sh_vslot : -1;
    pf.dead_blk = vcount == 1 ? sh_dead : -1;
    pf.k_new = reinterpret_cast<const KT*>(sm.pf_row);
    pf.v_new = reinterpret_cast<const KT*>(sm.pf_row) + d;
    lane_finish<KT>(A, L, l, n, k, vcount, dead, nan_all, sh_work, sh_scan,
                    sh_pfnb <= kPfBlocks ? &pf : nullptr);
    cluster_wait();
    return;
  } else if (k > 1) {
    cluster.sync();   // every rank's pooled keys are written
    if (rank == 0) {
      auto candf = [&](int i) { return L.pos[i] < cut; };
      auto posf = [&](int i) { return static_cast<uint32_t>(L.pos[i]); };
      auto keyf = [&](int i) { return pooled[i]; };
      const SelectResult sel = block_bottom_k(n, k, 64, keyf, posf, candf, sh_hist, sh_misc);
      auto isv = [&](int i) { return candf(i) && select_is_victim(sel, keyf(i), posf(i)); };
      vcount = lane_remove(L, n, plain_victims(isv), vout, nullptr, &dead, dm.P, A.ws.status, sh_scan);
    }
  }
  if (A.has_q && policy != KVEVICT_DROPKV) {
    const int per = (ghd + kRingCluster - 1) / kRingCluster;
    combine(rank * per, max(0, min(ghd, rank * per + per) - rank * per));
  }
  // the ranks' NaN counts (final once a cluster barrier followed the keys:
  // the selection's, or one here); nothing reads another rank's shared
  // memory after the last barrier
  if (k == 0) cluster.sync();
  int nan_tot = 0;
  if (rank == 0 && tid == 0)
    for (int rr = 0; rr < kRingCluster; ++rr) nan_tot += *cluster.map_shared_rank(&sh_nanr, rr);
  cluster.sync();
  if (rank != 0) return;
  if (A.has_q && tid == 0) A.ls.ring_slot[l] = (rs + 1) % W;
  // admission from the block state read ahead when at most one token left
  // (its live bit and released block known) and the list fitted
  LanePrefetch<KT> pf;
  pf.blocks = sm.pf_blocks;
  pf.masks = sm.pf_masks;
  pf.nb = sh_pfnb;
  pf.victim_slot = vcount == 1 ? sh_vslot : -1;
  pf.dead_blk = vcount == 1 ? sh_dead : -1;
  pf.k_new = reinterpret_cast<const KT*>(sm.pf_row);
  pf.v_new = reinterpret_cast<const KT*>(sm.pf_row) + d;
  const bool use_pf = k <= 1 && sh_pfnb <= kPfBlocks;
  lane_finish<KT>(A, L, l, n, k, vcount, dead, nan_tot, sh_work, sh_scan, use_pf ? &pf : nullptr);
}

template <typename KT>
__global__ void __cluster_dims__(kRingCluster, 1, 1) __launch_bounds__(kEpiThreads, 1)
    decode_epilogue_ring_cluster_kernel(EpiArgs A) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ int sh_scan[40];
  __shared__ int sh_work, sh_last, sh_flag, sh_sig, sh_gen;
  const Dims& dm = A.dm;
  const int rank = static_cast<int>(cg::this_cluster().block_rank());
  const int l = blockIdx.x / kRingCluster, tid = threadIdx.x;
  LaneRefs L = lane_refs(A.ls, dm, l);
  const int n = __ldcg(A.ls.count + l);
  if (tid == 0) { sh_work = 0; sh_sig = 0; sh_gen = 0; }
  if (n < 0 || n >= dm.cap) {
    grid_dep_wait();
    grid_dep_launch();
    if (rank == 0) {
      read_generation(A, &sh_gen);
      if (tid == 0) {
        set_status(A.ws.status, ST_CAPACITY);
        A.n_victims[l] = 0; A.ws.need_admit[l] = 0; A.ws.want_dst[l] = 0; A.ws.plan_tlive[l] = 0;
      }
    }
  } else if (ring_cluster_fits(dm, n)) {
    lane_step_cluster<KT>(A, L, l, rank, n, dsm, &sh_work, &sh_gen);
  } else if (rank == 0) {
    lane_step<KT, true>(A, L, l, n, dsm, &sh_work, &sh_gen);
  } else {
    grid_dep_wait();
    grid_dep_launch();
  }
  if (rank != 0) return;
  // rank 0 signals for the lane (the others are done with the scratch copy:
  // the step's last cluster barrier follows their last read)
  int* mv = reinterpret_cast<int*>(dsm);
  epilogue_tail<KT>(A, sh_scan, &sh_work, &sh_last, &sh_flag, &sh_sig, &sh_gen, mv, mv + kApplyThreads,
                    static_cast<int>(gridDim.x) / kRingCluster);
  scratch_released(A);
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
    if (tid == 0) { ws.counters[1] = 0; ws.counters[2] = 0; ws.counters[kApplyCount] = 0; }
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
  // the lanes left with work for apply, ascending (each thread reads the
  // requests of the lanes it updated above)
  int nwork = 0;
  for (int base = 0; base < dm.lanes; base += blockDim.x) {
    const int l = base + tid;
    const int has = (l < dm.lanes && (__ldcg(ws.need_admit + l) != 0 || __ldcg(ws.want_dst + l) > 0)) ? 1 : 0;
    int tot;
    const int ex = block_excl_scan(has, sh_scan, &tot);
    if (has) ws.apply_list[nwork + ex] = l;
    nwork += tot;
  }
  if (tid == 0) {
    ws.counters[1] = 1;
    ws.counters[2] = deferred ? 0 : totM;
    ws.counters[kApplyCount] = nwork;
    ws.counters[kApplyClaim] = 0;
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
// One lane's admission into its fresh block and its relocation plan (vToken
// review, Sec. 3.3 Stage 3), after the layer allocator assigned the blocks;
// all threads of a kApplyThreads CTA.
template <typename KT>
__device__ void apply_lane(const LayerState& ls, const Workspace& ws, const Dims& dm, const int l,
                           const void* k_new, const void* v_new, int mark_freed, int32_t* moves, int* sh_scan,
                           int* sh_mv_src, int* sh_mv_dst) {
  const int tid = threadIdx.x;
  // the allocator (another CTA) wrote these; read them from L2
  const int need = __ldcg(ws.need_admit + l);
  const int ndst = __ldcg(ws.want_dst + l);
  if (!need && ndst == 0) return;
  LaneRefs L = lane_refs(ls, dm, l);
  const int d = dm.d;
  KT* kp = static_cast<KT*>(ls.k_pool);
  KT* vp = static_cast<KT*>(ls.v_pool);
  const int m = __ldcg(ls.count + l);
  if (need) {
    const int blk = __ldcg(ws.admit_block + l);
    const size_t s = static_cast<size_t>(blk) * kBlock;
    copy_row(kp + s * d, static_cast<const KT*>(k_new) + static_cast<size_t>(l) * d, d);
    copy_row(vp + s * d, static_cast<const KT*>(v_new) + static_cast<size_t>(l) * d, d);
    if (L.ring)
      for (int t = tid; t < L.W; t += blockDim.x) L.ring[s * L.W + t] = 0.f;
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
    const int dbeg = __ldcg(ws.dst_begin + l);
    const int mbeg = __ldcg(ws.move_begin + l);
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
        const int db = __ldcg(ws.alloc_ids + dbeg + q / kBlock);
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
      if (L.ring) move_history_rows(L.ring, L.W, sh_mv_src, sh_mv_dst, tot);
      __syncthreads();
      q_total += tot;
    }
    __syncthreads();
    for (int j = tid; j < ndst; j += blockDim.x) {
      const int db = __ldcg(ws.alloc_ids + dbeg + j);
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
    for (int j = tid; j < ndst; j += blockDim.x) L.blocks[nb2 + j] = __ldcg(ws.alloc_ids + dbeg + j);
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

// Admission into a fresh block and relocation of each lane, after the layer
// allocator, when the epilogue does not do it itself.
template <typename KT>
__global__ void __launch_bounds__(kApplyThreads, 1) apply_kernel(LayerState ls, Workspace ws, Dims dm,
                                                           const void* k_new, const void* v_new,
                                                           int mark_freed, int32_t* moves) {
  __shared__ int sh_scan[40];
  __shared__ int sh_mv_src[kApplyThreads], sh_mv_dst[kApplyThreads];
  grid_dep_launch();    // the next layer's attention may start (it touches other state)
  grid_dep_wait();      // the epilogue and its allocator are complete
  if (ws.counters[1] == 0) return;
  apply_lane<KT>(ls, ws, dm, blockIdx.x, k_new, v_new, mark_freed, moves, sh_scan, sh_mv_src, sh_mv_dst);
}

}  // namespace

cudaError_t launch_epilogue(const Ctx& ctx, int layer, bool has_q, int new_pos, const void* k_new,
                            const void* v_new, float* out, float* lse, int32_t* victims,
                            int32_t* n_victims, cudaStream_t stream, bool* needs_apply_kernel) {
  EpiArgs A;
  A.ls = layer_state(ctx, layer);
  A.ws = ctx.ws;
  A.dm = ctx.dims;
  A.dm.budget = ctx.layer_budget[layer];
  A.dm.R = ctx.layer_recent[layer];
  // deferred relocation: Eq. (1)'s test never passes here (F <= 1)
  if (ctx.defer_reloc) A.dm.theta_f = INFINITY;
  A.has_q = has_q ? 1 : 0;
  A.new_pos = new_pos;
  A.layer = layer;
  A.k_new = k_new; A.v_new = v_new;
  A.out = out; A.lse = lse; A.victims = victims; A.n_victims = n_victims;
  // Early start (programmatic dependent launch) only right after this
  // layer's attention launch: the epilogue then reads, before its dependency
  // wait, tables no running kernel writes.  A query-less epilogue waits for
  // its predecessor.
  const bool pdl = has_q && ctx.last_kind == kLaunchAttend && ctx.last_layer == layer;
  const bool ring = ctx.dims.policy != KVEVICT_H2O;
  const dim3 grid(ctx.dims.lanes);
  // the lean H2O epilogue when every lane is within its budget (a hint from
  // the host's record of the layer; either kernel is correct in every case)
  const bool lean = !ring && ctx.lean_epi && ctx.layer_steady[layer];
  A.applies = (lean || ctx.epi_applies) ? 1 : 0;
  if (needs_apply_kernel) *needs_apply_kernel = !A.applies;
  if (lean)   // bf16 pools only (see kvevict_create)
    return launch_k(decode_epilogue_lean_kernel<__nv_bfloat16>, grid, dim3(kLeanThreads), 0, stream, pdl, A);
  const dim3 block(kEpiThreads);
  if (ring && ctx.ring_cluster) {
    const dim3 cgrid(ctx.dims.lanes * kRingCluster);
    if (ctx.dims.dtype == KVEVICT_BF16)
      return launch_k(decode_epilogue_ring_cluster_kernel<__nv_bfloat16>, cgrid, block, kEpiDynSmem, stream, pdl, A);
    return launch_k(decode_epilogue_ring_cluster_kernel<float>, cgrid, block, kEpiDynSmem, stream, pdl, A);
  }
  if (ctx.dims.dtype == KVEVICT_BF16)
    return ring ? launch_k(decode_epilogue_kernel<__nv_bfloat16, true>, grid, block, kEpiDynSmem, stream, pdl, A)
                : launch_k(decode_epilogue_kernel<__nv_bfloat16, false>, grid, block, kEpiDynSmem, stream, pdl, A);
  return ring ? launch_k(decode_epilogue_kernel<float, true>, grid, block, kEpiDynSmem, stream, pdl, A)
              : launch_k(decode_epilogue_kernel<float, false>, grid, block, kEpiDynSmem, stream, pdl, A);
}

cudaError_t prepare_epilogue() {
  const int bytes = static_cast<int>(kEpiDynSmem);
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(decode_epilogue_kernel<__nv_bfloat16, false>, a, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_epilogue_kernel<__nv_bfloat16, true>, a, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_epilogue_kernel<float, false>, a, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_epilogue_kernel<float, true>, a, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_epilogue_ring_cluster_kernel<__nv_bfloat16>, a, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_epilogue_ring_cluster_kernel<float>, a, bytes);
  // the lean kernel shares SMs with the attention kernel, which needs the
  // largest shared-memory carveout: ask for the same one
  const cudaFuncAttribute c = cudaFuncAttributePreferredSharedMemoryCarveout;
  if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_epilogue_lean_kernel<__nv_bfloat16>, c, 100);
  return e;
}

// The smallest occupancy over the large kernel's four instantiations (any
// of them may run a decode step).
int epilogue_ctas_per_sm() {
  int best = 1 << 30;
  auto take = [&](auto kernel) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kEpiThreads, kEpiDynSmem) != cudaSuccess) n = 0;
    best = n < best ? n : best;
  };
  take(decode_epilogue_kernel<__nv_bfloat16, false>);
  take(decode_epilogue_kernel<__nv_bfloat16, true>);
  take(decode_epilogue_kernel<float, false>);
  take(decode_epilogue_kernel<float, true>);
  return best;
}

// kRingCluster when a cluster of the ring epilogue can be resident (one
// CTA per SM of a cluster, for both storage types), else 0.
int ring_cluster_ctas() {
  int best = 1 << 30;
  auto take = [&](auto kernel) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kEpiThreads, kEpiDynSmem) != cudaSuccess) n = 0;
    best = n < best ? n : best;
  };
  take(decode_epilogue_ring_cluster_kernel<__nv_bfloat16>);
  take(decode_epilogue_ring_cluster_kernel<float>);
  return best >= 1 ? kRingCluster : 0;
}

cudaError_t lean_epilogue_attributes(cudaFuncAttributes* a, int* threads) {
  *threads = kLeanThreads;
  return cudaFuncGetAttributes(a, decode_epilogue_lean_kernel<__nv_bfloat16>);
}

int lean_epilogue_ctas_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_epilogue_lean_kernel<__nv_bfloat16>, kLeanThreads,
                                                    0) != cudaSuccess)
    return 0;
  return n;
}

cudaError_t launch_allocate(const Ctx& ctx, const Workspace& ws, int layer, cudaStream_t stream) {
  allocate_kernel<<<1, 1024, 0, stream>>>(layer_state(ctx, layer), ws, ctx.dims);
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
