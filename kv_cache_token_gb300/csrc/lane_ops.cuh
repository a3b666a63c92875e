// Lane-level device routines shared by the decode epilogue and the forced
// compaction: in-place stable removal of victims from a token table,
// release of emptied blocks, pruning of the lane's block list, and the
// relocation plan (vToken review, Sec. 3.3 Stages 1 and 3).  Each routine is
// executed by all threads of one CTA that owns the lane.
#pragma once
#include "kvevict_internal.cuh"

namespace kve {

struct LaneRefs {
  int32_t* pos; int32_t* slot; float* score;                // lane slices
  float* ring;                                              // layer: history row per slot
  int32_t* blocks; int32_t* nblocks;                        // lane block list
  int32_t* owner; int32_t* mask;                            // layer pool
  int W;
};

__device__ __forceinline__ LaneRefs lane_refs(const LayerState& ls, const Dims& dm, int l) {
  LaneRefs r;
  const size_t off = static_cast<size_t>(l) * dm.cap;
  r.pos = ls.pos + off;
  r.slot = ls.slot + off;
  r.score = ls.score ? ls.score + off : nullptr;
  r.ring = ls.ring;
  r.blocks = ls.lane_blocks + off;
  r.nblocks = ls.lane_nblocks + l;
  r.owner = ls.owner;
  r.mask = ls.mask;
  r.W = dm.W;
  return r;
}

// A victim predicate without per-chunk preparation.
template <typename F>
struct PlainVictims {
  F f;
  __device__ __forceinline__ void prepare(int) {}
  __device__ __forceinline__ bool operator()(int i) const { return f(i); }
};
template <typename F>
__device__ __forceinline__ PlainVictims<F> plain_victims(F f) { return PlainVictims<F>{f}; }

// Removes the entries i < n for which is_victim(i) holds, keeping the order
// of the survivors.  Victim positions are appended (ascending) to vout (if
// not null).  Each victim's live bit is cleared (fire-and-forget atomics);
// afterwards every block of the lane's list left without a live bit (each
// held one before) is released (owner -1) and, if freed_flag is given,
// flagged.  is_victim.prepare(base) runs on every thread at the start of each
// chunk of blockDim entries, before any entry of the chunk is tested.
// Returns the number of victims.  sh_scan: 40 ints.  History rows stay at
// their slots.
template <typename VictimFn>
__device__ __forceinline__ int lane_remove(const LaneRefs& L, int n, VictimFn is_victim, int32_t* vout,
                           int32_t* freed_flag, int* n_dead, int P, uint32_t* status,
                           int* sh_scan) {
  int kept_total = 0, vict_total = 0;
  for (int base = 0; base < n; base += blockDim.x) {
    is_victim.prepare(base);
    const int i = base + threadIdx.x;
    int p = 0, s = 0;
    float sc = 0.f;
    bool isv = false, keep = false;
    if (i < n) {
      p = L.pos[i];
      s = L.slot[i];
      if (L.score) sc = L.score[i];
      isv = is_victim(i);
      keep = !isv;
    }
    // one scan of both counts: survivors in the low half-word, victims in the high
    int tot2;
    const int ex2 = block_excl_scan((keep ? 1 : 0) | (isv ? 0x10000 : 0), sh_scan, &tot2);
    const int kex = ex2 & 0xFFFF, vex = ex2 >> 16;
    const int ktot = tot2 & 0xFFFF, vtot = tot2 >> 16;
    const int ni = kept_total + kex;
    // every read of this chunk happened before the scans' barriers
    if (keep) {
      L.pos[ni] = p;
      L.slot[ni] = s;
      if (L.score) L.score[ni] = sc;
    }
    if (isv) {
      if (vout) vout[vict_total + vex] = p;
      if (s >= 0 && s < P * kBlock) {
        atomicAnd(&L.mask[s >> 4], ~(1 << (s & 15)));
      } else if (s >= 0) {
        set_status(status, ST_BAD_INDEX);
      }
    }
    __syncthreads();
    kept_total += ktot;
    vict_total += vtot;
  }
  // blocks emptied by the removal
  __threadfence();
  __syncthreads();
  int dead = 0;
  const int nb = *L.nblocks;
  for (int j = threadIdx.x; j < nb; j += blockDim.x) {
    const int b = L.blocks[j];
    if (b >= 0 && b < P && (__ldcg(L.mask + b) & 0xFFFF) == 0 && L.owner[b] >= 0) {
      L.owner[b] = -1;
      if (freed_flag) freed_flag[b] = 1;
      ++dead;
    }
  }
  int tot;
  (void)block_excl_scan(dead, sh_scan, &tot);
  if (n_dead) *n_dead = tot;
  return vict_total;
}

// Block-wide minimum of (key, position) with the entry index; returns the
// index of the minimum (-1 if no thread had a candidate).  Every thread
// returns the same value.  sh_a: 256 ints of scratch, 8-byte aligned (it
// also holds 64-bit keys), sh_b: 40 ints.
__device__ __forceinline__ int block_argmin3(unsigned long long bk, uint32_t bp, int bi, int* sh_a, int* sh_b) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long ok = __shfl_xor_sync(0xffffffffu, bk, o);
    const uint32_t op = __shfl_xor_sync(0xffffffffu, bp, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (oi >= 0 && (bi < 0 || ok < bk || (ok == bk && op < bp))) { bk = ok; bp = op; bi = oi; }
  }
  unsigned long long* shk = reinterpret_cast<unsigned long long*>(sh_a);   // 32 x 8 bytes
  uint32_t* shp = reinterpret_cast<uint32_t*>(sh_a + 64);
  const int wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) { shk[wid] = bk; shp[wid] = bp; sh_b[wid] = bi; }
  __syncthreads();
  bk = ~0ull; bp = 0xFFFFFFFFu; bi = -1;
  for (int w = 0; w < nw; ++w) {
    const int oi = sh_b[w];
    if (oi >= 0 && (bi < 0 || shk[w] < bk || (shk[w] == bk && shp[w] < bp))) { bk = shk[w]; bp = shp[w]; bi = oi; }
  }
  __syncthreads();
  return bi;
}

// History rows (ring policies) of tot moved tokens, W floats each, from
// slot src[j] to slot dst[j] (src -1: not moved).  Destinations are fresh
// blocks, never a source of the same plan, so each row is read before any
// write can reach it.
__device__ __forceinline__ void move_history_rows(float* ring, const int W, const int* src, const int* dst,
                                                  const int tot) {
  // a warp per row
  const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int j = threadIdx.x >> 5; j < tot; j += nw) {
    const int so = src[j];
    if (so < 0) continue;
    const size_t a = static_cast<size_t>(so) * W, b = static_cast<size_t>(dst[j]) * W;
    for (int t = lane; t < W; t += 32) ring[b + t] = ring[a + t];
  }
}

// Removes the single entry v (the step's only victim): its position goes to
// vout[0], its live bit clears (an emptied block is released and dropped
// from the lane's block list by swapping in the last entry), and entries
// v+1 .. n-1 shift down by one.  Returns 1 if a block was released.
__device__ __forceinline__ int lane_remove_one(const LaneRefs& L, int n, int v, int32_t* vout, int P,
                                               uint32_t* status, int* sh_b) {
  if (threadIdx.x == 0) {
    const int s = L.slot[v];
    vout[0] = L.pos[v];
    int dead_blk = -1;
    if (s >= 0 && s < P * kBlock) {
      const int b = s >> 4, bit = 1 << (s & 15);
      const int old = atomicAnd(&L.mask[b], ~bit);
      if ((old & ~bit) == 0 && (old & bit)) {
        L.owner[b] = -1;
        dead_blk = b;
      }
    } else if (s >= 0) {
      set_status(status, ST_BAD_INDEX);
    }
    sh_b[0] = dead_blk;
  }
  // shift the table: every read of a chunk precedes the barrier, the chunk's
  // writes (one index lower) follow it
  for (int base = v + 1; base < n; base += blockDim.x) {
    const int i = base + threadIdx.x;
    int p = 0, s = 0;
    float sc = 0.f;
    if (i < n) {
      p = L.pos[i];
      s = L.slot[i];
      if (L.score) sc = L.score[i];
    }
    __syncthreads();
    if (i < n) {
      L.pos[i - 1] = p;
      L.slot[i - 1] = s;
      if (L.score) L.score[i - 1] = sc;
    }
  }
  __syncthreads();
  const int dead_blk = sh_b[0];
  if (dead_blk >= 0) {
    const int nb = *L.nblocks;
    for (int j = threadIdx.x; j < nb; j += blockDim.x) {
      if (L.blocks[j] == dead_blk) {
        L.blocks[j] = L.blocks[nb - 1];
        *L.nblocks = nb - 1;
      }
    }
    __syncthreads();
  }
  return dead_blk >= 0 ? 1 : 0;
}

// Drops released blocks (owner != l) from the lane's block list, stably.
__device__ __forceinline__ int lane_prune_blocks(const LaneRefs& L, int l, int* sh_scan) {
  const int nb = *L.nblocks;
  int out = 0;
  for (int base = 0; base < nb; base += blockDim.x) {
    const int j = base + threadIdx.x;
    int b = -1;
    bool keep = false;
    if (j < nb) {
      b = L.blocks[j];
      keep = b >= 0 && L.owner[b] == l;
    }
    int tot;
    const int ex = block_excl_scan(keep ? 1 : 0, sh_scan, &tot);
    if (keep) L.blocks[out + ex] = b;
    __syncthreads();
    out += tot;
  }
  __syncthreads();
  if (threadIdx.x == 0) *L.nblocks = out;
  __syncthreads();
  return out;
}

// Eq. (1)'s fragmentation test F > theta for N blocks holding n_live tokens,
// in double (theta_f is widened exactly); N > 0.
__device__ __forceinline__ bool frag_over(int n_live, int N, float theta_f) {
  const double Fd = 1.0 - static_cast<double>(n_live) / (static_cast<double>(N) * kBlock);
  return Fd > static_cast<double>(theta_f);
}

// Relocation plan of a lane after its evictions and admission, given the
// outcome of the fragmentation test (over); a pending admission counts as
// one more block holding one token.
// Returns the number of destination blocks (0 = no plan); *t_live = tokens to move.
__device__ __forceinline__ int lane_plan_given(const LaneRefs& L, int nb, bool over, bool forced, bool pending_admit,
                                               int* t_live_out, int* sh_scan) {
  const int N = nb + (pending_admit ? 1 : 0);
  if (N == 0 || (!forced && !over)) { *t_live_out = 0; return 0; }
  int src = 0, tl = 0;
  for (int j = threadIdx.x; j < nb; j += blockDim.x) {
    const int c = __popc(L.mask[L.blocks[j]] & 0xFFFF);
    if (c > 0 && c < kBlock) { ++src; tl += c; }
  }
  int src_tot, tl_tot;
  (void)block_excl_scan(src, sh_scan, &src_tot);
  (void)block_excl_scan(tl, sh_scan, &tl_tot);
  if (pending_admit) { src_tot += 1; tl_tot += 1; }
  const int ndst = (tl_tot + kBlock - 1) / kBlock;
  if (!(src_tot > ndst)) { *t_live_out = 0; return 0; }
  *t_live_out = tl_tot;
  return ndst;
}

// The same with the test evaluated here: one lane of each warp divides
// (double arithmetic is slow on this part).
__device__ __forceinline__ int lane_plan(const LaneRefs& L, int nb, int n_live, bool forced, float theta_f,
                         bool pending_admit, int* t_live_out, int* sh_scan) {
  const int N = nb + (pending_admit ? 1 : 0);
  int over = 0;
  if ((threadIdx.x & 31) == 0 && N > 0) over = frag_over(n_live, N, theta_f) ? 1 : 0;
  over = __shfl_sync(0xffffffffu, over, 0);
  return lane_plan_given(L, nb, over != 0, forced, pending_admit, t_live_out, sh_scan);
}

}  // namespace kve
