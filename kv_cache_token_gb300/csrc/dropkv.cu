// D3: DropKV prefill-window scoring (DropKV explainer: Lemma 1; the fused
// scoring paragraph: stream K/V tiles, recompute each weight from the
// log-sum-exp, expand ||a - v||^2 = ||a||^2 + ||v||^2 - 2<a, v> so every V
// tile is read once per pass, never build the window x context x d tensor).
//
// Rows of a lane are its g query heads x w window queries (row = h * w + i).
// pass 1 (grid: key chunks x lanes x 128-row groups): causal flash attention
//   of the rows over one key chunk -> per-chunk (max, sum, unnormalised a).
// combine: per row, LSE and a = out (fp32 outputs), a split into bf16 hi + lo
//   for the tensor cores, ||a||^2.
// pass 2 (same grid): S = Q K^T and G = a V^T on the tensor cores;
//   per (row, key): p = exp(s - LSE), term = p / (1 - p) * sqrt(max(0,
//   ||a||^2 + ||v||^2 - 2 G)) (+inf where 1 - p <= 0); column sums over the
//   CTA's rows -> one partial per row group.
// finalize: scores = sum of the row-group partials.
#include <cudaTypedefs.h>
#include <new>
#include <type_traits>

#include "kvevict_internal.cuh"
#include "tcgen05.cuh"

namespace kve {
namespace {

constexpr int kD = 128;
constexpr int kRowStride = kD * 2 + 16;         // bytes per staged row
constexpr int kKeyTile = 32;                    // keys per tile
constexpr int kChunkMin = 1024;                 // keys per CTA, at least (the workspace holds cap / kChunkMin chunks)
constexpr int kWarps = 8;                       // 8 x 16 = 128 rows per CTA
constexpr int kRowsPerCta = kWarps * 16;
constexpr int kMaxRowGroups = 4;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void split_bf16(float p0, float p1, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
  float2 hf = __bfloat1622float2(h);
  __nv_bfloat162 l = __floats2bfloat162_rn(p0 - hf.x, p1 - hf.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}

struct D3Args {
  LayerState ls;
  Workspace ws;
  Dims dm;
  const __nv_bfloat16* q;   // [B][Hq][w][d]
  const int32_t* qpos;      // [w]
  int w, rows, rows_cap, chunks, chunk_keys;   // chunk_keys: keys per CTA, a multiple of 128
  float* lse_out; float* a_out; float* scores;
  float* col_out;   // where pass 2 leaves each key's column sum (scores, or scratch ahead of pooling)
  float scale2;
};

// What pass 2 sums per (row, key):
//   kResidual  the DropKV term p / (1 - p) ||a - v||, keys at or before the row;
//   kMassCausal  the weight p, keys at or before the row (SnapKV's prefill
//                observation: the window rows' attention paid to each key);
//   kMassLater   the weight p, keys strictly before the row (H2O's
//                cumulative score, which sums the rows t >= j + 1).
enum D3Mode { kResidual = 0, kMassCausal = 1, kMassLater = 2 };

// Shared staging of one key tile: K rows, V rows, positions, |v|^2.
struct Tile {
  unsigned char k[kKeyTile * kRowStride];
  unsigned char v[kKeyTile * kRowStride];
  int pos[kKeyTile];
  float vn[kKeyTile];
};

// Issue the cp.async copies of key tile [j0, j0 + 32) of lane l into t
// (K rows only when kV is false).
template <bool kV = true>
__device__ __forceinline__ void load_tile(Tile& t, const D3Args& A, int l, int n, int j0) {
  const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(A.ls.k_pool);
  const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(A.ls.v_pool);
  const size_t lo = static_cast<size_t>(l) * A.dm.cap;
  const size_t pool_rows = static_cast<size_t>(A.dm.P) * kBlock;
  // 32 keys x 2 tensors x 16 pieces of 16 bytes = 1024 pieces
  for (int e = threadIdx.x; e < kKeyTile * 2 * 16; e += blockDim.x) {
    const int key = e >> 5, tens = (e >> 4) & 1, piece = e & 15;
    const int j = j0 + key;
    if (!kV && tens) continue;
    unsigned char* dst = (tens ? t.v : t.k) + key * kRowStride + piece * 16;
    if (j < n) {
      int s = A.ls.slot[lo + j];
      if (s < 0 || static_cast<size_t>(s) >= pool_rows) { set_status(A.ws.status, ST_BAD_INDEX); s = 0; }
      const __nv_bfloat16* src = (tens ? vp : kp) + static_cast<size_t>(s) * kD + piece * 8;
      cp_async16(dst, src);
    } else {
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
  }
  for (int e = threadIdx.x; e < kKeyTile; e += blockDim.x) {
    const int j = j0 + e;
    t.pos[e] = j < n ? A.ls.pos[lo + j] : 0x7FFFFFFF;
  }
}

// Q (or any [rows][d] bf16 operand) as the A fragments of the warp's 16 rows.
__device__ __forceinline__ void load_afrag_q(uint32_t (&fa)[8][4], const D3Args& A, int b, int kh, int r0) {
  const int gq = (threadIdx.x & 31) >> 2, cq = threadIdx.x & 3;
  const int rr[2] = {r0 + gq, r0 + gq + 8};
  const __nv_bfloat16* ptr[2];
  bool ok[2];
  for (int u = 0; u < 2; ++u) {
    const int r = rr[u];
    ok[u] = r < A.rows;
    const int h = ok[u] ? r / A.w : 0, i = ok[u] ? r % A.w : 0;
    ptr[u] = A.q + ((static_cast<size_t>(b) * A.dm.Hq + kh * A.dm.g + h) * A.w + i) * kD;
  }
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int c0 = ks * 16 + cq * 2;
    fa[ks][0] = ok[0] ? *reinterpret_cast<const uint32_t*>(ptr[0] + c0) : 0u;
    fa[ks][1] = ok[1] ? *reinterpret_cast<const uint32_t*>(ptr[1] + c0) : 0u;
    fa[ks][2] = ok[0] ? *reinterpret_cast<const uint32_t*>(ptr[0] + c0 + 8) : 0u;
    fa[ks][3] = ok[1] ? *reinterpret_cast<const uint32_t*>(ptr[1] + c0 + 8) : 0u;
  }
}
__device__ __forceinline__ void load_afrag_rows(uint32_t (&fa)[8][4], const __nv_bfloat16* base, int rows, int r0) {
  const int gq = (threadIdx.x & 31) >> 2, cq = threadIdx.x & 3;
  const int ra = r0 + gq, rb = r0 + gq + 8;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int c0 = ks * 16 + cq * 2;
    fa[ks][0] = ra < rows ? *reinterpret_cast<const uint32_t*>(base + static_cast<size_t>(ra) * kD + c0) : 0u;
    fa[ks][1] = rb < rows ? *reinterpret_cast<const uint32_t*>(base + static_cast<size_t>(rb) * kD + c0) : 0u;
    fa[ks][2] = ra < rows ? *reinterpret_cast<const uint32_t*>(base + static_cast<size_t>(ra) * kD + c0 + 8) : 0u;
    fa[ks][3] = rb < rows ? *reinterpret_cast<const uint32_t*>(base + static_cast<size_t>(rb) * kD + c0 + 8) : 0u;
  }
}

// S[16 rows][32 keys] = A B^T with B rows staged in smem (K or V tile)
__device__ __forceinline__ void tile_rows_dot(float (&acc)[4][4], const uint32_t (&fa)[8][4], const unsigned char* rowsm) {
  const int lane = threadIdx.x & 31;
  const int tok = (lane & 7) + ((lane >> 4) << 3);
  const int colb = ((lane >> 3) & 1) * 16;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint32_t addr = smem_u32(rowsm + (half * 16 + tok) * kRowStride + colb);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(addr + ks * 32, b0, b1, b2, b3);
      mma_bf16(acc[half * 2 + 0], fa[ks], b0, b1);
      mma_bf16(acc[half * 2 + 1], fa[ks], b2, b3);
    }
  }
}

// ---------------------------------------------------------------------------
// pass 1
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kWarps * 32) d3_pass1_kernel(D3Args A) {
  __shared__ __align__(128) Tile tiles[2];
  const int chunk = blockIdx.x, l = blockIdx.y, rg = blockIdx.z;
  const int n = min(max(A.ls.count[l], 0), A.dm.cap);
  const int j_begin = chunk * A.chunk_keys;
  if (j_begin >= n) return;
  const int j_end = min(n, j_begin + A.chunk_keys);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, cq = lane & 3;
  const int b = l / A.dm.Hkv, kh = l % A.dm.Hkv;
  const int r0 = rg * kRowsPerCta + warp * 16;
  uint32_t qa[8][4];
  load_afrag_q(qa, A, b, kh, r0);
  const int ra = r0 + gq, rb = r0 + gq + 8;
  const int qpa = ra < A.rows ? A.qpos[ra % A.w] : -1;
  const int qpb = rb < A.rows ? A.qpos[rb % A.w] : -1;
  float o[16][4];
#pragma unroll
  for (int dn = 0; dn < 16; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
  float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;

  const int ntiles = (j_end - j_begin + kKeyTile - 1) / kKeyTile;
  load_tile(tiles[0], A, l, n, j_begin);
  cp_commit();
  for (int t = 0; t < ntiles; ++t) {
    if (t + 1 < ntiles) load_tile(tiles[(t + 1) & 1], A, l, n, j_begin + (t + 1) * kKeyTile);
    cp_commit();
    cp_wait<1>();
    __syncthreads();
    const Tile& T = tiles[t & 1];
    float s[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    tile_rows_dot(s, qa, T.k);
    float tma = -INFINITY, tmb = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int kp = T.pos[nt * 8 + cq * 2 + e];
        s[nt][e] = kp <= qpa ? s[nt][e] * A.scale2 : -INFINITY;
        s[nt][2 + e] = kp <= qpb ? s[nt][2 + e] * A.scale2 : -INFINITY;
        tma = fmaxf(tma, s[nt][e]);
        tmb = fmaxf(tmb, s[nt][2 + e]);
      }
    }
    tma = fmaxf(tma, __shfl_xor_sync(0xffffffffu, tma, 1));
    tma = fmaxf(tma, __shfl_xor_sync(0xffffffffu, tma, 2));
    tmb = fmaxf(tmb, __shfl_xor_sync(0xffffffffu, tmb, 1));
    tmb = fmaxf(tmb, __shfl_xor_sync(0xffffffffu, tmb, 2));
    const float mna = fmaxf(ma, tma), mnb = fmaxf(mb, tmb);
    const float ca = (mna == -INFINITY) ? 1.f : exp2f(ma - mna);
    const float cb = (mnb == -INFINITY) ? 1.f : exp2f(mb - mnb);
    ma = mna;
    mb = mnb;
    float p[4][4];
    float psa = 0.f, psb = 0.f;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        p[nt][e] = (mna == -INFINITY) ? 0.f : exp2f(s[nt][e] - mna);
        p[nt][2 + e] = (mnb == -INFINITY) ? 0.f : exp2f(s[nt][2 + e] - mnb);
        psa += p[nt][e];
        psb += p[nt][2 + e];
      }
    }
    la = la * ca + psa;
    lb = lb * cb + psb;
#pragma unroll
    for (int dn = 0; dn < 16; ++dn) {
      o[dn][0] *= ca; o[dn][1] *= ca; o[dn][2] *= cb; o[dn][3] *= cb;
    }
    // PV: two 16-key k-steps
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      uint32_t ah[4], al[4];
      split_bf16(p[2 * kk][0], p[2 * kk][1], ah[0], al[0]);
      split_bf16(p[2 * kk][2], p[2 * kk][3], ah[1], al[1]);
      split_bf16(p[2 * kk + 1][0], p[2 * kk + 1][1], ah[2], al[2]);
      split_bf16(p[2 * kk + 1][2], p[2 * kk + 1][3], ah[3], al[3]);
      const int tok = (lane & 7) + (((lane >> 3) & 1) << 3) + kk * 16;
      const uint32_t addr = smem_u32(T.v + tok * kRowStride) + (lane >> 4) * 16;
#pragma unroll
      for (int dn = 0; dn < 16; dn += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(addr + dn * 16, b0, b1, b2, b3);
        mma_bf16(o[dn], ah, b0, b1);
        mma_bf16(o[dn], al, b0, b1);
        mma_bf16(o[dn + 1], ah, b2, b3);
        mma_bf16(o[dn + 1], al, b2, b3);
      }
    }
    __syncthreads();
  }
  la += __shfl_xor_sync(0xffffffffu, la, 1);
  la += __shfl_xor_sync(0xffffffffu, la, 2);
  lb += __shfl_xor_sync(0xffffffffu, lb, 1);
  lb += __shfl_xor_sync(0xffffffffu, lb, 2);
  const size_t stride = kD + 2;
  float* part = A.ws.d3_part + (static_cast<size_t>(l) * A.chunks + chunk) * static_cast<size_t>(A.rows_cap) * stride;
  if (ra < A.rows) {
    float* pr = part + static_cast<size_t>(ra) * stride;
#pragma unroll
    for (int dn = 0; dn < 16; ++dn) *reinterpret_cast<float2*>(pr + dn * 8 + cq * 2) = make_float2(o[dn][0], o[dn][1]);
    if (cq == 0) { pr[kD] = ma; pr[kD + 1] = la; }
  }
  if (rb < A.rows) {
    float* pr = part + static_cast<size_t>(rb) * stride;
#pragma unroll
    for (int dn = 0; dn < 16; ++dn) *reinterpret_cast<float2*>(pr + dn * 8 + cq * 2) = make_float2(o[dn][2], o[dn][3]);
    if (cq == 0) { pr[kD] = mb; pr[kD + 1] = lb; }
  }
}

// ---------------------------------------------------------------------------
// combine: grid (row groups of 8, lanes), one warp per row; the chunks'
// (max, sum) in lanes of the warp, then each lane accumulates 4 of the d
// columns over the chunks.
// ---------------------------------------------------------------------------
// kA false: the LSE alone (the chunks' partial outputs were not written).
template <bool kA>
__global__ void __launch_bounds__(256) d3_combine_kernel(D3Args A) {
  // launched as a dependent of pass 1: its partials are complete past the
  // wait; pass 2 may launch at once (all of this grid is resident, and pass
  // 2 waits for it before reading what it writes)
  grid_dep_wait();
  grid_dep_launch();
  const int l = blockIdx.y;
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= A.rows) return;
  const int n = min(max(A.ls.count[l], 0), A.dm.cap);
  const int nch = (n + A.chunk_keys - 1) / A.chunk_keys;
  const int b = l / A.dm.Hkv, kh = l % A.dm.Hkv;
  const size_t stride = kD + 2;
  const size_t chunk_stride = static_cast<size_t>(A.rows_cap) * stride;
  const int h = r / A.w, i = r % A.w;
  const float* base = A.ws.d3_part + static_cast<size_t>(l) * A.chunks * chunk_stride + static_cast<size_t>(r) * stride;
  float M = -INFINITY;
  for (int c = lane; c < nch; c += 32) M = fmaxf(M, base[c * chunk_stride + kD]);
  M = warp_max(M);
  float Lp = 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  // 32 chunks at a time: lane c holds chunk c's scale, broadcast by shuffle,
  // so the partial rows' loads do not wait on one another
  for (int c0 = 0; c0 < nch; c0 += 32) {
    const int c = c0 + lane;
    const float m = c < nch ? base[c * chunk_stride + kD] : -INFINITY;
    const float sc_mine = m == -INFINITY ? 0.f : exp2f(m - M);
    if (c < nch) Lp += base[c * chunk_stride + kD + 1] * sc_mine;
    const int cnt = kA ? min(32, nch - c0) : 0;
    const float* bc = base + static_cast<size_t>(c0) * chunk_stride + lane * 4;
#pragma unroll 8
    for (int u = 0; u < cnt; ++u) {
      const float sc = __shfl_sync(0xffffffffu, sc_mine, u);
      // partial rows are 130 floats: 8-byte aligned, so two float2 loads
      const float2 x0 = *reinterpret_cast<const float2*>(bc + u * chunk_stride);
      const float2 x1 = *reinterpret_cast<const float2*>(bc + u * chunk_stride + 2);
      acc[0] = fmaf(x0.x, sc, acc[0]);
      acc[1] = fmaf(x0.y, sc, acc[1]);
      acc[2] = fmaf(x1.x, sc, acc[2]);
      acc[3] = fmaf(x1.y, sc, acc[3]);
    }
  }
  for (int o = 16; o > 0; o >>= 1) Lp += __shfl_xor_sync(0xffffffffu, Lp, o);
  const float lse2 = M + log2f(Lp);
  const size_t orow = (static_cast<size_t>(b) * A.dm.Hq + kh * A.dm.g + h) * A.w + i;
  const size_t wrow = static_cast<size_t>(l) * A.rows_cap + r;
  if (!kA) {
    if (lane == 0) {
      A.lse_out[orow] = lse2 * kLn2;
      A.ws.d3_rowc[wrow * 2 + 0] = lse2;
      A.ws.d3_rowc[wrow * 2 + 1] = 0.f;
    }
    return;
  }
  float nrm = 0.f;
  float av[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    av[u] = acc[u] / Lp;
    nrm += av[u] * av[u];
  }
  *reinterpret_cast<float4*>(A.a_out + orow * kD + lane * 4) = make_float4(av[0], av[1], av[2], av[3]);
#pragma unroll
  for (int u = 0; u < 4; u += 2) {
    const __nv_bfloat162 hi = __floats2bfloat162_rn(av[u], av[u + 1]);
    const float2 hf = __bfloat1622float2(hi);
    const __nv_bfloat162 lo = __floats2bfloat162_rn(av[u] - hf.x, av[u + 1] - hf.y);
    *reinterpret_cast<__nv_bfloat162*>(A.ws.d3_ahi + wrow * kD + lane * 4 + u) = hi;
    *reinterpret_cast<__nv_bfloat162*>(A.ws.d3_alo + wrow * kD + lane * 4 + u) = lo;
  }
  for (int o = 16; o > 0; o >>= 1) nrm += __shfl_xor_sync(0xffffffffu, nrm, o);
  if (lane == 0) {
    A.lse_out[orow] = lse2 * kLn2;
    A.ws.d3_rowc[wrow * 2 + 0] = lse2;
    A.ws.d3_rowc[wrow * 2 + 1] = nrm;
  }
}

// One (row, key) term of the DropKV score: p / (1 - p) * ||a - v||, with
// x = log2 p.  ||a - v||^2 comes from the expansion r2 = |a|^2 + |v|^2 - 2<a,v>
// except where p > 1/2: there a is within (1 - p) of v and the expansion
// cancels, so the distance is taken directly from the fp32 a and the staged v
// row (at most one key per row can have p > 1/2).  1 - p uses expm1 near 1.
__device__ __forceinline__ float residual_term(float x, float r2, const float* arow, const unsigned char* vrow) {
  const float p = exp2f(x);
  if (!(p > 0.f)) return 0.f;
  if (p <= 0.5f) return p / (1.f - p) * sqrtf(fmaxf(0.f, r2));
  const float om = -expm1f(x * kLn2);
  if (!(om > 0.f)) return INFINITY;
  const __nv_bfloat16* v = reinterpret_cast<const __nv_bfloat16*>(vrow);
  float acc = 0.f;
  for (int e = 0; e < kD; ++e) {
    const float df = arow[e] - __bfloat162float(v[e]);
    acc = fmaf(df, df, acc);
  }
  return p / om * sqrtf(acc);
}

// ---------------------------------------------------------------------------
// pass 2
// ---------------------------------------------------------------------------
template <int kMode>
__global__ void __launch_bounds__(kWarps * 32) d3_pass2_kernel(D3Args A) {
  constexpr bool kRes = kMode == kResidual;
  __shared__ __align__(128) Tile tiles[2];
  __shared__ float colsum[kWarps][kKeyTile];
  const int chunk = blockIdx.x, l = blockIdx.y, rg = blockIdx.z;
  const int n = min(max(A.ls.count[l], 0), A.dm.cap);
  const int j_begin = chunk * A.chunk_keys;
  if (j_begin >= n) return;
  const int j_end = min(n, j_begin + A.chunk_keys);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, cq = lane & 3;
  const int b = l / A.dm.Hkv, kh = l % A.dm.Hkv;
  const int r0 = rg * kRowsPerCta + warp * 16;
  const size_t wbase = static_cast<size_t>(l) * A.rows_cap;
  uint32_t qa[8][4], ah[8][4], al[8][4];
  load_afrag_q(qa, A, b, kh, r0);
  if (kRes) {
    load_afrag_rows(ah, A.ws.d3_ahi + wbase * kD, A.rows, r0);
    load_afrag_rows(al, A.ws.d3_alo + wbase * kD, A.rows, r0);
  }
  const int ra = r0 + gq, rb = r0 + gq + 8;
  const bool oka = ra < A.rows, okb = rb < A.rows;
  const int qpa = oka ? A.qpos[ra % A.w] : -1;
  const int qpb = okb ? A.qpos[rb % A.w] : -1;
  const float lsa = oka ? A.ws.d3_rowc[(wbase + ra) * 2] : 0.f;
  const float lsb = okb ? A.ws.d3_rowc[(wbase + rb) * 2] : 0.f;
  const float ana = oka ? A.ws.d3_rowc[(wbase + ra) * 2 + 1] : 0.f;
  const float anb = okb ? A.ws.d3_rowc[(wbase + rb) * 2 + 1] : 0.f;
  float* out = A.ws.d3_score_part + (static_cast<size_t>(rg) * A.dm.lanes + l) * A.dm.cap;
  auto arow_of = [&](int r, bool ok) -> const float* {
    if (!ok) return A.a_out;
    const int h = r / A.w, i = r % A.w;
    return A.a_out + ((static_cast<size_t>(b) * A.dm.Hq + kh * A.dm.g + h) * A.w + i) * kD;
  };
  const float* arow_a = arow_of(ra, oka);
  const float* arow_b = arow_of(rb, okb);

  const int ntiles = (j_end - j_begin + kKeyTile - 1) / kKeyTile;
  load_tile<kRes>(tiles[0], A, l, n, j_begin);
  cp_commit();
  for (int t = 0; t < ntiles; ++t) {
    if (t + 1 < ntiles) load_tile<kRes>(tiles[(t + 1) & 1], A, l, n, j_begin + (t + 1) * kKeyTile);
    cp_commit();
    cp_wait<1>();
    __syncthreads();
    Tile& T = tiles[t & 1];
    // |v|^2 of the tile's keys (warp 0)
    if (kRes && warp == 0) {
      const __nv_bfloat16* vr = reinterpret_cast<const __nv_bfloat16*>(T.v + lane * kRowStride);
      float acc = 0.f;
      for (int e = 0; e < kD; ++e) {
        const float x = __bfloat162float(vr[(e + lane * 4) & (kD - 1)]);
        acc = fmaf(x, x, acc);
      }
      T.vn[lane] = acc;
    }
    float s[4][4], g[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
      g[nt][0] = g[nt][1] = g[nt][2] = g[nt][3] = 0.f;
    }
    tile_rows_dot(s, qa, T.k);
    if (kRes) {
      tile_rows_dot(g, ah, T.v);
      tile_rows_dot(g, al, T.v);
    }
    __syncthreads();   // |v|^2 ready
    float cs[4][2];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = nt * 8 + cq * 2 + e;
        const int kp = T.pos[key];
        const float vn = T.vn[key];
        float term = 0.f;
        if (kRes) {
          if (kp <= qpa) term += residual_term(s[nt][e] * A.scale2 - lsa, ana + vn - 2.f * g[nt][e], arow_a,
                                               T.v + key * kRowStride);
          if (kp <= qpb) term += residual_term(s[nt][2 + e] * A.scale2 - lsb, anb + vn - 2.f * g[nt][2 + e], arow_b,
                                               T.v + key * kRowStride);
        } else {
          const bool ca = kMode == kMassLater ? kp < qpa : kp <= qpa;
          const bool cb = kMode == kMassLater ? kp < qpb : kp <= qpb;
          if (ca) term += exp2f(s[nt][e] * A.scale2 - lsa);
          if (cb) term += exp2f(s[nt][2 + e] * A.scale2 - lsb);
        }
        // sum over the 8 row groups of the warp (lanes with equal cq)
        term += __shfl_xor_sync(0xffffffffu, term, 4);
        term += __shfl_xor_sync(0xffffffffu, term, 8);
        term += __shfl_xor_sync(0xffffffffu, term, 16);
        cs[nt][e] = term;
      }
    }
    if (gq == 0) {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        colsum[warp][nt * 8 + cq * 2 + 0] = cs[nt][0];
        colsum[warp][nt * 8 + cq * 2 + 1] = cs[nt][1];
      }
    }
    __syncthreads();
    if (threadIdx.x < kKeyTile) {
      const int j = j_begin + t * kKeyTile + threadIdx.x;
      float tot = 0.f;
      for (int w = 0; w < kWarps; ++w) tot += colsum[w][threadIdx.x];
      if (j < j_end) out[j] = tot;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(256) d3_finalize_kernel(D3Args A, int groups) {
  const int l = blockIdx.y;
  const int n = min(max(A.ls.count[l], 0), A.dm.cap);
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < n; j += gridDim.x * blockDim.x) {
    float tot = 0.f;
    for (int rg = 0; rg < groups; ++rg)
      tot += A.ws.d3_score_part[(static_cast<size_t>(rg) * A.dm.lanes + l) * A.dm.cap + j];
    A.col_out[static_cast<size_t>(l) * A.dm.cap + j] = tot;
  }
}

// SnapKV pooling of the column sums (SnapKV, "How it works": pooled[i] =
// max of sums[i - r .. i + r], clamped at the lane's ends; a NaN sum wins,
// as a max over a set holding NaN is NaN).  One CTA per 1024 kept entries of
// a lane, sums staged with a halo of r on each side.
constexpr int kPoolTile = 1024;
__global__ void __launch_bounds__(256) d3_pool_kernel(const float* __restrict__ sums, float* __restrict__ out,
                                                      const int32_t* __restrict__ count, int cap, int r) {
  extern __shared__ float pool_sm[];
  const int l = blockIdx.y;
  const int n = min(max(count[l], 0), cap);
  const int j0 = blockIdx.x * kPoolTile;
  if (j0 >= n) return;
  const int lo = max(0, j0 - r), hi = min(n, j0 + kPoolTile + r);
  const float* src = sums + static_cast<size_t>(l) * cap;
  for (int j = lo + threadIdx.x; j < hi; j += blockDim.x) pool_sm[j - lo] = src[j];
  __syncthreads();
  const int jend = min(n, j0 + kPoolTile);
  for (int j = j0 + threadIdx.x; j < jend; j += blockDim.x) {
    const int a = max(0, j - r), b = min(n - 1, j + r);
    float m = pool_sm[a - lo];
    for (int i = a + 1; i <= b; ++i) {
      const float x = pool_sm[i - lo];
      if (x != x || x > m) m = x;
    }
    out[static_cast<size_t>(l) * cap + j] = m;
  }
}

// ---------------------------------------------------------------------------
// tcgen05 path.  A CTA owns one 128-row tile of a lane's window rows (rows
// 0-127, and 128-255 when there are more) and one chunk of the lane's keys;
// the CTAs of the two row tiles of a chunk are grid neighbours, run side by
// side and read the same K and V rows (the second read is served by L2).
//
// pass 1, per 64-key tile: S = Q K^T on the tensor cores.  Two groups of four
//   row warps (one thread per row) take alternate tiles.  Each group keeps its
//   own running max and sum per row and its own output accumulator O_g in
//   tensor memory; the two are merged at the end like two chunks, so no two
//   threads ever share a row's softmax state.  A thread masks and
//   exponentiates its row of S (lazy rescale of the running max), writes P as
//   bf16 hi + lo over S, and O_g += P V takes P from tensor memory and V
//   (MN-major) from shared memory.  The group also takes |v|^2 of the tile's
//   keys for pass 2.  Tensor-memory columns: O_A 0, O_B 128, four S/P buffers
//   at 256 + 64 b (tile t in b = t % 4); S runs three tiles ahead of P V.  K
//   and V have rings of their own: a K stage is free once its S is computed,
//   a V stage once P V and the |v|^2 job are done with it.
// pass 2, per 128-key tile: S^T = K Q^T and G^T = V a^T (a as bf16 hi + lo;
//   Q, a hi and a lo stay in shared memory).  Tensor-memory lanes are keys
//   and columns rows, so a thread owns one key and sums its terms over 64
//   rows in a register: no reduction across threads.  The two warps sharing a
//   key add their sums in a fixed order; with two row tiles both CTAs add
//   theirs into the output, which pass 1 zeroed (two addends onto zero: the
//   result is the same whichever lands first).  Tensor-memory columns:
//   buffer b (tile t % 2) holds S^T at 256 b and G^T at 256 b + 128.
// The attention-mass modes skip V: pass 1 keeps (max, sum) per row and
// pass 2 sums the weights p themselves.
// K and V rows arrive by TMA: a 64-row box per 64 consecutive slots (the
// layout a prefill leaves), 16-row boxes for runs of 16, else gathers of four
// rows; the copy engine applies the 128-byte swizzle the MMAs read.
// ---------------------------------------------------------------------------
constexpr int kTcRows = 256;                 // window rows per lane on this path (two row tiles)
constexpr int kRowTile = 128;
constexpr int kQBytes = 2 * kRowTile * 128;  // [d half][128 rows][128 B]
constexpr int kP1Keys = 128;
constexpr int kP1Bufs = 2;                   // S/P buffers in tensor memory (after O_0, O_1)
constexpr int kP1KSt = 3, kP1VSt = 2;        // K and V ring depths
constexpr int kP1Tile = kP1Keys * 256;       // one K or V tile (32 KB)
constexpr int kP1Smem = kQBytes + (kP1KSt + kP1VSt) * kP1Tile + 1024;
constexpr int kP1KProd = 8, kP1VProd = 9, kP1Issuer = 10, kP1VnWarp0 = 11, kP1VnWarps = 2;
constexpr int kP1Depth = 3;                  // tiles of slots the producers read ahead
constexpr int kP1Threads = 13 * 32;
constexpr int kP2Keys = 128;
constexpr int kP2St = 2;                     // K/V stages
constexpr int kP2Tile = kP2Keys * 256;       // one K or V tile (32 KB)
constexpr int kP2RowWarps = 16;             // 4 per lane quarter, 32 rows each
constexpr int kP2Producer = 16, kP2Issuer = 17;
constexpr int kP2Threads = 18 * 32;
constexpr int kTileKeys = kP2Keys;           // chunks hold whole tiles of both passes
constexpr float kTcRescale = 8.f;
constexpr uint32_t kIdPV = tc::idesc_bf16(128, kD, 1);
constexpr uint32_t kId128 = tc::idesc_bf16(128, 128, 0);
static_assert(kChunkMin % kTileKeys == 0, "chunks hold whole tiles");

// Hardware approximations (PTX ex2/rcp/sqrt .approx.ftz, relative error
// about 2^-22; results below 2^-126 flush to zero).
__device__ __forceinline__ float hw_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Two fp32 lanes per instruction (the packed .f32x2 arithmetic): each lane
// is rounded exactly as the scalar fmaf, + or * rounds it.
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 a, b, c, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n mov.b64 c, {%6, %7};\n"
      " fma.rn.f32x2 d, a, b, c;\n mov.b64 {%0, %1}, d;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n add.rn.f32x2 d, a, b;\n"
      " mov.b64 {%0, %1}, d;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 f2_sub(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n sub.rn.f32x2 d, a, b;\n"
      " mov.b64 {%0, %1}, d;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n mul.rn.f32x2 d, a, b;\n"
      " mov.b64 {%0, %1}, d;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float hw_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float hw_sqrt(float x) {
  float y;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float hw_rsqrt(float x) {
  float y;
  asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}
// byte offset of bf16 element e of key row k in a swizzled tile of kKeys rows
// ([d half][kKeys rows][128 B])
template <int kKeys>
__device__ __forceinline__ int sw_off(int k, int e) {
  return (e >> 6) * (kKeys * 128) + k * 128 + ((((e & 63) >> 3) ^ (k & 7)) << 4) + (e & 7) * 2;
}
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy reads of them (the tensor cores reading an operand).
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void cp_async16_zf(void* dst, const void* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(ok ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async4i(int* dst, const int* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int threads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// The K and V pool tensor maps of one layer (see kTmapsPerLayer).
struct D3Maps {
  CUtensorMap m[kTmapsPerLayer];   // K gather, V gather, K 16 rows, V 16 rows, K 64 rows, V 64 rows
};

// One tiled TMA copy: rows y .. y + box - 1 of the 64-element half row at
// column x into consecutive 128-byte rows at dst (128-byte swizzle), the box
// bytes completing on bar.
__device__ __forceinline__ void tma_rows(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// One TMA gather: the 64-element half rows at column x of four pool rows
// (slots r0..r3) into four consecutive 128-byte rows at dst, swizzled by
// their shared-memory address (the UMMA 128-byte K-major layout when dst
// lies in a 1024-byte aligned tile); 512 bytes complete on bar.  A row past
// the pool reads as zeros.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* map, int x, int r0, int r1, int r2, int r3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

// One producer warp streaming the chunk's tiles of kKeys keys into a ring of
// kStages stages.  A stage holds the K tile (kK) and then the V tile (kV),
// each [d half][kKeys rows][128 B]; with kPos the keys' positions go to
// pos[stage][key] for the row warps.  Per tile: wait until the stage is
// empty, store the positions, arm the stage's full barrier with the bytes to
// come, issue the copies.  The keys' slots (and positions) are read ahead, so
// the producer does not wait a global round trip per tile: kDepth > 0 tiles
// ahead by 4-byte cp.async into pf_s / pf_p ([kDepth][kKeys], one commit
// group per tile; each lane copies and reads back only its own keys), or,
// with kDepth 0, one tile ahead into registers (enough when the producer
// mostly waits for empty stages).  A key past the chunk reads a pool row past
// the end: zeros.  A tile whose keys sit
// in consecutive slots takes one 64-row copy per 64 keys, tensor and d half;
// otherwise each 16-key group in consecutive slots takes a 16-row copy and
// the rest are gathered four rows per copy (a TMA instruction costs tens of
// nanoseconds to issue, so the fewer the better).
template <int kKeys, int kStages, bool kK, bool kV, bool kPos, int kDepth>
__device__ __forceinline__ void d3_produce(const D3Args& A, const D3Maps& mp, int l, int j_begin, int j_end,
                                           int ntiles, unsigned char* ring, uint64_t* full, uint64_t* empty,
                                           int* pos, int* pf_s, int* pf_p) {
  constexpr int kpl = kKeys / 32;   // keys per lane
  constexpr int kHalfB = kKeys * 128;
  constexpr int kTileB = 2 * kHalfB;
  constexpr uint32_t kStageB = (kK ? kTileB : 0) + (kV ? kTileB : 0);
  constexpr int kGl = kKeys / 4;    // gather lanes: lane L < kGl takes keys 4L .. 4L + 3
  const int lane = threadIdx.x & 31;
  const size_t lo = static_cast<size_t>(l) * A.dm.cap;
  const int rows_max = A.dm.P * kBlock;
  int sl[kpl], ps[kpl];
  auto read = [&](int t, int (&s)[kpl], int (&p)[kpl]) {
#pragma unroll
    for (int i = 0; i < kpl; ++i) {
      const int j = j_begin + t * kKeys + kpl * lane + i;
      const bool ok = t < ntiles && j < j_end;
      s[i] = ok ? A.ls.slot[lo + j] : rows_max;
      p[i] = (kPos && ok) ? A.ls.pos[lo + j] : 0x7FFFFFFF;
    }
  };
  auto prefetch = [&](int t) {
    if (t < ntiles) {
      const int bb = t % (kDepth > 0 ? kDepth : 1);
#pragma unroll
      for (int i = 0; i < kpl; ++i) {
        const int key = kpl * lane + i, j = j_begin + t * kKeys + key;
        if (j < j_end) {
          cp_async4i(pf_s + bb * kKeys + key, A.ls.slot + lo + j);
          if (kPos) cp_async4i(pf_p + bb * kKeys + key, A.ls.pos + lo + j);
        }
      }
    }
    cp_commit();
  };
  if (kDepth > 0) {
#pragma unroll
    for (int u = 0; u < kDepth; ++u) prefetch(u);
  } else {
    read(0, sl, ps);
  }
#pragma unroll 1
  for (int t = 0; t < ntiles; ++t) {
    int sn[kpl], pn[kpl];
    if (kDepth > 0) {
      cp_wait<(kDepth > 0 ? kDepth - 1 : 0)>();   // tile t's group has landed
      const int bb = t % (kDepth > 0 ? kDepth : 1);
#pragma unroll
      for (int i = 0; i < kpl; ++i) {
        const int key = kpl * lane + i, j = j_begin + t * kKeys + key;
        sl[i] = j < j_end ? pf_s[bb * kKeys + key] : rows_max;
        ps[i] = (kPos && j < j_end) ? pf_p[bb * kKeys + key] : 0x7FFFFFFF;
      }
      prefetch(t + kDepth);   // into the buffer just read (its values are in registers)
    } else {
      read(t + 1, sn, pn);
    }
    const int st = t % kStages;
    if (t >= kStages) (void)mbar_wait_bounded(&empty[st], ((t / kStages) - 1) & 1, A.ws.status);
#pragma unroll
    for (int i = 0; i < kpl; ++i) {
      const int j = j_begin + t * kKeys + kpl * lane + i;
      if (j < j_end && (sl[i] < 0 || sl[i] >= rows_max)) {
        set_status(A.ws.status, ST_BAD_INDEX);
        sl[i] = 0;
      }
      if (kPos) pos[st * kKeys + kpl * lane + i] = ps[i];
    }
    if (kK || kV) {
      // consecutive slots: the whole tile, and each 16-key group
      const int tbase = __shfl_sync(0xffffffffu, sl[0], 0);
      const int g16 = (kpl * lane) >> 4;   // this lane's 16-key group
      const int gfirst = __shfl_sync(0xffffffffu, sl[0], (16 * g16) / kpl);
      bool run_t = true, run_g = true;
#pragma unroll
      for (int i = 0; i < kpl; ++i) {
        run_t = run_t && sl[i] == tbase + kpl * lane + i;
        run_g = run_g && sl[i] == gfirst + kpl * lane + i - 16 * g16;
      }
      const bool tile_run = __all_sync(0xffffffffu, run_t) && tbase + kKeys <= rows_max;
      const unsigned runs = __ballot_sync(0xffffffffu, run_g);
      const int gl = lane % kGl;             // lanes past kGl compute harmless copies of lane gl's values
      const int ggrp = gl >> 2;              // the gather lane's 16-key group
      const unsigned gmask = ((1u << (16 / kpl)) - 1u) << ((16 * ggrp) / kpl);
      const int gbase = __shfl_sync(0xffffffffu, sl[0], (16 * ggrp) / kpl);
      const bool grp_run = (runs & gmask) == gmask && gbase + 16 <= rows_max;
      int g4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) g4[i] = __shfl_sync(0xffffffffu, sl[i % kpl], (4 * gl + i) / kpl);
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&full[st], kStageB);
      __syncwarp();
      unsigned char* stage = ring + static_cast<size_t>(st) * kStageB;
#pragma unroll
      for (int ten = 0; ten < 2; ++ten) {
        if ((ten == 0 && !kK) || (ten == 1 && !kV)) continue;
        unsigned char* dst = stage + ((ten == 1 && kK) ? kTileB : 0);
        const int mg = ten, m16 = 2 + ten, m64 = 4 + ten;
        if (tile_run) {
          if (lane == 0) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
              for (int c = 0; c < kKeys / 64; ++c)
                tma_rows(dst + hf * kHalfB + c * 8192, &mp.m[m64], hf * 64, tbase + 64 * c, &full[st]);
          }
        } else if (lane < kGl) {
          if (grp_run) {
            if ((lane & 3) == 0) {
#pragma unroll
              for (int hf = 0; hf < 2; ++hf)
                tma_rows(dst + hf * kHalfB + ggrp * 2048, &mp.m[m16], hf * 64, gbase, &full[st]);
            }
          } else {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
              tma_gather4(dst + hf * kHalfB + lane * 512, &mp.m[mg], hf * 64, g4[0], g4[1], g4[2], g4[3],
                          &full[st]);
          }
        }
      }
    } else {
      __syncwarp();
      if (lane == 0) mbar_arrive1(&full[st]);   // positions only
    }
    if (kDepth == 0) {
#pragma unroll
      for (int i = 0; i < kpl; ++i) {
        sl[i] = sn[i];
        ps[i] = pn[i];
      }
    }
  }
}

// The CTA's 128 window rows of Q (which = 0) or of a hi / a lo (1 / 2) into
// shared memory at dst in the UMMA 128-byte K-major layout, by 16-byte
// cp.async pieces (zeros past the rows), split over `threads` threads.
__device__ __forceinline__ void stage_rows(unsigned char* dst, int which, const D3Args& A, int l, int rt, int tid,
                                           int threads) {
  const int b = l / A.dm.Hkv, kh = l % A.dm.Hkv;
  for (int e = tid; e < kRowTile * 16; e += threads) {
    const int rr = e >> 4, c = e & 15, r = rt * kRowTile + rr;
    const bool ok = r < A.rows;
    const __nv_bfloat16* src = A.q;
    if (ok) {
      if (which == 0)
        src = A.q + ((static_cast<size_t>(b) * A.dm.Hq + kh * A.dm.g + r / A.w) * A.w + r % A.w) * kD + c * 8;
      else
        src = (which == 1 ? A.ws.d3_ahi : A.ws.d3_alo) + (static_cast<size_t>(l) * A.rows_cap + r) * kD + c * 8;
    }
    cp_async16_zf(dst + (c >> 3) * 16384 + rr * 128 + (((c & 7) ^ (rr & 7)) << 4), src, ok);
  }
}

struct P1Bars {
  uint64_t qfull;
  uint64_t kfull[kP1KSt], kempty[kP1KSt];
  uint64_t vfull[kP1VSt], vempty[kP1VSt];
  uint64_t x_full[kP1Bufs], x_free[kP1Bufs];
};

// pass 1.  Barriers: x_full[b] S(t) done (b = t % 2); x_free[b] the 8 row
// warps have read S(t) and written P(t); kfull / kempty and vfull / vempty
// the two rings (a K stage also carries the keys' positions, released by
// S(t) and the rows; vempty[s] completes once P V(t) and the |v|^2 warps are
// done with V stage s, which also tells the rows that P V(t) is complete).  Issue order: S(0),
// then per tile S(t + 1), P V(t): S(t + 1) reuses the buffer of P(t - 1),
// which P V(t - 1) read before it in the tensor core's order.
template <bool kWithV>
__global__ void __launch_bounds__(kP1Threads, 1) d3_p1_kernel(D3Args A, const __grid_constant__ D3Maps mp) {
  extern __shared__ unsigned char d3_dsm[];
  __shared__ __align__(8) P1Bars bar;
  __shared__ int sh_pos[kP1KSt * kP1Keys];
  __shared__ float sh_ml[2][kRowTile][2];
  __shared__ int pf_k[kP1Depth * kP1Keys], pf_v[kP1Depth * kP1Keys], pf_p[kP1Depth * kP1Keys];
  __shared__ uint32_t sh_taddr;
  const int nrt = (A.rows + kRowTile - 1) / kRowTile;
  const int rt = blockIdx.x % nrt, chunk = blockIdx.x / nrt, l = blockIdx.y;
  const int n = min(max(A.ls.count[l], 0), A.dm.cap);
  const int j_begin = chunk * A.chunk_keys;
  if (j_begin >= n) return;
  const int j_end = min(n, j_begin + A.chunk_keys);
  const int ntiles = (j_end - j_begin + kP1Keys - 1) / kP1Keys;
  unsigned char* sq = align1024(d3_dsm);
  unsigned char* skr = sq + kQBytes;
  unsigned char* svr = skr + kP1KSt * kP1Tile;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == kP1Issuer) tc::alloc(&sh_taddr, 512);
  if (tid == 0) {
    mbar_init(&bar.qfull, 8);
    for (int s = 0; s < kP1KSt; ++s) {
      mbar_init(&bar.kfull[s], 1);
      mbar_init(&bar.kempty[s], 1 + 8);   // S(t) and the 8 row warps (the keys' positions)
    }
    for (int s = 0; s < kP1VSt; ++s) {
      mbar_init(&bar.vfull[s], 1);
      mbar_init(&bar.vempty[s], 1 + kP1VnWarps);   // P V(t) and the |v|^2 warps
    }
    for (int b = 0; b < kP1Bufs; ++b) {
      mbar_init(&bar.x_full[b], 1);
      mbar_init(&bar.x_free[b], 8);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tl = sh_taddr;
  const size_t lo = static_cast<size_t>(l) * A.dm.cap;

  if (warp == kP1KProd) {
    d3_produce<kP1Keys, kP1KSt, true, false, true, kP1Depth>(A, mp, l, j_begin, j_end, ntiles, skr, bar.kfull,
                                                             bar.kempty, sh_pos, pf_k, pf_p);
  } else if (warp == kP1VProd) {
    if (kWithV)
      d3_produce<kP1Keys, kP1VSt, false, true, false, kP1Depth>(A, mp, l, j_begin, j_end, ntiles, svr, bar.vfull,
                                                                bar.vempty, nullptr, pf_v, nullptr);
  } else if (warp == kP1Issuer) {
    if (lane == 0) {
      // descriptors built once; each MMA advances one by a constant
      const uint64_t dq = tc::desc_sw128(smem_u32(sq), 16, 1024);
      const uint64_t dk0 = tc::desc_sw128(smem_u32(skr), 16, 1024);
      const uint64_t dv0 = tc::desc_sw128(smem_u32(svr), kP1Keys * 128, 1024);
      (void)mbar_wait_bounded(&bar.qfull, 0, A.ws.status);
      auto issue_s = [&](int u) {
        const int b = u % kP1Bufs, ks = u % kP1KSt;
        // without P V, the rows' reading of S(u - 2) is what frees its buffer
        // (with it, P V(u - 2) read that buffer before S(u) in issue order)
        if (!kWithV && u >= kP1Bufs)
          (void)mbar_wait_bounded(&bar.x_free[b], ((u / kP1Bufs) - 1) & 1, A.ws.status);
        (void)mbar_wait_bounded(&bar.kfull[ks], (u / kP1KSt) & 1, A.ws.status);
        tc::fence_after();
        const uint64_t dk = tc::desc_add(dk0, ks * kP1Tile);
        const uint32_t dS = tl + 256 + b * kP1Keys;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int off = (kk >> 2) * (kP1Keys * 128) + (kk & 3) * 32;   // d half, 16-element step
          tc::mma_ss(dS, tc::desc_add(dq, off), tc::desc_add(dk, off), kId128, kk > 0 ? 1u : 0u);
        }
        tc::commit(&bar.x_full[b]);
        tc::commit(&bar.kempty[ks]);
      };
      if (ntiles > 0) issue_s(0);
#pragma unroll 1
      for (int t = 0; t < ntiles; ++t) {
        if (t + 1 < ntiles) issue_s(t + 1);
        if (kWithV) {
          const int b = t % kP1Bufs, vs = t % kP1VSt;
          (void)mbar_wait_bounded(&bar.x_free[b], (t / kP1Bufs) & 1, A.ws.status);
          (void)mbar_wait_bounded(&bar.vfull[vs], (t / kP1VSt) & 1, A.ws.status);
          tc::fence_after();
          const uint64_t dv = tc::desc_add(dv0, vs * kP1Tile);
          const uint32_t aP = tl + 256 + b * kP1Keys;
#pragma unroll
          for (int ks = 0; ks < kP1Keys / 16; ++ks) {
            // keys 16 ks ..: half h = ks / 4 accumulates into O_h; P hi at
            // column 16 ks of the buffer, lo at 16 ks + 8
            const int hh = ks >> 2, kin = ks & 3;
            const uint32_t ac = aP + ks * 16;
            const uint64_t bd = tc::desc_add(dv, ks * 2048);
            tc::mma_ts(tl + hh * 128, ac, bd, kIdPV, (t > 0 || kin > 0) ? 1u : 0u);
            tc::mma_ts(tl + hh * 128, ac + 8, bd, kIdPV, 1u);
          }
          tc::commit(&bar.vempty[vs]);
        }
      }
    }
  } else if (warp >= kP1VnWarp0) {
    // |v|^2 of every tile's keys for pass 2 (with two row tiles each CTA
    // takes half of them), a key per thread (two with one row tile)
    if (kWithV) {
      const int vt = tid - kP1VnWarp0 * 32;   // 0 .. 63
      const int kpc = kP1Keys / nrt;
#pragma unroll 1
      for (int t = 0; t < ntiles; ++t) {
        const int vs = t % kP1VSt;
        (void)mbar_wait_bounded(&bar.vfull[vs], (t / kP1VSt) & 1, A.ws.status);
        const unsigned char* vst = svr + vs * kP1Tile;
#pragma unroll 1
        for (int key = rt * kpc + vt; key < (rt + 1) * kpc; key += 64) {
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
          for (int c = 0; c < 16; ++c) {
            const uint4 x = *reinterpret_cast<const uint4*>(vst + sw_off<kP1Keys>(key, c * 8));
            const __nv_bfloat162* pr = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float2 f = __bfloat1622float2(pr[u]);
              acc[(2 * u) & 3] = fmaf(f.x, f.x, acc[(2 * u) & 3]);
              acc[(2 * u + 1) & 3] = fmaf(f.y, f.y, acc[(2 * u + 1) & 3]);
            }
          }
          const int j = j_begin + t * kP1Keys + key;
          if (j < j_end) A.ws.d3_vn[lo + j] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive1(&bar.vempty[vs]);
      }
    }
  } else {
    // row warps: warps w and w + 4 share rows 32 (w % 4) .. + 31 (their
    // tensor-memory lanes); warp w / 4 = h takes keys 64 h .. 64 h + 63 of
    // every tile with its own running max and sum and its own output
    // accumulator O_h (columns 128 h ..): the two key halves are two
    // sub-chunks, merged at the end
    const int qd = warp & 3, h = warp >> 2;
    const int rr = qd * 32 + lane, r = rt * kRowTile + rr;
    const bool row_ok = r < A.rows;
    const int qp = row_ok ? A.qpos[r % A.w] : -1;
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    const int nkeys = j_end - j_begin;
    stage_rows(sq, 0, A, l, rt, tid, 256);
    cp_commit();
    cp_wait<0>();
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) mbar_arrive1(&bar.qfull);
    // pass 2 adds both row tiles' sums into the output: zero it first
    if (nrt > 1 && rt == 0)
      for (int j = j_begin + tid; j < j_end; j += 256) A.col_out[lo + j] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    // the position of the last key of this half of tile t, read from the
    // table a tile ahead (INT_MAX when the half runs past the chunk): a row
    // at or after it sees the whole half, and needs no staged positions
    auto half_last = [&](int t) {
      const int k0 = t * kP1Keys + h * 64;
      return (t < ntiles && k0 + 64 <= nkeys) ? A.ls.pos[lo + j_begin + k0 + 63] : 0x7FFFFFFF;
    };
    int last_next = half_last(0);
#pragma unroll 1
    for (int t = 0; t < ntiles; ++t) {
      const int b = t % kP1Bufs, ks = t % kP1KSt;
      const int last = last_next;
      last_next = half_last(t + 1);
      (void)mbar_wait_bounded(&bar.x_full[b], (t / kP1Bufs) & 1, A.ws.status);
      tc::fence_after();
      const uint32_t aS = tl + lane_off + 256 + b * kP1Keys + h * 64;
      const bool full = __all_sync(0xffffffffu, row_ok && last <= qp);   // no key of the half masked for the warp
      int vis = 64;
      if (!full) {
        // the half's keys the row sees: a prefix (positions ascend), found
        // by a binary search of the staged positions
        (void)mbar_wait_bounded(&bar.kfull[ks], (t / kP1KSt) & 1, A.ws.status);
        const int* tpos = sh_pos + ks * kP1Keys + h * 64;
        const int k0 = t * kP1Keys + h * 64;   // first key of the half within the chunk
        vis = 0;
        if (row_ok) {
          const int lim = max(0, min(64, nkeys - k0));
          if (lim > 0 && tpos[lim - 1] <= qp) {
            vis = lim;
          } else {
            int lo_ = 0, hi_ = lim;
            while (lo_ < hi_) {
              const int mid = (lo_ + hi_) >> 1;
              if (tpos[mid] <= qp) lo_ = mid + 1; else hi_ = mid;
            }
            vis = lo_;
          }
        }
      }
      // the stage is free once S(t) is done (x_full) and the rows are past
      // its positions
      __syncwarp();
      if (lane == 0) mbar_arrive1(&bar.kempty[ks]);
      // The row loops stay compact (16 keys at a time, S read twice: max,
      // then P): the kernel's warp roles share the instruction cache, and
      // fully unrolled loops stalled them on instruction fetch.  Without P V
      // a half whose 64 keys the whole warp sees (every tile but the last
      // few) is read once, into registers, and summed from there.
      const bool regs = !kWithV && full;
      uint32_t s0[16], s1[16], s2[16], s3[16];
      float tmax;
      if (regs) {
        tc::ld16(aS, s0);
        tc::ld16(aS + 16, s1);
        tc::ld16(aS + 32, s2);
        tc::ld16(aS + 48, s3);
        tc::wait_ld();
        tc::hold16(s0);
        tc::hold16(s1);
        tc::hold16(s2);
        tc::hold16(s3);
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int k = 0; k < 16; k += 2) {
          mq[0] = fmaxf(mq[0], fmaxf(__uint_as_float(s0[k]), __uint_as_float(s0[k + 1])));
          mq[1] = fmaxf(mq[1], fmaxf(__uint_as_float(s1[k]), __uint_as_float(s1[k + 1])));
          mq[2] = fmaxf(mq[2], fmaxf(__uint_as_float(s2[k]), __uint_as_float(s2[k + 1])));
          mq[3] = fmaxf(mq[3], fmaxf(__uint_as_float(s3[k]), __uint_as_float(s3[k + 1])));
        }
        tmax = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      } else if (full) {
        // every key visible: the four 16-column loads in flight at once
        tc::ld16(aS, s0);
        tc::ld16(aS + 16, s1);
        tc::ld16(aS + 32, s2);
        tc::ld16(aS + 48, s3);
        tc::wait_ld();
        tc::hold16(s0);
        tc::hold16(s1);
        tc::hold16(s2);
        tc::hold16(s3);
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int k = 0; k < 16; k += 2) {
          mq[0] = fmaxf(mq[0], fmaxf(__uint_as_float(s0[k]), __uint_as_float(s0[k + 1])));
          mq[1] = fmaxf(mq[1], fmaxf(__uint_as_float(s1[k]), __uint_as_float(s1[k + 1])));
          mq[2] = fmaxf(mq[2], fmaxf(__uint_as_float(s2[k]), __uint_as_float(s2[k + 1])));
          mq[3] = fmaxf(mq[3], fmaxf(__uint_as_float(s3[k]), __uint_as_float(s3[k + 1])));
        }
        tmax = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      } else {
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[16];
          tc::ld16(aS + c * 16, v);
          tc::wait_ld();
          tc::hold16(v);
          const int vc = full ? 16 : vis - 16 * c;
#pragma unroll
          for (int k = 0; k < 16; ++k) mx[k & 3] = fmaxf(mx[k & 3], k < vc ? __uint_as_float(v[k]) : -INFINITY);
        }
        tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      }
      // the largest raw score (scale2 > 0 keeps the order; the scale is
      // applied once, and inside the exponent's FMA below)
      tmax *= A.scale2;
      float factor = 1.f;
      if (tmax > m_run + kTcRescale) {
        factor = (m_run == -INFINITY) ? 0.f : exp2f(m_run - tmax);
        m_run = tmax;
        l_run *= factor;
      }
      const float negm = m_run == -INFINITY ? 0.f : -m_run;
      if (!kWithV) {
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
        if (regs) {
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            ps[0] += hw_exp2(fmaf(__uint_as_float(s0[k]), A.scale2, negm));
            ps[1] += hw_exp2(fmaf(__uint_as_float(s1[k]), A.scale2, negm));
            ps[2] += hw_exp2(fmaf(__uint_as_float(s2[k]), A.scale2, negm));
            ps[3] += hw_exp2(fmaf(__uint_as_float(s3[k]), A.scale2, negm));
          }
        } else {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t v[16];
            tc::ld16(aS + c * 16, v);
            tc::wait_ld();
            tc::hold16(v);
            const int vc = vis - 16 * c;
#pragma unroll
            for (int k = 0; k < 16; ++k)
              ps[k & 3] += hw_exp2(k < vc ? fmaf(__uint_as_float(v[k]), A.scale2, negm) : -INFINITY);
          }
        }
        l_run += (ps[0] + ps[1]) + (ps[2] + ps[3]);
        // S is read: release the buffer
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive1(&bar.x_free[b]);
        continue;
      }
      // p = 2^(s scale2 - m); a key the row does not see gives 0, and so does
      // every key while the row has seen none (m = -inf, offset taken as 0).
      // P of the 16 keys of chunk c goes over their own (already read) S
      // columns: hi in the first 8, lo in the next 8.
      float2 psum = make_float2(0.f, 0.f);
      auto p_store = [&](int c, const uint32_t (&v)[16], int vc, auto masked) {
        uint32_t hi[8], lo2[8];
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2) {
          float2 xx = f2_fma(make_float2(__uint_as_float(v[2 * k2]), __uint_as_float(v[2 * k2 + 1])),
                             make_float2(A.scale2, A.scale2), make_float2(negm, negm));
          if (decltype(masked)::value) {
            xx.x = 2 * k2 < vc ? xx.x : -INFINITY;
            xx.y = 2 * k2 + 1 < vc ? xx.y : -INFINITY;
          }
          const float2 pp = make_float2(hw_exp2(xx.x), hw_exp2(xx.y));
          psum = f2_add(psum, pp);
          // the split into bf16 hi + lo by integer and add instructions
          // only (the conversion instructions run at a fraction of the
          // rate): hi is p truncated to bf16 (its upper 16 bits), lo = p - hi
          // exactly in fp32, rounded to the nearest bf16 (ties away from
          // zero) by adding half an ulp to its bits; hi + lo is p to 2^-16
          // relative (p finite and >= 0)
          const uint32_t b0 = __float_as_uint(pp.x), b1 = __float_as_uint(pp.y);
          hi[k2] = __byte_perm(b0, b1, 0x7632);
          const float2 rem =
              f2_sub(pp, make_float2(__uint_as_float(b0 & 0xFFFF0000u), __uint_as_float(b1 & 0xFFFF0000u)));
          lo2[k2] = __byte_perm(__float_as_uint(rem.x) + 0x8000u, __float_as_uint(rem.y) + 0x8000u, 0x7632);
        }
        tc::st8(aS + c * 16, hi);
        tc::st8(aS + c * 16 + 8, lo2);
      };
      if (full) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[16];
          tc::ld16(aS + c * 16, v);
          tc::wait_ld();
          tc::hold16(v);
          p_store(c, v, 16, std::false_type{});
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[16];
          tc::ld16(aS + c * 16, v);
          tc::wait_ld();
          tc::hold16(v);
          p_store(c, v, vis - 16 * c, std::true_type{});
        }
      }
      // O_h is rescaled after P(t) is written, so that P V(t - 1), which
      // must be complete first, has run meanwhile; P V(t) is issued only
      // once the rows are past this point (x_free)
      if (t >= 1 && __any_sync(0xffffffffu, factor != 1.f)) {
        const int tp = t - 1, vp = tp % kP1VSt;
        (void)mbar_wait_bounded(&bar.vempty[vp], (tp / kP1VSt) & 1, A.ws.status);
        tc::fence_after();
        const uint32_t aO = tl + lane_off + h * 128;
#pragma unroll 1
        for (int q = 0; q < 2; ++q) {
          uint32_t o0[16], o1[16], o2[16], o3[16];
          tc::ld16(aO + q * 64, o0);
          tc::ld16(aO + q * 64 + 16, o1);
          tc::ld16(aO + q * 64 + 32, o2);
          tc::ld16(aO + q * 64 + 48, o3);
          tc::wait_ld();
          tc::hold16(o0);
          tc::hold16(o1);
          tc::hold16(o2);
          tc::hold16(o3);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            o0[k] = __float_as_uint(__uint_as_float(o0[k]) * factor);
            o1[k] = __float_as_uint(__uint_as_float(o1[k]) * factor);
            o2[k] = __float_as_uint(__uint_as_float(o2[k]) * factor);
            o3[k] = __float_as_uint(__uint_as_float(o3[k]) * factor);
          }
          tc::st16(aO + q * 64, o0);
          tc::st16(aO + q * 64 + 16, o1);
          tc::st16(aO + q * 64 + 32, o2);
          tc::st16(aO + q * 64 + 48, o3);
        }
      }
      l_run += psum.x + psum.y;
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive1(&bar.x_free[b]);
    }
    // merge the two key halves' (max, sum, O) per row, like two chunks;
    // this thread writes output columns [64 h, 64 h + 64)
    sh_ml[h][rr][0] = m_run;
    sh_ml[h][rr][1] = l_run;
    named_sync(1, 256);
    const float m0 = sh_ml[0][rr][0], l0 = sh_ml[0][rr][1], m1 = sh_ml[1][rr][0], l1 = sh_ml[1][rr][1];
    const float M = fmaxf(m0, m1);
    const float s0 = m0 == -INFINITY ? 0.f : exp2f(m0 - M);
    const float s1 = m1 == -INFINITY ? 0.f : exp2f(m1 - M);
    const size_t stride = kD + 2;
    float* part = A.ws.d3_part + (static_cast<size_t>(l) * A.chunks + chunk) * static_cast<size_t>(A.rows_cap) * stride +
                  static_cast<size_t>(row_ok ? r : 0) * stride;
    if (kWithV) {
      // every P V is complete once the last one is (its commit covers all earlier MMAs)
      (void)mbar_wait_bounded(&bar.vempty[(ntiles - 1) % kP1VSt], ((ntiles - 1) / kP1VSt) & 1, A.ws.status);
      tc::fence_after();
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int c0 = h * 64 + q4 * 16;
        uint32_t va[16], vb[16];
        tc::ld16(tl + lane_off + c0, va);
        tc::ld16(tl + lane_off + 128 + c0, vb);
        tc::wait_ld();
        if (row_ok) {
#pragma unroll
          for (int k = 0; k < 16; k += 2) {
            float2 o;
            o.x = s0 * __uint_as_float(va[k]) + s1 * __uint_as_float(vb[k]);
            o.y = s0 * __uint_as_float(va[k + 1]) + s1 * __uint_as_float(vb[k + 1]);
            *reinterpret_cast<float2*>(part + c0 + k) = o;
          }
        }
      }
    }
    if (row_ok && h == 0) {
      part[kD] = M;
      part[kD + 1] = s0 * l0 + s1 * l1;
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == kP1Issuer) tc::dealloc(tl, 512);
}

// p / (1 - p) * sqrt(d2) for a (row, key) pair with p > 1/2, x = log2 p, d2
// = ||a - v||^2 taken directly (the expansion would cancel there); 1 - p
// from expm1.
__device__ __forceinline__ float direct_term(float x, float d2) {
  const float p = exp2f(x);
  const float om = -expm1f(x * kLn2);
  if (!(om > 0.f)) return INFINITY;
  return p / om * sqrtf(d2);
}

constexpr float kSmallLog2 = -7.f;   // p < 2^-7: p / (1 - p) = p + p^2 + p^3 within 2^-21
constexpr float kR2Floor = 1e-30f;   // r2 floor: sqrt(r2) = r2 rsqrt(r2) stays finite (1e-15 for r2 = 0)

// Pass-2 state past the big operands, in dynamic shared memory (the operands
// fill all but a few KB of it).
struct P2Small {
  uint64_t full[kP2St], empty[kP2St], x_full[2], x_free[2], qfull;
  uint32_t taddr, pad;
  float nlse2[kRowTile];   // per row of the CTA: -LSE (base 2; -inf past the rows) and |a|^2
  float an[kRowTile];
};
constexpr int p2_smem(bool res) {
  return (res ? 3 : 1) * kQBytes + kP2St * (res ? 2 : 1) * kP2Tile + static_cast<int>(sizeof(P2Small)) + 1008;
}

// pass 2.  Barriers: full / empty the K/V stages (empty: the tile's MMAs are
// done with it); x_full[b] S^T and G^T of tile t done; x_free[b] the 8 row
// warps have read them into registers; qfull the resident operands staged.
template <int kMode>
__global__ void __launch_bounds__(kP2Threads, 1) d3_p2_kernel(D3Args A, const __grid_constant__ D3Maps mp) {
  constexpr bool kRes = kMode == kResidual;
  constexpr int kStageB = (kRes ? 2 : 1) * kP2Tile;
  constexpr uint32_t kCols = kRes ? 512 : 256;
  constexpr int kBufCols = kRes ? 256 : 128;
  extern __shared__ unsigned char d3_dsm[];
  const int nrt = (A.rows + kRowTile - 1) / kRowTile;
  const int rt = blockIdx.x % nrt, chunk = blockIdx.x / nrt, l = blockIdx.y;
  const int n = min(max(A.ls.count[l], 0), A.dm.cap);
  const int j_begin = chunk * A.chunk_keys;
  if (j_begin >= n) return;
  const int j_end = min(n, j_begin + A.chunk_keys);
  const int ntiles = (j_end - j_begin + kP2Keys - 1) / kP2Keys;
  unsigned char* sq = align1024(d3_dsm);
  unsigned char* sah = sq + kQBytes;
  unsigned char* sal = sah + kQBytes;
  unsigned char* ring = sq + (kRes ? 3 : 1) * kQBytes;
  P2Small& sm = *reinterpret_cast<P2Small*>(ring + kP2St * kStageB);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == kP2Issuer) tc::alloc(&sm.taddr, kCols);
  if (tid == 0) {
    for (int s = 0; s < kP2St; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.x_full[b], 1);
      mbar_init(&sm.x_free[b], kP2RowWarps);
    }
    mbar_init(&sm.qfull, kP2RowWarps);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tl = sm.taddr;
  const size_t lo = static_cast<size_t>(l) * A.dm.cap;

  if (warp == kP2Producer) {
    d3_produce<kP2Keys, kP2St, true, kRes, false, 0>(A, mp, l, j_begin, j_end, ntiles, ring, sm.full, sm.empty,
                                                     nullptr, nullptr, nullptr);
  } else if (warp == kP2Issuer) {
    if (lane == 0) {
      // descriptors built once; each MMA advances one by a constant
      const uint64_t dq = tc::desc_sw128(smem_u32(sq), 16, 1024);
      const uint64_t dah = tc::desc_sw128(smem_u32(sah), 16, 1024);
      const uint64_t dal = tc::desc_sw128(smem_u32(sal), 16, 1024);
      const uint64_t dr0 = tc::desc_sw128(smem_u32(ring), 16, 1024);
      (void)mbar_wait_bounded(&sm.qfull, 0, A.ws.status);
#pragma unroll 1
      for (int t = 0; t < ntiles; ++t) {
        const int st = t & 1;
        (void)mbar_wait_bounded(&sm.full[st], (t >> 1) & 1, A.ws.status);
        if (t >= 2) (void)mbar_wait_bounded(&sm.x_free[st], ((t >> 1) - 1) & 1, A.ws.status);
        tc::fence_after();
        const uint64_t dk = tc::desc_add(dr0, st * kStageB), dv = tc::desc_add(dk, kP2Tile);
        const uint32_t dS = tl + st * kBufCols, dG = dS + 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int off = (kk >> 2) * (kP2Keys * 128) + (kk & 3) * 32;   // d half, 16-element step
          tc::mma_ss(dS, tc::desc_add(dk, off), tc::desc_add(dq, off), kId128, kk > 0 ? 1u : 0u);
        }
        if (kRes) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const int off = (kk >> 2) * (kP2Keys * 128) + (kk & 3) * 32;
            tc::mma_ss(dG, tc::desc_add(dv, off), tc::desc_add(dah, off), kId128, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const int off = (kk >> 2) * (kP2Keys * 128) + (kk & 3) * 32;
            tc::mma_ss(dG, tc::desc_add(dv, off), tc::desc_add(dal, off), kId128, 1u);
          }
        }
        tc::commit(&sm.x_full[st]);
        tc::commit(&sm.empty[st]);
      }
    }
  } else {
    // row warps: warp w owns keys 32 (w % 4) .. + 31 of every tile (its
    // tensor-memory lanes) and the CTA's rows 32 (w / 4) .. + 31 (columns)
    constexpr int kRowThreads = kP2RowWarps * 32;
    const int qd = warp & 3, c = warp >> 2;
    const int kk = qd * 32 + lane;
    const int r0 = rt * kRowTile + c * 32;   // first row of this warp
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    const int b = l / A.dm.Hkv, kh = l % A.dm.Hkv;
    stage_rows(sq, 0, A, l, rt, tid, kRowThreads);
    // launched as a dependent of the combine: everything above (the barriers,
    // tensor memory, Q, and the producers' K/V copies) overlaps it; a, the
    // row statistics, |v|^2 and the output are read or written past the wait
    grid_dep_wait();
    if (kRes) {
      stage_rows(sah, 1, A, l, rt, tid, kRowThreads);
      stage_rows(sal, 2, A, l, rt, tid, kRowThreads);
    }
    if (tid < kRowTile) {
      const int r = rt * kRowTile + tid;
      const size_t wrow = static_cast<size_t>(l) * A.rows_cap + r;
      // a row past the window's rows: +inf LSE, so every weight of it is 0
      sm.nlse2[tid] = r < A.rows ? -A.ws.d3_rowc[wrow * 2] : -INFINITY;
      sm.an[tid] = (kRes && r < A.rows) ? A.ws.d3_rowc[wrow * 2 + 1] : 0.f;
    }
    cp_commit();
    cp_wait<0>();
    fence_proxy_async();
    named_sync(1, kRowThreads);
    if (lane == 0) mbar_arrive1(&sm.qfull);
    // the query position of row r0 + lane, and the warp's minimum: a key at
    // or before it is seen by all of the warp's rows
    const int qp_mine = r0 + lane < A.rows ? A.qpos[(r0 + lane) % A.w] : 0x7FFFFFFF;
    const int qmin = __reduce_min_sync(0xffffffffu, qp_mine);
    const int nv = min(32, A.rows - r0);   // rows of this warp (<= 0: none)
    const int nch = nv <= 0 ? 0 : (nv + 15) >> 4;
    auto meta = [&](int t, int& p, float& v, int& sl) {
      const int j = j_begin + t * kP2Keys + kk;
      const bool ok = t < ntiles && j < j_end;
      p = ok ? A.ls.pos[lo + j] : 0x7FFFFFFF;
      v = (kRes && ok) ? A.ws.d3_vn[lo + j] : 0.f;
      sl = (kRes && ok) ? A.ls.slot[lo + j] : 0;
    };
    int pj, sj;
    float vj;
    meta(0, pj, vj, sj);
#pragma unroll 1
    for (int t = 0; t < ntiles; ++t) {
      const int st = t & 1;
      const int j = j_begin + t * kP2Keys + kk;
      const bool key_ok = j < j_end;
      int pj_n, sj_n;
      float vj_n;
      meta(t + 1, pj_n, vj_n, sj_n);   // in flight while this tile is scored
      // every (row, key) pair of the warp counted: no mask (a key past the
      // chunk has position INT_MAX)
      const int wmax = __reduce_max_sync(0xffffffffu, pj);
      const bool no_mask = kMode == kMassLater ? wmax < qmin : wmax <= qmin;
      (void)mbar_wait_bounded(&sm.x_full[st], (t >> 1) & 1, A.ws.status);
      tc::fence_after();
      const uint32_t aS = tl + lane_off + st * kBufCols + c * 32;
      float acc = 0.f;
      // 16 rows at a time: the chunk's S^T (and G^T) columns into registers
#pragma unroll 1
      for (int ch = 0; ch < nch; ++ch) {
        uint32_t v[16], g[16];
        tc::ld16(aS + ch * 16, v);
        if (kRes) tc::ld16(aS + 128 + ch * 16, g);
        tc::wait_ld();
        tc::hold16(v);
        if (kRes) tc::hold16(g);
        const float* nlse_c = sm.nlse2 + c * 32 + ch * 16;
        const float* an_c = sm.an + c * 32 + ch * 16;
        // two rows per packed instruction
        float x[16];
        float xm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int k = 0; k < 16; k += 2) {
          const float2 nl = *reinterpret_cast<const float2*>(nlse_c + k);
          float2 xx = f2_fma(make_float2(__uint_as_float(v[k]), __uint_as_float(v[k + 1])),
                             make_float2(A.scale2, A.scale2), nl);
          if (!no_mask) {
            const int qp0 = __shfl_sync(0xffffffffu, qp_mine, ch * 16 + k);
            const int qp1 = __shfl_sync(0xffffffffu, qp_mine, ch * 16 + k + 1);
            const bool vis0 = key_ok && (kMode == kMassLater ? pj < qp0 : pj <= qp0);
            const bool vis1 = key_ok && (kMode == kMassLater ? pj < qp1 : pj <= qp1);
            xx.x = vis0 ? xx.x : -INFINITY;
            xx.y = vis1 ? xx.y : -INFINITY;
          }
          x[k] = xx.x;
          x[k + 1] = xx.y;
          xm[k & 3] = fmaxf(xm[k & 3], xx.x);
          xm[(k + 1) & 3] = fmaxf(xm[(k + 1) & 3], xx.y);
        }
        if (!kRes) {
          float2 a2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int k = 0; k < 16; k += 2) a2 = f2_add(a2, make_float2(hw_exp2(x[k]), hw_exp2(x[k + 1])));
          acc += a2.x + a2.y;
          continue;
        }
        const float xmax = fmaxf(fmaxf(xm[0], xm[1]), fmaxf(xm[2], xm[3]));
        if (!__any_sync(0xffffffffu, xmax >= kSmallLog2)) {
          // every weight of the warp's pairs is small: no reciprocal, and
          // sqrt(r2) = r2 rsqrt(r2) (a pair not counted has p = 0)
          float2 a2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int k = 0; k < 16; k += 2) {
            const float2 n2 = *reinterpret_cast<const float2*>(an_c + k);
            const float2 p = make_float2(hw_exp2(x[k]), hw_exp2(x[k + 1]));
            float2 r2 = f2_fma(make_float2(__uint_as_float(g[k]), __uint_as_float(g[k + 1])), make_float2(-2.f, -2.f),
                               f2_add(n2, make_float2(vj, vj)));
            r2.x = fmaxf(kR2Floor, r2.x);
            r2.y = fmaxf(kR2Floor, r2.y);
            const float2 q = f2_fma(f2_fma(p, p, p), p, p);   // p + p^2 + p^3
            a2 = f2_fma(f2_mul(q, r2), make_float2(hw_rsqrt(r2.x), hw_rsqrt(r2.y)), a2);
          }
          acc += a2.x + a2.y;
        } else {
          unsigned big = 0;
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const float4 N4 = *reinterpret_cast<const float4*>(an_c + 4 * k4);
            const float Ns[4] = {N4.x, N4.y, N4.z, N4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int k = 4 * k4 + u;
              const float p = hw_exp2(x[k]);
              const float r2 = fmaxf(0.f, fmaf(-2.f, __uint_as_float(g[k]), Ns[u] + vj));
              const float tm = p * hw_rcp(1.f - p) * hw_sqrt(r2);
              if (p > 0.5f) big |= 1u << k;
              acc += (p > 0.f && p <= 0.5f) ? tm : 0.f;
            }
          }
          // pairs with p > 1/2 (at most one key per row has one): the direct
          // distance, each pair's 128 elements shared by the warp's lanes, so
          // its loads (the fp32 a row, just written by the combine, and the
          // key's V row, just copied for the tile) take one round trip
          unsigned pend = __ballot_sync(0xffffffffu, big != 0);
          while (pend) {
            const int src = __ffs(pend) - 1;
            const int k = __ffs(__shfl_sync(0xffffffffu, big, src)) - 1;
            float xk = 0.f;
#pragma unroll
            for (int k2 = 0; k2 < 16; ++k2)
              if (k2 == k) xk = x[k2];
            xk = __shfl_sync(0xffffffffu, xk, src);
            int slot = __shfl_sync(0xffffffffu, sj, src);
            if (slot < 0 || slot >= A.dm.P * kBlock) {
              if (lane == 0) set_status(A.ws.status, ST_BAD_INDEX);
              slot = 0;
            }
            const int r = r0 + ch * 16 + k;
            const float4 av = *reinterpret_cast<const float4*>(
                A.a_out + ((static_cast<size_t>(b) * A.dm.Hq + kh * A.dm.g + r / A.w) * A.w + r % A.w) * kD + 4 * lane);
            const uint2 vr = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(A.ls.v_pool) +
                                                             static_cast<size_t>(slot) * kD + 4 * lane);
            const float2 v01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vr.x));
            const float2 v23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vr.y));
            float d, d2 = 0.f;
            d = av.x - v01.x; d2 = fmaf(d, d, d2);
            d = av.y - v01.y; d2 = fmaf(d, d, d2);
            d = av.z - v23.x; d2 = fmaf(d, d, d2);
            d = av.w - v23.y; d2 = fmaf(d, d, d2);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) d2 += __shfl_xor_sync(0xffffffffu, d2, o);
            if (lane == src) {
              acc += direct_term(xk, d2);
              big &= big - 1;
            }
            pend = __ballot_sync(0xffffffffu, big != 0);
          }
        }
      }
      // the four warps sharing these keys: warps c = 1..3 leave their sums in
      // the first (already read) S^T column of their rows, warp c = 0 adds
      // them to its own in order c = 0..3; a barrier per tile parity, so a
      // warp a tile ahead cannot arrive on the one still being waited on
      const int hb = 2 + qd + 4 * (t & 1);
      if (c != 0) {
        tc::st1(aS, __float_as_uint(acc));
        tc::wait_st();
        tc::fence_before();
        named_arrive(hb, 128);
        __syncwarp();
        if (lane == 0) mbar_arrive1(&sm.x_free[st]);
      } else {
        named_sync(hb, 128);
        tc::fence_after();
        const uint32_t a1 = tc::ld1(aS + 32), a2 = tc::ld1(aS + 64), a3 = tc::ld1(aS + 96);
        tc::wait_ld();
        const float tot = ((acc + __uint_as_float(a1)) + __uint_as_float(a2)) + __uint_as_float(a3);
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive1(&sm.x_free[st]);
        if (key_ok) {
          if (nrt == 1)
            A.col_out[lo + j] = tot;
          else
            atomicAdd(A.col_out + lo + j, tot);
        }
      }
      pj = pj_n;
      vj = vj_n;
      sj = sj_n;
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == kP2Issuer) tc::dealloc(tl, kCols);
}

}  // namespace

int d3_rows_max(const Dims& dm) { return dm.g * dm.max_window; }

cudaError_t prepare_dropkv() {
  struct {
    const void* f;
    int smem;
  } fns[] = {{reinterpret_cast<const void*>(d3_p1_kernel<true>), kP1Smem},
             {reinterpret_cast<const void*>(d3_p1_kernel<false>), kP1Smem},
             {reinterpret_cast<const void*>(d3_p2_kernel<kResidual>), p2_smem(true)},
             {reinterpret_cast<const void*>(d3_p2_kernel<kMassCausal>), p2_smem(false)},
             {reinterpret_cast<const void*>(d3_p2_kernel<kMassLater>), p2_smem(false)}};
  for (const auto& x : fns) {
    const cudaError_t e = cudaFuncSetAttribute(x.f, cudaFuncAttributeMaxDynamicSharedMemorySize, x.smem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}
// Keys per CTA: each lane's keys split over floor(SMs / (lanes x row tiles))
// CTAs (one wave when the lanes are few), in whole 128-key tiles, at least
// kChunkMin.  sm_count 0 gives the most chunks any device can use
// (workspace sizing).
static int d3_chunk_keys(const Dims& dm, int sm_count, int row_tiles) {
  const int per_lane = sm_count > 0 ? max(1, sm_count / max(1, dm.lanes * row_tiles)) : 1 << 30;
  const int k = (dm.cap + per_lane - 1) / per_lane;
  return max(kChunkMin, (k + kTileKeys - 1) / kTileKeys * kTileKeys);
}
int d3_chunks(const Dims& dm, int sm_count) {
  const int ck = d3_chunk_keys(dm, sm_count, 1);
  return (dm.cap + ck - 1) / ck;
}

cudaError_t prepare_tensor_maps(Ctx& ctx) {
  const Dims& dm = ctx.dims;
  if (!(dm.max_window > 0 && dm.dtype == KVEVICT_BF16 && dm.d == kD)) return cudaSuccess;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess) return e;
  if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
  const auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  ctx.tmaps = new (std::nothrow) CUtensorMap[kTmapsPerLayer * static_cast<size_t>(dm.L)];
  if (!ctx.tmaps) return cudaErrorMemoryAllocation;
  // [P * 16 rows][d] bf16, rows 2 d bytes apart; boxes of 64 elements (128
  // bytes) by 1, 16 or 64 rows
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(dm.P) * kBlock};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(kD) * 2};
  const cuuint32_t box_rows[3] = {1, 16, 64};
  const cuuint32_t estride[2] = {1, 1};
  for (int layer = 0; layer < dm.L; ++layer) {
    const LayerState ls = layer_state(ctx, layer);
    for (int i = 0; i < kTmapsPerLayer; ++i) {
      const cuuint32_t box[2] = {64, box_rows[i / 2]};
      const CUresult r = encode(&ctx.tmaps[static_cast<size_t>(layer) * kTmapsPerLayer + i],
                                CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (i & 1) ? ls.v_pool : ls.k_pool, gdim, gstride,
                                box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
  }
  return cudaSuccess;
}

// The window passes of one layer.  mode (D3Mode) picks the pass-2 term;
// pool_r >= 0 max-pools the mass sums over kept neighbours (radius pool_r)
// into scores, pool_r < 0 writes the sums themselves.
static cudaError_t launch_window(const Ctx& ctx, int layer, const void* q_win, int w, const int32_t* q_pos,
                                 int mode, int pool_r, float* lse, float* a_out, float* scores, cudaStream_t stream) {
  const Dims& dm = ctx.dims;
  D3Args A;
  A.ls = layer_state(ctx, layer);
  A.ws = ctx.ws;
  A.dm = dm;
  A.q = static_cast<const __nv_bfloat16*>(q_win);
  A.qpos = q_pos;
  A.w = w;
  A.rows = dm.g * w;
  A.rows_cap = d3_rows_max(dm);
  // the tensor-core path splits the rows into 128-row tiles, one CTA each
  const bool tcp = A.rows <= kTcRows;
  const int nrt = tcp ? (A.rows + kRowTile - 1) / kRowTile : 1;
  A.chunk_keys = d3_chunk_keys(dm, ctx.sm_count, nrt);
  A.chunks = (dm.cap + A.chunk_keys - 1) / A.chunk_keys;
  A.lse_out = lse; A.a_out = a_out; A.scores = scores;
  A.col_out = pool_r >= 0 ? ctx.ws.d3_score_part : scores;
  A.scale2 = 1.4426950408889634f / sqrtf(static_cast<float>(dm.d));
  if (A.rows > A.rows_cap || A.rows > kMaxRowGroups * kRowsPerCta || dm.d != kD || dm.dtype != KVEVICT_BF16)
    return cudaErrorInvalidValue;
  const bool res = mode == kResidual;
  if (tcp) {
    const dim3 grid(nrt * A.chunks, dm.lanes);
    if (!ctx.tmaps) return cudaErrorInvalidValue;
    D3Maps mp;
    for (int i = 0; i < kTmapsPerLayer; ++i) mp.m[i] = ctx.tmaps[static_cast<size_t>(layer) * kTmapsPerLayer + i];
    const dim3 cgrid((A.rows + 7) / 8, dm.lanes);
    // the combine and pass 2 are dependent launches (each orders itself
    // with griddepcontrol.wait before it reads its predecessor's results)
    cudaError_t e;
    if (res) {
      d3_p1_kernel<true><<<grid, kP1Threads, kP1Smem, stream>>>(A, mp);
      e = launch_k(d3_combine_kernel<true>, cgrid, dim3(256), 0, stream, true, A);
      if (e == cudaSuccess) e = launch_k(d3_p2_kernel<kResidual>, grid, dim3(kP2Threads), p2_smem(true), stream, true, A, mp);
    } else {
      d3_p1_kernel<false><<<grid, kP1Threads, kP1Smem, stream>>>(A, mp);
      e = launch_k(d3_combine_kernel<false>, cgrid, dim3(256), 0, stream, true, A);
      if (e == cudaSuccess)
        e = mode == kMassLater
                ? launch_k(d3_p2_kernel<kMassLater>, grid, dim3(kP2Threads), p2_smem(false), stream, true, A, mp)
                : launch_k(d3_p2_kernel<kMassCausal>, grid, dim3(kP2Threads), p2_smem(false), stream, true, A, mp);
    }
    if (e != cudaSuccess) return e;
  } else {
    const int groups = (A.rows + kRowsPerCta - 1) / kRowsPerCta;
    dim3 grid(A.chunks, dm.lanes, groups);
    d3_pass1_kernel<<<grid, kWarps * 32, 0, stream>>>(A);
    if (res) {
      d3_combine_kernel<true><<<dim3((A.rows + 7) / 8, dm.lanes), 256, 0, stream>>>(A);
      d3_pass2_kernel<kResidual><<<grid, kWarps * 32, 0, stream>>>(A);
    } else {
      d3_combine_kernel<false><<<dim3((A.rows + 7) / 8, dm.lanes), 256, 0, stream>>>(A);
      if (mode == kMassLater)
        d3_pass2_kernel<kMassLater><<<grid, kWarps * 32, 0, stream>>>(A);
      else
        d3_pass2_kernel<kMassCausal><<<grid, kWarps * 32, 0, stream>>>(A);
    }
    dim3 fgrid((dm.cap + 255) / 256 < 64 ? (dm.cap + 255) / 256 : 64, dm.lanes);
    d3_finalize_kernel<<<fgrid, 256, 0, stream>>>(A, groups);
  }
  if (pool_r >= 0) {
    const dim3 pgrid((dm.cap + kPoolTile - 1) / kPoolTile, dm.lanes);
    const size_t sm = static_cast<size_t>(kPoolTile + 2 * pool_r) * sizeof(float);
    d3_pool_kernel<<<pgrid, 256, sm, stream>>>(A.col_out, scores, A.ls.count, dm.cap, pool_r);
  }
  return cudaGetLastError();
}

cudaError_t launch_score(const Ctx& ctx, int layer, const void* q_win, int w, const int32_t* q_pos,
                         float* lse, float* a_out, float* scores, cudaStream_t stream) {
  return launch_window(ctx, layer, q_win, w, q_pos, kResidual, -1, lse, a_out, scores, stream);
}

cudaError_t launch_score_mass(const Ctx& ctx, int layer, const void* q_win, int w, const int32_t* q_pos,
                              bool later, int pool_r, float* lse, float* scores, cudaStream_t stream) {
  return launch_window(ctx, layer, q_win, w, q_pos, later ? kMassLater : kMassCausal, pool_r, lse, nullptr,
                       scores, stream);
}

}  // namespace kve
