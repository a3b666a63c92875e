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
  int w, rows, rows_cap, chunks, chunk_keys;   // chunk_keys: keys per CTA, a multiple of 64
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
// tcgen05 path: all window rows of a lane (up to 256 = two 128-row tiles) per
// CTA, one thread per row, accumulators in tensor memory.
//
// pass 1, per 64-key tile:  S = Q K^T (Q and K in shared memory, 128-byte
//   swizzle); each thread masks and exponentiates its row (lazy rescale of
//   the running max), writes P as bf16 hi + lo over S in tensor memory, and
//   O += P V takes P from tensor memory and V (MN-major) from shared memory.
//   Tensor-memory columns: O of tile 0 / 1 at 0 / 128; S-P double buffer at
//   256 + 128 * (t & 1) (+ 64 for row tile 1).  The row warps also take
//   |v|^2 of every key for pass 2.
// pass 2, per 64-key tile:  S = Q K^T and G = a V^T (a as bf16 hi + lo held
//   in tensor memory); each thread copies its row of S and G to registers,
//   which frees the buffer for the next tile's MMAs, and turns them into
//   residual terms (32 keys at a time through one copy of the code); each warp sums its 32 rows per key
//   by a butterfly, and the producer adds the 8 warp sums in a fixed order
//   when the tile's stage is recycled and writes the final scores.  While
//   every weight of a warp's rows is below 2^-7, p / (1 - p) is the series
//   p (1 + p (1 + p)) instead of a reciprocal.
//   Tensor-memory columns: a hi 0 / 64, a lo 128 / 192, S 256 / 320,
//   G 384 / 448 (row tile 0 / 1).  (MMAs of 32 keys, which would let two
//   buffers fit, re-read Q from shared memory for half the keys and ran
//   at a fraction of the rate.)
// K/V rows arrive by TMA gathers (four pool rows per copy, 128-byte swizzle
// applied by the copy engine) into a four-stage ring.
// ---------------------------------------------------------------------------
constexpr int kTcKeys = 64;
constexpr int kTcStages = 4;
constexpr int kTcRows = 256;
constexpr int kTcHalf = kTcKeys * 128;                 // one d half of a K or V tile (8 KB)
constexpr int kTcKV = 4 * kTcHalf;                     // K (2 halves) then V (2 halves)
constexpr int kTcQ = 2 * 2 * 128 * 128;                // [row tile][d half][128 rows][128 B]
constexpr int kTcSmem = kTcQ + kTcStages * kTcKV + 1024;
constexpr uint32_t kTcCols = 512;
constexpr float kTcRescale = 8.f;
constexpr uint32_t kIdS = tc::idesc_bf16(128, kTcKeys, 0);
constexpr uint32_t kIdPV = tc::idesc_bf16(128, kD, 1);
static_assert(kChunkMin % kTcKeys == 0, "chunks hold whole tiles");

// Hardware approximations (PTX ex2/rcp/sqrt .approx.ftz, relative error
// about 2^-22; results below 2^-126 flush to zero).
__device__ __forceinline__ float hw_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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
// byte offset of bf16 element e of key row k in a swizzled K or V tile
__device__ __forceinline__ int sw_off(int k, int e) {
  return (e >> 6) * kTcHalf + k * 128 + ((((e & 63) >> 3) ^ (k & 7)) << 4) + (e & 7) * 2;
}

// S[row tile mm] = Q K^T for stage st into tensor-memory column dS (thread 0)
__device__ __forceinline__ void tc_issue_s(uint32_t dS, const unsigned char* sq, const unsigned char* kst, int mm) {
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int half = ks >> 2, kin = ks & 3;
    const uint64_t ad = tc::desc_sw128(smem_u32(sq + mm * 32768 + half * 16384) + kin * 32, 16, 1024);
    const uint64_t bd = tc::desc_sw128(smem_u32(kst + half * kTcHalf) + kin * 32, 16, 1024);
    tc::mma_ss(dS, ad, bd, kIdS, ks > 0 ? 1u : 0u);
  }
}

// Warp roles of the tcgen05 passes: warps 0-7 own one window row per thread,
// warp 8 produces (Q, then K/V tiles into the stage ring by TMA row gathers),
// warp 9 lane 0 issues the MMAs.  Hand-offs are mbarriers only.
constexpr int kWsRowThreads = 256;
constexpr int kWsThreads = kWsRowThreads + 64;
constexpr int kWsProducer = 8, kWsIssuer = 9;
constexpr int kPrefetch = 4;   // tiles of key slots / positions the producer has in flight

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async16_zf(void* dst, const void* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(ok ? 16 : 0)
               : "memory");
}
// one arrival on the barrier once this thread's earlier cp.async copies land
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
struct WsBars {
  uint64_t qfull;
  uint64_t full[kTcStages], empty[kTcStages];
  uint64_t x_full[2], x_free[2], pv_done[2];
};

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

// Producer warp.  Q rows first (8 per lane, 16-byte cp.async, once); then per
// tile the K and V rows of its 64 keys by TMA, after the keys' positions
// (and in pass 2 their |v|^2), loaded one tile ahead, are stored to the
// stage and lane 0 has armed the stage's full barrier with the tile's bytes.
// A tile whose 64 slots are consecutive (the layout a prefill leaves) takes
// one 64-row copy per tensor and row half; otherwise each group of 16 keys
// in consecutive slots takes a 16-row copy, and the other keys are gathered
// four rows per copy (lanes 0-15, four keys each; a key past the chunk
// gathers a row past the pool, which reads as zeros).  A TMA instruction
// costs tens of nanoseconds to issue, so the fewer the better.
// In pass 2 it also retires each tile's column sums: once the tile's stage
// is empty (its MMAs and the 8 row warps are done with it), the 8 warps'
// partial sums are added in warp order and stored.
template <bool kPass2, bool kLoadV = true>
__device__ __forceinline__ void ws_produce(const D3Args& A, const D3Maps& mp, int l,
                                           int j_begin, int j_end, int ntiles, unsigned char* sq, unsigned char* skv,
                                           int (*pos)[kTcKeys], float (*vn)[kTcKeys],
                                           float (*col)[kWsRowThreads / 32][kTcKeys], WsBars& bar) {
  const int lane = threadIdx.x & 31;
  const int b = l / A.dm.Hkv, kh = l % A.dm.Hkv;
#pragma unroll 1
  for (int q = 0; q < 8; ++q) {
    const int r = lane * 8 + q, rr = r & 127;
    unsigned char* row = sq + (r >> 7) * 32768 + rr * 128;
    const bool ok = r < A.rows;
    const int h = ok ? r / A.w : 0, i = ok ? r % A.w : 0;
    const __nv_bfloat16* src = A.q + ((static_cast<size_t>(b) * A.dm.Hq + kh * A.dm.g + h) * A.w + i) * kD;
#pragma unroll
    for (int c = 0; c < 16; ++c)
      cp_async16_zf(row + (c >> 3) * 16384 + (((c & 7) ^ (rr & 7)) << 4), ok ? src + c * 8 : A.q, ok);
  }
  cp_async_arrive(&bar.qfull);
  const size_t lo = static_cast<size_t>(l) * A.dm.cap;
  const int rows_max = A.dm.P * kBlock;
  // The keys' slots, positions (and |v|^2) reach shared memory by 4-byte
  // cp.async kPrefetch tiles ahead, one commit group per tile, so the
  // producer does not wait a global round trip per tile before it can
  // issue the tile's copies.  Each lane copies and later reads only its own
  // two keys of a tile.
  __shared__ int pf_slot[kPrefetch][kTcKeys], pf_pos[kPrefetch][kTcKeys];
  __shared__ float pf_vn[kPrefetch][kTcKeys];
  auto prefetch = [&](int t) {
    if (t < ntiles) {
      const int b = t % kPrefetch;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int key = 2 * lane + kk, j = j_begin + t * kTcKeys + key;
        if (j < j_end) {
          cp_async4(&pf_slot[b][key], A.ls.slot + lo + j);
          cp_async4(&pf_pos[b][key], A.ls.pos + lo + j);
          if (kPass2 && kLoadV) cp_async4(&pf_vn[b][key], A.ws.d3_vn + lo + j);
        }
      }
    }
    cp_commit();
  };
  auto fetch = [&](int t, int key, int& sl, int& ps, float& v) {
    const int j = j_begin + t * kTcKeys + key;
    sl = rows_max;
    ps = 0x7FFFFFFF;
    v = 0.f;
    if (t >= ntiles || j >= j_end) return;
    const int b = t % kPrefetch;
    int s = pf_slot[b][key];
    if (s < 0 || s >= rows_max) { set_status(A.ws.status, ST_BAD_INDEX); s = 0; }
    sl = s;
    ps = pf_pos[b][key];
    if (kPass2 && kLoadV) v = pf_vn[b][key];
  };
  auto retire = [&](int u) {
    const int su = u % kTcStages;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const int key = 2 * lane + kk;
      float tot = 0.f;
#pragma unroll
      for (int w8 = 0; w8 < kWsRowThreads / 32; ++w8) tot += col[su][w8][key];
      const int j = j_begin + u * kTcKeys + key;
      if (j < j_end) A.col_out[lo + j] = tot;
    }
  };
  int s0, s1, p0, p1;
  float v0, v1;
#pragma unroll
  for (int u = 0; u < kPrefetch; ++u) prefetch(u);
#pragma unroll 1
  for (int t = 0; t < ntiles; ++t) {
    const int st = t % kTcStages;
    cp_wait<kPrefetch - 1>();   // tile t's group has landed
    fetch(t, 2 * lane, s0, p0, v0);
    fetch(t, 2 * lane + 1, s1, p1, v1);
    if (t >= kTcStages) {
      (void)mbar_wait_bounded(&bar.empty[st], ((t / kTcStages) - 1) & 1, A.ws.status);
      if (kPass2) retire(t - kTcStages);
    }
    pos[st][2 * lane] = p0;
    pos[st][2 * lane + 1] = p1;
    if (kPass2 && kLoadV) {
      vn[st][2 * lane] = v0;
      vn[st][2 * lane + 1] = v1;
    }
    // lane g < 16 takes keys 4g .. 4g + 3, held by lanes 2g and 2g + 1
    const int g0 = __shfl_sync(0xffffffffu, s0, (2 * lane) & 31);
    const int g1 = __shfl_sync(0xffffffffu, s1, (2 * lane) & 31);
    const int g2 = __shfl_sync(0xffffffffu, s0, (2 * lane + 1) & 31);
    const int g3 = __shfl_sync(0xffffffffu, s1, (2 * lane + 1) & 31);
    // consecutive slots: the whole tile (lane 0's key 0 first), and each
    // 16-key group q (keys 16q.., held by lanes 8q .. 8q + 7)
    const int tbase = __shfl_sync(0xffffffffu, s0, 0);
    const bool tile_run = __all_sync(0xffffffffu, s0 == tbase + 2 * lane && s1 == tbase + 2 * lane + 1) &&
                          tbase + kTcKeys <= rows_max;
    const int qbase = __shfl_sync(0xffffffffu, s0, lane & ~7);
    const unsigned qrun = __ballot_sync(0xffffffffu, s0 == qbase + 2 * (lane & 7) && s1 == qbase + 2 * (lane & 7) + 1);
    const int grp = (lane >> 2) & 3;                                  // the group of lane g < 16
    const int gbase = __shfl_sync(0xffffffffu, qbase, 8 * grp);
    const bool grp_run = ((qrun >> (8 * grp)) & 0xFFu) == 0xFFu && gbase + 16 <= rows_max;
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(&bar.full[st], static_cast<uint32_t>(kLoadV ? kTcKV : 2 * kTcHalf));
    __syncwarp();
    unsigned char* kst = skv + st * kTcKV;
    unsigned char* vst = kst + 2 * kTcHalf;
    if (tile_run) {
      if (lane == 0) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          tma_rows(kst + hf * kTcHalf, &mp.m[4], hf * 64, tbase, &bar.full[st]);
          if (kLoadV) tma_rows(vst + hf * kTcHalf, &mp.m[5], hf * 64, tbase, &bar.full[st]);
        }
      }
    } else if (lane < kTcKeys / 4) {
      if (grp_run) {
        if ((lane & 3) == 0) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            tma_rows(kst + hf * kTcHalf + grp * 2048, &mp.m[2], hf * 64, gbase, &bar.full[st]);
            if (kLoadV) tma_rows(vst + hf * kTcHalf + grp * 2048, &mp.m[3], hf * 64, gbase, &bar.full[st]);
          }
        }
      } else {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          tma_gather4(kst + hf * kTcHalf + lane * 512, &mp.m[0], hf * 64, g0, g1, g2, g3, &bar.full[st]);
          if (kLoadV) tma_gather4(vst + hf * kTcHalf + lane * 512, &mp.m[1], hf * 64, g0, g1, g2, g3, &bar.full[st]);
        }
      }
    }
    prefetch(t + kPrefetch);   // into the buffer tile t was read from (its values are in registers)
  }
  if (kPass2) {
#pragma unroll 1
    for (int u = ntiles > kTcStages ? ntiles - kTcStages : 0; u < ntiles; ++u) {
      (void)mbar_wait_bounded(&bar.empty[u % kTcStages], (u / kTcStages) & 1, A.ws.status);
      retire(u);
    }
  }
}

__device__ __forceinline__ void ws_init_bars(WsBars& bar, uint32_t full_count, uint32_t empty_count,
                                             uint32_t free_count) {
  mbar_init(&bar.qfull, 32);
  for (int s = 0; s < kTcStages; ++s) {
    mbar_init(&bar.full[s], full_count);
    mbar_init(&bar.empty[s], empty_count);
  }
  for (int b = 0; b < 2; ++b) {
    mbar_init(&bar.x_full[b], 1);
    mbar_init(&bar.x_free[b], free_count);
    mbar_init(&bar.pv_done[b], 1);
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// pass 1.  Issue order S(0), then per tile S(t+1), P V(t): the tensor core
// computes the next scores while the row warps exponentiate.  x_full[b]:
// S(t) done (b = t & 1); x_free[b]: P(t) written by the 8 row warps;
// pv_done[b]: P V(t) done; empty[s]: P V and the 8 row warps (which also
// take |v|^2 of the tile's keys for pass 2) are done with the stage.
// Without V (kWithV false: the attention-mass scores need only the LSE) the
// stages hold K alone, no P V is issued and the rows keep only (max, sum).
template <bool kWithV>
__global__ void __launch_bounds__(kWsThreads, 1)
    d3_tc_pass1_kernel(D3Args A, const __grid_constant__ D3Maps mp) {
  extern __shared__ unsigned char d3_dsm[];
  __shared__ int sh_pos[kTcStages][kTcKeys];
  __shared__ float sh_ml[128][2];
  __shared__ __align__(8) WsBars bar;
  __shared__ uint32_t sh_taddr;
  const int chunk = blockIdx.x, l = blockIdx.y;
  const int n = min(max(A.ls.count[l], 0), A.dm.cap);
  const int j_begin = chunk * A.chunk_keys;
  if (j_begin >= n) return;
  const int j_end = min(n, j_begin + A.chunk_keys);
  const int ntiles = (j_end - j_begin + kTcKeys - 1) / kTcKeys;
  unsigned char* sq = align1024(d3_dsm);
  unsigned char* skv = sq + kTcQ;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == kWsIssuer) tc::alloc(&sh_taddr, kTcCols);
  if (tid == 0) ws_init_bars(bar, 1, 1 + kWsRowThreads / 32, kWsRowThreads / 32);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tl = sh_taddr;
  // at most 128 rows without V: one row tile; warps w and w + 4 share its
  // rows, each taking 32 keys of every tile
  const bool split = !kWithV && A.rows <= 128;

  if (warp == kWsProducer) {
    ws_produce<false, kWithV>(A, mp, l, j_begin, j_end, ntiles, sq, skv, sh_pos, nullptr, nullptr, bar);
  } else if (warp == kWsIssuer) {
    if ((tid & 31) == 0) {
      (void)mbar_wait_bounded(&bar.qfull, 0, A.ws.status);
      auto issue_s = [&](int t) {
        const int st = t % kTcStages, buf = t & 1;
        (void)mbar_wait_bounded(&bar.full[st], (t / kTcStages) & 1, A.ws.status);
        tc::fence_after();
        const unsigned char* kst = skv + st * kTcKV;
        tc_issue_s(tl + 256 + buf * 128, sq, kst, 0);
        if (!split) tc_issue_s(tl + 256 + buf * 128 + 64, sq, kst, 1);
        tc::commit(&bar.x_full[buf]);
      };
      issue_s(0);
#pragma unroll 1
      for (int t = 0; t < ntiles; ++t) {
        if (t + 1 < ntiles) issue_s(t + 1);
        const int st = t % kTcStages, buf = t & 1;
        (void)mbar_wait_bounded(&bar.x_free[buf], (t >> 1) & 1, A.ws.status);
        tc::fence_after();
        const uint32_t vbase = smem_u32(skv + st * kTcKV + 2 * kTcHalf);
#pragma unroll
        for (int mm = 0; mm < (kWithV ? 2 : 0); ++mm) {
          const uint32_t aP = tl + 256 + buf * 128 + mm * 64;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t bd = tc::desc_sw128(vbase + ks * 2048, kTcHalf, 1024);
            tc::mma_ts(tl + mm * 128, aP + ks * 8, bd, kIdPV, (t > 0 || ks > 0) ? 1u : 0u);
            tc::mma_ts(tl + mm * 128, aP + 32 + ks * 8, bd, kIdPV, 1u);
          }
        }
        tc::commit(&bar.empty[st]);
        tc::commit(&bar.pv_done[buf]);
      }
    }
  } else if (!kWithV) {
    // row warps without V: each row's running (max, sum); split: rows
    // tid & 127, keys [32 h0, 32 h0 + 32) of each tile with h0 = warp / 4
    const int r = split ? (tid & 127) : tid, m = r >> 7, h0 = split ? (warp >> 2) : 0;
    const bool row_ok = r < A.rows;
    const int qp = row_ok ? A.qpos[r % A.w] : -1;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int nkeys = j_end - j_begin;
    float m_run = -INFINITY, l_run = 0.f;
#pragma unroll 1
    for (int t = 0; t < ntiles; ++t) {
      const int st = t % kTcStages, buf = t & 1;
      (void)mbar_wait_bounded(&bar.x_full[buf], (t >> 1) & 1, A.ws.status);
      (void)mbar_wait_bounded(&bar.full[st], (t / kTcStages) & 1, A.ws.status);   // key positions
      tc::fence_after();
      const uint32_t aS = tl + lane_off + 256 + buf * 128 + m * 64;
      float s[kTcKeys];
      {
        uint32_t v[4][16];
        tc::ld16(aS + h0 * 32, v[0]);
        tc::ld16(aS + h0 * 32 + 16, v[1]);
        if (!split) {
          tc::ld16(aS + 32, v[2]);
          tc::ld16(aS + 48, v[3]);
        }
        tc::wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
          for (int k = 0; k < 16; ++k) s[q4 * 16 + k] = __uint_as_float(v[q4][k]);
      }
      // the keys at or before the row: a prefix of the tile (positions ascend)
      int vis = 0;
      if (row_ok) {
        const int lim = min(kTcKeys, nkeys - t * kTcKeys);
        if (lim > 0 && sh_pos[st][lim - 1] <= qp) {
          vis = lim;
        } else {
          int lo = 0, hi = lim;
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (sh_pos[st][mid] <= qp) lo = mid + 1; else hi = mid;
          }
          vis = lo;
        }
      }
      // S read, positions read: the buffer and the stage are free
      tc::fence_before();
      __syncwarp();
      if ((tid & 31) == 0) {
        mbar_arrive1(&bar.x_free[buf]);
        mbar_arrive1(&bar.empty[st]);
      }
#pragma unroll 1
      for (int hh = 0; hh < (split ? 1 : 2); ++hh) {
        const int kv = vis - (h0 + hh) * 32;
        float tmax = -INFINITY;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          s[k] = k < kv ? s[k] : -INFINITY;
          tmax = fmaxf(tmax, s[k]);
        }
        tmax *= A.scale2;
        if (tmax > m_run + kTcRescale) {
          l_run *= (m_run == -INFINITY) ? 0.f : exp2f(m_run - tmax);
          m_run = tmax;
        }
        const float negm = m_run == -INFINITY ? 0.f : -m_run;
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 32; ++k) ps[k & 3] += hw_exp2(fmaf(s[k], A.scale2, negm));
        l_run += (ps[0] + ps[1]) + (ps[2] + ps[3]);
#pragma unroll
        for (int k = 0; k < 32; ++k) s[k] = s[32 + k];
      }
    }
    const size_t stride = kD + 2;
    if (split) {
      // merge the two key halves of each row (named barrier of the row warps)
      if (h0 == 1) {
        sh_ml[r][0] = m_run;
        sh_ml[r][1] = l_run;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (h0 == 0) {
        const float m1 = sh_ml[r][0], l1 = sh_ml[r][1];
        const float M = fmaxf(m_run, m1);
        if (M != -INFINITY) {
          l_run = l_run * exp2f(m_run - M) + l1 * exp2f(m1 - M);
          m_run = M;
        }
      }
    }
    float* part = A.ws.d3_part + (static_cast<size_t>(l) * A.chunks + chunk) * static_cast<size_t>(A.rows_cap) * stride +
                  static_cast<size_t>(r) * stride;
    if (row_ok && h0 == 0) {
      part[kD] = m_run;
      part[kD + 1] = l_run;
    }
  } else {
    // row warps: one window row per thread
    const int r = tid, m = r >> 7;
    const bool row_ok = r < A.rows;
    const int qp = row_ok ? A.qpos[r % A.w] : -1;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int nkeys = j_end - j_begin;
    float m_run = -INFINITY, l_run = 0.f;
#pragma unroll 1
    for (int t = 0; t < ntiles; ++t) {
      const int st = t % kTcStages, buf = t & 1;
      (void)mbar_wait_bounded(&bar.x_full[buf], (t >> 1) & 1, A.ws.status);
      (void)mbar_wait_bounded(&bar.full[st], (t / kTcStages) & 1, A.ws.status);   // key positions
      tc::fence_after();
      const uint32_t aS = tl + lane_off + 256 + buf * 128 + m * 64;
      float s[kTcKeys];
      {
        uint32_t v[4][16];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) tc::ld16(aS + q4 * 16, v[q4]);
        tc::wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
          for (int k = 0; k < 16; ++k) s[q4 * 16 + k] = __uint_as_float(v[q4][k]);
      }
      // a full tile whose last (largest) position precedes the row is wholly visible
      const bool all_vis = row_ok && (t + 1) * kTcKeys <= nkeys && sh_pos[st][kTcKeys - 1] <= qp;
      // the largest raw score of the tile (scale2 > 0 keeps the order; the
      // scale is applied once, and inside the exponent's FMA below)
      float tmax = -INFINITY;
      if (all_vis) {
#pragma unroll
        for (int k = 0; k < kTcKeys; ++k) tmax = fmaxf(tmax, s[k]);
      } else {
#pragma unroll
        for (int k = 0; k < kTcKeys; ++k) {
          const bool ok = row_ok && t * kTcKeys + k < nkeys && sh_pos[st][k] <= qp;
          s[k] = ok ? s[k] : -INFINITY;
          tmax = fmaxf(tmax, s[k]);
        }
      }
      tmax *= A.scale2;
      float factor = 1.f;
      if (tmax > m_run + kTcRescale) {
        factor = (m_run == -INFINITY) ? 0.f : exp2f(m_run - tmax);
        m_run = tmax;
        l_run *= factor;
      }
      if (kWithV && t > 0 && __any_sync(0xffffffffu, factor != 1.f)) {
        // P V(t - 1) must be complete before O is rescaled
        (void)mbar_wait_bounded(&bar.pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, A.ws.status);
        tc::fence_after();
        const uint32_t aO = tl + lane_off + m * 128;
#pragma unroll 1
        for (int q8 = 0; q8 < 8; ++q8) {
          uint32_t v[16];
          tc::ld16(aO + q8 * 16, v);
          tc::wait_ld();
#pragma unroll
          for (int k = 0; k < 16; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * factor);
          tc::st16(aO + q8 * 16, v);
        }
      }
      // p = 2^(s scale2 - m); a masked key (s = -inf) gives 0, and so does
      // every key while the row has seen none (m = -inf, offset taken as 0)
      const float negm = m_run == -INFINITY ? 0.f : -m_run;
      float psum = 0.f;
      uint32_t hi[32], lo[32];
#pragma unroll
      for (int k2 = 0; k2 < 32; ++k2) {
        const float p0 = hw_exp2(fmaf(s[2 * k2], A.scale2, negm));
        const float p1 = hw_exp2(fmaf(s[2 * k2 + 1], A.scale2, negm));
        psum += p0 + p1;
        split_bf16(p0, p1, hi[k2], lo[k2]);
      }
      l_run += psum;
      {
        uint32_t v[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = hi[k];
        tc::st16(aS, v);
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = hi[16 + k];
        tc::st16(aS + 16, v);
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = lo[k];
        tc::st16(aS + 32, v);
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = lo[16 + k];
        tc::st16(aS + 48, v);
      }
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if ((tid & 31) == 0) mbar_arrive1(&bar.x_free[buf]);
      // |v|^2 of the tile's keys for pass 2: four threads per key, 32 elements each
      {
        const int key = tid >> 2, part = tid & 3;
        const unsigned char* vst = skv + st * kTcKV + 2 * kTcHalf;
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 x = *reinterpret_cast<const uint4*>(vst + sw_off(key, (part * 4 + c) * 8));
          const __nv_bfloat162* pr = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float2 f = __bfloat1622float2(pr[u]);
            acc = fmaf(f.x, f.x, fmaf(f.y, f.y, acc));
          }
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        const int j = j_begin + t * kTcKeys + key;
        if (part == 0 && j < j_end) A.ws.d3_vn[static_cast<size_t>(l) * A.dm.cap + j] = acc;
      }
      __syncwarp();
      if ((tid & 31) == 0) mbar_arrive1(&bar.empty[st]);
    }
    const size_t stride = kD + 2;
    float* part = A.ws.d3_part + (static_cast<size_t>(l) * A.chunks + chunk) * static_cast<size_t>(A.rows_cap) * stride +
                  static_cast<size_t>(r) * stride;
    if (kWithV) {
      (void)mbar_wait_bounded(&bar.pv_done[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, A.ws.status);
      tc::fence_after();
    }
    const uint32_t aO = tl + lane_off + m * 128;
#pragma unroll
    for (int q8 = 0; q8 < (kWithV ? 8 : 0); ++q8) {
      uint32_t v[16];
      tc::ld16(aO + q8 * 16, v);
      tc::wait_ld();
      if (row_ok) {
#pragma unroll
        for (int k = 0; k < 16; k += 2)
          *reinterpret_cast<float2*>(part + q8 * 16 + k) = make_float2(__uint_as_float(v[k]), __uint_as_float(v[k + 1]));
      }
    }
    if (row_ok) {
      part[kD] = m_run;
      part[kD + 1] = l_run;
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == kWsIssuer) tc::dealloc(tl, kTcCols);
}

// p / (1 - p) * ||a - v|| for the one key of a row with p > 1/2, x = log2 p:
// the distance directly from the fp32 a row and the swizzled V tile (the
// expansion would cancel), 1 - p from expm1.
__device__ __noinline__ float residual_direct(float x, const float* arow, const unsigned char* vtile, int key) {
  const float p = exp2f(x);
  const float om = -expm1f(x * kLn2);
  if (!(om > 0.f)) return INFINITY;
  const float4* a4 = reinterpret_cast<const float4*>(arow);
  float acc = 0.f;
#pragma unroll 4
  for (int c = 0; c < kD / 8; ++c) {
    const uint4 raw = *reinterpret_cast<const uint4*>(vtile + sw_off(key, c * 8));
    const __nv_bfloat162* pr = reinterpret_cast<const __nv_bfloat162*>(&raw);
    const float4 x0 = a4[c * 2], x1 = a4[c * 2 + 1];
    const float2 v0 = __bfloat1622float2(pr[0]), v1 = __bfloat1622float2(pr[1]);
    const float2 v2 = __bfloat1622float2(pr[2]), v3 = __bfloat1622float2(pr[3]);
    float d;
    d = x0.x - v0.x; acc = fmaf(d, d, acc);
    d = x0.y - v0.y; acc = fmaf(d, d, acc);
    d = x0.z - v1.x; acc = fmaf(d, d, acc);
    d = x0.w - v1.y; acc = fmaf(d, d, acc);
    d = x1.x - v2.x; acc = fmaf(d, d, acc);
    d = x1.y - v2.y; acc = fmaf(d, d, acc);
    d = x1.z - v3.x; acc = fmaf(d, d, acc);
    d = x1.w - v3.y; acc = fmaf(d, d, acc);
  }
  return p / om * sqrtf(acc);
}

// pass 2.  x_full[0]: S(t) and G(t) done; x_free[0]: the 8 row warps have
// read them (the buffer may be overwritten); empty[s]: the MMAs and the 8 row
// warps are done with the stage.  Each row warp leaves its 32 rows' sum per
// key of the tile in col[stage][warp]; the producer adds the 8 when it
// recycles the stage.
constexpr float kSmallLog2 = -7.f;   // p < 2^-7: p / (1 - p) = p + p^2 + p^3 within 2^-21
constexpr float kR2Floor = 1e-30f;   // r2 floor: sqrt(r2) = r2 rsqrt(r2) stays finite (1e-15 for r2 = 0)

// kMode (D3Mode): kResidual as above; the mass modes issue S alone, load no
// V and sum the weights of the keys the row counts.
template <int kMode>
__global__ void __launch_bounds__(kWsThreads, 1)
    d3_tc_pass2_kernel(D3Args A, const __grid_constant__ D3Maps mp) {
  extern __shared__ unsigned char d3_dsm[];
  __shared__ int sh_pos[kTcStages][kTcKeys];
  __shared__ __align__(16) float sh_vn[kTcStages][kTcKeys];
  __shared__ float sh_col[kTcStages][kWsRowThreads / 32][kTcKeys];
  __shared__ __align__(8) WsBars bar;
  __shared__ uint32_t sh_taddr;
  const int chunk = blockIdx.x, l = blockIdx.y;
  const int n = min(max(A.ls.count[l], 0), A.dm.cap);
  const int j_begin = chunk * A.chunk_keys;
  if (j_begin >= n) return;
  const int j_end = min(n, j_begin + A.chunk_keys);
  const int ntiles = (j_end - j_begin + kTcKeys - 1) / kTcKeys;
  unsigned char* sq = align1024(d3_dsm);
  unsigned char* skv = sq + kTcQ;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == kWsIssuer) tc::alloc(&sh_taddr, kTcCols);
  if (tid == 0) ws_init_bars(bar, 1, 1 + kWsRowThreads / 32, kWsRowThreads / 32);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tl = sh_taddr;
  const int b = l / A.dm.Hkv, kh = l % A.dm.Hkv;
  // mass modes with at most 128 rows: one row tile; warps w and w + 4 share
  // its rows, warp w summing keys 0-31 of each tile and warp w + 4 keys 32-63
  const bool split = kMode != kResidual && A.rows <= 128;
  const int r = split ? (tid & 127) : tid, m = r >> 7, h0 = split && tid < kWsRowThreads ? (warp >> 2) : 0;
  const bool row_ok = r < A.rows;
  const size_t wrow = static_cast<size_t>(l) * A.rows_cap + (row_ok ? r : 0);
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  if (kMode == kResidual && warp < kWsProducer) {
    // a of this row (bf16 hi and lo) into tensor memory
    const uint4* hsrc = reinterpret_cast<const uint4*>(A.ws.d3_ahi + wrow * kD);
    const uint4* lsrc = reinterpret_cast<const uint4*>(A.ws.d3_alo + wrow * kD);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      uint32_t vh[16], vl[16];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 x = row_ok ? hsrc[q4 * 4 + u] : make_uint4(0, 0, 0, 0);
        const uint4 y = row_ok ? lsrc[q4 * 4 + u] : make_uint4(0, 0, 0, 0);
        vh[u * 4 + 0] = x.x; vh[u * 4 + 1] = x.y; vh[u * 4 + 2] = x.z; vh[u * 4 + 3] = x.w;
        vl[u * 4 + 0] = y.x; vl[u * 4 + 1] = y.y; vl[u * 4 + 2] = y.z; vl[u * 4 + 3] = y.w;
      }
      tc::st16(tl + lane_off + m * 64 + q4 * 16, vh);
      tc::st16(tl + lane_off + 128 + m * 64 + q4 * 16, vl);
    }
    tc::wait_st();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();

  if (warp == kWsProducer) {
    ws_produce<true, kMode == kResidual>(A, mp, l, j_begin, j_end, ntiles, sq, skv, sh_pos, sh_vn, sh_col, bar);
  } else if (warp == kWsIssuer) {
    if (lane == 0) {
      (void)mbar_wait_bounded(&bar.qfull, 0, A.ws.status);
#pragma unroll 1
      for (int t = 0; t < ntiles; ++t) {
        const int st = t % kTcStages;
        (void)mbar_wait_bounded(&bar.full[st], (t / kTcStages) & 1, A.ws.status);
        if (t > 0) (void)mbar_wait_bounded(&bar.x_free[0], (t - 1) & 1, A.ws.status);
        tc::fence_after();
        const unsigned char* kst = skv + st * kTcKV;
        const unsigned char* vst = kst + 2 * kTcHalf;
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
          if (split && mm == 1) break;
          tc_issue_s(tl + 256 + mm * 64, sq, kst, mm);
#pragma unroll
          for (int ks = 0; ks < (kMode == kResidual ? 8 : 0); ++ks) {
            const int half = ks >> 2, kin = ks & 3;
            const uint64_t bd = tc::desc_sw128(smem_u32(vst + half * kTcHalf) + kin * 32, 16, 1024);
            tc::mma_ts(tl + 384 + mm * 64, tl + mm * 64 + ks * 8, bd, kIdS, ks > 0 ? 1u : 0u);
            tc::mma_ts(tl + 384 + mm * 64, tl + 128 + mm * 64 + ks * 8, bd, kIdS, 1u);
          }
        }
        tc::commit(&bar.x_full[0]);
        tc::commit(&bar.empty[st]);
      }
    }
  } else {
    const int qp = row_ok ? A.qpos[r % A.w] : -1;
    const float lse2 = row_ok ? A.ws.d3_rowc[wrow * 2] : 0.f;
    const float an = row_ok ? A.ws.d3_rowc[wrow * 2 + 1] : 0.f;
    const float* arow = A.a_out;
    if (row_ok) {
      const int h = r / A.w, i = r % A.w;
      arow = A.a_out + ((static_cast<size_t>(b) * A.dm.Hq + kh * A.dm.g + h) * A.w + i) * kD;
    }
    const int nkeys = j_end - j_begin;
    if (kMode != kResidual) {
#pragma unroll 1
      for (int t = 0; t < ntiles; ++t) {
        const int st = t % kTcStages;
        (void)mbar_wait_bounded(&bar.full[st], (t / kTcStages) & 1, A.ws.status);   // positions
        (void)mbar_wait_bounded(&bar.x_full[0], t & 1, A.ws.status);
        tc::fence_after();
        float sv[kTcKeys];
        {
          uint32_t v[4][16];
          const uint32_t aS = tl + lane_off + 256 + m * 64;
          tc::ld16(aS + h0 * 32, v[0]);
          tc::ld16(aS + h0 * 32 + 16, v[1]);
          if (!split) {
            tc::ld16(aS + 32, v[2]);
            tc::ld16(aS + 48, v[3]);
          }
          tc::wait_ld();
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
            for (int k = 0; k < 16; ++k) sv[q4 * 16 + k] = __uint_as_float(v[q4][k]);
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive1(&bar.x_free[0]);
        // the keys the row counts are a prefix of the tile (positions ascend)
        int vis = 0;
        if (row_ok) {
          const int lim = min(kTcKeys, nkeys - t * kTcKeys);
          auto counted = [&](int k) { return kMode == kMassLater ? sh_pos[st][k] < qp : sh_pos[st][k] <= qp; };
          if (lim > 0 && counted(lim - 1)) {
            vis = lim;
          } else {
            int lo = 0, hi = lim;
            while (lo < hi) {
              const int mid = (lo + hi) >> 1;
              if (counted(mid)) lo = mid + 1; else hi = mid;
            }
            vis = lo;
          }
        }
        if (split) sh_col[st][warp][(1 - h0) * 32 + lane] = 0.f;   // the other warp of the pair sums those keys
#pragma unroll 1
        for (int hf = h0; hf < (split ? h0 + 1 : 2); ++hf) {
          const int kv = vis - hf * 32;
#pragma unroll
          for (int k2 = 0; k2 < kTcKeys / 2; ++k2)
            sv[k2] = k2 < kv ? hw_exp2(fmaf(sv[k2], A.scale2, -lse2)) : 0.f;
#pragma unroll
          for (int o = 16, cnt = kTcKeys / 2; o >= 1; o >>= 1, cnt >>= 1) {
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < cnt / 2; ++i) {
              const float send = up ? sv[i] : sv[cnt / 2 + i];
              const float keep = up ? sv[cnt / 2 + i] : sv[i];
              sv[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
          }
          sh_col[st][warp][hf * 32 + lane] = sv[0];
#pragma unroll
          for (int k2 = 0; k2 < kTcKeys / 2; ++k2) sv[k2] = sv[kTcKeys / 2 + k2];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive1(&bar.empty[st]);
      }
    } else {
#pragma unroll 1
    for (int t = 0; t < ntiles; ++t) {
      const int st = t % kTcStages;
      const unsigned char* vst = skv + st * kTcKV + 2 * kTcHalf;
      (void)mbar_wait_bounded(&bar.full[st], (t / kTcStages) & 1, A.ws.status);   // positions, |v|^2, V
      // S and G of the tile's 64 keys; once read, the next tile's MMAs may
      // overwrite them
      (void)mbar_wait_bounded(&bar.x_full[0], t & 1, A.ws.status);
      tc::fence_after();
      float sv[kTcKeys], gv[kTcKeys];
      {
        uint32_t v[4][16], w[4][16];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          tc::ld16(tl + lane_off + 256 + m * 64 + q4 * 16, v[q4]);
          tc::ld16(tl + lane_off + 384 + m * 64 + q4 * 16, w[q4]);
        }
        tc::wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            sv[q4 * 16 + k] = __uint_as_float(v[q4][k]);
            gv[q4 * 16 + k] = __uint_as_float(w[q4][k]);
          }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive1(&bar.x_free[0]);
      // keys visible to the row: positions ascend within the tile, so they
      // are a prefix (binary search of the row's query position)
      int vis = 0;
      if (row_ok) {
        const int lim = min(kTcKeys, nkeys - t * kTcKeys);
        if (lim > 0 && sh_pos[st][lim - 1] <= qp) {
          vis = lim;
        } else {
          int lo = 0, hi = lim;   // first key with position > qp lies in [lo, hi)
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (sh_pos[st][mid] <= qp) lo = mid + 1; else hi = mid;
          }
          vis = lo;
        }
      }
      // the two halves go through one copy of the code (the row loop is long
      // and instruction fetch stalls when it is duplicated); after the first,
      // the second half's registers move down
#pragma unroll 1
      for (int hf = 0; hf < 2; ++hf) {
        const int kv = vis - hf * 32;   // visible keys of this half: k2 < kv
        // weights p = 2^x of the half's keys in place of S (x = -inf, p = 0
        // where not visible), and the largest x
        float xmax = -INFINITY;
        if (__all_sync(0xffffffffu, kv >= kTcKeys / 2)) {
#pragma unroll
          for (int k2 = 0; k2 < kTcKeys / 2; ++k2) {
            const float x = fmaf(sv[k2], A.scale2, -lse2);
            xmax = fmaxf(xmax, x);
            sv[k2] = hw_exp2(x);
          }
        } else {
#pragma unroll
          for (int k2 = 0; k2 < kTcKeys / 2; ++k2) {
            const float x = k2 < kv ? fmaf(sv[k2], A.scale2, -lse2) : -INFINITY;
            xmax = fmaxf(xmax, x);
            sv[k2] = hw_exp2(x);
          }
        }
        if (!__any_sync(0xffffffffu, xmax >= kSmallLog2)) {
          // every weight of the warp's rows is small: no reciprocal, and
          // sqrt(r2) = r2 rsqrt(r2) (a key that is not visible has p = 0)
          const float4* vn4 = reinterpret_cast<const float4*>(&sh_vn[st][hf * 32]);
#pragma unroll
          for (int k4 = 0; k4 < kTcKeys / 8; ++k4) {
            const float4 vq = vn4[k4];
            const float vv[4] = {vq.x, vq.y, vq.z, vq.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int k2 = k4 * 4 + u;
              const float p = sv[k2];
              const float r2 = fmaxf(kR2Floor, fmaf(-2.f, gv[k2], an + vv[u]));
              const float q = fmaf(fmaf(p, p, p), p, p);   // p + p^2 + p^3
              sv[k2] = q * r2 * hw_rsqrt(r2);
            }
          }
        } else {
          int xk = -1;
#pragma unroll
          for (int k2 = 0; k2 < kTcKeys / 2; ++k2) {
            const float p = sv[k2];
            const float r2 = fmaxf(0.f, fmaf(-2.f, gv[k2], an + sh_vn[st][hf * 32 + k2]));
            float tm = p * hw_rcp(1.f - p) * hw_sqrt(r2);
            if (p > 0.5f) { xk = k2; tm = 0.f; }
            sv[k2] = p > 0.f ? tm : 0.f;
          }
          // the one key of the row with p > 1/2 (the largest x): direct
          // distance, out of line
          if (xk >= 0) {
            const float dterm = residual_direct(xmax, arow, vst, hf * 32 + xk);
#pragma unroll
            for (int k2 = 0; k2 < kTcKeys / 2; ++k2)
              if (k2 == xk) sv[k2] = dterm;
          }
        }
        // butterfly: each lane ends with the warp's sum of one key
#pragma unroll
        for (int o = 16, cnt = kTcKeys / 2; o >= 1; o >>= 1, cnt >>= 1) {
          const bool up = (lane & o) != 0;
#pragma unroll
          for (int i = 0; i < cnt / 2; ++i) {
            const float send = up ? sv[i] : sv[cnt / 2 + i];
            const float keep = up ? sv[cnt / 2 + i] : sv[i];
            sv[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
        sh_col[st][warp][hf * 32 + lane] = sv[0];
#pragma unroll
        for (int k2 = 0; k2 < kTcKeys / 2; ++k2) {
          sv[k2] = sv[kTcKeys / 2 + k2];
          gv[k2] = gv[kTcKeys / 2 + k2];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive1(&bar.empty[st]);    // this warp is done with the stage
    }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == kWsIssuer) tc::dealloc(tl, kTcCols);
}

}  // namespace

int d3_rows_max(const Dims& dm) { return dm.g * dm.max_window; }

cudaError_t prepare_dropkv() {
  const void* fns[] = {reinterpret_cast<const void*>(d3_tc_pass1_kernel<true>),
                       reinterpret_cast<const void*>(d3_tc_pass1_kernel<false>),
                       reinterpret_cast<const void*>(d3_tc_pass2_kernel<kResidual>),
                       reinterpret_cast<const void*>(d3_tc_pass2_kernel<kMassCausal>),
                       reinterpret_cast<const void*>(d3_tc_pass2_kernel<kMassLater>)};
  for (const void* f : fns) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}
// Keys per CTA: each lane's keys split over floor(SMs / lanes) CTAs (one
// wave when the lanes are few), in whole 64-key tiles, at least kChunkMin.
// sm_count 0 gives the most chunks any device can use (workspace sizing).
static int d3_chunk_keys(const Dims& dm, int sm_count) {
  const int per_lane = sm_count > 0 ? max(1, sm_count / max(1, dm.lanes)) : 1 << 30;
  const int k = (dm.cap + per_lane - 1) / per_lane;
  return max(kChunkMin, (k + kTcKeys - 1) / kTcKeys * kTcKeys);
}
int d3_chunks(const Dims& dm, int sm_count) {
  const int ck = d3_chunk_keys(dm, sm_count);
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
  const cuuint32_t box_rows[3] = {1, 16, static_cast<cuuint32_t>(kTcKeys)};
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
  A.chunk_keys = d3_chunk_keys(dm, ctx.sm_count);
  A.chunks = d3_chunks(dm, ctx.sm_count);
  A.lse_out = lse; A.a_out = a_out; A.scores = scores;
  A.col_out = pool_r >= 0 ? ctx.ws.d3_score_part : scores;
  A.scale2 = 1.4426950408889634f / sqrtf(static_cast<float>(dm.d));
  if (A.rows > A.rows_cap || A.rows > kMaxRowGroups * kRowsPerCta || dm.d != kD || dm.dtype != KVEVICT_BF16)
    return cudaErrorInvalidValue;
  const bool res = mode == kResidual;
  if (A.rows <= kTcRows) {
    const dim3 grid(A.chunks, dm.lanes);
    if (!ctx.tmaps) return cudaErrorInvalidValue;
    D3Maps mp;
    for (int i = 0; i < kTmapsPerLayer; ++i) mp.m[i] = ctx.tmaps[static_cast<size_t>(layer) * kTmapsPerLayer + i];
    const dim3 cgrid((A.rows + 7) / 8, dm.lanes);
    if (res) {
      d3_tc_pass1_kernel<true><<<grid, kWsThreads, kTcSmem, stream>>>(A, mp);
      d3_combine_kernel<true><<<cgrid, 256, 0, stream>>>(A);
      d3_tc_pass2_kernel<kResidual><<<grid, kWsThreads, kTcSmem, stream>>>(A, mp);
    } else {
      d3_tc_pass1_kernel<false><<<grid, kWsThreads, kTcSmem, stream>>>(A, mp);
      d3_combine_kernel<false><<<cgrid, 256, 0, stream>>>(A);
      if (mode == kMassLater)
        d3_tc_pass2_kernel<kMassLater><<<grid, kWsThreads, kTcSmem, stream>>>(A, mp);
      else
        d3_tc_pass2_kernel<kMassCausal><<<grid, kWsThreads, kTcSmem, stream>>>(A, mp);
    }
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
