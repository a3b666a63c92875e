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
#include "kvevict_internal.cuh"

namespace kve {
namespace {

constexpr int kD = 128;
constexpr int kRowStride = kD * 2 + 16;         // bytes per staged row
constexpr int kKeyTile = 32;                    // keys per tile
constexpr int kChunk = 1024;                    // keys per CTA
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
  int w, rows, rows_cap, chunks;
  float* lse_out; float* a_out; float* scores;
  float scale2;
};

// Shared staging of one key tile: K rows, V rows, positions, |v|^2.
struct Tile {
  unsigned char k[kKeyTile * kRowStride];
  unsigned char v[kKeyTile * kRowStride];
  int pos[kKeyTile];
  float vn[kKeyTile];
};

// Issue the cp.async copies of key tile [j0, j0 + 32) of lane l into t.
__device__ __forceinline__ void load_tile(Tile& t, const D3Args& A, int l, int n, int j0) {
  const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(A.ls.k_pool);
  const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(A.ls.v_pool);
  const size_t lo = static_cast<size_t>(l) * A.dm.cap;
  const size_t pool_rows = static_cast<size_t>(A.dm.P) * kBlock;
  // 32 keys x 2 tensors x 16 pieces of 16 bytes = 1024 pieces
  for (int e = threadIdx.x; e < kKeyTile * 2 * 16; e += blockDim.x) {
    const int key = e >> 5, tens = (e >> 4) & 1, piece = e & 15;
    const int j = j0 + key;
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
  const int j_begin = chunk * kChunk;
  if (j_begin >= n) return;
  const int j_end = min(n, j_begin + kChunk);
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
// combine: grid (lanes), one warp per row
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) d3_combine_kernel(D3Args A) {
  const int l = blockIdx.x;
  const int n = min(max(A.ls.count[l], 0), A.dm.cap);
  const int nch = (n + kChunk - 1) / kChunk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = l / A.dm.Hkv, kh = l % A.dm.Hkv;
  const size_t stride = kD + 2;
  const size_t chunk_stride = static_cast<size_t>(A.rows_cap) * stride;
  for (int r = warp; r < A.rows; r += blockDim.x >> 5) {
    const int h = r / A.w, i = r % A.w;
    const float* base = A.ws.d3_part + static_cast<size_t>(l) * A.chunks * chunk_stride + static_cast<size_t>(r) * stride;
    float M = -INFINITY;
    for (int c = 0; c < nch; ++c) M = fmaxf(M, base[c * chunk_stride + kD]);
    float Ls = 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c = 0; c < nch; ++c) {
      const float m = base[c * chunk_stride + kD];
      if (m == -INFINITY) continue;
      const float sc = exp2f(m - M);
      Ls += base[c * chunk_stride + kD + 1] * sc;
#pragma unroll
      for (int u = 0; u < 4; ++u) acc[u] += base[c * chunk_stride + lane + 32 * u] * sc;
    }
    const float lse2 = M + log2f(Ls);
    const size_t orow = (static_cast<size_t>(b) * A.dm.Hq + kh * A.dm.g + h) * A.w + i;
    float nrm = 0.f;
    const size_t wrow = static_cast<size_t>(l) * A.rows_cap + r;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float a = acc[u] / Ls;
      const int e = lane + 32 * u;
      A.a_out[orow * kD + e] = a;
      nrm += a * a;
      const __nv_bfloat16 hi = __float2bfloat16_rn(a);
      const __nv_bfloat16 lo = __float2bfloat16_rn(a - __bfloat162float(hi));
      A.ws.d3_ahi[wrow * kD + e] = hi;
      A.ws.d3_alo[wrow * kD + e] = lo;
    }
    for (int o = 16; o > 0; o >>= 1) nrm += __shfl_xor_sync(0xffffffffu, nrm, o);
    if (lane == 0) {
      A.lse_out[orow] = lse2 * kLn2;
      A.ws.d3_rowc[wrow * 2 + 0] = lse2;
      A.ws.d3_rowc[wrow * 2 + 1] = nrm;
    }
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
__global__ void __launch_bounds__(kWarps * 32) d3_pass2_kernel(D3Args A) {
  __shared__ __align__(128) Tile tiles[2];
  __shared__ float colsum[kWarps][kKeyTile];
  const int chunk = blockIdx.x, l = blockIdx.y, rg = blockIdx.z;
  const int n = min(max(A.ls.count[l], 0), A.dm.cap);
  const int j_begin = chunk * kChunk;
  if (j_begin >= n) return;
  const int j_end = min(n, j_begin + kChunk);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, cq = lane & 3;
  const int b = l / A.dm.Hkv, kh = l % A.dm.Hkv;
  const int r0 = rg * kRowsPerCta + warp * 16;
  const size_t wbase = static_cast<size_t>(l) * A.rows_cap;
  uint32_t qa[8][4], ah[8][4], al[8][4];
  load_afrag_q(qa, A, b, kh, r0);
  load_afrag_rows(ah, A.ws.d3_ahi + wbase * kD, A.rows, r0);
  load_afrag_rows(al, A.ws.d3_alo + wbase * kD, A.rows, r0);
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
  load_tile(tiles[0], A, l, n, j_begin);
  cp_commit();
  for (int t = 0; t < ntiles; ++t) {
    if (t + 1 < ntiles) load_tile(tiles[(t + 1) & 1], A, l, n, j_begin + (t + 1) * kKeyTile);
    cp_commit();
    cp_wait<1>();
    __syncthreads();
    Tile& T = tiles[t & 1];
    // |v|^2 of the tile's keys (warp 0)
    if (warp == 0) {
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
    tile_rows_dot(g, ah, T.v);
    tile_rows_dot(g, al, T.v);
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
        if (kp <= qpa) term += residual_term(s[nt][e] * A.scale2 - lsa, ana + vn - 2.f * g[nt][e], arow_a,
                                             T.v + key * kRowStride);
        if (kp <= qpb) term += residual_term(s[nt][2 + e] * A.scale2 - lsb, anb + vn - 2.f * g[nt][2 + e], arow_b,
                                             T.v + key * kRowStride);
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
    A.scores[static_cast<size_t>(l) * A.dm.cap + j] = tot;
  }
}

}  // namespace

int d3_rows_max(const Dims& dm) { return dm.g * dm.max_window; }
int d3_chunks(const Dims& dm, int) { return (dm.cap + kChunk - 1) / kChunk; }

cudaError_t launch_score(const Ctx& ctx, int layer, const void* q_win, int w, const int32_t* q_pos,
                         float* lse, float* a_out, float* scores, cudaStream_t stream) {
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
  A.chunks = d3_chunks(dm, ctx.sm_count);
  A.lse_out = lse; A.a_out = a_out; A.scores = scores;
  A.scale2 = 1.4426950408889634f / sqrtf(static_cast<float>(dm.d));
  if (A.rows > A.rows_cap || A.rows > kMaxRowGroups * kRowsPerCta || dm.d != kD || dm.dtype != KVEVICT_BF16)
    return cudaErrorInvalidValue;
  const int groups = (A.rows + kRowsPerCta - 1) / kRowsPerCta;
  dim3 grid(A.chunks, dm.lanes, groups);
  d3_pass1_kernel<<<grid, kWarps * 32, 0, stream>>>(A);
  d3_combine_kernel<<<dm.lanes, 256, 0, stream>>>(A);
  d3_pass2_kernel<<<grid, kWarps * 32, 0, stream>>>(A);
  dim3 fgrid((dm.cap + 255) / 256 < 64 ? (dm.cap + 255) / 256 : 64, dm.lanes);
  d3_finalize_kernel<<<fgrid, 256, 0, stream>>>(A, groups);
  return cudaGetLastError();
}

}  // namespace kve
