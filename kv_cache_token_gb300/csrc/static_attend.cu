// Decode attention that allocates nothing.
//
// Some callers cannot hand the library device memory for scratch: code that
// runs while a CUDA graph is being captured (cudaMalloc is not a capturable
// operation and breaks the capture), hosts whose device memory is owned by
// their own allocator and never cede raw allocations, and serving loops that
// forbid allocation on the hot path because cudaMalloc synchronises the whole
// device.  kvevict_attend_static serves them: it runs the engine's split-K
// attention for one layer and writes each lane's attention output and
// log-sum-exp, using as scratch a fixed array compiled into this library
// instead of the caller's workspace.  The engine's tables are read, never
// changed.
//
// The array is KVEVICT_STATIC_SCRATCH_BYTES long and lives on every GPU that
// loads the library until the process exits.  Host code cannot use the
// array's name as a device address, so the first call on each device looks
// the address up (cudaGetSymbolAddress) with that device current and keeps
// it, together with the CUDA context it belongs to; that first call should
// therefore happen before any stream capture.  A later call that finds
// another context current on the device (after cudaDeviceReset, say) looks
// the address up again.
// All calls share the one array: calls whose kernels overlap on the GPU (two
// streams, or two host threads) race on it and give undefined results.
// Nothing in it needs to start at zero: every scratch word a call reads was
// written earlier by the same call.
#include <mutex>

#include "kvevict_internal.cuh"

namespace {

constexpr size_t kStaticBytes = KVEVICT_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_attend_scratch[kStaticBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

// The calling thread's current CUDA context (null if none or not known),
// through the runtime's driver entry point.
CUcontext current_context() {
  using GetCurrent = CUresult (*)(CUcontext*);
  static GetCurrent fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<GetCurrent>(f);
  }();
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

inline size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Bytes of scratch a layer of this configuration needs, carved in the order
// logits, partial outputs, partial (max, sum), segment counts.
size_t scratch_bytes(const kve::Dims& dm, size_t* off) {
  const size_t lanes = dm.lanes, g = dm.g, d = dm.d;
  off[0] = 0;
  off[1] = off[0] + up256(lanes * g * dm.lcap * 4);
  off[2] = off[1] + up256(lanes * kve::kMaxSeg * g * d * 4);
  off[3] = off[2] + up256(lanes * kve::kMaxSeg * g * 2 * 4);
  return off[3] + up256(lanes * 4);
}

// Per lane: merge the split-K segments into the output and log-sum-exp.
__global__ void __launch_bounds__(256) static_combine_kernel(const float* part_o, const float* part_ml,
                                                              const int32_t* lane_nseg, int g, int d, int Hkv,
                                                              int Hq, float* out, float* lse) {
  __shared__ float sh_scale[kve::kMaxSeg][kve::kMaxG];
  __shared__ float sh_L[kve::kMaxG];
  const int l = blockIdx.x, tid = threadIdx.x;
  const int b = l / Hkv, kh = l % Hkv;
  const int nseg = min(lane_nseg[l], kve::kMaxSeg);
  const float2* ml = reinterpret_cast<const float2*>(part_ml) + static_cast<size_t>(l) * kve::kMaxSeg * g;
  const int warp = tid >> 5, lane = tid & 31;
  for (int h = warp; h < g; h += blockDim.x >> 5) {
    const float2 v0 = lane < nseg ? ml[lane * g + h] : make_float2(-INFINITY, 0.f);
    const float2 v1 = lane + 32 < nseg ? ml[(lane + 32) * g + h] : make_float2(-INFINITY, 0.f);
    const float M = kve::warp_max(fmaxf(v0.x, v1.x));
    const float s0 = v0.x == -INFINITY ? 0.f : exp2f(v0.x - M);
    const float s1 = v1.x == -INFINITY ? 0.f : exp2f(v1.x - M);
    if (lane < nseg) sh_scale[lane][h] = s0;
    if (lane + 32 < nseg) sh_scale[lane + 32][h] = s1;
    float Ls = v0.y * s0 + v1.y * s1;
    for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
    if (lane == 0) {
      sh_L[h] = Ls;
      lse[static_cast<size_t>(b) * Hq + kh * g + h] = (M + log2f(Ls)) * 0.6931471805599453f;
    }
  }
  __syncthreads();
  const float* po = part_o + static_cast<size_t>(l) * kve::kMaxSeg * g * d;
  for (int he = tid; he < g * d; he += blockDim.x) {
    const int h = he / d, e = he - h * d;
    float acc = 0.f;
    for (int s = 0; s < nseg; ++s) acc = fmaf(po[(static_cast<size_t>(s) * g + h) * d + e], sh_scale[s][h], acc);
    out[(static_cast<size_t>(b) * Hq + kh * g + h) * d + e] = acc / sh_L[h];
  }
}

}  // namespace

extern "C" kvevict_status kvevict_attend_static(kvevict_ctx* ctx, int layer, const void* q, const void* k_new,
                                                const void* v_new, float* out, float* lse, void* stream) {
  if (!ctx || layer < 0 || layer >= ctx->c.dims.L || !q || !k_new || !v_new || !out || !lse)
    return KVEVICT_E_INVALID_ARG;
  const kve::Dims& dm = ctx->c.dims;
  size_t off[4];
  if (scratch_bytes(dm, off) > kStaticBytes) return KVEVICT_E_SCRATCH_LIMIT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVEVICT_E_CUDA;
  char* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    const CUcontext cur = current_context();
    if (!g_scratch_addr[dev] || !cur || cur != g_scratch_ctx[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_attend_scratch) != cudaSuccess || !p) return KVEVICT_E_CUDA;
      g_scratch_addr[dev] = p;
      g_scratch_ctx[dev] = current_context();   // the lookup made the device's context current
    }
    base = static_cast<char*>(g_scratch_addr[dev]);
  }
  float* logits = reinterpret_cast<float*>(base + off[0]);
  float* part_o = reinterpret_cast<float*>(base + off[1]);
  float* part_ml = reinterpret_cast<float*>(base + off[2]);
  int32_t* nseg = reinterpret_cast<int32_t*>(base + off[3]);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = kve::launch_attend_into(ctx->c, layer, q, k_new, v_new, logits, part_o, part_ml, nseg, st);
  if (e != cudaSuccess) return KVEVICT_E_CUDA;
  static_combine_kernel<<<dm.lanes, 256, 0, st>>>(part_o, part_ml, nseg, dm.g, dm.d, dm.Hkv, dm.Hq, out, lse);
  return cudaGetLastError() == cudaSuccess ? KVEVICT_OK : KVEVICT_E_CUDA;
}
