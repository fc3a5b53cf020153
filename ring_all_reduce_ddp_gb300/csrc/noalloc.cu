// The C ABI (include/ddp_ring.h): the reduce-scatter that allocates nothing.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <string>
#include <utility>

#include "host.h"

using namespace ddp;
using namespace ddp::host;

// ======================================= reduce-scatter that allocates nothing
// For callers that cannot allocate device memory: a framework whose caching
// allocator owns the whole device, or code that must not risk an allocation's
// failure or its implicit synchronisation in the middle of a step. The literal
// ring reduce-scatter keeps its fp32 partials in the fixed array below instead
// of a stream-ordered temporary. Every GPU that loads this library holds the
// array until the process exits.
namespace {

constexpr int64_t kNoAllocScratchBytes = int64_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
std::mutex g_noalloc_mutex;
struct ScratchAddr {
  unsigned long long ctx_id = 0;  // the context the address belongs to (0: none looked up yet)
  void* ptr = nullptr;
};
ScratchAddr g_noalloc_addr[64];

// The driver's cuCtxGetId, reached through the runtime (the library does not
// link the driver library itself). It returns an id that no other context of
// the process ever gets, so a destroyed and re-created primary context
// (cudaDeviceReset) is told apart from the one an address was looked up in.
using CtxGetIdFn = int (*)(void* ctx, unsigned long long* id);

ddp_status current_context_id(unsigned long long* id) {
  static CtxGetIdFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    (void)cudaGetLastError();
    return reinterpret_cast<CtxGetIdFn>(f);
  }();
  DDP_CHECK(fn != nullptr, DDP_ERR_CUDA, "the driver has no cuCtxGetId");
  if (fn(nullptr, id) != 0) {
    // No context current on this thread yet: cudaSetDevice binds the current
    // device's primary context (and allocates nothing on it).
    int dev = 0;
    DDP_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
    DDP_CUDA(cudaSetDevice(dev), "cudaSetDevice");
    DDP_CHECK(fn(nullptr, id) == 0, DDP_ERR_CUDA, "cuCtxGetId of the current context failed");
  }
  return DDP_OK;
}

// The array's device address in the current device's context, looked up once
// per device and context. In host code the array's name is only a stand-in:
// the address a kernel may use is the one cudaGetSymbolAddress returns with
// that device current, and it lasts as long as the context does.
ddp_status noalloc_scratch(float** out) {
  int dev = 0;
  DDP_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  DDP_CHECK(dev >= 0 && dev < 64, DDP_ERR_ARG, "device index out of range");
  unsigned long long ctx = 0;
  DDP_TRY(current_context_id(&ctx));
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  ScratchAddr& a = g_noalloc_addr[dev];
  if (a.ptr == nullptr || a.ctx_id != ctx) {
    void* ptr = nullptr;
    DDP_CUDA(cudaGetSymbolAddress(&ptr, g_noalloc_scratch), "cudaGetSymbolAddress of the scratch array");
    a.ptr = ptr;
    a.ctx_id = ctx;
  }
  *out = static_cast<float*>(a.ptr);
  return DDP_OK;
}

// Pairwise-disjoint byte ranges, sorted in place (no allocation).
bool disjoint_inplace(std::pair<uintptr_t, uintptr_t>* r, int count) {
  int m = 0;
  for (int i = 0; i < count; ++i)
    if (r[i].second > r[i].first) r[m++] = r[i];
  std::sort(r, r + m);
  for (int i = 1; i < m; ++i)
    if (r[i].first < r[i - 1].second) return false;
  return true;
}

}  // namespace

extern "C" ddp_status ddp_reduce_scatter_noalloc(const void* const* in, void* const* out, int32_t p, int64_t n,
                                                 ddp_dtype dtype, float divisor, ddp_own own,
                                                 cudaStream_t stream) {
  DDP_TRY(check_common(p, n, dtype));
  DDP_TRY(check_divisor(divisor));
  DDP_TRY(check_own(own));
  if (n == 0) return DDP_OK;  // a no-op whatever the pointers, as in ddp_reduce_scatter
  DDP_TRY(check_ptrs(in, p, "in"));
  DDP_TRY(check_ptrs(const_cast<const void* const*>(out), p, "out"));
  if (own == DDP_OWN_RANK)
    DDP_CHECK(n % p == 0, DDP_ERR_NOT_DIVISIBLE,
              "reduce_scatter: " + std::to_string(n) + " elements are not divisible by " + std::to_string(p) + " ranks");
  const int es = esize(dtype);
  const int64_t cs = chunk_size(n, p);
  const int64_t need = 2 * static_cast<int64_t>(p) * cs * static_cast<int64_t>(sizeof(float));
  DDP_CHECK(p == 1 || need <= kNoAllocScratchBytes, DDP_ERR_ARG,
            "ddp_reduce_scatter_noalloc: needs " + std::to_string(need) +
                " bytes of scratch (2 * p * ceil(n/p) fp32 partials), more than its fixed " +
                std::to_string(kNoAllocScratchBytes) + "-byte array; call ddp_reduce_scatter instead");
  std::pair<uintptr_t, uintptr_t> outs[DDP_MAX_P], all[DDP_MAX_P + 1];
  for (int r = 0; r < p; ++r) outs[r] = range_of(out[r], cs * es);
  for (int r = 0; r < p; ++r) all[r] = outs[r];
  DDP_CHECK(disjoint_inplace(all, p), DDP_ERR_ARG, "output buffers overlap");
  for (int r = 0; r < p; ++r) {
    for (int q = 0; q < p; ++q) all[q] = outs[q];
    all[p] = range_of(in[r], n * es);
    DDP_CHECK(disjoint_inplace(all, p + 1), DDP_ERR_ARG, "an output buffer overlaps an input");
  }
  if (p == 1)  // one scale step, no partials
    return run_fused(in, out, 1, n, dtype, divisor, true, 0, false, stream);
  float* scratch = nullptr;
  DDP_TRY(noalloc_scratch(&scratch));
  // Nothing in the array needs to start at zero: every slot a step reads was
  // written by the step before it in this same call.
  RingStepArgs a;
  for (int s = 0; s < p - 1; ++s) {
    std::memset(&a, 0, sizeof(a));
    for (int r = 0; r < p; ++r) {
      a.x[r] = const_cast<void*>(in[r]);
      a.out[r] = out[r];
    }
    a.w = scratch; a.n = n; a.cs = cs; a.divisor = divisor; a.p = p; a.step = s;
    a.shift = (own == DDP_OWN_RANK) ? 1 : 0; a.last = (s == p - 2); a.out_rel = 1;
    DDP_CUDA(launch_rs_step_ws(a, dtype, stream), "reduce-scatter step launch");
  }
  return DDP_OK;
}
