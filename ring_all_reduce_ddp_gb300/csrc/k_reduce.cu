// Reduction kernels: the fused one-pass ring-order reduction (all-reduce and
// reduce-scatter) and the literal reduce-scatter steps of the ring.
//
// Sources: "Collective Ops From Scratch", "Ring allreduce in two passes"
// (reduce-scatter: at step s rank r sends chunk (r - s) mod N to rank r + 1,
// which accumulates it; rank r ends owning chunk (r + 1) mod N; zero padding to
// a multiple of N); "Data parallelism", "Ring all-reduce, derived" (same
// phases) and "Overlapping communication with the backward pass" (the sum is
// divided by the number of ranks).
//
// The fused kernel does in one pass what the 2(p-1) ring steps do: chunk c's
// elements are first sent by rank c, so its sum is the left fold
// ((x_c + x_{c+1}) + ...) + x_{c+p-1}; the owner divides once and the
// all-gather copies the result to every replica. Padding never meets a real
// element, so it is never materialised.
#include <atomic>

#include "launch.h"

namespace ddp {

__device__ int g_device_error = 0;

// ------------------------------------------------ fused, register-only path
template <typename T, int P>
__global__ void __launch_bounds__(kThreads) k_fused_reduce_ldst(const __grid_constant__ FusedArgs a) {
  const int p = (P > 0) ? P : a.p;
  const int c = blockIdx.y;
  const int64_t lo = static_cast<int64_t>(c) * a.cs;
  const int64_t hi = min(a.n, lo + a.cs);
  if (lo >= hi) return;
  const int o = (c + a.shift) % p;            // origin rank of chunk c
  const int owner = (o + p - 1) % p;          // the rank pass 1 leaves it on
  const T* const* src = reinterpret_cast<const T* const*>(&a.src[o]);
  T* sdst = a.scatter ? reinterpret_cast<T*>(a.dst[owner]) : nullptr;  // chunk-relative
  constexpr int V = Vec<T>::N;
  const int64_t len = hi - lo;

  // Elements before the first 16-byte boundary (and all of them when the
  // replicas do not share an alignment) take the scalar path.
  int64_t head = len;
  if (a.same_align) {
    const uintptr_t addr = reinterpret_cast<uintptr_t>(src[0] + lo);
    const int64_t h = static_cast<int64_t>(((16u - (addr & 15u)) & 15u) / sizeof(T));
    bool ok = (addr % sizeof(T)) == 0;
    if (a.scatter) ok = ok && ((reinterpret_cast<uintptr_t>(sdst + h) & 15u) == 0);
    if (ok) head = min(h, len);
  }
  const int64_t nvec = (len - head) / V;
  const int64_t tail0 = head + nvec * V;
  const int64_t nscalar = head + (len - tail0);
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t gstride = static_cast<int64_t>(gridDim.x) * blockDim.x;

  for (int64_t e = gtid; e < nscalar; e += gstride) {
    const int64_t i = lo + (e < head ? e : tail0 + (e - head));
    float acc = widen(src[0][i]);
    for (int j = 1; j < p; ++j) acc = __fadd_rn(acc, widen(src[j][i]));
    const T y = narrow<T>(__fdiv_rn(acc, a.divisor));
    if (a.scatter) {
      sdst[i - lo] = y;
    } else {
      for (int r = 0; r < p; ++r) reinterpret_cast<T*>(a.dst[r])[i] = y;
    }
  }

  for (int64_t v = gtid; v < nvec; v += gstride) {
    const int64_t i = lo + head + v * V;
    float acc[V];
    if constexpr (P > 0) {
      uint4 x[P];
#pragma unroll
      for (int j = 0; j < P; ++j) x[j] = *reinterpret_cast<const uint4*>(src[j] + i);
      Vec<T>::unpack(x[0], acc);
#pragma unroll
      for (int j = 1; j < P; ++j) {
        float t[V];
        Vec<T>::unpack(x[j], t);
#pragma unroll
        for (int l = 0; l < V; ++l) acc[l] = __fadd_rn(acc[l], t[l]);
      }
    } else {
      constexpr int B = 8;
#pragma unroll
      for (int l = 0; l < V; ++l) acc[l] = 0.f;
      for (int j0 = 0; j0 < p; j0 += B) {
        uint4 x[B];
#pragma unroll
        for (int q = 0; q < B; ++q)
          if (j0 + q < p) x[q] = *reinterpret_cast<const uint4*>(src[j0 + q] + i);
#pragma unroll
        for (int q = 0; q < B; ++q) {
          if (j0 + q < p) {
            float t[V];
            Vec<T>::unpack(x[q], t);
            if (j0 + q == 0) {
#pragma unroll
              for (int l = 0; l < V; ++l) acc[l] = t[l];
            } else {
#pragma unroll
              for (int l = 0; l < V; ++l) acc[l] = __fadd_rn(acc[l], t[l]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int l = 0; l < V; ++l) acc[l] = __fdiv_rn(acc[l], a.divisor);
    const uint4 y = Vec<T>::pack(acc);
    if (a.scatter) {
      *reinterpret_cast<uint4*>(sdst + (i - lo)) = y;
    } else if constexpr (P > 0) {
#pragma unroll
      for (int r = 0; r < P; ++r) *reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.dst[r]) + i) = y;
    } else {
      for (int r = 0; r < p; ++r) *reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.dst[r]) + i) = y;
    }
  }
}

// ----------------------------------------------------- literal ring steps
constexpr int kU = 4;  // independent elements in flight per thread

__device__ __forceinline__ int sent_chunk(int r, int step, int shift, int p) {
  return ((r - step - shift) % p + p) % p;
}

// fp32 all-reduce, partials in the replicas themselves: rank r+1's copy of
// chunk (r - s) mod p becomes local + received; the last step also divides.
__global__ void __launch_bounds__(kThreads) k_rs_step_inplace_f32(const __grid_constant__ RingStepArgs a) {
  const int p = a.p;
  const int r = blockIdx.y;
  const int d = (r + 1) % p;
  const int c = sent_chunk(r, a.step, a.shift, p);
  const int64_t lo = static_cast<int64_t>(c) * a.cs;
  const int64_t hi = min(a.n, lo + a.cs);
  if (lo >= hi) return;
  const float* xs = reinterpret_cast<const float*>(a.x[r]) + lo;
  float* xd = reinterpret_cast<float*>(a.x[d]) + lo;
  const int64_t len = hi - lo;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kThreads * kU; base < len;
       base += static_cast<int64_t>(gridDim.x) * kThreads * kU) {
    float loc[kU], rcv[kU];
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      const int64_t e = base + q * kThreads + threadIdx.x;
      if (e < len) { loc[q] = xd[e]; rcv[q] = xs[e]; }
    }
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      const int64_t e = base + q * kThreads + threadIdx.x;
      if (e < len) {
        float y = __fadd_rn(loc[q], rcv[q]);
        if (a.last) y = __fdiv_rn(y, a.divisor);
        xd[e] = y;
      }
    }
  }
}

// Partials in the fp32 workspace w[2][p][cs] (bf16 all-reduce; reduce-scatter
// with const inputs). Step s: the sender's partial is its own input at s == 0,
// else the slot it received into at step s-1; the receiver adds its input and
// stores into its slot of half (s & 1), or, on the last step, writes
// round(fl32(sum / divisor)) to its output.
template <typename T>
__global__ void __launch_bounds__(kThreads) k_rs_step_ws(const __grid_constant__ RingStepArgs a) {
  const int p = a.p;
  const int r = blockIdx.y;
  const int d = (r + 1) % p;
  const int c = sent_chunk(r, a.step, a.shift, p);
  const int64_t lo = static_cast<int64_t>(c) * a.cs;
  const int64_t hi = min(a.n, lo + a.cs);
  if (lo >= hi) return;
  const int64_t len = hi - lo;
  const T* xs = reinterpret_cast<const T*>(a.x[r]) + lo;
  const T* xd = reinterpret_cast<const T*>(a.x[d]) + lo;
  const float* wprev = a.w + (static_cast<int64_t>((a.step + 1) & 1) * p + r) * a.cs;
  float* wcur = a.w + (static_cast<int64_t>(a.step & 1) * p + d) * a.cs;
  T* od = reinterpret_cast<T*>(a.out[d]) + (a.out_rel ? 0 : lo);
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kThreads * kU; base < len;
       base += static_cast<int64_t>(gridDim.x) * kThreads * kU) {
    float part[kU], loc[kU];
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      const int64_t e = base + q * kThreads + threadIdx.x;
      if (e < len) {
        part[q] = (a.step == 0) ? widen(xs[e]) : wprev[e];
        loc[q] = widen(xd[e]);
      }
    }
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      const int64_t e = base + q * kThreads + threadIdx.x;
      if (e < len) {
        const float v = __fadd_rn(part[q], loc[q]);
        if (a.last) od[e] = narrow<T>(__fdiv_rn(v, a.divisor));
        else wcur[e] = v;
      }
    }
  }
}

// ------------------------------------------------------------- launchers
namespace {
std::atomic<int64_t> g_launches{0};
int g_sm_count[64] = {0};

int blocks_per_chunk(int64_t work_items, int per_block, int chunks) {
  const int64_t target = static_cast<int64_t>(sm_count()) * (2048 / kThreads);
  int64_t bx = (target + chunks - 1) / chunks;
  const int64_t need = (work_items + per_block - 1) / per_block;
  if (bx > need) bx = need;
  if (bx < 1) bx = 1;
  if (bx > 65535 * 32) bx = 65535 * 32;
  return static_cast<int>(bx);
}

template <typename T>
cudaError_t fused_ldst(const FusedArgs& a, cudaStream_t s) {
  constexpr int V = Vec<T>::N;
  const dim3 grid(blocks_per_chunk(a.cs / V + 1, kThreads, a.p), a.p);
  switch (a.p) {
    case 2: k_fused_reduce_ldst<T, 2><<<grid, kThreads, 0, s>>>(a); break;
    case 4: k_fused_reduce_ldst<T, 4><<<grid, kThreads, 0, s>>>(a); break;
    case 8: k_fused_reduce_ldst<T, 8><<<grid, kThreads, 0, s>>>(a); break;
    case 16: k_fused_reduce_ldst<T, 16><<<grid, kThreads, 0, s>>>(a); break;
    default: k_fused_reduce_ldst<T, 0><<<grid, kThreads, 0, s>>>(a); break;
  }
  count_launch();
  return cudaGetLastError();
}
}  // namespace

int sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (g_sm_count[dev] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    g_sm_count[dev] = v > 0 ? v : 1;
  }
  return g_sm_count[dev];
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
int64_t launches() { return g_launches.load(std::memory_order_relaxed); }

cudaError_t launch_fused_reduce(const FusedArgs& a, ddp_dtype dt, bool staged, cudaStream_t s) {
  (void)staged;
  return dt == DDP_FLOAT32 ? fused_ldst<float>(a, s) : fused_ldst<__nv_bfloat16>(a, s);
}

cudaError_t launch_rs_step_inplace_f32(const RingStepArgs& a, cudaStream_t s) {
  const dim3 grid(blocks_per_chunk(a.cs, kThreads * kU, a.p), a.p);
  k_rs_step_inplace_f32<<<grid, kThreads, 0, s>>>(a);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_rs_step_ws(const RingStepArgs& a, ddp_dtype dt, cudaStream_t s) {
  const dim3 grid(blocks_per_chunk(a.cs, kThreads * kU, a.p), a.p);
  if (dt == DDP_FLOAT32) k_rs_step_ws<float><<<grid, kThreads, 0, s>>>(a);
  else k_rs_step_ws<__nv_bfloat16><<<grid, kThreads, 0, s>>>(a);
  count_launch();
  return cudaGetLastError();
}

cudaError_t read_device_error(cudaStream_t s, int* code) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
  }
  *code = v;
  return e;
}

}  // namespace ddp
