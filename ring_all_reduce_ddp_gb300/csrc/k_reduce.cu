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
#include <algorithm>
#include <atomic>
#include <cstring>

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


// ------------------------------------ fused, staged through shared memory
// Bulk asynchronous copies (the TMA's non-tensor form): one elected thread
// loads a tile of every replica into shared memory and signals an mbarrier;
// all threads fold the p copies in ring order into a result tile; the elected
// thread writes that tile back to every replica with p bulk stores. Stages are
// recycled in a ring so several tiles are in flight per SM.
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase with the given parity to complete; give up after
// timeout_ns nanoseconds and return false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, int64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (static_cast<int64_t>(global_ns() - t0) > timeout_ns) return false;
  }
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Block until at most n committed store groups may still be reading shared memory.
__device__ __forceinline__ void bulk_wait_read(int n) {
  switch (n) {
    case 0: asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.bulk.wait_group.read 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.bulk.wait_group.read 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.bulk.wait_group.read 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.bulk.wait_group.read 6;" ::: "memory"); break;
    default: asm volatile("cp.async.bulk.wait_group.read 7;" ::: "memory"); break;
  }
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

constexpr int kMaxStages = 8;
constexpr int kErrBulkWait = 1;  // device error code: a bulk copy did not complete in time

template <typename T>
__device__ __forceinline__ void staged_scalar(const StagedArgs& a, int c, int64_t i) {
  const int p = a.p;
  const int o = (c + a.shift) % p;
  float acc = widen(reinterpret_cast<const T*>(a.rep[o])[i]);
  int r = o;
  for (int j = 1; j < p; ++j) {
    r = (r + 1 == p) ? 0 : r + 1;
    acc = __fadd_rn(acc, widen(reinterpret_cast<const T*>(a.rep[r])[i]));
  }
  const T y = narrow<T>(__fdiv_rn(acc, a.divisor));
  if (a.scatter) {
    reinterpret_cast<T*>(a.out[(o + p - 1) % p])[i - static_cast<int64_t>(c) * a.cs] = y;
  } else {
    for (int q = 0; q < p; ++q) reinterpret_cast<T*>(a.rep[q])[i] = y;
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) k_fused_reduce_staged(const __grid_constant__ StagedArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int V = Vec<T>::N;
  const int p = a.p;
  const int S = a.stages;
  const int tile_bytes = a.tile_elems * static_cast<int>(sizeof(T));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  unsigned char* data = smem + 128;                        // [S][p][tile_bytes]
  unsigned char* res = data + static_cast<size_t>(S) * p * tile_bytes;  // [S][tile_bytes]
  __shared__ int s_abort;

  // 1. elements outside the aligned bodies, scalar, chunks round-robin over CTAs
  for (int c = blockIdx.x; c < p; c += gridDim.x) {
    const int64_t lo = min(a.n, static_cast<int64_t>(c) * a.cs);
    const int64_t hi = min(a.n, lo + a.cs);
    const int64_t b0 = a.body_lo[c], b1 = a.body_lo[c] + a.body_len[c];
    for (int64_t i = lo + threadIdx.x; i < b0; i += blockDim.x) staged_scalar<T>(a, c, i);
    for (int64_t i = b1 + threadIdx.x; i < hi; i += blockDim.x) staged_scalar<T>(a, c, i);
  }

  // 2. the aligned bodies, tile by tile
  const int32_t total = a.tile0[p];
  const int my_tiles = (blockIdx.x < total) ? (total - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
  if (my_tiles == 0) return;
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int st = 0; st < S; ++st) mbar_init(smem_addr(&bars[st]), 1);
    fence_mbar_init();
  }
  __syncthreads();

  // tile geometry: chunk, first element, element count
  auto tile_at = [&](int j, int& c, int64_t& i0, int& len) {
    const int32_t g = static_cast<int32_t>(blockIdx.x) + j * static_cast<int32_t>(gridDim.x);
    int lo = 0, hi = p;  // tile0[lo] <= g < tile0[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (a.tile0[mid] <= g) lo = mid; else hi = mid;
    }
    c = lo;
    const int64_t off = static_cast<int64_t>(g - a.tile0[c]) * a.tile_elems;
    i0 = a.body_lo[c] + off;
    len = static_cast<int>(min(static_cast<int64_t>(a.tile_elems), a.body_len[c] - off));
  };
  auto issue_loads = [&](int j, int st) {
    int c, len;
    int64_t i0;
    tile_at(j, c, i0, len);
    const uint32_t bytes = static_cast<uint32_t>(len) * sizeof(T);
    const uint32_t bar = smem_addr(&bars[st]);
    mbar_arrive_expect_tx(bar, bytes * p);
    for (int r = 0; r < p; ++r)
      bulk_load(smem_addr(data + (static_cast<size_t>(st) * p + r) * tile_bytes),
                reinterpret_cast<const T*>(a.rep[r]) + i0, bytes, bar);
  };

  if (threadIdx.x == 0)
    for (int j = 0; j < S && j < my_tiles; ++j) issue_loads(j, j);

  int j = 0;
  for (; j < my_tiles; ++j) {
    const int st = j % S;
    const uint32_t parity = static_cast<uint32_t>(j / S) & 1u;
    if (threadIdx.x == 0) {
      bulk_wait_read(S - 1);  // the stores that last read res[st] are done with it
      if (!mbar_wait_bounded(smem_addr(&bars[st]), parity, a.timeout_ns)) {
        atomicCAS(&g_device_error, 0, kErrBulkWait);
        s_abort = 1;
      }
    }
    __syncthreads();
    if (s_abort) break;
    (void)mbar_try_wait(smem_addr(&bars[st]), parity);  // completed: acquire for this thread

    int c, len;
    int64_t i0;
    tile_at(j, c, i0, len);
    const int o = (c + a.shift) % p;
    const unsigned char* stage = data + static_cast<size_t>(st) * p * tile_bytes;
    unsigned char* out = res + static_cast<size_t>(st) * tile_bytes;
    const int nvec = len / V;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      float acc[V];
      Vec<T>::unpack(*reinterpret_cast<const uint4*>(stage + static_cast<size_t>(o) * tile_bytes + v * 16), acc);
      int r = o;
      for (int q = 1; q < p; ++q) {
        r = (r + 1 == p) ? 0 : r + 1;
        float t[V];
        Vec<T>::unpack(*reinterpret_cast<const uint4*>(stage + static_cast<size_t>(r) * tile_bytes + v * 16), t);
#pragma unroll
        for (int l = 0; l < V; ++l) acc[l] = __fadd_rn(acc[l], t[l]);
      }
#pragma unroll
      for (int l = 0; l < V; ++l) acc[l] = __fdiv_rn(acc[l], a.divisor);
      *reinterpret_cast<uint4*>(out + v * 16) = Vec<T>::pack(acc);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      const uint32_t bytes = static_cast<uint32_t>(len) * sizeof(T);
      if (a.scatter) {
        T* d = reinterpret_cast<T*>(a.out[(o + p - 1) % p]) + (i0 - static_cast<int64_t>(c) * a.cs);
        bulk_store(d, smem_addr(out), bytes);
      } else {
        for (int r = 0; r < p; ++r) bulk_store(reinterpret_cast<T*>(a.rep[r]) + i0, smem_addr(out), bytes);
      }
      bulk_commit();
      if (j + S < my_tiles) issue_loads(j + S, st);
    }
  }

  if (threadIdx.x == 0) {
    bulk_wait_all();
    if (s_abort) {  // let the loads still in flight land before the CTA's shared memory goes away
      for (int k = j + 1; k < my_tiles && k < j + S; ++k)
        (void)mbar_wait_bounded(smem_addr(&bars[k % S]), static_cast<uint32_t>(k / S) & 1u, a.timeout_ns);
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

namespace {
constexpr int kStagedSmemBudget = 220 * 1024;

// Plan the staged kernel; false when its conditions do not hold (more than
// kMaxStagedP replicas, replicas not sharing an alignment, a scatter output
// that is not 16-byte aligned where its chunk's body starts).
template <typename T>
bool plan_staged(const FusedArgs& f, StagedArgs& a) {
  constexpr int V = Vec<T>::N;
  const int p = f.p;
  if (p > kMaxStagedP || !f.same_align) return false;
  const uintptr_t base = reinterpret_cast<uintptr_t>(f.src[0]);
  if (base % sizeof(T) != 0) return false;
  std::memset(&a, 0, sizeof(a));
  int tile_bytes = 16384;
  while (tile_bytes > 512 && static_cast<int64_t>(p + 1) * tile_bytes * 3 > kStagedSmemBudget) tile_bytes /= 2;
  int stages = static_cast<int>(kStagedSmemBudget / (static_cast<int64_t>(p + 1) * tile_bytes));
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return false;
  a.tile_elems = tile_bytes / static_cast<int>(sizeof(T));
  a.stages = stages;
  a.n = f.n; a.cs = f.cs; a.divisor = f.divisor; a.p = p; a.scatter = f.scatter; a.shift = f.shift;
  a.timeout_ns = 2000000000LL;
  int64_t tiles = 0;
  for (int c = 0; c < p; ++c) {
    a.rep[c] = const_cast<void*>(f.src[c]);
    a.out[c] = f.dst[c];
  }
  for (int c = 0; c < p; ++c) {
    const int64_t lo = std::min(f.n, static_cast<int64_t>(c) * f.cs);
    const int64_t hi = std::min(f.n, lo + f.cs);
    const uintptr_t addr = base + static_cast<uintptr_t>(lo) * sizeof(T);
    int64_t head = static_cast<int64_t>(((16u - (addr & 15u)) & 15u) / sizeof(T));
    if (head > hi - lo) head = hi - lo;
    const int64_t body = (hi - lo - head) / V * V;
    a.body_lo[c] = lo + head;
    a.body_len[c] = body;
    if (f.scatter && body > 0) {
      const int owner = ((c + f.shift) % p + p - 1) % p;
      const uintptr_t d = reinterpret_cast<uintptr_t>(f.dst[owner]) + static_cast<uintptr_t>(head) * sizeof(T);
      if (d & 15u) return false;
    }
    a.tile0[c] = static_cast<int32_t>(tiles);
    tiles += (body + a.tile_elems - 1) / a.tile_elems;
    if (tiles > 0x7FFFFFFF) return false;
  }
  a.tile0[p] = static_cast<int32_t>(tiles);
  return true;
}

template <typename T>
cudaError_t fused_staged(const StagedArgs& a, cudaStream_t s) {
  const size_t smem = 128 + static_cast<size_t>(a.stages) * (a.p + 1) * a.tile_elems * sizeof(T);
  static bool configured[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(k_fused_reduce_staged<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kStagedSmemBudget + 1024);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  int grid = sm_count();
  if (a.tile0[a.p] < grid) grid = a.tile0[a.p] > a.p ? a.tile0[a.p] : a.p;
  if (grid < 1) grid = 1;
  k_fused_reduce_staged<T><<<grid, kThreads, smem, s>>>(a);
  count_launch();
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_fused_reduce(const FusedArgs& a, ddp_dtype dt, bool staged, cudaStream_t s) {
  if (staged) {
    StagedArgs sa;
    if (dt == DDP_FLOAT32 ? plan_staged<float>(a, sa) : plan_staged<__nv_bfloat16>(a, sa))
      return dt == DDP_FLOAT32 ? fused_staged<float>(sa, s) : fused_staged<__nv_bfloat16>(sa, s);
  }
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
