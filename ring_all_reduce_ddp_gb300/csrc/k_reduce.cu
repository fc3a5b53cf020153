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

#include "bulk.cuh"
#include "launch.h"

namespace ddp {

__device__ int g_device_error = 0;

// ------------------------------------------------ fused, register-only path
// Blocks of 128 threads, one 16-byte vector per thread and replica (U = 1).
// Measured on GB300 against 256-thread blocks, flat fp32 all-reduce, CUDA
// graph of launches after an L2 flush: 1 MiB per replica 0.239 -> 0.249 of
// measured HBM at p = 2, 0.49 -> 0.51 at p = 8, 0.655 -> 0.70 at p = 64;
// from 64 MiB within 0.002 either way (p = 8, 1 GiB: 1.036 both).
constexpr int kFusedThreads = 128;

// Vectors per thread (U): with few replicas a vector needs few loads, so on
// large chunks a thread may take two vectors to keep more 16-byte loads in
// flight. Measured on GB300, flat fp32, CUDA graph of launches after an L2
// flush, fraction of measured HBM at 16 / 25 / 64 / 256 MiB:
//   all-reduce p = 2, U = 2: 0.867 / 0.917 / 0.988 / 1.035; U = 4: 0.844 /
//     0.904 / 0.981 / 1.029; U = 1: 0.724 / 0.772 / 0.818 / 0.845;
//   all-reduce p = 4, U = 1: 0.935 / 0.974 / 1.014 / 1.036; U = 2: 0.935 /
//     0.968 / 1.012 / 1.031;
//   reduce-scatter p = 2, U = 2: 0.819 / 0.902 / 1.007 / 1.068; U = 4: 0.801
//     / 0.888 / 0.990 / 1.047;
//   reduce-scatter p = 4, U = 2: 0.918 / 0.975 / 1.050 / 1.073; U = 1: 0.834
//     / 0.887 / 0.941 / 0.990 (it writes one output per p inputs, so its
//     stores do not keep the memory system busy the way p stores do).
// So U = 2 for p = 2, and for the reduce-scatter at p = 4; U = 1 otherwise.
constexpr int ldst_unroll(int p, bool scatter) { return (p == 2 || (p == 4 && scatter)) ? 2 : 1; }

// Vectors per thread of the one-shot staged kernel's window, as measured
// with it (a 16 KB staging buffer per block at p = 2 and 4).
template <int P>
__host__ __device__ constexpr int oneshot_unroll() { return P == 2 ? 4 : P == 4 ? 2 : 1; }

template <typename T, int P, bool HOP = false, int U = 1>
__global__ void __launch_bounds__(kFusedThreads) k_fused_reduce_ldst(const __grid_constant__ FusedArgs a) {
  pdl_trigger();
  pdl_wait();
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
    for (int j = 1; j < p; ++j) {
      acc = __fadd_rn(acc, widen(src[j][i]));
      if constexpr (HOP) acc = round_bf16(acc);
    }
    const T y = narrow<T>(__fdiv_rn(acc, a.divisor));
    if (a.scatter) {
      sdst[i - lo] = y;
    } else {
      for (int r = 0; r < p; ++r) reinterpret_cast<T*>(a.dst[r])[i] = y;
    }
  }

  if constexpr (P > 0 && U > 1) {
    // block b takes vectors [b * U * blockDim, (b + 1) * U * blockDim) of the chunk;
    // all U * P loads are issued before the first fold
    const int64_t bstride = static_cast<int64_t>(gridDim.x) * blockDim.x * U;
    for (int64_t v0 = static_cast<int64_t>(blockIdx.x) * blockDim.x * U + threadIdx.x; v0 < nvec; v0 += bstride) {
      uint4 x[U][P];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t v = v0 + static_cast<int64_t>(u) * blockDim.x;
        if (v < nvec) {
#pragma unroll
          for (int j = 0; j < P; ++j) x[u][j] = *reinterpret_cast<const uint4*>(src[j] + lo + head + v * V);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t v = v0 + static_cast<int64_t>(u) * blockDim.x;
        if (v >= nvec) continue;
        const int64_t i = lo + head + v * V;
        float acc[V];
        Vec<T>::unpack(x[u][0], acc);
#pragma unroll
        for (int j = 1; j < P; ++j) {
          float t[V];
          Vec<T>::unpack(x[u][j], t);
#pragma unroll
          for (int l = 0; l < V; ++l) {
            acc[l] = __fadd_rn(acc[l], t[l]);
            if constexpr (HOP) acc[l] = round_bf16(acc[l]);
          }
        }
#pragma unroll
        for (int l = 0; l < V; ++l) acc[l] = __fdiv_rn(acc[l], a.divisor);
        const uint4 y = Vec<T>::pack(acc);
        if (a.scatter) {
          *reinterpret_cast<uint4*>(sdst + (i - lo)) = y;
        } else {
#pragma unroll
          for (int r = 0; r < P; ++r) *reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.dst[r]) + i) = y;
        }
      }
    }
    return;
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
        for (int l = 0; l < V; ++l) {
          acc[l] = __fadd_rn(acc[l], t[l]);
          if constexpr (HOP) acc[l] = round_bf16(acc[l]);
        }
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
              for (int l = 0; l < V; ++l) {
                acc[l] = __fadd_rn(acc[l], t[l]);
                if constexpr (HOP) acc[l] = round_bf16(acc[l]);
              }
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


// ------------------------------- fused, one-shot staging through shared memory
// The register kernel's grid (one block of 128 threads per window of 128 * U
// vectors of a chunk, in index order), with the loads staged: lane j of warp
// 0 issues one bulk asynchronous copy (cp.async.bulk) of replica j's window,
// all P completing on one mbarrier; each thread then folds its U vectors from
// shared memory in ring order and stores with 128-bit stores. No pipeline and
// no hand-off between warps: the many resident blocks keep the copies in
// flight. A block loops over further windows only when the grid had to be
// capped. Every wait is bounded; the block decides together (a barrier vote)
// whether its copies landed, and on a timeout records kErrBulkWait, waits
// once more (bounded) for the copies and stops.
constexpr int64_t kBulkWaitNs = 2000000000LL;  // bound of every wait on a bulk copy

template <typename T, int P>
__global__ void __launch_bounds__(kFusedThreads) k_fused_reduce_oneshot(const __grid_constant__ FusedArgs a) {
  constexpr int U = oneshot_unroll<P>();
  constexpr int W = kFusedThreads * U;  // vectors per window
  constexpr int V = Vec<T>::N;
  __shared__ __align__(128) uint4 stage[P][W];
  __shared__ __align__(8) uint64_t full;
  __shared__ T* dst[P];
  pdl_trigger();
  pdl_wait();
  const int c = blockIdx.y;
  const int64_t lo = static_cast<int64_t>(c) * a.cs;
  const int64_t hi = min(a.n, lo + a.cs);
  if (lo >= hi) return;
  const int o = (c + a.shift) % P;
  const int owner = (o + P - 1) % P;
  const T* const* src = reinterpret_cast<const T* const*>(&a.src[o]);
  T* sdst = a.scatter ? reinterpret_cast<T*>(a.dst[owner]) : nullptr;
  const int64_t len = hi - lo;
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
  // The few elements outside the aligned body, one loaded value at a time
  // (not unrolled: P values in flight here would set the register count of
  // the whole kernel, 80 instead of 44 at p = 16).
  for (int64_t e = gtid; e < nscalar; e += gstride) {
    const int64_t i = lo + (e < head ? e : tail0 + (e - head));
    float acc = widen(src[0][i]);
#pragma unroll 1
    for (int j = 1; j < P; ++j) acc = __fadd_rn(acc, widen(src[j][i]));
    const T y = narrow<T>(__fdiv_rn(acc, a.divisor));
    if (a.scatter) {
      sdst[i - lo] = y;
    } else {
#pragma unroll 1
      for (int r = 0; r < P; ++r) reinterpret_cast<T*>(a.dst[r])[i] = y;
    }
  }
  int64_t v0 = static_cast<int64_t>(blockIdx.x) * W;
  if (v0 >= nvec) return;
  const uint32_t bar = smem_addr(&full);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  // the destinations in shared memory, read as each store needs them, rather
  // than P pointers held in registers across the loop
  if (threadIdx.x < P) dst[threadIdx.x] = reinterpret_cast<T*>(a.dst[threadIdx.x]);
  __syncthreads();
  for (uint32_t phase = 0; v0 < nvec; v0 += static_cast<int64_t>(gridDim.x) * W, phase ^= 1u) {
    const int cnt = static_cast<int>(min(static_cast<int64_t>(W), nvec - v0));
    if (threadIdx.x < 32) {
      const uint32_t bytes = static_cast<uint32_t>(cnt) * 16u;
      if (threadIdx.x == 0) mbar_arrive_expect_tx(bar, bytes * P);
      __syncwarp();
      if (static_cast<int>(threadIdx.x) < P)
        bulk_load(smem_addr(stage[threadIdx.x]), src[threadIdx.x] + lo + head + v0 * V, bytes, bar);
    }
    const bool landed = mbar_wait_bounded(bar, phase, kBulkWaitNs);
    if (!__syncthreads_and(landed)) {
      if (threadIdx.x == 0) atomicCAS(&g_device_error, 0, kErrBulkWait);
      (void)mbar_wait_bounded(bar, phase, kBulkWaitNs);  // the copies must land before shared memory goes away
      return;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = threadIdx.x + u * kFusedThreads;
      if (v >= cnt) break;
      float acc[V];
      Vec<T>::unpack(stage[0][v], acc);
#pragma unroll 1
      for (int j = 1; j < P; ++j) {  // one staged vector at a time: shared memory is close, registers are not free
        float t[V];
        Vec<T>::unpack(stage[j][v], t);
#pragma unroll
        for (int l = 0; l < V; ++l) acc[l] = __fadd_rn(acc[l], t[l]);
      }
#pragma unroll
      for (int l = 0; l < V; ++l) acc[l] = __fdiv_rn(acc[l], a.divisor);
      const uint4 y = Vec<T>::pack(acc);
      const int64_t i = lo + head + (v0 + v) * V;
      if (a.scatter) {
        *reinterpret_cast<uint4*>(sdst + (i - lo)) = y;
      } else {
#pragma unroll
        for (int r = 0; r < P; ++r) *reinterpret_cast<uint4*>(dst[r] + i) = y;
      }
    }
    __syncthreads();  // every thread is done with this window before the next one's copies land
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
  pdl_trigger();
  pdl_wait();
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
  auto one = [&](int64_t e) {
    float y = __fadd_rn(xd[e], xs[e]);
    if (a.last) y = __fdiv_rn(y, a.divisor);
    xd[e] = y;
  };
  // 16-byte vectors where both replicas sit at the same address mod 16
  int64_t head = len;
  const uintptr_t ad = reinterpret_cast<uintptr_t>(xd), as = reinterpret_cast<uintptr_t>(xs);
  if (((ad ^ as) & 15u) == 0 && (ad & 3u) == 0) head = min(static_cast<int64_t>(((16u - (ad & 15u)) & 15u) / 4), len);
  const int64_t nvec = (len - head) / 4;
  const int64_t tail0 = head + nvec * 4;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t gstride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = gtid; e < head; e += gstride) one(e);
  for (int64_t e = tail0 + gtid; e < len; e += gstride) one(e);
  const float4* s4 = reinterpret_cast<const float4*>(xs + head);
  float4* d4 = reinterpret_cast<float4*>(xd + head);
  for (int64_t v0 = gtid; v0 < nvec; v0 += gstride * kU) {
    float4 loc[kU], rcv[kU];
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      const int64_t v = v0 + q * gstride;
      if (v < nvec) { loc[q] = d4[v]; rcv[q] = s4[v]; }
    }
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      const int64_t v = v0 + q * gstride;
      if (v < nvec) {
        float4 y;
        y.x = __fadd_rn(loc[q].x, rcv[q].x);
        y.y = __fadd_rn(loc[q].y, rcv[q].y);
        y.z = __fadd_rn(loc[q].z, rcv[q].z);
        y.w = __fadd_rn(loc[q].w, rcv[q].w);
        if (a.last) {
          y.x = __fdiv_rn(y.x, a.divisor);
          y.y = __fdiv_rn(y.y, a.divisor);
          y.z = __fdiv_rn(y.z, a.divisor);
          y.w = __fdiv_rn(y.w, a.divisor);
        }
        d4[v] = y;
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
  pdl_trigger();
  pdl_wait();
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
        float v = __fadd_rn(part[q], loc[q]);
        if (a.hop_round) v = round_bf16(v);
        if (a.last) od[e] = narrow<T>(__fdiv_rn(v, a.divisor));
        else wcur[e] = v;
      }
    }
  }
}


// ------------------------------------------- persistent literal ring (fp32)
// The literal 2(p-1)-step schedule in one cooperative launch ("Collective Ops
// From Scratch", "Ring allreduce in two passes": each rank receives one chunk
// per step from its left neighbour; its exercise of a configurable receive
// timeout that surfaces a deadline error). Receiver d at step t needs the
// chunk its sender d-1 finished at step t-1, so it waits until the sender has
// posted t steps; every other ordering follows from that chain. Waits are
// bounded by %globaltimer; a wait that runs out records where it gave up and
// the block stops, so its own successors time out after it and the kernel
// ends. Data of other ranks is read through L2 (ld.global.cg): L1 is not
// coherent across SMs.
//
// Each (rank, slice) flag has a 128-byte line of its own (kFlagStride ints):
// with flags packed side by side, every posting store contended with the many
// receivers polling the same line, which doubled the time per step at 1-4 MiB
// buffers on GB300. A step is posted by bar.sync followed by one thread's
// st.release.gpu: the release is cumulative over the block's writes ordered
// before it by the barrier, so no separate fence is needed (an extra
// fence.acq_rel cost 7-12 % of the step time).

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__global__ void __launch_bounds__(kThreads) k_ring_persistent_f32(const __grid_constant__ PersistArgs a) {
  const int B = a.blocks_per_rank, p = a.p;
  const int r = blockIdx.x / B, b = blockIdx.x % B;
  const int snd = (r + p - 1) % p;  // this rank's left neighbour
  const int T = 2 * (p - 1);
  float* mine = reinterpret_cast<float*>(a.buf[r]);
  const float* theirs = reinterpret_cast<const float*>(a.buf[snd]);
  __shared__ int s_ok;
  // Bounded wait until the sender has posted `need` steps; on a timeout record
  // (rank, need) and return false.
  auto wait_sender = [&](int need) -> bool {
    if (threadIdx.x == 0) {
      const int* f = a.flags + (snd * B + b) * kFlagStride;
      int ok = 1;
      if (ld_acquire_gpu(f) < need) {
        const uint64_t t0 = global_ns();
        while (ld_acquire_gpu(f) < need) {
          if (static_cast<int64_t>(global_ns() - t0) > a.timeout_ns) {
            ok = 0;
            break;
          }
          __nanosleep(256);
        }
      }
      if (!ok) {
        if (a.status) {
          if (atomicCAS(&a.status[0], 0, static_cast<int>(DDP_ERR_TIMEOUT)) == 0) {
            a.status[1] = r;
            a.status[2] = need;
          }
          atomicAdd(&a.status[3], 1);
        }
        atomicCAS(&g_device_error, 0, kErrRingWait);
      }
      s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
  };
  for (int t = 0; t < T; ++t) {
    if (r == a.fault_rank && t == a.fault_step) return;  // injected fault: never posts step t
    if (t > 0 && !wait_sender(t)) return;
    const bool rs = t < p - 1;
    const int c = rs ? ((snd - t) % p + p) % p : ((snd + 1 - (t - (p - 1))) % p + p) % p;
    const int64_t lo = min(a.n, static_cast<int64_t>(c) * a.cs);
    const int64_t hi = min(a.n, lo + a.cs);
    const int64_t span = (hi - lo + B - 1) / B;
    const int64_t x0 = min(hi, lo + static_cast<int64_t>(b) * span);
    const int64_t x1 = min(hi, x0 + span);
    const bool last_rs = (t == p - 2);
    auto one = [&](int64_t i) {
      const float recv = __ldcg(theirs + i);
      if (rs) {
        float y = __fadd_rn(mine[i], recv);
        if (last_rs) y = __fdiv_rn(y, a.divisor);
        mine[i] = y;
      } else {
        mine[i] = recv;
      }
    };
    // 16-byte vectors where both replicas sit at the same address mod 16
    int64_t head = x1 - x0;
    const uintptr_t am = reinterpret_cast<uintptr_t>(mine + x0), at = reinterpret_cast<uintptr_t>(theirs + x0);
    if (((am ^ at) & 15u) == 0 && (am & 3u) == 0)
      head = min(static_cast<int64_t>(((16u - (am & 15u)) & 15u) / 4), x1 - x0);
    const int64_t nvec = (x1 - x0 - head) / 4;
    const int64_t tail0 = x0 + head + nvec * 4;
    for (int64_t e = threadIdx.x; e < head; e += blockDim.x) one(x0 + e);
    for (int64_t i = tail0 + threadIdx.x; i < x1; i += blockDim.x) one(i);
    float4* m4 = reinterpret_cast<float4*>(mine + x0 + head);
    const float4* t4 = reinterpret_cast<const float4*>(theirs + x0 + head);
    for (int64_t v = threadIdx.x; v < nvec; v += blockDim.x) {
      const float4 rcv = __ldcg(t4 + v);
      if (rs) {
        float4 y = m4[v];
        y.x = __fadd_rn(y.x, rcv.x);
        y.y = __fadd_rn(y.y, rcv.y);
        y.z = __fadd_rn(y.z, rcv.z);
        y.w = __fadd_rn(y.w, rcv.w);
        if (last_rs) {
          y.x = __fdiv_rn(y.x, a.divisor);
          y.y = __fdiv_rn(y.y, a.divisor);
          y.z = __fdiv_rn(y.z, a.divisor);
          y.w = __fdiv_rn(y.w, a.divisor);
        }
        m4[v] = y;
      } else {
        m4[v] = rcv;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) st_release_gpu(a.flags + (r * B + b) * kFlagStride, t + 1);
  }
  // The sender's last step is read by no later step: wait for it too, so a
  // rank that stops before its final step is still caught.
  (void)wait_sender(T);
}

// ------------------------------------------------------------- launchers
namespace {
std::atomic<int64_t> g_launches{0};
std::atomic<int> g_sm_count[64];  // zero-initialised (static storage)

int blocks_per_chunk(int64_t work_items, int per_block, int chunks) {
  const int64_t target = static_cast<int64_t>(sm_count()) * (2048 / kThreads);
  int64_t bx = (target + chunks - 1) / chunks;
  const int64_t need = (work_items + per_block - 1) / per_block;
  if (bx > need) bx = need;
  if (bx < 1) bx = 1;
  if (bx > 65535 * 32) bx = 65535 * 32;
  return static_cast<int>(bx);
}

// One block per kFusedThreads * U vectors of a chunk, no striding: blocks are
// dispatched in index order, so the resident ones sweep one contiguous window
// of each replica, chunk after chunk. Measured on GB300, flat fp32 buffers of
// 256 MiB-1 GiB per replica: 0.94-0.95 of measured HBM peak at p = 8 and 0.94
// at p = 2 with a striding grid of 8 blocks per SM, 1.02-1.04 this way.
int fused_blocks_per_chunk(int64_t vectors, int per_block) {
  int64_t bx = (vectors + per_block - 1) / per_block;
  if (bx < 1) bx = 1;
  if (bx > (int64_t(1) << 30)) bx = int64_t(1) << 30;  // the kernel strides past this
  return static_cast<int>(bx);
}

// The unrolled form only while its grid still holds 8 blocks (of 128 threads)
// per SM: on small chunks, more blocks beat more loads per thread.
template <typename T, int P, bool HOP>
cudaError_t launch_ldst(const FusedArgs& a, cudaStream_t s) {
  constexpr int V = Vec<T>::N;
  const int64_t vectors = a.cs / V + 1;
  if constexpr (P == 2 || P == 4) {
    if (ldst_unroll(P, a.scatter != 0) == 2) {
      const int bx = fused_blocks_per_chunk(vectors, kFusedThreads * 2);
      if (static_cast<int64_t>(bx) * a.p >= 8 * static_cast<int64_t>(sm_count()))
        return launch_pdl(k_fused_reduce_ldst<T, P, HOP, 2>, dim3(bx, a.p), dim3(kFusedThreads), 0, s, a);
    }
  }
  return launch_pdl(k_fused_reduce_ldst<T, P, HOP, 1>, dim3(fused_blocks_per_chunk(vectors, kFusedThreads), a.p),
                    dim3(kFusedThreads), 0, s, a);
}

template <typename T, bool HOP>
cudaError_t fused_ldst(const FusedArgs& a, cudaStream_t s) {
  cudaError_t e;
  switch (a.p) {
    case 2: e = launch_ldst<T, 2, HOP>(a, s); break;
    case 4: e = launch_ldst<T, 4, HOP>(a, s); break;
    case 8: e = launch_ldst<T, 8, HOP>(a, s); break;
    case 16: e = launch_ldst<T, 16, HOP>(a, s); break;
    default: e = launch_ldst<T, 0, HOP>(a, s); break;
  }
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}
}  // namespace

int sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  int c = g_sm_count[dev].load(std::memory_order_relaxed);
  if (c == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
    g_sm_count[dev].store(v, std::memory_order_relaxed);
    c = v;
  }
  return c;
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
int64_t launches() { return g_launches.load(std::memory_order_relaxed); }

namespace {
// No shared-memory carveout preference is set: measured on GB300, setting
// it to the maximum changed no time (64 MiB at p = 8: 156.1-156.8 us either
// way), so a first call may also be made inside a stream capture.
template <typename T, int P>
cudaError_t launch_oneshot(const FusedArgs& a, cudaStream_t s) {
  constexpr int V = Vec<T>::N;
  constexpr int W = kFusedThreads * oneshot_unroll<P>();
  const cudaError_t e = launch_pdl(k_fused_reduce_oneshot<T, P>,
                                   dim3(fused_blocks_per_chunk(a.cs / V + 1, W), a.p), dim3(kFusedThreads), 0, s, a);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

// The one-shot staged kernel for p = 2, 4, 8 and 16 with every replica at
// the same address mod 16; false when it does not apply.
template <typename T>
bool oneshot(const FusedArgs& a, cudaStream_t s, cudaError_t* e) {
  if (!a.same_align || a.hop_round) return false;
  switch (a.p) {
    case 2: *e = launch_oneshot<T, 2>(a, s); return true;
    case 4: *e = launch_oneshot<T, 4>(a, s); return true;
    case 8: *e = launch_oneshot<T, 8>(a, s); return true;
    case 16: *e = launch_oneshot<T, 16>(a, s); return true;
    default: return false;
  }
}
}  // namespace

cudaError_t launch_fused_reduce(const FusedArgs& a, ddp_dtype dt, bool staged, cudaStream_t s) {
  if (staged) {
    cudaError_t e = cudaSuccess;
    if (dt == DDP_FLOAT32 ? oneshot<float>(a, s, &e) : oneshot<__nv_bfloat16>(a, s, &e)) return e;
  }
  if (dt == DDP_FLOAT32) return fused_ldst<float, false>(a, s);
  return a.hop_round ? fused_ldst<__nv_bfloat16, true>(a, s) : fused_ldst<__nv_bfloat16, false>(a, s);
}

cudaError_t launch_rs_step_inplace_f32(const RingStepArgs& a, cudaStream_t s) {
  const dim3 grid(blocks_per_chunk(a.cs / 4 + 1, kThreads * kU, a.p), a.p);
  const cudaError_t e = launch_pdl(k_rs_step_inplace_f32, grid, dim3(kThreads), 0, s, a);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_rs_step_ws(const RingStepArgs& a, ddp_dtype dt, cudaStream_t s) {
  const dim3 grid(blocks_per_chunk(a.cs, kThreads * kU, a.p), a.p);
  const cudaError_t e = dt == DDP_FLOAT32 ? launch_pdl(k_rs_step_ws<float>, grid, dim3(kThreads), 0, s, a)
                                          : launch_pdl(k_rs_step_ws<__nv_bfloat16>, grid, dim3(kThreads), 0, s, a);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

int ring_persistent_max_blocks() {
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k_ring_persistent_f32, kThreads, 0) != cudaSuccess)
    return 0;
  return blocks * sm_count();
}

cudaError_t launch_ring_persistent(const PersistArgs& a, cudaStream_t s) {
  void* args[] = {const_cast<PersistArgs*>(&a)};
  const cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(k_ring_persistent_f32),
                                                    dim3(a.p * a.blocks_per_rank), dim3(kThreads), args, 0, s);
  count_launch();
  return e;
}

int* device_error_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_error) == cudaSuccess) return static_cast<int*>(p);
  (void)cudaGetLastError();  // leave no error behind for a later launch check to misreport
  return nullptr;
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
