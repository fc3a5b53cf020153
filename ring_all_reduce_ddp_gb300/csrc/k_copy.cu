// Copy kernels: ring all-gather steps and doubling-tree broadcast steps (copy
// jobs), the fused all-gather and broadcast (one read, many writes), bucket
// flatten / unflatten (segment copies, optionally dividing), and the coalesced
// broadcast (multi-tensor fan-out).
//
// Sources: "Data parallelism", "Ring all-reduce, derived" (all-gather: the
// receiver overwrites its copy); "Collective Ops From Scratch", code/main.py
// list (doubling-tree broadcast, N-1 rotations for all-gather); "PyTorch DDP
// Deep Dive", Part 2 (mark_variable_ready copies each gradient into its bucket
// slice, pre-dividing; finalize_backward copies back; _broadcast_coalesced
// flattens, broadcasts and unflattens).
//
// Every copy picks the widest word (16, 8, 4, 2 or 1 bytes) on which source
// and destination agree modulo its size, copies the bytes before the first
// boundary and after the last one singly, and the words in between.
#include "bulk.cuh"
#include "launch.h"

namespace ddp {
namespace {

constexpr int kWordsInFlight = 4;
constexpr int64_t kTileBytes = kSegTileBytes;  // = kThreads * 16 bytes * kWordsInFlight
// The one-read, many-write fan-out: with more than kFanFewDst destinations it
// keeps 2 words in flight per thread on 8 KB tiles, otherwise 4 on 16 KB.
// Measured on GB300 (all-gather and broadcast, 1 MiB to 1 GiB): 2 words were
// 2 to 4 % faster from 256 MiB at p = 8 and 64 and far faster at 1-4 MiB,
// but 3 to 10 % slower with 1 to 4 destinations.
constexpr int kFanFewDst = 4;
template <int U> __host__ __device__ constexpr int64_t fan_tile_bytes() { return static_cast<int64_t>(kThreads) * 16 * U; }

template <typename W, int U>
__device__ __forceinline__ void copy_words(const char* s, char* const* d, int nd, int64_t nbytes,
                                           int tid, int nthr) {
  constexpr int64_t w = sizeof(W);
  int64_t head = static_cast<int64_t>((w - (reinterpret_cast<uintptr_t>(s) & (w - 1))) & (w - 1));
  if (head > nbytes) head = nbytes;
  const int64_t nw = (nbytes - head) / w;
  const int64_t tail0 = head + nw * w;
  for (int64_t b = tid; b < head; b += nthr) {
    const char v = s[b];
    for (int q = 0; q < nd; ++q) d[q][b] = v;
  }
  for (int64_t b = tail0 + tid; b < nbytes; b += nthr) {
    const char v = s[b];
    for (int q = 0; q < nd; ++q) d[q][b] = v;
  }
  const W* sw = reinterpret_cast<const W*>(s + head);
  for (int64_t k0 = tid; k0 < nw; k0 += static_cast<int64_t>(nthr) * U) {
    W v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t k = k0 + static_cast<int64_t>(u) * nthr;
      if (k < nw) v[u] = sw[k];
    }
    for (int q = 0; q < nd; ++q) {
      W* dw = reinterpret_cast<W*>(d[q] + head);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t k = k0 + static_cast<int64_t>(u) * nthr;
        if (k < nw) dw[k] = v[u];
      }
    }
  }
}

// Copy nbytes from s to each of the nd destinations d[q] (one read, nd
// writes), U words per thread in flight.
template <int U = kWordsInFlight>
__device__ __forceinline__ void copy_to_all(const char* s, char* const* d, int nd, int64_t nbytes,
                                            int tid, int nthr) {
  uintptr_t x = 0;
  for (int q = 0; q < nd; ++q) x |= reinterpret_cast<uintptr_t>(s) ^ reinterpret_cast<uintptr_t>(d[q]);
  if ((x & 15) == 0) copy_words<uint4, U>(s, d, nd, nbytes, tid, nthr);
  else if ((x & 7) == 0) copy_words<uint2, U>(s, d, nd, nbytes, tid, nthr);
  else if ((x & 3) == 0) copy_words<uint32_t, U>(s, d, nd, nbytes, tid, nthr);
  else if ((x & 1) == 0) copy_words<uint16_t, U>(s, d, nd, nbytes, tid, nthr);
  else copy_words<uint8_t, U>(s, d, nd, nbytes, tid, nthr);
}

// ---------------------------------------------------------------- kernels
__global__ void __launch_bounds__(kThreads) k_pair_copy(const __grid_constant__ PairCopyArgs a) {
  pdl_trigger();
  pdl_wait();
  const int j = blockIdx.y;
  const int64_t nb = a.nbytes[j];
  const int64_t ntiles = (nb + kTileBytes - 1) / kTileBytes;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t b0 = t * kTileBytes;
    const int64_t len = min(kTileBytes, nb - b0);
    char* d = a.dst[j] + b0;
    copy_to_all(a.src[j] + b0, &d, 1, len, threadIdx.x, blockDim.x);
  }
}

template <int U>
__global__ void __launch_bounds__(kThreads) k_fanout(const __grid_constant__ FanoutArgs a) {
  pdl_trigger();
  pdl_wait();
  constexpr int64_t kTile = fan_tile_bytes<U>();
  const int j = blockIdx.y;
  const int64_t ntiles = (a.nbytes + kTile - 1) / kTile;
  __shared__ char* dst[kMaxP];
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t b0 = t * kTile;
    const int64_t len = min(kTile, a.nbytes - b0);
    __syncthreads();
    for (int q = threadIdx.x; q < a.ndst; q += blockDim.x) dst[q] = a.dst[q] + a.job_off[j] + b0;
    __syncthreads();
    copy_to_all<U>(a.src[j] + b0, dst, a.ndst, len, threadIdx.x, blockDim.x);
  }
}

// The fused fan-out with the TMA's bulk copies: each block is one warp with
// one tile of the job's source. Lane 0 loads the tile into shared memory with
// one bulk copy (completing on an mbarrier); then the lanes write it to the
// destinations, one bulk store each, so the copy engine of the SM moves every
// byte and no thread holds data in registers. Every source and destination
// must agree modulo 16 bytes (the host checks); the bytes before the first
// 16-byte boundary of the source and after the last one go singly. The wait
// for the load is bounded: past kBulkFanWaitNs the block records kErrBulkWait,
// waits once more (bounded) and stops. A block waits for its stores to
// complete before it ends.
// 8 KB tiles: measured on GB300 against 16 and 32 KB, broadcast and
// all-gather at 64 MiB per replica, p = 8 / 16 / 64: 0.98 / 1.00 / 1.04 of
// measured HBM against 0.96 / 0.96 / 1.00 (16 KB) and 0.97 / 0.95 / 0.96
// (32 KB); from 256 MiB all three within 1 %.
constexpr int kBulkFanTile = 8192;
constexpr int64_t kBulkFanWaitNs = 2000000000LL;

__global__ void __launch_bounds__(32) k_fanout_bulk(const __grid_constant__ FanoutArgs a) {
  __shared__ __align__(128) unsigned char buf[kBulkFanTile];
  __shared__ __align__(8) uint64_t full;
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x;
  const int j = blockIdx.y;
  const char* src = a.src[j];
  const int64_t nb = a.nbytes;
  const int64_t head = min(nb, static_cast<int64_t>((16u - (reinterpret_cast<uintptr_t>(src) & 15u)) & 15u));
  const int64_t body = (nb - head) & ~static_cast<int64_t>(15);
  if (blockIdx.x == 0) {
    for (int64_t b = lane; b < nb - body; b += 32) {
      const int64_t x = b < head ? b : body + b;
      const char v = src[x];
      for (int q = 0; q < a.ndst; ++q) a.dst[q][a.job_off[j] + x] = v;
    }
  }
  const uint32_t bar = smem_addr(&full);
  if (lane == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  uint32_t phase = 0;
  for (int64_t t0 = static_cast<int64_t>(blockIdx.x) * kBulkFanTile; t0 < body;
       t0 += static_cast<int64_t>(gridDim.x) * kBulkFanTile, phase ^= 1u) {
    const uint32_t len = static_cast<uint32_t>(min(static_cast<int64_t>(kBulkFanTile), body - t0));
    if (lane == 0) {
      mbar_arrive_expect_tx(bar, len);
      bulk_load(smem_addr(buf), src + head + t0, len, bar);
    }
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar, phase, kBulkFanWaitNs))) {
      if (lane == 0 && a.err) atomicCAS(a.err, 0, kErrBulkWait);
      (void)mbar_wait_bounded(bar, phase, kBulkFanWaitNs);  // the load must land before shared memory goes away
      return;
    }
    for (int q = lane; q < a.ndst; q += 32) bulk_store(a.dst[q] + a.job_off[j] + head + t0, smem_addr(buf), len);
    bulk_commit();
    bulk_wait_read(0);  // the tile has been read out before the next load overwrites it
    __syncwarp();
  }
  bulk_wait_all();  // this lane's stores are complete
}

__device__ __forceinline__ int find_tile_owner(const int32_t* tile0, int nseg, int32_t b) {
  int lo = 0, hi = nseg;  // tile0[lo] <= b < tile0[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile0[mid] <= b) lo = mid; else hi = mid;
  }
  return lo;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) k_seg_copy(const __grid_constant__ SegCopyArgs a) {
  pdl_trigger();
  pdl_wait();
  const int32_t b = blockIdx.x;
  const int s = find_tile_owner(a.tile0, a.nseg, b);
  const int64_t b0 = static_cast<int64_t>(b - a.tile0[s]) * kSegTileBytes;
  const int64_t len = min(static_cast<int64_t>(kSegTileBytes), a.bytes[s] - b0);
  if (len <= 0) return;
  const char* src = a.src[s] + b0;
  char* dst = a.dst[s] + b0;
  if (a.predivide == 1.0f) {
    copy_to_all(src, &dst, 1, len, threadIdx.x, blockDim.x);
  } else {
    const T* xs = reinterpret_cast<const T*>(src);
    T* xd = reinterpret_cast<T*>(dst);
    const int64_t ne = len / static_cast<int64_t>(sizeof(T));
    for (int64_t e = threadIdx.x; e < ne; e += blockDim.x)
      xd[e] = narrow<T>(__fdiv_rn(widen(xs[e]), a.predivide));
  }
}

__global__ void __launch_bounds__(kThreads) k_multi_fanout(const __grid_constant__ MultiFanoutArgs a) {
  // a programmatic dependent (the Reducer's sync) may start its prologue now;
  // it still waits for this grid to finish before it touches memory
  asm volatile("griddepcontrol.launch_dependents;");
  const int32_t b = blockIdx.x;
  const int t = find_tile_owner(a.tile0, a.ntensors, b);
  const int64_t b0 = static_cast<int64_t>(b - a.tile0[t]) * kTileBytes;
  const int64_t len = min(kTileBytes, a.bytes[t] - b0);
  if (len <= 0) return;
  __shared__ char* dst[kMaxP];  // ndst <= p - 1
  for (int q = threadIdx.x; q < a.ndst; q += blockDim.x) dst[q] = a.dst[t * a.ndst + q] + b0;
  __syncthreads();
  copy_to_all(a.src[t] + b0, dst, a.ndst, len, threadIdx.x, blockDim.x);
}

// One job per blockIdx.y. Eight elements per thread and step (16 bytes of
// bf16, 32 of fp32) when the bf16 side is 16-byte aligned and the fp32 side
// 32-byte aligned; the rest element by element.
__global__ void __launch_bounds__(kThreads) k_convert(const __grid_constant__ ConvertArgs a) {
  pdl_trigger();
  pdl_wait();
  const int j = blockIdx.y;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const uintptr_t bf = reinterpret_cast<uintptr_t>(a.to_bf16 ? a.dst[j] : a.src[j]);
  const uintptr_t f32 = reinterpret_cast<uintptr_t>(a.to_bf16 ? a.src[j] : a.dst[j]);
  const int64_t nv = (bf % 16 == 0 && f32 % 32 == 0) ? a.n / 8 : 0;
  if (a.to_bf16) {
    const float4* s = static_cast<const float4*>(a.src[j]);
    uint4* d = static_cast<uint4*>(a.dst[j]);
    for (int64_t v = tid; v < nv; v += stride) {
      const float4 x = s[2 * v], y = s[2 * v + 1];
      const float f[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
      d[v] = Vec<__nv_bfloat16>::pack(f);
    }
    const float* ss = static_cast<const float*>(a.src[j]);
    __nv_bfloat16* dd = static_cast<__nv_bfloat16*>(a.dst[j]);
    for (int64_t i = nv * 8 + tid; i < a.n; i += stride) dd[i] = narrow<__nv_bfloat16>(ss[i]);
  } else {
    const uint4* s = static_cast<const uint4*>(a.src[j]);
    float4* d = static_cast<float4*>(a.dst[j]);
    for (int64_t v = tid; v < nv; v += stride) {
      float f[8];
      Vec<__nv_bfloat16>::unpack(s[v], f);
      d[2 * v] = make_float4(f[0], f[1], f[2], f[3]);
      d[2 * v + 1] = make_float4(f[4], f[5], f[6], f[7]);
    }
    const __nv_bfloat16* ss = static_cast<const __nv_bfloat16*>(a.src[j]);
    float* dd = static_cast<float*>(a.dst[j]);
    for (int64_t i = nv * 8 + tid; i < a.n; i += stride) dd[i] = widen(ss[i]);
  }
}

// One block per tile of each row, no striding: blocks are dispatched in index
// order, so the resident ones sweep one contiguous window of the source and of
// every destination. Measured on GB300 (fused all-gather and broadcast, p = 8,
// 64 MiB-1 GiB per replica): 0.88-0.92 of measured HBM peak with a striding
// grid of 8 blocks per SM, 0.97-0.98 this way; at p = 2 and 64, 1.01-1.05.
int grid_x_for(int64_t tiles) {
  int64_t bx = tiles;
  if (bx < 1) bx = 1;
  if (bx > (int64_t(1) << 30)) bx = int64_t(1) << 30;  // the kernels stride past this
  return static_cast<int>(bx);
}

}  // namespace

cudaError_t launch_pair_copy(const PairCopyArgs& a, cudaStream_t s) {
  if (a.njobs <= 0) return cudaSuccess;
  int64_t maxb = 0;
  for (int j = 0; j < a.njobs; ++j) maxb = a.nbytes[j] > maxb ? a.nbytes[j] : maxb;
  if (maxb == 0) return cudaSuccess;
  const dim3 grid(grid_x_for((maxb + kTileBytes - 1) / kTileBytes), a.njobs);
  const cudaError_t e = launch_pdl(k_pair_copy, grid, dim3(kThreads), 0, s, a);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Every job's source and every destination of it agree modulo 16 bytes.
bool fanout_aligned(const FanoutArgs& a) {
  for (int j = 0; j < a.njobs; ++j)
    for (int q = 0; q < a.ndst; ++q)
      if (((reinterpret_cast<uintptr_t>(a.dst[q]) + static_cast<uintptr_t>(a.job_off[j])) ^
           reinterpret_cast<uintptr_t>(a.src[j])) & 15u)
        return false;
  return true;
}

// Which fan-out DDP_ALGO_FUSED takes: the bulk-copy form with 7 or more
// destinations once the job reads 64 MiB or more in all, where it measured
// faster on GB300 (broadcast / all-gather, fraction of measured HBM, bulk
// against registers: p = 8 at 256 MiB 1.002 / 1.002 against 0.991 / 0.989,
// at 1 GiB 1.004 / 1.003 against 0.997 / 0.994; p = 16 at 64 MiB 1.003 /
// 1.007 against 0.980 / 0.979, at 256 MiB 1.016 / 1.016 against 0.978 /
// 0.982; p = 64 at 64 MiB 1.037 / 1.036 against 1.012 / 1.012, at 256 MiB
// 1.061 / 1.054 against 1.025 / 1.013). With fewer destinations, or below
// 64 MiB where its grid holds too few blocks, the register form was faster
// (p = 2 at 1 GiB: 1.034 against 1.046; p = 8 at 16 MiB with 16 KB tiles:
// 0.73 against 0.91).
bool fanout_bulk_by_default(const FanoutArgs& a) {
  return a.ndst >= 7 && static_cast<int64_t>(a.njobs) * a.nbytes >= (int64_t(64) << 20);
}

cudaError_t launch_fanout(const FanoutArgs& a, cudaStream_t s, ddp_algo algo) {
  if (a.njobs <= 0 || a.nbytes <= 0 || a.ndst <= 0) return cudaSuccess;
  cudaError_t e;
  const bool bulk = algo == DDP_ALGO_FUSED_TMA || (algo == DDP_ALGO_FUSED && fanout_bulk_by_default(a));
  if (bulk && fanout_aligned(a)) {
    FanoutArgs b = a;
    b.err = device_error_word();
    e = launch_pdl(k_fanout_bulk, dim3(grid_x_for((a.nbytes + kBulkFanTile - 1) / kBulkFanTile), a.njobs),
                   dim3(32), 0, s, b);
  } else if (a.ndst <= kFanFewDst) {
    constexpr int64_t t = fan_tile_bytes<4>();
    e = launch_pdl(k_fanout<4>, dim3(grid_x_for((a.nbytes + t - 1) / t), a.njobs), dim3(kThreads), 0, s, a);
  } else {
    constexpr int64_t t = fan_tile_bytes<2>();
    e = launch_pdl(k_fanout<2>, dim3(grid_x_for((a.nbytes + t - 1) / t), a.njobs), dim3(kThreads), 0, s, a);
  }
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_seg_copy(const SegCopyArgs& a, ddp_dtype dt, cudaStream_t s) {
  const int32_t ntiles = a.tile0[a.nseg];
  if (a.nseg <= 0 || ntiles <= 0) return cudaSuccess;
  const cudaError_t e = dt == DDP_BFLOAT16
                            ? launch_pdl(k_seg_copy<__nv_bfloat16>, dim3(ntiles), dim3(kThreads), 0, s, a)
                            : launch_pdl(k_seg_copy<float>, dim3(ntiles), dim3(kThreads), 0, s, a);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_convert(const ConvertArgs& a, cudaStream_t s) {
  if (a.njobs <= 0 || a.n <= 0) return cudaSuccess;
  const dim3 grid(grid_x_for((a.n + 8 * kThreads - 1) / (8 * kThreads)), a.njobs);
  const cudaError_t e = launch_pdl(k_convert, grid, dim3(kThreads), 0, s, a);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_multi_fanout(const MultiFanoutArgs& a, cudaStream_t s) {
  const int32_t ntiles = a.tile0[a.ntensors];
  if (a.ntensors <= 0 || ntiles <= 0 || a.ndst <= 0) return cudaSuccess;
  k_multi_fanout<<<ntiles, kThreads, 0, s>>>(a);
  count_launch();
  return cudaGetLastError();
}

}  // namespace ddp
