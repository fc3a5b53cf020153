// Bucket all-reduce straight on the gradient tensors: what DDP's Reducer does
// as copy-into-bucket, ring all-reduce of the bucket and copy-back
// ("PyTorch DDP Deep Dive", Part 2, mark_variable_ready and
// finalize_backward; "Collective Ops From Scratch", "Ring allreduce in two
// passes"), done in one pass that reads each replica's gradients once and
// writes the result once.
//
// The bucket's flat layout exists only as index arithmetic: element e of the
// tensor in slot s sits at bucket position offset_s + e, which belongs to
// chunk c = position / ceil(n/p) and is therefore summed starting at rank c,
// ((x_c + x_{c+1}) + ...) + x_{c+p-1}, then divided once by the divisor: the
// same bits as the ring on the flat bucket. Work is cut into pieces (a tensor
// intersected with a chunk: one origin each) and pieces into tiles of
// bucket_tile_elems elements per replica; one block per tile.
//
// A Reducer's table may end with copy pieces, one per attached buffer: the
// per-forward buffer broadcast ("PyTorch DDP Deep Dive", Part 2,
// _sync_buffers -> _broadcast_coalesced) rides in the same launch as the
// gradient sync (ddp_reducer_step).
//
// The whole-Reducer table kernel comes in two forms with the same bits: the
// register fold (k_bucket_allreduce_table) and a form that stages each tile
// in shared memory by bulk copies (k_bucket_table_staged); staged_by_default
// says which one DDP_ALGO_FUSED and the step take. A single bucket's launch
// (k_bucket_allreduce, table by value) always folds in registers.
#include <algorithm>

#include "bulk.cuh"
#include "launch.h"

namespace ddp {
namespace {

// A replica's 16 bytes, with a hint that L2 fetch the surrounding 256-byte
// block from DRAM. Measured on GB300, back to back: plain loads take 249.7 us
// against 244.8 us on the ResNet-50-shaped sync and 5,781 against 5,520 us on
// the bf16 Llama-1B one. (With the earlier persistent-grid form of this kernel
// the hint gained 0.4 %, and L1::no_allocate or an L2 evict-first policy
// instead cost 3 %.)
__device__ __forceinline__ uint4 ld_prefetch256(const void* p) {
  uint4 v;
  asm volatile("ld.global.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

struct View {
  void* const* ptr;
  const int64_t* start;
  const int64_t* len;
  const int32_t* slot;
  const int32_t* origin;
  const int32_t* tile0;
  int npieces, p;
};

// The piece that tile b belongs to: the last i < n with tile0[i] <= b
// (tile0 is non-decreasing and tile0[n] > b). Each warp searches on its own,
// 32 probes per round: the lanes whose probe is <= b form a prefix, whose
// length moves the lower bound, so every round shrinks the range 32-fold and
// a table of up to 1,024 pieces takes two dependent loads instead of ten.
// Measured on GB300 against a binary search in every thread, two runs each:
// ResNet-50-shaped step 240.3-240.8 -> 239.1-239.6 us, bf16 Llama-1B 5,498-
// 5,508 -> 5,453-5,455 us, GPT-2 unchanged (1,136-1,138 us), although the
// kernel now takes 48 registers at p = 8 (five blocks per SM) instead of 40
// (six). Forcing six blocks back with a launch bound gained nothing more.
__device__ __forceinline__ int find_piece(const int32_t* tile0, int n, int32_t b) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = n;  // tile0[lo] <= b < tile0[hi]
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) >> 5;  // probes at lo + step, lo + 2 step, ..., below hi
    const int q = lo + step * (lane + 1);
    const bool le = q < hi && tile0[q] <= b;
    const int c = __popc(__ballot_sync(0xffffffffu, le));
    hi = min(hi, lo + step * (c + 1));
    lo += step * c;
  }
  return lo;
}

// Launched as a programmatic dependent of the previous kernel in the stream:
// the piece table (static since the Reducer was built) may be read before
// that kernel has finished, gradient data only after griddepcontrol.wait,
// which each block executes once, before its first data access.
__device__ __forceinline__ void wait_previous_grid(bool& waited) {
  if (!waited) {
    pdl_wait();
    waited = true;
  }
}

template <typename T, int P>
__device__ __forceinline__ void bucket_tile(const View& a, int32_t b, float divisor, bool& waited) {
  constexpr int V = Vec<T>::N;
  constexpr int64_t kTile = bucket_tile_elems(sizeof(T));
  const int p = (P > 0) ? P : a.p;
  const int i = find_piece(a.tile0, a.npieces, b);
  const int64_t t0 = a.start[i] + static_cast<int64_t>(b - a.tile0[i]) * kTile;  // first element of the tile
  const int64_t len = min(kTile, a.start[i] + a.len[i] - t0);
  if (len <= 0) return;
  void* const* rep = a.ptr + static_cast<int64_t>(a.slot[i]) * p;
  // origin >= p marks a copy piece, one of the per-forward buffers that the
  // Reducer's one-launch step broadcasts ("PyTorch DDP Deep Dive", Part 2,
  // _sync_buffers -> _broadcast_coalesced): replica origin - p's bits are
  // written to every other replica, nothing is summed, the root is not written.
  const int oi = a.origin[i];
  const bool copy = oi >= p;
  const int o = copy ? oi - p : oi;

  // The replicas in ring order o, o+1, ... (mod p), staged in shared memory
  // rather than held in registers: with the binary search this kernel had
  // then, 40 registers instead of 74 at p = 8, so six blocks fit on an SM
  // instead of three, which is what hides each tile's table lookups.
  // Measured on GB300, one block per 4 KB tile against the earlier persistent
  // grid over 16 KB tiles with the pointers in registers: ResNet-50-shaped
  // sync 258.7 -> 244.4 us, GPT-2 1,222 -> 1,142 us, bf16 Llama-1B 5,678 ->
  // 5,499 us.
  __shared__ T* base[P > 0 ? P : 1];
  if constexpr (P > 0) {
    __syncthreads();  // every thread is done with the previous tile's bases
    if (threadIdx.x < P) base[threadIdx.x] = reinterpret_cast<T*>(rep[(o + threadIdx.x) % P]);
    __syncthreads();
  }

  wait_previous_grid(waited);

  // a vector path needs every replica at the same address mod 16
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(reinterpret_cast<const T*>(rep[0]) + t0);
  bool same = (a0 % sizeof(T)) == 0;
  for (int r = 1; r < p && same; ++r)
    same = ((reinterpret_cast<uintptr_t>(reinterpret_cast<const T*>(rep[r]) + t0) ^ a0) & 15u) == 0;
  int64_t head = len;
  if (same) head = min(static_cast<int64_t>(((16u - (a0 & 15u)) & 15u) / sizeof(T)), len);
  const int64_t nvec = (len - head) / V;
  const int64_t tail0 = head + nvec * V;

  if (copy) {
    for (int64_t e = threadIdx.x; e < head + (len - tail0); e += blockDim.x) {
      const int64_t x = t0 + (e < head ? e : tail0 + (e - head));
      const T y = reinterpret_cast<const T*>(rep[o])[x];
      for (int q = 0; q < p; ++q)
        if (q != o) reinterpret_cast<T*>(rep[q])[x] = y;
    }
    for (int64_t v = threadIdx.x; v < nvec; v += blockDim.x) {
      const int64_t x = t0 + head + v * V;
      const uint4 y = *reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(rep[o]) + x);
      for (int q = 0; q < p; ++q)
        if (q != o) *reinterpret_cast<uint4*>(reinterpret_cast<T*>(rep[q]) + x) = y;
    }
    return;
  }

  for (int64_t e = threadIdx.x; e < head + (len - tail0); e += blockDim.x) {
    const int64_t x = t0 + (e < head ? e : tail0 + (e - head));
    float acc = widen(reinterpret_cast<const T*>(rep[o])[x]);
    int r = o;
    for (int j = 1; j < p; ++j) {
      r = (r + 1 == p) ? 0 : r + 1;
      acc = __fadd_rn(acc, widen(reinterpret_cast<const T*>(rep[r])[x]));
    }
    const T y = narrow<T>(__fdiv_rn(acc, divisor));
    for (int q = 0; q < p; ++q) reinterpret_cast<T*>(rep[q])[x] = y;
  }

  for (int64_t v = threadIdx.x; v < nvec; v += blockDim.x) {
    const int64_t x = t0 + head + v * V;
    float acc[V];
    if constexpr (P > 0) {
      uint4 w[P];
#pragma unroll
      for (int j = 0; j < P; ++j) w[j] = ld_prefetch256(base[j] + x);
      Vec<T>::unpack(w[0], acc);
#pragma unroll
      for (int j = 1; j < P; ++j) {
        float t[V];
        Vec<T>::unpack(w[j], t);
#pragma unroll
        for (int l = 0; l < V; ++l) acc[l] = __fadd_rn(acc[l], t[l]);
      }
#pragma unroll
      for (int l = 0; l < V; ++l) acc[l] = __fdiv_rn(acc[l], divisor);
      const uint4 y = Vec<T>::pack(acc);
#pragma unroll
      for (int q = 0; q < P; ++q) *reinterpret_cast<uint4*>(base[q] + x) = y;
    } else {
      Vec<T>::unpack(*reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(rep[o]) + x), acc);
      int r = o;
      for (int j = 1; j < p; ++j) {
        r = (r + 1 == p) ? 0 : r + 1;
        float t[V];
        Vec<T>::unpack(*reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(rep[r]) + x), t);
#pragma unroll
        for (int l = 0; l < V; ++l) acc[l] = __fadd_rn(acc[l], t[l]);
      }
#pragma unroll
      for (int l = 0; l < V; ++l) acc[l] = __fdiv_rn(acc[l], divisor);
      const uint4 y = Vec<T>::pack(acc);
      for (int q = 0; q < p; ++q) *reinterpret_cast<uint4*>(reinterpret_cast<T*>(rep[q]) + x) = y;
    }
  }
}

template <typename T, int P>
__device__ __forceinline__ void bucket_tiles(const View& v, float divisor) {
  const int32_t total = v.tile0[v.npieces];
  bool waited = false;
  for (int32_t b = blockIdx.x; b < total; b += gridDim.x) bucket_tile<T, P>(v, b, divisor, waited);
  wait_previous_grid(waited);  // a block with no data to touch still orders after the previous grid
}

// Arguments by value (one bucket, from ddp_bucket_allreduce).
template <typename T, int P>
__global__ void __launch_bounds__(kBucketThreads) k_bucket_allreduce(const __grid_constant__ BucketArgs a) {
  pdl_trigger();
  const View v{a.ptr, a.start, a.len, a.slot, a.origin, a.tile0, a.npieces, a.p};
  bucket_tiles<T, P>(v, a.divisor);
}

// Piece table in device memory (every bucket of a Reducer in one launch).
template <typename T, int P>
__global__ void __launch_bounds__(kBucketThreads) k_bucket_allreduce_table(const BucketTable t, float divisor) {
  pdl_trigger();
  const View v{t.ptr, t.start, t.len, t.slot, t.origin, t.tile0, t.npieces, t.p};
  bucket_tiles<T, P>(v, divisor);
}

// ------------------------------------------------------------ staged form
// The same tiles with the loads staged through shared memory: lane j of warp
// 0 issues a bulk asynchronous copy (cp.async.bulk, the TMA's non-tensor
// form) of the tile's 16-byte-aligned body from replica j, all P completing
// on one mbarrier; every thread then folds its 16 bytes from the P
// staged copies in ring order and stores the result to every replica with
// 128-bit stores. The few elements outside the aligned body (a tensor's
// misaligned start or end) take the register form's plain loads while the
// copies are in flight. The wait on the copies is bounded: past kStagedWaitNs
// the block records kErrBulkWait in the device error word, waits once more
// (bounded) for its copies to land, and stores nothing.
constexpr int64_t kStagedWaitNs = 2000000000LL;

template <typename T, int P>
__global__ void __launch_bounds__(kBucketThreads) k_bucket_table_staged(const BucketTable t, float divisor) {
  static_assert(P >= 2 && P * kBucketTileBytes <= 40 * 1024, "staged tiles of every replica must fit");
  constexpr int V = Vec<T>::N;
  constexpr int64_t kTile = bucket_tile_elems(sizeof(T));
  __shared__ __align__(128) uint4 stage[P][kBucketThreads];  // replica (ring position) j's tile body
  __shared__ __align__(8) uint64_t full;
  __shared__ T* base[P];
  pdl_trigger();
  bool waited = false;
  const View a{t.ptr, t.start, t.len, t.slot, t.origin, t.tile0, t.npieces, t.p};
  const int32_t b = blockIdx.x;
  if (b >= a.tile0[a.npieces]) {
    wait_previous_grid(waited);
    return;
  }
  const int i = find_piece(a.tile0, a.npieces, b);
  const int64_t t0 = a.start[i] + static_cast<int64_t>(b - a.tile0[i]) * kTile;
  const int64_t len = min(kTile, a.start[i] + a.len[i] - t0);
  if (len <= 0) {
    wait_previous_grid(waited);
    return;
  }
  void* const* rep = a.ptr + static_cast<int64_t>(a.slot[i]) * P;
  const int oi = a.origin[i];
  const bool copy = oi >= P;  // a copy piece: replica oi - P's bits to the others
  const int o = copy ? oi - P : oi;
  const uint32_t bar = smem_addr(&full);
  if (threadIdx.x < P) base[threadIdx.x] = reinterpret_cast<T*>(rep[(o + threadIdx.x) % P]);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  wait_previous_grid(waited);

  const uintptr_t a0 = reinterpret_cast<uintptr_t>(base[0] + t0);
  bool same = (a0 % sizeof(T)) == 0;
  for (int r = 1; r < P && same; ++r) same = ((reinterpret_cast<uintptr_t>(base[r] + t0) ^ a0) & 15u) == 0;
  int64_t head = len;
  if (same) head = min(static_cast<int64_t>(((16u - (a0 & 15u)) & 15u) / sizeof(T)), len);
  const int nvec = static_cast<int>((len - head) / V);
  const int64_t tail0 = head + static_cast<int64_t>(nvec) * V;
  const int loads = copy ? 1 : P;

  if (threadIdx.x < 32 && nvec > 0) {  // warp 0: lane j copies replica j's body
    const uint32_t bytes = static_cast<uint32_t>(nvec) * 16u;
    if (threadIdx.x == 0) mbar_arrive_expect_tx(bar, bytes * loads);
    __syncwarp();
    if (static_cast<int>(threadIdx.x) < loads)
      bulk_load(smem_addr(stage[threadIdx.x]), base[threadIdx.x] + t0 + head, bytes, bar);
  }

  for (int64_t e = threadIdx.x; e < head + (len - tail0); e += blockDim.x) {
    const int64_t x = t0 + (e < head ? e : tail0 + (e - head));
    if (copy) {
      const T y = base[0][x];
      for (int q = 1; q < P; ++q) base[q][x] = y;
      continue;
    }
    float acc = widen(base[0][x]);
    for (int j = 1; j < P; ++j) acc = __fadd_rn(acc, widen(base[j][x]));
    const T y = narrow<T>(__fdiv_rn(acc, divisor));
    for (int q = 0; q < P; ++q) base[q][x] = y;
  }
  if (nvec == 0) return;

  if (!mbar_wait_bounded(bar, 0, kStagedWaitNs)) {
    if (t.err) atomicCAS(t.err, 0, kErrBulkWait);
    (void)mbar_wait_bounded(bar, 0, kStagedWaitNs);  // the copies must land before shared memory goes away
    return;
  }
  const int v = threadIdx.x;
  if (v >= nvec) return;
  const int64_t x = t0 + head + static_cast<int64_t>(v) * V;
  if (copy) {
    const uint4 y = stage[0][v];
#pragma unroll
    for (int q = 1; q < P; ++q) *reinterpret_cast<uint4*>(base[q] + x) = y;
    return;
  }
  float acc[V];
  Vec<T>::unpack(stage[0][v], acc);
#pragma unroll
  for (int j = 1; j < P; ++j) {
    float u[V];
    Vec<T>::unpack(stage[j][v], u);
#pragma unroll
    for (int l = 0; l < V; ++l) acc[l] = __fadd_rn(acc[l], u[l]);
  }
#pragma unroll
  for (int l = 0; l < V; ++l) acc[l] = __fdiv_rn(acc[l], divisor);
  const uint4 y = Vec<T>::pack(acc);
#pragma unroll
  for (int q = 0; q < P; ++q) *reinterpret_cast<uint4*>(base[q] + x) = y;
}

// One block per tile: blocks are dispatched in index order, so the resident
// ones work on consecutive tiles. Measured on GB300 and slower: a persistent
// grid striding over the tiles, and one taking tiles in order from a device
// counter. Each bucket's launch is a programmatic dependent of the previous
// kernel in the stream (usually the previous bucket's), so its blocks start
// while that kernel's last wave drains.
template <typename T>
cudaError_t by_value(const BucketArgs& a, cudaStream_t s, int32_t max_blocks) {
  const int32_t tiles = a.tile0[a.npieces];
  const dim3 grid(max_blocks > 0 ? std::min(tiles, max_blocks) : tiles), block(kBucketThreads);
  cudaError_t e;
  switch (a.p) {
    case 2: e = launch_pdl(k_bucket_allreduce<T, 2>, grid, block, 0, s, a); break;
    case 4: e = launch_pdl(k_bucket_allreduce<T, 4>, grid, block, 0, s, a); break;
    case 8: e = launch_pdl(k_bucket_allreduce<T, 8>, grid, block, 0, s, a); break;
    case 16: e = launch_pdl(k_bucket_allreduce<T, 16>, grid, block, 0, s, a); break;
    default: e = launch_pdl(k_bucket_allreduce<T, 0>, grid, block, 0, s, a); break;
  }
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

// The whole-Reducer launch may start while the previous kernel in the stream
// finishes (programmatic stream serialisation): its blocks fetch their first
// piece while that kernel drains, and wait for it before touching gradients.
// Measured on GB300 on the ResNet-50-shaped step (buffer broadcast, then this
// kernel): 263.1 -> 259.6 us per step.
// The staged form needs no shared-memory carveout preference: the driver
// already gives its blocks the largest split (13 blocks per SM at p = 8).
// Measured on GB300 with the preference set to the maximum: the same times
// within 0.1 us on the ResNet-50-shaped sync.
template <typename T, int P>
cudaError_t launch_table(const BucketTable& t, int32_t tiles, float divisor, cudaStream_t s, bool staged = false) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles);
  cfg.blockDim = dim3(kBucketThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if constexpr (P >= 2) {
    if (staged) return cudaLaunchKernelEx(&cfg, k_bucket_table_staged<T, P>, t, divisor);
  }
  return cudaLaunchKernelEx(&cfg, k_bucket_allreduce_table<T, P>, t, divisor);
}

// staged: the shared-memory staged form for p = 2, 4, 8 and 16; any other p
// takes the register form.
template <typename T>
cudaError_t by_table(const BucketTable& t, int32_t tiles, float divisor, cudaStream_t s, bool staged) {
  cudaError_t e;
  switch (t.p) {
    case 2: e = launch_table<T, 2>(t, tiles, divisor, s, staged); break;
    case 4: e = launch_table<T, 4>(t, tiles, divisor, s, staged); break;
    case 8: e = launch_table<T, 8>(t, tiles, divisor, s, staged); break;
    case 16: e = launch_table<T, 16>(t, tiles, divisor, s, staged); break;
    default: e = launch_table<T, 0>(t, tiles, divisor, s); break;
  }
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_bucket_allreduce(const BucketArgs& a, ddp_dtype dt, cudaStream_t s, int32_t max_blocks) {
  if (a.npieces <= 0 || a.tile0[a.npieces] <= 0) return cudaSuccess;
  return dt == DDP_FLOAT32 ? by_value<float>(a, s, max_blocks) : by_value<__nv_bfloat16>(a, s, max_blocks);
}

// Which form DDP_ALGO_FUSED takes: the staged one where it measured faster
// on GB300 than the register one. In-place sync, launches back to back, best
// of four, staged against registers:
//   ResNet-50-shaped set (25.6 M gradients), fp32, p = 2, 4, 8, 16:
//     70.7 / 120.2 / 236.2 / 480.9 us against 67.3 / 120.6 / 237.7 / 474.6;
//   GPT-2-shaped set (124 M), fp32, p = 2, 4, 16: 321.9 / 566.1 / 2,303
//     against 295.5 / 567.5 / 2,278 us (p = 8: 1,135.4 against 1,137.0);
//   Llama-1B-shaped set (1.2 B), bf16, p = 2, 4, 8: 1,661 / 2,746 / 5,475
//     against 1,724 / 2,777 / 5,460 us.
// (The ResNet-50-shaped set in bf16 also favoured the staged form at p = 2
// and 4, 38.0 / 62.4 against 41.7 / 70.0 us, but partly from L2.) The
// one-launch step on the ResNet-50-shaped set, with its 159 buffers: 236.9
// against 238.8 us. At p = 16 the staged tiles (32 KB a block) leave room for
// six blocks per SM; at p = 2 a tile is too little work to repay the mbarrier
// round trip.
bool staged_by_default(ddp_dtype dt, int p) {
  return dt == DDP_FLOAT32 ? (p == 4 || p == 8) : (p == 2 || p == 4);
}

cudaError_t launch_bucket_table(const BucketTable& t, int32_t total_tiles, float divisor, ddp_dtype dt,
                                cudaStream_t s, ddp_algo algo) {
  if (t.npieces <= 0 || total_tiles <= 0) return cudaSuccess;
  const bool staged = algo == DDP_ALGO_FUSED_TMA || (algo == DDP_ALGO_FUSED && staged_by_default(dt, t.p));
  return dt == DDP_FLOAT32 ? by_table<float>(t, total_tiles, divisor, s, staged)
                           : by_table<__nv_bfloat16>(t, total_tiles, divisor, s, staged);
}

}  // namespace ddp
