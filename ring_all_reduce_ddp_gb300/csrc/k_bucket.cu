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
// same bits as the ring on the flat bucket.
#include "launch.h"

namespace ddp {
namespace {

constexpr int kVecPerThread = kBucketTileBytes / 16 / kThreads;  // 4

__device__ __forceinline__ int find_piece(const int32_t* tile0, int n, int32_t b) {
  int lo = 0, hi = n;  // tile0[lo] <= b < tile0[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile0[mid] <= b) lo = mid; else hi = mid;
  }
  return lo;
}

template <typename T, int P>
__global__ void __launch_bounds__(kThreads) k_bucket_allreduce(const __grid_constant__ BucketArgs a) {
  constexpr int V = Vec<T>::N;
  constexpr int64_t kTile = kBucketTileBytes / sizeof(T);
  const int p = (P > 0) ? P : a.p;
  const int32_t b = blockIdx.x;
  const int i = find_piece(a.tile0, a.npieces, b);
  const int64_t t0 = a.start[i] + static_cast<int64_t>(b - a.tile0[i]) * kTile;  // first element of this tile
  const int64_t len = min(kTile, a.start[i] + a.len[i] - t0);
  if (len <= 0) return;
  void* const* rep = &a.ptr[static_cast<int64_t>(a.slot[i]) * p];
  const int o = a.origin[i];

  // the ring order o, o+1, ..., o+p-1 (mod p) as replica indices
  int order[P > 0 ? P : 1];
  if constexpr (P > 0) {
#pragma unroll
    for (int j = 0; j < P; ++j) order[j] = (o + j) % P;
  }

  // a vector path needs every replica at the same address mod 16
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(reinterpret_cast<const T*>(rep[0]) + t0);
  bool same = (a0 % sizeof(T)) == 0;
  for (int r = 1; r < p && same; ++r)
    same = ((reinterpret_cast<uintptr_t>(reinterpret_cast<const T*>(rep[r]) + t0) ^ a0) & 15u) == 0;
  int64_t head = len;
  if (same) head = min(static_cast<int64_t>(((16u - (a0 & 15u)) & 15u) / sizeof(T)), len);
  const int64_t nvec = (len - head) / V;
  const int64_t tail0 = head + nvec * V;

  // scalar elements: the head, the tail, or all of them
  for (int64_t e = threadIdx.x; e < head + (len - tail0); e += blockDim.x) {
    const int64_t x = t0 + (e < head ? e : tail0 + (e - head));
    float acc = widen(reinterpret_cast<const T*>(rep[o])[x]);
    int r = o;
    for (int j = 1; j < p; ++j) {
      r = (r + 1 == p) ? 0 : r + 1;
      acc = __fadd_rn(acc, widen(reinterpret_cast<const T*>(rep[r])[x]));
    }
    const T y = narrow<T>(__fdiv_rn(acc, a.divisor));
    for (int q = 0; q < p; ++q) reinterpret_cast<T*>(rep[q])[x] = y;
  }

  for (int64_t v = threadIdx.x; v < nvec; v += blockDim.x) {
    const int64_t x = t0 + head + v * V;
    float acc[V];
    if constexpr (P > 0) {
      uint4 w[P];
#pragma unroll
      for (int j = 0; j < P; ++j) w[j] = *reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(rep[order[j]]) + x);
      Vec<T>::unpack(w[0], acc);
#pragma unroll
      for (int j = 1; j < P; ++j) {
        float t[V];
        Vec<T>::unpack(w[j], t);
#pragma unroll
        for (int l = 0; l < V; ++l) acc[l] = __fadd_rn(acc[l], t[l]);
      }
#pragma unroll
      for (int l = 0; l < V; ++l) acc[l] = __fdiv_rn(acc[l], a.divisor);
      const uint4 y = Vec<T>::pack(acc);
#pragma unroll
      for (int q = 0; q < P; ++q) *reinterpret_cast<uint4*>(reinterpret_cast<T*>(rep[q]) + x) = y;
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
      for (int l = 0; l < V; ++l) acc[l] = __fdiv_rn(acc[l], a.divisor);
      const uint4 y = Vec<T>::pack(acc);
      for (int q = 0; q < p; ++q) *reinterpret_cast<uint4*>(reinterpret_cast<T*>(rep[q]) + x) = y;
    }
  }
}

template <typename T>
cudaError_t bucket_launch(const BucketArgs& a, cudaStream_t s) {
  const int32_t tiles = a.tile0[a.npieces];
  switch (a.p) {
    case 2: k_bucket_allreduce<T, 2><<<tiles, kThreads, 0, s>>>(a); break;
    case 4: k_bucket_allreduce<T, 4><<<tiles, kThreads, 0, s>>>(a); break;
    case 8: k_bucket_allreduce<T, 8><<<tiles, kThreads, 0, s>>>(a); break;
    case 16: k_bucket_allreduce<T, 16><<<tiles, kThreads, 0, s>>>(a); break;
    default: k_bucket_allreduce<T, 0><<<tiles, kThreads, 0, s>>>(a); break;
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bucket_allreduce(const BucketArgs& a, ddp_dtype dt, cudaStream_t s) {
  if (a.npieces <= 0 || a.tile0[a.npieces] <= 0) return cudaSuccess;
  return dt == DDP_FLOAT32 ? bucket_launch<float>(a, s) : bucket_launch<__nv_bfloat16>(a, s);
}

}  // namespace ddp
