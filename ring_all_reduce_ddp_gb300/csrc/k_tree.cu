// The add step of the tree-shaped all-reduces ("Data parallelism",
// "Latency, trees, and choosing an algorithm": recursive doubling, and
// recursive halving and doubling; "Collective Ops From Scratch": tree
// all-reduce). Each job adds two replicas' copies of a range, in fp32, and
// writes the sum to one or both of them. Both partners of an exchange compute
// the same a + b (addition is commutative), so one thread per element writes
// both copies and no workspace is needed.
#include "launch.h"

namespace ddp {
namespace {

constexpr int kAddU = 4;  // float4 vectors in flight per thread

__global__ void __launch_bounds__(kThreads) k_pair_add(const __grid_constant__ PairAddArgs a) {
  pdl_trigger();
  pdl_wait();
  const int j = blockIdx.y;
  const int64_t lo = a.lo[j], hi = a.hi[j];
  if (hi <= lo) return;
  const float* A = a.a[j];
  const float* B = a.b[j];
  float* D1 = a.d1[j];
  float* D2 = a.d2[j];
  const float div = a.divisor;
  const bool divide = a.divide != 0;
  auto one = [&](int64_t i) {
    float y = __fadd_rn(A[i], B[i]);
    if (divide) y = __fdiv_rn(y, div);
    D1[i] = y;
    if (D2) D2[i] = y;
  };
  // vector body when every pointer sits at the same address mod 16
  const uintptr_t y = (reinterpret_cast<uintptr_t>(A + lo) ^ reinterpret_cast<uintptr_t>(B + lo)) |
                      (reinterpret_cast<uintptr_t>(A + lo) ^ reinterpret_cast<uintptr_t>(D1 + lo)) |
                      (D2 ? (reinterpret_cast<uintptr_t>(A + lo) ^ reinterpret_cast<uintptr_t>(D2 + lo)) : 0);
  int64_t head = hi - lo;
  if ((y & 15u) == 0 && (reinterpret_cast<uintptr_t>(A + lo) & 3u) == 0)
    head = min(static_cast<int64_t>(((16u - (reinterpret_cast<uintptr_t>(A + lo) & 15u)) & 15u) / 4), hi - lo);
  const int64_t nvec = (hi - lo - head) / 4;
  const int64_t tail0 = lo + head + nvec * 4;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t gstride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = gtid; e < head; e += gstride) one(lo + e);
  for (int64_t i = tail0 + gtid; i < hi; i += gstride) one(i);
  const float4* A4 = reinterpret_cast<const float4*>(A + lo + head);
  const float4* B4 = reinterpret_cast<const float4*>(B + lo + head);
  float4* D14 = reinterpret_cast<float4*>(D1 + lo + head);
  float4* D24 = D2 ? reinterpret_cast<float4*>(D2 + lo + head) : nullptr;
  for (int64_t v0 = gtid; v0 < nvec; v0 += gstride * kAddU) {
    float4 u[kAddU], w[kAddU];
#pragma unroll
    for (int q = 0; q < kAddU; ++q) {
      const int64_t v = v0 + q * gstride;
      if (v < nvec) { u[q] = A4[v]; w[q] = B4[v]; }
    }
#pragma unroll
    for (int q = 0; q < kAddU; ++q) {
      const int64_t v = v0 + q * gstride;
      if (v < nvec) {
        float4 r;
        r.x = __fadd_rn(u[q].x, w[q].x);
        r.y = __fadd_rn(u[q].y, w[q].y);
        r.z = __fadd_rn(u[q].z, w[q].z);
        r.w = __fadd_rn(u[q].w, w[q].w);
        if (divide) {
          r.x = __fdiv_rn(r.x, div);
          r.y = __fdiv_rn(r.y, div);
          r.z = __fdiv_rn(r.z, div);
          r.w = __fdiv_rn(r.w, div);
        }
        D14[v] = r;
        if (D24) D24[v] = r;
      }
    }
  }
}

}  // namespace

cudaError_t launch_pair_add(const PairAddArgs& a, cudaStream_t s) {
  if (a.njobs <= 0) return cudaSuccess;
  int64_t maxlen = 0;
  for (int j = 0; j < a.njobs; ++j) maxlen = (a.hi[j] - a.lo[j]) > maxlen ? (a.hi[j] - a.lo[j]) : maxlen;
  if (maxlen <= 0) return cudaSuccess;
  const int64_t target = static_cast<int64_t>(sm_count()) * (2048 / kThreads);
  int64_t bx = (target + a.njobs - 1) / a.njobs;
  const int64_t need = (maxlen / 4 + kThreads * kAddU - 1) / (kThreads * kAddU);
  if (bx > need) bx = need;
  if (bx < 1) bx = 1;
  const cudaError_t e = launch_pdl(k_pair_add, dim3(static_cast<unsigned>(bx), a.njobs), dim3(kThreads), 0, s, a);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace ddp
