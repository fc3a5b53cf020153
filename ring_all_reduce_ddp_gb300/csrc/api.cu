// The C ABI (include/ddp_ring.h), collectives part: bucket assignment,
// flatten / unflatten, the all-reduce family, reduce-scatter, all-gather,
// broadcast and coalesced broadcast, the stepwise ddp_ring handle, and the
// library's status calls. Host code only plans and launches; every step that
// touches data runs in the library's kernels. The exported collectives are
// thin wrappers (calllog.cu) around the *_impl bodies here.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <string>
#include <utility>
#include <vector>

#include "host.h"

using namespace ddp;
using namespace ddp::host;

namespace ddp {
namespace host {

ddp_status allreduce_impl(void* const* bufs, int32_t p, int64_t n, ddp_dtype dtype, float divisor,
                          ddp_algo algo, cudaStream_t stream) {
  DDP_NVTX("ddp_allreduce");
  if (is_tree_algo(algo)) {
    DDP_TRY(check_common(p, n, dtype));
    DDP_TRY(check_divisor(divisor));
    if (n == 0) return DDP_OK;  // a no-op whatever the pointers
    DDP_TRY(check_ptrs(const_cast<const void* const*>(bufs), p, "bufs"));
    const int es = esize(dtype);
    std::vector<std::pair<uintptr_t, uintptr_t>> rg;
    for (int r = 0; r < p; ++r) rg.push_back(range_of(bufs[r], n * es));
    DDP_CHECK(disjoint(rg), DDP_ERR_ARG, "replica buffers overlap");
    if (n == 0) return DDP_OK;
    if (algo != DDP_ALGO_TREE) {
      const bool pow2 = (p & (p - 1)) == 0;
      DDP_CHECK(pow2, DDP_ERR_ARG, "recursive doubling and Rabenseifner need p a power of two");
    }
    std::vector<float*> B(p);
    if (dtype == DDP_FLOAT32) {
      for (int r = 0; r < p; ++r) B[r] = static_cast<float*>(bufs[r]);
      return run_tree_allreduce(B.data(), p, n, divisor, algo, stream);
    }
    if (p == 1)
      return run_fused(const_cast<const void* const*>(bufs), bufs, 1, n, dtype, divisor, false, 0, false, stream);
    // bf16: the schedule runs on fp32 partials (widened exactly), and each
    // replica's finished fp32 value is rounded to bf16 once at the end.
    const int64_t slot = (n * 4 + 255) / 256 * 256;
    void* wsv = nullptr;
    DDP_TRY(alloc_async(&wsv, slot * p, stream, "tree workspace"));
    char* ws = static_cast<char*>(wsv);
    for (int r = 0; r < p; ++r) B[r] = reinterpret_cast<float*>(ws + slot * r);
    ConvertArgs cv;
    std::memset(&cv, 0, sizeof(cv));
    cv.n = n;
    cv.njobs = p;
    for (int r = 0; r < p; ++r) { cv.src[r] = bufs[r]; cv.dst[r] = B[r]; }
    cudaError_t e = launch_convert(cv, stream);
    ddp_status rc = e == cudaSuccess ? run_tree_allreduce(B.data(), p, n, divisor, algo, stream)
                                     : cuda_fail(e, "widen launch");
    if (rc == DDP_OK) {
      cv.to_bf16 = 1;
      for (int r = 0; r < p; ++r) { cv.src[r] = B[r]; cv.dst[r] = bufs[r]; }
      e = launch_convert(cv, stream);
      if (e != cudaSuccess) rc = cuda_fail(e, "narrow launch");
    }
    const cudaError_t ef = cudaFreeAsync(wsv, stream);
    if (rc != DDP_OK) return rc;
    if (ef != cudaSuccess) return cuda_fail(ef, "tree workspace release");
    return DDP_OK;
  }
  return allreduce_ex_impl(bufs, p, n, dtype, divisor, algo, 0u, stream);
}

ddp_status allreduce_ex_impl(void* const* bufs, int32_t p, int64_t n, ddp_dtype dtype, float divisor,
                             ddp_algo algo, uint32_t flags, cudaStream_t stream) {
  DDP_NVTX("ddp_allreduce_ex");
  DDP_TRY(check_common(p, n, dtype));
  DDP_TRY(check_divisor(divisor));
  DDP_TRY(check_algo(algo));
  DDP_CHECK((flags & ~static_cast<uint32_t>(DDP_FLAG_ROUND_EACH_HOP)) == 0, DDP_ERR_ARG, "unknown flags");
  const bool hop = (flags & DDP_FLAG_ROUND_EACH_HOP) != 0;
  DDP_CHECK(!hop || dtype == DDP_BFLOAT16, DDP_ERR_DTYPE, "DDP_FLAG_ROUND_EACH_HOP is a bf16 variant");
  if (n == 0) return DDP_OK;  // a no-op whatever the pointers
  DDP_TRY(check_ptrs(const_cast<const void* const*>(bufs), p, "bufs"));
  const int es = esize(dtype);
  std::vector<std::pair<uintptr_t, uintptr_t>> rg;
  for (int r = 0; r < p; ++r) rg.push_back(range_of(bufs[r], n * es));
  DDP_CHECK(disjoint(rg), DDP_ERR_ARG, "replica buffers overlap");
  if (n == 0) return DDP_OK;
  if (algo == DDP_ALGO_RING_STEPS) {
    Plan pl;
    pl.op = DDP_OP_ALLREDUCE; pl.p = p; pl.n = n; pl.dt = dtype; pl.divisor = divisor; pl.hop_round = hop;
    pl.in.assign(bufs, bufs + p);
    return run_plan_once(pl, stream);
  }
  return run_fused(const_cast<const void* const*>(bufs), bufs, p, n, dtype, divisor, false, 0,
                   algo == DDP_ALGO_FUSED_TMA && !hop, stream, hop);
}

ddp_status reduce_scatter_impl(const void* const* in, void* const* out, int32_t p, int64_t n, ddp_dtype dtype,
                               float divisor, ddp_own own, ddp_algo algo, cudaStream_t stream) {
  DDP_NVTX("ddp_reduce_scatter");
  DDP_TRY(check_common(p, n, dtype));
  DDP_TRY(check_divisor(divisor));
  DDP_TRY(check_algo(algo));
  DDP_TRY(check_own(own));
  if (n == 0) return DDP_OK;  // a no-op whatever the pointers
  DDP_TRY(check_ptrs(in, p, "in"));
  DDP_TRY(check_ptrs(const_cast<const void* const*>(out), p, "out"));
  if (own == DDP_OWN_RANK)
    DDP_CHECK(n % p == 0, DDP_ERR_NOT_DIVISIBLE,
              "reduce_scatter: " + std::to_string(n) + " elements are not divisible by " + std::to_string(p) + " ranks");
  const int es = esize(dtype);
  const int64_t cs = chunk_size(n, p);
  std::vector<std::pair<uintptr_t, uintptr_t>> outs, all;
  for (int r = 0; r < p; ++r) outs.push_back(range_of(out[r], cs * es));
  DDP_CHECK(disjoint(outs), DDP_ERR_ARG, "output buffers overlap");
  for (int r = 0; r < p; ++r) {
    all = outs;
    all.push_back(range_of(in[r], n * es));
    DDP_CHECK(disjoint(all), DDP_ERR_ARG, "an output buffer overlaps an input");
  }
  if (n == 0) return DDP_OK;
  if (algo == DDP_ALGO_RING_STEPS) {
    Plan pl;
    pl.op = DDP_OP_REDUCE_SCATTER; pl.p = p; pl.n = n; pl.dt = dtype; pl.divisor = divisor; pl.own = own;
    pl.in.assign(const_cast<void* const*>(in), const_cast<void* const*>(in) + p);
    pl.out.assign(out, out + p);
    return run_plan_once(pl, stream);
  }
  return run_fused(in, out, p, n, dtype, divisor, true, own == DDP_OWN_RANK ? 1 : 0,
                   algo == DDP_ALGO_FUSED_TMA, stream);
}

ddp_status allgather_impl(const void* const* in, void* const* out, int32_t p, int64_t m, ddp_dtype dtype,
                          ddp_own own, ddp_algo algo, cudaStream_t stream) {
  DDP_NVTX("ddp_allgather");
  DDP_TRY(check_common(p, m, dtype));
  DDP_TRY(check_algo(algo));
  DDP_TRY(check_own(own));
  if (m == 0) return DDP_OK;  // a no-op whatever the pointers
  DDP_TRY(check_ptrs(in, p, "in"));
  DDP_TRY(check_ptrs(const_cast<const void* const*>(out), p, "out"));
  const int es = esize(dtype);
  std::vector<std::pair<uintptr_t, uintptr_t>> outs, all;
  for (int r = 0; r < p; ++r) outs.push_back(range_of(out[r], static_cast<int64_t>(p) * m * es));
  DDP_CHECK(disjoint(outs), DDP_ERR_ARG, "output buffers overlap");
  for (int r = 0; r < p; ++r) {
    all = outs;
    all.push_back(range_of(in[r], m * es));
    DDP_CHECK(disjoint(all), DDP_ERR_ARG, "an output buffer overlaps an input");
  }
  if (m == 0) return DDP_OK;
  if (algo == DDP_ALGO_RING_STEPS) {
    Plan pl;
    pl.op = DDP_OP_ALLGATHER; pl.p = p; pl.n = m; pl.dt = dtype; pl.own = own;
    pl.in.assign(const_cast<void* const*>(in), const_cast<void* const*>(in) + p);
    pl.out.assign(out, out + p);
    return run_plan_once(pl, stream);
  }
  FanoutArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int c = 0; c < p; ++c) {
    const int holder = (own == DDP_OWN_RANK) ? c : (c + p - 1) % p;
    a.src[c] = static_cast<const char*>(in[holder]);
    a.job_off[c] = static_cast<int64_t>(c) * m * es;
  }
  for (int r = 0; r < p; ++r) a.dst[r] = static_cast<char*>(out[r]);
  a.nbytes = m * es;
  a.njobs = p;
  a.ndst = p;
  DDP_CUDA(launch_fanout(a, stream, algo), "all-gather launch");
  return DDP_OK;
}

ddp_status broadcast_impl(void* const* bufs, int32_t p, int64_t nbytes, int32_t root, ddp_algo algo,
                          cudaStream_t stream) {
  DDP_NVTX("ddp_broadcast");
  DDP_TRY(check_common(p, nbytes, DDP_FLOAT32));
  DDP_TRY(check_algo(algo));
  DDP_CHECK(root >= 0 && root < p, DDP_ERR_ARG, "root out of range");
  if (nbytes == 0) return DDP_OK;  // a no-op whatever the pointers
  DDP_TRY(check_ptrs(const_cast<const void* const*>(bufs), p, "bufs"));
  std::vector<std::pair<uintptr_t, uintptr_t>> rg;
  for (int r = 0; r < p; ++r) rg.push_back(range_of(bufs[r], nbytes));
  DDP_CHECK(disjoint(rg), DDP_ERR_ARG, "replica buffers overlap");
  if (nbytes == 0 || p == 1) return DDP_OK;
  if (algo == DDP_ALGO_RING_STEPS) {
    Plan pl;
    pl.op = DDP_OP_BROADCAST; pl.p = p; pl.n = nbytes; pl.root = root;
    pl.in.assign(bufs, bufs + p);
    return run_plan_once(pl, stream);
  }
  FanoutArgs a;
  std::memset(&a, 0, sizeof(a));
  a.src[0] = static_cast<const char*>(bufs[root]);
  int q = 0;
  for (int r = 0; r < p; ++r)
    if (r != root) a.dst[q++] = static_cast<char*>(bufs[r]);
  a.nbytes = nbytes;
  a.njobs = 1;
  a.ndst = q;
  DDP_CUDA(launch_fanout(a, stream, algo), "broadcast launch");
  return DDP_OK;
}

ddp_status broadcast_coalesced_impl(int32_t p, int32_t k, void* const* tensors, const int64_t* nbytes,
                                    int32_t root, int64_t bucket_cap_bytes, ddp_algo algo,
                                    cudaStream_t stream) {
  DDP_NVTX("ddp_broadcast_coalesced");
  DDP_TRY(check_common(p, 0, DDP_FLOAT32));
  DDP_TRY(check_algo(algo));
  DDP_CHECK(k >= 0, DDP_ERR_ARG, "k must be >= 0");
  DDP_CHECK(root >= 0 && root < p, DDP_ERR_ARG, "root out of range");
  DDP_CHECK(bucket_cap_bytes >= 0, DDP_ERR_ARG, "bucket_cap_bytes must be >= 0");
  if (k == 0) return DDP_OK;
  DDP_CHECK(tensors && nbytes, DDP_ERR_ARG, "tensors / nbytes arrays are null");
  std::vector<std::pair<uintptr_t, uintptr_t>> rg;
  for (int32_t j = 0; j < k; ++j) {
    DDP_CHECK(nbytes[j] >= 0, DDP_ERR_ARG, "nbytes must be >= 0");
    if (nbytes[j] == 0) continue;
    for (int32_t r = 0; r < p; ++r) {
      const void* t = tensors[static_cast<int64_t>(r) * k + j];
      DDP_CHECK(t != nullptr, DDP_ERR_ARG, "tensors[" + std::to_string(r * k + j) + "] is null");
      rg.push_back(range_of(t, nbytes[j]));
    }
  }
  DDP_CHECK(disjoint(rg), DDP_ERR_ARG, "tensors overlap");
  if (p == 1) return DDP_OK;
  const int64_t cap = bucket_cap_bytes > 0 ? bucket_cap_bytes : int64_t(250) * 1024 * 1024;
  auto T = [&](int r, int j) { return tensors[static_cast<int64_t>(r) * k + j]; };

  if (algo != DDP_ALGO_RING_STEPS) {
    // Every root tensor straight to the p-1 other replicas, kFanD destinations per launch.
    const int ndst = p - 1;
    const int per_launch = std::max(1, std::min(kFanT, kFanD / ndst));
    MultiFanoutArgs a;
    std::memset(&a, 0, sizeof(a));
    a.ndst = ndst;
    auto flush = [&]() -> ddp_status {
      if (a.ntensors == 0) return DDP_OK;
      DDP_CUDA(launch_multi_fanout(a, stream), "coalesced broadcast launch");
      std::memset(&a, 0, sizeof(a));
      a.ndst = ndst;
      return DDP_OK;
    };
    for (int32_t j = 0; j < k; ++j) {
      if (nbytes[j] == 0) continue;
      const int64_t tiles = (nbytes[j] + kSegTileBytes - 1) / kSegTileBytes;
      if (a.ntensors == per_launch || static_cast<int64_t>(a.tile0[a.ntensors]) + tiles > 0x7FFFFFFF)
        DDP_TRY(flush());
      const int t = a.ntensors;
      a.src[t] = static_cast<const char*>(T(root, j));
      a.bytes[t] = nbytes[j];
      int q = 0;
      for (int r = 0; r < p; ++r)
        if (r != root) a.dst[t * ndst + q++] = static_cast<char*>(T(r, j));
      a.tile0[t + 1] = a.tile0[t] + static_cast<int32_t>(tiles);
      ++a.ntensors;
    }
    return flush();
  }

  // Literal: coalesce into buckets of at most `cap` bytes; per bucket pack on
  // the root, broadcast the packed buffer by the doubling tree, unpack.
  std::vector<std::vector<int32_t>> groups;
  std::vector<int64_t> gbytes;
  {
    std::vector<int32_t> cur;
    int64_t size = 0;
    for (int32_t j = 0; j < k; ++j) {
      if (!cur.empty() && size + nbytes[j] > cap) {
        groups.push_back(cur);
        gbytes.push_back(size);
        cur.clear();
        size = 0;
      }
      cur.push_back(j);
      size += nbytes[j];
    }
    if (!cur.empty()) { groups.push_back(cur); gbytes.push_back(size); }
  }
  const int64_t gmax = *std::max_element(gbytes.begin(), gbytes.end());
  if (gmax == 0) return DDP_OK;
  const int64_t slot = (gmax + 255) / 256 * 256;
  void* wsv = nullptr;
  DDP_TRY(alloc_async(&wsv, slot * p, stream, "broadcast workspace allocation"));
  char* ws = static_cast<char*>(wsv);
  ddp_status rc = DDP_OK;
  for (size_t g = 0; g < groups.size() && rc == DDP_OK; ++g) {
    if (gbytes[g] == 0) continue;
    SegBatcher pack(DDP_FLOAT32, 1.0f, stream);
    int64_t pos = 0;
    for (int32_t j : groups[g]) {
      rc = pack.add(T(root, j), ws + root * slot + pos, nbytes[j]);
      if (rc != DDP_OK) break;
      pos += nbytes[j];
    }
    if (rc == DDP_OK) rc = pack.flush();
    if (rc != DDP_OK) break;
    Plan pl;
    pl.op = DDP_OP_BROADCAST; pl.p = p; pl.n = gbytes[g]; pl.root = root;
    for (int r = 0; r < p; ++r) pl.in.push_back(ws + r * slot);
    pl.init();
    rc = pl.run_all(stream);
    if (rc != DDP_OK) break;
    SegBatcher unpack(DDP_FLOAT32, 1.0f, stream);
    for (int r = 0; r < p && rc == DDP_OK; ++r) {
      if (r == root) continue;
      pos = 0;
      for (int32_t j : groups[g]) {
        rc = unpack.add(ws + r * slot + pos, T(r, j), nbytes[j]);
        if (rc != DDP_OK) break;
        pos += nbytes[j];
      }
    }
    if (rc == DDP_OK) rc = unpack.flush();
  }
  const cudaError_t e = cudaFreeAsync(ws, stream);
  if (rc == DDP_OK && e != cudaSuccess) return cuda_fail(e, "broadcast workspace release");
  return rc;
}


ddp_status bucket_allreduce_impl(int32_t p, int32_t k, void* const* grads, const int64_t* numel,
                                 const int64_t* offset, ddp_dtype dtype, float divisor, cudaStream_t stream) {
  DDP_NVTX("ddp_bucket_allreduce");
  DDP_TRY(check_bucket_args(p, k, numel, offset, dtype));
  DDP_TRY(check_divisor(divisor));
  const int es = esize(dtype);
  DDP_CHECK(grads != nullptr || k == 0, DDP_ERR_ARG, "grads array is null");
  std::vector<std::pair<uintptr_t, uintptr_t>> slots, ranges;
  for (int32_t j = 0; j < k; ++j)
    slots.push_back({static_cast<uintptr_t>(offset[j]), static_cast<uintptr_t>(offset[j] + numel[j])});
  DDP_CHECK(disjoint(slots), DDP_ERR_ARG, "bucket slots of different tensors overlap");
  for (int32_t r = 0; r < p; ++r)
    for (int32_t j = 0; j < k; ++j) {
      if (numel[j] == 0) continue;
      const void* g = grads[static_cast<int64_t>(r) * k + j];
      DDP_CHECK(g != nullptr, DDP_ERR_ARG, "grads[" + std::to_string(r * k + j) + "] is null");
      ranges.push_back(range_of(g, numel[j] * es));
    }
  DDP_CHECK(disjoint(ranges), DDP_ERR_ARG, "gradient tensors overlap");
  std::vector<BucketArgs> launches;
  DDP_TRY(plan_bucket_launches(p, k, const_cast<const void* const*>(grads), numel, offset, dtype, divisor, launches));
  return run_bucket_launches(launches, dtype, divisor, stream);
}

ddp_status allreduce_persistent_impl(void* const* bufs, int32_t p, int64_t n, ddp_dtype dtype, float divisor,
                                     int64_t timeout_ns, int32_t fault_rank, int32_t fault_step, int32_t* status,
                                     cudaStream_t stream) {
  DDP_NVTX("ddp_allreduce_persistent");
  DDP_TRY(check_common(p, n, dtype));
  DDP_TRY(check_divisor(divisor));
  DDP_CHECK(timeout_ns >= 0, DDP_ERR_ARG, "timeout_ns must be >= 0");
  const int32_t T = 2 * (p - 1);
  DDP_CHECK(fault_rank == -1 || (fault_rank >= 0 && fault_rank < p && fault_step >= 0 && fault_step < T),
            DDP_ERR_ARG, "fault_rank must be -1 or a rank, fault_step a step in [0, 2(p-1))");
  if (n == 0) {  // a no-op whatever the pointers; the status block still reads "no error"
    if (status) DDP_CUDA(cudaMemsetAsync(status, 0, 4 * sizeof(int32_t), stream), "status reset");
    return DDP_OK;
  }
  DDP_TRY(check_ptrs(const_cast<const void* const*>(bufs), p, "bufs"));
  std::vector<std::pair<uintptr_t, uintptr_t>> rg;
  for (int r = 0; r < p; ++r) rg.push_back(range_of(bufs[r], n * esize(dtype)));
  DDP_CHECK(disjoint(rg), DDP_ERR_ARG, "replica buffers overlap");
  if (status) DDP_CUDA(cudaMemsetAsync(status, 0, 4 * sizeof(int32_t), stream), "status reset");
  if (p == 1) return run_fused(const_cast<const void* const*>(bufs), bufs, 1, n, dtype, divisor, false, 0, false,
                               stream);
  const int max_blocks = ring_persistent_max_blocks();
  DDP_CHECK(max_blocks >= p, DDP_ERR_ARG, "more ranks than co-resident blocks for the persistent ring");
  if (dtype == DDP_BFLOAT16) {
    // fp32 partials for the whole ring (reading A10): widen into a workspace,
    // run the fp32 ring there, round each finished value to bf16 once.
    const int64_t slot = (n * 4 + 255) / 256 * 256;
    void* wsv = nullptr;
    DDP_TRY(alloc_async(&wsv, slot * p, stream, "persistent ring workspace"));
    std::vector<void*> W(p);
    ConvertArgs cv;
    std::memset(&cv, 0, sizeof(cv));
    cv.n = n;
    cv.njobs = p;
    for (int r = 0; r < p; ++r) {
      W[r] = static_cast<char*>(wsv) + slot * r;
      cv.src[r] = bufs[r];
      cv.dst[r] = W[r];
    }
    cudaError_t e = launch_convert(cv, stream);
    ddp_status rc = e == cudaSuccess
                        ? allreduce_persistent_impl(W.data(), p, n, DDP_FLOAT32, divisor, timeout_ns, fault_rank,
                                                   fault_step, status, stream)
                        : cuda_fail(e, "widen launch");
    if (rc == DDP_OK) {
      cv.to_bf16 = 1;
      for (int r = 0; r < p; ++r) { cv.src[r] = W[r]; cv.dst[r] = bufs[r]; }
      e = launch_convert(cv, stream);
      if (e != cudaSuccess) rc = cuda_fail(e, "narrow launch");
    }
    const cudaError_t ef = cudaFreeAsync(wsv, stream);
    if (rc != DDP_OK) return rc;
    if (ef != cudaSuccess) return cuda_fail(ef, "persistent ring workspace release");
    return DDP_OK;
  }
  const int64_t cs = chunk_size(n, p);
  int B = max_blocks / p;
  const int64_t useful = std::max<int64_t>(1, (cs + kThreads * 4 - 1) / (kThreads * 4));
  if (B > useful) B = static_cast<int>(useful);
  PersistArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int r = 0; r < p; ++r) a.buf[r] = bufs[r];
  a.n = n; a.cs = cs; a.divisor = divisor; a.p = p; a.blocks_per_rank = B;
  a.fault_rank = fault_rank; a.fault_step = fault_step;
  a.timeout_ns = timeout_ns > 0 ? timeout_ns : 1000000000LL;
  a.status = status;
  void* flags = nullptr;
  DDP_TRY(alloc_async(&flags, static_cast<size_t>(p) * B * kFlagStride * sizeof(int), stream, "step flags allocation"));
  a.flags = static_cast<int*>(flags);
  cudaError_t e = cudaMemsetAsync(flags, 0, static_cast<size_t>(p) * B * kFlagStride * sizeof(int), stream);
  if (e == cudaSuccess) e = launch_ring_persistent(a, stream);
  const cudaError_t e2 = cudaFreeAsync(flags, stream);
  if (e != cudaSuccess) return cuda_fail(e, "persistent ring launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "step flags release");
  return DDP_OK;
}

}  // namespace host
}  // namespace ddp

// =================================================================== C ABI
extern "C" {

struct ddp_ring {
  Plan plan;
  cudaStream_t stream;
};

ddp_status ddp_bucket_assign(int32_t k, const int64_t* numel, int32_t elem_size,
                             int64_t first_bucket_cap_bytes, int64_t bucket_cap_bytes,
                             ddp_border order, int32_t* n_buckets, int32_t* bucket_of,
                             int64_t* offset, int32_t* bucket_ptr, int32_t* bucket_tensors,
                             int64_t* bucket_numel) {
  DDP_CHECK(k >= 0, DDP_ERR_ARG, "k must be >= 0");
  DDP_CHECK(n_buckets && bucket_ptr, DDP_ERR_ARG, "output arrays are null");
  DDP_CHECK(k == 0 || (numel && bucket_of && offset && bucket_tensors && bucket_numel), DDP_ERR_ARG,
            "input or output arrays are null");
  DDP_CHECK(elem_size > 0, DDP_ERR_ARG, "elem_size must be > 0");
  DDP_CHECK(first_bucket_cap_bytes >= 0 && bucket_cap_bytes >= 0, DDP_ERR_ARG, "caps must be >= 0");
  DDP_CHECK(order == DDP_ORDER_REVERSED || order == DDP_ORDER_REGISTRATION, DDP_ERR_ARG, "unknown order");
  for (int32_t t = 0; t < k; ++t) DDP_CHECK(numel[t] >= 0, DDP_ERR_ARG, "numel must be >= 0");

  std::vector<int32_t> walk(k);
  for (int32_t w = 0; w < k; ++w) walk[w] = (order == DDP_ORDER_REVERSED) ? k - 1 - w : w;
  auto buckets = walk_buckets(walk, numel, elem_size, first_bucket_cap_bytes, bucket_cap_bytes);
  if (order == DDP_ORDER_REGISTRATION) std::reverse(buckets.begin(), buckets.end());
  write_assignment(buckets, numel, n_buckets, bucket_of, offset, bucket_ptr, bucket_tensors, bucket_numel);
  return DDP_OK;
}

ddp_status ddp_bucket_assign_order(int32_t k, const int64_t* numel, int32_t elem_size,
                                   int64_t first_bucket_cap_bytes, int64_t bucket_cap_bytes, const int32_t* walk,
                                   int32_t* n_buckets, int32_t* bucket_of, int64_t* offset, int32_t* bucket_ptr,
                                   int32_t* bucket_tensors, int64_t* bucket_numel) {
  DDP_CHECK(k >= 0, DDP_ERR_ARG, "k must be >= 0");
  DDP_CHECK(n_buckets && bucket_ptr, DDP_ERR_ARG, "output arrays are null");
  DDP_CHECK(k == 0 || (numel && walk && bucket_of && offset && bucket_tensors && bucket_numel), DDP_ERR_ARG,
            "input or output arrays are null");
  DDP_CHECK(elem_size > 0, DDP_ERR_ARG, "elem_size must be > 0");
  DDP_CHECK(first_bucket_cap_bytes >= 0 && bucket_cap_bytes >= 0, DDP_ERR_ARG, "caps must be >= 0");
  std::vector<char> seen(k, 0);
  for (int32_t w = 0; w < k; ++w) {
    DDP_CHECK(walk[w] >= 0 && walk[w] < k && !seen[walk[w]], DDP_ERR_ARG, "walk must be a permutation of 0..k-1");
    seen[walk[w]] = 1;
    DDP_CHECK(numel[walk[w]] >= 0, DDP_ERR_ARG, "numel must be >= 0");
  }
  const auto buckets = walk_buckets(std::vector<int32_t>(walk, walk + k), numel, elem_size, first_bucket_cap_bytes,
                                    bucket_cap_bytes);
  write_assignment(buckets, numel, n_buckets, bucket_of, offset, bucket_ptr, bucket_tensors, bucket_numel);
  return DDP_OK;
}

ddp_status ddp_bucket_flatten(int32_t p, int32_t k, const void* const* grads, const int64_t* numel,
                              const int64_t* offset, void* const* bucket, ddp_dtype dtype,
                              float predivide, cudaStream_t stream) {
  DDP_NVTX("ddp_bucket_flatten");
  DDP_TRY(check_bucket_args(p, k, numel, offset, dtype));
  DDP_TRY(check_divisor(predivide));
  const int es = esize(dtype);
  DDP_TRY(check_bucket_layout(p, k, grads, numel, offset, const_cast<const void* const*>(bucket), es));
  SegBatcher sb(dtype, predivide, stream);
  for (int32_t r = 0; r < p; ++r)
    for (int32_t j = 0; j < k; ++j)
      DDP_TRY(sb.add(grads[static_cast<int64_t>(r) * k + j], static_cast<char*>(bucket[r]) + offset[j] * es,
                     numel[j] * es));
  return sb.flush();
}

ddp_status ddp_bucket_unflatten(int32_t p, int32_t k, const void* const* bucket, const int64_t* numel,
                                const int64_t* offset, void* const* grads, ddp_dtype dtype,
                                cudaStream_t stream) {
  DDP_NVTX("ddp_bucket_unflatten");
  DDP_TRY(check_bucket_args(p, k, numel, offset, dtype));
  const int es = esize(dtype);
  DDP_TRY(check_bucket_layout(p, k, const_cast<const void* const*>(grads), numel, offset, bucket, es));
  SegBatcher sb(dtype, 1.0f, stream);
  for (int32_t r = 0; r < p; ++r)
    for (int32_t j = 0; j < k; ++j)
      DDP_TRY(sb.add(static_cast<const char*>(bucket[r]) + offset[j] * es, grads[static_cast<int64_t>(r) * k + j],
                     numel[j] * es));
  return sb.flush();
}

ddp_status ddp_ring_create(ddp_ring** handle, ddp_op op, void* const* in, void* const* out, int32_t p,
                           int64_t n, ddp_dtype dtype, float divisor, ddp_own own, int32_t root,
                           cudaStream_t stream) {
  DDP_CHECK(handle != nullptr, DDP_ERR_ARG, "handle pointer is null");
  *handle = nullptr;
  DDP_CHECK(op >= DDP_OP_ALLREDUCE && op <= DDP_OP_BROADCAST, DDP_ERR_ARG, "unknown op");
  DDP_TRY(check_common(p, n, op == DDP_OP_BROADCAST ? DDP_FLOAT32 : dtype));
  DDP_CHECK(in != nullptr, DDP_ERR_ARG, "in array is null");
  if (n > 0) DDP_TRY(check_ptrs(const_cast<const void* const*>(in), p, "in"));
  const bool needs_out = (op == DDP_OP_REDUCE_SCATTER || op == DDP_OP_ALLGATHER);
  DDP_CHECK(!needs_out || out != nullptr, DDP_ERR_ARG, "out array is null");
  if (needs_out && n > 0) DDP_TRY(check_ptrs(const_cast<const void* const*>(out), p, "out"));
  if (op == DDP_OP_ALLREDUCE || op == DDP_OP_REDUCE_SCATTER) DDP_TRY(check_divisor(divisor));
  if (op != DDP_OP_BROADCAST) DDP_TRY(check_own(own));
  if (op == DDP_OP_BROADCAST) DDP_CHECK(root >= 0 && root < p, DDP_ERR_ARG, "root out of range");
  if (op == DDP_OP_REDUCE_SCATTER && own == DDP_OWN_RANK)
    DDP_CHECK(n % p == 0, DDP_ERR_NOT_DIVISIBLE,
              "reduce_scatter: " + std::to_string(n) + " elements are not divisible by " + std::to_string(p) + " ranks");
  const int es = (op == DDP_OP_BROADCAST) ? 1 : esize(dtype);
  {
    std::vector<std::pair<uintptr_t, uintptr_t>> rg;
    const int64_t in_bytes = n * es;
    const int64_t out_bytes = (op == DDP_OP_ALLGATHER) ? static_cast<int64_t>(p) * n * es : chunk_size(n, p) * es;
    for (int r = 0; r < p; ++r) {
      rg.push_back(range_of(in[r], in_bytes));
      if (needs_out) rg.push_back(range_of(out[r], out_bytes));
    }
    DDP_CHECK(disjoint(rg), DDP_ERR_ARG, "buffers overlap");
  }
  ddp_ring* h = new ddp_ring();
  Plan& pl = h->plan;
  pl.op = op; pl.p = p; pl.n = n; pl.dt = dtype; pl.divisor = divisor; pl.own = own; pl.root = root;
  pl.in.assign(in, in + p);
  if (needs_out) pl.out.assign(out, out + p);
  pl.init();
  if (n == 0) pl.nsteps = 0;
  h->stream = stream;
  if (pl.needs_ws() && n > 0) {
    void* w = nullptr;
    const ddp_status st = alloc_device(&w, pl.ws_elems() * sizeof(float), "handle workspace allocation");
    if (st != DDP_OK) {
      delete h;
      return st;
    }
    pl.ws = static_cast<float*>(w);
  }
  *handle = h;
  return DDP_OK;
}

int32_t ddp_ring_num_steps(const ddp_ring* h) { return h ? h->plan.nsteps : -1; }
int32_t ddp_ring_steps_done(const ddp_ring* h) { return h ? h->plan.done : -1; }

ddp_status ddp_ring_step(ddp_ring* h) {
  DDP_NVTX("ddp_ring_step");
  DDP_CHECK(h != nullptr, DDP_ERR_ARG, "handle is null");
  return h->plan.step(h->stream);
}

ddp_status ddp_ring_workspace(const ddp_ring* h, void** fp32_partials, int64_t* elems_per_slot) {
  DDP_CHECK(h && fp32_partials && elems_per_slot, DDP_ERR_ARG, "null argument");
  *fp32_partials = h->plan.ws;
  *elems_per_slot = h->plan.ws ? h->plan.cs : 0;
  return DDP_OK;
}

ddp_status ddp_ring_bytes_sent(const ddp_ring* h, int32_t rank, int64_t* bytes) {
  DDP_CHECK(h && bytes, DDP_ERR_ARG, "null argument");
  DDP_CHECK(rank >= 0 && rank < h->plan.p, DDP_ERR_ARG, "rank out of range");
  *bytes = h->plan.sent[rank];
  return DDP_OK;
}

ddp_status ddp_ring_sync(ddp_ring* h) {
  DDP_CHECK(h != nullptr, DDP_ERR_ARG, "handle is null");
  int32_t code = 0;
  return ddp_device_error(h->stream, &code);
}

ddp_status ddp_ring_destroy(ddp_ring* h) {
  if (!h) return DDP_OK;
  cudaError_t e = cudaSuccess;
  if (h->plan.ws) e = cudaFree(h->plan.ws);
  delete h;
  if (e != cudaSuccess) return cuda_fail(e, "handle workspace release");
  return DDP_OK;
}

ddp_status ddp_device_error(cudaStream_t stream, int32_t* code) {
  DDP_CHECK(code != nullptr, DDP_ERR_ARG, "code pointer is null");
  int v = 0;
  DDP_CUDA(read_device_error(stream, &v), "device status read");
  *code = v;
  if (v != 0) return fail(DDP_ERR_TIMEOUT, "a kernel gave up a bounded wait (code " + std::to_string(v) + ")");
  return DDP_OK;
}

int64_t ddp_kernel_launches(void) { return launches(); }

const char* ddp_last_error(void) { return t_error.c_str(); }

const char* ddp_status_string(ddp_status s) {
  switch (s) {
    case DDP_OK: return "DDP_OK";
    case DDP_ERR_ARG: return "DDP_ERR_ARG";
    case DDP_ERR_DTYPE: return "DDP_ERR_DTYPE";
    case DDP_ERR_NOT_DIVISIBLE: return "DDP_ERR_NOT_DIVISIBLE";
    case DDP_ERR_ALIGN: return "DDP_ERR_ALIGN";
    case DDP_ERR_NOMEM: return "DDP_ERR_NOMEM";
    case DDP_ERR_CUDA: return "DDP_ERR_CUDA";
    case DDP_ERR_TIMEOUT: return "DDP_ERR_TIMEOUT";
    case DDP_ERR_STATE: return "DDP_ERR_STATE";
  }
  return "DDP_ERR_UNKNOWN";
}

}  // extern "C"
