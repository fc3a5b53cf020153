// The C ABI (include/ddp_ring.h): the exported collectives, each a thin
// wrapper that runs its body (*_impl) and appends the per-call log record.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <string>
#include <vector>

#include "host.h"

using namespace ddp;
using namespace ddp::host;

// ================================================================ call log
// With DDP_RING_LOG=<path> in the environment, every collective call appends
// one JSON line to <path>: the entry point, algo, p, element count, dtype,
// the algorithmic bytes (every replica's input read once and every output
// written once), the bytes each simulated rank sends in the method's own
// schedule (the ring's 2(p-1) chunk sends for an all-reduce, as the pages'
// per-rank byte counter counts them), the status, and the call's device time
// from events around it. Timing waits for the call to finish, so a logged
// call is synchronous; inside a stream capture the time is left out. Without
// the variable nothing is recorded and nothing waits.
namespace {

std::mutex g_log_mu;
std::FILE* g_log = nullptr;
bool g_log_checked = false;

std::FILE* log_file() {
  std::lock_guard<std::mutex> lk(g_log_mu);
  if (!g_log_checked) {
    g_log_checked = true;
    const char* path = std::getenv("DDP_RING_LOG");
    if (path && *path) g_log = std::fopen(path, "a");
  }
  return g_log;
}

int ceil_log2(int32_t p) {
  int L = 0;
  while ((int64_t(1) << L) < p) ++L;
  return L;
}

// Events around one call, when the log is on and the stream is not capturing.
class CallTimer {
 public:
  explicit CallTimer(cudaStream_t s) : s_(s), on_(log_file() != nullptr) {
    if (!on_) return;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s_, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
      (void)cudaGetLastError();
      return;
    }
    if (cudaEventCreate(&e0_) != cudaSuccess || cudaEventCreate(&e1_) != cudaSuccess ||
        cudaEventRecord(e0_, s_) != cudaSuccess) {
      (void)cudaGetLastError();
      release();
      return;
    }
    timing_ = true;
  }
  ~CallTimer() { release(); }
  CallTimer(const CallTimer&) = delete;
  CallTimer& operator=(const CallTimer&) = delete;

  bool on() const { return on_; }

  // Device microseconds of the call, or a negative number when not timed.
  double finish(ddp_status st) {
    if (!timing_ || st != DDP_OK) return -1.0;
    float ms = 0.f;
    if (cudaEventRecord(e1_, s_) != cudaSuccess || cudaEventSynchronize(e1_) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0_, e1_) != cudaSuccess) {
      (void)cudaGetLastError();
      return -1.0;
    }
    return 1e3 * static_cast<double>(ms);
  }

 private:
  void release() {
    if (e0_) cudaEventDestroy(e0_);
    if (e1_) cudaEventDestroy(e1_);
    e0_ = e1_ = nullptr;
  }
  cudaStream_t s_;
  bool on_;
  bool timing_ = false;
  cudaEvent_t e0_ = nullptr, e1_ = nullptr;
};

void log_call(CallTimer& t, const char* op, int algo, int32_t p, int64_t n, ddp_dtype dt, int64_t alg_bytes,
              int64_t rank_bytes, ddp_status st) {
  if (!t.on()) return;
  const double us = t.finish(st);
  char line[512];
  int len = std::snprintf(line, sizeof(line),
                          "{\"op\": \"%s\", \"algo\": %d, \"p\": %d, \"n\": %lld, \"dtype\": \"%s\", "
                          "\"bytes_algorithmic\": %lld, \"bytes_per_rank\": %lld, \"status\": \"%s\", ",
                          op, algo, p, static_cast<long long>(n), dt == DDP_BFLOAT16 ? "bf16" : "f32",
                          static_cast<long long>(alg_bytes), static_cast<long long>(rank_bytes),
                          ddp_status_string(st));
  if (len < 0 || len >= static_cast<int>(sizeof(line))) return;
  if (us >= 0.0)
    len += std::snprintf(line + len, sizeof(line) - len, "\"elapsed_us\": %.3f}\n", us);
  else
    len += std::snprintf(line + len, sizeof(line) - len, "\"elapsed_us\": null}\n");
  std::lock_guard<std::mutex> lk(g_log_mu);
  if (g_log) {
    std::fputs(line, g_log);
    std::fflush(g_log);
  }
}

// Bytes one simulated rank sends in an all-reduce of n elements, in the
// schedule the algo names (the maximum over ranks where ranks differ).
int64_t allreduce_rank_bytes(int algo, int32_t p, int64_t n, int es) {
  if (p <= 1 || n <= 0) return 0;
  const int64_t cs = chunk_size(n, p);
  const int L = ceil_log2(p);
  switch (algo) {
    case DDP_ALGO_RECURSIVE_DOUBLING: return static_cast<int64_t>(L) * n * es;
    case DDP_ALGO_TREE: return static_cast<int64_t>(L) * n * es;  // the root sends at every broadcast level
    default: return 2 * static_cast<int64_t>(p - 1) * cs * es;    // the ring's chunks (Rabenseifner's equal them)
  }
}

}  // namespace

extern "C" {

ddp_status ddp_allreduce(void* const* bufs, int32_t p, int64_t n, ddp_dtype dtype, float divisor, ddp_algo algo,
                         cudaStream_t stream) {
  CallTimer t(stream);
  const ddp_status st = allreduce_impl(bufs, p, n, dtype, divisor, algo, stream);
  const int es = esize(dtype);
  log_call(t, "ddp_allreduce", algo, p, n, dtype, 2 * static_cast<int64_t>(p) * n * es,
           allreduce_rank_bytes(algo, p, n, es), st);
  return st;
}

ddp_status ddp_allreduce_ex(void* const* bufs, int32_t p, int64_t n, ddp_dtype dtype, float divisor,
                            ddp_algo algo, uint32_t flags, cudaStream_t stream) {
  CallTimer t(stream);
  const ddp_status st = allreduce_ex_impl(bufs, p, n, dtype, divisor, algo, flags, stream);
  const int es = esize(dtype);
  log_call(t, "ddp_allreduce_ex", algo, p, n, dtype, 2 * static_cast<int64_t>(p) * n * es,
           allreduce_rank_bytes(algo, p, n, es), st);
  return st;
}

ddp_status ddp_allreduce_persistent(void* const* bufs, int32_t p, int64_t n, ddp_dtype dtype, float divisor,
                                    int64_t timeout_ns, int32_t fault_rank, int32_t fault_step, int32_t* status,
                                    cudaStream_t stream) {
  CallTimer t(stream);
  const ddp_status st =
      allreduce_persistent_impl(bufs, p, n, dtype, divisor, timeout_ns, fault_rank, fault_step, status, stream);
  const int es = esize(dtype);
  log_call(t, "ddp_allreduce_persistent", DDP_ALGO_RING_STEPS, p, n, dtype, 2 * static_cast<int64_t>(p) * n * es,
           allreduce_rank_bytes(DDP_ALGO_RING_STEPS, p, n, es), st);
  return st;
}

ddp_status ddp_reduce_scatter(const void* const* in, void* const* out, int32_t p, int64_t n, ddp_dtype dtype,
                              float divisor, ddp_own own, ddp_algo algo, cudaStream_t stream) {
  CallTimer t(stream);
  const ddp_status st = reduce_scatter_impl(in, out, p, n, dtype, divisor, own, algo, stream);
  const int es = esize(dtype);
  const int64_t cs = (p > 0 && n > 0) ? chunk_size(n, p) : 0;
  log_call(t, "ddp_reduce_scatter", algo, p, n, dtype, (static_cast<int64_t>(p) + 1) * n * es,
           p > 1 ? static_cast<int64_t>(p - 1) * cs * es : 0, st);
  return st;
}

ddp_status ddp_allgather(const void* const* in, void* const* out, int32_t p, int64_t m, ddp_dtype dtype,
                         ddp_own own, ddp_algo algo, cudaStream_t stream) {
  CallTimer t(stream);
  const ddp_status st = allgather_impl(in, out, p, m, dtype, own, algo, stream);
  const int es = esize(dtype);
  const int64_t whole = static_cast<int64_t>(p) * m;  // elements of the gathered buffer
  log_call(t, "ddp_allgather", algo, p, whole, dtype, (static_cast<int64_t>(p) + 1) * whole * es,
           p > 1 ? static_cast<int64_t>(p - 1) * m * es : 0, st);
  return st;
}

ddp_status ddp_broadcast(void* const* bufs, int32_t p, int64_t nbytes, int32_t root, ddp_algo algo,
                         cudaStream_t stream) {
  CallTimer t(stream);
  const ddp_status st = broadcast_impl(bufs, p, nbytes, root, algo, stream);
  log_call(t, "ddp_broadcast", algo, p, nbytes, DDP_FLOAT32, static_cast<int64_t>(p) * nbytes,
           static_cast<int64_t>(ceil_log2(p)) * nbytes, st);
  return st;
}

ddp_status ddp_broadcast_coalesced(int32_t p, int32_t k, void* const* tensors, const int64_t* nbytes, int32_t root,
                                   int64_t bucket_cap_bytes, ddp_algo algo, cudaStream_t stream) {
  CallTimer t(stream);
  const ddp_status st = broadcast_coalesced_impl(p, k, tensors, nbytes, root, bucket_cap_bytes, algo, stream);
  int64_t total = 0;
  if (st == DDP_OK && nbytes)
    for (int32_t j = 0; j < k; ++j) total += nbytes[j];
  log_call(t, "ddp_broadcast_coalesced", algo, p, total, DDP_FLOAT32, static_cast<int64_t>(p) * total,
           static_cast<int64_t>(ceil_log2(p)) * total, st);
  return st;
}

ddp_status ddp_bucket_allreduce(int32_t p, int32_t k, void* const* grads, const int64_t* numel,
                                const int64_t* offset, ddp_dtype dtype, float divisor, cudaStream_t stream) {
  CallTimer t(stream);
  const ddp_status st = bucket_allreduce_impl(p, k, grads, numel, offset, dtype, divisor, stream);
  int64_t n = 0, extent = 0;
  if (st == DDP_OK && numel && offset)
    for (int32_t j = 0; j < k; ++j) {
      n += numel[j];
      extent = std::max(extent, offset[j] + numel[j]);
    }
  const int es = esize(dtype);
  log_call(t, "ddp_bucket_allreduce", DDP_ALGO_FUSED, p, n, dtype, 2 * static_cast<int64_t>(p) * n * es,
           allreduce_rank_bytes(DDP_ALGO_FUSED, p, extent, es), st);
  return st;
}

ddp_status ddp_reducer_sync(ddp_reducer* h, float divisor, float predivide, ddp_algo algo, ddp_sync_mode mode,
                            cudaStream_t stream) {
  CallTimer t(stream);
  const ddp_status st = reducer_sync_impl(h, divisor, predivide, algo, mode, stream);
  int32_t p = 0;
  ddp_dtype dt = DDP_FLOAT32;
  std::vector<int64_t> bn;
  reducer_shape(h, &p, &dt, &bn);
  int64_t n = 0, rank_bytes = 0;
  for (int64_t nb : bn) {
    n += nb;
    rank_bytes += allreduce_rank_bytes(algo, p, nb, esize(dt));
  }
  const int64_t ar = 2 * static_cast<int64_t>(p) * n * esize(dt);
  // the flatten form also copies every gradient into its bucket and back: 4pM more
  log_call(t, "ddp_reducer_sync", algo, p, n, dt, mode == DDP_SYNC_FLATTEN ? 3 * ar : ar, rank_bytes, st);
  return st;
}

ddp_status ddp_reducer_step(ddp_reducer* h, float divisor, cudaStream_t stream) {
  CallTimer t(stream);
  const ddp_status st = reducer_step_impl(h, divisor, stream);
  int32_t p = 0;
  ddp_dtype dt = DDP_FLOAT32;
  std::vector<int64_t> bn;
  reducer_shape(h, &p, &dt, &bn);
  int64_t n = 0, rank_bytes = 0;
  for (int64_t nb : bn) {
    n += nb;
    rank_bytes += allreduce_rank_bytes(DDP_ALGO_FUSED, p, nb, esize(dt));
  }
  const int64_t buf = reducer_buffer_bytes(h);
  // the sync reads and writes every replica once (2pM); the broadcast reads the
  // root's buffers once and writes the p - 1 others (p B)
  log_call(t, "ddp_reducer_step", DDP_ALGO_FUSED, p, n, dt, 2 * static_cast<int64_t>(p) * n * esize(dt) + p * buf,
           rank_bytes + static_cast<int64_t>(ceil_log2(p)) * buf, st);
  return st;
}

}  // extern "C"
