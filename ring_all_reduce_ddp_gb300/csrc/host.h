// Host-side internals of the C ABI, shared by its translation units: error
// text, argument checks, the literal schedule of one collective (Plan), the
// tree-shaped schedules, multi-tensor copies, the bucket planner, and the
// bodies of the entry points that the per-call log wraps. Nothing here
// touches data: every step runs in the library's kernels.
#pragma once

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>
#include <utility>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "launch.h"

namespace ddp {
namespace host {

extern thread_local std::string t_error;  // this thread's last error text (ddp_last_error)

#define DDP_CUDA(call, where)                         \
  do {                                                \
    cudaError_t e_ = (call);                          \
    if (e_ != cudaSuccess) return cuda_fail(e_, where); \
  } while (0)

#define DDP_CHECK(cond, code, msg) \
  do {                             \
    if (!(cond)) return fail(code, msg); \
  } while (0)

#define DDP_TRY(expr)                 \
  do {                                \
    const ddp_status rc_ = (expr);    \
    if (rc_ != DDP_OK) return rc_;    \
  } while (0)

// One NVTX range per C-ABI call that enqueues device work, named after the
// entry point, and nested ones per literal ring step and per bucket, for
// timeline tools and ncu's --nvtx filters. Without a tool attached a range
// costs a pointer check.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  // "<what> <i>", e.g. "bucket 3" or "reduce-scatter step 2"
  NvtxRange(const char* what, int i) {
    char buf[64];
    std::snprintf(buf, sizeof(buf), "%s %d", what, i);
    nvtxRangePushA(buf);
  }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
#define DDP_NVTX(name) ::ddp::host::NvtxRange nvtx_range_(name)
#define DDP_NVTX_I(what, i) ::ddp::host::NvtxRange nvtx_range_i_(what, i)

struct Plan;

// A stream-ordered temporary (cudaMallocAsync on s). A failure returns
// DDP_ERR_NOMEM with `what` in the error text, and clears CUDA's last error:
// an allocation failure is not sticky and must not surface at a later launch.
ddp_status alloc_async(void** ptr, size_t bytes, cudaStream_t s, const char* what);
// The same for a handle's long-lived memory (cudaMalloc).
ddp_status alloc_device(void** ptr, size_t bytes, const char* what);

ddp_status fail(ddp_status s, const std::string& msg);
ddp_status cuda_fail(cudaError_t e, const char* where);
int esize(ddp_dtype dt);
ddp_status check_common(int32_t p, int64_t n, int dtype);
ddp_status check_divisor(float d);
ddp_status check_ptrs(const void* const* v, int32_t count, const char* what);
bool disjoint(std::vector<std::pair<uintptr_t, uintptr_t>> r);
std::pair<uintptr_t, uintptr_t> range_of(const void* ptr, int64_t bytes);
int64_t chunk_size(int64_t n, int32_t p);
bool same_align16(const void* const* v, int32_t count);
ddp_status run_fused(const void* const* in, void* const* out, int32_t p, int64_t n, ddp_dtype dt,
                     float divisor, bool scatter, int shift, bool staged, cudaStream_t s,
                     bool hop_round = false);
ddp_status run_plan_once(Plan& pl, cudaStream_t s);
ddp_status check_algo(int algo);
bool is_tree_algo(int algo);
ddp_status run_tree_allreduce(float* const* B, int32_t p, int64_t n, float divisor, int algo, cudaStream_t s);
ddp_status check_own(int own);
ddp_status check_bucket_args(int32_t p, int32_t k, const int64_t* numel, const int64_t* offset, int dtype);
ddp_status check_bucket_layout(int32_t p, int32_t k, const void* const* grads, const int64_t* numel,
                               const int64_t* offset, const void* const* bucket, int es);
ddp_status plan_bucket_launches(int32_t p, int32_t k, const void* const* grads, const int64_t* numel,
                                const int64_t* offset, ddp_dtype dt, float divisor,
                                std::vector<BucketArgs>& out);
ddp_status run_bucket_launches(std::vector<BucketArgs>& launches, ddp_dtype dt, float divisor, cudaStream_t s,
                                int32_t max_blocks = 0);
void write_assignment(const std::vector<std::vector<int32_t>>& buckets, const int64_t* numel, int32_t* n_buckets,
                      int32_t* bucket_of, int64_t* offset, int32_t* bucket_ptr, int32_t* bucket_tensors,
                      int64_t* bucket_numel);
std::vector<std::vector<int32_t>> walk_buckets(const std::vector<int32_t>& walk, const int64_t* numel,
                                               int32_t elem_size, int64_t first_cap, int64_t cap);

// The literal schedule of one collective, one step at a time.
struct Plan {
  ddp_op op = DDP_OP_ALLREDUCE;
  int32_t p = 1;
  int64_t n = 0;  // AR/RS: elements per input; AG: elements per input (m); BC: bytes
  ddp_dtype dt = DDP_FLOAT32;
  float divisor = 1.0f;
  ddp_own own = DDP_OWN_RANK;
  int32_t root = 0;
  std::vector<void*> in, out;
  int64_t cs = 0;
  float* ws = nullptr;
  bool ws_async = false;
  bool hop_round = false;  // bf16 all-reduce: round every partial to bf16
  int32_t nsteps = 0, done = 0;
  std::vector<int64_t> sent;

  bool needs_ws() const {
    return p > 1 && ((op == DDP_OP_ALLREDUCE && dt == DDP_BFLOAT16) || op == DDP_OP_REDUCE_SCATTER);
  }
  int64_t ws_elems() const { return 2 * static_cast<int64_t>(p) * cs; }

  void init() {
    cs = (op == DDP_OP_ALLGATHER) ? n : chunk_size(n, p);
    switch (op) {
      case DDP_OP_ALLREDUCE: nsteps = p == 1 ? 1 : 2 * (p - 1); break;
      case DDP_OP_REDUCE_SCATTER:
      case DDP_OP_ALLGATHER: nsteps = p == 1 ? 1 : p - 1; break;
      case DDP_OP_BROADCAST: {
        int steps = 0;
        for (int64_t span = 1; span < p; span *= 2) ++steps;
        nsteps = steps;
        break;
      }
    }
    sent.assign(p, 0);
  }

  ddp_status step(cudaStream_t s) {
    if (done >= nsteps) return fail(DDP_ERR_STATE, "all steps of this schedule are already enqueued");
    const int st = done;
    DDP_NVTX_I(op == DDP_OP_BROADCAST ? "broadcast step"
               : (op == DDP_OP_ALLGATHER || (op == DDP_OP_ALLREDUCE && st >= p - 1 && p > 1)) ? "all-gather step"
                                                                                             : "reduce-scatter step",
               st);
    const int es = (op == DDP_OP_BROADCAST) ? 1 : esize(dt);
    ddp_status rc = DDP_OK;
    if (op == DDP_OP_ALLREDUCE) {
      if (p == 1) {
        rc = run_fused(in.data(), in.data(), 1, n, dt, divisor, false, 0, false, s);
      } else if (st < p - 1) {
        RingStepArgs a;
        std::memset(&a, 0, sizeof(a));
        for (int r = 0; r < p; ++r) { a.x[r] = in[r]; a.out[r] = in[r]; }
        a.w = ws; a.n = n; a.cs = cs; a.divisor = divisor; a.p = p; a.step = st;
        a.shift = 0; a.last = (st == p - 2); a.out_rel = 0; a.hop_round = hop_round ? 1 : 0;
        DDP_CUDA(dt == DDP_FLOAT32 ? launch_rs_step_inplace_f32(a, s) : launch_rs_step_ws(a, dt, s),
                 "reduce-scatter step launch");
        for (int r = 0; r < p; ++r) sent[r] += cs * es;
      } else {
        const int k = st - (p - 1);
        PairCopyArgs a;
        std::memset(&a, 0, sizeof(a));
        for (int r = 0; r < p; ++r) {
          const int c = ((r + 1 - k) % p + p) % p;
          const int64_t lo = std::min(n, c * cs), hi = std::min(n, (c + 1) * cs);
          a.src[r] = static_cast<const char*>(in[r]) + lo * es;
          a.dst[r] = static_cast<char*>(in[(r + 1) % p]) + lo * es;
          a.nbytes[r] = (hi - lo) * es;
          sent[r] += cs * es;
        }
        a.njobs = p;
        DDP_CUDA(launch_pair_copy(a, s), "all-gather step launch");
      }
    } else if (op == DDP_OP_REDUCE_SCATTER) {
      if (p == 1) {
        rc = run_fused(in.data(), out.data(), 1, n, dt, divisor, true, 0, false, s);
      } else {
        RingStepArgs a;
        std::memset(&a, 0, sizeof(a));
        for (int r = 0; r < p; ++r) { a.x[r] = in[r]; a.out[r] = out[r]; }
        a.w = ws; a.n = n; a.cs = cs; a.divisor = divisor; a.p = p; a.step = st;
        a.shift = (own == DDP_OWN_RANK) ? 1 : 0; a.last = (st == p - 2); a.out_rel = 1;
        DDP_CUDA(launch_rs_step_ws(a, dt, s), "reduce-scatter step launch");
        for (int r = 0; r < p; ++r) sent[r] += cs * es;
      }
    } else if (op == DDP_OP_ALLGATHER) {
      const int64_t mb = n * es;
      if (p == 1) {
        PairCopyArgs a;
        std::memset(&a, 0, sizeof(a));
        a.src[0] = static_cast<const char*>(in[0]); a.dst[0] = static_cast<char*>(out[0]);
        a.nbytes[0] = mb; a.njobs = 1;
        DDP_CUDA(launch_pair_copy(a, s), "all-gather copy launch");
      } else {
        auto held = [&](int r) { return own == DDP_OWN_RANK ? r : (r + 1) % p; };
        if (st == 0) {  // each rank's own chunk goes to its place in its output
          PairCopyArgs a;
          std::memset(&a, 0, sizeof(a));
          for (int r = 0; r < p; ++r) {
            a.src[r] = static_cast<const char*>(in[r]);
            a.dst[r] = static_cast<char*>(out[r]) + held(r) * mb;
            a.nbytes[r] = mb;
          }
          a.njobs = p;
          DDP_CUDA(launch_pair_copy(a, s), "all-gather placement launch");
        }
        PairCopyArgs a;
        std::memset(&a, 0, sizeof(a));
        for (int r = 0; r < p; ++r) {
          const int c = ((held(r) - st) % p + p) % p;
          a.src[r] = (st == 0) ? static_cast<const char*>(in[r]) : static_cast<const char*>(out[r]) + c * mb;
          a.dst[r] = static_cast<char*>(out[(r + 1) % p]) + c * mb;
          a.nbytes[r] = mb;
          sent[r] += mb;
        }
        a.njobs = p;
        DDP_CUDA(launch_pair_copy(a, s), "all-gather step launch");
      }
    } else {  // broadcast: doubling tree
      const int64_t span = int64_t(1) << st;
      PairCopyArgs a;
      std::memset(&a, 0, sizeof(a));
      int jobs = 0;
      for (int64_t v = 0; v < span; ++v) {
        if (v + span >= p) continue;
        const int src = static_cast<int>((root + v) % p), dst = static_cast<int>((root + v + span) % p);
        a.src[jobs] = static_cast<const char*>(in[src]);
        a.dst[jobs] = static_cast<char*>(in[dst]);
        a.nbytes[jobs] = n;
        sent[src] += n;
        ++jobs;
      }
      a.njobs = jobs;
      DDP_CUDA(launch_pair_copy(a, s), "broadcast step launch");
    }
    if (rc != DDP_OK) return rc;
    ++done;
    return DDP_OK;
  }

  ddp_status run_all(cudaStream_t s) {
    while (done < nsteps) {
      const ddp_status rc = step(s);
      if (rc != DDP_OK) return rc;
    }
    return DDP_OK;
  }
};


// Multi-tensor copies, split into launches of at most kSegCap segments.
struct SegBatcher {
  SegCopyArgs a;
  ddp_dtype dt;
  cudaStream_t s;
  SegBatcher(ddp_dtype dt_, float predivide, cudaStream_t s_) : dt(dt_), s(s_) {
    std::memset(&a, 0, sizeof(a));
    a.elem_size = esize(dt_);
    a.predivide = predivide;
  }
  ddp_status add(const void* src, void* dst, int64_t bytes) {
    if (bytes <= 0) return DDP_OK;
    const int64_t tiles = (bytes + kSegTileBytes - 1) / kSegTileBytes;
    if (a.nseg == kSegCap || static_cast<int64_t>(a.tile0[a.nseg]) + tiles > 0x7FFFFFFF) DDP_TRY(flush());
    DDP_CHECK(tiles <= 0x7FFFFFFF, DDP_ERR_ARG, "tensor too large");
    a.src[a.nseg] = static_cast<const char*>(src);
    a.dst[a.nseg] = static_cast<char*>(dst);
    a.bytes[a.nseg] = bytes;
    a.tile0[a.nseg + 1] = a.tile0[a.nseg] + static_cast<int32_t>(tiles);
    ++a.nseg;
    return DDP_OK;
  }
  ddp_status flush() {
    if (a.nseg == 0) return DDP_OK;
    DDP_CUDA(launch_seg_copy(a, dt, s), "segment copy launch");
    const int elem = a.elem_size;
    const float pd = a.predivide;
    std::memset(&a, 0, sizeof(a));
    a.elem_size = elem;
    a.predivide = pd;
    return DDP_OK;
  }
};


// The entry points' bodies, wrapped by the exported functions that add the
// per-call log (calllog.cu).
ddp_status allreduce_impl(void* const* bufs, int32_t p, int64_t n, ddp_dtype dtype, float divisor, ddp_algo algo,
                          cudaStream_t stream);
ddp_status allreduce_ex_impl(void* const* bufs, int32_t p, int64_t n, ddp_dtype dtype, float divisor,
                             ddp_algo algo, uint32_t flags, cudaStream_t stream);
ddp_status allreduce_persistent_impl(void* const* bufs, int32_t p, int64_t n, ddp_dtype dtype, float divisor,
                                     int64_t timeout_ns, int32_t fault_rank, int32_t fault_step, int32_t* status,
                                     cudaStream_t stream);
ddp_status reduce_scatter_impl(const void* const* in, void* const* out, int32_t p, int64_t n, ddp_dtype dtype,
                               float divisor, ddp_own own, ddp_algo algo, cudaStream_t stream);
ddp_status allgather_impl(const void* const* in, void* const* out, int32_t p, int64_t m, ddp_dtype dtype,
                          ddp_own own, ddp_algo algo, cudaStream_t stream);
ddp_status broadcast_impl(void* const* bufs, int32_t p, int64_t nbytes, int32_t root, ddp_algo algo,
                          cudaStream_t stream);
ddp_status broadcast_coalesced_impl(int32_t p, int32_t k, void* const* tensors, const int64_t* nbytes,
                                    int32_t root, int64_t bucket_cap_bytes, ddp_algo algo, cudaStream_t stream);
ddp_status bucket_allreduce_impl(int32_t p, int32_t k, void* const* grads, const int64_t* numel,
                                 const int64_t* offset, ddp_dtype dtype, float divisor, cudaStream_t stream);
ddp_status reducer_sync_impl(ddp_reducer* h, float divisor, float predivide, ddp_algo algo, ddp_sync_mode mode,
                             cudaStream_t stream);
ddp_status reducer_step_impl(ddp_reducer* h, float divisor, cudaStream_t stream);
// Bytes of one replica's buffers attached for ddp_reducer_step (0 if none).
int64_t reducer_buffer_bytes(const ddp_reducer* h);
// A reducer's replica count, dtype and bucket sizes (elements), for the log.
void reducer_shape(const ddp_reducer* h, int32_t* p, ddp_dtype* dt, std::vector<int64_t>* bucket_numel);

}  // namespace host
}  // namespace ddp
