// The C ABI (include/ddp_ring.h): argument checks, the host planner (bucket
// assignment, chunk plan, coalescing groups, the literal schedule's steps) and
// dispatch to the kernels. Everything that touches the data runs in the
// library's kernels; this file only plans and launches.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "launch.h"

using namespace ddp;

namespace {

thread_local std::string t_error;

// One NVTX range per C-ABI call that enqueues device work, named after the
// entry point, for timeline tools and ncu's --nvtx filters. Without a tool
// attached a range costs a pointer check.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
#define DDP_NVTX(name) NvtxRange nvtx_range_(name)

ddp_status fail(ddp_status s, const std::string& msg) {
  t_error = msg;
  return s;
}

ddp_status cuda_fail(cudaError_t e, const char* where) {
  t_error = std::string(where) + ": " + cudaGetErrorString(e);
  return DDP_ERR_CUDA;
}

#define DDP_CUDA(call, where)                         \
  do {                                                \
    cudaError_t e_ = (call);                          \
    if (e_ != cudaSuccess) return cuda_fail(e_, where); \
  } while (0)

#define DDP_CHECK(cond, code, msg) \
  do {                             \
    if (!(cond)) return fail(code, msg); \
  } while (0)

int esize(ddp_dtype dt) { return dt == DDP_FLOAT32 ? 4 : 2; }

ddp_status check_common(int32_t p, int64_t n, int dtype) {
  DDP_CHECK(p >= 1 && p <= DDP_MAX_P, DDP_ERR_ARG, "p must be in [1, " + std::to_string(DDP_MAX_P) + "]");
  DDP_CHECK(n >= 0, DDP_ERR_ARG, "element count must be >= 0");
  DDP_CHECK(dtype == DDP_FLOAT32 || dtype == DDP_BFLOAT16, DDP_ERR_DTYPE, "dtype must be DDP_FLOAT32 or DDP_BFLOAT16");
  return DDP_OK;
}

ddp_status check_divisor(float d) {
  DDP_CHECK(std::isfinite(d) && d != 0.0f, DDP_ERR_ARG, "divisor must be finite and non-zero");
  return DDP_OK;
}

ddp_status check_ptrs(const void* const* v, int32_t count, const char* what) {
  DDP_CHECK(v != nullptr, DDP_ERR_ARG, std::string(what) + " array is null");
  for (int32_t i = 0; i < count; ++i)
    DDP_CHECK(v[i] != nullptr, DDP_ERR_ARG, std::string(what) + "[" + std::to_string(i) + "] is null");
  return DDP_OK;
}

// Byte ranges [begin, end) must be pairwise disjoint (empty ranges ignored).
bool disjoint(std::vector<std::pair<uintptr_t, uintptr_t>> r) {
  r.erase(std::remove_if(r.begin(), r.end(), [](const auto& x) { return x.second <= x.first; }), r.end());
  std::sort(r.begin(), r.end());
  for (size_t i = 1; i < r.size(); ++i)
    if (r[i].first < r[i - 1].second) return false;
  return true;
}

std::pair<uintptr_t, uintptr_t> range_of(const void* ptr, int64_t bytes) {
  const uintptr_t b = reinterpret_cast<uintptr_t>(ptr);
  return {b, b + static_cast<uintptr_t>(bytes)};
}

int64_t chunk_size(int64_t n, int32_t p) { return n > 0 ? (n + p - 1) / p : 0; }

bool same_align16(const void* const* v, int32_t count) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(v[0]) & 15u;
  for (int32_t i = 1; i < count; ++i)
    if ((reinterpret_cast<uintptr_t>(v[i]) & 15u) != a0) return false;
  return true;
}

// ------------------------------------------------------------------ planner

// Fused one-pass reduction of p replicas.
ddp_status run_fused(const void* const* in, void* const* out, int32_t p, int64_t n, ddp_dtype dt,
                     float divisor, bool scatter, int shift, bool staged, cudaStream_t s,
                     bool hop_round = false) {
  FusedArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int j = 0; j < 2 * p; ++j) a.src[j] = in[j % p];
  for (int r = 0; r < p; ++r) a.dst[r] = out[r];
  a.n = n;
  a.cs = chunk_size(n, p);
  a.divisor = divisor;
  a.p = p;
  a.scatter = scatter ? 1 : 0;
  a.shift = shift;
  // All-reduce reads and writes the same p replicas; a scatter's outputs are
  // checked per chunk in the kernel.
  a.same_align = same_align16(in, p) ? 1 : 0;
  a.hop_round = hop_round ? 1 : 0;
  DDP_CUDA(launch_fused_reduce(a, dt, staged, s), "fused reduction launch");
  return DDP_OK;
}

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

// One-shot literal schedule with a stream-ordered temporary workspace.
ddp_status run_plan_once(Plan& pl, cudaStream_t s) {
  pl.init();
  if (pl.needs_ws()) {
    void* w = nullptr;
    DDP_CUDA(cudaMallocAsync(&w, pl.ws_elems() * sizeof(float), s), "workspace allocation");
    pl.ws = static_cast<float*>(w);
  }
  const ddp_status rc = pl.run_all(s);
  if (pl.ws) {
    const cudaError_t e = cudaFreeAsync(pl.ws, s);
    pl.ws = nullptr;
    if (rc == DDP_OK && e != cudaSuccess) return cuda_fail(e, "workspace release");
  }
  return rc;
}

ddp_status check_algo(int algo) {
  DDP_CHECK(algo == DDP_ALGO_FUSED || algo == DDP_ALGO_RING_STEPS || algo == DDP_ALGO_FUSED_LDST ||
                algo == DDP_ALGO_FUSED_TMA,
            DDP_ERR_ARG, "unknown algo (the tree-shaped algos are for ddp_allreduce only)");
  return DDP_OK;
}

bool is_tree_algo(int algo) {
  return algo == DDP_ALGO_RECURSIVE_DOUBLING || algo == DDP_ALGO_RABENSEIFNER || algo == DDP_ALGO_TREE;
}

// The tree-shaped literal all-reduces, fp32 in place. See the oracle's
// readings: recursive doubling pairs r, r ^ 2^j; Rabenseifner halves with
// distance d = p / 2^(k+1), the rank with bit d clear keeping the lower half,
// then doubles back; the tree reduces binomially to rank 0 and broadcasts.
ddp_status run_tree_allreduce(float* const* B, int32_t p, int64_t n, float divisor, int algo, cudaStream_t s) {
  auto pow2 = [](int32_t x) { return x >= 1 && (x & (x - 1)) == 0; };
  if (algo != DDP_ALGO_TREE)
    DDP_CHECK(pow2(p), DDP_ERR_ARG, "recursive doubling and Rabenseifner need p a power of two");
  if (p == 1) return run_fused(reinterpret_cast<const void* const*>(B), reinterpret_cast<void* const*>(B), 1, n,
                               DDP_FLOAT32, divisor, false, 0, false, s);
  int L = 0;
  while ((int64_t(1) << L) < p) ++L;
  if (algo == DDP_ALGO_RECURSIVE_DOUBLING) {
    for (int j = 0; j < L; ++j) {
      const int d = 1 << j;
      PairAddArgs a;
      std::memset(&a, 0, sizeof(a));
      for (int r = 0; r < p; ++r) {
        if (r & d) continue;
        const int k = a.njobs++;
        a.a[k] = B[r]; a.b[k] = B[r | d]; a.d1[k] = B[r]; a.d2[k] = B[r | d];
        a.lo[k] = 0; a.hi[k] = n;
      }
      a.divide = (j == L - 1); a.divisor = divisor;
      DDP_CUDA(launch_pair_add(a, s), "recursive doubling step launch");
    }
    return DDP_OK;
  }
  if (algo == DDP_ALGO_RABENSEIFNER) {
    const int64_t cs = chunk_size(n, p);
    auto clip = [&](int64_t chunk) { return std::min(n, chunk * cs); };
    for (int k = 0; k < L; ++k) {  // recursive halving
      const int d = p >> (k + 1);
      PairAddArgs a;
      std::memset(&a, 0, sizeof(a));
      for (int r = 0; r < p; ++r) {
        if (r & d) continue;
        const int64_t lo = r & ~(2 * d - 1);  // the pair's common segment, in chunks
        const int q = r | d;
        int j = a.njobs++;
        a.a[j] = B[r]; a.b[j] = B[q]; a.d1[j] = B[r]; a.lo[j] = clip(lo); a.hi[j] = clip(lo + d);
        j = a.njobs++;
        a.a[j] = B[r]; a.b[j] = B[q]; a.d1[j] = B[q]; a.lo[j] = clip(lo + d); a.hi[j] = clip(lo + 2 * d);
      }
      a.divide = (k == L - 1); a.divisor = divisor;
      DDP_CUDA(launch_pair_add(a, s), "recursive halving step launch");
    }
    for (int k = 0; k < L; ++k) {  // recursive doubling of the owned segments
      const int d = 1 << k;
      PairCopyArgs a;
      std::memset(&a, 0, sizeof(a));
      for (int r = 0; r < p; ++r) {
        const int64_t lo = r & ~(d - 1);  // rank r's owned segment (d chunks)
        a.src[r] = reinterpret_cast<const char*>(B[r] + clip(lo));
        a.dst[r] = reinterpret_cast<char*>(B[r ^ d] + clip(lo));
        a.nbytes[r] = (clip(lo + d) - clip(lo)) * 4;
      }
      a.njobs = p;
      DDP_CUDA(launch_pair_copy(a, s), "recursive doubling copy launch");
    }
    return DDP_OK;
  }
  // tree: binomial reduce to rank 0, then the doubling-tree broadcast from rank 0
  for (int64_t span = 1; span < p; span *= 2) {
    PairAddArgs a;
    std::memset(&a, 0, sizeof(a));
    for (int64_t r = 0; r + span < p; r += 2 * span) {
      const int k = a.njobs++;
      a.a[k] = B[r]; a.b[k] = B[r + span]; a.d1[k] = B[r]; a.lo[k] = 0; a.hi[k] = n;
    }
    a.divide = (2 * span >= p); a.divisor = divisor;
    DDP_CUDA(launch_pair_add(a, s), "tree reduce step launch");
  }
  for (int64_t span = 1; span < p; span *= 2) {
    PairCopyArgs a;
    std::memset(&a, 0, sizeof(a));
    for (int64_t v = 0; v < span && v + span < p; ++v) {
      const int k = a.njobs++;
      a.src[k] = reinterpret_cast<const char*>(B[v]);
      a.dst[k] = reinterpret_cast<char*>(B[v + span]);
      a.nbytes[k] = n * 4;
    }
    DDP_CUDA(launch_pair_copy(a, s), "tree broadcast step launch");
  }
  return DDP_OK;
}

ddp_status check_own(int own) {
  DDP_CHECK(own == DDP_OWN_RANK || own == DDP_OWN_RING, DDP_ERR_ARG, "unknown ownership");
  return DDP_OK;
}

#define DDP_TRY(expr)                 \
  do {                                \
    const ddp_status rc_ = (expr);    \
    if (rc_ != DDP_OK) return rc_;    \
  } while (0)

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

ddp_status check_bucket_args(int32_t p, int32_t k, const int64_t* numel, const int64_t* offset, int dtype) {
  DDP_TRY(check_common(p, 0, dtype));
  DDP_CHECK(k >= 0, DDP_ERR_ARG, "k must be >= 0");
  if (k > 0) DDP_CHECK(numel && offset, DDP_ERR_ARG, "numel / offset arrays are null");
  for (int32_t j = 0; j < k; ++j)
    DDP_CHECK(numel[j] >= 0 && offset[j] >= 0, DDP_ERR_ARG, "numel and offset must be >= 0");
  return DDP_OK;
}

ddp_status check_bucket_layout(int32_t p, int32_t k, const void* const* grads, const int64_t* numel,
                               const int64_t* offset, const void* const* bucket, int es) {
  DDP_TRY(check_ptrs(bucket, p, "bucket"));
  DDP_CHECK(grads != nullptr || k == 0, DDP_ERR_ARG, "grads array is null");
  int64_t extent = 0;
  std::vector<std::pair<uintptr_t, uintptr_t>> slots, ranges;
  for (int32_t j = 0; j < k; ++j) {
    extent = std::max(extent, offset[j] + numel[j]);
    slots.push_back({static_cast<uintptr_t>(offset[j]), static_cast<uintptr_t>(offset[j] + numel[j])});
  }
  DDP_CHECK(disjoint(slots), DDP_ERR_ARG, "bucket slots of different tensors overlap");
  for (int32_t r = 0; r < p; ++r) {
    ranges.push_back(range_of(bucket[r], extent * es));
    for (int32_t j = 0; j < k; ++j) {
      if (numel[j] == 0) continue;
      const void* g = grads[static_cast<int64_t>(r) * k + j];
      DDP_CHECK(g != nullptr, DDP_ERR_ARG, "grads[" + std::to_string(r * k + j) + "] is null");
      ranges.push_back(range_of(g, numel[j] * es));
    }
  }
  DDP_CHECK(disjoint(ranges), DDP_ERR_ARG, "gradient tensors and buckets must not overlap");
  return DDP_OK;
}


// Pieces of one bucket for the in-place kernel: every tensor cut at chunk
// boundaries, so each piece has one summation origin. Launches hold at most
// kBucketPieces pieces and kBucketPtrs replica pointers; a longer bucket goes
// out in several launches (pieces are independent).
ddp_status plan_bucket_launches(int32_t p, int32_t k, const void* const* grads, const int64_t* numel,
                                const int64_t* offset, ddp_dtype dt, float divisor,
                                std::vector<BucketArgs>& out) {
  out.clear();
  int64_t n = 0;
  for (int32_t j = 0; j < k; ++j) n = std::max(n, offset[j] + numel[j]);
  if (n == 0) return DDP_OK;
  const int64_t cs = chunk_size(n, p);
  const int64_t tile = bucket_tile_elems(esize(dt));
  const int slots_per_launch = kBucketPtrs / p;
  DDP_CHECK(slots_per_launch >= 1, DDP_ERR_ARG, "too many replicas for the in-place bucket kernel");
  BucketArgs a;
  std::memset(&a, 0, sizeof(a));
  a.p = p;
  a.divisor = divisor;
  int nslots = 0;
  auto flush = [&]() {
    if (a.npieces > 0) out.push_back(a);
    std::memset(&a, 0, sizeof(a));
    a.p = p;
    a.divisor = divisor;
    nslots = 0;
  };
  for (int32_t j = 0; j < k; ++j) {
    if (numel[j] == 0) continue;
    const int64_t lo = offset[j], hi = offset[j] + numel[j];
    const int64_t c0 = lo / cs, c1 = (hi - 1) / cs;
    if (nslots == slots_per_launch || a.npieces + (c1 - c0 + 1) > kBucketPieces) flush();
    DDP_CHECK(c1 - c0 + 1 <= kBucketPieces, DDP_ERR_ARG, "a tensor spans too many chunks");
    const int slot = nslots++;
    for (int r = 0; r < p; ++r) a.ptr[slot * p + r] = const_cast<void*>(grads[static_cast<int64_t>(r) * k + j]);
    for (int64_t c = c0; c <= c1; ++c) {
      const int64_t plo = std::max(lo, c * cs), phi = std::min(hi, (c + 1) * cs);
      const int i = a.npieces++;
      a.start[i] = plo - lo;
      a.len[i] = phi - plo;
      a.slot[i] = slot;
      a.origin[i] = static_cast<int32_t>(c);
      const int64_t tiles = (phi - plo + tile - 1) / tile;
      DDP_CHECK(static_cast<int64_t>(a.tile0[i]) + tiles <= 0x7FFFFFFF, DDP_ERR_ARG, "bucket too large");
      a.tile0[i + 1] = a.tile0[i] + static_cast<int32_t>(tiles);
    }
  }
  flush();
  return DDP_OK;
}

ddp_status run_bucket_launches(std::vector<BucketArgs>& launches, ddp_dtype dt, float divisor, cudaStream_t s) {
  for (BucketArgs& a : launches) {
    a.divisor = divisor;
    DDP_CUDA(launch_bucket_allreduce(a, dt, s), "bucket all-reduce launch");
  }
  return DDP_OK;
}

// Write a bucket list (tensor indices per bucket, walk order) in the
// ddp_bucket_assign output format.
void write_assignment(const std::vector<std::vector<int32_t>>& buckets, const int64_t* numel, int32_t* n_buckets,
                      int32_t* bucket_of, int64_t* offset, int32_t* bucket_ptr, int32_t* bucket_tensors,
                      int64_t* bucket_numel) {
  int32_t pos = 0;
  bucket_ptr[0] = 0;
  for (size_t b = 0; b < buckets.size(); ++b) {
    int64_t off = 0;
    for (int32_t t : buckets[b]) {
      bucket_of[t] = static_cast<int32_t>(b);
      offset[t] = off;
      off += numel[t];
      bucket_tensors[pos++] = t;
    }
    bucket_numel[b] = off;
    bucket_ptr[b + 1] = pos;
  }
  *n_buckets = static_cast<int32_t>(buckets.size());
}

// Walk `walk` (tensor indices), closing a bucket once its bytes reach its cap.
std::vector<std::vector<int32_t>> walk_buckets(const std::vector<int32_t>& walk, const int64_t* numel,
                                               int32_t elem_size, int64_t first_cap, int64_t cap) {
  std::vector<std::vector<int32_t>> buckets;
  std::vector<int32_t> open;
  int64_t bytes = 0;
  for (int32_t t : walk) {
    open.push_back(t);
    bytes += numel[t] * elem_size;
    if (bytes >= (buckets.empty() ? first_cap : cap)) {
      buckets.push_back(open);
      open.clear();
      bytes = 0;
    }
  }
  if (!open.empty()) buckets.push_back(open);
  return buckets;
}

}  // namespace

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

static ddp_status impl_allreduce_ex(void* const* bufs, int32_t p, int64_t n, ddp_dtype dtype, float divisor,
                                    ddp_algo algo, uint32_t flags, cudaStream_t stream);

static ddp_status impl_allreduce(void* const* bufs, int32_t p, int64_t n, ddp_dtype dtype, float divisor,
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
    const cudaError_t ea = cudaMallocAsync(&wsv, slot * p, stream);
    if (ea != cudaSuccess) {
      (void)cudaGetLastError();  // an allocation failure is not sticky: do not let a later launch report it
      return fail(DDP_ERR_NOMEM, std::string("tree workspace: ") + cudaGetErrorString(ea));
    }
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
  return impl_allreduce_ex(bufs, p, n, dtype, divisor, algo, 0u, stream);
}

static ddp_status impl_allreduce_ex(void* const* bufs, int32_t p, int64_t n, ddp_dtype dtype, float divisor,
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

static ddp_status impl_reduce_scatter(const void* const* in, void* const* out, int32_t p, int64_t n, ddp_dtype dtype,
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

static ddp_status impl_allgather(const void* const* in, void* const* out, int32_t p, int64_t m, ddp_dtype dtype,
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
  DDP_CUDA(launch_fanout(a, stream), "all-gather launch");
  return DDP_OK;
}

static ddp_status impl_broadcast(void* const* bufs, int32_t p, int64_t nbytes, int32_t root, ddp_algo algo,
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
  DDP_CUDA(launch_fanout(a, stream), "broadcast launch");
  return DDP_OK;
}

static ddp_status impl_broadcast_coalesced(int32_t p, int32_t k, void* const* tensors, const int64_t* nbytes,
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
  DDP_CUDA(cudaMallocAsync(&wsv, slot * p, stream), "broadcast workspace allocation");
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


static ddp_status impl_bucket_allreduce(int32_t p, int32_t k, void* const* grads, const int64_t* numel,
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

// ------------------------------------------------------------- reducer
struct ddp_reducer {
  int32_t p = 0, k = 0;
  ddp_dtype dt = DDP_FLOAT32;
  int64_t first_cap = 0, cap = 0;
  std::vector<void*> grads;  // [p * k]
  std::vector<int64_t> numel;
  struct Bucket {
    std::vector<int32_t> members;
    std::vector<int64_t> numel, offset;  // per member
    int64_t n = 0;
    std::vector<void*> flat;             // [p]
    std::vector<const void*> grads;      // [p * members], replica-major
    std::vector<BucketArgs> launches;    // this bucket alone, in place (readiness-driven firing)
  };
  std::vector<Bucket> buckets;
  std::vector<int32_t> bucket_of;  // per tensor
  std::vector<void*> arenas;  // one flat-bucket arena per replica
  float* ws = nullptr;        // fp32 partials for the literal bf16 schedule
  int64_t ws_elems = 0;
  void* table_mem = nullptr;  // the in-place sync's piece table, every bucket, in device memory
  BucketTable table{};
  int32_t table_tiles = 0;
  // readiness ("PyTorch DDP Deep Dive", Part 2: pending counts, next_bucket_)
  std::vector<int32_t> pending;
  std::vector<char> marked;
  std::vector<int32_t> observed;  // ready order seen since the last prepare
  int32_t next_bucket = 0;
};

namespace {

// Free the reducer's device memory; returns the first cudaFree error.
cudaError_t reducer_free_device(ddp_reducer* h) {
  cudaError_t first = cudaSuccess;
  auto release = [&](void* ptr) {
    if (!ptr) return;
    const cudaError_t e = cudaFree(ptr);
    if (first == cudaSuccess) first = e;
  };
  for (void* a : h->arenas) release(a);
  h->arenas.clear();
  release(h->ws);
  h->ws = nullptr;
  release(h->table_mem);
  h->table_mem = nullptr;
  h->table = BucketTable{};
  h->table_tiles = 0;
  return first;
}

// Cut every bucket of the reducer into pieces (tensor x chunk, one summation
// origin each), in bucket order, and upload the table to device memory once.
ddp_status build_reducer_table(ddp_reducer* h) {
  const int p = h->p;
  const int64_t tile = bucket_tile_elems(esize(h->dt));
  std::vector<void*> ptr;
  std::vector<int64_t> start, len;
  std::vector<int32_t> slot, origin, tile0{0};
  int32_t nslots = 0;
  for (const auto& B : h->buckets) {
    if (B.n == 0) continue;
    const int64_t cs = chunk_size(B.n, p);
    const int32_t m = static_cast<int32_t>(B.members.size());
    for (int32_t j = 0; j < m; ++j) {
      if (B.numel[j] == 0) continue;
      const int32_t sl = nslots++;
      for (int r = 0; r < p; ++r) ptr.push_back(const_cast<void*>(B.grads[static_cast<int64_t>(r) * m + j]));
      const int64_t lo = B.offset[j], hi = B.offset[j] + B.numel[j];
      for (int64_t c = lo / cs; c <= (hi - 1) / cs; ++c) {
        const int64_t plo = std::max(lo, c * cs), phi = std::min(hi, (c + 1) * cs);
        start.push_back(plo - lo);
        len.push_back(phi - plo);
        slot.push_back(sl);
        origin.push_back(static_cast<int32_t>(c));
        const int64_t t = static_cast<int64_t>(tile0.back()) + (phi - plo + tile - 1) / tile;
        DDP_CHECK(t <= 0x7FFFFFFF, DDP_ERR_ARG, "gradient set too large for one in-place launch");
        tile0.push_back(static_cast<int32_t>(t));
      }
    }
  }
  const size_t np = start.size();
  if (np == 0) return DDP_OK;
  auto up16 = [](size_t x) { return (x + 15) / 16 * 16; };
  const size_t o_ptr = 0, o_start = up16(o_ptr + ptr.size() * sizeof(void*)), o_len = up16(o_start + np * 8),
               o_slot = up16(o_len + np * 8), o_origin = up16(o_slot + np * 4), o_tile0 = up16(o_origin + np * 4),
               total = up16(o_tile0 + (np + 1) * 4);
  std::vector<unsigned char> host(total, 0);
  std::memcpy(host.data() + o_ptr, ptr.data(), ptr.size() * sizeof(void*));
  std::memcpy(host.data() + o_start, start.data(), np * 8);
  std::memcpy(host.data() + o_len, len.data(), np * 8);
  std::memcpy(host.data() + o_slot, slot.data(), np * 4);
  std::memcpy(host.data() + o_origin, origin.data(), np * 4);
  std::memcpy(host.data() + o_tile0, tile0.data(), (np + 1) * 4);
  void* mem = nullptr;
  cudaError_t e = cudaMalloc(&mem, total);
  if (e != cudaSuccess) return fail(DDP_ERR_NOMEM, std::string("reducer piece table: ") + cudaGetErrorString(e));
  h->table_mem = mem;
  DDP_CUDA(cudaMemcpy(mem, host.data(), total, cudaMemcpyHostToDevice), "reducer piece table upload");
  unsigned char* d = static_cast<unsigned char*>(mem);
  h->table.ptr = reinterpret_cast<void* const*>(d + o_ptr);
  h->table.start = reinterpret_cast<const int64_t*>(d + o_start);
  h->table.len = reinterpret_cast<const int64_t*>(d + o_len);
  h->table.slot = reinterpret_cast<const int32_t*>(d + o_slot);
  h->table.origin = reinterpret_cast<const int32_t*>(d + o_origin);
  h->table.tile0 = reinterpret_cast<const int32_t*>(d + o_tile0);
  h->table.npieces = static_cast<int>(np);
  h->table.p = p;
  h->table_tiles = tile0.back();
  return DDP_OK;
}

// (Re)build buckets from a walk order over the tensors: the flat-bucket
// arenas, the bf16 workspace, each bucket's own in-place launches and the
// whole-set piece table. Frees whatever device memory a previous build held.
ddp_status reducer_build(ddp_reducer* h, const std::vector<int32_t>& walk, bool reverse_list) {
  const int p = h->p, k = h->k, es = esize(h->dt);
  auto lists = walk_buckets(walk, h->numel.data(), es, h->first_cap, h->cap);
  if (reverse_list) std::reverse(lists.begin(), lists.end());
  DDP_CUDA(reducer_free_device(h), "reducer rebuild: release");
  h->buckets.clear();
  h->bucket_of.assign(k, -1);
  h->ws_elems = 0;
  int64_t arena = 0;
  std::vector<int64_t> base;
  for (const auto& members : lists) {
    int64_t n = 0;
    for (int32_t t : members) n += h->numel[t];
    base.push_back(arena);
    arena += (n * es + 255) / 256 * 256;
    h->ws_elems = std::max(h->ws_elems, 2 * static_cast<int64_t>(p) * chunk_size(n, p));
  }
  for (int32_t r = 0; r < p; ++r) {
    void* a = nullptr;
    const cudaError_t e = cudaMalloc(&a, std::max<int64_t>(arena, 256));
    if (e != cudaSuccess) return fail(DDP_ERR_NOMEM, std::string("reducer buckets: ") + cudaGetErrorString(e));
    h->arenas.push_back(a);
  }
  if (h->dt == DDP_BFLOAT16 && p > 1 && h->ws_elems > 0) {
    void* w = nullptr;
    const cudaError_t e = cudaMalloc(&w, h->ws_elems * sizeof(float));
    if (e != cudaSuccess) return fail(DDP_ERR_NOMEM, std::string("reducer workspace: ") + cudaGetErrorString(e));
    h->ws = static_cast<float*>(w);
  }
  for (size_t b = 0; b < lists.size(); ++b) {
    ddp_reducer::Bucket B;
    int64_t off = 0;
    for (int32_t t : lists[b]) {
      B.members.push_back(t);
      B.numel.push_back(h->numel[t]);
      B.offset.push_back(off);
      off += h->numel[t];
      h->bucket_of[t] = static_cast<int32_t>(b);
    }
    B.n = off;
    const int32_t m = static_cast<int32_t>(B.members.size());
    for (int32_t r = 0; r < p; ++r) {
      B.flat.push_back(static_cast<char*>(h->arenas[r]) + base[b]);
      for (int32_t t : B.members) B.grads.push_back(h->grads[static_cast<int64_t>(r) * k + t]);
    }
    DDP_TRY(plan_bucket_launches(p, m, B.grads.data(), B.numel.data(), B.offset.data(), h->dt, 1.0f, B.launches));
    h->buckets.push_back(std::move(B));
  }
  DDP_TRY(build_reducer_table(h));
  h->pending.assign(h->buckets.size(), 0);
  for (size_t b = 0; b < h->buckets.size(); ++b) h->pending[b] = static_cast<int32_t>(h->buckets[b].members.size());
  h->marked.assign(k, 0);
  h->observed.clear();
  h->next_bucket = 0;
  return DDP_OK;
}

}  // namespace

ddp_status ddp_reducer_create(ddp_reducer** handle, int32_t p, int32_t k, void* const* grads,
                              const int64_t* numel, ddp_dtype dtype, int64_t first_bucket_cap_bytes,
                              int64_t bucket_cap_bytes, ddp_border order) {
  DDP_CHECK(handle != nullptr, DDP_ERR_ARG, "handle pointer is null");
  *handle = nullptr;
  DDP_TRY(check_common(p, 0, dtype));
  DDP_CHECK(k >= 1 && numel && grads, DDP_ERR_ARG, "need k >= 1 tensors, numel and grads");
  DDP_CHECK(first_bucket_cap_bytes >= 0 && bucket_cap_bytes >= 0, DDP_ERR_ARG, "caps must be >= 0");
  DDP_CHECK(order == DDP_ORDER_REVERSED || order == DDP_ORDER_REGISTRATION, DDP_ERR_ARG, "unknown order");
  const int es = esize(dtype);
  {
    std::vector<std::pair<uintptr_t, uintptr_t>> ranges;
    for (int32_t t = 0; t < k; ++t) DDP_CHECK(numel[t] >= 0, DDP_ERR_ARG, "numel must be >= 0");
    for (int32_t r = 0; r < p; ++r)
      for (int32_t t = 0; t < k; ++t) {
        if (numel[t] == 0) continue;
        const void* g = grads[static_cast<int64_t>(r) * k + t];
        DDP_CHECK(g != nullptr, DDP_ERR_ARG, "grads[" + std::to_string(r * k + t) + "] is null");
        ranges.push_back(range_of(g, numel[t] * es));
      }
    DDP_CHECK(disjoint(ranges), DDP_ERR_ARG, "gradient tensors overlap");
  }
  ddp_reducer* h = new ddp_reducer();
  h->p = p; h->k = k; h->dt = dtype;
  h->first_cap = first_bucket_cap_bytes;
  h->cap = bucket_cap_bytes;
  h->grads.assign(grads, grads + static_cast<int64_t>(p) * k);
  h->numel.assign(numel, numel + k);
  std::vector<int32_t> walk(k);
  for (int32_t w = 0; w < k; ++w) walk[w] = (order == DDP_ORDER_REVERSED) ? k - 1 - w : w;
  const ddp_status st = reducer_build(h, walk, order == DDP_ORDER_REGISTRATION);
  if (st != DDP_OK) {
    reducer_free_device(h);
    delete h;
    return st;
  }
  *handle = h;
  return DDP_OK;
}

int32_t ddp_reducer_num_buckets(const ddp_reducer* h) { return h ? static_cast<int32_t>(h->buckets.size()) : -1; }

ddp_status ddp_reducer_bucket(const ddp_reducer* h, int32_t b, int64_t* numel, void** flat) {
  DDP_CHECK(h && numel, DDP_ERR_ARG, "null argument");
  DDP_CHECK(b >= 0 && b < static_cast<int32_t>(h->buckets.size()), DDP_ERR_ARG, "bucket index out of range");
  *numel = h->buckets[b].n;
  if (flat)
    for (int32_t r = 0; r < h->p; ++r) flat[r] = h->buckets[b].flat[r];
  return DDP_OK;
}

static ddp_status impl_reducer_sync(ddp_reducer* h, float divisor, float predivide, ddp_algo algo, ddp_sync_mode mode,
                                    cudaStream_t stream) {
  DDP_NVTX("ddp_reducer_sync");
  DDP_CHECK(h != nullptr, DDP_ERR_ARG, "handle is null");
  DDP_TRY(check_divisor(divisor));
  DDP_TRY(check_divisor(predivide));
  DDP_TRY(check_algo(algo));
  DDP_CHECK(mode == DDP_SYNC_FLATTEN || mode == DDP_SYNC_IN_PLACE, DDP_ERR_ARG, "unknown sync mode");
  const int p = h->p;
  if (mode == DDP_SYNC_IN_PLACE) {
    DDP_CHECK(algo != DDP_ALGO_RING_STEPS, DDP_ERR_ARG, "the in-place sync is the fused form only");
    DDP_CHECK(predivide == 1.0f, DDP_ERR_ARG, "the in-place sync has no pre-divide");
    DDP_CUDA(launch_bucket_table(h->table, h->table_tiles, divisor, h->dt, stream), "in-place sync launch");
    return DDP_OK;
  }
  const int es = esize(h->dt);
  for (auto& B : h->buckets) {
    const int32_t m = static_cast<int32_t>(B.members.size());
    SegBatcher sb(h->dt, predivide, stream);
    for (int32_t r = 0; r < p; ++r)
      for (int32_t j = 0; j < m; ++j)
        DDP_TRY(sb.add(B.grads[static_cast<int64_t>(r) * m + j], static_cast<char*>(B.flat[r]) + B.offset[j] * es,
                       B.numel[j] * es));
    DDP_TRY(sb.flush());
    if (B.n == 0) continue;
    if (algo == DDP_ALGO_RING_STEPS) {
      Plan pl;
      pl.op = DDP_OP_ALLREDUCE; pl.p = p; pl.n = B.n; pl.dt = h->dt; pl.divisor = divisor;
      pl.in.assign(B.flat.begin(), B.flat.end());
      pl.init();
      pl.ws = h->ws;
      DDP_TRY(pl.run_all(stream));
    } else {
      DDP_TRY(run_fused(const_cast<const void* const*>(B.flat.data()), B.flat.data(), p, B.n, h->dt, divisor, false,
                        0, algo == DDP_ALGO_FUSED_TMA, stream));
    }
  }
  for (auto& B : h->buckets) {
    const int32_t m = static_cast<int32_t>(B.members.size());
    SegBatcher sb(h->dt, 1.0f, stream);
    for (int32_t r = 0; r < p; ++r)
      for (int32_t j = 0; j < m; ++j)
        DDP_TRY(sb.add(static_cast<const char*>(B.flat[r]) + B.offset[j] * es,
                       const_cast<void*>(B.grads[static_cast<int64_t>(r) * m + j]), B.numel[j] * es));
    DDP_TRY(sb.flush());
  }
  return DDP_OK;
}

ddp_status ddp_reducer_destroy(ddp_reducer* h) {
  if (!h) return DDP_OK;
  const cudaError_t e = reducer_free_device(h);
  delete h;
  if (e != cudaSuccess) return cuda_fail(e, "reducer release");
  return DDP_OK;
}

ddp_status ddp_reducer_prepare(ddp_reducer* h) {
  DDP_CHECK(h != nullptr, DDP_ERR_ARG, "handle is null");
  for (size_t b = 0; b < h->buckets.size(); ++b) h->pending[b] = static_cast<int32_t>(h->buckets[b].members.size());
  std::fill(h->marked.begin(), h->marked.end(), 0);
  h->observed.clear();
  h->next_bucket = 0;
  return DDP_OK;
}

ddp_status ddp_reducer_mark_ready(ddp_reducer* h, int32_t tensor, float divisor, cudaEvent_t ready,
                                  cudaStream_t comm_stream, int32_t* fired) {
  DDP_NVTX("ddp_reducer_mark_ready");
  DDP_CHECK(h != nullptr, DDP_ERR_ARG, "handle is null");
  DDP_CHECK(tensor >= 0 && tensor < h->k, DDP_ERR_ARG, "tensor index out of range");
  DDP_TRY(check_divisor(divisor));
  DDP_CHECK(!h->marked[tensor], DDP_ERR_STATE,
            "tensor " + std::to_string(tensor) + " was already marked ready since the last ddp_reducer_prepare");
  h->marked[tensor] = 1;
  h->observed.push_back(tensor);
  h->pending[h->bucket_of[tensor]] -= 1;
  int32_t n = 0;
  bool waited = false;
  const int32_t nb = static_cast<int32_t>(h->buckets.size());
  while (h->next_bucket < nb && h->pending[h->next_bucket] == 0) {  // mark_bucket_ready: strictly in order
    if (ready && !waited) {
      DDP_CUDA(cudaStreamWaitEvent(comm_stream, ready, 0), "wait on the gradient's ready event");
      waited = true;
    }
    DDP_TRY(run_bucket_launches(h->buckets[h->next_bucket].launches, h->dt, divisor, comm_stream));
    ++h->next_bucket;
    ++n;
  }
  if (fired) *fired = n;
  return DDP_OK;
}

int32_t ddp_reducer_observed(const ddp_reducer* h, int32_t* order) {
  if (!h) return -1;
  if (order)
    for (size_t i = 0; i < h->observed.size(); ++i) order[i] = h->observed[i];
  return static_cast<int32_t>(h->observed.size());
}

ddp_status ddp_reducer_rebuild(ddp_reducer* h, const int32_t* order) {
  DDP_CHECK(h != nullptr, DDP_ERR_ARG, "handle is null");
  std::vector<int32_t> walk;
  if (order) {
    walk.assign(order, order + h->k);
  } else {
    DDP_CHECK(static_cast<int32_t>(h->observed.size()) == h->k, DDP_ERR_STATE,
              "rebuild from the observed order needs every tensor marked ready since the last prepare");
    walk = h->observed;
  }
  std::vector<char> seen(h->k, 0);
  for (int32_t t : walk) {
    DDP_CHECK(t >= 0 && t < h->k && !seen[t], DDP_ERR_ARG, "order must be a permutation of 0..k-1");
    seen[t] = 1;
  }
  DDP_CUDA(cudaDeviceSynchronize(), "synchronize before rebuilding buckets");
  return reducer_build(h, walk, false);
}

static ddp_status impl_allreduce_persistent(void* const* bufs, int32_t p, int64_t n, ddp_dtype dtype, float divisor,
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
    const cudaError_t ea = cudaMallocAsync(&wsv, slot * p, stream);
    if (ea != cudaSuccess) {
      (void)cudaGetLastError();  // an allocation failure is not sticky: do not let a later launch report it
      return fail(DDP_ERR_NOMEM, std::string("persistent ring workspace: ") + cudaGetErrorString(ea));
    }
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
                        ? impl_allreduce_persistent(W.data(), p, n, DDP_FLOAT32, divisor, timeout_ns, fault_rank,
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
  DDP_CUDA(cudaMallocAsync(&flags, static_cast<size_t>(p) * B * kFlagStride * sizeof(int), stream), "step flags allocation");
  a.flags = static_cast<int*>(flags);
  cudaError_t e = cudaMemsetAsync(flags, 0, static_cast<size_t>(p) * B * kFlagStride * sizeof(int), stream);
  if (e == cudaSuccess) e = launch_ring_persistent(a, stream);
  const cudaError_t e2 = cudaFreeAsync(flags, stream);
  if (e != cudaSuccess) return cuda_fail(e, "persistent ring launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "step flags release");
  return DDP_OK;
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
    const cudaError_t e = cudaMalloc(&w, pl.ws_elems() * sizeof(float));
    if (e != cudaSuccess) {
      delete h;
      t_error = std::string("handle workspace allocation: ") + cudaGetErrorString(e);
      return DDP_ERR_NOMEM;
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

// ======================================= reduce-scatter that allocates nothing
// For callers that cannot allocate device memory: a framework whose caching
// allocator owns the whole device, or code that must not risk an allocation's
// failure or its implicit synchronisation in the middle of a step. The literal
// ring reduce-scatter keeps its fp32 partials in the fixed array below instead
// of a stream-ordered temporary. Every GPU that loads this library holds the
// array until the process exits.
namespace {

constexpr int64_t kNoAllocScratchBytes = int64_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[64] = {nullptr};

// The array's device address on the current device, looked up once per device.
// In host code the array's name is only a stand-in: the address a kernel may
// use is the one cudaGetSymbolAddress returns with that device current.
ddp_status noalloc_scratch(float** out) {
  int dev = 0;
  DDP_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  DDP_CHECK(dev >= 0 && dev < 64, DDP_ERR_ARG, "device index out of range");
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    DDP_CUDA(cudaGetSymbolAddress(&ptr, g_noalloc_scratch), "cudaGetSymbolAddress of the scratch array");
    g_noalloc_ptr[dev] = ptr;
  }
  *out = static_cast<float*>(g_noalloc_ptr[dev]);
  return DDP_OK;
}

// Pairwise-disjoint byte ranges, sorted in place (no allocation).
bool disjoint_inplace(std::pair<uintptr_t, uintptr_t>* r, int count) {
  int m = 0;
  for (int i = 0; i < count; ++i)
    if (r[i].second > r[i].first) r[m++] = r[i];
  std::sort(r, r + m);
  for (int i = 1; i < m; ++i)
    if (r[i].first < r[i - 1].second) return false;
  return true;
}

}  // namespace

extern "C" ddp_status ddp_reduce_scatter_noalloc(const void* const* in, void* const* out, int32_t p, int64_t n,
                                                 ddp_dtype dtype, float divisor, ddp_own own,
                                                 cudaStream_t stream) {
  DDP_TRY(check_common(p, n, dtype));
  DDP_TRY(check_divisor(divisor));
  DDP_TRY(check_own(own));
  DDP_TRY(check_ptrs(in, p, "in"));
  DDP_TRY(check_ptrs(const_cast<const void* const*>(out), p, "out"));
  if (own == DDP_OWN_RANK)
    DDP_CHECK(n % p == 0, DDP_ERR_NOT_DIVISIBLE,
              "reduce_scatter: " + std::to_string(n) + " elements are not divisible by " + std::to_string(p) + " ranks");
  const int es = esize(dtype);
  const int64_t cs = chunk_size(n, p);
  const int64_t need = 2 * static_cast<int64_t>(p) * cs * static_cast<int64_t>(sizeof(float));
  DDP_CHECK(p == 1 || need <= kNoAllocScratchBytes, DDP_ERR_ARG,
            "ddp_reduce_scatter_noalloc: needs " + std::to_string(need) +
                " bytes of scratch (2 * p * ceil(n/p) fp32 partials), more than its fixed " +
                std::to_string(kNoAllocScratchBytes) + "-byte array; call ddp_reduce_scatter instead");
  std::pair<uintptr_t, uintptr_t> outs[DDP_MAX_P], all[DDP_MAX_P + 1];
  for (int r = 0; r < p; ++r) outs[r] = range_of(out[r], cs * es);
  for (int r = 0; r < p; ++r) all[r] = outs[r];
  DDP_CHECK(disjoint_inplace(all, p), DDP_ERR_ARG, "output buffers overlap");
  for (int r = 0; r < p; ++r) {
    for (int q = 0; q < p; ++q) all[q] = outs[q];
    all[p] = range_of(in[r], n * es);
    DDP_CHECK(disjoint_inplace(all, p + 1), DDP_ERR_ARG, "an output buffer overlaps an input");
  }
  if (n == 0) return DDP_OK;
  if (p == 1)  // one scale step, no partials
    return run_fused(in, out, 1, n, dtype, divisor, true, 0, false, stream);
  float* scratch = nullptr;
  DDP_TRY(noalloc_scratch(&scratch));
  // Nothing in the array needs to start at zero: every slot a step reads was
  // written by the step before it in this same call.
  RingStepArgs a;
  for (int s = 0; s < p - 1; ++s) {
    std::memset(&a, 0, sizeof(a));
    for (int r = 0; r < p; ++r) {
      a.x[r] = const_cast<void*>(in[r]);
      a.out[r] = out[r];
    }
    a.w = scratch; a.n = n; a.cs = cs; a.divisor = divisor; a.p = p; a.step = s;
    a.shift = (own == DDP_OWN_RANK) ? 1 : 0; a.last = (s == p - 2); a.out_rel = 1;
    DDP_CUDA(launch_rs_step_ws(a, dtype, stream), "reduce-scatter step launch");
  }
  return DDP_OK;
}

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
  const ddp_status st = impl_allreduce(bufs, p, n, dtype, divisor, algo, stream);
  const int es = esize(dtype);
  log_call(t, "ddp_allreduce", algo, p, n, dtype, 2 * static_cast<int64_t>(p) * n * es,
           allreduce_rank_bytes(algo, p, n, es), st);
  return st;
}

ddp_status ddp_allreduce_ex(void* const* bufs, int32_t p, int64_t n, ddp_dtype dtype, float divisor,
                            ddp_algo algo, uint32_t flags, cudaStream_t stream) {
  CallTimer t(stream);
  const ddp_status st = impl_allreduce_ex(bufs, p, n, dtype, divisor, algo, flags, stream);
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
      impl_allreduce_persistent(bufs, p, n, dtype, divisor, timeout_ns, fault_rank, fault_step, status, stream);
  const int es = esize(dtype);
  log_call(t, "ddp_allreduce_persistent", DDP_ALGO_RING_STEPS, p, n, dtype, 2 * static_cast<int64_t>(p) * n * es,
           allreduce_rank_bytes(DDP_ALGO_RING_STEPS, p, n, es), st);
  return st;
}

ddp_status ddp_reduce_scatter(const void* const* in, void* const* out, int32_t p, int64_t n, ddp_dtype dtype,
                              float divisor, ddp_own own, ddp_algo algo, cudaStream_t stream) {
  CallTimer t(stream);
  const ddp_status st = impl_reduce_scatter(in, out, p, n, dtype, divisor, own, algo, stream);
  const int es = esize(dtype);
  const int64_t cs = (p > 0 && n > 0) ? chunk_size(n, p) : 0;
  log_call(t, "ddp_reduce_scatter", algo, p, n, dtype, (static_cast<int64_t>(p) + 1) * n * es,
           p > 1 ? static_cast<int64_t>(p - 1) * cs * es : 0, st);
  return st;
}

ddp_status ddp_allgather(const void* const* in, void* const* out, int32_t p, int64_t m, ddp_dtype dtype,
                         ddp_own own, ddp_algo algo, cudaStream_t stream) {
  CallTimer t(stream);
  const ddp_status st = impl_allgather(in, out, p, m, dtype, own, algo, stream);
  const int es = esize(dtype);
  const int64_t whole = static_cast<int64_t>(p) * m;  // elements of the gathered buffer
  log_call(t, "ddp_allgather", algo, p, whole, dtype, (static_cast<int64_t>(p) + 1) * whole * es,
           p > 1 ? static_cast<int64_t>(p - 1) * m * es : 0, st);
  return st;
}

ddp_status ddp_broadcast(void* const* bufs, int32_t p, int64_t nbytes, int32_t root, ddp_algo algo,
                         cudaStream_t stream) {
  CallTimer t(stream);
  const ddp_status st = impl_broadcast(bufs, p, nbytes, root, algo, stream);
  log_call(t, "ddp_broadcast", algo, p, nbytes, DDP_FLOAT32, static_cast<int64_t>(p) * nbytes,
           static_cast<int64_t>(ceil_log2(p)) * nbytes, st);
  return st;
}

ddp_status ddp_broadcast_coalesced(int32_t p, int32_t k, void* const* tensors, const int64_t* nbytes, int32_t root,
                                   int64_t bucket_cap_bytes, ddp_algo algo, cudaStream_t stream) {
  CallTimer t(stream);
  const ddp_status st = impl_broadcast_coalesced(p, k, tensors, nbytes, root, bucket_cap_bytes, algo, stream);
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
  const ddp_status st = impl_bucket_allreduce(p, k, grads, numel, offset, dtype, divisor, stream);
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
  const ddp_status st = impl_reducer_sync(h, divisor, predivide, algo, mode, stream);
  int64_t n = 0, rank_bytes = 0;
  int32_t p = 0;
  ddp_dtype dt = DDP_FLOAT32;
  if (h) {
    p = h->p;
    dt = h->dt;
    for (const auto& b : h->buckets) {
      n += b.n;
      rank_bytes += allreduce_rank_bytes(algo, p, b.n, esize(dt));
    }
  }
  const int64_t ar = 2 * static_cast<int64_t>(p) * n * esize(dt);
  // the flatten form also copies every gradient into its bucket and back: 4pM more
  log_call(t, "ddp_reducer_sync", algo, p, n, dt, mode == DDP_SYNC_FLATTEN ? 3 * ar : ar, rank_bytes, st);
  return st;
}

}  // extern "C"
