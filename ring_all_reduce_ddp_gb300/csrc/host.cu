// Host-side internals of the C ABI (declared in host.h): error text, argument
// checks, the fused and tree-shaped launches, and the bucket planner.
#include <algorithm>
#include <cmath>

#include "host.h"

namespace ddp {
namespace host {

thread_local std::string t_error;

ddp_status fail(ddp_status s, const std::string& msg) {
  t_error = msg;
  return s;
}

ddp_status alloc_async(void** ptr, size_t bytes, cudaStream_t s, const char* what) {
  *ptr = nullptr;
  const cudaError_t e = cudaMallocAsync(ptr, bytes, s);
  if (e == cudaSuccess) return DDP_OK;
  (void)cudaGetLastError();
  *ptr = nullptr;
  return fail(DDP_ERR_NOMEM, std::string(what) + ": " + cudaGetErrorString(e));
}

ddp_status alloc_device(void** ptr, size_t bytes, const char* what) {
  *ptr = nullptr;
  const cudaError_t e = cudaMalloc(ptr, bytes);
  if (e == cudaSuccess) return DDP_OK;
  (void)cudaGetLastError();
  *ptr = nullptr;
  return fail(DDP_ERR_NOMEM, std::string(what) + ": " + cudaGetErrorString(e));
}

ddp_status cuda_fail(cudaError_t e, const char* where) {
  t_error = std::string(where) + ": " + cudaGetErrorString(e);
  return DDP_ERR_CUDA;
}



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
                     bool hop_round) {
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


// One-shot literal schedule with a stream-ordered temporary workspace.
ddp_status run_plan_once(Plan& pl, cudaStream_t s) {
  pl.init();
  if (pl.needs_ws()) {
    void* w = nullptr;
    DDP_TRY(alloc_async(&w, pl.ws_elems() * sizeof(float), s, "workspace allocation"));
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

ddp_status run_bucket_launches(std::vector<BucketArgs>& launches, ddp_dtype dt, float divisor, cudaStream_t s,
                                int32_t max_blocks) {
  for (BucketArgs& a : launches) {
    a.divisor = divisor;
    DDP_CUDA(launch_bucket_allreduce(a, dt, s, max_blocks), "bucket all-reduce launch");
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

}  // namespace host
}  // namespace ddp
