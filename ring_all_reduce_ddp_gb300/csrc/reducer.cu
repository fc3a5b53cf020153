// The C ABI (include/ddp_ring.h), Reducer part: a gradient set's bucket plan
// ("PyTorch DDP Deep Dive", Part 1, _ddp_init_helper), its flat buckets and
// launch tables built once, the whole-set sync, and readiness-driven firing
// (Part 2, mark_variable_ready / mark_bucket_ready, _rebuild_buckets).
#include <algorithm>
#include <cstring>
#include <string>
#include <utility>
#include <vector>

#include "host.h"

using namespace ddp;
using namespace ddp::host;

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
  // A rebuild that failed part way leaves no buckets; until a later rebuild
  // succeeds, sync and readiness calls refuse to run rather than do nothing.
  bool unbuilt = false;
  // Per-forward buffers that ddp_reducer_step broadcasts (kept across
  // rebuilds). They sit at the end of the piece table as copy pieces; the
  // in-place sync launches only the first sync_pieces pieces (sync_tiles).
  std::vector<void*> buf_ptrs;  // [p * kb], replica-major
  std::vector<int64_t> buf_bytes;
  int32_t buf_root = 0;
  int64_t bc_bytes = 0;  // bytes of one replica's buffers
  int32_t sync_pieces = 0, sync_tiles = 0;
  // grid cap of the bucket launches mark_ready fires (0: one block per tile)
  int32_t comm_blocks = 0;
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
  h->sync_pieces = 0;
  h->sync_tiles = 0;
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
  const int32_t sync_pieces = static_cast<int32_t>(start.size());
  const int32_t sync_tiles = tile0.back();
  // the attached buffers: one copy piece each, root replica = origin - p
  const int es = esize(h->dt);
  const int32_t kb = static_cast<int32_t>(h->buf_bytes.size());
  for (int32_t j = 0; j < kb && p > 1; ++j) {
    if (h->buf_bytes[j] == 0) continue;
    const int32_t sl = nslots++;
    for (int r = 0; r < p; ++r) ptr.push_back(h->buf_ptrs[static_cast<int64_t>(r) * kb + j]);
    const int64_t n = h->buf_bytes[j] / es;
    start.push_back(0);
    len.push_back(n);
    slot.push_back(sl);
    origin.push_back(p + h->buf_root);
    const int64_t t = static_cast<int64_t>(tile0.back()) + (n + tile - 1) / tile;
    DDP_CHECK(t <= 0x7FFFFFFF, DDP_ERR_ARG, "gradients and buffers too large for one launch");
    tile0.push_back(static_cast<int32_t>(t));
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
  DDP_TRY(alloc_device(&mem, total, "reducer piece table"));
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
  h->table.err = device_error_word();
  h->table_tiles = tile0.back();
  h->sync_pieces = sync_pieces;
  h->sync_tiles = sync_tiles;
  return DDP_OK;
}

// (Re)build buckets from a walk order over the tensors: the flat-bucket
// arenas, the bf16 workspace, each bucket's own in-place launches and the
// whole-set piece table. Frees whatever device memory an earlier call held.
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
    DDP_TRY(alloc_device(&a, std::max<int64_t>(arena, 256), "reducer buckets"));
    h->arenas.push_back(a);
  }
  if (h->dt == DDP_BFLOAT16 && p > 1 && h->ws_elems > 0) {
    void* w = nullptr;
    DDP_TRY(alloc_device(&w, h->ws_elems * sizeof(float), "reducer workspace"));
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

namespace ddp {
namespace host {

ddp_status reducer_sync_impl(ddp_reducer* h, float divisor, float predivide, ddp_algo algo, ddp_sync_mode mode,
                             cudaStream_t stream) {
  DDP_NVTX("ddp_reducer_sync");
  DDP_CHECK(h != nullptr, DDP_ERR_ARG, "handle is null");
  DDP_TRY(check_divisor(divisor));
  DDP_TRY(check_divisor(predivide));
  DDP_TRY(check_algo(algo));
  DDP_CHECK(mode == DDP_SYNC_FLATTEN || mode == DDP_SYNC_IN_PLACE, DDP_ERR_ARG, "unknown sync mode");
  DDP_CHECK(!h->unbuilt, DDP_ERR_STATE, "the reducer's last rebuild failed; rebuild it again or destroy it");
  const int p = h->p;
  if (mode == DDP_SYNC_IN_PLACE) {
    DDP_CHECK(algo != DDP_ALGO_RING_STEPS, DDP_ERR_ARG, "the in-place sync is the fused form only");
    DDP_CHECK(predivide == 1.0f, DDP_ERR_ARG, "the in-place sync has no pre-divide");
    BucketTable sync = h->table;  // the gradient pieces only: the copy pieces come after them
    sync.npieces = h->sync_pieces;
    DDP_CUDA(launch_bucket_table(sync, h->sync_tiles, divisor, h->dt, stream, algo), "in-place sync launch");
    return DDP_OK;
  }
  const int es = esize(h->dt);
  for (auto& B : h->buckets) {
    DDP_NVTX_I("bucket", static_cast<int>(&B - h->buckets.data()));
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

ddp_status reducer_step_impl(ddp_reducer* h, float divisor, cudaStream_t stream) {
  DDP_NVTX("ddp_reducer_step");
  DDP_CHECK(h != nullptr, DDP_ERR_ARG, "handle is null");
  DDP_TRY(check_divisor(divisor));
  DDP_CHECK(!h->unbuilt, DDP_ERR_STATE, "the reducer's last rebuild failed; rebuild it again or destroy it");
  DDP_CUDA(launch_bucket_table(h->table, h->table_tiles, divisor, h->dt, stream, DDP_ALGO_FUSED),
           "reducer step launch");
  return DDP_OK;
}

int64_t reducer_buffer_bytes(const ddp_reducer* h) { return h ? h->bc_bytes : 0; }

void reducer_shape(const ddp_reducer* h, int32_t* p, ddp_dtype* dt, std::vector<int64_t>* bucket_numel) {
  *p = h ? h->p : 0;
  *dt = h ? h->dt : DDP_FLOAT32;
  bucket_numel->clear();
  if (h)
    for (const auto& b : h->buckets) bucket_numel->push_back(b.n);
}

}  // namespace host
}  // namespace ddp

extern "C" {

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

int32_t ddp_reducer_staged(const ddp_reducer* h) { return h ? (ddp::staged_by_default(h->dt, h->p) ? 1 : 0) : -1; }

ddp_status ddp_reducer_bucket(const ddp_reducer* h, int32_t b, int64_t* numel, void** flat) {
  DDP_CHECK(h && numel, DDP_ERR_ARG, "null argument");
  DDP_CHECK(b >= 0 && b < static_cast<int32_t>(h->buckets.size()), DDP_ERR_ARG, "bucket index out of range");
  *numel = h->buckets[b].n;
  if (flat)
    for (int32_t r = 0; r < h->p; ++r) flat[r] = h->buckets[b].flat[r];
  return DDP_OK;
}


ddp_status ddp_reducer_destroy(ddp_reducer* h) {
  if (!h) return DDP_OK;
  const cudaError_t e = reducer_free_device(h);
  delete h;
  if (e != cudaSuccess) return cuda_fail(e, "reducer release");
  return DDP_OK;
}

ddp_status ddp_reducer_set_buffers(ddp_reducer* h, int32_t k, void* const* tensors, const int64_t* nbytes,
                                   int32_t root) {
  DDP_CHECK(h != nullptr, DDP_ERR_ARG, "handle is null");
  DDP_CHECK(k >= 0, DDP_ERR_ARG, "k must be >= 0");
  DDP_CHECK(root >= 0 && root < h->p, DDP_ERR_ARG, "root out of range");
  DDP_CHECK(k == 0 || (tensors && nbytes), DDP_ERR_ARG, "tensors / nbytes arrays are null");
  DDP_CHECK(!h->unbuilt, DDP_ERR_STATE, "the reducer's last rebuild failed; rebuild it again or destroy it");
  const int p = h->p, es = esize(h->dt);
  std::vector<std::pair<uintptr_t, uintptr_t>> ranges;
  for (int32_t r = 0; r < p; ++r)
    for (int32_t t = 0; t < h->k; ++t)
      if (h->numel[t] > 0) ranges.push_back(range_of(h->grads[static_cast<int64_t>(r) * h->k + t], h->numel[t] * es));
  const size_t ngrad = ranges.size();
  for (int32_t j = 0; j < k; ++j) {
    DDP_CHECK(nbytes[j] >= 0, DDP_ERR_ARG, "nbytes must be >= 0");
    if (nbytes[j] == 0) continue;
    DDP_CHECK(nbytes[j] % es == 0, DDP_ERR_ARG,
              "buffer " + std::to_string(j) + ": its bytes must be a multiple of the gradients' element size");
    for (int32_t r = 0; r < p; ++r) {
      const void* t = tensors[static_cast<int64_t>(r) * k + j];
      DDP_CHECK(t != nullptr, DDP_ERR_ARG, "tensors[" + std::to_string(r * k + j) + "] is null");
      DDP_CHECK(reinterpret_cast<uintptr_t>(t) % es == 0, DDP_ERR_ALIGN,
                "tensors[" + std::to_string(r * k + j) + "] is not aligned to the gradients' element size");
      ranges.push_back(range_of(t, nbytes[j]));
    }
  }
  {
    std::vector<std::pair<uintptr_t, uintptr_t>> bufs(ranges.begin() + ngrad, ranges.end());
    DDP_CHECK(disjoint(bufs), DDP_ERR_ARG, "buffers overlap");
  }
  DDP_CHECK(disjoint(ranges), DDP_ERR_ARG, "a buffer overlaps a gradient of the reducer");
  // the old table may still be read by launches in flight
  DDP_CUDA(cudaDeviceSynchronize(), "synchronize before replacing the piece table");
  h->buf_ptrs.assign(tensors, tensors + static_cast<int64_t>(p) * k);
  h->buf_bytes.assign(nbytes, nbytes + k);
  h->buf_root = root;
  h->bc_bytes = 0;
  for (int32_t j = 0; j < k && p > 1; ++j) h->bc_bytes += nbytes[j];
  if (h->table_mem) {
    DDP_CUDA(cudaFree(h->table_mem), "release of the previous piece table");
    h->table_mem = nullptr;
  }
  h->table = BucketTable{};
  h->table_tiles = h->sync_pieces = h->sync_tiles = 0;
  const ddp_status st = build_reducer_table(h);
  if (st != DDP_OK) {  // keep the handle usable for nothing until a later set or rebuild succeeds
    const std::string msg = t_error;
    if (h->table_mem) cudaFree(h->table_mem);
    h->table_mem = nullptr;
    h->table = BucketTable{};
    h->table_tiles = h->sync_pieces = h->sync_tiles = 0;
    h->buf_ptrs.clear();
    h->buf_bytes.clear();
    h->bc_bytes = 0;
    h->unbuilt = true;
    return fail(st, msg + " (the reducer has no piece table until a rebuild succeeds)");
  }
  return DDP_OK;
}

ddp_status ddp_reducer_set_comm_blocks(ddp_reducer* h, int32_t max_blocks) {
  DDP_CHECK(h != nullptr, DDP_ERR_ARG, "handle is null");
  DDP_CHECK(max_blocks >= 0, DDP_ERR_ARG, "max_blocks must be >= 0");
  h->comm_blocks = max_blocks;
  return DDP_OK;
}

ddp_status ddp_reducer_prepare(ddp_reducer* h) {
  DDP_CHECK(h != nullptr, DDP_ERR_ARG, "handle is null");
  DDP_CHECK(!h->unbuilt, DDP_ERR_STATE, "the reducer's last rebuild failed; rebuild it again or destroy it");
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
  DDP_CHECK(!h->unbuilt, DDP_ERR_STATE, "the reducer's last rebuild failed; rebuild it again or destroy it");
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
    DDP_NVTX_I("bucket", h->next_bucket);
    DDP_TRY(run_bucket_launches(h->buckets[h->next_bucket].launches, h->dt, divisor, comm_stream, h->comm_blocks));
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
  const ddp_status st = reducer_build(h, walk, false);
  if (st != DDP_OK) {  // release what the failed build allocated; keep the handle, bucket-less
    const std::string msg = t_error;
    reducer_free_device(h);
    h->buckets.clear();
    h->unbuilt = true;
    return fail(st, msg + " (the reducer has no buckets until a rebuild succeeds)");
  }
  h->unbuilt = false;
  return DDP_OK;
}

}  // extern "C"
