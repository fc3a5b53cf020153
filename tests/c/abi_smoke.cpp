// The C ABI driven from C++ with nothing but the CUDA runtime: no Python, no
// torch. Small-integer inputs make every sum exact, so the expected values are
// plain arithmetic and the check does not depend on the summation order.
// Prints "ok" and exits 0 when every check passes.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include <cuda_runtime.h>

#include "ddp_ring.h"

#define CHECK(cond, msg)                                          \
  do {                                                            \
    if (!(cond)) {                                                \
      std::printf("FAIL %s (line %d): %s\n", msg, __LINE__, ddp_last_error()); \
      return 1;                                                   \
    }                                                             \
  } while (0)

static int allreduce_case(int p, int64_t n, ddp_algo algo, cudaStream_t s) {
  std::vector<void*> bufs(p);
  std::vector<float> host(n);
  for (int r = 0; r < p; ++r) {
    CHECK(cudaMalloc(&bufs[r], n * sizeof(float)) == cudaSuccess, "cudaMalloc");
    for (int64_t i = 0; i < n; ++i) host[i] = static_cast<float>((i * 7 + r * 3) % 11) - 5.0f;
    CHECK(cudaMemcpy(bufs[r], host.data(), n * sizeof(float), cudaMemcpyHostToDevice) == cudaSuccess, "upload");
  }
  CHECK(ddp_allreduce(bufs.data(), p, n, DDP_FLOAT32, 1.0f, algo, s) == DDP_OK, "ddp_allreduce");
  CHECK(cudaStreamSynchronize(s) == cudaSuccess, "sync");
  for (int r = 0; r < p; ++r) {
    CHECK(cudaMemcpy(host.data(), bufs[r], n * sizeof(float), cudaMemcpyDeviceToHost) == cudaSuccess, "download");
    for (int64_t i = 0; i < n; ++i) {
      float want = 0.0f;
      for (int q = 0; q < p; ++q) want += static_cast<float>((i * 7 + q * 3) % 11) - 5.0f;
      CHECK(host[i] == want, "all-reduce value");
    }
    cudaFree(bufs[r]);
  }
  return 0;
}

int main() {
  cudaStream_t s;
  if (cudaStreamCreate(&s) != cudaSuccess) {
    std::printf("FAIL no stream\n");
    return 1;
  }
  // the all-reduce in its fused, literal and tree-shaped forms, ragged sizes
  const ddp_algo algos[] = {DDP_ALGO_FUSED, DDP_ALGO_RING_STEPS, DDP_ALGO_TREE};
  for (ddp_algo a : algos)
    for (int p : {2, 3, 8})
      if (allreduce_case(p, 10007, a, s)) return 1;

  // reduce-scatter, ring ownership: rank q gets chunk (q + 1) mod p
  {
    const int p = 4;
    const int64_t n = 1003, cs = (n + p - 1) / p;
    std::vector<void*> in(p), out(p);
    std::vector<float> host(n, 0.0f);
    for (int r = 0; r < p; ++r) {
      for (int64_t i = 0; i < n; ++i) host[i] = static_cast<float>(r + 1);
      CHECK(cudaMalloc(&in[r], n * sizeof(float)) == cudaSuccess, "cudaMalloc in");
      CHECK(cudaMalloc(&out[r], cs * sizeof(float)) == cudaSuccess, "cudaMalloc out");
      CHECK(cudaMemcpy(in[r], host.data(), n * sizeof(float), cudaMemcpyHostToDevice) == cudaSuccess, "upload");
    }
    CHECK(ddp_reduce_scatter(in.data(), out.data(), p, n, DDP_FLOAT32, 2.0f, DDP_OWN_RING, DDP_ALGO_FUSED, s) == DDP_OK,
          "ddp_reduce_scatter");
    CHECK(cudaStreamSynchronize(s) == cudaSuccess, "sync");
    for (int q = 0; q < p; ++q) {
      const int64_t c = (q + 1) % p, lo = c * cs, hi = (lo + cs < n) ? lo + cs : n;
      std::vector<float> got(cs);
      CHECK(cudaMemcpy(got.data(), out[q], cs * sizeof(float), cudaMemcpyDeviceToHost) == cudaSuccess, "download");
      for (int64_t i = 0; i < hi - lo; ++i) CHECK(got[i] == 5.0f, "reduce-scatter value");  // (1+2+3+4)/2
      cudaFree(in[q]);
      cudaFree(out[q]);
    }
  }

  // a Reducer over two tensors per replica, whole-set sync in place, then the one-launch step
  {
    const int p = 2, k = 2;
    const int64_t numel[k] = {300, 5000};
    std::vector<void*> grads(p * k);
    for (int r = 0; r < p; ++r)
      for (int t = 0; t < k; ++t) {
        CHECK(cudaMalloc(&grads[r * k + t], numel[t] * sizeof(float)) == cudaSuccess, "cudaMalloc grad");
        std::vector<float> v(numel[t], static_cast<float>(10 * (r + 1) + t));
        CHECK(cudaMemcpy(grads[r * k + t], v.data(), numel[t] * sizeof(float), cudaMemcpyHostToDevice) == cudaSuccess,
              "upload grad");
      }
    ddp_reducer* h = nullptr;
    CHECK(ddp_reducer_create(&h, p, k, grads.data(), numel, DDP_FLOAT32, 1024, 4096, DDP_ORDER_REVERSED) == DDP_OK,
          "ddp_reducer_create");
    CHECK(ddp_reducer_num_buckets(h) >= 1, "buckets");
    CHECK(ddp_reducer_staged(h) == 0 && ddp_reducer_staged(nullptr) == -1, "ddp_reducer_staged");  // fp32, p = 2: registers
    CHECK(ddp_reducer_sync(h, 2.0f, 1.0f, DDP_ALGO_FUSED, DDP_SYNC_IN_PLACE, s) == DDP_OK, "ddp_reducer_sync");
    CHECK(cudaStreamSynchronize(s) == cudaSuccess, "sync");
    for (int r = 0; r < p; ++r)
      for (int t = 0; t < k; ++t) {
        std::vector<float> v(numel[t]);
        CHECK(cudaMemcpy(v.data(), grads[r * k + t], numel[t] * sizeof(float), cudaMemcpyDeviceToHost) == cudaSuccess,
              "download grad");
        const float want = (10.0f + t + 20.0f + t) / 2.0f;
        for (int64_t i = 0; i < numel[t]; ++i) CHECK(v[i] == want, "reducer value");
      }
    // one buffer per replica attached: the step copies replica 1's to replica 0 and syncs again
    const int64_t nb = 64;
    std::vector<void*> bufs(p);
    for (int r = 0; r < p; ++r) {
      CHECK(cudaMalloc(&bufs[r], nb * sizeof(float)) == cudaSuccess, "cudaMalloc buffer");
      std::vector<float> v(nb, static_cast<float>(100 + r));
      CHECK(cudaMemcpy(bufs[r], v.data(), nb * sizeof(float), cudaMemcpyHostToDevice) == cudaSuccess, "upload buffer");
    }
    const int64_t nbytes[1] = {nb * static_cast<int64_t>(sizeof(float))};
    CHECK(ddp_reducer_set_buffers(h, 1, bufs.data(), nbytes, 1) == DDP_OK, "ddp_reducer_set_buffers");
    CHECK(ddp_reducer_step(h, 1.0f, s) == DDP_OK, "ddp_reducer_step");
    CHECK(cudaStreamSynchronize(s) == cudaSuccess, "sync");
    for (int r = 0; r < p; ++r) {
      std::vector<float> v(nb);
      CHECK(cudaMemcpy(v.data(), bufs[r], nb * sizeof(float), cudaMemcpyDeviceToHost) == cudaSuccess, "download buffer");
      for (int64_t i = 0; i < nb; ++i) CHECK(v[i] == 101.0f, "buffer broadcast from replica 1");
      for (int t = 0; t < k; ++t) {
        std::vector<float> g(numel[t]);
        CHECK(cudaMemcpy(g.data(), grads[r * k + t], numel[t] * sizeof(float), cudaMemcpyDeviceToHost) == cudaSuccess,
              "download grad");
        const float want = 2.0f * (10.0f + t + 20.0f + t) / 2.0f;  // two equal copies summed, divisor 1
        for (int64_t i = 0; i < numel[t]; ++i) CHECK(g[i] == want, "step value");
      }
    }
    CHECK(ddp_reducer_destroy(h) == DDP_OK, "ddp_reducer_destroy");
    for (void* g : grads) cudaFree(g);
    for (void* b : bufs) cudaFree(b);
  }

  // errors come back as codes, with this thread's text
  {
    void* nothing[2] = {nullptr, nullptr};
    const ddp_status st = ddp_allreduce(nothing, 2, 16, DDP_FLOAT32, 0.0f, DDP_ALGO_FUSED, s);
    CHECK(st == DDP_ERR_ARG, "bad divisor is an argument error");
    CHECK(std::strstr(ddp_last_error(), "divisor") != nullptr, "error text");
    CHECK(std::strcmp(ddp_status_string(DDP_ERR_ARG), "DDP_ERR_ARG") == 0, "status string");
    int32_t code = -1;
    CHECK(ddp_device_error(s, &code) == DDP_OK && code == 0, "no device error");
  }
  cudaStreamDestroy(s);
  std::printf("ok\n");
  return 0;
}
