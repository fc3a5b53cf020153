// Device helpers and kernel argument blocks shared by the library's kernels.
//
// Arithmetic rules of the whole library: a sum of p contributions is a left
// fold of IEEE round-to-nearest fp32 additions (__fadd_rn, never contracted or
// reassociated), the scale is one IEEE division (__fdiv_rn), bf16 values are
// widened exactly (bits << 16) and narrowed once with round-to-nearest-even.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "ddp_ring.h"

namespace ddp {

constexpr int kThreads = 256;
constexpr int kMaxP = DDP_MAX_P;

// ---------------------------------------------------------------- elements
__device__ __forceinline__ float widen(float x) { return x; }
__device__ __forceinline__ float widen(__nv_bfloat16 x) {
  return __uint_as_float(static_cast<uint32_t>(__bfloat16_as_ushort(x)) << 16);
}

template <typename T> __device__ __forceinline__ T narrow(float x);
template <> __device__ __forceinline__ float narrow<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 narrow<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// The fp32 value rounded to bf16 (nearest even) and widened back: what a
// partial becomes when it is stored as bf16 between hops.
__device__ __forceinline__ float round_bf16(float x) { return widen(__float2bfloat16_rn(x)); }

// A 16-byte vector seen as N fp32 lanes.
template <typename T> struct Vec;
template <> struct Vec<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                      __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
};
template <> struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void unpack2(uint32_t w, float* f) {
    f[0] = __uint_as_float(w << 16);          // element 2i: low half (little endian)
    f[1] = __uint_as_float(w & 0xFFFF0000u);  // element 2i+1: high half
  }
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    unpack2(v.x, f); unpack2(v.y, f + 2); unpack2(v.z, f + 4); unpack2(v.w, f + 6);
  }
  __device__ __forceinline__ static uint32_t pack2(float a, float b) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(a))) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(b))) << 16);
  }
  __device__ __forceinline__ static uint4 pack(const float* f) {
    return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
  }
};

// ------------------------------------------ programmatic dependent launch
// A kernel started by launch_pdl may begin while the kernel before it in the
// stream drains. It calls pdl_wait() before its first memory access; that
// returns once the earlier kernel has completed and its writes are visible
// (at once for a kernel launched without the attribute). pdl_trigger() lets
// the next such kernel start launching; it fires for a grid only once every
// block has executed it, so a dependent never takes the place of a block of
// the grid before it.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ------------------------------------------------------------ argument blocks

// Fused one-pass reduction (all-reduce, reduce-scatter).
// src holds the p input replicas twice over (src[j] = replica j mod p), so the
// ring order of chunk c, replicas o, o+1, ..., o+p-1 (mod p) with origin o,
// is src[o .. o+p-1] without a modulo.
struct FusedArgs {
  const void* src[2 * kMaxP];
  void* dst[kMaxP];  // all-reduce: the p replicas; reduce-scatter: out[rank]
  int64_t n;         // elements per input replica
  int64_t cs;        // chunk size, ceil(n / p)
  float divisor;
  int p;
  int scatter;       // 0: write y to every dst at index i; 1: to dst[owner] at i - c*cs
  int shift;         // origin of chunk c is (c + shift) mod p
  int same_align;    // every src / dst base has the same address mod 16
  int hop_round;     // bf16 only: round each partial to bf16 after every add
};

// Bucket all-reduce straight on the gradients (flatten + all-reduce +
// unflatten in one pass). A bucket's virtual flat layout is cut into pieces:
// the intersections of its tensors with its chunks, so each piece has one
// summation origin (its chunk index). ptr[slot * p + r] is replica r's tensor
// in local slot `slot`; piece i covers elements [start, start + len) of that
// tensor; tile0 is the prefix of each piece's tiles of bucket_tile_elems
// elements. A tile is 2 KB per replica: one 16-byte vector per thread of a
// 128-thread block, one block per tile. Measured on GB300 that way on the
// ResNet-50-shaped set, with a binary piece search: 4, 8, 16, 32 and 64 KB
// tiles took 244.4, 246.6, 250.4, 259.4 and 264.1 us; on the bf16 Llama-1B
// set 4 KB beat 8 and 64 KB (5,499, 5,517 and 5,677 us). With the warps'
// 32-way piece search, 2, 4 and 8 KB took 238.8-239.0, 239.0-239.9 and
// 247.4-248.1 us on ResNet-50, 1,135-1,136, 1,136-1,138 and 1,159-1,167 us
// on GPT-2, and 5,443-5,444, 5,454-5,455 and 5,843-5,846 us on Llama-1B.
constexpr int kBucketPtrs = 1024;
constexpr int kBucketPieces = 256;
constexpr int kBucketTileBytes = 2048;
constexpr int kBucketThreads = kBucketTileBytes / 16;  // one 16-byte vector per thread and replica
__host__ __device__ constexpr int64_t bucket_tile_elems(int elem_size) { return kBucketTileBytes / elem_size; }
struct BucketArgs {
  void* ptr[kBucketPtrs];
  int64_t start[kBucketPieces];
  int64_t len[kBucketPieces];
  int32_t slot[kBucketPieces];
  int32_t origin[kBucketPieces];
  int32_t tile0[kBucketPieces + 1];
  int npieces, p;
  float divisor;
};

// The same piece table held in device memory (a Reducer's whole set of
// buckets, uploaded once): arrays of npieces entries, ptr of (slots * p).
struct BucketTable {
  void* const* ptr;
  const int64_t* start;
  const int64_t* len;
  const int32_t* slot;
  const int32_t* origin;
  const int32_t* tile0;  // npieces + 1 entries
  int npieces, p;
  int* err;              // the library's device error word (the staged form's bounded waits), or null
};

// Codes of the library's device error word (ddp_device_error).
constexpr int kErrBulkWait = 1;  // a bulk copy did not complete in time
constexpr int kErrRingWait = 2;  // a ring step's wait ran out

// Literal reduce-scatter step. x[r]: replica r's input (const except in the
// fp32 in-place all-reduce); w: fp32 partials [2][p][cs]; out[d]: where the
// last step writes (at chunk-relative index if out_rel, else at i).
struct RingStepArgs {
  void* x[kMaxP];
  void* out[kMaxP];
  float* w;
  int64_t n, cs;
  float divisor;
  int p, step, shift, last, out_rel;
  int hop_round;  // bf16 only: round each partial to bf16 after every add
};

// Persistent literal ring (fp32, in place): every rank's blocks in one
// cooperative launch; block b of rank d handles slice b of each step's chunk
// and waits for block b of rank d-1 to have posted the previous step.
constexpr int kFlagStride = 32;  // ints between two step flags: one 128-byte line each
struct PersistArgs {
  void* buf[kMaxP];
  int* flags;          // [p][blocks_per_rank][kFlagStride]: steps posted (first int); zero at launch
  int* status;         // caller's 4 device words, or null: {code, rank, step, waits that gave up}
  int64_t n, cs;
  float divisor;
  int p, blocks_per_rank;
  int fault_rank, fault_step;  // injected: that rank never posts that step (-1: none)
  int64_t timeout_ns;          // bound of every wait
};

// Pair-add step of the tree-shaped all-reduces (fp32, in place): job j sets
// y = a[j][i] + b[j][i] (then y / divisor if divide) for i in [lo[j], hi[j])
// and stores y to d1[j][i] and, if d2[j] is set, to d2[j][i].
struct PairAddArgs {
  const float* a[kMaxP];
  const float* b[kMaxP];
  float* d1[kMaxP];
  float* d2[kMaxP];
  int64_t lo[kMaxP], hi[kMaxP];
  int njobs, divide;
  float divisor;
};

// Copy jobs: job j copies nbytes[j] bytes from src[j] to dst[j].
struct PairCopyArgs {
  const char* src[kMaxP];
  char* dst[kMaxP];
  int64_t nbytes[kMaxP];
  int njobs;
};

// Precision change of p buffers of n elements each: job j converts src[j]
// into dst[j]; to_bf16 = 0 widens bf16 to fp32 (exact), 1 narrows fp32 to
// bf16 (round to nearest even).
struct ConvertArgs {
  const void* src[kMaxP];
  void* dst[kMaxP];
  int64_t n;
  int njobs;
  int to_bf16;
};

// Fan-out: job j copies nbytes from src[j] to every dst[q] + job_off[j].
struct FanoutArgs {
  const char* src[kMaxP];
  int64_t job_off[kMaxP];
  char* dst[kMaxP];
  int64_t nbytes;
  int njobs, ndst;
  int* err;  // the library's device error word (the bulk-copy form's bounded waits), or null
};

// Segment copy (multi-tensor): segment s copies bytes[s] bytes from src[s] to
// dst[s]; tile0 is the prefix sum of each segment's tile count.
constexpr int kSegCap = 512;
constexpr int kSegTileBytes = 16384;
struct SegCopyArgs {
  const char* src[kSegCap];
  char* dst[kSegCap];
  int64_t bytes[kSegCap];
  int32_t tile0[kSegCap + 1];
  int nseg;
  int elem_size;     // for the dividing copy
  float predivide;   // 1: plain byte copy
};

// Multi-tensor fan-out (coalesced broadcast): tensor t goes from src[t] to
// dst[t * ndst + q] for q < ndst. Sized so that a whole model's buffer set
// (ResNet-50 has 159 BN buffers) goes out in one launch at p = 8; the struct
// (about 21 KB) stays inside the 32 KB kernel-parameter limit.
constexpr int kFanT = 256;
constexpr int kFanD = 2048;
struct MultiFanoutArgs {
  const char* src[kFanT];
  int64_t bytes[kFanT];
  int32_t tile0[kFanT + 1];
  char* dst[kFanD];
  int ntensors, ndst;
};
static_assert(sizeof(MultiFanoutArgs) <= 32764, "kernel parameters are limited to 32764 bytes");

}  // namespace ddp
