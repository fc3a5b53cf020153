/*
 * ddp_ring.h -- C ABI of a single-GPU library for the hot path of PyTorch
 * DDP's Reducer: bucketed gradient all-reduce by the two-pass ring, with p
 * simulated ranks whose replica buffers all live in one GPU's memory.
 *
 * Sources, by page title and section:
 *   [DDP]  "PyTorch DDP Deep Dive -- Initialization, Buffer Broadcast, the
 *          Reducer, and the torch.compile Story"
 *   [COLL] "Collective Ops From Scratch"
 *   [DP]   "Data parallelism"
 *
 * Conventions (every call):
 *   - Pointer arrays (bufs, in, out, grads, tensors, bucket) are HOST arrays of
 *     DEVICE pointers. They are read during the call and not kept, except by a
 *     ddp_ring handle, which keeps a copy until ddp_ring_destroy.
 *   - The caller owns every replica, input and output buffer. The library
 *     allocates only:
 *       a handle's device memory, freed by its destroy call: a ddp_ring's
 *       workspace; a ddp_reducer's flat buckets, piece table, buffer table and
 *       workspace;
 *       stream-ordered temporaries (cudaMallocAsync / cudaFreeAsync on the
 *       caller's stream) for the literal schedules of one-shot calls, the
 *       persistent ring's step flags, and the fp32 workspace of the bf16
 *       tree-shaped and persistent all-reduces.
 *     ddp_reduce_scatter_noalloc allocates nothing.
 *   - Work is enqueued on the caller's stream and runs asynchronously to the
 *     host, as DDP's per-bucket futures do ([DDP] Part 2, "Step 3:
 *     finalize_backward"). Only these wait for the device: ddp_ring_sync,
 *     ddp_device_error, ddp_reducer_create (its piece-table upload),
 *     ddp_reducer_set_buffers (its table upload),
 *     ddp_reducer_rebuild (drains the device first), the destroy calls, and
 *     every collective while the call log (DDP_RING_LOG) is on.
 *   - Threads: calls on different handles, or handle-free calls, may run
 *     from several host threads at once. One handle must not be used from
 *     two threads at the same time.
 *   - Errors: every call returns a ddp_status. Argument errors are found on the
 *     host before anything is enqueued. A failed launch returns
 *     DDP_ERR_CUDA. A stream-ordered temporary that cannot be allocated
 *     returns DDP_ERR_NOMEM before any kernel of the call is enqueued, and
 *     leaves no CUDA error pending. ddp_last_error() gives this thread's
 *     last message.
 *   - Replica buffers of one call must be distinct and must not overlap.
 *     Alignment is not required; misaligned heads and tails take a scalar path.
 *   - 1 <= p <= DDP_MAX_P. n == 0 (or nbytes == 0) is a no-op returning DDP_OK
 *     once the scalar arguments are valid; the buffer pointers are then not
 *     read and may be NULL (an empty tensor has no storage). A ddp_ring
 *     handle of n == 0 (zero steps) still needs non-NULL pointer arrays.
 *   - Call log: with the environment variable DDP_RING_LOG=<path> set when
 *     the library first logs, each collective call (ddp_allreduce, _ex,
 *     _persistent, ddp_reduce_scatter, ddp_allgather, ddp_broadcast,
 *     _coalesced, ddp_bucket_allreduce, ddp_reducer_sync, ddp_reducer_step)
 *     appends one JSON
 *     line to <path>: op, algo, p, n, dtype, bytes_algorithmic (inputs read
 *     once, outputs written once), bytes_per_rank (what one simulated rank
 *     sends in the method's schedule, the pages' per-rank byte counter),
 *     status and elapsed_us (CUDA events around the call; null inside a stream
 *     capture or on failure). A timed call waits for its own completion, so
 *     with the log on, calls are synchronous. Without the variable nothing is
 *     recorded and nothing waits.
 *   - Floating point: the sum of p contributions is accumulated in fp32 in
 *     ring order, by IEEE round-to-nearest additions (no FMA contraction, no
 *     reassociation); the scale is one IEEE division; bf16 results are
 *     rounded to nearest even once, at the end.
 */
#ifndef DDP_RING_H
#define DDP_RING_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The library is built with hidden symbol visibility; the entry points
 * declared in this header are the only symbols it exports. */
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

#define DDP_MAX_P 256

typedef enum {
  DDP_OK = 0,
  DDP_ERR_ARG = 1,            /* bad argument (null pointer, range, aliasing)      */
  DDP_ERR_DTYPE = 2,          /* unsupported or mismatched element type            */
  DDP_ERR_NOT_DIVISIBLE = 3,  /* torch-contract reduce_scatter with p not dividing n */
  DDP_ERR_ALIGN = 4,          /* reserved                                          */
  DDP_ERR_NOMEM = 5,          /* a device allocation failed                        */
  DDP_ERR_CUDA = 6,           /* a CUDA call or launch failed                      */
  DDP_ERR_TIMEOUT = 7,        /* a bounded device-side wait gave up                */
  DDP_ERR_STATE = 8           /* handle used out of order (e.g. step after the last) */
} ddp_status;

typedef enum { DDP_FLOAT32 = 0, DDP_BFLOAT16 = 1 } ddp_dtype;

typedef enum {
  DDP_ALGO_FUSED = 0,       /* one pass: read p contributions, write p results; the
                               library picks its fastest one-pass kernel             */
  DDP_ALGO_RING_STEPS = 1,  /* the literal schedule: one launch per ring step         */
  DDP_ALGO_FUSED_LDST = 2,  /* one pass through registers (128-bit loads and stores) */
  DDP_ALGO_FUSED_TMA = 3,   /* one pass staged through shared memory by bulk
                               asynchronous copies, p = 2, 4, 8 or 16 (any other p,
                               replicas at different addresses mod 16, or the
                               per-hop bf16 flag take the register path)            */
  /* Tree-shaped literal all-reduces ([DP] "Latency, trees, and choosing an
   * algorithm"; [COLL] tree all-reduce). ddp_allreduce only; the pairwise
   * tree order, not the ring's. bf16 buffers are widened into a stream-ordered
   * fp32 workspace of p * n floats, reduced there and rounded once at the end
   * (one launch more on each side; DDP_ERR_NOMEM if the workspace fails). */
  DDP_ALGO_RECURSIVE_DOUBLING = 4, /* log2 p steps: pairs r, r^2^j swap and add; p = 2^k */
  DDP_ALGO_RABENSEIFNER = 5,       /* recursive halving (keep lower half if bit d clear),
                                      then recursive doubling of owned chunks; p = 2^k */
  DDP_ALGO_TREE = 6                /* binomial reduce to rank 0, divide there, then the
                                      doubling-tree broadcast; any p                  */
} ddp_algo;

typedef enum {
  DDP_OWN_RANK = 0,  /* rank r <-> chunk r: the torch contract, chunks pre-rotated */
  DDP_OWN_RING = 1   /* rank r <-> chunk (r+1) mod p: where pass 1 leaves them     */
} ddp_own;

typedef enum {
  DDP_ORDER_REVERSED = 0,     /* walk last-registered first; bucket 0 gets the first cap   */
  DDP_ORDER_REGISTRATION = 1  /* walk in registration order, first cap on that walk's
                                 bucket 0, then reverse the bucket list                  */
} ddp_border;

/* Flags of ddp_allreduce_ex. */
#define DDP_FLAG_ROUND_EACH_HOP 1u

typedef enum {
  DDP_SYNC_FLATTEN = 0,  /* per bucket: flatten, all-reduce the flat bucket; then unflatten */
  DDP_SYNC_IN_PLACE = 1  /* per bucket: one pass over the gradients themselves            */
} ddp_sync_mode;

typedef enum {
  DDP_OP_ALLREDUCE = 0,
  DDP_OP_REDUCE_SCATTER = 1,
  DDP_OP_ALLGATHER = 2,
  DDP_OP_BROADCAST = 3
} ddp_op;

/* ------------------------------------------------------------------ buckets */

/* Bucket assignment by size. [DDP] Part 1, "What _ddp_init_helper actually
 * does" (buckets handed to the Reducer reversed; small first bucket, 1 MB by
 * default) and Part 3, DDPOptimizer's compile_fn (reverse walk; a new bucket
 * once the current one reaches bucket_bytes_cap, or first_bucket_cap for the
 * first); [DP] "Overlapping communication with the backward pass" (~25 MB).
 *
 * Walks the k tensors in `order`; each whole tensor joins the open bucket; the
 * bucket closes once its byte size (elements * elem_size) is >= its cap:
 * first_bucket_cap_bytes for bucket 0, bucket_cap_bytes after. Tensors are
 * never split; no empty bucket is produced. Host-only: no CUDA call.
 *   numel[k]            element count of tensor t, registration order, >= 0
 *   out n_buckets       number of buckets B (0 when k == 0)
 *   out bucket_of[k]    bucket of tensor t
 *   out offset[k]       element offset of tensor t inside its bucket
 *                       (exclusive prefix sum in walk order)
 *   out bucket_ptr[k+1] CSR row pointers: bucket b's tensors are
 *                       bucket_tensors[bucket_ptr[b] .. bucket_ptr[b+1])
 *   out bucket_tensors[k] tensor indices in walk order
 *   out bucket_numel[k] element count of each bucket (first B entries used)
 * Errors: DDP_ERR_ARG for k < 0, null arrays (k > 0), elem_size <= 0,
 * negative numel or caps, or an unknown order. */
ddp_status ddp_bucket_assign(int32_t k, const int64_t* numel, int32_t elem_size,
                             int64_t first_bucket_cap_bytes, int64_t bucket_cap_bytes,
                             ddp_border order, int32_t* n_buckets, int32_t* bucket_of,
                             int64_t* offset, int32_t* bucket_ptr, int32_t* bucket_tensors,
                             int64_t* bucket_numel);

/* Bucket assignment along an explicit walk: the rebuild of [DDP] Part 2
 * ("_rebuild_buckets": buckets rebuilt from the order in which gradients were
 * observed to become ready). walk[k] is a permutation of 0..k-1, first-ready
 * first; bucket 0 gets the first cap; a bucket closes once its bytes reach its
 * cap; the list is not reversed. Outputs as ddp_bucket_assign. Host-only.
 * DDP_ERR_ARG if walk is not a permutation. */
ddp_status ddp_bucket_assign_order(int32_t k, const int64_t* numel, int32_t elem_size,
                                   int64_t first_bucket_cap_bytes, int64_t bucket_cap_bytes,
                                   const int32_t* walk, int32_t* n_buckets, int32_t* bucket_of,
                                   int64_t* offset, int32_t* bucket_ptr, int32_t* bucket_tensors,
                                   int64_t* bucket_numel);

/* Copy each replica's k gradients into its flat bucket. [DDP] Part 2
 * "Step 2: backward", mark_variable_ready: each parameter's gradient is
 * copied into its slice of the bucket's flat tensor, optionally pre-divided.
 *   grads[p*k]  grads[r*k + j]: replica r's tensor j (numel[j] elements, dtype)
 *   numel[k], offset[k]: element count and bucket offset of tensor j
 *   bucket[p]   replica r's flat bucket (>= max(offset[j]+numel[j]) elements)
 *   predivide   1.0f: plain copy; otherwise y = round(fl32(x / predivide))
 * Tensors must not overlap the buckets. Zero-element tensors are skipped. */
ddp_status ddp_bucket_flatten(int32_t p, int32_t k, const void* const* grads,
                              const int64_t* numel, const int64_t* offset,
                              void* const* bucket, ddp_dtype dtype, float predivide,
                              cudaStream_t stream);

/* Copy each replica's flat bucket back into its k gradients (the inverse of
 * ddp_bucket_flatten). [DDP] Part 2 "Step 3: finalize_backward": the reduced
 * flat tensor is copied back into the per-parameter gradient views (skipped by
 * callers whose gradients are already bucket views). Same layout as above. */
ddp_status ddp_bucket_unflatten(int32_t p, int32_t k, const void* const* bucket,
                                const int64_t* numel, const int64_t* offset,
                                void* const* grads, ddp_dtype dtype, cudaStream_t stream);

/* ------------------------------------------------------------ collectives */

/* All-reduce in place over p replica buffers of n elements. [COLL] "Ring
 * allreduce in two passes"; [DP] "Ring all-reduce, derived" and "Overlapping
 * communication with the backward pass" (DDP divides the sum by the number of
 * ranks); [DP] "Why averaging gradients is exactly large-batch training"
 * (divide once by the global token count).
 * With cs = ceil(n/p) and chunk c = [c*cs, min(n, (c+1)*cs)), every element i
 * of chunk c becomes, on every replica,
 *     y = fl32( (((x_c + x_{c+1}) + x_{c+2}) + ... + x_{c+p-1}) / divisor )
 * with replica indices mod p: the order in which the ring's reduce-scatter
 * accumulates chunk c, starting at rank c. bf16 inputs are widened to fp32,
 * and y is rounded to bf16 (nearest even). divisor: 1 (sum), p (average) or a
 * token count; must be finite and non-zero.
 * algo DDP_ALGO_FUSED / _FUSED_LDST / _FUSED_TMA: one pass, the same bits;
 * RING_STEPS: 2(p-1) launches of the literal schedule (bf16 keeps fp32
 * partials in a stream-ordered temporary). */
ddp_status ddp_allreduce(void* const* bufs, int32_t p, int64_t n, ddp_dtype dtype,
                         float divisor, ddp_algo algo, cudaStream_t stream);

/* ddp_allreduce with variant flags (0 gives ddp_allreduce exactly).
 *   DDP_FLAG_ROUND_EACH_HOP (bf16 only, else DDP_ERR_DTYPE): the partials
 *   travel as bf16, as a bf16 wire format would carry them ([COLL] "Ring
 *   allreduce in two passes": the receiver accumulates the received chunk into
 *   its local copy, here a bf16 copy). After every local + received (an fp32
 *   add) the sum is rounded to bf16; the owner's y = RNE_bf16(fl32(sum / D)).
 *   Literal (RING_STEPS) and fused forms give the same bits; _FUSED_TMA runs
 *   the register-path kernel for this variant. */
ddp_status ddp_allreduce_ex(void* const* bufs, int32_t p, int64_t n, ddp_dtype dtype, float divisor,
                            ddp_algo algo, uint32_t flags, cudaStream_t stream);

/* The literal 2(p-1)-step ring as one persistent cooperative kernel with
 * device-side step synchronisation, bounded waits and host-set fault
 * injection. [COLL] "Ring allreduce in two passes" (rank r receives from
 * r - 1 each step) and its exercise on a configurable receive timeout that
 * surfaces a deadline error instead of waiting forever.
 * Same result as ddp_allreduce, bit for bit. bf16 buffers are widened into a
 * stream-ordered fp32 workspace of p * n floats, the ring runs there and each
 * finished value is rounded to bf16 once (DDP_ERR_NOMEM if the workspace
 * cannot be had); after a wait ran out their contents are unspecified.
 * Each simulated rank gets blocks of its own; receiver d waits, before step t,
 * until its sender d-1 has posted t steps. A wait gives up after timeout_ns
 * (0 means 1 s); the kernel then records the failure and ends (no trap).
 *   fault_rank, fault_step: inject "rank fault_rank never posts step
 *     fault_step" (it stops before that step); -1 for no fault.
 *   status: NULL, or 4 device int32 words the caller owns, zeroed by the call
 *     and written by the kernel: {0 or DDP_ERR_TIMEOUT, the rank whose wait
 *     gave up first, the step it waited for, number of waits that gave up}.
 * A wait that ran out also sets the library's device error word
 * (ddp_device_error returns DDP_ERR_TIMEOUT). Buffers are then only partly
 * reduced. Needs p co-resident blocks (DDP_ERR_ARG otherwise); the step flags
 * are a stream-ordered temporary. */
ddp_status ddp_allreduce_persistent(void* const* bufs, int32_t p, int64_t n, ddp_dtype dtype, float divisor,
                                    int64_t timeout_ns, int32_t fault_rank, int32_t fault_step,
                                    int32_t* status, cudaStream_t stream);

/* Reduce-scatter: pass 1 alone. [COLL] code/main.py list (reduce_scatter
 * pre-rotates so rank r returns the sum of chunk r and rejects element counts
 * not divisible by the world size); [DP] "The collective operations".
 *   in[p]:  n elements each (not modified)
 *   out[p]: DDP_OWN_RANK: out[r] = chunk r, summed from rank r+1 around to
 *           rank r; needs p | n (else DDP_ERR_NOT_DIVISIBLE), n/p elements.
 *           DDP_OWN_RING: out[q] = chunk (q+1) mod p, summed from rank q+1;
 *           only the chunk's real elements are written (the padding is
 *           trimmed); out[q] needs room for ceil(n/p) elements.
 * Each value is fl32(sum / divisor), rounded to dtype. out must not overlap in. */
ddp_status ddp_reduce_scatter(const void* const* in, void* const* out, int32_t p, int64_t n,
                              ddp_dtype dtype, float divisor, ddp_own own, ddp_algo algo,
                              cudaStream_t stream);

/* All-gather: pass 2 alone. [COLL] code/main.py list (N-1 rotations);
 * [DP] "Ring all-reduce, derived" (all-gather step k sends chunk (r+1-k) mod p).
 *   in[p]:  m elements each: rank r's finished chunk, chunk r (DDP_OWN_RANK) or
 *           chunk (r+1) mod p (DDP_OWN_RING)
 *   out[p]: p*m elements each; every out[r] ends holding all chunks in order.
 * A copy: bit-exact, no scaling. out must not overlap in. The fused forms
 * read each chunk once and write it p times: _FUSED_LDST through registers,
 * _FUSED_TMA by bulk copies through shared memory (8 KB tiles; where a source
 * and a destination differ modulo 16 bytes, registers), _FUSED the bulk
 * copies with 7 or more destinations from 64 MiB read in all, else registers.
 * Same fan-out for ddp_broadcast. */
ddp_status ddp_allgather(const void* const* in, void* const* out, int32_t p, int64_t m,
                         ddp_dtype dtype, ddp_own own, ddp_algo algo, cudaStream_t stream);

/* Broadcast nbytes from bufs[root] to every other replica. [COLL] code/main.py
 * list (broadcast over a doubling tree). RING_STEPS runs the tree: with
 * v = (r - root) mod p, at step j every v < 2^j copies to v + 2^j (< p);
 * ceil(log2 p) launches. FUSED reads the root once and writes p-1 copies
 * (the fused forms as for ddp_allgather). */
ddp_status ddp_broadcast(void* const* bufs, int32_t p, int64_t nbytes, int32_t root,
                         ddp_algo algo, cudaStream_t stream);

/* Coalesced broadcast of k tensors from replica root. [DDP] Part 2, the
 * annotated trace: dist._broadcast_coalesced packs tensors into buckets of at
 * most 250 * 1024 * 1024 bytes, flattens each, broadcasts it from the root,
 * unflattens and copies back; this is the per-forward buffer sync of DDP
 * (BatchNorm running statistics).
 *   tensors[p*k]: tensors[r*k + j] is replica r's tensor j, nbytes[j] bytes
 *   bucket_cap_bytes: 0 means 250 MiB. Tensors join a bucket in order; a new
 *   bucket starts when the next tensor would take it over the cap.
 * RING_STEPS packs each bucket on the root, runs the doubling tree on the
 * packed buffers (a temporary of p * bucket bytes) and unpacks; FUSED copies
 * each root tensor straight to the p-1 others (same bytes). */
ddp_status ddp_broadcast_coalesced(int32_t p, int32_t k, void* const* tensors,
                                   const int64_t* nbytes, int32_t root,
                                   int64_t bucket_cap_bytes, ddp_algo algo,
                                   cudaStream_t stream);

/* All-reduce of one bucket straight on the gradients: the result of
 * ddp_bucket_flatten, ddp_allreduce(DDP_ALGO_FUSED) on the flat bucket and
 * ddp_bucket_unflatten, bit for bit, in one pass that reads every replica's
 * gradients once and writes them once (no flat buffer). [DDP] Part 2,
 * mark_variable_ready / all_reduce_bucket / finalize_backward; [COLL] "Ring
 * allreduce in two passes". Element e of tensor j sits at bucket position
 * offset[j] + e, in chunk (offset[j] + e) / ceil(n/p) with n = max(offset[j] +
 * numel[j]); it is summed in that chunk's ring order and divided by divisor.
 *   grads[p*k]: grads[r*k + j] is replica r's tensor j (in place);
 *   numel[k], offset[k]: as from ddp_bucket_assign. Tensors must not overlap. */
ddp_status ddp_bucket_allreduce(int32_t p, int32_t k, void* const* grads, const int64_t* numel,
                                const int64_t* offset, ddp_dtype dtype, float divisor,
                                cudaStream_t stream);

/* ------------------------------------------------------------- reducer */

/* A Reducer for p replicas: the gradient synchronisation of [DDP] Part 2 in
 * one call. ddp_reducer_create assigns the buckets (ddp_bucket_assign with
 * the given caps and order), allocates every replica's flat buckets (handle
 * workspace, freed by ddp_reducer_destroy) and plans every launch once.
 *   grads[p*k]: grads[r*k + t] is replica r's gradient t (registration order),
 *   numel[k] elements each; kept (not copied) until destroy.
 * ddp_reducer_sync enqueues, on `stream`, one synchronisation:
 *   DDP_SYNC_FLATTEN: for every bucket in order, ddp_bucket_flatten (with
 *     predivide) then ddp_allreduce with `algo`; then ddp_bucket_unflatten of
 *     every bucket ([DDP] "Step 3: finalize_backward").
 *   DDP_SYNC_IN_PLACE: every bucket's ddp_bucket_allreduce, all in ONE launch
 *     driven by a piece table uploaded to device memory at create (fused
 *     algos only; predivide must be 1). Tiles are ordered bucket by bucket.
 *     DDP_ALGO_FUSED_TMA stages each 2 KB tile of every replica in shared
 *     memory by bulk asynchronous copies before the fold (p = 2, 4, 8 or 16;
 *     other p take the register form); a copy that does not complete within
 *     2 s sets ddp_device_error() to 1 and leaves that tile unwritten.
 *     DDP_ALGO_FUSED_LDST folds in registers; DDP_ALGO_FUSED takes the form
 *     that ddp_reducer_staged reports.
 * Both give the same bits. */
typedef struct ddp_reducer ddp_reducer;
ddp_status ddp_reducer_create(ddp_reducer** handle, int32_t p, int32_t k, void* const* grads,
                              const int64_t* numel, ddp_dtype dtype, int64_t first_bucket_cap_bytes,
                              int64_t bucket_cap_bytes, ddp_border order);
/* Number of buckets; -1 for a null handle. */
int32_t ddp_reducer_num_buckets(const ddp_reducer* handle);
/* 1 if this reducer's ddp_reducer_step and its in-place ddp_reducer_sync
 * with DDP_ALGO_FUSED stage every tile in shared memory by bulk copies (the
 * _FUSED_TMA form), 0 if they fold in registers (the _FUSED_LDST form); -1
 * for a null handle. The choice depends only on the dtype and p: the form
 * that measured faster on GB300 (staged for fp32 at p = 4 or 8 and for bf16
 * at p = 2 or 4). Both give the same bits. */
int32_t ddp_reducer_staged(const ddp_reducer* handle);
/* Bucket b's element count and (if flat != NULL) its p flat buffers. */
ddp_status ddp_reducer_bucket(const ddp_reducer* handle, int32_t b, int64_t* numel, void** flat);
ddp_status ddp_reducer_sync(ddp_reducer* handle, float divisor, float predivide, ddp_algo algo,
                            ddp_sync_mode mode, cudaStream_t stream);
ddp_status ddp_reducer_destroy(ddp_reducer* handle);

/* The per-forward buffer broadcast and the gradient sync in ONE launch.
 * [DDP] Part 2: every forward starts with _sync_buffers, a
 * _broadcast_coalesced of the module's buffers from rank 0 (the annotated
 * trace), and every backward ends with the Reducer's bucket all-reduces
 * (mark_variable_ready / finalize_backward).
 * ddp_reducer_set_buffers attaches k buffers to the reducer:
 *   tensors[p*k]: tensors[r*k + j] is replica r's buffer j (device pointers,
 *   kept, not copied, until the next set_buffers or destroy), nbytes[k] bytes
 *   each, root: the replica whose buffers are copied to the others. The copy
 *   is bitwise, whatever the buffers' own dtypes, but each buffer's bytes must
 *   be a multiple of the gradients' element size (DDP_ERR_ARG) and every
 *   pointer aligned to it (DDP_ERR_ALIGN). Buffers must not overlap one
 *   another or any gradient of the reducer (DDP_ERR_ARG). The buffers join the
 *   reducer's piece table, which is rebuilt in device memory: the call waits
 *   for the device. If that allocation fails (DDP_ERR_NOMEM), no buffers stay
 *   attached and the reducer refuses sync, step, prepare and mark_ready
 *   (DDP_ERR_STATE) until a ddp_reducer_rebuild succeeds. k == 0 detaches.
 *   A null handle, k < 0, root outside [0, p), null arrays with k > 0 or a
 *   null buffer of nonzero size: DDP_ERR_ARG, and nothing changes. The
 *   buffers stay attached across ddp_reducer_rebuild.
 * ddp_reducer_step enqueues on `stream` one launch that does both: the
 *   attached buffers copied from root to every other replica (the bits of
 *   ddp_broadcast_coalesced; the root's buffers are read, not written) and
 *   every bucket's in-place sync with `divisor` (the bits of
 *   ddp_reducer_sync with DDP_SYNC_IN_PLACE, which never touches the
 *   buffers). The two touch disjoint memory, so the result equals the two
 *   calls in either order. In a training loop it is the sync at the end of
 *   backward together with the buffer broadcast that the next forward needs
 *   (nothing between the two reads or writes the buffers). With no buffers
 *   attached it is ddp_reducer_sync(DDP_SYNC_IN_PLACE). Same errors as
 *   ddp_reducer_sync. */
ddp_status ddp_reducer_set_buffers(ddp_reducer* handle, int32_t k, void* const* tensors,
                                   const int64_t* nbytes, int32_t root);
ddp_status ddp_reducer_step(ddp_reducer* handle, float divisor, cudaStream_t stream);

/* Readiness-driven firing, as the Reducer's hooks do it during backward
 * ([DDP] Part 2 "Step 2: backward": mark_variable_ready decrements the
 * bucket's pending count; mark_bucket_ready reduces every contiguous complete
 * bucket from next_bucket_ on, strictly in order; [DP] "Overlapping
 * communication with the backward pass": the all-reduce runs on a separate
 * stream while backward continues).
 * ddp_reducer_prepare resets the pending counts and the observed order.
 * ddp_reducer_mark_ready marks gradient `tensor` (registration index) ready:
 *   if that completes bucket next_bucket_ (and the ones after it), each of
 *   them is all-reduced in place (ddp_bucket_allreduce with divisor; the grid
 *   as ddp_reducer_set_comm_blocks set it) on comm_stream, which first waits
 *   on `ready` (if not NULL: the event after
 *   which the gradient holds its final value; events must complete in marking
 *   order, e.g. all recorded on one producing stream). *fired (if not NULL)
 *   = number of buckets launched by this call. DDP_ERR_STATE if the tensor was
 *   already marked since the last prepare.
 * ddp_reducer_observed writes the ready order seen since the last prepare
 *   into order (if not NULL) and returns its length (-1 for a null handle).
 * ddp_reducer_rebuild rebuilds the buckets along `order` (a permutation of
 *   0..k-1, first-ready first) or, if order is NULL, along the observed order
 *   (DDP_ERR_STATE unless every tensor was marked); reallocates the flat
 *   buckets and tables (it synchronizes the device) and resets readiness.
 *   If the rebuild fails after the old buckets were released (an allocation
 *   returns DDP_ERR_NOMEM), the handle keeps no buckets and no device memory:
 *   ddp_reducer_sync, _prepare and _mark_ready then return DDP_ERR_STATE
 *   until a rebuild succeeds; destroy works as always. */
ddp_status ddp_reducer_prepare(ddp_reducer* handle);
/* The grid of the bucket launches ddp_reducer_mark_ready fires: max_blocks
 * == 0 (the default) gives one block per 2 KB tile; max_blocks > 0 at most
 * that many blocks, each striding over the bucket's tiles, as a collective
 * library bounds its kernels to a few channels. A bounded grid holds at most
 * max_blocks / (blocks resident per SM) SMs, so a backward pass running on
 * another stream keeps the others ([DP] "Overlapping communication with the
 * backward pass"). Results are the same bits for every value.
 * DDP_ERR_ARG if max_blocks < 0. */
ddp_status ddp_reducer_set_comm_blocks(ddp_reducer* handle, int32_t max_blocks);
ddp_status ddp_reducer_mark_ready(ddp_reducer* handle, int32_t tensor, float divisor, cudaEvent_t ready,
                                  cudaStream_t comm_stream, int32_t* fired);
int32_t ddp_reducer_observed(const ddp_reducer* handle, int32_t* order);
ddp_status ddp_reducer_rebuild(ddp_reducer* handle, const int32_t* order);


/* Reduce-scatter that allocates nothing. No counterpart in the paper: it exists
 * for callers that cannot allocate device memory during a call -- for example a
 * framework whose caching allocator already owns all of the device's memory, or
 * code that must not risk an allocation failing, or synchronising, in the
 * middle of a training step.
 * Same arguments, layout, ownerships, results and errors as ddp_reduce_scatter
 * with DDP_ALGO_RING_STEPS (the literal p-1 step ring), but the fp32 partials
 * live in a fixed 8 MiB device array inside the library instead of a
 * temporary: it calls no cudaMalloc, cudaMallocAsync or cudaFree.
 *   Limit: 2 * p * ceil(n/p) * 4 bytes <= 8 MiB (p * ceil(n/p) <= 1,048,576
 *   elements); larger calls return DDP_ERR_ARG with a message and enqueue
 *   nothing. p == 1 needs no scratch and has no limit.
 *   The array is one per device, shared by every call, and keeps the last
 *   call's contents (no call depends on them). Calls whose work overlaps on the
 *   GPU (different streams, or threads) race on it: order them on one stream.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture. The address is kept for as long as the
 *   device's context lives: after a cudaDeviceReset the next call looks it
 *   up again in the new context (so that call, too, should come before any
 *   capture). Every GPU that loads the library holds the 8 MiB until the
 *   process exits.
 *   n == 0 returns DDP_OK without reading the pointers, as ddp_reduce_scatter
 *   does. */
ddp_status ddp_reduce_scatter_noalloc(const void* const* in, void* const* out, int32_t p, int64_t n,
                                      ddp_dtype dtype, float divisor, ddp_own own, cudaStream_t stream);

/* ------------------------------------------- literal schedule, stepwise */

/* A handle that runs one collective's literal schedule one step at a time, so
 * the state after every step can be read. [COLL] "Ring allreduce in two
 * passes"; [DP] "Ring all-reduce, derived".
 *   op ALLREDUCE:      bufs = in (in place, n elements), out = NULL.
 *                      2(p-1) steps (1 for p == 1): step s < p-1 is
 *                      reduce-scatter step s (rank r's chunk (r-s) mod p is
 *                      accumulated into rank r+1; the last one also divides the
 *                      owner's chunk by divisor); then all-gather steps.
 *                      fp32 partials live in the buffers; bf16 partials in the
 *                      handle's fp32 workspace.
 *   op REDUCE_SCATTER: in (n elements), out (as ddp_reduce_scatter); p-1 steps
 *                      (1 for p == 1); partials in the workspace.
 *   op ALLGATHER:      in (m = n elements), out (p*n); p-1 steps (1 for p == 1);
 *                      step 0 also places each rank's own chunk.
 *   op BROADCAST:      in = bufs (n bytes), out = NULL, root; ceil(log2 p) steps.
 * Workspace (REDUCE_SCATTER, and bf16 ALLREDUCE): 2 * p * ceil(n/p) fp32,
 * laid out [2][p][ceil(n/p)]; reduce-scatter step s writes half (s & 1), slot
 * d = receiving rank, element e = offset inside the chunk.
 * The handle keeps copies of the pointer arrays and enqueues on `stream`. */
typedef struct ddp_ring ddp_ring;

ddp_status ddp_ring_create(ddp_ring** handle, ddp_op op, void* const* in, void* const* out,
                           int32_t p, int64_t n, ddp_dtype dtype, float divisor, ddp_own own,
                           int32_t root, cudaStream_t stream);
/* Total number of steps; -1 for a null handle. */
int32_t ddp_ring_num_steps(const ddp_ring* handle);
/* Steps enqueued so far; -1 for a null handle. */
int32_t ddp_ring_steps_done(const ddp_ring* handle);
/* Enqueue the next step. DDP_ERR_STATE once all steps are enqueued. */
ddp_status ddp_ring_step(ddp_ring* handle);
/* The fp32 workspace (NULL and 0 if this handle has none). */
ddp_status ddp_ring_workspace(const ddp_ring* handle, void** fp32_partials,
                              int64_t* elems_per_slot);
/* Bytes rank `rank` has sent so far on the simulated wire: each ring send is
 * one chunk of ceil(n/p) elements (padding included) at the buffer's element
 * size; each tree send is n bytes. */
ddp_status ddp_ring_bytes_sent(const ddp_ring* handle, int32_t rank, int64_t* bytes);
/* Wait for the handle's stream and report any device-side error. */
ddp_status ddp_ring_sync(ddp_ring* handle);
/* Free the handle and its workspace (after the stream's work is done). */
ddp_status ddp_ring_destroy(ddp_ring* handle);

/* ----------------------------------------------------------------- misc */

/* Synchronize `stream`, then read and clear the library's device error word:
 * *code = 0 when no kernel reported a problem, else the first code a kernel
 * recorded (a bounded wait that gave up): 1 a bulk copy of a shared-memory
 * staged kernel (DDP_ALGO_FUSED_TMA, or a staged in-place sync or step) did
 * not complete within 2 s, and that block stored nothing; 2 a persistent
 * ring step's wait ran out. Returns DDP_ERR_TIMEOUT if set. */
ddp_status ddp_device_error(cudaStream_t stream, int32_t* code);
/* Number of kernels this library has launched in this process. */
int64_t ddp_kernel_launches(void);
/* Text of this thread's last error (empty if none). */
const char* ddp_last_error(void);
/* Fixed name of a status code. */
const char* ddp_status_string(ddp_status s);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#ifdef __cplusplus
}
#endif
#endif /* DDP_RING_H */
