"""CPU oracle for the bucketed ring all-reduce of DDP's Reducer.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's CPU
baseline may import this package. The library's product path never imports,
links or runs it, and it shares no code with the CUDA library.

Plain, slow and literal: the ring is simulated step by step on a list of numpy
arrays, one per simulated rank, with explicit send payloads, in the order and
notation of the pages it cites. Floating point: the pages fix the arithmetic to
fp32 sums in ring order (bf16 inputs are widened to fp32 and rounded back once),
so the ring runs in fp32; the closed forms and the data-parallel checks that
pin it run in fp64.

Modules
  buckets   bucket assignment, flatten/unflatten, broadcast coalescing
  ring      chunk plan, ring reduce-scatter / all-gather / all-reduce, scale,
            naive send-to-root sum, doubling-tree broadcast, byte counters
  bf16      bf16 <-> fp32 conversions from their definitions
  costs     the cost-model closed forms
  linear_dp data-parallel gradient averaging on a linear model
  trees     recursive doubling, Rabenseifner and binomial-tree all-reduces
  reducer_sim  bucket readiness (mark_variable_ready / mark_bucket_ready),
            overlap timelines, and rebuilding buckets from a ready order

Parity unpinned: none. Every function is pinned by a CPU test against values
the pages print, closed forms, brute force or an independent library routine.
"""
