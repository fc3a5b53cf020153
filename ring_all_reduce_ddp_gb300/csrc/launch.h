// Host-side launchers of the library's kernels (internal interface between the
// C ABI in api.cu and the kernel translation units).
#pragma once

#include "common.cuh"

namespace ddp {

int sm_count();               // SMs of the current device (cached per device)
void count_launch();          // one more kernel launched by this library
int64_t launches();

cudaError_t launch_fused_reduce(const FusedArgs& a, ddp_dtype dt, bool staged, cudaStream_t s);
cudaError_t launch_rs_step_inplace_f32(const RingStepArgs& a, cudaStream_t s);
cudaError_t launch_rs_step_ws(const RingStepArgs& a, ddp_dtype dt, cudaStream_t s);
// max_blocks > 0 caps the grid: each block then strides over the tiles.
cudaError_t launch_bucket_allreduce(const BucketArgs& a, ddp_dtype dt, cudaStream_t s, int32_t max_blocks = 0);
// algo: DDP_ALGO_FUSED_LDST the register form, DDP_ALGO_FUSED_TMA the
// shared-memory staged form (p = 2, 4, 8, 16; others take the register form),
// DDP_ALGO_FUSED whichever measured faster for the dtype and p.
cudaError_t launch_bucket_table(const BucketTable& t, int32_t total_tiles, float divisor, ddp_dtype dt,
                                cudaStream_t s, ddp_algo algo);
bool staged_by_default(ddp_dtype dt, int p);  // the form DDP_ALGO_FUSED takes in launch_bucket_table
cudaError_t launch_ring_persistent(const PersistArgs& a, cudaStream_t s);
int ring_persistent_max_blocks();  // co-resident blocks of the persistent ring kernel on this device
cudaError_t launch_pair_copy(const PairCopyArgs& a, cudaStream_t s);
cudaError_t launch_pair_add(const PairAddArgs& a, cudaStream_t s);
// algo: DDP_ALGO_FUSED_TMA the TMA bulk-copy form (k_fanout_bulk) when every
// source and destination agree modulo 16 bytes, DDP_ALGO_FUSED_LDST the
// register form (k_fanout), DDP_ALGO_FUSED whichever measured faster for the
// destination count and size.
cudaError_t launch_fanout(const FanoutArgs& a, cudaStream_t s, ddp_algo algo = DDP_ALGO_FUSED_LDST);
cudaError_t launch_seg_copy(const SegCopyArgs& a, ddp_dtype dt, cudaStream_t s);
cudaError_t launch_multi_fanout(const MultiFanoutArgs& a, cudaStream_t s);
cudaError_t launch_convert(const ConvertArgs& a, cudaStream_t s);

// Device address of the library's device error word in the current context.
int* device_error_word();
// Synchronize s, then read and clear the device error word.
cudaError_t read_device_error(cudaStream_t s, int* code);

}  // namespace ddp
