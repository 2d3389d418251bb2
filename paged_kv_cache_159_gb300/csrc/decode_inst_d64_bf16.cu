// decode_inst_d64_bf16.cu -- compiles the decode kernels for head_dim 64 with a bf16 pool.
#include "decode_kernels.cuh"

template cudaError_t pkv::decode::dispatch_nw_ns<64, false>(const pkv::decode::Plan &, int, bool, int *, cudaStream_t,
                                                        const pkv::decode::LaunchArgs *);
template cudaError_t pkv::decode::run_prefix<64, false>(const pkv::decode::LaunchArgs *, cudaStream_t);
