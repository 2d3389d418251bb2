// decode_inst_d64_fp8.cu -- compiles the decode kernels for head_dim 64 with a FP8 E4M3 pool.
#include "decode_kernels.cuh"

template cudaError_t pkv::decode::dispatch_nw_ns<64, true>(const pkv::decode::Plan &, int, bool, int *, cudaStream_t,
                                                        const pkv::decode::LaunchArgs *);
template cudaError_t pkv::decode::run_prefix<64, true>(const pkv::decode::LaunchArgs *, cudaStream_t);
