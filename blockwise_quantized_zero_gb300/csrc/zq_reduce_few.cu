// zq_reduce_few.cu -- launch unit for the quantized-reduce kernels built for
// three CTAs an SM, used by launches of at most kFewShards shards (the
// two-hop reduce's hops, the ring's hops, small shard counts). A separate
// unit so that it compiles in parallel with zq_reduce.cu.
#include "zq_reduce_launch.h"

namespace zq {

cudaError_t launch_reduce_few(const ReduceArgs &a, int fin, int fout, cudaStream_t st) {
  return go_r_io<3>(a, fin, fout, st);
}

cudaError_t launch_reduce_hop_few(const HopArgs &a, int fin, int fout, cudaStream_t st) {
  return go_r_io<3>(a, fin, fout, st);
}

unsigned take_reduce_few_device_error() { return take_unit_error_word(); }

}  // namespace zq
