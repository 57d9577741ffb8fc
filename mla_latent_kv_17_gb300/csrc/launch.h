// Kernel launchers shared between the translation units of libmla_decode.
#pragma once
#include <cuda_runtime.h>

#include "common.cuh"

namespace mla {

// Tensor-core kernel (bf16 cache dense or DSA-sparse when a.indices is set, or FP8 records
// when a.kv_fp8 is set): one cluster of two CTAs per work unit.
cudaError_t launch_decode_sm103(const DecodeArgs &a, int num_clusters, cudaStream_t stream);
// Clusters of that kernel that fit on the current device at once (0 if unknown).
int sm103_max_units();

}  // namespace mla
