// Kernel launchers shared between the translation units of libmla_decode.
#pragma once
#include <cuda_runtime.h>

#include "common.cuh"

namespace mla {

cudaError_t launch_decode_simt(const DecodeArgs &a, int num_units, cudaStream_t stream);

}  // namespace mla
