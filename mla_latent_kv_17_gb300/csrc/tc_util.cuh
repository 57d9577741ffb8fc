// Helpers shared by the tensor-core kernels around the decode (absorption, projection,
// prefill): bounded mbarrier waits, TMA tile stores, bf16 packing, tensor-map encoding and
// programmatic dependent launches.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sm103_ptx.cuh"

namespace mla {
namespace {

constexpr long long kWaitCycles = 4000000000LL;  // about two seconds

// Waits for phase `parity` of an mbarrier for at most kWaitCycles.  With an abort flag (a
// shared-memory int of the CTA) a wait also gives up once another wait of the CTA has, and
// a wait that runs out sets it.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, int *abort_flag = nullptr) {
    const long long t0 = (long long)ptx::clock64_now();
    for (uint32_t i = 0;; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u) {
            if (abort_flag && *reinterpret_cast<volatile int *>(abort_flag)) return false;
            if ((long long)ptx::clock64_now() - t0 > kWaitCycles) {
                if (abort_flag) *reinterpret_cast<volatile int *>(abort_flag) = 1;
                return false;
            }
        }
    }
}
// The same with the first probe inline, for an issuing thread whose barriers have mostly
// completed already (one try_wait then, no call and no clock read).
__device__ __forceinline__ bool wait_quick(uint32_t bar, uint32_t parity, int *abort_flag) {
    return ptx::mbar_try_wait(bar, parity) || wait_bounded(bar, parity, abort_flag);
}

// Gives copies or MMAs still in flight a bounded time to land before the CTA leaves.
__device__ __forceinline__ void drain_pause() {
    const long long t0 = (long long)ptx::clock64_now();
    while ((long long)ptx::clock64_now() - t0 < 20000000LL) {
    }
}

// Tile store shared -> global through a 3-D tensor map (bulk group), and the wait for it.
__device__ __forceinline__ void tma_store_3d(const void *tmap, uint32_t src, int32_t x, int32_t y, int32_t z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until the committed bulk stores have completed (written to global memory).
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ uint16_t bf16_bits(float f) {
    __nv_bfloat16 v = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&v);
}
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// Tensor of rank 2 or 3 (d[0] innermost; byte strides s[0 .. rank - 2]) with boxes b, 128-B
// swizzle; elements outside the tensor read as zero and are not written by stores.
inline bool tmap_tiled(CUtensorMap *m, CUtensorMapDataType dtype, const void *p, int rank, const uint64_t *d,
                       const uint64_t *s, const uint32_t *b) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc || rank < 2 || rank > 3) return false;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3], estr[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        dims[i] = d[i];
        box[i] = b[i];
    }
    for (int i = 0; i + 1 < rank; ++i) strides[i] = s[i];
    return enc(m, dtype, (cuuint32_t)rank, const_cast<void *>(p), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch with programmatic stream serialization: the kernel may start while the previous
// kernel of the stream runs, and waits for it in griddepcontrol.wait.
template <typename K, typename... Args>
cudaError_t launch_pdl(K kernel, int grid, int threads, uint32_t smem, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace
}  // namespace mla
