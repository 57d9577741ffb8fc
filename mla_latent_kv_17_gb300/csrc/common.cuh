// Device-side helpers shared by the decode kernels of libmla_decode.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_decode.h"
#include "plan.h"

namespace mla {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Everything a decode launch needs, passed by value.
struct DecodeArgs {
    const unsigned char *ws;      // workspace (plan, partials)
    int *status;                  // device status word inside the workspace
    const uint16_t *q_nope;       // bf16 [B][H][512]
    const uint16_t *q_rope;       // bf16 [B][H][64]
    const unsigned char *cache;   // bf16 [P][64][576] or fp8 records [P][64][656]
    int64_t num_pages;
    const int32_t *block_table;   // [B][max_pages]
    int max_pages;
    const int32_t *seq_lens;      // [B]
    const int32_t *indices;       // [B][topk] or null
    int topk;
    int B, H;
    float scale_log2;             // softmax_scale * log2(e)
    float *out;                   // [B][H][512]
    float *lse;                   // [B][H]
    int kv_fp8;
    size_t ws_bytes;
    long long wait_cycles;        // iteration limit of every pipeline wait, in SM clock cycles
    int stall_test;               // nonzero: the MMA issuer first waits on a barrier nothing completes
};

// Default limit of a pipeline wait: about two seconds of SM clock.  Nothing in a healthy run
// waits anywhere near this long; a wait that does records MLA_ERR_TIMEOUT and the kernel
// winds down instead of spinning forever.
constexpr long long kDefaultWaitCycles = 4000000000LL;

// True when the workspace holds a plan built for this call (same B, H, topk) that fits in
// ws_bytes.  Otherwise the caller's kernel records MLA_ERR_WORKSPACE and does nothing.
__device__ __forceinline__ bool plan_matches(const DecodeArgs &a) {
    const PlanHeader *hd = reinterpret_cast<const PlanHeader *>(a.ws);
    if (hd->magic != kPlanMagic || hd->B != a.B || hd->H != a.H || hd->topk != a.topk ||
        hd->num_units < 1 || ws_layout(hd->B, hd->H, hd->num_units).total > a.ws_bytes)
        return false;
    return true;
}

// Programmatic dependent launch: a kernel launched with programmatic stream serialization
// may start while the previous kernel of the stream still runs; grid_dep_wait() returns once
// that kernel has completed and its memory is visible.  grid_dep_launch() lets the next
// kernel of the stream start launching (its blocks still wait in their grid_dep_wait()).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// Records the first device-side error; later ones are dropped.
__device__ __forceinline__ void record_error(int *status, int code) {
    atomicCAS(status, 0, code);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t v) {
    return __uint_as_float(((uint32_t)v) << 16);
}

}  // namespace mla
