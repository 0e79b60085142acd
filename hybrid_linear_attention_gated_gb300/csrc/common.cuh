// Shared host/device helpers for the sm_103a kernels behind include/hla.h.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "hla.h"

namespace hla {

// ----------------------------------------------------------------------------- host side

void set_variant(const char *fmt, ...);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

void count_launch();

// Status of the launch just made (and count it).  Every kernel launch in the library is
// followed by this call.
inline int launch_status() {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return HLA_ERR_CUDA;
    count_launch();
    return HLA_OK;
}

// Optional per-kernel event timing (see hla_trace_enable).
enum TraceKernel { kTraceNone = 0, kTraceKda, kTraceDense, kTraceMoeGateup, kTraceMoeDown };
void trace_before(int kernel, cudaStream_t st);
void trace_after(int kernel, cudaStream_t st);

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Number of SMs of the current device (cached per device).
int sm_count();

// Which side-stream L2 prefetches run when a prefetch stream is given: a bit mask from the
// tuning override HLA_PREFETCH_MASK, or -1 for the measured default policy.
// kPrefetchLayer: output-projection + router weights during the KDA step;
// kPrefetchSharedGateUp / kPrefetchSharedDown: the shared experts' weights during dispatch.
enum { kPrefetchLayer = 1, kPrefetchSharedGateUp = 2, kPrefetchSharedDown = 4 };
int prefetch_mask();

#define HLA_REQUIRE(cond, status) \
    do {                          \
        if (!(cond)) return (status); \
    } while (0)

// ----------------------------------------------------------------------------- device side

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return static_cast<uint32_t>(float_to_bf16_bits(lo)) |
           (static_cast<uint32_t>(float_to_bf16_bits(hi)) << 16);
}

// 128-bit load of STATIC WEIGHTS only: read-only (non-coherent) path, no L1
// allocation, 256-byte L2 sector promotion.  Activations and states written by
// earlier kernels must not use this load: the non-coherent path lets the compiler
// hoist it across synchronisation (the hazard the vLLM K3 audit found).
__device__ __forceinline__ uint4 ld_weight_v4(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Plain coherent 128-bit load for activations / states.
__device__ __forceinline__ uint4 ld_act_v4(const void *p) {
    return *reinterpret_cast<const uint4 *>(p);
}

// D(16x8 fp32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }
__device__ __forceinline__ float sigmoid_f(float z) { return 1.0f / (1.0f + __expf(-z)); }

}  // namespace hla
