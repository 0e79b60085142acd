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

// Status of a launch made through launch_kernel (its error is also consumed from the runtime).
inline int launched(cudaError_t e) {
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return HLA_ERR_CUDA;
    }
    return launch_status();
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

// ----------------------------------------------------------------------------- launch chains
// Programmatic dependent launch.  Inside a chain (the decode layer's main stream, or calls a
// caller brackets with hla_chain_begin / hla_chain_end) every kernel after the chain's first is
// launched with programmatic stream serialisation: it may start while its predecessor still
// runs, does the work that does not depend on the predecessor (e.g. loading static weights or
// its own state), then waits (pdl_wait) until the predecessor has completed and its writes are
// visible.  Each kernel lets its successor start (pdl_trigger) only after its own wait, so when a
// kernel starts, every kernel before its immediate predecessor has completed: its pre-wait
// reads may touch anything the immediate predecessor does not write.  Every kernel of the
// library keeps to that, so any sequence of library kernels can form a chain.  Outside a chain
// every launch is plain and pdl_wait is a no-op.
//
// A PdlChain object opens a chain on a stream for its lifetime.  Inside a chain already open on
// the same stream it continues that chain (its first kernel follows the outer chain's last);
// otherwise its first kernel is launched plain, after whatever the caller queued before.
struct PdlChain {
    PdlChain(cudaStream_t st, bool on);
    ~PdlChain();
    bool prev_on, prev_started;
    cudaStream_t prev_st;
};
bool pdl_default(int M);             // do multi-kernel entry points chain their kernels at M tokens?
bool pdl_for(cudaStream_t st);       // launch with programmatic serialisation on this stream?
void pdl_launched(cudaStream_t st);  // a kernel was launched on st (the chain has started)

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_for(st) ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    if (e == cudaSuccess) pdl_launched(st);
    return e;
}

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

// ----------------------------------------------------------------------------- async copies

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Wait until the phase with the given parity completes, for at most limit_ns of %globaltimer.
// Returns false (after writing HLA_ERR_DEVICE_TIMEOUT to *status) if it has not by then.
__device__ __forceinline__ bool mbar_wait_for(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                              int *status) {
    const uint32_t a = smem_u32(bar);
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
        if ((i & 63) == 0) {  // the clock is read every 64 polls
            const uint64_t t = global_ns();
            if (i == 0) t0 = t;
            else if (t - t0 > limit_ns) break;
        }
    }
    atomicExch(status, HLA_ERR_DEVICE_TIMEOUT);
    return false;
}

// Per-thread asynchronous copies into shared memory (16 bytes through L2 only, or 4 bytes), in
// commit groups; wait_group<N> returns once at most N of this thread's groups are still pending.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from global memory
// into this CTA's shared memory, completing on the mbarrier's transaction count.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
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

// Wait for the stream predecessor of a programmatically launched kernel (no-op otherwise), then
// let this kernel's own successor start.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_trigger() {
    pdl_wait();
    pdl_trigger();
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }
__device__ __forceinline__ float sigmoid_f(float z) { return 1.0f / (1.0f + __expf(-z)); }

}  // namespace hla
