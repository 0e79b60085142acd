// Skinny projections (split-K), the KDA input projection with its epilogue, RMSNorm,
// the sigmoid top-k router and the L2 prefetch kernel.
//
// "Hyper-optimizing Kimi K3 in vLLM", Part 1 sec. 1: projections at decode batch
// sizes are skinny products; the pages use small-matrix kernels at batch 1-2 and
// split-K (K divided over more CTAs, then reduced) above.  Here, below 32 tokens, every
// projection runs on the warp-level streaming tile (stream_mma.cuh; a warp item is 32
// weight rows x one K slice x a group of tokens) with the split count chosen from the
// problem size so that enough items exist to keep every SM streaming; from 32 tokens the
// tcgen05 path (tc_gemm.cu) takes over.  Split partials are summed in a fixed slice
// order, so results are deterministic.
#include <cooperative_groups.h>
#include <cstdlib>

#include "common.cuh"
#include "stream_mma.cuh"

namespace hla {

int dense_auto_split(int M, int N, int K);   // shared with the layer executor
int router_split(int M, int Hd, int E);

// HLA_DENSE_XITEM=0 keeps one item per warp on the streaming path (A/B runs).
bool dense_cross_item() {
    const char *env = getenv("HLA_DENSE_XITEM");
    return !(env && env[0] == '0');
}

// The streaming path's persistent cross-item kernel applies (else one item per warp).
bool dense_xi_applies(int N, int K, int split) {
    return N % 32 == 0 && min_slice_steps(K, split) >= 4 && dense_cross_item();
}

namespace {

constexpr int kDenseThreads = 128;  // 4 warps, one item per warp
// RMSNorm kernels: one thread-block cluster of kNormCluster CTAs per row, each CTA a contiguous
// eighth of the columns (same layout in both kernels => same sums)
constexpr int kNormCluster = 8;
constexpr int kNormThreads = 128;

struct DenseParams {
    const uint16_t *W;
    const uint16_t *x;
    int M, N, K;
    int split, ntg;
    float *part;               // [split][M][N] partials, or nullptr for the direct epilogue
    void *y;                   // direct epilogue output [M][N]
    int y_bf16;
    const uint16_t *residual;  // direct epilogue residual [M][N] or nullptr
};

// Warp item: 32 weight rows (two 16-row MMA tiles that share the token fragments) x one K
// slice x one group of 8*NT tokens.
template <int NT, int UNROLL>
__global__ void __launch_bounds__(kDenseThreads) dense_stream_kernel(const DenseParams p) {
    const int item = (blockIdx.x * kDenseThreads + threadIdx.x) >> 5;
    const int nrb = (p.N + 31) >> 5;
    if (item >= nrb * p.split * p.ntg) return;  // whole warp leaves together
    const int tg = item % p.ntg;
    const int rest = item / p.ntg;
    const int ks = rest % p.split;
    const int rb = rest / p.split;
    const int g = (threadIdx.x & 31) >> 2;
    const int rbase = rb * 32;

    const uint16_t *wg[2] = {p.W + (size_t)min(rbase + g, p.N - 1) * p.K,
                             p.W + (size_t)min(rbase + 16 + g, p.N - 1) * p.K};
    const uint16_t *wg8[2] = {p.W + (size_t)min(rbase + g + 8, p.N - 1) * p.K,
                              p.W + (size_t)min(rbase + 16 + g + 8, p.N - 1) * p.K};
    const uint16_t *xr[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
        xr[nt] = p.x + (size_t)min(tg * 8 * NT + nt * 8 + g, p.M - 1) * p.K;
    int kb, ke;
    k_slice(p.K, p.split, ks, kb, ke);

    float acc[2][NT][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[h][nt][e] = 0.f;
    // the weights are static: their first loads go out before waiting for the tokens
    warp_stream_tile<2, NT, UNROLL>(wg, wg8, xr, kb, ke, acc, [] { pdl_wait_trigger(); });

#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = rbase + 16 * h + acc_row(e);
                const int m = tg * 8 * NT + acc_tok(nt, e);
                if (r >= p.N || m >= p.M) continue;
                const size_t o = (size_t)m * p.N + r;
                if (p.part) {
                    p.part[(size_t)ks * p.M * p.N + o] = acc[h][nt][e];
                } else {
                    float v = acc[h][nt][e];
                    if (p.residual) v = __fadd_rn(v, bf16_bits_to_float(p.residual[o]));
                    if (p.y_bf16)
                        reinterpret_cast<uint16_t *>(p.y)[o] = float_to_bf16_bits(v);
                    else
                        reinterpret_cast<float *>(p.y)[o] = v;
                }
            }
        }
    }
}

// The same items on persistent warps whose load ring runs across item boundaries
// (stream_items): warp w of nwarps takes items w, w + nwarps, ...; the host picks nwarps so
// that every warp gets the same number of items.  Needs N a multiple of 32 (rows g + 8 of a
// tile never pass the last row) and every K slice at least 4 steps long.
struct DenseCtx {
    int rbase, ks, m0;  // first of the item's 32 rows, K slice, first token of its group
};

constexpr int dense_xi_min_blocks(int NT) { return NT == 1 ? 4 : 3; }

template <int NT>
__global__ void __launch_bounds__(kDenseThreads, dense_xi_min_blocks(NT))
    dense_stream_xi_kernel(const DenseParams p, int nwarps) {
    const int warp = (blockIdx.x * kDenseThreads + threadIdx.x) >> 5;
    if (warp >= nwarps) return;  // whole warp leaves together
    const int total = (p.N >> 5) * p.split * p.ntg;
    const int g = (threadIdx.x & 31) >> 2;
    auto decode = [&](int item) {
        ItemRows<2, NT, DenseCtx> r;
        const int tg = item % p.ntg;
        const int rest = item / p.ntg;
        const int ks = rest % p.split;
        const int rbase = rest / p.split * 32;
        int kb, ke;
        k_slice(p.K, p.split, ks, kb, ke);
        r.w[0] = p.W + (size_t)(rbase + g) * p.K + kb;
        r.w[1] = p.W + (size_t)(rbase + 16 + g) * p.K + kb;
        const int m0 = tg * 8 * NT;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) r.x[nt] = p.x + (size_t)min(m0 + nt * 8 + g, p.M - 1) * p.K + kb;
        r.n = (ke - kb) >> 5;
        r.ctx = DenseCtx{rbase, ks, m0};
        return r;
    };
    auto epilogue = [&](const DenseCtx &c, float (&acc)[2][NT][4]) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = c.rbase + 16 * h + acc_row(e);
                    const int m = c.m0 + acc_tok(nt, e);
                    if (m >= p.M) continue;
                    const size_t o = (size_t)m * p.N + r;
                    if (p.part) {
                        p.part[(size_t)c.ks * p.M * p.N + o] = acc[h][nt][e];
                    } else {
                        float v = acc[h][nt][e];
                        if (p.residual) v = __fadd_rn(v, bf16_bits_to_float(p.residual[o]));
                        if (p.y_bf16)
                            reinterpret_cast<uint16_t *>(p.y)[o] = float_to_bf16_bits(v);
                        else
                            reinterpret_cast<float *>(p.y)[o] = v;
                    }
                }
            }
        }
    };
    StridedClaims claims{warp, nwarps};
    // the weights are static: the first ring's weight loads go out before waiting for the tokens
    stream_items<2, NT, 4, DenseCtx>(claims, total, (size_t)8 * p.K, decode, epilogue,
                                     [] { pdl_wait_trigger(); });
}

// y = sum over slices in increasing order (+ residual)
__global__ void splitk_reduce_kernel(const float *__restrict__ part, int split, int M, int N,
                                     const uint16_t *__restrict__ residual, void *y, int y_bf16) {
    pdl_wait_trigger();
    const size_t total = (size_t)M * N;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        float v = part[i];
        for (int s = 1; s < split; ++s) v = __fadd_rn(v, part[(size_t)s * total + i]);
        if (residual) v = __fadd_rn(v, bf16_bits_to_float(residual[i]));
        if (y_bf16)
            reinterpret_cast<uint16_t *>(y)[i] = float_to_bf16_bits(v);
        else
            reinterpret_cast<float *>(y)[i] = v;
    }
}

// o-projection epilogue fused with the next RMSNorm: r = (sum of split partials) + residual,
// stored bf16, then xn = RMSNorm(r) * gamma.  Same thread layout and arithmetic order as
// splitk_reduce_kernel followed by rmsnorm_kernel, so the results are bit-identical to them.
// Thread t owns the 8-column groups t, t + blockDim.x, ...; when it owns at most one (N up to
// 8 * blockDim.x) its r and gamma stay in registers between the two passes, the residual load
// is issued before the slice loads and the gamma load before the block reduction.
__device__ __forceinline__ void residual_slices(const float *pr, size_t plane, int split, int i,
                                                bool has_res, const uint4 res, float (&v)[8]) {
    const float4 *p4 = reinterpret_cast<const float4 *>(pr + 8 * i);
    float4 lo = p4[0], hi = p4[1];
    // slices summed in increasing order per element (as splitk_reduce_kernel), loaded as
    // float4 pairs several slices ahead
#pragma unroll 4
    for (int sl = 1; sl < split; ++sl) {
        const float4 *q4 = reinterpret_cast<const float4 *>(pr + (size_t)sl * plane + 8 * i);
        const float4 a = q4[0], b = q4[1];
        lo.x = __fadd_rn(lo.x, a.x); lo.y = __fadd_rn(lo.y, a.y);
        lo.z = __fadd_rn(lo.z, a.z); lo.w = __fadd_rn(lo.w, a.w);
        hi.x = __fadd_rn(hi.x, b.x); hi.y = __fadd_rn(hi.y, b.y);
        hi.z = __fadd_rn(hi.z, b.z); hi.w = __fadd_rn(hi.w, b.w);
    }
    v[0] = lo.x; v[1] = lo.y; v[2] = lo.z; v[3] = lo.w;
    v[4] = hi.x; v[5] = hi.y; v[6] = hi.z; v[7] = hi.w;
    if (has_res) {
        const uint32_t rs[4] = {res.x, res.y, res.z, res.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[2 * j] = __fadd_rn(v[2 * j], bf16_lo(rs[j]));
            v[2 * j + 1] = __fadd_rn(v[2 * j + 1], bf16_hi(rs[j]));
        }
    }
}

__device__ __forceinline__ float sum_squares8(const uint4 w, float ss) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float a = bf16_lo(ws[j]), b = bf16_hi(ws[j]);
        ss = __fmaf_rn(a, a, ss);
        ss = __fmaf_rn(b, b, ss);
    }
    return ss;
}

__device__ __forceinline__ uint4 scale8(const uint4 w, const uint4 gg, float inv) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w}, gs[4] = {gg.x, gg.y, gg.z, gg.w};
    uint32_t out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        out[j] = pack_bf16x2(__fmul_rn(__fmul_rn(bf16_lo(ws[j]), inv), bf16_lo(gs[j])),
                             __fmul_rn(__fmul_rn(bf16_hi(ws[j]), inv), bf16_hi(gs[j])));
    return make_uint4(out[0], out[1], out[2], out[3]);
}

__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
    return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7]));
}

// Fixed-order sum over one row's cluster (every thread gets the result): a warp butterfly,
// the warps of a CTA in order, then the CTAs in rank order, read from their shared memory
// through the cluster (distributed shared memory).
__device__ float cluster_row_sum(float v, float *red) {
    namespace cg = cooperative_groups;
    constexpr int NW = kNormThreads / 32;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        float s = red[0];
        for (int i = 1; i < NW; ++i) s = __fadd_rn(s, red[i]);
        red[NW] = s;
    }
    cg::cluster_group cl = cg::this_cluster();
    cl.sync();
    float tot = *cl.map_shared_rank(&red[NW], 0);
    for (int r = 1; r < kNormCluster; ++r) tot = __fadd_rn(tot, *cl.map_shared_rank(&red[NW], r));
    cl.sync();  // every CTA has read the others' sums before any of them exits
    return tot;
}

// Columns of a row handled by CTA `rank` of its cluster: 8-column groups [g0, g1).
__device__ __forceinline__ void norm_range(int nv, int rank, int &g0, int &g1) {
    const int per = (nv + kNormCluster - 1) / kNormCluster;
    g0 = min(nv, rank * per);
    g1 = min(nv, g0 + per);
}

__global__ void __launch_bounds__(kNormThreads) __cluster_dims__(kNormCluster, 1, 1)
    residual_rmsnorm_kernel(const float *__restrict__ part, int split, int M, int N,
                            const uint16_t *__restrict__ residual,
                            const uint16_t *__restrict__ gamma, float eps, uint16_t *r,
                            uint16_t *xn) {
    __shared__ float red[kNormThreads / 32 + 1];
    const int m = blockIdx.x / kNormCluster;
    const size_t plane = (size_t)M * N;
    const float *pr = part + (size_t)m * N;
    uint4 *rr = reinterpret_cast<uint4 *>(r + (size_t)m * N);
    const uint4 *gr = reinterpret_cast<const uint4 *>(gamma);
    const uint4 *resr = residual ? reinterpret_cast<const uint4 *>(residual + (size_t)m * N) : nullptr;
    uint4 *yr = reinterpret_cast<uint4 *>(xn + (size_t)m * N);
    int g0, g1;
    norm_range(N / 8, blockIdx.x % kNormCluster, g0, g1);
    float ss = 0.f;
    if (g1 - g0 <= kNormThreads) {
        const int i = g0 + threadIdx.x;
        uint4 w = make_uint4(0, 0, 0, 0), gg = w, rw = w;
        // gamma and the residual do not come from the projection before this kernel: loaded
        // before waiting for it
        if (i < g1) {
            if (resr) rw = ld_act_v4(resr + i);
            gg = ld_act_v4(gr + i);
        }
        pdl_wait_trigger();
        if (i < g1) {
            float v[8];
            residual_slices(pr, plane, split, i, resr != nullptr, rw, v);
            w = pack8(v);
            rr[i] = w;
            ss = sum_squares8(w, ss);
        }
        const float tot = cluster_row_sum(ss, red);
        const float inv = 1.0f / sqrtf(tot / (float)N + eps);
        if (i < g1) yr[i] = scale8(w, gg, inv);
        return;
    }
    pdl_wait_trigger();
    for (int i = g0 + threadIdx.x; i < g1; i += kNormThreads) {
        uint4 rw = make_uint4(0, 0, 0, 0);
        if (resr) rw = ld_act_v4(resr + i);
        float v[8];
        residual_slices(pr, plane, split, i, resr != nullptr, rw, v);
        const uint4 w = pack8(v);
        rr[i] = w;
        ss = sum_squares8(w, ss);
    }
    const float tot = cluster_row_sum(ss, red);
    const float inv = 1.0f / sqrtf(tot / (float)N + eps);
    for (int i = g0 + threadIdx.x; i < g1; i += kNormThreads) yr[i] = scale8(rr[i], ld_act_v4(gr + i), inv);
}

// Fixed-order block sum of two values at once (one pair of barriers instead of two).
__device__ float2 block_sum2(float a, float b, float2 *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, o));
        b = __fadd_rn(b, __shfl_xor_sync(0xffffffffu, b, o));
    }
    const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[w] = make_float2(a, b);
    __syncthreads();
    float2 s = red[0];
    for (int i = 1; i < nw; ++i) {
        s.x = __fadd_rn(s.x, red[i].x);
        s.y = __fadd_rn(s.y, red[i].y);
    }
    return s;
}

// q/k/v/gate/beta epilogue: one CTA of d threads per (token, head).  Each thread sums the
// split slices of its q, k, v and gate columns (and the head's beta column, the same address
// for every thread) in increasing slice order, all five sums advancing together so that
// the loads of several slices are in flight at once.
__global__ void qkvg_epilogue_kernel(const float *__restrict__ part, int split, int M, int H, int d,
                                     uint16_t *q, uint16_t *k, uint16_t *v, float *alpha,
                                     float *beta) {
    __shared__ float2 red[32];
    pdl_wait_trigger();
    const int m = blockIdx.x / H, h = blockIdx.x % H, i = threadIdx.x;
    const int Nq = 4 * H * d + H;
    const size_t plane = (size_t)M * Nq;
    const int Hd_ = H * d;
    const float *row = part + (size_t)m * Nq + h * d + i;
    const float *rb = part + (size_t)m * Nq + 4 * Hd_ + h;
    float zq = row[0], zk = row[Hd_], zv = row[2 * Hd_], zg = row[3 * Hd_], zb = rb[0];
#pragma unroll 4
    for (int sl = 1; sl < split; ++sl) {
        const float *r = row + (size_t)sl * plane;
        const float a = r[0], b = r[Hd_], c = r[2 * Hd_], e = r[3 * Hd_], f = rb[(size_t)sl * plane];
        zq = __fadd_rn(zq, a);
        zk = __fadd_rn(zk, b);
        zv = __fadd_rn(zv, c);
        zg = __fadd_rn(zg, e);
        zb = __fadd_rn(zb, f);
    }
    const float2 ss = block_sum2(zq * zq, zk * zk, red);
    const size_t o = ((size_t)m * H + h) * d + i;
    q[o] = float_to_bf16_bits(ss.x > 0.f ? zq / sqrtf(ss.x) : 0.f);
    k[o] = float_to_bf16_bits(ss.y > 0.f ? zk / sqrtf(ss.y) : 0.f);
    v[o] = float_to_bf16_bits(zv);
    alpha[o] = 1.0f / (1.0f + expf(zg));  // exp(-softplus(g)) = 1 / (1 + e^g)
    if (i == 0) beta[(size_t)m * H + h] = 1.0f / (1.0f + expf(-zb));
}

// RMSNorm of bf16 rows, one cluster per row; thread layout and arithmetic order as in
// residual_rmsnorm_kernel's second half (x kept in registers when a thread owns one group).
__global__ void __launch_bounds__(kNormThreads) __cluster_dims__(kNormCluster, 1, 1)
    rmsnorm_kernel(int Hd, const uint16_t *__restrict__ x, const uint16_t *__restrict__ gamma,
                   float eps, uint16_t *y) {
    __shared__ float red[kNormThreads / 32 + 1];
    const int m = blockIdx.x / kNormCluster;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)m * Hd);
    const uint4 *gr = reinterpret_cast<const uint4 *>(gamma);
    uint4 *yr = reinterpret_cast<uint4 *>(y + (size_t)m * Hd);
    int g0, g1;
    norm_range(Hd / 8, blockIdx.x % kNormCluster, g0, g1);
    float ss = 0.f;
    if (g1 - g0 <= kNormThreads) {
        const int i = g0 + threadIdx.x;
        uint4 w = make_uint4(0, 0, 0, 0), gg = w;
        if (i < g1) gg = ld_act_v4(gr + i);  // static: before the wait
        pdl_wait_trigger();
        if (i < g1) {
            w = ld_act_v4(xr + i);
            ss = sum_squares8(w, ss);
        }
        const float tot = cluster_row_sum(ss, red);
        const float inv = 1.0f / sqrtf(tot / (float)Hd + eps);
        if (i < g1) yr[i] = scale8(w, gg, inv);
        return;
    }
    pdl_wait_trigger();
    for (int i = g0 + threadIdx.x; i < g1; i += kNormThreads) ss = sum_squares8(ld_act_v4(xr + i), ss);
    const float tot = cluster_row_sum(ss, red);
    const float inv = 1.0f / sqrtf(tot / (float)Hd + eps);
    for (int i = g0 + threadIdx.x; i < g1; i += kNormThreads)
        yr[i] = scale8(ld_act_v4(xr + i), ld_act_v4(gr + i), inv);
}

// One CTA per token.  The split partials of the fp32 logits are summed by all 1024 threads:
// each expert's slices are cut into nq = 1024 / E contiguous chunks, a thread sums one chunk
// in increasing slice order with eight loads in flight, and the chunk sums are added in
// chunk order (a fixed order, independent of the GPU).  Then every expert's thread finds its
// rank on the logits (ties to the lower index) in one pass; the k first are the top k, whose
// sigmoid scores one thread renormalises.
constexpr int kRouterThreads = 1024;

__global__ void __launch_bounds__(kRouterThreads)
    router_topk_kernel(const float *__restrict__ part, int split, int M, int E, int k,
                       int32_t *topk_idx, float *topk_w, float *logits_out) {
    __shared__ __align__(16) float lg[1024];
    __shared__ float chunk[kRouterThreads];
    __shared__ float sel[16];
    pdl_wait_trigger();
    const int m = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
    const size_t plane = (size_t)M * E;
    const int nq = kRouterThreads / E;  // E <= 1024
    {
        const int e = tid % E, q = tid / E;
        const int s0 = q * split / nq, s1 = (q + 1) * split / nq;
        if (q < nq && s1 > s0) {
            const float *src = part + (size_t)m * E + e;
            float s = src[(size_t)s0 * plane];
            for (int sb = s0 + 1; sb < s1; sb += 8) {
                float v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = sb + j < s1 ? src[(size_t)(sb + j) * plane] : 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (sb + j < s1) s = __fadd_rn(s, v[j]);
            }
            chunk[tid] = s;
        }
    }
    __syncthreads();
    if (tid < E) {
        float s = 0.f;
        bool first = true;
        for (int q = 0; q < nq; ++q) {
            if ((q + 1) * split / nq == q * split / nq) continue;  // empty chunk
            s = first ? chunk[q * E + tid] : __fadd_rn(s, chunk[q * E + tid]);
            first = false;
        }
        lg[tid] = s;
        if (logits_out) logits_out[(size_t)m * E + tid] = s;
    }
    __syncthreads();
    // Selection by rank: expert e's place in the order (logit descending, index ascending) is the
    // number of experts ahead of it; the k experts with rank < k are the top k, listed by rank.
    // Every thread reads the same logit at a time (a shared-memory broadcast).
    if (tid < E) {
        const float v = lg[tid];
        int rank = 0;
        const int E4 = E & ~3;
        for (int e = 0; e < E4; e += 4) {
            const float4 o = *reinterpret_cast<const float4 *>(&lg[e]);
            rank += (o.x > v || (o.x == v && e < tid)) + (o.y > v || (o.y == v && e + 1 < tid)) +
                    (o.z > v || (o.z == v && e + 2 < tid)) + (o.w > v || (o.w == v && e + 3 < tid));
        }
        for (int e = E4; e < E; ++e) rank += lg[e] > v || (lg[e] == v && e < tid);
        if (rank < k) {
            topk_idx[(size_t)m * k + rank] = tid;
            sel[rank] = v;
        }
    }
    __syncthreads();
    if (tid >= 32) return;
    if (lane == 0) {
        float sc[16], tot = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (j >= k) break;
            sc[j] = 1.0f / (1.0f + expf(-sel[j]));
            tot = __fadd_rn(tot, sc[j]);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (j >= k) break;
            topk_w[(size_t)m * k + j] = sc[j] / tot;
        }
    }
}

__global__ void l2_prefetch_kernel(const char *p, size_t bytes, uint32_t chunk) {
    // it reads only static weights, but in a launch chain a kernel must not let its successor
    // start before its own predecessor has completed
    pdl_wait_trigger();
    const size_t stride = (size_t)gridDim.x * blockDim.x * chunk;
    for (size_t off = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) * chunk; off < bytes;
         off += stride) {
        size_t sz = bytes - off < chunk ? bytes - off : chunk;
        sz &= ~(size_t)15;
        if (sz)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p + off), "r"((uint32_t)sz)
                         : "memory");
    }
}

template <int NT>
int launch_dense_nt(const DenseParams &p, cudaStream_t st) {
    const long items = (long)((p.N + 31) / 32) * p.split * p.ntg;
    cudaError_t e;
    trace_before(kTraceDense, st);
    if (dense_xi_applies(p.N, p.K, p.split)) {
        // as many warps as keep every warp at the same item count within the resident set
        static int resident[2] = {0, 0};
        int &res = resident[NT - 1];
        if (!res) {
            int per_sm = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dense_stream_xi_kernel<NT>,
                                                              kDenseThreads, 0) != cudaSuccess ||
                per_sm < 1)
                per_sm = 1;
            res = per_sm * sm_count() * (kDenseThreads / 32);
        }
        const long per_warp = (items + res - 1) / res;
        const long nwarps = (items + per_warp - 1) / per_warp;
        const long blocks = (nwarps * 32 + kDenseThreads - 1) / kDenseThreads;
        e = launch_kernel(dense_stream_xi_kernel<NT>, dim3((unsigned)blocks), dim3(kDenseThreads), 0, st,
                          p, (int)nwarps);
    } else {
        const long blocks = (items * 32 + kDenseThreads - 1) / kDenseThreads;
        e = launch_kernel(dense_stream_kernel<NT, 4>, dim3((unsigned)blocks), dim3(kDenseThreads), 0, st, p);
    }
    trace_after(kTraceDense, st);
    return launched(e);
}

}  // namespace

bool dense_tc_enabled(int M);
int dense_tc_split(int M, int N, int K);
int dense_tc_tile(int M);
int run_dense_tc(int M, int N, int K, const hla_bf16 *x, const hla_bf16 *W, int split, float *part,
                 void *y, int y_bf16, const hla_bf16 *residual, cudaStream_t st);

// Tokens per tile: 8 or 16 on the mma.sync streaming path, the MMA N (32..256) on the
// tensor-core path used from 32 tokens up.
int dense_tokens_per_tile(int M) {
    if (dense_tc_enabled(M)) return dense_tc_tile(M);
    return M <= 8 ? 8 : 16;
}

// Split so that (32-row blocks x token groups x split) gives about 24 warp items per SM,
// with at least 4 K steps (128 K values) per item and no empty slice.
int dense_auto_split(int M, int N, int K) {
    const char *env = getenv("HLA_DENSE_SPLIT");
    const long nrb = (N + 31) / 32;
    const long ntg = (M + dense_tokens_per_tile(M) - 1) / dense_tokens_per_tile(M);
    const long base = nrb * ntg;
    const long maxs = K / 128 > 0 ? K / 128 : 1;
    if (!env && dense_tc_enabled(M)) return dense_tc_split(M, N, K);
    long s = env ? atol(env) : (24L * sm_count() + base - 1) / base;
    if (s < 1) s = 1;
    if (s > maxs) s = maxs;
    if (s > 64) s = 64;
    // fewest slices of the same length: no slice left empty (128 K steps in 17 slices of 8
    // would leave the last one with nothing to stream)
    const long steps = K / 32, per = (steps + s - 1) / s;
    return (int)((steps + per - 1) / per);
}

// HLA_ROUTER_SPLIT overrides the router's K split (A/B runs); the default is the projection rule.
int router_split(int M, int Hd, int E) {
    const char *env = getenv("HLA_ROUTER_SPLIT");
    if (env) {
        const int v = atoi(env);
        if (v >= 1 && v <= Hd / 128) return v;
    }
    return dense_auto_split(M, E, Hd);
}

// Run x W^T with the streaming tile.  part != nullptr -> fp32 partials [split][M][N].
int run_dense(int M, int N, int K, const hla_bf16 *x, const hla_bf16 *W, int split, float *part,
              void *y, int y_bf16, const hla_bf16 *residual, cudaStream_t st) {
    if (dense_tc_enabled(M))
        return run_dense_tc(M, N, K, x, W, split, part, y, y_bf16, residual, st);
    DenseParams p;
    p.W = W; p.x = x; p.M = M; p.N = N; p.K = K; p.split = split;
    const int tt = dense_tokens_per_tile(M);
    p.ntg = (M + tt - 1) / tt;
    p.part = part; p.y = y; p.y_bf16 = y_bf16; p.residual = residual;
    return tt == 8 ? launch_dense_nt<1>(p, st) : launch_dense_nt<2>(p, st);
}

int run_splitk_reduce(const float *part, int split, int M, int N, const hla_bf16 *residual, void *y,
                      int y_bf16, cudaStream_t st) {
    const size_t total = (size_t)M * N;
    const int threads = 256;
    long blocks = (long)((total + threads - 1) / threads);
    if (blocks > 8L * sm_count()) blocks = 8L * sm_count();
    return launched(launch_kernel(splitk_reduce_kernel, dim3((unsigned)blocks), dim3(threads), 0, st,
                                  part, split, M, N, reinterpret_cast<const uint16_t *>(residual), y, y_bf16));
}

int run_rmsnorm(int M, int Hd, const hla_bf16 *x, const hla_bf16 *gamma, float eps, hla_bf16 *y,
                cudaStream_t st) {
    return launched(launch_kernel(rmsnorm_kernel, dim3((unsigned)M * kNormCluster), dim3(kNormThreads), 0,
                                  st, Hd, reinterpret_cast<const uint16_t *>(x),
                                  reinterpret_cast<const uint16_t *>(gamma), eps, reinterpret_cast<uint16_t *>(y)));
}

int run_l2_prefetch(const void *ptr, size_t bytes, cudaStream_t st) {
    if (bytes < 16) return HLA_OK;
    const uint32_t chunk = 16384;
    long threads = (long)((bytes + chunk - 1) / chunk);
    int blocks = (int)((threads + 127) / 128);
    if (blocks > sm_count()) blocks = sm_count();
    return launched(launch_kernel(l2_prefetch_kernel, dim3(blocks), dim3(128), 0, st,
                                  reinterpret_cast<const char *>(ptr), bytes, chunk));
}

int run_qkvg(int M, int Hd, int H, int d, const hla_bf16 *x, const hla_bf16 *W, hla_bf16 *q,
             hla_bf16 *k, hla_bf16 *v, float *alpha, float *beta, int split, float *part,
             cudaStream_t st) {
    const int Nq = 4 * H * d + H;
    int s = run_dense(M, Nq, Hd, x, W, split, part, nullptr, 0, nullptr, st);
    if (s != HLA_OK) return s;
    return launched(launch_kernel(qkvg_epilogue_kernel, dim3(M * H), dim3(d), 0, st, (const float *)part,
                                  split, M, H, d, reinterpret_cast<uint16_t *>(q), reinterpret_cast<uint16_t *>(k),
                                  reinterpret_cast<uint16_t *>(v), alpha, beta));
}

int run_router(int M, int Hd, int E, int k, const hla_bf16 *x, const hla_bf16 *W_r, int32_t *idx,
               float *w, float *logits, float *part, cudaStream_t st) {
    const int split = router_split(M, Hd, E);
    int s = run_dense(M, E, Hd, x, W_r, split, part, nullptr, 0, nullptr, st);
    if (s != HLA_OK) return s;
    return launched(launch_kernel(router_topk_kernel, dim3(M), dim3(kRouterThreads), 0, st, (const float *)part,
                                  split, M, E, k, idx, w, logits));
}

}  // namespace hla

using namespace hla;

static int resolve_split(int M, int N, int K, int split) {
    return split > 0 ? (split > K / 32 ? K / 32 : split) : dense_auto_split(M, N, K);
}

extern "C" size_t skinny_proj_splitk_workspace_size(int M, int N, int K, int split) {
    if (M < 1 || N < 1 || K < 32) return 0;
    const int s = resolve_split(M, N, K, split);
    return s > 1 ? (size_t)s * M * N * sizeof(float) : 0;
}

extern "C" int skinny_proj_splitk(int M, int N, int K, const hla_bf16 *x, const hla_bf16 *W,
                                  const hla_bf16 *residual, void *y, int y_dtype, int split,
                                  void *ws, size_t ws_bytes, hla_stream stream) {
    HLA_REQUIRE(M >= 1 && N >= 1 && K >= 32 && split >= 0, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(M <= 256 && K % 32 == 0, HLA_ERR_UNSUPPORTED);
    HLA_REQUIRE(x && W && y, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(y_dtype == HLA_F32 || y_dtype == HLA_BF16, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(aligned16(x) && aligned16(W) && aligned16(y) && (!residual || aligned16(residual)),
                HLA_ERR_MISALIGNED);
    const int s = resolve_split(M, N, K, split);
    const size_t need = skinny_proj_splitk_workspace_size(M, N, K, split);
    HLA_REQUIRE(need == 0 || (ws && ws_bytes >= need), HLA_ERR_WORKSPACE);
    HLA_REQUIRE(need == 0 || aligned16(ws), HLA_ERR_MISALIGNED);
    cudaStream_t st = (cudaStream_t)stream;
    set_variant("skinny_proj<tt%d,%ssplit%d>", dense_tokens_per_tile(M),
                !dense_tc_enabled(M) && dense_xi_applies(N, K, s) ? "xi," : "", s);
    const PdlChain chain(st, pdl_default(M));  // the projection and its split reduction
    if (s == 1) return run_dense(M, N, K, x, W, 1, nullptr, y, y_dtype == HLA_BF16, residual, st);
    int r = run_dense(M, N, K, x, W, s, reinterpret_cast<float *>(ws), nullptr, 0, nullptr, st);
    if (r != HLA_OK) return r;
    return run_splitk_reduce(reinterpret_cast<float *>(ws), s, M, N, residual, y, y_dtype == HLA_BF16, st);
}

extern "C" size_t kda_qkvg_proj_workspace_size(int M, int Hd, int H, int dk, int dv, int split) {
    if (M < 1 || Hd < 32 || H < 1 || dk < 1 || dv != dk) return 0;
    const int Nq = 4 * H * dk + H;
    const int s = resolve_split(M, Nq, Hd, split);
    return (size_t)s * M * Nq * sizeof(float);
}

extern "C" int kda_qkvg_proj(int M, int Hd, int H, int dk, int dv, const hla_bf16 *x,
                             const hla_bf16 *W, hla_bf16 *q, hla_bf16 *k, hla_bf16 *v, float *alpha,
                             float *beta, int split, void *ws, size_t ws_bytes, hla_stream stream) {
    HLA_REQUIRE(M >= 1 && Hd >= 32 && H >= 1 && split >= 0, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(dk == dv && (dk == 64 || dk == 128) && M <= 256 && Hd % 32 == 0, HLA_ERR_UNSUPPORTED);
    HLA_REQUIRE(x && W && q && k && v && alpha && beta, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(aligned16(x) && aligned16(W) && aligned16(q) && aligned16(k) && aligned16(v) &&
                    aligned16(alpha) && aligned16(beta),
                HLA_ERR_MISALIGNED);
    const size_t need = kda_qkvg_proj_workspace_size(M, Hd, H, dk, dv, split);
    HLA_REQUIRE(ws && ws_bytes >= need, HLA_ERR_WORKSPACE);
    HLA_REQUIRE(aligned16(ws), HLA_ERR_MISALIGNED);
    const int s = resolve_split(M, 4 * H * dk + H, Hd, split);
    set_variant("qkvg_proj<tt%d,split%d>", dense_tokens_per_tile(M), s);
    const PdlChain chain((cudaStream_t)stream, pdl_default(M));  // the projection and its epilogue
    return run_qkvg(M, Hd, H, dk, x, W, q, k, v, alpha, beta, s, reinterpret_cast<float *>(ws),
                    (cudaStream_t)stream);
}

extern "C" int hla_rmsnorm(int M, int Hd, const hla_bf16 *x, const hla_bf16 *gamma, float eps,
                           hla_bf16 *y, hla_stream stream) {
    HLA_REQUIRE(M >= 1 && Hd >= 8 && eps >= 0.f, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(Hd % 8 == 0 && M <= 65535, HLA_ERR_UNSUPPORTED);
    HLA_REQUIRE(x && gamma && y, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(aligned16(x) && aligned16(gamma) && aligned16(y), HLA_ERR_MISALIGNED);
    set_variant("rmsnorm");
    return run_rmsnorm(M, Hd, x, gamma, eps, y, (cudaStream_t)stream);
}

extern "C" size_t moe_route_topk_workspace_size(int M, int Hd, int E) {
    if (M < 1 || Hd < 32 || E < 1) return 0;
    return (size_t)router_split(M, Hd, E) * M * E * sizeof(float);
}

extern "C" int moe_route_topk(int M, int Hd, int E, int k, const hla_bf16 *x, const hla_bf16 *W_r,
                              int32_t *topk_idx, float *topk_w, float *logits, void *ws,
                              size_t ws_bytes, hla_stream stream) {
    HLA_REQUIRE(M >= 1 && Hd >= 32 && E >= 1 && k >= 1, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(k <= 16 && k <= E && E <= 1024 && Hd % 32 == 0 && M <= 65535, HLA_ERR_UNSUPPORTED);
    HLA_REQUIRE(x && W_r && topk_idx && topk_w, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(aligned16(x) && aligned16(W_r) && aligned16(topk_idx) && aligned16(topk_w) &&
                    (!logits || aligned16(logits)),
                HLA_ERR_MISALIGNED);
    const size_t need = moe_route_topk_workspace_size(M, Hd, E);
    HLA_REQUIRE(ws && ws_bytes >= need, HLA_ERR_WORKSPACE);
    HLA_REQUIRE(aligned16(ws), HLA_ERR_MISALIGNED);
    set_variant("router<split%d>", router_split(M, Hd, E));
    const PdlChain chain((cudaStream_t)stream, pdl_default(M));  // the router GEMV and its top-k
    return run_router(M, Hd, E, k, x, W_r, topk_idx, topk_w, logits, reinterpret_cast<float *>(ws),
                      (cudaStream_t)stream);
}

extern "C" int hla_l2_prefetch(const void *ptr, size_t bytes, hla_stream stream) {
    HLA_REQUIRE(ptr || bytes == 0, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(bytes == 0 || aligned16(ptr), HLA_ERR_MISALIGNED);
    set_variant("l2_prefetch");
    return run_l2_prefetch(ptr, bytes, (cudaStream_t)stream);
}

// Default split of the projection fused with residual + RMSNorm: each thread of that epilogue
// sums every slice of its columns, so on the streaming path the split is capped at 8 (at batch 1
// and 8 with N = 7168, K = 4096: 17.6 / 17.9 us at split 8 against 19.9 / 20.5 us at the
// generic choice, then 17).
static int residual_norm_split(int M, int N, int K, int split) {
    const int s = resolve_split(M, N, K, split);
    return (split == 0 && !dense_tc_enabled(M) && s > 8) ? 8 : s;
}

extern "C" size_t skinny_proj_residual_rmsnorm_workspace_size(int M, int N, int K, int split) {
    if (M < 1 || N < 8 || K < 32) return 0;
    return (size_t)residual_norm_split(M, N, K, split) * M * N * sizeof(float);
}

extern "C" int skinny_proj_residual_rmsnorm(int M, int N, int K, const hla_bf16 *x,
                                            const hla_bf16 *W, const hla_bf16 *residual,
                                            const hla_bf16 *gamma, float eps, hla_bf16 *r,
                                            hla_bf16 *xn, int split, void *ws, size_t ws_bytes,
                                            hla_stream stream) {
    HLA_REQUIRE(M >= 1 && N >= 8 && K >= 32 && split >= 0 && eps >= 0.f, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(M <= 256 && K % 32 == 0 && N % 8 == 0, HLA_ERR_UNSUPPORTED);
    HLA_REQUIRE(x && W && gamma && r && xn, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(aligned16(x) && aligned16(W) && aligned16(gamma) && aligned16(r) && aligned16(xn) &&
                    (!residual || aligned16(residual)),
                HLA_ERR_MISALIGNED);
    const size_t need = skinny_proj_residual_rmsnorm_workspace_size(M, N, K, split);
    HLA_REQUIRE(ws && ws_bytes >= need, HLA_ERR_WORKSPACE);
    HLA_REQUIRE(aligned16(ws), HLA_ERR_MISALIGNED);
    const int s = residual_norm_split(M, N, K, split);
    cudaStream_t st = (cudaStream_t)stream;
    float *part = reinterpret_cast<float *>(ws);
    const PdlChain chain(st, pdl_default(M));  // the projection and its residual + RMSNorm epilogue
    int rc = run_dense(M, N, K, x, W, s, part, nullptr, 0, nullptr, st);
    if (rc != HLA_OK) return rc;
    const cudaError_t e = launch_kernel(
        residual_rmsnorm_kernel, dim3((unsigned)M * kNormCluster), dim3(kNormThreads), 0, st, (const float *)part, s,
        M, N, reinterpret_cast<const uint16_t *>(residual), reinterpret_cast<const uint16_t *>(gamma), eps,
        reinterpret_cast<uint16_t *>(r), reinterpret_cast<uint16_t *>(xn));
    set_variant("proj_residual_rmsnorm<tt%d,split%d>", dense_tokens_per_tile(M), s);
    return launched(e);
}
