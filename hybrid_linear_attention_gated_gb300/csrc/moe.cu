// Routed + shared SwiGLU experts at decode batch sizes.
//
// "Kimi K3: From Day-0 Availability to Optimized Inference": at low batch, moving
// expert weights through GPU memory is the limit.  "Hyper-optimizing Kimi K3 in
// vLLM", Part 1 sec. 3: routed experts plus a shared expert for every token;
// sec. 4: a side-stream kernel warms L2 with upcoming weights while a phase cannot
// use the memory bandwidth.
//
// Pipeline (all on device, no host round trip; sizes the host does not know -- the
// number of active experts -- are read by persistent kernels from the workspace, whose
// warps claim work items from a counter):
//   1. dispatch   : one CTA groups the M*k (token, slot) pairs by expert (counting
//                   sort, stable by pair index), lists the active experts (shared
//                   experts first) and prefix-sums their work items.
//   2. gate/up    : persistent warps stream 16 rows of W_gate[e] and W_up[e] over a
//                   K slice for up to 16 of expert e's tokens; SiLU(g)*u -> h (bf16),
//                   or fp32 partials when K is split (small M, to fill the GPU).
//   3. [reduce]   : h = SiLU(sum g) * (sum u) over the K slices, fixed order.
//   4. down       : persistent warps stream 32 rows of W_down[e] (two 16-row MMA tiles
//                   sharing the token fragments) for the tokens' h rows -> one fp32 row per
//                   (token, slot).
//   5. combine    : y[m] = sum_j w[m,j] * y[m,j] + sum_s y[m,k+s] (+ residual), fixed order.
// Each active expert's weights are read from HBM once per call; when an expert has
// more than 16 tokens, its token groups are adjacent work items that stream the same
// rows at the same time, so the repeats are served by L2.
// The shared experts are, by default, grouped work units 0..n_shared-1 of steps 2-4.  Two
// opt-in placements compute them instead as dense SwiGLU products into their output slots:
// on the tensor-core path before dispatch (HLA_SHARED_TC=1, past 16 tokens), or on the side
// stream concurrently with everything routed (HLA_SHARED_STREAM=1, moe_shared_side).
#include <cstdio>
#include <cstdlib>

#include "common.cuh"
#include "stream_mma.cuh"

namespace hla {

int run_l2_prefetch(const void *ptr, size_t bytes, cudaStream_t st);
int dense_tc_split(int M, int N, int K);
int dense_auto_split(int M, int N, int K);
int run_dense(int M, int N, int K, const hla_bf16 *x, const hla_bf16 *W, int split, float *part,
              void *y, int y_bf16, const hla_bf16 *residual, cudaStream_t st);
int run_dense_tc(int M, int N, int K, const hla_bf16 *x, const hla_bf16 *W, int split, float *part,
                 void *y, int y_bf16, const hla_bf16 *residual, cudaStream_t st);

namespace {

constexpr int kMoeThreads = 128;
constexpr int kDispatchThreads = 1024;

struct MoeLayout {
    int M, Hd, I, E, k, nsh, P, U_max, KS, KSD, TT;
    bool shared_tc;      // shared experts on the tensor-core path instead of grouped work units
    int s_gu, s_dn;      // K slices of the shared experts' tensor-core products
    int d_gu, d_dn;      // K slices of the shared experts' products when they run on a side stream
    size_t off_meta, off_unit_expert, off_unit_off, off_item_gu, off_item_dn, off_pos_token,
        off_pos_slot, off_h, off_part_g, off_part_u, off_ypart, off_sh_g, off_sh_u, off_sh_d, total;
};

struct MoeArgs {
    int M, Hd, I, E, k, nsh, P, KS, KSD, TT;
    int nsh_units;  // shared experts run as grouped work units (0 when on the tensor-core path)
    const uint16_t *x;
    const int32_t *topk_idx;
    const float *topk_w;
    const uint16_t *W_gate, *W_up, *W_down, *Ws_gate, *Ws_up, *Ws_down;
    const uint16_t *residual;
    uint16_t *y;
    int *meta, *unit_expert, *unit_off, *item_gu, *item_dn, *pos_token, *pos_slot;
    uint16_t *h;
    float *part_g, *part_u, *ypart;
};

int moe_tokens_per_tile(int M) { return M <= 8 ? 8 : 16; }

// K splits of the expert products.  Two rules, the larger wins:
//  * enough work items: about 24 warp items per SM (units x row blocks x split);
//  * short items at small batch: with the 8-token tile (batch <= 8) a gate/up item is cut
//    to about 128 KB of weights and a down item to about 64 KB, so that the last items
//    claimed end soon after the others (at batch 8: 726 us with splits 4 / 2 against 775 us
//    unsplit; at batch 32 and 64 splitting measured no better or slower, the partials then
//    being large).
// HLA_MOE_SHALLOW=0 keeps the per-item gate/up kernel at 4 K steps of loads from 32 tokens too
// (A/B measurements); the cross-item kernels take their ring depth from moe_ring_depth.
bool moe_shallow_gateup() {
    const char *env = getenv("HLA_MOE_SHALLOW");
    return !(env && env[0] == '0');
}

// HLA_MOE_XITEM=0 keeps the expert kernels whose loads stop at item boundaries (A/B runs).
bool moe_cross_item() {
    const char *env = getenv("HLA_MOE_XITEM");
    return !(env && env[0] == '0');
}

int moe_items_split(int M, int k, int E, int nsh, long row_blocks, long cap) {
    long units = (long)M * k < E ? (long)M * k : E;
    units += nsh;
    const long items = units * row_blocks;
    long s = (24L * sm_count() + items - 1) / items;
    if (s < 1) s = 1;
    return (int)(s > cap ? cap : s);
}

int moe_bytes_split(int M, long item_bytes, long target, long cap) {
    if (M > 8) return 1;
    long s = (item_bytes + target - 1) / target;
    if (s < 1) s = 1;
    return (int)(s > cap ? cap : s);
}

int moe_down_split(int M, int Hd, int I, int E, int k, int nsh) {
    const char *env = getenv("HLA_MOE_DOWN_SPLIT");
    if (env) {
        const int v = atoi(env);
        if (v >= 1 && v <= 4) return v;
    }
    const int a = moe_items_split(M, k, E, nsh, (Hd + 31) / 32, 4);
    const int b = moe_bytes_split(M, 32L * I * 2, 64L * 1024, 4);  // 32 rows of W_down
    return a > b ? a : b;
}

int moe_gateup_split(int M, int Hd, int I, int E, int k, int nsh) {
    const char *env = getenv("HLA_MOE_SPLIT");
    if (env) {
        const int v = atoi(env);
        if (v >= 1 && v <= 16) return v;
    }
    const int a = moe_items_split(M, k, E, nsh, (I + 15) / 16, 8);
    const int b = moe_bytes_split(M, 2L * 16 * Hd * 2, 128L * 1024, 8);  // 16 rows of W_gate and W_up
    return a > b ? a : b;
}

MoeLayout moe_layout(int M, int Hd, int I, int E, int k, int nsh) {
    MoeLayout L;
    L.M = M; L.Hd = Hd; L.I = I; L.E = E; L.k = k; L.nsh = nsh;
    L.P = M * (k + nsh);
    L.U_max = E + nsh;
    L.KS = moe_gateup_split(M, Hd, I, E, k, nsh);
    L.KSD = moe_down_split(M, Hd, I, E, k, nsh);
    L.TT = moe_tokens_per_tile(M);
    // Optional (HLA_SHARED_TC=1): past 16 tokens run each shared expert as a dense SwiGLU
    // over all M tokens on the tensor-core path instead of as a grouped work unit.  Off by
    // default: in the decode layer at batch 64 the grouped unit with its gate/up weights
    // warmed in L2 measured 3146 us per layer against 3515 us for this path.
    const char *env = getenv("HLA_SHARED_TC");
    L.shared_tc = nsh > 0 && M > 16 && env && env[0] == '1';
    L.s_gu = L.shared_tc ? dense_tc_split(M, I, Hd) : 0;
    L.s_dn = L.shared_tc ? dense_tc_split(M, Hd, I) : 0;
    // The side-stream placement (moe_shared_side) can be chosen per call, so its partial
    // buffers are always part of the workspace when there are shared experts.
    L.d_gu = nsh > 0 ? dense_auto_split(M, I, Hd) : 0;
    L.d_dn = nsh > 0 ? dense_auto_split(M, Hd, I) : 0;
    const size_t sgu = (size_t)(L.s_gu > L.d_gu ? L.s_gu : L.d_gu);
    const size_t sdn = (size_t)(L.s_dn > L.d_dn ? L.s_dn : L.d_dn);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = round_up(o + bytes, 256);
        return at;
    };
    L.off_meta = take(16 * sizeof(int));
    L.off_unit_expert = take((size_t)L.U_max * sizeof(int));
    L.off_unit_off = take((size_t)(L.U_max + 1) * sizeof(int));
    L.off_item_gu = take((size_t)(L.U_max + 1) * sizeof(int));
    L.off_item_dn = take((size_t)(L.U_max + 1) * sizeof(int));
    L.off_pos_token = take((size_t)L.P * sizeof(int));
    L.off_pos_slot = take((size_t)L.P * sizeof(int));
    L.off_h = take((size_t)L.P * I * sizeof(uint16_t));
    L.off_part_g = take(L.KS > 1 ? (size_t)L.KS * L.P * I * sizeof(float) : 0);
    L.off_part_u = take(L.KS > 1 ? (size_t)L.KS * L.P * I * sizeof(float) : 0);
    L.off_ypart = take((size_t)L.KSD * L.P * Hd * sizeof(float));
    L.off_sh_g = take(sgu * M * I * sizeof(float));
    L.off_sh_u = take(sgu * M * I * sizeof(float));
    L.off_sh_d = take(sdn * M * Hd * sizeof(float));
    L.total = o;
    return L;
}

// Exclusive prefix sum over one value per thread of the block (a whole number of warps,
// at most 1024 threads).
__device__ int block_exclusive_scan(int v, int *warp_tot, int &total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    __syncthreads();
    if (lane == 31) warp_tot[w] = incl;
    __syncthreads();
    if (w == 0) {
        const int t = lane < nw ? warp_tot[lane] : 0;
        int s = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += n;
        }
        warp_tot[lane] = s - t;  // exclusive warp offsets
        if (lane == 31) warp_tot[32] = s;
    }
    __syncthreads();
    total = warp_tot[32];
    return warp_tot[w] + incl - v;
}

// One CTA of round_up(E + n_shared, 32) threads (thread e owns expert e's count and unit).
__global__ void __launch_bounds__(kDispatchThreads) moe_dispatch_kernel(const MoeArgs a) {
    __shared__ int cnt[1024], base[1024], run[1024], uid[1024];
    __shared__ int warp_tot[33];
    pdl_wait_trigger();
    const int tid = threadIdx.x;
    const int npairs = a.M * a.k;
    const int nrb_gu = (a.I + 15) / 16, nrb_dn = (a.Hd + 31) / 32;

    cnt[tid] = 0;
    run[tid] = 0;
    __syncthreads();
    for (int p = tid; p < npairs; p += blockDim.x) {
        const int e = a.topk_idx[p];
        if (e >= 0 && e < a.E) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    const int c = tid < a.E ? cnt[tid] : 0;
    int nvalid, nact;
    base[tid] = block_exclusive_scan(c, warp_tot, nvalid);
    uid[tid] = block_exclusive_scan(c > 0 ? 1 : 0, warp_tot, nact);
    __syncthreads();

    const int routed0 = a.nsh * a.M;  // shared experts' positions come first
    if (tid < 32) {
        // stable placement: pairs in increasing index order within each expert
        const unsigned lt = (1u << tid) - 1u;
        for (int c0 = 0; c0 < npairs; c0 += 32) {
            const int p = c0 + tid;
            const int e = p < npairs ? a.topk_idx[p] : -1;
            const bool valid = e >= 0 && e < a.E;
            const unsigned grp = __match_any_sync(0xffffffffu, valid ? e : -1 - tid);
            if (valid) {
                const int pos = routed0 + base[e] + run[e] + __popc(grp & lt);
                const int m = p / a.k, j = p % a.k;
                a.pos_token[pos] = m;
                a.pos_slot[pos] = m * (a.k + a.nsh) + j;
            }
            __syncwarp();
            if (valid && (grp & lt) == 0) run[e] += __popc(grp);
            __syncwarp();
        }
    }
    for (int i = tid; i < routed0; i += blockDim.x) {
        const int s = i / a.M, m = i % a.M;
        a.pos_token[i] = m;
        a.pos_slot[i] = m * (a.k + a.nsh) + a.k + s;
    }
    // unit tables: shared experts (when grouped) are units 0..nsh-1, routed experts follow by id
    if (tid < a.nsh_units) {
        a.unit_expert[tid] = a.E + tid;
        a.unit_off[tid] = tid * a.M;
    }
    if (tid < a.E && c > 0) {
        a.unit_expert[a.nsh_units + uid[tid]] = tid;
        a.unit_off[a.nsh_units + uid[tid]] = routed0 + base[tid];
    }
    const int U = a.nsh_units + nact;
    if (tid == 0) {
        a.unit_off[U] = routed0 + nvalid;
        a.meta[0] = U;
        a.meta[3] = 0;  // next gate/up work item to hand out
        a.meta[4] = 0;  // next down work item to hand out
    }
    __syncthreads();
    int ig = 0, id = 0;
    if (tid < U) {
        const int n = a.unit_off[tid + 1] - a.unit_off[tid];
        const int ntg = (n + a.TT - 1) / a.TT;
        ig = nrb_gu * a.KS * ntg;
        id = nrb_dn * ntg * a.KSD;
    }
    int tot_g, tot_d;
    const int og = block_exclusive_scan(ig, warp_tot, tot_g);
    const int od = block_exclusive_scan(id, warp_tot, tot_d);
    if (tid < U) {
        a.item_gu[tid] = og;
        a.item_dn[tid] = od;
    }
    if (tid == 0) {
        a.item_gu[U] = tot_g;
        a.item_dn[U] = tot_d;
        a.meta[1] = tot_g;
        a.meta[2] = tot_d;
    }
}

// Work items are handed out dynamically: lane 0 of a warp claims the next index from a
// counter the dispatch kernel reset, so warps that start late or run slow simply take fewer
// items (the result of an item does not depend on which warp computes it).
__device__ __forceinline__ int claim_item(int *counter) {
    int it = 0;
    if ((threadIdx.x & 31) == 0) it = atomicAdd(counter, 1);
    return __shfl_sync(0xffffffffu, it, 0);
}

// largest u in [0, U) with pref[u] <= it
__device__ __forceinline__ int find_unit(const int *pref, int U, int it) {
    int lo = 0, hi = U - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pref[mid] <= it) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <int NT, int UNROLL>
__global__ void __launch_bounds__(kMoeThreads) moe_gateup_kernel(const MoeArgs a) {
    pdl_wait_trigger();
    const int U = a.meta[0];
    const int total = a.item_gu[U];
    const int g = (threadIdx.x & 31) >> 2;
    for (int it = claim_item(&a.meta[3]); it < total; it = claim_item(&a.meta[3])) {
        const int u = find_unit(a.item_gu, U, it);
        const int local = it - a.item_gu[u];
        const int p0 = a.unit_off[u], p1 = a.unit_off[u + 1];
        const int ntg = (p1 - p0 + a.TT - 1) / a.TT;
        const int tg = local % ntg;
        const int rest = local / ntg;
        const int ks = rest % a.KS;
        const int rb = rest / a.KS;
        const int e = a.unit_expert[u];
        const size_t eoff = (size_t)(e < a.E ? e : e - a.E) * a.I * a.Hd;
        const uint16_t *Wg = (e < a.E ? a.W_gate : a.Ws_gate) + eoff;
        const uint16_t *Wu = (e < a.E ? a.W_up : a.Ws_up) + eoff;
        const int r0 = min(rb * 16 + g, a.I - 1), r1 = min(rb * 16 + g + 8, a.I - 1);
        const uint16_t *wg[2] = {Wg + (size_t)r0 * a.Hd, Wu + (size_t)r0 * a.Hd};
        const uint16_t *wg8[2] = {Wg + (size_t)r1 * a.Hd, Wu + (size_t)r1 * a.Hd};
        const int pt = p0 + tg * a.TT;
        const uint16_t *xr[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int p = pt + nt * 8 + g;
            xr[nt] = a.x + (size_t)a.pos_token[p < p1 ? p : pt] * a.Hd;
        }
        int kb, ke;
        k_slice(a.Hd, a.KS, ks, kb, ke);
        float acc[2][NT][4];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[m][nt][q] = 0.f;
        warp_stream_tile<2, NT, UNROLL>(wg, wg8, xr, kb, ke, acc);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int row = rb * 16 + acc_row(q);
                const int p = pt + acc_tok(nt, q);
                if (row >= a.I || p >= p1) continue;
                if (a.KS == 1) {
                    a.h[(size_t)p * a.I + row] =
                        float_to_bf16_bits(__fmul_rn(silu_f(acc[0][nt][q]), acc[1][nt][q]));
                } else {
                    const size_t o = ((size_t)ks * a.P + p) * a.I + row;
                    a.part_g[o] = acc[0][nt][q];
                    a.part_u[o] = acc[1][nt][q];
                }
            }
        }
    }
}

__global__ void moe_swiglu_reduce_kernel(const MoeArgs a) {
    pdl_wait_trigger();
    const int n = a.meta[0];
    const int used = a.unit_off[n];  // positions in use
    // positions of shared experts on the tensor-core path are not grouped units: skip them
    const size_t first = (size_t)(a.nsh - a.nsh_units) * a.M * a.I;
    const size_t total = (size_t)used * a.I, plane = (size_t)a.P * a.I;
    for (size_t i = first + blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        float g = a.part_g[i], u = a.part_u[i];
#pragma unroll 4
        for (int s = 1; s < a.KS; ++s) {
            g = __fadd_rn(g, a.part_g[s * plane + i]);
            u = __fadd_rn(u, a.part_u[s * plane + i]);
        }
        a.h[i] = float_to_bf16_bits(__fmul_rn(silu_f(g), u));
    }
}

template <int NT>
__global__ void __launch_bounds__(kMoeThreads) moe_down_kernel(const MoeArgs a) {
    pdl_wait_trigger();
    const int U = a.meta[0];
    const int total = a.item_dn[U];
    const int g = (threadIdx.x & 31) >> 2;
    for (int it = claim_item(&a.meta[4]); it < total; it = claim_item(&a.meta[4])) {
        const int u = find_unit(a.item_dn, U, it);
        const int local = it - a.item_dn[u];
        const int p0 = a.unit_off[u], p1 = a.unit_off[u + 1];
        const int ntg = (p1 - p0 + a.TT - 1) / a.TT;
        const int tg = local % ntg;
        const int ks = (local / ntg) % a.KSD;
        const int rb = local / ntg / a.KSD;  // a block of 32 rows: two 16-row MMA tiles share the tokens
        const int e = a.unit_expert[u];
        const uint16_t *Wd = (e < a.E ? a.W_down : a.Ws_down) +
                             (size_t)(e < a.E ? e : e - a.E) * a.Hd * a.I;
        const int rbase = rb * 32;
        const uint16_t *wg[2] = {Wd + (size_t)min(rbase + g, a.Hd - 1) * a.I,
                                 Wd + (size_t)min(rbase + 16 + g, a.Hd - 1) * a.I};
        const uint16_t *wg8[2] = {Wd + (size_t)min(rbase + g + 8, a.Hd - 1) * a.I,
                                  Wd + (size_t)min(rbase + 16 + g + 8, a.Hd - 1) * a.I};
        const int pt = p0 + tg * a.TT;
        const uint16_t *xr[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int p = pt + nt * 8 + g;
            xr[nt] = a.h + (size_t)(p < p1 ? p : pt) * a.I;
        }
        float acc[2][NT][4];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[h][nt][q] = 0.f;
        int kb, ke;
        k_slice(a.I, a.KSD, ks, kb, ke);
        warp_stream_tile<2, NT, 4>(wg, wg8, xr, kb, ke, acc);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int row = rbase + 16 * h + acc_row(q);
                    const int p = pt + acc_tok(nt, q);
                    if (row >= a.Hd || p >= p1) continue;
                    a.ypart[((size_t)ks * a.P + a.pos_slot[p]) * a.Hd + row] = acc[h][nt][q];
                }
            }
        }
    }
}

// Work-item claims for stream_items (stream_mma.cuh): lane 0 takes the next index from the
// counter a few K steps before the item's first loads are due; the index is broadcast to the
// warp when the item is decoded, so the atomic's latency passes meanwhile.  Claiming late
// keeps the dynamic balance between warps as it was (at batch 1 a warp has about two items).
struct CounterClaims {
    int *counter;
    int pend = 0;
    __device__ __forceinline__ int first() { return claim_item(counter); }
    __device__ __forceinline__ void issue() {
        pend = (threadIdx.x & 31) == 0 ? atomicAdd(counter, 1) : 0;
    }
    __device__ __forceinline__ int take() { return __shfl_sync(0xffffffffu, pend, 0); }
};

struct GateupCtx {
    int ptn;   // first position of the token group << 5 | its number of tokens (1..16)
    int rbks;  // row block << 8 | K slice
};

// Resident CTAs per SM the cross-item kernels keep (at most 65536 / (128 x 128) registers
// each for 4): the same residency as the kernels without the cross-item ring.
constexpr int xi_min_blocks(int NT, int UNROLL) { return (NT == 1 || UNROLL == 2) ? 4 : 3; }

template <int NT, int UNROLL>
__global__ void __launch_bounds__(kMoeThreads, xi_min_blocks(NT, UNROLL))
    moe_gateup_xi_kernel(const MoeArgs a) {
    pdl_wait_trigger();
    const int U = a.meta[0];
    const int total = a.item_gu[U];
    const int g = (threadIdx.x & 31) >> 2;
    auto decode = [&](int it) {
        ItemRows<2, NT, GateupCtx> r;
        const int u = find_unit(a.item_gu, U, it);
        const int local = it - a.item_gu[u];
        const int p0 = a.unit_off[u], p1 = a.unit_off[u + 1];
        const int ntg = (p1 - p0 + a.TT - 1) / a.TT;
        const int tg = local % ntg;
        const int rest = local / ntg;
        const int ks = rest % a.KS;
        const int rb = rest / a.KS;
        const int e = a.unit_expert[u];
        int kb, ke;
        k_slice(a.Hd, a.KS, ks, kb, ke);
        // I is a multiple of 32, so rows rb*16 + g + 8 never pass the last row
        const size_t roff = (size_t)(e < a.E ? e : e - a.E) * a.I * a.Hd +
                            (size_t)(rb * 16 + g) * a.Hd + kb;
        r.w[0] = (e < a.E ? a.W_gate : a.Ws_gate) + roff;
        r.w[1] = (e < a.E ? a.W_up : a.Ws_up) + roff;
        const int pt = p0 + tg * a.TT;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int p = pt + nt * 8 + g;
            r.x[nt] = a.x + (size_t)a.pos_token[p < p1 ? p : pt] * a.Hd + kb;
        }
        r.n = (ke - kb) >> 5;
        r.ctx = GateupCtx{pt << 5 | min(p1 - pt, a.TT), rb << 8 | ks};
        return r;
    };
    auto epilogue = [&](const GateupCtx &c, float (&acc)[2][NT][4]) {
        const int pt = c.ptn >> 5, n = c.ptn & 31, rb = c.rbks >> 8, ks = c.rbks & 255;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int row = rb * 16 + acc_row(q);
                const int t = acc_tok(nt, q);
                if (t >= n) continue;
                const int p = pt + t;
                if (a.KS == 1) {
                    a.h[(size_t)p * a.I + row] =
                        float_to_bf16_bits(__fmul_rn(silu_f(acc[0][nt][q]), acc[1][nt][q]));
                } else {
                    const size_t o = ((size_t)ks * a.P + p) * a.I + row;
                    a.part_g[o] = acc[0][nt][q];
                    a.part_u[o] = acc[1][nt][q];
                }
            }
        }
    };
    CounterClaims claims{&a.meta[3]};
    stream_items<2, NT, UNROLL, GateupCtx>(claims, total, (size_t)8 * a.Hd, decode, epilogue);
}

template <int NT>
struct DownCtx {
    int ks, rbase;     // K slice, first of the item's 32 rows
    int slot[NT][2];   // output slot of the two tokens this lane holds in tile nt (-1: none)
};

template <int NT, int UNROLL>
__global__ void __launch_bounds__(kMoeThreads, xi_min_blocks(NT, UNROLL))
    moe_down_xi_kernel(const MoeArgs a) {
    pdl_wait_trigger();
    const int U = a.meta[0];
    const int total = a.item_dn[U];
    const int g = (threadIdx.x & 31) >> 2;
    const int t2 = (threadIdx.x & 3) * 2;
    auto decode = [&](int it) {
        ItemRows<2, NT, DownCtx<NT>> r;
        const int u = find_unit(a.item_dn, U, it);
        const int local = it - a.item_dn[u];
        const int p0 = a.unit_off[u], p1 = a.unit_off[u + 1];
        const int ntg = (p1 - p0 + a.TT - 1) / a.TT;
        const int tg = local % ntg;
        const int ks = (local / ntg) % a.KSD;
        const int rbase = local / ntg / a.KSD * 32;
        const int e = a.unit_expert[u];
        int kb, ke;
        k_slice(a.I, a.KSD, ks, kb, ke);
        // Hd is a multiple of 32, so rows rbase + 24 + g never pass the last row
        const uint16_t *Wd = (e < a.E ? a.W_down : a.Ws_down) +
                             (size_t)(e < a.E ? e : e - a.E) * a.Hd * a.I + kb;
        r.w[0] = Wd + (size_t)(rbase + g) * a.I;
        r.w[1] = Wd + (size_t)(rbase + 16 + g) * a.I;
        const int pt = p0 + tg * a.TT;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int p = pt + nt * 8 + g;
            r.x[nt] = a.h + (size_t)(p < p1 ? p : pt) * a.I + kb;
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const int q = pt + nt * 8 + t2 + e2;
                r.ctx.slot[nt][e2] = q < p1 ? a.pos_slot[q] : -1;
            }
        }
        r.n = (ke - kb) >> 5;
        r.ctx.ks = ks;
        r.ctx.rbase = rbase;
        return r;
    };
    auto epilogue = [&](const DownCtx<NT> &c, float (&acc)[2][NT][4]) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int slot = c.slot[nt][q & 1];
                    if (slot < 0) continue;
                    const int row = c.rbase + 16 * h + acc_row(q);
                    a.ypart[((size_t)c.ks * a.P + slot) * a.Hd + row] = acc[h][nt][q];
                }
            }
        }
    };
    CounterClaims claims{&a.meta[4]};
    stream_items<2, NT, UNROLL, DownCtx<NT>>(claims, total, (size_t)8 * a.I, decode, epilogue);
}

// y[m] = sum_j w[m,j] * (sum over down slices of y[m,j]) (+ residual): slots in increasing
// order, slices in increasing order.  Slots are taken four at a time with their routing
// entries and all their slice rows loaded before any of them is used, so each group of four
// slots costs one round of memory latency.
__global__ void moe_combine_kernel(const MoeArgs a) {
    pdl_wait_trigger();
    const int m = blockIdx.y;
    const int c4 = blockIdx.x * blockDim.x + threadIdx.x;
    if (c4 * 4 >= a.Hd) return;
    const int S = a.k + a.nsh;
    const size_t plane = (size_t)a.P * a.Hd;
    const float *base = a.ypart + (size_t)m * S * a.Hd + (size_t)c4 * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < S; j0 += 4) {
        float4 v[4][4];
        int e[4];
        float w[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int j = j0 + jj;
            const bool routed = j < a.k;
            e[jj] = routed ? a.topk_idx[(size_t)m * a.k + j] : 0;
            w[jj] = routed ? a.topk_w[(size_t)m * a.k + j] : 1.0f;
            const int nks = (j >= a.k && a.nsh_units == 0) ? 1 : a.KSD;  // tensor-core shared slot: one plane
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                v[jj][ks] = (j < S && ks < nks)
                                ? *reinterpret_cast<const float4 *>(base + ks * plane + (size_t)j * a.Hd)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int j = j0 + jj;
            if (j >= S) break;
            if (j < a.k && (e[jj] < 0 || e[jj] >= a.E)) continue;
            const int nks = (j >= a.k && a.nsh_units == 0) ? 1 : a.KSD;
            float4 t = v[jj][0];
#pragma unroll
            for (int ks = 1; ks < 4; ++ks) {
                if (ks >= nks) break;
                t.x = __fadd_rn(t.x, v[jj][ks].x); t.y = __fadd_rn(t.y, v[jj][ks].y);
                t.z = __fadd_rn(t.z, v[jj][ks].z); t.w = __fadd_rn(t.w, v[jj][ks].w);
            }
            acc.x = __fmaf_rn(w[jj], t.x, acc.x);
            acc.y = __fmaf_rn(w[jj], t.y, acc.y);
            acc.z = __fmaf_rn(w[jj], t.z, acc.z);
            acc.w = __fmaf_rn(w[jj], t.w, acc.w);
        }
    }
    const size_t o = (size_t)m * a.Hd + (size_t)c4 * 4;
    if (a.residual) {
        const uint2 r = *reinterpret_cast<const uint2 *>(a.residual + o);
        acc.x = __fadd_rn(acc.x, bf16_lo(r.x));
        acc.y = __fadd_rn(acc.y, bf16_hi(r.x));
        acc.z = __fadd_rn(acc.z, bf16_lo(r.y));
        acc.w = __fadd_rn(acc.w, bf16_hi(r.y));
    }
    *reinterpret_cast<uint2 *>(a.y + o) =
        make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
}

// Shared expert on the tensor-core path: h = SiLU(sum of gate slices) * (sum of up slices),
// written into the shared expert's h rows (positions s*M .. s*M+M-1).
__global__ void shared_swiglu_kernel(const float *__restrict__ pg, const float *__restrict__ pu,
                                     int split, int M, int I, uint16_t *h) {
    pdl_wait_trigger();
    const size_t total = (size_t)M * I;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        float g = pg[i], u = pu[i];
        for (int s = 1; s < split; ++s) {
            g = __fadd_rn(g, pg[s * total + i]);
            u = __fadd_rn(u, pu[s * total + i]);
        }
        h[i] = float_to_bf16_bits(__fmul_rn(silu_f(g), u));
    }
}

// Sum of the down-projection slices into the (token, slot) rows of the expert outputs.
__global__ void shared_down_reduce_kernel(const float *__restrict__ pd, int split, int M, int Hd,
                                          int S, int slot, float *ypart) {
    pdl_wait_trigger();
    const size_t total = (size_t)M * Hd;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        float d = pd[i];
        for (int s = 1; s < split; ++s) d = __fadd_rn(d, pd[s * total + i]);
        const size_t m = i / Hd, n = i % Hd;
        ypart[(m * S + slot) * Hd + n] = d;
    }
}

// SMs withheld from the routed experts' persistent grids while the shared experts run on the
// side stream, so that the side kernels find free SMs (HLA_SHARED_SM_BUDGET overrides the
// default of 16: at batch 8 the layer took 1029 us with no SMs withheld, 926 us with 16,
// 924 us with 38 and 1110 us with 76; at batch 1 and 2, 16 was best by a small margin).
int shared_sm_budget() {
    const char *env = getenv("HLA_SHARED_SM_BUDGET");
    const int b = env ? atoi(env) : 16;
    return b < 0 ? 0 : (b > sm_count() / 2 ? sm_count() / 2 : b);
}

template <typename K>
int persistent_grid(K kernel) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kMoeThreads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    return per_sm * sm_count();
}

// K steps in the load ring of the cross-item expert kernels: 4 for both at every batch
// (HLA_MOE_RING_GU / HLA_MOE_RING_DN = 2..4 override it for A/B runs).  Measured on the layer
// (CUDA graphs, same box, results bit-identical across depths): gate/up with 4 steps against 2
// took 2957 / 3041 us at batch 64 and 2132 / 2196 us at batch 32 (the 2-step ring that the
// per-item kernel prefers from 32 tokens), 819 / 828 us at batch 8 (3 steps: 845 us); down with
// 2 or 3 steps was slower at every batch (3222 / 3198 us against 3041 us at batch 64).
int moe_ring_depth(bool gateup) {
    const char *env = getenv(gateup ? "HLA_MOE_RING_GU" : "HLA_MOE_RING_DN");
    if (env) {
        const int v = atoi(env);
        if (v >= 2 && v <= 4) return v;
    }
    return 4;
}

template <int NT, int R, typename F>
cudaError_t launch_gateup_ring(F budgeted, const MoeArgs &a, cudaStream_t st) {
    static int g = 0;
    if (!g) g = persistent_grid(moe_gateup_xi_kernel<NT, R>);
    return launch_kernel(moe_gateup_xi_kernel<NT, R>, dim3(budgeted(g)), dim3(kMoeThreads), 0, st, a);
}

template <int NT, int R, typename F>
cudaError_t launch_down_ring(F budgeted, const MoeArgs &a, cudaStream_t st) {
    static int g = 0;
    if (!g) g = persistent_grid(moe_down_xi_kernel<NT, R>);
    return launch_kernel(moe_down_xi_kernel<NT, R>, dim3(budgeted(g)), dim3(kMoeThreads), 0, st, a);
}

template <typename F>
cudaError_t launch_gateup_xi(int TT, int ring, F budgeted, const MoeArgs &a, cudaStream_t st) {
    if (TT == 8) {
        if (ring == 2) return launch_gateup_ring<1, 2>(budgeted, a, st);
        if (ring == 3) return launch_gateup_ring<1, 3>(budgeted, a, st);
        return launch_gateup_ring<1, 4>(budgeted, a, st);
    }
    if (ring == 2) return launch_gateup_ring<2, 2>(budgeted, a, st);
    if (ring == 3) return launch_gateup_ring<2, 3>(budgeted, a, st);
    return launch_gateup_ring<2, 4>(budgeted, a, st);
}

template <typename F>
cudaError_t launch_down_xi(int TT, int ring, F budgeted, const MoeArgs &a, cudaStream_t st) {
    if (TT == 8) {
        if (ring == 2) return launch_down_ring<1, 2>(budgeted, a, st);
        if (ring == 3) return launch_down_ring<1, 3>(budgeted, a, st);
        return launch_down_ring<1, 4>(budgeted, a, st);
    }
    if (ring == 2) return launch_down_ring<2, 2>(budgeted, a, st);
    if (ring == 3) return launch_down_ring<2, 3>(budgeted, a, st);
    return launch_down_ring<2, 4>(budgeted, a, st);
}

// Fork/join events of a side stream, per host thread and per device (an event belongs to the
// device that was current when it was created).
struct SideStreamEvents {
    cudaEvent_t fork = nullptr, join = nullptr;
    bool ok() {
        if (!fork && cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess) return false;
        if (!join && cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess) return false;
        return true;
    }
};
constexpr int kMaxDevices = 64;
// role 0: the shared experts' L2 prefetch; role 1: the shared experts on the side stream
thread_local SideStreamEvents g_side_events[2][kMaxDevices];

SideStreamEvents *side_events(int role) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    SideStreamEvents *e = &g_side_events[role][dev];
    return e->ok() ? e : nullptr;
}


// The shared experts as dense SwiGLUs over all M tokens: gate and up products (split K,
// fp32 slices), h = SiLU(sum g) * (sum u) into the shared experts' h rows, the down product,
// and its slice sum into the shared slots of the expert-output rows (one plane), where the
// combine reads them.  tc: the tensor-core tiles (the optional path at more than 16 tokens);
// otherwise the projection entry point's own choice of path and split.
int run_shared_dense(const MoeLayout &L, bool tc, const hla_bf16 *x, const hla_bf16 *Ws_gate,
                     const hla_bf16 *Ws_up, const hla_bf16 *Ws_down, char *w, cudaStream_t st) {
    const int M = L.M, Hd = L.Hd, I = L.I;
    float *pg = reinterpret_cast<float *>(w + L.off_sh_g);
    float *pu = reinterpret_cast<float *>(w + L.off_sh_u);
    float *pd = reinterpret_cast<float *>(w + L.off_sh_d);
    uint16_t *h = reinterpret_cast<uint16_t *>(w + L.off_h);
    float *ypart = reinterpret_cast<float *>(w + L.off_ypart);
    const int sgu = tc ? L.s_gu : L.d_gu, sdn = tc ? L.s_dn : L.d_dn;
    const int grid = 2 * sm_count();
    auto proj = [&](int N, int K, const hla_bf16 *in, const hla_bf16 *W, int split, float *part) {
        return tc ? run_dense_tc(M, N, K, in, W, split, part, nullptr, 0, nullptr, st)
                  : run_dense(M, N, K, in, W, split, part, nullptr, 0, nullptr, st);
    };
    int r;
    for (int s = 0; s < L.nsh; ++s) {
        const size_t eo = (size_t)s * I * Hd;
        hla_bf16 *hs = h + (size_t)s * M * I;
        if ((r = proj(I, Hd, x, Ws_gate + eo, sgu, pg)) != HLA_OK) return r;
        if ((r = proj(I, Hd, x, Ws_up + eo, sgu, pu)) != HLA_OK) return r;
        if ((r = launched(launch_kernel(shared_swiglu_kernel, dim3(grid), dim3(256), 0, st, (const float *)pg,
                                        (const float *)pu, sgu, M, I, reinterpret_cast<uint16_t *>(hs)))) != HLA_OK)
            return r;
        if ((r = proj(Hd, I, hs, Ws_down + eo, sdn, pd)) != HLA_OK) return r;
        if ((r = launched(launch_kernel(shared_down_reduce_kernel, dim3(grid), dim3(256), 0, st, (const float *)pd,
                                        sdn, M, Hd, L.k + L.nsh, L.k + s, ypart))) != HLA_OK)
            return r;
    }
    return HLA_OK;
}


}  // namespace

size_t moe_workspace_bytes(int M, int Hd, int I, int E, int k, int nsh) {
    return moe_layout(M, Hd, I, E, k, nsh).total;
}

// Whether the shared experts run on the side stream, overlapping the router, dispatch and
// the routed experts ("Hyper-optimizing Kimi K3 in vLLM", Part 1 sec. 3: the shared expert
// does not depend on the routing).  Needs a side stream; the tensor-core shared path
// (HLA_SHARED_TC=1) takes precedence.  Off unless HLA_SHARED_STREAM=1: in the decode layer
// (CUDA graph, 16 SMs withheld from the routed kernels) it measured 212 vs 210 us at batch 1,
// 319 vs 321 us at batch 2, 926 vs 909 us at batch 8, and at batch 64 (no SMs withheld)
// 3980 vs 3105 us, where the grouped unit also profits from the L2 warming of its rows.
bool moe_shared_on_side(int M, int nsh, bool have_side) {
    if (nsh <= 0 || !have_side) return false;
    const char *tc = getenv("HLA_SHARED_TC");
    if (M > 16 && tc && tc[0] == '1') return false;
    const char *env = getenv("HLA_SHARED_STREAM");
    return env && env[0] == '1';
}

// Fork the shared experts onto `side` (after everything already queued on `st`); their
// outputs land in the workspace, and run_moe(..., shared_external = true) joins before its
// combine.  The side stream only touches the shared experts' partial buffers, h rows and
// output slots, which no routed kernel reads or writes.
int moe_shared_side(int M, int Hd, int I, int E, int k, int nsh, const hla_bf16 *x,
                    const hla_bf16 *Ws_gate, const hla_bf16 *Ws_up, const hla_bf16 *Ws_down,
                    void *ws, cudaStream_t st, cudaStream_t side) {
    const MoeLayout L = moe_layout(M, Hd, I, E, k, nsh);
    SideStreamEvents *ev = side_events(1);
    if (!ev) return HLA_ERR_CUDA;
    if (cudaEventRecord(ev->fork, st) != cudaSuccess) return HLA_ERR_CUDA;
    if (cudaStreamWaitEvent(side, ev->fork, 0) != cudaSuccess) return HLA_ERR_CUDA;
    const int r = run_shared_dense(L, false, x, Ws_gate, Ws_up, Ws_down, reinterpret_cast<char *>(ws),
                                   side);
    if (r != HLA_OK) return r;
    if (cudaEventRecord(ev->join, side) != cudaSuccess) return HLA_ERR_CUDA;
    return HLA_OK;
}

int run_moe(int M, int Hd, int I, int E, int k, int nsh, const hla_bf16 *x, const int32_t *topk_idx,
            const float *topk_w, const hla_bf16 *W_gate, const hla_bf16 *W_up,
            const hla_bf16 *W_down, const hla_bf16 *Ws_gate, const hla_bf16 *Ws_up,
            const hla_bf16 *Ws_down, const hla_bf16 *residual, hla_bf16 *y, void *ws,
            cudaStream_t st, cudaStream_t pf, bool shared_external) {
    const MoeLayout L = moe_layout(M, Hd, I, E, k, nsh);
    const bool shared_side = shared_external || moe_shared_on_side(M, nsh, pf != nullptr);
    char *w = reinterpret_cast<char *>(ws);
    MoeArgs a;
    a.M = M; a.Hd = Hd; a.I = I; a.E = E; a.k = k; a.nsh = nsh; a.P = L.P; a.KS = L.KS; a.TT = L.TT;
    a.KSD = L.KSD;
    a.nsh_units = (L.shared_tc || shared_side) ? 0 : nsh;
    a.x = x; a.topk_idx = topk_idx; a.topk_w = topk_w;
    a.W_gate = W_gate; a.W_up = W_up; a.W_down = W_down;
    a.Ws_gate = Ws_gate; a.Ws_up = Ws_up; a.Ws_down = Ws_down;
    a.residual = residual; a.y = y;
    a.meta = reinterpret_cast<int *>(w + L.off_meta);
    a.unit_expert = reinterpret_cast<int *>(w + L.off_unit_expert);
    a.unit_off = reinterpret_cast<int *>(w + L.off_unit_off);
    a.item_gu = reinterpret_cast<int *>(w + L.off_item_gu);
    a.item_dn = reinterpret_cast<int *>(w + L.off_item_dn);
    a.pos_token = reinterpret_cast<int *>(w + L.off_pos_token);
    a.pos_slot = reinterpret_cast<int *>(w + L.off_pos_slot);
    a.h = reinterpret_cast<uint16_t *>(w + L.off_h);
    a.part_g = reinterpret_cast<float *>(w + L.off_part_g);
    a.part_u = reinterpret_cast<float *>(w + L.off_part_u);
    a.ypart = reinterpret_cast<float *>(w + L.off_ypart);

    // Default: warm the shared experts' gate/up rows in L2 while dispatch runs, but only when
    // several token groups will stream those rows at the same time (more than one tile of
    // tokens); with a single token group any prefetch only competes with the weight stream
    // (measured +11% per layer at batch 1, +19% at batch 8).
    const int pm = prefetch_mask();
    const int mask = pm >= 0 ? pm & (kPrefetchSharedGateUp | kPrefetchSharedDown)
                             : ((a.nsh_units > 0 && M > L.TT) ? kPrefetchSharedGateUp : 0);
    const bool side = pf != nullptr && nsh > 0 && mask != 0 && !shared_side;
    SideStreamEvents *pev = side ? side_events(0) : nullptr;
    if (side) {
        if (!pev) return HLA_ERR_CUDA;
        if (cudaEventRecord(pev->fork, st) != cudaSuccess) return HLA_ERR_CUDA;
        if (cudaStreamWaitEvent(pf, pev->fork, 0) != cudaSuccess) return HLA_ERR_CUDA;
        const size_t mat = (size_t)nsh * I * Hd * sizeof(uint16_t);
        int r = HLA_OK;
        if (mask & kPrefetchSharedGateUp) {
            r = run_l2_prefetch(Ws_gate, mat, pf);
            if (r == HLA_OK) r = run_l2_prefetch(Ws_up, mat, pf);
        }
        if (r == HLA_OK && (mask & kPrefetchSharedDown)) r = run_l2_prefetch(Ws_down, mat, pf);
        if (r != HLA_OK) return r;
        if (cudaEventRecord(pev->join, pf) != cudaSuccess) return HLA_ERR_CUDA;
    }

    int r;
    if (L.shared_tc) {
        if ((r = run_shared_dense(L, true, x, Ws_gate, Ws_up, Ws_down, w, st)) != HLA_OK) return r;
    } else if (shared_side && !shared_external) {
        if ((r = moe_shared_side(M, Hd, I, E, k, nsh, x, Ws_gate, Ws_up, Ws_down, ws, st, pf)) != HLA_OK)
            return r;
    }
    // Per-item gate/up kernel (K slices shorter than the ring): loads 4 K steps ahead, or 2
    // from 32 tokens (fewer registers, 4 resident CTAs per SM instead of 3; measured on the
    // decode layer, CUDA graph, same box: gate/up at batch 64 1910 us against 1958, batch 32
    // 2224 us against 2283, slower at batch 16).
    const bool shallow = L.TT == 16 && M >= 32 && moe_shallow_gateup();
    // The cross-item kernels need every K slice to hold at least the ring's depth in steps.
    const int ring_gu = moe_ring_depth(true), ring_dn = moe_ring_depth(false);
    const bool xgu = moe_cross_item() && min_slice_steps(Hd, L.KS) >= ring_gu;
    const bool xdn = moe_cross_item() && min_slice_steps(I, L.KSD) >= ring_dn;
    const int dthreads = (int)round_up((size_t)(E + nsh), 32);
    r = launched(launch_kernel(moe_dispatch_kernel, dim3(1), dim3(dthreads), 0, st, a));
    if (r != HLA_OK) return r;
    const int keep = shared_side ? sm_count() - shared_sm_budget() : sm_count();
    auto budgeted = [&](int full) { return full / sm_count() * keep; };
    cudaError_t e;
    const dim3 mt(kMoeThreads);
    trace_before(kTraceMoeGateup, st);
    if (xgu) {
        e = launch_gateup_xi(L.TT, ring_gu, budgeted, a, st);
    } else if (L.TT == 8) {
        static int g = 0;
        if (!g) g = persistent_grid(moe_gateup_kernel<1, 4>);
        e = launch_kernel(moe_gateup_kernel<1, 4>, dim3(budgeted(g)), mt, 0, st, a);
    } else if (shallow) {
        static int g = 0;
        if (!g) g = persistent_grid(moe_gateup_kernel<2, 2>);
        e = launch_kernel(moe_gateup_kernel<2, 2>, dim3(budgeted(g)), mt, 0, st, a);
    } else {
        static int g = 0;
        if (!g) g = persistent_grid(moe_gateup_kernel<2, 4>);
        e = launch_kernel(moe_gateup_kernel<2, 4>, dim3(budgeted(g)), mt, 0, st, a);
    }
    trace_after(kTraceMoeGateup, st);
    if ((r = launched(e)) != HLA_OK) return r;
    if (L.KS > 1) {
        if ((r = launched(launch_kernel(moe_swiglu_reduce_kernel, dim3(4 * sm_count()), dim3(256), 0, st, a))) !=
            HLA_OK)
            return r;
    }
    trace_before(kTraceMoeDown, st);
    if (xdn) {
        e = launch_down_xi(L.TT, ring_dn, budgeted, a, st);
    } else if (L.TT == 8) {
        static int d = 0;
        if (!d) d = persistent_grid(moe_down_kernel<1>);
        e = launch_kernel(moe_down_kernel<1>, dim3(budgeted(d)), mt, 0, st, a);
    } else {
        static int d = 0;
        if (!d) d = persistent_grid(moe_down_kernel<2>);
        e = launch_kernel(moe_down_kernel<2>, dim3(budgeted(d)), mt, 0, st, a);
    }
    trace_after(kTraceMoeDown, st);
    if ((r = launched(e)) != HLA_OK) return r;
    if (shared_side) {
        SideStreamEvents *sev = side_events(1);
        if (!sev || cudaStreamWaitEvent(st, sev->join, 0) != cudaSuccess) return HLA_ERR_CUDA;
    }
    const dim3 cgrid((unsigned)((Hd / 4 + 127) / 128), (unsigned)M);
    if ((r = launched(launch_kernel(moe_combine_kernel, cgrid, dim3(128), 0, st, a))) != HLA_OK) return r;
    if (side && cudaStreamWaitEvent(st, pev->join, 0) != cudaSuccess) return HLA_ERR_CUDA;
    // kernel forms: ",xgu<ring>" / ",xdn<ring>" cross-item, ",u2" the shallow per-item gate/up
    char ringv[32] = "";
    int o = 0;
    if (xgu) o += snprintf(ringv, sizeof(ringv), ",xgu%d", ring_gu);
    else if (shallow) o += snprintf(ringv, sizeof(ringv), ",u2");
    if (xdn) snprintf(ringv + o, sizeof(ringv) - o, ",xdn%d", ring_dn);
    set_variant("moe<tt%d,ks%d,ksd%d%s%s%s>", L.TT, L.KS, L.KSD, ringv,
                L.shared_tc ? ",shared_tc" : (shared_side ? ",shared_side" : ""),
                side ? ",prefetch" : "");
    return HLA_OK;
}

}  // namespace hla

using namespace hla;

extern "C" size_t moe_expert_forward_workspace_size(int M, int Hd, int I, int E, int k,
                                                    int n_shared) {
    if (M < 1 || Hd < 32 || I < 32 || E < 1 || k < 1 || n_shared < 0) return 0;
    return moe_workspace_bytes(M, Hd, I, E, k, n_shared);
}

namespace hla {

// Argument checks of moe_expert_forward, then the pipeline.  shared_external: the shared
// experts were already forked onto the side stream by moe_shared_side (the layer does this
// before its router).
int moe_forward_checked(int M, int Hd, int I, int E, int k, int n_shared, const hla_bf16 *x,
                        const int32_t *topk_idx, const float *topk_w, const hla_bf16 *W_gate,
                        const hla_bf16 *W_up, const hla_bf16 *W_down, const hla_bf16 *Ws_gate,
                        const hla_bf16 *Ws_up, const hla_bf16 *Ws_down, const hla_bf16 *residual,
                        hla_bf16 *y, void *ws, size_t ws_bytes, cudaStream_t st, cudaStream_t pf,
                        bool shared_external) {
    HLA_REQUIRE(M >= 1 && Hd >= 32 && I >= 32 && E >= 1 && k >= 1 && n_shared >= 0,
                HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(M <= 256 && k <= 16 && k <= E && E + n_shared <= 1024 && n_shared <= 16 &&
                    Hd % 32 == 0 && I % 32 == 0,
                HLA_ERR_UNSUPPORTED);
    HLA_REQUIRE(x && topk_idx && topk_w && W_gate && W_up && W_down && y, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(n_shared == 0 || (Ws_gate && Ws_up && Ws_down), HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(aligned16(x) && aligned16(topk_idx) && aligned16(topk_w) && aligned16(W_gate) &&
                    aligned16(W_up) && aligned16(W_down) && aligned16(y) &&
                    (!residual || aligned16(residual)) &&
                    (n_shared == 0 || (aligned16(Ws_gate) && aligned16(Ws_up) && aligned16(Ws_down))),
                HLA_ERR_MISALIGNED);
    const size_t need = moe_workspace_bytes(M, Hd, I, E, k, n_shared);
    HLA_REQUIRE(ws && ws_bytes >= need, HLA_ERR_WORKSPACE);
    HLA_REQUIRE(aligned16(ws), HLA_ERR_MISALIGNED);
    const PdlChain chain(st, pdl_default(M));  // dispatch, experts and combine as one chain
    return run_moe(M, Hd, I, E, k, n_shared, x, topk_idx, topk_w, W_gate, W_up, W_down, Ws_gate,
                   Ws_up, Ws_down, residual, y, ws, st, pf, shared_external);
}

}  // namespace hla

extern "C" int moe_expert_forward(int M, int Hd, int I, int E, int k, int n_shared,
                                  const hla_bf16 *x, const int32_t *topk_idx, const float *topk_w,
                                  const hla_bf16 *W_gate, const hla_bf16 *W_up,
                                  const hla_bf16 *W_down, const hla_bf16 *Ws_gate,
                                  const hla_bf16 *Ws_up, const hla_bf16 *Ws_down,
                                  const hla_bf16 *residual, hla_bf16 *y, void *ws,
                                  size_t ws_bytes, hla_stream stream, hla_stream prefetch_stream) {
    return moe_forward_checked(M, Hd, I, E, k, n_shared, x, topk_idx, topk_w, W_gate, W_up, W_down,
                               Ws_gate, Ws_up, Ws_down, residual, y, ws, ws_bytes, (cudaStream_t)stream,
                               (cudaStream_t)prefetch_stream, false);
}
