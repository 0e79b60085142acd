// Warp-level weight-streaming tile for skinny products out[n, r] = sum_k W[r, k] x[n, k].
//
// At decode batch sizes the weights (16 rows per warp here) are read exactly once
// and each weight element meets only a handful of tokens, so the product is bound
// by how fast the weights stream from HBM ("moving expert weights through GPU
// memory was a major constraint", "Kimi K3: From Day-0 Availability to Optimized
// Inference").  The tile keeps the weight stream as wide as possible: every lane
// issues 128-bit loads straight into mma.sync A fragments, several K steps ahead.
//
// Fragment trick: m16n8k16 expects lane (g, t) (g = lane/4, t = lane%4) to hold
// A[g][2t,2t+1], A[g+8][2t,2t+1], A[g][2t+8,2t+9], A[g+8][2t+8,2t+9] and
// B[2t,2t+1][g], B[2t+8,2t+9][g].  A dot product does not care about the order of
// its K terms, so lane (g, t) instead loads 8 consecutive K values (16 bytes)
// k0+8t .. k0+8t+7 of weight rows g and g+8 and of token row g, and feeds them to
// two MMAs: physical (8t, 8t+1 | 8t+2, 8t+3) as logical (2t, 2t+1 | 2t+8, 2t+9) of
// the first MMA and (8t+4, 8t+5 | 8t+6, 8t+7) of the second.  A and B use the same
// permutation, so the products are exact dot products over 32 K values per pair.
#pragma once

#include "common.cuh"

namespace hla {

// One K step (32 values) for one warp: acc[m][nt] += W_m[16 rows] . X[8 tokens of tile nt]^T
// from the fragments this lane loaded (wa[m][0] / wa[m][1]: rows g / g+8; xb[nt]: its token row).
template <int NMAT, int NT>
__device__ __forceinline__ void mma_step(const uint4 (&wa)[NMAT][2], const uint4 (&xb)[NT],
                                         float (&acc)[NMAT][NT][4]) {
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            mma_bf16_16816(acc[m][nt], wa[m][0].x, wa[m][1].x, wa[m][0].y, wa[m][1].y, xb[nt].x,
                           xb[nt].y);
            mma_bf16_16816(acc[m][nt], wa[m][0].z, wa[m][1].z, wa[m][0].w, wa[m][1].w, xb[nt].z,
                           xb[nt].w);
        }
    }
}

// Accumulate, for one warp, acc[m][nt] += W_m[16 rows] . X[8 tokens of tile nt]^T over
// K in [kb, ke) (multiples of 32).  wg[m] / wg8[m] point at weight rows g and g+8 of
// matrix m (element 0 of the row); xr[nt] points at the token row that lane group g
// feeds to tile nt.  Lanes whose rows / tokens fall outside the problem point at any
// valid row; their outputs are simply not stored.  before_x() runs between the weight loads
// and the token loads of the first UNROLL steps (the place for a programmatic-launch wait: the
// weights are static, the tokens come from the preceding kernel).
struct NoHook {
    __device__ __forceinline__ void operator()() const {}
};

template <int NMAT, int NT, int UNROLL, class Hook = NoHook>
__device__ __forceinline__ void warp_stream_tile(const uint16_t *const (&wg)[NMAT],
                                                 const uint16_t *const (&wg8)[NMAT],
                                                 const uint16_t *const (&xr)[NT], int kb, int ke,
                                                 float (&acc)[NMAT][NT][4],
                                                 const Hook &before_x = Hook()) {
    const int t8 = (threadIdx.x & 3) * 8;
    const int nsteps = (ke - kb) >> 5;
    uint4 wa[UNROLL][NMAT][2];
    uint4 xb[UNROLL][NT];

#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        if (u < nsteps) {
            const int k = kb + 32 * u + t8;
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
                wa[u][m][0] = ld_weight_v4(wg[m] + k);
                wa[u][m][1] = ld_weight_v4(wg8[m] + k);
            }
        }
    }
    before_x();
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        if (u < nsteps) {
            const int k = kb + 32 * u + t8;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) xb[u][nt] = ld_act_v4(xr[nt] + k);
        }
    }

    for (int s0 = 0; s0 < nsteps; s0 += UNROLL) {
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int s = s0 + u;
            if (s < nsteps) {
                mma_step<NMAT, NT>(wa[u], xb[u], acc);
                if (s + UNROLL < nsteps) {
                    const int k = kb + 32 * (s + UNROLL) + t8;
#pragma unroll
                    for (int m = 0; m < NMAT; ++m) {
                        wa[u][m][0] = ld_weight_v4(wg[m] + k);
                        wa[u][m][1] = ld_weight_v4(wg8[m] + k);
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) xb[u][nt] = ld_act_v4(xr[nt] + k);
                }
            }
        }
    }
}

// Output coordinates of accumulator element e (0..3) of tile nt for this lane:
// row (within the 16-row block) and token (within the 8*NT token group).
__device__ __forceinline__ int acc_row(int e) { return (threadIdx.x & 31) / 4 + ((e & 2) ? 8 : 0); }
__device__ __forceinline__ int acc_tok(int nt, int e) { return nt * 8 + (threadIdx.x & 3) * 2 + (e & 1); }

// Split [0, K) into `split` slices that are multiples of 32 and return slice ks.
__device__ __forceinline__ void k_slice(int K, int split, int ks, int &kb, int &ke) {
    const int steps = K >> 5;
    const int per = (steps + split - 1) / split;
    kb = min(steps, ks * per) * 32;
    ke = min(steps, (ks + 1) * per) * 32;
}

// Fewest K steps of 32 in any of the `split` slices of [0, K) that k_slice hands out.
inline int min_slice_steps(int K, int split) {
    const int steps = K >> 5;
    const int per = (steps + split - 1) / split;
    int mn = steps;
    for (int s = 0; s < split; ++s) {
        const int kb = s * per < steps ? s * per : steps;
        const int ke = (s + 1) * per < steps ? (s + 1) * per : steps;
        if (ke - kb < mn) mn = ke - kb;
    }
    return mn;
}

// ---------------------------------------------------------------------------------------
// Cross-item pipeline.  A warp that runs warp_stream_tile once per work item stops loading
// at the end of every item: its ring drains, the next item is found and decoded, and only
// then are that item's first loads issued, so each item boundary leaves the warp with
// nothing in flight for about one memory latency (plus, with dynamic claiming, one atomic).
// With items of 64-128 KB of weights that gap is a visible share of an item.  stream_items
// keeps a ring of UNROLL K steps running across item boundaries: the next item is claimed
// kClaimAhead steps before its first loads are due, decoded just before them, and the last
// steps of one item are multiplied while the first loads of the next are in flight.  Every
// item must have at least UNROLL K steps (the caller checks the K slices with
// min_slice_steps), so the loads ahead reach at most into the next item.
constexpr int kClaimAhead = 2;

// What a warp streams for one work item: weight row g of each matrix (row g + 8 lies ld8
// elements further on) and the token row of each 8-token tile, all offset to the item's
// first K value; n K steps of 32 (0: no item); ctx is what the item's epilogue needs.
template <int NMAT, int NT, class Ctx>
struct ItemRows {
    const uint16_t *w[NMAT];
    const uint16_t *x[NT];
    int n;
    Ctx ctx;
    __device__ __forceinline__ void load_w(int s, size_t ld8, uint4 (&wa)[NMAT][2]) const {
        const int k = 32 * s + (threadIdx.x & 3) * 8;
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
            wa[m][0] = ld_weight_v4(w[m] + k);
            wa[m][1] = ld_weight_v4(w[m] + ld8 + k);
        }
    }
    __device__ __forceinline__ void load_x(int s, uint4 (&xb)[NT]) const {
        const int k = 32 * s + (threadIdx.x & 3) * 8;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) xb[nt] = ld_act_v4(x[nt] + k);
    }
    __device__ __forceinline__ void load(int s, size_t ld8, uint4 (&wa)[NMAT][2],
                                         uint4 (&xb)[NT]) const {
        load_w(s, ld8, wa);
        load_x(s, xb);
    }
};

template <int NMAT, int NT>
__device__ __forceinline__ void zero_acc(float (&acc)[NMAT][NT][4]) {
#pragma unroll
    for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[m][nt][q] = 0.f;
}

// Items handed out round-robin: warp w of nw takes items w, w + nw, w + 2 nw, ...
struct StridedClaims {
    int it, stride;
    __device__ __forceinline__ int first() { return it; }
    __device__ __forceinline__ void issue() {}
    __device__ __forceinline__ int take() { return it += stride; }
};

// claims: first() -> the warp's first item, issue() at the claim point, take() -> the next
// item (>= total: none).  decode(it) -> ItemRows of item it; epilogue(ctx, acc) stores an
// item's result.  before_x() runs between the weight loads and the token loads of the first
// ring (as in warp_stream_tile).
template <int NMAT, int NT, int UNROLL, class Ctx, class Claims, class Decode, class Epilogue,
          class Hook = NoHook>
__device__ __forceinline__ void stream_items(Claims &claims, int total, size_t ld8,
                                             const Decode &decode, const Epilogue &epilogue,
                                             const Hook &before_x = Hook()) {
    using Item = ItemRows<NMAT, NT, Ctx>;
    int it = claims.first();
    if (it >= total) return;
    Item cur = decode(it);
    Item nxt;
    nxt.n = 0;
    uint4 wa[UNROLL][NMAT][2];
    uint4 xb[UNROLL][NT];
    float acc[NMAT][NT][4];
    zero_acc<NMAT, NT>(acc);
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) cur.load_w(u, ld8, wa[u]);
    before_x();
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) cur.load_x(u, xb[u]);
    int ls = 0;  // the step of cur that ring slot u holds
    for (;;) {
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int first_next = cur.n - UNROLL;  // the step whose refill is next's step 0
            if (ls == (first_next > kClaimAhead ? first_next - kClaimAhead : 0)) claims.issue();
            mma_step<NMAT, NT>(wa[u], xb[u], acc);
            if (ls == first_next) {
                it = claims.take();
                if (it < total) nxt = decode(it);
            }
            int j = ls + UNROLL;  // the step that refills slot u, counted from cur's first
            if (ls == cur.n - 1) {
                epilogue(cur.ctx, acc);
                zero_acc<NMAT, NT>(acc);
                if (nxt.n == 0) return;
                cur = nxt;
                nxt.n = 0;
                ls = -1;
                j = UNROLL - 1;
            }
            if (j < cur.n) cur.load(j, ld8, wa[u], xb[u]);
            else if (j - cur.n < nxt.n) nxt.load(j - cur.n, ld8, wa[u], xb[u]);
            ++ls;
        }
    }
}

}  // namespace hla
