// KDA recurrent-state kernels: decode step, speculative verify, accepted-prefix replay,
// and the accepted-length bookkeeping.
//
// The update is the gated delta rule (KDA's fixed-size recurrent state, "Kimi K3:
// From Day-0 Availability to Optimized Inference"):
//     S' = diag(alpha) S                (rows scaled by the per-key decay)
//     u  = S'^T k,  w = S'^T q          (one pass over S' gives both)
//     S_t = S' + beta k (v - u)^T        (= (I - beta k k^T) S' + beta k v^T)
//     o   = w + beta (q.k) (v - u)       (= S_t^T q, read from the updated state)
// Column j of S_t depends only on column j of S, so a (sequence, head) state
// splits over d_v into independent column slices; small batches use narrow
// slices to put work on every SM ("KDA decode kernel ... scheduling tuned for the
// batch size and number of heads", "Hyper-optimizing Kimi K3 in vLLM", Part 1 sec. 1).
//
// Layout inside a CTA: 8 row groups x (CW/4) float4 column groups.  Thread
// (rg, cg) keeps rows rg, rg+8, rg+16, ... of 4 columns in registers, so the state
// is read from HBM once and written once.  The 8 row groups of a column group are
// lanes of one warp (lane = 4 rg + cg % 4; warp w holds column groups 4w..4w+3), so
// the sums over rows (u, w, q.k) finish with three butterfly shuffles inside the warp
// and a step needs no block barrier.  The row partition (and therefore the order of
// every reduction) is the same for every slice width, which makes the result
// independent of the variant chosen: replaying T tokens is bit-identical to T single
// decode steps.
#include <cstdlib>

#include "common.cuh"

namespace hla {
namespace {

constexpr int kRowGroups = 8;
constexpr int kMaxWindow = 8;

// component e (a compile-time constant after unrolling) of a float4
__device__ __forceinline__ float f4_at(const float4 v, int e) {
    return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

enum KdaMode { kDecode = 0, kVerify = 1, kReplay = 2, kReplayVerify = 3, kExtend = 4 };

struct KdaParams {
    float *S;
    const int32_t *state_idx;
    const uint16_t *q, *k, *v;          // this call's tokens [B, T, H, .] (T = 1 for decode);
    const float *alpha, *beta;          //   extend: packed [N, H, .] rows cu_seqlens[b]..[b+1]-1
    const uint16_t *qp, *kp, *vp;       // replay-verify: the previous window [B, Tp, H, .]
    const float *alphap, *betap;
    const int32_t *accepted;            // replay: of this window; replay-verify: of the previous one
    const int32_t *cu_seqlens;          // extend: [B + 1] token offsets of the sequences
    void *o;
    int o_bf16;
    int B, T, Tp, H;
    // the state may be read before waiting for the kernel before this one: set only where that
    // kernel is known not to write the state (the decode layer's projection epilogue); inside a
    // caller's launch chain the predecessor may be a KDA kernel that writes it
    int state_first;
};

// Extend programs take their sequences in two classes: first those with more than one block of
// TMAX tokens (serial chains), in batch order, then the others.  Returns the sequence at schedule
// position r, computed by the whole block from the sequence offsets.  In batch order, chains that
// come after many short programs start only once those have filled the SMs, and finish last,
// several to an SM.  Kept out of line: inlined, it changed the register allocation of the token
// loop and made long chains slower.
template <int NTHR, int TMAX>
__device__ __noinline__ int extend_sequence_at(int r, int B, const int32_t *cu) {
    __shared__ int s_cnt[NTHR / 32];
    __shared__ int s_seq;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    auto is_chain = [&](int j) { return j < B && cu[j + 1] - cu[j] > TMAX; };
    int n_chain = 0;
    for (int base = 0; base < B; base += NTHR) n_chain += __syncthreads_count(is_chain(base + tid));
    // position of sequence j: its rank among the chains, or n_chain + its rank among the others
    int before = 0;  // chains in earlier rounds
    for (int base = 0; base < B; base += NTHR) {
        const int j = base + tid;
        const bool chain = is_chain(j);
        const unsigned m = __ballot_sync(0xffffffffu, chain);
        if (lane == 0) s_cnt[warp] = __popc(m);
        __syncthreads();
        int lp = before + __popc(m & ((1u << lane) - 1u)), round = 0;
        for (int w = 0; w < NTHR / 32; ++w) {
            lp += w < warp ? s_cnt[w] : 0;
            round += s_cnt[w];
        }
        if (j < B && (chain ? lp : n_chain + (j - lp)) == r) s_seq = j;  // exactly one j matches
        before += round;
        __syncthreads();
    }
    return s_seq;
}

// Each CTA runs a short program over its (sequence, head, column slice):
//   n_pre steps from the previous window, then commit the state (replay-verify only);
//   n_main steps from this call's tokens, writing o (decode, verify, replay-verify, extend)
//   and/or committing the state at the end (decode, replay, extend).
// Tokens are staged through shared memory in blocks of TMAX; the state stays in registers
// for the whole program.  Every step is the same arithmetic, so any combination is
// bit-identical to the corresponding sequence of single steps.
// The multi-token verify programs are held to 128 registers per thread (4 CTAs of 128 threads,
// or 16 one-warp CTAs, per SM); left free they take up to 146 and lose a resident CTA.  The
// other programs stay near 128 on their own (decode, replay) or spill under the cap (extend),
// so they get no minimum (0: the compiler's own choice, as with no second bound).
constexpr int kda_min_blocks(int cw, int mode) {
    return (mode == 1 || mode == 3) ? 65536 / (kRowGroups * cw / 4 * 128) : 0;
}

template <int DK, int CW, int MODE>
__global__ void __launch_bounds__(kRowGroups *CW / 4, kda_min_blocks(CW, MODE))
    kda_recur_kernel(const KdaParams p) {
    constexpr int CG = CW / 4;
    constexpr int RPT = DK / kRowGroups;
    constexpr int DV = DK;
    constexpr int NSLICE = DV / CW;
    constexpr int NTHR = kRowGroups * CG;
    constexpr int TMAX = MODE == kDecode ? 1 : (MODE == kReplayVerify ? 2 * kMaxWindow : kMaxWindow);
    constexpr bool WRITE_O = MODE != kReplay;
    constexpr bool COMMIT_END = MODE == kDecode || MODE == kReplay || MODE == kExtend;
    static_assert(TMAX <= NTHR, "one thread per token loads beta");

    static_assert(CG % 4 == 0, "a warp holds 8 row groups x 4 column groups");
    // q, k and alpha of a token are stored row-group-major: row i at (i % 8) * PAD + i / 8, so a
    // thread's rows rg, rg+8, ... are contiguous (float4 reads) and the 8 row groups of a warp
    // start in distinct banks (PAD = RPT + 4)
    constexpr int PAD = RPT + 4;
    __shared__ __align__(16) float sq[TMAX][8 * PAD], sk[TMAX][8 * PAD], sa[TMAX][8 * PAD],
        sv[TMAX][CW];
    __shared__ float sb[TMAX];
    auto rowpos = [](int i) { return (i & 7) * PAD + (i >> 3); };

    // Only extend programs can exceed one block of TMAX tokens.  They copy the next block's raw
    // token vectors into shared memory (asynchronously, two buffers) while the current block runs,
    // so a long serial chain never waits on global memory between blocks.
    constexpr bool BLOCKED = MODE == kExtend;
    // per token: DK/8 16-byte chunks of q, DK/8 of k, DK/4 of alpha and CW/8 of v; item x of a
    // block is chunk x % PER_TOK of token x / PER_TOK
    constexpr int QC = DK / 8, AC = DK / 4, VC = CW / 8, PER_TOK = 2 * QC + AC + VC;
    __shared__ __align__(16) uint4 raw[BLOCKED ? 2 : 1][BLOCKED ? TMAX * PER_TOK : 1];
    __shared__ float rawb[BLOCKED ? 2 : 1][BLOCKED ? TMAX : 1];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int rg = lane >> 2;
    const int cg = (tid >> 5) * 4 + (lane & 3);
    const int slice = blockIdx.x % NSLICE;
    const int bh = blockIdx.x / NSLICE;
    const int h = bh % p.H;
    int b = bh / p.H;
    const int col0 = slice * CW;

    // Decode and verify may read their state slice before waiting for the kernel before them,
    // when the caller knows that kernel does not write the state (p.state_first); otherwise, and
    // for the programs that first read accepted lengths or sequence offsets, they wait first.
    const bool state_first = (MODE == kDecode || MODE == kVerify) && p.state_first;
    if (!state_first) pdl_wait_trigger();

    int n_pre = 0, n_main = MODE == kDecode ? 1 : p.T;
    int seq0 = 0;
    if (MODE == kReplay || MODE == kReplayVerify) {
        const int lim = MODE == kReplay ? p.T : p.Tp;
        const int a0 = p.accepted[b];
        const int a = a0 < 0 ? 0 : (a0 > lim ? lim : a0);
        if (MODE == kReplay) {
            n_main = a;
            if (a == 0) return;  // nothing accepted: the committed state is not touched
        } else {
            n_pre = a;
        }
    }
    if (MODE == kExtend) {
        b = extend_sequence_at<NTHR, TMAX>(b, p.B, p.cu_seqlens);
        seq0 = p.cu_seqlens[b];
        n_main = p.cu_seqlens[b + 1] - seq0;
        if (n_main <= 0) return;  // no new tokens: the state is not touched
    }
    const int steps = n_pre + n_main;
    const int Tld = MODE == kDecode ? 1 : p.T;

    // row of step t in its [., H, .] token tensor (previous window, this window, or packed)
    auto token_row = [&](int t) -> size_t {
        if (t < n_pre) return ((size_t)b * p.Tp + t) * p.H + h;
        const int tm = t - n_pre;
        if (MODE == kExtend) return ((size_t)seq0 + tm) * p.H + h;
        return ((size_t)b * Tld + tm) * p.H + h;
    };

    // global address of item x of the block starting at step t0
    auto item_src = [&](int x, int t0) -> const void * {
        const int tt = x / PER_TOK, c = x - tt * PER_TOK;
        const int t = t0 + tt;
        const bool pre = t < n_pre;
        const size_t tok = token_row(t);
        if (c < QC) return (pre ? p.qp : p.q) + tok * DK + 8 * c;
        if (c < 2 * QC) return (pre ? p.kp : p.k) + tok * DK + 8 * (c - QC);
        if (c < 2 * QC + AC) return (pre ? p.alphap : p.alpha) + tok * DK + 4 * (c - 2 * QC);
        return (pre ? p.vp : p.v) + tok * DV + col0 + 8 * (c - 2 * QC - AC);
    };
    // item x (16 bytes) into the staged layout: q, k and alpha row-group-major as fp32, v as fp32
    auto store_item = [&](int x, const uint4 w) {
        const int tt = x / PER_TOK, c = x - tt * PER_TOK;
        if (c < 2 * QC + AC && c >= 2 * QC) {  // 4 alphas (fp32 bits), rows i0..i0+3
            const int i0 = 4 * (c - 2 * QC);
            sa[tt][rowpos(i0 + 0)] = __uint_as_float(w.x);
            sa[tt][rowpos(i0 + 1)] = __uint_as_float(w.y);
            sa[tt][rowpos(i0 + 2)] = __uint_as_float(w.z);
            sa[tt][rowpos(i0 + 3)] = __uint_as_float(w.w);
        } else if (c < 2 * QC) {  // 8 bf16 of q or k, rows 8j .. 8j+7 (one per row group)
            float *dst = c < QC ? sq[tt] : sk[tt];
            const int j = c < QC ? c : c - QC;
            dst[0 * PAD + j] = bf16_lo(w.x); dst[1 * PAD + j] = bf16_hi(w.x);
            dst[2 * PAD + j] = bf16_lo(w.y); dst[3 * PAD + j] = bf16_hi(w.y);
            dst[4 * PAD + j] = bf16_lo(w.z); dst[5 * PAD + j] = bf16_hi(w.z);
            dst[6 * PAD + j] = bf16_lo(w.w); dst[7 * PAD + j] = bf16_hi(w.w);
        } else {
            float *dst = &sv[tt][8 * (c - 2 * QC - AC)];
            reinterpret_cast<float4 *>(dst)[0] =
                make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
            reinterpret_cast<float4 *>(dst)[1] =
                make_float4(bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w));
        }
    };
    // extend: raw copies of the block starting at step tb into buffer buf, as one commit group
    // (an empty group past the last block keeps the group count of every iteration the same)
    auto issue_raw = [&](int buf, int tb) {
        if (tb < steps) {
            const int tn_b = steps - tb < TMAX ? steps - tb : TMAX;
            for (int x = tid; x < tn_b * PER_TOK; x += NTHR) cp_async16(&raw[buf][x], item_src(x, tb));
            if (tid < tn_b) cp_async4(&rawb[buf][tid], p.beta + token_row(tb + tid));
        }
        cp_async_commit();
    };
    if constexpr (BLOCKED) issue_raw(0, 0);  // in flight together with the state loads

    const int slot = p.state_idx ? p.state_idx[b] : b;
    float *Sb = p.S + ((size_t)slot * p.H + h) * (size_t)(DK * DV) + col0 + cg * 4;

    // the thread's 4 columns as two float2 pairs (columns 0-1, 2-3), so that the per-row
    // arithmetic runs as packed fp32x2 operations: two correctly rounded fp32 results per
    // instruction, the same bits as two scalar operations
    float2 s[RPT][2];
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
        const float4 t = *reinterpret_cast<const float4 *>(Sb + (size_t)(rg + kRowGroups * j) * DV);
        s[j][0] = make_float2(t.x, t.y);
        s[j][1] = make_float2(t.z, t.w);
    }
    auto store_state = [&]() {
#pragma unroll
        for (int j = 0; j < RPT; ++j)
            *reinterpret_cast<float4 *>(Sb + (size_t)(rg + kRowGroups * j) * DV) =
                make_float4(s[j][0].x, s[j][0].y, s[j][1].x, s[j][1].y);
    };
    if (state_first) pdl_wait_trigger();

    // For the programs other than extend the loop body runs once with every step in it (and
    // compiles to straight-line code).
    for (int t0 = 0, blk = 0; BLOCKED ? t0 < steps : t0 == 0; t0 += TMAX, ++blk) {
        const int tn = !BLOCKED ? steps : (steps - t0 < TMAX ? steps - t0 : TMAX);

        // Token vectors of steps t0 .. t0+tn-1 into slots 0..tn-1.  The loaders fill the same
        // shared arrays with the same values (results do not depend on the choice); which is
        // faster depends on the CTA width and the program length.
        float beta_r = 0.f;
        if constexpr (BLOCKED) {
            const int buf = blk & 1;
            issue_raw(buf ^ 1, t0 + TMAX);  // the next block, into the buffer converted last time
            cp_async_wait<1>();             // this thread's copies of this block have landed
            __syncthreads();                // everyone's have; the previous block is no longer read
            for (int x = tid; x < tn * PER_TOK; x += NTHR) store_item(x, raw[buf][x]);
            if (tid < tn) beta_r = rawb[buf][tid];
        } else {
            // beta goes to a register first so its load overlaps the others
            if (tid < tn) {
                const int t = t0 + tid;
                beta_r = (t < n_pre ? p.betap : p.beta)[token_row(t)];
            }
            constexpr bool kVectorLoads = CW <= 32 || MODE == kReplayVerify;
            if constexpr (kVectorLoads) {
                // one 128-bit load per item; a thread issues LDEPTH loads before storing any of them
                constexpr int LDEPTH = 4;
                const int n_items = tn * PER_TOK;
                for (int x0 = tid; x0 < n_items; x0 += LDEPTH * NTHR) {
                    uint4 r[LDEPTH];
#pragma unroll
                    for (int u = 0; u < LDEPTH; ++u) {
                        const int x = x0 + u * NTHR;
                        if (x >= n_items) break;
                        r[u] = ld_act_v4(item_src(x, t0));
                    }
#pragma unroll
                    for (int u = 0; u < LDEPTH; ++u) {
                        const int x = x0 + u * NTHR;
                        if (x >= n_items) break;
                        store_item(x, r[u]);
                    }
                }
            } else {
                // scalar loads, one unrolled pass per token (measured faster for 64/128-column
                // slices in the decode, verify and replay programs)
                for (int tt = 0; tt < tn; ++tt) {
                    const int t = t0 + tt;
                    const bool pre = t < n_pre;
                    const uint16_t *q = pre ? p.qp : p.q, *k = pre ? p.kp : p.k, *v = pre ? p.vp : p.v;
                    const float *al = pre ? p.alphap : p.alpha;
                    const size_t tok = token_row(t);
                    for (int i = tid; i < DK; i += NTHR) {
                        sq[tt][rowpos(i)] = bf16_bits_to_float(q[tok * DK + i]);
                        sk[tt][rowpos(i)] = bf16_bits_to_float(k[tok * DK + i]);
                        sa[tt][rowpos(i)] = al[tok * DK + i];
                    }
                    for (int c = tid; c < CW; c += NTHR) sv[tt][c] = bf16_bits_to_float(v[tok * DV + col0 + c]);
                }
            }
        }
        if (tid < tn) sb[tid] = beta_r;
        __syncthreads();

        for (int tt = 0; tt < tn; ++tt) {
            const int t = t0 + tt;
            float2 pu[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)}, pw[2] = {pu[0], pu[1]};
            float pqk = 0.f;
            const float4 *a4 = reinterpret_cast<const float4 *>(&sa[tt][rg * PAD]);
            const float4 *k4 = reinterpret_cast<const float4 *>(&sk[tt][rg * PAD]);
            const float4 *q4 = reinterpret_cast<const float4 *>(&sq[tt][rg * PAD]);
#pragma unroll
            for (int j = 0; j < RPT; ++j) {  // row rg + 8 j
                const float a = f4_at(a4[j >> 2], j & 3), kk = f4_at(k4[j >> 2], j & 3),
                            qq = f4_at(q4[j >> 2], j & 3);
                const float2 a2 = make_float2(a, a), k2 = make_float2(kk, kk), q2 = make_float2(qq, qq);
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    s[j][h2] = __fmul2_rn(s[j][h2], a2);             // decay
                    pu[h2] = __ffma2_rn(k2, s[j][h2], pu[h2]);       // k . S'
                    pw[h2] = __ffma2_rn(q2, s[j][h2], pw[h2]);       // q . S'
                }
                pqk = __fmaf_rn(qq, kk, pqk);
            }
            // sums over the 8 row groups (lane bits 2..4): a butterfly, after which every lane
            // holds the same bits (each level adds the same two values in either order)
#pragma unroll
            for (int m = 4; m < 32; m <<= 1) {
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    pu[h2] = __fadd2_rn(pu[h2], make_float2(__shfl_xor_sync(0xffffffffu, pu[h2].x, m),
                                                            __shfl_xor_sync(0xffffffffu, pu[h2].y, m)));
                    pw[h2] = __fadd2_rn(pw[h2], make_float2(__shfl_xor_sync(0xffffffffu, pw[h2].x, m),
                                                            __shfl_xor_sync(0xffffffffu, pw[h2].y, m)));
                }
                pqk = __fadd_rn(pqk, __shfl_xor_sync(0xffffffffu, pqk, m));
            }
            const float bt = sb[tt];
            const float4 vv = *reinterpret_cast<const float4 *>(&sv[tt][cg * 4]);
            // d = beta (v - u), per column
            float2 d[2];
            d[0] = make_float2(__fmul_rn(bt, __fsub_rn(vv.x, pu[0].x)), __fmul_rn(bt, __fsub_rn(vv.y, pu[0].y)));
            d[1] = make_float2(__fmul_rn(bt, __fsub_rn(vv.z, pu[1].x)), __fmul_rn(bt, __fsub_rn(vv.w, pu[1].y)));
            // the state after a verify program's last token is never read (no commit, and o comes
            // from w, q.k and d): its update is skipped
            if (COMMIT_END || t != steps - 1) {
#pragma unroll
                for (int j = 0; j < RPT; ++j) {
                    const float kk = f4_at(k4[j >> 2], j & 3);
                    const float2 k2 = make_float2(kk, kk);
                    s[j][0] = __ffma2_rn(k2, d[0], s[j][0]);
                    s[j][1] = __ffma2_rn(k2, d[1], s[j][1]);
                }
            }
            if (WRITE_O && t >= n_pre && rg == 0) {
                const float2 qk2 = make_float2(pqk, pqk);
                const float2 o0 = __ffma2_rn(qk2, d[0], pw[0]), o1 = __ffma2_rn(qk2, d[1], pw[1]);
                const size_t oo = token_row(t) * DV + col0 + cg * 4;
                if (p.o_bf16) {
                    uint2 pk = make_uint2(pack_bf16x2(o0.x, o0.y), pack_bf16x2(o1.x, o1.y));
                    *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(p.o) + oo) = pk;
                } else {
                    *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.o) + oo) =
                        make_float4(o0.x, o0.y, o1.x, o1.y);
                }
            }
            if (MODE == kReplayVerify && t + 1 == n_pre) {
                // the replayed prefix is the new committed state; the new window is only verified
                store_state();
            }
        }
    }

    if (COMMIT_END) store_state();
}

template <int DK, int MODE>
int launch_dk(int cw, const KdaParams &p, cudaStream_t st) {
    const int grid_per_head = DK / cw;
    const dim3 grid((unsigned)((size_t)p.B * p.H * grid_per_head));
    cudaError_t e;
    trace_before(kTraceKda, st);
    switch (cw) {
        case 16: e = launch_kernel(kda_recur_kernel<DK, 16, MODE>, grid, dim3(kRowGroups * 4), 0, st, p); break;
        case 32: e = launch_kernel(kda_recur_kernel<DK, 32, MODE>, grid, dim3(kRowGroups * 8), 0, st, p); break;
        case 64: e = launch_kernel(kda_recur_kernel<DK, 64, MODE>, grid, dim3(kRowGroups * 16), 0, st, p); break;
        case 128:
            if constexpr (DK >= 128 && MODE != kReplayVerify) {
                e = launch_kernel(kda_recur_kernel<DK, 128, MODE>, grid, dim3(kRowGroups * 32), 0, st, p);
                break;
            } else {
                return HLA_ERR_UNSUPPORTED;
            }
        default: return HLA_ERR_UNSUPPORTED;
    }
    trace_after(kTraceKda, st);
    return launched(e);
}

// Column-slice width.  Measured on GB300 (d = 128, 32 heads, CUDA graphs, states rotated
// over 512 MB, the warp-shuffle row sums):
//   decode: 16 columns, one warp per CTA, at every batch (batch 1: 2.85-3.2 us vs 3.56 with
//           32; batch 32: 22.7 vs 23.4 with 32; batch 64: 42.1 vs 42.4);
//   verify / replay / fused window (several tokens per CTA): 64 columns, halved while the
//           heads do not cover the SMs twice (batch 16 separate window: 23.1 us vs 26.7 with
//           32 and 32.2 with 16; batch 64: 81.5 vs 96.3 and 132);
//   extend: whole heads (128 columns) while the heads fit one per SM, so each serial chain
//           has an SM to itself (4 x 512-token chunks: 314 us vs 349 with 64), else 64 (60
//           decodes + 4 x 128-token chunks: 128.6 us vs 141 with 128).
int choose_cw(int B, int H, int dv, int mode) {
    const char *env = getenv("HLA_KDA_CW");
    if (env) {
        const int v = atoi(env);
        if ((v == 16 || v == 32 || v == 64 || v == 128) && v <= dv) return v;
    }
    const long heads = (long)B * H;
    if (mode == kDecode) return 16 <= dv ? 16 : dv;
    if (mode == kExtend) return heads <= sm_count() ? dv : (dv < 64 ? dv : 64);
    // 64-column slices (128 threads, 32 KB of state per CTA) once there are enough heads;
    // narrower slices put work on every SM at small batch.
    const long target = 2L * sm_count();
    int cw = dv < 64 ? dv : 64;
    while (cw > 16 && heads * (dv / cw) < target) cw /= 2;
    return cw;
}

struct PrevWindow {
    const hla_bf16 *q = nullptr, *k = nullptr, *v = nullptr;
    const float *alpha = nullptr, *beta = nullptr;
    int T = 0;
};

int run_kda(int mode, int B, int T, int H, int dk, int dv, float *S, const int32_t *state_idx,
            const hla_bf16 *q, const hla_bf16 *k, const hla_bf16 *v, const float *alpha,
            const float *beta, const int32_t *accepted, void *o, int o_dtype, cudaStream_t st,
            const PrevWindow &prev = PrevWindow(), const int32_t *cu_seqlens = nullptr,
            bool state_first = false) {
    HLA_REQUIRE(B >= 1 && H >= 1 && T >= 1, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(dk == dv && (dk == 64 || dk == 128), HLA_ERR_UNSUPPORTED);
    HLA_REQUIRE(T <= kMaxWindow, HLA_ERR_UNSUPPORTED);
    HLA_REQUIRE((long)B * H * (dv / 16) < (1L << 31), HLA_ERR_UNSUPPORTED);
    HLA_REQUIRE(S && q && k && v && alpha && beta, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE((mode != kReplay && mode != kReplayVerify) || accepted, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(mode == kReplay || o, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(mode != kExtend || (cu_seqlens && aligned16(cu_seqlens)),
                cu_seqlens ? HLA_ERR_MISALIGNED : HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(o_dtype == HLA_F32 || o_dtype == HLA_BF16, HLA_ERR_INVALID_ARG);
    if (mode == kReplayVerify) {
        HLA_REQUIRE(prev.T >= 1, HLA_ERR_INVALID_ARG);
        HLA_REQUIRE(prev.T <= kMaxWindow, HLA_ERR_UNSUPPORTED);
        HLA_REQUIRE(prev.q && prev.k && prev.v && prev.alpha && prev.beta, HLA_ERR_INVALID_ARG);
        HLA_REQUIRE(aligned16(prev.q) && aligned16(prev.k) && aligned16(prev.v) &&
                        aligned16(prev.alpha) && aligned16(prev.beta),
                    HLA_ERR_MISALIGNED);
    }
    HLA_REQUIRE(aligned16(S) && aligned16(q) && aligned16(k) && aligned16(v) && aligned16(alpha) &&
                    aligned16(beta) && (o == nullptr || aligned16(o)) &&
                    (state_idx == nullptr || aligned16(state_idx)) &&
                    (accepted == nullptr || aligned16(accepted)),
                HLA_ERR_MISALIGNED);
    KdaParams p;
    p.S = S; p.state_idx = state_idx; p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.beta = beta;
    p.qp = prev.q; p.kp = prev.k; p.vp = prev.v; p.alphap = prev.alpha; p.betap = prev.beta;
    p.Tp = prev.T;
    p.accepted = accepted; p.o = o; p.o_bf16 = o_dtype == HLA_BF16; p.B = B; p.T = T; p.H = H;
    p.cu_seqlens = cu_seqlens;
    p.state_first = state_first ? 1 : 0;
    int cw = choose_cw(B, H, dv, mode);
    if (mode == kReplayVerify && cw > 64) cw = 64;  // two windows of token vectors in shared memory
    static const char *names[5] = {"decode", "verify", "replay", "replay_verify", "extend"};
    set_variant("kda_recur<dk%d,cw%d,%s>", dk, cw, names[mode]);
    int st_ = HLA_ERR_UNSUPPORTED;
    if (dk == 128) {
        st_ = mode == kDecode ? launch_dk<128, kDecode>(cw, p, st)
            : mode == kVerify ? launch_dk<128, kVerify>(cw, p, st)
            : mode == kReplay ? launch_dk<128, kReplay>(cw, p, st)
            : mode == kReplayVerify ? launch_dk<128, kReplayVerify>(cw, p, st)
                                    : launch_dk<128, kExtend>(cw, p, st);
    } else {
        st_ = mode == kDecode ? launch_dk<64, kDecode>(cw, p, st)
            : mode == kVerify ? launch_dk<64, kVerify>(cw, p, st)
            : mode == kReplay ? launch_dk<64, kReplay>(cw, p, st)
            : mode == kReplayVerify ? launch_dk<64, kReplayVerify>(cw, p, st)
                                    : launch_dk<64, kExtend>(cw, p, st);
    }
    return st_;
}

__global__ void accept_prefix_kernel(int B, int T, const int32_t *__restrict__ draft,
                                     const int32_t *__restrict__ target, int32_t *accepted,
                                     int32_t *committed) {
    pdl_wait_trigger();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int n = 0;
    while (n < T && draft[(size_t)b * T + n] == target[(size_t)b * T + n]) ++n;
    accepted[b] = n;
    committed[b] += n;
}

}  // namespace

// The decode layer's KDA step: its stream predecessor is the input projection's epilogue, which
// does not write the state, so the state slice is loaded before waiting for it.
int kda_decode_step_in_layer(int B, int H, int dk, float *S, const int32_t *state_idx, const hla_bf16 *q,
                             const hla_bf16 *k, const hla_bf16 *v, const float *alpha, const float *beta,
                             void *o, int o_dtype, cudaStream_t st) {
    return run_kda(kDecode, B, 1, H, dk, dk, S, state_idx, q, k, v, alpha, beta, nullptr, o, o_dtype, st,
                   PrevWindow(), nullptr, true);
}

}  // namespace hla

using namespace hla;

extern "C" int kda_decode_step(int B, int H, int dk, int dv, float *S, const int32_t *state_idx,
                               const hla_bf16 *q, const hla_bf16 *k, const hla_bf16 *v,
                               const float *alpha, const float *beta, void *o, int o_dtype,
                               hla_stream stream) {
    return run_kda(kDecode, B, 1, H, dk, dv, S, state_idx, q, k, v, alpha, beta, nullptr, o,
                   o_dtype, (cudaStream_t)stream);
}

extern "C" int kda_spec_verify_replay(int phase, int B, int T, int H, int dk, int dv, float *S,
                                      const int32_t *state_idx, const hla_bf16 *q,
                                      const hla_bf16 *k, const hla_bf16 *v, const float *alpha,
                                      const float *beta, const int32_t *accepted_len, void *o,
                                      int o_dtype, hla_stream stream) {
    if (phase == HLA_SPEC_VERIFY)
        return run_kda(kVerify, B, T, H, dk, dv, S, state_idx, q, k, v, alpha, beta, nullptr, o,
                       o_dtype, (cudaStream_t)stream);
    if (phase == HLA_SPEC_REPLAY)
        return run_kda(kReplay, B, T, H, dk, dv, S, state_idx, q, k, v, alpha, beta,
                       accepted_len, nullptr, o_dtype, (cudaStream_t)stream);
    // BOTH: a window's accepted length depends on what the target makes of that window's
    // verify outputs, so its verify and its replay cannot share one call; the one-pass
    // speculative step is kda_spec_replay_verify (previous window's replay + next verify)
    if (phase == HLA_SPEC_BOTH) return HLA_ERR_UNSUPPORTED;
    return HLA_ERR_INVALID_ARG;
}

extern "C" int kda_spec_replay_verify(int B, int T_prev, int T, int H, int dk, int dv, float *S,
                                      const int32_t *state_idx, const hla_bf16 *q_prev,
                                      const hla_bf16 *k_prev, const hla_bf16 *v_prev,
                                      const float *alpha_prev, const float *beta_prev,
                                      const int32_t *accepted_prev, const hla_bf16 *q,
                                      const hla_bf16 *k, const hla_bf16 *v, const float *alpha,
                                      const float *beta, void *o, int o_dtype, hla_stream stream) {
    PrevWindow prev;
    prev.q = q_prev; prev.k = k_prev; prev.v = v_prev; prev.alpha = alpha_prev; prev.beta = beta_prev;
    prev.T = T_prev;
    return run_kda(kReplayVerify, B, T, H, dk, dv, S, state_idx, q, k, v, alpha, beta, accepted_prev,
                   o, o_dtype, (cudaStream_t)stream, prev);
}

extern "C" int kda_extend(int B, const int32_t *cu_seqlens, int H, int dk, int dv, float *S,
                          const int32_t *state_idx, const hla_bf16 *q, const hla_bf16 *k,
                          const hla_bf16 *v, const float *alpha, const float *beta, void *o,
                          int o_dtype, hla_stream stream) {
    return run_kda(kExtend, B, 1, H, dk, dv, S, state_idx, q, k, v, alpha, beta, nullptr, o,
                   o_dtype, (cudaStream_t)stream, PrevWindow(), cu_seqlens);
}

extern "C" int spec_accept_prefix(int B, int T, const int32_t *draft_ids,
                                  const int32_t *target_ids, int32_t *accepted_len,
                                  int32_t *committed_len, hla_stream stream) {
    HLA_REQUIRE(B >= 1 && T >= 1 && T <= 64, B >= 1 && T >= 1 ? HLA_ERR_UNSUPPORTED : HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(draft_ids && target_ids && accepted_len && committed_len, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(aligned16(draft_ids) && aligned16(target_ids) && aligned16(accepted_len) &&
                    aligned16(committed_len),
                HLA_ERR_MISALIGNED);
    set_variant("accept_prefix");
    return launched(launch_kernel(accept_prefix_kernel, dim3((B + 127) / 128), dim3(128), 0,
                                  (cudaStream_t)stream, B, T, draft_ids, target_ids, accepted_len,
                                  committed_len));
}
