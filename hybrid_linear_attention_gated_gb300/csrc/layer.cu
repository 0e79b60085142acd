// One hybrid decode layer as a chain of the library's entry points, on one stream:
//   x -> RMSNorm -> q/k/v/gate/beta projection (+ L2 norm, decay, write strength)
//     -> KDA decode step (state in place) -> output projection + residual + RMSNorm (one
//     epilogue) -> router -> routed + shared experts + residual -> y
// ("Hyper-optimizing Kimi K3 in vLLM", Part 1 secs. 1-4; "Kimi K3: From Day-0
// Availability to Optimized Inference": residual adds and normalisation around the
// projections).  The prefetch stream is passed to the MoE call, which warms the shared
// expert's rows in L2 during dispatch when several token groups will read them (Part 1
// sec. 4); warming the output-projection and router weights during the KDA step is
// available through HLA_PREFETCH_MASK.  With HLA_SHARED_STREAM=1 the shared experts are
// forked onto the prefetch stream right after the second RMSNorm, so that they overlap the
// router and dispatch (Part 1 sec. 3).  All scratch lives in the caller's workspace;
// nothing here allocates or synchronises.
#include <cstdlib>

#include "common.cuh"

namespace hla {
namespace {

struct LayerLayout {
    size_t x1, q, k, v, alpha, beta, qkvg_ws, o, oproj_ws, r, x2, idx, w, router_ws, moe_ws, total;
    size_t qkvg_bytes, oproj_bytes, router_bytes, moe_bytes;
};

bool layer_ok(const hla_layer *L) {
    return L && L->hidden >= 32 && L->heads >= 1 && L->dk >= 1 && L->dv == L->dk &&
           L->n_experts >= 1 && L->top_k >= 1 && L->inter >= 32 && L->n_shared >= 0 &&
           L->gamma_attn && L->gamma_moe && L->W_qkvgb && L->W_o && L->W_router && L->W_gate &&
           L->W_up && L->W_down &&
           (L->n_shared == 0 || (L->Ws_gate && L->Ws_up && L->Ws_down));
}

LayerLayout layer_layout(const hla_layer *L, int M) {
    LayerLayout o;
    const size_t Hd = L->hidden, H = L->heads, d = L->dk, k = L->top_k;
    size_t at = 0;
    auto take = [&](size_t bytes) {
        const size_t p = at;
        at = round_up(at + bytes, 256);
        return p;
    };
    o.qkvg_bytes = kda_qkvg_proj_workspace_size(M, L->hidden, L->heads, L->dk, L->dv, 0);
    o.oproj_bytes = skinny_proj_residual_rmsnorm_workspace_size(M, L->hidden, L->heads * L->dv, 0);
    o.router_bytes = moe_route_topk_workspace_size(M, L->hidden, L->n_experts);
    o.moe_bytes = moe_expert_forward_workspace_size(M, L->hidden, L->inter, L->n_experts,
                                                   L->top_k, L->n_shared);
    o.x1 = take(M * Hd * 2);
    o.q = take(M * H * d * 2);
    o.k = take(M * H * d * 2);
    o.v = take(M * H * d * 2);
    o.alpha = take(M * H * d * 4);
    o.beta = take(M * H * 4);
    o.qkvg_ws = take(o.qkvg_bytes);
    o.o = take(M * H * d * 2);
    o.oproj_ws = take(o.oproj_bytes);
    o.r = take(M * Hd * 2);
    o.x2 = take(M * Hd * 2);
    o.idx = take(M * k * 4);
    o.w = take(M * k * 4);
    o.router_ws = take(o.router_bytes);
    o.moe_ws = take(o.moe_bytes);
    o.total = at;
    return o;
}

// Fork/join events of the side-stream prefetch, per host thread and per device (an event
// belongs to the device that was current when it was created).
constexpr int kMaxDevices = 64;
struct ForkJoin {
    cudaEvent_t fork = nullptr, join = nullptr;
};
thread_local ForkJoin g_events[kMaxDevices];

ForkJoin *fork_join_events() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    ForkJoin &e = g_events[dev];
    if (!e.fork && cudaEventCreateWithFlags(&e.fork, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    if (!e.join && cudaEventCreateWithFlags(&e.join, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    return &e;
}

}  // namespace

bool moe_shared_on_side(int M, int nsh, bool have_side);
int kda_decode_step_in_layer(int B, int H, int dk, float *S, const int32_t *state_idx, const hla_bf16 *q,
                             const hla_bf16 *k, const hla_bf16 *v, const float *alpha, const float *beta,
                             void *o, int o_dtype, cudaStream_t st);
int moe_shared_side(int M, int Hd, int I, int E, int k, int nsh, const hla_bf16 *x,
                    const hla_bf16 *Ws_gate, const hla_bf16 *Ws_up, const hla_bf16 *Ws_down,
                    void *ws, cudaStream_t st, cudaStream_t side);
int moe_forward_checked(int M, int Hd, int I, int E, int k, int n_shared, const hla_bf16 *x,
                        const int32_t *topk_idx, const float *topk_w, const hla_bf16 *W_gate,
                        const hla_bf16 *W_up, const hla_bf16 *W_down, const hla_bf16 *Ws_gate,
                        const hla_bf16 *Ws_up, const hla_bf16 *Ws_down, const hla_bf16 *residual,
                        hla_bf16 *y, void *ws, size_t ws_bytes, cudaStream_t st, cudaStream_t pf,
                        bool shared_external);
}  // namespace hla

using namespace hla;

extern "C" size_t hla_decode_layer_workspace_size(const hla_layer *L, int M) {
    if (!layer_ok(L) || M < 1) return 0;
    return layer_layout(L, M).total;
}

extern "C" int hla_decode_layer(const hla_layer *L, int M, const hla_bf16 *x, float *S,
                                const int32_t *state_idx, hla_bf16 *y, void *ws, size_t ws_bytes,
                                hla_stream stream, hla_stream prefetch_stream) {
    HLA_REQUIRE(layer_ok(L) && M >= 1 && x && S && y, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(M <= 256, HLA_ERR_UNSUPPORTED);
    HLA_REQUIRE(x != y, HLA_ERR_INVALID_ARG);
    const LayerLayout lo = layer_layout(L, M);
    HLA_REQUIRE(ws && ws_bytes >= lo.total, HLA_ERR_WORKSPACE);
    HLA_REQUIRE(aligned16(ws), HLA_ERR_MISALIGNED);
    char *w = reinterpret_cast<char *>(ws);
    auto bf = [&](size_t off) { return reinterpret_cast<hla_bf16 *>(w + off); };
    auto f32 = [&](size_t off) { return reinterpret_cast<float *>(w + off); };
    const int Hd = L->hidden, H = L->heads, d = L->dk;
    cudaStream_t st = (cudaStream_t)stream, pf = (cudaStream_t)prefetch_stream;
    int r;

    // Every kernel on `stream` after the first is a programmatic dependent of the one before it:
    // it loads its static weights or its state while its predecessor finishes.  The first is a
    // plain launch after whatever the caller queued (or, inside a chain the caller opened, the
    // next link of that chain).  Side-stream launches stay plain.
    const PdlChain chain(st, pdl_default(M));
    if ((r = hla_rmsnorm(M, Hd, x, L->gamma_attn, L->eps, bf(lo.x1), stream)) != HLA_OK) return r;
    if ((r = kda_qkvg_proj(M, Hd, H, d, d, bf(lo.x1), L->W_qkvgb, bf(lo.q), bf(lo.k), bf(lo.v),
                           f32(lo.alpha), f32(lo.beta), 0, w + lo.qkvg_ws, lo.qkvg_bytes,
                           stream)) != HLA_OK)
        return r;
    // W_o / W_r warming during the KDA step is off unless asked for: it measured neutral at
    // batch 64 and slower at batch 1-8 (the stream flushes L2 before the o-projection).
    const int pm = prefetch_mask();
    const bool layer_pf = pf && pm >= 0 && (pm & kPrefetchLayer);
    ForkJoin *ev = nullptr;
    if (layer_pf) {
        if (!(ev = fork_join_events())) return HLA_ERR_CUDA;
        if (cudaEventRecord(ev->fork, st) != cudaSuccess || cudaStreamWaitEvent(pf, ev->fork, 0) != cudaSuccess)
            return HLA_ERR_CUDA;
        if ((r = hla_l2_prefetch(L->W_o, (size_t)Hd * H * d * 2, prefetch_stream)) != HLA_OK) return r;
        if ((r = hla_l2_prefetch(L->W_router, (size_t)L->n_experts * Hd * 2, prefetch_stream)) != HLA_OK)
            return r;
        if (cudaEventRecord(ev->join, pf) != cudaSuccess) return HLA_ERR_CUDA;
    }
    if ((r = kda_decode_step_in_layer(M, H, d, S, state_idx, bf(lo.q), bf(lo.k), bf(lo.v), f32(lo.alpha),
                                      f32(lo.beta), bf(lo.o), HLA_BF16, st)) != HLA_OK)
        return r;
    if ((r = skinny_proj_residual_rmsnorm(M, Hd, H * d, bf(lo.o), L->W_o, x, L->gamma_moe, L->eps,
                                          bf(lo.r), bf(lo.x2), 0, w + lo.oproj_ws, lo.oproj_bytes,
                                          stream)) != HLA_OK)
        return r;
    // The shared experts do not depend on the routing: when they run on the side stream they
    // start here, overlapping the router and dispatch ("Hyper-optimizing Kimi K3 in vLLM",
    // Part 1 sec. 3).
    const bool shared_side = moe_shared_on_side(M, L->n_shared, pf != nullptr);
    if (shared_side &&
        (r = moe_shared_side(M, Hd, L->inter, L->n_experts, L->top_k, L->n_shared, bf(lo.x2),
                             L->Ws_gate, L->Ws_up, L->Ws_down, w + lo.moe_ws, st, pf)) != HLA_OK)
        return r;
    if ((r = moe_route_topk(M, Hd, L->n_experts, L->top_k, bf(lo.x2), L->W_router,
                            reinterpret_cast<int32_t *>(w + lo.idx), f32(lo.w), nullptr,
                            w + lo.router_ws, lo.router_bytes, stream)) != HLA_OK)
        return r;
    if ((r = moe_forward_checked(M, Hd, L->inter, L->n_experts, L->top_k, L->n_shared, bf(lo.x2),
                                 reinterpret_cast<int32_t *>(w + lo.idx), f32(lo.w), L->W_gate,
                                 L->W_up, L->W_down, L->Ws_gate, L->Ws_up, L->Ws_down, bf(lo.r), y,
                                 w + lo.moe_ws, lo.moe_bytes, st, pf, shared_side)) != HLA_OK)
        return r;
    if (layer_pf && cudaStreamWaitEvent(st, ev->join, 0) != cudaSuccess) return HLA_ERR_CUDA;
    set_variant("decode_layer%s%s", pf ? "<prefetch>" : "", pdl_default(M) ? "<pdl>" : "");
    return HLA_OK;
}

extern "C" int hla_decode_layer_routing(const hla_layer *L, int M, const void *ws,
                                        const int32_t **topk_idx, const float **topk_w) {
    HLA_REQUIRE(layer_ok(L) && M >= 1 && ws && topk_idx && topk_w, HLA_ERR_INVALID_ARG);
    const LayerLayout lo = layer_layout(L, M);
    const char *w = reinterpret_cast<const char *>(ws);
    *topk_idx = reinterpret_cast<const int32_t *>(w + lo.idx);
    *topk_w = reinterpret_cast<const float *>(w + lo.w);
    return HLA_OK;
}
