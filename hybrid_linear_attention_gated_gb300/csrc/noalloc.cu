// skinny_proj_splitk_noalloc: the split-K projection with its scratch in a fixed device array.
//
// Some callers cannot allocate device memory at the point where they need a projection:
// a serving process that reserves its whole memory budget at start-up and forbids later
// allocations (so a request never fails for lack of a workspace mid-traffic), a plugin
// whose host application owns every device allocation, or code that runs where a
// cudaMalloc would synchronise the device.  For them this entry point keeps the split-K
// partials in a file-scope device array instead of a caller workspace.  The array is part
// of the library's device image, so every GPU that loads the library holds it until the
// process exits.
#include "common.cuh"

namespace hla {

int run_dense(int M, int N, int K, const hla_bf16 *x, const hla_bf16 *W, int split, float *part,
              void *y, int y_bf16, const hla_bf16 *residual, cudaStream_t st);
int run_splitk_reduce(const float *part, int split, int M, int N, const hla_bf16 *residual, void *y,
                      int y_bf16, cudaStream_t st);
int dense_tokens_per_tile(int M);
bool dense_tc_enabled(int M);
bool dense_xi_applies(int N, int K, int split);

namespace {

// 4 Mi floats = 16 MiB of split partials (split x M x N fp32); HLA_NOALLOC_SCRATCH_BYTES.
constexpr size_t kScratchFloats = HLA_NOALLOC_SCRATCH_BYTES / sizeof(float);
__device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

// Device address of the scratch array on the current device.  The host-side name of a
// __device__ array is not a device address, so it is asked for with the device current.
// The answer is not cached: the query is a host-side table lookup, and a cached address
// would dangle after a device reset reloads the library's device image elsewhere.  On the
// first call on a device the runtime may load that image there.
int scratch_for_current_device(float **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return HLA_ERR_CUDA;
    *out = static_cast<float *>(p);
    return HLA_OK;
}

}  // namespace
}  // namespace hla

using namespace hla;

extern "C" int skinny_proj_splitk_noalloc(int M, int N, int K, const hla_bf16 *x,
                                          const hla_bf16 *W, const hla_bf16 *residual, void *y,
                                          int y_dtype, int split, hla_stream stream) {
    HLA_REQUIRE(M >= 1 && N >= 1 && K >= 32 && split >= 0, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(M <= 256 && K % 32 == 0, HLA_ERR_UNSUPPORTED);
    HLA_REQUIRE(x && W && y, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(y_dtype == HLA_F32 || y_dtype == HLA_BF16, HLA_ERR_INVALID_ARG);
    HLA_REQUIRE(aligned16(x) && aligned16(W) && aligned16(y) && (!residual || aligned16(residual)),
                HLA_ERR_MISALIGNED);
    // the same split the workspace version picks; its partials must fit the fixed scratch
    const size_t need = skinny_proj_splitk_workspace_size(M, N, K, split);
    HLA_REQUIRE(need <= kScratchFloats * sizeof(float), HLA_ERR_WORKSPACE);
    const int s = need == 0 ? 1 : (int)(need / ((size_t)M * N * sizeof(float)));
    cudaStream_t st = (cudaStream_t)stream;
    // same variant text as skinny_proj_splitk after the prefix (which streaming kernel, which split)
    set_variant("skinny_proj_noalloc<tt%d,%ssplit%d>", dense_tokens_per_tile(M),
                !dense_tc_enabled(M) && dense_xi_applies(N, K, s) ? "xi," : "", s);
    const PdlChain chain(st, pdl_default(M));  // the projection and its split reduction
    if (s == 1) return run_dense(M, N, K, x, W, 1, nullptr, y, y_dtype == HLA_BF16, residual, st);
    float *scratch = nullptr;
    int r = scratch_for_current_device(&scratch);
    if (r != HLA_OK) return r;
    // every partial is written by pass 1 before pass 2 reads it: no clearing is needed
    r = run_dense(M, N, K, x, W, s, scratch, nullptr, 0, nullptr, st);
    if (r != HLA_OK) return r;
    return run_splitk_reduce(scratch, s, M, N, residual, y, y_dtype == HLA_BF16, st);
}
