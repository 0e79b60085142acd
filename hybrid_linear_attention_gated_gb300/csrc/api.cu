// Status strings, variant reporting and small device queries for the C ABI.
#include <atomic>
#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <vector>

#include "common.cuh"

namespace {
thread_local char g_variant[128] = "";
int g_sm_count[64] = {0};
std::atomic<unsigned long long> g_launches{0};

struct Trace {
    int kernel = 0;
    int capacity = 0;
    int count = 0;
    std::vector<cudaEvent_t> start, stop;
} g_trace;
}  // namespace

namespace hla {

void set_variant(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_variant, sizeof(g_variant), fmt, ap);
    va_end(ap);
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void trace_before(int kernel, cudaStream_t st) {
    if (kernel == 0 || kernel != g_trace.kernel || g_trace.count >= g_trace.capacity) return;
    cudaEventRecord(g_trace.start[g_trace.count], st);
}

void trace_after(int kernel, cudaStream_t st) {
    if (kernel == 0 || kernel != g_trace.kernel || g_trace.count >= g_trace.capacity) return;
    cudaEventRecord(g_trace.stop[g_trace.count], st);
    ++g_trace.count;
}

namespace {
thread_local bool g_pdl_on = false;         // a chain is open ...
thread_local cudaStream_t g_pdl_stream = nullptr;  // ... on this stream
thread_local bool g_pdl_started = false;    // and a kernel of it has been launched
}  // namespace

PdlChain::PdlChain(cudaStream_t st, bool on)
    : prev_on(g_pdl_on), prev_started(g_pdl_started), prev_st(g_pdl_stream) {
    // inside a chain already open on this stream, the first kernel follows that chain's last
    const bool continues = g_pdl_on && g_pdl_stream == st && g_pdl_started;
    g_pdl_on = on;
    g_pdl_stream = st;
    g_pdl_started = continues;
}

PdlChain::~PdlChain() {
    const bool launched_inside = g_pdl_started;
    const bool same_stream = g_pdl_stream == prev_st;
    g_pdl_on = prev_on;
    g_pdl_stream = prev_st;
    // an outer chain on the same stream goes on after the kernels queued inside this one
    g_pdl_started = prev_started || (same_stream && launched_inside);
}

// Entry points that launch several kernels chain them up to 32 tokens.  Measured on the decode layer
// (CUDA graph of 8 calls with the prefetch stream, same box, medians of 5 interleaved repetitions,
// plain / chained): batch 1 198.3 / 194.2 us, 2 297.6 / 293.5, 8 812.6 / 809.5, 32 2094.5 / 2086.5,
// 64 2860.7 / 2871.0.  HLA_PDL=0 / 1 forces plain launches / chains.
bool pdl_default(int M) {
    const char *env = getenv("HLA_PDL");
    if (env) return env[0] == '1';
    return M <= 32;
}

bool pdl_for(cudaStream_t st) { return g_pdl_on && g_pdl_started && st == g_pdl_stream; }

// records that a kernel went out on the chain's stream (chained or not)
void pdl_launched(cudaStream_t st) {
    if (st == g_pdl_stream) g_pdl_started = true;
}

namespace {
// the chain a caller opened with hla_chain_begin (at most one per host thread)
thread_local PdlChain *g_user_chain = nullptr;
}  // namespace

int prefetch_mask() {
    const char *env = getenv("HLA_PREFETCH_MASK");
    return env ? (atoi(env) & 7) : -1;
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
    if (dev < 64 && g_sm_count[dev] > 0) return g_sm_count[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 148;
    if (dev < 64) g_sm_count[dev] = n;
    return n;
}

}  // namespace hla

extern "C" const char *hla_status_string(int status) {
    switch (status) {
        case HLA_OK: return "ok";
        case HLA_ERR_INVALID_ARG: return "invalid argument (null pointer or inconsistent size)";
        case HLA_ERR_UNSUPPORTED: return "unsupported shape";
        case HLA_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
        case HLA_ERR_WORKSPACE: return "workspace missing or too small";
        case HLA_ERR_CUDA: return "CUDA launch or runtime error";
        case HLA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        default: return "unknown status";
    }
}

extern "C" const char *hla_last_variant(void) { return g_variant; }

extern "C" int hla_version(void) { return 100; }

extern "C" int hla_chain_begin(hla_stream stream) {
    if (hla::g_user_chain) return HLA_ERR_INVALID_ARG;  // already open on this thread
    hla::g_user_chain = new hla::PdlChain((cudaStream_t)stream, true);
    return HLA_OK;
}

extern "C" int hla_chain_end(void) {
    if (!hla::g_user_chain) return HLA_ERR_INVALID_ARG;
    delete hla::g_user_chain;
    hla::g_user_chain = nullptr;
    return HLA_OK;
}

extern "C" unsigned long long hla_launch_count(void) {
    return g_launches.load(std::memory_order_relaxed);
}

extern "C" int hla_trace_enable(const char *kernel, int capacity) {
    int id = hla::kTraceNone;
    if (kernel && capacity > 0) {
        if (!strcmp(kernel, "kda")) id = hla::kTraceKda;
        else if (!strcmp(kernel, "dense")) id = hla::kTraceDense;
        else if (!strcmp(kernel, "moe_gateup")) id = hla::kTraceMoeGateup;
        else if (!strcmp(kernel, "moe_down")) id = hla::kTraceMoeDown;
        else return HLA_ERR_INVALID_ARG;
    }
    for (cudaEvent_t e : g_trace.start) cudaEventDestroy(e);
    for (cudaEvent_t e : g_trace.stop) cudaEventDestroy(e);
    g_trace.start.clear();
    g_trace.stop.clear();
    g_trace.kernel = hla::kTraceNone;
    g_trace.capacity = g_trace.count = 0;
    if (id == hla::kTraceNone) return HLA_OK;
    g_trace.start.resize(capacity);
    g_trace.stop.resize(capacity);
    for (int i = 0; i < capacity; ++i) {
        if (cudaEventCreate(&g_trace.start[i]) != cudaSuccess ||
            cudaEventCreate(&g_trace.stop[i]) != cudaSuccess) {
            g_trace.start.resize(i);
            g_trace.stop.resize(i);
            return HLA_ERR_CUDA;
        }
    }
    g_trace.kernel = id;
    g_trace.capacity = capacity;
    return HLA_OK;
}

extern "C" int hla_trace_read(float *ms_out, int max_n) {
    const int n = g_trace.count < max_n ? g_trace.count : max_n;
    for (int i = 0; i < n; ++i) {
        if (cudaEventSynchronize(g_trace.stop[i]) != cudaSuccess ||
            cudaEventElapsedTime(&ms_out[i], g_trace.start[i], g_trace.stop[i]) != cudaSuccess)
            return -HLA_ERR_CUDA;
    }
    return g_trace.count;
}
