// api.cu: the extern "C" boundary of the selector library (declared in include/dflash.h).
//
// This file validates arguments on the host, finds the device facts the launchers need,
// owns the device status word, and runs the fused selector and its stage tracing. All
// arithmetic of the method lives in topk.cu, projection.cu and edges.cu.
#include "dflash.h"
#include "common.cuh"
#include "ptx.cuh"

#include <nvtx3/nvToolsExt.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

namespace {

// In the fused selector, a projection of more than this many FLOPs is launched before the
// top-k, a smaller one after it (see dflash_selector). The measured cases on either side:
// 3.8 GFLOP (gemma_softcap) and 21.1 GFLOP (gemma_large).
constexpr double kProjectionFirstFlops = 8e9;

thread_local std::string g_last_error;

dflash_status fail(dflash_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

dflash_status ok() {
    g_last_error.clear();
    return DFLASH_OK;
}

dflash_status cuda_fail(cudaError_t e, const char* what) {
    return fail(DFLASH_CUDA_ERROR, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Bits the kernels set on problems they detect; read through dflash_device_status.
__device__ uint32_t g_device_status;

// Zeroed scratch of dflash_selftest_wait_timeout's queue check (1 KB).
__device__ __align__(16) uint32_t g_selftest_buffer[256];

constexpr int kMaxDevices = 64;
struct DeviceSlot {
    dflash::DeviceInfo info;
    uint32_t* status_word = nullptr;
    bool ready = false;
};

std::mutex g_dev_mu;
DeviceSlot g_dev[kMaxDevices];

// Facts about the current device, looked up once per device.
dflash_status current_device(dflash::DeviceInfo* info, uint32_t** status_word) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return fail(DFLASH_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    }
    if (dev < 0 || dev >= kMaxDevices) return fail(DFLASH_NO_DEVICE, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceSlot& s = g_dev[dev];
    if (!s.ready) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
        if (prop.major != 10 || prop.minor != 3)
            return fail(DFLASH_NO_DEVICE,
                        "device %d is sm_%d%d; this library is built for sm_103a (GB300)", dev,
                        prop.major, prop.minor);
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_status);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
        s.info.device = dev;
        s.info.sm_count = prop.multiProcessorCount;
        s.info.cc_major = prop.major;
        s.info.cc_minor = prop.minor;
        s.info.smem_optin = prop.sharedMemPerBlockOptin;
        s.status_word = static_cast<uint32_t*>(p);
        s.ready = true;
    }
    if (info) *info = s.info;
    if (status_word) *status_word = s.status_word;
    return DFLASH_OK;
}

// ---------------------------------------------------------------- argument checks

dflash_status check_dims_topk(int R, int S, int V, int K) {
    if (R < 1 || S < 1 || V < 1 || K < 1)
        return fail(DFLASH_INVALID_ARGUMENT, "R, S, V and K must be >= 1 (got R=%d S=%d V=%d K=%d)",
                    R, S, V, K);
    if (K > V) return fail(DFLASH_INVALID_ARGUMENT, "K=%d exceeds V=%d", K, V);
    if (K > 32) return fail(DFLASH_UNSUPPORTED, "K=%d: top-k supports K <= 32", K);
    if ((long long)R * S > (1LL << 31) - 1)
        return fail(DFLASH_INVALID_ARGUMENT, "R*S=%lld rows exceeds 2^31-1", (long long)R * S);
    return DFLASH_OK;
}

dflash_status check_rank(int rank) {
    if (rank < 1) return fail(DFLASH_INVALID_ARGUMENT, "rank=%d must be >= 1", rank);
    if (rank % 8 != 0 || rank > 256)
        return fail(DFLASH_UNSUPPORTED, "rank=%d: supported ranks are multiples of 8 up to 256", rank);
    return DFLASH_OK;
}

dflash_status check_dims_projection(int R, int S, int H, int rank) {
    if (R < 1 || S < 1 || H < 1)
        return fail(DFLASH_INVALID_ARGUMENT, "R, S and H must be >= 1 (got R=%d S=%d H=%d)", R, S, H);
    if (H % 8 != 0) return fail(DFLASH_UNSUPPORTED, "H=%d: must be a multiple of 8", H);
    if ((long long)R * S > (1LL << 31) - 1)
        return fail(DFLASH_INVALID_ARGUMENT, "R*S=%lld rows exceeds 2^31-1", (long long)R * S);
    return check_rank(rank);
}

dflash_status check_dims_edges(int R, int S, int K, int V, int rank) {
    if (R < 1 || S < 1 || V < 1 || K < 1)
        return fail(DFLASH_INVALID_ARGUMENT, "R, S, V and K must be >= 1 (got R=%d S=%d V=%d K=%d)",
                    R, S, V, K);
    if (K > V) return fail(DFLASH_INVALID_ARGUMENT, "K=%d exceeds V=%d", K, V);
    if (K > 32) return fail(DFLASH_UNSUPPORTED, "K=%d: edges support K <= 32", K);
    if ((long long)R * S > (1LL << 31) - 1)
        return fail(DFLASH_INVALID_ARGUMENT, "R*S=%lld rows exceeds 2^31-1", (long long)R * S);
    return check_rank(rank);
}

dflash_status check_processor(float softcap, float scale) {
    if (!(softcap >= 0.f) || isinf(softcap))
        return fail(DFLASH_INVALID_ARGUMENT, "softcap=%g must be finite and >= 0 (0 = no cap)",
                    (double)softcap);
    if (!(scale > 0.f) || isinf(scale))
        return fail(DFLASH_INVALID_ARGUMENT, "scale=%g must be finite and > 0", (double)scale);
    return DFLASH_OK;
}

dflash_status check_ptr(const void* p, const char* name) {
    if (!p) return fail(DFLASH_INVALID_ARGUMENT, "%s is NULL", name);
    if (!aligned16(p)) return fail(DFLASH_INVALID_ARGUMENT, "%s is not 16-byte aligned", name);
    return DFLASH_OK;
}

// For the arrays that need only their natural 4-byte alignment: the anchors, candidate ids,
// unary values, edge scores and best-path outputs (read and written one element at a time,
// or staged with copies as wide as their alignment allows) and the logits (the top-k finds
// the 16-byte boundaries itself), so a slice of requests out of larger arrays stays valid.
dflash_status check_ptr4(const void* p, const char* name) {
    if (!p) return fail(DFLASH_INVALID_ARGUMENT, "%s is NULL", name);
    if ((reinterpret_cast<uintptr_t>(p) & 3u) != 0)
        return fail(DFLASH_INVALID_ARGUMENT, "%s is not 4-byte aligned", name);
    return DFLASH_OK;
}

#define DFLASH_TRY(expr)                     \
    do {                                     \
        dflash_status _s = (expr);           \
        if (_s != DFLASH_OK) return _s;      \
    } while (0)

// A named NVTX range around one library call (host side: it brackets the argument checks and
// the enqueue, and profilers attach the call's CUDA launches to it). Free when no tool is
// attached.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// ---------------------------------------------------------------- stage tracing

struct Trace {
    std::mutex mu;
    int device = -1;
    int capacity = 0;   // calls
    int used = 0;
    std::vector<cudaEvent_t> events;   // 4 per call
};
Trace g_trace;

// Event slots for the next traced call, or nullptr when tracing is off or full.
cudaEvent_t* trace_slot(int device) {
    std::lock_guard<std::mutex> lock(g_trace.mu);
    if (g_trace.capacity == 0 || g_trace.used >= g_trace.capacity || g_trace.device != device)
        return nullptr;
    return &g_trace.events[4 * (g_trace.used++)];
}

}  // namespace

extern "C" {

const char* dflash_version(void) { return "0.1.0"; }

const char* dflash_status_string(int status) {
    switch (status) {
        case DFLASH_OK: return "DFLASH_OK";
        case DFLASH_INVALID_ARGUMENT: return "DFLASH_INVALID_ARGUMENT";
        case DFLASH_UNSUPPORTED: return "DFLASH_UNSUPPORTED";
        case DFLASH_WORKSPACE_TOO_SMALL: return "DFLASH_WORKSPACE_TOO_SMALL";
        case DFLASH_CUDA_ERROR: return "DFLASH_CUDA_ERROR";
        case DFLASH_NO_DEVICE: return "DFLASH_NO_DEVICE";
        default: return "DFLASH_UNKNOWN_STATUS";
    }
}

const char* dflash_last_error(void) { return g_last_error.c_str(); }

size_t dflash_topk_workspace_bytes(int R, int S, int V, int K) {
    if (check_dims_topk(R, S, V, K) != DFLASH_OK) return 0;
    dflash::DeviceInfo dev;
    if (current_device(&dev, nullptr) != DFLASH_OK) return 0;
    return dflash::topk_plan(dev, (long long)R * S, V).workspace_bytes();
}

size_t dflash_selector_workspace_bytes(int R, int S, int V, int K) {
    if (check_dims_topk(R, S, V, K) != DFLASH_OK) return 0;
    dflash::DeviceInfo dev;
    if (current_device(&dev, nullptr) != DFLASH_OK) return 0;
    const long long rows = (long long)R * S;
    // The top-k's workspace with the edge tiles' ready queue between its counters and its
    // partial lists (zeroed together).
    return dflash::topk_plan(dev, rows, V).workspace_bytes() + dflash::edge_queue_bytes(rows);
}

dflash_status dflash_topk_candidates(const float* logits, int R, int S, int V, int K,
                                     float softcap, float scale, int32_t* cand_ids,
                                     float* unary, void* workspace, size_t workspace_bytes,
                                     dflash_stream_t stream) {
    NvtxRange range("dflash_topk_candidates");
    DFLASH_TRY(check_dims_topk(R, S, V, K));
    DFLASH_TRY(check_processor(softcap, scale));
    DFLASH_TRY(check_ptr4(logits, "logits"));
    DFLASH_TRY(check_ptr4(cand_ids, "cand_ids"));
    DFLASH_TRY(check_ptr4(unary, "unary"));
    DFLASH_TRY(check_ptr(workspace, "workspace"));
    dflash::DeviceInfo dev;
    DFLASH_TRY(current_device(&dev, nullptr));
    const dflash::TopkPlan plan = dflash::topk_plan(dev, (long long)R * S, V);
    if (workspace_bytes < plan.workspace_bytes())
        return fail(DFLASH_WORKSPACE_TOO_SMALL, "workspace of %zu bytes; %zu needed",
                    workspace_bytes, plan.workspace_bytes());
    cudaError_t e = dflash::launch_topk(plan, logits, V, K, cand_ids, unary, workspace,
                                        reinterpret_cast<cudaStream_t>(stream), softcap, scale);
    if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
    return ok();
}

dflash_status dflash_topk_candidates_noalloc(const float* logits, int R, int S, int V, int K,
                                             int32_t* cand_ids, float* unary,
                                             dflash_stream_t stream) {
    NvtxRange range("dflash_topk_candidates_noalloc");
    DFLASH_TRY(check_dims_topk(R, S, V, K));
    DFLASH_TRY(check_ptr4(logits, "logits"));
    DFLASH_TRY(check_ptr4(cand_ids, "cand_ids"));
    DFLASH_TRY(check_ptr4(unary, "unary"));
    dflash::DeviceInfo dev;
    DFLASH_TRY(current_device(&dev, nullptr));
    const dflash::TopkPlan plan = dflash::topk_plan(dev, (long long)R * S, V);
    if (plan.workspace_bytes() > dflash::kStaticScratchBytes)
        return fail(DFLASH_UNSUPPORTED,
                    "R*S=%lld rows need %zu bytes of scratch; the built-in scratch holds %zu. "
                    "Use dflash_topk_candidates with a caller-owned workspace",
                    (long long)R * S, plan.workspace_bytes(), dflash::kStaticScratchBytes);
    void* scratch = nullptr;
    cudaError_t e = dflash::topk_static_scratch(dev.device, &scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(top-k scratch)");
    // launch_topk clears the arrival counters on the stream before the kernel runs.
    e = dflash::launch_topk(plan, logits, V, K, cand_ids, unary, scratch,
                            reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
    return ok();
}

size_t dflash_lmhead_topk_workspace_bytes(int R, int S, int V, int K) {
    if (check_dims_topk(R, S, V, K) != DFLASH_OK) return 0;
    dflash::DeviceInfo dev;
    if (current_device(&dev, nullptr) != DFLASH_OK) return 0;
    return dflash::lmhead_plan(dev, (long long)R * S, V).workspace_bytes();
}

dflash_status dflash_lmhead_topk(const uint16_t* hidden, const uint16_t* lm_head, int R, int S,
                                 int H, int V, int K, float softcap, float scale,
                                 int32_t* cand_ids, float* unary, void* workspace,
                                 size_t workspace_bytes, dflash_stream_t stream) {
    NvtxRange range("dflash_lmhead_topk");
    DFLASH_TRY(check_dims_topk(R, S, V, K));
    DFLASH_TRY(check_processor(softcap, scale));
    if (H < 1) return fail(DFLASH_INVALID_ARGUMENT, "H=%d must be >= 1", H);
    if (H % 8 != 0) return fail(DFLASH_UNSUPPORTED, "H=%d: must be a multiple of 8", H);
    DFLASH_TRY(check_ptr(hidden, "hidden"));
    DFLASH_TRY(check_ptr(lm_head, "lm_head"));
    DFLASH_TRY(check_ptr4(cand_ids, "cand_ids"));
    DFLASH_TRY(check_ptr4(unary, "unary"));
    DFLASH_TRY(check_ptr(workspace, "workspace"));
    dflash::DeviceInfo dev;
    uint32_t* status = nullptr;
    DFLASH_TRY(current_device(&dev, &status));
    const dflash::LmheadPlan plan = dflash::lmhead_plan(dev, (long long)R * S, V);
    if (workspace_bytes < plan.workspace_bytes())
        return fail(DFLASH_WORKSPACE_TOO_SMALL, "workspace of %zu bytes; %zu needed",
                    workspace_bytes, plan.workspace_bytes());
    cudaError_t e = dflash::launch_lmhead_topk(dev, plan, hidden, lm_head, R * S, H, V, K, softcap,
                                               scale, cand_ids, unary, workspace, status,
                                               reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "LM-head top-k launch");
    return ok();
}

dflash_status dflash_hidden_projection(const uint16_t* hidden, const uint16_t* w_proj, int R,
                                       int S, int H, int rank, uint16_t* h_out,
                                       dflash_stream_t stream) {
    NvtxRange range("dflash_hidden_projection");
    DFLASH_TRY(check_dims_projection(R, S, H, rank));
    DFLASH_TRY(check_ptr(hidden, "hidden"));
    DFLASH_TRY(check_ptr(w_proj, "w_proj"));
    DFLASH_TRY(check_ptr(h_out, "h_out"));
    dflash::DeviceInfo dev;
    uint32_t* status = nullptr;
    DFLASH_TRY(current_device(&dev, &status));
    cudaError_t e = dflash::launch_projection(dev, hidden, w_proj, R * S, H, rank, h_out, status,
                                              reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "projection launch");
    return ok();
}

dflash_status dflash_candidate_edges(const uint16_t* pred_cb, const uint16_t* succ_cb,
                                     const int32_t* cand_ids, const float* unary,
                                     const uint16_t* h, const int32_t* anchors, int R, int S,
                                     int K, int V, int rank, float* edges,
                                     dflash_stream_t stream) {
    NvtxRange range("dflash_candidate_edges");
    DFLASH_TRY(check_dims_edges(R, S, K, V, rank));
    DFLASH_TRY(check_ptr(pred_cb, "pred_cb"));
    DFLASH_TRY(check_ptr(succ_cb, "succ_cb"));
    DFLASH_TRY(check_ptr4(cand_ids, "cand_ids"));
    DFLASH_TRY(check_ptr4(unary, "unary"));
    DFLASH_TRY(check_ptr(h, "h"));
    DFLASH_TRY(check_ptr4(anchors, "anchors"));
    DFLASH_TRY(check_ptr4(edges, "edges"));
    dflash::DeviceInfo dev;
    uint32_t* status = nullptr;
    DFLASH_TRY(current_device(&dev, &status));
    cudaError_t e = dflash::launch_edges(dev, pred_cb, succ_cb, cand_ids, unary, h, anchors, R, S,
                                         K, V, rank, edges, status,
                                         reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "edges launch");
    return ok();
}

dflash_status dflash_selector(const float* logits, const uint16_t* hidden, const uint16_t* w_proj,
                              const uint16_t* pred_cb, const uint16_t* succ_cb,
                              const int32_t* anchors, int R, int S, int K, int V, int H, int rank,
                              float softcap, float scale, int32_t* cand_ids, float* unary,
                              uint16_t* h_out, float* edges, void* workspace,
                              size_t workspace_bytes, dflash_stream_t stream) {
    NvtxRange range("dflash_selector");
    DFLASH_TRY(check_dims_topk(R, S, V, K));
    DFLASH_TRY(check_processor(softcap, scale));
    DFLASH_TRY(check_dims_projection(R, S, H, rank));
    DFLASH_TRY(check_ptr4(logits, "logits"));
    DFLASH_TRY(check_ptr(hidden, "hidden"));
    DFLASH_TRY(check_ptr(w_proj, "w_proj"));
    DFLASH_TRY(check_ptr(pred_cb, "pred_cb"));
    DFLASH_TRY(check_ptr(succ_cb, "succ_cb"));
    DFLASH_TRY(check_ptr4(anchors, "anchors"));
    DFLASH_TRY(check_ptr4(cand_ids, "cand_ids"));
    DFLASH_TRY(check_ptr4(unary, "unary"));
    DFLASH_TRY(check_ptr(h_out, "h_out"));
    DFLASH_TRY(check_ptr4(edges, "edges"));
    DFLASH_TRY(check_ptr(workspace, "workspace"));
    dflash::DeviceInfo dev;
    uint32_t* status = nullptr;
    DFLASH_TRY(current_device(&dev, &status));
    const long long rows = (long long)R * S;
    const dflash::TopkPlan plan = dflash::topk_plan(dev, rows, V);
    const size_t qbytes = dflash::edge_queue_bytes(rows);
    if (workspace_bytes < plan.workspace_bytes() + qbytes)
        return fail(DFLASH_WORKSPACE_TOO_SMALL, "workspace of %zu bytes; %zu needed",
                    workspace_bytes, plan.workspace_bytes() + qbytes);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaEvent_t* ev = trace_slot(dev.device);
    // Workspace: the top-k's arrival counters, the edge tiles' ready queue, the top-k's partial
    // lists. The counters and the queue are zeroed first.
    dflash::EdgeQueue queue =
        dflash::edge_queue_at(static_cast<char*>(workspace) + plan.counter_bytes, rows, S);
    queue.proj_ctas = dflash::projection_ctas(dev, R * S, H, rank);
    // Schedule, one stream. Each kernel is the next one's programmatic dependent: it may start
    // once every CTA of the kernel before it has started, and takes only the resources that
    // kernel leaves. The edges come last and take the SMs that top-k CTAs leave as they
    // finish, each scoring a tile once the ready queue hands it over (its rows are written)
    // and the projection's count of finished CTAs is complete: most edges run in the top-k's
    // tail. The projection comes first when it is large (more than kProjectionFirstFlops):
    // it then runs beside the top-k (an SM holding a projection CTA takes one top-k CTA at
    // once and two more when the projection CTA ends: its shared-memory configuration leaves
    // room for only one more CTA) and h is ready long before the edges need it. A smaller
    // projection comes after the top-k instead and runs on the SMs the top-k's first finished
    // CTAs leave, so every top-k CTA starts at once. Measured on GB300 (same bits either way):
    // gemma_large (21.1 GFLOP of projection) 1174-1176 us projection first against 1205 us
    // after; gemma_softcap (3.8 GFLOP) 589-590 -> 585.5-585.7 us, qwen_zipf 122.7-123.0 ->
    // 119.1-119.4 us, small_ties 28.7-28.9 -> 27.2-27.5 us, tiny 17.4-18.7 -> 17.2 us with the
    // projection after the top-k. Either way every producer a wait depends on has all its CTAs
    // resident before any edge CTA exists, so nothing can stall. A traced call
    // (dflash_trace_begin) records events between the kernels, which then run one after
    // another in the first order, so that each can be timed.
    const bool chain = ev == nullptr;
    const double proj_flops = 2.0 * (double)rows * (double)H * (double)rank;
    const bool topk_first = chain && proj_flops <= kProjectionFirstFlops;
    cudaError_t e;
    if (ev && (e = cudaEventRecord(ev[0], st)) != cudaSuccess) return cuda_fail(e, "trace event");
    if ((e = cudaMemsetAsync(workspace, 0, plan.counter_bytes + qbytes, st)) != cudaSuccess)
        return cuda_fail(e, "clearing the workspace");
    if (topk_first) {
        e = dflash::launch_topk(plan, logits, V, K, cand_ids, unary, workspace, st, softcap, scale,
                                qbytes, /*clear_counters=*/false, queue, /*programmatic=*/false);
        if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
        e = dflash::launch_projection(dev, hidden, w_proj, R * S, H, rank, h_out, status, st,
                                      /*beside_topk=*/true, queue.proj_done,
                                      /*programmatic=*/true);
        if (e != cudaSuccess) return cuda_fail(e, "projection launch");
    } else {
        e = dflash::launch_projection(dev, hidden, w_proj, R * S, H, rank, h_out, status, st,
                                      /*beside_topk=*/true, queue.proj_done);
        if (e != cudaSuccess) return cuda_fail(e, "projection launch");
        if (ev && (e = cudaEventRecord(ev[1], st)) != cudaSuccess)
            return cuda_fail(e, "trace event");
        e = dflash::launch_topk(plan, logits, V, K, cand_ids, unary, workspace, st, softcap,
                                scale, qbytes, /*clear_counters=*/false, queue,
                                /*programmatic=*/chain);
        if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
    }
    if (ev && (e = cudaEventRecord(ev[2], st)) != cudaSuccess) return cuda_fail(e, "trace event");
    e = dflash::launch_edges(dev, pred_cb, succ_cb, cand_ids, unary, h_out, anchors, R, S, K, V,
                             rank, edges, status, st, /*after_h_producer=*/false, queue,
                             /*programmatic=*/chain);
    if (e != cudaSuccess) return cuda_fail(e, "edges launch");
    if (ev && (e = cudaEventRecord(ev[3], st)) != cudaSuccess) return cuda_fail(e, "trace event");
    return ok();
}

dflash_status dflash_selector_forward(const int32_t* cand_ids, const float* unary,
                                      const uint16_t* hidden, const int32_t* anchors,
                                      const uint16_t* w_proj, const uint16_t* pred_cb,
                                      const uint16_t* succ_cb, int R, int S, int K, int V, int H,
                                      int rank, uint16_t* h_out, float* edges,
                                      dflash_stream_t stream) {
    NvtxRange range("dflash_selector_forward");
    DFLASH_TRY(check_dims_edges(R, S, K, V, rank));
    DFLASH_TRY(check_dims_projection(R, S, H, rank));
    DFLASH_TRY(check_ptr4(cand_ids, "cand_ids"));
    DFLASH_TRY(check_ptr4(unary, "unary"));
    DFLASH_TRY(check_ptr(hidden, "hidden"));
    DFLASH_TRY(check_ptr4(anchors, "anchors"));
    DFLASH_TRY(check_ptr(w_proj, "w_proj"));
    DFLASH_TRY(check_ptr(pred_cb, "pred_cb"));
    DFLASH_TRY(check_ptr(succ_cb, "succ_cb"));
    DFLASH_TRY(check_ptr(h_out, "h_out"));
    DFLASH_TRY(check_ptr4(edges, "edges"));
    dflash::DeviceInfo dev;
    uint32_t* status = nullptr;
    DFLASH_TRY(current_device(&dev, &status));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = dflash::launch_projection(dev, hidden, w_proj, R * S, H, rank, h_out, status, st);
    if (e != cudaSuccess) return cuda_fail(e, "projection launch");
    // The edges start their gathers while the projection finishes and wait for it only to
    // read h (programmatic dependent launch).
    e = dflash::launch_edges(dev, pred_cb, succ_cb, cand_ids, unary, h_out, anchors, R, S, K, V,
                             rank, edges, status, st, /*after_h_producer=*/true);
    if (e != cudaSuccess) return cuda_fail(e, "edges launch");
    return ok();
}

dflash_status dflash_best_path(const float* edges, const int32_t* cand_ids, int R, int S, int K,
                               int32_t* path, int32_t* tokens, float* score,
                               dflash_stream_t stream) {
    NvtxRange range("dflash_best_path");
    if (R < 1 || S < 1 || K < 1)
        return fail(DFLASH_INVALID_ARGUMENT, "R, S and K must be >= 1 (got R=%d S=%d K=%d)", R, S,
                    K);
    if (K > 32) return fail(DFLASH_UNSUPPORTED, "K=%d: the best path supports K <= 32", K);
    if (S > dflash::kMaxPathSteps)
        return fail(DFLASH_UNSUPPORTED, "S=%d: the best path supports S <= %d", S,
                    dflash::kMaxPathSteps);
    DFLASH_TRY(check_ptr4(edges, "edges"));
    DFLASH_TRY(check_ptr4(cand_ids, "cand_ids"));
    DFLASH_TRY(check_ptr4(path, "path"));
    DFLASH_TRY(check_ptr4(tokens, "tokens"));
    DFLASH_TRY(check_ptr4(score, "score"));
    DFLASH_TRY(current_device(nullptr, nullptr));
    cudaError_t e = dflash::launch_best_path(edges, cand_ids, R, S, K, path, tokens, score,
                                             reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "best path launch");
    return ok();
}

size_t dflash_selector_lmhead_workspace_bytes(int R, int S, int V, int K) {
    return dflash_lmhead_topk_workspace_bytes(R, S, V, K);
}

dflash_status dflash_selector_lmhead(const uint16_t* hidden, const uint16_t* lm_head,
                                     const uint16_t* w_proj, const uint16_t* pred_cb,
                                     const uint16_t* succ_cb, const int32_t* anchors, int R,
                                     int S, int K, int V, int H, int rank, float softcap,
                                     float scale, int32_t* cand_ids, float* unary,
                                     uint16_t* h_out, float* edges, void* workspace,
                                     size_t workspace_bytes, dflash_stream_t stream) {
    NvtxRange range("dflash_selector_lmhead");
    DFLASH_TRY(check_dims_topk(R, S, V, K));
    DFLASH_TRY(check_processor(softcap, scale));
    DFLASH_TRY(check_dims_projection(R, S, H, rank));
    DFLASH_TRY(check_ptr(hidden, "hidden"));
    DFLASH_TRY(check_ptr(lm_head, "lm_head"));
    DFLASH_TRY(check_ptr(w_proj, "w_proj"));
    DFLASH_TRY(check_ptr(pred_cb, "pred_cb"));
    DFLASH_TRY(check_ptr(succ_cb, "succ_cb"));
    DFLASH_TRY(check_ptr4(anchors, "anchors"));
    DFLASH_TRY(check_ptr4(cand_ids, "cand_ids"));
    DFLASH_TRY(check_ptr4(unary, "unary"));
    DFLASH_TRY(check_ptr(h_out, "h_out"));
    DFLASH_TRY(check_ptr4(edges, "edges"));
    DFLASH_TRY(check_ptr(workspace, "workspace"));
    dflash::DeviceInfo dev;
    uint32_t* status = nullptr;
    DFLASH_TRY(current_device(&dev, &status));
    const dflash::LmheadPlan plan = dflash::lmhead_plan(dev, (long long)R * S, V);
    if (workspace_bytes < plan.workspace_bytes())
        return fail(DFLASH_WORKSPACE_TOO_SMALL, "workspace of %zu bytes; %zu needed",
                    workspace_bytes, plan.workspace_bytes());
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaEvent_t* ev = trace_slot(dev.device);
    // One stream: the LM-head top-k sizes its grid to one CTA per SM, and a projection CTA
    // beside it would push one of them into a second wave.
    cudaError_t e;
    if (ev && (e = cudaEventRecord(ev[0], st)) != cudaSuccess) return cuda_fail(e, "trace event");
    e = dflash::launch_projection(dev, hidden, w_proj, R * S, H, rank, h_out, status, st);
    if (e != cudaSuccess) return cuda_fail(e, "projection launch");
    if (ev && (e = cudaEventRecord(ev[1], st)) != cudaSuccess) return cuda_fail(e, "trace event");
    e = dflash::launch_lmhead_topk(dev, plan, hidden, lm_head, R * S, H, V, K, softcap, scale,
                                   cand_ids, unary, workspace, status, st);
    if (e != cudaSuccess) return cuda_fail(e, "LM-head top-k launch");
    if (ev && (e = cudaEventRecord(ev[2], st)) != cudaSuccess) return cuda_fail(e, "trace event");
    e = dflash::launch_edges(dev, pred_cb, succ_cb, cand_ids, unary, h_out, anchors, R, S, K, V,
                             rank, edges, status, st);
    if (e != cudaSuccess) return cuda_fail(e, "edges launch");
    if (ev && (e = cudaEventRecord(ev[3], st)) != cudaSuccess) return cuda_fail(e, "trace event");
    return ok();
}

namespace {

// One thread waits on an mbarrier that nothing arrives on; the bounded wait gives up.
__global__ void wait_timeout_kernel(uint32_t* status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        const uint32_t b = dflash::ptx::smem_u32(&bar);
        dflash::ptx::mbar_init(b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!dflash::ptx::mbar_wait(b, 0)) atomicOr(status, dflash::kStatusTimeout);
    }
}

}  // namespace

dflash_status dflash_selftest_wait_timeout(void) {
    dflash::DeviceInfo dev;
    uint32_t* status = nullptr;
    DFLASH_TRY(current_device(&dev, &status));
    wait_timeout_kernel<<<1, 32>>>(status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "wait self-check launch");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "wait self-check");
    // The edge tiles' ready queue: one edge CTA waits for a tile that is never pushed. Its
    // queue and every array it is given live in a zeroed static buffer; it gives up before it
    // reads any of them and writes nothing.
    void* buf = nullptr;
    e = cudaGetSymbolAddress(&buf, g_selftest_buffer);
    if (e == cudaSuccess) e = cudaMemset(buf, 0, sizeof(g_selftest_buffer));
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return cuda_fail(e, "queue self-check buffer");
    }
    uint32_t* w = static_cast<uint32_t*>(buf);
    dflash::EdgeQueue q = dflash::edge_queue_at(w, 1, 1);
    q.proj_ctas = 1;
    const uint16_t* b16 = reinterpret_cast<const uint16_t*>(w + 64);
    e = dflash::launch_edges(dev, b16, b16, reinterpret_cast<const int32_t*>(w + 64),
                             reinterpret_cast<const float*>(w + 64), b16,
                             reinterpret_cast<const int32_t*>(w + 64), 1, 1, 1, 1, 8,
                             reinterpret_cast<float*>(w + 128), status, nullptr, false, q);
    if (e != cudaSuccess) return cuda_fail(e, "queue self-check launch");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "queue self-check");
    return ok();
}

dflash_status dflash_device_status(uint32_t* flags, int clear) {
    if (!flags) return fail(DFLASH_INVALID_ARGUMENT, "flags is NULL");
    DFLASH_TRY(current_device(nullptr, nullptr));
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    e = cudaMemcpyFromSymbol(flags, g_device_status, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e, "read status word");
    if (clear) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(uint32_t));
        if (e != cudaSuccess) return cuda_fail(e, "clear status word");
    }
    return ok();
}

dflash_status dflash_trace_begin(int n_calls) {
    if (n_calls < 1 || n_calls > (1 << 20))
        return fail(DFLASH_INVALID_ARGUMENT, "n_calls=%d must be in [1, 2^20]", n_calls);
    dflash::DeviceInfo dev;
    DFLASH_TRY(current_device(&dev, nullptr));
    std::lock_guard<std::mutex> lock(g_trace.mu);
    if (g_trace.capacity != 0) return fail(DFLASH_INVALID_ARGUMENT, "a trace is already active");
    g_trace.events.assign(4 * (size_t)n_calls, nullptr);
    for (auto& ev : g_trace.events) {
        cudaError_t e = cudaEventCreate(&ev);
        if (e != cudaSuccess) {
            for (auto& x : g_trace.events)
                if (x) cudaEventDestroy(x);
            g_trace.events.clear();
            return cuda_fail(e, "cudaEventCreate");
        }
    }
    g_trace.device = dev.device;
    g_trace.capacity = n_calls;
    g_trace.used = 0;
    return ok();
}

dflash_status dflash_trace_end(float* stage_ms, int max_calls, int* n_calls) {
    std::lock_guard<std::mutex> lock(g_trace.mu);
    if (g_trace.capacity == 0) return fail(DFLASH_INVALID_ARGUMENT, "no trace is active");
    dflash_status st = DFLASH_OK;
    const int n = g_trace.used < max_calls ? g_trace.used : (max_calls > 0 ? max_calls : 0);
    for (int i = 0; i < n && st == DFLASH_OK; ++i) {
        cudaEvent_t* ev = &g_trace.events[4 * (size_t)i];
        cudaError_t e = cudaEventSynchronize(ev[3]);
        // Events: [0] start, [1] projection done, [2] top-k done, [3] edges done; a traced
        // call runs its kernels one after another, so each stage is the time between two.
        const int from[3] = {0, 1, 2}, to[3] = {1, 2, 3};
        for (int k = 0; k < 3 && e == cudaSuccess; ++k) {
            float ms = 0.f;
            e = cudaEventElapsedTime(&ms, ev[from[k]], ev[to[k]]);
            if (stage_ms) stage_ms[3 * i + k] = ms;
        }
        if (e != cudaSuccess) st = cuda_fail(e, "reading trace events");
    }
    for (auto& ev : g_trace.events) cudaEventDestroy(ev);
    g_trace.events.clear();
    g_trace.capacity = 0;
    g_trace.used = 0;
    g_trace.device = -1;
    if (n_calls) *n_calls = n;
    return st == DFLASH_OK ? ok() : st;
}

}  // extern "C"
