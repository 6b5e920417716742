// common.cuh: declarations shared by the selector's CUDA translation units.
//
// Each kernel file exposes one host launcher. dflash_api.cu validates the arguments and
// then calls the launchers. Kernels report problems through a device status word whose
// address api.cu passes in. Nothing here allocates memory.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dflash {

constexpr uint32_t kStatusBadId = 0x1u;     // matches DFLASH_DEVICE_BAD_ID
constexpr uint32_t kStatusTimeout = 0x2u;   // matches DFLASH_DEVICE_TIMEOUT

// Per-device facts the launchers size their grids with.
struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int cc_major = 0;
    int cc_minor = 0;
    size_t smem_optin = 0;   // max dynamic shared memory per block (opt-in)
};

// ---------------------------------------------------------------- top-k (topk.cu)

// How the flat stream of R*S*V logits is cut among warps. Every warp takes one
// contiguous span of `span` logits (the last one may be shorter). A row split across
// several warps is merged by whichever of them finishes last.
struct TopkPlan {
    long long total = 0;      // R * S * V
    long long span = 0;       // logits per warp, a multiple of 128
    int warps = 0;            // warps with work
    int blocks = 0;           // CTAs launched
    long long rows = 0;       // R * S
    int variant = 0;          // kernel build: 0 targets 3 CTAs per SM, 1 targets 2
    size_t counter_bytes = 0; // per-row arrival counters (uint32), padded to 256 B
    size_t partial_bytes = 0; // two 32-entry partial lists (uint64) per warp
    size_t workspace_bytes() const { return counter_bytes + partial_bytes; }
};

TopkPlan topk_plan(const DeviceInfo& dev, long long rows, int V);

// The fused selector's ready queue of edge tiles (one tile per (r, p) row), in the caller's
// workspace and zeroed before every call. The top-k counts, per tile, the rows it has
// written that the tile needs (rows p - 1 and p; only row 0 at p = 0) and pushes the tile
// once they are all written; the projection counts its finished CTAs; edge CTA k waits
// (bounded) for the tile pushed k-th and for the projection. A null `slots` means no queue.
struct EdgeQueue {
    uint32_t* tile_rows = nullptr;   // [rows] rows written that each tile needs
    uint32_t* slots = nullptr;       // [rows] tile + 1 of the k-th ready tile; 0 until pushed
    uint32_t* tail = nullptr;        // tiles pushed
    uint32_t* proj_done = nullptr;   // projection CTAs finished
    int S = 0;                       // steps per request
    int proj_ctas = 0;               // projection CTAs to wait for
};

// Bytes of the queue's arrays for `rows` tiles, padded to 256 B.
size_t edge_queue_bytes(long long rows);

// The queue laid out at `base` (edge_queue_bytes(rows) bytes).
EdgeQueue edge_queue_at(void* base, long long rows, int S);

// softcap > 0 and scale != 1 apply the logits processor to the reported unary values.
// `workspace` holds the arrival counters, then `extra_clear` more bytes that are zeroed with
// them (the fused selector's queue), then the partial lists. With clear_counters false the
// caller has zeroed them. A queue with non-null slots makes the kernel push edge tiles as
// their rows are written. programmatic: launched as the programmatic dependent of the kernel
// before it on the stream (it may start once that kernel's CTAs have all started; it reads
// nothing that kernel writes).
cudaError_t launch_topk(const TopkPlan& plan, const float* logits, int V, int K,
                        int32_t* cand_ids, float* unary, void* workspace,
                        cudaStream_t stream, float softcap = 0.f, float scale = 1.f,
                        size_t extra_clear = 0, bool clear_counters = true,
                        const EdgeQueue& queue = EdgeQueue(), bool programmatic = false);

// Size of the fixed device array that dflash_topk_candidates_noalloc uses as its workspace.
constexpr size_t kStaticScratchBytes = size_t(4) << 20;

// Device address of that array on `device`, which must be the current device. The first
// call per device looks it up (cudaGetSymbolAddress); later calls return the cached value.
cudaError_t topk_static_scratch(int device, void** ptr);

// ---------------------------------------------------------------- projection (projection.cu)

// Returns cudaSuccess, or an error if the tensor maps cannot be encoded or the launch
// fails. status_word receives kStatusTimeout if a bounded pipeline wait gives up.
// beside_topk selects the build that keeps to 32 registers per thread, so that by registers
// a projection CTA fits on an SM beside three top-k CTAs (the fused selector's schedule),
// with N tiles at most 128 wide. Below a rank of 256 both take the same plan and give identical bits; at 256
// the other build runs CTA pairs with a K split, so its fp32 sums may round differently
// (both stay within the accumulation bound of the exact product).
// done_counter, if not null, is incremented by every CTA once its part of h is written and
// visible device-wide (the fused selector's edges wait for it instead of a stream join).
// projection_ctas gives the number of CTAs a launch has, for that count.
cudaError_t launch_projection(const DeviceInfo& dev, const uint16_t* hidden,
                              const uint16_t* w_proj, int M, int H, int rank,
                              uint16_t* h_out, uint32_t* status_word, cudaStream_t stream,
                              bool beside_topk = false, uint32_t* done_counter = nullptr,
                              bool programmatic = false);
int projection_ctas(const DeviceInfo& dev, int M, int H, int rank);

// ---------------------------------------------------------------- edges (edges.cu)

// after_h_producer: h is written by the kernel launched just before on `stream`, and the ids,
// unary values and anchors are ready. The edges are then launched as that kernel's
// programmatic dependent (their gathers overlap its end; they wait for it before reading h).
// queue (non-null slots): the edges take their tiles from the fused selector's ready queue;
// with `programmatic` they are launched as the top-k's programmatic dependent.
cudaError_t launch_edges(const DeviceInfo& dev, const uint16_t* pred_cb,
                         const uint16_t* succ_cb, const int32_t* cand_ids, const float* unary,
                         const uint16_t* h, const int32_t* anchors, int R, int S, int K, int V,
                         int rank, float* edges, uint32_t* status_word, cudaStream_t stream,
                         bool after_h_producer = false, const EdgeQueue& queue = EdgeQueue(),
                         bool programmatic = false);

// ---------------------------------------------------------------- LM head + top-k (lmhead.cu)

// How the candidate head from the LM head is cut. One main unit per (row unit, vocabulary
// split); a unit is one CTA on a 128-row tile, or a CTA pair on 256 rows (two 128-row tiles).
// When the main units leave SMs idle, helper units take over the tail of every split's
// vocabulary range: the main unit stops at rows_per_helper / (rows_per_helper + 1) of its
// range, and each helper walks the tails of rows_per_helper consecutive row units in turn.
// The partial lists of a row tile are merged by whichever CTA finishes last.
struct LmheadPlan {
    int pair = 0;              // 1: CTA pairs on 256-row units
    int m_units = 0;           // row units: ceil(rows / 128), or ceil(rows / 256) for pairs
    int m_tiles = 0;           // 128-row tiles: m_units, or 2 m_units for pairs
    int n_tiles = 0;           // ceil(V / 256)
    int n_splits = 0;          // vocabulary ranges per row unit
    int rows_per_helper = 0;   // row units per helper (0: no helpers)
    int helpers_per_split = 0; // ceil(m_units / rows_per_helper), or 0
    int slots = 0;             // partial lists per row tile: n_splits, doubled with helpers
    int blocks = 0;            // CTAs launched
    size_t counter_bytes = 0;  // per-row-tile arrival counters, padded to 256 B
    size_t partial_bytes = 0;  // [m_tiles][slots][32][128] uint64 lists (0 if one slot)
    size_t workspace_bytes() const { return counter_bytes + partial_bytes; }
};

LmheadPlan lmhead_plan(const DeviceInfo& dev, long long rows, int V);

cudaError_t launch_lmhead_topk(const DeviceInfo& dev, const LmheadPlan& plan, const uint16_t* hidden,
                               const uint16_t* lm_head, int M, int H, int V, int K, float softcap,
                               float scale, int32_t* cand_ids, float* unary, void* workspace,
                               uint32_t* status_word, cudaStream_t stream);

// ---------------------------------------------------------------- best path (path.cu)

constexpr int kMaxPathSteps = 256;   // steps per request the best path supports

// One warp per request: the max-sum path through E [R,S,K,K] (K <= 32, S <= kMaxPathSteps).
cudaError_t launch_best_path(const float* edges, const int32_t* cand_ids, int R, int S, int K,
                             int32_t* path, int32_t* tokens, float* score, cudaStream_t stream);

}  // namespace dflash
