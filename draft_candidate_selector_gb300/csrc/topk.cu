// topk.cu: the top-K candidates of every logit row, in one streaming pass.
//
// Method: page "vllm.models.beam.nvidia.dflash2", DFlash2BeamForCausalLM.compute_candidates
// (the selector's top-k candidate ids and their logits at each position). Candidate
// order: logit descending, then token id ascending; -0 == +0; NaN with the sign clear
// above +inf, NaN with the sign set below -inf.
//
// Design (HBM-bound: every logit is read exactly once, 4 bytes, no re-reads):
//   * The R*S*V logits form one flat stream. It is cut into equal spans, one per warp
//     of a single full wave (SMs x resident CTAs x 8 warps). Every warp moves the same
//     number of bytes, whatever V is, and no CTA waits for a second wave.
//   * A warp reads its span with 128-bit non-allocating loads, eight in flight per lane
//     (each warp instruction covers 512 contiguous bytes).
//   * The warp's running top-K is a sorted list, one entry per lane. An entry is a
//     64-bit key: an order-preserving transform of the logit bits in the high word, the
//     complemented token id in the low word. Comparing two keys as integers gives the
//     candidate order, ties included.
//   * A float compare against the K-th entry's logit filters almost every element.
//     It is conservative: NaNs and ties with the threshold value pass. Survivors are
//     inserted one at a time, with a ballot for the position and a shuffle to shift.
//   * The first group of a row is different: the list is empty, so everything would pass.
//     Each lane takes the best of its own 32 values, the warp sorts those 32 lane-bests
//     once, and they become the starting list. Its K-th entry is a valid threshold for
//     the rest of the group, so only a handful of values go through the insert path.
//   * A row split across warps: each warp writes its sorted list to the workspace and
//     bumps the row's arrival counter. The warp that arrives last merges the lists with
//     warp-wide bitonic merges and writes the row. Nobody waits, so nothing can hang.
#include "common.cuh"

#include <algorithm>
#include <mutex>

namespace dflash {
namespace {

constexpr int kThreads = 256;
constexpr int kWarpsPerBlock = kThreads / 32;
constexpr int kUnroll = 8;              // 128-bit loads per lane per group (4 KB per warp)
// Two builds of the kernel differ only in the resident CTAs per SM that the register budget
// targets. Three (80 registers) streams large problems fastest. Two (94 registers, and so
// half again as many logits per warp) wins when the problem is small enough that list
// start-up is a noticeable share of each warp's span. Timed on GB300: gemma_large
// 1137 us vs 1184 us, qwen_zipf 118 us vs 111 us.
constexpr long long kSmallProblemBytes = 2LL << 30;
constexpr long long kMinSpan = 1024;    // smallest span given to one warp
constexpr long long kShortSpan = 4096;  // spans up to this long (4 groups) are "short"
constexpr long long kSpanAlign = 128;   // spans start 512 bytes apart (on 512-byte boundaries
                                        // when the logits are 16-byte aligned)
constexpr unsigned kFull = 0xffffffffu;

// Order-preserving map from float bits to uint32: a larger float gives a larger key.
// -0 is folded onto +0, and the NaNs of each sign are folded onto one key just outside
// the infinities.
__device__ __forceinline__ uint32_t order_key(uint32_t bits) {
    bits = (bits == 0x80000000u) ? 0u : bits;
    uint32_t k = bits ^ ((uint32_t)((int32_t)bits >> 31) | 0x80000000u);
    return min(max(k, 0x007FFFFEu), 0xFF800001u);
}

// Inverse of order_key (up to the folding of -0 and NaN payloads).
__device__ __forceinline__ float key_value(uint32_t key) {
    uint32_t bits = (key & 0x80000000u) ? (key ^ 0x80000000u) : ~key;
    return __uint_as_float(bits);
}

__device__ __forceinline__ uint64_t make_entry(float v, uint32_t id) {
    return ((uint64_t)order_key(__float_as_uint(v)) << 32) | (uint32_t)(~id);
}

__device__ __forceinline__ uint64_t shfl64(uint64_t v, int src) {
    uint32_t lo = __shfl_sync(kFull, (uint32_t)v, src);
    uint32_t hi = __shfl_sync(kFull, (uint32_t)(v >> 32), src);
    return ((uint64_t)hi << 32) | lo;
}

__device__ __forceinline__ uint64_t shfl_up64(uint64_t v, int d) {
    uint32_t lo = __shfl_up_sync(kFull, (uint32_t)v, d);
    uint32_t hi = __shfl_up_sync(kFull, (uint32_t)(v >> 32), d);
    return ((uint64_t)hi << 32) | lo;
}

__device__ __forceinline__ uint64_t shfl_xor64(uint64_t v, int m) {
    uint32_t lo = __shfl_xor_sync(kFull, (uint32_t)v, m);
    uint32_t hi = __shfl_xor_sync(kFull, (uint32_t)(v >> 32), m);
    return ((uint64_t)hi << 32) | lo;
}

// Streaming 128-bit load: read-only path, no L1 allocation, 256-byte L2 prefetch.
__device__ __forceinline__ float4 ld_stream(const float4* p) {
    float4 v;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.f32 {%0, %1, %2, %3}, [%4];"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(p));
    return v;
}

// A warp's running top list: lane i holds the entry of rank i (lane 0 is the best).
// Lanes at or past K hold leftovers that are never reported.
struct WarpList {
    uint64_t e;       // this lane's entry
    uint64_t thr;     // entry of rank K-1: a newcomer must beat it
    float thr_f;      // logit of that entry, for the float pre-filter
};

__device__ __forceinline__ void list_reset(WarpList& L) {
    L.e = 0;                               // sentinel: below every real entry
    L.thr = 0;
    L.thr_f = __uint_as_float(0xFFFFFFFFu);   // NaN: the pre-filter passes everything
}

// Insert c (uniform across the warp, known to beat L.thr) at its rank.
__device__ __forceinline__ void list_insert(WarpList& L, uint64_t c, int lane, int K) {
    const int pos = __popc(__ballot_sync(kFull, L.e > c));
    const uint64_t up = shfl_up64(L.e, 1);
    if (lane == pos) L.e = c;
    else if (lane > pos) L.e = up;
    L.thr = shfl64(L.e, K - 1);
    L.thr_f = key_value((uint32_t)(L.thr >> 32));
}

// The 32 best of two sorted 32-lists: a bitonic merge across the warp.
__device__ __forceinline__ uint64_t merge_lists(uint64_t a, uint64_t b, int lane) {
    const uint64_t br = shfl64(b, 31 - lane);
    uint64_t m = a > br ? a : br;             // bitonic, and holds the 32 best
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const uint64_t o = shfl_xor64(m, s);
        const bool lower = (lane & s) == 0;
        m = lower ? (m > o ? m : o) : (m < o ? m : o);
    }
    return m;
}

// Offer every lane's candidate entry to the list, lowest lane first.
__device__ __forceinline__ void list_offer(WarpList& L, uint64_t c, bool valid, int lane, int K) {
    unsigned m = __ballot_sync(kFull, valid && c > L.thr);
    while (m) {
        const int src = __ffs(m) - 1;
        m &= m - 1;
        const uint64_t x = shfl64(c, src);
        if (x > L.thr) list_insert(L, x, lane, K);
    }
}

// Sort one entry per lane across the warp, best first (a bitonic sorting network). It runs
// once per row segment, from one call site.
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const uint64_t o = shfl_xor64(v, j);
            const bool take_max = ((lane & j) == 0) == ((lane & k) == 0);
            v = take_max ? (v > o ? v : o) : (v < o ? v : o);
        }
    }
    return v;
}

// Conservative float pre-filter: false only if all four values surely lose to t.
__device__ __forceinline__ bool may_enter(const float4& v, float t) {
    return !(v.x < t) | !(v.y < t) | !(v.z < t) | !(v.w < t);
}

__device__ __forceinline__ void offer4(WarpList& L, const float4& v, uint32_t col, bool valid,
                                       int lane, int K) {
    list_offer(L, make_entry(v.x, col + 0), valid, lane, K);
    list_offer(L, make_entry(v.y, col + 1), valid, lane, K);
    list_offer(L, make_entry(v.z, col + 2), valid, lane, K);
    list_offer(L, make_entry(v.w, col + 3), valid, lane, K);
}

// The logits processor's options applied to a selected logit: scale * cap * tanh(x / cap),
// or scale * x when cap == 0. Selection and order use the raw logits (the map is
// increasing), so this touches only the K reported values.
__device__ __forceinline__ float processed(float x, float softcap, float scale) {
    if (softcap > 0.f) x = softcap * tanhf(x / softcap);
    return x * scale;
}

__device__ __forceinline__ void write_row(uint64_t e, long long row, int lane, int K,
                                          float softcap, float scale,
                                          int32_t* __restrict__ cand_ids,
                                          float* __restrict__ unary) {
    if (lane < K) {
        cand_ids[row * K + lane] = (int32_t)(~(uint32_t)e);
        unary[row * K + lane] = processed(key_value((uint32_t)(e >> 32)), softcap, scale);
    }
}

// The fused selector's ready queue: tile t (row t's edge scores) is pushed once the rows it
// needs are written.
__device__ __forceinline__ void enqueue_tile(const EdgeQueue& q, int t) {
    const unsigned k = atomicAdd(q.tail, 1u);
    atomicExch(q.slots + k, (unsigned)t + 1u);
}

// Row `row` is written: count it for the two tiles that need it (tile row, which also needs
// row - 1 unless it is a request's first step, and tile row + 1, unless row is the request's
// last step) and push each tile whose rows are now all written. Every lane's writes of the
// row are made visible device-wide before the counts.
__device__ __forceinline__ void push_ready(const EdgeQueue& q, long long row, int lane) {
    if (q.slots == nullptr) return;
    __threadfence();
    __syncwarp();
    if (lane == 0) {
        const int p = (int)(row % q.S);
        if (atomicAdd(q.tile_rows + row, 1u) + 1u == (p == 0 ? 1u : 2u)) enqueue_tile(q, (int)row);
        if (p + 1 < q.S && atomicAdd(q.tile_rows + row + 1, 1u) + 1u == 2u)
            enqueue_tile(q, (int)row + 1);
    }
    __syncwarp();
}

// First group of a row segment, with the list still empty. The lane-bests, sorted, start
// the list: they are K or more real entries, so the K-th of them is a valid threshold.
// The group is then read again (it is in L2 by now) and its other values are offered;
// each lane's best is already in. Not holding the group in registers across the sort keeps
// the kernel within its register budget.
template <int U>
__device__ __forceinline__ void first_group(WarpList& L, const float4* __restrict__ p,
                                            uint32_t col0, int lane, int K) {
    uint64_t best = 0;
    int best_slot = -1;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const float4 v = ld_stream(p + u * 32 + lane);
        const uint32_t col = col0 + (uint32_t)((u * 32 + lane) * 4);
        uint64_t e = make_entry(v.x, col + 0);
        if (e > best) { best = e; best_slot = u * 4 + 0; }
        e = make_entry(v.y, col + 1);
        if (e > best) { best = e; best_slot = u * 4 + 1; }
        e = make_entry(v.z, col + 2);
        if (e > best) { best = e; best_slot = u * 4 + 2; }
        e = make_entry(v.w, col + 3);
        if (e > best) { best = e; best_slot = u * 4 + 3; }
    }
    // Merge, not overwrite: an unaligned row head may already have put entries in the list.
    L.e = merge_lists(L.e, warp_sort_desc(best, lane), lane);
    L.thr = shfl64(L.e, K - 1);
    L.thr_f = key_value((uint32_t)(L.thr >> 32));
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const float4 v = ld_stream(p + u * 32 + lane);
        if (__any_sync(kFull, may_enter(v, L.thr_f))) {
            const uint32_t col = col0 + (uint32_t)((u * 32 + lane) * 4);
            list_offer(L, make_entry(v.x, col + 0), best_slot != u * 4 + 0, lane, K);
            list_offer(L, make_entry(v.y, col + 1), best_slot != u * 4 + 1, lane, K);
            list_offer(L, make_entry(v.z, col + 2), best_slot != u * 4 + 2, lane, K);
            list_offer(L, make_entry(v.w, col + 3), best_slot != u * 4 + 3, lane, K);
        }
    }
}

// Check one group of U float4 per lane (row float4 index j + u*32 + lane) against the list.
template <int U>
__device__ __forceinline__ void check_group(WarpList& L, const float4 (&v)[U], uint32_t col0,
                                            int j, int lane, int K) {
    bool hit = false;
#pragma unroll
    for (int u = 0; u < U; ++u) hit |= may_enter(v[u], L.thr_f);
    if (__any_sync(kFull, hit)) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (__any_sync(kFull, may_enter(v[u], L.thr_f))) {
                const uint32_t col = col0 + (uint32_t)((j + u * 32 + lane) * 4);
                offer4(L, v[u], col, true, lane, K);
            }
        }
    }
}

// Scan logits [lo, hi) of one row, given as indices within the row (0 <= lo < hi <= V), with
// `row` pointing at the row's first logit. `mis` is that pointer's offset, in floats, from a
// 16-byte boundary (0 to 3): the 128-bit loads start where the address, not the index, is a
// multiple of 16 bytes. All indices fit 32 bits because V does.
template <int U>
__device__ __forceinline__ void scan_range(WarpList& L, const float* __restrict__ row, int lo,
                                           int hi, int lane, int K, int mis) {
    // Unaligned head (fewer than 4 logits: V not a multiple of 4, or an offset base).
    const int a4 = (int)min((long long)hi, (((long long)lo + mis + 3) & ~3LL) - mis);
    if (lo < a4) {
        const int i = lo + lane;
        const bool valid = i < a4;
        const float v = valid ? row[i] : 0.f;
        list_offer(L, make_entry(v, (uint32_t)i), valid, lane, K);
    }
    const int b4 = (int)max((long long)a4, (((long long)hi + mis) & ~3LL) - mis);
    const float4* __restrict__ p = reinterpret_cast<const float4*>(row + a4);
    const int n4 = (b4 - a4) >> 2;
    const uint32_t col0 = (uint32_t)a4;

    constexpr int kGroup = 32 * U;                   // float4s per group: U lines of 512 B
    int j = 0;
    if (kGroup <= n4 && L.thr == 0) {                // a full first group, list still empty
        first_group<U>(L, p, col0, lane, K);
        j = kGroup;
    }
    for (; j + kGroup <= n4; j += kGroup) {
        float4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = ld_stream(p + j + u * 32 + lane);
        check_group<U>(L, v, col0, j, lane, K);
    }
    for (; j < n4; j += 32) {
        const int idx = j + lane;
        const bool valid = idx < n4;
        const float4 v = valid ? ld_stream(p + idx) : make_float4(0.f, 0.f, 0.f, 0.f);
        if (__any_sync(kFull, valid && may_enter(v, L.thr_f)))
            offer4(L, v, col0 + (uint32_t)(idx * 4), valid, lane, K);
    }
    // Unaligned tail (fewer than 4 logits).
    if (b4 < hi) {
        const int i = b4 + lane;
        const bool valid = i < hi;
        const float v = valid ? row[i] : 0.f;
        list_offer(L, make_entry(v, (uint32_t)i), valid, lane, K);
    }
}

template <int kMinBlocks, int U>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
topk_kernel(const float* __restrict__ logits, long long total, long long span, int warps, int V,
            int K, float softcap, float scale, int32_t* __restrict__ cand_ids,
            float* __restrict__ unary, uint32_t* __restrict__ counters,
            uint64_t* __restrict__ partials, const EdgeQueue queue) {
    // A grid launched as this one's programmatic dependent (the fused selector's edges) may
    // start once every CTA of this grid has: it takes only the resources this grid frees, and
    // it reads nothing of this grid's output until the ready queue says it is written.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (gw >= warps) return;
    // The warp's span [gw * span, min(total, (gw + 1) * span)) is recomputed where it is
    // needed rather than kept live across the scan, which holds the register budget.
    const int mis = (int)((reinterpret_cast<uintptr_t>(logits) >> 2) & 3);
    const int r_first = (int)(((long long)gw * span) / V);
    const int r_last = (int)((min(total, (long long)gw * span + span) - 1) / V);

    for (int r = r_first; r <= r_last; ++r) {
        const long long row_base = (long long)r * V;
        int lo, hi;                              // this warp's part of row r, within the row
        {
            const long long s = (long long)gw * span;
            const long long e = min(total, s + span);
            lo = (int)(max(s, row_base) - row_base);
            hi = (int)(min(e, row_base + V) - row_base);
        }
        WarpList L;
        list_reset(L);
        scan_range<U>(L, logits + row_base, lo, hi, lane, K, (int)((mis + row_base) & 3));

        // Warps whose spans touch this row.
        const int w0 = (int)(row_base / span);
        const int w1 = (int)((row_base + V - 1) / span);
        if (w0 == w1) {
            write_row(L.e, r, lane, K, softcap, scale, cand_ids, unary);
            push_ready(queue, r, lane);
            continue;
        }
        // Only a warp's first and last rows can be shared: one slot for each.
        const int slot = (r == r_first) ? 0 : 1;
        partials[((long long)gw * 2 + slot) * 32 + lane] = L.e;
        __threadfence();
        __syncwarp();
        unsigned arrived = 0;
        if (lane == 0) arrived = atomicAdd(&counters[r], 1u);
        arrived = __shfl_sync(kFull, arrived, 0);
        if (arrived != (unsigned)(w1 - w0)) continue;   // not the last one: done
        __threadfence();
        uint64_t m = L.e;
        for (int w = w0; w <= w1; ++w) {
            if (w == gw) continue;
            const int ws = (r == (int)(((long long)w * span) / V)) ? 0 : 1;
            const uint64_t other = __ldcg(reinterpret_cast<const unsigned long long*>(partials) +
                                          ((long long)w * 2 + ws) * 32 + lane);
            m = merge_lists(m, other, lane);
        }
        write_row(m, r, lane, K, softcap, scale, cand_ids, unary);
        push_ready(queue, r, lane);
    }
}

// Resident CTAs per SM of one build of the kernel (variant 0: 3 targeted, 1: 2 targeted).
int resident_blocks_per_sm(int device, int variant) {
    static std::mutex mu;
    static int cache[64][2] = {{0}};
    std::lock_guard<std::mutex> lock(mu);
    if (device < 0 || device >= 64) return 1;
    if (cache[device][variant] == 0) {
        int n = 0;
        cudaError_t e = variant == 0
            ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, topk_kernel<3, kUnroll>, kThreads, 0)
            : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, topk_kernel<2, kUnroll>, kThreads, 0);
        if (e != cudaSuccess || n < 1) {
            (void)cudaGetLastError();
            n = 1;
        }
        cache[device][variant] = n;
    }
    return cache[device][variant];
}

// Scratch of dflash_topk_candidates_noalloc: a fixed array in device memory, loaded with
// the library, so that callers which may not allocate device memory can still run the
// top-k. It holds the per-row arrival counters and the warps' partial lists.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

}  // namespace

cudaError_t topk_static_scratch(int device, void** ptr) {
    // Host code only sees a stand-in for the array's name, so its device address is looked
    // up per device, with that device current (the caller makes it current). Only a
    // successful lookup is kept: a failed one (for example a first call made while the
    // stream is capturing) is cleared from the thread's error state and tried again on the
    // next call.
    static std::mutex mu;
    static void* addr[64] = {nullptr};
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[device]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || !p) {
            (void)cudaGetLastError();
            *ptr = nullptr;
            return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
        }
        addr[device] = p;
    }
    *ptr = addr[device];
    return cudaSuccess;
}

TopkPlan topk_plan(const DeviceInfo& dev, long long rows, int V) {
    TopkPlan p;
    p.rows = rows;
    p.total = rows * (long long)V;
    p.variant = (p.total * 4 < kSmallProblemBytes) ? 1 : 0;
    const long long max_warps = (long long)std::max(1, dev.sm_count) *
                                resident_blocks_per_sm(dev.device, p.variant) * kWarpsPerBlock;
    long long span = (p.total + max_warps - 1) / max_warps;
    span = std::max(span, kMinSpan);
    // A row split over many warps ends in a chain of merges, one L2 round trip per list, so
    // short spans keep a row to about 8 warps (small_ties: 32 -> 8 warps a row, top-k 28 -> 22
    // us). Longer spans are left alone: fewer warps would read more slowly (qwen_zipf at 16
    // requests, 55 -> 61 us with the rule applied there too).
    span = std::max(span, std::min((long long)V / 8, kShortSpan));
    span = (span + kSpanAlign - 1) / kSpanAlign * kSpanAlign;
    p.span = span;
    p.warps = (int)((p.total + span - 1) / span);
    p.blocks = (p.warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    p.counter_bytes = (size_t)((rows * 4 + 255) / 256 * 256);
    p.partial_bytes = (size_t)p.warps * 2 * 32 * sizeof(uint64_t);
    return p;
}

size_t edge_queue_bytes(long long rows) {
    return (size_t)(((2 * rows + 2) * 4 + 255) / 256 * 256);
}

EdgeQueue edge_queue_at(void* base, long long rows, int S) {
    EdgeQueue q;
    uint32_t* w = static_cast<uint32_t*>(base);
    q.tile_rows = w;
    q.slots = w + rows;
    q.tail = w + 2 * rows;
    q.proj_done = w + 2 * rows + 1;
    q.S = S;
    return q;
}

cudaError_t launch_topk(const TopkPlan& plan, const float* logits, int V, int K,
                        int32_t* cand_ids, float* unary, void* workspace, cudaStream_t stream,
                        float softcap, float scale, size_t extra_clear, bool clear_counters,
                        const EdgeQueue& queue, bool programmatic) {
    uint32_t* counters = static_cast<uint32_t*>(workspace);
    uint64_t* partials = reinterpret_cast<uint64_t*>(static_cast<char*>(workspace) +
                                                     plan.counter_bytes + extra_clear);
    if (clear_counters) {
        cudaError_t err = cudaMemsetAsync(counters, 0, plan.counter_bytes + extra_clear, stream);
        if (err != cudaSuccess) return err;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)plan.blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 1 : 0;
    if (plan.variant == 0)
        return cudaLaunchKernelEx(&cfg, topk_kernel<3, kUnroll>, logits, plan.total, plan.span,
                                  plan.warps, V, K, softcap, scale, cand_ids, unary, counters,
                                  partials, queue);
    return cudaLaunchKernelEx(&cfg, topk_kernel<2, kUnroll>, logits, plan.total, plan.span,
                              plan.warps, V, K, softcap, scale, cand_ids, unary, counters,
                              partials, queue);
}

}  // namespace dflash
