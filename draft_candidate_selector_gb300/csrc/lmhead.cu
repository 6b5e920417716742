// lmhead.cu: the candidate head straight from the LM head. The top-K of
// logits = hidden . lm_head^T is taken without writing the logits anywhere.
//
// Method: page "vllm.models.beam.nvidia.dflash2", DFlash2BeamForCausalLM.compute_candidates:
// get_top_k_tokens(lm_head, hidden, top_k) yields the selector's top-k candidate ids and their
// logits at each position. The candidate order and the logits processor's options are those
// of the logits top-k (topk.cu). The logits are fp32 sums of bf16 products, taken by the
// tensor cores.
//
// GEMM view: logits[M = R*S, N = V] = hidden[M, H] . lm_head[V, H]^T, both operands
// K-major. One CTA (6 warps, one per SM) owns a 128-row tile of M and a contiguous range of
// 256-wide vocabulary tiles:
//   * warp 0, one lane: TMA producer. It streams 128x64 hidden tiles and 256x64 LM-head
//     tiles (128-byte swizzle) through a 4-stage shared-memory ring. All CTAs that share a
//     vocabulary range walk it in step, so each LM-head tile comes from HBM once and is
//     reused from L2.
//   * warp 1, one lane: MMA issuer. tcgen05.mma kind::f16 (bf16 x bf16 -> fp32),
//     M = 128, N = 256, K = 16, into one of two 256-column accumulators in tensor memory.
//     The epilogue drains one while the next tile accumulates in the other.
//   * warps 2-5: epilogue, one thread per row (tensor-memory lane). Each reads its row's
//     256 logits of the tile (tcgen05.ld, 32 columns at a time). One float compare per value
//     against the row's KC-th best so far turns the 32 values into a bit mask of survivors,
//     which is empty almost always. The thread then walks only its own survivors, so a warp
//     spends as many steps as its busiest row has survivors. Each survivor goes into the
//     row's sorted list, held in registers (KC = 8, 16 or 32 entries, the smallest that holds
//     K) and updated by a branch-free network of min/max steps.
// Where no helpers are needed and the rows fill 256-row units well, the CTAs work in pairs
// (cluster of 2, tcgen05.mma.cta_group::2, M = 256): each CTA stages its own 128 hidden rows
// and half of the LM-head tile, the even CTA issues the MMAs for both, and each CTA's
// epilogue reads its own rows from its own tensor memory. Per K block a pair stages 64 KB
// (32 KB per SM) where two single CTAs stage 96 KB, for the same MMA work.
// When the main CTAs (row tiles x splits) leave SMs idle, helper CTAs fill them: every main
// CTA stops early in its vocabulary range, and each helper takes the remaining tails of a few
// consecutive row tiles, one after the other. The helpers of a split walk the same vocabulary
// tiles at the same time, as the main CTAs do, so L2 still serves each LM-head tile to many.
// When a CTA has finished a row tile's range, it writes its lists to the workspace. The CTA
// of a row tile that arrives last merges all of them and writes the K candidates. Nobody
// waits on another CTA. Every mbarrier wait is bounded (about a second); on expiry the CTA sets
// kStatusTimeout and stops.
#include "common.cuh"
#include "ptx.cuh"

#include <algorithm>
#include <mutex>

namespace dflash {
namespace {

using namespace ptx;

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;                       // bf16 elements per 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kThreads = 192;                // producer, MMA, 4 epilogue warps
constexpr int kMaxK = 32;
constexpr uint32_t kATile = BM * BK * 2;     // 16 KB
constexpr uint32_t kBTile = BN * BK * 2;     // 32 KB
constexpr uint32_t kTmemCols = 2 * BN;       // two accumulators
constexpr int kMinHelperTiles = 8;           // vocabulary tiles per split before helpers pay
constexpr int kMaxHelperRows = 16;           // row tiles per helper, at most

__device__ __forceinline__ uint32_t order_key(uint32_t bits) {
    bits = (bits == 0x80000000u) ? 0u : bits;
    uint32_t k = bits ^ ((uint32_t)((int32_t)bits >> 31) | 0x80000000u);
    return min(max(k, 0x007FFFFEu), 0xFF800001u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
    uint32_t bits = (key & 0x80000000u) ? (key ^ 0x80000000u) : ~key;
    return __uint_as_float(bits);
}

__device__ __forceinline__ float processed(float x, float softcap, float scale) {
    if (softcap > 0.f) x = softcap * tanhf(x / softcap);
    return x * scale;
}

struct LmSmem {
    uint32_t a, b, bars, slot, flag, total;
};

__host__ __device__ inline LmSmem lm_smem_layout() {
    LmSmem L;
    L.a = 0;                                             // kStages x 16 KB
    L.b = L.a + kStages * kATile;                        // kStages x 32 KB
    L.bars = L.b + kStages * kBTile;                     // full, empty, tfull[2], tempty[2]
    L.slot = L.bars + (2 * kStages + 4) * 8;             // tensor-memory base address
    L.flag = L.slot + 8;                                 // "this CTA merges" flag
    L.total = L.flag + 8;
    return L;
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
                 : "memory");
}

__device__ __forceinline__ uint64_t max64(uint64_t a, uint64_t b) { return a > b ? a : b; }
__device__ __forceinline__ uint64_t min64(uint64_t a, uint64_t b) { return a < b ? a : b; }

// Insert c into the descending register list l, keeping its KC largest entries. Slot i takes
// max(l[i], min(l[i-1], c)), all from the old values: the slots above c keep their entries,
// c lands in its place and the rest move down by one. Fully unrolled, so l stays in
// registers; no branches.
template <int KC>
__device__ __forceinline__ void reg_insert(uint64_t (&l)[KC], uint64_t c) {
#pragma unroll
    for (int i = KC - 1; i > 0; --i) l[i] = max64(l[i], min64(l[i - 1], c));
    l[0] = max64(l[0], c);
}

// v[j] for a run-time j: a tree of selects on the bits of j (indexing a register array with
// a run-time index would move it to local memory).
__device__ __forceinline__ uint32_t pick32(const uint32_t (&v)[32], int j) {
    uint32_t a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) a[i] = (j & 1) ? v[2 * i + 1] : v[2 * i];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = (j & 2) ? a[2 * i + 1] : a[2 * i];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = (j & 4) ? a[2 * i + 1] : a[2 * i];
#pragma unroll
    for (int i = 0; i < 2; ++i) a[i] = (j & 8) ? a[2 * i + 1] : a[2 * i];
    return (j & 16) ? a[1] : a[0];
}

// The work of one CTA: n_seg row tiles (segments) from m_first on, each over the vocabulary
// tiles [n_begin, n_begin + T). A main CTA has one segment, the head of its split's range. A
// helper has the tails of the same split for rows_per_helper consecutive row tiles.
struct Work {
    int m_first, n_seg, n_begin, T, slots, slot;
};

__device__ __forceinline__ Work work_of(int w, int m_tiles, int n_tiles, int n_splits,
                                        int rows_per_helper, int helpers_per_split) {
    Work k;
    const int mains = m_tiles * n_splits;
    const bool helper = w >= mains;
    int split;
    if (!helper) {
        k.m_first = w / n_splits;
        split = w % n_splits;
        k.n_seg = 1;
    } else {
        const int hb = w - mains;
        split = hb / helpers_per_split;
        k.m_first = (hb % helpers_per_split) * rows_per_helper;
        k.n_seg = min(rows_per_helper, m_tiles - k.m_first);
    }
    const int s_begin = (int)((long long)split * n_tiles / n_splits);
    const int s_end = (int)((long long)(split + 1) * n_tiles / n_splits);
    const int cut = rows_per_helper > 0
                        ? s_begin + (s_end - s_begin) * rows_per_helper / (rows_per_helper + 1)
                        : s_end;
    k.n_begin = helper ? cut : s_begin;
    k.T = helper ? s_end - cut : cut - s_begin;
    k.slots = rows_per_helper > 0 ? 2 * n_splits : n_splits;
    k.slot = helper ? n_splits + split : split;    // this CTA's partial-list slot
    return k;
}

// One accumulator tile into this thread's row list: the row's 256 logits of the tile are
// read from tensor memory at taddr, 32 columns at a time; ids are n0 + column.
template <int KC>
__device__ __forceinline__ void scan_tile(uint32_t taddr, uint32_t n0, int V, uint64_t (&lst)[KC],
                                          float& thr_f) {
    for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        __syncwarp();
        tmem_ld_32x32b_x32(taddr + (uint32_t)c0, v);
        // A value equal to the threshold cannot enter: ids arrive in ascending order, so it
        // ties with the KC-th entry and loses on the id. NaN passes (exact order in the key),
        // and so does everything while the list has free slots.
        uint32_t pass = 0;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            pass |= (__uint_as_float(v[j]) <= thr_f ? 0u : 1u) << j;
        const uint32_t id0 = n0 + (uint32_t)c0;
        if (id0 + 32u > (uint32_t)V)                 // the zero-filled tail past V
            pass &= (id0 >= (uint32_t)V) ? 0u : ((1u << ((uint32_t)V - id0)) - 1u);
        while (pass) {
            const int j = __ffs(pass) - 1;
            pass &= pass - 1;
            const uint64_t e = ((uint64_t)order_key(pick32(v, j)) << 32) |
                               (uint32_t)(~(id0 + (uint32_t)j));
            if (e > lst[KC - 1]) reg_insert(lst, e);
        }
        thr_f = key_value((uint32_t)(lst[KC - 1] >> 32));
    }
}

// A segment's row lists (one per epilogue thread, 128 rows of 128-row tile m_tile) ->
// final candidates, or a partial list in the workspace, merged by the last CTA of the row
// tile to arrive. Every CTA's own top K holds all of the row's top K that fall in its range,
// so the merge of the partial top-K lists is exact. Called by all four epilogue
// warps together: the named barriers run in every epilogue thread for every segment, even
// after a timeout, so no thread is left waiting at one. A CTA that timed out still arrives;
// its lists are then wrong, and the status word says so.
template <int KC>
__device__ __forceinline__ void finish_segment(uint64_t (&lst)[KC], bool ok, int m_tile,
                                               int slots, int slot, int t_row, int M, int K,
                                               float softcap, float scale, int* merge_flag,
                                               int32_t* __restrict__ cand_ids,
                                               float* __restrict__ unary,
                                               uint32_t* __restrict__ counters,
                                               uint64_t* __restrict__ partials) {
    const long long row = (long long)m_tile * BM + t_row;
    bool write_final = ok && slots == 1;
    if (slots > 1) {
        uint64_t* mine = partials + ((long long)m_tile * slots + slot) * kMaxK * BM;
#pragma unroll
        for (int k = 0; k < KC; ++k)
            if (k < K) mine[k * BM + t_row] = lst[k];
        __threadfence();
        asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps
        if (t_row == 0) {
            const unsigned arrived = atomicAdd(&counters[m_tile], 1u);
            *merge_flag = (arrived == (unsigned)(slots - 1)) ? 1 : 0;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (*merge_flag) {
            __threadfence();
            for (int sp = 0; sp < slots; ++sp) {
                if (sp == slot) continue;
                const unsigned long long* other = reinterpret_cast<const unsigned long long*>(
                    partials + ((long long)m_tile * slots + sp) * kMaxK * BM);
                for (int k = 0; k < K; ++k) {
                    const uint64_t e = __ldcg(other + k * BM + t_row);
                    if (e > lst[KC - 1]) reg_insert(lst, e);
                }
            }
            write_final = true;
        }
    }
    if (write_final && row < M) {
#pragma unroll
        for (int k = 0; k < KC; ++k) {
            if (k < K) {
                const uint64_t e = lst[k];
                cand_ids[row * K + k] = (int32_t)(~(uint32_t)e);
                unary[row * K + k] = processed(key_value((uint32_t)(e >> 32)), softcap, scale);
            }
        }
    }
}

template <int KC, bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
lmhead_topk_kernel(const __grid_constant__ CUtensorMap map_a,
                   const __grid_constant__ CUtensorMap map_b, int M, int H, int V, int K,
                   int m_units, int n_tiles, int n_splits, int rows_per_helper,
                   int helpers_per_split, float softcap, float scale,
                   int32_t* __restrict__ cand_ids, float* __restrict__ unary,
                   uint32_t* __restrict__ counters, uint64_t* __restrict__ partials,
                   uint32_t* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const LmSmem L = lm_smem_layout();
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    uint64_t* tfull = bars + 2 * kStages;
    uint64_t* tempty = bars + 2 * kStages + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.slot);
    int* merge_flag = reinterpret_cast<int*>(smem + L.flag);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr int kCta = kPair ? 2 : 1;
    const int crank = kPair ? (int)cluster_ctarank() : 0;
    const int pr = crank & (kCta - 1);               // CTA within the pair (0 issues the MMAs)
    const Work wk = work_of(blockIdx.x / kCta, m_units, n_tiles, n_splits, rows_per_helper,
                            helpers_per_split);
    const int m_first = wk.m_first, n_seg = wk.n_seg, n_begin = wk.n_begin, T = wk.T;
    const int num_kb = (H + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tfull[b]), 1);
            mbar_init(smem_u32(&tempty[b]), BM * kCta);  // every epilogue thread (of both CTAs)
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&map_a) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&map_b) : "memory");
        *merge_flag = 0;
    }
    if (warp == 1) {
        if constexpr (kPair) {
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "r"(kTmemCols)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "r"(kTmemCols)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (kPair) cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint16_t pair_mask = (uint16_t)(3u << (crank & ~1));

    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer
            long long g = 0;
            bool ok = true;
            for (int tt = 0; tt < n_seg * T && ok; ++tt) {
                const int m_unit = m_first + tt / T;
                const int n0 = (n_begin + tt % T) * BN;
                for (int kb = 0; kb < num_kb; ++kb, ++g) {
                    const int s = (int)(g % kStages);
                    if (g >= kStages &&
                        !mbar_wait(smem_u32(&empty[s]), (uint32_t)(((g / kStages) - 1) & 1))) {
                        atomicOr(status, kStatusTimeout);
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full[s]);
                    if constexpr (kPair) {
                        // Both CTAs' bytes count on the even CTA's barrier: its rows of A and
                        // half of the LM-head tile each.
                        const uint32_t lead = mapa(fb, (uint32_t)(crank & ~1));
                        if (pr == 0) mbar_expect_tx(fb, 2u * (kATile + kBTile / 2));
                        tma_load_2d_pair(smem_u32(smem + L.a + s * kATile), &map_a, lead, kb * BK,
                                         (m_unit * 2 + pr) * BM);
                        tma_load_2d_pair(smem_u32(smem + L.b + s * kBTile), &map_b, lead, kb * BK,
                                         n0 + pr * (BN / 2));
                    } else {
                        mbar_expect_tx(fb, kATile + kBTile);
                        tma_load_2d(smem_u32(smem + L.a + s * kATile), &map_a, fb, kb * BK, m_unit * BM);
                        tma_load_2d(smem_u32(smem + L.b + s * kBTile), &map_b, fb, kb * BK, n0);
                    }
                }
            }
            // Let the last loads land before this thread leaves the role (in a pair the even
            // CTA's barriers count both CTAs' loads; the odd CTA waits for the MMAs that read
            // its last loads).
            const long long issued = g;
            for (long long q = std::max(0LL, issued - kStages); q < issued; ++q) {
                if (pr == 0) (void)mbar_wait(smem_u32(&full[q % kStages]), (uint32_t)((q / kStages) & 1));
                else (void)mbar_wait(smem_u32(&empty[q % kStages]), (uint32_t)((q / kStages) & 1));
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && pr == 0) {
            // ---- MMA issuer (in a pair, the even CTA's, for both)
            const uint32_t idesc = f16_idesc(BM * kCta, BN);
            long long g = 0;
            bool ok = true;
            for (int tt = 0; tt < n_seg * T && ok; ++tt) {
                const int buf = tt & 1;
                if (tt >= 2 &&
                    !mbar_wait(smem_u32(&tempty[buf]), (uint32_t)(((tt >> 1) - 1) & 1))) {
                    atomicOr(status, kStatusTimeout);
                    break;
                }
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(buf * BN);
                for (int kb = 0; kb < num_kb; ++kb, ++g) {
                    const int s = (int)(g % kStages);
                    if (!mbar_wait(smem_u32(&full[s]), (uint32_t)((g / kStages) & 1))) {
                        atomicOr(status, kStatusTimeout);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(smem + L.a + s * kATile);
                    const uint32_t b0 = smem_u32(smem + L.b + s * kBTile);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        if constexpr (kPair)
                            umma_bf16_pair(acc, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32),
                                           idesc, (kb | k) != 0);
                        else
                            umma_bf16(acc, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), idesc,
                                      (kb | k) != 0);
                    }
                    if constexpr (kPair) umma_commit_pair(smem_u32(&empty[s]), pair_mask);
                    else umma_commit(smem_u32(&empty[s]));
                }
                if constexpr (kPair) umma_commit_pair(smem_u32(&tfull[buf]), pair_mask);
                else umma_commit(smem_u32(&tfull[buf]));
            }
        }
    } else {
        // ---- epilogue: thread = row (tensor-memory lane) of the tile
        const int quad = warp & 3;                       // lanes 32*quad .. 32*quad + 31
        const int t_row = quad * 32 + lane;              // 0..127
        bool ok = true;
        for (int sg = 0; sg < n_seg; ++sg) {
            uint64_t lst[KC];                            // descending; 0 is below every entry
#pragma unroll
            for (int k = 0; k < KC; ++k) lst[k] = 0;
            float thr_f = __uint_as_float(0xFFFFFFFFu);  // NaN: everything passes at first
            for (int t = 0; t < T && ok; ++t) {
                const int tt = sg * T + t;
                const int buf = tt & 1;
                const bool ready = __all_sync(
                    0xffffffffu, mbar_wait(smem_u32(&tfull[buf]), (uint32_t)((tt >> 1) & 1)));
                if (!ready) {
                    if (lane == 0) atomicOr(status, kStatusTimeout);
                    ok = false;
                    break;
                }
                tc_fence_after();
                scan_tile(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * BN),
                          (uint32_t)(n_begin + t) * BN, V, lst, thr_f);
                tc_fence_before();
                if (kPair && pr != 0)
                    mbar_arrive_remote(mapa(smem_u32(&tempty[buf]), (uint32_t)(crank & ~1)));
                else
                    mbar_arrive(smem_u32(&tempty[buf]));
            }
            finish_segment(lst, ok, (m_first + sg) * kCta + pr, wk.slots, wk.slot, t_row, M, K,
                           softcap, scale, merge_flag, cand_ids, unary, counters, partials);
        }
    }
    tc_fence_before();
    __syncthreads();
    // A pair frees its tensor memory together, once both CTAs are done with it.
    if constexpr (kPair) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (kPair)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                         "r"(kTmemCols)
                         : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                         "r"(kTmemCols)
                         : "memory");
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous), box [box_rows, 64], 128-byte swizzle.
bool encode_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
               uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace {

// The plan for units of kCta CTAs (1: 128-row tiles; 2: CTA pairs on 256-row tiles).
LmheadPlan plan_for(const DeviceInfo& dev, long long rows, int V, int kCta) {
    LmheadPlan p;
    p.pair = kCta == 2 ? 1 : 0;
    p.m_units = (int)((rows + BM * kCta - 1) / (BM * kCta));
    p.m_tiles = p.m_units * kCta;
    p.n_tiles = (V + BN - 1) / BN;
    // One wave: as many vocabulary splits as fit next to the row units on the SMs. Timed on
    // GB300, this beat every other split count tried (1 to 38), also the ones that fill all
    // SMs in two waves: with every SM on the tensor cores the clock drops under the power
    // cap, and a second wave restarts the pipelines.
    const int slots_on_chip = std::max(1, dev.sm_count / kCta);
    p.n_splits = std::max(1, std::min(p.n_tiles, slots_on_chip / std::max(1, p.m_units)));
    // Helpers for the unit slots the main units leave idle (gemma-like shapes: 60 row tiles x 2
    // splits leave 32 of 152 SMs). Only when each split is long enough to cut, and a helper's
    // row count is small enough for the cut to pay.
    const int spare = p.m_units <= slots_on_chip ? slots_on_chip - p.m_units * p.n_splits : 0;
    const int g_max = spare / p.n_splits;
    if (g_max > 0 && p.n_tiles / p.n_splits >= kMinHelperTiles) {
        const int r = (p.m_units + g_max - 1) / g_max;
        if (r <= kMaxHelperRows) {
            p.rows_per_helper = r;
            p.helpers_per_split = (p.m_units + r - 1) / r;
        }
    }
    p.slots = p.rows_per_helper > 0 ? 2 * p.n_splits : p.n_splits;
    p.blocks = kCta * (p.m_units * p.n_splits + p.n_splits * p.helpers_per_split);
    p.counter_bytes = (size_t)((p.m_tiles * 4 + 255) / 256 * 256);
    p.partial_bytes = p.slots > 1 ? (size_t)p.m_tiles * p.slots * kMaxK * BM * 8 : 0;
    return p;
}

}  // namespace

// CTA pairs stage half the LM-head bytes per SM for the same MMA work. Measured on GB300
// (same ids bit for bit): faster where no helpers are needed (qwen_zipf 0.384 -> 0.372 ms,
// gemma_softcap 4.42 -> 4.30 ms sustained), no faster where helpers take the tails of the
// vocabulary ranges (gemma_large sustained: 12.8-12.9 -> 13.3 ms on one GPU, a tie on
// another), so pairs are used only without helpers, and only when 256-row units pad the rows
// by at most an eighth.
LmheadPlan lmhead_plan(const DeviceInfo& dev, long long rows, int V) {
    const LmheadPlan single = plan_for(dev, rows, V, 1);
    if (single.rows_per_helper > 0) return single;
    const LmheadPlan pair = plan_for(dev, rows, V, 2);
    const long long padding = (long long)pair.m_units * 2 * BM - rows;
    if (pair.rows_per_helper > 0 || padding * 8 > rows) return single;
    return pair;
}

cudaError_t launch_lmhead_topk(const DeviceInfo& dev, const LmheadPlan& plan, const uint16_t* hidden,
                               const uint16_t* lm_head, int M, int H, int V, int K, float softcap,
                               float scale, int32_t* cand_ids, float* unary, void* workspace,
                               uint32_t* status_word, cudaStream_t stream) {
    static std::once_flag once[2][3][64];
    static cudaError_t attr_err[2][3][64];
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    // The register list holds KC >= K entries: the smallest build of 8, 16 or 32.
    const int kc = K <= 8 ? 0 : (K <= 16 ? 1 : 2);
    const int kp = plan.pair ? 1 : 0;
    auto kernel = kp == 0 ? (kc == 0 ? lmhead_topk_kernel<8, false>
                                     : (kc == 1 ? lmhead_topk_kernel<16, false>
                                                : lmhead_topk_kernel<32, false>))
                          : (kc == 0 ? lmhead_topk_kernel<8, true>
                                     : (kc == 1 ? lmhead_topk_kernel<16, true>
                                                : lmhead_topk_kernel<32, true>));
    const size_t smem = 1024 + lm_smem_layout().total;
    std::call_once(once[kp][kc][dev.device], [&] {
        attr_err[kp][kc][dev.device] = cudaFuncSetAttribute(
            kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (attr_err[kp][kc][dev.device] != cudaSuccess) return attr_err[kp][kc][dev.device];
    CUtensorMap map_a, map_b;
    if (!encode_2d(&map_a, hidden, (uint64_t)M, (uint64_t)H, BM) ||
        !encode_2d(&map_b, lm_head, (uint64_t)V, (uint64_t)H, plan.pair ? BN / 2 : BN))
        return cudaErrorInvalidValue;
    uint32_t* counters = static_cast<uint32_t*>(workspace);
    uint64_t* partials = reinterpret_cast<uint64_t*>(static_cast<char*>(workspace) + plan.counter_bytes);
    cudaError_t err = cudaMemsetAsync(counters, 0, plan.counter_bytes, stream);
    if (err != cudaSuccess) return err;
    if (!plan.pair) {
        kernel<<<plan.blocks, kThreads, smem, stream>>>(
            map_a, map_b, M, H, V, K, plan.m_units, plan.n_tiles, plan.n_splits,
            plan.rows_per_helper, plan.helpers_per_split, softcap, scale, cand_ids, unary,
            counters, partials, status_word);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)plan.blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, map_a, map_b, M, H, V, K, plan.m_units, plan.n_tiles,
                              plan.n_splits, plan.rows_per_helper, plan.helpers_per_split, softcap,
                              scale, cand_ids, unary, counters, partials, status_word);
}

}  // namespace dflash
