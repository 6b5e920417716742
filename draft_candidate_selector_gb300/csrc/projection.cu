// projection.cu: h = hidden . W_proj^T on the 5th-generation tensor cores.
//
// Method: page "vllm.models.beam.nvidia.dflash2", DFlash2BeamCandidateSelector.__init__
// (hidden_projection: bias-free linear map hidden_size -> rank, params_dtype bf16) and
// forward (hidden must be bf16). Accumulation is fp32, and the output is rounded to
// bf16, nearest-even.
//
// GEMM view: D[M = R*S, N = rank] = A[M, K = H] . B[N, K]^T. A (hidden) and B (W_proj,
// Linear [out, in]) are both K-major, which is the native operand form of tcgen05.mma.
//
// Tiling. The output is cut into 128 x BN tiles, BN = the rank rounded up to 16, at most
// 256 (the widest N of one M = 128 tcgen05.mma). Wide tiles pay: measured on GB300, a CTA's
// ring (wait for a stage, four M = 128, K = 16 MMAs, commit) takes about 0.31 us per K block
// at N = 128 even with the loads taken out, while the same MMAs issued back to back take
// 0.17 us; at N = 256 the MMAs take 0.31 us, as long as the ring, so a 256-wide tile does
// about twice the work per K block.
// CTA pairs. Outside the fused selector a 256-wide tile runs on a pair of CTAs
// (tcgen05.mma.cta_group::2, M = 256): each CTA stages its own 128 rows of A and half of B's
// rows at the same shared-memory offsets, the even CTA issues the MMAs for both, and each
// CTA's tensor memory holds its 128 rows of the accumulator. The odd CTA's TMA loads count
// their bytes on the even CTA's barrier; commits arrive on both CTAs' barriers (multicast).
// A pair stages half the operand bytes per SM for the same MMA work.
// K split. A cluster of `ks` tiles' CTAs (times two for pairs) splits K: split s takes the
// contiguous K blocks [s * nkb / ks, (s + 1) * nkb / ks). The host doubles ks, from 1, while
// the CTAs still fit the SMs in one wave and every split keeps at least 8 K blocks
// (gemma_large standalone: 30 pair tiles of 256 x 256, ks = 2, clusters of 4; beside the
// top-k: 60 x 2 tiles of 128 x 128, ks = 1; gemma_softcap: 30 tiles, ks = 4; qwen_zipf: 8
// tiles, ks = 4). In each CTA:
//   * warp 0, one lane: TMA producer. Per 64-wide K block it loads a 128x64 A tile and a
//     BNx64 B tile (128-byte swizzle) into a ring of `stages` shared-memory stages (192 KB:
//     4 at BN = 256, 6 at BN = 128, up to 8). Completion is tracked on mbarriers by
//     transaction bytes.
//   * warp 1, one lane: MMA issuer (in a pair, the even CTA's only). tcgen05.mma kind::f16
//     (bf16 x bf16 -> fp32), M = 128 (256 for a pair), N = BN, K = 16, four per K block,
//     accumulating in tensor memory. tcgen05.commit frees each stage and finally signals
//     the accumulator.
//   * warps 0-3: epilogue; thread t owns row t of the tile (tensor-memory lane t).
//       ks = 1: tcgen05.ld 16 columns at a time (8 in the register-capped build), round
//       to bf16, store.
//       ks > 1: the tile's columns are cut into ks slices of BN / ks; CTA s owns slice s.
//       Once every CTA's MMAs are done (cluster barrier), each CTA writes its fp32
//       partials of the slices it does not own into the owners' shared memory
//       (distributed shared memory, over the now idle ring, in a layout where each warp
//       store covers 512 contiguous bytes), a second cluster barrier makes them visible,
//       and each owner adds the ks partials of its slice in split order (0, 1, ...), rounds
//       to bf16 and stores. The sum order is fixed, so the result does not depend on which
//       CTA owns which slice.
// Out-of-range rows, columns and K are zero-filled by TMA and never stored.
// Every mbarrier wait is bounded, about one second by %globaltimer. On expiry the kernel
// sets kStatusTimeout, skips the remaining work, still takes part in both cluster
// barriers, frees its tensor memory, and returns.
// The fused selector runs the projection beside the top-k: its build keeps to 32 registers
// per thread, so that by registers one projection CTA (128 threads) fits beside three top-k
// CTAs on an SM (65,536 registers exactly).
#include "common.cuh"
#include "ptx.cuh"

#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

namespace dflash {
namespace {

using namespace ptx;

constexpr int BM = 128;
constexpr int BK = 64;                 // bf16 elements in one 128-byte swizzle row
constexpr int kThreads = 128;
constexpr uint32_t kATileBytes = BM * BK * 2;
constexpr uint32_t kRingBudget = 192u * 1024u;   // shared memory for the stage ring
constexpr int kMaxStages = 8;
constexpr int kMaxSplit = 8;
constexpr int kMaxBN = 256;            // widest N tile: one tcgen05.mma (M = 128) takes N <= 256
constexpr int kMinKbPerSplit = 8;      // K blocks each split must keep

// Receive area of the K-split reduction. A slot holds one other CTA's fp32 partials of
// this CTA's slice as [slice / 4][BM rows][4 columns]: thread t (row t) moves 16 bytes at
// t * 16 within a 4-column group, so a warp's 32 stores or loads are 512 contiguous bytes
// and touch every bank once.
__host__ __device__ constexpr uint32_t recv_slot_bytes(int slice) { return (uint32_t)slice * BM * 4u; }
__host__ __device__ constexpr uint32_t recv_offset(int c, int row) {
    return (uint32_t)(c >> 2) * (BM * 16u) + (uint32_t)row * 16u;
}

// Two builds. kMinBlocks = 16 caps the registers at 32 per thread, so that by registers one
// projection CTA fits beside three top-k CTAs on an SM (the fused selector runs them side by
// side); kMinBlocks = 1 leaves the compiler free, for calls where nothing runs beside it.
template <int kMinBlocks, bool kPair>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
projection_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                  uint16_t* __restrict__ out, int M, int N, int Kdim, int BN, uint32_t tmem_cols,
                  int ks, int stages, uint32_t* __restrict__ status,
                  uint32_t* __restrict__ done_counter) {
    extern __shared__ uint8_t smem_raw[];
    // The 128-byte swizzle pattern repeats every 1024 B: tiles start on that boundary. Every
    // CTA has the same layout, so an offset names the same place in each CTA of a cluster.
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    // A CTA pair computes a 256 x BN tile: each CTA stages its own 128 rows of A and half of
    // B's BN rows, and holds its 128 rows of the accumulator.
    constexpr int kCta = kPair ? 2 : 1;
    const int bn_cta = BN / kCta;                // B rows this CTA stages
    const uint32_t b_tile_bytes = (uint32_t)bn_cta * BK * 2;
    uint8_t* sa = smem;
    uint8_t* sb = smem + stages * kATileBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sb + stages * b_tile_bytes);
    uint64_t* full = bars;                  // [stages] TMA landed
    uint64_t* empty = bars + stages;        // [stages] MMAs done reading
    uint64_t* accum = bars + 2 * stages;    // all MMAs done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * stages + 1);

    // A dependent grid launched with programmatic serialization (the edges of the forward
    // pass) may start now; it waits for this grid to finish before it reads h.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int crank = (ks > 1 || kPair) ? (int)cluster_ctarank() : 0;
    const int pr = kPair ? (crank & 1) : 0;      // CTA within the pair (0 issues the MMAs)
    const int split = crank / kCta;
    const int m0 = (blockIdx.x / (ks * kCta)) * (BM * kCta) + pr * BM;
    const int n0 = blockIdx.y * BN;
    const int nkb = (Kdim + BK - 1) / BK;
    const int kb0 = split * nkb / ks;
    const int n_kb = (split + 1) * nkb / ks - kb0;   // >= 1: the host keeps ks <= nkb

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(accum), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&map_a) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&map_b) : "memory");
    }
    if (warp == 1) {
        if constexpr (kPair) {
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "r"(tmem_cols)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "r"(tmem_cols)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    tc_fence_before();
    __syncthreads();
    // A pair's loads count on the even CTA's barriers and its commits arrive on both CTAs'
    // barriers: every barrier of the cluster is initialised before any of that starts.
    if constexpr (kPair) cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint16_t pair_mask = (uint16_t)(3u << (crank & ~1));

    if (warp == 0 && lane == 0) {
        // TMA producer.
        // The stage and its phase advance with the K block (no division on the way).
        int issued = 0;
        for (int i = 0, s = 0, ph = 0; i < n_kb; ++i) {
            if (i >= stages && !mbar_wait(smem_u32(&empty[s]), ph ^ 1)) {
                atomicOr(status, kStatusTimeout);
                break;
            }
            const uint32_t fb = smem_u32(&full[s]);
            if constexpr (kPair) {
                // Both CTAs' bytes count on the even CTA's barrier, which that CTA arms.
                const uint32_t lead = mapa(fb, (uint32_t)(crank & ~1));
                if (pr == 0) mbar_expect_tx(fb, 2u * (kATileBytes + b_tile_bytes));
                tma_load_2d_pair(smem_u32(sa + s * kATileBytes), &map_a, lead, (kb0 + i) * BK, m0);
                tma_load_2d_pair(smem_u32(sb + s * b_tile_bytes), &map_b, lead, (kb0 + i) * BK,
                                 n0 + pr * bn_cta);
            } else {
                mbar_expect_tx(fb, kATileBytes + b_tile_bytes);
                tma_load_2d(smem_u32(sa + s * kATileBytes), &map_a, fb, (kb0 + i) * BK, m0);
                tma_load_2d(smem_u32(sb + s * b_tile_bytes), &map_b, fb, (kb0 + i) * BK, n0);
            }
            issued = i + 1;
            if (++s == stages) {
                s = 0;
                ph ^= 1;
            }
        }
        // The last load into each stage must land before the CTA may leave, or its ring be
        // reused for the partial sums, also after a timeout. Each wait is bounded; in the
        // normal case those loads were consumed long ago and every wait returns at once.
        // In a pair the even CTA's barriers count both CTAs' loads; the odd CTA waits until
        // the MMAs that read its last loads are done.
        for (int q = issued > stages ? issued - stages : 0; q < issued; ++q) {
            if (pr == 0) (void)mbar_wait(smem_u32(&full[q % stages]), (q / stages) & 1);
            else (void)mbar_wait(smem_u32(&empty[q % stages]), (q / stages) & 1);
        }
    } else if (warp == 1 && lane == 0 && pr == 0) {
        // MMA issuer (in a pair, the even CTA's, for both).
        const uint32_t idesc = f16_idesc(BM * kCta, BN);
        for (int i = 0, s = 0, ph = 0; i < n_kb; ++i) {
            if (!mbar_wait(smem_u32(&full[s]), ph)) {
                atomicOr(status, kStatusTimeout);
                break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(sa + s * kATileBytes);
            const uint32_t b0 = smem_u32(sb + s * b_tile_bytes);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
                // Advancing 16 bf16 (32 B) along K inside the swizzled 128-byte row.
                if constexpr (kPair)
                    umma_bf16_pair(tmem, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), idesc,
                                   (i | k) != 0);
                else
                    umma_bf16(tmem, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), idesc,
                              (i | k) != 0);
            }
            if constexpr (kPair) umma_commit_pair(smem_u32(&empty[s]), pair_mask);
            else umma_commit(smem_u32(&empty[s]));
            if (++s == stages) {
                s = 0;
                ph ^= 1;
            }
        }
        // Signals once every MMA issued above has completed (also after a timeout).
        if constexpr (kPair) umma_commit_pair(smem_u32(accum), pair_mask);
        else umma_commit(smem_u32(accum));
    }
    __syncwarp();

    // Epilogue: every warp drains its 32 TMEM lanes (= 32 output rows).
    const bool ready = __all_sync(0xffffffffu, mbar_wait(smem_u32(accum), 0));
    tc_fence_after();
    if (!ready && lane == 0) atomicOr(status, kStatusTimeout);
    const int trow = warp * 32 + lane;          // row of the tile, and its tensor-memory lane
    const uint32_t tlane = tmem + ((uint32_t)(warp * 32) << 16);
    if (ks == 1) {
        if (ready) {
            // Columns past N (the rank rounded up to 16) are loaded and dropped; N % 8 == 0,
            // so each 8-column piece is all in or all out.
            const int cols = min(BN, N - n0);
            uint4* orow = reinterpret_cast<uint4*>(out + (long long)(m0 + trow) * N + n0);
            const bool live = m0 + trow < M;
            if constexpr (kMinBlocks == 1) {
                // 16 columns per tensor-memory load: one wait per 16.
                for (int c0 = 0; c0 < cols; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(tlane + (uint32_t)c0, v);
                    if (live) {
                        orow[c0 >> 3] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                                   pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
                        if (c0 + 8 < cols)
                            orow[(c0 >> 3) + 1] =
                                make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]),
                                           pack_bf16x2(v[12], v[13]), pack_bf16x2(v[14], v[15]));
                    }
                }
            } else {
                // 8 columns per load: a 16-column load does not fit in 32 registers.
                for (int c0 = 0; c0 < cols; c0 += 8) {
                    uint32_t v[8];
                    tmem_ld_32x32b_x8(tlane + (uint32_t)c0, v);
                    if (live)
                        orow[c0 >> 3] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                                   pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
                }
            }
        }
    } else {
        // Receive area of this CTA, over its ring (idle from here on): slot j holds the
        // partials of the j-th other CTA (in split order), one padded row per tile row.
        // Barrier 1: every CTA of the cluster is done with its ring.
        cluster_sync();
        const int me = split;
        const int slice = BN / ks;                   // a multiple of 16
        if (ready) {
            for (int o = 0; o < ks; ++o) {
                if (o == me) continue;
                // In owner o's receive area, sender `me` uses slot me (or me - 1).
                // The CTAs holding the same rows: cluster rank o * kCta + pr.
                const uint32_t dst = mapa(smem_u32(smem) + (uint32_t)(me < o ? me : me - 1) *
                                              recv_slot_bytes(slice) + recv_offset(0, trow),
                                          (uint32_t)(o * kCta + pr));
                if constexpr (kMinBlocks == 1) {
                    for (int c = 0; c < slice; c += 16) {
                        uint32_t v[16];
                        tmem_ld_32x32b_x16(tlane + (uint32_t)(o * slice + c), v);
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            st_cluster_v4(dst + recv_offset(c + j, 0), v[j], v[j + 1], v[j + 2],
                                          v[j + 3]);
                    }
                } else {
                    for (int c = 0; c < slice; c += 4) {
                        uint32_t v[4];
                        tmem_ld_32x32b_x4(tlane + (uint32_t)(o * slice + c), v);
                        st_cluster_v4(dst + recv_offset(c, 0), v[0], v[1], v[2], v[3]);
                    }
                }
            }
        }
        // Barrier 2: the partials written to peers are visible to them.
        cluster_sync();
        if (ready) {
            // Every lane runs the warp-wide tensor-memory loads; only rows < M are stored. The
            // sum runs in split order 0, 1, ...: acc = p0, then acc += p1, and so on, so it
            // does not depend on which CTA owns the slice.
            constexpr int kChunk = kMinBlocks == 1 ? 16 : 8;
            const int row = m0 + trow;
            for (int c = 0; c < slice; c += kChunk) {
                const int col = me * slice + c;      // within the tile
                if (n0 + col >= N) break;            // warp-uniform; N % 8 == 0
                uint32_t v[kChunk];
                if constexpr (kChunk == 16) tmem_ld_32x32b_x16(tlane + (uint32_t)col, v);
                else tmem_ld_32x32b_x8(tlane + (uint32_t)col, v);
                float acc[kChunk];
                if (me == 0) {
#pragma unroll
                    for (int j = 0; j < kChunk; ++j) acc[j] = __uint_as_float(v[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < kChunk; j += 4) {
                        const float4 a = *reinterpret_cast<const float4*>(smem + recv_offset(c + j, trow));
                        acc[j] = a.x; acc[j + 1] = a.y; acc[j + 2] = a.z; acc[j + 3] = a.w;
                    }
                }
                for (int s = 1; s < ks; ++s) {
                    if (s == me) {
#pragma unroll
                        for (int j = 0; j < kChunk; ++j) acc[j] += __uint_as_float(v[j]);
                    } else {
                        const uint8_t* slot = smem + (size_t)(s < me ? s : s - 1) * recv_slot_bytes(slice);
#pragma unroll
                        for (int j = 0; j < kChunk; j += 4) {
                            const float4 a = *reinterpret_cast<const float4*>(slot + recv_offset(c + j, trow));
                            acc[j] += a.x; acc[j + 1] += a.y; acc[j + 2] += a.z; acc[j + 3] += a.w;
                        }
                    }
                }
                if (row < M) {
                    uint4* o4 = reinterpret_cast<uint4*>(out + (long long)row * N + n0 + col);
#pragma unroll
                    for (int j = 0; j < kChunk; j += 8) {
                        // N % 8 == 0: each 8-column piece is all in or all out.
                        if (n0 + col + j < N)
                            o4[j >> 3] = make_uint4(
                                pack_bf16x2(__float_as_uint(acc[j]), __float_as_uint(acc[j + 1])),
                                pack_bf16x2(__float_as_uint(acc[j + 2]), __float_as_uint(acc[j + 3])),
                                pack_bf16x2(__float_as_uint(acc[j + 4]), __float_as_uint(acc[j + 5])),
                                pack_bf16x2(__float_as_uint(acc[j + 6]), __float_as_uint(acc[j + 7])));
                    }
                }
            }
        }
    }
    // This CTA's part of h is written: make it visible device-wide, then count the CTA (the
    // fused selector's edges wait for the count rather than for the stream).
    if (done_counter != nullptr) __threadfence();
    tc_fence_before();
    __syncthreads();
    if (done_counter != nullptr && threadIdx.x == 0) atomicAdd(done_counter, 1u);
    // A pair frees its tensor memory together, once both CTAs have drained it.
    if constexpr (kPair) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (kPair)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                         "r"(tmem_cols)
                         : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                         "r"(tmem_cols)
                         : "memory");
    }
}

// ---------------------------------------------------------------- host side

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

struct ProjPlan {
    bool pair = false;      // CTA pairs (cta_group::2): 256-row tiles over two CTAs
    int BN = 0;             // N tile: the rank rounded up to 16 (32 for pairs), at most 256
    uint32_t tmem_cols = 0; // power of two >= max(32, BN)
    int stages = 0;         // ring stages
    int ks = 1;             // K splits per tile
    int m_tiles = 0;        // row tiles (of 128 rows, or 256 for pairs)
    int n_tiles = 0;
    size_t smem = 0;        // dynamic shared memory per CTA
    int cluster() const { return ks * (pair ? 2 : 1); }
};

uint32_t recv_bytes(int BN, int ks) {
    return ks > 1 ? (uint32_t)(ks - 1) * recv_slot_bytes(BN / ks) : 0u;
}

size_t smem_bytes(int bn_cta, int stages) {
    return 1024 + (size_t)stages * (kATileBytes + (size_t)bn_cta * BK * 2) +
           (2 * stages + 1) * sizeof(uint64_t) + 16;
}

int ring_stages(int bn_cta) {
    const uint32_t stage = kATileBytes + (uint32_t)bn_cta * BK * 2;
    const int st = (int)(kRingBudget / stage);
    return st < 2 ? 2 : (st > kMaxStages ? kMaxStages : st);
}

// Largest dynamic shared memory any plan asks for (set once per device).
size_t max_smem_bytes() {
    size_t m = 0;
    for (int bn = 16; bn <= kMaxBN; bn += 16) {
        const size_t b = smem_bytes(bn, ring_stages(bn));
        m = b > m ? b : m;
    }
    return m;
}

// Whether clusters of `size` CTAs of this kernel, with smem bytes each, can be resident.
bool cluster_fits(int device, int size, bool pair, size_t smem) {
    static std::mutex mu;
    static int cache[64][2][2 * kMaxSplit + 1] = {{{0}}};   // 0 unknown, 1 fits, 2 does not
    std::lock_guard<std::mutex> lock(mu);
    if (device < 0 || device >= 64 || size > 2 * kMaxSplit) return false;
    int& c = cache[device][pair ? 1 : 0][size];
    if (c == 0) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)size;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3((unsigned)size);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        const cudaError_t e =
            pair ? cudaOccupancyMaxActiveClusters(&n, projection_kernel<1, true>, &cfg)
                 : cudaOccupancyMaxActiveClusters(&n, projection_kernel<16, false>, &cfg);
        if (e != cudaSuccess) (void)cudaGetLastError();
        c = (e == cudaSuccess && n > 0) ? 1 : 2;
    }
    return c == 1;
}

// Beside the top-k (the fused selector) the N tile stays at most 128 wide and CTAs work
// alone: measured there on GB300, 256-wide tiles split over K made the whole fused step
// slower (gemma_large 1183 -> 1195 us), although the projection alone is faster with them.
// Elsewhere a rank of 256 runs on CTA pairs, which stage half the operand bytes per SM for
// the same MMA work (gemma_large: main loop 20.3 -> 14.5 us per CTA); narrower tiles were
// no faster with pairs (qwen_zipf 13 -> 15 us).
ProjPlan projection_plan(const DeviceInfo& dev, int M, int H, int rank, bool beside_topk) {
    ProjPlan p;
    const int max_bn = beside_topk ? 128 : kMaxBN;
    p.BN = rank >= max_bn ? max_bn : ((rank + 15) / 16) * 16;
    const bool pair = !beside_topk && p.BN == kMaxBN;
    p.pair = pair;
    p.n_tiles = (rank + p.BN - 1) / p.BN;
    p.tmem_cols = 32;
    while (p.tmem_cols < (uint32_t)p.BN) p.tmem_cols <<= 1;
    const int bn_cta = pair ? p.BN / 2 : p.BN;
    p.stages = ring_stages(bn_cta);
    p.smem = smem_bytes(bn_cta, p.stages);
    const int rows = pair ? 2 * BM : BM;
    p.m_tiles = (M + rows - 1) / rows;
    const int nkb = (H + BK - 1) / BK;
    const uint32_t ring = (uint32_t)p.stages * (kATileBytes + (uint32_t)bn_cta * BK * 2);
    const int cta = pair ? 2 : 1;
    if (pair && !cluster_fits(dev.device, 2, true, p.smem))
        return projection_plan(dev, M, H, rank, true);
    // Double the split while the tiles times the splits still fit in one wave, each split
    // keeps enough K blocks to run its pipeline, and each slice stays a multiple of 16 wide.
    while (2 * p.ks <= kMaxSplit &&
           (long long)p.m_tiles * p.n_tiles * cta * 2 * p.ks <= dev.sm_count &&
           nkb >= 2 * p.ks * kMinKbPerSplit && p.BN % (2 * p.ks * 16) == 0 &&
           recv_bytes(p.BN, 2 * p.ks) <= ring &&
           cluster_fits(dev.device, cta * 2 * p.ks, pair, p.smem))
        p.ks *= 2;
    return p;
}

}  // namespace

cudaError_t launch_projection(const DeviceInfo& dev, const uint16_t* hidden,
                              const uint16_t* w_proj, int M, int H, int rank, uint16_t* h_out,
                              uint32_t* status_word, cudaStream_t stream, bool beside_topk,
                              uint32_t* done_counter, bool programmatic) {
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    // Allow the largest layout once per device, for every build; every plan fits under it.
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    std::call_once(once[dev.device], [&] {
        const int smem = (int)max_smem_bytes();
        cudaError_t e = cudaFuncSetAttribute(projection_kernel<16, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(projection_kernel<1, false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(projection_kernel<1, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        attr_err[dev.device] = e;
    });
    if (attr_err[dev.device] != cudaSuccess) return attr_err[dev.device];
    const ProjPlan plan = projection_plan(dev, M, H, rank, beside_topk);
    CUtensorMap map_a, map_b;
    if (!encode_2d(&map_a, hidden, (uint64_t)M, (uint64_t)H, BM) ||
        !encode_2d(&map_b, w_proj, (uint64_t)rank, (uint64_t)H,
                   (uint32_t)(plan.pair ? plan.BN / 2 : plan.BN)))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)plan.cluster();
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // As the programmatic dependent of the kernel before it (the top-k of the fused selector),
    // the projection may start once that kernel's CTAs have all started. It reads nothing that
    // kernel writes, so it never waits for it.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)(plan.m_tiles * plan.cluster()), (unsigned)plan.n_tiles);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 2 : 1;
    if (beside_topk)
        return cudaLaunchKernelEx(&cfg, projection_kernel<16, false>, map_a, map_b, h_out, M, rank,
                                  H, plan.BN, plan.tmem_cols, plan.ks, plan.stages, status_word,
                                  done_counter);
    if (plan.pair)
        return cudaLaunchKernelEx(&cfg, projection_kernel<1, true>, map_a, map_b, h_out, M, rank,
                                  H, plan.BN, plan.tmem_cols, plan.ks, plan.stages, status_word,
                                  done_counter);
    return cudaLaunchKernelEx(&cfg, projection_kernel<1, false>, map_a, map_b, h_out, M, rank, H,
                              plan.BN, plan.tmem_cols, plan.ks, plan.stages, status_word,
                              done_counter);
}

int projection_ctas(const DeviceInfo& dev, int M, int H, int rank) {
    const ProjPlan plan = projection_plan(dev, M, H, rank, true);
    return plan.m_tiles * plan.cluster() * plan.n_tiles;
}

}  // namespace dflash
