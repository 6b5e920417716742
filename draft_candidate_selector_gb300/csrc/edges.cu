// edges.cu: K x K edge scores of every (request, step).
//
// Method: page "vllm.models.beam.nvidia.dflash2", class DFlash2BeamCandidateSelector
// (docstring and forward). The score of position p, candidate c and predecessor q is
// the candidate's own logit plus <predecessor[q] * h_p, successor[c]>. The predecessor
// of the first position is the anchor token. The output is [requests, steps,
// top_k (predecessor), top_k].
//
// Design: one CTA (4 warps) per (r, p) tile, six CTAs per SM (35 KB of shared memory each),
// so six tiles' gathers are in flight on every SM.
//   1. Gather. Warp w owns row slots 16w..16w+15 (slots 0..31: predecessors q, 32..63:
//      successors c). Its lanes read those 16 ids with one load, then the warp copies
//      one whole codebook row per instruction: 32 lanes x 16 B cp.async (rank*2 bytes per
//      row). Predecessor q is pred_cb[cand[r,p-1,q]] (at p = 0, the anchor row, K times);
//      successor c is succ_cb[cand[r,p,c]]. Rows are stored with a 16-byte pad (stride
//      2*rank + 16 B), so the fragment loads below are bank-conflict free.
//   2. Contract. E[q][c] = sum_j G[q][j] S[c][j] with G = pred * h, on the tensor cores:
//      mma.sync m16n8k16 bf16 x bf16 -> fp32. Each A fragment is built in registers from
//      shared memory. G = pred * h is a product of two bf16 values, so it has at most 16
//      significant bits, and G = hi + lo exactly with hi = bf16(G), lo = bf16(G - hi).
//      Both halves are multiplied (two MMAs), so each product is exact and the sums run
//      in fp32. B fragments (successor rows) come from ldmatrix.
//   3. Epilogue: add unary[c], store rows q < K, columns c < K (a pair of columns per 8-byte
//      store when K is even and the output 8-byte aligned).
// In the forward pass (projection, then edges on one stream) the edges are launched as the
// projection's programmatic dependent: their CTAs start on free SMs, issue the id loads and
// codebook gathers, and wait (griddepcontrol.wait) for the projection only before copying h.
// In the fused selector they are the top-k's programmatic dependent instead: they take only
// the SMs top-k CTAs leave as they finish, and each CTA scores the tile the ready queue hands
// it (a tile whose rows the top-k has written), so most of the edges run in the top-k's tail.
// Ids are checked against [0, V) before any copy. A bad id is never dereferenced: its
// smem row is zeroed, its row or column of E is NaN, and the status word records
// kStatusBadId. No thread waits on another CTA.
#include "common.cuh"

#include <mutex>

namespace dflash {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxK = 32;
constexpr int kSlotsPerWarp = 2 * kMaxK / kWarps;   // 16

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte asynchronous copy global -> shared (not cached in L1).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// D += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two products pred*h from one 32-bit word (two bf16) of each, split into a packed hi pair
// and a packed lo pair with hi + lo = pred*h exactly (see the file comment). Each half is
// one bf16x2 fused multiply-add, which rounds the exact product once: hi = RN(a*b) (the
// addend is -0), lo = RN(a*b - hi). The product of two 8-bit significands has at most 16
// bits and its rounding remainder at most 8, so lo is exact.
__device__ __forceinline__ void split_pair(uint32_t a, uint32_t b, uint32_t& hi, uint32_t& lo) {
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(hi) : "r"(a), "r"(b), "r"(0x80008000u));
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(lo) : "r"(a), "r"(b), "r"(hi ^ 0x80008000u));
}

struct EdgeSmem {
    // Byte offsets inside the dynamic shared memory block.
    uint32_t stride;     // bytes per staged row: 2 * rank + 16
    uint32_t pred;       // [32][stride] predecessor rows
    uint32_t succ;       // [32][stride] successor rows
    uint32_t h;          // [stride]
    uint32_t flags;      // int bad_q[32], bad_c[32]
    uint32_t total;
};

__host__ __device__ inline EdgeSmem edge_smem_layout(int rank) {
    EdgeSmem L;
    L.stride = 2u * (uint32_t)rank + 16u;
    L.pred = 0;
    L.succ = kMaxK * L.stride;
    L.h = 2 * kMaxK * L.stride;
    L.flags = L.h + L.stride;
    L.total = L.flags + 2 * kMaxK * 4;
    return L;
}

// A wait in the ready queue gives up after this long; the CTA then sets kStatusTimeout and
// writes nothing.
constexpr unsigned long long kQueueWaitNs = 1000000000ull;

__device__ __forceinline__ unsigned long long now_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ unsigned ld_acquire(const uint32_t* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// One thread: wait for the tile pushed k-th (k = this CTA's index: every tile is pushed once,
// and the top-k that pushes them is resident before any edge CTA starts, so slot k always
// fills) and for every projection CTA to be done, then return the tile (or -1 after a
// timeout). Both counters are read with acquire loads, issued together; they pair with the
// writers' fences, and the barrier after this call carries the order to the CTA's other
// threads, so the tile's rows and h are visible to them.
__device__ int take_ready_tile(const EdgeQueue& q, uint32_t* status) {
    const uint32_t* slot = q.slots + blockIdx.x;
    unsigned v = ld_acquire(slot);
    unsigned done = ld_acquire(q.proj_done);
    if (v != 0u && done >= (unsigned)q.proj_ctas) return (int)v - 1;
    const unsigned long long t0 = now_ns();
    while (v == 0u || done < (unsigned)q.proj_ctas) {
        if (now_ns() - t0 > kQueueWaitNs) {
            atomicOr(status, kStatusTimeout);
            return -1;
        }
        __nanosleep(200);
        if (v == 0u) v = ld_acquire(slot);
        if (done < (unsigned)q.proj_ctas) done = ld_acquire(q.proj_done);
    }
    return (int)v - 1;
}

__global__ void __launch_bounds__(kThreads)
edges_kernel(const uint16_t* __restrict__ pred_cb, const uint16_t* __restrict__ succ_cb,
             const int32_t* __restrict__ cand_ids, const float* __restrict__ unary,
             const uint16_t* __restrict__ h, const int32_t* __restrict__ anchors, int S, int K,
             int V, int rank, float* __restrict__ edges, uint32_t* __restrict__ status,
             const EdgeQueue q) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int s_tile;
    const EdgeSmem L = edge_smem_layout(rank);
    const uint32_t sbase = smem_u32(smem);
    int* bad = reinterpret_cast<int*>(smem + L.flags);   // bad_q[32], then bad_c[32]

    long long row = blockIdx.x;                  // r * S + p
    if (q.slots != nullptr) {
        // Fused selector: CTA k runs whichever tile comes k-th in the ready queue, once the
        // projection has finished (all waits bounded).
        if (threadIdx.x == 0) s_tile = take_ready_tile(q, status);
        __syncthreads();
        if (s_tile < 0) return;
        row = s_tile;
    }
    const int r = (int)(row / S);
    const int p = (int)(row % S);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int chunks = rank >> 3;                // 16-byte chunks per codebook row
    const int kpad = (rank + 15) & ~15;          // contraction length, padded to 16

    // ---- 1. gather: ids first (one load per lane), then one row per warp instruction
    {
        const int slot = warp * kSlotsPerWarp + (lane & (kSlotsPerWarp - 1));
        const bool is_pred = slot < kMaxK;
        const int k = is_pred ? slot : slot - kMaxK;
        int id = -1;
        if (lane < kSlotsPerWarp && k < K)
            id = is_pred ? ((p == 0) ? anchors[r] : cand_ids[(row - 1) * K + k])
                         : cand_ids[row * K + k];
        const bool ok = id >= 0 && id < V;
        if (lane < kSlotsPerWarp) {
            bad[slot] = (k < K && !ok) ? 1 : 0;
            if (k < K && !ok) atomicOr(status, kStatusBadId);
        }
#pragma unroll 4
        for (int j = 0; j < kSlotsPerWarp; ++j) {
            const int s_j = warp * kSlotsPerWarp + j;
            const bool pred_j = s_j < kMaxK;
            const int k_j = pred_j ? s_j : s_j - kMaxK;
            if (k_j >= K) continue;                                     // warp-uniform
            const int id_j = __shfl_sync(0xffffffffu, id, j);
            const uint32_t dst_row = (pred_j ? L.pred : L.succ) + k_j * L.stride;
            if (lane < chunks) {
                if (id_j >= 0 && id_j < V)
                    cp_async16(sbase + dst_row + lane * 16,
                               (pred_j ? pred_cb : succ_cb) + (long long)id_j * rank + lane * 8);
                else
                    *reinterpret_cast<uint4*>(smem + dst_row + lane * 16) = make_uint4(0, 0, 0, 0);
            }
            // The K-padding tail [rank, kpad) of the row is zero.
            if (kpad != rank && lane == 0)
                *reinterpret_cast<uint4*>(smem + dst_row + 2 * rank) = make_uint4(0, 0, 0, 0);
        }
        // h may come from the grid launched just before this one (the forward pass launches
        // the edges as its programmatic dependent): the gathers above need only ids, so they
        // are already in flight. The wait returns at once when there is no such grid. With the
        // ready queue, the tile's rows and h are already known to be written.
        if (q.slots == nullptr) asm volatile("griddepcontrol.wait;" ::: "memory");
        if (warp == 0) {
            if (lane < chunks) cp_async16(sbase + L.h + lane * 16, h + row * rank + lane * 8);
            if (kpad != rank && lane == 0)
                *reinterpret_cast<uint4*>(smem + L.h + 2 * rank) = make_uint4(0, 0, 0, 0);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();
    }

    // ---- 2. contraction on the tensor cores, 3. epilogue
    const int m_tiles = (K + 15) >> 4;           // 16 predecessor rows per tile
    const int n_pairs = (K + 15) >> 4;           // two 8-wide candidate tiles per item
    const int g = lane >> 2;                     // fragment row
    const int t = lane & 3;                      // fragment column pair
    const int* bad_q = bad;
    const int* bad_c = bad + kMaxK;
    float* out = edges + row * K * K;
    const float* un = unary + row * K;
    // A candidate pair (c, c + 1) is stored with one 8-byte store when K is even and the
    // output is 8-byte aligned (then every pair is); otherwise one value at a time.
    const bool pair_store = (K & 1) == 0 && (reinterpret_cast<uintptr_t>(edges) & 7u) == 0;
    for (int item = warp; item < m_tiles * n_pairs; item += kWarps) {
        const int m0 = (item % m_tiles) * 16;
        const int n0 = (item / m_tiles) * 16;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        // This lane's unary values, loaded before the contraction hides their latency.
        float u[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int cc = n0 + nt * 8 + 2 * t + e;
                u[nt][e] = cc < K ? un[cc] : 0.f;
            }
        // A fragment words: rows m0+g and m0+g+8, columns k0+2t (+8).
        const uint32_t a_r0 = sbase + L.pred + (uint32_t)(m0 + g) * L.stride + 4u * t;
        const uint32_t a_r1 = a_r0 + 8u * L.stride;
        const uint32_t h_w = sbase + L.h + 4u * t;
        // B fragments by ldmatrix: matrix (lane >> 3), row (lane & 7) of it.
        const int mi = lane >> 3;
        const uint32_t b_ad = sbase + L.succ + (uint32_t)(n0 + (mi >> 1) * 8 + (lane & 7)) * L.stride +
                              (uint32_t)((mi & 1) * 16);
#pragma unroll 4
        for (int k0 = 0; k0 < kpad; k0 += 16) {
            const uint32_t hw0 = lds32(h_w + 2 * k0), hw1 = lds32(h_w + 2 * k0 + 16);
            uint32_t hi0, hi1, hi2, hi3, lo0, lo1, lo2, lo3;
            split_pair(lds32(a_r0 + 2 * k0), hw0, hi0, lo0);
            split_pair(lds32(a_r1 + 2 * k0), hw0, hi1, lo1);
            split_pair(lds32(a_r0 + 2 * k0 + 16), hw1, hi2, lo2);
            split_pair(lds32(a_r1 + 2 * k0 + 16), hw1, hi3, lo3);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(b_ad + 2 * k0, b0, b1, b2, b3);
            mma_bf16_16816(acc[0], hi0, hi1, hi2, hi3, b0, b1);
            mma_bf16_16816(acc[1], hi0, hi1, hi2, hi3, b2, b3);
            mma_bf16_16816(acc[0], lo0, lo1, lo2, lo3, b0, b1);
            mma_bf16_16816(acc[1], lo0, lo1, lo2, lo3, b2, b3);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int c = n0 + nt * 8 + 2 * t;           // even
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int q = m0 + g + half * 8;
                if (q >= K || c >= K) continue;
                float v0 = acc[nt][2 * half] + u[nt][0];
                float v1 = acc[nt][2 * half + 1] + u[nt][1];
                if (bad_q[q] || bad_c[c]) v0 = __int_as_float(0x7FC00000);
                if (pair_store) {
                    // K even: c + 1 < K as well, and q * K + c is even.
                    if (bad_q[q] || bad_c[c + 1]) v1 = __int_as_float(0x7FC00000);
                    *reinterpret_cast<float2*>(out + q * K + c) = make_float2(v0, v1);
                } else {
                    out[q * K + c] = v0;
                    if (c + 1 < K) {
                        if (bad_q[q] || bad_c[c + 1]) v1 = __int_as_float(0x7FC00000);
                        out[q * K + c + 1] = v1;
                    }
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_edges(const DeviceInfo& dev, const uint16_t* pred_cb,
                         const uint16_t* succ_cb, const int32_t* cand_ids, const float* unary,
                         const uint16_t* h, const int32_t* anchors, int R, int S, int K, int V,
                         int rank, float* edges, uint32_t* status_word, cudaStream_t stream,
                         bool after_h_producer, const EdgeQueue& queue, bool programmatic) {
    // Allow the largest layout (rank = 256) once per device; smaller ranks fit under it.
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    std::call_once(once[dev.device], [&] {
        attr_err[dev.device] = cudaFuncSetAttribute(
            edges_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
            (int)edge_smem_layout(256).total);
    });
    if (attr_err[dev.device] != cudaSuccess) return attr_err[dev.device];
    const long long rows = (long long)R * S;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)rows);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = edge_smem_layout(rank).total;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = (after_h_producer || programmatic) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, edges_kernel, pred_cb, succ_cb, cand_ids, unary, h, anchors,
                              S, K, V, rank, edges, status_word, queue);
}

}  // namespace dflash
