// edges.cu: K x K edge scores of every (request, step).
//
// Method: page "vllm.models.beam.nvidia.dflash2", class DFlash2BeamCandidateSelector
// (docstring and forward). The score of position p, candidate c and predecessor q is
// the candidate's own logit plus <predecessor[q] * h_p, successor[c]>. The predecessor
// of the first position is the anchor token. The output is [requests, steps,
// top_k (predecessor), top_k].
//
// Design: one CTA (4 warps) per (r, p), several CTAs per SM.
//   1. Gather. Lanes of warp 0 issue one bulk copy (cp.async.bulk, the TMA engine) per
//      codebook row into shared memory: the K predecessor rows pred_cb[pid_q] (at p = 0,
//      the anchor row, K times) and the K successor rows succ_cb[cid_c], plus h[r,p]. All
//      copies are in flight at once and land on one mbarrier. Rows are stored with a
//      16-byte pad (stride 2*rank + 16 B), so ldmatrix reads are bank-conflict free.
//   2. Split. G = pred * h is the product of two bf16 values, so it has at most 16
//      significant bits, and G = hi + lo exactly with hi = bf16(G) and lo = bf16(G - hi).
//      hi overwrites the predecessor rows in place; lo goes to its own buffer.
//   3. Contract. E[q][c] = sum_j hi[q][j] S[c][j] + sum_j lo[q][j] S[c][j] on the tensor
//      cores: mma.sync m16n8k16 bf16 x bf16 -> fp32, with operands loaded by ldmatrix.
//      Each product is exact, and the sums run in fp32.
//   4. Epilogue: add unary[c], store rows q < K, columns c < K.
// Ids are checked against [0, V) before any copy. A bad id is never dereferenced: its
// row or column of E is NaN, and the status word records kStatusBadId. The mbarrier wait
// is bounded (about one second); on expiry the CTA sets kStatusTimeout and writes NaN.
#include "common.cuh"

#include <cuda_bf16.h>

#include <mutex>

namespace dflash {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxK = 32;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > kWaitLimitNs) return false;
    }
}

// One bulk copy global -> shared, completing `bytes` on the mbarrier.
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
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

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// (x, y) -> packed bf16 pair (x in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack2(float x, float y) {
    __nv_bfloat162 v = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Two exact products pred*h from one 32-bit word of each, split into a packed hi pair
// and a packed lo pair (see the file comment).
__device__ __forceinline__ void split_pair(uint32_t a, uint32_t b, uint32_t& hi, uint32_t& lo) {
    const float x = bf16_lo(a) * bf16_lo(b);
    const float y = bf16_hi(a) * bf16_hi(b);
    hi = pack2(x, y);
    lo = pack2(x - bf16_lo(hi), y - bf16_hi(hi));
}

struct EdgeSmem {
    // Byte offsets inside the dynamic shared memory block.
    uint32_t stride;     // bytes per staged row: 2 * rank + 16
    uint32_t pred;       // [32][stride]: predecessor rows, then hi in place
    uint32_t lo;         // [32][stride]
    uint32_t succ;       // [32][stride]
    uint32_t h;          // [stride]
    uint32_t flags;      // int bad_q[32], bad_c[32]
    uint32_t bar;        // mbarrier (8 B)
    uint32_t total;
};

__host__ __device__ inline EdgeSmem edge_smem_layout(int rank) {
    EdgeSmem L;
    L.stride = 2u * (uint32_t)rank + 16u;
    L.pred = 0;
    L.lo = L.pred + kMaxK * L.stride;
    L.succ = L.lo + kMaxK * L.stride;
    L.h = L.succ + kMaxK * L.stride;
    L.flags = L.h + L.stride;
    L.bar = L.flags + 2 * kMaxK * 4;
    L.total = L.bar + 8;
    return L;
}

__global__ void __launch_bounds__(kThreads, 4)
edges_kernel(const uint16_t* __restrict__ pred_cb, const uint16_t* __restrict__ succ_cb,
             const int32_t* __restrict__ cand_ids, const float* __restrict__ unary,
             const uint16_t* __restrict__ h, const int32_t* __restrict__ anchors, int S, int K,
             int V, int rank, float* __restrict__ edges, uint32_t* __restrict__ status) {
    extern __shared__ __align__(16) uint8_t smem[];
    const EdgeSmem L = edge_smem_layout(rank);
    int* bad_q = reinterpret_cast<int*>(smem + L.flags);
    int* bad_c = bad_q + kMaxK;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar = sbase + L.bar;

    const long long row = blockIdx.x;            // r * S + p
    const int r = (int)(row / S);
    const int p = (int)(row % S);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t row_bytes = 2u * (uint32_t)rank;
    const int kpad = (rank + 15) & ~15;          // contraction length, padded to 16

    // ---- 1. gather (warp 0 issues every copy)
    if (warp == 0) {
        int pid = -1, cid = -1;
        if (lane < K) {
            pid = (p == 0) ? anchors[r] : cand_ids[(row - 1) * K + lane];
            cid = cand_ids[row * K + lane];
        }
        const bool pok = lane < K && pid >= 0 && pid < V;
        const bool cok = lane < K && cid >= 0 && cid < V;
        bad_q[lane] = (lane < K && !pok) ? 1 : 0;
        bad_c[lane] = (lane < K && !cok) ? 1 : 0;
        if ((lane < K) && (!pok || !cok)) atomicOr(status, kStatusBadId);
        const int copies = __popc(__ballot_sync(0xffffffffu, pok)) +
                           __popc(__ballot_sync(0xffffffffu, cok)) + 1;   // + h
        if (lane == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                         "r"(copies * row_bytes)
                         : "memory");
        }
        __syncwarp();
        if (pok)
            bulk_copy(sbase + L.pred + lane * L.stride, pred_cb + (long long)pid * rank,
                      row_bytes, bar);
        if (cok)
            bulk_copy(sbase + L.succ + lane * L.stride, succ_cb + (long long)cid * rank,
                      row_bytes, bar);
        if (lane == 0) bulk_copy(sbase + L.h, h + row * rank, row_bytes, bar);
    }
    __syncthreads();   // flags and barrier init visible to all
    // Zero what the copies do not write: rows of bad ids, and the K-padding tail
    // [rank, kpad) of every row. These bytes are disjoint from the copies' targets.
    {
        const int pad = (kpad - rank) * 2;       // 0 or 16 bytes
        for (int q = tid; q < kMaxK; q += kThreads) {
            if (pad) {
                *reinterpret_cast<uint4*>(smem + L.pred + q * L.stride + row_bytes) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(smem + L.lo + q * L.stride + row_bytes) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(smem + L.succ + q * L.stride + row_bytes) = make_uint4(0, 0, 0, 0);
            }
        }
        const int chunks = rank >> 3;
        for (int item = tid; item < K * chunks; item += kThreads) {
            const int q = item / chunks;
            const int ch = item - q * chunks;
            if (bad_q[q]) *reinterpret_cast<uint4*>(smem + L.pred + q * L.stride + ch * 16) = make_uint4(0, 0, 0, 0);
            if (bad_c[q]) *reinterpret_cast<uint4*>(smem + L.succ + q * L.stride + ch * 16) = make_uint4(0, 0, 0, 0);
        }
    }
    const bool landed = mbar_wait(bar, 0);
    const bool ok = __syncthreads_and(landed ? 1 : 0) != 0;
    if (!ok) {
        if (tid == 0) atomicOr(status, kStatusTimeout);
        // Give copies still in flight one more bounded wait before the CTA may exit.
        (void)mbar_wait(bar, 0);
    }

    // ---- 2. split G = pred * h into hi (in place) + lo
    if (ok) {
        const int chunks = rank >> 3;
        for (int item = tid; item < K * chunks; item += kThreads) {
            const int q = item / chunks;
            const int ch = item - q * chunks;
            uint4* pq = reinterpret_cast<uint4*>(smem + L.pred + q * L.stride + ch * 16);
            const uint4 a = *pq;
            const uint4 b = *reinterpret_cast<const uint4*>(smem + L.h + ch * 16);
            uint4 hi, lo;
            split_pair(a.x, b.x, hi.x, lo.x);
            split_pair(a.y, b.y, hi.y, lo.y);
            split_pair(a.z, b.z, hi.z, lo.z);
            split_pair(a.w, b.w, hi.w, lo.w);
            *pq = hi;
            *reinterpret_cast<uint4*>(smem + L.lo + q * L.stride + ch * 16) = lo;
        }
    }
    __syncthreads();

    // ---- 3. contraction on the tensor cores; 4. epilogue
    const int m_tiles = (K + 15) >> 4;           // 16 predecessor rows per tile
    const int n_pairs = (K + 15) >> 4;           // two 8-wide candidate tiles per item
    const int g = lane >> 2;                     // accumulator row within the tile
    const int t = lane & 3;                      // accumulator column pair
    float* out = edges + row * K * K;
    for (int item = warp; item < m_tiles * n_pairs; item += kWarps) {
        const int m0 = (item % m_tiles) * 16;
        const int n0 = (item / m_tiles) * 16;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        if (ok) {
            // ldmatrix lane addresses: matrix (lane >> 3), row (lane & 7) of it.
            const int mi = lane >> 3;
            const uint32_t a_row = (uint32_t)(m0 + (mi & 1) * 8 + (lane & 7));
            const uint32_t a_col = (uint32_t)((mi >> 1) * 8);
            const uint32_t b_row = (uint32_t)(n0 + (mi >> 1) * 8 + (lane & 7));
            const uint32_t b_col = (uint32_t)((mi & 1) * 8);
            const uint32_t a_hi = sbase + L.pred + a_row * L.stride + a_col * 2;
            const uint32_t a_lo = sbase + L.lo + a_row * L.stride + a_col * 2;
            const uint32_t b_ad = sbase + L.succ + b_row * L.stride + b_col * 2;
            for (int k0 = 0; k0 < kpad; k0 += 16) {
                uint32_t h0, h1, h2, h3, l0, l1, l2, l3, b0, b1, b2, b3;
                ldmatrix_x4(a_hi + k0 * 2, h0, h1, h2, h3);
                ldmatrix_x4(a_lo + k0 * 2, l0, l1, l2, l3);
                ldmatrix_x4(b_ad + k0 * 2, b0, b1, b2, b3);
                mma_bf16_16816(acc[0], h0, h1, h2, h3, b0, b1);
                mma_bf16_16816(acc[0], l0, l1, l2, l3, b0, b1);
                mma_bf16_16816(acc[1], h0, h1, h2, h3, b2, b3);
                mma_bf16_16816(acc[1], l0, l1, l2, l3, b2, b3);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int c = n0 + nt * 8 + 2 * t;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int q = m0 + g + half * 8;
                if (q >= K) continue;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int cc = c + e;
                    if (cc >= K) continue;
                    float v = acc[nt][2 * half + e] + unary[row * K + cc];
                    if (!ok || bad_q[q] || bad_c[cc]) v = __int_as_float(0x7FC00000);
                    out[q * K + cc] = v;
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_edges(const DeviceInfo& dev, const uint16_t* pred_cb,
                         const uint16_t* succ_cb, const int32_t* cand_ids, const float* unary,
                         const uint16_t* h, const int32_t* anchors, int R, int S, int K, int V,
                         int rank, float* edges, uint32_t* status_word, cudaStream_t stream) {
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
    edges_kernel<<<(unsigned)rows, kThreads, edge_smem_layout(rank).total, stream>>>(
        pred_cb, succ_cb, cand_ids, unary, h, anchors, S, K, V, rank, edges, status_word);
    return cudaGetLastError();
}

}  // namespace dflash
