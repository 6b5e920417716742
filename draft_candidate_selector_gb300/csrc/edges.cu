// edges.cu: K x K edge scores of every (request, step).
//
// Method: page "vllm.models.beam.nvidia.dflash2", class DFlash2BeamCandidateSelector
// (docstring and forward). The score of position p, candidate c and predecessor q is
// the candidate's own logit plus <predecessor[q] * h_p, successor[c]>. The predecessor
// of the first position is the anchor token. The output is [requests, steps,
// top_k (predecessor), top_k].
//
// Design: one CTA per (r, p). The CTA gathers the (up to) K predecessor codebook rows
// and the K successor rows, each rank bf16 = rank*2 bytes contiguous, into shared
// memory:
//   G[q][j]  = pred_cb[pid_q][j] * h[r,p][j]     (fp32, row-major)
//   St[j][c] = succ_cb[cid_c][j]                 (fp32, transposed: lanes read along c)
// Warp w then owns predecessor rows q = w, w+4, ...; lane c accumulates
// sum_j G[q][j] * St[j][c] for up to 8 rows at once. G reads are warp-broadcast and
// St reads are consecutive, so shared memory has no bank conflicts. At p = 0 all
// predecessors are the anchor, so one row is computed and stored K times.
// Gathered ids are checked against [0, V). A bad id is never dereferenced: its row or
// column is NaN, and the status word records kStatusBadId.
#include "common.cuh"

#include <cuda_bf16.h>

#include <mutex>

namespace dflash {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerPass = 8;   // predecessor rows a lane accumulates at once

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__global__ void __launch_bounds__(kThreads)
edges_kernel(const uint16_t* __restrict__ pred_cb, const uint16_t* __restrict__ succ_cb,
             const int32_t* __restrict__ cand_ids, const float* __restrict__ unary,
             const uint16_t* __restrict__ h, const int32_t* __restrict__ anchors, int S, int K,
             int V, int rank, float* __restrict__ edges, uint32_t* __restrict__ status) {
    extern __shared__ float4 smem4[];
    float* G = reinterpret_cast<float*>(smem4);          // [K][rank]
    float* St = G + K * rank;                            // [rank][32]
    int* bad_q = reinterpret_cast<int*>(St + rank * 32); // [32]
    int* bad_c = bad_q + 32;                             // [32]

    const long long row = blockIdx.x;                    // r * S + p
    const int r = (int)(row / S);
    const int p = (int)(row % S);
    const int nq = (p == 0) ? 1 : K;
    const int chunks = rank >> 3;                        // 16-byte chunks per codebook row
    const int tid = threadIdx.x;

    if (tid < 32) {
        bad_q[tid] = 0;
        bad_c[tid] = 0;
    }
    __syncthreads();

    // Predecessor rows times h, chunk index fastest: a warp reads contiguous bytes.
    const uint4* h4 = reinterpret_cast<const uint4*>(h + row * rank);
    for (int item = tid; item < nq * chunks; item += kThreads) {
        const int q = item / chunks;
        const int ch = item - q * chunks;
        const int pid = (p == 0) ? anchors[r] : cand_ids[(row - 1) * K + q];
        float4 lo, hi;
        if (pid < 0 || pid >= V) {
            if (ch == 0) {
                bad_q[q] = 1;
                atomicOr(status, kStatusBadId);
            }
            lo = hi = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            const uint4 a = __ldg(reinterpret_cast<const uint4*>(pred_cb + (long long)pid * rank) + ch);
            const uint4 b = __ldg(h4 + ch);
            lo = make_float4(bf16_lo(a.x) * bf16_lo(b.x), bf16_hi(a.x) * bf16_hi(b.x),
                             bf16_lo(a.y) * bf16_lo(b.y), bf16_hi(a.y) * bf16_hi(b.y));
            hi = make_float4(bf16_lo(a.z) * bf16_lo(b.z), bf16_hi(a.z) * bf16_hi(b.z),
                             bf16_lo(a.w) * bf16_lo(b.w), bf16_hi(a.w) * bf16_hi(b.w));
        }
        float4* dst = reinterpret_cast<float4*>(G + q * rank + ch * 8);
        dst[0] = lo;
        dst[1] = hi;
    }
    // Successor rows, candidate index fastest: transposed stores hit distinct banks.
    for (int item = tid; item < K * chunks; item += kThreads) {
        const int ch = item / K;
        const int c = item - ch * K;
        const int cid = cand_ids[row * K + c];
        float v[8];
        if (cid < 0 || cid >= V) {
            if (ch == 0) {
                bad_c[c] = 1;
                atomicOr(status, kStatusBadId);
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) v[t] = 0.f;
        } else {
            const uint4 a = __ldg(reinterpret_cast<const uint4*>(succ_cb + (long long)cid * rank) + ch);
            v[0] = bf16_lo(a.x); v[1] = bf16_hi(a.x); v[2] = bf16_lo(a.y); v[3] = bf16_hi(a.y);
            v[4] = bf16_lo(a.z); v[5] = bf16_hi(a.z); v[6] = bf16_lo(a.w); v[7] = bf16_hi(a.w);
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) St[(ch * 8 + t) * 32 + c] = v[t];
    }
    __syncthreads();

    const int warp = tid >> 5;
    const int c = tid & 31;
    const bool c_ok = c < K;
    const float u = c_ok ? unary[row * K + c] : 0.f;
    const bool c_bad = c_ok && bad_c[c];
    float* out = edges + row * K * K;

    // Predecessor rows of this warp: q = warp + kWarps * i.
    for (int q0 = warp; q0 < nq; q0 += kWarps * kRowsPerPass) {
        float acc[kRowsPerPass];
#pragma unroll
        for (int i = 0; i < kRowsPerPass; ++i) acc[i] = 0.f;
        for (int j = 0; j < rank; j += 4) {
            const float s0 = St[(j + 0) * 32 + c];
            const float s1 = St[(j + 1) * 32 + c];
            const float s2 = St[(j + 2) * 32 + c];
            const float s3 = St[(j + 3) * 32 + c];
#pragma unroll
            for (int i = 0; i < kRowsPerPass; ++i) {
                const int q = q0 + i * kWarps;
                if (q < nq) {
                    const float4 g = *reinterpret_cast<const float4*>(G + q * rank + j);
                    acc[i] = fmaf(g.x, s0, acc[i]);
                    acc[i] = fmaf(g.y, s1, acc[i]);
                    acc[i] = fmaf(g.z, s2, acc[i]);
                    acc[i] = fmaf(g.w, s3, acc[i]);
                }
            }
        }
        if (c_ok) {
#pragma unroll
            for (int i = 0; i < kRowsPerPass; ++i) {
                const int q = q0 + i * kWarps;
                if (q < nq) {
                    const float e = (c_bad || bad_q[q]) ? __int_as_float(0x7FC00000) : u + acc[i];
                    if (p == 0) {
                        for (int qq = 0; qq < K; ++qq) out[qq * K + c] = e;
                    } else {
                        out[q * K + c] = e;
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
                         int rank, float* edges, uint32_t* status_word, cudaStream_t stream) {
    const size_t smem = (size_t)(K * rank + rank * 32) * sizeof(float) + 64 * sizeof(int);
    // The largest layout (K = 32, rank = 256) is allowed once per device; smaller ones fit.
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    std::call_once(once[dev.device], [&] {
        const size_t max_smem = (size_t)(32 * 256 + 256 * 32) * sizeof(float) + 64 * sizeof(int);
        attr_err[dev.device] = cudaFuncSetAttribute(
            edges_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
    });
    if (attr_err[dev.device] != cudaSuccess) return attr_err[dev.device];
    const long long rows = (long long)R * S;
    edges_kernel<<<(unsigned)rows, kThreads, smem, stream>>>(pred_cb, succ_cb, cand_ids, unary, h,
                                                             anchors, S, K, V, rank, edges,
                                                             status_word);
    return cudaGetLastError();
}

}  // namespace dflash
