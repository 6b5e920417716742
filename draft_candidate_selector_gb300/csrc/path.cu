// path.cu: the best path through each request's edge scores.
//
// Reading (the pages show no consumer of the edge scores): page
// "vllm.models.beam.nvidia.dflash2", module docstring: the selector rescores the top-k tokens
// at each block position against the token before it. The best path picks one candidate per
// step so that the sum over p of E[r,p,c_{p-1},c_p] is largest; at p = 0 the predecessor row is
// q = 0 (every q row there is the anchor's). Max-sum dynamic programming over the steps in
// fp32, in a fixed order with a fixed tie rule, so the choice is exactly reproducible:
//   V_0[c] = E[r,0,0,c];
//   V_p[c] = running maximum over q = 0..K-1 of V_{p-1}[q] + E[r,p,q,c], replaced only by a
//            strictly larger sum (ties keep the lower q; a NaN neither replaces nor is
//            replaced);
//   the last step's candidate is the running maximum of V_{S-1} (same rule), and the path
//   follows the kept predecessors back.
//
// Design: one 128-thread CTA per request. Thread (c, g), c = 0..31 the candidate column and
// g = 0..3 a quarter of the predecessors (q = 8g .. 8g+7), forms its 8 sums V_{p-1}[q] +
// E[r,p,q,c], reduces them with a 3-level tree, and two ordered shuffle levels combine the
// four quarters; every combine keeps exactly the running maximum's choice (scan_combine). The
// CTA stages the K x K blocks of the next steps in a shared-memory ring with cp.async
// (16-byte copies when K is even and the scores are 16-byte aligned, 4-byte ones otherwise), so a step's update runs while
// later steps' blocks are in flight; one barrier per step. V_{p-1} is double-buffered in
// shared memory, and the kept predecessors go to shared memory (S x 32 bytes). Thread 0
// takes the last step's choice and walks the kept predecessors back; the threads then write
// the path and its token ids in parallel. Reads R*S*K*K*4 bytes of E once. No waits on other
// CTAs.
#include "common.cuh"

namespace dflash {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kThreads = 128;
constexpr int kDepth = 8;                // ring stages (steps in flight: kDepth - 1)
constexpr int kMaxK = 32;
constexpr int kQuarter = kMaxK / 4;      // predecessors per thread

// Shared bytes: the ring [kDepth][K*K] floats, V [2][32] floats, the kept predecessors
// [S][32] and the path [S], 16-byte rounded.
__host__ __device__ inline size_t path_ring_bytes(int K) { return (size_t)kDepth * K * K * 4; }
__host__ __device__ inline size_t path_smem_bytes(int S, int K) {
    return path_ring_bytes(K) + 2 * kMaxK * 4 + (((size_t)S * 33 + 15) & ~(size_t)15);
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// All but the newest kDepth - 2 groups of this thread have landed.
__device__ __forceinline__ void cp_async_wait_ring() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kDepth - 2) : "memory");
}

// This thread's share of the copy of step p's K x K block into ring stage p % kDepth. When
// every block starts on a 16-byte boundary (K even and a 16-byte aligned base; `wide`), the
// copy moves 16 bytes per thread and instruction; otherwise 4.
__device__ __forceinline__ void stage_step(float* ring, const float* E, int p, int K, int tid,
                                           bool wide) {
    const int n = K * K;
    float* dst = ring + (size_t)(p % kDepth) * n;
    const float* src = E + (size_t)p * n;
    if (wide) {
        for (int i = tid * 4; i < n; i += kThreads * 4) cp_async16(dst + i, src + i);
    } else {
        for (int i = tid; i < n; i += kThreads) cp_async4(dst + i, src + i);
    }
}

// Combine two pieces of a left-to-right running maximum: (av, ai) covers lower indices than
// (bv, bi). The result is what the scan keeps over both: a strictly larger value replaces;
// ties keep the lower index; a NaN at index 0 sticks (nothing compares larger than it), and
// any other NaN is passed over (it never compares larger). Associative for adjacent pieces,
// so a tree over the indices gives exactly the scan's choice.
__device__ __forceinline__ void scan_combine(float& av, int& ai, float bv, int bi) {
    const bool a_nan = av != av;
    const bool take_b = a_nan ? (ai != 0) : (bv > av);
    if (take_b) {
        av = bv;
        ai = bi;
    }
}

// One ordered level across lanes lane and lane ^ m: the lane whose bit m is clear holds the
// lower indices. Both lanes end with the combined piece.
__device__ __forceinline__ void lane_combine(float& v, int& i, int lane, int m) {
    const float ov = __shfl_xor_sync(kFull, v, m);
    const int oi = __shfl_xor_sync(kFull, i, m);
    if (lane & m) {
        float lv = ov;
        int li = oi;
        scan_combine(lv, li, v, i);
        v = lv;
        i = li;
    } else {
        scan_combine(v, i, ov, oi);
    }
}

__global__ void __launch_bounds__(kThreads)
best_path_kernel(const float* __restrict__ edges, const int32_t* __restrict__ cand, int R, int S,
                 int K, int32_t* __restrict__ path, int32_t* __restrict__ tokens,
                 float* __restrict__ score) {
    extern __shared__ __align__(16) uint8_t path_smem[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int c = (tid >> 5) * 8 + (lane >> 2);          // candidate column
    const int g = lane & 3;                              // predecessor quarter
    const long long r = blockIdx.x;
    float* ring = reinterpret_cast<float*>(path_smem);                   // [kDepth][K*K]
    float* vbuf = reinterpret_cast<float*>(path_smem + path_ring_bytes(K));   // [2][32]
    uint8_t* keep = reinterpret_cast<uint8_t*>(vbuf + 2 * kMaxK);        // [S][32]
    uint8_t* chosen = keep + (size_t)S * 32;                             // [S]
    const float* E = edges + (size_t)r * S * K * K;
    const bool live = c < K;
    const bool wide = (K & 1) == 0 && (reinterpret_cast<uintptr_t>(edges) & 15) == 0;

    for (int p = 0; p < kDepth; ++p) {                   // prologue: steps 0 .. kDepth-1
        if (p < S) stage_step(ring, E, p, K, tid, wide);
        cp_async_commit();
    }
    for (int p = 0; p < S; ++p) {
        cp_async_wait_ring();                            // step p has landed (this thread's part)
        __syncthreads();                                 // ... everyone's; step p-1 is finished
        if (p >= 1) {
            // Refill the stage step p-1 used. One group per step, empty past the last step,
            // so that before step p's wait exactly p + kDepth - 1 groups are committed and
            // waiting for all but the newest kDepth - 2 covers step p.
            if (p - 1 + kDepth < S) stage_step(ring, E, p - 1 + kDepth, K, tid, wide);
            cp_async_commit();
        }
        const float* Ep = ring + (size_t)(p % kDepth) * K * K;
        if (p == 0) {
            if (g == 0 && live) vbuf[c] = Ep[c];         // predecessor row q = 0
            continue;
        }
        const float* vprev = vbuf + ((p - 1) & 1) * kMaxK;
        float s[kQuarter];
        int at[kQuarter];
#pragma unroll
        for (int j = 0; j < kQuarter; ++j) {
            const int q = g * kQuarter + j;
            at[j] = q;
            s[j] = (live && q < K) ? vprev[q] + Ep[q * K + c] : -INFINITY;
        }
#pragma unroll
        for (int w = 1; w < kQuarter; w <<= 1) {
#pragma unroll
            for (int j = 0; j + w < kQuarter; j += 2 * w) scan_combine(s[j], at[j], s[j + w], at[j + w]);
        }
        float v = s[0];
        int bq = at[0];
        lane_combine(v, bq, lane, 1);                    // quarters 0+1 and 2+3
        lane_combine(v, bq, lane, 2);                    // then the halves
        if (g == 0 && live) {
            vbuf[(p & 1) * kMaxK + c] = v;
            keep[p * 32 + c] = (uint8_t)bq;
        }
    }
    __syncthreads();
    if (tid == 0) {
        // The last step's choice: the running maximum over c, then the kept predecessors.
        const float* vl = vbuf + ((S - 1) & 1) * kMaxK;
        int cur = 0;
        float vb = vl[0];
        for (int j = 1; j < K; ++j) {
            if (vl[j] > vb) {
                vb = vl[j];
                cur = j;
            }
        }
        score[r] = vb;
        for (int p = S - 1; p >= 0; --p) {
            chosen[p] = (uint8_t)cur;
            if (p > 0) cur = keep[p * 32 + cur];
        }
    }
    __syncthreads();
    for (int p = tid; p < S; p += kThreads) {
        const int cc = chosen[p];
        path[(size_t)r * S + p] = cc;
        tokens[(size_t)r * S + p] = cand[((size_t)r * S + p) * K + cc];
    }
}

}  // namespace

cudaError_t launch_best_path(const float* edges, const int32_t* cand_ids, int R, int S, int K,
                             int32_t* path, int32_t* tokens, float* score, cudaStream_t stream) {
    // At most 32 KB of ring + 8.5 KB (S = 256): under the default 48 KB, no opt-in needed.
    const size_t smem = path_smem_bytes(S, K);
    best_path_kernel<<<(unsigned)R, kThreads, smem, stream>>>(edges, cand_ids, R, S, K, path,
                                                             tokens, score);
    return cudaGetLastError();
}

}  // namespace dflash
