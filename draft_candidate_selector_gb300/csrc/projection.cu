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
// One CTA computes one 128 x BN tile of D, with BN = min(rank rounded up to 16, 128):
//   * warp 0, one lane: TMA producer. Per 64-wide K block it loads a 128x64 A tile and a
//     BNx64 B tile (128-byte swizzle) into a 6-stage shared-memory ring. Completion is
//     tracked on mbarriers by transaction bytes.
//   * warp 1, one lane: MMA issuer. tcgen05.mma kind::f16 (bf16 x bf16 -> fp32), M=128,
//     N=BN, K=16, four per K block, accumulating in tensor memory. tcgen05.commit
//     frees each stage and finally signals the accumulator.
//   * warps 0-3: epilogue. tcgen05.ld 32 lanes x 16 columns per warp, convert to bf16,
//     store to global memory.
// Out-of-range rows, columns and K are zero-filled by TMA and never stored.
// Every mbarrier wait is bounded, about one second by %globaltimer. On expiry the kernel
// sets kStatusTimeout, skips the remaining work, still frees its tensor memory, and
// returns.
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
constexpr int kStages = 6;
constexpr int kThreads = 128;
constexpr uint32_t kATileBytes = BM * BK * 2;

__global__ void __launch_bounds__(kThreads, 1)
projection_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                  uint16_t* __restrict__ out, int M, int N, int Kdim, int BN, uint32_t tmem_cols,
                  uint32_t* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    // The 128-byte swizzle pattern repeats every 1024 B: tiles start on that boundary.
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t b_tile_bytes = (uint32_t)BN * BK * 2;
    uint8_t* sa = smem;
    uint8_t* sb = smem + kStages * kATileBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sb + kStages * b_tile_bytes);
    uint64_t* full = bars;                  // [kStages] TMA landed
    uint64_t* empty = bars + kStages;       // [kStages] MMAs done reading
    uint64_t* accum = bars + 2 * kStages;   // all MMAs done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BM;
    const int n0 = blockIdx.y * BN;
    const int num_kb = (Kdim + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(accum), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&map_a) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&map_b) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // TMA producer.
        int issued = 0;
        for (int kb = 0; kb < num_kb; ++kb) {
            const int s = kb % kStages;
            if (kb >= kStages && !mbar_wait(smem_u32(&empty[s]), ((kb / kStages) - 1) & 1)) {
                atomicOr(status, kStatusTimeout);
                break;
            }
            const uint32_t fb = smem_u32(&full[s]);
            mbar_expect_tx(fb, kATileBytes + b_tile_bytes);
            tma_load_2d(smem_u32(sa + s * kATileBytes), &map_a, fb, kb * BK, m0);
            tma_load_2d(smem_u32(sb + s * b_tile_bytes), &map_b, fb, kb * BK, n0);
            issued = kb + 1;
        }
        // The last load into each stage must land before the CTA may leave and its shared
        // memory be reused, also after a timeout. Each wait is bounded; in the normal case
        // those loads were consumed long ago and every wait returns at once.
        for (int q = issued > kStages ? issued - kStages : 0; q < issued; ++q)
            (void)mbar_wait(smem_u32(&full[q % kStages]), (q / kStages) & 1);
    } else if (warp == 1 && lane == 0) {
        // MMA issuer.
        const uint32_t idesc = f16_idesc(BM, BN);
        int kb = 0;
        for (; kb < num_kb; ++kb) {
            const int s = kb % kStages;
            if (!mbar_wait(smem_u32(&full[s]), (kb / kStages) & 1)) {
                atomicOr(status, kStatusTimeout);
                break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(sa + s * kATileBytes);
            const uint32_t b0 = smem_u32(sb + s * b_tile_bytes);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
                // Advancing 16 bf16 (32 B) along K inside the swizzled 128-byte row.
                umma_bf16(tmem, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), idesc,
                          (kb | k) != 0);
            }
            umma_commit(smem_u32(&empty[s]));
        }
        // Signals once every MMA issued above has completed (also after a timeout).
        umma_commit(smem_u32(accum));
    }
    __syncwarp();

    // Epilogue: every warp drains its 32 TMEM lanes (= 32 output rows).
    const bool ready = __all_sync(0xffffffffu, mbar_wait(smem_u32(accum), 0));
    tc_fence_after();
    if (ready) {
        const int row = m0 + warp * 32 + lane;
        uint16_t* orow = out + (long long)row * N;
        for (int c0 = 0; c0 < BN; c0 += 16) {
            uint32_t v[16];
            tmem_ld_32x32b_x16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
            const int col = n0 + c0;
            if (row < M && col < N) {
                uint4 w0, w1;
                w0.x = pack_bf16x2(v[0], v[1]);
                w0.y = pack_bf16x2(v[2], v[3]);
                w0.z = pack_bf16x2(v[4], v[5]);
                w0.w = pack_bf16x2(v[6], v[7]);
                w1.x = pack_bf16x2(v[8], v[9]);
                w1.y = pack_bf16x2(v[10], v[11]);
                w1.z = pack_bf16x2(v[12], v[13]);
                w1.w = pack_bf16x2(v[14], v[15]);
                reinterpret_cast<uint4*>(orow + col)[0] = w0;          // N % 8 == 0
                if (col + 8 < N) reinterpret_cast<uint4*>(orow + col)[1] = w1;
            }
        }
    } else if (threadIdx.x == 0) {
        atomicOr(status, kStatusTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
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

size_t smem_bytes(int BN) {
    return 1024 + (size_t)kStages * (kATileBytes + (size_t)BN * BK * 2) +
           (2 * kStages + 1) * sizeof(uint64_t) + 16;
}

}  // namespace

cudaError_t launch_projection(const DeviceInfo& dev, const uint16_t* hidden,
                              const uint16_t* w_proj, int M, int H, int rank, uint16_t* h_out,
                              uint32_t* status_word, cudaStream_t stream) {
    const int BN = rank >= 128 ? 128 : ((rank + 15) / 16) * 16;
    const uint32_t tmem_cols = BN <= 32 ? 32u : (BN <= 64 ? 64u : 128u);
    CUtensorMap map_a, map_b;
    if (!encode_2d(&map_a, hidden, (uint64_t)M, (uint64_t)H, BM) ||
        !encode_2d(&map_b, w_proj, (uint64_t)rank, (uint64_t)H, (uint32_t)BN))
        return cudaErrorInvalidValue;
    const size_t smem = smem_bytes(BN);
    // Allow the largest layout (BN = 128) once per device; smaller tiles fit under it.
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    std::call_once(once[dev.device], [&] {
        attr_err[dev.device] = cudaFuncSetAttribute(
            projection_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes(128));
    });
    if (attr_err[dev.device] != cudaSuccess) return attr_err[dev.device];
    dim3 grid((unsigned)((M + BM - 1) / BM), (unsigned)((rank + BN - 1) / BN));
    projection_kernel<<<grid, kThreads, smem, stream>>>(map_a, map_b, h_out, M, rank, H, BN,
                                                        tmem_cols, status_word);
    return cudaGetLastError();
}

}  // namespace dflash
