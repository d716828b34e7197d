// Tensor-core GEMM for the prefill (and wide-batch) projections on sm_103a:
//   C[M, N] (+)= A[M, K] * B[N, K]^T,  A = activations, B = weights, both bf16,
//   K-major ("[out, in]" row-major weights, as ggml_mul_mat reads them), fp32 accumulation.
//
// One CTA computes a 128 x BN tile over a range of K blocks (split-K over gridDim.z):
//   warp 0, one lane: TMA producer - 2-D tiled bulk tensor copies of 128x64 (A) and
//                     BNx64 (B) bf16 tiles with 128-byte swizzle into a STAGES-deep ring;
//   warp 1:           allocates the TMEM accumulator (128 lanes x BN fp32 columns); one
//                     lane issues tcgen05.mma (kind::f16, M=128, N=BN, K=16) from shared
//                     memory descriptors and commits each stage back to the producer;
//   warps 2..5:       epilogue - tcgen05.ld of their 32-lane quadrant, then plain stores
//                     or vector reductions (red.add) into the fp32 output.
// Every mbarrier wait is bounded; a wait that gives up sets the device status word.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"

using namespace talker_dev;

namespace talker_k {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;                 // 64 bf16 = one 128-byte swizzle row
constexpr int NTHREADS = 192;

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile stored with the
// 128-byte swizzle (rows of 64 bf16, 8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);      // start address >> 4
    d |= (uint64_t)1u << 16;                       // leading byte offset >> 4 (not used with swizzle)
    d |= (uint64_t)(1024u >> 4) << 32;             // stride byte offset >> 4: 8 rows x 128 B
    d |= (uint64_t)1u << 46;                       // descriptor version
    d |= (uint64_t)2u << 61;                       // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16 with bf16 A/B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(NTHREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b, const GemmParams p) {
    constexpr uint32_t A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2;
    constexpr uint32_t IDESC = instr_desc(BM, BN);
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment for the swizzled tiles
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char *sA = smem;
    unsigned char *sB = smem + STAGES * A_BYTES;
    __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], done;
    __shared__ uint32_t tmem_base_s;
    __shared__ int fail_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
    const int nk_total = p.K / BK;
    const int per = (nk_total + gridDim.z - 1) / gridDim.z;
    const int kb0 = blockIdx.z * per;
    const int nk = max(0, min(per, nk_total - kb0));

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        fail_s = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_s)),
                     "r"((uint32_t)BN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    if (nk > 0) {
        if (warp == 0 && lane == 0) {
            // ---- TMA producer
            for (int i = 0; i < nk; ++i) {
                const int s = i % STAGES;
                if (i >= STAGES && !mbar_wait(&empty[s], ((i / STAGES) - 1) & 1, p.status)) {
                    fail_s = 1;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], A_BYTES + B_BYTES);
                tma_load_2d(sA + s * A_BYTES, &map_a, (kb0 + i) * BK, m0, &full[s]);
                tma_load_2d(sB + s * B_BYTES, &map_b, (kb0 + i) * BK, n0, &full[s]);
            }
            // let the last copies land before the CTA can exit (no-op when they were consumed)
            for (int i = max(0, nk - STAGES); i < nk; ++i) mbar_wait(&full[i % STAGES], (i / STAGES) & 1, p.status);
        } else if (warp == 1 && lane == 0) {
            // ---- MMA issuer
            bool ok = true;
            for (int i = 0; i < nk && ok; ++i) {
                const int s = i % STAGES;
                if (!mbar_wait(&full[s], (i / STAGES) & 1, p.status)) {
                    ok = false;
                    fail_s = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_u32(sA + s * A_BYTES), b0 = smem_u32(sB + s * B_BYTES);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    umma_bf16(tmem, smem_desc(a0 + k * 32), smem_desc(b0 + k * 32), IDESC, (i > 0 || k > 0) ? 1u : 0u);
                umma_commit(&empty[s]);
            }
            umma_commit(&done);   // arrives once every MMA issued so far has completed
        } else if (warp >= 2) {
            // ---- epilogue: TMEM quadrant (warp % 4) holds tile rows 32*(warp%4) .. +31
            const bool ok = mbar_wait(&done, 0, p.status);
            tc_fence_after();
            const int q = warp & 3;
            const int row = m0 + q * 32 + lane;
            if (ok && !fail_s) {
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 32), v);
                    if (row < p.M) {
                        float *o = p.out + (size_t)row * p.ld_out + n0 + c * 32;
                        if (p.accumulate) {
#pragma unroll
                            for (int i = 0; i < 32; i += 4) red_add_v4(o + i, v[i], v[i + 1], v[i + 2], v[i + 3]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; i += 4)
                                *reinterpret_cast<float4 *>(o + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                        }
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)BN) : "memory");
    }
}

// Persistent variant: one CTA per SM walks the tile list (tile t = blockIdx.x, +gridDim.x,
// ...; each tile is (row block, column block, K split)). The accumulator is double
// buffered in TMEM (2 x BN columns): while warps 2..5 drain tile j from buffer j & 1,
// the MMA thread already accumulates tile j + 1 into the other buffer, and the producer
// keeps the shared-memory ring full across tile boundaries.
template <int BN, int STAGES>
__global__ void __launch_bounds__(NTHREADS, 1)
    k_gemm_tc_persist(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                      const GemmParams p, int splits) {
    constexpr uint32_t A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2;
    constexpr uint32_t IDESC = instr_desc(BM, BN);
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char *sA = smem;
    unsigned char *sB = smem + STAGES * A_BYTES;
    __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2];
    __shared__ uint32_t tmem_base_s;
    __shared__ int fail_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_n = p.N / BN, tiles_m = (p.M + BM - 1) / BM;
    const int n_tiles = tiles_m * tiles_n * splits;
    const int nk_total = p.K / BK;
    const int per = (nk_total + splits - 1) / splits;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);   // one arrival per epilogue warp
        }
        fail_s = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_s)),
                     "r"((uint32_t)(2 * BN))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    // tile t -> (row block, column block, split); column blocks vary fastest
    auto tile_of = [&](int t, int &m0, int &n0, int &kb0, int &nk) {
        const int sp = t / (tiles_m * tiles_n), rem = t - sp * tiles_m * tiles_n;
        m0 = (rem / tiles_n) * BM;
        n0 = (rem % tiles_n) * BN;
        kb0 = sp * per;
        nk = max(0, min(per, nk_total - kb0));
    };

    if (warp == 0 && lane == 0) {
        // ---- TMA producer: one ring across all tiles of this CTA
        uint32_t it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
            int m0, n0, kb0, nk;
            tile_of(t, m0, n0, kb0, nk);
            for (int i = 0; i < nk; ++i, ++it) {
                const int s = it % STAGES;
                if (it >= (uint32_t)STAGES && !mbar_wait(&empty[s], ((it / STAGES) - 1) & 1, p.status)) {
                    fail_s = 1;
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], A_BYTES + B_BYTES);
                tma_load_2d(sA + s * A_BYTES, &map_a, (kb0 + i) * BK, m0, &full[s]);
                tma_load_2d(sB + s * B_BYTES, &map_b, (kb0 + i) * BK, n0, &full[s]);
            }
        }
        // let the last copies land before the CTA can exit (no-op when they were consumed)
        for (uint32_t j = (it > (uint32_t)STAGES ? it - STAGES : 0); j < it; ++j)
            mbar_wait(&full[j % STAGES], (j / STAGES) & 1, p.status);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        uint32_t it = 0;
        int j = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++j) {
            int m0, n0, kb0, nk;
            tile_of(t, m0, n0, kb0, nk);
            const int b = j & 1;
            if (j >= 2 && !mbar_wait(&tempty[b], ((j >> 1) - 1) & 1, p.status)) {
                fail_s = 1;
                break;
            }
            tc_fence_after();
            const uint32_t acc = tmem + (uint32_t)(b * BN);
            for (int i = 0; i < nk; ++i, ++it) {
                const int s = it % STAGES;
                if (!mbar_wait(&full[s], (it / STAGES) & 1, p.status)) {
                    fail_s = 1;
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_u32(sA + s * A_BYTES), b0 = smem_u32(sB + s * B_BYTES);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    umma_bf16(acc, smem_desc(a0 + k * 32), smem_desc(b0 + k * 32), IDESC, (i > 0 || k > 0) ? 1u : 0u);
                umma_commit(&empty[s]);
            }
            umma_commit(&tfull[b]);   // arrives once this tile's MMAs have completed
        }
    } else if (warp >= 2) {
        // ---- epilogue: TMEM lane quadrant (warp % 4) holds tile rows 32*(warp%4) .. +31
        const int q = warp & 3;
        int j = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++j) {
            int m0, n0, kb0, nk;
            tile_of(t, m0, n0, kb0, nk);
            const int b = j & 1;
            const bool ok = mbar_wait(&tfull[b], (j >> 1) & 1, p.status);
            tc_fence_after();
            if (!ok || fail_s) break;
            const int row = m0 + q * 32 + lane;
            if (nk > 0) {
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN + c * 32), v);
                    if (row < p.M) {
                        float *o = p.out + (size_t)row * p.ld_out + n0 + c * 32;
                        if (p.accumulate) {
#pragma unroll
                            for (int i = 0; i < 32; i += 4) red_add_v4(o + i, v[i], v[i + 1], v[i + 2], v[i + 3]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; i += 4)
                                *reinterpret_cast<float4 *>(o + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[b]);   // this warp's quadrant of buffer b is free
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)(2 * BN))
                     : "memory");
    }
}

}  // namespace tc
}  // namespace talker_k

namespace talker_k {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// 2-D map over a row-major bf16 matrix [rows, K]: box of 64 (K) x box_rows, 128-byte swizzle,
// zero fill outside the matrix.
bool make_map(CUtensorMap *m, const void *ptr, int rows, int K, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)tc::BK, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kBN = 128, kStages = 6;
constexpr size_t kGemmSmem = (size_t)kStages * (tc::BM + kBN) * tc::BK * 2 + 1024;

}  // namespace

bool gemm_tc_supported(int N, int K) { return N % kBN == 0 && K % tc::BK == 0 && K >= tc::BK; }

int gemm_tc_splits(int M, int N, int K, int n_sm) {
    const int tiles = ((M + tc::BM - 1) / tc::BM) * (N / kBN);
    const int nk = K / tc::BK;
    int s = (n_sm + tiles - 1) / tiles;
    s = std::min(s, std::max(1, nk / 4));   // keep at least 4 K blocks per split
    return std::max(1, s);
}

cudaError_t prepare_gemm_tc() {
    cudaError_t e = cudaFuncSetAttribute(tc::k_gemm_tc<kBN, kStages>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kGemmSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(tc::k_gemm_tc_persist<kBN, kStages>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kGemmSmem);
}

namespace {
int sm_count_current() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0 && cudaDeviceGetAttribute(&cached[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        cached[dev] = 0;
    return cached[dev];
}
}  // namespace

cudaError_t launch_gemm_tc(const void *A, int M, int K, const void *B, int N, float *out, int ld_out, int accumulate,
                           int splits, int *status, cudaStream_t st) {
    if (!gemm_tc_supported(N, K) || M < 1) return cudaErrorInvalidValue;
    CUtensorMap ma, mb;
    if (!make_map(&ma, A, M, K, tc::BM) || !make_map(&mb, B, N, K, kBN)) return cudaErrorInvalidValue;
    GemmParams p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.out = out;
    p.ld_out = ld_out;
    p.accumulate = (accumulate || splits > 1) ? 1 : 0;
    p.status = status;
    const int s = std::max(1, splits);
    const int n_tiles = (N / kBN) * ((M + tc::BM - 1) / tc::BM) * s;
    const int n_sm = sm_count_current();
    if (n_sm <= 0) return cudaErrorInvalidDevice;
    // persistent: one CTA per SM over the tile list, TMEM accumulators double buffered
    tc::k_gemm_tc_persist<kBN, kStages><<<std::min(n_tiles, n_sm), tc::NTHREADS, kGemmSmem, st>>>(ma, mb, p, s);
    return cudaGetLastError();
}

}  // namespace talker_k
