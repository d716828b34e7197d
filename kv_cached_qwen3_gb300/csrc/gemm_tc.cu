// Tensor-core GEMM for the prefill (and wide-batch) projections on sm_103a:
//   C[M, N] (+)= A[M, K] * B[N, K]^T,  A = activations, B = weights, both bf16,
//   K-major ("[out, in]" row-major weights, as ggml_mul_mat reads them), fp32 accumulation.
//
// Three kernels by shape:
//   k_gemm_tc_pair    tall products (1024 rows or more) with N % 256 == 0: CTA pairs on
//                     256 x 256 tiles (cta_group::2 MMAs of M = 256), persistent over the tiles;
//   k_gemm_tc_persist other products above 128 rows: one CTA per SM over 128 x 128 tiles;
//   k_gemm_tc_swap    at most 128 rows (decode batches, small prefills): the weights as the
//                     MMA's M operand, the rows as N.
// Each persistent CTA runs:
//   warp 0, one lane: TMA producer - 2-D tiled bulk tensor copies of 64-wide K slices with the
//                     128-byte swizzle into a STAGES-deep ring;
//   warp 1:           allocates two TMEM accumulators; one lane issues tcgen05.mma (kind::f16,
//                     K=16) from shared memory descriptors and commits each stage back to the
//                     producer;
//   warps 2..5:       epilogue - tcgen05.ld of their 32-lane quadrant (one row per lane),
//                     staged through per-warp shared blocks so that whole 128-byte row segments
//                     of the fp32 output are stored or reduce-added, or (gate/up projection)
//                     silu(gate) * up of interleaved column pairs is stored as bf16.
// Every mbarrier wait is bounded; a wait that gives up sets the device status word.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"
#include "tcgen05.cuh"

using namespace talker_dev;

namespace talker_k {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;                 // 64 bf16 = one 128-byte swizzle row
constexpr int NTHREADS = 192;

// One 32-column chunk of a warp's 32 accumulator rows (v: this lane's row, global rows row0 ..
// row0 + 31, columns col0 .. col0 + 31) through the warp's 32 x 32 staging block: with the
// SwiGLU epilogue, silu(gate) * up of the interleaved column pairs as bf16; else the fp32
// values stored or reduce-added. The caller syncs the warp before the block is reused.
__device__ __forceinline__ void epi_chunk32(const GemmParams &p, float *stg, const float (&v)[32], int row0, int col0,
                                            int lane) {
    if (p.swiglu_out != nullptr) {
        // columns (2j, 2j + 1) = (gate_j, up_j): 16 bf16 outputs = 32 bytes of this lane's
        // row, staged as [32 rows][2 x 16 B] with the halves swapped on every other group of
        // 4 rows (conflict-free), then written 16 rows x 32 bytes per instruction
        uint32_t h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float g0 = v[4 * i], u0 = v[4 * i + 1], g1 = v[4 * i + 2], u1 = v[4 * i + 3];
            const __nv_bfloat16 lo = __float2bfloat16_rn(g0 / (1.0f + expf(-g0)) * u0);
            const __nv_bfloat16 hi = __float2bfloat16_rn(g1 / (1.0f + expf(-g1)) * u1);
            h[i] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
        }
        uint4 *w = reinterpret_cast<uint4 *>(stg);
        const int sw = (lane >> 2) & 1;
        w[lane * 2 + sw] = make_uint4(h[0], h[1], h[2], h[3]);
        w[lane * 2 + (sw ^ 1)] = make_uint4(h[4], h[5], h[6], h[7]);
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int r = it * 16 + (lane >> 1), half = lane & 1;
            const uint4 x = w[r * 2 + (half ^ ((r >> 2) & 1))];
            const int grow = row0 + r;
            if (grow < p.M)
                *reinterpret_cast<uint4 *>(p.swiglu_out + (size_t)grow * p.ld_swiglu + col0 / 2 +
                                           half * 8) = x;
        }
    } else {
        // this lane's 32 values of its row go to the warp's 32 x 32 block (16-byte chunks
        // XOR-swizzled by row, conflict-free), then each instruction stores or reduce-adds
        // 4 rows x 128 contiguous bytes
        float4 *w = reinterpret_cast<float4 *>(stg);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            w[lane * 8 + (i ^ (lane & 7))] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int r = it * 4 + (lane >> 3), ch = lane & 7;
            const float4 x = w[r * 8 + (ch ^ (r & 7))];
            const int grow = row0 + r;
            if (grow < p.M) {
                float *o = p.out + (size_t)grow * p.ld_out + col0 + ch * 4;
                if (p.accumulate)
                    red_add_v4(o, x.x, x.y, x.z, x.w);
                else
                    *reinterpret_cast<float4 *>(o) = x;
            }
        }
    }
}

// One CTA per SM walks the tile list; each tile is (row block, column block, K split),
// and every CTA loads its own A and B boxes. The accumulator is double buffered in TMEM
// (2 x BN columns): while warps 2..5 drain tile j from buffer j & 1, the MMA thread already accumulates tile j + 1 into the other
// buffer, and the producer keeps the shared-memory ring full across tile boundaries.
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
    const int cid = blockIdx.x, n_ctas = gridDim.x;
    const int tiles_n = p.N / BN;
    const int tiles_m = (p.M + BM - 1) / BM;
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

    // tile t -> (row block of this CTA, column block, split); column blocks vary fastest
    auto tile_of = [&](int t, int &m0, int &n0, int &kb0, int &nk) {
        const int sp = t / (tiles_m * tiles_n), rem = t - sp * tiles_m * tiles_n;
        m0 = (rem / tiles_n) * BM;
        n0 = (rem % tiles_n) * BN;
        kb0 = sp * per;
        nk = max(0, min(per, nk_total - kb0));
    };

    pdl_launch_dependents();
    if (warp == 0 && lane == 0) {
        // ---- TMA producer: one ring across all tiles of this CTA. The weight boxes of the
        // first STAGES slots do not depend on the previous kernel: they are requested before
        // the dependency wait, the activation boxes after it.
        uint32_t pre = 0;
        for (int t = cid; t < n_tiles && pre < (uint32_t)STAGES; t += n_ctas) {
            int m0, n0, kb0, nk;
            tile_of(t, m0, n0, kb0, nk);
            for (int i = 0; i < nk && pre < (uint32_t)STAGES; ++i, ++pre) {
                mbar_arrive_expect_tx(&full[pre], A_BYTES + B_BYTES);
                tma_load_2d(sB + pre * B_BYTES, &map_b, (kb0 + i) * BK, n0, &full[pre]);
            }
        }
        pdl_wait();
        uint32_t it = 0;
        bool ok = true;
        for (int t = cid; t < n_tiles && ok; t += n_ctas) {
            int m0, n0, kb0, nk;
            tile_of(t, m0, n0, kb0, nk);
            for (int i = 0; i < nk; ++i, ++it) {
                const int s = it % STAGES;
                if (it < pre) {   // weights already requested
                    tma_load_2d(sA + s * A_BYTES, &map_a, (kb0 + i) * BK, m0, &full[s]);
                    continue;
                }
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
        // Tail: wait until the MMAs have consumed every slot still in flight, so no copy
        // lands in shared memory after the CTA has moved on.
        for (uint32_t j = (it > (uint32_t)STAGES ? it - STAGES : 0); j < it; ++j)
            mbar_wait(&empty[j % STAGES], (j / STAGES) & 1, p.status);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        uint32_t it = 0;
        int j = 0;
        bool ok = true;
        for (int t = cid; t < n_tiles && ok; t += n_ctas, ++j) {
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
        // ---- epilogue: TMEM lane quadrant (warp % 4) holds tile rows 32*(warp%4) .. +31;
        // it writes (or reduce-adds into) buffers of the previous kernels: wait for them first
        pdl_wait();
        const int q = warp & 3;
        float *stg = reinterpret_cast<float *>(sB + STAGES * B_BYTES) + q * 32 * 32;   // this warp's staging block
        int j = 0;
        for (int t = cid; t < n_tiles; t += n_ctas, ++j) {
            int m0, n0, kb0, nk;
            tile_of(t, m0, n0, kb0, nk);
            const int b = j & 1;
            const bool ok = mbar_wait(&tfull[b], (j >> 1) & 1, p.status);
            tc_fence_after();
            if (!ok || fail_s) break;
            if (nk > 0) {
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN + c * 32), v);
                    epi_chunk32(p, stg, v, m0 + q * 32, n0 + c * 32, lane);
                    __syncwarp();   // the block is rewritten by the next chunk
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


// Tall products on CTA pairs (a cluster of 2): tiles of 256 x 256, CTA r of the pair holding rows
// 128 r .. 128 r + 127 of A and columns 128 r .. 128 r + 127 of B in its own 6-stage ring; the
// even CTA issues M = 256, N = 256 MMAs (cta_group::2) that read both CTAs' shared memory and
// accumulate each CTA's 128 rows x 256 columns in its own TMEM (two buffers of 256 columns).
// Per CTA and K block 32 KB of operands feed 2 x 128 x 256 x 64 FLOP, 1.5 times the single-CTA
// 128 x 256 tile, and the deeper ring covers twice its copy latency. Both CTAs' copies count on
// the even CTA's full barriers; its commits arrive on both CTAs' empty and TMEM-full barriers, and
// all eight epilogue warps release a TMEM buffer on the even CTA's barrier. The fp32 epilogue
// stages each 32 x 32 chunk in the swizzled layout of the output's tensor map and hands it to the
// TMA (a bulk store, or an element-wise reduce-add for the residual stream and split-K), with two
// staging blocks per warp so that the next chunk is written while the previous one drains.
constexpr int kPairStages = 6;
__global__ void __launch_bounds__(NTHREADS, 1)
    k_gemm_tc_pair(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_o, const GemmParams p, int splits) {
    constexpr int STAGES = kPairStages;
    constexpr int BN = 256;                                // pair tile: 256 x 256
    constexpr uint32_t A_BYTES = BM * BK * 2, B_BYTES = (BN / 2) * BK * 2;
    constexpr uint32_t IDESC = instr_desc(2 * BM, BN);
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char *sA = smem;
    unsigned char *sB = smem + STAGES * A_BYTES;
    __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2];
    __shared__ uint32_t tmem_base_s;
    __shared__ int fail_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t rank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
    const int tiles_n = p.N / BN;
    const int tiles_m = (p.M + 2 * BM - 1) / (2 * BM);
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
            mbar_init(&tempty[b], 8);   // the four epilogue warps of both CTAs
        }
        fail_s = 0;
        fence_barrier_init();
    }
    // both CTAs' barriers are initialised before either signals the other's
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_s)),
                     "r"((uint32_t)(2 * BN))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    auto at_rank = [&](const void *local, uint32_t r) {   // a barrier's copy in CTA r (shared::cluster address)
        uint32_t a;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(r));
        return a;
    };
    auto lead = [&](const void *local) { return at_rank(local, 0u); };

    // tile t -> (256-row block, 256-column block, split); column blocks vary fastest
    auto tile_of = [&](int t, int &m0, int &n0, int &kb0, int &nk) {
        const int sp = t / (tiles_m * tiles_n), rem = t - sp * tiles_m * tiles_n;
        m0 = (rem / tiles_n) * 2 * BM;
        n0 = (rem % tiles_n) * BN;
        kb0 = sp * per;
        nk = max(0, min(per, nk_total - kb0));
    };

    pdl_launch_dependents();
    if (warp == 0 && lane == 0) {
        // ---- TMA producer of this CTA's halves; the even CTA arms each stage for both
        const int ra = (int)rank * BM, rb = (int)rank * (BN / 2);
        uint32_t pre = 0;
        for (int t = pair; t < n_tiles && pre < (uint32_t)STAGES; t += n_pairs) {
            int m0, n0, kb0, nk;
            tile_of(t, m0, n0, kb0, nk);
            for (int i = 0; i < nk && pre < (uint32_t)STAGES; ++i, ++pre) {
                if (rank == 0) mbar_arrive_expect_tx(&full[pre], 2 * (A_BYTES + B_BYTES));
                tma_load_2d_pair(sB + pre * B_BYTES, &map_b, (kb0 + i) * BK, n0 + rb, lead(&full[pre]));
            }
        }
        pdl_wait();
        uint32_t it = 0;
        bool ok = true;
        for (int t = pair; t < n_tiles && ok; t += n_pairs) {
            int m0, n0, kb0, nk;
            tile_of(t, m0, n0, kb0, nk);
            for (int i = 0; i < nk; ++i, ++it) {
                const int s = it % STAGES;
                if (it < pre) {   // weights already requested
                    tma_load_2d_pair(sA + s * A_BYTES, &map_a, (kb0 + i) * BK, m0 + ra, lead(&full[s]));
                    continue;
                }
                if (it >= (uint32_t)STAGES && !mbar_wait(&empty[s], ((it / STAGES) - 1) & 1, p.status)) {
                    fail_s = 1;
                    ok = false;
                    break;
                }
                if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * (A_BYTES + B_BYTES));
                tma_load_2d_pair(sA + s * A_BYTES, &map_a, (kb0 + i) * BK, m0 + ra, lead(&full[s]));
                tma_load_2d_pair(sB + s * B_BYTES, &map_b, (kb0 + i) * BK, n0 + rb, lead(&full[s]));
            }
        }
        for (uint32_t j = (it > (uint32_t)STAGES ? it - STAGES : 0); j < it; ++j)
            mbar_wait(&empty[j % STAGES], (j / STAGES) & 1, p.status);
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ---- MMA issuer (even CTA)
        uint32_t it = 0;
        int j = 0;
        bool ok = true;
        for (int t = pair; t < n_tiles && ok; t += n_pairs, ++j) {
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
                    umma_bf16_pair(acc, smem_desc(a0 + k * 32), smem_desc(b0 + k * 32), IDESC,
                                   (i > 0 || k > 0) ? 1u : 0u);
                umma_commit_pair(at_rank(&empty[s], 0u));   // the stage is free in both CTAs
                umma_commit_pair(at_rank(&empty[s], 1u));
            }
            umma_commit_pair(at_rank(&tfull[b], 0u));   // both CTAs' accumulator halves are complete
            umma_commit_pair(at_rank(&tfull[b], 1u));
        }
    } else if (warp >= 2) {
        // ---- epilogue: this CTA's 128 rows of the tile, TMEM lane quadrant (warp % 4)
        pdl_wait();
        const int q = warp & 3;
        float *stg = reinterpret_cast<float *>(sB + STAGES * B_BYTES) + q * 2 * 32 * 32;   // two 4 KB blocks
        int nst = 0;   // chunks this warp has handed to the TMA
        int j = 0;
        for (int t = pair; t < n_tiles; t += n_pairs, ++j) {
            int m0, n0, kb0, nk;
            tile_of(t, m0, n0, kb0, nk);
            const int b = j & 1;
            const bool ok = mbar_wait(&tfull[b], (j >> 1) & 1, p.status);
            tc_fence_after();
            if (!ok) break;
            if (nk > 0) {
                const int row0 = m0 + (int)rank * BM + q * 32;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN + c * 32), v);
                    if (p.swiglu_out != nullptr) {
                        epi_chunk32(p, stg, v, row0, n0 + c * 32, lane);
                    } else {
                        float4 *w = reinterpret_cast<float4 *>(stg + (nst & 1) * 32 * 32);
                        if (nst >= 2) {   // the block's previous store has been read out
                            if (lane == 0) bulk_wait_read_1();
                            __syncwarp();
                        }
                        // row = lane, 16-byte chunk i at i ^ (row % 8): the tensor map's 128-byte swizzle
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            w[lane * 8 + (i ^ (lane & 7))] =
                                make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {   // rows past M are clipped by the copy (a block wholly past M is skipped)
                            if (row0 < p.M) {
                                if (p.accumulate) tma_reduce_add_2d(&map_o, n0 + c * 32, row0, w);
                                else tma_store_2d(&map_o, n0 + c * 32, row0, w);
                            }
                            bulk_commit();
                        }
                        ++nst;
                    }
                    __syncwarp();   // the block is rewritten by the next chunk
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)   // this warp's quadrant of buffer b is free (on the even CTA's barrier)
                asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(lead(&tempty[b]))
                             : "memory");
        }
        if (lane == 0) bulk_wait_all();   // every store has landed before the CTA moves on
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    // neither CTA releases TMEM (or leaves) while the other may still use the pair's resources
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)(2 * BN))
                     : "memory");
    }
}


// Short products (M <= 128 activation rows: decode batches, small prefills) with the weights as
// the MMA's M operand: D^T[f, r] = sum_k W[f, k] X[r, k] for one tile of 128 weight rows
// (output features) and all rows at once (N = M rounded up to 16), a K range per CTA.
// The shared-memory ring holds 128 x 64 weight boxes and only N x 64 activation boxes, so
// a CTA fits next to the previous kernel's CTAs and streams its first weight boxes before the
// dependency wait. Epilogue: TMEM lane = feature, column = row; each warp turns 16 rows x its
// 32 features around in shared memory and stores or reduce-adds (split-K, the residual) 4 rows
// x 128 bytes per instruction, or writes silu(gate) * up of the interleaved feature pairs as bf16.
constexpr int kSwapStages = 4;
__global__ void __launch_bounds__(NTHREADS, 1)
    k_gemm_tc_swap(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                   const GemmParams p, int splits) {
    constexpr uint32_t W_BYTES = BM * BK * 2;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int ncol = (p.M + 15) / 16 * 16;                 // MMA N: rows rounded up to 16
    const uint32_t X_BYTES = (uint32_t)ncol * BK * 2;      // a multiple of 2048
    unsigned char *sW = smem;
    unsigned char *sX = smem + kSwapStages * W_BYTES;
    __shared__ __align__(8) uint64_t full[kSwapStages], empty[kSwapStages], tfull;
    __shared__ uint32_t tmem_base_s;
    __shared__ int last_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x / splits, sp = blockIdx.x - tile * splits;
    const int f0 = tile * BM;
    const int nk_total = p.K / BK;
    const int kb0 = sp * nk_total / splits, kb1 = (sp + 1) * nk_total / splits;
    const int nk = kb1 - kb0;
    uint32_t tcols = 32;
    while ((int)tcols < ncol) tcols <<= 1;
    const uint32_t idesc = instr_desc(BM, ncol);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSwapStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&tfull, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_s)),
                     "r"(tcols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    pdl_launch_dependents();

    if (warp == 0 && lane == 0) {
        // ---- TMA producer: weight boxes of the first stages before the dependency wait
        const int pre = nk < kSwapStages ? nk : kSwapStages;
        for (int i = 0; i < pre; ++i) {
            mbar_arrive_expect_tx(&full[i], W_BYTES + X_BYTES);
            tma_load_2d(sW + i * W_BYTES, &map_w, (kb0 + i) * BK, f0, &full[i]);
        }
        pdl_wait();
        for (int i = 0; i < nk; ++i) {
            const int s = i % kSwapStages;
            if (i >= pre) {
                if (!mbar_wait(&empty[s], ((i / kSwapStages) - 1) & 1, p.status)) break;
                mbar_arrive_expect_tx(&full[s], W_BYTES + X_BYTES);
                tma_load_2d(sW + s * W_BYTES, &map_w, (kb0 + i) * BK, f0, &full[s]);
            }
            tma_load_2d(sX + s * X_BYTES, &map_x, (kb0 + i) * BK, 0, &full[s]);
        }
        for (int j = (nk > kSwapStages ? nk - kSwapStages : 0); j < nk; ++j)
            mbar_wait(&empty[j % kSwapStages], (j / kSwapStages) & 1, p.status);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        for (int i = 0; i < nk; ++i) {
            const int s = i % kSwapStages;
            if (!mbar_wait(&full[s], (i / kSwapStages) & 1, p.status)) break;
            tc_fence_after();
            const uint32_t w0 = smem_u32(sW + s * W_BYTES), x0 = smem_u32(sX + s * X_BYTES);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
                umma_bf16(tmem, smem_desc(w0 + k * 32), smem_desc(x0 + k * 32), idesc, (i > 0 || k > 0) ? 1u : 0u);
            umma_commit(&empty[s]);
        }
        umma_commit(&tfull);
    } else if (warp >= 2) {
        // ---- epilogue: warp q holds features f0 + 32 q + lane (its TMEM lane quadrant)
        pdl_wait();
        const int q = warp & 3;
        const int f = f0 + q * 32 + lane;
        float *stg = reinterpret_cast<float *>(sX + kSwapStages * X_BYTES) + q * 16 * 32;
        const bool ok = mbar_wait(&tfull, 0, p.status);
        tc_fence_after();
        const bool direct_swiglu = p.swiglu_out != nullptr && p.fin_cnt == nullptr;
        if (ok) {
            for (int c0 = 0; c0 < ncol; c0 += 16) {
                float v[16];
                tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, v);
                if (direct_swiglu) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        // features 2i (gate) and 2i + 1 (up) sit in neighbouring lanes
                        const int r = c0 + j;
                        const float u = __shfl_xor_sync(0xffffffffu, v[j], 1);
                        if (r < p.M && (lane & 1) == 0) {
                            const float g = v[j];
                            p.swiglu_out[(size_t)r * p.ld_swiglu + f / 2] = __float2bfloat16_rn(g / (1.0f + expf(-g)) * u);
                        }
                    }
                } else {
                    // through the warp's 16 x 32 staging block: lane = feature on the way in, then
                    // each instruction stores or reduce-adds 4 rows x 128 contiguous bytes
#pragma unroll
                    for (int j = 0; j < 16; ++j) stg[j * 32 + lane] = v[j];
                    __syncwarp();
#pragma unroll
                    for (int it = 0; it < 4; ++it) {
                        const int rr = it * 4 + (lane >> 3), ch = lane & 7;
                        const float4 x = reinterpret_cast<const float4 *>(stg)[rr * 8 + ch];
                        const int r = c0 + rr;
                        if (r < p.M) {
                            float *o = p.out + (size_t)r * p.ld_out + f0 + q * 32 + ch * 4;
                            if (p.accumulate)
                                red_add_v4(o, x.x, x.y, x.z, x.w);
                            else
                                *reinterpret_cast<float4 *>(o) = x;
                        }
                    }
                    __syncwarp();   // the block is rewritten by the next chunk
                }
            }
        }
        if (p.fin_cnt != nullptr) {
            // split-K SwiGLU: the CTA whose reduce-adds complete the tile finishes it (release by
            // the fence before the count, acquire by the fence after it)
            __threadfence();
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (threadIdx.x == 64) last_s = atomicAdd(&p.fin_cnt[tile], 1) == splits - 1;
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (last_s) {
                __threadfence();
                // 8 independent L2 reads in flight per thread, then their outputs
                const int t = threadIdx.x - 64, n4 = p.M * 32;
                for (int i0 = t; i0 < n4; i0 += 128 * 8) {
                    float4 x[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int i = i0 + u * 128;
                        if (i < n4)
                            x[u] = __ldcg(reinterpret_cast<const float4 *>(p.out + (size_t)(i >> 5) * p.ld_out + f0 +
                                                                           (i & 31) * 4));
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int i = i0 + u * 128;
                        if (i < n4) {
                            const int r = i >> 5, c = i & 31;
                            __stcg(reinterpret_cast<float4 *>(p.out + (size_t)r * p.ld_out + f0 + c * 4),
                                   make_float4(0.f, 0.f, 0.f, 0.f));
                            *reinterpret_cast<__nv_bfloat162 *>(p.swiglu_out + (size_t)r * p.ld_swiglu + f0 / 2 + c * 2) =
                                __floats2bfloat162_rn(x[u].x / (1.0f + expf(-x[u].x)) * x[u].y,
                                                      x[u].z / (1.0f + expf(-x[u].z)) * x[u].w);
                        }
                    }
                }
                if (t == 0) p.fin_cnt[tile] = 0;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tcols) : "memory");
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

}  // namespace

// 2-D map over a bf16 matrix [rows][cols] with the given row stride: boxes of box_cols
// (64 = one 128-byte swizzle row) x box_rows, 128-byte swizzle, zero fill outside.
bool make_map_bf16_2d(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint64_t row_stride_bytes,
                      int box_cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_stride_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// fp32 matrix [rows][cols] (row stride in bytes) in boxes of 32 x 32 with the 128-byte swizzle:
// the destination of the bulk tensor stores and reduce-adds of an epilogue.
bool make_map_f32_2d(CUtensorMap *m, void *ptr, uint64_t rows, uint64_t cols, uint64_t row_stride_bytes) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_stride_bytes};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// row-major [rows, K] operand, boxes of 64 (K) x box_rows
bool make_map(CUtensorMap *m, const void *ptr, int rows, int K, int box_rows) {
    return make_map_bf16_2d(m, ptr, (uint64_t)rows, (uint64_t)K, (uint64_t)K * 2, tc::BK, box_rows);
}

// Two tile widths: 256 x 256 pair tiles for tall products where N allows (per CTA and K block
// 32 KB of operands for 128 x 256 outputs), and 128 x 128 single-CTA tiles (6-stage ring)
// otherwise. TMEM holds two accumulators either way.
constexpr int kBNNarrow = 128, kStagesNarrow = 6;
constexpr int kBNWide = 256;
// ring + the epilogue's staging blocks (4 warps x 32 x 32 f32) + alignment slack
constexpr size_t smem_for(int bn, int stages) {
    return (size_t)stages * (tc::BM + bn) * tc::BK * 2 + 4 * 32 * 32 * 4 + 1024;
}

// Wide tiles only for tall activations (8 or more row blocks). A short M
// (small prefills, decode batches) streams the weights once, and there the narrow tiles
// give twice as many CTAs pulling them from HBM.
constexpr int kWideMinRowBlocks = 8;
bool tall(int M) { return (M + tc::BM - 1) / tc::BM >= kWideMinRowBlocks; }
int tile_n_for(int M, int N) { return (tall(M) && N % kBNWide == 0) ? kBNWide : kBNNarrow; }

}  // namespace

bool gemm_tc_supported(int N, int K) { return N % kBNNarrow == 0 && K % tc::BK == 0 && K >= tc::BK; }

int gemm_tc_splits(int M, int N, int K, int n_sm) {
    if (gemm_tc_swap_ok(M, N, K)) return gemm_tc_swap_splits(M, N, K, n_sm);
    const int tiles = ((M + tc::BM - 1) / tc::BM) * (N / tile_n_for(M, N));
    const int nk = K / tc::BK;
    int s = (n_sm + tiles - 1) / tiles;
    s = std::min(s, std::max(1, nk / 4));   // keep at least 4 K blocks per split
    return std::max(1, s);
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

template <int BN, int STAGES>
static cudaError_t raise_smem() {
    return cudaFuncSetAttribute(tc::k_gemm_tc_persist<BN, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_for(BN, STAGES));
}

namespace {
// The swapped kernel's shared memory: weight and activation boxes of each stage, the
// epilogue's staging blocks (4 warps x 16 x 32 f32) and alignment slack.
size_t smem_swap(int M) {
    const size_t ncol = (size_t)(M + 15) / 16 * 16;
    return (size_t)tc::kSwapStages * (tc::BM + ncol) * tc::BK * 2 + 4 * 16 * 32 * 4 + 1024;
}
constexpr int kSwapMaxRows = 128;
}  // namespace

// CTA pair kernel: 6 stages of 16 KB (A) + 16 KB (half of B) per CTA, two staging blocks per
// epilogue warp, slack.
constexpr size_t kPairSmem = (size_t)tc::kPairStages * 2 * tc::BM * tc::BK * 2 + 4 * 2 * 32 * 32 * 4 + 1024;

cudaError_t prepare_gemm_tc() {
    cudaError_t e = raise_smem<kBNNarrow, kStagesNarrow>();
    e = e ? e : cudaFuncSetAttribute(tc::k_gemm_tc_pair, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPairSmem);
    return e ? e : cudaFuncSetAttribute(tc::k_gemm_tc_swap, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)smem_swap(kSwapMaxRows));
}

bool gemm_tc_swap_ok(int M, int N, int K) {
    return M >= 1 && M <= kSwapMaxRows && N % tc::BM == 0 && K % tc::BK == 0 && K >= tc::BK;
}

// K splits of the swapped kernel: one wave of CTAs (as many per SM as the shared memory of
// this row count allows, at most two), at least two K blocks each.
int gemm_tc_swap_splits(int M, int N, int K, int n_sm) {
    const int tiles = N / tc::BM, nkb = K / tc::BK;
    const int per_sm = std::max(1, std::min(2, (int)((228 * 1024) / (smem_swap(M) + 1024))));
    const int s = std::max(1, n_sm * per_sm / tiles);
    return std::max(1, std::min(s, nkb / 2));
}

cudaError_t launch_gemm_tc_swap(const void *X, int M, int K, const void *W, int N, float *out, int ld_out,
                                int accumulate, int splits, __nv_bfloat16 *swiglu_out, int ld_swiglu, int *status,
                                cudaStream_t st, int *fin_cnt) {
    if (!gemm_tc_swap_ok(M, N, K) || splits < 1 || splits > K / tc::BK ||
        (swiglu_out != nullptr && fin_cnt == nullptr && splits != 1))
        return cudaErrorInvalidValue;
    if ((swiglu_out == nullptr || fin_cnt != nullptr) &&
        (out == nullptr || ld_out % 4 != 0 || (reinterpret_cast<uintptr_t>(out) & 15u) != 0))
        return cudaErrorInvalidValue;
    if (fin_cnt != nullptr && (swiglu_out == nullptr || ld_swiglu % 2 != 0)) return cudaErrorInvalidValue;
    GemmParams p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.out = out;
    p.ld_out = ld_out;
    p.accumulate = (accumulate || splits > 1) ? 1 : 0;
    p.status = status;
    p.swiglu_out = swiglu_out;
    p.ld_swiglu = ld_swiglu;
    p.fin_cnt = fin_cnt;
    if (fin_cnt != nullptr) p.accumulate = 1;
    CUtensorMap mw, mx;
    const int ncol = (M + 15) / 16 * 16;
    if (!make_map(&mw, W, N, K, tc::BM) || !make_map(&mx, X, M, K, ncol)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N / tc::BM) * splits, 1, 1);
    cfg.blockDim = dim3(tc::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = smem_swap(M);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc::k_gemm_tc_swap, mw, mx, p, splits);
}

cudaError_t launch_gemm_tc_swiglu_split(const void *A, int M, int K, const void *B, int N, float *acc,
                                        __nv_bfloat16 *out_bf16, int ld, int *cnt, int splits, int *status,
                                        cudaStream_t st) {
    if (acc == nullptr || cnt == nullptr || out_bf16 == nullptr) return cudaErrorInvalidValue;
    return launch_gemm_tc_swap(A, M, K, B, N, acc, N, 1, splits, out_bf16, ld, status, st, cnt);
}

namespace {
// Persistent launch: one CTA per SM (the shared-memory ring allows no more), at most one
// per tile.
template <int BN, int STAGES>
cudaError_t launch_cfg(const CUtensorMap &ma, const CUtensorMap &mb, const GemmParams &p, int splits, int n_sm,
                       cudaStream_t st) {
    const int tiles = ((p.M + tc::BM - 1) / tc::BM) * (p.N / BN) * splits;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(tc::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = smem_for(BN, STAGES);
    cfg.stream = st;
    cfg.gridDim = dim3(std::min(tiles, n_sm), 1, 1);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc::k_gemm_tc_persist<BN, STAGES>, ma, mb, p, splits);
}

// Tall products with N % 256 == 0 on CTA pairs: 256 x 256 tiles, one pair per two SMs.
cudaError_t launch_pair(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mo, const GemmParams &p,
                        int splits, int n_sm, cudaStream_t st) {
    const int tiles = ((p.M + 2 * tc::BM - 1) / (2 * tc::BM)) * (p.N / kBNWide) * splits;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(tc::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = kPairSmem;
    cfg.stream = st;
    cfg.gridDim = dim3(2 * std::min(tiles, std::max(1, n_sm / 2)), 1, 1);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, tc::k_gemm_tc_pair, ma, mb, mo, p, splits);
}

cudaError_t launch_persist(const void *A, const void *B, GemmParams &p, int splits, cudaStream_t st) {
    const int M = p.M, N = p.N, K = p.K;
    if (!gemm_tc_supported(N, K) || M < 1) return cudaErrorInvalidValue;
    const int bn = tile_n_for(M, N);
    const int s = std::max(1, splits);
    const int n_sm = sm_count_current();
    if (n_sm <= 0) return cudaErrorInvalidDevice;
    CUtensorMap ma, mb;
    if (bn == kBNWide) {   // CTA pairs: each CTA loads its 128 rows of A and 128 rows (half) of B
        if (!make_map(&ma, A, M, K, tc::BM) || !make_map(&mb, B, N, K, kBNWide / 2)) return cudaErrorInvalidValue;
        CUtensorMap mo{};
        if (p.swiglu_out == nullptr) {   // fp32 output [M][N], row stride ld_out: 32 x 32 boxes, 128-byte swizzle
            if (p.out == nullptr || p.ld_out % 4 != 0 || (reinterpret_cast<uintptr_t>(p.out) & 15u) != 0 ||
                !make_map_f32_2d(&mo, p.out, (uint64_t)M, (uint64_t)N, (uint64_t)p.ld_out * 4))
                return cudaErrorInvalidValue;
        }
        return launch_pair(ma, mb, mo, p, s, n_sm, st);
    }
    if (!make_map(&ma, A, M, K, tc::BM) || !make_map(&mb, B, N, K, bn)) return cudaErrorInvalidValue;
    return launch_cfg<kBNNarrow, kStagesNarrow>(ma, mb, p, s, n_sm, st);
}
}  // namespace

cudaError_t launch_gemm_tc(const void *A, int M, int K, const void *B, int N, float *out, int ld_out, int accumulate,
                           int splits, int *status, cudaStream_t st) {
    if (gemm_tc_swap_ok(M, N, K) && splits <= K / tc::BK)
        return launch_gemm_tc_swap(A, M, K, B, N, out, ld_out, accumulate, splits, nullptr, 0, status, st);
    GemmParams p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.out = out;
    p.ld_out = ld_out;
    p.accumulate = (accumulate || splits > 1) ? 1 : 0;
    p.status = status;
    return launch_persist(A, B, p, splits, st);
}

cudaError_t launch_gemm_tc_swiglu(const void *A, int M, int K, const void *B, int N, __nv_bfloat16 *out_bf16, int ld,
                                  int *status, cudaStream_t st) {
    if (out_bf16 == nullptr || N % 32 != 0 || ld % 8 != 0 || (reinterpret_cast<uintptr_t>(out_bf16) & 15u) != 0)
        return cudaErrorInvalidValue;
    if (gemm_tc_swap_ok(M, N, K))
        return launch_gemm_tc_swap(A, M, K, B, N, nullptr, 0, 0, 1, out_bf16, ld, status, st);
    GemmParams p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.status = status;
    p.swiglu_out = out_bf16;
    p.ld_swiglu = ld;
    return launch_persist(A, B, p, 1, st);
}

}  // namespace talker_k
