// Causal prefill attention on the fifth-generation tensor cores, head_dim 128
// ("qwentts.cpp/src/talker-forward.h", talker_layer_forward / talker_forward_core with
// n_past: query row r of a call starting at position pos0 attends keys [0, pos0 + r]; softmax
// of the scaled dot products, weighted sum of the values). One stream per launch: a prefill
// from position 0, an appended chunk (pos0 > 0, the earlier keys read from the cache), or one
// stream of a batched prefill.
//
// Per layer, k_kv_dense_tc first writes the KV group's keys densely, K [n_kv][L][128], and
// its values transposed, V^T [n_kv][128][L] (L = pos0 + T keys rounded up to 128, zero rows
// past them), so that both products read K-major operands; with Q8_0 storage the earlier
// rows are dequantized there and the call's own rows come from their exact bf16 copy.
//
// k_attn_prefill_tc: one CTA per 128 query rows of one q head (longest tiles first),
// walking key blocks of 128:
//   warp 0, one lane: TMA producer of K and V^T blocks (double buffered);
//   warp 1:           allocates TMEM (S[2], 128 columns each, and one O of 128 columns); one
//                     lane issues S_j = Q K_j^T (tcgen05.mma M=128 N=128, K=16 steps over
//                     head_dim) and O += P_j V_j (over the 128 keys), S_{j+1} ahead of P_j V_j;
//   warps 2..9:       two threads per query row (its TMEM lane), each owning half of the
//                     head dimension and half of each key block: stage the row of q (scaled by
//                     log2(e)/sqrt(head_dim), bf16) as the A operand, then per block read its
//                     64 scores of S_j once from TMEM (the row max, exchanged between the two
//                     halves through shared memory; then p = 2^(s - m), partial row sums, P_j
//                     as bf16 into shared memory for the second MMA). m is the exponent reference: it moves
//                     to the new row maximum only when that exceeds it by more than 8 (p stays
//                     below 2^8, exact enough in bf16 and f32), and then the threads rescale
//                     their half of O in TMEM before P_j is released; at the end O is read once,
//                     divided by the row sum and stored as bf16 rows through shared memory.
// Every mbarrier wait is bounded; a wait that gives up sets the device status word.
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"
#include "tcgen05.cuh"

using namespace talker_dev;

namespace talker_k {
namespace atc {

constexpr int HD = 128;
constexpr int BM = 128;                     // query rows per CTA
constexpr int BN = 128;                     // keys per block
constexpr int NTHREADS = 320;         // warp 0 TMA, warp 1 MMA, warps 2..9 softmax
constexpr uint32_t CB = 128 * 128;          // one swizzle column block: 128 rows x 128 bytes
constexpr uint32_t TILE = 2 * CB;           // a 128 x 128 bf16 operand (two column blocks of 64)
constexpr size_t SMEM = 1024 + 6 * (size_t)TILE;   // Q, K[2], V^T[2], P (+ alignment slack)
constexpr uint32_t IDESC = tc::instr_desc(128, 128);

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Byte offset of 16-byte chunk `ch` (0..15, 8 elements each) of row r in a K-major
// 128 x 128 bf16 operand stored as two 128-byte-swizzled column blocks.
__device__ __forceinline__ uint32_t op_off(int r, int ch) {
    return (uint32_t)(ch >> 3) * CB + (uint32_t)r * 128 + ((uint32_t)((ch & 7) ^ (r & 7)) << 4);
}

// 2^x on the special-function unit (ex2.approx.ftz: relative error ~2^-22, 2^-inf = +0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}


struct Params {
    const float *q;        // [T][n_q * HD] f32, QK-normed and rotated, unscaled
    __nv_bfloat16 *out;    // [T][n_q * HD] bf16
    int T, n_q, group, Lpad;
    int pos0;              // position of row 0 (keys [0, pos0 + T) are in the dense copy)
    float scale_log2;
    int *status;
};

__global__ void __launch_bounds__(NTHREADS, 1)
    k_attn_prefill_tc(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_vt,
                      const Params p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char *sQ = smem, *sK = smem + TILE, *sV = sK + 2 * TILE, *sP = sV + 2 * TILE;
    __shared__ __align__(8) uint64_t kv_full[2], kv_empty[2], s_full[2], s_free[2], o_full;
    __shared__ __align__(8) uint64_t p_full, q_full, mma_done;
    __shared__ uint32_t tmem_base_s;
    __shared__ __align__(8) uint64_t pair_bar[4];   // the two softmax warps of a lane quadrant
    __shared__ float mx_s[2][2][BM];   // [block parity][half][row]: the halves' row maxima
    __shared__ float l_s[2][BM];       // [half][row]: the halves' row sums

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_qt = (p.T + BM - 1) / BM;
    const int qt = n_qt - 1 - (int)blockIdx.x;
    const int h = blockIdx.y, kvh = h / p.group;
    const int last_row = min(p.T, (qt + 1) * BM) - 1;
    const int nb = (p.pos0 + last_row) / BN + 1;

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&kv_full[b], 1);
            mbar_init(&kv_empty[b], 1);
            mbar_init(&s_full[b], 1);
            mbar_init(&s_free[b], 8);   // one arrival per softmax warp
        }
        mbar_init(&o_full, 1);
        mbar_init(&p_full, 8);
        mbar_init(&q_full, 8);
        mbar_init(&mma_done, 1);
        for (int i = 0; i < 4; ++i) mbar_init(&pair_bar[i], 2);
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_s)),
                     "r"(512u)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        tc::tc_fence_before();
    }
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = tmem_base_s;   // columns [0,256): S[2]; [256,384): O

    if (warp == 0 && lane == 0) {
        // ---- producer
        for (int j = 0; j < nb; ++j) {
            const int b = j & 1;
            if (j >= 2 && !mbar_wait(&kv_empty[b], ((j >> 1) - 1) & 1, p.status)) break;
            mbar_arrive_expect_tx(&kv_full[b], 2 * TILE);
            for (int c = 0; c < 2; ++c) {
                tc::tma_load_2d(sK + b * TILE + c * CB, &map_k, c * 64, kvh * p.Lpad + j * BN, &kv_full[b]);
                tc::tma_load_2d(sV + b * TILE + c * CB, &map_vt, j * BN + c * 64, kvh * HD, &kv_full[b]);
            }
        }
        // every block consumed before the CTA can exit
        for (int j = max(0, nb - 2); j < nb; ++j) mbar_wait(&kv_empty[j & 1], (j >> 1) & 1, p.status);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        bool ok = mbar_wait(&q_full, 0, p.status);
        auto issue_s = [&](int j) -> bool {
            const int b = j & 1;
            if (!mbar_wait(&kv_full[b], (j >> 1) & 1, p.status)) return false;
            if (j >= 2 && !mbar_wait(&s_free[b], ((j >> 1) - 1) & 1, p.status)) return false;
            tc::tc_fence_after();
            const uint32_t qa = smem_u32(sQ), kb = smem_u32(sK + b * TILE);
#pragma unroll
            for (int k = 0; k < HD / 16; ++k) {
                const uint32_t off = (uint32_t)(k >> 2) * CB + (uint32_t)(k & 3) * 32;
                tc::umma_bf16(tmem + (uint32_t)(b * 128), tc::smem_desc(qa + off), tc::smem_desc(kb + off), IDESC,
                              k > 0 ? 1u : 0u);
            }
            tc::umma_commit(&s_full[b]);
            return true;
        };
        if (ok) ok = issue_s(0);
        for (int j = 0; j < nb && ok; ++j) {
            if (j + 1 < nb && !issue_s(j + 1)) break;
            const int b = j & 1;
            // P_j is staged and O rescaled (when the reference moved): O += P_j V_j
            if (!mbar_wait(&p_full, j & 1, p.status)) break;
            tc::tc_fence_after();
            const uint32_t pa = smem_u32(sP), vb = smem_u32(sV + b * TILE);
#pragma unroll
            for (int k = 0; k < BN / 16; ++k) {
                const uint32_t off = (uint32_t)(k >> 2) * CB + (uint32_t)(k & 3) * 32;
                tc::umma_bf16(tmem + 256u, tc::smem_desc(pa + off), tc::smem_desc(vb + off), IDESC,
                              (j > 0 || k > 0) ? 1u : 0u);
            }
            tc::umma_commit(&o_full);
            tc::umma_commit(&kv_empty[b]);
        }
        tc::umma_commit(&mma_done);   // arrives once every MMA issued above has completed
    } else if (warp >= 2) {
        // ---- softmax: warps w and w + 4 share TMEM lane quadrant w % 4 (query rows); half 0
        // takes keys 0..63 of each block and O columns 0..63, half 1 the other 64
        const int q4 = warp & 3, half = (warp - 2) >> 2;
        const int r = q4 * 32 + lane;
        const int grow = qt * BM + r;   // row of the call
        const int qpos = p.pos0 + grow;  // its position
        const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
        const int qd = p.n_q * HD;
        // exchange point of the warp pair: both warps' shared-memory writes before it are
        // visible after it; a bounded wait (a partner that gave up cannot stall this warp)
        uint32_t pair_phase = 0;
        auto pair_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(&pair_bar[q4]);
            const bool done = mbar_wait(&pair_bar[q4], pair_phase & 1, p.status);
            ++pair_phase;
            return done;
        };
        {
            const float *qs = p.q + (size_t)grow * qd + (size_t)h * HD;
#pragma unroll 4
            for (int c8 = 0; c8 < 8; ++c8) {
                const int ch = half * 8 + c8;
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f), c = a;
                if (grow < p.T) {
                    a = *reinterpret_cast<const float4 *>(qs + ch * 8);
                    c = *reinterpret_cast<const float4 *>(qs + ch * 8 + 4);
                }
                const float s = p.scale_log2;
                *reinterpret_cast<uint4 *>(sQ + op_off(r, ch)) =
                    make_uint4(pack2(a.x * s, a.y * s), pack2(a.z * s, a.w * s), pack2(c.x * s, c.y * s),
                               pack2(c.z * s, c.w * s));
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_full);
        }

        float m = -INFINITY, l = 0.f;   // exponent reference; this half's share of the row sum
        bool ok = true;
        const uint32_t o_base = lane_base + 256u + (uint32_t)(half * 64);   // this half's 64 O columns
        for (int j = 0; j < nb; ++j) {
            const int b = j & 1;
            if (!mbar_wait(&s_full[b], (j >> 1) & 1, p.status)) {
                ok = false;
                break;
            }
            tc::tc_fence_after();
            const int key0 = j * BN + half * 64;                 // first key of this half
            const bool masked = j * BN + BN - 1 > p.pos0 + qt * BM;   // the block reaches past the tile's first row
            const uint32_t sb = lane_base + (uint32_t)(b * 128 + half * 64);
            // pass 1: this half's 64 scores of the block (kept in registers) and their max over
            // the keys this row may see (key <= position)
            float sv[2][32];
            tc::tmem_ld32(sb, sv[0]);
            tc::tmem_ld32(sb + 32u, sv[1]);
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[b]);   // S_j is in registers: its buffer may take S_{j+2}
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (masked) {
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        if (key0 + c * 32 + t <= qpos) mx = fmaxf(mx, sv[c][t]);
                } else {
#pragma unroll
                    for (int t = 0; t < 32; ++t) mx = fmaxf(mx, sv[c][t]);
                }
            }
            mx_s[b][half][r] = mx;
            if (!pair_sync()) {
                ok = false;
                break;
            }
            // both halves see the same maxima: they move the reference together
            const float m_blk = fmaxf(mx_s[b][0][r], mx_s[b][1][r]);
            const bool move = m == -INFINITY || m_blk > m + 8.0f;
            // P's buffer is free, and O settled, once P_{j-1} V_{j-1} has completed
            if (j >= 1 && !mbar_wait(&o_full, (j - 1) & 1, p.status)) {
                ok = false;
                break;
            }
            tc::tc_fence_after();
            if (move) {
                const float m_new = fmaxf(m, m_blk);
                if (j >= 1) {   // O and l were formed against the old reference
                    const float sc = fast_exp2(m - m_new);
#pragma unroll 1
                    for (int c = 0; c < 2; ++c) {
                        float v[32];
                        tc::tmem_ld32(o_base + (uint32_t)(c * 32), v);
#pragma unroll
                        for (int t = 0; t < 32; ++t) v[t] *= sc;
                        tc::tmem_st32(o_base + (uint32_t)(c * 32), v);
                    }
                    l *= sc;
                }
                m = m_new;
            }
            // pass 2: p = 2^(s - m) (0 past the position), this half's row sum, P_j as bf16
            float ps = 0.f;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const float(&v)[32] = sv[c];
                uint32_t pk[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const int k = key0 + c * 32 + 2 * t;
                    float p0 = fast_exp2(v[2 * t] - m), p1 = fast_exp2(v[2 * t + 1] - m);
                    if (masked) {
                        p0 = (k <= qpos) ? p0 : 0.f;
                        p1 = (k + 1 <= qpos) ? p1 : 0.f;
                    }
                    ps += p0 + p1;
                    pk[t] = pack2(p0, p1);
                }
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    *reinterpret_cast<uint4 *>(sP + op_off(r, half * 8 + c * 4 + t)) =
                        make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
            }
            l += ps;
            tc::tc_fence_before();
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full);
        }
        if (ok && mbar_wait(&o_full, (nb - 1) & 1, p.status)) {
            tc::tc_fence_after();
            float o[64];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float v[32];
                tc::tmem_ld32(o_base + (uint32_t)(c * 32), v);
#pragma unroll
                for (int t = 0; t < 32; ++t) o[c * 32 + t] = v[t];
            }
            // row sum = both halves' shares; rows go out through shared memory (P's buffer: no
            // MMA reads it any more)
            l_s[half][r] = l;
            pair_sync();
            const float inv = 1.0f / (l_s[0][r] + l_s[1][r]);
            unsigned char *stg = sP;   // [128 rows][256 bytes], 16-byte chunks XOR-swizzled by row
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                const int ch = half * 8 + c8;
                *reinterpret_cast<uint4 *>(stg + r * 256 + ((ch ^ (r & 15)) << 4)) =
                    make_uint4(pack2(o[c8 * 8] * inv, o[c8 * 8 + 1] * inv), pack2(o[c8 * 8 + 2] * inv, o[c8 * 8 + 3] * inv),
                               pack2(o[c8 * 8 + 4] * inv, o[c8 * 8 + 5] * inv),
                               pack2(o[c8 * 8 + 6] * inv, o[c8 * 8 + 7] * inv));
            }
            pair_sync();   // both halves of the pair's 32 rows are staged
#pragma unroll 4
            for (int it = half * 8; it < half * 8 + 8; ++it) {
                const int rr = q4 * 32 + it * 2 + (lane >> 4), ch = lane & 15;
                const uint4 x = *reinterpret_cast<const uint4 *>(stg + rr * 256 + ((ch ^ (rr & 15)) << 4));
                const int g = qt * BM + rr;
                if (g < p.T) *reinterpret_cast<uint4 *>(p.out + (size_t)g * qd + (size_t)h * HD + ch * 8) = x;
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        mbar_wait(&mma_done, 0, p.status);   // no MMA may still write TMEM when it is released
        tc::tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512u) : "memory");
    }
}

// 8 dims (16-byte chunk ch) of row `row` of a Q8_0 tile ([64][HD] int8 codes, then [64][HD/32]
// fp16 scales), dequantized (code x scale, exact in f32) and rounded to bf16.
__device__ __forceinline__ uint4 q8_chunk_bf16(const unsigned char *tile, int row, int ch) {
    const uint2 cw = *reinterpret_cast<const uint2 *>(tile + row * HD + ch * 8);
    const float sc = __half2float(*reinterpret_cast<const __half *>(tile + kPage * HD + (row * (HD / 32) + ch / 4) * 2));
    const uint32_t w[2] = {cw.x, cw.y};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int b0 = (int)(signed char)((w[i >> 1] >> (16 * (i & 1))) & 0xffu);
        const int b1 = (int)(signed char)((w[i >> 1] >> (16 * (i & 1) + 8)) & 0xffu);
        o[i] = pack2((float)b0 * sc, (float)b1 * sc);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Dense K rows and transposed V rows of one (64-key block, KV head); keys at or past
// nkeys are written as zeros. Sources: the paged bf16 cache of `stream`; with Q8_0 storage,
// the dense bf16 copy of the call's rows [rows][n_kv][HD] for keys >= pos0 and the cache's
// Q8_0 tiles, dequantized, for the earlier keys.
__global__ void __launch_bounds__(256) k_kv_dense_tc(const CacheView c, int layer, int stream, int nkeys, int Lpad,
                                                     int pos0, const __nv_bfloat16 *dense_k,
                                                     const __nv_bfloat16 *dense_v, __nv_bfloat16 *kd,
                                                     __nv_bfloat16 *vt) {
    __shared__ __align__(16) __nv_bfloat16 vs[64][HD + 8];
    const int j0 = blockIdx.x * 64, kvh = blockIdx.y;
    for (int idx = threadIdx.x; idx < 64 * 16; idx += 256) {
        const int r = idx >> 4, ch = idx & 15, key = j0 + r;
        uint4 kx = make_uint4(0u, 0u, 0u, 0u), vx = kx;
        if (key < nkeys) {
            if (dense_k != nullptr && key >= pos0) {   // the call's own rows, exact up to bf16
                kx = *reinterpret_cast<const uint4 *>(dense_k + ((size_t)(key - pos0) * c.n_kv + kvh) * HD + ch * 8);
                vx = *reinterpret_cast<const uint4 *>(dense_v + ((size_t)(key - pos0) * c.n_kv + kvh) * HD + ch * 8);
            } else if (c.kv_q8) {   // a row of an earlier call, as stored
                const size_t tile = (size_t)kPage * HD + (size_t)kPage * (HD / 32) * 2;
                const size_t off = (size_t)c.page_table[stream * c.pages_per_stream + key / kPage] * c.page_elems +
                                   (size_t)(layer * c.n_kv + kvh) * tile;
                kx = q8_chunk_bf16(static_cast<const unsigned char *>(c.k) + off, key % kPage, ch);
                vx = q8_chunk_bf16(static_cast<const unsigned char *>(c.v) + off, key % kPage, ch);
            } else {
                const size_t off = (size_t)c.page_table[stream * c.pages_per_stream + key / kPage] * c.page_elems +
                                   ((size_t)(layer * c.n_kv + kvh) * kPage + key % kPage) * HD;
                kx = *reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(c.k) + off + ch * 8);
                vx = *reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(c.v) + off + ch * 8);
            }
        }
        *reinterpret_cast<uint4 *>(kd + ((size_t)kvh * Lpad + key) * HD + ch * 8) = kx;
        *reinterpret_cast<uint4 *>(&vs[r][ch * 8]) = vx;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < HD * 8; idx += 256) {
        const int d = idx % HD, kc = idx / HD;   // consecutive lanes: consecutive dims (conflict-free reads)
        uint32_t w[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const __nv_bfloat162 pr = __halves2bfloat162(vs[kc * 8 + 2 * t][d], vs[kc * 8 + 2 * t + 1][d]);
            w[t] = *reinterpret_cast<const uint32_t *>(&pr);
        }
        *reinterpret_cast<uint4 *>(vt + ((size_t)kvh * HD + d) * Lpad + j0 + kc * 8) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

}  // namespace atc

int attn_prefill_tc_lpad(int nkeys) { return (nkeys + atc::BN - 1) / atc::BN * atc::BN; }

bool attn_prefill_tc_supported(const AttnParams &a, int T) {
    const bool one_stream = a.rowmap.rows_per_stream == 0 || a.rowmap.rows_per_stream == T;
    // bf16 cache: the dense copy reads every key from the pages; Q8_0: the call's own rows from
    // their dense bf16 copy, earlier rows dequantized from the cache (any start position)
    return a.rowmap.mode == 1 && one_stream && a.out_bf16 && a.cache.head_dim == atc::HD && T >= 1 &&
           (a.cache.kv_bf16 || (a.cache.kv_q8 && a.dense_k != nullptr));
}

cudaError_t prepare_attn_prefill_tc() {
    return cudaFuncSetAttribute(atc::k_attn_prefill_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)atc::SMEM);
}

cudaError_t launch_attn_prefill_tc(const AttnParams &a, int T, __nv_bfloat16 *kd, __nv_bfloat16 *vt,
                                   cudaStream_t st) {
    if (!attn_prefill_tc_supported(a, T) || kd == nullptr || vt == nullptr) return cudaErrorInvalidValue;
    const int nkeys = a.rowmap.pos0 + T, Lpad = attn_prefill_tc_lpad(nkeys);
    const int n_kv = a.cache.n_kv;
    atc::k_kv_dense_tc<<<dim3(Lpad / 64, n_kv), 256, 0, st>>>(a.cache, a.layer, a.rowmap.stream0, nkeys, Lpad,
                                                               a.rowmap.pos0, a.dense_k, a.dense_v, kd, vt);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap mk, mv;
    if (!make_map_bf16_2d(&mk, kd, (uint64_t)n_kv * Lpad, atc::HD, atc::HD * 2, 64, 128) ||
        !make_map_bf16_2d(&mv, vt, (uint64_t)n_kv * atc::HD, (uint64_t)Lpad, (uint64_t)Lpad * 2, 64, 128))
        return cudaErrorInvalidValue;
    atc::Params p{};
    p.q = a.q;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.T = T;
    p.n_q = a.n_q;
    p.group = a.group;
    p.Lpad = Lpad;
    p.pos0 = a.rowmap.pos0;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.status = a.status;
    const dim3 grid((T + atc::BM - 1) / atc::BM, a.n_q);
    atc::k_attn_prefill_tc<<<grid, atc::NTHREADS, atc::SMEM, st>>>(mk, mv, p);
    return cudaGetLastError();
}

}  // namespace talker_k
