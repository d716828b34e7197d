// Causal attention of a prefill on the tensor cores ("qwentts.cpp/src/talker-forward.h",
// talker_layer_forward, attention step, every row r at position pos0 + r attending the
// cached keys [0, pos0 + r]).
//
// One CTA: 64 query rows of one q head (16 per warp), walking the KV group's cached pages
// (64 keys each, [pos][hd] bf16) in order. S = Q K^T and O += P V run on mma.sync
// m16n8k16 (bf16 in, f32 accumulate); the softmax is online in base 2 with the
// 1/sqrt(hd) * log2(e) scale folded into q. K and V pages are staged by cp.async into
// double-buffered shared memory with the 16-byte chunks of each row XOR-swizzled by the
// row index, so the ldmatrix reads are free of bank conflicts. Output rows are bf16
// (the o_proj GEMM's A operand).
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

using namespace talker_dev;

namespace talker_k {
namespace {

constexpr int kBM = 64;    // query rows per CTA (per head)
constexpr int kWarpsPerHead = 4;   // 16 query rows per warp

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// d += a * b for one m16n8k16 tile (bf16 inputs, f32 accumulators)
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Byte offset of 16-byte chunk c of row r in a [64][HD] bf16 tile (rows of HD * 2 bytes).
template <int HD>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)(r * HD * 2 + ((c ^ (r & 7)) << 4));
}

}  // namespace

// q: f32 rows [T][n_q * HD] (QK-normed, rotated, unscaled); out: bf16 rows [T][n_q * HD].
// Query row r sits at position pos0 + r of stream `stream`; the cache already holds the
// keys and values of positions [0, pos0 + T).
// HPC q heads of one KV group per CTA (warps 4*i..4*i+3 take head i): each K / V page
// staged in shared memory serves all of them.
template <int HD, int HPC>
__global__ void __launch_bounds__(kWarpsPerHead * HPC * 32) k_attn_prefill(const float *q, __nv_bfloat16 *out, int T, int pos0,
                                                               int stream, int n_q, int group, int layer,
                                                               float scale_log2, CacheView cache,
                                                               const __nv_bfloat16 *dense_k,
                                                               const __nv_bfloat16 *dense_v, int n_streams) {
    constexpr int NKS = HD / 16;        // k-steps of S = Q K^T
    constexpr int NNO = HD / 8;         // n-tiles of O
    constexpr int TILE = kPage * HD;    // elements of one K (or V) page of one head
    constexpr int CHUNKS = TILE * 2 / 16;
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t sbase = smem_u32(smem);   // [2 buffers][K, V][TILE] bf16
    constexpr int NTH = kWarpsPerHead * HPC * 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g8 = lane >> 2, t4 = lane & 3;
    // n_streams streams of T rows each (stream s = rows s*T .. s*T + T - 1); the longest tiles
    // of every stream go first
    const int tiles_ps = (T + kBM - 1) / kBM;
    const int qt = tiles_ps - 1 - (int)(blockIdx.x / n_streams);
    const int sb = blockIdx.x % n_streams;
    const size_t rbase = (size_t)sb * T;   // this stream's first row in q, out and the dense copy
    stream += sb;
    const int h = blockIdx.y * HPC + warp / kWarpsPerHead;
    const int kvh = (blockIdx.y * HPC) / group;
    const int qd = n_q * HD;
    const int row0 = qt * kBM + (warp % kWarpsPerHead) * 16;   // this warp's first query row
    // launched with programmatic dependent launch: q and the call's K/V rows come from the
    // previous kernel
    pdl_launch_dependents();
    pdl_wait();

    // Q fragments (A operand, row-major 16 x HD), scaled for base-2 exponentials
    uint32_t qa[NKS][4];
#pragma unroll
    for (int ks = 0; ks < NKS; ++ks) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = row0 + g8 + 8 * half;
            float2 lo = make_float2(0.f, 0.f), hi = make_float2(0.f, 0.f);
            if (r < T) {
                const float *src = q + (rbase + r) * qd + (size_t)h * HD + ks * 16 + 2 * t4;
                lo = *reinterpret_cast<const float2 *>(src);
                hi = *reinterpret_cast<const float2 *>(src + 8);
            }
            qa[ks][half] = pack_bf16(lo.x * scale_log2, lo.y * scale_log2);
            qa[ks][2 + half] = pack_bf16(hi.x * scale_log2, hi.y * scale_log2);
        }
    }

    // last query position of the CTA decides how many key pages it reads
    const int last_row = min(T, (qt + 1) * kBM) - 1;
    const int n_blocks = (pos0 + last_row) / kPage + 1;
    const int *ptab = cache.page_table + (size_t)stream * cache.pages_per_stream;
    const __nv_bfloat16 *kpool = static_cast<const __nv_bfloat16 *>(cache.k);
    const __nv_bfloat16 *vpool = static_cast<const __nv_bfloat16 *>(cache.v);
    const size_t head_off = (size_t)(layer * cache.n_kv + kvh) * kPage * HD;

    // Keys [0, pos0 + T) exist; rows of a block past them are zero-filled, so that a stale or
    // poisoned cache tail never reaches the products (a masked weight is 0, and 0 * NaN = NaN).
    const int nkeys = pos0 + T;
    auto load_block = [&](int kb, int buf) {
        const __nv_bfloat16 *ks, *vs;
        size_t rs;   // row stride (elements)
        if (dense_k != nullptr) {   // the call's own rows (Q8_0 storage; pos0 = 0)
            ks = dense_k + ((rbase + (size_t)kb * kPage) * cache.n_kv + kvh) * HD;
            vs = dense_v + ((rbase + (size_t)kb * kPage) * cache.n_kv + kvh) * HD;
            rs = (size_t)cache.n_kv * HD;
        } else {
            const size_t off = (size_t)ptab[kb] * cache.page_elems + head_off;
            ks = kpool + off;
            vs = vpool + off;
            rs = HD;
        }
        const uint32_t kdst = sbase + (uint32_t)(buf * 2) * TILE * 2, vdst = kdst + TILE * 2;
        for (int i = threadIdx.x; i < CHUNKS; i += NTH) {
            const int r = i / (HD / 8), c = i % (HD / 8);
            if (kb * kPage + r < nkeys) {
                cp_async16(kdst + swz<HD>(r, c), ks + r * rs + c * 8);
                cp_async16(vdst + swz<HD>(r, c), vs + r * rs + c * 8);
            } else {
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(kdst + swz<HD>(r, c)), "r"(0) : "memory");
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vdst + swz<HD>(r, c)), "r"(0) : "memory");
            }
        }
    };

    float o[NNO][4];
#pragma unroll
    for (int n = 0; n < NNO; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
    const int qpos0 = pos0 + row0 + g8, qpos1 = qpos0 + 8;   // positions of this thread's two rows

    load_block(0, 0);
    cp_async_commit();
    for (int kb = 0; kb < n_blocks; ++kb) {
        const int buf = kb & 1;
        if (kb + 1 < n_blocks) load_block(kb + 1, buf ^ 1);
        cp_async_commit();
        cp_async_wait<1>();   // block kb has landed (for this thread)
        __syncthreads();      // ... and for every thread
        const uint32_t kbase = sbase + (uint32_t)(buf * 2) * TILE * 2, vbase = kbase + TILE * 2;

        // S = Q K^T for 64 keys: 8 n-tiles of 8 keys
        float s[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int ks = 0; ks < NKS; ks += 2) {
                // matrices: keys nt*8..+7 x dims (ks, lo), (ks, hi), (ks+1, lo), (ks+1, hi)
                const int r = nt * 8 + (lane & 7), c = 2 * ks + (lane >> 3);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kbase + swz<HD>(r, c), b0, b1, b2, b3);
                mma_bf16(s[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                mma_bf16(s[nt], qa[ks + 1][0], qa[ks + 1][1], qa[ks + 1][2], qa[ks + 1][3], b2, b3);
            }
        }
        // causal mask (only the blocks that reach past a row's position have masked keys)
        const int key0 = kb * kPage;
        if (key0 + kPage - 1 > qpos0) {
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int k0 = key0 + nt * 8 + 2 * t4;
                if (k0 > qpos0) s[nt][0] = -INFINITY;
                if (k0 + 1 > qpos0) s[nt][1] = -INFINITY;
                if (k0 > qpos1) s[nt][2] = -INFINITY;
                if (k0 + 1 > qpos1) s[nt][3] = -INFINITY;
            }
        }
        // online softmax: this thread holds rows g8 (s[.][0..1]) and g8 + 8 (s[.][2..3]);
        // the four lanes of a quad share a row
        float mx[2] = {m_r[0], m_r[1]};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            mx[0] = fmaxf(mx[0], fmaxf(s[nt][0], s[nt][1]));
            mx[1] = fmaxf(mx[1], fmaxf(s[nt][2], s[nt][3]));
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
            mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
        }
        const float alpha0 = exp2f(m_r[0] - mx[0]), alpha1 = exp2f(m_r[1] - mx[1]);   // 0 on the first block
        m_r[0] = mx[0];
        m_r[1] = mx[1];
        float ps0 = 0.f, ps1 = 0.f;
        uint32_t pa[4][4];   // P as A fragments, one per 16 keys
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const float p0 = exp2f(s[nt][0] - mx[0]), p1 = exp2f(s[nt][1] - mx[0]);
            const float p2 = exp2f(s[nt][2] - mx[1]), p3 = exp2f(s[nt][3] - mx[1]);
            ps0 += p0 + p1;
            ps1 += p2 + p3;
            pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p0, p1);
            pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p2, p3);
        }
        l_r[0] = l_r[0] * alpha0 + ps0;   // per-thread partial sums; the quad adds them at the end
        l_r[1] = l_r[1] * alpha1 + ps1;
#pragma unroll
        for (int n = 0; n < NNO; ++n) {
            o[n][0] *= alpha0;
            o[n][1] *= alpha0;
            o[n][2] *= alpha1;
            o[n][3] *= alpha1;
        }
        // O += P V: k-steps of 16 keys, n-tiles of 8 dims; V^T fragments by transposed ldmatrix
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
            for (int n = 0; n < NNO; n += 2) {
                // matrices: keys kk*16 + (0..7 | 8..15) x dims n*8.. (and (n+1)*8..)
                const int r = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, c = n + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vbase + swz<HD>(r, c), b0, b1, b2, b3);
                mma_bf16(o[n], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
                mma_bf16(o[n + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
            }
        }
        __syncthreads();   // every warp is done with buffer `buf` before it is refilled
    }
    cp_async_wait<0>();

    // normalise and store rows < T
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        l_r[i] += __shfl_xor_sync(0xffffffffu, l_r[i], 1);
        l_r[i] += __shfl_xor_sync(0xffffffffu, l_r[i], 2);
    }
    const float inv0 = 1.0f / l_r[0], inv1 = 1.0f / l_r[1];
    const int r0 = row0 + g8, r1 = r0 + 8;
#pragma unroll
    for (int n = 0; n < NNO; ++n) {
        const int d = n * 8 + 2 * t4;
        if (r0 < T)
            *reinterpret_cast<uint32_t *>(out + (rbase + r0) * qd + (size_t)h * HD + d) =
                pack_bf16(o[n][0] * inv0, o[n][1] * inv0);
        if (r1 < T)
            *reinterpret_cast<uint32_t *>(out + (rbase + r1) * qd + (size_t)h * HD + d) =
                pack_bf16(o[n][2] * inv1, o[n][3] * inv1);
    }
}

template <int HD>
constexpr size_t ap_smem() {   // (independent of the heads per CTA)
    return (size_t)2 * 2 * kPage * HD * 2;   // two buffers of a K page and a V page
}

template <int HD, int HPC>
static cudaError_t launch_ap(const AttnParams &a, int T, cudaStream_t st) {
    // rows_per_stream > 0: n_streams = T / rows_per_stream streams of rows_per_stream rows
    const int rps = a.rowmap.rows_per_stream > 0 ? a.rowmap.rows_per_stream : T;
    const int ns = T / rps;
    const dim3 grid(ns * ((rps + kBM - 1) / kBM), a.n_q / HPC);
    const float scale_log2 = a.scale * 1.4426950408889634f;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kWarpsPerHead * HPC * 32, 1, 1);
    cfg.dynamicSmemBytes = ap_smem<HD>();
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_attn_prefill<HD, HPC>, a.q, static_cast<__nv_bfloat16 *>(a.out), rps,
                              a.rowmap.pos0, a.rowmap.stream0, a.n_q, a.group, a.layer, scale_log2, a.cache,
                              static_cast<const __nv_bfloat16 *>(a.dense_k), static_cast<const __nv_bfloat16 *>(a.dense_v),
                              ns);
}

template <int HD, int HPC>
static cudaError_t raise_ap() {
    return cudaFuncSetAttribute(k_attn_prefill<HD, HPC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)ap_smem<HD>());
}

cudaError_t prepare_attn_prefill() {
    cudaError_t e = raise_ap<128, 1>();
    e = e ? e : raise_ap<128, 2>();
    e = e ? e : raise_ap<64, 1>();
    return e ? e : raise_ap<64, 2>();
}

// bf16 cache, or Q8_0 storage (whose prefill reads the call's rows from the dense bf16 copy)
bool attn_prefill_supported(int kv_kind, int head_dim) {
    return (kv_kind == 1 || kv_kind == 2) && (head_dim == 64 || head_dim == 128);
}

cudaError_t launch_attn_prefill(int head_dim, const AttnParams &a, int T, cudaStream_t st) {
    if (a.rowmap.mode != 1 || !a.out_bf16) return cudaErrorInvalidValue;
    if (a.rowmap.rows_per_stream > 0 && T % a.rowmap.rows_per_stream) return cudaErrorInvalidValue;
    if ((a.dense_k != nullptr) != (a.dense_v != nullptr) || (a.dense_k != nullptr && a.rowmap.pos0 != 0))
        return cudaErrorInvalidValue;
    if (a.cache.kv_q8 && a.dense_k == nullptr) return cudaErrorInvalidValue;
    const bool pair = a.group % 2 == 0;   // two q heads of a KV group share each staged page
    if (head_dim == 128) return pair ? launch_ap<128, 2>(a, T, st) : launch_ap<128, 1>(a, T, st);
    if (head_dim == 64) return pair ? launch_ap<64, 2>(a, T, st) : launch_ap<64, 1>(a, T, st);
    return cudaErrorInvalidValue;
}

}  // namespace talker_k
