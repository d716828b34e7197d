// Element-wise stages of the tensor-core prefill path (the projections run on
// the tcgen05 GEMM):
//   k_rmsnorm_bf16 (tall inputs: k_rmsnorm_bf16_rows, a warp per row):
//                   x / sqrt(mean(x^2) + eps) * w, rounded to bf16 as the next
//                   GEMM's A operand ("talker-forward.h", talker_layer_forward
//                   pre-norm and MLP pre-norm); it also clears the split-K
//                   accumulator of the GEMM that follows, when there is one;
//   k_qkv_post (k_qkv_post_v: head_dim 128 without Q8_0, 16-byte accesses):
//                   per (row, head) of the raw projections: QK-RMSNorm with the
//                   [hd] gain and NEOX RoPE at the row's position for q and k,
//                   k and v appended to the cache at that position (set_rows),
//                   q kept in f32 for attention;
//   k_swiglu_bf16:  silu(gate) * up from the row-interleaved [gate; up]
//                   projection (columns 2j, 2j+1), rounded to bf16; the f32 split-K
//                   sum is zeroed behind the read, ready for the next accumulation.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"

using namespace talker_dev;

namespace talker_k {

// Launch with programmatic dependent launch: the kernel starts while its predecessor drains
// and waits for it (griddepcontrol.wait) before touching the predecessor's outputs.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// One CTA per row: every thread stages its float4s of the row (one round trip), the sum of
// squares is reduced across the CTA, then the scaled bf16 row is written.
__global__ void k_rmsnorm_bf16(float *x, int ld, const float *w, float eps, int rows, int H,
                               __nv_bfloat16 *out, CodeGather gather, int *status, float4 *zero, size_t zero_n4) {
    __shared__ float red[32];
    const int row = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_launch_dependents();
    pdl_wait();
    if (zero != nullptr) {   // this CTA's share of the next GEMM's split-K accumulator
        const size_t per = (zero_n4 + gridDim.x - 1) / gridDim.x;
        const size_t b = (size_t)blockIdx.x * per, e = b + per < zero_n4 ? b + per : zero_n4;
        for (size_t i = b + threadIdx.x; i < e; i += blockDim.x) zero[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float *xr = x + (size_t)row * ld;
    constexpr int MAXV = 4;   // float4s per thread (H <= 4 * 4 * blockDim.x)
    float4 v[MAXV];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
        const int k = (threadIdx.x + i * blockDim.x) * 4;
        if (gather.n > 0) {   // the row from codebook tables, kept as the residual stream
            v[i] = k < H ? gather_row4(gather, row, k, H, status) : make_float4(0.f, 0.f, 0.f, 0.f);
            if (k < H) *reinterpret_cast<float4 *>(x + (size_t)row * ld + k) = v[i];
        } else {
            v[i] = k < H ? *reinterpret_cast<const float4 *>(xr + k) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
    const float inv = 1.0f / sqrtf(t / (float)H + eps);
    __nv_bfloat16 *o = out + (size_t)row * H;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
        const int k = (threadIdx.x + i * blockDim.x) * 4;
        if (k < H) {
            const float4 g = *reinterpret_cast<const float4 *>(w + k);
            *reinterpret_cast<__nv_bfloat162 *>(o + k) = __floats2bfloat162_rn(v[i].x * inv * g.x, v[i].y * inv * g.y);
            *reinterpret_cast<__nv_bfloat162 *>(o + k + 2) = __floats2bfloat162_rn(v[i].z * inv * g.z, v[i].w * inv * g.w);
        }
    }
}

// Tall inputs: one warp per row (4 rows per CTA), the row held in registers (H <= 1024).
__global__ void k_rmsnorm_bf16_rows(float *x, int ld, const float *w, float eps, int rows, int H,
                                    __nv_bfloat16 *out, CodeGather gather, int *status, float4 *zero, size_t zero_n4) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * 4 + warp;
    pdl_launch_dependents();
    pdl_wait();
    if (zero != nullptr) {
        const size_t per = (zero_n4 + gridDim.x - 1) / gridDim.x;
        const size_t b = (size_t)blockIdx.x * per, e = b + per < zero_n4 ? b + per : zero_n4;
        for (size_t i = b + threadIdx.x; i < e; i += blockDim.x) zero[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (row >= rows) return;
    constexpr int MAXV = 8;   // float4s per lane
    float4 v[MAXV];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
        const int k = (lane + 32 * i) * 4;
        if (k < H) {
            if (gather.n > 0) {
                v[i] = gather_row4(gather, row, k, H, status);
                *reinterpret_cast<float4 *>(x + (size_t)row * ld + k) = v[i];
            } else {
                v[i] = *reinterpret_cast<const float4 *>(x + (size_t)row * ld + k);
            }
        } else {
            v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
    }
    ss = warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss / (float)H + eps);
    __nv_bfloat16 *o = out + (size_t)row * H;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
        const int k = (lane + 32 * i) * 4;
        if (k < H) {
            const float4 g = *reinterpret_cast<const float4 *>(w + k);
            const __nv_bfloat162 lo = __floats2bfloat162_rn(v[i].x * inv * g.x, v[i].y * inv * g.y);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(v[i].z * inv * g.z, v[i].w * inv * g.w);
            uint2 u;
            u.x = *reinterpret_cast<const uint32_t *>(&lo);
            u.y = *reinterpret_cast<const uint32_t *>(&hi);
            *reinterpret_cast<uint2 *>(o + k) = u;
        }
    }
}

// One warp per (row, head); the row map gives each row's stream and position
// (prefill: stream0 at pos0 + r; decode: stream r at cur_len[r]).
__global__ void k_qkv_post(const float *raw, int rows, int n_q, int n_kv, int hd, const float *q_norm,
                           const float *k_norm, const float2 *rope, float eps, float *q_out, CacheView cache, int layer,
                           RowMap rm, int *status, __nv_bfloat16 *dense_kv) {
    const int n_heads = n_q + 2 * n_kv;
    const int item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    pdl_launch_dependents();
    pdl_wait();
    if (item >= rows * n_heads) return;
    const int r = item / n_heads, h = item - r * n_heads;
    const int half = hd >> 1;
    const int qkv_n = n_heads * hd;
    const float *src = raw + (size_t)r * qkv_n + (size_t)h * hd;
    const bool is_q = h < n_q, is_k = !is_q && h < n_q + n_kv;
    float a[2], b[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int i = lane + 32 * t;
        a[t] = (i < half) ? src[i] : 0.f;
        b[t] = (i < half) ? src[i + half] : 0.f;
    }
    const int pos = rowmap_pos(rm, r);
    const int stream = rowmap_stream(rm, r);
    if (pos < 0 || pos >= cache.max_seq) {
        if (lane == 0) atomicOr(status, ST_BAD_POSITION);
        return;
    }
    if (is_q || is_k) {
        const float *gain = is_q ? q_norm : k_norm;
        const float ss = warp_sum(a[0] * a[0] + b[0] * b[0] + a[1] * a[1] + b[1] * b[1]);
        const float inv = 1.0f / sqrtf(ss / (float)hd + eps);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int i = lane + 32 * t;
            if (i < half) {
                const float x0 = a[t] * inv * gain[i], x1 = b[t] * inv * gain[i + half];
                const float2 cs = rope[(size_t)pos * half + i];
                a[t] = x0 * cs.x - x1 * cs.y;
                b[t] = x1 * cs.x + x0 * cs.y;
            }
        }
    }
    if (is_q) {
        float *d = q_out + (size_t)r * n_q * hd + (size_t)h * hd;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int i = lane + 32 * t;
            if (i < half) {
                d[i] = a[t];
                d[i + half] = b[t];
            }
        }
        return;
    }
    const int kvh = is_k ? h - n_q : h - n_q - n_kv;
    const int page = cache.page_table[(size_t)stream * cache.pages_per_stream + pos / kPage];
    if (cache.kv_q8) {
        // Q8_0 tile of (page, layer, head): [64][hd] codes, then [64][hd/32] fp16 scales; each valid
        // register of the warp holds one block of 32 dims (lane = dim % 32, hd is 64 or 128)
        const size_t tile = (size_t)kPage * hd + (size_t)kPage * (hd / 32) * 2;
        unsigned char *t = static_cast<unsigned char *>(is_k ? cache.k : cache.v) + (size_t)page * cache.page_elems +
                           (size_t)(layer * n_kv + kvh) * tile;
        const int row = pos % kPage;
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                if (32 * j >= half) continue;
                const int d0 = 32 * j + u * half;
                q8_store_block(t, row * hd + d0, kPage * hd + (row * (hd / 32) + d0 / 32) * 2, u ? b[j] : a[j], lane);
            }
        // the call itself attends its rows unquantized
        __nv_bfloat16 *dk = dense_kv + ((size_t)(is_k ? 0 : rows) * n_kv + (size_t)r * n_kv + kvh) * hd;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int i = lane + 32 * j;
            if (i < half) {
                dk[i] = __float2bfloat16_rn(a[j]);
                dk[i + half] = __float2bfloat16_rn(b[j]);
            }
        }
        return;
    }
    const size_t off = (size_t)page * cache.page_elems + ((size_t)(layer * n_kv + kvh) * kPage + pos % kPage) * hd;
    void *base = is_k ? cache.k : cache.v;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int i = lane + 32 * t;
        if (i < half) {
            if (cache.kv_bf16) {
                __nv_bfloat16 *d = static_cast<__nv_bfloat16 *>(base) + off;
                d[i] = __float2bfloat16_rn(a[t]);
                d[i + half] = __float2bfloat16_rn(b[t]);
            } else {
                float *d = static_cast<float *>(base) + off;
                d[i] = a[t];
                d[i + half] = b[t];
            }
        }
    }
}

// head_dim 128, bf16 or f32 storage: the same per (row, head) steps with 16-byte accesses. Lane l
// holds dims 64 (l / 16) + 4 (l % 16) .. +3; the RoPE partner (dim +- 64) is lane l ^ 16.
__global__ void k_qkv_post_v(const float *raw, int rows, int n_q, int n_kv, const float *q_norm, const float *k_norm,
                             const float2 *rope, float eps, float *q_out, CacheView cache, int layer, RowMap rm,
                             int *status) {
    constexpr int HD = 128, HALF = 64;
    const int n_heads = n_q + 2 * n_kv;
    const int item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    pdl_launch_dependents();
    pdl_wait();
    if (item >= rows * n_heads) return;
    const int r = item / n_heads, h = item - r * n_heads;
    const int part = lane >> 4, i0 = (lane & 15) * 4, d0 = part * HALF + i0;
    const float4 x = *reinterpret_cast<const float4 *>(raw + ((size_t)r * n_heads + h) * HD + d0);
    const int pos = rowmap_pos(rm, r);
    const int stream = rowmap_stream(rm, r);
    if (pos < 0 || pos >= cache.max_seq) {
        if (lane == 0) atomicOr(status, ST_BAD_POSITION);
        return;
    }
    const bool is_q = h < n_q, is_k = !is_q && h < n_q + n_kv;
    float y[4] = {x.x, x.y, x.z, x.w};
    if (is_q || is_k) {
        const float *gain = is_q ? q_norm : k_norm;
        const float ss = warp_sum(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w);
        const float inv = 1.0f / sqrtf(ss / (float)HD + eps);
        const float4 g = *reinterpret_cast<const float4 *>(gain + d0);
        const float n[4] = {x.x * inv * g.x, x.y * inv * g.y, x.z * inv * g.z, x.w * inv * g.w};
        const float4 cs01 = *reinterpret_cast<const float4 *>(rope + (size_t)pos * HALF + i0);
        const float4 cs23 = *reinterpret_cast<const float4 *>(rope + (size_t)pos * HALF + i0 + 2);
        const float c[4] = {cs01.x, cs01.z, cs23.x, cs23.z}, sn[4] = {cs01.y, cs01.w, cs23.y, cs23.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float o = __shfl_xor_sync(0xffffffffu, n[e], 16);
            y[e] = part == 0 ? n[e] * c[e] - o * sn[e] : n[e] * c[e] + o * sn[e];
        }
    }
    if (is_q) {
        *reinterpret_cast<float4 *>(q_out + ((size_t)r * n_q + h) * HD + d0) = make_float4(y[0], y[1], y[2], y[3]);
        return;
    }
    const int kvh = is_k ? h - n_q : h - n_q - n_kv;
    const int page = cache.page_table[(size_t)stream * cache.pages_per_stream + pos / kPage];
    const size_t off = (size_t)page * cache.page_elems + ((size_t)(layer * n_kv + kvh) * kPage + pos % kPage) * HD + d0;
    void *base = is_k ? cache.k : cache.v;
    if (cache.kv_bf16) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(y[0], y[1]), hi = __floats2bfloat162_rn(y[2], y[3]);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t *>(&lo);
        u.y = *reinterpret_cast<const uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(base) + off) = u;
    } else {
        *reinterpret_cast<float4 *>(static_cast<float *>(base) + off) = make_float4(y[0], y[1], y[2], y[3]);
    }
}

__global__ void k_swiglu_bf16(float *gu, int rows, int I, __nv_bfloat16 *out) {
    const size_t n = (size_t)rows * I;
    pdl_launch_dependents();
    pdl_wait();
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t r = i / I, j = i - r * I;
        float2 *src = reinterpret_cast<float2 *>(gu + r * 2 * I + 2 * j);
        const float2 v = *src;
        *src = make_float2(0.f, 0.f);
        out[i] = __float2bfloat16_rn(v.x / (1.0f + expf(-v.x)) * v.y);
    }
}

// from this many rows on, the one-warp-per-row form (below it, a CTA per row spreads the work wider)
constexpr int kRmsRowsMin = 2048;

cudaError_t launch_rmsnorm_bf16(float *x, int ld, const float *w, float eps, int rows, int H, void *out,
                                cudaStream_t st, const CodeGather *gather, int *status, float *zero, size_t zero_n) {
    const int threads = 256;
    if (H % 4 || H > 4 * 4 * threads || (gather != nullptr && gather->n > 0 && status == nullptr))
        return cudaErrorInvalidValue;
    if (zero != nullptr && (zero_n % 4 != 0 || (reinterpret_cast<uintptr_t>(zero) & 15u) != 0))
        return cudaErrorInvalidValue;
    const CodeGather none{};
    if (rows >= kRmsRowsMin && H <= 1024)   // tall: a warp per row
        return launch_pdl(k_rmsnorm_bf16_rows, dim3((rows + 3) / 4), dim3(128), st, x, ld, w, eps, rows, H,
                          static_cast<__nv_bfloat16 *>(out), gather ? *gather : none, status,
                          reinterpret_cast<float4 *>(zero), zero != nullptr ? zero_n / 4 : (size_t)0);
    return launch_pdl(k_rmsnorm_bf16, dim3(rows), dim3(threads), st, x, ld, w, eps, rows, H,
                      static_cast<__nv_bfloat16 *>(out), gather ? *gather : none, status,
                      reinterpret_cast<float4 *>(zero), zero != nullptr ? zero_n / 4 : (size_t)0);
}

cudaError_t launch_qkv_post(const float *raw, int rows, int n_q, int n_kv, int hd, const float *q_norm,
                            const float *k_norm, const float2 *rope, float eps, float *q_out, const CacheView &cache,
                            int layer, const RowMap &rm, int *status, cudaStream_t st, __nv_bfloat16 *dense_kv) {
    if (cache.kv_q8 && dense_kv == nullptr) return cudaErrorInvalidValue;
    const long long items = (long long)rows * (n_q + 2 * n_kv);
    const int per_block = 8;
    if (!cache.kv_q8 && hd == 128)
        return launch_pdl(k_qkv_post_v, dim3((unsigned)((items + per_block - 1) / per_block)), dim3(per_block * 32), st,
                          raw, rows, n_q, n_kv, q_norm, k_norm, rope, eps, q_out, cache, layer, rm, status);
    return launch_pdl(k_qkv_post, dim3((unsigned)((items + per_block - 1) / per_block)), dim3(per_block * 32), st,
                      raw, rows, n_q, n_kv, hd, q_norm, k_norm, rope, eps, q_out, cache, layer, rm, status, dense_kv);
}

cudaError_t launch_swiglu_bf16(float *gu, int rows, int I, void *out, cudaStream_t st) {
    const size_t n = (size_t)rows * I;
    const int blocks = (int)std::min<size_t>((n + 255) / 256, 4096);
    return launch_pdl(k_swiglu_bf16, dim3(blocks), dim3(256), st, gu, rows, I, static_cast<__nv_bfloat16 *>(out));
}

}  // namespace talker_k
